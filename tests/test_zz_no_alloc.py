"""qmoe_forward_noalloc (library-owned static device workspace) through the
C ABI, against qmoe_forward with a caller workspace.  Collected last so it
runs both after the other GPU tests and, on its own, in a fresh process."""
import pytest
import torch

from int4_block_quantized_gb300 import binding as B
from int4_block_quantized_gb300 import synthetic as S
from qmoe_check import assert_close_layer, to_f64

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from int4_block_quantized_gb300 import build
    build.build()
    assert torch.cuda.is_available()


@pytest.mark.parametrize("name", ["tiny", "decode", "verify"])
def test_noalloc_matches_workspace_entry_point_twice(name):
    wl = S.WORKLOADS[name]
    L = S.make_layer(wl, seed=21, device=DEV)
    ref, rw, ri = B.qmoe_forward(L, return_routing=True)
    for _ in range(2):  # the second call sees the scratch the first one left
        o, tw, ti = B.qmoe_forward_noalloc(L, return_routing=True)
        torch.cuda.synchronize()
        assert B.qmoe_noalloc_status() == (0, 0)
        assert torch.equal(ti, ri)
        assert torch.allclose(tw, rw, rtol=0, atol=1e-6)
        assert_close_layer(o, to_f64(ref), name + " noalloc")


def test_noalloc_residual_accumulate():
    wl = S.WORKLOADS["verify"]
    L = S.make_layer(wl, seed=22, device=DEV)
    base = torch.randn(wl.T, wl.H, generator=torch.Generator(device=DEV).manual_seed(5), device=DEV).half()
    ref = B.qmoe_forward(L, out=base.clone(), accumulate=True)
    o = B.qmoe_forward_noalloc(L, out=base.clone(), accumulate=True)
    assert B.qmoe_noalloc_status() == (0, 0)
    assert_close_layer(o, to_f64(ref), "noalloc accumulate")


def test_noalloc_rejects_shapes_beyond_its_scratch():
    """T = 512 at the full layer size needs far more than 2 MiB of workspace."""
    wl = S.WORKLOADS["prefill"]
    assert B.qmoe_workspace_size(wl.T, wl.H, wl.I, wl.E, wl.k) > (2 << 20)
    L = S.make_layer(wl.with_(T=512), seed=1, device=DEV)
    with pytest.raises(RuntimeError, match="unsupported"):
        B.qmoe_forward_noalloc(L)
