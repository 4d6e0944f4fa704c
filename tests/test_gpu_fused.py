"""The fused decode layer (router, gate-up and down in one cooperative
kernel, T <= 4; the default decode path at T = 1) against the three-kernel
decode path: the same arithmetic in the same order, so outputs and routing
must agree bit for bit.  Also the
grid barrier over many back-to-back calls (its counter resets itself), the
residual add, and the shapes that fall back to three kernels."""
import pytest
import torch

from int4_block_quantized_gb300 import binding as B
from int4_block_quantized_gb300 import synthetic as S

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from int4_block_quantized_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def _both(L, wl, accumulate=False, seed=0):
    x = L["x"]
    base = None
    if accumulate:
        base = torch.randn(x.shape, generator=torch.Generator(device=DEV).manual_seed(seed + 5),
                           device=DEV).to(x.dtype)
    res = []
    for path in (B.PATH_DECODE_FUSED, B.PATH_DECODE_SPLIT):
        ws = B.Workspace(x.shape[0], wl.H, wl.I, wl.E, wl.k)
        out = base.clone() if accumulate else None
        o, tw, ti = B.qmoe_forward(L, out=out, ws=ws, accumulate=accumulate, path=path, return_routing=True)
        torch.cuda.synchronize()
        assert ws.status() == (0, 0)
        res.append((o, tw, ti))
    return res


FUSED_CASES = [
    S.WORKLOADS["tiny"],
    S.WORKLOADS["decode"],
    S.WORKLOADS["decode"].with_(name="decode_t2", T=2),
    S.WORKLOADS["decode"].with_(name="decode_t3", T=3),
    S.WORKLOADS["decode"].with_(name="decode_t4", T=4),
    S.Workload("t3_bf16", 3, 512, 384, 16, 4, 64, S.BF16, S.BF16, False, -6),
    S.Workload("k1_e128", 1, 512, 256, 128, 1, 32, S.F16, S.F16, True, -5),
    S.Workload("k8_e128", 4, 512, 256, 128, 8, 32, S.BF16, S.BF16, True, -5),
    S.Workload("ragged", 3, 320, 96, 24, 3, 32, S.F16, S.F16, True, -5),
    S.WORKLOADS["e128_decode"],
    S.WORKLOADS["e256_decode"],
]


@pytest.mark.parametrize("wl", FUSED_CASES, ids=[w.name for w in FUSED_CASES])
def test_fused_equals_three_kernels(wl):
    L = S.make_layer(wl, seed=3, device=DEV)
    (o1, w1, i1), (o2, w2, i2) = _both(L, wl)
    assert torch.equal(i1, i2)
    assert torch.equal(w1, w2)
    assert torch.equal(o1, o2)


def test_fused_residual_equals_three_kernels():
    wl = S.WORKLOADS["decode"].with_(name="decode_t2", T=2)
    L = S.make_layer(wl, seed=4, device=DEV)
    (o1, _, _), (o2, _, _) = _both(L, wl, accumulate=True, seed=4)
    assert torch.equal(o1, o2)


def test_fused_repeated_calls_keep_the_barrier_consistent():
    wl = S.WORKLOADS["decode"]
    L = S.make_layer(wl, seed=7, device=DEV)
    ws = B.Workspace(1, wl.H, wl.I, wl.E, wl.k)
    ref = B.qmoe_forward(L, ws=ws, path=B.PATH_DECODE_SPLIT)
    out = torch.empty_like(ref)
    for _ in range(200):
        B.qmoe_forward(L, out=out, ws=ws, path=B.PATH_DECODE)
    torch.cuda.synchronize()
    assert ws.status() == (0, 0)
    assert torch.equal(out, ref)


def test_fused_in_a_cuda_graph():
    wl = S.WORKLOADS["decode"]
    L = S.make_layer(wl, seed=8, device=DEV)
    ws = B.Workspace(1, wl.H, wl.I, wl.E, wl.k)
    ref = B.qmoe_forward(L, ws=ws, path=B.PATH_DECODE_SPLIT)
    out = torch.empty_like(ref)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        B.qmoe_forward(L, out=out, ws=ws, path=B.PATH_DECODE)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        B.qmoe_forward(L, out=out, ws=ws, path=B.PATH_DECODE)
    out.zero_()
    for _ in range(5):
        g.replay()
    torch.cuda.synchronize()
    assert ws.status() == (0, 0)
    assert torch.equal(out, ref)


def test_mixed_zero_points_fall_back_and_agree():
    """Gate/up with zero points and down without: no fused plan.  The forced
    fused path refuses; DECODE runs three kernels, equal to DECODE_SPLIT."""
    wl = S.WORKLOADS["decode"]
    L = dict(S.make_layer(wl, seed=9, device=DEV))
    L["down_zp"] = None
    with pytest.raises(B.QMoEError):
        B.qmoe_forward(L, path=B.PATH_DECODE_FUSED)
    outs = []
    for path in (B.PATH_DECODE, B.PATH_DECODE_SPLIT):
        o, _, i = B.qmoe_forward(L, path=path, return_routing=True)
        outs.append((o, i))
    torch.cuda.synchronize()
    assert torch.equal(outs[0][1], outs[1][1]) and torch.equal(outs[0][0], outs[1][0])
    assert B.qmoe_forward_kernels(L, 1) == 3


def test_kernel_count_query():
    L = S.make_layer(S.WORKLOADS["decode"], seed=10, device=DEV)
    assert B.qmoe_forward_kernels(L, 1) == 1
    assert B.qmoe_forward_kernels(L, 2) == 3
    for T in (1, 2, 3, 4):
        assert B.qmoe_forward_kernels(L, T, path=B.PATH_DECODE_FUSED) == 1
    assert B.qmoe_forward_kernels(L, 1, path=B.PATH_DECODE_SPLIT) == 3
    assert B.qmoe_forward_kernels(L, 16) == 3
    assert B.qmoe_forward_kernels(L, 512) == 5
