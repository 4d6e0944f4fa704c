"""The fused decode layer (router, gate-up and down in one launch; the
default decode path at T = 1) against the fp64 oracle and against the
three-kernel decode path.  Both paths compute the routing with the same fp32
arithmetic in the same order, so ids and weights agree bit for bit; the
fused layer splits the down projection along I and sums the partial outputs
in a fixed order, so its output is compared with the oracle elementwise and
must be bit-identical from call to call.  Also the per-slice completion
counters over many back-to-back calls and graph replays, the residual add,
and the shapes that fall back to three kernels."""
import pytest
import torch

from int4_block_quantized_gb300 import binding as B
from int4_block_quantized_gb300 import synthetic as S
from qmoe_check import assert_close_layer, run_layer_and_check, to_f64

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from int4_block_quantized_gb300 import build
    build.build()
    assert torch.cuda.is_available()


FUSED_CASES = [
    S.WORKLOADS["tiny"],
    S.WORKLOADS["decode"],
    S.WORKLOADS["decode"].with_(name="decode_bf16_bs128", act_dtype=S.BF16, scale_dtype=S.BF16, block_size=128,
                                has_zp=False, scale_exp=-6),
    S.Workload("t3_bf16", 3, 512, 384, 16, 4, 64, S.BF16, S.BF16, False, -6),
    S.Workload("k1_e128", 1, 512, 256, 128, 1, 32, S.F16, S.F16, True, -5),
    S.Workload("k8_e128", 4, 512, 256, 128, 8, 32, S.BF16, S.BF16, True, -5),
    S.Workload("ragged", 3, 320, 96, 24, 3, 32, S.F16, S.F16, True, -5),
    S.Workload("t1_h256", 1, 256, 128, 8, 2, 32, S.F16, S.BF16, True, -5),
    S.WORKLOADS["e128_decode"],
    S.WORKLOADS["e256_decode"],
]


@pytest.mark.parametrize("wl", FUSED_CASES, ids=[w.name for w in FUSED_CASES])
def test_fused_matches_oracle_and_routes_like_three_kernels(wl):
    L = S.make_layer(wl, seed=3, device=DEV)
    assert B.qmoe_forward_kernels(L, wl.T, path=B.PATH_DECODE_FUSED) == 1
    o1, w1, i1, _, _ = run_layer_and_check(wl, L, B.PATH_DECODE_FUSED)
    o2, w2, i2, _, _ = run_layer_and_check(wl, L, B.PATH_DECODE_SPLIT)
    assert torch.equal(i1, i2)
    assert torch.equal(w1, w2)
    assert_close_layer(o1, to_f64(o2), wl.name + " fused vs three kernels")


@pytest.mark.parametrize("name", ["tiny", "decode"])
def test_fused_residual_accumulate(name):
    wl = S.WORKLOADS[name]
    L = S.make_layer(wl, seed=4, device=DEV)
    run_layer_and_check(wl, L, B.PATH_DECODE_FUSED, accumulate=True, seed=4)


def test_fused_repeated_calls_bit_identical():
    """Fixed summation order: every call gives the same bits, and the
    per-slice counters are back at zero after each call."""
    wl = S.WORKLOADS["decode"]
    L = S.make_layer(wl, seed=7, device=DEV)
    ws = B.Workspace(1, wl.H, wl.I, wl.E, wl.k)
    ref = B.qmoe_forward(L, ws=ws, path=B.PATH_DECODE).clone()
    outs = [torch.empty_like(ref) for _ in range(4)]
    for i in range(200):
        B.qmoe_forward(L, out=outs[i % 4], ws=ws, path=B.PATH_DECODE)
    torch.cuda.synchronize()
    assert ws.status() == (0, 0)
    for o in outs:
        assert torch.equal(o, ref)
    ctl = ws.buf[:64].cpu().view(torch.int32)
    assert torch.equal(ctl[8:12], torch.zeros(4, dtype=torch.int32))
    # the fixed-point output accumulator after the control words is clear again
    assert int(ws.buf[1024:1024 + 8 * wl.H].count_nonzero()) == 0


def test_fused_workspace_shared_with_other_paths():
    """One workspace alternating between the fused layer, the three-kernel
    path and the prefill path keeps giving the fused layer's exact result."""
    wl = S.WORKLOADS["decode"]
    L = S.make_layer(wl, seed=12, device=DEV)
    ws = B.Workspace(64, wl.H, wl.I, wl.E, wl.k)
    ref = B.qmoe_forward(L, ws=ws, path=B.PATH_DECODE_FUSED).clone()
    L64 = S.make_layer(wl.with_(T=64), seed=13, device=DEV)
    for _ in range(3):
        B.qmoe_forward(L, ws=ws, path=B.PATH_DECODE_SPLIT)
        B.qmoe_forward(L64, ws=ws)
        assert torch.equal(B.qmoe_forward(L, ws=ws, path=B.PATH_DECODE_FUSED), ref)
    torch.cuda.synchronize()
    assert ws.status() == (0, 0)


def test_fused_in_a_cuda_graph():
    wl = S.WORKLOADS["decode"]
    L = S.make_layer(wl, seed=8, device=DEV)
    ws = B.Workspace(1, wl.H, wl.I, wl.E, wl.k)
    ref = B.qmoe_forward(L, ws=ws, path=B.PATH_DECODE).clone()
    out = torch.empty_like(ref)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        B.qmoe_forward(L, out=out, ws=ws, path=B.PATH_DECODE)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(3):
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
    assert B.qmoe_forward_kernels(L, 1, path=B.PATH_DECODE_FUSED) == 1
    assert B.qmoe_forward_kernels(L, 2) == 3
    # at the full layer shape a CTA's share of T >= 2 tokens' experts no
    # longer fits in shared memory: three kernels only
    for T in (2, 3, 4):
        with pytest.raises(B.QMoEError, match="unsupported"):
            B.qmoe_forward_kernels(L, T, path=B.PATH_DECODE_FUSED)
    assert B.qmoe_forward_kernels(L, 1, path=B.PATH_DECODE_SPLIT) == 3
    assert B.qmoe_forward_kernels(L, 5) == 3
    assert B.qmoe_forward_kernels(L, 16) == 5  # AUTO: the grouped GEMM beyond 5 tokens
    assert B.qmoe_forward_kernels(L, 16, path=B.PATH_DECODE) == 3
    assert B.qmoe_forward_kernels(L, 512) == 5
    Lt = S.make_layer(S.WORKLOADS["tiny"], seed=10, device=DEV)
    assert B.qmoe_forward_kernels(Lt, 4, path=B.PATH_DECODE_FUSED) == 1
