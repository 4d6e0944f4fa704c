"""GPU parity of the prefill path (tokens grouped by expert, grouped GEMM on
the tensor cores with on-chip dequantisation) against the fp64 oracle.

Every token of every case is compared, the full-size workloads included
(the oracle runs over the host's cores: each token's output depends only on
that token).  The prefill path's operands are exact (one fp16 weight
operand for bf16 block scales, hi + lo for fp16 scales; the SwiGLU output
as hi + lo), so it meets the decode path's bar: ids exact outside near
ties, output within 1e-2 * (1 + |ref|) elementwise."""
import numpy as np
import pytest
import torch

import oracle
from int4_block_quantized_gb300 import binding as B
from int4_block_quantized_gb300 import synthetic as S
from qmoe_check import assert_close_layer, check_routing, oracle_forward_parallel, tokens_covering_tile_columns

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from int4_block_quantized_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def check_prefill(wl, L=None, seed=0, sample=None, accumulate=False, path=B.PATH_PREFILL, cover=None):
    """cover = n: compare the tokens whose assignments sit at every column
    position of the GEMM's token tiles (from the GPU's routing) plus n more
    at random, instead of every token."""
    L = L or S.make_layer(wl, seed=seed, device=DEV)
    x = L["x"]
    T = x.shape[0]
    out = out0 = None
    if accumulate:
        out0 = torch.randn(x.shape, generator=torch.Generator(device=DEV).manual_seed(seed + 7),
                           device=DEV).to(x.dtype)
        out = out0.clone()
    ws = B.Workspace(T, wl.H, wl.I, wl.E, wl.k)
    o, tw, ti = B.qmoe_forward(L, out=out, ws=ws, accumulate=accumulate, path=path, return_routing=True)
    torch.cuda.synchronize()
    rc, bits = ws.status()
    assert rc == 0 and bits == 0
    if cover is not None:
        idx = np.asarray(tokens_covering_tile_columns(ti.cpu().numpy(), wl.E, cover, seed + 11))
    elif sample is None:
        idx = np.arange(T)
    else:
        idx = np.sort(np.random.default_rng(seed + 11).choice(T, size=min(sample, T), replace=False))
    tidx = torch.as_tensor(idx, device=DEV)
    Ls = dict(L, x=x[tidx].contiguous(), T=len(idx))
    ref, ref_ids, ref_w, probs = oracle_forward_parallel(Ls) if len(idx) > 64 else oracle.qmoe_forward(Ls)
    ids = ti[tidx].cpu().numpy()
    w = tw[tidx].cpu()
    near = check_routing(ids, w.numpy(), probs, ref_ids, wl.k)
    if near.any():
        ref2, _, _, _ = oracle.qmoe_forward(Ls, forced_ids=ids, forced_w=w.double().numpy())
        ref[near] = ref2[near]
    if accumulate:
        ref = ref + out0[tidx].double().cpu().numpy()
    return assert_close_layer(o[tidx], ref, wl.name + " (prefill)")


SMALL_CASES = [
    S.WORKLOADS["tiny"],
    S.Workload("pf_ragged", 37, 256, 128, 8, 2, 32, S.F16, S.F16, True, -5),
    S.Workload("pf_multi_tile", 300, 256, 128, 8, 2, 32, S.F16, S.F16, True, -5),
    S.Workload("pf_bf16_bs64", 100, 512, 384, 16, 4, 64, S.BF16, S.BF16, False, -6),
    S.Workload("pf_mixed_zp", 64, 512, 256, 16, 4, 32, S.BF16, S.F16, True, -5),
    S.Workload("pf_f16_bf16s", 48, 384, 192, 12, 3, 64, S.F16, S.BF16, False, -6),
    S.Workload("pf_bs128", 80, 1024, 640, 32, 4, 128, S.BF16, S.BF16, True, -6),
    S.Workload("pf_k8_e128", 40, 512, 256, 128, 8, 32, S.BF16, S.BF16, True, -5),
    S.Workload("pf_e256_k8", 33, 256, 128, 256, 8, 32, S.F16, S.BF16, False, -6),
    S.Workload("pf_k1", 130, 256, 128, 4, 1, 32, S.F16, S.F16, True, -5),
    # token tiles wider than 128 columns (up to 160): ~150 tokens per expert
    # (one tile of 160), and ~500 (four tiles of 125)
    S.Workload("pf_wide_tile", 300, 256, 128, 2, 1, 32, S.F16, S.F16, True, -5),
    S.Workload("pf_three_wide", 500, 512, 256, 2, 2, 64, S.BF16, S.F16, True, -5),
]


@pytest.mark.parametrize("wl", SMALL_CASES, ids=[w.name for w in SMALL_CASES])
def test_prefill_matches_oracle(wl):
    check_prefill(wl, seed=3)


def test_prefill_decode_shape_forced():
    """T = 16 at the full layer size through the grouped GEMM (every token)."""
    check_prefill(S.WORKLOADS["verify"], seed=5)


def test_prefill_full_size_every_token():
    """T = 512, bf16, block 128, no zero points, Zipf-skewed routing: all 512
    tokens (fp16 operands: one exact weight operand per bf16-scaled weight)."""
    check_prefill(S.WORKLOADS["prefill"], seed=1)


@pytest.mark.parametrize("name", ["e128_prefill", "e256_prefill"])
def test_larger_e_prefill_full_size_tile_columns(name):
    """Larger-E family shapes: 128 experts / I = 768 and 256 experts / I = 512,
    top-8, T = 512 through the grouped GEMM: tokens at every tile column
    position that occurs, plus 128 more."""
    check_prefill(S.WORKLOADS[name], seed=4, cover=128)


def test_stack_layer_full_size_tile_columns():
    """One layer of the T = 2048 stack shape (bf16 tokens, fp16 scales, zp):
    the tokens whose assignments sit at every column position of the 160-
    token tiles (all positions that occur), plus 256 more at random."""
    check_prefill(S.WORKLOADS["stack"], seed=2, cover=256)


def test_prefill_residual_accumulate():
    check_prefill(S.Workload("pf_res", 50, 256, 128, 8, 2, 32, S.BF16, S.BF16, True, -5), seed=4,
                  accumulate=True)


def test_prefill_one_expert_gets_every_token():
    """A large bias sends all 300 tokens to one expert first: that expert
    needs three token tiles, the rest are thin."""
    wl = S.Workload("pf_hot", 300, 256, 128, 8, 2, 32, S.F16, S.F16, True, -5)
    L = S.make_layer(wl, seed=6, device=DEV)
    bias = torch.zeros(wl.E, device=DEV)
    bias[5] = 30.0
    L["router_bias"] = bias
    check_prefill(wl, L=L)


def test_auto_path_above_decode_limit_is_prefill():
    """T = 17 takes the grouped GEMM under the automatic path choice."""
    check_prefill(S.Workload("pf_auto", 17, 256, 128, 8, 2, 32, S.F16, S.F16, True, -5), seed=8,
                  path=B.PATH_AUTO)


def test_prefill_repeat_calls_close():
    """fp32 atomics make the order of the k expert contributions vary, so
    repeated calls agree to rounding, not bit for bit."""
    wl = S.Workload("pf_rep", 64, 256, 128, 8, 2, 32, S.BF16, S.BF16, False, -6)
    L = S.make_layer(wl, seed=9, device=DEV)
    ws = B.Workspace(wl.T, wl.H, wl.I, wl.E, wl.k)
    a = B.qmoe_forward(L, ws=ws, path=B.PATH_PREFILL).float()
    for _ in range(3):
        b = B.qmoe_forward(L, ws=ws, path=B.PATH_PREFILL).float()
        assert torch.allclose(a, b, rtol=1e-2, atol=1e-2)


def test_prefill_rejects_unsupported_shape():
    """H not a multiple of 128: the grouped GEMM reports UNSUPPORTED and
    enqueues nothing."""
    wl = S.Workload("pf_bad", 20, 320, 96, 8, 2, 32, S.F16, S.F16, True, -5)
    L = S.make_layer(wl, seed=1, device=DEV)
    with pytest.raises(RuntimeError, match="unsupported"):
        B.qmoe_forward(L, path=B.PATH_PREFILL)


def test_withdrawn_path_value_is_rejected():
    """Path value 3 (a single-rounded-operand form that missed the
    elementwise tolerance) is not accepted any more."""
    wl = S.WORKLOADS["tiny"]
    L = S.make_layer(wl, seed=1, device=DEV)
    with pytest.raises(RuntimeError, match="invalid argument"):
        B.qmoe_forward(L, path=3)


def test_gemm_wait_timeout_is_reported_and_the_workspace_recovers():
    """Drive the grouped GEMM's bounded waits to expiry: the dequantisers
    wait for a copy that cannot arrive (a flag nothing sets) under a wait
    limit of 2^20 SM cycles (about 0.5 ms).  The wait gives up, every role
    drains what it has in flight, TMEM is freed and both GEMM kernels
    return; the status reads QMOE_ERR_TIMEOUT.  With the diagnostics cleared
    the same workspace computes the same output bit for bit."""
    wl = S.Workload("pf_timeout", 40, 256, 128, 8, 2, 32, S.F16, S.F16, True, -5)
    L = S.make_layer(wl, seed=3, device=DEV)
    ws = B.Workspace(wl.T, wl.H, wl.I, wl.E, wl.k)
    ref = B.qmoe_forward(L, ws=ws, path=B.PATH_PREFILL).clone()
    torch.cuda.synchronize()
    assert ws.status() == (0, 0)
    ws.set_diagnostics(1024, B.DIAG_STALL_GEMM)
    B.qmoe_forward(L, ws=ws, path=B.PATH_PREFILL)
    torch.cuda.synchronize()
    rc, bits = ws.status()
    assert rc == 5 and (bits & 1), (rc, bits)
    ws.set_diagnostics(0, 0)
    out = B.qmoe_forward(L, ws=ws, path=B.PATH_PREFILL)
    torch.cuda.synchronize()
    assert ws.status() == (0, 0)
    assert torch.equal(out, ref)


def test_bf16_beyond_fp16_range_sets_the_range_bit():
    """bf16 activations are converted to the fp16 operands exactly inside
    fp16's range; a value beyond it is reported (QMOE_ERR_DEVICE_CHECK)."""
    wl = S.Workload("pf_big", 40, 256, 128, 8, 2, 128, S.BF16, S.BF16, False, -6)
    L = S.make_layer(wl, seed=2, device=DEV)
    L["x"] = L["x"].clone()
    L["x"][3, 7] = 1.0e6
    ws = B.Workspace(wl.T, wl.H, wl.I, wl.E, wl.k)
    B.qmoe_forward(L, ws=ws, path=B.PATH_PREFILL)
    torch.cuda.synchronize()
    rc, bits = ws.status()
    assert rc == 6 and (bits & 4)
    assert ws.status() == (0, 0)  # read and cleared


def test_prefill_repeated_many_tiles_per_cta():
    """T = 16 at the full layer size gives each persistent CTA several
    weight tiles in a row, which exercises every ring wrap-around; repeated
    calls must all match the oracle (an ordering bug in the packed-code
    ring once corrupted a few rows of random tiles here)."""
    wl = S.WORKLOADS["verify"]
    L = S.make_layer(wl, seed=3, device=DEV)
    ws = B.Workspace(wl.T, wl.H, wl.I, wl.E, wl.k)
    o, tw, ti = B.qmoe_forward(L, ws=ws, path=B.PATH_PREFILL, return_routing=True)
    ids = ti.cpu().numpy()
    ref, ref_ids, _, probs = oracle.qmoe_forward(L)
    near = check_routing(ids, tw.cpu().numpy(), probs, ref_ids, wl.k)
    if near.any():
        ref2, _, _, _ = oracle.qmoe_forward(L, forced_ids=ids, forced_w=tw.cpu().double().numpy())
        ref[near] = ref2[near]
    for rep in range(4):
        o = B.qmoe_forward(L, ws=ws, path=B.PATH_PREFILL)
        torch.cuda.synchronize()
        assert_close_layer(o, ref, "verify prefill rep %d" % rep)
    rc, bits = ws.status()
    assert rc == 0 and bits == 0
