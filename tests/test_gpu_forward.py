"""GPU parity of the whole layer (qmoe_forward, C ABI) against the fp64
oracle on seeded synthetic inputs: routing ids exact outside near ties,
output within 1e-2 * (1 + |ref|) elementwise."""
import numpy as np
import pytest
import torch

import oracle
from int4_block_quantized_gb300 import binding as B
from int4_block_quantized_gb300 import synthetic as S
from qmoe_check import assert_close_layer, check_routing

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from int4_block_quantized_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def run_and_check(wl, seed=0, path=B.PATH_AUTO, layer=None, accumulate=False, x=None):
    L = layer or S.make_layer(wl, seed=seed, device=DEV)
    if x is not None:
        L = dict(L, x=x, T=x.shape[0])
    x = L["x"]
    out0 = None
    if accumulate:
        out0 = torch.randn(x.shape, generator=torch.Generator(device=DEV).manual_seed(seed + 7),
                           device=DEV).to(x.dtype)
        out = out0.clone()
    else:
        out = None
    ws = B.Workspace(x.shape[0], wl.H, wl.I, wl.E, wl.k)
    o, tw, ti = B.qmoe_forward(L, out=out, ws=ws, accumulate=accumulate, path=path, return_routing=True)
    torch.cuda.synchronize()
    rc, bits = ws.status()
    assert rc == 0 and bits == 0
    ref, ref_ids, ref_w, probs = oracle.qmoe_forward(L)
    ids = ti.cpu().numpy()
    near = check_routing(ids, tw.cpu().numpy(), probs, ref_ids, wl.k)
    if near.any():
        # re-run the oracle on the GPU's routing for the near-tie tokens
        ref2, _, _, _ = oracle.qmoe_forward(L, forced_ids=ids, forced_w=tw.cpu().double().numpy())
        ref[near] = ref2[near]
    if accumulate:
        ref = ref + out0.double().cpu().numpy()
    return assert_close_layer(o, ref, wl.name), int(near.sum())


DECODE_CASES = [
    S.WORKLOADS["tiny"],
    S.WORKLOADS["decode"],
    S.WORKLOADS["verify"],
    S.Workload("t2_e16", 2, 512, 384, 16, 4, 32, S.F16, S.F16, True, -5),
    S.Workload("t3_bf16", 3, 512, 384, 16, 4, 64, S.BF16, S.BF16, False, -6),
    S.Workload("t5_bs128", 5, 1024, 640, 32, 4, 128, S.BF16, S.F16, True, -5),
    S.Workload("k1_e128", 7, 512, 256, 128, 1, 32, S.F16, S.F16, True, -5),
    S.Workload("k8_e128", 9, 512, 256, 128, 8, 32, S.BF16, S.BF16, True, -5),
    S.Workload("e256_k8", 16, 256, 128, 256, 8, 32, S.F16, S.BF16, False, -6),
    S.Workload("ragged", 11, 320, 96, 24, 3, 32, S.F16, S.F16, True, -5),
    S.Workload("zipf", 16, 2048, 1408, 60, 4, 128, S.BF16, S.BF16, False, -6, zipf_s=1.1),
    S.WORKLOADS["e128_decode"],
    S.WORKLOADS["e256_decode"],
    S.WORKLOADS["e128_decode"].with_(name="e128_t8", T=8),
]


@pytest.mark.parametrize("wl", DECODE_CASES, ids=[w.name for w in DECODE_CASES])
def test_forward_decode_matches_oracle(wl):
    run_and_check(wl, seed=1, path=B.PATH_DECODE)


@pytest.mark.parametrize("T,expect", [(1, B.PATH_DECODE), (5, B.PATH_DECODE), (6, B.PATH_PREFILL),
                                      (16, B.PATH_PREFILL)])
def test_auto_path_choice(T, expect):
    """AUTO takes the decode path up to AUTO_DECODE_MAX_TOKENS tokens and the
    grouped GEMM beyond: AUTO and the forced path both match the oracle, and
    the kernel count says which path AUTO runs."""
    base = S.WORKLOADS["verify"]
    wl = S.Workload("auto%d" % T, T, base.H, base.I, base.E, base.k, base.block_size, base.act_dtype,
                    base.scale_dtype, base.has_zp, base.scale_exp)
    L = S.make_layer(wl, seed=11, device=DEV)
    auto, _ = run_and_check(wl, layer=L, path=B.PATH_AUTO)
    forced, _ = run_and_check(wl, layer=L, path=expect)
    n = B.qmoe_forward_kernels(L, T)
    assert n == (5 if expect == B.PATH_PREFILL else (1 if T == 1 else 3))


def test_forward_decode_residual_accumulate():
    run_and_check(S.WORKLOADS["tiny"], seed=2, accumulate=True, path=B.PATH_DECODE)
    run_and_check(S.WORKLOADS["verify"], seed=2, accumulate=True, path=B.PATH_DECODE)


def test_forward_all_tokens_one_expert():
    """A large bias on one expert sends every token there first: one expert
    with 16 tokens (four token groups) plus the rest spread thinly."""
    wl = S.WORKLOADS["verify"]
    L = S.make_layer(wl, seed=4, device=DEV)
    bias = torch.zeros(wl.E, device=DEV)
    bias[17] = 30.0
    L["router_bias"] = bias
    run_and_check(wl, layer=L, path=B.PATH_DECODE)
    run_and_check(wl, layer=L, path=B.PATH_PREFILL)


def test_forward_identical_experts_closed_form():
    """All experts share weights: out = (sum of routing weights) * FFN(x),
    with FFN from the single-expert oracle (E = k = 1)."""
    wl = S.Workload("same", 6, 512, 256, 8, 2, 32, S.F16, S.F16, True, -5)
    L = S.make_layer(wl, seed=9, device=DEV)
    for p in ("gate", "up", "down"):
        for t in ("_w", "_s", "_zp"):
            L[p + t] = L[p + t][:1].repeat(wl.E, *([1] * (L[p + t].dim() - 1))).contiguous()
    o, tw, ti = B.qmoe_forward(L, return_routing=True)
    L1 = dict(L, E=1, k=1, router_w=L["router_w"][:, :1].contiguous(), router_bias=None)
    for p in ("gate", "up", "down"):
        for t in ("_w", "_s", "_zp"):
            L1[p + t] = L[p + t][:1].contiguous()
    ffn, _, _, _ = oracle.qmoe_forward(L1)
    ref = ffn * tw.double().sum(dim=1, keepdim=True).cpu().numpy()
    assert_close_layer(o, ref, "identical experts")


def test_forward_repeat_calls_identical():
    wl = S.WORKLOADS["verify"]
    L = S.make_layer(wl, seed=6, device=DEV)
    ws = B.Workspace(wl.T, wl.H, wl.I, wl.E, wl.k)
    a = B.qmoe_forward(L, ws=ws, path=B.PATH_DECODE).clone()
    for _ in range(3):
        assert torch.equal(B.qmoe_forward(L, ws=ws, path=B.PATH_DECODE), a)


def test_forward_decode_full_size_workspace_reuse_across_shapes():
    """One workspace sized for T=16 serves T=1 calls too (smaller needs)."""
    wl = S.WORKLOADS["decode"]
    L = S.make_layer(wl, seed=8, device=DEV)
    ws = B.Workspace(16, wl.H, wl.I, wl.E, wl.k)
    ref, _, _, _ = oracle.qmoe_forward(L)
    o = B.qmoe_forward(L, ws=ws)
    assert_close_layer(o, ref, "decode, large workspace")
