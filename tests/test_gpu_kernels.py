"""GPU parity of the individual entry points against the fp64 oracle:
DequantizeLinear (bit-exact), the router (ids exact outside near ties,
grouping bit-exact), MatMulNBits and RMSNorm (within tolerance).  Every call
goes through the C ABI."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from int4_block_quantized_gb300 import binding as B
from int4_block_quantized_gb300 import synthetic as S
from qmoe_check import assert_close_layer, check_routing

pytestmark = pytest.mark.gpu
DEV = "cuda"
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from int4_block_quantized_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def _gen(seed):
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    return g


def _qmat(N, K, bs, sdt, zp, seed):
    g = _gen(seed)
    w = torch.randint(0, 256, (N, K // 2), generator=g, device=DEV, dtype=torch.uint8)
    s = ((torch.rand((N, K // bs), generator=g, device=DEV) + 0.5) / 32).to(
        torch.bfloat16 if sdt == S.BF16 else torch.float16)
    z = torch.randint(0, 16, (N, K // bs), generator=g, device=DEV, dtype=torch.uint8) if zp else None
    return w, s, z


# ------------------------------------------------------------------ dequant

@pytest.mark.parametrize("bs", [32, 64, 128])
@pytest.mark.parametrize("sdt", [S.F16, S.BF16])
@pytest.mark.parametrize("zp", [True, False])
def test_dequant_bit_exact(bs, sdt, zp):
    N, K = 96, 1408 if bs != 128 else 1280
    w, s, z = _qmat(N, K, bs, sdt, zp, 100 + bs + sdt)
    got = B.qmoe_dequant(w, s, z, bs).cpu().double().numpy()
    ref = oracle.dequant(w, s, sdt, z, N, K, bs)
    assert np.array_equal(got, ref)


def test_dequant_hand_example():
    g = json.load(open(os.path.join(GOLDEN, "dequant_two_blocks.json")))
    w = torch.tensor([list(bytes.fromhex(h)) for h in g["packed_hex"]], dtype=torch.uint8, device=DEV)
    s = torch.tensor(g["scales"], dtype=torch.float16, device=DEV)
    z = torch.tensor(g["zero_points"], dtype=torch.uint8, device=DEV)
    d = B.qmoe_dequant(w, s, z, g["block_size"]).cpu().double()
    assert d.sum(dim=1).tolist() == g["row_sums"]
    for n, k, v in g["elements"]:
        assert d[n, k].item() == v
    x = torch.tensor([[(-1) ** k * (1 + k % 4) for k in range(g["K"])]], dtype=torch.float16, device=DEV)
    y = B.matmul_nbits(x, w, s, z, g["block_size"])
    assert y.double().cpu()[0].tolist() == g["y_for_x_alternating"]


# ------------------------------------------------------------------- router

ROUTE_CASES = [
    # name, T, H, E, k, act dtype, zipf
    ("tiny", 4, 256, 8, 2, S.F16, 0.0),
    ("decode", 1, 2048, 60, 4, S.F16, 0.0),
    ("verify", 16, 2048, 60, 4, S.F16, 0.0),
    ("prefill", 512, 2048, 60, 4, S.BF16, 1.1),
    ("ragged", 37, 320, 60, 4, S.BF16, 0.0),
    ("k1", 33, 512, 128, 1, S.F16, 0.0),
    ("k8", 17, 512, 128, 8, S.BF16, 0.0),
    ("e256", 5, 256, 256, 8, S.F16, 0.0),
    ("e1", 3, 64, 1, 1, S.F16, 0.0),
    ("stack", 2048, 2048, 60, 4, S.BF16, 0.0),
    # T > 16 takes the tensor-core router: ragged last tile, E not a
    # multiple of 16, H whose 64-wide chunks do not divide over 8 CTAs
    ("tc_tail", 300, 256, 16, 2, S.F16, 0.0),
    ("tc_e100", 129, 1024, 100, 6, S.BF16, 0.0),
    ("tc_h192", 64, 192, 24, 3, S.F16, 0.0),
]


@pytest.mark.parametrize("case", ROUTE_CASES, ids=[c[0] for c in ROUTE_CASES])
def test_route_matches_oracle(case):
    name, T, H, E, k, dt, zipf = case
    wl = S.Workload(name, T, H, 128, E, k, 32, dt, dt, True, -5, zipf_s=zipf)
    x = S.make_x(wl, seed=3, device=DEV)
    d = S.make_weights(wl, seed=3, device=DEV)
    tw, ti, off, perm = B.qmoe_route(x, d["router_w"], k, d["router_bias"])
    torch.cuda.synchronize()
    probs = oracle.router_probs(x, dt, d["router_w"], d["router_bias"], T, H, E)
    ref_ids, _ = oracle.topk(probs, k)
    ids = ti.cpu().numpy()
    near = check_routing(ids, tw.cpu().numpy(), probs, ref_ids, k)
    print("%s: %d near-tie token(s) of %d" % (name, int(near.sum()), T))
    # grouping is deterministic: bit-exact against the oracle's on the GPU's ids
    ro, rp = oracle.group_by_expert(ids, E)
    assert np.array_equal(off.cpu().numpy(), ro)
    assert np.array_equal(perm.cpu().numpy(), rp)


def test_route_ties_lower_id_first():
    """Identical router columns make exact ties; the lower expert id wins."""
    T, H, E, k = 8, 64, 16, 4
    g = _gen(7)
    x = torch.randn((T, H), generator=g, device=DEV).half()
    col = torch.randn((H, 1), generator=g, device=DEV) * 0.1
    rw = col.repeat(1, E).half()  # all logits equal
    tw, ti, off, perm = B.qmoe_route(x, rw, k)
    assert ti.cpu().tolist() == [[0, 1, 2, 3]] * T
    assert torch.allclose(tw.cpu(), torch.full((T, k), 1.0 / E))


def test_route_ties_lower_id_first_many_tokens():
    """The same on the tensor-core router (T > 16): identical columns give
    bit-identical logits, and the lower expert id wins."""
    T, H, E, k = 40, 256, 16, 4
    g = _gen(8)
    x = torch.randn((T, H), generator=g, device=DEV).half()
    col = torch.randn((H, 1), generator=g, device=DEV) * 0.1
    rw = col.repeat(1, E).half()
    tw, ti, off, perm = B.qmoe_route(x, rw, k)
    assert ti.cpu().tolist() == [[0, 1, 2, 3]] * T
    assert torch.allclose(tw.cpu(), torch.full((T, k), 1.0 / E))


def test_route_is_deterministic():
    wl = S.WORKLOADS["prefill"]
    x = S.make_x(wl, seed=5, device=DEV)
    d = S.make_weights(wl, seed=5, device=DEV)
    first = [t.clone() for t in B.qmoe_route(x, d["router_w"], wl.k, d["router_bias"])]
    for _ in range(5):
        again = B.qmoe_route(x, d["router_w"], wl.k, d["router_bias"])
        for a, b in zip(first, again):
            assert torch.equal(a, b)


# -------------------------------------------------------------- matmul_nbits

MM_CASES = [
    # M, N, K, bs, act, scale, zp
    (1, 1408, 2048, 32, S.F16, S.F16, True),
    (3, 2048, 1408, 32, S.F16, S.F16, True),
    (16, 256, 2048, 128, S.BF16, S.BF16, False),
    (17, 320, 512, 64, S.BF16, S.F16, True),
    (5, 1, 64, 32, S.F16, S.BF16, False),
    (40, 96, 4096, 128, S.F16, S.F16, True),
]


@pytest.mark.parametrize("case", MM_CASES, ids=[str(c[:4]) for c in MM_CASES])
def test_matmul_nbits_matches_oracle(case):
    M, N, K, bs, adt, sdt, zp = case
    w, s, z = _qmat(N, K, bs, sdt, zp, 11 + M)
    x = torch.randn((M, K), generator=_gen(12), device=DEV).to(torch.bfloat16 if adt else torch.float16)
    y = B.matmul_nbits(x, w, s, z, bs)
    ref = oracle.matmul_nbits(x, adt, w, s, sdt, z, M, N, K, bs)
    assert_close_layer(y, ref, "matmul_nbits")
    # fp32 accumulation: within one rounding of the output type plus a small sum error
    ulp = 2.0 ** -8 if adt == S.BF16 else 2.0 ** -11
    err = np.abs(y.double().cpu().numpy() - ref)
    assert (err <= ulp * np.abs(ref) + 1e-3 * (1 + np.abs(ref))).all()


# ------------------------------------------------------------------ RMSNorm

@pytest.mark.parametrize("dt", [S.F16, S.BF16])
def test_rmsnorm_matches_oracle(dt):
    T, H = 33, 2048
    x = (torch.randn((T, H), generator=_gen(13), device=DEV) * 3).to(torch.bfloat16 if dt else torch.float16)
    y = B.qmoe_rmsnorm(x, 1e-6)
    ref = oracle.rmsnorm(x, dt, T, H, 1e-6)
    got = y.double().cpu().numpy()
    ulp = 2.0 ** -8 if dt == S.BF16 else 2.0 ** -11
    assert (np.abs(got - ref) <= ulp * np.abs(ref) + 1e-6).all()
