"""GPU parity of the weight-format adapters (C ABI) against oracle/formats.py:
bit-exact canonical bytes from GPTQ tensors and from packed zero points,
the device zero-offset rule, and a whole layer run from GPTQ-converted
weights against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from oracle import formats as F
from int4_block_quantized_gb300 import binding as B
from int4_block_quantized_gb300 import synthetic as S
from qmoe_check import assert_close_layer

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from int4_block_quantized_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def _gptq(E, K, N, bs, seed, zero_mask=0x77777777, stored_zero=None, scale_dtype=torch.float16):
    g = torch.Generator().manual_seed(seed)
    qweight = torch.randint(-2 ** 31, 2 ** 31 - 1, (E, K // 8, N), generator=g, dtype=torch.int64).to(torch.int32)
    if stored_zero is None:
        qzeros = torch.randint(-2 ** 31, 2 ** 31 - 1, (E, K // bs, N // 8), generator=g, dtype=torch.int64)
        qzeros = (qzeros & zero_mask).to(torch.int32)
    else:
        qzeros = torch.full((E, K // bs, N // 8), stored_zero * 0x11111111, dtype=torch.int64).to(torch.int32)
    scales = ((torch.rand((E, K // bs, N), generator=g) + 0.5) * 2 ** -5).to(scale_dtype)
    return qweight, qzeros, scales


def _np_u32(t):
    return t.numpy().view(np.uint32)


@pytest.mark.parametrize("E,K,N,bs,offset", [(2, 256, 64, 32, 1), (1, 512, 40, 128, 0), (3, 128, 24, 64, 1)])
def test_repack_gptq_bit_exact(E, K, N, bs, offset):
    qw, qz, sc = _gptq(E, K, N, bs, seed=E * 100 + K)
    w, s, zp = B.qmoe_repack_gptq(qw.to(DEV), qz.to(DEV), sc.to(DEV), bs, zero_offset=offset)
    torch.cuda.synchronize()
    for e in range(E):
        rw, rs, rz = F.gptq_to_canonical(_np_u32(qw[e]), _np_u32(qz[e]), sc[e].view(torch.int16).numpy(), K, N,
                                         bs, offset)
        assert np.array_equal(w[e].cpu().numpy(), rw)
        assert np.array_equal(s[e].view(torch.int16).cpu().numpy(), rs)
        assert np.array_equal(zp[e].cpu().numpy(), rz)


def test_repack_gptq_without_zeros_and_bf16_scales():
    E, K, N, bs = 2, 256, 32, 128
    qw, _, sc = _gptq(E, K, N, bs, seed=11, scale_dtype=torch.bfloat16)
    w, s, zp = B.qmoe_repack_gptq(qw.to(DEV), None, sc.to(DEV), bs)
    torch.cuda.synchronize()
    assert zp is None
    for e in range(E):
        rw, rs, _ = F.gptq_to_canonical(_np_u32(qw[e]), None, sc[e].view(torch.int16).numpy(), K, N, bs, 0)
        assert np.array_equal(w[e].cpu().numpy(), rw)
        assert np.array_equal(s[e].view(torch.int16).cpu().numpy(), rs)


def test_repack_gptq_full_layer_shape_sampled():
    """A Qwen1.5-MoE-A2.7B gate projection (E = 60, K = H = 2048, N = I = 1408,
    bs = 32): every weight word is a transposed input word; zero points and
    scales checked on sampled (e, n, g) against the oracle's definitions."""
    E, K, N, bs = 60, 2048, 1408, 32
    qw, qz, sc = _gptq(E, K, N, bs, seed=5)
    w, s, zp = B.qmoe_repack_gptq(qw.to(DEV), qz.to(DEV), sc.to(DEV), bs, zero_offset=1)
    torch.cuda.synchronize()
    # canonical byte 4i + b of row n is byte b of word (i, n): the word transpose
    assert torch.equal(w.view(torch.int32).cpu(), qw.transpose(1, 2).contiguous())
    assert torch.equal(s.cpu(), sc.transpose(1, 2).contiguous())
    rng = np.random.default_rng(0)
    zc = zp.cpu().numpy()
    for _ in range(2000):
        e, n, g = int(rng.integers(E)), int(rng.integers(N)), int(rng.integers(K // bs))
        assert zc[e, n, g] == min(F.gptq_stored_zero(_np_u32(qz[e]), g, n) + 1, 15)
    # and sampled weight nibbles against the GPTQ definition
    wc = w.cpu().numpy()
    for _ in range(2000):
        e, n, k = int(rng.integers(E)), int(rng.integers(N)), int(rng.integers(K))
        assert (int(wc[e, n, k // 2]) >> (4 * (k % 2))) & 15 == F.gptq_nibble(_np_u32(qw[e]), k, n)


def test_zero_point_16_is_reported():
    """A stored zero of 15 with offset 1 is 16, outside the 4-bit zero point:
    the converter writes 15 (like the oracle) and sets the range bit; the
    binding's default check raises.  Offset 0 converts the same words
    silently."""
    E, K, N, bs = 1, 128, 16, 32
    qw, qz, sc = _gptq(E, K, N, bs, seed=9, stored_zero=15)
    with pytest.raises(B.QMoEError, match="above 15"):
        B.qmoe_repack_gptq(qw.to(DEV), qz.to(DEV), sc.to(DEV), bs, zero_offset=1)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    _, _, zp = B.qmoe_repack_gptq(qw.to(DEV), qz.to(DEV), sc.to(DEV), bs, zero_offset=1, check=False, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 4
    assert not F.gptq_zero_points_fit(_np_u32(qz[0]), K, N, bs, 1)
    _, _, rz = F.gptq_to_canonical(_np_u32(qw[0]), _np_u32(qz[0]), sc[0].view(torch.int16).numpy(), K, N, bs, 1)
    assert np.array_equal(zp[0].cpu().numpy(), rz)
    _, _, zp0 = B.qmoe_repack_gptq(qw.to(DEV), qz.to(DEV), sc.to(DEV), bs, zero_offset=0)
    assert (zp0 == 15).all() and F.gptq_zero_points_fit(_np_u32(qz[0]), K, N, bs, 0)


@pytest.mark.parametrize("stored,expect", [(7, 1), (8, 0)])
def test_device_zero_offset_rule(stored, expect):
    _, qz, _ = _gptq(4, 256, 64, 32, seed=stored, stored_zero=stored)
    off = B.qmoe_gptq_zero_offset(qz.to(DEV))
    torch.cuda.synchronize()
    assert int(off.item()) == expect == F.gptq_zero_offset(_np_u32(qz))


def test_device_zero_offset_random_matches_oracle():
    for seed in range(4):
        _, qz, _ = _gptq(2, 256, 64, 32, seed=40 + seed, zero_mask=0x77777777 if seed % 2 == 0 else 0xFFFFFFFF)
        off = B.qmoe_gptq_zero_offset(qz.to(DEV))
        torch.cuda.synchronize()
        assert int(off.item()) == F.gptq_zero_offset(_np_u32(qz))


def test_repack_reads_the_device_offset():
    E, K, N, bs = 2, 256, 64, 32
    qw, qz, sc = _gptq(E, K, N, bs, seed=3, stored_zero=7)
    qzd = qz.to(DEV)
    off = B.qmoe_gptq_zero_offset(qzd)
    _, _, zp = B.qmoe_repack_gptq(qw.to(DEV), qzd, sc.to(DEV), bs, zero_offset=0, zero_offset_dev=off)
    torch.cuda.synchronize()
    assert (zp == 8).all()


@pytest.mark.parametrize("rows,nb", [(7, 5), (1408, 64), (256, 11)])
def test_unpack_zero_points_bit_exact(rows, nb):
    g = torch.Generator().manual_seed(rows + nb)
    packed = torch.randint(0, 256, (rows, (nb + 1) // 2), generator=g, dtype=torch.int32).to(torch.uint8)
    out = B.qmoe_unpack_zero_points(packed.to(DEV), nb)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), F.unpack_zero_points(packed.numpy(), rows, nb))


def test_layer_from_gptq_weights_matches_oracle():
    """A tiny-workload layer whose three projections arrive as GPTQ tensors
    (zero-point offset detected on the device), converted, then run."""
    wl = S.WORKLOADS["tiny"]
    L = dict(S.make_layer(wl, seed=12, device=DEV))
    E, H, I, bs = wl.E, wl.H, wl.I, wl.block_size
    for name, (K, N), seed in (("gate", (H, I), 21), ("up", (H, I), 22), ("down", (I, H), 23)):
        qw, qz, sc = _gptq(E, K, N, bs, seed=seed)
        qzd = qz.to(DEV)
        off = B.qmoe_gptq_zero_offset(qzd)
        w, s, zp = B.qmoe_repack_gptq(qw.to(DEV), qzd, sc.to(DEV), bs, zero_offset_dev=off)
        L[name + "_w"], L[name + "_s"], L[name + "_zp"] = w, s, zp
    out = B.qmoe_forward(L)
    torch.cuda.synchronize()
    ref, _, _, _ = oracle.qmoe_forward(L)
    assert_close_layer(out, ref, "gptq layer")
