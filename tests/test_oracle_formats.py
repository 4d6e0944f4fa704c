"""Pins of the weight-format oracle (oracle/formats.py), CPU only.

Hand-derived byte images (the hex literals below were worked out by hand
from the format definitions, not produced by the oracle), the pages'
zero-point offset rule ("Qwen MoE BringUp", "Bugs/Issues Found", item 1),
and a cross-check of the GPTQ dequantisation against the independent C
oracle's DequantizeLinear on the converted weights."""
import numpy as np
import pytest

import oracle
from oracle import formats as F

# K = 32 (one block of 32), N = 8.  Column n holds q[k, n] = (k + n) mod 16
# for n = 0 and 1; the other columns are zero.  GPTQ words, column 0:
# k = 0..7 -> 0x76543210, k = 8..15 -> 0xFEDCBA98, then the same again.
# Column 1: k = 0..7 -> q = 1..8 -> 0x87654321, k = 8..15 -> q = 9..15, 0 ->
# 0x0FEDCBA9, then the same again.
QWEIGHT_HAND = np.zeros((4, 8), dtype=np.uint32)
QWEIGHT_HAND[:, 0] = [0x76543210, 0xFEDCBA98, 0x76543210, 0xFEDCBA98]
QWEIGHT_HAND[:, 1] = [0x87654321, 0x0FEDCBA9, 0x87654321, 0x0FEDCBA9]
# canonical row 0: pairs (0,1) (2,3) ... -> 10 32 54 76 98 ba dc fe, twice
W_ROW0_HAND = bytes.fromhex("1032547698badcfe" * 2)
# canonical row 1: (1,2) (3,4) ... (15,0) -> 21 43 65 87 a9 cb ed 0f, twice
W_ROW1_HAND = bytes.fromhex("21436587a9cbed0f" * 2)
# stored zeros of columns 0..7 = 7 7 3 0 15 8 1 2: nibble j = column j,
# so the word reads (high to low) 2 1 8 F 0 3 7 7
QZEROS_HAND = np.array([[0x218F0377]], dtype=np.uint32)


def test_gptq_weights_match_hand_bytes():
    scales = np.ones((1, 8), dtype=np.float64)
    w, s, zp = F.gptq_to_canonical(QWEIGHT_HAND, None, scales, 32, 8, 32, 0)
    assert w.shape == (8, 16)
    assert bytes(w[0]) == W_ROW0_HAND
    assert bytes(w[1]) == W_ROW1_HAND
    assert not w[2:].any()
    assert zp is None
    assert s.shape == (8, 1)


def test_gptq_zero_points_match_hand_values():
    scales = np.ones((1, 8), dtype=np.float64)
    _, _, z0 = F.gptq_to_canonical(QWEIGHT_HAND, QZEROS_HAND, scales, 32, 8, 32, 0)
    _, _, z1 = F.gptq_to_canonical(QWEIGHT_HAND, QZEROS_HAND, scales, 32, 8, 32, 1)
    assert z0[:, 0].tolist() == [7, 7, 3, 0, 15, 8, 1, 2]
    # offset 1; the stored 15 would be 16, outside 4 bits: written as 15 and
    # reported as not fitting
    assert z1[:, 0].tolist() == [8, 8, 4, 1, 15, 9, 2, 3]
    assert F.gptq_zero_points_fit(QZEROS_HAND, 32, 8, 32, 0)
    assert not F.gptq_zero_points_fit(QZEROS_HAND, 32, 8, 32, 1)
    assert F.gptq_zero_points_fit(None, 32, 8, 32, 1)


def test_zero_offset_rule_of_the_pages():
    # auto_gptq symmetric: every stored zero 7 -> offset 1 (real zero 8)
    assert F.gptq_zero_offset(np.full((4, 2), 0x77777777, dtype=np.uint32)) == 1
    # stored as is (Qwen3.5 symmetric): 8 -> offset 0
    assert F.gptq_zero_offset(np.full((4, 2), 0x88888888, dtype=np.uint32)) == 0
    # lower median: 5 sevens and 3 eights among 8 entries -> median 7
    assert F.gptq_zero_offset(np.array([[0x88877777]], dtype=np.uint32)) == 1
    # 4 sevens, 4 eights: the 4th of 8 sorted values is 7 -> 1
    assert F.gptq_zero_offset(np.array([[0x88887777]], dtype=np.uint32)) == 1
    # 3 sevens, 5 eights -> median 8 -> 0
    assert F.gptq_zero_offset(np.array([[0x88888777]], dtype=np.uint32)) == 0


def test_unpack_zero_points_hand_example():
    # nb = 5 per row: bytes 0x21 0x43 0x05 -> 1 2 3 4 5; second row 0xf0 0x7e 0x0a -> 0 15 14 7 10
    packed = np.array([[0x21, 0x43, 0x05], [0xF0, 0x7E, 0x0A]], dtype=np.uint8)
    out = F.unpack_zero_points(packed, 2, 5)
    assert out.tolist() == [[1, 2, 3, 4, 5], [0, 15, 14, 7, 10]]


def _random_gptq(rng, K, N, bs, stored_zero=None):
    qweight = rng.integers(0, 2 ** 32, size=(K // 8, N), dtype=np.uint64).astype(np.uint32)
    if stored_zero is None:
        qzeros = rng.integers(0, 2 ** 32, size=(K // bs, N // 8), dtype=np.uint64).astype(np.uint32)
        # keep stored zeros <= 14 so that offset 1 stays inside 4 bits
        qzeros &= np.uint32(0x77777777)
    else:
        qzeros = np.full((K // bs, N // 8), stored_zero * 0x11111111, dtype=np.uint32)
    scales16 = (rng.uniform(0.5, 1.5, size=(K // bs, N)) * 2 ** -5).astype(np.float16)
    return qweight, qzeros, scales16


@pytest.mark.parametrize("offset", [0, 1])
def test_gptq_dequant_agrees_with_the_c_oracle(offset):
    """The converted weights through the C oracle's DequantizeLinear equal
    the GPTQ definition (q - (stored + offset)) * s, element by element."""
    rng = np.random.default_rng(7)
    K, N, bs = 64, 16, 32
    qweight, qzeros, s16 = _random_gptq(rng, K, N, bs)
    w, s, zp = F.gptq_to_canonical(qweight, qzeros, s16.view(np.uint16), K, N, bs, offset)
    got = oracle.dequant(w, s, oracle.F16, zp, N, K, bs)
    ref = F.gptq_dequant(qweight, qzeros, s16.astype(np.float64), K, N, bs, offset)
    assert np.array_equal(got, ref)


def test_symmetric_auto_gptq_equals_implied_zero_point_8():
    """Stored zeros all 7 with offset 1 dequantise exactly like the canonical
    layout without zero points (zero point 8)."""
    rng = np.random.default_rng(8)
    K, N, bs = 64, 16, 32
    qweight, qzeros, s16 = _random_gptq(rng, K, N, bs, stored_zero=7)
    assert F.gptq_zero_offset(qzeros) == 1
    w, s, zp = F.gptq_to_canonical(qweight, qzeros, s16.view(np.uint16), K, N, bs, 1)
    assert (zp == 8).all()
    with_zp = oracle.dequant(w, s, oracle.F16, zp, N, K, bs)
    without = oracle.dequant(w, s, oracle.F16, None, N, K, bs)
    assert np.array_equal(with_zp, without)


def test_planted_nibble_order_mistake_is_caught():
    """Swapping the nibbles of a canonical byte (a plausible packing mistake)
    breaks the hand image."""
    scales = np.ones((1, 8), dtype=np.float64)
    w, _, _ = F.gptq_to_canonical(QWEIGHT_HAND, None, scales, 32, 8, 32, 0)
    swapped = ((w[0] >> 4) | (w[0] << 4)).astype(np.uint8)
    assert bytes(swapped) != W_ROW0_HAND
