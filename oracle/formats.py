"""Weight-format adapters, plain CPU definition (numpy, integers only).

TEST INFRASTRUCTURE ONLY: the tests may import this module; the library's
product path never does.  It shares no code with the CUDA path.

The library's canonical layout for one projection of E experts:
  w      [E, N, K/2]  uint8, element 2j of a row in the low nibble of byte j
  scales [E, N, K/bs] 16-bit
  zp     [E, N, K/bs] uint8, one zero point 0..15 per block (or absent: 8)
and the dequantised weight is (q - zp) * scale ("Qwen MoE BringUp", local
fix A1, DequantizeLinear with block_size).

Two source formats are converted to it:

GPTQ checkpoints ("Qwen MoE BringUp", "Bugs/Issues Found", item 1: the
qzeros offset).  The pages name the format and its zero-point offset but not
its bit layout; the reading taken here is the common GPTQ packing:
  qweight [K/8, N]    int32, bits 4j..4j+3 of word (i, n) hold q[8i + j, n]
  qzeros  [K/bs, N/8] int32, bits 4j..4j+3 of word (g, i) hold the stored
                      zero point of block g, column 8i + j
  scales  [K/bs, N]   16-bit
with the matrix stored input-major (K rows, N output columns).  The real
zero point is the stored one plus an offset: 1 for checkpoints that store
zero - 1 (the pages: auto_gptq writes 7 for a symmetric model whose zero is
8), 0 for those that store it as is (the pages: 8 for Qwen3.5 symmetric).
The pages detect the offset from the median stored zero; the reading here:
offset 1 if that median is 7, else 0 (the median is the lower median, the
smallest v whose cumulative count reaches half of all entries, rounded up).

Packed 4-bit zero points.  The pages' model stores one byte per block
("Qwen MoE BringUp", the MoE lowering: zeros [60, 2048, 11] ui8), which is
the canonical layout; the pages give no packed zero-point layout.  The
reading taken is the usual 4-bit packing of ONNX MatMulNBits: two zero
points per byte, block 2b in the low nibble and 2b + 1 in the high nibble,
each row padded to a whole byte: [rows, ceil(nb / 2)].
"""
import numpy as np


def gptq_nibble(qweight, k, n):
    """q[k, n] of a GPTQ qweight [K/8, N] (int32 words)."""
    word = int(np.uint32(qweight[k // 8, n]))
    return (word >> (4 * (k % 8))) & 15


def gptq_stored_zero(qzeros, g, n):
    """Stored zero point of block g, column n of a GPTQ qzeros [K/bs, N/8]."""
    word = int(np.uint32(qzeros[g, n // 8]))
    return (word >> (4 * (n % 8))) & 15


def gptq_zero_offset(qzeros):
    """1 if the median stored zero point is 7 (zero - 1 stored), else 0."""
    words = np.asarray(qzeros).astype(np.uint32).reshape(-1)
    counts = [0] * 16
    for wv in words:
        v = int(wv)
        for j in range(8):
            counts[(v >> (4 * j)) & 15] += 1
    total = sum(counts)
    half = (total + 1) // 2
    run = 0
    for v in range(16):
        run += counts[v]
        if run >= half:
            return 1 if v == 7 else 0
    return 0


def gptq_to_canonical(qweight, qzeros, scales, K, N, block_size, zero_offset):
    """One GPTQ matrix -> canonical (w [N, K/2] u8, scales [N, K/bs], zp [N, K/bs] u8 or None).

    `scales` is any 2-D array [K/bs, N] (16-bit patterns or floats); it is
    transposed as stored.  A zero point above 15 after the offset (a stored
    15 with offset 1) does not fit the canonical 4-bit zero point: it is
    written as 15, which changes that block's weights by one scale step, and
    gptq_zero_points_fit() reports it; the converter reports the same
    condition as a device status bit."""
    nb = K // block_size
    qweight = np.asarray(qweight)
    w = np.zeros((N, K // 2), dtype=np.uint8)
    for n in range(N):
        for j in range(K // 2):
            lo = gptq_nibble(qweight, 2 * j, n)
            hi = gptq_nibble(qweight, 2 * j + 1, n)
            w[n, j] = lo | (hi << 4)
    s = np.asarray(scales).reshape(nb, N).T.copy()
    zp = None
    if qzeros is not None:
        qzeros = np.asarray(qzeros)
        zp = np.zeros((N, nb), dtype=np.uint8)
        for n in range(N):
            for g in range(nb):
                zp[n, g] = min(gptq_stored_zero(qzeros, g, n) + zero_offset, 15)
    return w, s, zp


def gptq_zero_points_fit(qzeros, K, N, block_size, zero_offset):
    """True when every stored zero + offset is at most 15, i.e. the GPTQ
    matrix converts to the canonical layout without changing a weight."""
    if qzeros is None:
        return True
    qzeros = np.asarray(qzeros)
    return all(gptq_stored_zero(qzeros, g, n) + zero_offset <= 15
               for n in range(N) for g in range(K // block_size))


def gptq_dequant(qweight, qzeros, scales, K, N, block_size, zero_offset):
    """fp64 [N, K] weight of a GPTQ matrix: (q - (stored zero + offset)) * scale,
    scales given as floats [K/bs, N]; no qzeros: zero point 8."""
    out = np.zeros((N, K), dtype=np.float64)
    for n in range(N):
        for k in range(K):
            g = k // block_size
            z = 8 if qzeros is None else gptq_stored_zero(qzeros, g, n) + zero_offset
            out[n, k] = (gptq_nibble(qweight, k, n) - z) * float(scales[g, n])
    return out


def unpack_zero_points(zp_packed, rows, nb):
    """[rows, ceil(nb/2)] packed 4-bit zero points -> [rows, nb] uint8."""
    zp_packed = np.asarray(zp_packed).reshape(rows, (nb + 1) // 2)
    out = np.zeros((rows, nb), dtype=np.uint8)
    for r in range(rows):
        for b in range(nb):
            byte = int(zp_packed[r, b // 2])
            out[r, b] = (byte >> (4 * (b % 2))) & 15
    return out
