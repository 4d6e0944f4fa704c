"""GPU parity of MatMulNBits on the tensor-core path (matmul_nbits_ex with
M above the decode token limit) against the fp64 oracle, plus an exactness
pin: with one-hot rows of x, each output is one dequantised weight, which
the exact hi + lo split must reproduce after a single rounding to the
output type.  Every call goes through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
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


def _gen(seed):
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    return g


def _tdt(dt):
    return torch.bfloat16 if dt == S.BF16 else torch.float16


def _qmat(N, K, bs, sdt, zp, seed):
    g = _gen(seed)
    w = torch.randint(0, 256, (N, K // 2), generator=g, device=DEV, dtype=torch.uint8)
    s = ((torch.rand((N, K // bs), generator=g, device=DEV) + 0.5) / 32).to(_tdt(sdt))
    z = torch.randint(0, 16, (N, K // bs), generator=g, device=DEV, dtype=torch.uint8) if zp else None
    return w, s, z


DENSE_CASES = [
    # M, N, K, bs, act, scale, zp
    (17, 128, 64, 32, S.F16, S.F16, True),         # smallest tile shapes, M just above the GEMV limit
    (200, 256, 512, 64, S.BF16, S.BF16, False),    # two ragged token tiles
    (300, 384, 1024, 128, S.BF16, S.F16, True),    # bf16 x with fp16 scales (split scales)
    (129, 128, 2048, 32, S.F16, S.BF16, True),     # one row past a tile
    (512, 2048, 1408, 32, S.F16, S.F16, True),     # the layer's down-projection shape
    (512, 1408, 2048, 128, S.BF16, S.BF16, False),  # the layer's gate/up shape
]


@pytest.mark.parametrize("case", DENSE_CASES, ids=[str(c[:4]) for c in DENSE_CASES])
def test_dense_matches_oracle(case, path=B.PATH_AUTO):
    M, N, K, bs, adt, sdt, zp = case
    w, s, z = _qmat(N, K, bs, sdt, zp, 31 + M + N)
    x = torch.randn((M, K), generator=_gen(32 + K), device=DEV).to(_tdt(adt))
    y = B.matmul_nbits_ex(x, w, s, z, bs, path=path)
    torch.cuda.synchronize()
    ref = oracle.matmul_nbits(x, adt, w, s, sdt, z, M, N, K, bs)
    assert_close_layer(y, ref, "matmul_nbits_ex")
    # exact operands add only fp32 summation error to one output rounding
    ulp = 2.0 ** -8 if adt == S.BF16 else 2.0 ** -11
    err = np.abs(to_f64(y) - ref)
    assert (err <= ulp * np.abs(ref) + 1e-3 * (1 + np.abs(ref))).all()


@pytest.mark.parametrize("adt,sdt,zp,bs", [(S.F16, S.F16, True, 32), (S.BF16, S.BF16, False, 128),
                                           (S.BF16, S.F16, True, 64), (S.F16, S.BF16, True, 32)])
def test_dense_one_hot_rows_give_the_dequantised_weights(adt, sdt, zp, bs):
    """x[r] = e_(r mod K): y[r, n] = RN(dequant(W)[n, r mod K]) bit for bit."""
    M, N, K = 320, 256, 256
    w, s, z = _qmat(N, K, bs, sdt, zp, 41 + bs)
    x = torch.zeros((M, K), device=DEV, dtype=_tdt(adt))
    rows = torch.arange(M, device=DEV)
    x[rows, rows % K] = 1
    y = B.matmul_nbits_ex(x, w, s, z, bs, path=B.PATH_PREFILL)
    deq = oracle.dequant(w, s, sdt, z, N, K, bs)            # exact in fp64, <= 15 significant bits
    want = torch.from_numpy(deq.T[np.arange(M) % K].copy()).float().to(_tdt(adt))
    assert torch.equal(y.cpu(), want)


def test_dense_auto_small_m_uses_the_gemv_path():
    M, N, K, bs = 8, 256, 512, 32
    w, s, z = _qmat(N, K, bs, S.F16, True, 51)
    x = torch.randn((M, K), generator=_gen(52), device=DEV).half()
    a = B.matmul_nbits_ex(x, w, s, z, bs)
    b = B.matmul_nbits(x, w, s, z, bs)
    assert torch.equal(a, b)


def test_dense_repeat_is_deterministic():
    M, N, K, bs = 384, 512, 1024, 64
    w, s, z = _qmat(N, K, bs, S.BF16, False, 61)
    x = torch.randn((M, K), generator=_gen(62), device=DEV).bfloat16()
    ws = B.Workspace(M, N, K, 1, 1)
    a = B.matmul_nbits_ex(x, w, s, z, bs, ws=ws)
    b = B.matmul_nbits_ex(x, w, s, z, bs, ws=ws)
    assert torch.equal(a, b)
    assert ws.status()[1] == 0


def test_dense_rejects_unsupported_shape():
    w, s, z = _qmat(200, 512, 32, S.F16, False, 71)
    x = torch.randn((64, 512), generator=_gen(72), device=DEV).half()
    with pytest.raises(RuntimeError):
        B.matmul_nbits_ex(x, w, s, z, 32, path=B.PATH_PREFILL)
