"""Host-side checks of the C ABI (no GPU): the library builds and loads,
exports every entry point include/qmoe.h declares, and rejects bad
arguments with the documented status before enqueueing anything."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qmoe.h")


@pytest.fixture(scope="module")
def L():
    from int4_block_quantized_gb300 import build as b
    b.build()
    from int4_block_quantized_gb300 import binding
    return binding.lib()


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\**\s+\**([A-Za-z_][A-Za-z0-9_]*)\s*\(",
                       src, flags=re.M)
    return sorted(set(n for n in names if n not in ("typedef",)))


def test_header_declares_the_entry_points():
    names = _declared()
    for n in ("qmoe_route", "matmul_nbits", "qmoe_forward", "qmoe_forward_ex", "qmoe_dequant",
              "qmoe_rmsnorm", "qmoe_workspace_size", "qmoe_workspace_init", "qmoe_status_string",
              "qmoe_get_device_status", "qmoe_forward_noalloc", "qmoe_shared_expert",
              "matmul_nbits_ex"):
        assert n in names, n


def test_library_exports_every_declared_symbol(L):
    for n in _declared():
        assert hasattr(L, n), "libqmoe.so does not export %s" % n


def test_status_strings(L):
    for code in range(7):
        s = L.qmoe_status_string(code)
        assert s and s.decode() != "unknown status"
    assert L.qmoe_status_string(99).decode() == "unknown status"


def test_workspace_size(L):
    a = L.qmoe_workspace_size(1, 2048, 1408, 60, 4)
    b = L.qmoe_workspace_size(16, 2048, 1408, 60, 4)
    c = L.qmoe_workspace_size(2048, 2048, 1408, 60, 4)
    assert 0 < a < b < c
    assert c % 256 == 0
    assert L.qmoe_workspace_size(0, 2048, 1408, 60, 4) == 0


FAKE = 0x10000  # 16-byte aligned, never dereferenced: every call below fails its checks first


def _route(L, **kw):
    a = dict(x=FAKE, rw=FAKE, dt=0, bias=None, T=4, H=256, E=8, k=2, tw=FAKE, ti=FAKE, off=None,
             perm=None, ws=FAKE, wsb=1 << 30, st=None)
    a.update(kw)
    return L.qmoe_route(a["x"], a["rw"], a["dt"], a["bias"], a["T"], a["H"], a["E"], a["k"], a["tw"],
                        a["ti"], a["off"], a["perm"], a["ws"], a["wsb"], a["st"])


def test_route_rejects_bad_arguments(L):
    assert _route(L, x=None) == 1
    assert _route(L, dt=7) == 1
    assert _route(L, T=0) == 1
    assert _route(L, k=9, E=8) == 1          # k > E
    assert _route(L, E=300, k=2) == 2        # more experts than supported
    assert _route(L, E=60, k=9) == 2         # k above 8
    assert _route(L, x=FAKE + 2) == 1        # x not 16-byte aligned
    assert _route(L, tw=None) == 1
    assert _route(L, ws=None) == 3
    assert _route(L, wsb=16) == 3
    assert _route(L, ws=FAKE + 64) == 3      # workspace not 256-byte aligned


def test_matmul_nbits_rejects_bad_arguments(L):
    call = lambda **kw: L.matmul_nbits(kw.get("x", FAKE), 0, kw.get("w", FAKE), kw.get("s", FAKE), 0,
                                       None, kw.get("M", 1), kw.get("N", 8), kw.get("K", 64),
                                       kw.get("bs", 32), kw.get("y", FAKE), None)
    assert call(w=None) == 1
    assert call(K=48) == 1                   # K not a multiple of 32
    assert call(bs=16) == 1                  # unsupported block size
    assert call(K=96, bs=64) == 1            # K not a multiple of block_size
    assert call(M=0) == 1
    assert call(w=FAKE + 8) == 1             # packed weights must be 16-byte aligned


def test_matmul_nbits_ex_rejects_bad_arguments(L):
    big = 1 << 40
    def call(**kw):
        return L.matmul_nbits_ex(kw.get("x", FAKE), 0, kw.get("w", FAKE), kw.get("s", FAKE), 0, None,
                                 kw.get("M", 64), kw.get("N", 256), kw.get("K", 512), kw.get("bs", 32),
                                 kw.get("y", FAKE), kw.get("path", 2), kw.get("ws", FAKE),
                                 kw.get("wsb", big), None)
    assert call(path=4) == 1 and call(path=-1) == 1
    assert call(M=0) == 1
    assert call(x=None) == 1
    assert call(K=48) == 1                   # K not a multiple of 32
    assert call(x=FAKE + 2) == 1             # x must be 16-byte aligned on the tensor-core path
    assert call(ws=None) == 3
    assert call(wsb=16) == 3
    assert call(ws=FAKE + 64) == 3           # workspace not 256-byte aligned
    assert call(N=200) == 2                  # N not a multiple of 128
    assert call(K=96) == 2                   # K not a multiple of 64
    assert call(M=4, path=1, K=48) == 1      # the decode path keeps its own checks


def test_forward_rejects_bad_arguments(L):
    from int4_block_quantized_gb300.binding import QWeight
    q = QWeight(FAKE, FAKE, None)
    qz = QWeight(FAKE, FAKE, FAKE)
    def call(**kw):
        return L.qmoe_forward_ex(FAKE, 0, FAKE, None, kw.get("g", q), kw.get("u", q), kw.get("d", q), 0,
                                 kw.get("T", 1), kw.get("H", 256), kw.get("I", 128), kw.get("E", 8),
                                 kw.get("k", 2), kw.get("bs", 32), kw.get("out", FAKE), None, None, 0,
                                 kw.get("path", 0), kw.get("ws", FAKE), kw.get("wsb", 1 << 30), None)
    assert call(g=QWeight(None, FAKE, None)) == 1
    assert call(g=qz) == 1                   # gate and up must agree on zero points
    assert call(I=100) == 1                  # I not a multiple of 32
    assert call(H=256, bs=128, I=64) == 1    # I not a multiple of block_size
    assert call(path=6) == 1
    assert call(out=None) == 1
    assert call(wsb=100) == 3
    assert call(k=3, E=2) == 1


def test_oracle_and_product_share_no_code():
    """The oracle is test infrastructure: the product package never imports
    or loads it, and the oracle never imports the product package."""
    pkg = os.path.join(ROOT, "int4_block_quantized_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                src = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(from|import)\s+oracle\b", src, flags=re.M), f
                assert "qmoe_oracle" not in src and "oracle_" not in src, f
    for f in os.listdir(os.path.join(ROOT, "oracle")):
        if f.endswith((".py", ".c")):
            assert "int4_block_quantized_gb300" not in open(os.path.join(ROOT, "oracle", f)).read(), f


def test_noalloc_rejects_oversize_shapes_on_the_host(L):
    """The size check precedes any CUDA call: UNSUPPORTED for a workspace
    beyond the 2 MiB static array, INVALID_ARG for T = 0."""
    from int4_block_quantized_gb300.binding import QWeight
    q = QWeight(FAKE, FAKE, None)
    args = lambda T: (FAKE, 1, FAKE, None, q, q, q, 1, T, 2048, 1408, 60, 4, 128, FAKE, None, None, 0, None)
    assert L.qmoe_forward_noalloc(*args(512)) == 2
    assert L.qmoe_forward_noalloc(*args(0)) == 1


def test_shared_expert_requires_gate_vector(L):
    from int4_block_quantized_gb300.binding import QWeight
    q = QWeight(FAKE, FAKE, None)
    assert L.qmoe_shared_expert(FAKE, 0, None, q, q, q, 0, 1, 2048, 5632, 32, FAKE, 0, FAKE, 1 << 30, None) == 1


def test_adapters_reject_bad_arguments(L):
    """GPTQ repack / zero-offset / packed zero-point unpack: argument checks
    happen on the host before anything is enqueued (no GPU needed)."""
    vp = ctypes.c_void_p

    def repack(**kw):
        return L.qmoe_repack_gptq(kw.get("qw", FAKE), kw.get("qz", FAKE), kw.get("s", FAKE), kw.get("E", 2),
                                  kw.get("K", 256), kw.get("N", 64), kw.get("bs", 32), kw.get("off", 1),
                                  kw.get("offdev", None), kw.get("w", FAKE), kw.get("so", FAKE),
                                  kw.get("zp", FAKE), kw.get("st", None), None)
    assert repack(qw=None) == 1
    assert repack(w=None) == 1
    assert repack(qz=None) == 1              # zp_out given without qzeros
    assert repack(zp=None) == 1              # qzeros given without zp_out
    assert repack(N=60) == 1                 # N not a multiple of 8
    assert repack(K=48) == 1                 # K not a multiple of 32
    assert repack(bs=16) == 1                # block size outside {32, 64, 128}
    assert repack(K=320, bs=128) == 1        # K not a multiple of the block size
    assert repack(off=2) == 1                # offset 0 or 1 only
    assert repack(st=FAKE + 2) == 1          # status word not 4-byte aligned
    assert repack(E=0) == 1
    assert repack(qw=FAKE + 2) == 1          # int32 words must be 4-byte aligned
    assert repack(s=FAKE + 1) == 1           # scales must be 2-byte aligned
    assert repack(offdev=vp(FAKE + 2)) == 1  # device offset word must be 4-byte aligned
    assert L.qmoe_gptq_zero_offset(None, 16, FAKE, None) == 1
    assert L.qmoe_gptq_zero_offset(FAKE, 0, FAKE, None) == 1
    assert L.qmoe_gptq_zero_offset(FAKE, 16, None, None) == 1
    assert L.qmoe_unpack_zero_points(None, 4, 5, FAKE, None) == 1
    assert L.qmoe_unpack_zero_points(FAKE, 0, 5, FAKE, None) == 1
    assert L.qmoe_unpack_zero_points(FAKE, 4, 0, FAKE, None) == 1


def test_kernel_count_query_rejects_bad_arguments(L):
    assert L.qmoe_forward_kernels(0, 2048, 1408, 60, 4, 32, 0, 0, 1, 1, 0) == -1
    assert L.qmoe_forward_kernels(1, 2048, 1408, 60, 61, 32, 0, 0, 1, 1, 0) == -1   # k > E
    assert L.qmoe_forward_kernels(1, 2048, 1408, 300, 4, 32, 0, 0, 1, 1, 0) == -1   # E > 256
    assert L.qmoe_forward_kernels(1, 2048, 1408, 60, 4, 48, 0, 0, 1, 1, 0) == -1    # block size
    assert L.qmoe_forward_kernels(1, 2048, 1408, 60, 4, 32, 0, 0, 1, 1, 6) == -1    # path


def test_diagnostics_reject_bad_arguments(L):
    """qmoe_workspace_set_diagnostics: workspace and flag checks happen on the
    host before anything is enqueued."""
    import ctypes
    f = L.qmoe_workspace_set_diagnostics
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_uint32, ctypes.c_uint32, ctypes.c_void_p]
    assert f(None, 1 << 30, 0, 0, None) == 3          # no workspace
    assert f(FAKE + 16, 1 << 30, 0, 0, None) == 3     # not 256-byte aligned
    assert f(FAKE, 64, 0, 0, None) == 3               # smaller than the control block
    assert f(FAKE, 1 << 30, 0, 2, None) == 1          # unknown flag
