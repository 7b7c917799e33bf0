"""The C-ABI library loads, exports every symbol its header declares, and
rejects bad arguments on the host (no GPU needed for any of this)."""
import ctypes
import os
import re
import subprocess

import pytest

import oracle
import structured_sparse_gemm_gb300 as st

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in sorted(os.listdir(os.path.join(ROOT, "include")))
           if f.endswith(".h")]


def declared_functions():
    names = set()
    for h in HEADERS:
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"\b(st24_\w+)\s*\(", text))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    from structured_sparse_gemm_gb300 import _build_lib
    _build_lib.build()
    return st.load()


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert {"st24_prune_compress", "st24_decompress", "st24_spmm"} <= set(names)
    out = subprocess.run(["nm", "-D", "--defined-only", st._build_lib.LIB], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (st24_\w+)$", out, flags=re.M))
    for n in names:
        assert n in exported, n
        getattr(lib, n)
    # nothing else leaks out under the st24_ prefix
    assert exported == set(names)


def test_sizes_match_oracle_closed_form(lib):
    # 256 x 1024 at 2 bytes per value: 256 KiB of values + 32 KiB of metadata = 288.0 KB.
    assert st.st24_values_bytes("f16", 256, 1024) == oracle.values_bytes("f16", 256, 1024) == 262144
    assert st.st24_meta_bytes(256, 1024) == oracle.meta_bytes(256, 1024) == 32768
    for dt in ("f16", "bf16", "e4m3", "s8"):
        for M, K in ((1, 4), (3, 12), (7, 1000), (28672, 8192)):
            assert st.st24_values_bytes(dt, M, K) == oracle.values_bytes(dt, M, K)
            assert st.st24_meta_bytes(M, K) == oracle.meta_bytes(M, K)
    assert st.st24_values_bytes("f16", 4, 6) == 0       # K % 4 != 0
    assert st.st24_values_bytes("f32", 4, 8) == 0       # not an input type


def test_status_strings(lib):
    for s in range(7):
        assert st.st24_status_string(s) and st.st24_status_string(s) != "unknown status"
    assert st.st24_status_string(99) == "unknown status"
    assert st.st24_version() > 0


FAKE = 1 << 20   # an aligned non-null address; never dereferenced: the checks run first


def test_prune_compress_rejects_bad_arguments(lib):
    f = lib.st24_prune_compress
    assert f(st.BF16, FAKE, 4, 6, 6, FAKE, FAKE, None) == 1        # K % 4
    assert f(st.F32, FAKE, 4, 8, 8, FAKE, FAKE, None) == 1         # not an input type
    assert f(st.BF16, None, 4, 8, 8, FAKE, FAKE, None) == 1        # null W
    assert f(st.BF16, FAKE, 4, 8, 4, FAKE, FAKE, None) == 1        # ldw < K
    assert f(st.BF16, FAKE, -1, 8, 8, FAKE, FAKE, None) == 1       # negative M
    assert f(st.BF16, None, 0, 8, 8, None, None, None) == 0        # empty: no-op
    assert lib.st24_decompress(st.E4M3, FAKE, None, 4, 8, FAKE, 8, None) == 1


def test_prune_compress_nm_rejects_bad_arguments(lib):
    def call(t=st.BF16, n=1, m=4, W=FAKE, M=8, K=64, ldw=64, values=FAKE, meta=FAKE):
        return lib.st24_prune_compress_nm(t, n, m, W, M, K, ldw, values, meta, None)

    assert call(t=st.F32) == 1 and call(K=6) == 1 and call(M=-1) == 1
    assert call(n=3, m=8) == 2 and call(m=16) == 2 and call(n=0) == 2
    assert call(m=8, K=12, ldw=12) == 1                   # K % m
    assert call(M=0) == 0
    assert call(W=None) == 1 and call(ldw=32) == 1
    assert call(W=FAKE + 1) == 3 and call(values=FAKE + 2) == 3


def test_quantize_prune_compress_rejects_bad_arguments(lib):
    def call(src=st.BF16, dst=st.E4M3, W=FAKE, M=8, K=64, ldw=64, values=FAKE, meta=FAKE, scales=FAKE):
        return lib.st24_quantize_prune_compress(src, dst, W, M, K, ldw, values, meta, scales, None)

    assert call(M=-1) == 1 and call(K=6) == 1              # invalid sizes
    assert call(src=st.F32) == 2 and call(dst=st.BF16) == 2 and call(src=st.E4M3, dst=st.S8) == 2
    assert call(M=0) == 0                                  # nothing to do
    assert call(W=None) == 1 and call(scales=None) == 1 and call(ldw=32) == 1
    assert call(K=8, ldw=8) == 2                           # K % 16 != 0
    assert call(W=FAKE + 2) == 3 and call(ldw=68) == 3 and call(values=FAKE + 4) == 3
    assert call(meta=FAKE + 1) == 3 and call(scales=FAKE + 2) == 3


def test_spmm_rejects_bad_arguments(lib):
    f = lib.st24_spmm

    def call(ab=st.BF16, c=st.BF16, M=128, N=8, K=256, alpha=1.0, beta=0.0, v=FAKE, e=FAKE, B=FAKE,
             ldb=256, C=FAKE, ldc=128, scale=None):
        return f(ab, c, M, N, K, alpha, v, e, B, ldb, beta, C, ldc, scale, None, 0, None)

    assert call(K=130) == 1                              # K % 4
    assert call(K=132) == 2                              # K % 128: unsupported
    assert call(c=st.S32) == 2                           # int32 out needs int8 in
    assert call(ab=st.S8, c=st.S32, alpha=2.0) == 2      # int32 out: plain sums only
    assert call(ab=st.F32) == 1
    assert call(v=None) == 1
    assert call(ldb=128) == 1                            # ldb < K
    assert call(ldc=64) == 1                             # ldc < M
    assert call(v=FAKE + 8) == 3                         # A values not 16-byte aligned
    assert call(ldb=260) == 3                            # ldb * 2 bytes not a multiple of 16
    assert call(C=FAKE + 1) == 3                         # C not aligned to its element
    assert call(M=0, v=None, e=None, B=None, C=None) == 0    # empty: no-op


def test_direct_kernel_rejects_what_it_does_not_cover(lib):
    # the register-direct family takes 1 <= N <= 32 only
    def call(ab, c, N):
        return lib.st24_spmm_ex(st.KERNEL_MMA_SP_DIRECT, 0, ab, c, 128, N, 256, 1.0, FAKE, FAKE, FAKE, 256, 0.0,
                                FAKE, 128, None, None, 0, None)

    for ab, c in ((st.BF16, st.BF16), (st.F16, st.F32), (st.E4M3, st.BF16), (st.S8, st.S32)):
        assert call(ab, c, 33) == 2


def test_two_forms_flag_checks(lib):
    # two 2:4 forms side by side: K must be a multiple of 256, and the register-direct family declines them
    def call(kernel, K):
        return lib.st24_spmm_ex(kernel, st.SPMM_TWO_FORMS, st.BF16, st.BF16, 128, 8, K, 1.0, FAKE, FAKE, FAKE, K, 0.0,
                                FAKE, 128, None, None, 0, None)

    assert call(st.KERNEL_AUTO, 384) == 2
    assert call(st.KERNEL_MMA_SP_DIRECT, 512) == 2


def test_narrow_kernel_rejects_what_it_does_not_cover(lib):
    # the narrow tcgen05 family takes 1 <= N <= 64 and no int8 (no int8 tcgen05 kind on sm_103a)
    def call(ab, c, N):
        return lib.st24_spmm_ex(st.KERNEL_TCGEN05_NARROW, 0, ab, c, 128, N, 256, 1.0, FAKE, FAKE, FAKE, 256, 0.0,
                                FAKE, 128, None, None, 0, None)

    for ab, c in ((st.BF16, st.BF16), (st.F16, st.F32), (st.E4M3, st.BF16)):
        assert call(ab, c, 65) == 2
    assert call(st.S8, st.S32, 16) == 2


def test_spmm_ex_rejects_unknown_kernel_and_flags(lib):
    def call(kernel=0, flags=0):
        return lib.st24_spmm_ex(kernel, flags, st.BF16, st.BF16, 128, 8, 256, 1.0, FAKE, FAKE, FAKE, 256, 0.0,
                                FAKE, 128, None, None, 0, None)

    assert call(kernel=5) == 1
    assert call(kernel=-1) == 1
    assert call(flags=4) == 1
    assert call(flags=1 << 31) == 1
    assert call(kernel=7, flags=1) == 1
