"""CPU oracle for 2:4 structured sparsity -- TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously correct implementation of what the sparse path
computes (magnitude prune, compress, decompress, sparse x dense product),
written in C (``st24_oracle.c``, fp64 / int64 arithmetic) and wrapped here
with ctypes + numpy.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import it.  It shares no code with the CUDA
library and never imports it.

What each function follows (web pages, cited by title and section):

* ``prune_compress`` / ``decompress``: "Chapter 26 -- Sparsity: The Hardware
  View", sections "2:4 Fine-Grained Structured Sparsity" (worked example) and
  "Python: Build a 2:4 Mask, Compress It, ..." (keep the 2 largest |w| of each
  group of 4 along K; kept positions sorted ascending); "10.4g Structured
  Sparsity (2:4)", section "What is 2:4 Structured Sparsity?".
* ``spmm`` / ``gemm_dense`` / ``spmm_sampled``: the same chapter, section
  "2:4 Fine-Grained Structured Sparsity" (the stored pair multiplies the two
  activations its indices select; the other two products are zero), with
  C = alpha * (A_sparse * B) + beta * C as the product's definition.
* ``values_bytes`` / ``meta_bytes``: the chapter's storage accounting (half
  the values plus a 2-bit index per kept value).
* ``quantize_prune_compress`` / ``encode_e4m3``: the same chapter, section
  "Sparsity + Quantization Combine", and "Establishing a Scalable Sparse
  Ecosystem with the Universal Sparse Tensor Abstraction", section "Building
  a Practical Compression Pipeline" (2:4 pruning stacked with 8-bit weights);
  the per-row absmax arithmetic is a reading (R7 in ``st24_oracle.c``).
* ``prune_compress_nm``: the same chapter, section "Block Sparsity, N:M
  Generalizations, and Channel Pruning" (keep N of every M; 1:4, 2:8, ...),
  written in the 2:4 form (reading R8).
* ``prune_compress_nm2``: the same section, for patterns that keep up to four
  of a 4-element subgroup (4:8, 3:8), written as two 2:4 forms whose sum is
  the pruned matrix (reading R10).
* ``spmm_t`` / ``spmm_t_sampled``: the transposed use of a compressed weight,
  dX = dY * W (the same chapter, section "2:4: ~2x on the Matmul, Less
  End-to-End": retraining after the prune needs the layer's input gradient),
  summed along M in ascending order (reading R9).

Pins (tests/test_oracle_pins.py): the worked example, the listing's printed
invariants and byte counts, brute force over all 6 masks of every group,
decompress(compress(W)) == prune(W), and agreement of the compressed-form
product with a dense triple loop and with numpy's float64 / int64 matmul.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "st24_oracle.c")
_LIB = os.path.join(_HERE, "_build", "libst24_oracle.so")

# The oracle's own element-type codes.
F16, BF16, E4M3, S8, F32, S32 = 0, 1, 2, 3, 4, 5
NAMES = {"f16": F16, "bf16": BF16, "e4m3": E4M3, "s8": S8, "f32": F32, "s32": S32}
_NP_STORAGE = {F16: np.uint16, BF16: np.uint16, E4M3: np.uint8, S8: np.int8, F32: np.uint32, S32: np.int32}


def build(force: bool = False) -> str:
    """Compile the oracle shared library with gcc (plain C, no CUDA)."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp.%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        i64, p, d, i = ctypes.c_int64, ctypes.c_void_p, ctypes.c_double, ctypes.c_int
        _lib.orc_prune_compress.argtypes = [i, p, i64, i64, i64, p, p, p, p]
        _lib.orc_decompress.argtypes = [i, p, p, i64, i64, p, i64]
        _lib.orc_spmm.argtypes = [i, i, i64, i64, i64, d, p, p, p, i64, d, p, i64, p, p, p, i]
        _lib.orc_gemm_dense.argtypes = [i, i, i64, i64, i64, d, p, i64, p, i64, d, p, i64, p, p, p, i]
        _lib.orc_spmm_sampled.argtypes = [i, i, i64, i64, i64, d, p, p, p, i64, d, p, i64, p,
                                          p, p, i64, p, p, i]
        _lib.orc_decode.argtypes = [i, p, i64, p]
        _lib.orc_spmm_t.argtypes = [i, i, i64, i64, i64, d, p, p, p, i64, d, p, i64, p, p, i]
        _lib.orc_spmm_t_sampled.argtypes = [i, i, i64, i64, i64, d, p, p, p, i64, d, p, i64, p, p, i64, p, p, i]
        _lib.orc_quantize_prune_compress.argtypes = [i, i, p, i64, i64, i64, p, p, p, p]
        _lib.orc_prune_compress_nm.argtypes = [i, i, i, p, i64, i64, i64, p, p, p]
        _lib.orc_prune_compress_nm2.argtypes = [i, i, i, p, i64, i64, i64, p, p, p]
        _lib.orc_enc_e4m3.argtypes = [ctypes.c_float]
        _lib.orc_enc_e4m3.restype = ctypes.c_uint8
        _lib.orc_meta_row_bytes.argtypes = [i64]
        _lib.orc_meta_row_bytes.restype = i64
        _lib.orc_values_bytes.argtypes = [i, i64, i64]
        _lib.orc_values_bytes.restype = i64
        _lib.orc_meta_bytes.argtypes = [i64, i64]
        _lib.orc_meta_bytes.restype = i64
    return _lib


def _code(dt) -> int:
    return NAMES[dt] if isinstance(dt, str) else int(dt)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _as_storage(dt: int, a: np.ndarray) -> np.ndarray:
    want = _NP_STORAGE[dt]
    a = np.ascontiguousarray(a)
    if a.dtype != want:
        if a.dtype.itemsize != np.dtype(want).itemsize:
            raise TypeError(f"array of {a.dtype} is not raw storage for oracle type {dt}")
        a = a.view(want)
    return a


def meta_row_bytes(K: int) -> int:
    return int(lib().orc_meta_row_bytes(K))


def values_bytes(dt, M: int, K: int) -> int:
    return int(lib().orc_values_bytes(_code(dt), M, K))


def meta_bytes(M: int, K: int) -> int:
    return int(lib().orc_meta_bytes(M, K))


def decode(dt, bits: np.ndarray) -> np.ndarray:
    """Real values (float64) of raw element storage."""
    dt = _code(dt)
    bits = _as_storage(dt, bits)
    out = np.empty(bits.shape, np.float64)
    lib().orc_decode(dt, _ptr(bits), bits.size, _ptr(out))
    return out


def prune_compress(dt, W: np.ndarray):
    """Prune W (M x K raw storage) to 2:4 and compress it.

    Returns (pruned M x K, mask M x K uint8, values M x K/2, meta M x ceil(K/8) uint8).
    """
    dt = _code(dt)
    W = _as_storage(dt, W)
    M, K = W.shape
    pruned = np.empty_like(W)
    mask = np.empty((M, K), np.uint8)
    values = np.empty((M, K // 2), W.dtype)
    meta = np.empty((M, meta_row_bytes(K)), np.uint8)
    rc = lib().orc_prune_compress(dt, _ptr(W), M, K, K, _ptr(pruned), _ptr(mask), _ptr(values), _ptr(meta))
    if rc != 0:
        raise ValueError("oracle prune_compress: K must be a multiple of 4 and the type known")
    return pruned, mask, values, meta


def quantize_prune_compress(src, dst, W: np.ndarray):
    """Per-row quantisation of a 16-bit weight (raw storage, M x K) to e4m3 or
    int8 (reading R7 of st24_oracle.c), then prune + compress of the codes.

    Returns (codes M x K before pruning, values M x K/2, meta M x ceil(K/8)
    uint8, scales M float32), codes and values as raw storage of ``dst``.
    """
    src, dst = _code(src), _code(dst)
    W = _as_storage(src, W)
    M, K = W.shape
    st = _NP_STORAGE[dst]
    codes = np.empty((M, K), st)
    values = np.empty((M, K // 2), st)
    meta = np.empty((M, meta_row_bytes(K)), np.uint8)
    scales = np.empty(M, np.float32)
    rc = lib().orc_quantize_prune_compress(src, dst, _ptr(W), M, K, K, _ptr(codes), _ptr(values), _ptr(meta),
                                           _ptr(scales))
    if rc != 0:
        raise ValueError("oracle quantize_prune_compress: 16-bit source, 8-bit destination, K % 4 == 0")
    return codes, values, meta, scales


def prune_compress_nm(dt, n: int, m: int, W: np.ndarray):
    """Keep the n largest |w| of every m consecutive elements along K (ties to the
    lower index; reading R8 of st24_oracle.c) and write the result in the 2:4 form.

    Returns (pruned M x K, values M x K/2, meta M x ceil(K/8) uint8)."""
    dt = _code(dt)
    W = _as_storage(dt, W)
    M, K = W.shape
    pruned = np.empty_like(W)
    values = np.empty((M, K // 2), W.dtype)
    meta = np.empty((M, meta_row_bytes(K)), np.uint8)
    rc = lib().orc_prune_compress_nm(dt, n, m, _ptr(W), M, K, K, _ptr(pruned), _ptr(values), _ptr(meta))
    if rc != 0:
        raise ValueError("oracle prune_compress_nm: (n, m) in {1, 2} x {4, 8}, K % m == 0, a known type")
    return pruned, values, meta


def prune_compress_nm2(dt, n: int, m: int, W: np.ndarray):
    """Keep the n largest |w| of every m along K (n <= 4; reading R10) and write the result
    as two 2:4 forms concatenated along K.

    Returns (pruned M x K, values M x K -- form 0's K/2 then form 1's K/2 per row,
    meta M x 2*ceil(K/8) uint8 -- form 0's bytes then form 1's per row)."""
    dt = _code(dt)
    W = _as_storage(dt, W)
    M, K = W.shape
    pruned = np.empty_like(W)
    values = np.empty((M, K), W.dtype)
    meta = np.empty((M, 2 * meta_row_bytes(K)), np.uint8)
    rc = lib().orc_prune_compress_nm2(dt, n, m, _ptr(W), M, K, K, _ptr(pruned), _ptr(values), _ptr(meta))
    if rc != 0:
        raise ValueError("oracle prune_compress_nm2: m in {4, 8}, 1 <= n <= min(4, m), K % m == 0, a known type")
    return pruned, values, meta


def encode_e4m3(x: np.ndarray) -> np.ndarray:
    """fp32 -> e4m3 codes, nearest-even, saturated to +-448 (reading R7)."""
    x = np.ascontiguousarray(x, np.float32).ravel()
    f = lib().orc_enc_e4m3
    return np.array([f(float(v)) for v in x], np.uint8)


def decompress(dt, values: np.ndarray, meta: np.ndarray, K: int) -> np.ndarray:
    dt = _code(dt)
    values = _as_storage(dt, values)
    meta = np.ascontiguousarray(meta, np.uint8)
    M = values.shape[0]
    out = np.empty((M, K), values.dtype)
    rc = lib().orc_decompress(dt, _ptr(values), _ptr(meta), M, K, _ptr(out), K)
    if rc == -2:
        raise ValueError("oracle decompress: metadata with non-ascending indices")
    if rc != 0:
        raise ValueError("oracle decompress: bad arguments")
    return out


def _c_args(dt_c, C_in, beta):
    if beta == 0.0 or C_in is None:
        return None, 0
    C_in = _as_storage(dt_c, C_in)
    return C_in, C_in.shape[1]


def spmm(dt_ab, dt_c, values, meta, B, K, alpha=1.0, beta=0.0, C_in=None, scale=None, nthreads=0):
    """C = alpha*scale[m]*(A_sparse @ B) + beta*C_in from the compressed form.

    B is given as X[N, K] (element (k, n) at X[n, k]); C_in and the result are
    Y[N, M] (element (m, n) at Y[n, m]).  Returns (out float64 [N, M],
    acc int64 [N, M] -- the exact integer accumulator for int8, else zeros).
    """
    dt_ab, dt_c = _code(dt_ab), _code(dt_c)
    values = _as_storage(dt_ab, values)
    B = _as_storage(dt_ab, B)
    meta = np.ascontiguousarray(meta, np.uint8)
    M, N = values.shape[0], B.shape[0]
    C_in, ldc = _c_args(dt_c, C_in, beta)
    scale = None if scale is None else np.ascontiguousarray(scale, np.float32)
    out = np.empty((N, M), np.float64)
    acc = np.zeros((N, M), np.int64)
    rc = lib().orc_spmm(dt_ab, dt_c, M, N, K, alpha, _ptr(values), _ptr(meta), _ptr(B), B.shape[1],
                        beta, _ptr(C_in), ldc, _ptr(scale), _ptr(out), _ptr(acc), nthreads)
    if rc < 0:
        raise ValueError("oracle spmm: bad arguments")
    return out, acc


def gemm_dense(dt_ab, dt_c, A, B, alpha=1.0, beta=0.0, C_in=None, scale=None, nthreads=0):
    """Plain triple-loop product of a dense A[M, K] (already pruned) with B given as X[N, K]."""
    dt_ab, dt_c = _code(dt_ab), _code(dt_c)
    A = _as_storage(dt_ab, A)
    B = _as_storage(dt_ab, B)
    M, K = A.shape
    N = B.shape[0]
    C_in, ldc = _c_args(dt_c, C_in, beta)
    scale = None if scale is None else np.ascontiguousarray(scale, np.float32)
    out = np.empty((N, M), np.float64)
    acc = np.zeros((N, M), np.int64)
    rc = lib().orc_gemm_dense(dt_ab, dt_c, M, N, K, alpha, _ptr(A), K, _ptr(B), B.shape[1],
                              beta, _ptr(C_in), ldc, _ptr(scale), _ptr(out), _ptr(acc), nthreads)
    if rc < 0:
        raise ValueError("oracle gemm_dense: bad arguments")
    return out, acc


def spmm_sampled(dt_ab, dt_c, values, meta, B, K, rows, cols, alpha=1.0, beta=0.0, C_in=None,
                 scale=None, nthreads=0):
    """Outputs (rows[s], cols[s]) of the compressed-form product, one by one."""
    dt_ab, dt_c = _code(dt_ab), _code(dt_c)
    values = _as_storage(dt_ab, values)
    B = _as_storage(dt_ab, B)
    meta = np.ascontiguousarray(meta, np.uint8)
    M, N = values.shape[0], B.shape[0]
    rows = np.ascontiguousarray(rows, np.int64)
    cols = np.ascontiguousarray(cols, np.int64)
    C_in, ldc = _c_args(dt_c, C_in, beta)
    scale = None if scale is None else np.ascontiguousarray(scale, np.float32)
    out = np.empty(rows.shape, np.float64)
    acc = np.zeros(rows.shape, np.int64)
    rc = lib().orc_spmm_sampled(dt_ab, dt_c, M, N, K, alpha, _ptr(values), _ptr(meta), _ptr(B),
                                B.shape[1], beta, _ptr(C_in), ldc, _ptr(scale), _ptr(rows),
                                _ptr(cols), rows.size, _ptr(out), _ptr(acc), nthreads)
    if rc < 0:
        raise ValueError("oracle spmm_sampled: bad arguments")
    return out, acc


def spmm_t(dt_ab, dt_c, values, meta, dY, K, alpha=1.0, beta=0.0, C_in=None, nthreads=0):
    """dX = alpha * (dY @ A) + beta * C_in for A (M x K) in the compressed form.

    dY is [N, M] (element (m, n) of the transposed product's right operand at
    dY[n, m]); C_in and the result are dX[N, K].  Returns (out float64 [N, K],
    acc int64 [N, K] -- the exact integer sums for int8, else zeros)."""
    dt_ab, dt_c = _code(dt_ab), _code(dt_c)
    values = _as_storage(dt_ab, values)
    dY = _as_storage(dt_ab, dY)
    meta = np.ascontiguousarray(meta, np.uint8)
    M, N = values.shape[0], dY.shape[0]
    C_in, ldc = _c_args(dt_c, C_in, beta)
    out = np.empty((N, K), np.float64)
    acc = np.zeros((N, K), np.int64)
    rc = lib().orc_spmm_t(dt_ab, dt_c, M, N, K, alpha, _ptr(values), _ptr(meta), _ptr(dY), dY.shape[1],
                          beta, _ptr(C_in), ldc, _ptr(out), _ptr(acc), nthreads)
    if rc < 0:
        raise ValueError("oracle spmm_t: bad arguments")
    return out, acc


def spmm_t_sampled(dt_ab, dt_c, values, meta, dY, K, ks, ns, alpha=1.0, beta=0.0, C_in=None, nthreads=0):
    """Outputs (ks[s], ns[s]) of the transposed product, one by one."""
    dt_ab, dt_c = _code(dt_ab), _code(dt_c)
    values = _as_storage(dt_ab, values)
    dY = _as_storage(dt_ab, dY)
    meta = np.ascontiguousarray(meta, np.uint8)
    M, N = values.shape[0], dY.shape[0]
    ks = np.ascontiguousarray(ks, np.int64)
    ns = np.ascontiguousarray(ns, np.int64)
    C_in, ldc = _c_args(dt_c, C_in, beta)
    out = np.empty(ks.shape, np.float64)
    acc = np.zeros(ks.shape, np.int64)
    rc = lib().orc_spmm_t_sampled(dt_ab, dt_c, M, N, K, alpha, _ptr(values), _ptr(meta), _ptr(dY), dY.shape[1],
                                  beta, _ptr(C_in), ldc, _ptr(ks), _ptr(ns), ks.size, _ptr(out), _ptr(acc),
                                  nthreads)
    if rc < 0:
        raise ValueError("oracle spmm_t_sampled: bad arguments")
    return out, acc


def default_threads() -> int:
    return int(lib().orc_default_threads())
