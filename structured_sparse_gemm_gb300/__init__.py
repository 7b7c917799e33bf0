"""Python binding of libst24 (2:4 structured-sparse GEMM for GB300, sm_103a).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  The functions keep the C ABI's names (include/st24.h) and take
torch tensors for the buffers; they raise ``St24Error`` on a non-OK status.
There is no CPU fallback: if the library is missing the import of the
binding's functions raises.

Layouts (as in the C ABI): A is the sparse weight [M, K] (pruned along K),
B is passed as the activation X[N, K] (K-major B), C is Y[N, M].
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import _build_lib

__all__ = [
    "St24Error", "load", "st24_version", "st24_status_string", "st24_values_bytes",
    "st24_meta_bytes", "st24_prune_compress", "st24_decompress", "st24_spmm_workspace_bytes",
    "st24_spmm", "st24_spmm_ex", "st24_spmm_noalloc", "st24_spmm_t", "st24_prune_compress_nm2", "compress_nm2", "st24_device_status", "dtype_code", "compress", "spmm", "Workspace",
]

F16, BF16, E4M3, S8, F32, S32 = 0, 1, 2, 3, 4, 5
KERNEL_AUTO, KERNEL_TCGEN05, KERNEL_MMA_SP, KERNEL_MMA_SP_DIRECT, KERNEL_TCGEN05_NARROW = 0, 1, 2, 3, 4
SPMM_FIXED_A = 1   # st24_spmm_flags: A is fixed weights no in-flight work on the stream writes
SPMM_TWO_FORMS = 2   # st24_spmm_flags: A is two 2:4 forms side by side (st24_prune_compress_nm2)
_KERNELS = {"auto": KERNEL_AUTO, "tcgen05": KERNEL_TCGEN05, "mma_sp": KERNEL_MMA_SP,
            "mma_sp_direct": KERNEL_MMA_SP_DIRECT, "tcgen05_narrow": KERNEL_TCGEN05_NARROW}
_TORCH_CODE = {
    torch.float16: F16, torch.bfloat16: BF16, torch.float8_e4m3fn: E4M3, torch.int8: S8,
    torch.float32: F32, torch.int32: S32,
}


class St24Error(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {st24_status_string(status)} (status {status})")


_lib = None


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libst24.so (built in-tree by ``_build_lib.build``)."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or _build_lib.LIB
    if not os.path.exists(path):
        raise RuntimeError(f"libst24 is not built ({path} missing); run __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    i64, p, f, sz, i = ctypes.c_int64, ctypes.c_void_p, ctypes.c_float, ctypes.c_size_t, ctypes.c_int
    lib.st24_version.restype = i
    lib.st24_status_string.argtypes = [i]
    lib.st24_status_string.restype = ctypes.c_char_p
    lib.st24_values_bytes.argtypes = [i, i64, i64]
    lib.st24_values_bytes.restype = sz
    lib.st24_meta_bytes.argtypes = [i64, i64]
    lib.st24_meta_bytes.restype = sz
    lib.st24_prune_compress.argtypes = [i, p, i64, i64, i64, p, p, p]
    lib.st24_prune_compress.restype = i
    lib.st24_prune_compress_nm.argtypes = [i, i, i, p, i64, i64, i64, p, p, p]
    lib.st24_prune_compress_nm.restype = i
    lib.st24_prune_compress_nm2.argtypes = [i, i, i, p, i64, i64, i64, p, p, p]
    lib.st24_prune_compress_nm2.restype = i
    lib.st24_quantize_prune_compress.argtypes = [i, i, p, i64, i64, i64, p, p, p, p]
    lib.st24_quantize_prune_compress.restype = i
    lib.st24_decompress.argtypes = [i, p, p, i64, i64, p, i64, p]
    lib.st24_decompress.restype = i
    lib.st24_spmm_workspace_bytes.argtypes = [i, i, i64, i64, i64]
    lib.st24_spmm_workspace_bytes.restype = sz
    lib.st24_spmm.argtypes = [i, i, i64, i64, i64, f, p, p, p, i64, f, p, i64, p, p, sz, p]
    lib.st24_spmm.restype = i
    lib.st24_spmm_ex.argtypes = [i, ctypes.c_uint, i, i, i64, i64, i64, f, p, p, p, i64, f, p, i64, p, p, sz, p]
    lib.st24_spmm_ex.restype = i
    lib.st24_spmm_noalloc.argtypes = [i, i, i64, i64, i64, f, p, p, p, i64, f, p, i64, p, p]
    lib.st24_spmm_noalloc.restype = i
    lib.st24_spmm_t.argtypes = [i, i, i64, i64, i64, f, p, p, p, i64, f, p, i64, p]
    lib.st24_spmm_t.restype = i
    lib.st24_selftest_wait_timeout.argtypes = [p]
    lib.st24_selftest_wait_timeout.restype = i
    lib.st24_device_status.argtypes = [p]
    lib.st24_device_status.restype = i
    _lib = lib
    return lib


def dtype_code(dt) -> int:
    if isinstance(dt, int):
        return dt
    if isinstance(dt, torch.dtype):
        return _TORCH_CODE[dt]
    return {"f16": F16, "bf16": BF16, "e4m3": E4M3, "s8": S8, "f32": F32, "s32": S32}[dt]


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, what: str) -> None:
    if status != 0:
        raise St24Error(status, what)


def st24_version() -> int:
    return load().st24_version()


def st24_status_string(status: int) -> str:
    return load().st24_status_string(status).decode()


def st24_values_bytes(dt, M: int, K: int) -> int:
    return load().st24_values_bytes(dtype_code(dt), M, K)


def st24_meta_bytes(M: int, K: int) -> int:
    return load().st24_meta_bytes(M, K)


def st24_prune_compress(W: torch.Tensor, values: torch.Tensor, meta: torch.Tensor, *, stream=None) -> None:
    """Prune W [M, K] (row stride W.stride(0)) to 2:4 and write its compressed form."""
    M, K = W.shape
    if W.stride(1) != 1:
        raise ValueError("W must have unit stride along K")
    _check(load().st24_prune_compress(dtype_code(W.dtype), _ptr(W), M, K, W.stride(0), _ptr(values),
                                      _ptr(meta), _stream(stream)), "st24_prune_compress")


def st24_prune_compress_nm(W: torch.Tensor, values: torch.Tensor, meta: torch.Tensor, n: int, m: int, *,
                           stream=None) -> None:
    """Keep the n largest-|w| of every m consecutive elements of W [M, K] along K ((n, m) in
    {1, 2} x {4, 8}) and write the result in the 2:4 compressed form."""
    M, K = W.shape
    if W.stride(1) != 1:
        raise ValueError("W must have unit stride along K")
    _check(load().st24_prune_compress_nm(dtype_code(W.dtype), n, m, _ptr(W), M, K, W.stride(0), _ptr(values),
                                         _ptr(meta), _stream(stream)), "st24_prune_compress_nm")


def st24_prune_compress_nm2(W: torch.Tensor, values: torch.Tensor, meta: torch.Tensor, n: int, m: int, *,
                            stream=None) -> None:
    """Keep the n largest |w| of every m along K (n <= 4) as two 2:4 forms: values [M, K]
    (form 0's K/2 then form 1's per row), meta [M, 2 * ceil(K/8)]."""
    M, K = W.shape
    if W.stride(1) != 1:
        raise ValueError("W must have unit stride along K")
    _check(load().st24_prune_compress_nm2(dtype_code(W.dtype), n, m, _ptr(W), M, K, W.stride(0), _ptr(values),
                                          _ptr(meta), _stream(stream)), "st24_prune_compress_nm2")


def st24_quantize_prune_compress(W: torch.Tensor, values: torch.Tensor, meta: torch.Tensor, scales: torch.Tensor,
                                 *, stream=None) -> None:
    """Quantise each row of W [M, K] (f16/bf16) to values' 8-bit type (e4m3 or int8) with a
    per-row absmax scale, prune the codes to 2:4 and write their compressed form and the scales."""
    M, K = W.shape
    if W.stride(1) != 1:
        raise ValueError("W must have unit stride along K")
    _check(load().st24_quantize_prune_compress(dtype_code(W.dtype), dtype_code(values.dtype), _ptr(W), M, K,
                                               W.stride(0), _ptr(values), _ptr(meta), _ptr(scales),
                                               _stream(stream)), "st24_quantize_prune_compress")


def st24_decompress(values: torch.Tensor, meta: torch.Tensor, W: torch.Tensor, *, stream=None) -> None:
    """Expand a compressed form into W [M, K] (+0 at dropped positions)."""
    M, K = W.shape
    if W.stride(1) != 1:
        raise ValueError("W must have unit stride along K")
    _check(load().st24_decompress(dtype_code(W.dtype), _ptr(values), _ptr(meta), M, K, _ptr(W),
                                  W.stride(0), _stream(stream)), "st24_decompress")


def st24_spmm_workspace_bytes(ab, c, M: int, N: int, K: int) -> int:
    return load().st24_spmm_workspace_bytes(dtype_code(ab), dtype_code(c), M, N, K)


def st24_spmm(values: torch.Tensor, meta: torch.Tensor, X: torch.Tensor, Y: torch.Tensor, *, K: int | None = None,
              alpha: float = 1.0, beta: float = 0.0, row_scale: torch.Tensor | None = None,
              workspace: torch.Tensor | None = None, M: int | None = None, stream=None,
              kernel: str | int = "auto", fixed_a: bool = False, two_forms: bool = False) -> None:
    """Y[N, M] = alpha * row_scale * (A_sparse @ X.T).T + beta * Y, A given by (values, meta).

    ``kernel`` picks the kernel family ("auto", "tcgen05", "mma_sp",
    "mma_sp_direct" or "tcgen05_narrow");
    ``fixed_a`` declares (values, meta) fixed weights that no work still in
    flight on the stream writes (ST24_SPMM_FIXED_A); ``two_forms`` says they
    hold two 2:4 forms side by side (ST24_SPMM_TWO_FORMS; K is B's K).
    Anything but the defaults goes through st24_spmm_ex."""
    N, Kx = X.shape
    K = Kx if K is None else K
    M = Y.shape[1] if M is None else M
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if X.stride(1) != 1 or Y.stride(1) != 1:
        raise ValueError("X and Y must have unit stride along their last dimension")
    args = (dtype_code(X.dtype), dtype_code(Y.dtype), M, N, K, float(alpha), _ptr(values), _ptr(meta), _ptr(X),
            X.stride(0), float(beta), _ptr(Y), Y.stride(0), _ptr(row_scale), _ptr(workspace), ws_bytes,
            _stream(stream))
    k = _KERNELS[kernel] if isinstance(kernel, str) else int(kernel)
    flags = (SPMM_FIXED_A if fixed_a else 0) | (SPMM_TWO_FORMS if two_forms else 0)
    if k == KERNEL_AUTO and flags == 0:
        _check(load().st24_spmm(*args), "st24_spmm")
    else:
        _check(load().st24_spmm_ex(k, flags, *args), "st24_spmm_ex")


def st24_spmm_t(values: torch.Tensor, meta: torch.Tensor, dY: torch.Tensor, dX: torch.Tensor, *, K: int | None = None,
                alpha: float = 1.0, beta: float = 0.0, M: int | None = None, stream=None) -> None:
    """dX[N, K] = alpha * dY[N, M] @ A + beta * dX, A (M x K) given by (values, meta)."""
    N, Mx = dY.shape
    M = Mx if M is None else M
    K = dX.shape[1] if K is None else K
    if dY.stride(1) != 1 or dX.stride(1) != 1:
        raise ValueError("dY and dX must have unit stride along their last dimension")
    _check(load().st24_spmm_t(dtype_code(dY.dtype), dtype_code(dX.dtype), M, N, K, float(alpha), _ptr(values),
                              _ptr(meta), _ptr(dY), dY.stride(0), float(beta), _ptr(dX), dX.stride(0),
                              _stream(stream)), "st24_spmm_t")


def st24_spmm_noalloc(values: torch.Tensor, meta: torch.Tensor, X: torch.Tensor, Y: torch.Tensor, *,
                      K: int | None = None, alpha: float = 1.0, beta: float = 0.0,
                      row_scale: torch.Tensor | None = None, M: int | None = None, stream=None) -> None:
    """st24_spmm with the library's own fixed-size scratch (for callers that cannot allocate)."""
    N, Kx = X.shape
    K = Kx if K is None else K
    M = Y.shape[1] if M is None else M
    if X.stride(1) != 1 or Y.stride(1) != 1:
        raise ValueError("X and Y must have unit stride along their last dimension")
    _check(load().st24_spmm_noalloc(dtype_code(X.dtype), dtype_code(Y.dtype), M, N, K, float(alpha), _ptr(values),
                                    _ptr(meta), _ptr(X), X.stride(0), float(beta), _ptr(Y), Y.stride(0),
                                    _ptr(row_scale), _stream(stream)), "st24_spmm_noalloc")


def st24_selftest_wait_timeout(*, stream=None) -> None:
    """Enqueue the self-test whose bounded wait runs out (about a second); the next
    st24_device_status() returns ST24_ERR_TIMEOUT (5)."""
    _check(load().st24_selftest_wait_timeout(_stream(stream)), "st24_selftest_wait_timeout")


def st24_device_status(stream=None) -> int:
    return load().st24_device_status(_stream(stream))


# ---- conveniences (allocation through torch; compute still in the library) ----

def compress(W: torch.Tensor, *, stream=None):
    """(values, meta) of W [M, K] on W's device."""
    M, K = W.shape
    values = torch.empty((M, K // 2), dtype=W.dtype, device=W.device)
    meta = torch.empty((M, (K // 4 + 1) // 2), dtype=torch.uint8, device=W.device)
    st24_prune_compress(W, values, meta, stream=stream)
    return values, meta


def compress_nm(W: torch.Tensor, n: int, m: int, *, stream=None):
    """(values, meta) of W [M, K] pruned n:m, in the 2:4 compressed form."""
    M, K = W.shape
    values = torch.empty((M, K // 2), dtype=W.dtype, device=W.device)
    meta = torch.empty((M, (K // 4 + 1) // 2), dtype=torch.uint8, device=W.device)
    st24_prune_compress_nm(W, values, meta, n, m, stream=stream)
    return values, meta


def compress_nm2(W: torch.Tensor, n: int, m: int, *, stream=None):
    """(values [M, K], meta [M, 2 * ceil(K/8)]): the two 2:4 forms of W's n:m pruning."""
    M, K = W.shape
    values = torch.empty((M, K), dtype=W.dtype, device=W.device)
    meta = torch.empty((M, 2 * ((K // 4 + 1) // 2)), dtype=torch.uint8, device=W.device)
    st24_prune_compress_nm2(W, values, meta, n, m, stream=stream)
    return values, meta


def quantize_compress(W: torch.Tensor, dtype=torch.float8_e4m3fn, *, stream=None):
    """(values, meta, scales) of W [M, K] quantised per row to ``dtype`` (float8_e4m3fn or int8)."""
    M, K = W.shape
    values = torch.empty((M, K // 2), dtype=dtype, device=W.device)
    meta = torch.empty((M, (K // 4 + 1) // 2), dtype=torch.uint8, device=W.device)
    scales = torch.empty(M, dtype=torch.float32, device=W.device)
    st24_quantize_prune_compress(W, values, meta, scales, stream=stream)
    return values, meta, scales


class Workspace:
    """A zero-filled workspace per (device, size), reused across calls on one stream."""

    def __init__(self):
        self._bufs = {}

    def get(self, nbytes: int, device) -> torch.Tensor | None:
        if nbytes == 0:
            return None
        key = (str(device),)
        buf = self._bufs.get(key)
        if buf is None or buf.numel() < nbytes:
            buf = torch.zeros(nbytes, dtype=torch.uint8, device=device)
            self._bufs[key] = buf
        return buf


_default_ws = Workspace()


def spmm(values: torch.Tensor, meta: torch.Tensor, X: torch.Tensor, *, out_dtype=torch.bfloat16,
         alpha: float = 1.0, beta: float = 0.0, C: torch.Tensor | None = None,
         row_scale: torch.Tensor | None = None, workspace: Workspace | None = None, stream=None):
    """Y[N, M] = alpha * row_scale * (A_sparse @ X.T).T + beta * C."""
    M = values.shape[0]
    N, K = X.shape
    if C is not None:
        Y = C
    else:
        Y = torch.empty((N, M), dtype=out_dtype, device=X.device)
    ws = (workspace or _default_ws).get(st24_spmm_workspace_bytes(X.dtype, Y.dtype, M, N, K), X.device)
    st24_spmm(values, meta, X, Y, K=K, alpha=alpha, beta=beta, row_scale=row_scale, workspace=ws,
              M=M, stream=stream)
    return Y
