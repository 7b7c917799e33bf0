// spmm_t.cu -- C ABI entry of the transposed use of a compressed weight
// (st24_spmm_t): argument checks, then the per-type kernel launch.
#include "spmm_t.cuh"

using namespace st24;

extern "C" st24_status st24_spmm_t(st24_dtype ab_type, st24_dtype c_type, int64_t M, int64_t N, int64_t K,
                                   float alpha, const void* A_values, const void* A_meta, const void* B,
                                   int64_t ldb, float beta, void* C, int64_t ldc, void* stream) {
  if (M < 0 || N < 0 || K < 0 || K % 4 != 0) return ST24_ERR_INVALID_ARG;
  if (ab_type != ST24_F16 && ab_type != ST24_BF16) return ST24_ERR_UNSUPPORTED;
  if (c_type != ST24_F32 && c_type != ST24_BF16 && c_type != ST24_F16) return ST24_ERR_UNSUPPORTED;
  if (K == 0 || N == 0) return ST24_OK;
  if (!C || ldc < K) return ST24_ERR_INVALID_ARG;
  if (M > 0 && (!A_values || !A_meta || !B || ldb < M)) return ST24_ERR_INVALID_ARG;
  if (K % 128 != 0) return ST24_ERR_UNSUPPORTED;
  auto aligned = [](const void* ptr, int al) { return reinterpret_cast<uintptr_t>(ptr) % al == 0; };
  if (M > 0 && (!aligned(A_values, 16) || !aligned(A_meta, 16) || !aligned(B, 16) || (ldb * 2) % 16 != 0))
    return ST24_ERR_MISALIGNED;
  if (!aligned(C, elem_size(c_type))) return ST24_ERR_MISALIGNED;
  SpmmArgs a{};
  a.ab = ab_type;
  a.c = c_type;
  a.M = M;
  a.N = N;
  a.K = K;
  a.alpha = alpha;
  a.beta = beta;
  a.values = A_values;
  a.meta = A_meta;
  a.B = B;
  a.ldb = ldb;
  a.C = C;
  a.ldc = ldc;
  const DeviceInfo* dev = current_device_info();
  if (!dev) return ST24_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (M == 0) {   // an empty sum: dX = beta * dX
    SpmmArgs e = a;
    e.M = K;      // scale_c works on the (k, n) output
    return launch_scale_c(e, *dev, s);
  }
  return ab_type == ST24_BF16 ? spt::launch_dt<kBF16>(a, *dev, s) : spt::launch_dt<kF16>(a, *dev, s);
}
