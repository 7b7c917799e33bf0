// st24_epilogue.cuh -- the SpMM output stage shared by the kernels:
// out(m, n) = round(alpha * row_scale[m] * acc + beta * C(m, n)), with C
// element (m, n) at C[n*ldc + m].  The fp32 operations are done in this fixed
// order without contraction, so every kernel rounds the same way.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "st24_device.cuh"
#include "st24_schedule.cuh"

namespace st24 {

struct OutParams {
  int64_t M, N;
  float alpha, beta;
  void* C;
  int64_t ldc;
  int c_type;
  const float* row_scale;
};

__device__ __forceinline__ float load_c(const OutParams& p, int64_t idx) {
  switch (p.c_type) {
    case kF32: return static_cast<const float*>(p.C)[idx];
    case kBF16: return __bfloat162float(static_cast<const __nv_bfloat16*>(p.C)[idx]);
    default: return __half2float(static_cast<const __half*>(p.C)[idx]);
  }
}

// Row factor alpha * row_scale[m] (alpha when there is no scale).
__device__ __forceinline__ float row_factor(const OutParams& p, int64_t m) {
  return p.row_scale ? __fmul_rn(p.alpha, p.row_scale[m]) : p.alpha;
}

// beta * C(m, n) as read before any output of the chunk is written (0 when
// beta == 0: C is not read).  Load a chunk's inputs first, then store the
// chunk: C is read and written through the same pointer, so a load placed
// after a store to C has to wait for it.
__device__ __forceinline__ float load_beta_c(const OutParams& p, int64_t m, int64_t n) {
  return p.beta != 0.0f ? __fmul_rn(p.beta, load_c(p, n * p.ldc + m)) : 0.0f;
}

// The same, with the output type a compile-time constant: no per-element
// branch on the type, so a chunk's loads issue back to back as predicated
// instructions and their latencies overlap.
template <int CT>
__device__ __forceinline__ float c_load(const void* C, int64_t idx) {
  if constexpr (CT == kF32) return static_cast<const float*>(C)[idx];
  else if constexpr (CT == kBF16) return __bfloat162float(static_cast<const __nv_bfloat16*>(C)[idx]);
  else return __half2float(static_cast<const __half*>(C)[idx]);
}

template <int CT>
__device__ __forceinline__ void c_store(void* C, int64_t idx, float r) {
  if constexpr (CT == kF32) static_cast<float*>(C)[idx] = r;
  else if constexpr (CT == kBF16) static_cast<__nv_bfloat16*>(C)[idx] = __float2bfloat16_rn(r);
  else static_cast<__half*>(C)[idx] = __float2half_rn(r);
}

// Calls f(std::integral_constant<int, CT>) for the floating-point output
// type p.c_type (the branch is taken once, outside the caller's loops).
template <typename F>
__device__ __forceinline__ void with_float_c_type(int c_type, F&& f) {
  switch (c_type) {
    case kF32: f(std::integral_constant<int, kF32>{}); break;
    case kBF16: f(std::integral_constant<int, kBF16>{}); break;
    default: f(std::integral_constant<int, kF16>{}); break;
  }
}

// Column chunk [n0, n0 + CH) of output row m from fp32 sums v: every beta*C
// input of the chunk is loaded before any output is stored (the epilogue
// formula and rounding are those of store_out).
template <int CT, int CH>
__device__ __forceinline__ void store_row_chunk(const OutParams& p, int64_t m, int64_t n0, const float (&v)[CH],
                                                float factor) {
  float bc[CH];
  if (p.beta != 0.0f) {
#pragma unroll
    for (int j = 0; j < CH; ++j) bc[j] = (n0 + j < p.N) ? c_load<CT>(p.C, (n0 + j) * p.ldc + m) : 0.0f;
#pragma unroll
    for (int j = 0; j < CH; ++j) bc[j] = __fmul_rn(p.beta, bc[j]);
  }
#pragma unroll
  for (int j = 0; j < CH; ++j) {
    if (n0 + j < p.N) {
      float r = __fmul_rn(v[j], factor);
      if (p.beta != 0.0f) r = __fadd_rn(r, bc[j]);
      c_store<CT>(p.C, (n0 + j) * p.ldc + m, r);
    }
  }
}

template <typename Acc>
__device__ __forceinline__ void store_out(const OutParams& p, int64_t m, int64_t n, Acc acc, float factor,
                                          float beta_c) {
  const int64_t idx = n * p.ldc + m;
  if constexpr (std::is_same<Acc, int>::value) {
    if (p.c_type == kS32) {
      static_cast<int*>(p.C)[idx] = acc;
      return;
    }
  }
  float r = __fmul_rn(static_cast<float>(acc), factor);
  if (p.beta != 0.0f) r = __fadd_rn(r, beta_c);
  switch (p.c_type) {
    case kF32: static_cast<float*>(p.C)[idx] = r; break;
    case kBF16: static_cast<__nv_bfloat16*>(p.C)[idx] = __float2bfloat16_rn(r); break;
    default: static_cast<__half*>(p.C)[idx] = __float2half_rn(r); break;
  }
}

// C = beta * C over the whole M x N output (the product is empty when K == 0).
__global__ void scale_c_kernel(OutParams p);

}  // namespace st24
