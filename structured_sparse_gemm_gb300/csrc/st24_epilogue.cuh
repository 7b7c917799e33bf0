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

// beta * C(m, n0 + j) for the CH columns of a chunk (0 past N), loaded as
// back-to-back predicated loads.  Called before the chunk's sums are fetched,
// so the loads' latency overlaps that fetch and few registers are live.
template <int CT, int CH>
__device__ __forceinline__ void load_row_chunk_beta_c(const OutParams& p, int64_t m, int64_t n0, float (&bc)[CH]) {
#pragma unroll
  for (int j = 0; j < CH; ++j) bc[j] = (n0 + j < p.N) ? c_load<CT>(p.C, (n0 + j) * p.ldc + m) : 0.0f;
#pragma unroll
  for (int j = 0; j < CH; ++j) bc[j] = __fmul_rn(p.beta, bc[j]);
}

// Column chunk [n0, n0 + CH) of output row m from fp32 sums (given as bit
// patterns) and the chunk's beta * C inputs bc (used only when beta != 0);
// the epilogue formula and rounding are those of store_out.
template <int CT, int CH>
__device__ __forceinline__ void store_row_chunk_bits(const OutParams& p, int64_t m, int64_t n0,
                                                     const uint32_t (&acc)[CH], const float (&bc)[CH], float factor) {
  using E = typename std::conditional<CT == kF32, float,
                                      typename std::conditional<CT == kBF16, __nv_bfloat16, __half>::type>::type;
  E* out = static_cast<E*>(p.C) + n0 * p.ldc + m;   // one running pointer: few registers live
  const int64_t cols = p.N - n0;
#pragma unroll
  for (int j = 0; j < CH; ++j) {
    if (j < cols) {
      float r = __fmul_rn(__uint_as_float(acc[j]), factor);
      if (p.beta != 0.0f) r = __fadd_rn(r, bc[j]);
      if constexpr (CT == kF32) *out = r;
      else if constexpr (CT == kBF16) *out = __float2bfloat16_rn(r);
      else *out = __float2half_rn(r);
    }
    out += p.ldc;
  }
}

// beta * C for a chunk staged in shared memory as [32 columns][32 rows] of
// the output type, row `lane` (32-bit shared address of the chunk).
template <int CT, int CH>
__device__ __forceinline__ void staged_beta_c(uint32_t chunk, int lane, float beta, float (&bc)[CH]) {
#pragma unroll
  for (int j = 0; j < CH; ++j) {
    float c;
    if constexpr (CT == kF32) c = lds_f32(chunk + (j * 32 + lane) * 4);
    else if constexpr (CT == kBF16) c = __uint_as_float(lds_u16(chunk + (j * 32 + lane) * 2) << 16);
    else c = __half2float(__ushort_as_half(static_cast<unsigned short>(lds_u16(chunk + (j * 32 + lane) * 2))));
    bc[j] = __fmul_rn(beta, c);
  }
}

// Column chunk [n0, n0 + CH) of output row m from fp32 sums v: every beta*C
// input of the chunk is loaded before any output is stored.
template <int CT, int CH>
__device__ __forceinline__ void store_row_chunk(const OutParams& p, int64_t m, int64_t n0, const float (&v)[CH],
                                                float factor) {
  float bc[CH];
  if (p.beta != 0.0f) load_row_chunk_beta_c<CT, CH>(p, m, n0, bc);
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

// The contributor that finishes a split tile (stream-K): for output row m,
// sum the contributors' fp32 partial rows in k order (contributor c_lo first)
// and apply the epilogue.  Contributor c's partial tile sits at partial slot
// slot_mul * sch.slot(c, tile) + slot_add, BM x BNW floats column-major, this
// row at index row.  RCH columns at a time, up to 4 contributors' loads in
// flight together.  Not inlined: its registers stay out of the main loop's.
template <int BM, int BNW, int RCH>
__device__ __noinline__ void reduce_split_row(const OutParams& p, const float* partials, const Schedule& sch,
                                              int64_t tile, int slot_mul, int slot_add, int64_t c_lo, int64_t c_hi,
                                              int row, int64_t m, int64_t n_base, float factor) {
#pragma unroll 1
  for (int c0 = 0; c0 < BNW; c0 += RCH) {
    if (n_base + c0 >= p.N) break;
    float t[RCH];
    for (int64_t cb = c_lo; cb <= c_hi; cb += 4) {
      float v[4][RCH];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (cb + u <= c_hi) {
          const float* src = partials + (slot_mul * sch.slot(cb + u, tile) + slot_add) * (BM * BNW) + row;
#pragma unroll
          for (int j = 0; j < RCH; ++j) v[u][j] = __ldcg(src + (c0 + j) * BM);
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (cb + u <= c_hi) {
#pragma unroll
          for (int j = 0; j < RCH; ++j) t[j] = (cb + u == c_lo) ? v[u][j] : t[j] + v[u][j];
        }
      }
    }
    with_float_c_type(p.c_type, [&](auto ct) { store_row_chunk<decltype(ct)::value, RCH>(p, m, n_base + c0, t, factor); });
  }
}

// C = beta * C over the whole M x N output (the product is empty when K == 0).
__global__ void scale_c_kernel(OutParams p);

}  // namespace st24
