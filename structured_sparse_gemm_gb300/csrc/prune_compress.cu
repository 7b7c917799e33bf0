// prune_compress.cu -- 2:4 magnitude prune + compress, and its inverse.
//
// Method ("Chapter 26 -- Sparsity: The Hardware View", sections "2:4
// Fine-Grained Structured Sparsity" and "Python: Build a 2:4 Mask, Compress
// It, ..."): in every group of 4 consecutive elements along K keep the two of
// largest magnitude, store their values in ascending position order and their
// two 2-bit in-group indices as metadata.
//
// Both directions are pure data movement, bound by HBM bandwidth.  The fast
// kernel gives every lane 16-byte pieces of the input such that each warp
// instruction reads 512 contiguous bytes and writes 256 contiguous bytes of
// values and 32 or 64 contiguous bytes of metadata; both pieces of a lane are
// loaded before either is used, and the kernel fits 32 registers so that 64
// warps per SM keep enough bytes in flight.  The N:M patterns are in
// prune_nm.cuh.
#include "prune_common.cuh"

#include <cuda_fp16.h>
#include <cuda_fp8.h>

namespace st24 {
using namespace prune;
namespace {

// Fast path.  The matrix is a sequence of 16-byte pieces, `ppr` per row; warp
// w handles pieces [w*64, w*64+64) of each grid-stride round, lane l the
// pieces l and l+32 of that span.  Piece p (counted row by row)
// owns bytes [8p, 8p+8) of the values and its metadata at p * (16 / ES / 8)
// bytes, since both outputs are dense; only the input may have a row stride.
// Where it has one, a lane divides once per round (Idx is 32-bit whenever the
// piece count allows) and carries (row, col) forward for its other pieces.
template <int DT, int ES, typename Idx>
__global__ void __launch_bounds__(kThreads) prune_compress_vec(
    const uint8_t* __restrict__ W, int64_t w_row_bytes, Idx total, Idx ppr,
    uint8_t* __restrict__ values, uint8_t* __restrict__ meta) {
  const int lane = threadIdx.x & 31;
  const Idx warp = (static_cast<Idx>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
  const Idx nwarps = (static_cast<Idx>(gridDim.x) * kThreads) >> 5;
  const bool dense = w_row_bytes == static_cast<int64_t>(ppr) * 16;
  for (Idx base = warp * kWarpSpan; base < total; base += nwarps * kWarpSpan) {
    uint4 in[kPiecesPerLane];
    if (dense) {
#pragma unroll
      for (int i = 0; i < kPiecesPerLane; ++i) {
        const Idx q = base + i * 32 + lane;
        if (q < total) in[i] = __ldcs(reinterpret_cast<const uint4*>(W) + q);
      }
    } else {
      Idx r = (base + lane) / ppr, c = base + lane - r * ppr;
#pragma unroll
      for (int i = 0; i < kPiecesPerLane; ++i) {
        if (base + i * 32 + lane < total)
          in[i] = __ldcs(reinterpret_cast<const uint4*>(W + static_cast<int64_t>(r) * w_row_bytes) + c);
        advance<Idx>(r, c, 32, ppr);
      }
    }
#pragma unroll
    for (int i = 0; i < kPiecesPerLane; ++i) {
      const Idx q = base + i * 32 + lane;
      if (q >= total) break;
      uint32_t mb;
      uint2 v;
      if (!compress_piece_lanes<DT, ES>(in[i], v, mb)) v = compress_piece<DT, ES>(in[i], mb);
      reinterpret_cast<uint2*>(values)[q] = v;
      if constexpr (ES == 2)
        meta[q] = static_cast<uint8_t>(mb);
      else
        reinterpret_cast<uint16_t*>(meta)[q] = static_cast<uint16_t>(mb);
    }
  }
}

template <int ES, typename Idx>
__global__ void __launch_bounds__(kThreads) decompress_vec(
    const uint8_t* __restrict__ values, const uint8_t* __restrict__ meta, Idx total, Idx ppr,
    uint8_t* __restrict__ W, int64_t w_row_bytes) {
  const int lane = threadIdx.x & 31;
  const Idx warp = (static_cast<Idx>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
  const Idx nwarps = (static_cast<Idx>(gridDim.x) * kThreads) >> 5;
  const bool dense = w_row_bytes == static_cast<int64_t>(ppr) * 16;
  for (Idx base = warp * kWarpSpan; base < total; base += nwarps * kWarpSpan) {
    uint2 v[kPiecesPerLane];
    uint32_t mb[kPiecesPerLane];
#pragma unroll
    for (int i = 0; i < kPiecesPerLane; ++i) {
      const Idx q = base + i * 32 + lane;
      if (q < total) {
        v[i] = __ldcs(reinterpret_cast<const uint2*>(values) + q);
        if constexpr (ES == 2)
          mb[i] = __ldcs(meta + q);
        else
          mb[i] = __ldcs(reinterpret_cast<const uint16_t*>(meta) + q);
      }
    }
    Idx r = 0, c = 0;
    if (!dense) {
      r = (base + lane) / ppr;
      c = base + lane - r * ppr;
    }
#pragma unroll
    for (int i = 0; i < kPiecesPerLane; ++i) {
      const Idx q = base + i * 32 + lane;
      if (q >= total) break;
      uint4* dst = dense ? reinterpret_cast<uint4*>(W) + q
                         : reinterpret_cast<uint4*>(W + static_cast<int64_t>(r) * w_row_bytes) + c;
      *dst = expand_piece<ES>(v[i], mb[i]);
      if (!dense) advance<Idx>(r, c, 32, ppr);
    }
  }
}

// ---- general path: any K % 4 == 0, any strides and alignments --------------
// One thread per metadata byte (two groups, or one for the last byte of a row
// when K % 8 == 4).
template <int ES>
__device__ __forceinline__ uint32_t load_raw(const uint8_t* p) {
  if constexpr (ES == 2) {
    return static_cast<uint32_t>(p[0]) | (static_cast<uint32_t>(p[1]) << 8);
  } else {
    return p[0];
  }
}

template <int ES>
__device__ __forceinline__ void store_raw(uint8_t* p, uint32_t v) {
  p[0] = static_cast<uint8_t>(v);
  if constexpr (ES == 2) p[1] = static_cast<uint8_t>(v >> 8);
}

template <int DT, int ES>
__global__ void __launch_bounds__(kThreads) prune_compress_any(
    const uint8_t* __restrict__ W, int64_t ldw, int64_t M, int64_t K, uint8_t* __restrict__ values,
    uint8_t* __restrict__ meta) {
  const int64_t groups = K / 4, mrb = meta_row_bytes(K);
  const int64_t total = M * mrb;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; t < total;
       t += static_cast<int64_t>(gridDim.x) * kThreads) {
    const int64_t m = t / mrb, b = t - m * mrb;
    uint32_t byte = 0;
    for (int h = 0; h < 2; ++h) {
      const int64_t g = 2 * b + h;
      if (g >= groups) break;
      uint32_t e[4];
      for (int i = 0; i < 4; ++i) e[i] = load_raw<ES>(W + (m * ldw + 4 * g + i) * ES);
      uint32_t v0, v1;
      byte |= compress_group<DT>(e, v0, v1) << (4 * h);
      store_raw<ES>(values + (m * (K / 2) + 2 * g) * ES, v0);
      store_raw<ES>(values + (m * (K / 2) + 2 * g + 1) * ES, v1);
    }
    meta[m * mrb + b] = static_cast<uint8_t>(byte);
  }
}

template <int ES>
__global__ void __launch_bounds__(kThreads) decompress_any(
    const uint8_t* __restrict__ values, const uint8_t* __restrict__ meta, int64_t M, int64_t K,
    uint8_t* __restrict__ W, int64_t ldw) {
  const int64_t groups = K / 4, mrb = meta_row_bytes(K);
  const int64_t total = M * mrb;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; t < total;
       t += static_cast<int64_t>(gridDim.x) * kThreads) {
    const int64_t m = t / mrb, b = t - m * mrb;
    const uint32_t byte = meta[m * mrb + b];
    for (int h = 0; h < 2; ++h) {
      const int64_t g = 2 * b + h;
      if (g >= groups) break;
      const uint32_t v0 = load_raw<ES>(values + (m * (K / 2) + 2 * g) * ES);
      const uint32_t v1 = load_raw<ES>(values + (m * (K / 2) + 2 * g + 1) * ES);
      uint32_t e[4];
      expand_group(v0, v1, (byte >> (4 * h)) & 0xFu, e);
      for (int i = 0; i < 4; ++i) store_raw<ES>(W + (m * ldw + 4 * g + i) * ES, e[i]);
    }
  }
}


// ---- quantise to 8 bits, then prune and compress --------------------------
// Per row of a 16-bit weight: amax = max |w|; inv = Q / amax and every
// scaled value w * inv in fp32 (round to nearest, no contraction); the codes
// are e4m3 (nearest-even, saturated to +-448) or int8 (nearest-even, clamped
// to [-127, 127]); scale = amax / Q; a zero row gets scale 0 and zero codes.
// ("Chapter 26 -- Sparsity: The Hardware View", section "Sparsity +
// Quantization Combine": 2:4 sparsity and 8-bit weights stack.)  The codes
// of each 16-value piece are then pruned and compressed like an 8-bit
// weight's.  One CTA per row (grid-stride over rows): when the row fits in
// registers (K <= 256 threads x QP pieces x 16, QP = 1, 2 or 4: the fewest
// that hold it, so short rows keep the register count and occupancy up), it
// is read once.

template <int ST>
__device__ __forceinline__ float to_f32(uint32_t bits16) {
  if constexpr (ST == kBF16) return __uint_as_float(bits16 << 16);
  else return __half2float(__ushort_as_half(static_cast<unsigned short>(bits16)));
}

// |w| of 8 16-bit values (exact).
template <int ST>
__device__ __forceinline__ float absmax8(const uint4 v, float m) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    m = fmaxf(m, fabsf(to_f32<ST>(w[i] & 0xFFFFu)));
    m = fmaxf(m, fabsf(to_f32<ST>(w[i] >> 16)));
  }
  return m;
}

// The 16 codes (byte j = value j) of a piece of 16 values given as two uint4.
template <int ST, int DT>
__device__ __forceinline__ uint4 quantize16(const uint4 lo, const uint4 hi, float inv) {
  const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
  uint32_t out[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t word = 0;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t pair = w[2 * i + h];
      const float y0 = __fmul_rn(to_f32<ST>(pair & 0xFFFFu), inv);
      const float y1 = __fmul_rn(to_f32<ST>(pair >> 16), inv);
      uint32_t two;
      if constexpr (DT == kE4M3) {
        two = __nv_cvt_float2_to_fp8x2(make_float2(y0, y1), __NV_SATFINITE, __NV_E4M3);
      } else {
        const int q0 = min(127, max(-127, __float2int_rn(y0)));
        const int q1 = min(127, max(-127, __float2int_rn(y1)));
        two = (static_cast<uint32_t>(q0) & 0xFFu) | ((static_cast<uint32_t>(q1) & 0xFFu) << 8);
      }
      word |= (two & 0xFFFFu) << (16 * h);
    }
    out[i] = word;
  }
  return make_uint4(out[0], out[1], out[2], out[3]);
}

template <int ST, int DT, int QP>
__global__ void __launch_bounds__(kThreads) quantize_prune_compress_rows(
    const uint8_t* __restrict__ W, int64_t w_row_bytes, int64_t M, int64_t K, uint8_t* __restrict__ values,
    uint8_t* __restrict__ meta, float* __restrict__ scales) {
  __shared__ float red[kThreads / 32];
  const int64_t P = K / 16;   // pieces per row
  const float Q = DT == kE4M3 ? 448.0f : 127.0f;
  for (int64_t m = blockIdx.x; m < M; m += gridDim.x) {
    const uint8_t* row = W + m * w_row_bytes;
    constexpr bool FITS = QP > 0;
    uint4 held[FITS ? QP : 1][2];
    float amax = 0.0f;
    if constexpr (FITS) {
#pragma unroll
      for (int i = 0; i < QP; ++i) {
        const int64_t pc = threadIdx.x + static_cast<int64_t>(i) * kThreads;
        if (pc < P) {
          held[i][0] = __ldcs(reinterpret_cast<const uint4*>(row + pc * 32));
          held[i][1] = __ldcs(reinterpret_cast<const uint4*>(row + pc * 32 + 16));
        }
      }
#pragma unroll
      for (int i = 0; i < QP; ++i)
        if (threadIdx.x + static_cast<int64_t>(i) * kThreads < P)
          amax = absmax8<ST>(held[i][1], absmax8<ST>(held[i][0], amax));
    } else {
      for (int64_t pc = threadIdx.x; pc < P; pc += kThreads) {
        const uint4 lo = __ldcg(reinterpret_cast<const uint4*>(row + pc * 32));
        const uint4 hi = __ldcg(reinterpret_cast<const uint4*>(row + pc * 32 + 16));
        amax = absmax8<ST>(hi, absmax8<ST>(lo, amax));
      }
    }
    // the row's absolute maximum, in every thread
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kThreads / 32; ++i) amax = fmaxf(amax, red[i]);
    const float inv = amax > 0.0f ? __fdiv_rn(Q, amax) : 0.0f;
    if (threadIdx.x == 0) scales[m] = amax > 0.0f ? __fdiv_rn(amax, Q) : 0.0f;
    uint8_t* vrow = values + m * (K / 2);
    uint8_t* erow = meta + m * (K / 8);
    auto emit = [&](int64_t pc, const uint4 lo, const uint4 hi) {
      const uint4 codes = quantize16<ST, DT>(lo, hi, inv);
      uint2 v;
      uint32_t mb;
      if (!compress_piece_lanes<DT, 1>(codes, v, mb)) v = compress_piece<DT, 1>(codes, mb);
      *reinterpret_cast<uint2*>(vrow + pc * 8) = v;
      *reinterpret_cast<uint16_t*>(erow + pc * 2) = static_cast<uint16_t>(mb);
    };
    if constexpr (FITS) {
#pragma unroll
      for (int i = 0; i < QP; ++i) {
        const int64_t pc = threadIdx.x + static_cast<int64_t>(i) * kThreads;
        if (pc < P) emit(pc, held[i][0], held[i][1]);
      }
    } else {
      for (int64_t pc = threadIdx.x; pc < P; pc += kThreads)
        emit(pc, __ldcs(reinterpret_cast<const uint4*>(row + pc * 32)),
             __ldcs(reinterpret_cast<const uint4*>(row + pc * 32 + 16)));
    }
    __syncthreads();   // red[] is reused by the next row
  }
}

template <int DT, int ES>
void launch_pc(const void* W, int64_t M, int64_t K, int64_t ldw, void* values, void* meta,
               int num_sms, bool fast, cudaStream_t s) {
  if (fast) {
    const int64_t ppr = K * ES / 16, total = M * ppr;
    const auto* w = static_cast<const uint8_t*>(W);
    auto* v = static_cast<uint8_t*>(values);
    auto* e = static_cast<uint8_t*>(meta);
    if (fits_u32(total)) {
      auto k = prune_compress_vec<DT, ES, uint32_t>;
      k<<<grid_for(k, total, kThreads / 32 * kWarpSpan, num_sms), kThreads, 0, s>>>(
          w, ldw * ES, static_cast<uint32_t>(total), static_cast<uint32_t>(ppr), v, e);
    } else {
      auto k = prune_compress_vec<DT, ES, int64_t>;
      k<<<grid_for(k, total, kThreads / 32 * kWarpSpan, num_sms), kThreads, 0, s>>>(
          w, ldw * ES, total, ppr, v, e);
    }
  } else {
    auto k = prune_compress_any<DT, ES>;
    k<<<grid_for(k, M * meta_row_bytes(K), kThreads, num_sms), kThreads, 0, s>>>(
        static_cast<const uint8_t*>(W), ldw, M, K, static_cast<uint8_t*>(values), static_cast<uint8_t*>(meta));
  }
}

template <int ES>
void launch_dc(const void* values, const void* meta, int64_t M, int64_t K, void* W, int64_t ldw,
               int num_sms, bool fast, cudaStream_t s) {
  if (fast) {
    const int64_t ppr = K * ES / 16, total = M * ppr;
    const auto* v = static_cast<const uint8_t*>(values);
    const auto* e = static_cast<const uint8_t*>(meta);
    auto* w = static_cast<uint8_t*>(W);
    if (fits_u32(total)) {
      auto k = decompress_vec<ES, uint32_t>;
      k<<<grid_for(k, total, kThreads / 32 * kWarpSpan, num_sms), kThreads, 0, s>>>(
          v, e, static_cast<uint32_t>(total), static_cast<uint32_t>(ppr), w, ldw * ES);
    } else {
      auto k = decompress_vec<ES, int64_t>;
      k<<<grid_for(k, total, kThreads / 32 * kWarpSpan, num_sms), kThreads, 0, s>>>(
          v, e, total, ppr, w, ldw * ES);
    }
  } else {
    auto k = decompress_any<ES>;
    k<<<grid_for(k, M * meta_row_bytes(K), kThreads, num_sms), kThreads, 0, s>>>(
        static_cast<const uint8_t*>(values), static_cast<const uint8_t*>(meta), M, K, static_cast<uint8_t*>(W), ldw);
  }
}

}  // namespace

st24_status launch_prune_compress(int dt, const void* W, int64_t M, int64_t K, int64_t ldw,
                                  void* values, void* meta, cudaStream_t stream) {
  const DeviceInfo* dev = current_device_info();
  if (!dev) return ST24_ERR_CUDA;
  const bool fast = fast_layout(elem_size(dt), K, ldw, W, values, meta);
  switch (dt) {
    case kF16: launch_pc<kF16, 2>(W, M, K, ldw, values, meta, dev->num_sms, fast, stream); break;
    case kBF16: launch_pc<kBF16, 2>(W, M, K, ldw, values, meta, dev->num_sms, fast, stream); break;
    case kE4M3: launch_pc<kE4M3, 1>(W, M, K, ldw, values, meta, dev->num_sms, fast, stream); break;
    case kS8: launch_pc<kS8, 1>(W, M, K, ldw, values, meta, dev->num_sms, fast, stream); break;
    default: return ST24_ERR_UNSUPPORTED;
  }
  return cudaGetLastError() == cudaSuccess ? ST24_OK : ST24_ERR_CUDA;
}

st24_status launch_quantize_prune_compress(int src, int dst, const void* W, int64_t M, int64_t K, int64_t ldw,
                                           void* values, void* meta, float* scales, cudaStream_t stream) {
  const DeviceInfo* dev = current_device_info();
  if (!dev) return ST24_ERR_CUDA;
  const int64_t per_piece = static_cast<int64_t>(kThreads) * 16;   // K covered by one piece per thread
  const int qp = K <= per_piece ? 1 : K <= 2 * per_piece ? 2 : K <= 4 * per_piece ? 4 : 0;
  const auto* w = static_cast<const uint8_t*>(W);
  auto* v = static_cast<uint8_t*>(values);
  auto* e = static_cast<uint8_t*>(meta);
  auto go = [&](auto kern) {
    const int64_t cap = static_cast<int64_t>(dev->num_sms) * resident_blocks(kern);
    const int grid = static_cast<int>(M < cap ? M : cap);
    kern<<<grid, kThreads, 0, stream>>>(w, ldw * 2, M, K, v, e, scales);
  };
#define ST24_QPC(S, D)                                                          \
  if (src == S && dst == D) {                                                  \
    if (qp == 1) go(quantize_prune_compress_rows<S, D, 1>);                    \
    else if (qp == 2) go(quantize_prune_compress_rows<S, D, 2>);               \
    else if (qp == 4) go(quantize_prune_compress_rows<S, D, 4>);               \
    else go(quantize_prune_compress_rows<S, D, 0>);                            \
  }
  ST24_QPC(kBF16, kE4M3) else ST24_QPC(kBF16, kS8) else ST24_QPC(kF16, kE4M3) else ST24_QPC(kF16, kS8) else
    return ST24_ERR_UNSUPPORTED;
#undef ST24_QPC
  return cudaGetLastError() == cudaSuccess ? ST24_OK : ST24_ERR_CUDA;
}

st24_status launch_decompress(int dt, const void* values, const void* meta, int64_t M, int64_t K,
                              void* W, int64_t ldw, cudaStream_t stream) {
  const DeviceInfo* dev = current_device_info();
  if (!dev) return ST24_ERR_CUDA;
  const int es = elem_size(dt);
  const bool fast = fast_layout(es, K, ldw, W, values, meta);
  if (es == 2)
    launch_dc<2>(values, meta, M, K, W, ldw, dev->num_sms, fast, stream);
  else if (es == 1)
    launch_dc<1>(values, meta, M, K, W, ldw, dev->num_sms, fast, stream);
  else
    return ST24_ERR_UNSUPPORTED;
  return cudaGetLastError() == cudaSuccess ? ST24_OK : ST24_ERR_CUDA;
}

}  // namespace st24
