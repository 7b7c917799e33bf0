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
// values and 32 or 64 contiguous bytes of metadata; four pieces per lane are
// loaded before any is used, which keeps enough bytes in flight per SM.
#include "st24_device.cuh"

namespace st24 {
namespace {

// A key whose unsigned order is the order of |x|: the sign-cleared bit
// pattern for the floating-point types (sign-magnitude encodings), with every
// NaN mapped to one value above infinity so that NaNs tie with each other;
// |x| for int8 (|-128| = 128).
template <int DT>
__device__ __forceinline__ uint32_t mag_key(uint32_t raw);
template <>
__device__ __forceinline__ uint32_t mag_key<kF16>(uint32_t raw) {
  const uint32_t k = raw & 0x7FFFu;
  return k > 0x7C00u ? 0x7C01u : k;
}
template <>
__device__ __forceinline__ uint32_t mag_key<kBF16>(uint32_t raw) {
  const uint32_t k = raw & 0x7FFFu;
  return k > 0x7F80u ? 0x7F81u : k;
}
template <>
__device__ __forceinline__ uint32_t mag_key<kE4M3>(uint32_t raw) {
  return raw & 0x7Fu;  // 0x7F is the only NaN magnitude; there is no infinity
}
template <>
__device__ __forceinline__ uint32_t mag_key<kS8>(uint32_t raw) {
  const int v = static_cast<int>(static_cast<int8_t>(raw & 0xFFu));
  return static_cast<uint32_t>(v < 0 ? -v : v);
}

// Element i of a group outranks element j when its key is larger, or equal
// with i < j.  With c_ij = (k_i >= k_j) for i < j, element i is kept when it is
// outranked by fewer than two others, i.e. when a majority of its three
// comparisons go its way:
//   keep0 = maj(c01, c02, c03)      keep1 = maj(!c01, c12, c13)
//   keep2 = maj(!c02, !c12, c23)    keep3 = maj(!c03, !c13, !c23)
// Exactly two of the four are kept (the relation is a strict total order).
// Returns the nibble i0 | i1 << 2 of the kept pair and its two raw values.
template <int DT>
__device__ __forceinline__ uint32_t compress_group(const uint32_t (&e)[4], uint32_t& v0,
                                                   uint32_t& v1) {
  const uint32_t k0 = mag_key<DT>(e[0]), k1 = mag_key<DT>(e[1]), k2 = mag_key<DT>(e[2]),
                 k3 = mag_key<DT>(e[3]);
  const bool c01 = k0 >= k1, c02 = k0 >= k2, c03 = k0 >= k3;
  const bool c12 = k1 >= k2, c13 = k1 >= k3, c23 = k2 >= k3;
  const bool keep0 = (c01 & c02) | (c01 & c03) | (c02 & c03);
  const bool keep1 = (!c01 & c12) | (!c01 & c13) | (c12 & c13);
  const bool keep2 = (!c02 & !c12) | (!c02 & c23) | (!c12 & c23);
  const bool keep3 = (!c03 & !c13) | (!c03 & !c23) | (!c13 & !c23);
  const uint32_t i0 = keep0 ? 0u : (keep1 ? 1u : 2u);
  const uint32_t i1 = keep3 ? 3u : (keep2 ? 2u : 1u);
  v0 = keep0 ? e[0] : (keep1 ? e[1] : e[2]);
  v1 = keep3 ? e[3] : (keep2 ? e[2] : e[1]);
  return i0 | (i1 << 2);
}

// The 4 raw elements of a group rebuilt from its two values and nibble.
__device__ __forceinline__ void expand_group(uint32_t v0, uint32_t v1, uint32_t nib,
                                             uint32_t (&e)[4]) {
  const uint32_t i0 = nib & 3u, i1 = (nib >> 2) & 3u;
#pragma unroll
  for (uint32_t i = 0; i < 4; ++i) e[i] = (i == i0) ? v0 : ((i == i1) ? v1 : 0u);
}

// ---- one 16-byte piece of input ----------------------------------------------
// 16-bit types: 8 elements = 2 groups -> 8 bytes of values, 1 metadata byte.
// 8-bit types: 16 elements = 4 groups -> 8 bytes of values, 2 metadata bytes.
template <int DT, int ES>
__device__ __forceinline__ uint2 compress_piece(const uint4 in, uint32_t& meta_bits) {
  const uint32_t w[4] = {in.x, in.y, in.z, in.w};
  uint32_t out[2];
  meta_bits = 0;
  if constexpr (ES == 2) {
#pragma unroll
    for (int g = 0; g < 2; ++g) {
      const uint32_t e[4] = {w[2 * g] & 0xFFFFu, w[2 * g] >> 16, w[2 * g + 1] & 0xFFFFu,
                             w[2 * g + 1] >> 16};
      uint32_t v0, v1;
      meta_bits |= compress_group<DT>(e, v0, v1) << (4 * g);
      out[g] = v0 | (v1 << 16);
    }
  } else {
    uint32_t pair[4];
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const uint32_t e[4] = {w[g] & 0xFFu, (w[g] >> 8) & 0xFFu, (w[g] >> 16) & 0xFFu, w[g] >> 24};
      uint32_t v0, v1;
      meta_bits |= compress_group<DT>(e, v0, v1) << (4 * g);
      pair[g] = v0 | (v1 << 8);
    }
    out[0] = pair[0] | (pair[1] << 16);
    out[1] = pair[2] | (pair[3] << 16);
  }
  return make_uint2(out[0], out[1]);
}

template <int ES>
__device__ __forceinline__ uint4 expand_piece(const uint2 vals, uint32_t meta_bits) {
  uint32_t w[4];
  if constexpr (ES == 2) {
    const uint32_t v[2] = {vals.x, vals.y};
#pragma unroll
    for (int g = 0; g < 2; ++g) {
      uint32_t e[4];
      expand_group(v[g] & 0xFFFFu, v[g] >> 16, (meta_bits >> (4 * g)) & 0xFu, e);
      w[2 * g] = e[0] | (e[1] << 16);
      w[2 * g + 1] = e[2] | (e[3] << 16);
    }
  } else {
    const uint32_t pairs[4] = {vals.x & 0xFFFFu, vals.x >> 16, vals.y & 0xFFFFu, vals.y >> 16};
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      uint32_t e[4];
      expand_group(pairs[g] & 0xFFu, pairs[g] >> 8, (meta_bits >> (4 * g)) & 0xFu, e);
      w[g] = e[0] | (e[1] << 8) | (e[2] << 16) | (e[3] << 24);
    }
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

constexpr int kThreads = 256;
constexpr int kPiecesPerLane = 4;
constexpr int kWarpSpan = 32 * kPiecesPerLane;  // pieces one warp handles per iteration

// Fast path.  The matrix is a sequence of 16-byte pieces, `ppr` per row; warp
// w handles pieces [w*128, w*128+128) of each grid-stride round, lane l the
// pieces l, l+32, l+64 and l+96 of that span.  A lane divides once per round
// (Idx is 32-bit whenever the piece count allows) and carries (row, col)
// forward for its other pieces.
template <typename Idx>
__device__ __forceinline__ void advance(Idx& row, Idx& col, Idx step, Idx ppr) {
  col += step;
  while (col >= ppr) {
    col -= ppr;
    ++row;
  }
}

template <int DT, int ES, typename Idx>
__global__ void __launch_bounds__(kThreads) prune_compress_vec(
    const uint8_t* __restrict__ W, int64_t w_row_bytes, Idx total, Idx ppr,
    uint8_t* __restrict__ values, int64_t v_row_bytes, uint8_t* __restrict__ meta,
    int64_t m_row_bytes) {
  const int lane = threadIdx.x & 31;
  const Idx warp = (static_cast<Idx>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
  const Idx nwarps = (static_cast<Idx>(gridDim.x) * kThreads) >> 5;
  for (Idx base = warp * kWarpSpan; base < total; base += nwarps * kWarpSpan) {
    uint4 in[kPiecesPerLane];
    Idx row[kPiecesPerLane], col[kPiecesPerLane];
    Idx r = (base + lane) / ppr, c = base + lane - r * ppr;
#pragma unroll
    for (int i = 0; i < kPiecesPerLane; ++i) {
      row[i] = r;
      col[i] = c;
      if (base + i * 32 + lane < total)
        in[i] = __ldcs(reinterpret_cast<const uint4*>(W + static_cast<int64_t>(r) * w_row_bytes +
                                                      static_cast<int64_t>(c) * 16));
      advance<Idx>(r, c, 32, ppr);
    }
#pragma unroll
    for (int i = 0; i < kPiecesPerLane; ++i) {
      if (base + i * 32 + lane >= total) break;
      uint32_t mb;
      const uint2 v = compress_piece<DT, ES>(in[i], mb);
      const int64_t rr = row[i], cc = col[i];
      *reinterpret_cast<uint2*>(values + rr * v_row_bytes + cc * 8) = v;
      if constexpr (ES == 2)
        meta[rr * m_row_bytes + cc] = static_cast<uint8_t>(mb);
      else
        *reinterpret_cast<uint16_t*>(meta + rr * m_row_bytes + cc * 2) = static_cast<uint16_t>(mb);
    }
  }
}

template <int ES, typename Idx>
__global__ void __launch_bounds__(kThreads) decompress_vec(
    const uint8_t* __restrict__ values, int64_t v_row_bytes, const uint8_t* __restrict__ meta,
    int64_t m_row_bytes, Idx total, Idx ppr, uint8_t* __restrict__ W, int64_t w_row_bytes) {
  const int lane = threadIdx.x & 31;
  const Idx warp = (static_cast<Idx>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
  const Idx nwarps = (static_cast<Idx>(gridDim.x) * kThreads) >> 5;
  for (Idx base = warp * kWarpSpan; base < total; base += nwarps * kWarpSpan) {
    uint2 v[kPiecesPerLane];
    uint32_t mb[kPiecesPerLane];
    Idx row[kPiecesPerLane], col[kPiecesPerLane];
    Idx r = (base + lane) / ppr, c = base + lane - r * ppr;
#pragma unroll
    for (int i = 0; i < kPiecesPerLane; ++i) {
      row[i] = r;
      col[i] = c;
      if (base + i * 32 + lane < total) {
        const int64_t rr = r, cc = c;
        v[i] = __ldcs(reinterpret_cast<const uint2*>(values + rr * v_row_bytes + cc * 8));
        if constexpr (ES == 2)
          mb[i] = __ldcs(meta + rr * m_row_bytes + cc);
        else
          mb[i] = __ldcs(reinterpret_cast<const uint16_t*>(meta + rr * m_row_bytes + cc * 2));
      }
      advance<Idx>(r, c, 32, ppr);
    }
#pragma unroll
    for (int i = 0; i < kPiecesPerLane; ++i) {
      if (base + i * 32 + lane >= total) break;
      const int64_t rr = row[i], cc = col[i];
      *reinterpret_cast<uint4*>(W + rr * w_row_bytes + cc * 16) = expand_piece<ES>(v[i], mb[i]);
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

bool aligned(const void* p, int a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Blocks that stay resident on one SM for kernel `k` (queried once per kernel).
template <typename Kernel>
int resident_blocks(Kernel k) {
  static int blocks = 0;
  if (blocks == 0) {
    int b = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, k, kThreads, 0) != cudaSuccess || b <= 0) b = 1;
    blocks = b;
  }
  return blocks;
}

// A grid of at most one resident wave: every block stays on the GPU for the
// whole launch and grid-strides over the work.
template <typename Kernel>
int grid_for(Kernel k, int64_t work_items, int items_per_block, int num_sms) {
  const int64_t want = (work_items + items_per_block - 1) / items_per_block;
  const int64_t cap = static_cast<int64_t>(num_sms) * resident_blocks(k);
  return static_cast<int>(want < cap ? (want > 0 ? want : 1) : cap);
}

// 32-bit piece indices whenever the last grid-stride round cannot overflow them.
inline bool fits_u32(int64_t total) { return total + (int64_t(1) << 26) < (int64_t(1) << 32); }

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
          w, ldw * ES, static_cast<uint32_t>(total), static_cast<uint32_t>(ppr), v, (K / 2) * ES, e,
          meta_row_bytes(K));
    } else {
      auto k = prune_compress_vec<DT, ES, int64_t>;
      k<<<grid_for(k, total, kThreads / 32 * kWarpSpan, num_sms), kThreads, 0, s>>>(
          w, ldw * ES, total, ppr, v, (K / 2) * ES, e, meta_row_bytes(K));
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
          v, (K / 2) * ES, e, meta_row_bytes(K), static_cast<uint32_t>(total), static_cast<uint32_t>(ppr), w,
          ldw * ES);
    } else {
      auto k = decompress_vec<ES, int64_t>;
      k<<<grid_for(k, total, kThreads / 32 * kWarpSpan, num_sms), kThreads, 0, s>>>(
          v, (K / 2) * ES, e, meta_row_bytes(K), total, ppr, w, ldw * ES);
    }
  } else {
    auto k = decompress_any<ES>;
    k<<<grid_for(k, M * meta_row_bytes(K), kThreads, num_sms), kThreads, 0, s>>>(
        static_cast<const uint8_t*>(values), static_cast<const uint8_t*>(meta), M, K, static_cast<uint8_t*>(W), ldw);
  }
}

bool fast_layout(int es, int64_t K, int64_t ldw, const void* W, const void* values,
                 const void* meta) {
  return (K * es) % 16 == 0 && (ldw * es) % 16 == 0 && aligned(W, 16) && aligned(values, 8) &&
         aligned(meta, es == 1 ? 2 : 1);
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
