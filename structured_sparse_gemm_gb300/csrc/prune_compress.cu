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
// with i < j.  The kept pair is the two elements outranked by fewer than two
// others.  Returns the 4-bit keep mask (exactly two bits set).
__device__ __forceinline__ uint32_t keep_mask(uint32_t k0, uint32_t k1, uint32_t k2, uint32_t k3) {
  const uint32_t b0 = (k1 > k0) + (k2 > k0) + (k3 > k0);
  const uint32_t b1 = (k0 >= k1) + (k2 > k1) + (k3 > k1);
  const uint32_t b2 = (k0 >= k2) + (k1 >= k2) + (k3 > k2);
  const uint32_t b3 = (k0 >= k3) + (k1 >= k3) + (k2 >= k3);
  return (b0 < 2u) | ((b1 < 2u) << 1) | ((b2 < 2u) << 2) | ((b3 < 2u) << 3);
}

// One group: raw elements e[0..3] -> (v0, v1) with v0 at the lower index, and
// the metadata nibble i0 | i1 << 2.
template <int DT>
__device__ __forceinline__ uint32_t compress_group(const uint32_t (&e)[4], uint32_t& v0,
                                                   uint32_t& v1) {
  const uint32_t keep =
      keep_mask(mag_key<DT>(e[0]), mag_key<DT>(e[1]), mag_key<DT>(e[2]), mag_key<DT>(e[3]));
  const uint32_t i0 = __ffs(keep) - 1;
  const uint32_t i1 = 31 - __clz(keep);
  v0 = i0 == 0 ? e[0] : (i0 == 1 ? e[1] : e[2]);
  v1 = i1 == 3 ? e[3] : (i1 == 2 ? e[2] : e[1]);
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
// pieces l, l+32, l+64 and l+96 of that span.
template <int DT, int ES>
__global__ void __launch_bounds__(kThreads) prune_compress_vec(
    const uint8_t* __restrict__ W, int64_t w_row_bytes, int64_t M, int64_t ppr,
    uint8_t* __restrict__ values, int64_t v_row_bytes, uint8_t* __restrict__ meta,
    int64_t m_row_bytes) {
  const int64_t total = M * ppr;
  const int lane = threadIdx.x & 31;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * kThreads) >> 5;
  for (int64_t base = warp * kWarpSpan; base < total; base += nwarps * kWarpSpan) {
    uint4 in[kPiecesPerLane];
    int64_t row[kPiecesPerLane], col[kPiecesPerLane];
#pragma unroll
    for (int i = 0; i < kPiecesPerLane; ++i) {
      const int64_t p = base + i * 32 + lane;
      row[i] = p / ppr;
      col[i] = p - row[i] * ppr;
      if (p < total)
        in[i] = __ldcs(reinterpret_cast<const uint4*>(W + row[i] * w_row_bytes + col[i] * 16));
    }
#pragma unroll
    for (int i = 0; i < kPiecesPerLane; ++i) {
      if (base + i * 32 + lane >= total) break;
      uint32_t mb;
      const uint2 v = compress_piece<DT, ES>(in[i], mb);
      *reinterpret_cast<uint2*>(values + row[i] * v_row_bytes + col[i] * 8) = v;
      if constexpr (ES == 2)
        meta[row[i] * m_row_bytes + col[i]] = static_cast<uint8_t>(mb);
      else
        *reinterpret_cast<uint16_t*>(meta + row[i] * m_row_bytes + col[i] * 2) =
            static_cast<uint16_t>(mb);
    }
  }
}

template <int ES>
__global__ void __launch_bounds__(kThreads) decompress_vec(
    const uint8_t* __restrict__ values, int64_t v_row_bytes, const uint8_t* __restrict__ meta,
    int64_t m_row_bytes, int64_t M, int64_t ppr, uint8_t* __restrict__ W, int64_t w_row_bytes) {
  const int64_t total = M * ppr;
  const int lane = threadIdx.x & 31;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * kThreads) >> 5;
  for (int64_t base = warp * kWarpSpan; base < total; base += nwarps * kWarpSpan) {
    uint2 v[kPiecesPerLane];
    uint32_t mb[kPiecesPerLane];
    int64_t row[kPiecesPerLane], col[kPiecesPerLane];
#pragma unroll
    for (int i = 0; i < kPiecesPerLane; ++i) {
      const int64_t p = base + i * 32 + lane;
      row[i] = p / ppr;
      col[i] = p - row[i] * ppr;
      if (p < total) {
        v[i] = __ldcs(reinterpret_cast<const uint2*>(values + row[i] * v_row_bytes + col[i] * 8));
        if constexpr (ES == 2)
          mb[i] = __ldcs(meta + row[i] * m_row_bytes + col[i]);
        else
          mb[i] = __ldcs(reinterpret_cast<const uint16_t*>(meta + row[i] * m_row_bytes + col[i] * 2));
      }
    }
#pragma unroll
    for (int i = 0; i < kPiecesPerLane; ++i) {
      if (base + i * 32 + lane >= total) break;
      *reinterpret_cast<uint4*>(W + row[i] * w_row_bytes + col[i] * 16) = expand_piece<ES>(v[i], mb[i]);
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

int grid_for(int64_t work_items, int items_per_block, int num_sms) {
  const int64_t want = (work_items + items_per_block - 1) / items_per_block;
  const int64_t cap = static_cast<int64_t>(num_sms) * (2048 / kThreads);
  return static_cast<int>(want < cap ? (want > 0 ? want : 1) : cap);
}

template <int DT, int ES>
void launch_pc(const void* W, int64_t M, int64_t K, int64_t ldw, void* values, void* meta,
               int num_sms, bool fast, cudaStream_t s) {
  if (fast) {
    const int64_t ppr = K * ES / 16;
    const int grid = grid_for(M * ppr, kThreads / 32 * kWarpSpan, num_sms);
    prune_compress_vec<DT, ES><<<grid, kThreads, 0, s>>>(
        static_cast<const uint8_t*>(W), ldw * ES, M, ppr, static_cast<uint8_t*>(values),
        (K / 2) * ES, static_cast<uint8_t*>(meta), meta_row_bytes(K));
  } else {
    const int grid = grid_for(M * meta_row_bytes(K), kThreads, num_sms);
    prune_compress_any<DT, ES><<<grid, kThreads, 0, s>>>(static_cast<const uint8_t*>(W), ldw, M, K,
                                                         static_cast<uint8_t*>(values),
                                                         static_cast<uint8_t*>(meta));
  }
}

template <int ES>
void launch_dc(const void* values, const void* meta, int64_t M, int64_t K, void* W, int64_t ldw,
               int num_sms, bool fast, cudaStream_t s) {
  if (fast) {
    const int64_t ppr = K * ES / 16;
    const int grid = grid_for(M * ppr, kThreads / 32 * kWarpSpan, num_sms);
    decompress_vec<ES><<<grid, kThreads, 0, s>>>(static_cast<const uint8_t*>(values), (K / 2) * ES,
                                                 static_cast<const uint8_t*>(meta),
                                                 meta_row_bytes(K), M, ppr,
                                                 static_cast<uint8_t*>(W), ldw * ES);
  } else {
    const int grid = grid_for(M * meta_row_bytes(K), kThreads, num_sms);
    decompress_any<ES><<<grid, kThreads, 0, s>>>(static_cast<const uint8_t*>(values),
                                                 static_cast<const uint8_t*>(meta), M, K,
                                                 static_cast<uint8_t*>(W), ldw);
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
