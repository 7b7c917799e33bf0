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
#include "st24_schedule.cuh"

#include <type_traits>

#include <cuda_fp16.h>
#include <cuda_fp8.h>

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

// ---- the same selection on several groups at once ("SIMD within a register")
// Lanes of a 32-bit word hold one group each (16-bit lanes: 2 groups, 8-bit
// lanes: 4 groups).  With every magnitude key below its lane's top bit,
// (k_i | TOP) - k_j has the lane's top bit set exactly when k_i >= k_j and
// never borrows from the next lane, so one subtraction compares all lanes.
// The keep rule is the majority formulation of compress_group, evaluated on
// the lanes' top bits; a byte permute that replicates each lane's top bit
// turns the result into lane masks for the selects.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

template <int LANE>
struct Lanes {
  static constexpr uint32_t TOP = LANE == 16 ? 0x80008000u : 0x80808080u;
  static constexpr uint32_t ONE = LANE == 16 ? 0x00010001u : 0x01010101u;
  // prmt selector: every byte takes the sign (top bit) of its lane's top byte.
  static constexpr uint32_t SPREAD = LANE == 16 ? 0xBB99u : 0xBA98u;
};

__device__ __forceinline__ uint32_t maj(uint32_t a, uint32_t b, uint32_t c) { return (a & b) | (a & c) | (b & c); }

// k[i]: keys of element i of every lane's group; x[i]: the raw elements.
// v0, v1: the kept pair of every lane (lower index first); nib: its nibble
// i0 | i1 << 2 in the low bits of every lane.
template <int LANE>
__device__ __forceinline__ void select_lanes(const uint32_t (&k)[4], const uint32_t (&x)[4], uint32_t& v0,
                                             uint32_t& v1, uint32_t& nib) {
  using L = Lanes<LANE>;
  const uint32_t T = L::TOP;
  const uint32_t c01 = ((k[0] | T) - k[1]) & T, c02 = ((k[0] | T) - k[2]) & T, c03 = ((k[0] | T) - k[3]) & T;
  const uint32_t c12 = ((k[1] | T) - k[2]) & T, c13 = ((k[1] | T) - k[3]) & T, c23 = ((k[2] | T) - k[3]) & T;
  const uint32_t m0 = prmt(maj(c01, c02, c03), 0, L::SPREAD);
  const uint32_t m1 = prmt(maj(c01 ^ T, c12, c13), 0, L::SPREAD);
  const uint32_t m2 = prmt(maj(c02 ^ T, c12 ^ T, c23), 0, L::SPREAD);
  const uint32_t m3 = prmt(maj(c03 ^ T, c13 ^ T, c23 ^ T), 0, L::SPREAD);
  v0 = (x[0] & m0) | (~m0 & ((x[1] & m1) | (~m1 & x[2])));
  v1 = (x[3] & m3) | (~m3 & ((x[2] & m2) | (~m2 & x[1])));
  const uint32_t one = L::ONE, two = L::ONE << 1;
  const uint32_t i0 = ~m0 & ((m1 & one) | (~m1 & two));
  const uint32_t i1 = (m3 & (one | two)) | (~m3 & ((m2 & two) | (~m2 & one)));
  nib = i0 | (i1 << 2);
}

// compress_piece on lanes.  Returns false (16-bit types only) when the piece
// holds a NaN, whose keys need the clamp of mag_key; the caller then uses
// compress_piece.
template <int DT, int ES>
__device__ __forceinline__ bool compress_piece_lanes(const uint4 in, uint2& out, uint32_t& meta_bits) {
  if constexpr (ES == 2) {
    // x[i] = element i of group 0 (low lane) and of group 1 (high lane).
    const uint32_t x[4] = {prmt(in.x, in.z, 0x5410), prmt(in.x, in.z, 0x7632), prmt(in.y, in.w, 0x5410),
                           prmt(in.y, in.w, 0x7632)};
    uint32_t k[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) k[i] = x[i] & 0x7FFF7FFFu;
    // a lane holds a NaN when its key is above the infinity pattern
    constexpr uint32_t below_top = DT == kBF16 ? 0x007F007Fu : 0x03FF03FFu;
    if (((k[0] + below_top) | (k[1] + below_top) | (k[2] + below_top) | (k[3] + below_top)) & 0x80008000u)
      return false;
    uint32_t v0, v1, nib;
    select_lanes<16>(k, x, v0, v1, nib);
    out = make_uint2(prmt(v0, v1, 0x5410), prmt(v0, v1, 0x7632));
    meta_bits = (nib & 0xFu) | ((nib >> 12) & 0xF0u);
    return true;
  } else {
    // 8-bit types, 8-bit lanes: 4x4 byte transpose, x[i] = element i of
    // groups 0..3 (lane g = group g).
    const uint32_t t0 = prmt(in.x, in.y, 0x5140), t1 = prmt(in.x, in.y, 0x7362);
    const uint32_t t2 = prmt(in.z, in.w, 0x5140), t3 = prmt(in.z, in.w, 0x7362);
    const uint32_t x[4] = {prmt(t0, t2, 0x5410), prmt(t0, t2, 0x7632), prmt(t1, t3, 0x5410),
                           prmt(t1, t3, 0x7632)};
    uint32_t k[4];
    bool lanes8 = true;
    if constexpr (DT == kE4M3) {
      // |x| order is the order of the low 7 bits; 0x7F, the only NaN
      // magnitude, is above every number and ties with itself.
#pragma unroll
      for (int i = 0; i < 4; ++i) k[i] = x[i] & 0x7F7F7F7Fu;
    } else {
      // int8: |v| fits in 7 bits unless v = -128 (a 0x80 byte); such pieces
      // take 16-bit lanes below.
      uint32_t has_min = 0;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t y = x[i] ^ 0x80808080u;   // 0x80 bytes become zero bytes
        has_min |= (y - 0x01010101u) & ~y & 0x80808080u;
        const uint32_t neg = prmt(x[i], 0, 0xBA98);   // all-ones in negative bytes
        k[i] = (x[i] ^ neg) + (neg & 0x01010101u);
      }
      lanes8 = has_min == 0;
    }
    if (lanes8) {
      uint32_t v0, v1, nib;
      select_lanes<8>(k, x, v0, v1, nib);
      out = make_uint2(prmt(v0, v1, 0x5140), prmt(v0, v1, 0x7362));
      const uint32_t t = nib | (nib >> 4);   // bytes 0 and 2: two nibbles each
      meta_bits = prmt(t, 0, 0x4420) & 0xFFFFu;
      return true;
    }
  }
  if constexpr (DT == kS8) {
    // int8 with a -128: |-128| = 128 needs 8 bits, so 16-bit lanes, two
    // groups per pass; each element sign-extended into its lane.
    const uint32_t w[4] = {in.x, in.y, in.z, in.w};
    uint32_t pairs[2];
    meta_bits = 0;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t a = w[2 * h], b = w[2 * h + 1];
      const uint32_t x[4] = {prmt(a, b, 0xC480), prmt(a, b, 0xD591), prmt(a, b, 0xE6A2), prmt(a, b, 0xF7B3)};
      uint32_t k[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t neg = prmt(x[i], 0, 0xBB99);   // all-ones in negative lanes
        k[i] = (x[i] ^ neg) + (neg & 0x00010001u);
      }
      uint32_t v0, v1, nib;
      select_lanes<16>(k, x, v0, v1, nib);
      pairs[h] = prmt(v0, v1, 0x6240);
      meta_bits |= ((nib & 0xFu) | ((nib >> 12) & 0xF0u)) << (8 * h);
    }
    out = make_uint2(pairs[0], pairs[1]);
    return true;
  }
  return false;   // not reached: e4m3 always takes the 8-bit lanes
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
constexpr int kPiecesPerLane = 2;
constexpr int kWarpSpan = 32 * kPiecesPerLane;  // pieces one warp handles per iteration

// Fast path.  The matrix is a sequence of 16-byte pieces, `ppr` per row; warp
// w handles pieces [w*64, w*64+64) of each grid-stride round, lane l the
// pieces l and l+32 of that span.  Piece p (counted row by row)
// owns bytes [8p, 8p+8) of the values and its metadata at p * (16 / ES / 8)
// bytes, since both outputs are dense; only the input may have a row stride.
// Where it has one, a lane divides once per round (Idx is 32-bit whenever the
// piece count allows) and carries (row, col) forward for its other pieces.
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

bool aligned(const void* p, int a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// ---- N:M prune into one or two 2:4 forms -----------------------------------
// ("Chapter 26 -- Sparsity: The Hardware View", section "Block Sparsity, N:M
// Generalizations, and Channel Pruning": keep N of every M consecutive
// weights.)  In every group of M_ elements along K the N_ of largest
// magnitude are kept (the order of mag_key; ties to the lower index).  Each
// aligned 4-element subgroup then holds some of the kept elements in
// ascending index order: the first two go to form 0, the rest (TWO: up to two
// more, for N_ up to 4) to form 1; a form holding fewer than two of a
// subgroup's elements takes as the missing slots the lowest indices of the
// subgroup not among its own, with +0 values.  With N_ <= 2 form 0 is the
// whole result, a 2:4 compressed form st24_spmm multiplies exactly; with two
// forms (values M x K and metadata M x 2 ceil(K/8), form 0 then form 1 in
// each row) the forms together are the 2:4 form of an M x 2K matrix whose
// product with B stacked twice is the pruned matrix times B.  One thread per
// 8 elements of a row (two subgroups: one metadata byte per form);
// neighbouring threads take neighbouring elements, so the warp's loads and
// stores are contiguous.

// The pair a form stores for one subgroup: its own kept elements (bits of
// `own`, at most two) and the lowest other indices as +0 fillers, ascending.
__device__ __forceinline__ void form_pair(uint32_t own, int& i0, int& i1, bool& v0, bool& v1) {
  int idx[2] = {0, 0};
  bool isv[2] = {false, false};
  int c = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j)
    if (((own >> j) & 1u) && c < 2) { idx[c] = j; isv[c] = true; ++c; }
#pragma unroll
  for (int j = 0; j < 4; ++j)
    if (c < 2 && !((own >> j) & 1u) && (c == 0 || idx[0] != j)) { idx[c] = j; isv[c] = false; ++c; }
  const bool lo = idx[0] < idx[1];
  i0 = lo ? idx[0] : idx[1];
  i1 = lo ? idx[1] : idx[0];
  v0 = lo ? isv[0] : isv[1];
  v1 = lo ? isv[1] : isv[0];
}

template <int DT, int ES, int N_, int M_, bool TWO>
__global__ void __launch_bounds__(kThreads) prune_compress_nm_kernel(const uint8_t* __restrict__ W, int64_t w_row_bytes,
                                                                     int64_t M, int64_t K, uint8_t* __restrict__ values,
                                                                     uint8_t* __restrict__ meta, int vec) {
  static_assert(M_ == 4 || M_ == 8, "group size");
  static_assert(N_ >= 1 && N_ <= (TWO ? 4 : 2) && N_ <= M_, "kept per group");
  const int64_t upr = (K + 7) / 8;   // 8-element units per row
  const int64_t total = M * upr;
  const int64_t mrb = meta_row_bytes(K);
  const int64_t vrow = TWO ? K : K / 2;          // values per row (both forms)
  const int64_t erow = TWO ? 2 * mrb : mrb;      // metadata bytes per row (both forms)
  for (int64_t u = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; u < total;
       u += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = div_nn(u, upr), c0 = (u - r * upr) * 8;
    const int cnt = K - c0 < 8 ? static_cast<int>(K - c0) : 8;   // 4 or 8
    const uint8_t* src = W + r * w_row_bytes + c0 * ES;
    uint32_t e[8], k[8];
    if (vec && cnt == 8) {
      // the unit in one load (16-byte aligned rows of 16-bit values, 8-byte of 8-bit ones)
      if constexpr (ES == 2) {
        const uint4 v = __ldcs(reinterpret_cast<const uint4*>(src));
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 8; ++j) e[j] = (w[j / 2] >> (16 * (j & 1))) & 0xFFFFu;
      } else {
        const uint2 v = __ldcs(reinterpret_cast<const uint2*>(src));
        const uint32_t w[2] = {v.x, v.y};
#pragma unroll
        for (int j = 0; j < 8; ++j) e[j] = (w[j / 4] >> (8 * (j & 3))) & 0xFFu;
      }
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        e[j] = 0u;
        if (j < cnt) e[j] = ES == 2 ? static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(src)[j]) : src[j];
      }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) k[j] = mag_key<DT>(e[j]);
    uint32_t kept = 0;   // bit j: element j of the unit is kept
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      constexpr int m = M_;
      const int b = (j / m) * m;   // this element's m-group inside the unit
      int above = 0;               // elements of the group that outrank it
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (i >= b && i < b + m && i != j && (k[i] > k[j] || (k[i] == k[j] && i < j))) ++above;
      if (j < cnt && above < N_) kept |= 1u << j;
    }
    uint32_t mb[2] = {0u, 0u};
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      if (4 * q >= cnt) break;
      const uint32_t km = (kept >> (4 * q)) & 0xFu;
      uint32_t own[2];
      if constexpr (TWO) {
        const uint32_t b1 = km & (0u - km), rest = km ^ b1, b2 = rest & (0u - rest);
        own[0] = b1 | b2;        // the subgroup's first two kept elements
        own[1] = km & ~own[0];   // the rest
      } else {
        own[0] = km;
        own[1] = 0u;
      }
#pragma unroll
      for (int f = 0; f < (TWO ? 2 : 1); ++f) {
        int i0, i1;
        bool v0, v1;
        form_pair(own[f], i0, i1, v0, v1);
        const uint32_t a0 = v0 ? e[4 * q + i0] : 0u, a1 = v1 ? e[4 * q + i1] : 0u;
        uint8_t* vrow_ptr = values + (r * vrow + f * (K / 2)) * ES;
        const int64_t col = c0 / 2 + 2 * q;   // value column of the pair
        if constexpr (ES == 2) {
          *reinterpret_cast<uint32_t*>(vrow_ptr + col * 2) = a0 | (a1 << 16);
        } else {
          *reinterpret_cast<uint16_t*>(vrow_ptr + col) = static_cast<uint16_t>(a0 | (a1 << 8));
        }
        mb[f] |= static_cast<uint32_t>(i0 | (i1 << 2)) << (4 * q);
      }
    }
    meta[r * erow + c0 / 8] = static_cast<uint8_t>(mb[0]);
    if constexpr (TWO) meta[r * erow + mrb + c0 / 8] = static_cast<uint8_t>(mb[1]);
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

st24_status launch_prune_compress_nm(int dt, int n, int m, bool two, const void* W, int64_t M, int64_t K,
                                     int64_t ldw, void* values, void* meta, cudaStream_t stream) {
  const DeviceInfo* dev = current_device_info();
  if (!dev) return ST24_ERR_CUDA;
  const int64_t units = M * ((K + 7) / 8);
  auto go = [&](auto kern, int es) {
    const int va = 8 * es;   // bytes of one unit: its vector load needs this alignment
    const int vec = aligned(W, va) && (ldw * es) % va == 0 ? 1 : 0;
    kern<<<grid_for(kern, units, kThreads, dev->num_sms), kThreads, 0, stream>>>(
        static_cast<const uint8_t*>(W), ldw * es, M, K, static_cast<uint8_t*>(values), static_cast<uint8_t*>(meta),
        vec);
    return true;
  };
  // (n, m, two) -> the compiled pattern, for one element type
  auto pattern = [&](auto dtc, auto esc) {
    constexpr int DT = decltype(dtc)::value, ES = decltype(esc)::value;
#define ST24_NM(N_, M_, TWO)                                                                  \
  if (n == N_ && m == M_ && two == TWO) return go(prune_compress_nm_kernel<DT, ES, N_, M_, TWO>, ES);
    ST24_NM(1, 4, false) ST24_NM(2, 4, false) ST24_NM(1, 8, false) ST24_NM(2, 8, false)
    ST24_NM(1, 4, true) ST24_NM(2, 4, true) ST24_NM(3, 4, true) ST24_NM(4, 4, true)
    ST24_NM(1, 8, true) ST24_NM(2, 8, true) ST24_NM(3, 8, true) ST24_NM(4, 8, true)
#undef ST24_NM
    return false;
  };
  bool ok = false;
  switch (dt) {
    case kF16: ok = pattern(std::integral_constant<int, kF16>{}, std::integral_constant<int, 2>{}); break;
    case kBF16: ok = pattern(std::integral_constant<int, kBF16>{}, std::integral_constant<int, 2>{}); break;
    case kE4M3: ok = pattern(std::integral_constant<int, kE4M3>{}, std::integral_constant<int, 1>{}); break;
    case kS8: ok = pattern(std::integral_constant<int, kS8>{}, std::integral_constant<int, 1>{}); break;
    default: break;
  }
  if (!ok) return ST24_ERR_UNSUPPORTED;
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
