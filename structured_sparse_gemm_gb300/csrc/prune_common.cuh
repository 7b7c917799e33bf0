// prune_common.cuh -- pieces shared by the prune/compress kernels: the
// magnitude key, the 2:4 selection on one group and on lanes of a word, the
// 16-byte piece codecs, and the host-side grid and layout helpers.
#pragma once

#include "st24_device.cuh"

#include <cstdint>

namespace st24 {
namespace prune {

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

// Moves (row, col) of a piece `step` pieces forward in a matrix of `ppr`
// pieces per row.
template <typename Idx>
__device__ __forceinline__ void advance(Idx& row, Idx& col, Idx step, Idx ppr) {
  col += step;
  while (col >= ppr) {
    col -= ppr;
    ++row;
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

inline bool aligned(const void* p, int a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

inline bool fast_layout(int es, int64_t K, int64_t ldw, const void* W, const void* values,
                 const void* meta) {
  return (K * es) % 16 == 0 && (ldw * es) % 16 == 0 && aligned(W, 16) && aligned(values, 8) &&
         aligned(meta, es == 1 ? 2 : 1);
}

}  // namespace prune
}  // namespace st24
