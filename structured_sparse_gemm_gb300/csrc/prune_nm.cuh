// prune_nm.cuh -- N:M magnitude prune into one or two 2:4 compressed forms
// (the kernels and their launcher, instantiated per element type by
// prune_nm_16.cu and prune_nm_8.cu).
#pragma once

#include "prune_common.cuh"
#include "st24_internal.h"
#include "st24_schedule.cuh"

namespace st24 {
namespace prune {

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

// One 8-element unit (cnt = 8, or 4 at the end of a row with K % 8 == 4),
// element by element: the kept mask by rank, then for form f and subgroup q
// the stored pair packed as a0 | a1 << (8 ES) in pv[f][q], and form f's
// metadata byte in mb[f].
template <int DT, int ES, int N_, int M_, bool TWO>
__device__ __forceinline__ void nm_unit(const uint32_t (&e)[8], int cnt, uint32_t (&pv)[2][2], uint32_t (&mb)[2]) {
  uint32_t k[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) k[j] = mag_key<DT>(e[j]);
  uint32_t kept = 0;   // bit j: element j of the unit is kept
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int b = (j / M_) * M_;   // this element's group inside the unit
    int above = 0;                 // elements of the group that outrank it
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (i >= b && i < b + M_ && i != j && (k[i] > k[j] || (k[i] == k[j] && i < j))) ++above;
    if (j < cnt && above < N_) kept |= 1u << j;
  }
  mb[0] = mb[1] = 0u;
  pv[0][0] = pv[0][1] = pv[1][0] = pv[1][1] = 0u;
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
      pv[f][q] = a0 | (a1 << (8 * ES));
      mb[f] |= static_cast<uint32_t>(i0 | (i1 << 2)) << (4 * q);
    }
  }
}

// Any layout: one thread per unit.
template <int DT, int ES, int N_, int M_, bool TWO>
__global__ void __launch_bounds__(kThreads) prune_compress_nm_kernel(const uint8_t* __restrict__ W, int64_t w_row_bytes,
                                                                     int64_t M, int64_t K, uint8_t* __restrict__ values,
                                                                     uint8_t* __restrict__ meta) {
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
    uint32_t e[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      e[j] = 0u;
      if (j < cnt) e[j] = ES == 2 ? static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(src)[j]) : src[j];
    }
    uint32_t pv[2][2], mb[2];
    nm_unit<DT, ES, N_, M_, TWO>(e, cnt, pv, mb);
#pragma unroll
    for (int f = 0; f < (TWO ? 2 : 1); ++f) {
      uint8_t* dst = values + (r * vrow + f * (K / 2) + c0 / 2) * ES;   // this unit's pairs in form f
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        if (4 * q >= cnt) break;
        if constexpr (ES == 2) {
          reinterpret_cast<uint16_t*>(dst)[2 * q] = static_cast<uint16_t>(pv[f][q]);
          reinterpret_cast<uint16_t*>(dst)[2 * q + 1] = static_cast<uint16_t>(pv[f][q] >> 16);
        } else {
          dst[2 * q] = static_cast<uint8_t>(pv[f][q]);
          dst[2 * q + 1] = static_cast<uint8_t>(pv[f][q] >> 8);
        }
      }
      meta[r * erow + f * mrb + c0 / 8] = static_cast<uint8_t>(mb[f]);
    }
  }
}

// ---- the same on lanes -------------------------------------------------------
// A thread holds two 16-byte pieces and arranges their units in lanes: word j
// holds element j of every unit (16-bit types: the two pieces' units; 8-bit:
// the four units of the two pieces, piece 0's first).  The rank of an element
// is the number of its group's elements that outrank it; with
// c_ab = (k_a >= k_b) on the lanes' top bits (the subtraction of
// select_lanes), element j loses to a < j where c_aj and to b > j where not
// c_jb, and is kept when it loses fewer than N_ times: for groups of 4 a
// boolean function of the three losses, for groups of 8 a count of the seven
// taken with bit-sliced full adders.  A form's own elements of a subgroup
// (masks o0..o3) plus its fillers (the lowest other indices while fewer than
// two are owned) are exactly two positions, stored in ascending order with the
// fillers' values +0: the select of select_lanes on those positions.

// Element j of every unit in words x, magnitude keys in k (below each lane's
// top bit).  False when a key would need the clamp of mag_key (a NaN in a
// 16-bit type) or 8 bits (an int8 -128); the caller then goes unit by unit.
template <int DT, int ES>
__device__ __forceinline__ bool nm_lane_words(const uint4 a, const uint4 b, uint32_t (&x)[8], uint32_t (&k)[8]) {
  if constexpr (ES == 2) {
    const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[2 * i] = prmt(wa[i], wb[i], 0x5410);
      x[2 * i + 1] = prmt(wa[i], wb[i], 0x7632);
    }
    constexpr uint32_t below_top = DT == kBF16 ? 0x007F007Fu : 0x03FF03FFu;
    uint32_t nan = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      k[j] = x[j] & 0x7FFF7FFFu;
      nan |= k[j] + below_top;
    }
    return (nan & 0x80008000u) == 0;
  } else {
    // bytes (piece 0 unit 0, piece 0 unit 1, piece 1 unit 0, piece 1 unit 1)
    const uint32_t lo[2][2] = {{a.x, a.z}, {b.x, b.z}}, hi[2][2] = {{a.y, a.w}, {b.y, b.w}};
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const uint32_t(&w)[2][2] = half ? hi : lo;
      const uint32_t p01 = prmt(w[0][0], w[0][1], 0x5140), p23 = prmt(w[0][0], w[0][1], 0x7362);
      const uint32_t q01 = prmt(w[1][0], w[1][1], 0x5140), q23 = prmt(w[1][0], w[1][1], 0x7362);
      x[4 * half + 0] = prmt(p01, q01, 0x5410);
      x[4 * half + 1] = prmt(p01, q01, 0x7632);
      x[4 * half + 2] = prmt(p23, q23, 0x5410);
      x[4 * half + 3] = prmt(p23, q23, 0x7632);
    }
    if constexpr (DT == kE4M3) {
#pragma unroll
      for (int j = 0; j < 8; ++j) k[j] = x[j] & 0x7F7F7F7Fu;   // 0x7F (NaN) is above every number
      return true;
    } else {
      uint32_t has_min = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t y = x[j] ^ 0x80808080u;
        has_min |= (y - 0x01010101u) & ~y & 0x80808080u;
        const uint32_t neg = prmt(x[j], 0, 0xBA98);
        k[j] = (x[j] ^ neg) + (neg & 0x01010101u);
      }
      return has_min == 0;
    }
  }
}

// kept when fewer than N_ of the losses l[] are set (top bits).
template <int N_>
__device__ __forceinline__ uint32_t keep_of3(uint32_t l1, uint32_t l2, uint32_t l3) {
  if constexpr (N_ == 1) return ~(l1 | l2 | l3);
  else if constexpr (N_ == 2) return ~maj(l1, l2, l3);
  else if constexpr (N_ == 3) return ~(l1 & l2 & l3);
  else return ~0u;
}
template <int N_>
__device__ __forceinline__ uint32_t keep_of7(const uint32_t (&l)[7]) {
  if constexpr (N_ == 1) {
    return ~(l[0] | l[1] | l[2] | l[3] | l[4] | l[5] | l[6]);
  } else {
    // the count of set losses, bit-sliced: b0 + 2 b1 + 4 b2
    const uint32_t s1 = l[0] ^ l[1] ^ l[2], c1 = maj(l[0], l[1], l[2]);
    const uint32_t s2 = l[3] ^ l[4] ^ l[5], c2 = maj(l[3], l[4], l[5]);
    const uint32_t b0 = s1 ^ s2 ^ l[6], c3 = maj(s1, s2, l[6]);
    const uint32_t b1 = c1 ^ c2 ^ c3, b2 = maj(c1, c2, c3);
    if constexpr (N_ == 2) return ~(b1 | b2);
    else if constexpr (N_ == 3) return ~(b2 | (b1 & b0));
    else return ~b2;
  }
}

// The stored pair of every lane's subgroup for one form, from the form's own
// lane masks o[0..3] and the subgroup's raw words xs[0..3].
template <int LANE, bool ALWAYS_TWO>
__device__ __forceinline__ void nm_form_pair(const uint32_t (&o)[4], const uint32_t (&xs)[4], uint32_t& v0,
                                             uint32_t& v1, uint32_t& nib) {
  using L = Lanes<LANE>;
  uint32_t f0 = o[0], f1 = o[1];
  if constexpr (!ALWAYS_TWO) {
    const uint32_t two = (o[0] & o[1]) | (o[2] & o[3]) | ((o[0] | o[1]) & (o[2] | o[3]));
    const uint32_t any = o[0] | o[1] | o[2] | o[3];
    f0 = o[0] | ~two;
    f1 = o[1] | ~any | (~two & o[0]);
  }
  const uint32_t f2 = o[2], f3 = o[3];
  const uint32_t y0 = xs[0] & o[0], y1 = xs[1] & o[1], y2 = xs[2] & o[2], y3 = xs[3] & o[3];
  v0 = (y0 & f0) | (~f0 & ((y1 & f1) | (~f1 & y2)));
  v1 = (y3 & f3) | (~f3 & ((y2 & f2) | (~f2 & y1)));
  const uint32_t one = L::ONE, two2 = L::ONE << 1;
  const uint32_t i0 = ~f0 & ((f1 & one) | (~f1 & two2));
  const uint32_t i1 = (f3 & (one | two2)) | (~f3 & ((f2 & two2) | (~f2 & one)));
  nib = i0 | (i1 << 2);
}

// v0[f][h], v1[f][h], nib[f][h]: form f's pair of subgroup h (elements 4h..4h+3) in every lane.
template <int LANE, int N_, int M_, bool TWO>
__device__ __forceinline__ void nm_select_lanes(const uint32_t (&x)[8], const uint32_t (&k)[8],
                                                uint32_t (&v0)[2][2], uint32_t (&v1)[2][2], uint32_t (&nib)[2][2]) {
  using L = Lanes<LANE>;
  constexpr uint32_t T = L::TOP;
  uint32_t keep[8];
  if constexpr (M_ == 4) {
#pragma unroll
    for (int g = 0; g < 8; g += 4) {
      const uint32_t t0 = k[g] | T, t1 = k[g + 1] | T, t2 = k[g + 2] | T;
      const uint32_t c01 = t0 - k[g + 1], c02 = t0 - k[g + 2], c03 = t0 - k[g + 3];
      const uint32_t c12 = t1 - k[g + 2], c13 = t1 - k[g + 3], c23 = t2 - k[g + 3];
      keep[g] = keep_of3<N_>(~c01, ~c02, ~c03);
      keep[g + 1] = keep_of3<N_>(c01, ~c12, ~c13);
      keep[g + 2] = keep_of3<N_>(c02, c12, ~c23);
      keep[g + 3] = keep_of3<N_>(c03, c13, c23);
    }
  } else {
    uint32_t c[8][8];
#pragma unroll
    for (int a = 0; a < 7; ++a) {
      const uint32_t t = k[a] | T;
#pragma unroll
      for (int b = a + 1; b < 8; ++b) c[a][b] = t - k[b];
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      uint32_t l[7];
      int n = 0;
#pragma unroll
      for (int a = 0; a < 8; ++a) {
        if (a < j) l[n++] = c[a][j];
        else if (a > j) l[n++] = ~c[j][a];
      }
      keep[j] = keep_of7<N_>(l);
    }
  }
  uint32_t m[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) m[j] = prmt(keep[j], 0, L::SPREAD);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint32_t s[4] = {m[4 * h], m[4 * h + 1], m[4 * h + 2], m[4 * h + 3]};
    const uint32_t xs[4] = {x[4 * h], x[4 * h + 1], x[4 * h + 2], x[4 * h + 3]};
    if constexpr (TWO) {
      const uint32_t s012 = maj(s[0], s[1], s[2]);
      const uint32_t o0[4] = {s[0], s[1], s[2] & ~(s[0] & s[1]), s[3] & ~s012};   // the first two kept
      const uint32_t o1[4] = {0u, 0u, s[2] & s[0] & s[1], s[3] & s012};            // the rest
      nm_form_pair<LANE, M_ == 4 && N_ == 4>(o0, xs, v0[0][h], v1[0][h], nib[0][h]);
      nm_form_pair<LANE, M_ == 4 && N_ == 4>(o1, xs, v0[1][h], v1[1][h], nib[1][h]);
    } else {
      nm_form_pair<LANE, M_ == 4 && N_ == 2>(s, xs, v0[0][h], v1[0][h], nib[0][h]);
    }
  }
}

// Fast layout (K * ES % 16 == 0, 16-byte rows): lane l of warp w takes the
// pieces w*64 + l and w*64 + l + 32 of each grid-stride round.  Piece q of row
// r, column c (16-byte pieces from the row start) holds 16 / ES elements: its
// pairs go to form f at 8 bytes per piece and its metadata at 16 / ES / 8
// bytes per piece.
template <int DT, int ES, int N_, int M_, bool TWO, typename Idx>
__global__ void __launch_bounds__(kThreads) prune_compress_nm_vec(const uint8_t* __restrict__ W, int64_t w_row_bytes,
                                                                  Idx total, Idx ppr, int64_t K,
                                                                  uint8_t* __restrict__ values,
                                                                  uint8_t* __restrict__ meta) {
  static_assert(M_ == 4 || M_ == 8, "group size");
  static_assert(N_ >= 1 && N_ <= (TWO ? 4 : 2) && N_ <= M_, "kept per group");
  static_assert(kPiecesPerLane == 2, "two pieces per lane");
  constexpr int LANE = ES == 2 ? 16 : 8;
  constexpr int UPP = 2 / ES;   // 8-element units per piece
  const int lane = threadIdx.x & 31;
  const Idx warp = (static_cast<Idx>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
  const Idx nwarps = (static_cast<Idx>(gridDim.x) * kThreads) >> 5;
  const bool dense = w_row_bytes == static_cast<int64_t>(ppr) * 16;
  const int64_t mrb = K / 8;                          // one form's metadata bytes per row
  const int64_t vrb = (TWO ? K : K / 2) * ES;         // values bytes per row (both forms)
  const int64_t erb = TWO ? 2 * mrb : mrb;            // metadata bytes per row (both forms)
  for (Idx base = warp * kWarpSpan; base < total; base += nwarps * kWarpSpan) {
    const Idx q[2] = {base + lane, base + 32 + lane};
    if (q[0] >= total) break;
    const bool has1 = q[1] < total;
    Idx r[2] = {0, 0}, c[2] = {0, 0};
    if (TWO || !dense) {
      r[0] = q[0] / ppr;
      c[0] = q[0] - r[0] * ppr;
      r[1] = r[0];
      c[1] = c[0];
      advance<Idx>(r[1], c[1], 32, ppr);
    }
    uint4 in[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      in[i] = make_uint4(0u, 0u, 0u, 0u);
      if (i == 0 || has1)
        in[i] = __ldcs(dense ? reinterpret_cast<const uint4*>(W) + q[i]
                             : reinterpret_cast<const uint4*>(W + static_cast<int64_t>(r[i]) * w_row_bytes) + c[i]);
    }
    // where piece i's form f pairs and metadata go
    auto vptr = [&](int i, int f) -> uint8_t* {
      if constexpr (TWO) return values + static_cast<int64_t>(r[i]) * vrb + f * (K / 2) * ES + static_cast<int64_t>(c[i]) * 8;
      else return values + static_cast<int64_t>(q[i]) * 8;
    };
    auto eptr = [&](int i, int f) -> uint8_t* {
      if constexpr (TWO) return meta + static_cast<int64_t>(r[i]) * erb + f * mrb + static_cast<int64_t>(c[i]) * UPP;
      else return meta + static_cast<int64_t>(q[i]) * UPP;
    };
    uint32_t x[8], k[8];
    if (nm_lane_words<DT, ES>(in[0], in[1], x, k)) {
      uint32_t v0[2][2], v1[2][2], nib[2][2];
      nm_select_lanes<LANE, N_, M_, TWO>(x, k, v0, v1, nib);
#pragma unroll
      for (int f = 0; f < (TWO ? 2 : 1); ++f) {
        const uint32_t t = nib[f][0] | (nib[f][1] << 4);   // every lane's metadata byte
        uint2 out[2];
        uint32_t mb[2];
        if constexpr (ES == 2) {
          out[0] = make_uint2(prmt(v0[f][0], v1[f][0], 0x5410), prmt(v0[f][1], v1[f][1], 0x5410));
          out[1] = make_uint2(prmt(v0[f][0], v1[f][0], 0x7632), prmt(v0[f][1], v1[f][1], 0x7632));
          mb[0] = t & 0xFFu;
          mb[1] = (t >> 16) & 0xFFu;
        } else {
          const uint32_t p01 = prmt(v0[f][0], v1[f][0], 0x5140), q01 = prmt(v0[f][1], v1[f][1], 0x5140);
          const uint32_t p23 = prmt(v0[f][0], v1[f][0], 0x7362), q23 = prmt(v0[f][1], v1[f][1], 0x7362);
          out[0] = make_uint2(prmt(p01, q01, 0x5410), prmt(p01, q01, 0x7632));
          out[1] = make_uint2(prmt(p23, q23, 0x5410), prmt(p23, q23, 0x7632));
          mb[0] = t & 0xFFFFu;
          mb[1] = t >> 16;
        }
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          if (i == 1 && !has1) break;
          *reinterpret_cast<uint2*>(vptr(i, f)) = out[i];
          if constexpr (ES == 2)
            *eptr(i, f) = static_cast<uint8_t>(mb[i]);
          else
            *reinterpret_cast<uint16_t*>(eptr(i, f)) = static_cast<uint16_t>(mb[i]);
        }
      }
    } else {
      // unit by unit
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        if (i == 1 && !has1) break;
        const uint32_t w[4] = {in[i].x, in[i].y, in[i].z, in[i].w};
#pragma unroll
        for (int u = 0; u < UPP; ++u) {
          uint32_t e[8];
#pragma unroll
          for (int j = 0; j < 8; ++j)
            e[j] = ES == 2 ? (w[j / 2] >> (16 * (j & 1))) & 0xFFFFu : (w[2 * u + j / 4] >> (8 * (j & 3))) & 0xFFu;
          uint32_t pv[2][2], mbu[2];
          nm_unit<DT, ES, N_, M_, TWO>(e, 8, pv, mbu);
#pragma unroll
          for (int f = 0; f < (TWO ? 2 : 1); ++f) {
            if constexpr (ES == 2)
              *reinterpret_cast<uint2*>(vptr(i, f)) = make_uint2(pv[f][0], pv[f][1]);
            else
              reinterpret_cast<uint32_t*>(vptr(i, f))[u] = pv[f][0] | (pv[f][1] << 16);
            eptr(i, f)[u] = static_cast<uint8_t>(mbu[f]);
          }
        }
      }
    }
  }
}

// The launch for element type DT: the lanes kernel on the fast layout, the
// unit-by-unit kernel otherwise.  False for a pattern that is not compiled.
template <int DT, int ES>
bool launch_nm(int n, int m, bool two, const void* W, int64_t M, int64_t K, int64_t ldw, void* values, void* meta,
               int num_sms, cudaStream_t stream) {
  const bool fast = fast_layout(ES, K, ldw, W, values, meta);
  auto go = [&](auto vec32, auto vec64, auto any) {
    auto* w = static_cast<const uint8_t*>(W);
    auto* v = static_cast<uint8_t*>(values);
    auto* e = static_cast<uint8_t*>(meta);
    if (fast) {
      const int64_t ppr = K * ES / 16, total = M * ppr;
      if (fits_u32(total))
        vec32<<<grid_for(vec32, total, kThreads / 32 * kWarpSpan, num_sms), kThreads, 0, stream>>>(
            w, ldw * ES, static_cast<uint32_t>(total), static_cast<uint32_t>(ppr), K, v, e);
      else
        vec64<<<grid_for(vec64, total, kThreads / 32 * kWarpSpan, num_sms), kThreads, 0, stream>>>(
            w, ldw * ES, total, ppr, K, v, e);
    } else {
      any<<<grid_for(any, M * ((K + 7) / 8), kThreads, num_sms), kThreads, 0, stream>>>(w, ldw * ES, M, K, v, e);
    }
    return true;
  };
#define ST24_NM(N_, M_, TWO)                                                                   \
  if (n == N_ && m == M_ && two == TWO)                                                        \
    return go(prune_compress_nm_vec<DT, ES, N_, M_, TWO, uint32_t>,                            \
              prune_compress_nm_vec<DT, ES, N_, M_, TWO, int64_t>, prune_compress_nm_kernel<DT, ES, N_, M_, TWO>);
  ST24_NM(1, 4, false) ST24_NM(2, 4, false) ST24_NM(1, 8, false) ST24_NM(2, 8, false)
  ST24_NM(1, 4, true) ST24_NM(2, 4, true) ST24_NM(3, 4, true) ST24_NM(4, 4, true)
  ST24_NM(1, 8, true) ST24_NM(2, 8, true) ST24_NM(3, 8, true) ST24_NM(4, 8, true)
#undef ST24_NM
  return false;
}

// The 8-bit element types' launch (prune_nm_8.cu).
bool launch_nm_8bit(int dt, int n, int m, bool two, const void* W, int64_t M, int64_t K, int64_t ldw, void* values,
                    void* meta, int num_sms, cudaStream_t stream);

}  // namespace prune
}  // namespace st24
