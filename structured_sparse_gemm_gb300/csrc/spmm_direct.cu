// spmm_direct.cu -- decode-shaped products (N <= 32), every input type:
// C = alpha * row_scale * (A_sparse * B) + beta * C on the warp-level sparse
// MMA (mma.sp::ordered_metadata m16n8k32, f16/bf16), with the compressed
// weights loaded straight from HBM into registers.  8-bit inputs (e4m3,
// int8) are widened to f16 in registers, exactly (every e4m3 and int8 value
// is an f16 value), and take the f16 MMA: on this GPU the warp-level e4m3
// sparse MMA runs at ~1/50 and the int8 one at ~1/3 of the f16 rate.
//
// Method ("Chapter 26 -- Sparsity: The Hardware View", sections "2:4
// Fine-Grained Structured Sparsity" and "2:4 in the Memory-Bound Regime"):
// each group's metadata picks the two activations its two stored weights
// multiply; for small N the product is bound by streaming the compressed
// weights (values + metadata, ~56% of the dense bytes), so the kernel is built
// to keep as many of those bytes in flight as it can and to add little after
// they land.
//
// Structure:
//  * A 128-row tile is split along K over S = 1, 2, 4 or 8 CTAs, which form a
//    thread-block cluster.  Each of a CTA's 8 warps owns a 16-row slab and
//    streams that slab's values and metadata for the CTA's K-range in rounds
//    of 8 windows: every lane issues all of its 16-byte loads of a round at
//    once (into registers; no shared-memory ring), then the round's B by
//    bulk copies (TMA), which do not queue behind those loads.  With ST24_SPMM_FIXED_A the first round's weight loads
//    are issued before the grid-dependency wait, while the previous kernel
//    on the stream finishes (measured 0.5-1 us faster per launch).
//  * K order inside the MMA: within each window (64 K of 16-bit or 128 K of
//    8-bit values: one 16-byte load per lane and row), the groups are handed
//    to the MMA in the order that lets a lane's 16-byte load of a row (the
//    kept pairs of 4 or 8 consecutive groups) feed two or four MMAs
//    directly.  B (staged in shared memory once per round) and the metadata
//    are permuted the same way, so every product meets its own activation and
//    the sum is unchanged.
//  * Each warp's partial slab goes to the shared memory of the cluster CTA
//    that finishes that slab (st.async, counted on that CTA's mbarrier); that
//    CTA sums the S partials in K order (deterministic) and applies the
//    epilogue.  No CTA waits for the whole cluster at the end.
#include "st24_epilogue.cuh"

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <type_traits>

namespace st24 {
namespace direct {

constexpr int kWarps = 8;              // 16-row slabs per CTA
constexpr int kThreads = kWarps * 32;
constexpr int kBM = 16 * kWarps;       // rows per tile
constexpr int kWPW = 8;                // windows per warp per round

// Per input type: ES bytes per value; a window is the logical K of one
// 16-byte load of a row (32 bytes of groups' kept pairs per 4 lanes).
template <int DT>
struct Shape {
  static constexpr int ES = (DT == kF16 || DT == kBF16) ? 2 : 1;
  static constexpr bool k8 = ES == 1;
  static constexpr bool kInt = DT == kS8;
  static constexpr int WK = 64 * (2 / ES);       // logical K per window
  static constexpr int MPW = 2 * (2 / ES);       // MMAs (k32) per window
  static constexpr int ROUND_K = kWPW * WK;      // logical K per round
  static constexpr int META_V4 = 2 / ES;         // 16-byte metadata loads per row and lane
  static constexpr int MMA_DT = k8 ? kF16 : DT;  // type the MMA takes
};

struct Params : OutParams {
  const uint8_t* values;   // M x K/2 values, row-major
  const uint8_t* meta;     // M x K/8 bytes, canonical nibbles
  const uint8_t* B;        // element (k, n) at byte ES * (n * ldb + k)
  int64_t K, ldb_bytes;
  int parts;               // CTAs per tile (cluster size): 1, 2, 4 or 8
  int rounds;              // rounds per CTA
  int a_fixed;             // issue the first round's weight loads before the grid-dependency wait
  unsigned* status;        // device status word (a bounded wait that ran out)
};

// 16-byte load cached in L2 only (streamed once; coherent with earlier grids).
__device__ __forceinline__ uint4 ld_cg_v4(const void* ptr) {
  uint4 v;
  asm volatile("ld.global.cg.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(ptr));
  return v;
}

__device__ __forceinline__ uint32_t word_of(const uint4& v, int i) {
  return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

// Two 8-bit values (low byte first) as an f16x2 word, exactly.
template <int DT>
__device__ __forceinline__ uint32_t widen2(uint32_t two) {
  if constexpr (DT == kE4M3) {
    const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two & 0xFFFFu), __NV_E4M3);
    return static_cast<uint32_t>(h.x) | (static_cast<uint32_t>(h.y) << 16);
  } else {
    // int8 b as the f16 1024 + (b + 128) (its byte in the low mantissa bits),
    // minus 1152.
    const uint32_t w = __byte_perm(two ^ 0x8080u, 0x64646464u, 0x5140u);
    const __half2 d = __hsub2(*reinterpret_cast<const __half2*>(&w), __floats2half2_rn(1152.0f, 1152.0f));
    return *reinterpret_cast<const uint32_t*>(&d);
  }
}

// Metadata nibbles of one MMA's 4 groups, from 4 bytes holding them (byte i
// = group i's byte): the low nibbles (sh = 0) or the high nibbles (sh = 4),
// packed with group 0 in the lowest nibble, for rows g (bits 0-15) and g+8
// (bits 16-31).
__device__ __forceinline__ uint32_t pack_meta(uint32_t ug, uint32_t uh, int sh) {
  uint32_t vg = (ug >> sh) & 0x0F0F0F0Fu;
  uint32_t vh = (uh >> sh) & 0x0F0F0F0Fu;
  vg |= vg >> 4;   // bytes 0 and 2 now hold nibble pairs (0,1) and (2,3)
  vh |= vh >> 4;
  return __byte_perm(vg, vh, 0x6420u);
}

// Dynamic shared memory of one CTA: B of a round as loaded (natural order,
// NR columns of 1 KB), B in fragment order as f16/bf16 (NR columns of
// ROUND_K * 2 bytes), the partial slabs pushed to this CTA (8 slots x NT x
// 512 B), the reduction barrier and the B barrier.
template <int DT, int NT>
struct Smem {
  static constexpr int NR = 8 * NT;
  static constexpr int NAT = 0;
  static constexpr int FRAG = NAT + NR * 1024;
  static constexpr int PART = FRAG + NR * Shape<DT>::ROUND_K * 2;
  static constexpr int BAR = PART + kWarps * NT * 512;
  static constexpr int BYTES = BAR + 16;
};

template <int DT, int NT>
__global__ void __launch_bounds__(kThreads, 2) spmm_direct_kernel(const Params p) {
  using Sh = Shape<DT>;
  using L = Smem<DT, NT>;
  using Acc = typename std::conditional<Sh::kInt, int, float>::type;
  constexpr int NR = L::NR;                                 // B columns of the fragment layout (only n < N staged)
  // Independent accumulator chains (fewer for 8-bit inputs: four MMAs per
  // window already, and the registers go to the metadata and int sums).
  constexpr int KACC = Sh::k8 ? (NT == 1 && !Sh::kInt ? 2 : 1) : (NT == 1 ? 4 : (NT == 2 ? 2 : 1));
  constexpr int MPW = Sh::MPW, WK = Sh::WK, ES = Sh::ES;
  extern __shared__ __align__(16) uint8_t smem[];
  uint8_t* sBn = smem + L::NAT;                                        // [column][round, as loaded]
  uint32_t* sB = reinterpret_cast<uint32_t*>(smem + L::FRAG);          // [window][mma][column][lane % 4][4 words]
  float4* sP = reinterpret_cast<float4*>(smem + L::PART);              // [slot][n8 tile][lane]
  uint64_t* red_bar = reinterpret_cast<uint64_t*>(smem + L::BAR);
  uint64_t* b_bar = red_bar + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gid = lane >> 2, t = lane & 3;
  const int S = p.parts;
  const int r = S > 1 ? static_cast<int>(cluster_ctarank()) : 0;
  const int64_t tile = blockIdx.x / S;
  const int64_t K = p.K;
  const int N = static_cast<int>(p.N);
  const int64_t rowA = tile * kBM + warp * 16 + gid, rowB = rowA + 8;
  const bool inA = rowA < p.M, inB = rowB < p.M;
  const int64_t k_begin = static_cast<int64_t>(r) * p.rounds * Sh::ROUND_K;
  // Byte offsets: logical k sits at byte k * ES / 2 of a values row (two
  // kept values per group of 4) and at byte k / 8 of a metadata row.
  const uint8_t* va = p.values + rowA * (K * ES / 2) + 16 * t;
  const uint8_t* vb = va + 8 * (K * ES / 2);
  const uint8_t* ma = p.meta + rowA * (K / 8) + 16 * Sh::META_V4 * t;
  const uint8_t* mb = ma + K;   // 8 rows down: 8 * K / 8 bytes
  const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
  const uint4 pair01 = make_uint4(0x44444444u, 0x44444444u, 0x44444444u, 0x44444444u);

  if (threadIdx.x == 0) {
    grid_launch_dependents();
    // B barrier: one phase per round.  Reduction barrier (clusters): this CTA
    // receives 8 slots of NT x 512 bytes.
    mbar_init(smem_u32(b_bar), 1);
    mbar_init(smem_u32(red_bar), 1);
    fence_barrier_init();
    if (S > 1) mbar_arrive_expect_tx(smem_u32(red_bar), kWarps * NT * 512);
  }
  __syncthreads();
  if (S > 1) cluster_arrive_release();   // waited on before the first DSMEM store

  float acc[KACC][NT][4];
  Acc iacc[NT][4];   // int8: the exact running sums (unused otherwise)
#pragma unroll
  for (int i = 0; i < NT; ++i)
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      iacc[i][x] = 0;
#pragma unroll
      for (int u = 0; u < KACC; ++u) acc[u][i][x] = 0.0f;
    }
  const int sh = (t & 1) * 4;

  for (int ro = 0; ro < p.rounds; ++ro) {
    const int64_t kr = k_begin + static_cast<int64_t>(ro) * Sh::ROUND_K;
    if (ro > 0) __syncthreads();   // every warp is done with the previous round's B
    if (ro == 0 && !p.a_fixed) grid_dependency_wait();   // inputs may come from the previous kernel
    // The weights: lane (g, t) loads, for each window j, the kept pairs of
    // its 16 bytes of the window (groups 4t..4t+3, or 8t..8t+7 for 8-bit
    // values) in rows g and g+8, and the metadata of windows 2t, 2t+1 of
    // both rows.  Rows past M and windows past K read nothing: zero values
    // with a valid index pair.
    uint4 ra[kWPW], rb[kWPW];
#pragma unroll
    for (int j = 0; j < kWPW; ++j) {
      const int64_t k = kr + WK * j;
      ra[j] = (inA && k < K) ? ld_cg_v4(va + k * ES / 2) : zero;
      rb[j] = (inB && k < K) ? ld_cg_v4(vb + k * ES / 2) : zero;
    }
    uint4 mg[Sh::META_V4], mh[Sh::META_V4];
#pragma unroll
    for (int v = 0; v < Sh::META_V4; ++v) {
      // 16-bit: one load holds windows 2t and 2t+1; 8-bit: load v holds window 2t+v.
      const bool kin = kr + WK * (2 * t + v) < K;
      mg[v] = (inA && kin) ? ld_cg_v4(ma + kr / 8 + 16 * v) : pair01;
      mh[v] = (inB && kin) ? ld_cg_v4(mb + kr / 8 + 16 * v) : pair01;
    }
    if (ro == 0 && p.a_fixed) grid_dependency_wait();    // the weights are in flight already

    // Then B: columns n < N of the round as they lie in memory, one bulk
    // copy (TMA) per column, so they do not queue behind the weights' loads;
    // the part of a round past K is zero.
    const int64_t kv = K - kr < Sh::ROUND_K ? (K - kr > 0 ? K - kr : 0) : Sh::ROUND_K;   // valid K of the round
    if (threadIdx.x == 0) {
      fence_proxy_async_smem();   // earlier reads of the staging area come before the copies' writes
      if (kv > 0) {
        mbar_arrive_expect_tx(smem_u32(b_bar), static_cast<uint32_t>(N * ES * kv));
        for (int n = 0; n < N; ++n)
          bulk_load(smem_u32(sBn + n * 1024), p.B + n * p.ldb_bytes + ES * kr, static_cast<uint32_t>(ES * kv),
                    smem_u32(b_bar));
      } else {
        mbar_arrive(smem_u32(b_bar));
      }
    }
    const int chunks = N * 64;   // 16-byte chunks of the staged columns
    for (int c = threadIdx.x; c < chunks; c += kThreads)
      if (kr + (c % 64) * (16 / ES) >= K) *reinterpret_cast<uint4*>(sBn + 16 * c) = zero;

    // B into fragment order (and, for 8-bit inputs, f16), columns n < N only.  Values (k, k+1)
    // of column n at K offset kk = WK j + 4 G + e (group G of window j,
    // element e even) are MMA mp's word jj of lane t, with G split as
    // G = 2 MPW (2 h + a) + 2 mp + s:  jj = h + 2 s, t = 2 a + e / 2.
    mbar_wait(smem_u32(b_bar), static_cast<uint32_t>(ro & 1), p.status);   // (a timeout is reported; the round goes on)
    __syncthreads();
    for (int c = threadIdx.x; c < chunks; c += kThreads) {
      const int n = c / 64, q = c % 64;
      const uint4 v = *reinterpret_cast<const uint4*>(sBn + 16 * c);
#pragma unroll
      for (int u = 0; u < 8 / ES; ++u) {   // value pairs of the chunk
        uint32_t wv;
        if constexpr (ES == 2)
          wv = word_of(v, u);
        else
          wv = widen2<DT>(word_of(v, u >> 1) >> (16 * (u & 1)));
        const int kk = q * (16 / ES) + 2 * u;
        const int j = kk / WK, kw = kk % WK;
        const int G = kw >> 2, e = kw & 3;
        const int s = G & 1, mp = (G >> 1) % MPW, a = (G / (2 * MPW)) & 1, h = G / (4 * MPW);
        const int tt = 2 * a + (e >> 1), jj = h + 2 * s;
        sB[(((j * MPW + mp) * NR + n) * 4 + tt) * 4 + jj] = wv;
      }
    }
    __syncthreads();

#pragma unroll
    for (int j = 0; j < kWPW; ++j) {
      // Window j's metadata lives in lane (g, j / 2).
      const int src = 4 * gid + (j >> 1);
      uint32_t gw[4 / ES], hw[4 / ES];   // the window's metadata words: 2 (16-bit) or 4 (8-bit) per row
      if constexpr (ES == 2) {
        gw[0] = __shfl_sync(0xffffffffu, (j & 1) ? mg[0].z : mg[0].x, src);
        gw[1] = __shfl_sync(0xffffffffu, (j & 1) ? mg[0].w : mg[0].y, src);
        hw[0] = __shfl_sync(0xffffffffu, (j & 1) ? mh[0].z : mh[0].x, src);
        hw[1] = __shfl_sync(0xffffffffu, (j & 1) ? mh[0].w : mh[0].y, src);
      } else {
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          gw[w] = __shfl_sync(0xffffffffu, word_of(mg[j & 1], w), src);
          hw[w] = __shfl_sync(0xffffffffu, word_of(mh[j & 1], w), src);
        }
      }
#pragma unroll
      for (int mp = 0; mp < MPW; ++mp) {
        // MMA mp takes, as its groups 0-3, the window's groups
        // 2 MPW v + 2 mp (v = 0..3: the low nibbles of bytes MPW v + mp) and,
        // as its groups 4-7, the next group of each (the high nibbles).
        uint32_t ug, uh;
        if constexpr (ES == 2) {
          const uint32_t sel = mp ? 0x7531u : 0x6420u;
          ug = __byte_perm(gw[0], gw[1], sel);
          uh = __byte_perm(hw[0], hw[1], sel);
        } else {
          const uint32_t sel = static_cast<uint32_t>(mp | ((mp + 4) << 4));
          ug = __byte_perm(__byte_perm(gw[0], gw[1], sel), __byte_perm(gw[2], gw[3], sel), 0x5410u);
          uh = __byte_perm(__byte_perm(hw[0], hw[1], sel), __byte_perm(hw[2], hw[3], sel), 0x5410u);
        }
        const uint32_t e = pack_meta(ug, uh, sh);
        // MMA mp: its group t is the kept pair of the lane's load in word
        // 2 mp (16-bit) or in the low half of word mp (8-bit), its group
        // t + 4 the pair after it; rows g and g+8.
        uint32_t a[4];
        if constexpr (ES == 2) {
          a[0] = word_of(ra[j], 2 * mp); a[1] = word_of(rb[j], 2 * mp);
          a[2] = word_of(ra[j], 2 * mp + 1); a[3] = word_of(rb[j], 2 * mp + 1);
        } else {
          a[0] = widen2<DT>(word_of(ra[j], mp)); a[1] = widen2<DT>(word_of(rb[j], mp));
          a[2] = widen2<DT>(word_of(ra[j], mp) >> 16); a[3] = widen2<DT>(word_of(rb[j], mp) >> 16);
        }
#pragma unroll
        for (int i = 0; i < NT; ++i) {
          // columns past N multiply as zeros (their slots are never staged)
          const uint4 bv = i * 8 + gid < N
                               ? *reinterpret_cast<const uint4*>(&sB[(((j * MPW + mp) * NR + i * 8 + gid) * 4 + t) * 4])
                               : zero;
          const uint32_t b[4] = {bv.x, bv.y, bv.z, bv.w};
          mma_sp_16832<Sh::MMA_DT>(acc[(MPW * j + mp) % KACC][i], a, b, e);
        }
      }
      if constexpr (Sh::kInt) {
        // Move the window's exact integer sums into int32.
#pragma unroll
        for (int u = 0; u < KACC; ++u)
#pragma unroll
          for (int i = 0; i < NT; ++i)
#pragma unroll
            for (int x = 0; x < 4; ++x) {
              iacc[i][x] += __float2int_rn(acc[u][i][x]);
              acc[u][i][x] = 0.0f;
            }
      }
    }
  }

  // This CTA's partial of its slab: the accumulator chains summed in a fixed order.
  Acc tot[NT][4];
#pragma unroll
  for (int i = 0; i < NT; ++i)
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      if constexpr (Sh::kInt) {
        tot[i][x] = iacc[i][x];
      } else {
        float v = acc[0][i][x];
#pragma unroll
        for (int u = 1; u < KACC; ++u) v += acc[u][i][x];
        tot[i][x] = v;
      }
    }

  // Slab w is finished by CTA w % S of the cluster; this CTA's partial of it
  // goes to that CTA's slot (w / S) * S + r.  In a cluster the partials move
  // by st.async, counted on the owner's reduction barrier: no CTA waits for
  // the others to finish, only the owner for what it sums.
  const int per = kWarps / S;   // slabs this CTA finishes
  {
    const int owner = warp % S, slot = (warp / S) * S + r;
    if (S > 1) cluster_wait();   // every CTA of the cluster has started and set up its barrier
#pragma unroll
    for (int i = 0; i < NT; ++i) {
      float4 v;
      if constexpr (Sh::kInt)
        v = make_float4(__int_as_float(tot[i][0]), __int_as_float(tot[i][1]), __int_as_float(tot[i][2]),
                        __int_as_float(tot[i][3]));
      else
        v = make_float4(tot[i][0], tot[i][1], tot[i][2], tot[i][3]);
      if (S > 1)
        st_async_cluster_f4(&sP[(slot * NT + i) * 32 + lane], red_bar, static_cast<uint32_t>(owner), v);
      else
        sP[(slot * NT + i) * 32 + lane] = v;
    }
  }
  if (S == 1) __syncthreads();    // (every warp has epilogue work when S = 1: per * NT >= 8)
  if (warp >= per * NT) return;   // no epilogue work in this warp
  if (S > 1 && !mbar_wait_cluster(smem_u32(red_bar), 0u, p.status)) return;

  // Epilogue for the slabs this CTA finishes: (slab, n8 tile) pairs over the warps.
  for (int pr = warp; pr < per * NT; pr += kWarps) {
    const int si = pr / NT, i = pr % NT;
    const int w = r + si * S;
    Acc v[4];
    for (int q = 0; q < S; ++q) {   // K order
      const float4 f = sP[((si * S + q) * NT + i) * 32 + lane];
      Acc fv[4];
      if constexpr (Sh::kInt) {
        fv[0] = __float_as_int(f.x); fv[1] = __float_as_int(f.y); fv[2] = __float_as_int(f.z); fv[3] = __float_as_int(f.w);
      } else {
        fv[0] = f.x; fv[1] = f.y; fv[2] = f.z; fv[3] = f.w;
      }
#pragma unroll
      for (int x = 0; x < 4; ++x) v[x] = (q == 0) ? fv[x] : v[x] + fv[x];
    }
    const int64_t m_lo = tile * kBM + 16 * w + gid, n_lo = 8 * i + 2 * t;
    float bc[4];
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      const int64_t m = m_lo + 8 * (x >> 1), n = n_lo + (x & 1);
      bc[x] = (m < p.M && n < p.N && p.c_type != kS32) ? load_beta_c(p, m, n) : 0.0f;
    }
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      const int64_t m = m_lo + 8 * (x >> 1), n = n_lo + (x & 1);
      if (m < p.M && n < p.N) store_out<Acc>(p, m, n, v[x], p.c_type == kS32 ? 1.0f : row_factor(p, m), bc[x]);
    }
  }
}

// CTAs per tile (a power of two up to 8) and rounds per CTA.
void split_k(int64_t K, int64_t round_k, int& parts, int& rounds) {
  const int64_t need = (K + round_k - 1) / round_k;
  parts = need <= 1 ? 1 : (need <= 2 ? 2 : (need <= 4 ? 4 : 8));
  rounds = static_cast<int>((K + round_k * parts - 1) / (round_k * parts));
}

template <int DT, int NT>
st24_status launch_nt(const Params& p, int64_t tiles, const DeviceInfo& dev, cudaStream_t stream) {
  auto kern = spmm_direct_kernel<DT, NT>;
  static bool attr_set[64] = {};
  if (!attr_set[dev.device % 64]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Smem<DT, NT>::BYTES) != cudaSuccess)
      return ST24_ERR_CUDA;
    attr_set[dev.device % 64] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(tiles * p.parts));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Smem<DT, NT>::BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attrs[2];
  int n = 0;
  attrs[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (p.parts > 1) {
    attrs[n].id = cudaLaunchAttributeClusterDimension;
    attrs[n].val.clusterDim.x = static_cast<unsigned>(p.parts);
    attrs[n].val.clusterDim.y = 1;
    attrs[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attrs;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, p) == cudaSuccess ? ST24_OK : ST24_ERR_CUDA;
}

template <int DT>
st24_status launch_dt(const SpmmArgs& a, const DeviceInfo& dev, cudaStream_t stream) {
  Params p{};
  p.M = a.M;
  p.N = a.N;
  p.alpha = a.alpha;
  p.beta = a.beta;
  p.C = a.C;
  p.ldc = a.ldc;
  p.c_type = a.c;
  p.row_scale = a.row_scale;
  p.values = static_cast<const uint8_t*>(a.values);
  p.meta = static_cast<const uint8_t*>(a.meta);
  p.B = static_cast<const uint8_t*>(a.B);
  p.K = a.K;
  p.ldb_bytes = a.ldb * Shape<DT>::ES;
  p.a_fixed = (a.flags & ST24_SPMM_FIXED_A) ? 1 : 0;
  p.status = dev.status;
  split_k(a.K, Shape<DT>::ROUND_K, p.parts, p.rounds);
  const int64_t tiles = (a.M + kBM - 1) / kBM;
  if (a.N <= 8) return launch_nt<DT, 1>(p, tiles, dev, stream);
  if (a.N <= 16) return launch_nt<DT, 2>(p, tiles, dev, stream);
  return launch_nt<DT, 4>(p, tiles, dev, stream);
}

}  // namespace direct

bool direct_applies(const SpmmArgs& a) {
  return (a.ab == kF16 || a.ab == kBF16 || a.ab == kE4M3 || a.ab == kS8) && a.N >= 1 && a.N <= 32 &&
         (a.M + direct::kBM - 1) / direct::kBM * 8 <= 0x7fffffff;
}

bool direct_one_wave(const SpmmArgs& a, int num_sms) {
  int parts = 1, rounds = 1;
  const bool k8 = a.ab == kE4M3 || a.ab == kS8;
  direct::split_k(a.K, k8 ? direct::Shape<kS8>::ROUND_K : direct::Shape<kBF16>::ROUND_K, parts, rounds);
  return (a.M + direct::kBM - 1) / direct::kBM * parts <= 2 * static_cast<int64_t>(num_sms);
}

st24_status launch_spmm_direct(const SpmmArgs& a, const DeviceInfo& dev, cudaStream_t stream) {
  if (!direct_applies(a)) return ST24_ERR_UNSUPPORTED;
  switch (a.ab) {
    case kF16: return direct::launch_dt<kF16>(a, dev, stream);
    case kBF16: return direct::launch_dt<kBF16>(a, dev, stream);
    case kE4M3: return direct::launch_dt<kE4M3>(a, dev, stream);
    default: return direct::launch_dt<kS8>(a, dev, stream);
  }
}

}  // namespace st24
