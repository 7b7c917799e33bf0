// spmm_direct.cu -- decode-shaped products, 16-bit inputs, N <= 32:
// C = alpha * row_scale * (A_sparse * B) + beta * C on the warp-level sparse
// MMA (mma.sp::ordered_metadata m16n8k32), with the compressed weights
// loaded straight from HBM into registers.
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
//    of 512 K: every lane issues all 18 of its 16-byte loads of a round at
//    once (into registers; no shared-memory ring), then the round's B by
//    bulk copies (TMA), which do not queue behind those loads.  With ST24_SPMM_FIXED_A the first round's weight loads
//    are issued before the grid-dependency wait, while the previous kernel
//    on the stream finishes (measured 0.5-1 us faster per launch).
//  * K order inside the MMA: within each 64-K window (16 groups of 4), the
//    groups are handed to the MMA in the order that lets one lane's 16-byte
//    load of a row (the kept pairs of 4 consecutive groups) feed two MMAs
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

namespace st24 {
namespace direct {

constexpr int kWarps = 8;              // 16-row slabs per CTA
constexpr int kThreads = kWarps * 32;
constexpr int kBM = 16 * kWarps;       // rows per tile
constexpr int kWPW = 8;                // 64-K windows per warp per round
constexpr int kRoundK = 64 * kWPW;     // logical K per round

struct Params : OutParams {
  const uint8_t* values;   // M x K/2 16-bit values, row-major
  const uint8_t* meta;     // M x K/8 bytes, canonical nibbles
  const uint8_t* B;        // element (k, n) at byte 2 * (n * ldb + k)
  int64_t K, ldb_bytes;
  int parts;               // CTAs per tile (cluster size): 1, 2, 4 or 8
  int rounds;              // 512-K rounds per CTA
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

// Metadata word of one MMA of a window for this lane, from the window's 8
// metadata bytes of row g (lo, hi words) and of row g+8.  MMA p takes groups
// 2p, 2p+4, 2p+8, 2p+12 of the window as its groups 0-3 (the low nibbles of
// bytes p, p+2, p+4, p+6) and groups 2p+1, 2p+5, ... as its groups 4-7 (the
// high nibbles).  Lane 4g supplies groups 0-3 (row g in bits 0-15, row g+8 in
// bits 16-31), lane 4g+1 groups 4-7: `sh` is 0 or 4 accordingly.
__device__ __forceinline__ uint32_t window_meta(uint32_t g_lo, uint32_t g_hi, uint32_t h_lo, uint32_t h_hi,
                                                int p, int sh) {
  const uint32_t sel = p ? 0x7531u : 0x6420u;
  uint32_t vg = (__byte_perm(g_lo, g_hi, sel) >> sh) & 0x0F0F0F0Fu;
  uint32_t vh = (__byte_perm(h_lo, h_hi, sel) >> sh) & 0x0F0F0F0Fu;
  vg |= vg >> 4;   // bytes 0 and 2 now hold nibble pairs (0,1) and (2,3)
  vh |= vh >> 4;
  return __byte_perm(vg, vh, 0x6420u);
}

// Dynamic shared memory of one CTA: B of a round as loaded (natural order,
// NR columns of 1 KB), B in fragment order (NR x 1 KB), the partial slabs
// pushed to this CTA (8 slots x NT x 512 B) and the reduction barrier.
template <int NT>
struct Smem {
  static constexpr int NR = 8 * NT;
  static constexpr int NAT = 0;
  static constexpr int FRAG = NAT + NR * 1024;
  static constexpr int PART = FRAG + NR * 1024;
  static constexpr int BAR = PART + kWarps * NT * 512;   // reduction barrier, then B barrier
  static constexpr int BYTES = BAR + 16;
};

template <int DT, int NT>
__global__ void __launch_bounds__(kThreads, 2) spmm_direct_kernel(const Params p) {
  using L = Smem<NT>;
  constexpr int NR = L::NR;                                 // B columns staged (zero past N)
  constexpr int KACC = NT == 1 ? 4 : (NT == 2 ? 2 : 1);     // independent accumulator chains
  extern __shared__ __align__(16) uint8_t smem[];
  uint8_t* sBn = smem + L::NAT;                                        // [column][512 K]
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
  const int64_t k_begin = static_cast<int64_t>(r) * p.rounds * kRoundK;
  // Byte offsets: logical k sits at byte k of a values row (two 2-byte values
  // per group of 4), and at byte k / 8 of a metadata row.
  const uint8_t* va = p.values + rowA * K + 16 * t;
  const uint8_t* vb = va + 8 * K;
  const uint8_t* ma = p.meta + rowA * (K / 8) + 16 * t;
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
#pragma unroll
  for (int u = 0; u < KACC; ++u)
#pragma unroll
    for (int i = 0; i < NT; ++i)
#pragma unroll
      for (int x = 0; x < 4; ++x) acc[u][i][x] = 0.0f;
  const int sh = (t & 1) * 4;

  for (int ro = 0; ro < p.rounds; ++ro) {
    const int64_t kr = k_begin + static_cast<int64_t>(ro) * kRoundK;
    if (ro > 0) __syncthreads();   // every warp is done with the previous round's B
    if (ro == 0 && !p.a_fixed) grid_dependency_wait();   // inputs may come from the previous kernel
    // The weights: lane (g, t) loads, for each window j, the kept pairs of
    // groups 4t..4t+3 of the window in rows g and g+8, and the metadata of
    // windows 2t, 2t+1 of both rows.  Rows past M and windows past K read
    // nothing: zero values with a valid index pair.
    uint4 ra[kWPW], rb[kWPW];
#pragma unroll
    for (int j = 0; j < kWPW; ++j) {
      const int64_t k = kr + 64 * j;
      ra[j] = (inA && k < K) ? ld_cg_v4(va + k) : zero;
      rb[j] = (inB && k < K) ? ld_cg_v4(vb + k) : zero;
    }
    const bool kin = kr + 128 * t < K;
    const uint4 mg = (inA && kin) ? ld_cg_v4(ma + kr / 8) : pair01;
    const uint4 mh = (inB && kin) ? ld_cg_v4(mb + kr / 8) : pair01;
    if (ro == 0 && p.a_fixed) grid_dependency_wait();    // the weights are in flight already
    // Then B: columns n < N of the round as they lie in memory, one bulk
    // copy (TMA) per column, so they do not queue behind the weights' loads;
    // the part of a round past K is zero.
    const int64_t kv = K - kr < kRoundK ? (K - kr > 0 ? K - kr : 0) : kRoundK;   // valid K of the round
    if (threadIdx.x == 0) {
      fence_proxy_async_smem();   // earlier reads of the staging area come before the copies' writes
      if (kv > 0) {
        mbar_arrive_expect_tx(smem_u32(b_bar), static_cast<uint32_t>(N * 2 * kv));
        for (int n = 0; n < N; ++n)
          bulk_load(smem_u32(sBn + n * 1024), p.B + n * p.ldb_bytes + 2 * kr, static_cast<uint32_t>(2 * kv),
                    smem_u32(b_bar));
      } else {
        mbar_arrive(smem_u32(b_bar));
      }
    }
    const int chunks = N * (kRoundK / 8);
    for (int c = threadIdx.x; c < chunks; c += kThreads)
      if (kr + 8 * (c % (kRoundK / 8)) >= K) *reinterpret_cast<uint4*>(sBn + 16 * c) = zero;

    // B into fragment order.  Word (k, k+1) of column n, at K offset
    // kk = 64 j + 4 G + 2 e (group G of window j, half e), is MMA
    // p = (G >> 1) & 1's word jj = (G >> 3) + 2 (G & 1) of lane
    // t = 2 ((G >> 2) & 1) + e.  Columns N..NR-1 are zero.
    mbar_wait(smem_u32(b_bar), static_cast<uint32_t>(ro & 1), p.status);   // (a timeout is reported; the round goes on)
    __syncthreads();
    for (int c = threadIdx.x; c < chunks; c += kThreads) {
      const int n = c / (kRoundK / 8), q = c % (kRoundK / 8);
      const uint4 v = *reinterpret_cast<const uint4*>(sBn + 16 * c);
      const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int kk = 8 * q + 2 * u;
        const int j = kk >> 6, G = (kk & 63) >> 2, e = (kk >> 1) & 1;
        const int mp = (G >> 1) & 1, tt = 2 * ((G >> 2) & 1) + e, jj = (G >> 3) + 2 * (G & 1);
        sB[(((j * 2 + mp) * NR + n) * 4 + tt) * 4 + jj] = w4[u];
      }
    }
    const int pad = (NR - N) * 16;   // words of the zero columns, per (window, mma)
    for (int c = threadIdx.x; c < kWPW * 2 * pad; c += kThreads) sB[(c / pad) * NR * 16 + N * 16 + c % pad] = 0u;
    __syncthreads();

#pragma unroll
    for (int j = 0; j < kWPW; ++j) {
      // Window j's metadata lives in lane (g, j / 2).
      const int src = 4 * gid + (j >> 1);
      const uint32_t g_lo = __shfl_sync(0xffffffffu, (j & 1) ? mg.z : mg.x, src);
      const uint32_t g_hi = __shfl_sync(0xffffffffu, (j & 1) ? mg.w : mg.y, src);
      const uint32_t h_lo = __shfl_sync(0xffffffffu, (j & 1) ? mh.z : mh.x, src);
      const uint32_t h_hi = __shfl_sync(0xffffffffu, (j & 1) ? mh.w : mh.y, src);
#pragma unroll
      for (int mp = 0; mp < 2; ++mp) {
        const uint32_t e = window_meta(g_lo, g_hi, h_lo, h_hi, mp, sh);
        // MMA mp: its group t is the lane's group 4t + 2mp, its group t + 4 the
        // lane's group 4t + 2mp + 1; rows g and g+8.
        const uint32_t a[4] = {mp ? ra[j].z : ra[j].x, mp ? rb[j].z : rb[j].x, mp ? ra[j].w : ra[j].y,
                               mp ? rb[j].w : rb[j].y};
#pragma unroll
        for (int i = 0; i < NT; ++i) {
          const uint4 bv = *reinterpret_cast<const uint4*>(&sB[(((j * 2 + mp) * NR + i * 8 + gid) * 4 + t) * 4]);
          const uint32_t b[4] = {bv.x, bv.y, bv.z, bv.w};
          mma_sp_16832<DT>(acc[(2 * j + mp) % KACC][i], a, b, e);
        }
      }
    }
  }

  // Sum the accumulator chains in a fixed order.
#pragma unroll
  for (int u = 1; u < KACC; ++u)
#pragma unroll
    for (int i = 0; i < NT; ++i)
#pragma unroll
      for (int x = 0; x < 4; ++x) acc[0][i][x] += acc[u][i][x];

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
      const float4 v = make_float4(acc[0][i][0], acc[0][i][1], acc[0][i][2], acc[0][i][3]);
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
    float v[4];
#pragma unroll
    for (int x = 0; x < 4; ++x) v[x] = 0.0f;
    for (int q = 0; q < S; ++q) {   // K order
      const float4 f = sP[((si * S + q) * NT + i) * 32 + lane];
      if (q == 0) {
        v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
      } else {
        v[0] += f.x; v[1] += f.y; v[2] += f.z; v[3] += f.w;
      }
    }
    const int64_t m_lo = tile * kBM + 16 * w + gid, n_lo = 8 * i + 2 * t;
    float bc[4];
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      const int64_t m = m_lo + 8 * (x >> 1), n = n_lo + (x & 1);
      bc[x] = (m < p.M && n < p.N) ? load_beta_c(p, m, n) : 0.0f;
    }
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      const int64_t m = m_lo + 8 * (x >> 1), n = n_lo + (x & 1);
      if (m < p.M && n < p.N) store_out<float>(p, m, n, v[x], row_factor(p, m), bc[x]);
    }
  }
}

// CTAs per tile (a power of two up to 8) and 512-K rounds per CTA.
void split_k(int64_t K, int& parts, int& rounds) {
  const int64_t need = (K + kRoundK - 1) / kRoundK;
  parts = need <= 1 ? 1 : (need <= 2 ? 2 : (need <= 4 ? 4 : 8));
  rounds = static_cast<int>((K + static_cast<int64_t>(kRoundK) * parts - 1) / (static_cast<int64_t>(kRoundK) * parts));
}

template <int DT, int NT>
st24_status launch_nt(const Params& p, int64_t tiles, const DeviceInfo& dev, cudaStream_t stream) {
  auto kern = spmm_direct_kernel<DT, NT>;
  static bool attr_set[64] = {};
  if (!attr_set[dev.device % 64]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Smem<NT>::BYTES) != cudaSuccess)
      return ST24_ERR_CUDA;
    attr_set[dev.device % 64] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(tiles * p.parts));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Smem<NT>::BYTES;
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
  p.ldb_bytes = a.ldb * 2;
  p.a_fixed = (a.flags & ST24_SPMM_FIXED_A) ? 1 : 0;
  p.status = dev.status;
  split_k(a.K, p.parts, p.rounds);
  const int64_t tiles = (a.M + kBM - 1) / kBM;
  if (a.N <= 8) return launch_nt<DT, 1>(p, tiles, dev, stream);
  if (a.N <= 16) return launch_nt<DT, 2>(p, tiles, dev, stream);
  return launch_nt<DT, 4>(p, tiles, dev, stream);
}

}  // namespace direct

bool direct_applies(const SpmmArgs& a) {
  return (a.ab == kF16 || a.ab == kBF16) && a.N >= 1 && a.N <= 32 &&
         (a.M + direct::kBM - 1) / direct::kBM * 8 <= 0x7fffffff;
}

st24_status launch_spmm_direct(const SpmmArgs& a, const DeviceInfo& dev, cudaStream_t stream) {
  if (!direct_applies(a)) return ST24_ERR_UNSUPPORTED;
  return a.ab == kF16 ? direct::launch_dt<kF16>(a, dev, stream) : direct::launch_dt<kBF16>(a, dev, stream);
}

}  // namespace st24
