// spmm_mmasp.cuh -- C = alpha * row_scale * (A_sparse * B) + beta * C on the
// warp-level sparse tensor-core instruction (mma.sp::ordered_metadata).
//
// Method ("Chapter 26 -- Sparsity: The Hardware View", section "2:4
// Fine-Grained Structured Sparsity"): the metadata of each group selects the
// two activations its two stored weights multiply; the other two products are
// zero and never computed.  A is streamed in its compressed form (values +
// metadata), so for small N the kernel reads ~56% of the dense weight bytes
// (section "2:4 in the Memory-Bound Regime").
//
// Structure (one CTA per SM, persistent):
//  * Schedule: stream-K.  The (output tile, k-block) iterations are flattened
//    and each CTA takes one contiguous run of them, so every SM streams the
//    same number of A bytes whatever the tile count.  A tile whose k-blocks
//    are spread over several CTAs is finished by whichever of them arrives
//    last: each writes its fp32 (or int32) partial tile to the workspace and
//    bumps the tile's counter; the last one sums the partials in k order
//    (deterministic), applies the epilogue and resets the counter.
//  * Producer warp: TMA loads of the compressed A tile (128-byte swizzle), the
//    A metadata tile and the B tile (128-byte swizzle) into a ring of stages
//    guarded by full/empty mbarriers.
//  * Consumer warps (4 x WARPS_N): ldmatrix fragments, mma.sp into registers.
//  * Epilogue: alpha, per-row scale, beta * C, rounding to the output type.
#pragma once
#include "st24_epilogue.cuh"

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

namespace st24 {
namespace mmasp {

// Per element type: 16-bit types use m16n8k32 (32 logical K per MMA, 128 per
// k-block); 8-bit types use m16n8k64 (64 per MMA, 256 per k-block).  Either
// way one k-block is 128 bytes of compressed A per row, 256 bytes of B per
// column, and EB bytes of metadata per row.
template <int DT>
struct Traits {
  static constexpr int ES = (DT == kF16 || DT == kBF16) ? 2 : 1;
  static constexpr int KSTEP = 64 / ES;      // logical K of one MMA
  static constexpr int BK = 4 * KSTEP;       // logical K of one k-block
  static constexpr int EB = BK / 8;          // metadata bytes per row per k-block
  static constexpr bool kInt = DT == kS8;
};

template <int DT, int BN_, int WARPS_N_, int STAGES_, int WMT_ = 2>
struct Config {
  using T = Traits<DT>;
  static constexpr int BM = 128;
  static constexpr int BN = BN_;
  static constexpr int WMT = WMT_;                    // m16 tiles per warp
  static constexpr int WARPS_M = BM / (16 * WMT_);
  static constexpr int WARPS_N = WARPS_N_;
  static constexpr int CONSUMERS = WARPS_M * WARPS_N;
  static constexpr int THREADS = (CONSUMERS + 1) * 32;
  static constexpr int WN = BN / 8 / WARPS_N;        // n8 tiles per warp
  static constexpr int STAGES = STAGES_;
  static constexpr int A_BYTES = BM * 128;
  static constexpr int B_BYTES = BN * 256;           // two 128-byte-wide boxes
  static constexpr int E_BYTES = BM * T::EB;
  static constexpr int STAGE_TX = A_BYTES + B_BYTES + E_BYTES;
  static constexpr int STAGE_BYTES = (STAGE_TX + 1023) / 1024 * 1024;
  static constexpr int PARTIAL_ELEMS = BM * BN;      // one fp32/int32 partial tile
  // In-cluster split-K: partial fragments pushed by the cluster's CTAs land
  // here (a region of its own, so no CTA has to wait for another to leave
  // its main loop before pushing).
  static constexpr int PUSH_BYTES = BN <= 64 ? BM * BN * 4 : 0;   // wide tiles never run in cluster mode
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + PUSH_BYTES + 1024 /*align*/ + 256 /*barriers*/;
  // Narrow (decode) tiles are sized so two CTAs fit on an SM: shared memory
  // below half the SM's, and registers within what the sub-partition holding
  // the most of the two CTAs' warps can give (16384 per sub-partition; e.g.
  // 168 for 2 x 5 warps, 96 for 2 x 9).
  static constexpr bool TWO_PER_SM = BN <= 32;
  // Independent accumulator sets per fragment (k-step ks feeds set ks % KACC,
  // summed in set order at the end of the tile's k-range).  A warp-level MMA
  // has a long latency on this GPU: with one set, the narrow tiles' few
  // fragments form a chain of 4 dependent MMAs per k-block, which bounded
  // the decode-shaped products.
  static constexpr int KACC = BN > 32 ? 1 : (WMT_ * WN >= 8 ? 1 : (WMT_ * WN >= 4 ? 2 : 4));
  static constexpr bool FRAGS_FIRST = BN <= 8;   // all of a stage's fragments in registers at once
  static constexpr int WARPS_2 = 2 * (CONSUMERS + 1);
  static constexpr int REGS_2 = (16384 / ((WARPS_2 + 3) / 4 * 32)) & ~7;
  static constexpr int MAX_REGS = TWO_PER_SM ? (REGS_2 < 168 ? REGS_2 : 168) : (THREADS > 256 ? 168 : 255);
  static_assert(WN >= 1 && BN % (8 * WARPS_N) == 0, "tile split");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
  static_assert(!TWO_PER_SM || 2 * (SMEM_BYTES + 1024) <= 228 * 1024, "two CTAs per SM");
};

struct Params : OutParams {
  int64_t K;
  int64_t tiles_m, tiles_n, group_m, k_iters, dp_tiles, sk_tiles;
  int a_evict_first;      // A is streamed once (by the tiles running at the same time): evict it first
  int b_evict_first;      // B likewise (the raster keeps the A panel resident instead)
  int a_fixed;            // A is not written by earlier work on the stream: load it before the dependency wait
  int b3d;                // tmB is 3-D (128-byte K chunk, row, chunk index): one copy per stage
  int64_t kb_wrap;        // two-form product: k-blocks per form (B's k-block of k-block kb is kb mod kb_wrap); 0: one form
  int cluster;            // > 1: the CTAs of each split tile form a cluster and reduce in shared memory
  float* partials;       // [2 * gridDim.x][PARTIAL_ELEMS]
  unsigned* counters;    // one per output tile
  unsigned* status;
};

__device__ __forceinline__ void consumer_sync(int threads) {
  asm volatile("bar.sync 1, %0;" ::"r"(threads) : "memory");
}

// Metadata register of lane `lane` for each k-step of an m16 tile whose rows
// start at `row0` in the stage's metadata block (EB bytes per row, canonical
// order: 8 groups per 32-bit word, lowest K in the lowest nibble).
// Lane layout of the metadata operand (sparsity selector 0), with g = lane/4:
//  m16n8k32, 16-bit types: lane 4g supplies groups 0-3 of the k-step, row g in
//    its low 16 bits and row g+8 in its high 16 bits; lane 4g+1 the same for
//    groups 4-7.  (Lanes 4g+2, 4g+3 are not read.)
//  m16n8k64, 8-bit types: lane 4g+t supplies 8 groups of row g + 8*(t&1),
//    groups 0-7 of the k-step for t < 2 and groups 8-15 for t >= 2.
// Rows past M were zero-filled by the TMA; they get a valid index pair (0, 1).
template <int DT>
__device__ __forceinline__ void meta_words(const uint8_t* sE, int row0, int lane, int64_t rows_left,
                                           uint32_t (&w)[4]) {
  using T = Traits<DT>;
  const int g = lane >> 2, t = lane & 3;
  if constexpr (T::ES == 2) {
    uint4 lo = *reinterpret_cast<const uint4*>(sE + (row0 + g) * T::EB);
    uint4 hi = *reinterpret_cast<const uint4*>(sE + (row0 + g + 8) * T::EB);
    if (g >= rows_left) lo = make_uint4(0x44444444u, 0x44444444u, 0x44444444u, 0x44444444u);
    if (g + 8 >= rows_left) hi = make_uint4(0x44444444u, 0x44444444u, 0x44444444u, 0x44444444u);
    const uint32_t sel = (t & 1) ? 0x7632u : 0x5410u;
    w[0] = __byte_perm(lo.x, hi.x, sel);
    w[1] = __byte_perm(lo.y, hi.y, sel);
    w[2] = __byte_perm(lo.z, hi.z, sel);
    w[3] = __byte_perm(lo.w, hi.w, sel);
  } else {
    const int r = g + 8 * (t & 1);
    const int half = t >> 1;
    const uint8_t* rowp = sE + (row0 + r) * T::EB;
    const uint4 lo = *reinterpret_cast<const uint4*>(rowp);
    const uint4 hi = *reinterpret_cast<const uint4*>(rowp + 16);
    w[0] = half ? lo.y : lo.x;
    w[1] = half ? lo.w : lo.z;
    w[2] = half ? hi.y : hi.x;
    w[3] = half ? hi.w : hi.z;
    if (r >= rows_left) w[0] = w[1] = w[2] = w[3] = 0x44444444u;
  }
}

template <int DT, int BN, int WARPS_N, int STAGES, int WMT>
__global__ void __launch_bounds__((Config<DT, BN, WARPS_N, STAGES, WMT>::THREADS))
    __maxnreg__((Config<DT, BN, WARPS_N, STAGES, WMT>::MAX_REGS))
    spmm_mmasp_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmE,
                      const __grid_constant__ CUtensorMap tmB, const Params p) {
  using Cfg = Config<DT, BN, WARPS_N, STAGES, WMT>;
  using T = Traits<DT>;
  using Acc = typename std::conditional<T::kInt, int, float>::type;
  constexpr int WROWS = WMT * 16;   // rows of a warp tile
  constexpr int WN = Cfg::WN;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float4* push_slots = reinterpret_cast<float4*>(smem + STAGES * Cfg::STAGE_BYTES);
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + STAGES * Cfg::STAGE_BYTES + Cfg::PUSH_BYTES);
  uint64_t* empty_bar = full_bar + STAGES;
  int* s_last = reinterpret_cast<int*>(empty_bar + STAGES);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t G = gridDim.x, cta = blockIdx.x;
  const int64_t KI = p.k_iters;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), Cfg::CONSUMERS);
    }
    fence_barrier_init();
  }
  __syncthreads();
  // Everything up to grid_dependency_wait overlaps the previous kernel in the
  // stream.  Inputs are read only after it has completed -- except, when the
  // caller declares A fixed (weights no earlier work on the stream writes),
  // the A and metadata tiles of the first STAGES k-blocks, which the producer
  // loads into the ring straight away.  Before waiting it also warms L2 with
  // the weight tiles of the k-blocks after those (an L2 prefetch cannot
  // observe stale data), so they stream from HBM meanwhile.
  // The consumers read only shared memory until their epilogue, where they
  // wait for the previous kernel; their schedule math runs before.
  if (threadIdx.x == 0) grid_launch_dependents();
  // Cluster mode: every thread arrives once here and waits once before its
  // part in the in-cluster reduction, so no CTA stores into another's shared
  // memory before that CTA has started.
  if (p.cluster > 1) cluster_arrive_relaxed();

  if (warp == Cfg::CONSUMERS) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmE);
      tma_prefetch_desc(&tmB);
      const uint64_t stream_once = p.a_evict_first ? policy_evict_first() : policy_evict_last();
      const uint64_t reuse = p.b_evict_first ? policy_evict_first() : policy_evict_last();
      uint32_t issued = 0, issued_parity = 0;   // per stage (bit s): a copy was issued, and its phase
      // This CTA's first piece of work, computed before the wait (the
      // schedule math is off the critical path that starts at the wait).
      Schedule sch(KI, p.dp_tiles, p.sk_tiles, G, cta);
      Segment sg;
      bool have = sch.next(sg);
      int64_t mt64 = 0, nt64 = 0;
      if (have) tile_coords(sg.tile, p.tiles_m, p.tiles_n, p.group_m, mt64, nt64);
      int preloaded = 0;   // leading k-blocks whose A and metadata were loaded before the wait
      {
        Schedule pre(KI, p.dp_tiles, p.sk_tiles, G, cta);
        Segment sg;
        int warm = 2 * STAGES;   // k-blocks to warm in L2
        while (warm > 0 && pre.next(sg)) {
          int64_t mt, nt;
          tile_coords(sg.tile, p.tiles_m, p.tiles_n, p.group_m, mt, nt);
          for (int64_t kb = sg.kb0; kb < sg.kb1 && warm > 0; ++kb) {
            const int32_t ka = static_cast<int32_t>(kb * (128 / T::ES));
            const int32_t ke = static_cast<int32_t>(kb * T::EB);
            const int32_t m0 = static_cast<int32_t>(mt * Cfg::BM);
            if (p.a_fixed && preloaded < STAGES) {
              // The ring starts empty: stage `preloaded` is free.  Its full
              // barrier expects the whole stage; B follows after the wait.
              const uint32_t fb = smem_u32(&full_bar[preloaded]);
              uint8_t* st = smem + preloaded * Cfg::STAGE_BYTES;
              mbar_arrive_expect_tx(fb, Cfg::STAGE_TX);
              tma_load_2d(smem_u32(st), &tmA, ka, m0, fb, stream_once);
              tma_load_2d(smem_u32(st + Cfg::A_BYTES + Cfg::B_BYTES), &tmE, ke, m0, fb, stream_once);
              issued |= 1u << preloaded;
              ++preloaded;
            } else {
              tma_prefetch_l2_2d(&tmA, ka, m0);
              tma_prefetch_l2_2d(&tmE, ke, m0);
              --warm;
            }
          }
        }
      }
      grid_dependency_wait();
      int stage = 0;
      uint32_t phase = 0;
      int done = 0;   // k-blocks issued so far
      bool ok = true;
      while (ok && have) {
        const int64_t kb0 = sg.kb0, kb1 = sg.kb1;
        const int32_t mt = static_cast<int32_t>(mt64), nt = static_cast<int32_t>(nt64);
        for (int64_t kb = kb0; kb < kb1; ++kb, ++done) {
          const uint32_t fb = smem_u32(&full_bar[stage]);
          uint8_t* st = smem + stage * Cfg::STAGE_BYTES;
          if (done >= preloaded) {
            if (!mbar_wait(smem_u32(&empty_bar[stage]), phase ^ 1u, p.status)) { ok = false; break; }
            mbar_arrive_expect_tx(fb, Cfg::STAGE_TX);
            const int32_t ka = static_cast<int32_t>(kb * (128 / T::ES));   // compressed A column
            tma_load_2d(smem_u32(st), &tmA, ka, mt * Cfg::BM, fb, stream_once);
            tma_load_2d(smem_u32(st + Cfg::A_BYTES + Cfg::B_BYTES), &tmE,
                        static_cast<int32_t>(kb * T::EB), mt * Cfg::BM, fb, stream_once);
            issued |= 1u << stage;
            issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          }
          const int64_t kbb = (p.kb_wrap && kb >= p.kb_wrap) ? kb - p.kb_wrap : kb;
          if (p.b3d) {
            // Both 128-byte-wide K chunks of the stage in one copy (3-D map).
            tma_load_3d(smem_u32(st + Cfg::A_BYTES), &tmB, 0, nt * BN, static_cast<int32_t>(2 * kbb), fb, reuse);
          } else {
            const int32_t kB = static_cast<int32_t>(kbb * T::BK);
            tma_load_2d(smem_u32(st + Cfg::A_BYTES), &tmB, kB, nt * BN, fb, reuse);
            tma_load_2d(smem_u32(st + Cfg::A_BYTES + BN * 128), &tmB, kB + 128 / T::ES, nt * BN, fb, reuse);
          }
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        have = sch.next(sg);
        if (have) tile_coords(sg.tile, p.tiles_m, p.tiles_n, p.group_m, mt64, nt64);
      }
      // Never leave with copies in flight into this CTA's shared memory.
      for (int s = 0; s < STAGES; ++s)
        if ((issued >> s) & 1u) mbar_wait(smem_u32(&full_bar[s]), (issued_parity >> s) & 1u, p.status);
    }
    __syncwarp();
    if (p.cluster > 1) {   // the producer warp's part in the in-cluster reduction
      cluster_wait();
      cluster_sync();
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int wm = warp % Cfg::WARPS_M, wn = warp / Cfg::WARPS_M;
  int cluster_done = 0;   // cluster barrier phases passed (cluster mode: exactly one per CTA)
  const int gid = lane >> 2, tig = lane & 3;
  int stage = 0;
  uint32_t phase = 0;
  Schedule sch(KI, p.dp_tiles, p.sk_tiles, G, cta);
  Segment sg;
  while (sch.next(sg)) {
    const int64_t tile = sg.tile, kb0 = sg.kb0, kb1 = sg.kb1;
    int64_t mt, nt;
    tile_coords(tile, p.tiles_m, p.tiles_n, p.group_m, mt, nt);
    const int64_t m_base = mt * Cfg::BM, n_base = nt * BN;
    constexpr int KACC = Cfg::KACC;
    Acc accs[KACC][WMT][WN][4];
#pragma unroll
    for (int u = 0; u < KACC; ++u)
#pragma unroll
      for (int i = 0; i < WMT; ++i)
#pragma unroll
        for (int j = 0; j < WN; ++j)
#pragma unroll
          for (int r = 0; r < 4; ++r) accs[u][i][j][r] = 0;

    bool ok = true;
    for (int64_t kb = kb0; kb < kb1; ++kb) {
      if (!mbar_wait(smem_u32(&full_bar[stage]), phase, p.status)) { ok = false; break; }
      const uint8_t* st = smem + stage * Cfg::STAGE_BYTES;
      const uint32_t sA = smem_u32(st);
      const uint32_t sB = smem_u32(st + Cfg::A_BYTES);
      const uint8_t* sE = st + Cfg::A_BYTES + Cfg::B_BYTES;
      uint32_t e[WMT][4];
#pragma unroll
      for (int i = 0; i < WMT; ++i)
        meta_words<DT>(sE, wm * WROWS + i * 16, lane, p.M - m_base - wm * WROWS - i * 16, e[i]);
      const int64_t ks_left = (p.K - kb * T::BK) / T::KSTEP;
      const int ksteps = ks_left < 4 ? static_cast<int>(ks_left) : 4;
      if constexpr (Cfg::FRAGS_FIRST) {
        // Narrow tiles: every fragment of the stage is loaded before the
        // first MMA, so the loads' latencies overlap instead of adding up
        // k-step by k-step (the inline-asm loads and MMAs keep program order).
        uint32_t a[4][WMT][4], b[4][WN][4];
        const int q = lane >> 3, r8 = lane & 7;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          if (ks < ksteps) {
#pragma unroll
            for (int i = 0; i < WMT; ++i) {
              const int row = wm * WROWS + i * 16 + (q & 1) * 8 + r8;
              const int chunk = ks * 2 + (q >> 1);
              ldmatrix_x4(sA + row * 128 + ((chunk ^ (row & 7)) << 4), a[ks][i][0], a[ks][i][1], a[ks][i][2],
                          a[ks][i][3]);
            }
#pragma unroll
            for (int j = 0; j < WN; ++j) {
              const int n = wn * WN * 8 + j * 8 + r8;
              const int box = ks >> 1, cb = (ks & 1) * 4 + q;
              ldmatrix_x4(sB + box * (BN * 128) + n * 128 + ((cb ^ (n & 7)) << 4), b[ks][j][0], b[ks][j][1],
                          b[ks][j][2], b[ks][j][3]);
            }
          }
        }
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          if (ks < ksteps) {
#pragma unroll
            for (int j = 0; j < WN; ++j)
#pragma unroll
              for (int i = 0; i < WMT; ++i) {
                if constexpr (DT == kS8)
                  mma_sp_16864_s8(accs[ks % KACC][i][j], a[ks][i], b[ks][j], e[i][ks]);
                else if constexpr (DT == kE4M3)
                  mma_sp_16864_e4m3(accs[ks % KACC][i][j], a[ks][i], b[ks][j], e[i][ks]);
                else
                  mma_sp_16832<DT>(accs[ks % KACC][i][j], a[ks][i], b[ks][j], e[i][ks]);
              }
          }
        }
      } else {
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        if (ks >= ksteps) break;
        uint32_t a[WMT][4];
#pragma unroll
        for (int i = 0; i < WMT; ++i) {
          const int q = lane >> 3, r8 = lane & 7;
          const int row = wm * WROWS + i * 16 + (q & 1) * 8 + r8;
          const int chunk = ks * 2 + (q >> 1);
          ldmatrix_x4(sA + row * 128 + ((chunk ^ (row & 7)) << 4), a[i][0], a[i][1], a[i][2], a[i][3]);
        }
#pragma unroll
        for (int j = 0; j < WN; ++j) {
          const int q = lane >> 3, r8 = lane & 7;
          const int n = wn * WN * 8 + j * 8 + r8;
          const int box = ks >> 1, cb = (ks & 1) * 4 + q;
          uint32_t b[4];
          ldmatrix_x4(sB + box * (BN * 128) + n * 128 + ((cb ^ (n & 7)) << 4), b[0], b[1], b[2], b[3]);
#pragma unroll
          for (int i = 0; i < WMT; ++i) {
            if constexpr (DT == kS8)
              mma_sp_16864_s8(accs[ks % KACC][i][j], a[i], b, e[i][ks]);
            else if constexpr (DT == kE4M3)
              mma_sp_16864_e4m3(accs[ks % KACC][i][j], a[i], b, e[i][ks]);
            else
              mma_sp_16832<DT>(accs[ks % KACC][i][j], a[i], b, e[i][ks]);
          }
        }
      }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&empty_bar[stage]));
      if (++stage == STAGES) { stage = 0; phase ^= 1u; }
    }
    if (!ok) break;
    // Sum the accumulator sets in set order (a fixed order: deterministic).
    Acc (&acc)[WMT][WN][4] = accs[0];
#pragma unroll
    for (int u = 1; u < KACC; ++u)
#pragma unroll
      for (int i = 0; i < WMT; ++i)
#pragma unroll
        for (int j = 0; j < WN; ++j)
#pragma unroll
          for (int r = 0; r < 4; ++r) acc[i][j][r] += accs[u][i][j][r];

    // ---- epilogue ----
    grid_dependency_wait();   // C, the workspace and the row scales are read or written from here on
    const bool whole = (kb0 == 0 && kb1 == KI);
    bool write_out = whole;
    bool mine[WMT][WN];        // fragments this CTA writes out
#pragma unroll
    for (int i = 0; i < WMT; ++i)
#pragma unroll
      for (int j = 0; j < WN; ++j) mine[i][j] = true;
    if (!whole && p.cluster > 1) {
      // Split-K inside the cluster: CTA rank r of the cluster holds the r-th
      // k-range of this tile.  Fragment f of the tile is finished by CTA
      // f % cluster; every CTA pushes its partial of f straight into that
      // CTA's push region, slot [r][f / cluster].  One cluster barrier makes
      // the pushes visible; each CTA then sums its own fragments over the
      // ranks in order (k order) from local memory and writes them out.  No
      // CTA touches another's memory after the barrier, so none waits for the
      // others before exiting.
      constexpr int F = Cfg::CONSUMERS * WMT * WN;            // fragments of the tile
      const int cs = p.cluster;
      const int owned_max = (F + cs - 1) / cs;
      const int rank = static_cast<int>(cluster_ctarank());
      float4* slots = push_slots;                            // [cluster][owned_max][32 lanes]
      cluster_wait();                                        // every CTA of the cluster has started
#pragma unroll
      for (int i = 0; i < WMT; ++i)
#pragma unroll
        for (int j = 0; j < WN; ++j) {
          const int f = (warp * WMT + i) * WN + j;
          float4 v;
          if constexpr (T::kInt)
            v = make_float4(__int_as_float(acc[i][j][0]), __int_as_float(acc[i][j][1]),
                            __int_as_float(acc[i][j][2]), __int_as_float(acc[i][j][3]));
          else
            v = make_float4(acc[i][j][0], acc[i][j][1], acc[i][j][2], acc[i][j][3]);
          st_shared_cluster_f4(slots + (rank * owned_max + f / cs) * 32 + lane, static_cast<uint32_t>(f % cs), v);
        }
      cluster_sync();
      cluster_done = 1;
#pragma unroll
      for (int i = 0; i < WMT; ++i)
#pragma unroll
        for (int j = 0; j < WN; ++j) {
          const int f = (warp * WMT + i) * WN + j;
          mine[i][j] = (f % cs) == rank;
          if (!mine[i][j]) continue;
          Acc t[4];
          for (int q = 0; q < cs; ++q) {
            const float4 v = slots[(q * owned_max + f / cs) * 32 + lane];
            Acc w[4];
            if constexpr (T::kInt) {
              w[0] = __float_as_int(v.x); w[1] = __float_as_int(v.y);
              w[2] = __float_as_int(v.z); w[3] = __float_as_int(v.w);
            } else {
              w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
            }
#pragma unroll
            for (int r = 0; r < 4; ++r) t[r] = (q == 0) ? w[r] : t[r] + w[r];
          }
#pragma unroll
          for (int r = 0; r < 4; ++r) acc[i][j][r] = t[r];
        }
      write_out = true;
    } else if (!whole) {
      // Partial tile: publish it, and let the last contributor finish the tile.
      const int64_t c_lo = sch.first_cta(tile);
      const int64_t c_hi = sch.last_cta(tile);
      auto slot_of = [&](int64_t c) -> int64_t { return sch.slot(c, tile); };
      float4* mine = reinterpret_cast<float4*>(p.partials + slot_of(cta) * Cfg::PARTIAL_ELEMS);
#pragma unroll
      for (int i = 0; i < WMT; ++i)
#pragma unroll
        for (int j = 0; j < WN; ++j) {
          const int idx = ((warp * WMT + i) * WN + j) * 32 + lane;
          float4 v;
          if constexpr (T::kInt) {
            v = make_float4(__int_as_float(acc[i][j][0]), __int_as_float(acc[i][j][1]),
                            __int_as_float(acc[i][j][2]), __int_as_float(acc[i][j][3]));
          } else {
            v = make_float4(acc[i][j][0], acc[i][j][1], acc[i][j][2], acc[i][j][3]);
          }
          __stcg(mine + idx, v);
        }
      __threadfence();
      consumer_sync(Cfg::CONSUMERS * 32);
      if (threadIdx.x == 0) {
        const unsigned nseg = static_cast<unsigned>(c_hi - c_lo + 1);
        const unsigned old = atomicAdd(p.counters + tile, 1u);
        const int last = (old == nseg - 1) ? 1 : 0;
        if (last) p.counters[tile] = 0;   // every contributor has arrived: reset for the next call
        __threadfence();
        *s_last = last;
      }
      consumer_sync(Cfg::CONSUMERS * 32);
      write_out = *s_last != 0;
      if (write_out) {
        // Sum the partials in k order (segment c_lo first).  Each segment's
        // fragments are loaded as one batch of independent loads, so a segment
        // costs one memory latency; this CTA's own partial comes from registers.
#pragma unroll
        for (int i = 0; i < WMT; ++i) {
          Acc t[WN][4];
          constexpr int U = WN >= 4 ? 1 : 4 / WN;   // segments whose loads are issued together
          for (int64_t cb = c_lo; cb <= c_hi; cb += U) {
            float4 f[U][WN];
#pragma unroll
            for (int u = 0; u < U; ++u) {
              if (cb + u <= c_hi && cb + u != cta) {
                const float4* src = reinterpret_cast<const float4*>(p.partials + slot_of(cb + u) * Cfg::PARTIAL_ELEMS);
#pragma unroll
                for (int j = 0; j < WN; ++j) f[u][j] = __ldcg(src + ((warp * WMT + i) * WN + j) * 32 + lane);
              }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
              const int64_t c = cb + u;
              if (c > c_hi) break;
#pragma unroll
              for (int j = 0; j < WN; ++j) {
                Acc v[4];
                if (c == cta) {
#pragma unroll
                  for (int r = 0; r < 4; ++r) v[r] = acc[i][j][r];
                } else if constexpr (T::kInt) {
                  v[0] = __float_as_int(f[u][j].x); v[1] = __float_as_int(f[u][j].y);
                  v[2] = __float_as_int(f[u][j].z); v[3] = __float_as_int(f[u][j].w);
                } else {
                  v[0] = f[u][j].x; v[1] = f[u][j].y; v[2] = f[u][j].z; v[3] = f[u][j].w;
                }
#pragma unroll
                for (int r = 0; r < 4; ++r) t[j][r] = (c == c_lo) ? v[r] : t[j][r] + v[r];
              }
            }
          }
#pragma unroll
          for (int j = 0; j < WN; ++j)
#pragma unroll
            for (int r = 0; r < 4; ++r) acc[i][j][r] = t[j][r];
        }
      }
    }
    if (write_out) {
      // A fragment's four C inputs are read before its four outputs are written.
#pragma unroll
      for (int i = 0; i < WMT; ++i)
#pragma unroll
        for (int j = 0; j < WN; ++j) {
          if (!mine[i][j]) continue;
          float bc[4];
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const int64_t m = m_base + wm * WROWS + i * 16 + gid + 8 * (r >> 1);
            const int64_t n = n_base + wn * WN * 8 + j * 8 + 2 * tig + (r & 1);
            bc[r] = (m < p.M && n < p.N) ? load_beta_c(p, m, n) : 0.0f;
          }
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const int64_t m = m_base + wm * WROWS + i * 16 + gid + 8 * (r >> 1);
            const int64_t n = n_base + wn * WN * 8 + j * 8 + 2 * tig + (r & 1);
            if (m < p.M && n < p.N) store_out<Acc>(p, m, n, acc[i][j][r], row_factor(p, m), bc[r]);
          }
        }
    }
  }
  // A wait that ran out of time skipped the reduction: still meet the peers
  // at the cluster barrier.
  if (p.cluster > 1 && cluster_done == 0) {
    cluster_wait();
    cluster_sync();
  }
}

template <int DT, int BN, int WARPS_N, int STAGES, int WMT = 2>
st24_status launch_cfg(const SpmmArgs& a, const StreamKPlan& plan, const DeviceInfo& dev,
                       cudaStream_t stream) {
  using Cfg = Config<DT, BN, WARPS_N, STAGES, WMT>;
  using T = Traits<DT>;
  const CUtensorMapDataType ty = T::ES == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  CUtensorMap tmA, tmE, tmB;
  const uint64_t kc = a.K / 2;  // compressed columns
  if (!encode_tensor_map_2d(&tmA, ty, a.values, kc, a.M, kc * T::ES, 128 / T::ES, Cfg::BM,
                            CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tensor_map_2d(&tmE, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.meta, a.K / 8, a.M, a.K / 8,
                            T::EB, Cfg::BM, CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !encode_tensor_map_2d(&tmB, ty, a.B, a.Kb ? a.Kb : a.K, a.N, a.ldb * T::ES, 128 / T::ES, BN,
                            CU_TENSOR_MAP_SWIZZLE_128B))
    return ST24_ERR_CUDA;
  // B as (128-byte K chunk, row, chunk index): a stage's two chunks in one
  // copy, laid out like the two 2-D boxes (chunk 0's rows, then chunk 1's).
  // Issuing copies costs the producer thread ~0.1 us each, which paced the
  // decode-shaped products.
  CUtensorMap tmB3;
  const uint64_t bdims[3] = {static_cast<uint64_t>(128 / T::ES), static_cast<uint64_t>(a.N),
                             static_cast<uint64_t>((a.Kb ? a.Kb : a.K) / (128 / T::ES))};
  const uint64_t bstrides[2] = {static_cast<uint64_t>(a.ldb * T::ES), 128};
  const uint32_t bbox[3] = {128u / T::ES, static_cast<uint32_t>(BN), 2u};
  const bool b3d = encode_tensor_map_3d(&tmB3, ty, a.B, bdims, bstrides, bbox, CU_TENSOR_MAP_SWIZZLE_128B);
  if (b3d) tmB = tmB3;
  Params p{};
  p.b3d = b3d ? 1 : 0;
  p.M = a.M; p.N = a.N; p.K = a.K;
  p.kb_wrap = (a.Kb && a.Kb != a.K) ? a.Kb / T::BK : 0;
  p.tiles_m = plan.tiles_m;
  p.tiles_n = plan.tiles_n;
  p.group_m = plan.group_m;
  p.k_iters = plan.k_iters;
  p.dp_tiles = plan.dp_tiles;
  p.sk_tiles = plan.sk_tiles;
  // A is streamed through L2 only when a single tile column reads it; B
  // stays (it is re-read by every m-tile group).  Marking the operand the
  // raster streams as evict-first was measured: it raised DRAM re-reads when
  // the output stream (C) competes for L2.
  p.a_evict_first = plan.tiles_n == 1 ? 1 : 0;
  p.b_evict_first = 0;
  p.a_fixed = (a.flags & ST24_SPMM_FIXED_A) ? 1 : 0;
  p.cluster = plan.cluster;
  p.alpha = a.alpha; p.beta = a.beta;
  p.C = a.C; p.ldc = a.ldc; p.c_type = a.c;
  p.row_scale = a.row_scale;
  p.partials = static_cast<float*>(a.workspace);
  p.counters = plan.ws_bytes
                   ? reinterpret_cast<unsigned*>(static_cast<uint8_t*>(a.workspace) +
                                                 2 * static_cast<size_t>(plan.grid) * plan.partial_bytes)
                   : nullptr;
  p.status = dev.status;
  auto kern = spmm_mmasp_kernel<DT, BN, WARPS_N, STAGES, WMT>;
  static bool attr_set[64] = {};
  if (!attr_set[dev.device % 64]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES) !=
        cudaSuccess)
      return ST24_ERR_CUDA;
    attr_set[dev.device % 64] = true;
  }
  // Launched as a programmatic dependent of the previous kernel in the stream
  // (its prologue overlaps that kernel's tail), and in clusters of
  // plan.cluster CTAs when split tiles are reduced inside the cluster.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(plan.grid));
  cfg.blockDim = dim3(Cfg::THREADS);
  cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attrs[2];
  unsigned n = 0;
  attrs[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (plan.cluster > 1) {
    attrs[n].id = cudaLaunchAttributeClusterDimension;
    attrs[n].val.clusterDim.x = static_cast<unsigned>(plan.cluster);
    attrs[n].val.clusterDim.y = 1;
    attrs[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attrs;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, tmA, tmE, tmB, p) == cudaSuccess ? ST24_OK : ST24_ERR_CUDA;
}

template <int DT>
st24_status launch_dt_impl(const SpmmArgs& a, const StreamKPlan& plan, const DeviceInfo& dev,
                      cudaStream_t s) {
  constexpr bool k16 = Traits<DT>::ES == 2;
  switch (plan.bn) {
    // Decode-shaped tiles.  From N = 9 on, 8 consumer warps of 16 rows each
    // (half the dependent MMA chain per warp) measured faster; for N <= 8,
    // 4 warps of 32 rows.
    case 8: return launch_cfg<DT, 8, 1, k16 ? 5 : 4>(a, plan, dev, s);
    case 16: return launch_cfg<DT, 16, 1, 4, 1>(a, plan, dev, s);
    case 32: return launch_cfg<DT, 32, 1, 3, 1>(a, plan, dev, s);
    case 64: return launch_cfg<DT, 64, 1, 5>(a, plan, dev, s);
    default: return launch_cfg<DT, 128, 2, 4>(a, plan, dev, s);
  }
}

// Entry per element type (defined, one per translation unit, in spmm_mmasp_<type>.cu).
template <int DT>
st24_status launch_dt(const SpmmArgs& a, const StreamKPlan& plan, const DeviceInfo& dev,
                      cudaStream_t s);

}  // namespace mmasp
}  // namespace st24
