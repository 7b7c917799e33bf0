// spmm_tc2.cuh -- the tcgen05 sparse-MMA SpMM on CTA pairs, for wide N.
//
// Same product and epilogue as spmm_tc.cuh ("Chapter 26 -- Sparsity: The
// Hardware View", section "2:4 Fine-Grained Structured Sparsity"), with the
// output tile shared by the two CTAs of a cluster: tcgen05.mma.sp with
// cta_group::2 computes M = 256 rows (128 rows of A and of the accumulator in
// each CTA) by N = BNP columns (each CTA stages BNP / 2 rows of B, the MMA
// reads both halves).  Per CTA this halves the B bytes staged per output
// element against a one-CTA tile of the same N, which is what bounds the wide
// products: the pipeline's bytes in flight per SM against L2 latency.
//
// Roles (352 threads per CTA, both CTAs):
//  * warp 0, weight producer: per stage, first its CTA's metadata (on its own
//    metadata barrier), then its 128 rows of compressed A; warp 10, B
//    producer: its BNP / 2 rows of B.  The A and B loads of both CTAs complete
//    on the leader's full barrier (the cta_group::2 form of the tensor load),
//    which the leader's weight producer arms for the bytes of both; each CTA
//    refills a stage when its own empty barrier (the MMA commit, multicast)
//    says it is free.  Two issuing threads, because one thread issues tensor
//    loads at a bounded rate (~90 cycles per box plus ~1 cycle per 117 bytes,
//    measured by a load-only probe), which put the metadata, A and the two B
//    boxes of a stage at ~800 cycles of issue against ~450 of MMA work.
//  * warps 6-9, metadata: once this CTA's metadata has landed, shared memory
//    -> this CTA's TMEM (as in the one-CTA kernel), then signal the leader
//    CTA's meta barrier: the leader's warps arrive on it (4 arrivals, each
//    expecting 4 bytes), the peer's warps complete those bytes with an
//    asynchronous 4-byte store into the leader's shared memory (st.async,
//    whose barrier signal releases at cluster scope without stalling the
//    warp).  The metadata is small and loaded first, so this path runs ahead
//    of the operand bytes instead of after them.
//  * warp 1 of the leader (cluster rank 0), MMA issuer: waits on the full
//    barrier (operands of both CTAs) and the meta barrier, issues the pair
//    MMAs and commits them to the empty barriers and accumulator barriers of
//    both CTAs (multicast).  Warp 1 of each CTA allocates and frees TMEM
//    (cta_group::2, both CTAs together).
//  * warps 2-5, epilogue: this CTA's 128 rows of the accumulator; they arrive
//    on the leader's accumulator-empty barrier (8 arrivals).  With beta != 0
//    each warp stages its 32 x 32 chunks of C in shared memory by TMA, one
//    chunk ahead (double-buffered), instead of 32 scattered loads per chunk.
// Stream-K over pair tiles: each CTA keeps its own partial tile and counter.
#pragma once

#include "spmm_tc.cuh"

namespace st24 {
namespace tc2 {

// One staged C value (output type CT) at a 32-bit shared address, as fp32.
template <int CT>
__device__ __forceinline__ float staged_c(uint32_t at) {
  if constexpr (CT == kF32) return lds_f32(at);
  else if constexpr (CT == kBF16) return __uint_as_float(lds_u16(at) << 16);
  else return __half2float(__ushort_as_half(static_cast<unsigned short>(lds_u16(at))));
}

using tc::TcParams;
using tc::TcTraits;

template <int DT, int BNP_, int STAGES_, bool CST = true>
struct PairConfig {
  using T = TcTraits<DT>;
  static constexpr int BM = 128;                     // rows of A and D per CTA (M = 256 per pair)
  static constexpr int BNP = BNP_;                   // N of the pair tile
  static constexpr int BH = BNP / 2;                 // rows of B staged per CTA
  static constexpr int STAGES = STAGES_;
  static constexpr int THREADS = 352;
  static constexpr int A_BYTES = BM * 128;
  static constexpr int B_BYTES = BH * 256;           // two 128-byte-wide boxes of BH rows
  static constexpr int E_BYTES = BM * T::EB;
  static constexpr int STAGE_TX = A_BYTES + B_BYTES + E_BYTES;
  static constexpr int PAIR_TX = 2 * (A_BYTES + B_BYTES);   // operand bytes of both CTAs per stage
  static constexpr int STAGE_BYTES = (STAGE_TX + 1023) / 1024 * 1024;
  // Two accumulators (the epilogue of one tile overlaps the next tile's
  // MMAs) where they fit beside the metadata ring, else one.
  static constexpr int ACC_BUFS = 2 * BNP + STAGES * T::META_COLS <= 512 ? 2 : 1;
  static constexpr int META_COL0 = ACC_BUFS * BNP;   // after the accumulators
  static constexpr int TMEM_COLS = 512;
  static constexpr int CBUF_BYTES = 32 * 32 * 4;                     // one warp's 32 x 32 chunk of C (fp32 at most)
  // 4 epilogue warps, double-buffered; none (CST false) when the shared
  // memory goes to one more operand stage and the outputs leave by direct
  // coalesced stores (beta = 0: no C to stage).
  static constexpr int C_BYTES = CST ? 4 * 2 * CBUF_BYTES : 0;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + C_BYTES + 1024 + 512;   // + alignment, barriers, signal words
  static constexpr int CH = 32;                      // columns per tcgen05.ld
  // Instruction descriptor: sparse, fp32 accumulator, K-major A and B, N = BNP, M = 256.
  static constexpr uint32_t IDESC = (1u << 2) | (1u << 4) | (T::FMT << 7) | (T::FMT << 10) |
                                    (static_cast<uint32_t>(BNP >> 3) << 17) | (static_cast<uint32_t>(256 >> 4) << 24);
  static_assert(BNP % 32 == 0 && BNP >= 64 && BNP <= 256, "N of the pair MMA; B halves of whole swizzle atoms");
  static_assert(ACC_BUFS * BNP + STAGES * T::META_COLS <= TMEM_COLS, "tensor memory");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
  static_assert((4 * STAGES + 5 + 8) * 8 + 8 + STAGES * 16 <= 512, "barrier region");
};

template <int DT, int BNP, int STAGES, bool CST>
__global__ void __launch_bounds__(352, 1)
    spmm_tc2_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmE,
                    const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmC,
                    const __grid_constant__ CUtensorMap tmCc, const TcParams p) {
  using Cfg = PairConfig<DT, BNP, STAGES, CST>;
  using T = TcTraits<DT>;
  constexpr uint16_t kBoth = 0x3;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* cbuf = smem + STAGES * Cfg::STAGE_BYTES;   // [4 warps][2][CBUF_BYTES] staged chunks of C
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(cbuf + Cfg::C_BYTES);   // [STAGES] leader: A and B of both CTAs
  uint64_t* empty_bar = full_bar + STAGES;
  uint64_t* efull_bar = empty_bar + STAGES;     // [STAGES] this CTA's metadata landed
  uint64_t* meta_bar = efull_bar + STAGES;      // [STAGES] leader: metadata of both CTAs in TMEM
  uint64_t* tfull_bar = meta_bar + STAGES;      // [2] accumulator ready
  uint64_t* tempty_bar = tfull_bar + 2;         // [2] leader: accumulator drained in both CTAs
  uint64_t* drain_bar = tempty_bar + 2;
  uint64_t* cbar = drain_bar + 1;               // [4 warps][2] staged C chunk landed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(cbar + 8);
  int* s_last = reinterpret_cast<int*>(tmem_slot + 1);
  uint32_t* meta_sink = reinterpret_cast<uint32_t*>(s_last + 1);   // [STAGES][4] targets of the peer's signals

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();      // 0: the leader, which issues the pair MMAs
  const int64_t G = gridDim.x / 2, pair = blockIdx.x / 2;
  const int64_t KI = p.k_iters;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), 1);
      mbar_init(smem_u32(&efull_bar[s]), 1);
      mbar_init(smem_u32(&meta_bar[s]), 4);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&tfull_bar[b]), 1);
      mbar_init(smem_u32(&tempty_bar[b]), 8);
    }
    mbar_init(smem_u32(drain_bar), 1);
    for (int i = 0; i < 8; ++i) mbar_init(smem_u32(&cbar[i]), 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), Cfg::TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();   // both CTAs' barriers initialised and TMEM allocated before any cross-CTA use
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // As in the one-CTA kernel: inputs are read after the dependency wait,
  // except fixed weights (ST24_SPMM_FIXED_A), whose first stages are loaded
  // before it; L2 is warmed with the weight tiles after those.
  // Only the producers (after the weight preloads) and the epilogue warps (C,
  // the workspace, the row scales) touch global memory; they wait for the
  // previous kernel, the MMA and metadata warps never need to.
  if (threadIdx.x == 0) grid_launch_dependents();
  if (warp >= 2 && warp <= 5) grid_dependency_wait();

  if (warp == 0) {
    // ------------------------------------------------------------ weight producer
    if (lane == 0) {
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmE);
      const uint64_t stream_once = p.a_evict_first ? policy_evict_first() : policy_evict_last();
      uint32_t issued = 0, issued_parity = 0;   // per stage (bit s): a copy was issued, and its phase
      // Arm stage s (the leader: for both CTAs' operand bytes, B included)
      // and load its metadata, then its A rows.
      auto load_weights = [&](int s, int64_t kb, int32_t m0) {
        uint8_t* st = smem + s * Cfg::STAGE_BYTES;
        const uint32_t fb = smem_u32(&full_bar[s]), eb = smem_u32(&efull_bar[s]);
        if (rank == 0) mbar_arrive_expect_tx(fb, Cfg::PAIR_TX);
        mbar_arrive_expect_tx(eb, Cfg::E_BYTES);
        uint8_t* se = st + Cfg::A_BYTES + Cfg::B_BYTES;
        const int32_t ke = static_cast<int32_t>(kb * T::EB);
        tma_load_2d(smem_u32(se), &tmE, ke, m0, eb, stream_once);
        if constexpr (T::EB == 32) tma_load_2d(smem_u32(se + 2048), &tmE, ke + 16, m0, eb, stream_once);
        tma_load_2d_pair(smem_u32(st), &tmA, static_cast<int32_t>(kb * (128 / T::ES)), m0, fb, 0, stream_once);
      };
      int preloaded = 0;
      {
        Schedule pre(KI, p.dp_tiles, p.sk_tiles, G, pair);
        Segment sg;
        int warm = 2 * STAGES;
        while (warm > 0 && pre.next(sg)) {
          int64_t mt, nt;
          tile_coords(sg.tile, p.tiles_m, p.tiles_n, p.group_m, mt, nt);
          const int32_t m0 = static_cast<int32_t>((2 * mt + rank) * Cfg::BM);
          for (int64_t kb = sg.kb0; kb < sg.kb1 && warm > 0; ++kb) {
            if (p.a_fixed && preloaded < STAGES) {
              load_weights(preloaded, kb, m0);
              issued |= 1u << preloaded;
              ++preloaded;
            } else {
              tma_prefetch_l2_2d(&tmA, static_cast<int32_t>(kb * (128 / T::ES)), m0);
              tma_prefetch_l2_2d(&tmE, static_cast<int32_t>(kb * T::EB), m0);
              --warm;
            }
          }
        }
      }
      // The first piece of work is computed before the wait.
      Schedule sch(KI, p.dp_tiles, p.sk_tiles, G, pair);
      Segment sg;
      bool have = sch.next(sg);
      int64_t mt64 = 0, nt64 = 0;
      if (have) tile_coords(sg.tile, p.tiles_m, p.tiles_n, p.group_m, mt64, nt64);
      grid_dependency_wait();
      int stage = 0;
      uint32_t phase = 0;
      int done = 0;
      bool ok = true;
      while (ok && have) {
        const int32_t m0 = static_cast<int32_t>((2 * mt64 + rank) * Cfg::BM);
        if (p.prefetch_c && sg.kb1 == KI) tma_prefetch_l2_2d(&tmC, m0, static_cast<int32_t>(nt64 * BNP));
        for (int64_t kb = sg.kb0; kb < sg.kb1; ++kb, ++done) {
          if (done >= preloaded) {
            if (!mbar_wait(smem_u32(&empty_bar[stage]), phase ^ 1u, p.status)) { ok = false; break; }
            load_weights(stage, kb, m0);
            issued |= 1u << stage;
            issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          }
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        have = sch.next(sg);
        if (have) tile_coords(sg.tile, p.tiles_m, p.tiles_n, p.group_m, mt64, nt64);
      }
      // No copy may still be landing when the CTA exits: the leader's full
      // barrier counts both CTAs' operand bytes, B included (the peer waits
      // for the leader at the final cluster barrier), each CTA's metadata
      // barrier its own.
      for (int s = 0; s < STAGES; ++s)
        if ((issued >> s) & 1u) {
          const uint32_t par = (issued_parity >> s) & 1u;
          if (rank == 0) mbar_wait_cluster(smem_u32(&full_bar[s]), par, p.status);
          mbar_wait(smem_u32(&efull_bar[s]), par, p.status);
        }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (leader)
    // The whole warp runs the loop, so the addresses and descriptors are
    // warp-uniform; one elected lane issues the MMAs and commits (issued from
    // a single-lane branch, every operand had to be moved to the uniform
    // datapath per instruction, which made the issue, not the tensor pipe,
    // the limit).
    if (rank == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int abuf = 0;
      uint32_t aphase = 0;
      bool ok = true;
      const uint32_t smem0 = smem_u32(smem);
      // whole K-steps in the last k-block (every other k-block has 4)
      const int64_t k_last = p.K - (KI - 1) * T::BK;
      const int ksteps_last = k_last / T::KSTEP < 4 ? static_cast<int>(k_last / T::KSTEP) : 4;
      Schedule sch(KI, p.dp_tiles, p.sk_tiles, G, pair);
      Segment sg;
      while (ok && sch.next(sg)) {
        ok = __all_sync(0xffffffffu, mbar_wait_cluster(smem_u32(&tempty_bar[abuf]), aphase ^ 1u, p.status));
        if (!ok) break;
        tc_fence_after();
        const uint32_t d = tmem + static_cast<uint32_t>(abuf * BNP);
        for (int64_t kb = sg.kb0; kb < sg.kb1; ++kb) {
          // The operands of both CTAs, then the metadata of both in TMEM.
          ok = __all_sync(0xffffffffu, mbar_wait_cluster(smem_u32(&full_bar[stage]), phase, p.status) &&
                                           mbar_wait_cluster(smem_u32(&meta_bar[stage]), phase, p.status));
          if (!ok) break;
          tc_fence_after();
          const uint32_t a0 = smem0 + static_cast<uint32_t>(stage * Cfg::STAGE_BYTES);
          const uint64_t da = smem_desc(a0, 16, 1024, kSwizzle128B);
          const uint64_t db = smem_desc(a0 + Cfg::A_BYTES, 16, 1024, kSwizzle128B);
          const uint32_t mcol = tmem + static_cast<uint32_t>(Cfg::META_COL0 + stage * T::META_COLS);
          const int ksteps = kb == KI - 1 ? ksteps_last : 4;
          if (elect_one_lane()) {
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
              if (ks >= ksteps) break;
              // descriptor start addresses advance in 16-byte units (no carry: shared memory < 256 KB)
              const uint64_t dak = da + static_cast<uint64_t>(ks * 2);
              const uint64_t dbk = db + static_cast<uint64_t>(((ks >> 1) * (Cfg::BH * 128) + (ks & 1) * 64) >> 4);
              const uint32_t acc = (kb > sg.kb0 || ks > 0) ? 1u : 0u;
              if constexpr (T::ES == 2)
                tc_mma_sp_f16_pair(d, dak, dbk, mcol + 4 * ks, Cfg::IDESC, acc);
              else
                tc_mma_sp_f8f6f4_pair(d, dak, dbk, mcol + 4 * ks, Cfg::IDESC, acc);
            }
            tc_commit_pair(smem_u32(&empty_bar[stage]), kBoth);
          }
          __syncwarp();
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        if (elect_one_lane()) tc_commit_pair(smem_u32(&tfull_bar[abuf]), kBoth);
        __syncwarp();
        if (++abuf == Cfg::ACC_BUFS) { abuf = 0; aphase ^= 1u; }
      }
      // Both CTAs learn when every pair MMA has completed (before TMEM is freed).
      if (elect_one_lane()) tc_commit_pair(smem_u32(drain_bar), kBoth);
      __syncwarp();
      mbar_wait(smem_u32(drain_bar), 0, p.status);
    } else if (lane == 0) {
      mbar_wait(smem_u32(drain_bar), 0, p.status);
    }
  } else if (warp == 10) {
    // ------------------------------------------------------------ B producer
    if (lane == 0) {
      tma_prefetch_desc(&tmB);
      const uint64_t reuse = p.b_evict_first ? policy_evict_first() : policy_evict_last();
      Schedule sch(KI, p.dp_tiles, p.sk_tiles, G, pair);
      Segment sg;
      grid_dependency_wait();
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      while (ok && sch.next(sg)) {
        int64_t mt, nt;
        tile_coords(sg.tile, p.tiles_m, p.tiles_n, p.group_m, mt, nt);
        const int32_t n0 = static_cast<int32_t>(nt * BNP + rank * Cfg::BH);
        for (int64_t kb = sg.kb0; kb < sg.kb1; ++kb) {
          // the slot's previous operands are consumed (both producers wait on the same phase)
          if (!mbar_wait(smem_u32(&empty_bar[stage]), phase ^ 1u, p.status)) { ok = false; break; }
          const uint32_t fb = smem_u32(&full_bar[stage]);
          uint8_t* st = smem + stage * Cfg::STAGE_BYTES;
          const int64_t kbb = (p.kb_wrap && kb >= p.kb_wrap) ? kb - p.kb_wrap : kb;
          const int32_t kB = static_cast<int32_t>(kbb * T::BK);
          tma_load_2d_pair(smem_u32(st + Cfg::A_BYTES), &tmB, kB, n0, fb, 0, reuse);
          tma_load_2d_pair(smem_u32(st + Cfg::A_BYTES + Cfg::BH * 128), &tmB, kB + 128 / T::ES, n0, fb, 0, reuse);
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
    }
  } else if (warp >= 6) {
    // ------------------------------------------------------------ metadata
    const int q = warp & 3;
    const int row = 32 * q + lane;
    const uint4 fill = make_uint4(0x44444444u, 0x44444444u, 0x44444444u, 0x44444444u);  // index pair (0, 1)
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    Schedule sch(KI, p.dp_tiles, p.sk_tiles, G, pair);
    Segment sg;
    while (ok && sch.next(sg)) {
      int64_t mt, nt;
      tile_coords(sg.tile, p.tiles_m, p.tiles_n, p.group_m, mt, nt);
      const int64_t rows_valid = p.M - (2 * mt + rank) * Cfg::BM;   // rows past M hold zero-filled metadata
      for (int64_t kb = sg.kb0; kb < sg.kb1; ++kb) {
        if (!mbar_wait(smem_u32(&efull_bar[stage]), phase, p.status)) { ok = false; break; }
        const uint8_t* se = smem + stage * Cfg::STAGE_BYTES + Cfg::A_BYTES + Cfg::B_BYTES;
        const uint32_t taddr = tmem + (static_cast<uint32_t>(32 * q) << 16) +
                               static_cast<uint32_t>(Cfg::META_COL0 + stage * T::META_COLS);
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) w[i] = fill.x;
        if constexpr (T::ES == 2) {
          const int j = row & 15;
          const int partner = j < 8 ? row + 8 : row - 8;
          const uint4 own = row < rows_valid ? *reinterpret_cast<const uint4*>(se + row * 16) : fill;
          const uint4 oth = partner < rows_valid ? *reinterpret_cast<const uint4*>(se + partner * 16) : fill;
          const uint4 lo = j < 8 ? own : oth, hi = j < 8 ? oth : own;
          const uint32_t sel = j < 8 ? 0x5410u : 0x7632u;
          w[0] = __byte_perm(lo.x, hi.x, sel);
          w[4] = __byte_perm(lo.y, hi.y, sel);
          w[8] = __byte_perm(lo.z, hi.z, sel);
          w[12] = __byte_perm(lo.w, hi.w, sel);
        } else {
          const bool in = row < rows_valid;
          const uint4 a = in ? *reinterpret_cast<const uint4*>(se + row * 16) : fill;
          const uint4 b = in ? *reinterpret_cast<const uint4*>(se + 2048 + row * 16) : fill;
          w[0] = a.x; w[1] = a.y; w[4] = a.z; w[5] = a.w;
          w[8] = b.x; w[9] = b.y; w[12] = b.z; w[13] = b.w;
        }
        tmem_st_x16(taddr, w);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (rank == 0)
            mbar_arrive_expect_tx(smem_u32(&meta_bar[stage]), 4);
          else
            signal_tx_cluster(smem_u32(&meta_sink[stage * 4 + q]), smem_u32(&meta_bar[stage]), 0);
        }
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    int abuf = 0;
    uint32_t aphase = 0;
    constexpr int CH = Cfg::CH;
    // beta * C from staged chunks when C has a tensor map (else scattered loads).
    const bool stage_c = p.beta != 0.0f && p.c_tma;
    uint8_t* my_cbuf = cbuf + q * 2 * Cfg::CBUF_BYTES;
    uint64_t* my_cbar = cbar + 2 * q;
    uint32_t cpar[2] = {0u, 0u};
    const uint64_t c_once = policy_evict_first();
    Schedule sch(KI, p.dp_tiles, p.sk_tiles, G, pair);
    Segment sg;
    while (sch.next(sg)) {
      const int64_t tile = sg.tile, kb0 = sg.kb0, kb1 = sg.kb1;
      int64_t mt, nt;
      tile_coords(tile, p.tiles_m, p.tiles_n, p.group_m, mt, nt);
      const int64_t m = (2 * mt + rank) * Cfg::BM + 32 * q + lane;
      const int64_t n_base = nt * BNP;
      if (!mbar_wait(smem_u32(&tfull_bar[abuf]), aphase, p.status)) break;
      tc_fence_after();
      const uint32_t tacc = tmem + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(abuf * BNP);
      const bool whole = (kb0 == 0 && kb1 == KI);
      const bool row_ok = m < p.M;
      const float f = row_ok ? row_factor(p, m) : 0.0f;
      if (whole && p.c_tma) {
        // Through shared memory both ways: chunk c of C (32 rows x 32
        // columns, [column][row]) is staged by TMA one chunk ahead when
        // beta != 0; the chunk's outputs overwrite it in place and leave by a
        // TMA store, which clips rows and columns past the output.
        with_float_c_type(p.c_type, [&](auto ct) {
          constexpr int CT = decltype(ct)::value;
          constexpr uint32_t CS = CT == kF32 ? 4u : 2u;
          const int32_t cm = static_cast<int32_t>((2 * mt + rank) * Cfg::BM + 32 * q);   // this warp's 32 rows
          auto stage_chunk = [&](int c) {   // lane 0
            const int b = (c / CH) & 1;
            bulk_wait_read<0>();            // the store that last used this buffer has read it
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(smem_u32(&my_cbar[b]), 32u * 32u * CS);
            tma_load_2d(smem_u32(my_cbuf + b * Cfg::CBUF_BYTES), &tmCc, cm, static_cast<int32_t>(n_base + c),
                        smem_u32(&my_cbar[b]), c_once);
          };
          // Buffer b holds chunks c with (c / CH) & 1 == b of every tile; the
          // previous tile's last stores may still be reading either buffer.
          if (lane == 0) {
            if (stage_c)
              stage_chunk(0);
            else
              bulk_wait_read<0>();
          }
#pragma unroll 1
          for (int c = 0; c < BNP; c += CH) {
            if (stage_c && lane == 0 && c + CH < BNP && n_base + c + CH < p.N) stage_chunk(c + CH);
            uint32_t r[CH];
            tmem_ld_x32(tacc + c, r);
            tmem_ld_wait();
            if (n_base + c >= p.N) continue;   // warp-uniform: nothing of this chunk is in the output
            const int b = (c / CH) & 1;
            const uint32_t buf = smem_u32(my_cbuf + b * Cfg::CBUF_BYTES);
            if (stage_c) {
              mbar_wait(smem_u32(&my_cbar[b]), cpar[b], p.status);
              cpar[b] ^= 1u;
            } else {
              if (lane == 0) bulk_wait_read<1>();   // the store of two chunks ago has read this buffer
              __syncwarp();
            }
            // each lane overwrites in place only the staged values it read
#pragma unroll
            for (int j = 0; j < CH; ++j) {
              float o = __fmul_rn(__uint_as_float(r[j]), f);
              const uint32_t at = buf + (j * 32 + lane) * CS;
              if (p.beta != 0.0f) o = __fadd_rn(o, __fmul_rn(p.beta, staged_c<CT>(at)));
              if constexpr (CT == kF32) sts_f32(at, o);
              else if constexpr (CT == kBF16) sts_u16(at, __bfloat16_as_ushort(__float2bfloat16_rn(o)));
              else sts_u16(at, __half_as_ushort(__float2half_rn(o)));
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmCc, cm, static_cast<int32_t>(n_base + c), buf, c_once);   // the output streams through L2
              bulk_commit();
            }
          }
        });
      } else if (whole) {
        with_float_c_type(p.c_type, [&](auto ct) {
          constexpr int CT = decltype(ct)::value;
#pragma unroll 1
          for (int c = 0; c < BNP; c += CH) {
            const bool live = row_ok && n_base + c < p.N;
            uint32_t r[CH];
            tmem_ld_x32(tacc + c, r);
            tmem_ld_wait();
            if (live) {
#pragma unroll
              for (int g = 0; g < CH; g += 8) {   // 8 columns at a time: few registers live
                float bc[8];
                uint32_t rg[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) rg[j] = r[g + j];
                if (p.beta != 0.0f) load_row_chunk_beta_c<CT, 8>(p, m, n_base + c + g, bc);
                store_row_chunk_bits<CT, 8>(p, m, n_base + c + g, rg, bc, f);
              }
            }
          }
        });
      }
      if (whole) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(smem_u32(&tempty_bar[abuf]), 0);
      } else {
        // This CTA's half of the pair tile: slot 2 * (pair slot) + rank.
        float* mine = p.partials + (2 * sch.slot(pair, tile) + rank) * (Cfg::BM * BNP);
#pragma unroll 1
        for (int c = 0; c < BNP; c += CH) {
          uint32_t r[CH];
          tmem_ld_x32(tacc + c, r);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < CH; ++j) __stcg(mine + (c + j) * Cfg::BM + 32 * q + lane, __uint_as_float(r[j]));
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(smem_u32(&tempty_bar[abuf]), 0);
        __threadfence();
        named_barrier_sync(1, 128);
        const int64_t c_lo = sch.first_cta(tile);
        const int64_t c_hi = sch.last_cta(tile);
        if (threadIdx.x == 64) {
          unsigned* counter = p.counters + 2 * tile + rank;
          const unsigned nseg = static_cast<unsigned>(c_hi - c_lo + 1);
          const unsigned old = atomicAdd(counter, 1u);
          const int last = (old == nseg - 1) ? 1 : 0;
          if (last) *counter = 0;   // all contributors have arrived: ready for the next call
          __threadfence();
          *s_last = last;
        }
        named_barrier_sync(1, 128);
        if (*s_last && row_ok)
          reduce_split_row<Cfg::BM, BNP, 8>(p, p.partials, sch, tile, 2, static_cast<int>(rank), c_lo, c_hi,
                                             32 * q + lane, m, n_base, f);
      }
      if (++abuf == Cfg::ACC_BUFS) { abuf = 0; aphase ^= 1u; }
    }
    if (lane == 0) bulk_wait_all();   // this warp's output stores have completed
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem, Cfg::TMEM_COLS);
  // Neither CTA leaves while the other may still arrive on its barriers.
  cluster_sync();
}

// Pairs that can be resident at once for this kernel (its clusters of 2).
template <int DT, int BNP, int STAGES, bool CST>
int resident_pairs(int num_sms) {
  using Cfg = PairConfig<DT, BNP, STAGES, CST>;
  static int pairs = 0;
  if (pairs == 0) {
    auto kern = spmm_tc2_kernel<DT, BNP, STAGES, CST>;
    int n = 0;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES) == cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(static_cast<unsigned>(num_sms / 2 * 2));
      cfg.blockDim = dim3(Cfg::THREADS);
      cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
      cudaLaunchAttribute attr;
      attr.id = cudaLaunchAttributeClusterDimension;
      attr.val.clusterDim.x = 2;
      attr.val.clusterDim.y = 1;
      attr.val.clusterDim.z = 1;
      cfg.attrs = &attr;
      cfg.numAttrs = 1;
      if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) n = 0;
    }
    pairs = n > 0 ? (n < num_sms / 2 ? n : num_sms / 2) : num_sms / 2;
  }
  return pairs;
}

template <int DT, int BNP, int STAGES, bool CST = true>
st24_status launch_pair(const SpmmArgs& a, const StreamKPlan& plan, const DeviceInfo& dev, cudaStream_t stream) {
  using Cfg = PairConfig<DT, BNP, STAGES, CST>;
  using T = TcTraits<DT>;
  const CUtensorMapDataType ty = T::ES == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  CUtensorMap tmA, tmE, tmB;
  const uint64_t kc = a.K / 2;
  if (!encode_tensor_map_2d(&tmA, ty, a.values, kc, a.M, kc * T::ES, 128 / T::ES, Cfg::BM,
                            CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tensor_map_2d(&tmE, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.meta, a.K / 8, a.M, a.K / 8, 16, Cfg::BM,
                            CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !encode_tensor_map_2d(&tmB, ty, a.B, a.Kb ? a.Kb : a.K, a.N, a.ldb * T::ES, 128 / T::ES, Cfg::BH,
                            CU_TENSOR_MAP_SWIZZLE_128B))
    return ST24_ERR_CUDA;
  // C (element (m, n) at C[n*ldc + m]) as an M-inner 2-D tensor: 32 x 32
  // boxes for the epilogue's chunks, and a whole-tile box for the L2
  // prefetch of each tile's C block when beta != 0.
  CUtensorMap tmC, tmCc;
  const int cs = elem_size(a.c);
  const CUtensorMapDataType cty = cs == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_UINT16;
  const bool c_map = (reinterpret_cast<uintptr_t>(a.C) % 16 == 0) && ((a.ldc * cs) % 16 == 0) &&
                     encode_tensor_map_2d(&tmCc, cty, a.C, a.M, a.N, a.ldc * cs, 32, 32, CU_TENSOR_MAP_SWIZZLE_NONE);
  const bool c_prefetch = c_map && a.beta != 0.0f &&
                          encode_tensor_map_2d(&tmC, cty, a.C, a.M, a.N, a.ldc * cs, Cfg::BM, BNP,
                                               CU_TENSOR_MAP_SWIZZLE_NONE);
  if (!c_map) tmCc = tmA;        // unused
  if (!c_prefetch) tmC = tmA;    // unused
  TcParams p{};
  p.c_tma = (c_map && CST) ? 1 : 0;
  p.prefetch_c = c_prefetch ? 1 : 0;
  p.M = a.M; p.N = a.N; p.K = a.K;
  p.kb_wrap = (a.Kb && a.Kb != a.K) ? a.Kb / T::BK : 0;
  p.alpha = a.alpha; p.beta = a.beta;
  p.C = a.C; p.ldc = a.ldc; p.c_type = a.c;
  p.row_scale = a.row_scale;
  p.tiles_m = plan.tiles_m;
  p.tiles_n = plan.tiles_n;
  p.group_m = plan.group_m;
  p.k_iters = plan.k_iters;
  p.dp_tiles = plan.dp_tiles;
  p.sk_tiles = plan.sk_tiles;
  // L2 policy per operand.  A is streamed once when a single tile column
  // reads it.  When the raster keeps the whole A resident (one group of all
  // m-tiles, n-tiles outer), each B panel is read by the m-tiles of one wave
  // and never again: evict-first, so that the panels passing through do not
  // push A out (measured on 4096x11008, N = 4096: DRAM reads 355 -> 240 MB,
  // same time).  Otherwise B stays: it is re-read by every m-tile group.
  // (Marking A evict-first in the row-major raster was measured to raise
  // DRAM re-reads when the output stream C competes for L2.)
  p.a_evict_first = plan.tiles_n == 1 ? 1 : 0;
  p.b_evict_first = (plan.group_m >= plan.tiles_m && plan.tiles_m > 1 && plan.tiles_n > 1) ? 1 : 0;
  p.a_fixed = (a.flags & ST24_SPMM_FIXED_A) ? 1 : 0;
  p.partials = static_cast<float*>(a.workspace);
  p.counters = plan.ws_bytes ? reinterpret_cast<unsigned*>(static_cast<uint8_t*>(a.workspace) +
                                                          2 * static_cast<size_t>(plan.grid) * plan.partial_bytes)
                             : nullptr;
  p.status = dev.status;
  auto kern = spmm_tc2_kernel<DT, BNP, STAGES, CST>;
  resident_pairs<DT, BNP, STAGES, CST>(dev.num_sms);   // sets the kernel's shared-memory attribute once
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(2 * plan.grid));
  cfg.blockDim = dim3(Cfg::THREADS);
  cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attrs[2];
  attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[0].val.programmaticStreamSerializationAllowed = 1;
  attrs[1].id = cudaLaunchAttributeClusterDimension;
  attrs[1].val.clusterDim.x = 2;
  attrs[1].val.clusterDim.y = 1;
  attrs[1].val.clusterDim.z = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, tmA, tmE, tmB, tmC, tmCc, p) == cudaSuccess ? ST24_OK : ST24_ERR_CUDA;
}

}  // namespace tc2
}  // namespace st24
