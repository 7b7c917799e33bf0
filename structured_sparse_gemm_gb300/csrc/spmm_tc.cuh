// spmm_tc.cuh -- C = alpha * row_scale * (A_sparse * B) + beta * C on the
// 5th-generation tensor cores (tcgen05.mma.sp), for f16, bf16 and fp8-e4m3.
//
// Method ("Chapter 26 -- Sparsity: The Hardware View", section "2:4
// Fine-Grained Structured Sparsity"): each group's two stored weights multiply
// the two activations its metadata selects; the sparse MMA reads the
// compressed A (M x K/2) and a 4-bit-per-group metadata operand, so a 2:4 tile
// costs half the multiply work of its dense shape.
//
// One persistent CTA per SM, 6 warps:
//  * warp 0, TMA producer: per stage the compressed-A tile (128 rows x 128 B,
//    128-byte swizzle), the B tile (BN rows x 256 B as two 128-byte swizzled
//    boxes) and the metadata tile (128 rows x 16 B per box, no swizzle) into a
//    ring of stages guarded by full/empty mbarriers.
//  * warps 6-9, metadata: move the stage's metadata tile from shared memory
//    into TMEM with tcgen05.st (each warp its 32-lane quadrant), in the order
//    the sparse MMA reads it, and give rows past M a valid index pair.
//  * warp 1, MMA issuer (one thread): issues 4 sparse MMAs per stage (M=128,
//    N=BN, K=32 for 16-bit or 64 for 8-bit inputs) into a TMEM accumulator and
//    commits the stage back to the producer.  Two accumulators alternate so
//    the epilogue of a tile overlaps the next tile.  Warp 1 also owns the TMEM
//    allocation.
//  * warps 2-5, epilogue: tcgen05.ld of their 32-lane quadrant, then the fused
//    alpha / row-scale / beta / rounding store; partial tiles of the stream-K
//    schedule go through the workspace and are summed in k order by the last
//    contributor.
// Metadata order in TMEM (lane = row of the tile, one 32-bit column per 32
// logical K of an MMA, the columns of each MMA starting on a 4-column
// boundary): for 8-bit inputs each column is the row's canonical metadata word
// (8 groups, lowest K lowest).  For 16-bit inputs rows pair up
// as (r, r+8) inside each 16-row block: lane r holds groups 0-3 of row r in
// its low half and groups 0-3 of row r+8 in its high half, lane r+8 holds
// groups 4-7 of the two rows the same way.
#pragma once

#include "st24_epilogue.cuh"

namespace st24 {
namespace tc {

template <int DT>
struct TcTraits {
  static constexpr int ES = (DT == kF16 || DT == kBF16) ? 2 : 1;
  static constexpr int KSTEP = 64 / ES;              // logical K per MMA
  static constexpr int BK = 4 * KSTEP;               // logical K per stage
  static constexpr int EB = BK / 8;                  // metadata bytes per row per stage
  // Metadata of MMA ks of a stage sits at column 4*ks of the stage's 16-column
  // slot (4-column aligned, read with sparsity selector 0): one column for
  // 16-bit inputs, two for 8-bit inputs.
  static constexpr int META_COLS_PER_MMA = KSTEP / 32;
  static constexpr int META_COLS = 16;               // TMEM columns of metadata per stage
  static constexpr uint32_t FMT = (DT == kBF16) ? 1u : 0u;   // f16 0, bf16 1; e4m3 0 (kind::f8f6f4)
};

constexpr int pow2_at_least(int v) {
  int p = 32;
  while (p < v) p <<= 1;
  return p;
}

template <int DT, int BN_, int STAGES_>
struct TcConfig {
  using T = TcTraits<DT>;
  static constexpr int BM = 128;
  static constexpr int BN = BN_;
  static constexpr int STAGES = STAGES_;
  static constexpr int THREADS = 320;
  static constexpr int A_BYTES = BM * 128;
  static constexpr int B_BYTES = BN * 256;
  static constexpr int E_BYTES = BM * T::EB;
  static constexpr int STAGE_TX = A_BYTES + B_BYTES + E_BYTES;
  static constexpr int STAGE_BYTES = (STAGE_TX + 1023) / 1024 * 1024;
  static constexpr int META_COL0 = 2 * BN;           // after the two accumulators
  static constexpr int TMEM_COLS = pow2_at_least(2 * BN + STAGES * T::META_COLS);
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 256;
  static constexpr int CH = BN < 32 ? BN : 32;       // columns per tcgen05.ld
  // Instruction descriptor: sparse, fp32 accumulator, K-major A and B, N = BN, M = 128.
  static constexpr uint32_t IDESC = (1u << 2) | (1u << 4) | (T::FMT << 7) | (T::FMT << 10) |
                                    (static_cast<uint32_t>(BN >> 3) << 17) | (static_cast<uint32_t>(BM >> 4) << 24);
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 128, "N of the MMA");
  static_assert(TMEM_COLS <= 512, "tensor memory");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
};

struct TcParams : OutParams {
  int64_t K;
  int prefetch_c;          // beta != 0 and C has a tensor map: warm L2 with each tile's C early
  int c_tma;               // C has a tensor map with 32 x 32 boxes (pair kernel: TMA epilogue)
  int64_t tiles_m, tiles_n, group_m, k_iters, dp_tiles, sk_tiles;
  int a_evict_first;      // A is streamed once (by the tiles running at the same time): evict it first
  int b_evict_first;      // B likewise (the raster keeps the A panel resident instead)
  int a_fixed;            // A is not written by earlier work on the stream: load it before the dependency wait
  int64_t kb_wrap;        // two-form product: k-blocks per form (B's k-block of k-block kb is kb mod kb_wrap); 0: one form
  float* partials;
  unsigned* counters;
  unsigned* status;
};

template <int DT, int BN, int STAGES>
__global__ void __launch_bounds__(320, 1)
    spmm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmE,
                   const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmC,
                   const TcParams p) {
  using Cfg = TcConfig<DT, BN, STAGES>;
  using T = TcTraits<DT>;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + STAGES * Cfg::STAGE_BYTES);
  uint64_t* empty_bar = full_bar + STAGES;
  uint64_t* meta_bar = empty_bar + STAGES;      // [STAGES] metadata in TMEM
  uint64_t* tfull_bar = meta_bar + STAGES;      // [2] accumulator ready
  uint64_t* tempty_bar = tfull_bar + 2;         // [2] accumulator drained
  uint64_t* drain_bar = tempty_bar + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain_bar + 1);
  int* s_last = reinterpret_cast<int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t G = gridDim.x, cta = blockIdx.x;
  const int64_t KI = p.k_iters;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), 1);
      mbar_init(smem_u32(&meta_bar[s]), 4);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&tfull_bar[b]), 1);
      mbar_init(smem_u32(&tempty_bar[b]), 4);
    }
    mbar_init(smem_u32(drain_bar), 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), Cfg::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Everything up to grid_dependency_wait overlaps the previous kernel in the
  // stream.  Inputs are read only after it has completed -- except, when the
  // caller declares A fixed (weights no earlier work on the stream writes),
  // the A and metadata tiles of the first STAGES k-blocks, which the producer
  // loads into the ring straight away.  Before waiting it also warms L2 with
  // the weight tiles of the k-blocks after those (an L2 prefetch cannot
  // observe stale data), so they stream from HBM meanwhile.
  // Only the producer (B, after its preloads) and the epilogue warps (C, the
  // workspace, the row scales) touch global memory; they wait for the
  // previous kernel, the MMA and metadata warps never need to.
  if (threadIdx.x == 0) grid_launch_dependents();
  if (warp >= 2 && warp <= 5) grid_dependency_wait();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmE);
      tma_prefetch_desc(&tmB);
      const uint64_t stream_once = p.a_evict_first ? policy_evict_first() : policy_evict_last();
      const uint64_t reuse = p.b_evict_first ? policy_evict_first() : policy_evict_last();
      uint32_t issued = 0, issued_parity = 0;   // per stage (bit s): a copy was issued, and its phase
      // A and metadata of k-block kb of m-tile mt into stage st (full barrier fb).
      auto load_weights = [&](uint8_t* st, uint32_t fb, int64_t kb, int32_t m0) {
        tma_load_2d(smem_u32(st), &tmA, static_cast<int32_t>(kb * (128 / T::ES)), m0, fb, stream_once);
        uint8_t* se = st + Cfg::A_BYTES + Cfg::B_BYTES;
        const int32_t ke = static_cast<int32_t>(kb * T::EB);
        tma_load_2d(smem_u32(se), &tmE, ke, m0, fb, stream_once);
        if constexpr (T::EB == 32) tma_load_2d(smem_u32(se + 2048), &tmE, ke + 16, m0, fb, stream_once);
      };
      int preloaded = 0;   // leading k-blocks whose A and metadata were loaded before the wait
      {
        Schedule pre(KI, p.dp_tiles, p.sk_tiles, G, cta);
        Segment sg;
        int warm = 2 * STAGES;   // k-blocks to warm in L2
        while (warm > 0 && pre.next(sg)) {
          int64_t mt, nt;
          tile_coords(sg.tile, p.tiles_m, p.tiles_n, p.group_m, mt, nt);
          const int32_t m0 = static_cast<int32_t>(mt * Cfg::BM);
          for (int64_t kb = sg.kb0; kb < sg.kb1 && warm > 0; ++kb) {
            if (p.a_fixed && preloaded < STAGES) {
              // The ring starts empty: stage `preloaded` is free.  Its full
              // barrier expects the whole stage; B follows after the wait.
              const uint32_t fb = smem_u32(&full_bar[preloaded]);
              mbar_arrive_expect_tx(fb, Cfg::STAGE_TX);
              load_weights(smem + preloaded * Cfg::STAGE_BYTES, fb, kb, m0);
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
      // The first piece of work is computed before the wait (off the
      // critical path that starts there).
      Schedule sch(KI, p.dp_tiles, p.sk_tiles, G, cta);
      Segment sg;
      bool have = sch.next(sg);
      int64_t mt64 = 0, nt64 = 0;
      if (have) tile_coords(sg.tile, p.tiles_m, p.tiles_n, p.group_m, mt64, nt64);
      grid_dependency_wait();
      int stage = 0;
      uint32_t phase = 0;
      int done = 0;   // k-blocks issued so far
      bool ok = true;
      while (ok && have) {
        const int64_t kb0 = sg.kb0, kb1 = sg.kb1;
        const int32_t mt = static_cast<int32_t>(mt64), nt = static_cast<int32_t>(nt64);
        // The epilogue of this tile reads C (beta != 0): start it towards L2 now.
        if (p.prefetch_c && kb1 == KI) tma_prefetch_l2_2d(&tmC, mt * Cfg::BM, nt * BN);
        for (int64_t kb = kb0; kb < kb1; ++kb, ++done) {
          const uint32_t fb = smem_u32(&full_bar[stage]);
          uint8_t* st = smem + stage * Cfg::STAGE_BYTES;
          if (done >= preloaded) {
            if (!mbar_wait(smem_u32(&empty_bar[stage]), phase ^ 1u, p.status)) { ok = false; break; }
            mbar_arrive_expect_tx(fb, Cfg::STAGE_TX);
            load_weights(st, fb, kb, mt * Cfg::BM);
            issued |= 1u << stage;
            issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          }
          const int64_t kbb = (p.kb_wrap && kb >= p.kb_wrap) ? kb - p.kb_wrap : kb;
          const int32_t kB = static_cast<int32_t>(kbb * T::BK);
          tma_load_2d(smem_u32(st + Cfg::A_BYTES), &tmB, kB, nt * BN, fb, reuse);
          tma_load_2d(smem_u32(st + Cfg::A_BYTES + BN * 128), &tmB, kB + 128 / T::ES, nt * BN, fb, reuse);
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        have = sch.next(sg);
        if (have) tile_coords(sg.tile, p.tiles_m, p.tiles_n, p.group_m, mt64, nt64);
      }
      // Never leave with copies in flight into this CTA's shared memory.
      for (int s = 0; s < STAGES; ++s)
        if ((issued >> s) & 1u) mbar_wait(smem_u32(&full_bar[s]), (issued_parity >> s) & 1u, p.status);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the loop (its addresses and descriptors stay
    // warp-uniform); one elected lane issues the MMAs and commits.
    int stage = 0;
    uint32_t phase = 0;
    int abuf = 0;
    uint32_t aphase = 0;
    bool ok = true;
    const uint32_t smem0 = smem_u32(smem);
    const int64_t k_last = p.K - (KI - 1) * T::BK;   // whole K-steps in the last k-block (others: 4)
    const int ksteps_last = k_last / T::KSTEP < 4 ? static_cast<int>(k_last / T::KSTEP) : 4;
    Schedule sch(KI, p.dp_tiles, p.sk_tiles, G, cta);
    Segment sg;
    while (ok && sch.next(sg)) {
      const int64_t kb0 = sg.kb0, kb1 = sg.kb1;
      ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&tempty_bar[abuf]), aphase ^ 1u, p.status));
      if (!ok) break;
      tc_fence_after();
      const uint32_t d = tmem + static_cast<uint32_t>(abuf * BN);
      for (int64_t kb = kb0; kb < kb1; ++kb) {
        ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&meta_bar[stage]), phase, p.status) &&
                                         mbar_wait(smem_u32(&full_bar[stage]), phase, p.status));
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
            const uint64_t dbk = db + static_cast<uint64_t>(((ks >> 1) * (BN * 128) + (ks & 1) * 64) >> 4);
            const uint32_t acc = (kb > kb0 || ks > 0) ? 1u : 0u;
            if constexpr (T::ES == 2)
              tc_mma_sp_f16(d, dak, dbk, mcol + 4 * ks, Cfg::IDESC, acc);
            else
              tc_mma_sp_f8f6f4(d, dak, dbk, mcol + 4 * ks, Cfg::IDESC, acc);
          }
          tc_commit(smem_u32(&empty_bar[stage]));
        }
        __syncwarp();
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
      if (!ok) break;
      if (elect_one_lane()) tc_commit(smem_u32(&tfull_bar[abuf]));
      __syncwarp();
      if (++abuf == 2) { abuf = 0; aphase ^= 1u; }
    }
    // Every tcgen05 operation of this warp has completed before TMEM is freed.
    if (elect_one_lane()) tc_commit(smem_u32(drain_bar));
    __syncwarp();
    mbar_wait(smem_u32(drain_bar), 0, p.status);
  } else if (warp >= 6) {
    // ------------------------------------------------------------ metadata
    const int q = warp & 3;                 // TMEM lane quadrant of this warp
    const int row = 32 * q + lane;          // row of the tile this lane moves
    const uint4 fill = make_uint4(0x44444444u, 0x44444444u, 0x44444444u, 0x44444444u);  // index pair (0, 1)
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    Schedule sch(KI, p.dp_tiles, p.sk_tiles, G, cta);
    Segment sg;
    while (ok && sch.next(sg)) {
      const int64_t tile = sg.tile, kb0 = sg.kb0, kb1 = sg.kb1;
      int64_t mt, nt;
      tile_coords(tile, p.tiles_m, p.tiles_n, p.group_m, mt, nt);
      const int64_t rows_valid = p.M - mt * Cfg::BM;   // rows past M hold zero-filled metadata
      for (int64_t kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait(smem_u32(&full_bar[stage]), phase, p.status)) { ok = false; break; }
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
        if (lane == 0) mbar_arrive(smem_u32(&meta_bar[stage]));
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;                 // TMEM lane quadrant of this warp
    int abuf = 0;
    uint32_t aphase = 0;
    constexpr int CH = Cfg::CH;
    Schedule sch(KI, p.dp_tiles, p.sk_tiles, G, cta);
    Segment sg;
    while (sch.next(sg)) {
      const int64_t tile = sg.tile, kb0 = sg.kb0, kb1 = sg.kb1;
      int64_t mt, nt;
      tile_coords(tile, p.tiles_m, p.tiles_n, p.group_m, mt, nt);
      const int64_t m = mt * Cfg::BM + 32 * q + lane;
      const int64_t n_base = nt * BN;
      if (!mbar_wait(smem_u32(&tfull_bar[abuf]), aphase, p.status)) break;
      tc_fence_after();
      const uint32_t tacc = tmem + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(abuf * BN);
      const bool whole = (kb0 == 0 && kb1 == KI);
      const bool row_ok = m < p.M;
      const float f = row_ok ? row_factor(p, m) : 0.0f;
      if (whole) {
        with_float_c_type(p.c_type, [&](auto ct) {
          constexpr int CT = decltype(ct)::value;
#pragma unroll 1
          for (int c = 0; c < BN; c += CH) {
            uint32_t r[CH];
            if constexpr (CH == 32) tmem_ld_x32(tacc + c, r); else tmem_ld_x16(tacc + c, r);
            tmem_ld_wait();
            if (row_ok) {
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
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&tempty_bar[abuf]));
      } else {
        float* mine = p.partials + sch.slot(cta, tile) * (Cfg::BM * BN);
#pragma unroll 1
        for (int c = 0; c < BN; c += CH) {
          uint32_t r[CH];
          if constexpr (CH == 32) tmem_ld_x32(tacc + c, r); else tmem_ld_x16(tacc + c, r);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < CH; ++j) __stcg(mine + (c + j) * Cfg::BM + 32 * q + lane, __uint_as_float(r[j]));
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&tempty_bar[abuf]));
        __threadfence();
        named_barrier_sync(1, 128);
        const int64_t c_lo = sch.first_cta(tile);
        const int64_t c_hi = sch.last_cta(tile);
        if (threadIdx.x == 64) {
          const unsigned nseg = static_cast<unsigned>(c_hi - c_lo + 1);
          const unsigned old = atomicAdd(p.counters + tile, 1u);
          const int last = (old == nseg - 1) ? 1 : 0;
          if (last) p.counters[tile] = 0;   // all contributors have arrived: ready for the next call
          __threadfence();
          *s_last = last;
        }
        named_barrier_sync(1, 128);
        if (*s_last && row_ok)
          reduce_split_row<Cfg::BM, BN, (BN < 8 ? BN : 8)>(p, p.partials, sch, tile, 1, 0, c_lo, c_hi,
                                                             32 * q + lane, m, n_base, f);
      }
      if (++abuf == 2) { abuf = 0; aphase ^= 1u; }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, Cfg::TMEM_COLS);
}

template <int DT, int BN, int STAGES>
st24_status launch_cfg(const SpmmArgs& a, const StreamKPlan& plan, const DeviceInfo& dev, cudaStream_t stream) {
  using Cfg = TcConfig<DT, BN, STAGES>;
  using T = TcTraits<DT>;
  const CUtensorMapDataType ty = T::ES == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  CUtensorMap tmA, tmE, tmB;
  const uint64_t kc = a.K / 2;
  if (!encode_tensor_map_2d(&tmA, ty, a.values, kc, a.M, kc * T::ES, 128 / T::ES, Cfg::BM,
                            CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tensor_map_2d(&tmE, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.meta, a.K / 8, a.M, a.K / 8, 16, Cfg::BM,
                            CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !encode_tensor_map_2d(&tmB, ty, a.B, a.Kb ? a.Kb : a.K, a.N, a.ldb * T::ES, 128 / T::ES, BN,
                            CU_TENSOR_MAP_SWIZZLE_128B))
    return ST24_ERR_CUDA;
  // C (element (m, n) at C[n*ldc + m]) as an M-inner 2-D tensor, for the L2
  // prefetch of each tile's C block when beta != 0.
  CUtensorMap tmC;
  bool have_c = false;
  if (a.beta != 0.0f) {
    const int cs = elem_size(a.c);
    const CUtensorMapDataType cty = cs == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_UINT16;
    have_c = (reinterpret_cast<uintptr_t>(a.C) % 16 == 0) && ((a.ldc * cs) % 16 == 0) &&
             encode_tensor_map_2d(&tmC, cty, a.C, a.M, a.N, a.ldc * cs, Cfg::BM, BN,
                                  CU_TENSOR_MAP_SWIZZLE_NONE);
  }
  if (!have_c) tmC = tmA;   // unused
  TcParams p{};
  p.prefetch_c = have_c ? 1 : 0;
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
  // A is streamed through L2 only when a single tile column reads it; B
  // stays (it is re-read by every m-tile group).  Marking the operand the
  // raster streams as evict-first was measured: it raised DRAM re-reads when
  // the output stream (C) competes for L2.
  p.a_evict_first = plan.tiles_n == 1 ? 1 : 0;
  p.b_evict_first = 0;
  p.a_fixed = (a.flags & ST24_SPMM_FIXED_A) ? 1 : 0;
  p.partials = static_cast<float*>(a.workspace);
  p.counters = plan.ws_bytes ? reinterpret_cast<unsigned*>(static_cast<uint8_t*>(a.workspace) +
                                                          2 * static_cast<size_t>(plan.grid) * plan.partial_bytes)
                             : nullptr;
  p.status = dev.status;
  auto kern = spmm_tc_kernel<DT, BN, STAGES>;
  static bool attr_set[64] = {};
  if (!attr_set[dev.device % 64]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES) != cudaSuccess)
      return ST24_ERR_CUDA;
    attr_set[dev.device % 64] = true;
  }
  // Launched as a programmatic dependent of the previous kernel in the stream.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(plan.grid));
  cfg.blockDim = dim3(Cfg::THREADS);
  cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tmA, tmE, tmB, tmC, p) == cudaSuccess ? ST24_OK : ST24_ERR_CUDA;
}

}  // namespace tc
}  // namespace st24

#include "spmm_tc2.cuh"

namespace st24 {
namespace tc {

template <int DT>
st24_status launch_dt_impl(const SpmmArgs& a, const StreamKPlan& plan, const DeviceInfo& dev, cudaStream_t s) {
  constexpr bool k16 = TcTraits<DT>::ES == 2;
  if (plan.pair) {
    if (plan.bn == 128) return tc2::launch_pair<DT, 128, 5>(a, plan, dev, s);
    // 256-column tiles: 4 stages when beta = 0 (no C staging buffers;
    // e4m3 28672x8192 at N = 512: 71.9 -> 66.8 us against 3 stages)
    if (plan.bn == 256)
      return a.beta == 0.0f ? tc2::launch_pair<DT, 256, 4, false>(a, plan, dev, s)
                            : tc2::launch_pair<DT, 256, 3>(a, plan, dev, s);
    return tc2::launch_pair<DT, 224, 4>(a, plan, dev, s);
  }
  switch (plan.bn) {
    case 16: return launch_cfg<DT, 16, 8>(a, plan, dev, s);
    case 32: return launch_cfg<DT, 32, 7>(a, plan, dev, s);
    case 64: return launch_cfg<DT, 64, k16 ? 6 : 6>(a, plan, dev, s);
    default: return launch_cfg<DT, 128, 4>(a, plan, dev, s);
  }
}

// Entry per element type (one translation unit each: spmm_tc_<type>.cu).
template <int DT>
st24_status launch_dt(const SpmmArgs& a, const StreamKPlan& plan, const DeviceInfo& dev, cudaStream_t s);

}  // namespace tc
}  // namespace st24
