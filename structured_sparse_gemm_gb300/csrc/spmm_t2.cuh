// spmm_t2.cuh -- the transposed use of a compressed weight on CTA pairs:
// dX = alpha * dY * A + beta * dX, the same product and expansion as
// spmm_t.cuh ("Chapter 26 -- Sparsity: The Hardware View", section "2:4: ~2x
// on the Matmul, Less End-to-End"), with each output tile of 256 k x BN n
// shared by the two CTAs of a cluster: a dense tcgen05.mma with cta_group::2
// computes M = 256 rows (128 k per CTA, from that CTA's expanded tile) by
// N = BN columns, each CTA staging half of the tile's dY rows.  Per CTA this
// halves the dY bytes staged per output element against the one-CTA kernel,
// whose small tiles re-read dY from L2 at ~100 flops per byte.
//
// Two rings per CTA: the operand ring (OPS stages of the dense tile and the
// dY half) and, deeper, the compressed-tile ring (VES stages of values and
// metadata, 9 KB each), so that the compressed tiles are in shared memory
// long before their dense slot frees and the expansion is the only step
// between a slot freeing and the MMA that refills it.
// Roles (480 threads per CTA, both CTAs):
//  * warp 14, compressed-tile producer: per stage, this CTA's values and
//    metadata of 64 rows of A x its 128 k into the next compressed slot, once
//    the expansion warps have released it.
//  * warp 0, dY producer: per stage, its half of dY (BN / 2 rows x 64
//    m-elements) completing on the leader's full barrier (the cta_group::2
//    form of the tensor load), which the leader's producer arms for both
//    halves, once this CTA's own empty barrier (the MMA commit, multicast)
//    says the operand slot is free.
//  * warps 6-13, expansion, in two groups of 4 that take alternate stages:
//    once the compressed tile has landed and the operand slot is free, the
//    compressed tile -> this CTA's dense tile; the group releases the
//    compressed slot and signals the leader's expansion barrier: the leader's
//    warps arrive (4 arrivals, each expecting 4 bytes), the peer's warps
//    complete those bytes with a 4-byte st.async.
//  * warp 1 of the leader (cluster rank 0), MMA issuer: the whole warp waits
//    on the full and expansion barriers, one elected lane issues the pair
//    MMAs (M = 256, N = BN, K = 16, A transposed) and commits them to the
//    empty and accumulator barriers of both CTAs (multicast).  Warp 1 of each
//    CTA allocates and frees TMEM (cta_group::2, both CTAs together).
//  * warps 2-5, epilogue: this CTA's 128 rows of the accumulator; they arrive
//    on the leader's accumulator-empty barrier (8 arrivals, 4 of them remote).
#pragma once

#include "spmm_t.cuh"

namespace st24 {
namespace spt2 {

using spt::Params;

template <int DT, int BN_, int OPS_, int VES_>
struct Config {
  static constexpr int BM = 128;                 // output rows (k) per CTA (256 per pair)
  static constexpr int BN = BN_;                 // output columns (n) per pair tile
  static constexpr int BH = BN / 2;              // dY rows staged per CTA
  static constexpr int SM = 64;                  // rows of A (the reduction) per stage
  static constexpr int STAGES = OPS_;            // operand ring
  static constexpr int VES = VES_;               // compressed-tile ring
  static constexpr int THREADS = 480;
  static constexpr int V_BYTES = SM * 128;       // compressed values: [64 rows][128 B], 128-byte swizzle
  static constexpr int E_BYTES = SM * 16;        // metadata: [64 rows][16 B]
  static constexpr int B_BYTES = BH * 128;       // this CTA's half of dY: [BH rows][64 m], 128-byte swizzle
  static constexpr int A_BYTES = SM * BM * 2;    // dense tile: [2 k-blocks][8 m-groups][8 rows][128 B]
  static constexpr int A_OFF = 0;                // 1024-aligned (swizzle atoms)
  static constexpr int B_OFF = A_OFF + A_BYTES;
  static constexpr int STAGE_BYTES = (B_OFF + B_BYTES + 1023) / 1024 * 1024;
  static constexpr int V_OFF = 0;                // in a compressed slot
  static constexpr int E_OFF = V_OFF + V_BYTES;
  static constexpr int VE_STAGE_BYTES = (E_OFF + E_BYTES + 1023) / 1024 * 1024;
  static constexpr int VE_BASE = STAGES * STAGE_BYTES;
  static constexpr int VE_TX = V_BYTES + E_BYTES;          // this CTA's compressed tile
  static constexpr int PAIR_B_TX = 2 * B_BYTES;            // both CTAs' dY halves
  static constexpr int TMEM_COLS = 2 * BN;
  static constexpr int BAR_BYTES = 1024;
  static constexpr int BAR_OFF = VE_BASE + VES * VE_STAGE_BYTES;
  static constexpr int SMEM_BYTES = BAR_OFF + BAR_BYTES + 64 + 1024;   // barriers, selectors, alignment
  static constexpr uint32_t FMT = (DT == kBF16) ? 1u : 0u;
  // Instruction descriptor: dense, fp32 accumulator, A MN-major (transposed), B K-major, N = BN, M = 256.
  static constexpr uint32_t IDESC = (1u << 4) | (FMT << 7) | (FMT << 10) | (1u << 15) |
                                    (static_cast<uint32_t>(BN >> 3) << 17) | (static_cast<uint32_t>(256 >> 4) << 24);
  static_assert(BN % 32 == 0 && BN >= 64 && BN <= 256, "N of the pair MMA; dY halves of whole 16-row blocks");
  static_assert(VE_BASE % 1024 == 0 && VE_STAGE_BYTES % 1024 == 0, "128-byte swizzle atoms of the values");
  static_assert(TMEM_COLS <= 512, "tensor memory");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
  static_assert(VES >= STAGES && VES <= 32, "compressed ring at least as deep as the operand ring");
  // full, expd, empty per operand stage; vfull, vempty per compressed stage; tfull, tempty (2 each);
  // drain; tmem slot; st.async sinks
  static_assert((3 * STAGES + 2 * VES + 5) * 8 + 8 + STAGES * 8 * 4 <= BAR_BYTES, "barrier region");
};

template <int DT, int BN, int STAGES, int VES>
__global__ void __launch_bounds__(480, 1)
    spmm_t2_kernel(const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmE,
                   const __grid_constant__ CUtensorMap tmB, const Params p) {
  using Cfg = Config<DT, BN, STAGES, VES>;
  constexpr uint16_t kBoth = 0x3;
  if (threadIdx.x == 0) grid_launch_dependents();

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + Cfg::BAR_OFF);   // [STAGES] leader: dY halves
  uint64_t* expd_bar = full_bar + STAGES;      // [STAGES] leader: both dense tiles written
  uint64_t* empty_bar = expd_bar + STAGES;     // [STAGES] MMAs done with the operand slot (both CTAs)
  uint64_t* vfull_bar = empty_bar + STAGES;    // [VES] this CTA's compressed tile landed
  uint64_t* vempty_bar = vfull_bar + VES;      // [VES] the expansion warps are done with the compressed slot
  uint64_t* tfull_bar = vempty_bar + VES;      // [2] accumulator ready (both CTAs)
  uint64_t* tempty_bar = tfull_bar + 2;        // [2] leader: accumulator drained in both CTAs
  uint64_t* drain_bar = tempty_bar + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain_bar + 1);
  uint32_t* sink = tmem_slot + 2;              // [STAGES][8] targets of the peer's expansion signals
  uint32_t* sel_tab = reinterpret_cast<uint32_t*>(smem + Cfg::BAR_OFF + Cfg::BAR_BYTES);   // [16]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();     // 0: the leader, which issues the pair MMAs
  const int64_t G = gridDim.x / 2, pair = blockIdx.x / 2;
  const int64_t tiles = p.tiles_k * p.tiles_n, MI = p.m_iters;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&expd_bar[s]), 4);   // the 4 warps of the group expanding the stage
      mbar_init(smem_u32(&empty_bar[s]), 1);
    }
    for (int v = 0; v < VES; ++v) {
      mbar_init(smem_u32(&vfull_bar[v]), 1);
      mbar_init(smem_u32(&vempty_bar[v]), 4);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&tfull_bar[b]), 1);
      mbar_init(smem_u32(&tempty_bar[b]), 8);
    }
    mbar_init(smem_u32(drain_bar), 1);
    fence_barrier_init();
  }
  if (threadIdx.x < 16) {
    // Byte-permute selectors of one group (as in the one-CTA kernel).
    const int i0 = threadIdx.x & 3, i1 = threadIdx.x >> 2;
    uint32_t sel = 0;
    for (int pos = 0; pos < 4; ++pos) {
      const uint32_t src = pos == i0 ? 0x10u : (pos == i1 ? 0x32u : 0x44u);
      sel |= src << (8 * pos);
    }
    sel_tab[threadIdx.x] = sel;
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), Cfg::TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();   // both CTAs' barriers initialised and TMEM allocated before any cross-CTA use
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  grid_dependency_wait();   // every input may come from the previous kernel on the stream

  if (warp == 14) {
    // ------------------------------------------------------------ compressed-tile producer
    if (lane == 0) {
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmE);
      const uint64_t keep = policy_evict_last();
      int vs = 0;
      uint32_t vph = 0;
      uint32_t issued = 0, issued_parity = 0;
      bool ok = true;
      for (int64_t t = pair; ok && t < tiles; t += G) {
        const int64_t kt = t % p.tiles_k;
        const int64_t k0 = kt * 256 + rank * Cfg::BM;          // this CTA's first output row
        for (int64_t mi = 0; mi < MI; ++mi) {
          if (!mbar_wait(smem_u32(&vempty_bar[vs]), vph ^ 1u, p.status)) { ok = false; break; }
          uint8_t* sv = smem + Cfg::VE_BASE + vs * Cfg::VE_STAGE_BYTES;
          const uint32_t vb = smem_u32(&vfull_bar[vs]);
          const int32_t m0 = static_cast<int32_t>(mi * Cfg::SM);
          mbar_arrive_expect_tx(vb, Cfg::VE_TX);
          tma_load_2d(smem_u32(sv + Cfg::V_OFF), &tmV, static_cast<int32_t>(k0 / 2), m0, vb, keep);
          tma_load_2d(smem_u32(sv + Cfg::E_OFF), &tmE, static_cast<int32_t>(k0 / 8), m0, vb, keep);
          issued |= 1u << vs;
          issued_parity = (issued_parity & ~(1u << vs)) | (vph << vs);
          if (++vs == VES) { vs = 0; vph ^= 1u; }
        }
      }
      // No copy may still be landing when the CTA exits.
      for (int v = 0; v < VES; ++v)
        if ((issued >> v) & 1u) mbar_wait(smem_u32(&vfull_bar[v]), (issued_parity >> v) & 1u, p.status);
    }
  } else if (warp == 0) {
    // ------------------------------------------------------------ dY producer
    if (lane == 0) {
      tma_prefetch_desc(&tmB);
      // dY evict-first: each panel is read by the tiles of one wave, while the
      // compressed weight is re-read by every panel and stays resident
      // (11008x4096 at N = 4096: DRAM reads 282 -> 215 MB per launch).
      const uint64_t keep = policy_evict_first();
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0, issued_parity = 0;
      bool ok = true;
      for (int64_t t = pair; ok && t < tiles; t += G) {
        const int64_t nt = t / p.tiles_k;
        for (int64_t mi = 0; mi < MI; ++mi) {
          if (!mbar_wait(smem_u32(&empty_bar[stage]), phase ^ 1u, p.status)) { ok = false; break; }
          uint8_t* st = smem + stage * Cfg::STAGE_BYTES;
          const uint32_t fb = smem_u32(&full_bar[stage]);
          const int32_t m0 = static_cast<int32_t>(mi * Cfg::SM);
          if (rank == 0) mbar_arrive_expect_tx(fb, Cfg::PAIR_B_TX);
          tma_load_2d_pair(smem_u32(st + Cfg::B_OFF), &tmB, m0, static_cast<int32_t>(nt * BN + rank * Cfg::BH), fb, 0,
                           keep);
          issued |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      // The leader's full barrier counts both CTAs' dY bytes (the peer waits
      // for the leader at the final cluster barrier).
      if (rank == 0)
        for (int s = 0; s < STAGES; ++s)
          if ((issued >> s) & 1u) mbar_wait_cluster(smem_u32(&full_bar[s]), (issued_parity >> s) & 1u, p.status);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (leader)
    // The whole warp runs the loop (warp-uniform addresses and descriptors);
    // one elected lane issues the MMAs and commits.
    if (rank == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int abuf = 0;
      uint32_t aphase = 0;
      bool ok = true;
      const uint32_t smem0 = smem_u32(smem);
      for (int64_t t = pair; ok && t < tiles; t += G) {
        ok = __all_sync(0xffffffffu, mbar_wait_cluster(smem_u32(&tempty_bar[abuf]), aphase ^ 1u, p.status));
        if (!ok) break;
        tc_fence_after();
        const uint32_t d = tmem + static_cast<uint32_t>(abuf * BN);
        for (int64_t mi = 0; mi < MI; ++mi) {
          // both CTAs' dY halves, then both CTAs' dense tiles
          ok = __all_sync(0xffffffffu, mbar_wait_cluster(smem_u32(&full_bar[stage]), phase, p.status) &&
                                           mbar_wait_cluster(smem_u32(&expd_bar[stage]), phase, p.status));
          if (!ok) break;
          tc_fence_after();
          const uint32_t st = smem0 + static_cast<uint32_t>(stage * Cfg::STAGE_BYTES);
          const uint64_t da = smem_desc(st + Cfg::A_OFF, 8192, 1024, kSwizzle128B);
          const uint64_t db = smem_desc(st + Cfg::B_OFF, 16, 1024, kSwizzle128B);
          if (elect_one_lane()) {
#pragma unroll
            for (int j = 0; j < Cfg::SM / 16; ++j) {
              // A: rows 16j..16j+15 of the dense tile (two 8-row groups, 1 KB
              // apart); B: 16 m-elements = 32 B.  Start addresses advance in
              // 16-byte units (no carry: shared memory < 256 KB).
              tc_mma_f16_pair(d, da + static_cast<uint64_t>(j * (2048 >> 4)), db + static_cast<uint64_t>(j * (32 >> 4)),
                              Cfg::IDESC, (mi > 0 || j > 0) ? 1u : 0u);
            }
            tc_commit_pair(smem_u32(&empty_bar[stage]), kBoth);
          }
          __syncwarp();
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        if (elect_one_lane()) tc_commit_pair(smem_u32(&tfull_bar[abuf]), kBoth);
        __syncwarp();
        if (++abuf == 2) { abuf = 0; aphase ^= 1u; }
      }
      // Both CTAs learn when every pair MMA has completed (before TMEM is freed).
      if (elect_one_lane()) tc_commit_pair(smem_u32(drain_bar), kBoth);
      __syncwarp();
      mbar_wait(smem_u32(drain_bar), 0, p.status);
    } else if (lane == 0) {
      mbar_wait(smem_u32(drain_bar), 0, p.status);
    }
  } else if (warp >= 6) {
    // ------------------------------------------------------------ expansion
    // Two groups of 4 warps take alternate stages (group 0 the even ones of
    // this CTA's sequence), so that two stages expand at once: a stage's
    // expansion is a chain of dependent shared-memory steps, and one group
    // alone left the MMA waiting on it.  Thread e of a group: row r of the
    // stage, chunks c = 8h..8h+7, chunk c = the 8 k of groups 2c, 2c+1 = one
    // 16-byte run of the dense row.  The 8 lanes of each quarter-warp take 8
    // consecutive rows with the same h, so that their 16-byte reads (values
    // stored with the 128-byte swizzle) and writes (the dense tile's swizzle)
    // fall in 8 different bank quads.
    const int ew = warp - 6;                     // expansion warp 0-7
    const int grp = ew >> 2;
    const int e = (threadIdx.x - 192) & 127;
    const int r = ((e >> 4) << 3) | (e & 7), h = (e >> 3) & 1;
    const int g = r >> 3, rr = r & 7;
    int stage = 0, vs = 0;
    uint32_t phase = 0, vph = 0;
    int par = 0;                                  // parity of this CTA's stage sequence
    for (int64_t t = pair; t < tiles; t += G) {
      bool ok = true;
      for (int64_t mi = 0; mi < MI; ++mi) {
        if (par == grp) {
          // the compressed tile has landed, and the MMAs of this operand slot's last use are done
          if (!mbar_wait(smem_u32(&vfull_bar[vs]), vph, p.status) ||
              !mbar_wait(smem_u32(&empty_bar[stage]), phase ^ 1u, p.status)) { ok = false; break; }
          uint8_t* st = smem + stage * Cfg::STAGE_BYTES;
          const uint8_t* sv = smem + Cfg::VE_BASE + vs * Cfg::VE_STAGE_BYTES;
          uint32_t vw[16];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const uint4 v = *reinterpret_cast<const uint4*>(sv + Cfg::V_OFF + r * 128 + (((4 * h + u) ^ rr) << 4));
            vw[4 * u] = v.x; vw[4 * u + 1] = v.y; vw[4 * u + 2] = v.z; vw[4 * u + 3] = v.w;
          }
          const uint2 mb = *reinterpret_cast<const uint2*>(sv + Cfg::E_OFF + r * 16 + h * 8);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            // chunk c = 8h + i of the row: k in [8c, 8c + 8); its metadata byte holds groups 2c and 2c+1
            const uint32_t byte = ((i < 4 ? mb.x : mb.y) >> (8 * (i & 3))) & 0xFFu;
            const uint32_t s0 = sel_tab[byte & 15u], s1 = sel_tab[byte >> 4];
            uint4 o;
            o.x = __byte_perm(vw[2 * i], 0u, s0 & 0xFFFFu);
            o.y = __byte_perm(vw[2 * i], 0u, s0 >> 16);
            o.z = __byte_perm(vw[2 * i + 1], 0u, s1 & 0xFFFFu);
            o.w = __byte_perm(vw[2 * i + 1], 0u, s1 >> 16);
            // k-block h, 16-byte run i inside it
            *reinterpret_cast<uint4*>(st + Cfg::A_OFF + h * 8192 + g * 1024 + rr * 128 + ((i ^ rr) << 4)) = o;
          }
          fence_proxy_async_smem();   // the dense tile is read by the tensor core (async proxy)
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(smem_u32(&vempty_bar[vs]));   // the compressed slot may be refilled
            if (rank == 0)
              mbar_arrive_expect_tx(smem_u32(&expd_bar[stage]), 4);
            else
              signal_tx_cluster(smem_u32(&sink[stage * 8 + ew]), smem_u32(&expd_bar[stage]), 0);
          }
        }
        par ^= 1;
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        if (++vs == VES) { vs = 0; vph ^= 1u; }
      }
      if (!ok) break;
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    int abuf = 0;
    uint32_t aphase = 0;
    for (int64_t t = pair; t < tiles; t += G) {
      const int64_t kt = t % p.tiles_k, nt = t / p.tiles_k;
      const int64_t k = kt * 256 + rank * Cfg::BM + 32 * q + lane;   // output row
      const int64_t n_base = nt * BN;
      if (!mbar_wait(smem_u32(&tfull_bar[abuf]), aphase, p.status)) break;
      tc_fence_after();
      const uint32_t tacc = tmem + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(abuf * BN);
      with_float_c_type(p.c_type, [&](auto ct) {
        constexpr int CT = decltype(ct)::value;
        constexpr int CH = 16;
#pragma unroll 1
        for (int c = 0; c < BN; c += CH) {
          if (n_base + c >= p.N) break;
          float bc[CH];
          if (p.beta != 0.0f) load_row_chunk_beta_c<CT, CH>(p, k, n_base + c, bc);
          uint32_t v[CH];
          tmem_ld_x16(tacc + c, v);
          tmem_ld_wait();
          store_row_chunk_bits<CT, CH>(p, k, n_base + c, v, bc, p.alpha);
        }
      });
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(smem_u32(&tempty_bar[abuf]), 0);
      if (++abuf == 2) { abuf = 0; aphase ^= 1u; }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem, Cfg::TMEM_COLS);
  // Neither CTA leaves while the other may still arrive on its barriers.
  cluster_sync();
}

}  // namespace spt2
}  // namespace st24
