// spmm_t.cuh -- the transposed use of a compressed weight: dX = alpha * dY * A
// + beta * dX for A (M x K) in the 2:4 compressed form, on the
// 5th-generation tensor cores (dense tcgen05.mma, f16 / bf16).
//
// Method ("Chapter 26 -- Sparsity: The Hardware View", section "2:4: ~2x on
// the Matmul, Less End-to-End": train dense, prune to 2:4, retrain).
// Retraining a layer Y = X * A^T needs its input gradient dX = dY * A, a sum
// over M, along which A has no 2:4 structure: the sparse MMA cannot take it.
// Instead each stage's compressed tile (64 rows of A x 128 K: kept values and
// their 2-bit indices) is expanded in shared memory into the dense tile it
// stands for -- every kept pair written to the two K positions its indices
// name, zeros elsewhere -- and a dense MMA multiplies that tile, read
// transposed (K is its contiguous dimension), by the matching tile of dY.
// The weight is read from HBM in its compressed form (~56% of the dense
// bytes); the dense form exists only in shared memory.
//
//   out(k, n) = alpha * sum_m A(m, k) * dY(n, m) + beta * C(k, n),
//   dY(n, m) at B[n * ldb + m] (row-major [N, M]), C(k, n) at C[n * ldc + k].
//
// One persistent CTA per SM over output tiles of 128 k x BN n, each tile a
// full sweep over M in stages of 64 rows.  Roles (448 threads):
//  * warp 0: TMA producer -- per stage the values (64 rows x 128 B), the
//    metadata (64 rows x 16 B) and dY (BN rows x 128 B, 128-byte swizzle);
//  * warps 6-13: expansion -- each thread turns 4 groups-pairs of one row
//    into 16-byte runs of the dense tile (two byte permutes per group, the
//    selector taken from a 16-entry table of index pairs), written in the
//    MN-major 128-byte-swizzled layout the MMA reads;
//  * warp 1: MMA issuer (M = 128, N = BN, K = 16, A transposed) into a
//    double-buffered TMEM accumulator, and the TMEM allocation;
//  * warps 2-5: epilogue (alpha / beta / rounding), one 32-lane quadrant each.
#pragma once

#include "st24_epilogue.cuh"

namespace st24 {
namespace spt {

template <int DT, int BN_, int STAGES_>
struct Config {
  static constexpr int BM = 128;                 // output rows (k) per tile
  static constexpr int BN = BN_;                 // output columns (n) per tile
  static constexpr int SM = 64;                  // rows of A (the reduction) per stage
  static constexpr int STAGES = STAGES_;
  static constexpr int THREADS = 448;
  static constexpr int EXPAND_THREADS = 256;
  static constexpr int V_BYTES = SM * 128;       // compressed values: [64 rows][128 B], 128-byte swizzle
  static constexpr int E_BYTES = SM * 16;        // metadata: [64 rows][16 B]
  static constexpr int B_BYTES = BN * 128;       // dY: [BN rows][64 m-elements], 128-byte swizzle
  static constexpr int A_BYTES = SM * BM * 2;    // dense tile: [2 k-blocks][8 m-groups][8 rows][128 B]
  static constexpr int A_OFF = 0;                // 1024-aligned (swizzle atoms)
  static constexpr int B_OFF = A_OFF + A_BYTES;
  static constexpr int V_OFF = B_OFF + B_BYTES;
  static constexpr int E_OFF = V_OFF + V_BYTES;
  static constexpr int STAGE_BYTES = (E_OFF + E_BYTES + 1023) / 1024 * 1024;
  static constexpr int TX = B_BYTES + V_BYTES + E_BYTES;
  static constexpr int TMEM_COLS = 2 * BN;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 256 + 64 + 1024;   // barriers, selector table, alignment
  static constexpr uint32_t FMT = (DT == kBF16) ? 1u : 0u;
  // Instruction descriptor: dense, fp32 accumulator, A MN-major (transposed), B K-major, N = BN, M = 128.
  static constexpr uint32_t IDESC = (1u << 4) | (FMT << 7) | (FMT << 10) | (1u << 15) |
                                    (static_cast<uint32_t>(BN >> 3) << 17) | (static_cast<uint32_t>(BM >> 4) << 24);
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "N of the MMA");
  static_assert(V_OFF % 1024 == 0, "128-byte swizzle atoms of the values");
  static_assert(TMEM_COLS <= 512, "tensor memory");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
  static_assert((4 * STAGES + 5) * 8 + 8 <= 256, "barrier region");
};

struct Params : OutParams {        // OutParams: M = K of the weight (output rows), N, C (the dX), ldc
  int64_t Mw;                      // rows of the weight (the reduction)
  int64_t tiles_k, tiles_n, m_iters;
  unsigned* status;
};

template <int DT, int BN, int STAGES>
__global__ void __launch_bounds__(448, 1)
    spmm_t_kernel(const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmE,
                  const __grid_constant__ CUtensorMap tmB, const Params p) {
  using Cfg = Config<DT, BN, STAGES>;
  if (threadIdx.x == 0) grid_launch_dependents();

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + STAGES * Cfg::STAGE_BYTES);   // [STAGES] TMA landed
  uint64_t* expd_bar = full_bar + STAGES;      // [STAGES] dense tile written
  uint64_t* empty_bar = expd_bar + STAGES;     // [STAGES] MMAs done with the stage
  uint64_t* tfull_bar = empty_bar + STAGES;    // [2]
  uint64_t* tempty_bar = tfull_bar + 2;        // [2]
  uint64_t* drain_bar = tempty_bar + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain_bar + 1);
  uint32_t* sel_tab = reinterpret_cast<uint32_t*>(smem + STAGES * Cfg::STAGE_BYTES + 256);   // [16]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t G = gridDim.x, cta = blockIdx.x;
  const int64_t tiles = p.tiles_k * p.tiles_n, MI = p.m_iters;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&expd_bar[s]), 8);
      mbar_init(smem_u32(&empty_bar[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&tfull_bar[b]), 1);
      mbar_init(smem_u32(&tempty_bar[b]), 4);
    }
    mbar_init(smem_u32(drain_bar), 1);
    fence_barrier_init();
  }
  if (threadIdx.x < 16) {
    // Byte-permute selectors of one group: index pair (i0, i1) = (nib & 3,
    // nib >> 2); the group's 4 outputs (two 32-bit words) take bytes 0-1 of
    // the value pair at position i0, bytes 2-3 at position i1, zero elsewhere.
    const int i0 = threadIdx.x & 3, i1 = threadIdx.x >> 2;
    uint32_t sel = 0;
    for (int pos = 0; pos < 4; ++pos) {
      const uint32_t src = pos == i0 ? 0x10u : (pos == i1 ? 0x32u : 0x44u);
      sel |= src << (8 * pos);
    }
    sel_tab[threadIdx.x] = sel;
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), Cfg::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  grid_dependency_wait();   // every input may come from the previous kernel on the stream

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmE);
      tma_prefetch_desc(&tmB);
      const uint64_t keep = policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0, issued_parity = 0;
      bool ok = true;
      for (int64_t t = cta; ok && t < tiles; t += G) {
        const int64_t kt = t % p.tiles_k, nt = t / p.tiles_k;
        for (int64_t mi = 0; mi < MI; ++mi) {
          if (!mbar_wait(smem_u32(&empty_bar[stage]), phase ^ 1u, p.status)) { ok = false; break; }
          uint8_t* st = smem + stage * Cfg::STAGE_BYTES;
          const uint32_t fb = smem_u32(&full_bar[stage]);
          const int32_t m0 = static_cast<int32_t>(mi * Cfg::SM);
          mbar_arrive_expect_tx(fb, Cfg::TX);
          tma_load_2d(smem_u32(st + Cfg::V_OFF), &tmV, static_cast<int32_t>(kt * 64), m0, fb, keep);
          tma_load_2d(smem_u32(st + Cfg::E_OFF), &tmE, static_cast<int32_t>(kt * 16), m0, fb, keep);
          tma_load_2d(smem_u32(st + Cfg::B_OFF), &tmB, m0, static_cast<int32_t>(nt * BN), fb, keep);
          issued |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      for (int s = 0; s < STAGES; ++s)
        if ((issued >> s) & 1u) mbar_wait(smem_u32(&full_bar[s]), (issued_parity >> s) & 1u, p.status);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the loop (warp-uniform addresses and descriptors);
    // one elected lane issues the MMAs and commits.
    int stage = 0;
    uint32_t phase = 0;
    int abuf = 0;
    uint32_t aphase = 0;
    bool ok = true;
    const uint32_t smem0 = smem_u32(smem);
    for (int64_t t = cta; ok && t < tiles; t += G) {
      ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&tempty_bar[abuf]), aphase ^ 1u, p.status));
      if (!ok) break;
      tc_fence_after();
      const uint32_t d = tmem + static_cast<uint32_t>(abuf * BN);
      for (int64_t mi = 0; mi < MI; ++mi) {
        ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&expd_bar[stage]), phase, p.status) &&
                                         mbar_wait(smem_u32(&full_bar[stage]), phase, p.status));
        if (!ok) break;
        tc_fence_after();
        const uint32_t st = smem0 + static_cast<uint32_t>(stage * Cfg::STAGE_BYTES);
        const uint64_t da = smem_desc(st + Cfg::A_OFF, 8192, 1024, kSwizzle128B);
        const uint64_t db = smem_desc(st + Cfg::B_OFF, 16, 1024, kSwizzle128B);
        if (elect_one_lane()) {
#pragma unroll
          for (int j = 0; j < Cfg::SM / 16; ++j) {
            // A: rows 16j..16j+15 of the dense tile (two 8-row groups, 1 KB apart),
            // the 128 k in two 64-element blocks 8 KB apart; B: 16 m-elements = 32 B.
            // Start addresses advance in 16-byte units (no carry: shared memory < 256 KB).
            tc_mma_f16(d, da + static_cast<uint64_t>(j * (2048 >> 4)), db + static_cast<uint64_t>(j * (32 >> 4)),
                       Cfg::IDESC, (mi > 0 || j > 0) ? 1u : 0u);
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
    if (elect_one_lane()) tc_commit(smem_u32(drain_bar));
    __syncwarp();
    mbar_wait(smem_u32(drain_bar), 0, p.status);
  } else if (warp >= 6) {
    // ------------------------------------------------------------ expansion
    // Thread e: row r of the stage, chunks c = 4q..4q+3, chunk c = the 8 k of
    // groups 2c, 2c+1 = one 16-byte run of the dense row.  The 8 lanes of each
    // quarter-warp take 8 consecutive rows with the same q, so that their
    // 16-byte reads (values stored with the 128-byte swizzle) and writes (the
    // dense tile's swizzle) fall in 8 different bank quads.
    const int e = threadIdx.x - 192;
    const int r = ((e >> 5) << 3) | (e & 7), q = (e >> 3) & 3;
    const int g = r >> 3, rr = r & 7;
    int stage = 0;
    uint32_t phase = 0;
    for (int64_t t = cta; t < tiles; t += G) {
      bool ok = true;
      for (int64_t mi = 0; mi < MI; ++mi) {
        if (!mbar_wait(smem_u32(&full_bar[stage]), phase, p.status)) { ok = false; break; }
        uint8_t* st = smem + stage * Cfg::STAGE_BYTES;
        const uint4 v0 = *reinterpret_cast<const uint4*>(st + Cfg::V_OFF + r * 128 + (((2 * q) ^ rr) << 4));
        const uint4 v1 = *reinterpret_cast<const uint4*>(st + Cfg::V_OFF + r * 128 + (((2 * q + 1) ^ rr) << 4));
        const uint32_t mb = *reinterpret_cast<const uint32_t*>(st + Cfg::E_OFF + r * 16 + q * 4);
        const uint32_t vw[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int c = 4 * q + i;                       // chunk of the row: k in [8c, 8c + 8)
          const uint32_t byte = (mb >> (8 * i)) & 0xFFu;  // groups 2c (low nibble) and 2c+1
          const uint32_t s0 = sel_tab[byte & 15u], s1 = sel_tab[byte >> 4];
          uint4 o;
          o.x = __byte_perm(vw[2 * i], 0u, s0 & 0xFFFFu);
          o.y = __byte_perm(vw[2 * i], 0u, s0 >> 16);
          o.z = __byte_perm(vw[2 * i + 1], 0u, s1 & 0xFFFFu);
          o.w = __byte_perm(vw[2 * i + 1], 0u, s1 >> 16);
          const int b = c >> 3, cc = c & 7;               // k-block, 16-byte run inside it
          *reinterpret_cast<uint4*>(st + Cfg::A_OFF + b * 8192 + g * 1024 + rr * 128 + ((cc ^ rr) << 4)) = o;
        }
        fence_proxy_async_smem();   // the dense tile is read by the tensor core (async proxy)
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&expd_bar[stage]));
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
      if (!ok) break;
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    int abuf = 0;
    uint32_t aphase = 0;
    for (int64_t t = cta; t < tiles; t += G) {
      const int64_t kt = t % p.tiles_k, nt = t / p.tiles_k;
      const int64_t k = kt * Cfg::BM + 32 * q + lane;   // output row
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
      if (lane == 0) mbar_arrive(smem_u32(&tempty_bar[abuf]));
      if (++abuf == 2) { abuf = 0; aphase ^= 1u; }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, Cfg::TMEM_COLS);
}

template <int DT>
st24_status launch_dt(const SpmmArgs& a, const DeviceInfo& dev, cudaStream_t s);

}  // namespace spt
}  // namespace st24
