// spmm_nt.cuh -- narrow products (N <= 64) on the 5th-generation tensor cores:
// C = alpha * row_scale * (A_sparse * B) + beta * C with tcgen05.mma.sp, for
// f16, bf16 and fp8-e4m3 inputs.
//
// Method ("Chapter 26 -- Sparsity: The Hardware View", sections "2:4
// Fine-Grained Structured Sparsity" and "2:4 in the Memory-Bound Regime"):
// the stored pair of every group multiplies the two activations its metadata
// selects; with few activation columns the product is bound by streaming the
// compressed weights (values + metadata, ~56% of the dense bytes), so the
// kernel exists to keep HBM busy from the first byte to the last:
//
//  * Few, large copies.  A stage is C 128-byte chunks of K for 128 rows of
//    values (one 3-D TMA copy of C x 16 KB), their metadata (one copy) and
//    the matching 2C chunks of B (one 3-D copy): issuing a TMA copy costs the
//    issuing thread time in proportion to the rows it moves, and with one
//    2-D copy per 16 KB plus separate metadata and B copies a single producer
//    could not keep up with HBM (measured: 0.63 of the copy rate against 0.86
//    with this mix).
//  * Each 128-row tile's K range is split evenly over the S CTAs (1, 2, 4 or
//    8) of a thread-block cluster.  When its MMAs are done, each CTA pushes
//    its fp32 partial through distributed shared memory into a receive
//    buffer of the rows' owner (CTA r owns rows [r*128/S, (r+1)*128/S)) with
//    asynchronous stores counted on the owner's barrier; the owner sums the
//    S partials of its rows in rank (= K) order, deterministically.  No
//    workspace, no atomics, no global round trip, and no CTA waits for its
//    peers to finish -- only for the bytes it sums.
//  * Half an SM per CTA (registers, shared memory, tensor memory), so the CTA
//    of the next product on the stream (a programmatic dependent launch) is
//    resident beside this one: with fixed weights (ST24_SPMM_FIXED_A) it
//    fills its ring with weight tiles and warms L2 with the rest of its K
//    range before its dependency wait, and its metadata warps move the ring's
//    metadata into TMEM meanwhile, so HBM streams the next product's weights
//    while this one finishes and only B is read after the wait.
//  * Roles (320 threads): warp 0 issues the TMA copies; warp 1 issues the
//    sparse MMAs (M = 128, N = BN, one CTA) into a TMEM accumulator and owns
//    the allocation; warps 6-9 move each stage's metadata from shared memory
//    into TMEM in the order the sparse MMA reads it; warps 2-5 read the
//    accumulator out; the partial exchange and the output use every thread.
#pragma once

#include "st24_epilogue.cuh"

namespace st24 {
namespace nt {

template <int DT>
struct Traits {
  static constexpr int ES = (DT == kF16 || DT == kBF16) ? 2 : 1;
  static constexpr int KSTEP = 64 / ES;        // logical K per MMA
  static constexpr int CK = 4 * KSTEP;         // logical K per 128-byte chunk of values
  static constexpr int CHUNK_ELEMS = 128 / ES; // stored values (or B elements) per 128-byte chunk
  static constexpr uint32_t FMT = (DT == kBF16) ? 1u : 0u;   // f16 0, bf16 1; e4m3 0 (kind::f8f6f4)
};

constexpr int tmem_cols_for(int v) {
  int p = 32;
  while (p < v) p <<= 1;
  return p;
}

template <int DT, int BN_, int C_, int STAGES_, bool SPLIT_>
struct Config {
  using T = Traits<DT>;
  static constexpr bool SPLIT = SPLIT_;                // tiles split over a cluster: a receive buffer
  static constexpr int BM = 128;
  static constexpr int BN = BN_;
  static constexpr int C = C_;                         // 128-byte chunks of values per stage
  static constexpr int STAGES = STAGES_;
  static constexpr int THREADS = 320;
  static constexpr int BK = C * T::CK;                 // logical K per stage
  static constexpr int KSTEPS = 4 * C;                 // MMAs per stage
  static constexpr int EB = BK / 8;                    // metadata bytes per row per stage
  static constexpr int A_BYTES = C * BM * 128;         // [chunk][128 rows][128 B], 128-byte swizzle
  static constexpr int B_BYTES = 2 * C * BN * 128;     // [2C chunks][BN rows][128 B], 128-byte swizzle
  static constexpr int E_BYTES = BM * EB;              // [128 rows][EB B]
  static constexpr int STAGE_BYTES = (A_BYTES + B_BYTES + E_BYTES + 1023) / 1024 * 1024;
  static constexpr int RING_BYTES = STAGES * STAGE_BYTES;
  static constexpr int RECV_BYTES = SPLIT ? BM * BN * 4 : 0;   // [S][N][128/S] fp32 partials of owned rows
  static constexpr int META_COL0 = BN;                 // after the accumulator
  static constexpr int META_COLS = 4 * KSTEPS;         // per stage: MMA ks at column 4 * ks
  static constexpr int TMEM_COLS = tmem_cols_for(BN + STAGES * META_COLS);
  static constexpr int BAR_BYTES = 192;
  static constexpr int SMEM_BYTES = RING_BYTES + RECV_BYTES + BAR_BYTES + 1024;   // + alignment slack
  // Instruction descriptor: sparse, fp32 accumulator, K-major A and B, N = BN, M = 128.
  static constexpr uint32_t IDESC = (1u << 2) | (1u << 4) | (T::FMT << 7) | (T::FMT << 10) |
                                    (static_cast<uint32_t>(BN >> 3) << 17) | (static_cast<uint32_t>(BM >> 4) << 24);
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 64, "N of the MMA");
  static_assert(C == 1 || C == 2, "chunks per stage");
  static_assert(TMEM_COLS <= 256, "two CTAs share an SM's tensor memory");
  static_assert(SMEM_BYTES <= 113 * 1024, "two CTAs share an SM's shared memory");
  static_assert((4 * STAGES + 3) * 8 + 8 <= BAR_BYTES, "barrier region");
};

struct Params : OutParams {
  int64_t K;
  int64_t k_iters;   // k-blocks (stages) of the whole K
  int parts;         // S: CTAs per tile = cluster size (1, 2, 4 or 8)
  int a_fixed;       // load weight stages before the dependency wait
  int64_t kb_wrap;   // two-form product: k-blocks per form (B's k-block of k-block kb is kb mod kb_wrap); 0: one form
  unsigned* status;
};

template <int DT, int BN, int C, int STAGES, bool SPLIT>
__global__ void __launch_bounds__(320, 2)
    spmm_nt_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmE,
                   const __grid_constant__ CUtensorMap tmB, const Params p) {
  using Cfg = Config<DT, BN, C, STAGES, SPLIT>;
  using T = Traits<DT>;

  // The next kernel on the stream may start launching now: its CTAs fit
  // beside this one and begin streaming their own fixed weights.
  if (threadIdx.x == 0) grid_launch_dependents();

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* recv = reinterpret_cast<float*>(smem + Cfg::RING_BYTES);                 // partials of the rows this CTA owns
  uint64_t* fulla_bar = reinterpret_cast<uint64_t*>(smem + Cfg::RING_BYTES + Cfg::RECV_BYTES);   // [STAGES] values + metadata landed
  uint64_t* fullb_bar = fulla_bar + STAGES;     // [STAGES] B landed
  uint64_t* empty_bar = fullb_bar + STAGES;     // [STAGES] the MMAs are done with the stage
  uint64_t* meta_bar = empty_bar + STAGES;      // [STAGES] the stage's metadata is in TMEM
  uint64_t* tfull_bar = meta_bar + STAGES;      // the accumulator is complete
  uint64_t* drain_bar = tfull_bar + 1;
  uint64_t* recv_bar = drain_bar + 1;           // every partial of the owned rows has arrived
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(recv_bar + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = SPLIT ? p.parts : 1;
  const int r = S > 1 ? static_cast<int>(cluster_ctarank()) : 0;
  const int64_t tile = blockIdx.x / S;
  const int64_t KI = p.k_iters;
  const int64_t kb0 = div_nn(r * KI, S), kb1 = div_nn((r + 1) * KI, S);   // this CTA's k-blocks
  const int64_t n_units = kb1 - kb0;
  const int32_t m0 = static_cast<int32_t>(tile * Cfg::BM);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&fulla_bar[s]), 1);
      mbar_init(smem_u32(&fullb_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), 1);
      mbar_init(smem_u32(&meta_bar[s]), 4);
    }
    mbar_init(smem_u32(tfull_bar), 1);
    mbar_init(smem_u32(drain_bar), 1);
    mbar_init(smem_u32(recv_bar), 1);
    // S partials of (128 / S) rows x N columns, pushed by the cluster's CTAs
    if (SPLIT) mbar_arrive_expect_tx(smem_u32(recv_bar), static_cast<uint32_t>(Cfg::BM * p.N * 4));
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
  // Peers push partials into this CTA's receive buffer only after this
  // cluster barrier phase completes (waited on just before the first push):
  // every CTA's barriers are initialised by then.
  if (SPLIT) cluster_arrive_release();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      constexpr uint32_t kWeightTx = Cfg::A_BYTES + Cfg::E_BYTES;
      const uint64_t once = policy_evict_first();    // every weight byte is read once
      const uint64_t reuse = policy_evict_last();    // B is read by every tile
      auto load_weights = [&](int stage, int64_t kb) {
        uint8_t* st = smem + stage * Cfg::STAGE_BYTES;
        const uint32_t fb = smem_u32(&fulla_bar[stage]);
        mbar_arrive_expect_tx(fb, kWeightTx);
        tma_load_3d(smem_u32(st), &tmA, 0, m0, static_cast<int32_t>(kb * C), fb, once);
        tma_load_2d(smem_u32(st + Cfg::A_BYTES + Cfg::B_BYTES), &tmE, static_cast<int32_t>(kb * Cfg::EB), m0, fb,
                    once);
      };
      int pre = 0;
      if (p.a_fixed) {
        // The ring starts empty: fill it, then warm L2 with the k-blocks
        // after it (up to ~192 KB per CTA), so that after the dependency wait
        // the rest of this CTA's range streams from L2.
        pre = static_cast<int>(n_units < STAGES ? n_units : STAGES);
        for (int s = 0; s < pre; ++s) load_weights(s, kb0 + s);
        constexpr int kPrefetch = (192 * 1024) / (Cfg::A_BYTES + Cfg::E_BYTES);
        const int64_t pf_end = kb0 + pre + kPrefetch < kb1 ? kb0 + pre + kPrefetch : kb1;
        for (int64_t kb = kb0 + pre; kb < pf_end; ++kb) {
          tma_prefetch_l2_3d(&tmA, 0, m0, static_cast<int32_t>(kb * C));
          tma_prefetch_l2_2d(&tmE, static_cast<int32_t>(kb * Cfg::EB), m0);
        }
      }
      grid_dependency_wait();
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0, issued_parity = 0;   // per stage: copies were issued, and their phase
      for (int64_t j = 0; j < n_units; ++j) {
        const int64_t kb = kb0 + j;
        if (j >= pre) {
          if (!mbar_wait(smem_u32(&empty_bar[stage]), phase ^ 1u, p.status)) break;
          load_weights(stage, kb);
        }
        issued |= 1u << stage;
        issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
        const uint32_t bb = smem_u32(&fullb_bar[stage]);
        const int64_t kbb = (p.kb_wrap && kb >= p.kb_wrap) ? kb - p.kb_wrap : kb;
        mbar_arrive_expect_tx(bb, Cfg::B_BYTES);
        tma_load_3d(smem_u32(smem + stage * Cfg::STAGE_BYTES + Cfg::A_BYTES), &tmB, 0, 0,
                    static_cast<int32_t>(kbb * 2 * C), bb, reuse);
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
      // Never leave with copies in flight into this CTA's shared memory.
      for (int s = 0; s < STAGES; ++s)
        if ((issued >> s) & 1u) {
          mbar_wait(smem_u32(&fulla_bar[s]), (issued_parity >> s) & 1u, p.status);
          mbar_wait(smem_u32(&fullb_bar[s]), (issued_parity >> s) & 1u, p.status);
        }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the loop (warp-uniform addresses and descriptors);
    // one elected lane issues the MMAs and commits.
    int stage = 0;
    uint32_t phase = 0;
    const uint32_t smem0 = smem_u32(smem);
    const int64_t k_last = p.K - (KI - 1) * Cfg::BK;   // whole K-steps in the last k-block (others: KSTEPS)
    const int ksteps_last = k_last / T::KSTEP < Cfg::KSTEPS ? static_cast<int>(k_last / T::KSTEP) : Cfg::KSTEPS;
    for (int64_t kb = kb0; kb < kb1; ++kb) {
      const bool ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&meta_bar[stage]), phase, p.status) &&
                                                  mbar_wait(smem_u32(&fulla_bar[stage]), phase, p.status) &&
                                                  mbar_wait(smem_u32(&fullb_bar[stage]), phase, p.status));
      if (!ok) break;
      tc_fence_after();
      const uint32_t a0 = smem0 + static_cast<uint32_t>(stage * Cfg::STAGE_BYTES);
      const uint64_t da = smem_desc(a0, 16, 1024, kSwizzle128B);
      const uint64_t db = smem_desc(a0 + Cfg::A_BYTES, 16, 1024, kSwizzle128B);
      const uint32_t mcol = tmem + static_cast<uint32_t>(Cfg::META_COL0 + stage * Cfg::META_COLS);
      const int ksteps = kb == KI - 1 ? ksteps_last : Cfg::KSTEPS;
      if (elect_one_lane()) {
#pragma unroll
        for (int ks = 0; ks < Cfg::KSTEPS; ++ks) {
          if (ks >= ksteps) break;
          // descriptor start addresses advance in 16-byte units (no carry: shared memory < 256 KB)
          const uint64_t dak = da + static_cast<uint64_t>(((ks >> 2) * (Cfg::BM * 128) + (ks & 3) * 32) >> 4);
          const uint64_t dbk = db + static_cast<uint64_t>(((ks >> 1) * (BN * 128) + (ks & 1) * 64) >> 4);
          const uint32_t acc = (kb > kb0 || ks > 0) ? 1u : 0u;
          if constexpr (T::ES == 2)
            tc_mma_sp_f16(tmem, dak, dbk, mcol + 4 * ks, Cfg::IDESC, acc);
          else
            tc_mma_sp_f8f6f4(tmem, dak, dbk, mcol + 4 * ks, Cfg::IDESC, acc);
        }
        tc_commit(smem_u32(&empty_bar[stage]));
      }
      __syncwarp();
      if (++stage == STAGES) { stage = 0; phase ^= 1u; }
    }
    if (elect_one_lane()) {
      tc_commit(smem_u32(tfull_bar));
      // Every tcgen05 operation of this warp has completed before TMEM is freed.
      tc_commit(smem_u32(drain_bar));
    }
    __syncwarp();
    mbar_wait(smem_u32(drain_bar), 0, p.status);
  } else if (warp >= 6) {
    // ------------------------------------------------------------ metadata
    // Needs only the stage's values and metadata, not B: the stages loaded
    // before the dependency wait are moved into TMEM while the previous
    // kernel still runs.
    const int q = warp & 3;                 // TMEM lane quadrant of this warp
    const int row = 32 * q + lane;          // row of the tile this lane moves
    const uint32_t fill = 0x44444444u;      // index pair (0, 1): rows past M hold zero values
    const int64_t rows_valid = p.M - tile * Cfg::BM;
    int stage = 0;
    uint32_t phase = 0;
    for (int64_t kb = kb0; kb < kb1; ++kb) {
      if (!mbar_wait(smem_u32(&fulla_bar[stage]), phase, p.status)) break;
      const uint8_t* se = smem + stage * Cfg::STAGE_BYTES + Cfg::A_BYTES + Cfg::B_BYTES;
      const uint32_t taddr = tmem + (static_cast<uint32_t>(32 * q) << 16) +
                             static_cast<uint32_t>(Cfg::META_COL0 + stage * Cfg::META_COLS);
#pragma unroll
      for (int h = 0; h < C; ++h) {   // 16 columns (4 MMAs) at a time
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) w[i] = fill;
        if constexpr (T::ES == 2) {
          // Rows pair up as (r, r+8) in each 16-row block: lane r holds groups
          // 0-3 of both rows (low and high halfword), lane r+8 groups 4-7.
          const int j = row & 15;
          const int partner = j < 8 ? row + 8 : row - 8;
          const uint4 f4 = make_uint4(fill, fill, fill, fill);
          const uint4 own = row < rows_valid ? *reinterpret_cast<const uint4*>(se + row * Cfg::EB + 16 * h) : f4;
          const uint4 oth =
              partner < rows_valid ? *reinterpret_cast<const uint4*>(se + partner * Cfg::EB + 16 * h) : f4;
          const uint4 lo = j < 8 ? own : oth, hi = j < 8 ? oth : own;
          const uint32_t sel = j < 8 ? 0x5410u : 0x7632u;
          w[0] = __byte_perm(lo.x, hi.x, sel);
          w[4] = __byte_perm(lo.y, hi.y, sel);
          w[8] = __byte_perm(lo.z, hi.z, sel);
          w[12] = __byte_perm(lo.w, hi.w, sel);
        } else {
          // One row per lane, the canonical words in order, two per MMA.
          if (row < rows_valid) {
            const uint4 a = *reinterpret_cast<const uint4*>(se + row * Cfg::EB + 32 * h);
            const uint4 b = *reinterpret_cast<const uint4*>(se + row * Cfg::EB + 32 * h + 16);
            w[0] = a.x; w[1] = a.y; w[4] = a.z; w[5] = a.w;
            w[8] = b.x; w[9] = b.y; w[12] = b.z; w[13] = b.w;
          }
        }
        tmem_st_x16(taddr + 16 * h, w);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&meta_bar[stage]));
      if (++stage == STAGES) { stage = 0; phase ^= 1u; }
    }
  }

  // ------------------------------------------------------------ output
  // Warps 2-5 read the accumulator (one 32-lane quadrant each).  C and the
  // row scales are read only after the previous kernel has completed.
  const bool epi = warp >= 2 && warp <= 5;
  const int q = warp & 3;
  const int row = 32 * q + lane;
  const int64_t m = tile * Cfg::BM + row;
  const uint32_t tacc = tmem + (static_cast<uint32_t>(32 * q) << 16);
  constexpr int CH = 16;
  grid_dependency_wait();
  if (epi) {
    mbar_wait(smem_u32(tfull_bar), 0, p.status);
    tc_fence_after();
  }
  if (!SPLIT) {
    if (epi) {
      const bool row_ok = m < p.M;
      const float f = row_ok ? row_factor(p, m) : 0.0f;
      with_float_c_type(p.c_type, [&](auto ct) {
        constexpr int CT = decltype(ct)::value;
#pragma unroll 1
        for (int c = 0; c < BN; c += CH) {
          if (c >= p.N) break;
          float bc[CH];
          if (row_ok && p.beta != 0.0f) load_row_chunk_beta_c<CT, CH>(p, m, c, bc);
          uint32_t v[CH];
          tmem_ld_x16(tacc + c, v);
          tmem_ld_wait();
          if (row_ok) store_row_chunk_bits<CT, CH>(p, m, c, v, bc, f);
        }
      });
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, Cfg::TMEM_COLS);
    return;
  }

  // Split tile: push this CTA's partial of every row to the row's owner --
  // slot [r][n][row % RPO] of its receive buffer, columns n < N -- with
  // asynchronous stores counted on the owner's receive barrier.
  const int RPO = Cfg::BM / S;   // rows each CTA of the cluster owns
  const int N = static_cast<int>(p.N);
  cluster_wait();                // every CTA of the cluster has initialised its barriers
  if (epi) {
    const uint32_t owner = static_cast<uint32_t>(row / RPO);
    const uint32_t local = smem_u32(recv) + static_cast<uint32_t>((r * N * RPO + row % RPO) * 4);
    uint32_t remote, rbar;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(owner));
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rbar) : "r"(smem_u32(recv_bar)), "r"(owner));
#pragma unroll 1
    for (int c = 0; c < BN; c += CH) {
      if (c >= N) break;
      uint32_t v[CH];
      tmem_ld_x16(tacc + c, v);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < CH; ++j)
        if (c + j < N)
          asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(
                           remote + static_cast<uint32_t>((c + j) * RPO * 4)),
                       "r"(v[j]), "r"(rbar)
                       : "memory");
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, Cfg::TMEM_COLS);
  // This CTA sums its rows' S partials in rank (K) order and stores them.
  if (!mbar_wait_cluster(smem_u32(recv_bar), 0, p.status)) return;
  with_float_c_type(p.c_type, [&](auto ct) {
    constexpr int CT = decltype(ct)::value;
#pragma unroll 1
    for (int it = threadIdx.x; it < RPO * N; it += Cfg::THREADS) {
      const int n = it / RPO, lr = it - n * RPO;
      const int64_t mo = tile * Cfg::BM + r * RPO + lr;
      if (mo >= p.M) continue;
      const float* src = recv + n * RPO + lr;
      float t = src[0];
      for (int s = 1; s < S; ++s) t = t + src[s * N * RPO];
      float out = __fmul_rn(t, row_factor(p, mo));
      if (p.beta != 0.0f) out = __fadd_rn(out, __fmul_rn(p.beta, c_load<CT>(p.C, n * p.ldc + mo)));
      c_store<CT>(p.C, n * p.ldc + mo, out);
    }
  });
}

template <int DT>
st24_status launch_dt(const SpmmArgs& a, const StreamKPlan& plan, const DeviceInfo& dev, cudaStream_t s);

}  // namespace nt
}  // namespace st24
