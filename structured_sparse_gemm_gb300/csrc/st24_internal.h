// st24_internal.h -- declarations shared between the C-ABI layer (st24_api.cu)
// and the kernel translation units.  Not part of the public interface.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "st24.h"

namespace st24 {

constexpr int kF16 = ST24_F16;
constexpr int kBF16 = ST24_BF16;
constexpr int kE4M3 = ST24_E4M3;
constexpr int kS8 = ST24_S8;
constexpr int kF32 = ST24_F32;
constexpr int kS32 = ST24_S32;

__host__ __device__ inline int elem_size(int dt) {
  switch (dt) {
    case kF16: case kBF16: return 2;
    case kE4M3: case kS8: return 1;
    case kF32: case kS32: return 4;
    default: return 0;
  }
}

__host__ __device__ inline int64_t meta_row_bytes(int64_t K) { return (K / 4 + 1) / 2; }

// Per-device state the launchers need.
struct DeviceInfo {
  int device = -1;
  int num_sms = 0;
  unsigned* status = nullptr;   // device address of this device's status word
};
// Info for the current device (queried once per device).  nullptr on failure.
const DeviceInfo* current_device_info();

// ---------------------------------------------------------- prune / compress
st24_status launch_prune_compress(int dt, const void* W, int64_t M, int64_t K, int64_t ldw,
                                  void* values, void* meta, cudaStream_t stream);
// N:M prune into one 2:4 form (two = false, n <= 2) or two (two = true, n <= 4).
st24_status launch_prune_compress_nm(int dt, int n, int m, bool two, const void* W, int64_t M, int64_t K,
                                     int64_t ldw, void* values, void* meta, cudaStream_t stream);
st24_status launch_quantize_prune_compress(int src, int dst, const void* W, int64_t M, int64_t K, int64_t ldw,
                                           void* values, void* meta, float* scales, cudaStream_t stream);
st24_status launch_decompress(int dt, const void* values, const void* meta, int64_t M, int64_t K,
                              void* W, int64_t ldw, cudaStream_t stream);

// ---------------------------------------------------------------- SpMM
struct SpmmArgs {
  int ab, c;
  int64_t M, N, K;         // K: A's extent along K (twice B's for a two-form product)
  int64_t Kb;              // K of B (the contraction); 0 means K
  float alpha, beta;
  const void* values;
  const void* meta;
  const void* B;
  int64_t ldb;
  void* C;
  int64_t ldc;
  const float* row_scale;
  void* workspace;
  size_t ws_bytes;
  unsigned flags;          // st24_spmm_flags
};

// A split of the output into BM x BN tiles and of each tile's K loop into
// k-blocks, shared out over a persistent grid: dp_tiles whole tiles in
// data-parallel waves, then sk_tiles tiles whose (tile, k-block) iterations are
// split evenly over the grid (stream-K).
struct StreamKPlan {
  int bm, bn, bk;          // tile shape; bk in logical K
  int64_t tiles_m, tiles_n, k_iters;
  int64_t dp_tiles, sk_tiles;
  int64_t group_m;         // raster: tiles run in groups of group_m m-tiles, n-tile outer inside a group
  int grid;                // CTAs
  int cluster;             // > 1: each split tile's CTAs form one cluster and reduce through DSMEM
  int pair;                // tcgen05 CTA-pair tiles (bm = 256): `grid` counts pairs of CTAs
  size_t partial_bytes;    // bytes of one fp32 partial tile
  size_t ws_bytes;         // workspace bytes (0 if no tile is split)
};

// A stream-K plan over a persistent grid of at most num_sms CTAs.
// a_row_bytes / b_col_bytes: HBM bytes of one row of A (values + metadata) and
// of one column of B, used to pick the tile raster that keeps one operand in L2.
// allow_cluster: the kernel can reduce split tiles inside a thread-block
// cluster (no workspace) when every tile is split over the same 2..8 CTAs.
StreamKPlan make_stream_k_plan(int bm, int bn, int bk, int64_t M, int64_t N, int64_t K, int num_sms,
                               double a_row_bytes, double b_col_bytes, bool allow_cluster);

// Host-side argument checks of st24_spmm (no CUDA call is made).
st24_status check_spmm_args(const SpmmArgs& a);

// The plan of the kernel family st24_spmm picks for these arguments.
StreamKPlan plan_auto(const SpmmArgs& a, int num_sms);

// The mma.sp (warp-level sparse MMA) path: every element type.
StreamKPlan plan_spmm_mmasp(const SpmmArgs& a, int num_sms);
st24_status launch_spmm_mmasp(const SpmmArgs& a, const StreamKPlan& plan, const DeviceInfo& dev,
                              cudaStream_t stream);

// The register-direct mma.sp path: N <= 32, every input type (no workspace).
bool direct_applies(const SpmmArgs& a);
// Whether its grid (two CTAs per SM) runs in one wave on num_sms SMs.
bool direct_one_wave(const SpmmArgs& a, int num_sms);
st24_status launch_spmm_direct(const SpmmArgs& a, const DeviceInfo& dev, cudaStream_t stream);

// The narrow-N tcgen05 path (N <= 64; f16, bf16, e4m3): balanced stream-K,
// two CTAs per SM so consecutive products overlap.
bool narrow_applies(const SpmmArgs& a);
StreamKPlan plan_spmm_nt(const SpmmArgs& a, int num_sms);
st24_status launch_spmm_nt(const SpmmArgs& a, const StreamKPlan& plan, const DeviceInfo& dev,
                           cudaStream_t stream);

// The tcgen05 (5th-generation tensor core) path: f16, bf16, e4m3.
StreamKPlan plan_spmm_tc(const SpmmArgs& a, int num_sms);
st24_status launch_spmm_tc(const SpmmArgs& a, const StreamKPlan& plan, const DeviceInfo& dev,
                           cudaStream_t stream);
// C = beta * C when K == 0.
st24_status launch_scale_c(const SpmmArgs& a, const DeviceInfo& dev, cudaStream_t stream);

// Tensor maps (driver entry point fetched through the runtime, so the library
// has no link-time dependency on libcuda).
bool encode_tensor_map_2d(CUtensorMap* map, CUtensorMapDataType type, const void* base,
                          uint64_t inner, uint64_t outer, uint64_t row_stride_bytes,
                          uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle);
// A 3-D tiled tensor map: dims[0] innermost (contiguous), strides_bytes[i] =
// stride of dimension i + 1.
bool encode_tensor_map_3d(CUtensorMap* map, CUtensorMapDataType type, const void* base, const uint64_t dims[3],
                          const uint64_t strides_bytes[2], const uint32_t box[3], CUtensorMapSwizzle swizzle);

}  // namespace st24
