// spmm_t_launch.cuh -- host launch of the transposed-use kernel for one
// element type (included by the per-type translation units).
#pragma once

#include "spmm_t2.cuh"

namespace st24 {
namespace spt {

template <int DT, int BN, int STAGES>
st24_status launch_cfg(const SpmmArgs& a, const DeviceInfo& dev, cudaStream_t stream) {
  using Cfg = Config<DT, BN, STAGES>;
  // A's values (K/2 per row) and metadata (K/8 bytes per row); dY as (M, N) with M inner.
  CUtensorMap tmV, tmE, tmB;
  const uint64_t kc = a.K / 2;
  // Values with the 128-byte swizzle: the expansion threads of one 8-lane
  // phase read the same 16-byte column of 8 consecutive rows, which the
  // swizzle spreads over all 32 banks.
  if (!encode_tensor_map_2d(&tmV, CU_TENSOR_MAP_DATA_TYPE_UINT16, a.values, kc, a.M, kc * 2, 64, Cfg::SM,
                            CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tensor_map_2d(&tmE, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.meta, a.K / 8, a.M, a.K / 8, 16, Cfg::SM,
                            CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !encode_tensor_map_2d(&tmB, CU_TENSOR_MAP_DATA_TYPE_UINT16, a.B, a.M, a.N, a.ldb * 2, 64, BN,
                            CU_TENSOR_MAP_SWIZZLE_128B))
    return ST24_ERR_CUDA;
  Params p{};
  p.M = a.K;   // rows of the output dX^T (the weight's K)
  p.N = a.N;
  p.alpha = a.alpha;
  p.beta = a.beta;
  p.C = a.C;
  p.ldc = a.ldc;
  p.c_type = a.c;
  p.row_scale = nullptr;
  p.Mw = a.M;
  p.tiles_k = a.K / Cfg::BM;
  p.tiles_n = (a.N + BN - 1) / BN;
  p.m_iters = (a.M + Cfg::SM - 1) / Cfg::SM;
  p.status = dev.status;
  const int64_t tiles = p.tiles_k * p.tiles_n;
  auto kern = spmm_t_kernel<DT, BN, STAGES>;
  static bool attr_set[64] = {};
  if (!attr_set[dev.device % 64]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES) != cudaSuccess)
      return ST24_ERR_CUDA;
    attr_set[dev.device % 64] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(tiles < dev.num_sms ? tiles : dev.num_sms));
  cfg.blockDim = dim3(Cfg::THREADS);
  cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tmV, tmE, tmB, p) == cudaSuccess ? ST24_OK : ST24_ERR_CUDA;
}

// The CTA-pair form: 256 output rows (k) per tile, half of dY's tile rows
// staged by each CTA of the cluster.
template <int DT, int BN, int STAGES, int VES>
st24_status launch_pair(const SpmmArgs& a, const DeviceInfo& dev, cudaStream_t stream) {
  using Cfg = spt2::Config<DT, BN, STAGES, VES>;
  CUtensorMap tmV, tmE, tmB;
  const uint64_t kc = a.K / 2;
  // Values with the 128-byte swizzle: the expansion threads of one 8-lane
  // phase read the same 16-byte column of 8 consecutive rows, which the
  // swizzle spreads over all 32 banks.
  if (!encode_tensor_map_2d(&tmV, CU_TENSOR_MAP_DATA_TYPE_UINT16, a.values, kc, a.M, kc * 2, 64, Cfg::SM,
                            CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tensor_map_2d(&tmE, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.meta, a.K / 8, a.M, a.K / 8, 16, Cfg::SM,
                            CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !encode_tensor_map_2d(&tmB, CU_TENSOR_MAP_DATA_TYPE_UINT16, a.B, a.M, a.N, a.ldb * 2, 64, Cfg::BH,
                            CU_TENSOR_MAP_SWIZZLE_128B))
    return ST24_ERR_CUDA;
  Params p{};
  p.M = a.K;   // rows of the output dX^T (the weight's K)
  p.N = a.N;
  p.alpha = a.alpha;
  p.beta = a.beta;
  p.C = a.C;
  p.ldc = a.ldc;
  p.c_type = a.c;
  p.row_scale = nullptr;
  p.Mw = a.M;
  p.tiles_k = a.K / 256;
  p.tiles_n = (a.N + BN - 1) / BN;
  p.m_iters = (a.M + Cfg::SM - 1) / Cfg::SM;
  p.status = dev.status;
  const int64_t tiles = p.tiles_k * p.tiles_n, pairs = dev.num_sms / 2;
  auto kern = spt2::spmm_t2_kernel<DT, BN, STAGES, VES>;
  static bool attr_set[64] = {};
  if (!attr_set[dev.device % 64]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES) != cudaSuccess)
      return ST24_ERR_CUDA;
    attr_set[dev.device % 64] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(2 * (tiles < pairs ? tiles : pairs)));
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
  return cudaLaunchKernelEx(&cfg, kern, tmV, tmE, tmB, p) == cudaSuccess ? ST24_OK : ST24_ERR_CUDA;
}

// Output tile width for N: 64 / 128 / 256 columns (with the deepest ring that
// fits); CTA pairs when K fills whole 256-row pair tiles.
template <int DT>
st24_status launch_dt_impl(const SpmmArgs& a, const DeviceInfo& dev, cudaStream_t s) {
  if (a.K % 256 == 0) {
    if (a.N <= 64) return launch_pair<DT, 64, 6, 10>(a, dev, s);
    if (a.N <= 128) return launch_pair<DT, 128, 5, 10>(a, dev, s);
    return launch_pair<DT, 256, 4, 10>(a, dev, s);
  }
  if (a.N <= 64) return launch_cfg<DT, 64, 6>(a, dev, s);
  if (a.N <= 128) return launch_cfg<DT, 128, 5>(a, dev, s);
  return launch_cfg<DT, 256, 3>(a, dev, s);
}

}  // namespace spt
}  // namespace st24
