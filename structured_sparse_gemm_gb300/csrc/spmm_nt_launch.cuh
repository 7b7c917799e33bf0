// spmm_nt_launch.cuh -- host launch of the narrow-N tcgen05 SpMM for one
// element type (included by the per-type translation units).
#pragma once

#include "spmm_nt.cuh"

namespace st24 {
namespace nt {

template <int DT, int BN, int C, int STAGES, bool SPLIT>
st24_status launch_cfg(const SpmmArgs& a, const StreamKPlan& plan, const DeviceInfo& dev, cudaStream_t stream) {
  using Cfg = Config<DT, BN, C, STAGES, SPLIT>;
  using T = Traits<DT>;
  const CUtensorMapDataType ty = T::ES == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  // Values as (128-byte chunk of a row, row, chunk index): a stage's C chunks
  // of 128 rows in one copy, chunk-major ([chunk][row][128 B]).
  const uint64_t vrow = static_cast<uint64_t>(a.K / 2) * T::ES;   // bytes per row of values
  const uint64_t adims[3] = {static_cast<uint64_t>(T::CHUNK_ELEMS), static_cast<uint64_t>(a.M), vrow / 128};
  const uint64_t astr[2] = {vrow, 128};
  const uint32_t abox[3] = {static_cast<uint32_t>(T::CHUNK_ELEMS), static_cast<uint32_t>(Cfg::BM),
                            static_cast<uint32_t>(C)};
  // B likewise: (128-byte chunk of a column of B, column n, chunk index), 2C chunks per stage.
  const uint64_t bdims[3] = {static_cast<uint64_t>(T::CHUNK_ELEMS), static_cast<uint64_t>(a.N),
                             static_cast<uint64_t>(a.Kb ? a.Kb : a.K) * T::ES / 128};
  const uint64_t bstr[2] = {static_cast<uint64_t>(a.ldb) * T::ES, 128};
  const uint32_t bbox[3] = {static_cast<uint32_t>(T::CHUNK_ELEMS), static_cast<uint32_t>(BN),
                            static_cast<uint32_t>(2 * C)};
  CUtensorMap tmA, tmE, tmB;
  if (!encode_tensor_map_3d(&tmA, ty, a.values, adims, astr, abox, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tensor_map_2d(&tmE, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.meta, a.K / 8, a.M, a.K / 8, Cfg::EB, Cfg::BM,
                            CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !encode_tensor_map_3d(&tmB, ty, a.B, bdims, bstr, bbox, CU_TENSOR_MAP_SWIZZLE_128B))
    return ST24_ERR_CUDA;
  Params p{};
  p.M = a.M; p.N = a.N; p.K = a.K;
  p.alpha = a.alpha; p.beta = a.beta;
  p.C = a.C; p.ldc = a.ldc; p.c_type = a.c;
  p.row_scale = a.row_scale;
  p.k_iters = plan.k_iters;
  p.parts = plan.cluster;
  p.kb_wrap = (a.Kb && a.Kb != a.K) ? a.Kb / plan.bk : 0;
  p.a_fixed = (a.flags & ST24_SPMM_FIXED_A) ? 1 : 0;
  p.status = dev.status;
  auto kern = spmm_nt_kernel<DT, BN, C, STAGES, SPLIT>;
  static bool attr_set[64] = {};
  if (!attr_set[dev.device % 64]) {
    // Two CTAs per SM (this product's and the next one's) need the largest shared-memory carveout.
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES) != cudaSuccess ||
        cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100) != cudaSuccess)
      return ST24_ERR_CUDA;
    attr_set[dev.device % 64] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(plan.grid));
  cfg.blockDim = dim3(Cfg::THREADS);
  cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attrs[2];
  attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[0].val.programmaticStreamSerializationAllowed = 1;
  int nattr = 1;
  if (plan.cluster > 1) {
    attrs[1].id = cudaLaunchAttributeClusterDimension;
    attrs[1].val.clusterDim.x = static_cast<unsigned>(plan.cluster);
    attrs[1].val.clusterDim.y = 1;
    attrs[1].val.clusterDim.z = 1;
    nattr = 2;
  }
  cfg.attrs = attrs;
  cfg.numAttrs = nattr;
  return cudaLaunchKernelEx(&cfg, kern, tmA, tmE, tmB, p) == cudaSuccess ? ST24_OK : ST24_ERR_CUDA;
}

// Tile width -> chunks per stage and ring depth.  Unsplit tiles (large
// products): two 128-byte chunks per stage where two stages fit in half an
// SM (fewer copies per byte for the single producer), else one chunk and
// three stages.  Split tiles: one chunk per stage (a finer-grained ring that
// refills from L2 sooner) and room for the partials the CTA receives.
template <int DT>
st24_status launch_dt_impl(const SpmmArgs& a, const StreamKPlan& plan, const DeviceInfo& dev, cudaStream_t s) {
  constexpr bool k16 = Traits<DT>::ES == 2;
  if (plan.cluster > 1) {
    switch (plan.bn) {
      case 16: return launch_cfg<DT, 16, 1, 4, true>(a, plan, dev, s);
      case 32: return launch_cfg<DT, 32, 1, 3, true>(a, plan, dev, s);
      case 48: return launch_cfg<DT, 48, 1, 2, true>(a, plan, dev, s);
      default: return launch_cfg<DT, 64, 1, 2, true>(a, plan, dev, s);
    }
  }
  switch (plan.bn) {
    case 16: return launch_cfg<DT, 16, 2, 2, false>(a, plan, dev, s);
    case 32:
      if constexpr (k16) return launch_cfg<DT, 32, 2, 2, false>(a, plan, dev, s);
      else return launch_cfg<DT, 32, 1, 3, false>(a, plan, dev, s);
    case 48: return launch_cfg<DT, 48, 1, 3, false>(a, plan, dev, s);
    default: return launch_cfg<DT, 64, 1, 3, false>(a, plan, dev, s);
  }
}

// Logical K of one stage (the plan's k-block) for a tile width and split.
inline int stage_k(int es, int bn, bool split) {
  const int ck = es == 2 ? 128 : 256;
  const int c = split ? 1 : ((bn == 16 || (bn == 32 && es == 2)) ? 2 : 1);
  return c * ck;
}

}  // namespace nt
}  // namespace st24
