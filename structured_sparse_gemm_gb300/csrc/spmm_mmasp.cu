// spmm_mmasp.cu -- schedule choice and dispatch of the warp-level sparse-MMA
// SpMM (the kernel template lives in spmm_mmasp.cuh; one translation unit per
// element type instantiates it).
#include "spmm_mmasp.cuh"

namespace st24 {
namespace mmasp {
// C = beta * C (K == 0: the product is empty).
__global__ void scale_c_kernel(Params p) {
  const int64_t total = p.M * p.N;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < total;
       t += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t n = t / p.M, m = t - n * p.M;
    const int64_t idx = n * p.ldc + m;
    const float r = p.beta != 0.0f ? __fmul_rn(p.beta, load_c(p, idx)) : 0.0f;
    switch (p.c_type) {
      case kF32: static_cast<float*>(p.C)[idx] = r; break;
      case kBF16: static_cast<__nv_bfloat16*>(p.C)[idx] = __float2bfloat16_rn(r); break;
      case kF16: static_cast<__half*>(p.C)[idx] = __float2half_rn(r); break;
      default: static_cast<int*>(p.C)[idx] = 0; break;
    }
  }
}

// Tile width for a given N: the smallest of 8/16/32/64 that covers N, else 128.
int pick_bn(int64_t N) {
  if (N <= 8) return 8;
  if (N <= 16) return 16;
  if (N <= 32) return 32;
  if (N <= 64) return 64;
  return 128;
}

}  // namespace mmasp

using namespace mmasp;

StreamKPlan plan_spmm_mmasp(const SpmmArgs& a, int num_sms) {
  StreamKPlan pl{};
  const int es = elem_size(a.ab);
  pl.bm = 128;
  pl.bn = pick_bn(a.N);
  pl.bk = es == 2 ? 128 : 256;
  pl.tiles_m = (a.M + pl.bm - 1) / pl.bm;
  pl.tiles_n = (a.N + pl.bn - 1) / pl.bn;
  pl.k_iters = (a.K + pl.bk - 1) / pl.bk;
  pl.total_iters = pl.tiles_m * pl.tiles_n * pl.k_iters;
  const int64_t grid = pl.total_iters < num_sms ? pl.total_iters : num_sms;
  pl.grid = static_cast<int>(grid > 0 ? grid : 1);
  pl.partial_bytes = static_cast<size_t>(pl.bm) * pl.bn * 4;
  // Is any tile split between CTAs?
  bool split = false;
  for (int64_t c = 1; c < pl.grid && !split; ++c)
    if ((c * pl.total_iters / pl.grid) % pl.k_iters != 0) split = true;
  const size_t tiles = static_cast<size_t>(pl.tiles_m * pl.tiles_n);
  pl.ws_bytes = split ? 2 * static_cast<size_t>(pl.grid) * pl.partial_bytes + (tiles * 4 + 255) / 256 * 256 : 0;
  return pl;
}

st24_status launch_spmm_mmasp(const SpmmArgs& a, const StreamKPlan& plan, const DeviceInfo& dev,
                              cudaStream_t stream) {
  if (a.K == 0) {
    Params p{};
    p.M = a.M; p.N = a.N; p.beta = a.beta; p.C = a.C; p.ldc = a.ldc; p.c_type = a.c;
    const int64_t want = (a.M * a.N + 255) / 256;
    const int grid = static_cast<int>(want < dev.num_sms * 8 ? want : dev.num_sms * 8);
    scale_c_kernel<<<grid, 256, 0, stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? ST24_OK : ST24_ERR_CUDA;
  }
  switch (a.ab) {
    case kF16: return launch_dt<kF16>(a, plan, dev, stream);
    case kBF16: return launch_dt<kBF16>(a, plan, dev, stream);
    case kE4M3: return launch_dt<kE4M3>(a, plan, dev, stream);
    case kS8: return launch_dt<kS8>(a, plan, dev, stream);
    default: return ST24_ERR_UNSUPPORTED;
  }
}

}  // namespace st24
