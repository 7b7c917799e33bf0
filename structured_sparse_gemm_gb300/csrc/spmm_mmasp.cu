// spmm_mmasp.cu -- schedule choice and dispatch of the warp-level sparse-MMA
// SpMM (the kernel template lives in spmm_mmasp.cuh; one translation unit per
// element type instantiates it).
#include "spmm_mmasp.cuh"

namespace st24 {
namespace mmasp {
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

// Narrow tiles (BN <= 32) fit two CTAs per SM: with no more tiles than SMs,
// split each tile over the CTAs of twice the SMs, at most 8 so every split
// tile still reduces inside one cluster (measured: int8 8192x8192, N = 16,
// 21.7 -> 15.7 us; bf16 11008x4096, N = 8, 15.5 -> 12.2 us).  More tiles
// keep the balanced stream-K schedule over one CTA per SM.
StreamKPlan plan_spmm_mmasp(const SpmmArgs& a, int num_sms) {
  int slots = num_sms;
  const int64_t tiles = (a.M + 127) / 128;
  if (pick_bn(a.N) <= 32 && tiles <= num_sms) {
    const int64_t cap = 8 * tiles > num_sms ? 8 * tiles : num_sms;
    slots = static_cast<int>(2 * static_cast<int64_t>(num_sms) < cap ? 2 * static_cast<int64_t>(num_sms) : cap);
  }
  return make_stream_k_plan(128, pick_bn(a.N), elem_size(a.ab) == 2 ? 128 : 256, a.M, a.N, a.K, slots,
                            a.K * (elem_size(a.ab) / 2.0 + 0.125), static_cast<double>(a.K) * elem_size(a.ab),
                            /*allow_cluster=*/pick_bn(a.N) <= 64);
}

st24_status launch_scale_c(const SpmmArgs& a, const DeviceInfo& dev, cudaStream_t stream) {
  OutParams p{};
  p.M = a.M; p.N = a.N; p.beta = a.beta; p.C = a.C; p.ldc = a.ldc; p.c_type = a.c;
  const int64_t want = (a.M * a.N + 255) / 256;
  const int grid = static_cast<int>(want < dev.num_sms * 8 ? want : dev.num_sms * 8);
  scale_c_kernel<<<grid, 256, 0, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? ST24_OK : ST24_ERR_CUDA;
}

st24_status launch_spmm_mmasp(const SpmmArgs& a, const StreamKPlan& plan, const DeviceInfo& dev,
                              cudaStream_t stream) {
  switch (a.ab) {
    case kF16: return launch_dt<kF16>(a, plan, dev, stream);
    case kBF16: return launch_dt<kBF16>(a, plan, dev, stream);
    case kE4M3: return launch_dt<kE4M3>(a, plan, dev, stream);
    case kS8: return launch_dt<kS8>(a, plan, dev, stream);
    default: return ST24_ERR_UNSUPPORTED;
  }
}

// C = beta * C (K == 0: the product is empty).
__global__ void scale_c_kernel(OutParams p) {
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

}  // namespace st24
