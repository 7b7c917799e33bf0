// peak_mma_sp.cu -- issue-rate ceiling of the warp-level sparse tensor-core
// instruction (mma.sp::ordered_metadata) on this GPU, for the roofline of the
// kernels built on it.  int8 products run on that instruction (the 5th
// generation tensor-core MMA of this architecture has no 8-bit integer kind),
// so its measured rate, not a datasheet figure, is their tensor peak.
//
// Each warp keeps 8 independent accumulators and issues back-to-back MMAs on
// register operands only: no memory traffic, so the rate is the tensor pipe's.
// Reported as dense-equivalent operations (2 * 16 * 8 * logical K per MMA),
// the unit every throughput figure of this library uses.
#include <cstdint>
#include <cuda_runtime.h>

namespace {

constexpr int kChains = 8;

template <int KIND>   // 0: s8 m16n8k64, 1: bf16 m16n8k32
__global__ void __launch_bounds__(128) mma_sp_loop(int iters, int* sink) {
  uint32_t a[4], b[4];
  for (int i = 0; i < 4; ++i) {
    a[i] = 0x01010101u * (threadIdx.x + i);
    b[i] = 0x00010001u * (i + 1);
  }
  const uint32_t e = 0x44444444u;   // every group: indices (0, 1)
  int ai[kChains][4] = {};
  float af[kChains][4] = {};
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int c = 0; c < kChains; ++c) {
      if constexpr (KIND == 0) {
        asm volatile(
            "mma.sp::ordered_metadata.sync.aligned.m16n8k64.row.col.s32.s8.s8.s32 "
            "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9,%10,%11}, {%0,%1,%2,%3}, %12, 0x0;"
            : "+r"(ai[c][0]), "+r"(ai[c][1]), "+r"(ai[c][2]), "+r"(ai[c][3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]), "r"(b[2]), "r"(b[3]), "r"(e));
      } else {
        asm volatile(
            "mma.sp::ordered_metadata.sync.aligned.m16n8k32.row.col.f32.bf16.bf16.f32 "
            "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9,%10,%11}, {%0,%1,%2,%3}, %12, 0x0;"
            : "+f"(af[c][0]), "+f"(af[c][1]), "+f"(af[c][2]), "+f"(af[c][3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]), "r"(b[2]), "r"(b[3]), "r"(e));
      }
    }
  }
  int s = 0;
  for (int c = 0; c < kChains; ++c)
    for (int r = 0; r < 4; ++r) s += ai[c][r] + static_cast<int>(af[c][r]);
  if (s == 0x7fffffff) sink[0] = s;   // keeps the loop alive; practically never taken
}

}  // namespace

// kind 0: int8 (m16n8k64), kind 1: bf16 (m16n8k32).  Writes the best of three
// timed runs, in dense-equivalent TOPS, to *tops.  Returns 0, or a CUDA error
// code.  Runs on the current device and stream 0, and synchronises it.
extern "C" __attribute__((visibility("default"))) int st24peak_mma_sp(int kind, double* tops) {
  if (kind != 0 && kind != 1) return -1;
  int dev = 0, sms = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err == cudaSuccess) err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int* sink = nullptr;
  if (err == cudaSuccess) err = cudaMalloc(&sink, sizeof(int));
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  if (err == cudaSuccess) err = cudaEventCreate(&e0);
  if (err == cudaSuccess) err = cudaEventCreate(&e1);
  const int blocks = 4 * sms, threads = 128, iters = kind == 0 ? 2048 : 8192;
  float best = 0.f;
  for (int rep = 0; rep < 4 && err == cudaSuccess; ++rep) {
    cudaEventRecord(e0);
    if (kind == 0)
      mma_sp_loop<0><<<blocks, threads>>>(iters, sink);
    else
      mma_sp_loop<1><<<blocks, threads>>>(iters, sink);
    cudaEventRecord(e1);
    err = cudaEventSynchronize(e1);
    float ms = 0.f;
    if (err == cudaSuccess) err = cudaEventElapsedTime(&ms, e0, e1);
    if (err == cudaSuccess && rep > 0 && (best == 0.f || ms < best)) best = ms;
  }
  if (err == cudaSuccess) {
    const double mmas = double(blocks) * (threads / 32) * iters * kChains;
    const double k = kind == 0 ? 64.0 : 32.0;
    *tops = mmas * 2.0 * 16 * 8 * k / (best * 1e-3) / 1e12;
  }
  if (e0) cudaEventDestroy(e0);
  if (e1) cudaEventDestroy(e1);
  if (sink) cudaFree(sink);
  return err == cudaSuccess ? 0 : static_cast<int>(err);
}
