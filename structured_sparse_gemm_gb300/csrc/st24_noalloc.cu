// st24_noalloc.cu -- st24_spmm for callers that cannot allocate device memory.
//
// The split-K / stream-K schedule of st24_spmm keeps partial tiles and one
// counter per output tile in a workspace the caller allocates.  Some callers
// cannot allocate: a plugin inside a serving runtime whose device memory is
// owned by the runtime's own pool, code running while a stream is captured
// in the global capture mode (where cudaMalloc is not a permitted call), or a
// latency-critical path that must not take the allocator's lock or
// synchronise the device.  st24_spmm_noalloc runs the same kernels with that
// scratch in a fixed-size array in device global memory that this library
// owns: kScratchBytes, created with the library's module on every GPU that
// loads it and held until the process exits.  It calls no cudaMalloc, no
// cudaFree and no allocating library routine.
#include <mutex>

#include "st24_device.cuh"

namespace st24 {
namespace {

// 16 MiB: enough for every product with N <= 64 on GPUs of up to 160 SMs
// (two fp32 partial tiles of 128 x 64 per CTA plus the tile counters).
constexpr size_t kScratchBytes = size_t(16) << 20;

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices];
std::once_flag g_scratch_once[kMaxDevices];

// Device address of the current device's scratch array, looked up once per
// device with that device current; nullptr if the lookup failed.
void* scratch_of_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::call_once(g_scratch_once[dev], [dev] {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_scratch) == cudaSuccess) g_scratch_addr[dev] = ptr;
  });
  return g_scratch_addr[dev];
}

}  // namespace
}  // namespace st24

using namespace st24;

extern "C" st24_status st24_spmm_noalloc(st24_dtype ab_type, st24_dtype c_type, int64_t M, int64_t N,
                                         int64_t K, float alpha, const void* A_values, const void* A_meta,
                                         const void* B, int64_t ldb, float beta, void* C, int64_t ldc,
                                         const float* row_scale, void* stream) {
  SpmmArgs a{};
  a.ab = ab_type;
  a.c = c_type;
  a.M = M;
  a.N = N;
  a.K = K;
  a.alpha = alpha;
  a.beta = beta;
  a.values = A_values;
  a.meta = A_meta;
  a.B = B;
  a.ldb = ldb;
  a.C = C;
  a.ldc = ldc;
  a.row_scale = row_scale;
  // Argument errors are reported before anything is enqueued.
  const st24_status st = check_spmm_args(a);
  if (st != ST24_OK) return st;
  size_t need = 0;
  size_t counters_at = 0;
  if (M > 0 && N > 0 && K > 0) {
    const DeviceInfo* dev = current_device_info();
    if (!dev) return ST24_ERR_CUDA;
    const StreamKPlan plan = plan_auto(a, dev->num_sms);   // the plan st24_spmm will use
    need = plan.ws_bytes;
    counters_at = 2 * static_cast<size_t>(plan.grid) * plan.partial_bytes;
  }
  if (need > kScratchBytes) return ST24_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (need > 0) {
    scratch = scratch_of_current_device();
    if (!scratch) return ST24_ERR_CUDA;
    // The array keeps the previous call's contents: the tile counters must
    // start at zero (the partial tiles are always written before being read).
    if (cudaMemsetAsync(static_cast<unsigned char*>(scratch) + counters_at, 0, need - counters_at,
                        static_cast<cudaStream_t>(stream)) != cudaSuccess)
      return ST24_ERR_CUDA;
  }
  return st24_spmm(ab_type, c_type, M, N, K, alpha, A_values, A_meta, B, ldb, beta, C, ldc, row_scale, scratch,
                   need > 0 ? kScratchBytes : 0, stream);
}
