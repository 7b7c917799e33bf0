// st24_api.cu -- the C ABI (include/st24.h): argument checks, per-device state,
// schedule choice and kernel launch.  Every argument error is caught here, on
// the host, before any CUDA call is made.
#include <mutex>

#include "st24_device.cuh"

namespace st24 {

namespace {

// The status word kernels write when a bounded wait runs out.  One per device
// that loads the library; its address is looked up per device.
__device__ unsigned g_status_word;

constexpr int kMaxDevices = 64;
DeviceInfo g_info[kMaxDevices];
std::once_flag g_once[kMaxDevices];

bool is_ab_type(int t) { return t == kF16 || t == kBF16 || t == kE4M3 || t == kS8; }

bool aligned(const void* p, int a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<EncodeTiledFn>(nullptr);
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

}  // namespace

const DeviceInfo* current_device_info() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::call_once(g_once[dev], [dev] {
    DeviceInfo info;
    int sms = 0;
    void* word = nullptr;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return;
    if (cudaGetSymbolAddress(&word, g_status_word) != cudaSuccess) return;
    info.device = dev;
    info.num_sms = sms;
    info.status = static_cast<unsigned*>(word);
    g_info[dev] = info;
  });
  return g_info[dev].device == dev ? &g_info[dev] : nullptr;
}

bool encode_tensor_map_2d(CUtensorMap* map, CUtensorMapDataType type, const void* base,
                          uint64_t inner, uint64_t outer, uint64_t row_stride_bytes,
                          uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_stride_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, type, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_tensor_map_3d(CUtensorMap* map, CUtensorMapDataType type, const void* base, const uint64_t dims[3],
                          const uint64_t strides_bytes[2], const uint32_t box[3], CUtensorMapSwizzle swizzle) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t d[3] = {dims[0], dims[1], dims[2]};
  const cuuint64_t st[2] = {strides_bytes[0], strides_bytes[1]};
  const cuuint32_t b[3] = {box[0], box[1], box[2]};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, type, 3, const_cast<void*>(base), d, st, b, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

StreamKPlan make_stream_k_plan(int bm, int bn, int bk, int64_t M, int64_t N, int64_t K, int num_sms,
                               double a_row_bytes, double b_col_bytes, bool allow_cluster) {
  StreamKPlan pl{};
  pl.bm = bm;
  pl.bn = bn;
  pl.bk = bk;
  pl.tiles_m = (M + bm - 1) / bm;
  pl.tiles_n = (N + bn - 1) / bn;
  pl.k_iters = (K + bk - 1) / bk;
  const int64_t tiles = pl.tiles_m * pl.tiles_n;
  const int64_t total_iters = tiles * pl.k_iters;
  // Fewer tiles than SMs: split every tile over the same number of CTAs
  // (tiles * floor(SMs / tiles)) so each CTA streams an equal, whole-k-block
  // share and every split tile has the same few contributors.
  int64_t grid = num_sms;
  if (tiles > 0 && tiles < num_sms) grid = tiles * (num_sms / tiles);
  if (grid > total_iters) grid = total_iters;
  pl.grid = static_cast<int>(grid > 0 ? grid : 1);
  // Whole waves of tiles run data-parallel; the remainder plus one wave (so
  // that each of its tiles is split over only one or two CTAs) runs stream-K.
  // With many waves and a nearly full last one, whole tiles throughout:
  // a stream-K tail costs each split tile a partial-tile round trip through
  // the workspace, more than the last wave's idle share (measured on
  // 11008x4096, N = 4096: 10.75 waves of CTA pairs).
  if (tiles <= pl.grid) {
    pl.sk_tiles = tiles;
  } else {
    const int64_t rem = tiles % pl.grid;
    const int64_t waves = (tiles + pl.grid - 1) / pl.grid;
    const bool tail_cheap = rem == 0 || (pl.grid - rem) * 100 <= 3 * waves * pl.grid;   // idle share <= 3%
    pl.sk_tiles = tail_cheap ? 0 : rem + pl.grid;
  }
  pl.dp_tiles = tiles - pl.sk_tiles;
  // Raster.  Consecutive tiles run at the same time; keep one operand's panel
  // in L2 and stream the other once.  If all of B fits in the budget, go
  // row by row (m-tile outer): B stays resident, A is read once.  Otherwise
  // group as many m-tiles as fit (their A panel stays resident) and sweep the
  // n-tiles inside each group, so B is read once per group.
  const double kResident = 56.0 * (1 << 20);
  if (b_col_bytes * static_cast<double>(N) <= kResident) {
    pl.group_m = 1;
  } else {
    const double per_mtile = a_row_bytes * bm;
    int64_t g = static_cast<int64_t>(kResident / (per_mtile > 1.0 ? per_mtile : 1.0));
    pl.group_m = g < 1 ? 1 : (g > pl.tiles_m ? pl.tiles_m : g);
  }
  pl.partial_bytes = static_cast<size_t>(bm) * bn * 4;
  // Every tile split over the same s = grid / tiles CTAs (2 <= s <= 8, whole
  // k-blocks each): those CTAs can form one cluster and sum in shared memory.
  pl.cluster = 1;
  if (allow_cluster && pl.dp_tiles == 0 && tiles > 0 && pl.grid % tiles == 0) {
    const int64_t sp = pl.grid / tiles;
    if (sp >= 2 && sp <= 8 && pl.k_iters >= sp) pl.cluster = static_cast<int>(sp);
  }
  if (pl.cluster > 1) {
    pl.ws_bytes = 0;
    return pl;
  }
  // Is any stream-K tile split between CTAs?  (CTA c starts at c*I/G.)
  const int64_t sk_iters = pl.sk_tiles * pl.k_iters;
  bool split = false;
  for (int64_t c = 1; c < pl.grid && !split && sk_iters > 0; ++c)
    if ((c * sk_iters / pl.grid) % pl.k_iters != 0) split = true;
  pl.ws_bytes = split ? 2 * static_cast<size_t>(pl.grid) * pl.partial_bytes +
                            (static_cast<size_t>(tiles) * 4 + 255) / 256 * 256
                      : 0;
  return pl;
}

}  // namespace st24

using namespace st24;

namespace {

// Which kernel family st24_spmm uses (measured on GB300):
//  * int8: the warp-level kernels (there is no int8 tcgen05 kind on sm_103a):
//    the TMA-ring one (the register-direct one measured slower on the int8
//    workload's shapes).
//  * narrow products (N <= 64; for e4m3 with K a multiple of 256), bound by
//    streaming the compressed weights: the narrow tcgen05 kernel -- except
//    16-bit inputs with N <= 4 whose grid fits in one wave, where the
//    register-direct kernel's shorter chain wins by a little.  Left over:
//    the TMA-ring kernel (e4m3 with other K: tcgen05; the warp-level e4m3
//    sparse MMA runs at ~1/50 of the 16-bit rate).
//  * wider products: tcgen05 (CTA pairs for N > 64).
int resolve_kernel(int requested, const SpmmArgs& a, int num_sms) {
  if (requested != ST24_KERNEL_AUTO) return requested;
  if (a.ab == kS8) return ST24_KERNEL_MMA_SP;
  if (a.N > 64) return ST24_KERNEL_TCGEN05;
  const bool k16 = a.ab == kF16 || a.ab == kBF16;
  if (k16 && a.N <= 4 && direct_applies(a) && direct_one_wave(a, num_sms)) return ST24_KERNEL_MMA_SP_DIRECT;
  if (narrow_applies(a)) return ST24_KERNEL_TCGEN05_NARROW;
  return k16 ? ST24_KERNEL_MMA_SP : ST24_KERNEL_TCGEN05;
}

StreamKPlan plan_for(int kernel, const SpmmArgs& a, int num_sms) {
  if (kernel == ST24_KERNEL_MMA_SP_DIRECT) return StreamKPlan{};   // one launch shape, no workspace
  if (kernel == ST24_KERNEL_TCGEN05_NARROW) return plan_spmm_nt(a, num_sms);
  return kernel == ST24_KERNEL_TCGEN05 ? plan_spmm_tc(a, num_sms) : plan_spmm_mmasp(a, num_sms);
}

}  // namespace

StreamKPlan st24::plan_auto(const SpmmArgs& a, int num_sms) {
  return plan_for(resolve_kernel(ST24_KERNEL_AUTO, a, num_sms), a, num_sms);
}

st24_status st24::check_spmm_args(const SpmmArgs& a) {
  if (!is_ab_type(a.ab) || a.M < 0 || a.N < 0 || a.K < 0 || a.K % 4 != 0)
    return ST24_ERR_INVALID_ARG;
  const bool float_out = a.c == kF32 || a.c == kBF16 || a.c == kF16;
  if (!float_out && !(a.c == kS32 && a.ab == kS8)) return ST24_ERR_UNSUPPORTED;
  if (a.c == kS32 && (a.alpha != 1.0f || a.beta != 0.0f || a.row_scale))
    return ST24_ERR_UNSUPPORTED;
  if (a.M == 0 || a.N == 0) return ST24_OK;
  if (!a.C || a.ldc < a.M) return ST24_ERR_INVALID_ARG;
  if (a.K > 0 && (!a.values || !a.meta || !a.B || a.ldb < a.K)) return ST24_ERR_INVALID_ARG;
  if (a.K % 128 != 0) return ST24_ERR_UNSUPPORTED;
  const int es = elem_size(a.ab);
  if (a.K > 0 && (!aligned(a.values, 16) || !aligned(a.meta, 16) || !aligned(a.B, 16) ||
                  (a.ldb * es) % 16 != 0))
    return ST24_ERR_MISALIGNED;
  if (!aligned(a.C, elem_size(a.c)) || (a.row_scale && !aligned(a.row_scale, 4)))
    return ST24_ERR_MISALIGNED;
  return ST24_OK;
}

extern "C" {

int st24_version(void) { return (0 << 16) | (1 << 8) | 0; }

const char* st24_status_string(int status) {
  switch (status) {
    case ST24_OK: return "ok";
    case ST24_ERR_INVALID_ARG: return "invalid argument";
    case ST24_ERR_UNSUPPORTED: return "unsupported (type pair or shape)";
    case ST24_ERR_MISALIGNED: return "misaligned pointer or stride";
    case ST24_ERR_CUDA: return "CUDA error";
    case ST24_ERR_TIMEOUT: return "a kernel wait timed out";
    case ST24_ERR_WORKSPACE: return "workspace too small";
    default: return "unknown status";
  }
}

size_t st24_values_bytes(st24_dtype type, int64_t M, int64_t K) {
  if (!is_ab_type(type) || M < 0 || K < 0 || K % 4 != 0) return 0;
  return static_cast<size_t>(M) * static_cast<size_t>(K / 2) * elem_size(type);
}

size_t st24_meta_bytes(int64_t M, int64_t K) {
  if (M < 0 || K < 0 || K % 4 != 0) return 0;
  return static_cast<size_t>(M) * static_cast<size_t>(meta_row_bytes(K));
}

st24_status st24_prune_compress(st24_dtype type, const void* W, int64_t M, int64_t K, int64_t ldw,
                                void* values, void* meta, void* stream) {
  if (!is_ab_type(type) || M < 0 || K < 0 || K % 4 != 0) return ST24_ERR_INVALID_ARG;
  if (M == 0 || K == 0) return ST24_OK;
  if (!W || !values || !meta || ldw < K) return ST24_ERR_INVALID_ARG;
  return launch_prune_compress(type, W, M, K, ldw, values, meta, static_cast<cudaStream_t>(stream));
}

st24_status st24_prune_compress_nm(st24_dtype type, int n, int m, const void* W, int64_t M, int64_t K, int64_t ldw,
                                   void* values, void* meta, void* stream) {
  if (!is_ab_type(type) || M < 0 || K < 0 || K % 4 != 0) return ST24_ERR_INVALID_ARG;
  if ((m != 4 && m != 8) || n < 1 || n > 2) return ST24_ERR_UNSUPPORTED;
  if (K % m != 0) return ST24_ERR_INVALID_ARG;
  if (M == 0 || K == 0) return ST24_OK;
  if (!W || !values || !meta || ldw < K) return ST24_ERR_INVALID_ARG;
  const int es = elem_size(type);
  if (!aligned(W, es) || !aligned(values, 2 * es)) return ST24_ERR_MISALIGNED;
  return launch_prune_compress_nm(type, n, m, false, W, M, K, ldw, values, meta, static_cast<cudaStream_t>(stream));
}

st24_status st24_prune_compress_nm2(st24_dtype type, int n, int m, const void* W, int64_t M, int64_t K, int64_t ldw,
                                    void* values, void* meta, void* stream) {
  if (!is_ab_type(type) || M < 0 || K < 0 || K % 4 != 0) return ST24_ERR_INVALID_ARG;
  if ((m != 4 && m != 8) || n < 1 || n > 4 || n > m) return ST24_ERR_UNSUPPORTED;
  if (K % m != 0) return ST24_ERR_INVALID_ARG;
  if (M == 0 || K == 0) return ST24_OK;
  if (!W || !values || !meta || ldw < K) return ST24_ERR_INVALID_ARG;
  const int es = elem_size(type);
  if (!aligned(W, es) || !aligned(values, 2 * es)) return ST24_ERR_MISALIGNED;
  return launch_prune_compress_nm(type, n, m, true, W, M, K, ldw, values, meta, static_cast<cudaStream_t>(stream));
}

st24_status st24_quantize_prune_compress(st24_dtype src_type, st24_dtype dst_type, const void* W, int64_t M,
                                         int64_t K, int64_t ldw, void* values, void* meta, float* scales,
                                         void* stream) {
  if (M < 0 || K < 0 || K % 4 != 0) return ST24_ERR_INVALID_ARG;
  if ((src_type != ST24_F16 && src_type != ST24_BF16) || (dst_type != ST24_E4M3 && dst_type != ST24_S8))
    return ST24_ERR_UNSUPPORTED;
  if (M == 0) return ST24_OK;
  if (!scales || (K > 0 && (!W || !values || !meta || ldw < K))) return ST24_ERR_INVALID_ARG;
  if (K % 16 != 0) return ST24_ERR_UNSUPPORTED;
  if ((K > 0 && (!aligned(W, 16) || (ldw * 2) % 16 != 0 || !aligned(values, 8) || !aligned(meta, 2))) ||
      !aligned(scales, 4))
    return ST24_ERR_MISALIGNED;
  return launch_quantize_prune_compress(src_type, dst_type, W, M, K, ldw, values, meta, scales,
                                        static_cast<cudaStream_t>(stream));
}

st24_status st24_decompress(st24_dtype type, const void* values, const void* meta, int64_t M,
                            int64_t K, void* W, int64_t ldw, void* stream) {
  if (!is_ab_type(type) || M < 0 || K < 0 || K % 4 != 0) return ST24_ERR_INVALID_ARG;
  if (M == 0 || K == 0) return ST24_OK;
  if (!W || !values || !meta || ldw < K) return ST24_ERR_INVALID_ARG;
  return launch_decompress(type, values, meta, M, K, W, ldw, static_cast<cudaStream_t>(stream));
}


size_t st24_spmm_workspace_bytes(st24_dtype ab_type, st24_dtype c_type, int64_t M, int64_t N,
                                 int64_t K) {
  if (!is_ab_type(ab_type) || M <= 0 || N <= 0 || K <= 0 || K % 128 != 0) return 0;
  const DeviceInfo* dev = current_device_info();
  if (!dev) return 0;
  SpmmArgs a{};
  a.ab = ab_type;
  a.c = c_type;
  a.M = M;
  a.N = N;
  a.K = K;
  // Enough for whichever kernel family a call with these sizes may run on.
  size_t ws = plan_spmm_mmasp(a, dev->num_sms).ws_bytes;
  if (ab_type != ST24_S8) {
    const size_t t = plan_spmm_tc(a, dev->num_sms).ws_bytes;
    ws = t > ws ? t : ws;
    if (narrow_applies(a)) {
      const size_t n = plan_spmm_nt(a, dev->num_sms).ws_bytes;
      ws = n > ws ? n : ws;
    }
  }
  return ws;
}

st24_status st24_spmm_ex(st24_kernel kernel, unsigned flags, st24_dtype ab_type, st24_dtype c_type, int64_t M,
                         int64_t N, int64_t K, float alpha, const void* A_values, const void* A_meta, const void* B,
                         int64_t ldb, float beta, void* C, int64_t ldc, const float* row_scale,
                         void* workspace, size_t ws_bytes, void* stream) {
  if (kernel != ST24_KERNEL_AUTO && kernel != ST24_KERNEL_TCGEN05 && kernel != ST24_KERNEL_MMA_SP &&
      kernel != ST24_KERNEL_MMA_SP_DIRECT && kernel != ST24_KERNEL_TCGEN05_NARROW)
    return ST24_ERR_INVALID_ARG;
  if (flags & ~static_cast<unsigned>(ST24_SPMM_FIXED_A | ST24_SPMM_TWO_FORMS)) return ST24_ERR_INVALID_ARG;
  const bool two = (flags & ST24_SPMM_TWO_FORMS) != 0;
  SpmmArgs a{};
  a.flags = flags;
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
  a.workspace = workspace;
  a.ws_bytes = ws_bytes;
  a.Kb = K;
  st24_status st = check_spmm_args(a);   // B and C as for K
  if (st != ST24_OK || M == 0 || N == 0) return st;
  if (two) {
    // A holds two 2:4 forms of M x K side by side: the M x 2K matrix [form 0 | form 1],
    // multiplied by B once per form (B's k-coordinate wraps at K).
    if (K % 256 != 0) return ST24_ERR_UNSUPPORTED;
    if (kernel == ST24_KERNEL_MMA_SP_DIRECT) return ST24_ERR_UNSUPPORTED;
    a.K = 2 * K;
  }
  if (kernel == ST24_KERNEL_TCGEN05 && ab_type == ST24_S8) return ST24_ERR_UNSUPPORTED;
  if (kernel == ST24_KERNEL_MMA_SP_DIRECT && !direct_applies(a)) return ST24_ERR_UNSUPPORTED;
  if (kernel == ST24_KERNEL_TCGEN05_NARROW && !narrow_applies(a)) return ST24_ERR_UNSUPPORTED;
  const DeviceInfo* dev = current_device_info();
  if (!dev) return ST24_ERR_CUDA;
  int k = resolve_kernel(kernel, a, dev->num_sms);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (K == 0) return launch_scale_c(a, *dev, s);
  if (two) {
    // every k-block must lie in one form: the plan's k-block must divide K
    if (k == ST24_KERNEL_MMA_SP_DIRECT) k = ST24_KERNEL_TCGEN05_NARROW;
    if (plan_for(k, a, dev->num_sms).bk <= 0 || K % plan_for(k, a, dev->num_sms).bk != 0) {
      if (kernel != ST24_KERNEL_AUTO) return ST24_ERR_UNSUPPORTED;
      k = ab_type == ST24_S8 || ab_type == ST24_F16 || ab_type == ST24_BF16 ? ST24_KERNEL_MMA_SP : ST24_KERNEL_TCGEN05;
    }
  }
  if (k == ST24_KERNEL_MMA_SP_DIRECT) return launch_spmm_direct(a, *dev, s);
  const StreamKPlan plan = plan_for(k, a, dev->num_sms);
  if (plan.ws_bytes > 0 && (!workspace || ws_bytes < plan.ws_bytes || !aligned(workspace, 16)))
    return ST24_ERR_WORKSPACE;
  if (k == ST24_KERNEL_TCGEN05_NARROW) return launch_spmm_nt(a, plan, *dev, s);
  return k == ST24_KERNEL_TCGEN05 ? launch_spmm_tc(a, plan, *dev, s) : launch_spmm_mmasp(a, plan, *dev, s);
}

st24_status st24_spmm(st24_dtype ab_type, st24_dtype c_type, int64_t M, int64_t N, int64_t K,
                      float alpha, const void* A_values, const void* A_meta, const void* B,
                      int64_t ldb, float beta, void* C, int64_t ldc, const float* row_scale,
                      void* workspace, size_t ws_bytes, void* stream) {
  return st24_spmm_ex(ST24_KERNEL_AUTO, 0u, ab_type, c_type, M, N, K, alpha, A_values, A_meta, B, ldb, beta, C, ldc,
                      row_scale, workspace, ws_bytes, stream);
}

st24_status st24_device_status(void* stream) {
  const DeviceInfo* dev = current_device_info();
  if (!dev) return ST24_ERR_CUDA;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return ST24_ERR_CUDA;
  unsigned word = 0;
  if (cudaMemcpy(&word, dev->status, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess)
    return ST24_ERR_CUDA;
  if (word == 0) return ST24_OK;
  if (cudaMemset(dev->status, 0, sizeof word) != cudaSuccess) return ST24_ERR_CUDA;
  return (word & kStatusTimeout) ? ST24_ERR_TIMEOUT : ST24_ERR_CUDA;
}

}  // extern "C"
