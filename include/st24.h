/*
 * st24.h -- C ABI of a 2:4 structured-sparse GEMM library for GB300 (sm_103a).
 *
 * The library implements the data-parallel hot path of 2:4 structured
 * sparsity as described in:
 *   [CH26] "Chapter 26 -- Sparsity: The Hardware View" (sections "2:4
 *          Fine-Grained Structured Sparsity", "2:4 in the Memory-Bound Regime",
 *          "Sparsity + Quantization Combine", and "Python: Build a 2:4 Mask,
 *          Compress It, and Show Why Unstructured Doesn't Help");
 *   [SS24] "10.4g Structured Sparsity (2:4)" (sections "What is 2:4
 *          Structured Sparsity?" and "How Tensor Cores Leverage This Pattern").
 *
 * Conventions shared by every call:
 *  - All pointers named as device buffers must point to device memory (or
 *    memory the device can access) owned by the caller.  The library
 *    allocates no device memory per call and keeps no pointer after a call
 *    returns.
 *  - `stream` is a cudaStream_t passed as void*; NULL is the legacy default
 *    stream.  Work is enqueued asynchronously on it; a call returns once the
 *    work is enqueued.
 *  - Matrices use element strides (not bytes).  A is the sparse weight
 *    (M x K, pruned along K), B the dense activation (K x N), C the output
 *    (M x N).
 *  - Argument errors are detected on the host before anything is enqueued
 *    and return a status; nothing is launched in that case.  A launch failure
 *    returns ST24_ERR_CUDA.  Errors the kernels detect while running (a wait
 *    that ran out of time) are recorded in a per-device status word read by
 *    st24_device_status().
 *
 * Compressed form (the output of st24_prune_compress, the input of
 * st24_spmm), for an M x K matrix with K a multiple of 4:
 *  - values: M x K/2 elements, row-major with row stride K/2; the two kept
 *    values of group g (elements 4g..4g+3 of a row) at columns 2g and 2g+1,
 *    in ascending order of their position in the group.  ([CH26] worked
 *    example: values [w0 w3 | w5 w6].)
 *  - meta: M x ceil(K/8) bytes, row-major with row stride ceil(K/8); group g
 *    of a row is the 4-bit nibble (i0 | i1 << 2) with i0 < i1 the in-group
 *    indices of the kept values, stored in bits 4*(g%2)..4*(g%2)+3 of byte
 *    g/2.  ([CH26] worked example: indices [0 3 | 1 2], 2 bits each, 4 bits
 *    per group.)  Each 32-bit little-endian word of a row therefore holds the
 *    8 groups of 32 consecutive K, lowest K in the lowest bits, which is the
 *    order the sparse tensor-core instructions read their metadata in.
 */
#ifndef ST24_H
#define ST24_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define ST24_API __attribute__((visibility("default")))
#else
#define ST24_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Element types. */
typedef enum st24_dtype {
    ST24_F16 = 0,   /* IEEE binary16 */
    ST24_BF16 = 1,  /* bfloat16 */
    ST24_E4M3 = 2,  /* OCP FP8 E4M3 (finite-only "fn" variant, max 448) */
    ST24_S8 = 3,    /* int8 */
    ST24_F32 = 4,   /* IEEE binary32 (output only) */
    ST24_S32 = 5    /* int32 (output only, int8 inputs) */
} st24_dtype;

typedef enum st24_status {
    ST24_OK = 0,
    ST24_ERR_INVALID_ARG = 1,   /* null pointer, negative size, bad stride, K % 4 != 0 */
    ST24_ERR_UNSUPPORTED = 2,   /* valid but not handled: a type pair or a K this build rejects */
    ST24_ERR_MISALIGNED = 3,    /* a pointer or stride breaks an alignment the call states */
    ST24_ERR_CUDA = 4,          /* a CUDA runtime call or a launch failed */
    ST24_ERR_TIMEOUT = 5,       /* a kernel gave up on a wait (bounded spin) and returned early */
    ST24_ERR_WORKSPACE = 6      /* the workspace passed to st24_spmm is too small */
} st24_status;

/* Kernel families st24_spmm_ex can be asked to use. */
typedef enum st24_kernel {
    ST24_KERNEL_AUTO = 0,     /* what st24_spmm uses: MMA_SP for int8; for N <= 64 (bound by the
                                 weights' bytes) TCGEN05_NARROW -- MMA_SP_DIRECT for 16-bit inputs
                                 with N <= 4 whose grid fits in one wave; e4m3 with K not a multiple
                                 of 256 on TCGEN05 -- and TCGEN05 for wider products */
    ST24_KERNEL_TCGEN05 = 1,  /* tcgen05.mma.sp with TMEM accumulators (f16, bf16, e4m3 only) */
    ST24_KERNEL_MMA_SP = 2,   /* warp-level mma.sp fed by a TMA ring in shared memory (all input types) */
    ST24_KERNEL_MMA_SP_DIRECT = 3, /* warp-level mma.sp with the weights loaded straight into registers
                                      (1 <= N <= 32 only; 8-bit inputs widened exactly to f16; no
                                      workspace) */
    ST24_KERNEL_TCGEN05_NARROW = 4 /* tcgen05.mma.sp for narrow products (1 <= N <= 64; f16, bf16, and
                                      e4m3 with K % 256 == 0): each 128-row tile's K range split over a
                                      cluster of up to 8 CTAs that sum their partials in distributed
                                      shared memory; half an SM per CTA, so the next product's CTAs fit
                                      beside it; no workspace */
} st24_kernel;

/* Option bits for st24_spmm_ex (OR them together; 0 = none). */
typedef enum st24_spmm_flags {
    /* A_values and A_meta are fixed weights: no work that may still be running
       on `stream` when the call is enqueued writes them (they were written by
       work that has completed, or earlier on the stream behind a kernel that
       does not overlap its successor).  The kernel may then start loading them
       while the preceding kernel on the stream is still running, which hides
       the launch-to-launch gap of back-to-back decode-shaped products.  B and C
       are always read only after the preceding kernel has completed. */
    ST24_SPMM_FIXED_A = 1,
    /* A_values and A_meta hold TWO 2:4 compressed forms of M x K side by side
       along K, as written by st24_prune_compress_nm2 (values M x K, meta
       M x 2*ceil(K/8)): the compressed form of the M x 2K matrix
       [form 0 | form 1].  The product multiplies it by B read once per form --
       B's k-coordinate wraps at K -- into one accumulator, so the result is
       (form 0 + form 1) * B, e.g. a 4:8-pruned weight times B.  K is B's K and
       must be a multiple of 256 (else ST24_ERR_UNSUPPORTED); the workspace is
       st24_spmm_workspace_bytes(ab_type, c_type, M, N, 2K) bytes.  Not taken by
       ST24_KERNEL_MMA_SP_DIRECT. */
    ST24_SPMM_TWO_FORMS = 2
} st24_spmm_flags;

/* Library version, (major << 16) | (minor << 8) | patch. */
ST24_API int st24_version(void);

/* A static, human-readable name for a status value. */
ST24_API const char* st24_status_string(int status);

/*
 * Storage of the compressed form in bytes ([CH26] "The wins, quantified" and
 * the storage accounting of its listing: half the values plus a 2-bit index
 * per kept value).  values: M * (K/2) * sizeof(type); meta: M * ceil(K/8).
 * For 256 x 1024 at 2 bytes per value these are 262144 and 32768 bytes
 * (288.0 KB of a 512.0 KB dense matrix).  Return 0 for invalid arguments.
 */
ST24_API size_t st24_values_bytes(st24_dtype type, int64_t M, int64_t K);
ST24_API size_t st24_meta_bytes(int64_t M, int64_t K);

/*
 * Prune and compress ([CH26] "Python: Build a 2:4 Mask, Compress It, ...":
 * in every group of 4 consecutive elements along K keep the 2 with the
 * largest magnitude; [SS24] "What is 2:4 Structured Sparsity?").
 *   type   : ST24_F16, ST24_BF16, ST24_E4M3 or ST24_S8.
 *   W      : device, M x K dense matrix, row-major, row stride ldw >= K.
 *   values : device, st24_values_bytes(type, M, K) bytes, written.
 *   meta   : device, st24_meta_bytes(M, K) bytes, written.
 * Magnitude is |x|; ties go to the lower index; +0 and -0 tie; a NaN
 * outranks every number; a group always keeps exactly two slots (a group
 * with fewer non-zeros keeps zeros).  The result is bit-exact and
 * deterministic.  K must be a multiple of 4; M or K == 0 is a no-op.
 * Fast path when K*sizeof(type) % 16 == 0, W and ldw*sizeof(type) are
 * 16-byte aligned, values 8-byte aligned and meta 2-byte aligned; any other
 * valid layout takes a slower general kernel.
 */
ST24_API st24_status st24_prune_compress(st24_dtype type, const void* W, int64_t M, int64_t K, int64_t ldw,
                                void* values, void* meta, void* stream);

/*
 * N:M prune and compress into the 2:4 form ([CH26] "Block Sparsity, N:M
 * Generalizations, and Channel Pruning": keep N of every M consecutive
 * weights; 1:4, 2:8, ...).  In every group of m consecutive elements along K
 * the n of largest magnitude are kept (magnitude and ties as for
 * st24_prune_compress).  Supported: n in {1, 2}, m in {4, 8} (else
 * ST24_ERR_UNSUPPORTED); every aligned 4-element subgroup then keeps at most
 * two, so the output is the compressed form of st24_prune_compress (same
 * sizes and layout): a subgroup with one kept element stores it with a +0
 * partner at its lowest dropped index, one with none stores +0 at indices 0
 * and 1.  st24_spmm multiplies it exactly; st24_decompress gives the N:M
 * pruned matrix.  (2, 4) is st24_prune_compress.  K must be a multiple of 4
 * and of m; W aligned to the element size and values to twice it (else
 * ST24_ERR_MISALIGNED).  M or K == 0 is a no-op.  Bit-exact and
 * deterministic.
 */
ST24_API st24_status st24_prune_compress_nm(st24_dtype type, int n, int m, const void* W, int64_t M, int64_t K,
                                            int64_t ldw, void* values, void* meta, void* stream);

/*
 * N:M prune and compress into TWO 2:4 forms, for patterns that keep up to
 * four of an aligned 4-element subgroup ([CH26] "Block Sparsity, N:M
 * Generalizations, and Channel Pruning": 4:8, 3:8, ...).  The n largest
 * magnitudes of every m consecutive weights along K are kept (as for
 * st24_prune_compress_nm); in each 4-element subgroup the kept elements in
 * ascending index order go first to form 0 (its first two) and then to form 1
 * (the rest), a form holding fewer than two of them storing +0 partners at the
 * lowest indices of the subgroup not among its own.  The two forms are the
 * pruned matrix's two halves: their sum is the pruned matrix.
 *   values : device, st24_values_bytes(type, M, 2K) bytes: an M x K row-major
 *            matrix whose row r is form 0's K/2 values, then form 1's.
 *   meta   : device, st24_meta_bytes(M, 2K) bytes: row r is form 0's
 *            ceil(K/8) bytes, then form 1's.
 * Together they are the compressed form of the M x 2K matrix [form 0 | form 1]:
 * st24_spmm_ex with ST24_SPMM_TWO_FORMS multiplies it by B (read once per
 * form) into one accumulator, giving the pruned matrix times B.  Supported:
 * m in {4, 8}, 1 <= n <= min(4, m) (else ST24_ERR_UNSUPPORTED); K a multiple
 * of 4 and of m; W aligned to the element size and values to twice it (else
 * ST24_ERR_MISALIGNED).  M or K == 0 is a no-op.  Bit-exact and deterministic.
 */
ST24_API st24_status st24_prune_compress_nm2(st24_dtype type, int n, int m, const void* W, int64_t M, int64_t K,
                                             int64_t ldw, void* values, void* meta, void* stream);

/*
 * Quantise, then prune and compress ([CH26] "Sparsity + Quantization
 * Combine": 2:4 sparsity and 8-bit weights stack; "Establishing a Scalable
 * Sparse Ecosystem with the Universal Sparse Tensor Abstraction", section
 * "Building a Practical Compression Pipeline": prune plus INT8 post-training
 * quantisation).  Per row m of the 16-bit weight W, in fp32 arithmetic with
 * round-to-nearest and no contraction:
 *   amax      = max_k |W[m][k]|,  Q = 448 (ST24_E4M3) or 127 (ST24_S8),
 *   inv       = Q / amax,  code = encode(W[m][k] * inv),
 *   scales[m] = amax / Q   (so W ~ code * scales[m]);
 * encode is nearest-even with saturation to +-448 (e4m3) or nearest-even
 * clamped to [-127, 127] (int8); a row with amax == 0 gets scales[m] = 0
 * and zero codes.  The codes are then pruned and compressed exactly as by
 * st24_prune_compress with type dst_type, in one pass over W (read once when
 * K <= 16384).  Pass the result to st24_spmm with row_scale = scales (times
 * any activation scale) to get the dequantised product.
 *   src_type : ST24_F16 or ST24_BF16;  dst_type : ST24_E4M3 or ST24_S8.
 *   W        : device, M x K, row stride ldw >= K; must be finite (NaN or
 *              Inf give unspecified codes).
 *   values   : device, st24_values_bytes(dst_type, M, K) bytes, written.
 *   meta     : device, st24_meta_bytes(M, K) bytes, written.
 *   scales   : device, M floats, written.
 * K must be a multiple of 16 (else ST24_ERR_UNSUPPORTED); W and
 * ldw*2 16-byte aligned, values 8-byte, meta 2-byte and scales 4-byte
 * aligned (else ST24_ERR_MISALIGNED).  M == 0 is a no-op.  Bit-exact and
 * deterministic.
 */
ST24_API st24_status st24_quantize_prune_compress(st24_dtype src_type, st24_dtype dst_type, const void* W,
                                                  int64_t M, int64_t K, int64_t ldw, void* values, void* meta,
                                                  float* scales, void* stream);

/*
 * Inverse of compression ([SS24] "How Engineers Enable 2:4 Sparsity": the
 * libraries handle compression and decompression; [CH26] pruned row
 * [w0 0 0 w3 | 0 w5 w6 0]): writes the M x K dense matrix W (row stride
 * ldw >= K) with the kept values at their indices and +0 elsewhere.
 * Metadata nibbles whose two indices are not strictly ascending are not a
 * valid compressed form; the result for such groups is unspecified (no
 * memory outside W is written).  Same alignment fast path as above.
 */
ST24_API st24_status st24_decompress(st24_dtype type, const void* values, const void* meta, int64_t M,
                            int64_t K, void* W, int64_t ldw, void* stream);

/*
 * Bytes of workspace st24_spmm needs for these sizes (0 when the chosen
 * schedule needs none).  The workspace holds fp32 partial tiles of the
 * split-K / stream-K schedule and one 32-bit counter per output tile.
 * It must be zero-filled before its first use; every successful st24_spmm
 * leaves the counters at zero again, so a workspace can be reused by later
 * calls on the same stream without clearing.  After a call whose kernels gave
 * up on a wait (st24_device_status returns ST24_ERR_TIMEOUT) some counters
 * may be left nonzero: zero-fill the workspace again before reusing it.
 * Calls that run at the same time must not share a workspace.
 */
ST24_API size_t st24_spmm_workspace_bytes(st24_dtype ab_type, st24_dtype c_type, int64_t M, int64_t N,
                                 int64_t K);

/*
 * Sparse x dense product ([CH26] "2:4 Fine-Grained Structured Sparsity": the
 * two stored weights of each group multiply the two activations their
 * indices select; the other two products are zero and never computed):
 *
 *   C(m, n) = alpha * row_scale[m] * sum_k A(m, k) * B(k, n) + beta * C(m, n)
 *
 *   ab_type  : ST24_F16, ST24_BF16, ST24_E4M3 (fp32 accumulation) or ST24_S8
 *              (int32 accumulation, exact).
 *   c_type   : ST24_F32, ST24_BF16 or ST24_F16 for any ab_type; ST24_S32
 *              only for ST24_S8 with alpha == 1, beta == 0 and no row_scale
 *              (the raw int32 sums).
 *   A_values, A_meta : device, the compressed form of A (M x K).
 *   B        : device, element (k, n) at B[n*ldb + k] (K-major; a row-major
 *              activation X[N, K] with ldb >= K).
 *   C        : device, element (m, n) at C[n*ldc + m] (ldc >= M; a
 *              row-major Y[N, M]); read when beta != 0, always written.
 *   row_scale: device, M fp32 values, or NULL for 1.
 *   workspace: device, ws_bytes >= st24_spmm_workspace_bytes(...), or NULL
 *              when that is 0.  See st24_spmm_workspace_bytes.
 * The output is rounded to nearest-even from fp32 (int32 is exact).
 * Requirements: K % 128 == 0 (ST24_ERR_UNSUPPORTED otherwise); A_values, B
 * and A_meta 16-byte aligned; ldb*sizeof(ab_type) % 16 == 0; C aligned to
 * its element size.  M, N == 0 is a no-op.
 */
ST24_API st24_status st24_spmm(st24_dtype ab_type, st24_dtype c_type, int64_t M, int64_t N, int64_t K,
                      float alpha, const void* A_values, const void* A_meta,
                      const void* B, int64_t ldb, float beta, void* C, int64_t ldc,
                      const float* row_scale, void* workspace, size_t ws_bytes, void* stream);

/*
 * st24_spmm with options: an explicitly chosen kernel family (for testing one
 * family against another, or a family against the oracle) and `flags`, a set
 * of st24_spmm_flags bits.  ST24_KERNEL_TCGEN05 or ST24_KERNEL_TCGEN05_NARROW
 * with ab_type ST24_S8, ST24_KERNEL_MMA_SP_DIRECT with N > 32 and
 * ST24_KERNEL_TCGEN05_NARROW with N > 64 return ST24_ERR_UNSUPPORTED.  Arguments, workspace and results are as for
 * st24_spmm (which is st24_spmm_ex with ST24_KERNEL_AUTO and no flags);
 * st24_spmm_workspace_bytes covers every family.  An unknown `kernel` or an
 * unknown flag bit returns ST24_ERR_INVALID_ARG.
 */
ST24_API st24_status st24_spmm_ex(st24_kernel kernel, unsigned flags, st24_dtype ab_type, st24_dtype c_type, int64_t M,
                                  int64_t N, int64_t K, float alpha, const void* A_values,
                                  const void* A_meta, const void* B, int64_t ldb, float beta, void* C,
                                  int64_t ldc, const float* row_scale, void* workspace, size_t ws_bytes,
                                  void* stream);

/*
 * st24_spmm for callers that cannot allocate device memory.  No counterpart
 * in the source pages: it is a deployment variant of st24_spmm.
 *
 * Some callers cannot call cudaMalloc or take memory from an allocator: a
 * plugin inside a serving runtime whose device memory is owned entirely by
 * the runtime's pool, code that runs while a stream is being captured in the
 * global capture mode (where cudaMalloc is not allowed), or a latency-critical
 * path that must not take the allocator's lock or synchronise the device.
 * This call takes the same arguments as st24_spmm without the workspace and
 * keeps the split-K / stream-K partial tiles and tile counters in a
 * fixed-size array in device global memory owned by the library: 16 MiB on
 * every GPU that loads the library, held until the process exits.  It calls
 * no cudaMalloc, cudaFree or allocating library routine.
 *   - A product whose schedule needs more scratch than 16 MiB (for example
 *     N > 64 with a stream-K tail on a large M) returns ST24_ERR_WORKSPACE and
 *     launches nothing; every product with N <= 64 fits.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture begins.
 *   - Every call on a device shares the one array, which keeps the last
 *     call's contents; each call clears the tile counters (a cudaMemsetAsync
 *     on `stream`) before its kernel.  Calls whose work overlaps on the GPU
 *     (on different streams, or from different host threads) race on the
 *     array and give wrong results: serialise them.
 * Results are identical to st24_spmm with a workspace of its own.
 */
ST24_API st24_status st24_spmm_noalloc(st24_dtype ab_type, st24_dtype c_type, int64_t M, int64_t N,
                                       int64_t K, float alpha, const void* A_values, const void* A_meta,
                                       const void* B, int64_t ldb, float beta, void* C, int64_t ldc,
                                       const float* row_scale, void* stream);

/*
 * The transposed use of a compressed weight ([CH26] "2:4: ~2x on the Matmul,
 * Less End-to-End": after pruning to 2:4 the model is retrained, and the
 * input gradient of a layer Y = X * A^T is dX = dY * A, a sum over M, along
 * which A has no 2:4 structure):
 *
 *   C(k, n) = alpha * sum_m A(m, k) * B(m, n) + beta * C(k, n)
 *
 *   ab_type  : ST24_F16 or ST24_BF16 (fp32 accumulation); c_type: ST24_F32,
 *              ST24_BF16 or ST24_F16.
 *   A_values, A_meta : device, the compressed form of A (M x K), as for
 *              st24_spmm; it is read compressed and expanded on chip.
 *   B        : device, element (m, n) at B[n*ldb + m] (a row-major dY[N, M],
 *              ldb >= M).
 *   C        : device, element (k, n) at C[n*ldc + k] (a row-major dX[N, K],
 *              ldc >= K); read when beta != 0, always written.
 * The output is rounded to nearest-even from fp32.  Requirements: K % 128 ==
 * 0 (ST24_ERR_UNSUPPORTED otherwise); A_values, A_meta and B 16-byte aligned,
 * ldb*2 % 16 == 0, C aligned to its element size (ST24_ERR_MISALIGNED).  No
 * workspace.  N or K == 0 is a no-op; M == 0 gives C = beta * C.
 */
ST24_API st24_status st24_spmm_t(st24_dtype ab_type, st24_dtype c_type, int64_t M, int64_t N, int64_t K,
                                 float alpha, const void* A_values, const void* A_meta, const void* B,
                                 int64_t ldb, float beta, void* C, int64_t ldc, void* stream);

/*
 * Synchronises `stream`, then reads and clears the status word the kernels
 * of the current device write when a bounded wait runs out
 * (ST24_ERR_TIMEOUT), or returns ST24_ERR_CUDA if the stream reports an
 * error.  ST24_OK otherwise.
 */
ST24_API st24_status st24_device_status(void* stream);

#ifdef __cplusplus
}
#endif

#endif /* ST24_H */
