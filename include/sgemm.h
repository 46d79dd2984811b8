/*
 * sgemm.h — C ABI of the GB300 (sm_103a) dense fp32 matrix multiplication
 * library, libsgemm_gb300.so.
 *
 * The operation is the plain product of row-major single-precision matrices
 *
 *     C[i][j] = sum over k = 0 .. K-1 of A[i][k] * B[k][j]
 *
 * with A of M x K, B of K x N and C of M x N. This is the definition stated
 * in "CUDA算子优化(4)：矩阵乘法", section "矩阵乘法的数学定义", and in
 * "CUDA内存优化入门：从Naive到Tiled矩阵乘法", section 三 (formula block);
 * both index row-major storage as A[i*K + k], B[k*N + j], C[i*N + j]. This
 * ABI adds a row stride per matrix: element (r, c) of a matrix with row
 * stride ld sits at offset r*ld + c (in elements, not bytes).
 *
 * Conventions shared by every entry point
 *   - Sizes and strides are int64_t element counts.
 *   - Matrix pointers are device pointers (memory that the current CUDA
 *     device can read and write), except where an entry point says "host".
 *   - The caller owns every buffer. The library keeps no pointer after a
 *     call returns and never synchronises the stream. It allocates device
 *     memory in one case only: a tensor-core product whose A or B rows are
 *     not 16-byte aligned (row stride or base address), from 1.25 * 2^30
 *     multiply-adds on, copies those operands into aligned rows in scratch
 *     taken from a stream-ordered pool the library creates per device on
 *     first use (cudaMallocFromPoolAsync on `stream`, freed with
 *     cudaFreeAsync on `stream` behind the product; the pool keeps up to
 *     512 MiB between calls). If that allocation fails the product runs
 *     without the copies. No host memory is allocated.
 *   - Calls are asynchronous: they enqueue work on `stream` and return. A
 *     NULL stream means the legacy default stream. Errors raised by a kernel
 *     while it runs surface on the stream (cudaStreamSynchronize), not here.
 *   - The library runs only on devices of compute capability 10.3 (sm_103a).
 *   - No entry point ever calls exit() or falls back to the CPU.
 */
#ifndef DENSE_FP32_SGEMM_GB300_H
#define DENSE_FP32_SGEMM_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t, declared here so the header needs no CUDA include. */
typedef struct CUstream_st *sgemm_stream_t;

/* Status codes returned by every int-returning entry point. */
enum sgemm_status {
    SGEMM_OK = 0,
    SGEMM_ERR_INVALID_ARG = 1, /* negative size, stride shorter than a row, NULL
                                  pointer with a non-empty extent, C overlapping
                                  A or B, unknown variant or tuning key */
    SGEMM_ERR_UNSUPPORTED = 2, /* a forced variant cannot run this shape or
                                  alignment (SGEMM_AUTO never returns this) */
    SGEMM_ERR_LAUNCH = 3,      /* a CUDA call failed while enqueueing */
    SGEMM_ERR_DEVICE = 4,      /* no usable device, or not compute capability 10.3 */
    SGEMM_ERR_TIMEOUT = 5,     /* a kernel gave up a bounded wait (see sgemm_device_status) */
    SGEMM_ERR_SCRATCH = 6      /* sgemm_f32_noalloc: the product needs more scratch than its
                                  fixed buffer (SGEMM_NOALLOC_SCRATCH_BYTES) holds */
};

/* Kernel variants. */
enum sgemm_variant {
    SGEMM_AUTO = 0,   /* pick per shape and alignment: TF32X3 from 2^14 multiply-adds (tile
                         padding discounted), FFMA below */
    SGEMM_FFMA = 1,   /* register-blocked fp32 fused multiply-add on the CUDA cores */
    SGEMM_TF32X3 = 2  /* tensor cores (tcgen05) with the three-term TF32 split */
};

/*
 * C = A * B.
 *   M, N, K   sizes; each >= 0.
 *   A, lda    M x K, row stride lda >= K; read only.
 *   B, ldb    K x N, row stride ldb >= N; read only.
 *   C, ldc    M x N, row stride ldc >= N; every element of the M x N box is
 *             overwritten (no alpha, no beta: C's old contents are not read).
 *             Elements between column N and the next row start are never
 *             written. C must not overlap A or B.
 *   stream    CUDA stream to enqueue on.
 * M == 0 or N == 0: nothing is enqueued, SGEMM_OK. K == 0: C is set to zero
 * (the empty sum). A NULL pointer is accepted only for a matrix with no
 * elements. Results: every output is the exact sum rounded with fp32
 * arithmetic in an order the library chooses; the acceptance bound is
 * max |C - C_exact| / sum_k |A[i][k]| |B[k][j]| <= 1e-5, and inputs whose
 * products and partial sums are integers below 2^24 give exact results.
 * Non-finite inputs follow IEEE arithmetic on both variants: an infinity
 * gives +-inf by the signs of the products it takes part in, inf * 0 and
 * inf - inf give NaN, a NaN input gives NaN in every output that uses it.
 * (SGEMM_TF32X3's split alone would turn an infinity into NaN: it finds
 * every NaN it produced and recomputes that output over its k-range with
 * fp32 fused multiply-adds, at no cost when no output is NaN.)
 * Returns SGEMM_OK or an sgemm_status code; on error nothing is enqueued.
 */
int sgemm_f32(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda, const float *B,
              int64_t ldb, float *C, int64_t ldc, sgemm_stream_t stream);

/* Operand forms for sgemm_f32_ex. */
enum sgemm_op {
    SGEMM_OP_N = 0, /* op(X) = X */
    SGEMM_OP_T = 1  /* op(X) = X^T */
};

/*
 * C = alpha * op(A) * op(B) + beta * C, the general (BLAS GEMM) form; the
 * source pages define only C = A * B, which is sgemm_f32 (alpha = 1,
 * beta = 0, no transposes).
 *   transA    SGEMM_OP_N: A is stored M x K, row stride lda >= K.
 *             SGEMM_OP_T: A is stored K x M, row stride lda >= M (op(A) = A^T).
 *   transB    SGEMM_OP_N: B is stored K x N, row stride ldb >= N.
 *             SGEMM_OP_T: B is stored N x K, row stride ldb >= K.
 *   C, ldc    M x N, row stride ldc >= N. beta == 0: C is only written (it may
 *             hold NaN); otherwise C is read and updated in place.
 *   alpha     alpha == 0 or K == 0: C = beta * C (C = 0 when beta == 0) and A,
 *             B are not read.
 * Same conventions, errors and accuracy bound as sgemm_f32, with the error
 * scale |alpha| sum_k |op(A)[i][k]| |op(B)[k][j]| + |beta| |C[i][j]|.
 * Both variants serve every operand form at any alignment.
 */
int sgemm_f32_ex(int transA, int transB, int64_t M, int64_t N, int64_t K, float alpha, const float *A,
                 int64_t lda, const float *B, int64_t ldb, float beta, float *C, int64_t ldc,
                 sgemm_stream_t stream);

/*
 * Strided batch of independent products: for b = 0 .. batch-1,
 *     C_b = alpha * op(A_b) * op(B_b) + beta * C_b
 * with A_b = A + b*strideA, B_b = B + b*strideB, C_b = C + b*strideC
 * (strides in elements). Each item follows sgemm_f32_ex (same transA, transB,
 * M, N, K, alpha, beta, lda, ldb, ldc for all items). strideA or strideB may
 * be 0 (one matrix shared by every item); C items must not overlap one
 * another (strideC >= (M-1)*ldc + N) nor any A or B item. batch == 0:
 * nothing is enqueued. The whole batch runs as one persistent launch (plus a
 * small scaling launch when some tiles are split along K, and one copy launch
 * when rows TMA cannot address are copied, see the conventions above).
 */
int sgemm_f32_batched(int transA, int transB, int64_t M, int64_t N, int64_t K, float alpha, const float *A,
                      int64_t lda, int64_t strideA, const float *B, int64_t ldb, int64_t strideB, float beta,
                      float *C, int64_t ldc, int64_t strideC, int64_t batch, sgemm_stream_t stream);

/* Bias forms of the fused epilogue (sgemm_f32_fused). */
enum sgemm_bias {
    SGEMM_BIAS_NONE = 0,    /* no bias; `bias` is not read */
    SGEMM_BIAS_PER_COL = 1, /* N values: bias[j] is added to every element of column j */
    SGEMM_BIAS_PER_ROW = 2  /* M values: bias[i] is added to every element of row i */
};

/* Activations of the fused epilogue, applied to each element x. */
enum sgemm_activation {
    SGEMM_ACT_NONE = 0,
    SGEMM_ACT_RELU = 1, /* x < 0 ? 0 : x (NaN stays NaN) */
    SGEMM_ACT_GELU = 2, /* x * Phi(x) = x / 2 * (1 + erf(x / sqrt(2))), Phi the standard normal CDF,
                           Phi evaluated by a rational approximation of error below 7.5e-8
                           before fp32 rounding (not the tanh form) */
    SGEMM_ACT_SILU = 3  /* x / (1 + exp(-x)) */
};

/*
 * Product with a fused epilogue:
 *     C = act(alpha * op(A) * op(B) + beta * C + bias)
 * The source pages compute the product alone and motivate it as the core
 * operation of neural-network layers ("CUDA内存优化入门：从Naive到Tiled矩阵
 * 乘法", section 一); a layer's forward pass is this product followed by a
 * bias and an activation, and fusing them saves the extra pass over C.
 *   transA .. ldc   as sgemm_f32_ex.
 *   bias            device pointer, read only: N floats (SGEMM_BIAS_PER_COL)
 *                   or M floats (SGEMM_BIAS_PER_ROW), contiguous, any
 *                   alignment, not overlapping C; ignored for SGEMM_BIAS_NONE.
 *   bias_kind       an sgemm_bias value.
 *   activation      an sgemm_activation value.
 * The bias is added and the activation applied to the fp32 value
 * alpha * acc + beta * C, once per element, in the kernel that writes C.
 * Tiles split along K (stream-K) take the bias in the pre-pass that scales C
 * by beta, and the activation in one more small launch over those tiles
 * after the product. Accuracy: the error scale becomes |alpha| sum_k |op(A)|
 * |op(B)| + |beta| |C| + |bias|; the activations are at most 1.13-Lipschitz
 * (GELU), so the product's bound carries over up to that factor plus a few
 * fp32 roundings of the activation itself. Same errors as sgemm_f32_ex, plus
 * SGEMM_ERR_INVALID_ARG for an unknown bias_kind or activation, a null bias
 * with a bias kind other than NONE, or a bias overlapping C.
 */
int sgemm_f32_fused(int transA, int transB, int64_t M, int64_t N, int64_t K, float alpha, const float *A,
                    int64_t lda, const float *B, int64_t ldb, float beta, float *C, int64_t ldc,
                    const float *bias, int bias_kind, int activation, sgemm_stream_t stream);

/*
 * C = A * B for matrices that live in HOST memory, through caller-owned
 * device buffers. Enqueues, on `stream`: the copy of A_host into dA and of
 * B_host into dB (row strides kept), the product into dC, and the copy of
 * dC back into C_host. dA, dB, dC are device buffers with the same row
 * strides as the host matrices (lda, ldb, ldc) and at least that many rows.
 * Host buffers should be page-locked (cudaHostAlloc) for the copies to be
 * asynchronous; the caller synchronises the stream before reading C_host.
 * Same sizes, strides, errors and results as sgemm_f32, except that an
 * error may come back after part of the work was enqueued: the buffers are
 * then in use until `stream` has been synchronised, as on success (`stream`
 * still waits for whatever the call enqueued on the library streams).
 * Products of at least 2^30 multiply-adds with N >= 512 are pipelined over
 * up to eight column panels of B and C (widths in multiples of 256): A and
 * the B panels are copied in on `stream`, panel j's product runs on a
 * library stream as soon as its B panel is in, and its C panel is copied
 * out on a second library stream, so copies in, products and copies out
 * overlap. `stream` waits for the last
 * copy out, so the call behaves as if everything ran in order on `stream`.
 * The two library streams and their events are created on the first
 * pipelined call on a device and kept for the process (creating them takes
 * no device memory); concurrent pipelined calls on one device are serialised
 * while they enqueue.
 */
int sgemm_f32_from_host(int64_t M, int64_t N, int64_t K, const float *A_host, int64_t lda,
                        const float *B_host, int64_t ldb, float *C_host, int64_t ldc, float *dA,
                        float *dB, float *dC, sgemm_stream_t stream);

/*
 * C = A * B like sgemm_f32 (same arguments, results and errors), without
 * allocating memory. The pages define no such entry point; it exists because
 * of sgemm_f32's one allocation (see the conventions above: the aligned
 * copies of A or B whose rows are not 16-byte aligned, for tensor-core
 * products of at least 1.25 * 2^30 multiply-adds).
 * Some callers cannot let a library take device memory during a call: a
 * program whose device memory is all reserved up front by its own allocator
 * (a framework's caching allocator holding most of HBM), a service that must
 * know before the first request how much memory the library uses, or code
 * that may not risk an allocation failing in the middle of a step. This entry
 * point puts those copies into one fixed buffer of SGEMM_NOALLOC_SCRATCH_BYTES
 * per device instead: a file-scope __device__ array of the library, created
 * with the library's device code when the module is loaded, not by this call.
 *   - A product whose copies would need more than SGEMM_NOALLOC_SCRATCH_BYTES
 *     is rejected with SGEMM_ERR_SCRATCH before anything is enqueued. The
 *     copies take 4 * rows * round_up(columns, 4) bytes for each operand whose
 *     rows are not aligned (A: M x K, B: K x N), each rounded up to 256 bytes;
 *     products that make no copies (aligned rows, or fewer multiply-adds)
 *     have no limit.
 *   - Nothing in the buffer needs to start at zero: every value a product
 *     reads from it was written by the copy pass of the same call.
 *   - The buffer is shared by every call of this entry point on a device. Two
 *     calls whose work may overlap on the GPU (different streams with no
 *     ordering between them, or calls from several host threads) race on it
 *     and give wrong results; order them (one stream, or events).
 *   - The first call on each device looks up the buffer's device address
 *     (cudaGetSymbolAddress, with that device current); make that first call
 *     before any stream capture begins. If the lookup fails the call returns
 *     SGEMM_ERR_DEVICE.
 */
#define SGEMM_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
int sgemm_f32_noalloc(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda, const float *B,
                      int64_t ldb, float *C, int64_t ldc, sgemm_stream_t stream);

/* Variant selection, process-wide (all threads, all devices). Returns SGEMM_OK
 * or SGEMM_ERR_INVALID_ARG for an unknown value. The initial value is
 * SGEMM_AUTO, or the value of the environment variable SGEMM_VARIANT (0, 1, 2
 * or a variant name) read at the first call. */
int sgemm_set_variant(int variant);
int sgemm_get_variant(void);
/* Name of a variant ("auto", "ffma", "tf32x3"), or "unknown". Static storage. */
const char *sgemm_variant_name(int variant);
/* Variant that the most recent successful product call (any entry point) in
 * this process enqueued (SGEMM_AUTO before any call). For reporting only. */
int sgemm_last_variant_used(void);
/* Number of kernel launches that the most recent successful product call
 * (any entry point) enqueued (0 for an empty product). For reporting only. */
int sgemm_last_launch_count(void);

/* Human-readable text of a status code. Static storage. */
const char *sgemm_strerror(int status);

/*
 * Bounded waits. Kernels that wait on an mbarrier give up after a fixed time
 * (SGEMM_TUNE_WATCHDOG_MS), record the event in a per-device flag, stop
 * issuing work and return; C is then incomplete. This call waits for all work on the current
 * device (cudaDeviceSynchronize), then returns SGEMM_ERR_TIMEOUT if a kernel
 * gave up since the last call (and clears the flag), SGEMM_ERR_LAUNCH if the
 * device reported an error, else SGEMM_OK.
 */
int sgemm_device_status(void);

/*
 * Exercises the bounded-wait reporting path without faulting the device:
 * enqueues on `stream` a one-warp kernel whose single mbarrier wait can never
 * complete (nothing arrives). The wait gives up after wait_ms (1 .. 60000),
 * records the event in the watchdog flag and the kernel exits normally, so a
 * following sgemm_device_status() returns SGEMM_ERR_TIMEOUT (once) and the
 * CUDA context stays usable. Returns SGEMM_OK once enqueued,
 * SGEMM_ERR_INVALID_ARG for wait_ms out of range, SGEMM_ERR_DEVICE or
 * SGEMM_ERR_LAUNCH.
 */
int sgemm_watchdog_selftest(int64_t wait_ms, sgemm_stream_t stream);

/*
 * Tuning keys for sgemm_set_tuning / sgemm_get_tuning (process-wide).
 *   SGEMM_TUNE_FFMA_TILE     0 = choose per shape; 1 = 128x256; 2 = 128x128;
 *                            3 = 64x64 (FFMA block tile, M x N)
 *   SGEMM_TUNE_STREAM_K      0 = choose per shape; 1 = data-parallel only;
 *                            2 = data-parallel waves plus a stream-K remainder;
 *                            3 = stream-K over all tiles
 *   SGEMM_TUNE_WATCHDOG_MS   milliseconds a bounded wait polls before it gives
 *                            up (1 .. 60000; default 2000)
 *   SGEMM_TUNE_TF32X3_KERNEL  tensor-core kernel: 0 = automatic (default):
 *                            where A and B have 16-byte aligned bases and
 *                            row strides, the SM-pair kernel from 2^20
 *                            multiply-adds on and the TMA kernel with A in
 *                            tensor memory below; otherwise, from 1.25 * 2^30
 *                            multiply-adds on, the unaligned operands are
 *                            first copied into aligned rows (scratch from a
 *                            stream-ordered pool, see sgemm_f32) and the TMA
 *                            kernels run; below that per-thread loads (the
 *                            SM-pair kernel for the transposed forms);
 *                            1 = per-thread loads, 2 = TMA, 3 = TMA with A's
 *                            operands in tensor memory, 4 = SM pairs (tcgen05
 *                            cta_group::2 on clusters of two CTAs; TMA loads
 *                            for 16-byte aligned rows, cp.async otherwise),
 *                            5 = as 0, but unaligned operands are copied at
 *                            any size. Kernels 2 and 3 need 16-byte aligned
 *                            rows (else kernel 1 runs, or kernel 4 for the
 *                            transposed forms); kernel 1 serves op(A) = A,
 *                            op(B) = B only (the transposed forms take kernel
 *                            3 when the rows are aligned, else kernel 4).
 * Returns SGEMM_OK or SGEMM_ERR_INVALID_ARG. sgemm_get_tuning returns the
 * value, or -1 for an unknown key.
 */
enum sgemm_tuning_key {
    SGEMM_TUNE_FFMA_TILE = 1,
    SGEMM_TUNE_STREAM_K = 2,
    SGEMM_TUNE_WATCHDOG_MS = 3,
    SGEMM_TUNE_TF32X3_KERNEL = 4,
    SGEMM_TUNE_LAST_TC_KERNEL = 5  /* read only: the tensor-core kernel (1-4) the
                                      last SGEMM_TF32X3 call on this process ran */
};
int sgemm_set_tuning(int key, int64_t value);
int64_t sgemm_get_tuning(int key);

/* Library version as "major.minor.patch". Static storage. */
const char *sgemm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DENSE_FP32_SGEMM_GB300_H */
