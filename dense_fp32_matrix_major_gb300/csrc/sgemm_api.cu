// C ABI of libsgemm_gb300: argument checks, variant selection and dispatch.
// The declarations and the contract of every entry point are in sgemm.h.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "sgemm.h"
#include "sgemm_internal.h"

namespace sgemm {
namespace {

constexpr int kMaxDevices = 64;

std::once_flag g_env_once;
std::atomic<int> g_variant{SGEMM_AUTO};
std::atomic<int> g_last_variant{SGEMM_AUTO};
std::atomic<int> g_last_launches{0};
std::atomic<int64_t> g_tune_tile{0};
std::atomic<int64_t> g_tune_sk{0};

struct DevCache {
    std::once_flag once[kMaxDevices];
    DeviceInfo info[kMaxDevices];
    int status[kMaxDevices];
};
DevCache g_dev;

int parse_variant(const char *s) {
    if (!s || !*s) return -1;
    if (!strcmp(s, "0") || !strcmp(s, "auto")) return SGEMM_AUTO;
    if (!strcmp(s, "1") || !strcmp(s, "ffma")) return SGEMM_FFMA;
    if (!strcmp(s, "2") || !strcmp(s, "tf32x3")) return SGEMM_TF32X3;
    return -1;
}

void read_env() {
    std::call_once(g_env_once, [] {
        const int v = parse_variant(getenv("SGEMM_VARIANT"));
        if (v >= 0) g_variant.store(v);
    });
}

// Byte range [lo, hi) spanned by a rows x cols matrix with row stride ld.
void span(const void *p, int64_t rows, int64_t cols, int64_t ld, uintptr_t *lo, uintptr_t *hi) {
    *lo = reinterpret_cast<uintptr_t>(p);
    *hi = *lo + static_cast<uintptr_t>(((rows - 1) * ld + cols) * static_cast<int64_t>(sizeof(float)));
}

bool overlaps(const void *x, int64_t xr, int64_t xc, int64_t xld, const void *y, int64_t yr, int64_t yc,
              int64_t yld) {
    if (xr == 0 || xc == 0 || yr == 0 || yc == 0) return false;
    uintptr_t a0, a1, b0, b1;
    span(x, xr, xc, xld, &a0, &a1);
    span(y, yr, yc, yld, &b0, &b1);
    return a0 < b1 && b0 < a1;
}

int check_args(int transA, int transB, int64_t M, int64_t N, int64_t K, const float *A, int64_t lda,
               const float *B, int64_t ldb, const float *C, int64_t ldc) {
    if (transA != SGEMM_OP_N && transA != SGEMM_OP_T) return SGEMM_ERR_INVALID_ARG;
    if (transB != SGEMM_OP_N && transB != SGEMM_OP_T) return SGEMM_ERR_INVALID_ARG;
    if (M < 0 || N < 0 || K < 0) return SGEMM_ERR_INVALID_ARG;
    // Stored shapes: A is M x K (K x M when transposed), B is K x N (N x K).
    const int64_t a_rows = transA ? K : M, a_cols = transA ? M : K;
    const int64_t b_rows = transB ? N : K, b_cols = transB ? K : N;
    if (lda < a_cols || ldb < b_cols || ldc < N) return SGEMM_ERR_INVALID_ARG;
    if (lda < 1 || ldb < 1 || ldc < 1) return SGEMM_ERR_INVALID_ARG;
    // Element offsets must fit in int64 with room to spare.
    const int64_t lim = INT64_C(1) << 60;
    if ((a_rows > 0 && lda > lim / a_rows) || (b_rows > 0 && ldb > lim / b_rows) || (M > 0 && ldc > lim / M))
        return SGEMM_ERR_INVALID_ARG;
    if (M > 0 && K > 0 && !A) return SGEMM_ERR_INVALID_ARG;
    if (K > 0 && N > 0 && !B) return SGEMM_ERR_INVALID_ARG;
    if (M > 0 && N > 0 && !C) return SGEMM_ERR_INVALID_ARG;
    if (M > 0 && N > 0) {
        if (overlaps(C, M, N, ldc, A, a_rows, a_cols, lda) || overlaps(C, M, N, ldc, B, b_rows, b_cols, ldb))
            return SGEMM_ERR_INVALID_ARG;
    }
    return SGEMM_OK;
}

// Checks of the fused epilogue's arguments: known bias kind and activation,
// a bias vector (M or N floats) that exists and does not overlap C.
int check_epilogue(int64_t M, int64_t N, const float *C, int64_t ldc, const float *bias, int bias_kind,
                   int act) {
    if (bias_kind < SGEMM_BIAS_NONE || bias_kind > SGEMM_BIAS_PER_ROW) return SGEMM_ERR_INVALID_ARG;
    if (act < SGEMM_ACT_NONE || act > SGEMM_ACT_SILU) return SGEMM_ERR_INVALID_ARG;
    if (bias_kind == SGEMM_BIAS_NONE || M == 0 || N == 0) return SGEMM_OK;
    const int64_t len = bias_kind == SGEMM_BIAS_PER_COL ? N : M;
    if (!bias) return SGEMM_ERR_INVALID_ARG;
    if (overlaps(C, M, N, ldc, bias, 1, len, len)) return SGEMM_ERR_INVALID_ARG;
    return SGEMM_OK;
}

// AUTO: the tensor-core path from 2^14 useful multiply-adds up, at any K:
// its accumulation rounds toward zero, so beyond K = 8192 it splits every
// tile along K into units of K <= 4096 (2.9e-6 of the 1e-5 bound) added with
// round-to-nearest fp32 adds. "Useful" discounts the padding of the
// tensor-core path's 128 x 256 tiles, which matters for batches of small
// products (the FFMA path has 64 x 64 tiles for those).
int auto_variant(const Problem &p, const DeviceInfo &dev) {
    const double m_pad = static_cast<double>((p.M + 127) / 128 * 128);
    const double n_pad = static_cast<double>((p.N + 255) / 256 * 256);
    const double fill = static_cast<double>(p.M) * static_cast<double>(p.N) / (m_pad * n_pad);
    const double work = static_cast<double>(p.M) * static_cast<double>(p.N) * static_cast<double>(p.K) *
                        static_cast<double>(p.batch) * fill;
    // Measured on GB300 (CUDA events, L2 flushed): the tensor-core kernels
    // are faster from 64^3 on (64^3: 11.6 vs 16.4 us; 256^3: 19.7 vs 28.7;
    // 2048 x 128 x 512: 20.0 vs 30.7; 300 x 257 x 513, rows not 16-byte
    // aligned: 36.3 vs 42.0), FFMA only on the tiniest products (16^3: 8.3
    // vs 10.5 us), where launch latency is all there is.
    if (work >= 16384.0 && tf32x3_supports(p, dev)) return SGEMM_TF32X3;
    return SGEMM_FFMA;
}

// Extra checks for a strided batch: non-negative strides, C items that do
// not overlap one another, and no C item overlapping any A or B item (checked
// on the ranges the whole batch spans).
int check_batch(const Problem &p) {
    if (p.batch < 0 || p.strideA < 0 || p.strideB < 0 || p.strideC < 0) return SGEMM_ERR_INVALID_ARG;
    if (p.batch <= 1 || p.M == 0 || p.N == 0) return SGEMM_OK;
    const int64_t lim = INT64_C(1) << 60;
    if (p.strideA > lim / p.batch || p.strideB > lim / p.batch || p.strideC > lim / p.batch)
        return SGEMM_ERR_INVALID_ARG;
    if (p.strideC < (p.M - 1) * p.ldc + p.N) return SGEMM_ERR_INVALID_ARG;  // C items would overlap
    const int64_t a_rows = p.transA ? p.K : p.M, a_cols = p.transA ? p.M : p.K;
    const int64_t b_rows = p.transB ? p.N : p.K, b_cols = p.transB ? p.K : p.N;
    const int64_t c_span = (p.batch - 1) * p.strideC + (p.M - 1) * p.ldc + p.N;
    if (p.K > 0) {
        const int64_t a_span = (p.batch - 1) * p.strideA + (a_rows - 1) * p.lda + a_cols;
        const int64_t b_span = (p.batch - 1) * p.strideB + (b_rows - 1) * p.ldb + b_cols;
        if (overlaps(p.C, 1, c_span, c_span, p.A, 1, a_span, a_span) ||
            overlaps(p.C, 1, c_span, c_span, p.B, 1, b_span, b_span))
            return SGEMM_ERR_INVALID_ARG;
    }
    return SGEMM_OK;
}

int enqueue(const Problem &p, cudaStream_t stream) {
    read_env();
    DeviceInfo dev;
    int rc = current_device(&dev);
    if (rc != SGEMM_OK) return rc;
    int launches = 0;
    if (p.M == 0 || p.N == 0 || p.batch == 0) {
        g_last_launches.store(0);
        return SGEMM_OK;
    }
    if (p.K == 0 || p.alpha == 0.0f) {
        // The empty sum (or alpha = 0): C = act(beta * C + bias).
        rc = scale_launch(p, dev, stream, &launches);
        if (rc == SGEMM_OK) {
            g_last_variant.store(SGEMM_FFMA);
            g_last_launches.store(launches);
        }
        return rc;
    }
    int variant = g_variant.load();
    if (variant == SGEMM_AUTO) variant = auto_variant(p, dev);
    if (variant == SGEMM_TF32X3) {
        if (!tf32x3_supports(p, dev)) return SGEMM_ERR_UNSUPPORTED;
        rc = tf32x3_launch(p, dev, static_cast<int>(g_tune_sk.load()), stream, &launches);
    } else {
        rc = ffma_launch(p, dev, static_cast<int>(g_tune_tile.load()), static_cast<int>(g_tune_sk.load()),
                         stream, &launches);
    }
    if (rc == SGEMM_OK) {
        g_last_variant.store(variant);
        g_last_launches.store(launches);
    }
    return rc;
}

// sgemm_f32_noalloc's fixed scratch: one buffer per device (the copies of
// operands whose rows TMA cannot address), looked up once per device.
static __device__ __align__(256) float g_noalloc_scratch[SGEMM_NOALLOC_SCRATCH_BYTES / sizeof(float)];

struct NoallocSlot {
    std::once_flag once;
    float *ptr = nullptr;
};
NoallocSlot g_noalloc[kMaxDevices];

// The device address of the fixed buffer on the current device, or nullptr.
float *noalloc_scratch(int device) {
    std::call_once(g_noalloc[device].once, [device] {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess) {
            cudaGetLastError();
            return;
        }
        g_noalloc[device].ptr = static_cast<float *>(ptr);
    });
    return g_noalloc[device].ptr;
}

// enqueue() with the fixed buffer in place of pool memory; SGEMM_ERR_SCRATCH
// when the copies do not fit (nothing enqueued).
int enqueue_noalloc(const Problem &p, cudaStream_t stream) {
    read_env();
    DeviceInfo dev;
    int rc = current_device(&dev);
    if (rc != SGEMM_OK) return rc;
    int launches = 0;
    if (p.M == 0 || p.N == 0 || p.batch == 0) {
        g_last_launches.store(0);
        return SGEMM_OK;
    }
    if (p.K == 0 || p.alpha == 0.0f) {
        rc = scale_launch(p, dev, stream, &launches);
        if (rc == SGEMM_OK) {
            g_last_variant.store(SGEMM_FFMA);
            g_last_launches.store(launches);
        }
        return rc;
    }
    int variant = g_variant.load();
    if (variant == SGEMM_AUTO) variant = auto_variant(p, dev);
    if (variant == SGEMM_TF32X3) {
        if (!tf32x3_supports(p, dev)) return SGEMM_ERR_UNSUPPORTED;
        const size_t bytes = tf32x3_copy_bytes(p);
        float *scratch = nullptr;
        if (bytes > 0) {
            if (bytes > SGEMM_NOALLOC_SCRATCH_BYTES) return SGEMM_ERR_SCRATCH;
            scratch = noalloc_scratch(dev.device);
            if (!scratch) return SGEMM_ERR_DEVICE;
        }
        rc = tf32x3_launch_with_scratch(p, dev, static_cast<int>(g_tune_sk.load()), stream, &launches, scratch,
                                        scratch ? SGEMM_NOALLOC_SCRATCH_BYTES : 0);
    } else {
        rc = ffma_launch(p, dev, static_cast<int>(g_tune_tile.load()), static_cast<int>(g_tune_sk.load()),
                         stream, &launches);
    }
    if (rc == SGEMM_OK) {
        g_last_variant.store(variant);
        g_last_launches.store(launches);
    }
    return rc;
}

}  // namespace

int current_device(DeviceInfo *info) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return SGEMM_ERR_DEVICE;
    }
    std::call_once(g_dev.once[dev], [dev] {
        DeviceInfo d{};
        d.device = dev;
        int optin = 0;
        bool ok = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
                  cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) == cudaSuccess &&
                  cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) == cudaSuccess &&
                  cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) == cudaSuccess;
        d.smem_optin = static_cast<size_t>(optin);
        g_dev.info[dev] = d;
        if (!ok) {
            cudaGetLastError();
            g_dev.status[dev] = SGEMM_ERR_DEVICE;
        } else {
            // The kernels are built for sm_103a only.
            g_dev.status[dev] = (d.cc_major == 10 && d.cc_minor == 3) ? SGEMM_OK : SGEMM_ERR_DEVICE;
        }
    });
    *info = g_dev.info[dev];
    return g_dev.status[dev];
}

}  // namespace sgemm

using sgemm::Problem;

extern "C" {

int sgemm_f32(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda, const float *B, int64_t ldb,
              float *C, int64_t ldc, sgemm_stream_t stream) {
    int rc = sgemm::check_args(SGEMM_OP_N, SGEMM_OP_N, M, N, K, A, lda, B, ldb, C, ldc);
    if (rc != SGEMM_OK) return rc;
    Problem p{M, N, K, A, lda, B, ldb, C, ldc};
    return sgemm::enqueue(p, reinterpret_cast<cudaStream_t>(stream));
}

int sgemm_f32_noalloc(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda, const float *B, int64_t ldb,
                      float *C, int64_t ldc, sgemm_stream_t stream) {
    int rc = sgemm::check_args(SGEMM_OP_N, SGEMM_OP_N, M, N, K, A, lda, B, ldb, C, ldc);
    if (rc != SGEMM_OK) return rc;
    Problem p{M, N, K, A, lda, B, ldb, C, ldc};
    return sgemm::enqueue_noalloc(p, reinterpret_cast<cudaStream_t>(stream));
}

int sgemm_f32_ex(int transA, int transB, int64_t M, int64_t N, int64_t K, float alpha, const float *A,
                 int64_t lda, const float *B, int64_t ldb, float beta, float *C, int64_t ldc,
                 sgemm_stream_t stream) {
    int rc = sgemm::check_args(transA, transB, M, N, K, A, lda, B, ldb, C, ldc);
    if (rc != SGEMM_OK) return rc;
    Problem p{M, N, K, A, lda, B, ldb, C, ldc};
    p.transA = transA;
    p.transB = transB;
    p.alpha = alpha;
    p.beta = beta;
    return sgemm::enqueue(p, reinterpret_cast<cudaStream_t>(stream));
}

int sgemm_f32_fused(int transA, int transB, int64_t M, int64_t N, int64_t K, float alpha, const float *A,
                    int64_t lda, const float *B, int64_t ldb, float beta, float *C, int64_t ldc,
                    const float *bias, int bias_kind, int activation, sgemm_stream_t stream) {
    int rc = sgemm::check_args(transA, transB, M, N, K, A, lda, B, ldb, C, ldc);
    if (rc != SGEMM_OK) return rc;
    rc = sgemm::check_epilogue(M, N, C, ldc, bias, bias_kind, activation);
    if (rc != SGEMM_OK) return rc;
    Problem p{M, N, K, A, lda, B, ldb, C, ldc};
    p.transA = transA;
    p.transB = transB;
    p.alpha = alpha;
    p.beta = beta;
    p.bias = bias_kind == SGEMM_BIAS_NONE ? nullptr : bias;
    p.bias_kind = bias_kind;
    p.act = activation;
    return sgemm::enqueue(p, reinterpret_cast<cudaStream_t>(stream));
}

// rows x cols of a matrix with row stride ld: one linear copy when the rows
// are contiguous, else a strided copy that leaves the row padding untouched.
static cudaError_t copy_rows(float *dst, const float *src, int64_t rows, int64_t cols, int64_t ld,
                             cudaMemcpyKind kind, cudaStream_t s) {
    const size_t f = sizeof(float);
    if (ld == cols || rows == 1)
        return cudaMemcpyAsync(dst, src, static_cast<size_t>(rows * cols) * f, kind, s);
    return cudaMemcpy2DAsync(dst, ld * f, src, ld * f, cols * f, rows, kind, s);
}

int sgemm_f32_batched(int transA, int transB, int64_t M, int64_t N, int64_t K, float alpha, const float *A,
                      int64_t lda, int64_t strideA, const float *B, int64_t ldb, int64_t strideB, float beta,
                      float *C, int64_t ldc, int64_t strideC, int64_t batch, sgemm_stream_t stream) {
    int rc = sgemm::check_args(transA, transB, M, N, K, A, lda, B, ldb, C, ldc);
    if (rc != SGEMM_OK) return rc;
    Problem p{M, N, K, A, lda, B, ldb, C, ldc};
    p.transA = transA;
    p.transB = transB;
    p.alpha = alpha;
    p.beta = beta;
    p.batch = batch;
    p.strideA = strideA;
    p.strideB = strideB;
    p.strideC = strideC;
    rc = sgemm::check_batch(p);
    if (rc != SGEMM_OK) return rc;
    return sgemm::enqueue(p, reinterpret_cast<cudaStream_t>(stream));
}

namespace sgemm {
namespace {

// Streams and events of the pipelined host-buffer product, made once per
// device on first use and kept for the process; `lock` serialises the
// enqueueing of pipelined calls on one device (the events are re-recorded
// by every call).
constexpr int kMaxPanels = 8;
struct HostPipe {
    std::once_flag once;
    int status = SGEMM_ERR_LAUNCH;
    cudaStream_t compute = nullptr, d2h = nullptr;
    cudaEvent_t fork = nullptr, done = nullptr, b_in[kMaxPanels] = {}, c_out[kMaxPanels] = {};
    std::mutex lock;
};
HostPipe g_pipe[kMaxDevices];

HostPipe *host_pipe(int device) {
    HostPipe &hp = g_pipe[device];
    std::call_once(hp.once, [&hp] {
        const unsigned f = cudaEventDisableTiming;
        bool ok = cudaStreamCreateWithFlags(&hp.compute, cudaStreamNonBlocking) == cudaSuccess &&
                  cudaStreamCreateWithFlags(&hp.d2h, cudaStreamNonBlocking) == cudaSuccess &&
                  cudaEventCreateWithFlags(&hp.fork, f) == cudaSuccess &&
                  cudaEventCreateWithFlags(&hp.done, f) == cudaSuccess;
        for (int j = 0; ok && j < kMaxPanels; ++j)
            ok = cudaEventCreateWithFlags(&hp.b_in[j], f) == cudaSuccess &&
                 cudaEventCreateWithFlags(&hp.c_out[j], f) == cudaSuccess;
        if (!ok) cudaGetLastError();
        hp.status = ok ? SGEMM_OK : SGEMM_ERR_LAUNCH;
    });
    return hp.status == SGEMM_OK ? &hp : nullptr;
}

// Column panels of the pipelined host-buffer product: their widths in
// `widths`, their count returned; 0 for one product without panels. Panels
// pay only when the copies are long enough to hide a panel's product behind
// the next panel's copy.
int panel_plan(int64_t M, int64_t N, int64_t K, int64_t (&widths)[kMaxPanels]) {
    const double work = static_cast<double>(M) * static_cast<double>(N) * static_cast<double>(K);
    if (N < 512 || work < 1073741824.0) return 0;
    const int64_t w = ((N + kMaxPanels - 1) / kMaxPanels + 255) / 256 * 256;  // 256-column multiples
    if (w >= N) return 0;
    int n = 0;
    for (int64_t c0 = 0; c0 < N; c0 += w) widths[n++] = (N - c0 < w) ? N - c0 : w;
    return n;
}

}  // namespace
}  // namespace sgemm

int sgemm_f32_from_host(int64_t M, int64_t N, int64_t K, const float *A_host, int64_t lda,
                        const float *B_host, int64_t ldb, float *C_host, int64_t ldc, float *dA, float *dB,
                        float *dC, sgemm_stream_t stream) {
    int rc = sgemm::check_args(SGEMM_OP_N, SGEMM_OP_N, M, N, K, dA, lda, dB, ldb, dC, ldc);
    if (rc != SGEMM_OK) return rc;
    if ((M > 0 && K > 0 && !A_host) || (K > 0 && N > 0 && !B_host) || (M > 0 && N > 0 && !C_host))
        return SGEMM_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int64_t widths[sgemm::kMaxPanels];
    const int panels = (M > 0 && K > 0) ? sgemm::panel_plan(M, N, K, widths) : 0;
    int device = -1;
    sgemm::HostPipe *hp = nullptr;
    if (panels > 0 && cudaGetDevice(&device) == cudaSuccess && device >= 0 && device < sgemm::kMaxDevices)
        hp = sgemm::host_pipe(device);
    cudaGetLastError();
    if (!hp) {
        // One product: copies in, product, copy out, all in order on `stream`.
        if (M > 0 && K > 0 && copy_rows(dA, A_host, M, K, lda, cudaMemcpyHostToDevice, s) != cudaSuccess)
            return cudaGetLastError(), SGEMM_ERR_LAUNCH;
        if (K > 0 && N > 0 && copy_rows(dB, B_host, K, N, ldb, cudaMemcpyHostToDevice, s) != cudaSuccess)
            return cudaGetLastError(), SGEMM_ERR_LAUNCH;
        Problem p{M, N, K, dA, lda, dB, ldb, dC, ldc};
        rc = sgemm::enqueue(p, s);
        if (rc != SGEMM_OK) return rc;
        if (M > 0 && N > 0 && copy_rows(C_host, dC, M, N, ldc, cudaMemcpyDeviceToHost, s) != cudaSuccess)
            return cudaGetLastError(), SGEMM_ERR_LAUNCH;
        return SGEMM_OK;
    }
    // Column panels: A, then B panel by panel in on `stream`; panel j's
    // product on the compute stream once its B panel is in; its C panel out
    // on the copy-out stream once the product is done. `stream` waits for the
    // last copy out, so the call keeps the one-stream semantics.
    std::lock_guard<std::mutex> guard(hp->lock);
    const size_t f = sizeof(float);
    // On a failure after the fork, `stream` still waits for what the two
    // library streams hold (best effort), so that, as on success, the
    // buffers are free for reuse once `stream` has been synchronised.
    auto fail = [&](int code = SGEMM_ERR_LAUNCH) {
        cudaGetLastError();
        if (cudaEventRecord(hp->fork, hp->compute) == cudaSuccess) cudaStreamWaitEvent(s, hp->fork, 0);
        if (cudaEventRecord(hp->done, hp->d2h) == cudaSuccess) cudaStreamWaitEvent(s, hp->done, 0);
        cudaGetLastError();
        return code;
    };
    if (cudaEventRecord(hp->fork, s) != cudaSuccess || cudaStreamWaitEvent(hp->compute, hp->fork, 0) != cudaSuccess ||
        cudaStreamWaitEvent(hp->d2h, hp->fork, 0) != cudaSuccess)
        return fail();
    if (copy_rows(dA, A_host, M, K, lda, cudaMemcpyHostToDevice, s) != cudaSuccess) return fail();
    int64_t c0 = 0;
    for (int j = 0; j < panels; c0 += widths[j], ++j) {
        const int64_t wj = widths[j];
        if (cudaMemcpy2DAsync(dB + c0, ldb * f, B_host + c0, ldb * f, wj * f, K, cudaMemcpyHostToDevice, s) !=
                cudaSuccess ||
            cudaEventRecord(hp->b_in[j], s) != cudaSuccess ||
            cudaStreamWaitEvent(hp->compute, hp->b_in[j], 0) != cudaSuccess)
            return fail();
        Problem p{M, wj, K, dA, lda, dB + c0, ldb, dC + c0, ldc};
        rc = sgemm::enqueue(p, hp->compute);
        if (rc != SGEMM_OK) return fail(rc);
        if (cudaEventRecord(hp->c_out[j], hp->compute) != cudaSuccess ||
            cudaStreamWaitEvent(hp->d2h, hp->c_out[j], 0) != cudaSuccess ||
            cudaMemcpy2DAsync(C_host + c0, ldc * f, dC + c0, ldc * f, wj * f, M, cudaMemcpyDeviceToHost, hp->d2h) !=
                cudaSuccess)
            return fail();
    }
    if (cudaEventRecord(hp->done, hp->d2h) != cudaSuccess || cudaStreamWaitEvent(s, hp->done, 0) != cudaSuccess)
        return fail();
    return SGEMM_OK;
}

int sgemm_set_variant(int variant) {
    sgemm::read_env();
    if (variant < SGEMM_AUTO || variant > SGEMM_TF32X3) return SGEMM_ERR_INVALID_ARG;
    sgemm::g_variant.store(variant);
    return SGEMM_OK;
}

int sgemm_get_variant(void) {
    sgemm::read_env();
    return sgemm::g_variant.load();
}

const char *sgemm_variant_name(int variant) {
    switch (variant) {
        case SGEMM_AUTO: return "auto";
        case SGEMM_FFMA: return "ffma";
        case SGEMM_TF32X3: return "tf32x3";
        default: return "unknown";
    }
}

int sgemm_last_variant_used(void) { return sgemm::g_last_variant.load(); }

int sgemm_last_launch_count(void) { return sgemm::g_last_launches.load(); }

const char *sgemm_strerror(int status) {
    switch (status) {
        case SGEMM_OK: return "success";
        case SGEMM_ERR_INVALID_ARG: return "invalid argument";
        case SGEMM_ERR_UNSUPPORTED: return "variant does not support this shape or alignment";
        case SGEMM_ERR_LAUNCH: return "CUDA launch or copy failed";
        case SGEMM_ERR_DEVICE: return "no usable sm_103a device";
        case SGEMM_ERR_TIMEOUT: return "a kernel gave up a bounded wait";
        case SGEMM_ERR_SCRATCH: return "product needs more scratch than the fixed no-allocation buffer holds";
        default: return "unknown status";
    }
}

int sgemm_device_status(void) {
    if (cudaDeviceSynchronize() != cudaSuccess) {
        cudaGetLastError();
        return SGEMM_ERR_LAUNCH;
    }
    int code = 0;
    if (sgemm::watchdog_read_and_clear(&code) != 0) return SGEMM_ERR_LAUNCH;
    return code ? SGEMM_ERR_TIMEOUT : SGEMM_OK;
}

int sgemm_watchdog_selftest(int64_t wait_ms, sgemm_stream_t stream) {
    if (wait_ms < 1 || wait_ms > 60000) return SGEMM_ERR_INVALID_ARG;
    sgemm::DeviceInfo dev;
    const int rc = sgemm::current_device(&dev);
    if (rc != SGEMM_OK) return rc;
    return sgemm::watchdog_selftest_launch(wait_ms, reinterpret_cast<cudaStream_t>(stream));
}

int sgemm_set_tuning(int key, int64_t value) {
    switch (key) {
        case SGEMM_TUNE_FFMA_TILE:
            if (value < 0 || value > 3) return SGEMM_ERR_INVALID_ARG;
            sgemm::g_tune_tile.store(value);
            return SGEMM_OK;
        case SGEMM_TUNE_STREAM_K:
            if (value < 0 || value > 3) return SGEMM_ERR_INVALID_ARG;
            sgemm::g_tune_sk.store(value);
            return SGEMM_OK;
        case SGEMM_TUNE_WATCHDOG_MS:
            return sgemm::watchdog_set_ms(value);
        case SGEMM_TUNE_TF32X3_KERNEL:
            return sgemm::tf32x3_set_kernel(value);
        default: return SGEMM_ERR_INVALID_ARG;
    }
}

int64_t sgemm_get_tuning(int key) {
    switch (key) {
        case SGEMM_TUNE_FFMA_TILE: return sgemm::g_tune_tile.load();
        case SGEMM_TUNE_STREAM_K: return sgemm::g_tune_sk.load();
        case SGEMM_TUNE_WATCHDOG_MS: return sgemm::watchdog_ms();
        case SGEMM_TUNE_TF32X3_KERNEL: return sgemm::tf32x3_get_kernel();
        case SGEMM_TUNE_LAST_TC_KERNEL: return sgemm::tf32x3_last_kernel();
        default: return -1;
    }
}

const char *sgemm_version(void) { return "0.1.0"; }

}  // extern "C"
