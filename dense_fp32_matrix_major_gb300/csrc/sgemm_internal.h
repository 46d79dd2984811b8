// Internal declarations shared by the translation units of libsgemm_gb300.
// Not installed; the public ABI is include/sgemm.h.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace sgemm {

// One product request after argument checks: C = alpha * op(A) * op(B) +
// beta * C with op(X) = X or X^T (transA / transB); all pointers are device
// pointers, strides are in elements, M, N, K > 0 and alpha != 0. A is stored
// M x K (K x M when transA), B is stored K x N (N x K when transB).
struct Problem {
    int64_t M, N, K;
    const float *A;
    int64_t lda;
    const float *B;
    int64_t ldb;
    float *C;
    int64_t ldc;
    int transA = 0, transB = 0;
    float alpha = 1.0f, beta = 0.0f;
    // Strided batch: item b uses A + b*strideA, B + b*strideB, C + b*strideC.
    int64_t batch = 1, strideA = 0, strideB = 0, strideC = 0;
    // Fused epilogue: C = act(alpha * op(A) op(B) + beta * C + bias), with
    // bias_kind / act the sgemm_bias / sgemm_activation values of sgemm.h
    // (the bias is shared by all items of a batch).
    const float *bias = nullptr;
    int bias_kind = 0, act = 0;
    bool has_epilogue() const { return bias_kind != 0 || act != 0; }
};

// Properties of the current device that the launchers need.
struct DeviceInfo {
    int device;
    int sm_count;
    int cc_major, cc_minor;
    size_t smem_optin;  // max dynamic shared memory per block (opt-in)
};

// Returns 0 and fills `info` for the current device, or an sgemm_status code.
int current_device(DeviceInfo *info);

// Schedules of the FFMA kernel family.
enum FfmaTile { FFMA_TILE_AUTO = 0, FFMA_TILE_128x256 = 1, FFMA_TILE_128x128 = 2, FFMA_TILE_64x64 = 3 };
enum StreamKMode { SK_AUTO = 0, SK_DP_ONLY = 1, SK_HYBRID = 2, SK_ALL = 3 };

// Work split of a persistent grid over a tiles x k_steps iteration space:
// tiles [0, dp_tiles) go whole, round-robin over the CTAs; the rest are split
// along K into sk_iters (tile, k-step) iterations shared evenly by CTAs
// [0, sk_ctas) (stream-K). A split tile's outputs are set to beta * C (plus
// the bias) first and its partial sums added with atomics.
struct Schedule {
    int dp_tiles;
    int sk_ctas;
    int grid;
    int64_t sk_iters;
};

// slots = CTAs that can be resident at once; min_share = fewest k-steps worth
// giving one stream-K CTA; idle_for_split = the fraction of slots a single
// partial wave would leave idle above which splitting every tile along K
// pays for its atomic fix-up (measured per kernel family on GB300: 0.10 for
// FFMA, 0.25 for the tensor-core kernels, whose k-steps are far shorter).
inline Schedule make_schedule(int tiles, int64_t k_steps, int slots, int mode, int64_t min_share,
                              double idle_for_split, bool split_all_for_remainder = false) {
    if (mode == SK_AUTO) {
        const int rem = tiles % slots;
        if (tiles >= slots) {
            const int split = split_all_for_remainder ? SK_ALL : SK_HYBRID;
            mode = (rem != 0 && static_cast<int64_t>(rem) * k_steps >= min_share * slots) ? split : SK_DP_ONLY;
        } else {
            const double idle = 1.0 - static_cast<double>(tiles) / static_cast<double>(slots);
            mode = (idle >= idle_for_split && k_steps >= 2 * min_share) ? SK_ALL : SK_DP_ONLY;
        }
    }
    Schedule s{};
    if (mode == SK_DP_ONLY) {
        s.dp_tiles = tiles;
        s.sk_iters = 0;
        s.sk_ctas = 0;
        s.grid = tiles < slots ? tiles : slots;
        return s;
    }
    s.dp_tiles = (mode == SK_ALL) ? 0 : (tiles / slots) * slots;
    s.sk_iters = static_cast<int64_t>(tiles - s.dp_tiles) * k_steps;
    int64_t ctas = s.sk_iters / min_share;
    if (ctas > slots) ctas = slots;
    if (ctas < 1) ctas = 1;
    s.sk_ctas = static_cast<int>(ctas);
    const int dp_grid = s.dp_tiles < slots ? s.dp_tiles : slots;
    s.grid = dp_grid > s.sk_ctas ? dp_grid : s.sk_ctas;
    return s;
}

// Passes over the tiles that a schedule splits along K: `count` tiles from
// tile `first_tile` of a bm x bn tile grid with tiles_n tiles per row and
// tiles_per_item tiles per batch item. The prepare pass runs before the
// product and sets C = beta * C + bias (C is not read when beta = 0), so the
// product can add its partial sums with atomics; the finish pass runs after
// it and applies the activation (it enqueues nothing when p.act is NONE).
int split_tiles_prepare(const Problem &p, int bm, int bn, int tiles_n, int tiles_per_item, int first_tile,
                        int count, cudaStream_t stream, int *launches);
// after_signal: the product just enqueued executes
// griddepcontrol.launch_dependents, so the finish pass is launched as its
// programmatic dependent (its launch overlaps the product's tail).
int split_tiles_finish(const Problem &p, int bm, int bn, int tiles_n, int tiles_per_item, int first_tile,
                       int count, cudaStream_t stream, int *launches, bool after_signal = false);

// Enqueue the FFMA product. `launches` receives the number of kernels enqueued.
int ffma_launch(const Problem &p, const DeviceInfo &dev, int tile, int sk_mode, cudaStream_t stream,
                int *launches);
// The transposed forms (op(A) = A^T and/or op(B) = B^T).
int ffma_launch_t(const Problem &p, const DeviceInfo &dev, int tile, int sk_mode, cudaStream_t stream,
                  int *launches);

// Enqueue C[0:M, 0:N] = act(beta * C + bias) for every item (C not read
// when beta = 0): the result when K = 0 (the empty sum) or alpha = 0.
int scale_launch(const Problem &p, const DeviceInfo &dev, cudaStream_t stream, int *launches);

// Tensor-core three-term TF32 variant. Returns SGEMM_ERR_UNSUPPORTED when it
// cannot run the request.
bool tf32x3_supports(const Problem &p, const DeviceInfo &dev);
int tf32x3_launch(const Problem &p, const DeviceInfo &dev, int sk_mode, cudaStream_t stream, int *launches);
// The part of tf32x3_launch for operands a tensor map cannot describe. With
// `scratch` (16-byte aligned, scratch_bytes long) the aligned copies go
// there instead of into pool memory; SGEMM_ERR_INVALID_ARG when it is too
// small.
int tf32x3_launch_unaligned(const Problem &p, const DeviceInfo &dev, int sk_mode, cudaStream_t stream,
                            int *launches, float *scratch, size_t scratch_bytes);
// Scratch bytes tf32x3_launch would take from the pool for p (0: none), and
// tf32x3_launch with the caller's scratch buffer in place of the pool.
size_t tf32x3_copy_bytes(const Problem &p);
int tf32x3_launch_with_scratch(const Problem &p, const DeviceInfo &dev, int sk_mode, cudaStream_t stream,
                               int *launches, float *scratch, size_t scratch_bytes);
// The SM-pair kernel (every operand form; cpa: A and B rows not 16-byte
// aligned, loaded with cp.async instead of TMA; after_copy: the last kernel
// enqueued is the aligned copy of A and B, which this launch may overlap).
int tf32x3_pair_launch(const Problem &p, const DeviceInfo &dev, int sk_mode, bool cpa, cudaStream_t stream,
                       int *launches, bool after_copy = false);

// Operands whose rows TMA cannot address (repack.cu). tma_operand_ok: the
// stored matrix X (rows x ld floats per item, items `stride` apart) can be
// described by a tensor map. repack_bytes: scratch needed to copy every
// operand of p that fails that test into rows of a multiple of 4 floats (0
// when none does). repack_into: enqueue those copies on `stream` into
// `scratch` (16-byte aligned, at least repack_bytes(p) bytes) and set *q to
// p with the copied operands in place of the originals; nothing is enqueued
// on error. scratch_alloc / scratch_free: stream-ordered scratch from a pool
// the library keeps per device (nullptr when it cannot allocate).
bool tma_operand_ok(const float *X, int64_t ld, int64_t stride, int64_t rows, int64_t batch);
size_t repack_bytes(const Problem &p);
int repack_into(const Problem &p, const DeviceInfo &dev, float *scratch, size_t bytes, cudaStream_t stream,
                Problem *q, int *launches);
float *scratch_alloc(const DeviceInfo &dev, size_t bytes, cudaStream_t stream);
void scratch_free(float *ptr, cudaStream_t stream);

// Watchdog flag shared by kernels with bounded waits (one per device, in the
// tf32x3 translation unit). Read-and-clear; returns 0 or the first recorded code.
int watchdog_read_and_clear(int *code);
int64_t watchdog_ms();
int watchdog_set_ms(int64_t ms);
// Which tensor-core kernel serves TMA-compatible operands (tuning key
// SGEMM_TUNE_TF32X3_KERNEL).
int tf32x3_set_kernel(int64_t mode);
int watchdog_selftest_launch(int64_t wait_ms, cudaStream_t stream);
int64_t tf32x3_get_kernel();
int64_t tf32x3_last_kernel();  // 1-4: the tensor-core kernel of the last TF32X3 launch
int *watchdog_flag_device_ptr();  // device address of the current device's flag, or nullptr

}  // namespace sgemm
