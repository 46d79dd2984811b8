// Register-blocked fp32 SGEMM on the CUDA cores (FFMA), sm_103a.
//
// Computes C = A * B for row-major fp32 A (M x K), B (K x N), C (M x N): the
// sum of products of "CUDA算子优化(4)：矩阵乘法", section "矩阵乘法的数学定义".
// The pages' tiled kernels ("CUDA内存优化入门：从Naive到Tiled矩阵乘法" section 六,
// and the shared-memory version of "CUDA算子优化(4)：矩阵乘法") stage square
// 16x16 / 32x32 tiles of A and B in shared memory with one output per thread.
// This kernel keeps their two ideas -- stage tiles of A and B on chip and
// reuse them, and fill out-of-range tile elements with zeros so ragged sizes
// need no special case ("CUDA内存优化入门" section 六, "边界检查的重要性") --
// and replaces the rest with a design for a 128-FP32-lane-per-SM part:
//
//   * Block tile BM x BN (128x256, 128x128 or 64x64), k-step BK = 16; each
//     thread owns an 8 x TN register tile (TN = 16 or 8), so one k-step costs
//     a thread 8*TN fused multiply-adds against 2 + TN/4 128-bit shared-memory
//     loads. The multiply-adds are issued as packed fma.rn.f32x2 on pairs of
//     adjacent columns (two IEEE fp32 FMAs each, the same results as fmaf):
//     half the issue slots (measured 48.5 -> 53.3 TFLOP/s at 2048x3072x4096;
//     56.0 with a two-stage ring).
//   * A and B move global -> shared with cp.async through a STAGES-deep ring
//     (one __syncthreads per k-tile; two stages for the 128x256 tile). A is
//     transposed on the way (4-byte copies into As[k][m]) so each thread
//     reads four rows with one 128-bit load; As is XOR-swizzled on 16-byte
//     groups by (k & 7) so the transposing stores spread over the banks. B
//     keeps its layout (16-byte copies when its rows are 16-byte aligned,
//     else 4-byte copies).
//   * Out-of-range elements are copied as zeros (cp.async src-size 0), the
//     store is guarded by row < M and col < N on both sides (the '&&' guard,
//     not the '||' guard that writes out of bounds), and nothing is written
//     between column N and the row stride.
//   * Work is scheduled over a persistent grid: whole tiles round-robin
//     (data-parallel), and the tiles left after the last full wave are split
//     along K across all CTAs (stream-K). A split tile is first scaled by
//     beta (zeroed when beta = 0) by a small kernel and its partial sums,
//     times alpha, are added with fp32 atomics, so the summation order of
//     those outputs varies from run to run (every order stays within the
//     acceptance bound, and integer-exact inputs stay exact).
//   * The general form C = alpha * op(A) * op(B) + beta * C (op = the matrix
//     or its transpose, the standard BLAS form; the pages compute only
//     C = A * B) changes the loads and the epilogue only: a transposed A is
//     copied row for row (16 bytes when aligned), a transposed B is
//     transposed by 4-byte copies into a swizzled Bs; the epilogue writes
//     alpha * acc + beta * C and reads C only when beta != 0.
//   * The fused epilogue (bias, activation; sgemm_f32_fused) is applied in
//     the same store to whole tiles; split tiles get the bias in the beta
//     pre-pass and the activation in a pass after the product.
//
// This file instantiates op(A) = A, op(B) = B and holds the C passes (beta,
// bias, activation) that run outside the product kernels;
// sgemm_ffma_t.cu instantiates the transposed forms.
#include <cuda_runtime.h>
#include <stdint.h>

#include "epilogue.cuh"
#include "ffma_impl.cuh"

namespace sgemm {
namespace {

using namespace ffma;

// C = act(beta * C + bias) over `count` tiles starting at `first_tile` of a
// bm x bn tile grid (C is not read when beta = 0); tiles run item-major over
// a batch whose items are strideC elements apart. blockIdx.x picks the tile
// (up to 2^31 - 1 of them), blockIdx.y a band of 8 rows; a warp handles one
// row (float4 when aligned).
__global__ void tile_pass_kernel(float *C, int64_t M, int64_t N, int64_t ldc, int64_t strideC, float beta,
                                 const float *bias, int bias_kind, int act, int bm, int bn, int tiles_n,
                                 int tiles_per_item, int first_tile) {
    // Launched behind a product (the activation pass) this waits for it; the
    // product launched behind this pass (the beta pre-pass) may start its
    // main loop at once and waits only before it writes C.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    const int tile = first_tile + static_cast<int>(blockIdx.x);
    const int item = tile / tiles_per_item, rest = tile % tiles_per_item;
    C += item * strideC;
    const int64_t m0 = static_cast<int64_t>(rest / tiles_n) * bm;
    const int64_t n0 = static_cast<int64_t>(rest % tiles_n) * bn;
    const int64_t row = m0 + blockIdx.y * 8 + (threadIdx.x >> 5);
    if (row >= M || row >= m0 + bm) return;
    const int cols = static_cast<int>(min64(bn, N - n0));
    float *p = C + row * ldc + n0;
    const int lane = threadIdx.x & 31;
    const bool ep = bias_kind != SGEMM_BIAS_NONE || act != SGEMM_ACT_NONE;
    auto one = [&](float c, int i) {
        const float x = beta != 0.0f ? beta * c : 0.0f;
        return ep ? epilogue_value(x, bias, bias_kind, act, row, n0 + i) : x;
    };
    int done = 0;
    if ((reinterpret_cast<uintptr_t>(p) & 15) == 0) {
        const int v4 = cols >> 2;
        float4 *p4 = reinterpret_cast<float4 *>(p);
        for (int i = lane; i < v4; i += 32) {
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (beta != 0.0f) v = p4[i];
            v.x = one(v.x, 4 * i);
            v.y = one(v.y, 4 * i + 1);
            v.z = one(v.z, 4 * i + 2);
            v.w = one(v.w, 4 * i + 3);
            p4[i] = v;
        }
        done = 4 * v4;
    }
    for (int i = done + lane; i < cols; i += 32) p[i] = one(beta != 0.0f ? p[i] : 0.0f, i);
}

// C[0:M, 0:N] = act(beta * C + bias) (C not read when beta = 0) for every
// item of a batch, with a grid-stride loop.
__global__ void scale_rect_kernel(float *C, int64_t M, int64_t N, int64_t ldc, int64_t strideC, int64_t batch,
                                  float beta, const float *bias, int bias_kind, int act) {
    const int64_t per_item = M * N, total = per_item * batch;
    const bool ep = bias_kind != SGEMM_BIAS_NONE || act != SGEMM_ACT_NONE;
    for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < total;
         e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t item = e / per_item, r = e % per_item;
        const int64_t row = r / N, col = r % N;
        float *p = C + item * strideC + row * ldc + col;
        const float x = beta != 0.0f ? beta * *p : 0.0f;
        *p = ep ? epilogue_value(x, bias, bias_kind, act, row, col) : x;
    }
}

template <class C>
int launch_nn(const Problem &p, const DeviceInfo &dev, int sk_mode, cudaStream_t stream, int *launches) {
    const bool vb = (p.ldb % 4 == 0) && (p.strideB % 4 == 0) && (reinterpret_cast<uintptr_t>(p.B) % 16 == 0);
    const bool vc = (p.ldc % 4 == 0) && (p.strideC % 4 == 0) && (reinterpret_cast<uintptr_t>(p.C) % 16 == 0);
    if (vb && vc) return launch_cfg<C, false, false, true, true>(p, dev, sk_mode, stream, launches);
    if (vb) return launch_cfg<C, false, false, true, false>(p, dev, sk_mode, stream, launches);
    if (vc) return launch_cfg<C, false, false, false, true>(p, dev, sk_mode, stream, launches);
    return launch_cfg<C, false, false, false, false>(p, dev, sk_mode, stream, launches);
}

}  // namespace

int ffma_launch(const Problem &p, const DeviceInfo &dev, int tile, int sk_mode, cudaStream_t stream,
                int *launches) {
    if (p.transA || p.transB) return ffma_launch_t(p, dev, tile, sk_mode, stream, launches);
    switch (pick_tile(p, dev, tile)) {
        case FFMA_TILE_128x256: return launch_nn<CfgBig>(p, dev, sk_mode, stream, launches);
        case FFMA_TILE_128x128: return launch_nn<CfgMid>(p, dev, sk_mode, stream, launches);
        case FFMA_TILE_64x64: return launch_nn<CfgSmall>(p, dev, sk_mode, stream, launches);
        default: return SGEMM_ERR_INVALID_ARG;
    }
}

int split_tiles_prepare(const Problem &p, int bm, int bn, int tiles_n, int tiles_per_item, int first_tile,
                        int count, cudaStream_t stream, int *launches) {
    if (count <= 0) return SGEMM_OK;
    const dim3 grid(static_cast<unsigned>(count), static_cast<unsigned>((bm + 7) / 8));
    tile_pass_kernel<<<grid, 256, 0, stream>>>(p.C, p.M, p.N, p.ldc, p.strideC, p.beta, p.bias, p.bias_kind,
                                                SGEMM_ACT_NONE, bm, bn, tiles_n, tiles_per_item, first_tile);
    ++*launches;
    return cudaGetLastError() == cudaSuccess ? SGEMM_OK : SGEMM_ERR_LAUNCH;
}

int split_tiles_finish(const Problem &p, int bm, int bn, int tiles_n, int tiles_per_item, int first_tile,
                       int count, cudaStream_t stream, int *launches, bool after_signal) {
    if (count <= 0 || p.act == SGEMM_ACT_NONE) return SGEMM_OK;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(count), static_cast<unsigned>((bm + 7) / 8));
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    // Behind a product that signals griddepcontrol.launch_dependents this
    // pass may be scheduled during the product's tail; it waits for the
    // whole product (griddepcontrol.wait) before it touches C.
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = after_signal ? 1 : 0;
    if (cudaLaunchKernelEx(&cfg, tile_pass_kernel, p.C, p.M, p.N, p.ldc, p.strideC, 1.0f,
                           static_cast<const float *>(nullptr), static_cast<int>(SGEMM_BIAS_NONE), p.act, bm, bn,
                           tiles_n, tiles_per_item, first_tile) != cudaSuccess) {
        cudaGetLastError();
        return SGEMM_ERR_LAUNCH;
    }
    ++*launches;
    return SGEMM_OK;
}

int scale_launch(const Problem &p, const DeviceInfo &dev, cudaStream_t stream, int *launches) {
    const int64_t total = p.M * p.N * p.batch;
    const int64_t blocks = min64(ceil_div(total, 256), static_cast<int64_t>(dev.sm_count) * 8);
    scale_rect_kernel<<<static_cast<int>(blocks > 1 ? blocks : 1), 256, 0, stream>>>(
        p.C, p.M, p.N, p.ldc, p.strideC, p.batch, p.beta, p.bias, p.bias_kind, p.act);
    ++*launches;
    return cudaGetLastError() == cudaSuccess ? SGEMM_OK : SGEMM_ERR_LAUNCH;
}

}  // namespace sgemm
