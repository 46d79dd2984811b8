// Register-blocked fp32 FFMA kernel family: the template shared by the
// translation units that instantiate it (sgemm_ffma.cu: op(A) = A,
// op(B) = B; sgemm_ffma_t.cu: the transposed forms). The design notes are at
// the top of sgemm_ffma.cu.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <mutex>

#include "epilogue.cuh"
#include "sgemm.h"
#include "sgemm_internal.h"

namespace sgemm {
namespace ffma {

struct FfmaArgs {
    int64_t M, N, K;
    const float *A;
    int64_t lda;
    const float *B;
    int64_t ldb;
    float *C;
    int64_t ldc;
    float alpha, beta;  // C = alpha * op(A) op(B) + beta * C; beta == 0: C not read
    int64_t strideA, strideB, strideC;  // elements between the items of a batch
    int tiles_per_item;                 // tiles of one product (tiles run item-major)
    int vec_a;          // op(A) = A^T and its rows allow 16-byte copies
    int vec_c;          // C rows allow 16-byte stores (used when VEC_C is not set)
    int tiles_n;        // tiles along N (tiles are numbered row-major over the tile grid)
    int k_tiles;        // ceil(K / BK)
    int dp_tiles;       // tiles [0, dp_tiles) go round-robin to CTAs, whole
    int total_tiles;    // tiles [dp_tiles, total_tiles) are split along K
    int64_t sk_iters;   // (total_tiles - dp_tiles) * k_tiles
    int sk_ctas;        // CTAs [0, sk_ctas) share the split iterations evenly
    const float *bias;  // fused epilogue: C = act(... + bias) on whole tiles
    int bias_kind, act;
    int ep;             // bias_kind or act set
};

template <int WARPS_M_, int WARPS_N_, int CN_, int STAGES_, int MIN_BLOCKS_, int KU_>
struct Cfg {
    static constexpr int WARPS_M = WARPS_M_, WARPS_N = WARPS_N_, CN = CN_, STAGES = STAGES_;
    static constexpr int KU = KU_;  // k-steps unrolled per pass of the inner loop (8 or 16)
    static constexpr int MIN_BLOCKS = MIN_BLOCKS_;  // resident CTAs per SM the registers must allow
    static constexpr int BK = 16;
    static constexpr int THREADS = 32 * WARPS_M * WARPS_N;
    static constexpr int WM = 64;       // warp tile rows: 8 lanes x 2 groups x 4 rows
    static constexpr int WN = 16 * CN;  // warp tile cols: 4 lanes x CN chunks x 4 cols
    static constexpr int BM = WM * WARPS_M;
    static constexpr int BN = WN * WARPS_N;
    static constexpr int TN = 4 * CN;
    static constexpr int A_STAGE = BK * BM;  // floats
    static constexpr int B_STAGE = BK * BN;
    static constexpr int SMEM_BYTES = STAGES * (A_STAGE + B_STAGE) * 4;
    static constexpr int A_PER_THREAD = BM * BK / THREADS;
    static constexpr int A4_PER_THREAD = BM * BK / 4 / THREADS;
    static constexpr int B_PER_THREAD = BK * BN / THREADS;
    static constexpr int B4_PER_THREAD = BK * BN / 4 / THREADS;
    static_assert(BM * BK / 4 % THREADS == 0, "A tile must split evenly over threads");
    static_assert(BK * BN / 4 % THREADS == 0, "B tile must split evenly over threads");
};

// 128 x 256, 256 threads, 8 x 16 per thread, two stages: measured on GB300
// at 2048 x 3072 x 4096 (L2 flushed), 2 / 3 / 4 / 5 stages gave 56.0 / 55.6 /
// 53.2 / 54.6 TFLOP/s (a smaller shared-memory carve-out leaves more L1).
using CfgBig = Cfg<2, 4, 4, 2, 1, 16>;
using CfgMid = Cfg<2, 4, 2, 4, 2, 16>;    // 128 x 128, 256 threads, 8 x 8 per thread
using CfgSmall = Cfg<1, 2, 2, 3, 6, 16>;  // 64 x 64, 64 threads, 8 x 8 per thread

__host__ __device__ __forceinline__ int64_t min64(int64_t x, int64_t y) { return x < y ? x : y; }

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 4-byte asynchronous copy; src_bytes 0 writes a zero.
__device__ __forceinline__ void cp_async_4(uint32_t dst, const float *src, int src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes)
                 : "memory");
}

// 16-byte asynchronous copy of src_bytes (0..16) bytes; the rest is zero-filled.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const float *src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }

template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// Position of op(A) element (m, k) in one stage of As: k-major rows of BM,
// 16-byte groups XOR-swizzled by (k & 7) so the transposing 4-byte copies
// spread over the banks and 4 consecutive m stay one aligned float4.
template <class C>
__device__ __forceinline__ int as_index(int k, int m) {
    return k * C::BM + (m ^ ((k & 7) << 2));
}

// Position of op(B) element (k, n) in one stage of Bs: k-major rows of BN,
// swizzled the same way when op(B) = B^T (the copies transpose).
template <class C, bool TB>
__device__ __forceinline__ int bs_index(int k, int n) {
    return k * C::BN + (TB ? (n ^ ((k & 7) << 2)) : n);
}

template <class C, bool TA, bool TB, bool VEC_B>
__device__ __forceinline__ void load_stage(const FfmaArgs &a, const float *__restrict__ Ab,
                                           const float *__restrict__ Bb, float *As, float *Bs, int64_t m0,
                                           int64_t n0, int64_t k0, int tid) {
    constexpr int BK = C::BK;
    if constexpr (!TA) {
        // A is M x K: 4 consecutive threads read one row along k; copies transpose.
#pragma unroll
        for (int r = 0; r < C::A_PER_THREAD; ++r) {
            const int e = r * C::THREADS + tid;
            const int m = e / BK, k = e % BK;
            const int64_t gm = m0 + m, gk = k0 + k;
            const bool ok = gm < a.M && gk < a.K;
            const float *src = ok ? Ab + gm * a.lda + gk : Ab;
            cp_async_4(smem_addr(As + as_index<C>(k, m)), src, ok ? 4 : 0);
        }
    } else if (a.vec_a) {
        // A is stored K x M: rows of As come straight from rows of A, 16 bytes at a time.
#pragma unroll
        for (int r = 0; r < C::A4_PER_THREAD; ++r) {
            const int e = r * C::THREADS + tid;
            const int k = e / (C::BM / 4), m = (e % (C::BM / 4)) * 4;
            const int64_t gk = k0 + k, gm = m0 + m;
            int bytes = 0;
            if (gk < a.K && gm < a.M) bytes = static_cast<int>(min64(4, a.M - gm)) * 4;
            const float *src = bytes ? Ab + gk * a.lda + gm : Ab;
            cp_async_16(smem_addr(As + as_index<C>(k, m)), src, bytes);
        }
    } else {
#pragma unroll
        for (int r = 0; r < C::A_PER_THREAD; ++r) {
            const int e = r * C::THREADS + tid;
            const int k = e / C::BM, m = e % C::BM;
            const int64_t gk = k0 + k, gm = m0 + m;
            const bool ok = gk < a.K && gm < a.M;
            const float *src = ok ? Ab + gk * a.lda + gm : Ab;
            cp_async_4(smem_addr(As + as_index<C>(k, m)), src, ok ? 4 : 0);
        }
    }
    if constexpr (TB) {
        // B is stored N x K: consecutive threads read along k; copies transpose.
#pragma unroll
        for (int r = 0; r < C::B_PER_THREAD; ++r) {
            const int e = r * C::THREADS + tid;
            const int n = e / BK, k = e % BK;
            const int64_t gn = n0 + n, gk = k0 + k;
            const bool ok = gk < a.K && gn < a.N;
            const float *src = ok ? Bb + gn * a.ldb + gk : Bb;
            cp_async_4(smem_addr(Bs + bs_index<C, TB>(k, n)), src, ok ? 4 : 0);
        }
    } else if constexpr (VEC_B) {
#pragma unroll
        for (int r = 0; r < C::B4_PER_THREAD; ++r) {
            const int e = r * C::THREADS + tid;
            const int k = e / (C::BN / 4), n = (e % (C::BN / 4)) * 4;
            const int64_t gk = k0 + k, gn = n0 + n;
            int bytes = 0;
            if (gk < a.K && gn < a.N) bytes = static_cast<int>(min64(4, a.N - gn)) * 4;
            const float *src = bytes ? Bb + gk * a.ldb + gn : Bb;
            cp_async_16(smem_addr(Bs + bs_index<C, TB>(k, n)), src, bytes);
        }
    } else {
#pragma unroll
        for (int r = 0; r < C::B_PER_THREAD; ++r) {
            const int e = r * C::THREADS + tid;
            const int k = e / C::BN, n = e % C::BN;
            const int64_t gk = k0 + k, gn = n0 + n;
            const bool ok = gk < a.K && gn < a.N;
            const float *src = ok ? Bb + gk * a.ldb + gn : Bb;
            cp_async_4(smem_addr(Bs + bs_index<C, TB>(k, n)), src, ok ? 4 : 0);
        }
    }
}

// One tile over k-tiles [kb, ke). atomic: add alpha * the partial sum into C
// (C was set to beta * C + bias beforehand; the activation comes after the
// product) instead of storing. Otherwise the store applies the whole
// epilogue: act(alpha * acc + beta * C + bias).
template <class C, bool TA, bool TB, bool VEC_B, bool VEC_C>
__device__ __forceinline__ void process_tile(const FfmaArgs &a, float *As, float *Bs, int tile, int kb,
                                             int ke, bool atomic) {
    constexpr int BK = C::BK, S = C::STAGES, TN = C::TN;
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int wm0 = (warp / C::WARPS_N) * C::WM;
    const int wn0 = (warp % C::WARPS_N) * C::WN;
    const int tm = lane >> 2, tn = lane & 3;
    const int item = tile / a.tiles_per_item, rest = tile % a.tiles_per_item;
    const int64_t m0 = static_cast<int64_t>(rest / a.tiles_n) * C::BM;
    const int64_t n0 = static_cast<int64_t>(rest % a.tiles_n) * C::BN;
    const float *Ab = a.A + item * a.strideA;
    const float *Bb = a.B + item * a.strideB;
    float *Cb = a.C + item * a.strideC;
    const int nk = ke - kb;

    // Accumulators in pairs of adjacent columns: each update is one packed
    // fma.rn.f32x2 (two fp32 fused multiply-adds, each rounded to nearest as
    // fmaf would), half the issue slots of scalar FFMAs.
    unsigned long long acc2[8][TN / 2];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < TN / 2; ++j) acc2[i][j] = 0ull;

    __syncthreads();  // the previous tile of this CTA is done with the ring
#pragma unroll
    for (int s = 0; s < S - 1; ++s) {
        if (s < nk)
            load_stage<C, TA, TB, VEC_B>(a, Ab, Bb, As + s * C::A_STAGE, Bs + s * C::B_STAGE, m0, n0,
                                         static_cast<int64_t>(kb + s) * BK, tid);
        cp_async_commit();
    }

    for (int t = 0; t < nk; ++t) {
        cp_async_wait<S - 2>();
        __syncthreads();
        {
            const int tl = t + S - 1;
            if (tl < nk) {
                const int sl = tl % S;
                load_stage<C, TA, TB, VEC_B>(a, Ab, Bb, As + sl * C::A_STAGE, Bs + sl * C::B_STAGE, m0, n0,
                                             static_cast<int64_t>(kb + tl) * BK, tid);
            }
            cp_async_commit();
        }
        const float *as = As + (t % S) * C::A_STAGE;
        const float *bs = Bs + (t % S) * C::B_STAGE;
        // Rolled passes of KU unrolled k-steps (KU = BK: one pass; with scalar
        // FFMAs the 8 x 16 register tile's full unroll overflowed the
        // instruction cache, with packed ones it fits); the swizzle term
        // ((k8 + kk) & 7 = kk & 7) stays a compile-time constant.
#pragma unroll 1
        for (int k8 = 0; k8 < BK; k8 += C::KU)
#pragma unroll
        for (int kk = 0; kk < C::KU; ++kk) {
            float av[8], bv[TN];
#pragma unroll
            for (int g = 0; g < 2; ++g) {
                const float4 v = *reinterpret_cast<const float4 *>(
                    as + (k8 + kk) * C::BM + ((wm0 + g * 32 + tm * 4) ^ ((kk & 7) << 2)));
                av[g * 4 + 0] = v.x;
                av[g * 4 + 1] = v.y;
                av[g * 4 + 2] = v.z;
                av[g * 4 + 3] = v.w;
            }
#pragma unroll
            for (int c = 0; c < C::CN; ++c) {
                const int n = wn0 + c * 16 + tn * 4;
                const float4 v = *reinterpret_cast<const float4 *>(
                    bs + (k8 + kk) * C::BN + (TB ? (n ^ ((kk & 7) << 2)) : n));
                bv[c * 4 + 0] = v.x;
                bv[c * 4 + 1] = v.y;
                bv[c * 4 + 2] = v.z;
                bv[c * 4 + 3] = v.w;
            }
            unsigned long long b2[TN / 2];
#pragma unroll
            for (int j = 0; j < TN / 2; ++j)
                asm("mov.b64 %0, {%1, %2};" : "=l"(b2[j]) : "f"(bv[2 * j]), "f"(bv[2 * j + 1]));
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                unsigned long long a2;  // av[i] in both halves
                asm("mov.b64 %0, {%1, %1};" : "=l"(a2) : "f"(av[i]));
#pragma unroll
                for (int j = 0; j < TN / 2; ++j)
                    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc2[i][j]) : "l"(a2), "l"(b2[j]));
            }
        }
    }
    cp_async_wait<0>();
    float acc[8][TN];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < TN / 2; ++j)
            asm("mov.b64 {%0, %1}, %2;" : "=f"(acc[i][2 * j]), "=f"(acc[i][2 * j + 1]) : "l"(acc2[i][j]));

    // Epilogue: rows wm0 + g*32 + tm*4 + r, columns wn0 + c*16 + tn*4 + q.
    // Everything the stores need, read from the parameters before the first
    // store (a store through a generic pointer would force re-reads).
    const float alpha = a.alpha, beta = a.beta;
    const bool vec_c = VEC_C || a.vec_c;
    const int64_t M = a.M, N = a.N, ldc = a.ldc;
    const float *bias = a.bias;
    const int bias_kind = a.bias_kind, act = a.act;
    const bool ep = a.ep;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int64_t row = m0 + wm0 + (i >> 2) * 32 + tm * 4 + (i & 3);
        if (row >= M) continue;
        float *crow = Cb + row * ldc;
#pragma unroll
        for (int c = 0; c < C::CN; ++c) {
            const int64_t col = n0 + wn0 + c * 16 + tn * 4;
            if (col >= N) continue;
            float v[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) v[q] = alpha * acc[i][c * 4 + q];
            if (atomic) {
                if (vec_c && col + 3 < N) {
                    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(crow + col), "f"(v[0]),
                                 "f"(v[1]), "f"(v[2]), "f"(v[3])
                                 : "memory");
                } else {
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        if (col + q < N) atomicAdd(crow + col + q, v[q]);
                }
            } else if (vec_c && col + 3 < N) {
                float4 *p = reinterpret_cast<float4 *>(crow + col);
                if (beta != 0.0f) {
                    const float4 o = *p;
                    v[0] = fmaf(beta, o.x, v[0]);
                    v[1] = fmaf(beta, o.y, v[1]);
                    v[2] = fmaf(beta, o.z, v[2]);
                    v[3] = fmaf(beta, o.w, v[3]);
                }
                if (ep) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) v[q] = epilogue_value(v[q], bias, bias_kind, act, row, col + q);
                }
                *p = make_float4(v[0], v[1], v[2], v[3]);
            } else {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    if (col + q >= N) continue;
                    float x = v[q];
                    if (beta != 0.0f) x = fmaf(beta, crow[col + q], x);
                    if (ep) x = epilogue_value(x, bias, bias_kind, act, row, col + q);
                    crow[col + q] = x;
                }
            }
        }
    }
}

template <class C, bool TA, bool TB, bool VEC_B, bool VEC_C>
__global__ void __launch_bounds__(C::THREADS, C::MIN_BLOCKS) ffma_kernel(const FfmaArgs a) {
    extern __shared__ float4 smem_f4[];
    float *As = reinterpret_cast<float *>(smem_f4);
    float *Bs = As + C::STAGES * C::A_STAGE;

    for (int t = blockIdx.x; t < a.dp_tiles; t += gridDim.x)
        process_tile<C, TA, TB, VEC_B, VEC_C>(a, As, Bs, t, 0, a.k_tiles, false);

    if (static_cast<int>(blockIdx.x) < a.sk_ctas) {
        int64_t it = a.sk_iters * blockIdx.x / a.sk_ctas;
        const int64_t end = a.sk_iters * (blockIdx.x + 1) / a.sk_ctas;
        while (it < end) {
            const int tile = a.dp_tiles + static_cast<int>(it / a.k_tiles);
            const int kb = static_cast<int>(it % a.k_tiles);
            const int ke = static_cast<int>(min64(a.k_tiles, kb + (end - it)));
            // Stream-K tiles were scaled by beta beforehand: every unit adds,
            // also one that happens to cover the whole K range.
            process_tile<C, TA, TB, VEC_B, VEC_C>(a, As, Bs, tile, kb, ke, true);
            it += ke - kb;
        }
    }
}

// ------------------------------------------------------------------ host side

constexpr int kMaxDevices = 64;

struct KernelSlot {
    std::once_flag once[kMaxDevices];
    int ctas_per_sm[kMaxDevices];
    cudaError_t err[kMaxDevices];
};

template <class C, bool TA, bool TB, bool VEC_B, bool VEC_C>
KernelSlot &slot() {
    static KernelSlot s;
    return s;
}

template <class C, bool TA, bool TB, bool VEC_B, bool VEC_C>
int occupancy(const DeviceInfo &dev, int *ctas_per_sm) {
    if (dev.device < 0 || dev.device >= kMaxDevices) return SGEMM_ERR_DEVICE;
    KernelSlot &s = slot<C, TA, TB, VEC_B, VEC_C>();
    std::call_once(s.once[dev.device], [&] {
        auto fn = ffma_kernel<C, TA, TB, VEC_B, VEC_C>;
        cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
        int n = 0;
        if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, C::THREADS, C::SMEM_BYTES);
        s.err[dev.device] = e;
        s.ctas_per_sm[dev.device] = n;
    });
    if (s.err[dev.device] != cudaSuccess || s.ctas_per_sm[dev.device] < 1) {
        cudaGetLastError();
        return SGEMM_ERR_LAUNCH;
    }
    *ctas_per_sm = s.ctas_per_sm[dev.device];
    return SGEMM_OK;
}

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

template <class C, bool TA, bool TB, bool VEC_B, bool VEC_C>
int launch_cfg(const Problem &p, const DeviceInfo &dev, int sk_mode, cudaStream_t stream, int *launches) {
    int per_sm = 0;
    int rc = occupancy<C, TA, TB, VEC_B, VEC_C>(dev, &per_sm);
    if (rc != SGEMM_OK) return rc;

    const int64_t tiles_m = ceil_div(p.M, C::BM), tiles_n = ceil_div(p.N, C::BN);
    const int64_t tiles64 = tiles_m * tiles_n * p.batch;
    const int64_t k_tiles = ceil_div(p.K, C::BK);
    if (tiles64 > INT32_MAX / 2 || k_tiles > INT32_MAX / 2) return SGEMM_ERR_UNSUPPORTED;
    const int tiles = static_cast<int>(tiles64);
    const int slots = dev.sm_count * per_sm;
    // A stream-K share below this many k-steps costs more in fix-up than it saves.
    // A partial last wave: every tile split along K (stream-K over all) beats
    // whole tiles plus a split remainder here (measured on GB300, 128 x 256
    // tiles, L2 flushed: 2048 x 3072 x 4096 887.7 vs 920.6 us, 4096^3 2334
    // vs 2392, 3072^3 1003 vs 1035, 4096 x 2048 x 1024 319.5 vs 350.4).
    const Schedule sch = make_schedule(tiles, k_tiles, slots, sk_mode, 8, 0.10, true);

    FfmaArgs a;
    a.M = p.M;
    a.N = p.N;
    a.K = p.K;
    a.A = p.A;
    a.lda = p.lda;
    a.B = p.B;
    a.ldb = p.ldb;
    a.C = p.C;
    a.ldc = p.ldc;
    a.alpha = p.alpha;
    a.beta = p.beta;
    a.strideA = p.strideA;
    a.strideB = p.strideB;
    a.strideC = p.strideC;
    a.tiles_per_item = static_cast<int>(tiles_m * tiles_n);
    a.vec_a = (p.lda % 4 == 0) && (p.strideA % 4 == 0) && (reinterpret_cast<uintptr_t>(p.A) % 16 == 0);
    a.vec_c = (p.ldc % 4 == 0) && (p.strideC % 4 == 0) && (reinterpret_cast<uintptr_t>(p.C) % 16 == 0);
    a.tiles_n = static_cast<int>(tiles_n);
    a.k_tiles = static_cast<int>(k_tiles);
    a.total_tiles = tiles;
    a.dp_tiles = sch.dp_tiles;
    a.sk_iters = sch.sk_iters;
    a.sk_ctas = sch.sk_ctas;
    a.bias = p.bias;
    a.bias_kind = p.bias_kind;
    a.act = p.act;
    a.ep = p.has_epilogue();
    const int split = tiles - sch.dp_tiles;
    rc = split_tiles_prepare(p, C::BM, C::BN, a.tiles_n, a.tiles_per_item, sch.dp_tiles, split, stream, launches);
    if (rc != SGEMM_OK) return rc;
    ffma_kernel<C, TA, TB, VEC_B, VEC_C><<<sch.grid, C::THREADS, C::SMEM_BYTES, stream>>>(a);
    ++*launches;
    if (cudaGetLastError() != cudaSuccess) return SGEMM_ERR_LAUNCH;
    return split_tiles_finish(p, C::BM, C::BN, a.tiles_n, a.tiles_per_item, sch.dp_tiles, split, stream, launches);
}

// Block tile for AUTO: large outputs take the widest register tile (fewest
// shared-memory loads per FFMA); below a full wave of those, 128 x 128 tiles
// with stream-K (measured faster than 64 x 64 at 512^3 and 1024^3 on GB300);
// 64 x 64 only for outputs of a handful of tiles.
inline int pick_tile(const Problem &p, const DeviceInfo &dev, int tile) {
    if (tile != FFMA_TILE_AUTO) return tile;
    const int64_t big_tiles = ceil_div(p.M, CfgBig::BM) * ceil_div(p.N, CfgBig::BN) * p.batch;
    const int64_t mid_tiles = ceil_div(p.M, CfgMid::BM) * ceil_div(p.N, CfgMid::BN) * p.batch;
    if (big_tiles >= dev.sm_count) return FFMA_TILE_128x256;
    if (mid_tiles >= 8) return FFMA_TILE_128x128;
    return FFMA_TILE_64x64;
}

}  // namespace ffma
}  // namespace sgemm
