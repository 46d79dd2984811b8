// Tensor-core SGEMM for sm_103a: tcgen05.mma (kind::tf32) with TMEM
// accumulators and the three-term TF32 split, so the result keeps fp32-level
// accuracy.
//
// The product is the plain sum of "CUDA算子优化(4)：矩阵乘法", section
// "矩阵乘法的数学定义". The pages name tensor cores only as a further
// optimisation ("CUDA内存优化入门：从Naive到Tiled矩阵乘法", section 八); they
// give no design for them, and this kernel is not derived from their code.
//
// Split. Each fp32 value x becomes hi = x truncated to tf32 (sign, exponent,
// top 10 mantissa bits) and lo = tf32(x - hi), where x - hi is exact in fp32.
// Then
//     a*b = hi_a*hi_b + hi_a*lo_b + lo_a*hi_b + lo_a*lo_b,
// and the kernel sums the first three products on the tensor cores with fp32
// accumulation. |lo| < 2^-10 |x|, so the dropped term (< 2^-20 |a*b|) and the
// rounding of lo (< 2^-21 |x|) stay far inside the 1e-5 acceptance bound on
// max |C - C_exact| / sum_k |a_ik||b_kj|. Values with at most 11 significant
// bits (small integers) have lo = 0 and give exact products.
//
// Layout and roles (one persistent CTA per SM, 13 warps):
//   * Block tile 128 x 256 of C, k-block 32. The 128 x 256 fp32 accumulator
//     lives in TMEM (columns 0-255) and is restarted every FOLD_KB k-blocks:
//     the epilogue warps add it, rounded to nearest, into a running sum of
//     the tile in columns 256-511 (the tensor core truncates as it
//     accumulates, so no accumulator may chain many MMAs), and the MMAs of
//     the next interval wait for that fold.
//   * Warps 1-8 (producers) read a k-block of A (128 x 32) and B (32 x 256)
//     from global memory (any alignment; 16-byte loads where the rows allow,
//     unguarded loads for k-blocks inside the matrices), split
//     each value, and write four K-major tiles -- A_hi, A_lo, B_hi, B_lo, each
//     row 32 values = 128 bytes -- into shared memory in the 128-byte swizzled
//     layout that the tensor core reads (16-byte chunk c of row r stored at
//     chunk c ^ (r mod 8)). B is transposed on the way (row n of the B tile is
//     column n of B). Two such stages form a ring.
//   * Warp 0, one thread: per k-block 4 x 3 tcgen05.mma of 128 x 256 x 8
//     (hi*hi, hi*lo, lo*hi for each 8-wide slice of k), then tcgen05.commit to
//     free the stage; after a tile's last k-block, commit to the accumulator.
//   * Warps 9-12 (epilogue): tcgen05.ld the accumulator (each warp reads its
//     32-lane quarter = 32 rows) and store C, guarded by row < M and col < N.
//   * Scheduling: whole tiles round-robin, and the tiles after the last full
//     wave split along K (stream-K), with the split tiles zeroed first and
//     their partial sums added by fp32 atomics.
//   * Every mbarrier wait is bounded in time: past the limit the thread
//     records the event in a device flag and in a CTA abort flag, every role
//     stops issuing work, the MMA thread waits (bounded) for its own MMAs to
//     drain, and the CTA frees its TMEM and exits.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "sgemm.h"
#include "sgemm_internal.h"
#include "tc_common.cuh"

namespace sgemm {

// Per-device watchdog flag: 0, or the code of the first bounded wait that gave up.
__device__ int g_watchdog_code;

namespace {

std::atomic<int64_t> g_watchdog_ms{2000};
// Tensor-core kernel (tuning key SGEMM_TUNE_TF32X3_KERNEL): 0 = automatic,
// 1 = per-thread loads only, 2 = TMA kernel, 3 = TMA kernel with A in TMEM,
// 4 = the SM-pair kernel of sgemm_tf32x3_pair.cu (every form; TMA for
// aligned rows, cp.async otherwise), 5 = automatic, with operands whose rows
// TMA cannot address copied into aligned scratch at any size.
std::atomic<int> g_use_tma{0};
std::atomic<int> g_last_tc_kernel{0};

using namespace tc;

constexpr int STAGES = 2;
constexpr int STAGE_BYTES = 2 * A_TILE + 2 * B_TILE;  // A_hi, A_lo, B_hi, B_lo
constexpr int PRODUCER_WARPS = 8;
constexpr int THREADS = 32 * (1 + PRODUCER_WARPS + EPILOGUE_WARPS);
constexpr int PRODUCER_THREADS = 32 * PRODUCER_WARPS;
// C rows that are not 16-byte aligned leave through one 32 x 32 staging
// chunk per epilogue warp (coalesced row stores, store_staged_rows).
constexpr int STAGE_C = STAGES * STAGE_BYTES;
constexpr int C_CHUNK_BYTES = 32 * 32 * 4;
constexpr int SMEM_BYTES = STAGE_C + EPILOGUE_WARPS * C_CHUNK_BYTES + BAR_BYTES + 1024;  // + slack to align to 1024
constexpr int A_TASKS = BM * (BK / 4);  // 16-byte chunks per A tile
constexpr int B_TASKS = BN * (BK / 4);
static_assert(A_TASKS % PRODUCER_THREADS == 0 && B_TASKS % PRODUCER_THREADS == 0, "even producer split");

template <bool VEC_A, bool VEC_B, bool VEC_C>
__global__ void __launch_bounds__(THREADS, 1) tf32x3_kernel(const Args a) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;  // 1024-aligned: the swizzle uses address bits 4-9
    uint8_t *smem = smem_raw + (base - raw);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + STAGE_C + EPILOGUE_WARPS * C_CHUNK_BYTES);
    // bars[0..1] full, [2..3] empty, [4] acc_full, [6] acc_empty, [8] drain
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(bars + 9);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + 10);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    auto bar = [&](int i) { return smem_u32(bars + i); };

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar(s), PRODUCER_THREADS);
            mbar_init(bar(2 + s), 1);
        }
        mbar_init(bar(4), 1);
        mbar_init(bar(6), 32 * EPILOGUE_WARPS);
        mbar_init(bar(8), 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_holder)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    if (warp == 0) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            uint32_t it = 0, iv = 0;  // k-blocks and fold intervals issued so far
            for_each_unit(a, abort_flag, [&](int, int kb, int ke) {
                for (int k0 = kb; k0 < ke; k0 += FOLD_KB) {
                    const int k1 = ke - k0 > FOLD_KB ? k0 + FOLD_KB : ke;
                    // The accumulator is free once the previous interval is folded.
                    if (!mbar_wait(bar(6), (iv & 1) ^ 1, a, abort_flag, WD_MMA_ACC)) return;
                    tc_fence_after();
                    for (int kblk = k0; kblk < k1; ++kblk, ++it) {
                        const int s = it & 1;
                        if (!mbar_wait(bar(s), (it >> 1) & 1, a, abort_flag, WD_MMA_FULL)) return;
                        tc_fence_after();
                        const uint32_t st = base + static_cast<uint32_t>(s * STAGE_BYTES);
                        const uint64_t a_hi = sw128_desc(st), a_lo = sw128_desc(st + A_TILE);
                        const uint64_t b_hi = sw128_desc(st + 2 * A_TILE), b_lo = sw128_desc(st + 2 * A_TILE + B_TILE);
#pragma unroll
                        for (int ks = 0; ks < BK / 8; ++ks) {
                            // 8 tf32 = 32 bytes along K: advance the start address (field units of 16 B).
                            const uint64_t adv = static_cast<uint64_t>(ks * 2);
                            const uint32_t first = (kblk == k0 && ks == 0) ? 0u : 1u;
                            tc_mma(tmem_base, a_lo + adv, b_hi + adv, first);
                            tc_mma(tmem_base, a_hi + adv, b_lo + adv, 1u);
                            tc_mma(tmem_base, a_hi + adv, b_hi + adv, 1u);
                        }
                        tc_commit(bar(2 + s));  // the stage is free once these MMAs finish
                    }
                    tc_commit(bar(4));  // interval done: the epilogue folds or stores it
                    ++iv;
                }
            });
            // Drain: every MMA this thread issued has finished before TMEM is freed.
            tc_commit(bar(8));
            const bool was_aborted = *abort_flag != 0;
            if (!mbar_wait(bar(8), 0, a, abort_flag, WD_DRAIN) && was_aborted) {
                // Already aborted: one more bounded wait for the drain, ignoring the flag.
                const uint64_t t0 = global_timer();
                while (!mbar_try_wait(bar(8), 0) && global_timer() - t0 < a.timeout_ns) {
                }
            }
        }
    } else if (warp <= PRODUCER_WARPS) {
        // -------------------------------------------------------------- producers
        const int pt = threadIdx.x - 32;  // 0 .. PRODUCER_THREADS-1
        // A: task r is row r*32 + pt/8, 16-byte chunk pt%8 (8 lanes = one row).
        const int a_row0 = pt >> 3, a_ch = pt & 7;
        const uint32_t a_off0 = sw128_offset(a_row0, a_ch);  // + r * 32 rows * 128 B
        // B with 16-byte loads: task r covers B rows 4c..4c+3 (c = pt%8) and
        // columns 4g..4g+3 (g = pt/8 + 32r); a quarter-warp shares g and spans
        // the 8 chunks, so its swizzled stores hit 8 distinct bank groups.
        const int b_c = pt & 7, b_g0 = pt >> 3;
        uint32_t it = 0;
        bool ok = true;
        for_each_unit(a, abort_flag, [&](int tile, int kb, int ke) {
            if (!ok) return;
            const TileAt at = tile_at(a, tile);
            const int64_t m0 = at.m0, n0 = at.n0;
            const float *Ai = a.A + at.item * a.strideA;
            const float *Bi = a.B + at.item * a.strideB;
            const bool full_mn = (m0 + BM <= a.M) && (n0 + BN <= a.N);
            const float *a_base = Ai + (m0 + a_row0) * a.lda + a_ch * 4;
            const float *b_base = VEC_B ? Bi + static_cast<int64_t>(4 * b_c) * a.ldb + n0 + 4 * b_g0
                                        : Bi + n0 + pt;
            for (int kblk = kb; kblk < ke; ++kblk, ++it) {
                const int s = it & 1;
                const int64_t k0 = static_cast<int64_t>(kblk) * BK;
                const bool interior = full_mn && (k0 + BK <= a.K);
                // Loads first (all in flight together), then split and store.
                float4 av[4], bv[8];
                if (interior) {
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const float *src = a_base + static_cast<int64_t>(r * 32) * a.lda + k0;
                        if (VEC_A) {
                            av[r] = __ldg(reinterpret_cast<const float4 *>(src));
                        } else {
                            av[r] = make_float4(__ldg(src), __ldg(src + 1), __ldg(src + 2), __ldg(src + 3));
                        }
                    }
                    if (VEC_B) {
#pragma unroll
                        for (int r = 0; r < 2; ++r)
#pragma unroll
                            for (int q = 0; q < 4; ++q)
                                bv[r * 4 + q] = __ldg(reinterpret_cast<const float4 *>(
                                    b_base + (k0 + q) * a.ldb + 128 * r));
                    } else {
#pragma unroll
                        for (int r = 0; r < 8; ++r) {
                            const float *src = b_base + (k0 + 4 * r) * a.ldb;
                            bv[r] = make_float4(__ldg(src), __ldg(src + a.ldb), __ldg(src + 2 * a.ldb),
                                                __ldg(src + 3 * a.ldb));
                        }
                    }
                } else {
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const int64_t gm = m0 + a_row0 + r * 32, gk = k0 + a_ch * 4;
                        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                        if (gm < a.M) {
                            const float *src = Ai + gm * a.lda + gk;
                            if (gk + 0 < a.K) v.x = __ldg(src + 0);
                            if (gk + 1 < a.K) v.y = __ldg(src + 1);
                            if (gk + 2 < a.K) v.z = __ldg(src + 2);
                            if (gk + 3 < a.K) v.w = __ldg(src + 3);
                        }
                        av[r] = v;
                    }
                    if (VEC_B) {
#pragma unroll
                        for (int r = 0; r < 2; ++r)
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                const int64_t gk = k0 + 4 * b_c + q, gn = n0 + 4 * (b_g0 + 32 * r);
                                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                                if (gk < a.K) {
                                    const float *src = Bi + gk * a.ldb + gn;
                                    if (gn + 3 < a.N) {
                                        v = __ldg(reinterpret_cast<const float4 *>(src));
                                    } else {
                                        if (gn + 0 < a.N) v.x = __ldg(src + 0);
                                        if (gn + 1 < a.N) v.y = __ldg(src + 1);
                                        if (gn + 2 < a.N) v.z = __ldg(src + 2);
                                    }
                                }
                                bv[r * 4 + q] = v;
                            }
                    } else {
#pragma unroll
                        for (int r = 0; r < 8; ++r) {
                            const int64_t gn = n0 + pt, gk = k0 + 4 * r;
                            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                            if (gn < a.N) {
                                const float *src = Bi + gk * a.ldb + gn;
                                if (gk + 0 < a.K) v.x = __ldg(src);
                                if (gk + 1 < a.K) v.y = __ldg(src + a.ldb);
                                if (gk + 2 < a.K) v.z = __ldg(src + 2 * a.ldb);
                                if (gk + 3 < a.K) v.w = __ldg(src + 3 * a.ldb);
                            }
                            bv[r] = v;
                        }
                    }
                }
                if (!mbar_wait(bar(2 + s), ((it >> 1) & 1) ^ 1, a, abort_flag, WD_PRODUCER)) {
                    ok = false;
                    return;
                }
                const uint32_t st = base + static_cast<uint32_t>(s * STAGE_BYTES);
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const uint32_t off = a_off0 + static_cast<uint32_t>(r * 32 * 128);
                    split_store(st + off, st + A_TILE + off, av[r].x, av[r].y, av[r].z, av[r].w);
                }
                const uint32_t bh = st + 2 * A_TILE, bl = bh + B_TILE;
                if (VEC_B) {
                    // bv[r*4 + q] holds B row 4c+q, columns 4g..4g+3: column j of
                    // that 4 x 4 block is chunk c of tile row 4g + j.
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        const int g = b_g0 + 32 * r;
                        const float4 q0 = bv[r * 4 + 0], q1 = bv[r * 4 + 1], q2 = bv[r * 4 + 2], q3 = bv[r * 4 + 3];
                        uint32_t off = sw128_offset(4 * g + 0, b_c);
                        split_store(bh + off, bl + off, q0.x, q1.x, q2.x, q3.x);
                        off = sw128_offset(4 * g + 1, b_c);
                        split_store(bh + off, bl + off, q0.y, q1.y, q2.y, q3.y);
                        off = sw128_offset(4 * g + 2, b_c);
                        split_store(bh + off, bl + off, q0.z, q1.z, q2.z, q3.z);
                        off = sw128_offset(4 * g + 3, b_c);
                        split_store(bh + off, bl + off, q0.w, q1.w, q2.w, q3.w);
                    }
                } else {
                    // bv[r] holds B rows 4r..4r+3 of column pt: chunk r of tile row pt.
#pragma unroll
                    for (int r = 0; r < 8; ++r) {
                        const uint32_t off = sw128_offset(pt, r);
                        split_store(bh + off, bl + off, bv[r].x, bv[r].y, bv[r].z, bv[r].w);
                    }
                }
                fence_proxy_async_smem();  // generic-proxy stores -> visible to the tensor core
                mbar_arrive(bar(s));
            }
        });
    } else {
        // -------------------------------------------------------------- epilogue
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const uint32_t tq = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
        uint32_t iv = 0;
        for_each_unit(a, abort_flag, [&](int tile, int kb, int ke) {
            const TileAt at = tile_at(a, tile);
            const int64_t m0 = at.m0, n0 = at.n0;
            const int64_t row = m0 + q * 32 + lane;
            // Stream-K tiles hold beta * C + bias already: every unit adds.
            const bool atomic = tile >= a.dp_tiles;
            float *crow = a.C + at.item * a.strideC + row * a.ldc;
            for (int k0 = kb; k0 < ke; k0 += FOLD_KB) {
                const bool first = k0 == kb, last = ke - k0 <= FOLD_KB;
                if (!mbar_wait(bar(4), iv & 1, a, abort_flag, WD_EPILOGUE)) return;
                tc_fence_after();
                ++iv;
#pragma unroll 1
                for (int ch = 0; ch < BN / 32; ++ch) {
                    const uint32_t td = tq + static_cast<uint32_t>(ch * 32), tr = td + BN;
                    float v[32];
                    tmem_load32(td, v);
                    if (!first) {
                        float r[32];
                        tmem_load32(tr, r);
#pragma unroll
                        for (int j = 0; j < 32; ++j) v[j] += r[j];
                    }
                    if (ch == BN / 32 - 1) {
                        // The accumulator is out: the next interval's MMAs may start.
                        tmem_wait_st();
                        tc_fence_before();
                        mbar_arrive(bar(6));
                    }
                    if (last) {
                        fix_nonfinite(a, at.item, row, n0 + ch * 32, static_cast<int64_t>(kb) * BK,
                                      static_cast<int64_t>(ke) * BK, v);
                        if (VEC_C || (a.ep && !atomic)) {
                            store_chunk_regs<VEC_C>(a, crow, row, n0 + ch * 32, v, atomic);
                        } else if (n0 + ch * 32 < a.N) {
                            // Unaligned C rows: through shared memory, one coalesced row per step.
                            const uint32_t cs = base + static_cast<uint32_t>(STAGE_C + q * C_CHUNK_BYTES);
#pragma unroll
                            for (int j = 0; j < 8; ++j)
                                st_shared_v4(cs + sw128_offset(lane, j), v[4 * j], v[4 * j + 1], v[4 * j + 2],
                                             v[4 * j + 3]);
                            __syncwarp();
                            store_staged_rows(a, cs, a.C + at.item * a.strideC, m0 + q * 32, n0 + ch * 32, atomic);
                            __syncwarp();  // the chunk is read before the next one is written
                        }
                    } else {
                        float h[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j) h[j] = v[j];
                        tmem_store16(tr, h);
#pragma unroll
                        for (int j = 0; j < 16; ++j) h[j] = v[16 + j];
                        tmem_store16(tr + 16, h);
                    }
                }
                if (!last) tmem_wait_st();  // the running sum is written before it is read again
            }
        });
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS)
                     : "memory");
    }
}


// ---------------------------------------------------------------------------
// TMA variant, for A and B whose base addresses and row strides are 16-byte
// aligned. The tensor core reads an fp32 value of a kind::tf32 operand as its
// truncation to tf32, so a raw tile can serve as the high part:
//   * TMA copies the A tile (K-major, as stored) straight into the stage in
//     the 128-byte swizzled layout: that is A's high part. Converter warps add
//     A's low part chunk for chunk at the same offsets.
//   * B is stored N-contiguous, and the operand must be K-major, so TMA copies
//     the raw B tile (32 rows of K x 256 of N, unswizzled) into a staging
//     buffer; converter warps read it in 4 x 4 blocks and write B's high and
//     low parts transposed into the stage. Lane l of each group of eight
//     takes column block g = g0 + l and k-chunk c = (l + s) mod 8, which keeps
//     both the staging reads and the swizzled stores free of bank conflicts.
//     The staging buffer is released as soon as its values are in registers.
// Out-of-range elements arrive as zeros from TMA.
//   warp 0: MMA issuer; warp 1: TMA issuer; warps 2-9: converters;
//   warps 10-13: epilogue.
// Shared memory: two 96 KB stages (A raw = hi | A lo | B hi | B lo) and the
// 32 KB B staging buffer.
namespace tma {

constexpr int CONV_WARPS = 8;
constexpr int CONV_THREADS = 32 * CONV_WARPS;
constexpr int EPI_WARP0 = 2 + CONV_WARPS;
constexpr int THREADS = 32 * (EPI_WARP0 + EPILOGUE_WARPS);
constexpr int A_RAW = 0, A_LO = A_TILE, B_HI = 2 * A_TILE, B_LO = 2 * A_TILE + B_TILE;
constexpr int STAGING = STAGES * STAGE_BYTES;  // B raw: BK rows x BN floats
constexpr int STAGING_BYTES = BK * BN * 4;
constexpr int BAR_OFFSET = STAGING + STAGING_BYTES;
constexpr int SMEM_BYTES = BAR_OFFSET + BAR_BYTES + 1024;
constexpr int A_CHUNKS = A_TILE / 16;
static_assert(A_CHUNKS % CONV_THREADS == 0, "even converter split of A");
static_assert((BN / 4) * (BK / 4) == 2 * CONV_THREADS, "two 4 x 4 B blocks per converter thread");
static_assert(BK == 32 && BN % 32 == 0, "diagonal mapping assumes 8 k-chunks");

}  // namespace tma

template <bool VEC_C>
__global__ void __launch_bounds__(tma::THREADS, 1)
    tf32x3_tma_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const Args a) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (base - raw);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + tma::BAR_OFFSET);
    // [0..1] a_full (TMA of A), [2..3] empty (MMA done with the stage),
    // [4..5] acc_full, [6..7] acc_empty, [8] drain, [9..10] op_full
    // (converters done), [11] b_staged (TMA of B), [12] staging free
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(bars + 13);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + 14);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    auto bar = [&](int i) { return smem_u32(bars + i); };
    const uint32_t staging = base + tma::STAGING;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar(s), 1);
            mbar_init(bar(2 + s), 1);
            mbar_init(bar(9 + s), tma::CONV_THREADS);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(4 + b), 1);
            mbar_init(bar(6 + b), 32 * EPILOGUE_WARPS);
        }
        mbar_init(bar(8), 1);
        mbar_init(bar(11), 1);
        mbar_init(bar(12), tma::CONV_THREADS);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_holder)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    if (warp == 0) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            uint32_t it = 0, unit = 0;
            for_each_unit(a, abort_flag, [&](int, int kb, int ke) {
                const int buf = unit & 1;
                if (!mbar_wait(bar(6 + buf), ((unit >> 1) & 1) ^ 1, a, abort_flag, WD_MMA_ACC)) return;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * BN);
                for (int kblk = kb; kblk < ke; ++kblk, ++it) {
                    const int s = it & 1;
                    const uint32_t ph = (it >> 1) & 1;
                    if (!mbar_wait(bar(9 + s), ph, a, abort_flag, WD_MMA_FULL)) return;
                    if (!mbar_wait(bar(s), ph, a, abort_flag, WD_MMA_FULL)) return;
                    tc_fence_after();
                    const uint32_t st = base + static_cast<uint32_t>(s * STAGE_BYTES);
                    const uint64_t a_hi = sw128_desc(st + tma::A_RAW), a_lo = sw128_desc(st + tma::A_LO);
                    const uint64_t b_hi = sw128_desc(st + tma::B_HI), b_lo = sw128_desc(st + tma::B_LO);
#pragma unroll
                    for (int ks = 0; ks < BK / 8; ++ks) {
                        const uint64_t adv = static_cast<uint64_t>(ks * 2);  // 32 bytes along K
                        const uint32_t first = (kblk == kb && ks == 0) ? 0u : 1u;
                        tc_mma(d_tmem, a_lo + adv, b_hi + adv, first);
                        tc_mma(d_tmem, a_hi + adv, b_lo + adv, 1u);
                        tc_mma(d_tmem, a_hi + adv, b_hi + adv, 1u);
                    }
                    tc_commit(bar(2 + s));
                }
                tc_commit(bar(4 + buf));
                ++unit;
            });
            tc_commit(bar(8));
            const bool was_aborted = *abort_flag != 0;
            if (!mbar_wait(bar(8), 0, a, abort_flag, WD_DRAIN) && was_aborted) {
                const uint64_t t0 = global_timer();
                while (!mbar_try_wait(bar(8), 0) && global_timer() - t0 < a.timeout_ns) {
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ TMA issuer
        if (lane == 0) {
            uint32_t it = 0;
            bool ok = true;
            for_each_unit(a, abort_flag, [&](int tile, int kb, int ke) {
                if (!ok) return;
                const TileAt at = tile_at(a, tile);
                const int m0 = static_cast<int>(at.m0), n0 = static_cast<int>(at.n0);
                const int za = a.a_shared ? 0 : at.item, zb = a.b_shared ? 0 : at.item;
                for (int kblk = kb; kblk < ke; ++kblk, ++it) {
                    const int s = it & 1;
                    const int k0 = kblk * BK;
                    // B into the staging buffer once the converters have read the last one.
                    if (!mbar_wait(bar(12), (it & 1) ^ 1, a, abort_flag, WD_PRODUCER)) {
                        ok = false;
                        return;
                    }
                    mbar_arrive_expect_tx(bar(11), tma::STAGING_BYTES);
                    tma_load_3d(staging, &tmB, n0, k0, zb, bar(11));
                    // A straight into the stage once the MMA is done with it.
                    if (!mbar_wait(bar(2 + s), ((it >> 1) & 1) ^ 1, a, abort_flag, WD_PRODUCER)) {
                        ok = false;
                        return;
                    }
                    mbar_arrive_expect_tx(bar(s), A_TILE);
                    tma_load_3d(base + static_cast<uint32_t>(s * STAGE_BYTES) + tma::A_RAW, &tmA, k0, m0, za, bar(s));
                }
            });
        }
    } else if (warp < tma::EPI_WARP0) {
        // ------------------------------------------------------------ converters
        const int ct = threadIdx.x - 64;
        const int l = ct & 7, quarter = ct >> 3;  // 32 groups of eight lanes
        uint32_t it = 0;
        bool ok = true;
        for_each_unit(a, abort_flag, [&](int, int kb, int ke) {
            if (!ok) return;
            for (int kblk = kb; kblk < ke; ++kblk, ++it) {
                const int s = it & 1;
                // B: two 4 x 4 blocks per thread from the staging buffer.
                if (!mbar_wait(bar(11), it & 1, a, abort_flag, WD_PRODUCER)) {
                    ok = false;
                    return;
                }
                float4 bv[2][4];
                int bg[2], bc[2];
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const int tb = quarter * 2 + r;  // 0..63
                    const int g = (tb >> 3) * 8 + l, c = (l + tb) & 7;
                    bg[r] = g;
                    bc[r] = c;
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        bv[r][q] = ld_shared_v4(staging + static_cast<uint32_t>((4 * c + q) * BN * 4 + g * 16));
                }
                // The next TMA (async proxy) overwrites what these generic loads
                // read: order them first, then release the staging buffer.
                fence_proxy_async_smem();
                mbar_arrive(bar(12));
                if (!mbar_wait(bar(s), (it >> 1) & 1, a, abort_flag, WD_PRODUCER)) {
                    ok = false;
                    return;
                }
                const uint32_t st = base + static_cast<uint32_t>(s * STAGE_BYTES);
                float4 av[tma::A_CHUNKS / tma::CONV_THREADS];
#pragma unroll
                for (int r = 0; r < tma::A_CHUNKS / tma::CONV_THREADS; ++r)
                    av[r] = ld_shared_v4(st + tma::A_RAW + (r * tma::CONV_THREADS + ct) * 16);
#pragma unroll
                for (int r = 0; r < tma::A_CHUNKS / tma::CONV_THREADS; ++r)
                    st_shared_v4(st + tma::A_LO + (r * tma::CONV_THREADS + ct) * 16, lo_of(av[r].x), lo_of(av[r].y),
                                 lo_of(av[r].z), lo_of(av[r].w));
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    // bv[r][q] = B row 4c+q, columns 4g..4g+3; column j of the block is
                    // chunk c of operand row 4g + j.
                    const float4 q0 = bv[r][0], q1 = bv[r][1], q2 = bv[r][2], q3 = bv[r][3];
                    const int g = bg[r], c = bc[r];
                    uint32_t off = sw128_offset(4 * g + 0, c);
                    split_store(st + tma::B_HI + off, st + tma::B_LO + off, q0.x, q1.x, q2.x, q3.x);
                    off = sw128_offset(4 * g + 1, c);
                    split_store(st + tma::B_HI + off, st + tma::B_LO + off, q0.y, q1.y, q2.y, q3.y);
                    off = sw128_offset(4 * g + 2, c);
                    split_store(st + tma::B_HI + off, st + tma::B_LO + off, q0.z, q1.z, q2.z, q3.z);
                    off = sw128_offset(4 * g + 3, c);
                    split_store(st + tma::B_HI + off, st + tma::B_LO + off, q0.w, q1.w, q2.w, q3.w);
                }
                fence_proxy_async_smem();
                mbar_arrive(bar(9 + s));
            }
        });
    } else {
        // -------------------------------------------------------------- epilogue
        const int q = warp & 3;
        uint32_t unit = 0;
        for_each_unit(a, abort_flag, [&](int tile, int kb, int ke) {
            const int buf = unit & 1;
            if (!mbar_wait(bar(4 + buf), (unit >> 1) & 1, a, abort_flag, WD_EPILOGUE)) return;
            tc_fence_after();
            const TileAt at = tile_at(a, tile);
            const int64_t m0 = at.m0, n0 = at.n0;
            const int64_t row = m0 + q * 32 + lane;
            // Stream-K tiles hold beta * C + bias already: every unit adds.
            const bool atomic = tile >= a.dp_tiles;
            float *crow = a.C + at.item * a.strideC + row * a.ldc;
#pragma unroll 1
            for (int ch = 0; ch < BN / 32; ++ch)
                epilogue_chunk<VEC_C>(
                    a, tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(buf * BN + ch * 32),
                    crow, row, n0 + ch * 32, atomic, false, 0, at.item, static_cast<int64_t>(kb) * BK,
                    static_cast<int64_t>(ke) * BK);
            tc_fence_before();
            mbar_arrive(bar(6 + buf));
            ++unit;
        });
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS)
                     : "memory");
    }
}


// ---------------------------------------------------------------------------
// Variant with A in TMEM (same alignment needs as the TMA variant). A's high
// and low parts go to TMEM, which frees the shared memory for a raw staging
// ring two k-blocks deep, so TMA latency stays off the critical path:
//   shared: two B operand stages (B hi | B lo, 64 KB each) and two raw slots
//   (A tile 16 KB with 128-byte swizzle | B tile 32 KB unswizzled);
//   TMEM: the 128 x 256 accumulator (columns 0-255) and two A stages
//   (columns 256 + 64 s: hi in the first 32, lo in the next 32).
// Sixteen converter warps: each takes one TMEM lane quarter (warp mod 4) and
// one quarter of the 32 k-columns, so every thread splits 8 values of one row
// of A and stores them with tcgen05.st; each thread also transposes one 4 x 4
// block of B into the stage (mapping as in the TMA variant).
// One accumulator: the MMA of the next unit waits for the epilogue to drain.
namespace tm3 {

constexpr int CONV_WARPS = 16;
constexpr int CONV_THREADS = 32 * CONV_WARPS;
constexpr int EPI_WARP0 = 2 + CONV_WARPS;
constexpr int THREADS = 32 * (EPI_WARP0 + EPILOGUE_WARPS);
constexpr int B_STAGE = 2 * B_TILE;  // hi | lo
constexpr int SLOT = A_TILE + B_TILE;  // raw A | raw B
constexpr int RAW0 = STAGES * B_STAGE;
constexpr int BAR_OFFSET = RAW0 + 2 * SLOT;
constexpr int SMEM_BYTES = BAR_OFFSET + BAR_BYTES + 1024;
constexpr uint32_t TMEM_A = BN;  // first A column
static_assert((BN / 4) * (BK / 4) == CONV_THREADS, "one 4 x 4 B block per converter thread");
static_assert(CONV_WARPS == 16, "four converter warps per TMEM lane quarter, 8 k-columns each");

}  // namespace tm3

template <bool VEC_C, bool TA, bool TB>
__global__ void __launch_bounds__(tm3::THREADS, 1)
    tf32x3_tmem_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const Args a) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (base - raw);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + tm3::BAR_OFFSET);
    // [0..1] raw_full (TMA), [2..3] raw_free (converters read the slot),
    // [4..5] op_full (converters wrote the stage), [6..7] empty (MMA done),
    // [8] acc_full, [9] acc_empty, [10] drain
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(bars + 11);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + 12);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    auto bar = [&](int i) { return smem_u32(bars + i); };

    if (threadIdx.x == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(s), 1);
            mbar_init(bar(2 + s), tm3::CONV_THREADS);
            mbar_init(bar(4 + s), tm3::CONV_THREADS);
            mbar_init(bar(6 + s), 1);
        }
        mbar_init(bar(8), 1);
        mbar_init(bar(9), 32 * EPILOGUE_WARPS);
        mbar_init(bar(10), 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_holder)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    if (warp == 0) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            uint32_t it = 0, unit = 0;
            for_each_unit(a, abort_flag, [&](int, int kb, int ke) {
                if (!mbar_wait(bar(9), (unit & 1) ^ 1, a, abort_flag, WD_MMA_ACC)) return;
                tc_fence_after();
                for (int kblk = kb; kblk < ke; ++kblk, ++it) {
                    const int s = it & 1;
                    if (!mbar_wait(bar(4 + s), (it >> 1) & 1, a, abort_flag, WD_MMA_FULL)) return;
                    tc_fence_after();
                    const uint32_t st = base + static_cast<uint32_t>(s * tm3::B_STAGE);
                    const uint64_t b_hi = sw128_desc(st), b_lo = sw128_desc(st + B_TILE);
                    const uint32_t a_hi = tmem_base + tm3::TMEM_A + static_cast<uint32_t>(64 * s);
                    const uint32_t a_lo = a_hi + 32;
#pragma unroll
                    for (int ks = 0; ks < BK / 8; ++ks) {
                        const uint64_t adv = static_cast<uint64_t>(ks * 2);
                        const uint32_t ac = static_cast<uint32_t>(ks * 8);
                        const uint32_t first = (kblk == kb && ks == 0) ? 0u : 1u;
                        tc_mma_ts(tmem_base, a_lo + ac, b_hi + adv, first);
                        tc_mma_ts(tmem_base, a_hi + ac, b_lo + adv, 1u);
                        tc_mma_ts(tmem_base, a_hi + ac, b_hi + adv, 1u);
                    }
                    tc_commit(bar(6 + s));
                }
                tc_commit(bar(8));
                ++unit;
            });
            tc_commit(bar(10));
            const bool was_aborted = *abort_flag != 0;
            if (!mbar_wait(bar(10), 0, a, abort_flag, WD_DRAIN) && was_aborted) {
                const uint64_t t0 = global_timer();
                while (!mbar_try_wait(bar(10), 0) && global_timer() - t0 < a.timeout_ns) {
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ TMA issuer
        if (lane == 0) {
            uint32_t it = 0;
            bool ok = true;
            for_each_unit(a, abort_flag, [&](int tile, int kb, int ke) {
                if (!ok) return;
                const TileAt at = tile_at(a, tile);
                const int m0 = static_cast<int>(at.m0), n0 = static_cast<int>(at.n0);
                const int za = a.a_shared ? 0 : at.item, zb = a.b_shared ? 0 : at.item;
                for (int kblk = kb; kblk < ke; ++kblk, ++it) {
                    const int slot = it & 1;
                    if (!mbar_wait(bar(2 + slot), ((it >> 1) & 1) ^ 1, a, abort_flag, WD_PRODUCER)) {
                        ok = false;
                        return;
                    }
                    const uint32_t sl = base + tm3::RAW0 + static_cast<uint32_t>(slot * tm3::SLOT);
                    mbar_arrive_expect_tx(bar(slot), tm3::SLOT);
                    if (TA) {  // A stored K x M: four boxes of 32 m x 32 k
#pragma unroll
                        for (int b = 0; b < BM / 32; ++b)
                            tma_load_3d(sl + b * 4096, &tmA, m0 + 32 * b, kblk * BK, za, bar(slot));
                    } else {
                        tma_load_3d(sl, &tmA, kblk * BK, m0, za, bar(slot));
                    }
                    if (TB)  // B stored N x K: already K-major, 256 rows of 32 k
                        tma_load_3d(sl + A_TILE, &tmB, kblk * BK, n0, zb, bar(slot));
                    else
                        tma_load_3d(sl + A_TILE, &tmB, n0, kblk * BK, zb, bar(slot));
                }
            });
        }
    } else if (warp < tm3::EPI_WARP0) {
        // ------------------------------------------------------------ converters
        const int ct = threadIdx.x - 64;
        const int l = ct & 7, tb = ct >> 3;  // 64 groups of eight lanes
        const int g = (tb >> 3) * 8 + l, c = (l + tb) & 7;  // this thread's 4 x 4 B block
        const int q = warp & 3, part = (warp - 2) >> 2;     // TMEM lane quarter, k-columns 8*part..+7
        const int arow = 32 * q + lane;                     // A row this thread converts
        uint32_t it = 0;
        bool ok = true;
        for_each_unit(a, abort_flag, [&](int, int kb, int ke) {
            if (!ok) return;
            for (int kblk = kb; kblk < ke; ++kblk, ++it) {
                const int s = it & 1;
                const uint32_t ph = (it >> 1) & 1;
                if (!mbar_wait(bar(s), ph, a, abort_flag, WD_PRODUCER)) {
                    ok = false;
                    return;
                }
                const uint32_t sl = base + tm3::RAW0 + static_cast<uint32_t>(s * tm3::SLOT);
                // A: 8 k-values of row arow.
                float av[8];
                if (TA) {
                    // Box q holds rows k = 0..31 of columns m = 32q..32q+31 (128-byte
                    // swizzled): column arow is lane `lane` of each row.
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int k = 8 * part + j;
                        av[j] = ld_shared_f32(sl + static_cast<uint32_t>(q * 4096) + sw128_offset(k, lane >> 2) +
                                              static_cast<uint32_t>((lane & 3) * 4));
                    }
                } else {
                    const float4 a0 = ld_shared_v4(sl + sw128_offset(arow, 2 * part));
                    const float4 a1 = ld_shared_v4(sl + sw128_offset(arow, 2 * part + 1));
                    av[0] = a0.x;
                    av[1] = a0.y;
                    av[2] = a0.z;
                    av[3] = a0.w;
                    av[4] = a1.x;
                    av[5] = a1.y;
                    av[6] = a1.z;
                    av[7] = a1.w;
                }
                // B: rows 4c..4c+3, columns 4g..4g+3 of the unswizzled staging tile
                // (op(B) = B), or four 16-byte chunks of the K-major tile (B^T).
                float4 bq[4];
#pragma unroll
                for (int qq = 0; qq < 4; ++qq)
                    bq[qq] = TB ? ld_shared_v4(sl + A_TILE + static_cast<uint32_t>((qq * tm3::CONV_THREADS + ct) * 16))
                                : ld_shared_v4(sl + A_TILE + static_cast<uint32_t>((4 * c + qq) * BN * 4 + g * 16));
                fence_proxy_async_smem();  // order these loads before the next TMA into the slot
                mbar_arrive(bar(2 + s));
                // The stage (B in shared memory, A in TMEM) is free once the MMA
                // two k-blocks back has finished.
                if (!mbar_wait(bar(6 + s), ph ^ 1, a, abort_flag, WD_PRODUCER)) {
                    ok = false;
                    return;
                }
                tc_fence_after();
                const uint32_t st = base + static_cast<uint32_t>(s * tm3::B_STAGE);
                if (TB) {
                    // Same swizzled K-major layout: chunk for chunk.
#pragma unroll
                    for (int qq = 0; qq < 4; ++qq) {
                        const uint32_t off = static_cast<uint32_t>((qq * tm3::CONV_THREADS + ct) * 16);
                        split_store(st + off, st + B_TILE + off, bq[qq].x, bq[qq].y, bq[qq].z, bq[qq].w);
                    }
                } else {
                    // Column j of the 4 x 4 block is chunk c of operand row 4g + j.
                    uint32_t off = sw128_offset(4 * g + 0, c);
                    split_store(st + off, st + B_TILE + off, bq[0].x, bq[1].x, bq[2].x, bq[3].x);
                    off = sw128_offset(4 * g + 1, c);
                    split_store(st + off, st + B_TILE + off, bq[0].y, bq[1].y, bq[2].y, bq[3].y);
                    off = sw128_offset(4 * g + 2, c);
                    split_store(st + off, st + B_TILE + off, bq[0].z, bq[1].z, bq[2].z, bq[3].z);
                    off = sw128_offset(4 * g + 3, c);
                    split_store(st + off, st + B_TILE + off, bq[0].w, bq[1].w, bq[2].w, bq[3].w);
                }
                float hi[8], lo[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) split_tf32(av[j], hi[j], lo[j]);
                const uint32_t ta = tmem_base + (static_cast<uint32_t>(32 * q) << 16) + tm3::TMEM_A +
                                    static_cast<uint32_t>(64 * s + 8 * part);
                tmem_store8(ta, hi);
                tmem_store8(ta + 32, lo);
                tmem_wait_st();
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(bar(4 + s));
            }
        });
    } else {
        // -------------------------------------------------------------- epilogue
        const int q = warp & 3;
        uint32_t unit = 0;
        for_each_unit(a, abort_flag, [&](int tile, int kb, int ke) {
            if (!mbar_wait(bar(8), unit & 1, a, abort_flag, WD_EPILOGUE)) return;
            tc_fence_after();
            const TileAt at = tile_at(a, tile);
            const int64_t m0 = at.m0, n0 = at.n0;
            const int64_t row = m0 + q * 32 + lane;
            // Stream-K tiles hold beta * C + bias already: every unit adds.
            const bool atomic = tile >= a.dp_tiles;
            float *crow = a.C + at.item * a.strideC + row * a.ldc;
#pragma unroll 1
            for (int ch = 0; ch < BN / 32; ++ch)  // the last chunk frees the accumulator for the next unit
                epilogue_chunk<VEC_C>(a, tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(ch * 32),
                                      crow, row, n0 + ch * 32, atomic, ch == BN / 32 - 1, bar(9), at.item,
                                      static_cast<int64_t>(kb) * BK, static_cast<int64_t>(ke) * BK);
            ++unit;
        });
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS)
                     : "memory");
    }
}

// One bounded wait on an mbarrier that nothing arrives at: it must give up
// after timeout_ns, record WD_SELFTEST in the watchdog flag and return.
__global__ void watchdog_selftest_kernel(uint64_t timeout_ns, int *flag) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        Args a{};
        a.timeout_ns = timeout_ns;
        a.watchdog = flag;
        mbar_wait(smem_u32(&bar), 0, a, &abort_flag, WD_SELFTEST);
    }
    __syncthreads();
}

constexpr int kMaxDevices = 64;
std::once_flag g_attr_once[kMaxDevices][8];
cudaError_t g_attr_err[kMaxDevices][8];

template <bool VEC_A, bool VEC_B, bool VEC_C>
int launch(const Problem &p, const DeviceInfo &dev, int sk_mode, cudaStream_t stream, int *launches) {
    constexpr int idx = (VEC_A ? 4 : 0) + (VEC_B ? 2 : 0) + (VEC_C ? 1 : 0);
    auto kernel = tf32x3_kernel<VEC_A, VEC_B, VEC_C>;
    std::call_once(g_attr_once[dev.device][idx], [&] {
        g_attr_err[dev.device][idx] =
            cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    });
    if (g_attr_err[dev.device][idx] != cudaSuccess) {
        cudaGetLastError();
        return SGEMM_ERR_LAUNCH;
    }
    int *flag = watchdog_flag_device_ptr();
    if (!flag) return SGEMM_ERR_LAUNCH;

    const int64_t tiles_m = (p.M + BM - 1) / BM, tiles_n = (p.N + BN - 1) / BN;
    const int64_t k_blocks = (p.K + BK - 1) / BK;
    if (tiles_m * tiles_n * p.batch > INT32_MAX / 2 || k_blocks > INT32_MAX / 2) return SGEMM_ERR_UNSUPPORTED;
    const int tiles = static_cast<int>(tiles_m * tiles_n * p.batch);
    // One CTA per SM (the stage ring takes most of shared memory). A stream-K
    // share below 4 k-blocks costs more in fix-up than it saves.
    // Accumulation chains are bounded by the folds inside the kernel, so
    // units may span any number of k-blocks.
    const Schedule sch = make_schedule(tiles, k_blocks, dev.sm_count, sk_mode, 4, 0.25);
    const int split = tiles - sch.dp_tiles;
    int rc = split_tiles_prepare(p, BM, BN, static_cast<int>(tiles_n), static_cast<int>(tiles_m * tiles_n),
                                 sch.dp_tiles, split, stream, launches);
    if (rc != SGEMM_OK) return rc;
    Args a;
    a.M = p.M;
    a.N = p.N;
    a.K = p.K;
    a.A = p.A;
    a.lda = p.lda;
    a.B = p.B;
    a.ldb = p.ldb;
    a.C = p.C;
    a.ldc = p.ldc;
    a.tiles_n = static_cast<int>(tiles_n);
    a.k_blocks = static_cast<int>(k_blocks);
    a.dp_tiles = sch.dp_tiles;
    a.sk_ctas = sch.sk_ctas;
    a.sk_iters = sch.sk_iters;
    a.timeout_ns = static_cast<uint64_t>(g_watchdog_ms.load()) * 1000000ull;
    a.watchdog = flag;
    a.alpha = p.alpha;
    a.beta = p.beta;
    a.strideA = p.strideA;
    a.strideB = p.strideB;
    a.strideC = p.strideC;
    a.tiles_per_item = static_cast<int>(tiles_m * tiles_n);
    a.a_shared = p.strideA == 0;
    a.b_shared = p.strideB == 0;
    a.bias = p.bias;
    a.bias_kind = p.bias_kind;
    a.act = p.act;
    a.ep = p.has_epilogue();
    a.kb_cap = 0;
    kernel<<<sch.grid, THREADS, SMEM_BYTES, stream>>>(a);
    ++*launches;
    if (cudaGetLastError() != cudaSuccess) return SGEMM_ERR_LAUNCH;
    return split_tiles_finish(p, BM, BN, static_cast<int>(tiles_n), static_cast<int>(tiles_m * tiles_n),
                              sch.dp_tiles, split, stream, launches);
}


PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        else
            cudaGetLastError();
    });
    return fn;
}

// TMA requirements: 16-byte aligned bases and row strides, coordinates that
// fit int32.
// Sizes a tensor map can describe, and the driver entry point that encodes one.
bool tma_sizes_ok(const Problem &p) {
    return p.M < INT32_MAX / 2 && p.N < INT32_MAX / 2 && p.K < INT32_MAX / 2 && p.batch < INT32_MAX / 2 &&
           tensor_map_encoder() != nullptr;
}

bool tma_ok(const Problem &p) {
    return tma_operand_ok(p.A, p.lda, p.strideA, p.transA ? p.K : p.M, p.batch) &&
           tma_operand_ok(p.B, p.ldb, p.strideB, p.transB ? p.N : p.K, p.batch) && tma_sizes_ok(p);
}

std::once_flag g_tma_attr_once[kMaxDevices][16];
cudaError_t g_tma_attr_err[kMaxDevices][16];

// V3 = A in TMEM (tf32x3_tmem_kernel, every operand form), else the TMA
// variant (tf32x3_tma_kernel, op(A) = A and op(B) = B only).
template <bool V3, bool VEC_C, bool TA = false, bool TB = false>
int launch_tma(const Problem &p, const DeviceInfo &dev, int sk_mode, cudaStream_t stream, int *launches) {
    static_assert(V3 || (!TA && !TB), "the TMA variant serves op(A) = A, op(B) = B only");
    auto kernel = V3 ? tf32x3_tmem_kernel<VEC_C, TA, TB> : tf32x3_tma_kernel<VEC_C>;
    constexpr int smem = V3 ? tm3::SMEM_BYTES : tma::SMEM_BYTES;
    constexpr int threads = V3 ? tm3::THREADS : tma::THREADS;
    constexpr int idx = (V3 ? 2 : 0) + (VEC_C ? 1 : 0) + (TA ? 4 : 0) + (TB ? 8 : 0);
    std::call_once(g_tma_attr_once[dev.device][idx], [&] {
        g_tma_attr_err[dev.device][idx] = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    });
    if (g_tma_attr_err[dev.device][idx] != cudaSuccess) {
        cudaGetLastError();
        return SGEMM_ERR_LAUNCH;
    }
    int *flag = watchdog_flag_device_ptr();
    if (!flag) return SGEMM_ERR_LAUNCH;
    alignas(64) CUtensorMap mapA, mapB;
    const bool ok_a =
        TA ? encode_map(&mapA, p.A, p.K, p.M, p.lda, p.batch, p.strideA, 32, 32, CU_TENSOR_MAP_SWIZZLE_128B)
           : encode_map(&mapA, p.A, p.M, p.K, p.lda, p.batch, p.strideA, BK, BM, CU_TENSOR_MAP_SWIZZLE_128B);
    const bool ok_b =
        TB ? encode_map(&mapB, p.B, p.N, p.K, p.ldb, p.batch, p.strideB, BK, BN, CU_TENSOR_MAP_SWIZZLE_128B)
           : encode_map(&mapB, p.B, p.K, p.N, p.ldb, p.batch, p.strideB, BN, BK, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (!ok_a || !ok_b) return SGEMM_ERR_LAUNCH;

    const int64_t tiles_m = (p.M + BM - 1) / BM, tiles_n = (p.N + BN - 1) / BN;
    const int64_t k_blocks = (p.K + BK - 1) / BK;
    if (tiles_m * tiles_n * p.batch > INT32_MAX / 2) return SGEMM_ERR_UNSUPPORTED;
    const int tiles = static_cast<int>(tiles_m * tiles_n * p.batch);
    const bool long_k = k_blocks > KB_CAP;  // every tile split, units of <= KB_CAP k-blocks
    const Schedule sch = make_schedule(tiles, k_blocks, dev.sm_count, long_k ? SK_ALL : sk_mode, 4, 0.25);
    const int split = tiles - sch.dp_tiles;
    int rc = split_tiles_prepare(p, BM, BN, static_cast<int>(tiles_n), static_cast<int>(tiles_m * tiles_n),
                                 sch.dp_tiles, split, stream, launches);
    if (rc != SGEMM_OK) return rc;
    Args a{};
    a.M = p.M;
    a.N = p.N;
    a.K = p.K;
    a.A = p.A;
    a.lda = p.lda;
    a.B = p.B;
    a.ldb = p.ldb;
    a.ta = TA ? 1 : 0;
    a.tb = TB ? 1 : 0;
    a.C = p.C;
    a.ldc = p.ldc;
    a.tiles_n = static_cast<int>(tiles_n);
    a.k_blocks = static_cast<int>(k_blocks);
    a.dp_tiles = sch.dp_tiles;
    a.sk_ctas = sch.sk_ctas;
    a.sk_iters = sch.sk_iters;
    a.timeout_ns = static_cast<uint64_t>(g_watchdog_ms.load()) * 1000000ull;
    a.watchdog = flag;
    a.alpha = p.alpha;
    a.beta = p.beta;
    a.strideA = p.strideA;
    a.strideB = p.strideB;
    a.strideC = p.strideC;
    a.tiles_per_item = static_cast<int>(tiles_m * tiles_n);
    a.a_shared = p.strideA == 0;
    a.b_shared = p.strideB == 0;
    a.bias = p.bias;
    a.bias_kind = p.bias_kind;
    a.act = p.act;
    a.ep = p.has_epilogue();
    a.kb_cap = long_k ? KB_CAP : 0;
    kernel<<<sch.grid, threads, smem, stream>>>(mapA, mapB, a);
    ++*launches;
    if (cudaGetLastError() != cudaSuccess) return SGEMM_ERR_LAUNCH;
    return split_tiles_finish(p, BM, BN, static_cast<int>(tiles_n), static_cast<int>(tiles_m * tiles_n),
                              sch.dp_tiles, split, stream, launches);
}

}  // namespace

namespace tc {

// A batch of row-major rows x cols fp32 matrices as a rank-3 tensor map (see
// tc_common.cuh).
bool encode_map(CUtensorMap *map, const float *ptr, int64_t rows, int64_t cols, int64_t ld, int64_t batch,
                int64_t stride, uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle swizzle) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    const int64_t items = stride == 0 ? 1 : batch;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                                static_cast<cuuint64_t>(items)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld) * sizeof(float),
                                   static_cast<cuuint64_t>(stride == 0 ? ld * rows : stride) * sizeof(float)};
    const cuuint32_t box[3] = {box_cols, box_rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(ptr), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace tc

int *watchdog_flag_device_ptr() {
    static std::once_flag once[kMaxDevices];
    static int *ptrs[kMaxDevices];
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return nullptr;
    }
    // Host code must not use the symbol itself: its device address comes from
    // the runtime, once per device.
    std::call_once(once[dev], [dev] {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_watchdog_code) != cudaSuccess) {
            cudaGetLastError();
            ptr = nullptr;
        }
        ptrs[dev] = static_cast<int *>(ptr);
    });
    return ptrs[dev];
}

int watchdog_read_and_clear(int *code) {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_watchdog_code, sizeof(int)) != cudaSuccess) {
        cudaGetLastError();
        return 1;
    }
    if (v != 0) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_watchdog_code, &zero, sizeof(int)) != cudaSuccess) {
            cudaGetLastError();
            return 1;
        }
    }
    *code = v;
    return 0;
}

int64_t watchdog_ms() { return g_watchdog_ms.load(); }

int watchdog_selftest_launch(int64_t wait_ms, cudaStream_t stream) {
    if (wait_ms < 1 || wait_ms > 60000) return SGEMM_ERR_INVALID_ARG;
    int *flag = watchdog_flag_device_ptr();
    if (!flag) return SGEMM_ERR_LAUNCH;
    watchdog_selftest_kernel<<<1, 32, 0, stream>>>(static_cast<uint64_t>(wait_ms) * 1000000ull, flag);
    return cudaGetLastError() == cudaSuccess ? SGEMM_OK : SGEMM_ERR_LAUNCH;
}

int tf32x3_set_kernel(int64_t mode) {
    if (mode < 0 || mode > 5) return SGEMM_ERR_INVALID_ARG;
    g_use_tma.store(static_cast<int>(mode));
    return SGEMM_OK;
}

int64_t tf32x3_get_kernel() { return g_use_tma.load(); }

int64_t tf32x3_last_kernel() { return g_last_tc_kernel.load(); }

int watchdog_set_ms(int64_t ms) {
    if (ms < 1 || ms > 60000) return SGEMM_ERR_INVALID_ARG;
    g_watchdog_ms.store(ms);
    return SGEMM_OK;
}

bool tf32x3_supports(const Problem &p, const DeviceInfo &dev) {
    // Every operand form at any alignment (the SM-pair kernel loads rows that
    // TMA cannot address with cp.async).
    return p.M > 0 && p.N > 0 && p.K > 0 && dev.cc_major == 10 && dev.cc_minor == 3 &&
           dev.smem_optin >= static_cast<size_t>(tma::SMEM_BYTES);
}

namespace {

// The TMA kernels, for operands a tensor map can describe: the SM-pair
// kernel from 2^20 multiply-adds on (or when forced), else the single-SM
// kernels. Measured on GB300, L2 flushed, pair vs tensor-memory kernel:
// 128^3 14.4 vs 15.7 us, 512^3 17.5 vs 22.2, 2048 x 128 x 512 17.2 vs 20.5,
// 200 x 4096 x 4096 52.4 vs 68.6, 1024^3 27.5 vs 33.4; all four forms.
// Batches of short products (K <= 256: at most 8 k-blocks per tile) stay on
// the tensor-memory kernel, whose tiles switch at less cost: 512 x 128^3
// 43.0 vs 55.8 us, 64 x 256^3 24.6 vs 31.8, 256 x 64^3 17.9 vs 26.6 (but
// 32 x 512^3 73.2 vs 51.2, and single products keep the pair kernel:
// 8192 x 8192 x 256 201.7 vs 148.1).
int launch_aligned(const Problem &p, const DeviceInfo &dev, int sk_mode, int mode, cudaStream_t stream,
                   int *launches, bool after_copy = false) {
    const bool vc = (p.ldc % 4 == 0) && (p.strideC % 4 == 0) && (reinterpret_cast<uintptr_t>(p.C) % 16 == 0);
    const double work = static_cast<double>(p.M) * static_cast<double>(p.N) * static_cast<double>(p.K) *
                        static_cast<double>(p.batch);
    const bool pair = mode == 4 || (mode == 0 && work >= 1048576.0 && !(p.batch > 1 && p.K <= 256));
    if (pair) {
        g_last_tc_kernel.store(4);
        return tf32x3_pair_launch(p, dev, sk_mode, false, stream, launches, after_copy);
    }
    g_last_tc_kernel.store(mode == 2 && !p.transA && !p.transB ? 2 : 3);
    if (p.transA && p.transB)
        return vc ? launch_tma<true, true, true, true>(p, dev, sk_mode, stream, launches)
                  : launch_tma<true, false, true, true>(p, dev, sk_mode, stream, launches);
    if (p.transA)
        return vc ? launch_tma<true, true, true, false>(p, dev, sk_mode, stream, launches)
                  : launch_tma<true, false, true, false>(p, dev, sk_mode, stream, launches);
    if (p.transB)
        return vc ? launch_tma<true, true, false, true>(p, dev, sk_mode, stream, launches)
                  : launch_tma<true, false, false, true>(p, dev, sk_mode, stream, launches);
    if (mode == 2)
        return vc ? launch_tma<false, true>(p, dev, sk_mode, stream, launches)
                  : launch_tma<false, false>(p, dev, sk_mode, stream, launches);
    return vc ? launch_tma<true, true>(p, dev, sk_mode, stream, launches)
              : launch_tma<true, false>(p, dev, sk_mode, stream, launches);
}

// Smallest product (multiply-adds) for which copying operands with
// unaligned rows into aligned scratch and running the TMA kernels beats the
// per-thread-load kernel (measured on GB300, L2 flushed, rows of K + 1 and
// N + 1 floats, per-thread loads vs copies + TMA kernels: 1023 x 1023 x 1025
// 39.5 vs 44.1 us, 1151 x 1151 x 1153 47.9 vs 47.1, 1279 x 1279 x 1281 53.8
// vs 52.5, 1407 x 1407 x 1409 66.1 vs 42.5, 511 x 4095 x 1025 53.8 vs 35.9,
// 1023 x 2049 x 1537 72.4 vs 50.4): 1.25 * 2^30.
constexpr double kRepackMinWork = 1342177280.0;

}  // namespace

int tf32x3_launch(const Problem &p, const DeviceInfo &dev, int sk_mode, cudaStream_t stream, int *launches) {
    if (!tf32x3_supports(p, dev) || dev.device < 0 || dev.device >= kMaxDevices) return SGEMM_ERR_UNSUPPORTED;
    const int mode = g_use_tma.load();
    // The transposed forms always take a TMA kernel (the per-thread-load
    // kernel serves op(A) = A, op(B) = B only).
    if (tma_ok(p) && (mode != 1 || p.transA || p.transB))
        return launch_aligned(p, dev, sk_mode, mode == 5 ? 0 : mode, stream, launches);
    return tf32x3_launch_unaligned(p, dev, sk_mode, stream, launches, nullptr, 0);
}

int tf32x3_launch_unaligned(const Problem &p, const DeviceInfo &dev, int sk_mode, cudaStream_t stream,
                            int *launches, float *scratch, size_t scratch_bytes) {
    const int mode = g_use_tma.load();
    const double work = static_cast<double>(p.M) * static_cast<double>(p.N) * static_cast<double>(p.K) *
                        static_cast<double>(p.batch);
    // Automatic (from kRepackMinWork on) or forced (5): copy the operands
    // whose rows TMA cannot address into rows of a multiple of 4 floats (a
    // memory-bound pass) and run the TMA kernels. Scratch: the caller's
    // buffer, else the library's stream-ordered pool, freed on `stream`
    // behind the product.
    if (((mode == 0 && work >= kRepackMinWork) || mode == 5) && tma_sizes_ok(p)) {
        const size_t bytes = repack_bytes(p);
        float *buf = scratch;
        if (!buf) buf = scratch_alloc(dev, bytes, stream);
        if (buf && (scratch == nullptr || scratch_bytes >= bytes)) {
            Problem q;
            int rc = repack_into(p, dev, buf, bytes, stream, &q, launches);
            if (rc == SGEMM_OK) rc = launch_aligned(q, dev, sk_mode, 0, stream, launches, true);
            if (!scratch) scratch_free(buf, stream);
            return rc;
        }
        if (scratch) return SGEMM_ERR_INVALID_ARG;
    }
    // Per-thread loads: the per-thread-load kernel for op(A) = A, op(B) = B;
    // the SM-pair kernel with cp.async loaders for the transposed forms
    // (which the per-thread-load kernel does not serve) or when forced (4).
    // Its 4-byte copies are slow to issue (measured on GB300: ~5.5 us for
    // one warp's half of a k-block, so 1023 x 2049 x 1537 with rows of 1537
    // and 2049 floats takes 309 us there against 86 us on the
    // per-thread-load kernel).
    if (p.transA || p.transB || mode == 4) {
        g_last_tc_kernel.store(4);
        return tf32x3_pair_launch(p, dev, sk_mode, true, stream, launches);
    }
    g_last_tc_kernel.store(1);
    const bool vc = (p.ldc % 4 == 0) && (p.strideC % 4 == 0) && (reinterpret_cast<uintptr_t>(p.C) % 16 == 0);
    const bool va = (p.lda % 4 == 0) && (p.strideA % 4 == 0) && (reinterpret_cast<uintptr_t>(p.A) % 16 == 0);
    const bool vb = (p.ldb % 4 == 0) && (p.strideB % 4 == 0) && (reinterpret_cast<uintptr_t>(p.B) % 16 == 0);
    const int idx = (va ? 4 : 0) + (vb ? 2 : 0) + (vc ? 1 : 0);
    switch (idx) {
        case 0: return launch<false, false, false>(p, dev, sk_mode, stream, launches);
        case 1: return launch<false, false, true>(p, dev, sk_mode, stream, launches);
        case 2: return launch<false, true, false>(p, dev, sk_mode, stream, launches);
        case 3: return launch<false, true, true>(p, dev, sk_mode, stream, launches);
        case 4: return launch<true, false, false>(p, dev, sk_mode, stream, launches);
        case 5: return launch<true, false, true>(p, dev, sk_mode, stream, launches);
        case 6: return launch<true, true, false>(p, dev, sk_mode, stream, launches);
        default: return launch<true, true, true>(p, dev, sk_mode, stream, launches);
    }
}

size_t tf32x3_copy_bytes(const Problem &p) {
    const int mode = g_use_tma.load();
    if (tma_ok(p) && (mode != 1 || p.transA || p.transB)) return 0;
    const double work = static_cast<double>(p.M) * static_cast<double>(p.N) * static_cast<double>(p.K) *
                        static_cast<double>(p.batch);
    if (((mode == 0 && work >= kRepackMinWork) || mode == 5) && tma_sizes_ok(p)) return repack_bytes(p);
    return 0;
}

int tf32x3_launch_with_scratch(const Problem &p, const DeviceInfo &dev, int sk_mode, cudaStream_t stream,
                               int *launches, float *scratch, size_t scratch_bytes) {
    if (!tf32x3_supports(p, dev) || dev.device < 0 || dev.device >= kMaxDevices) return SGEMM_ERR_UNSUPPORTED;
    const int mode = g_use_tma.load();
    if (tma_ok(p) && (mode != 1 || p.transA || p.transB))
        return launch_aligned(p, dev, sk_mode, mode == 5 ? 0 : mode, stream, launches);
    return tf32x3_launch_unaligned(p, dev, sk_mode, stream, launches, scratch, scratch_bytes);
}

}  // namespace sgemm
