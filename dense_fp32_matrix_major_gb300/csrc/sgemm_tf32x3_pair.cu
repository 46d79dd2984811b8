// Tensor-core SGEMM on SM pairs: tcgen05.mma.cta_group::2 (kind::tf32) with
// the three-term TF32 split of sgemm_tf32x3.cu, for all four operand forms
// (op(A) = A or A^T, op(B) = B or B^T) at any alignment: TMA loads the raw
// tiles where the rows are 16-byte aligned, 4-byte cp.async copies elsewhere.
//
// The product is the plain sum of "CUDA算子优化(4)：矩阵乘法", section
// "矩阵乘法的数学定义"; the pages give no tensor-core design (they name
// tensor cores once, "CUDA内存优化入门：从Naive到Tiled矩阵乘法", section 八).
//
// Accuracy: short accumulation chains, folded on chip. The tensor core adds
// each MMA's products into its fp32 accumulator with truncation (measured on
// GB300: about one unit in the last place of the running value per
// tcgen05.mma), so one accumulator that chains every MMA of a long K drifts
// in one direction when the terms share a sign (3.5e-5 of sum |a||b| at
// K = 16384 on U[0,1] inputs). Here an accumulator never chains more than
// FOLD_KB k-blocks (12 MMAs each): the pair's MMAs alternate between two
// accumulators in TMEM, and while the tensor core fills one, the epilogue
// warps add the other, rounded to nearest, into an fp32 running sum of the
// tile held in shared memory. The MMAs never wait for a fold.
//
// Why pairs. Two CTAs on two SMs of a cluster share one 256 x 128 tile: each
// holds 128 rows of A (split into hi / lo, in its TMEM) and 64 columns of B
// (hi / lo in its shared memory), and one MMA of 256 x 128 x 8 issued by the
// even CTA reads both halves. Each SM's shared memory then serves only half
// of the B operand the tensor core reads. (Measured on GB300: the 256 x 128
// x 8 and 256 x 256 x 8 tf32 MMAs run at the same multiply-add rate, 32.7
// and 65.4 ns each.) TMEM per CTA: two 128-column accumulators and four A
// stages of 64 columns (hi | lo for 32 values of k), all 512 columns.
//
// Roles in each CTA (23 warps):
//   * warp 0: in the even CTA, one thread issues the pair's MMAs (4 k-slices
//     x 3 products per k-block, lo*hi + hi*lo + hi*hi) into accumulator
//     d = (fold interval) mod 2 and commits them to the mbarriers of both
//     CTAs (multicast).
//   * warps 1 and 22: TMA of this CTA's A rows (128 x 32, 128-byte swizzled)
//     and B columns (32 x 64) into a 4-slot raw ring (one lane each), or,
//     for rows TMA cannot address, all lanes of both copying half of each
//     tile with 4-byte cp.async.
//   * warps 2-17 (converters, four groups of four warps, group g taking the
//     k-blocks it with it mod 4 = g; each warp of a group serves one TMEM
//     lane quarter): each thread splits one row of A (32 values) into hi /
//     lo and writes them to TMEM (tcgen05.st), and transposes and splits one
//     4 x 4 block of B into the K-major, 128-byte-swizzled hi / lo tiles of a
//     4-stage shared ring; then one lane per warp signals the even CTA's
//     stage-full barrier (a local arrival, or from the odd CTA an st.async
//     that completes transaction bytes on it).
//   * warps 18-21 (epilogue, one per TMEM lane quarter): for each fold
//     interval, read the finished accumulator's 128 columns of its 32 rows
//     (four 32 x 32 chunks), add them into the running sum (or start it) and
//     free the accumulator; after a unit's last interval, form the output
//     alpha * sum (+ bias, activation) in the running-sum chunk itself and
//     write it to C with one TMA bulk store (bulk reduce-add for tiles split
//     along K) per chunk. Chunks crossing the last row or column, C that TMA
//     cannot address, or beta != 0 take per-thread stores.
// Every wait is bounded in time as in the single-SM kernels; the pair meets
// at cluster barriers only at the start (mbarriers initialised) and at the
// end (before the TMEM of both is released).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "sgemm.h"
#include "sgemm_internal.h"
#include "tc_common.cuh"

namespace sgemm {
namespace {

using namespace tc;

namespace pr {

constexpr int PM = 256, PN = 128;  // C tile of a pair
constexpr int HM = 128, HN = 64;   // this CTA's rows of A, columns of B
// Longest chain of k-blocks one accumulator sums before it is folded into the
// running sum (tc::FOLD_KB = 8): 96 MMAs, ~5e-6 of sum |a||b| on non-negative
// inputs at any K.
constexpr int FOLD_KB = tc::FOLD_KB;
// Four operand stages (a stage is refilled only after the MMAs that read it
// have completed, and completions trail issue by the tensor pipe's queue)
// and four raw slots, one of each per converter group.
constexpr int OP_STAGES = 4, RAW_SLOTS = 4;
constexpr int B_HALF = HN * BK * 4;   // 8 KB: one of B hi / B lo, or raw B
constexpr int A_RAW = HM * BK * 4;    // 16 KB
constexpr int OP_STAGE = 2 * B_HALF;  // hi | lo
constexpr int SLOT = A_RAW + B_HALF;  // raw A | raw B
constexpr int RAW0 = OP_STAGES * OP_STAGE;
// Running sum: this CTA's 128 x 128 fp32 share of the tile as 16 chunks of
// 32 x 32 (chunk (q, c): rows 32q.., columns 32c..), rows of 128 bytes in the
// 128-byte swizzle, so a chunk is also the source of one TMA store of C.
constexpr int C_CHUNK = 32 * 32 * 4;
constexpr int R0 = RAW0 + RAW_SLOTS * SLOT;
constexpr int R_BYTES = (HM / 32) * (PN / 32) * C_CHUNK;
constexpr int CHUNKS = PN / 32;  // chunks per lane quarter
constexpr int GROUP_WARPS = 4, CONV_GROUPS = 4, CONV_WARPS = GROUP_WARPS * CONV_GROUPS, EPI_WARPS = 4;
constexpr int CONV_THREADS = 32 * GROUP_WARPS;  // threads converting one k-block
constexpr int EPI_WARP0 = 2 + CONV_WARPS;
// A second TMA issuer: a warp keeps only about one box in processing at a
// time (measured on GB300: ~0.4 us per box of 16-64 KB, whatever the ring
// depth), so A and B come from separate warps.
constexpr int TMA_B_WARP = EPI_WARP0 + EPI_WARPS;
constexpr int THREADS = 32 * (TMA_B_WARP + 1);
constexpr int BAR_OFFSET = R0 + R_BYTES;
constexpr int PBAR_BYTES = 256;
constexpr int SMEM_BYTES = BAR_OFFSET + PBAR_BYTES + 1024;
constexpr uint32_t TMEM_A = 2 * PN;  // A stages after the two 128-column accumulators
// Instruction descriptor: D fp32, A and B tf32, both K-major, N = 128, M = 256.
constexpr uint32_t kIdesc2 = (1u << 4) | (2u << 7) | (2u << 10) | (static_cast<uint32_t>(PN >> 3) << 17) |
                             (static_cast<uint32_t>(PM >> 4) << 24);
// mbarrier indices
constexpr int RAW_FULL = 0, RAW_FREE = RAW_FULL + RAW_SLOTS, OP_FULL = RAW_FREE + RAW_SLOTS,
              OP_EMPTY = OP_FULL + OP_STAGES, ACC_FULL = OP_EMPTY + OP_STAGES, ACC_EMPTY = ACC_FULL + 2,
              DRAIN = ACC_EMPTY + 2, NBARS = DRAIN + 1;
// The odd CTA's converter warps report a filled stage with st.async: a 4-byte
// store into the even CTA's shared memory that completes 4 bytes of
// transactions on its stage-full barrier with release semantics at cluster
// scope, without stalling the warp (a remote mbarrier.arrive.release.cluster
// held the arriving thread ~0.8 us per k-block on GB300, measured).
constexpr uint32_t SIGNAL_BYTES = 4 * GROUP_WARPS;
static_assert(NBARS * 8 + 24 <= PBAR_BYTES, "barrier block");
static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
static_assert(TMEM_A + OP_STAGES * 64 <= TMEM_COLS, "TMEM columns");
static_assert((HN / 4) * (BK / 4) == CONV_THREADS, "one 4 x 4 B block per converter thread");
static_assert(CONV_GROUPS == OP_STAGES && RAW_SLOTS == OP_STAGES, "group g owns raw slot g and stage g");
static_assert(SLOT % 1024 == 0 && RAW0 % 1024 == 0 && R0 % 1024 == 0, "1024-byte aligned swizzled buffers");

}  // namespace pr

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_sync() {
    cluster_arrive();
    cluster_wait();
}

// Arrive on the mbarrier at this CTA's shared offset `bar` in CTA `cta` of
// the cluster, releasing this thread's prior writes at cluster scope.
__device__ __forceinline__ void mbar_arrive_at(uint32_t bar, uint32_t cta) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(bar), "r"(cta));
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote) : "memory");
}

// st.async of a 4-byte word into CTA `cta`'s shared memory at this CTA's
// offset `word`, completing 4 bytes of transactions on the mbarrier at offset
// `bar` there. The completion has release semantics at cluster scope (this
// thread's prior writes, and those it has observed, are visible to a thread
// that sees the phase complete) and the issuing thread does not wait for it.
__device__ __forceinline__ void st_async_signal(uint32_t word, uint32_t bar, uint32_t cta) {
    uint32_t rw, rb;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rw) : "r"(word), "r"(cta));
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rb) : "r"(bar), "r"(cta));
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(rw), "r"(0u),
                 "r"(rb)
                 : "memory");
}

// One 256 x 128 x 8 product of the pair: A (128 rows per CTA) from TMEM, B
// (64 columns per CTA) from shared memory.
__device__ __forceinline__ void tc_mma2_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t accumulate) {
    asm volatile(
        "{\n"
        " .reg .pred p;\n"
        " setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::2.kind::tf32 [%0], [%1], %2, %3, p;\n"
        "}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(pr::kIdesc2), "r"(accumulate)
        : "memory");
}

// Arrive on the mbarrier at offset `bar` of both CTAs once the pair's MMAs
// issued so far have completed.
__device__ __forceinline__ void tc_commit2(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            bar),
        "h"(static_cast<uint16_t>(3))
        : "memory");
}

// Fused-epilogue values of 16 columns (chunk columns base .. base + 15)
// written to the swizzled chunk row of this lane: ACT(alpha * v + bias), the
// bias per row (bl) or per column (lane (base + j)'s bl, by shuffle).
template <int ACT>
__device__ __forceinline__ void stage16_ep(uint32_t buf, int lane, int base, float alpha, bool col_bias, float bl,
                                           const float *v) {
#pragma unroll
    for (int j = 0; j < 16; j += 4) {
        float b[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) b[t] = col_bias ? __shfl_sync(0xffffffffu, bl, base + j + t) : bl;
        st_shared_v4(buf + sw128_offset(lane, (base + j) >> 2), activate(alpha * v[j] + b[0], ACT),
                     activate(alpha * v[j + 1] + b[1], ACT), activate(alpha * v[j + 2] + b[2], ACT),
                     activate(alpha * v[j + 3] + b[3], ACT));
    }
}

__device__ __forceinline__ void stage32_fused(int act, uint32_t buf, int lane, float alpha, bool col_bias, float bl,
                                              const float (&v)[32]) {
    switch (act) {
        case SGEMM_ACT_RELU:
            stage16_ep<SGEMM_ACT_RELU>(buf, lane, 0, alpha, col_bias, bl, v);
            stage16_ep<SGEMM_ACT_RELU>(buf, lane, 16, alpha, col_bias, bl, v + 16);
            break;
        case SGEMM_ACT_GELU:
            stage16_ep<SGEMM_ACT_GELU>(buf, lane, 0, alpha, col_bias, bl, v);
            stage16_ep<SGEMM_ACT_GELU>(buf, lane, 16, alpha, col_bias, bl, v + 16);
            break;
        case SGEMM_ACT_SILU:
            stage16_ep<SGEMM_ACT_SILU>(buf, lane, 0, alpha, col_bias, bl, v);
            stage16_ep<SGEMM_ACT_SILU>(buf, lane, 16, alpha, col_bias, bl, v + 16);
            break;
        default:
            stage16_ep<SGEMM_ACT_NONE>(buf, lane, 0, alpha, col_bias, bl, v);
            stage16_ep<SGEMM_ACT_NONE>(buf, lane, 16, alpha, col_bias, bl, v + 16);
            break;
    }
}

// The last fold of a unit for a chunk written with per-thread stores: the
// unit's finished sum for rows row0 .. row0 + 31, columns col0 .. col0 + 31
// (chunk rc of shared memory, swizzled, lane l holding row row0 + l),
// repaired where it is NaN (recomputed over the unit's k-range [k_begin,
// k_end) of batch item `item`), then written one row per step with the lanes
// along the row (coalesced): C = act(alpha * v + beta * C + bias) for a
// whole tile, C += alpha * v with atomics for a tile split along K. Used for
// chunks that cross the last row or column of C, for C that TMA cannot
// address and for chunks holding a NaN; called by all 32 lanes. Out of line:
// it is rare, and inlined it would compete for registers with the interior
// path.
template <bool VEC_C>
__device__ __noinline__ void edge_final_chunk(const Args &a, uint32_t rc, float *citem, int64_t row0, int64_t col0,
                                              bool atomic, int item, int64_t k_begin, int64_t k_end) {
    const int lane = static_cast<int>(threadIdx.x & 31);
    if (col0 >= a.N) return;  // uniform over the warp
    const int64_t row = row0 + lane;
    bool nan = false;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const float4 r = ld_shared_v4(rc + sw128_offset(lane, j));
        nan |= r.x != r.x || r.y != r.y || r.z != r.z || r.w != r.w;
    }
    if (nan && row < a.M) {
        // Repair in shared memory, one column at a time (few registers).
        const float *A = a.A + (a.a_shared ? 0 : item * a.strideA);
        const float *B = a.B + (a.b_shared ? 0 : item * a.strideB);
        if (k_end > a.K) k_end = a.K;
#pragma unroll 1
        for (int j = 0; j < 32 && col0 + j < a.N; ++j) {
            const uint32_t addr = rc + sw128_offset(lane, j >> 2) + static_cast<uint32_t>((j & 3) * 4);
            const float x = ld_shared_f32(addr);
            if (x != x) st_shared_f32(addr, dot_ieee(A, a.lda, a.ta, B, a.ldb, a.tb, row, col0 + j, k_begin, k_end));
        }
    }
    __syncwarp();
    store_staged_rows(a, rc, citem, row0, col0, atomic);
}

// TA: A stored K x M (op(A) = A^T); TB: B stored N x K (op(B) = B^T).
template <bool VEC_C, bool TA, bool TB>
__global__ void __launch_bounds__(pr::THREADS, 1)
    tf32x3_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                       const __grid_constant__ CUtensorMap tmC, const __grid_constant__ Args a) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (base - raw);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + pr::BAR_OFFSET);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(bars + pr::NBARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + pr::NBARS + 1);
    // Target word of the odd CTA's st.async signals (its value is not used).
    const uint32_t signal_word = smem_u32(bars + pr::NBARS + 2);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const int pair = static_cast<int>(blockIdx.x >> 1), pairs = static_cast<int>(gridDim.x >> 1);
    auto bar = [&](int i) { return smem_u32(bars + i); };

    // TMA of this CTA's A rows (warp 1) or B columns (warp TMA_B_WARP) for
    // the k-blocks it = from .. to - 1 of its units, into the raw ring.
    const bool tma_warp = warp == 1 || warp == pr::TMA_B_WARP;
    auto tma_pass = [&](uint32_t from, uint32_t to) {
        if (a.wait_inputs) asm volatile("griddepcontrol.wait;" ::: "memory");
        const bool is_a = warp == 1;
        uint32_t it = 0;
        bool ok = true;
        for_each_unit_of(a, abort_flag, pair, pairs, [&](int tile, int kb, int ke) {
            if (!ok || it >= to) return;
            if (it + static_cast<uint32_t>(ke - kb) <= from) {
                it += static_cast<uint32_t>(ke - kb);
                return;
            }
            const TileAt at = tile_at<pr::PM, pr::PN>(a, tile);
            const int m0 = static_cast<int>(at.m0) + pr::HM * static_cast<int>(rank);
            const int n0 = static_cast<int>(at.n0) + pr::HN * static_cast<int>(rank);
            const int za = a.a_shared ? 0 : at.item, zb = a.b_shared ? 0 : at.item;
            for (int kblk = kb; kblk < ke && it < to; ++kblk, ++it) {
                if (it < from) continue;
                const int slot = static_cast<int>(it % pr::RAW_SLOTS);
                const uint32_t ph = (it / pr::RAW_SLOTS) & 1;
                if (!mbar_wait(bar(pr::RAW_FREE + slot), ph ^ 1, a, abort_flag, WD_PRODUCER)) {
                    ok = false;
                    return;
                }
                const uint32_t sl = base + pr::RAW0 + static_cast<uint32_t>(slot * pr::SLOT);
                if (is_a) {
                    mbar_arrive_expect_tx(bar(pr::RAW_FULL + slot), pr::A_RAW);
                    if (TA) {  // A stored K x M: four boxes of 32 m x 32 k
#pragma unroll
                        for (int b = 0; b < pr::HM / 32; ++b)
                            tma_load_3d(sl + b * 4096, &tmA, m0 + 32 * b, kblk * BK, za, bar(pr::RAW_FULL + slot));
                    } else {
                        tma_load_3d(sl, &tmA, kblk * BK, m0, za, bar(pr::RAW_FULL + slot));
                    }
                } else {
                    mbar_arrive_expect_tx(bar(pr::RAW_FULL + slot), pr::B_HALF);
                    if (TB)  // B stored N x K: already K-major, 64 rows of 32 k
                        tma_load_3d(sl + pr::A_RAW, &tmB, kblk * BK, n0, zb, bar(pr::RAW_FULL + slot));
                    else
                        tma_load_3d(sl + pr::A_RAW, &tmB, n0, kblk * BK, zb, bar(pr::RAW_FULL + slot));
                }
            }
        });
    };

    // The same ring filled with 4-byte cp.async copies (a.cpa: rows that TMA
    // cannot address), by all lanes of warps 1 and TMA_B_WARP, each copying
    // half of this CTA's A tile and half of its B tile in the layouts the TMA
    // boxes have (A, and B stored N x K, in the 128-byte swizzle; B stored
    // K x N plain), zero outside the matrices. Every lane's copies for a slot
    // are tracked by one cp.async arrival on the slot's full barrier.
    auto load_pass = [&](uint32_t from, uint32_t to) {
        if (a.wait_inputs) asm volatile("griddepcontrol.wait;" ::: "memory");
        const int half = warp == 1 ? 0 : 1;
        uint32_t it = 0;
        bool ok = true;
        for_each_unit_of(a, abort_flag, pair, pairs, [&](int tile, int kb, int ke) {
            if (!ok || it >= to) return;
            if (it + static_cast<uint32_t>(ke - kb) <= from) {
                it += static_cast<uint32_t>(ke - kb);
                return;
            }
            const TileAt at = tile_at<pr::PM, pr::PN>(a, tile);
            const int64_t m0 = at.m0 + pr::HM * static_cast<int64_t>(rank);
            const int64_t n0 = at.n0 + pr::HN * static_cast<int64_t>(rank);
            const float *Ai = a.A + (a.a_shared ? 0 : at.item * a.strideA);
            const float *Bi = a.B + (a.b_shared ? 0 : at.item * a.strideB);
            for (int kblk = kb; kblk < ke && it < to; ++kblk, ++it) {
                if (it < from) continue;
                const int slot = static_cast<int>(it % pr::RAW_SLOTS);
                const bool free = mbar_wait(bar(pr::RAW_FREE + slot), ((it / pr::RAW_SLOTS) & 1) ^ 1, a, abort_flag,
                                            WD_PRODUCER);
                if (!__all_sync(0xffffffffu, free)) {
                    ok = false;
                    return;
                }
                const uint32_t sl = base + pr::RAW0 + static_cast<uint32_t>(slot * pr::SLOT);
                const int64_t k0 = static_cast<int64_t>(kblk) * BK;
                const uint32_t lo4 = static_cast<uint32_t>((lane & 3) * 4);
                if (TA) {
                    // A stored K x M: boxes 2 half, 2 half + 1 of 32 k-rows x 32 m; lane = m.
                    for (int bx = 2 * half; bx < 2 * half + 2; ++bx) {
                        const int64_t m = m0 + 32 * bx + lane;
                        for (int r = 0; r < 32; ++r) {
                            const int64_t k = k0 + r;
                            const bool v = k < a.K && m < a.M;
                            cp_async4(sl + static_cast<uint32_t>(bx * 4096) + sw128_offset(r, lane >> 2) + lo4,
                                      v ? Ai + k * a.lda + m : Ai, v);
                        }
                    }
                } else {
                    // A rows 64 half .. 64 half + 63 of the tile; lane = k.
                    const int64_t k = k0 + lane;
                    for (int r = 64 * half; r < 64 * half + 64; ++r) {
                        const int64_t m = m0 + r;
                        const bool v = k < a.K && m < a.M;
                        cp_async4(sl + sw128_offset(r, lane >> 2) + lo4, v ? Ai + m * a.lda + k : Ai, v);
                    }
                }
                const uint32_t sb = sl + pr::A_RAW;
                if (TB) {
                    // B stored N x K: n-rows 32 half .. 32 half + 31 of 32 k; lane = k.
                    const int64_t k = k0 + lane;
                    for (int r = 32 * half; r < 32 * half + 32; ++r) {
                        const int64_t n = n0 + r;
                        const bool v = k < a.K && n < a.N;
                        cp_async4(sb + sw128_offset(r, lane >> 2) + lo4, v ? Bi + n * a.ldb + k : Bi, v);
                    }
                } else {
                    // B stored K x N: k-rows 16 half .. 16 half + 15 of 64 n (plain rows of 256 bytes).
                    for (int r = 16 * half; r < 16 * half + 16; ++r) {
                        const int64_t k = k0 + r;
#pragma unroll
                        for (int c2 = 0; c2 < 2; ++c2) {
                            const int64_t n = n0 + 32 * c2 + lane;
                            const bool v = k < a.K && n < a.N;
                            cp_async4(sb + static_cast<uint32_t>(r * pr::HN * 4 + (32 * c2 + lane) * 4),
                                      v ? Bi + k * a.ldb + n : Bi, v);
                        }
                    }
                }
                cp_async_arrive(bar(pr::RAW_FULL + slot));
            }
        });
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < pr::RAW_SLOTS; ++s) {
            // One expect_tx arrival per TMA issuer, or one cp.async arrival
            // per lane of the two loader warps.
            mbar_init(bar(pr::RAW_FULL + s), a.cpa ? 64 : 2);
            mbar_init(bar(pr::RAW_FREE + s), pr::GROUP_WARPS);  // one lane per converter warp
        }
        for (int s = 0; s < pr::OP_STAGES; ++s) {
            // Even CTA: one arrival per own converter warp (the first also
            // expects SIGNAL_BYTES), and SIGNAL_BYTES of transactions from the
            // odd CTA's converter warps (st.async, see below).
            mbar_init(bar(pr::OP_FULL + s), pr::GROUP_WARPS);
            mbar_init(bar(pr::OP_EMPTY + s), 1);
        }
        for (int d = 0; d < 2; ++d) {
            mbar_init(bar(pr::ACC_FULL + d), 1);
            mbar_init(bar(pr::ACC_EMPTY + d), 2 * pr::EPI_WARPS);
        }
        mbar_init(bar(pr::DRAIN), 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (tma_warp && lane == 0 && !a.cpa) {
        const bool is_a = warp == 1;
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(is_a ? &tmA : &tmB)) : "memory");
    }
    __syncthreads();  // this CTA's mbarriers are initialised
    if (warp == 0) {
        // Both CTAs allocate: the pair's MMAs use the same columns in each.
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_holder)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    // The cluster barrier publishes the peer's mbarriers before anyone
    // arrives on them, and the TMEM address to this CTA. The first loads
    // signal only this CTA's barriers, so the TMA issuers send them while the
    // pair meets (after their arrival, whose release would otherwise wait for
    // the loads).
    cluster_arrive();
    if (tma_warp) {
        if (a.cpa)
            load_pass(0, pr::RAW_SLOTS);
        else if (lane == 0)
            tma_pass(0, pr::RAW_SLOTS);
    }
    __syncwarp();
    cluster_wait();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    // A pass launched behind this kernel (the activation of split tiles) may
    // be scheduled now; it waits for this grid to finish before touching C.
    if (a.signal_dependents && threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;");

    if (warp == 0) {
        // ------------------------------------------------------------ MMA issuer
        // A 256 x 128 x 8 MMA takes ~33 ns and the tensor core queues only a
        // few, so the issuer's own work between MMAs shows as idle tensor
        // time. The whole warp runs the loop (its values stay warp-uniform)
        // and one elected lane issues; the stage addresses are one add from
        // precomputed bases, and the next stage's barrier is tested while this
        // k-block's last k-slice is still queued.
        if (rank == 0) {
            const bool leader = elect_one();
            uint32_t it = 0, iv = 0;  // k-blocks and fold intervals issued so far
            const uint64_t desc0 = sw128_desc(base);
            const uint32_t a0 = tmem_base + pr::TMEM_A;
            bool ready = false;  // the stage of k-block `it` was seen full (and fenced) early
            for_each_unit_of(a, abort_flag, pair, pairs, [&](int, int kb, int ke) {
                for (int k0 = kb; k0 < ke; k0 += pr::FOLD_KB) {
                    const int k1 = ke - k0 > pr::FOLD_KB ? k0 + pr::FOLD_KB : ke;
                    const uint32_t d = iv & 1;
                    // Accumulator d is free once the epilogue has folded the
                    // interval that used it two intervals back.
                    const bool ok = mbar_wait<true>(bar(pr::ACC_EMPTY + d), ((iv >> 1) & 1) ^ 1, a, abort_flag,
                                                    WD_MMA_ACC);
                    if (!__all_sync(0xffffffffu, ok)) return;
                    tc_fence_after();
                    const uint32_t dt = tmem_base + d * pr::PN;
                    for (int kblk = k0; kblk < k1; ++kblk, ++it) {
                        const uint32_t s = it % pr::OP_STAGES;
                        if (!ready) {
                            const bool full = mbar_wait<true>(bar(pr::OP_FULL + s), (it / pr::OP_STAGES) & 1, a,
                                                              abort_flag, WD_MMA_FULL);
                            if (!__all_sync(0xffffffffu, full)) return;
                            tc_fence_after();
                        }
                        const uint64_t b_hi = desc0 + static_cast<uint64_t>(s * (pr::OP_STAGE >> 4));
                        const uint64_t b_lo = b_hi + (pr::B_HALF >> 4);
                        const uint32_t a_hi = a0 + 64 * s, a_lo = a_hi + 32;
                        const uint32_t acc0 = kblk == k0 ? 0u : 1u;  // each interval starts its accumulator
#pragma unroll
                        for (int ks = 0; ks < BK / 8; ++ks) {
                            const uint64_t adv = static_cast<uint64_t>(ks * 2);
                            const uint32_t ac = static_cast<uint32_t>(ks * 8);
                            if (ks == BK / 8 - 1) {
                                // The next k-block's stage, tested without blocking.
                                const uint32_t nx = it + 1;
                                ready = __all_sync(0xffffffffu, mbar_test_wait<true>(bar(pr::OP_FULL + nx % pr::OP_STAGES),
                                                                                     (nx / pr::OP_STAGES) & 1));
                                if (ready) tc_fence_after();
                            }
                            if (leader) {
                                tc_mma2_ts(dt, a_lo + ac, b_hi + adv, ks == 0 ? acc0 : 1u);
                                tc_mma2_ts(dt, a_hi + ac, b_lo + adv, 1u);
                                tc_mma2_ts(dt, a_hi + ac, b_hi + adv, 1u);
                            }
                            __syncwarp();
                        }
                        if (leader) tc_commit2(bar(pr::OP_EMPTY + s));
                        __syncwarp();
                    }
                    if (leader) tc_commit2(bar(pr::ACC_FULL + d));
                    __syncwarp();
                    ++iv;
                }
            });
            if (leader) tc_commit2(bar(pr::DRAIN));
            __syncwarp();
            if (lane == 0) {
                const bool was_aborted = *abort_flag != 0;
                if (!mbar_wait(bar(pr::DRAIN), 0, a, abort_flag, WD_DRAIN) && was_aborted) {
                    const uint64_t t0 = global_timer();
                    while (!mbar_try_wait(bar(pr::DRAIN), 0) && global_timer() - t0 < a.timeout_ns) {
                    }
                }
            }
        }
    } else if (tma_warp) {
        // ---------------------------------------------------- TMA issuers (A, B)
        if (a.cpa)
            load_pass(pr::RAW_SLOTS, 0xffffffffu);
        else if (lane == 0)
            tma_pass(pr::RAW_SLOTS, 0xffffffffu);
    } else if (warp < pr::EPI_WARP0) {
        // ------------------------------------------------------------ converters
        const int cw = warp - 2;                                 // 0 .. 15
        const uint32_t group = static_cast<uint32_t>(cw >> 2);  // k-blocks with it % 4 == group
        const int ct = ((cw & 3) << 5) + lane;                   // 0 .. 127 within the group
        const int l = ct & 7, tb = ct >> 3;                      // 16 groups of eight lanes
        const int g = (tb >> 3) * 8 + l, c = (l + tb) & 7;       // this thread's 4 x 4 B block
        const int q = warp & 3;                                  // TMEM lane quarter
        const int arow = 32 * q + lane;                          // A row this thread converts
        uint32_t it = 0;
        bool ok = true;
        for_each_unit_of(a, abort_flag, pair, pairs, [&](int, int kb, int ke) {
            if (!ok) return;
            for (int kblk = kb; kblk < ke; ++kblk, ++it) {
                if (it % pr::CONV_GROUPS != group) continue;
                const int slot = static_cast<int>(it % pr::RAW_SLOTS);
                const int s = static_cast<int>(it % pr::OP_STAGES);
                if (!mbar_wait(bar(pr::RAW_FULL + slot), (it / pr::RAW_SLOTS) & 1, a, abort_flag, WD_PRODUCER)) {
                    ok = false;
                    return;
                }
                const uint32_t sl = base + pr::RAW0 + static_cast<uint32_t>(slot * pr::SLOT);
                // A: the 32 k-values of row arow.
                float av[32];
                if (TA) {
                    // Box q holds rows k = 0..31 of columns m = 32q..32q+31 (128-byte
                    // swizzled): column arow is lane `lane` of each row.
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        av[j] = ld_shared_f32(sl + static_cast<uint32_t>(q * 4096) + sw128_offset(j, lane >> 2) +
                                              static_cast<uint32_t>((lane & 3) * 4));
                } else {
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const float4 t = ld_shared_v4(sl + sw128_offset(arow, j));
                        av[4 * j] = t.x;
                        av[4 * j + 1] = t.y;
                        av[4 * j + 2] = t.z;
                        av[4 * j + 3] = t.w;
                    }
                }
                // B: op(B) = B: rows 4c..4c+3, columns 4g..4g+3 of the unswizzled 32 x 64
                // staging tile; op(B) = B^T: four 16-byte chunks of the K-major tile.
                float4 bq[4];
#pragma unroll
                for (int qq = 0; qq < 4; ++qq)
                    bq[qq] = TB ? ld_shared_v4(sl + pr::A_RAW + static_cast<uint32_t>((qq * pr::CONV_THREADS + ct) * 16))
                                : ld_shared_v4(sl + pr::A_RAW +
                                               static_cast<uint32_t>((4 * c + qq) * pr::HN * 4 + g * 16));
                fence_proxy_async_smem();  // order these loads before the next TMA into the slot
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(pr::RAW_FREE + slot));
                // The stage is free once the pair's MMAs four k-blocks back are done.
                if (!mbar_wait<true>(bar(pr::OP_EMPTY + s), ((it / pr::OP_STAGES) & 1) ^ 1, a, abort_flag,
                                     WD_PRODUCER)) {
                    ok = false;
                    return;
                }
                tc_fence_after();
                const uint32_t st = base + static_cast<uint32_t>(s * pr::OP_STAGE);
                if (TB) {
                    // Same swizzled K-major layout: chunk for chunk.
#pragma unroll
                    for (int qq = 0; qq < 4; ++qq) {
                        const uint32_t off = static_cast<uint32_t>((qq * pr::CONV_THREADS + ct) * 16);
                        split_store(st + off, st + pr::B_HALF + off, bq[qq].x, bq[qq].y, bq[qq].z, bq[qq].w);
                    }
                } else {
                    // Column j of the 4 x 4 block is chunk c of operand row 4g + j.
                    uint32_t off = sw128_offset(4 * g + 0, c);
                    split_store(st + off, st + pr::B_HALF + off, bq[0].x, bq[1].x, bq[2].x, bq[3].x);
                    off = sw128_offset(4 * g + 1, c);
                    split_store(st + off, st + pr::B_HALF + off, bq[0].y, bq[1].y, bq[2].y, bq[3].y);
                    off = sw128_offset(4 * g + 2, c);
                    split_store(st + off, st + pr::B_HALF + off, bq[0].z, bq[1].z, bq[2].z, bq[3].z);
                    off = sw128_offset(4 * g + 3, c);
                    split_store(st + off, st + pr::B_HALF + off, bq[0].w, bq[1].w, bq[2].w, bq[3].w);
                }
                const uint32_t ta =
                    tmem_base + (static_cast<uint32_t>(32 * q) << 16) + pr::TMEM_A + static_cast<uint32_t>(64 * s);
#pragma unroll
                for (int h = 0; h < 4; ++h) {  // 8 values at a time: fewer live registers
                    float hi[8], lo[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) split_tf32(av[8 * h + j], hi[j], lo[j]);
                    tmem_store8(ta + 8 * h, hi);
                    tmem_store8(ta + 32 + 8 * h, lo);
                }
                tmem_wait_st();
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if (rank != 0)
                        st_async_signal(signal_word, bar(pr::OP_FULL + s), 0);  // the even CTA issues the MMAs
                    else if ((cw & 3) == 0)
                        mbar_arrive_expect_tx(bar(pr::OP_FULL + s), pr::SIGNAL_BYTES);
                    else
                        mbar_arrive(bar(pr::OP_FULL + s));
                }
            }
        });
    } else {
        // -------------------------------------------------------------- epilogue
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const uint32_t rq = base + pr::R0 + static_cast<uint32_t>(q * pr::CHUNKS * pr::C_CHUNK);  // its chunks
        // C may still be in the beta pre-pass launched just before this
        // kernel (programmatic dependent launch): only the epilogue waits.
        asm volatile("griddepcontrol.wait;" ::: "memory");
        uint32_t iv = 0;  // fold intervals consumed so far
        auto release = [&](uint32_t d) {
            // Accumulator d is out of TMEM: one lane per warp frees it on the
            // even CTA's barrier.
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_at(bar(pr::ACC_EMPTY + d), 0);
        };
        for_each_unit_of(a, abort_flag, pair, pairs, [&](int tile, int kb, int ke) {
            const TileAt at = tile_at<pr::PM, pr::PN>(a, tile);
            const int64_t row0 = at.m0 + pr::HM * static_cast<int64_t>(rank) + q * 32;
            const int64_t row = row0 + lane;
            // Stream-K tiles hold beta * C + bias already: every unit adds.
            const bool atomic = tile >= a.dp_tiles;
            const bool fused = a.ep && !atomic;
            const bool col_bias = a.bias_kind == SGEMM_BIAS_PER_COL;
            const float rb = (a.bias_kind == SGEMM_BIAS_PER_ROW && row < a.M) ? __ldg(a.bias + row) : 0.0f;
            // The previous unit's TMA stores read the running sum: wait until
            // they have, before this unit overwrites it.
            if (lane == 0) bulk_wait_read<0>();
            __syncwarp();
            for (int k0 = kb; k0 < ke; k0 += pr::FOLD_KB) {
                const bool first = k0 == kb, last = ke - k0 <= pr::FOLD_KB;
                const uint32_t d = iv & 1;
                if (!mbar_wait<true>(bar(pr::ACC_FULL + d), (iv >> 1) & 1, a, abort_flag, WD_EPILOGUE)) return;
                tc_fence_after();
                ++iv;
                const uint32_t dt = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + d * pr::PN;
#pragma unroll 1
                for (int ch = 0; ch < pr::CHUNKS; ++ch) {
                    const uint32_t rc = rq + static_cast<uint32_t>(ch * pr::C_CHUNK);
                    const int64_t col0 = at.n0 + ch * 32;
                    float v[32];
                    tmem_load32(dt + static_cast<uint32_t>(ch * 32), v);
                    if (ch == pr::CHUNKS - 1) release(d);
                    if (!first) {
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const float4 r = ld_shared_v4(rc + sw128_offset(lane, j));
                            v[4 * j] += r.x;
                            v[4 * j + 1] += r.y;
                            v[4 * j + 2] += r.z;
                            v[4 * j + 3] += r.w;
                        }
                    }
                    if (!last) {
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            st_shared_v4(rc + sw128_offset(lane, j), v[4 * j], v[4 * j + 1], v[4 * j + 2],
                                         v[4 * j + 3]);
                        continue;
                    }
                    // The unit's sum is complete: write this chunk of C.
                    bool nan = false;
#pragma unroll
                    for (int j = 0; j < 32; ++j) nan |= v[j] != v[j];
                    if (__any_sync(0xffffffffu, nan) || !a.c_tma || col0 + 32 > a.N || row0 + 32 > a.M) {
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            st_shared_v4(rc + sw128_offset(lane, j), v[4 * j], v[4 * j + 1], v[4 * j + 2],
                                         v[4 * j + 3]);
                        edge_final_chunk<VEC_C>(a, rc, a.C + at.item * a.strideC, row0, col0, atomic, at.item,
                                                static_cast<int64_t>(kb) * BK, static_cast<int64_t>(ke) * BK);
                        continue;
                    }
                    if (fused) {
                        // Per-column bias of this chunk: lane l holds column col0 + l.
                        const float bl = col_bias ? __ldg(a.bias + col0 + lane) : rb;
                        stage32_fused(a.act, rc, lane, a.alpha, col_bias, bl, v);
                    } else {
                        const float alpha = a.alpha;
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            st_shared_v4(rc + sw128_offset(lane, j), alpha * v[4 * j], alpha * v[4 * j + 1],
                                         alpha * v[4 * j + 2], alpha * v[4 * j + 3]);
                    }
                    fence_proxy_async_smem();  // chunk writes -> visible to the TMA engine
                    __syncwarp();
                    if (lane == 0) {
                        const int x = static_cast<int>(col0), y = static_cast<int>(row0);
                        if (atomic)
                            tma_reduce_add_3d(&tmC, x, y, at.item, rc);
                        else
                            tma_store_3d(&tmC, x, y, at.item, rc);
                        bulk_commit();
                    }
                }
            }
        });
        if (lane == 0) bulk_wait<0>();  // every store of this warp has landed
    }

    // The odd CTA's TMEM is written by the even CTA's MMAs: wait for them to
    // drain before the pair releases it.
    tc_fence_before();
    __syncthreads();
    if (rank != 0 && threadIdx.x == 0) {
        if (!mbar_wait<true>(bar(pr::DRAIN), 0, a, abort_flag, WD_DRAIN)) {
            const uint64_t t0 = global_timer();
            while (!mbar_try_wait<true>(bar(pr::DRAIN), 0) && global_timer() - t0 < a.timeout_ns) {
            }
        }
    }
    __syncthreads();
    cluster_sync();
    tc_fence_after();
    if (warp == 0) {
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS)
                     : "memory");
    }
}

constexpr int kMaxDevices = 64;
std::once_flag g_pair_once[kMaxDevices][8];
cudaError_t g_pair_err[kMaxDevices][8];
int g_pair_clusters[kMaxDevices][8];

template <bool VEC_C, bool TA, bool TB>
int launch_pair(const Problem &p, const DeviceInfo &dev, int sk_mode, bool cpa, bool after_copy, cudaStream_t stream,
                int *launches) {
    auto kernel = tf32x3_pair_kernel<VEC_C, TA, TB>;
    constexpr int idx = (VEC_C ? 1 : 0) + (TA ? 2 : 0) + (TB ? 4 : 0);
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg{};
    cfg.blockDim = dim3(pr::THREADS);
    cfg.dynamicSmemBytes = pr::SMEM_BYTES;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    std::call_once(g_pair_once[dev.device][idx], [&] {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, pr::SMEM_BYTES);
        int n = 0;
        if (e == cudaSuccess) {
            cudaLaunchConfig_t q = cfg;
            q.gridDim = dim3(2 * (dev.sm_count / 2));
            e = cudaOccupancyMaxActiveClusters(&n, kernel, &q);
        }
        g_pair_err[dev.device][idx] = e;
        g_pair_clusters[dev.device][idx] = n;
    });
    const int clusters = g_pair_clusters[dev.device][idx];
    if (g_pair_err[dev.device][idx] != cudaSuccess || clusters < 1) {
        cudaGetLastError();
        return SGEMM_ERR_LAUNCH;
    }
    int *flag = watchdog_flag_device_ptr();
    if (!flag) return SGEMM_ERR_LAUNCH;
    alignas(64) CUtensorMap mapA{}, mapB{}, mapC{};
    if (!cpa) {  // operands through TMA; otherwise the kernel's cp.async loaders read A and B
        const bool ok_a =
            TA ? encode_map(&mapA, p.A, p.K, p.M, p.lda, p.batch, p.strideA, 32, 32, CU_TENSOR_MAP_SWIZZLE_128B)
               : encode_map(&mapA, p.A, p.M, p.K, p.lda, p.batch, p.strideA, BK, pr::HM, CU_TENSOR_MAP_SWIZZLE_128B);
        const bool ok_b =
            TB ? encode_map(&mapB, p.B, p.N, p.K, p.ldb, p.batch, p.strideB, BK, pr::HN, CU_TENSOR_MAP_SWIZZLE_128B)
               : encode_map(&mapB, p.B, p.K, p.N, p.ldb, p.batch, p.strideB, pr::HN, BK, CU_TENSOR_MAP_SWIZZLE_NONE);
        if (!ok_a || !ok_b) return SGEMM_ERR_LAUNCH;
    }
    // C through TMA when its rows allow 16-byte aligned boxes and C is not
    // read (beta = 0; split tiles are reduce-added either way).
    const bool c_tma = VEC_C && p.beta == 0.0f &&
                       encode_map(&mapC, p.C, p.M, p.N, p.ldc, p.batch, p.strideC, 32, 32, CU_TENSOR_MAP_SWIZZLE_128B);
    if (!c_tma) mapC = mapA;  // not read by the kernel

    const int64_t tiles_m = (p.M + pr::PM - 1) / pr::PM, tiles_n = (p.N + pr::PN - 1) / pr::PN;
    const int64_t k_blocks = (p.K + BK - 1) / BK;
    if (tiles_m * tiles_n * p.batch > INT32_MAX / 2 || k_blocks > INT32_MAX / 2) return SGEMM_ERR_UNSUPPORTED;
    const int tiles = static_cast<int>(tiles_m * tiles_n * p.batch);
    // One pair per two SMs, as many pairs as fit at once. A stream-K share
    // below 4 k-blocks costs more in fix-up than it saves. Accumulation
    // chains are bounded by the folds inside the kernel, so units may span
    // any number of k-blocks.
    const Schedule sch = make_schedule(tiles, k_blocks, clusters, sk_mode, 4, 0.25);
    const int split = tiles - sch.dp_tiles;
    int rc = split_tiles_prepare(p, pr::PM, pr::PN, static_cast<int>(tiles_n), static_cast<int>(tiles_m * tiles_n),
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
    a.cpa = cpa ? 1 : 0;
    a.ta = TA ? 1 : 0;
    a.tb = TB ? 1 : 0;
    a.C = p.C;
    a.ldc = p.ldc;
    a.tiles_n = static_cast<int>(tiles_n);
    a.k_blocks = static_cast<int>(k_blocks);
    a.dp_tiles = sch.dp_tiles;
    a.sk_ctas = sch.sk_ctas;
    a.sk_iters = sch.sk_iters;
    a.timeout_ns = static_cast<uint64_t>(watchdog_ms()) * 1000000ull;
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
    a.sk_switch_kb = 0;  // a unit switch costs no MMA time: the accumulators alternate
    a.signal_dependents = (split > 0 && p.act != SGEMM_ACT_NONE) ? 1 : 0;
    a.c_tma = c_tma ? 1 : 0;
    cfg.gridDim = dim3(2 * sch.grid);
    // Behind our own beta pre-pass (which touches only C, and which started
    // after everything before it in the stream had finished) the main loop
    // may overlap it; the epilogue waits for it (griddepcontrol.wait).
    // Right behind the aligned copies of A and B the prologue overlaps them
    // and the loaders wait.
    a.wait_inputs = (after_copy && split == 0) ? 1 : 0;
    cfg.numAttrs = (split > 0 || a.wait_inputs) ? 2 : 1;
    if (cudaLaunchKernelEx(&cfg, kernel, mapA, mapB, mapC, a) != cudaSuccess) {
        cudaGetLastError();
        return SGEMM_ERR_LAUNCH;
    }
    ++*launches;
    return split_tiles_finish(p, pr::PM, pr::PN, static_cast<int>(tiles_n), static_cast<int>(tiles_m * tiles_n),
                              sch.dp_tiles, split, stream, launches, a.signal_dependents != 0);
}

}  // namespace

int tf32x3_pair_launch(const Problem &p, const DeviceInfo &dev, int sk_mode, bool cpa, cudaStream_t stream,
                       int *launches, bool after_copy) {
    if (dev.device < 0 || dev.device >= kMaxDevices) return SGEMM_ERR_DEVICE;
    const bool vc = (p.ldc % 4 == 0) && (p.strideC % 4 == 0) && (reinterpret_cast<uintptr_t>(p.C) % 16 == 0);
    const int form = (vc ? 1 : 0) + (p.transA ? 2 : 0) + (p.transB ? 4 : 0);
    switch (form) {
        case 0: return launch_pair<false, false, false>(p, dev, sk_mode, cpa, after_copy, stream, launches);
        case 1: return launch_pair<true, false, false>(p, dev, sk_mode, cpa, after_copy, stream, launches);
        case 2: return launch_pair<false, true, false>(p, dev, sk_mode, cpa, after_copy, stream, launches);
        case 3: return launch_pair<true, true, false>(p, dev, sk_mode, cpa, after_copy, stream, launches);
        case 4: return launch_pair<false, false, true>(p, dev, sk_mode, cpa, after_copy, stream, launches);
        case 5: return launch_pair<true, false, true>(p, dev, sk_mode, cpa, after_copy, stream, launches);
        case 6: return launch_pair<false, true, true>(p, dev, sk_mode, cpa, after_copy, stream, launches);
        default: return launch_pair<true, true, true>(p, dev, sk_mode, cpa, after_copy, stream, launches);
    }
}

}  // namespace sgemm
