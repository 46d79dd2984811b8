// Tensor-core SGEMM on SM pairs: tcgen05.mma.cta_group::2 (kind::tf32) with
// the three-term TF32 split of sgemm_tf32x3.cu, for all four operand forms
// (op(A) = A or A^T, op(B) = B or B^T) with 16-byte aligned rows.
//
// The product is the plain sum of "CUDA算子优化(4)：矩阵乘法", section
// "矩阵乘法的数学定义"; the pages give no tensor-core design (they name
// tensor cores once, "CUDA内存优化入门：从Naive到Tiled矩阵乘法", section 八).
//
// Why pairs. On one SM the 128 x 256 kernel moves about 256 KB through
// shared memory per 32-deep k-block (TMA writes of the raw tiles, the
// converters' reads and their hi / lo writes of B, and the tensor core's
// reads of B, 8 KB per 128 x 256 x 8 MMA), which holds the tensor pipe near
// 83% of its rate. Two CTAs on two SMs of a cluster share one 256 x 256 tile:
// each holds 128 rows of A (in its TMEM) and 128 columns of B (in its shared
// memory), and one MMA of 256 x 256 x 8 issued by the even CTA reads both
// halves. Per SM that halves B's traffic: about 144 KB per k-block for the
// same flops, under what the shared-memory pipe sustains.
//
// Roles in each CTA (23 warps):
//   * warp 0: in the even CTA, one thread issues the pair's MMAs (4 k-slices
//     x 3 products per k-block, lo*hi + hi*lo + hi*hi) and commits them to
//     the mbarriers of both CTAs (multicast); in the odd CTA, one thread
//     forwards "stage filled" to the even CTA (one cluster-scope arrival per
//     k-block instead of one per converter warp).
//   * warps 1 and 22: TMA of this CTA's A rows (128 x 32, 128-byte swizzled)
//     and B columns (32 x 128, unswizzled) into a 2-slot raw ring.
//   * warps 2-17 (converters, two groups of 8 taking alternate k-blocks):
//     split A into hi / lo and write them to this CTA's TMEM (the A
//     operand), transpose and split B into K-major, 128-byte-swizzled hi / lo
//     tiles in a 4-stage shared ring, then one lane per warp arrives on a
//     local mbarrier (the even CTA's stage-full barrier, or the odd CTA's
//     forwarding barrier).
//   * warps 18-21 (epilogue): one per TMEM lane quarter, reading the
//     accumulator's 256 columns for its 32 rows in 32 x 32 chunks, each
//     staged in shared memory and written by one TMA bulk store (or bulk
//     reduce-add for tiles split along K); chunks crossing the last row or
//     column, C that TMA cannot address, or beta != 0 take per-thread
//     stores. After the last chunk's TMEM load one lane per warp frees the
//     accumulator on the even CTA's mbarrier.
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

constexpr int PM = 256, PN = 256;  // C tile of a pair
constexpr int HM = 128, HN = 128;  // this CTA's rows of A, columns of B
// Four operand stages: a stage is refilled only after the MMAs that read it
// have completed, and completions trail issue by the tensor pipe's queue,
// so three stages left the MMA issuer waiting ~480 cycles per k-block.
constexpr int OP_STAGES = 4, RAW_SLOTS = 2;
constexpr int B_HALF = HN * BK * 4;   // 16 KB: one of B hi / B lo, or raw B
constexpr int A_RAW = HM * BK * 4;    // 16 KB
constexpr int OP_STAGE = 2 * B_HALF;  // hi | lo
constexpr int SLOT = A_RAW + B_HALF;  // raw A | raw B
constexpr int RAW0 = OP_STAGES * OP_STAGE;
// C staging: per epilogue warp two 32 x 32 fp32 chunks (128-byte swizzled
// rows) that TMA stores or reduce-adds into C.
constexpr int C_CHUNK = 32 * 32 * 4;
constexpr int C_STAGE0 = RAW0 + RAW_SLOTS * SLOT;
// Converters: two groups of 8 warps taking alternate k-blocks (one group's
// chain of waits, loads, stores and arrivals takes longer than one k-block
// of MMA, so one group alone would hold the tensor pipe back).
constexpr int GROUP_WARPS = 8, CONV_GROUPS = 2, CONV_WARPS = GROUP_WARPS * CONV_GROUPS, EPI_WARPS = 4;
// Epilogue: EPI_WARPS / 4 warps per TMEM lane quarter, each reading an equal
// share of the accumulator's 32-column chunks; C_BUFS staging chunks each.
constexpr int EPI_PER_QUAD = EPI_WARPS / 4, CHUNKS_PER_WARP = (PN / 32) / EPI_PER_QUAD, C_BUFS = 2;
constexpr int CONV_THREADS = 32 * GROUP_WARPS;  // threads converting one k-block
constexpr int EPI_WARP0 = 2 + CONV_WARPS;
// A second TMA issuer: a warp keeps only about one box in processing at a
// time (measured on GB300: ~0.4 us per box of 16-64 KB, whatever the ring
// depth), so A and B come from separate warps.
constexpr int TMA_B_WARP = EPI_WARP0 + EPI_WARPS;
constexpr int THREADS = 32 * (TMA_B_WARP + 1);
constexpr int BAR_OFFSET = C_STAGE0 + EPI_WARPS * C_BUFS * C_CHUNK;
constexpr int PBAR_BYTES = 256;
constexpr int SMEM_BYTES = BAR_OFFSET + PBAR_BYTES + 1024;
constexpr uint32_t TMEM_A = PN;  // A stages after the 256-column accumulator
// Instruction descriptor: D fp32, A and B tf32, both K-major, N = 256, M = 256.
constexpr uint32_t kIdesc2 = (1u << 4) | (2u << 7) | (2u << 10) | (static_cast<uint32_t>(PN >> 3) << 17) |
                             (static_cast<uint32_t>(PM >> 4) << 24);
// mbarrier indices
constexpr int RAW_FULL = 0, RAW_FREE = RAW_FULL + RAW_SLOTS, OP_FULL = RAW_FREE + RAW_SLOTS,
              OP_EMPTY = OP_FULL + OP_STAGES, ACC_FULL = OP_EMPTY + OP_STAGES, ACC_EMPTY = ACC_FULL + 1,
              DRAIN = ACC_EMPTY + 1, OP_FWD = DRAIN + 1, NBARS = OP_FWD + OP_STAGES;
// A pair that moves from one split tile to the next waits ~5 us on GB300
// for its accumulator to be read out: about 6 k-blocks of MMAs. The split
// work is shared with that cost counted, so the pairs whose share crosses a
// tile boundary are not the last to finish.
constexpr int SWITCH_KB = 6;
static_assert(NBARS * 8 + 16 <= PBAR_BYTES, "barrier block");
static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
static_assert(TMEM_A + OP_STAGES * 64 <= TMEM_COLS, "TMEM columns");
static_assert((HN / 4) * (BK / 4) == CONV_THREADS, "one 4 x 4 B block per converter thread");

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

// One 256 x 256 x 8 product of the pair: A (128 rows per CTA) from TMEM, B
// (128 columns per CTA) from shared memory.
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

// Fused-epilogue values of 16 accumulator columns (chunk columns base ..
// base + 15) written to the staging row of this lane: ACT(alpha * v + bias),
// the bias per row (bl) or per column (lane (base + j)'s bl, by shuffle).
template <int ACT>
__device__ __forceinline__ void stage16_ep(uint32_t buf, int lane, int base, float alpha, bool col_bias, float bl,
                                           const float (&v)[16]) {
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

__device__ __forceinline__ void stage16_fused(int act, uint32_t buf, int lane, int base, float alpha, bool col_bias,
                                              float bl, const float (&v)[16]) {
    switch (act) {
        case SGEMM_ACT_RELU: stage16_ep<SGEMM_ACT_RELU>(buf, lane, base, alpha, col_bias, bl, v); break;
        case SGEMM_ACT_GELU: stage16_ep<SGEMM_ACT_GELU>(buf, lane, base, alpha, col_bias, bl, v); break;
        case SGEMM_ACT_SILU: stage16_ep<SGEMM_ACT_SILU>(buf, lane, base, alpha, col_bias, bl, v); break;
        default: stage16_ep<SGEMM_ACT_NONE>(buf, lane, base, alpha, col_bias, bl, v); break;
    }
}

// A chunk that crosses the last row or column of C: per-thread stores, and
// on the tile's last chunk the accumulator release (one lane per warp, on
// the even CTA's barrier acc_empty). Out of line: it is rare, and inlined it
// would compete for registers with the interior path.
template <bool VEC_C>
__device__ __noinline__ void edge_chunk(const Args &a, uint32_t taddr, float *crow, int64_t row, int64_t col0,
                                        bool atomic, bool last, uint32_t acc_empty) {
    const int lane = static_cast<int>(threadIdx.x & 31);
    epilogue_chunk_then<VEC_C>(a, taddr, crow, row, col0, atomic, last, [&] {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_at(acc_empty, 0);
    });
}

// TA: A stored K x M (op(A) = A^T); TB: B stored N x K (op(B) = B^T).
template <bool VEC_C, bool TA, bool TB>
__global__ void __launch_bounds__(pr::THREADS, 1)
    tf32x3_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                       const __grid_constant__ CUtensorMap tmC, const Args a) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (base - raw);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + pr::BAR_OFFSET);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(bars + pr::NBARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + pr::NBARS + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const int pair = static_cast<int>(blockIdx.x >> 1), pairs = static_cast<int>(gridDim.x >> 1);
    auto bar = [&](int i) { return smem_u32(bars + i); };

    // TMA of this CTA's A rows (warp 1) or B columns (warp TMA_B_WARP) for
    // the k-blocks it = from .. to - 1 of its units, into the raw ring.
    auto tma_pass = [&](uint32_t from, uint32_t to) {
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
                    if (TB)  // B stored N x K: already K-major, 128 rows of 32 k
                        tma_load_3d(sl + pr::A_RAW, &tmB, kblk * BK, n0, zb, bar(pr::RAW_FULL + slot));
                    else
                        tma_load_3d(sl + pr::A_RAW, &tmB, n0, kblk * BK, zb, bar(pr::RAW_FULL + slot));
                }
            }
        });
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < pr::RAW_SLOTS; ++s) {
            mbar_init(bar(pr::RAW_FULL + s), 2);  // one expect_tx arrival per TMA issuer
            mbar_init(bar(pr::RAW_FREE + s), pr::GROUP_WARPS);  // one lane per converter warp
        }
        for (int s = 0; s < pr::OP_STAGES; ++s) {
            // Even CTA: its own converter warps plus one forwarded arrival for
            // the odd CTA's warps (OP_FWD there), so the converters never pay
            // a cluster-scope release.
            mbar_init(bar(pr::OP_FULL + s), pr::GROUP_WARPS + 1);
            mbar_init(bar(pr::OP_FWD + s), pr::GROUP_WARPS);
            mbar_init(bar(pr::OP_EMPTY + s), 1);
        }
        mbar_init(bar(pr::ACC_FULL), 1);
        mbar_init(bar(pr::ACC_EMPTY), 2 * pr::EPI_WARPS);
        mbar_init(bar(pr::DRAIN), 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if ((warp == 1 || warp == pr::TMA_B_WARP) && lane == 0)
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(warp == 1 ? &tmA : &tmB)) : "memory");
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
    if ((warp == 1 || warp == pr::TMA_B_WARP) && lane == 0) tma_pass(0, pr::RAW_SLOTS);
    __syncwarp();
    cluster_wait();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    // A pass launched behind this kernel (the activation of split tiles) may
    // be scheduled now; it waits for this grid to finish before touching C.
    if (a.signal_dependents && threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;");

    if (warp == 0) {
        // ------------------------------------------------------------ MMA issuer
        if (rank == 0 && lane == 0) {
            uint32_t it = 0, unit = 0;
            for_each_unit_of(a, abort_flag, pair, pairs, [&](int, int kb, int ke) {
                if (!mbar_wait<true>(bar(pr::ACC_EMPTY), (unit & 1) ^ 1, a, abort_flag, WD_MMA_ACC)) return;
                tc_fence_after();
                for (int kblk = kb; kblk < ke; ++kblk, ++it) {
                    const int s = static_cast<int>(it % pr::OP_STAGES);
                    const uint32_t ph = (it / pr::OP_STAGES) & 1;
                    if (!mbar_wait<true>(bar(pr::OP_FULL + s), ph, a, abort_flag, WD_MMA_FULL)) return;
                    tc_fence_after();
                    const uint32_t st = base + static_cast<uint32_t>(s * pr::OP_STAGE);
                    const uint64_t b_hi = sw128_desc(st), b_lo = sw128_desc(st + pr::B_HALF);
                    const uint32_t a_hi = tmem_base + pr::TMEM_A + static_cast<uint32_t>(64 * s);
                    const uint32_t a_lo = a_hi + 32;
#pragma unroll
                    for (int ks = 0; ks < BK / 8; ++ks) {
                        const uint64_t adv = static_cast<uint64_t>(ks * 2);
                        const uint32_t ac = static_cast<uint32_t>(ks * 8);
                        const uint32_t first = (kblk == kb && ks == 0) ? 0u : 1u;
                        tc_mma2_ts(tmem_base, a_lo + ac, b_hi + adv, first);
                        tc_mma2_ts(tmem_base, a_hi + ac, b_lo + adv, 1u);
                        tc_mma2_ts(tmem_base, a_hi + ac, b_hi + adv, 1u);
                    }
                    tc_commit2(bar(pr::OP_EMPTY + s));
                }
                tc_commit2(bar(pr::ACC_FULL));
                ++unit;
            });
            tc_commit2(bar(pr::DRAIN));
            const bool was_aborted = *abort_flag != 0;
            if (!mbar_wait(bar(pr::DRAIN), 0, a, abort_flag, WD_DRAIN) && was_aborted) {
                const uint64_t t0 = global_timer();
                while (!mbar_try_wait(bar(pr::DRAIN), 0) && global_timer() - t0 < a.timeout_ns) {
                }
            }
        }
        if (rank != 0 && lane == 0) {
            // Forwarder: once this CTA's converters have filled stage s, one
            // cluster-scope arrival tells the even CTA's MMA issuer.
            uint32_t it = 0;
            bool ok = true;
            for_each_unit_of(a, abort_flag, pair, pairs, [&](int, int kb, int ke) {
                for (int kblk = kb; kblk < ke && ok; ++kblk, ++it) {
                    const int s = static_cast<int>(it % pr::OP_STAGES);
                    if (!mbar_wait(bar(pr::OP_FWD + s), (it / pr::OP_STAGES) & 1, a, abort_flag, WD_PRODUCER)) {
                        ok = false;
                        return;
                    }
                    mbar_arrive_at(bar(pr::OP_FULL + s), 0);
                }
            });
        }
    } else if (warp == 1 || warp == pr::TMA_B_WARP) {
        // ---------------------------------------------------- TMA issuers (A, B)
        if (lane == 0) tma_pass(pr::RAW_SLOTS, 0xffffffffu);
    } else if (warp < pr::EPI_WARP0) {
        // ------------------------------------------------------------ converters
        const int cw = warp - 2;                            // 0 .. 15
        const uint32_t group = static_cast<uint32_t>(cw >> 3);  // k-blocks with it % 2 == group
        const int ct = threadIdx.x - 64 - 256 * static_cast<int>(group);
        const int l = ct & 7, tb = ct >> 3;                 // 32 groups of eight lanes
        const int g = (tb >> 3) * 8 + l, c = (l + tb) & 7;  // this thread's 4 x 4 B block
        const int q = warp & 3, part = (cw >> 2) & 1;       // TMEM lane quarter, k-columns 16*part..+15
        const int arow = 32 * q + lane;                     // A row this thread converts
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
                // A: 16 k-values of row arow.
                float4 av[4];
                if (TA) {
                    // Box q holds rows k = 0..31 of columns m = 32q..32q+31 (128-byte
                    // swizzled): column arow is lane `lane` of each row.
                    float t[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        t[j] = ld_shared_f32(sl + static_cast<uint32_t>(q * 4096) + sw128_offset(16 * part + j, lane >> 2) +
                                             static_cast<uint32_t>((lane & 3) * 4));
#pragma unroll
                    for (int j = 0; j < 4; ++j) av[j] = make_float4(t[4 * j], t[4 * j + 1], t[4 * j + 2], t[4 * j + 3]);
                } else {
                    // Chunks 4*part .. 4*part+3 of the swizzled K-major row.
#pragma unroll
                    for (int j = 0; j < 4; ++j) av[j] = ld_shared_v4(sl + sw128_offset(arow, 4 * part + j));
                }
                // B: op(B) = B: rows 4c..4c+3, columns 4g..4g+3 of the unswizzled 32 x 128
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
                const uint32_t ta = tmem_base + (static_cast<uint32_t>(32 * q) << 16) + pr::TMEM_A +
                                    static_cast<uint32_t>(64 * s + 16 * part);
#pragma unroll
                for (int h = 0; h < 2; ++h) {  // 8 values at a time: fewer live registers
                    float hi[8], lo[8];
                    split_tf32(av[2 * h].x, hi[0], lo[0]);
                    split_tf32(av[2 * h].y, hi[1], lo[1]);
                    split_tf32(av[2 * h].z, hi[2], lo[2]);
                    split_tf32(av[2 * h].w, hi[3], lo[3]);
                    split_tf32(av[2 * h + 1].x, hi[4], lo[4]);
                    split_tf32(av[2 * h + 1].y, hi[5], lo[5]);
                    split_tf32(av[2 * h + 1].z, hi[6], lo[6]);
                    split_tf32(av[2 * h + 1].w, hi[7], lo[7]);
                    tmem_store8(ta + 8 * h, hi);
                    tmem_store8(ta + 32 + 8 * h, lo);
                }
                tmem_wait_st();
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar((rank == 0 ? pr::OP_FULL : pr::OP_FWD) + s));
            }
        });
    } else {
        // -------------------------------------------------------------- epilogue
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const uint32_t stage0 =
            base + pr::C_STAGE0 + static_cast<uint32_t>((warp - pr::EPI_WARP0) * pr::C_BUFS * pr::C_CHUNK);
        const int ch0 = ((warp - pr::EPI_WARP0) >> 2) * pr::CHUNKS_PER_WARP;  // this warp's chunks
        const int ch_end = ch0 + pr::CHUNKS_PER_WARP;
        // C may still be in the beta pre-pass launched just before this
        // kernel (programmatic dependent launch): only the epilogue waits.
        asm volatile("griddepcontrol.wait;" ::: "memory");
        uint32_t unit = 0, nchunk = 0;
        auto release = [&] {
            // The accumulator is out of TMEM: one lane per warp frees it on the
            // even CTA's barrier.
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_at(bar(pr::ACC_EMPTY), 0);
        };
        for_each_unit_of(a, abort_flag, pair, pairs, [&](int tile, int kb, int ke) {
            if (!mbar_wait<true>(bar(pr::ACC_FULL), unit & 1, a, abort_flag, WD_EPILOGUE)) return;
            tc_fence_after();
            const TileAt at = tile_at<pr::PM, pr::PN>(a, tile);
            const int64_t row0 = at.m0 + pr::HM * static_cast<int64_t>(rank) + q * 32;
            const int64_t row = row0 + lane;
            // Stream-K tiles hold beta * C + bias already: every unit adds.
            const bool atomic = tile >= a.dp_tiles;
            if (a.c_tma) {
                // Each 32 x 32 chunk inside the matrix: TMEM -> registers ->
                // (epilogue) -> swizzled staging rows -> one TMA store (or
                // reduce-add) of the chunk. Chunks that cross the last row or
                // column use the per-thread stores.
                const bool fused = a.ep && !atomic;
                const bool col_bias = a.bias_kind == SGEMM_BIAS_PER_COL;
                const float alpha = a.alpha;
                const float rb = (a.bias_kind == SGEMM_BIAS_PER_ROW && row < a.M) ? __ldg(a.bias + row) : 0.0f;
                float *crow = a.C + at.item * a.strideC + row * a.ldc;
#pragma unroll 1
                for (int ch = ch0; ch < ch_end; ++ch) {
                    const uint32_t taddr =
                        tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(ch * 32);
                    const int64_t col0 = at.n0 + ch * 32;
                    const bool last = ch == ch_end - 1;
                    if (col0 + 32 > a.N || row0 + 32 > a.M) {
                        edge_chunk<VEC_C>(a, taddr, crow, row, col0, atomic, last, bar(pr::ACC_EMPTY));
                        continue;
                    }
                    const uint32_t buf = stage0 + (nchunk % pr::C_BUFS) * pr::C_CHUNK;
                    ++nchunk;
                    // Per-column bias of this chunk: lane l holds column col0 + l.
                    const float bl = (fused && col_bias) ? __ldg(a.bias + col0 + lane) : rb;
                    if (lane == 0) bulk_wait_read<pr::C_BUFS - 1>();  // the store C_BUFS chunks back has read this buffer
                    __syncwarp();
                    if (fused) {
                        float v[16];
                        tmem_load16(taddr, v);
                        stage16_fused(a.act, buf, lane, 0, alpha, col_bias, bl, v);
                        tmem_load16(taddr + 16, v);
                        if (last) release();
                        stage16_fused(a.act, buf, lane, 16, alpha, col_bias, bl, v);
                    } else {
                        float v[32];
                        tmem_load32(taddr, v);
                        if (last) release();
#pragma unroll
                        for (int j = 0; j < 32; j += 4)
                            st_shared_v4(buf + sw128_offset(lane, j >> 2), alpha * v[j], alpha * v[j + 1],
                                         alpha * v[j + 2], alpha * v[j + 3]);
                    }
                    fence_proxy_async_smem();  // staging writes -> visible to the TMA engine
                    __syncwarp();
                    if (lane == 0) {
                        const int x = static_cast<int>(col0), y = static_cast<int>(row0);
                        if (atomic)
                            tma_reduce_add_3d(&tmC, x, y, at.item, buf);
                        else
                            tma_store_3d(&tmC, x, y, at.item, buf);
                        bulk_commit();
                    }
                }
            } else {
                float *crow = a.C + at.item * a.strideC + row * a.ldc;
#pragma unroll 1
                for (int ch = ch0; ch < ch_end; ++ch)
                    epilogue_chunk_then<VEC_C>(
                        a, tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(ch * 32), crow,
                        row, at.n0 + ch * 32, atomic, ch == ch_end - 1, release);
            }
            ++unit;
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
int launch_pair(const Problem &p, const DeviceInfo &dev, int sk_mode, cudaStream_t stream, int *launches) {
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
    alignas(64) CUtensorMap mapA, mapB, mapC;
    const bool ok_a =
        TA ? encode_map(&mapA, p.A, p.K, p.M, p.lda, p.batch, p.strideA, 32, 32, CU_TENSOR_MAP_SWIZZLE_128B)
           : encode_map(&mapA, p.A, p.M, p.K, p.lda, p.batch, p.strideA, BK, pr::HM, CU_TENSOR_MAP_SWIZZLE_128B);
    const bool ok_b =
        TB ? encode_map(&mapB, p.B, p.N, p.K, p.ldb, p.batch, p.strideB, BK, pr::HN, CU_TENSOR_MAP_SWIZZLE_128B)
           : encode_map(&mapB, p.B, p.K, p.N, p.ldb, p.batch, p.strideB, pr::HN, BK, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (!ok_a || !ok_b) return SGEMM_ERR_LAUNCH;
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
    // below 4 k-blocks costs more in fix-up than it saves.
    const bool long_k = k_blocks > 2 * KB_CAP;  // every tile split, units of <= KB_CAP k-blocks
    const Schedule sch = make_schedule(tiles, k_blocks, clusters, long_k ? SK_ALL : sk_mode, 4, 0.25);
    const int split = tiles - sch.dp_tiles;
    int rc = split_tiles_prepare(p, pr::PM, pr::PN, static_cast<int>(tiles_n), static_cast<int>(tiles_m * tiles_n),
                                 sch.dp_tiles, split, stream, launches);
    if (rc != SGEMM_OK) return rc;
    Args a{};
    a.M = p.M;
    a.N = p.N;
    a.K = p.K;
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
    a.kb_cap = long_k ? KB_CAP : 0;
    count_switches(a, pr::SWITCH_KB);
    a.signal_dependents = (split > 0 && p.act != SGEMM_ACT_NONE) ? 1 : 0;
    a.c_tma = c_tma ? 1 : 0;
    cfg.gridDim = dim3(2 * sch.grid);
    // Behind our own beta pre-pass (which touches only C, and which started
    // after everything before it in the stream had finished) the main loop
    // may overlap it; the epilogue waits for it (griddepcontrol.wait).
    cfg.numAttrs = split > 0 ? 2 : 1;
    if (cudaLaunchKernelEx(&cfg, kernel, mapA, mapB, mapC, a) != cudaSuccess) {
        cudaGetLastError();
        return SGEMM_ERR_LAUNCH;
    }
    ++*launches;
    return split_tiles_finish(p, pr::PM, pr::PN, static_cast<int>(tiles_n), static_cast<int>(tiles_m * tiles_n),
                              sch.dp_tiles, split, stream, launches, a.signal_dependents != 0);
}

}  // namespace

int tf32x3_pair_launch(const Problem &p, const DeviceInfo &dev, int sk_mode, cudaStream_t stream, int *launches) {
    if (dev.device < 0 || dev.device >= kMaxDevices) return SGEMM_ERR_DEVICE;
    const bool vc = (p.ldc % 4 == 0) && (p.strideC % 4 == 0) && (reinterpret_cast<uintptr_t>(p.C) % 16 == 0);
    const int form = (vc ? 1 : 0) + (p.transA ? 2 : 0) + (p.transB ? 4 : 0);
    switch (form) {
        case 0: return launch_pair<false, false, false>(p, dev, sk_mode, stream, launches);
        case 1: return launch_pair<true, false, false>(p, dev, sk_mode, stream, launches);
        case 2: return launch_pair<false, true, false>(p, dev, sk_mode, stream, launches);
        case 3: return launch_pair<true, true, false>(p, dev, sk_mode, stream, launches);
        case 4: return launch_pair<false, false, true>(p, dev, sk_mode, stream, launches);
        case 5: return launch_pair<true, false, true>(p, dev, sk_mode, stream, launches);
        case 6: return launch_pair<false, true, true>(p, dev, sk_mode, stream, launches);
        default: return launch_pair<true, true, true>(p, dev, sk_mode, stream, launches);
    }
}

}  // namespace sgemm
