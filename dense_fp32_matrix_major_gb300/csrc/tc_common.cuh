// Device-side building blocks of the tcgen05 kernels (sm_103a): the kernel
// argument block, mbarrier waits bounded in time, tcgen05 MMA / TMEM access,
// TMA loads, the three-term TF32 split, the 128-byte swizzle, the C stores
// (plain, atomic for split tiles, and the fused epilogue) and the persistent
// unit loop. Shared by the translation units that hold the kernels.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "epilogue.cuh"
#include "sgemm.h"

namespace sgemm {
namespace tc {

constexpr int BM = 128, BN = 256, BK = 32;  // BK fp32 = 128 bytes = one swizzle row
constexpr int A_TILE = BM * BK * 4;         // bytes of one A tile (hi or lo)
constexpr int B_TILE = BN * BK * 4;         // bytes of one B tile (hi or lo)
constexpr int EPILOGUE_WARPS = 4;
constexpr int TMEM_COLS = 512;
constexpr int BAR_BYTES = 128;
// The tensor core adds each MMA's products into the fp32 accumulator in TMEM
// with truncation (measured on GB300: about one unit in the last place of
// the running sum lost per tcgen05.mma, all in the same direction when the
// terms share a sign). The error therefore grows with the number of MMAs
// that one accumulator chains, whatever K is: ~6.7e-7 of sum |a||b| per
// 32-deep k-block (12 MMAs) on non-negative inputs. Products with more than
// KB_CAP k-blocks are split along K into units of at most KB_CAP k-blocks
// (~5.4e-6 on non-negative inputs), whose partial sums are added into C
// with round-to-nearest fp32 adds (the TMA kernels of sgemm_tf32x3.cu).
constexpr int KB_CAP = 8;
// Kernels that fold on chip restart their accumulator every FOLD_KB
// k-blocks and add it, rounded to nearest, into an fp32 running sum of the
// tile (TMEM or shared memory), so units of any length keep that error.
constexpr int FOLD_KB = 8;

// Watchdog codes (which wait gave up).
enum : int { WD_PRODUCER = 1, WD_MMA_FULL = 2, WD_MMA_ACC = 3, WD_EPILOGUE = 4, WD_DRAIN = 5, WD_SELFTEST = 6 };

struct Args {
    int64_t M, N, K;
    const float *A;
    int64_t lda;
    const float *B;
    int64_t ldb;
    float *C;
    int64_t ldc;
    int tiles_n, k_blocks, dp_tiles;
    int sk_ctas;
    int64_t sk_iters;
    uint64_t timeout_ns;
    int *watchdog;
    float alpha = 1.0f, beta = 0.0f;  // C = alpha * op(A) op(B) + beta * C; beta == 0: C not read
    // Strided batch: tiles run item-major, tiles_per_item per product; item b
    // uses A + b*strideA, B + b*strideB, C + b*strideC. In the TMA kernels the
    // item is the third tensor-map coordinate (0 for an operand shared by all
    // items, stride 0).
    int64_t strideA = 0, strideB = 0, strideC = 0;
    int tiles_per_item = 1;
    int a_shared = 0, b_shared = 0;
    // Fused epilogue on whole tiles: C = act(alpha * acc + beta * C + bias).
    const float *bias = nullptr;
    int bias_kind = 0, act = 0, ep = 0;
    // Kernels with a C tensor map: write C through shared memory with TMA
    // bulk stores (and bulk reduce-adds for split tiles).
    int c_tma = 0;
    // Operands whose rows TMA cannot address (not 16-byte aligned): the raw
    // ring is filled with 4-byte cp.async copies instead (pair kernel).
    int cpa = 0;
    // Operand forms (A stored K x M, B stored N x K), for the recomputation of
    // non-finite outputs (fix_nonfinite).
    int ta = 0, tb = 0;
    // Longest run of k-blocks one unit may accumulate in TMEM (0: no limit);
    // split units start at multiples of it (see for_each_unit_of).
    int kb_cap = 0;
    // A pass (the activation of split tiles) follows as a programmatic
    // dependent: signal griddepcontrol.launch_dependents.
    int signal_dependents = 0;
    // Launched as the programmatic dependent of the kernel that writes A and
    // B (aligned copies): the loaders wait for it (griddepcontrol.wait)
    // before their first read.
    int wait_inputs = 0;
    // Cost, in k-blocks, of a switch from one split tile to the next inside
    // one worker's share (the next unit's MMAs wait for the accumulator to be
    // read out). With it the split iterations are shared so that k-blocks
    // plus switches come out even; 0 shares the k-blocks evenly. Not used
    // with kb_cap.
    int sk_switch_kb = 0;
};

// Item and top-left corner of tile `tile` of the item-major tile order.
struct TileAt {
    int item;
    int64_t m0, n0;
};

template <int TM = BM, int TN = BN>
__device__ __forceinline__ TileAt tile_at(const Args &a, int tile) {
    const int rest = tile % a.tiles_per_item;
    return TileAt{tile / a.tiles_per_item, static_cast<int64_t>(rest / a.tiles_n) * TM,
                  static_cast<int64_t>(rest % a.tiles_n) * TN};
}

// Instruction descriptor of tcgen05.mma kind::tf32: D fp32 (bits 4-5 = 1),
// A and B tf32 (bits 7-9 and 10-12 = 2), both K-major (bits 15, 16 = 0),
// N >> 3 in bits 17-22, M >> 4 in bits 24-28.
constexpr uint32_t kIdesc = (1u << 4) | (2u << 7) | (2u << 10) | (static_cast<uint32_t>(BN >> 3) << 17) |
                            (static_cast<uint32_t>(BM >> 4) << 24);

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of
// 128 bytes, 8-row groups 1024 bytes apart. Bits 0-13 start address >> 4,
// 16-29 leading byte offset >> 4 (unused for this layout), 32-45 stride byte
// offset >> 4, bit 46 descriptor version 1, bits 61-63 swizzle mode (2 = 128 B).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(1) << 16) |
           (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
           (static_cast<uint64_t>(2) << 61);
}

__device__ __forceinline__ uint32_t tf32_rna_bits(float x);

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// CLUSTER: acquire at cluster scope (arrivals may come from the peer CTA).
template <bool CLUSTER = false>
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    if (CLUSTER) {
        asm volatile(
            "{\n"
            " .reg .pred p;\n"
            " mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
            " selp.u32 %0, 1, 0, p;\n"
            "}\n"
            : "=r"(ok)
            : "r"(bar), "r"(parity)
            : "memory");
    } else {
        asm volatile(
            "{\n"
            " .reg .pred p;\n"
            " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
            " selp.u32 %0, 1, 0, p;\n"
            "}\n"
            : "=r"(ok)
            : "r"(bar), "r"(parity)
            : "memory");
    }
    return ok != 0;
}

// Whether the phase with the given parity has completed, without waiting
// (test_wait never suspends the thread).
template <bool CLUSTER = false>
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    if (CLUSTER) {
        asm volatile(
            "{\n"
            " .reg .pred p;\n"
            " mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
            " selp.u32 %0, 1, 0, p;\n"
            "}\n"
            : "=r"(ok)
            : "r"(bar), "r"(parity)
            : "memory");
    } else {
        asm volatile(
            "{\n"
            " .reg .pred p;\n"
            " mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
            " selp.u32 %0, 1, 0, p;\n"
            "}\n"
            : "=r"(ok)
            : "r"(bar), "r"(parity)
            : "memory");
    }
    return ok != 0;
}

// Wait for the phase with the given parity to complete, within the time
// limit; false if the limit passed or another role already aborted.
template <bool CLUSTER = false>
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, const Args &a, volatile int *abort_flag,
                                          int code) {
    if (mbar_try_wait<CLUSTER>(bar, parity)) return true;
    const uint64_t t0 = global_timer();
    for (uint32_t n = 1;; ++n) {
        if (mbar_try_wait<CLUSTER>(bar, parity)) return true;
        if ((n & 63) == 0) {
            if (*abort_flag) return false;
            if (global_timer() - t0 > a.timeout_ns) {
                *abort_flag = 1;
                atomicCAS(a.watchdog, 0, code);
                return false;
            }
        }
    }
}

// True in exactly one lane of the (converged, full) warp.
__device__ __forceinline__ bool elect_one() {
    uint32_t e;
    asm volatile(
        "{\n"
        " .reg .pred p;\n"
        " elect.sync _|p, 0xffffffff;\n"
        " selp.u32 %0, 1, 0, p;\n"
        "}\n"
        : "=r"(e));
    return e != 0;
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t accumulate) {
    asm volatile(
        "{\n"
        " .reg .pred p;\n"
        " setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n"
        "}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(kIdesc), "r"(accumulate)
        : "memory");
}

// MMA with the A operand in TMEM (128 lanes = rows, 8 columns = the k-slice).
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t accumulate) {
    asm volatile(
        "{\n"
        " .reg .pred p;\n"
        " setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n"
        "}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(kIdesc), "r"(accumulate)
        : "memory");
}

// 16 consecutive TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_store16(uint32_t taddr, const float (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15]))
        : "memory");
}

// 8 consecutive TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_store8(uint32_t taddr, const float (&v)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
                 "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
                 "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
                 "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7]))
                 : "memory");
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

// 3-D tiled TMA load of the box at (x, y, z) (x innermost, in elements; z is
// the batch item) into shared memory, completing its bytes of transactions
// on the mbarrier.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, int x, int y, int z,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}

// TMA bulk store of the box at (x, y, z) from shared memory, and the same as
// an element-wise fp32 add into global memory; both tracked as a bulk group
// of the issuing thread.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap *map, int x, int y, int z, uint32_t src) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(z), "r"(src)
                 : "memory");
}

__device__ __forceinline__ void tma_reduce_add_3d(const CUtensorMap *map, int x, int y, int z, uint32_t src) {
    asm volatile("cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(z), "r"(src)
                 : "memory");
}

// 4-byte asynchronous copy global -> shared; valid == false writes zero and
// reads nothing (src must still be a valid address).
__device__ __forceinline__ void cp_async4(uint32_t dst, const float *src, bool valid) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst),
                 "l"(__cvta_generic_to_global(src)), "r"(valid ? 4 : 0)
                 : "memory");
}

// The mbarrier gets one arrival once every cp.async this thread issued so far
// has completed (its expected count must include that arrival).
__device__ __forceinline__ void cp_async_arrive(uint32_t bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Wait until at most N bulk groups of this thread are still reading shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Wait until at most N bulk groups of this thread are incomplete.
template <int N>
__device__ __forceinline__ void bulk_wait() {
    asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ float ld_shared_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ void st_shared_f32(uint32_t addr, float v) {
    asm volatile("st.shared.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

__device__ __forceinline__ float4 ld_shared_v4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

// Low part of a value whose high part the tensor core takes by truncation.
__device__ __forceinline__ float lo_of(float x) {
    const float hi = __uint_as_float(__float_as_uint(x) & 0xFFFFE000u);
    return __uint_as_float(tf32_rna_bits(x - hi));
}

__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// 32 consecutive accumulator columns of this thread's lane.
__device__ __forceinline__ void tmem_load32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    // The registers are valid only after wait::ld; tying them to the wait keeps
    // every use after it.
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                   "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                   "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                   "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
                 :
                 : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 16 consecutive accumulator columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_load16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                   "+r"(r[15])
                 :
                 : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ uint32_t tf32_rna_bits(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}

// hi + lo split of one value: hi keeps the sign, the exponent and the top 10
// mantissa bits of x (an exact tf32, so it never overflows), and lo is
// x - hi (exact in fp32) rounded to tf32. Non-finite x gives a NaN lo, so the
// products that use it are NaN.
__device__ __forceinline__ void split_tf32(float x, float &hi, float &lo) {
    hi = __uint_as_float(__float_as_uint(x) & 0xFFFFE000u);
    lo = __uint_as_float(tf32_rna_bits(x - hi));
}

__device__ __forceinline__ void split_store(uint32_t hi_addr, uint32_t lo_addr, float a, float b, float c,
                                            float d);

__device__ __forceinline__ void st_shared_v4(uint32_t addr, float a, float b, float c, float d) {
    asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
                 : "memory");
}

// Split four values and store the high parts at hi_addr, the low parts at lo_addr.
__device__ __forceinline__ void split_store(uint32_t hi_addr, uint32_t lo_addr, float a, float b, float c,
                                            float d) {
    float h0, h1, h2, h3, l0, l1, l2, l3;
    split_tf32(a, h0, l0);
    split_tf32(b, h1, l1);
    split_tf32(c, h2, l2);
    split_tf32(d, h3, l3);
    st_shared_v4(hi_addr, h0, h1, h2, h3);
    st_shared_v4(lo_addr, l0, l1, l2, l3);
}

// Byte offset of 16-byte chunk `chunk` of row `row` in a 128-byte-swizzled tile.
__device__ __forceinline__ uint32_t sw128_offset(int row, int chunk) {
    return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}

// Atomic add of four consecutive floats at a 16-byte aligned address.
__device__ __forceinline__ void red_add_v4(float *p, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c), "f"(d)
                 : "memory");
}

// Fused epilogue for 16 values of one row: C[col0 + j] = ACT(alpha * v[j] +
// beta * C[col0 + j] + bias_j) for the columns below N (C read only when
// beta != 0), stores only when `valid` (row < M). The bias of column j is
// bl (per row or absent) or, per column, lane (base + j)'s value of bl (the
// warp loaded bias[chunk column + lane] in one coalesced load): the whole
// warp runs the shuffles, so no lane may have left before.
template <bool VEC_C, int ACT>
__device__ __forceinline__ void store16_ep(float *crow, bool valid, int64_t col0, int base, int64_t N, float alpha,
                                           float beta, bool col_bias, float bl, const float (&v)[16]) {
    if (VEC_C && col0 + 15 < N) {
#pragma unroll
        for (int j = 0; j < 16; j += 4) {
            float4 bb = make_float4(bl, bl, bl, bl);
            if (col_bias) {
                bb.x = __shfl_sync(0xffffffffu, bl, base + j);
                bb.y = __shfl_sync(0xffffffffu, bl, base + j + 1);
                bb.z = __shfl_sync(0xffffffffu, bl, base + j + 2);
                bb.w = __shfl_sync(0xffffffffu, bl, base + j + 3);
            }
            if (!valid) continue;
            float4 *p = reinterpret_cast<float4 *>(crow + col0 + j);
            float4 o = make_float4(alpha * v[j], alpha * v[j + 1], alpha * v[j + 2], alpha * v[j + 3]);
            if (beta != 0.0f) {
                const float4 c = *p;
                o.x = fmaf(beta, c.x, o.x);
                o.y = fmaf(beta, c.y, o.y);
                o.z = fmaf(beta, c.z, o.z);
                o.w = fmaf(beta, c.w, o.w);
            }
            o.x = activate(o.x + bb.x, ACT);
            o.y = activate(o.y + bb.y, ACT);
            o.z = activate(o.z + bb.z, ACT);
            o.w = activate(o.w + bb.w, ACT);
            *p = o;
        }
    } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const float b = col_bias ? __shfl_sync(0xffffffffu, bl, base + j) : bl;
            if (!valid || col0 + j >= N) continue;
            float x = alpha * v[j];
            if (beta != 0.0f) x = fmaf(beta, crow[col0 + j], x);
            crow[col0 + j] = activate(x + b, ACT);
        }
    }
}

// The 16 columns col0 .. col0 + 15 (= chunk column base .. base + 15) of one
// row; called by all 32 lanes of the warp (see store16_ep).
template <bool VEC_C>
__device__ __forceinline__ void store16_fused(const Args &a, float *crow, int64_t row, int64_t col0, int base,
                                              float bl, const float (&v)[16]) {
    const int64_t N = a.N;
    if (col0 >= N) return;  // uniform over the warp
    const bool valid = row < a.M;
    const float alpha = a.alpha, beta = a.beta;
    const bool cb = a.bias_kind == SGEMM_BIAS_PER_COL;
    switch (a.act) {
        case SGEMM_ACT_RELU:
            store16_ep<VEC_C, SGEMM_ACT_RELU>(crow, valid, col0, base, N, alpha, beta, cb, bl, v);
            break;
        case SGEMM_ACT_GELU:
            store16_ep<VEC_C, SGEMM_ACT_GELU>(crow, valid, col0, base, N, alpha, beta, cb, bl, v);
            break;
        case SGEMM_ACT_SILU:
            store16_ep<VEC_C, SGEMM_ACT_SILU>(crow, valid, col0, base, N, alpha, beta, cb, bl, v);
            break;
        default: store16_ep<VEC_C, SGEMM_ACT_NONE>(crow, valid, col0, base, N, alpha, beta, cb, bl, v); break;
    }
}

// Writes 32 accumulator values (columns col0 .. col0 + 31 of one row of C):
// C = alpha * v + beta * C (C read only when beta != 0), or, for a tile split
// along K (C already holds beta * C + bias; the activation follows in a
// later pass), C += alpha * v with atomics.
template <bool VEC_C>
__device__ __forceinline__ void store_chunk(const Args &a, float *crow, int64_t row, int64_t col0, const float (&v)[32],
                                            bool atomic) {
    const int64_t N = a.N;
    if (row >= a.M || col0 >= N) return;
    const float alpha = a.alpha, beta = a.beta;
    if (atomic) {
        if (VEC_C && col0 + 31 < N) {
#pragma unroll
            for (int j = 0; j < 32; j += 4)
                red_add_v4(crow + col0 + j, alpha * v[j], alpha * v[j + 1], alpha * v[j + 2], alpha * v[j + 3]);
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (col0 + j < N) atomicAdd(crow + col0 + j, alpha * v[j]);
        }
    } else if (VEC_C && col0 + 31 < N) {
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
            float4 *p = reinterpret_cast<float4 *>(crow + col0 + j);
            float4 o = make_float4(alpha * v[j], alpha * v[j + 1], alpha * v[j + 2], alpha * v[j + 3]);
            if (beta != 0.0f) {
                const float4 c = *p;
                o.x = fmaf(beta, c.x, o.x);
                o.y = fmaf(beta, c.y, o.y);
                o.z = fmaf(beta, c.z, o.z);
                o.w = fmaf(beta, c.w, o.w);
            }
            *p = o;
        }
    } else if (beta == 0.0f) {
        // Separate loops: with beta in the store expression the compiler
        // loads C ahead of every store, beta or not.
#pragma unroll
        for (int j = 0; j < 32; ++j)
            if (col0 + j < N) crow[col0 + j] = alpha * v[j];
    } else {
#pragma unroll
        for (int j = 0; j < 32; ++j)
            if (col0 + j < N) crow[col0 + j] = fmaf(beta, crow[col0 + j], alpha * v[j]);
    }
}

// op(A)[row][k] * op(B)[k][col] summed over k in [k_begin, k_end) with fp32
// fused multiply-adds in k order: IEEE arithmetic, infinities and NaN
// propagating as they do on the CUDA cores. A and B point at the batch
// item's operands; ta: A stored K x M, tb: B stored N x K.
__device__ __forceinline__ float dot_ieee(const float *A, int64_t lda, int ta, const float *B, int64_t ldb, int tb,
                                          int64_t row, int64_t col, int64_t k_begin, int64_t k_end) {
    float s = 0.0f;
#pragma unroll 1
    for (int64_t k = k_begin; k < k_end; ++k) {
        const float x = ta ? A[k * lda + row] : A[row * lda + k];
        const float y = tb ? B[col * ldb + k] : B[k * ldb + col];
        s = fmaf(x, y, s);
    }
    return s;
}

// Non-finite inputs: the three-term split multiplies an infinite high part
// by the NaN low part (inf - inf) of its own value, so an output that summed
// an infinity comes out NaN where IEEE arithmetic gives +-inf. Finite inputs
// never give NaN, so every NaN among v (columns col0 .. col0 + N - 1 of one
// row of batch item `item`, the sum over the k-range [k_begin, k_end)) is
// recomputed there with IEEE arithmetic (dot_ieee); NaN inputs give NaN
// again. Adding such per-range results keeps IEEE's rules (inf + finite =
// inf, inf - inf = NaN). Called by all 32 lanes: one comparison per value
// and a warp vote when nothing is NaN. The repair walks the columns in a
// rolled loop (one copy of the dot product, v kept in registers by selects).
template <int N>
__device__ __forceinline__ void fix_nonfinite(const Args &a, int item, int64_t row, int64_t col0, int64_t k_begin,
                                              int64_t k_end, float (&v)[N]) {
    bool bad = false;
#pragma unroll
    for (int j = 0; j < N; ++j) bad |= v[j] != v[j];
    if (!__any_sync(0xffffffffu, bad)) return;
    const float *A = a.A + (a.a_shared ? 0 : item * a.strideA);
    const float *B = a.B + (a.b_shared ? 0 : item * a.strideB);
    if (k_end > a.K) k_end = a.K;
    const bool in_rows = row < a.M;
#pragma unroll 1
    for (int j = 0; j < N; ++j) {
        float x = 0.0f;
#pragma unroll
        for (int i = 0; i < N; ++i)
            if (i == j) x = v[i];
        if (x == x || !in_rows || col0 + j >= a.N) continue;
        x = dot_ieee(A, a.lda, a.ta, B, a.ldb, a.tb, row, col0 + j, k_begin, k_end);
#pragma unroll
        for (int i = 0; i < N; ++i)
            if (i == j) v[i] = x;
    }
}

// Writes 32 finished values of one row held in registers (columns col0 ..
// col0 + 31): C = act(alpha * v + beta * C + bias) for a whole tile (the bias
// and activation with a fused epilogue), C += alpha * v with atomics for a
// tile split along K. Called by all 32 lanes of the warp (the bias shuffles).
template <bool VEC_C>
__device__ __forceinline__ void store_chunk_regs(const Args &a, float *crow, int64_t row, int64_t col0,
                                                 const float (&v)[32], bool atomic) {
    if (col0 >= a.N) return;  // uniform over the warp
    if (a.ep && !atomic) {
        const int lane = static_cast<int>(threadIdx.x & 31);
        float bl = 0.0f;
        if (a.bias_kind == SGEMM_BIAS_PER_COL && col0 + lane < a.N) bl = __ldg(a.bias + col0 + lane);
        if (a.bias_kind == SGEMM_BIAS_PER_ROW && row < a.M) bl = __ldg(a.bias + row);
        float h[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) h[j] = v[j];
        store16_fused<VEC_C>(a, crow, row, col0, 0, bl, h);
#pragma unroll
        for (int j = 0; j < 16; ++j) h[j] = v[16 + j];
        store16_fused<VEC_C>(a, crow, row, col0 + 16, 16, bl, h);
    } else {
        store_chunk<VEC_C>(a, crow, row, col0, v, atomic);
    }
}

// Writes a 32 x 32 chunk of C held in shared memory (chunk rc, 128-byte
// swizzled rows, row r = row row0 + r, the unit's finished sums) one row per
// step with the lanes along the row, so that each warp store covers 128
// contiguous bytes whatever C's alignment: C = act(alpha * v + beta * C +
// bias) for a whole tile, C += alpha * v with atomics for a tile split along
// K. Rows from M and columns from N on are skipped. Called by all 32 lanes
// after the chunk is complete in shared memory (__syncwarp).
__device__ __forceinline__ void store_staged_rows(const Args &a, uint32_t rc, float *citem, int64_t row0,
                                                  int64_t col0, bool atomic) {
    const int lane = static_cast<int>(threadIdx.x & 31);
    // Parameters in registers: the shared-memory loads below are ordered
    // against all memory, so fields read through `a` would be reloaded on
    // every row.
    const int64_t M = a.M, ldc = a.ldc, col = col0 + lane;
    const bool col_ok = col < a.N;
    const bool fused = a.ep && !atomic;
    const int bias_kind = fused ? a.bias_kind : SGEMM_BIAS_NONE, act = a.act;
    const float *bias = a.bias;
    const float bcol = (bias_kind == SGEMM_BIAS_PER_COL && col_ok) ? __ldg(bias + col) : 0.0f;
    const float alpha = a.alpha, beta = a.beta;
    float *p = citem + row0 * ldc + col;
    if (!fused) {
        // All 32 values first (independent shared loads), then the stores.
        float x[32];
#pragma unroll
        for (int r = 0; r < 32; ++r)
            x[r] = ld_shared_f32(rc + sw128_offset(r, lane >> 2) + static_cast<uint32_t>((lane & 3) * 4));
        if (!col_ok) return;
        const int rows = M - row0 < 32 ? static_cast<int>(M - row0) : 32;
        // Separate loops: with beta in the store expression the compiler
        // loads C ahead of every store, beta or not.
        if (atomic) {
#pragma unroll
            for (int r = 0; r < 32; ++r)
                if (r < rows) atomicAdd(p + r * ldc, alpha * x[r]);
        } else if (beta == 0.0f) {
#pragma unroll
            for (int r = 0; r < 32; ++r)
                if (r < rows) p[r * ldc] = alpha * x[r];
        } else {
#pragma unroll
            for (int r = 0; r < 32; ++r)
                if (r < rows) p[r * ldc] = fmaf(beta, p[r * ldc], alpha * x[r]);
        }
        return;
    }
#pragma unroll 1
    for (int r = 0; r < 32 && row0 + r < M; ++r, p += ldc) {  // the row bound is uniform over the warp
        const float x = ld_shared_f32(rc + sw128_offset(r, lane >> 2) + static_cast<uint32_t>((lane & 3) * 4));
        if (!col_ok) continue;
        float y = alpha * x;
        if (beta != 0.0f) y = fmaf(beta, *p, y);
        y += bias_kind == SGEMM_BIAS_PER_COL ? bcol : (bias_kind == SGEMM_BIAS_PER_ROW ? __ldg(bias + row0 + r) : 0.0f);
        *p = activate(y, act);
    }
}

// Epilogue of one 32-column chunk of the accumulator at TMEM address taddr
// (this thread's lane, the sum over the unit's k-range [k_begin, k_end) of
// batch item `item`): loads it, repairs non-finite outputs (fix_nonfinite)
// and writes C (store_chunk_regs). release: call on_release() once the chunk
// is out of TMEM (the accumulator may be reused).
template <bool VEC_C, class Release>
__device__ __forceinline__ void epilogue_chunk_then(const Args &a, uint32_t taddr, float *crow, int64_t row, int64_t col0,
                                               bool atomic, bool release, Release &&on_release, int item,
                                               int64_t k_begin, int64_t k_end) {
    float v[32];
    tmem_load32(taddr, v);
    if (release) on_release();
    fix_nonfinite(a, item, row, col0, k_begin, k_end, v);
    store_chunk_regs<VEC_C>(a, crow, row, col0, v, atomic);
}

// The same, arriving on the CTA's own mbarrier release_bar to free the
// accumulator.
template <bool VEC_C>
__device__ __forceinline__ void epilogue_chunk(const Args &a, uint32_t taddr, float *crow, int64_t row, int64_t col0,
                                               bool atomic, bool release, uint32_t release_bar, int item,
                                               int64_t k_begin, int64_t k_end) {
    epilogue_chunk_then<VEC_C>(
        a, taddr, crow, row, col0, atomic, release,
        [&] {
            tc_fence_before();
            mbar_arrive(release_bar);
        },
        item, k_begin, k_end);
}

// First split iteration of worker `index` (index = sk_ctas: the end). With
// a.sk_switch_kb = P the split tiles are laid on a line where each is
// followed by a gap of P (none after the last), the line is cut evenly, and
// a cut that falls in a gap moves to the start of the next tile.
__host__ __device__ __forceinline__ int64_t sk_share_start(const Args &a, int index) {
    if (a.sk_switch_kb <= 0 || a.kb_cap > 0 || a.sk_iters <= 0) return a.sk_iters * index / a.sk_ctas;
    const int64_t seg = a.k_blocks + a.sk_switch_kb;
    const int64_t line = (a.sk_iters / a.k_blocks) * seg - a.sk_switch_kb;
    const int64_t v = line * index / a.sk_ctas;
    const int64_t r = v % seg;
    return (v / seg) * a.k_blocks + (r < a.k_blocks ? r : a.k_blocks);
}

// The slowest share of the split iterations: its k-blocks plus `cost` for
// each switch from one split tile to the next inside it (every worker that
// has a share runs the same number of whole tiles).
__host__ __device__ inline int64_t slowest_share(const Args &a, int64_t cost) {
    int64_t worst = 0;
    for (int i = 0; i < a.sk_ctas; ++i) {
        const int64_t s0 = sk_share_start(a, i), s1 = sk_share_start(a, i + 1);
        if (s1 <= s0) continue;
        const int64_t c = (s1 - s0) + cost * ((s1 - 1) / a.k_blocks - s0 / a.k_blocks);
        worst = c > worst ? c : worst;
    }
    return worst;
}

// Sets a.sk_switch_kb: `cost` where counting the switches makes the slowest
// share faster than the even split does, else 0 (an even split that already
// falls on tile boundaries loses to nothing).
inline void count_switches(Args &a, int cost) {
    a.sk_switch_kb = 0;
    if (cost <= 0 || a.sk_ctas <= 0 || a.kb_cap > 0) return;
    const int64_t even = slowest_share(a, cost);
    a.sk_switch_kb = cost;
    if (slowest_share(a, cost) >= even) a.sk_switch_kb = 0;
}

// Calls f(tile, kb, ke) for the units of work of worker `index` of `count`
// (whole tiles round-robin, then its share of the split iterations), in
// order. With a.kb_cap a split unit also ends at every multiple of kb_cap
// k-blocks, so no unit accumulates more than kb_cap k-blocks in TMEM.
template <class F>
__host__ __device__ __forceinline__ void for_each_unit_of(const Args &a, volatile int *abort_flag, int index, int count,
                                                          F &&f) {
    for (int t = index; t < a.dp_tiles; t += count) {
        if (*abort_flag) return;
        f(t, 0, a.k_blocks);
    }
    if (index < a.sk_ctas) {
        int64_t it = sk_share_start(a, index);
        const int64_t end = sk_share_start(a, index + 1);
        while (it < end) {
            if (*abort_flag) return;
            const int tile = a.dp_tiles + static_cast<int>(it / a.k_blocks);
            const int kb = static_cast<int>(it % a.k_blocks);
            const int64_t rest = end - it;
            int ke = static_cast<int>(rest < a.k_blocks - kb ? kb + rest : a.k_blocks);
            if (a.kb_cap > 0) {
                const int lim = (kb / a.kb_cap + 1) * a.kb_cap;
                if (ke > lim) ke = lim;
            }
            f(tile, kb, ke);
            it += ke - kb;
        }
    }
}

// This CTA's units: worker blockIdx.x of gridDim.x.
template <class F>
__device__ __forceinline__ void for_each_unit(const Args &a, volatile int *abort_flag, F &&f) {
    for_each_unit_of(a, abort_flag, static_cast<int>(blockIdx.x), static_cast<int>(gridDim.x), f);
}

// Host side, defined with the kernels in sgemm_tf32x3.cu: a rank-3 tensor
// map over a batch of row-major rows x cols fp32 matrices with row stride ld
// and item stride `stride` (elements; 0 = one matrix shared by all items),
// boxes of box_cols x box_rows x 1, out-of-range elements read as zero.
bool encode_map(CUtensorMap *map, const float *ptr, int64_t rows, int64_t cols, int64_t ld, int64_t batch,
                int64_t stride, uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle swizzle);

}  // namespace tc
}  // namespace sgemm
