// Aligned copies of operands whose rows TMA cannot address.
//
// A tensor map needs a 16-byte aligned base and row strides that are
// multiples of 16 bytes. A row-major operand with, say, 1537 floats per row
// ("CUDA内存优化入门：从Naive到Tiled矩阵乘法", section 六: sizes that are not
// multiples of the tile) has neither, so the tensor-core path would have to
// load it with per-thread copies, several times slower than TMA. Instead the
// operand is copied once into rows of a multiple of 4 floats in scratch
// memory (a memory-bound pass over the operand: read once, written once) and
// the product runs on the TMA kernels. Scratch comes from a stream-ordered
// pool the library owns per device, or from a buffer the caller supplies.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "sgemm.h"
#include "sgemm_internal.h"

namespace sgemm {
namespace {

constexpr int kMaxDevices = 64;
constexpr int COPY_THREADS = 256;
constexpr uint64_t kPoolKeepBytes = 512ull << 20;  // retained by the pool between calls

// One matrix (or strided batch of matrices) to copy: `items` matrices of
// rows x cols floats, row stride ld_src / ld_dst, item stride stride_src /
// stride_dst (dst rows 16-byte aligned: ld_dst % 4 == 0, dst 16-byte aligned).
struct CopyJob {
    const float *src;
    float *dst;
    int64_t rows, cols, ld_src, ld_dst, stride_src, stride_dst, items;
};

// Two copies in one launch. A block copies whole rows (job 0's rows first,
// then job 1's); its warps take the row's segments of 128 floats in turn,
// two at a time, with four scalar loads and four scalar stores per lane per
// segment, each warp instruction covering 128 contiguous bytes on both sides.
// The product kernel is launched as this grid's programmatic dependent: every
// block signals at once (all blocks are resident together, see repack_into)
// and the product waits (griddepcontrol.wait) before it reads the copies.
constexpr int SEG = 128;
constexpr int WARPS = COPY_THREADS / 32;

__global__ void __launch_bounds__(COPY_THREADS, 8) repack_kernel(const CopyJob j0, const CopyJob j1) {
    asm volatile("griddepcontrol.launch_dependents;");
    const int64_t rows0 = j0.rows * j0.items;
    const int64_t total = rows0 + j1.rows * j1.items;
    const int lane = static_cast<int>(threadIdx.x & 31), warp = static_cast<int>(threadIdx.x >> 5);
    for (int64_t r = blockIdx.x; r < total; r += gridDim.x) {
        const bool first = r < rows0;
        const int64_t rr = first ? r : r - rows0;
        const int64_t rows = first ? j0.rows : j1.rows, cols = first ? j0.cols : j1.cols;
        const int64_t item = rr / rows, row = rr - item * rows;
        const float *s = (first ? j0.src : j1.src) + item * (first ? j0.stride_src : j1.stride_src) +
                         row * (first ? j0.ld_src : j1.ld_src);
        float *d = (first ? j0.dst : j1.dst) + item * (first ? j0.stride_dst : j1.stride_dst) +
                   row * (first ? j0.ld_dst : j1.ld_dst);
        for (int64_t c0 = static_cast<int64_t>(warp) * SEG + lane; c0 < cols; c0 += 2 * WARPS * SEG) {
            float v[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int64_t c = c0 + (q >> 2) * WARPS * SEG + 32 * (q & 3);
                v[q] = c < cols ? __ldg(s + c) : 0.0f;
            }
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int64_t c = c0 + (q >> 2) * WARPS * SEG + 32 * (q & 3);
                if (c < cols) d[c] = v[q];
            }
        }
    }
}

struct PoolSlot {
    std::once_flag once;
    cudaMemPool_t pool = nullptr;
};
PoolSlot g_pool[kMaxDevices];

cudaMemPool_t scratch_pool(int device) {
    if (device < 0 || device >= kMaxDevices) return nullptr;
    std::call_once(g_pool[device].once, [device] {
        cudaMemPoolProps props{};
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = device;
        cudaMemPool_t pool = nullptr;
        if (cudaMemPoolCreate(&pool, &props) != cudaSuccess) {
            cudaGetLastError();
            return;
        }
        uint64_t keep = kPoolKeepBytes;
        if (cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep) != cudaSuccess) cudaGetLastError();
        g_pool[device].pool = pool;
    });
    return g_pool[device].pool;
}

int64_t round4(int64_t x) { return (x + 3) / 4 * 4; }
int64_t round64(int64_t x) { return (x + 63) / 64 * 64; }

// The stored shape of an operand: op(A) = A is M x K, A^T is stored K x M.
void stored_a(const Problem &p, int64_t *rows, int64_t *cols) {
    *rows = p.transA ? p.K : p.M;
    *cols = p.transA ? p.M : p.K;
}
void stored_b(const Problem &p, int64_t *rows, int64_t *cols) {
    *rows = p.transB ? p.N : p.K;
    *cols = p.transB ? p.K : p.N;
}

// Layout of the copies in the scratch buffer (offsets in floats).
struct Plan {
    bool copy_a = false, copy_b = false;
    int64_t a_rows = 0, a_cols = 0, a_ld = 0, a_items = 0, a_stride = 0, a_off = 0;
    int64_t b_rows = 0, b_cols = 0, b_ld = 0, b_items = 0, b_stride = 0, b_off = 0;
    int64_t floats = 0;
};

Plan plan_for(const Problem &p) {
    Plan pl;
    pl.copy_a = !tma_operand_ok(p.A, p.lda, p.strideA, p.transA ? p.K : p.M, p.batch);
    pl.copy_b = !tma_operand_ok(p.B, p.ldb, p.strideB, p.transB ? p.N : p.K, p.batch);
    int64_t off = 0;
    if (pl.copy_a) {
        stored_a(p, &pl.a_rows, &pl.a_cols);
        pl.a_ld = round4(pl.a_cols);
        pl.a_items = p.strideA == 0 ? 1 : p.batch;
        pl.a_stride = pl.a_items > 1 ? pl.a_rows * pl.a_ld : 0;
        pl.a_off = off;
        off = round64(off + pl.a_items * pl.a_rows * pl.a_ld);
    }
    if (pl.copy_b) {
        stored_b(p, &pl.b_rows, &pl.b_cols);
        pl.b_ld = round4(pl.b_cols);
        pl.b_items = p.strideB == 0 ? 1 : p.batch;
        pl.b_stride = pl.b_items > 1 ? pl.b_rows * pl.b_ld : 0;
        pl.b_off = off;
        off = round64(off + pl.b_items * pl.b_rows * pl.b_ld);
    }
    pl.floats = off;
    return pl;
}

}  // namespace

bool tma_operand_ok(const float *X, int64_t ld, int64_t stride, int64_t rows, int64_t batch) {
    return reinterpret_cast<uintptr_t>(X) % 16 == 0 && ld % 4 == 0 && stride % 4 == 0 &&
           // batch items that overlap cannot be described as a tensor
           (batch == 1 || stride == 0 || stride >= rows * ld);
}

size_t repack_bytes(const Problem &p) {
    if (p.M <= 0 || p.N <= 0 || p.K <= 0 || p.batch <= 0) return 0;
    return static_cast<size_t>(plan_for(p).floats) * sizeof(float);
}

int repack_into(const Problem &p, const DeviceInfo &dev, float *scratch, size_t bytes, cudaStream_t stream,
                Problem *q, int *launches) {
    const Plan pl = plan_for(p);
    *q = p;
    if (!pl.copy_a && !pl.copy_b) return SGEMM_OK;
    if (!scratch || reinterpret_cast<uintptr_t>(scratch) % 16 != 0 ||
        bytes < static_cast<size_t>(pl.floats) * sizeof(float))
        return SGEMM_ERR_INVALID_ARG;
    CopyJob j[2] = {};
    int n = 0;
    if (pl.copy_a) {
        j[n++] = CopyJob{p.A, scratch + pl.a_off, pl.a_rows, pl.a_cols, p.lda, pl.a_ld, p.strideA, pl.a_stride,
                         pl.a_items};
        q->A = scratch + pl.a_off;
        q->lda = pl.a_ld;
        q->strideA = pl.a_stride;
    }
    if (pl.copy_b) {
        j[n++] = CopyJob{p.B, scratch + pl.b_off, pl.b_rows, pl.b_cols, p.ldb, pl.b_ld, p.strideB, pl.b_stride,
                         pl.b_items};
        q->B = scratch + pl.b_off;
        q->ldb = pl.b_ld;
        q->strideB = pl.b_stride;
    }
    // j[1] stays empty (zero rows) when only one operand is copied. At most
    // 8 blocks of 256 threads per SM: the whole grid is resident at once, so
    // a product launched as its programmatic dependent never waits for SMs
    // that blocks of this grid still have to reach.
    const int64_t rows = j[0].rows * j[0].items + j[1].rows * j[1].items;
    const int64_t blocks = rows < 8LL * dev.sm_count ? rows : 8LL * dev.sm_count;
    repack_kernel<<<static_cast<unsigned>(blocks > 0 ? blocks : 1), COPY_THREADS, 0, stream>>>(j[0], j[1]);
    if (cudaGetLastError() != cudaSuccess) return SGEMM_ERR_LAUNCH;
    ++*launches;
    return SGEMM_OK;
}

float *scratch_alloc(const DeviceInfo &dev, size_t bytes, cudaStream_t stream) {
    cudaMemPool_t pool = scratch_pool(dev.device);
    if (!pool || bytes == 0) return nullptr;
    void *ptr = nullptr;
    if (cudaMallocFromPoolAsync(&ptr, bytes, pool, stream) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    return static_cast<float *>(ptr);
}

void scratch_free(float *ptr, cudaStream_t stream) {
    if (ptr && cudaFreeAsync(ptr, stream) != cudaSuccess) cudaGetLastError();
}

}  // namespace sgemm
