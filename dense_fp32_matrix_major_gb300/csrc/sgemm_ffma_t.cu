// FFMA kernel family, transposed forms: op(A) = A^T and/or op(B) = B^T (the
// template and its design notes are in ffma_impl.cuh and sgemm_ffma.cu).
// A transposed A is copied row for row (16-byte copies when its rows are
// aligned); a transposed B goes through 4-byte transposing copies into a
// swizzled Bs, so every alignment is served.
#include <cuda_runtime.h>
#include <stdint.h>

#include "ffma_impl.cuh"

namespace sgemm {
namespace {

using namespace ffma;

template <class C>
int launch_t(const Problem &p, const DeviceInfo &dev, int sk_mode, cudaStream_t stream, int *launches) {
    const bool vb = (p.ldb % 4 == 0) && (p.strideB % 4 == 0) && (reinterpret_cast<uintptr_t>(p.B) % 16 == 0);
    if (p.transA && p.transB) return launch_cfg<C, true, true, false, false>(p, dev, sk_mode, stream, launches);
    if (p.transB) return launch_cfg<C, false, true, false, false>(p, dev, sk_mode, stream, launches);
    if (vb) return launch_cfg<C, true, false, true, false>(p, dev, sk_mode, stream, launches);
    return launch_cfg<C, true, false, false, false>(p, dev, sk_mode, stream, launches);
}

}  // namespace

int ffma_launch_t(const Problem &p, const DeviceInfo &dev, int tile, int sk_mode, cudaStream_t stream,
                  int *launches) {
    switch (pick_tile(p, dev, tile)) {
        case FFMA_TILE_128x256: return launch_t<CfgBig>(p, dev, sk_mode, stream, launches);
        case FFMA_TILE_128x128: return launch_t<CfgMid>(p, dev, sk_mode, stream, launches);
        case FFMA_TILE_64x64: return launch_t<CfgSmall>(p, dev, sk_mode, stream, launches);
        default: return SGEMM_ERR_INVALID_ARG;
    }
}

}  // namespace sgemm
