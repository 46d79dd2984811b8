// Internal declarations shared by the translation units of libsgemm_gb300.
// Not installed; the public ABI is include/sgemm.h.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace sgemm {

// One product request after argument checks: all pointers are device
// pointers, strides are in elements, M, N, K > 0.
struct Problem {
    int64_t M, N, K;
    const float *A;
    int64_t lda;
    const float *B;
    int64_t ldb;
    float *C;
    int64_t ldc;
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

// Enqueue the FFMA product. `launches` receives the number of kernels enqueued.
int ffma_launch(const Problem &p, const DeviceInfo &dev, int tile, int sk_mode, cudaStream_t stream,
                int *launches);

// Enqueue C[0:M, 0:N] = 0 (the empty sum).
int zero_launch(float *C, int64_t M, int64_t N, int64_t ldc, const DeviceInfo &dev,
                cudaStream_t stream, int *launches);

// Tensor-core three-term TF32 variant. Returns SGEMM_ERR_UNSUPPORTED when it
// cannot run the request.
bool tf32x3_supports(const Problem &p, const DeviceInfo &dev);
int tf32x3_launch(const Problem &p, const DeviceInfo &dev, cudaStream_t stream, int *launches);

// Watchdog flag shared by kernels with bounded waits (one per device, in the
// tf32x3 translation unit). Read-and-clear; returns 0 or the first recorded code.
int watchdog_read_and_clear(int *code);
int64_t watchdog_polls();
int watchdog_set_polls(int64_t polls);

}  // namespace sgemm
