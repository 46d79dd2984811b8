// Tensor-core variant (tcgen05, three-term TF32 split). Placeholder until the
// kernel lands: it reports every shape as unsupported, so AUTO picks FFMA.
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "sgemm.h"
#include "sgemm_internal.h"

namespace sgemm {

// Per-device watchdog flag: 0, or the code of the first bounded wait that gave up.
__device__ int g_watchdog_code;

namespace {
std::atomic<int64_t> g_polls{INT64_C(1) << 24};
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

int64_t watchdog_polls() { return g_polls.load(); }

int watchdog_set_polls(int64_t polls) {
    if (polls < 1024) return SGEMM_ERR_INVALID_ARG;
    g_polls.store(polls);
    return SGEMM_OK;
}

bool tf32x3_supports(const Problem &, const DeviceInfo &) { return false; }

int tf32x3_launch(const Problem &, const DeviceInfo &, cudaStream_t, int *) { return SGEMM_ERR_UNSUPPORTED; }

}  // namespace sgemm
