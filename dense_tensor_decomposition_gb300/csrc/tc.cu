// Tensor-core (tcgen05 / TMEM) MTTKRP path.
#include <cstdio>

#include "tc.h"

namespace mk {

// Error word set by kernels whose bounded waits expire (read by the host
// through mttkrp_device_status).
__device__ uint32_t g_device_status = 0;

size_t tc_binner_bytes(const ModePlan&) { return 0; }

bool tc_prefer(const ModePlan&) { return false; }

bool tc_plan(ModePlan&) { return false; }

int tc_run(const Plan&, const ModePlan&, const float*, const float* const*, const float*,
           const int64_t*, void*, float*, cudaStream_t, int* nlaunch, cudaEvent_t*, char* errbuf,
           size_t errlen) {
    *nlaunch = 0;
    snprintf(errbuf, errlen, "tensor-core path not available");
    return MTTKRP_ERR_UNSUPPORTED;
}

cudaError_t tc_read_and_clear_status(uint32_t* word) {
    cudaError_t err = cudaDeviceSynchronize();
    if (err != cudaSuccess) return err;
    err = cudaMemcpyFromSymbol(word, g_device_status, sizeof(uint32_t));
    if (err != cudaSuccess) return err;
    const uint32_t zero = 0;
    return cudaMemcpyToSymbol(g_device_status, &zero, sizeof(uint32_t));
}

}  // namespace mk
