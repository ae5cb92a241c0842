// wq_tc.cu -- the large-M tensor-core path (tcgen05 / TMEM) and the device
// status word that its bounded waits report into.
#include "wq_common.cuh"
#include "wq_internal.h"

namespace wq {

// WQ_OK, or WQ_ERR_DEVICE_TIMEOUT once a bounded wait of a kernel gave up.
__device__ int g_device_status = 0;

int read_and_clear_device_status() {
    int v = 0;
    const int zero = 0;
    if (cudaDeviceSynchronize() != cudaSuccess) return WQ_ERR_CUDA;
    if (cudaMemcpyFromSymbol(&v, g_device_status, sizeof(int)) != cudaSuccess) return WQ_ERR_CUDA;
    if (cudaMemcpyToSymbol(g_device_status, &zero, sizeof(int)) != cudaSuccess) return WQ_ERR_CUDA;
    return v;
}

int launch_tc(const void*, const uint8_t*, const void*, const uint8_t*, void*, int, int, int, int, int, bool,
              cudaStream_t) {
    return WQ_ERR_UNSUPPORTED;
}

}  // namespace wq
