// wq_internal.h -- host-side launchers behind the C ABI (not exported).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/wq.h"

namespace wq {

// All launchers assume validated arguments and return a WQ_* status.
int launch_dequant(const uint8_t* packed, const void* scales, const uint8_t* zeros, void* W, int N,
                   int K, int fmt, int group, cudaStream_t stream);

// pdl: launch with programmatic dependent launch (the kernel streams its
// weights before the preceding kernel on the stream has finished)
int launch_gemv(const void* A, const uint8_t* packed, const void* scales, const uint8_t* zeros,
                void* C, int M, int N, int K, int fmt, int group, bool out_f32, bool pdl, cudaStream_t stream);

// Returns WQ_ERR_UNSUPPORTED (without launching) for shapes the tensor-core
// kernel does not take.
int launch_tc(const void* A, const uint8_t* packed, const void* scales, const uint8_t* zeros,
              void* C, int M, int N, int K, int fmt, int group, bool out_f32, cudaStream_t stream);

// A kernel whose bounded wait is bound to run out (tests the failure path).
int launch_timeout_selftest(cudaStream_t stream);

// Device status word of the current device: read and clear.
int read_and_clear_device_status();

}  // namespace wq
