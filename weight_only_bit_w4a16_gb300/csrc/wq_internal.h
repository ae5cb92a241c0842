// wq_internal.h -- host-side launchers behind the C ABI (not exported).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/wq.h"
#include "wq_common.cuh"

namespace wq {

// All launchers assume validated arguments and return a WQ_* status.
int launch_dequant(const uint8_t* packed, const void* scales, const uint8_t* zeros, void* W, int N,
                   int K, int fmt, int group, cudaStream_t stream);

// pdl: launch with programmatic dependent launch (the kernel streams its
// weights before the preceding kernel on the stream has finished)
// inputs_ready: A was complete before the chain of overlapped launches
// began, so the kernel may read it at once and wait for its predecessor only
// before storing C (implies pdl)
int launch_gemv(const void* A, const uint8_t* packed, const void* scales, const uint8_t* zeros,
                void* C, int M, int N, int K, int fmt, int group, bool out_f32, bool pdl, bool inputs_ready,
                const Epilogue& epi, cudaStream_t stream);

// The streaming small-M kernel (all of a CTA's weights requested by TMA up
// front).  Returns WQ_ERR_UNSUPPORTED (without launching) for shapes it does
// not take; launch_gemv then uses the register-streaming kernels.
int launch_gemv_tma(const void* A, const uint8_t* packed, const void* scales, const uint8_t* zeros,
                    void* C, int M, int N, int K, int fmt, int group, bool out_f32, bool pdl, bool inputs_ready,
                    const Epilogue& epi, cudaStream_t stream);

// Returns WQ_ERR_UNSUPPORTED (without launching) for shapes the tensor-core
// kernel does not take.  With a workspace of at least tc_workspace_bytes()
// (zero-initialised before its first use; every completed call leaves it
// zero) the kernel may split tiles across CTAs (stream-K); without one each
// CTA computes whole tiles.  pdl: launched with programmatic dependent
// launch -- the grid may start while its predecessor on the stream runs, and
// reads A, and writes C, only after the predecessor has completed.
int launch_tc(const void* A, const uint8_t* packed, const void* scales, const uint8_t* zeros,
              void* C, int M, int N, int K, int fmt, int group, bool out_f32, void* workspace,
              size_t workspace_bytes, const Epilogue& epi, bool pdl, cudaStream_t stream);
size_t tc_workspace_bytes(int M, int N, int K, int fmt);

// The tensor-core kernel on prepacked weights (same contract as launch_tc;
// one k-step of 128 rows is 8 row blocks' half blocks).
int launch_tc_prepacked(const void* A, const void* prepacked, void* C, int M, int N, int K, int fmt, int group,
                        bool out_f32, void* workspace, size_t workspace_bytes, const Epilogue& epi, bool pdl,
                        cudaStream_t stream);

// The prepacked layout (include/wq.h, above wq_prepack_bytes): its size,
// the repack kernel, and the small-M kernel that reads it (any M, up to 16
// activation rows per CTA; WQ_ERR_UNSUPPORTED for K > 16384).
size_t prepack_bytes(int N, int K, int fmt);
int launch_prepack(const uint8_t* packed, const void* scales, const uint8_t* zeros, void* out, int N, int K,
                   int fmt, cudaStream_t stream);
int launch_gemv_prepacked(const void* A, const void* prepacked, void* C, int M, int N, int K, int fmt,
                          bool out_f32, bool pdl, bool inputs_ready, const Epilogue& epi, cudaStream_t stream);
// the staged small-M kernel on prepacked weights (dependent and plain calls)
int launch_gemv_staged(const void* A, const void* prepacked, void* C, int M, int N, int K, int fmt, bool out_f32,
                       bool pdl, bool inputs_ready, const Epilogue& epi, cudaStream_t stream);

// The library's own stream-K scratch (a file-scope device array of the
// tensor-core module) on the current device and its size; NULL if the
// address cannot be had (status WQ_ERR_CUDA).  After a call reported a
// timeout (read_and_clear_device_status), it first zeroes the scratch's flag
// words on `stream`.
void* static_workspace(size_t* bytes, cudaStream_t stream, int* status);

// A kernel whose bounded wait is bound to run out (tests the failure path).
int launch_timeout_selftest(cudaStream_t stream);

// Device status words of the current device (one per kernel module): read
// and clear; the first non-zero one wins.
int read_and_clear_device_status();
int read_and_clear_gemv_status();
int read_and_clear_pre_status();
int read_and_clear_staged_status();

// WQ_DEBUG=1 in the environment prints why a call was refused.
bool debug_on();

// 2D tiled tensor map (row-major, `inner` elements per row, `outer` rows,
// rows `row_bytes` apart) through the driver entry point, no libcuda link.
bool encode_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
               uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw);

}  // namespace wq
