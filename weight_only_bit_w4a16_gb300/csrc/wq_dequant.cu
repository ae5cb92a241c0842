// wq_dequant.cu -- W = deq(packed, scales, zeros) as an (N, K) bf16 matrix.
//
// One thread per 16-byte chunk of a packed row (32 codes = 4 words): one
// coalesced 128-bit load, the register decode of wq_common.cuh (the same
// routine the GEMM kernels feed to the tensor cores), four 128-bit stores.
// Each weight is the round-to-nearest-even bf16 image of its exact value, so
// the result equals the oracle's bf16 image bit for bit.  The decode always
// takes the two-step form here: the extra exact step (x - 0, x * 1) changes
// no bit and keeps every thread on one path.
#include "wq_common.cuh"
#include "wq_internal.h"

namespace wq {

template <int FMT>
__global__ void __launch_bounds__(256) dequant_kernel(const uint8_t* __restrict__ packed,
                                                     const void* __restrict__ scales,
                                                     const uint8_t* __restrict__ zeros,
                                                     uint16_t* __restrict__ W, int N, int K, int group) {
    const int chunks_per_row = K >> 5;
    const long long total = (long long)N * chunks_per_row;
    const int groups_per_row = K / group;
    for (long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x; t < total;
         t += (long long)gridDim.x * blockDim.x) {
        const int n = (int)(t / chunks_per_row);
        const int j = (int)(t - (long long)n * chunks_per_row);
        const uint4 q = ldg_stream_v4(packed + (size_t)n * (K >> 1) + (size_t)j * 16);
        const uint32_t wds[4] = {q.x, q.y, q.z, q.w};
        const size_t gbase = (size_t)n * groups_per_row;
        uint4* out = reinterpret_cast<uint4*>(W + (size_t)n * K + (size_t)j * 32);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            // element index of the word's first code within the row
            const int k = j * 32 + i * 8;
            const GroupKey key = load_key<FMT>(scales, zeros, gbase + (size_t)(k / group));
            uint32_t p[4];
            word_scaled<FMT, true>(wds[i], key, p);
            out[i] = make_uint4(p[0], p[1], p[2], p[3]);
        }
    }
}

int launch_dequant(const uint8_t* packed, const void* scales, const uint8_t* zeros, void* W, int N,
                   int K, int fmt, int group, cudaStream_t stream) {
    const long long total = (long long)N * (K >> 5);
    if (total == 0) return WQ_OK;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int threads = 256;
    long long blocks = (total + threads - 1) / threads;
    const long long cap = (long long)sms * 16;
    if (blocks > cap) blocks = cap;
    uint16_t* Wp = static_cast<uint16_t*>(W);
    switch (fmt) {
        case kNVFP4:
            dequant_kernel<kNVFP4><<<(int)blocks, threads, 0, stream>>>(packed, scales, zeros, Wp, N, K, group);
            break;
        case kMXFP4:
            dequant_kernel<kMXFP4><<<(int)blocks, threads, 0, stream>>>(packed, scales, zeros, Wp, N, K, group);
            break;
        default:
            dequant_kernel<kINT4><<<(int)blocks, threads, 0, stream>>>(packed, scales, zeros, Wp, N, K, group);
            break;
    }
    return cudaGetLastError() == cudaSuccess ? WQ_OK : WQ_ERR_CUDA;
}

}  // namespace wq
