// wq_prepack.cu -- the offline repack of a weight into the prepacked layout
// defined above wq_prepack_bytes in include/wq.h.
//
// The KBench megakernel_int4_weight_decode.py spec lets the untimed build
// step store the weights in whatever layout suits the kernel (nibble order,
// fragment order, scales apart from the codes) as long as the 4-bit codes
// are what is streamed per call.  This layout serves the small-M
// kernel (wq_gemv_pre.cu):
//   - a 16-row x 128-k block is 1024 contiguous bytes, so a warp's whole
//     slice (16 rows x its k range) is one bulk copy, with no row padding;
//   - in a half-row the words are stored w0 w4 w1 w5 | w2 w6 w3 w7 and the
//     two 16-byte halves of rows with bit 2 set are exchanged: a lane of the
//     mma.sync fragment reads its two words of a half as one 8-byte load, a
//     half-warp's loads cover 128 distinct bytes, and a lane's four words of a
//     128-k block are the k units c, c + 4, c + 8, c + 12 -- exactly the
//     activation units at 16-byte offsets 16c + 64j of the natural row, so
//     the activations are copied as they are (no permutation);
//   - int4 words hold the pairs (k0 + 2s, k0 + 2s + 1) in nibbles (s, s + 4),
//     so the one-mask decode gives bf16 pairs of consecutive k;
//   - the int4 records hold each row's bf16 scale and uint8 zero point, rows
//     r and r + 8 side by side (one 4-byte and one 2-byte load per lane);
//     the loop forms the subtrahend 128 + z from the zero byte with one
//     byte permute, and a flag after the records says whether any zero
//     point exceeds 128 (then it is subtracted in two exact steps).
// A half block (16 rows x 64 k, 512 bytes) has the byte placement of a tile
// of 32-byte rows under the 32-byte swizzle (16-byte chunks exchanged on bit
// 2 of the row), the placement a tensor-map copy of 64 k of the natural rows
// would give, up to the order of the words.
#include <cstdint>

#include "wq_internal.h"

namespace wq {
namespace {

constexpr int kBlockBytes = 1024;

__host__ __device__ constexpr int record_block_bytes(int fmt) {
    return fmt == kINT4 ? 48 : (fmt == kNVFP4 ? 128 : 64);
}
// int4: the flag block after the record blocks (byte 0: a zero point > 128)
constexpr int kFlagBytes = 16;

// int4: nibble q of the input word holds k0 + q; the output word holds
// k0 + 2s in nibble s and k0 + 2s + 1 in nibble s + 4
__device__ __forceinline__ uint32_t int4_pair_order(uint32_t v) {
    uint32_t o = 0;
#pragma unroll
    for (int s = 0; s < 4; ++s) {
        o |= ((v >> (8 * s)) & 0xFu) << (4 * s);
        o |= ((v >> (8 * s + 4)) & 0xFu) << (16 + 4 * s);
    }
    return o;
}

// One warp per code block (b, i); lane = (row r, half h).  Lanes of half 0
// also write their row's record.
template <int FMT>
__global__ void __launch_bounds__(256) prepack_kernel(const uint8_t* __restrict__ packed,
                                                      const void* __restrict__ scales,
                                                      const uint8_t* __restrict__ zeros, uint8_t* __restrict__ out,
                                                      int N, int K, int Nb, int I) {
    const long long blk = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (blk >= (long long)Nb * I) return;
    const int lane = threadIdx.x & 31;
    const int b = (int)(blk / I), i = (int)(blk % I);
    const int r = lane >> 1, h = lane & 1;
    const int n = 16 * b + r;
    const int kh = K >> 1;                       // packed bytes per row (a multiple of 8)
    const int byte0 = 64 * i + 32 * h;           // first packed byte of this half-row
    uint32_t w[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        uint32_t v = 0;
        const int bo = byte0 + 4 * u;
        if (n < N && bo < kh) v = __ldg(reinterpret_cast<const uint32_t*>(packed + (size_t)n * kh + bo));
        if constexpr (FMT == kINT4) v = int4_pair_order(v);
        w[u] = v;
    }
    uint4 lo = make_uint4(w[0], w[4], w[1], w[5]), hi = make_uint4(w[2], w[6], w[3], w[7]);
    if ((r >> 2) & 1) {
        const uint4 t = lo;
        lo = hi;
        hi = t;
    }
    uint8_t* dst = out + (size_t)blk * kBlockBytes + 512 * h + 32 * r;
    reinterpret_cast<uint4*>(dst)[0] = lo;
    reinterpret_cast<uint4*>(dst)[1] = hi;

    if (h != 0) return;
    uint8_t* rec = out + (size_t)Nb * I * kBlockBytes + (size_t)blk * record_block_bytes(FMT);
    if constexpr (FMT == kINT4) {
        uint32_t s = 0, z = 0;
        if (n < N) {
            const size_t gi = (size_t)n * (K >> 7) + i;
            s = static_cast<const uint16_t*>(scales)[gi];
            z = zeros[gi];
        }
        *reinterpret_cast<uint16_t*>(rec + 4 * (r & 7) + 2 * (r >> 3)) = (uint16_t)s;
        rec[32 + 2 * (r & 7) + (r >> 3)] = (uint8_t)z;
        if (z > 128u) {   // the flag block follows the last record block (zeroed before this kernel)
            const size_t at = (size_t)Nb * I * (kBlockBytes + record_block_bytes(kINT4));
            uint32_t* flag = reinterpret_cast<uint32_t*>(out + at);
            atomicOr(flag, 1u);
        }
    } else {
        constexpr int per = FMT == kNVFP4 ? 8 : 4;   // groups of a row in a 128-k block
        const int ng = K / (FMT == kNVFP4 ? 16 : 32);
        const uint8_t* sc = static_cast<const uint8_t*>(scales);
#pragma unroll
        for (int g = 0; g < per; ++g) {
            const int gi = per * i + g;
            rec[per * r + g] = (n < N && gi < ng) ? sc[(size_t)n * ng + gi] : (uint8_t)0;
        }
    }
}

}  // namespace

size_t prepack_bytes(int N, int K, int fmt) {
    const size_t nb = (size_t)(N + 15) / 16, nk = (size_t)(K + 127) / 128;
    return nb * nk * (size_t)(kBlockBytes + record_block_bytes(fmt)) + (fmt == kINT4 ? kFlagBytes : 0);
}

int launch_prepack(const uint8_t* packed, const void* scales, const uint8_t* zeros, void* out, int N, int K,
                   int fmt, cudaStream_t stream) {
    const int Nb = (N + 15) / 16, I = (K + 127) / 128;
    const long long blocks = ((long long)Nb * I + 7) / 8;
    if (blocks > 0x7FFFFFFFLL) return WQ_ERR_UNSUPPORTED;
    uint8_t* o = static_cast<uint8_t*>(out);
    if (fmt == kINT4 &&
        cudaMemsetAsync(o + (size_t)Nb * I * (kBlockBytes + record_block_bytes(kINT4)), 0, kFlagBytes, stream) !=
            cudaSuccess)
        return WQ_ERR_CUDA;
    if (fmt == kINT4)
        prepack_kernel<kINT4><<<(unsigned)blocks, 256, 0, stream>>>(packed, scales, zeros, o, N, K, Nb, I);
    else if (fmt == kNVFP4)
        prepack_kernel<kNVFP4><<<(unsigned)blocks, 256, 0, stream>>>(packed, scales, zeros, o, N, K, Nb, I);
    else
        prepack_kernel<kMXFP4><<<(unsigned)blocks, 256, 0, stream>>>(packed, scales, zeros, o, N, K, Nb, I);
    return cudaGetLastError() == cudaSuccess ? WQ_OK : WQ_ERR_CUDA;
}

}  // namespace wq
