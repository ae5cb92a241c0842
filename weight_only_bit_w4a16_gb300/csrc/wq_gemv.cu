// wq_gemv.cu -- the small-M path: split-K GEMV with register decode feeding
// warp-level tensor-core MMAs.
//
// Shape of the work (C = A . deq(B)^T, M <= 16 per pass):
//   * A warp owns 16 weight rows (n) and a K-slice; per iteration it covers
//     128 k: lane (r = lane/4, c = lane%4) issues one coalesced 128-bit load
//     of rows r and r+8 at k = 32c .. 32c+31 (4 lanes read 64 contiguous
//     bytes of a row).  Up to kPF iterations of packed data are in flight per
//     lane, so the loads are all issued before the first decode.
//   * The codes are unpacked and dequantised in registers (wq_common.cuh) and
//     go straight into mma.sync.m16n8k16 bf16 as the A operand -- the weight
//     rows are the MMA's M dimension and the activations its N = 8 dimension
//     ("swap AB").  The m16n8k16 fragment maps follow the TVM TIRx gemm tile
//     primitive page (Demonstration program, register layouts); since the
//     order of the 16 k slots inside one MMA is free as long as both operands
//     agree, each lane feeds the natural bf16 pairs of its own 32 codes and
//     the matching 16-byte slice of the activation row, with no repacking.
//   * int4 with group % 128 == 0: one iteration is one group, so the MMA runs
//     on the exact integers (code - zero) and the group's scale multiplies the
//     fp32 partial sums afterwards; other formats multiply the decoded weights
//     by their scale before the MMA (bf16 RNE of the exact weight).
//   * K is split over the CTAs of a thread-block cluster (up to 8 CTAs); each
//     CTA stages its K-slice of A once in shared memory (swizzled so that the
//     quarter-warp 128-bit reads hit 8 distinct bank groups), and the partial
//     sums are reduced through distributed shared memory in a fixed rank
//     order -- deterministic, with no global workspace and no atomics.
#include <cooperative_groups.h>

#include "wq_common.cuh"
#include "wq_internal.h"

namespace cg = cooperative_groups;

namespace wq {

namespace {

constexpr int kItK = 128;   // k per warp-iteration
constexpr int kPF = 4;      // iterations of packed data in flight per lane

struct GemvArgs {
    const uint16_t* A;
    const uint8_t* packed;
    const void* scales;
    const uint8_t* zeros;
    void* C;
    int M, N, K, group;
    int out_f32;
    int total_its;     // ceil(K / 128)
    int its_per_cta;   // iterations per CTA of a cluster
};

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 16-byte unit u of activation row m, swizzled inside aligned groups of 16
// units: the 8 lanes of a quarter-warp (2 rows x 4 chunk lanes) land on 8
// different bank groups.
__device__ __forceinline__ int a_unit(int u, int m) { return u ^ ((((u >> 3) & 1) << 1) | (m & 1)); }

__device__ __forceinline__ uint4 lds128(const uint8_t* p) {
    return *reinterpret_cast<const uint4*>(p);
}

// raw scale data of one lane-row for iteration g (k = 128 g + 32 c)
template <int FMT, bool POST>
__device__ __forceinline__ uint32_t load_raw(const GemvArgs& a, int n, int kk) {
    const int gpr = a.K / a.group;
    if constexpr (POST) {
        const size_t gi = (size_t)n * gpr + (size_t)((kk & ~127) / a.group);
        return ldg_u16(static_cast<const uint16_t*>(a.scales) + gi) | (ldg_u8(a.zeros + gi) << 16);
    } else if constexpr (FMT == kNVFP4) {
        // two scales (groups of 16) per 32-code chunk, adjacent bytes
        const uint8_t* s = static_cast<const uint8_t*>(a.scales) + (size_t)n * gpr + (size_t)(kk >> 4);
        return ldg_u8(s) | (ldg_u8(s + 1) << 8);
    } else if constexpr (FMT == kMXFP4) {
        const size_t gi = (size_t)n * gpr + (size_t)(kk >> 5);
        return ldg_u8(static_cast<const uint8_t*>(a.scales) + gi);
    } else {
        const size_t gi = (size_t)n * gpr + (size_t)(kk / a.group);
        return ldg_u16(static_cast<const uint16_t*>(a.scales) + gi) | (ldg_u8(a.zeros + gi) << 16);
    }
}

template <int FMT, bool POST>
__device__ __forceinline__ void keys_of(uint32_t raw, GroupKey& k0, GroupKey& k1, float& s) {
    if constexpr (FMT == kNVFP4) {
        k0 = key_nvfp4(raw & 0xFF);
        k1 = key_nvfp4((raw >> 8) & 0xFF);
        s = 0.f;
    } else if constexpr (FMT == kMXFP4) {
        k0 = key_mxfp4(raw & 0xFF);
        k1 = k0;
        s = 0.f;
    } else {
        k0 = key_int4(raw & 0xFFFF, raw >> 16);
        k1 = k0;
        s = __uint_as_float((raw & 0xFFFFu) << 16);   // bf16 scale as fp32 (exact)
    }
}

// decode + MMA of one iteration (16 rows x 128 k) for one warp
template <int FMT, int NT, bool POST, bool TWO>
__device__ __forceinline__ void iteration_body(const uint4& qa, const uint4& qb, const GroupKey (&ka)[2],
                                               const GroupKey (&kb)[2], const uint8_t* arow0,
                                               const uint8_t* arow1, int ubase, int r, float (&acc)[NT][4],
                                               float sa, float sb) {
    const uint32_t wa[4] = {qa.x, qa.y, qa.z, qa.w};
    const uint32_t wb[4] = {qb.x, qb.y, qb.z, qb.w};
    float part[NT][4];
    if constexpr (POST) {
#pragma unroll
        for (int t = 0; t < NT; ++t)
#pragma unroll
            for (int e = 0; e < 4; ++e) part[t][e] = 0.f;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint32_t pa[4], pb[4];
        const GroupKey& keyA = ka[j >> 1];
        const GroupKey& keyB = kb[j >> 1];
        if constexpr (POST) {
            int4_word_centered<TWO>(wa[j], keyA, pa);
            int4_word_centered<TWO>(wb[j], keyB, pb);
        } else {
            word_scaled<FMT, TWO>(wa[j], keyA, pa);
            word_scaled<FMT, TWO>(wb[j], keyB, pb);
        }
        const int u = ubase + j;
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            const int m = t * 8 + r;
            const uint4 bv = lds128((t == 0 ? arow0 : arow1) + (a_unit(u, m) << 4));
            float (&d)[4] = POST ? part[t] : acc[t];
            mma16816(d, pa[0], pb[0], pa[1], pb[1], bv.x, bv.y);
            mma16816(d, pa[2], pb[2], pa[3], pb[3], bv.z, bv.w);
        }
    }
    if constexpr (POST) {
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            acc[t][0] = fmaf(sa, part[t][0], acc[t][0]);
            acc[t][1] = fmaf(sa, part[t][1], acc[t][1]);
            acc[t][2] = fmaf(sb, part[t][2], acc[t][2]);
            acc[t][3] = fmaf(sb, part[t][3], acc[t][3]);
        }
    }
}

template <int FMT, int NT, bool POST>
__global__ void __launch_bounds__(256) gemv_kernel(const GemvArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int warps = blockDim.x >> 5;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int r = lane >> 2, c = lane & 3;
    const int ks = gridDim.x;          // CTAs of a cluster split K
    const int rank = blockIdx.x;       // == rank inside the cluster
    const int rows_per_cta = warps * 16;
    const int n_cta = blockIdx.y * rows_per_cta;
    const int mz = blockIdx.z * 16;
    const int Mc = min(16, a.M - mz);
    const int it0 = rank * a.its_per_cta;
    const int nit = max(0, min(a.total_its, it0 + a.its_per_cta) - it0);
    const int U = a.its_per_cta * (kItK / 8);   // 16-byte units per staged A row
    uint8_t* a_s = smem;
    float* red = reinterpret_cast<float*>(smem + (size_t)NT * 8 * U * 16);

    // ---- issue the first kPF iterations of packed loads -------------------
    const int nA = n_cta + warp * 16 + r, nB = nA + 8;
    const bool vA = nA < a.N, vB = nB < a.N;
    const uint8_t* pA = a.packed + (size_t)(vA ? nA : 0) * (a.K >> 1) + c * 16;
    const uint8_t* pB = a.packed + (size_t)(vB ? nB : 0) * (a.K >> 1) + c * 16;
    uint4 qa[kPF], qb[kPF];
    uint32_t ra[kPF], rb[kPF];
    const uint4 z4 = make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int s = 0; s < kPF; ++s) {
        if (s < nit) {
            const int kk = (it0 + s) * kItK + c * 32;
            const bool ok = kk < a.K;
            qa[s] = (vA && ok) ? ldg_stream_v4(pA + (size_t)(it0 + s) * 64) : z4;
            qb[s] = (vB && ok) ? ldg_stream_v4(pB + (size_t)(it0 + s) * 64) : z4;
            ra[s] = (vA && ok) ? load_raw<FMT, POST>(a, nA, kk) : 0u;
            rb[s] = (vB && ok) ? load_raw<FMT, POST>(a, nB, kk) : 0u;
        }
    }

    // ---- stage this CTA's K-slice of A (rows mz .. mz+8NT-1) --------------
    {
        const int k0 = it0 * kItK;
        const int units = NT * 8 * U;
        for (int idx = threadIdx.x; idx < units; idx += blockDim.x) {
            const int m = idx / U, u = idx - m * U;
            const int k = k0 + u * 8;
            uint4 v = z4;
            if (m < Mc && u < nit * (kItK / 8) && k < a.K)
                v = *reinterpret_cast<const uint4*>(a.A + (size_t)(mz + m) * a.K + k);
            *reinterpret_cast<uint4*>(a_s + ((size_t)m * U + a_unit(u, m)) * 16) = v;
        }
    }
    __syncthreads();

    float acc[NT][4];
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[t][e] = 0.f;

    const uint8_t* arow0 = a_s + (size_t)(0 * 8 + r) * U * 16;
    const uint8_t* arow1 = a_s + (size_t)((NT - 1) * 8 + r) * U * 16;

    for (int base = 0; base < nit; base += kPF) {
#pragma unroll
        for (int s = 0; s < kPF; ++s) {
            const int i = base + s;
            if (i < nit) {
                const uint4 cqa = qa[s], cqb = qb[s];
                const uint32_t cra = ra[s], crb = rb[s];
                if (i + kPF < nit) {
                    const int g = it0 + i + kPF;
                    const int kk = g * kItK + c * 32;
                    const bool ok = kk < a.K;
                    qa[s] = (vA && ok) ? ldg_stream_v4(pA + (size_t)g * 64) : z4;
                    qb[s] = (vB && ok) ? ldg_stream_v4(pB + (size_t)g * 64) : z4;
                    ra[s] = (vA && ok) ? load_raw<FMT, POST>(a, nA, kk) : 0u;
                    rb[s] = (vB && ok) ? load_raw<FMT, POST>(a, nB, kk) : 0u;
                }
                GroupKey ka[2], kb[2];
                float sa, sb;
                keys_of<FMT, POST>(cra, ka[0], ka[1], sa);
                keys_of<FMT, POST>(crb, kb[0], kb[1], sb);
                const int ubase = i * (kItK / 8) + 4 * c;
                bool two = false;
                if constexpr (FMT != kNVFP4) two = __any_sync(0xffffffffu, ka[0].two || kb[0].two);
                if (two)
                    iteration_body<FMT, NT, POST, true>(cqa, cqb, ka, kb, arow0, arow1, ubase, r, acc, sa, sb);
                else
                    iteration_body<FMT, NT, POST, false>(cqa, cqb, ka, kb, arow0, arow1, ubase, r, acc, sa, sb);
            }
        }
    }

    // ---- partial sums -> shared memory ------------------------------------
    const int MP = NT * 8;
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        const int rowA = warp * 16 + r, rowB = rowA + 8;
        const int m = t * 8 + 2 * c;
        red[rowA * MP + m] = acc[t][0];
        red[rowA * MP + m + 1] = acc[t][1];
        red[rowB * MP + m] = acc[t][2];
        red[rowB * MP + m + 1] = acc[t][3];
    }

    // ---- reduce over the cluster (fixed rank order) and store C -----------
    const int rows_mine = rows_per_cta / ks;
    const int row0 = rank * rows_mine;
    if (ks > 1) {
        cg::cluster_group cluster = cg::this_cluster();
        cluster.sync();
        for (int idx = threadIdx.x; idx < rows_mine * Mc; idx += blockDim.x) {
            const int m = idx / rows_mine, rl = row0 + (idx - m * rows_mine);
            const int n = n_cta + rl;
            float v = 0.f;
            for (int q = 0; q < ks; ++q) v += cluster.map_shared_rank(red, q)[rl * MP + m];
            if (n < a.N) {
                const size_t o = (size_t)(mz + m) * a.N + n;
                if (a.out_f32) static_cast<float*>(a.C)[o] = v;
                else static_cast<__nv_bfloat16*>(a.C)[o] = __float2bfloat16_rn(v);
            }
        }
        cluster.sync();   // keep this CTA's partials alive until all ranks read them
    } else {
        __syncthreads();
        for (int idx = threadIdx.x; idx < rows_per_cta * Mc; idx += blockDim.x) {
            const int m = idx / rows_per_cta, rl = idx - m * rows_per_cta;
            const int n = n_cta + rl;
            if (n < a.N) {
                const float v = red[rl * MP + m];
                const size_t o = (size_t)(mz + m) * a.N + n;
                if (a.out_f32) static_cast<float*>(a.C)[o] = v;
                else static_cast<__nv_bfloat16*>(a.C)[o] = __float2bfloat16_rn(v);
            }
        }
    }
}

template <int FMT, int NT, bool POST>
int launch_inst(const GemvArgs& args, dim3 grid, int threads, size_t smem, cudaStream_t stream) {
    auto kern = gemv_kernel<FMT, NT, POST>;
    if (smem > 48 * 1024) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
            return WQ_ERR_CUDA;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(threads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = grid.x;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = grid.x > 1 ? 1 : 0;
    if (cudaLaunchKernelEx(&cfg, kern, args) != cudaSuccess) return WQ_ERR_CUDA;
    return WQ_OK;
}

}  // namespace

int launch_gemv(const void* A, const uint8_t* packed, const void* scales, const uint8_t* zeros, void* C,
                int M, int N, int K, int fmt, int group, bool out_f32, cudaStream_t stream) {
    if (M == 0 || N == 0) return WQ_OK;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);

    const int total_its = (K + kItK - 1) / kItK;
    const int rowblocks = (N + 15) / 16;
    const int mchunks = (M + 15) / 16;
    // K split over a cluster: enough warps to keep ~kPF iterations of loads
    // in flight on every SM, at most 8 CTAs per cluster
    int ks = 1;
    while (ks < 8 && ks * 2 <= total_its && (long long)rowblocks * ks * mchunks < 2048) ks *= 2;
    const int its_per_cta = total_its ? (total_its + ks - 1) / ks : 0;
    // warps per CTA: the largest power of two that still gives >= 2 CTAs per SM
    int W = 8;
    while (W > 1 && (long long)((rowblocks + W - 1) / W) * ks * mchunks < 2LL * sms) W >>= 1;
    const int NT = (M <= 8) ? 1 : 2;
    const int U = its_per_cta * (kItK / 8);
    const size_t smem = (size_t)NT * 8 * U * 16 + (size_t)W * 16 * NT * 8 * sizeof(float);
    if (smem > 200 * 1024) return WQ_ERR_UNSUPPORTED;
    if ((long long)(rowblocks + W - 1) / W > 65535 || mchunks > 65535) return WQ_ERR_UNSUPPORTED;

    GemvArgs args;
    args.A = static_cast<const uint16_t*>(A);
    args.packed = packed;
    args.scales = scales;
    args.zeros = zeros;
    args.C = C;
    args.M = M;
    args.N = N;
    args.K = K;
    args.group = group;
    args.out_f32 = out_f32 ? 1 : 0;
    args.total_its = total_its;
    args.its_per_cta = its_per_cta;
    const dim3 grid(ks, (rowblocks + W - 1) / W, mchunks);
    const int threads = W * 32;
    const bool post = (fmt == kINT4) && (group % kItK == 0);

    if (fmt == kNVFP4) {
        return NT == 1 ? launch_inst<kNVFP4, 1, false>(args, grid, threads, smem, stream)
                       : launch_inst<kNVFP4, 2, false>(args, grid, threads, smem, stream);
    }
    if (fmt == kMXFP4) {
        return NT == 1 ? launch_inst<kMXFP4, 1, false>(args, grid, threads, smem, stream)
                       : launch_inst<kMXFP4, 2, false>(args, grid, threads, smem, stream);
    }
    if (post) {
        return NT == 1 ? launch_inst<kINT4, 1, true>(args, grid, threads, smem, stream)
                       : launch_inst<kINT4, 2, true>(args, grid, threads, smem, stream);
    }
    return NT == 1 ? launch_inst<kINT4, 1, false>(args, grid, threads, smem, stream)
                   : launch_inst<kINT4, 2, false>(args, grid, threads, smem, stream);
}

}  // namespace wq
