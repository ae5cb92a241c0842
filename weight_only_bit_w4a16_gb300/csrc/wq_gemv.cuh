// wq_gemv.cuh -- device pieces shared by the small-M kernels: the warp-level
// bf16 MMA, the swizzled activation addressing, the in-register int4 decode
// in (k, k+4) pair order and one 16-row x 128-k iteration of work.
//
// Fragment maps of mma.sync.m16n8k16 follow the TVM TIRx gemm tile primitive
// page (Demonstration program, register layouts).  The weight rows are the
// MMA's M dimension and the activations its N = 8 dimension ("swap AB").  The
// order of the 16 k slots inside one MMA is free as long as both operands
// agree, so each lane feeds the bf16 pairs of its own 32 codes and the
// matching 16-byte slice of the activation row, with no repacking.
#pragma once

#include "wq_common.cuh"
#include "wq_tc.cuh"

namespace wq {
namespace gemv {

constexpr int kItK = 128;          // k per warp-iteration
constexpr int kModeInt4 = 0;       // int4 with group 128: exact (code - zero), scale after the MMA
constexpr int kModeScaled = 1;     // every other case: weights scaled before the MMA

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

// defined with the tensor-core primitives (wq_tc.cuh)
using sm100::fence_proxy_async_smem;
using sm100::grid_dependency_wait;
using sm100::grid_dependents_launch;

__device__ __forceinline__ uint4 lds128(uint32_t saddr) {
    uint4 v;
    asm("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(saddr));
    return v;
}

__device__ __forceinline__ uint2 lds64(uint32_t saddr) {
    uint2 v;
    asm("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(saddr));
    return v;
}

__device__ __forceinline__ uint32_t lds16(uint32_t saddr) {
    uint16_t v;
    asm("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(saddr));
    return v;
}

// global -> shared bulk copy completing on an mbarrier (16-byte aligned
// addresses, size a multiple of 16)
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}

__device__ __forceinline__ void named_barrier(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// D = A . B with a zero accumulator input (the chain starts fresh; no
// per-iteration re-zeroing of partial sums)
__device__ __forceinline__ void mma16816_z(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                           uint32_t b0, uint32_t b1) {
    const float z = 0.f;
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%10, %11, %12, %13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(z), "f"(z), "f"(z), "f"(z));
}

template <int FMT>
__device__ __forceinline__ void keys_of(uint32_t raw, GroupKey& k0, GroupKey& k1) {
    if constexpr (FMT == kNVFP4) {
        k0 = key_nvfp4(raw & 0xFF);
        k1 = key_nvfp4((raw >> 8) & 0xFF);
    } else if constexpr (FMT == kMXFP4) {
        k0 = key_mxfp4(raw & 0xFF);
        k1 = k0;
    } else {
        k0 = key_int4(raw & 0xFFFF, raw >> 16);
        k1 = k0;
    }
}

// bf16x2 subtrahends of a zero point: (128 + z) for z <= 128 (0x4300 + z is
// exactly 128 + z, the carry of z = 128 moving into the exponent), else 128
// and then z itself
// Branch-free: zz = 128 + min(z, 128) (exact; 0x4300 + z is 128 + z, the
// carry of z = 128 moving into the exponent), zz2 = z - min(z, 128) as a bf16
// integer (0..127: exact, its float bits truncate to bf16 without rounding).
__device__ __forceinline__ void zero_subtrahends(uint32_t z, uint32_t& zz, uint32_t& zz2) {
    const uint32_t zc = min(z, 128u);
    zz = 0x43004300u + zc * 0x10001u;
    const float d = __uint_as_float(0x4B000000u | (z - zc)) - 8388608.0f;
    zz2 = (__float_as_uint(d) >> 16) * 0x10001u;
}

// One iteration (16 rows x 128 k) of the int4 group-128 path: the MMAs run on
// the exact integers (code - zero); the group's scale multiplies the fp32
// partial sums afterwards ("subtract before multiply").  Two accumulation
// chains shorten the dependent MMA sequence.
template <int NT, bool TWO>
__device__ __forceinline__ void iteration_int4(const uint4& qa, const uint4& qb, const uint32_t (&abase)[NT][4],
                                               int ioff, float (&acc)[NT][4], uint32_t zzA,
                                               uint32_t zzA2, uint32_t zzB, uint32_t zzB2, float sa, float sb) {
    const uint32_t wa[4] = {qa.x, qa.y, qa.z, qa.w};
    const uint32_t wb[4] = {qb.x, qb.y, qb.z, qb.w};
    float part[2][NT][4];
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int t = 0; t < NT; ++t)
#pragma unroll
            for (int e = 0; e < 4; ++e) part[h][t][e] = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint32_t pa[4], pb[4];
        int4_word_kk4<TWO>(wa[j], zzA, zzA2, pa);
        int4_word_kk4<TWO>(wb[j], zzB, zzB2, pb);
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            const uint4 bv = lds128(abase[t][j] + ioff);
            mma16816(part[j & 1][t], pa[0], pb[0], pa[1], pb[1], bv.x, bv.y);
            mma16816(part[j & 1][t], pa[2], pb[2], pa[3], pb[3], bv.z, bv.w);
        }
    }
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        acc[t][0] = fmaf(sa, part[0][t][0] + part[1][t][0], acc[t][0]);
        acc[t][1] = fmaf(sa, part[0][t][1] + part[1][t][1], acc[t][1]);
        acc[t][2] = fmaf(sb, part[0][t][2] + part[1][t][2], acc[t][2]);
        acc[t][3] = fmaf(sb, part[0][t][3] + part[1][t][3], acc[t][3]);
    }
}

// One iteration of the generic path: weights decoded with their scale (bf16
// RNE of the exact weight) in natural pair order, then the MMAs.
template <int FMT, int NT, bool TWO>
__device__ __forceinline__ void iteration_scaled(const uint4& qa, const uint4& qb, const GroupKey (&ka)[2],
                                                 const GroupKey (&kb)[2], const uint32_t (&abase)[NT][4],
                                                 int ioff, float (&acc)[NT][4]) {
    const uint32_t wa[4] = {qa.x, qa.y, qa.z, qa.w};
    const uint32_t wb[4] = {qb.x, qb.y, qb.z, qb.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint32_t pa[4], pb[4];
        word_scaled<FMT, TWO>(wa[j], ka[j >> 1], pa);
        word_scaled<FMT, TWO>(wb[j], kb[j >> 1], pb);
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            const uint4 bv = lds128(abase[t][j] + ioff);
            mma16816(acc[t], pa[0], pb[0], pa[1], pb[1], bv.x, bv.y);
            mma16816(acc[t], pa[2], pb[2], pa[3], pb[3], bv.z, bv.w);
        }
    }
}

// One iteration (16 rows x 128 k), int4 group 128: the MMAs run on the exact
// integers (code - zero) in one chain per activation tile, the group's scale
// multiplies the fp32 partial sums afterwards ("subtract before multiply").
//   ap[t] : the lane's activation address for tile t in this iteration
template <int NT, bool TWO>
__device__ __forceinline__ void it_int4(const uint4& qa, const uint4& qb, const uint32_t (&ap)[NT],
                                        float (&acc)[NT][4], uint32_t zzA, uint32_t zzA2, uint32_t zzB,
                                        uint32_t zzB2, float sa, float sb) {
    const uint32_t wa[4] = {qa.x, qa.y, qa.z, qa.w};
    const uint32_t wb[4] = {qb.x, qb.y, qb.z, qb.w};
    // CH independent MMA chains per tile (words j = h mod CH): with one tile
    // two chains keep the dependent sequence 4 deep; two tiles already are
    // two chains
    constexpr int CH = NT == 1 ? 2 : 1;
    float part[CH][NT][4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint32_t pa[4], pb[4];
        int4_word_kk4<TWO>(wa[j], zzA, zzA2, pa);
        int4_word_kk4<TWO>(wb[j], zzB, zzB2, pb);
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            const uint4 bv = lds128(ap[t] + 64 * j);
            if (j < CH) mma16816_z(part[j % CH][t], pa[0], pb[0], pa[1], pb[1], bv.x, bv.y);
            else mma16816(part[j % CH][t], pa[0], pb[0], pa[1], pb[1], bv.x, bv.y);
            mma16816(part[j % CH][t], pa[2], pb[2], pa[3], pb[3], bv.z, bv.w);
        }
    }
#pragma unroll
    for (int t = 0; t < NT; ++t) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            float p = part[0][t][e];
            if constexpr (CH == 2) p += part[CH - 1][t][e];
            acc[t][e] = fmaf(e < 2 ? sa : sb, p, acc[t][e]);
        }
    }
}

// two outputs rounded to bf16 (RNE), the first in the low half
__device__ __forceinline__ uint32_t bf16x2_bits(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

// The final stores of a small-M CTA, plain output in 16-byte pieces: 8 bf16
// or 4 fp32 outputs per thread and pass.  red holds the Wk warps' partial
// sums, [warp][MP activation rows][ld] floats with the CTA's 2^outs_log2
// weight rows contiguous (ld a multiple of 4, the rows 16-byte aligned);
// each output sums them in warp order from 0, as the scalar stores do, so
// both give the same bits.  C must be 16-byte aligned and N a multiple of 8
// (bf16) or 4 (fp32); n0 and n_end are then multiples of a piece.
// These stores run after the preceding call has completed and before this
// one can, so on a chain of calls they are on its critical path: a 16-row
// ring call's scalar 2-byte stores took ~2.4 us there (per-CTA stamps).
template <int MP>
__device__ __forceinline__ void store_pieces(const float* red, int ld, int Wk, int Mc, int outs_log2, int n0,
                                             int n_end, int mz, int N, void* C, bool out_f32, int tid, int nthreads) {
    const int vl2 = out_f32 ? 2 : 3;       // log2 outputs per piece
    const int pl2 = outs_log2 - vl2;       // log2 pieces per activation row
    for (int i = tid; i < (Mc << pl2); i += nthreads) {
        const int m = i >> pl2, rl = (i & ((1 << pl2) - 1)) << vl2;
        const int n = n0 + rl;
        if (n >= n_end) continue;
        const float* src = red + (size_t)m * ld + rl;
        float4 v0 = make_float4(0.f, 0.f, 0.f, 0.f), v1 = v0;
        for (int q = 0; q < Wk; ++q) {
            const float4 x0 = *reinterpret_cast<const float4*>(src + (size_t)q * MP * ld);
            v0.x += x0.x;
            v0.y += x0.y;
            v0.z += x0.z;
            v0.w += x0.w;
            if (!out_f32) {
                const float4 x1 = *reinterpret_cast<const float4*>(src + (size_t)q * MP * ld + 4);
                v1.x += x1.x;
                v1.y += x1.y;
                v1.z += x1.z;
                v1.w += x1.w;
            }
        }
        const size_t o = (size_t)(mz + m) * N + n;
        if (out_f32) {
            *reinterpret_cast<float4*>(static_cast<float*>(C) + o) = v0;
        } else {
            const uint4 w = make_uint4(bf16x2_bits(v0.x, v0.y), bf16x2_bits(v0.z, v0.w), bf16x2_bits(v1.x, v1.y),
                                       bf16x2_bits(v1.z, v1.w));
            *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(C) + o) = w;
        }
    }
}

}  // namespace gemv
}  // namespace wq
