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
//     fp32 partial sums afterwards.  The codes are unpacked in the (k, k+4)
//     pair order a mask-and-or produces directly (no byte permutes), and the
//     activations are staged in that same order once per CTA.  Other formats
//     multiply the decoded weights by their scale before the MMA (bf16 RNE of
//     the exact weight) in natural pair order.
//   * K is split over the CTAs of a thread-block cluster (up to 8 CTAs); each
//     CTA stages its K-slice of A once in shared memory (swizzled so that the
//     quarter-warp 128-bit reads hit 8 distinct bank groups), and the partial
//     sums are reduced through distributed shared memory in a fixed rank
//     order -- deterministic, with no global workspace and no atomics.
#include <cooperative_groups.h>
#include <cstdlib>
#include <cstring>

#include "wq_gemv.cuh"
#include "wq_internal.h"

namespace cg = cooperative_groups;

namespace wq {

namespace {

using namespace gemv;

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
    int its_per_cta;   // iterations per CTA of a cluster (cluster kernel) / per warp (split kernel)
    int row_blocks;    // split kernel: 16-row blocks per CTA
    int wk_log2;       // split kernel: log2 of the warps that split K for one row block
    Epilogue epi;
};

// Scale / zero-point sources of one row: its scale bytes and zero points.
struct RowScales {
    const uint8_t* s;   // scales of the row (bytes)
    const uint8_t* z;   // zero points of the row (int4), else unused
};

template <int FMT>
__device__ __forceinline__ RowScales row_scales(const GemvArgs& a, int n) {
    const size_t g0 = (size_t)n * (a.K / a.group);
    RowScales rs;
    if constexpr (FMT == kINT4) rs.s = reinterpret_cast<const uint8_t*>(static_cast<const uint16_t*>(a.scales) + g0);
    else rs.s = static_cast<const uint8_t*>(a.scales) + g0;
    rs.z = (FMT == kINT4) ? a.zeros + g0 : nullptr;
    return rs;
}

// Raw scale word of one lane-row for iteration g (k = 128 g + 32 c):
//   int4 group 128    : bf16 scale | zero << 16 of group g
//   nvfp4             : the two e4m3 bytes of groups 8g + 2c, 8g + 2c + 1
//   mxfp4             : the e8m0 byte of group 4g + c
//   int4 otherwise    : bf16 scale | zero << 16 of group (128 g + 32 c) / group
// A chunk past K reads group 0 and returns 0, a zero scale that zeroes its
// weights (its activations are zero as well).
template <int FMT, int MODE>
__device__ __forceinline__ uint32_t load_raw(const GemvArgs& a, const RowScales& rs, int g, int c, bool ok) {
    if constexpr (MODE == kModeInt4) {
        const int gi = ok ? g : 0;
        const uint32_t v = ldg_u16(rs.s + 2 * (size_t)gi) | (ldg_u8(rs.z + gi) << 16);
        return ok ? v : 0u;
    } else if constexpr (FMT == kNVFP4) {
        const uint8_t* p = rs.s + (ok ? (size_t)g * 8 + 2 * c : 0);
        const uint32_t v = ldg_u8(p) | (ldg_u8(p + 1) << 8);
        return ok ? v : 0u;
    } else if constexpr (FMT == kMXFP4) {
        const uint32_t v = ldg_u8(rs.s + (ok ? (size_t)g * 4 + c : 0));
        return ok ? v : 0u;
    } else {
        const int gi = ok ? (g * kItK + c * 32) / a.group : 0;
        const uint32_t v = ldg_u16(rs.s + 2 * (size_t)gi) | (ldg_u8(rs.z + gi) << 16);
        return ok ? v : 0u;
    }
}

// 16 packed bytes and the raw scale word of one lane-row for iteration g,
// with no branches: rows past N read row 0 (their results are never stored),
// a chunk past K reads the row's first chunk under a zero scale word.
template <int FMT, int MODE>
__device__ __forceinline__ void fetch(const GemvArgs& a, const uint8_t* prow, const RowScales& rs, int g, int c,
                                      uint4& q, uint32_t& raw) {
    const bool ok = g * kItK + c * 32 < a.K;
    q = ldg_stream_v4(prow + (ok ? (size_t)g * 64 + c * 16 : 0));
    raw = load_raw<FMT, MODE>(a, rs, g, c, ok);
}

template <int FMT, int NT, int MODE>
__global__ void __launch_bounds__(256) gemv_cluster_kernel(const GemvArgs a) {
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
    constexpr int MP = NT * 8;                  // staged activation rows
    uint8_t* a_s = smem;
    float* red = reinterpret_cast<float*>(smem + (size_t)MP * U * 16);   // [rows][MP]

    // ---- issue the first kPF iterations of packed loads -------------------
    const int nA = n_cta + warp * 16 + r, nB = nA + 8;
    const bool vA = nA < a.N, vB = nB < a.N;
    const uint8_t* pA = a.packed + (size_t)(vA ? nA : 0) * (a.K >> 1);
    const uint8_t* pB = a.packed + (size_t)(vB ? nB : 0) * (a.K >> 1);
    const RowScales sA = row_scales<FMT>(a, vA ? nA : 0);
    const RowScales sB = row_scales<FMT>(a, vB ? nB : 0);
    uint4 qa[kPF], qb[kPF];
    uint32_t ra[kPF], rb[kPF];
    const uint4 z4 = make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int s = 0; s < kPF; ++s) {
        if (s < nit) {
            fetch<FMT, MODE>(a, pA, sA, it0 + s, c, qa[s], ra[s]);
            fetch<FMT, MODE>(a, pB, sB, it0 + s, c, qb[s], rb[s]);
        }
    }

    // the next kernel on the stream may start (programmatic dependent launch);
    // A is read, and C written, only after the preceding kernel has finished
    grid_dependents_launch();
    grid_dependency_wait();

    // ---- stage this CTA's K-slice of A (rows mz .. mz+MP-1) ---------------
    {
        const int k0 = it0 * kItK;
        const int ulim = min(nit * (kItK / 8), (a.K - k0) >> 3);   // units holding data
#pragma unroll 1
        for (int m = 0; m < MP; ++m) {
            const bool mv = m < Mc;
            const uint16_t* arow = a.A + (size_t)(mz + (mv ? m : 0)) * a.K + k0;
            uint8_t* srow = a_s + (size_t)m * U * 16;
            for (int u = threadIdx.x; u < U; u += blockDim.x) {
                uint4 v = z4;
                if (mv && u < ulim) v = *reinterpret_cast<const uint4*>(arow + u * 8);
                if constexpr (MODE == kModeInt4) {
                    // the (k, k+4) pair order the int4 decode produces
                    v = make_uint4(prmt(v.x, v.z, 0x5410u), prmt(v.x, v.z, 0x7632u), prmt(v.y, v.w, 0x5410u),
                                   prmt(v.y, v.w, 0x7632u));
                }
                *reinterpret_cast<uint4*>(srow + a_unit(u, m) * 16) = v;
            }
        }
    }
    __syncthreads();

    float acc[NT][4];
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[t][e] = 0.f;

    // per-lane shared-memory addresses of the activation fragments of word j
    // in iteration 0 (iteration i adds 256 bytes * i): unit 4c + (j ^ x)
    uint32_t abase[NT][4];   // rows past M are staged as zeros
    {
        const int x = (((c >> 1) & 1) << 1) | (r & 1);
        const uint32_t s0 = static_cast<uint32_t>(__cvta_generic_to_shared(a_s));
#pragma unroll
        for (int t = 0; t < NT; ++t)
#pragma unroll
            for (int j = 0; j < 4; ++j) abase[t][j] = s0 + ((t * 8 + r) * U + 4 * c + (j ^ x)) * 16;
    }

    for (int base = 0; base < nit; base += kPF) {
#pragma unroll
        for (int s = 0; s < kPF; ++s) {
            const int i = base + s;
            if (i < nit) {
                const uint4 cqa = qa[s], cqb = qb[s];
                const uint32_t cra = ra[s], crb = rb[s];
                if (i + kPF < nit) {
                    fetch<FMT, MODE>(a, pA, sA, it0 + i + kPF, c, qa[s], ra[s]);
                    fetch<FMT, MODE>(a, pB, sB, it0 + i + kPF, c, qb[s], rb[s]);
                }
                const int ioff = i * (kItK / 8) * 16;
                if constexpr (MODE == kModeInt4) {
                    uint32_t zzA, zzA2, zzB, zzB2;
                    zero_subtrahends(cra >> 16, zzA, zzA2);
                    zero_subtrahends(crb >> 16, zzB, zzB2);
                    const float sa = __uint_as_float((cra & 0xFFFFu) << 16);   // bf16 scale, exact in fp32
                    const float sb = __uint_as_float((crb & 0xFFFFu) << 16);
                    if (__any_sync(0xffffffffu, (zzA2 | zzB2) != 0))
                        iteration_int4<NT, true>(cqa, cqb, abase, ioff, acc, zzA, zzA2, zzB, zzB2, sa, sb);
                    else
                        iteration_int4<NT, false>(cqa, cqb, abase, ioff, acc, zzA, zzA2, zzB, zzB2, sa, sb);
                } else {
                    GroupKey ka[2], kb[2];
                    keys_of<FMT>(cra, ka[0], ka[1]);
                    keys_of<FMT>(crb, kb[0], kb[1]);
                    bool two = false;
                    if constexpr (FMT != kNVFP4) two = __any_sync(0xffffffffu, ka[0].two || kb[0].two);
                    if (two)
                        iteration_scaled<FMT, NT, true>(cqa, cqb, ka, kb, abase, ioff, acc);
                    else
                        iteration_scaled<FMT, NT, false>(cqa, cqb, ka, kb, abase, ioff, acc);
                }
            }
        }
    }

    // ---- partial sums -> shared memory ------------------------------------
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
        for (int rl = row0 + (int)threadIdx.x; rl < row0 + rows_mine; rl += blockDim.x) {
            const int n = n_cta + rl;
            if (n >= a.N) continue;
            if (a.epi.gated && (rl & 8)) continue;   // an up row: stored with its gate row
            float v[MP], u[MP];
#pragma unroll
            for (int m = 0; m < MP; ++m) v[m] = u[m] = 0.f;
            for (int q = 0; q < ks; ++q) {
                const float* src = cluster.map_shared_rank(red, q) + rl * MP;
#pragma unroll
                for (int m = 0; m < MP; ++m) v[m] += src[m];
                if (a.epi.gated) {
#pragma unroll
                    for (int m = 0; m < MP; ++m) u[m] += src[8 * MP + m];
                }
            }
#pragma unroll
            for (int m = 0; m < MP; ++m)
                if (m < Mc) store_epilogue(a.epi, a.C, a.out_f32, a.N, mz + m, n, v[m], u[m]);
        }
        cluster.sync();   // keep this CTA's partials alive until all ranks read them
    } else {
        __syncthreads();
        for (int rl = threadIdx.x; rl < rows_per_cta; rl += blockDim.x) {
            const int n = n_cta + rl;
            if (n >= a.N) continue;
            if (a.epi.gated && (rl & 8)) continue;   // an up row: stored with its gate row
            for (int m = 0; m < Mc; ++m)
                store_epilogue(a.epi, a.C, a.out_f32, a.N, mz + m, n, red[rl * MP + m],
                               a.epi.gated ? red[(rl + 8) * MP + m] : 0.f);
        }
    }
}

// The split-K-in-CTA kernel: a CTA owns `row_blocks` blocks of 16 rows and
// all of K; its row_blocks x Wk warps split K Wk ways, the activations
// (M <= 16 rows, all of K) are staged once per CTA, and the partial sums meet
// in one shared-memory reduction in a fixed warp order.  No cluster, no
// global workspace.  Used whenever the staged activations fit comfortably in
// shared memory; larger M x K goes to the cluster kernel above.
template <int FMT, int NT, int MODE>
__global__ void __launch_bounds__(NT == 1 ? 512 : 256) gemv_kernel(const GemvArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int r = lane >> 2, c = lane & 3;
    const int Wk = 1 << a.wk_log2;
    const int rb = warp >> a.wk_log2, kw = warp & (Wk - 1);
    const int rows_per_cta = a.row_blocks * 16;
    const int n_cta = blockIdx.x * rows_per_cta;
    const int mz = blockIdx.y * 16;
    const int Mc = min(16, a.M - mz);
    const int it0 = kw * a.its_per_cta;
    const int nit = max(0, min(a.total_its, it0 + a.its_per_cta) - it0);
    const int U = a.total_its * (kItK / 8);     // 16-byte units per staged A row (all of K)
    constexpr int MP = NT * 8;
    uint8_t* a_s = smem;                                                     // [Mc][U]
    float* red = reinterpret_cast<float*>(smem + (size_t)Mc * U * 16);      // [rows][Wk][MP]

    // ---- issue the first kPF iterations of packed loads -------------------
    const int nA = n_cta + rb * 16 + r, nB = nA + 8;
    const bool vA = nA < a.N, vB = nB < a.N;
    const uint8_t* pA = a.packed + (size_t)(vA ? nA : 0) * (a.K >> 1);
    const uint8_t* pB = a.packed + (size_t)(vB ? nB : 0) * (a.K >> 1);
    const RowScales sA = row_scales<FMT>(a, vA ? nA : 0);
    const RowScales sB = row_scales<FMT>(a, vB ? nB : 0);
    uint4 qa[kPF], qb[kPF];
    uint32_t ra[kPF], rb_[kPF];
    const uint4 z4 = make_uint4(0, 0, 0, 0);
    // int4 group 128 (K % 128 == 0): this lane's chunk, scale and zero of
    // iteration it0, advanced by pointer bumps with immediate offsets
    const uint8_t* qpA = pA + (size_t)it0 * 64 + c * 16;
    const uint8_t* qpB = pB + (size_t)it0 * 64 + c * 16;
    const uint16_t* spA = reinterpret_cast<const uint16_t*>(sA.s) + it0;
    const uint16_t* spB = reinterpret_cast<const uint16_t*>(sB.s) + it0;
    const uint8_t* zpA = sA.z + it0;
    const uint8_t* zpB = sB.z + it0;
#pragma unroll
    for (int s = 0; s < kPF; ++s) {
        if (s < nit) {
            if constexpr (MODE == kModeInt4) {
                qa[s] = ldg_stream_v4(qpA + s * 64);
                qb[s] = ldg_stream_v4(qpB + s * 64);
                ra[s] = ldg_u16(spA + s) | (ldg_u8(zpA + s) << 16);
                rb_[s] = ldg_u16(spB + s) | (ldg_u8(zpB + s) << 16);
            } else {
                fetch<FMT, MODE>(a, pA, sA, it0 + s, c, qa[s], ra[s]);
                fetch<FMT, MODE>(a, pB, sB, it0 + s, c, qb[s], rb_[s]);
            }
        }
    }

    // the next kernel on the stream may start (programmatic dependent launch);
    // A is read, and C written, only after the preceding kernel has finished
    grid_dependents_launch();
    grid_dependency_wait();

    // ---- stage the activations (rows mz .. mz+Mc-1, all of K) -------------
    {
        const int ulim = a.K >> 3;
#pragma unroll 1
        for (int m = 0; m < Mc; ++m) {
            const uint16_t* arow = a.A + (size_t)(mz + m) * a.K;
            uint8_t* srow = a_s + (size_t)m * U * 16;
            for (int u = threadIdx.x; u < U; u += blockDim.x) {
                uint4 v = z4;
                if (u < ulim) v = *reinterpret_cast<const uint4*>(arow + u * 8);
                if constexpr (MODE == kModeInt4) {
                    v = make_uint4(prmt(v.x, v.z, 0x5410u), prmt(v.x, v.z, 0x7632u), prmt(v.y, v.w, 0x5410u),
                                   prmt(v.y, v.w, 0x7632u));
                }
                *reinterpret_cast<uint4*>(srow + a_unit(u, m) * 16) = v;
            }
        }
    }
    __syncthreads();

    float acc[NT][4];
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[t][e] = 0.f;

    // activation rows past Mc are not staged: those lanes read row 0, which
    // only feeds MMA columns (m >= Mc) that are never stored
    uint32_t abase[NT][4];
    {
        const int x = (((c >> 1) & 1) << 1) | (r & 1);
        const uint32_t s0 = static_cast<uint32_t>(__cvta_generic_to_shared(a_s));
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            const int m = t * 8 + r;
            const int ms = m < Mc ? m : 0;
#pragma unroll
            for (int j = 0; j < 4; ++j) abase[t][j] = s0 + (ms * U + 4 * c + (j ^ x)) * 16;
        }
    }

    if constexpr (MODE == kModeInt4) {
        // compute from the ring slot first, then refill it kPF iterations ahead
        int ioff = it0 * (kItK / 8) * 16;
        for (int base = 0; base < nit; base += kPF) {
#pragma unroll
            for (int s = 0; s < kPF; ++s) {
                if (base + s < nit) {
                    uint32_t zzA, zzA2, zzB, zzB2;
                    zero_subtrahends(ra[s] >> 16, zzA, zzA2);
                    zero_subtrahends(rb_[s] >> 16, zzB, zzB2);
                    const float sa = __uint_as_float((ra[s] & 0xFFFFu) << 16);   // bf16 scale, exact in fp32
                    const float sb = __uint_as_float((rb_[s] & 0xFFFFu) << 16);
                    const int off = ioff + s * (kItK / 8) * 16;
                    if (__any_sync(0xffffffffu, (zzA2 | zzB2) != 0))
                        iteration_int4<NT, true>(qa[s], qb[s], abase, off, acc, zzA, zzA2, zzB, zzB2, sa, sb);
                    else
                        iteration_int4<NT, false>(qa[s], qb[s], abase, off, acc, zzA, zzA2, zzB, zzB2, sa, sb);
                    if (base + s + kPF < nit) {
                        qa[s] = ldg_stream_v4(qpA + (s + kPF) * 64);
                        qb[s] = ldg_stream_v4(qpB + (s + kPF) * 64);
                        ra[s] = ldg_u16(spA + s + kPF) | (ldg_u8(zpA + s + kPF) << 16);
                        rb_[s] = ldg_u16(spB + s + kPF) | (ldg_u8(zpB + s + kPF) << 16);
                    }
                }
            }
            qpA += kPF * 64;
            qpB += kPF * 64;
            spA += kPF;
            spB += kPF;
            zpA += kPF;
            zpB += kPF;
            ioff += kPF * (kItK / 8) * 16;
        }
    } else {
    for (int base = 0; base < nit; base += kPF) {
#pragma unroll
        for (int s = 0; s < kPF; ++s) {
            const int i = base + s;
            if (i < nit) {
                const uint4 cqa = qa[s], cqb = qb[s];
                const uint32_t cra = ra[s], crb = rb_[s];
                if (i + kPF < nit) {
                    fetch<FMT, MODE>(a, pA, sA, it0 + i + kPF, c, qa[s], ra[s]);
                    fetch<FMT, MODE>(a, pB, sB, it0 + i + kPF, c, qb[s], rb_[s]);
                }
                const int ioff = (it0 + i) * (kItK / 8) * 16;
                if constexpr (false) {
                    uint32_t zzA, zzA2, zzB, zzB2;
                    zero_subtrahends(cra >> 16, zzA, zzA2);
                    zero_subtrahends(crb >> 16, zzB, zzB2);
                    const float sa = __uint_as_float((cra & 0xFFFFu) << 16);
                    const float sb = __uint_as_float((crb & 0xFFFFu) << 16);
                    if (__any_sync(0xffffffffu, (zzA2 | zzB2) != 0))
                        iteration_int4<NT, true>(cqa, cqb, abase, ioff, acc, zzA, zzA2, zzB, zzB2, sa, sb);
                    else
                        iteration_int4<NT, false>(cqa, cqb, abase, ioff, acc, zzA, zzA2, zzB, zzB2, sa, sb);
                } else {
                    GroupKey ka[2], kb[2];
                    keys_of<FMT>(cra, ka[0], ka[1]);
                    keys_of<FMT>(crb, kb[0], kb[1]);
                    bool two = false;
                    if constexpr (FMT != kNVFP4) two = __any_sync(0xffffffffu, ka[0].two || kb[0].two);
                    if (two)
                        iteration_scaled<FMT, NT, true>(cqa, cqb, ka, kb, abase, ioff, acc);
                    else
                        iteration_scaled<FMT, NT, false>(cqa, cqb, ka, kb, abase, ioff, acc);
                }
            }
        }
    }

    }

    // ---- warp partials -> shared memory, reduce in fixed order, store -----
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        const int rowA = rb * 16 + r, rowB = rowA + 8;
        const int m = t * 8 + 2 * c;
        float* ra_ = red + ((size_t)rowA * Wk + kw) * MP;
        float* rb2 = red + ((size_t)rowB * Wk + kw) * MP;
        ra_[m] = acc[t][0];
        ra_[m + 1] = acc[t][1];
        rb2[m] = acc[t][2];
        rb2[m + 1] = acc[t][3];
    }
    __syncthreads();
    for (int rl = threadIdx.x; rl < rows_per_cta; rl += blockDim.x) {
        const int n = n_cta + rl;
        if (n >= a.N) continue;
        if (a.epi.gated && (rl & 8)) continue;   // an up row: stored with its gate row
        float v[MP], u[MP];
#pragma unroll
        for (int m = 0; m < MP; ++m) v[m] = u[m] = 0.f;
        for (int q = 0; q < Wk; ++q) {
            const float* src = red + ((size_t)rl * Wk + q) * MP;
#pragma unroll
            for (int m = 0; m < MP; ++m) v[m] += src[m];
            if (a.epi.gated) {
                const float* up = red + ((size_t)(rl + 8) * Wk + q) * MP;
#pragma unroll
                for (int m = 0; m < MP; ++m) u[m] += up[m];
            }
        }
#pragma unroll
        for (int m = 0; m < MP; ++m)
            if (m < Mc) store_epilogue(a.epi, a.C, a.out_f32, a.N, mz + m, n, v[m], u[m]);
    }
}

template <typename Kern>
int launch_kernel(Kern kern, const GemvArgs& args, dim3 grid, int threads, size_t smem, int cluster_x, bool pdl,
                  cudaStream_t stream) {
    if (smem > 48 * 1024) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
            return WQ_ERR_CUDA;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(threads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (cluster_x > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = cluster_x;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    if (pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    if (cudaLaunchKernelEx(&cfg, kern, args) != cudaSuccess) return WQ_ERR_CUDA;
    return WQ_OK;
}

template <int FMT, int NT, int MODE>
int launch_inst(const GemvArgs& args, dim3 grid, int threads, size_t smem, int cluster_x, bool split_kernel,
                bool pdl, cudaStream_t stream) {
    if (split_kernel)
        return launch_kernel(gemv_kernel<FMT, NT, MODE>, args, grid, threads, smem, 1, pdl, stream);
    return launch_kernel(gemv_cluster_kernel<FMT, NT, MODE>, args, grid, threads, smem, cluster_x, pdl, stream);
}

}  // namespace

int launch_gemv(const void* A, const uint8_t* packed, const void* scales, const uint8_t* zeros, void* C,
                int M, int N, int K, int fmt, int group, bool out_f32, bool pdl, bool inputs_ready,
                const Epilogue& epi, cudaStream_t stream) {
    // the register-streaming kernels below read A after the dependency wait
    // whatever the caller declared, which is always correct
    if (inputs_ready) pdl = true;
    if (M == 0 || N == 0) return WQ_OK;
    // WQ_GEMV_KERNEL=split|cluster (tests, tuning) skips the streaming kernel
    const char* force = getenv("WQ_GEMV_KERNEL");
    const bool force_cluster = getenv("WQ_GEMV_FORCE_CLUSTER") || (force && !strcmp(force, "cluster"));
    const bool force_split = force && !strcmp(force, "split");
    if (!force_cluster && !force_split) {
        const int st = launch_gemv_tma(A, packed, scales, zeros, C, M, N, K, fmt, group, out_f32, pdl, inputs_ready,
                                       epi, stream);
        if (st != WQ_ERR_UNSUPPORTED) return st;
    }
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);

    const int total_its = (K + kItK - 1) / kItK;
    const int rowblocks = (N + 15) / 16;
    const int mchunks = (M + 15) / 16;
    const int Mc = M < 16 ? M : 16;
    const int NT = (Mc <= 8) ? 1 : 2;
    const int MP = NT * 8;
    const bool int4_g128 = (fmt == kINT4) && (group == kItK);

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
    args.epi = epi;

    // split-K inside one CTA when the staged activations (Mc rows, all of K)
    // leave room for two CTAs per SM
    const int R = (Mc > 8) ? 2 : 1;
    const int max_warps = NT == 1 ? 16 : 8;   // the kernel's launch bounds
    int wk_log2 = 0;
    while ((2 << wk_log2) * R <= max_warps && (2 << wk_log2) <= total_its &&
           (long long)rowblocks * (1 << wk_log2) * mchunks < 2048)
        ++wk_log2;
    if (const char* e = getenv("WQ_GEMV_WK_LOG2")) {
        const int v = atoi(e);
        if (v >= 0 && v <= 4 && (1 << v) * R <= max_warps) wk_log2 = v;
    }
    const int Wk = 1 << wk_log2;
    const size_t smem_split = (size_t)Mc * total_its * kItK * 2 + (size_t)R * 16 * Wk * MP * sizeof(float);
    const bool split_kernel = smem_split <= 112 * 1024 && !force_cluster;

    dim3 grid;
    int threads, cluster_x = 1;
    size_t smem;
    if (split_kernel) {
        args.its_per_cta = total_its ? (total_its + Wk - 1) / Wk : 0;
        args.row_blocks = R;
        args.wk_log2 = wk_log2;
        grid = dim3((rowblocks + R - 1) / R, mchunks, 1);
        threads = R * Wk * 32;
        smem = smem_split;
        if (grid.x > 0x7FFFFFFF || mchunks > 65535) return WQ_ERR_UNSUPPORTED;
    } else {
        // K split over a cluster: enough warps to keep ~kPF iterations of loads
        // in flight on every SM, at most 8 CTAs per cluster
        int ks = 1;
        while (ks < 8 && ks * 2 <= total_its && (long long)rowblocks * ks * mchunks < 2048) ks *= 2;
        // and at most 8 iterations per CTA where possible, bounding the staged A slice
        while (ks < 8 && (total_its + ks - 1) / ks > 8) ks *= 2;
        // warps per CTA: the largest power of two that still gives >= 2 CTAs per SM
        int W = 8;
        while (W > 1 && (long long)((rowblocks + W - 1) / W) * ks * mchunks < 2LL * sms) W >>= 1;
        if (const char* e = getenv("WQ_GEMV_KSPLIT")) {
            const int v = atoi(e);
            if (v == 1 || v == 2 || v == 4 || v == 8) ks = v;
        }
        if (const char* e = getenv("WQ_GEMV_WARPS")) {
            const int v = atoi(e);
            if (v == 1 || v == 2 || v == 4 || v == 8) W = v;
        }
        const int its_per_cta = total_its ? (total_its + ks - 1) / ks : 0;
        const int U = its_per_cta * (kItK / 8);
        smem = (size_t)MP * U * 16 + (size_t)W * 16 * MP * sizeof(float);
        if (smem > 200 * 1024) return WQ_ERR_UNSUPPORTED;
        if ((long long)(rowblocks + W - 1) / W > 65535 || mchunks > 65535) return WQ_ERR_UNSUPPORTED;
        args.its_per_cta = its_per_cta;
        args.row_blocks = W;
        args.wk_log2 = 0;
        grid = dim3(ks, (rowblocks + W - 1) / W, mchunks);
        threads = W * 32;
        cluster_x = ks;
    }

#define WQ_GEMV_DISPATCH(F, MODE)                                                                          \
    return NT == 1 ? launch_inst<F, 1, MODE>(args, grid, threads, smem, cluster_x, split_kernel, pdl, stream) \
                   : launch_inst<F, 2, MODE>(args, grid, threads, smem, cluster_x, split_kernel, pdl, stream)
    if (fmt == kNVFP4) WQ_GEMV_DISPATCH(kNVFP4, kModeScaled);
    if (fmt == kMXFP4) WQ_GEMV_DISPATCH(kMXFP4, kModeScaled);
    if (int4_g128) WQ_GEMV_DISPATCH(kINT4, kModeInt4);
    WQ_GEMV_DISPATCH(kINT4, kModeScaled);
#undef WQ_GEMV_DISPATCH
}

}  // namespace wq
