// wq_gemv_tma.cu -- the small-M path's streaming kernel: every packed weight
// byte a warp needs is requested by bulk copy (cp.async.bulk) the moment the
// warp starts, and the warps run the register decode + mma.sync work of
// wq_gemv.cuh out of shared memory.
//
// Why this shape (the KBench megakernel_int4_weight_decode.py spec, "Why
// this is hard": at batch 1 the GEMV is pure weight bandwidth, and the decode
// has to sit between the load and the FMA): a kernel that holds only a few
// iterations of weights in registers per warp waits out several DRAM round
// trips per warp.  Here each warp's whole weight slice (16 rows x its K
// range) is in flight at once, issued before anything else -- and, under
// programmatic dependent launch, before the preceding kernel on the stream
// has finished -- and no warp waits for another before its first MMA.
//
// CTA = rb blocks of 16 weight rows x all of K.  Each block's K is split over
// Wk warps (warp = block * Wk + kw), each owning a contiguous run of 128-k
// iterations.  Per warp, at start:
//   1. its scale / zero-point loads (global -> registers),
//   2. one mbarrier and 16 bulk copies: row i of the block, the warp's byte
//      range of K, into a shared row of stride S = 64 (mod 128) bytes, so the
//      two rows a quarter-warp reads sit in opposite halves of the banks,
//   3. its decode records (shared memory, warp-private),
// then, after the preceding kernel's writes are visible, the rb warps that
// share a K range stage those activations once (named barrier), and each
// warp waits for its own copies only.  Partial sums meet in shared memory and
// are added in a fixed order (deterministic, no atomics, no workspace).
//
// Shared memory (from a 128-byte aligned base):
//   bars [warps] mbarrier             one per warp, used once
//   W    [rows][S]                    packed rows as stored (low nibble = even k)
//   A    [Mc][n_its * 16][16 B]       activations, swizzled units (a_unit), in
//                                     the (k, k+4) pair order for int4 g128
//   rec8 [warps][16][R] uint2         per row and iteration (int4 g128:
//                                     {fp32 scale, bf16x2 (128 + zero)}) or
//                                     per row and 32-k chunk (other modes: the
//                                     decode multipliers of the chunk's groups)
//   rec4 [warps][16][R] u32           int4 only: second zero-point subtrahend
//   red  [Wk][MP][rows + 4] f32       partial sums (aliases W, A and the
//                                     records once every warp is done)
#include <cuda.h>
#include <cstdio>
#include <cstdlib>
#include <map>
#include <mutex>
#include <tuple>

#include "wq_gemv.cuh"
#include "wq_internal.h"
#include "wq_tc.cuh"

namespace wq {

__device__ int g_gemv_status = 0;

int read_and_clear_gemv_status() {
    int v = 0;
    const int zero = 0;
    if (cudaDeviceSynchronize() != cudaSuccess) return WQ_ERR_CUDA;
    if (cudaMemcpyFromSymbol(&v, g_gemv_status, sizeof(int)) != cudaSuccess) return WQ_ERR_CUDA;
    if (cudaMemcpyToSymbol(g_gemv_status, &zero, sizeof(int)) != cudaSuccess) return WQ_ERR_CUDA;
    return v;
}

namespace {

using namespace gemv;
using namespace sm100;

constexpr int kMaxIpw = 16;                             // iterations per warp
constexpr int kMaxWkLog2 = 3;                           // warps per K split <= 8 (named barriers 1..8)
constexpr unsigned long long kWaitNs = 2000000000ull;   // 2 s: far above any legal wait

struct TmaGemvArgs {
    const uint8_t* packed;
    const uint16_t* A;
    const void* scales;
    const uint8_t* zeros;
    void* C;
    int M, N, K, group;
    int out_f32;
    int n_its;          // ceil(K / 128)
    int rb;             // 16-row blocks per CTA
    int wk_log2;        // log2 of the warps splitting one block's K
    int ipw;            // iterations per warp
    int R;              // decode records per row and warp
    uint32_t S;         // shared row stride of the packed weights (bytes)
    uint32_t SA;        // shared row stride of the activations (bytes)
    uint32_t w_off, a_off, r8_off, r4_off, bar_off, red_off;
    int inputs_ready;   // A may be read before the preceding kernel completes
    int vec_store;      // plain output in 16-byte pieces: C 16-byte aligned, N a multiple of 8 (bf16) or 4 (fp32)
    Epilogue epi;
};

__device__ __forceinline__ void record_gemv_timeout() { atomicExch(&g_gemv_status, WQ_ERR_DEVICE_TIMEOUT); }

// Decode records of weight row n (n < N), record q of the scaled modes
// (q = 32-k chunk).  Returns true when the record needs the second exact step.
//   nvfp4: {mul of group 2q, mul of group 2q + 1}
//   mxfp4: {mul, mul2}
//   int4 other groups: {mul, zz}, zz2
// Chunks past K get all-zero records (zero multipliers; their weights and
// activations are zero as well).
template <int FMT>
__device__ __forceinline__ bool scaled_record(const TmaGemvArgs& a, int n, int q, uint2& r8, uint32_t& r4) {
    r8 = make_uint2(0, 0);
    r4 = 0;
    if (q * 32 >= a.K) return false;
    if constexpr (FMT == kNVFP4) {
        const uint8_t* p = static_cast<const uint8_t*>(a.scales) + (size_t)n * (a.K >> 4) + 2 * q;
        r8 = make_uint2(splat16(nvfp4_mul_bits(ldg_u8(p))), splat16(nvfp4_mul_bits(ldg_u8(p + 1))));
        return false;
    } else if constexpr (FMT == kMXFP4) {
        const GroupKey k = key_mxfp4(ldg_u8(static_cast<const uint8_t*>(a.scales) + (size_t)n * (a.K >> 5) + q));
        r8 = make_uint2(k.mul, k.mul2);
        return k.two;
    } else {
        const size_t gi = (size_t)n * (a.K / a.group) + (q * 32) / a.group;
        const GroupKey k = key_int4(ldg_u16(static_cast<const uint16_t*>(a.scales) + gi), ldg_u8(a.zeros + gi));
        r8 = make_uint2(k.mul, k.zz);
        r4 = k.zz2;
        return k.two;
    }
}

template <int FMT>
__device__ __forceinline__ void keys_from_record(uint2 r8, uint32_t r4, GroupKey (&k)[2]) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        k[h].mul2 = 0x3F803F80u;
        k[h].zz = 0;
        k[h].zz2 = 0;
        k[h].two = false;
    }
    if constexpr (FMT == kNVFP4) {
        k[0].mul = r8.x;
        k[1].mul = r8.y;
    } else if constexpr (FMT == kMXFP4) {
        k[0].mul = k[1].mul = r8.x;
        k[0].mul2 = k[1].mul2 = r8.y;
    } else {
        k[0].mul = k[1].mul = r8.x;
        k[0].zz = k[1].zz = r8.y;
        k[0].zz2 = k[1].zz2 = r4;
    }
}

// Staged activation position of 16-byte unit u: inside each iteration's 16
// units, unit 4c + j (lane chunk c, word j) sits at c + 4j, so a lane's four
// reads are its base + 64 j and the 8 lanes of a quarter-warp hit 4 bank
// groups x 2 row parities.
__device__ __forceinline__ int a_pos(int u) { return (u & ~15) | ((u >> 2) & 3) | ((u & 3) << 2); }

// One iteration of the scaled modes: weights decoded with their scale (bf16
// RNE of the exact weight) in natural pair order, accumulated directly.
template <int FMT, int NT, bool TWO>
__device__ __forceinline__ void it_scaled(const uint4& qa, const uint4& qb, const GroupKey (&ka)[2],
                                          const GroupKey (&kb)[2], const uint32_t (&ap)[NT], float (&acc)[NT][4]) {
    const uint32_t wa[4] = {qa.x, qa.y, qa.z, qa.w};
    const uint32_t wb[4] = {qb.x, qb.y, qb.z, qb.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint32_t pa[4], pb[4];
        word_scaled<FMT, TWO>(wa[j], ka[j >> 1], pa);
        word_scaled<FMT, TWO>(wb[j], kb[j >> 1], pb);
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            const uint4 bv = lds128(ap[t] + 64 * j);
            mma16816(acc[t], pa[0], pb[0], pa[1], pb[1], bv.x, bv.y);
            mma16816(acc[t], pa[2], pb[2], pa[3], pb[3], bv.z, bv.w);
        }
    }
}

// The compute loop of one warp over its nit iterations, all addresses bumped:
//   wp : the lane's 16 packed bytes of row r (row r + 8 is S8 on), +64 / iteration
//   rp : the lane's record pair {row r, row r + 8}, +16 (int4 g128) or +64
//        (scaled modes, chunk c of 4) per iteration; rq likewise for the
//        second zero-point subtrahends
//   ap : the lane's activation address per tile, +256 / iteration
template <int FMT, int NT, int MODE, bool TWO>
__device__ __forceinline__ void warp_loop(uint32_t wp, uint32_t S8, uint32_t rp, uint32_t rq, uint32_t (&ap)[NT],
                                          int nit, float (&acc)[NT][4]) {
    // int4 g128: a record pair {row r, row r + 8} is 2 x 4 bytes per iteration
    // (bf16 scale | bf16 (128 + zero) << 16) and the raw zero points 2 x 1
    // byte; scaled modes: 2 x 8 bytes and 2 x 4 bytes per 32-k chunk
    constexpr uint32_t kRecStep = MODE == kModeInt4 ? 8 : 64;
    constexpr uint32_t kRqStep = MODE == kModeInt4 ? 2 : 32;
#pragma unroll 2
    for (int i = 0; i < nit; ++i) {
        const uint4 qa = lds128(wp);
        const uint4 qb = lds128(wp + S8);
        if constexpr (MODE == kModeInt4) {
            const uint2 rr = lds64(rp);   // {row r, row r + 8}
            uint32_t zzA = prmt(rr.x, rr.x, 0x3232u), zzB = prmt(rr.y, rr.y, 0x3232u), zA2 = 0, zB2 = 0;
            if constexpr (TWO) {
                const uint32_t zb = lds16(rq);
                zero_subtrahends(zb & 0xFFu, zzA, zA2);
                zero_subtrahends(zb >> 8, zzB, zB2);
            }
            it_int4<NT, TWO>(qa, qb, ap, acc, zzA, zA2, zzB, zB2, __uint_as_float(rr.x << 16),
                             __uint_as_float(rr.y << 16));
        } else {
            const uint4 rr = lds128(rp);   // {row r: x, y; row r + 8: z, w}
            uint32_t zA2 = 0, zB2 = 0;
            if constexpr (TWO && FMT == kINT4) {
                const uint2 q2 = lds64(rq);
                zA2 = q2.x;
                zB2 = q2.y;
            }
            GroupKey ka[2], kb[2];
            keys_from_record<FMT>(make_uint2(rr.x, rr.y), zA2, ka);
            keys_from_record<FMT>(make_uint2(rr.z, rr.w), zB2, kb);
            it_scaled<FMT, NT, TWO>(qa, qb, ka, kb, ap, acc);
        }
        wp += 64;
        rp += kRecStep;
        rq += kRqStep;
#pragma unroll
        for (int t = 0; t < NT; ++t) ap[t] += 256;
    }
}

// One tile of activations (M <= 8) keeps to 64 registers, so that two
// launches' CTAs fit on an SM; two tiles (M <= 16) hold 96 KB of activations
// per CTA and never share an SM, so they take the registers to have all 16
// rows of their activation loads in flight at once.
// store_pieces as a call of its own: inlined, its registers pushed the
// one-tile int4 instance (two 512-thread CTAs per SM, 64 registers) into
// spilling
template <int MP>
__device__ __noinline__ void store_pieces_apart(const float* red, int ld, int Wk, int Mc, int outs_log2, int n0,
                                                int n_end, int mz, int N, void* C, bool out_f32, int tid,
                                                int nthreads) {
    store_pieces<MP>(red, ld, Wk, Mc, outs_log2, n0, n_end, mz, N, C, out_f32, tid, nthreads);
}

template <int FMT, int NT, int MODE, bool EPI>
__global__ void __launch_bounds__(512, NT == 1 ? 2 : 1) gemv_stream_kernel(const TmaGemvArgs a) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t sbase = (smem_u32(smem_raw) + 127u) & ~127u;
    uint8_t* sgen = smem_raw + (sbase - smem_u32(smem_raw));
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int r = lane >> 2, c = lane & 3;
    const int rows = a.rb * 16;
    const int n0 = blockIdx.x * rows;
    const int mz = blockIdx.y * 16;
    const int Mc = min(16, a.M - mz);
    const int Wk = 1 << a.wk_log2;
    const int blk = warp >> a.wk_log2, kw = warp & (Wk - 1);
    const int it0 = kw * a.ipw;
    const int nit = max(0, min(a.n_its, it0 + a.ipw) - it0);
    const int nb = n0 + blk * 16;   // first weight row of this warp's block
    const uint32_t bar = sbase + a.bar_off + 8 * warp;
    const int rr = lane & 15, rh = lane >> 4;   // record loads: row rr, every other record
    const int nrow = min(nb + rr, a.N - 1);
    // records of row rr live at pair (rr & 7), half (rr >> 3): [8][R][2]
    constexpr uint32_t kR8 = MODE == kModeInt4 ? 4 : 8, kR4 = MODE == kModeInt4 ? 1 : 4;   // record bytes
    const uint32_t rec8_w = a.r8_off + (uint32_t)warp * 16 * a.R * kR8;
    const uint32_t rec4_w = a.r4_off + (uint32_t)warp * 16 * a.R * kR4;
    const uint32_t rec_row = (uint32_t)(rr & 7) * a.R * 2 + (rr >> 3);

    // ---- 1. scale / zero-point loads of the int4 g128 records -------------
    uint32_t raw[kMaxIpw / 2];
    if constexpr (MODE == kModeInt4) {
        const size_t g0 = (size_t)nrow * (a.K >> 7) + it0;
        const uint16_t* sp = static_cast<const uint16_t*>(a.scales) + g0;
        const uint8_t* zp = a.zeros + g0;
#pragma unroll
        for (int t = 0; t < kMaxIpw / 2; ++t) {
            const int j = rh + 2 * t;
            raw[t] = 0;
            if (j < nit) raw[t] = ldg_u16(sp + j) | (ldg_u8(zp + j) << 16);
        }
    }

    // ---- 2. this warp's weight slice: 16 rows x its K range, one barrier
    // (issued after the scale loads: measured faster for chained calls of one
    // shape than the other order, whose barrier fences then wait on nothing
    // but whose scale loads queue behind the weight stream) --
    const int kb0 = it0 * 64;                                         // first packed byte of the range
    const int seg = max(0, min((it0 + nit) * 64, a.K >> 1) - kb0);    // bytes per row
    const int vrows = max(0, min(16, a.N - nb));
    if (lane == 0) {
        mbar_init(bar, 1);
        fence_mbarrier_init();
        fence_proxy_async_smem();
    }
    __syncwarp();
    if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)(seg * vrows));
    __syncwarp();
    if (lane < vrows && seg > 0)
        bulk_copy_g2s(sbase + a.w_off + (uint32_t)(blk * 16 + lane) * a.S + kb0,
                      a.packed + (size_t)(nb + lane) * (a.K >> 1) + kb0, (uint32_t)seg, bar);

    // ---- 3. decode records (warp-private) ----------------------------------
    bool two = false;
    if constexpr (MODE == kModeInt4) {
#pragma unroll
        for (int t = 0; t < kMaxIpw / 2; ++t) {
            const int j = rh + 2 * t;
            if (j < nit) {
                const uint32_t z = raw[t] >> 16;
                const uint32_t idx = rec_row + 2 * j;
                *reinterpret_cast<uint32_t*>(sgen + rec8_w + idx * 4) = (raw[t] & 0xFFFFu) | ((0x4300u + min(z, 128u)) << 16);
                sgen[rec4_w + idx] = (uint8_t)z;
                two |= z > 128;
            }
        }
    } else {
        const int nq = 4 * nit;
#pragma unroll 4
        for (int q = rh; q < nq; q += 2) {
            uint2 r8;
            uint32_t r4;
            two |= scaled_record<FMT>(a, nrow, 4 * it0 + q, r8, r4);
            const uint32_t idx = rec_row + 2 * q;
            *reinterpret_cast<uint2*>(sgen + rec8_w + idx * 8) = r8;
            if constexpr (FMT == kINT4) *reinterpret_cast<uint32_t*>(sgen + rec4_w + idx * 4) = r4;
        }
    }
    two = __any_sync(0xffffffffu, two);

    // the next kernel on the stream may start (programmatic dependent launch:
    // triggered once this CTA's own weight requests are out, so the next
    // call's stream follows this one's instead of competing with it); A is
    // read, and C written, only after the preceding kernel has finished --
    // A before it when the caller declared A complete already (inputs_ready)
    grid_dependents_launch();
    if (!a.inputs_ready) grid_dependency_wait();

    // ---- 4. activations of this K range, staged once by the rb warps that
    // share it (rows SA bytes apart, SA = 64 mod 128; units at a_pos) -------
    {
        const int gt = blk * 32 + lane, gsz = a.rb * 32;
        const int u0 = it0 * (kItK / 8), nu = nit * (kItK / 8);
        const int ulim = a.K >> 3;
        uint8_t* a_s = sgen + a.a_off;
        for (int e = gt; e < nu; e += gsz) {
            const int u = u0 + e;
            const uint32_t pos = (uint32_t)a_pos(u) * 16;
            constexpr int MB = NT * 8;   // activation rows in flight per thread
            for (int m0 = 0; m0 < Mc; m0 += MB) {
                uint4 v[MB];
#pragma unroll
                for (int q = 0; q < MB; ++q) {
                    v[q] = make_uint4(0, 0, 0, 0);
                    if (m0 + q < Mc && u < ulim)
                        v[q] = *reinterpret_cast<const uint4*>(a.A + (size_t)(mz + m0 + q) * a.K + u * 8);
                }
#pragma unroll
                for (int q = 0; q < MB; ++q) {
                    if (m0 + q < Mc) {
                        uint4 w = v[q];
                        if constexpr (MODE == kModeInt4) {
                            w = make_uint4(prmt(w.x, w.z, 0x5410u), prmt(w.x, w.z, 0x7632u),
                                           prmt(w.y, w.w, 0x5410u), prmt(w.y, w.w, 0x7632u));
                        }
                        *reinterpret_cast<uint4*>(a_s + (size_t)(m0 + q) * a.SA + pos) = w;
                    }
                }
            }
        }
        if (a.rb > 1) named_barrier(1 + kw, gsz);
        else __syncwarp();
    }

    // ---- 5. wait for this warp's copies, then its iterations --------------
    constexpr int MP = NT * 8;
    float acc[NT][4];
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[t][e] = 0.f;
    const bool ok = mbar_wait_timeout(bar, 0, kWaitNs);
    if (ok && nit > 0) {
        // activation rows past Mc are not staged: those lanes read row 0 or 1
        // (same row parity as a staged neighbour would break the bank split)
        uint32_t ap[NT];
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            const int m = t * 8 + r;
            const int ms = m < Mc ? m : (Mc > 1 ? (m & 1) : 0);
            ap[t] = sbase + a.a_off + (uint32_t)ms * a.SA + (uint32_t)(it0 * 256 + c * 16);
        }
        uint32_t wp = sbase + a.w_off + (uint32_t)(blk * 16 + r) * a.S + (uint32_t)(kb0 + c * 16);
        uint32_t rp = sbase + rec8_w + ((uint32_t)(r * a.R * 2) + 2u * (MODE == kModeInt4 ? 0u : (uint32_t)c)) * kR8;
        uint32_t rq = sbase + rec4_w + ((uint32_t)(r * a.R * 2) + 2u * (MODE == kModeInt4 ? 0u : (uint32_t)c)) * kR4;
        // the shared loads below must not move above the barrier wait
        asm volatile("" : "+r"(wp), "+r"(rp), "+r"(rq)::"memory");
#pragma unroll
        for (int t = 0; t < NT; ++t) asm volatile("" : "+r"(ap[t])::"memory");
        if (two)
            warp_loop<FMT, NT, MODE, true>(wp, 8 * a.S, rp, rq, ap, nit, acc);
        else
            warp_loop<FMT, NT, MODE, false>(wp, 8 * a.S, rp, rq, ap, nit, acc);
    }
    if (!ok && lane == 0) record_gemv_timeout();
    if (a.inputs_ready) grid_dependency_wait();   // completion order: stores after the predecessor's
    if (__syncthreads_or(!ok)) return;   // a copy never landed: store nothing

    // ---- 6. partial sums -> shared memory, fixed-order reduction, store ----
    // red[kw][m][row], row stride rows + 4: conflict-free on both sides
    const int ld = rows + 4;
    float* red = reinterpret_cast<float*>(sgen + a.red_off);
    {
        const int y = blk * 16 + r;
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            const int m = t * 8 + 2 * c;
            float* p = red + ((size_t)kw * MP + m) * ld + y;
            p[0] = acc[t][0];
            p[ld] = acc[t][1];
            p[8] = acc[t][2];
            p[ld + 8] = acc[t][3];
        }
    }
    __syncthreads();
    // (m, output) pairs over all threads; consecutive threads take
    // consecutive rows (coalesced stores, conflict-free reads).  Gated: an
    // output reads its gate row 16b + j and its up row 16b + 8 + j.  The
    // plain instance (EPI false) carries no epilogue code at all.
    const bool gated = EPI && a.epi.gated;
    const int outs = gated ? rows >> 1 : rows;   // a power of two
    const int outs_log2 = 31 - __clz(outs);
    if constexpr (!EPI) {
        if (a.vec_store) {
            store_pieces_apart<MP>(red, ld, Wk, Mc, outs_log2, n0, a.N, mz, a.N, a.C, a.out_f32, tid, blockDim.x);
            return;
        }
    }
    for (int i = tid; i < Mc * outs; i += blockDim.x) {
        const int m = i >> outs_log2, o = i & (outs - 1);
        const int rl = gated ? (((o >> 3) << 4) | (o & 7)) : o;
        const int n = n0 + rl;
        if (n >= a.N) continue;
        const float* src = red + (size_t)m * ld + rl;
        float v = 0.f;
        for (int q = 0; q < Wk; ++q) v += src[(size_t)q * MP * ld];
        if constexpr (EPI) {
            float u = 0.f;
            if (gated)
                for (int q = 0; q < Wk; ++q) u += src[(size_t)q * MP * ld + 8];
            store_epilogue(a.epi, a.C, a.out_f32, a.N, mz + m, n, v, u);
        } else {
            const size_t o2 = (size_t)(mz + m) * a.N + n;
            if (a.out_f32) static_cast<float*>(a.C)[o2] = v;
            else static_cast<__nv_bfloat16*>(a.C)[o2] = __float2bfloat16_rn(v);
        }
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
struct Plan {
    int rb = 0, wk_log2 = 0, threads = 0, ipw = 0, R = 0;
    size_t smem = 0;
    uint32_t S = 0, SA = 0, w_off = 0, a_off = 0, r8_off = 0, r4_off = 0, bar_off = 0, red_off = 0;
};

using KernFn = void (*)(TmaGemvArgs);

template <int FMT, int NT, int MODE>
KernFn kernel_for(bool epi) {
    return epi ? gemv_stream_kernel<FMT, NT, MODE, true> : gemv_stream_kernel<FMT, NT, MODE, false>;
}

KernFn select_kernel(int fmt, int NT, int mode, bool epi) {
    if (fmt == kNVFP4)
        return NT == 1 ? kernel_for<kNVFP4, 1, kModeScaled>(epi) : kernel_for<kNVFP4, 2, kModeScaled>(epi);
    if (fmt == kMXFP4)
        return NT == 1 ? kernel_for<kMXFP4, 1, kModeScaled>(epi) : kernel_for<kMXFP4, 2, kModeScaled>(epi);
    if (mode == kModeInt4)
        return NT == 1 ? kernel_for<kINT4, 1, kModeInt4>(epi) : kernel_for<kINT4, 2, kModeInt4>(epi);
    return NT == 1 ? kernel_for<kINT4, 1, kModeScaled>(epi) : kernel_for<kINT4, 2, kModeScaled>(epi);
}

constexpr size_t kMaxSmem = 227 * 1024;

// Shared-memory layout of one candidate (offsets from the aligned base).
Plan layout(int rb, int wk_log2, int Mc, int K, int n_its, int mode, int fmt, int MP, bool pad) {
    Plan p;
    p.rb = rb;
    p.wk_log2 = wk_log2;
    p.threads = (rb << wk_log2) * 32;
    p.ipw = (n_its + (1 << wk_log2) - 1) >> wk_log2;
    p.R = mode == kModeInt4 ? p.ipw : 4 * p.ipw;
    const size_t rows = (size_t)rb * 16, warps = (size_t)rb << wk_log2;
    // row stride = 64 (mod 128) bytes and at least K / 2 (conflict-free
    // quarter-warp reads), or K / 2 itself where shared memory is short
    p.S = pad ? (uint32_t)(((size_t)(K / 2) + 63) / 128 * 128 + 64) : (uint32_t)(K / 2);
    p.bar_off = 0;                   // warps * 8 <= 128 bytes
    p.w_off = 128;
    size_t off = p.w_off + rows * p.S;
    p.a_off = (uint32_t)off;
    p.SA = (uint32_t)n_its * 256 + 64;   // 64 (mod 128): row parities in opposite bank halves
    off += (size_t)Mc * p.SA;
    p.r8_off = (uint32_t)off;
    off += warps * 16 * p.R * (mode == kModeInt4 ? 4 : 8);
    p.r4_off = (uint32_t)off;
    if (fmt == kINT4) off += warps * 16 * p.R * (mode == kModeInt4 ? 1 : 4);
    off = (off + 15) & ~(size_t)15;
    p.red_off = 128;                 // aliases W, A and the records at the end
    const size_t red = ((size_t)1 << wk_log2) * MP * (rows + 4) * sizeof(float);
    if (p.red_off + red > off) off = p.red_off + red;
    p.smem = off + 128;              // base alignment slack
    return p;
}

int env_int(const char* name, int dflt) {
    const char* e = getenv(name);
    return e ? atoi(e) : dflt;
}

// Pick the CTA shape.  Cost, in SM issue cycles of the busiest SM: its block
// iterations x cycles per iteration / 4 schedulers, the activation bytes it
// stages, one warp's run (the tail after its slice lands) and a latency round
// per extra wave.
bool choose_plan(KernFn kern, int fmt, int mode, int NT, int Mc, int mchunks, int N, int K, int n_its, int sms,
                 bool pdl, Plan& best) {
    const int MP = NT * 8;
    const int force_rb = env_int("WQ_GEMV_RB", 0), force_wk = env_int("WQ_GEMV_TMA_WK", -1);
    const double c_it = NT == 1 ? 130.0 : 150.0;
    double best_cost = -1.0;
    for (int rb = 1; rb <= 8; rb *= 2) {
        if (force_rb && rb != force_rb) continue;
        for (int wk = 0; wk <= kMaxWkLog2; ++wk) {
            if (force_wk >= 0 && wk != force_wk) continue;
            if ((rb << wk) * 32 > 512) continue;
            if (force_wk < 0 && wk > 0 && (1 << wk) > n_its) continue;
            for (int pad = 1; pad >= 0; --pad) {
                const Plan p = layout(rb, wk, Mc, K, n_its, mode, fmt, MP, pad != 0);
                if (p.ipw > kMaxIpw || p.smem > kMaxSmem) continue;
                int occ = 0;
                if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, p.threads, p.smem) != cudaSuccess ||
                    occ < 1)
                    continue;
                const long long ctas = (long long)((N + rb * 16 - 1) / (rb * 16)) * mchunks;
                const long long per_sm = (ctas + sms - 1) / sms;
                const long long waves = (ctas + (long long)sms * occ - 1) / ((long long)sms * occ);
                double cost = per_sm * rb * n_its * c_it / 4.0 + per_sm * (double)Mc * n_its * kItK * 2 / 48.0 +
                              p.ipw * c_it + (waves - 1) * 2500.0 + (pad ? 0.0 : 300.0);
                // chained launches stream the next call's weights while this one
                // computes only if the next kernel's CTAs fit beside this
                // kernel's own: room for a second generation on every SM
                if (pdl && occ < 2 * per_sm) cost += 4000.0;
                if (best_cost < 0 || cost < best_cost) {
                    best_cost = cost;
                    best = p;
                }
            }
        }
    }
    return best_cost >= 0;
}

struct PlanKey {
    int dev, fmt, mode, NT, Mc, mchunks, N, K, pdl, epi;
    bool operator<(const PlanKey& o) const {
        return std::tie(dev, fmt, mode, NT, Mc, mchunks, N, K, pdl, epi) <
               std::tie(o.dev, o.fmt, o.mode, o.NT, o.Mc, o.mchunks, o.N, o.K, o.pdl, o.epi);
    }
};

}  // namespace

// Returns WQ_ERR_UNSUPPORTED (without launching) when the shape does not fit
// this kernel: K = 0, K > 16384, or a CTA's activations + weights + records
// above the shared-memory limit.
int launch_gemv_tma(const void* A, const uint8_t* packed, const void* scales, const uint8_t* zeros, void* C,
                    int M, int N, int K, int fmt, int group, bool out_f32, bool pdl, bool inputs_ready,
                    const Epilogue& epi, cudaStream_t stream) {
    if (inputs_ready) pdl = true;
    if (M == 0 || N == 0) return WQ_OK;
    if (K <= 0 || K > kMaxIpw * (1 << kMaxWkLog2) * kItK) return WQ_ERR_UNSUPPORTED;
    const int n_its = (K + kItK - 1) / kItK;
    const int Mc = M < 16 ? M : 16;
    const int mchunks = (M + 15) / 16;
    const int NT = Mc <= 8 ? 1 : 2;
    const int mode = (fmt == kINT4 && group == kItK) ? kModeInt4 : kModeScaled;
    if (mchunks > 65535) return WQ_ERR_UNSUPPORTED;

    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const bool has_epi = epi.bias || epi.residual || epi.gated;
    KernFn kern = select_kernel(fmt, NT, mode, has_epi);

    Plan plan;
    {
        static std::mutex mu;
        static std::map<PlanKey, Plan> cache;
        static std::map<std::pair<int, KernFn>, bool> attr_set;
        const bool overridden = getenv("WQ_GEMV_RB") || getenv("WQ_GEMV_TMA_WK");
        const PlanKey key{dev, fmt, mode, NT, Mc, mchunks, N, K, pdl ? 1 : 0, has_epi ? 1 : 0};
        std::lock_guard<std::mutex> lock(mu);
        if (!attr_set[{dev, kern}]) {
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kMaxSmem) !=
                cudaSuccess)
                return WQ_ERR_CUDA;
            attr_set[{dev, kern}] = true;
        }
        auto it = overridden ? cache.end() : cache.find(key);
        if (it != cache.end()) {
            plan = it->second;
        } else {
            if (!choose_plan(kern, fmt, mode, NT, Mc, mchunks, N, K, n_its, sms, pdl, plan)) {
                if (debug_on()) fprintf(stderr, "wq: streaming GEMV: no CTA shape fits M=%d N=%d K=%d\n", M, N, K);
                return WQ_ERR_UNSUPPORTED;
            }
            if (!overridden) cache[key] = plan;
        }
    }
    if (debug_on())
        fprintf(stderr, "wq: streaming GEMV M=%d N=%d K=%d: rb=%d wk=%d threads=%d smem=%zu S=%u\n", M, N, K,
                plan.rb, 1 << plan.wk_log2, plan.threads, plan.smem, plan.S);

    const int rows = plan.rb * 16;
    TmaGemvArgs args;
    args.packed = packed;
    args.A = static_cast<const uint16_t*>(A);
    args.scales = scales;
    args.zeros = zeros;
    args.C = C;
    args.M = M;
    args.N = N;
    args.K = K;
    args.group = group;
    args.out_f32 = out_f32 ? 1 : 0;
    args.n_its = n_its;
    args.rb = plan.rb;
    args.wk_log2 = plan.wk_log2;
    args.ipw = plan.ipw;
    args.R = plan.R;
    args.S = plan.S;
    args.SA = plan.SA;
    args.w_off = plan.w_off;
    args.a_off = plan.a_off;
    args.r8_off = plan.r8_off;
    args.r4_off = plan.r4_off;
    args.bar_off = plan.bar_off;
    args.red_off = plan.red_off;
    args.inputs_ready = inputs_ready ? 1 : 0;
    args.vec_store = (reinterpret_cast<uintptr_t>(C) & 15) == 0 && N % (out_f32 ? 4 : 8) == 0 && !getenv("WQ_GEMV_SCALAR_STORE");
    args.epi = epi;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((N + rows - 1) / rows, mchunks, 1);
    cfg.blockDim = dim3(plan.threads, 1, 1);
    cfg.dynamicSmemBytes = plan.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if (pdl) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
    }
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    if (cudaLaunchKernelEx(&cfg, kern, args) != cudaSuccess) return WQ_ERR_CUDA;
    return WQ_OK;
}

}  // namespace wq
