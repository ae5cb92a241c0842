// wq_gemv_staged.cu -- the small-M kernel for prepacked weights whose call
// depends on the kernel before it (a plain launch, or WQ_LAUNCH_OVERLAP
// without WQ_LAUNCH_INPUTS_READY); calls that declare their inputs ready run
// the ring kernel of wq_gemv_pre.cu instead.
//
// A dependent call cannot start its product before its predecessor has
// finished, so this kernel stages ALL of a CTA's weights while that one runs
// and then needs many warps to run the product fast once the wait is over:
// a CTA takes rb blocks of 16 weight rows x all of K, each block's K split
// over Wk warps; the weights are the M operand of mma.sync.m16n8k16 and the
// activations its N = 8 operand; int4 g128 runs the MMAs on the exact
// integers (code - zero) and scales the fp32 partial sums per iteration.
//   - per warp, its codes are ONE bulk copy (nit contiguous 1024-byte
//     blocks) and, for int4, its records a second one (nit x 48 bytes of
//     scales and zero points);
//   - the activations need no permutation (a lane's four words of a block
//     are the natural k units c + 4j), so after the dependency wait the first
//     warp of each K range copies them with one bulk copy per row and the
//     other warps of the range wait on that copy's mbarrier.
//
// Shared memory (from a 128-byte aligned base):
//   bars  [warps] u64 at 0, [Wk] u64 at 128   codes / activations landed
//   W     [warps][ipw][1024]                  the warps' code blocks
//   A     [Mc][SA]                            activation rows, natural order
//   R     [warps][ipw][48]  int4              the copied record blocks
//         [warps][ipw][512] fp4               decoded multipliers, per lane
//   red   [Wk][MP][rows + 4] f32 at 256       partial sums (aliases W, A, R)
#include <cstdio>
#include <cstdlib>
#include <map>
#include <mutex>
#include <tuple>

#include "wq_gemv.cuh"
#include "wq_internal.h"
#include "wq_tc.cuh"

namespace wq {

__device__ int g_staged_status = 0;

int read_and_clear_staged_status() {
    int v = 0;
    const int zero = 0;
    if (cudaDeviceSynchronize() != cudaSuccess) return WQ_ERR_CUDA;
    if (cudaMemcpyFromSymbol(&v, g_staged_status, sizeof(int)) != cudaSuccess) return WQ_ERR_CUDA;
    if (cudaMemcpyToSymbol(g_staged_status, &zero, sizeof(int)) != cudaSuccess) return WQ_ERR_CUDA;
    return v;
}

namespace {

using namespace gemv;
using namespace sm100;

constexpr int kMaxIpw = 16;                             // 128-k blocks per warp
constexpr int kMaxWkLog2 = 3;                           // warps per K split <= 8
constexpr unsigned long long kWaitNs = 2000000000ull;   // 2 s: far above any legal wait
constexpr uint32_t kBarBytes = 256;

struct PreArgs {
    const uint8_t* codes;   // code blocks
    const uint8_t* recs;    // record blocks
    const uint16_t* A;
    void* C;
    int M, N, K;
    int I, Nb;              // 128-k blocks per row, 16-row blocks
    int out_f32;
    int mrows;              // activation rows per CTA (16, 8, 4, 2 or 1)
    int rb, wk_log2, ipw;
    uint32_t SA;            // shared row stride of the activations (bytes)
    uint32_t w_off, a_off, r_off, red_off;
    int inputs_ready;       // A may be read before the preceding kernel completes
    int vec_store;          // plain output in 16-byte pieces: C 16-byte aligned, N a multiple of 8 (bf16) or 4 (fp32)
    Epilogue epi;
};

__device__ __forceinline__ void record_pre_timeout() { atomicExch(&g_staged_status, WQ_ERR_DEVICE_TIMEOUT); }

__device__ __forceinline__ uint32_t lds32(uint32_t saddr) {
    uint32_t v;
    asm("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(saddr));
    return v;
}

__device__ __forceinline__ void sts128_zero(uint32_t saddr) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(saddr), "r"(0) : "memory");
}

// The lane's four words of one 128-k block, rows r (qa) and r + 8 (qb), in
// the order of the k units c, c + 4, c + 8, c + 12.  wp: the lane's 8 bytes
// of half 0, row r (row r + 8 is 256 bytes on, half 1 is 512 bytes on).
__device__ __forceinline__ void block_words(uint32_t wp, uint4& qa, uint4& qb) {
    const uint2 a0 = lds64(wp), b0 = lds64(wp + 256), a1 = lds64(wp + 512), b1 = lds64(wp + 768);
    qa = make_uint4(a0.x, a0.y, a1.x, a1.y);
    qb = make_uint4(b0.x, b0.y, b1.x, b1.y);
}

// int4 g128 loop.  rp: the lane's scale pair {row r, row r + 8} (bf16 each);
// rq: its zero-point pair (a byte each).  TWO: some zero point exceeds 128,
// so each is subtracted in two exact steps.
template <int NT, bool TWO>
__device__ __forceinline__ void loop_int4(uint32_t wp, uint32_t rp, uint32_t rq, uint32_t (&ap)[NT], int nit,
                                          float (&acc)[NT][4]) {
    // the rare second-subtrahend instance runs unrolled once (register cap)
#pragma unroll(TWO ? 1 : 2)
    for (int i = 0; i < nit; ++i) {
        uint4 qa, qb;
        block_words(wp, qa, qb);
        const uint32_t sp = lds32(rp), zp = lds16(rq);
        uint32_t zA, zB, zA2 = 0, zB2 = 0;
        if constexpr (TWO) {
            zsub_two(zp & 0xFFu, zA, zA2);
            zsub_two(zp >> 8, zB, zB2);
        } else {
            zA = zsub_lo(zp);
            zB = zsub_hi(zp);
        }
        it_int4<NT, TWO>(qa, qb, ap, acc, zA, zA2, zB, zB2, __uint_as_float(sp << 16),
                         __uint_as_float(sp & 0xFFFF0000u));
        wp += 1024;
        rp += 48;
        rq += 48;
#pragma unroll
        for (int t = 0; t < NT; ++t) ap[t] += 256;
    }
}

// fp4 loop.  rp: the lane's decoded multipliers, words j = 0..3 of row r
// (16 bytes) then of row r + 8; the second multipliers (MXFP4 scales above
// 2^15) 256 bytes on.
template <int NT, bool TWO>
__device__ __forceinline__ void loop_fp4(uint32_t wp, uint32_t rp, uint32_t (&ap)[NT], int nit, float (&acc)[NT][4]) {
#pragma unroll 2
    for (int i = 0; i < nit; ++i) {
        uint4 qa, qb;
        block_words(wp, qa, qb);
        const uint4 ma = lds128(rp), mb = lds128(rp + 16);
        uint4 na = make_uint4(0, 0, 0, 0), nb = na;
        if constexpr (TWO) {
            na = lds128(rp + 256);
            nb = lds128(rp + 272);
        }
        const uint32_t wa[4] = {qa.x, qa.y, qa.z, qa.w}, wb[4] = {qb.x, qb.y, qb.z, qb.w};
        const uint32_t mua[4] = {ma.x, ma.y, ma.z, ma.w}, mub[4] = {mb.x, mb.y, mb.z, mb.w};
        const uint32_t m2a[4] = {na.x, na.y, na.z, na.w}, m2b[4] = {nb.x, nb.y, nb.z, nb.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint32_t pa[4], pb[4];
            e2m1_word_raw(wa[j], pa);
            e2m1_word_raw(wb[j], pb);
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                pa[s] = bf16x2_mul(pa[s], mua[j]);
                pb[s] = bf16x2_mul(pb[s], mub[j]);
                if constexpr (TWO) {
                    pa[s] = bf16x2_mul(pa[s], m2a[j]);
                    pb[s] = bf16x2_mul(pb[s], m2b[j]);
                }
            }
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                const uint4 bv = lds128(ap[t] + 64 * j);
                mma16816(acc[t], pa[0], pb[0], pa[1], pb[1], bv.x, bv.y);
                mma16816(acc[t], pa[2], pb[2], pa[3], pb[3], bv.z, bv.w);
            }
        }
        wp += 1024;
        rp += 512;
#pragma unroll
        for (int t = 0; t < NT; ++t) ap[t] += 256;
    }
}

template <int FMT, int NT, bool EPI>
__global__ void __launch_bounds__(512, NT == 1 ? 2 : 1) gemv_staged_kernel(const PreArgs a) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t sbase = (smem_u32(smem_raw) + 127u) & ~127u;
    uint8_t* sgen = smem_raw + (sbase - smem_u32(smem_raw));
    constexpr bool kInt4 = FMT == kINT4;
    constexpr uint32_t kRec = kInt4 ? 48 : 512;   // shared record bytes per warp and block
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int r = lane >> 2, c = lane & 3;
    const int Wk = 1 << a.wk_log2;
    const int blk = warp >> a.wk_log2, kw = warp & (Wk - 1);
    const int rows = a.rb * 16;                                // rows of the widest CTA
    // this CTA's row blocks: an even share of the Nb blocks (counts differ
    // by at most one, never above rb)
    const int bs = (int)((long long)blockIdx.x * a.Nb / gridDim.x);
    const int be = (int)((long long)(blockIdx.x + 1) * a.Nb / gridDim.x);
    const int n0 = bs * 16, n_end = min(a.N, be * 16);
    const int b = bs + blk;                                    // this warp's row block
    const int mz = blockIdx.y * a.mrows;
    const int Mc = min(a.mrows, a.M - mz);
    const int it0 = kw * a.ipw;
    const int nrange = max(0, min(a.I, it0 + a.ipw) - it0);   // blocks of this K range
    const int nit = b < be ? nrange : 0;                      // ... this warp computes
    const uint32_t bar = sbase + 8 * warp, abar = sbase + 128 + 8 * kw;
    const uint32_t wslice = sbase + a.w_off + (uint32_t)(warp * a.ipw) * 1024u;
    const uint32_t rslice = sbase + a.r_off + (uint32_t)(warp * a.ipw) * kRec;
    const size_t blk0 = (size_t)b * a.I + it0;
    // int4: the prepacked weight's flag (a zero point above 128 anywhere)
    const uint32_t large_zero = kInt4 ? ldg_u32(a.recs + (size_t)a.Nb * a.I * 48) : 0u;

    if (tid == 0) {
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) mbar_init(sbase + 8 * w, 1);
        for (int q = 0; q < Wk; ++q) mbar_init(sbase + 128 + 8 * q, 1);
        fence_mbarrier_init();
    }
    __syncthreads();

    // ---- 1. this warp's code blocks (and int4 record blocks), one copy each
    if (lane == 0) {
        mbar_arrive_expect_tx(bar, (uint32_t)nit * (1024u + (kInt4 ? 48u : 0u)));
        if (nit > 0) {
            bulk_copy_g2s(wslice, a.codes + blk0 * 1024, (uint32_t)nit * 1024u, bar);
            if constexpr (kInt4) bulk_copy_g2s(rslice, a.recs + blk0 * 48, (uint32_t)nit * 48u, bar);
        }
    }

    // ---- 2. fp4: decode multipliers into the lane order of the loop; zero
    // the activation tail of a partial last block (its codes are 0, and
    // 0 x garbage could be NaN)
    bool two = false;
    if constexpr (!kInt4) {
        uint8_t* s8 = sgen + (rslice - sbase);
        if constexpr (FMT == kNVFP4) {
            // record block: row rho's 8 bytes at 8 rho; lane = (rho, half of
            // the groups); group g feeds word j = g >> 1 of the lanes with
            // (c >> 1) == (g & 1)
            const int rho = lane >> 1, g0 = 4 * (lane & 1);
            for (int t = 0; t < nit; ++t) {
                const uint32_t raw = ldg_u32(a.recs + (blk0 + t) * 128 + 4 * lane);
                const uint32_t f01 = e4m3x2_to_f16x2(raw & 0xFFFFu), f23 = e4m3x2_to_f16x2(raw >> 16);
                const uint32_t hv[4] = {f01 & 0xFFFFu, f01 >> 16, f23 & 0xFFFFu, f23 >> 16};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int g = g0 + q;
                    const uint32_t off = t * 512 + (((rho & 7) * 2 + (g & 1)) * 32) + (rho >> 3) * 16 + (g >> 1) * 4;
                    *reinterpret_cast<uint32_t*>(s8 + off) = splat16(nvfp4_mul_from_f16(hv[q]));
                }
            }
        } else {
            // record block: row rho's 4 bytes at 4 rho, group g = word j
            const int rho = lane & 15;
            for (int t = lane >> 4; t < nit; t += 2) {
                const uint32_t raw = ldg_u32(a.recs + (blk0 + t) * 64 + 4 * rho);
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    const GroupKey k = key_mxfp4((raw >> (8 * g)) & 0xFFu);
                    two |= k.two;
                    const uint32_t off = t * 512 + (rho & 7) * 32 + (rho >> 3) * 16 + g * 4;
                    *reinterpret_cast<uint32_t*>(s8 + off) = k.mul;
                    *reinterpret_cast<uint32_t*>(s8 + off + 256) = k.mul2;
                }
            }
        }
        if (nit > 0 && (it0 + nit) * 128 > a.K) {
            const int t0 = (a.K - it0 * 128) * 2, t1 = nit * 256;   // bytes of the range
            for (int m = 0; m < Mc; ++m)
                for (int o = t0 + 16 * lane; o < t1; o += 512)
                    sts128_zero(sbase + a.a_off + (uint32_t)m * a.SA + (uint32_t)it0 * 256 + o);
        }
        two = __any_sync(0xffffffffu, two);
    }

    // the next kernel on the stream may start.  C is written only after the
    // preceding kernel has finished; A is read after it too, unless the
    // caller declared it complete already (inputs_ready)
    grid_dependents_launch();
    if (!a.inputs_ready) grid_dependency_wait();

    // ---- 3. activations of this K range: the range's first warp copies them
    if (blk == 0) {
        const int kb = it0 * 128, ke = min(a.K, (it0 + nrange) * 128);
        const uint32_t bytes = ke > kb ? (uint32_t)(ke - kb) * 2u : 0u;
        if (lane == 0) mbar_arrive_expect_tx(abar, bytes * (uint32_t)Mc);
        __syncwarp();
        if (lane < Mc && bytes > 0)
            bulk_copy_g2s(sbase + a.a_off + (uint32_t)lane * a.SA + (uint32_t)it0 * 256,
                          a.A + (size_t)(mz + lane) * a.K + kb, bytes, abar);
    }

    // ---- 4. wait for this warp's codes and the range's activations --------
    constexpr int MP = NT * 8;
    float acc[NT][4];
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[t][e] = 0.f;
    bool ok = mbar_wait_timeout(bar, 0, kWaitNs);
    ok = mbar_wait_timeout(abar, 0, kWaitNs) && ok;
    if constexpr (kInt4) two = (large_zero & 0xFFu) != 0;   // some zero point above 128: two subtrahends
    if (ok && nit > 0) {
        // activation rows past Mc are not staged: those lanes read row 0 or 1
        // (keeping the row parity of a staged neighbour)
        uint32_t ap[NT];
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            const int m = t * 8 + r;
            const int ms = m < Mc ? m : (Mc > 1 ? (m & 1) : 0);
            ap[t] = sbase + a.a_off + (uint32_t)ms * a.SA + (uint32_t)(it0 * 256 + c * 16);
        }
        const uint32_t lane_w = 32u * r + 16u * ((c >> 1) ^ ((r >> 2) & 1)) + 8u * (c & 1);
        uint32_t wp = wslice + lane_w;
        // the shared loads below must not move above the barrier waits
        asm volatile("" : "+r"(wp)::"memory");
#pragma unroll
        for (int t = 0; t < NT; ++t) asm volatile("" : "+r"(ap[t])::"memory");
        if constexpr (kInt4) {
            const uint32_t rp = rslice + 4u * r, rq = rslice + 32u + 2u * r;
            if (two) loop_int4<NT, true>(wp, rp, rq, ap, nit, acc);
            else loop_int4<NT, false>(wp, rp, rq, ap, nit, acc);
        } else {
            const uint32_t rp = rslice + (FMT == kNVFP4 ? (2u * r + (c >> 1)) * 32u : 32u * r);
            if (two) loop_fp4<NT, true>(wp, rp, ap, nit, acc);
            else loop_fp4<NT, false>(wp, rp, ap, nit, acc);
        }
    }
    if (!ok && lane == 0) record_pre_timeout();
    if (a.inputs_ready) grid_dependency_wait();   // completion order: stores after the predecessor's
    if (__syncthreads_or(!ok)) return;   // a copy never landed: store nothing

    // ---- 5. partial sums -> shared memory, fixed-order reduction, store ----
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
    const bool gated = EPI && a.epi.gated;
    const int outs = gated ? rows >> 1 : rows;   // a power of two
    const int outs_log2 = 31 - __clz(outs);
    if constexpr (!EPI) {
        if (a.vec_store) {
            store_pieces<MP>(red, ld, Wk, Mc, outs_log2, n0, n_end, mz, a.N, a.C, a.out_f32, tid, blockDim.x);
            return;
        }
    }
    for (int i = tid; i < Mc * outs; i += blockDim.x) {
        const int m = i >> outs_log2, o = i & (outs - 1);
        const int rl = gated ? (((o >> 3) << 4) | (o & 7)) : o;
        const int n = n0 + rl;
        if (n >= n_end) continue;
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
    int rb = 0, wk_log2 = 0, threads = 0, ipw = 0;
    size_t smem = 0;
    uint32_t SA = 0, w_off = 0, a_off = 0, r_off = 0, red_off = 0;
};

using KernFn = void (*)(PreArgs);

template <int FMT, int NT>
KernFn kernel_for(bool epi) {
    return epi ? gemv_staged_kernel<FMT, NT, true> : gemv_staged_kernel<FMT, NT, false>;
}

KernFn select_kernel(int fmt, int NT, bool epi) {
    if (fmt == kNVFP4) return NT == 1 ? kernel_for<kNVFP4, 1>(epi) : kernel_for<kNVFP4, 2>(epi);
    if (fmt == kMXFP4) return NT == 1 ? kernel_for<kMXFP4, 1>(epi) : kernel_for<kMXFP4, 2>(epi);
    return NT == 1 ? kernel_for<kINT4, 1>(epi) : kernel_for<kINT4, 2>(epi);
}

constexpr size_t kMaxSmem = 227 * 1024;

Plan layout(int rb, int wk_log2, int Mc, int I, int fmt, int MP) {
    Plan p;
    p.rb = rb;
    p.wk_log2 = wk_log2;
    p.threads = (rb << wk_log2) * 32;
    p.ipw = (I + (1 << wk_log2) - 1) >> wk_log2;
    const size_t rows = (size_t)rb * 16, warps = (size_t)rb << wk_log2;
    p.w_off = kBarBytes;
    size_t off = p.w_off + warps * p.ipw * 1024;
    p.a_off = (uint32_t)off;
    p.SA = (uint32_t)I * 256 + 64;   // 64 (mod 128): row parities in opposite bank halves
    off += (size_t)Mc * p.SA;
    p.r_off = (uint32_t)off;
    // int4 records take 48 bytes per block; 96 are reserved, the footprint
    // of the format before (its plans and the overlap between calls that
    // the CTA size sets were measured with it)
    off += warps * p.ipw * (fmt == kINT4 ? 96 : 512);
    p.red_off = kBarBytes;           // aliases W, A and R once every warp is done
    const size_t red = ((size_t)1 << wk_log2) * MP * (rows + 4) * sizeof(float);
    if (p.red_off + red > off) off = p.red_off + red;
    p.smem = off + 128;              // base alignment slack
    return p;
}

int env_int(const char* name, int dflt) {
    const char* e = getenv(name);
    return e ? atoi(e) : dflt;
}

// The CTA shape and grid.  A CTA takes an even share of the row blocks
// (rb = the largest share) x all of K, split over Wk warps.  Cost, in SM
// issue cycles of the busiest SM: its block iterations / 4 schedulers, the
// activation bytes it receives, one warp's run and a latency round per extra
// wave.  Chained launches (pdl) stream the next call's weights while this
// one computes only if its CTAs fit beside this kernel's own; and a grid
// smaller than the SM count lets the next call put two CTAs on an SM this
// call left idle, which then runs twice the work -- so a grid of exactly one
// CTA per SM is preferred there.
bool choose_plan(KernFn kern, int fmt, int NT, int Mc, int mchunks, int Nb, int I, int sms, bool pdl, Plan& best,
                 int& grid) {
    const int MP = NT * 8;
    const int force_rb = env_int("WQ_GEMV_RB", 0), force_wk = env_int("WQ_GEMV_TMA_WK", -1);
    const double c_it = NT == 1 ? 130.0 : 150.0;
    double best_cost = -1.0;
    // (grid, blocks per CTA at most): fixed CTA widths, and one or two CTAs
    // per SM with the blocks shared out evenly
    int cg[6], crb[6], nc = 0;
    for (int rb = 1; rb <= 8; rb *= 2, ++nc) {
        cg[nc] = (Nb + rb - 1) / rb;
        crb[nc] = rb;
    }
    for (int q = 1; q <= 2; ++q, ++nc) {
        cg[nc] = Nb < q * sms ? Nb : q * sms;
        crb[nc] = (Nb + cg[nc] - 1) / cg[nc];
    }
    for (int ci = 0; ci < nc; ++ci) {
        const int G = cg[ci], rb = crb[ci];
        if (rb > 8 || (force_rb && rb != force_rb)) continue;
        for (int wk = 0; wk <= kMaxWkLog2; ++wk) {
            if (force_wk >= 0 && wk != force_wk) continue;
            if ((rb << wk) * 32 > 512) continue;
            if (force_wk < 0 && wk > 0 && (1 << wk) > I) continue;
            const Plan p = layout(rb, wk, Mc, I, fmt, MP);
            if (p.ipw > kMaxIpw || p.smem > kMaxSmem) continue;
            int occ = 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, p.threads, p.smem) != cudaSuccess || occ < 1)
                continue;
            const long long ctas = (long long)G * mchunks;
            long long per_sm = (ctas + sms - 1) / sms;
            if (pdl && occ >= 2 && ctas < sms) per_sm = 2;   // the next call doubles up on idle SMs
            const long long waves = (ctas + (long long)sms * occ - 1) / ((long long)sms * occ);
            double cost = per_sm * rb * I * c_it / 4.0 + per_sm * (double)Mc * I * 128 * 2 / 64.0 + p.ipw * c_it +
                          (waves - 1) * 2500.0;
            if (pdl && occ < 2 * ((ctas + sms - 1) / sms)) cost += 4000.0;
            if (best_cost < 0 || cost < best_cost) {
                best_cost = cost;
                best = p;
                grid = G;
            }
        }
    }
    return best_cost >= 0;
}

struct PlanKey {
    int dev, fmt, NT, Mc, mchunks, N, K, pdl, epi;
    bool operator<(const PlanKey& o) const {
        return std::tie(dev, fmt, NT, Mc, mchunks, N, K, pdl, epi) <
               std::tie(o.dev, o.fmt, o.NT, o.Mc, o.mchunks, o.N, o.K, o.pdl, o.epi);
    }
};

}  // namespace

int launch_gemv_staged(const void* A, const void* prepacked, void* C, int M, int N, int K, int fmt, bool out_f32,
                       bool pdl, bool inputs_ready, const Epilogue& epi, cudaStream_t stream) {
    if (inputs_ready) pdl = true;
    if (M == 0 || N == 0) return WQ_OK;
    if (K <= 0 || K > kMaxIpw * (1 << kMaxWkLog2) * 128) return WQ_ERR_UNSUPPORTED;
    const int I = (K + 127) / 128, Nb = (N + 15) / 16;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const bool has_epi = epi.bias || epi.residual || epi.gated;

    // 16 activation rows per CTA (two mma tiles) when they fit beside the
    // weights, else 8, 4, 2 or 1 (one tile; long rows leave room for few)
    Plan plan;
    KernFn kern = nullptr;
    int mrows = 0, grid = 0;
    {
        static std::mutex mu;
        static std::map<PlanKey, std::tuple<Plan, int, bool>> cache;   // shape -> (plan, grid, fits)
        static std::map<std::pair<int, KernFn>, bool> attr_set;
        const bool overridden = getenv("WQ_GEMV_RB") || getenv("WQ_GEMV_TMA_WK");
        std::lock_guard<std::mutex> lock(mu);
        for (int mr = (M > 8 ? 16 : 8); mr >= 1 && !kern; mr = mr == 16 ? 8 : mr / 2) {
            const int NT = mr == 16 ? 2 : 1;
            const int Mc = M < mr ? M : mr;
            const int mchunks = (M + mr - 1) / mr;
            if (mchunks > 65535) return WQ_ERR_UNSUPPORTED;
            KernFn kf = select_kernel(fmt, NT, has_epi);
            if (!attr_set[{dev, kf}]) {
                if (cudaFuncSetAttribute(kf, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kMaxSmem) !=
                    cudaSuccess)
                    return WQ_ERR_CUDA;
                attr_set[{dev, kf}] = true;
            }
            const PlanKey key{dev, fmt, NT, Mc, mchunks, N, K, pdl ? 1 : 0, has_epi ? 1 : 0};
            auto it = overridden ? cache.end() : cache.find(key);
            bool fits;
            if (it != cache.end()) {
                std::tie(plan, grid, fits) = it->second;
            } else {
                fits = choose_plan(kf, fmt, NT, Mc, mchunks, Nb, I, sms, pdl, plan, grid);
                if (!overridden) cache[key] = std::make_tuple(plan, grid, fits);
            }
            if (fits) {
                kern = kf;
                mrows = mr;
            }
        }
    }
    if (!kern) {
        if (debug_on()) fprintf(stderr, "wq: staged GEMV: no CTA shape fits M=%d N=%d K=%d\n", M, N, K);
        return WQ_ERR_UNSUPPORTED;
    }
    if (debug_on())
        fprintf(stderr, "wq: staged GEMV M=%d N=%d K=%d: rows/CTA=%d grid=%d rb=%d wk=%d threads=%d smem=%zu\n", M,
                N, K, mrows, grid, plan.rb, 1 << plan.wk_log2, plan.threads, plan.smem);

    const uint8_t* base = static_cast<const uint8_t*>(prepacked);
    PreArgs args;
    args.codes = base;
    args.recs = base + (size_t)Nb * I * 1024;
    args.A = static_cast<const uint16_t*>(A);
    args.C = C;
    args.M = M;
    args.N = N;
    args.K = K;
    args.I = I;
    args.Nb = Nb;
    args.out_f32 = out_f32 ? 1 : 0;
    args.mrows = mrows;
    args.rb = plan.rb;
    args.wk_log2 = plan.wk_log2;
    args.ipw = plan.ipw;
    args.SA = plan.SA;
    args.w_off = plan.w_off;
    args.a_off = plan.a_off;
    args.r_off = plan.r_off;
    args.red_off = plan.red_off;
    args.inputs_ready = inputs_ready ? 1 : 0;
    args.vec_store = (reinterpret_cast<uintptr_t>(C) & 15) == 0 && N % (out_f32 ? 4 : 8) == 0 && !getenv("WQ_GEMV_SCALAR_STORE");
    args.epi = epi;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, (M + mrows - 1) / mrows, 1);
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
