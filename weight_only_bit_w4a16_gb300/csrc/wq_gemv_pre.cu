// wq_gemv_pre.cu -- the small-M kernel for weights in the prepacked layout
// (wq_prepack.cu; definition above wq_prepack_bytes in include/wq.h).
//
// Arithmetic as in the streaming kernel (wq_gemv_tma.cu): the weights are
// the M operand of mma.sync.m16n8k16 and the activations its N = 8 operand;
// int4 g128 runs the MMAs on the exact integers (code - zero) and scales the
// fp32 partial sums per 128-k block; fp4 weights are decoded with their
// scale (exact in bf16).
//
// Work split.  A CTA takes up to RB blocks of 16 weight rows x all of K; its
// Wk warps split K into equal ranges, and each warp runs its range for ALL of
// the CTA's row blocks, so an activation fragment read from shared memory
// feeds RB row blocks and the CTA fetches each activation byte once.
//
// Data movement.  Nothing is staged whole: every warp streams its range
// through a ring of P slots.  The slot of step t (k-block it0 + t) holds the
// RB code blocks of that k-block (1024 bytes each) and its activation slice
// (Mc rows x 128 k).  The lanes fill a slot with 16-byte cp.async copies and
// then arrive (without a count increment) on the slot's mbarrier, an arrival
// that happens once their copies have landed; a phase of 32 arrivals
// therefore means the whole slot is in shared memory.  The warp refills the
// slot with step t + P once step t's MMAs are done.  The int4 records of the
// warp's range (48 bytes per block: scales and zero points) are copied once,
// ahead of step 0.  The small CTA footprint lets the
// CTAs of several consecutive calls share an SM, so that one call's weights
// stream while another's decode runs.
//
// Dependencies (programmatic dependent launch).  The code blocks of the first
// P steps are requested at once; the activation copies wait for the
// preceding kernel, unless the caller declared A complete already
// (inputs_ready), in which case the kernel waits only before storing C.
//
// Shared memory (from a 128-byte aligned base):
//   bars  [Wk][P] u64 at 0                     slot landed (32 arrivals)
//   ring  [Wk][P][slot_bytes] at ring_off      RB code blocks, then the
//                                              activation rows (256 B, swizzled)
//   recs  [Wk][RB][ipw][48]  int4 at rec_off   the copied record blocks
//         [Wk][RB][ipw][512] fp4               decoded multipliers, per lane
//   red   [Wk][MP][RB*16 + 4] f32 at ring_off  partial sums (aliases ring/recs)
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>

#include "wq_gemv.cuh"
#include "wq_internal.h"
#include "wq_tc.cuh"

namespace wq {

__device__ int g_pre_status = 0;

int read_and_clear_pre_status() {
    int v = 0;
    const int zero = 0;
    if (cudaDeviceSynchronize() != cudaSuccess) return WQ_ERR_CUDA;
    if (cudaMemcpyFromSymbol(&v, g_pre_status, sizeof(int)) != cudaSuccess) return WQ_ERR_CUDA;
    if (cudaMemcpyToSymbol(g_pre_status, &zero, sizeof(int)) != cudaSuccess) return WQ_ERR_CUDA;
    return v;
}

namespace {

using namespace gemv;
using namespace sm100;

constexpr unsigned long long kWaitNs = 2000000000ull;   // 2 s: far above any legal wait
constexpr int kMaxWkLog2 = 3;                           // K ranges (warps) per CTA <= 8
// Activation rows in a slot are 256 bytes apart (128 k), their 16-byte units
// swizzled: unit u of row m sits at position u ^ (4 (m & 1)).  The lanes of a
// quarter-warp read units c + 4j of two adjacent rows, which then fall in
// opposite 64-byte halves of a 128-byte window: no bank conflict, no padding.
constexpr uint32_t kAStride = 256;

struct PreArgs {
    const uint8_t* codes;   // code blocks
    const uint8_t* recs;    // record blocks
    const uint16_t* A;
    void* C;
    int M, N, K;
    int I, Nb;              // 128-k blocks per row, 16-row blocks
    int out_f32;
    int mrows;              // activation rows per CTA (16 or 8)
    int ipw;                // k-blocks per warp (its K range)
    int P;                  // ring slots per warp
    uint32_t slot_bytes;    // RB x 1024 + activation rows x kAStride (128-aligned)
    uint32_t ring_off, rec_off;
    int wide;               // grid x Nb does not fit 32 bits
    int inputs_ready;       // A may be read before the preceding kernel completes
    int vec_store;          // plain output in 16-byte pieces: C 16-byte aligned, N a multiple of 8 (bf16) or 4 (fp32)
    Epilogue epi;
};

__device__ __forceinline__ void record_pre_timeout() { atomicExch(&g_pre_status, WQ_ERR_DEVICE_TIMEOUT); }

__device__ __forceinline__ uint32_t lds32(uint32_t saddr) {
    uint32_t v;
    asm("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(saddr));
    return v;
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
// copies `bytes` (0 or 16) and zero-fills the rest of the 16-byte unit
__device__ __forceinline__ void cp_async16_zfill(uint32_t dst, const void* src, uint32_t bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(bytes) : "memory");
}
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// The lane's four words of one 128-k block, rows r (qa) and r + 8 (qb), in
// the order of the k units c, c + 4, c + 8, c + 12.  wp: the lane's 8 bytes
// of half 0, row r (row r + 8 is 256 bytes on, half 1 is 512 bytes on).
__device__ __forceinline__ void block_words(uint32_t wp, uint4& qa, uint4& qb) {
    const uint2 a0 = lds64(wp), b0 = lds64(wp + 256), a1 = lds64(wp + 512), b1 = lds64(wp + 768);
    qa = make_uint4(a0.x, a0.y, a1.x, a1.y);
    qb = make_uint4(b0.x, b0.y, b1.x, b1.y);
}

// One warp's stream: step t (k-block it0 + t) lands in slot t mod P.
template <int RB, int NT>
struct Ring {
    uint32_t slots;           // slot 0 (shared address)
    uint32_t bar;             // barrier of slot 0 (8 bytes per slot)
    uint32_t slot_bytes;
    const uint8_t* codes;     // code block (bs, it0) in global memory
    size_t row_stride;        // bytes between the blocks of consecutive row blocks (I x 1024)
    const uint16_t* asrc;     // the lane's first activation unit: row mz + (lane >> 4), k = it0 * 128 + 8 (lane & 15)
    const uint16_t* azero;    // a valid address for the zero-filled units (no byte is read there)
    size_t lda2;              // two activation rows (2 K elements)
    int krem;                 // k left in the row from it0 * 128, minus 8 (lane & 15)
    uint32_t adst;            // the lane's first unit in a slot's activation rows
    int aunits;               // 16-byte units the lane copies per step: rows lane >> 4, + 2, ... < Mc
    uint32_t lda2b;           // bytes between two activation rows
    int kfull;                // steps that lie wholly inside K
    int nb, nit, P, lane;

    __device__ __forceinline__ void issue_codes(int t, int slot) const {
        const uint32_t d = slots + slot_bytes * slot + 16u * lane;
        const uint8_t* g = codes + (size_t)t * 1024 + 16 * lane;
#pragma unroll
        for (int q = 0; q < RB; ++q) {
            if (q < nb) {
                cp_async16(d + 1024u * q, g + row_stride * q);
                cp_async16(d + 1024u * q + 512, g + row_stride * q + 512);
            }
        }
    }
    // the activation slice of step t (16-byte units past K zero-filled: K is
    // a multiple of 32, so a unit is wholly inside or outside), then the
    // lane's arrival on the slot's barrier, which covers every copy the lane
    // issued before it
    __device__ __forceinline__ void issue_acts(int t, int slot) const {
        // two tiles, a step inside K, all 16 rows: the lane's 8 units at
        // fixed offsets (v * 2 rows), no loop
        if constexpr (NT == 2) {
            if (t < kfull && aunits == 8) {
                const uint32_t d = slots + slot_bytes * slot + adst;
                const uint8_t* g = reinterpret_cast<const uint8_t*>(asrc + t * 128);
#pragma unroll
                for (int v = 0; v < 8; ++v) cp_async16(d + 2u * kAStride * v, g + (uint32_t)v * lda2b);
                cp_async_arrive_noinc(bar + 8u * slot);
                return;
            }
        }
        uint32_t d = slots + slot_bytes * slot + adst;
        const bool in = t * 128 < krem;
        const uint16_t* g = in ? asrc + t * 128 : azero;
        const uint32_t bytes = in ? 16u : 0u;
        for (int v = 0; v < aunits; ++v) {
            cp_async16_zfill(d, g, bytes);
            d += 2 * kAStride;
            if (in) g += lda2;
        }
        cp_async_arrive_noinc(bar + 8u * slot);
    }
    // wait for the slot whose current phase has parity ph; ties sb to the
    // wait so that the compiler cannot hoist the slot's shared loads above it
    __device__ __forceinline__ bool wait(int slot, uint32_t ph, uint32_t& sb) const {
        const bool ok = mbar_wait_sleep(bar + 8u * slot, ph, kWaitNs);
        asm volatile("" : "+r"(sb)::"memory");
        return ok;
    }
    // after a failed wait: let the steps still in flight, [from, upto), land
    // (bounded) before the CTA's shared memory can be reused
    __device__ __forceinline__ void drain(int from, int upto) const {
        for (int j = from; j < upto; ++j) {
            uint32_t dummy = 0;
            if (!wait(j % P, (uint32_t)(j / P) & 1u, dummy)) break;
        }
    }
};

// Every shared load of a step's slot feeds an MMA whose result ends up in
// the accumulators; this volatile asm needs them, so the compiler has the
// step's loads and MMAs done before it, and therefore before the refill
// copies that follow it.
template <int RB, int NT>
__device__ __forceinline__ void slot_consumed(float (&acc)[RB][NT][4]) {
#pragma unroll
    for (int q = 0; q < RB; ++q)
#pragma unroll
        for (int t = 0; t < NT; ++t)
            asm volatile("" ::"f"(acc[q][t][0]), "f"(acc[q][t][1]), "f"(acc[q][t][2]), "f"(acc[q][t][3])
                         : "memory");
    __syncwarp();
}

// int4 g128, row blocks q0 .. q0 + QI - 1 of a step, their MMA chains
// interleaved word by word (independent accumulators in flight together).
// rec0: record block of row block 0 of this step; rec_stride: bytes between
// the record blocks of consecutive row blocks.
// Activation fragments come from the slot (sa0): unit c + 4j of the lane's
// row sits at aoffE + 64j for even j and aoffO + 64j for odd j (the row's
// swizzle).  One tile (M <= 8) reads all four 32-k slices up front; two tiles
// read each slice as its MMAs need it (the registers that holding all four
// would take are what a 16-row step lacks).
template <int NT, int QI, bool TWO>
__device__ __forceinline__ void step_int4_group(uint32_t wp0, uint32_t rec0, uint32_t rec_stride, uint32_t r,
                                                uint32_t sa0, const uint32_t (&aoffE)[NT], const uint32_t (&aoffO)[NT],
                                                float (*acc)[NT][4]) {
    uint4 bv1[4];
    if constexpr (NT == 1) {
#pragma unroll
        for (int j = 0; j < 4; ++j) bv1[j] = lds128(sa0 + ((j & 1) ? aoffO[0] : aoffE[0]) + 64u * j);
    }
    uint32_t wa[QI][4], wb[QI][4], zzA[QI], zzB[QI], zzA2[QI], zzB2[QI];
    float sa[QI], sb[QI];
#pragma unroll
    for (int q = 0; q < QI; ++q) {
        uint4 qa, qb;
        block_words(wp0 + 1024u * q, qa, qb);
        wa[q][0] = qa.x; wa[q][1] = qa.y; wa[q][2] = qa.z; wa[q][3] = qa.w;
        wb[q][0] = qb.x; wb[q][1] = qb.y; wb[q][2] = qb.z; wb[q][3] = qb.w;
        // rows r and r + 8: bf16 scales at 4r, zero points at 32 + 2r
        const uint32_t rec = rec0 + rec_stride * q;
        const uint32_t sp = lds32(rec + 4u * r), zp = lds16(rec + 32u + 2u * r);
        sa[q] = __uint_as_float(sp << 16);
        sb[q] = __uint_as_float(sp & 0xFFFF0000u);
        if constexpr (TWO) {
            zsub_two(zp & 0xFFu, zzA[q], zzA2[q]);
            zsub_two(zp >> 8, zzB[q], zzB2[q]);
        } else {
            zzA[q] = zsub_lo(zp);
            zzB[q] = zsub_hi(zp);
            zzA2[q] = zzB2[q] = 0;
        }
    }
    // one MMA chain per tile and row block: the QI row blocks' chains are
    // already independent (a second chain per tile measured 1-2 % slower)
    constexpr int CH = 1;
    float part[QI][CH][NT][4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint4 bj[NT];
#pragma unroll
        for (int t = 0; t < NT; ++t)
            bj[t] = NT == 1 ? bv1[j] : lds128(sa0 + ((j & 1) ? aoffO[t] : aoffE[t]) + 64u * j);
#pragma unroll
        for (int q = 0; q < QI; ++q) {
            uint32_t pa[4], pb[4];
            int4_word_kk4<TWO>(wa[q][j], zzA[q], zzA2[q], pa);
            int4_word_kk4<TWO>(wb[q][j], zzB[q], zzB2[q], pb);
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                if (j < CH) mma16816_z(part[q][j % CH][t], pa[0], pb[0], pa[1], pb[1], bj[t].x, bj[t].y);
                else mma16816(part[q][j % CH][t], pa[0], pb[0], pa[1], pb[1], bj[t].x, bj[t].y);
                mma16816(part[q][j % CH][t], pa[2], pb[2], pa[3], pb[3], bj[t].z, bj[t].w);
            }
        }
    }
#pragma unroll
    for (int q = 0; q < QI; ++q)
#pragma unroll
        for (int t = 0; t < NT; ++t)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float p = part[q][0][t][e];
                if constexpr (CH == 2) p += part[q][CH - 1][t][e];
                acc[q][t][e] = fmaf(e < 2 ? sa[q] : sb[q], p, acc[q][t][e]);
            }
}

// fp4, one row block of a step.  rp: the lane's decoded multipliers, words
// j = 0..3 of row r (16 bytes) then of row r + 8; the second multipliers
// (MXFP4 scales above 2^15) 256 bytes on.
template <int NT, bool TWO>
__device__ __forceinline__ void step_fp4(uint32_t wp, uint32_t rp, const uint4 (&bv)[NT][4], float (&acc)[NT][4]) {
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
            mma16816(acc[t], pa[0], pb[0], pa[1], pb[1], bv[t][j].x, bv[t][j].y);
            mma16816(acc[t], pa[2], pb[2], pa[3], pb[3], bv[t][j].z, bv[t][j].w);
        }
    }
}

// The warp's whole range, step by step as the slots land: every row block of
// the step, then the refill of the slot.  Returns false if a copy never
// landed (the ones still in flight are drained first).
//   lane_w : the lane's weight offset in a code block
//   aoff   : the lane's activation offset in a slot, per MMA tile
//   rlane  : the lane's offset in a record block (int4: its row r)
template <int FMT, int NT, int RB, bool TWO>
__device__ __forceinline__ bool run_range(const Ring<RB, NT>& ring, uint32_t lane_w, const uint32_t (&aoffE)[NT],
                                          const uint32_t (&aoffO)[NT], uint32_t rslice, uint32_t rlane, int ipw,
                                          float (&acc)[RB][NT][4]) {
    constexpr uint32_t kRec = FMT == kINT4 ? 48 : 512;
    int slot = 0;
    uint32_t ph = 0;
    for (int i = 0; i < ring.nit; ++i) {
        uint32_t sb = ring.slots + ring.slot_bytes * slot;
        if (!ring.wait(slot, ph, sb)) {
            ring.drain(i + 1, min(ring.nit, i + ring.P));
            return false;
        }
        if constexpr (FMT == kINT4) {
            // row blocks in groups of two, each group's MMA chains
            // interleaved; a CTA's row blocks past nb compute on stale slot
            // bytes and are never stored
            constexpr int QI = RB < 2 ? RB : 2;
#pragma unroll
            for (int q0 = 0; q0 < RB; q0 += QI)
                step_int4_group<NT, QI, TWO>(sb + 1024u * q0 + lane_w, rslice + (uint32_t)(q0 * ipw + i) * kRec,
                                             (uint32_t)ipw * kRec, rlane, sb, aoffE, aoffO, &acc[q0]);
        } else {
            // the step's activation fragments, read once for all its row blocks
            uint4 bv[NT][4];
#pragma unroll
            for (int t = 0; t < NT; ++t)
#pragma unroll
                for (int j = 0; j < 4; ++j) bv[t][j] = lds128(sb + ((j & 1) ? aoffO[t] : aoffE[t]) + 64u * j);
#pragma unroll
            for (int q = 0; q < RB; ++q) {
                if (q < ring.nb) {
                    const uint32_t rec = rslice + (uint32_t)(q * ipw + i) * kRec;
                    step_fp4<NT, TWO>(sb + 1024u * q + lane_w, rec + rlane, bv, acc[q]);
                }
            }
        }
        slot_consumed<RB, NT>(acc);
        if (i + ring.P < ring.nit) {
            ring.issue_codes(i + ring.P, slot);
            ring.issue_acts(i + ring.P, slot);
        }
        if (++slot == ring.P) {
            slot = 0;
            ph ^= 1u;
        }
    }
    return true;
}

template <int FMT, int NT, bool EPI, int RB>
__global__ void __launch_bounds__(256, 2) gemv_pre_kernel(const PreArgs a) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t sbase = (smem_u32(smem_raw) + 127u) & ~127u;
    uint8_t* sgen = smem_raw + (sbase - smem_u32(smem_raw));
    constexpr bool kInt4 = FMT == kINT4;
    constexpr uint32_t kRec = kInt4 ? 48 : 512;   // shared record bytes per row block and k-block
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int Wk = blockDim.x >> 5;
    const int r = lane >> 2, c = lane & 3;
    constexpr int rows = RB * 16;
    // this CTA's row blocks: an even share of the Nb blocks (at most RB)
    const int bs = a.wide ? (int)((long long)blockIdx.x * a.Nb / gridDim.x)
                          : (int)(blockIdx.x * (unsigned)a.Nb / gridDim.x);
    const int be = a.wide ? (int)((long long)(blockIdx.x + 1) * a.Nb / gridDim.x)
                          : (int)((blockIdx.x + 1) * (unsigned)a.Nb / gridDim.x);
    const int nb = be - bs;
    const int n0 = bs * 16, n_end = min(a.N, be * 16);
    const int mz = blockIdx.y * a.mrows;
    const int Mc = min(a.mrows, a.M - mz);
    const int it0 = warp * a.ipw;
    const int nit = max(0, min(a.I, it0 + a.ipw) - it0);   // this warp's k-blocks
    const uint32_t rslice = sbase + a.rec_off + (uint32_t)(warp * RB * a.ipw) * kRec;

    Ring<RB, NT> ring;
    ring.slots = sbase + a.ring_off + (uint32_t)(warp * a.P) * a.slot_bytes;
    ring.bar = sbase + 8u * (uint32_t)(warp * a.P);
    ring.slot_bytes = a.slot_bytes;
    ring.codes = a.codes + ((size_t)bs * a.I + it0) * 1024;
    ring.row_stride = (size_t)a.I * 1024;
    ring.asrc = a.A + (size_t)(mz + (lane >> 4)) * a.K + (size_t)it0 * 128 + 8 * (lane & 15);
    ring.azero = a.A;
    ring.lda2 = 2 * (size_t)a.K;
    ring.krem = a.K - it0 * 128 - 8 * (lane & 15);
    // the lane's rows all have the parity of lane >> 4: one swizzled position
    ring.adst = 1024u * RB + kAStride * (uint32_t)(lane >> 4) + 16u * ((lane & 15) ^ (4 * (lane >> 4)));
    ring.aunits = Mc > (lane >> 4) ? (Mc - (lane >> 4) + 1) >> 1 : 0;
    ring.lda2b = 4u * (uint32_t)a.K;
    ring.kfull = a.K / 128 - it0;
    ring.nb = nb;
    ring.nit = nit;
    ring.P = a.P;
    ring.lane = lane;
    const int npro = min(a.P, nit);
    // int4: the prepacked weight's flag (a zero point above 128 anywhere),
    // read now and needed once step 0 has landed
    const uint32_t large_zero = kInt4 ? ldg_u32(a.recs + (size_t)a.Nb * a.I * 48) : 0u;

    // with the inputs declared ready nothing waits on the preceding kernel
    // before the stores, so the next call may be scheduled at once
    if (a.inputs_ready) grid_dependents_launch();
    if (lane < npro) mbar_init(ring.bar + 8 * lane, 32);
    fence_mbarrier_init();
    __syncthreads();

    // ---- 1. records (int4: copied ahead of step 0's arrival, so that its
    // barrier covers them) and the code blocks of the first P steps
    if (nit > 0) {
        if constexpr (kInt4) {
            for (int q = 0; q < nb; ++q)
                for (int u = lane; u < nit * 3; u += 32)
                    cp_async16(rslice + (uint32_t)(q * a.ipw) * 48u + 16u * u,
                               a.recs + ((size_t)(bs + q) * a.I + it0) * 48 + 16 * u);
        }
        for (int t = 0; t < npro; ++t) ring.issue_codes(t, t);
    }

    // ---- 2. fp4: decode multipliers into the lane order of the loop
    bool two = false;
    if constexpr (!kInt4) {
        uint8_t* s8 = sgen + (rslice - sbase);
        for (int q = 0; q < nb; ++q) {
            const size_t blk0 = (size_t)(bs + q) * a.I + it0;
            uint8_t* sq = s8 + (size_t)q * a.ipw * 512;
            if constexpr (FMT == kNVFP4) {
                // record block: row rho's 8 bytes at 8 rho; lane = (rho, half
                // of the groups); group g feeds word j = g >> 1 of the lanes
                // with (c >> 1) == (g & 1)
                const int rho = lane >> 1, g0 = 4 * (lane & 1);
                for (int t = 0; t < nit; ++t) {
                    const uint32_t raw = ldg_u32(a.recs + (blk0 + t) * 128 + 4 * lane);
                    const uint32_t f01 = e4m3x2_to_f16x2(raw & 0xFFFFu), f23 = e4m3x2_to_f16x2(raw >> 16);
                    const uint32_t hv[4] = {f01 & 0xFFFFu, f01 >> 16, f23 & 0xFFFFu, f23 >> 16};
#pragma unroll
                    for (int g4 = 0; g4 < 4; ++g4) {
                        const int g = g0 + g4;
                        const uint32_t off =
                            t * 512 + (((rho & 7) * 2 + (g & 1)) * 32) + (rho >> 3) * 16 + (g >> 1) * 4;
                        *reinterpret_cast<uint32_t*>(sq + off) = splat16(nvfp4_mul_from_f16(hv[g4]));
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
                        *reinterpret_cast<uint32_t*>(sq + off) = k.mul;
                        *reinterpret_cast<uint32_t*>(sq + off + 256) = k.mul2;
                    }
                }
            }
        }
        two = __any_sync(0xffffffffu, two);
        __syncwarp();   // the lanes read multipliers other lanes wrote
    }

    // ---- 3. the next kernel may start.  C is written only after the
    // preceding kernel has finished; A is read after it too, unless the
    // caller declared it complete already (inputs_ready)
    grid_dependents_launch();
    if (!a.inputs_ready) grid_dependency_wait();
    for (int t = 0; t < npro; ++t) ring.issue_acts(t, t);

    // ---- 4. the range, step by step as the slots land ----------------------
    constexpr int MP = NT * 8;
    float acc[RB][NT][4];
#pragma unroll
    for (int q = 0; q < RB; ++q)
#pragma unroll
        for (int t = 0; t < NT; ++t)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[q][t][e] = 0.f;
    bool ok = true;
    if (nit > 0) {
        uint32_t dummy = 0;
        ok = ring.wait(0, 0u, dummy);   // step 0 (and the int4 records)
        if (!ok) ring.drain(1, npro);
    }
    if constexpr (kInt4) two = (large_zero & 0xFFu) != 0;   // some zero point above 128: two subtrahends
    if (ok && nit > 0) {
        // activation rows past Mc are not copied: those lanes read row 0 or 1
        // (keeping the row parity of a copied neighbour); their outputs are
        // never stored
        // (unit c + 4j of row ms sits at 16 c + 64 (j ^ (ms & 1)): +64 bytes
        // for even j and -64 for odd j on odd rows)
        uint32_t aoffE[NT], aoffO[NT];
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            const int m = t * 8 + r;
            const int ms = m < Mc ? m : (Mc > 1 ? (m & 1) : 0);
            const uint32_t aoff = 1024u * RB + kAStride * (uint32_t)ms + 16u * c, sw = 64u * (uint32_t)(ms & 1);
            aoffE[t] = aoff + sw;
            aoffO[t] = aoff - sw;
        }
        const uint32_t lane_w = 32u * r + 16u * ((c >> 1) ^ ((r >> 2) & 1)) + 8u * (c & 1);
        const uint32_t rlane = kInt4 ? (uint32_t)r : (FMT == kNVFP4 ? (2u * r + (c >> 1)) * 32u : 32u * r);
        ok = two ? run_range<FMT, NT, RB, true>(ring, lane_w, aoffE, aoffO, rslice, rlane, a.ipw, acc)
                 : run_range<FMT, NT, RB, false>(ring, lane_w, aoffE, aoffO, rslice, rlane, a.ipw, acc);
    }
    if (!ok && lane == 0) record_pre_timeout();
    if (a.inputs_ready) grid_dependency_wait();   // completion order: stores after the predecessor's
    if (__syncthreads_or(!ok)) return;           // a copy never landed: store nothing

    // ---- 5. partial sums -> shared memory, fixed-order reduction, store ----
    const int ld = rows + 4;
    float* red = reinterpret_cast<float*>(sgen + a.ring_off);
#pragma unroll
    for (int q = 0; q < RB; ++q) {
        if (q < nb) {
            const int y = q * 16 + r;
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                const int m = t * 8 + 2 * c;
                float* p = red + ((size_t)warp * MP + m) * ld + y;
                p[0] = acc[q][t][0];
                p[ld] = acc[q][t][1];
                p[8] = acc[q][t][2];
                p[ld + 8] = acc[q][t][3];
            }
        }
    }
    __syncthreads();
    const bool gated = EPI && a.epi.gated;
    constexpr int outs_full = rows;
    const int outs = gated ? outs_full >> 1 : outs_full;   // a power of two
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
constexpr int kMaxK = 16384;
constexpr size_t kMaxSmem = 227 * 1024;

struct Plan {
    int RB = 0, Wk = 0, P = 0, ipw = 0, grid = 0;
    size_t smem = 0;
    uint32_t slot_bytes = 0, ring_off = 0, rec_off = 0;
};

using KernFn = void (*)(PreArgs);

template <int FMT, int NT, int RB>
KernFn kernel_for(bool epi) {
    return epi ? gemv_pre_kernel<FMT, NT, true, RB> : gemv_pre_kernel<FMT, NT, false, RB>;
}
template <int FMT, int NT>
KernFn kernel_rb(int RB, bool epi) {
    return RB == 1 ? kernel_for<FMT, NT, 1>(epi) : RB == 2 ? kernel_for<FMT, NT, 2>(epi) : kernel_for<FMT, NT, 4>(epi);
}
KernFn select_kernel(int fmt, int NT, int RB, bool epi) {
    if (fmt == kNVFP4) return NT == 1 ? kernel_rb<kNVFP4, 1>(RB, epi) : kernel_rb<kNVFP4, 2>(RB, epi);
    if (fmt == kMXFP4) return NT == 1 ? kernel_rb<kMXFP4, 1>(RB, epi) : kernel_rb<kMXFP4, 2>(RB, epi);
    return NT == 1 ? kernel_rb<kINT4, 1>(RB, epi) : kernel_rb<kINT4, 2>(RB, epi);
}

uint32_t round128(size_t x) { return (uint32_t)((x + 127) & ~(size_t)127); }

// Shared memory of a CTA shape (section comment at the top of the file).
Plan layout(int RB, int Wk, int P, int Mc, int I, int fmt, int MP) {
    Plan p;
    p.RB = RB;
    p.Wk = Wk;
    p.ipw = (I + Wk - 1) / Wk;
    p.P = P < p.ipw ? P : p.ipw;
    p.ring_off = round128((size_t)8 * Wk * p.P);
    p.slot_bytes = round128((size_t)1024 * RB + (size_t)kAStride * Mc);
    p.rec_off = p.ring_off + (uint32_t)(Wk * p.P) * p.slot_bytes;
    // int4 records take 48 bytes per block, but 96 are reserved: with the
    // smaller CTAs more calls overlap on an SM, and a chain of calls of
    // mixed M then collapses in some orders (same GPU: M = 1, 4, 16 in turn
    // 9.5 -> 22.5 us per step), later calls taking the issue slots of the
    // oldest one, whose completion every later store waits for
    const size_t end = p.rec_off + (size_t)Wk * RB * p.ipw * (fmt == kINT4 ? 96 : 512);
    const size_t red = p.ring_off + (size_t)Wk * MP * (RB * 16 + 4) * sizeof(float);
    p.smem = (end > red ? end : red) + 128;   // + base alignment slack
    return p;
}

int env_int(const char* name, int dflt) {
    const char* e = getenv(name);
    return e ? atoi(e) : dflt;
}

// Kernels take up to 227 KB of dynamic shared memory (set once per device
// and kernel, before any occupancy query or launch).
bool allow_smem(int dev, KernFn kern) {
    static std::mutex mu;
    static std::map<std::pair<int, KernFn>, bool> done;
    std::lock_guard<std::mutex> lock(mu);
    if (done[{dev, kern}]) return true;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kMaxSmem) != cudaSuccess)
        return false;
    done[{dev, kern}] = true;
    return true;
}

// The CTA shape: RB row blocks per CTA (grid = ceil(Nb / RB)), Wk warps (K
// ranges) per CTA, P ring slots per warp.  Two regimes:
//   inputs ready  the call overlaps the calls before and after it end to
//                 end, so what counts is how many calls' CTAs share an SM
//                 (small CTAs, a ring of 3) and the activation bytes each SM
//                 copies (all of K per CTA);
//   otherwise     the call's product can only start once its predecessor
//                 has finished, so the whole range is requested at once
//                 (P = the range) while that one runs, and the product after
//                 the wait needs enough warps to keep the SM busy; a chained
//                 call only streams early if its CTAs fit beside the
//                 previous call's.
// Overlapped and plain launches share a plan, so that flag never changes the
// result's bits (the ready plan may split K differently: a rounding-level
// difference, within the gate).  Costs are SM cycles of one call.
// WQ_RING_RB / WQ_RING_WK (log2 of Wk) / WQ_RING_P force a shape (tests,
// sweeps).
bool choose_plan(int dev, int fmt, int NT, bool epi, int Mc, int mchunks, int Nb, int I, int K, int sms, bool ready,
                 Plan& best) {
    const int MP = NT * 8;
    const int force_rb = env_int("WQ_RING_RB", 0), force_wk = env_int("WQ_RING_WK", -1);
    const int force_p = env_int("WQ_RING_P", 0);
    const double c_it = NT == 1 ? 140.0 : 170.0;   // issue cycles of one warp per 16 x 128 block
    if (ready && !force_rb && force_wk < 0 && force_p <= 0) {
        // Measured on GB300 (chained int4 calls with their inputs ready, every
        // (RB, Wk, P) in {1,2,4} x {1,2,4,8} x {2,3}, on the decoder's q/o,
        // k/v, gate/up, down and LM-head shapes at M = 1, 4, 16): two-slot
        // rings; up to 8 activation rows, four row blocks per CTA once there
        // are 128 row blocks and ~256 warps per call; 16 rows, two row
        // blocks and ~384 warps.  Within 5 % of the best shape everywhere.
        // Take that shape when it fits, else fall through to the cost model.
        const int RB = NT == 1 ? (Nb >= 128 ? 4 : (Nb >= 64 ? 2 : 1)) : (Nb >= 64 ? 2 : 1);
        const int G = (Nb + RB - 1) / RB;
        const double want = (NT == 1 ? 256.0 : 384.0) / ((double)G * mchunks);
        int Wk = 1;
        while (Wk < (1 << kMaxWkLog2) && 2 * Wk <= want && 2 * Wk <= I) Wk *= 2;
        const KernFn kern = select_kernel(fmt, NT, RB, epi);
        if (!allow_smem(dev, kern)) return false;
        const Plan p = layout(RB, Wk, 2, Mc, I, fmt, MP);
        int occ = 0;
        if (p.smem <= kMaxSmem &&
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, Wk * 32, p.smem) == cudaSuccess && occ >= 1) {
            best = p;
            best.grid = G;
            return true;
        }
    }
    double best_cost = -1.0;
    for (int RB = 1; RB <= 4; RB *= 2) {
        if (force_rb && RB != force_rb) continue;
        const KernFn kern = select_kernel(fmt, NT, RB, epi);
        if (!allow_smem(dev, kern)) return false;
        const int G = (Nb + RB - 1) / RB;
        for (int wk = 0; wk <= kMaxWkLog2; ++wk) {
            const int Wk = 1 << wk;
            if (force_wk >= 0 && wk != force_wk) continue;
            if (force_wk < 0 && wk > 0 && Wk > I) continue;
            const int ipw = (I + Wk - 1) / Wk;
            int P = force_p > 0 ? force_p : (ready ? 3 : ipw);
            Plan p = layout(RB, Wk, P, Mc, I, fmt, MP);
            // not ready: the deepest ring that fits (steps beyond it stream
            // after the dependency wait)
            while (p.smem > kMaxSmem && !ready && force_p <= 0 && P > 2) p = layout(RB, Wk, --P, Mc, I, fmt, MP);
            if (p.smem > kMaxSmem) continue;
            int occ = 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, Wk * 32, p.smem) != cudaSuccess || occ < 1)
                continue;
            const double ctas = (double)G * mchunks, per_sm = ctas / sms;
            const double act = per_sm * (double)Mc * K * 2 / 64.0;
            double cost;
            if (ready) {
                cost = act + per_sm * 800.0 + (double)RB * p.ipw * c_it * 0.5;
                const double depth = occ / per_sm;   // calls whose CTAs fit on an SM together
                if (depth < 3.0) cost += (3.0 - depth) * 1500.0;
            } else {
                const double busiest = ceil(per_sm);
                const double loop_sm = busiest * RB * I * c_it / 4.0;                   // issue-bound
                const double loop_warp = (double)RB * p.ipw * c_it * 3.0;               // latency-bound
                cost = act + busiest * 800.0 + (loop_sm > loop_warp ? loop_sm : loop_warp);
                const double waves = ceil(ctas / ((double)sms * occ));
                cost += (waves - 1.0) * 2500.0;
                if (occ < 2.0 * busiest) cost += 4000.0;   // no room for the next call's CTAs
                cost += (double)(p.ipw - p.P) / p.ipw * 3000.0;   // steps fetched after the wait
            }
            if (best_cost < 0 || cost < best_cost) {
                best_cost = cost;
                best = p;
                best.grid = G;
            }
        }
    }
    return best_cost >= 0;
}

struct PlanKey {
    int dev, fmt, NT, Mc, mchunks, N, K, epi, ready;
    bool operator<(const PlanKey& o) const {
        return std::tie(dev, fmt, NT, Mc, mchunks, N, K, epi, ready) <
               std::tie(o.dev, o.fmt, o.NT, o.Mc, o.mchunks, o.N, o.K, o.epi, o.ready);
    }
};

}  // namespace

// Calls that declare their inputs ready run this file's ring kernel;
// dependent and plain calls the staged kernel (wq_gemv_staged.cu), which
// requests a CTA's whole slice before its dependency wait.
// WQ_GEMV_PRE_KERNEL=ring|staged forces one of them (tests).
int launch_gemv_prepacked(const void* A, const void* prepacked, void* C, int M, int N, int K, int fmt,
                          bool out_f32, bool pdl, bool inputs_ready, const Epilogue& epi, cudaStream_t stream) {
    const char* force = getenv("WQ_GEMV_PRE_KERNEL");
    const bool ring = force ? strcmp(force, "staged") != 0 : inputs_ready;
    if (!ring) return launch_gemv_staged(A, prepacked, C, M, N, K, fmt, out_f32, pdl, inputs_ready, epi, stream);
    if (inputs_ready) pdl = true;
    if (M == 0 || N == 0) return WQ_OK;
    if (K <= 0 || K > kMaxK) return WQ_ERR_UNSUPPORTED;
    const int I = (K + 127) / 128, Nb = (N + 15) / 16;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const bool has_epi = epi.bias || epi.residual || epi.gated;

    // 16 activation rows per CTA (two MMA tiles) above 8 rows, else one tile
    const int mrows = M > 8 ? 16 : 8;
    const int NT = mrows == 16 ? 2 : 1;
    const int Mc = M < mrows ? M : mrows;
    const int mchunks = (M + mrows - 1) / mrows;
    if (mchunks > 65535) return WQ_ERR_UNSUPPORTED;
    Plan plan;
    bool fits;
    {
        static std::mutex mu;
        static std::map<PlanKey, std::pair<Plan, bool>> cache;   // shape -> (plan, fits)
        const bool overridden = getenv("WQ_RING_RB") || getenv("WQ_RING_WK") || getenv("WQ_RING_P");
        std::lock_guard<std::mutex> lock(mu);
        const PlanKey key{dev, fmt, NT, Mc, mchunks, N, K, has_epi ? 1 : 0, inputs_ready ? 1 : 0};
        auto it = overridden ? cache.end() : cache.find(key);
        if (it != cache.end()) {
            std::tie(plan, fits) = it->second;
        } else {
            fits = choose_plan(dev, fmt, NT, has_epi, Mc, mchunks, Nb, I, K, sms, inputs_ready, plan);
            if (!overridden) cache[key] = std::make_pair(plan, fits);
        }
    }
    if (!fits) {
        if (debug_on()) fprintf(stderr, "wq: prepacked GEMV: no CTA shape fits M=%d N=%d K=%d\n", M, N, K);
        return WQ_ERR_UNSUPPORTED;
    }
    KernFn kern = select_kernel(fmt, NT, plan.RB, has_epi);
    if (!allow_smem(dev, kern)) return WQ_ERR_CUDA;
    if (debug_on())
        fprintf(stderr, "wq: prepacked GEMV M=%d N=%d K=%d: rows/CTA=%d grid=%d RB=%d Wk=%d P=%d threads=%d smem=%zu\n",
                M, N, K, mrows, plan.grid, plan.RB, plan.Wk, plan.P, plan.Wk * 32, plan.smem);

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
    args.ipw = plan.ipw;
    args.P = plan.P;
    args.slot_bytes = plan.slot_bytes;
    args.ring_off = plan.ring_off;
    args.rec_off = plan.rec_off;
    args.wide = (unsigned long long)(plan.grid + 1) * (unsigned long long)Nb >= (1ull << 32) ? 1 : 0;
    args.inputs_ready = inputs_ready ? 1 : 0;
    args.vec_store = (reinterpret_cast<uintptr_t>(C) & 15) == 0 && N % (out_f32 ? 4 : 8) == 0 && !getenv("WQ_GEMV_SCALAR_STORE");
    args.epi = epi;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(plan.grid, mchunks, 1);
    cfg.blockDim = dim3(plan.Wk * 32, 1, 1);
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
