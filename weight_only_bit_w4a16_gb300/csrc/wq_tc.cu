// wq_tc.cu -- the large-M path: TMA-fed, warp-specialised tcgen05 kernel with
// the dequantised weights in tensor memory, and the device status word that
// its bounded waits report into.
//
// Tile: 128 weight rows (n) x bm activation rows (m, a multiple of 32 up to
// 256 for int4 and 384 for the fp4 formats, chosen per call to limit the
// last partial wave) x all of K, in k-steps of 64.  The product is computed
// transposed, D = W . A^T, so that the dequantised weights are the A operand
// of tcgen05.mma and can live in TMEM:
//   * warp 0, one lane: TMA producer.  Per k-step it loads the activation
//     tile (bm x 64 bf16, 128-byte swizzle, the MMA's B operand in shared
//     memory; above 256 rows as two boxes of bm / 2) and the packed weight
//     tile (128 rows x 32 bytes, 32-byte swizzle) into a ring of kStages
//     stages, completing on the stage's "full" mbarrier.
//   * warps 2.. (kDecodeSets sets of 4 warps, thread = weight row; set j
//     takes the k-steps ks = j mod kDecodeSets): decode.  Each thread reads
//     its row's 32 packed bytes, dequantises them in registers (the routine
//     of wq_common.cuh) and writes the 64 bf16 weights into TMEM with one
//     tcgen05.st (32 columns of its lane); int4 weights go in as the exact
//     two-term split hi + lo, two stores.  The weights never pass through
//     shared memory.
//   * warp 1, one lane: issues 4 (int4: 8) tcgen05.mma.kind::f16 (M=128,
//     N=bm, K=16) per k-step with A from TMEM, B from shared memory, the
//     fp32 accumulator in TMEM; tcgen05.commit frees the stage and the TMEM
//     weight buffer.  Above 256 rows (fp4) the tile is two MMAs of N = bm / 2
//     on the same decoded weights: one decode of a k-step feeds up to 384
//     activation rows.  This is what the fp4 weight buffers' 32 TMEM columns
//     leave room for (384 accumulator + 4 x 32 = 512 columns); int4 keeps
//     256 + 4 x 64 (its hi and lo terms).
//   * the decode warps again: epilogue, tcgen05.ld of the accumulator (their
//     lane quarter; the sets split the columns), fp32 -> bf16/fp32, stores.
//     A whole tile of plain bf16 output goes to a shared staging tile
//     instead: the accumulator is released as soon as it is read, and one
//     thread writes the tile with a bulk tensor store that runs while the
//     next tile starts.
// Every wait is bounded in wall time (%globaltimer); a wait that runs out
// records WQ_ERR_DEVICE_TIMEOUT in the device status word, the CTA unwinds
// (outstanding TMA copies and MMAs are waited for, again with a bound) and
// frees its tensor memory.
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "wq_common.cuh"
#include "wq_internal.h"
#include "wq_tc.cuh"

namespace wq {

// WQ_OK, or WQ_ERR_DEVICE_TIMEOUT once a bounded wait of a kernel gave up.
__device__ int g_device_status = 0;

// Devices whose library scratch (wq_gemm_static) may hold flags a timed-out
// call left set: a wait that ran out leaves its tile's flags as they were.
static bool g_static_dirty[64];
static std::mutex g_static_mu;

int read_and_clear_device_status() {
    int v = 0;
    const int zero = 0;
    if (cudaDeviceSynchronize() != cudaSuccess) return WQ_ERR_CUDA;
    if (cudaMemcpyFromSymbol(&v, g_device_status, sizeof(int)) != cudaSuccess) return WQ_ERR_CUDA;
    if (cudaMemcpyToSymbol(g_device_status, &zero, sizeof(int)) != cudaSuccess) return WQ_ERR_CUDA;
    int dev = 0;
    if (v != 0 && cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < 64) {
        std::lock_guard<std::mutex> lock(g_static_mu);
        g_static_dirty[dev] = true;
    }
    return v;
}

namespace {

using namespace sm100;

constexpr int kBN = 128;        // weight rows per tile (MMA M)
constexpr int kBMMax = 256;     // activation rows of one MMA (its N), of an int4 tile and of a stream-K tile
constexpr int kBMMaxFp4 = 384;  // activation rows of an fp4 data-parallel tile: two MMAs of N = bm / 2
constexpr int kBK = 64;         // k per stage
// Stages of the ring, and TMEM weight buffers (as many: stage s and weight
// buffer s are freed by one commit).  A k-step's copy is issued when the MMAs
// kStages k-steps back complete, and it must land (~1,500 cycles) and be
// decoded (~600) before its own MMAs: with 4 stages that chain, not the
// tensor pipe, set the k-step of one-MMA fp4 tiles (~700 cycles against
// ~512 of MMA at 256 rows).  Their 32-column weight buffers leave TMEM room
// for 6 beside a 256-column accumulator (same GPU, bit-identical: 8192^3
// NVFP4 724 -> 654 (5 stages) -> 626 us; 128 x 8192 x 3072 17.2 -> 15.6
// us).  int4 (64-column buffers) and the two-MMA fp4 tiles (a 384-column
// accumulator) keep 4.
constexpr int kStagesMax = 6;
template <int FMT, bool SPLIT>
constexpr int kStagesOf = (FMT != kINT4 && !SPLIT) ? 6 : 4;
constexpr int kTmemCols = 512;
// TMEM columns per weight buffer (bf16 pairs of a row's 64 weights: int4 hi
// then lo, fp4 the weights alone) and the fp32 accumulator's columns before them
template <int FMT>
constexpr int kWColsOf = FMT == kINT4 ? 2 * kBK / 2 : kBK / 2;
template <int FMT, bool SPLIT>
constexpr int kAccColsOf = kTmemCols - kStagesOf<FMT, SPLIT> * kWColsOf<FMT>;
static_assert(kAccColsOf<kINT4, false> >= kBMMax && kAccColsOf<kNVFP4, false> >= kBMMax &&
                  kAccColsOf<kNVFP4, true> >= kBMMaxFp4,
              "TMEM budget");
constexpr int kDecodeSets = 3;                      // decode warp sets, taking the k-steps in turn
constexpr int kThreads = 64 + kDecodeSets * 128;    // producer, MMA, decode/epilogue warps
constexpr int kPTileBytes = kBN * kBK / 2;          // 4 KB of packed weights per stage
constexpr uint64_t kWaitNs = 2000000000ull;        // 2 s
constexpr uint64_t kDrainNs = 100000000ull;        // 0.1 s


struct TcArgs {
    const uint8_t* scales;   // prepacked weights: the record blocks
    const uint8_t* zeros;
    void* C;
    float* ws;          // stream-K partial sums [G][bm / 32][8][128] float4; null: one tile per CTA
    unsigned* flags;    // stream-K "partial of CTA c is ready" flags [G], zero between calls
    int M, N, K, group;
    int out_f32;
    int bm;             // activation rows per tile, a multiple of 32
    int bh;             // activation rows per MMA and per TMA box: bm, or bm / 2 above kBMMax
    int a_tile_bytes;   // bm * 128: the activation tile of a stage
    int stage_bytes;    // a_tile_bytes + packed tile; a multiple of 1024 (128-byte swizzle period)
    uint32_t idesc;     // instruction descriptor: M = 128, N = bh
    int nt_n;           // tiles along N; tile t covers rows (t % nt_n) * 128, activations (t / nt_n) * bm
    int nks;            // k-steps per tile
    long long units;    // tiles * nks
    int G;              // CTAs of a stream-K launch
    int csk;            // cluster split-K: CTAs per tile, one thread-block cluster (0: not this mode)
    int tma_store;      // whole tiles, plain bf16 C: staged in shared memory at stg_off, bulk tensor store (tmapC)
    int stg_off;        // the staging tile: beside the stage ring, or over it when each CTA has one tile
    int pdl;            // launched with programmatic dependent launch
    int kblocks;        // prepacked weights: 128-k blocks per row
    int vec_store;      // C rows 16-byte aligned and the store scratch allocated: vector stores of C
    int scr_off;        // byte offset of the decode warps' store scratch (2 KB each) in shared memory
    unsigned long long flag_wait_ns;   // bound of a stream-K owner's wait for a partial (0: give up at once)
    Epilogue epi;
};

struct __align__(8) TcShared {
    uint64_t full[kStagesMax];
    uint64_t empty[kStagesMax];
    uint64_t wfull[kStagesMax];
    uint64_t accfull;
    uint64_t accempty;
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};

__device__ __forceinline__ void record_timeout() { atomicExch(&g_device_status, WQ_ERR_DEVICE_TIMEOUT); }

// raw scale data of one row for one k-step (64 k):
//   nvfp4: the 4 e4m3 bytes of groups 4ks..4ks+3
//   mxfp4: the 2 e8m0 bytes of groups 2ks, 2ks+1
//   int4 : (bf16 scale | zero << 16) of the groups of k = 64ks and 64ks + 32
template <int FMT>
__device__ __forceinline__ uint2 tc_raw(const TcArgs& a, int n, int ks) {
    const int gpr = a.K / a.group;
    uint2 r;
    if constexpr (FMT == kNVFP4) {
        const uint8_t* p = a.scales + (size_t)n * gpr + 4 * ks;
        r.x = ldg_u8(p) | (ldg_u8(p + 1) << 8) | (ldg_u8(p + 2) << 16) | (ldg_u8(p + 3) << 24);
        r.y = 0;
    } else if constexpr (FMT == kMXFP4) {
        const uint8_t* p = a.scales + (size_t)n * gpr + 2 * ks;
        r.x = ldg_u8(p) | (ldg_u8(p + 1) << 8);
        r.y = 0;
    } else {
        const int g0 = (ks * kBK) / a.group, g1 = (ks * kBK + 32) / a.group;
        const uint16_t* s = reinterpret_cast<const uint16_t*>(a.scales) + (size_t)n * gpr;
        const uint8_t* z = a.zeros + (size_t)n * gpr;
        r.x = ldg_u16(s + g0) | (ldg_u8(z + g0) << 16);
        r.y = ldg_u16(s + g1) | (ldg_u8(z + g1) << 16);
    }
    return r;
}

// the decode key of word i (codes k = 8i .. 8i+7 of the k-step)
template <int FMT>
__device__ __forceinline__ void tc_keys(uint2 raw, GroupKey (&key)[4]) {
    if constexpr (FMT == kNVFP4) {
        const uint32_t h01 = e4m3x2_to_f16x2(raw.x & 0xFFFF), h23 = e4m3x2_to_f16x2(raw.x >> 16);
        const uint32_t hv[4] = {h01 & 0xFFFF, h01 >> 16, h23 & 0xFFFF, h23 >> 16};
#pragma unroll
        for (int j = 0; j < 4; ++j) {                 // words 2j, 2j+1
            key[j].mul = splat16(nvfp4_mul_from_f16(hv[j]));
            key[j].mul2 = 0x3F803F80u;
            key[j].zz = 0;
            key[j].zz2 = 0;
            key[j].two = false;
        }
    } else if constexpr (FMT == kMXFP4) {
        key[0] = key_mxfp4(raw.x & 0xFF);            // words 0..3
        key[1] = key_mxfp4((raw.x >> 8) & 0xFF);     // words 4..7
        key[2] = key[0];
        key[3] = key[1];
    } else {
        key[0] = key_int4(raw.x & 0xFFFF, raw.x >> 16);
        key[1] = key_int4(raw.y & 0xFFFF, raw.y >> 16);
        key[2] = key[0];
        key[3] = key[1];
    }
}

template <int FMT>
__device__ __forceinline__ const GroupKey& key_of_word(const GroupKey (&key)[4], int i) {
    if constexpr (FMT == kNVFP4) return key[i >> 1];
    else return key[i >> 2];
}

// One row's 64 weights of a k-step as bf16 pairs.  fp4 weights are exact in
// bf16 (at most 6 significant bits); int4 weights come as the exact split
// hi + lo (w2 = lo), so the tensor cores see the exact weight.
template <int FMT, bool TWO>
__device__ __forceinline__ void decode_row(const uint4& c0, const uint4& c1, const GroupKey (&key)[4],
                                           uint32_t (&w)[32], uint32_t (&w2)[32]) {
    const uint32_t wd[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        uint32_t p[4], r[4];
        if constexpr (FMT == kINT4) {
            int4_word_split<TWO>(wd[i], key_of_word<FMT>(key, i), p, r);
        } else {
            word_scaled<FMT, TWO>(wd[i], key_of_word<FMT>(key, i), p);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            w[4 * i + e] = p[e];
            if constexpr (FMT == kINT4) w2[4 * i + e] = r[e];
        }
    }
}

// The same raw scale data from a prepacked weight's record blocks (block
// (n / 16, ks / 2), row n % 16, half ks % 2):
//   nvfp4: the 4 bytes of groups 4ks..4ks+3 (the row's 8 bytes at 8 r)
//   mxfp4: the 2 bytes of groups 2ks, 2ks+1 (the row's 4 bytes at 4 r)
//   int4 : the row's bf16 scale (at 4 (r & 7) + 2 (r >> 3)) and zero point
//          (at 32 + 2 (r & 7) + (r >> 3)), returned as the input layout's
//          {bf16 scale | bf16 (128 + min(z, 128)) << 16}, bf16 (z - min(z, 128))
template <int FMT>
__device__ __forceinline__ uint2 tc_raw_pre(const TcArgs& a, int n, int ks) {
    const size_t blk = (size_t)(n >> 4) * a.kblocks + (ks >> 1);
    const int r = n & 15, h = ks & 1;
    uint2 raw;
    if constexpr (FMT == kNVFP4) {
        raw.x = ldg_u32(a.scales + blk * 128 + 8 * r + 4 * h);
        raw.y = 0;
    } else if constexpr (FMT == kMXFP4) {
        raw.x = ldg_u16(a.scales + blk * 64 + 4 * r + 2 * h);
        raw.y = 0;
    } else {
        const uint8_t* rec = a.scales + blk * 48;
        const uint32_t s = ldg_u16(rec + 4 * (r & 7) + 2 * (r >> 3));
        const uint32_t z = __ldg(rec + 32 + 2 * (r & 7) + (r >> 3));
        const uint32_t zc = min(z, 128u);
        raw.x = s | ((0x4300u + zc) << 16);   // 128 + zc, exact in bf16
        raw.y = z > 128u ? (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn((float)(z - zc))) : 0u;
    }
    return raw;
}

template <int FMT>
__device__ __forceinline__ void tc_keys_pre(uint2 raw, GroupKey (&key)[4]) {
    if constexpr (FMT == kINT4) {
        GroupKey k;
        k.mul = splat16(raw.x);
        k.mul2 = 0x3F803F80u;
        k.zz = splat16(raw.x >> 16);
        k.zz2 = splat16(raw.y);
        k.two = (raw.y & 0xFFFFu) != 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) key[j] = k;
    } else {
        tc_keys<FMT>(raw, key);   // the same bytes as the input layout's
    }
}

// One row's 64 weights of a k-step from the prepacked layout: the row's two
// 16-byte chunks hold the words w0 w4 w1 w5 | w2 w6 w3 w7; int4 words hold
// natural k pairs in nibbles (s, s + 4).
template <int FMT, bool TWO>
__device__ __forceinline__ void decode_row_pre(const uint4& c0, const uint4& c1, const GroupKey (&key)[4],
                                               uint32_t (&w)[32], uint32_t (&w2)[32]) {
    const uint32_t wd[8] = {c0.x, c0.z, c1.x, c1.z, c0.y, c0.w, c1.y, c1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        uint32_t p[4], r[4];
        if constexpr (FMT == kINT4) {
            int4_word_split_pairs<TWO>(wd[i], key_of_word<FMT>(key, i), p, r);
        } else {
            word_scaled<FMT, TWO>(wd[i], key_of_word<FMT>(key, i), p);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            w[4 * i + e] = p[e];
            if constexpr (FMT == kINT4) w2[4 * i + e] = r[e];
        }
    }
}

// ---------------------------------------------------------------------------
// work split
// ---------------------------------------------------------------------------
// Whole-tile launch (no workspace): G = min(tiles, SMs) persistent CTAs; CTA
// c computes tiles c, c + G, c + 2G, ... all k-steps, its stage ring and
// weight buffers running on from one tile to the next, so a tile's first
// loads and decode overlap the previous tile's epilogue (measured on the same
// GPU against one CTA per tile: 2-5 % faster on every shape).
// Stream-K launch: the tiles * nks (tile, k-step) units are cut into G equal
// contiguous ranges, one per CTA; a tile met by several CTAs is finished by
// the CTA holding its last k-step (the owner), which adds the fp32 partial
// sums the others left in the workspace, in increasing CTA order.
// Cluster split-K launch (few tiles, no workspace): each tile is one cluster
// of S = csk CTAs, CTA c taking the (c mod S)-th of tile c / S's k-steps in
// equal contiguous parts; the CTAs add up their partial sums through
// distributed shared memory (tc_cluster_reduce).
__device__ __forceinline__ long long unit_start(const TcArgs& a, int c) {
    return a.ws ? (long long)c * a.units / a.G : (long long)c * a.nks;
}

// CTA whose range holds unit u (stream-K)
__device__ __forceinline__ int cta_of_unit(const TcArgs& a, long long u) {
    int c = (int)((u * a.G) / a.units);
    while (c + 1 < a.G && unit_start(a, c + 1) <= u) ++c;
    while (c > 0 && unit_start(a, c) > u) --c;
    return c;
}

// Segment i of CTA c in processing order: the last segment first when it
// does not end its tile (its partial is then written before anyone waits on
// it), then the tile-ending segments in order.  Every role of the CTA walks
// the same sequence.  Returns false past the last segment.
__device__ __forceinline__ bool get_seg(const TcArgs& a, int c, int i, int& tile, int& kb, int& ke) {
    if (a.csk) {   // cluster split-K: one segment
        if (i > 0) return false;
        const int r = c % a.csk;
        tile = c / a.csk;
        kb = (int)((long long)r * a.nks / a.csk);
        ke = (int)((long long)(r + 1) * a.nks / a.csk);
        return true;
    }
    if (!a.ws) {   // whole tiles: c, c + G, c + 2G, ...
        const long long t = (long long)c + (long long)i * a.G;
        if (t * a.nks >= a.units) return false;
        tile = (int)t;
        kb = 0;
        ke = a.nks;
        return true;
    }
    const long long u0 = unit_start(a, c), u1 = unit_start(a, c + 1);
    if (u1 <= u0) return false;
    const long long nks = a.nks;
    const int t_first = (int)(u0 / nks), t_last = (int)((u1 - 1) / nks);
    const bool last_partial = (u1 % nks) != 0;
    if (last_partial) {
        if (i == 0) {
            tile = t_last;
            kb = (int)((u0 > t_last * nks ? u0 : t_last * nks) - t_last * nks);
            ke = (int)(u1 - t_last * nks);
            return true;
        }
        --i;
    }
    const int t = t_first + i;
    if (t > (last_partial ? t_last - 1 : t_last)) return false;
    tile = t;
    kb = (int)((u0 > t * nks ? u0 : t * nks) - t * nks);
    ke = (int)nks;
    return true;
}

// the fp32 partial of CTA `slot`: columns 32 ch + 4 j .. + 3 of row `row`,
// laid out [slot][ch][j][row] in float4 so that a warp's 32 rows of one
// (ch, j) are one contiguous 512-byte run
__device__ __forceinline__ float4* partial_ptr(const TcArgs& a, int slot, int ch, int j, int row) {
    return reinterpret_cast<float4*>(a.ws) + (((size_t)slot * (a.bm / 32) + ch) * 8 + j) * kBN + row;
}

// A limit of 0 gives up at once without reading the flag (the host sets it
// only to run the failure path in tests; see WQ_TC_FLAG_WAIT_NS).
__device__ __forceinline__ bool wait_flag(const unsigned* f, volatile int* abort, uint64_t limit_ns) {
    if (limit_ns == 0) {
        *abort = 1;
        return false;
    }
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 0;; ++i) {
        unsigned v;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(f) : "memory");
        if (v) return true;
        if ((i & 15) == 15) {
            if (*abort) return false;
            if (globaltimer_ns() - t0 > limit_ns) {
                *abort = 1;
                return false;
            }
        }
        __nanosleep(32);
    }
}

// Cluster split-K: the cluster's CTA of rank r adds up, for its share of the
// tile's column groups (4 activation rows x 128 weight rows each, group p =
// ch * 8 + j of the [ch][j][row] float4 partials), the S partial sums in
// increasing rank order -- a fixed order: the same inputs give the same bits
// -- and stores them, through the fused epilogue where there is one.  t: the
// decode warps' thread index; 128 consecutive threads take one group, one
// thread per weight row, so a gate row's up row (row + 8) is in its warp.
template <bool EPI>
__device__ __forceinline__ void tc_cluster_reduce(const TcArgs& a, uint8_t* smem, int t) {
    constexpr int kMaxS = 8;
    const int S = a.csk, r = (int)cluster_ctarank(), tile = (int)blockIdx.x / S;
    const int n0 = (tile % a.nt_n) * kBN, m0 = (tile / a.nt_n) * a.bm;
    const int row = t & (kBN - 1), n = n0 + row;
    const int ngroups = a.bm / 4;
    const int p0 = r * ngroups / S, p1 = (r + 1) * ngroups / S;
    const uint32_t base = smem_u32(smem);
    uint32_t src[kMaxS];
#pragma unroll
    for (int s = 0; s < kMaxS; ++s) src[s] = s < S ? mapa_shared(base, (uint32_t)s) : 0u;
    // A group's S loads go out together, and the thread's next group's loads
    // before this group's sums and stores (same GPU, bit-identical: int4
    // M = 128 k / v 10.72 -> 10.53 us, q 12.75 -> 12.52 us).  Tried and
    // slower: each CTA pushing its partials into the owners' shared memory
    // (remote stores, one cluster barrier, local sums): k / v 14.8 us.
    auto load = [&](int p, float4 (&x)[kMaxS]) {
        const uint32_t off = ((uint32_t)p * kBN + row) * 16u;
#pragma unroll
        for (int s = 0; s < kMaxS; ++s)
            if (s < S) x[s] = ld_dsmem_f4(src[s] + off);
    };
    float4 cur[kMaxS], nxt[kMaxS];
    int p = p0 + (t >> 7);
    if (p < p1) load(p, cur);
    for (; p < p1; p += kDecodeSets) {
        if (p + kDecodeSets < p1) load(p + kDecodeSets, nxt);
        float f[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int s = 0; s < kMaxS; ++s) {   // rank order
            if (s < S) {
                f[0] += cur[s].x;
                f[1] += cur[s].y;
                f[2] += cur[s].z;
                f[3] += cur[s].w;
            }
        }
#pragma unroll
        for (int s = 0; s < kMaxS; ++s) cur[s] = nxt[s];
        const int mb = m0 + 4 * p;
        if constexpr (EPI) {
            const bool mine = n < a.N && !(a.epi.gated && (row & 8));
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float u = a.epi.gated ? __shfl_xor_sync(0xffffffffu, f[e], 8) : 0.f;
                if (mine && mb + e < a.M) store_epilogue(a.epi, a.C, a.out_f32, a.N, mb + e, n, f[e], u);
            }
        } else if (n < a.N) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                if (mb + e < a.M) {
                    const size_t o = (size_t)(mb + e) * a.N + n;
                    if (a.out_f32) static_cast<float*>(a.C)[o] = f[e];
                    else static_cast<__nv_bfloat16*>(a.C)[o] = __float2bfloat16_rn(f[e]);
                }
            }
        }
    }
}

// PRE: the weights are in the prepacked layout (tmapP a 3-D map of its code
// blocks: 512-byte half blocks x 2 per 128-k block x row blocks; scales
// from its record blocks).  EPI: the fused epilogue; the plain instance
// carries no epilogue code at all.  SPLIT (fp4): tiles of bm = 2 bh rows, two
// MMAs per 16-k slice.  It is a template parameter, not a runtime test: a
// never-taken branch around the second MMA in the issuing loop cost the
// one-MMA tiles 27 % (8192^3 NVFP4 prepacked, same GPU: 776 -> 983 us).
template <int FMT, bool PRE, bool EPI, bool SPLIT>
__global__ void __launch_bounds__(kThreads, 1)
    tc_kernel(const __grid_constant__ CUtensorMap tmapA, const __grid_constant__ CUtensorMap tmapP, const TcArgs a,
              const __grid_constant__ CUtensorMap tmapC) {
    static_assert(!(SPLIT && FMT == kINT4), "int4 tiles use one MMA per slice and its residual");
    constexpr int kStages = kStagesOf<FMT, SPLIT>, kWBufs = kStages;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // stages 1024-byte aligned (the 128-byte swizzle pattern repeats every 1 KB)
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int kStageBytes = a.stage_bytes, kATileBytes = a.a_tile_bytes;
    TcShared& sh = *reinterpret_cast<TcShared*>(smem + kStages * kStageBytes);
    volatile int* abort = &sh.abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cta = blockIdx.x;
    const int nks = a.nks;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&sh.full[s]), 1);
            mbar_init(smem_u32(&sh.empty[s]), 1);
        }
        for (int b = 0; b < kWBufs; ++b) {
            mbar_init(smem_u32(&sh.wfull[b]), 128);
        }
        mbar_init(smem_u32(&sh.accfull), 1);
        mbar_init(smem_u32(&sh.accempty), kDecodeSets * 128);
        mbar_init(smem_u32(&sh.drain), 1);
        sh.abort = 0;
        fence_mbarrier_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&sh.tmem_base), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh.tmem_base;
    // Programmatic dependent launch (no-ops otherwise).  This grid reads A
    // only after its predecessor has completed (the producer's wait below),
    // and every write it makes to global memory -- C, stream-K partials and
    // flags, the bulk stores -- follows from copies the producer issued after
    // that wait.  The next grid may be scheduled once every CTA has begun its
    // last segment (the producer's trigger below): at once in a one-wave
    // launch, late in a longer one.

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            prefetch_tensormap(&tmapA);
            prefetch_tensormap(&tmapP);
            if (a.pdl) grid_dependency_wait();
            int g = 0;   // k-steps issued so far (the stage ring runs across segments)
            bool ok = true;
            int tile, kb, ke;
            for (int i = 0; ok && get_seg(a, cta, i, tile, kb, ke); ++i) {
                const int n0 = (tile % a.nt_n) * kBN, m0 = (tile / a.nt_n) * a.bm;
                if (a.pdl) {
                    int t2, kb2, ke2;
                    if (!get_seg(a, cta, i + 1, t2, kb2, ke2)) grid_dependents_launch();   // the last segment
                }
                for (int k = kb; k < ke; ++k, ++g) {
                    const int s = g % kStages;
                    const uint32_t ph = (g / kStages) & 1;
                    if (!mbar_wait_bounded(smem_u32(&sh.empty[s]), ph ^ 1, abort, kWaitNs)) {
                        record_timeout();
                        ok = false;
                        break;
                    }
                    uint8_t* st = smem + s * kStageBytes;
                    const uint32_t fb = smem_u32(&sh.full[s]);
                    mbar_arrive_expect_tx(fb, kStageBytes);
                    tma_load_2d(smem_u32(st), &tmapA, fb, k * kBK, m0);
                    if constexpr (SPLIT) tma_load_2d(smem_u32(st + a.bh * 128), &tmapA, fb, k * kBK, m0 + a.bh);
                    if constexpr (PRE) tma_load_3d(smem_u32(st + kATileBytes), &tmapP, fb, 0, k, n0 >> 4);
                    else tma_load_2d(smem_u32(st + kATileBytes), &tmapP, fb, k * (kBK / 2), n0);
                }
            }
            // never leave the CTA with copies in flight
            for (int k = (g > kStages ? g - kStages : 0); k < g; ++k)
                mbar_wait_timeout(smem_u32(&sh.full[k % kStages]), (k / kStages) & 1, kDrainNs);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            int g = 0;
            bool ok = true;
            int tile, kb, ke;
            for (int i = 0; ok && get_seg(a, cta, i, tile, kb, ke); ++i) {
                // the epilogue of the previous segment has read the accumulator
                if (i > 0 && !mbar_wait_bounded(smem_u32(&sh.accempty), (i - 1) & 1, abort, kWaitNs)) {
                    record_timeout();
                    break;
                }
                for (int k = kb; k < ke; ++k, ++g) {
                    const int s = g % kStages, b = g % kWBufs;
                    const uint32_t phb = (g / kWBufs) & 1;
                    // One wait, for the decoded weights: the decode set waited
                    // for this k-step's stage copy (full[s]) before decoding and
                    // arrived on wfull[b] after, so the copy is ordered before
                    // this acquire through its arrivals.  This thread is the
                    // pipeline's critical path -- a satisfied mbarrier wait costs
                    // it ~120 cycles, against ~590 of MMA in a k-step -- and
                    // dropping the second wait measured (same GPU): MXFP4
                    // 2048 x 3072^2 32.1 -> 30.4 us, int4 128 x 128256 x 3072
                    // 187 -> 176 us, 8192^3 NVFP4 761 -> 748 us.
                    if (!mbar_wait_bounded(smem_u32(&sh.wfull[b]), phb, abort, kWaitNs)) {
                        record_timeout();
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // The descriptors are formed once per k-step and stepped by
                    // 32 bytes (2 in the 16-byte address field, which cannot
                    // carry below 256 KB) per 16-k slice: the issuing thread's
                    // work per MMA is on the critical path (same GPU: 8192^3
                    // NVFP4 776 -> 764 us, the prefill 33.5 -> 32.8 us against
                    // a descriptor formed per MMA).
                    const uint32_t a_addr = smem_u32(smem + s * kStageBytes);
                    const uint64_t bdesc0 = smem_desc_sw128_kmajor(a_addr);
                    const uint64_t bdesc1 = SPLIT ? smem_desc_sw128_kmajor(a_addr + a.bh * 128) : 0;
                    const uint32_t wcol0 = tmem + kAccColsOf<FMT, SPLIT> + b * kWColsOf<FMT>;
                    const uint32_t acc0 = k != kb ? 1u : 0u;
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk) {
                        const uint32_t acc = kk ? 1u : acc0;
                        mma_ts_f16(tmem, wcol0 + kk * 8, bdesc0 + 2 * kk, a.idesc, acc);
                        // the tile's second half: the same weights, activation rows
                        // bh.., accumulator columns bh..
                        if constexpr (SPLIT) mma_ts_f16(tmem + a.bh, wcol0 + kk * 8, bdesc1 + 2 * kk, a.idesc, acc);
                    }
                    if constexpr (FMT == kINT4) {
#pragma unroll
                        for (int kk = 0; kk < kBK / 16; ++kk)   // the residuals, after the leading terms
                            mma_ts_f16(tmem, wcol0 + 32 + kk * 8, bdesc0 + 2 * kk, a.idesc, 1);
                    }
                    // one commit frees both stage s and weight buffer b == s: a
                    // second commit per k-step to a barrier of its own measured
                    // 2-4 % slower (8192^3 NVFP4 775 -> 760 us without it)
                    tc_commit(smem_u32(&sh.empty[s]));
                }
                if (ok) tc_commit(smem_u32(&sh.accfull));
            }
            // every MMA of this thread has completed before the CTA tears down
            tc_commit(smem_u32(&sh.drain));
            mbar_wait_timeout(smem_u32(&sh.drain), 0, kDrainNs);
        }
    } else {
        // ---------------- decode, then epilogue (warps 2..) ----------------
        // set `dset` decodes the k-steps g = dset (mod kDecodeSets) of the
        // CTA's running k-step count; each set has one warp per TMEM lane
        // quarter.  Failures do not leave the segment loop: every epilogue
        // thread passes the same named barriers.
        const int dset = (warp - 2) >> 2;
        const int q = warp & 3;                 // TMEM lane quarter this warp may access
        const int row = q * 32 + lane;          // weight row inside the tile
        const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);
        constexpr int D = 4;                    // this set's k-steps of scales in flight
        constexpr int KS = kDecodeSets;
        // Decode k-step gg (running count) from its scale keys into weight
        // buffer gg mod kWBufs; false once a wait gave up (decided per warp:
        // the TMEM store is warp-collective).
        auto decode_kstep = [&](int gg, const GroupKey (&key)[4]) -> bool {
            const int s = gg % kStages, b = gg % kWBufs;
            const uint32_t ph = (gg / kStages) & 1, phb = (gg / kWBufs) & 1;
            // Weight buffer first, stage second.  A set never waits on
            // the stage phase of k-step gg - kStages (another set's), so
            // on its own the parity test on full[s] could match that
            // older phase when copies land out of order, and the decode
            // would read the stage before this k-step's copy.  The MMA
            // of k-step gg - kWBufs has consumed every copy up to it,
            // that of gg - kStages included, so the full[s] wait after
            // it can only match this k-step's phase.
            static_assert(kWBufs == kStages,
                          "weight buffer b is freed by the commit that frees stage b; the "
                          "weight-buffer wait must imply the older stage phase");
            const bool got = mbar_wait_bounded(smem_u32(&sh.empty[b]), phb ^ 1, abort, kWaitNs) &&
                             mbar_wait_bounded(smem_u32(&sh.full[s]), ph, abort, kWaitNs);
            if (!__all_sync(0xffffffffu, got)) {
                if (!got) record_timeout();
                return false;
            }
            tc_fence_after();
            // this row's 32 packed bytes; 32-byte swizzle: chunk c of row r
            // sits at 32 r + 16 (c ^ ((r >> 2) & 1))
            const uint8_t* prow = smem + s * kStageBytes + kATileBytes + row * 32;
            const int x = (row >> 2) & 1;
            const uint4 lo = *reinterpret_cast<const uint4*>(prow + 16 * x);
            const uint4 hi = *reinterpret_cast<const uint4*>(prow + 16 * (x ^ 1));
            uint32_t w[32], w2[32];
            bool two = false;
            if constexpr (FMT != kNVFP4) two = __any_sync(0xffffffffu, key[0].two || key[1].two);
            if constexpr (PRE) {
                if (two) decode_row_pre<FMT, true>(lo, hi, key, w, w2);
                else decode_row_pre<FMT, false>(lo, hi, key, w, w2);
            } else {
                if (two) decode_row<FMT, true>(lo, hi, key, w, w2);
                else decode_row<FMT, false>(lo, hi, key, w, w2);
            }
            const uint32_t wbuf = lane_base + kAccColsOf<FMT, SPLIT> + b * kWColsOf<FMT>;
            if constexpr (FMT == kINT4)
                tmem_st2_32x32b_x32_sync(wbuf, w, wbuf + 32, w2);
            else
                tmem_st_32x32b_x32_sync(wbuf, w);
            tc_fence_before();
            mbar_arrive(smem_u32(&sh.wfull[b]));
            return true;
        };
        auto raw_of = [&](int nrow, int k) -> uint2 {
            return PRE ? tc_raw_pre<FMT>(a, nrow, k) : tc_raw<FMT>(a, nrow, k);
        };
        auto keys_of = [&](const uint2& r, GroupKey (&key)[4]) {
            if constexpr (PRE) tc_keys_pre<FMT>(r, key);
            else tc_keys<FMT>(r, key);
        };
        int g = 0;
        bool ok = true;
        bool ahead = false;   // this set's first k-step of the segment was decoded during the previous one
        int tile, kb, ke;
        for (int i = 0; get_seg(a, cta, i, tile, kb, ke); ++i) {
            const int n0 = (tile % a.nt_n) * kBN, m0 = (tile / a.nt_n) * a.bm;
            const int n = n0 + row;
            const int nc = n < a.N ? n : a.N - 1;   // rows past N decode row N-1 (never stored)
            const int g0 = g;
            // this set's first k-step of the segment still to decode
            const int k1 = kb + ((dset - g0) % KS + KS) % KS + (ahead ? KS : 0);
            uint2 raw[D];
#pragma unroll
            for (int d = 0; d < D; ++d)
                if (k1 + d * KS < ke) raw[d] = raw_of(nc, k1 + d * KS);
            for (int kk0 = k1; kk0 < ke && ok; kk0 += D * KS) {
#pragma unroll
                for (int d = 0; d < D; ++d) {
                    const int k = kk0 + d * KS;
                    if (k < ke && ok) {
                        GroupKey key[4];
                        keys_of(raw[d], key);
                        if (k + D * KS < ke) raw[d] = raw_of(nc, k + D * KS);
                        if (!decode_kstep(g0 + (k - kb), key)) {
                            ok = false;
                            break;
                        }
                    }
                }
            }
            g = g0 + (ke - kb);
            // Look-ahead: this set's first k-step of the next segment, decoded
            // before this segment's epilogue.  Its weight buffer is freed by
            // MMAs of this segment, not by the epilogue, so the issuer finds
            // the next tile's first weights ready once the accumulator is
            // released (per-k-step stamps: the issuer had waited ~4,500 cycles
            // for them at every tile boundary of int4 2048 x 128256 x 3072).
            ahead = false;
            {
                int tile2, kb2, ke2;
                if (ok && get_seg(a, cta, i + 1, tile2, kb2, ke2)) {
                    const int k1n = kb2 + ((dset - g) % KS + KS) % KS;
                    if (k1n < ke2) {
                        const int n2 = (tile2 % a.nt_n) * kBN + row;
                        GroupKey key2[4];
                        keys_of(raw_of(n2 < a.N ? n2 : a.N - 1, k1n), key2);
                        ok = decode_kstep(g + (k1n - kb2), key2);
                        ahead = true;
                    }
                }
            }

            // ---------------- epilogue of the segment ----------------
            // (cluster split-K: no CTA owns its tile; all add up on chip later)
            const bool owner = ke == nks && !a.csk;
            const int cfirst = (owner && a.ws) ? cta_of_unit(a, (long long)tile * nks) : cta;
            if (ok) ok = mbar_wait_bounded(smem_u32(&sh.accfull), i & 1, abort, kWaitNs);
            ok = __all_sync(0xffffffffu, ok);
            if (a.tma_store) {
                // Plain bf16 C of a whole tile: the accumulator to bf16 in the
                // staging tile [bm][128] (a warp's 32 weight rows of one
                // activation row are 64 contiguous bytes), the accumulator
                // released, then one bulk tensor store by one thread, which
                // the next tile's work overlaps.  Same GPU, against scalar
                // stores from the decode warps: 8192^3 NVFP4 747 -> 727 us,
                // int4 2048 x 8192 x 3072 129.3 -> 121.3 us, MXFP4 2048 x
                // 3072^2 30.4 -> 29.8 us.
                if (warp == 2 && lane == 0) bulk_wait_read0();   // the previous tile's store has read the staging
                asm volatile("bar.sync 1, %0;" ::"n"(kDecodeSets * 128) : "memory");
                if (!ok && lane == 0) record_timeout();
                tc_fence_after();
                __nv_bfloat16* stg = reinterpret_cast<__nv_bfloat16*>(smem + a.stg_off);
#pragma unroll 1
                for (int ch = dset; ch < a.bm / 32 && ok; ch += kDecodeSets) {
                    uint32_t v[32];
                    tmem_ld_32x32b_x32_sync(lane_base + ch * 32, v);
#pragma unroll
                    for (int j = 0; j < 32; ++j) stg[(ch * 32 + j) * kBN + row] = __float2bfloat16_rn(__uint_as_float(v[j]));
                }
                tc_fence_before();
                mbar_arrive(smem_u32(&sh.accempty));
                fence_proxy_async_smem();
                asm volatile("bar.sync 1, %0;" ::"n"(kDecodeSets * 128) : "memory");
                if (warp == 2 && lane == 0 && ok) {
                    // boxes of bh rows: two for a two-MMA tile
                    tma_store_2d(&tmapC, smem_u32(stg), n0, m0);
                    if (a.bh < a.bm) tma_store_2d(&tmapC, smem_u32(stg) + (uint32_t)a.bh * kBN * 2, n0, m0 + a.bh);
                    bulk_commit();
                }
                continue;
            }
            if (ok && owner) {
                // the lanes poll the contributors' flags together (one memory
                // round trip per pass, not per contributor)
                for (int c0 = cfirst; c0 < cta && ok; c0 += 32) {
                    const int c2 = c0 + lane;
                    const bool mine = c2 < cta;
                    const bool got = !mine || wait_flag(a.flags + c2, abort, a.flag_wait_ns);
                    ok = __all_sync(0xffffffffu, got);
                }
            }
            // the warp's reads of the partials below are ordered after the
            // lanes' acquires of their flags
            __syncwarp();
            if (!ok && lane == 0) record_timeout();
            tc_fence_after();
#pragma unroll 1
            for (int ch = dset; ch < a.bm / 32; ch += kDecodeSets) {
                uint32_t v[32];
                if (!ok) continue;
                tmem_ld_32x32b_x32_sync(lane_base + ch * 32, v);
                if (!owner) {
                    // a tile this CTA starts but does not end: its partial sums,
                    // to the workspace (stream-K) or, cluster split-K, to its own
                    // shared memory over the stage ring ([ch][j][row] float4;
                    // every MMA, and with it every copy into the ring, has
                    // completed once accfull has) for tc_cluster_reduce
                    float4* part = reinterpret_cast<float4*>(smem) + (size_t)ch * 8 * kBN + row;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const float4 x = make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                                                     __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3]));
                        if (a.csk) part[j * kBN] = x;
                        else __stcg(partial_ptr(a, cta, ch, j, row), x);
                    }
                    continue;
                }
                float f[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) f[j] = __uint_as_float(v[j]);
                // the contributors' partials in increasing CTA order, two at a
                // time: their 16 loads are in flight together, the sums keep
                // the order (a tile of M = 128 rows split over ~19 CTAs waited
                // ~18 L2 round trips per chunk one partial at a time)
                auto add4 = [&](const float4 (&t)[8]) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        f[4 * j] += t[j].x;
                        f[4 * j + 1] += t[j].y;
                        f[4 * j + 2] += t[j].z;
                        f[4 * j + 3] += t[j].w;
                    }
                };
                int c2 = cfirst;
                for (; c2 + 1 < cta; c2 += 2) {
                    float4 t0[8], t1[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        t0[j] = __ldcg(partial_ptr(a, c2, ch, j, row));
                        t1[j] = __ldcg(partial_ptr(a, c2 + 1, ch, j, row));
                    }
                    add4(t0);
                    add4(t1);
                }
                if (c2 < cta) {
                    float4 t0[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) t0[j] = __ldcg(partial_ptr(a, c2, ch, j, row));
                    add4(t0);
                }
                const int mb = m0 + ch * 32;
                if constexpr (EPI) {
                    // gated: the up row of this gate row is row + 8, held by lane + 8
                    const bool mine = n < a.N && !(a.epi.gated && (row & 8));
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float u = a.epi.gated ? __shfl_xor_sync(0xffffffffu, f[j], 8) : 0.f;
                        if (mine && mb + j < a.M) store_epilogue(a.epi, a.C, a.out_f32, a.N, mb + j, n, f[j], u);
                    }
                } else if (a.vec_store) {
                    // This warp's 32 weight rows x 32 activation rows through its
                    // 2 KB of shared memory, transposed, then out as 16-byte
                    // pieces of C rows: 4 vector stores per lane where 32 scalar
                    // ones wrote 64-byte pieces.
                    const int nb = n - lane;                        // the warp's first weight row
                    uint8_t* scr = smem + a.scr_off + (warp - 2) * 2048;
                    if (a.out_f32) {
                        float* t = reinterpret_cast<float*>(scr);   // [16 activation rows][32]
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
#pragma unroll
                            for (int j = 0; j < 16; ++j) t[j * 32 + lane] = f[16 * h + j];
                            __syncwarp();
#pragma unroll
                            for (int r = 0; r < 4; ++r) {
                                const int v = r * 32 + lane, row = v >> 3, c = (v & 7) * 4;
                                const int m = mb + 16 * h + row;
                                const float4 x = *reinterpret_cast<const float4*>(t + row * 32 + c);
                                if (m < a.M && nb + c < a.N)
                                    *reinterpret_cast<float4*>(static_cast<float*>(a.C) + (size_t)m * a.N + nb + c) = x;
                            }
                            __syncwarp();
                        }
                    } else {
                        __nv_bfloat16* t = reinterpret_cast<__nv_bfloat16*>(scr);   // [32 activation rows][32]
#pragma unroll
                        for (int j = 0; j < 32; ++j) t[j * 32 + lane] = __float2bfloat16_rn(f[j]);
                        __syncwarp();
#pragma unroll
                        for (int r = 0; r < 4; ++r) {
                            const int v = r * 32 + lane, row = v >> 2, c = (v & 3) * 8;
                            const int m = mb + row;
                            const uint4 x = *reinterpret_cast<const uint4*>(t + row * 32 + c);
                            if (m < a.M && nb + c < a.N)
                                *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.C) + (size_t)m * a.N + nb + c) = x;
                        }
                        __syncwarp();
                    }
                } else if (n < a.N) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        if (mb + j < a.M) {
                            const size_t o = (size_t)(mb + j) * a.N + n;
                            if (a.out_f32) static_cast<float*>(a.C)[o] = f[j];
                            else static_cast<__nv_bfloat16*>(a.C)[o] = __float2bfloat16_rn(f[j]);
                        }
                    }
                }
            }
            // the accumulator may be overwritten by the next segment's MMAs
            tc_fence_before();
            mbar_arrive(smem_u32(&sh.accempty));
            if (a.ws && (!owner || cfirst < cta)) {
                // every epilogue thread is done with the partials it writes / reads
                asm volatile("bar.sync 1, %0;" ::"n"(kDecodeSets * 128) : "memory");
                if (warp == 2 && lane == 0 && ok) {
                    if (!owner) {
                        __threadfence();
                        asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(a.flags + cta), "r"(1u) : "memory");
                    } else {
                        // consumed: leave the flags zero for the next call
                        for (int c2 = cfirst; c2 < cta; ++c2)
                            asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(a.flags + c2), "r"(0u) : "memory");
                    }
                }
            }
        }
    }

    if (a.tma_store && warp == 2 && lane == 0) bulk_wait0();   // the stores complete before the CTA exits (and its smem goes)
    if (a.csk) {
        // every role of every CTA of the tile's cluster passes both barriers,
        // a failed wait included (its partial is then garbage, its status
        // recorded)
        cluster_sync_all();   // each CTA's partial is in its shared memory
        if (warp >= 2) tc_cluster_reduce<EPI>(a, smem, (int)threadIdx.x - 64);
        cluster_sync_all();   // no CTA leaves while another still reads its partial
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <int FMT, bool PRE>
int launch_fmt(const CUtensorMap& ta, const CUtensorMap& tp, const TcArgs& args, dim3 grid, size_t smem,
               cudaStream_t stream, const CUtensorMap& tcm) {
    const bool epi = args.epi.bias || args.epi.residual || args.epi.gated;
    auto kern = epi ? tc_kernel<FMT, PRE, true, false> : tc_kernel<FMT, PRE, false, false>;
    if constexpr (FMT != kINT4) {
        if (args.bh < args.bm) kern = epi ? tc_kernel<FMT, PRE, true, true> : tc_kernel<FMT, PRE, false, true>;
    }
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return WQ_ERR_CUDA;
    if (args.csk || args.pdl) {
        // one cluster of csk CTAs per tile; programmatic dependent launch
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = grid;
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = stream;
        cudaLaunchAttribute attr[2];
        unsigned na = 0;
        if (args.csk) {
            attr[na].id = cudaLaunchAttributeClusterDimension;
            attr[na].val.clusterDim.x = (unsigned)args.csk;
            attr[na].val.clusterDim.y = 1;
            attr[na].val.clusterDim.z = 1;
            ++na;
        }
        if (args.pdl) {
            attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[na].val.programmaticStreamSerializationAllowed = 1;
            ++na;
        }
        cfg.attrs = attr;
        cfg.numAttrs = na;
        return cudaLaunchKernelEx(&cfg, kern, ta, tp, args, tcm) == cudaSuccess ? WQ_OK : WQ_ERR_CUDA;
    }
    kern<<<grid, kThreads, smem, stream>>>(ta, tp, args, tcm);
    return cudaGetLastError() == cudaSuccess ? WQ_OK : WQ_ERR_CUDA;
}

// Clusters of S CTAs of the tensor-core kernel (one CTA per SM) with `smem`
// bytes of dynamic shared memory that the device can hold at once; cached.
int csk_max_clusters(int S, size_t smem) {
    static std::mutex mu;
    static long long keys[64];
    static int vals[64];
    static int n = 0;
    int dev = 0;
    cudaGetDevice(&dev);
    const long long key = ((long long)dev << 40) | ((long long)S << 32) | (long long)smem;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < n; ++i)
        if (keys[i] == key) return vals[i];
    auto kern = tc_kernel<kINT4, true, false, false>;
    int clusters = 0;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) == cudaSuccess) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)S, 1, 1);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)S;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) != cudaSuccess) clusters = 0;
    }
    cudaGetLastError();   // a refused query leaves no error behind
    if (n < 64) {
        keys[n] = key;
        vals[n] = clusters;
        ++n;
    }
    return clusters;
}

// Failure-path self test: one thread waits, with a short wall-time bound, on
// an mbarrier that nothing will ever arrive on, then records the timeout the
// way the GEMM kernels do.  No GPU is hung and the context stays usable.
__global__ void timeout_selftest_kernel(unsigned long long limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(smem_u32(&bar), 1);
        fence_mbarrier_init();
        if (!mbar_wait_bounded(smem_u32(&bar), 0, &abort_flag, limit_ns)) record_timeout();
    }
}

}  // namespace

// ---------------------------------------------------------------------------
// host side: tensor maps through the driver entry point (no libcuda link)
// ---------------------------------------------------------------------------
// WQ_DEBUG=1 in the environment prints why a call was refused
bool debug_on() { return getenv("WQ_DEBUG") != nullptr; }   // read per call: tests switch it on and off

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        const cudaError_t e =
            cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
        if (e == cudaSuccess && q == cudaDriverEntryPointSuccess) fn = reinterpret_cast<EncodeTiledFn>(p);
        else if (debug_on())
            fprintf(stderr, "wq: driver entry point lookup failed (%s, %d)\n", cudaGetErrorString(e), (int)q);
    });
    return fn;
}

bool encode_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
               uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) {
        if (debug_on()) fprintf(stderr, "wq: cuTensorMapEncodeTiled entry point not found\n");
        return false;
    }
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS && debug_on())
        fprintf(stderr, "wq: cuTensorMapEncodeTiled failed (%d): dims %llu x %llu, stride %llu, box %u x %u\n",
                (int)r, (unsigned long long)inner, (unsigned long long)outer, (unsigned long long)row_bytes,
                box_inner, box_outer);
    return r == CUDA_SUCCESS;
}

// 3-D tiled map, no swizzle: dims / box inner-first, strides of dims 1, 2
static bool encode_3d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, const uint64_t (&dims)[3],
                      const uint64_t (&strides)[2], const uint32_t (&box)[3]) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t d[3] = {dims[0], dims[1], dims[2]};
    const cuuint64_t st[2] = {strides[0], strides[1]};
    const cuuint32_t b[3] = {box[0], box[1], box[2]};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = fn(map, dt, 3, const_cast<void*>(base), d, st, b, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS && debug_on())
        fprintf(stderr, "wq: cuTensorMapEncodeTiled (3-D) failed (%d): dims %llu x %llu x %llu\n", (int)r,
                (unsigned long long)dims[0], (unsigned long long)dims[1], (unsigned long long)dims[2]);
    return r == CUDA_SUCCESS;
}

int launch_timeout_selftest(cudaStream_t stream) {
    timeout_selftest_kernel<<<1, 32, 0, stream>>>(20000000ull);   // 20 ms
    return cudaGetLastError() == cudaSuccess ? WQ_OK : WQ_ERR_CUDA;
}

namespace {

int device_sms() {
    int sms = 148, dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms;
}

// Cycles of an fp4 data-parallel tile of bm rows: a fixed ~10,200 per tile
// (the first copies and decode, the accumulator's readout) and per k-step
// ~450 + 0.75 bm for one MMA (six stages; the copy and decode chain, not
// the MMA's ~2 cycles per row, sets it), ~2.8 per row for two (four
// stages).  Fitted to forced tile heights on the prepacked layout at 2070
// MHz: NVFP4 8192^3 and 2048 x 8192 x 3072, 4096^3, MXFP4 4096 x 3072^2,
// 2048 x 3072^2 and 1024 x 3072^2, tiles of 128..352 rows.
constexpr long long kFp4TileCycles = 10200;
long long fp4_kstep_cycles(int bm) { return bm <= kBMMax ? 450 + 3LL * bm / 4 : 28LL * bm / 10; }

// Tile height (activation rows) for M rows.  Data-parallel: least time, the
// waves of one-CTA-per-SM tiles times a tile's cost -- for int4 about
// (bm + 64) per k-step (MMA time grows with bm, the decode of a k-step does
// not), for the fp4 formats kFp4TileCycles + nks fp4_kstep_cycles, up to
// 384 rows (two MMAs on one decode, chosen where they save enough waves:
// the 2048 x 3072 x 3072 prefill runs 144 tiles of 352 rows in one wave
// instead of 264 of 192 in two).  Stream-K: least total work, tiles x
// (bm + 64), as the CTAs share it evenly, up to 256 rows.
int choose_bm(int M, int N, int nks, int sms, bool streamk, int fmt) {
    const int nt = (N + kBN - 1) / kBN;
    const int bm_max = (fmt != kINT4 && !streamk) ? kBMMaxFp4 : kBMMax;
    int bm = 0;
    long long best = -1;
    for (int cand = bm_max; cand >= 32; cand -= 32) {
        if (cand < 128 && cand < ((M + 31) / 32) * 32) continue;   // small tiles only to fit a small M
        const long long tiles = (long long)nt * ((M + cand - 1) / cand);
        const long long waves = (tiles + sms - 1) / sms;
        const long long cost = streamk ? tiles * (cand + 64)
                               : fmt == kINT4 ? waves * (cand + 64)
                                              : waves * (kFp4TileCycles + nks * fp4_kstep_cycles(cand));
        // candidates run from tall to short.  On a tie of the fp4 model the
        // shorter tile wins (fewer padded rows).  The int4 and stream-K models
        // keep the taller tile (2048 x 8192 x 3072 int4: 4 waves of 256 rows
        // run 122 us, 5 of 192 rows 142 us, which the (bm + 64) model scores
        // alike).
        const bool fp4_dp = fmt != kINT4 && !streamk;
        if (best < 0 || cost < best || (fp4_dp && cost == best)) {
            best = cost;
            bm = cand;
        }
    }
    if (const char* e = getenv("WQ_TC_BM")) {
        const int v = atoi(e);
        if (v >= 32 && v <= bm_max && v % 32 == 0) bm = v;
    }
    return bm;
}

struct TcPlan {
    int bm, nt_n, tiles, nks, G;
    long long units;
    bool streamk;
    int csk;           // cluster split-K: CTAs per tile (0: off)
    size_t ws_bytes;   // workspace a stream-K launch needs (0 if none)
};

// Cluster split-K policy (WQ_TC_CSK): 0 off, 1 automatic (the default), S >=
// 2 that many CTAs per tile where the shape allows.  Measured against
// stream-K on the decoder's shapes at M = 128 (int4, prepacked, same GPU):
// q / o 17.3 -> 12.9 us, k / v 17.1 -> 10.7, gate / up 22.6 -> 19.7, down
// 23.3 -> 20.6; and it needs no workspace.
int csk_setting() {
    const char* e = getenv("WQ_TC_CSK");
    return e ? atoi(e) : 1;
}

constexpr size_t kFlagBytes(int G) { return ((size_t)G * sizeof(unsigned) + 255) / 256 * 256; }

TcPlan plan_tc(int M, int N, int K, int sms, bool allow_streamk, int fmt, bool allow_csk = true) {
    TcPlan p{};
    p.nks = K / kBK;
    p.nt_n = (N + kBN - 1) / kBN;
    // stream-K where whole tiles would leave the waves badly filled: below 75%
    // the balance wins; above it the extra epilogue of a split tile (partials
    // out, partials in) costs more than the idle SMs (measured: 2048 x 3072 x
    // 3072 runs 87% full on whole tiles and is faster that way; 128 x 3072 x
    // 3072 -- 24 tiles on 152 SMs -- runs 1.8x faster split)
    int bm = choose_bm(M, N, p.nks, sms, false, fmt);
    long long tiles = (long long)p.nt_n * ((M + bm - 1) / bm);
    const long long waves = (tiles + sms - 1) / sms;
    const bool thin = (double)tiles / (double)(waves * sms) < 0.75;
    bool sk = allow_streamk && thin;
    if (allow_streamk && getenv("WQ_TC_STREAMK")) sk = atoi(getenv("WQ_TC_STREAMK")) != 0;   // tests, tuning
    // Cluster split-K where the tiles are so few that each can take a
    // cluster of at least two CTAs (S <= 8, the portable cluster size): the
    // k-steps split as in stream-K, the partial sums added on chip, no
    // workspace.
    p.csk = 0;
    const int csk_mode = csk_setting();
    if (allow_csk && thin && csk_mode != 0 && !(getenv("WQ_TC_STREAMK") && sk)) {
        const int bmc = choose_bm(M, N, p.nks, sms, true, fmt);
        const long long tc = (long long)p.nt_n * ((M + bmc - 1) / bmc);
        long long S = csk_mode >= 2 ? csk_mode : sms / tc;
        if (S > 8) S = 8;
        if (S > p.nks) S = p.nks;
        if (S >= 2 && tc * S <= sms) {
            p.csk = (int)S;
            sk = false;
            bm = bmc;
            tiles = tc;
        }
    }
    p.bm = bm;
    p.tiles = (int)tiles;
    p.units = tiles * p.nks;
    p.streamk = sk;
    p.G = (int)(p.csk ? tiles * p.csk : sk ? (p.units < sms ? p.units : sms) : (tiles < sms ? tiles : sms));
    if (sk) {
        // Fewer CTAs than SMs when the tiles are few: a CTA's k-steps shrink
        // as 1 / G, but the owner of a tile adds the partials (bm x 128 fp32
        // each) of the G / tiles CTAs sharing it.  The sum of the two is least
        // near tiles x sqrt(nks x 128 / bm) (same GPU, CTA counts 16..152:
        // int4 128 x 1024 x 3072 flat from 32 to 80 CTAs at 16.3 us against
        // 23.5 us on 152; 256 x 3072 x 3072 21.7 us on 96 against 28.9 us).
        const int g_max = p.G;
        const double g = (double)tiles * std::sqrt((double)p.nks * 128.0 / bm);
        const long long gi = (long long)(g + 0.5);
        if (gi >= tiles && gi < g_max) p.G = (int)gi;
        if (const char* e = getenv("WQ_TC_SK_G")) {   // tests, tuning: the stream-K CTA count, clamped
            const int v = atoi(e);
            if (v >= 1) p.G = v < g_max ? v : g_max;
        }
    }
    // the flag words cover every CTA a launch on this device can have, so a
    // later call with more CTAs never reads an earlier call's partials as flags
    p.ws_bytes = sk ? kFlagBytes(sms) + (size_t)p.G * kBN * bm * sizeof(float) : 0;
    return p;
}

}  // namespace

// Library-owned scratch of wq_gemm_static: the stream-K flags and partials
// of up to kStaticCtas CTAs with 128 x 256 fp32 tiles (zero at module load;
// every completed call leaves the flags zero).
constexpr int kStaticCtas = 160;
constexpr size_t kStaticWsBytes = kFlagBytes(kStaticCtas) + (size_t)kStaticCtas * kBN * kBMMax * sizeof(float);
static __device__ __align__(256) uint8_t g_static_ws[kStaticWsBytes];

void* static_workspace(size_t* bytes, cudaStream_t stream, int* status) {
    static void* addr[64] = {};
    *status = WQ_OK;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(g_static_mu);
    if (!addr[dev] && cudaGetSymbolAddress(&addr[dev], g_static_ws) != cudaSuccess) addr[dev] = nullptr;
    *bytes = addr[dev] ? kStaticWsBytes : 0;
    if (addr[dev] && g_static_dirty[dev]) {
        // a call reported a timeout since: zero the flag words before this
        // call's kernel reads them (on its stream; nothing is allocated)
        if (cudaMemsetAsync(addr[dev], 0, kFlagBytes(kStaticCtas), stream) != cudaSuccess) {
            *status = WQ_ERR_CUDA;
            return nullptr;
        }
        g_static_dirty[dev] = false;
    }
    return addr[dev];
}

size_t tc_workspace_bytes(int M, int N, int K, int fmt) {
    if (M <= 0 || N <= 0 || K <= 0 || K % kBK != 0) return 0;
    return plan_tc(M, N, K, device_sms(), true, fmt).ws_bytes;
}

namespace {

// The launch shared by both weight layouts: tp maps the weight tiles (2-D
// packed rows, or 3-D prepacked code blocks when pre), scales / zeros are the
// scale arrays or the record blocks.
int run_tc(const void* A, const CUtensorMap& tp, bool pre, const uint8_t* scales, const uint8_t* zeros,
           int kblocks, void* C, int M, int N, int K, int fmt, int group, bool out_f32, void* workspace,
           size_t workspace_bytes, const Epilogue& epi, bool pdl, cudaStream_t stream) {
    const int sms = device_sms();
    TcPlan plan = plan_tc(M, N, K, sms, workspace != nullptr, fmt);
    if (plan.streamk && workspace_bytes < plan.ws_bytes) plan = plan_tc(M, N, K, sms, false, fmt);
    if (plan.csk) {
        // every tile's cluster resident at once, else fewer CTAs per tile
        const int st_c = fmt == kINT4 ? kStagesOf<kINT4, false> : kStagesOf<kNVFP4, false>;
        const size_t smem_c = 1024 + (size_t)st_c * (plan.bm * kBK * 2 + kPTileBytes) + sizeof(TcShared);
        while (plan.csk >= 2 && csk_max_clusters(plan.csk, smem_c) < plan.tiles) --plan.csk;
        if (plan.csk >= 2) {
            plan.G = plan.tiles * plan.csk;
        } else {
            plan = plan_tc(M, N, K, sms, workspace != nullptr, fmt, false);
            if (plan.streamk && workspace_bytes < plan.ws_bytes) plan = plan_tc(M, N, K, sms, false, fmt, false);
        }
    }
    const int bm = plan.bm;
    const int bh = bm > kBMMax ? bm / 2 : bm;   // rows of one MMA and one TMA box
    if (bm > kBMMax && (fmt == kINT4 || plan.streamk || bh % 16 != 0)) return WQ_ERR_UNSUPPORTED;
    if (!plan.streamk && plan.tiles > 0x7FFFFFFF) return WQ_ERR_UNSUPPORTED;

    CUtensorMap ta;
    if (!encode_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, A, (uint64_t)K, (uint64_t)M, (uint64_t)K * 2, kBK, bh,
                   CU_TENSOR_MAP_SWIZZLE_128B))
        return WQ_ERR_UNSUPPORTED;

    TcArgs args;
    args.scales = scales;
    args.zeros = zeros;
    args.C = C;
    args.ws = nullptr;
    args.flags = nullptr;
    if (plan.streamk) {
        args.flags = static_cast<unsigned*>(workspace);
        args.ws = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + kFlagBytes(sms));
    }
    args.M = M;
    args.N = N;
    args.K = K;
    args.group = group;
    args.out_f32 = out_f32 ? 1 : 0;
    args.bm = bm;
    args.bh = bh;
    args.a_tile_bytes = bm * kBK * 2;
    args.stage_bytes = args.a_tile_bytes + kPTileBytes;
    args.idesc = idesc_bf16_f32(kBN, bh);
    args.nt_n = plan.nt_n;
    args.nks = plan.nks;
    args.units = plan.units;
    args.G = plan.G;
    args.csk = plan.csk;
    // Programmatic dependent launch for launches of up to two waves (and
    // every split plan): same GPU, MXFP4 2048 x 3072^2 29.5 -> 28.6 us, int4
    // 128 x 1024 x 3072 10.7 -> 9.7 us, 128 x 3072^2 12.7 -> 11.8 us.  A
    // longer persistent launch gained nothing and lost up to 2 % (8192^3
    // NVFP4, 13.5 tiles per CTA: the dependent CTAs land on SMs in the
    // order the predecessor frees them, not the placement whole-tile
    // scheduling relies on for sharing activation tiles in L2).
    args.pdl = (pdl && (plan.streamk || plan.csk || plan.tiles <= 2LL * plan.G)) ? 1 : 0;
    args.kblocks = kblocks;
    args.flag_wait_ns = kWaitNs;
    if (const char* e = getenv("WQ_TC_FLAG_WAIT_NS")) args.flag_wait_ns = strtoull(e, nullptr, 10);   // tests
    args.epi = epi;
    if (debug_on())
        fprintf(stderr, "wq: tcgen05%s M=%d N=%d K=%d: bm=%d tiles=%d %s grid=%d\n", pre ? " (prepacked)" : "", M, N,
                K, bm, plan.tiles, plan.csk ? "cluster split-K" : plan.streamk ? "stream-K" : "data-parallel", plan.G);
    const dim3 grid(plan.G, 1, 1);
    const int nst = fmt == kINT4 ? kStagesOf<kINT4, false>
                    : (bh < bm ? kStagesOf<kNVFP4, true> : kStagesOf<kNVFP4, false>);
    size_t smem = 1024 + (size_t)nst * args.stage_bytes + sizeof(TcShared);
    // Stream-K launches stage C through the decode warps' store scratch (2 KB
    // each) and write it in 16-byte pieces, where the output rows are 16-byte
    // aligned: there the owner's stores are on the critical path (same GPU:
    // int4 128 x 3072 x 3072 17.7 -> 16.8 us, 128 x 3072 x 8192 24.1 -> 23.3
    // us).  Whole-tile launches keep the scalar stores, which overlap other
    // tiles' work (with the scratch: 8192^3 NVFP4 778 -> 782 us).
    constexpr size_t kScrBytes = (size_t)kDecodeSets * 4 * 2048;
    constexpr size_t kMaxDynSmem = 227 * 1024;
    args.scr_off = (int)(((size_t)nst * args.stage_bytes + sizeof(TcShared) + 255) / 256 * 256);
    args.vec_store = plan.streamk && (N % (out_f32 ? 4 : 8) == 0) &&
                     1024 + (size_t)args.scr_off + kScrBytes <= kMaxDynSmem;
    if (args.vec_store) smem = 1024 + (size_t)args.scr_off + kScrBytes;
    // whole tiles of plain bf16 output: staged C, one bulk tensor store per
    // tile (WQ_TC_NO_TMA_STORE: the decode warps' stores, for tests)
    CUtensorMap tcm;
    memset(&tcm, 0, sizeof(tcm));
    const bool any_epi = epi.bias || epi.residual || epi.gated;
    // The staging tile (bm x 128 bf16) sits beside the stage ring where it
    // fits; a tile of more than 256 rows (two-MMA fp4) stages over the ring
    // itself when every CTA has one tile: its ring is idle once its MMAs
    // have completed, and no later tile's copies come (same GPU, MXFP4
    // 2048 x 3072^2, 144 tiles of 352 rows: 29.5 -> 28.6 us).
    const bool one_tile_per_cta = !plan.streamk && !plan.csk && plan.tiles <= plan.G;
    const bool beside = 1024 + (size_t)args.scr_off + (size_t)bm * 256 <= kMaxDynSmem;
    const bool over = bm > kBMMax && one_tile_per_cta && (size_t)nst * args.stage_bytes >= (size_t)bm * 256;
    args.stg_off = beside ? args.scr_off : 0;
    args.tma_store = !any_epi && !out_f32 && !plan.streamk && !plan.csk && (beside || over) && N % 8 == 0 &&
                     (reinterpret_cast<uintptr_t>(C) & 15) == 0 && !getenv("WQ_TC_NO_TMA_STORE") &&
                     encode_2d(&tcm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, C, (uint64_t)N, (uint64_t)M, (uint64_t)N * 2, kBN, bh,
                               CU_TENSOR_MAP_SWIZZLE_NONE);
    if (args.tma_store && beside) smem = 1024 + (size_t)args.scr_off + (size_t)bm * 256;
    if (debug_on()) fprintf(stderr, "wq: tensor-core C stores: %s\n", args.tma_store ? "bulk tensor" : "threads");
    switch (fmt) {
        case kNVFP4:
            return pre ? launch_fmt<kNVFP4, true>(ta, tp, args, grid, smem, stream, tcm)
                       : launch_fmt<kNVFP4, false>(ta, tp, args, grid, smem, stream, tcm);
        case kMXFP4:
            return pre ? launch_fmt<kMXFP4, true>(ta, tp, args, grid, smem, stream, tcm)
                       : launch_fmt<kMXFP4, false>(ta, tp, args, grid, smem, stream, tcm);
        default:
            return pre ? launch_fmt<kINT4, true>(ta, tp, args, grid, smem, stream, tcm)
                       : launch_fmt<kINT4, false>(ta, tp, args, grid, smem, stream, tcm);
    }
}

}  // namespace

int launch_tc(const void* A, const uint8_t* packed, const void* scales, const uint8_t* zeros, void* C, int M,
              int N, int K, int fmt, int group, bool out_f32, void* workspace, size_t workspace_bytes,
              const Epilogue& epi, bool pdl, cudaStream_t stream) {
    if (M == 0 || N == 0) return WQ_OK;
    // shapes this kernel takes: whole k-steps, TMA-legal strides, aligned
    // scale rows for the per-k-step scale loads
    if (K <= 0 || K % kBK != 0) return WQ_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(A) & 15) || (reinterpret_cast<uintptr_t>(packed) & 15))
        return WQ_ERR_UNSUPPORTED;
    CUtensorMap tp;
    if (!encode_2d(&tp, CU_TENSOR_MAP_DATA_TYPE_UINT8, packed, (uint64_t)K / 2, (uint64_t)N, (uint64_t)K / 2,
                   kBK / 2, kBN, CU_TENSOR_MAP_SWIZZLE_32B))
        return WQ_ERR_UNSUPPORTED;
    return run_tc(A, tp, false, static_cast<const uint8_t*>(scales), zeros, 0, C, M, N, K, fmt, group, out_f32,
                  workspace, workspace_bytes, epi, pdl, stream);
}

int launch_tc_prepacked(const void* A, const void* prepacked, void* C, int M, int N, int K, int fmt, int group,
                        bool out_f32, void* workspace, size_t workspace_bytes, const Epilogue& epi, bool pdl,
                        cudaStream_t stream) {
    if (M == 0 || N == 0) return WQ_OK;
    if (K <= 0 || K % kBK != 0) return WQ_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(A) & 15) || (reinterpret_cast<uintptr_t>(prepacked) & 15))
        return WQ_ERR_UNSUPPORTED;
    const uint64_t I = (uint64_t)(K + 127) / 128, Nb = (uint64_t)(N + 15) / 16;
    // the code blocks as [Nb][2 I][512 bytes]: one k-step of 128 rows is the
    // half blocks (ks) of 8 consecutive row blocks, 4 KB
    CUtensorMap tp;
    const uint64_t dims[3] = {128, 2 * I, Nb};          // 4-byte elements
    const uint64_t strides[2] = {512, I * 1024};
    const uint32_t box[3] = {128, 1, kBN / 16};
    if (!encode_3d(&tp, CU_TENSOR_MAP_DATA_TYPE_UINT32, prepacked, dims, strides, box)) return WQ_ERR_UNSUPPORTED;
    const uint8_t* recs = static_cast<const uint8_t*>(prepacked) + Nb * I * 1024;
    return run_tc(A, tp, true, recs, nullptr, (int)I, C, M, N, K, fmt, group, out_f32, workspace, workspace_bytes,
                  epi, pdl, stream);
}

}  // namespace wq
