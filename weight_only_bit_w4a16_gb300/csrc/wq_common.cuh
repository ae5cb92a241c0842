// wq_common.cuh -- shared device helpers of the W4A16 kernels: the 4-bit
// decode into bf16 pairs and thin PTX wrappers.
//
// Decode contract (all three kernels use it, so the bf16 weights seen by the
// tensor cores are exactly the ones wq_dequant writes):
//   one 32-bit word holds 8 codes, element k0..k7 in nibbles 0..7 (byte j =
//   elements 2j (low nibble) and 2j+1 (high nibble), KBench
//   megakernel_int4_weight_decode.py spec, "The weight format").  A word
//   decodes into 4 bf16x2 registers holding the natural pairs (k0,k1),
//   (k2,k3), (k4,k5), (k6,k7), low half = even element, so they line up with
//   bf16 activations read straight from a row-major A.
//
//   int4:  x = bf16(128 + code) built with the exponent-bias trick (0x4300 is
//          128.0, the code lands in the low mantissa bits), then
//          (x - (128 + zero)) is an exact small integer and one bf16x2
//          multiply by the scale rounds the exact product to nearest even --
//          "subtract before multiply" as the KBench spec's Precision section
//          asks.  Zero points above 128 take a second exact subtraction.
//   e2m1:  the hardware e2m1x2 -> f16x2 conversion gives the exact value; the
//          f16 bit pattern shifted right by 3 is a bf16 pattern of the same
//          value times 2^-112 (all e2m1 values are normal f16 numbers), the
//          sign is moved back to bit 15, and one bf16x2 multiply by
//          (scale * 2^112) -- exact, as the product has at most 6 significant
//          bits -- restores e2m1 * scale.  MXFP4 scales with E > 142 (where
//          2^(E-15) would not fit bf16) use two exact multiplies.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

namespace wq {

constexpr int kNVFP4 = 0;
constexpr int kMXFP4 = 1;
constexpr int kINT4 = 2;

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

__device__ __forceinline__ uint32_t bf16x2_sub(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// two e2m1 codes in one byte -> f16x2 (low nibble -> low half)
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte_in_low8) {
    uint32_t d;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t}"
        : "=r"(d) : "r"(byte_in_low8));
    return d;
}

// four e2m1 pairs (the 4 bytes of w) -> four f16x2
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t (&h)[4]) {
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3]) : "r"(w));
}

// Loads of read-only inputs (weights and scales never change while a kernel
// runs): plain asm, so the compiler may schedule and predicate them freely.
__device__ __forceinline__ uint4 ldg_stream_v4(const void* p) {
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t ldg_u8(const uint8_t* p) {
    uint16_t v;
    asm("ld.global.nc.u8 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t ldg_u32(const void* p) {
    uint32_t v;
    asm("ld.global.nc.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t ldg_u16(const void* p) {
    uint16_t v;
    asm("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

// ---------------------------------------------------------------------------
// Per-group multipliers
// ---------------------------------------------------------------------------
// A decode "key" carries what one group needs, as bf16x2 words (both halves
// equal):
//   mul  : the multiplier (the scale, or scale * 2^112 for fp4)
//   mul2 : second multiplier, 1.0 unless an MXFP4 scale has E > 142
//   zz   : int4 only, 128 + zero (or 128 when zero > 128)
//   zz2  : int4 only, 0 (or the zero point itself when zero > 128)
// `two` marks the rare keys that need the second exact step; kernels branch
// on it warp-uniformly (ONE_STEP / TWO_STEP template argument below).
struct GroupKey {
    uint32_t mul;
    uint32_t mul2;
    uint32_t zz;
    uint32_t zz2;
    bool two;
};

__device__ __forceinline__ uint32_t splat16(uint32_t h) { return (h & 0xFFFFu) * 0x10001u; }

// int4 subtrahends from a prepacked record's zero-point pair zp = {z_r,
// z_(r+8)} (bytes 0, 1): the bf16x2 splat of 128 + z for row r (zsub_lo) and
// row r + 8 (zsub_hi).  0x43 over the byte z is 128 + z exactly for z <= 127,
// and z = 128 carries into the exponent: 0x4380 = 256.  Larger zero points
// take zsub_two.
__device__ __forceinline__ uint32_t zsub_lo(uint32_t zp) { return prmt(zp, 0x43u, 0x4040u); }
__device__ __forceinline__ uint32_t zsub_hi(uint32_t zp) { return prmt(zp, 0x43u, 0x4141u); }
// Any uint8 zero point z: the two exact subtrahends 128 + min(z, 128) and
// z - min(z, 128), as bf16x2 splats.
__device__ __forceinline__ void zsub_two(uint32_t z, uint32_t& first, uint32_t& second) {
    const uint32_t zc = min(z, 128u);
    first = splat16(0x4300u + zc);
    second = splat16(__bfloat16_as_ushort(__float2bfloat16_rn((float)(z - zc))));
}

// bf16 bits of |e4m3(b)| * 2^112 (exact: at most 4 significant bits, range
// 2^103 .. 1.75*2^120).  NaN (S.1111.111) gives a NaN multiplier; the sign
// bit is ignored (the weight uses |scale|).
__device__ __forceinline__ uint32_t nvfp4_mul_bits(uint32_t b) {
    const uint32_t e = (b >> 3) & 0xF, m = b & 7;
    if (e == 15 && m == 7) return 0x7FC0u;
    if (e != 0) return ((e + 232u) << 7) | (m << 4);   // 2^(e-7+112) * (1 + m/8)
    // subnormal e4m3: (m/8) * 2^-6 * 2^112 = m * 2^103
    if (m == 0) return 0u;
    const uint32_t lz = (m >= 4) ? 2u : (m >= 2 ? 1u : 0u);   // floor(log2 m)
    return ((230u + lz) << 7) | ((m << (7 - lz)) & 0x7Fu);
}

// Two NVFP4 multipliers at once, without branches: the hardware e4m3x2 ->
// f16x2 conversion is exact (every e4m3 value, subnormals included, is a
// normal f16 number or zero), and a normal f16 pattern h maps to the bf16
// pattern of |value| * 2^112 as ((h & 0x7FFF) >> 3) + (224 << 7): the f16
// exponent field rebased (-15 + 127 + 112) and the mantissa's top 7 bits,
// which hold all 3 e4m3 mantissa bits.  Zero stays zero; NaN stays NaN.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_bytes) {
    uint32_t d;
    asm("{\n\t.reg .b16 lo, hi;\n\t"
        "mov.b32 {lo, hi}, %1;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, lo;\n\t}"
        : "=r"(d) : "r"(two_bytes));
    return d;
}

__device__ __forceinline__ uint32_t nvfp4_mul_from_f16(uint32_t h16) {
    const uint32_t m = h16 & 0x7FFFu;
    const uint32_t b = (m >> 3) + (224u << 7);
    return m ? b : 0u;
}

__device__ __forceinline__ GroupKey key_nvfp4(uint32_t sbyte) {
    GroupKey k;
    k.mul = splat16(nvfp4_mul_bits(sbyte));
    k.mul2 = 0x3F803F80u;
    k.zz = 0;
    k.zz2 = 0;
    k.two = false;
    return k;
}

__device__ __forceinline__ GroupKey key_mxfp4(uint32_t E) {
    GroupKey k;
    k.zz = 0;
    k.zz2 = 0;
    k.mul2 = 0x3F803F80u;
    k.two = false;
    if (E == 0xFF) {
        k.mul = 0x7FC07FC0u;
    } else if (E <= 142) {
        k.mul = splat16((E + 112u) << 7);   // 2^(E-127) * 2^112
    } else {
        k.mul = splat16(0x7780u);           // 2^112
        k.mul2 = splat16(E << 7);           // 2^(E-127), normal for E in 143..254
        k.two = true;
    }
    return k;
}

__device__ __forceinline__ GroupKey key_int4(uint32_t sbits, uint32_t zero) {
    GroupKey k;
    k.mul = splat16(sbits);
    k.mul2 = 0x3F803F80u;
    if (zero <= 128) {
        // 128 + zero in [128, 256]: exactly representable (8 significant bits)
        k.zz = splat16(__bfloat16_as_ushort(__float2bfloat16_rn(128.0f + (float)zero)));
        k.zz2 = 0;
        k.two = false;
    } else {
        k.zz = splat16(0x4300u);   // 128
        k.zz2 = splat16(__bfloat16_as_ushort(__float2bfloat16_rn((float)zero)));
        k.two = true;
    }
    return k;
}

// ---------------------------------------------------------------------------
// Word decode: 8 codes -> 4 natural bf16x2 pairs
// ---------------------------------------------------------------------------
// int4, exact integer (code - zero) as bf16 (no scale applied)
template <bool TWO>
__device__ __forceinline__ void int4_word_centered(uint32_t w, const GroupKey& key, uint32_t (&p)[4]) {
    const uint32_t v = w >> 4;
    const uint32_t sel[4] = {0x0400u, 0x0501u, 0x0602u, 0x0703u};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint32_t x = (prmt(w, v, sel[i]) & 0x000F000Fu) | 0x43004300u;   // 128 + code
        x = bf16x2_sub(x, key.zz);
        if constexpr (TWO) x = bf16x2_sub(x, key.zz2);
        p[i] = x;
    }
}

// int4 codes of one word minus the zero point, as exact bf16 integers, with
// nibble s paired with nibble s + 4: (n0,n4), (n1,n5), (n2,n6), (n3,n7).  In
// the input layout these are the k pairs (k, k+4); the prepacked layout
// stores k0 + 2s in nibble s and k0 + 2s + 1 in nibble s + 4, so there they
// are natural pairs.  The exponent-bias trick makes bf16(128 + code) with one
// mask-and-or, and one exact bf16x2 subtraction of (128 + zero) leaves
// (code - zero).  Zero points above 128 take a second exact subtraction (TWO).
// (x & 0x000F000F) | magic as one lop3 with the magic in a register
__device__ __forceinline__ uint32_t nib_or_magic(uint32_t x, uint32_t magic) {
    uint32_t d;
    asm("lop3.b32 %0, %1, 0x000F000F, %2, 0xEA;" : "=r"(d) : "r"(x), "r"(magic));
    return d;
}

template <bool TWO>
__device__ __forceinline__ void int4_word_kk4(uint32_t w, uint32_t zz, uint32_t zz2, uint32_t (&p)[4]) {
    const uint32_t magic = 0x43004300u;
    p[0] = bf16x2_sub(nib_or_magic(w, magic), zz);
    p[1] = bf16x2_sub(nib_or_magic(w >> 4, magic), zz);
    p[2] = bf16x2_sub(nib_or_magic(w >> 8, magic), zz);
    p[3] = bf16x2_sub(nib_or_magic(w >> 12, magic), zz);
    if constexpr (TWO) {
#pragma unroll
        for (int i = 0; i < 4; ++i) p[i] = bf16x2_sub(p[i], zz2);
    }
}

// e2m1 codes as bf16 values times 2^-112 (exact), natural pairs
__device__ __forceinline__ void e2m1_word_raw(uint32_t w, uint32_t (&p)[4]) {
    uint32_t h[4];
    e2m1x8_to_f16x2(w, h);
#pragma unroll
    for (int i = 0; i < 4; ++i)
        p[i] = ((h[i] >> 3) & 0x0FFF0FFFu) | (h[i] & 0x80008000u);
}

// one word with its group's scale applied: bf16 RNE of the exact weight
template <int FMT, bool TWO>
__device__ __forceinline__ void word_scaled(uint32_t w, const GroupKey& key, uint32_t (&p)[4]) {
    if constexpr (FMT == kINT4) {
        int4_word_centered<TWO>(w, key, p);
#pragma unroll
        for (int i = 0; i < 4; ++i) p[i] = bf16x2_mul(p[i], key.mul);
    } else {
        e2m1_word_raw(w, p);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            p[i] = bf16x2_mul(p[i], key.mul);
            if constexpr (TWO) p[i] = bf16x2_mul(p[i], key.mul2);
        }
    }
}

__device__ __forceinline__ uint32_t bf16x2_fma(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// int4 word as an exact two-term bf16 sum: hi = RNE(w), lo = w - hi.  The
// weight (code - zero) * scale has at most 13 significant bits, so the
// residual (at most 6 bits) is a bf16 number and fma(x, s, -hi), which rounds
// the exact x*s - hi once, returns it exactly: hi + lo == w.
template <bool TWO>
__device__ __forceinline__ void int4_word_split(uint32_t w, const GroupKey& key, uint32_t (&hi)[4], uint32_t (&lo)[4]) {
    uint32_t x[4];
    int4_word_centered<TWO>(w, key, x);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        hi[i] = bf16x2_mul(x[i], key.mul);
        lo[i] = bf16x2_fma(x[i], key.mul, hi[i] ^ 0x80008000u);
    }
}

// The same split for a prepacked int4 word (k0 + 2s in nibble s, k0 + 2s + 1
// in nibble s + 4): natural pairs straight from the nibble pairs.
template <bool TWO>
__device__ __forceinline__ void int4_word_split_pairs(uint32_t w, const GroupKey& key, uint32_t (&hi)[4],
                                                      uint32_t (&lo)[4]) {
    uint32_t x[4];
    int4_word_kk4<TWO>(w, key.zz, key.zz2, x);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        hi[i] = bf16x2_mul(x[i], key.mul);
        lo[i] = bf16x2_fma(x[i], key.mul, hi[i] ^ 0x80008000u);
    }
}

// ---------------------------------------------------------------------------
// Fused epilogue of every GEMM kernel
// ---------------------------------------------------------------------------
// Optional, per output element, in fp32 before the cast to C:
//   y = acc (+ bias[n])                              bias: bf16 per weight row
//   gated: y = silu(y_gate) * y_up                   the SiLU-gated product of a
//          gate/up projection pair whose rows interleave in groups of 8 --
//          weight rows 16b .. 16b+7 are the gate rows of outputs 8b .. 8b+7,
//          rows 16b+8 .. 16b+15 their up rows (KBench spec, the decoder MLP
//          down(silu(gate(x)) * up(x)))
//   y += residual[m, o]                              bf16, row-major (M, outputs)
struct Epilogue {
    const uint16_t* bias;
    const uint16_t* residual;
    int gated;
};

__device__ __forceinline__ float bf16_at(const uint16_t* p, size_t i) {
    return __uint_as_float((uint32_t)__ldg(p + i) << 16);
}

__device__ __forceinline__ float silu_f32(float x) { return x / (1.0f + expf(-x)); }

// Write output (m, weight row n): v is the accumulated value of row n, u that
// of row n + 8 (gated mode only; n must then be a gate row).  Nw: weight rows.
__device__ __forceinline__ void store_epilogue(const Epilogue& e, void* C, int out_f32, int Nw, int m, int n,
                                               float v, float u) {
    float y = v;
    if (e.bias) y += bf16_at(e.bias, n);
    int ldc = Nw, o = n;
    if (e.gated) {
        if (e.bias) u += bf16_at(e.bias, n + 8);
        y = silu_f32(y) * u;
        ldc = Nw >> 1;
        o = ((n >> 4) << 3) | (n & 7);
    }
    const size_t idx = (size_t)m * ldc + o;
    if (e.residual) y += bf16_at(e.residual, idx);
    if (out_f32) static_cast<float*>(C)[idx] = y;
    else static_cast<__nv_bfloat16*>(C)[idx] = __float2bfloat16_rn(y);
}

// key of group gi from the raw scale / zero arrays
template <int FMT>
__device__ __forceinline__ GroupKey load_key(const void* scales, const uint8_t* zeros, size_t gi) {
    if constexpr (FMT == kNVFP4) return key_nvfp4(ldg_u8(static_cast<const uint8_t*>(scales) + gi));
    else if constexpr (FMT == kMXFP4) return key_mxfp4(ldg_u8(static_cast<const uint8_t*>(scales) + gi));
    else return key_int4(ldg_u16(static_cast<const uint16_t*>(scales) + gi), ldg_u8(zeros + gi));
}

}  // namespace wq
