// Coded-cache arithmetic (e4m3 and int8 codes of one byte, int4 codes of
// half a byte), shared by the append kernel and the fused decode step so that
// both write identical bytes.
//
// The rule ("KV cache & continuous batching", section "KV cache memory math":
// fp8 = 1 byte per element; "LLM Inference Optimization", section "Memory
// Bandwidth Optimization": KV-cache quantization, INT8 halving the reads):
// one fp32 scale per (block, kv head).  When a call writes tokens into a
// block starting at offset `first`:  old = first == 0 ? 0 : scale;
// s = max(old, fp32(absmax) / QMAX);  if s > old > 0 every older row
// (offset < first) is re-encoded as Q(fp32(value * old) / s);  each new value
// x becomes Q(x / s) (all codes 0 when s == 0);  scale = s.
//   e4m3 (KV_FP8):  QMAX = 448, Q = E4M3 round to nearest even, saturating;
//   int8 (KV_INT8): QMAX = 127, Q = clamp(round half to even, -127, 127);
//   int4 (KV_INT4): QMAX = 7, Q = clamp(round half to even, -7, 7), stored as
//                   4-bit two's complement, element 2j of a row in the low
//                   nibble of byte j and element 2j+1 in the high nibble
//                   (half a byte per element: "KV cache memory math").
#pragma once

#include <cuda_fp8.h>

#include <type_traits>

#include "pa_device.cuh"

namespace pa {

enum KvType { KV_BF16 = 0, KV_FP8 = 1, KV_INT8 = 2, KV_INT4 = 3 };

// e4m3 code -> fp32, exact (the e4m3 -> f16 conversion is exact).
__device__ __forceinline__ float e4m3_to_f32(uint32_t code) {
    const uint32_t h2 = e4m3x2_to_f16x2((uint16_t)(code & 0xFF));
    return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFF)));
}

__device__ __forceinline__ uint32_t f32_to_e4m3(float x) {
    return (uint32_t)__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3);
}

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

// int8 code (two's-complement byte) -> fp32, exact.
__device__ __forceinline__ float s8_to_f32(uint32_t code) { return (float)(int8_t)(code & 0xFF); }

__device__ __forceinline__ uint32_t f32_to_s8(float x) {
    const int q = max(-127, min(127, __float2int_rn(x)));   // NaN converts to 0
    return (uint32_t)q & 0xFF;
}

// four one-byte codes of the cache type KVT (bytes 0..3 of w) -> two f16x2:
// lo = {byte 0, byte 1}, hi = {byte 2, byte 3}; exact for both code types.
// int8: with its sign bit flipped a code c becomes the byte u = c + 128; one
// byte permute places two such bytes under the f16 pattern 0x64.., whose
// value is 1024 + u, and subtracting 1152 leaves c (every step exact).
template <int KVT>
__device__ __forceinline__ void code4_to_f16x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
    if constexpr (KVT == KV_INT8) {
        const uint32_t u = w ^ 0x80808080u;
        const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
        uint32_t a, b;
        asm("prmt.b32 %0, %1, %2, 0x4140;" : "=r"(a) : "r"(u), "r"(0x64646464u));
        asm("prmt.b32 %0, %1, %2, 0x4342;" : "=r"(b) : "r"(u), "r"(0x64646464u));
        __half2 ha = __hsub2(*reinterpret_cast<__half2*>(&a), bias);
        __half2 hb = __hsub2(*reinterpret_cast<__half2*>(&b), bias);
        lo = *reinterpret_cast<uint32_t*>(&ha);
        hi = *reinterpret_cast<uint32_t*>(&hb);
    } else {
        lo = e4m3x2_to_f16x2((uint16_t)(w & 0xFFFF));
        hi = e4m3x2_to_f16x2((uint16_t)(w >> 16));
    }
}

// four int8 codes -> two f16x2 holding 1152 + c (the step of code4_to_f16x2
// before its subtraction; exact).  A dot product with these values exceeds the
// one with the codes by 1152 * (sum of the other operand), a constant per
// query head that the caller removes once per score.
__device__ __forceinline__ void s8x4_to_f16x2_biased(uint32_t w, uint32_t& lo, uint32_t& hi) {
    const uint32_t u = w ^ 0x80808080u;
    asm("prmt.b32 %0, %1, %2, 0x4140;" : "=r"(lo) : "r"(u), "r"(0x64646464u));
    asm("prmt.b32 %0, %1, %2, 0x4342;" : "=r"(hi) : "r"(u), "r"(0x64646464u));
}
// The same values with the even bytes (0, 2) in lo and the odd bytes (1, 3)
// in hi: a byte reorder and the conversion in the same two permutes.
__device__ __forceinline__ void s8x4_eo_to_f16x2_biased(uint32_t w, uint32_t& lo, uint32_t& hi) {
    const uint32_t u = w ^ 0x80808080u;
    asm("prmt.b32 %0, %1, %2, 0x4240;" : "=r"(lo) : "r"(u), "r"(0x64646464u));
    asm("prmt.b32 %0, %1, %2, 0x4341;" : "=r"(hi) : "r"(u), "r"(0x64646464u));
}
constexpr float kS8Bias = 1152.f;

// int4 code (low nibble, two's complement) -> fp32, exact.
__device__ __forceinline__ float s4_to_f32(uint32_t code) { return (float)((int)(code << 28) >> 28); }

__device__ __forceinline__ uint32_t f32_to_s4(float x) {
    const int q = max(-7, min(7, __float2int_rn(x)));   // NaN converts to 0
    return (uint32_t)q & 0xF;
}

// eight int4 codes (nibbles 0..7 of w, element j in nibble j) -> four f16x2:
// f[0] = {e0, e4}, f[1] = {e1, e5}, f[2] = {e2, e6}, f[3] = {e3, e7}; exact.
// With its sign bit flipped a code c becomes the nibble u = c + 8.  Masking
// nibbles 0 and 4 (or 2 and 6 after a shift by 8) under the f16 pattern
// 0x64.. gives 1024 + u, and subtracting 1032 leaves c; nibbles 1 and 5 (3 and
// 7) land 4 bits higher, giving 1024 + 16u, and x / 16 - 72 leaves c.  The mask,
// the sign flip and the exponent bits are one three-input logic operation.
__device__ __forceinline__ void nib8_to_f16x2(uint32_t w, uint32_t (&f)[4]) {
    const uint32_t w8 = w >> 8;
    uint32_t r[4];
    asm("lop3.b32 %0, %1, %2, %3, 0x6a;" : "=r"(r[0]) : "r"(w), "r"(0x000F000Fu), "r"(0x64086408u));
    asm("lop3.b32 %0, %1, %2, %3, 0x6a;" : "=r"(r[1]) : "r"(w), "r"(0x00F000F0u), "r"(0x64806480u));
    asm("lop3.b32 %0, %1, %2, %3, 0x6a;" : "=r"(r[2]) : "r"(w8), "r"(0x000F000Fu), "r"(0x64086408u));
    asm("lop3.b32 %0, %1, %2, %3, 0x6a;" : "=r"(r[3]) : "r"(w8), "r"(0x00F000F0u), "r"(0x64806480u));
    const __half2 b1032 = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));
    const __half2 s16 = __halves2half2(__ushort_as_half(0x2C00), __ushort_as_half(0x2C00));    // 1/16
    const __half2 m72 = __halves2half2(__ushort_as_half(0xD480), __ushort_as_half(0xD480));    // -72
#pragma unroll
    for (int i = 0; i < 4; i += 2) {
        __half2 a = __hsub2(*reinterpret_cast<__half2*>(&r[i]), b1032);
        __half2 b = __hfma2(*reinterpret_cast<__half2*>(&r[i + 1]), s16, m72);
        f[i] = *reinterpret_cast<uint32_t*>(&a);
        f[i + 1] = *reinterpret_cast<uint32_t*>(&b);
    }
}

// The same eight codes before the final subtraction / scaling (exact): f[0],
// f[2] hold 1032 + c (nibbles 0, 4 and 2, 6), f[1], f[3] hold 1152 + 16c
// (nibbles 1, 5 and 3, 7).  The caller removes the offsets and the factor 16
// after the products are summed.
__device__ __forceinline__ void nib8_to_f16x2_raw(uint32_t w, uint32_t (&f)[4]) {
    const uint32_t w8 = w >> 8;
    asm("lop3.b32 %0, %1, %2, %3, 0x6a;" : "=r"(f[0]) : "r"(w), "r"(0x000F000Fu), "r"(0x64086408u));
    asm("lop3.b32 %0, %1, %2, %3, 0x6a;" : "=r"(f[1]) : "r"(w), "r"(0x00F000F0u), "r"(0x64806480u));
    asm("lop3.b32 %0, %1, %2, %3, 0x6a;" : "=r"(f[2]) : "r"(w8), "r"(0x000F000Fu), "r"(0x64086408u));
    asm("lop3.b32 %0, %1, %2, %3, 0x6a;" : "=r"(f[3]) : "r"(w8), "r"(0x00F000F0u), "r"(0x64806480u));
}
constexpr float kS4BiasLo = 1032.f, kS4BiasHi = 1152.f;

// BITS: bits per code; a lane's four codes pack into BITS * 4 bits, code e at
// bit BITS * e (int4: the nibble order of the row).
template <int KVT>
struct Codec;
template <>
struct Codec<KV_FP8> {
    static constexpr int BITS = 8;
    static constexpr float QMAX = 448.f;
    __device__ __forceinline__ static float value(uint32_t c) { return e4m3_to_f32(c); }
    __device__ __forceinline__ static uint32_t encode(float x) { return f32_to_e4m3(x); }
};
template <>
struct Codec<KV_INT8> {
    static constexpr int BITS = 8;
    static constexpr float QMAX = 127.f;
    __device__ __forceinline__ static float value(uint32_t c) { return s8_to_f32(c); }
    __device__ __forceinline__ static uint32_t encode(float x) { return f32_to_s8(x); }
};
template <>
struct Codec<KV_INT4> {
    static constexpr int BITS = 4;
    static constexpr float QMAX = 7.f;
    __device__ __forceinline__ static float value(uint32_t c) { return s4_to_f32(c); }
    __device__ __forceinline__ static uint32_t encode(float x) { return f32_to_s4(x); }
};
// the codec of a coded cache type (bf16 maps to e4m3 only so that templates
// instantiated for every type compile; bf16 paths never call it)
template <int KVT>
using CodecOf = Codec<KVT == KV_BF16 ? KV_FP8 : KVT>;

// The block's new scale from its current one (`old`, already 0 when the call
// starts the block at offset 0) and the absmax `a` of the new values; when it
// grows, the older rows (offsets < first) are re-encoded through
// load_old(o) / store_old(o, codes), 4 codes per lane.  One full warp.
template <int KVT, typename LoadOld, typename StoreOld>
__device__ __forceinline__ float q8_rescale(float old, float a, int first, LoadOld load_old, StoreOld store_old) {
    using Q = Codec<KVT>;
    constexpr uint32_t MASK = (1u << Q::BITS) - 1;
    float s = __fdiv_rn(a, Q::QMAX);
    if (old > s) s = old;
    if (s > old && old > 0.f) {
#pragma unroll 1
        for (int o = 0; o < first; ++o) {
            const uint32_t w = load_old(o);
            uint32_t nw = 0;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float v = Q::value((w >> (Q::BITS * e)) & MASK);
                nw |= Q::encode(__fdiv_rn(__fmul_rn(v, old), s)) << (Q::BITS * e);
            }
            store_old(o, nw);
        }
    }
    return s;
}

// 4 bf16 values (packed in w) -> 4 codes Q(x / s); all 0 when s == 0.
template <int KVT>
__device__ __forceinline__ uint32_t q8_encode4(uint2 w, float s) {
    const float x[4] = {bf16_bits_to_f32(w.x & 0xFFFF), bf16_bits_to_f32(w.x >> 16), bf16_bits_to_f32(w.y & 0xFFFF),
                        bf16_bits_to_f32(w.y >> 16)};
    uint32_t nw = 0;
    if (s != 0.f) {
#pragma unroll
        for (int e = 0; e < 4; ++e) nw |= Codec<KVT>::encode(__fdiv_rn(x[e], s)) << (Codec<KVT>::BITS * e);
    }
    return nw;
}

__device__ __forceinline__ float absmax4(uint2 w) {
    float a = fabsf(bf16_bits_to_f32(w.x & 0xFFFF));
    a = fmaxf(a, fabsf(bf16_bits_to_f32(w.x >> 16)));
    a = fmaxf(a, fabsf(bf16_bits_to_f32(w.y & 0xFFFF)));
    return fmaxf(a, fabsf(bf16_bits_to_f32(w.y >> 16)));
}

__device__ __forceinline__ float warp_max(float a) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    return a;
}

// Quantise r bf16 rows of 128 values (row j at src + j * src_stride) into
// `page` (rows of 128 codes) at offsets off_of(j), for one (block, kv head)
// with scale *scale_p; `first` is the smallest offset written.  One full warp;
// lane owns the codes of elements 4*lane .. 4*lane+3 of every row (one 32-bit
// word of a one-byte row, one 16-bit word of an int4 row).  Returns the new
// scale.
template <int KVT, typename OffFn>
__device__ __forceinline__ float q8_quantise_run(uint8_t* __restrict__ page, float* __restrict__ scale_p,
                                                 const uint16_t* __restrict__ src, int64_t src_stride, int r,
                                                 int first, OffFn off_of) {
    const int lane = threadIdx.x & 31;
    float a = 0.f;
#pragma unroll 1
    for (int j = 0; j < r; ++j) a = fmaxf(a, absmax4(*reinterpret_cast<const uint2*>(src + j * src_stride + lane * 4)));
    a = warp_max(a);
    const float old = (first == 0) ? 0.f : *scale_p;
    using W = typename std::conditional<Codec<KVT>::BITS == 8, uint32_t, uint16_t>::type;
    W* rows = reinterpret_cast<W*>(page);
    const float s = q8_rescale<KVT>(
        old, a, first, [&](int o) { return rows[o * 32 + lane]; },
        [&](int o, uint32_t nw) { rows[o * 32 + lane] = (W)nw; });
#pragma unroll 1
    for (int j = 0; j < r; ++j)
        rows[off_of(j) * 32 + lane] =
            (W)q8_encode4<KVT>(*reinterpret_cast<const uint2*>(src + j * src_stride + lane * 4), s);
    __syncwarp();
    if (lane == 0) *scale_p = s;
    return s;
}

}  // namespace pa
