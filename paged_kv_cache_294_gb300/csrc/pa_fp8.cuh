// fp8 (e4m3) cache append arithmetic, shared by the append kernel and the
// fused decode step so that both write identical bytes.
//
// The rule ("KV cache & continuous batching", section "KV cache memory math":
// fp8 = 1 byte per element; "LLM Inference Optimization", section "Memory
// Bandwidth Optimization": KV-cache quantization): one fp32 scale per (block,
// kv head).  When a call writes tokens into a block starting at offset
// `first`:  old = first == 0 ? 0 : scale;  s = max(old, fp32(absmax) / 448);
// if s > old > 0 every older row (offset < first) is re-encoded as
// E4M3(fp32(value * old) / s);  each new value x becomes E4M3(x / s) (all +0
// when s == 0);  scale = s.  E4M3 rounds to nearest even and saturates at 448.
#pragma once

#include <cuda_fp8.h>

#include "pa_device.cuh"

namespace pa {

// e4m3 code -> fp32, exact (the e4m3 -> f16 conversion is exact).
__device__ __forceinline__ float e4m3_to_f32(uint32_t code) {
    const uint32_t h2 = e4m3x2_to_f16x2((uint16_t)(code & 0xFF));
    return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFF)));
}

__device__ __forceinline__ uint32_t f32_to_e4m3(float x) {
    return (uint32_t)__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3);
}

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

// The block's new scale from its current one (`old`, already 0 when the call
// starts the block at offset 0) and the absmax `a` of the new values; when it
// grows, the older rows (offsets < first) are re-encoded through
// load_old(o) / store_old(o, codes), 4 codes per lane.  One full warp.
template <typename LoadOld, typename StoreOld>
__device__ __forceinline__ float fp8_rescale(float old, float a, int first, LoadOld load_old, StoreOld store_old) {
    float s = __fdiv_rn(a, 448.0f);
    if (old > s) s = old;
    if (s > old && old > 0.f) {
#pragma unroll 1
        for (int o = 0; o < first; ++o) {
            const uint32_t w = load_old(o);
            uint32_t nw = 0;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float v = e4m3_to_f32((w >> (8 * e)) & 0xFF);
                nw |= f32_to_e4m3(__fdiv_rn(__fmul_rn(v, old), s)) << (8 * e);
            }
            store_old(o, nw);
        }
    }
    return s;
}

// 4 bf16 values (packed in w) -> 4 codes E4M3(x / s); all +0 when s == 0.
__device__ __forceinline__ uint32_t fp8_encode4(uint2 w, float s) {
    const float x[4] = {bf16_bits_to_f32(w.x & 0xFFFF), bf16_bits_to_f32(w.x >> 16), bf16_bits_to_f32(w.y & 0xFFFF),
                        bf16_bits_to_f32(w.y >> 16)};
    uint32_t nw = 0;
    if (s != 0.f) {
#pragma unroll
        for (int e = 0; e < 4; ++e) nw |= f32_to_e4m3(__fdiv_rn(x[e], s)) << (8 * e);
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
// lane owns bytes 4*lane .. 4*lane+3 of every row.  Returns the new scale.
template <typename OffFn>
__device__ __forceinline__ float fp8_quantise_run(uint8_t* __restrict__ page, float* __restrict__ scale_p,
                                                 const uint16_t* __restrict__ src, int64_t src_stride, int r,
                                                 int first, OffFn off_of) {
    const int lane = threadIdx.x & 31;
    float a = 0.f;
#pragma unroll 1
    for (int j = 0; j < r; ++j) a = fmaxf(a, absmax4(*reinterpret_cast<const uint2*>(src + j * src_stride + lane * 4)));
    a = warp_max(a);
    const float old = (first == 0) ? 0.f : *scale_p;
    uint32_t* rows = reinterpret_cast<uint32_t*>(page);
    const float s = fp8_rescale(
        old, a, first, [&](int o) { return rows[o * 32 + lane]; },
        [&](int o, uint32_t nw) { rows[o * 32 + lane] = nw; });
#pragma unroll 1
    for (int j = 0; j < r; ++j)
        rows[off_of(j) * 32 + lane] = fp8_encode4(*reinterpret_cast<const uint2*>(src + j * src_stride + lane * 4), s);
    __syncwarp();
    if (lane == 0) *scale_p = s;
    return s;
}

}  // namespace pa
