// KV append: scatter the new tokens' K/V into the paged cache through
// slot_mapping (bf16 copy, or e4m3 / int8 / int4 quantisation with
// per-(block, kv_head) absmax scales).
//
// Definitions: "LLM Serving - KV Cache, Batching, Speculative Decoding",
// section "Recall and stretch" item 3 (keys/values appended in decode);
// "KV cache & continuous batching", sections "The core insight" and "KV cache
// memory math" (fp8 and int8 = 1 byte per element, int4 = half a byte);
// "LLM Inference Optimization",
// section "Memory Bandwidth Optimization" (KV-cache quantization).
#include <cuda_fp8.h>

#include "pa_device.cuh"
#include "pa_fp8.cuh"
#include "pa_internal.h"

namespace pa {

// One thread per 16-byte unit of one (token, kv_head) row, K and V.
__global__ void __launch_bounds__(256) kv_append_bf16_kernel(
    uint4* __restrict__ k_cache, uint4* __restrict__ v_cache, const uint4* __restrict__ k_new,
    const uint4* __restrict__ v_new, const int64_t* __restrict__ slots, int T, int Hkv, int units,
    int bs, int64_t cap_slots) {
    griddep_launch_dependents();  // the decode that follows may start its prologue
    const int64_t total = (int64_t)T * Hkv * units;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int u = (int)(i % units);
        const int64_t th = i / units;
        const int h = (int)(th % Hkv);
        const int64_t t = th / Hkv;
        const int64_t slot = slots[t];
        if (slot < 0) continue;
        if (slot >= cap_slots) {
            if (u == 0 && h == 0) raise_error(PA_DEVERR_SLOT);
            continue;
        }
        const int64_t blk = slot / bs, off = slot - blk * bs;
        const int64_t dst = ((blk * Hkv + h) * bs + off) * units + u;
        const int64_t src = (t * Hkv + h) * units + u;
        k_cache[dst] = k_new[src];
        v_cache[dst] = v_new[src];
    }
}

// Coded caches (e4m3, int8 or int4 codes, KVT).  One warp per (token, kv_head).
// Only the first token of each run of consecutive tokens that land in the
// same block does work: it quantises the whole run (at most bs tokens) for its
// head, K then V.
template <int KVT>
__global__ void __launch_bounds__(256) kv_append_q8_kernel(
    uint8_t* __restrict__ k_cache, uint8_t* __restrict__ v_cache, float* __restrict__ k_scale,
    float* __restrict__ v_scale, const uint16_t* __restrict__ k_new,
    const uint16_t* __restrict__ v_new, const int64_t* __restrict__ slots, int T, int Hkv, int bs,
    int64_t cap_slots) {
    griddep_launch_dependents();  // the decode that follows may start its prologue
    const int64_t wid = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (wid >= (int64_t)T * Hkv) return;
    const int t = (int)(wid / Hkv), h = (int)(wid % Hkv);
    const int64_t slot = slots[t];
    if (slot < 0) return;
    if (slot >= cap_slots) {
        if (h == 0 && (threadIdx.x & 31) == 0) raise_error(PA_DEVERR_SLOT);
        return;
    }
    const int64_t blk = slot / bs;
    if (t > 0) {
        const int64_t ps = slots[t - 1];
        if (ps >= 0 && ps < cap_slots && ps / bs == blk) return;  // not the run's first token
    }
    int r = 1;
    while (t + r < T && r < bs) {
        const int64_t s2 = slots[t + r];
        if (s2 < 0 || s2 >= cap_slots || s2 / bs != blk) break;
        ++r;
    }
    const int first = (int)(slot - blk * bs);
    constexpr int ROWB = Codec<KVT>::BITS * 128 / 8;   // bytes of one coded row of 128 elements
    const int64_t page = (blk * Hkv + h) * (int64_t)bs * ROWB;
    const int64_t row0 = ((int64_t)t * Hkv + h) * 128;
    auto off_of = [&](int j) { return (int)(slots[t + j] % bs); };
    q8_quantise_run<KVT>(k_cache + page, k_scale + blk * Hkv + h, k_new + row0, (int64_t)Hkv * 128, r, first,
                         off_of);
    q8_quantise_run<KVT>(v_cache + page, v_scale + blk * Hkv + h, v_new + row0, (int64_t)Hkv * 128, r, first,
                         off_of);
}

cudaError_t launch_kv_append(const AppendLaunch& L, cudaStream_t stream) {
    const int64_t cap = (int64_t)L.num_blocks * L.bs;
    if (L.kvt != PA_KV_BF16) {
        const int64_t warps = (int64_t)L.T * L.Hkv;
        const int blocks = (int)((warps * 32 + 255) / 256);
        auto kern = (L.kvt == PA_KV_INT4)   ? kv_append_q8_kernel<KV_INT4>
                    : (L.kvt == PA_KV_INT8) ? kv_append_q8_kernel<KV_INT8>
                                            : kv_append_q8_kernel<KV_FP8>;
        kern<<<blocks, 256, 0, stream>>>((uint8_t*)L.k_cache, (uint8_t*)L.v_cache, L.k_scale, L.v_scale,
                                         (const uint16_t*)L.k_new, (const uint16_t*)L.v_new, L.slots, L.T, L.Hkv,
                                         L.bs, cap);
    } else {
        const int units = L.d / 8;
        const int64_t total = (int64_t)L.T * L.Hkv * units;
        int blocks = (int)std::min<int64_t>((total + 255) / 256, 1 << 20);
        kv_append_bf16_kernel<<<blocks, 256, 0, stream>>>(
            (uint4*)L.k_cache, (uint4*)L.v_cache, (const uint4*)L.k_new, (const uint4*)L.v_new,
            L.slots, L.T, L.Hkv, units, L.bs, cap);
    }
    return cudaGetLastError();
}

// Whole-block copies (copy-on-write): for each pair i, every kv head's K and
// V page of block dst[i] becomes a copy of block src[i] (and the scales of a
// coded cache).
// One thread per 16-byte unit of a block's K (and V) data.
__global__ void __launch_bounds__(256) copy_blocks_kernel(uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                                                          float* __restrict__ k_scale, float* __restrict__ v_scale,
                                                          const int32_t* __restrict__ src,
                                                          const int32_t* __restrict__ dst, int n,
                                                          int64_t units, int Hkv, int num_blocks) {
    const int64_t total = (int64_t)n * units;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int p = (int)(i / units);
        const int64_t u = i - (int64_t)p * units;
        const int s = src[p], d = dst[p];
        if (s < 0 || s >= num_blocks || d < 0 || d >= num_blocks) {
            if (u == 0) raise_error(PA_DEVERR_BLOCK_ID);
            continue;
        }
        k_cache[(int64_t)d * units + u] = k_cache[(int64_t)s * units + u];
        v_cache[(int64_t)d * units + u] = v_cache[(int64_t)s * units + u];
        if (k_scale && u < Hkv) {
            k_scale[(int64_t)d * Hkv + u] = k_scale[(int64_t)s * Hkv + u];
            v_scale[(int64_t)d * Hkv + u] = v_scale[(int64_t)s * Hkv + u];
        }
    }
}

cudaError_t launch_copy_blocks(void* k_cache, void* v_cache, float* k_scale, float* v_scale, const int32_t* src,
                               const int32_t* dst, int n, int num_blocks, int Hkv, int d, int bs, int kvt,
                               cudaStream_t stream) {
    // bytes of one token row: 2 per element (bf16), 1 (e4m3, int8), 1/2 (int4)
    const int64_t rowb = kvt == PA_KV_BF16 ? 2 * d : (kvt == PA_KV_INT4 ? d / 2 : d);
    const int64_t units = (int64_t)Hkv * bs * rowb / 16;
    const int64_t total = (int64_t)n * units;
    const int blocks = (int)std::min<int64_t>((total + 255) / 256, 1 << 20);
    copy_blocks_kernel<<<blocks, 256, 0, stream>>>((uint4*)k_cache, (uint4*)v_cache,
                                                   kvt == PA_KV_BF16 ? nullptr : k_scale,
                                                   kvt == PA_KV_BF16 ? nullptr : v_scale, src, dst, n, units, Hkv,
                                                   num_blocks);
    return cudaGetLastError();
}

// Self-test of the bounded wait: one warp waits on a barrier phase that no
// thread or copy will ever complete.  The wait must give up on its own,
// record PA_DEVERR_TIMEOUT and let the kernel finish.
__global__ void bounded_wait_selftest_kernel() {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncwarp();
    mbar_wait(&bar, 0);
}

cudaError_t launch_wait_selftest(cudaStream_t stream) {
    bounded_wait_selftest_kernel<<<1, 32, 0, stream>>>();
    return cudaGetLastError();
}

cudaError_t append_unit_error(unsigned int* v, bool clear) { return read_unit_error(v, clear); }

}  // namespace pa
