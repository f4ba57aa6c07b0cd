// Launch descriptors shared between the C entry points (pa_api.cu) and the
// kernel translation units.  Host-side only.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <nvtx3/nvToolsExt.h>

#include <algorithm>

#include "../../include/pa.h"

namespace pa {

// An NVTX range named after a C entry point, open for the host side of the
// call (checks, planning, launch), so that a profiler's timeline shows which
// call queued which kernels.  Without a profiler attached, a push or a pop is
// one call through an empty hook.
struct CallRange {
    explicit CallRange(const char* name) { nvtxRangePushA(name); }
    ~CallRange() { nvtxRangePop(); }
    CallRange(const CallRange&) = delete;
    CallRange& operator=(const CallRange&) = delete;
};

struct AppendLaunch {
    void* k_cache;
    void* v_cache;
    float* k_scale;
    float* v_scale;
    const void* k_new;
    const void* v_new;
    const int64_t* slots;
    int T, num_blocks, Hkv, d, bs;
    int kvt;            // PA_KV_BF16 / PA_KV_FP8_E4M3 / PA_KV_INT8 / PA_KV_INT4
};

struct DecodeLaunch {
    void* out;
    const void* q;
    const float* k_scale;
    const float* v_scale;
    const int32_t* tables;
    const int32_t* lens;
    float* o_part;      // workspace, [B][Hq][S][d] (S > 1 only)
    float* lse;         // workspace, [B][Hq][S]
    int* counters;      // workspace, [B][Hkv], zero between calls
    const CUtensorMap* tm_k;
    const CUtensorMap* tm_v;
    // fused step: each sequence's new token (position len-1) is written first
    const void* k_new;  // bf16 [B][Hkv][d], NULL: attention only
    const void* v_new;
    void* k_cache_w;
    void* v_cache_w;
    float* k_scale_w;
    float* v_scale_w;
    int B, Hq, Hkv, d, bs, M, num_blocks;
    int part_blocks;    // blocks per split partition
    int hpc;            // kv heads per CTA (1 or 2); the tensor maps' boxes span hpc heads' pages
    int S;              // partitions per sequence at most (grid x)
    float scale;
    int kvt;            // PA_KV_BF16 / PA_KV_FP8_E4M3 / PA_KV_INT8 / PA_KV_INT4
    int Sw;             // partial slots per output row in the workspace (S without shared prefixes)
    // shared prefixes (n_chunks > 0): the plan of pa_decode_step_shared
    const int32_t* chunk_of = nullptr;
    const int32_t* chunk_members = nullptr;
    const int32_t* chunk_blocks = nullptr;
    int n_chunks = 0, chunk_parts = 0, max_chunk_blocks = 0;
};

struct PrefillLaunch {
    void* out;          // bf16 [total_q][Hq][d]
    const void* q;      // bf16 [total_q][Hq][d]
    const float* k_scale;   // coded caches: [num_blocks][Hkv]
    const float* v_scale;
    const int32_t* tables;
    const int32_t* lens;
    const int32_t* q_start;   // [B + 1]
    const CUtensorMap* tm_k;
    const CUtensorMap* tm_v;
    int B, Hq, Hkv, bs, M, num_blocks, max_q;
    float scale;
    int kvt;            // PA_KV_BF16 / PA_KV_FP8_E4M3 / PA_KV_INT8 / PA_KV_INT4
};

// Checks of a decode call's arguments other than its workspace (pa_api.cu);
// returns the status the call would return, PA_OK if it may launch.
pa_status decode_check(const void* out, const void* q, const void* k_cache, const void* v_cache, const float* k_scale,
                       const float* v_scale, const int32_t* block_tables, const int32_t* seq_lens, int batch,
                       int num_q_heads, int num_kv_heads, int head_dim, int block_size, int max_blocks_per_seq,
                       int num_blocks, float scale, int num_splits, int kv_dtype, const void* k_new,
                       const void* v_new);

cudaError_t launch_kv_append(const AppendLaunch& L, cudaStream_t stream);
cudaError_t launch_prefill(const PrefillLaunch& L, cudaStream_t stream);
cudaError_t prefill_unit_error(unsigned int* v, bool clear);
cudaError_t launch_decode(const DecodeLaunch& L, cudaStream_t stream);

cudaError_t launch_wait_selftest(cudaStream_t stream);
cudaError_t launch_copy_blocks(void* k_cache, void* v_cache, float* k_scale, float* v_scale, const int32_t* src,
                               const int32_t* dst, int n, int num_blocks, int Hkv, int d, int bs, int kvt,
                               cudaStream_t stream);
cudaError_t append_unit_error(unsigned int* v, bool clear);
cudaError_t decode_unit_error(unsigned int* v, bool clear);

}  // namespace pa
