// C entry points for the device operations of libpagedattn.so: argument
// validation, split planning, TMA descriptor encoding, dispatch.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <mutex>

#include "../../include/pa.h"
#include "pa_internal.h"

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

pa_status cuda_status(cudaError_t e) { return e == cudaSuccess ? PA_OK : PA_ERR_CUDA; }

bool shape_ok(int num_blocks, int Hkv, int d, int bs, int kv_dtype) {
    if (num_blocks <= 0 || Hkv <= 0 || bs <= 0 || d <= 0) return false;
    if (kv_dtype != PA_KV_BF16 && kv_dtype != PA_KV_FP8_E4M3 && kv_dtype != PA_KV_INT8 && kv_dtype != PA_KV_INT4)
        return false;
    if ((int64_t)num_blocks * Hkv * bs >= (int64_t)1 << 31) return false;  // TMA row coordinate
    return true;
}

// PA_OK, PA_ERR_INVALID or PA_ERR_UNSUPPORTED for head_dim / block_size / dtype.
pa_status kernel_shape(int d, int bs, int kv_dtype) {
    if (bs != 16 && bs != 32) return PA_ERR_UNSUPPORTED;
    if (kv_dtype != PA_KV_BF16) return d == 128 ? PA_OK : PA_ERR_UNSUPPORTED;   // coded rows: 128 (int4: 64) bytes
    return (d == 64 || d == 128) ? PA_OK : PA_ERR_UNSUPPORTED;
}

// ---------------------------------------------------------------- TMA maps
PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

struct MapKey {
    const void* ptr;
    int64_t rows;
    int d, box_tok, dtype, device;
    bool operator==(const MapKey& o) const {
        return ptr == o.ptr && rows == o.rows && d == o.d && box_tok == o.box_tok && dtype == o.dtype &&
               device == o.device;
    }
};

struct MapCache {
    static constexpr int N = 32;
    MapKey key[N];
    CUtensorMap map[N];
    bool used[N] = {};
    int next = 0;
    std::mutex mu;
};

MapCache& map_cache() {
    static MapCache c;
    return c;
}

// The cache viewed as a 2-D tensor: rows = num_blocks * Hkv * bs token rows of
// d elements; one box = box_tok rows x 128 bytes (a page, or the adjacent
// pages of several kv heads of one block), written to shared memory with the
// 128-byte swizzle (head_dim 128 bf16 takes two boxes per row range).  An int4
// row of 128 codes is 64 bytes: the tensor is then rows / 2 lines of 128 bytes
// (two tokens each) and a box is box_tok / 2 lines.
bool encode_cache_map(const void* base, int64_t rows, int d, int box_tok, int dtype, CUtensorMap* out) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = get_encode();
    if (!enc) return false;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    const MapKey k{base, rows, d, box_tok, dtype, dev};
    MapCache& c = map_cache();
    std::lock_guard<std::mutex> lock(c.mu);
    for (int i = 0; i < MapCache::N; ++i)
        if (c.used[i] && c.key[i] == k) {
            *out = c.map[i];
            return true;
        }
    const bool q8 = dtype != PA_KV_BF16;   // coded: byte elements (e4m3, int8; int4 two per byte)
    const bool i4 = dtype == PA_KV_INT4;
    const int elt = q8 ? 1 : 2;
    cuuint64_t gdim[2] = {(cuuint64_t)d, (cuuint64_t)rows};
    cuuint64_t gstride[1] = {(cuuint64_t)d * elt};
    cuuint32_t box[2] = {(cuuint32_t)(128 / elt), (cuuint32_t)box_tok};
    if (i4) {
        gdim[0] = 128;
        gdim[1] = (cuuint64_t)(rows / 2);
        gstride[0] = 128;
        box[0] = 128;
        box[1] = (cuuint32_t)(box_tok / 2);
    }
    cuuint32_t estride[2] = {1, 1};
    CUtensorMap m;
    CUresult r = enc(&m, q8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                     const_cast<void*>(base), gdim, gstride, box, estride,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return false;
    const int slot = c.next;
    c.next = (c.next + 1) % MapCache::N;
    c.key[slot] = k;
    c.map[slot] = m;
    c.used[slot] = true;
    *out = m;
    return true;
}

// The current device's SM count; without a device (host-side planning), a
// GB300's 152.
int device_sms() {
    constexpr int kGb300Sms = 152;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return kGb300Sms;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        return kGb300Sms;
    return sms;
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

constexpr int kMaxSplits = 512;  // partitions per sequence

struct WsLayout {
    size_t o_off, lse_off, cnt_off, total;
};

// o_part fp32 [B][Hq][S][d] | lse fp32 [B][Hq][S]   (S > 1 only)
// counters int32 [B][Hkv]                            (always)
// each part 256-byte aligned
WsLayout ws_layout(int B, int Hq, int Hkv, int d, int S) {
    const size_t rows = S > 1 ? (size_t)B * Hq * S : 0;
    auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
    WsLayout w;
    w.o_off = 0;
    w.lse_off = up(rows * d * sizeof(float));
    w.cnt_off = w.lse_off + up(rows * sizeof(float));
    w.total = w.cnt_off + up((size_t)B * Hkv * sizeof(int));
    return w;
}

// Blocks per partition for a resolved split count.
int part_blocks_for(int M, int S) { return (int)ceil_div(M, S < 1 ? 1 : S); }

// PA_FORCE_SPLITS=n (a positive integer) in the environment stands in for an
// explicit split count wherever the automatic one is asked for; read once.
int forced_splits() {
    static const int n = [] {
        const char* v = getenv("PA_FORCE_SPLITS");
        if (!v || !*v) return 0;
        char* end = nullptr;
        const long x = strtol(v, &end, 10);
        return (*end == '\0' && x > 0 && x <= kMaxSplits) ? (int)x : 0;
    }();
    return n;
}

}  // namespace

extern "C" {

const char* pa_status_string(pa_status s) {
    switch (s) {
        case PA_OK: return "PA_OK";
        case PA_ERR_INVALID: return "PA_ERR_INVALID";
        case PA_ERR_OOM: return "PA_ERR_OOM";
        case PA_ERR_CUDA: return "PA_ERR_CUDA";
        case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED";
    }
    return "PA_ERR_UNKNOWN";
}

pa_status pa_kv_append(void* k_cache, void* v_cache, float* k_scale, float* v_scale,
                       const void* k_new, const void* v_new, const int64_t* slot_mapping,
                       int num_tokens, int num_blocks, int num_kv_heads, int head_dim,
                       int block_size, int kv_dtype, void* stream) {
    pa::CallRange range("pa_kv_append");
    if (num_tokens < 0 || !shape_ok(num_blocks, num_kv_heads, head_dim, block_size, kv_dtype))
        return PA_ERR_INVALID;
    const pa_status ks = kernel_shape(head_dim, block_size, kv_dtype);
    if (ks != PA_OK) return ks;
    if (num_tokens == 0) return PA_OK;
    if (!k_cache || !v_cache || !k_new || !v_new || !slot_mapping) return PA_ERR_INVALID;
    if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(k_new) || !aligned16(v_new) ||
        (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
        return PA_ERR_INVALID;
    const bool q8 = kv_dtype != PA_KV_BF16;   // one-byte codes with scales
    if (q8 != (k_scale != nullptr) || q8 != (v_scale != nullptr)) return PA_ERR_INVALID;
    pa::AppendLaunch L{k_cache, v_cache, k_scale, v_scale, k_new, v_new, slot_mapping,
                       num_tokens, num_blocks, num_kv_heads, head_dim, block_size, kv_dtype};
    return cuda_status(pa::launch_kv_append(L, static_cast<cudaStream_t>(stream)));
}

int pa_decode_resolve_splits(int batch, int num_kv_heads, int max_blocks_per_seq, int num_splits) {
    if (batch <= 0 || num_kv_heads <= 0 || max_blocks_per_seq <= 0) return 1;
    const int M = max_blocks_per_seq;
    if (num_splits <= 0) num_splits = forced_splits();
    if (num_splits > 0) {
        int S = num_splits > M ? M : num_splits;
        if (S > kMaxSplits) S = kMaxSplits;
        return (int)ceil_div(M, part_blocks_for(M, S));
    }
    // Automatic: about two waves of the three CTAs an SM holds, assuming the
    // tables are half full on average; a CTA streams 32 .. 256 pages (enough
    // to amortise its start-up, few enough to keep the last wave short; the
    // many (sequence, head set) groups of large batches already fill the GPU,
    // so more partitions there only add merges: shared-prefix fp8 batch 344
    // -> 328 us at 256 pages against 128).  A CTA covers two kv heads when
    // their count is even, so its partition is half as many blocks.
    const int hpc = num_kv_heads % 2 == 0 ? 2 : 1;
    // Few (sequence, kv-head set) groups (long contexts): one wave of long
    // partitions instead.  The CTAs start together and stream evenly, and
    // fewer CTAs start and end (4 x 131072 tokens: 28 partitions, 0.99-1.01
    // of the copy peak, against 0.97 at 128 partitions of 64 blocks).
    const int64_t groups = (int64_t)batch * (num_kv_heads / hpc);
    const int64_t slots = (int64_t)device_sms() * 3;
    if (groups * 4 <= slots && (int64_t)M * hpc >= 2 * 128 * (slots / groups)) {
        int64_t S = slots / groups;
        if (S > M) S = M;
        if (S > kMaxSplits) S = kMaxSplits;
        return (int)ceil_div(M, ceil_div(M, S));
    }
    const int64_t pages = (int64_t)batch * num_kv_heads * M / 2;
    const int64_t target = (int64_t)device_sms() * 6;
    int64_t P = ceil_div(pages, target);
    if (P < 32) P = 32;
    if (P > 256) P = 256;
    P = ceil_div(P, hpc);
    if (P > M) P = M;
    if (ceil_div(M, P) > kMaxSplits) P = ceil_div(M, kMaxSplits);
    return (int)ceil_div(M, P);
}

size_t pa_decode_workspace_bytes(int batch, int num_q_heads, int num_kv_heads, int head_dim,
                                 int max_blocks_per_seq, int num_splits) {
    if (batch <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0) return 0;
    const int S = pa_decode_resolve_splits(batch, num_kv_heads, max_blocks_per_seq, num_splits);
    return ws_layout(batch, num_q_heads, num_kv_heads, head_dim, S).total;
}

}  // extern "C"

namespace pa {

// Every check of a decode call's arguments but the workspace's.  PA_OK for a
// call that may launch (batch == 0 included: it launches nothing).
pa_status decode_check(const void* out, const void* q, const void* k_cache, const void* v_cache,
                       const float* k_scale, const float* v_scale, const int32_t* block_tables,
                       const int32_t* seq_lens, int batch, int num_q_heads, int num_kv_heads, int head_dim,
                       int block_size, int max_blocks_per_seq, int num_blocks, float scale, int num_splits,
                       int kv_dtype, const void* k_new, const void* v_new) {
    if (batch < 0 || num_q_heads <= 0 || max_blocks_per_seq <= 0 || num_splits < 0 ||
        !shape_ok(num_blocks, num_kv_heads, head_dim, block_size, kv_dtype))
        return PA_ERR_INVALID;
    if (num_q_heads % num_kv_heads != 0) return PA_ERR_INVALID;
    if (num_q_heads / num_kv_heads > 8) return PA_ERR_UNSUPPORTED;
    if ((int64_t)max_blocks_per_seq * block_size >= (int64_t)1 << 31) return PA_ERR_INVALID;
    {   // one CTA per work item: at most S x (kv-head sets) x batch of them
        const int64_t items = (int64_t)pa_decode_resolve_splits(batch, num_kv_heads, max_blocks_per_seq, num_splits) *
                              (num_kv_heads % 2 == 0 ? num_kv_heads / 2 : num_kv_heads) * batch;
        if (items > INT32_MAX) return PA_ERR_UNSUPPORTED;
    }
    const pa_status ks = kernel_shape(head_dim, block_size, kv_dtype);
    if (ks != PA_OK) return ks;
    if (!(scale == scale)) return PA_ERR_INVALID;  // NaN
    if (batch == 0) return PA_OK;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !seq_lens) return PA_ERR_INVALID;
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) ||
        (reinterpret_cast<uintptr_t>(block_tables) & 3u) || (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
        return PA_ERR_INVALID;
    const bool q8 = kv_dtype != PA_KV_BF16;
    if (q8 && (!k_scale || !v_scale)) return PA_ERR_INVALID;
    if ((k_new != nullptr) != (v_new != nullptr)) return PA_ERR_INVALID;
    if (k_new && (!aligned16(k_new) || !aligned16(v_new))) return PA_ERR_INVALID;
    return PA_OK;
}

}  // namespace pa

namespace {

// Chunk partitions per chunk item set for a shared-prefix launch: chunks of up
// to max_chunk_blocks blocks in partitions of at most part_blocks.
int chunk_parts_for(int max_blocks_per_seq, int S, int max_chunk_blocks) {
    return max_chunk_blocks > 0 ? (int)ceil_div(max_chunk_blocks, part_blocks_for(max_blocks_per_seq, S)) : 0;
}

// The shared-prefix plan of one launch (n_chunks == 0: none).
struct SharePlan {
    const int32_t* chunk_of = nullptr;
    const int32_t* chunk_members = nullptr;
    const int32_t* chunk_blocks = nullptr;
    int n_chunks = 0, max_chunk_blocks = 0;
};

// Shared by pa_decode_attention (k_new == NULL), pa_decode_step and
// pa_decode_step_shared (plan.n_chunks > 0).
pa_status decode_impl(void* out, const void* q, const void* k_cache, const void* v_cache,
                      const float* k_scale, const float* v_scale, const int32_t* block_tables,
                      const int32_t* seq_lens, int batch, int num_q_heads, int num_kv_heads, int head_dim,
                      int block_size, int max_blocks_per_seq, int num_blocks, float scale, int num_splits,
                      void* workspace, size_t workspace_bytes, int kv_dtype, void* stream, const void* k_new,
                      const void* v_new, const SharePlan& plan = SharePlan()) {
    const pa_status chk = pa::decode_check(out, q, k_cache, v_cache, k_scale, v_scale, block_tables, seq_lens, batch,
                                           num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq,
                                           num_blocks, scale, num_splits, kv_dtype, k_new, v_new);
    if (chk != PA_OK || batch == 0) return chk;
    const int S = pa_decode_resolve_splits(batch, num_kv_heads, max_blocks_per_seq, num_splits);
    const int cparts = plan.n_chunks > 0 ? chunk_parts_for(max_blocks_per_seq, S, plan.max_chunk_blocks) : 0;
    const size_t need = plan.n_chunks > 0
                            ? pa_decode_shared_workspace_bytes(batch, num_q_heads, num_kv_heads, head_dim,
                                                               max_blocks_per_seq, num_splits, plan.max_chunk_blocks)
                            : pa_decode_workspace_bytes(batch, num_q_heads, num_kv_heads, head_dim,
                                                        max_blocks_per_seq, num_splits);
    if (!workspace || workspace_bytes < need || !aligned16(workspace)) return PA_ERR_INVALID;
    const int Sw = S + cparts;   // partial slots per output row

    const int64_t rows = (int64_t)num_blocks * num_kv_heads * block_size;
    // two kv heads per CTA when their count is even: one box holds a block's
    // pages of both
    const int hpc = num_kv_heads % 2 == 0 ? 2 : 1;
    CUtensorMap tm_k, tm_v;
    if (!encode_cache_map(k_cache, rows, head_dim, hpc * block_size, kv_dtype, &tm_k) ||
        !encode_cache_map(v_cache, rows, head_dim, hpc * block_size, kv_dtype, &tm_v))
        return PA_ERR_CUDA;

    pa::DecodeLaunch L;
    L.hpc = hpc;
    L.out = out;
    L.q = q;
    L.k_scale = k_scale;
    L.v_scale = v_scale;
    L.tables = block_tables;
    L.lens = seq_lens;
    L.o_part = nullptr;
    L.lse = nullptr;
    {
        const WsLayout wl = ws_layout(batch, num_q_heads, num_kv_heads, head_dim, Sw);
        char* base = static_cast<char*>(workspace);
        if (Sw > 1) {
            L.o_part = reinterpret_cast<float*>(base + wl.o_off);
            L.lse = reinterpret_cast<float*>(base + wl.lse_off);
        }
        L.counters = reinterpret_cast<int*>(base + wl.cnt_off);
    }
    L.tm_k = &tm_k;
    L.tm_v = &tm_v;
    L.B = batch;
    L.Hq = num_q_heads;
    L.Hkv = num_kv_heads;
    L.d = head_dim;
    L.bs = block_size;
    L.M = max_blocks_per_seq;
    L.num_blocks = num_blocks;
    L.part_blocks = part_blocks_for(max_blocks_per_seq, S);
    L.S = S;
    L.scale = scale;
    L.kvt = kv_dtype;
    L.k_new = k_new;
    L.v_new = v_new;
    L.k_cache_w = const_cast<void*>(k_cache);
    L.v_cache_w = const_cast<void*>(v_cache);
    L.k_scale_w = const_cast<float*>(k_scale);
    L.v_scale_w = const_cast<float*>(v_scale);
    L.Sw = Sw;
    L.chunk_of = plan.chunk_of;
    L.chunk_members = plan.chunk_members;
    L.chunk_blocks = plan.chunk_blocks;
    L.n_chunks = plan.n_chunks;
    L.chunk_parts = cparts;
    L.max_chunk_blocks = plan.max_chunk_blocks;
    return cuda_status(pa::launch_decode(L, static_cast<cudaStream_t>(stream)));
}

}  // namespace

extern "C" {

pa_status pa_decode_attention(void* out, const void* q, const void* k_cache, const void* v_cache,
                              const float* k_scale, const float* v_scale,
                              const int32_t* block_tables, const int32_t* seq_lens, int batch,
                              int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                              int max_blocks_per_seq, int num_blocks, float scale, int num_splits,
                              void* workspace, size_t workspace_bytes, int kv_dtype,
                              void* stream) {
    pa::CallRange range("pa_decode_attention");
    return decode_impl(out, q, k_cache, v_cache, k_scale, v_scale, block_tables, seq_lens, batch,
                       num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq, num_blocks,
                       scale, num_splits, workspace, workspace_bytes, kv_dtype, stream, nullptr, nullptr);
}

pa_status pa_decode_step(void* out, const void* q, const void* k_new, const void* v_new, void* k_cache,
                         void* v_cache, float* k_scale, float* v_scale, const int32_t* block_tables,
                         const int32_t* seq_lens, int batch, int num_q_heads, int num_kv_heads,
                         int head_dim, int block_size, int max_blocks_per_seq, int num_blocks, float scale,
                         int num_splits, void* workspace, size_t workspace_bytes, int kv_dtype, void* stream) {
    pa::CallRange range("pa_decode_step");
    if (batch > 0 && (!k_new || !v_new)) return PA_ERR_INVALID;
    return decode_impl(out, q, k_cache, v_cache, k_scale, v_scale, block_tables, seq_lens, batch,
                       num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq, num_blocks,
                       scale, num_splits, workspace, workspace_bytes, kv_dtype, stream, k_new, v_new);
}

size_t pa_decode_shared_workspace_bytes(int batch, int num_q_heads, int num_kv_heads, int head_dim,
                                        int max_blocks_per_seq, int num_splits, int max_chunk_blocks) {
    if (batch <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || max_chunk_blocks < 0) return 0;
    const int S = pa_decode_resolve_splits(batch, num_kv_heads, max_blocks_per_seq, num_splits);
    return ws_layout(batch, num_q_heads, num_kv_heads, head_dim,
                     S + chunk_parts_for(max_blocks_per_seq, S, max_chunk_blocks))
        .total;
}

pa_status pa_decode_step_shared(void* out, const void* q, const void* k_new, const void* v_new, void* k_cache,
                                void* v_cache, float* k_scale, float* v_scale, const int32_t* block_tables,
                                const int32_t* seq_lens, const int32_t* chunk_of, const int32_t* chunk_members,
                                const int32_t* chunk_blocks, int n_chunks, int max_chunk_blocks, int batch,
                                int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                int max_blocks_per_seq, int num_blocks, float scale, int num_splits,
                                void* workspace, size_t workspace_bytes, int kv_dtype, void* stream) {
    pa::CallRange range("pa_decode_step_shared");
    if (n_chunks < 0 || max_chunk_blocks < 0) return PA_ERR_INVALID;
    if (n_chunks > 0) {
        if (!chunk_of || !chunk_members || !chunk_blocks || max_chunk_blocks < 1 ||
            max_chunk_blocks > max_blocks_per_seq)
            return PA_ERR_INVALID;
        // chunk items: n_chunks x kv-head sets x chunk partitions must fit the grid with the rest
        const int S = pa_decode_resolve_splits(batch, num_kv_heads, max_blocks_per_seq, num_splits);
        const int64_t sets = num_kv_heads % 2 == 0 ? num_kv_heads / 2 : num_kv_heads;
        if ((int64_t)n_chunks * sets * chunk_parts_for(max_blocks_per_seq, S, max_chunk_blocks) +
                (int64_t)S * sets * batch > INT32_MAX)
            return PA_ERR_UNSUPPORTED;
    }
    SharePlan plan;
    plan.chunk_of = chunk_of;
    plan.chunk_members = chunk_members;
    plan.chunk_blocks = chunk_blocks;
    plan.n_chunks = n_chunks;
    plan.max_chunk_blocks = n_chunks > 0 ? max_chunk_blocks : 0;
    return decode_impl(out, q, k_cache, v_cache, k_scale, v_scale, block_tables, seq_lens, batch, num_q_heads,
                       num_kv_heads, head_dim, block_size, max_blocks_per_seq, num_blocks, scale, num_splits,
                       workspace, workspace_bytes, kv_dtype, stream, k_new, v_new, plan);
}

pa_status pa_copy_blocks(void* k_cache, void* v_cache, float* k_scale, float* v_scale, const int32_t* src,
                         const int32_t* dst, int n, int num_blocks, int num_kv_heads, int head_dim, int block_size,
                         int kv_dtype, void* stream) {
    pa::CallRange range("pa_copy_blocks");
    if (n < 0 || !shape_ok(num_blocks, num_kv_heads, head_dim, block_size, kv_dtype)) return PA_ERR_INVALID;
    const pa_status ks = kernel_shape(head_dim, block_size, kv_dtype);
    if (ks != PA_OK) return ks;
    if (n == 0) return PA_OK;
    if (!k_cache || !v_cache || !src || !dst || !aligned16(k_cache) || !aligned16(v_cache)) return PA_ERR_INVALID;
    const bool q8 = kv_dtype != PA_KV_BF16;   // coded cache with scales
    if (q8 != (k_scale != nullptr) || q8 != (v_scale != nullptr)) return PA_ERR_INVALID;
    return cuda_status(pa::launch_copy_blocks(k_cache, v_cache, k_scale, v_scale, src, dst, n, num_blocks,
                                              num_kv_heads, head_dim, block_size, kv_dtype,
                                              static_cast<cudaStream_t>(stream)));
}

pa_status pa_prefill_attention(void* out, const void* q, const void* k_cache, const void* v_cache,
                               const float* k_scale, const float* v_scale, const int32_t* block_tables,
                               const int32_t* seq_lens, const int32_t* q_start, int batch, int num_q_heads,
                               int num_kv_heads, int head_dim, int block_size, int max_blocks_per_seq,
                               int num_blocks, int max_q_len, float scale, int kv_dtype, void* stream) {
    pa::CallRange range("pa_prefill_attention");
    if (batch < 0 || num_q_heads <= 0 || max_blocks_per_seq <= 0 || max_q_len < 0 ||
        !shape_ok(num_blocks, num_kv_heads, head_dim, block_size, kv_dtype))
        return PA_ERR_INVALID;
    if (num_q_heads % num_kv_heads != 0) return PA_ERR_INVALID;
    if ((int64_t)max_blocks_per_seq * block_size >= (int64_t)1 << 31) return PA_ERR_INVALID;
    if (!(scale == scale)) return PA_ERR_INVALID;
    const int G = num_q_heads / num_kv_heads;
    if (head_dim != 128 || (block_size != 16 && block_size != 32) || 128 % G != 0) return PA_ERR_UNSUPPORTED;
    if (batch > 65535 || num_kv_heads > 65535) return PA_ERR_UNSUPPORTED;  // grid z / y
    if (batch == 0 || max_q_len == 0) return PA_OK;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !seq_lens || !q_start) return PA_ERR_INVALID;
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) ||
        (reinterpret_cast<uintptr_t>(block_tables) & 3u) || (reinterpret_cast<uintptr_t>(seq_lens) & 3u) ||
        (reinterpret_cast<uintptr_t>(q_start) & 3u))
        return PA_ERR_INVALID;
    const bool q8 = kv_dtype != PA_KV_BF16;   // coded cache with scales
    if (q8 != (k_scale != nullptr) || q8 != (v_scale != nullptr)) return PA_ERR_INVALID;
    const int64_t rows = (int64_t)num_blocks * num_kv_heads * block_size;
    CUtensorMap tm_k, tm_v;
    if (!encode_cache_map(k_cache, rows, head_dim, block_size, kv_dtype, &tm_k) ||
        !encode_cache_map(v_cache, rows, head_dim, block_size, kv_dtype, &tm_v))
        return PA_ERR_CUDA;
    pa::PrefillLaunch L;
    L.out = out;
    L.q = q;
    L.tables = block_tables;
    L.lens = seq_lens;
    L.q_start = q_start;
    L.tm_k = &tm_k;
    L.tm_v = &tm_v;
    L.B = batch;
    L.Hq = num_q_heads;
    L.Hkv = num_kv_heads;
    L.bs = block_size;
    L.M = max_blocks_per_seq;
    L.num_blocks = num_blocks;
    L.max_q = max_q_len;
    L.scale = scale;
    L.k_scale = k_scale;
    L.v_scale = v_scale;
    L.kvt = kv_dtype;
    return cuda_status(pa::launch_prefill(L, static_cast<cudaStream_t>(stream)));
}

pa_status pa_selftest_bounded_wait(void* stream) {
    return cuda_status(pa::launch_wait_selftest(static_cast<cudaStream_t>(stream)));
}

pa_status pa_get_device_error(uint32_t* flags, int clear) {
    if (!flags) return PA_ERR_INVALID;
    unsigned int a = 0, d = 0, p = 0;
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = pa::append_unit_error(&a, clear != 0);
    if (e == cudaSuccess) e = pa::decode_unit_error(&d, clear != 0);
    if (e == cudaSuccess) e = pa::prefill_unit_error(&p, clear != 0);
    if (e != cudaSuccess) return PA_ERR_CUDA;
    *flags = a | d | p;
    return PA_OK;
}

}  // extern "C"
