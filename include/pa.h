/*
 * pa.h - C ABI of libpagedattn.so: attention over a paged KV cache for
 * NVIDIA GB300 (sm_103a): single-token decode, multi-query (chunked-prefill /
 * speculative-verify) attention, the cache append, and the host-side block
 * allocator, prefix cache and schedulers.
 *
 * Pages this interface follows (cited by title and section):
 *   [P1] "KV cache & continuous batching" (docs.masst.dev/ai/inference/kv-cache-batching)
 *   [P2] "LLM Serving - KV Cache, Batching, Speculative Decoding"
 *        (dineshblog.com/blog/session-124-llm-serving)
 *   [P3] "LLM Inference Optimization: KV Cache, Batching, and Speculative
 *        Decoding" (adaptiverecall.com/open-source-llms/inference-optimization.php)
 *
 * Conventions for every call
 *   - Device pointers are owned by the caller (for example allocated by
 *     PyTorch).  The device entry points allocate no device memory, never
 *     synchronise the device, and enqueue their kernels on the caller's
 *     stream, passed as `void* stream` (a cudaStream_t; NULL = legacy default
 *     stream).  Host pointers are read only during the call.
 *   - Errors are return codes (pa_status); nothing throws, nothing aborts.
 *     Argument errors are found on the host before any launch and leave every
 *     buffer untouched.
 *   - Values that only the device can check (block ids read from a block
 *     table, lengths read from seq_lens, slots read from slot_mapping) are
 *     range-checked inside the kernels: an offending element is skipped or
 *     clamped (no out-of-bounds access is ever made) and a bit is set in a
 *     per-device error word that pa_get_device_error() returns.
 *
 * Memory layout (all row-major, innermost last)
 *   k_cache, v_cache  [num_blocks][num_kv_heads][block_size][head_dim]
 *                     bf16 (PA_KV_BF16), e4m3 bytes (PA_KV_FP8_E4M3),
 *                     two's-complement int8 codes (PA_KV_INT8) or 4-bit codes
 *                     two per byte (PA_KV_INT4: a row is head_dim / 2 bytes,
 *                     element 2j in the low nibble of byte j, 2j+1 in the high).
 *                     One (block, kv_head) page is contiguous.
 *   k_scale, v_scale  [num_blocks][num_kv_heads] fp32 (coded caches only:
 *                     e4m3, int8, int4)
 *   q, out            [batch][num_q_heads][head_dim] bf16
 *   k_new, v_new      [num_tokens][num_kv_heads][head_dim] bf16
 *   block_tables      [batch][max_blocks_per_seq] int32: physical block of
 *                     logical block j of sequence b ([P1] "2. PagedAttention")
 *   seq_lens          [batch] int32, tokens of each sequence including the one
 *                     appended this step
 *   slot_mapping      [num_tokens] int64, slot = block * block_size + offset
 *
 * Query head i reads KV head i / (num_q_heads / num_kv_heads) (grouped-query
 * attention, [P1] "KV cache memory math"; consecutive query heads share a KV
 * head, the pages leave the order open).
 */
#ifndef PAGEDATTN_PA_H
#define PAGEDATTN_PA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PA_OK = 0,
    PA_ERR_INVALID = 1,     /* bad argument (shape, null pointer, range, workspace too small) */
    PA_ERR_OOM = 2,         /* allocator: not enough free blocks (nothing was taken) */
    PA_ERR_CUDA = 3,        /* a CUDA runtime call or kernel launch failed */
    PA_ERR_UNSUPPORTED = 4  /* a valid request the library does not implement (e.g. fp8 with head_dim 64) */
} pa_status;

typedef enum {
    PA_KV_BF16 = 0,
    PA_KV_FP8_E4M3 = 1,
    PA_KV_INT8 = 2,     /* int8 codes c in [-127, 127], value c * scale ([P3] "Memory
                           Bandwidth Optimization": INT8 KV quantization) */
    PA_KV_INT4 = 3      /* 4-bit two's-complement codes c in [-7, 7], value c * scale,
                           two per byte ([P1] "KV cache memory math": int4 = 0.5 byte
                           per element) */
} pa_kv_dtype;

/* Bits of the per-device error word (pa_get_device_error). */
#define PA_DEVERR_BLOCK_ID   0x1u   /* a block table entry outside [0, num_blocks) (clamped to block 0) */
#define PA_DEVERR_SEQ_LEN    0x2u   /* seq_len < 0 or > max_blocks_per_seq * block_size (clamped) */
#define PA_DEVERR_SLOT       0x4u   /* slot >= num_blocks * block_size (token skipped) */
#define PA_DEVERR_TIMEOUT    0x8u   /* a pipeline wait exceeded its bound; the kernel gave up */

/* Human-readable name of a status code (static string). */
const char* pa_status_string(pa_status s);

/* ---------------------------------------------------------------------------
 * pa_kv_append - write the K/V of new tokens into the paged cache.
 *
 * Defines: [P2] "Recall and stretch" item 3 (keys/values are written in
 * prefill and appended in decode) and [P1] "The core insight" (decode
 * computes K/V for the new token only).  Token t, KV head h is written to
 * cache[slot / block_size][h][slot % block_size][:], slot = slot_mapping[t];
 * a negative slot skips the token.
 *
 * PA_KV_BF16: an exact copy of the bf16 bits; k_scale / v_scale must be NULL.
 *
 * PA_KV_FP8_E4M3 ([P1] "KV cache memory math": fp8 = 1 byte per element;
 * [P3] "Memory Bandwidth Optimization": KV-cache quantization): one fp32
 * scale per (block, kv_head), separately for K and V.  For each block p that
 * this call writes, with f = the smallest offset written:
 *     old = 0 if f == 0 else scale[p][h]
 *     s   = max(old, fp32(max|x| over the new values) / 448)
 *     if s > old > 0, each older entry (offset < f) is re-encoded as
 *         E4M3(fp32(value(e) * old) / s)
 *     each new value x is stored as E4M3(x / s) (round to nearest even,
 *     saturating at +-448); all codes are +0 when s == 0;  scale[p][h] = s.
 * PA_KV_INT8 ([P3] "Memory Bandwidth Optimization": INT8 KV quantization
 * halves the cache reads): the same rule with 127 in place of 448 and the
 * code Q(y) = clamp(round-half-to-even(y), -127, 127) in place of E4M3; an
 * element's value is code * scale.
 * PA_KV_INT4 ([P1] "KV cache memory math": int4 takes half a byte per
 * element): the same rule with 7 in place of 127 and Q(y) = clamp(round-half-
 * to-even(y), -7, 7), stored as 4-bit two's complement, two codes per byte
 * (element 2j of a row in the low nibble of byte j, 2j+1 in the high nibble).
 * Precondition (coded caches only): the tokens a call writes into one block form one
 * run of consecutive entries of slot_mapping with increasing offsets (true for
 * one decode token per sequence and for a prefill of one sequence).  A
 * violation gives unspecified cache contents but no out-of-bounds access.
 *
 * num_blocks * num_kv_heads * block_size must be below 2^31.  head_dim in
 * {64, 128} (coded caches: 128), block_size in {16, 32}.  num_tokens == 0 is a no-op.
 * ------------------------------------------------------------------------- */
pa_status pa_kv_append(void* k_cache, void* v_cache, float* k_scale, float* v_scale,
                       const void* k_new, const void* v_new, const int64_t* slot_mapping,
                       int num_tokens, int num_blocks, int num_kv_heads, int head_dim,
                       int block_size, int kv_dtype, void* stream);

/* ---------------------------------------------------------------------------
 * Split-K (flash-decoding) planning for pa_decode_attention.
 *
 * With S = num_splits (at most 512, at most max_blocks_per_seq) and
 * P = ceil(max_blocks_per_seq / S), sequence b with n = ceil(seq_len_b /
 * block_size) blocks uses k = ceil(n / P) partitions of ceil(n / k) blocks
 * each (the last one possibly shorter).
 * Each partition yields a normalised partial output and its log-sum-exp,
 * combined as
 *     out = sum_i exp(lse_i - L) o_i,  L = log sum_i exp(lse_i)
 * which equals the unsplit result in exact arithmetic.  The combination runs
 * inside pa_decode_attention: the last partition of a (sequence, kv head) to
 * finish merges them.  num_splits == 0 picks S from the batch shape and the
 * current device's SM count (152, a GB300's, when no device is visible).
 *
 * pa_decode_resolve_splits returns the S that pa_decode_attention will use for
 * the request (0 asks for the automatic choice); the workspace must hold
 * pa_decode_workspace_bytes(...) bytes for that S (always at least 256).
 * Workspace layout, each part 256-byte aligned: when S > 1, o_part fp32
 * [batch][num_q_heads][S][head_dim] and lse fp32 [batch][num_q_heads][S]
 * (base-2 log-sum-exp of the scaled scores); then merge counters int32
 * [batch][num_kv_heads].  The workspace must be zero-filled before its
 * first use; every call that completes leaves the counters at zero again
 * (after a PA_DEVERR_TIMEOUT, zero it again).  The counters' place follows
 * from the layout (batch, heads, S): a workspace reused for a request of
 * another layout must be zero-filled again.  Calls that share a workspace
 * must not overlap on the device.
 * ------------------------------------------------------------------------- */
/* PA_FORCE_SPLITS=n in the environment (an integer in 1 .. 512, read once, at
 * the first call) makes every request for the automatic choice use n as if it
 * were passed: the split sweeps of long contexts without a code change.
 * Other values are ignored; an explicit num_splits always wins. */
int pa_decode_resolve_splits(int batch, int num_kv_heads, int max_blocks_per_seq, int num_splits);
size_t pa_decode_workspace_bytes(int batch, int num_q_heads, int num_kv_heads, int head_dim,
                                 int max_blocks_per_seq, int num_splits);

/* ---------------------------------------------------------------------------
 * pa_decode_attention - one decode step's attention for a batch.
 *
 * Defines: [P1] "The core insight" (the new token's query attends over all
 * cached K and V), [P2] "Hands-on: cache equivalence and scheduling oracles"
 * (cached attention = softmax(q . K^T * scale) . V, the last row of causal
 * attention), [P1] "2. PagedAttention" (K and V gathered through the block
 * table, blocks need not be contiguous), [P3] "FlashAttention" (scores,
 * softmax and P.V fused on chip, fp32 online softmax).
 *
 *   out[b][i][:] = sum_t softmax_t(scale * q[b][i] . K_t) V_t,
 *   t = 0 .. seq_lens[b]-1,  K_t = k_cache[block_tables[b][t / bs]][i / G][t % bs]
 * fp8 / int8 / int4: K_t and V_t elements are value(code) * scale[block][kv_head].
 * A sequence with seq_len 0 gives a zero row.  The outputs are bf16.
 *
 * num_blocks * num_kv_heads * block_size must be below 2^31; head_dim in
 * {64, 128} (coded caches: 128); block_size in {16, 32}; num_q_heads a multiple of
 * num_kv_heads with a group size of at most 8.  batch == 0 is a no-op.  The
 * launch has one CTA per (sequence, kv-head set, partition), a kv-head set
 * being two heads when num_kv_heads is even, else one: S * sets * batch must
 * stay below 2^31 (PA_ERR_UNSUPPORTED otherwise).
 * ------------------------------------------------------------------------- */
pa_status pa_decode_attention(void* out, const void* q, const void* k_cache, const void* v_cache,
                              const float* k_scale, const float* v_scale,
                              const int32_t* block_tables, const int32_t* seq_lens, int batch,
                              int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                              int max_blocks_per_seq, int num_blocks, float scale, int num_splits,
                              void* workspace, size_t workspace_bytes, int kv_dtype, void* stream);

/* ---------------------------------------------------------------------------
 * pa_decode_step - one whole decode step of a layer in one launch: the append
 * of every sequence's new token followed by decode attention.
 *
 * Equivalent to pa_kv_append(k_new, v_new, slot_mapping) with slot_mapping[b]
 * = block_tables[b][(seq_lens[b]-1) / block_size] * block_size +
 * (seq_lens[b]-1) % block_size (the new token is position seq_lens[b]-1,
 * [P1] "The core insight"; [P2] "Recall and stretch" 3), followed by
 * pa_decode_attention with the same arguments: the cache bytes, fp8 scales
 * and outputs are the same as those two calls give.  Sequences with
 * seq_len 0 append nothing.  The block receiving a sequence's new token must
 * belong to that sequence alone (a shared block must be copied first).
 *   k_new, v_new  bf16 [batch][num_kv_heads][head_dim], 16-byte aligned
 * Everything else as pa_decode_attention; k_cache / v_cache (and the fp8
 * scales) are written.
 * ------------------------------------------------------------------------- */
pa_status pa_decode_step(void* out, const void* q, const void* k_new, const void* v_new, void* k_cache,
                         void* v_cache, float* k_scale, float* v_scale, const int32_t* block_tables,
                         const int32_t* seq_lens, int batch, int num_q_heads, int num_kv_heads,
                         int head_dim, int block_size, int max_blocks_per_seq, int num_blocks, float scale,
                         int num_splits, void* workspace, size_t workspace_bytes, int kv_dtype,
                         void* stream);

/* ---------------------------------------------------------------------------
 * pa_decode_attention_static_ws - pa_decode_attention for callers that cannot
 * allocate device memory.  (The pages have no counterpart to this entry
 * point: it is a convenience of this library.)
 *
 * Some callers only ever receive their input and output buffers and may not
 * call cudaMalloc themselves: plugins of inference runtimes that plan every
 * byte of device memory ahead of time, or code that runs while another
 * component owns the allocator, where an allocation would fail, upset the
 * memory plan or implicitly synchronise the device.  This entry point takes
 * the same arguments as pa_decode_attention minus the workspace and uses a
 * workspace owned by the library instead: a device array of
 * PA_STATIC_WORKSPACE_BYTES that every GPU which loads the library keeps
 * until the process exits.  It allocates nothing (no cudaMalloc, no
 * cudaFree) and gives the same outputs as pa_decode_attention.
 *   - Requests whose workspace (pa_decode_workspace_bytes) exceeds
 *     PA_STATIC_WORKSPACE_BYTES return PA_ERR_INVALID and launch nothing;
 *     use pa_decode_attention with a caller workspace for those.
 *   - Arguments are checked exactly as pa_decode_attention checks them, and
 *     a refused call queues no work at all.
 *   - The first call in a device's context looks up the array's device
 *     address (cudaGetSymbolAddress, which may load the library's device
 *     code) and keeps it for that context; after cudaDeviceReset the next
 *     call looks it up again.  Make the first call on each device (and the
 *     first after a reset) before any stream capture.
 *   - Every call uses the same array: each call zeroes its counter words with
 *     cudaMemsetAsync on `stream` before the kernel, and calls whose work
 *     overlaps on the GPU (other streams, other threads) race on the array
 *     and must be serialised by the caller.
 * ------------------------------------------------------------------------- */
#define PA_STATIC_WORKSPACE_BYTES ((size_t)16 << 20)

pa_status pa_decode_attention_static_ws(void* out, const void* q, const void* k_cache,
                                        const void* v_cache, const float* k_scale,
                                        const float* v_scale, const int32_t* block_tables,
                                        const int32_t* seq_lens, int batch, int num_q_heads,
                                        int num_kv_heads, int head_dim, int block_size,
                                        int max_blocks_per_seq, int num_blocks, float scale,
                                        int num_splits, int kv_dtype, void* stream);

/* ---------------------------------------------------------------------------
 * Shared prefixes in one decode step ([P3] "KV Cache Management": 100
 * requests with one system prompt share its KV; [P1] "4. Prefix caching").
 *
 * When several sequences' tables name the same physical blocks for their
 * first positions, pa_decode_step_shared reads those blocks once per chunk
 * of up to PA_SHARE_MAX_ROWS / G sequences instead of once per sequence: a
 * chunk's work item takes its members' query heads as the rows of one
 * contraction over the shared pages and writes one (partial, log-sum-exp)
 * per member and head, which the split-K merge combines with the member's
 * own pages.  The outputs are the same attention (within the parity bound;
 * the summation order differs from pa_decode_step's).
 *
 * The plan (pa_share_plan builds it on the host from the block tables and
 * lengths; the caller copies its arrays to the device):
 *   chunk_of       [batch] int32: chunk of sequence b, -1 for none
 *   chunk_members  [n_chunks][PA_SHARE_MAX_ROWS] int32: member sequences, -1 padded
 *   chunk_blocks   [n_chunks] int32: shared blocks of the chunk, taken from
 *                  its first member's table row
 * Requirements (checked on the device; a sequence or member that fails them
 * is attended without sharing and PA_DEVERR_BLOCK_ID is set): b appears once
 * in chunk chunk_of[b]; 1 <= chunk_blocks[c] <= max_chunk_blocks and
 * chunk_blocks[c] <= (seq_lens[b] - 1) / block_size for every member (the
 * shared blocks lie before each member's newest token); a chunk holds at most
 * PA_SHARE_MAX_ROWS / (num_q_heads / num_kv_heads) members.  The caller
 * guarantees that the members' tables agree on those blocks (pa_share_plan's
 * plans do); if they do not, the members attend the first member's blocks.
 * ------------------------------------------------------------------------- */
#define PA_SHARE_MAX_ROWS 8

/* Build a plan: sequences whose first physical block is the same form a
 * group; its shared length is the number of leading blocks every member holds
 * at the same positions, capped by each member's (seq_lens - 1) / block_size;
 * groups sharing at least max(min_blocks, 1) blocks are cut, in batch order,
 * into chunks of group_rows sequences (group_rows = PA_SHARE_MAX_ROWS / G for
 * the decode launch; below 2 nothing is shared).  Host arrays; at most
 * max_chunks chunks (later groups are left unshared).  *max_chunk_blocks =
 * the largest chunk_blocks. */
pa_status pa_share_plan(const int32_t* block_tables, int max_blocks_per_seq, const int32_t* seq_lens, int batch,
                        int block_size, int group_rows, int min_blocks, int32_t* chunk_of, int32_t* chunk_members,
                        int32_t* chunk_blocks, int max_chunks, int* n_chunks, int* max_chunk_blocks);

/* Workspace for pa_decode_step_shared: pa_decode_workspace_bytes' layout
 * with room for the chunk partials (max_chunk_blocks as passed to the step). */
size_t pa_decode_shared_workspace_bytes(int batch, int num_q_heads, int num_kv_heads, int head_dim,
                                        int max_blocks_per_seq, int num_splits, int max_chunk_blocks);

/* pa_decode_step (k_new / v_new given) or pa_decode_attention (both NULL)
 * with the plan above (device arrays; n_chunks == 0 reads none of them).
 * Other arguments, layouts and errors as pa_decode_step; the workspace must
 * hold pa_decode_shared_workspace_bytes. */
pa_status pa_decode_step_shared(void* out, const void* q, const void* k_new, const void* v_new, void* k_cache,
                                void* v_cache, float* k_scale, float* v_scale, const int32_t* block_tables,
                                const int32_t* seq_lens, const int32_t* chunk_of, const int32_t* chunk_members,
                                const int32_t* chunk_blocks, int n_chunks, int max_chunk_blocks, int batch,
                                int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                int max_blocks_per_seq, int num_blocks, float scale, int num_splits,
                                void* workspace, size_t workspace_bytes, int kv_dtype, void* stream);

/* Read (and optionally clear) the current device's error word; synchronises
 * the device.  *flags receives an OR of PA_DEVERR_* bits set since the last
 * clear. */
pa_status pa_get_device_error(uint32_t* flags, int clear);

/* Enqueue a one-warp kernel that waits on a shared-memory barrier phase that
 * nothing completes, through the same bounded wait the decode pipeline uses.
 * The wait gives up after about two seconds, the kernel ends normally and
 * PA_DEVERR_TIMEOUT is set in the device error word: a check, without any
 * GPU fault, that no barrier wait in this library can hang a GPU. */
pa_status pa_selftest_bounded_wait(void* stream);

/* ---------------------------------------------------------------------------
 * Host side: block allocator, accounting, slots, scheduler simulator.
 * No device access.  Not thread-safe per allocator object.
 * ------------------------------------------------------------------------- */

/* Paged KV-block pool: [P1] "2. PagedAttention" (fixed-size blocks allocated
 * on demand and freed when done, not necessarily contiguous) and [P2] "KV
 * memory, paging and prefix identity" (physical blocks shared between
 * sequences).  Reference counted; an allocation takes the lowest free ids in
 * increasing order (a deterministic policy: the pages fix none). */
typedef struct pa_allocator pa_allocator;

/* NULL on bad arguments (num_blocks < 0, block_size <= 0) or out of memory. */
pa_allocator* pa_allocator_create(int num_blocks, int block_size);
/* Releases the allocator (deferred while prefix caches created on it remain,
 * see pa_prefix_cache_destroy). */
void pa_allocator_destroy(pa_allocator* a);
/* n blocks, all or nothing; ids written to out_ids[0..n-1].  PA_ERR_OOM if
 * fewer than n are free (nothing taken). */
pa_status pa_block_alloc(pa_allocator* a, int n, int32_t* out_ids);
/* Drop one reference per listed id; a block is free again at zero.  Any id
 * out of range or without enough references: PA_ERR_INVALID and no change. */
pa_status pa_block_free(pa_allocator* a, const int32_t* ids, int n);
/* Take one more reference per listed id (prefix sharing, [P3] "KV Cache
 * Management": 100 requests sharing one system prompt).  Every id must be
 * allocated; otherwise PA_ERR_INVALID and no change. */
pa_status pa_block_share(pa_allocator* a, const int32_t* ids, int n);
/* Fault injection for host-side failure tests ([P1] "KV cache memory math"
 * and [P2] "Static versus continuous scheduling": a request is refused when
 * the pool cannot hold its blocks): the n-th later pa_block_alloc call on this
 * allocator that asks for at least one block fails with PA_ERR_OOM and takes
 * nothing, whatever is free; that includes the allocations made inside
 * pa_block_cow, pa_seq_admit, pa_seq_append_slot and pa_sched_continuous_kv.
 * One shot: later calls succeed as usual.  n <= 0 disarms it.  PA_ERR_INVALID
 * for a NULL allocator. */
pa_status pa_allocator_fail_nth_alloc(pa_allocator* a, int64_t n);
int pa_allocator_num_free(const pa_allocator* a);
int pa_allocator_num_blocks(const pa_allocator* a);
int pa_allocator_block_size(const pa_allocator* a);
/* References held on block id (0 = free); -1 if id is out of range. */
int pa_allocator_refcount(const pa_allocator* a, int32_t id);

/* Multi-query attention over the paged cache: a prefill chunk ([P1] "3.
 * Chunked prefill": a long prompt is processed a chunk at a time, each chunk
 * attending to the cache that holds the earlier chunks) or a speculative
 * verification pass ([P2] "Speculative decoding": the target model scores
 * the K proposed tokens in one pass).
 *
 * Sequence b has C_b = q_start[b+1] - q_start[b] query tokens, which are the
 * last C_b of its seq_lens[b] cached positions: query token i of the
 * sequence sits at position seq_lens[b] - C_b + i and attends to positions
 * 0 .. that position.  The chunk's own K/V must already be in the cache
 * (pa_kv_append with its slots).  Query head i uses kv head i / G.
 *
 *   out, q        bf16 [total_q][num_q_heads][head_dim], total_q = q_start[batch];
 *                 sequence b's rows start at q_start[b]
 *   q_start       device int32 [batch + 1], non-decreasing, q_start[0] = 0
 *   max_q_len     host bound on every C_b (sizes the grid)
 *   other arguments as for pa_decode_attention (no workspace).
 *
 * Every cache type (bf16, e4m3, int8, int4; the coded ones with k_scale /
 * v_scale, PA_ERR_INVALID without) at head_dim 128, block_size 16 or 32, G
 * dividing 128 (PA_ERR_UNSUPPORTED otherwise).  A coded cache's codes are
 * expanded exactly to f16 and the tensor cores then take q and the
 * probabilities as f16 too, so q must lie in the f16 range (|q| < 65504).
 * A sequence with C_b < 0, C_b > seq_lens[b],
 * seq_lens[b] > max_blocks_per_seq * block_size or C_b > max_q_len is
 * skipped (PA_DEVERR_SEQ_LEN); out-of-range block ids raise
 * PA_DEVERR_BLOCK_ID and leave that sequence's outputs unspecified (finite).
 * Enqueued on `stream`; no allocation, no synchronisation. */
pa_status pa_prefill_attention(void* out, const void* q, const void* k_cache, const void* v_cache,
                               const float* k_scale, const float* v_scale, const int32_t* block_tables,
                               const int32_t* seq_lens, const int32_t* q_start, int batch, int num_q_heads,
                               int num_kv_heads, int head_dim, int block_size, int max_blocks_per_seq,
                               int num_blocks, int max_q_len, float scale, int kv_dtype, void* stream);

/* ---------------------------------------------------------------------------
 * Prefix cache and copy-on-write ([P1] "4. Prefix caching": a shared prefix's
 * KV is computed once and reused, vLLM hashing prefix blocks, a radix tree
 * sharing any common prefix; [P3] "KV Cache Management": 100 requests with
 * one system prompt share its KV; [P2] "KV memory, paging and prefix
 * identity": reuse requires the exact token prefix).
 *
 * Block j of a sequence (tokens [j*bs, (j+1)*bs)) is cached under the whole
 * token prefix [0, (j+1)*bs): two sequences share it exactly when those
 * tokens agree.  Only full blocks are cached; the cache holds one reference
 * on each block it lists (on the allocator it was created with).
 * The cache keeps a clock that every match and insert call advances by one;
 * an entry's last use is the clock of the last call that matched or
 * inserted it.
 * ------------------------------------------------------------------------- */
typedef struct pa_prefix_cache pa_prefix_cache;

pa_prefix_cache* pa_prefix_cache_create(pa_allocator* a);
/* Drops the cache's references.  Caches and their allocator may be destroyed
 * in any order: an allocator destroyed while caches created on it remain is
 * released when the last of them is destroyed. */
void pa_prefix_cache_destroy(pa_prefix_cache* c);
int pa_prefix_cache_size(const pa_prefix_cache* c);
/* The longest cached prefix of tokens[0..n_tokens): the physical blocks of
 * its first *n_blocks full blocks (at most max_out) are written to out_blocks
 * and the caller receives one reference on each. */
pa_status pa_prefix_match(pa_prefix_cache* c, const int32_t* tokens, int64_t n_tokens, int32_t* out_blocks,
                          int max_out, int* n_blocks);
/* Registers the full blocks of a sequence: blocks[j] holds tokens
 * [j*bs, (j+1)*bs) of tokens[0..n_tokens).  A prefix already cached keeps its
 * existing block; each new entry takes one reference.  Every listed block
 * must be allocated (PA_ERR_INVALID otherwise, nothing changed). */
pa_status pa_prefix_insert(pa_prefix_cache* c, const int32_t* tokens, int64_t n_tokens, const int32_t* blocks,
                           int n_blocks);
/* Frees up to `want` cached blocks, one at a time, each time taking among
 * the entries that end a chain (no cached entry continues them) and that no
 * sequence references any more (refcount 1: only the cache holds them) the
 * least recently used, then the deepest, then the lowest block id.  Freeing
 * a chain's end can make its parent eligible.  *freed = count. */
pa_status pa_prefix_evict(pa_prefix_cache* c, int want, int* freed);

/* Copy-on-write of one block the caller holds a reference on, before the
 * caller writes into it: if the caller is its only user (refcount 1) the
 * block is returned as it is (*needs_copy = 0); otherwise a fresh block is
 * allocated (lowest free id), the caller's reference moves from `block` to
 * it and *needs_copy = 1: the caller then copies the data with
 * pa_copy_blocks.  PA_ERR_OOM if no block is free (nothing changed). */
pa_status pa_block_cow(pa_allocator* a, int32_t block, int32_t* out_block, int* needs_copy);

/* Admit a sequence of n_tokens tokens ([P1] "2. PagedAttention" and "4.
 * Prefix caching"): blocks[0 .. *n_blocks) receives
 * pa_blocks_for_tokens(n_tokens, bs) physical blocks, first the longest
 * cached prefix of `tokens` (pa_prefix_match; c may be NULL: no reuse), then
 * fresh blocks (lowest free ids).  When the pool is short, blocks only the
 * cache still references are evicted first (pa_prefix_evict).  The caller
 * holds one reference on each listed block.  *first_new_pos = the first
 * position whose KV the caller must still write (matched blocks x bs).
 * All or nothing: PA_ERR_OOM leaves the allocator and cache references as
 * they were (*n_blocks = 0).  PA_ERR_INVALID if the blocks needed exceed
 * max_blocks, c belongs to another allocator, or a pointer is NULL. */
pa_status pa_seq_admit(pa_allocator* a, pa_prefix_cache* c, const int32_t* tokens, int64_t n_tokens,
                       int32_t* blocks, int max_blocks, int* n_blocks, int64_t* first_new_pos);

/* Reserve the slot of token position `pos` in a sequence holding
 * blocks[0 .. *n_blocks) (capacity max_blocks).  If pos opens a new block
 * (pos / bs == *n_blocks) a fresh block is appended (*n_blocks grows by one);
 * otherwise the block holding pos goes through pa_block_cow, and when it was
 * shared, blocks[] names the private copy and *copy_src / *copy_dst the page
 * copy the caller must run (pa_copy_blocks) before writing the slot (both -1
 * when no copy is needed).  *slot = block * bs + pos % bs.  A pool that is
 * short first gives up blocks only the cache references (c may be NULL).
 * PA_ERR_OOM if no block can be had (nothing changed); PA_ERR_INVALID if
 * pos < 0, pos / bs > *n_blocks or pos / bs >= max_blocks. */
pa_status pa_seq_append_slot(pa_allocator* a, pa_prefix_cache* c, int32_t* blocks, int* n_blocks, int max_blocks,
                             int64_t pos, int64_t* slot, int32_t* copy_src, int32_t* copy_dst);

/* Device copy of whole blocks: for i < n, block dst[i] (every kv head's K and
 * V page, and for a coded cache both scales) becomes a copy of block src[i].
 * src / dst are device int32 arrays; no dst may appear as a src of the same
 * call.  Ids out of range are skipped (PA_DEVERR_BLOCK_ID).  Same layout
 * rules as pa_kv_append. */
pa_status pa_copy_blocks(void* k_cache, void* v_cache, float* k_scale, float* v_scale, const int32_t* src,
                         const int32_t* dst, int n, int num_blocks, int num_kv_heads, int head_dim,
                         int block_size, int kv_dtype, void* stream);

/* Blocks needed for `tokens` tokens: ceil(tokens / block_size) ([P1] "Visual:
 * the lifecycle of a request": 50 tokens use 4 blocks, 5000 use 313).
 * 0 for tokens <= 0 or block_size <= 0. */
int64_t pa_blocks_for_tokens(int64_t tokens, int block_size);

/* KV-cache bytes: 2 x layers x kv_heads x head_dim x tokens x batch x
 * dtype_bits / 8 ([P1] "KV cache memory math"; [P2] "KV memory, paging and
 * prefix identity": GQA/MQA count KV heads).  dtype_bits 16 for bf16/fp16, 8
 * for fp8/int8, 4 for int4.  Returns 0 if an argument is negative. */
uint64_t pa_kv_bytes(int layers, int kv_heads, int head_dim, int dtype_bits, int64_t tokens,
                     int64_t batch);

/* slots[t] = block_tables[seq_ids[t]][positions[t] / block_size] * block_size
 *            + positions[t] % block_size
 * ([P1] "2. PagedAttention": the table maps logical positions to physical
 * blocks).  PA_ERR_INVALID if a position is negative or beyond the table. */
pa_status pa_slot_mapping(const int32_t* block_tables, int max_blocks_per_seq,
                          const int32_t* seq_ids, const int32_t* positions, int num_tokens,
                          int block_size, int64_t* slots);

/* The slot of each sequence's new token in a decode step: position
 * seq_lens[b] - 1 (the new token counts in its sequence's length), mapped as
 * pa_slot_mapping maps it ([P1] "2. PagedAttention").  slots[b] = -1 where
 * seq_lens[b] <= 0 (the sequence gets no token; pa_kv_append skips it).
 * block_tables [batch][max_blocks_per_seq] and seq_lens [batch] are host
 * arrays; slots [batch] is written by the call.  PA_ERR_INVALID if a
 * position lies beyond its table row or an argument is bad. */
pa_status pa_step_slots(const int32_t* block_tables, int max_blocks_per_seq, const int32_t* seq_lens, int batch,
                        int block_size, int64_t* slots);

/* Unit-time scheduler simulator ([P2] "Static versus continuous scheduling"
 * and "Hands-on"): mode 0 = static cohorts of `slots` requests (each cohort
 * lasts as long as its longest member), mode 1 = iteration-level (a freed
 * slot is refilled before the next iteration).  out_lens are the requests'
 * output lengths in arrival order.  Requires slots > 0 and out_lens > 0
 * (zero slots would never finish): otherwise PA_ERR_INVALID.  n == 0 gives
 * 0 iterations.  [5,20,10,15,10] with 3 slots: 35 static, 20 continuous. */
pa_status pa_sched_simulate(const int64_t* out_lens, int n, int slots, int mode, int64_t* iters);

/* Iteration-level scheduler with KV admission ([P1] "1. Continuous
 * (iteration-level) batching": admit while KV blocks remain, decode one
 * token for every active request, free a finished request's blocks at once;
 * [P1] "Pitfalls" 1 and 5: a request is admitted only when its reserved
 * tokens fit, at most max_num_seqs run at once).
 * Request r needs prompt_lens[r] + out_lens[r] tokens; admission reserves
 * blocks for them all (pa_blocks_for_tokens) from `a`, in arrival order, and
 * the head of the queue blocks later ones when it does not fit.  Runs until
 * every request has finished or until `stop_iter` iterations (stop_iter < 0:
 * run to the end).  Outputs (may be NULL): *iters = iterations run;
 * admitted_at[r] / finished_at[r] = iteration of admission / completion
 * (-1 if not reached); tables (n x max_blocks_per_seq, -1 padded) and
 * lens (tokens held) of the requests still active when it stops.
 * PA_ERR_INVALID on bad arguments or if a single request can never fit.  A
 * reservation the pool refuses although the blocks looked free (see
 * pa_allocator_fail_nth_alloc) leaves the request at the head of the queue
 * for the next iteration; PA_ERR_OOM if no request is running then (every
 * block this call took has been returned). */
pa_status pa_sched_continuous_kv(pa_allocator* a, const int64_t* prompt_lens,
                                 const int64_t* out_lens, int n, int max_num_seqs,
                                 int64_t stop_iter, int max_blocks_per_seq, int64_t* iters,
                                 int64_t* admitted_at, int64_t* finished_at, int32_t* tables,
                                 int32_t* lens);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDATTN_PA_H */
