/*
 * Plain CPU oracle for single-token decode attention over a paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline / reference arm load this file's library.  It
 * shares no code, header, table or constant with the CUDA library; the two
 * are written separately from the same definitions.
 *
 * Everything here is the slow, obvious form of each definition: loops in
 * logical order, fp64 for attention arithmetic, fp32 only where the encoding
 * itself is defined in fp32 (the fp8 append's scale and quotient).
 *
 * Sources (pages of the subject, cited by title and section):
 *   [P1] "KV cache & continuous batching" (docs.masst.dev/ai/inference/kv-cache-batching)
 *   [P2] "LLM Serving - KV Cache, Batching, Speculative Decoding"
 *        (dineshblog.com/blog/session-124-llm-serving)
 *   [P3] "LLM Inference Optimization: KV Cache, Batching, and Speculative
 *        Decoding" (adaptiverecall.com/open-source-llms/inference-optimization.php)
 *
 * Cache layout shared by both implementations (it is an interface, not
 * arithmetic): k_cache / v_cache are [num_blocks][Hkv][block_size][d]
 * elements: bf16 bit patterns, e4m3 or int8 codes (one byte each) or int4
 * codes (two per byte, a row taking d / 2 bytes); the scales of the coded
 * caches are [num_blocks][Hkv] fp32.  block_tables is [B][M] int32, row b listing the physical block of
 * logical block j of sequence b.
 *
 * Build: gcc -O2 -std=c99 -fPIC -shared -ffp-contract=off pa_oracle.c -lm
 * (-ffp-contract=off keeps every fp32 product and quotient separately rounded.)
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_OK 0
#define OR_ERR -1

/* ------------------------------------------------------------------------ */
/* Number formats                                                            */
/* ------------------------------------------------------------------------ */

/* bfloat16 is the upper 16 bits of an IEEE binary32; widening is exact. */
double or_bf16_value(uint16_t bits) {
    uint32_t w = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

static float bf16_to_float(uint16_t bits) {
    uint32_t w = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return f;
}

/* OCP 8-bit floating point, E4M3: 1 sign, 4 exponent (bias 7), 3 mantissa
 * bits.  Exponent field 0 is subnormal: m * 2^-9.  S.1111.111 is NaN; there
 * is no infinity, so the largest finite magnitude is 1.75 * 2^8 = 448.
 * The fp8 cache follows [P1] "KV cache memory math" (1 byte per element for
 * fp8) and [P3] "Memory Bandwidth Optimization" (KV cache quantization). */
double or_e4m3_value(uint8_t code) {
    int s = code >> 7;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double v;
    if (e == 0xF && m == 0x7) return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp(1.0 + m / 8.0, e - 7);
    return s ? -v : v;
}

/* Round a binary32 value to E4M3: round to nearest, ties to even, magnitudes
 * beyond 448 saturate to 448 (no infinity exists), NaN maps to 0x7F.  The
 * sign of zero is kept.  All steps are exact in double except the final
 * rint(), which rounds half to even under the default rounding mode. */
uint8_t or_e4m3_encode(float x) {
    double a;
    int s, ex;
    double q;
    int code;
    if (isnan(x)) return 0x7F;
    s = signbit(x) ? 1 : 0;
    a = fabs((double)x);
    if (a >= 448.0) return (uint8_t)((s << 7) | 0x7E);
    if (a < ldexp(1.0, -6)) {
        /* subnormal range: multiples of 2^-9; 8 * 2^-9 is the first normal */
        q = rint(a * 512.0);
        code = (int)q; /* 0..8; 8 encodes 2^-6 = exponent 1, mantissa 0 */
    } else {
        double mant;
        frexp(a, &ex);          /* a = f * 2^ex, f in [0.5, 1) */
        ex -= 1;                /* a = mant * 2^ex, mant in [1, 2) */
        mant = ldexp(a, -ex);
        q = rint((mant - 1.0) * 8.0);
        if (q >= 8.0) { q = 0.0; ex += 1; }
        code = ((ex + 7) << 3) | (int)q;
        if (code > 0x7E) code = 0x7E;
    }
    return (uint8_t)((s << 7) | code);
}

/* int8 cache ([P3] "Memory Bandwidth Optimization": INT8 KV quantization):
 * a code c in [-127, 127] stands for c * scale.  Encoding rounds a binary32
 * quotient to the nearest integer, ties to even (rint under the default
 * rounding mode), and clamps to +-127; NaN maps to 0.  Codes are stored as
 * two's-complement bytes. */
double or_int8_value(uint8_t code) { return (double)(int8_t)code; }

uint8_t or_int8_encode(float x) {
    double q;
    if (isnan(x)) return 0;
    q = rint((double)x);
    if (q > 127.0) q = 127.0;
    if (q < -127.0) q = -127.0;
    return (uint8_t)(int8_t)q;
}

/* int4 cache ([P1] "KV cache memory math": half a byte per element for
 * int4): a code c in [-7, 7] stands for c * scale, the symmetric range, like
 * int8's [-127, 127].  Encoding as for int8, clamped to +-7.  A code is a
 * 4-bit two's-complement nibble; element 2j of a row sits in the low nibble
 * of the row's byte j and element 2j+1 in its high nibble. */
double or_int4_value(uint8_t nibble) {
    int v = nibble & 0xF;
    return (double)(v >= 8 ? v - 16 : v);
}

uint8_t or_int4_encode(float x) {
    double q;
    if (isnan(x)) return 0;
    q = rint((double)x);
    if (q > 7.0) q = 7.0;
    if (q < -7.0) q = -7.0;
    return (uint8_t)((int)q & 0xF);
}

/* The scaled codecs: 1 = e4m3 (largest code value 448), 2 = int8 (127),
 * 3 = int4 (7). */
static double q8_value(int codec, uint8_t c) {
    return codec == 3 ? or_int4_value(c) : codec == 2 ? or_int8_value(c) : or_e4m3_value(c);
}
static uint8_t q8_encode(int codec, float x) {
    return codec == 3 ? or_int4_encode(x) : codec == 2 ? or_int8_encode(x) : or_e4m3_encode(x);
}
static float q8_max(int codec) { return codec == 3 ? 7.0f : codec == 2 ? 127.0f : 448.0f; }

/* Bytes of one token row of one head: d for one-byte codes, d / 2 for int4. */
static int64_t row_bytes(int codec, int d) { return codec == 3 ? d / 2 : d; }

/* The code of element i of row o of a page, and its update. */
static uint8_t page_get(const uint8_t* page, int codec, int d, int o, int i) {
    if (codec == 3) {
        uint8_t b = page[(int64_t)o * (d / 2) + i / 2];
        return (uint8_t)((i & 1) ? (b >> 4) : (b & 0xF));
    }
    return page[(int64_t)o * d + i];
}

static void page_set(uint8_t* page, int codec, int d, int o, int i, uint8_t c) {
    if (codec == 3) {
        uint8_t* b = page + (int64_t)o * (d / 2) + i / 2;
        *b = (i & 1) ? (uint8_t)((*b & 0x0F) | ((c & 0xF) << 4)) : (uint8_t)((*b & 0xF0) | (c & 0xF));
        return;
    }
    page[(int64_t)o * d + i] = c;
}

/* ------------------------------------------------------------------------ */
/* Accounting: [P1] "KV cache memory math" and [P2] "KV memory, paging and   */
/* prefix identity": bytes = 2 x layers x kv_heads x head_dim x tokens x     */
/* batch x bytes-per-element (dtype given in bits so int4 is exact).        */
/* ------------------------------------------------------------------------ */
uint64_t or_kv_bytes(int64_t layers, int64_t kv_heads, int64_t head_dim, int64_t dtype_bits,
                     int64_t tokens, int64_t batch) {
    uint64_t bits = 2ull * (uint64_t)layers * (uint64_t)kv_heads * (uint64_t)head_dim *
                    (uint64_t)tokens * (uint64_t)batch * (uint64_t)dtype_bits;
    return bits / 8ull;
}

/* [P1] "Visual: the lifecycle of a request": memory is allocated per block of
 * block_size tokens; a request of n tokens holds the smallest number of
 * blocks whose capacity covers n. */
int64_t or_blocks_for_tokens(int64_t tokens, int64_t block_size) {
    int64_t n = 0;
    if (tokens <= 0 || block_size <= 0) return 0;
    while (n * block_size < tokens) n++;
    return n;
}

/* ------------------------------------------------------------------------ */
/* Scheduler simulator: [P2] "Static versus continuous scheduling" and the   */
/* hands-on program.  Unit-time iterations; each request needs lens[i]       */
/* iterations of one token each.                                             */
/* ------------------------------------------------------------------------ */

/* Both simulators take the hands-on program's stated domain: a positive
 * slot count and positive output lengths (zero slots would never finish);
 * anything else is rejected.  An empty request list takes zero ticks. */
static int sched_args_ok(const int64_t* lens, int n, int slots) {
    int i;
    if (slots <= 0 || n < 0) return 0;
    for (i = 0; i < n; i++)
        if (lens[i] <= 0) return 0;
    return 1;
}

/* Static cohorts: consecutive groups of `slots` requests run together and the
 * group lasts as long as its longest member. */
int or_sched_static(const int64_t* lens, int n, int slots, int64_t* iters) {
    int64_t total = 0;
    int i, j;
    if (!sched_args_ok(lens, n, slots)) return OR_ERR;
    for (i = 0; i < n; i += slots) {
        int64_t mx = 0;
        for (j = i; j < n && j < i + slots; j++)
            if (lens[j] > mx) mx = lens[j];
        total += mx;
    }
    *iters = total;
    return OR_OK;
}

/* Iteration-level: before every tick, free slots are refilled from the
 * waiting requests in arrival order; every active request then advances one
 * token and leaves when its last token is produced. */
int or_sched_continuous(const int64_t* lens, int n, int slots, int64_t* iters) {
    int64_t* remaining;
    int next = 0, active = 0, i;
    int64_t ticks = 0;
    if (!sched_args_ok(lens, n, slots)) return OR_ERR;
    if (n == 0) { *iters = 0; return OR_OK; }
    remaining = (int64_t*)calloc((size_t)n, sizeof(int64_t));
    if (!remaining) return OR_ERR;
    for (;;) {
        /* admit */
        while (next < n && active < slots) {
            remaining[next] = lens[next];
            active++;
            next++;
        }
        if (active == 0 && next >= n) break;
        /* one iteration: every active request emits one token */
        for (i = 0; i < next; i++) {
            if (remaining[i] > 0) {
                remaining[i]--;
                if (remaining[i] == 0) active--;
            }
        }
        ticks++;
    }
    free(remaining);
    *iters = ticks;
    return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* Block allocator: [P1] "2. PagedAttention" (fixed-size blocks, allocated on */
/* demand, freed when done, not contiguous) and [P2] "KV memory, paging and   */
/* prefix identity" (physical blocks may be shared).  Policy (the pages fix   */
/* none): reference counted; an allocation takes the lowest free ids in      */
/* increasing order, all or nothing.                                          */
/* ------------------------------------------------------------------------ */
typedef struct {
    int n;
    int* refcnt;
} or_alloc;

or_alloc* or_alloc_create(int num_blocks) {
    or_alloc* a;
    if (num_blocks < 0) return NULL;
    a = (or_alloc*)malloc(sizeof(or_alloc));
    if (!a) return NULL;
    a->n = num_blocks;
    a->refcnt = (int*)calloc((size_t)(num_blocks > 0 ? num_blocks : 1), sizeof(int));
    if (!a->refcnt) { free(a); return NULL; }
    return a;
}

void or_alloc_destroy(or_alloc* a) {
    if (!a) return;
    free(a->refcnt);
    free(a);
}

int or_alloc_num_free(const or_alloc* a) {
    int i, c = 0;
    for (i = 0; i < a->n; i++)
        if (a->refcnt[i] == 0) c++;
    return c;
}

/* returns 0, or -1 (invalid) / -2 (not enough free blocks; nothing taken) */
int or_alloc_alloc(or_alloc* a, int n, int32_t* out) {
    int i, k = 0;
    if (n < 0) return -1;
    if (or_alloc_num_free(a) < n) return -2;
    for (i = 0; i < a->n && k < n; i++) {
        if (a->refcnt[i] == 0) {
            a->refcnt[i] = 1;
            out[k++] = i;
        }
    }
    return 0;
}

/* drop one reference per listed id; a block returns to the free set at 0.
 * Any id out of range or not allocated: -1 and no change at all. */
int or_alloc_free(or_alloc* a, const int32_t* ids, int n) {
    int i, j, cnt;
    for (i = 0; i < n; i++) {
        if (ids[i] < 0 || ids[i] >= a->n) return -1;
        cnt = 0;
        for (j = 0; j < n; j++)
            if (ids[j] == ids[i]) cnt++;
        if (a->refcnt[ids[i]] < cnt) return -1;
    }
    for (i = 0; i < n; i++) a->refcnt[ids[i]]--;
    return 0;
}

/* take one more reference per listed id (prefix sharing) */
int or_alloc_share(or_alloc* a, const int32_t* ids, int n) {
    int i;
    for (i = 0; i < n; i++)
        if (ids[i] < 0 || ids[i] >= a->n || a->refcnt[ids[i]] == 0) return -1;
    for (i = 0; i < n; i++) a->refcnt[ids[i]]++;
    return 0;
}

int or_alloc_refcount(const or_alloc* a, int id) {
    if (id < 0 || id >= a->n) return -1;
    return a->refcnt[id];
}

/* ------------------------------------------------------------------------ */
/* Slot of a token: [P1] "2. PagedAttention": the block table maps a logical  */
/* position to its physical block; position p of a sequence lives in logical  */
/* block p / bs at offset p mod bs, so slot = table[p / bs] * bs + p mod bs.  */
/* ------------------------------------------------------------------------ */
int or_slot_mapping(const int32_t* tables, int M, const int32_t* seq, const int32_t* pos, int T,
                    int bs, int64_t* slots) {
    int i;
    for (i = 0; i < T; i++) {
        int j = pos[i] / bs;
        if (pos[i] < 0 || j >= M) return -1;
        slots[i] = (int64_t)tables[(int64_t)seq[i] * M + j] * bs + pos[i] % bs;
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* KV append: [P2] "Recall and stretch" item 3 (keys/values written in      */
/* prefill and appended in decode) and [P1] "The core insight" (decode       */
/* computes only the new token's K/V).  Token t, head h goes to              */
/* cache[slot / bs][h][slot mod bs][:]; a negative slot means "skip".        */
/* ------------------------------------------------------------------------ */
int or_kv_append_bf16(uint16_t* k_cache, uint16_t* v_cache, const uint16_t* k_new,
                      const uint16_t* v_new, const int64_t* slots, int T, int64_t num_blocks,
                      int Hkv, int d, int bs) {
    int t, h, i;
    for (t = 0; t < T; t++) {
        int64_t blk, off;
        if (slots[t] < 0) continue;
        blk = slots[t] / bs;
        off = slots[t] % bs;
        if (blk >= num_blocks) return -1;
        for (h = 0; h < Hkv; h++) {
            int64_t dst = ((blk * Hkv + h) * bs + off) * d;
            int64_t src = ((int64_t)t * Hkv + h) * d;
            for (i = 0; i < d; i++) {
                k_cache[dst + i] = k_new[src + i];
                v_cache[dst + i] = v_new[src + i];
            }
        }
    }
    return 0;
}

/* fp8 append with one fp32 absmax scale per (block, kv_head), applied to K
 * and V separately.  For every block p that this call writes (tokens W, first
 * offset f = smallest offset written):
 *   old = 0 if f == 0 (the block starts afresh) else scale[p][h]
 *   a   = max |x| over the new values (fp32)
 *   s   = max(old, a / 448)               (fp32 quotient)
 *   if s > old > 0: each older entry e at offset < f becomes
 *          E4M3( fp32( value(e) * old ) / s )
 *   each new value x becomes E4M3(x / s), or +0 when s == 0
 *   scale[p][h] = s
 * so that the block's scale is always its absmax / 448 and no stored code
 * saturates by more than rounding.  448 is the largest finite E4M3 value. */
static void q8_block_head(int codec, uint8_t* cache, float* scale, const uint16_t* src,
                          const int64_t* slots, const int* toks, int ntok, int64_t p, int h, int Hkv,
                          int d, int bs, int first) {
    float old, a = 0.0f, s;
    int k, i, o;
    int64_t sidx = p * Hkv + h;
    uint8_t* page = cache + (p * Hkv + h) * (int64_t)bs * row_bytes(codec, d);
    old = (first == 0) ? 0.0f : scale[sidx];
    for (k = 0; k < ntok; k++) {
        const uint16_t* x = src + ((int64_t)toks[k] * Hkv + h) * d;
        for (i = 0; i < d; i++) {
            float v = fabsf(bf16_to_float(x[i]));
            if (v > a) a = v;
        }
    }
    s = a / q8_max(codec);
    if (old > s) s = old;
    if (s > old && old > 0.0f) {
        for (o = 0; o < first; o++)
            for (i = 0; i < d; i++) {
                float prod = (float)q8_value(codec, page_get(page, codec, d, o, i)) * old;
                page_set(page, codec, d, o, i, q8_encode(codec, prod / s));
            }
    }
    for (k = 0; k < ntok; k++) {
        const uint16_t* x = src + ((int64_t)toks[k] * Hkv + h) * d;
        int64_t off = slots[toks[k]] % bs;
        for (i = 0; i < d; i++)
            page_set(page, codec, d, (int)off, i,
                     (s == 0.0f) ? (uint8_t)0 : q8_encode(codec, bf16_to_float(x[i]) / s));
    }
    scale[sidx] = s;
}

static int q8_append(int codec, uint8_t* k_cache, uint8_t* v_cache, float* k_scale, float* v_scale,
                     const uint16_t* k_new, const uint16_t* v_new, const int64_t* slots, int T,
                     int64_t num_blocks, int Hkv, int d, int bs) {
    int t, u, h;
    int* toks = (int*)malloc(sizeof(int) * (size_t)(T > 0 ? T : 1));
    char* done = (char*)calloc((size_t)(T > 0 ? T : 1), 1);
    if (!toks || !done) { free(toks); free(done); return -1; }
    for (t = 0; t < T; t++)
        if (slots[t] >= 0 && slots[t] / bs >= num_blocks) { free(toks); free(done); return -1; }
    for (t = 0; t < T; t++) {
        int64_t p;
        int n = 0, first;
        if (done[t] || slots[t] < 0) continue;
        p = slots[t] / bs;
        first = bs;
        /* gather every token of this call that lands in block p */
        for (u = t; u < T; u++) {
            if (!done[u] && slots[u] >= 0 && slots[u] / bs == p) {
                toks[n++] = u;
                done[u] = 1;
                if ((int)(slots[u] % bs) < first) first = (int)(slots[u] % bs);
            }
        }
        for (h = 0; h < Hkv; h++) {
            q8_block_head(codec, k_cache, k_scale, k_new, slots, toks, n, p, h, Hkv, d, bs, first);
            q8_block_head(codec, v_cache, v_scale, v_new, slots, toks, n, p, h, Hkv, d, bs, first);
        }
    }
    free(toks);
    free(done);
    return 0;
}

int or_kv_append_fp8(uint8_t* k_cache, uint8_t* v_cache, float* k_scale, float* v_scale,
                     const uint16_t* k_new, const uint16_t* v_new, const int64_t* slots, int T,
                     int64_t num_blocks, int Hkv, int d, int bs) {
    return q8_append(1, k_cache, v_cache, k_scale, v_scale, k_new, v_new, slots, T, num_blocks, Hkv, d, bs);
}

/* The same rule for the int8 cache: s = max(old, fp32(absmax) / 127), codes
 * clamp(rint(x / s), -127, 127), older codes re-encoded as
 * clamp(rint(fp32(c * old) / s)) when s grows. */
int or_kv_append_int8(uint8_t* k_cache, uint8_t* v_cache, float* k_scale, float* v_scale,
                      const uint16_t* k_new, const uint16_t* v_new, const int64_t* slots, int T,
                      int64_t num_blocks, int Hkv, int d, int bs) {
    return q8_append(2, k_cache, v_cache, k_scale, v_scale, k_new, v_new, slots, T, num_blocks, Hkv, d, bs);
}

/* The same rule for the int4 cache with 7 in place of 127: s = max(old,
 * fp32(absmax) / 7), codes clamp(rint(x / s), -7, 7), two per byte.  A row's
 * d codes fill d / 2 bytes (d even). */
int or_kv_append_int4(uint8_t* k_cache, uint8_t* v_cache, float* k_scale, float* v_scale,
                      const uint16_t* k_new, const uint16_t* v_new, const int64_t* slots, int T,
                      int64_t num_blocks, int Hkv, int d, int bs) {
    if (d % 2) return -1;
    return q8_append(3, k_cache, v_cache, k_scale, v_scale, k_new, v_new, slots, T, num_blocks, Hkv, d, bs);
}

/* ------------------------------------------------------------------------ */
/* Decode attention: [P1] "The core insight" (the new token's query attends  */
/* over all cached keys and values), [P2] "Hands-on" (cached attention of    */
/* position t: softmax(q . K^T * scale) . V, equal to the last row of causal */
/* attention), [P1] "2. PagedAttention" (K and V gathered through the block  */
/* table), [P1] "KV cache memory math" / [P3] "Memory Bandwidth              */
/* Optimization" (GQA: several query heads share one KV head).               */
/*                                                                           */
/* Query head i of a sequence uses KV head i / G, G = Hq / Hkv (consecutive  */
/* query heads share a KV head; the pages do not fix the mapping).  Token t  */
/* of sequence b is row t mod bs of physical block table[b][t / bs].  For    */
/* the fp8 / int8 / int4 cache an element's value is value(code) *          */
/* scale[block][head]; the attention functions' `fp8` argument is the cache  */
/* type: 0 bf16, 1 e4m3, 2 int8, 3 int4.                                     */
/* A sequence of length 0 yields a zero output row.                          */
/* ------------------------------------------------------------------------ */
static double kv_elem(const void* cache, const float* sc, int fp8, int64_t blk, int h, int off,
                      int i, int Hkv, int d, int bs) {
    int64_t idx = ((blk * Hkv + h) * bs + off) * (int64_t)d + i;
    if (fp8) {
        const uint8_t* page = (const uint8_t*)cache + (blk * Hkv + h) * (int64_t)bs * row_bytes(fp8, d);
        return q8_value(fp8, page_get(page, fp8, d, off, i)) * (double)sc[blk * Hkv + h];
    }
    return or_bf16_value(((const uint16_t*)cache)[idx]);
}

/* Attention of one query head over tokens [t0, t1) of one sequence.
 * Writes the softmax-weighted sum of the values into acc[d] and returns the
 * log-sum-exp (natural log) of the scaled scores; -INFINITY when empty. */
static double attend_range(double* acc, const uint16_t* qrow, const void* k_cache,
                           const void* v_cache, const float* k_scale, const float* v_scale,
                           const int32_t* table, int h, int Hkv, int d, int bs, double scale,
                           int fp8, int t0, int t1, int64_t num_blocks, int* bad) {
    int n = t1 - t0, t, i;
    double* s;
    double m = -INFINITY, l = 0.0;
    for (i = 0; i < d; i++) acc[i] = 0.0;
    if (n <= 0) return -INFINITY;
    s = (double*)malloc(sizeof(double) * (size_t)n);
    if (!s) { *bad = 1; return -INFINITY; }
    for (t = t0; t < t1; t++) {
        int64_t blk = table[t / bs];
        double dot = 0.0;
        if (blk < 0 || blk >= num_blocks) { *bad = 1; free(s); return -INFINITY; }
        for (i = 0; i < d; i++)
            dot += or_bf16_value(qrow[i]) * kv_elem(k_cache, k_scale, fp8, blk, h, t % bs, i, Hkv, d, bs);
        s[t - t0] = scale * dot;
        if (s[t - t0] > m) m = s[t - t0];
    }
    for (t = t0; t < t1; t++) {
        int64_t blk = table[t / bs];
        double w = exp(s[t - t0] - m);
        l += w;
        for (i = 0; i < d; i++)
            acc[i] += w * kv_elem(v_cache, v_scale, fp8, blk, h, t % bs, i, Hkv, d, bs);
    }
    free(s);
    for (i = 0; i < d; i++) acc[i] /= l;
    return m + log(l);
}

int or_decode_attention(double* out, const uint16_t* q, const void* k_cache, const void* v_cache,
                        const float* k_scale, const float* v_scale, const int32_t* block_tables,
                        const int32_t* seq_lens, int B, int Hq, int Hkv, int d, int bs, int M,
                        int64_t num_blocks, double scale, int fp8) {
    int b, i, G, bad = 0;
    if (Hkv <= 0 || Hq % Hkv != 0 || d <= 0 || bs <= 0) return -1;
    G = Hq / Hkv;
    for (b = 0; b < B; b++) {
        int len = seq_lens[b];
        if (len > M * bs) return -1;
        for (i = 0; i < Hq; i++) {
            double* o = out + ((int64_t)b * Hq + i) * d;
            attend_range(o, q + ((int64_t)b * Hq + i) * d, k_cache, v_cache, k_scale, v_scale,
                         block_tables + (int64_t)b * M, i / G, Hkv, d, bs, scale, fp8, 0, len,
                         num_blocks, &bad);
            if (bad) return -1;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Multi-query attention over the paged cache: [P1] "3. Chunked prefill" (a  */
/* long prompt is processed a chunk at a time; the chunk's queries attend to */
/* the cache holding the earlier chunks and the chunk itself) and [P2]       */
/* "Speculative decoding" (the target model scores the K proposed tokens in  */
/* one pass).  Sequence b has C_b = q_start[b+1] - q_start[b] query tokens:  */
/* the last C_b of its seq_lens[b] cached positions.  Query token i of the   */
/* sequence sits at position p = seq_lens[b] - C_b + i and attends causally  */
/* to positions 0..p; head mapping and the fp8 value rule as above.  q and   */
/* out are [total queries][Hq][d], sequence b's rows starting at q_start[b]. */
/* ------------------------------------------------------------------------ */
int or_prefill_attention(double* out, const uint16_t* q, const void* k_cache, const void* v_cache,
                         const float* k_scale, const float* v_scale, const int32_t* block_tables,
                         const int32_t* seq_lens, const int32_t* q_start, int B, int Hq, int Hkv, int d,
                         int bs, int M, int64_t num_blocks, double scale, int fp8) {
    int b, i, c, G, bad = 0;
    if (Hkv <= 0 || Hq % Hkv != 0 || d <= 0 || bs <= 0) return -1;
    G = Hq / Hkv;
    for (b = 0; b < B; b++) {
        int len = seq_lens[b], C = q_start[b + 1] - q_start[b];
        if (len > M * bs || C < 0 || C > len) return -1;
        for (c = 0; c < C; c++) {
            int64_t row = (int64_t)q_start[b] + c;
            for (i = 0; i < Hq; i++) {
                attend_range(out + (row * Hq + i) * d, q + (row * Hq + i) * d, k_cache, v_cache, k_scale,
                             v_scale, block_tables + (int64_t)b * M, i / G, Hkv, d, bs, scale, fp8, 0,
                             len - C + c + 1, num_blocks, &bad);
                if (bad) return -1;
            }
        }
    }
    return 0;
}

/* Split-K form of the same quantity (flash-decoding): the tokens of every
 * sequence are cut into contiguous partitions of part_blocks blocks; each
 * partition yields its normalised output o_i and log-sum-exp lse_i, and the
 * partitions combine as  out = sum_i exp(lse_i - L) o_i,  L = log sum_i
 * exp(lse_i).  Empty partitions have lse = -inf and weight 0.  In exact
 * arithmetic this equals or_decode_attention. */
int or_decode_attention_split(double* out, const uint16_t* q, const void* k_cache,
                              const void* v_cache, const float* k_scale, const float* v_scale,
                              const int32_t* block_tables, const int32_t* seq_lens, int B, int Hq,
                              int Hkv, int d, int bs, int M, int64_t num_blocks, double scale,
                              int fp8, int part_blocks) {
    int b, i, G, k, bad = 0, nparts;
    double *po, *plse;
    if (Hkv <= 0 || Hq % Hkv != 0 || part_blocks <= 0) return -1;
    G = Hq / Hkv;
    nparts = (M + part_blocks - 1) / part_blocks;
    if (nparts < 1) nparts = 1;
    po = (double*)malloc(sizeof(double) * (size_t)nparts * (size_t)d);
    plse = (double*)malloc(sizeof(double) * (size_t)nparts);
    if (!po || !plse) { free(po); free(plse); return -1; }
    for (b = 0; b < B; b++) {
        int len = seq_lens[b];
        if (len > M * bs) { free(po); free(plse); return -1; }
        for (i = 0; i < Hq; i++) {
            double* o = out + ((int64_t)b * Hq + i) * d;
            double L = -INFINITY, tot = 0.0;
            for (k = 0; k < nparts; k++) {
                int t0 = k * part_blocks * bs, t1 = (k + 1) * part_blocks * bs;
                if (t1 > len) t1 = len;
                plse[k] = attend_range(po + (int64_t)k * d, q + ((int64_t)b * Hq + i) * d, k_cache,
                                       v_cache, k_scale, v_scale, block_tables + (int64_t)b * M,
                                       i / G, Hkv, d, bs, scale, fp8, t0, t1, num_blocks, &bad);
                if (bad) { free(po); free(plse); return -1; }
                if (plse[k] > L) L = plse[k];
            }
            for (k = 0; k < d; k++) o[k] = 0.0;
            if (L == -INFINITY) continue;
            for (k = 0; k < nparts; k++) {
                double w;
                int c;
                if (plse[k] == -INFINITY) continue;
                w = exp(plse[k] - L);
                tot += w;
                for (c = 0; c < d; c++) o[c] += w * po[(int64_t)k * d + c];
            }
            for (k = 0; k < d; k++) o[k] /= tot;
        }
    }
    free(po);
    free(plse);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Iteration-level scheduling with KV admission: [P1] "1. Continuous        */
/* (iteration-level) batching" (admit while KV memory remains, decode one    */
/* token for every active request in one pass, free a finished request's     */
/* blocks immediately) and [P1] "Pitfalls" 1 and 5 (a request reserves KV    */
/* for its whole budget; admission is refused when it does not fit; at most  */
/* max_seqs requests run).  Request r reserves ceil((prompt+out)/bs) blocks. */
/* Waiting requests are admitted strictly in arrival order.                  */
/* ------------------------------------------------------------------------ */
int or_sched_continuous_kv(or_alloc* a, int bs, const int64_t* prompt, const int64_t* outl, int n,
                           int max_seqs, int64_t stop_iter, int M, int64_t* iters, int64_t* admitted,
                           int64_t* finished, int32_t* tables, int32_t* lens) {
    int r, j, head = 0, active = 0;
    int64_t it = 0;
    int* state;          /* 0 waiting, 1 active, 2 done */
    int64_t* gen;
    int64_t* nblk;
    int32_t* blocks;     /* n x maxb */
    int64_t maxb = 1;
    if (n < 0 || max_seqs <= 0 || bs <= 0) return -1;
    for (r = 0; r < n; r++) {
        int64_t need;
        if (prompt[r] < 0 || outl[r] <= 0) return -1;
        need = or_blocks_for_tokens(prompt[r] + outl[r], bs);
        if (need > a->n || (tables && need > M)) return -1;
        if (need > maxb) maxb = need;
    }
    state = (int*)calloc((size_t)(n > 0 ? n : 1), sizeof(int));
    gen = (int64_t*)calloc((size_t)(n > 0 ? n : 1), sizeof(int64_t));
    nblk = (int64_t*)calloc((size_t)(n > 0 ? n : 1), sizeof(int64_t));
    blocks = (int32_t*)calloc((size_t)(n > 0 ? n : 1) * (size_t)maxb, sizeof(int32_t));
    if (!state || !gen || !nblk || !blocks) { free(state); free(gen); free(nblk); free(blocks); return -1; }
    for (r = 0; r < n; r++) {
        if (admitted) admitted[r] = -1;
        if (finished) finished[r] = -1;
    }
    while ((head < n || active > 0) && (stop_iter < 0 || it < stop_iter)) {
        /* admit from the head of the queue */
        while (head < n && active < max_seqs) {
            int64_t need = or_blocks_for_tokens(prompt[head] + outl[head], bs);
            if (or_alloc_num_free(a) < need) break;
            or_alloc_alloc(a, (int)need, blocks + (int64_t)head * maxb);
            nblk[head] = need;
            state[head] = 1;
            if (admitted) admitted[head] = it;
            active++;
            head++;
        }
        if (active == 0) { free(state); free(gen); free(nblk); free(blocks); return -1; }
        /* one iteration: every active request emits a token */
        for (r = 0; r < n; r++) {
            if (state[r] != 1) continue;
            gen[r]++;
            if (gen[r] >= outl[r]) {
                or_alloc_free(a, blocks + (int64_t)r * maxb, (int)nblk[r]);
                state[r] = 2;
                active--;
                if (finished) finished[r] = it;
            }
        }
        it++;
    }
    if (iters) *iters = it;
    for (r = 0; r < n; r++) {
        if (lens) lens[r] = state[r] == 1 ? (int32_t)(prompt[r] + gen[r]) : 0;
        if (tables)
            for (j = 0; j < M; j++)
                tables[(int64_t)r * M + j] = (state[r] == 1 && j < nblk[r]) ? blocks[(int64_t)r * maxb + j] : -1;
    }
    free(state);
    free(gen);
    free(nblk);
    free(blocks);
    return 0;
}
