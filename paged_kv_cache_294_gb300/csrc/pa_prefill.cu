// Multi-query attention over the paged KV cache on the 5th-generation tensor
// cores: the queries of a prefill chunk ("KV cache & continuous batching",
// section "3. Chunked prefill") or of a speculative-verification pass ("LLM
// Serving - KV Cache, Batching, Speculative Decoding", section "Speculative
// decoding") attend causally to the cache, which already holds the chunk's
// own keys and values.
//
// One CTA computes one tile of 128 query rows of one (sequence, kv head):
// with G query heads per kv head a row is a (token, head) pair, row =
// token * G + head, so the G heads share every K/V tile.  KV is walked in
// tiles of 128 tokens (128 / block_size pages, each page fetched by TMA from
// its physical block with the 128-byte swizzle).
//
//   warp 0      TMA producer of the K tile ring (3 stages), one lane per page
//   warp 18     TMA producer of the V tile ring (3 stages), one lane per page
//   warp 1      owns the tensor memory; one lane issues S[j%2] = Q K_j^T
//   warp 19     one lane issues O += P_j V_j
//               (tcgen05.mma, A operand in tensor memory, B in shared
//               memory: K tile K-major, V tile MN-major; two issuing
//               threads because one cannot keep the tensor core busy with
//               M=128 x N=128 instructions)
//   warps 2-17  softmax: a thread holds one query row (its tensor-memory
//               lane) and a quarter of its columns; keeps the running max
//               m and sum l in fp32 (log2 domain), writes P (bf16) into
//               tensor memory, rescales O only when the max grows by more
//               than 2^8, and finally writes out = O / l.  These warps
//               also place Q in tensor memory at the start.
//
// Coded caches (e4m3, int8, int4 codes with one fp32 scale per (block, kv
// head)): the producers land each page's codes in the upper part of its
// stage, and four more warps (20-23; two for K, two for V) expand them in
// place to exact f16 values in the layout a bf16 tile would have (int4:
// with each 8-dim unit in the expansion's own order, which Q and the output
// store follow).  The MMAs then run on f16 operands (Q, K, P, V all f16).
// The K producer also passes each page's K and V scales through a four-slot
// ring; the softmax folds the K scale into the scores and the V scale into
// the probabilities, relative to the largest V scale of the tile's sequence
// seen so far (vref), so O accumulates in units of vref and is rescaled when
// vref grows.
//
// Tensor memory (32-bit columns): S0 [0,128), S1 [128,256), O [256,384)
// in fp32; Q [384,448) as bf16 pairs.  P_j (bf16 pairs) is written over the
// S columns it came from: each softmax warp's quarter of S_j holds its
// quarter of P_j in its first 16 columns, so P is double-buffered with S.  Shared memory holds
// only the K and V rings, so the tensor core reads one operand per MMA from
// it.  Every wait is bounded; on a
// timeout the CTA records PA_DEVERR_TIMEOUT, drains its own copies and MMAs,
// frees the tensor memory and ends.
#include "pa_device.cuh"
#include "pa_fp8.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int D = 128;                 // head_dim
constexpr int TN = 128;                // KV tokens per tile
constexpr int TM = 128;                // query rows per CTA
constexpr int HALF = TN * 128;         // one 64-column half of a 128-row tile (bytes)
constexpr int TILEB = 2 * HALF;        // a 128 x 128 bf16 tile (32 KB)
constexpr int KST = 3;                 // K tile stages
constexpr int VST = 3;                 // V tile stages
constexpr int OFF_K = 0;
constexpr int OFF_V = OFF_K + KST * TILEB;
constexpr int SMEM_TILES = OFF_V + VST * TILEB;   // 192 KB
constexpr int SMEM_BYTES = SMEM_TILES + 1024;
constexpr int NSW = 16;                // softmax warps: four per tensor-memory lane quadrant
constexpr int NSOFT = NSW * 32;
constexpr int NCOL = TN / (NSW / 4);   // S / P / O columns one softmax warp handles (32)
constexpr int W_KPROD = 0, W_QK = 1, W_SOFT0 = 2, W_VPROD = W_SOFT0 + NSW, W_PV = W_VPROD + 1;
constexpr int W_KCONV = W_PV + 1, W_VCONV = W_KCONV + 2;   // coded caches: code -> f16 warps
constexpr int NTHREADS = (W_PV + 1) * 32;   // 640
constexpr int NCONV = 64;                   // threads expanding one K (or V) tile
constexpr int SC_SLOTS = 4;                 // scale ring (coded caches), by tile index

// Per cache type: threads per CTA and where a stage holds the raw codes
// before they are expanded in place (one-byte codes: the upper half, which
// row r of the f16 tile's upper half overwrites only after the same thread
// has read raw row r; int4 codes: the last 8 KB, read whole before any write).
template <int KVT>
struct PfCfg {
    static constexpr bool CODED = KVT != KV_BF16;
    static constexpr int NT = CODED ? NTHREADS + 4 * 32 : NTHREADS;
    static constexpr int RAW_OFF = KVT == KV_INT4 ? TILEB - TN * 64 : HALF;
    static constexpr int ROWB = KVT == KV_INT4 ? 64 : 128;   // raw bytes of one token row
};
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t COL_O = 256;
constexpr uint32_t COL_Q = 384;
constexpr float RESCALE_LOG2 = 8.f;    // lazy rescale threshold (a factor of 256)

struct PrefillArgs {
    __nv_bfloat16* out;
    const __nv_bfloat16* q;
    const float* k_scale;    // coded caches: [num_blocks][Hkv]
    const float* v_scale;
    const int32_t* tables;
    const int32_t* lens;
    const int32_t* q_start;
    int Hq, Hkv, G, M, num_blocks, max_q;
    float scale_log2;
};

struct Bars {
    uint64_t kfull[KST], kempty[KST], vfull[VST], vempty[VST];
    uint64_t q_full, s_full[2], p_full[2], o_done[2], drain[2];   // [2]: by tile parity
    uint64_t pair[4];            // the four softmax warps of a lane quadrant
    float red[2][4][128];        // partial row maxima [tile parity][column quarter][row]
    float red_l[4][128];         // partial row sums [column quarter][row]
    uint32_t kbad[KST], vbad[VST];   // pages of the stage whose block id was out of range
    uint64_t kconv[KST], vconv[VST]; // coded caches: the stage's f16 tile is ready
    uint64_t krd, vrd;               // int4: the converter group has read the tile's codes
    uint64_t sc_full[SC_SLOTS], sc_empty[SC_SLOTS];
    float2 sc[SC_SLOTS][TN / 16];    // (K, V) scale of each page of a tile (coded caches)
    uint32_t tmem_base;
    int abort;
};

// ------------------------------------------------------------------ tcgen05
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    // shared-memory matrix descriptor: start >> 4, leading / stride byte
    // offsets >> 4, descriptor version 1, 128-byte swizzle
    return (uint64_t)((saddr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// instruction descriptor of kind::f16: bf16 A and B, fp32 accumulator,
// A K-major, B K-major (b_mn = 0) or MN-major (b_mn = 1), M x N
__host__ __device__ constexpr uint32_t instr_desc(int M, int N, int b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)b_mn << 16) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

// the same for f16 A and B (format code 0 at bits 7 and 10): the coded caches'
// codes expand to f16 exactly, and Q and P are f16 to match
__host__ __device__ constexpr uint32_t instr_desc_f16(int M, int N, int b_mn) {
    return (1u << 4) | ((uint32_t)b_mn << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// D (+)= A B, both operands described by shared-memory matrix descriptors
__device__ __forceinline__ void umma_ss(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

// D (+)= A B with the A operand (M x K, bf16 pairs along the columns) in tensor memory
// and B described by a shared-memory matrix descriptor
__device__ __forceinline__ void umma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

__device__ __forceinline__ void umma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
          "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
          "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st16u(uint32_t taddr, const uint32_t* v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
        "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float* v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]), "f"(v[8]),
        "f"(v[9]), "f"(v[10]), "f"(v[11]), "f"(v[12]), "f"(v[13]), "f"(v[14]), "f"(v[15]), "f"(v[16]),
        "f"(v[17]), "f"(v[18]), "f"(v[19]), "f"(v[20]), "f"(v[21]), "f"(v[22]), "f"(v[23]), "f"(v[24]),
        "f"(v[25]), "f"(v[26]), "f"(v[27]), "f"(v[28]), "f"(v[29]), "f"(v[30]), "f"(v[31])
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 2^x on the special-function unit (flushes subnormal results to zero).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// acc + lo + hi for the two bf16 halves of pk, in fp32: a mixed-precision
// FMA with 1.0 takes each 16-bit half as it is
__device__ __forceinline__ float add_bf16_halves(float acc, uint32_t pk) {
    unsigned short lo, hi;
    asm("mov.b32 {%0, %1}, %2;" : "=h"(lo), "=h"(hi) : "r"(pk));
    const unsigned short one = 0x3F80;   // bf16 1.0
    asm("fma.rn.f32.bf16 %0, %1, %2, %0;" : "+f"(acc) : "h"(lo), "h"(one));
    asm("fma.rn.f32.bf16 %0, %1, %2, %0;" : "+f"(acc) : "h"(hi), "h"(one));
    return acc;
}

// two bf16 values -> the same two values as f16 (round to nearest; exact
// for the f16 normal range)
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t v) {
    return pack_f16x2(__uint_as_float(v << 16), __uint_as_float(v & 0xFFFF0000u));
}

// Sum, in fp32, of a q row's values as the f16 operand holds them (int8 K
// tiles carry 1152 + c: each score then carries 1152 times this sum).
__device__ __forceinline__ float q_row_f16_sum(const __nv_bfloat16* qrow, bool valid) {
    float sum = 0.f;
    if (valid) {
        const uint4* src = reinterpret_cast<const uint4*>(qrow);
#pragma unroll
        for (int u = 0; u < D / 8; ++u) {
            const uint4 v = __ldg(src + u);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint32_t h = bf16x2_to_f16x2(w[k]);
                const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h));
                sum += f.x + f.y;
            }
        }
    }
    return sum;
}

// The offset that int4 K tiles holding 1032 + c (even dims, low nibbles) and
// 1152 + 16c (odd dims, high nibbles, met by q / 16) add to each score of a q
// row: 1032 * (sum of its even-dim f16 q) + 72 * (sum of its odd-dim ones).
__device__ __forceinline__ float q_row_int4_bias(const __nv_bfloat16* qrow, bool valid) {
    float even = 0.f, odd = 0.f;
    if (valid) {
        const uint4* src = reinterpret_cast<const uint4*>(qrow);
#pragma unroll
        for (int u = 0; u < D / 8; ++u) {
            const uint4 v = __ldg(src + u);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint32_t h = bf16x2_to_f16x2(w[k]);
                const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h));
                even += f.x;
                odd += f.y;
            }
        }
    }
    return kS4BiasLo * even + (kS4BiasHi / 16.f) * odd;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}


// Rows [r0, TN) of both 64-column halves of a tile, and every row of the
// pages flagged in `bad`, set to zero (generic stores; one warp).
__device__ __forceinline__ void zero_tile_rows(uint32_t tile, int r0, uint32_t bad, int bs, int lane) {
    for (int row = r0 + (lane >> 3); row < TN; row += 4)
        for (int hh = 0; hh < 2; ++hh) st_shared_v4(tile + hh * HALF + row * 128 + (lane & 7) * 16, 0, 0, 0, 0);
    while (bad) {
        const int pg = __ffs(bad) - 1;
        bad &= bad - 1;
        for (int row = pg * bs + (lane >> 3); row < (pg + 1) * bs; row += 4)
            for (int hh = 0; hh < 2; ++hh)
                st_shared_v4(tile + hh * HALF + row * 128 + (lane & 7) * 16, 0, 0, 0, 0);
    }
}

// int4 caches: the f16 K and V tiles hold each 8-dim unit in the order the
// nibble expansion yields it, dims {0, 4, 1, 5, 2, 6, 3, 7} (four operations
// per eight codes fewer than putting it back).  Q takes the same order, so
// Q.K^T is unchanged; O's columns come out in it, and the output store puts
// them back.  This turns a unit of four f16x2 words in dim order into that
// order.
__device__ __forceinline__ void to_nibble_order(uint32_t& x, uint32_t& y, uint32_t& z, uint32_t& w) {
    uint32_t a, b, c, d;
    asm("prmt.b32 %0, %1, %2, 0x5410;" : "=r"(a) : "r"(x), "r"(z));   // dims 0, 4
    asm("prmt.b32 %0, %1, %2, 0x7632;" : "=r"(b) : "r"(x), "r"(z));   // dims 1, 5
    asm("prmt.b32 %0, %1, %2, 0x5410;" : "=r"(c) : "r"(y), "r"(w));   // dims 2, 6
    asm("prmt.b32 %0, %1, %2, 0x7632;" : "=r"(d) : "r"(y), "r"(w));   // dims 3, 7
    x = a;
    y = b;
    z = c;
    w = d;
}

// Eight O columns of one output unit (o[0..7], int4 caches: in the nibble
// order above) scaled by inv, as bf16 in dim order.
template <int KVT>
__device__ __forceinline__ uint4 out_unit(const float* o, float inv) {
    if constexpr (KVT == KV_INT4)
        return make_uint4(pack_bf16x2(o[0] * inv, o[2] * inv), pack_bf16x2(o[4] * inv, o[6] * inv),
                          pack_bf16x2(o[1] * inv, o[3] * inv), pack_bf16x2(o[5] * inv, o[7] * inv));
    else
        return make_uint4(pack_bf16x2(o[0] * inv, o[1] * inv), pack_bf16x2(o[2] * inv, o[3] * inv),
                          pack_bf16x2(o[4] * inv, o[5] * inv), pack_bf16x2(o[6] * inv, o[7] * inv));
}

// Shared address of the 16-byte f16 unit holding dims 8u .. 8u + 7 of row r
// of a tile (two 64-column halves of 128 rows x 128 bytes, 128-byte swizzle:
// the layout a bf16 tile loaded by TMA has).
__device__ __forceinline__ uint32_t f16_unit(uint32_t tile, int r, int u) {
    return tile + (u >> 3) * HALF + r * 128 + (((u & 7) ^ (r & 7)) << 4);
}

// Expand a stage's raw codes (landed by TMA at PfCfg::RAW_OFF, 128-byte
// swizzled) in place into exact f16 values.  Thread i < NCONV of the
// converter group; int4 codes: `rd` is the group's read barrier (count
// NCONV), in phase `rd_parity` for this tile.  Returns false on an abort.
// BIASED (K tiles of the one-tile kernel): int8 codes expand to 1152 + c
// (the decode kernel's trick, two operations per four codes fewer), int4
// codes to 1032 + c and 1152 + 16c (four fewer per eight codes); every score
// then carries a per-row offset, which the softmax takes off.
template <int KVT, bool BIASED = false>
__device__ __forceinline__ bool expand_tile(uint32_t tile, int i, uint64_t* rd, uint32_t rd_parity,
                                            volatile int* abort) {
    const uint32_t raw = tile + PfCfg<KVT>::RAW_OFF;
    if constexpr (KVT == KV_INT4) {
        // line i holds tokens 2i (bytes 0..63) and 2i + 1 (bytes 64..127);
        // 16-byte chunk c: token 2i + c / 4, dims 32 (c % 4) .. + 31.  Every
        // line is read before any f16 row is written (the f16 rows overlap
        // other threads' lines): the group meets at a bounded barrier wait.
        uint4 ch[8];
#pragma unroll
        for (int c = 0; c < 8; ++c)
            asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(ch[c].x), "=r"(ch[c].y), "=r"(ch[c].z), "=r"(ch[c].w)
                         : "r"(raw + i * 128 + ((c ^ (i & 7)) << 4)));
        mbar_arrive(rd);
        if (!cta_wait(rd, rd_parity, abort)) return false;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const int r = 2 * i + (c >> 2);
            const uint32_t w[4] = {ch[c].x, ch[c].y, ch[c].z, ch[c].w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {   // word k: dims 32 (c % 4) + 8 k .. + 7, in nibble order
                uint32_t o[4];
                if constexpr (BIASED)
                    nib8_to_f16x2_raw(w[k], o);   // 1032 + c, 1152 + 16c: the softmax takes the offset off
                else
                    nib8_to_f16x2(w[k], o);
                st_shared_v4(f16_unit(tile, r, 4 * (c & 3) + k), o[0], o[1], o[2], o[3]);
            }
        }
    } else {
        // rows i and i + 64: each thread reads its raw row whole before it
        // writes the row's f16 units (the upper half's row r lies on raw row r)
#pragma unroll 1
        for (int r = i; r < TN; r += NCONV) {
            uint4 ch[8];
#pragma unroll
            for (int c = 0; c < 8; ++c)
                asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                             : "=r"(ch[c].x), "=r"(ch[c].y), "=r"(ch[c].z), "=r"(ch[c].w)
                             : "r"(raw + r * 128 + ((c ^ (r & 7)) << 4)));
#pragma unroll
            for (int c = 0; c < 8; ++c) {   // chunk c: dims 16 c .. 16 c + 15 -> units 2c, 2c + 1
                uint32_t a0, a1, b0, b1, c0, c1, d0, d1;
                if constexpr (BIASED && KVT == KV_INT8) {
                    s8x4_to_f16x2_biased(ch[c].x, a0, a1);
                    s8x4_to_f16x2_biased(ch[c].y, b0, b1);
                    s8x4_to_f16x2_biased(ch[c].z, c0, c1);
                    s8x4_to_f16x2_biased(ch[c].w, d0, d1);
                } else {
                    code4_to_f16x2<KVT>(ch[c].x, a0, a1);
                    code4_to_f16x2<KVT>(ch[c].y, b0, b1);
                    code4_to_f16x2<KVT>(ch[c].z, c0, c1);
                    code4_to_f16x2<KVT>(ch[c].w, d0, d1);
                }
                st_shared_v4(f16_unit(tile, r, 2 * c), a0, a1, b0, b1);
                st_shared_v4(f16_unit(tile, r, 2 * c + 1), c0, c1, d0, d1);
            }
        }
    }
    fence_proxy_async_smem();   // the f16 tile, written by generic stores, is read by the tensor core
    return true;
}

// Converter group (two warps): for each tile j of the ring, wait for its raw
// codes, expand them, and arrive on conv[stage].  Ends early on an abort.
template <int KVT, int NS, bool BIASED = false>
__device__ __forceinline__ void convert_ring(uint64_t* full, uint64_t* conv, uint64_t* rd, uint32_t ring, int nT,
                                             int i, volatile int* abort) {
    int st = 0, use = 0;
    for (int j = 0; j < nT; ++j) {
        if (!cta_wait(&full[st], use & 1, abort)) return;
        if (!expand_tile<KVT, BIASED>(ring + st * TILEB, i, rd, j & 1, abort)) return;
        mbar_arrive(&conv[st]);
        if (++st == NS) {
            st = 0;
            ++use;
        }
    }
}

// TMA producer of one ring of NS tile stages (one warp).  Tile j (128 tokens)
// goes into stage j % NS.  Lane i < 128/BS handles page i of each tile: it
// reads the page's block id one tile ahead and issues the page's two
// 128-byte-swizzled boxes.  Lane 0 waits for the stage to be free and posts the
// bytes to expect.  Out-of-range ids are skipped and reported in badw[stage]
// (and, when report_bad, in the device error word).  On an abort, lane 0 waits
// for the copies this warp issued.
// Coded caches: the codes of page i land at PfCfg::RAW_OFF + i * BS * ROWB
// (one box per page), and when `sc` is given (the K producer) each page's
// (K, V) scales are published through the scale ring: slot j % SC_SLOTS,
// sc_full arrived once the tile's scales are written, sc_empty arrived by
// every softmax thread once it has read them.
template <int BS, int NS, int KVT>
__device__ __forceinline__ void produce_ring(const CUtensorMap* map, uint64_t* full, uint64_t* empty, uint32_t* badw,
                                             uint32_t ring, const int32_t* table, int nT, int npages, int num_blocks,
                                             int Hkv, int h, bool report_bad, volatile int* abort, int lane,
                                             float2 (*sc)[TN / 16] = nullptr, uint64_t* sc_full = nullptr,
                                             uint64_t* sc_empty = nullptr, const float* k_scale = nullptr,
                                             const float* v_scale = nullptr) {
    constexpr int PPT = TN / BS;
    constexpr bool CODED = PfCfg<KVT>::CODED;
    constexpr uint32_t PAGE_BYTES = CODED ? (uint32_t)BS * PfCfg<KVT>::ROWB : 2u * BS * 128u;
    const bool pl = lane < PPT;   // a page lane
    if (lane == 0) prefetch_tensormap(map);
    int issued[NS];               // last use of each stage that was loaded
#pragma unroll
    for (int i = 0; i < NS; ++i) issued[i] = -1;
    int nxt = (pl && lane < npages) ? table[lane] : -1;
    // scales of the next tile's page, loaded alongside its block id
    auto load_sc = [&](int id) {
        return (id >= 0 && id < num_blocks) ? make_float2(k_scale[(int64_t)id * Hkv + h], v_scale[(int64_t)id * Hkv + h])
                                            : make_float2(0.f, 0.f);
    };
    float2 nsc = make_float2(0.f, 0.f);
    if (sc) nsc = load_sc(nxt);
    int st = 0, use = 0;          // stage of tile j, and how often it was used before
    for (int j = 0; j < nT; ++j) {
        const int p = j * PPT + lane;
        const int id = nxt;
        const float2 psc = nsc;
        if (j + 1 < nT) {
            nxt = (pl && p + PPT < npages) ? table[p + PPT] : -1;
            if (sc) nsc = load_sc(nxt);
        }
        const bool inside = pl && p < npages;
        const bool valid = inside && id >= 0 && id < num_blocks;
        const uint32_t bad = __ballot_sync(0xffffffffu, inside && !valid);
        const int nvalid = __popc(__ballot_sync(0xffffffffu, valid));
        int ok = 1;
        if (sc) {
            // the tile's scales into ring slot j % SC_SLOTS, once its last reader is done
            const int slot = j % SC_SLOTS;
            if (lane == 0 && j >= SC_SLOTS) ok = cta_wait(&sc_empty[slot], ((j / SC_SLOTS) - 1) & 1, abort) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            if (pl) sc[slot][lane] = valid ? psc : make_float2(0.f, 0.f);
            __syncwarp();
            if (lane == 0) mbar_arrive(&sc_full[slot]);
        }
        if (lane == 0) {
            if (bad && report_bad) raise_error(PA_DEVERR_BLOCK_ID);
            ok = cta_wait(&empty[st], (use & 1) ^ 1, abort) ? 1 : 0;
            if (ok) {
                badw[st] = bad;
                mbar_arrive_expect_tx(&full[st], (uint32_t)nvalid * PAGE_BYTES);
            }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        if (valid) {
            if constexpr (CODED) {
                // one box of BS rows (int4: BS / 2 lines of two rows) of the page's codes
                constexpr int LINES = KVT == KV_INT4 ? BS / 2 : BS;
                const uint32_t dst = ring + st * TILEB + PfCfg<KVT>::RAW_OFF + lane * BS * PfCfg<KVT>::ROWB;
                tma_load_2d_at(dst, map, 0, (id * Hkv + h) * LINES, &full[st]);
            } else {
                const uint32_t dst = ring + st * TILEB + lane * BS * 128;
                const int y = (id * Hkv + h) * BS;
                tma_load_2d_at(dst, map, 0, y, &full[st]);
                tma_load_2d_at(dst + HALF, map, 64, y, &full[st]);
            }
        }
        issued[st] = use;
        if (++st == NS) {
            st = 0;
            ++use;
        }
    }
    if (lane == 0 && *abort) {
        for (int i = 0; i < NS; ++i)
            if (issued[i] >= 0) mbar_wait(&full[i], issued[i] & 1);
    }
}

template <int BS, int KVT>
__global__ void __launch_bounds__(PfCfg<KVT>::NT, 1)
    paged_prefill_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                         const PrefillArgs a) {
    constexpr int PPT = TN / BS;  // pages per KV tile
    constexpr bool CODED = PfCfg<KVT>::CODED;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    __shared__ Bars bars;
    const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int b = blockIdx.z, h = blockIdx.y;
    const int qt = gridDim.x - 1 - blockIdx.x;  // later (longer) query tiles first
    const int G = a.G, T = TM / G;

    // ---- this tile's work (uniform over the CTA)
    const int qs0 = a.q_start[b];
    const int C = a.q_start[b + 1] - qs0;
    const int L = a.lens[b];
    if (C < 0 || C > L || L > a.M * BS || C > a.max_q) {
        if (tid == 0 && h == 0 && qt == 0) raise_error(PA_DEVERR_SEQ_LEN);
        return;
    }
    const int t0 = qt * T;
    if (t0 >= C) return;
    const int tv = min(T, C - t0);              // valid query tokens in the tile
    const int nkv = L - C + t0 + tv;            // KV positions needed: 0 .. nkv-1
    const int nT = (nkv + TN - 1) / TN;
    const int npages = (nkv + BS - 1) / BS;
    const int32_t* table = a.tables + (int64_t)b * a.M;
    volatile int* abort = &bars.abort;

    if (tid == 0) {
        for (int i = 0; i < KST; ++i) {
            mbar_init(&bars.kfull[i], 1);
            mbar_init(&bars.kempty[i], 1);
        }
        for (int i = 0; i < VST; ++i) {
            mbar_init(&bars.vfull[i], 1);
            mbar_init(&bars.vempty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars.s_full[i], 1);
            mbar_init(&bars.o_done[i], 1);
            mbar_init(&bars.p_full[i], NSOFT);
        }
        for (int i = 0; i < 4; ++i) mbar_init(&bars.pair[i], NSW / 4 * 32);
        mbar_init(&bars.q_full, NSOFT);
        mbar_init(&bars.drain[0], 1);
        mbar_init(&bars.drain[1], 1);
        for (int i = 0; i < KST; ++i) mbar_init(&bars.kconv[i], NCONV);
        for (int i = 0; i < VST; ++i) mbar_init(&bars.vconv[i], NCONV);
        mbar_init(&bars.krd, NCONV);
        mbar_init(&bars.vrd, NCONV);
        for (int i = 0; i < SC_SLOTS; ++i) {
            mbar_init(&bars.sc_full[i], 1);
            mbar_init(&bars.sc_empty[i], NSOFT);
        }
        bars.abort = 0;
        fence_mbar_init();
    }
    if (warp == W_QK) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&bars.tmem_base)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars.tmem_base;

    if (warp == W_KPROD || warp == W_VPROD) {
        // ------------------------------------------------------------ producers
        const bool is_k = warp == W_KPROD;
        if (is_k) {
            if constexpr (CODED)
                produce_ring<BS, KST, KVT>(&tm_k, bars.kfull, bars.kempty, bars.kbad, sbase + OFF_K, table, nT, npages,
                                           a.num_blocks, a.Hkv, h, true, abort, lane, bars.sc, bars.sc_full,
                                           bars.sc_empty, a.k_scale, a.v_scale);
            else
                produce_ring<BS, KST, KVT>(&tm_k, bars.kfull, bars.kempty, bars.kbad, sbase + OFF_K, table, nT, npages,
                                           a.num_blocks, a.Hkv, h, true, abort, lane);
        } else {
            produce_ring<BS, VST, KVT>(&tm_v, bars.vfull, bars.vempty, bars.vbad, sbase + OFF_V, table, nT, npages,
                                       a.num_blocks, a.Hkv, h, false, abort, lane);
        }
    } else if (CODED && warp >= W_KCONV) {
        // ------------------------------------------------------------ code -> f16 expansion
        const bool is_k = warp < W_VCONV;
        const int i = tid - (is_k ? W_KCONV : W_VCONV) * 32;
        if (is_k)
            convert_ring<KVT, KST, KVT == KV_INT8 || KVT == KV_INT4>(bars.kfull, bars.kconv, &bars.krd, sbase + OFF_K,
                                                                     nT, i, abort);
        else
            convert_ring<KVT, VST>(bars.vfull, bars.vconv, &bars.vrd, sbase + OFF_V, nT, i, abort);
    } else if (warp == W_QK) {
        // ------------------------------------------------------------ S = Q K^T issuer
        constexpr uint32_t ID_S = CODED ? instr_desc_f16(TM, TN, 0) : instr_desc(TM, TN, 0);
        uint64_t* kready = CODED ? bars.kconv : bars.kfull;
        const uint64_t kd0 = smem_desc(sbase + OFF_K, 16, 1024);   // + (byte offset >> 4) per MMA
        bool ok = cta_wait(&bars.q_full, 0, abort);
        tc_fence_after();
        int ks = 0, kuse = 0;   // K stage of tile j and its use count
        for (int j = 0; ok && j < nT; ++j) {
            const int sb = j & 1;
            if (!(ok = cta_wait(&kready[ks], kuse & 1, abort))) break;
            const uint32_t kbad = bars.kbad[ks];
            if (kbad) {
                zero_tile_rows(sbase + OFF_K + ks * TILEB, TN, kbad, BS, lane);
                fence_proxy_async_smem();
            }
            __syncwarp();
            // S buffer j%2 holds P_{j-2} until P_{j-2} V_{j-2} has finished
            if (j >= 2 && !(ok = cta_wait(&bars.o_done[sb], ((j >> 1) & 1) ^ 1, abort))) break;
            tc_fence_after();
            if (lane == 0) {
                const uint32_t d_tmem = tmem + (uint32_t)sb * TN;
                const uint64_t kd = kd0 + (uint64_t)((ks * TILEB) >> 4);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    umma_ts(d_tmem, tmem + COL_Q + kk * 8, kd + (uint64_t)((((kk >> 2) * HALF) + (kk & 3) * 32) >> 4),
                            ID_S, kk > 0);
                umma_commit(&bars.s_full[sb]);
                umma_commit(&bars.kempty[ks]);
            }
            __syncwarp();
            if (++ks == KST) {
                ks = 0;
                ++kuse;
            }
        }
        // every MMA this thread issued has completed before the CTA frees the tensor memory
        if (lane == 0) {
            umma_commit(&bars.drain[0]);
            mbar_wait(&bars.drain[0], 0);
        }
        __syncwarp();
    } else if (warp == W_PV) {
        // ------------------------------------------------------------ O += P V issuer
        // (a second issuing thread: one thread alone cannot issue MMAs of this
        // size as fast as the tensor core retires them)
        constexpr uint32_t ID_O = CODED ? instr_desc_f16(TM, D, 1) : instr_desc(TM, D, 1);
        uint64_t* vready = CODED ? bars.vconv : bars.vfull;
        const uint64_t vd0 = smem_desc(sbase + OFF_V, HALF, 1024);
        bool ok = true;
        int vs = 0, vuse = 0;   // V stage of tile j and its use count
        for (int j = 0; ok && j < nT; ++j) {
            if (!(ok = cta_wait(&vready[vs], vuse & 1, abort))) break;
            const int rz = (j == nT - 1) ? nkv - j * TN : TN;   // rows past the last needed position
            const uint32_t vbad = bars.vbad[vs];
            if (rz < TN || vbad) {
                zero_tile_rows(sbase + OFF_V + vs * TILEB, rz, vbad, BS, lane);
                fence_proxy_async_smem();
            }
            __syncwarp();
            if (!(ok = cta_wait(&bars.p_full[j & 1], (j >> 1) & 1, abort))) break;
            tc_fence_after();
            if (lane == 0) {
                const uint64_t vd = vd0 + (uint64_t)((vs * TILEB) >> 4);
#pragma unroll
                for (int kk = 0; kk < TN / 16; ++kk)   // P_j: quarter kk/2 of S buffer j%2, 16 packed columns each
                    umma_ts(tmem + COL_O, tmem + (uint32_t)(j & 1) * TN + (kk >> 1) * NCOL + (kk & 1) * 8,
                            vd + (uint64_t)((kk * 2048) >> 4), ID_O, (j > 0 || kk > 0) ? 1u : 0u);
                umma_commit(&bars.o_done[j & 1]);
                umma_commit(&bars.vempty[vs]);
            }
            __syncwarp();
            if (++vs == VST) {
                vs = 0;
                ++vuse;
            }
        }
        if (lane == 0) {
            umma_commit(&bars.drain[1]);
            mbar_wait(&bars.drain[1], 0);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax
        // warps W_SOFT0 .. W_SOFT0+15: quad = warp % 4 selects the tensor-
        // memory lanes (query rows) the warp may access; qc the quarter of the
        // 128 columns of S, P and O it handles.  The four warps of a quad
        // exchange their partial row maxima (and, at the end, row sums)
        // through shared memory.
        const int quad = warp & 3, qc = (warp - W_SOFT0) >> 2;
        const int r = quad * 32 + lane;
        const int tok = t0 + r / G, g = r % G;
        const bool valid_row = tok < C;
        const int qpos = valid_row ? L - C + tok : -1;
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        // a lane quadrant whose 32 rows all lie past the chunk's last query
        // (short chunks: verify passes) computes nothing: its Q rows are zero,
        // so its S and P rows are zero and P V leaves its O rows at zero; it
        // only keeps pace with the barriers the other roles count it in
        const bool live = t0 + (quad * 32) / G < C;
        {
            // this quarter of the Q row -> tensor memory (bf16 pairs, element
            // 2i in the low half of column i)
            const uint4* src =
                reinterpret_cast<const uint4*>(a.q + ((int64_t)(qs0 + tok) * a.Hq + h * G + g) * D) + qc * 4;
            uint32_t qv[16];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                uint4 v = make_uint4(0, 0, 0, 0);
                if (valid_row) v = __ldg(src + u);
                qv[4 * u] = v.x;
                qv[4 * u + 1] = v.y;
                qv[4 * u + 2] = v.z;
                qv[4 * u + 3] = v.w;
            }
            if constexpr (CODED) {   // f16 operands throughout
#pragma unroll
                for (int i = 0; i < 16; ++i) qv[i] = bf16x2_to_f16x2(qv[i]);
            }
            if constexpr (KVT == KV_INT4) {
                // the K tiles' odd dims hold 1152 + 16c: their q enters as q / 16
                const __half2 s16 = __halves2half2(__ushort_as_half(0x2C00), __ushort_as_half(0x2C00));
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    to_nibble_order(qv[4 * u], qv[4 * u + 1], qv[4 * u + 2], qv[4 * u + 3]);
#pragma unroll
                    for (int o = 1; o < 4; o += 2) {
                        __half2 hq = __hmul2(*reinterpret_cast<const __half2*>(&qv[4 * u + o]), s16);
                        qv[4 * u + o] = *reinterpret_cast<uint32_t*>(&hq);
                    }
                }
            }
            tmem_st16u(tmem + lane_off + COL_Q + qc * 16, qv);
            tc_fence_before();
            mbar_arrive(&bars.q_full);
        }
        const float sl2 = a.scale_log2;
        float m = -INFINITY, l = 0.f;   // running max (scaled, log2 units) and this quarter's sum
        // coded caches: O is kept in units of vref, the largest V scale seen
        float vref = 0.f, inv_vref = 0.f;
        // int8 / int4: the offset the K tiles' offset codes add to this row's scores
        const __nv_bfloat16* qrow = a.q + ((int64_t)(qs0 + tok) * a.Hq + h * G + g) * D;
        const float kbias = !live               ? 0.f
                            : KVT == KV_INT8 ? kS8Bias * q_row_f16_sum(qrow, valid_row)
                            : KVT == KV_INT4 ? q_row_int4_bias(qrow, valid_row)
                                             : 0.f;
        bool ok = true;
        for (int j = 0; j < nT; ++j) {
            const int s = j & 1;
            // coded caches: this tile's page scales (K on the scores, V on the probabilities)
            constexpr int PQ = CODED ? (NCOL + BS - 1) / BS : 1;   // pages under this thread's columns
            float sl2k[PQ], vr[PQ];
            float vmax = 0.f;
            if constexpr (CODED) {
                const int slot = j % SC_SLOTS;
                if (!(ok = cta_wait(&bars.sc_full[slot], (j / SC_SLOTS) & 1, abort))) break;
#pragma unroll
                for (int i = 0; i < PPT; ++i) vmax = fmaxf(vmax, bars.sc[slot][i].y);
#pragma unroll
                for (int i = 0; i < PQ; ++i) {
                    const float2 sv = bars.sc[slot][(qc * NCOL) / BS + i];
                    sl2k[i] = sl2 * sv.x;
                    vr[i] = sv.y;
                }
                mbar_arrive(&bars.sc_empty[slot]);
            }
            if (!(ok = cta_wait(&bars.s_full[s], (j >> 1) & 1, abort))) break;
            if (!live) {
                mbar_arrive(&bars.p_full[s]);
                continue;
            }
            tc_fence_after();
            float x[NCOL];
            tmem_ld32(tmem + lane_off + s * TN + qc * NCOL, x);
            const int lim = qpos - j * TN - qc * NCOL;   // columns c <= lim are visible to this row
            if constexpr (CODED) {
                // scores in log2 units (K scale of the column's page; int8: the
                // biased codes' offset off), masked after scaling
#pragma unroll
                for (int c = 0; c < NCOL; ++c)
                    x[c] = (c <= lim) ? fmaf(x[c], sl2k[c / BS], -kbias * sl2k[c / BS]) : -INFINITY;
            } else if (lim < NCOL - 1) {
#pragma unroll
                for (int c = 0; c < NCOL; ++c) x[c] = (c <= lim) ? x[c] : -INFINITY;
            }
            float mx8[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) mx8[i] = x[i];
#pragma unroll
            for (int c = 8; c < NCOL; ++c) mx8[c & 7] = fmaxf(mx8[c & 7], x[c]);
            const float mxs = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                                    fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]))) * (CODED ? 1.f : sl2);
            bars.red[j & 1][qc][r] = mxs;
            mbar_arrive(&bars.pair[quad]);
            if (!(ok = cta_wait(&bars.pair[quad], j & 1, abort))) break;
            const float mt = fmaxf(fmaxf(bars.red[j & 1][0][r], bars.red[j & 1][1][r]),
                                   fmaxf(bars.red[j & 1][2][r], bars.red[j & 1][3][r]));
            const float m_new = fmaxf(m, mt);
            const bool rescale = m_new > m + RESCALE_LOG2;
            const float m_next = rescale ? m_new : m;
            const float mb = (m_next == -INFINITY) ? 0.f : m_next;
            uint32_t w[NCOL / 2];
            float ls[4] = {0.f, 0.f, 0.f, 0.f};
            // coded caches: a larger V scale than any before moves vref (O rescales below)
            const float vref_old = vref;
            if (CODED && vmax > vref) {
                vref = vmax;
                inv_vref = 1.f / vmax;
            }
            if constexpr (CODED) {
                // P' = P * vsc / vref as f16 (exact codes times these probabilities
                // accumulate O in units of vref); l sums P itself
#pragma unroll
                for (int c = 0; c < NCOL; c += 2) {
                    const float p0 = ex2(x[c] - mb), p1 = ex2(x[c + 1] - mb);
                    const float ratio = vr[c / BS] * inv_vref;   // 0 while every V scale seen is 0
                    ls[(c >> 1) & 3] += p0 + p1;
                    w[c >> 1] = pack_f16x2(p0 * ratio, p1 * ratio);
                }
            } else {
#pragma unroll
                for (int c = 0; c < NCOL; c += 2) {
                    // l sums the probabilities as the P V product sees them (bf16):
                    // the output is then a convex combination of V rows whose weights
                    // carry the rounding, so its error scales with the spread of V
                    // rather than with |V|
                    const uint32_t pk = pack_bf16x2(ex2(fmaf(x[c], sl2, -mb)), ex2(fmaf(x[c + 1], sl2, -mb)));
                    ls[(c >> 1) & 3] = add_bf16_halves(ls[(c >> 1) & 3], pk);
                    w[c >> 1] = pk;
                }
            }
            const bool mrescale = rescale && m != -INFINITY;
            const bool vrescale = CODED && vref > vref_old && vref_old > 0.f;
            if (mrescale || vrescale) {
                // O must be stable: P_{j-1} V_{j-1} has finished
                if (!(ok = cta_wait(&bars.o_done[(j - 1) & 1], ((j - 1) >> 1) & 1, abort))) break;
                tc_fence_after();
                const float alpha = mrescale ? ex2(m - m_new) : 1.f;
                if (mrescale) l *= alpha;
                const float f = vrescale ? alpha * (vref_old * inv_vref) : alpha;
                float o[NCOL];
                tmem_ld32(tmem + lane_off + COL_O + qc * NCOL, o);
#pragma unroll
                for (int i = 0; i < NCOL; ++i) o[i] *= f;
                tmem_st32(tmem + lane_off + COL_O + qc * NCOL, o);
            }
            m = m_next;
            l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
            // P_j over the S columns this warp has just read (its own quarter)
            tmem_st16u(tmem + lane_off + s * TN + qc * NCOL, w);
            tc_fence_before();
            mbar_arrive(&bars.p_full[s]);
        }
        if (ok && live && cta_wait(&bars.o_done[(nT - 1) & 1], ((nT - 1) >> 1) & 1, abort)) {
            tc_fence_after();
            bars.red_l[qc][r] = l;
            mbar_arrive(&bars.pair[quad]);
            if (cta_wait(&bars.pair[quad], nT & 1, abort)) {
                const float lt = (bars.red_l[0][r] + bars.red_l[1][r]) + (bars.red_l[2][r] + bars.red_l[3][r]);
                // coded caches: O is in units of vref
                const float inv = lt > 0.f ? (CODED ? vref : 1.f) / lt : 0.f;
                uint4* dst =
                    reinterpret_cast<uint4*>(a.out + ((int64_t)(qs0 + tok) * a.Hq + h * G + g) * D) + qc * (NCOL / 8);
                float o[NCOL];
                tmem_ld32(tmem + lane_off + COL_O + qc * NCOL, o);
                if (valid_row) {
#pragma unroll
                    for (int v = 0; v < NCOL / 8; ++v) dst[v] = out_unit<KVT>(o + 8 * v, inv);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == W_QK) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS)
                     : "memory");
    }
}

// ------------------------------------------------------------------ two query tiles per CTA
// For chunks longer than one tile: the CTA owns 256 query rows (tiles A and
// B, consecutive tokens) of one (sequence, kv head), so every K/V tile feeds
// twice the MMA work.  Same warp roles as above; the softmax warps alternate
// between the tiles, so the tensor core works on one tile while the softmax
// works on the other.  Q_A / Q_B are in shared memory (A operand of Q K^T by
// descriptor), the K and V rings have two stages each, and tensor memory holds
// S_A [0,128), S_B [128,256), O_A [256,384), O_B [384,512); P_t is written
// over the S_t quarter its warp has just read, so Q K_{j+1}^T of tile t waits
// for P_t(j) V_j.
constexpr int P2_OFF_Q = 0;
constexpr int P2_OFF_K = 2 * TILEB;
constexpr int P2_OFF_V = P2_OFF_K + 2 * TILEB;
constexpr int P2_SMEM_BYTES = P2_OFF_V + 2 * TILEB + 1024;   // 192 KB + alignment

struct Bars2 {
    uint64_t kfull[2], kempty[2], vfull[2], vempty[2];
    uint64_t q_full, s_full[2], p_full[2], o_done[2], drain[2];   // [2]: query tile
    uint64_t pair[2][4];                                          // [tile][lane quadrant]
    float red[2][2][4][128];     // partial row maxima [tile][tile parity j][column quarter][row]
    float red_l[2][4][128];      // partial row sums [tile][column quarter][row]
    uint32_t kbad[2], vbad[2];
    uint64_t kconv[2], vconv[2];     // coded caches: the stage's f16 tile is ready
    uint64_t krd, vrd;               // int4: the converter group has read the tile's codes
    uint64_t sc_full[SC_SLOTS], sc_empty[SC_SLOTS];
    float2 sc[SC_SLOTS][TN / 16];    // (K, V) scale of each page of a tile (coded caches)
    uint32_t tmem_base;
    int abort;
};

template <int BS, int KVT>
__global__ void __launch_bounds__(PfCfg<KVT>::NT, 1)
    paged_prefill2_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                          const PrefillArgs a) {
    constexpr int PPT = TN / BS;  // pages per KV tile
    constexpr bool CODED = PfCfg<KVT>::CODED;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    __shared__ Bars2 bars;
    const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int b = blockIdx.z, h = blockIdx.y;
    const int qt = gridDim.x - 1 - blockIdx.x;  // later (longer) query tiles first
    const int G = a.G, T = TM / G;

    const int qs0 = a.q_start[b];
    const int C = a.q_start[b + 1] - qs0;
    const int L = a.lens[b];
    if (C < 0 || C > L || L > a.M * BS || C > a.max_q) {
        if (tid == 0 && h == 0 && qt == 0) raise_error(PA_DEVERR_SEQ_LEN);
        return;
    }
    const int t0 = qt * 2 * T;                  // first token of tile A
    if (t0 >= C) return;
    const int tv = min(2 * T, C - t0);          // valid query tokens in the two tiles
    const int nkv = L - C + t0 + tv;            // KV positions needed: 0 .. nkv-1
    const int nT = (nkv + TN - 1) / TN;
    const int npages = (nkv + BS - 1) / BS;
    const int32_t* table = a.tables + (int64_t)b * a.M;
    volatile int* abort = &bars.abort;

    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars.kfull[i], 1);
            mbar_init(&bars.kempty[i], 1);
            mbar_init(&bars.vfull[i], 1);
            mbar_init(&bars.vempty[i], 1);
            mbar_init(&bars.s_full[i], 1);
            mbar_init(&bars.o_done[i], 1);
            mbar_init(&bars.p_full[i], NSOFT);
            mbar_init(&bars.drain[i], 1);
            for (int q = 0; q < 4; ++q) mbar_init(&bars.pair[i][q], NSW / 4 * 32);
            mbar_init(&bars.kconv[i], NCONV);
            mbar_init(&bars.vconv[i], NCONV);
        }
        mbar_init(&bars.krd, NCONV);
        mbar_init(&bars.vrd, NCONV);
        for (int i = 0; i < SC_SLOTS; ++i) {
            mbar_init(&bars.sc_full[i], 1);
            mbar_init(&bars.sc_empty[i], NSOFT);
        }
        mbar_init(&bars.q_full, NSOFT);
        bars.abort = 0;
        fence_mbar_init();
    }
    if (warp == W_QK) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&bars.tmem_base)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars.tmem_base;

    if (warp == W_KPROD || warp == W_VPROD) {
        if (warp == W_KPROD) {
            if constexpr (CODED)
                produce_ring<BS, 2, KVT>(&tm_k, bars.kfull, bars.kempty, bars.kbad, sbase + P2_OFF_K, table, nT,
                                         npages, a.num_blocks, a.Hkv, h, true, abort, lane, bars.sc, bars.sc_full,
                                         bars.sc_empty, a.k_scale, a.v_scale);
            else
                produce_ring<BS, 2, KVT>(&tm_k, bars.kfull, bars.kempty, bars.kbad, sbase + P2_OFF_K, table, nT,
                                         npages, a.num_blocks, a.Hkv, h, true, abort, lane);
        } else {
            produce_ring<BS, 2, KVT>(&tm_v, bars.vfull, bars.vempty, bars.vbad, sbase + P2_OFF_V, table, nT, npages,
                                     a.num_blocks, a.Hkv, h, false, abort, lane);
        }
    } else if (CODED && warp >= W_KCONV) {
        // ------------------------------------------------------------ code -> f16 expansion
        const bool is_k = warp < W_VCONV;
        const int i = tid - (is_k ? W_KCONV : W_VCONV) * 32;
        if (is_k)
            convert_ring<KVT, 2>(bars.kfull, bars.kconv, &bars.krd, sbase + P2_OFF_K, nT, i, abort);
        else
            convert_ring<KVT, 2>(bars.vfull, bars.vconv, &bars.vrd, sbase + P2_OFF_V, nT, i, abort);
    } else if (warp == W_QK) {
        // ------------------------------------------------------------ S_t = Q_t K_j^T issuer
        constexpr uint32_t ID_S = CODED ? instr_desc_f16(TM, TN, 0) : instr_desc(TM, TN, 0);
        uint64_t* kready = CODED ? bars.kconv : bars.kfull;
        const uint64_t qd0 = smem_desc(sbase + P2_OFF_Q, 16, 1024);
        const uint64_t kd0 = smem_desc(sbase + P2_OFF_K, 16, 1024);
        bool ok = cta_wait(&bars.q_full, 0, abort);
        tc_fence_after();
        for (int j = 0; ok && j < nT; ++j) {
            const int ks = j & 1;
            if (!(ok = cta_wait(&kready[ks], (j >> 1) & 1, abort))) break;
            const uint32_t kbad = bars.kbad[ks];
            if (kbad) {
                zero_tile_rows(sbase + P2_OFF_K + ks * TILEB, TN, kbad, BS, lane);
                fence_proxy_async_smem();
            }
            __syncwarp();
            for (int t = 0; ok && t < 2; ++t) {
                // S_t holds P_t(j-1) until P_t(j-1) V_{j-1} has finished
                if (j > 0 && !(ok = cta_wait(&bars.o_done[t], (j - 1) & 1, abort))) break;
                tc_fence_after();
                if (lane == 0) {
                    const uint64_t qd = qd0 + (uint64_t)((t * TILEB) >> 4);
                    const uint64_t kd = kd0 + (uint64_t)((ks * TILEB) >> 4);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint64_t off = (uint64_t)(((kk >> 2) * HALF + (kk & 3) * 32) >> 4);
                        umma_ss(tmem + (uint32_t)t * TN, qd + off, kd + off, ID_S, kk > 0);
                    }
                    umma_commit(&bars.s_full[t]);
                }
                __syncwarp();
            }
            if (!ok) break;
            if (lane == 0) umma_commit(&bars.kempty[ks]);
            __syncwarp();
        }
        if (lane == 0) {
            umma_commit(&bars.drain[0]);
            mbar_wait(&bars.drain[0], 0);
        }
        __syncwarp();
    } else if (warp == W_PV) {
        // ------------------------------------------------------------ O_t += P_t V_j issuer
        constexpr uint32_t ID_O = CODED ? instr_desc_f16(TM, D, 1) : instr_desc(TM, D, 1);
        uint64_t* vready = CODED ? bars.vconv : bars.vfull;
        const uint64_t vd0 = smem_desc(sbase + P2_OFF_V, HALF, 1024);
        bool ok = true;
        for (int j = 0; ok && j < nT; ++j) {
            const int vs = j & 1;
            if (!(ok = cta_wait(&vready[vs], (j >> 1) & 1, abort))) break;
            const int rz = (j == nT - 1) ? nkv - j * TN : TN;   // rows past the last needed position
            const uint32_t vbad = bars.vbad[vs];
            if (rz < TN || vbad) {
                zero_tile_rows(sbase + P2_OFF_V + vs * TILEB, rz, vbad, BS, lane);
                fence_proxy_async_smem();
            }
            __syncwarp();
            for (int t = 0; ok && t < 2; ++t) {
                if (!(ok = cta_wait(&bars.p_full[t], j & 1, abort))) break;
                tc_fence_after();
                if (lane == 0) {
                    const uint64_t vd = vd0 + (uint64_t)((vs * TILEB) >> 4);
#pragma unroll
                    for (int kk = 0; kk < TN / 16; ++kk)   // P_t: quarter kk/2 of S_t, 16 packed columns each
                        umma_ts(tmem + COL_O + (uint32_t)t * TN, tmem + (uint32_t)t * TN + (kk >> 1) * NCOL + (kk & 1) * 8,
                                vd + (uint64_t)((kk * 2048) >> 4), ID_O, (j > 0 || kk > 0) ? 1u : 0u);
                    umma_commit(&bars.o_done[t]);
                }
                __syncwarp();
            }
            if (!ok) break;
            if (lane == 0) umma_commit(&bars.vempty[vs]);
            __syncwarp();
        }
        if (lane == 0) {
            umma_commit(&bars.drain[1]);
            mbar_wait(&bars.drain[1], 0);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax (both tiles)
        const int quad = warp & 3, qc = (warp - W_SOFT0) >> 2;
        const int r = quad * 32 + lane;
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        int tok[2], qpos[2];
        bool valid_row[2];
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            tok[t] = t0 + t * T + r / G;
            valid_row[t] = tok[t] < C;
            qpos[t] = valid_row[t] ? L - C + tok[t] : -1;
        }
        const int g = r % G;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            // this quarter of the Q row of tile t -> shared memory, 128-byte swizzled
            const uint4* src =
                reinterpret_cast<const uint4*>(a.q + ((int64_t)(qs0 + tok[t]) * a.Hq + h * G + g) * D) + qc * 4;
            const uint32_t row = sbase + P2_OFF_Q + t * TILEB + (qc >> 1) * HALF + r * 128;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                uint4 v = make_uint4(0, 0, 0, 0);
                if (valid_row[t]) v = __ldg(src + i);
                if constexpr (CODED) {   // f16 operands throughout
                    v.x = bf16x2_to_f16x2(v.x);
                    v.y = bf16x2_to_f16x2(v.y);
                    v.z = bf16x2_to_f16x2(v.z);
                    v.w = bf16x2_to_f16x2(v.w);
                }
                if constexpr (KVT == KV_INT4) to_nibble_order(v.x, v.y, v.z, v.w);
                const int u = (qc & 1) * 4 + i;
                st_shared_v4(row + ((u ^ (r & 7)) << 4), v.x, v.y, v.z, v.w);
            }
        }
        fence_proxy_async_smem();
        mbar_arrive(&bars.q_full);
        const float sl2 = a.scale_log2;
        float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
        // coded caches: O_t is kept in units of vref[t], the largest V scale seen
        float vref[2] = {0.f, 0.f}, inv_vref[2] = {0.f, 0.f};
        bool ok = true;
        for (int j = 0; ok && j < nT; ++j) {
            // coded caches: this K/V tile's page scales, shared by both query tiles
            constexpr int PQ = CODED ? (NCOL + BS - 1) / BS : 1;   // pages under this thread's columns
            float sl2k[PQ], vr[PQ];
            float vmax = 0.f;
            if constexpr (CODED) {
                const int slot = j % SC_SLOTS;
                if (!(ok = cta_wait(&bars.sc_full[slot], (j / SC_SLOTS) & 1, abort))) break;
#pragma unroll
                for (int i = 0; i < PPT; ++i) vmax = fmaxf(vmax, bars.sc[slot][i].y);
#pragma unroll
                for (int i = 0; i < PQ; ++i) {
                    const float2 sv = bars.sc[slot][(qc * NCOL) / BS + i];
                    sl2k[i] = sl2 * sv.x;
                    vr[i] = sv.y;
                }
                mbar_arrive(&bars.sc_empty[slot]);
            }
#pragma unroll 1
            for (int t = 0; t < 2; ++t) {
                if (!(ok = cta_wait(&bars.s_full[t], j & 1, abort))) break;
                tc_fence_after();
                float x[NCOL];
                tmem_ld32(tmem + lane_off + t * TN + qc * NCOL, x);
                const int lim = qpos[t] - j * TN - qc * NCOL;
                if constexpr (CODED) {
                    // scores in log2 units (K scale of the column's page), masked after
                    // scaling; only a tile the causal limit cuts pays for the mask
                    if (lim < NCOL - 1) {
#pragma unroll
                        for (int c = 0; c < NCOL; ++c) x[c] = (c <= lim) ? x[c] * sl2k[c / BS] : -INFINITY;
                    } else {
#pragma unroll
                        for (int c = 0; c < NCOL; ++c) x[c] *= sl2k[c / BS];
                    }
                } else if (lim < NCOL - 1) {
#pragma unroll
                    for (int c = 0; c < NCOL; ++c) x[c] = (c <= lim) ? x[c] : -INFINITY;
                }
                float mx8[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) mx8[i] = x[i];
#pragma unroll
                for (int c = 8; c < NCOL; ++c) mx8[c & 7] = fmaxf(mx8[c & 7], x[c]);
                const float mxs = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                                        fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]))) * (CODED ? 1.f : sl2);
                bars.red[t][j & 1][qc][r] = mxs;
                mbar_arrive(&bars.pair[t][quad]);
                if (!(ok = cta_wait(&bars.pair[t][quad], j & 1, abort))) break;
                const float mt = fmaxf(fmaxf(bars.red[t][j & 1][0][r], bars.red[t][j & 1][1][r]),
                                       fmaxf(bars.red[t][j & 1][2][r], bars.red[t][j & 1][3][r]));
                const float m_new = fmaxf(m[t], mt);
                const bool rescale = m_new > m[t] + RESCALE_LOG2;
                const float m_next = rescale ? m_new : m[t];
                const float mb = (m_next == -INFINITY) ? 0.f : m_next;
                uint32_t w[NCOL / 2];
                float ls[4] = {0.f, 0.f, 0.f, 0.f};
                const float vref_old = vref[t];
                if (CODED && vmax > vref[t]) {
                    vref[t] = vmax;
                    inv_vref[t] = 1.f / vmax;
                }
                if constexpr (CODED) {
                    // P' = P * vsc / vref as f16; l sums P itself
#pragma unroll
                    for (int c = 0; c < NCOL; c += 2) {
                        const float p0 = ex2(x[c] - mb), p1 = ex2(x[c + 1] - mb);
                        const float ratio = vr[c / BS] * inv_vref[t];   // 0 while every V scale seen is 0
                        ls[(c >> 1) & 3] += p0 + p1;
                        w[c >> 1] = pack_f16x2(p0 * ratio, p1 * ratio);
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < NCOL; c += 2) {
                        // l sums the bf16 probabilities the P V product uses
                        const uint32_t pk = pack_bf16x2(ex2(fmaf(x[c], sl2, -mb)), ex2(fmaf(x[c + 1], sl2, -mb)));
                        ls[(c >> 1) & 3] = add_bf16_halves(ls[(c >> 1) & 3], pk);
                        w[c >> 1] = pk;
                    }
                }
                const bool mrescale = rescale && m[t] != -INFINITY;
                const bool vrescale = CODED && vref[t] > vref_old && vref_old > 0.f;
                if (mrescale || vrescale) {
                    // O_t must be stable: P_t(j-1) V_{j-1} has finished (Q K_j^T waited for it)
                    if (!(ok = cta_wait(&bars.o_done[t], (j - 1) & 1, abort))) break;
                    tc_fence_after();
                    const float alpha = mrescale ? ex2(m[t] - m_new) : 1.f;
                    if (mrescale) l[t] *= alpha;
                    const float f = vrescale ? alpha * (vref_old * inv_vref[t]) : alpha;
                    float o[NCOL];
                    tmem_ld32(tmem + lane_off + COL_O + t * TN + qc * NCOL, o);
#pragma unroll
                    for (int i = 0; i < NCOL; ++i) o[i] *= f;
                    tmem_st32(tmem + lane_off + COL_O + t * TN + qc * NCOL, o);
                }
                m[t] = m_next;
                l[t] += (ls[0] + ls[1]) + (ls[2] + ls[3]);
                tmem_st16u(tmem + lane_off + t * TN + qc * NCOL, w);
                tc_fence_before();
                mbar_arrive(&bars.p_full[t]);
            }
        }
#pragma unroll 1
        for (int t = 0; ok && t < 2; ++t) {
            if (!(ok = cta_wait(&bars.o_done[t], (nT - 1) & 1, abort))) break;
            tc_fence_after();
            bars.red_l[t][qc][r] = l[t];
            mbar_arrive(&bars.pair[t][quad]);
            if (!(ok = cta_wait(&bars.pair[t][quad], nT & 1, abort))) break;
            const float lt = (bars.red_l[t][0][r] + bars.red_l[t][1][r]) + (bars.red_l[t][2][r] + bars.red_l[t][3][r]);
            // coded caches: O_t is in units of vref[t]
            const float inv = lt > 0.f ? (CODED ? vref[t] : 1.f) / lt : 0.f;
            float o[NCOL];
            tmem_ld32(tmem + lane_off + COL_O + t * TN + qc * NCOL, o);
            if (valid_row[t]) {
                uint4* dst = reinterpret_cast<uint4*>(a.out + ((int64_t)(qs0 + tok[t]) * a.Hq + h * G + g) * D) +
                             qc * (NCOL / 8);
#pragma unroll
                for (int v = 0; v < NCOL / 8; ++v) dst[v] = out_unit<KVT>(o + 8 * v, inv);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == W_QK) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS)
                     : "memory");
    }
}

template <int BS, int KVT>
cudaError_t launch_typed(const PrefillLaunch& L, cudaStream_t stream) {
    constexpr int NT = PfCfg<KVT>::NT;
    static bool attr_set[64][2] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    PrefillArgs a;
    a.out = static_cast<__nv_bfloat16*>(L.out);
    a.q = static_cast<const __nv_bfloat16*>(L.q);
    a.k_scale = L.k_scale;
    a.v_scale = L.v_scale;
    a.tables = L.tables;
    a.lens = L.lens;
    a.q_start = L.q_start;
    a.Hq = L.Hq;
    a.Hkv = L.Hkv;
    a.G = L.Hq / L.Hkv;
    a.M = L.M;
    a.num_blocks = L.num_blocks;
    a.max_q = L.max_q;
    a.scale_log2 = L.scale * 1.4426950408889634f;
    const int T = TM / a.G;
    // chunks longer than one 128-row tile: two tiles per CTA share each K/V tile
    const bool two = L.max_q > T;
    if (dev >= 0 && dev < 64 && !attr_set[dev][two]) {
        e = two ? cudaFuncSetAttribute(paged_prefill2_kernel<BS, KVT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       P2_SMEM_BYTES)
                : cudaFuncSetAttribute(paged_prefill_kernel<BS, KVT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_set[dev][two] = true;
    }
    if (two) {
        dim3 grid((unsigned)((L.max_q + 2 * T - 1) / (2 * T)), (unsigned)L.Hkv, (unsigned)L.B);
        paged_prefill2_kernel<BS, KVT><<<grid, NT, P2_SMEM_BYTES, stream>>>(*L.tm_k, *L.tm_v, a);
    } else {
        dim3 grid((unsigned)((L.max_q + T - 1) / T), (unsigned)L.Hkv, (unsigned)L.B);
        paged_prefill_kernel<BS, KVT><<<grid, NT, SMEM_BYTES, stream>>>(*L.tm_k, *L.tm_v, a);
    }
    return cudaGetLastError();
}

template <int BS>
cudaError_t launch_kv(const PrefillLaunch& L, cudaStream_t stream) {
    switch (L.kvt) {
        case PA_KV_BF16: return launch_typed<BS, KV_BF16>(L, stream);
        case PA_KV_FP8_E4M3: return launch_typed<BS, KV_FP8>(L, stream);
        case PA_KV_INT8: return launch_typed<BS, KV_INT8>(L, stream);
        case PA_KV_INT4: return launch_typed<BS, KV_INT4>(L, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_prefill(const PrefillLaunch& L, cudaStream_t stream) {
    if (L.bs == 16) return launch_kv<16>(L, stream);
    if (L.bs == 32) return launch_kv<32>(L, stream);
    return cudaErrorInvalidValue;
}

cudaError_t prefill_unit_error(unsigned int* v, bool clear) { return read_unit_error(v, clear); }

}  // namespace pa
