// Paged decode attention for sm_103a, with split-K partitions merged by
// log-sum-exp inside the same launch.
//
// What it computes ("KV cache & continuous batching", sections "The core
// insight" and "2. PagedAttention"; "LLM Serving - KV Cache, Batching,
// Speculative Decoding", section "Hands-on"): for every sequence b and query
// head i, out = softmax(scale * q . K^T) . V over the sequence's cached
// tokens, K/V rows gathered through the block table; query head i reads KV
// head i / G.  Scores, softmax and P.V stay on chip ("LLM Inference
// Optimization", section "FlashAttention") with an fp32 online softmax.
//
// One CTA per (partition of P blocks, pair of kv heads, sequence); one kv
// head per CTA when their count is odd.  The pages of one block for
// consecutive kv heads are adjacent in the cache, so one copy fetches a block
// for both heads.  A CTA has 5 warps:
//   * warp 4, the producer, issues TMA tile loads of each block's K and V rows
//     for the CTA's heads into a ring of shared-memory stages written with the
//     128-byte swizzle; completion is counted in bytes on one mbarrier per
//     stage;
//   * warps 0-3 consume the pages, two warps per kv head taking alternate
//     pages.  Per page a warp forms S^T = Q K^T with m16n8k16 MMAs (the G query
//     heads of the group are the M rows, the page's tokens the N columns,
//     head_dim the K depth; q lives in registers), updates its fp32 online
//     softmax in registers and accumulates O^T += V^T P^T with MMAs whose B
//     operand is the probability tile taken straight from the score registers;
//   * each head's warp states merge in shared memory; a one-partition
//     sequence writes bf16 out, otherwise the partition writes its normalised
//     partials and base-2 log-sum-exps to the workspace and the group's last
//     partition to finish merges them (an atomic counter per group; nothing
//     waits on another CTA).
// Coded caches (e4m3, int8, int4): codes convert exactly to f16 in registers
// (q and the probabilities are f16 there).  The K scale folds into the
// scores; the V scale folds into the probabilities relative to the largest V
// scale seen so far, so P.V accumulates straight into O.  The integer codes
// enter the products with a constant offset that comes off per score (K) or
// once per CTA (V).  An int4 row (64 bytes) is half of a 128-byte line: the
// TMA map views a page as bs / 2 lines of two tokens each.
#include <cuda_fp8.h>
#include <math.h>
#include <stdlib.h>

#include "pa_device.cuh"
#include "pa_fp8.cuh"
#include "pa_internal.h"

namespace pa {

struct DecodeArgs {
    __nv_bfloat16* out;
    const uint16_t* q;
    const float* k_scale;
    const float* v_scale;
    const int32_t* tables;
    const int32_t* lens;
    float* o_part;
    float* lse;
    int* counters;   // [B][Hkv] merge counters
    // fused step (APPEND): new K/V rows written before their page is loaded
    const uint16_t* k_new;
    const uint16_t* v_new;
    uint8_t* k_cache_w;
    uint8_t* v_cache_w;
    float* k_scale_w;
    float* v_scale_w;
    int B, Hq, Hkv, G, M, num_blocks, part_blocks, S;
    int b_early, part_early;   // sequences b < b_early: partitions of part_early blocks
    int scan;                  // 1: the grid lists work items only (see find_later_item)
    float scale_log2;
    int Sw;                    // partial slots per output row in the workspace
    // shared prefixes (SHARED launches): chunk_of[b] = PA_SHARE_MAX_ROWS * c + slot
    // of sequence b in chunk c, -1 for none; chunk c's members and shared blocks
    const int32_t* chunk_of;
    const int32_t* chunk_members;
    const int32_t* chunk_blocks;
    int n_chunks, chunk_parts, max_chunk_blocks;
};

// HPC: kv heads per CTA.  The pages of one block for consecutive kv heads
// are adjacent in the cache, so one copy fetches a block for HPC heads.
template <int D, int BS, int KVT, int HPC = 1>
struct Cfg {
    static constexpr bool FP8 = KVT != KV_BF16;   // coded cache with scales (e4m3, int8 or int4)
    static constexpr bool I4 = KVT == KV_INT4;
    static constexpr int ELT = FP8 ? 1 : 2;
    static constexpr int ROWB = I4 ? D / 2 : D * ELT;   // bytes of one token row of one head
    static constexpr int NCH = I4 ? 1 : ROWB / 128;    // TMA boxes per page (128-byte columns)
    static constexpr int LINES = I4 ? BS / 2 : BS;     // 128-byte lines of a page's box
    static constexpr int PAGEB = BS * ROWB;     // one (block, kv_head) page of K (or V)
    static constexpr int STAGEB = 2 * HPC * PAGEB;   // a block's K pages, then its V pages, for HPC heads
    static constexpr int CHS = HPC * BS * 128;  // stride of the 128-byte column tiles of a stage's K (or V)
    static constexpr int NCW = 4;               // consumer warps
    static constexpr int WPH = NCW / HPC;       // consumer warps per kv head
    static constexpr int NTHREADS = (NCW + 1) * 32;
    static constexpr int KS = D / 16;           // 16-deep steps over head_dim (QK)
    static constexpr int MT = D / 16;           // 16-row tiles of head_dim (PV)
    static constexpr int KT = BS / 16;          // 16-token row tiles (QK) and steps (PV) per page
    static constexpr int COMBINE_FLOATS = NCW * (8 * D + 16);
    static_assert(I4 ? ROWB == 64 : ROWB % 128 == 0, "rows must be whole 128-byte chunks (int4: half of one)");
};

// Shared address of byte `byte` of token row t of a page tile: NCH column
// tiles of BS rows x 128 bytes, CHS bytes apart, or (int4) one tile of BS / 2
// lines holding tokens 2L and 2L + 1 in bytes 0..63 and 64..127 of line L;
// 128-byte swizzle.
template <int BS, int KVT, int CHS>
__device__ __forceinline__ uint32_t tok_addr(uint32_t tile, int t, int byte) {
    if constexpr (KVT == KV_INT4)
        return swz128(tile, t >> 1, ((t & 1) << 6) + byte);
    else
        return swz128(tile + (byte >> 7) * CHS, t, byte & 127);
}


// ------------------------------------------------------------------ per warp
template <int D, int BS, int KVT, int HPC>
struct WarpAcc {
    static constexpr bool FP8 = KVT != KV_BF16;
    static constexpr int CHS = Cfg<D, BS, KVT, HPC>::CHS;
    // Lane (g, c) = (lane / 4, lane % 4) keeps the softmax state of query
    // heads 2c and 2c + 1 (index e), the columns its O fragment holds: m[e] is
    // the same in the 8 lanes of column c, l[e] and psi[e] sum this lane's
    // tokens only (publish() adds the 8 lanes up).
    float m[2], l[2];
    float o[D / 16][4];
    uint32_t qa[D / 16][2];   // q of head g as the Q.K^T B operand
    float qbias[2];   // int8 / int4 caches: the K codes' offset times head 2c + e's q (see load_q)
    // coded caches: O is kept in units of vref (the largest V scale so far) and
    // psi sums the f16 probabilities P' = P * vsc / vref of each head (see the
    // P.V product); publish() turns O back into values
    float vref, inv_vref, psi[2];

    __device__ __forceinline__ void reset() {
        m[0] = m[1] = -INFINITY;
        l[0] = l[1] = 0.f;
        vref = inv_vref = psi[0] = psi[1] = 0.f;
#pragma unroll
        for (int i = 0; i < D / 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    }

    // q of query head h*G + g as the Q.K^T B operand (column g; the k order
    // within a 16-deep step is that of the K operand's codes); columns g >= G
    // stay zero.  `qrow` is a generic pointer (global or shared) to that
    // head's bf16 row.
    __device__ __forceinline__ void load_q(const uint16_t* qrow, bool valid, int c) {
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            if (!valid) {
                qa[ks][0] = qa[ks][1] = 0u;
            } else if (KVT == KV_INT4) {
                // step 2ch + j2 of chunk ch: lane c's elements e_i = 32ch + 8c + i in
                // the order the nibble conversion yields them: {e0,e4},{e1,e5} then
                // {e2,e6},{e3,e7}.  The K operand holds 1032 + c for the even
                // elements (low nibbles) and 1152 + 16c for the odd ones (high
                // nibbles): q of an odd element enters as q / 16
                const int ch = ks >> 1, j2 = ks & 1;
                const uint4 w = *reinterpret_cast<const uint4*>(qrow + ch * 32 + 8 * c);
                const uint32_t u[4] = {w.x, w.y, w.z, w.w};
                auto el = [&](int i) { return __uint_as_float((i & 1) ? (u[i >> 1] & 0xFFFF0000u) : (u[i >> 1] << 16)); };
                qa[ks][0] = pack_f16x2(el(2 * j2), el(2 * j2 + 4));
                qa[ks][1] = pack_f16x2(el(2 * j2 + 1) * 0.0625f, el(2 * j2 + 5) * 0.0625f);
            } else if (FP8) {
                // k order inside a 16-deep step matches the e4m3 byte order 4c .. 4c+3
                const uint2 w = *reinterpret_cast<const uint2*>(qrow + ks * 16 + 4 * c);
                qa[ks][0] = pack_f16x2(__uint_as_float((w.x & 0xFFFF) << 16), __uint_as_float(w.x & 0xFFFF0000u));
                qa[ks][1] = pack_f16x2(__uint_as_float((w.y & 0xFFFF) << 16), __uint_as_float(w.y & 0xFFFF0000u));
            } else {
                qa[ks][0] = *reinterpret_cast<const uint32_t*>(qrow + ks * 16 + 2 * c);
                qa[ks][1] = *reinterpret_cast<const uint32_t*>(qrow + ks * 16 + 2 * c + 8);
            }
        }
        qbias[0] = qbias[1] = 0.f;
        if (KVT == KV_INT8 || KVT == KV_INT4) {
            // the K operand carries an offset per element (int8: 1152 + c;
            // int4: 1032 + c, and 1152 + 16c against q / 16): the scores carry
            // sum_k q_k * offset_k on top, summed here over the same f16 values
            float sum = 0.f, sum_hi = 0.f;
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&qa[ks][j]));
                    if (KVT == KV_INT4 && j == 1)
                        sum_hi += f.x + f.y;
                    else
                        sum += f.x + f.y;
                }
            }
            if (KVT == KV_INT4) sum = kS4BiasLo * sum + kS4BiasHi * sum_hi;
            sum += __shfl_xor_sync(0xffffffffu, sum, 1);
            sum += __shfl_xor_sync(0xffffffffu, sum, 2);
            if (KVT == KV_INT8) sum *= kS8Bias;
            // lanes 8c and 8c + 4 hold heads 2c and 2c + 1
            qbias[0] = __shfl_sync(0xffffffffu, sum, 8 * c);
            qbias[1] = __shfl_sync(0xffffffffu, sum, 8 * c + 4);
        }
    }

    // One page: kt / vt are the shared addresses of its K and V tiles, `valid`
    // the number of its tokens inside the sequence, sl2 = scale * log2(e)
    // (times the K scale for fp8), vsc the V scale (fp8).
    __device__ __forceinline__ void page(uint32_t kt, uint32_t vt, int valid, float sl2, float vsc, int lane) {
        using C = Cfg<D, BS, KVT, HPC>;
        const int g = lane >> 2, c = lane & 3;
        const int mi = lane >> 3, r = lane & 7;

        // ------------------------------------------------ S^T = K Q^T
        // Tokens are the MMA's M (16 per m-tile) and the query heads its N:
        // acc[kk] holds tokens 16kk + g and 16kk + g + 8 (e >> 1) of heads 2c
        // and 2c + 1 (e & 1).  A 16-token page takes D / 16 MMAs.
        float acc[C::KT][4];
#pragma unroll
        for (int kk = 0; kk < C::KT; ++kk) acc[kk][0] = acc[kk][1] = acc[kk][2] = acc[kk][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < C::KS; ++ks) {
            if (KVT == KV_INT4) {
                // one 32-bit word = 8 codes of chunk ks / 2 of a token feeds steps ks and ks + 1
                if (ks & 1) continue;
#pragma unroll
                for (int kk = 0; kk < C::KT; ++kk) {
                    const int t = kk * 16 + g;
                    uint32_t f0[4], f1[4];
                    // offset codes; qbias comes off each score below
                    nib8_to_f16x2_raw(ld_shared_u32(tok_addr<BS, KVT, CHS>(kt, t, (ks >> 1) * 16 + 4 * c)), f0);
                    nib8_to_f16x2_raw(ld_shared_u32(tok_addr<BS, KVT, CHS>(kt, t + 8, (ks >> 1) * 16 + 4 * c)), f1);
                    const uint32_t A0[4] = {f0[0], f1[0], f0[1], f1[1]};
                    const uint32_t A1[4] = {f0[2], f1[2], f0[3], f1[3]};
                    mma_f16(acc[kk], A0, qa[ks][0], qa[ks][1]);
                    mma_f16(acc[kk], A1, qa[ks + 1][0], qa[ks + 1][1]);
                }
            } else if (FP8) {
#pragma unroll
                for (int kk = 0; kk < C::KT; ++kk) {
                    const int t = kk * 16 + g;
                    const uint32_t w0 = ld_shared_u32(swz128(kt, t, ks * 16 + 4 * c));
                    const uint32_t w1 = ld_shared_u32(swz128(kt, t + 8, ks * 16 + 4 * c));
                    uint32_t A[4];
                    if (KVT == KV_INT8) {   // qbias comes off each score below
                        s8x4_to_f16x2_biased(w0, A[0], A[2]);
                        s8x4_to_f16x2_biased(w1, A[1], A[3]);
                    } else {
                        code4_to_f16x2<KVT>(w0, A[0], A[2]);
                        code4_to_f16x2<KVT>(w1, A[1], A[3]);
                    }
                    mma_f16(acc[kk], A, qa[ks][0], qa[ks][1]);
                }
            } else {
                // matrices: tokens 0-7 / 8-15 (mi & 1) x dims 8 (mi >> 1) .. of the step
                const int jg = 2 * ks + (mi >> 1);  // 16-byte unit along the row
                const uint32_t ktile = kt + (jg >> 3) * C::CHS;
#pragma unroll
                for (int kk = 0; kk < C::KT; ++kk) {
                    const int t = kk * 16 + (mi & 1) * 8 + r;
                    uint32_t A[4];
                    ldsm_x4(swz128(ktile, t, (jg & 7) * 16), A[0], A[1], A[2], A[3]);
                    mma_bf16(acc[kk], A, qa[ks][0], qa[ks][1]);
                }
            }
        }

        // ------------------------------------------------ online softmax
        float sc[C::KT][4];
        float mx[2] = {-INFINITY, -INFINITY};
        const float sb[2] = {-qbias[0] * sl2, -qbias[1] * sl2};   // 0 but for the int8 and int4 caches
#pragma unroll
        for (int kk = 0; kk < C::KT; ++kk) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int tok = kk * 16 + g + 8 * (e >> 1);
                const float v = tok < valid ? fmaf(acc[kk][e], sl2, sb[e & 1]) : -INFINITY;
                sc[kk][e] = v;
                mx[e & 1] = fmaxf(mx[e & 1], v);
            }
        }
        // Lazy rescale: m is a reference point, not the running max.  It moves
        // (and O and l are rescaled) only when a score exceeds it by more than
        // 2^8, so that the probabilities 2^(s - m) stay below 256 (exact range
        // for the f16 / bf16 operands) and the O rescale is skipped on almost
        // every page.  The result is the same: O / l with l = sum 2^(s - m).
        // Each lane tests its own scores (m == -inf: any finite one); only on
        // a page where one passes does the warp form the column maxima, which
        // the 8 lanes of a column then share as their new m.
        if (__any_sync(0xffffffffu, mx[0] > m[0] + 8.f || mx[1] > m[1] + 8.f)) {
#pragma unroll
            for (int x = 4; x < 32; x <<= 1) {
                mx[0] = fmaxf(mx[0], __shfl_xor_sync(0xffffffffu, mx[0], x));
                mx[1] = fmaxf(mx[1], __shfl_xor_sync(0xffffffffu, mx[1], x));
            }
            float al[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const float m_new = mx[e] > m[e] + 8.f ? mx[e] : m[e];
                al[e] = m_new == m[e] ? 1.f : exp2f(m[e] - m_new);   // m == -inf: 0
                l[e] *= al[e];
                psi[e] *= al[e];
                m[e] = m_new;
            }
            // accumulator columns are query heads 2c and 2c+1
#pragma unroll
            for (int mt = 0; mt < C::MT; ++mt) {
                o[mt][0] *= al[0];
                o[mt][1] *= al[1];
                o[mt][2] *= al[0];
                o[mt][3] *= al[1];
            }
        }
        const float m_use[2] = {m[0] == -INFINITY ? 0.f : m[0], m[1] == -INFINITY ? 0.f : m[1]};
#pragma unroll
        for (int kk = 0; kk < C::KT; ++kk) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                sc[kk][e] = ex2_approx(sc[kk][e] - m_use[e & 1]);
                // bf16 cache: l sums the probabilities as the P.V product sees
                // them (bf16), so the output is a convex combination of V rows
                // whose weights carry the rounding
                if (!FP8) sc[kk][e] = __bfloat162float(__float2bfloat16_rn(sc[kk][e]));
                l[e & 1] += sc[kk][e];
            }
        }

        // rows past the sequence end hold stale bytes: zero them so that
        // 0-probability x non-finite garbage cannot reach the accumulator
        // (integer codes are always finite)
        constexpr bool ZERO_TAIL = KVT == KV_BF16 || KVT == KV_FP8;
        if (ZERO_TAIL && valid < BS) {
            for (int idx = valid * C::ROWB / 16 + lane; idx < BS * C::ROWB / 16; idx += 32) {
                const int row = idx / (C::ROWB / 16), u = idx % (C::ROWB / 16);
                const uint32_t tile = vt + (u >> 3) * C::CHS;
                asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(swz128(tile, row, (u & 7) * 16)), "r"(0u)
                             : "memory");
            }
            __syncwarp();
        }

        // ------------------------------------------------ O^T += V^T P^T
        // The B operand of k-step kk (tokens 16kk .. 16kk + 15) is P^T: the
        // (token, head) 8x8 blocks of acc[kk] transposed in registers.
        uint32_t pq[C::KT][2];   // coded caches: P' = P * vsc / vref as f16
        if (FP8) {
            // O is kept in units of vref: a page with a larger V scale rescales
            // O (and psi) once; every other page scales its probabilities
            if (vsc > vref) {   // uniform over the warp
                const float rs = vref / vsc;   // 0 on the first page
#pragma unroll
                for (int mt = 0; mt < C::MT; ++mt) o[mt][0] *= rs, o[mt][1] *= rs, o[mt][2] *= rs, o[mt][3] *= rs;
                psi[0] *= rs;
                psi[1] *= rs;
                vref = vsc;
                inv_vref = 1.f / vsc;
            }
            const float ratio = vsc * inv_vref;   // 0 while every V scale seen is 0
#pragma unroll
            for (int kk = 0; kk < C::KT; ++kk) {
                const uint32_t lo = pack_f16x2(sc[kk][0] * ratio, sc[kk][1] * ratio);   // token 16kk + g
                const uint32_t hi = pack_f16x2(sc[kk][2] * ratio, sc[kk][3] * ratio);   // token 16kk + g + 8
                if (KVT == KV_INT8 || KVT == KV_INT4) {   // the integer codes enter P.V with an offset
                    const float2 a0 = __half22float2(*reinterpret_cast<const __half2*>(&lo));
                    const float2 a1 = __half22float2(*reinterpret_cast<const __half2*>(&hi));
                    psi[0] += a0.x + a1.x;
                    psi[1] += a0.y + a1.y;
                }
                pq[kk][0] = movm_t(lo);
                pq[kk][1] = movm_t(hi);
            }
        }
        if (KVT == KV_INT4) {
            // ldmatrix.trans of 16-bit units (4 dims of one token; a unit is 16
            // bytes = 32 dims of a row): lane (g, c) gets tokens 2c, 2c+1 of dims
            // 4g..4g+3 of a unit; the nibble split turns that into one A register
            // per dim.  MMA mt = 2 * unit + jp has rows g -> dim 32 unit + 4g + 2jp
            // (operand 1032 + c) and g + 8 -> that dim + 1 (operand 1152 + 16c).
            // one ldmatrix.x4 covers 32 (token, unit) rows: two units of a
            // 16-token page, or one unit of a 32-token page (matrices 2kk and
            // 2kk + 1 are that unit's tokens 16kk .. 16kk + 15)
            constexpr int UPL = BS == 16 ? 2 : 1;   // units per ldmatrix.x4
#pragma unroll
            for (int u0 = 0; u0 < D / 32; u0 += UPL) {
                const int tok = BS == 16 ? (mi & 1) * 8 + r : mi * 8 + r;
                const int unit = BS == 16 ? u0 + (mi >> 1) : u0;
                uint32_t rr[4];
                ldsm_x4_t(tok_addr<BS, KVT, CHS>(vt, tok, unit * 16), rr[0], rr[1], rr[2], rr[3]);
#pragma unroll
                for (int hm = 0; hm < 2; ++hm) {   // matrix pair (2hm, 2hm+1): tokens 0-7 and 8-15 of a k-step
                    const int kk = BS == 16 ? 0 : hm, ti = BS == 16 ? 2 * hm : 0;
                    uint32_t fa[4], fb[4];
                    nib8_to_f16x2_raw(rr[2 * hm], fa);
                    nib8_to_f16x2_raw(rr[2 * hm + 1], fb);
                    const uint32_t A0[4] = {fa[0], fa[1], fb[0], fb[1]};
                    const uint32_t A1[4] = {fa[2], fa[3], fb[2], fb[3]};
                    mma_f16(o[2 * u0 + ti], A0, pq[kk][0], pq[kk][1]);
                    mma_f16(o[2 * u0 + ti + 1], A1, pq[kk][0], pq[kk][1]);
                }
            }
        } else if (FP8) {
#pragma unroll
            for (int mp = 0; mp < C::MT / 2; ++mp) {
#pragma unroll
                for (int kk = 0; kk < C::KT; ++kk) {
                    const int t = kk * 16 + (mi & 1) * 8 + r;
                    const int unit = 2 * mp + (mi >> 1);
                    uint32_t r0, r1, r2, r3;
                    ldsm_x4_t(swz128(vt, t, unit * 16), r0, r1, r2, r3);
                    // r = {v[2c][2n], v[2c][2n+1], v[2c+1][2n], v[2c+1][2n+1]} bytes;
                    // the A operand wants the even bytes, then the odd ones
                    uint32_t A0[4], A1[4];
                    if (KVT == KV_INT8) {   // operands 1152 + c
                        s8x4_eo_to_f16x2_biased(r0, A0[0], A0[1]);
                        s8x4_eo_to_f16x2_biased(r1, A0[2], A0[3]);
                        s8x4_eo_to_f16x2_biased(r2, A1[0], A1[1]);
                        s8x4_eo_to_f16x2_biased(r3, A1[2], A1[3]);
                    } else {
                        const uint32_t x0 = prmt(r0, 0x3120), x1 = prmt(r1, 0x3120);
                        const uint32_t x2 = prmt(r2, 0x3120), x3 = prmt(r3, 0x3120);
                        code4_to_f16x2<KVT>(x0, A0[0], A0[1]);
                        code4_to_f16x2<KVT>(x1, A0[2], A0[3]);
                        code4_to_f16x2<KVT>(x2, A1[0], A1[1]);
                        code4_to_f16x2<KVT>(x3, A1[2], A1[3]);
                    }
                    mma_f16(o[2 * mp], A0, pq[kk][0], pq[kk][1]);
                    mma_f16(o[2 * mp + 1], A1, pq[kk][0], pq[kk][1]);
                }
            }
        } else {
            uint32_t pb[C::KT][2];
#pragma unroll
            for (int kk = 0; kk < C::KT; ++kk) {
                pb[kk][0] = movm_t(pack_bf16x2(sc[kk][0], sc[kk][1]));
                pb[kk][1] = movm_t(pack_bf16x2(sc[kk][2], sc[kk][3]));
            }
#pragma unroll
            for (int mt = 0; mt < C::MT; ++mt) {
                const int jg = 2 * mt + (mi & 1);
                const uint32_t vtile = vt + (jg >> 3) * C::CHS;
#pragma unroll
                for (int kk = 0; kk < C::KT; ++kk) {
                    const int t = kk * 16 + (mi >> 1) * 8 + r;
                    uint32_t A[4];
                    ldsm_x4_t(swz128(vtile, t, (jg & 7) * 16), A[0], A[1], A[2], A[3]);
                    mma_bf16(o[mt], A, pb[kk][0], pb[kk][1]);
                }
            }
        }
        if (ZERO_TAIL && valid < BS) fence_proxy_async_smem();  // generic writes before the next TMA fill
    }

    // Publish this warp's state for the item-level combine.
    __device__ __forceinline__ void publish(float* cm, float* cl, float* co, int warp, int lane) {
        // the 8 lanes of column c (lane bits 2-4) hold heads 2c and 2c + 1
#pragma unroll
        for (int x = 4; x < 32; x <<= 1) {
            l[0] += __shfl_xor_sync(0xffffffffu, l[0], x);
            l[1] += __shfl_xor_sync(0xffffffffu, l[1], x);
        }
        const int g = lane >> 2, c = lane & 3, n = lane >> 2;
        if (FP8) {
            // back from units of vref; the integer codes' offsets (times the sum
            // of the probabilities they met) come off, int4's odd dims were x16
#pragma unroll
            for (int x = 4; x < 32; x <<= 1) {
                psi[0] += __shfl_xor_sync(0xffffffffu, psi[0], x);
                psi[1] += __shfl_xor_sync(0xffffffffu, psi[1], x);
            }
            const float ps0 = psi[0], ps1 = psi[1];
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float ps = (e & 1) ? ps1 : ps0;
                    if (KVT == KV_INT8)
                        o[mt][e] = (o[mt][e] - kS8Bias * ps) * vref;
                    else if (KVT == KV_INT4)
                        o[mt][e] = (e >> 1) ? (o[mt][e] - kS4BiasHi * ps) * (vref * 0.0625f)
                                            : (o[mt][e] - kS4BiasLo * ps) * vref;
                    else
                        o[mt][e] *= vref;
                }
            }
        }
        if (g == 0) {
            cm[warp * 8 + 2 * c] = m[0];
            cm[warp * 8 + 2 * c + 1] = m[1];
            cl[warp * 8 + 2 * c] = l[0];
            cl[warp * 8 + 2 * c + 1] = l[1];
        }
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int gq = 2 * c + (e & 1);
                const int dim = KVT == KV_INT4 ? 32 * (mt >> 1) + 4 * n + 2 * (mt & 1) + (e >> 1)
                                : FP8          ? mt * 16 + 2 * n + (e >> 1)
                                               : mt * 16 + n + 8 * (e >> 1);
                co[(warp * 8 + gq) * D + dim] = o[mt][e];
            }
        }
    }
};

// The same page step on the CUDA cores (bf16 cache, head_dim 128, 16-token
// pages, G query heads per kv head fixed at compile time): S = Q K^T, the
// lazy-rescaled fp32 online softmax and O += P V, with packed two-wide fp32
// FMAs (fma.rn.f32x2) in place of the tensor-core MMAs.  It exists so that
// the two contractions can be timed against each other on the same kernel;
// PA_DECODE_FMA=1 selects it (see launch_heads).
//   Q K^T: lane (t, h) = (lane / 2, lane % 2) forms token t's G scores over
//     half h of head_dim, with q read as fp32 from shared memory (this head's
//     copy, [G][8 chunks of 8 dims][2 halves][8 floats]); the halves add with
//     one shuffle.
//   P V: lane owns dims 4 lane .. 4 lane + 3 of O for the G heads.  Token t's
//     probabilities reach every lane through the first 1 KB of this head's K
//     rows of the stage, which Q K^T no longer needs, as {p, p} pairs.  Rows
//     past the sequence's end are skipped, never multiplied.
template <int D, int BS, int HPC, int G>
struct WarpAccFma {
    static_assert(D == 128 && BS == 16 && (G == 4 || G == 8), "CUDA-core variant: d 128, 16-token pages, G 4 or 8");
    static constexpr int CHS = Cfg<D, BS, KV_BF16, HPC>::CHS;
    static_assert(BS * G * 8 <= BS * 128, "the probabilities fit in the head's K rows of one column tile");
    static constexpr int QS_BYTES = G * D * 4;   // this head's fp32 q
    float m[G], l[G];
    float o[G][4];
    uint32_t qs;   // shared address of this head's fp32 q

    __device__ __forceinline__ void reset() {
#pragma unroll
        for (int g = 0; g < G; ++g) {
            m[g] = -INFINITY;
            l[g] = 0.f;
            o[g][0] = o[g][1] = o[g][2] = o[g][3] = 0.f;
        }
    }

    // q rows of the head's G query heads (qrow: bf16 [G][D] in global memory)
    // into the head's shared copy, written by the head's first warp; every
    // warp of the head then meets at named barrier `bar`.
    __device__ __forceinline__ void load_q(const uint16_t* qrow, uint32_t qs_head, bool writer, int bar, int nthr,
                                           int lane) {
        qs = qs_head;
        if (writer) {
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const uint2 w = *reinterpret_cast<const uint2*>(qrow + g * D + lane * 4);
                const int d0 = lane * 4, half = d0 >> 6, j = (d0 & 63) >> 3, e = d0 & 7;
                const uint32_t a = qs + (((g * 8 + j) * 2 + half) * 8 + e) * 4;
                asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(a), "f"(__uint_as_float(w.x << 16)),
                             "f"(__uint_as_float(w.x & 0xFFFF0000u)), "f"(__uint_as_float(w.y << 16)),
                             "f"(__uint_as_float(w.y & 0xFFFF0000u))
                             : "memory");
            }
        }
        // literal barrier ids (1 per head) keep the kernel's barrier count at 3
        if (bar == 1)
            asm volatile("bar.sync 1, %0;" ::"r"(nthr) : "memory");
        else
            asm volatile("bar.sync 2, %0;" ::"r"(nthr) : "memory");
    }

    static __device__ __forceinline__ void fma2(float2& acc, float2 a, float2 b) {
        uint64_t d, x, y;
        asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(acc.x), "f"(acc.y));
        asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(a.x), "f"(a.y));
        asm("mov.b64 %0, {%1, %2};" : "=l"(y) : "f"(b.x), "f"(b.y));
        asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(d) : "l"(x), "l"(y));
        asm("mov.b64 {%0, %1}, %2;" : "=f"(acc.x), "=f"(acc.y) : "l"(d));
    }

    static __device__ __forceinline__ float2 bf2(uint32_t w) {
        return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
    }

    __device__ __forceinline__ void page(uint32_t kt, uint32_t vt, int valid, float sl2, float, int lane) {
        const int t = lane >> 1, h = lane & 1;
        // ------------------------------------------------ S^T = Q K^T
        float2 acc[G];
#pragma unroll
        for (int g = 0; g < G; ++g) acc[g] = make_float2(0.f, 0.f);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            uint32_t k0, k1, k2, k3;
            asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(k0), "=r"(k1), "=r"(k2), "=r"(k3)
                         : "r"(swz128(kt + h * CHS, t, j * 16)));
            const float2 kp0 = bf2(k0), kp1 = bf2(k1), kp2 = bf2(k2), kp3 = bf2(k3);
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const uint32_t qa = qs + ((g * 8 + j) * 2 + h) * 32;
                float4 q0, q1;
                asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                             : "=f"(q0.x), "=f"(q0.y), "=f"(q0.z), "=f"(q0.w)
                             : "r"(qa));
                asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                             : "=f"(q1.x), "=f"(q1.y), "=f"(q1.z), "=f"(q1.w)
                             : "r"(qa + 16));
                fma2(acc[g], make_float2(q0.x, q0.y), kp0);
                fma2(acc[g], make_float2(q0.z, q0.w), kp1);
                fma2(acc[g], make_float2(q1.x, q1.y), kp2);
                fma2(acc[g], make_float2(q1.z, q1.w), kp3);
            }
        }
        // ------------------------------------------------ online softmax
        float sc[G];
        bool grow = false;
#pragma unroll
        for (int g = 0; g < G; ++g) {
            float sv = acc[g].x + acc[g].y;
            sv += __shfl_xor_sync(0xffffffffu, sv, 1);
            sc[g] = t < valid ? sv * sl2 : -INFINITY;
            grow |= sc[g] > m[g] + 8.f;   // m == -inf: any finite score
        }
        // Lazy rescale, as in WarpAcc: the reference m moves only when a score
        // exceeds it by more than 2^8
        if (__any_sync(0xffffffffu, grow)) {
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float pm = sc[g];
#pragma unroll
                for (int o2 = 2; o2 < 32; o2 <<= 1) pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, o2));
                const float m_new = pm > m[g] + 8.f ? pm : m[g];
                const float alpha = m_new == m[g] ? 1.f : exp2f(m[g] - m_new);   // m == -inf: 0
                l[g] *= alpha;
                o[g][0] *= alpha;
                o[g][1] *= alpha;
                o[g][2] *= alpha;
                o[g][3] *= alpha;
                m[g] = m_new;
            }
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
            sc[g] = ex2_approx(sc[g] - (m[g] == -INFINITY ? 0.f : m[g]));
            if (h == 0) l[g] += sc[g];
        }
        __syncwarp();   // every lane's K reads are done: the rows take the probabilities
        // layout [G / 2 head pairs][BS tokens] of {p_g, p_g, p_g+1, p_g+1}
        if (h == 0) {
#pragma unroll
            for (int g = 0; g < G; g += 2)
                asm volatile("st.shared.v4.f32 [%0], {%1, %1, %2, %2};" ::"r"(kt + ((g / 2) * BS + t) * 16),
                             "f"(sc[g]), "f"(sc[g + 1])
                             : "memory");
        }
        __syncwarp();
        // ------------------------------------------------ O += P V
        const uint32_t vcol = vt + (lane >> 4) * CHS;
        const int vbyte = (lane * 8) & 127;
#pragma unroll
        for (int tt = 0; tt < BS; ++tt) {
            if (tt < valid) {
                uint32_t v0, v1;
                asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v0), "=r"(v1) : "r"(swz128(vcol, tt, vbyte)));
                const float2 vp0 = bf2(v0), vp1 = bf2(v1);
#pragma unroll
                for (int g = 0; g < G; g += 2) {
                    float4 pp;
                    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                                 : "=f"(pp.x), "=f"(pp.y), "=f"(pp.z), "=f"(pp.w)
                                 : "r"(kt + ((g / 2) * BS + tt) * 16));
                    float2 a0 = make_float2(o[g][0], o[g][1]), a1 = make_float2(o[g][2], o[g][3]);
                    float2 b0 = make_float2(o[g + 1][0], o[g + 1][1]), b1 = make_float2(o[g + 1][2], o[g + 1][3]);
                    fma2(a0, make_float2(pp.x, pp.y), vp0);
                    fma2(a1, make_float2(pp.x, pp.y), vp1);
                    fma2(b0, make_float2(pp.z, pp.w), vp0);
                    fma2(b1, make_float2(pp.z, pp.w), vp1);
                    o[g][0] = a0.x, o[g][1] = a0.y, o[g][2] = a1.x, o[g][3] = a1.y;
                    o[g + 1][0] = b0.x, o[g + 1][1] = b0.y, o[g + 1][2] = b1.x, o[g + 1][3] = b1.y;
                }
            }
        }
        fence_proxy_async_smem();   // generic writes into the stage before its next TMA fill
    }

    __device__ __forceinline__ void publish(float* cm, float* cl, float* co, int warp, int lane) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
            float ls = l[g];
#pragma unroll
            for (int o2 = 1; o2 < 32; o2 <<= 1) ls += __shfl_xor_sync(0xffffffffu, ls, o2);
            if (lane == 0) {
                cm[warp * 8 + g] = m[g];
                cl[warp * 8 + g] = ls;
            }
            *reinterpret_cast<float4*>(co + (warp * 8 + g) * D + lane * 4) =
                make_float4(o[g][0], o[g][1], o[g][2], o[g][3]);
        }
    }
};

// CTA-level combine of the consumer warps' states, then the output: bf16 out
// for a one-partition sequence, else the partition's normalised partial and
// base-2 log-sum-exp.  Kv head h0 + hh is combined from warps hh * WPH ..
// hh * WPH + WPH - 1.  Threads tid < nthr take part.
template <int D, int WPH, int HPC>
__device__ __forceinline__ void combine_store(const DecodeArgs& a, const float* cm, const float* cl, const float* co,
                                              int b, int h0, int split, int nsplit, int tid, int nthr) {
    const int G = a.G;
    for (int idx = tid; idx < HPC * G * D; idx += nthr) {
        const int hg = idx / D, dim = idx - hg * D;
        const int hh = hg / G, gq = hg - hh * G;
        const int w0 = hh * WPH;
        float M = -INFINITY;
#pragma unroll
        for (int w = w0; w < w0 + WPH; ++w) M = fmaxf(M, cm[w * 8 + gq]);
        float L = 0.f, O = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = w0; w < w0 + WPH; ++w) {
                const float f = exp2f(cm[w * 8 + gq] - M);
                L += cl[w * 8 + gq] * f;
                O += co[(w * 8 + gq) * D + dim] * f;
            }
        }
        const int64_t row = (int64_t)b * a.Hq + (h0 + hh) * G + gq;
        const float val = (M == -INFINITY) ? 0.f : O / L;
        if (nsplit <= 1) {
            a.out[row * D + dim] = __float2bfloat16_rn(val);
        } else {
            a.o_part[(row * a.Sw + split) * D + dim] = val;
            if (dim == 0) a.lse[row * a.Sw + split] = (M == -INFINITY) ? -INFINITY : M + log2f(L);
        }
    }
}

// Log-sum-exp merge of a group's nsplit partials (the G query heads of each
// of the CTA's kv heads: rows row0 .. row0 + G - 1 of the output), by the
// group's last partition to finish:  out = sum_k 2^(lse_k - L) o_k.
// `sw` holds G * nsplit floats of shared memory.  A thread owns columns of 4
// consecutive dims of one row and keeps U partitions' float4 loads in flight
// per round trip (the first batch while the weights are computed).
template <int D>
__device__ __forceinline__ void merge_group(const DecodeArgs& a, float* sw, int64_t row0, int G, int nsplit,
                                           int tid, int nthr, int warp, int nwarps, int lane, void (*sync)()) {
    constexpr int U = 16, D4 = D / 4;
    const int ncol = G * D4;
    float4 pv[U];
    auto load_batch = [&](int col, int k0) {
        const int gq = col / D4, d4 = col - gq * D4;
        const float4* op = reinterpret_cast<const float4*>(a.o_part + (row0 + gq) * a.Sw * D) + d4;
#pragma unroll
        for (int u = 0; u < U; ++u)
            pv[u] = k0 + u < nsplit ? __ldcg(op + (int64_t)(k0 + u) * D4) : make_float4(0.f, 0.f, 0.f, 0.f);
    };
    if (tid < ncol) load_batch(tid, 0);
    for (int i = tid; i < G * nsplit; i += nthr) {
        const int gq = i / nsplit, k = i - gq * nsplit;
        sw[i] = __ldcg(&a.lse[(row0 + gq) * a.Sw + k]);
    }
    sync();
    for (int gq = warp; gq < G; gq += nwarps) {
        float* wr = sw + gq * nsplit;
        float mx = -INFINITY;
        for (int k = lane; k < nsplit; k += 32) mx = fmaxf(mx, wr[k]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        float den = 0.f;
        for (int k = lane; k < nsplit; k += 32) den += exp2f(wr[k] - mx);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
        const float inv = 1.f / den;
        __syncwarp();
        for (int k = lane; k < nsplit; k += 32) wr[k] = exp2f(wr[k] - mx) * inv;
    }
    sync();
    for (int col = tid; col < ncol; col += nthr) {
        const int gq = col / D4, d4 = col - gq * D4;
        const float* wr = sw + gq * nsplit;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int k0 = 0; k0 < nsplit; k0 += U) {
            if (k0 > 0 || col != tid) load_batch(col, k0);
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (k0 + u < nsplit) {
                    const float w = wr[k0 + u];
                    acc.x = fmaf(w, pv[u].x, acc.x);
                    acc.y = fmaf(w, pv[u].y, acc.y);
                    acc.z = fmaf(w, pv[u].z, acc.z);
                    acc.w = fmaf(w, pv[u].w, acc.w);
                }
            }
        }
        const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y), hi = __floats2bfloat162_rn(acc.z, acc.w);
        uint2 pk;
        pk.x = *reinterpret_cast<const uint32_t*>(&lo);
        pk.y = *reinterpret_cast<const uint32_t*>(&hi);
        *reinterpret_cast<uint2*>(a.out + (row0 + gq) * D + d4 * 4) = pk;
    }
}

__device__ __forceinline__ void sync_cta() { __syncthreads(); }

__device__ __forceinline__ int clamp_len(int len, int cap) { return len < 0 ? 0 : (len > cap ? cap : len); }

// Work items.  Sequence b of nblk blocks has max(1, ceil(nblk / pblk))
// partitions for each of the NH = Hkv / HPC kv-head sets (pblk = part_early
// for b < b_early, else part_blocks).  For batches of up to 256 sequences and
// at most 32 partitions (where partitions past a sequence's end are a large
// share of S * NH * B and each would hold a CTA slot for a while) the grid
// lists only these items: first partition 0 of every (sequence, head
// set), CTA r = b * NH + head set, mapped without any lookup; then the later
// partitions, sequence by sequence, then by head set, then by partition,
// which a CTA finds with one warp scan over the lengths.  CTAs past the last
// item have nothing to do, so no CTA slot goes to a partition past its
// sequence's end.  Other launches take every (sequence, head set, partition
// < S) in that order, with no scan; a partition past its sequence's end
// leaves once it has read the length.
struct WorkItem {
    int b, hs, split, raw_len;   // b < 0: no item
    int sh;                      // leading blocks attended by b's chunk (0: none)
    int chunk;                   // >= 0: a chunk item (b = its first member)
};

// Shared prefixes: the blocks of sequence b (clamped length len) that its
// chunk attends, or 0.  The same test decides, in b's own items and in its
// chunk's item, whether b takes part, so both count the same partials: b is
// member slot k of chunk c (chunk_of[b] = 8c + k, chunk_members[8c + k] = b,
// k < 8 / G, c < n_chunks) and the chunk's blocks lie before b's newest
// token.  A plan that fails it sets PA_DEVERR_BLOCK_ID; b is then attended
// without sharing.
template <int BS>
__device__ __forceinline__ int shared_blocks_of(const DecodeArgs& a, int b, int len) {
    const int v = a.chunk_of[b];
    if (v < 0) return 0;
    const int c = v / PA_SHARE_MAX_ROWS, k = v % PA_SHARE_MAX_ROWS;
    int cb = 0;
    const bool ok = c < a.n_chunks && k < PA_SHARE_MAX_ROWS / a.G && a.chunk_members[v] == b &&
                    (cb = a.chunk_blocks[c]) >= 1 && cb <= a.max_chunk_blocks && cb <= a.M && len >= 1 &&
                    cb <= (len - 1) / BS;
    if (!ok) {
        raise_error(PA_DEVERR_BLOCK_ID);
        return 0;
    }
    return cb;
}

// Partials of sequence b's output rows: its own partitions (blocks sh ..
// nblk - 1 in partitions of at most pblk) and, with a shared prefix, its
// chunk's partitions (sh blocks in partitions of at most part_blocks).
__device__ __forceinline__ int own_parts(int nblk, int sh, int pblk) {
    return (nblk - sh + pblk - 1) / pblk;
}
__device__ __forceinline__ int chunk_parts_of(const DecodeArgs& a, int sh) {
    return sh > 0 ? (sh + a.part_blocks - 1) / a.part_blocks : 0;
}

template <int BS>
__device__ __forceinline__ int partitions_of(const DecodeArgs& a, int b, int raw_len) {
    const int nblk = (clamp_len(raw_len, a.M * BS) + BS - 1) / BS;
    const int pblk = b < a.b_early ? a.part_early : a.part_blocks;
    return max(1, (nblk + pblk - 1) / pblk);
}

constexpr int kScanMaxBatch = 256;

// Later partition r (counted from the first item after the B * NH partitions
// 0), B <= kScanMaxBatch.  Called by one full warp.  Lane L covers sequences
// 8L .. 8L + 7; all lengths are loaded before the scan.
template <int BS, int HPC>
__device__ __forceinline__ WorkItem find_later_item(const DecodeArgs& a, int r, int lane) {
    const int NH = a.Hkv / HPC;
    int raw[8], ns[8], mine = 0;   // ns: partitions after the first
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const int bb = 8 * lane + k;
        raw[k] = bb < a.B ? a.lens[bb] : 0;
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const int bb = 8 * lane + k;
        ns[k] = bb < a.B ? partitions_of<BS>(a, bb, raw[k]) - 1 : 0;
        mine += ns[k] * NH;
    }
    int inc = mine;   // inclusive scan of the lanes' item counts
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += t;
    }
    WorkItem it{-1, 0, 0, 0, 0, -1};
    if (r >= __shfl_sync(0xffffffffu, inc, 31)) return it;   // past the last item
    const int src = __ffs(__ballot_sync(0xffffffffu, r < inc)) - 1;
    if (lane == src) {
        int off = r - (inc - mine);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int cnt = ns[k] * NH;
            if (it.b < 0 && off < cnt) {
                const int n = max(ns[k], 1);
                it.b = 8 * lane + k;
                it.hs = off / n;
                it.split = 1 + off - it.hs * n;
                it.raw_len = raw[k];
            }
            off -= cnt;
        }
    }
    it.b = __shfl_sync(0xffffffffu, it.b, src);
    it.hs = __shfl_sync(0xffffffffu, it.hs, src);
    it.split = __shfl_sync(0xffffffffu, it.split, src);
    it.raw_len = __shfl_sync(0xffffffffu, it.raw_len, src);
    return it;
}

// ========================================================================
// grid: the work items (see find_item), one CTA each
// ========================================================================
// Fused step.  The warp that consumes the page holding sequence b's position
// len-1 prepares this head's new row when the CTA starts (fp8: the block's new
// scale and the row's codes, computed while the first pages are in flight),
// then, once that page is in shared memory, writes the row into the page so
// that this page's attention sees it, and into the cache in global memory
// exactly as pa_kv_append would (no other CTA reads this page in this launch).
struct NewRow {
    uint2 kraw, vraw;    // this lane's 4 new bf16 values of K / V
    uint32_t kc, vc;     // fp8: their codes under the new scales
    float kold, vold;    // fp8: scales the older rows were encoded with (0 when the block restarts)
    float ks, vs;        // fp8: the block's new scales
};

template <int D, int KVT>
__device__ __forceinline__ NewRow prepare_new_row(const DecodeArgs& a, int b, int h, int phys, int off, int lane) {
    constexpr bool FP8 = KVT != KV_BF16;
    constexpr int CK = KVT == KV_BF16 ? KV_FP8 : KVT;
    using QC = Codec<CK>;
    NewRow r;
    const int64_t src = ((int64_t)b * a.Hkv + h) * D;
    r.kraw = r.vraw = make_uint2(0u, 0u);
    if (lane < D / 4) {
        r.kraw = *reinterpret_cast<const uint2*>(a.k_new + src + lane * 4);
        r.vraw = *reinterpret_cast<const uint2*>(a.v_new + src + lane * 4);
    }
    r.kc = r.vc = 0u;
    r.kold = r.vold = r.ks = r.vs = 1.f;
    if (FP8) {
        r.kold = off == 0 ? 0.f : a.k_scale_w[(int64_t)phys * a.Hkv + h];
        r.vold = off == 0 ? 0.f : a.v_scale_w[(int64_t)phys * a.Hkv + h];
        r.ks = fmaxf(r.kold, __fdiv_rn(warp_max(absmax4(r.kraw)), QC::QMAX));
        r.vs = fmaxf(r.vold, __fdiv_rn(warp_max(absmax4(r.vraw)), QC::QMAX));
        r.kc = q8_encode4<CK>(r.kraw, r.ks);
        r.vc = q8_encode4<CK>(r.vraw, r.vs);
    }
    return r;
}

template <int D, int BS, int KVT, int HPC>
__device__ __forceinline__ void patch_new_row_body(const DecodeArgs& a, int h, int phys, int off, uint32_t kt,
                                                   uint32_t vt, const NewRow& r, int lane) {
    constexpr bool FP8 = KVT != KV_BF16;
    constexpr int CHS = Cfg<D, BS, KVT, HPC>::CHS;
    using QC = CodecOf<KVT>;
    constexpr uint32_t MASK = (1u << QC::BITS) - 1;
    constexpr int ROWB = QC::BITS * D / 8;    // bytes of a coded row; lane owns QC::BITS / 2 of them
    const int64_t prow = ((int64_t)phys * a.Hkv + h) * BS;  // first row of the page
    if (FP8) {
        // a lane's 4 codes: one 32-bit word of a one-byte row, one 16-bit word of an int4 row
        auto ld4 = [&](uint32_t tile, int o) {
            uint32_t w;
            if (QC::BITS == 8)
                w = ld_shared_u32(tok_addr<BS, KVT, CHS>(tile, o, lane * 4));
            else {
                unsigned short hw;
                asm volatile("ld.shared.u16 %0, [%1];" : "=h"(hw) : "r"(tok_addr<BS, KVT, CHS>(tile, o, lane * 2)));
                w = hw;
            }
            return w;
        };
        auto st4 = [&](uint32_t tile, uint8_t* gpage, int o, uint32_t nw) {
            if (QC::BITS == 8) {
                asm volatile("st.shared.u32 [%0], %1;" ::"r"(tok_addr<BS, KVT, CHS>(tile, o, lane * 4)), "r"(nw) : "memory");
                reinterpret_cast<uint32_t*>(gpage)[o * 32 + lane] = nw;
            } else {
                asm volatile("st.shared.u16 [%0], %1;" ::"r"(tok_addr<BS, KVT, CHS>(tile, o, lane * 2)),
                             "h"((unsigned short)nw)
                             : "memory");
                reinterpret_cast<uint16_t*>(gpage)[o * 32 + lane] = (uint16_t)nw;
            }
        };
#pragma unroll
        for (int kv = 0; kv < 2; ++kv) {
            const uint32_t tile = kv == 0 ? kt : vt;
            uint8_t* gpage = (kv == 0 ? a.k_cache_w : a.v_cache_w) + prow * ROWB;
            const float old = kv == 0 ? r.kold : r.vold, sn = kv == 0 ? r.ks : r.vs;
            if (sn > old && old > 0.f) {  // the scale grew: re-encode the older rows (same rule as the append)
#pragma unroll 1
                for (int o = 0; o < off; ++o) {
                    const uint32_t w = ld4(tile, o);
                    uint32_t nw = 0;
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        nw |= QC::encode(__fdiv_rn(__fmul_rn(QC::value((w >> (QC::BITS * e)) & MASK), old), sn))
                              << (QC::BITS * e);
                    st4(tile, gpage, o, nw);
                }
            }
            st4(tile, gpage, off, kv == 0 ? r.kc : r.vc);
            if (lane == 0) (kv == 0 ? a.k_scale_w : a.v_scale_w)[(int64_t)phys * a.Hkv + h] = sn;
        }
    } else if (lane < D / 4) {
        const int ct = (lane * 4) / 64, byte = (lane * 4 % 64) * 2;
        asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(swz128(kt + ct * CHS, off, byte)), "r"(r.kraw.x),
                     "r"(r.kraw.y)
                     : "memory");
        asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(swz128(vt + ct * CHS, off, byte)), "r"(r.vraw.x),
                     "r"(r.vraw.y)
                     : "memory");
        *reinterpret_cast<uint2*>(reinterpret_cast<uint16_t*>(a.k_cache_w) + (prow + off) * D + lane * 4) = r.kraw;
        *reinterpret_cast<uint2*>(reinterpret_cast<uint16_t*>(a.v_cache_w) + (prow + off) * D + lane * 4) = r.vraw;
    }
    __syncwarp();
}

// The coded caches' patch (with the re-encode of older rows when the block
// scale grows) runs out of line: it runs once per CTA, and inlined into the
// page loop it cost that loop about 8% (register allocation and scheduling).
// The bf16 patch is a few stores and stays inline.
template <int D, int BS, int KVT, int HPC>
__device__ __noinline__ void patch_new_row_call(const DecodeArgs& a, int h, int phys, int off, uint32_t kt,
                                                uint32_t vt, const NewRow& r, int lane) {
    patch_new_row_body<D, BS, KVT, HPC>(a, h, phys, off, kt, vt, r, lane);
}

template <int D, int BS, int KVT, int HPC>
__device__ __forceinline__ void patch_new_row(const DecodeArgs& a, int h, int phys, int off, uint32_t kt, uint32_t vt,
                                              const NewRow& r, int lane) {
    if constexpr (KVT == KV_BF16)
        patch_new_row_body<D, BS, KVT, HPC>(a, h, phys, off, kt, vt, r, lane);
    else
        patch_new_row_call<D, BS, KVT, HPC>(a, h, phys, off, kt, vt, r, lane);
}

// GF = 0: tensor-core page step (WarpAcc); GF = G: the CUDA-core page step
// (WarpAccFma) for exactly G query heads per kv head.
template <int D, int BS, int KVT, int HPC, int GF, bool CUDA_CORES = (GF > 0 && KVT == KV_BF16)>
struct AccOf {
    using type = WarpAcc<D, BS, KVT, HPC>;
};
template <int D, int BS, int KVT, int HPC, int GF>
struct AccOf<D, BS, KVT, HPC, GF, true> {
    using type = WarpAccFma<D, BS, HPC, GF>;
};

// Epilogue of a chunk item: the CTA's rows (member m's query head g at row
// m * G + g of each kv head) go out as partial p of their member's output
// rows, in the slot after the member's own partitions; then each member's
// merge counter counts the partial, and the CTA merges every member whose
// partials it completed.
template <int D, int BS, int WPH, int HPC>
__device__ __noinline__ void chunk_epilogue(const DecodeArgs& a, const float* cm, const float* cl, const float* co,
                                            const int* members, int cb, int h0, int hs, int p, int warp, int lane) {
    constexpr int NTHR = (4 + 1) * 32;
    const int G = a.G, NH = a.Hkv / HPC, R = PA_SHARE_MAX_ROWS / G;
    __shared__ int s_slot[PA_SHARE_MAX_ROWS], s_tot[PA_SHARE_MAX_ROWS];
    __shared__ unsigned s_last;
    const int tid = threadIdx.x;
    if (tid < R) {
        const int bm = members[tid];
        if (bm >= 0) {
            const int nb = (clamp_len(a.lens[bm], a.M * BS) + BS - 1) / BS;
            const int own = own_parts(nb, cb, bm < a.b_early ? a.part_early : a.part_blocks);
            s_slot[tid] = own + p;
            s_tot[tid] = own + chunk_parts_of(a, cb);
        }
    }
    __syncthreads();
    for (int idx = tid; idx < HPC * R * G * D; idx += NTHR) {
        const int hr = idx / D, dim = idx - hr * D;
        const int hh = hr / (R * G), r = hr - hh * (R * G);
        const int m = r / G, gq = r - m * G;
        const int bm = members[m];
        if (bm < 0) continue;
        const int w0 = hh * WPH;
        float M = -INFINITY;
#pragma unroll
        for (int w = w0; w < w0 + WPH; ++w) M = fmaxf(M, cm[w * 8 + r]);
        float L = 0.f, O = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = w0; w < w0 + WPH; ++w) {
                const float f = exp2f(cm[w * 8 + r] - M);
                L += cl[w * 8 + r] * f;
                O += co[(w * 8 + r) * D + dim] * f;
            }
        }
        const int64_t row = (int64_t)bm * a.Hq + (h0 + hh) * G + gq;
        a.o_part[(row * a.Sw + s_slot[m]) * D + dim] = (M == -INFINITY) ? 0.f : O / L;
        if (dim == 0) a.lse[row * a.Sw + s_slot[m]] = (M == -INFINITY) ? -INFINITY : M + log2f(L);
    }
    __syncthreads();   // every thread's partial stores precede the counts
    if (tid == 0) {
        unsigned last = 0;
        for (int m = 0; m < R; ++m) {
            const int bm = members[m];
            if (bm < 0) continue;
            int old;
            asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;"
                         : "=r"(old)
                         : "l"(&a.counters[bm * NH + hs])
                         : "memory");
            if (old == s_tot[m] - 1) last |= 1u << m;
        }
        s_last = last;
    }
    __syncthreads();
    // the merge scratch: the combine area, free once the partials are out
    float* sw = const_cast<float*>(cm);
    for (unsigned last = s_last; last; last &= last - 1) {
        const int m = __ffs(last) - 1, bm = members[m];
        merge_group<D>(a, sw, (int64_t)bm * a.Hq + h0 * G, HPC * G, s_tot[m], tid, NTHR, warp, 5, lane, sync_cta);
        if (tid == 0) a.counters[bm * NH + hs] = 0;
        __syncthreads();
    }
}

// SHARED: the launch also lists chunk items (shared prefixes) ahead of the
// sequences' own items, always on the direct grid.
template <int D, int BS, int KVT, int NSTAGE, bool APPEND, int HPC, int GF = 0, bool SHARED = false>
__global__ void __launch_bounds__(Cfg<D, BS, KVT, HPC>::NTHREADS, 3)
    paged_decode_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                        const DecodeArgs a) {
    using C = Cfg<D, BS, KVT, HPC>;
    using Acc = typename AccOf<D, BS, KVT, HPC, GF>::type;
    constexpr bool FP8 = C::FP8;
    constexpr int BAR_OFF = NSTAGE * C::STAGEB;
    constexpr int WPH = C::WPH;
    static_assert(C::COMBINE_FLOATS * 4 <= NSTAGE * C::STAGEB, "combine area must fit in the stages");
    // stage s is always consumed by warps hh * WPH + s % WPH (one per kv head),
    // so no waiter can run two phases ahead of a stage's oldest unconsumed
    // fill (parity waits alias)
    static_assert(NSTAGE % WPH == 0, "ring depth must be a multiple of the consumer warps per head");
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    const uint32_t sbase = (raw_u32 + 1023u) & ~1023u;
    uint8_t* sgen = smem_raw + (sbase - raw_u32);
    uint64_t* full = reinterpret_cast<uint64_t*>(sgen + BAR_OFF);
    uint64_t* empty = full + NSTAGE;
    // Coded caches: the (K, V) scales per head of the pages of a 32-page batch,
    // in two slots (batch n in slot n % 2), each published by the producer at
    // the batch's start with one arrival on its barrier.  A slot is rewritten
    // two batches later, when every page of its batch has been released (the
    // ring holds at most 32 pages).
    __shared__ float2 batch_sc[FP8 ? 2 : 1][32][HPC];
    __shared__ uint64_t batch_bar[2];
    static_assert(NSTAGE <= 32, "a batch slot is reused only after its pages are released");

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool scan = !SHARED && a.scan != 0;
    // SHARED: the first n_chunks * NH * chunk_parts CTAs are chunk items
    const int n_citems = SHARED ? a.n_chunks * (a.Hkv / HPC) * a.chunk_parts : 0;
    const bool is_chunk = SHARED && (int)blockIdx.x < n_citems;
    const int rid = (int)blockIdx.x - n_citems;   // regular item index
    if (!scan && !is_chunk) {
        // a partition this sequence can never use (a table holds at most M
        // blocks): leave before any set-up or load
        const int b0 = rid / a.S / (a.Hkv / HPC), split0 = rid % a.S;
        const int pblk0 = b0 < a.b_early ? a.part_early : a.part_blocks;
        if (split0 > 0 && split0 >= (a.M + pblk0 - 1) / pblk0) return;
    }

    if (threadIdx.x == 0) {
        for (int s = 0; s < NSTAGE; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], HPC);   // released once per kv head
        }
        mbar_init(&batch_bar[0], 1);
        mbar_init(&batch_bar[1], 1);
        fence_mbar_init();
    }
    // Inputs may come from the preceding kernel in the stream (this step's
    // append): wait for it before the first global read.
    griddep_wait();

    __shared__ WorkItem s_item;
    __shared__ int s_members[PA_SHARE_MAX_ROWS];   // chunk items: member sequences that take part (-1: none)
    const int NH = a.Hkv / HPC;
    // partition 0 of (b, head set): mapped directly, the table read with the
    // length (not with shared prefixes: a sequence's own blocks start later)
    const bool first = !SHARED && (scan ? (int)blockIdx.x < a.B * NH : (int)blockIdx.x % a.S == 0);
    int phys0 = 0;
    if (warp == C::NCW) {
        if (is_chunk) {
            const int per = NH * a.chunk_parts;
            const int c = (int)blockIdx.x / per, hs = ((int)blockIdx.x % per) / a.chunk_parts,
                      p = (int)blockIdx.x % a.chunk_parts;
            const int cb = a.chunk_blocks[c];
            // member slot `lane`: the sequence takes part when its own items
            // count this chunk's partials (the same test, shared_blocks_of)
            int mb = -1;
            if (lane < PA_SHARE_MAX_ROWS / a.G) {
                const int bm = a.chunk_members[c * PA_SHARE_MAX_ROWS + lane];
                if (bm >= 0 && bm < a.B && a.chunk_of[bm] == c * PA_SHARE_MAX_ROWS + lane &&
                    shared_blocks_of<BS>(a, bm, clamp_len(a.lens[bm], a.M * BS)) == cb)
                    mb = bm;
            }
            if (lane < PA_SHARE_MAX_ROWS) s_members[lane] = mb;
            const int lead = __shfl_sync(0xffffffffu, mb, __ffs(__ballot_sync(0xffffffffu, mb >= 0)) - 1);
            const bool any = __any_sync(0xffffffffu, mb >= 0);
            // the first member's table row names the shared blocks; every page is full
            if (lane == 0) s_item = WorkItem{any ? lead : -1, hs, p, cb * BS, cb, c};
        } else if (!scan) {
            const int q = rid / a.S, b0 = q / NH;
            if (first && lane < a.M) phys0 = a.tables[(int64_t)b0 * a.M + lane];
            if (lane == 0) {
                const int l0 = a.lens[b0];
                const int sh0 = SHARED ? shared_blocks_of<BS>(a, b0, clamp_len(l0, a.M * BS)) : 0;
                s_item = WorkItem{b0, q - b0 * NH, rid - q * a.S, l0, sh0, -1};
            }
        } else if (first) {
            const int b0 = blockIdx.x / NH;
            // partition 0 starts at block 0: the first table entries come
            // alongside the length (entries past the sequence are not used)
            if (lane < a.M) phys0 = a.tables[(int64_t)b0 * a.M + lane];
            if (lane == 0) s_item = WorkItem{b0, (int)blockIdx.x - b0 * NH, 0, a.lens[b0], 0, -1};
        } else {
            const WorkItem it = find_later_item<BS, HPC>(a, blockIdx.x - a.B * NH, lane);
            if (lane == 0) s_item = it;
        }
    }
    __syncthreads();   // also publishes the barrier initialisation
    const WorkItem it = s_item;
    if (it.b < 0) return;   // past the last item
    const int b = it.b, split = it.split;
    const int h0 = it.hs * HPC;   // this CTA's kv heads: h0 .. h0 + HPC - 1
    int len = it.raw_len;
    const int cap = a.M * BS;
    if (len < 0 || len > cap) {
        if (threadIdx.x == 0 && split == 0 && h0 == 0) raise_error(PA_DEVERR_SEQ_LEN);
        len = clamp_len(len, cap);
    }
    const int nblk = (len + BS - 1) / BS;
    // a chunk item covers the chunk's sh blocks; a sequence's own items its blocks sh .. nblk - 1
    const int sh = SHARED ? it.sh : 0;
    const bool chunk = SHARED && it.chunk >= 0;
    const int base = chunk ? 0 : sh;
    const int span = chunk ? sh : nblk - sh;
    const int pblk = chunk ? a.part_blocks : (b < a.b_early ? a.part_early : a.part_blocks);
    const int nsplit = (span + pblk - 1) / pblk;  // 0 when len == 0 (one item, no pages)
    if (split > 0 && split >= nsplit) return;     // (direct grid) past the sequence's end
    // the blocks split evenly over the partitions (at most P each)
    const int pb = nsplit > 0 ? (span + nsplit - 1) / nsplit : 0;
    const int j0 = base + split * pb;
    const int npages = max(0, min(base + span, j0 + pb) - j0);
    const int32_t* trow = a.tables + (int64_t)b * a.M + j0;
    if (!first && warp == C::NCW && lane < npages) phys0 = trow[lane];

    Acc st;
    st.reset();
    if (warp == C::NCW) {
        if (lane == 0) {
            prefetch_tensormap(&tm_k);
            prefetch_tensormap(&tm_v);
        }
        bool alive = true;
        int issued = 0;   // lane 0: pages whose copies were issued
        // batch n's block ids (and, coded caches, scales): loaded during batch
        // n - 1, so that neither a copy nor the consumers wait for them
        auto load_batch = [&](int base, int& phys, float (&ks)[HPC], float (&vs)[HPC]) {
            phys = 0;
#pragma unroll
            for (int hh = 0; hh < HPC; ++hh) ks[hh] = vs[hh] = 1.f;
            if (base + lane < npages) {
                phys = base == 0 ? phys0 : trow[base + lane];   // batch 0's were loaded at the start
                if (phys < 0 || phys >= a.num_blocks) {
                    raise_error(PA_DEVERR_BLOCK_ID);
                    phys = -1;  // loads read block 0; nothing is written through it
                }
                if (FP8) {
                    const int64_t si = (int64_t)(phys < 0 ? 0 : phys) * a.Hkv + h0;
#pragma unroll
                    for (int hh = 0; hh < HPC; ++hh) {
                        ks[hh] = a.k_scale[si + hh];
                        vs[hh] = a.v_scale[si + hh];
                    }
                }
            }
        };
        int myphys;
        float mks[HPC], mvs[HPC];
        load_batch(0, myphys, mks, mvs);
        for (int base = 0; base < npages; base += 32) {
            const int nb = base / 32;
            if (FP8) {   // this batch's scales for the consumers
#pragma unroll
                for (int hh = 0; hh < HPC; ++hh) batch_sc[nb & 1][lane][hh] = make_float2(mks[hh], mvs[hh]);
                __syncwarp();
                if (lane == 0) mbar_arrive(&batch_bar[nb & 1]);
            }
            int nphys = 0;
            float nks[HPC], nvs[HPC];
            if (base + 32 < npages) load_batch(base + 32, nphys, nks, nvs);
            const int cnt = min(32, npages - base);
            for (int k = 0; k < cnt; ++k) {
                const int phys_raw = __shfl_sync(0xffffffffu, myphys, k);
                const int phys = phys_raw < 0 ? 0 : phys_raw;
                if (lane == 0 && alive) {
                    const int i = base + k;
                    const int s = i % NSTAGE;
                    if (i >= NSTAGE) alive = mbar_wait(&empty[s], ((i / NSTAGE) - 1) & 1);
                    if (alive) {
                        mbar_arrive_expect_tx(&full[s], C::STAGEB);
                        // one box: the block's rows for kv heads h0 .. h0 + HPC - 1
                        const int y = (phys * a.Hkv + h0) * C::LINES;
                        uint8_t* stg = sgen + s * C::STAGEB;
#pragma unroll
                        for (int ch = 0; ch < C::NCH; ++ch)
                            tma_load_2d(stg + ch * C::CHS, &tm_k, ch * (128 / C::ELT), y, &full[s]);
#pragma unroll
                        for (int ch = 0; ch < C::NCH; ++ch)
                            tma_load_2d(stg + HPC * C::PAGEB + ch * C::CHS, &tm_v, ch * (128 / C::ELT), y, &full[s]);
                        issued = i + 1;
                    }
                }
            }
            myphys = nphys;
#pragma unroll
            for (int hh = 0; hh < HPC; ++hh) {
                mks[hh] = nks[hh];
                mvs[hh] = nvs[hh];
            }
        }
        // every issued load lands before the shared memory is reused or released
        if (lane == 0) {
            for (int s = 0; s < NSTAGE && s < issued; ++s) {
                const int last = s + ((issued - 1 - s) / NSTAGE) * NSTAGE;
                mbar_wait(&full[s], (last / NSTAGE) & 1);
            }
        }
    } else {
        // consumer warp: kv head h = h0 + hh, pages i with i mod WPH == wi
        const int hh = warp / WPH, wi = warp - hh * WPH, h = h0 + hh;
        if constexpr (GF > 0) {
            // the head's q in shared memory (after the barriers), written by its first warp
            const uint32_t qs_head = sbase + BAR_OFF + 2 * NSTAGE * 8 + hh * Acc::QS_BYTES;
            st.load_q(a.q + ((int64_t)b * a.Hq + h * GF) * D, qs_head, wi == 0, 1 + hh, WPH * 32, lane);
        } else if (chunk) {
            // q column g: query head g % G of member g / G
            const int g = lane >> 2, m = g / a.G;
            const int bm = m < PA_SHARE_MAX_ROWS / a.G ? s_members[m] : -1;
            st.load_q(a.q + ((int64_t)max(bm, 0) * a.Hq + h * a.G + g % a.G) * D, bm >= 0, lane & 3);
        } else {
            const int g = lane >> 2;
            st.load_q(a.q + ((int64_t)b * a.Hq + h * a.G + g) * D, g < a.G, lane & 3);
        }
        // fused step: the warp that consumes the page holding position len-1 fetches
        // its head's new K/V row (and the block's scales) up front
        const bool appends = APPEND && !chunk && split == nsplit - 1 && npages > 0 && wi == (npages - 1) % WPH;
        int app_phys = -1;
        // the row waits in shared memory, not in registers, until its page arrives
        __shared__ NewRow s_nr[APPEND ? HPC : 1][32];
        if (appends) {
            app_phys = trow[npages - 1];
            if (app_phys < 0 || app_phys >= a.num_blocks) app_phys = -1;
            if (app_phys >= 0) s_nr[hh][lane] = prepare_new_row<D, KVT>(a, b, h, app_phys, (len - 1) % BS, lane);
        }
        for (int i = wi; i < npages; i += WPH) {
            const int s = i % NSTAGE;
            float ksc = 1.f, vsc = 1.f;
            if (FP8) {   // the batch's scales, published at the batch's start
                const int nb = i / 32;
                if ((i & 31) == wi && !mbar_wait(&batch_bar[nb & 1], (nb >> 1) & 1)) break;   // warp's first page of it
                const float2 sv = batch_sc[nb & 1][i & 31][hh];
                ksc = sv.x;
                vsc = sv.y;
            }
            if (!mbar_wait(&full[s], (i / NSTAGE) & 1)) break;
            // this head's rows of the stage: line hh * LINES of each column tile
            const uint32_t kt = sbase + s * C::STAGEB + hh * C::LINES * 128;
            const uint32_t vt = kt + HPC * C::PAGEB;
            const bool patched = appends && i == npages - 1 && app_phys >= 0;
            if (patched) {
                const NewRow nr = s_nr[hh][lane];
                patch_new_row<D, BS, KVT, HPC>(a, h, app_phys, (len - 1) % BS, kt, vt, nr, lane);
                if (FP8) {
                    ksc = nr.ks;
                    vsc = nr.vs;
                }
            }
            st.page(kt, vt, min(BS, len - (j0 + i) * BS), FP8 ? a.scale_log2 * ksc : a.scale_log2, vsc, lane);
            if (patched) fence_proxy_async_smem();  // generic writes before the next TMA fill
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }
    }

    __syncthreads();  // pipeline drained: the stage memory becomes the combine area
    // the item again, from shared memory: none of it stays in registers
    // across the page loop
    const WorkItem ie = s_item;
    const int eb = ie.b, eh0 = ie.hs * HPC, esplit = ie.split;
    float* cm = reinterpret_cast<float*>(sgen);
    float* cl = cm + C::NCW * 8;
    float* co = cl + C::NCW * 8;
    if (warp < C::NCW) st.publish(cm, cl, co, warp, lane);
    __syncthreads();
    if constexpr (SHARED) {
        if (ie.chunk >= 0) {
            chunk_epilogue<D, BS, WPH, HPC>(a, cm, cl, co, s_members, ie.sh, eh0, ie.hs, esplit, warp, lane);
            return;
        }
    }
    // the sequence's partials: its own partitions and, with a shared prefix, its chunk's
    const int esh = SHARED ? ie.sh : 0;
    const int ensplit = own_parts((clamp_len(ie.raw_len, cap) + BS - 1) / BS, esh,
                                  eb < a.b_early ? a.part_early : a.part_blocks) + chunk_parts_of(a, esh);
    combine_store<D, WPH, HPC>(a, cm, cl, co, eb, eh0, esplit, ensplit, threadIdx.x, C::NTHREADS);
    if (ensplit <= 1) return;

    // the group: this CTA's kv heads of sequence b, counted per head set
    const int grp = eb * (a.Hkv / HPC) + ie.hs;
    __shared__ int s_last;
    __syncthreads();   // every thread's partial stores precede the count
    if (threadIdx.x == 0) {
        // one acquire-release count: it releases this CTA's partials (ordered
        // before it by the barrier) and, for the group's last partition,
        // acquires the others' (the barrier below passes that on)
        int old;
        asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(old) : "l"(&a.counters[grp]) : "memory");
        s_last = (old == ensplit - 1);
    }
    __syncthreads();
    if (!s_last) return;
    merge_group<D>(a, cm, (int64_t)eb * a.Hq + eh0 * a.G, HPC * a.G, ensplit, threadIdx.x, C::NTHREADS, warp,
                   C::NCW + 1, lane, sync_cta);
    if (threadIdx.x == 0) a.counters[grp] = 0;
}

// ------------------------------------------------------------------ launch
template <typename K>
static cudaError_t set_smem_once(K kernel, int smem, int& configured_device) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured_device != dev) {  // the attribute is per device
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    return cudaSuccess;
}

template <int D, int BS, int KVT, bool APPEND, int HPC, int GF = 0, bool SHARED = false>
static cudaError_t launch_typed(const DecodeLaunch& L, cudaStream_t stream) {
    using C = Cfg<D, BS, KVT, HPC>;
    DecodeArgs a;
    a.out = (__nv_bfloat16*)L.out;
    a.q = (const uint16_t*)L.q;
    a.k_scale = L.k_scale;
    a.v_scale = L.v_scale;
    a.tables = L.tables;
    a.lens = L.lens;
    a.o_part = L.o_part;
    a.lse = L.lse;
    a.counters = L.counters;
    a.k_new = (const uint16_t*)L.k_new;
    a.v_new = (const uint16_t*)L.v_new;
    a.k_cache_w = (uint8_t*)L.k_cache_w;
    a.v_cache_w = (uint8_t*)L.v_cache_w;
    a.k_scale_w = L.k_scale_w;
    a.v_scale_w = L.v_scale_w;
    a.B = L.B;
    a.Hq = L.Hq;
    a.Hkv = L.Hkv;
    a.G = L.Hq / L.Hkv;
    a.M = L.M;
    a.num_blocks = L.num_blocks;
    a.part_blocks = L.part_blocks;
    // Short partitions (under 128 pages per CTA): the first half of the
    // batch, whose CTAs start first, takes partitions up to twice as long (at
    // most 128 pages per CTA), so fewer CTAs start and finish in the early
    // waves and the last CTAs to start are the short ones.
    a.b_early = L.part_blocks * HPC < 128 ? L.B / 2 : 0;
    a.part_early = std::min(std::min(2 * L.part_blocks, 128 / HPC), L.M);
    a.S = L.S;
    a.scan = L.B <= kScanMaxBatch && L.S <= 32;
    a.scale_log2 = L.scale * 1.4426950408889634f;
    a.Sw = L.Sw;
    a.chunk_of = L.chunk_of;
    a.chunk_members = L.chunk_members;
    a.chunk_blocks = L.chunk_blocks;
    a.n_chunks = SHARED ? L.n_chunks : 0;
    a.chunk_parts = L.chunk_parts;
    a.max_chunk_blocks = L.max_chunk_blocks;
    if (SHARED) {
        // every partition count follows from (length, shared blocks): no early doubling, direct grid
        a.b_early = 0;
        a.scan = 0;
    }
    constexpr int NST = 65536 / C::STAGEB;   // 64 KB of stages
    // the CUDA-core page step keeps each head's q (fp32) after the barriers
    constexpr int QS = GF > 0 ? HPC * GF * D * 4 : 0;
    constexpr int SMEM = NST * C::STAGEB + 2 * NST * 8 + QS + 1024;
    static int configured = -1;
    cudaError_t e = set_smem_once(paged_decode_kernel<D, BS, KVT, NST, APPEND, HPC, GF, SHARED>, SMEM, configured);
    if (e != cudaSuccess) return e;
    // programmatic stream serialisation: the CTAs may be scheduled while the
    // previous kernel (typically this step's append) finishes; they wait for it
    // in griddep_wait() before reading any input
    cudaLaunchConfig_t cfg = {};
    // an upper bound on the work items: every sequence at most S partitions
    // (shared prefixes: the chunk items first)
    cfg.gridDim = dim3((unsigned)L.S * (unsigned)(L.Hkv / HPC) * (unsigned)L.B +
                       (SHARED ? (unsigned)L.n_chunks * (unsigned)(L.Hkv / HPC) * (unsigned)L.chunk_parts : 0u));
    cfg.blockDim = dim3(C::NTHREADS);
    cfg.dynamicSmemBytes = SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, paged_decode_kernel<D, BS, KVT, NST, APPEND, HPC, GF, SHARED>, *L.tm_k, *L.tm_v,
                              a);
}

// PA_DECODE_FMA=1 in the environment selects the CUDA-core page step
// (WarpAccFma) where it exists (bf16 cache, head_dim 128, 16-token pages,
// G = 4 or 8); the tensor-core step is the default.  A measurement switch:
// both give the same quantity within the parity bound.
static bool fma_requested() {
    const char* e = getenv("PA_DECODE_FMA");
    return e && e[0] == '1';
}

// Kv heads per CTA: 2 when the count is even (the tensor maps' boxes then
// span two heads' pages), else 1.
template <int D, int BS, int KVT, bool APPEND>
static cudaError_t launch_heads(const DecodeLaunch& L, cudaStream_t stream) {
    if (L.n_chunks > 0)   // shared prefixes
        return L.hpc == 2 ? launch_typed<D, BS, KVT, APPEND, 2, 0, true>(L, stream)
                          : launch_typed<D, BS, KVT, APPEND, 1, 0, true>(L, stream);
    if constexpr (KVT == KV_BF16 && D == 128 && BS == 16) {
        const int G = L.Hq / L.Hkv;
        if (fma_requested() && (G == 4 || G == 8)) {
            if (L.hpc == 2)
                return G == 4 ? launch_typed<D, BS, KVT, APPEND, 2, 4>(L, stream)
                              : launch_typed<D, BS, KVT, APPEND, 2, 8>(L, stream);
            return G == 4 ? launch_typed<D, BS, KVT, APPEND, 1, 4>(L, stream)
                          : launch_typed<D, BS, KVT, APPEND, 1, 8>(L, stream);
        }
    }
    return L.hpc == 2 ? launch_typed<D, BS, KVT, APPEND, 2>(L, stream) : launch_typed<D, BS, KVT, APPEND, 1>(L, stream);
}

template <bool APPEND>
static cudaError_t launch_shape(const DecodeLaunch& L, cudaStream_t stream) {
    if (L.kvt == PA_KV_FP8_E4M3) {
        if (L.d == 128 && L.bs == 16) return launch_heads<128, 16, KV_FP8, APPEND>(L, stream);
        if (L.d == 128 && L.bs == 32) return launch_heads<128, 32, KV_FP8, APPEND>(L, stream);
    } else if (L.kvt == PA_KV_INT8) {
        if (L.d == 128 && L.bs == 16) return launch_heads<128, 16, KV_INT8, APPEND>(L, stream);
        if (L.d == 128 && L.bs == 32) return launch_heads<128, 32, KV_INT8, APPEND>(L, stream);
    } else if (L.kvt == PA_KV_INT4) {
        if (L.d == 128 && L.bs == 16) return launch_heads<128, 16, KV_INT4, APPEND>(L, stream);
        if (L.d == 128 && L.bs == 32) return launch_heads<128, 32, KV_INT4, APPEND>(L, stream);
    } else {
        if (L.d == 128 && L.bs == 16) return launch_heads<128, 16, KV_BF16, APPEND>(L, stream);
        if (L.d == 128 && L.bs == 32) return launch_heads<128, 32, KV_BF16, APPEND>(L, stream);
        if (L.d == 64 && L.bs == 16) return launch_heads<64, 16, KV_BF16, APPEND>(L, stream);
        if (L.d == 64 && L.bs == 32) return launch_heads<64, 32, KV_BF16, APPEND>(L, stream);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_decode(const DecodeLaunch& L, cudaStream_t stream) {
    return L.k_new ? launch_shape<true>(L, stream) : launch_shape<false>(L, stream);
}

cudaError_t decode_unit_error(unsigned int* v, bool clear) { return read_unit_error(v, clear); }

}  // namespace pa
