// Decode attention with the sequence's K/V blocks staged in shared memory.
//
// Same arithmetic as attention_core (scores by dp4a, base-2 logits, exact
// row maximum, 15-bit E_j, num = 256 sum E_hi v8 + sum E_lo v8, one deferred
// division; DetLLM blog footnote on 15-bit probabilities), arranged for the
// latency of one decode step:
//  * every key before this step's token was written by earlier steps, so
//    its cache blocks are copied into shared memory (1D bulk copies, one
//    mbarrier) before the wait on the QKV GEMV; only the new token's key and
//    value arrive afterwards, written by the K/V warp into the staged block;
//  * scores and the P·V products read shared memory only, in orders that
//    spread each warp's 16-byte reads over all banks (key rows by a rotated
//    chunk order; value rows as 8 channels x 4 key chunks per warp);
//  * a ninth warp forms the row sums and the reciprocal RS while the others
//    run the P·V products.
// The staged layout holds ctx_cap keys (a multiple of 64); longer contexts
// use the per-token kernel.
#pragma once
#include "kernels.h"
#include "ptx.cuh"
#include "int_device.cuh"

namespace detint {

constexpr int AD_THREADS = 288;
constexpr int AD_MAXB = 64;   // staged cache blocks at most
constexpr int AD_SMEM_MAX = 220 * 1024;   // dynamic shared memory budget

// dynamic shared memory of the staged decode attention: K [cap][d],
// V^T [cap/64][d][64], q [MAXG][d], S [G][cap] int32, E_lo/E_hi [G][cap],
// P·V limbs [G][d][2] int32
__host__ __device__ inline size_t attn_dec_smem_bytes(int G, int d, int cap) {
    return (size_t)2 * cap * d + (size_t)MAXG * d + (size_t)G * cap * 4 + (size_t)2 * G * cap +
           (size_t)G * d * 8;
}

// G: q heads per kv head (a template constant, so that every per-head loop
// compiles to exactly G copies: the kernel runs once per SM per step, and its
// code arrives through a cold instruction cache)
template <int EPL, int G>
__global__ void __launch_bounds__(AD_THREADS) k_attn_dec_staged(AttnArgs a, QkvPostArgs qa) {
    extern __shared__ __align__(128) unsigned char sm[];
    constexpr int D = EPL * 32, NC = D >> 4;
    __shared__ int32_t mqs[MAXG], kqs[MAXG];
    __shared__ __align__(16) int16_t s_cos[64], s_sin[64], s_gq[128], s_gk[128];
    __shared__ int32_t s_kvp[8 + 64];
    __shared__ int s_bt[AD_MAXB];
    __shared__ unsigned long long cbar;
    __shared__ i64 umax_s[MAXG], rs_s[MAXG];
    __shared__ int bl_s[MAXG];
    __shared__ int red_i[8][MAXG];
    __shared__ i64 red_l[8][MAXG];

    const int t = blockIdx.x, g = blockIdx.y, tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
    const int dh2 = D >> 1, cap = a.ctx_cap;
    const int seq = a.tok_seq[t];
    const int p0 = a.seq_len[seq];            // keys before this step; the new key sits at p0
    const int ctx = p0 + 1, ctx16 = (ctx + 15) & ~15;
    const int nb = (ctx + KV_BLK - 1) >> 6;
    int8_t* Ks = (int8_t*)sm;                                  // [cap][D]
    int8_t* Vs = Ks + (size_t)cap * D;                         // [cap/64][D][64]
    int8_t* qs = Vs + (size_t)cap * D;                         // [MAXG][D]
    int32_t* S = (int32_t*)(qs + MAXG * D);                    // [G][cap]
    unsigned char* Elo = (unsigned char*)(S + (size_t)G * cap);
    unsigned char* Ehi = Elo + (size_t)G * cap;
    int32_t* pv = (int32_t*)(Ehi + (size_t)G * cap);           // [G][D][2]

    // ---- before the wait: everything that does not depend on this step.
    // The sequence length, block table and cache rows below p0 were written
    // by earlier steps; every step starts with a launch in plain stream order
    // (the embedding), so all of those writes are complete here even though
    // the kernels of this step overlap one another under PDL.
    if (tid < dh2) {
        s_cos[tid] = qa.rope_cos[(size_t)p0 * dh2 + tid];
        s_sin[tid] = qa.rope_sin[(size_t)p0 * dh2 + tid];
    }
    if (tid < D) { s_gq[tid] = qa.q_gamma[tid]; s_gk[tid] = qa.k_gamma[tid]; }
    if (tid < 8 + dh2) s_kvp[tid] = qa.kvp[(size_t)g * (8 + dh2) + tid];
    if (tid < nb) s_bt[tid] = a.block_table[(size_t)seq * a.mbs + tid];
    if (tid == 0) {
        mbar_init(smem_u32(&cbar), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    const uint32_t cb = smem_u32(&cbar);
    if (tid == 0) {
        constexpr uint32_t BLK = (uint32_t)KV_BLK * D;
        mbar_arrive_expect_tx(cb, (uint32_t)nb * 2u * BLK);
        for (int b = 0; b < nb; ++b) {
            const size_t unit = (size_t)s_bt[b] * a.nkv + g;
            bulk_g2s(smem_u32(Ks + (size_t)b * BLK), a.kc + unit * BLK, BLK, cb);
            bulk_g2s(smem_u32(Vs + (size_t)b * BLK), a.vc + unit * BLK, BLK, cb);
        }
    }
    pdl_wait();

    // ---- q heads of this kv group (one warp each) and the new key/value
    if (w < G) {
        qkv_head_p<EPL>(qa, t, (g << a.lg_grp) + w, qs + w * D, &mqs[w], &kqs[w], s_cos, s_sin, s_kvp,
                        s_gq, s_gk);
    } else if (w == G) {
        // the staged block must have landed before its new row is written
        if (!mbar_wait(cb, 0)) a.status[ST_TIMEOUT] = 1;
        qkv_head_p<EPL>(qa, t, a.nq + g, nullptr, nullptr, nullptr, s_cos, s_sin, s_kvp, s_gq, s_gk,
                        Ks + (size_t)p0 * D, Vs + (size_t)(nb - 1) * KV_BLK * D + (p0 & (KV_BLK - 1)));
    }
    if (!mbar_wait(cb, 0)) a.status[ST_TIMEOUT] = 1;
    __syncthreads();
    pdl_launch();

    const int32_t* kvp = s_kvp;
    const i64 CSTM = kvp[6], MV = kvp[4];
    const int CSTK = kvp[7], KVS = kvp[5];

    // ---- phase 1: scores and per-head maxima
    if (tid < 256) {
        int smax[G];
#pragma unroll
        for (int hh = 0; hh < G; ++hh) smax[hh] = -2147483647;
        for (int j = tid; j < ctx; j += 256) {
            const int8_t* kr = Ks + (size_t)j * D;
            int acc[G];
#pragma unroll
            for (int hh = 0; hh < G; ++hh) acc[hh] = 0;
#pragma unroll
            for (int v = 0; v < NC; ++v) {
                const int c = (v + j) & (NC - 1);
                const int4 kw = *(const int4*)(kr + c * 16);
#pragma unroll
                for (int hh = 0; hh < G; ++hh) {
                    const int4 qw = *(const int4*)(qs + hh * D + c * 16);
                    acc[hh] = __dp4a(kw.x, qw.x, acc[hh]);
                    acc[hh] = __dp4a(kw.y, qw.y, acc[hh]);
                    acc[hh] = __dp4a(kw.z, qw.z, acc[hh]);
                    acc[hh] = __dp4a(kw.w, qw.w, acc[hh]);
                }
            }
#pragma unroll
            for (int hh = 0; hh < G; ++hh) { S[hh * cap + j] = acc[hh]; smax[hh] = max(smax[hh], acc[hh]); }
        }
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
            const int v = __reduce_max_sync(0xffffffffu, smax[hh]);
            if (lane == 0) red_i[w][hh] = v;
        }
    }
    __syncthreads();
    if (tid < G) {
        int v = red_i[0][tid];
        for (int w2 = 1; w2 < 8; ++w2) v = max(v, red_i[w2][tid]);
        umax_s[tid] = rshr((i64)v * (i64)mqs[tid] * CSTM, kqs[tid] + CSTK - 10);
    }
    __syncthreads();

    // ---- phase 2: E_j (15 bits) as two byte planes, and the row sums
    if (tid < 256) {
        i64 sum[G];
#pragma unroll
        for (int hh = 0; hh < G; ++hh) sum[hh] = 0;
        for (int j = tid; j < ctx16; j += 256) {
#pragma unroll
            for (int hh = 0; hh < G; ++hh) {
                int E = 0;
                if (j < ctx) {
                    const i64 u = rshr((i64)S[hh * cap + j] * (i64)mqs[hh] * CSTM, kqs[hh] + CSTK - 10);
                    E = min(32767, exp2q_dev(u - umax_s[hh]));
                }
                Elo[hh * cap + j] = (unsigned char)(E & 255);
                Ehi[hh * cap + j] = (unsigned char)(E >> 8);
                sum[hh] += E;
            }
        }
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
            const i64 v = warp_sum_i64(sum[hh]);
            if (lane == 0) red_l[w][hh] = v;
        }
    }
    __syncthreads();

    if (w == 8) {
        // ---- row sums and RS = floor(2^(bl + 23) / sum), beside phase 3
        for (int hh = 0; hh < G; ++hh) {
            i64 v = 0;
            for (int w2 = 0; w2 < 8; ++w2) v += red_l[w2][hh];
            const int bl = bitlen_u64((u64)v);
            const i64 rs = (i64)pow2_recip((u64)v, bl, 1, 23);
            if (lane == 0) { rs_s[hh] = rs; bl_s[hh] = bl; }
        }
    } else {
        // ---- phase 3: lane (channel c of 8, key chunk q of 4) of warp w
        const int q = lane & 3, cl = lane >> 2;
        for (int cg = w; cg < (D >> 3); cg += 8) {
            const int c = cg * 8 + cl;
            int lo[G], hi[G];
#pragma unroll
            for (int hh = 0; hh < G; ++hh) { lo[hh] = 0; hi[hh] = 0; }
            for (int b = 0; b < nb; ++b) {
                const int j0 = b * KV_BLK + q * 16;
                if (j0 >= ctx16) break;
                const int4 vw = *(const int4*)(Vs + (size_t)b * KV_BLK * D + c * KV_BLK + q * 16);
#pragma unroll
                for (int hh = 0; hh < G; ++hh) {
                    const uint4 el = *(const uint4*)(Elo + hh * cap + j0);
                    const int4 eh = *(const int4*)(Ehi + hh * cap + j0);
                    lo[hh] = dp4a_us(el.x, vw.x, lo[hh]);
                    lo[hh] = dp4a_us(el.y, vw.y, lo[hh]);
                    lo[hh] = dp4a_us(el.z, vw.z, lo[hh]);
                    lo[hh] = dp4a_us(el.w, vw.w, lo[hh]);
                    hi[hh] = __dp4a(eh.x, vw.x, hi[hh]);
                    hi[hh] = __dp4a(eh.y, vw.y, hi[hh]);
                    hi[hh] = __dp4a(eh.z, vw.z, hi[hh]);
                    hi[hh] = __dp4a(eh.w, vw.w, hi[hh]);
                }
            }
#pragma unroll
            for (int hh = 0; hh < G; ++hh) {
                int l2 = lo[hh], h2 = hi[hh];
                l2 += __shfl_xor_sync(0xffffffffu, l2, 1);
                l2 += __shfl_xor_sync(0xffffffffu, l2, 2);
                h2 += __shfl_xor_sync(0xffffffffu, h2, 1);
                h2 += __shfl_xor_sync(0xffffffffu, h2, 2);
                if (q == 0) { pv[(hh * D + c) * 2] = l2; pv[(hh * D + c) * 2 + 1] = h2; }
            }
        }
    }
    __syncthreads();

    // ---- normalisation and the output row (Q12)
    for (int idx = tid; idx < (G << (EPL == 4 ? 7 : 6)); idx += AD_THREADS) {
        const int hh = idx >> (EPL == 4 ? 7 : 6), c = idx & (D - 1);
        const i64 num = (i64)pv[idx * 2 + 1] * 256 + pv[idx * 2];
        const i64 tq = rshr(num * rs_s[hh], bl_s[hh] + 7);
        const i64 ov = rshr(tq * MV, KVS + 16 - 12);
        a.o[(size_t)t * a.nq * D + ((g << a.lg_grp) + hh) * D + c] = (int32_t)ov;
    }
}

}  // namespace detint
