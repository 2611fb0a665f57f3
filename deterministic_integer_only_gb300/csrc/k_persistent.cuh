// One decode step in one launch (B <= 8 sequences).
//
// A cooperative grid of one CTA per SM runs every phase of the step in
// order: embedding, then per layer QKV GEMV, attention, o_proj GEMV (+
// residual), gate/up GEMV (+ SwiGLU), down GEMV (+ residual), then the
// lm_head GEMV with argmax partials and the final argmax. Each phase waits on
// a grid barrier for the previous phase's outputs (the per-token
// quantisation needs a whole row, the attention all of q/k/v), exactly the
// dependencies of the multi-kernel step, so the arithmetic and every result
// are the same. What changes is the cost around the arithmetic:
//  * the producer warp of each CTA streams the weight slices of ALL of the
//    step's GEMV phases through one shared-memory ring without ever waiting
//    on a barrier, so a phase's weights are in shared memory while the
//    compute warps still wait for its inputs;
//  * one code image serves every layer, so the instruction cache stays warm
//    after the first layer, and no CTA is launched or scheduled per phase.
// Grid barriers use one arrival counter in global memory (release adds,
// acquire polls at GPU scope, bounded polling that records a timeout in the
// status word instead of hanging). Only the 256 compute
// threads take part in barriers; the producer warp never does.
#pragma once
#include "kernels.h"
#include "ptx.cuh"
#include "int_device.cuh"

namespace detint {

constexpr int PD_SPIN = 1 << 20;        // bounded polls of a grid barrier
constexpr int PD_PMAX = 1024 + 64;      // largest ring row pitch (K chunks of 1024 + pad)
constexpr size_t PD_SB = (size_t)16 * PD_PMAX;   // ring stage stride

__device__ __forceinline__ unsigned pd_ld_acquire(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void pd_red_release(unsigned* p, unsigned v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Grid barrier of the compute threads (256 per CTA) in two halves, so that a
// CTA can issue its next phase's independent loads between them. bar[0]
// counts arrivals over the whole step (the host zeroes it before each
// launch); barrier k of the step is complete when it reaches (k + 1) CTAs x
// grid. Arrival is one release add per CTA; the wait polls with acquire
// loads (bounded: once any wait has timed out, later barriers stop waiting,
// so a broken step ends quickly with the flag set).
__device__ __forceinline__ void pd_arrive(unsigned* bar) {
    bar_named(1, 256);
    if (threadIdx.x == 0) pd_red_release(bar, 1u);
}
__device__ __forceinline__ void pd_wait(unsigned* bar, unsigned target, int32_t* status) {
    if (threadIdx.x == 0 && *(volatile int32_t*)&status[ST_TIMEOUT] == 0) {
        int i = 0;
        while (pd_ld_acquire(bar) < target) {
            if (++i > PD_SPIN) { status[ST_TIMEOUT] = 1; break; }
        }
    }
    bar_named(1, 256);
}

enum { PD_QKV = 0, PD_O = 1, PD_GU = 2, PD_D = 3, PD_LOGITS = 4 };

// the streaming-GEMV arguments of phase ph (layer l)
__device__ __forceinline__ SgArgs pd_sgargs(const PdArgs& a, int ph, const PdLayer& L) {
    SgArgs s{};
    const int nqkv = (a.nq + 2 * a.nkv) * a.d;
    s.M = a.T;
    s.ep.status = a.status;
    s.rows = nullptr;
    s.eps = a.eps_h;
    s.lg_k = a.lg_H;
    switch (ph) {
        case PD_QKV:
            s.W = L.w_qkv; s.N = nqkv; s.K = a.H; s.xin = a.h; s.gamma = L.attn_gamma;
            s.pro = PRO_NORMQUANT; s.mode = EPI_QKV;
            s.ep.out = a.qkv; s.ep.ldo = nqkv; s.ep.mc = L.m_qkv; s.ep.fout = 12;
            break;
        case PD_O:
            s.W = L.w_o; s.N = a.H; s.K = a.nq * a.d; s.xin = a.o; s.F = 12;
            s.pro = PRO_ACTQUANT; s.mode = EPI_RESADD;
            s.ep.out = a.h; s.ep.ldo = a.H; s.ep.mc = L.m_o; s.ep.fout = 16;
            break;
        case PD_GU:
            s.W = L.w_gu; s.N = 2 * a.F; s.K = a.H; s.xin = a.h; s.gamma = L.ffn_gamma;
            s.pro = PRO_NORMQUANT; s.mode = EPI_SWIGLU;
            s.ep.out = a.sbuf; s.ep.ldo = a.F; s.ep.mc = L.m_gu; s.ep.fout = 12;
            break;
        case PD_D:
            s.W = L.w_d; s.N = a.H; s.K = a.F; s.xin = a.sbuf; s.F = 10;
            s.pro = PRO_ACTQUANT; s.mode = EPI_RESADD;
            s.ep.out = a.h; s.ep.ldo = a.H; s.ep.mc = L.m_d; s.ep.fout = 16;
            break;
        default:
            s.W = a.embed; s.N = a.V; s.K = a.H; s.xin = a.h; s.gamma = a.final_gamma;
            s.pro = PRO_NORMQUANT; s.mode = EPI_LOGITS;
            s.ep.out = a.logits; s.ep.ldo = a.V; s.ep.mc = a.embed_m; s.ep.fout = 16;
            s.ep.pval = a.pval; s.ep.pidx = a.pidx; s.ep.npart = a.npart;
            break;
    }
    s.KC = s.K <= 1024 ? s.K : 1024;
    s.nkc = s.K <= 1024 ? 1 : (s.K >> 10);
    s.rg_q = a.rg[ph][0];
    s.rg_r = a.rg[ph][1];
    s.lg_ns = a.lg_ns;
    return s;
}

__device__ __forceinline__ void pd_groups(const SgArgs& s, int c, int* g0, int* g1) {
    *g0 = c * s.rg_q + min(c, s.rg_r);
    *g1 = *g0 + s.rg_q + (c < s.rg_r ? 1 : 0);
}

// one GEMV phase on the compute warps: arrive at the barrier that ends the
// previous phase, stage the immutable gamma and channel scales while it
// completes, then quantise, dot products and epilogue
__device__ void pd_gemv(const PdArgs& a, const SgArgs& s, SgShared& sh, unsigned char* smem, int c,
                        int& u, unsigned& nbar) {
    const int tid = threadIdx.x;
    int g0, g1;
    pd_groups(s, c, &g0, &g1);
    int8_t* xs = (int8_t*)(smem + a.off_xs);
    int32_t* red = (int32_t*)(smem + a.off_red);
    int16_t* gam = (int16_t*)(smem + a.off_gam);
    int32_t* hold = (int32_t*)(smem + a.off_hold);
    int32_t* mcs = hold + 256;
    const int XP = s.K + 64;
    const int P = s.nkc == 1 ? s.K : s.KC + 64;
    pd_arrive(a.bar);
    if (s.pro == PRO_NORMQUANT)
        for (int i = tid * 8; i < s.K; i += 256 * 8) *(int4*)(gam + i) = *(const int4*)(s.gamma + i);
    const bool mc_pre = (g1 - g0) * 16 <= 256;
    if (mc_pre && tid < (g1 - g0) * 16) mcs[tid] = s.ep.mc[min(g0 * 16 + tid, s.N - 1)];
    pd_wait(a.bar, ++nbar * gridDim.x, a.status);
    const bool pre = s.mode == EPI_RESADD && (g1 - g0) * 128 <= 256;
    int hv = 0;
    if (pre && tid < (g1 - g0) * 128) {
        const int tk = tid & 7, n = g0 * 16 + (tid >> 3);
        if (tk < s.M && n < s.N) hv = s.ep.out[(size_t)tk * s.ep.ldo + n];
    }
    sg_prologue(s, sh, xs, XP, gam, false);
    if (pre && tid < (g1 - g0) * 128) hold[tid] = hv;
    bar_named(1, 256);
    sg_consume(s, sh, smem, P, PD_SB, 1 << a.lg_ns, a.lg_ns, xs, XP, red, g0, g1, u,
               pre ? hold : nullptr, mc_pre ? mcs : nullptr, false);
}

// attention of token t's q heads of kv group g (compute warps of one CTA):
// QK-post of the G q heads and the K/V head (one warp each), then scores,
// maximum, 15-bit weights and the two P·V limbs with the K/V cache read from
// global memory, the same arithmetic as attention_core
template <int EPL, int G>
__device__ void pd_attention(const PdArgs& a, const PdLayer& L, int t, int g, unsigned char* scr) {
    constexpr int D = EPL * 32, NC = D >> 4;
    __shared__ int32_t mqs[G], kqs[G];
    __shared__ int red_i[8][G];
    __shared__ i64 red_l[8][G], umax_s[G], rs_s[G];
    __shared__ int bl_s[G];
    const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31, dh2 = D >> 1;
    const int cap = a.attn_cap;
    int8_t* qs = (int8_t*)scr;                          // [G][D]
    int32_t* S = (int32_t*)(scr + G * D);               // [G][cap]
    unsigned char* Elo = (unsigned char*)(S + (size_t)G * cap);
    unsigned char* Ehi = Elo + (size_t)G * cap;
    int32_t* pv = (int32_t*)(Ehi + (size_t)G * cap);    // [G][D][2]
    QkvPostArgs qa{};
    qa.qkv = a.qkv; qa.q_gamma = L.q_gamma; qa.k_gamma = L.k_gamma; qa.qk_norm = a.qk_norm;
    qa.eps_qk = a.eps_qk; qa.rope_cos = a.rope_cos; qa.rope_sin = a.rope_sin; qa.kvp = L.kvp;
    qa.tok_seq = a.tok_seq; qa.tok_pos = a.tok_pos; qa.block_table = a.block_table; qa.mbs = a.mbs;
    qa.kc = L.kc; qa.vc = L.vc; qa.T = a.T; qa.nq = a.nq; qa.nkv = a.nkv; qa.d = D; qa.lg_grp = a.lg_grp;
    const int pos = a.tok_pos[t];
    const int32_t* kvp = L.kvp + (size_t)g * (8 + dh2);
    const int16_t* cr = a.rope_cos + (size_t)pos * dh2;
    const int16_t* sr = a.rope_sin + (size_t)pos * dh2;
    if (w < G)
        qkv_head_p<EPL>(qa, t, (g << a.lg_grp) + w, qs + w * D, &mqs[w], &kqs[w], cr, sr, kvp, L.q_gamma,
                        L.k_gamma);
    else if (w == G)
        qkv_head_p<EPL>(qa, t, a.nq + g, nullptr, nullptr, nullptr, cr, sr, kvp, L.q_gamma, L.k_gamma);
    bar_named(1, 256);

    const i64 CSTM = kvp[6], MV = kvp[4];
    const int CSTK = kvp[7], KVS = kvp[5];
    const int ctx = pos + 1, ctx16 = (ctx + 15) & ~15;
    const int* bt = a.block_table + (size_t)a.tok_seq[t] * a.mbs;
    // ---- scores and per-head maxima
    {
        int smax[G];
#pragma unroll
        for (int hh = 0; hh < G; ++hh) smax[hh] = -2147483647;
        for (int j = tid; j < ctx; j += 256) {
            const int8_t* kr = L.kc + (((size_t)bt[j >> 6] * a.nkv + g) * KV_BLK + (j & 63)) * D;
            int acc[G];
#pragma unroll
            for (int hh = 0; hh < G; ++hh) acc[hh] = 0;
#pragma unroll
            for (int v = 0; v < NC; ++v) {
                const int4 kw = *(const int4*)(kr + v * 16);
#pragma unroll
                for (int hh = 0; hh < G; ++hh) {
                    const int4 qw = *(const int4*)(qs + hh * D + v * 16);
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
            int v = smax[hh];
#pragma unroll
            for (int o = 16; o; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
            if (lane == 0) red_i[w][hh] = v;
        }
    }
    bar_named(1, 256);
    if (tid < G) {
        int v = red_i[0][tid];
        for (int w2 = 1; w2 < 8; ++w2) v = max(v, red_i[w2][tid]);
        umax_s[tid] = rshr((i64)v * (i64)mqs[tid] * CSTM, kqs[tid] + CSTK - 10);
    }
    bar_named(1, 256);
    // ---- 15-bit weights as two byte planes, and the row sums
    {
        i64 sum[G];
#pragma unroll
        for (int hh = 0; hh < G; ++hh) sum[hh] = 0;
        for (int j = tid; j < ctx16; j += 256) {
#pragma unroll
            for (int hh = 0; hh < G; ++hh) {
                int E = 0;
                if (j < ctx) {
                    const i64 uu = rshr((i64)S[hh * cap + j] * (i64)mqs[hh] * CSTM, kqs[hh] + CSTK - 10);
                    E = min(32767, exp2q_dev(uu - umax_s[hh]));
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
    bar_named(1, 256);
    if (w < G) {
        i64 v = 0;
        for (int w2 = 0; w2 < 8; ++w2) v += red_l[w2][w];
        const int bl = bitlen_u64((u64)v);
        const i64 rs = (i64)pow2_recip((u64)v, bl, 1, 23);
        if (lane == 0) { rs_s[w] = rs; bl_s[w] = bl; }
    }
    // ---- P·V: lane (channel c of 8, key chunk q of 4) of warp w
    {
        const int q = lane & 3, cl = lane >> 2;
        for (int cg = w; cg < (D >> 3); cg += 8) {
            const int c = cg * 8 + cl;
            int lo[G], hi[G];
#pragma unroll
            for (int hh = 0; hh < G; ++hh) { lo[hh] = 0; hi[hh] = 0; }
            for (int j0 = q * 16; j0 < ctx16; j0 += 64) {
                const int4 vw = *(const int4*)(L.vc + (((size_t)bt[j0 >> 6] * a.nkv + g) * D + c) * KV_BLK +
                                               (j0 & 63));
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
    bar_named(1, 256);
    for (int idx = tid; idx < G * D; idx += 256) {
        const int hh = idx >> (EPL == 4 ? 7 : 6), c = idx & (D - 1);
        const i64 num = (i64)pv[idx * 2 + 1] * 256 + pv[idx * 2];
        const i64 tq = rshr(num * rs_s[hh], bl_s[hh] + 7);
        const i64 ov = rshr(tq * MV, KVS + 16 - 12);
        a.o[(size_t)t * a.nq * D + ((g << a.lg_grp) + hh) * D + c] = (int32_t)ov;
    }
    bar_named(1, 256);
}

template <int EPL, int G>
__global__ void __launch_bounds__(SG_THREADS, 1) k_decode_persistent(PdArgs a) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ SgShared sh;
    __shared__ int sv[8], si[8];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = blockIdx.x, nblk = gridDim.x;
    const int NS = 1 << a.lg_ns;
    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(smem_u32(&sh.full[s]), 1);
            mbar_init(smem_u32(&sh.empty[s]), 8);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    if (warp == 8) {
        // the weight slices of every GEMV phase of the step, in phase order
        const uint64_t pol = l2_evict_first();
        int u = 0;
        for (int l = 0; l <= a.L; ++l) {
            const int nph = l < a.L ? 4 : 1;
            for (int p = 0; p < nph; ++p) {
                const int ph = l < a.L ? p : PD_LOGITS;
                const SgArgs s = pd_sgargs(a, ph, a.layers[l < a.L ? l : 0]);
                int g0, g1;
                pd_groups(s, c, &g0, &g1);
                const int P = s.nkc == 1 ? s.K : s.KC + 64;
                sg_produce(s, sh, smem, P, PD_SB, NS, a.lg_ns, g0, g1, u, pol);
            }
        }
        return;
    }

    int u = 0;
    unsigned nbar = 0;          // barriers passed in this step
    // ---- embedding (every CTA a slice of the T x H residual rows)
    if (c == 0 && tid < a.T) {
        int p = a.seq_len[a.tok_seq[tid]];
        if (p >= a.max_pos) { a.status[ST_CTX] = 1; p = a.max_pos - 1; }
        a.tok_pos[tid] = p;
    }
    for (int e = c * 256 + tid; e < a.T * a.H; e += nblk * 256) {
        const int t = e >> a.lg_H, i = e & (a.H - 1);
        int id = a.tokens[t];
        if (id < 0 || id >= a.V) {
            if (i == 0) a.status[ST_TOKEN] = 1;
            id = 0;
        }
        a.h[e] = (int32_t)rshr((i64)a.embed[(size_t)id * a.H + i] * (i64)a.embed_m[id], 6);
    }
    unsigned char* scr = smem + a.off_xs;      // attention scratch aliases the GEMV tile
    for (int l = 0; l < a.L; ++l) {
        const PdLayer& L = a.layers[l];
        // this layer's cached K/V blocks of the CTA's attention items into L2
        // (all positions before this step's are already written)
        for (int it = c; it < a.T * a.nkv; it += nblk) {
            int t = 0, g = it;
            while (g >= a.nkv) { g -= a.nkv; ++t; }
            const int seq = a.tok_seq[t];
            const int nb = (a.seq_len[seq] + KV_BLK) >> 6;
            const size_t blk_bytes = (size_t)KV_BLK * a.d;
            for (int b = tid; b < nb; b += 256) {
                const size_t off = ((size_t)a.block_table[(size_t)seq * a.mbs + b] * a.nkv + g) * blk_bytes;
                prefetch_l2(L.kc + off, (uint32_t)blk_bytes);
                prefetch_l2(L.vc + off, (uint32_t)blk_bytes);
            }
        }
        pd_gemv(a, pd_sgargs(a, PD_QKV, L), sh, smem, c, u, nbar);
        pd_arrive(a.bar);
        pd_wait(a.bar, ++nbar * nblk, a.status);
        {
            // work items (token, kv head): CTA c takes items c, c + nblk, ...
            const int items = a.T * a.nkv;
            for (int it = c; it < items; it += nblk) {
                int t = 0, g = it;
                while (g >= a.nkv) { g -= a.nkv; ++t; }
                pd_attention<EPL, G>(a, L, t, g, scr);
            }
        }
        pd_gemv(a, pd_sgargs(a, PD_O, L), sh, smem, c, u, nbar);
        pd_gemv(a, pd_sgargs(a, PD_GU, L), sh, smem, c, u, nbar);
        pd_gemv(a, pd_sgargs(a, PD_D, L), sh, smem, c, u, nbar);
    }
    pd_gemv(a, pd_sgargs(a, PD_LOGITS, a.layers[0]), sh, smem, c, u, nbar);
    pd_arrive(a.bar);
    pd_wait(a.bar, ++nbar * nblk, a.status);
    // ---- final argmax of each row (lowest id on ties), CTA t for row t
    if (c < a.T) {
        const int r = c;
        int bv = -2147483647 - 1, bi = 2147483647;
        for (int i = tid; i < a.npart; i += 256) {
            const int v = a.pval[(size_t)r * a.npart + i], ix = a.pidx[(size_t)r * a.npart + i];
            if (v > bv || (v == bv && ix < bi)) { bv = v; bi = ix; }
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            const int v = __shfl_xor_sync(0xffffffffu, bv, o);
            const int ix = __shfl_xor_sync(0xffffffffu, bi, o);
            if (v > bv || (v == bv && ix < bi)) { bv = v; bi = ix; }
        }
        if (lane == 0) { sv[warp] = bv; si[warp] = bi; }
        bar_named(1, 256);
        if (tid == 0) {
            bv = sv[0]; bi = si[0];
            for (int w2 = 1; w2 < 8; ++w2)
                if (sv[w2] > bv || (sv[w2] == bv && si[w2] < bi)) { bv = sv[w2]; bi = si[w2]; }
            a.next_tok[r] = bi;
            a.seq_len[a.tok_seq[r]] += 1;
        }
    }
}

}  // namespace detint
