// Streaming decode GEMV with a fused quantisation prologue (M <= 8 tokens).
//
// One CTA per SM owns a contiguous run of 16-row weight groups. A producer
// warp streams that run through a 4-stage shared-memory ring with 1D bulk
// TMA copies (one per weight row and K-chunk, completion on an mbarrier).
// Weights never depend on the previous kernel, so the first stages are
// issued before griddepcontrol.wait: with programmatic dependent launch the
// next GEMV's weight stream overlaps the tail of the current kernel.
// After the wait, the 8 compute warps quantise the int32 activation rows
// themselves (NormQuant of the residual, or ActQuant of the attention or
// SwiGLU output — the per-token quantisation of the DetLLM blog, section
// "DetLLM") into an int8 tile, then run mma.sync m16n8k32 s8 over the ring
// and apply the requantisation epilogue (one integer multiply and one
// rounding shift per output).
#pragma once
#include "int_device.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace detint {

constexpr int SG_STAGES = 8;           // most ring stages (the launch picks 4 or 8)
constexpr int SG_THREADS = 288;      // 8 compute warps + 1 producer warp

enum { PRO_NONE = 0, PRO_NORMQUANT = 1, PRO_ACTQUANT = 2 };

constexpr int SG_GB = 4;             // row groups whose partial sums are reduced together

struct SgArgs {
    const int8_t* W;          // weights [N][K]
    int N, K, KC, nkc;        // K-chunk width KC (K = nkc * KC, KC <= 1024, KC % 64 == 0)
    int M;                    // tokens, 1..8
    const int32_t* xin;       // int32 activation rows [M][K]
    const int32_t* rows;      // optional row indirection for xin (final norm), or null
    const int16_t* gamma;     // PRO_NORMQUANT
    long long eps;
    int lg_k;                 // log2 K (NormQuant mean)
    int F;                    // PRO_ACTQUANT fixed point
    int pro;                  // PRO_NORMQUANT, PRO_ACTQUANT or PRO_NONE
    const int8_t* x8;         // PRO_NONE: quantised rows [M][K]
    const int32_t* mt_in;     // PRO_NONE: token scales [M]
    const int32_t* kt_in;
    int mode;                 // EPI_QKV, EPI_RESADD, EPI_SWIGLU or EPI_LOGITS
    int rg_q, rg_r;           // CTA c owns rg_q + (c < rg_r) row groups
    int lg_ns;                // log2 of the ring stages used (2 or 3)
    Epi ep;
};

struct SgShared {
    unsigned long long full[SG_STAGES];
    unsigned long long empty[SG_STAGES];
    int mt[8], kt[8];
    long long red64[8][5];     // prologue group reductions (per warp)
};

__device__ __forceinline__ size_t sg_ring_bytes(int KC, int ns) { return (size_t)ns * 16 * (KC + 64); }

// ---- prologue: one group of (8 / Mp) warps per token row quantises it into
// the int8 tile. The row is read once; up to SG_NV 16-byte vectors per thread
// stay in registers for the later passes. The integer square root and the
// two divisions run on different warps of the group where it has more than
// one.
constexpr int SG_NV = 6;

__device__ __forceinline__ int4 sg_vec(const int4 (&v)[SG_NV], const int32_t* xr, int j, int i) {
    // vector j of this thread (element offset i): from registers when held
    int4 r = make_int4(0, 0, 0, 0);
#pragma unroll
    for (int q = 0; q < SG_NV; ++q)
        if (q == j) r = v[q];
    if (j >= SG_NV) r = *(const int4*)(xr + i);
    return r;
}

// token scale (m_t, k_t) of row r, by one warp, from the prologue's partial
// reductions of the row's warp group w0 .. w0 + wpr - 1; only the epilogue
// needs it
__device__ void sg_token_scale(const SgArgs& a, SgShared& sh, int r, int w0, int wpr) {
    u64 axl = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w)
        if (w < wpr) axl = umax64(axl, (u64)sh.red64[(w0 + w) & 7][0]);
    int m = 0, k = 0;
    if (axl != 0) {
        if (a.pro == PRO_NORMQUANT) {
            const int sig = bitlen_u64(axl) - 24;
            i64 ss = 0;
            u64 az = 0;
            const int js = sig <= 0 ? 2 : 3, jz = sig <= 0 ? 1 : 4;
#pragma unroll
            for (int w = 0; w < 8; ++w) {
                if (w < wpr) {
                    ss += sh.red64[(w0 + w) & 7][js];
                    az = umax64(az, (u64)sh.red64[(w0 + w) & 7][jz]);
                }
            }
            if (sig <= 0) {
                ss <<= -2 * sig;
                az <<= -sig;
            }
            i64 eps_s;
            if (sig >= 0) eps_s = (2 * sig >= 62) ? 0 : (a.eps >> (2 * sig));
            else eps_s = a.eps * (1LL << (-2 * sig));
            const u64 rr = isqrt_fast((u64)((ss >> a.lg_k) + eps_s));
            dyadic_fast(az, 127ull * rr, &m, &k);
            k += 12;
        } else {
            dyadic_fast(axl, 127ull, &m, &k);
            k += a.F;
        }
    }
    if ((threadIdx.x & 31) == 0) { sh.mt[r] = m; sh.kt[r] = k; }
}

// sp: the token scales are left to the producer warp (sg_token_scale after
// the prologue), off the path to the dot products
__device__ void sg_prologue(const SgArgs& a, SgShared& sh, int8_t* xs, int XP, const int16_t* gam,
                            bool sp) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int M = a.M, K = a.K;
    const bool norm = a.pro == PRO_NORMQUANT;
    const int lgw = M > 4 ? 0 : (M > 2 ? 1 : (M > 1 ? 2 : 3));   // log2 warps per row
    const int wpr = 1 << lgw;
    const int r = warp >> lgw;              // row of this warp's group
    const int gw = warp & (wpr - 1);        // warp index in its group
    const int gt = gw * 32 + lane;          // thread index in its group
    const int gn = wpr * 32;
    const int bar = 2 + r;
    const int w0 = r << lgw;                // first warp of the group
    int8_t* qr = xs + (size_t)r * XP;
    if (r >= M) {
        for (int i = gt * 16; i < K; i += gn * 16) *(int4*)(qr + i) = make_int4(0, 0, 0, 0);
        return;
    }
    const int src = a.rows ? a.rows[r] : r;
    const int32_t* xr = a.xin + (size_t)src * K;
    const int nvec = K >> 2;                                  // 16-byte vectors in the row
    const int nv = (nvec + gn - 1) >> (5 + lgw);              // per thread (the last may be empty)
    int4 v[SG_NV];
#pragma unroll
    for (int j = 0; j < SG_NV; ++j)
        v[j] = (j < nv && gt + j * gn < nvec) ? *(const int4*)(xr + (gt + j * gn) * 4)
                                              : make_int4(0, 0, 0, 0);
    // pass 1: max |x|; for NormQuant also max |x gamma| and the sum of x^2
    // (modulo 2^64), which are the normalised row's max |x' gamma| and sum of
    // squares up to the exact power-of-two factor whenever the row needs no
    // right shift (every |x| < 2^24: then each x^2 < 2^48 and the sum is exact)
    unsigned ax = 0;                        // |x| <= 2^31
    u64 ag = 0, sq = 0;
    for (int j = 0; j < nv; ++j) {
        if (gt + j * gn >= nvec) break;
        const int i = (gt + j * gn) * 4;
        const int4 w = sg_vec(v, xr, j, i);
        const int xv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) ax = max(ax, (unsigned)absu(xv[q]));
        if (norm) {
            const short4 gm = *(const short4*)(gam + i);
            const int gv[4] = {gm.x, gm.y, gm.z, gm.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                ag = umax64(ag, absu((i64)xv[q] * (i64)gv[q]));
                sq += (u64)((i64)xv[q] * (i64)xv[q]);
            }
        }
    }
    ax = __reduce_max_sync(0xffffffffu, ax);
    if (norm) {
        ag = redux_max_u64(ag);
        sq = redux_sum_u64(sq);
    }
    if (lane == 0) {
        sh.red64[warp][0] = ax;
        sh.red64[warp][1] = (long long)ag;
        sh.red64[warp][2] = (long long)sq;
    }
    bar_named(bar, gn);
    u64 axl = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w)
        if (w < wpr) axl = umax64(axl, (u64)sh.red64[(w0 + w) & 7][0]);
    if (axl == 0) {
        if (sp) bar_arrive_named(14, 288);
        for (int i = gt * 16; i < K; i += gn * 16) *(int4*)(qr + i) = make_int4(0, 0, 0, 0);
        if (gt == 0) { sh.mt[r] = 0; sh.kt[r] = 0; }
        return;
    }
    int sig = 0;
    u64 amax = axl;                         // the maximum the int8 codes are scaled to
    if (norm) {
        sig = bitlen_u64(axl) - 24;
        if (sig <= 0) {
            // x' = x 2^-sig exactly: max |x' gamma| is the pass-1 maximum scaled
            amax = 0;
#pragma unroll
            for (int w = 0; w < 8; ++w)
                if (w < wpr) amax = umax64(amax, (u64)sh.red64[(w0 + w) & 7][1]);
            amax <<= -sig;
        } else {
            // pass 2: sum of squares of the 24-bit row and max |x' gamma|
            i64 ss = 0;
            u64 az = 0;
            for (int j = 0; j < nv; ++j) {
                if (gt + j * gn >= nvec) break;
                const int i = (gt + j * gn) * 4;
                const int4 w = sg_vec(v, xr, j, i);
                const short4 gm = *(const short4*)(gam + i);
                const int xv[4] = {w.x, w.y, w.z, w.w};
                const int gv[4] = {gm.x, gm.y, gm.z, gm.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const i64 xp = norm24(xv[q], sig);
                    ss += xp * xp;
                    az = umax64(az, absu(xp * (i64)gv[q]));
                }
            }
            ss = (i64)redux_sum_u64((u64)ss);
            az = redux_max_u64(az);
            if (lane == 0) { sh.red64[warp][3] = ss; sh.red64[warp][4] = (long long)az; }
            bar_named(bar, gn);
            amax = 0;
#pragma unroll
            for (int w = 0; w < 8; ++w)
                if (w < wpr) amax = umax64(amax, (u64)sh.red64[(w0 + w) & 7][4]);
        }
    }
    // the partial reductions are final: the producer warp may start on the
    // token scale (sp) while this thread quantises; else one warp of the
    // group takes it. The quantisation multiplier in every thread, from the
    // maximum it already holds
    if (sp) bar_arrive_named(14, 288);
    else if (gw == 0) sg_token_scale(a, sh, r, w0, wpr);
    const int e = bitlen_u64(amax);
    const i64 R = (i64)pow2_recip(amax, e, 127, 16);
    const int shq = e + 16;
    // pass 3: quantise
    for (int j = 0; j < nv; ++j) {
        if (gt + j * gn >= nvec) break;
        const int i = (gt + j * gn) * 4;
        const int4 w = sg_vec(v, xr, j, i);
        const int xv[4] = {w.x, w.y, w.z, w.w};
        i64 z[4];
        if (norm) {
            const short4 gm = *(const short4*)(gam + i);
            const int gv[4] = {gm.x, gm.y, gm.z, gm.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) z[q] = norm24(xv[q], sig) * (i64)gv[q];
        } else {
#pragma unroll
            for (int q = 0; q < 4; ++q) z[q] = xv[q];
        }
        char4 c4;
        c4.x = (signed char)rshr(z[0] * R, shq);
        c4.y = (signed char)rshr(z[1] * R, shq);
        c4.z = (signed char)rshr(z[2] * R, shq);
        c4.w = (signed char)rshr(z[3] * R, shq);
        *(char4*)(qr + i) = c4;
    }
}

// PRO_NONE: the rows were quantised by a row kernel; load the int8 tile and
// the token scales
__device__ void sg_load_x8(const SgArgs& a, SgShared& sh, int8_t* xs, int XP) {
    const int tid = threadIdx.x;
    const int kv = a.K >> 4;
    // every load of a pass is issued before its stores, so the L2 round trips
    // overlap instead of following one another
    int mt = 0, kt = 0;
    if (tid < a.M) {
        if (a.mt_in) mt = a.mt_in[tid];
        if (a.kt_in) kt = a.kt_in[tid];
    }
    for (int v = tid; v < kv; v += 256) {
        int4 val[8];
#pragma unroll
        for (int r = 0; r < 8; ++r)
            val[r] = r < a.M ? *(const int4*)(a.x8 + (size_t)r * a.K + v * 16) : make_int4(0, 0, 0, 0);
#pragma unroll
        for (int r = 0; r < 8; ++r) *(int4*)(xs + (size_t)r * XP + v * 16) = val[r];
    }
    if (tid < 8) {
        sh.mt[tid] = mt;
        sh.kt[tid] = kt;
    }
}

// weight-channel scale of output row n: from the CTA's shared-memory copy when
// it was staged (mcs, rows from nbase), else from global memory
__device__ __forceinline__ i64 sg_requant(int acc, const SgShared& sh, const Epi& ep, int tk, int n,
                                          const int32_t* mcs, int nbase) {
    const i64 mc = mcs ? mcs[n - nbase] : ep.mc[n];
    const i64 M = (i64)sh.mt[tk] * mc;
    return rshr((i64)acc * M, sh.kt[tk] + 22 - ep.fout);
}

// epilogue of nb row groups starting at group gb, from the per-warp partial
// tiles red[b][warp][16 rows][8 tokens]
// nw: partial tiles per group to add (8 for the mma path, 1 for dp4a)
__device__ void sg_epilogue(const SgArgs& a, const SgShared& sh, int32_t* red, int gb, int nb,
                            const int32_t* hold, int g0, const int32_t* mcs, int nw) {
    const int nbase = g0 * 16;
    const int tid = threadIdx.x;
    const Epi& ep = a.ep;
    if (a.mode == EPI_SWIGLU) {
        for (int it = tid; it < nb * 64; it += 256) {
            const int b = it >> 6, p = (it >> 3) & 7, tk = it & 7;
            const int32_t* rb = red + b * 1024;
            int sg = 0, su = 0;
            for (int w = 0; w < nw; ++w) {
                sg += rb[w * 128 + (2 * p) * 8 + tk];
                su += rb[w * 128 + (2 * p + 1) * 8 + tk];
            }
            const int n = (gb + b) * 16 + 2 * p;
            if (tk < a.M && n < a.N) {
                i64 yg = sg_requant(sg, sh, ep, tk, n, mcs, nbase), yu = sg_requant(su, sh, ep, tk, n + 1, mcs, nbase);
                if (yg > (1 << 24) || yg < -(1 << 24) || yu > (1 << 24) || yu < -(1 << 24))
                    ep.status[ST_SAT_GU] = 1;
                yg = sat_b(yg, 1 << 24);
                yu = sat_b(yu, 1 << 24);
                ep.out[(size_t)tk * ep.ldo + (n >> 1)] = swiglu_dev((int)yg, (int)yu);
            }
        }
        return;
    }
    for (int it = tid; it < nb * 128; it += 256) {
        const int b = it >> 7, rr = (it >> 3) & 15, tk = it & 7;
        const int32_t* rb = red + b * 1024;
        int sum = 0;
        for (int w = 0; w < nw; ++w) sum += rb[w * 128 + (it & 127)];
        const int n = (gb + b) * 16 + rr;
        int outv = -2147483647;
        if (a.mode == EPI_RAW) {
            if (tk < a.M && n < a.N) ep.out[(size_t)tk * ep.ldo + n] = sum;
            continue;
        }
        if (tk < a.M && n < a.N) {
            const i64 y = sg_requant(sum, sh, ep, tk, n, mcs, nbase);
            if (a.mode == EPI_QKV) {
                if (y > 2147483647LL || y < -2147483647LL) ep.status[ST_SAT_QKV] = 1;
                ep.out[(size_t)tk * ep.ldo + n] = sat32(y);
            } else if (a.mode == EPI_RESADD) {
                int32_t* hp = ep.out + (size_t)tk * ep.ldo + n;
                const int li = ((gb + b - g0) * 16 + rr) * 8 + tk;      // preloaded slot
                const i64 hv = hold ? hold[li] : *hp;
                const i64 s2 = hv + (i64)sat32(y);
                if (s2 > 2147483647LL || s2 < -2147483647LL) ep.status[ST_SAT_RES] = 1;
                *hp = sat32(s2);
            } else {
                if (y > 2147483647LL || y < -2147483647LL) ep.status[ST_SAT_LOGIT] = 1;
                outv = sat32(y);
                ep.out[(size_t)tk * ep.ldo + n] = outv;
            }
        }
        if (a.mode == EPI_LOGITS) red[b * 1024 + (it & 127)] = outv;   // warp 0's slot, summed already
    }
    if (a.mode == EPI_LOGITS) {
        bar_named(1, 256);
        // per (group, token): the largest logit of the 16 rows, lowest row on ties
        for (int it = tid; it < nb * 8; it += 256) {
            const int b = it >> 3, tk = it & 7;
            if (tk >= a.M) continue;
            const int n0 = (gb + b) * 16;
            const int32_t* lg = red + b * 1024;
            int bv = lg[tk], bi = n0;
            for (int q = 1; q < 16; ++q) {
                const int v = lg[q * 8 + tk];
                if (v > bv && n0 + q < a.N) { bv = v; bi = n0 + q; }
            }
            ep.pval[(size_t)tk * ep.npart + gb + b] = bv;
            ep.pidx[(size_t)tk * ep.npart + gb + b] = bi;
        }
    }
}

// producer warp: the weight rows of each (row group, K-chunk) unit of row
// groups [g0, g1) into the ring; u counts ring units across calls (stage
// u mod NS, phase parity from u / NS), SB is the ring's stage stride
__device__ __forceinline__ void sg_produce(const SgArgs& a, SgShared& sh, unsigned char* ring, int P,
                                           size_t SB, int NS, int lg_ns, int g0, int g1, int& u,
                                           uint64_t pol) {
    const int lane = threadIdx.x & 31;
    for (int g = g0; g < g1; ++g) {
        for (int kc = 0; kc < a.nkc; ++kc, ++u) {
            const int s = u & (NS - 1);
            if (u >= NS && lane == 0) {
                // bounded: on a timeout the status word records it and the
                // stream continues (results are then invalid, nothing hangs)
                if (!mbar_wait(smem_u32(&sh.empty[s]), ((u >> lg_ns) - 1) & 1))
                    a.ep.status[ST_TIMEOUT] = 1;
            }
            __syncwarp();
            const uint32_t fb = smem_u32(&sh.full[s]);
            if (a.nkc == 1) {
                // the group's rows are contiguous: one copy (the last group
                // may hold fewer than 16 rows; its missing rows are never stored)
                const int rows = min(16, a.N - g * 16);
                const uint32_t bytes = (uint32_t)rows * (uint32_t)a.K;
                if (lane == 0) {
                    mbar_arrive_expect_tx(fb, bytes);
                    bulk_g2s_hint(smem_u32(ring + (size_t)s * SB), a.W + (size_t)g * 16 * a.K, bytes, fb, pol);
                }
            } else {
                if (lane == 0) mbar_arrive_expect_tx(fb, 16u * a.KC);
                __syncwarp();
                if (lane < 16) {
                    const int row = min(g * 16 + lane, a.N - 1);
                    bulk_g2s_hint(smem_u32(ring + (size_t)s * SB + (size_t)lane * P),
                                  a.W + (size_t)row * a.K + (size_t)kc * a.KC, a.KC, fb, pol);
                }
            }
        }
    }
}

// compute warps: dot products of the quantised tile with the ring's weight
// units of row groups [g0, g1), then the epilogue per SG_GB groups; hold:
// preloaded residual values (or null), mcs: staged channel scales (or null)
__device__ __forceinline__ void sg_consume(const SgArgs& a, SgShared& sh, const unsigned char* ring,
                                           int P, size_t SB, int NS, int lg_ns, const int8_t* xs,
                                           int XP, int32_t* red, int g0, int g1, int& u,
                                           const int32_t* hold, const int32_t* mcs,
                                           bool wait_scale) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, tq = lane & 3;
    const int nch = a.KC >> 6;
    // up to 4 tokens: dp4a on the integer pipe (one multiply per weight per
    // token); more: mma.sync m16n8k32 over 8 token columns. On sm_103a both
    // run at the same int8 rate, so the m16n8 tile's unused columns would
    // cost up to 8x the integer work at one token.
    const bool dp = a.M <= 4;
    for (int gb = g0; gb < g1; gb += SG_GB) {
        const int nb = min(SG_GB, g1 - gb);
        if (dp) {
            // a half-warp per weight row: thread t of the half reads 16-byte
            // chunks t, t+16, ... of the row's K-chunk and the same chunks of
            // each token's activations; a 4-step shuffle sums the half. Each
            // 32-bit word lane of a chunk has its own accumulator and the
            // chunk loads are issued before any multiply, so the dp4a
            // latencies overlap instead of forming one dependent chain.
            const int r = tid >> 4, hl = tid & 15;
            const int nc = a.KC >> 4;                 // 16-byte chunks per row chunk
            for (int b = 0; b < nb; ++b) {
                int acc[4][4];
#pragma unroll
                for (int tk = 0; tk < 4; ++tk) acc[tk][0] = acc[tk][1] = acc[tk][2] = acc[tk][3] = 0;
                for (int kc = 0; kc < a.nkc; ++kc, ++u) {
                    const int s = u & (NS - 1);
                    if (!mbar_wait(smem_u32(&sh.full[s]), (u >> lg_ns) & 1)) a.ep.status[ST_TIMEOUT] = 1;
                    const unsigned char* wr = ring + (size_t)s * SB + (size_t)r * P;
                    const int8_t* xk = xs + (size_t)kc * a.KC;
                    for (int c0 = hl; c0 < nc; c0 += 64) {
                        int4 w[4];
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            w[j] = (c0 + 16 * j < nc) ? *(const int4*)(wr + (c0 + 16 * j) * 16) : make_int4(0, 0, 0, 0);
#pragma unroll
                        for (int tk = 0; tk < 4; ++tk) {
                            if (tk < a.M) {
                                int4 xv[4];
#pragma unroll
                                for (int j = 0; j < 4; ++j)
                                    xv[j] = (c0 + 16 * j < nc)
                                                ? *(const int4*)(xk + (size_t)tk * XP + (c0 + 16 * j) * 16)
                                                : make_int4(0, 0, 0, 0);
#pragma unroll
                                for (int j = 0; j < 4; ++j) {
                                    acc[tk][0] = __dp4a(w[j].x, xv[j].x, acc[tk][0]);
                                    acc[tk][1] = __dp4a(w[j].y, xv[j].y, acc[tk][1]);
                                    acc[tk][2] = __dp4a(w[j].z, xv[j].z, acc[tk][2]);
                                    acc[tk][3] = __dp4a(w[j].w, xv[j].w, acc[tk][3]);
                                }
                            }
                        }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&sh.empty[s]));
                }
                int tot[4];
#pragma unroll
                for (int tk = 0; tk < 4; ++tk) {
                    int v = (acc[tk][0] + acc[tk][1]) + (acc[tk][2] + acc[tk][3]);
                    if (tk < a.M) {
                        v += __shfl_xor_sync(0xffffffffu, v, 8);
                        v += __shfl_xor_sync(0xffffffffu, v, 4);
                        v += __shfl_xor_sync(0xffffffffu, v, 2);
                        v += __shfl_xor_sync(0xffffffffu, v, 1);
                    }
                    tot[tk] = v;
                }
                if (hl < 8) {
                    int v = 0;
#pragma unroll
                    for (int tk = 0; tk < 4; ++tk)
                        if (hl == tk && tk < a.M) v = tot[tk];
                    red[b * 1024 + r * 8 + hl] = v;
                }
            }
            if (wait_scale && gb == g0) bar_named(15, 288);    // token scales from the producer
            bar_named(1, 256);
            sg_epilogue(a, sh, red, gb, nb, hold, g0, mcs, 1);
            bar_named(1, 256);
            continue;
        }
        for (int b = 0; b < nb; ++b) {
            int acc[4] = {0, 0, 0, 0}, acc2[4] = {0, 0, 0, 0};
            for (int kc = 0; kc < a.nkc; ++kc, ++u) {
                const int s = u & (NS - 1);
                if (!mbar_wait(smem_u32(&sh.full[s]), (u >> lg_ns) & 1)) a.ep.status[ST_TIMEOUT] = 1;
                const int8_t* st = (const int8_t*)ring + (size_t)s * SB;
                const int8_t* wlo = st + g * P + 16 * tq;
                const int8_t* whi = wlo + 8 * P;
                const int8_t* xb = xs + g * XP + kc * a.KC + 16 * tq;
                for (int ch = warp; ch < nch; ch += 8) {
                    const int4 al = *(const int4*)(wlo + ch * 64);
                    const int4 ah = *(const int4*)(whi + ch * 64);
                    const int4 bx = *(const int4*)(xb + ch * 64);
                    mma_s8(acc, al.x, ah.x, al.y, ah.y, bx.x, bx.y);
                    mma_s8(acc2, al.z, ah.z, al.w, ah.w, bx.z, bx.w);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&sh.empty[s]));
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[q] += acc2[q];
            // accumulator fragment: c0 (row g, tok 2tq), c1, c2 (row g+8), c3
            int32_t* rw = red + b * 1024 + warp * 128;
            rw[g * 8 + 2 * tq] = acc[0];
            rw[g * 8 + 2 * tq + 1] = acc[1];
            rw[(g + 8) * 8 + 2 * tq] = acc[2];
            rw[(g + 8) * 8 + 2 * tq + 1] = acc[3];
        }
        if (wait_scale && gb == g0) bar_named(15, 288);
        bar_named(1, 256);
        sg_epilogue(a, sh, red, gb, nb, hold, g0, mcs, 8);
        bar_named(1, 256);
    }
}

// MINB = 2: the long-stream variant (two CTAs per SM, registers capped to fit)
template <int MINB>
__global__ void __launch_bounds__(SG_THREADS, MINB) k_sgemv(SgArgs a) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ SgShared sh;
    const int tid = threadIdx.x, warp = tid >> 5;
    // ring row pitch: a whole 16-row group arrives in one bulk copy when the
    // rows are not chunked (pitch K); chunked rows get a 64-byte pad so
    // fragment loads of neighbouring rows fall in different banks
    const int P = a.nkc == 1 ? a.K : a.KC + 64;
    const int XP = a.K + 64;                      // activation row pitch
    unsigned char* ring = smem;
    const int NS = 1 << a.lg_ns;
    int8_t* xs = (int8_t*)(smem + sg_ring_bytes(a.KC, NS));
    int32_t* red = (int32_t*)(xs + (size_t)8 * XP);     // [SG_GB][8 warps][16][8]
    const int c = blockIdx.x;
    const int g0 = c * a.rg_q + min(c, a.rg_r);
    const int g1 = g0 + a.rg_q + (c < a.rg_r ? 1 : 0);
    const int units = (g1 - g0) * a.nkc;

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(smem_u32(&sh.full[s]), 1);
            mbar_init(smem_u32(&sh.empty[s]), 8);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    pdl_launch();

    // with at most two token rows and the CTA's whole weight run fitting the
    // ring, the producer warp is idle once its copies are issued: it then
    // computes the token scales while the compute warps quantise and multiply
    const bool sp = a.pro != PRO_NONE && a.M <= 2 && units <= NS && g1 > g0;
    if (warp == 8) {
        const uint64_t pol = l2_evict_first();
        int u = 0;
        sg_produce(a, sh, ring, P, (size_t)16 * P, NS, a.lg_ns, g0, g1, u, pol);
        if (sp) {
            bar_named(14, 288);                     // the prologue's partial reductions are final
            const int lgw = a.M > 1 ? 2 : 3;        // the prologue's warps per row
            for (int r = 0; r < a.M; ++r) sg_token_scale(a, sh, r, r << lgw, 1 << lgw);
            __syncwarp();
            bar_arrive_named(15, 288);
        }
        return;
    }

    // compute warps: copy the (immutable) RMSNorm gamma and this CTA's weight
    // channel scales before the wait
    int16_t* gam = (int16_t*)(red + SG_GB * 1024);
    if (a.pro == PRO_NORMQUANT)
        for (int i = tid * 8; i < a.K; i += 256 * 8) *(int4*)(gam + i) = *(const int4*)(a.gamma + i);
    int32_t* hold = (int32_t*)(gam + a.K);
    int32_t* mcs = hold + 256;
    const bool mc_pre = a.ep.mc && (g1 - g0) * 16 <= 256;
    if (mc_pre && tid < (g1 - g0) * 16) mcs[tid] = a.ep.mc[min(g0 * 16 + tid, a.N - 1)];
    // the prologue's first pass reads gamma elements that other warps copied
    bar_named(1, 256);
    pdl_wait();
    // residual add: issue the loads of this CTA's old residual values now so
    // they overlap the quantisation prologue
    const bool pre = a.mode == EPI_RESADD && (g1 - g0) * 128 <= 256;
    int hv = 0;
    if (pre && tid < (g1 - g0) * 128) {
        const int tk = tid & 7, n = g0 * 16 + (tid >> 3);
        if (tk < a.M && n < a.N) hv = a.ep.out[(size_t)tk * a.ep.ldo + n];
    }
    if (a.pro == PRO_NONE) sg_load_x8(a, sh, xs, XP);
    else sg_prologue(a, sh, xs, XP, gam, sp);
    if (pre && tid < (g1 - g0) * 128) hold[tid] = hv;
    bar_named(1, 256);

    int u = 0;
    sg_consume(a, sh, ring, P, (size_t)16 * P, NS, a.lg_ns, xs, XP, red, g0, g1, u,
               pre ? hold : nullptr, mc_pre ? mcs : nullptr, sp);
    // every issued copy has completed before the CTA exits (bounded wait;
    // normally these phases completed long ago)
    if (tid == 0) {
        for (int s = 0; s < NS && s < units; ++s) {
            const int ul = s + ((units - 1 - s) >> a.lg_ns) * NS;    // last unit on stage s
            if (!mbar_wait(smem_u32(&sh.full[s]), (ul >> a.lg_ns) & 1)) a.ep.status[ST_TIMEOUT] = 1;
        }
    }
}

}  // namespace detint
