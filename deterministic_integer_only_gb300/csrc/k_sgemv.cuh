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

constexpr int SG_STAGES = 4;
constexpr int SG_THREADS = 288;      // 8 compute warps + 1 producer warp

enum { PRO_NORMQUANT = 1, PRO_ACTQUANT = 2 };

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
    int pro;
    int rg_q, rg_r;           // CTA c owns rg_q + (c < rg_r) row groups
    Epi ep;
};

struct SgShared {
    unsigned long long full[SG_STAGES];
    unsigned long long empty[SG_STAGES];
    int mt[8], kt[8];
    long long red64[8][2];     // prologue group reductions (per warp)
    long long bc[8][4];        // per-row broadcast of R, shift, sigma, flag
};

__device__ __forceinline__ size_t sg_ring_bytes(int KC) { return (size_t)SG_STAGES * 16 * (KC + 64); }

// ---- prologue: one group of (8 / Mp) warps per token row
template <int PRO>
__device__ void sg_prologue(const SgArgs& a, SgShared& sh, int8_t* xs, int XP) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int M = a.M, K = a.K;
    const int lgw = M > 4 ? 0 : (M > 2 ? 1 : (M > 1 ? 2 : 3));   // log2 warps per row
    const int wpr = 1 << lgw;
    const int r = warp >> lgw;              // row of this warp's group
    const int gw = warp & (wpr - 1);        // warp index in its group
    const int gt = gw * 32 + lane;          // thread index in its group
    const int gn = wpr * 32;
    const int bar = 2 + r;
    int8_t* qr = xs + (size_t)r * XP;
    if (r >= M) {
        for (int i = gt * 16; i < K; i += gn * 16) *(int4*)(qr + i) = make_int4(0, 0, 0, 0);
        return;
    }
    const int src = a.rows ? a.rows[r] : r;
    const int32_t* xr = a.xin + (size_t)src * K;
    // pass 1: max |x|
    u64 ax = 0;
    for (int i = gt * 4; i < K; i += gn * 4) {
        const int4 v = *(const int4*)(xr + i);
        ax = umax64(ax, umax64(umax64(absu(v.x), absu(v.y)), umax64(absu(v.z), absu(v.w))));
    }
    ax = warp_max_u64(ax);
    if (lane == 0) sh.red64[warp][0] = (long long)ax;
    bar_named(bar, gn);
    ax = 0;
    for (int w = 0; w < wpr; ++w) ax = umax64(ax, (u64)sh.red64[(r << lgw) + w][0]);
    bar_named(bar, gn);
    if (ax == 0) {
        for (int i = gt * 16; i < K; i += gn * 16) *(int4*)(qr + i) = make_int4(0, 0, 0, 0);
        if (gt == 0) { sh.mt[r] = 0; sh.kt[r] = 0; }
        return;
    }
    int sig = 0;
    u64 amax = ax;
    if (PRO == PRO_NORMQUANT) {
        sig = bitlen_u64(ax) - 24;
        // pass 2: sum of squares of the 24-bit row and max |x' gamma|
        i64 ss = 0;
        u64 az = 0;
        for (int i = gt * 4; i < K; i += gn * 4) {
            const int4 v = *(const int4*)(xr + i);
            const int xv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const i64 xp = norm24(xv[j], sig);
                ss += xp * xp;
                az = umax64(az, absu(xp * (i64)a.gamma[i + j]));
            }
        }
        ss = warp_sum_i64(ss);
        az = warp_max_u64(az);
        if (lane == 0) { sh.red64[warp][0] = ss; sh.red64[warp][1] = (long long)az; }
        bar_named(bar, gn);
        ss = 0;
        az = 0;
        for (int w = 0; w < wpr; ++w) {
            ss += sh.red64[(r << lgw) + w][0];
            az = umax64(az, (u64)sh.red64[(r << lgw) + w][1]);
        }
        amax = az;
        if (gw == 0) {
            i64 eps_s;
            if (sig >= 0) eps_s = (2 * sig >= 62) ? 0 : (a.eps >> (2 * sig));
            else eps_s = a.eps * (1LL << (-2 * sig));
            const u64 rr = warp_isqrt64((u64)((ss >> a.lg_k) + eps_s));
            const int e = bitlen_u64(az);
            const u64 R = warp_udiv64(127ull << (e + 16), az);
            int m, k;
            warp_dyadic(az, 127ull * rr, &m, &k);
            if (lane == 0) {
                sh.bc[r][0] = (long long)R;
                sh.bc[r][1] = e + 16;
                sh.mt[r] = m;
                sh.kt[r] = k + 12;
            }
        }
    } else {
        if (gw == 0) {
            const int e = bitlen_u64(ax);
            const u64 R = warp_udiv64(127ull << (e + 16), ax);
            int m, k;
            warp_dyadic(ax, 127ull, &m, &k);
            if (lane == 0) {
                sh.bc[r][0] = (long long)R;
                sh.bc[r][1] = e + 16;
                sh.mt[r] = m;
                sh.kt[r] = k + a.F;
            }
        }
    }
    (void)amax;
    bar_named(bar, gn);
    const i64 R = sh.bc[r][0];
    const int shq = (int)sh.bc[r][1];
    // pass 3: quantise
    for (int i = gt * 4; i < K; i += gn * 4) {
        const int4 v = *(const int4*)(xr + i);
        const int xv[4] = {v.x, v.y, v.z, v.w};
        char4 q;
        i64 z[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            z[j] = (PRO == PRO_NORMQUANT) ? norm24(xv[j], sig) * (i64)a.gamma[i + j] : (i64)xv[j];
        q.x = (signed char)rshr(z[0] * R, shq);
        q.y = (signed char)rshr(z[1] * R, shq);
        q.z = (signed char)rshr(z[2] * R, shq);
        q.w = (signed char)rshr(z[3] * R, shq);
        *(char4*)(qr + i) = q;
    }
}

__device__ __forceinline__ i64 sg_requant(int acc, const SgShared& sh, const Epi& ep, int tk, int n) {
    const i64 M = (i64)sh.mt[tk] * (i64)ep.mc[n];
    return rshr((i64)acc * M, sh.kt[tk] + 22 - ep.fout);
}

template <int PRO, int MODE>
__global__ void __launch_bounds__(SG_THREADS, 1) k_sgemv(SgArgs a) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ SgShared sh;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int P = a.KC + 64;                      // ring row pitch (bank-conflict-free pairs)
    const int XP = a.K + 64;                      // activation row pitch
    unsigned char* ring = smem;
    int8_t* xs = (int8_t*)(smem + sg_ring_bytes(a.KC));
    int32_t* red = (int32_t*)(xs + (size_t)8 * XP);     // [8 warps][16][8]
    const int c = blockIdx.x;
    const int g0 = c * a.rg_q + min(c, a.rg_r);
    const int g1 = g0 + a.rg_q + (c < a.rg_r ? 1 : 0);
    const int units = (g1 - g0) * a.nkc;

    if (tid == 0) {
        for (int s = 0; s < SG_STAGES; ++s) {
            mbar_init(smem_u32(&sh.full[s]), 1);
            mbar_init(smem_u32(&sh.empty[s]), 8);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    pdl_launch();

    if (warp == 8) {
        // producer: weight rows of each (row group, K-chunk) unit into the ring
        int u = 0;
        for (int g = g0; g < g1; ++g) {
            for (int kc = 0; kc < a.nkc; ++kc, ++u) {
                const int s = u & (SG_STAGES - 1);
                if (u >= SG_STAGES && lane == 0) {
                    // bounded: on a timeout the status word records it and the
                    // stream continues (results are then invalid, nothing hangs)
                    if (!mbar_wait(smem_u32(&sh.empty[s]), ((u >> 2) - 1) & 1))
                        a.ep.status[ST_TIMEOUT] = 1;
                }
                __syncwarp();
                const uint32_t fb = smem_u32(&sh.full[s]);
                if (lane == 0) mbar_arrive_expect_tx(fb, 16u * a.KC);
                __syncwarp();
                if (lane < 16) {
                    const int row = min(g * 16 + lane, a.N - 1);
                    bulk_g2s(smem_u32(ring + ((size_t)s * 16 + lane) * P),
                             a.W + (size_t)row * a.K + (size_t)kc * a.KC, a.KC, fb);
                }
            }
        }
        return;
    }

    // compute warps
    pdl_wait();
    sg_prologue<PRO>(a, sh, xs, XP);
    bar_named(1, 256);

    const int g = lane >> 2, tq = lane & 3;
    const int nch = a.KC >> 6;
    int u = 0;
    for (int grp = g0; grp < g1; ++grp) {
        int acc[4] = {0, 0, 0, 0};
        for (int kc = 0; kc < a.nkc; ++kc, ++u) {
            const int s = u & (SG_STAGES - 1);
            if (!mbar_wait(smem_u32(&sh.full[s]), (u >> 2) & 1)) a.ep.status[ST_TIMEOUT] = 1;
            const int8_t* st = (const int8_t*)ring + (size_t)s * 16 * P;
            const int8_t* wlo = st + g * P + 16 * tq;
            const int8_t* whi = wlo + 8 * P;
            const int8_t* xb = xs + g * XP + kc * a.KC + 16 * tq;
            for (int ch = warp; ch < nch; ch += 8) {
                const int4 al = *(const int4*)(wlo + ch * 64);
                const int4 ah = *(const int4*)(whi + ch * 64);
                const int4 b = *(const int4*)(xb + ch * 64);
                mma_s8(acc, al.x, ah.x, al.y, ah.y, b.x, b.y);
                mma_s8(acc, al.z, ah.z, al.w, ah.w, b.z, b.w);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&sh.empty[s]));
        }
        int32_t* rw = red + warp * 128;
        rw[g * 8 + 2 * tq] = acc[0];
        rw[g * 8 + 2 * tq + 1] = acc[1];
        rw[(g + 8) * 8 + 2 * tq] = acc[2];
        rw[(g + 8) * 8 + 2 * tq + 1] = acc[3];
        bar_named(1, 256);
        const int n0 = grp * 16;
        const Epi& ep = a.ep;
        if (MODE == EPI_SWIGLU) {
            if (tid < 64) {
                const int p = tid >> 3, tk = tid & 7;
                int sg = 0, su = 0;
#pragma unroll
                for (int w = 0; w < 8; ++w) {
                    sg += red[w * 128 + (2 * p) * 8 + tk];
                    su += red[w * 128 + (2 * p + 1) * 8 + tk];
                }
                const int n = n0 + 2 * p;
                if (tk < a.M && n < a.N) {
                    i64 yg = sg_requant(sg, sh, ep, tk, n), yu = sg_requant(su, sh, ep, tk, n + 1);
                    if (yg > (1 << 24) || yg < -(1 << 24) || yu > (1 << 24) || yu < -(1 << 24))
                        ep.status[ST_SAT_GU] = 1;
                    yg = sat_b(yg, 1 << 24);
                    yu = sat_b(yu, 1 << 24);
                    ep.out[(size_t)tk * ep.ldo + (n >> 1)] = swiglu_dev((int)yg, (int)yu);
                }
            }
        } else if (tid < 128) {
            const int rr = tid >> 3, tk = tid & 7;
            int sum = 0;
#pragma unroll
            for (int w = 0; w < 8; ++w) sum += red[w * 128 + tid];
            const int n = n0 + rr;
            int outv = -2147483647;
            if (tk < a.M && n < a.N) {
                const i64 y = sg_requant(sum, sh, ep, tk, n);
                if (MODE == EPI_QKV) {
                    if (y > 2147483647LL || y < -2147483647LL) ep.status[ST_SAT_QKV] = 1;
                    ep.out[(size_t)tk * ep.ldo + n] = sat32(y);
                } else if (MODE == EPI_RESADD) {
                    int32_t* hp = ep.out + (size_t)tk * ep.ldo + n;
                    const i64 s2 = (i64)*hp + (i64)sat32(y);
                    if (s2 > 2147483647LL || s2 < -2147483647LL) ep.status[ST_SAT_RES] = 1;
                    *hp = sat32(s2);
                } else if (MODE == EPI_LOGITS) {
                    if (y > 2147483647LL || y < -2147483647LL) ep.status[ST_SAT_LOGIT] = 1;
                    outv = sat32(y);
                    ep.out[(size_t)tk * ep.ldo + n] = outv;
                }
            }
            if (MODE == EPI_LOGITS) {
                // per-token (max, lowest row) of this row group, via the red tile
                bar_named(2, 128);
                red[tid] = outv;          // warp 0's slot is free again after the sums
                bar_named(2, 128);
                if (tid < a.M) {
                    int bv = red[tid], bi = n0;
                    for (int q = 1; q < 16; ++q) {
                        const int v = red[q * 8 + tid];
                        if (v > bv && n0 + q < a.N) { bv = v; bi = n0 + q; }
                    }
                    ep.pval[(size_t)tid * ep.npart + grp] = bv;
                    ep.pidx[(size_t)tid * ep.npart + grp] = bi;
                }
            }
        }
        bar_named(1, 256);
    }
    // every issued copy has completed before the CTA exits (bounded wait;
    // normally these phases completed long ago)
    if (tid == 0) {
        for (int s = 0; s < SG_STAGES && s < units; ++s) {
            const int ul = s + ((units - 1 - s) >> 2) * SG_STAGES;   // last unit on stage s
            if (!mbar_wait(smem_u32(&sh.full[s]), (ul >> 2) & 1)) a.ep.status[ST_TIMEOUT] = 1;
        }
    }
}

}  // namespace detint
