// One decode step of up to 8 sequences in one cooperative launch.
//
// The integer arithmetic is exactly the multi-kernel step's (per-token
// NormQuant / ActQuant, int8 GEMVs with dyadic requantisation, QK-norm,
// RoPE from the int16 tables, fixed K/V scales, the shift-based softmax with
// 15-bit probabilities and two exact P·V limbs, SwiGLU, tie-low argmax;
// DetLLM blog, section "DetLLM" and its footnote on 15-bit probabilities),
// so every logit equals the oracle's. What this kernel changes is how the
// phases of a step wait for one another:
//
//  * Tagged words. Every activation row a phase hands to the next (q/k/v,
//    the attention output, the residual, the SwiGLU output, the argmax
//    partials) is written as 64-bit words holding the value in the low half
//    and a phase tag in the high half, by single-copy-atomic 64-bit stores.
//    A consumer polls the words it needs until their tags match: the data
//    and its readiness arrive in one L2 round trip, and no grid barrier,
//    counter or flag exists. Tags grow by one per phase (the step's base tag
//    lives in device memory and advances at the end of each step), so words
//    left from earlier phases or steps never match.
//  * Roles. CTAs [0, NG) run the GEMVs: a producer warp streams the CTA's
//    weight rows of every GEMV phase of the step through a ring of 16 KB
//    shared-memory slots (1D bulk copies, mbarrier completion), never
//    waiting on activations; 8 compute warps quantise the polled input row
//    into an int8 tile, take one weight row per warp (dp4a, lane-strided
//    16-byte chunks, one redux add per token) and apply the epilogue in the
//    same warp, with no block barrier between the dot products and the
//    stores; a ninth warp computes the per-token scales (integer square root
//    and dyadic division) beside them. CTAs [NG, NG + NA) run attention
//    only: each copies its items' cached K/V blocks into shared memory while
//    the GEMV phases of the previous layer run, so the attention phase reads
//    no global memory but the new token's q/k/v.
//  * Ordering. Every buffer a phase overwrites was last read by a phase that
//    each writer has (transitively) waited on, because every GEMV CTA owns
//    rows in every GEMV phase and every attention item waits on the q/k/v
//    rows of its head: the residual is rewritten only after all o rows, the
//    q/k/v rows only after the whole residual of the next layer, and so on.
//
// Every wait is bounded: after `spin` polls it records ST_TIMEOUT, marks the
// step as aborted (later waits of the step return at once) and continues,
// so a broken step ends with the flag set instead of hanging. At exit every
// bulk copy a CTA issued has completed (bounded wait).
#pragma once
#include "kernels.h"
#include "ptx.cuh"
#include "int_device.cuh"

namespace detint {

constexpr int MG_W = 8;                  // compute warps (+ producer warp 8 + scale warp 9)
constexpr int MG_MAXS = 16;              // ring slots at most
constexpr int MG_IPC = 4;                // attention items per attention CTA at most

enum { MG_BAR_STAT = 1, MG_BAR_Q = 2, MG_BAR_TS = 3, MG_BAR_ATT = 4, MG_BAR_END = 5, MG_BAR_STAT2 = 6,
       MG_BAR_INIT = 8 };
enum { MG_K_QKV = 0, MG_K_O = 1, MG_K_GU = 2, MG_K_D = 3, MG_K_LM = 4 };

// ---- tagged words
__device__ __forceinline__ void ll_put(u64* p, int v, unsigned tag) {
    const u64 w = ((u64)tag << 32) | (u64)(unsigned)v;
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}
__device__ __forceinline__ u64 ll_get(const u64* p) {
    u64 w;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(w) : "l"(p) : "memory");
    return w;
}
__device__ __forceinline__ void ll_get2(const u64* p, u64& a, u64& b) {
    asm volatile("ld.relaxed.gpu.global.v2.u64 {%0,%1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}
__device__ __forceinline__ unsigned ll_tag(u64 w) { return (unsigned)(w >> 32); }
__device__ __forceinline__ int ll_val(u64 w) { return (int)(unsigned)(w & 0xffffffffull); }
__device__ __forceinline__ unsigned ld_u32_relaxed(const unsigned* p) {
    unsigned v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

struct MgShared {
    unsigned long long full[MG_MAXS], empty[MG_MAXS];
    unsigned long long kvbar[MG_IPC];
    long long red[MG_W][5];
    int mt[8], kt[8];
    int bv[MG_W][8], bi[MG_W][8];
    int pos[8];
    unsigned base;
    int abort;
    int rw[5][2];                 // this GEMV CTA's weight rows per GEMV kind
};

// ---- bounded waits: poll until `ok`, else record the timeout and abort the step
__device__ __forceinline__ bool mg_aborted(const StepArgs& a, MgShared& sh, int it) {
    if (*(volatile int*)&sh.abort) return true;
    if ((it & 31) != 31) return false;
    if (ld_u32_relaxed(a.ctl + 1) == sh.base) { sh.abort = 1; return true; }
    return false;
}
__device__ __noinline__ void mg_timeout(const StepArgs& a, MgShared& sh) {
    a.status[ST_TIMEOUT] = 1;
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(a.ctl + 1), "r"(sh.base) : "memory");
    sh.abort = 1;
}

// ---------------------------------------------------------------- producer
__device__ void mg_phase_w(const StepArgs& a, int kind, const StepLayer& Lw, const int8_t** W, int* K) {
    const int nqkv = (a.nq + 2 * a.nkv) * a.d;
    (void)nqkv;
    switch (kind) {
        case MG_K_QKV: *W = Lw.w_qkv; *K = a.H; break;
        case MG_K_O: *W = Lw.w_o; *K = a.nq * a.d; break;
        case MG_K_GU: *W = Lw.w_gu; *K = a.H; break;
        case MG_K_D: *W = Lw.w_d; *K = a.F; break;
        default: *W = a.embed; *K = a.H; break;
    }
}

__device__ void mg_produce(const StepArgs& a, MgShared& sh, unsigned char* ring, int c) {
    const int lane = threadIdx.x & 31;
    const int NS = 1 << a.lg_ns;
    const uint64_t pol = l2_evict_first();
    int u = 0;
    for (int l = 0; l <= a.L; ++l) {
        const int nph = l < a.L ? 4 : 1;
        for (int p = 0; p < nph; ++p) {
            const int kind = l < a.L ? p : MG_K_LM;
            const int8_t* W;
            int K;
            mg_phase_w(a, kind, a.layers[l < a.L ? l : 0], &W, &K);
            const int r0 = a.rows[kind * (a.NG + 1) + c], r1 = a.rows[kind * (a.NG + 1) + c + 1];
            const int R = step_rows_per_slot(K);
            for (int r = r0; r < r1; r += R, ++u) {
                const int s = u & (NS - 1);
                if (u >= NS && lane == 0) {
                    if (!mbar_wait(smem_u32(&sh.empty[s]), ((u >> a.lg_ns) - 1) & 1)) a.status[ST_TIMEOUT] = 1;
                }
                __syncwarp();
                if (lane == 0) {
                    const int nr = min(R, r1 - r);
                    const uint32_t bytes = (uint32_t)nr * (uint32_t)K;
                    const uint32_t fb = smem_u32(&sh.full[s]);
                    mbar_arrive_expect_tx(fb, bytes);
                    bulk_g2s_hint(smem_u32(ring + (size_t)s * STEP_SLOT), W + (size_t)r * K, bytes, fb, pol);
                }
            }
        }
    }
}

// ------------------------------------------------------------ GEMV phases
struct MgPhase {
    int kind, K, N, r0, r1;
    const int32_t* mc;
    const int16_t* gamma;        // NormQuant gamma, or null for ActQuant
    int F_in;                    // ActQuant fixed point
    const u64* src;              // tagged input rows [T][K], or null: the embedding rows
    unsigned tin, tout;
    u64* dst;                    // tagged output rows (QKV, RESADD, SWIGLU)
    int ldo;
    int fout;
};

// token groups: 8 >> lgT warps per token row
__device__ __forceinline__ int mg_lgT(int T) { return T <= 1 ? 0 : (T <= 2 ? 1 : (T <= 4 ? 2 : 3)); }

// input value j of this thread: tagged pair q = gt + gn * j of token row r
// (its two values), from the embedding at layer 0
__device__ __forceinline__ void mg_embed_pair(const StepArgs& a, int id, int k, int& v0, int& v1) {
    const i64 m = a.embed_m[id];
    const char2 e = *(const char2*)(a.embed + (size_t)id * a.H + k);
    v0 = (int)rshr((i64)e.x * m, 6);
    v1 = (int)rshr((i64)e.y * m, 6);
}

__device__ __forceinline__ int mg_token_id(const StepArgs& a, int t) {
    int id = a.tokens[t];
    if (id < 0 || id >= a.V) id = 0;    // flagged once by CTA 0 at the start of the step
    return id;
}

// quantisation prologue: poll (or compute) the T input rows into the int32
// row buffer xin, gathering the per-token statistics as the values arrive,
// then the multiplier and the int8 tile x8. Compact runtime loops: this code
// runs once per phase on every GEMV CTA, and its instructions must stay in
// the SM's instruction cache. The scale warp (warp 9) joins the statistics
// barriers and computes (m_t, k_t).
__device__ void mg_prologue(const StepArgs& a, MgShared& sh, const MgPhase& P, int8_t* x8, int XP,
                            int32_t* xin, int16_t* gs) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int T = a.T, K = P.K, lgT = mg_lgT(T);
    const int lgw = 3 - lgT;                      // log2 warps per token row
    const int r = warp >> lgw, gw = warp & ((1 << lgw) - 1);
    const int gt = gw * 32 + lane, lgn = 5 + lgw, gn = 1 << lgn;
    const int npair = K >> 1;
    const bool norm = P.gamma != nullptr;
    const bool live = r < T;
    int32_t* xr = xin + (size_t)r * XP;
    // this thread's gamma pairs into shared memory (only this thread reads them)
    if (norm && live)
        for (int q = gt; q < npair; q += gn) *(short2*)(gs + 2 * q) = *(const short2*)(P.gamma + 2 * q);
    unsigned ax = 0;
    u64 ag = 0, sq = 0;
    auto take = [&](int q, int v0, int v1) {
        *(int2*)(xr + 2 * q) = make_int2(v0, v1);
        ax = max(ax, max((unsigned)absu(v0), (unsigned)absu(v1)));
        if (norm) {
            const short2 g2 = *(const short2*)(gs + 2 * q);
            ag = umax64(ag, umax64(absu((i64)v0 * g2.x), absu((i64)v1 * g2.y)));
            sq += (u64)((i64)v0 * v0) + (u64)((i64)v1 * v1);
        }
    };
    if (live) {
        if (!P.src) {
            const int id = mg_token_id(a, r);
            const i64 m = a.embed_m[id];
            const int8_t* er = a.embed + (size_t)id * a.H;
            for (int q = gt; q < npair; q += gn) {
                const char2 e = *(const char2*)(er + 2 * q);
                take(q, (int)rshr((i64)e.x * m, 6), (int)rshr((i64)e.y * m, 6));
            }
        } else {
            const u64* src = P.src + (size_t)r * K;
            unsigned long long got = 0;          // pairs q = gt + gn j received (j < 64)
            for (int it = 0;; ++it) {
                bool all = true;
                int j = 0;
                for (int q = gt; q < npair; q += gn, ++j) {
                    if ((got >> j) & 1ull) continue;
                    u64 w0, w1;
                    ll_get2(src + 2 * q, w0, w1);
                    if (ll_tag(w0) == P.tin && ll_tag(w1) == P.tin) {
                        take(q, ll_val(w0), ll_val(w1));
                        got |= 1ull << j;
                    } else {
                        all = false;
                    }
                }
                if (all) break;
                if (it >= a.spin || mg_aborted(a, sh, it)) {
                    if (!sh.abort) mg_timeout(a, sh);
                    break;
                }
            }
        }
    }
    // pass 1 (gathered above): max |x|; NormQuant also max |x gamma| and the
    // sum of x^2, exact when every |x| < 2^24 (the 24-bit normalisation is
    // then a left shift)
    ax = __reduce_max_sync(0xffffffffu, ax);
    if (norm) { ag = redux_max_u64(ag); sq = redux_sum_u64(sq); }
    if (lane == 0) { sh.red[warp][0] = ax; sh.red[warp][1] = (long long)ag; sh.red[warp][2] = (long long)sq; }
    bar_named(MG_BAR_STAT, 288);
    // ---- per-token statistics of the group's warps: lane i reads warp
    // w0 + (i mod wpr), and one warp-wide reduction combines them (maxima
    // tolerate the repeats; sums count lanes i < wpr only)
    const int w0 = r << lgw, wpr = 1 << lgw;
    const int wsrc = w0 + (lane & (wpr - 1));
    const u64 axl = redux_max_u64((u64)sh.red[wsrc][0]);
    // any token needing the 24-bit right shift (uniform: the maximum over every warp)
    const bool pass2 = norm && bitlen_u64(redux_max_u64((u64)sh.red[lane & 7][0])) > 24;
    const int sig = norm ? bitlen_u64(axl) - 24 : 0;
    u64 amax = axl;
    if (norm) amax = sig <= 0 ? redux_max_u64((u64)sh.red[wsrc][1]) << -sig : 0;
    if (pass2) {
        i64 ss = 0;
        u64 az = 0;
        if (live && sig > 0)
            for (int q = gt; q < npair; q += gn) {
                const int2 v = *(const int2*)(xr + 2 * q);
                const short2 g2 = *(const short2*)(gs + 2 * q);
                const i64 x0 = norm24(v.x, sig), x1 = norm24(v.y, sig);
                ss += x0 * x0 + x1 * x1;
                az = umax64(az, umax64(absu(x0 * g2.x), absu(x1 * g2.y)));
            }
        ss = (i64)redux_sum_u64((u64)ss);
        az = redux_max_u64(az);
        if (lane == 0) { sh.red[warp][3] = ss; sh.red[warp][4] = (long long)az; }
        bar_named(MG_BAR_STAT2, 288);
        if (sig > 0) amax = redux_max_u64((u64)sh.red[wsrc][4]);
    }
    // ---- quantise with the per-row multiplier R = floor(127 2^(e+16) / amax)
    if (live) {
        int8_t* qr = x8 + (size_t)r * XP;
        const int e = bitlen_u64(amax);
        const i64 R = amax ? (i64)pow2_recip(amax, e, 127, 16) : 0;
        const int shq = e + 16;
#pragma unroll 2
        for (int q = gt; q < npair; q += gn) {
            const int2 v = *(const int2*)(xr + 2 * q);
            i64 z0 = v.x, z1 = v.y;
            if (norm) {
                const short2 g2 = *(const short2*)(gs + 2 * q);
                z0 = norm24(v.x, sig) * (i64)g2.x;
                z1 = norm24(v.y, sig) * (i64)g2.y;
            }
            char2 c2;
            c2.x = (signed char)rshr(z0 * R, shq);
            c2.y = (signed char)rshr(z1 * R, shq);
            *(char2*)(qr + 2 * q) = c2;
        }
    }
    bar_named(MG_BAR_Q, 256);
}

// the scale warp's share of a prologue: joins the statistics barriers, then
// computes every token's (m_t, k_t) and releases the epilogues
__device__ void mg_scales(const StepArgs& a, MgShared& sh, const MgPhase& P) {
    const int T = a.T, lgw = 3 - mg_lgT(T), wpr = 1 << lgw, lane = threadIdx.x & 31;
    const bool norm = P.gamma != nullptr;
    bar_named(MG_BAR_STAT, 288);
    const bool pass2 = norm && bitlen_u64(redux_max_u64((u64)sh.red[lane & 7][0])) > 24;
    if (pass2) bar_named(MG_BAR_STAT2, 288);
    int lg_k = 0;
    while ((1 << lg_k) < P.K) ++lg_k;
    for (int t = 0; t < T; ++t) {
        const int wsrc = (t << lgw) + (lane & (wpr - 1));
        const bool first = lane < wpr;            // counts each warp of the group once in sums
        const u64 axl = redux_max_u64((u64)sh.red[wsrc][0]);
        int m = 0, k = 0;
        if (axl != 0) {
            if (norm) {
                const int sig = bitlen_u64(axl) - 24;
                i64 ss;
                u64 az;
                if (sig <= 0) {
                    ss = (i64)redux_sum_u64(first ? (u64)sh.red[wsrc][2] : 0) << (-2 * sig);
                    az = redux_max_u64((u64)sh.red[wsrc][1]) << -sig;
                } else {
                    ss = (i64)redux_sum_u64(first ? (u64)sh.red[wsrc][3] : 0);
                    az = redux_max_u64((u64)sh.red[wsrc][4]);
                }
                i64 eps_s;
                if (sig >= 0) eps_s = (2 * sig >= 62) ? 0 : (a.eps_h >> (2 * sig));
                else eps_s = a.eps_h * (1LL << (-2 * sig));
                const u64 rr = isqrt_fast((u64)((ss >> lg_k) + eps_s));
                dyadic_fast(az, 127ull * rr, &m, &k);
                k += 12;
            } else {
                dyadic_fast(axl, 127ull, &m, &k);
                k += P.F_in;
            }
        }
        if (lane == 0) { sh.mt[t] = m; sh.kt[t] = k; }
    }
    __syncwarp();
    bar_arrive_named(MG_BAR_TS, 288);
}

// dot products of the ring slots of this phase and the epilogues (compute
// warps). The two halves of the compute warps (warps 0-3, 4-7) take
// alternate slots, so two slots are in flight at once. In a slot of 16 rows
// each half-warp takes two rows (lane l of the half reads 16-byte chunks l,
// l + 16, ...; a 4-step shuffle sums the half), a gate/up pair being the
// same rows of the two halves of a warp; in a slot of fewer rows each warp
// takes rows wg and wg + 4 (a gate/up pair: rows 2 wg and 2 wg + 1). Tokens
// run in a loop (the weight row is re-read from shared memory per token),
// so the code stays small; lane t of a row keeps token t's sum and applies
// its epilogue.
__device__ __forceinline__ void mg_epilogue(const StepArgs& a, MgShared& sh, const MgPhase& P, int t, int n,
                                            int sa, int sb, int32_t* hown, const int32_t* mcs, int& bestv,
                                            int& besti) {
    const i64 mt = sh.mt[t];
    const int shf = sh.kt[t] + 22 - P.fout;
    const i64 mca = mcs[n - P.r0];
    const i64 y = rshr((i64)sa * (mt * mca), shf);
    if (P.kind == MG_K_GU) {
        const i64 mcb = mcs[n + 1 - P.r0];
        const i64 yu = rshr((i64)sb * (mt * mcb), shf);
        if (y > (1 << 24) || y < -(1 << 24) || yu > (1 << 24) || yu < -(1 << 24)) a.status[ST_SAT_GU] = 1;
        ll_put(P.dst + (size_t)t * P.ldo + (n >> 1), swiglu_dev((int)sat_b(y, 1 << 24), (int)sat_b(yu, 1 << 24)),
               P.tout);
    } else if (P.kind == MG_K_QKV) {
        if (y > 2147483647LL || y < -2147483647LL) a.status[ST_SAT_QKV] = 1;
        ll_put(P.dst + (size_t)t * P.ldo + n, sat32(y), P.tout);
    } else if (P.kind == MG_K_LM) {
        if (y > 2147483647LL || y < -2147483647LL) a.status[ST_SAT_LOGIT] = 1;
        const int lv = sat32(y);
        a.logits[(size_t)t * a.V + n] = lv;
        if (lv > bestv) { bestv = lv; besti = n; }   // a lane's rows ascend: ties keep the lower id
    } else {
        int32_t* hp = hown + t * STEP_HOWN + (n - P.r0);
        const i64 s2 = (i64)*hp + (i64)sat32(y);
        if (s2 > 2147483647LL || s2 < -2147483647LL) a.status[ST_SAT_RES] = 1;
        const int hv = sat32(s2);
        *hp = hv;
        ll_put(P.dst + (size_t)t * P.ldo + n, hv, P.tout);
    }
}

// token t's dot product of weight row w with the int8 tile row x over this
// lane's chunks ch = li, li + lstep, ... (partial; the caller sums the lanes)
__device__ __forceinline__ int mg_dot_part(const unsigned char* w, const int8_t* x, int li, int lstep, int nch) {
    int acc = 0;
#pragma unroll 4
    for (int ch = li; ch < nch; ch += lstep) {
        const int4 wv = *(const int4*)(w + ch * 16);
        const int4 xv = *(const int4*)(x + ch * 16);
        acc = __dp4a(wv.x, xv.x, acc);
        acc = __dp4a(wv.y, xv.y, acc);
        acc = __dp4a(wv.z, xv.z, acc);
        acc = __dp4a(wv.w, xv.w, acc);
    }
    return acc;
}

__device__ void mg_consume(const StepArgs& a, MgShared& sh, const MgPhase& P, const unsigned char* ring,
                           const int8_t* x8, int XP, int32_t* hown, const int32_t* mcs, int& u,
                           int& bestv, int& besti) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int grp = warp >> 2, wg = warp & 3;
    const int NS = 1 << a.lg_ns, T = a.T, K = P.K;
    const int R = step_rows_per_slot(K);
    const int nch = K >> 4;                        // 16-byte chunks per row
    const bool swi = P.kind == MG_K_GU;
    const bool hrow = R >= 16;                     // a half-warp per row
    const int li = hrow ? (lane & 15) : lane;      // lane within the row's group
    const int lstep = hrow ? 16 : 32;
    // the two rows of this lane in a slot
    int r0, r1;
    if (hrow) {
        const int hw = 2 * wg + (lane >> 4);
        if (swi) { r0 = 4 * wg + (lane >> 4); r1 = r0 + 2; }   // pairs 2wg, 2wg+1: gate in half 0, up in half 1
        else { r0 = hw; r1 = hw + 8; }
    } else {
        if (swi) { r0 = 2 * wg; r1 = 2 * wg + 1; }
        else { r0 = wg; r1 = wg + 4; }
    }
    bool scales = false;
    for (int k = 0, rb = P.r0; rb < P.r1; ++k, rb += R, ++u) {
        if ((u & 1) != grp) continue;              // the other group's slot
        const int s = u & (NS - 1);
        const int nr = min(R, P.r1 - rb);
        const bool h0 = r0 < nr, h1 = r1 < nr;
        // every warp of the group waits for the slot's copy before it releases
        // the slot, so that no release can count towards an earlier use
        const uint32_t fb = smem_u32(&sh.full[s]);
        if (!mbar_test_wait(fb, (u >> a.lg_ns) & 1) && !mbar_wait(fb, (u >> a.lg_ns) & 1))
            a.status[ST_TIMEOUT] = 1;
        const unsigned char* slot = ring + (size_t)s * STEP_SLOT;
        int s0 = 0, s1 = 0;                        // token li's sums of rows r0, r1
        for (int t = 0; t < T; ++t) {
            const int8_t* xt = x8 + (size_t)t * XP;
            int a0 = h0 ? mg_dot_part(slot + (size_t)r0 * K, xt, li, lstep, nch) : 0;
            int a1 = h1 ? mg_dot_part(slot + (size_t)r1 * K, xt, li, lstep, nch) : 0;
            if (hrow) {
#pragma unroll
                for (int o = 8; o; o >>= 1) {
                    a0 += __shfl_xor_sync(0xffffffffu, a0, o);
                    a1 += __shfl_xor_sync(0xffffffffu, a1, o);
                }
            } else {
                if (h0) a0 = __reduce_add_sync(0xffffffffu, a0);
                if (h1) a1 = __reduce_add_sync(0xffffffffu, a1);
            }
            if (li == t) { s0 = a0; s1 = a1; }
        }
        int u0 = 0, u1 = 0;                        // gate/up in halves: the up rows' sums
        if (hrow && swi) {
            u0 = __shfl_down_sync(0xffffffffu, s0, 16);
            u1 = __shfl_down_sync(0xffffffffu, s1, 16);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sh.empty[s]));
        // every warp takes the token-scale barrier in its first slot of the
        // phase (or after the loop when it has none): deferring it could leave
        // warps waiting on slots that are refilled only after the warps
        // blocked at the barrier release theirs
        if (!scales) { bar_named(MG_BAR_TS, 288); scales = true; }
        if (li >= T) continue;
        if (swi) {
            if (hrow) {
                if (lane >= 16) continue;
                if (h0) mg_epilogue(a, sh, P, li, rb + r0, s0, u0, hown, mcs, bestv, besti);
                if (h1) mg_epilogue(a, sh, P, li, rb + r1, s1, u1, hown, mcs, bestv, besti);
            } else if (h0) {
                mg_epilogue(a, sh, P, li, rb + r0, s0, s1, hown, mcs, bestv, besti);
            }
            continue;
        }
        if (h0) mg_epilogue(a, sh, P, li, rb + r0, s0, 0, hown, mcs, bestv, besti);
        if (h1) mg_epilogue(a, sh, P, li, rb + r1, s1, 0, hown, mcs, bestv, besti);
    }
    if (!scales) bar_named(MG_BAR_TS, 288);
}

// ----------------------------------------------------------- attention
template <int EPL>
__device__ void mg_qk_norm(i64 (&y)[EPL], const int16_t* gamma, int lane, i64 eps) {
    constexpr int LG_D = EPL == 4 ? 7 : 6;
    u64 ax = 0;
#pragma unroll
    for (int j = 0; j < EPL; ++j) ax = umax64(ax, absu(y[j]));
    ax = redux_max_u64(ax);
    if (ax == 0) return;
    const int sig = bitlen_u64(ax) - 24;
    i64 xp[EPL];
    i64 ss = 0;
#pragma unroll
    for (int j = 0; j < EPL; ++j) { xp[j] = norm24(y[j], sig); ss += xp[j] * xp[j]; }
    ss = (i64)redux_sum_u64((u64)ss);
    i64 eps_s;
    if (sig >= 0) eps_s = (2 * sig >= 62) ? 0 : (eps >> (2 * sig));
    else eps_s = eps * (1LL << (-2 * sig));
    const i64 rr = (i64)isqrt_fast((u64)((ss >> LG_D) + eps_s));
    const i64 Rr = (i64)pow2_recip((u64)rr, bitlen_u64((u64)rr), 1, 23);
    const int shn = bitlen_u64((u64)rr) + 21;
#pragma unroll
    for (int j = 0; j < EPL; ++j) y[j] = rshr(xp[j] * (i64)gamma[lane + 32 * j] * Rr, shn);
}

template <int EPL>
__device__ __forceinline__ void mg_rope(i64 (&y)[EPL], const int16_t* cr, const int16_t* sr, int lane) {
#pragma unroll
    for (int j = 0; j < EPL / 2; ++j) {
        const int i = lane + 32 * j;
        const i64 c = cr[i], s = sr[i];
        const i64 x0 = y[j], x1 = y[j + EPL / 2];
        y[j] = rshr(x0 * c - x1 * s, 14);
        y[j + EPL / 2] = rshr(x1 * c + x0 * s, 14);
    }
}

// poll the tagged words p[lane + 32 j] (and p2[...] when given) of one warp (bounded)
template <int EPL>
__device__ void mg_poll_head(const StepArgs& a, MgShared& sh, const u64* p, unsigned tag, i64 (&y)[EPL],
                             const u64* p2 = nullptr, i64* y2 = nullptr) {
    const int lane = threadIdx.x & 31;
    unsigned got = 0;
    const unsigned want = p2 ? (1u << (2 * EPL)) - 1 : (1u << EPL) - 1;
    for (int it = 0;; ++it) {
#pragma unroll
        for (int j = 0; j < EPL; ++j) {
            if (!((got >> j) & 1u)) {
                const u64 w = ll_get(p + lane + 32 * j);
                if (ll_tag(w) == tag) { y[j] = ll_val(w); got |= 1u << j; }
            }
            if (p2 && !((got >> (EPL + j)) & 1u)) {
                const u64 w = ll_get(p2 + lane + 32 * j);
                if (ll_tag(w) == tag) { y2[j] = ll_val(w); got |= 1u << (EPL + j); }
            }
        }
        if (__all_sync(0xffffffffu, got == want)) break;
        if (it >= a.spin || mg_aborted(a, sh, it)) {
            if (lane == 0 && !sh.abort) mg_timeout(a, sh);
            __syncwarp();
            break;
        }
    }
}

// offsets of the parameter rows in an item's staging region (after K and V)
template <int D>
struct MgAux {
    static constexpr int KVP = 0, QG = (8 + D / 2) * 4, KG = QG + 2 * D, CS = KG + 2 * D, SN = CS + D, BT = SN + D;
};

// one attention item (token t, kv head g) of layer l on warps 0..8 of an
// attention CTA; the sequence's earlier K/V blocks are in Ks / Vs when
// staged, the item's parameter rows in aux (both completing on kvb)
template <int EPL, int G>
__device__ void mg_attention(const StepArgs& a, MgShared& sh, const StepLayer& Lw, int l, int t, int g,
                             int8_t* Ks, int8_t* Vs, const unsigned char* aux, bool staged, uint32_t kvb,
                             unsigned char* scr) {
    constexpr int D = EPL * 32, NC = D >> 4, DH2 = D / 2;
    using X = MgAux<D>;
    __shared__ int32_t mqs[G], kqs[G];
    __shared__ unsigned long long amq[G];
    __shared__ int red_i[8][G];
    __shared__ i64 red_l[8][G], rs_s[G];
    __shared__ int bl_s[G];
    const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
    const int scap = a.scap;
    int8_t* qs = (int8_t*)scr;                          // [G][D]
    int32_t* S = (int32_t*)(scr + G * D);               // [G][scap]
    unsigned char* Elo = (unsigned char*)(S + (size_t)G * scap);
    unsigned char* Ehi = Elo + (size_t)G * scap;
    int32_t* pv = (int32_t*)(Ehi + (size_t)G * scap);   // [G][D][2]
    const unsigned tag = sh.base + 5 * l;               // q/k/v of this layer
    const int nqkv = (a.nq + 2 * a.nkv) * D;
    const int pos = sh.pos[t];
    const int ctx = pos + 1, ctx16 = (ctx + 15) & ~15;
    const int nb = (ctx + KV_BLK - 1) >> 6;
    const int32_t* kvp = (const int32_t*)(aux + X::KVP);
    const int* bt = (const int*)(aux + X::BT);
    const u64* row = a.xqkv + (size_t)t * nqkv;

    // ---- q heads (warps 0..G-1) and the new key / value (warp G)
    if (w <= G) {
        const int16_t* cr = (const int16_t*)(aux + X::CS);
        const int16_t* sr = (const int16_t*)(aux + X::SN);
        if (!mbar_wait(kvb, l & 1)) a.status[ST_TIMEOUT] = 1;    // parameter rows (and K/V) staged
        int E = 0;
        for (int i = lane; i < DH2; i += 32) E = max(E, kvp[8 + i]);
        E = __reduce_max_sync(0xffffffffu, (unsigned)E);
        i64 y[EPL];
        if (w < G) {
            const int hq = (g << a.lg_grp) + w;
            mg_poll_head<EPL>(a, sh, row + (size_t)hq * D, tag, y);
            if (a.qk_norm) mg_qk_norm<EPL>(y, (const int16_t*)(aux + X::QG), lane, a.eps_qk);
            else {
#pragma unroll
                for (int j = 0; j < EPL; ++j) y[j] *= 4;
            }
            mg_rope<EPL>(y, cr, sr, lane);
            u64 am = 0;
#pragma unroll
            for (int j = 0; j < EPL; ++j) {
                const int i = lane + 32 * j;
                const int ec = kvp[8 + (i & (DH2 - 1))];
                y[j] = y[j] * (1LL << (E - ec));
                am = umax64(am, absu(y[j]));
            }
            am = redux_max_u64(am);
            int8_t* qo = qs + w * D;
            // the head's scale (m_q, k_q) = dyadic(am, 127) is formed by warp 8
            // during the score pass; only the multiplier is on this path
            if (lane == 0) amq[w] = am;
            const int e = bitlen_u64(am);
            const i64 R = am ? (i64)pow2_recip(am, e, 127, 16) : 0;
#pragma unroll
            for (int j = 0; j < EPL; ++j) qo[lane + 32 * j] = (int8_t)rshr(y[j] * R, e + 16);
        } else {
            i64 v[EPL];
            mg_poll_head<EPL>(a, sh, row + (size_t)(a.nq + g) * D, tag, y, row + (size_t)(a.nq + a.nkv + g) * D, v);
            if (a.qk_norm) mg_qk_norm<EPL>(y, (const int16_t*)(aux + X::KG), lane, a.eps_qk);
            else {
#pragma unroll
                for (int j = 0; j < EPL; ++j) y[j] *= 4;
            }
            mg_rope<EPL>(y, cr, sr, lane);
            const int blk = bt[pos >> 6];
            const int off = pos & (KV_BLK - 1);
            int8_t* kd = Lw.kc + (((size_t)blk * a.nkv + g) * KV_BLK + off) * D;
            int8_t* vd = Lw.vc + ((size_t)blk * a.nkv + g) * D * KV_BLK + off;
            const i64 KQM = kvp[0], VQM = kvp[2];
            const int KQS = kvp[1], VQS = kvp[3];
            int8_t* ks = Ks + (size_t)pos * D;
            int8_t* vs = Vs + (size_t)(nb - 1) * KV_BLK * D + off;
#pragma unroll
            for (int j = 0; j < EPL; ++j) {
                const int i = lane + 32 * j;
                const int ec = kvp[8 + (i & (DH2 - 1))];
                const int8_t k8 = (int8_t)sat127(rshr(y[j] * (1LL << ec) * KQM, KQS));
                const int8_t v8 = (int8_t)sat127(rshr(v[j] * VQM, VQS));
                kd[i] = k8;
                vd[(size_t)i * KV_BLK] = v8;
                if (staged) {
                    ks[i] = k8;
                    vs[(size_t)i * KV_BLK] = v8;
                }
            }
        }
    }
    if (w > G && lane == 0 && !mbar_wait(kvb, l & 1)) a.status[ST_TIMEOUT] = 1;
    bar_named(MG_BAR_ATT, 288);

    const i64 CSTM = kvp[6], MV = kvp[4];
    const int CSTK = kvp[7], KVS = kvp[5];
    // ---- scores and per-head maxima (warps 0..7); warp 8: the q heads' scales
    if (w == 8 && lane < G) {          // lane hh: head hh
        int m = 0, k = 0;
        if (amq[lane]) {
            dyadic_fast(amq[lane], 127ull, &m, &k);
            k += 14;
        }
        mqs[lane] = m;
        kqs[lane] = k;
    }
    if (tid < 256) {
        int smax[G];
#pragma unroll
        for (int hh = 0; hh < G; ++hh) smax[hh] = -2147483647;
        for (int j = tid; j < ctx; j += 256) {
            const int8_t* kr = staged ? Ks + (size_t)j * D
                                      : Lw.kc + (((size_t)bt[j >> 6] * a.nkv + g) * KV_BLK + (j & 63)) * D;
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
            for (int hh = 0; hh < G; ++hh) { S[hh * scap + j] = acc[hh]; smax[hh] = max(smax[hh], acc[hh]); }
        }
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
            const int v = (int)__reduce_max_sync(0xffffffffu, (unsigned)(smax[hh] ^ 0x80000000)) ^ 0x80000000;
            if (lane == 0) red_i[w][hh] = v;
        }
    }
    bar_named(MG_BAR_ATT, 288);
    // ---- 15-bit weights as two byte planes, and the row sums; every thread
    // forms the heads' maximum logits from the warps' maximum scores
    if (tid < 256) {
        i64 umax_s[G];
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
            int v = red_i[0][hh];
            for (int w2 = 1; w2 < 8; ++w2) v = max(v, red_i[w2][hh]);
            umax_s[hh] = rshr((i64)v * (i64)mqs[hh] * CSTM, kqs[hh] + CSTK - 10);
        }
        i64 sum[G];
#pragma unroll
        for (int hh = 0; hh < G; ++hh) sum[hh] = 0;
        for (int j = tid; j < ctx16; j += 256) {
#pragma unroll
            for (int hh = 0; hh < G; ++hh) {
                int Ej = 0;
                if (j < ctx) {
                    const i64 uu = rshr((i64)S[hh * scap + j] * (i64)mqs[hh] * CSTM, kqs[hh] + CSTK - 10);
                    Ej = min(32767, exp2q_dev(uu - umax_s[hh]));
                }
                Elo[hh * scap + j] = (unsigned char)(Ej & 255);
                Ehi[hh * scap + j] = (unsigned char)(Ej >> 8);
                sum[hh] += Ej;
            }
        }
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
            const i64 v = (i64)__reduce_add_sync(0xffffffffu, (unsigned)sum[hh]);   // < 2^15 * 2^11 per warp
            if (lane == 0) red_l[w][hh] = v;
        }
    }
    bar_named(MG_BAR_ATT, 288);
    if (w == 8) {
        // ---- row sums and RS = floor(2^(bl + 23) / sum), beside the P·V products
        for (int hh = 0; hh < G; ++hh) {
            i64 v = 0;
            for (int w2 = 0; w2 < 8; ++w2) v += red_l[w2][hh];
            const int bl = bitlen_u64((u64)v);
            const i64 rs = (i64)pow2_recip((u64)v, bl, 1, 23);
            if (lane == 0) { rs_s[hh] = rs; bl_s[hh] = bl; }
        }
    } else {
        // ---- P·V: lane (channel c of 8, key chunk q of 4) of warp w
        const int q = lane & 3, cl = lane >> 2;
        for (int cg = w; cg < (D >> 3); cg += 8) {
            const int c = cg * 8 + cl;
            int lo[G], hi[G];
#pragma unroll
            for (int hh = 0; hh < G; ++hh) { lo[hh] = 0; hi[hh] = 0; }
            for (int b = 0; b < nb; ++b) {
                const int j0 = b * KV_BLK + q * 16;
                if (j0 >= ctx16) break;
                const int8_t* vp = staged ? Vs + (size_t)b * KV_BLK * D + c * KV_BLK + q * 16
                                          : Lw.vc + (((size_t)bt[b] * a.nkv + g) * D + c) * KV_BLK + q * 16;
                const int4 vw = *(const int4*)vp;
#pragma unroll
                for (int hh = 0; hh < G; ++hh) {
                    const uint4 el = *(const uint4*)(Elo + hh * scap + j0);
                    const int4 eh = *(const int4*)(Ehi + hh * scap + j0);
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
    bar_named(MG_BAR_ATT, 288);
    // ---- normalisation and the output rows (Q12), as tagged words
    const unsigned tout = sh.base + 5 * l + 1;
    u64* orow = a.xo + (size_t)t * a.nq * D + (size_t)(g << a.lg_grp) * D;
    for (int idx = tid; idx < G * D; idx += 288) {
        const int hh = idx / D;
        const i64 num = (i64)pv[idx * 2 + 1] * 256 + pv[idx * 2];
        const i64 tq = rshr(num * rs_s[hh], bl_s[hh] + 7);
        const i64 ov = rshr(tq * MV, KVS + 16 - 12);
        ll_put(orow + idx, (int)ov, tout);
    }
    bar_named(MG_BAR_ATT, 288);
}

// item (t, g) of layer l, by thread 0: its parameter rows into aux (the
// block-table row by plain loads, the rest by 1D bulk copies) and, when
// staged, the K/V blocks of every position before this step's into Ks / Vs;
// the copies complete on kvb (one phase per layer)
template <int D>
__device__ void mg_stage(const StepArgs& a, MgShared& sh, const StepLayer& Lw, int t, int g, int8_t* Ks,
                         int8_t* Vs, unsigned char* aux, bool staged, uint32_t kvb) {
    using X = MgAux<D>;
    constexpr int DH2 = D / 2;
    constexpr uint32_t BLK = (uint32_t)KV_BLK * D;
    constexpr uint32_t PAR = (uint32_t)X::BT;            // parameter bytes copied in bulk
    const int pos = sh.pos[t];
    const int nb = (pos + 1 + KV_BLK - 1) >> 6;
    const int* bt = a.block_table + (size_t)a.tok_seq[t] * a.mbs;
    int* bts = (int*)(aux + X::BT);
    for (int b = 0; b < nb; ++b) bts[b] = bt[b];
    mbar_arrive_expect_tx(kvb, PAR + (staged ? (uint32_t)nb * 2u * BLK : 0u));
    bulk_g2s(smem_u32(aux + X::KVP), Lw.kvp + (size_t)g * (8 + DH2), (8 + DH2) * 4, kvb);
    bulk_g2s(smem_u32(aux + X::QG), Lw.q_gamma, 2 * D, kvb);
    bulk_g2s(smem_u32(aux + X::KG), Lw.k_gamma, 2 * D, kvb);
    bulk_g2s(smem_u32(aux + X::CS), a.rope_cos + (size_t)pos * DH2, 2 * DH2, kvb);
    bulk_g2s(smem_u32(aux + X::SN), a.rope_sin + (size_t)pos * DH2, 2 * DH2, kvb);
    if (!staged) return;
    for (int b = 0; b < nb; ++b) {
        const size_t unit = (size_t)bts[b] * a.nkv + g;
        bulk_g2s(smem_u32(Ks + (size_t)b * BLK), Lw.kc + unit * BLK, BLK, kvb);
        bulk_g2s(smem_u32(Vs + (size_t)b * BLK), Lw.vc + unit * BLK, BLK, kvb);
    }
}

template <int EPL, int G>
__global__ void __launch_bounds__(STEP_THREADS, 1) k_decode_step(StepArgs a) {
    constexpr int D = EPL * 32;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ MgShared sh;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = blockIdx.x;
    const int NS = 1 << a.lg_ns;
    if (tid == 0) {
        sh.base = *(volatile unsigned*)a.ctl;
        sh.abort = 0;
        for (int s = 0; s < NS; ++s) {
            mbar_init(smem_u32(&sh.full[s]), 1);
            mbar_init(smem_u32(&sh.empty[s]), MG_W / 2);
        }
        for (int j = 0; j < MG_IPC; ++j) mbar_init(smem_u32(&sh.kvbar[j]), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (tid < a.T) {
        int p = a.seq_len[a.tok_seq[tid]];
        if (p >= a.max_pos) {
            if (c == 0) a.status[ST_CTX] = 1;
            p = a.max_pos - 1;
        }
        sh.pos[tid] = p;
        const int id = a.tokens[tid];
        if (c == 0 && (id < 0 || id >= a.V)) a.status[ST_TOKEN] = 1;
    }
    __syncthreads();
    const unsigned base = sh.base;

    if (c >= a.NG) {
        // ================= attention CTA
        if (warp == 9) return;
        const int ai = c - a.NG;
        const int items = a.T << a.lg_nkv;
        int8_t* att = (int8_t*)smem;
        const size_t ist = 2 * (size_t)a.cap * D + step_aux_bytes(D, a.mbs);   // item region stride
        unsigned char* scr = (unsigned char*)(att + (size_t)a.ipc * ist);
        for (int l = -1; l < a.L; ++l) {
            for (int j = 0; j < a.ipc; ++j) {
                const int it = ai + j * a.NA;
                if (it >= items) break;
                const int t = it >> a.lg_nkv, g = it & ((1 << a.lg_nkv) - 1);
                const bool staged = sh.pos[t] + 1 <= a.cap;
                int8_t* Ks = att + (size_t)j * ist;
                int8_t* Vs = Ks + (size_t)a.cap * D;
                unsigned char* aux = (unsigned char*)(Vs + (size_t)a.cap * D);
                const uint32_t kvb = smem_u32(&sh.kvbar[j]);
                if (l >= 0) mg_attention<EPL, G>(a, sh, a.layers[l], l, t, g, Ks, Vs, aux, staged, kvb, scr);
                // this item's next layer (the region is free again)
                if (tid == 0 && l + 1 < a.L) mg_stage<D>(a, sh, a.layers[l + 1], t, g, Ks, Vs, aux, staged, kvb);
            }
        }
        return;
    }

    // ================= GEMV CTA
    unsigned char* ring = smem;
    if (warp == 8) {
        mg_produce(a, sh, ring, c);
        return;
    }
    const int nqkv = (a.nq + 2 * a.nkv) * a.d;
    const int Kmax = max(max(a.H, a.nq * a.d), a.F);
    const int XP = Kmax + 16;
    int8_t* x8 = (int8_t*)(smem + a.off_x8);
    int32_t* xin = (int32_t*)(smem + a.off_xin);
    int16_t* gs = (int16_t*)(smem + a.off_gs);           // [H]
    int32_t* hown = (int32_t*)(smem + a.off_hown);
    StepLayer* lay = (StepLayer*)(smem + a.off_lay);
    int32_t* mct = (int32_t*)(smem + a.off_mct);
    // ---- everything small the phases read, staged once per step (a global
    // read of a small parameter under the weight stream can cost a microsecond
    // or two on the critical path): this CTA's row bounds per GEMV kind, the
    // layer table, and by asynchronous copies every phase's channel scales of
    // this CTA's rows
    if (tid < 10) sh.rw[tid >> 1][tid & 1] = a.rows[(tid >> 1) * (a.NG + 1) + c + (tid & 1)];
    if (warp < 8)                                         // threads 0..255 (warp 8 has left)
        for (int i = tid; i < a.L * (int)(sizeof(StepLayer) / 8); i += 256)
            ((u64*)lay)[i] = ((const u64*)a.layers)[i];
    bar_named(MG_BAR_INIT, 288);
    if (warp < 8) {
        for (int l = 0; l < a.L; ++l)
            for (int k = 0, off = l * a.ms; k < 4; ++k) {
                const int32_t* m = k == 0 ? lay[l].m_qkv : k == 1 ? lay[l].m_o : k == 2 ? lay[l].m_gu : lay[l].m_d;
                const int r0 = sh.rw[k][0], n = sh.rw[k][1] - r0;
                for (int i = tid; i < n; i += 256) cp_async4(mct + off + i, m + r0 + i);
                off += n;
            }
        const int r0 = sh.rw[MG_K_LM][0], n = sh.rw[MG_K_LM][1] - r0;
        for (int i = tid; i < n; i += 256) cp_async4(mct + a.L * a.ms + i, a.embed_m + r0 + i);
    }
    // the residual rows this CTA updates (o_proj and down share the rows), from the embedding
    const int h0 = sh.rw[MG_K_O][0], h1 = sh.rw[MG_K_O][1];
    if (warp < 8) {
        for (int e = tid; e < a.T * STEP_HOWN; e += 256) {
            const int t = e / STEP_HOWN, n = h0 + (e - t * STEP_HOWN);
            if (n < h1) {
                const int id = mg_token_id(a, t);
                hown[e] = (int)rshr((i64)a.embed[(size_t)id * a.H + n] * (i64)a.embed_m[id], 6);
            }
        }
    }
    int u = 0;
    bool first = true;
    int bestv = -2147483647 - 1, besti = 2147483647;
    for (int l = 0; l <= a.L; ++l) {
        const StepLayer& Lw = lay[l < a.L ? l : 0];
        const int nph = l < a.L ? 4 : 1;
        int moff = l * a.ms;                              // this layer's channel scales in mct
        for (int p = 0; p < nph; ++p) {
            MgPhase P{};
            P.kind = l < a.L ? p : MG_K_LM;
            switch (P.kind) {
                case MG_K_QKV:
                    P.K = a.H; P.N = nqkv; P.mc = Lw.m_qkv; P.gamma = Lw.attn_gamma;
                    P.src = l ? a.xh : nullptr; P.tin = base + 5 * (l - 1) + 4;
                    P.dst = a.xqkv; P.ldo = nqkv; P.fout = 12; P.tout = base + 5 * l;
                    break;
                case MG_K_O:
                    P.K = a.nq * a.d; P.N = a.H; P.mc = Lw.m_o; P.F_in = 12;
                    P.src = a.xo; P.tin = base + 5 * l + 1;
                    P.dst = a.xh; P.ldo = a.H; P.fout = 16; P.tout = base + 5 * l + 2;
                    break;
                case MG_K_GU:
                    P.K = a.H; P.N = 2 * a.F; P.mc = Lw.m_gu; P.gamma = Lw.ffn_gamma;
                    P.src = a.xh; P.tin = base + 5 * l + 2;
                    P.dst = a.xs; P.ldo = a.F; P.fout = 12; P.tout = base + 5 * l + 3;
                    break;
                case MG_K_D:
                    P.K = a.F; P.N = a.H; P.mc = Lw.m_d; P.F_in = 10;
                    P.src = a.xs; P.tin = base + 5 * l + 3;
                    P.dst = a.xh; P.ldo = a.H; P.fout = 16; P.tout = base + 5 * l + 4;
                    break;
                default:
                    P.K = a.H; P.N = a.V; P.mc = a.embed_m; P.gamma = a.final_gamma;
                    P.src = a.L ? a.xh : nullptr; P.tin = base + 5 * (a.L - 1) + 4;
                    P.fout = 16;
                    break;
            }
            P.r0 = sh.rw[P.kind][0];
            P.r1 = sh.rw[P.kind][1];
            if (warp == 9) {
                mg_scales(a, sh, P);
                continue;
            }
            const int32_t* mcs = mct + (P.kind == MG_K_LM ? a.L * a.ms : moff);
            moff += P.r1 - P.r0;
            // the scale table has landed (each thread its own copies; the
            // prologue's statistics barrier then publishes them to all)
            if (first) { cp_async_wait_all(); first = false; }
            mg_prologue(a, sh, P, x8, XP, xin, gs);
            mg_consume(a, sh, P, ring, x8, XP, hown, mcs, u, bestv, besti);
        }
    }
    if (warp == 9) return;
    // ---- lm_head argmax partials: lanes t and 16 + t hold token t's best of
    // their rows; per warp, then per CTA (ties to the lower id)
    {
        const int v = __shfl_down_sync(0xffffffffu, bestv, 16), i = __shfl_down_sync(0xffffffffu, besti, 16);
        if (v > bestv || (v == bestv && i < besti)) { bestv = v; besti = i; }
    }
    if (lane < 8) { sh.bv[warp][lane] = bestv; sh.bi[warp][lane] = besti; }
    bar_named(MG_BAR_END, 256);
    const unsigned tfin = base + 5 * a.L;
    if (tid < a.T) {
        int bv = sh.bv[0][tid], bi = sh.bi[0][tid];
        for (int w = 1; w < MG_W; ++w) {
            const int v = sh.bv[w][tid], i = sh.bi[w][tid];
            if (v > bv || (v == bv && i < bi)) { bv = v; bi = i; }
        }
        ll_put(a.xpart + ((size_t)c * 8 + tid) * 2, bv, tfin);
        ll_put(a.xpart + ((size_t)c * 8 + tid) * 2 + 1, bi, tfin);
    }
    if (c != 0) return;
    // ---- CTA 0: the final argmax of every row, sequence lengths, next base tag
    if (warp < a.T) {
        const int t = warp;
        const unsigned want = a.stall ? tfin + 1 : tfin;
        const int bound = a.stall ? a.stall : a.spin;
        int bv = -2147483647 - 1, bi = 2147483647;
        unsigned got = 0;                       // partials q = lane + 32 j received
        for (int it = 0;; ++it) {
            bool all = true;
            for (int j = 0; lane + 32 * j < a.NG; ++j) {
                if ((got >> j) & 1u) continue;
                u64 w0, w1;
                ll_get2(a.xpart + ((size_t)(lane + 32 * j) * 8 + t) * 2, w0, w1);
                if (ll_tag(w0) == want && ll_tag(w1) == want) {
                    const int v = ll_val(w0), i = ll_val(w1);
                    if (v > bv || (v == bv && i < bi)) { bv = v; bi = i; }
                    got |= 1u << j;
                } else {
                    all = false;
                }
            }
            if (all) break;
            if (it >= bound || mg_aborted(a, sh, it)) {
                if (!sh.abort) mg_timeout(a, sh);
                break;
            }
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            const int v = __shfl_xor_sync(0xffffffffu, bv, o);
            const int i = __shfl_xor_sync(0xffffffffu, bi, o);
            if (v > bv || (v == bv && i < bi)) { bv = v; bi = i; }
        }
        if (lane == 0) {
            a.next_tok[t] = bi;
            a.seq_len[a.tok_seq[t]] += 1;
        }
    }
    bar_named(MG_BAR_END, 256);
    if (tid == 0) *(volatile unsigned*)a.ctl = base + 5 * a.L + 1;
}

}  // namespace detint
