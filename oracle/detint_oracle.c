/*
 * detint CPU oracle: a plain, slow, scalar-int64 implementation of the
 * integer-only decoder forward pass.
 *
 * TEST INFRASTRUCTURE ONLY. This file defines the expected bits that the
 * CUDA library must reproduce. Only the tests, the package's smoke check and
 * the benchmark's CPU-baseline leg may load it; the product path never does.
 * It shares no code, header, table or helper with the CUDA path: both read
 * the same artifact file and implement the same written arithmetic.
 *
 * Sources (cited by page title and section):
 *   [README]  "DetLLM — Fully Deterministic LLM Inference" (GitHub README):
 *             intro (int32 logits, exact integer arithmetic), "Layout"
 *             (intmath, dyadic, DI-Exp/Softmax/RMSNorm/SwiGLU, int RoPE).
 *   [BLOG]    "Eliminating Nondeterminism in LLM Inference with Integer-Only
 *             Arithmetic" (DetLLM blog): section "DetLLM" (dyadic scales
 *             m/2^k, per-token activation quantisation, fixed K/V scales,
 *             int16 RoPE tables, tie-low argmax) and its footnote on QK^T
 *             error attribution (per-channel key rescale with inverse query
 *             scale, 15-bit probabilities, P.V as two int8 GEMMs).
 *   [BITEXACT] BitExact LLM post, "Fix the arithmetic, not just the random
 *             seed" (scales, rounding, tables and bounds must be specified).
 * Where the pages leave a step open the readings are the ones frozen in the
 * arithmetic specification shipped with this repository.
 *
 * Bounds: every quoted bound is checked with CHECK(); a violation is recorded
 * (first message kept) and reported through or_error_count()/or_last_error().
 *
 * Parity pins: every function here is pinned by tests against closed forms,
 * float64 restatements of the real-valued operation, library routines or
 * brute force; none is "parity unpinned".
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef int64_t i64;
typedef uint64_t u64;

/* ------------------------------------------------------------------ errors */
static int g_err_count = 0;
static char g_err_msg[256] = "";

static void record_error(const char* what, const char* file, int line) {
#ifdef _OPENMP
#pragma omp critical(or_err)
#endif
    {
        if (g_err_count == 0)
            snprintf(g_err_msg, sizeof g_err_msg, "%s:%d: bound violated: %s", file, line, what);
        g_err_count++;
    }
}
#define CHECK(c) do { if (!(c)) record_error(#c, __FILE__, __LINE__); } while (0)

int or_error_count(void) { return g_err_count; }
const char* or_last_error(void) { return g_err_msg; }
void or_clear_error(void) { g_err_count = 0; g_err_msg[0] = 0; }

void or_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int or_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* -------------------------------------------------------------- primitives */
#define P2(s) ((i64)1 << (s))

/* number of binary digits of x >= 0 */
static int bitlen(u64 x) {
    int n = 0;
    while (x) { n++; x >>= 1; }
    return n;
}

/* floor(x / 2^s), written without relying on the sign behaviour of >> */
static i64 floor_pow2(i64 x, int s) {
    if (x >= 0) return x >> s;
    return -(((-x) + (P2(s) - 1)) >> s);
}

/* rshr: x / 2^s rounded to nearest, ties toward +infinity ([README] "Layout":
 * intmath freezes one rounding rule; [BLOG] "DetLLM": a fixed rounding rule) */
i64 or_rshr(i64 x, int s) {
    CHECK(s >= 0 && s <= 62);
    if (s <= 0) return x;
    CHECK(x < P2(62) && x > -P2(62));
    return floor_pow2(x + P2(s - 1), s);
}

/* floor division of non-negative integers */
static u64 fdiv(u64 n, u64 d) {
    CHECK(d >= 1);
    return n / d;
}

/* largest r with r*r <= n (binary search: obviously correct) */
u64 or_isqrt(u64 n) {
    u64 lo = 0, hi = 1ull << 32;  /* r < 2^32 for n < 2^64 */
    while (hi - lo > 1) {
        u64 mid = lo + (hi - lo) / 2;
        if (mid * mid <= n && mid <= 0xFFFFFFFFull) lo = mid; else hi = mid;
    }
    return lo;
}

static i64 sat(i64 x, i64 b) { return x > b ? b : (x < -b ? -b : x); }
static i64 sat32(i64 x) { return sat(x, 2147483647LL); }

/* dyadic(N, D): (m, k) with m = N*2^k/D rounded (ties up), k the unique
 * integer with 2^14 <= N*2^k/D < 2^15 ([BLOG] "DetLLM": every tensor carries
 * a scale m/2^k). */
void or_dyadic(i64 N, i64 D, int32_t* m_out, int32_t* k_out) {
    CHECK(N >= 1 && D >= 1);
    CHECK(N < P2(50) && D < P2(50));
    /* find k: compare N*2^k with D*2^14 and D*2^15 exactly */
    int k = 14 + bitlen((u64)D) - bitlen((u64)N);   /* within 1 of the answer */
    for (;;) {
        /* want 2^14 D <= N 2^k < 2^15 D */
        u64 lhs, lo, hi;
        if (k >= 0) { lhs = (u64)N << k; lo = (u64)D << 14; hi = (u64)D << 15; }
        else        { lhs = (u64)N;      lo = (u64)D << (14 - k); hi = (u64)D << (15 - k); }
        if (lhs < lo) { k++; continue; }
        if (lhs >= hi) { k--; continue; }
        break;
    }
    i64 m;
    if (k >= 0) {
        CHECK(k <= 40);
        m = (i64)fdiv(((u64)N << (k + 1)) + (u64)D, 2 * (u64)D);
    } else {
        CHECK(-k <= 40);
        u64 dd = (u64)D << (-k);
        m = (i64)fdiv(2 * (u64)N + dd, 2 * dd);
    }
    CHECK(m >= P2(14) && m <= P2(15));
    *m_out = (int32_t)m;
    *k_out = k;
}

/* exp2q(delta): 2^(delta/1024) in Q15 for delta <= 0 ([README] "Layout":
 * DI-Exp, a shift-based integer exp). Fraction part by the cubic
 * 1 + x(A + x(B + C x))/2^15 on [0, 1) in Horner form with a rounding shift
 * after each step; integer part by a right shift. */
#define EXP2_A 22787
#define EXP2_B 7419
#define EXP2_C 2562
i64 or_exp2q(i64 delta) {
    CHECK(delta <= 0);
    i64 ip = floor_pow2(delta, 10);
    i64 f = delta - ip * 1024;
    CHECK(f >= 0 && f < 1024);
    i64 inner = EXP2_B + or_rshr(EXP2_C * f, 10);
    i64 mid = EXP2_A + or_rshr(f * inner, 10);
    i64 p2 = P2(15) + or_rshr(f * mid, 10);
    CHECK(p2 >= P2(15) && p2 < P2(16));
    if (-ip >= 24) return 0;
    return or_rshr(p2, (int)(-ip));
}

/* ------------------------------------------------------------ quantisers */

/* R = floor(127 * 2^(e+16) / a) with e = bitlen(a) */
static i64 quant_mult(i64 a, int* e_out) {
    int e = bitlen((u64)a);
    CHECK(e + 16 <= 56);
    i64 R = (i64)fdiv((u64)127 << (e + 16), (u64)a);
    CHECK(R <= 127 * P2(17));
    *e_out = e;
    return R;
}

/* ActQuant(x, F): per-token symmetric int8 quantisation of one row from its
 * own maximum ([BLOG] "DetLLM": each token's activation is quantised from
 * that token's own values, so its bits cannot depend on the batch). */
int or_actquant(const int32_t* x, int n, int F, int8_t* q, int32_t* mt, int32_t* kt) {
    i64 a = 0;
    for (int i = 0; i < n; i++) { i64 v = x[i] < 0 ? -(i64)x[i] : x[i]; if (v > a) a = v; }
    if (a == 0) {
        for (int i = 0; i < n; i++) q[i] = 0;
        *mt = 0; *kt = 0;
        return 0;
    }
    int e;
    i64 R = quant_mult(a, &e);
    for (int i = 0; i < n; i++) {
        i64 p = (i64)x[i] * R;
        i64 v = or_rshr(p, e + 16);
        CHECK(v >= -127 && v <= 127);
        q[i] = (int8_t)v;
    }
    int32_t m, k;
    or_dyadic(a, 127, &m, &k);
    *mt = m; *kt = k + F;
    return 0;
}

/* shared first half of the integer RMSNorm: normalise the row width and
 * return x' (magnitude-truncated to 24 bits) and r = isqrt(mean x'^2 + eps) */
static int rms_core(const int32_t* x, int n, i64 eps, i64* xp, i64* r_out) {
    i64 ax = 0;
    for (int i = 0; i < n; i++) { i64 v = x[i] < 0 ? -(i64)x[i] : x[i]; if (v > ax) ax = v; }
    if (ax == 0) return 0;
    int sig = bitlen((u64)ax) - 24;
    for (int i = 0; i < n; i++) {
        i64 v = x[i];
        if (sig >= 0) xp[i] = v < 0 ? -((-v) >> sig) : (v >> sig);
        else xp[i] = v * P2(-sig);
        CHECK(xp[i] < P2(24) && xp[i] > -P2(24));
    }
    int lg = bitlen((u64)n) - 1;
    CHECK(P2(lg) == n);
    i64 ss = 0;
    for (int i = 0; i < n; i++) ss += xp[i] * xp[i];
    CHECK(ss >= 0 && ss < P2(62));
    i64 eps_s;
    if (sig >= 0) eps_s = (2 * sig >= 62) ? 0 : (eps >> (2 * sig));
    else { CHECK(-2 * sig <= 48); eps_s = eps * P2(-2 * sig); }
    i64 ms = (ss >> lg) + eps_s;
    CHECK(ms >= 1 && ms < P2(62));
    *r_out = (i64)or_isqrt((u64)ms);
    CHECK(*r_out >= 1);
    return 1;
}

/* NormQuant: integer RMSNorm fused with per-token quantisation ([README]
 * "Layout": DI-RMSNorm). The real output x*gamma/rms enters only through the
 * ratio to its own maximum, so the division by the RMS lands in the scale. */
int or_normquant(const int32_t* x, int n, const int16_t* gamma, i64 eps,
                 int8_t* q, int32_t* mt, int32_t* kt) {
    i64* xp = (i64*)malloc(sizeof(i64) * (size_t)n);
    i64 r;
    if (!rms_core(x, n, eps, xp, &r)) {
        for (int i = 0; i < n; i++) q[i] = 0;
        *mt = 0; *kt = 0;
        free(xp);
        return 0;
    }
    i64 a = 0;
    for (int i = 0; i < n; i++) {
        xp[i] = xp[i] * (i64)gamma[i];      /* z_i, |z| < 2^37 */
        i64 v = xp[i] < 0 ? -xp[i] : xp[i];
        if (v > a) a = v;
    }
    CHECK(a >= 1 && a < P2(37));
    int e;
    i64 R = quant_mult(a, &e);
    for (int i = 0; i < n; i++) {
        i64 v = or_rshr(xp[i] * R, e + 16);
        CHECK(v >= -127 && v <= 127);
        q[i] = (int8_t)v;
    }
    int32_t m, k;
    or_dyadic(a, 127 * r, &m, &k);
    *mt = m; *kt = k + 12;
    free(xp);
    return 0;
}

/* QKNorm: integer RMSNorm of one head, output Q14 ([BLOG] footnote on QK^T:
 * the keys are examined after QK-Norm and RoPE, the Qwen3 order) */
int or_qknorm(const int32_t* x, int n, const int16_t* gamma, i64 eps, int32_t* y) {
    i64* xp = (i64*)malloc(sizeof(i64) * (size_t)n);
    i64 r;
    if (!rms_core(x, n, eps, xp, &r)) {
        for (int i = 0; i < n; i++) y[i] = 0;
        free(xp);
        return 0;
    }
    int bl = bitlen((u64)r);
    i64 Rr = (i64)fdiv((u64)1 << (bl + 23), (u64)r);
    CHECK(Rr <= P2(24));
    for (int i = 0; i < n; i++) {
        i64 z = xp[i] * (i64)gamma[i];
        i64 v = or_rshr(z * Rr, bl + 21);
        CHECK(v < P2(31) && v > -P2(31));
        y[i] = (int32_t)v;
    }
    free(xp);
    return 0;
}

/* RoPE with the artifact's int16 Q14 tables, rotate-half pairing ([BLOG]
 * "DetLLM": RoPE uses precomputed int16 sine and cosine tables) */
void or_rope(int32_t* y, int d, const int16_t* c, const int16_t* s) {
    int h = d / 2;
    for (int i = 0; i < h; i++) {
        i64 a = y[i], b = y[i + h];
        i64 ya = or_rshr(a * c[i] - b * s[i], 14);
        i64 yb = or_rshr(b * c[i] + a * s[i], 14);
        CHECK(ya < P2(31) && ya > -P2(31) && yb < P2(31) && yb > -P2(31));
        y[i] = (int32_t)ya;
        y[i + h] = (int32_t)yb;
    }
}

/* GEMM requantisation: one int64 multiply and one rounding shift ([BLOG]
 * "DetLLM": rescaling is one integer multiply and one shift) */
i64 or_requant(i64 acc, int32_t mt, int32_t kt, int32_t mc, int Fout) {
    i64 M = (i64)mt * (i64)mc;
    CHECK(M >= 0 && M < P2(31));
    CHECK(acc < P2(31) && acc > -P2(31));
    return or_rshr(acc * M, kt + 22 - Fout);
}

/* GEMM requantisation for 16-bit weights (the exact mode of the BitExact
 * post, "Three execution paths": wide weights against fixed-point
 * activations): the int64 accumulator times m_t m_c as one exact 128-bit
 * product, then one rounding shift; the weight scale is m_c / 2^30 */
i64 or_requant_wide(i64 acc, int32_t mt, int32_t kt, int32_t mc, int Fout) {
    const i64 M = (i64)mt * (i64)mc;
    CHECK(M >= 0 && M < P2(31));
    CHECK(acc < P2(36) && acc > -P2(36));
    const int s = kt + 30 - Fout;
    CHECK(s >= 1 && s <= 100);
    const __int128 p = (__int128)acc * (__int128)M;
    /* floor((p + 2^(s-1)) / 2^s) without relying on the sign behaviour of >> */
    const __int128 q = p + ((__int128)1 << (s - 1));
    const __int128 one = (__int128)1 << s;
    __int128 f = q >= 0 ? q / one : -((-q + one - 1) / one);
    CHECK(f < (__int128)P2(62) && f > -(__int128)P2(62));
    return (i64)f;
}

/* SwiGLU of one channel ([README] "Layout": DI-SwiGLU) */
int32_t or_swiglu(int32_t g, int32_t u) {
    CHECK(g <= (1 << 24) && g >= -(1 << 24) && u <= (1 << 24) && u >= -(1 << 24));
    i64 ag = g < 0 ? -(i64)g : g;
    i64 z = or_rshr(ag * 47274, 17);
    i64 Ez = or_exp2q(-z);
    i64 D = P2(15) + Ez;
    i64 sp = (i64)fdiv((u64)P2(31) + (u64)D, 2 * (u64)D);
    i64 sg = g >= 0 ? sp : P2(15) - sp;
    i64 silu = or_rshr((i64)g * sg, 15);
    i64 prod = silu * (i64)u;
    CHECK(prod < P2(49) && prod > -P2(49));
    return (int32_t)sat32(or_rshr(prod, 14));
}

/* brute-force int8 x int8 -> int32 GEMM: C[m][n] = sum_k A[m][k] * B[n][k]
 * ([README] "Layout": int_gemm, the only hardware-dispatched operation) */
void or_gemm_i8(const int8_t* A, const int8_t* B, int32_t* C, int M, int N, int K) {
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (int m = 0; m < M; m++)
        for (int n = 0; n < N; n++) {
            int32_t acc = 0;
            const int8_t* a = A + (size_t)m * K;
            const int8_t* b = B + (size_t)n * K;
            for (int k = 0; k < K; k++) acc += (int32_t)a[k] * (int32_t)b[k];
            C[(size_t)m * N + n] = acc;
        }
}

/* Attention for one query against ctx cached keys/values of its kv head
 * ([BLOG] footnote on QK^T: 15-bit probabilities, P.V exact; [README]
 * "Layout": DI-Softmax). kvp = KQM,KQS,VQM,VQS,MV,KV,CSTM,CSTK,e[...].
 * K8, V8: [ctx][d]. o: [d] Q12. P (optional): div-rounded probabilities Q15.
 */
int or_attention_row(const int8_t* q8, int32_t mq, int32_t kq, const int8_t* K8,
                     const int8_t* V8, int ctx, int d, const int32_t* kvp, int32_t* o,
                     int32_t* P, i64* sigma_out) {
    CHECK(ctx >= 1 && ctx <= (1 << 14));
    i64* u = (i64*)malloc(sizeof(i64) * (size_t)ctx);
    i64 CSTM = kvp[6], CSTK = kvp[7], MV = kvp[4], KVs = kvp[5];
    i64 umax = 0;
    for (int j = 0; j < ctx; j++) {
        i64 S = 0;
        for (int c = 0; c < d; c++) S += (i64)q8[c] * (i64)K8[(size_t)j * d + c];
        CHECK(S < P2(21) && S > -P2(21));
        u[j] = or_rshr(S * (i64)mq * CSTM, (int)(kq + CSTK - 10));
        if (j == 0 || u[j] > umax) umax = u[j];
    }
    i64 sigma = 0;
    for (int j = 0; j < ctx; j++) {
        i64 E = or_exp2q(u[j] - umax);
        if (E > P2(15) - 1) E = P2(15) - 1;
        u[j] = E;
        sigma += E;
    }
    CHECK(sigma >= P2(15) - 1);
    int bl = bitlen((u64)sigma);
    i64 RS = (i64)fdiv((u64)1 << (bl + 23), (u64)sigma);
    for (int c = 0; c < d; c++) {
        i64 num = 0;
        for (int j = 0; j < ctx; j++) num += u[j] * (i64)V8[(size_t)j * d + c];
        i64 t = or_rshr(num * RS, bl + 7);
        i64 ov = or_rshr(t * MV, (int)(KVs + 16 - 12));
        CHECK(ov < P2(31) && ov > -P2(31));
        o[c] = (int32_t)ov;
    }
    if (P)
        for (int j = 0; j < ctx; j++)
            P[j] = (int32_t)fdiv((u64)(u[j] * 2 * P2(15)) + (u64)sigma, 2 * (u64)sigma);
    if (sigma_out) *sigma_out = sigma;
    free(u);
    return 0;
}

/* argmax with ties to the lowest index ([BLOG] "DetLLM") */
int or_argmax(const int32_t* x, int n) {
    int best = 0;
    for (int i = 1; i < n; i++) if (x[i] > x[best]) best = i;
    return best;
}

/* ------------------------------------------------------- integer sampling */
/* Next-token draw from one logits row: temperature, top-k, top-p and one
 * draw by cumulative integer weights, all in integers ([BITEXACT] "Fix the
 * arithmetic, not just the random seed" and "Reproducibility has a cost":
 * integer sampling rules, deterministic sampling). The pages give no
 * algorithm; the steps follow the reading written in the arithmetic
 * specification (section "Integer sampling"), in that order. */

/* the (counter+1)-th output of SplitMix64 seeded with `seed` (Steele, Lea
 * and Flood, "Fast splittable pseudorandom number generators", 2014) */
uint64_t or_splitmix64(uint64_t seed, uint64_t counter) {
    uint64_t z = seed + (counter + 1) * 0x9E3779B97F4A7C15ULL;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

static const int32_t* g_sort_keys;   /* qsort has no context argument */
static int cmp_logit_desc(const void* a, const void* b) {
    const int ia = *(const int*)a, ib = *(const int*)b;
    const int32_t la = g_sort_keys[ia], lb = g_sort_keys[ib];
    if (la != lb) return la > lb ? -1 : 1;
    return ia < ib ? -1 : (ia > ib ? 1 : 0);
}

/* steps 1-5: the kept set K2 (keep_out), every weight E_i and S = sum over
 * K2; returns |K2| */
int or_sample_set(const int32_t* logits, int n, int32_t inv_temp, int32_t top_k, int32_t top_p,
                  char* keep_out, i64* E_out, i64* S_out) {
    CHECK(n >= 1);
    CHECK(inv_temp >= 0 && inv_temp <= (1 << 20));
    CHECK(top_p >= 1 && top_p <= 65536);
    if (n < 1) { *S_out = 0; return 0; }
    i64* u = (i64*)malloc(sizeof(i64) * (size_t)n);
    int* order = (int*)malloc(sizeof(int) * (size_t)n);
    /* 1. base-2 logits in Q10 at the temperature */
    for (int i = 0; i < n; i++) {
        const i64 a = or_rshr((i64)logits[i] * 47274, 21);
        u[i] = or_rshr(a * inv_temp, 16);
    }
    /* 2. weights relative to the maximum */
    i64 M = u[0];
    for (int i = 1; i < n; i++) if (u[i] > M) M = u[i];
    for (int i = 0; i < n; i++) E_out[i] = or_exp2q(u[i] - M);
    /* 3. logits descending, ties by index */
    for (int i = 0; i < n; i++) order[i] = i;
    g_sort_keys = logits;
    qsort(order, (size_t)n, sizeof(int), cmp_logit_desc);
    /* 4. top-k */
    const int k1 = (top_k > 0 && top_k < n) ? top_k : n;
    i64 S1 = 0;
    for (int j = 0; j < k1; j++) S1 += E_out[order[j]];
    /* 5. top-p: shortest prefix reaching top_p / 65536 of S1, boundary ties kept */
    int k2 = k1;
    if (top_p < 65536) {
        i64 P = 0;
        int L = 0;
        while (L < k1) {
            P += E_out[order[L]];
            L++;
            if ((__int128)P * 65536 >= (__int128)top_p * S1) break;
        }
        const i64 dstar = u[order[L - 1]] - M;
        k2 = L;
        while (k2 < k1 && u[order[k2]] - M >= dstar) k2++;
    }
    i64 S = 0;
    memset(keep_out, 0, (size_t)n);
    for (int j = 0; j < k2; j++) { keep_out[order[j]] = 1; S += E_out[order[j]]; }
    CHECK(S >= 32768);
    *S_out = S;
    free(u); free(order);
    return k2;
}

/* steps 1-7: the sampled token */
int or_sample(const int32_t* logits, int n, int32_t inv_temp, int32_t top_k, int32_t top_p,
              uint64_t seed, uint64_t counter) {
    if (n < 1) { CHECK(n >= 1); return -1; }
    char* keep = (char*)malloc((size_t)n);
    i64* E = (i64*)malloc(sizeof(i64) * (size_t)n);
    i64 S = 0;
    or_sample_set(logits, n, inv_temp, top_k, top_p, keep, E, &S);
    /* 6-7. one draw by cumulative weights in index order */
    const uint64_t r = or_splitmix64(seed, counter);
    const i64 t = (i64)(((unsigned __int128)r * (unsigned __int128)(u64)S) >> 64);
    int tok = -1;
    i64 cum = 0;
    for (int i = 0; i < n; i++) {
        if (!keep[i]) continue;
        cum += E[i];
        if (cum > t) { tok = i; break; }
    }
    CHECK(tok >= 0);
    free(keep);
    free(E);
    return tok;
}

/* ------------------------------------------------------------- the model */
/* weight matrices are int8 (wbits 8) or int16 (wbits 16, the exact mode);
 * the pointers below address either, by the model's wbits */
typedef struct {
    const int16_t *attn_gamma, *ffn_gamma, *q_gamma, *k_gamma;
    const void* w_qkv; const int32_t* m_qkv;
    const void* w_o; const int32_t* m_o;
    const void* w_gate; const int32_t* m_gate;
    const void* w_up; const int32_t* m_up;
    const void* w_down; const int32_t* m_down;
    const int32_t* kvp;
} or_layer;

typedef struct {
    int L, H, nq, nkv, d, F, V, max_pos, qk_norm, wbits;
    i64 eps_h, eps_qk;
    const void* embed; const int32_t* embed_m; const int16_t* final_gamma;
    const int16_t *rope_cos, *rope_sin;
    or_layer* layers;
    uint8_t* blob; size_t size;
} or_model;

typedef struct {
    int len, max_ctx;
    int8_t* K;   /* [L][nkv][max_ctx][d] */
    int8_t* V;   /* [L][nkv][max_ctx][d] */
} or_seq;

static int rd32(const uint8_t* p) { int32_t v; memcpy(&v, p, 4); return v; }
static i64 rd64(const uint8_t* p) { int64_t v; memcpy(&v, p, 8); return v; }

static const void* take(or_model* m, size_t* cur, size_t bytes, int* ok) {
    *cur = (*cur + 255) & ~(size_t)255;
    if (*cur + bytes > m->size) { *ok = 0; return NULL; }
    const void* p = m->blob + *cur;
    *cur += bytes;
    return p;
}

void* or_model_load(const char* path, int* err) {
    *err = 0;
    FILE* f = fopen(path, "rb");
    if (!f) { *err = 1; return NULL; }
    fseek(f, 0, SEEK_END);
    long sz = ftell(f);
    fseek(f, 0, SEEK_SET);
    or_model* m = (or_model*)calloc(1, sizeof(or_model));
    m->size = (size_t)sz;
    m->blob = (uint8_t*)malloc(m->size);
    if (fread(m->blob, 1, m->size, f) != m->size) { fclose(f); *err = 2; free(m->blob); free(m); return NULL; }
    fclose(f);
    if (m->size < 256 || memcmp(m->blob, "DETINT01", 8) != 0 ||
        (rd32(m->blob + 8) != 1 && !(rd32(m->blob + 8) == 2 && rd32(m->blob + 72) == 16))) {
        *err = 3; free(m->blob); free(m); return NULL;
    }
    m->wbits = rd32(m->blob + 8) == 2 ? 16 : 8;
    const uint8_t* h = m->blob;
    m->L = rd32(h + 12); m->H = rd32(h + 16); m->nq = rd32(h + 20); m->nkv = rd32(h + 24);
    m->d = rd32(h + 28); m->F = rd32(h + 32); m->V = rd32(h + 36); m->max_pos = rd32(h + 40);
    m->qk_norm = rd32(h + 44); m->eps_h = rd32(h + 48); m->eps_qk = rd32(h + 52);
    (void)rd64;
    int ok = 1;
    size_t cur = 256;
    int H = m->H, d = m->d, F = m->F, V = m->V, nqkv = (m->nq + 2 * m->nkv) * d;
    const size_t wb = (size_t)m->wbits / 8;
    m->embed = take(m, &cur, (size_t)V * H * wb, &ok);
    m->embed_m = (const int32_t*)take(m, &cur, (size_t)V * 4, &ok);
    m->final_gamma = (const int16_t*)take(m, &cur, (size_t)H * 2, &ok);
    m->rope_cos = (const int16_t*)take(m, &cur, (size_t)m->max_pos * (d / 2) * 2, &ok);
    m->rope_sin = (const int16_t*)take(m, &cur, (size_t)m->max_pos * (d / 2) * 2, &ok);
    m->layers = (or_layer*)calloc((size_t)m->L, sizeof(or_layer));
    for (int l = 0; l < m->L && ok; l++) {
        or_layer* y = &m->layers[l];
        y->attn_gamma = (const int16_t*)take(m, &cur, (size_t)H * 2, &ok);
        y->ffn_gamma = (const int16_t*)take(m, &cur, (size_t)H * 2, &ok);
        y->q_gamma = (const int16_t*)take(m, &cur, (size_t)d * 2, &ok);
        y->k_gamma = (const int16_t*)take(m, &cur, (size_t)d * 2, &ok);
        y->w_qkv = take(m, &cur, (size_t)nqkv * H * wb, &ok);
        y->m_qkv = (const int32_t*)take(m, &cur, (size_t)nqkv * 4, &ok);
        y->w_o = take(m, &cur, (size_t)H * m->nq * d * wb, &ok);
        y->m_o = (const int32_t*)take(m, &cur, (size_t)H * 4, &ok);
        y->w_gate = take(m, &cur, (size_t)F * H * wb, &ok);
        y->m_gate = (const int32_t*)take(m, &cur, (size_t)F * 4, &ok);
        y->w_up = take(m, &cur, (size_t)F * H * wb, &ok);
        y->m_up = (const int32_t*)take(m, &cur, (size_t)F * 4, &ok);
        y->w_down = take(m, &cur, (size_t)H * F * wb, &ok);
        y->m_down = (const int32_t*)take(m, &cur, (size_t)H * 4, &ok);
        y->kvp = (const int32_t*)take(m, &cur, (size_t)m->nkv * (8 + d / 2) * 4, &ok);
    }
    if (!ok) { *err = 4; free(m->layers); free(m->blob); free(m); return NULL; }
    return m;
}

void or_model_free(void* p) {
    or_model* m = (or_model*)p;
    if (!m) return;
    free(m->layers); free(m->blob); free(m);
}

/* info: L, H, nq, nkv, d, F, V, max_pos, qk_norm, wbits */
void or_model_info(void* p, int32_t* info) {
    or_model* m = (or_model*)p;
    info[0] = m->L; info[1] = m->H; info[2] = m->nq; info[3] = m->nkv; info[4] = m->d;
    info[5] = m->F; info[6] = m->V; info[7] = m->max_pos; info[8] = m->qk_norm; info[9] = m->wbits;
}

void* or_seq_new(void* p, int max_ctx) {
    or_model* m = (or_model*)p;
    or_seq* s = (or_seq*)calloc(1, sizeof(or_seq));
    s->max_ctx = max_ctx;
    size_t n = (size_t)m->L * m->nkv * max_ctx * m->d;
    s->K = (int8_t*)calloc(n, 1);
    s->V = (int8_t*)calloc(n, 1);
    return s;
}

void or_seq_free(void* p) {
    or_seq* s = (or_seq*)p;
    if (!s) return;
    free(s->K); free(s->V); free(s);
}

int or_seq_len(void* p) { return ((or_seq*)p)->len; }

/* sum_k x[k] w[row][k] over a weight row of width K (int8 rows: exact in
 * int32; int16 rows: exact in int64, |sum| < 127 * 2^15 * K) */
static i64 dot_row(const or_model* m, const void* w, size_t row, int K, const int8_t* x) {
    if (m->wbits == 16) {
        const int16_t* r = (const int16_t*)w + row * (size_t)K;
        i64 acc = 0;
        for (int k = 0; k < K; k++) acc += (i64)x[k] * (i64)r[k];
        return acc;
    }
    const int8_t* r = (const int8_t*)w + row * (size_t)K;
    int32_t acc = 0;
    for (int k = 0; k < K; k++) acc += (int32_t)x[k] * (int32_t)r[k];
    return acc;
}

/* requantisation by the model's weight width (section 5 or section 15) */
static i64 requant_w(const or_model* m, i64 acc, int32_t mt, int32_t kt, int32_t mc, int Fout) {
    return m->wbits == 16 ? or_requant_wide(acc, mt, kt, mc, Fout) : or_requant(acc, mt, kt, mc, Fout);
}

/* One token through the whole decoder at position s->len; appends its K/V.
 * Writes the int32 logits (if logits != NULL) and, if hid != NULL, the
 * residual after the embedding and after every layer ([L+1][H]). */
static void forward_token(or_model* m, or_seq* s, int32_t tok, int32_t* logits, int32_t* hid) {
    const int H = m->H, d = m->d, nq = m->nq, nkv = m->nkv, F = m->F, half = d / 2;
    const int nqkv = (nq + 2 * nkv) * d, grp = nq / nkv, pos = s->len;
    const int wmax = (nq * d > F ? nq * d : F) > H ? (nq * d > F ? nq * d : F) : H;
    int32_t* h = (int32_t*)malloc(sizeof(int32_t) * H);
    int8_t* x8 = (int8_t*)malloc((size_t)wmax);
    int32_t* qkv = (int32_t*)malloc(sizeof(int32_t) * nqkv);
    int8_t* q8 = (int8_t*)malloc((size_t)nq * d);
    int32_t* mq = (int32_t*)malloc(sizeof(int32_t) * nq);
    int32_t* kq = (int32_t*)malloc(sizeof(int32_t) * nq);
    int32_t* o = (int32_t*)malloc(sizeof(int32_t) * nq * d);
    int32_t* g = (int32_t*)malloc(sizeof(int32_t) * F);
    int32_t* u = (int32_t*)malloc(sizeof(int32_t) * F);
    int32_t* sv = (int32_t*)malloc(sizeof(int32_t) * F);
    int32_t* y = (int32_t*)malloc(sizeof(int32_t) * d);
    int32_t mt, kt;
    CHECK(tok >= 0 && tok < m->V);
    CHECK(pos < s->max_ctx && pos < m->max_pos);

    /* a1 embedding: tied int8 row times its row scale, onto the Q16 grid
     * (int16 rows: scale m / 2^30) */
    for (int i = 0; i < H; i++) {
        if (m->wbits == 16)
            h[i] = (int32_t)or_rshr((i64)((const int16_t*)m->embed)[(size_t)tok * H + i] * m->embed_m[tok], 30 - 16);
        else
            h[i] = (int32_t)or_rshr((i64)((const int8_t*)m->embed)[(size_t)tok * H + i] * m->embed_m[tok], 22 - 16);
    }
    if (hid) memcpy(hid, h, sizeof(int32_t) * H);

    for (int l = 0; l < m->L; l++) {
        const or_layer* ly = &m->layers[l];
        /* a2 + a3: NormQuant, QKV GEMM, requant to Q12 */
        or_normquant(h, H, ly->attn_gamma, m->eps_h, x8, &mt, &kt);
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
        for (int n = 0; n < nqkv; n++)
            qkv[n] = (int32_t)sat32(requant_w(m, dot_row(m, ly->w_qkv, n, H, x8), mt, kt, ly->m_qkv[n], 12));
        /* a4: QK-norm, RoPE, per-channel key rescale, quantisation, cache write */
        const int16_t* cr = m->rope_cos + (size_t)pos * half;
        const int16_t* sr = m->rope_sin + (size_t)pos * half;
        for (int hq = 0; hq < nq; hq++) {
            const int32_t* kvp = ly->kvp + (size_t)(hq / grp) * (8 + half);
            int E = 0;
            for (int i = 0; i < half; i++) if (kvp[8 + i] > E) E = kvp[8 + i];
            if (m->qk_norm) or_qknorm(qkv + hq * d, d, ly->q_gamma, m->eps_qk, y);
            else for (int i = 0; i < d; i++) {
                CHECK(qkv[hq * d + i] < (1 << 29) && qkv[hq * d + i] > -(1 << 29));
                y[i] = qkv[hq * d + i] * 4;
            }
            or_rope(y, d, cr, sr);
            for (int c = 0; c < d; c++) {
                i64 v = (i64)y[c] * P2(E - kvp[8 + (c % half)]);
                CHECK(v < P2(31) && v > -P2(31));
                y[c] = (int32_t)v;
            }
            or_actquant(y, d, 14, q8 + hq * d, &mq[hq], &kq[hq]);
        }
        for (int g2 = 0; g2 < nkv; g2++) {
            const int32_t* kvp = ly->kvp + (size_t)g2 * (8 + half);
            const int32_t* kin = qkv + (nq + g2) * d;
            const int32_t* vin = qkv + (nq + nkv + g2) * d;
            int8_t* Kd = s->K + (((size_t)l * nkv + g2) * s->max_ctx + pos) * d;
            int8_t* Vd = s->V + (((size_t)l * nkv + g2) * s->max_ctx + pos) * d;
            if (m->qk_norm) or_qknorm(kin, d, ly->k_gamma, m->eps_qk, y);
            else for (int i = 0; i < d; i++) {
                CHECK(kin[i] < (1 << 29) && kin[i] > -(1 << 29));
                y[i] = kin[i] * 4;
            }
            or_rope(y, d, cr, sr);
            for (int c = 0; c < d; c++) {
                i64 v = (i64)y[c] * P2(kvp[8 + (c % half)]);
                Kd[c] = (int8_t)sat(or_rshr(v * kvp[0], kvp[1]), 127);
                Vd[c] = (int8_t)sat(or_rshr((i64)vin[c] * kvp[2], kvp[3]), 127);
            }
        }
        /* a5: attention of every q head over keys 0..pos of this sequence */
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
        for (int hq = 0; hq < nq; hq++) {
            int g2 = hq / grp;
            const int8_t* Kb = s->K + ((size_t)l * nkv + g2) * s->max_ctx * d;
            const int8_t* Vb = s->V + ((size_t)l * nkv + g2) * s->max_ctx * d;
            or_attention_row(q8 + hq * d, mq[hq], kq[hq], Kb, Vb, pos + 1, d,
                             ly->kvp + (size_t)g2 * (8 + half), o + hq * d, NULL, NULL);
        }
        /* a6: ActQuant(o), o_proj, residual add */
        or_actquant(o, nq * d, 12, x8, &mt, &kt);
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
        for (int n = 0; n < H; n++) {
            const i64 acc = dot_row(m, ly->w_o, n, nq * d, x8);
            h[n] = (int32_t)sat32((i64)h[n] + sat32(requant_w(m, acc, mt, kt, ly->m_o[n], 16)));
        }
        /* a7 + a8: NormQuant, gate/up GEMMs, SwiGLU */
        or_normquant(h, H, ly->ffn_gamma, m->eps_h, x8, &mt, &kt);
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
        for (int n = 0; n < F; n++) {
            const i64 ag = dot_row(m, ly->w_gate, n, H, x8), au = dot_row(m, ly->w_up, n, H, x8);
            g[n] = (int32_t)sat(requant_w(m, ag, mt, kt, ly->m_gate[n], 12), P2(24));
            u[n] = (int32_t)sat(requant_w(m, au, mt, kt, ly->m_up[n], 12), P2(24));
            sv[n] = or_swiglu(g[n], u[n]);
        }
        /* a9: ActQuant(s), down projection, residual add */
        or_actquant(sv, F, 10, x8, &mt, &kt);
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
        for (int n = 0; n < H; n++) {
            const i64 acc = dot_row(m, ly->w_down, n, F, x8);
            h[n] = (int32_t)sat32((i64)h[n] + sat32(requant_w(m, acc, mt, kt, ly->m_down[n], 16)));
        }
        if (hid) memcpy(hid + (size_t)(l + 1) * H, h, sizeof(int32_t) * H);
    }
    s->len = pos + 1;
    if (logits) {
        /* a10: final NormQuant, lm_head against the tied embedding, Q16 logits */
        or_normquant(h, H, m->final_gamma, m->eps_h, x8, &mt, &kt);
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
        for (int v = 0; v < m->V; v++)
            logits[v] = (int32_t)sat32(requant_w(m, dot_row(m, m->embed, v, H, x8), mt, kt, m->embed_m[v], 16));
    }
    free(h); free(x8); free(qkv); free(q8); free(mq); free(kq); free(o);
    free(g); free(u); free(sv); free(y);
}

/* Feed n tokens to a sequence in order (a prefill when n > 1, a decode step
 * when n == 1). Returns the argmax of the last token's logits and writes
 * those logits to `logits` (length V) when it is not NULL. */
int or_seq_feed(void* pm, void* ps, int n, const int32_t* tokens, int32_t* logits, int32_t* hid) {
    or_model* m = (or_model*)pm;
    or_seq* s = (or_seq*)ps;
    int32_t* lg = (int32_t*)malloc(sizeof(int32_t) * (size_t)m->V);
    for (int i = 0; i < n; i++)
        forward_token(m, s, tokens[i], i == n - 1 ? lg : NULL, i == n - 1 ? hid : NULL);
    int am = or_argmax(lg, m->V);
    if (logits) memcpy(logits, lg, sizeof(int32_t) * (size_t)m->V);
    free(lg);
    return am;
}

/* ------------------------------------------- array helpers for the tests */
void or_rshr_vec(const i64* x, const int32_t* s, i64* out, int n) {
    for (int i = 0; i < n; i++) out[i] = or_rshr(x[i], s[i]);
}
void or_exp2q_vec(const i64* delta, i64* out, int n) {
    for (int i = 0; i < n; i++) out[i] = or_exp2q(delta[i]);
}
void or_swiglu_vec(const int32_t* g, const int32_t* u, int32_t* out, int n) {
    for (int i = 0; i < n; i++) out[i] = or_swiglu(g[i], u[i]);
}
void or_isqrt_vec(const u64* x, u64* out, int n) {
    for (int i = 0; i < n; i++) out[i] = or_isqrt(x[i]);
}
void or_dyadic_vec(const i64* N, const i64* D, int32_t* m, int32_t* k, int n) {
    for (int i = 0; i < n; i++) or_dyadic(N[i], D[i], &m[i], &k[i]);
}
void or_requant_wide_vec(const i64* acc, const int32_t* mt, const int32_t* kt, const int32_t* mc,
                         int Fout, i64* out, int n) {
    for (int i = 0; i < n; i++) out[i] = or_requant_wide(acc[i], mt[i], kt[i], mc[i], Fout);
}
void or_requant_vec(const i64* acc, const int32_t* mt, const int32_t* kt, const int32_t* mc,
                    int Fout, i64* out, int n) {
    for (int i = 0; i < n; i++) out[i] = or_requant(acc[i], mt[i], kt[i], mc[i], Fout);
}
/* actquant of `rows` rows of length n */
void or_actquant_rows(const int32_t* x, int rows, int n, int F, int8_t* q, int32_t* mt, int32_t* kt) {
    for (int r = 0; r < rows; r++)
        or_actquant(x + (size_t)r * n, n, F, q + (size_t)r * n, mt + r, kt + r);
}
void or_normquant_rows(const int32_t* x, int rows, int n, const int16_t* gamma, i64 eps,
                       int8_t* q, int32_t* mt, int32_t* kt) {
    for (int r = 0; r < rows; r++)
        or_normquant(x + (size_t)r * n, n, gamma, eps, q + (size_t)r * n, mt + r, kt + r);
}
void or_qknorm_rows(const int32_t* x, int rows, int n, const int16_t* gamma, i64 eps, int32_t* y) {
    for (int r = 0; r < rows; r++)
        or_qknorm(x + (size_t)r * n, n, gamma, eps, y + (size_t)r * n);
}
