// Host launchers of the detint kernels: grid sizing, shared-memory
// attributes, programmatic dependent launch. Kernel code lives in the
// .cuh files.
#include <cudaTypedefs.h>
#include <algorithm>

#include "kernels.cuh"

namespace detint {

static size_t gemv_smem_bytes(int NT, int K) {
    return (size_t)8 * NT * (K + 64) + (size_t)8 * 16 * 8 * NT * 4;
}
constexpr size_t GEMV_SMEM_MAX = 200 * 1024;

template <int NT, int MODE>
static cudaError_t gemv_attr() {
    return cudaFuncSetAttribute(k_gemv<NT, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)GEMV_SMEM_MAX);
}

template <int NT, int MODE>
static cudaError_t gemv_launch_t(const int8_t* W, const int8_t* X, int M, int N, int K,
                                 const Epi& ep, cudaStream_t s) {
    const size_t smem = gemv_smem_bytes(NT, K);
    const int grid = (N + 15) / 16;
    k_gemv<NT, MODE><<<grid, 256, smem, s>>>(W, X, M, N, K, ep);
    return cudaGetLastError();
}

// the Epi of rows m0.. of a larger launch
static Epi epi_rows(const Epi& ep, int m0) {
    Epi e = ep;
    if (e.out) e.out += (size_t)m0 * ep.ldo;
    if (e.mt) e.mt += m0;
    if (e.kt) e.kt += m0;
    if (e.pval) e.pval += (size_t)m0 * ep.npart;
    if (e.pidx) e.pidx += (size_t)m0 * ep.npart;
    return e;
}

template <int MODE>
static cudaError_t gemv_nt(const int8_t* W, const int8_t* X, int M, int N, int K, const Epi& ep,
                           cudaStream_t s) {
    if (M <= 8) return gemv_launch_t<1, MODE>(W, X, M, N, K, ep, s);
    if (M <= 16 || gemv_smem_bytes(4, K) > GEMV_SMEM_MAX) {
        if (M <= 16) return gemv_launch_t<2, MODE>(W, X, M, N, K, ep, s);
        cudaError_t e = gemv_launch_t<2, MODE>(W, X, 16, N, K, ep, s);
        if (e != cudaSuccess) return e;
        return gemv_nt<MODE>(W, X + (size_t)16 * K, M - 16, N, K, epi_rows(ep, 16), s);
    }
    return gemv_launch_t<4, MODE>(W, X, M, N, K, ep, s);
}

cudaError_t launch_gemv(const int8_t* W, const int8_t* X, int M, int N, int K, int mode,
                        const Epi& ep, cudaStream_t s) {
    if (M < 1 || M > 32 || N < 1 || (K & 63) || K < 64) return cudaErrorInvalidValue;
    switch (mode) {
        case EPI_RAW: return gemv_nt<EPI_RAW>(W, X, M, N, K, ep, s);
        case EPI_QKV: return gemv_nt<EPI_QKV>(W, X, M, N, K, ep, s);
        case EPI_RESADD: return gemv_nt<EPI_RESADD>(W, X, M, N, K, ep, s);
        case EPI_SWIGLU: return gemv_nt<EPI_SWIGLU>(W, X, M, N, K, ep, s);
        case EPI_LOGITS: return gemv_nt<EPI_LOGITS>(W, X, M, N, K, ep, s);
    }
    return cudaErrorInvalidValue;
}


// ------------------------------------------------------------- launchers
cudaError_t launch_embed(const int32_t* tokens, int T, const int32_t* tok_seq, int32_t* tok_pos,
                         const int32_t* seq_len, int decode, int max_pos, const int8_t* E,
                         const uint8_t* Elo, const int32_t* Em, int H, int V, int32_t* h,
                         int32_t* status, cudaStream_t s) {
    k_embed<<<T, 256, 0, s>>>(tokens, tok_seq, tok_pos, seq_len, decode, max_pos, E, Elo, Em, H, V, h,
                              status);
    return cudaGetLastError();
}

static int ilog2(int n) { int l = 0; while ((1 << l) < n) ++l; return l; }

template <typename... KArgs, typename... Args>
static cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t s, Args... args);

cudaError_t launch_normquant(const int32_t* x, const int32_t* rows, int R, int n,
                             const int16_t* gamma, long long eps, int8_t* q, int32_t* mt,
                             int32_t* kt, cudaStream_t s, bool pdl) {
    if (pdl) return launch_pdl(k_normquant, dim3(R), dim3(256), 0, s, x, rows, n, ilog2(n), gamma,
                               (i64)eps, q, mt, kt);
    k_normquant<<<R, 256, 0, s>>>(x, rows, n, ilog2(n), gamma, eps, q, mt, kt);
    return cudaGetLastError();
}

cudaError_t launch_actquant(const int32_t* x, int R, int n, int F, int8_t* q, int32_t* mt,
                            int32_t* kt, cudaStream_t s, bool pdl) {
    if (pdl) return launch_pdl(k_actquant, dim3(R), dim3(256), 0, s, x, n, F, q, mt, kt);
    k_actquant<<<R, 256, 0, s>>>(x, n, F, q, mt, kt);
    return cudaGetLastError();
}

cudaError_t launch_qkv_post(const QkvPostArgs& a, cudaStream_t s) {
    dim3 grid((a.nq + a.nkv + 3) / 4, a.T);
    if (a.d == 128) k_qkv_post<4><<<grid, 128, 0, s>>>(a);
    else if (a.d == 64) k_qkv_post<2><<<grid, 128, 0, s>>>(a);
    else return cudaErrorInvalidValue;
    return cudaGetLastError();
}

using AttnFn = void (*)(AttnArgs);
static AttnFn attention_kernel(int d, int lg_grp) {
    static const AttnFn k128[4] = {k_attention<4, 1>, k_attention<4, 2>, k_attention<4, 4>, k_attention<4, 8>};
    static const AttnFn k64[4] = {k_attention<2, 1>, k_attention<2, 2>, k_attention<2, 4>, k_attention<2, 8>};
    if (lg_grp < 0 || lg_grp > 3) return nullptr;
    return d == 128 ? k128[lg_grp] : (d == 64 ? k64[lg_grp] : nullptr);
}

cudaError_t launch_attention(const AttnArgs& a, cudaStream_t s) {
    const size_t smem = attention_smem_bytes(1 << a.lg_grp, a.d, a.ctx_cap);
    dim3 grid(a.T, a.nkv);
    auto k = attention_kernel(a.d, a.lg_grp);
    if (!k) return cudaErrorInvalidValue;
    k<<<grid, 256, smem, s>>>(a);
    return cudaGetLastError();
}

// launch with programmatic stream serialization: the kernel may start while
// its predecessor drains and must griddepcontrol.wait before reading its output
template <typename... KArgs, typename... Args>
static cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t s, Args... args) {
#ifdef DETINT_NO_PDL
    kern<<<grid, block, smem, s>>>(args...);
    return cudaGetLastError();
#endif
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

cudaError_t launch_argmax_final(const int32_t* pval, const int32_t* pidx, int rows, int npart,
                                int32_t* next_tok, const int32_t* tok_seq, int32_t* seq_len,
                                cudaStream_t s, bool pdl) {
    if (pdl) return launch_pdl(k_argmax_final, dim3(rows), dim3(256), 0, s, pval, pidx, npart,
                               next_tok, tok_seq, seq_len);
    k_argmax_final<<<rows, 256, 0, s>>>(pval, pidx, npart, next_tok, tok_seq, seq_len);
    return cudaGetLastError();
}

static int g_num_sms = 0;

static size_t sgemv_smem(int K, int KC, int ns) {
    // ring + int8 activation tile + partial tiles + gamma copy + preloaded
    // residual (256 int32) + weight-channel scales (256 int32)
    return (size_t)ns * 16 * (KC + 64) + (size_t)8 * (K + 64) + (size_t)SG_GB * 8 * 16 * 8 * 4 +
           (size_t)2 * K + 2048;
}
constexpr size_t SG_SMEM_MAX = 200 * 1024;

cudaError_t launch_sgemv(const int8_t* W, int N, int K, int M, const int32_t* xin,
                         const int32_t* rows, const int16_t* gamma, long long eps, int F, int pro,
                         int mode, const Epi& ep, cudaStream_t s, const int8_t* x8,
                         const int32_t* mt, const int32_t* kt, bool pdl, int spare_sms) {
    if (M < 1 || M > 8 || N < 1 || K < 64 || (K & 63)) return cudaErrorNotSupported;
    const int KC = K <= 1024 ? K : 1024;
    if (K % KC) return cudaErrorNotSupported;
    if (pro == PRO_NORMQUANT && (K & (K - 1))) return cudaErrorNotSupported;
    // long streams (many 16-row units per CTA): two CTAs per SM, each with a
    // 4-stage ring, so one CTA's consumer latency overlaps the other's and
    // twice the bytes are in flight; short ones: one CTA per SM (the next
    // kernel's CTA takes the other slot while this one drains)
    const int G0 = (N + 15) / 16;
    const int units_per_cta = ((G0 + g_num_sms - 1) / g_num_sms) * (K / KC);
    int lg_ns = 2, cta_per_sm = 1;
    size_t smem = sgemv_smem(K, KC, 4);
    if (units_per_cta > 4) {
        if (smem <= 113 * 1024) cta_per_sm = 2;
        else if (sgemv_smem(K, KC, 8) <= SG_SMEM_MAX) { lg_ns = 3; smem = sgemv_smem(K, KC, 8); }
    }
    if (smem > SG_SMEM_MAX) return cudaErrorNotSupported;
    SgArgs a{};
    a.W = W; a.N = N; a.K = K; a.KC = KC; a.nkc = K / KC; a.M = M; a.xin = xin; a.rows = rows;
    a.gamma = gamma; a.eps = eps; a.F = F; a.pro = pro; a.mode = mode; a.ep = ep;
    a.x8 = x8; a.mt_in = mt; a.kt_in = kt; a.lg_ns = lg_ns;
    int lg = 0;
    while ((1 << lg) < K) ++lg;
    a.lg_k = lg;
    const int G = (N + 15) / 16;
    int ncta = G < g_num_sms * cta_per_sm ? G : g_num_sms * cta_per_sm;
    if (cta_per_sm == 1 && spare_sms > 0 && spare_sms < ncta) {
        // spare_sms fewer CTAs when the most row groups a CTA holds stays the
        // same: the SMs left free take all of the next kernel's CTAs, which
        // under programmatic dependent launch stage their inputs while this
        // kernel runs (freeing only some of the SMs it needs measured slower)
        const int fewer = ncta - spare_sms;
        if ((G + fewer - 1) / fewer == (G + ncta - 1) / ncta) ncta = fewer;
    }
    a.rg_q = G / ncta;
    a.rg_r = G % ncta;
    if (pro != PRO_NORMQUANT && pro != PRO_ACTQUANT && pro != PRO_NONE) return cudaErrorNotSupported;
    if (mode != EPI_QKV && mode != EPI_RESADD && mode != EPI_SWIGLU && mode != EPI_LOGITS &&
        !(mode == EPI_RAW && pro == PRO_NONE))
        return cudaErrorNotSupported;
    if (!pdl) {
        // the weights may come from the previous kernel: plain stream order
        if (cta_per_sm == 2) k_sgemv<2><<<ncta, SG_THREADS, smem, s>>>(a);
        else k_sgemv<1><<<ncta, SG_THREADS, smem, s>>>(a);
        return cudaGetLastError();
    }
    if (cta_per_sm == 2) return launch_pdl(k_sgemv<2>, dim3(ncta), dim3(SG_THREADS), smem, s, a);
    return launch_pdl(k_sgemv<1>, dim3(ncta), dim3(SG_THREADS), smem, s, a);
}

size_t attn_dec_smem(int grp, int d, int cap) { return attn_dec_smem_bytes(grp, d, cap); }

using AttnDecFn = void (*)(AttnArgs, QkvPostArgs);
// the decode attention that reads K/V from the cache (contexts beyond the
// staged kernel's shared-memory budget)
static AttnDecFn attn_dec_global_kernel(int d, int lg_grp) {
    static const AttnDecFn k128[4] = {k_attn_decode<4, 1>, k_attn_decode<4, 2>, k_attn_decode<4, 4>,
                                      k_attn_decode<4, 8>};
    static const AttnDecFn k64[4] = {k_attn_decode<2, 1>, k_attn_decode<2, 2>, k_attn_decode<2, 4>,
                                     k_attn_decode<2, 8>};
    if (lg_grp < 0 || lg_grp > 3) return nullptr;
    return d == 128 ? k128[lg_grp] : (d == 64 ? k64[lg_grp] : nullptr);
}

static AttnDecFn attn_dec_kernel(int d, int lg_grp) {
    static const AttnDecFn k128[4] = {k_attn_dec_staged<4, 1>, k_attn_dec_staged<4, 2>,
                                      k_attn_dec_staged<4, 4>, k_attn_dec_staged<4, 8>};
    static const AttnDecFn k64[4] = {k_attn_dec_staged<2, 1>, k_attn_dec_staged<2, 2>,
                                     k_attn_dec_staged<2, 4>, k_attn_dec_staged<2, 8>};
    if (lg_grp < 0 || lg_grp > 3) return nullptr;
    return d == 128 ? k128[lg_grp] : (d == 64 ? k64[lg_grp] : nullptr);
}

cudaError_t launch_attn_decode(const AttnArgs& a, const QkvPostArgs& qa, cudaStream_t s, bool staged) {
    if (staged) {
        if ((a.ctx_cap & 63) || a.ctx_cap > AD_MAXB * KV_BLK || a.lg_grp > 3) return cudaErrorInvalidValue;
        const size_t sm2 = attn_dec_smem_bytes(1 << a.lg_grp, a.d, a.ctx_cap);
        const dim3 grid(a.T, a.nkv);
        auto k = attn_dec_kernel(a.d, a.lg_grp);
        if (!k) return cudaErrorInvalidValue;
        return launch_pdl(k, grid, dim3(AD_THREADS), sm2, s, a, qa);
    }
    const size_t smem = attention_smem_bytes(1 << a.lg_grp, a.d, a.ctx_cap);
    const dim3 grid(a.T, a.nkv);
    auto k = attn_dec_global_kernel(a.d, a.lg_grp);
    if (!k) return cudaErrorInvalidValue;
    return launch_pdl(k, grid, dim3(256), smem, s, a, qa);
}

// ------------------------------------------------------------ tiled GEMM
static PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

static cudaError_t get_encode() {
    if (g_encode) return cudaSuccess;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                     cudaEnableDefault, &q);
    if (e != cudaSuccess) return e;
    if (q != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
    g_encode = (PFN_cuTensorMapEncodeTiled_v12000)fn;
    return cudaSuccess;
}

// int8 matrix [rows][K] (K % 16 == 0), 128 x 128-byte boxes, 128-byte swizzle,
// zero fill outside the matrix
static cudaError_t make_map(CUtensorMap* map, const void* base, int rows, int K, int box_rows = 128) {
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)K};
    cuuint32_t box[2] = {(cuuint32_t)GM_BK, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

using GemmFn = void (*)(CUtensorMap, CUtensorMap, int, int, int, Epi, int, int32_t*, int*);
static GemmFn gemm_kernel(int mode, int bm) {
    if (bm == 32) {
        switch (mode) {
            case EPI_RAW: return k_gemm_tma<EPI_RAW, 32>;
            case EPI_QKV: return k_gemm_tma<EPI_QKV, 32>;
            case EPI_RESADD: return k_gemm_tma<EPI_RESADD, 32>;
            case EPI_SWIGLU: return k_gemm_tma<EPI_SWIGLU, 32>;
            case EPI_LOGITS: return k_gemm_tma<EPI_LOGITS, 32>;
            default: return nullptr;
        }
    }
    if (bm == 64) {
        switch (mode) {
            case EPI_RAW: return k_gemm_tma<EPI_RAW, 64>;
            case EPI_QKV: return k_gemm_tma<EPI_QKV, 64>;
            case EPI_RESADD: return k_gemm_tma<EPI_RESADD, 64>;
            case EPI_SWIGLU: return k_gemm_tma<EPI_SWIGLU, 64>;
            case EPI_LOGITS: return k_gemm_tma<EPI_LOGITS, 64>;
            default: return nullptr;
        }
    }
    switch (mode) {
        case EPI_RAW: return k_gemm_tma<EPI_RAW, 128>;
        case EPI_QKV: return k_gemm_tma<EPI_QKV, 128>;
        case EPI_RESADD: return k_gemm_tma<EPI_RESADD, 128>;
        case EPI_SWIGLU: return k_gemm_tma<EPI_SWIGLU, 128>;
        case EPI_LOGITS: return k_gemm_tma<EPI_LOGITS, 128>;
        default: return nullptr;
    }
}

cudaError_t launch_gemm(const int8_t* A, const int8_t* W, int M, int N, int K, int mode,
                        const Epi& ep, cudaStream_t s, int32_t* wsp, size_t ws_elems, int* tcnt,
                        int tcnt_n) {
    if ((K & 15) || K < 16 || M < 1 || N < 1) return cudaErrorInvalidValue;
    if (((uintptr_t)A & 15) || ((uintptr_t)W & 15)) return cudaErrorInvalidValue;
    cudaError_t e = get_encode();
    if (e != cudaSuccess) return e;
    CUtensorMap ma, mw;
    const int BM = M <= 32 ? 32 : (M <= 64 ? 64 : 128);    // few tile rows past a short M
    e = make_map(&ma, A, M, K, BM);
    if (e == cudaSuccess) e = make_map(&mw, W, N, K);
    if (e != cudaSuccess) return e;
    const int tiles_n = (N + GM_BN - 1) / GM_BN, tiles_m = (M + BM - 1) / BM;
    const int nk = (K + GM_BK - 1) / GM_BK;
    // raw output with fewer tiles than SMs: split K over up to two CTAs per
    // SM, at least two k-tiles each, partial sums added into a zeroed C
    int splits = 1, ksl = nk;
    const int tiles = tiles_n * tiles_m;
    // under an epilogue the partial tiles go through the caller's workspace
    const bool fixup_ok = mode != EPI_RAW && wsp && tcnt && tiles <= tcnt_n;
    // as many splits as fit one wave of two CTAs per SM, each of at least 2
    // k-tiles (raw: partials added by atomics) or 4 (epilogues: partials
    // written and re-read through the workspace)
    const int min_kt = mode == EPI_RAW ? 2 : 4;
    if ((mode == EPI_RAW || fixup_ok) && g_num_sms > 0 && tiles < g_num_sms && nk >= 2 * min_kt) {
        splits = std::max(1, std::min(nk / min_kt, (2 * g_num_sms) / tiles));
        if (mode != EPI_RAW)
            splits = std::min<long long>(splits, (long long)(ws_elems / ((size_t)tiles_m * BM * N)));
        splits = std::max(splits, 1);
        ksl = (nk + splits - 1) / splits;
        splits = (nk + ksl - 1) / ksl;
        if (splits > 1 && mode == EPI_RAW) {
            e = cudaMemsetAsync(ep.out, 0, (size_t)M * ep.ldo * sizeof(int32_t), s);
            if (e != cudaSuccess) return e;
        }
    }
    const dim3 grid(tiles_n, tiles_m, splits);
    auto k = gemm_kernel(mode, BM);
    if (!k) return cudaErrorInvalidValue;
    k<<<grid, GM_THREADS, GM_SMEM, s>>>(ma, mw, M, N, K, ep, ksl, wsp, tcnt);
    return cudaGetLastError();
}

cudaError_t make_kv_maps(CUtensorMap* kmap, CUtensorMap* vmap, const int8_t* kc, const int8_t* vc,
                         long long units, int d) {
    if ((d != 64 && d != 128) || units < 1 || units * 128 > 2147483647LL) return cudaErrorInvalidValue;
    if (((uintptr_t)kc & 15) || ((uintptr_t)vc & 15)) return cudaErrorInvalidValue;
    cudaError_t e = get_encode();
    if (e != cudaSuccess) return e;
    const cuuint32_t estr[2] = {1, 1};
    // K: rows of d bytes, a 64-key box; the swizzle span equals the row
    cuuint64_t kdims[2] = {(cuuint64_t)d, (cuuint64_t)units * 64};
    cuuint64_t kstr[1] = {(cuuint64_t)d};
    cuuint32_t kbox[2] = {(cuuint32_t)d, 64};
    CUresult r = g_encode(kmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<int8_t*>(kc), kdims, kstr,
                          kbox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          d == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    // V^T: rows of 64 key bytes, a d-channel box
    cuuint64_t vdims[2] = {64, (cuuint64_t)units * d};
    cuuint64_t vstr[1] = {64};
    cuuint32_t vbox[2] = {64, (cuuint32_t)d};
    r = g_encode(vmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<int8_t*>(vc), vdims, vstr, vbox, estr,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t launch_attn_prefill(const PfArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                                int d, cudaStream_t s) {
    if (a.lg_grp > 6 || a.nqb < 1) return cudaErrorInvalidValue;
    // grid x: kv heads (fastest, so the heaviest query blocks of every head
    // start first), grid y: query blocks in chunks of at most 65535
    for (int b0 = 0; b0 < a.nqb; b0 += 65535) {
        PfArgs c = a;
        c.qblk = a.qblk + 4 * (size_t)b0;
        c.nqb = std::min(65535, a.nqb - b0);
        const dim3 grid(a.nkv, c.nqb);
        if (d == 128)
            k_attn_prefill<128><<<grid, PF_THREADS, PfCfg<128>::SMEM, s>>>(kmap, vmap, c);
        else if (d == 64)
            k_attn_prefill<64><<<grid, PF_THREADS, PfCfg<64>::SMEM, s>>>(kmap, vmap, c);
        else
            return cudaErrorInvalidValue;
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

template <int MODE>
static cudaError_t gemv_attr_all() {
    cudaError_t e = gemv_attr<1, MODE>();
    if (e == cudaSuccess) e = gemv_attr<2, MODE>();
    if (e == cudaSuccess) e = gemv_attr<4, MODE>();
    return e;
}

cudaError_t launch_split_w16(const int16_t* W, int8_t* hi, uint8_t* lo, long long n, cudaStream_t s) {
    if (n < 1) return cudaErrorInvalidValue;
    const long long per_block = 256LL * SPLIT_PER_THREAD;
    const long long blocks = (n + per_block - 1) / per_block;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    k_split_w16<<<(unsigned)blocks, 256, 0, s>>>((const uint8_t*)W, (uint8_t*)hi, lo, n);
    return cudaGetLastError();
}

cudaError_t launch_epi_w16(const int64_t* C, int M, int N, int mode, const Epi& ep, cudaStream_t s) {
    if (M < 1 || M > 65535 || N < 1) return cudaErrorInvalidValue;
    const int cols = mode == EPI_SWIGLU ? (N >> 1) : mode == EPI_LOGITS ? ((N + 15) >> 4) : N;
    k_epi_w16<<<dim3((cols + 255) / 256, M), 256, 0, s>>>(C, N, mode, ep);
    return cudaGetLastError();
}

cudaError_t launch_gemm_w16(const int8_t* A, const int8_t* Wh, const uint8_t* Wl, int64_t* C, int M,
                            int N, int K, int32_t* status, cudaStream_t s) {
    if ((K & 15) || K < 16 || K > 65536 || M < 1 || N < 1) return cudaErrorInvalidValue;
    if (((uintptr_t)A & 15) || ((uintptr_t)Wh & 15) || ((uintptr_t)Wl & 15)) return cudaErrorInvalidValue;
    cudaError_t e = get_encode();
    if (e != cudaSuccess) return e;
    CUtensorMap ma, mh, ml;
    e = make_map(&ma, A, M, K, W16_BM);
    if (e == cudaSuccess) e = make_map(&mh, Wh, N, K);
    if (e == cudaSuccess) e = make_map(&ml, Wl, N, K);
    if (e != cudaSuccess) return e;
    const int tiles_n = (N + GM_BN - 1) / GM_BN, tiles_m = (M + W16_BM - 1) / W16_BM;
    const int nk = (K + GM_BK - 1) / GM_BK, tiles = tiles_n * tiles_m;
    int splits = 1, ksl = nk;
    if (g_num_sms > 0 && tiles < g_num_sms && nk >= 4) {
        splits = std::min(nk / 2, (2 * g_num_sms + tiles - 1) / tiles);
        ksl = (nk + splits - 1) / splits;
        splits = (nk + ksl - 1) / ksl;
        if (splits > 1) {
            e = cudaMemsetAsync(C, 0, (size_t)M * N * sizeof(int64_t), s);
            if (e != cudaSuccess) return e;
        }
    }
    k_gemm_w16<<<dim3(tiles_n, tiles_m, splits), GM_THREADS, W16_SMEM, s>>>(ma, mh, ml, M, N, K, C, ksl,
                                                                            status);
    return cudaGetLastError();
}

__device__ int32_t g_free_status[ST_N];
int32_t* standalone_status() {
    static int32_t* addr[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    if (!addr[dev] && cudaGetSymbolAddress((void**)&addr[dev], g_free_status) != cudaSuccess) return nullptr;
    return addr[dev];
}

using StepFn = void (*)(StepArgs);
static StepFn step_kernel(int d, int grp) {
    if (d == 128 && grp == 2) return k_decode_step<4, 2>;
    if (d == 64 && grp == 4) return k_decode_step<2, 4>;
    if (d == 64 && grp == 2) return k_decode_step<2, 2>;
    return nullptr;
}
bool decode_step_supported(int d, int grp) { return step_kernel(d, grp) != nullptr; }
bool decode_step_fits(int d, int grp, size_t smem) {
    StepFn k = step_kernel(d, grp);
    if (!k || smem > 227 * 1024) return false;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return false;
    int nb = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, k, STEP_THREADS, smem) != cudaSuccess) return false;
    return nb >= 1;
}

cudaError_t launch_decode_step(const StepArgs& a, int grid, size_t smem, cudaStream_t s) {
    StepFn k = step_kernel(a.d, 1 << a.lg_grp);
    if (!k) return cudaErrorNotSupported;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(STEP_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeCooperative;   // every CTA resident: CTAs poll one another's rows
    at[0].val.cooperative = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k, a);
}

cudaError_t kernels_init() {
    cudaError_t e = gemv_attr_all<EPI_RAW>();
    if (e == cudaSuccess) e = gemv_attr_all<EPI_QKV>();
    if (e == cudaSuccess) e = gemv_attr_all<EPI_RESADD>();
    if (e == cudaSuccess) e = gemv_attr_all<EPI_SWIGLU>();
    if (e == cudaSuccess) e = gemv_attr_all<EPI_LOGITS>();
    for (int lg = 0; lg < 4 && e == cudaSuccess; ++lg) {
        e = cudaFuncSetAttribute(attention_kernel(128, lg), cudaFuncAttributeMaxDynamicSharedMemorySize, 220 * 1024);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(attention_kernel(64, lg), cudaFuncAttributeMaxDynamicSharedMemorySize, 220 * 1024);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(attn_dec_global_kernel(128, lg), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     220 * 1024);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(attn_dec_global_kernel(64, lg), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     220 * 1024);
    }
    const int sgm = (int)SG_SMEM_MAX;
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k_sgemv<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, sgm);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k_sgemv<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, sgm);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k_gemm_w16, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)W16_SMEM);
    for (int bm : {32, 64, 128})
        for (int mode : {EPI_RAW, EPI_QKV, EPI_RESADD, EPI_SWIGLU, EPI_LOGITS})
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(gemm_kernel(mode, bm), cudaFuncAttributeMaxDynamicSharedMemorySize, (int)GM_SMEM);
    for (int lg = 0; lg < 4 && e == cudaSuccess; ++lg) {
        e = cudaFuncSetAttribute(attn_dec_kernel(128, lg), cudaFuncAttributeMaxDynamicSharedMemorySize, AD_SMEM_MAX);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(attn_dec_kernel(64, lg), cudaFuncAttributeMaxDynamicSharedMemorySize, AD_SMEM_MAX);
    }
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k_attn_prefill<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, PfCfg<128>::SMEM);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k_attn_prefill<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, PfCfg<64>::SMEM);
    if (e == cudaSuccess) {
        k_sig_table<<<(SIG_TAB_N + 255) / 256, 256>>>();
        e = cudaGetLastError();
    }
    if (e == cudaSuccess) e = cudaStreamSynchronize(0);
    int dev = 0;
    if (e == cudaSuccess) e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev);
    return e;
}

}  // namespace detint
