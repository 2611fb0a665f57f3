// detint host runtime: artifact loading (SHA-256 checked), device memory
// layout, the per-step launch sequence, CUDA-graph replay of decode steps,
// and the C ABI declared in include/detint.h.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <array>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/detint.h"
#include "kernels.h"

using namespace detint;

// ------------------------------------------------------------ last error
static thread_local std::string g_last_error;
static int fail(int code, const std::string& msg) {
    g_last_error = msg;
    return code;
}
#define CK(call)                                                                         \
    do {                                                                                 \
        cudaError_t e_ = (call);                                                         \
        if (e_ != cudaSuccess)                                                           \
            return fail(DETINT_E_CUDA, std::string(#call) + ": " + cudaGetErrorString(e_)); \
    } while (0)

// ------------------------------------------------ SHA-256 (FIPS 180-4)
namespace {
struct Sha256 {
    uint32_t h[8];
    uint8_t buf[64];
    uint64_t len = 0;
    size_t fill = 0;
    static uint32_t rotr(uint32_t x, int n) { return (x >> n) | (x << (32 - n)); }
    Sha256() {
        static const uint32_t init[8] = {0x6a09e667, 0xbb67ae85, 0x3c6ef372, 0xa54ff53a,
                                         0x510e527f, 0x9b05688c, 0x1f83d9ab, 0x5be0cd19};
        memcpy(h, init, sizeof h);
    }
    void block(const uint8_t* p) {
        static const uint32_t k[64] = {
            0x428a2f98, 0x71374491, 0xb5c0fbcf, 0xe9b5dba5, 0x3956c25b, 0x59f111f1, 0x923f82a4,
            0xab1c5ed5, 0xd807aa98, 0x12835b01, 0x243185be, 0x550c7dc3, 0x72be5d74, 0x80deb1fe,
            0x9bdc06a7, 0xc19bf174, 0xe49b69c1, 0xefbe4786, 0x0fc19dc6, 0x240ca1cc, 0x2de92c6f,
            0x4a7484aa, 0x5cb0a9dc, 0x76f988da, 0x983e5152, 0xa831c66d, 0xb00327c8, 0xbf597fc7,
            0xc6e00bf3, 0xd5a79147, 0x06ca6351, 0x14292967, 0x27b70a85, 0x2e1b2138, 0x4d2c6dfc,
            0x53380d13, 0x650a7354, 0x766a0abb, 0x81c2c92e, 0x92722c85, 0xa2bfe8a1, 0xa81a664b,
            0xc24b8b70, 0xc76c51a3, 0xd192e819, 0xd6990624, 0xf40e3585, 0x106aa070, 0x19a4c116,
            0x1e376c08, 0x2748774c, 0x34b0bcb5, 0x391c0cb3, 0x4ed8aa4a, 0x5b9cca4f, 0x682e6ff3,
            0x748f82ee, 0x78a5636f, 0x84c87814, 0x8cc70208, 0x90befffa, 0xa4506ceb, 0xbef9a3f7,
            0xc67178f2};
        uint32_t w[64];
        for (int i = 0; i < 16; ++i)
            w[i] = (uint32_t)p[4 * i] << 24 | (uint32_t)p[4 * i + 1] << 16 |
                   (uint32_t)p[4 * i + 2] << 8 | p[4 * i + 3];
        for (int i = 16; i < 64; ++i) {
            uint32_t s0 = rotr(w[i - 15], 7) ^ rotr(w[i - 15], 18) ^ (w[i - 15] >> 3);
            uint32_t s1 = rotr(w[i - 2], 17) ^ rotr(w[i - 2], 19) ^ (w[i - 2] >> 10);
            w[i] = w[i - 16] + s0 + w[i - 7] + s1;
        }
        uint32_t a = h[0], b = h[1], c = h[2], d = h[3], e = h[4], f = h[5], g = h[6], hh = h[7];
        for (int i = 0; i < 64; ++i) {
            uint32_t S1 = rotr(e, 6) ^ rotr(e, 11) ^ rotr(e, 25);
            uint32_t ch = (e & f) ^ (~e & g);
            uint32_t t1 = hh + S1 + ch + k[i] + w[i];
            uint32_t S0 = rotr(a, 2) ^ rotr(a, 13) ^ rotr(a, 22);
            uint32_t mj = (a & b) ^ (a & c) ^ (b & c);
            uint32_t t2 = S0 + mj;
            hh = g; g = f; f = e; e = d + t1; d = c; c = b; b = a; a = t1 + t2;
        }
        h[0] += a; h[1] += b; h[2] += c; h[3] += d; h[4] += e; h[5] += f; h[6] += g; h[7] += hh;
    }
    void update(const uint8_t* p, size_t n) {
        len += n;
        if (fill) {
            while (n && fill < 64) { buf[fill++] = *p++; --n; }
            if (fill == 64) { block(buf); fill = 0; }
        }
        while (n >= 64) { block(p); p += 64; n -= 64; }
        while (n) { buf[fill++] = *p++; --n; }
    }
    std::string hex() {
        uint64_t bits = len * 8;
        uint8_t pad = 0x80;
        update(&pad, 1);
        uint8_t z = 0;
        while (fill != 56) update(&z, 1);
        uint8_t lb[8];
        for (int i = 0; i < 8; ++i) lb[i] = (uint8_t)(bits >> (56 - 8 * i));
        update(lb, 8);
        char out[65];
        for (int i = 0; i < 8; ++i) snprintf(out + 8 * i, 9, "%08x", h[i]);
        return std::string(out, 64);
    }
};
}  // namespace

// ---------------------------------------------------------------- model
struct LayerW {
    int16_t *attn_gamma, *ffn_gamma, *q_gamma, *k_gamma;
    int8_t *w_qkv, *w_o, *w_gu, *w_d;          // int8 weights, or the high limbs of 16-bit ones
    uint8_t *l_qkv, *l_o, *l_gu, *l_d;          // exact mode: the low limbs (else null)
    int32_t *m_qkv, *m_o, *m_gu, *m_d, *kvp;
};

struct GraphEntry {
    cudaGraphExec_t exec = nullptr;
    int32_t* seq_dev = nullptr;
};

struct detint_model {
    int L, H, nq, nkv, d, F, V, max_pos, qk_norm, lg_grp;
    long long eps_h, eps_qk;
    int max_batch, max_ctx, mbs, nblocks, ctx_cap;
    unsigned char* wblob = nullptr;
    int wide = 0;            // exact mode: 16-bit weights as two limbs, channel shift 30
    int8_t* embed;
    uint8_t* embed_lo = nullptr;
    int32_t* embed_m;
    int16_t *final_gamma, *rope_cos, *rope_sin;
    std::vector<LayerW> layers;
    int8_t *kcache = nullptr, *vcache = nullptr;
    size_t kv_layer_elems;
    int32_t* block_table = nullptr;
    // paged KV pool: blocks are taken from a free list as sequences grow and
    // shared (reference counted) between sequences forked from one prefix
    std::vector<int32_t> bt_host;          // [max_batch][mbs] mirror of block_table
    std::vector<std::vector<int>> seq_blocks;
    std::vector<int> refcnt, free_blocks;
    bool bt_dirty = false;
    int32_t* seq_len_dev = nullptr;
    std::vector<int> seq_len;
    // scratch for up to Tcap tokens
    int Tcap = 0;
    unsigned char* scratch = nullptr;
    int32_t *h, *qkv, *o, *sbuf, *mt, *kt, *mq, *kq, *tok_seq, *tok_pos, *rows;
    int8_t *x8, *q8;
    int32_t *pval, *pidx, *logits_int;
    int64_t* c64 = nullptr;  // exact mode: the limb GEMM's int64 accumulators
    int npart;
    int32_t* status = nullptr;
    int use_graph = 1;
    int fused_decode = 1;    // 0: decode through the separate row kernels (tests compare both)
    int tc_prefill = 1;      // 0: prefill attention through the per-token kernel (tests compare both)
    int staged_decode = 1;   // 0: decode attention through the per-token kernel (tests compare both)
    int dec_cap = 0;         // keys the staged decode attention holds (0: unsupported shape)
    int dec_staged = 0;      // this step's decode: 0 kernels (global K/V), 1 kernels (staged K/V), 2 one launch
    int persistent = 0;      // 1: decode steps of up to 8 sequences as one launch where supported
    // the one-launch decode step (k_decode_step.cuh): per batch size T = 1..8,
    // its CTA roles and attention staging; its tagged exchange rows and tags
    struct StepCfg { int ok, NG, NA, ipc, cap, lg_ns, ms, off[6]; } st_cfg[8] = {};
    StepLayer* st_layers = nullptr;
    unsigned long long* st_x = nullptr;
    unsigned* st_ctl = nullptr;
    int32_t* st_rows = nullptr;    // [8][5 x (NG + 1), in a stride of 5 (nsm + 1)]
    size_t st_smem = 0, st_xoff[5] = {0, 0, 0, 0, 0};
    int st_scap = 0, st_stall = 0, nsm = 0;
    int32_t* gws = nullptr;  // split-K workspace of the short-M tiled GEMMs
    size_t gws_elems = 0;
    int* gcnt = nullptr;     // their tile counters (self-resetting)
    int gcnt_n = 0;
    int pf_ok = 0;           // the tensor-core prefill attention supports this shape
    CUtensorMap kmap, vmap;  // whole K / V^T caches for the prefill attention
    int32_t* qblk = nullptr; // prefill query blocks [Tcap + max_batch][4]
    int nqb = 0;
    std::map<std::string, GraphEntry> graphs;
    int32_t* pinned = nullptr;       // host staging for small copies
    size_t pinned_elems = 0;
    cudaEvent_t pinned_done = nullptr;
};

// Copy host int32 arrays to device through pinned staging, asynchronously on
// s; the staging area is reused only after the previous copies completed.
static int stage_copies(detint_model* m, cudaStream_t s,
                        const std::vector<std::pair<int32_t*, std::vector<int32_t>*>>& jobs) {
    size_t total = 0;
    for (auto& j : jobs) total += j.second->size();
    if (m->pinned_done) CK(cudaEventSynchronize(m->pinned_done));
    if (total > m->pinned_elems) {
        if (m->pinned) cudaFreeHost(m->pinned);
        m->pinned = nullptr;
        size_t n = std::max(total, (size_t)4096);
        CK(cudaMallocHost(&m->pinned, n * 4));
        m->pinned_elems = n;
    }
    if (!m->pinned_done) CK(cudaEventCreateWithFlags(&m->pinned_done, cudaEventDisableTiming));
    size_t off = 0;
    for (auto& j : jobs) {
        memcpy(m->pinned + off, j.second->data(), j.second->size() * 4);
        CK(cudaMemcpyAsync(j.first, m->pinned + off, j.second->size() * 4, cudaMemcpyHostToDevice, s));
        off += j.second->size();
    }
    CK(cudaEventRecord(m->pinned_done, s));
    return DETINT_OK;
}

static size_t al256(size_t x) { return (x + 255) & ~(size_t)255; }
static int ilog2i(int n) { int l = 0; while ((1 << l) < n) ++l; return l; }

// every captured step graph; waits for the device first, since one may be in flight
static void free_graphs(detint_model* m) {
    if (m->graphs.empty()) return;
    cudaDeviceSynchronize();
    for (auto& kv : m->graphs) {
        if (kv.second.exec) cudaGraphExecDestroy(kv.second.exec);
        if (kv.second.seq_dev) cudaFree(kv.second.seq_dev);
    }
    m->graphs.clear();
}

// (Re)allocate token scratch for T tokens; synchronises the device when it grows.
static int ensure_scratch(detint_model* m, int T) {
    if (T <= m->Tcap) return DETINT_OK;
    int Tn = T < 64 ? 64 : T;
    CK(cudaDeviceSynchronize());
    free_graphs(m);
    if (m->scratch) cudaFree(m->scratch);
    m->scratch = nullptr;
    const int nqkv = (m->nq + 2 * m->nkv) * m->d;
    const int wmax = std::max(std::max(m->H, m->nq * m->d), m->F);
    const int rows_out = m->max_batch;   // logits rows: one per sequence
    m->npart = (m->V + 15) / 16;
    size_t off = 0;
    auto take = [&](size_t bytes) { size_t o = off; off = al256(off + bytes); return o; };
    size_t o_h = take((size_t)Tn * m->H * 4), o_qkv = take((size_t)Tn * nqkv * 4),
           o_o = take((size_t)Tn * m->nq * m->d * 4), o_s = take((size_t)Tn * m->F * 4),
           o_mt = take((size_t)Tn * 4), o_kt = take((size_t)Tn * 4),
           o_mq = take((size_t)Tn * m->nq * 4), o_kq = take((size_t)Tn * m->nq * 4),
           o_ts = take((size_t)Tn * 4), o_tp = take((size_t)Tn * 4), o_rows = take((size_t)Tn * 4),
           o_x8 = take((size_t)Tn * wmax), o_q8 = take((size_t)Tn * m->nq * m->d),
           o_pv = take((size_t)rows_out * m->npart * 4), o_pi = take((size_t)rows_out * m->npart * 4),
           o_lg = take((size_t)rows_out * m->V * 4),
           o_qb = take((size_t)(Tn + m->max_batch) * 16),
           o_c64 = m->wide ? take(std::max((size_t)Tn * std::max(std::max(nqkv, m->H), 2 * m->F),
                                           (size_t)rows_out * m->V) * 8) : 0;
    cudaError_t e = cudaMalloc(&m->scratch, off);
    if (e != cudaSuccess) { m->scratch = nullptr; m->Tcap = 0; return fail(DETINT_E_OOM, "scratch allocation failed"); }
    unsigned char* b = m->scratch;
    m->h = (int32_t*)(b + o_h); m->qkv = (int32_t*)(b + o_qkv); m->o = (int32_t*)(b + o_o);
    m->sbuf = (int32_t*)(b + o_s); m->mt = (int32_t*)(b + o_mt); m->kt = (int32_t*)(b + o_kt);
    m->mq = (int32_t*)(b + o_mq); m->kq = (int32_t*)(b + o_kq); m->tok_seq = (int32_t*)(b + o_ts);
    m->tok_pos = (int32_t*)(b + o_tp); m->rows = (int32_t*)(b + o_rows);
    m->x8 = (int8_t*)(b + o_x8); m->q8 = (int8_t*)(b + o_q8);
    m->pval = (int32_t*)(b + o_pv); m->pidx = (int32_t*)(b + o_pi); m->logits_int = (int32_t*)(b + o_lg);
    m->qblk = (int32_t*)(b + o_qb);
    m->c64 = m->wide ? (int64_t*)(b + o_c64) : nullptr;
    m->Tcap = Tn;
    return DETINT_OK;
}

// GEMM of X[M][K] by W[N][K] with an epilogue.
static cudaError_t gemm_epi(detint_model* m, const int8_t* X, const int8_t* W, int M, int N, int K,
                            int mode, const Epi& ep, cudaStream_t s) {
    // up to 8 rows the register GEMV streams the weights once; beyond, the
    // tiled GEMM (32/64/128-row tiles) keeps the int8 tensor pipe busy
    if (mode == EPI_LOGITS && M <= 8) {
        // few rows: the GEMV streams the vocabulary once
        for (int r0 = 0; r0 < M; r0 += 32) {
            Epi e = ep;
            e.out = ep.out + (size_t)r0 * ep.ldo;
            e.mt = ep.mt + r0;
            e.kt = ep.kt + r0;
            e.pval = ep.pval + (size_t)r0 * ep.npart;
            e.pidx = ep.pidx + (size_t)r0 * ep.npart;
            cudaError_t ce = launch_gemv(W, X + (size_t)r0 * K, std::min(32, M - r0), N, K, mode, e, s);
            if (ce != cudaSuccess) return ce;
        }
        return cudaSuccess;
    }
    if (M <= 8 || (K & 15)) return launch_gemv(W, X, M, N, K, mode, ep, s);
    // short M: small grids split K through the model's workspace
    if (M <= 64) return launch_gemm(X, W, M, N, K, mode, ep, s, m->gws, m->gws_elems, m->gcnt, m->gcnt_n);
    return launch_gemm(X, W, M, N, K, mode, ep, s);
}

// exact mode: the limb GEMM (int64 accumulators) then the 128-bit epilogue
static cudaError_t gemm_wide(detint_model* m, const int8_t* X, const int8_t* Whi, const uint8_t* Wlo, int M,
                             int N, int K, int mode, const Epi& ep, cudaStream_t s) {
    cudaError_t e = launch_gemm_w16(X, Whi, Wlo, m->c64, M, N, K, m->status, s);
    if (e != cudaSuccess) return e;
    return launch_epi_w16(m->c64, M, N, mode, ep, s);
}

// The forward pass of T tokens whose (sequence, position) are in tok_seq /
// tok_pos on the device (decode: positions are read from seq_len_dev by the
// embedding kernel). Produces logits and argmax for the R rows listed in
// m->rows (prefill) or for every token (decode, rows == nullptr).
// Decode with at most 8 sequences: 5 kernels per layer chained by
// programmatic dependent launch (weights stream ahead of the dependency).
static int run_decode_step(detint_model* m, int T, const int32_t* tokens, int32_t* logits,
                           int32_t* next_tok, cudaStream_t s);

static int run_decode_fused(detint_model* m, int T, const int32_t* tokens, int32_t* logits,
                            int32_t* next_tok, cudaStream_t s) {
    if (m->dec_staged == 2) return run_decode_step(m, T, tokens, logits, next_tok, s);
    const int H = m->H, d = m->d, nq = m->nq, nkv = m->nkv, F = m->F;
    const int nqkv = (nq + 2 * nkv) * d;
    // from 3 sequences on, each row is quantised once by a row kernel (one CTA
    // per row) instead of redundantly by every GEMV CTA (measured steps: 2
    // sequences 868 us fused against 1002 us with row kernels; 3 and 4
    // sequences 1136 and 1213 us fused against 1052 and 1066 us)
    const bool sep = T >= 3;
    auto gemv = [&](const int8_t* W, int N, int K, const int32_t* xin, const int16_t* gamma, int F_in,
                    int pro, int mode, const Epi& e, int spare = 0) -> int {
        if (sep) {
            if (pro == 1) CK(launch_normquant(xin, nullptr, T, K, gamma, m->eps_h, m->x8, m->mt, m->kt, s, true));
            else CK(launch_actquant(xin, T, K, F_in, m->x8, m->mt, m->kt, s, true));
            CK(launch_sgemv(W, N, K, T, nullptr, nullptr, nullptr, 0, 0, 0, mode, e, s, m->x8, m->mt, m->kt,
                            true, spare));
        } else {
            CK(launch_sgemv(W, N, K, T, xin, nullptr, gamma, m->eps_h, F_in, pro, mode, e, s, nullptr, nullptr,
                            nullptr, true, spare));
        }
        return DETINT_OK;
    };
    // the staged attention's CTAs (one per token and kv head) need more shared
    // memory than is left beside a GEMV CTA: SMs left free by the QKV GEMV
    // take them early, and they copy the cached K/V while the GEMV runs
    const int att_ctas = m->dec_staged ? T * nkv : 0;
    CK(launch_embed(tokens, T, m->tok_seq, m->tok_pos, m->seq_len_dev, 1, m->max_ctx,
                    m->embed, nullptr, m->embed_m, H, m->V, m->h, m->status, s));
    for (int l = 0; l < m->L; ++l) {
        const LayerW& w = m->layers[l];
        Epi e{};
        e.status = m->status;
        e.out = m->qkv; e.ldo = nqkv; e.mc = w.m_qkv; e.fout = 12;
        int rc = gemv(w.w_qkv, nqkv, H, m->h, w.attn_gamma, 0, 1, EPI_QKV, e, att_ctas);
        if (rc) return rc;
        QkvPostArgs qa{};
        qa.qkv = m->qkv; qa.q_gamma = w.q_gamma; qa.k_gamma = w.k_gamma; qa.qk_norm = m->qk_norm;
        qa.eps_qk = m->eps_qk; qa.rope_cos = m->rope_cos; qa.rope_sin = m->rope_sin; qa.kvp = w.kvp;
        qa.tok_seq = m->tok_seq; qa.tok_pos = m->tok_pos; qa.block_table = m->block_table;
        qa.mbs = m->mbs; qa.kc = m->kcache + (size_t)l * m->kv_layer_elems;
        qa.vc = m->vcache + (size_t)l * m->kv_layer_elems;
        qa.T = T; qa.nq = nq; qa.nkv = nkv; qa.d = d; qa.lg_grp = m->lg_grp;
        AttnArgs aa{};
        aa.kc = qa.kc; aa.vc = qa.vc; aa.block_table = m->block_table; aa.mbs = m->mbs;
        aa.tok_seq = m->tok_seq; aa.tok_pos = m->tok_pos; aa.kvp = w.kvp; aa.o = m->o; aa.T = T;
        aa.nq = nq; aa.nkv = nkv; aa.d = d; aa.lg_grp = m->lg_grp;
        aa.ctx_cap = m->dec_staged ? m->dec_cap : m->ctx_cap;
        aa.seq_len = m->seq_len_dev; aa.status = m->status;
        CK(launch_attn_decode(aa, qa, s, m->dec_staged != 0));
        e.out = m->h; e.ldo = H; e.mc = w.m_o; e.fout = 16;
        if ((rc = gemv(w.w_o, H, nq * d, m->o, nullptr, 12, 2, EPI_RESADD, e))) return rc;
        e.out = m->sbuf; e.ldo = F; e.mc = w.m_gu; e.fout = 12;
        if ((rc = gemv(w.w_gu, 2 * F, H, m->h, w.ffn_gamma, 0, 1, EPI_SWIGLU, e))) return rc;
        e.out = m->h; e.ldo = H; e.mc = w.m_d; e.fout = 16;
        if ((rc = gemv(w.w_d, H, F, m->sbuf, nullptr, 10, 2, EPI_RESADD, e))) return rc;
    }
    Epi e{};
    e.status = m->status;
    e.out = logits ? logits : m->logits_int; e.ldo = m->V; e.mc = m->embed_m; e.fout = 16;
    e.pval = m->pval; e.pidx = m->pidx; e.npart = m->npart;
    int rc = gemv(m->embed, m->V, H, m->h, m->final_gamma, 0, 1, EPI_LOGITS, e);
    if (rc) return rc;
    CK(launch_argmax_final(m->pval, m->pidx, T, m->npart, next_tok, m->tok_seq, m->seq_len_dev, s, true));
    return DETINT_OK;
}

// every shape the fused decode path supports
static bool decode_fusable(const detint_model* m, int T) {
    if (T > 8 || m->fused_decode == 0 || m->wide) return false;
    const int d = m->d, nq = m->nq, nkv = m->nkv;
    const int Ks[4] = {m->H, nq * d, m->H, m->F};
    for (int K : Ks) {
        if (K & 63) return false;
        const int KC = K <= 1024 ? K : 1024;
        if (K % KC) return false;
        const size_t smem = (size_t)4 * 16 * (KC + 64) + (size_t)8 * (K + 64) + 16384 + 2 * K + 2048;
        if (smem > 200 * 1024) return false;
    }
    // one warp per q head of a kv group plus one for the K/V head
    return ((m->H & (m->H - 1)) == 0) && nkv >= 1 && (1 << m->lg_grp) < 8;
}

static int run_forward(detint_model* m, int T, const int32_t* tokens, int decode, int R,
                       const int32_t* rows, int32_t* logits, int32_t* next_tok, cudaStream_t s) {
    const int H = m->H, d = m->d, nq = m->nq, nkv = m->nkv, F = m->F;
    const int nqkv = (nq + 2 * nkv) * d;
    if (decode && decode_fusable(m, T)) return run_decode_fused(m, T, tokens, logits, next_tok, s);
    CK(launch_embed(tokens, T, m->tok_seq, m->tok_pos, m->seq_len_dev, decode, m->max_ctx,
                    m->embed, m->embed_lo, m->embed_m, H, m->V, m->h, m->status, s));
    // the layer GEMMs: int8 weights (tiled GEMM / GEMV with fused epilogues) or
    // 16-bit weights as limbs (exact mode)
    auto gemm = [&](const int8_t* W, const uint8_t* Wl, int M, int N, int K, int mode, const Epi& e) {
        return m->wide ? gemm_wide(m, m->x8, W, Wl, M, N, K, mode, e, s)
                       : gemm_epi(m, m->x8, W, M, N, K, mode, e, s);
    };
    for (int l = 0; l < m->L; ++l) {
        const LayerW& w = m->layers[l];
        int8_t* kc = m->kcache + (size_t)l * m->kv_layer_elems;
        int8_t* vc = m->vcache + (size_t)l * m->kv_layer_elems;
        CK(launch_normquant(m->h, nullptr, T, H, w.attn_gamma, m->eps_h, m->x8, m->mt, m->kt, s));
        Epi e{};
        e.status = m->status;
        e.mt = m->mt; e.kt = m->kt;
        e.out = m->qkv; e.ldo = nqkv; e.mc = w.m_qkv; e.fout = 12;
        CK(gemm(w.w_qkv, w.l_qkv, T, nqkv, H, EPI_QKV, e));
        QkvPostArgs qa{};
        qa.qkv = m->qkv; qa.q_gamma = w.q_gamma; qa.k_gamma = w.k_gamma; qa.qk_norm = m->qk_norm;
        qa.eps_qk = m->eps_qk; qa.rope_cos = m->rope_cos; qa.rope_sin = m->rope_sin; qa.kvp = w.kvp;
        qa.tok_seq = m->tok_seq; qa.tok_pos = m->tok_pos; qa.block_table = m->block_table;
        qa.mbs = m->mbs; qa.q8 = m->q8; qa.mq = m->mq; qa.kq = m->kq; qa.kc = kc; qa.vc = vc;
        qa.T = T; qa.nq = nq; qa.nkv = nkv; qa.d = d; qa.lg_grp = m->lg_grp;
        AttnArgs aa{};
        aa.q8 = m->q8; aa.mq = m->mq; aa.kq = m->kq; aa.kc = kc; aa.vc = vc;
        aa.block_table = m->block_table; aa.mbs = m->mbs; aa.tok_seq = m->tok_seq;
        aa.tok_pos = m->tok_pos; aa.kvp = w.kvp; aa.o = m->o; aa.T = T; aa.nq = nq; aa.nkv = nkv;
        aa.d = d; aa.lg_grp = m->lg_grp; aa.ctx_cap = m->ctx_cap;
        if (decode) {
            // one token per sequence: QKV post-processing fused into the decode
            // attention, the sequence's K/V staged in shared memory while every
            // context fits, else read from the cache
            aa.ctx_cap = m->dec_staged == 1 ? m->dec_cap : m->ctx_cap;
            aa.seq_len = m->seq_len_dev; aa.status = m->status;
            CK(launch_attn_decode(aa, qa, s, m->dec_staged == 1));
        } else if (!decode && m->pf_ok && m->tc_prefill) {
            CK(launch_qkv_post(qa, s));
            PfArgs pa{};
            pa.q8 = m->q8; pa.mq = m->mq; pa.kq = m->kq; pa.block_table = m->block_table;
            pa.mbs = m->mbs; pa.qblk = m->qblk; pa.nqb = m->nqb; pa.kvp = w.kvp; pa.o = m->o;
            pa.nq = nq; pa.nkv = nkv; pa.lg_grp = m->lg_grp;
            pa.krow0 = (int)((long long)l * m->nblocks * nkv * KV_BLK);
            pa.vrow0 = (int)((long long)l * m->nblocks * nkv * d);
            pa.status = m->status;
            CK(launch_attn_prefill(pa, m->kmap, m->vmap, d, s));
        } else {
            CK(launch_qkv_post(qa, s));
            CK(launch_attention(aa, s));
        }
        CK(launch_actquant(m->o, T, nq * d, 12, m->x8, m->mt, m->kt, s));
        e.out = m->h; e.ldo = H; e.mc = w.m_o; e.fout = 16;
        CK(gemm(w.w_o, w.l_o, T, H, nq * d, EPI_RESADD, e));
        CK(launch_normquant(m->h, nullptr, T, H, w.ffn_gamma, m->eps_h, m->x8, m->mt, m->kt, s));
        e.out = m->sbuf; e.ldo = F; e.mc = w.m_gu; e.fout = 12;
        CK(gemm(w.w_gu, w.l_gu, T, 2 * F, H, EPI_SWIGLU, e));
        CK(launch_actquant(m->sbuf, T, F, 10, m->x8, m->mt, m->kt, s));
        e.out = m->h; e.ldo = H; e.mc = w.m_d; e.fout = 16;
        CK(gemm(w.w_d, w.l_d, T, H, F, EPI_RESADD, e));
    }
    CK(launch_normquant(m->h, rows, R, H, m->final_gamma, m->eps_h, m->x8, m->mt, m->kt, s));
    Epi e{};
    e.status = m->status; e.mt = m->mt; e.kt = m->kt;
    e.out = logits ? logits : m->logits_int; e.ldo = m->V; e.mc = m->embed_m; e.fout = 16;
    e.pval = m->pval; e.pidx = m->pidx; e.npart = m->npart;
    CK(gemm(m->embed, m->embed_lo, R, m->V, H, EPI_LOGITS, e));
    CK(launch_argmax_final(m->pval, m->pidx, R, m->npart, next_tok, m->tok_seq,
                           decode ? m->seq_len_dev : nullptr, s));
    return DETINT_OK;
}

// Blocks for positions [0, len) of sequence sid: take free blocks for the
// missing tail. Returns CTX when the pool is exhausted.
static int ensure_blocks(detint_model* m, int sid, int len) {
    std::vector<int>& sb = m->seq_blocks[sid];
    const int need = (len + KV_BLK - 1) / KV_BLK;
    if (need > m->mbs) return fail(DETINT_E_CTX, "context exceeds max_ctx");
    while ((int)sb.size() < need) {
        if (m->free_blocks.empty()) return fail(DETINT_E_CTX, "KV block pool exhausted");
        const int b = m->free_blocks.back();
        m->free_blocks.pop_back();
        m->refcnt[b] = 1;
        m->bt_host[(size_t)sid * m->mbs + sb.size()] = b;
        sb.push_back(b);
        m->bt_dirty = true;
    }
    return DETINT_OK;
}

static void release_blocks(detint_model* m, int sid) {
    for (int b : m->seq_blocks[sid])
        if (--m->refcnt[b] == 0) m->free_blocks.push_back(b);
    m->seq_blocks[sid].clear();
    for (int i = 0; i < m->mbs; ++i) m->bt_host[(size_t)sid * m->mbs + i] = 0;
    m->bt_dirty = true;
}

// upload the block table when it changed (stream-ordered, before the kernels
// that read it)
static int sync_block_table(detint_model* m, cudaStream_t s) {
    if (!m->bt_dirty) return DETINT_OK;
    int rc = stage_copies(m, s, {{m->block_table, &m->bt_host}});
    if (rc == DETINT_OK) m->bt_dirty = false;
    return rc;
}

// The one-launch decode step: for each batch size T = 1..8 the CTA roles
// (NA attention CTAs for T x nkv items, the rest GEMV CTAs), each GEMV CTA's
// weight rows per GEMV kind, the attention staging capacity; the shared
// memory layout; the tagged exchange rows (zeroed: tag 0 is never expected)
// and the tag base (starting at 1). Leaves every st_cfg[].ok = 0 for shapes
// it does not cover (decode then runs one kernel per phase).
static int setup_step(detint_model* m) {
    const int H = m->H, d = m->d, G = 1 << m->lg_grp, nqd = m->nq * d, F = m->F, nkv = m->nkv;
    const int nqkv = (m->nq + 2 * nkv) * d;
    if (m->wide || (H & (H - 1)) || (nkv & (nkv - 1)) || G > 7 || !decode_step_supported(d, G))
        return DETINT_OK;                           // (16-bit weights: the layer-by-layer path)
    for (int K : {H, nqd, F})
        if ((K & 15) || K > STEP_SLOT) return DETINT_OK;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&m->nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return DETINT_OK;
    const size_t dyn = 220 * 1024;
    if (!decode_step_fits(d, G, dyn)) return DETINT_OK;
    m->st_smem = dyn;
    m->st_scap = (m->max_ctx + 15) & ~15;
    const int nsm = m->nsm;
    std::vector<int32_t> rows((size_t)8 * 5 * (nsm + 1), 0);
    const int Ns[5] = {nqkv, H, 2 * F, H, m->V}, unit[5] = {1, 1, 2, 1, 1}, Ks[5] = {H, nqd, H, F, H};
    bool any = false;
    for (int T = 1; T <= 8; ++T) {
        auto& c = m->st_cfg[T - 1];
        c.ok = 0;
        const int items = T * nkv;
        const int NA = items <= 16 ? items : std::min(items, 32);
        const int ipc = (items + NA - 1) / NA;
        const int NG = nsm - NA;
        if (NG < 1 || ipc > 4) continue;
        bool fit = (H + NG - 1) / NG <= STEP_HOWN;
        const int lgT = T <= 1 ? 0 : (T <= 2 ? 1 : (T <= 4 ? 2 : 3));
        const int gn = 32 * (8 >> lgT);
        for (int k = 0; k < 5; ++k) {
            if (k < 4 && Ns[k] / unit[k] < NG) fit = false;       // every GEMV CTA owns rows of every layer phase
            if ((Ks[k] / 2 + gn - 1) / gn > STEP_NP) fit = false;  // prologue pairs per thread
        }
        // the row ranges first: the GEMV layout holds every phase's scales of a CTA's rows
        int32_t* rt = rows.data() + (size_t)(T - 1) * 5 * (nsm + 1);
        for (int k = 0; k < 5; ++k)
            for (int i = 0; i <= NG; ++i)
                rt[k * (NG + 1) + i] = (int32_t)(unit[k] * (((long long)i * (Ns[k] / unit[k])) / NG));
        int ms = 0, nlm = 0;
        for (int i = 0; i < NG; ++i) {
            int sum = 0;
            for (int k = 0; k < 4; ++k) sum += rt[k * (NG + 1) + i + 1] - rt[k * (NG + 1) + i];
            ms = std::max(ms, sum);
            nlm = std::max(nlm, rt[4 * (NG + 1) + i + 1] - rt[4 * (NG + 1) + i]);
        }
        // attention CTA layout: per item K, V and parameter rows, then the score rows
        const int aux = step_aux_bytes(d, m->mbs);
        const size_t fixed = (size_t)G * d + (size_t)G * m->st_scap * 6 + (size_t)G * d * 8 + (size_t)ipc * aux;
        if (!fit || fixed > dyn) continue;
        int cap = (int)((dyn - fixed) / ((size_t)ipc * 2 * d)) & ~(KV_BLK - 1);
        cap = std::min(cap, (m->st_scap + KV_BLK - 1) & ~(KV_BLK - 1));
        // GEMV CTA layout: ring of 8 (else 4) slots, the int8 tile and the
        // int32 input rows of T tokens, gamma, owned residual rows,
        // the layer table, the channel-scale table
        const int Kmax = std::max(H, std::max(nqd, F)), XP = Kmax + 16;
        auto a16 = [](size_t x) { return (x + 15) & ~(size_t)15; };
        const size_t x8b = a16((size_t)T * XP), xinb = (size_t)T * XP * 4, gsb = a16((size_t)H * 2),
                     hownb = (size_t)8 * STEP_HOWN * 4, layb = a16(sizeof(StepLayer) * m->L),
                     mctb = a16((size_t)4 * ((size_t)m->L * ms + nlm));
        const size_t rest = x8b + xinb + gsb + hownb + layb + mctb;
        int lg_ns = 3;
        while (lg_ns > 2 && ((size_t)STEP_SLOT << lg_ns) + rest > dyn) --lg_ns;
        if (((size_t)STEP_SLOT << lg_ns) + rest > dyn) continue;
        c.lg_ns = lg_ns;
        c.off[0] = STEP_SLOT << lg_ns;
        c.off[1] = (int)(c.off[0] + x8b);
        c.off[2] = (int)(c.off[1] + xinb);
        c.off[3] = (int)(c.off[2] + gsb);
        c.off[4] = (int)(c.off[3] + hownb);
        c.off[5] = (int)(c.off[4] + layb);
        c.ms = ms;
        c.NG = NG; c.NA = NA; c.ipc = ipc; c.cap = std::max(cap, 0);
        c.ok = 1;
        any = true;
    }
    if (!any) return DETINT_OK;
    std::vector<StepLayer> pl(m->L);
    for (int l = 0; l < m->L; ++l) {
        const LayerW& w = m->layers[l];
        StepLayer& p = pl[l];
        p.w_qkv = w.w_qkv; p.w_o = w.w_o; p.w_gu = w.w_gu; p.w_d = w.w_d;
        p.m_qkv = w.m_qkv; p.m_o = w.m_o; p.m_gu = w.m_gu; p.m_d = w.m_d; p.kvp = w.kvp;
        p.attn_gamma = w.attn_gamma; p.ffn_gamma = w.ffn_gamma; p.q_gamma = w.q_gamma; p.k_gamma = w.k_gamma;
        p.kc = m->kcache + (size_t)l * m->kv_layer_elems;
        p.vc = m->vcache + (size_t)l * m->kv_layer_elems;
    }
    const size_t nx[5] = {(size_t)8 * H, (size_t)8 * nqkv, (size_t)8 * nqd, (size_t)8 * F, (size_t)nsm * 16};
    size_t tot = 0;
    for (int k = 0; k < 5; ++k) { m->st_xoff[k] = tot; tot += (nx[k] + 1) & ~(size_t)1; }
    const unsigned ctl0[2] = {1u, 0u};
    if (cudaMalloc(&m->st_layers, sizeof(StepLayer) * pl.size()) != cudaSuccess ||
        cudaMalloc(&m->st_x, tot * 8) != cudaSuccess || cudaMalloc(&m->st_ctl, 2 * sizeof(unsigned)) != cudaSuccess ||
        cudaMalloc(&m->st_rows, rows.size() * 4) != cudaSuccess)
        return fail(DETINT_E_OOM, "decode step tables");
    if (cudaMemcpy(m->st_layers, pl.data(), sizeof(StepLayer) * pl.size(), cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMemset(m->st_x, 0, tot * 8) != cudaSuccess ||
        cudaMemcpy(m->st_ctl, ctl0, sizeof ctl0, cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMemcpy(m->st_rows, rows.data(), rows.size() * 4, cudaMemcpyHostToDevice) != cudaSuccess)
        return fail(DETINT_E_CUDA, "decode step tables");
    return DETINT_OK;
}

static int run_decode_step(detint_model* m, int T, const int32_t* tokens, int32_t* logits,
                           int32_t* next_tok, cudaStream_t s) {
    const auto& c = m->st_cfg[T - 1];
    StepArgs a{};
    a.layers = m->st_layers;
    a.L = m->L; a.T = T; a.H = m->H; a.nq = m->nq; a.nkv = m->nkv; a.d = m->d; a.F = m->F; a.V = m->V;
    a.lg_grp = m->lg_grp; a.lg_nkv = ilog2i(m->nkv); a.qk_norm = m->qk_norm; a.max_pos = m->max_ctx;
    a.mbs = m->mbs; a.eps_h = m->eps_h; a.eps_qk = m->eps_qk;
    a.embed = m->embed; a.embed_m = m->embed_m; a.final_gamma = m->final_gamma;
    a.rope_cos = m->rope_cos; a.rope_sin = m->rope_sin; a.block_table = m->block_table;
    a.tokens = tokens; a.tok_seq = m->tok_seq; a.seq_len = m->seq_len_dev;
    a.xh = m->st_x + m->st_xoff[0]; a.xqkv = m->st_x + m->st_xoff[1]; a.xo = m->st_x + m->st_xoff[2];
    a.xs = m->st_x + m->st_xoff[3]; a.xpart = m->st_x + m->st_xoff[4];
    a.ctl = m->st_ctl;
    a.rows = m->st_rows + (size_t)(T - 1) * 5 * (m->nsm + 1);
    a.logits = logits ? logits : m->logits_int; a.next_tok = next_tok; a.status = m->status;
    a.NG = c.NG; a.NA = c.NA; a.ipc = c.ipc; a.lg_ns = c.lg_ns; a.cap = c.cap; a.scap = m->st_scap;
    a.spin = 1 << 20;
    a.stall = m->st_stall;
    a.off_x8 = c.off[0]; a.off_xin = c.off[1]; a.off_gs = c.off[2]; a.off_hown = c.off[3];
    a.off_lay = c.off[4]; a.off_mct = c.off[5]; a.ms = c.ms;
    CK(launch_decode_step(a, c.NG + c.NA, m->st_smem, s));
    return DETINT_OK;
}

// ------------------------------------------------------------------ ABI
extern "C" {

const char* detint_strerror(int code) {
    switch (code) {
        case DETINT_OK: return "ok";
        case DETINT_E_ARG: return "invalid argument";
        case DETINT_E_SHAPE: return "unsupported shape";
        case DETINT_E_TOKEN: return "token id outside the vocabulary";
        case DETINT_E_CTX: return "context capacity exceeded";
        case DETINT_E_ARTIFACT: return "unreadable or malformed artifact";
        case DETINT_E_SHA: return "artifact sha256 mismatch";
        case DETINT_E_CUDA: return "CUDA error";
        case DETINT_E_OOM: return "device out of memory";
        case DETINT_E_SEQ: return "bad sequence id";
        case DETINT_E_SAT: return "saturation recorded";
    }
    return "unknown error";
}

const char* detint_last_error(void) { return g_last_error.c_str(); }

void detint_free(detint_model* m) {
    if (!m) return;
    cudaDeviceSynchronize();
    free_graphs(m);
    if (m->scratch) cudaFree(m->scratch);
    if (m->wblob) cudaFree(m->wblob);
    if (m->kcache) cudaFree(m->kcache);
    if (m->vcache) cudaFree(m->vcache);
    if (m->block_table) cudaFree(m->block_table);
    if (m->seq_len_dev) cudaFree(m->seq_len_dev);
    if (m->status) cudaFree(m->status);
    if (m->st_layers) cudaFree(m->st_layers);
    if (m->st_x) cudaFree(m->st_x);
    if (m->st_ctl) cudaFree(m->st_ctl);
    if (m->st_rows) cudaFree(m->st_rows);
    if (m->gws) cudaFree(m->gws);
    if (m->gcnt) cudaFree(m->gcnt);
    if (m->pinned) cudaFreeHost(m->pinned);
    if (m->pinned_done) cudaEventDestroy(m->pinned_done);
    delete m;
}

static int rd32(const unsigned char* p) { int32_t v; memcpy(&v, p, 4); return v; }

int detint_load(const char* path, int max_batch, int max_ctx, detint_stream_t stream,
                detint_model** out) {
    if (!path || !out || max_batch < 1 || max_ctx < 1) return fail(DETINT_E_ARG, "detint_load: bad arguments");
    *out = nullptr;
    (void)stream;
    FILE* f = fopen(path, "rb");
    if (!f) return fail(DETINT_E_ARTIFACT, std::string("cannot open ") + path);
    fseek(f, 0, SEEK_END);
    long sz = ftell(f);
    fseek(f, 0, SEEK_SET);
    if (sz < 256) { fclose(f); return fail(DETINT_E_ARTIFACT, "artifact too small"); }
    std::vector<unsigned char> blob((size_t)sz);
    size_t got = fread(blob.data(), 1, blob.size(), f);
    fclose(f);
    if (got != blob.size()) return fail(DETINT_E_ARTIFACT, "short read");
    // SHA-256 against the sidecar
    std::string want;
    {
        FILE* g = fopen((std::string(path) + ".sha256").c_str(), "rb");
        if (!g) return fail(DETINT_E_SHA, "missing .sha256 sidecar");
        char buf[80] = {0};
        size_t n = fread(buf, 1, 64, g);
        fclose(g);
        want.assign(buf, n);
    }
    Sha256 sh;
    sh.update(blob.data(), blob.size());
    if (sh.hex() != want) return fail(DETINT_E_SHA, "artifact sha256 mismatch");
    const unsigned char* hd = blob.data();
    if (memcmp(hd, "DETINT01", 8) != 0 || (rd32(hd + 8) != 1 && rd32(hd + 8) != 2))
        return fail(DETINT_E_ARTIFACT, "bad magic/version");
    // version 2: the exact mode's 16-bit weights (weight bits at byte 72)
    const int wide = rd32(hd + 8) == 2;
    if (wide && rd32(hd + 72) != 16) return fail(DETINT_E_ARTIFACT, "unsupported weight width");
    const size_t wb = wide ? 2 : 1;                 // bytes per weight
    detint_model* m = new detint_model();
    m->wide = wide;
    m->L = rd32(hd + 12); m->H = rd32(hd + 16); m->nq = rd32(hd + 20); m->nkv = rd32(hd + 24);
    m->d = rd32(hd + 28); m->F = rd32(hd + 32); m->V = rd32(hd + 36); m->max_pos = rd32(hd + 40);
    m->qk_norm = rd32(hd + 44); m->eps_h = rd32(hd + 48); m->eps_qk = rd32(hd + 52);
    const int H = m->H, d = m->d, F = m->F, V = m->V, nq = m->nq, nkv = m->nkv;
    auto bad_shape = [&](const char* why) { delete m; return fail(DETINT_E_SHAPE, why); };
    if (m->L < 1 || H < 64 || (H & (H - 1)) || (d != 64 && d != 128) || nkv < 1 || nq % nkv)
        return bad_shape("unsupported model shape");
    const int grp = nq / nkv;
    if (grp & (grp - 1) || grp > 8) return bad_shape("q heads per kv head must be a power of two <= 8");
    if ((F & 63) || ((nq * d) & 63) || V < 1) return bad_shape("unsupported model shape");
    if (max_ctx > m->max_pos) return bad_shape("max_ctx exceeds the RoPE table length");
    m->lg_grp = ilog2i(grp);
    m->max_batch = max_batch;
    m->max_ctx = max_ctx;
    m->mbs = (max_ctx + KV_BLK - 1) / KV_BLK;
    m->ctx_cap = m->mbs * KV_BLK;
    m->nblocks = m->mbs * max_batch;
    if (attention_smem_bytes(grp, d, m->ctx_cap) > 220 * 1024) return bad_shape("max_ctx too large for the attention row");
    // section walk (256-byte aligned, file order)
    const int nqkv = (nq + 2 * nkv) * d;
    size_t cur = 256;
    bool ok = true;
    auto take = [&](size_t bytes) -> const unsigned char* {
        cur = (cur + 255) & ~(size_t)255;
        if (cur + bytes > blob.size()) { ok = false; return blob.data(); }
        const unsigned char* p = blob.data() + cur;
        cur += bytes;
        return p;
    };
    // device weight blob layout (same order, gate/up interleaved)
    size_t dsz = 0;
    auto dtake = [&](size_t bytes) { size_t o = dsz; dsz = al256(dsz + bytes); return o; };
    // kind 0: copied as is; kind 1: gate/up, interleaved below; kind 2: 16-bit
    // weights, copied then split on the device into the high limbs (int8, at
    // doff) and the low limbs (uint8, at doff + count)
    struct Sec { const unsigned char* src; size_t bytes; size_t doff; int kind; };
    std::vector<Sec> secs;
    auto add = [&](size_t bytes, int kind = 0) {
        const unsigned char* p = take(bytes);
        secs.push_back({p, bytes, dtake(bytes), kind});
        return secs.size() - 1;
    };
    const int wk = wide ? 2 : 0;                    // kind of a weight section
    size_t s_embed = add((size_t)V * H * wb, wk), s_em = add((size_t)V * 4), s_fg = add((size_t)H * 2),
           s_rc = add((size_t)m->max_pos * (d / 2) * 2), s_rs = add((size_t)m->max_pos * (d / 2) * 2);
    struct LS { size_t ag, fg, qg, kg, wqkv, mqkv, wo, mo, wg, mg, wu, mu, wd, md, kvp, wgu, mgu; };
    std::vector<LS> ls(m->L);
    for (int l = 0; l < m->L; ++l) {
        LS& x = ls[l];
        x.ag = add((size_t)H * 2); x.fg = add((size_t)H * 2); x.qg = add((size_t)d * 2);
        x.kg = add((size_t)d * 2); x.wqkv = add((size_t)nqkv * H * wb, wk); x.mqkv = add((size_t)nqkv * 4);
        x.wo = add((size_t)H * nq * d * wb, wk); x.mo = add((size_t)H * 4);
        x.wg = secs.size(); secs.push_back({take((size_t)F * H * wb), (size_t)F * H * wb, 0, 1});
        x.mg = secs.size(); secs.push_back({take((size_t)F * 4), (size_t)F * 4, 0, 1});
        x.wu = secs.size(); secs.push_back({take((size_t)F * H * wb), (size_t)F * H * wb, 0, 1});
        x.mu = secs.size(); secs.push_back({take((size_t)F * 4), (size_t)F * 4, 0, 1});
        x.wgu = dtake((size_t)2 * F * H * wb);
        x.mgu = dtake((size_t)2 * F * 4);
        x.wd = add((size_t)H * F * wb, wk); x.md = add((size_t)H * 4);
        x.kvp = add((size_t)nkv * (8 + d / 2) * 4);
    }
    if (!ok) { delete m; return fail(DETINT_E_ARTIFACT, "artifact truncated"); }
    cudaError_t ce = cudaMalloc(&m->wblob, dsz);
    if (ce != cudaSuccess) { m->wblob = nullptr; detint_free(m); return fail(DETINT_E_OOM, "weight allocation failed"); }
    // 16-bit weights pass through a device staging buffer and are split there
    // into limbs: W = 256 hi + lo (hi = W >> 8, lo = W & 255)
    int16_t* w16 = nullptr;
    auto put16 = [&](size_t doff, const void* src, size_t count) -> cudaError_t {
        cudaError_t e = cudaMemcpy(w16, src, count * 2, cudaMemcpyHostToDevice);
        if (e == cudaSuccess)
            e = launch_split_w16(w16, (int8_t*)(m->wblob + doff), (uint8_t*)(m->wblob + doff + count),
                                 (long long)count, nullptr);
        return e == cudaSuccess ? cudaDeviceSynchronize() : e;
    };
    if (wide) {
        size_t mx = (size_t)2 * F * H;
        for (const Sec& sc : secs)
            if (sc.kind == 2) mx = std::max(mx, sc.bytes / 2);
        if (cudaMalloc(&w16, mx * 2) != cudaSuccess) { detint_free(m); return fail(DETINT_E_OOM, "staging allocation failed"); }
    }
    for (const Sec& sc : secs) {
        if (sc.kind == 0) ce = cudaMemcpy(m->wblob + sc.doff, sc.src, sc.bytes, cudaMemcpyHostToDevice);
        else if (sc.kind == 2) ce = put16(sc.doff, sc.src, sc.bytes / 2);
        if (ce != cudaSuccess) { if (w16) cudaFree(w16); detint_free(m); return fail(DETINT_E_CUDA, cudaGetErrorString(ce)); }
    }
    // gate/up interleaved as rows (gate_i, up_i) so one CTA holds both of a channel
    std::vector<unsigned char> gu((size_t)2 * F * H * wb);
    std::vector<int32_t> mgu((size_t)2 * F);
    m->layers.resize(m->L);
    for (int l = 0; l < m->L; ++l) {
        const LS& x = ls[l];
        const unsigned char* wg = secs[x.wg].src;
        const unsigned char* wu = secs[x.wu].src;
        const int32_t* mg = (const int32_t*)secs[x.mg].src;
        const int32_t* mu = (const int32_t*)secs[x.mu].src;
        const size_t rb = (size_t)H * wb;             // bytes per weight row
        for (int i = 0; i < F; ++i) {
            memcpy(&gu[(size_t)(2 * i) * rb], wg + (size_t)i * rb, rb);
            memcpy(&gu[(size_t)(2 * i + 1) * rb], wu + (size_t)i * rb, rb);
            int32_t a, b;
            memcpy(&a, mg + i, 4); memcpy(&b, mu + i, 4);
            mgu[2 * i] = a; mgu[2 * i + 1] = b;
        }
        ce = wide ? put16(x.wgu, gu.data(), (size_t)2 * F * H)
                  : cudaMemcpy(m->wblob + x.wgu, gu.data(), gu.size(), cudaMemcpyHostToDevice);
        if (ce == cudaSuccess) ce = cudaMemcpy(m->wblob + x.mgu, mgu.data(), mgu.size() * 4, cudaMemcpyHostToDevice);
        if (ce != cudaSuccess) { detint_free(m); return fail(DETINT_E_CUDA, cudaGetErrorString(ce)); }
        LayerW& w = m->layers[l];
        auto P = [&](size_t si) { return m->wblob + secs[si].doff; };
        w.attn_gamma = (int16_t*)P(x.ag); w.ffn_gamma = (int16_t*)P(x.fg);
        w.q_gamma = (int16_t*)P(x.qg); w.k_gamma = (int16_t*)P(x.kg);
        w.w_qkv = (int8_t*)P(x.wqkv); w.m_qkv = (int32_t*)P(x.mqkv);
        w.w_o = (int8_t*)P(x.wo); w.m_o = (int32_t*)P(x.mo);
        w.w_gu = (int8_t*)(m->wblob + x.wgu); w.m_gu = (int32_t*)(m->wblob + x.mgu);
        w.w_d = (int8_t*)P(x.wd); w.m_d = (int32_t*)P(x.md);
        w.kvp = (int32_t*)P(x.kvp);
        w.l_qkv = w.l_o = w.l_gu = w.l_d = nullptr;
        if (wide) {
            w.l_qkv = (uint8_t*)w.w_qkv + (size_t)nqkv * H;
            w.l_o = (uint8_t*)w.w_o + (size_t)H * nq * d;
            w.l_gu = (uint8_t*)w.w_gu + (size_t)2 * F * H;
            w.l_d = (uint8_t*)w.w_d + (size_t)H * F;
        }
    }
    if (w16) cudaFree(w16);
    m->embed = (int8_t*)(m->wblob + secs[s_embed].doff);
    if (wide) m->embed_lo = (uint8_t*)m->embed + (size_t)V * H;
    m->embed_m = (int32_t*)(m->wblob + secs[s_em].doff);
    m->final_gamma = (int16_t*)(m->wblob + secs[s_fg].doff);
    m->rope_cos = (int16_t*)(m->wblob + secs[s_rc].doff);
    m->rope_sin = (int16_t*)(m->wblob + secs[s_rs].doff);
    // paged int8 KV cache: K [L][NB][nkv][64][d], V [L][NB][nkv][d][64]
    m->kv_layer_elems = (size_t)m->nblocks * nkv * KV_BLK * d;
    if (cudaMalloc(&m->kcache, m->kv_layer_elems * m->L) != cudaSuccess ||
        cudaMalloc(&m->vcache, m->kv_layer_elems * m->L) != cudaSuccess) {
        detint_free(m);
        return fail(DETINT_E_OOM, "KV cache allocation failed");
    }
    // every entry starts at block 0 (a valid block whose keys lie past every
    // sequence's length, so they are never used); blocks are assigned on demand
    std::vector<int32_t> bt((size_t)max_batch * m->mbs, 0);
    m->bt_host = bt;
    m->seq_blocks.assign(max_batch, {});
    m->refcnt.assign(m->nblocks, 0);
    m->free_blocks.clear();
    for (int b = m->nblocks - 1; b >= 0; --b) m->free_blocks.push_back(b);
    if (cudaMalloc(&m->block_table, bt.size() * 4) != cudaSuccess ||
        cudaMalloc(&m->seq_len_dev, (size_t)max_batch * 4) != cudaSuccess ||
        cudaMalloc(&m->status, ST_N * 4) != cudaSuccess) {
        detint_free(m);
        return fail(DETINT_E_OOM, "allocation failed");
    }
    ce = cudaMemcpy(m->block_table, bt.data(), bt.size() * 4, cudaMemcpyHostToDevice);
    if (ce == cudaSuccess) ce = cudaMemset(m->seq_len_dev, 0, (size_t)max_batch * 4);
    if (ce == cudaSuccess) ce = cudaMemset(m->status, 0, ST_N * 4);
    if (ce == cudaSuccess) ce = cudaMemset(m->kcache, 0, m->kv_layer_elems * m->L);
    if (ce == cudaSuccess) ce = cudaMemset(m->vcache, 0, m->kv_layer_elems * m->L);
    if (ce != cudaSuccess) { detint_free(m); return fail(DETINT_E_CUDA, cudaGetErrorString(ce)); }
    m->seq_len.assign(max_batch, 0);
    // the tensor-core prefill attention takes head_dim 64 or 128 and up to 64 q heads per kv head
    m->pf_ok = (d == 64 || d == 128) && m->lg_grp <= 6 &&
               make_kv_maps(&m->kmap, &m->vmap, m->kcache, m->vcache,
                            (long long)m->L * m->nblocks * nkv, d) == cudaSuccess;
    // staged decode attention: the largest block multiple of keys whose K/V
    // copies and score rows fit the shared-memory budget
    m->dec_cap = 0;
    if ((d == 64 || d == 128) && m->lg_grp <= 3) {
        const int want = std::min(m->mbs * KV_BLK, 64 * KV_BLK);
        for (int cap = KV_BLK; cap <= want; cap += KV_BLK)
            if (attn_dec_smem(1 << m->lg_grp, d, cap) <= 220 * 1024) m->dec_cap = cap;
    }
    int rc = ensure_scratch(m, std::max(64, max_batch));
    if (rc != DETINT_OK) { detint_free(m); return rc; }
    ce = kernels_init();
    if (ce != cudaSuccess) { detint_free(m); return fail(DETINT_E_CUDA, cudaGetErrorString(ce)); }
    rc = setup_step(m);
    if (rc != DETINT_OK) { detint_free(m); return rc; }
    {
        // split-K workspace for GEMMs of at most 64 rows: 8 splits of 64 x N
        const int nqkv = (m->nq + 2 * m->nkv) * m->d;
        const int nmax = std::max(std::max(nqkv, m->H), 2 * m->F);
        m->gws_elems = (size_t)8 * 64 * nmax;
        m->gcnt_n = 2 * ((nmax + 127) / 128);
        if (cudaMalloc(&m->gws, m->gws_elems * 4) != cudaSuccess ||
            cudaMalloc(&m->gcnt, (size_t)m->gcnt_n * 4) != cudaSuccess ||
            cudaMemset(m->gcnt, 0, (size_t)m->gcnt_n * 4) != cudaSuccess) {
            detint_free(m);
            return fail(DETINT_E_OOM, "GEMM workspace allocation failed");
        }
    }
    ce = cudaDeviceSynchronize();
    if (ce != cudaSuccess) { detint_free(m); return fail(DETINT_E_CUDA, cudaGetErrorString(ce)); }
    *out = m;
    return DETINT_OK;
}

static int check_seqs(detint_model* m, int n_seq, const int32_t* seq_ids) {
    if (n_seq < 1 || !seq_ids) return fail(DETINT_E_ARG, "no sequences");
    std::vector<char> seen(m->max_batch, 0);
    for (int i = 0; i < n_seq; ++i) {
        const int s = seq_ids[i];
        if (s < 0 || s >= m->max_batch || seen[s]) return fail(DETINT_E_SEQ, "sequence id out of range or repeated");
        seen[s] = 1;
    }
    return DETINT_OK;
}

int detint_prefill(detint_model* m, int n_seq, const int32_t* seq_ids, const int32_t* cu_lens,
                   const int32_t* tokens, int32_t* logits, int32_t* next_tok, detint_stream_t sp) {
    if (!m || !cu_lens || !tokens || !next_tok) return fail(DETINT_E_ARG, "detint_prefill: null pointer");
    int rc = check_seqs(m, n_seq, seq_ids);
    if (rc) return rc;
    if (cu_lens[0] != 0) return fail(DETINT_E_ARG, "cu_lens[0] must be 0");
    for (int i = 0; i < n_seq; ++i) {
        const int len = cu_lens[i + 1] - cu_lens[i];
        if (len < 1) return fail(DETINT_E_ARG, "empty prompt");
        if (m->seq_len[seq_ids[i]] + len > m->max_ctx) return fail(DETINT_E_CTX, "prompt exceeds max_ctx");
    }
    const int T = cu_lens[n_seq];
    cudaStream_t s = (cudaStream_t)sp;
    rc = ensure_scratch(m, std::max(T, n_seq));
    if (rc) return rc;
    std::vector<int32_t> ts(T), tp(T), rows(n_seq);
    for (int i = 0; i < n_seq; ++i) {
        const int sid = seq_ids[i];
        for (int j = cu_lens[i]; j < cu_lens[i + 1]; ++j) {
            ts[j] = sid;
            tp[j] = m->seq_len[sid] + (j - cu_lens[i]);
        }
        rows[i] = cu_lens[i + 1] - 1;
    }
    std::vector<int32_t> newlen(m->seq_len.begin(), m->seq_len.end());
    for (int i = 0; i < n_seq; ++i) newlen[seq_ids[i]] += cu_lens[i + 1] - cu_lens[i];
    for (int i = 0; i < n_seq; ++i) {
        rc = ensure_blocks(m, seq_ids[i], newlen[seq_ids[i]]);
        if (rc) return rc;
    }
    rc = sync_block_table(m, s);
    if (rc) return rc;
    // query blocks of up to 64 / G tokens of one sequence, the longest key
    // ranges first so that the heaviest CTAs start first
    const int bq = PF_ROWS >> m->lg_grp;
    std::vector<std::array<int32_t, 4>> blocks;
    for (int i = 0; i < n_seq; ++i) {
        const int sid = seq_ids[i];
        for (int j = cu_lens[i]; j < cu_lens[i + 1]; j += bq)
            blocks.push_back({j, std::min(bq, cu_lens[i + 1] - j), sid, m->seq_len[sid] + (j - cu_lens[i])});
    }
    std::stable_sort(blocks.begin(), blocks.end(), [](const std::array<int32_t, 4>& x,
                                                      const std::array<int32_t, 4>& y) {
        return x[3] + x[1] > y[3] + y[1];
    });
    std::vector<int32_t> qb(blocks.size() * 4);
    for (size_t b = 0; b < blocks.size(); ++b)
        for (int k = 0; k < 4; ++k) qb[4 * b + k] = blocks[b][k];
    m->nqb = (int)blocks.size();
    rc = stage_copies(m, s, {{m->tok_seq, &ts}, {m->tok_pos, &tp}, {m->rows, &rows}, {m->qblk, &qb}});
    if (rc) return rc;
    rc = run_forward(m, T, tokens, 0, n_seq, m->rows, logits, next_tok, s);
    if (rc) return rc;
    rc = stage_copies(m, s, {{m->seq_len_dev, &newlen}});
    if (rc) return rc;
    for (int i = 0; i < m->max_batch; ++i) m->seq_len[i] = newlen[i];
    return DETINT_OK;
}

int detint_decode_step(detint_model* m, int n_seq, const int32_t* seq_ids, const int32_t* tok,
                       int32_t* logits, int32_t* next_tok, detint_stream_t sp) {
    if (!m || !tok || !next_tok) return fail(DETINT_E_ARG, "detint_decode_step: null pointer");
    int rc = check_seqs(m, n_seq, seq_ids);
    if (rc) return rc;
    for (int i = 0; i < n_seq; ++i)
        if (m->seq_len[seq_ids[i]] + 1 > m->max_ctx) return fail(DETINT_E_CTX, "decode exceeds max_ctx");
    cudaStream_t s = (cudaStream_t)sp;
    rc = ensure_scratch(m, n_seq);
    if (rc) return rc;
    for (int i = 0; i < n_seq; ++i) {
        rc = ensure_blocks(m, seq_ids[i], m->seq_len[seq_ids[i]] + 1);
        if (rc) return rc;
    }
    rc = sync_block_table(m, s);
    if (rc) return rc;
    {
        int mx = 0;
        for (int i = 0; i < n_seq; ++i) mx = std::max(mx, m->seq_len[seq_ids[i]] + 1);
        m->dec_staged = (m->staged_decode && m->dec_cap > 0 && mx <= m->dec_cap) ? 1 : 0;
        if (m->persistent && n_seq <= 8 && m->st_cfg[n_seq - 1].ok && m->fused_decode && mx <= m->st_scap)
            m->dec_staged = 2;
    }
    const bool graph = m->use_graph && s != nullptr && s != cudaStreamLegacy && s != cudaStreamPerThread;
    if (!graph) {
        std::vector<int32_t> ids(seq_ids, seq_ids + n_seq);
        rc = stage_copies(m, s, {{m->tok_seq, &ids}});
        if (rc) return rc;
        rc = run_forward(m, n_seq, tok, 1, n_seq, nullptr, logits, next_tok, s);
        if (rc) return rc;
    } else {
        char key[128];
        snprintf(key, sizeof key, "%d|%d|%p|%p|%p|", n_seq, m->dec_staged, (const void*)tok, (void*)logits,
                 (void*)next_tok);
        std::string k(key);
        for (int i = 0; i < n_seq; ++i) k += std::to_string(seq_ids[i]) + ",";
        auto it = m->graphs.find(k);
        if (it == m->graphs.end()) {
            // one graph per (batch composition, mode, buffers): bound the cache
            if (m->graphs.size() >= 512) free_graphs(m);
            GraphEntry ge;
            CK(cudaMalloc(&ge.seq_dev, (size_t)n_seq * 4));
            CK(cudaMemcpy(ge.seq_dev, seq_ids, (size_t)n_seq * 4, cudaMemcpyHostToDevice));
            int32_t* saved = m->tok_seq;
            m->tok_seq = ge.seq_dev;
            cudaGraph_t gph;
            CK(cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal));
            rc = run_forward(m, n_seq, tok, 1, n_seq, nullptr, logits, next_tok, s);
            cudaError_t ce = cudaStreamEndCapture(s, &gph);
            m->tok_seq = saved;
            if (rc) {
                if (ce == cudaSuccess) cudaGraphDestroy(gph);
                cudaFree(ge.seq_dev);
                return rc;
            }
            if (ce != cudaSuccess) { cudaFree(ge.seq_dev); return fail(DETINT_E_CUDA, cudaGetErrorString(ce)); }
            ce = cudaGraphInstantiate(&ge.exec, gph, 0);
            cudaGraphDestroy(gph);
            if (ce != cudaSuccess) { cudaFree(ge.seq_dev); return fail(DETINT_E_CUDA, cudaGetErrorString(ce)); }
            it = m->graphs.emplace(k, ge).first;
        }
        CK(cudaGraphLaunch(it->second.exec, s));
    }
    for (int i = 0; i < n_seq; ++i) m->seq_len[seq_ids[i]] += 1;
    return DETINT_OK;
}

// per-device kernel set-up for the entry points that take no model
static int ensure_kernels() {
    static std::mutex mu;
    static int inited[64] = {};
    int dev = 0;
    CK(cudaGetDevice(&dev));
    if (dev < 0 || dev >= 64) return fail(DETINT_E_CUDA, "device ordinal out of range");
    std::lock_guard<std::mutex> lk(mu);
    if (!inited[dev]) { CK(kernels_init()); inited[dev] = 1; }
    return DETINT_OK;
}

int detint_split_w16(const int16_t* W, int8_t* w_hi, uint8_t* w_lo, long long count, detint_stream_t sp) {
    if (!W || !w_hi || !w_lo || count < 1) return fail(DETINT_E_ARG, "detint_split_w16: bad arguments");
    int rc = ensure_kernels();
    if (rc) return rc;
    CK(launch_split_w16(W, w_hi, w_lo, count, (cudaStream_t)sp));
    return DETINT_OK;
}

int detint_gemm_w16(const int8_t* A, const int8_t* w_hi, const uint8_t* w_lo, int64_t* C, int M, int N,
                    int K, detint_stream_t sp) {
    if (!A || !w_hi || !w_lo || !C || M < 1 || N < 1 || K < 1) return fail(DETINT_E_ARG, "detint_gemm_w16: bad arguments");
    if (K % 16 || K > 65536) return fail(DETINT_E_SHAPE, "detint_gemm_w16: K must be a multiple of 16, at most 65536");
    if (((uintptr_t)A & 15) || ((uintptr_t)w_hi & 15) || ((uintptr_t)w_lo & 15))
        return fail(DETINT_E_ARG, "detint_gemm_w16: operands must be 16-byte aligned");
    int rc = ensure_kernels();
    if (rc) return rc;
    CK(launch_gemm_w16(A, w_hi, w_lo, C, M, N, K, standalone_status(), (cudaStream_t)sp));
    return DETINT_OK;
}

int detint_gemm_i8(const int8_t* A, const int8_t* B, int32_t* C, int M, int N, int K,
                   detint_stream_t sp) {
    if (!A || !B || !C || M < 1 || N < 1 || K < 1) return fail(DETINT_E_ARG, "detint_gemm_i8: bad arguments");
    if (K % 16) return fail(DETINT_E_SHAPE, "detint_gemm_i8: K must be a multiple of 16");
    if (((uintptr_t)A & 15) || ((uintptr_t)B & 15)) return fail(DETINT_E_ARG, "detint_gemm_i8: A and B must be 16-byte aligned");
    cudaStream_t s = (cudaStream_t)sp;
    {
        static std::mutex mu;
        static int inited_dev = -1;
        int dev = 0;
        CK(cudaGetDevice(&dev));
        std::lock_guard<std::mutex> lk(mu);
        if (inited_dev != dev) { CK(kernels_init()); inited_dev = dev; }
    }
    Epi e{};
    e.out = C; e.ldo = N; e.status = standalone_status();
    // up to 8 rows: the streaming decode GEMV (weights through the bulk-TMA
    // ring) where the shape fits it; otherwise and beyond 8 rows the tiled
    // GEMM (32/64/128-row tiles, split K for small grids)
    if (M <= 8) {
        cudaError_t ce = launch_sgemv(B, N, K, M, nullptr, nullptr, nullptr, 0, 0, 0, EPI_RAW, e, s,
                                      A, nullptr, nullptr, false);
        if (ce == cudaSuccess) return DETINT_OK;
        if (ce != cudaErrorNotSupported) return fail(DETINT_E_CUDA, cudaGetErrorString(ce));
        cudaGetLastError();
    }
    CK(launch_gemm(A, B, M, N, K, EPI_RAW, e, s));
    return DETINT_OK;
}

int detint_reset_seq(detint_model* m, int seq_id) {
    if (!m) return fail(DETINT_E_ARG, "null model");
    if (seq_id < 0 || seq_id >= m->max_batch) return fail(DETINT_E_SEQ, "sequence id out of range");
    CK(cudaDeviceSynchronize());
    m->seq_len[seq_id] = 0;
    release_blocks(m, seq_id);
    const int32_t z = 0;
    CK(cudaMemcpy(m->seq_len_dev + seq_id, &z, 4, cudaMemcpyHostToDevice));
    return DETINT_OK;
}

int detint_fork_seq(detint_model* m, int src, int dst, int n_tokens, detint_stream_t sp) {
    if (!m) return fail(DETINT_E_ARG, "null model");
    if (src < 0 || src >= m->max_batch || dst < 0 || dst >= m->max_batch || src == dst)
        return fail(DETINT_E_SEQ, "sequence id out of range or equal");
    if (m->seq_len[dst] != 0) return fail(DETINT_E_SEQ, "the destination sequence is not empty");
    if (n_tokens < 0 || n_tokens > m->seq_len[src]) return fail(DETINT_E_ARG, "n_tokens outside the source");
    cudaStream_t s = (cudaStream_t)sp;
    const int full = n_tokens / KV_BLK, part = n_tokens % KV_BLK;
    std::vector<int>& sb = m->seq_blocks[src];
    std::vector<int>& db = m->seq_blocks[dst];
    for (int i = 0; i < full; ++i) {          // whole blocks: shared
        const int b = sb[i];
        ++m->refcnt[b];
        m->bt_host[(size_t)dst * m->mbs + i] = b;
        db.push_back(b);
    }
    if (part) {                               // the partial block: a private copy
        if (m->free_blocks.empty()) { release_blocks(m, dst); return fail(DETINT_E_CTX, "KV block pool exhausted"); }
        const int b = m->free_blocks.back();
        m->free_blocks.pop_back();
        m->refcnt[b] = 1;
        m->bt_host[(size_t)dst * m->mbs + full] = b;
        db.push_back(b);
        const size_t blk = (size_t)m->nkv * KV_BLK * m->d;   // bytes of one block of one layer
        for (int l = 0; l < m->L; ++l) {
            const size_t base = (size_t)l * m->kv_layer_elems;
            CK(cudaMemcpyAsync(m->kcache + base + (size_t)b * blk, m->kcache + base + (size_t)sb[full] * blk,
                               blk, cudaMemcpyDeviceToDevice, s));
            CK(cudaMemcpyAsync(m->vcache + base + (size_t)b * blk, m->vcache + base + (size_t)sb[full] * blk,
                               blk, cudaMemcpyDeviceToDevice, s));
        }
    }
    m->bt_dirty = true;
    int rc = sync_block_table(m, s);
    if (rc) return rc;
    std::vector<int32_t> nl(1, n_tokens);
    rc = stage_copies(m, s, {{m->seq_len_dev + dst, &nl}});
    if (rc) return rc;
    m->seq_len[dst] = n_tokens;
    return DETINT_OK;
}

int detint_seq_len(detint_model* m, int seq_id, int32_t* len) {
    if (!m || !len) return fail(DETINT_E_ARG, "null pointer");
    if (seq_id < 0 || seq_id >= m->max_batch) return fail(DETINT_E_SEQ, "sequence id out of range");
    *len = m->seq_len[seq_id];
    return DETINT_OK;
}

int detint_status(detint_model* m, int32_t* flags, detint_stream_t sp) {
    if (!m) return fail(DETINT_E_ARG, "null model");
    int32_t st[ST_N];
    CK(cudaStreamSynchronize((cudaStream_t)sp));
    CK(cudaMemcpy(st, m->status, sizeof st, cudaMemcpyDeviceToHost));
    CK(cudaMemset(m->status, 0, sizeof st));
    if (flags) memcpy(flags, st, sizeof st);
    if (st[ST_TOKEN]) return DETINT_E_TOKEN;
    if (st[ST_CTX]) return DETINT_E_CTX;
    return DETINT_OK;
}

int detint_set_graph(detint_model* m, int enable) {
    if (!m || (enable != 0 && enable != 1)) return fail(DETINT_E_ARG, "bad argument");
    m->use_graph = enable;
    return DETINT_OK;
}

int detint_set_option(detint_model* m, int option, int value) {
    if (!m) return fail(DETINT_E_ARG, "bad argument");
    if (option == DETINT_OPT_WAIT_TEST) {
        if (value < 0) return fail(DETINT_E_ARG, "bad argument");
        m->st_stall = value;
        free_graphs(m);
        return DETINT_OK;
    }
    if (value != 0 && value != 1) return fail(DETINT_E_ARG, "bad argument");
    if (option == DETINT_OPT_GRAPH) m->use_graph = value;
    else if (option == DETINT_OPT_FUSED_DECODE) { m->fused_decode = value; free_graphs(m); }
    else if (option == DETINT_OPT_TC_PREFILL) m->tc_prefill = value;
    else if (option == DETINT_OPT_STAGED_DECODE) { m->staged_decode = value; free_graphs(m); }
    else if (option == DETINT_OPT_PERSISTENT) { m->persistent = value; free_graphs(m); }
    else return fail(DETINT_E_ARG, "unknown option");
    return DETINT_OK;
}

int detint_model_info(detint_model* m, int32_t* info) {
    if (!m || !info) return fail(DETINT_E_ARG, "null pointer");
    int32_t v[11] = {m->L, m->H, m->nq, m->nkv, m->d, m->F, m->V, m->max_pos, m->qk_norm,
                     m->max_batch, m->max_ctx};
    memcpy(info, v, sizeof v);
    return DETINT_OK;
}

}  // extern "C"
