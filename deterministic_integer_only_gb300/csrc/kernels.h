// Host-side launchers of the detint CUDA kernels (internal to the library).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace detint {

// status word slots (plain stores of 1; never atomics into results)
enum {
    ST_TOKEN = 0,     // a token id outside [0, V) was replaced by 0
    ST_CTX = 1,       // a position beyond the KV capacity was clamped
    ST_SAT_RES = 2,   // a residual add saturated
    ST_SAT_GU = 3,    // a gate/up output saturated at 2^24
    ST_SAT_LOGIT = 4, // a logit saturated
    ST_SAT_QKV = 5,   // a q/k/v output saturated
    ST_TIMEOUT = 6,   // a bounded pipeline wait gave up (results invalid)
    ST_N = 8
};

enum EpiMode { EPI_RAW = 0, EPI_QKV = 1, EPI_RESADD = 2, EPI_SWIGLU = 3, EPI_LOGITS = 4 };

constexpr int KV_BLK = 64;   // tokens per KV-cache block

struct Epi {
    int32_t* out;          // output base (int32)
    int ldo;               // output row stride (elements)
    const int32_t* mt;     // per-token scale mantissa [M]
    const int32_t* kt;     // per-token scale shift [M]
    const int32_t* mc;     // per-weight-row scale mantissa [N]
    int fout;              // output fixed point
    int32_t* status;
    int32_t* pval;         // EPI_LOGITS: argmax partial values [M][npart]
    int32_t* pidx;         // EPI_LOGITS: argmax partial indices [M][npart]
    int npart;
};

// C[m][n] epilogue of sum_k X[m][k] W[n][k]; W row-major [N][K], X [M][K];
// requires K % 64 == 0, M <= 32 per call (rows of X beyond M are not read)
cudaError_t launch_gemv(const int8_t* W, const int8_t* X, int M, int N, int K, int mode,
                        const Epi& ep, cudaStream_t s);

// tiled GEMM for any M (TMA + mma.sync); K % 16 == 0. Grids with fewer
// tiles than SMs split K: raw outputs add partials into a zeroed C; the other
// epilogues need a workspace of ws_elems int32 and tcnt_n zeroed tile
// counters (else they run unsplit)
cudaError_t launch_gemm(const int8_t* A, const int8_t* W, int M, int N, int K, int mode,
                        const Epi& ep, cudaStream_t s, int32_t* wsp = nullptr, size_t ws_elems = 0,
                        int* tcnt = nullptr, int tcnt_n = 0);

cudaError_t launch_embed(const int32_t* tokens, int T, const int32_t* tok_seq, int32_t* tok_pos,
                         const int32_t* seq_len, int decode, int max_pos, const int8_t* E,
                         const uint8_t* Elo, const int32_t* Em, int H, int V, int32_t* h,
                         int32_t* status, cudaStream_t s);

cudaError_t launch_normquant(const int32_t* x, const int32_t* rows, int R, int n,
                             const int16_t* gamma, long long eps, int8_t* q, int32_t* mt,
                             int32_t* kt, cudaStream_t s, bool pdl = false);

cudaError_t launch_actquant(const int32_t* x, int R, int n, int F, int8_t* q, int32_t* mt,
                            int32_t* kt, cudaStream_t s, bool pdl = false);

struct QkvPostArgs {
    const int32_t* qkv;      // [T][(nq + 2 nkv) d] Q12
    const int16_t* q_gamma;
    const int16_t* k_gamma;
    int qk_norm;
    long long eps_qk;
    const int16_t* rope_cos; // [max_pos][d/2]
    const int16_t* rope_sin;
    const int32_t* kvp;      // [nkv][8 + d/2]
    const int32_t* tok_seq;
    const int32_t* tok_pos;
    const int32_t* block_table;
    int mbs;                 // block-table entries per sequence
    int8_t* q8;              // [T][nq][d]
    int32_t* mq;             // [T][nq]
    int32_t* kq;
    int8_t* kc;              // this layer's K cache [NB][nkv][64][d]
    int8_t* vc;              // this layer's V cache [NB][nkv][d][64]
    int T, nq, nkv, d, lg_grp;
};
cudaError_t launch_qkv_post(const QkvPostArgs& a, cudaStream_t s);

struct AttnArgs {
    const int8_t* q8;
    const int32_t* mq;
    const int32_t* kq;
    const int8_t* kc;
    const int8_t* vc;
    const int32_t* block_table;
    int mbs;
    const int32_t* tok_seq;
    const int32_t* tok_pos;
    const int32_t* kvp;
    int32_t* o;              // [T][nq d] Q12
    int T, nq, nkv, d, lg_grp;
    int ctx_cap;             // keys that fit the shared-memory row
    const int32_t* seq_len;  // decode: lengths before this step
    int32_t* status;         // staged decode: timeout flag of its bounded waits
};
cudaError_t launch_attention(const AttnArgs& a, cudaStream_t s);
size_t attention_smem_bytes(int grp, int d, int ctx_cap);

// streaming decode GEMV (M <= 8) with a fused quantisation prologue:
// pro 1 = NormQuant(xin rows, gamma, eps), 2 = ActQuant(xin rows, F),
// 0 = rows already quantised (x8 [M][K] with scales mt/kt).
// Returns cudaErrorNotSupported when the shape does not fit (the caller
// then uses the separate row kernels and launch_gemv).
cudaError_t launch_sgemv(const int8_t* W, int N, int K, int M, const int32_t* xin,
                         const int32_t* rows, const int16_t* gamma, long long eps, int F, int pro,
                         int mode, const Epi& ep, cudaStream_t s, const int8_t* x8 = nullptr,
                         const int32_t* mt = nullptr, const int32_t* kt = nullptr,
                         bool pdl = true,    // pdl: W is immutable (streamed before the wait)
                         int spare_sms = 0); // SMs left free for the next kernel's CTAs, where
                                             // no CTA then holds more row groups
// decode attention fused with the QKV post-processing (one token per sequence)
// staged: the variant that copies the sequence's K/V blocks into shared
// memory before the wait (a.ctx_cap = its staged key capacity, a multiple of
// 64; every sequence's context after the step must fit)
cudaError_t launch_attn_decode(const AttnArgs& a, const QkvPostArgs& qa, cudaStream_t s,
                               bool staged = false);
// dynamic shared memory of the staged variant for a capacity of cap keys
size_t attn_dec_smem(int grp, int d, int cap);

// prefill attention on the int8 tensor pipe: one CTA per (query block, kv
// head); a query block is up to 64 / G consecutive tokens of one sequence
struct PfArgs {
    const int8_t* q8;          // [T][nq][d]
    const int32_t* mq;         // [T][nq]
    const int32_t* kq;
    const int32_t* block_table;
    int mbs;
    const int32_t* qblk;       // [nqb][4]: first token, tokens, sequence, first position
    int nqb;
    const int32_t* kvp;        // [nkv][8 + d/2]
    int32_t* o;                // [T][nq d] Q12
    int nq, nkv, lg_grp;
    int krow0, vrow0;          // this layer's first row in the K / V^T cache maps
    int32_t* status;
};
// tensor maps over the whole K cache ([units * 64][d] bytes) and V^T cache
// ([units * d][64] bytes), units = layers * blocks * kv heads
cudaError_t make_kv_maps(CUtensorMap* kmap, CUtensorMap* vmap, const int8_t* kc,
                         const int8_t* vc, long long units, int d);
cudaError_t launch_attn_prefill(const PfArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                                int d, cudaStream_t s);
constexpr int PF_ROWS = 64;   // query rows (token x q head) per prefill attention CTA

// one decode step in one cooperative launch (k_decode_step.cuh)
// the layer's weights, scales and caches (a device array of these)
struct StepLayer {
    const int8_t *w_qkv, *w_o, *w_gu, *w_d;
    const int32_t *m_qkv, *m_o, *m_gu, *m_d, *kvp;
    const int16_t *attn_gamma, *ffn_gamma, *q_gamma, *k_gamma;
    int8_t *kc, *vc;
};

struct StepArgs {
    const StepLayer* layers;
    int L, T, H, nq, nkv, d, F, V, lg_grp, lg_nkv, qk_norm, max_pos, mbs;
    long long eps_h, eps_qk;
    const int8_t* embed;
    const int32_t* embed_m;
    const int16_t *final_gamma, *rope_cos, *rope_sin;
    const int32_t* block_table;
    const int32_t* tokens;       // [T] this step's input ids (may alias next_tok)
    const int32_t* tok_seq;      // [T] sequence of each token
    int32_t* seq_len;            // [max_batch], advanced at the end of the step
    // tagged rows (value | tag << 32): [8][H], [8][nqkv], [8][nq d], [8][F], [NG][8][2]
    unsigned long long *xh, *xqkv, *xo, *xs, *xpart;
    unsigned* ctl;               // [0] base tag of the next step, [1] base tag of a step that timed out
    const int32_t* rows;         // [5][NG + 1]: first weight row of each GEMV CTA per GEMV kind
    int32_t *logits, *next_tok, *status;
    int NG, NA, ipc, lg_ns;      // GEMV CTAs, attention CTAs, items per attention CTA, log2 ring slots
    int cap;                     // staged keys per attention item (a multiple of 64)
    int scap;                    // score-row capacity (a multiple of 16 >= every context)
    int spin;                    // polls before a wait gives up
    int stall;                   // > 0: the final wait expects a tag nobody writes, bounded by stall polls
    // dynamic shared memory of a GEMV CTA: weight ring, int8 tile [T][XP],
    // int32 input rows [T][XP], gamma [H], owned residual
    // rows, the layer table [L], the CTA's channel scales of every phase
    // (ms per layer for the four layer phases, then the lm_head rows)
    int off_x8, off_xin, off_gs, off_hown, off_lay, off_mct;
    int ms;
};
constexpr int STEP_THREADS = 320;
constexpr int STEP_SLOT = 16384;        // weight ring slot bytes
constexpr int STEP_HOWN = 64;           // residual rows a GEMV CTA owns at most
constexpr int STEP_NP = 64;             // tagged pairs per thread a prologue can track
// weight rows per ring slot for reduction length K (<= 16)
__host__ __device__ inline int step_rows_per_slot(int K) {
    int q = 16;
    while (q * K > STEP_SLOT) --q;
    return q;
}
// an attention item's parameter rows in shared memory: the kv head's
// parameters [8 + d/2] int32, q and k gammas [d] int16, this position's RoPE
// cos and sin rows [d/2] int16, the sequence's block-table row [mbs] int32
__host__ __device__ inline int step_aux_bytes(int d, int mbs) {
    return (8 + d / 2) * 4 + 4 * d + 2 * d + ((mbs * 4 + 15) & ~15);
}
// attention CTA shared memory: per item K [cap][d], V^T [cap/64][d][64] and
// the parameter rows; then q [G][d], scores [G][scap] int32, E_lo/E_hi
// [G][scap], P.V limbs [G][d][2]
__host__ __device__ inline size_t step_att_bytes(int G, int d, int cap, int ipc, int scap, int aux) {
    return (size_t)ipc * (2 * (size_t)cap * d + aux) + (size_t)G * d + (size_t)G * scap * 6 + (size_t)G * d * 8;
}
// d: head_dim, grp: q heads per kv head; false for shapes without an instantiation
bool decode_step_supported(int d, int grp);
// sets the kernel's shared-memory limit; true when one CTA of smem bytes fits an SM
bool decode_step_fits(int d, int grp, size_t smem);
cudaError_t launch_decode_step(const StepArgs& a, int grid, size_t smem, cudaStream_t s);

cudaError_t launch_argmax_final(const int32_t* pval, const int32_t* pidx, int rows, int npart,
                                int32_t* next_tok, const int32_t* tok_seq, int32_t* seq_len,
                                cudaStream_t s, bool pdl = false);

// exact int8 x int16 GEMM from two int8 weight limbs (k_gemm_w16.cuh):
// C int64 [M][N]; K % 16 == 0, K <= 65536, operands 16-byte aligned
cudaError_t launch_gemm_w16(const int8_t* A, const int8_t* Wh, const uint8_t* Wl, int64_t* C, int M,
                            int N, int K, int32_t* status, cudaStream_t s);
cudaError_t launch_split_w16(const int16_t* W, int8_t* hi, uint8_t* lo, long long n, cudaStream_t s);
// exact-mode epilogue of a limb GEMM's int64 output C [M][N] (EPI_QKV,
// EPI_RESADD, EPI_SWIGLU of interleaved gate/up rows, EPI_LOGITS with
// argmax partials): the 128-bit requantisation with channel shift 30
cudaError_t launch_epi_w16(const int64_t* C, int M, int N, int mode, const Epi& ep, cudaStream_t s);
// a status word in device memory for the entry points that take no model
int32_t* standalone_status();

cudaError_t kernels_init();

}  // namespace detint
