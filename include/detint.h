/*
 * detint — C ABI of the GB300 (sm_103a) integer-only LLM decoder.
 *
 * The library runs the integer-only decoder forward pass of a Qwen3- or
 * Llama-shaped model: every operation from input ids to int32 logits is
 * exact integer arithmetic, so logits and greedy tokens are bit-identical
 * across batch composition, prefill vs decode and backends ("DetLLM — Fully
 * Deterministic LLM Inference", intro; DetLLM blog "Eliminating
 * Nondeterminism in LLM Inference with Integer-Only Arithmetic", section
 * "DetLLM"). The user-level API of the pages is
 * `IntQwen3(path, backend).generate(ids, max_new, use_graph)` (README,
 * "Usage"); its C counterpart is detint_load + detint_prefill +
 * detint_decode_step.
 *
 * Conventions
 *  - Streams are `cudaStream_t` values passed as `detint_stream_t`. All
 *    compute calls are stream-ordered and asynchronous; they return after
 *    enqueueing work. The legacy default stream (NULL) is accepted but CUDA
 *    graphs are only used on a non-default stream.
 *  - Device pointers are owned by the caller unless stated. The model owns
 *    its weights, KV cache and scratch, released by detint_free.
 *  - Every call returns 0 (DETINT_OK) or a positive DETINT_E_* code; nothing
 *    aborts. detint_strerror names a code; detint_last_error gives the
 *    detail of the last failure in this process.
 *  - Conditions only the device can see (a token id >= vocab, a saturated
 *    residual/logit) are recorded in a status word read by detint_status.
 */
#ifndef DETINT_H
#define DETINT_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct detint_model detint_model;
typedef struct CUstream_st* detint_stream_t;   /* == cudaStream_t */

enum {
    DETINT_OK = 0,
    DETINT_E_ARG = 1,       /* null pointer, bad count or option */
    DETINT_E_SHAPE = 2,     /* unsupported sizes (e.g. K not a multiple of 16) */
    DETINT_E_TOKEN = 3,     /* status: a token id outside [0, vocab) */
    DETINT_E_CTX = 4,       /* a sequence would exceed max_ctx */
    DETINT_E_ARTIFACT = 5,  /* unreadable or malformed artifact file */
    DETINT_E_SHA = 6,       /* artifact SHA-256 differs from its .sha256 file */
    DETINT_E_CUDA = 7,      /* a CUDA call failed */
    DETINT_E_OOM = 8,       /* device allocation failed */
    DETINT_E_SEQ = 9,       /* sequence id outside [0, max_batch) or repeated */
    DETINT_E_SAT = 10       /* status: a saturation was recorded */
};

/* Load an artifact (format: the artifact section of the arithmetic
 * specification; header, int8 weights, dyadic channel scales, int16 gammas,
 * int16 Q14 RoPE tables, per-kv-head fixed K/V scales) after checking its
 * SHA-256 against `<path>.sha256` (README, "Demo": comparisons are valid only
 * for the same artifact hash). Allocates the weights, a paged int8 KV cache
 * for `max_batch` sequences of up to `max_ctx` positions, and scratch.
 * `max_ctx` <= the artifact's RoPE table length. Synchronous.
 * Errors: ARG, ARTIFACT, SHA, OOM, CUDA, SHAPE. */
int detint_load(const char* artifact_path, int max_batch, int max_ctx, detint_stream_t s,
                detint_model** out);

/* Prefill: append a ragged batch of prompts to the KV caches of `n_seq`
 * distinct sequences and return the logits of each sequence's last new
 * position (DetLLM blog, "DetLLM": prefill and decode see the same cached
 * bits). seq_ids: host int32[n_seq], each in [0, max_batch), distinct.
 * cu_lens: host int32[n_seq + 1] (a host array, not a device one: the
 * library plans KV blocks and attention query blocks from the lengths
 * before it enqueues any kernel), cu_lens[0] = 0, non-decreasing, each
 * length >= 1; tokens of sequence i are tokens[cu_lens[i] .. cu_lens[i+1]).
 * tokens: device int32[cu_lens[n_seq]]. logits: device int32[n_seq][vocab]
 * or NULL. next_tok: device int32[n_seq] (argmax, ties to the lowest id).
 * Positions continue from each sequence's current length, so a prompt may
 * be split across calls (split prefill) with identical results.
 * Errors: ARG, SEQ, CTX, CUDA, OOM. */
int detint_prefill(detint_model* m, int n_seq, const int32_t* seq_ids, const int32_t* cu_lens,
                   const int32_t* tokens, int32_t* logits, int32_t* next_tok, detint_stream_t s);

/* One greedy decode step: one new token per sequence, appended to its KV
 * cache, then int32 logits and the tie-low argmax of the new position
 * (DetLLM blog, "DetLLM": decode reads the same cached integers a prefill
 * writes, and argmax prefers the smallest token id on ties; README, "Usage":
 * generate(ids, max_new, use_graph) is a prefill followed by such steps).
 * seq_ids: host int32[n_seq]; tok: device int32[n_seq]; logits: device
 * int32[n_seq][vocab] or NULL; next_tok: device int32[n_seq] (may alias
 * tok). With graphs enabled (default) the step is one CUDA-graph launch,
 * re-captured when the sequence set or a pointer changes.
 * Errors: ARG, SEQ, CTX, CUDA. */
int detint_decode_step(detint_model* m, int n_seq, const int32_t* seq_ids, const int32_t* tok,
                       int32_t* logits, int32_t* next_tok, detint_stream_t s);

/* Exact int8 x int8 -> int32 GEMM: C[m][n] = sum_k A[m][k] * B[n][k].
 * A: device int8 [M][K] row-major; B: device int8 [N][K] row-major (the
 * weight layout); C: device int32 [M][N]. M, N >= 1; K >= 16 and a multiple
 * of 16; A, B 16-byte aligned. The integer GEMM is the one operation the
 * pages dispatch per device (README, "Layout": int_gemm). Errors: ARG,
 * SHAPE, CUDA. */
int detint_gemm_i8(const int8_t* A, const int8_t* B, int32_t* C, int M, int N, int K,
                   detint_stream_t s);

/* Tie-low argmax of `rows` int32 rows of length `n` (device, row-major) into
 * out[rows] (device int32), for callers that cannot allocate device memory:
 * code running inside a stream capture that must stay allocation-free, in a
 * host callback, or under an application that owns every allocation. This
 * entry point calls no cudaMalloc/cudaFree or allocating library routine;
 * its per-block partial results live in one fixed device array of 128 KB
 * that every GPU loading this library holds until the process exits.
 * Limits: rows <= DETINT_ARGMAX_NOALLOC_MAX_ROWS, n <=
 * DETINT_ARGMAX_NOALLOC_MAX_COLS; larger sizes return DETINT_E_SHAPE.
 * The first call on a device looks up that array's device address (with the
 * device current), so make it before any stream capture. All calls share the
 * one array: calls that overlap on the GPU (different streams, no ordering)
 * race and give wrong results; calls ordered on one stream are safe. Each
 * call writes every partial slot it reads, so no clearing is needed.
 * Ties go to the lowest column, as in the decode steps' token choice. The
 * pages have no counterpart to this entry point.
 * Errors: ARG, SHAPE, CUDA. */
#define DETINT_ARGMAX_NOALLOC_MAX_ROWS 64
#define DETINT_ARGMAX_NOALLOC_MAX_COLS 1048576
int detint_argmax_noalloc(const int32_t* logits, int rows, int n, int32_t* out, detint_stream_t s);

/* Forget a sequence's cached context (length back to 0) and return its KV
 * blocks to the pool. No passage of the pages defines this: it is library
 * housekeeping for reusing a sequence slot (the scheduler cases of the
 * BitExact LLM post, "What the checks actually compare": preemption then
 * recomputation, start from an emptied slot). Synchronises the device
 * first. Errors: ARG, SEQ, CUDA. */
int detint_reset_seq(detint_model* m, int seq_id);

/* Current length of a sequence (host-side bookkeeping). */
int detint_seq_len(detint_model* m, int seq_id, int32_t* len);

/* Read and clear the device status word after synchronising `s`.
 * flags: host int32[8] or NULL; slots 0 token id out of range, 1 context
 * clamp, 2 residual saturation, 3 gate/up saturation, 4 logit saturation,
 * 5 q/k/v saturation, 6 a bounded wait of a kernel timed out (its results
 * are invalid). Returns DETINT_E_TOKEN if slot 0 is set, else
 * DETINT_E_CTX if slot 1 is set, else DETINT_OK. */
int detint_status(detint_model* m, int32_t* flags, detint_stream_t s);

/* Enable (1, default) or disable (0) CUDA-graph replay of decode steps
 * (README, "Usage": use_graph). */
int detint_set_graph(detint_model* m, int enable);

/* Exact int8 x int16 GEMM for wide-weight ("exact mode") linear layers:
 * C[m][n] = sum_k A[m][k] W[n][k] in int64, with int8 activations A
 * [M][K] and int16 weights W [N][K] given as two int8 limbs,
 * W = 256 * w_hi + w_lo (w_hi int8, w_lo uint8; detint_split_w16 makes them).
 * Both limb products run on the int8 tensor pipe in one pass and are
 * combined exactly (BitExact LLM post, "Fix the arithmetic, not just the
 * random seed": products of split integer limbs combined in wider
 * accumulators; its exact mode keeps wide weights). Device pointers, all
 * 16-byte aligned, caller-owned; K % 16 == 0 and K <= 65536. Asynchronous
 * on s. Errors: ARG, SHAPE, CUDA. */
int detint_gemm_w16(const int8_t* A, const int8_t* w_hi, const uint8_t* w_lo, int64_t* C, int M, int N,
                    int K, detint_stream_t s);
/* w_hi[i] = W[i] >> 8 (floor), w_lo[i] = W[i] & 255, for count elements
 * (device pointers). Errors: ARG, CUDA. */
int detint_split_w16(const int16_t* W, int8_t* w_hi, uint8_t* w_lo, long long count, detint_stream_t s);

/* Start sequence dst (which must be empty) with the first n_tokens positions
 * of sequence src, without recomputing them: whole 64-token KV blocks are
 * shared by reference count, the partial last block is copied, and later
 * appends to either sequence go to blocks of its own. Continuing dst gives
 * the same logits, bit for bit, as prefilling the same tokens afresh
 * (scheduler invariance: BitExact LLM post, "What the checks actually
 * compare" lists shared prefixes among the tested scheduler changes).
 * Stream-ordered on s. Errors: ARG, SEQ (ids out of range or equal, dst not
 * empty), CTX (block pool exhausted), CUDA. */
int detint_fork_seq(detint_model* m, int src, int dst, int n_tokens, detint_stream_t s);

/* Integer sampling parameters of one row (see detint_sample). */
typedef struct {
    uint64_t seed;      /* SplitMix64 seed */
    uint64_t counter;   /* draw index: output counter + 1 of the generator */
    int32_t inv_temp;   /* Q16 of 1/temperature, 0 .. 2^20 (65536: T = 1; 0: uniform) */
    int32_t top_k;      /* keep the top_k largest logits (0 or >= n: off) */
    int32_t top_p;      /* Q16 nucleus mass, 1 .. 65536 (65536: off) */
    int32_t reserved;   /* set to 0 */
} detint_sampling_t;

/* Draw one token per logits row with integer arithmetic only: weights
 * E_i = exp2q(u_i - max u), u = the logit in base-2 Q10 at the temperature;
 * the top_k largest logits (ties by lower index), then the shortest prefix
 * of them (logit order) holding top_p of their weight plus its boundary ties;
 * then t = floor(r S / 2^64) with r = SplitMix64(seed, counter) and S the
 * kept weight, and the token is the first index (index order) whose
 * cumulative kept weight exceeds t. The pages ask for integer sampling rules
 * and deterministic sampling (BitExact LLM post, "Fix the arithmetic, not
 * just the random seed"; "Reproducibility has a cost") without an algorithm;
 * this is the reading in the arithmetic specification, section "Integer
 * sampling". top_k = 1 gives the tie-low argmax for every seed.
 * logits: device int32 [rows][n] (caller-owned); params: host [rows];
 * out: device int32 [rows]. Asynchronous on s; allocates nothing.
 * Errors: ARG (null pointer, rows or n < 1, a parameter out of range), CUDA. */
int detint_sample(const int32_t* logits, int rows, int n, const detint_sampling_t* params,
                  int32_t* out, detint_stream_t s);

/* Options: DETINT_OPT_GRAPH (1 = replay decode steps as CUDA graphs, the
 * default; same as detint_set_graph), DETINT_OPT_FUSED_DECODE (1 = decode
 * batches of up to 8 sequences through the fused streaming kernels, the
 * default; 0 = through the separate row kernels) and DETINT_OPT_TC_PREFILL
 * (1 = prefill attention on the int8 tensor pipe in two sweeps over the keys,
 * the default where head_dim is 64 or 128; 0 = the per-token attention
 * kernel) and DETINT_OPT_STAGED_DECODE (1 = fused decode attention with the
 * sequence's cached K/V copied into shared memory before the step's data is
 * ready, the default while every context fits that copy; 0 = the attention
 * kernel that reads the cache from global memory) and DETINT_OPT_PERSISTENT
 * (1 = a fused decode step of up to 8 sequences runs as one cooperative
 * launch of one CTA per SM whose phases hand rows to one another as tagged
 * words, where the shape fits; 0 = one kernel per phase). Every setting gives
 * bit-identical results.
 * DETINT_OPT_WAIT_TEST (value >= 0) exercises the failure path of the
 * one-launch step's bounded waits: while it is positive, the step's final
 * wait expects a tag that no CTA writes and gives up after `value` polls,
 * so the step ends with status slot 6 (a wait timed out) set and an invalid
 * token, without hanging; 0 (the default) turns it off. No passage of the
 * pages: a test hook of the library's failure detection.
 * Errors: ARG. */
enum { DETINT_OPT_GRAPH = 0, DETINT_OPT_FUSED_DECODE = 1, DETINT_OPT_TC_PREFILL = 2,
       DETINT_OPT_STAGED_DECODE = 3, DETINT_OPT_PERSISTENT = 4, DETINT_OPT_WAIT_TEST = 5 };
int detint_set_option(detint_model* m, int option, int value);

/* Integer-pipe peak loop, the measured denominator of the int8 GEMM and
 * prefill roofline fractions (no passage of the pages: a measurement
 * routine). kind 0: blocks x 256 threads of independent mma.sync m16n8k32
 * s8 operations on register operands; kind 1: the same with dp4a. Each
 * thread runs `iters` rounds and stores its 8 accumulators' checksums
 * into sink (device int32[blocks * 256 * 8], caller-owned); *ops (host) receives the integer
 * operations the launch performs (2 per multiply-add). Time it with events
 * on `s`. Asynchronous; allocates nothing. Errors: ARG, CUDA. */
int detint_int8_peak_loop(int kind, int blocks, int iters, int32_t* sink, long long* ops,
                          detint_stream_t s);

/* Shape of the loaded model: info[0..9] = n_layers, hidden, n_q, n_kv,
 * head_dim, ffn, vocab, max_pos, qk_norm, max_batch; info[10] = max_ctx. */
int detint_model_info(detint_model* m, int32_t* info);

/* Release everything the model owns. NULL is a no-op. No passage of the
 * pages: library housekeeping. */
void detint_free(detint_model* m);

/* A static English name of an error code ("unknown error" for other
 * values); detint_last_error gives the detail of this thread's last
 * failure. No passage of the pages: library housekeeping. */
const char* detint_strerror(int code);
const char* detint_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* DETINT_H */
