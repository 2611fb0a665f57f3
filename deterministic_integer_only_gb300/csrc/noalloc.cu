// detint_argmax_noalloc: the two-stage tie-low argmax with its per-block
// partial results kept in a fixed device array instead of allocated memory.
//
// Who needs it: code that runs where device allocation is not allowed or
// not possible — inside a CUDA-graph capture that must not allocate, in a
// host callback or signal-style context, or under a memory budget enforced
// by an embedding application that owns every allocation. Such callers pass
// their logits and output buffer and this entry point allocates nothing
// (no cudaMalloc, cudaFree, or allocating library routine).
//
// Stage 1: block (p, r) finds the largest value of row r within columns
// [p*CHUNK, (p+1)*CHUNK), lowest column on ties, and writes it to the
// partial slot (r, p). Stage 2: one block per row reduces its partial slots
// the same way. Every slot stage 2 reads was written by stage 1 of the same
// call, so nothing needs clearing between calls.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/detint.h"

namespace {

constexpr int NA_CHUNK = 4096;                      // columns per stage-1 block
constexpr int NA_MAX_ROWS = DETINT_ARGMAX_NOALLOC_MAX_ROWS;
constexpr int NA_MAX_PARTS = DETINT_ARGMAX_NOALLOC_MAX_COLS / NA_CHUNK;

// the scratch: [value, index] x NA_MAX_PARTS x NA_MAX_ROWS int32 (128 KB),
// resident on every device that loads this library until process exit
static __device__ __align__(256) int32_t g_argmax_scratch[2 * NA_MAX_ROWS * NA_MAX_PARTS];

__device__ __forceinline__ void na_better(int& bv, int& bi, int v, int i) {
    if (v > bv || (v == bv && i < bi)) { bv = v; bi = i; }
}

__device__ __forceinline__ void na_block_reduce(int& bv, int& bi, int* sv, int* si) {
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        const int v = __shfl_xor_sync(0xffffffffu, bv, o);
        const int i = __shfl_xor_sync(0xffffffffu, bi, o);
        na_better(bv, bi, v, i);
    }
    if ((threadIdx.x & 31) == 0) { sv[threadIdx.x >> 5] = bv; si[threadIdx.x >> 5] = bi; }
    __syncthreads();
    if (threadIdx.x == 0) {
        bv = sv[0]; bi = si[0];
        for (int w = 1; w < 8; ++w) na_better(bv, bi, sv[w], si[w]);
    }
}

__global__ void __launch_bounds__(256) k_na_partial(const int32_t* __restrict__ logits, int n,
                                                    int nparts, int32_t* __restrict__ scratch) {
    __shared__ int sv[8], si[8];
    const int p = blockIdx.x, r = blockIdx.y;
    const int c0 = p * NA_CHUNK;
    const int c1 = min(n, c0 + NA_CHUNK);
    const int32_t* row = logits + (size_t)r * n;
    int bv = -2147483647 - 1, bi = 2147483647;
    for (int c = c0 + (int)threadIdx.x; c < c1; c += 256) na_better(bv, bi, row[c], c);
    na_block_reduce(bv, bi, sv, si);
    if (threadIdx.x == 0) {
        scratch[2 * ((size_t)r * nparts + p)] = bv;
        scratch[2 * ((size_t)r * nparts + p) + 1] = bi;
    }
}

__global__ void __launch_bounds__(256) k_na_final(const int32_t* __restrict__ scratch, int nparts,
                                                  int32_t* __restrict__ out) {
    __shared__ int sv[8], si[8];
    const int r = blockIdx.x;
    int bv = -2147483647 - 1, bi = 2147483647;
    for (int p = threadIdx.x; p < nparts; p += 256)
        na_better(bv, bi, scratch[2 * ((size_t)r * nparts + p)],
                  scratch[2 * ((size_t)r * nparts + p) + 1]);
    na_block_reduce(bv, bi, sv, si);
    if (threadIdx.x == 0) out[r] = bi;
}

// device address of g_argmax_scratch, looked up once per device with that
// device current (the host-side name is only a stand-in for the symbol)
constexpr int NA_MAX_DEVICES = 64;
std::mutex g_na_mu;
int32_t* g_na_ptr[NA_MAX_DEVICES] = {};

int na_scratch(int32_t** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= NA_MAX_DEVICES) return DETINT_E_CUDA;
    std::lock_guard<std::mutex> lk(g_na_mu);
    if (!g_na_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_argmax_scratch) != cudaSuccess || !p) return DETINT_E_CUDA;
        g_na_ptr[dev] = (int32_t*)p;
    }
    *out = g_na_ptr[dev];
    return DETINT_OK;
}

}  // namespace

extern "C" int detint_argmax_noalloc(const int32_t* logits, int rows, int n, int32_t* out,
                                     detint_stream_t stream) {
    if (!logits || !out || rows < 1 || n < 1) return DETINT_E_ARG;
    if (rows > NA_MAX_ROWS || n > DETINT_ARGMAX_NOALLOC_MAX_COLS) return DETINT_E_SHAPE;
    int32_t* scratch = nullptr;
    int rc = na_scratch(&scratch);
    if (rc != DETINT_OK) return rc;
    cudaStream_t s = (cudaStream_t)stream;
    const int nparts = (n + NA_CHUNK - 1) / NA_CHUNK;
    k_na_partial<<<dim3(nparts, rows), 256, 0, s>>>(logits, n, nparts, scratch);
    k_na_final<<<rows, 256, 0, s>>>(scratch, nparts, out);
    return cudaGetLastError() == cudaSuccess ? DETINT_OK : DETINT_E_CUDA;
}
