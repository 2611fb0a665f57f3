// Integer-pipe peak loops: the measured denominator of the int8 GEMM and
// prefill roofline fractions. The tcgen05 tensor cores have no integer kind
// on sm_103a, so the int8 rate this GPU offers is that of warp-level
// mma.sync m16n8k32 s8 and of dp4a; these loops keep independent operations
// in flight on register operands only (no memory traffic) and store one
// checksum per thread so that nothing is eliminated.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/detint.h"

namespace {

constexpr int PK_THREADS = 256;
constexpr int PK_CHAINS = 8;          // independent accumulators per warp / thread

__global__ void __launch_bounds__(PK_THREADS) k_peak_mma(int iters, int32_t* sink) {
    const int t = threadIdx.x;
    int a0 = 0x01020304 * (t + 1), a1 = a0 ^ 0x55, a2 = a0 + 7, a3 = a0 - 9;
    int b0 = 0x0a0b0c0d ^ t, b1 = b0 + 3;
    int c[PK_CHAINS][4];
#pragma unroll
    for (int k = 0; k < PK_CHAINS; ++k) c[k][0] = c[k][1] = c[k][2] = c[k][3] = t ^ k;
    for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int k = 0; k < PK_CHAINS; ++k)
            asm volatile(
                "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                "{%0,%1,%2,%3};"
                : "+r"(c[k][0]), "+r"(c[k][1]), "+r"(c[k][2]), "+r"(c[k][3])
                : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
#pragma unroll
    for (int k = 0; k < PK_CHAINS; ++k)
        sink[(blockIdx.x * PK_THREADS + t) * PK_CHAINS + k] = c[k][0] ^ c[k][1] ^ c[k][2] ^ c[k][3];
}

__global__ void __launch_bounds__(PK_THREADS) k_peak_dp4a(int iters, int32_t* sink) {
    const int t = threadIdx.x;
    const int b = 0x0a0b0c0d ^ t;
    int a[PK_CHAINS], c[PK_CHAINS];
#pragma unroll
    for (int k = 0; k < PK_CHAINS; ++k) {
        a[k] = __byte_perm(0x01020304 ^ t, k, 0x3210);     // one operand word per chain
        c[k] = t ^ k;
    }
#pragma unroll 1
    for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int k = 0; k < PK_CHAINS; ++k)
            asm volatile("dp4a.s32.s32 %0, %1, %2, %0;" : "+r"(c[k]) : "r"(a[k]), "r"(b));
    }
#pragma unroll
    for (int k = 0; k < PK_CHAINS; ++k) sink[(blockIdx.x * PK_THREADS + t) * PK_CHAINS + k] = c[k];
}

}  // namespace

extern "C" int detint_int8_peak_loop(int kind, int blocks, int iters, int32_t* sink, long long* ops,
                                     detint_stream_t stream) {
    if ((kind != 0 && kind != 1) || blocks < 1 || iters < 1 || !sink || !ops) return DETINT_E_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    const long long threads = (long long)blocks * PK_THREADS;
    if (kind == 0) {
        // a warp's mma.sync m16n8k32: 16 x 8 x 32 multiply-adds = 8192 integer operations
        k_peak_mma<<<blocks, PK_THREADS, 0, s>>>(iters, sink);
        *ops = (threads / 32) * (long long)iters * PK_CHAINS * 8192;
    } else {
        // a thread's dp4a: 4 multiply-adds = 8 integer operations
        k_peak_dp4a<<<blocks, PK_THREADS, 0, s>>>(iters, sink);
        *ops = threads * (long long)iters * PK_CHAINS * 8;
    }
    return cudaGetLastError() == cudaSuccess ? DETINT_OK : DETINT_E_CUDA;
}
