// Exact GEMM with 16-bit weights as two int8 limbs (BitExact LLM post,
// "Fix the arithmetic, not just the random seed": matrix products split
// values into small integer limbs, compute partial products and combine them
// in wider accumulators; its exact mode keeps wide weights against
// fixed-point activations).
//
// C[m][n] = sum_k A[m][k] W[n][k] in int64, with int8 activations A and
// int16 weights stored as W = 256 W_hi + W_lo (W_hi int8 = W >> 8, W_lo the
// low byte as uint8). Both limb products run on the int8 tensor pipe in one
// pass over K: s8 x s8 for the high limb, s8 x u8 for the low limb, two int32
// accumulators per output (exact for K <= 65536: |a w_hi| <= 2^14 and
// |a w_lo| < 2^15 per term), combined as 256 acc_hi + acc_lo in int64.
// Tiles: 64 rows x 128 columns x 128 k, A / W_hi / W_lo by 2D TMA with the
// 128-byte swizzle into a 3-stage ring; 8 MMA warps of 64 x 16 and one
// producer warp. Grids smaller than the SM count split K, adding int64
// partials into a zeroed C (exact, so the order of the adds does not matter).
#pragma once
#include <cuda.h>
#include "kernels.h"
#include "ptx.cuh"

namespace detint {

constexpr int W16_BM = 64;
constexpr int W16_STAGE = (W16_BM + 2 * GM_BN) * GM_BK;   // A + W_hi + W_lo tiles, 40 KB
constexpr size_t W16_SMEM = (size_t)GM_STAGES * W16_STAGE + 1024;

// the limbs of little-endian int16 weights are their bytes: the high limb
// (W >> 8, floor, as int8) is the high byte and the low limb the low byte,
// so the split only moves bytes
// Thread i moves the 16 weights from 16 i on (the launch covers n with
// n / 16 threads rounded up, so no thread loops: a loop with a run-time stride
// would have its trip count formed by a division)
constexpr int SPLIT_PER_THREAD = 16;
__global__ void k_split_w16(const uint8_t* __restrict__ W, uint8_t* __restrict__ hi,
                            uint8_t* __restrict__ lo, long long n) {
    const long long i0 = ((long long)blockIdx.x * blockDim.x + threadIdx.x) * SPLIT_PER_THREAD;
#pragma unroll
    for (int k = 0; k < SPLIT_PER_THREAD; ++k) {
        const long long i = i0 + k;
        if (i < n) {
            lo[i] = W[2 * i];
            hi[i] = W[2 * i + 1];
        }
    }
}

__device__ __forceinline__ void mma_s8u8(int (&c)[4], int a0, int a1, int a2, int a3, int b0, int b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.s32.s8.u8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+r"(c[0]), "+r"(c[1]), "+r"(c[2]), "+r"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__global__ void __launch_bounds__(GM_THREADS, 1)
    k_gemm_w16(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapH,
               const __grid_constant__ CUtensorMap mapL, int M, int N, int K, int64_t* C, int ksl,
               int32_t* status) {
    extern __shared__ unsigned char wsm_raw[];
    __shared__ unsigned long long full[GM_STAGES], empty[GM_STAGES];
    unsigned char* sm = (unsigned char*)(((uintptr_t)wsm_raw + 1023) & ~(uintptr_t)1023);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int m0 = blockIdx.y * W16_BM, n0 = blockIdx.x * GM_BN;
    const int nk_all = (K + GM_BK - 1) / GM_BK;
    const int kt0 = blockIdx.z * ksl;
    const int nk = min(nk_all, kt0 + ksl) - kt0;

    if (tid == 0) {
        for (int s = 0; s < GM_STAGES; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 8);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    if (warp == 8) {
        if (lane == 0) {
            for (int kt = 0; kt < nk; ++kt) {
                const int s = kt % GM_STAGES;
                if (kt >= GM_STAGES && !mbar_wait(smem_u32(&empty[s]), ((kt / GM_STAGES) - 1) & 1))
                    status[ST_TIMEOUT] = 1;
                const uint32_t fb = smem_u32(&full[s]);
                mbar_arrive_expect_tx(fb, W16_STAGE);
                const uint32_t base = smem_u32(sm + (size_t)s * W16_STAGE);
                const int kx = (kt0 + kt) * GM_BK;
                tma_load_2d(base, &mapA, kx, m0, fb);
                tma_load_2d(base + W16_BM * GM_BK, &mapH, kx, n0, fb);
                tma_load_2d(base + (W16_BM + GM_BN) * GM_BK, &mapL, kx, n0, fb);
            }
        }
        return;
    }

    const int wn = warp;                          // 8 warps along N, 16 columns each
    const int g = lane >> 2, tq = lane & 3;
    const int mi = lane >> 3, ri = lane & 7;
    int ah[4][2][4], al[4][2][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 2; ++b)
#pragma unroll
            for (int e = 0; e < 4; ++e) ah[a][b][e] = al[a][b][e] = 0;

    for (int kt = 0; kt < nk; ++kt) {
        const int s = kt % GM_STAGES;
        if (!mbar_wait(smem_u32(&full[s]), (kt / GM_STAGES) & 1)) status[ST_TIMEOUT] = 1;
        const uint32_t tA = smem_u32(sm + (size_t)s * W16_STAGE);
        const uint32_t tH = tA + W16_BM * GM_BK;
        const uint32_t tL = tH + GM_BN * GM_BK;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            int af[4][4], bh[2][2], bl[2][2];
#pragma unroll
            for (int mt = 0; mt < 4; ++mt) {
                const int r = mt * 16 + ri + 8 * (mi & 1);
                ldsm_x4(tA + swz(r, 2 * kk + (mi >> 1)), af[mt][0], af[mt][1], af[mt][2], af[mt][3]);
            }
            {
                const int r = wn * 16 + ri + 8 * (mi >> 1);
                ldsm_x4(tH + swz(r, 2 * kk + (mi & 1)), bh[0][0], bh[0][1], bh[1][0], bh[1][1]);
                ldsm_x4(tL + swz(r, 2 * kk + (mi & 1)), bl[0][0], bl[0][1], bl[1][0], bl[1][1]);
            }
#pragma unroll
            for (int mt = 0; mt < 4; ++mt)
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    mma_s8(ah[mt][nt], af[mt][0], af[mt][1], af[mt][2], af[mt][3], bh[nt][0], bh[nt][1]);
                    mma_s8u8(al[mt][nt], af[mt][0], af[mt][1], af[mt][2], af[mt][3], bl[nt][0], bl[nt][1]);
                }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
    }

#pragma unroll
    for (int mt = 0; mt < 4; ++mt)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const int n = n0 + wn * 16 + nt * 8 + 2 * tq;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int m = m0 + mt * 16 + g + 8 * h;
                if (m >= M) continue;
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    if (n + e >= N) continue;
                    const int64_t v = (int64_t)ah[mt][nt][2 * h + e] * 256 + al[mt][nt][2 * h + e];
                    int64_t* p = C + (size_t)m * N + n + e;
                    if (gridDim.z > 1) atomicAdd((unsigned long long*)p, (unsigned long long)v);
                    else *p = v;
                }
            }
        }
}

// Exact-mode epilogues on the limb GEMM's int64 accumulators (16-bit
// weights, channel scale m_c / 2^30): y = rshr(acc * (m_t * m_c), k_t + 30 -
// F_out), the product formed exactly in 128 bits, then the int8 path's
// consumers: q/k/v saturation, saturating residual add, SwiGLU of an
// interleaved (gate, up) pair, or int32 logits with per-16-column argmax
// partials (lowest column on ties). One thread per output (per gate/up pair,
// per 16 logits).
__device__ __forceinline__ i64 w16_requant(const int64_t* C, const Epi& ep, int N, int m, int n) {
    const u64 M = (u64)((i64)ep.mt[m] * (i64)ep.mc[n]);
    return rshr_mul128((i64)C[(size_t)m * N + n], M, ep.kt[m] + 30 - ep.fout);
}

// grid: (column blocks of 256, M rows); columns are outputs, gate/up pairs
// or 16-column logit groups
__global__ void __launch_bounds__(256) k_epi_w16(const int64_t* __restrict__ C, int N, int mode, Epi ep) {
    const int m = blockIdx.y;
    const int j = blockIdx.x * 256 + threadIdx.x;
    if (mode == EPI_SWIGLU) {
        if (j >= (N >> 1)) return;                 // channel j: rows 2j (gate), 2j + 1 (up)
        i64 yg = w16_requant(C, ep, N, m, 2 * j), yu = w16_requant(C, ep, N, m, 2 * j + 1);
        if (yg > (1 << 24) || yg < -(1 << 24) || yu > (1 << 24) || yu < -(1 << 24)) ep.status[ST_SAT_GU] = 1;
        ep.out[(size_t)m * ep.ldo + j] = swiglu_dev((int)sat_b(yg, 1 << 24), (int)sat_b(yu, 1 << 24));
        return;
    }
    if (mode == EPI_LOGITS) {
        if (j >= ((N + 15) >> 4)) return;          // logit group j: columns 16j .. 16j + 15
        int bv = -2147483647 - 1, bi = 2147483647;
        for (int n = j * 16; n < min(N, j * 16 + 16); ++n) {
            const i64 y = w16_requant(C, ep, N, m, n);
            if (y > 2147483647LL || y < -2147483647LL) ep.status[ST_SAT_LOGIT] = 1;
            const int v = sat32(y);
            ep.out[(size_t)m * ep.ldo + n] = v;
            if (v > bv) { bv = v; bi = n; }
        }
        ep.pval[(size_t)m * ep.npart + j] = bv;
        ep.pidx[(size_t)m * ep.npart + j] = bi;
        return;
    }
    if (j >= N) return;
    const i64 y = w16_requant(C, ep, N, m, j);
    if (mode == EPI_QKV) {
        if (y > 2147483647LL || y < -2147483647LL) ep.status[ST_SAT_QKV] = 1;
        ep.out[(size_t)m * ep.ldo + j] = sat32(y);
    } else {
        int32_t* hp = ep.out + (size_t)m * ep.ldo + j;
        const i64 s2 = (i64)*hp + (i64)sat32(y);
        if (s2 > 2147483647LL || s2 < -2147483647LL) ep.status[ST_SAT_RES] = 1;
        *hp = sat32(s2);
    }
}

}  // namespace detint
