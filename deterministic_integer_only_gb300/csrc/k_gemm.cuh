// Tiled int8 x int8 -> int32 GEMM for many tokens (prefill, and the exact
// GEMM entry point): C[m][n] = sum_k A[m][k] W[n][k], with the same
// requantisation epilogues as the decode GEMV.
//
// sm_103a has no integer tcgen05 kind, so the integer tensor instruction is
// the warp-level mma.sync m16n8k32 (s8 x s8 -> s32). Operand tiles move by
// TMA (cp.async.bulk.tensor.2d, 128-byte swizzle, zero fill past the matrix
// edges, which leaves exact integer sums unchanged) into a 3-stage
// shared-memory ring guarded by mbarriers; a producer warp issues the copies
// and 8 consumer warps read fragments with conflict-free ldmatrix.
// CTA tile 128 x 128 x 128 bytes; warp tile 64 (M) x 32 (N).
#pragma once
#include <cuda.h>
#include "kernels.h"
#include "ptx.cuh"

namespace detint {

constexpr int GM_BM = 128, GM_BN = 128, GM_BK = 128;
constexpr int GM_STAGES = 3;
constexpr int GM_THREADS = 288;
constexpr int GM_STAGE_BYTES = (GM_BM + GM_BN) * GM_BK;   // 32 KB
constexpr size_t GM_SMEM = (size_t)GM_STAGES * GM_STAGE_BYTES + 1024;

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            dst),
        "l"(map), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, int& r0, int& r1, int& r2, int& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// byte offset of 16-byte chunk c of tile row r under the 128-byte swizzle
__device__ __forceinline__ uint32_t swz(int r, int c) { return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4)); }

// BM: rows of the CTA tile (128; 64 or 32 for short M, so that few MMAs work
// on zero rows); the 8 consumer warps tile it as WM x WN, each warp
// MT m16 tiles by NTW n8 tiles
template <int MODE, int BM>
__global__ void __launch_bounds__(GM_THREADS, 1) k_gemm_tma(const __grid_constant__ CUtensorMap mapA,
                                                            const __grid_constant__ CUtensorMap mapW,
                                                            int M, int N, int K, Epi ep, int ksl,
                                                            int32_t* wsp, int* tcnt) {
    extern __shared__ unsigned char gsm_raw[];
    __shared__ unsigned long long full[GM_STAGES], empty[GM_STAGES];
    unsigned char* gsm = (unsigned char*)(((uintptr_t)gsm_raw + 1023) & ~(uintptr_t)1023);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    constexpr int WN = BM == 128 ? 4 : 8;            // warps along N
    constexpr int NTW = GM_BN / WN / 8;              // 8-column n-tiles per warp
    constexpr int MT = BM == 32 ? 2 : 4;             // 16-row m-tiles per warp
    constexpr int STAGE = (BM + GM_BN) * GM_BK;
    const int m0 = blockIdx.y * BM, n0 = blockIdx.x * GM_BN;
    // split K (raw int32 output only): this CTA takes k-tiles [kt0, kt0 + nk)
    // and adds its partial sums into the zeroed output; integer addition is
    // exact, so the result does not depend on the order of the adds
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
                if (kt >= GM_STAGES &&
                    !mbar_wait(smem_u32(&empty[s]), ((kt / GM_STAGES) - 1) & 1))
                    ep.status[ST_TIMEOUT] = 1;
                const uint32_t fb = smem_u32(&full[s]);
                mbar_arrive_expect_tx(fb, STAGE);
                const uint32_t base = smem_u32(gsm + (size_t)s * STAGE);
                tma_load_2d(base, &mapA, (kt0 + kt) * GM_BK, m0, fb);
                tma_load_2d(base + BM * GM_BK, &mapW, (kt0 + kt) * GM_BK, n0, fb);
            }
        }
        return;
    }

    const int wm = warp / WN, wn = warp % WN;
    const int g = lane >> 2, tq = lane & 3;
    const int mi = lane >> 3, ri = lane & 7;     // ldmatrix matrix / row within it
    int acc[MT][NTW][4];
#pragma unroll
    for (int a = 0; a < MT; ++a)
#pragma unroll
        for (int b = 0; b < NTW; ++b) acc[a][b][0] = acc[a][b][1] = acc[a][b][2] = acc[a][b][3] = 0;

    for (int kt = 0; kt < nk; ++kt) {
        const int s = kt % GM_STAGES;
        if (!mbar_wait(smem_u32(&full[s]), (kt / GM_STAGES) & 1)) ep.status[ST_TIMEOUT] = 1;
        const uint32_t tA = smem_u32(gsm + (size_t)s * STAGE);
        const uint32_t tW = tA + BM * GM_BK;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            int af[MT][4], bf[NTW][2];
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                const int r = wm * 64 + mt * 16 + ri + 8 * (mi & 1);
                ldsm_x4(tA + swz(r, 2 * kk + (mi >> 1)), af[mt][0], af[mt][1], af[mt][2], af[mt][3]);
            }
#pragma unroll
            for (int np = 0; np < NTW / 2; ++np) {
                const int r = wn * (NTW * 8) + np * 16 + ri + 8 * (mi >> 1);
                ldsm_x4(tW + swz(r, 2 * kk + (mi & 1)), bf[2 * np][0], bf[2 * np][1],
                        bf[2 * np + 1][0], bf[2 * np + 1][1]);
            }
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int nt = 0; nt < NTW; ++nt)
                    mma_s8(acc[mt][nt], af[mt][0], af[mt][1], af[mt][2], af[mt][3], bf[nt][0], bf[nt][1]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
    }

    if (MODE != EPI_RAW && gridDim.z > 1) {
        // split K under an epilogue: every split stores its partial tile in
        // the workspace [split][rows][N]; the tile's last split (counted on
        // the tile's counter, which it resets) adds the partials in split
        // order and applies the epilogue
        const size_t TM = (size_t)gridDim.y * BM;
        __shared__ int last_split;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int nt = 0; nt < NTW; ++nt) {
                const int n = n0 + wn * (NTW * 8) + nt * 8 + 2 * tq;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int m = m0 + wm * 64 + mt * 16 + g + 8 * h;
                    if (m >= M) continue;
                    int32_t* w = wsp + ((size_t)blockIdx.z * TM + m) * N + n;
                    if (n < N) w[0] = acc[mt][nt][2 * h];
                    if (n + 1 < N) w[1] = acc[mt][nt][2 * h + 1];
                }
            }
        __threadfence();
        bar_named(1, 256);
        if (tid == 0) {
            int* c = tcnt + blockIdx.y * gridDim.x + blockIdx.x;
            const int old = atomicAdd(c, 1);
            last_split = old == (int)gridDim.z - 1;
            if (last_split) *c = 0;
        }
        bar_named(1, 256);
        if (!last_split) return;
        __threadfence();
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int nt = 0; nt < NTW; ++nt) {
                const int n = n0 + wn * (NTW * 8) + nt * 8 + 2 * tq;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int m = m0 + wm * 64 + mt * 16 + g + 8 * h;
                    if (m >= M) continue;
                    int c0 = 0, c1 = 0;
                    for (int z = 0; z < (int)gridDim.z; ++z) {
                        const int32_t* w = wsp + ((size_t)z * TM + m) * N + n;
                        if (n < N) c0 += __ldcg(w);
                        if (n + 1 < N) c1 += __ldcg(w + 1);
                    }
                    acc[mt][nt][2 * h] = c0;
                    acc[mt][nt][2 * h + 1] = c1;
                }
            }
    }

    if (MODE == EPI_LOGITS) {
        // int32 logits, and per 16-column group the largest (lowest column on
        // ties) as the argmax partial of that group: a group is two n-tiles
        // of one warp, spread over the 4 lanes of a quad
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int m = m0 + wm * 64 + mt * 16 + g + 8 * h;
#pragma unroll
                for (int j = 0; j < NTW / 2; ++j) {
                    int bv = -2147483647 - 1, bi = 2147483647;
#pragma unroll
                    for (int q = 0; q < 2; ++q)
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int n = n0 + wn * (NTW * 8) + (2 * j + q) * 8 + 2 * tq + e;
                            if (m < M && n < N) {
                                const i64 y = requant_dev(acc[mt][2 * j + q][2 * h + e], ep, m, n);
                                if (y > 2147483647LL || y < -2147483647LL) ep.status[ST_SAT_LOGIT] = 1;
                                const int v = sat32(y);
                                ep.out[(size_t)m * ep.ldo + n] = v;
                                if (v > bv || (v == bv && n < bi)) { bv = v; bi = n; }
                            }
                        }
#pragma unroll
                    for (int o = 1; o <= 2; o <<= 1) {
                        const int v = __shfl_xor_sync(0xffffffffu, bv, o);
                        const int i = __shfl_xor_sync(0xffffffffu, bi, o);
                        if (v > bv || (v == bv && i < bi)) { bv = v; bi = i; }
                    }
                    const int grp = (n0 + wn * (NTW * 8) + j * 16) >> 4;
                    if (tq == 0 && m < M && grp * 16 < N) {
                        ep.pval[(size_t)m * ep.npart + grp] = bv;
                        ep.pidx[(size_t)m * ep.npart + grp] = bi;
                    }
                }
            }
        return;
    }

    // epilogue straight from the accumulator fragments
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
        for (int nt = 0; nt < NTW; ++nt) {
            const int n = n0 + wn * (NTW * 8) + nt * 8 + 2 * tq;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int m = m0 + wm * 64 + mt * 16 + g + 8 * h;
                if (m >= M) continue;
                const int c0 = acc[mt][nt][2 * h], c1 = acc[mt][nt][2 * h + 1];
                if (MODE == EPI_SWIGLU) {
                    if (n < N) {
                        i64 yg = requant_dev(c0, ep, m, n), yu = requant_dev(c1, ep, m, n + 1);
                        if (yg > (1 << 24) || yg < -(1 << 24) || yu > (1 << 24) || yu < -(1 << 24))
                            ep.status[ST_SAT_GU] = 1;
                        yg = sat_b(yg, 1 << 24);
                        yu = sat_b(yu, 1 << 24);
                        ep.out[(size_t)m * ep.ldo + (n >> 1)] = swiglu_tab((int)yg, (int)yu);
                    }
                } else if (MODE == EPI_RAW && gridDim.z > 1) {
                    if (n < N) atomicAdd(ep.out + (size_t)m * ep.ldo + n, c0);
                    if (n + 1 < N) atomicAdd(ep.out + (size_t)m * ep.ldo + n + 1, c1);
                } else {
                    if (n < N) epi_store<MODE>(ep, m, n, c0);
                    if (n + 1 < N) epi_store<MODE>(ep, m, n + 1, c1);
                }
            }
        }
    }
    // the consumers waited for every stage the producer filled, so no copy
    // is in flight when the CTA exits
}

}  // namespace detint
