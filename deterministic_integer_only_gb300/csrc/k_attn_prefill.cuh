// Prefill attention on the int8 tensor pipe.
//
// The integer attention of one query row needs the row maximum of its
// logits before any probability exists (E_j = exp2q(u_j - max u), 15 bits),
// and the normalisation is one deferred division by the row sum (DetLLM
// blog, "DetLLM": 15-bit probabilities, P·V exactly as two int8 products).
// An online rescaling would round differently, so every CTA sweeps its keys
// twice:
//   sweep 1: S = Q K^T (mma.sync s8), running row maxima of the valid S;
//   sweep 2: S again, E from the fixed maxima, E split into its high and low
//            bytes, num += E_hi V (s8 x s8) and E_lo V (u8 x s8), sum E.
// Both limbs stay exact in int32 (|E_hi V| sums < 2^30, |E_lo V| < 2^31 for
// contexts up to 2^16 keys); the epilogue applies the same rounding chain as
// the per-token attention: t = rshr(num RS, bl + 7), o = rshr(t MV, KV + 4).
//
// CTA: 64 query rows (64 / G consecutive tokens of one sequence times the G
// q heads of one kv head), 8 consumer warps and one TMA producer warp. Warp
// (rg, hf) owns rows 16 rg .. 16 rg + 15; it computes S for key half hf of
// each 64-key tile and the P·V output for channel half hf, so the two warps
// of a row group exchange their E bytes through shared memory. K tiles
// ([64 keys][d] bytes) and V^T tiles ([d][64 keys] bytes) arrive by 2D TMA
// from the paged cache with the 128-byte (d = 128) or 64-byte swizzle, which
// makes every ldmatrix conflict-free; a 4-stage ring of mbarriers carries
// sweep 1 (K only) and then sweep 2 (K and V).
#pragma once
#include <cuda.h>
#include "kernels.h"
#include "ptx.cuh"
#include "int_device.cuh"

namespace detint {

constexpr int PF_THREADS = 288;
constexpr int PF_STAGES = 4;
constexpr int PF_LG_STAGES = 2;
constexpr int PF_EP = 80;     // row pitch of the E byte planes: 64 keys + 16 bytes of padding

template <int D>
struct PfCfg {
    static constexpr int KT = 64 * D;                       // K tile bytes
    static constexpr int STAGE = 2 * 64 * D;                // K tile + V^T tile
    static constexpr int QP = D + 16;                       // Q row pitch
    static constexpr int O_ES = PF_STAGES * STAGE;          // 2 buffers x (hi, lo) planes
    static constexpr int ES_BUF = 2 * PF_ROWS * PF_EP;
    static constexpr int O_Q = O_ES + 2 * ES_BUF;
    static constexpr int SMEM = O_Q + PF_ROWS * QP + 1024;  // + alignment slack
};

// byte offset of 16-byte chunk c of key row r in a K tile (TMA swizzle:
// bits 4..6 ^= bits 7..9 for 128-byte rows, bits 4..5 ^= bits 7..8 for 64)
template <int D>
__device__ __forceinline__ uint32_t pf_koff(int r, int c) {
    if (D == 128) return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
    return (uint32_t)(r * 64 + ((c ^ ((r >> 1) & 3)) << 4));
}
// same for channel row r of a V^T tile (64-byte rows)
__device__ __forceinline__ uint32_t pf_voff(int r, int c) {
    return (uint32_t)(r * 64 + ((c ^ ((r >> 1) & 3)) << 4));
}

__device__ __forceinline__ void mma_u8s8(int (&c)[4], int a0, int a1, int a2, int a3, int b0, int b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.s32.u8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+r"(c[0]), "+r"(c[1]), "+r"(c[2]), "+r"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 15-bit unnormalised probability of one logit (zero for a masked key)
__device__ __forceinline__ int pf_e(bool valid, int S, i64 M, int sh, i64 umax) {
    if (!valid) return 0;
    return min(32767, exp2q_dev(rshr((i64)S * M, sh) - umax));
}

template <int D>
__global__ void __launch_bounds__(PF_THREADS, 1)
    k_attn_prefill(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                   PfArgs a) {
    using C = PfCfg<D>;
    constexpr int KS = D >> 5;        // k-steps of 32 channels in Q K^T
    constexpr int NT2 = D >> 4;       // 8-channel n-tiles in a warp's half of P V
    constexpr int LG_CPR = D == 128 ? 3 : 2;   // log2 of 16-byte chunks per Q row
    extern __shared__ unsigned char pf_raw[];
    unsigned char* sm = (unsigned char*)(((uintptr_t)pf_raw + 1023) & ~(uintptr_t)1023);
    __shared__ unsigned long long full[PF_STAGES], empty[PF_STAGES];
    __shared__ int r_pos[PF_ROWS], r_sh[PF_ROWS], r_max2[2][PF_ROWS], r_sum2[2][PF_ROWS];
    __shared__ i64 r_m[PF_ROWS];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = blockIdx.x, qb = blockIdx.y;
    const int lgBQ = 6 - a.lg_grp;                     // tokens per block = 64 / G
    const int t0 = a.qblk[4 * qb], ntok = a.qblk[4 * qb + 1];
    const int seq = a.qblk[4 * qb + 2], pos0 = a.qblk[4 * qb + 3];
    const int nt = ((pos0 + ntok - 1) >> 6) + 1;       // key tiles up to the last position
    const int32_t* kvp = a.kvp + (size_t)g * (8 + (D >> 1));

    if (tid == 0) {
        for (int s = 0; s < PF_STAGES; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 8);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // row r = hh * (64 / G) + i: token t0 + i, q head (g << lg_grp) + hh
    if (tid < PF_ROWS) {
        const int hh = tid >> lgBQ, i = tid & ((1 << lgBQ) - 1);
        if (i < ntok) {
            const size_t th = (size_t)(t0 + i) * a.nq + (g << a.lg_grp) + hh;
            r_pos[tid] = pos0 + i;
            r_m[tid] = (i64)a.mq[th] * (i64)kvp[6];
            r_sh[tid] = a.kq[th] + kvp[7] - 10;
        } else {
            r_pos[tid] = -1;
            r_m[tid] = 0;
            r_sh[tid] = 0;
        }
    }
    {
        unsigned char* qs = sm + C::O_Q;
        for (int idx = tid; idx < (PF_ROWS << LG_CPR); idx += PF_THREADS) {
            const int r = idx >> LG_CPR, ch = idx & ((1 << LG_CPR) - 1);
            const int hh = r >> lgBQ, i = r & ((1 << lgBQ) - 1);
            int4 v = make_int4(0, 0, 0, 0);
            if (i < ntok)
                v = *(const int4*)(a.q8 + ((size_t)(t0 + i) * a.nq + (g << a.lg_grp) + hh) * D + ch * 16);
            *(int4*)(qs + r * C::QP + ch * 16) = v;
        }
    }
    __syncthreads();

    if (warp == 8) {
        // producer: sweep 1 streams K tiles, sweep 2 K and V^T tiles
        if (lane == 0) {
            const int* bt = a.block_table + (size_t)seq * a.mbs;
            int it = 0;
            for (int sw = 0; sw < 2; ++sw) {
                for (int kt = 0; kt < nt; ++kt, ++it) {
                    const int s = it & (PF_STAGES - 1);
                    if (it >= PF_STAGES &&
                        !mbar_wait(smem_u32(&empty[s]), ((it >> PF_LG_STAGES) - 1) & 1))
                        a.status[ST_TIMEOUT] = 1;
                    const uint32_t fb = smem_u32(&full[s]);
                    const int unit = bt[kt] * a.nkv + g;
                    const uint32_t dst = smem_u32(sm + (size_t)s * C::STAGE);
                    mbar_arrive_expect_tx(fb, sw ? C::STAGE : C::KT);
                    tma_load_2d(dst, &kmap, 0, a.krow0 + unit * 64, fb);
                    if (sw) tma_load_2d(dst + C::KT, &vmap, 0, a.vrow0 + unit * D, fb);
                }
            }
        }
        return;
    }

    const int rg = warp >> 1, hf = warp & 1;
    const int gid = lane >> 2, tig = lane & 3;
    const int mi = lane >> 3, ri = lane & 7;
    const int rA = rg * 16 + gid, rB = rA + 8;
    const int posA = r_pos[rA], posB = r_pos[rB];
    const i64 MA = r_m[rA], MB = r_m[rB];
    const int shA = r_sh[rA], shB = r_sh[rB];

    int qf[KS][4];
    {
        const uint32_t qb0 = smem_u32(sm + C::O_Q);
#pragma unroll
        for (int kk = 0; kk < KS; ++kk)
            ldsm_x4(qb0 + (rg * 16 + ri + 8 * (mi & 1)) * C::QP + ((2 * kk + (mi >> 1)) << 4),
                    qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3]);
    }
    // S for this warp's 16 rows and 32 keys of the tile at tK
    auto qk = [&](uint32_t tK, int (&S)[4][4]) {
#pragma unroll
        for (int n = 0; n < 4; ++n) S[n][0] = S[n][1] = S[n][2] = S[n][3] = 0;
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
#pragma unroll
            for (int np = 0; np < 2; ++np) {
                const int key = hf * 32 + np * 16 + ri + 8 * (mi >> 1);
                int b0, b1, b2, b3;
                ldsm_x4(tK + pf_koff<D>(key, 2 * kk + (mi & 1)), b0, b1, b2, b3);
                mma_s8(S[2 * np], qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3], b0, b1);
                mma_s8(S[2 * np + 1], qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3], b2, b3);
            }
        }
    };

    // ---- sweep 1: row maxima of S over the valid keys
    int mxA = -2147483647 - 1, mxB = -2147483647 - 1;
    int it = 0;
    for (int kt = 0; kt < nt; ++kt, ++it) {
        const int s = it & (PF_STAGES - 1);
        if (!mbar_wait(smem_u32(&full[s]), (it >> PF_LG_STAGES) & 1)) a.status[ST_TIMEOUT] = 1;
        int S[4][4];
        qk(smem_u32(sm + (size_t)s * C::STAGE), S);
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
        const int kb = kt * 64 + hf * 32 + 2 * tig;
#pragma unroll
        for (int n = 0; n < 4; ++n) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int key = kb + n * 8 + e;
                if (key <= posA) mxA = max(mxA, S[n][e]);
                if (key <= posB) mxB = max(mxB, S[n][2 + e]);
            }
        }
    }
    mxA = max(mxA, __shfl_xor_sync(0xffffffffu, mxA, 1));
    mxA = max(mxA, __shfl_xor_sync(0xffffffffu, mxA, 2));
    mxB = max(mxB, __shfl_xor_sync(0xffffffffu, mxB, 1));
    mxB = max(mxB, __shfl_xor_sync(0xffffffffu, mxB, 2));
    if (tig == 0) {
        r_max2[hf][rA] = mxA;
        r_max2[hf][rB] = mxB;
    }
    bar_named(1 + rg, 64);
    // u is non-decreasing in S, so max u = u(max S)
    const i64 umA = rshr((i64)max(r_max2[0][rA], r_max2[1][rA]) * MA, shA);
    const i64 umB = rshr((i64)max(r_max2[0][rB], r_max2[1][rB]) * MB, shB);

    // ---- sweep 2: probabilities, their sums and the two P·V limbs
    int accH[NT2][4], accL[NT2][4];
#pragma unroll
    for (int n = 0; n < NT2; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) accH[n][e] = accL[n][e] = 0;
    int sumA = 0, sumB = 0;
    for (int kt = 0; kt < nt; ++kt, ++it) {
        const int s = it & (PF_STAGES - 1);
        if (!mbar_wait(smem_u32(&full[s]), (it >> PF_LG_STAGES) & 1)) a.status[ST_TIMEOUT] = 1;
        const uint32_t tK = smem_u32(sm + (size_t)s * C::STAGE);
        int S[4][4];
        qk(tK, S);
        unsigned char* eh = sm + C::O_ES + (kt & 1) * C::ES_BUF;
        unsigned char* el = eh + PF_ROWS * PF_EP;
        const int kb = kt * 64 + hf * 32 + 2 * tig;
#pragma unroll
        for (int n = 0; n < 4; ++n) {
            const int key = kb + n * 8;
            const int a0 = pf_e(key <= posA, S[n][0], MA, shA, umA);
            const int a1 = pf_e(key + 1 <= posA, S[n][1], MA, shA, umA);
            const int b0 = pf_e(key <= posB, S[n][2], MB, shB, umB);
            const int b1 = pf_e(key + 1 <= posB, S[n][3], MB, shB, umB);
            sumA += a0 + a1;
            sumB += b0 + b1;
            const int col = hf * 32 + n * 8 + 2 * tig;
            *(uint16_t*)(eh + rA * PF_EP + col) = (uint16_t)((a0 >> 8) | ((a1 >> 8) << 8));
            *(uint16_t*)(el + rA * PF_EP + col) = (uint16_t)((a0 & 255) | ((a1 & 255) << 8));
            *(uint16_t*)(eh + rB * PF_EP + col) = (uint16_t)((b0 >> 8) | ((b1 >> 8) << 8));
            *(uint16_t*)(el + rB * PF_EP + col) = (uint16_t)((b0 & 255) | ((b1 & 255) << 8));
        }
        bar_named(1 + rg, 64);   // both key halves of the row group's E are in place
        int ah[2][4], al[2][4];
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
            const uint32_t off = (rg * 16 + ri + 8 * (mi & 1)) * PF_EP + ((2 * kk + (mi >> 1)) << 4);
            ldsm_x4(smem_u32(eh) + off, ah[kk][0], ah[kk][1], ah[kk][2], ah[kk][3]);
            ldsm_x4(smem_u32(el) + off, al[kk][0], al[kk][1], al[kk][2], al[kk][3]);
        }
        const uint32_t tV = tK + C::KT;
#pragma unroll
        for (int n = 0; n < NT2; n += 2) {
            // matrices: 16-key chunks 0..3 of channels c .. c + 7; two n-tiles
            // at a time so that dependent MMAs are four issues apart
            int v[2][4];
#pragma unroll
            for (int j = 0; j < 2; ++j)
                ldsm_x4(tV + pf_voff(hf * (D >> 1) + (n + j) * 8 + ri, mi), v[j][0], v[j][1], v[j][2],
                        v[j][3]);
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    mma_s8(accH[n + j], ah[kk][0], ah[kk][1], ah[kk][2], ah[kk][3], v[j][2 * kk],
                           v[j][2 * kk + 1]);
                    mma_u8s8(accL[n + j], al[kk][0], al[kk][1], al[kk][2], al[kk][3], v[j][2 * kk],
                             v[j][2 * kk + 1]);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
    }
    sumA += __shfl_xor_sync(0xffffffffu, sumA, 1);
    sumA += __shfl_xor_sync(0xffffffffu, sumA, 2);
    sumB += __shfl_xor_sync(0xffffffffu, sumB, 1);
    sumB += __shfl_xor_sync(0xffffffffu, sumB, 2);
    if (tig == 0) {
        r_sum2[hf][rA] = sumA;
        r_sum2[hf][rB] = sumB;
    }
    bar_named(1 + rg, 64);

    // ---- epilogue: one deferred division per row, then the output rounding
    const i64 MV = kvp[4];
    const int KVS = kvp[5];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int r = h ? rB : rA;
        const i64 sg = (i64)r_sum2[0][r] + (i64)r_sum2[1][r];   // >= 32767 for a valid row
        const int bl = bitlen_u64((u64)sg);
        i64 rs = 0;
        if (tig == 0 && sg > 0) rs = (i64)pow2_recip((u64)sg, bl, 1, 23);
        rs = __shfl_sync(0xffffffffu, rs, lane & ~3, 32);
        if (r_pos[r] < 0) continue;
        const int i = r & ((1 << lgBQ) - 1), hh = r >> lgBQ;
        int32_t* orow = a.o + ((size_t)(t0 + i) * a.nq + (g << a.lg_grp) + hh) * D;
#pragma unroll
        for (int n = 0; n < NT2; ++n) {
            const int c = hf * (D >> 1) + n * 8 + 2 * tig;
            int2 out;
            const i64 num0 = (i64)accH[n][2 * h] * 256 + accL[n][2 * h];
            const i64 num1 = (i64)accH[n][2 * h + 1] * 256 + accL[n][2 * h + 1];
            out.x = (int32_t)rshr(rshr(num0 * rs, bl + 7) * MV, KVS + 16 - 12);
            out.y = (int32_t)rshr(rshr(num1 * rs, bl + 7) * MV, KVS + 16 - 12);
            *(int2*)(orow + c) = out;
        }
    }
    // every stage the producer filled was waited for above, so no copy is
    // in flight when the CTA exits
}

}  // namespace detint
