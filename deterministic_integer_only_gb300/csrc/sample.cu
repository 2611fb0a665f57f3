// Integer sampling of logits rows (detint_sample): temperature, top-k,
// top-p and one SplitMix64 draw by cumulative integer weights, with the
// arithmetic of the specification's "Integer sampling" section (the pages
// ask for integer sampling rules and deterministic sampling: BitExact LLM
// post, "Fix the arithmetic, not just the random seed" and "Reproducibility
// has a cost"; they give no algorithm).
//
// Rows of 16384 or more logits run on a thread-block cluster of 8 CTAs of
// 1024 threads (one slice each, every count combined through distributed
// shared memory) while all rows' clusters fit the SMs at once; otherwise a
// row runs on one CTA. Nothing is allocated. Where the definition
// sorts the row by logit, the kernel uses order statistics instead:
//  * the top-k boundary logit by a 3-pass radix select (11 + 11 + 10 bits of
//    the order-preserving key), with the lowest-index ties taken first;
//  * the top-p boundary from a histogram of delta = u - max u over the top-k
//    set (24577 bins: every delta <= -24576 has weight 0 and shares bin 0),
//    since the weight E depends on delta alone and delta is non-increasing
//    along the logit order;
//  * the draw as one scan in index order (per-warp chunk sums, a block scan,
//    then one warp walks the chunk that holds the target).
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "../../include/detint.h"
#include "int_device.cuh"

#include <cooperative_groups.h>
namespace cg = cooperative_groups;

namespace detint {

constexpr int SP_THREADS = 1024;
constexpr int SP_BINS = 24577;
constexpr int SP_OFF = 24576;          // bin of delta = delta + SP_OFF, floored at 0
constexpr int SP_ROWS = 32;            // rows per launch (parameters travel in the argument)
constexpr int SP_CL = 8;               // CTAs per row for long rows (a thread-block cluster)

struct SpBatch {
    detint_sampling_t p[SP_ROWS];
};

__device__ __forceinline__ i64 sp_u(int32_t l, int32_t inv_temp) {
    const i64 a = rshr((i64)l * 47274, 21);
    return rshr(a * (i64)inv_temp, 16);
}
__device__ __forceinline__ uint32_t sp_key(int32_t l) { return (uint32_t)l ^ 0x80000000u; }
__device__ __forceinline__ int sp_bin(i64 delta) { return delta <= -SP_OFF ? 0 : (int)(delta + SP_OFF); }
__device__ __forceinline__ i64 sp_binE(int b) { return b == 0 ? 0 : (i64)exp2q_dev((i64)(b - SP_OFF)); }

__device__ __forceinline__ uint64_t sp_splitmix64(uint64_t seed, uint64_t counter) {
    uint64_t z = seed + (counter + 1) * 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

// block-wide reductions and scans over the 32 warps (every thread calls)
__device__ int sp_max_i32(int v, int* red) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
    __syncthreads();
    if (lane == 0) red[w] = v;
    __syncthreads();
    v = red[lane];
#pragma unroll
    for (int o = 16; o; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
// exclusive prefix of one i64 per warp (warp order); returns it to every
// lane of the warp, and the block total in *tot
__device__ i64 sp_warp_excl(i64 v, i64* red, i64* tot) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    __syncthreads();
    if (lane == 0) red[w] = v;
    __syncthreads();
    i64 x = red[lane], inc = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const i64 y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
    }
    *tot = __shfl_sync(0xffffffffu, inc, 31);
    return __shfl_sync(0xffffffffu, inc - x, w);
}
__device__ __forceinline__ i64 sp_warp_sum(i64 v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
// inclusive prefix over the lanes of a warp
__device__ __forceinline__ i64 sp_lane_incl(i64 v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const i64 y = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += y;
    }
    return v;
}

// CL: CTAs per row. CL = 1 is one CTA per row; CL > 1 runs the row on a
// thread-block cluster, each CTA on a contiguous slice, with every count
// combined through distributed shared memory (every CTA then takes the same
// decisions from the same cluster-wide counts)
template <int CL>
__global__ void __launch_bounds__(SP_THREADS) k_sample(const int32_t* __restrict__ logits, int n,
                                                      SpBatch batch, int32_t* out) {
    extern __shared__ int sp_sm[];
    int* hloc = sp_sm;                                   // this CTA's counts
    int* hsum = CL > 1 ? sp_sm + SP_BINS : sp_sm;        // the row's counts, later per-bin weights
    __shared__ int red_i[32];
    __shared__ i64 red_l[32];
    __shared__ int s_sel[4];
    __shared__ i64 s_sel64[2];
    __shared__ int c_max, c_ties;                        // read by the other CTAs of the cluster
    __shared__ i64 c_kept;
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    cg::cluster_group cl = cg::this_cluster();
    const int rank = CL > 1 ? (int)cl.block_rank() : 0;
    const int row = CL > 1 ? (int)(blockIdx.x / CL) : (int)blockIdx.x;
    const detint_sampling_t prm = batch.p[row];
    const int32_t* x = logits + (size_t)row * n;
    const int32_t invT = prm.inv_temp;
    // this CTA's slice [s0, s1) of the row, 32-aligned
    constexpr int SLICE_Q = CL * 32;                     // slice granule
    const int per = CL > 1 ? ((n + SLICE_Q - 1) / SLICE_Q) * 32 : n;
    const int s0 = min(n, rank * per), s1 = min(n, s0 + per);
    auto csync = [&]() {
        if (CL > 1) cl.sync();
        else __syncthreads();
    };

    // ---- 1-2: the maximum logit gives max u (u is non-decreasing in l)
    int lmax = -2147483647 - 1;
#pragma unroll 8
    for (int i = s0 + tid; i < s1; i += SP_THREADS) lmax = max(lmax, __ldg(x + i));
    lmax = sp_max_i32(lmax, red_i);
    if (CL > 1) {
        if (tid == 0) c_max = lmax;
        cl.sync();
#pragma unroll
        for (int r = 0; r < CL; ++r) lmax = max(lmax, *cl.map_shared_rank(&c_max, r));
    }
    const i64 M = sp_u(lmax, invT);

    // ---- 4: top-k boundary: the k-th largest logit lk and how many of its
    // ties (lowest indices first) belong to the set
    const bool topk = prm.top_k > 0 && prm.top_k < n;
    uint32_t kstar = 0;            // key of lk (0: no boundary, every element is in)
    int quota = 0;                 // ties of lk inside the set
    if (topk) {
        uint32_t prefix = 0, pmask = 0;
        int krem = prm.top_k;      // rank still to find among elements matching the prefix
        const int shifts[3] = {21, 10, 0};
        const int widths[3] = {11, 11, 10};
        for (int ps = 0; ps < 3; ++ps) {
            const int sh = shifts[ps], nb = 1 << widths[ps];
            for (int b = tid; b < nb; b += SP_THREADS) hloc[b] = 0;
            __syncthreads();
#pragma unroll 4
            for (int i = s0 + tid; i < s1; i += SP_THREADS) {
                const uint32_t k = sp_key(__ldg(x + i));
                if ((k & pmask) == prefix) atomicAdd(&hloc[(k >> sh) & (nb - 1)], 1);
            }
            csync();
            if (CL > 1)
                for (int b = tid; b < nb; b += SP_THREADS) {
                    int c = 0;
#pragma unroll
                    for (int r = 0; r < CL; ++r) c += cl.map_shared_rank(hloc, r)[b];
                    hsum[b] = c;
                }
            __syncthreads();
            // digit holding the krem-th largest: scan digits from the top
            if (w == 0) {
                int above = 0, found = -1, rem = krem;
                for (int base = nb - 1; base >= 0 && found < 0; base -= 32) {
                    const int b = base - lane;
                    const int c = b >= 0 ? hsum[b] : 0;
                    // inclusive count from the top within this group of 32 digits
                    int inc = c;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const int y = __shfl_up_sync(0xffffffffu, inc, o);
                        if (lane >= o) inc += y;
                    }
                    const unsigned hit = __ballot_sync(0xffffffffu, above + inc >= rem && b >= 0);
                    if (hit) {
                        const int l0 = __ffs(hit) - 1;
                        const int incl0 = __shfl_sync(0xffffffffu, inc, l0);
                        const int c0 = __shfl_sync(0xffffffffu, c, l0);
                        found = base - l0;
                        rem = rem - (above + incl0 - c0);
                    }
                    above += __shfl_sync(0xffffffffu, inc, 31);
                }
                if (lane == 0) { s_sel[0] = found; s_sel[1] = rem; }
            }
            __syncthreads();
            prefix |= (uint32_t)s_sel[0] << sh;
            pmask |= (uint32_t)(nb - 1) << sh;
            krem = s_sel[1];
            csync();               // every CTA has read the local counts before they are reset
        }
        kstar = prefix;
        quota = krem;              // the krem-th of lk's ties, counted from the lowest index
    }
    const int32_t lk = (int32_t)(kstar ^ 0x80000000u);

    // ---- delta histogram of the top-k set (weights depend on delta alone)
    for (int b = tid; b < SP_BINS; b += SP_THREADS) hloc[b] = 0;
    __syncthreads();
#pragma unroll 4
    for (int base = s0; base < s1; base += SP_THREADS) {   // every thread runs every round
        const int i = base + tid;
        const int32_t l = i < s1 ? __ldg(x + i) : 0;
        const bool in = i < s1 && (!topk || l > lk);
        const int b = in ? sp_bin(sp_u(l, invT) - M) : -1;
        const unsigned act = __ballot_sync(0xffffffffu, in);
        // one add per warp when its lanes share a bin (a flat or hot row),
        // else one per lane (bins of spread logits rarely collide)
        const int b0 = __shfl_sync(0xffffffffu, b, __ffs(act | 1u) - 1);
        const unsigned same = __ballot_sync(0xffffffffu, in && b == b0);
        if (same == act) {
            if (act && lane == __ffs(act) - 1) atomicAdd(&hloc[b0], __popc(act));
        } else if (in) {
            atomicAdd(&hloc[b], 1);
        }
    }
    __syncthreads();
    if (topk && rank == 0 && tid == 0) hloc[sp_bin(sp_u(lk, invT) - M)] += quota;
    csync();
    if (CL > 1) {
        for (int b = tid; b < SP_BINS; b += SP_THREADS) {
            int c = 0;
#pragma unroll
            for (int r = 0; r < CL; ++r) c += cl.map_shared_rank(hloc, r)[b];
            hsum[b] = c;
        }
        __syncthreads();
    }

    // ---- S1, and the top-p boundary bin: bins from the top, thread t owns
    // bins [SP_OFF - 24 t - 23, SP_OFF - 24 t] (thread 1023 also bin 0)
    const int bhi = SP_OFF - 24 * tid, blo = tid == SP_THREADS - 1 ? 0 : bhi - 23;
    i64 ce = 0;
    for (int b = bhi; b >= blo; --b) ce += (i64)hsum[b] * sp_binE(b);
    i64 S1;
    const i64 before = sp_warp_excl(sp_warp_sum(ce), red_l, &S1) + (sp_lane_incl(ce) - ce);
    const bool topp = prm.top_p < 65536;
    // first bin (from the top) where 65536 * cumulative >= top_p * S1
    int bstar = 0;
    i64 S = S1;
    if (topp) {
        const __int128 target = (__int128)prm.top_p * S1;
        const bool mine = (__int128)(before + ce) * 65536 >= target && (__int128)before * 65536 < target;
        if (mine) {
            i64 cum = before;
            for (int b = bhi; b >= blo; --b) {
                cum += (i64)hsum[b] * sp_binE(b);
                if ((__int128)cum * 65536 >= target) { s_sel[2] = b; s_sel64[0] = cum; break; }
            }
        }
        __syncthreads();
        bstar = s_sel[2];
        S = s_sel64[0];
    }
    // the row's histogram is no longer needed: it becomes the kept weight of
    // each bin (0 below the top-p boundary), looked up per element below
    __syncthreads();
    for (int b = tid; b < SP_BINS; b += SP_THREADS) hsum[b] = b >= bstar ? (int)sp_binE(b) : 0;
    __syncthreads();
    // ---- 6-7: the draw
    const uint64_t r = sp_splitmix64(prm.seed, prm.counter);
    const i64 tdraw = (i64)__umul64hi(r, (uint64_t)S);

    // membership in index order: delta bin >= bstar, and in the top-k set
    // (logit above lk, or one of lk's first `quota` ties by index)
    const int C = ((per + 32 * 32 - 1) / (32 * 32)) * 32;   // warp chunk of the slice, a multiple of 32
    const int c0 = min(s1, s0 + w * C), c1 = min(s1, c0 + C);
    // ties of lk before each warp's chunk: earlier CTAs of the cluster, then
    // earlier warps of this CTA
    int tie_before = 0;
    if (topk) {
        int cnt = 0;
#pragma unroll 8
        for (int i = c0 + lane; i < c1; i += 32) cnt += __ldg(x + i) == lk;
        i64 tot;
        tie_before = (int)sp_warp_excl(sp_warp_sum(cnt), red_l, &tot);
        if (CL > 1) {
            if (tid == 0) c_ties = (int)tot;
            cl.sync();
            for (int q = 0; q < rank; ++q) tie_before += *cl.map_shared_rank(&c_ties, q);
        }
    }
    // kept weight of each chunk
    auto kept_E = [&](int i, int rk) -> i64 {
        const int32_t l = __ldg(x + i);
        if (topk && (l < lk || (l == lk && rk >= quota))) return 0;
        return (i64)hsum[sp_bin(sp_u(l, invT) - M)];
    };
    i64 wsum = 0;
    {
        int rk = tie_before;
#pragma unroll 4
        for (int base = c0; base < c1; base += 32) {
            const int i = base + lane;
            const bool tie = topk && i < c1 && __ldg(x + i) == lk;
            const unsigned tb = __ballot_sync(0xffffffffu, tie);
            const int my = rk + __popc(tb & ((1u << lane) - 1));
            if (i < c1) wsum += kept_E(i, my);
            rk += __popc(tb);
        }
    }
    i64 ctot;
    i64 wpre = sp_warp_excl(sp_warp_sum(wsum), red_l, &ctot);
    const i64 wtot = sp_warp_sum(wsum);
    if (CL > 1) {
        // kept weight of the earlier CTAs of the cluster
        if (tid == 0) c_kept = ctot;
        cl.sync();
        for (int q = 0; q < rank; ++q) wpre += *cl.map_shared_rank(&c_kept, q);
    }
    if (wpre <= tdraw && tdraw < wpre + wtot) {
        // this warp's chunk holds the target: walk it in rounds of 32
        int rk = tie_before;
        i64 cum = wpre;
        for (int base = c0; base < c1; base += 32) {
            const int i = base + lane;
            const bool tie = topk && i < c1 && __ldg(x + i) == lk;
            const unsigned tb = __ballot_sync(0xffffffffu, tie);
            const int my = rk + __popc(tb & ((1u << lane) - 1));
            const i64 e = i < c1 ? kept_E(i, my) : 0;
            const i64 inc = sp_lane_incl(e);
            const unsigned hit = __ballot_sync(0xffffffffu, cum + inc > tdraw);
            if (hit) {
                if (lane == __ffs(hit) - 1) out[row] = i;
                break;
            }
            cum += __shfl_sync(0xffffffffu, inc, 31);
            rk += __popc(tb);
        }
    }
    // no CTA leaves while another may still read its shared memory
    if (CL > 1) cl.sync();
}

}  // namespace detint

using namespace detint;

extern "C" int detint_sample(const int32_t* logits, int rows, int n, const detint_sampling_t* params,
                             int32_t* out, detint_stream_t sp) {
    if (!logits || !params || !out || rows < 1 || n < 1) return DETINT_E_ARG;
    for (int r = 0; r < rows; ++r) {
        const detint_sampling_t& p = params[r];
        if (p.inv_temp < 0 || p.inv_temp > (1 << 20) || p.top_k < 0 || p.top_p < 1 || p.top_p > 65536)
            return DETINT_E_ARG;
    }
    int dev = 0, nsm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return DETINT_E_CUDA;
    cudaStream_t s = (cudaStream_t)sp;
    for (int r0 = 0; r0 < rows; r0 += SP_ROWS) {
        SpBatch b{};
        const int nr = std::min(SP_ROWS, rows - r0);
        // long rows run on a cluster of SP_CL CTAs while the clusters of all
        // rows fit the SMs at once; otherwise one CTA per row
        const bool clustered = n >= 16384 && nr * SP_CL <= nsm;
        const size_t smem = (size_t)(clustered ? 2 : 1) * SP_BINS * sizeof(int);
        void (*kern)(const int32_t*, int, SpBatch, int32_t*) = clustered ? k_sample<SP_CL> : k_sample<1>;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
            return DETINT_E_CUDA;
        for (int r = 0; r < nr; ++r) b.p[r] = params[r0 + r];
        const int32_t* lg = logits + (size_t)r0 * n;
        int32_t* o = out + r0;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(nr * (clustered ? SP_CL : 1));
        cfg.blockDim = dim3(SP_THREADS);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = s;
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = clustered ? SP_CL : 1;
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = 1;
        cfg.attrs = at;
        cfg.numAttrs = clustered ? 1 : 0;
        if (cudaLaunchKernelEx(&cfg, kern, lg, n, b, o) != cudaSuccess) return DETINT_E_CUDA;
    }
    return DETINT_OK;
}
