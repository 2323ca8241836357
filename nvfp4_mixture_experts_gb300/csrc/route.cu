// Routing: router logits, softmax top-k, and the local map + grouping ("compact
// pre-pass") that turns top-k ids into padded per-expert row groups.
//
// Solar Open 2 on DGX Spark, "Solar Open 2 개요": top-8 of 320 routed experts plus one
// shared expert.  "b12x에서의 Expert Parallelism 구현 추가": global expert ids are mapped
// to shard-relative ids with local_expert_offset and out-of-shard pairs are dropped.
#include <cuda_bf16.h>

#include "kernels.cuh"

namespace moe {

// ---------------------------------------------------------------- router logits
//
// logits[t][e] = sum_h x[t][h] * Wr[e][h] + bias[e], fp32 accumulation.
// Block: 4 warps, one expert per warp, a chunk of 64 tokens.  The x chunk is staged in
// shared memory 256 columns at a time; each lane accumulates all 64 tokens over its
// 8-column slice, then the partial sums are reduced across the warp.
constexpr int kRtTok = 64;
constexpr int kRtCols = 256;
constexpr int kRtExperts = 4;

__global__ void __launch_bounds__(128) router_logits_kernel(
    const uint16_t* __restrict__ x, const uint16_t* __restrict__ wr,
    const float* __restrict__ bias, int T, int H, int E, float* __restrict__ logits)
{
    __shared__ __align__(16) uint16_t xs[kRtTok][kRtCols];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = blockIdx.x * kRtExperts + warp;
    const int t0 = blockIdx.y * kRtTok;
    const int nt = min(kRtTok, T - t0);
    float acc[kRtTok];
#pragma unroll
    for (int i = 0; i < kRtTok; ++i) acc[i] = 0.0f;

    for (int h0 = 0; h0 < H; h0 += kRtCols) {
        __syncthreads();
        // stage x[t0 .. t0+nt)[h0 .. h0+512) (16-byte vectors)
        for (int v = threadIdx.x; v < kRtTok * (kRtCols / 8); v += blockDim.x) {
            const int r = v / (kRtCols / 8), c = (v % (kRtCols / 8)) * 8;
            uint4 val = make_uint4(0, 0, 0, 0);
            if (r < nt && h0 + c < H)
                val = *reinterpret_cast<const uint4*>(x + (size_t)(t0 + r) * H + h0 + c);
            *reinterpret_cast<uint4*>(&xs[r][c]) = val;
        }
        __syncthreads();
        if (e < E) {
            // this lane's 8 weights
            float w[8];
            const int c = lane * 8;
            if (h0 + c < H) {
                const uint4 a = *reinterpret_cast<const uint4*>(wr + (size_t)e * H + h0 + c);
                const uint32_t u[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    w[2 * i] = bf16_bits_to_f32(u[i] & 0xFFFFu);
                    w[2 * i + 1] = bf16_bits_to_f32(u[i] >> 16);
                }
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) w[i] = 0.0f;
            }
#pragma unroll
            for (int t = 0; t < kRtTok; ++t) {
                const uint4 a = *reinterpret_cast<const uint4*>(&xs[t][c]);
                const uint32_t u[4] = {a.x, a.y, a.z, a.w};
                float s = acc[t];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    s = fmaf(bf16_bits_to_f32(u[i] & 0xFFFFu), w[2 * i], s);
                    s = fmaf(bf16_bits_to_f32(u[i] >> 16), w[2 * i + 1], s);
                }
                acc[t] = s;
            }
        }
    }
    if (e >= E) return;
    const float b = bias ? bias[e] : 0.0f;
#pragma unroll
    for (int t = 0; t < kRtTok; ++t) {
        float s = acc[t];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (lane == (t & 31) && t < nt) logits[(size_t)(t0 + t) * E + e] = s + b;
    }
}

// ---------------------------------------------------------------- softmax top-k
//
// One warp per token.  k rounds of a warp arg-max over the remaining logits (larger value
// first, equal values: lower id first), then w_j = exp(l_j - l_0) / sum_i exp(l_i - l_0)
// over the selected logits.
__global__ void __launch_bounds__(256) topk_kernel(
    const float* __restrict__ logits_src, const float* __restrict__ bias, int T, int E, int k,
    int32_t* __restrict__ ids, float* __restrict__ wts, float* __restrict__ logits_out)
{
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (warp >= T) return;
    const int t = warp;
    constexpr int kPer = kMaxExperts / 32;
    float v[kPer];
    uint32_t used = 0;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int e = i * 32 + lane;
        float l = -INFINITY;
        if (e < E) {
            l = logits_src[(size_t)t * E + e] + (bias ? bias[e] : 0.0f);
            if (logits_out) logits_out[(size_t)t * E + e] = l;
        }
        v[i] = l;
    }
    float sel_l[kMaxTopK];
    int sel_e[kMaxTopK];
    for (int j = 0; j < k; ++j) {
        float best = -INFINITY;
        int be = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            const int e = i * 32 + lane;
            if (e < E && !((used >> i) & 1u)) {
                if (v[i] > best || (v[i] == best && e < be)) {
                    best = v[i];
                    be = e;
                }
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ob = __shfl_xor_sync(0xffffffffu, best, o);
            const int oe = __shfl_xor_sync(0xffffffffu, be, o);
            if (ob > best || (ob == best && oe < be)) {
                best = ob;
                be = oe;
            }
        }
        if ((be & 31) == lane) used |= 1u << (be >> 5);
        sel_l[j] = best;
        sel_e[j] = be;
    }
    if (lane == 0) {
        float z = 0.0f;
        for (int j = 0; j < k; ++j) z += expf(sel_l[j] - sel_l[0]);
        for (int j = 0; j < k; ++j) {
            ids[(size_t)t * k + j] = sel_e[j];
            wts[(size_t)t * k + j] = expf(sel_l[j] - sel_l[0]) / z;
        }
    }
}

// ---------------------------------------------------------------- grouping
//
// Stable counting sort of the local pairs by local expert, in three launches:
//   hist    per block of kPairsPerBlock pairs: count of each local expert
//   scan    per expert: prefix over blocks; per group: padded offsets, tile table,
//           shared-expert rows and padding markers
//   scatter per block: one warp walks its pairs in order; pairs of the same expert in a
//           32-pair step are ranked with a match mask, so rows keep ascending pair order.

__global__ void __launch_bounds__(256) perm_hist_kernel(const int32_t* __restrict__ ids, int P,
                                                        int E, int off, int El,
                                                        int32_t* __restrict__ hist,
                                                        uint32_t* status)
{
    __shared__ int32_t cnt[kMaxExperts];
    for (int e = threadIdx.x; e < El; e += blockDim.x) cnt[e] = 0;
    __syncthreads();
    const int p0 = blockIdx.x * kPairsPerBlock;
    const int p1 = min(P, p0 + kPairsPerBlock);
    bool bad = false;
    for (int p = p0 + threadIdx.x; p < p1; p += blockDim.x) {
        const int id = ids[p];
        if (id < 0 || id >= E) {
            bad = true;
            continue;
        }
        const int le = id - off;
        if (le >= 0 && le < El) atomicAdd(&cnt[le], 1);
    }
    if (bad) set_status(status, MOE_DEV_BAD_EXPERT_ID);
    __syncthreads();
    for (int e = threadIdx.x; e < El; e += blockDim.x) hist[(size_t)blockIdx.x * El + e] = cnt[e];
}

__global__ void __launch_bounds__(1024) perm_scan_kernel(
    const int32_t* __restrict__ hist, int nblk, int El, int T, int k, int shared_rows,
    int rows_cap, int32_t* __restrict__ blkoff, int32_t* __restrict__ counts,
    int32_t* __restrict__ offsets, int32_t* __restrict__ mb_start,
    int32_t* __restrict__ perm_src, uint32_t* status)
{
    __shared__ int32_t s_cnt[kMaxExperts + 1];
    __shared__ int32_t s_pad[kMaxExperts + 2];
    __shared__ int32_t s_mb[kMaxExperts + 2];
    const int G = El + 1;  // groups: routed experts, then the shared expert
    for (int g = threadIdx.x; g < G; g += blockDim.x) {
        int run = 0;
        if (g < El) {
            for (int b = 0; b < nblk; ++b) {
                blkoff[(size_t)b * El + g] = run;
                run += hist[(size_t)b * El + g];
            }
        } else {
            run = shared_rows;
        }
        s_cnt[g] = run;
        counts[g] = run;
    }
    __syncthreads();
    if (threadIdx.x == 0) {  // exclusive scans of padded sizes and 128-row blocks
        int a = 0, m = 0;
        for (int g = 0; g < G; ++g) {
            s_pad[g] = a;
            s_mb[g] = m;
            a += round_up(s_cnt[g], kRowAlign);
            m += (s_cnt[g] + kRowAlign - 1) / kRowAlign;
        }
        s_pad[G] = a;
        s_mb[G] = m;
        if (a > rows_cap) set_status(status, MOE_DEV_ROWS_OVERFLOW);
    }
    __syncthreads();
    for (int g = threadIdx.x; g <= G; g += blockDim.x) {
        offsets[g] = s_pad[g];
        mb_start[g] = s_mb[g];
    }
    // padding rows -> -1; shared rows -> T*k + t (routed rows are written by the scatter)
    const int total = min(s_pad[G], rows_cap);
    for (int r = threadIdx.x; r < total; r += blockDim.x) {
        int lo = 0, hi = G;  // s_pad[lo] <= r < s_pad[hi]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (s_pad[mid] <= r) lo = mid;
            else hi = mid;
        }
        const int i = r - s_pad[lo];
        if (i >= s_cnt[lo]) perm_src[r] = -1;
        else if (lo == El) perm_src[r] = T * k + i;
    }
}

__global__ void __launch_bounds__(32) perm_scatter_kernel(
    const int32_t* __restrict__ ids, int P, int E, int off, int El,
    const int32_t* __restrict__ blkoff, const int32_t* __restrict__ offsets, int rows_cap,
    int32_t* __restrict__ perm_src, int32_t* __restrict__ inv)
{
    __shared__ int32_t cursor[kMaxExperts];
    const int lane = threadIdx.x;
    for (int e = lane; e < El; e += 32)
        cursor[e] = offsets[e] + blkoff[(size_t)blockIdx.x * El + e];
    __syncwarp();
    const int p0 = blockIdx.x * kPairsPerBlock;
    const int p1 = min(P, p0 + kPairsPerBlock);
    const uint32_t lt = (1u << lane) - 1u;
    for (int base = p0; base < p1; base += 32) {
        const int p = base + lane;
        int le = -1;
        if (p < p1) {
            const int id = ids[p];
            if (id >= 0 && id < E) {
                le = id - off;
                if (le < 0 || le >= El) le = -1;
            }
        }
        const uint32_t grp = __match_any_sync(0xffffffffu, le);
        const int leader = __ffs(grp) - 1;
        int b = 0;
        if (le >= 0 && lane == leader) {
            b = cursor[le];
            cursor[le] = b + __popc(grp);
        }
        b = __shfl_sync(0xffffffffu, b, leader);
        __syncwarp();
        if (p < p1) {
            int row = -1;
            if (le >= 0) {
                row = b + __popc(grp & lt);
                if (row >= rows_cap) row = -1;
                else perm_src[row] = p;
            }
            inv[p] = row;
        }
    }
}

}  // namespace moe
