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
// logits = x . Wr^T on the tensor cores (kind::f16, bf16 operands, fp32 accumulation in
// TMEM).  Tile: 128 tokens x bn experts (64 or 160); grid (token tiles, expert tiles,
// k-splits).  Each
// k-split writes its partial sums to part[split][T][E]; the top-k kernel adds the splits
// in a fixed order (deterministic), then the bias.  Rows past T and experts past E are
// zero-filled by the TMA and never stored.
//   warp 0: TMA producer (x tile 128 x 64, Wr tile bn x 64 per stage)
//   warp 1: TMEM allocation, MMA issue (4 x K16 per stage)
//   warps 2..5: epilogue, one TMEM lane quarter (32 tokens) each
constexpr int kRgStages = 4;
constexpr int kRgStageBytes = 16384 + 160 * 128;  // x tile + the widest expert tile

// Expert-tile width: 64 experts for small T (more CTAs for the weight stream), 160 for
// large T (fewer re-reads of the x tile, more work per MMA).
int router_bn(int T, int E) { return (T >= 1024 && E > 64) ? 160 : 64; }

__global__ void __launch_bounds__(192, 1) router_gemm_kernel(
    const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW, int T,
    int E, int H, int k_per_split, int bn, float* __restrict__ part, uint32_t* status,
    uint32_t* clear0, uint32_t* clear1)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t u = smem_u32(smem_raw);
    uint8_t* st = smem_raw + (((u + 1023u) & ~1023u) - u);
    uint64_t* full = reinterpret_cast<uint64_t*>(st + kRgStages * kRgStageBytes);
    uint64_t* empty = full + kRgStages;
    uint64_t* acc = empty + kRgStages;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(acc + 1);
    int* flags = reinterpret_cast<int*>(tslot + 1);  // [0] abort, [1] zero
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.x * 128, n0 = blockIdx.y * bn;
    const int k0 = blockIdx.z * k_per_split;
    const int KB = min(k_per_split, H - k0) / 64;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kRgStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        mbar_init(acc, 1);
        flags[0] = flags[1] = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(tslot, 256);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    volatile int* abort = flags;
    pdl_wait();
    if (threadIdx.x == 0) {
        pdl_trigger();
        if (blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) {  // per-forward words
            if (clear0) *clear0 = 0u;
            if (clear1) clear1[0] = clear1[1] = 0u;  // both amax accumulators
        }
    }
    if (warp == 0 && lane == 0) {
        const uint64_t pol = policy_evict_last();
        uint32_t issued = 0, par = 0, phase = 0;
        int stg = 0;
        for (int kb = 0; kb < KB; ++kb) {
            if (!mbar_wait(&empty[stg], phase ^ 1u, abort)) {
                set_status(status, MOE_DEV_WAIT_TIMEOUT);
                flags[0] = 1;
                break;
            }
            uint8_t* sa = st + stg * kRgStageBytes;
            mbar_arrive_expect_tx(&full[stg], 16384u + (uint32_t)bn * 128u);
            tma_load_2d(sa, &tmX, &full[stg], k0 + kb * 64, m0, pol);
            tma_load_2d(sa + 16384, &tmW, &full[stg], k0 + kb * 64, n0, pol);
            issued |= 1u << stg;
            par = (par & ~(1u << stg)) | (phase << stg);
            if (++stg == kRgStages) {
                stg = 0;
                phase ^= 1u;
            }
        }
        for (int i = 0; i < kRgStages; ++i)
            if ((issued >> i) & 1u) mbar_wait(&full[i], (par >> i) & 1u, flags + 1);
    } else if (warp == 1 && lane == 0) {
        const uint32_t idesc = idesc_bf16(128, bn);
        uint32_t phase = 0;
        int stg = 0;
        bool ok = true;
        for (int kb = 0; kb < KB; ++kb) {
            if (!mbar_wait(&full[stg], phase, abort)) {
                set_status(status, MOE_DEV_WAIT_TIMEOUT);
                flags[0] = 1;
                ok = false;
                break;
            }
            tc_fence_after();
            uint8_t* sa = st + stg * kRgStageBytes;
            const uint64_t ad = sdesc_sw128(smem_u32(sa)), bd = sdesc_sw128(smem_u32(sa + 16384));
            for (int j = 0; j < 4; ++j) tc_mma_bf16(tmem, ad + 2 * j, bd + 2 * j, idesc, (kb | j) != 0);
            tc_commit(&empty[stg]);
            if (++stg == kRgStages) {
                stg = 0;
                phase ^= 1u;
            }
        }
        tc_commit(acc);  // also drains everything issued above
        if (!ok) mbar_wait(acc, 0, flags + 1);
    } else if (warp >= 2) {
        const int q = warp & 3;
        int ok = 1;
        if (lane == 0) ok = mbar_wait(acc, 0, abort) ? 1 : 0;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (ok && !flags[0]) {
            tc_fence_after();
            // each 32 x 32 piece (a lane per token) goes through shared memory, so that the
            // stores run along the rows (a lane per expert: 128 bytes a store) instead of one
            // 4-byte store per row.  The pipeline stages are free once acc completed (every
            // load they received was consumed by an MMA the commit covers).
            float* pc = reinterpret_cast<float*>(st) + (warp - 2) * 32 * 33;
            const int t0 = m0 + q * 32;
            float* dst = part + (size_t)blockIdx.z * T * E;
#pragma unroll 1
            for (int c = 0; c < bn / 32; ++c) {
                uint32_t r[32];
                tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + 32 * c, r);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; ++i) pc[lane * 33 + i] = __uint_as_float(r[i]);
                __syncwarp();
                const int col = n0 + 32 * c + lane;
                if (col < E)
#pragma unroll 4
                    for (int i = 0; i < 32 && t0 + i < T; ++i)
                        dst[(size_t)(t0 + i) * E + col] = pc[i * 33 + lane];
                __syncwarp();
            }
        } else if (lane == 0) {
            set_status(status, MOE_DEV_WAIT_TIMEOUT);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 256);
    }
}

int router_splits(int T, int E, int H, int num_sms)
{
    // Split K over more CTAs while the grid fills the GPU: up to 16 partial planes for small
    // batches (a weight stream, and the top-k's plane sum is small), 4 for large ones (where
    // that sum would dominate).  Each split is a whole number of 64-element k-steps, >= 256.
    const int bn = router_bn(T, E);
    const int tiles = ((T + 127) / 128) * ((E + bn - 1) / bn);
    const int cap = T <= 256 ? 16 : 4;
    int s = 1;
    while (s < cap && H % (2 * s * 64) == 0 && H / (2 * s) >= 256 && tiles * s * 2 <= num_sms)
        s *= 2;
    return s;
}

// ---------------------------------------------------------------- softmax top-k
//
// A block of 16 warps per topk_tokens_per_block(nsplit) consecutive tokens, so that the
// block holds 16 partial-sum rows (nsplit planes x tokens).  All threads first copy those
// rows, contiguous within each plane, into shared memory with every load in flight at once;
// then each logit is the sum of its nsplit partials in plane order plus the bias.  Warp j
// selects for token j: lane l holds experts l, l+32, ... as order-preserving integer keys,
// and each of the k rounds is a warp max over the keys, then a warp min over the ids that
// hold it (larger value first; equal values: lower id first); only the lane whose element
// was taken rescans.  Lane j keeps the j-th selection; w_j = exp(l_j - l_0) /
// sum_i exp(l_i - l_0) over the selected logits.  With amax_out, each block also folds
// max |x| over its tokens' rows of the layer input into *amax_out (fp32 bits, integer max;
// the router cleared it), so the forward needs no separate amax pass.
constexpr int kTopkWarps = 16;

__host__ __device__ int topk_tokens_per_block(int nsplit)
{
    return nsplit >= kTopkWarps ? 1 : kTopkWarps / nsplit;
}

size_t topk_smem(int nsplit, int E)
{
    return (size_t)nsplit * topk_tokens_per_block(nsplit) * E * sizeof(float);
}

// Unsigned keys in the order of the floats; -0 ranks with +0, and a NaN below -inf (key 1:
// key 0 marks an empty slot).
__device__ __forceinline__ uint32_t order_key(float f)
{
    if (f != f) return 1u;
    const uint32_t u = __float_as_uint(f == 0.0f ? 0.0f : f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_value(uint32_t key)
{
    return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

// PL: expert slots per lane (E <= 32 * PL), so the selection scans no more than it holds.
template <int PL>
__global__ void __launch_bounds__(32 * kTopkWarps) topk_kernel(
    const float* __restrict__ logits_src, int nsplit, const float* __restrict__ bias, int T,
    int E, int k, int32_t* __restrict__ ids, float* __restrict__ wts,
    float* __restrict__ logits_out, uint32_t* clear0, uint32_t* clear1,
    const uint16_t* __restrict__ x_amax, int H, uint32_t* amax_out, int32_t* zero_words,
    int nzero)
{
    extern __shared__ float s_part[];  // [nsplit][tokens of this block][E]
    __shared__ float s_xm[kTopkWarps];
    const int tpb = topk_tokens_per_block(nsplit);
    const int t0 = blockIdx.x * tpb;
    const int nt = min(tpb, T - t0);
    // max |x| over this block's token rows (the layer input is complete before the forward)
    float xm = 0.0f;
    if (amax_out) {
        const int64_t n8 = (int64_t)nt * H / 8;
        const uint4* xr = reinterpret_cast<const uint4*>(x_amax + (size_t)t0 * H);
        const int nthr = blockDim.x;
        for (int64_t q0 = threadIdx.x; q0 < n8; q0 += 4 * nthr) {  // four loads in flight
            uint4 v[4];
#pragma unroll
            for (int d = 0; d < 4; ++d)
                v[d] = q0 + d * nthr < n8 ? xr[q0 + d * nthr] : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int d = 0; d < 4; ++d) {
                const uint32_t u[4] = {v[d].x, v[d].y, v[d].z, v[d].w};
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    xm = fmaxf(xm, fmaxf(fabsf(bf16_bits_to_f32(u[j] & 0xFFFFu)),
                                         fabsf(bf16_bits_to_f32(u[j] >> 16))));
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) xm = fmaxf(xm, __shfl_xor_sync(0xffffffffu, xm, o));
        if ((threadIdx.x & 31) == 0) s_xm[threadIdx.x >> 5] = xm;
    }
    pdl_wait();
    if (threadIdx.x == 0) {
        pdl_trigger();
        if (blockIdx.x == 0) {  // per-forward words (when no router GEMM ran before)
            if (clear0) *clear0 = 0u;
            if (clear1) clear1[0] = clear1[1] = 0u;  // both amax accumulators
        }
    }
    // counters a later kernel of the forward starts from zero (the fused W4A16 GEMV's)
    if (blockIdx.x == 0)
        for (int i = threadIdx.x; i < nzero; i += blockDim.x) zero_words[i] = 0;
    const int per = nt * E;  // floats of this block in one plane
    uint32_t dyn_smem;
    asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn_smem));
    if (blockDim.x != 32 * kTopkWarps || dyn_smem < (uint32_t)(nsplit * per) * 4u) return;
    const size_t plane = (size_t)T * E;
    const float* src = logits_src + (size_t)t0 * E;
    const int nthr = blockDim.x;
    if ((E & 3) == 0 && (reinterpret_cast<uintptr_t>(logits_src) & 15) == 0) {  // 16-byte rows
        const int per4 = per >> 2, n4 = nsplit * per4;
        const size_t plane4 = plane >> 2;
        const float4* src4 = reinterpret_cast<const float4*>(src);
        float4* dst4 = reinterpret_cast<float4*>(s_part);
        for (int q0 = threadIdx.x; q0 < n4; q0 += 4 * nthr) {
            float4 r[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int q = q0 + u * nthr;
                if (q < n4) {
                    const int sp = q / per4;
                    r[u] = src4[sp * plane4 + (q - sp * per4)];
                }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (q0 + u * nthr < n4) dst4[q0 + u * nthr] = r[u];
        }
    } else {
        const int n = nsplit * per;
        for (int q0 = threadIdx.x; q0 < n; q0 += 8 * nthr) {
            float r[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int q = q0 + u * nthr;
                if (q < n) {
                    const int sp = q / per;
                    r[u] = src[sp * plane + (q - sp * per)];
                }
            }
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (q0 + u * nthr < n) s_part[q0 + u * nthr] = r[u];
        }
    }
    __syncthreads();
    if (amax_out && threadIdx.x == 0) {
        float m = 0.0f;
        for (int w = 0; w < kTopkWarps; ++w) m = fmaxf(m, s_xm[w]);
        atomicMax(amax_out, __float_as_uint(m));  // non-negative: bits order like values
    }
    for (int j = threadIdx.x; j < per; j += nthr) {
        float v = s_part[j];
        for (int sp = 1; sp < nsplit; ++sp) v += s_part[sp * per + j];
        if (bias) v += bias[j % E];
        if (logits_out) logits_out[(size_t)t0 * E + j] = v;
        s_part[j] = v;
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp >= nt) return;
    const float* lg = s_part + warp * E;
    const int ne = (E + 31) / 32;
    uint32_t key[PL];
    uint32_t live = 0;  // bit i: element i of this lane is a valid, unselected expert
#pragma unroll
    for (int i = 0; i < PL; ++i) {
        const int e = i * 32 + lane;
        const bool ok = i < ne && e < E;
        key[i] = ok ? order_key(lg[e]) : 0u;
        live |= (uint32_t)ok << i;
    }
    // this lane's best remaining element: the first (lowest id) of its largest key
    auto lane_best = [&](uint32_t& best, uint32_t& be) {
        best = 0u;
        be = 0xffffffffu;
#pragma unroll
        for (int i = 0; i < PL; ++i)
            if (((live >> i) & 1u) && key[i] > best) {
                best = key[i];
                be = (uint32_t)(i * 32 + lane);
            }
    };
    uint32_t lk, le;
    lane_best(lk, le);
    uint32_t my_key = 0u, my_e = 0u;
    for (int j = 0; j < k; ++j) {
        const uint32_t m = __reduce_max_sync(0xffffffffu, lk);
        const uint32_t be = __reduce_min_sync(0xffffffffu, lk == m ? le : 0xffffffffu);
        if (lane == j) {
            my_key = m;
            my_e = be;
        }
        if (le == be) {  // this lane's element was taken: drop it, rescan
            live &= ~(1u << (be >> 5));
            lane_best(lk, le);
        }
    }
    const float my_l = key_value(my_key);
    const float l0 = __shfl_sync(0xffffffffu, my_l, 0);
    const float ex = lane < k ? expf(my_l - l0) : 0.0f;
    float z = ex;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
    if (lane < k) {
        const int t = t0 + warp;
        ids[(size_t)t * k + lane] = (int32_t)my_e;
        wts[(size_t)t * k + lane] = ex / z;
    }
}

TopkKernel topk_kernel_for(int E)
{
    return E <= 128 ? topk_kernel<4> : E <= 256 ? topk_kernel<8> : E <= 384 ? topk_kernel<12>
         : E <= 512 ? topk_kernel<16> : topk_kernel<32>;
}

// ---------------------------------------------------------------- grouping
//
// Stable counting sort of the local pairs by local expert, in three launches:
//   hist    per block of kPairsPerBlock pairs: count of each local expert, stored
//           expert-major (hist[e][block]) so the scan reads each expert's counts in one piece
//   scan    per expert: prefix over blocks; per group: padded offsets, tile table,
//           shared-expert rows and padding markers
//   scatter a thread per pair: its rank among the pairs of its expert in its warp (match
//           mask), plus the counts of the earlier warps, plus the block's base, so rows keep
//           ascending pair order.

__global__ void __launch_bounds__(256) perm_hist_kernel(const int32_t* __restrict__ ids, int P,
                                                        int E, int off, int El,
                                                        int32_t* __restrict__ hist,
                                                        uint32_t* status)
{
    pdl_wait();
    if (threadIdx.x == 0) pdl_trigger();
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
    for (int e = threadIdx.x; e < El; e += blockDim.x) hist[(size_t)e * gridDim.x + blockIdx.x] = cnt[e];
}

__global__ void __launch_bounds__(1024) perm_scan_kernel(
    const int32_t* __restrict__ hist, int nblk, int El, int T, int k, int shared_rows,
    int rows_cap, int32_t* __restrict__ blkoff, int32_t* __restrict__ counts,
    int32_t* __restrict__ offsets, int32_t* __restrict__ mb_start,
    int32_t* __restrict__ perm_src, uint32_t* status)
{
    pdl_wait();
    if (threadIdx.x == 0) pdl_trigger();
    __shared__ int32_t s_cnt[kMaxExperts + 1];
    __shared__ int32_t s_pad[kMaxExperts + 2];
    __shared__ int32_t s_mb[kMaxExperts + 2];
    __shared__ int32_t s_wp[32], s_wm[32];
    const int G = El + 1;  // groups: routed experts, then the shared expert
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // per-group totals and per-block exclusive prefix: a warp per group, lanes over blocks;
    // each lane first loads its blocks' counts of all its groups (independent loads)
    constexpr int kMaxBlkPerLane = 2, kBatch = 8;  // loads in flight: kBatch x kMaxBlkPerLane
    if (nblk <= 32 * kMaxBlkPerLane) {
        for (int gb = warp; gb < G; gb += 32 * kBatch) {
            int v[kBatch][kMaxBlkPerLane];
#pragma unroll
            for (int gi = 0; gi < kBatch; ++gi)
#pragma unroll
                for (int i = 0; i < kMaxBlkPerLane; ++i) {
                    const int g = gb + 32 * gi, b = lane + 32 * i;
                    v[gi][i] = (g < El && b < nblk) ? hist[(size_t)g * nblk + b] : 0;
                }
#pragma unroll
            for (int gi = 0; gi < kBatch; ++gi) {
                const int g = gb + 32 * gi;
                if (g >= G) break;
                int total = 0;
                if (g < El) {
#pragma unroll
                    for (int i = 0; i < kMaxBlkPerLane; ++i) {
                        if (32 * i >= nblk) break;
                        int x = v[gi][i];
#pragma unroll
                        for (int o = 1; o < 32; o <<= 1) {
                            const int y = __shfl_up_sync(0xffffffffu, x, o);
                            if (lane >= o) x += y;
                        }
                        const int b = lane + 32 * i;
                        if (b < nblk) blkoff[(size_t)g * nblk + b] = total + x - v[gi][i];
                        total += __shfl_sync(0xffffffffu, x, 31);
                    }
                } else {
                    total = shared_rows;
                }
                if (lane == 0) {
                    s_cnt[g] = total;
                    counts[g] = total;
                }
            }
        }
    } else {
        for (int g = warp; g < G; g += 32) {
            int total = 0;
            if (g < El) {
                for (int b0 = 0; b0 < nblk; b0 += 32) {
                    const int b = b0 + lane;
                    const int v = b < nblk ? hist[(size_t)g * nblk + b] : 0;
                    int x = v;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const int y = __shfl_up_sync(0xffffffffu, x, o);
                        if (lane >= o) x += y;
                    }
                    if (b < nblk) blkoff[(size_t)g * nblk + b] = total + x - v;
                    total += __shfl_sync(0xffffffffu, x, 31);
                }
            } else {
                total = shared_rows;
            }
            if (lane == 0) {
                s_cnt[g] = total;
                counts[g] = total;
            }
        }
    }
    __syncthreads();
    // exclusive scans over groups of padded rows and 128-row blocks (2 groups per thread)
    const int g0 = 2 * threadIdx.x;
    const int c0 = g0 < G ? s_cnt[g0] : 0, c1 = g0 + 1 < G ? s_cnt[g0 + 1] : 0;
    const int p0 = round_up(c0, kRowAlign), p1 = round_up(c1, kRowAlign);
    const int m0 = (c0 + kRowAlign - 1) / kRowAlign, m1 = (c1 + kRowAlign - 1) / kRowAlign;
    int xp = p0 + p1, xm = m0 + m1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int yp = __shfl_up_sync(0xffffffffu, xp, o), ym = __shfl_up_sync(0xffffffffu, xm, o);
        if (lane >= o) {
            xp += yp;
            xm += ym;
        }
    }
    if (lane == 31) {
        s_wp[warp] = xp;
        s_wm[warp] = xm;
    }
    __syncthreads();
    if (warp == 0) {
        int a = s_wp[lane], b = s_wm[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int ya = __shfl_up_sync(0xffffffffu, a, o), yb = __shfl_up_sync(0xffffffffu, b, o);
            if (lane >= o) {
                a += ya;
                b += yb;
            }
        }
        s_wp[lane] = a;  // inclusive warp totals
        s_wm[lane] = b;
    }
    __syncthreads();
    const int bp = (warp ? s_wp[warp - 1] : 0) + xp - (p0 + p1);  // exclusive prefix
    const int bm = (warp ? s_wm[warp - 1] : 0) + xm - (m0 + m1);
    if (g0 <= G) {
        s_pad[g0] = bp;
        s_mb[g0] = bm;
    }
    if (g0 + 1 <= G) {
        s_pad[g0 + 1] = bp + p0;
        s_mb[g0 + 1] = bm + m0;
    }
    __syncthreads();
    if (threadIdx.x == 0 && s_pad[G] > rows_cap) set_status(status, MOE_DEV_ROWS_OVERFLOW);
    for (int g = threadIdx.x; g <= G; g += blockDim.x) {
        offsets[g] = s_pad[g];
        mb_start[g] = s_mb[g];
    }
    // padding rows -> -1; shared rows -> T*k + t (routed rows are written by the scatter);
    // a warp per group
    for (int g = warp; g < G; g += 32) {
        const int start = s_pad[g], n = s_cnt[g], end = min(s_pad[g + 1], rows_cap);
        for (int r = start + (g == El ? 0 : n) + lane; r < end; r += 32) {
            const int i = r - start;
            perm_src[r] = i < n ? T * k + i : -1;
        }
    }
}

// The whole grouping in one CTA when every pair fits one block (decode): per-expert counts,
// the scans, the stable scatter and (write_padding) the padding markers.  Same outputs as
// hist + scan + scatter.  Thread i takes pair i (P <= 1024 = 32 warps x 32 lanes): its rank
// inside its group is (pairs of that group in earlier warps) + (earlier lanes of its warp),
// the first from a per-warp count table (dynamic shared memory, [32][G] uint16) turned into
// an exclusive prefix over warps by one thread per group.
__global__ void __launch_bounds__(1024) perm_small_kernel(
    const int32_t* __restrict__ ids, int P, int E, int off, int El, int T, int k,
    int shared_rows, int rows_cap, int write_padding, int32_t* __restrict__ counts,
    int32_t* __restrict__ offsets, int32_t* __restrict__ mb_start, int32_t* __restrict__ perm_src,
    int32_t* __restrict__ inv, uint32_t* status)
{
    pdl_wait();
    if (threadIdx.x == 0) pdl_trigger();
    __shared__ int32_t s_cnt[kMaxExperts + 1];
    __shared__ int32_t s_pad[kMaxExperts + 2];
    __shared__ int32_t s_mb[kMaxExperts + 2];
    __shared__ int32_t s_wp[32], s_wm[32];
    extern __shared__ uint16_t s_wtab[];  // [32][G]: pairs of group g in warp w, then prefix
    const int G = El + 1;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nw = (P + 31) / 32;  // warps that hold pairs: only their rows of the table
    for (int g = threadIdx.x; g < G; g += blockDim.x) s_cnt[g] = g < El ? 0 : shared_rows;
    for (int x = threadIdx.x; x < nw * G; x += blockDim.x) s_wtab[x] = 0;
    __syncthreads();
    // local expert of pair i (-1: dropped), per-expert counts, per-warp counts and ranks
    const int i = threadIdx.x;
    int le = -1;
    if (i < P) {
        const int id = ids[i];
        if (id < 0 || id >= E) {
            set_status(status, MOE_DEV_BAD_EXPERT_ID);
        } else {
            le = id - off;
            if (le < 0 || le >= El) le = -1;
            else atomicAdd(&s_cnt[le], 1);
        }
    }
    const uint32_t grp = __match_any_sync(0xffffffffu, le);
    const int rank = __popc(grp & ((1u << lane) - 1u));
    if (le >= 0 && rank == 0) s_wtab[warp * G + le] = (uint16_t)__popc(grp);
    __syncthreads();
    const int g0 = 2 * threadIdx.x;
    const int c0 = g0 < G ? s_cnt[g0] : 0, c1 = g0 + 1 < G ? s_cnt[g0 + 1] : 0;
    const int p0 = round_up(c0, kRowAlign), p1 = round_up(c1, kRowAlign);
    const int m0 = (c0 + kRowAlign - 1) / kRowAlign, m1 = (c1 + kRowAlign - 1) / kRowAlign;
    int xp = p0 + p1, xm = m0 + m1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int yp = __shfl_up_sync(0xffffffffu, xp, o), ym = __shfl_up_sync(0xffffffffu, xm, o);
        if (lane >= o) {
            xp += yp;
            xm += ym;
        }
    }
    if (lane == 31) {
        s_wp[warp] = xp;
        s_wm[warp] = xm;
    }
    // per group: exclusive prefix of its per-warp counts over the warps
    if (threadIdx.x < G) {
        int run = 0;
        for (int w = 0; w < nw; ++w) {
            const int c = s_wtab[w * G + threadIdx.x];
            s_wtab[w * G + threadIdx.x] = (uint16_t)run;
            run += c;
        }
    }
    __syncthreads();
    if (warp == 0) {
        int a = s_wp[lane], b = s_wm[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int ya = __shfl_up_sync(0xffffffffu, a, o), yb = __shfl_up_sync(0xffffffffu, b, o);
            if (lane >= o) {
                a += ya;
                b += yb;
            }
        }
        s_wp[lane] = a;
        s_wm[lane] = b;
    }
    __syncthreads();
    const int bp = (warp ? s_wp[warp - 1] : 0) + xp - (p0 + p1);
    const int bm = (warp ? s_wm[warp - 1] : 0) + xm - (m0 + m1);
    if (g0 <= G) {
        s_pad[g0] = bp;
        s_mb[g0] = bm;
    }
    if (g0 + 1 <= G) {
        s_pad[g0 + 1] = bp + p0;
        s_mb[g0 + 1] = bm + m0;
    }
    __syncthreads();
    if (threadIdx.x == 0 && s_pad[G] > rows_cap) set_status(status, MOE_DEV_ROWS_OVERFLOW);
    for (int g = threadIdx.x; g <= G; g += blockDim.x) {
        offsets[g] = s_pad[g];
        mb_start[g] = s_mb[g];
        if (g < G) counts[g] = s_cnt[g];
    }
    // the stable scatter: the pair's row, and its inverse
    if (i < P) {
        int row = -1;
        if (le >= 0) {
            row = s_pad[le] + s_wtab[warp * G + le] + rank;
            if (row >= rows_cap) row = -1;
            else perm_src[row] = i;
        }
        inv[i] = row;
    }
    // shared rows, and the padding markers when asked for
    for (int g = warp; g < G; g += 32) {
        const int start = s_pad[g], n = s_cnt[g], end = min(s_pad[g + 1], rows_cap);
        const int r_end = (write_padding || g == El) ? end : start;
        for (int r = start + (g == El ? 0 : n) + lane; r < r_end; r += 32) {
            const int q = r - start;
            perm_src[r] = q < n ? T * k + q : -1;
        }
    }
}

__global__ void __launch_bounds__(kPairsPerBlock) perm_scatter_kernel(
    const int32_t* __restrict__ ids, int P, int E, int off, int El,
    const int32_t* __restrict__ blkoff, const int32_t* __restrict__ offsets, int rows_cap,
    int32_t* __restrict__ perm_src, int32_t* __restrict__ inv)
{
    pdl_wait();
    if (threadIdx.x == 0) pdl_trigger();
    __shared__ int32_t cursor[kMaxExperts];
    extern __shared__ uint16_t s_wtab[];  // [32][El]: pairs of expert e in warp w, then prefix
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int e = threadIdx.x; e < El; e += blockDim.x)
        cursor[e] = offsets[e] + blkoff[(size_t)e * gridDim.x + blockIdx.x];
    for (int x = threadIdx.x; x < 32 * El; x += blockDim.x) s_wtab[x] = 0;
    __syncthreads();
    // a thread per pair: local expert (-1: dropped), rank among the warp's pairs of that
    // expert, per-warp counts
    const int i = blockIdx.x * kPairsPerBlock + threadIdx.x;
    int le = -1;
    if (i < P) {
        const int id = ids[i];
        if (id >= 0 && id < E) {
            le = id - off;
            if (le < 0 || le >= El) le = -1;
        }
    }
    const uint32_t grp = __match_any_sync(0xffffffffu, le);
    const int rank = __popc(grp & ((1u << lane) - 1u));
    if (le >= 0 && rank == 0) s_wtab[warp * El + le] = (uint16_t)__popc(grp);
    __syncthreads();
    for (int e = threadIdx.x; e < El; e += blockDim.x) {  // exclusive prefix over the warps
        int run = 0;
        for (int w = 0; w < 32; ++w) {
            const int c = s_wtab[w * El + e];
            s_wtab[w * El + e] = (uint16_t)run;
            run += c;
        }
    }
    __syncthreads();
    // rows in ascending pair order within each expert: block base, warp prefix, rank
    if (i < P) {
        int row = -1;
        if (le >= 0) {
            row = cursor[le] + s_wtab[warp * El + le] + rank;
            if (row >= rows_cap) row = -1;
            else perm_src[row] = i;
        }
        inv[i] = row;
    }
}

}  // namespace moe
