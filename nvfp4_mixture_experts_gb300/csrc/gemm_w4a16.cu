// W4A16 grouped GEMMs (bf16 activations x NVFP4 weights) on tcgen05, shaped for decode.
//
// Swap-AB: the MMA's M side (128 rows) is a tile of one expert's weight rows and the N side
// a block of BN (16, 32 or 64) of that expert's token rows; D[weight row][token] is in TMEM.
// With few tokens per expert the tensor work is small and the kernel is a weight stream:
//   * raw weight blobs (one per (expert, 128-row tile, 256-element k-stage): FP4 codes in a
//     128-byte swizzled image + 4 E4M3 scale atoms, 18 KB) flow through a deep shared-memory
//     ring by 1-D bulk copies;
//   * eight warps expand each 64-element sub-stage into bf16 and write it straight into
//     TMEM, where tcgen05.mma reads its A operand, so the expanded weights never pass
//     through shared memory;
//   * the token tile (BN x 64 bf16) arrives by TMA into a second ring and is the B operand.
//
// Exact products: an E2M1 code placed in bf16 bit positions (magnitude bits at 6..8, sign at
// 15) is the code's value x 2^-126 (code 0.5 is a bf16 subnormal); multiplying it by the
// block scale in bf16 taken x 2^119 gives value x scale x 2^-7 with no rounding (at most 6
// significant bits, always in the normal range).  The epilogue multiplies by 2^7 / gs_w.
// For this the W4A16 blobs store the eight codes of each 32-bit word in the nibble order
// 0,2,4,6,1,3,5,7, so one shift and mask yields the bf16 pair of two neighbouring elements.
//
// Warp roles (480 threads):
//   warp 0     raw blob producer (constant data: starts without waiting for the previous
//              kernel)
//   warp 1     TMEM allocation; one thread issues the MMAs (kind::f16, M128 N=BN K16,
//              A from TMEM, B from shared memory)
//   warps 2-5  epilogue (TMEM lane quarter warp % 4 = 32 weight rows each)
//   warps 6-13 dequantisation: warp w writes lane quarter w % 4, half (w - 6) / 4 of each
//              64-element sub-stage
//   warp 14    token tile producer (after the previous kernel's writes are visible)
// TMEM columns: accumulators [0, 2 BN), A slots 128 + 32 s.  Every wait is bounded; a wait
// that runs out sets MOE_DEV_WAIT_TIMEOUT and every role stops.
#include <cuda_bf16.h>

#include "kernels.cuh"

namespace moe {

namespace {

constexpr uint32_t kTmemCols = 512;
constexpr int kAcol0 = 128;

struct W16Ctl {
    uint64_t* raw_full;    // [raw] blob landed (tx bytes)
    uint64_t* raw_empty;   // [raw] 8 dequantisation warps done with the blob
    uint64_t* b_full;      // [S] token tile landed (tx bytes)
    uint64_t* a_full;      // [S] 8 dequantisation warps wrote the A slot
    uint64_t* work_empty;  // [S] MMAs reading A slot / token tile s are complete
    uint64_t* acc_full;    // [2]
    uint64_t* acc_empty;   // [2] 128 epilogue threads
    uint64_t* drain;
    uint32_t* tmem_slot;
    volatile int* abort_flag;
    int* zero;
    int32_t* counts;       // [G]
    int32_t* offsets;      // [G+1]
    int32_t* tb_start;     // [G+1] first token block of each group
};

struct W16Tile {
    int g, nb, rows, brow0;
};

template <int BN>
__device__ __forceinline__ W16Tile w16_decode(const GemmArgs& a, const W16Ctl& c, int NB, int t)
{
    int lo = 0, hi = a.G;  // last group whose first tile index is <= t
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (c.tb_start[mid] * NB <= t) lo = mid;
        else hi = mid;
    }
    const int g = lo;
    const int ntb = c.tb_start[g + 1] - c.tb_start[g];
    const int local = t - c.tb_start[g] * NB;
    const int tb = local % ntb;  // consecutive tiles share a weight tile (L2 reuse)
    W16Tile ti;
    ti.g = g;
    ti.nb = local / ntb;
    ti.rows = min(BN, c.counts[g] - BN * tb);
    ti.brow0 = c.offsets[g] + BN * tb;
    return ti;
}

__device__ __forceinline__ bool w16_wait(uint64_t* bar, uint32_t parity, volatile int* abort)
{
    int ok = 1;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, abort) ? 1 : 0;
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// Nibbles j and j + 4 of a code word (elements 2j and 2j + 1 in the W4A16 nibble order)
// -> bf16 pair of value x 2^-126: shifted copies of each nibble by 6 and 12 bits do not
// overlap, so one multiply places magnitude bits at 6..8 and the sign at 15 in both halves.
__device__ __forceinline__ uint32_t e2m1_pair_bits(uint32_t w, int j)
{
    const uint32_t x = (w >> (4 * j)) & 0x000F000Fu;
    return (x * 0x1040u) & 0x81C081C0u;
}

__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// E4M3 scale byte -> bf16 pair (both halves) of scale x 2^119 (exact).
__device__ __forceinline__ uint32_t scale_pair(uint32_t byte)
{
    const float v = __fmul_rn(e4m3_to_f32(byte & 0xFFu), 0x1p119f);
    const uint32_t b = __bfloat16_as_ushort(__float2bfloat16_rn(v));
    return b | (b << 16);
}

}  // namespace

template <int BN>
__global__ void __launch_bounds__(kW16Threads, 1)
    gemm_w4a16_kernel(const __grid_constant__ CUtensorMap tmB, GemmArgs args)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t u0 = smem_u32(smem_raw);
    uint8_t* raw = smem_raw + (((u0 + 1023u) & ~1023u) - u0);
    const int RS = args.raw_slots, S = args.stages;
    constexpr int kBTile = BN * 128;
    uint8_t* btiles = raw + RS * kNvf4TileBytes;
    W16Ctl c;
    c.raw_full = reinterpret_cast<uint64_t*>(btiles + S * kBTile);
    c.raw_empty = c.raw_full + RS;
    c.b_full = c.raw_empty + RS;
    c.a_full = c.b_full + S;
    c.work_empty = c.a_full + S;
    c.acc_full = c.work_empty + S;
    c.acc_empty = c.acc_full + 2;
    c.drain = c.acc_empty + 2;
    c.tmem_slot = reinterpret_cast<uint32_t*>(c.drain + 1);
    c.abort_flag = reinterpret_cast<volatile int*>(c.tmem_slot + 1);
    c.zero = reinterpret_cast<int*>(c.tmem_slot + 2);
    c.counts = reinterpret_cast<int32_t*>(c.tmem_slot + 4);
    c.offsets = c.counts + args.G;
    c.tb_start = c.offsets + args.G + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int NB = args.N / 128;
    const int KB = (args.K + 255) / 256;
    const int KSUB = args.K / 64;

    // group tables (written by the grouping kernels, complete before the previous kernel)
    for (int i = threadIdx.x; i <= args.G; i += blockDim.x) {
        c.offsets[i] = args.offsets[i];
        if (i < args.G) c.counts[i] = args.counts[i];
    }
    if (threadIdx.x == 0) {
        for (int i = 0; i < RS; ++i) {
            mbar_init(&c.raw_full[i], 1);
            mbar_init(&c.raw_empty[i], 8);
        }
        for (int i = 0; i < S; ++i) {
            mbar_init(&c.b_full[i], 1);
            mbar_init(&c.a_full[i], 8);
            mbar_init(&c.work_empty[i], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&c.acc_full[b], 1);
            mbar_init(&c.acc_empty[b], 128);
        }
        mbar_init(c.drain, 1);
        *c.abort_flag = 0;
        *c.zero = 0;
        fence_barrier_init();
    }
    if (warp == 14 && lane == 0) prefetch_tmap(&tmB);
    if (warp == 1) {
        tmem_alloc(c.tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (threadIdx.x == 0) {
        int acc = 0;
        for (int g = 0; g < args.G; ++g) {
            c.tb_start[g] = acc;
            acc += (c.counts[g] + BN - 1) / BN;
        }
        c.tb_start[args.G] = acc;
    }
    __syncthreads();
    const uint32_t tmem = *c.tmem_slot;
    const int ntiles = c.tb_start[args.G] * NB;

    if (warp == 0) {
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_first();
            int rs = 0;
            uint32_t rph = 0, issued = 0, issued_par = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
                const W16Tile ti = w16_decode<BN>(args, c, NB, t);
                const uint8_t* wt =
                    args.b_tiles + ((size_t)ti.g * NB + ti.nb) * KB * (size_t)kNvf4TileBytes;
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait(&c.raw_empty[rs], rph ^ 1u, c.abort_flag)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&c.raw_full[rs], kNvf4TileBytes);
                    bulk_load(raw + rs * kNvf4TileBytes, wt + (size_t)kb * kNvf4TileBytes,
                              kNvf4TileBytes, &c.raw_full[rs], pol_w);
                    issued |= 1u << rs;
                    issued_par = (issued_par & ~(1u << rs)) | (rph << rs);
                    if (++rs == RS) {
                        rs = 0;
                        rph ^= 1u;
                    }
                }
            }
            if (!ok) {
                set_status(args.status, MOE_DEV_WAIT_TIMEOUT);
                *c.abort_flag = 1;
            }
            // copies still in flight land before the CTA exits
            for (int s = 0; s < RS; ++s)
                if ((issued >> s) & 1u) mbar_wait(&c.raw_full[s], (issued_par >> s) & 1u, c.zero);
        }
    } else if (warp == 14) {
        if (lane == 0) {
            const uint64_t pol_a = policy_evict_last();
            pdl_wait();
            pdl_trigger();
            int ws = 0;
            uint32_t wph = 0, issued = 0, issued_par = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
                const W16Tile ti = w16_decode<BN>(args, c, NB, t);
                for (int j = 0; j < KSUB; ++j) {
                    if (!mbar_wait(&c.work_empty[ws], wph ^ 1u, c.abort_flag)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&c.b_full[ws], kBTile);
                    tma_load_2d(btiles + ws * kBTile, &tmB, &c.b_full[ws], j * 64, ti.brow0,
                                pol_a);
                    issued |= 1u << ws;
                    issued_par = (issued_par & ~(1u << ws)) | (wph << ws);
                    if (++ws == S) {
                        ws = 0;
                        wph ^= 1u;
                    }
                }
            }
            if (!ok) {
                set_status(args.status, MOE_DEV_WAIT_TIMEOUT);
                *c.abort_flag = 1;
            }
            for (int s = 0; s < S; ++s)
                if ((issued >> s) & 1u) mbar_wait(&c.b_full[s], (issued_par >> s) & 1u, c.zero);
        }
    } else if (warp >= 6) {
        // dequantisation: lane = weight row r of quarter qd, 32 elements (16 columns) of
        // each 64-element sub-stage
        const int qd = warp & 3, hf = (warp - 6) >> 2;
        const int r = 32 * qd + lane;
        const uint32_t trow = tmem + ((uint32_t)(32 * qd) << 16) + kAcol0 + 16 * hf;
        int rs = 0, ws = 0;
        uint32_t rph = 0, wph = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
            for (int kb = 0; kb < KB && ok; ++kb) {
                if (!w16_wait(&c.raw_full[rs], rph, c.abort_flag)) {
                    ok = false;
                    break;
                }
                const uint8_t* blob = raw + rs * kNvf4TileBytes;
                const int nsub = min(4, (args.K - kb * 256) / 64);
                for (int j = 0; j < nsub; ++j) {
                    if (!w16_wait(&c.work_empty[ws], wph ^ 1u, c.abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint4 q = *reinterpret_cast<const uint4*>(
                        blob + r * 128 + (((2 * j + hf) ^ (r & 7)) << 4));
                    const uint32_t sw = *reinterpret_cast<const uint32_t*>(
                        blob + 16384 + 512 * j + (r & 31) * 16 + (r >> 5) * 4);
                    const uint32_t s0 = scale_pair(sw >> (16 * hf));
                    const uint32_t s1 = scale_pair(sw >> (16 * hf + 8));
                    const uint32_t cw[4] = {q.x, q.y, q.z, q.w};
                    uint32_t o[16];
#pragma unroll
                    for (int i = 0; i < 4; ++i)
#pragma unroll
                        for (int jj = 0; jj < 4; ++jj)
                            o[4 * i + jj] = bf16x2_mul(e2m1_pair_bits(cw[i], jj), i < 2 ? s0 : s1);
                    tmem_st16(trow + 32 * ws, o);
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&c.a_full[ws]);
                    if (++ws == S) {
                        ws = 0;
                        wph ^= 1u;
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&c.raw_empty[rs]);
                if (++rs == RS) {
                    rs = 0;
                    rph ^= 1u;
                }
            }
        }
        if (!ok && lane == 0) {
            set_status(args.status, MOE_DEV_WAIT_TIMEOUT);
            *c.abort_flag = 1;
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16(128, BN);
            int ws = 0, it = 0;
            uint32_t wph = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x, ++it) {
                const int buf = it & 1;
                if (!mbar_wait(&c.acc_empty[buf], ((it >> 1) & 1) ^ 1u, c.abort_flag)) {
                    ok = false;
                    break;
                }
                for (int j = 0; j < KSUB; ++j) {
                    if (!mbar_wait(&c.a_full[ws], wph, c.abort_flag) ||
                        !mbar_wait(&c.b_full[ws], wph, c.abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t bd = sdesc_sw128(smem_u32(btiles + ws * kBTile));
                    const uint32_t at = tmem + kAcol0 + 32 * ws;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        tc_mma_bf16_ts(tmem + buf * BN, at + 8 * kk, bd + 2 * kk, idesc,
                                       (j | kk) != 0);
                    tc_commit(&c.work_empty[ws]);
                    if (++ws == S) {
                        ws = 0;
                        wph ^= 1u;
                    }
                }
                if (!ok) break;
                tc_commit(&c.acc_full[buf]);
            }
            if (!ok) {
                set_status(args.status, MOE_DEV_WAIT_TIMEOUT);
                *c.abort_flag = 1;
            }
            tc_commit(c.drain);  // every MMA issued above is complete after this
            mbar_wait(c.drain, 0, c.zero);
        }
        __syncwarp();
    } else {
        // epilogue: thread = weight row m of the tile (TMEM lane), BN token columns
        constexpr int kNW = (BN + 31) / 32;
        const int q = warp & 3;
        const int m = q * 32 + lane;
        const int I = args.N / 2;
        int it = 0;
        pdl_wait();
        for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++it) {
            const W16Tile ti = w16_decode<BN>(args, c, NB, t);
            const int buf = it & 1;
            const float alpha = __fmul_rn(__frcp_rn(args.gs_w[ti.g]), 128.0f);
            float wl[kNW];  // kEpiDown: routing weight of token column lane + 32 i
#pragma unroll
            for (int i = 0; i < kNW; ++i) {
                wl[i] = 0.0f;
                const int n = lane + 32 * i;
                if (args.epilogue == kEpiDown && n < ti.rows) {
                    const int pair = args.perm_src[ti.brow0 + n];
                    wl[i] = pair < args.Tk ? args.topk_w[pair] : 1.0f;
                }
            }
            if (!w16_wait(&c.acc_full[buf], (it >> 1) & 1, c.abort_flag)) {
                if (lane == 0) {
                    set_status(args.status, MOE_DEV_WAIT_TIMEOUT);
                    *c.abort_flag = 1;
                }
                break;
            }
            tc_fence_after();
            uint32_t r[BN];
#pragma unroll
            for (int h = 0; h < BN / 16; ++h)
                tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + buf * BN + 16 * h,
                          *reinterpret_cast<uint32_t(*)[16]>(r + 16 * h));
            tmem_ld_wait();
            tc_fence_before();
            mbar_arrive(&c.acc_empty[buf]);  // the accumulator is free once in registers
            if (args.epilogue == kEpiDown) {
                float* ycol = args.out_f32 + 128 * ti.nb + m;
#pragma unroll
                for (int n = 0; n < BN; ++n) {
                    const float wn = __shfl_sync(0xffffffffu, wl[n >> 5], n & 31);
                    if (n < ti.rows)
                        ycol[(int64_t)(ti.brow0 + n) * args.N] =
                            __uint_as_float(r[n]) * __fmul_rn(alpha, wn);
                }
            } else {
                // tile row 32q + 16u + i is gate (u = 0) / up (u = 1) of feature
                // 64 nb + 16 q + i: the up value of a gate lane sits 16 lanes higher
                const int f = 64 * ti.nb + 16 * q + (lane & 15);
                const bool gate = lane < 16;
#pragma unroll
                for (int n = 0; n < BN; ++n) {
                    const float v = __fmul_rn(__uint_as_float(r[n]), alpha);
                    const float up = __shfl_down_sync(0xffffffffu, v, 16);
                    if (n >= ti.rows) continue;
                    const int64_t row = ti.brow0 + n;
                    if (args.epilogue == kEpiGateUpF32)
                        args.out_f32[row * args.N + (gate ? f : I + f)] = v;
                    else if (gate)
                        args.out_bf16[row * I + f] =
                            __bfloat16_as_ushort(__float2bfloat16_rn(silu_mul(v, up)));
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

W16Kernel w4a16_kernel(int bn)
{
    return bn == 16 ? gemm_w4a16_kernel<16> : bn == 32 ? gemm_w4a16_kernel<32>
                                                       : gemm_w4a16_kernel<64>;
}

}  // namespace moe
