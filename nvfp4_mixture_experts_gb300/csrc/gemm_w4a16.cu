// W4A16 grouped GEMMs (16-bit activations x NVFP4 weights) on tcgen05, shaped for decode.
//
// Swap-AB: the MMA's M side (128 rows) is a tile of one expert's weight rows and the N side
// a block of BN (16, 32 or 64) of that expert's token rows; D[weight row][token] is in TMEM.
// With few tokens per expert the tensor work is small and the kernel is a weight stream:
//   * raw weight blobs (one per (expert, 128-row tile, 256-element k-stage): FP4 codes in a
//     128-byte swizzled image + 4 E4M3 scale atoms, 18 KB) flow through a deep shared-memory
//     ring by 1-D bulk copies;
//   * eight warps expand each blob into 16-bit values and write them straight into TMEM,
//     where tcgen05.mma reads its A operand, so the expanded weights never pass through
//     shared memory; each warp issues its TMEM stores for one blob and waits for them only
//     after expanding the next;
//   * the token tiles (4 x BN x 64 16-bit values per blob) arrive by TMA into a second ring,
//     deeper than the 3 TMEM slots so that their L2 latency stays hidden, and are the B
//     operand.
//
// Two operand flavours, both with exact products (E2M1 x E4M3 has at most 6 significant
// bits and lies in [2^-10, 2688]):
//   kF16 (gate_up): A and B fp16.  Codes expand with cvt.rn.f16x2.e2m1x2, scales with
//     cvt.rn.f16x2.e4m3x2, one fp16x2 multiply per pair.  The activations are fp16 copies of
//     x * gs_a (gs_a a power of two, see gather_f16_kernel); alpha = 1 / (gs_a * gs_w).
//   bf16 (down): A and B bf16 (the intermediate stays bf16).  An E2M1 code placed in bf16
//     bit positions (magnitude bits at 6..8, sign at 15) is its value x 2^-126 (code 0.5 is
//     a bf16 subnormal); times the block scale in bf16 taken x 2^119 it is value x scale x
//     2^-7, exactly.  alpha = 2^7 / gs_w.  The blobs of this flavour store the 8 codes of
//     each 32-bit word in nibble order 0,2,4,6,1,3,5,7, so that nibbles j and j + 4 (elements
//     2j, 2j + 1) become one bf16 pair with a shift, a multiply and a mask.
//
// Warp roles (480 threads):
//   warp 0     raw blob producer (constant data: starts without waiting for the previous
//              kernel)
//   warp 1     TMEM allocation; one thread issues the MMAs (kind::f16, M128 N=BN K16,
//              A from TMEM, B from shared memory)
//   warps 2-5  epilogue (TMEM lane quarter warp % 4 = 32 weight rows each)
//   warps 6-13 expansion: warp w writes lane quarter w % 4, k-steps 2h, 2h + 1 of each
//              blob (h = (w - 6) / 4)
//   warp 14    token tile producer (after the previous kernel's writes are visible)
// TMEM columns: accumulators [0, 2 BN), A slots 128 (1 + s) (128 columns = 256 16-bit
// values per row).  Every wait is bounded; a wait that runs out sets MOE_DEV_WAIT_TIMEOUT
// and every role stops.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kernels.cuh"

namespace moe {

namespace {

constexpr uint32_t kTmemCols = 512;
constexpr int kAcol0 = 128;
constexpr int kASlots = 3;  // A slots in TMEM: one blob (128 columns) each

struct W16Ctl {
    uint64_t* raw_full;    // [raw] blob landed (tx bytes)
    uint64_t* raw_empty;   // [raw] 8 expansion warps done with the blob
    uint64_t* b_full;      // [SB] token tiles landed (tx bytes)
    uint64_t* b_empty;     // [SB] MMAs reading token tiles s are complete
    uint64_t* a_full;      // [3] 8 expansion warps wrote the A slot
    uint64_t* a_empty;     // [3] MMAs reading A slot s are complete
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

__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ uint32_t f16x2_mul(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Two E4M3 scales (low byte first) -> fp16x2 (exact).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two)
{
    uint32_t d;
    asm("{\n\t.reg .b16 s;\n\tcvt.u16.u32 s, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, s;\n\t}"
        : "=r"(d)
        : "r"(two));
    return d;
}

// One k-step (64 elements of row r) of a blob -> 32 columns of 16-bit pairs.
template <bool kF16>
__device__ __forceinline__ void expand_kstep(const uint8_t* blob, int r, int j, uint32_t (&o)[32])
{
    const uint4 q0 = *reinterpret_cast<const uint4*>(blob + r * 128 + (((2 * j) ^ (r & 7)) << 4));
    const uint4 q1 =
        *reinterpret_cast<const uint4*>(blob + r * 128 + (((2 * j + 1) ^ (r & 7)) << 4));
    const uint32_t sw =
        *reinterpret_cast<const uint32_t*>(blob + 16384 + 512 * j + (r & 31) * 16 + (r >> 5) * 4);
    const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
    if constexpr (kF16) {
        // scale of elements 16s..16s+15 in both halves
        const uint32_t s01 = e4m3x2_to_f16x2(sw & 0xFFFFu), s23 = e4m3x2_to_f16x2(sw >> 16);
        const uint32_t sc[4] = {__byte_perm(s01, 0, 0x1010), __byte_perm(s01, 0, 0x3232),
                                __byte_perm(s23, 0, 0x1010), __byte_perm(s23, 0, 0x3232)};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            uint32_t e0, e1, e2, e3;
            asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
                "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
                "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
                "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
                "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
                "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
                : "=r"(e0), "=r"(e1), "=r"(e2), "=r"(e3)
                : "r"(w[i]));
            const uint32_t s = sc[i >> 1];
            o[4 * i] = f16x2_mul(e0, s);
            o[4 * i + 1] = f16x2_mul(e1, s);
            o[4 * i + 2] = f16x2_mul(e2, s);
            o[4 * i + 3] = f16x2_mul(e3, s);
        }
    } else {
        uint32_t sc[4];
#pragma unroll
        for (int s = 0; s < 4; ++s) {
            const float v = __fmul_rn(e4m3_to_f32((sw >> (8 * s)) & 0xFFu), 0x1p119f);
            const uint32_t b = __bfloat16_as_ushort(__float2bfloat16_rn(v));
            sc[s] = b | (b << 16);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                // nibbles jj, jj + 4: shifted copies by 6 and 12 bits do not overlap, so one
                // multiply places magnitude bits at 6..8 and the sign at 15 in both halves
                const uint32_t x = (w[i] >> (4 * jj)) & 0x000F000Fu;
                o[4 * i + jj] = bf16x2_mul((x * 0x1040u) & 0x81C081C0u, sc[i >> 1]);
            }
    }
}

}  // namespace

template <int BN, bool kF16>
__global__ void __launch_bounds__(kW16Threads, 1)
    gemm_w4a16_kernel(const __grid_constant__ CUtensorMap tmB, GemmArgs args)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t u0 = smem_u32(smem_raw);
    uint8_t* raw = smem_raw + (((u0 + 1023u) & ~1023u) - u0);
    const int RS = args.raw_slots, SB = args.stages;
    constexpr int SA = kASlots;
    constexpr int kBTile = BN * 128;        // one k-step of BN token rows
    constexpr int kBSlot = 4 * kBTile;      // one blob's worth
    uint8_t* btiles = raw + RS * kNvf4TileBytes;
    W16Ctl c;
    c.raw_full = reinterpret_cast<uint64_t*>(btiles + SB * kBSlot);
    c.raw_empty = c.raw_full + RS;
    c.b_full = c.raw_empty + RS;
    c.b_empty = c.b_full + SB;
    c.a_full = c.b_empty + SB;
    c.a_empty = c.a_full + SA;
    c.acc_full = c.a_empty + SA;
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
        for (int i = 0; i < SB; ++i) {
            mbar_init(&c.b_full[i], 1);
            mbar_init(&c.b_empty[i], 1);
        }
        for (int i = 0; i < SA; ++i) {
            mbar_init(&c.a_full[i], 8);
            mbar_init(&c.a_empty[i], 1);
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
    if (warp == 0) {  // token-block starts: exclusive prefix over the groups, one warp
        const int per = (args.G + 31) / 32, g0 = lane * per, g1 = min(args.G, g0 + per);
        int sum = 0;
        for (int g = g0; g < g1; ++g) sum += (c.counts[g] + BN - 1) / BN;
        int x = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        int acc = x - sum;
        for (int g = g0; g < g1; ++g) {
            c.tb_start[g] = acc;
            acc += (c.counts[g] + BN - 1) / BN;
        }
        if (lane == 31) c.tb_start[args.G] = x;
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
                    if (!mbar_wait_lazy(&c.raw_empty[rs], rph ^ 1u, c.abort_flag, 256)) {
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
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait_lazy(&c.b_empty[ws], wph ^ 1u, c.abort_flag, 64)) {
                        ok = false;
                        break;
                    }
                    const int nsub = min(4, (args.K - kb * 256) / 64);
                    mbar_arrive_expect_tx(&c.b_full[ws], nsub * kBTile);
                    for (int j = 0; j < nsub; ++j)
                        tma_load_2d(btiles + ws * kBSlot + j * kBTile, &tmB, &c.b_full[ws],
                                    kb * 256 + j * 64, ti.brow0, pol_a);
                    issued |= 1u << ws;
                    issued_par = (issued_par & ~(1u << ws)) | (wph << ws);
                    if (++ws == SB) {
                        ws = 0;
                        wph ^= 1u;
                    }
                }
            }
            if (!ok) {
                set_status(args.status, MOE_DEV_WAIT_TIMEOUT);
                *c.abort_flag = 1;
            }
            for (int s = 0; s < SB; ++s)
                if ((issued >> s) & 1u) mbar_wait(&c.b_full[s], (issued_par >> s) & 1u, c.zero);
        }
    } else if (warp >= 6) {
        // expansion: lane = weight row r of quarter qd; k-steps 2h and 2h + 1 of each blob
        const int qd = warp & 3, h = (warp - 6) >> 2;
        const int r = 32 * qd + lane;
        const uint32_t trow = tmem + ((uint32_t)(32 * qd) << 16) + kAcol0;
        int rs = 0, ws = 0;
        uint32_t rph = 0, wph = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
            for (int kb = 0; kb < KB; ++kb) {
                if (!w16_wait(&c.raw_full[rs], rph, c.abort_flag) ||
                    !w16_wait(&c.a_empty[ws], wph ^ 1u, c.abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int nsub = min(4, (args.K - kb * 256) / 64);
                const uint8_t* blob = raw + rs * kNvf4TileBytes;
                uint32_t o0[32], o1[32];
                if (2 * h < nsub) expand_kstep<kF16>(blob, r, 2 * h, o0);
                if (2 * h + 1 < nsub) expand_kstep<kF16>(blob, r, 2 * h + 1, o1);
                __syncwarp();
                if (lane == 0) mbar_arrive(&c.raw_empty[rs]);
                const uint32_t ta = trow + 128 * ws + 64 * h;
                if (2 * h < nsub) tmem_st32(ta, o0);
                if (2 * h + 1 < nsub) tmem_st32(ta + 32, o1);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&c.a_full[ws]);
                if (++rs == RS) {
                    rs = 0;
                    rph ^= 1u;
                }
                if (++ws == kASlots) {
                    ws = 0;
                    wph ^= 1u;
                }
            }
        }
        if (!ok && lane == 0) {
            set_status(args.status, MOE_DEV_WAIT_TIMEOUT);
            *c.abort_flag = 1;
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // kind::f16, fp32 D, A and B fp16 (format 0) or bf16 (format 1), M = 128, N = BN
            constexpr uint32_t idesc = kF16 ? ((1u << 4) | ((uint32_t)(BN >> 3) << 17) |
                                               ((uint32_t)(128 >> 4) << 24))
                                            : idesc_bf16(128, BN);
            int as = 0, bs = 0, it = 0;
            uint32_t aph = 0, bph = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x, ++it) {
                const int buf = it & 1;
                if (!mbar_wait(&c.acc_empty[buf], ((it >> 1) & 1) ^ 1u, c.abort_flag)) {
                    ok = false;
                    break;
                }
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait(&c.a_full[as], aph, c.abort_flag) ||
                        !mbar_wait(&c.b_full[bs], bph, c.abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const int nsub = min(4, (args.K - kb * 256) / 64);
                    const uint32_t at = tmem + kAcol0 + 128 * as;
                    for (int j = 0; j < nsub; ++j) {
                        const uint64_t bd = sdesc_sw128(smem_u32(btiles + bs * kBSlot + j * kBTile));
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            tc_mma_bf16_ts(tmem + buf * BN, at + 32 * j + 8 * kk, bd + 2 * kk,
                                           idesc, (kb | j | kk) != 0);
                    }
                    tc_commit(&c.a_empty[as]);
                    tc_commit(&c.b_empty[bs]);
                    if (++as == kASlots) {
                        as = 0;
                        aph ^= 1u;
                    }
                    if (++bs == SB) {
                        bs = 0;
                        bph ^= 1u;
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
            const float gw = args.gs_w[ti.g];
            const float alpha = kF16 ? __frcp_rn(__fmul_rn(*args.gs_a, gw))
                                     : __fmul_rn(__frcp_rn(gw), 128.0f);
            float wl[kNW];  // kEpiDown: routing weight of token column lane + 32 i
#pragma unroll
            for (int i = 0; i < kNW; ++i) {
                wl[i] = 0.0f;
                const int n = lane + 32 * i;
                if (args.epilogue == kEpiDown && n < ti.rows) {
                    const int pair = args.perm_src[ti.brow0 + n];
                    wl[i] = !pair_ok(pair, args.status) ? 0.0f
                            : pair < args.Tk            ? args.topk_w[pair]
                                                        : 1.0f;
                }
            }
            int okw = 1;  // (a whole tile: the lane sleeps between polls)
            if (lane == 0) okw = mbar_wait_lazy(&c.acc_full[buf], (it >> 1) & 1, c.abort_flag, 256);
            if (!__shfl_sync(0xffffffffu, okw, 0)) {
                if (lane == 0) {
                    set_status(args.status, MOE_DEV_WAIT_TIMEOUT);
                    *c.abort_flag = 1;
                }
                break;
            }
            tc_fence_after();
            float r[BN];  // the tile's D
            {
                uint32_t p[BN];
#pragma unroll
                for (int hh = 0; hh < BN / 16; ++hh)
                    tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + buf * BN + 16 * hh,
                              *reinterpret_cast<uint32_t(*)[16]>(p + 16 * hh));
                tmem_ld_wait();
#pragma unroll
                for (int n = 0; n < BN; ++n) r[n] = __uint_as_float(p[n]);
            }
            tc_fence_before();
            mbar_arrive(&c.acc_empty[buf]);  // the accumulator is free once in registers
            if (args.epilogue == kEpiDown) {
                float* ycol = args.out_f32 + 128 * ti.nb + m;
#pragma unroll
                for (int n = 0; n < BN; ++n) {
                    const float wn = __shfl_sync(0xffffffffu, wl[n >> 5], n & 31);
                    if (n < ti.rows)
                        ycol[(int64_t)(ti.brow0 + n) * args.N] =
                            r[n] * __fmul_rn(alpha, wn);
                }
            } else {
                // tile row 32q + 16u + i is gate (u = 0) / up (u = 1) of feature
                // 64 nb + 16 q + i: the up value of a gate lane sits 16 lanes higher
                const int f = 64 * ti.nb + 16 * q + (lane & 15);
                const bool gate = lane < 16;
#pragma unroll
                for (int n = 0; n < BN; ++n) {
                    const float v = __fmul_rn(r[n], alpha);
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

W16Kernel w4a16_kernel(int bn, bool f16)
{
    if (f16)
        return bn == 16 ? gemm_w4a16_kernel<16, true>
                        : bn == 32 ? gemm_w4a16_kernel<32, true> : gemm_w4a16_kernel<64, true>;
    return bn == 16 ? gemm_w4a16_kernel<16, false>
                    : bn == 32 ? gemm_w4a16_kernel<32, false> : gemm_w4a16_kernel<64, false>;
}

}  // namespace moe
