// NVFP4 x NVFP4 (W4A4) grouped GEMMs for many rows per expert: the weight-stationary form.
//
// The MMA's M side is 128 rows of one expert's weight matrix and its N side is the expert's
// token rows, up to tile_n of them per tile (a multiple of 16), so a group of r rows costs
// round_up(r, 16) MMA columns instead of 128-row blocks, and each 128-row weight tile passes
// through shared memory once per token tile instead of once per 128-row block.  The
// accumulator D[weight row][token] sits in TMEM (lane = weight row, column = token); the
// epilogue reads it transposed: for gate_up a warp's 32 lanes are 16 gate and the matching
// 16 up features (the weights' interleave), so silu(gate)*up pairs lanes l and l+16 and one
// NVFP4 block of 16 intermediate features is one half-warp; for down each lane writes one
// output feature of a token row (32 consecutive features per warp store).
//
// Tiles: a group of r local rows (starting on a multiple of 128 padded rows) is cut into
// token tiles of 128 rows until at most tile_n remain, which form the last tile; each
// token tile pairs with every 128-row weight tile.  Tile order: group, weight tile, token
// tile, so consecutive tiles share a weight tile (read from L2 the second time).  The tile
// list is built in shared memory at kernel start from the group counts (a block scan).
//
// Warp roles:
//   warp 0       producer: weight blob (bulk copy), token codes (TMA, a 128-row box and
//                16-row boxes), token scale atoms (bulk copies), into a ring of stages
//   warp 1       TMEM allocation; one thread issues tcgen05.mma
//   warps 2..     epilogue: kSwHalves warps per TMEM lane quarter, alternate 32-column chunks
//   last 4 warps  scale warps: each stage's weight and token scale factors smem -> TMEM
//
// TMEM (512 columns): accumulator buffer b at column 256 b (tile_n columns); the scale
// slots fill the columns tile_n..255 and 256 + tile_n..511, each holding one stage's weight
// scales (4 columns per 64-element k-step, column c = rows 32c + lane) at +0 and token scales
// (4 columns per k-step for tile_n <= 128, else 8; column c = token rows 32c + lane) at +16.
// The slots decide how many k-stages can be in the tensor pipe at once (tile_n 128: 8 slots;
// 160: 4; 208: 2), against the weight traffic per token, which falls as tile_n grows.
//
// Every pipeline wait is bounded: a wait that runs out sets MOE_DEV_WAIT_TIMEOUT in the
// status word and makes all roles stop, drain their copies in flight, free TMEM and exit.
#include <cuda_fp16.h>

#include "kernels.cuh"

namespace moe {

namespace {

constexpr int kSwStageW = kNvf4TileBytes;        // weight blob: codes (SMEM image) + scales
constexpr int kSwEpiWarps = (kSwThreads / 32) - 6;  // after the producer, MMA, scale warps
constexpr int kSwHalves = kSwEpiWarps / 4;            // epilogue warps per TMEM lane quarter
constexpr int kSwChunks = ((kSwNmax + 31) / 32 + kSwHalves - 1) / kSwHalves;  // per warp
constexpr int kSwMaxSlots = 8;
constexpr int kSwCtlBytes = 512;  // barriers (4 x 8 + 5) and flags
// gate_up epilogue: each epilogue warp's [32 token columns][16 features] fp32 tile, rows
// padded to 20 floats (80 bytes: the 16-byte row reads of a quarter-warp hit distinct banks)
constexpr int kSwXposeStride = 20;
constexpr int kSwXposeBytes = kSwEpiWarps * 32 * kSwXposeStride * 4;

struct SwTile {
    int g;    // group
    int nb;   // 128-row weight tile
    int r0;   // first padded row of the token tile
    int n;    // token rows of the tile (1..tile_n)
};

struct SwTables {
    const int32_t* rows;   // [G] rows each group runs (its count, clamped to the capacity)
    const int32_t* ntt;    // [G] token tiles of each group
    const int32_t* off;    // [G] first padded row of each group
    const int32_t* ts;     // [G+1] first tile of each group
};

// Builds the tile tables in shared memory (all threads; ends with __syncthreads).
__device__ __forceinline__ SwTables sw_load_tables(const GemmArgs& a, int NB, int32_t* sm)
{
    const int Nmax = a.tile_n;
    const int G = a.G, cap = a.rb_cap * 128;
    int32_t* rows = sm;
    int32_t* ntt = rows + G;
    int32_t* off = ntt + G;
    int32_t* ts = off + G;
    int32_t* wsum = ts + G + 1;
    const int nthr = blockDim.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int per = (G + nthr - 1) / nthr;
    const int g0 = min(G, tid * per), g1 = min(G, g0 + per);
    int sum = 0;
    for (int g = g0; g < g1; ++g) {
        const int o = a.offsets[g];
        const int r = max(0, min(a.counts[g], cap - o));
        const int nt = r == 0 ? 0 : (r <= Nmax ? 1 : 1 + (r - Nmax + 127) / 128);
        rows[g] = r;
        ntt[g] = nt;
        off[g] = o;
        sum += nt * NB;
    }
    int v = sum;  // inclusive scan over the threads
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += t;
    }
    if (lane == 31) wsum[warp] = v;
    __syncthreads();
    if (warp == 0) {
        const int nw = nthr >> 5;
        int w = lane < nw ? wsum[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += t;
        }
        if (lane < nw) wsum[lane] = w;
    }
    __syncthreads();
    int pre = v - sum + (warp > 0 ? wsum[warp - 1] : 0);
    for (int g = g0; g < g1; ++g) {
        ts[g] = pre;
        pre += ntt[g] * NB;
    }
    if (tid == nthr - 1) ts[G] = pre;
    __syncthreads();
    SwTables tb;
    tb.rows = rows;
    tb.ntt = ntt;
    tb.off = off;
    tb.ts = ts;
    return tb;
}

inline int sw_table_bytes(int G) { return 4 * (4 * G + 1 + 32); }

// Tile t: the last group whose first tile is <= t (an empty group shares its first tile
// with the next one, so the last such group is the one that holds t).
__device__ __forceinline__ SwTile sw_decode(const SwTables& tb, int G, int t)
{
    int lo = 0, hi = G - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (tb.ts[mid] <= t) lo = mid;
        else hi = mid - 1;
    }
    const int nt = tb.ntt[lo];
    const int local = t - tb.ts[lo];
    const int nb = local / nt, j = local - nb * nt;
    SwTile ti;
    ti.g = lo;
    ti.nb = nb;
    ti.r0 = tb.off[lo] + 128 * j;
    ti.n = j == nt - 1 ? tb.rows[lo] - 128 * j : 128;
    return ti;
}

// Bytes one stage of tile ti receives: the weight blob, the token boxes (a 128-row box when
// the tile has >= 128 rows, then 16-row boxes), the token scale atoms (one or two row blocks).
__device__ __forceinline__ uint32_t sw_stage_tx(const SwTile& ti, int nk)
{
    const int nbig = ti.n >= 128 ? 1 : 0;
    const int nsmall = (ti.n - 128 * nbig + 15) >> 4;
    const int nrb = ti.n > 128 ? 2 : 1;
    return (uint32_t)kSwStageW + (uint32_t)(nbig * 16384 + nsmall * 2048) +
           (uint32_t)(nrb * 512 * nk);
}

// Lane 0 waits, sleeping sleep_ns between polls (the waiting warps leave the issue slots to
// the producer, MMA and working warps), and the warp follows.
__device__ __forceinline__ bool sw_warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                             uint32_t sleep_ns)
{
    int ok = 1;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait_lazy(bar, parity, abort, sleep_ns) ? 1 : 0;
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

}  // namespace

__global__ void __launch_bounds__(kSwThreads, 1)
    gemm_nvf4_swap_kernel(const __grid_constant__ CUtensorMap tmA,
                          const __grid_constant__ CUtensorMap tmA16,
                          const __grid_constant__ CUtensorMap tmY, GemmArgs args)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t su = smem_u32(smem_raw);
    uint8_t* stages = smem_raw + (((su + 1023u) & ~1023u) - su);
    const int NS = args.stages;
    const int Nmax = args.tile_n;
    const int SB = sw_stage_bytes(Nmax);
    const int kSwStageT = Nmax * 128;  // token codes of a stage
    const int NSL = sw_sf_slots(Nmax), SPR = NSL / 2;  // scale slots, per 256-column half
    const int SFS = sw_sfb_stride(Nmax), SLC = sw_slot_cols(Nmax);
    float* xpose = reinterpret_cast<float*>(stages + NS * SB);
    uint8_t* ctlb = stages + NS * SB + kSwXposeBytes;
    uint64_t* full = reinterpret_cast<uint64_t*>(ctlb);
    uint64_t* empty = full + kMaxStages;
    uint64_t* ready = empty + kMaxStages;  // a scale slot holds its stage's scales
    uint64_t* sfree = ready + kSwMaxSlots; // the MMAs that read a scale slot are done
    uint64_t* acc_full = sfree + kSwMaxSlots;
    uint64_t* acc_empty = acc_full + 2;
    uint64_t* drain = acc_empty + 2;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);
    int* zero = reinterpret_cast<int*>(tslot + 2);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int NB = args.N / 128;
    const int KB = (args.K + 255) / 256;
    const int G = args.G;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < NSL; ++b) {
            mbar_init(&ready[b], 4);  // one arrival per scale warp
            mbar_init(&sfree[b], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], kSwEpiWarps);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        *zero = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmA16);
    }
    if (warp == 1) {
        tmem_alloc(tslot, 512);
        tmem_relinquish();
    }
    const SwTables tb = sw_load_tables(args, NB, reinterpret_cast<int32_t*>(ctlb + kSwCtlBytes));
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const int ntiles = tb.ts[G];

    if (warp == 0) {
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_first(), pol_a = policy_evict_last();
            // the first NS stages' weights (constant) go out before the predecessor is done
            int i = 0;
            for (int t = blockIdx.x; t < ntiles && i < NS; t += gridDim.x) {
                const SwTile ti = sw_decode(tb, G, t);
                const uint8_t* wt =
                    args.b_tiles + ((size_t)ti.g * NB + ti.nb) * KB * (size_t)kNvf4TileBytes;
                for (int kb = 0; kb < KB && i < NS; ++kb, ++i) {
                    const int nk = min(4, (args.K - kb * 256) / 64);
                    mbar_arrive_expect_tx(&full[i], sw_stage_tx(ti, nk));
                    bulk_load(stages + i * SB, wt + (size_t)kb * kNvf4TileBytes,
                              kNvf4TileBytes, &full[i], pol_w);
                }
            }
            pdl_wait();
            pdl_trigger();
            int stage = 0;
            uint32_t phase = 0, issued = 0, issued_par = 0;
            bool ok = true;
            i = 0;
            for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
                const SwTile ti = sw_decode(tb, G, t);
                const int nbig = ti.n >= 128 ? 1 : 0;
                const int nsmall = (ti.n - 128 * nbig + 15) >> 4;
                const int nrb = ti.n > 128 ? 2 : 1;
                const uint8_t* wt =
                    args.b_tiles + ((size_t)ti.g * NB + ti.nb) * KB * (size_t)kNvf4TileBytes;
                const uint8_t* tsf = args.a_sf + (size_t)(ti.r0 >> 7) * (args.K / 64) * 512;
                for (int kb = 0; kb < KB; ++kb, ++i) {
                    const int nk = min(4, (args.K - kb * 256) / 64);
                    uint8_t* sW = stages + stage * SB;
                    uint8_t* sT = sW + kSwStageW;
                    uint8_t* sTSF = sT + kSwStageT;
                    if (i >= NS) {  // (the first NS stages were armed above)
                        if (!mbar_wait_lazy(&empty[stage], phase ^ 1u, abort_flag, 64)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(&full[stage], sw_stage_tx(ti, nk));
                        bulk_load(sW, wt + (size_t)kb * kNvf4TileBytes, kNvf4TileBytes,
                                  &full[stage], pol_w);
                    }
                    if (nbig) tma_load_2d(sT, &tmA, &full[stage], kb * 128, ti.r0, pol_a);
                    for (int b = 0; b < nsmall; ++b)
                        tma_load_2d(sT + nbig * 16384 + b * 2048, &tmA16, &full[stage], kb * 128,
                                    ti.r0 + 128 * nbig + 16 * b, pol_a);
                    for (int rb = 0; rb < nrb; ++rb)
                        bulk_load(sTSF + rb * 2048,
                                  tsf + (size_t)rb * (args.K / 64) * 512 + (size_t)kb * 2048,
                                  512u * nk, &full[stage], pol_a);
                    issued |= 1u << stage;
                    issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
                    if (++stage == NS) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                set_status(args.status, MOE_DEV_WAIT_TIMEOUT);
                *abort_flag = 1;
            }
            for (int s = 0; s < NS; ++s)  // copies in flight land before exit
                if ((issued >> s) & 1u) mbar_wait(&full[s], (issued_par >> s) & 1u, zero);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            int stage = 0, slot = 0, it = 0;
            uint32_t phase = 0, sphase = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x, ++it) {
                const SwTile ti = sw_decode(tb, G, t);
                const uint32_t idesc = idesc_nvf4(128, (ti.n + 15) & ~15);
                const int buf = it & 1;
                const uint32_t acc_par = (it >> 1) & 1;
                if (!mbar_wait(&acc_empty[buf], acc_par ^ 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_t = tmem + 256u * buf;
                for (int kb = 0; kb < KB; ++kb) {
                    // operands in smem and the stage's scales in the slot
                    if (!mbar_wait(&ready[slot], sphase, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const int nk = min(4, (args.K - kb * 256) / 64);
                    uint8_t* sW = stages + stage * SB;
                    uint8_t* sT = sW + kSwStageW;
                    const uint32_t sf_t =
                        tmem + (slot < SPR ? Nmax : 256 + Nmax) + (slot % SPR) * SLC;
                    const uint64_t ad = sdesc_sw128(smem_u32(sW)), bd = sdesc_sw128(smem_u32(sT));
                    for (int j = 0; j < nk; ++j)
                        tc_mma_nvf4(d_t, ad + 2 * j, bd + 2 * j, idesc, sf_t + 4 * j,
                                    sf_t + 16 + SFS * j, (kb | j) != 0);
                    tc_commit(&empty[stage]);
                    tc_commit(&sfree[slot]);
                    if (++stage == NS) {
                        stage = 0;
                        phase ^= 1u;
                    }
                    if (++slot == NSL) {
                        slot = 0;
                        sphase ^= 1u;
                    }
                }
                if (!ok) break;
                tc_commit(&acc_full[buf]);
            }
            if (!ok) {
                set_status(args.status, MOE_DEV_WAIT_TIMEOUT);
                *abort_flag = 1;
            }
            tc_commit(drain);  // every MMA issued above is complete after this
            mbar_wait(drain, 0, zero);
        }
        __syncwarp();
    } else if (warp >= 2 + kSwEpiWarps) {
        // scale warps (one per TMEM lane quarter), each writing the same slot contents into
        // its quarter: weight scales of rows 32c + lane (c < 4) and token scales of token
        // rows 32c + lane (c < 8; rows 128.. come from the second row block's atoms)
        const int q = warp & 3;
        int stage = 0, slot = 0;
        uint32_t phase = 0, sphase = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
            const SwTile ti = sw_decode(tb, G, t);
            const bool two = ti.n > 128;
            for (int kb = 0; kb < KB; ++kb) {
                if (!sw_warp_wait(&full[stage], phase, abort_flag, 32) ||
                    !sw_warp_wait(&sfree[slot], sphase ^ 1u, abort_flag, 32)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint8_t* sW = stages + stage * SB;
                const uint8_t* sWSF = sW + 16384;
                const uint8_t* sTSF = sW + kSwStageW + kSwStageT;
                uint32_t ra[16], rt[32];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint4 w = *reinterpret_cast<const uint4*>(sWSF + 512 * j + 16 * lane);
                    const uint4 a = *reinterpret_cast<const uint4*>(sTSF + 512 * j + 16 * lane);
                    const uint4 b = two ? *reinterpret_cast<const uint4*>(sTSF + 2048 + 512 * j +
                                                                         16 * lane)
                                        : make_uint4(0u, 0u, 0u, 0u);
                    ra[4 * j] = w.x;
                    ra[4 * j + 1] = w.y;
                    ra[4 * j + 2] = w.z;
                    ra[4 * j + 3] = w.w;
                    rt[8 * j] = a.x;
                    rt[8 * j + 1] = a.y;
                    rt[8 * j + 2] = a.z;
                    rt[8 * j + 3] = a.w;
                    rt[8 * j + 4] = b.x;
                    rt[8 * j + 5] = b.y;
                    rt[8 * j + 6] = b.z;
                    rt[8 * j + 7] = b.w;
                }
                const uint32_t base = tmem + ((uint32_t)(q * 32) << 16) +
                                      (slot < SPR ? Nmax : 256 + Nmax) + (slot % SPR) * SLC;
                tmem_st16(base, ra);
                if (SFS == 4) {  // token rows < 128: one row block, columns 4 j + c
                    uint32_t r4[16];
#pragma unroll
                    for (int j = 0; j < 4; ++j)
#pragma unroll
                        for (int c = 0; c < 4; ++c) r4[4 * j + c] = rt[8 * j + c];
                    tmem_st16(base + 16, r4);
                } else {
                    tmem_st32(base + 16, rt);
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&ready[slot]);
                if (++stage == NS) {
                    stage = 0;
                    phase ^= 1u;
                }
                if (++slot == NSL) {
                    slot = 0;
                    sphase ^= 1u;
                }
            }
        }
        if (!ok && lane == 0) {
            set_status(args.status, MOE_DEV_WAIT_TIMEOUT);
            *abort_flag = 1;
        }
    } else {
        // epilogue: quarter q of the weight rows, chunks h, h + 2, ... of 32 token columns
        const int q = warp & 3, h = (warp - 2) >> 2;  // (h < kSwHalves)
        const int ep = args.epilogue;
        const bool down = is_down(ep);
        const bool up_lane = lane >= 16;
        const int I = args.N / 2;  // gate_up: intermediate features
        float* xt = xpose + (warp - 2) * 32 * kSwXposeStride;
        float smax = 0.0f;         // kEpiGateUpSwigluF32: this lane's amax |s|
        int it = 0;
        pdl_wait();
        for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++it) {
            const SwTile ti = sw_decode(tb, G, t);
            const int nch = (ti.n + 31) >> 5;
            const float gw = args.gs_w[ti.g];
            const float gs_in = !down ? *args.gs_a : args.gs_i_dev ? *args.gs_i_dev : args.gs_i;
            const float alpha0 = __frcp_rn(__fmul_rn(gs_in, gw));
            float ys = 1.0f, yinv = 1.0f;
            if (ep == kEpiDownF16) {
                // 2^e_g: the largest power of two with K x 2688^2 x alpha_g x 2^e_g <= 65504
                const float tq = __fdiv_rd(
                    kYF16Max, __fmul_ru(__fmul_ru((float)args.K, kE2M1E4M3MaxSq), alpha0));
                const int ex =
                    max(-126, min(126, (int)((__float_as_uint(tq) >> 23) & 0xFFu) - 127));
                ys = __uint_as_float((uint32_t)(127 + ex) << 23);
                yinv = __uint_as_float((uint32_t)(127 - ex) << 23);
            }
            // per-column alpha of each of this warp's chunks (column 32 ch + lane)
            float av[kSwChunks];
#pragma unroll
            for (int c = 0; c < kSwChunks; ++c) {
                const int ch = h + kSwHalves * c, col = 32 * ch + lane;
                av[c] = alpha0;
                if (down && ch < nch && col < ti.n) {
                    const int pair = args.perm_src[ti.r0 + col];
                    const float wgt = !pair_ok(pair, args.status) ? 0.0f
                                      : pair < args.Tk          ? args.topk_w[pair]
                                                                : 1.0f;
                    av[c] = __fmul_rn(__fmul_rn(alpha0, wgt), ys);
                    if (ep == kEpiDownF16 && ti.nb == 0 && q == 0)
                        args.y_scale[ti.r0 + col] = yinv;  // one writer per row
                }
            }
            const int buf = it & 1;
            const uint32_t acc_par = (it >> 1) & 1;
            if (!sw_warp_wait(&acc_full[buf], acc_par, abort_flag, 256)) {
                if (lane == 0) {
                    set_status(args.status, MOE_DEV_WAIT_TIMEOUT);
                    *abort_flag = 1;
                }
                break;
            }
            tc_fence_after();
#pragma unroll
            for (int c = 0; c < kSwChunks; ++c) {
                const int ch = h + kSwHalves * c;
                if (ch >= nch) break;
                uint32_t r[32];
                tmem_ld32(tmem + 256u * buf + ((uint32_t)(q * 32) << 16) + 32 * ch, r);
                tmem_ld_wait();
                const int ncol = min(32, ti.n - 32 * ch);
                const int64_t row0 = (int64_t)ti.r0 + 32 * ch;
                if (down) {
                    const int64_t f = 128 * ti.nb + 32 * q + lane;  // output feature
                    if (ep == kEpiDownF16) {
                        // the 32 token rows x 32 features as a fp16 box in the warp's staging
                        // slice (64-byte rows, 64-byte swizzle: 16-byte piece c of row i at
                        // c ^ ((i >> 1) & 3)), written by one TMA tensor store; rows past the
                        // tile's tokens are padding rows of the group (never read)
                        uint8_t* stg = reinterpret_cast<uint8_t*>(xt);
                        if (lane == 0) bulk_wait_read0();  // the previous box has been read
                        __syncwarp();
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const float a = __shfl_sync(0xffffffffu, av[c], i);
                            *reinterpret_cast<__half*>(
                                stg + i * 64 + ((((lane >> 3) ^ ((i >> 1) & 3))) << 4) +
                                (lane & 7) * 2) = __float2half_rn(__uint_as_float(r[i]) * a);
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            tma_store_2d(&tmY, stg, 128 * ti.nb + 32 * q, ti.r0 + 32 * ch);
                            bulk_commit();
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const float a = __shfl_sync(0xffffffffu, av[c], i);
                            if (i < ncol)
                                args.out_f32[(row0 + i) * args.N + f] = __uint_as_float(r[i]) * a;
                        }
                    }
                    continue;
                }
                // gate_up: lanes 0..15 gate features f0 + lane, lanes 16..31 up f0 + lane - 16
                const int f0 = 64 * ti.nb + 16 * q;
                if (ep == kEpiGateUpF32) {
                    const int fl = f0 + (lane & 15);
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (i < ncol)
                            args.out_f32[(row0 + i) * args.N + (up_lane ? I : 0) + fl] =
                                __uint_as_float(r[i]) * alpha0;
                    continue;
                }
                // s = silu(gate) * up, two token columns at a time (gate lanes take column i,
                // their gate and the up of lane + 16; up lanes column i + 1, the gate of
                // lane - 16 and their up), into the warp's [column][feature] tile in shared
                // memory; then lane l holds token column l's 16 features and quantises them
                // as one NVFP4 block in registers
#pragma unroll
                for (int i = 0; i < 32; i += 2) {
                    const float send = __uint_as_float(up_lane ? r[i] : r[i + 1]);
                    const float recv = __shfl_xor_sync(0xffffffffu, send, 16);
                    const float g = up_lane ? recv : __uint_as_float(r[i]);
                    const float u = up_lane ? __uint_as_float(r[i + 1]) : recv;
                    xt[(i + (up_lane ? 1 : 0)) * kSwXposeStride + (lane & 15)] =
                        silu_mul(__fmul_rn(g, alpha0), __fmul_rn(u, alpha0));
                }
                __syncwarp();
                if (lane < ncol) {
                    float v[16];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float4 q4 =
                            *reinterpret_cast<const float4*>(xt + lane * kSwXposeStride + 4 * j);
                        v[4 * j] = q4.x;
                        v[4 * j + 1] = q4.y;
                        v[4 * j + 2] = q4.z;
                        v[4 * j + 3] = q4.w;
                    }
                    const int64_t prow = row0 + lane;
                    if (ep == kEpiGateUpSwigluF32) {
                        float4* dst = reinterpret_cast<float4*>(args.out_f32 + prow * I + f0);
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            dst[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                            smax = fmaxf(smax, fmaxf(fmaxf(fabsf(v[4 * j]), fabsf(v[4 * j + 1])),
                                                     fmaxf(fabsf(v[4 * j + 2]), fabsf(v[4 * j + 3]))));
                        }
                    } else {
                        uint32_t cw[2];
                        const uint32_t sb = quant16(v, args.gs_i, cw);
                        *reinterpret_cast<uint2*>(args.out_codes + prow * codes_pitch(I) + f0 / 2) =
                            make_uint2(cw[0], cw[1]);
                        args.out_sf[sf_atom_offset(prow, 4 * ti.nb + q, I)] = (uint8_t)sb;
                    }
                }
                __syncwarp();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[buf]);
        }
        if (lane == 0) bulk_wait_all();  // staged stores complete before the CTA exits
        if (ep == kEpiGateUpSwigluF32) {
            // one atomic per warp; |s| >= 0, so its fp32 bits order like the values
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
                smax = fmaxf(smax, __shfl_xor_sync(0xffffffffu, smax, o));
            if (lane == 0) atomicMax(args.inter_amax, __float_as_uint(smax));
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

int gemm_swap_smem_bytes(int stages, int tile_n, int G)
{
    return 1024 + stages * sw_stage_bytes(tile_n) + kSwXposeBytes + kSwCtlBytes +
           sw_table_bytes(G);
}

}  // namespace moe
