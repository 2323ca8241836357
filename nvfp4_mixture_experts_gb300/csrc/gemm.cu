// NVFP4 x NVFP4 (W4A4) grouped GEMMs of the expert MLPs on the 5th-generation tensor cores
// (tcgen05).  The W4A16 GEMMs are in gemm_w4a16.cu.
//
// Rows (M) are the padded rows of one expert group (tokens routed to that expert); columns
// (N) are 128 rows of that expert's weight matrix; the accumulator lives in TMEM.  One
// persistent CTA per SM walks the tile list (group, weight tile, row block), with
// consecutive tiles sharing the same weight tile so the second row block of an expert
// reads the weights from L2.
//
// Weights are re-laid out at create time as one contiguous blob per (expert, 128-row
// tile, k-stage): the codes exactly as the MMA reads them from shared memory, followed by
// their scale atoms, so each stage's weights arrive with one sequential bulk copy.
//
// Warp roles (warp-specialised pipeline):
//   warp 0   TMA producer: activation tile (tensor map), weight blob, activation scales
//   warp 1   TMEM allocation; one thread issues tcgen05.mma
//   warps 2-5 epilogue: TMEM -> registers -> fused output (one TMEM lane quarter each)
//   warps 6-9 the stage's scale factors smem -> TMEM with tcgen05.st (keeping the copies
//            out of the MMA thread's in-order tcgen05 queue, where they serialised with
//            the MMAs)
//
// kind::mxf4nvf4 block-scaled MMA, K = 64 per instruction, UE4M3 scales per 16 elements.
// The global scales are applied in the epilogue as alpha = 1 / (gs_a * gs_w).
//
// Every pipeline wait is bounded: a wait that runs out sets MOE_DEV_WAIT_TIMEOUT in the
// status word and makes all roles stop, drain their copies in flight, free TMEM and exit.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kernels.cuh"

namespace moe {

struct TileInfo {
    int g;       // group (local expert, or the shared slot)
    int nb;      // 128-row weight tile within the expert
    int rows;    // valid rows of this row block (1..128)
    int arow0;   // first padded row of the row block
    int brow0;   // first weight row (slot * N + 128 * nb)
};

// Group tables staged in shared memory at kernel start (the tile decode runs once per tile
// on the producer's critical path; global-memory latency there would stall the stream).
struct Tables {
    const int32_t* mb_start;  // [G+1]
    const int32_t* counts;    // [G]
    const int32_t* offsets;   // [G+1]
    const int32_t* rb_group;  // [rb_cap] group of each 128-row block
};

// Tile t of the list: groups in order; inside a group, weight tiles in order; inside a
// weight tile, the group's row blocks (so row blocks sharing weights run back to back).
// Group g owns tiles [mb_start[g] * NB, mb_start[g+1] * NB), so t / NB is one of its row
// blocks and the row-block table gives g directly.
__device__ __forceinline__ TileInfo decode_tile(const GemmArgs& a, const Tables& tb, int NB,
                                                int t)
{
    const int g = tb.rb_group[t / NB];
    const int nmb = tb.mb_start[g + 1] - tb.mb_start[g];
    const int local = t - tb.mb_start[g] * NB;
    const int nb = nmb == 1 ? local : local / nmb, mb = nmb == 1 ? 0 : local % nmb;
    TileInfo ti;
    ti.g = g;
    ti.nb = nb;
    ti.rows = min(128, tb.counts[g] - 128 * mb);
    ti.arow0 = tb.offsets[g] + 128 * mb;
    ti.brow0 = g * a.N + 128 * nb;
    return ti;
}

// Copies the group tables into shared memory (all threads; a __syncthreads follows).
__device__ __forceinline__ Tables load_tables(const GemmArgs& a, int32_t* smem)
{
    Tables tb;
    int32_t* m = smem;
    int32_t* c = m + (a.G + 1);
    int32_t* o = c + a.G;
    int32_t* r = o + (a.G + 1);
    for (int i = threadIdx.x; i <= a.G; i += blockDim.x) {
        const int m0 = a.mb_start[i];
        m[i] = m0;
        o[i] = a.offsets[i];
        if (i < a.G) {
            c[i] = a.counts[i];
            const int m1 = min(a.mb_start[i + 1], a.rb_cap);
            for (int b = max(m0, 0); b < m1; ++b) r[b] = i;
        }
    }
    tb.mb_start = m;
    tb.counts = c;
    tb.offsets = o;
    tb.rb_group = r;
    return tb;
}

// Lane 0 waits, the warp follows (keeps .sync.aligned tcgen05 ops converged).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort)
{
    int ok = 1;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, abort) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    return ok != 0;
}

// Per-row epilogue constants of one tile (global loads, issued before the accumulator
// wait so their latency overlaps the tile's mainloop).
// Eight fp32 accumulator words times alpha -> eight fp16 (round to nearest even).
__device__ __forceinline__ uint4 f32x8_to_f16x8(const uint32_t* r, float alpha)
{
    uint32_t h[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __half2 v = __floats2half2_rn(__uint_as_float(r[2 * i]) * alpha,
                                            __uint_as_float(r[2 * i + 1]) * alpha);
        h[i] = *reinterpret_cast<const uint32_t*>(&v);
    }
    return make_uint4(h[0], h[1], h[2], h[3]);
}

struct EpiPrep {
    int64_t prow;   // padded row of this thread
    float alpha;    // 1 / (global scales) (x routing weight for the down epilogues; x 2^e_g
                    // for kEpiDownF16)
    float yinv;     // kEpiDownF16: 2^-e_g
    int nvalid;     // valid rows in this warp's 32-row quarter (0..32)
    bool valid;
};

__device__ __forceinline__ EpiPrep epi_prep(const GemmArgs& a, const TileInfo& ti, int q,
                                            int lane)
{
    EpiPrep e;
    const int m = q * 32 + lane;
    e.valid = m < ti.rows;
    e.prow = (int64_t)ti.arow0 + m;
    const float gw = a.gs_w[ti.g];
    const float gs_in = !is_down(a.epilogue) ? *a.gs_a : a.gs_i_dev ? *a.gs_i_dev : a.gs_i;
    e.alpha = __frcp_rn(__fmul_rn(gs_in, gw));
    e.nvalid = max(0, min(32, ti.rows - q * 32));
    e.yinv = 1.0f;
    float ys = 1.0f;
    if (a.epilogue == kEpiDownF16) {
        // 2^e_g: the largest power of two with K x 2688^2 x alpha_g x 2^e_g <= 65504
        // (the bound rounded up, the quotient rounded down: 2^e_g never exceeds the exact one)
        const float t = __fdiv_rd(kYF16Max,
                                  __fmul_ru(__fmul_ru((float)a.K, kE2M1E4M3MaxSq), e.alpha));
        const int ex = max(-126, min(126, (int)((__float_as_uint(t) >> 23) & 0xFFu) - 127));
        ys = __uint_as_float((uint32_t)(127 + ex) << 23);
        e.yinv = __uint_as_float((uint32_t)(127 - ex) << 23);
    }
    if (is_down(a.epilogue) && e.valid) {
        const int pair = a.perm_src[e.prow];
        const float wgt = !pair_ok(pair, a.status) ? 0.0f : pair < a.Tk ? a.topk_w[pair] : 1.0f;
        e.alpha = __fmul_rn(__fmul_rn(e.alpha, wgt), ys);
    }
    return e;
}

// Epilogue of one tile for the 32 rows of TMEM lane quarter q (thread = row).  A warp
// whose quarter has no valid row does nothing.  The down epilogues with more than 8 valid
// rows stage each 32 x 32 chunk in shared memory (fp32: 128-byte swizzle; fp16: 64-byte
// swizzle; two buffers per warp) and write it with a TMA tensor store; sparse quarters store
// directly.
__device__ __forceinline__ void run_epilogue(const GemmArgs& a, const TileInfo& ti,
                                             const EpiPrep& ep, uint32_t tacc, int q, int lane,
                                             const CUtensorMap* tmY, uint8_t* stg, int& pp,
                                             int stg_stride = 4096)
{
    if (ep.nvalid == 0) return;
    const bool valid = ep.valid;
    const int64_t prow = ep.prow;
    const float alpha = ep.alpha;
    const bool staged = is_down(a.epilogue) && a.staging && ep.nvalid > 8;
    const bool f16 = a.epilogue == kEpiDownF16;
    if (f16 && ti.nb == 0 && valid) a.y_scale[prow] = ep.yinv;  // one writer per row
    const int I = a.N / 2;
    uint32_t sfword = 0;
    float smax = 0.0f;  // kEpiGateUpSwigluF32: this lane's amax |s|
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        tmem_ld32(tacc + ((uint32_t)(q * 32) << 16) + 32 * c, r);
        tmem_ld_wait();
        if (staged) {
            uint8_t* buf = stg + pp * stg_stride;
            if (lane == 0) bulk_wait_read1();  // this buffer's previous store has read it
            __syncwarp();
            if (f16) {  // row lane: 64 bytes, 16-byte piece i at i ^ ((lane >> 1) & 3)
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    *reinterpret_cast<uint4*>(buf + lane * 64 + ((i ^ ((lane >> 1) & 3)) << 4)) =
                        f32x8_to_f16x8(r + 8 * i, alpha);
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    *reinterpret_cast<float4*>(buf + lane * 128 + ((i ^ (lane & 7)) << 4)) =
                        make_float4(__uint_as_float(r[4 * i]) * alpha,
                                    __uint_as_float(r[4 * i + 1]) * alpha,
                                    __uint_as_float(r[4 * i + 2]) * alpha,
                                    __uint_as_float(r[4 * i + 3]) * alpha);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                tma_store_2d(tmY, buf, 128 * ti.nb + 32 * c, ti.arow0 + 32 * q);
                bulk_commit();
            }
            pp ^= 1;
            continue;
        }
        if (!valid) continue;
        if (f16) {
            uint4* dst = reinterpret_cast<uint4*>(a.out_bf16 + prow * a.N + 128 * ti.nb + 32 * c);
#pragma unroll
            for (int i = 0; i < 4; ++i) dst[i] = f32x8_to_f16x8(r + 8 * i, alpha);
        } else if (a.epilogue == kEpiDown) {
            float4* dst = reinterpret_cast<float4*>(a.out_f32 + prow * a.N + 128 * ti.nb + 32 * c);
#pragma unroll
            for (int i = 0; i < 8; ++i)
                dst[i] = make_float4(__uint_as_float(r[4 * i]) * alpha,
                                     __uint_as_float(r[4 * i + 1]) * alpha,
                                     __uint_as_float(r[4 * i + 2]) * alpha,
                                     __uint_as_float(r[4 * i + 3]) * alpha);
        } else if (a.epilogue == kEpiGateUpF32) {
            const int f = 64 * ti.nb + 16 * c;
            float4* dg = reinterpret_cast<float4*>(a.out_f32 + prow * a.N + f);
            float4* du = reinterpret_cast<float4*>(a.out_f32 + prow * a.N + I + f);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                dg[i] = make_float4(__uint_as_float(r[4 * i]) * alpha,
                                    __uint_as_float(r[4 * i + 1]) * alpha,
                                    __uint_as_float(r[4 * i + 2]) * alpha,
                                    __uint_as_float(r[4 * i + 3]) * alpha);
                du[i] = make_float4(__uint_as_float(r[16 + 4 * i]) * alpha,
                                    __uint_as_float(r[16 + 4 * i + 1]) * alpha,
                                    __uint_as_float(r[16 + 4 * i + 2]) * alpha,
                                    __uint_as_float(r[16 + 4 * i + 3]) * alpha);
            }
        } else {
            const int f = 64 * ti.nb + 16 * c;
            float s[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
                s[i] = silu_mul(__fmul_rn(__uint_as_float(r[i]), alpha),
                                __fmul_rn(__uint_as_float(r[16 + i]), alpha));
            if (a.epilogue == kEpiGateUpSwigluF32) {
                float4* dst = reinterpret_cast<float4*>(a.out_f32 + prow * I + f);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    dst[i] = make_float4(s[4 * i], s[4 * i + 1], s[4 * i + 2], s[4 * i + 3]);
                    smax = fmaxf(smax, fmaxf(fmaxf(fabsf(s[4 * i]), fabsf(s[4 * i + 1])),
                                             fmaxf(fabsf(s[4 * i + 2]), fabsf(s[4 * i + 3]))));
                }
                continue;
            }
            uint32_t cw[2];
            const uint32_t sb = quant16(s, a.gs_i, cw);
            *reinterpret_cast<uint2*>(a.out_codes + prow * codes_pitch(I) + f / 2) =
                make_uint2(cw[0], cw[1]);
            sfword |= sb << (8 * c);
        }
    }
    if (a.epilogue == kEpiGateUpSwiglu && valid)
        *reinterpret_cast<uint32_t*>(a.out_sf + sf_atom_offset(prow, 4 * ti.nb, I)) = sfword;
    if (a.epilogue == kEpiGateUpSwigluF32) {
        // one atomic per warp; |s| >= 0, so its fp32 bits order like the values
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) smax = fmaxf(smax, __shfl_xor_sync(0xffffffffu, smax, o));
        if (lane == 0) atomicMax(a.inter_amax, __float_as_uint(smax));
    }
}

// Shared-memory carve-up: stages, then barriers (room for kMaxStages), the TMEM address
// slot and flags, then the group tables.
struct Ctl {
    uint64_t* full;
    uint64_t* empty;
    uint64_t* ready;       // the stage's scale factors are in TMEM
    uint64_t* acc_full;
    uint64_t* acc_empty;
    uint64_t* drain;
    uint32_t* tmem_slot;
    volatile int* abort_flag;
    int* zero;
};

__device__ __forceinline__ Ctl carve(uint8_t* base, int stages)
{
    Ctl c;
    uint64_t* b = reinterpret_cast<uint64_t*>(base);
    c.full = b;
    c.empty = b + stages;
    c.ready = b + 2 * stages;
    c.acc_full = b + 3 * stages;
    c.acc_empty = c.acc_full + 2;
    c.drain = c.acc_empty + 2;
    c.tmem_slot = reinterpret_cast<uint32_t*>(c.drain + 1);
    c.abort_flag = reinterpret_cast<volatile int*>(c.tmem_slot + 1);
    c.zero = reinterpret_cast<int*>(c.tmem_slot + 2);
    return c;
}

__device__ __forceinline__ int32_t* tables_smem(uint8_t* ctl_base)
{
    return reinterpret_cast<int32_t*>(ctl_base + kCtlBytes);
}

__device__ __forceinline__ uint8_t* aligned_smem(uint8_t* raw)
{
    const uint32_t u = smem_u32(raw);
    return raw + (((u + 1023u) & ~1023u) - u);
}

// ============================================================== W4A4: NVFP4 x NVFP4

__global__ void __launch_bounds__(kNvf4Threads, 1)
    gemm_nvf4_kernel(const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ CUtensorMap tmA16,
                     const __grid_constant__ CUtensorMap tmY, GemmArgs args)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* stages = aligned_smem(smem_raw);
    const int NS = args.stages;
    uint8_t* staging = stages + NS * kNvf4StageBytes;  // epilogue staging (down epilogues)
    Ctl ctl = carve(staging + args.staging, kMaxStages);
    const Tables tb = load_tables(args, tables_smem(staging + args.staging));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int NB = args.N / 128;
    const int KB = (args.K + 255) / 256;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&ctl.full[s], 1);
            mbar_init(&ctl.empty[s], 1);
            mbar_init(&ctl.ready[s], 4);  // one arrival per scale warp
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&ctl.acc_full[b], 1);
            mbar_init(&ctl.acc_empty[b], 128);
        }
        mbar_init(ctl.drain, 1);
        *ctl.abort_flag = 0;
        *ctl.zero = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmA16);
    }
    if (warp == 1) {
        tmem_alloc(ctl.tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *ctl.tmem_slot;
    // (row blocks beyond the capacity were flagged by the grouping and are not run)
    const int ntiles = min(tb.mb_start[args.G], args.rb_cap) * NB;

    if (warp == 0) {
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_first(), pol_a = policy_evict_last();
            // the first NS stages' weights (constant) go out before the predecessor is done
            int i = 0;
            for (int t = blockIdx.x; t < ntiles && i < NS; t += gridDim.x) {
                const TileInfo ti = decode_tile(args, tb, NB, t);
                const int nbox = (ti.rows + 15) >> 4;
                const uint32_t a_bytes = nbox > 4 ? 16384u : (uint32_t)nbox * 2048u;
                const uint8_t* wt = args.b_tiles +
                                    ((size_t)ti.g * NB + ti.nb) * KB * (size_t)kNvf4TileBytes;
                for (int kb = 0; kb < KB && i < NS; ++kb, ++i) {
                    const int nk = min(4, (args.K - kb * 256) / 64);
                    mbar_arrive_expect_tx(&ctl.full[i],
                                          a_bytes + (uint32_t)kNvf4TileBytes + 512u * nk);
                    bulk_load(stages + i * kNvf4StageBytes + 16384,
                              wt + (size_t)kb * kNvf4TileBytes, kNvf4TileBytes, &ctl.full[i],
                              pol_w);
                }
            }
            pdl_wait();
            pdl_trigger();
            int stage = 0;
            uint32_t phase = 0, issued = 0, issued_par = 0;
            bool ok = true;
            i = 0;
            for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
                const TileInfo ti = decode_tile(args, tb, NB, t);
                const int nbox = (ti.rows + 15) >> 4;
                const bool big = nbox > 4;
                const uint32_t a_bytes = big ? 16384u : (uint32_t)nbox * 2048u;
                const uint8_t* sfa = args.a_sf + (size_t)(ti.arow0 >> 7) * (args.K / 64) * 512;
                // this weight tile's k-stages: contiguous blobs of codes (SMEM image) + scales
                const uint8_t* wt = args.b_tiles +
                                    ((size_t)ti.g * NB + ti.nb) * KB * (size_t)kNvf4TileBytes;
                for (int kb = 0; kb < KB; ++kb, ++i) {
                    const int nk = min(4, (args.K - kb * 256) / 64);
                    uint8_t* sA = stages + stage * kNvf4StageBytes;
                    uint8_t* sB = sA + 16384;    // weight codes, then their scales (contiguous)
                    uint8_t* sSFA = sB + kNvf4TileBytes;
                    if (i >= NS) {  // (the first NS stages were armed above)
                        if (!mbar_wait(&ctl.empty[stage], phase ^ 1u, ctl.abort_flag)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(&ctl.full[stage],
                                              a_bytes + (uint32_t)kNvf4TileBytes + 512u * nk);
                        bulk_load(sB, wt + (size_t)kb * kNvf4TileBytes, kNvf4TileBytes,
                                  &ctl.full[stage], pol_w);
                    }
                    if (big) {
                        tma_load_2d(sA, &tmA, &ctl.full[stage], kb * 128, ti.arow0, pol_a);
                    } else {
                        for (int b = 0; b < nbox; ++b)
                            tma_load_2d(sA + b * 2048, &tmA16, &ctl.full[stage], kb * 128,
                                        ti.arow0 + 16 * b, pol_a);
                    }
                    bulk_load(sSFA, sfa + kb * 2048, 512u * nk, &ctl.full[stage], pol_a);
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
                *ctl.abort_flag = 1;
            }
            for (int s = 0; s < NS; ++s)  // copies in flight land before exit
                if ((issued >> s) & 1u) mbar_wait(&ctl.full[s], (issued_par >> s) & 1u, ctl.zero);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_nvf4(128, 128);
            int stage = 0, it = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x, ++it) {
                const int buf = it & 1;
                const uint32_t acc_par = (it >> 1) & 1;
                if (!mbar_wait(&ctl.acc_empty[buf], acc_par ^ 1u, ctl.abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_t = tmem + buf * 128;
                for (int kb = 0; kb < KB; ++kb) {
                    // operands in smem and the stage's scales in TMEM
                    if (!mbar_wait(&ctl.ready[stage], phase, ctl.abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const int nk = min(4, (args.K - kb * 256) / 64);
                    uint8_t* sA = stages + stage * kNvf4StageBytes;
                    uint8_t* sB = sA + 16384;
                    const uint32_t sfa_t = tmem + 256 + stage * 32, sfb_t = sfa_t + 16;
                    const uint64_t ad = sdesc_sw128(smem_u32(sA)), bd = sdesc_sw128(smem_u32(sB));
                    for (int j = 0; j < nk; ++j)
                        tc_mma_nvf4(d_t, ad + 2 * j, bd + 2 * j, idesc, sfa_t + 4 * j,
                                    sfb_t + 4 * j, (kb | j) != 0);
                    tc_commit(&ctl.empty[stage]);
                    if (++stage == NS) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                tc_commit(&ctl.acc_full[buf]);
            }
            if (!ok) {
                set_status(args.status, MOE_DEV_WAIT_TIMEOUT);
                *ctl.abort_flag = 1;
            }
            tc_commit(ctl.drain);  // every MMA / copy issued above is complete after this
            mbar_wait(ctl.drain, 0, ctl.zero);
        }
        __syncwarp();
    } else if (warp >= 6) {
        // scale warps (one per TMEM lane quarter): each stage's activation and weight scale
        // atoms, smem -> registers -> TMEM columns 256 + 32*stage (the layout tc_cp_sf
        // describes: lane l, column c of a k-step = the 4 scales of row 32c + l)
        const int q = warp & 3;
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
            for (int kb = 0; kb < KB; ++kb) {
                if (!warp_wait(&ctl.full[stage], phase, ctl.abort_flag)) {
                    ok = false;
                    break;
                }
                const uint8_t* sB = stages + stage * kNvf4StageBytes + 16384;
                const uint8_t* sSFB = sB + 16384;
                const uint8_t* sSFA = sB + kNvf4TileBytes;
                uint32_t r[32];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint4 a = *reinterpret_cast<const uint4*>(sSFA + 512 * j + 16 * lane);
                    const uint4 b = *reinterpret_cast<const uint4*>(sSFB + 512 * j + 16 * lane);
                    r[4 * j] = a.x;
                    r[4 * j + 1] = a.y;
                    r[4 * j + 2] = a.z;
                    r[4 * j + 3] = a.w;
                    r[16 + 4 * j] = b.x;
                    r[16 + 4 * j + 1] = b.y;
                    r[16 + 4 * j + 2] = b.z;
                    r[16 + 4 * j + 3] = b.w;
                }
                tmem_st32(tmem + ((uint32_t)(q * 32) << 16) + 256 + stage * 32, r);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctl.ready[stage]);
                if (++stage == NS) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        if (!ok && lane == 0) {
            set_status(args.status, MOE_DEV_WAIT_TIMEOUT);
            *ctl.abort_flag = 1;
        }
    } else {
        const int q = warp & 3;
        int it = 0, pp = 0;
        pdl_wait();
        for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++it) {
            const TileInfo ti = decode_tile(args, tb, NB, t);
            const EpiPrep ep = epi_prep(args, ti, q, lane);
            const int buf = it & 1;
            const uint32_t acc_par = (it >> 1) & 1;
            if (!warp_wait(&ctl.acc_full[buf], acc_par, ctl.abort_flag)) {
                if (lane == 0) {
                    set_status(args.status, MOE_DEV_WAIT_TIMEOUT);
                    *ctl.abort_flag = 1;
                }
                break;
            }
            tc_fence_after();
            run_epilogue(args, ti, ep, tmem + buf * 128, q, lane, &tmY,
                             staging + (warp - 2) * 8192, pp);
            tc_fence_before();
            mbar_arrive(&ctl.acc_empty[buf]);
        }
        if (lane == 0) bulk_wait_all();  // staged stores complete before the CTA exits
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ============================================================== W4A4 with 256-column tiles
//
// The row-block kernel with each MMA covering two weight tiles (N = 256): measured in the
// row-block kernel, a block-scaled MMA holds its issuing thread about as long at N = 256 as at
// N = 128, so twice the columns per instruction halve the main loop's time per FLOP.  Two
// 256-column accumulators would fill TMEM, so there is one, beside the stage scale slots
// (256 + 48 s: the activation scales, 4 columns per k-step, then the 256 weight rows' scales,
// 8 columns per k-step); eight epilogue warps (two per TMEM lane quarter, one per weight tile)
// drain it while the producer and the scale warps fill the next tile's stages.  A stage holds
// the activation tile, the two weight tiles' codes back to back (the B operand's 256 rows),
// their scales, and the activation scales.  Tiles: groups in order; inside a group, pairs of
// weight tiles in order; inside those, the group's row blocks.
//   warp 0 producer, warp 1 TMEM + MMA, warps 2..9 epilogue, warps 10..13 scale warps

__device__ __forceinline__ TileInfo decode_wide_tile(const GemmArgs& a, const Tables& tb, int NB2,
                                                     int t)
{
    const int g = tb.rb_group[t / NB2];
    const int nmb = tb.mb_start[g + 1] - tb.mb_start[g];
    const int local = t - tb.mb_start[g] * NB2;
    const int nb2 = nmb == 1 ? local : local / nmb, mb = nmb == 1 ? 0 : local % nmb;
    TileInfo ti;
    ti.g = g;
    ti.nb = 2 * nb2;  // the first of the two weight tiles
    ti.rows = min(128, tb.counts[g] - 128 * mb);
    ti.arow0 = tb.offsets[g] + 128 * mb;
    ti.brow0 = g * a.N + 128 * ti.nb;
    return ti;
}

__global__ void __launch_bounds__(kWideThreads, 1)
    gemm_nvf4_wide_kernel(const __grid_constant__ CUtensorMap tmA,
                          const __grid_constant__ CUtensorMap tmA16,
                          const __grid_constant__ CUtensorMap tmY, GemmArgs args)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* stages = aligned_smem(smem_raw);
    const int NS = args.stages;
    uint8_t* staging = stages + NS * kWideStageBytes;  // epilogue staging (fp16 down)
    Ctl ctl = carve(staging + args.staging, kMaxStages);
    const Tables tb = load_tables(args, tables_smem(staging + args.staging));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int NB = args.N / 128, NB2 = NB / 2;
    const int KB = (args.K + 255) / 256;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&ctl.full[s], 1);
            mbar_init(&ctl.empty[s], 1);
            mbar_init(&ctl.ready[s], 4);  // one arrival per scale warp
        }
        mbar_init(&ctl.acc_full[0], 1);
        mbar_init(&ctl.acc_empty[0], 8);  // one arrival per epilogue warp
        mbar_init(ctl.drain, 1);
        *ctl.abort_flag = 0;
        *ctl.zero = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmA16);
    }
    if (warp == 1) {
        tmem_alloc(ctl.tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *ctl.tmem_slot;
    const int ntiles = min(tb.mb_start[args.G], args.rb_cap) * NB2;

    if (warp == 0) {
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_first(), pol_a = policy_evict_last();
            // the two weight tiles' k-stage blobs: codes back to back, then their scales
            auto weights = [&](const TileInfo& ti, int kb, uint8_t* sB, uint64_t* bar) {
                const uint8_t* b0 = args.b_tiles +
                                    (((size_t)ti.g * NB + ti.nb) * KB + kb) * (size_t)kNvf4TileBytes;
                const uint8_t* b1 = b0 + (size_t)KB * kNvf4TileBytes;
                bulk_load(sB, b0, 16384u, bar, pol_w);
                bulk_load(sB + 16384, b1, 16384u, bar, pol_w);
                bulk_load(sB + 32768, b0 + 16384, 2048u, bar, pol_w);
                bulk_load(sB + 34816, b1 + 16384, 2048u, bar, pol_w);
            };
            int i = 0;
            for (int t = blockIdx.x; t < ntiles && i < NS; t += gridDim.x) {
                const TileInfo ti = decode_wide_tile(args, tb, NB2, t);
                const int nbox = (ti.rows + 15) >> 4;
                const uint32_t a_bytes = nbox > 4 ? 16384u : (uint32_t)nbox * 2048u;
                for (int kb = 0; kb < KB && i < NS; ++kb, ++i) {
                    const int nk = min(4, (args.K - kb * 256) / 64);
                    mbar_arrive_expect_tx(&ctl.full[i], a_bytes + 36864u + 512u * nk);
                    weights(ti, kb, stages + i * kWideStageBytes + 16384, &ctl.full[i]);
                }
            }
            pdl_wait();
            pdl_trigger();
            int stage = 0;
            uint32_t phase = 0, issued = 0, issued_par = 0;
            bool ok = true;
            i = 0;
            for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
                const TileInfo ti = decode_wide_tile(args, tb, NB2, t);
                const int nbox = (ti.rows + 15) >> 4;
                const bool big = nbox > 4;
                const uint32_t a_bytes = big ? 16384u : (uint32_t)nbox * 2048u;
                const uint8_t* sfa = args.a_sf + (size_t)(ti.arow0 >> 7) * (args.K / 64) * 512;
                for (int kb = 0; kb < KB; ++kb, ++i) {
                    const int nk = min(4, (args.K - kb * 256) / 64);
                    uint8_t* sA = stages + stage * kWideStageBytes;
                    uint8_t* sB = sA + 16384;
                    uint8_t* sSFA = sB + 36864;
                    if (i >= NS) {
                        if (!mbar_wait(&ctl.empty[stage], phase ^ 1u, ctl.abort_flag)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(&ctl.full[stage], a_bytes + 36864u + 512u * nk);
                        weights(ti, kb, sB, &ctl.full[stage]);
                    }
                    if (big) {
                        tma_load_2d(sA, &tmA, &ctl.full[stage], kb * 128, ti.arow0, pol_a);
                    } else {
                        for (int b = 0; b < nbox; ++b)
                            tma_load_2d(sA + b * 2048, &tmA16, &ctl.full[stage], kb * 128,
                                        ti.arow0 + 16 * b, pol_a);
                    }
                    bulk_load(sSFA, sfa + kb * 2048, 512u * nk, &ctl.full[stage], pol_a);
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
                *ctl.abort_flag = 1;
            }
            for (int s = 0; s < NS; ++s)  // copies in flight land before exit
                if ((issued >> s) & 1u) mbar_wait(&ctl.full[s], (issued_par >> s) & 1u, ctl.zero);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_nvf4(128, 256);
            int stage = 0, it = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x, ++it) {
                if (!mbar_wait(&ctl.acc_empty[0], (it & 1) ^ 1u, ctl.abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait(&ctl.ready[stage], phase, ctl.abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const int nk = min(4, (args.K - kb * 256) / 64);
                    uint8_t* sA = stages + stage * kWideStageBytes;
                    uint8_t* sB = sA + 16384;
                    const uint32_t sfa_t = tmem + 256 + stage * 48, sfb_t = sfa_t + 16;
                    const uint64_t ad = sdesc_sw128(smem_u32(sA)), bd = sdesc_sw128(smem_u32(sB));
                    for (int j = 0; j < nk; ++j)
                        tc_mma_nvf4(tmem, ad + 2 * j, bd + 2 * j, idesc, sfa_t + 4 * j,
                                    sfb_t + 8 * j, (kb | j) != 0);
                    tc_commit(&ctl.empty[stage]);
                    if (++stage == NS) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                tc_commit(&ctl.acc_full[0]);
            }
            if (!ok) {
                set_status(args.status, MOE_DEV_WAIT_TIMEOUT);
                *ctl.abort_flag = 1;
            }
            tc_commit(ctl.drain);  // every MMA issued above is complete after this
            mbar_wait(ctl.drain, 0, ctl.zero);
        }
        __syncwarp();
    } else if (warp >= 10) {
        // scale warps (one per TMEM lane quarter): the stage's activation scales (columns
        // 256 + 48 s + 4 j + c: rows 32 c + lane) and the 256 weight rows' scales (columns
        // + 16 + 8 j + c: weight rows 32 c + lane, c < 4 from the first tile's atoms, c >= 4
        // from the second's)
        const int q = warp & 3;
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
            for (int kb = 0; kb < KB; ++kb) {
                if (!warp_wait(&ctl.full[stage], phase, ctl.abort_flag)) {
                    ok = false;
                    break;
                }
                const uint8_t* sSFB = stages + stage * kWideStageBytes + 16384 + 32768;
                const uint8_t* sSFA = sSFB + 4096;
                uint32_t ra[16], rb[32];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint4 a = *reinterpret_cast<const uint4*>(sSFA + 512 * j + 16 * lane);
                    const uint4 b0 = *reinterpret_cast<const uint4*>(sSFB + 512 * j + 16 * lane);
                    const uint4 b1 =
                        *reinterpret_cast<const uint4*>(sSFB + 2048 + 512 * j + 16 * lane);
                    ra[4 * j] = a.x;
                    ra[4 * j + 1] = a.y;
                    ra[4 * j + 2] = a.z;
                    ra[4 * j + 3] = a.w;
                    rb[8 * j] = b0.x;
                    rb[8 * j + 1] = b0.y;
                    rb[8 * j + 2] = b0.z;
                    rb[8 * j + 3] = b0.w;
                    rb[8 * j + 4] = b1.x;
                    rb[8 * j + 5] = b1.y;
                    rb[8 * j + 6] = b1.z;
                    rb[8 * j + 7] = b1.w;
                }
                const uint32_t base = tmem + ((uint32_t)(q * 32) << 16) + 256 + stage * 48;
                tmem_st16(base, ra);
                tmem_st32(base + 16, rb);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctl.ready[stage]);
                if (++stage == NS) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        if (!ok && lane == 0) {
            set_status(args.status, MOE_DEV_WAIT_TIMEOUT);
            *ctl.abort_flag = 1;
        }
    } else {
        // epilogue: quarter q, weight tile nb + h of the pair (accumulator columns 128 h ..)
        const int q = warp & 3, h = (warp - 2) >> 2;
        int it = 0, pp = 0;
        pdl_wait();
        for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++it) {
            TileInfo ti = decode_wide_tile(args, tb, NB2, t);
            ti.nb += h;
            ti.brow0 += 128 * h;
            const EpiPrep ep = epi_prep(args, ti, q, lane);
            if (!warp_wait(&ctl.acc_full[0], it & 1, ctl.abort_flag)) {
                if (lane == 0) {
                    set_status(args.status, MOE_DEV_WAIT_TIMEOUT);
                    *ctl.abort_flag = 1;
                }
                break;
            }
            tc_fence_after();
            run_epilogue(args, ti, ep, tmem + 128 * h, q, lane, &tmY,
                         staging + (warp - 2) * 4096, pp, 2048);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl.acc_empty[0]);
        }
        if (lane == 0) bulk_wait_all();  // staged stores complete before the CTA exits
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ============================================================== W4A4 on CTA pairs
//
// Two CTAs of a cluster share one 256-row tile: each holds its own 128-row block of an
// expert group's rows (the MMA's A, 128 of M = 256) and half of the 128-row weight tile (the
// MMA's B: weight rows 64 r .. 64 r + 63 of CTA r), so each CTA loads and keeps half of the
// weight bytes the one-CTA kernel does for the same work.  The leader (cluster rank 0) issues
// tcgen05.mma.cta_group::2 (M = 256, N = 128); each CTA's TMEM receives its own 128 rows x 128
// weight columns, so the epilogue is the one-CTA kernel's.  Each CTA's TMEM holds its own
// rows' activation scales and all 128 weight rows' scales (its scale warps write both).
//
// Synchronisation across the pair: the leader's MMA thread waits on its ready barrier, which
// the scale warps of both CTAs arrive on (the peer's remotely, after its stage has landed);
// its accumulator-empty barrier likewise counts the epilogue warps of both CTAs; the MMA
// commits arrive on the stage-empty and accumulator-full barriers of both CTAs (multicast).
// A group with an odd number of row blocks leaves the second CTA's half of its last pair
// empty (no rows loaded, nothing stored).

struct PairTables {
    const int32_t* mb_start;  // [G+1]
    const int32_t* counts;    // [G]
    const int32_t* offsets;   // [G+1]
    const int32_t* pb_start;  // [G+1] first pair block of each group
    const int32_t* pb_group;  // [pair blocks] group of each pair block
};

__host__ __device__ inline int pair_table_ints(int G, int rb_cap) { return 4 * G + 4 + rb_cap + 32; }

// Builds the pair tables in shared memory (all threads; ends with __syncthreads).
__device__ __forceinline__ PairTables load_pair_tables(const GemmArgs& a, int32_t* sm)
{
    const int G = a.G;
    int32_t* m = sm;
    int32_t* c = m + (G + 1);
    int32_t* o = c + G;
    int32_t* ps = o + (G + 1);
    int32_t* pg = ps + (G + 1);
    int32_t* ws = pg + a.rb_cap;
    const int nthr = blockDim.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int i = tid; i <= G; i += nthr) {
        m[i] = a.mb_start[i];
        o[i] = a.offsets[i];
        if (i < G) c[i] = a.counts[i];
    }
    __syncthreads();
    const int per = (G + nthr - 1) / nthr;
    const int g0 = min(G, tid * per), g1 = min(G, g0 + per);
    auto npb = [&](int g) {  // pair blocks of group g (its row blocks within the capacity)
        const int nmb = max(0, min(m[g + 1], a.rb_cap) - max(m[g], 0));
        return (nmb + 1) >> 1;
    };
    int sum = 0;
    for (int g = g0; g < g1; ++g) sum += npb(g);
    int v = sum;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, v, d);
        if (lane >= d) v += t;
    }
    if (lane == 31) ws[warp] = v;
    __syncthreads();
    if (warp == 0) {
        const int nw = nthr >> 5;
        int w = lane < nw ? ws[lane] : 0;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, w, d);
            if (lane >= d) w += t;
        }
        if (lane < nw) ws[lane] = w;
    }
    __syncthreads();
    int pre = v - sum + (warp > 0 ? ws[warp - 1] : 0);
    for (int g = g0; g < g1; ++g) {
        ps[g] = pre;
        const int n = npb(g);
        for (int b = 0; b < n; ++b) pg[pre + b] = g;
        pre += n;
    }
    if (tid == nthr - 1) ps[G] = pre;
    __syncthreads();
    PairTables tb;
    tb.mb_start = m;
    tb.counts = c;
    tb.offsets = o;
    tb.pb_start = ps;
    tb.pb_group = pg;
    return tb;
}

// Pair tile t (groups in order; inside a group, weight tiles in order; inside a weight tile,
// the group's pair blocks) as seen by the CTA of cluster rank `rank`: its row block is
// 2 mbp + rank of the group (rows 0 when the group has no such block).
__device__ __forceinline__ TileInfo decode_pair_tile(const GemmArgs& a, const PairTables& tb,
                                                     int NB, int t, int rank)
{
    const int g = tb.pb_group[t / NB];
    const int npb = tb.pb_start[g + 1] - tb.pb_start[g];
    const int local = t - tb.pb_start[g] * NB;
    const int nb = npb == 1 ? local : local / npb, mbp = npb == 1 ? 0 : local % npb;
    const int mb = 2 * mbp + rank;
    const int nmb = max(0, min(tb.mb_start[g + 1], a.rb_cap) - max(tb.mb_start[g], 0));
    TileInfo ti;
    ti.g = g;
    ti.nb = nb;
    ti.rows = mb < nmb ? min(128, tb.counts[g] - 128 * mb) : 0;
    ti.arow0 = tb.offsets[g] + 128 * mb;
    ti.brow0 = g * a.N + 128 * nb;
    return ti;
}

__global__ void __launch_bounds__(kNvf4Threads, 1)
    gemm_nvf4_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                          const __grid_constant__ CUtensorMap tmA16,
                          const __grid_constant__ CUtensorMap tmY, GemmArgs args)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* stages = aligned_smem(smem_raw);
    const int NS = args.stages;
    uint8_t* staging = stages + NS * kPairStageBytes;  // epilogue staging (down epilogues)
    Ctl ctl = carve(staging + args.staging, kMaxStages);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rank = (int)cluster_ctarank();
    const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
    const int NB = args.N / 128;
    const int KB = (args.K + 255) / 256;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&ctl.full[s], 1);
            mbar_init(&ctl.empty[s], 1);
            mbar_init(&ctl.ready[s], 8);  // the scale warps of both CTAs (the leader's)
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&ctl.acc_full[b], 1);
            mbar_init(&ctl.acc_empty[b], 8);  // the epilogue warps of both CTAs (leader's)
        }
        mbar_init(ctl.drain, 1);
        *ctl.abort_flag = 0;
        *ctl.zero = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmA16);
    }
    if (warp == 1) tmem_alloc_pair(ctl.tmem_slot, 512);
    const PairTables tb = load_pair_tables(args, tables_smem(staging + args.staging));
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // both CTAs' barriers exist before any arrives across the pair
    tc_fence_after();
    const uint32_t tmem = *ctl.tmem_slot;
    const int ntiles = tb.pb_start[args.G] * NB;

    if (warp == 0) {
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_first(), pol_a = policy_evict_last();
            auto arm = [&](const TileInfo& ti, int nk, uint64_t* bar) {
                const int nbox = (ti.rows + 15) >> 4;
                const uint32_t a_bytes = ti.rows == 0 ? 0u : nbox > 4 ? 16384u : (uint32_t)nbox * 2048u;
                mbar_arrive_expect_tx(bar, a_bytes + 8192u + 2048u + (ti.rows ? 512u * nk : 0u));
            };
            auto weights = [&](const TileInfo& ti, int kb, uint8_t* sB, uint64_t* bar) {
                const uint8_t* blob = args.b_tiles +
                                      (((size_t)ti.g * NB + ti.nb) * KB + kb) * (size_t)kNvf4TileBytes;
                bulk_load(sB, blob + rank * 8192, 8192u, bar, pol_w);     // this CTA's 64 rows
                bulk_load(sB + 8192, blob + 16384, 2048u, bar, pol_w);    // all 128 rows' scales
            };
            // the first NS stages' weights (constant) go out before the predecessor is done
            int i = 0;
            for (int t = pair; t < ntiles && i < NS; t += npairs) {
                const TileInfo ti = decode_pair_tile(args, tb, NB, t, rank);
                for (int kb = 0; kb < KB && i < NS; ++kb, ++i) {
                    arm(ti, min(4, (args.K - kb * 256) / 64), &ctl.full[i]);
                    weights(ti, kb, stages + i * kPairStageBytes + 16384, &ctl.full[i]);
                }
            }
            pdl_wait();
            pdl_trigger();
            int stage = 0;
            uint32_t phase = 0, issued = 0, issued_par = 0;
            bool ok = true;
            i = 0;
            for (int t = pair; t < ntiles && ok; t += npairs) {
                const TileInfo ti = decode_pair_tile(args, tb, NB, t, rank);
                const int nbox = (ti.rows + 15) >> 4;
                const bool big = nbox > 4;
                const uint8_t* sfa = args.a_sf + (size_t)(ti.arow0 >> 7) * (args.K / 64) * 512;
                for (int kb = 0; kb < KB; ++kb, ++i) {
                    const int nk = min(4, (args.K - kb * 256) / 64);
                    uint8_t* sA = stages + stage * kPairStageBytes;
                    uint8_t* sB = sA + 16384;     // weight codes (64 rows), then all their scales
                    uint8_t* sSFA = sB + 8192 + 2048;
                    if (i >= NS) {  // (the first NS stages were armed above)
                        if (!mbar_wait(&ctl.empty[stage], phase ^ 1u, ctl.abort_flag)) {
                            ok = false;
                            break;
                        }
                        arm(ti, nk, &ctl.full[stage]);
                        weights(ti, kb, sB, &ctl.full[stage]);
                    }
                    if (ti.rows) {
                        if (big) {
                            tma_load_2d(sA, &tmA, &ctl.full[stage], kb * 128, ti.arow0, pol_a);
                        } else {
                            for (int b = 0; b < nbox; ++b)
                                tma_load_2d(sA + b * 2048, &tmA16, &ctl.full[stage], kb * 128,
                                            ti.arow0 + 16 * b, pol_a);
                        }
                        bulk_load(sSFA, sfa + kb * 2048, 512u * nk, &ctl.full[stage], pol_a);
                    }
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
                *ctl.abort_flag = 1;
            }
            for (int s = 0; s < NS; ++s)  // copies in flight land before exit
                if ((issued >> s) & 1u) mbar_wait(&ctl.full[s], (issued_par >> s) & 1u, ctl.zero);
        }
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {
            constexpr uint32_t idesc = idesc_nvf4(256, 128);
            int stage = 0, it = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int t = pair; t < ntiles && ok; t += npairs, ++it) {
                const int buf = it & 1;
                const uint32_t acc_par = (it >> 1) & 1;
                if (!mbar_wait_cluster(&ctl.acc_empty[buf], acc_par ^ 1u, ctl.abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_t = tmem + buf * 128;
                for (int kb = 0; kb < KB; ++kb) {
                    // both CTAs' operands in smem and their stage scales in TMEM
                    if (!mbar_wait_cluster(&ctl.ready[stage], phase, ctl.abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const int nk = min(4, (args.K - kb * 256) / 64);
                    uint8_t* sA = stages + stage * kPairStageBytes;
                    uint8_t* sB = sA + 16384;
                    const uint32_t sfa_t = tmem + 256 + stage * 32, sfb_t = sfa_t + 16;
                    const uint64_t ad = sdesc_sw128(smem_u32(sA)), bd = sdesc_sw128(smem_u32(sB));
                    for (int j = 0; j < nk; ++j)
                        tc_mma_nvf4_pair(d_t, ad + 2 * j, bd + 2 * j, idesc, sfa_t + 4 * j,
                                         sfb_t + 4 * j, (kb | j) != 0);
                    tc_commit_pair(&ctl.empty[stage], 3);
                    if (++stage == NS) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                tc_commit_pair(&ctl.acc_full[buf], 3);
            }
            if (!ok) {
                set_status(args.status, MOE_DEV_WAIT_TIMEOUT);
                *ctl.abort_flag = 1;
            }
            tc_commit_pair(ctl.drain, 1);  // every MMA issued above is complete after this
            mbar_wait(ctl.drain, 0, ctl.zero);
        }
        __syncwarp();
    } else if (warp >= 6) {
        // scale warps (one per TMEM lane quarter): this CTA's activation scales and all 128
        // weight rows' scales of each stage, smem -> registers -> TMEM columns 256 + 32 stage,
        // then an arrival on the leader's ready barrier
        const int q = warp & 3;
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int t = pair; t < ntiles && ok; t += npairs) {
            for (int kb = 0; kb < KB; ++kb) {
                if (!warp_wait(&ctl.full[stage], phase, ctl.abort_flag)) {
                    ok = false;
                    break;
                }
                const uint8_t* sSFB = stages + stage * kPairStageBytes + 16384 + 8192;
                const uint8_t* sSFA = sSFB + 2048;
                uint32_t r[32];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint4 a = *reinterpret_cast<const uint4*>(sSFA + 512 * j + 16 * lane);
                    const uint4 b = *reinterpret_cast<const uint4*>(sSFB + 512 * j + 16 * lane);
                    r[4 * j] = a.x;
                    r[4 * j + 1] = a.y;
                    r[4 * j + 2] = a.z;
                    r[4 * j + 3] = a.w;
                    r[16 + 4 * j] = b.x;
                    r[16 + 4 * j + 1] = b.y;
                    r[16 + 4 * j + 2] = b.z;
                    r[16 + 4 * j + 3] = b.w;
                }
                tmem_st32(tmem + ((uint32_t)(q * 32) << 16) + 256 + stage * 32, r);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(&ctl.ready[stage], 0);
                if (++stage == NS) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        if (!ok && lane == 0) {
            set_status(args.status, MOE_DEV_WAIT_TIMEOUT);
            *ctl.abort_flag = 1;
        }
    } else {
        const int q = warp & 3;
        int it = 0, pp = 0;
        pdl_wait();
        for (int t = pair; t < ntiles; t += npairs, ++it) {
            const TileInfo ti = decode_pair_tile(args, tb, NB, t, rank);
            const EpiPrep ep = epi_prep(args, ti, q, lane);
            const int buf = it & 1;
            const uint32_t acc_par = (it >> 1) & 1;
            if (!warp_wait(&ctl.acc_full[buf], acc_par, ctl.abort_flag)) {
                if (lane == 0) {
                    set_status(args.status, MOE_DEV_WAIT_TIMEOUT);
                    *ctl.abort_flag = 1;
                }
                break;
            }
            tc_fence_after();
            run_epilogue(args, ti, ep, tmem + buf * 128, q, lane, &tmY,
                         staging + (warp - 2) * 8192, pp);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(&ctl.acc_empty[buf], 0);
        }
        if (lane == 0) bulk_wait_all();  // staged stores complete before the CTA exits
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // the leader's MMAs have read this CTA's smem; both CTAs leave together
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, 512);
    }
}

int gemm_pair_smem_bytes(int stages, int staging, int G, int rb_cap)
{
    return stages * kPairStageBytes + staging + 1024 + kCtlBytes + 4 * pair_table_ints(G, rb_cap);
}

}  // namespace moe
