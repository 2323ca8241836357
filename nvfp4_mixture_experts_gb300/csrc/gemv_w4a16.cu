// W4A16 grouped GEMV: 16-bit activation rows x NVFP4 weights for batches in which each
// expert sees a few tokens (up to 8 rows per pass over the weights).
//
// Solar Open 2 on DGX Spark, "b12x에서의 Expert Parallelism 구현 추가": the W4A16 backend
// (bf16 activations, NVFP4 weights dequantised in the main loop) among the fused-MoE
// backends, chosen by the local workload.  With one or two tokens per expert the layer is a
// weight stream, and what bounds it is how many weight elements per clock the SM can
// dequantise and feed to a multiplier.  Measured on this GPU: the tcgen05 kind::f16 MMA
// (M128 x K16) takes 46 cycles whatever N is up to 64, i.e. 44 weight elements per clock per
// SM; the warp-level mma.sync m16n8k16 (f16 in, f32 accumulate) issues 0.8 per clock per SM,
// i.e. 205 weight elements per clock, with its A operand straight from registers -- where the
// dequantised codes already are.  So this kernel decodes each weight fragment in registers
// (cvt.rn.f16x2.e2m1x2, then one exact f16x2 multiply by the block scale: E2M1 x E4M3 has at
// most 6 significant bits and lies in [2^-10, 2688]) and runs mma.sync with the token rows
// as the 8 columns of B: the instructions per weight element do not depend on the number of
// tokens up to 8.
//
// Data flow.  A copy warp streams the weight blobs of the block's work (one per (expert,
// 128-row tile, 256-element k-block): 128 rows x 128 bytes of swizzled codes and 4 scale
// atoms, 18 KB) by 1-D bulk copies into a ring of shared-memory slots; bytes in flight, not
// registers, carry the HBM stream.  Sixteen consumer warps read every blob: warp (u, a)
// takes rows 32u .. 32u + 31 of the tile and k-step a (64 elements) of the k-block, so each
// warp waits on every phase of every ring barrier in order.
//
// Fragment layout.  The dot product does not care in which order k is summed, so each
// lane's k positions are chosen to match the blob: lane (g = lane / 4, c = lane % 4) owns
// elements 16c .. 16c + 15 of its k-step (8 code bytes, one 16-element block: one scale) for
// rows g and g + 8 of each 16-row MMA block; MMA m (0..3) takes elements 16c + 4m ..
// 16c + 4m + 3 (code bytes 2m, 2m + 1: fragment registers a0/a1 and a2/a3), and the B
// fragment of token g holds the same four positions, read from shared memory in one
// 8-byte load.  The W4A16 down blobs store each 32-bit word's codes in nibble order
// 0,2,4,6,1,3,5,7, so there the staged activations of every 8-element group are permuted
// the same way.
//
// Activations in shared memory are fp16.  gate_up's rows are already fp16 copies of
// x * gs_a.  down's bf16 intermediate rows are staged as fp16 x * 2^k_t with k_t chosen per
// token so that the row's largest magnitude lands in [2^14, 2^15): every value above 2^-28
// of the row's largest converts exactly, and the epilogue multiplies by 2^-k_t.
//
// Work: an item is a chunk of up to 8 token rows of one group (local expert or the shared
// slot) and one 128-row weight tile; a block takes a contiguous run of items, chunk-major,
// so it restages activations (and the chunk's output scales: routing weights, global
// scales) only when its chunk changes.  The four k-step warps of a unit meet in shared
// memory and the epilogue is the tensor-core kernel's: gate_up times 1 / (gs_a * gs_w),
// SwiGLU, bf16 (or fp32 gate / up when unfused); down times 2^-k_t, 1 / gs_w and the pair's
// routing weight into y.  Every wait is bounded; one that runs out sets
// MOE_DEV_WAIT_TIMEOUT and every role stops.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>

#include "kernels.cuh"

namespace moe {

namespace {

constexpr int kGvTok = kGvChunk;  // token rows per pass over the weights (the MMA's N)

// Bytes of one staged activation row of KB k-blocks (2 bytes per element), the pitch 8
// modulo 128: the B-fragment loads of a half-warp (lanes g = 0..3, c = 0..3 at byte
// g pitch + 2 (64 a + 16 c + 4 m) + const) then fall on 16 distinct 8-byte slots.
__host__ __device__ __forceinline__ int gv_row_pitch(int KB) { return 512 * KB + 8; }

// Two E4M3 bytes (low first) -> f16x2, exact.
__device__ __forceinline__ uint32_t gv_e4m3x2(uint32_t two)
{
    uint32_t d;
    asm("{\n\t.reg .b16 s;\n\tcvt.u16.u32 s, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, s;\n\t}"
        : "=r"(d)
        : "r"(two));
    return d;
}

// Bytes 2h and 2h + 1 of w, each two E2M1 codes (low nibble -> low half), as f16x2.
template <int H>
__device__ __forceinline__ void gv_e2m1_pair(uint32_t w, uint32_t& lo, uint32_t& hi)
{
    if constexpr (H == 0)
        asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %2;\n\t"
            "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t}"
            : "=r"(lo), "=r"(hi)
            : "r"(w));
    else
        asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %2;\n\t"
            "cvt.rn.f16x2.e2m1x2 %0, b2;\n\tcvt.rn.f16x2.e2m1x2 %1, b3;\n\t}"
            : "=r"(lo), "=r"(hi)
            : "r"(w));
}

__device__ __forceinline__ uint32_t gv_hmul2(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// D += A B for one m16n8k16 tile, f16 operands, f32 accumulators.
__device__ __forceinline__ void gv_mma(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                       uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// One lane's share of one k-step (64 elements) of a blob for a warp's 32 weight rows: rows
// rbase + 16 mb + 8 hh + g (index 2 mb + hh), code bytes 8c .. 8c + 7 of the k-step
// (elements 16c .. 16c + 15) and the scale word of the k-step (its byte c is the lane's).
struct GvFrag {
    uint2 code[4];
    uint32_t sw[4];
};

__device__ __forceinline__ void gv_load(GvFrag& f, const uint8_t* blob, int rbase, int ks, int lane)
{
    const int g = lane >> 2, c = lane & 3;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = rbase + 16 * (i >> 1) + 8 * (i & 1) + g;
        f.code[i] = *reinterpret_cast<const uint2*>(
            blob + r * 128 + ((((2 * ks + (c >> 1)) ^ (r & 7)) << 4) | (8 * (c & 1))));
        f.sw[i] = *reinterpret_cast<const uint32_t*>(blob + 16384 + 512 * ks + (r & 31) * 16 +
                                                     (r >> 5) * 4);
    }
}

// The 8 MMAs of one k-step: xs = this lane's B base (token g, elements 16c .. of the
// k-step).  MMA m takes elements 16c + 4m .. 16c + 4m + 3: code bytes 2m, 2m + 1.  Four
// accumulator chains, d[m & 1][mb], summed by the caller.
__device__ __forceinline__ void gv_kstep(const GvFrag& f, const uint8_t* xs, int lane,
                                         float (&d)[2][2][4])
{
    // the lane's block scale of each row, in both halves: byte c twice -> one cvt
    const uint32_t sel = (uint32_t)(lane & 3) * 0x11u;
    uint32_t sc[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) sc[i] = gv_e4m3x2(__byte_perm(f.sw[i], 0, sel));
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        const uint2 b = *reinterpret_cast<const uint2*>(xs + 8 * m);
#pragma unroll
        for (int mb = 0; mb < 2; ++mb) {
            uint32_t a[4];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int i = 2 * mb + hh;
                const uint32_t w = m < 2 ? f.code[i].x : f.code[i].y;
                uint32_t lo, hi;
                if (m & 1)
                    gv_e2m1_pair<1>(w, lo, hi);
                else
                    gv_e2m1_pair<0>(w, lo, hi);
                a[hh] = gv_hmul2(lo, sc[i]);
                a[2 + hh] = gv_hmul2(hi, sc[i]);
            }
            gv_mma(d[m & 1][mb], a, b.x, b.y);
        }
    }
}

}  // namespace

namespace {

constexpr int kGvConsumers = kGvThreads / 32 - 1;  // 16 consumer warps, then the copy warp
constexpr int kGvUnits = 4;                        // 32-row units per 128-row tile
constexpr int kGvKsteps = 4;                       // 64-element k-steps per blob
constexpr int kGvScales = 48;                      // per-chunk output scales (floats)
constexpr int kGvScaleWmax = 32;                   // ... and 16 words for the staging maxima

// Consumer-warp wait on a full barrier: every lane polls; the vote keeps the outcome
// warp-uniform should the lanes' time limits run out at different polls.
__device__ __forceinline__ bool gv_all_wait(uint64_t* bar, uint32_t parity, volatile int* abort)
{
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort));
}

__device__ __forceinline__ void gv_consumer_sync()
{
    asm volatile("bar.sync 1, %0;" ::"n"(kGvConsumers * 32) : "memory");
}

struct GvSmem {
    uint8_t* ring;
    uint8_t* sx;
    float* red;
    float* tscale;  // [kGvScales]: 2^-k_t per token, then (down) rcp(gs_w) x routing weight
                    // per token, then (gate_up) 1 / (gs_a gs_w); 16 staging words at 32
    uint64_t* full;
    uint64_t* empty;
    volatile int* abort_flag;
    int* zero;
    int* n;
    volatile int* done;  // fused kernel: gate_up items whose stores are complete (consumers)
    int* list;
};

// Partial-sum buffers: two for short items (at most 8 k-blocks), so the next item's partial
// sums need not wait for this item's epilogue; one otherwise, leaving the ring its space.
__host__ __device__ __forceinline__ int gv_nred(int K) { return (K + 255) / 256 <= 8 ? 2 : 1; }

// Bytes of sx for `rows` staged rows, rounded up to 128 so that the buffers after it start
// 16-byte aligned.
__host__ __device__ __forceinline__ size_t gv_sx_bytes(int rows, int pitch)
{
    return ((size_t)rows * pitch + 127) / 128 * 128;
}

__host__ __device__ __forceinline__ size_t gv_fixed_bytes(int K)
{
    const int nred = gv_nred(K);
    return gv_sx_bytes(kGvTok, gv_row_pitch((K + 255) / 256)) +
           nred * kGvConsumers * 32 * kGvTok * 4 + kGvScales * 4 + 2 * kGvMaxSlots * 8 + 16;
}

// ring | sx (sx_bytes: the staged activation rows) | nred partial-sum buffers | scales |
// barriers | flags | work list
__device__ __forceinline__ GvSmem gv_carve(uint8_t* base, size_t sx_bytes, int nred, int slots)
{
    GvSmem m;
    m.ring = base;
    m.sx = m.ring + (size_t)slots * kNvf4TileBytes;
    m.red = reinterpret_cast<float*>(m.sx + sx_bytes);  // sx_bytes from gv_sx_bytes
    m.tscale = m.red + nred * kGvConsumers * 32 * kGvTok;
    m.full = reinterpret_cast<uint64_t*>(m.tscale + kGvScales);
    m.empty = m.full + kGvMaxSlots;
    m.abort_flag = reinterpret_cast<volatile int*>(m.empty + kGvMaxSlots);
    m.zero = const_cast<int*>(m.abort_flag + 1);
    m.n = m.zero + 1;
    m.done = m.n + 1;
    m.list = m.n + 2;
    return m;
}

// The work list: the chunks of up to kGvTok rows of the non-empty groups, in group order,
// each (group << 16) | first row; *m.n = their number.  Called by warp 0 with the G group
// counts in tmp (shared memory): each lane takes a contiguous range of groups, then a warp
// scan places the lanes' chunks.
__device__ __forceinline__ void gv_list_from_counts(const GemmArgs& a, const GvSmem& m,
                                                    int list_cap, const int* tmp)
{
    const int lane = threadIdx.x & 31;
    const int per = (a.G + 31) / 32;
    const int gb = lane * per, ge = min(a.G, gb + per);
    int nc = 0;  // chunks of this lane's groups
    for (int g = gb; g < ge; ++g) nc += (tmp[g] + kGvTok - 1) / kGvTok;
    int incl = nc;  // inclusive scan of the chunk counts over the warp
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    const int n = __shfl_sync(0xffffffffu, incl, 31);
    int slot = incl - nc;
    for (int g = gb; g < ge; ++g)
        for (int r = 0; r < tmp[g]; r += kGvTok, ++slot)
            if (slot < list_cap) m.list[slot] = (g << 16) | r;
    if (lane == 0) {
        if (n > list_cap) set_status(a.status, MOE_DEV_ROWS_OVERFLOW);
        *m.n = min(n, list_cap);
    }
}

// gv_list_from_counts from the grouping's counts (a.counts), loaded 16 per lane at a time
// (one load latency for up to 512 groups).
__device__ __forceinline__ void gv_build_list(const GemmArgs& a, const GvSmem& m, int list_cap,
                                              int* tmp)
{
    const int lane = threadIdx.x & 31;
    const int per = (a.G + 31) / 32;
    const int gb = lane * per, ge = min(a.G, gb + per);
    for (int g0 = gb; g0 < ge; g0 += 16) {
        int c[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) c[j] = g0 + j < ge ? a.counts[g0 + j] : 0;
#pragma unroll
        for (int j = 0; j < 16; ++j)
            if (g0 + j < ge) tmp[g0 + j] = max(c[j], 0);
    }
    __syncwarp();
    gv_list_from_counts(a, m, list_cap, tmp);
}

// The same list from the top-k ids (P <= 32 * kGvIdsLanePairs pairs): the counts the grouping
// kernel forms from them (an id outside [0, E) or outside the shard's experts off .. off +
// G - 2 has no row; the shared group, the last, has shared_rows), so the list needs nothing
// the grouping writes.
constexpr int kGvIdsLanePairs = 2;
__device__ __forceinline__ void gv_build_list_ids(const GemmArgs& a, const GvSmem& m,
                                                  int list_cap, int* tmp, const int32_t* ids,
                                                  int P, int E, int off, int shared_rows)
{
    const int lane = threadIdx.x & 31;
    const int El = a.G - 1;
    int id[kGvIdsLanePairs];
#pragma unroll
    for (int j = 0; j < kGvIdsLanePairs; ++j) {
        const int i = 32 * j + lane;
        id[j] = i < P ? ids[i] : -1;
    }
    for (int g = lane; g < a.G; g += 32) tmp[g] = g < El ? 0 : shared_rows;
    __syncwarp();
#pragma unroll
    for (int j = 0; j < kGvIdsLanePairs; ++j) {
        const int le = id[j] - off;
        if (id[j] >= 0 && id[j] < E && le >= 0 && le < El) atomicAdd(&tmp[le], 1);
    }
    __syncwarp();
    gv_list_from_counts(a, m, list_cap, tmp);
}

// bf16 pair -> two floats times `up`, rounded to an fp16 pair.
__device__ __forceinline__ uint32_t gv_bf16x2_to_f16x2(uint32_t u, float up)
{
    const __half2 v = __floats2half2_rn(__uint_as_float(u << 16) * up,
                                        __uint_as_float(u & 0xFFFF0000u) * up);
    return *reinterpret_cast<const uint32_t*>(&v);
}

// The chunk's nt token rows (K 16-bit values each, from row row0 of xin) -> sx as fp16,
// zeros past K, by all consumer warps: 16 / nt (rounded to a power of two) warps per row,
// each lane four 16-byte pieces in flight at a time.  down: each row's bf16 values are taken
// times 2^k_t (k_t from the row's largest magnitude, met across its warps in shared memory)
// and every 8-element group is stored in the blobs' nibble order 0,2,4,6,1,3,5,7.  Also the
// chunk's output scales: 2^-k_t, and rcp(gs_w) x the routing weight per row (down) or
// 1 / (gs_a gs_w) (gate_up).  Ends with the staged data visible to every consumer.
// kSrc: where row t of the chunk comes from -- kGvSrcRows: row row0 + t of xin;
// kGvSrcRowsL2: the same through L2 (ld.global.cg: rows written earlier in the same launch);
// kGvSrcTokens (gate_up): the layer input row of the row's token (from perm_src: pair / k,
// or pair - T k for a shared row) in bf16, times the prescale gs, rounded to fp16 -- the row
// the gather kernel would have written; kGvSrcSmem: row t of xin in shared memory.
constexpr int kGvSrcRows = 0, kGvSrcRowsL2 = 1, kGvSrcTokens = 2, kGvSrcSmem = 3;
template <bool kGateUp, int kSrc = kGvSrcRows>
__device__ __forceinline__ void gv_stage_chunk(const GemmArgs& a, const GvSmem& m,
                                               const uint16_t* xin, int64_t row0, int nt,
                                               int g, int K, int KB, int pitch, int T = 0,
                                               int k = 1, float gs = 1.0f)
{
    static_assert(kSrc != kGvSrcTokens || kGateUp, "token rows are gate_up's input");
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wpt = nt <= 1 ? 16 : nt <= 2 ? 8 : nt <= 4 ? 4 : 2;
    const int t = warp / wpt, sub = warp % wpt;
    const bool act = t < nt;
    const int npc = KB * 32;  // 8-element pieces of a staged row
    const int S = wpt * 32;   // the row's threads
    int64_t srow = (kSrc == kGvSrcSmem ? 0 : row0) + (act ? t : 0);
    bool rd = act;  // the row has a source (else it is staged as zeros)
    if constexpr (kSrc == kGvSrcTokens) {
        srow = 0;
        if (act) {
            const int pair = a.perm_src[row0 + t];
            const int tok = pair >= a.Tk ? pair - a.Tk : pair / k;
            if (pair < 0 || tok >= T) {  // not a row of this batch
                if (sub == 0 && lane == 0) set_status(a.status, MOE_DEV_BAD_INDEX);
                rd = false;
            } else {
                srow = tok;
            }
        }
    }
    const uint16_t* src = xin + srow * K;
    uint8_t* dst = m.sx + (act ? t : 0) * pitch;
    auto ld16 = [](const uint16_t* q) {
        if constexpr (kSrc == kGvSrcRowsL2)
            return __ldcg(reinterpret_cast<const uint4*>(q));
        else
            return *reinterpret_cast<const uint4*>(q);
    };
    // the chunk's output scales are loaded first, so their latency (a dependent pair of loads
    // for down: the pair index, then its routing weight) overlaps the row staging
    const bool scl = act && sub == 0 && lane == 0;
    float gw = 1.0f, sc = 1.0f;
    if (scl) {
        gw = a.gs_w[g];
        if constexpr (kGateUp) {
            if (t == 0) sc = kSrc == kGvSrcTokens ? gs : *a.gs_a;
        } else {
            const int pair = a.perm_src[row0 + t];
            sc = !pair_ok(pair, a.status) ? 0.0f : pair < a.Tk ? a.topk_w[pair] : 1.0f;
        }
    }
    float up = 1.0f;  // down: 2^k_t
    if constexpr (!kGateUp) {
        uint32_t mx = 0;  // largest bf16 magnitude (bits), this thread's pieces
        if (act)
            for (int p0 = sub * 32 + lane; p0 < npc; p0 += 4 * S) {
                uint4 q[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int p = p0 + j * S;
                    q[j] = (rd && p < npc && 8 * p < K) ? ld16(src + 8 * p) : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t u[4] = {q[j].x, q[j].y, q[j].z, q[j].w};
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        mx = max(mx, max(u[i] & 0x7FFFu, (u[i] >> 16) & 0x7FFFu));
                }
            }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        uint32_t* wmax = reinterpret_cast<uint32_t*>(m.tscale + kGvScaleWmax);
        if (lane == 0) wmax[warp] = mx;
        gv_consumer_sync();
        if (act) {
            for (int w = 0; w < wpt; ++w) mx = max(mx, wmax[t * wpt + w]);
            // bf16 exponent field of the largest magnitude -> k_t in [-113, 113]
            const int ex = (int)(mx >> 7) - 127;
            const int kt = mx ? max(-113, min(113, 14 - ex)) : 0;
            up = __uint_as_float((uint32_t)(127 + kt) << 23);
            if (sub == 0 && lane == 0) m.tscale[t] = __uint_as_float((uint32_t)(127 - kt) << 23);
        }
    }
    if (act)
        for (int p0 = sub * 32 + lane; p0 < npc; p0 += 4 * S) {
            uint4 q[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int p = p0 + j * S;
                q[j] = (rd && p < npc && 8 * p < K) ? ld16(src + 8 * p) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int p = p0 + j * S;
                if (p >= npc) break;
                uint2 lo, hi;  // elements (0..3, 4..7), or (0,2,4,6), (1,3,5,7) for down
                if constexpr (kSrc == kGvSrcTokens) {
                    lo = make_uint2(gv_bf16x2_to_f16x2(q[j].x, gs), gv_bf16x2_to_f16x2(q[j].y, gs));
                    hi = make_uint2(gv_bf16x2_to_f16x2(q[j].z, gs), gv_bf16x2_to_f16x2(q[j].w, gs));
                } else if constexpr (kGateUp) {
                    lo = make_uint2(q[j].x, q[j].y);
                    hi = make_uint2(q[j].z, q[j].w);
                } else {
                    const uint32_t h0 = gv_bf16x2_to_f16x2(q[j].x, up),
                                   h1 = gv_bf16x2_to_f16x2(q[j].y, up),
                                   h2 = gv_bf16x2_to_f16x2(q[j].z, up),
                                   h3 = gv_bf16x2_to_f16x2(q[j].w, up);
                    // h_i = (x_2i, x_2i+1) -> (x0, x2), (x4, x6) | (x1, x3), (x5, x7)
                    lo = make_uint2(__byte_perm(h0, h1, 0x5410), __byte_perm(h2, h3, 0x5410));
                    hi = make_uint2(__byte_perm(h0, h1, 0x7632), __byte_perm(h2, h3, 0x7632));
                }
                uint8_t* d = dst + 16 * p;
                *reinterpret_cast<uint2*>(d) = lo;
                *reinterpret_cast<uint2*>(d + 8) = hi;
            }
        }
    if (scl) {
        if constexpr (kGateUp) {
            if (t == 0) m.tscale[2 * kGvTok] = __frcp_rn(__fmul_rn(sc, gw));
        } else {
            m.tscale[kGvTok + t] = __fmul_rn(__frcp_rn(gw), sc);
        }
    }
    gv_consumer_sync();
}

// The k-slots' partials of tile nb summed, scaled and stored by the consumer threads.
// kNks: partial-sum sets in red (the k-step warps' 4, or 1 already summed).
template <bool kGateUp, int kNks = kGvKsteps>
__device__ __forceinline__ void gv_epilogue(const GemmArgs& a, const GvSmem& m,
                                            const float* red, int64_t row0, int nt, int nb)
{
    const int tid = threadIdx.x;  // consumers: 0 .. 32 kGvConsumers - 1
    if constexpr (kGateUp) {
        // output (token t, feature 64 nb + j): gate row j % 16, up row 16 + j % 16 of unit j / 16
        const float alpha = m.tscale[2 * kGvTok];
        const int I = a.N / 2;
        for (int o = tid; o < 64 * kGvTok; o += kGvConsumers * 32) {
            const int t = o & (kGvTok - 1), j = o / kGvTok;  // token fastest: every warp
            if (t >= nt) continue;                            // takes a share

            const int u = j >> 4, fi = j & 15;
            float vg = 0.0f, vu = 0.0f;
#pragma unroll
            for (int s = 0; s < kNks; ++s) {
                const float* rw = red + (s * kGvUnits + u) * 32 * kGvTok;
                vg += rw[fi * kGvTok + t];
                vu += rw[(16 + fi) * kGvTok + t];
            }
            vg = __fmul_rn(vg, alpha);
            vu = __fmul_rn(vu, alpha);
            const int64_t row = row0 + t;
            const int f = 64 * nb + j;
            if (a.epilogue == kEpiGateUpF32) {
                a.out_f32[row * a.N + f] = vg;
                a.out_f32[row * a.N + I + f] = vu;
            } else {
                a.out_bf16[row * I + f] = __bfloat16_as_ushort(__float2bfloat16_rn(silu_mul(vg, vu)));
            }
        }
    } else {
        // output (token t, row 128 nb + j)
        for (int o = tid; o < 128 * kGvTok; o += kGvConsumers * 32) {
            const int t = o & (kGvTok - 1), j = o / kGvTok;  // token fastest: every warp
            if (t >= nt) continue;                            // takes a share

            const int u = j >> 5, ri = j & 31;
            float v = 0.0f;
#pragma unroll
            for (int s = 0; s < kGvKsteps; ++s) v += red[((s * kGvUnits + u) * 32 + ri) * kGvTok + t];
            a.out_f32[(row0 + t) * a.N + 128 * nb + j] =
                __fmul_rn(v, m.tscale[t]) * m.tscale[kGvTok + t];
        }
    }
}

}  // namespace

size_t gemv_w4a16_smem(int K, int slots, int list_cap)
{
    return (size_t)slots * kNvf4TileBytes + gv_fixed_bytes(K) + 4 * (size_t)list_cap;
}

int gemv_w4a16_slots(int K, int list_cap)
{
    const size_t fixed = gv_fixed_bytes(K) + 4 * (size_t)list_cap;
    if (fixed >= (size_t)kSmemLimit) return 0;
    return (int)std::min<size_t>(kGvMaxSlots, ((size_t)kSmemLimit - fixed) / kNvf4TileBytes);
}

// kGateUp: N = 2I interleaved gate/up rows, x the fp16 rows x * gs_a, epilogue
// kEpiGateUpSwiglu or kEpiGateUpF32.  Else N = H rows of W2 (nibble-pair blobs), x the bf16
// intermediate, epilogue kEpiDown.  slots: weight blobs in the shared-memory ring.  Every
// consumer warp reads every blob (its unit's rows, its k-step), so each warp waits on every
// phase of every ring barrier in order and no parity wait can be satisfied by a stale phase.
template <bool kGateUp>
__global__ void __launch_bounds__(kGvThreads, 1)
    gemv_w4a16_kernel(GemmArgs a, const uint16_t* __restrict__ xin, int list_cap, int slots)
{
    extern __shared__ __align__(128) uint8_t gv_smem[];
    const int K = a.K, KB = (K + 255) / 256, NB = a.N / 128;
    const int pitch = gv_row_pitch(KB);
    const int nred = gv_nred(K);
    const GvSmem m = gv_carve(gv_smem, gv_sx_bytes(kGvTok, pitch), nred, slots);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < slots; ++i) {
            mbar_init(&m.full[i], 1);
            mbar_init(&m.empty[i], kGvConsumers);  // every consumer warp reads every blob
        }
        *m.abort_flag = 0;
        *m.zero = 0;
        fence_barrier_init();
    }
    // The group sizes and offsets come from the grouping kernels, which are complete when
    // this kernel starts (every kernel of the forward waits for its predecessor before it
    // lets the next one start, see pdl_wait), and the weights are constant: the work list
    // and the weight stream go ahead of the wait, which only the consumers (reading the
    // predecessor's activation rows) take.
    if (warp == 0) gv_build_list(a, m, list_cap, reinterpret_cast<int*>(m.red));
    __syncthreads();
    // items: (chunk, 128-row tile), chunk-major; a block takes a contiguous run of them
    const int nitems = *m.n * NB;
    const int i0 = (int)((int64_t)blockIdx.x * nitems / gridDim.x);
    const int i1 = (int)((int64_t)(blockIdx.x + 1) * nitems / gridDim.x);

    if (warp == kGvConsumers) {
        // copy warp: the run's blobs, in (item, k-block) order, into the ring
        if (lane == 0) {
            const uint64_t pol_stream = policy_evict_first(), pol_keep = policy_evict_last();
            uint32_t c = 0;   // blobs issued
            int sl = 0;       // their ring slot
            uint32_t ph = 0;  // the slot's phase parity
            bool ok = true;
            for (int item = i0; item < i1 && ok; ++item) {
                const int g = m.list[item / NB] >> 16, nb = item % NB;
                // the shared slot is read once per chunk: keep it in L2
                const uint64_t pol = g == a.G - 1 ? pol_keep : pol_stream;
                const uint8_t* src = a.b_tiles + (size_t)(g * NB + nb) * KB * kNvf4TileBytes;
                for (int kb = 0; kb < KB; ++kb, ++c) {
                    if (!mbar_wait(&m.empty[sl], ph ^ 1u, m.abort_flag)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&m.full[sl], kNvf4TileBytes);
                    bulk_load(m.ring + (size_t)sl * kNvf4TileBytes, src + (size_t)kb * kNvf4TileBytes,
                              kNvf4TileBytes, &m.full[sl], pol);
                    if (++sl == slots) {
                        sl = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (!ok) {
                set_status(a.status, MOE_DEV_WAIT_TIMEOUT);
                *m.abort_flag = 1;
            }
            // the copies in flight land before the block exits: the last min(c, slots)
            for (uint32_t j = c > (uint32_t)slots ? c - slots : 0; j < c; ++j)
                mbar_wait(&m.full[j % slots], (j / slots) & 1u, m.zero);
        }
        return;
    }

    pdl_wait();
    pdl_trigger();
    // consumer warps: unit my_u (rows 32 my_u .. of the tile), k-step my_ks of every blob
    const int my_u = warp % kGvUnits, my_ks = warp / kGvUnits;
    const int g8 = lane >> 2, c4 = lane & 3;
    bool ok = true;
    int staged = -1;  // chunk whose rows are in sx
    int g = 0, nt = 0;
    int64_t row0 = 0;
    int sl = 0;       // ring slot of the next blob
    uint32_t ph = 0;  // its full-barrier phase parity
    for (int item = i0; item < i1; ++item) {
        const int ci = item / NB, nb = item % NB;
        if (ci != staged) {
            const int e = m.list[ci];
            const int t0 = e & 0xFFFF;
            g = e >> 16;
            nt = min(kGvTok, a.counts[g] - t0);
            row0 = (int64_t)a.offsets[g] + t0;
        }
        // the previous item's readers of sx, the scales and (one buffer) red are done
        if (nred == 1 || ci != staged) gv_consumer_sync();
        if (ci != staged) {
            gv_stage_chunk<kGateUp>(a, m, xin, row0, nt, g, K, KB, pitch);
            staged = ci;
        }
        float d[2][2][4] = {};
        const uint8_t* xs = m.sx + g8 * pitch + 2 * (64 * my_ks + 16 * c4);
        for (int kb = 0; kb < KB; ++kb) {
            if (ok && !gv_all_wait(&m.full[sl], ph, m.abort_flag)) {
                ok = false;
                if (lane == 0) {
                    set_status(a.status, MOE_DEV_WAIT_TIMEOUT);
                    *m.abort_flag = 1;
                }
            }
            if (ok) {
                GvFrag f;
                gv_load(f, m.ring + (size_t)sl * kNvf4TileBytes, 32 * my_u, my_ks, lane);
                gv_kstep(f, xs + 512 * kb, lane, d);
                __syncwarp();
                if (lane == 0) mbar_arrive(&m.empty[sl]);
            }
            if (++sl == slots) {
                sl = 0;
                ph ^= 1u;
            }
        }
#pragma unroll
        for (int mb = 0; mb < 2; ++mb)
#pragma unroll
            for (int r = 0; r < 4; ++r) d[0][mb][r] += d[1][mb][r];
        // partial sums: red[warp][row][token], row = 16 mb + 8 hh + g, token 2c, 2c + 1
        float* redb = m.red + (nred == 2 ? ((item - i0) & 1) : 0) * kGvConsumers * 32 * kGvTok;
        float* rw = redb + warp * 32 * kGvTok;
#pragma unroll
        for (int mb = 0; mb < 2; ++mb)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh)
                *reinterpret_cast<float2*>(rw + (16 * mb + 8 * hh + g8) * kGvTok + 2 * c4) =
                    make_float2(d[0][mb][2 * hh], d[0][mb][2 * hh + 1]);
        gv_consumer_sync();
        if (ok) gv_epilogue<kGateUp>(a, m, redb, row0, nt, nb);
    }
}

// ---------------------------------------------------------------- fused gate_up + down
//
// The forward's two grouped GEMVs in one launch, for batches of a few tokens.  With one
// token the layer streams about 80 MB of weights in a few microseconds, and what two launches
// cost is their seams: the down launch's blocks cannot start until the gate_up blocks leave
// (each holds most of an SM's shared memory), then rebuild the work list and refill the ring,
// all while the stream is idle.  Here each block's copy warp streams its gate_up blobs and
// then its down blobs without a break, and a down item waits only for its own chunk: the
// chunk's intermediate rows are complete when all 2I / 128 of its gate_up tiles have been
// stored (ready[chunk] counts them: a block barrier after the stores, then one release add;
// the reader polls with acquire loads).  The activation rows are taken from the layer input
// directly (the gather kernel's fp16 rows x * gs, formed while staging).  With at most 64
// pairs the work list is formed from the top-k ids before the dependency wait (they are two
// launches back, so complete), and the weight stream starts while the grouping kernel runs.
//
// Few items: with one token the gate_up work is 9 chunks x 20 tiles = 180 items of 16 blobs
// on 152 SMs, and the SMs with two set the pace.  So when there are few items the contraction
// of each tile is cut into S parts (items of 16 / S blobs); each part stores its partial sums
// (fp32, 128 rows per token) and counts itself in ready[chunk], and the down stager of the
// chunk adds the S parts in the order of their k ranges and applies the gate_up epilogue's
// scale and SwiGLU (so the result does not depend on the order the parts finished in).
//
// Items: gate_up (chunk, tile, part), then down (chunk, tile), each list split evenly over the
// blocks in contiguous runs; a block takes its gate_up run, then its down run backwards
// (GvCursor).  Warps: 16 consumers, a copy warp, and a signal warp that publishes the
// finished gate_up items (a release add waits for the stores to land; the consumers go on
// meanwhile).  The launch is cooperative, so every block is resident at once (one block per
// SM, grid <= SMs) and every wait ends; each wait is bounded all the same, and one that runs
// out sets MOE_DEV_WAIT_TIMEOUT and stops the block's work.  The ready words are zeroed
// before the launch by the routing kernel.
__device__ __forceinline__ bool gv_wait_count(const int32_t* p, int target, volatile int* abort)
{
    if (ld_acquire_gpu(p) >= target) return true;
    const uint64_t t0 = globaltimer();
    for (;;) {
        __nanosleep(100);
        if (ld_acquire_gpu(p) >= target) return true;
        if (*abort) return false;
        if (globaltimer() - t0 > kWaitLimitNs) return false;
    }
}

// After the consumers' stores of gate_up item `it` (a tile or a part): the barrier orders every
// consumer's stores before thread 0's release of the block's count of finished items, which
// the signal warp turns into release adds on the chunks' ready words (so no consumer waits
// for its stores to land).
__device__ __forceinline__ void gv_item_done(const GvSmem& m, int it)
{
    gv_consumer_sync();
    if (threadIdx.x == 0) {
        __threadfence_block();
        *m.done = it + 1;
    }
}

// Split gate_up tiles: the chunk's intermediate rows from its parts' partial sums (part
// [tile][s][token][128 rows], s in k order), as the gate_up epilogue would form them: gate and
// up sums times alpha = 1 / (gs gs_w), SwiGLU, rounded to bf16 -> rows t < nt of dst (shared
// memory, I per row).  Each thread takes 4 features (adjacent gate rows, and their up rows).
__device__ __forceinline__ void gv_split_rows(const float* part, int ci, int NBg, int S, int nt,
                                              int I, float alpha, uint16_t* dst)
{
    const int q4 = I / 4;
    for (int e = threadIdx.x; e < nt * q4; e += kGvConsumers * 32) {
        const int t = e / q4, f0 = 4 * (e % q4);
        const int nb = f0 / 64, j = f0 % 64, u = j / 16, fi = j % 16;
        const float* base = part + (size_t)(ci * NBg + nb) * S * (128 * kGvTok) + t * 128 + u * 32 + fi;
        float4 vg = make_float4(0.f, 0.f, 0.f, 0.f), vu = vg;
        for (int q = 0; q < S; ++q) {
            const float4 pg = __ldcg(reinterpret_cast<const float4*>(base + (size_t)q * (128 * kGvTok)));
            const float4 pu = __ldcg(reinterpret_cast<const float4*>(base + (size_t)q * (128 * kGvTok) + 16));
            vg.x += pg.x; vg.y += pg.y; vg.z += pg.z; vg.w += pg.w;
            vu.x += pu.x; vu.y += pu.y; vu.z += pu.z; vu.w += pu.w;
        }
        const float g4[4] = {vg.x, vg.y, vg.z, vg.w}, u4[4] = {vu.x, vu.y, vu.z, vu.w};
        uint16_t* o = dst + t * I + f0;
#pragma unroll
        for (int i = 0; i < 4; ++i)
            o[i] = __bfloat16_as_ushort(__float2bfloat16_rn(
                silu_mul(__fmul_rn(g4[i], alpha), __fmul_rn(u4[i], alpha))));
    }
}

// A block's items in order, decoded one step at a time: its gate_up run ascending (chunk,
// tile, part), then its down run descending (chunk, tile).  Descending, because the runs are
// contiguous and chunk-major: the block's first down chunk is then its last gate_up chunk,
// whose other tiles the next block took first -- complete as soon as this block's own
// gate_up run is -- while the chunk it shares with the previous block (finished last there)
// comes last.
struct GvCursor {
    int ci, nb, s;  // the current item: chunk, tile, part
    bool isg;       // gate_up (else down)
    int left;       // gate_up items left, the current one included
    int S, NBg, NBd, d1;
    __device__ __forceinline__ void init(int u0, int nu, int d1_, int S_, int NBg_, int NBd_)
    {
        S = S_;
        NBg = NBg_;
        NBd = NBd_;
        d1 = d1_;
        left = nu;
        if (nu > 0) {
            isg = true;
            ci = u0 / (NBg * S);
            nb = (u0 / S) % NBg;
            s = u0 % S;
        } else {
            to_down();
        }
    }
    __device__ __forceinline__ void to_down()
    {
        isg = false;
        s = 0;
        ci = (d1 - 1) / NBd;  // (d1 - 1 < 0 only when the run is empty: never read)
        nb = (d1 - 1) % NBd;
    }
    __device__ __forceinline__ void next()
    {
        if (isg) {
            if (--left == 0) {
                to_down();
            } else if (++s == S) {
                s = 0;
                if (++nb == NBg) {
                    nb = 0;
                    ++ci;
                }
            }
        } else if (--nb < 0) {
            nb = NBd - 1;
            --ci;
        }
    }
};

// sx holds up to tok_rows staged rows of the gate_up width; one partial-sum buffer (a second
// one, letting warps start the next item before the slowest has read this item's sums, made
// every size slower: 321 vs 315 us at 32 tokens, 714 vs 699 us at 256)
__host__ __device__ __forceinline__ size_t gv_fused_fixed_bytes(int H, int tok_rows)
{
    return gv_sx_bytes(tok_rows, gv_row_pitch((H + 255) / 256)) +
           kGvConsumers * 32 * kGvTok * 4 + kGvScales * 4 + 2 * kGvMaxSlots * 8 + 16;
}

__global__ void __launch_bounds__(kGvFusedThreads, 1)
    gemv_w4a16_fused_kernel(GvFusedArgs f, int list_cap, int slots)
{
    extern __shared__ __align__(128) uint8_t gv_smem[];
    const GemmArgs& gu = f.gu;
    const GemmArgs& dn = f.dn;
    const int KBg = (gu.K + 255) / 256, NBg = gu.N / 128;
    const int KBd = (dn.K + 255) / 256, NBd = dn.N / 128;
    const int pg = gv_row_pitch(KBg), pd = gv_row_pitch(KBd);
    const GvSmem m = gv_carve(gv_smem, gv_sx_bytes(f.tok_rows, pg), 1, slots);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < slots; ++i) {
            mbar_init(&m.full[i], 1);
            mbar_init(&m.empty[i], kGvConsumers);  // every consumer warp reads every blob
        }
        *m.abort_flag = 0;
        *m.zero = 0;
        *m.done = 0;
        fence_barrier_init();
    }
    // The work list.  The group counts and the rows' pairs come from the predecessor (the
    // grouping kernel); with few pairs the list is formed from the top-k ids instead, which
    // the kernel before the predecessor wrote (complete when this kernel starts), so the copy
    // warp streams weights while the grouping kernel runs.  The consumers wait (pdl_wait)
    // before they read its output.
    const int npairs = f.T * f.k;
    const bool list_from_ids = npairs <= 32 * kGvIdsLanePairs;
    if (!list_from_ids) pdl_wait();
    if (warp == 0) {
        if (list_from_ids)
            gv_build_list_ids(gu, m, list_cap, reinterpret_cast<int*>(m.red), f.ids, npairs,
                              f.E, f.off, f.shared_rows);
        else
            gv_build_list(gu, m, list_cap, reinterpret_cast<int*>(m.red));
    }
    __syncthreads();
    const int n = *m.n;
    // parts per gate_up tile (uniform over the grid: it depends on n only); the down stager
    // forms a split chunk's rows in the partial-sum buffer (16 KB)
    int S = 1;
    const bool rows_fit = (int64_t)f.tok_rows * dn.K * 2 <= kGvConsumers * 32 * kGvTok * 4;
    while (rows_fit && 2 * S <= kGvMaxSplit && KBg % (2 * S) == 0 &&
           (int64_t)n * NBg * 2 * S <= min(6LL * gridDim.x, (long long)kGvSplitItems))
        S *= 2;
    const int nkg = KBg / S;
    const int64_t Ngu = (int64_t)n * NBg * S, Ndn = (int64_t)n * NBd;
    const int64_t b = blockIdx.x, P = gridDim.x;
    const int u0 = (int)(b * Ngu / P), nu = (int)((b + 1) * Ngu / P) - u0;
    const int d0 = (int)(b * Ndn / P), d1 = (int)((b + 1) * Ndn / P), nd = d1 - d0;
    GvCursor cur;
    cur.init(u0, nu, d1, S, NBg, NBd);

    if (warp == kGvConsumers + 1) {
        // signal warp: as the consumers finish gate_up items, adds them to their chunks'
        // ready words (runs of one chunk in one add).  Bounded: it gives up when the
        // consumers stop (abort) or finish no item for the wait limit.
        if (lane == 0) {
            int j = 0;  // gate_up items published; cur is item j
            uint64_t t0 = globaltimer();
            while (j < nu) {
                const int dn_ = *m.done;
                if (dn_ > j) {
                    __threadfence_block();
                    while (j < dn_) {
                        const int ci = cur.ci;
                        int cnt = 0;
                        for (; j < dn_ && cur.isg && cur.ci == ci; ++j, ++cnt) cur.next();
                        red_release_gpu(f.ready + ci, cnt);
                    }
                    t0 = globaltimer();
                } else {
                    if (*m.abort_flag) break;
                    if (globaltimer() - t0 > kWaitLimitNs) {
                        set_status(gu.status, MOE_DEV_WAIT_TIMEOUT);
                        *m.abort_flag = 1;
                        break;
                    }
                    __nanosleep(256);
                }
            }
        }
        return;
    }
    if (warp == kGvConsumers) {
        // copy warp: the blobs of the block's gate_up run, then of its down run
        if (lane == 0) {
            const uint64_t pol_stream = policy_evict_first(), pol_keep = policy_evict_last();
            uint32_t c = 0;
            int sl = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int it = 0; it < nu + nd && ok; ++it, cur.next()) {
                const int ci = cur.ci, nb = cur.nb, s = cur.s;
                const bool isg = cur.isg;
                const int g = m.list[ci] >> 16;
                const uint64_t pol = g == gu.G - 1 ? pol_keep : pol_stream;
                const uint8_t* src =
                    isg ? gu.b_tiles + ((size_t)(g * NBg + nb) * KBg + (size_t)s * nkg) * kNvf4TileBytes
                        : dn.b_tiles + (size_t)(g * NBd + nb) * KBd * kNvf4TileBytes;
                const int nkb = isg ? nkg : KBd;
                for (int kb = 0; kb < nkb; ++kb, ++c) {
                    if (!mbar_wait(&m.empty[sl], ph ^ 1u, m.abort_flag)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&m.full[sl], kNvf4TileBytes);
                    bulk_load(m.ring + (size_t)sl * kNvf4TileBytes, src + (size_t)kb * kNvf4TileBytes,
                              kNvf4TileBytes, &m.full[sl], pol);
                    if (++sl == slots) {
                        sl = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (!ok) {
                set_status(gu.status, MOE_DEV_WAIT_TIMEOUT);
                *m.abort_flag = 1;
            }
            for (uint32_t j = c > (uint32_t)slots ? c - slots : 0; j < c; ++j)
                mbar_wait(&m.full[j % slots], (j / slots) & 1u, m.zero);
        }
        return;
    }

    if (list_from_ids) pdl_wait();
    if (threadIdx.x == 0) pdl_trigger();
    const int my_u = warp % kGvUnits, my_ks = warp / kGvUnits;
    const int g8 = lane >> 2, c4 = lane & 3;
    const int xr = min(g8, f.tok_rows - 1);  // the B-fragment row (rows past tok_rows repeat)
    const float gs = f16_prescale(f.amax);
    if (blockIdx.x == 0 && threadIdx.x == 0 && f.gs_out) *f.gs_out = gs;
    bool ok = true;
    int staged = -1;  // 2 chunk + (1 for down) of the rows in sx
    int nt = 0;
    int64_t row0 = 0;
    int sl = 0;
    uint32_t ph = 0;
    for (int it = 0; it < nu + nd; ++it, cur.next()) {
        const int ci = cur.ci, nb = cur.nb, s = cur.s;
        const bool isg = cur.isg;
        const int key = 2 * ci + (isg ? 0 : 1);
        if (key != staged) {
            const int e = m.list[ci];
            const int t0 = e & 0xFFFF, g = e >> 16;
            nt = min(kGvTok, gu.counts[g] - t0);
            if (nt > f.tok_rows) {  // more rows in a group than the batch has tokens
                if (threadIdx.x == 0) set_status(gu.status, MOE_DEV_ROWS_OVERFLOW);
                nt = f.tok_rows;
            }
            row0 = (int64_t)gu.offsets[g] + t0;
            gv_consumer_sync();  // the previous chunk's readers of sx and the scales are done
            if (!isg) {
                // the chunk's intermediate rows: all NBg gate_up tiles (all their S parts)
                if (threadIdx.x == 0 && !*m.abort_flag &&
                    !gv_wait_count(f.ready + ci, NBg * S, m.abort_flag)) {
                    set_status(dn.status, MOE_DEV_WAIT_TIMEOUT);
                    *m.abort_flag = 1;
                }
                gv_consumer_sync();
                if (*m.abort_flag) ok = false;
                if (S == 1) {
                    gv_stage_chunk<false, kGvSrcRowsL2>(dn, m, gu.out_bf16, row0, nt, g, dn.K,
                                                        KBd, pd);
                } else {
                    uint16_t* rows = reinterpret_cast<uint16_t*>(m.red);
                    gv_split_rows(f.part, ci, NBg, S, nt, dn.K,
                                  __frcp_rn(__fmul_rn(gs, gu.gs_w[g])), rows);
                    gv_consumer_sync();
                    gv_stage_chunk<false, kGvSrcSmem>(dn, m, rows, row0, nt, g, dn.K, KBd, pd);
                }
            } else {
                gv_stage_chunk<true, kGvSrcTokens>(gu, m, f.x, row0, nt, g, gu.K, KBg, pg, f.T,
                                                   f.k, gs);
            }
            staged = key;
        } else {
            gv_consumer_sync();  // the previous item's readers of red are done
        }
        float d[2][2][4] = {};
        const int nkb = isg ? nkg : KBd;
        const uint8_t* xs = m.sx + xr * (isg ? pg : pd) + 2 * (64 * my_ks + 16 * c4) +
                            512 * (isg ? s * nkg : 0);
        for (int kb = 0; kb < nkb; ++kb) {
            if (ok && !gv_all_wait(&m.full[sl], ph, m.abort_flag)) {
                ok = false;
                if (lane == 0) {
                    set_status(gu.status, MOE_DEV_WAIT_TIMEOUT);
                    *m.abort_flag = 1;
                }
            }
            if (ok) {
                GvFrag fr;
                gv_load(fr, m.ring + (size_t)sl * kNvf4TileBytes, 32 * my_u, my_ks, lane);
                gv_kstep(fr, xs + 512 * kb, lane, d);
                __syncwarp();
                if (lane == 0) mbar_arrive(&m.empty[sl]);
            }
            if (++sl == slots) {
                sl = 0;
                ph ^= 1u;
            }
        }
#pragma unroll
        for (int mb = 0; mb < 2; ++mb)
#pragma unroll
            for (int r = 0; r < 4; ++r) d[0][mb][r] += d[1][mb][r];
        float* redb = m.red;
        float* rw = redb + warp * 32 * kGvTok;
#pragma unroll
        for (int mb = 0; mb < 2; ++mb)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh)
                *reinterpret_cast<float2*>(rw + (16 * mb + 8 * hh + g8) * kGvTok + 2 * c4) =
                    make_float2(d[0][mb][2 * hh], d[0][mb][2 * hh + 1]);
        gv_consumer_sync();
        if (!isg) {
            if (ok) gv_epilogue<false>(dn, m, redb, row0, nt, nb);
        } else if (S == 1) {
            if (ok) gv_epilogue<true>(gu, m, redb, row0, nt, nb);
            gv_item_done(m, it);
        } else {
            // this part's sums over its k range -> part[tile][s][token][row]; the down stagers
            // of the chunk add the parts
            float* mine = f.part + ((size_t)(ci * NBg + nb) * S + s) * (128 * kGvTok);
            for (int o = threadIdx.x; o < 128 * nt; o += kGvConsumers * 32) {
                const int t = o / 128, row = o % 128, u = row / 32, ri = row % 32;
                float v = 0.0f;
#pragma unroll
                for (int q = 0; q < kGvKsteps; ++q)
                    v += redb[((q * kGvUnits + u) * 32 + ri) * kGvTok + t];
                mine[o] = v;
            }
            gv_item_done(m, it);
        }
    }
}

size_t gemv_w4a16_fused_smem(int H, int tok_rows, int slots, int list_cap)
{
    return (size_t)slots * kNvf4TileBytes + gv_fused_fixed_bytes(H, tok_rows) +
           4 * (size_t)list_cap;
}

// At most 6 blobs in flight per block: with one token (where shared memory would allow 12)
// the deeper ring was slower (46.6 vs 45.2 us a forward; 8 tokens: 123.5 vs 123.1 us), as
// its first burst of requests delays every block's first blob; 32 and 256 tokens, where at
// most 7-8 fit, ran the same at 6.
constexpr int kGvFusedMaxSlots = 6;

int gemv_w4a16_fused_slots(int H, int tok_rows, int list_cap)
{
    const size_t fixed = gv_fused_fixed_bytes(H, tok_rows) + 4 * (size_t)list_cap;
    if (fixed >= (size_t)kSmemLimit) return 0;
    return (int)std::min<size_t>(kGvFusedMaxSlots, ((size_t)kSmemLimit - fixed) / kNvf4TileBytes);
}

FusedGemvKernel gemv_w4a16_fused_kernel_ptr() { return gemv_w4a16_fused_kernel; }

GemvKernel gemv_w4a16_kernel_for(bool gateup)
{
    return gateup ? gemv_w4a16_kernel<true> : gemv_w4a16_kernel<false>;
}

}  // namespace moe
