// NVFP4 quantisation (activations, standalone matrices, SwiGLU requantisation), the
// weighted combine, and the create-time weight re-layout.
//
// NVFP4 (Solar Open 2 on DGX Spark, "b12x 버전이 실제 NVFP4 체크포인트를 읽어들이도록
// 만들기": packed FP4 values, FP8 block scales clamped at 448, an FP32 global scale):
// E2M1 codes, one E4M3 scale per 16 consecutive elements, value = code * scale / gs.
#include <cuda_bf16.h>

#include <cuda_fp16.h>

#include "kernels.cuh"

namespace moe {

// ---------------------------------------------------------------- amax
// amax over n bf16 values, merged into *amax_bits with an integer max (non-negative
// floats order like their bit patterns).
__global__ void __launch_bounds__(256) amax_bf16_kernel(const uint16_t* __restrict__ x,
                                                        int64_t n, uint32_t* amax_bits)
{
    pdl_wait();
    if (threadIdx.x == 0) pdl_trigger();
    float m = 0.0f;
    const int64_t n8 = n / 8;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n8;
         i += (int64_t)gridDim.x * blockDim.x) {
        const uint4 v = reinterpret_cast<const uint4*>(x)[i];
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            m = fmaxf(m, fabsf(bf16_bits_to_f32(u[j] & 0xFFFFu)));
            m = fmaxf(m, fabsf(bf16_bits_to_f32(u[j] >> 16)));
        }
    }
    for (int64_t i = n8 * 8 + blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x)
        m = fmaxf(m, fabsf(bf16_bits_to_f32(x[i])));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    __shared__ float s[32];
    if ((threadIdx.x & 31) == 0) s[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x < 32) {
        m = threadIdx.x < (blockDim.x >> 5) ? s[threadIdx.x] : 0.0f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (threadIdx.x == 0) atomicMax(amax_bits, __float_as_uint(m));
    }
}

// Global encode scale: the static one if given, else 2688 / amax (1 when amax == 0).
__device__ __forceinline__ float global_scale(const float* gs_static, const uint32_t* amax_bits)
{
    if (gs_static) return *gs_static;
    const float a = __uint_as_float(*amax_bits);
    return a == 0.0f ? 1.0f : __fdiv_rn(2688.0f, a);
}

// Loads 16 bf16 values (32 bytes) as fp32.
__device__ __forceinline__ void load16_bf16(const uint16_t* p, float* v)
{
    const uint4 a = reinterpret_cast<const uint4*>(p)[0];
    const uint4 b = reinterpret_cast<const uint4*>(p)[1];
    const uint32_t u[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        v[2 * i] = bf16_bits_to_f32(u[i] & 0xFFFFu);
        v[2 * i + 1] = bf16_bits_to_f32(u[i] >> 16);
    }
}

// ---------------------------------------------------------------- gather-quantise
//
// Each warp handles 32 consecutive lanes' worth of one token: with BPL = 1 a lane per
// 16-element block (the 4 blocks of one 64-element k-step sit on 4 neighbouring lanes and
// their scale bytes are merged into one 32-bit atom word), with BPL = 4 a lane per k-step
// (its own scale word).  Code stores from a warp are contiguous.  Destinations: the padded
// rows of the token's local pairs (inv), then its shared row, read eight at a time.

template <int BPL>
__global__ void __launch_bounds__(256) gather_quant_kernel(
    const uint16_t* __restrict__ x, int T, int H, int k, const int32_t* __restrict__ inv,
    const int32_t* __restrict__ offsets, int shared_group, int add_shared,
    const float* gs_static, const uint32_t* amax_bits, uint8_t* __restrict__ codes,
    uint8_t* __restrict__ sf, float* gs_out, int64_t rows_cap, uint32_t* status)
{
    const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const int nb = H / 16;
    const int wpt = (nb + 32 * BPL - 1) / (32 * BPL);  // warps per token
    const bool live = gw < T * wpt;
    const int t = live ? gw / wpt : 0, chunk = live ? gw % wpt : 0;
    const int b = (chunk * 32 + lane) * BPL;  // this lane's first 16-element block
    const bool act = live && b < nb;  // nb % 4 == 0: the lanes of one k-step agree
    const int nrows = k + (add_shared ? 1 : 0);  // pairs in top-k order, then the shared row
    // destinations eight at a time (-1: a pair outside this shard)
    auto rows_of = [&](int j0, int64_t* row) {
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int j = j0 + u;
            row[u] = !act || j >= nrows ? -1
                     : checked_row(j < k ? (int64_t)inv[(size_t)t * k + j]
                                         : (int64_t)offsets[shared_group] + t,
                                   rows_cap, status);
        }
    };
    // the layer input is complete before the forward starts: its load goes out before the
    // wait; the destinations and the activation scale come from the preceding launches
    float v[16 * BPL];
    if (act)
#pragma unroll
        for (int i = 0; i < BPL; ++i) load16_bf16(x + (size_t)t * H + (b + i) * 16, v + 16 * i);
    pdl_wait();
    if (threadIdx.x == 0) pdl_trigger();
    if (!live) return;
    int64_t row[8];
    rows_of(0, row);
    const float gs = global_scale(gs_static, amax_bits);
    if (gw == 0 && lane == 0 && gs_out) *gs_out = gs;
    const int pitch = codes_pitch(H);
    uint32_t c[2 * BPL], word = 0u;
    if (BPL == 4) {  // a whole 64-element k-step per lane: its own scale word
        if (act)
#pragma unroll
            for (int i = 0; i < 4; ++i) word |= quant16(v + 16 * i, gs, c + 2 * i) << (8 * i);
    } else {  // merge the 4 scale bytes of a k-step into the lane with b % 4 == 0
        uint32_t sc = 0u;
        c[0] = c[1] = 0u;
        if (act) sc = quant16(v, gs, c);
        const uint32_t s1 = __shfl_down_sync(0xffffffffu, sc, 1);
        const uint32_t s2 = __shfl_down_sync(0xffffffffu, sc, 2);
        const uint32_t s3 = __shfl_down_sync(0xffffffffu, sc, 3);
        word = sc | (s1 << 8) | (s2 << 16) | (s3 << 24);
    }
    if (!act) return;
    for (int j0 = 0; j0 < nrows; j0 += 8) {
        if (j0) rows_of(j0, row);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            if (row[u] < 0) continue;
            uint8_t* dst = codes + row[u] * pitch + b * 8;
            if (BPL == 4) {
                reinterpret_cast<uint4*>(dst)[0] = make_uint4(c[0], c[1], c[2], c[3]);
                reinterpret_cast<uint4*>(dst)[1] = make_uint4(c[4], c[5], c[6], c[7]);
            } else {
                *reinterpret_cast<uint2*>(dst) = make_uint2(c[0], c[1]);
            }
            if ((b & 3) == 0)
                *reinterpret_cast<uint32_t*>(sf + sf_atom_offset(row[u], b, H)) = word;
        }
    }
}

GatherKernel gather_quant_kernel_for(int blocks_per_lane)
{
    return blocks_per_lane == 4 ? gather_quant_kernel<4> : gather_quant_kernel<1>;
}

// W4A16: copy token rows (bf16) times the prescale (f16_prescale), as fp16, to the padded
// rows of their pairs and shared row; a warp copies 256 elements of one token.
__global__ void __launch_bounds__(256) gather_f16_kernel(
    const uint16_t* __restrict__ x, int T, int H, int k, const int32_t* __restrict__ inv,
    const int32_t* __restrict__ offsets, int shared_group, int add_shared,
    const uint32_t* amax_bits, uint16_t* __restrict__ out, float* gs_out, int64_t rows_cap,
    uint32_t* status)
{
    const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const int wpt = (H + 255) / 256;
    const bool live = gw < T * wpt;
    const int t = live ? gw / wpt : 0, c = live ? (gw % wpt) * 256 + lane * 8 : 0;
    const bool act = live && c < H;
    // the layer input is complete before the forward starts: its load goes out before the
    // wait; the destinations and the prescale come from the preceding launches
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (act) v = *reinterpret_cast<const uint4*>(x + (size_t)t * H + c);
    pdl_wait();
    if (threadIdx.x == 0) pdl_trigger();
    const float gs = f16_prescale(amax_bits);
    if (blockIdx.x == 0 && threadIdx.x == 0 && gs_out) *gs_out = gs;
    if (!act) return;
    const uint32_t in[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __half2 h = __floats2half2_rn(__fmul_rn(bf16_bits_to_f32(in[i] & 0xFFFFu), gs),
                                            __fmul_rn(bf16_bits_to_f32(in[i] >> 16), gs));
        o[i] = *reinterpret_cast<const uint32_t*>(&h);
    }
    const int nrows = k + (add_shared ? 1 : 0);  // pairs in top-k order, then the shared row
    for (int j0 = 0; j0 < nrows; j0 += 8) {
        int64_t row[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int j = j0 + u;
            row[u] = j >= nrows ? -1
                     : checked_row(j < k ? (int64_t)inv[(size_t)t * k + j]
                                         : (int64_t)offsets[shared_group] + t,
                                   rows_cap, status);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u)
            if (row[u] >= 0)
                *reinterpret_cast<uint4*>(out + row[u] * H + c) = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

// ---------------------------------------------------------------- standalone quantiser
// rows x cols bf16 -> NVFP4; layout 0 canonical, 1 tiled.  One warp per row.
__global__ void __launch_bounds__(256) quant_rows_kernel(
    const uint16_t* __restrict__ x, int rows, int cols, const float* gs_static,
    const uint32_t* amax_bits, uint8_t* __restrict__ codes, uint8_t* __restrict__ sf,
    int layout, float* gs_out)
{
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (warp >= rows) return;
    const float gs = global_scale(gs_static, amax_bits);
    if (warp == 0 && lane == 0 && gs_out) *gs_out = gs;
    const int64_t r = warp;
    const int nb = cols / 16;
    const int pitch = layout ? codes_pitch(cols) : cols / 2;
    for (int b = lane; b < nb; b += 32) {
        float v[16];
        load16_bf16(x + r * cols + b * 16, v);
        uint32_t c[2];
        const uint32_t s = quant16(v, gs, c);
        *reinterpret_cast<uint2*>(codes + r * pitch + b * 8) = make_uint2(c[0], c[1]);
        if (layout) sf[sf_atom_offset(r, b, cols)] = (uint8_t)s;
        else sf[r * nb + b] = (uint8_t)s;
    }
}

// ---------------------------------------------------------------- SwiGLU + requant
// fp32 gate/up rows [rows][2I] (gate cols 0..I-1) -> s = silu(g) * u -> NVFP4 with gs_i.
__global__ void __launch_bounds__(256) swiglu_requant_kernel(
    const float* __restrict__ gu, int rows, int I, float gs_i, uint8_t* __restrict__ codes,
    uint8_t* __restrict__ sf, int layout)
{
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (warp >= rows) return;
    const int64_t r = warp;
    const int nb = I / 16;
    const int pitch = layout ? codes_pitch(I) : I / 2;
    for (int b = lane; b < nb; b += 32) {
        float v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
            v[i] = silu_mul(gu[r * 2 * I + b * 16 + i], gu[r * 2 * I + I + b * 16 + i]);
        uint32_t c[2];
        const uint32_t s = quant16(v, gs_i, c);
        *reinterpret_cast<uint2*>(codes + r * pitch + b * 8) = make_uint2(c[0], c[1]);
        if (layout) sf[sf_atom_offset(r, b, I)] = (uint8_t)s;
        else sf[r * nb + b] = (uint8_t)s;
    }
}

// ---------------------------------------------------------------- dynamic intermediate scale
// Second pass of the dynamic intermediate scale: the fp32 intermediate s [rows][I] of the
// gate_up epilogue (padded rows), NVFP4-quantised with gs_i = 2688 / amax |s| (amax from
// the first pass; 1 if 0) into the tiled codes / scale atoms the down GEMM reads.  Block b
// takes 128-row block b of the padded layout (mb_start maps it to its group); only the
// group's valid rows are written.  Block 0 stores gs_i.
__global__ void __launch_bounds__(256) quant_inter_kernel(
    const float* __restrict__ s, const int32_t* __restrict__ counts,
    const int32_t* __restrict__ offsets, const int32_t* __restrict__ mb_start, int G, int I,
    const uint32_t* amax_bits, uint8_t* __restrict__ codes, uint8_t* __restrict__ sf,
    float* gs_out)
{
    pdl_wait();
    if (threadIdx.x == 0) pdl_trigger();
    const float gs = global_scale(nullptr, amax_bits);
    if (blockIdx.x == 0 && threadIdx.x == 0) *gs_out = gs;
    const int b = blockIdx.x;
    if (b >= mb_start[G]) return;
    int lo = 0, hi = G;  // group of block b: last g with mb_start[g] <= b
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (mb_start[mid] <= b) lo = mid;
        else hi = mid;
    }
    const int blk = b - mb_start[lo];
    const int nrows = min(128, counts[lo] - 128 * blk);
    const int64_t row0 = offsets[lo] + 128 * blk;
    const int nb = I / 16, pitch = codes_pitch(I);
    for (int i = threadIdx.x; i < nrows * nb; i += blockDim.x) {
        const int64_t r = row0 + i / nb;
        const int q = i % nb;
        const float4* src = reinterpret_cast<const float4*>(s + r * I + q * 16);
        float v[16];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float4 f = src[j];
            v[4 * j] = f.x;
            v[4 * j + 1] = f.y;
            v[4 * j + 2] = f.z;
            v[4 * j + 3] = f.w;
        }
        uint32_t c[2];
        const uint32_t sb = quant16(v, gs, c);
        *reinterpret_cast<uint2*>(codes + r * pitch + q * 8) = make_uint2(c[0], c[1]);
        sf[sf_atom_offset(r, q, I)] = (uint8_t)sb;
    }
}

// ---------------------------------------------------------------- combine
// out[t][h] = sum_{j: inv >= 0} y[inv[t*k+j]][h] + (add_shared ? y[offsets[G_s] + t][h] : 0)
// in ascending j then the shared row, fp32, rounded to bf16.  y rows are padded rows (already
// multiplied by their routing weight).  One thread per 8 columns of one token.
// Eight fp16 (one 16-byte piece) -> fp32, exactly.
__device__ __forceinline__ void f16x8_to_f32(uint4 q, float (&f)[8])
{
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 p = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
        f[2 * i] = p.x;
        f[2 * i + 1] = p.y;
    }
}

__global__ void __launch_bounds__(256) combine_kernel(const void* __restrict__ y,
                                                      const float* __restrict__ y_scale,
                                                      const int32_t* __restrict__ inv,
                                                      const int32_t* __restrict__ offsets,
                                                      int shared_group, int T, int H, int k,
                                                      int add_shared, uint16_t* __restrict__ out,
                                                      int64_t rows_cap, uint32_t* status)
{
    const bool f16 = y_scale != nullptr;  // fp16 rows, each times y_scale[row]
    const int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    const int per = H / 8;
    const bool live = i < (int64_t)T * per;
    const int t = live ? (int)(i / per) : 0, c = live ? (int)(i % per) * 8 : 0;
    const int nrows = k + (add_shared ? 1 : 0);  // pairs in top-k order, then the shared row
    // rows of eight pairs at a time: their indices, then all their y loads, then the sums
    // in order (row -1: a pair outside this shard)
    auto rows_of = [&](int j0, int64_t* row) {
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int j = j0 + u;
            row[u] = !live || j >= nrows ? -1
                     : checked_row(j < k ? (int64_t)inv[(size_t)t * k + j]
                                         : (int64_t)offsets[shared_group] + t,
                                   rows_cap, status);
        }
    };
    int64_t row[8];
    rows_of(0, row);  // inv and offsets were complete before the predecessor started
    pdl_wait();
    if (threadIdx.x == 0) pdl_trigger();
    if (!live) return;
    float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    for (int j0 = 0; j0 < nrows; j0 += 8) {
        if (j0) rows_of(j0, row);
        float4 v[8][2];
        uint4 h[8];
        float sc[8];
#pragma unroll
        for (int u = 0; u < 8; ++u)
            if (row[u] >= 0) {
                if (f16) {
                    h[u] = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(y) +
                                                           row[u] * H + c);
                    sc[u] = y_scale[row[u]];
                } else {
                    const float4* src =
                        reinterpret_cast<const float4*>(static_cast<const float*>(y) + row[u] * H + c);
                    v[u][0] = src[0];
                    v[u][1] = src[1];
                }
            }
        if (f16)
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (row[u] >= 0) {
                    float f[8];
                    f16x8_to_f32(h[u], f);
                    v[u][0] = make_float4(f[0] * sc[u], f[1] * sc[u], f[2] * sc[u], f[3] * sc[u]);
                    v[u][1] = make_float4(f[4] * sc[u], f[5] * sc[u], f[6] * sc[u], f[7] * sc[u]);
                }
#pragma unroll
        for (int u = 0; u < 8; ++u)
            if (row[u] >= 0) {
                acc[0] += v[u][0].x; acc[1] += v[u][0].y; acc[2] += v[u][0].z; acc[3] += v[u][0].w;
                acc[4] += v[u][1].x; acc[5] += v[u][1].y; acc[6] += v[u][1].z; acc[7] += v[u][1].w;
            }
    }
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const __nv_bfloat162 p = __floats2bfloat162_rn(acc[2 * q], acc[2 * q + 1]);
        o[q] = *reinterpret_cast<const uint32_t*>(&p);
    }
    *reinterpret_cast<uint4*>(out + (size_t)t * H + c) = make_uint4(o[0], o[1], o[2], o[3]);
}

// The same combine for large batches, with the y rows moved by bulk copies: a work unit is
// one token and one cw-column piece; thread 0 of warp 0 copies the piece of each of the
// token's rows (pairs in top-k order, then its shared row; a pair outside the shard has none)
// into a ring slot of shared memory, and warps 1-16 add them in that order (the sums of
// combine_kernel, bit for bit), round to bf16 and store.  Every wait is bounded; a wait that
// runs out sets MOE_DEV_WAIT_TIMEOUT (when a status word is given) and ends the CTA's work.
__device__ __forceinline__ bool cmb_warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort)
{
    int ok = 1;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, abort) ? 1 : 0;
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

__global__ void __launch_bounds__(kCombineTmaThreads, 1) combine_tma_kernel(
    const void* __restrict__ y, const float* __restrict__ y_scale,
    const int32_t* __restrict__ inv, const int32_t* __restrict__ offsets, int shared_group,
    int T, int H, int k, int add_shared, int cw, int nslots, uint16_t* __restrict__ out,
    uint32_t* status, int64_t rows_cap)
{
    extern __shared__ __align__(128) uint8_t smem_cmb[];
    const bool f16 = y_scale != nullptr;  // fp16 rows, each times y_scale[row]
    const uint32_t es = f16 ? 2u : 4u;     // bytes per element
    const int nrows = k + (add_shared ? 1 : 0);
    const size_t slot_bytes = (size_t)nrows * cw * es;
    uint8_t* slots = smem_cmb;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem_cmb + nslots * slot_bytes);
    uint64_t* empty = full + kCombineMaxSlots;
    uint64_t* masks = empty + kCombineMaxSlots;  // valid rows of each slot's unit
    volatile int* abort_flag = reinterpret_cast<volatile int*>(masks + kCombineMaxSlots);
    int* zero = const_cast<int*>(reinterpret_cast<volatile int*>(abort_flag + 1));
    // [slot][row]: the fp16 rows' scales, after the two flag words (16 bytes)
    float* rsc = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(masks + kCombineMaxSlots) + 16);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < nslots; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kCombineTmaThreads / 32 - 1);  // one arrival per consumer warp
        }
        *abort_flag = 0;
        *zero = 0;
        fence_barrier_init();
    }
    __syncthreads();
    const int nchunk = H / cw;
    const int64_t nunits = (int64_t)T * nchunk;
    if (warp == 0) {
        // the copy warp: lane j looks up rows j and j + 32 of a unit (its index, then its
        // fp16 scale), so a unit's lookups take two load latencies; lane 0 issues the copies
        const uint64_t pol = policy_evict_first();
        pdl_wait();  // y and its scales are the predecessor's output
        pdl_trigger();
        uint32_t issued = 0, issued_par = 0;
        bool ok = true;
        int i = 0;
        int64_t row[2] = {-1, -1};  // rows lane and lane + 32 of the next unit (-1: none)
        float scl[2] = {1.0f, 1.0f};
        auto rows_of = [&](int64_t uu) {
            const int tt = (int)(uu / nchunk);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int j = lane + 32 * h;
                row[h] = j >= nrows ? -1
                         : checked_row(j < k ? (int64_t)inv[(size_t)tt * k + j]
                                             : (int64_t)offsets[shared_group] + tt,
                                       rows_cap, status);
            }
            if (f16)
#pragma unroll
                for (int h = 0; h < 2; ++h)
                    if (row[h] >= 0) scl[h] = y_scale[row[h]];
        };
        if (blockIdx.x < nunits) rows_of(blockIdx.x);
        for (int64_t u = blockIdx.x; u < nunits && ok; u += gridDim.x, ++i) {
            const int sl = i % nslots;
            const uint32_t ph = (uint32_t)(i / nslots) & 1u;
            int okw = 1;
            if (lane == 0) okw = mbar_wait(&empty[sl], ph ^ 1u, abort_flag) ? 1 : 0;
            if (!__shfl_sync(0xffffffffu, okw, 0)) {
                ok = false;
                break;
            }
            const int c0 = (int)(u % nchunk) * cw;
            // the unit's valid rows (a ballot per half) and their bytes; scales to the slot
            const uint64_t mask = (uint64_t)__ballot_sync(0xffffffffu, row[0] >= 0) |
                                  ((uint64_t)__ballot_sync(0xffffffffu, row[1] >= 0) << 32);
            if (f16) {
#pragma unroll
                for (int h = 0; h < 2; ++h)
                    if (row[h] >= 0) rsc[sl * (kMaxTopK + 1) + lane + 32 * h] = scl[h];
            }
            __syncwarp();
            if (lane == 0) {
                masks[sl] = mask;
                mbar_arrive_expect_tx(&full[sl], (uint32_t)__popcll(mask) * (uint32_t)cw * es);
            }
            uint8_t* dst = slots + (size_t)sl * slot_bytes;
            for (int j = 0; j < nrows; ++j) {
                const int64_t r = __shfl_sync(0xffffffffu, row[j >> 5], j & 31);
                if (lane == 0 && r >= 0)
                    bulk_load(dst + (size_t)j * cw * es,
                              static_cast<const uint8_t*>(y) + ((size_t)r * H + c0) * es,
                              (uint32_t)cw * es, &full[sl], pol);
            }
            issued |= 1u << sl;
            issued_par = (issued_par & ~(1u << sl)) | (ph << sl);
            if (u + gridDim.x < nunits) rows_of(u + gridDim.x);
        }
        if (lane == 0) {
            if (!ok) {
                set_status(status, MOE_DEV_WAIT_TIMEOUT);
                *abort_flag = 1;
            }
            for (int sl = 0; sl < nslots; ++sl)  // copies in flight land before the CTA exits
                if ((issued >> sl) & 1u) mbar_wait(&full[sl], (issued_par >> sl) & 1u, zero);
        }
    } else {
        // four columns per thread and segment of 4 x (consumer threads) columns
        const int tid = threadIdx.x - 32, seg = 4 * (kCombineTmaThreads - 32);
        int i = 0;
        for (int64_t u = blockIdx.x; u < nunits; u += gridDim.x, ++i) {
            const int sl = i % nslots;
            const uint32_t ph = (uint32_t)(i / nslots) & 1u;
            if (!cmb_warp_wait(&full[sl], ph, abort_flag)) {
                if (lane == 0) {
                    set_status(status, MOE_DEV_WAIT_TIMEOUT);
                    *abort_flag = 1;
                }
                break;
            }
            const uint64_t mask = masks[sl];
            const int t = (int)(u / nchunk), c0 = (int)(u % nchunk) * cw;
            const uint8_t* src = slots + (size_t)sl * slot_bytes;
            const float* sc = rsc + sl * (kMaxTopK + 1);
            for (int col = 4 * tid; col < cw; col += seg) {
                float a0 = 0.0f, a1 = 0.0f, a2 = 0.0f, a3 = 0.0f;
                for (int j = 0; j < nrows; ++j)
                    if ((mask >> j) & 1ull) {
                        float4 v;
                        if (f16) {
                            const uint2 hq = *reinterpret_cast<const uint2*>(
                                src + ((size_t)j * cw + col) * 2);
                            const float2 lo = __half22float2(*reinterpret_cast<const __half2*>(&hq.x));
                            const float2 hi = __half22float2(*reinterpret_cast<const __half2*>(&hq.y));
                            const float s = sc[j];
                            v = make_float4(lo.x * s, lo.y * s, hi.x * s, hi.y * s);
                        } else {
                            v = *reinterpret_cast<const float4*>(src + ((size_t)j * cw + col) * 4);
                        }
                        a0 += v.x;
                        a1 += v.y;
                        a2 += v.z;
                        a3 += v.w;
                    }
                const __nv_bfloat162 p0 = __floats2bfloat162_rn(a0, a1);
                const __nv_bfloat162 p1 = __floats2bfloat162_rn(a2, a3);
                *reinterpret_cast<uint2*>(out + (size_t)t * H + c0 + col) =
                    make_uint2(*reinterpret_cast<const uint32_t*>(&p0),
                               *reinterpret_cast<const uint32_t*>(&p1));
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[sl]);
        }
    }
}

// ---------------------------------------------------------------- checkpoint weights
// One matrix type of a checkpoint (codes [E][N][K/2], E4M3 scales [E][N][K/16], a global
// value per expert) -> the library's convention for experts off..off+count-1: global given
// as the encode scale (convention 0) or as a dequantisation multiplier m (1: gs = 1/m);
// fold_target > 0 folds each expert's global into its block scales relative to that
// common scale (r = gs_t / gs, sf' = E4M3(sf * r), nearest even, saturating at 448) and
// gives every expert gs_t; swap_halves puts rows N/2..N-1 first.  Codes are copied.
// A warp per output row: the row's codes in 16-byte pieces, its scales 4 bytes a lane.
__device__ __forceinline__ uint32_t fold_scale_byte(uint32_t v, float r)
{
    const float sv = e4m3_to_f32(v & 0x7Fu);  // the sign bit, if set, is kept
    return f32_to_e4m3(__fmul_rn((v & 0x80u) ? -sv : sv, r));
}

__global__ void __launch_bounds__(256) prepare_weights_kernel(
    const uint8_t* __restrict__ codes, const uint8_t* __restrict__ sf,
    const float* __restrict__ glob, int N, int K, int convention, float fold_target,
    int swap_halves, int off, int count, uint8_t* __restrict__ codes_out,
    uint8_t* __restrict__ sf_out, float* __restrict__ gs_out)
{
    const int lane = threadIdx.x & 31;
    const int64_t rows = (int64_t)count * N;
    const int cpr = K / 32, spr = K / 64;  // 16-byte code pieces, 4-byte scale words per row
    const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t row = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5; row < rows;
         row += nwarps) {
        const int64_t e = row / N;
        const int n = (int)(row - e * N);
        const int sn = swap_halves ? (n + N / 2) % N : n;
        const int64_t src = (off + e) * N + sn;
        const uint4* cs = reinterpret_cast<const uint4*>(codes) + src * cpr;
        uint4* cd = reinterpret_cast<uint4*>(codes_out) + row * cpr;
        for (int i = lane; i < cpr; i += 32) cd[i] = cs[i];
        const float g = glob[off + e];
        const float gs = convention == 1 ? __fdiv_rn(1.0f, g) : g;
        const uint32_t* ss = reinterpret_cast<const uint32_t*>(sf + src * (K / 16));
        uint32_t* sd = reinterpret_cast<uint32_t*>(sf_out + row * (K / 16));
        if (fold_target > 0.0f) {
            const float r = __fdiv_rn(fold_target, gs);
            for (int i = lane; i < spr; i += 32) {
                const uint32_t w = ss[i];
                sd[i] = fold_scale_byte(w & 0xFFu, r) | (fold_scale_byte((w >> 8) & 0xFFu, r) << 8) |
                        (fold_scale_byte((w >> 16) & 0xFFu, r) << 16) |
                        (fold_scale_byte(w >> 24, r) << 24);
            }
        } else {
            for (int i = lane; i < spr; i += 32) sd[i] = ss[i];
        }
        if (n == 0 && lane == 0) gs_out[e] = fold_target > 0.0f ? fold_target : gs;
    }
}

// ---------------------------------------------------------------- weight re-layout
//
// Canonical codes [nexp][N][K/2] and scales [nexp][N][K/16] -> one contiguous blob per
// (expert, 128-row tile nb, 256-element k-stage kb), the bytes a GEMM stage copies into
// shared memory: 128 rows x 128 code bytes in the 128-byte swizzled layout (byte c of row r
// at r*128 + ((c/16) ^ (r%8))*16 + c%16), then the 4 scale atoms of k-steps 4kb..4kb+3.
// With nibble_pairs (the W4A16 blobs) the 8 codes of each 32-bit word are stored in the
// nibble order 0,2,4,6,1,3,5,7 instead of 0..7.
// Scale atom byte (m%32)*16 + (m/32)*4 + kk holds scale kk of the k-step for tile row m.
// Bytes past K (a partial last stage) are zero.  With interleave (the gate/up matrix,
// N = 2I), tile row 128*nb + 32*c + 16*u + i holds source row u*I + 64*nb + 16*c + i, so
// each 128-row tile has 4 pairs of 16 gate rows and the 16 matching up rows -- the fused
// epilogue sees gate and up of the same features.
__device__ __forceinline__ int64_t src_row(int64_t r, int N, int interleave)
{
    if (!interleave) return r;
    const int I = N / 2;
    const int nb = (int)(r >> 7), c = (int)((r >> 5) & 3), u = (int)((r >> 4) & 1),
              i = (int)(r & 15);
    return (int64_t)u * I + 64 * nb + 16 * c + i;
}

__global__ void __launch_bounds__(256) repack_tiles_kernel(const uint8_t* __restrict__ codes,
                                                           const uint8_t* __restrict__ sf,
                                                           int nexp, int N, int K,
                                                           int interleave, int nibble_pairs,
                                                           uint8_t* __restrict__ dst)
{
    const int KB = (K + 255) / 256, NB = N / 128;
    const int64_t total = (int64_t)nexp * NB * KB * kNvf4TileBytes;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t blob = i / kNvf4TileBytes;
        const int o = (int)(i % kNvf4TileBytes);
        const int kb = (int)(blob % KB);
        const int64_t en = blob / KB;
        const int nb = (int)(en % NB);
        const int64_t e = en / NB;
        uint8_t v = 0;
        if (o < 16384) {
            const int r = o >> 7;
            const int c = ((((o >> 4) & 7) ^ (r & 7)) << 4) | (o & 15);  // byte of the row
            const uint8_t* row =
                codes + (e * N + src_row(nb * 128 + r, N, interleave)) * (int64_t)(K / 2);
            const int kbyte = kb * 128 + c;
            if (!nibble_pairs) {
                if (kbyte < K / 2) v = row[kbyte];
            } else if (kbyte < K / 2) {
                // byte b of a word holds nibbles 2b, 2b + 1; nibble n holds element
                // n < 4 ? 2n : 2(n - 4) + 1 of the word's eight
                const int b = c & 3, w0 = kbyte - b;  // first byte of the word
                const int n0 = 2 * b, n1 = 2 * b + 1;
                const int e0 = n0 < 4 ? 2 * n0 : 2 * (n0 - 4) + 1;
                const int e1 = n1 < 4 ? 2 * n1 : 2 * (n1 - 4) + 1;
                const uint32_t lo = (row[w0 + (e0 >> 1)] >> (4 * (e0 & 1))) & 15u;
                const uint32_t hi = (row[w0 + (e1 >> 1)] >> (4 * (e1 & 1))) & 15u;
                v = (uint8_t)(lo | (hi << 4));
            }
        } else {
            const int a = (o - 16384) / 512, w = (o - 16384) % 512;
            const int m = (w >> 4) + 32 * ((w & 15) >> 2), kk = w & 3;
            const int step = kb * 4 + a;
            if (step < K / 64)
                v = sf[(e * N + src_row(nb * 128 + m, N, interleave)) * (K / 16) + step * 4 + kk];
        }
        dst[i] = v;
    }
}

}  // namespace moe
