// Kernel declarations shared by the translation units of the library.
#pragma once

#include "common.cuh"

namespace moe {

constexpr int kPairsPerBlock = 1024;   // grouping: pairs per block of the counting sort

// Debug builds (MOE_DEBUG defined) check every padded-row index and pair index that a
// kernel reads from a buffer before using it: a bad one sets MOE_DEV_BAD_INDEX in the status
// word and the access is skipped (never a trap).  Release builds compile the checks away.
#ifdef MOE_DEBUG
constexpr bool kDebugChecks = true;
#else
constexpr bool kDebugChecks = false;
#endif

// A padded row r (-1: none) read from a buffer, against the row capacity.
__device__ __forceinline__ int64_t checked_row(int64_t r, int64_t cap, uint32_t* status)
{
    if (kDebugChecks && (r < -1 || r >= cap)) {
        set_status(status, MOE_DEV_BAD_INDEX);
        return -1;
    }
    return r;
}

// A pair index read from perm_src (>= T*k: a shared row), for a valid row: never negative.
__device__ __forceinline__ bool pair_ok(int pair, uint32_t* status)
{
    if (kDebugChecks && pair < 0) {
        set_status(status, MOE_DEV_BAD_INDEX);
        return false;
    }
    return true;
}

// W4A16 activation rows: x (bf16) times the power of two gs = 2^(141 - exponent field of
// amax(x)), clamped to 2^[-126, 127], rounded to fp16.  amax <= 2^(e - 126) for exponent
// field e, so |x * gs| <= 2^15 < 65504 and every bf16 value x with |x * gs| >= 2^-14 (all but
// values below amax * 2^-29) converts exactly; the GEMM divides by gs in its epilogue.
__device__ __forceinline__ float f16_prescale(const uint32_t* amax_bits)
{
    const uint32_t bits = *amax_bits;
    if (bits == 0u) return 1.0f;
    const int e = (int)((bits >> 23) & 0xFFu);
    const int p = min(127, max(-126, 141 - e));
    return __uint_as_float((uint32_t)(p + 127) << 23);
}

// silu(g) * u in fp32: g / (1 + exp(-g)) * u, each step an IEEE fp32 operation.
__device__ __forceinline__ float silu_mul(float g, float u)
{
    return __fmul_rn(__fdiv_rn(g, __fadd_rn(1.0f, expf(-g))), u);
}

// ---- route.cu
constexpr int kRouterSmem = 4 * (16384 + 160 * 128) + 1024 + 256;
__global__ void router_gemm_kernel(const __grid_constant__ CUtensorMap tmX,
                                   const __grid_constant__ CUtensorMap tmW, int T, int E, int H,
                                   int k_per_split, int bn, float* part, uint32_t* status,
                                   uint32_t* clear0, uint32_t* clear1);
int router_splits(int T, int E, int H, int num_sms);
int router_bn(int T, int E);
// top-k launch shape: 512 threads per block of topk_tokens_per_block(nsplit) tokens,
// topk_smem(nsplit, E) bytes of dynamic shared memory (at most 16 * E floats)
__host__ __device__ int topk_tokens_per_block(int nsplit);
size_t topk_smem(int nsplit, int E);
constexpr int kTopkThreads = 512;
using TopkKernel = void (*)(const float*, int, const float*, int, int, int, int32_t*, float*,
                            float*, uint32_t*, uint32_t*, const uint16_t*, int, uint32_t*,
                            int32_t*, int);
// the top-k kernel instantiated for E experts (E <= kMaxExperts)
TopkKernel topk_kernel_for(int E);
__global__ void perm_hist_kernel(const int32_t* ids, int P, int E, int off, int El,
                                 int32_t* hist, uint32_t* status);
__global__ void perm_scan_kernel(const int32_t* hist, int nblk, int El, int T, int k,
                                 int shared_rows, int rows_cap, int32_t* blkoff,
                                 int32_t* counts, int32_t* offsets, int32_t* mb_start,
                                 int32_t* perm_src, uint32_t* status);
// dynamic shared memory of perm_small_kernel (G groups) and perm_scatter_kernel (El
// experts): the per-warp count table [32][G] uint16
inline int perm_small_smem(int G) { return 32 * G * 2; }
__global__ void perm_small_kernel(const int32_t* ids, int P, int E, int off, int El, int T,
                                  int k, int shared_rows, int rows_cap, int write_padding,
                                  int32_t* counts, int32_t* offsets, int32_t* mb_start,
                                  int32_t* perm_src, int32_t* inv, uint32_t* status);
__global__ void perm_scatter_kernel(const int32_t* ids, int P, int E, int off, int El,
                                    const int32_t* blkoff, const int32_t* offsets,
                                    int rows_cap, int32_t* perm_src, int32_t* inv);

// ---- quant.cu
__global__ void amax_bf16_kernel(const uint16_t* x, int64_t n, uint32_t* amax_bits);
// NVFP4 gather-quantise of the activation rows; blocks_per_lane 1 (a lane per 16-element
// block: more threads, for small batches) or 4 (a lane per 64-element k-step: 1 KB pieces
// per destination row, for large batches).
using GatherKernel = void (*)(const uint16_t*, int, int, int, const int32_t*, const int32_t*,
                              int, int, const float*, const uint32_t*, uint8_t*, uint8_t*,
                              float*, int64_t, uint32_t*);
GatherKernel gather_quant_kernel_for(int blocks_per_lane);
__global__ void gather_f16_kernel(const uint16_t* x, int T, int H, int k, const int32_t* inv,
                                  const int32_t* offsets, int shared_group, int add_shared,
                                  const uint32_t* amax_bits, uint16_t* out, float* gs_out,
                                  int64_t rows_cap, uint32_t* status);
__global__ void quant_rows_kernel(const uint16_t* x, int rows, int cols, const float* gs_static,
                                  const uint32_t* amax_bits, uint8_t* codes, uint8_t* sf,
                                  int layout, float* gs_out);
__global__ void swiglu_requant_kernel(const float* gu, int rows, int I, float gs_i,
                                      uint8_t* codes, uint8_t* sf, int layout);
__global__ void quant_inter_kernel(const float* s, const int32_t* counts, const int32_t* offsets,
                                   const int32_t* mb_start, int G, int I,
                                   const uint32_t* amax_bits, uint8_t* codes, uint8_t* sf,
                                   float* gs_out);
// y: fp32 rows, or (y_scale non-null) fp16 rows to be multiplied by y_scale[row]
__global__ void combine_kernel(const void* y, const float* y_scale, const int32_t* inv,
                               const int32_t* offsets, int shared_group, int T, int H, int k,
                               int add_shared, uint16_t* out, int64_t rows_cap,
                               uint32_t* status);
// Bulk-copy combine for large batches: 544 threads (a copy thread, sixteen adding warps), a
// ring of nslots slots of (k + add_shared) row pieces of cw columns each.
constexpr int kCombineTmaThreads = 544;
constexpr int kCombineMaxSlots = 6;
inline size_t combine_tma_smem(int nrows, int cw, int nslots, int esize = 4)
{
    return (size_t)nslots * nrows * cw * esize + 3 * kCombineMaxSlots * 8 + 16 +
           (size_t)kCombineMaxSlots * (kMaxTopK + 1) * 4;
}
__global__ void combine_tma_kernel(const void* y, const float* y_scale, const int32_t* inv,
                                   const int32_t* offsets, int shared_group, int T, int H, int k,
                                   int add_shared, int cw, int nslots, uint16_t* out,
                                   uint32_t* status, int64_t rows_cap);
__global__ void prepare_weights_kernel(const uint8_t* codes, const uint8_t* sf,
                                       const float* glob, int N, int K, int convention,
                                       float fold_target, int swap_halves, int off, int count,
                                       uint8_t* codes_out, uint8_t* sf_out, float* gs_out);
__global__ void repack_tiles_kernel(const uint8_t* codes, const uint8_t* sf, int nexp, int N,
                                    int K, int interleave, int nibble_pairs, uint8_t* dst);

// ---- gemm.cu
enum GemmEpilogue : int {
    kEpiGateUpF32 = 0,     // G (alpha applied) -> fp32 rows, gate then up columns
    kEpiGateUpSwiglu = 1,  // silu(gate)*up -> NVFP4 (W4A4) or bf16 (W4A16)
    kEpiDown = 2,          // Y * routing weight -> fp32 rows indexed by padded row
    kEpiGateUpSwigluF32 = 3, // silu(gate)*up -> fp32 rows [rows][I], and amax |s| into
                             // inter_amax (first pass of the dynamic intermediate scale)
    kEpiDownF16 = 4          // as kEpiDown, as fp16 rows (out_bf16) of Y x 2^e_g, e_g per group
                             // from a bound on |Y| (kYF16Bound); y_scale[row] = 2^-e_g
};

// |Y| of a W4A4 down row is at most K x 2688^2 x alpha_g (every code x scale factor of the
// intermediate and of W2 is at most 6 x 448 = 2688 in magnitude, the routing weight at most
// 1, alpha_g = 1 / (gs_i gs_w)).  The fp16 form takes Y x 2^e_g with 2^e_g the largest power
// of two that keeps that bound within the fp16 range.
constexpr float kYF16Max = 65504.0f;
constexpr float kE2M1E4M3MaxSq = 2688.0f * 2688.0f;
__host__ __device__ __forceinline__ bool is_down(int epilogue)
{
    return epilogue == kEpiDown || epilogue == kEpiDownF16;
}

struct GemmArgs {
    const uint8_t* a_sf;      // W4A4: activation scale atoms (tiled, K-wide)
    const uint8_t* b_tiles;   // weight blobs [slots][N/128][k-stages][tile bytes]
    const float* gs_a;        // W4A4: activation global scale (device scalar)
    const float* gs_w;        // [slots] weight global scales
    const int32_t* counts;    // [G] rows per group
    const int32_t* offsets;   // [G+1] padded first row per group
    const int32_t* mb_start;  // [G+1] first 128-row block per group
    int G;                    // groups: E_loc routed + 1 shared
    int N;                    // weight rows per expert (2I or H)
    int K;                    // contraction length (elements)
    int epilogue;             // GemmEpilogue
    float gs_i;               // intermediate global scale (W4A4)
    float* out_f32;           // kEpiGateUpF32: [rows][2I]; kEpiDown: y [rows][H]
    uint8_t* out_codes;       // kEpiGateUpSwiglu W4A4: tiled codes [rows][pitch(I)]
    uint8_t* out_sf;          // kEpiGateUpSwiglu W4A4: scale atoms (K = I)
    uint16_t* out_bf16;       // kEpiGateUpSwiglu W4A16: [rows][I]
    const int32_t* perm_src;  // kEpiDown
    const float* topk_w;      // kEpiDown
    int Tk;                   // kEpiDown: first pair index of the shared rows (T*k)
    int stages;               // pipeline depth (<= kMaxStages; fits the shared memory)
    int staging;              // bytes of epilogue staging (kEpiDown: TMA stores of y), or 0
    int rb_cap;               // W4A4: 128-row blocks the padded rows hold (capacity / 128)
    int raw_slots;            // W4A16: raw weight blobs in flight
    uint32_t* inter_amax;     // kEpiGateUpSwigluF32: fp32 bits of amax |s| (atomic max)
    const float* gs_i_dev;    // kEpiDown: device intermediate scale (dynamic), else gs_i
    float* y_scale;           // kEpiDownF16: [rows] the inverse of each row's fp16 scale
    uint32_t* status;
    int tile_n;               // gemm_swap: token rows per tile at most (16..kSwNmax, % 16 == 0)
};

// W4A4: warp 0 TMA, warp 1 MMA, warps 2..5 epilogue, warps 6..9 scale factors
constexpr int kNvf4Threads = 320;
// Weight blob of one (expert, 128-row tile, 256-element k-stage): 128 rows x 128 bytes of
// codes (the 128-byte swizzled SMEM image) + 4 scale atoms of 512 bytes = 18432 bytes.
// W4A16 blobs have the same image with the 8 codes of each 32-bit word in nibble order
// 0,2,4,6,1,3,5,7 (the order its dequantisation unpacks in pairs).
constexpr int kNvf4TileBytes = 16384 + 2048;
constexpr int kMaxStages = 8;
constexpr int kCtlBytes = 256;          // barriers for kMaxStages + TMEM slot + flags
constexpr int kSmemLimit = 232448;      // dynamic shared memory per block (227 KB)
constexpr int kNvf4StageBytes = 16384 + 16384 + 2048 + 2048;
constexpr int kDownStaging = 4 * 2 * 4096;  // 4 epilogue warps x 2 buffers x 32x32 fp32
// Shared memory of a GEMM launch: stages, epilogue staging, 1 KB alignment slack, control
// block, the group tables (mb_start, counts, offsets) and the group of each row block.
inline int gemm_smem_bytes(int stages, int stage_bytes, int staging, int G, int rb_cap)
{
    return stages * stage_bytes + staging + 1024 + kCtlBytes + 4 * (3 * G + 2) + 4 * rb_cap;
}
inline int gemm_stages(int want, int stage_bytes, int staging, int G, int rb_cap)
{
    int s = want;
    while (s > 2 && gemm_smem_bytes(s, stage_bytes, staging, G, rb_cap) > kSmemLimit) --s;
    return s;
}
__global__ void gemm_nvf4_kernel(const __grid_constant__ CUtensorMap tmA,
                                 const __grid_constant__ CUtensorMap tmA16,
                                 const __grid_constant__ CUtensorMap tmY, GemmArgs args);
// The row-block grouped GEMM with 256-column tiles (two weight tiles per MMA, one
// accumulator, eight epilogue warps): 448 threads; a stage holds the activation tile 16 KB,
// the two weight tiles' codes 32 KB and scales 4 KB, the activation scales 2 KB.  The fp16 down
// epilogue stages 32 x 32 boxes, two 2 KB buffers per epilogue warp.
constexpr int kWideThreads = 448;
constexpr int kWideStageBytes = 16384 + 32768 + 4096 + 2048;
constexpr int kWideDownStaging = 8 * 2 * 2048;
__global__ void gemm_nvf4_wide_kernel(const __grid_constant__ CUtensorMap tmA,
                                      const __grid_constant__ CUtensorMap tmA16,
                                      const __grid_constant__ CUtensorMap tmY, GemmArgs args);
// The same grouped GEMM on CTA pairs (clusters of 2, tcgen05.mma.cta_group::2, M = 256): each
// CTA holds its own 128-row block and half of the 128-row weight tile.  A stage: activation
// tile 16 KB, 64 weight rows 8 KB, all 128 weight rows' scales 2 KB, activation scales 2 KB.
constexpr int kPairStageBytes = 16384 + 8192 + 2048 + 2048;
__global__ void gemm_nvf4_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                                      const __grid_constant__ CUtensorMap tmA16,
                                      const __grid_constant__ CUtensorMap tmY, GemmArgs args);
int gemm_pair_smem_bytes(int stages, int staging, int G, int rb_cap);

// ---- gemm_swap.cu: W4A4 with weight rows as the MMA's M side and up to kSwNmax token rows
// of one expert as its N side (many rows per expert).  448 threads: producer, MMA, eight
// epilogue warps, four scale warps.
constexpr int kSwThreads = 448;
constexpr int kSwNmax = 208;         // token rows per tile at most (GemmArgs::tile_n <= this)
// a stage: weight blob, token codes (tile_n rows of 128 bytes), token scale atoms of two
// 128-row blocks; a multiple of 1024 bytes for tile_n a multiple of 8
__host__ __device__ constexpr int sw_stage_bytes(int tile_n)
{
    return kNvf4TileBytes + tile_n * 128 + 2 * 2048;
}
// scale slots in TMEM beside two accumulators of tile_n columns (at columns 0 and 256): each
// slot holds a stage's weight scales (16 columns) and token scales (4 or 8 columns per
// 64-element k-step)
__host__ __device__ constexpr int sw_sfb_stride(int tile_n) { return tile_n <= 128 ? 4 : 8; }
__host__ __device__ constexpr int sw_slot_cols(int tile_n) { return 16 + 4 * sw_sfb_stride(tile_n); }
__host__ __device__ constexpr int sw_sf_slots(int tile_n)
{
    return 2 * ((256 - tile_n) / sw_slot_cols(tile_n));
}
__global__ void gemm_nvf4_swap_kernel(const __grid_constant__ CUtensorMap tmA,
                                      const __grid_constant__ CUtensorMap tmA16,
                                      const __grid_constant__ CUtensorMap tmY, GemmArgs args);
// dynamic shared memory of a launch with `stages` stages and G groups
int gemm_swap_smem_bytes(int stages, int tile_n, int G);

// ---- gemm_w4a16.cu: swap-AB weight stream, BN token rows per tile (16, 32 or 64)
constexpr int kW16Threads = 480;        // 15 warps: see the kernel's role table
constexpr int kW16MaxRaw = 8;           // raw blobs in flight at most
constexpr int kW16MaxB = 8;             // token-tile slots (one blob's k-range each) at most
// Shared memory: 1 KB alignment slack, raw blob ring, token-tile ring, barriers and flags,
// group tables (counts, offsets, first token block).
inline int w4a16_smem_bytes(int raw_slots, int b_slots, int bn, int G)
{
    return 1024 + raw_slots * kNvf4TileBytes + b_slots * 4 * bn * 128 +
           (2 * raw_slots + 2 * b_slots + 2 * 3 + 5) * 8 + 16 + 4 * (3 * G + 2);
}
// The kernel instantiated for BN = bn (16, 32 or 64) token rows per tile, with fp16 operands
// (gate_up: prescaled fp16 activations) or bf16 operands (down: the bf16 intermediate).
using W16Kernel = void (*)(CUtensorMap, GemmArgs);
W16Kernel w4a16_kernel(int bn, bool f16);

// ---- gemv_w4a16.cu: W4A16 for groups of a few token rows, weights decoded into mma.sync
// fragments.  544 threads: 16 consumer warps and a copy warp streaming the weight blobs
// through a ring of `slots` blobs in shared memory (gemv_w4a16_slots: as many as fit, at most
// kGvMaxSlots; 0 = the shape does not fit).  list_cap bounds the work list: the chunks of up
// to kGvChunk rows of the non-empty groups (at most G + rows / kGvChunk).
constexpr int kGvChunk = 8;
constexpr int kGvThreads = 544;
constexpr int kGvMaxSlots = 12;
using GemvKernel = void (*)(GemmArgs, const uint16_t*, int, int);
GemvKernel gemv_w4a16_kernel_for(bool gateup);
size_t gemv_w4a16_smem(int K, int slots, int list_cap);
int gemv_w4a16_slots(int K, int list_cap);

// The forward's gate_up and down GEMVs in one launch (gemv_w4a16.cu: items of both, a down
// chunk waiting for its gate_up tiles; activation rows taken from the layer input).  With few
// gate_up items each tile's contraction is cut into up to kGvMaxSplit parts, whose partial
// sums (kGvSplitItems parts at most) meet in `part`.  ready ([list_cap]) is zero at launch.
constexpr int kGvMaxSplit = 4;
constexpr int kGvFusedThreads = kGvThreads + 32;  // + the signal warp
constexpr int kGvSplitItems = 1024;
struct GvFusedArgs {
    GemmArgs gu;           // gate_up: W13 blobs, gs_w, counts/offsets/G, perm_src, Tk, status,
                           // out_bf16 = the intermediate rows [rows][I]
    GemmArgs dn;           // down: W2 blobs, gs_w, perm_src, topk_w, Tk, out_f32 = y [rows][H]
    const int32_t* ids;    // the top-k ids [T][k] (the work list is formed from them)
    int E, off;            // experts, and the shard's first expert
    int shared_rows;       // rows of the shared group (T, or 0)
    const uint16_t* x;     // the layer input [T][H], bf16
    const uint32_t* amax;  // fp32 bits of max |x|
    float* gs_out;         // receives the prescale gs (the forward's record of gs_a)
    int T, k;
    int tok_rows;          // rows of a chunk at most: min(kGvChunk, T)
    int32_t* ready;        // [list_cap] gate_up tiles (or tile parts) stored per chunk
    float* part;           // [kGvSplitItems][kGvChunk tokens][128 rows] partial sums
};
using FusedGemvKernel = void (*)(GvFusedArgs, int, int);
FusedGemvKernel gemv_w4a16_fused_kernel_ptr();
size_t gemv_w4a16_fused_smem(int H, int tok_rows, int slots, int list_cap);
int gemv_w4a16_fused_slots(int H, int tok_rows, int list_cap);

}  // namespace moe
