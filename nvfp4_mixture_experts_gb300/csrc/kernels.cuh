// Kernel declarations shared by the translation units of the library.
#pragma once

#include "common.cuh"

namespace moe {

constexpr int kPairsPerBlock = 1024;   // grouping: pairs per block of the counting sort

// silu(g) * u in fp32: g / (1 + exp(-g)) * u, each step an IEEE fp32 operation.
__device__ __forceinline__ float silu_mul(float g, float u)
{
    return __fmul_rn(__fdiv_rn(g, __fadd_rn(1.0f, expf(-g))), u);
}

// ---- route.cu
__global__ void router_logits_kernel(const uint16_t* x, const uint16_t* wr, const float* bias,
                                     int T, int H, int E, float* logits);
__global__ void topk_kernel(const float* logits_src, const float* bias, int T, int E, int k,
                            int32_t* ids, float* wts, float* logits_out);
__global__ void perm_hist_kernel(const int32_t* ids, int P, int E, int off, int El,
                                 int32_t* hist, uint32_t* status);
__global__ void perm_scan_kernel(const int32_t* hist, int nblk, int El, int T, int k,
                                 int shared_rows, int rows_cap, int32_t* blkoff,
                                 int32_t* counts, int32_t* offsets, int32_t* mb_start,
                                 int32_t* perm_src, uint32_t* status);
__global__ void perm_scatter_kernel(const int32_t* ids, int P, int E, int off, int El,
                                    const int32_t* blkoff, const int32_t* offsets,
                                    int rows_cap, int32_t* perm_src, int32_t* inv);

// ---- quant.cu
__global__ void amax_bf16_kernel(const uint16_t* x, int64_t n, uint32_t* amax_bits);
__global__ void gather_quant_kernel(const uint16_t* x, int T, int H, int k, const int32_t* inv,
                                    const int32_t* offsets, int shared_group, int add_shared,
                                    const float* gs_static, const uint32_t* amax_bits,
                                    uint8_t* codes, uint8_t* sf, float* gs_out);
__global__ void gather_bf16_kernel(const uint16_t* x, int T, int H, int k, const int32_t* inv,
                                   const int32_t* offsets, int shared_group, int add_shared,
                                   uint16_t* out);
__global__ void quant_rows_kernel(const uint16_t* x, int rows, int cols, const float* gs_static,
                                  const uint32_t* amax_bits, uint8_t* codes, uint8_t* sf,
                                  int layout, float* gs_out);
__global__ void swiglu_requant_kernel(const float* gu, int rows, int I, float gs_i,
                                      uint8_t* codes, uint8_t* sf, int layout);
__global__ void combine_kernel(const float* y, const int32_t* inv, int T, int H, int k,
                               int add_shared, uint16_t* out);
__global__ void repack_codes_kernel(const uint8_t* src, int nexp, int N, int K,
                                    int interleave, uint8_t* dst);
__global__ void repack_sf_kernel(const uint8_t* src, int nexp, int N, int K, int interleave,
                                 uint8_t* dst);

// ---- gemm.cu
enum GemmEpilogue : int {
    kEpiGateUpF32 = 0,     // G (alpha applied) -> fp32 rows, gate then up columns
    kEpiGateUpSwiglu = 1,  // silu(gate)*up -> NVFP4 (W4A4) or bf16 (W4A16)
    kEpiDown = 2           // Y * routing weight -> fp32 rows indexed by pair
};

struct GemmArgs {
    const uint8_t* a_sf;      // W4A4: activation scale atoms (tiled, K-wide)
    const uint8_t* b_sf;      // weight scale atoms [slots][N/128][K/64][512]
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
    float* out_f32;           // kEpiGateUpF32: [rows][2I]; kEpiDown: y [pairs][H]
    uint8_t* out_codes;       // kEpiGateUpSwiglu W4A4: tiled codes [rows][pitch(I)]
    uint8_t* out_sf;          // kEpiGateUpSwiglu W4A4: scale atoms (K = I)
    uint16_t* out_bf16;       // kEpiGateUpSwiglu W4A16: [rows][I]
    const int32_t* perm_src;  // kEpiDown
    const float* topk_w;      // kEpiDown
    int Tk;                   // kEpiDown: first pair index of the shared rows (T*k)
    uint32_t* status;
};

constexpr int kGemmThreads = 192;       // warp 0 TMA, warp 1 MMA, warps 2..5 epilogue
constexpr int kNvf4Stages = 6;
constexpr int kNvf4StageBytes = 16384 + 16384 + 2048 + 2048;
constexpr int kNvf4Smem = kNvf4Stages * kNvf4StageBytes + 1024 + 256;
constexpr int kBf16Stages = 6;
constexpr int kBf16StageBytes = 37888;   // A 16K + B 16K + raw FP4 4K + scales 512, padded to 1 KB
constexpr int kBf16Smem = kBf16Stages * kBf16StageBytes + 1024 + 256;
constexpr int kBf16Threads = 320;       // + 4 dequantisation warps

__global__ void gemm_nvf4_kernel(const __grid_constant__ CUtensorMap tmA,
                                 const __grid_constant__ CUtensorMap tmA16,
                                 const __grid_constant__ CUtensorMap tmB, GemmArgs args);
__global__ void gemm_w4a16_kernel(const __grid_constant__ CUtensorMap tmA,
                                  const __grid_constant__ CUtensorMap tmA16,
                                  const __grid_constant__ CUtensorMap tmB, GemmArgs args);

}  // namespace moe
