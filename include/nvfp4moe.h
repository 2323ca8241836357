/*
 * nvfp4moe.h -- C ABI of the NVFP4 fused mixture-of-experts layer forward (one GPU).
 *
 * The operation: a mixture-of-experts layer with routed experts plus one always-on
 * shared expert and top-k routing (Solar Open 2 on DGX Spark, "Solar Open 2 개요": 320
 * routed, 1 shared, top-8), NVFP4 weights (packed FP4 codes, FP8 E4M3 block scales of
 * 16 elements clamped at 448, one FP32 global scale per expert and projection; same
 * page, "b12x 버전이 실제 NVFP4 체크포인트를 읽어들이도록 만들기"), a fused gate/up
 * projection followed by silu(gate)*up and a down projection, and expert parallelism by
 * a contiguous shard of experts selected by local_expert_offset, whose output is the
 * shard's partial sum (same page, "b12x에서의 Expert Parallelism 구현 추가").
 *
 * Passages: every declaration below names the passage that defines its operation, as
 *   [OV] "Serving Solar Open 2 (NVFP4) on DGX Spark", section "Solar Open 2 개요";
 *   [EP] the same page, section "b12x에서의 Expert Parallelism 구현 추가";
 *   [CK] the same page, section "b12x 버전이 실제 NVFP4 체크포인트를 읽어들이도록 만들기";
 *   or "none" for this library's own plumbing, which the pages have no counterpart for.
 *
 * Conventions for every call:
 *   - Pointers named *_d are device pointers; all tensors are caller-owned unless stated.
 *     moe_create copies the weights into its own re-laid-out buffers: the caller may free
 *     its copies once moe_create returns.
 *   - Every call is asynchronous and ordered on the given stream (0 = legacy default).
 *   - Argument errors are reported synchronously, before anything is launched, with
 *     MOE_ERR_INVALID / MOE_ERR_UNSUPPORTED / MOE_ERR_WORKSPACE.  CUDA launch errors give
 *     MOE_ERR_CUDA.  Errors found on the device (an expert id outside [0, E), a bounded
 *     wait that ran out) set a status word in the workspace, drop the offending work and
 *     never trap; moe_get_status reads and clears it.  moe_forward clears the word when
 *     it starts; the staged calls only add to it, so a new workspace is zero-filled (or
 *     cleared with moe_get_status) before staged calls are checked.
 *   - No exceptions cross this boundary.  A handle is immutable after moe_create:
 *     concurrent calls on one handle are safe with separate workspaces.
 *   - bf16 tensors are passed as uint16_t bit patterns (void* in signatures).
 *
 * Layouts:
 *   canonical NVFP4 matrix [R][K]: codes uint8 [R][K/2], element 2i in the low nibble and
 *     2i+1 in the high nibble; block scales uint8 (E4M3) [R][K/16]; the value of an
 *     element is E2M1(code) * E4M3(scale) / gs, gs the FP32 global (encode) scale.
 *   padded rows: the grouped GEMMs work on "padded rows" -- the routed (token, expert)
 *     pairs grouped by local expert (ascending pair index p = t*k + j inside a group),
 *     each group starting on a multiple of 128 rows, followed by a group of T rows for the
 *     shared expert.  expert_offsets[g] is the first padded row of group g
 *     (g = 0..E_loc-1 routed, g = E_loc shared), expert_offsets[E_loc+1] the total.
 *   tiled NVFP4 activations (the GEMM operand layout): codes uint8 [rows][pitch] with
 *     pitch = round_up(K/2, 128) bytes; scales in 512-byte atoms, one per (128-row block
 *     rb, 64-element k-step s) at byte ((rb * K/64) + s) * 512, and inside an atom row m
 *     (0..127) scale kk (0..3) at byte (m % 32) * 16 + (m / 32) * 4 + kk.
 */
#ifndef NVFP4MOE_H
#define NVFP4MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

/* cudaStream_t without the CUDA headers. */
typedef struct CUstream_st* moe_stream_t;

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID = 1,        /* bad argument (null pointer, size out of range) */
    MOE_ERR_UNSUPPORTED = 2,    /* valid but unsupported shape or mode */
    MOE_ERR_CUDA = 3,           /* a CUDA runtime/driver call failed */
    MOE_ERR_WORKSPACE = 4,      /* workspace smaller than moe_workspace_size */
    MOE_ERR_TIMEOUT = 5,        /* a bounded device wait ran out (see moe_get_status) */
    MOE_ERR_DEVICE_STATUS = 6   /* the device flagged bad data (see moe_get_status) */
} moe_status;

typedef enum {
    MOE_W4A4_DYNAMIC = 0,   /* NVFP4 activations, global scale 2688/amax(x) per call */
    MOE_W4A4_STATIC = 1,    /* NVFP4 activations, global scale act_global_scale */
    MOE_W4A16 = 2           /* bf16 activations x NVFP4 weights */
} moe_act_mode;

/* How a checkpoint gives an expert's global scale (moe_prepare_weights). */
typedef enum {
    MOE_GS_ENCODE = 0,      /* the encode scale gs: value = code * sf / gs (reciprocal form) */
    MOE_GS_DEQUANT = 1      /* a dequantisation multiplier m: value = code * sf * m */
} moe_gs_convention;

/* Device status bits (moe_get_status's *bits). */
#define MOE_DEV_BAD_EXPERT_ID  0x1u   /* a top-k id outside [0, num_experts): pair dropped */
#define MOE_DEV_WAIT_TIMEOUT   0x2u   /* a pipeline wait ran out: that tile was abandoned */
#define MOE_DEV_ROWS_OVERFLOW  0x4u   /* padded rows exceeded capacity: pairs dropped */
#define MOE_DEV_BAD_INDEX      0x8u   /* library built with MOE_DEBUG only: a padded-row or
                                         pair index read from a buffer was out of range; the
                                         access was skipped */

typedef struct {
    int32_t hidden;               /* H: multiple of 128 */
    int32_t inter;                /* I: multiple of 64 */
    int32_t num_experts;          /* E: global routed experts, 1..1024 */
    int32_t top_k;                /* k: 1..min(E, 32) */
    int32_t num_local_experts;    /* E_loc: experts held by this shard, 0..E */
    int32_t local_expert_offset;  /* global id of local expert 0; off + E_loc <= E */
    int32_t has_shared;           /* 1 if the layer has the shared expert */
    int32_t shared_inter;         /* intermediate size of the shared expert (== inter) */
    int32_t add_shared;           /* 1: add the shared expert into THIS partial sum */
    int32_t act_mode;             /* moe_act_mode */
    float act_global_scale;       /* MOE_W4A4_STATIC only */
    float inter_global_scale;     /* global scale of the intermediate (W4A4): > 0 static;
                                     0 dynamic -- 2688 / amax of the fp32 intermediate over
                                     every row the call computes, in two passes (gate_up
                                     writes fp32 s and its amax, then s is quantised) */
    int32_t max_tokens;           /* largest T a call may pass */
    int32_t gemm_tiling;          /* W4A4 grouped GEMM form: 0 the library's choice (row
                                     blocks, the faster form at every measured size); 1 row
                                     blocks: 128 padded rows x 128 weight rows per MMA tile;
                                     2 token tiles: 128 weight rows x up to 208 token rows of
                                     one expert (no padding rows in the MMA); 3 row blocks on
                                     CTA pairs: 256 padded rows x 128 weight rows per pair,
                                     each CTA streaming half of the weight tile; 4 row blocks
                                     x 256 weight rows per MMA (weight matrices of a multiple of
                                     256 rows; others take form 1) */
} moe_config;

/* Device pointers, canonical layouts (see above). */
typedef struct {
    const void* router_w_d;       /* bf16 [E][H] (global E: routing is global) */
    const uint8_t* w13_d;         /* [E_loc][2I][H/2]; rows 0..I-1 gate, I..2I-1 up */
    const uint8_t* w13_sf_d;      /* [E_loc][2I][H/16] */
    const float* w13_gs_d;        /* [E_loc] */
    const uint8_t* w2_d;          /* [E_loc][H][I/2] */
    const uint8_t* w2_sf_d;       /* [E_loc][H][I/16] */
    const float* w2_gs_d;         /* [E_loc] */
    const uint8_t* sh13_d;        /* shared expert, [2I][H/2] (NULL when !has_shared) */
    const uint8_t* sh13_sf_d;     /* [2I][H/16] */
    const float* sh13_gs_d;       /* [1] */
    const uint8_t* sh2_d;         /* [H][I/2] */
    const uint8_t* sh2_sf_d;      /* [H][I/16] */
    const float* sh2_gs_d;        /* [1] */
} moe_weights;

typedef struct moe_layer* moe_handle;

/* Validates cfg, allocates the handle and device copies of the weights re-laid out for
 * the grouped GEMMs (gate/up rows interleaved in blocks of 16 inside each 128-row tile,
 * scales in 512-byte atoms, one extra expert slot for the shared expert).  Synchronises
 * the stream before returning.  *out receives the handle (NULL on error).
 * Passage: [OV] (320 routed + 1 shared experts) and [CK] (packed FP4
 * weights, FP8 block scales, a per-expert global scale, fused gate/up rows, MMA tile layout). */
MOE_API moe_status moe_create(const moe_config* cfg, const moe_weights* w, moe_stream_t stream,
                      moe_handle* out);
/* Passage: none; releases what moe_create allocated (the pages have no counterpart). */
MOE_API void moe_destroy(moe_handle h);

/* Bytes of workspace a call with T tokens needs (moe_forward and the staged calls).
 * One workspace may be shared by every layer of a model (calls on one stream).
 * Passage: [EP] (one module-level workspace pool
 * shared by the layers instead of per-layer scratch). */
MOE_API size_t moe_workspace_size(const moe_config* cfg, int32_t T);

/* Padded-row capacity for T tokens: every buffer indexed by padded row is sized to it.
 * Passage: [EP] (the compact pre-pass that groups the
 * local pairs by expert); the 128-row padding is this library's GEMM tile. */
MOE_API int32_t moe_rows_capacity(const moe_config* cfg, int32_t T);

/* Router (steps: logits, softmax + top-k).  logits = x . Wr^T (+ logit_bias) in fp32, or
 * logits_in (+ logit_bias) when given.  topk_ids_d[T][k]: the k largest logits,
 * descending, ties to the lower id (-0 equals +0; a NaN ranks below every number);
 * topk_w_d[T][k]: softmax over the selected logits.
 * logits_out_d (nullable): fp32 [T][E] including the bias.  x_bf16_d may be NULL when
 * logits_in_d is set.  ws: scratch for the logits when they are computed from x.
 * Passage: [OV] (top-8 of 320 routed experts; the softmax over the
 * selected logits and the tie rule are readings where the page is silent). */
MOE_API moe_status moe_route_topk(moe_handle h, const void* x_bf16_d, const float* logits_in_d,
                          const float* logit_bias_d, int32_t T, int32_t* topk_ids_d,
                          float* topk_w_d, float* logits_out_d, void* ws_d, size_t ws_bytes,
                          moe_stream_t stream);

/* Routing that allocates nothing: moe_route_topk's computation, for callers that cannot
 * allocate device memory at call time and have no workspace to lend -- for example code
 * running while another component owns every byte of device memory through its own pool,
 * or a caller in a phase where a cudaMalloc (which may synchronise the device) is not
 * allowed.  The pages have no counterpart; it is an addition of this library.
 * Result: the ids are the top-k of the returned logits exactly as moe_route_topk selects
 * them, and the logits and weights agree with moe_route_topk's to fp32 rounding (for
 * T * E * splits beyond the scratch this call sums fewer router k-splits, in another fp32
 * order, so near-ties may select differently).
 * The router's partial-sum planes and a status word live in one file-scope 8 MiB device
 * array that every device loading the library keeps until exit; T * E (tokens x global
 * experts) must not exceed 2,097,088, else MOE_ERR_WORKSPACE (with E = 320: T <= 6553).
 * The first call on a device (and again after the device's context changes, e.g. after a
 * cudaDeviceReset) looks the array's address up (cudaGetSymbolAddress, with the handle's
 * device current) and should come before any stream capture.  All calls share the array:
 * calls whose executions overlap on the GPU race (use one stream, or serialise them).  Each
 * call clears the status word and writes every plane value it reads.  If a bounded wait of
 * the router runs out, every id is written as -1 and every weight as 0 (moe_permute drops
 * such pairs and flags MOE_DEV_BAD_EXPERT_ID).  Given logits_in_d, no scratch is touched.
 * Passage: none -- the pages have no counterpart (see above). */
MOE_API moe_status moe_route_topk_noalloc(moe_handle h, const void* x_bf16_d,
                                          const float* logits_in_d, const float* logit_bias_d,
                                          int32_t T, int32_t* topk_ids_d, float* topk_w_d,
                                          float* logits_out_d, moe_stream_t stream);

/* Local map + grouping (the "compact pre-pass").  Pair p = t*k + j with local expert
 * e' = topk_ids[p] - local_expert_offset is kept iff 0 <= e' < E_loc (a pair with an id
 * outside [0, E) is dropped and sets MOE_DEV_BAD_EXPERT_ID).  Outputs:
 *   expert_counts_d[E_loc+1]  rows of each group (group E_loc: T if the shared expert is
 *                             added by this shard, else 0)
 *   expert_offsets_d[E_loc+2] padded first row of each group, [E_loc+1] = total
 *   perm_src_d[rows_capacity] pair index of each padded row (T*k + t for shared rows,
 *                             -1 for padding)
 *   inv_d[T*k]                padded row of each pair, -1 if dropped
 * ws: the workspace (its tile table is filled here and read by the grouped GEMMs).
 * Passage: [EP] (local_expert_offset maps global ids to the
 * shard; pairs outside it are filtered by a CTA-uniform guard; the compact pre-pass). */
MOE_API moe_status moe_permute(moe_handle h, const int32_t* topk_ids_d, int32_t T,
                       int32_t* expert_counts_d, int32_t* expert_offsets_d,
                       int32_t* perm_src_d, int32_t* inv_d, void* ws_d, size_t ws_bytes,
                       moe_stream_t stream);

/* NVFP4 quantiser of a bf16 matrix [rows][cols] (cols % 64 == 0).  gs_in_d NULL: dynamic
 * global scale 2688/amax over the whole matrix (written to gs_out_d); else the scale
 * *gs_in_d.  sf_layout 0: canonical codes [rows][cols/2], scales [rows][cols/16];
 * sf_layout 1: tiled (pitch-padded codes, 512-byte scale atoms).  ws: scratch for amax.
 * Passage: [CK] (packed FP4 codes, FP8 E4M3 block scales
 * clamped at 448, an FP32 global scale in reciprocal form). */
MOE_API moe_status moe_quant_nvfp4(const void* x_bf16_d, int32_t rows, int32_t cols,
                           const float* gs_in_d, float* gs_out_d, uint8_t* codes_d,
                           uint8_t* sf_d, int32_t sf_layout, void* ws_d, size_t ws_bytes,
                           moe_stream_t stream);

/* Gather-quantise: NVFP4-quantise the T rows of x with gs (dynamic or static per the
 * handle's act_mode) and write row t to every padded row of its local pairs and to its
 * shared row, in the tiled layout (W4A4).  W4A16: write fp16(x * gs) instead
 * (a_bf16_d [rows_capacity][H] fp16), gs = 2^(141 - e) for e the exponent field of
 * amax|x| (clamped to 2^[-126, 127]), so |x * gs| <= 2^15 and every x above amax * 2^-29
 * converts exactly.  gs_out_d receives the scale used (both modes).
 * Passage: [EP] (tokens reach the local experts of the
 * shard) and [CK] (the NVFP4 format of the operands). */
MOE_API moe_status moe_gather_activations(moe_handle h, const void* x_bf16_d, int32_t T,
                                  const int32_t* inv_d, const int32_t* expert_offsets_d,
                                  uint8_t* a_codes_d, uint8_t* a_sf_d, void* a_bf16_d,
                                  float* gs_out_d, void* ws_d, size_t ws_bytes,
                                  moe_stream_t stream);

/* Grouped GEMM gate_up over the padded rows: for group g with expert weights W13_g,
 * G = A_g . W13_g^T / (gs_a * gs13_g), A_g the NVFP4 rows (W4A4) or the fp16 rows of
 * moe_gather_activations (W4A16, gs_a its fp16 prescale).  gs_a_d (a device scalar) is
 * required in both modes.
 *   fuse_epilogue 0: gateup_f32_d [rows_capacity][2I] fp32 (gate cols 0..I-1, up I..2I-1)
 *   fuse_epilogue 1: s = silu(gate) * up, then
 *       W4A4 : NVFP4 with inter_global_scale -> inter_codes_d / inter_sf_d (tiled, K = I);
 *              with the dynamic scale (inter_global_scale 0) the call runs both passes,
 *              using the workspace for the fp32 intermediate, and leaves gs_i there for
 *              moe_grouped_gemm_down on the same workspace
 *       W4A16: bf16 -> inter_bf16_d [rows_capacity][I]
 * Padding rows of the outputs are left unwritten.
 * Passage: [CK] (the fused gate/up projection, its row
 * order, per-expert global scales) and [EP] (per-expert scales of the local experts). */
MOE_API moe_status moe_grouped_gemm_gateup(moe_handle h, const uint8_t* a_codes_d,
                                   const uint8_t* a_sf_d, const float* gs_a_d,
                                   const void* a_bf16_d, const int32_t* expert_counts_d,
                                   const int32_t* expert_offsets_d, int32_t fuse_epilogue,
                                   float* gateup_f32_d, uint8_t* inter_codes_d,
                                   uint8_t* inter_sf_d, void* inter_bf16_d, int32_t T,
                                   void* ws_d, size_t ws_bytes, moe_stream_t stream);

/* Checkpoint-convention weight preparation.  Passage: [CK] (packed FP4 weights, FP8 block
 * scales and a per-expert global scale in either convention; the reciprocal global scale
 * inverted and folded into the FP8 block scales with re-rounding, clamped at 448; the fused
 * gate/up row order; per-shard scale slicing).  One weight matrix type of num_experts
 * experts, each N x K NVFP4 in the canonical layout -- codes_d [E][N][K/2] (element 2i in the low
 * nibble), sf_d [E][N][K/16] E4M3, glob_d [E] fp32 -- becomes the moe_weights form of
 * experts off .. off+count-1:
 *   codes_out_d [count][N][K/2]: the codes (rows reordered by swap_halves);
 *   gs_out_d [count]: the encode scale gs (convention MOE_GS_DEQUANT: gs = 1/m in fp32);
 *   sf_out_d [count][N][K/16]: the scales, or with fold_target > 0 each expert's global
 *     folded in relative to the common scale gs_t = fold_target: r = gs_t / gs (fp32),
 *     sf' = E4M3(sf * r) rounded to nearest even and saturated at 448, and gs_out = gs_t
 *     for every expert (gs_t = 1 removes the global scale altogether);
 *   swap_halves != 0: output rows 0..N/2-1 are input rows N/2..N-1 and vice versa (a fused
 *     gate/up matrix stored up-then-gate becomes gate-then-up).
 * Scale bytes must not be the NaN pattern.  Device pointers, caller-owned; codes_d and
 * codes_out_d 16-byte aligned; K a multiple of 64; count 0 is a no-op (pointers unused).
 * Stream-ordered; argument errors return before any launch. */
MOE_API moe_status moe_prepare_weights(const uint8_t* codes_d, const uint8_t* sf_d,
                                       const float* glob_d, int32_t num_experts, int32_t N,
                                       int32_t K, int32_t convention, float fold_target,
                                       int32_t swap_halves, int32_t off, int32_t count,
                                       uint8_t* codes_out_d, uint8_t* sf_out_d,
                                       float* gs_out_d, moe_stream_t stream);

/* SwiGLU + NVFP4 requantisation of fp32 gate/up rows [rows][2I] (gate cols 0..I-1):
 * s = silu(g) * u in fp32, quantised with the static scale gs_i.  sf_layout as for
 * moe_quant_nvfp4 (0 canonical, 1 tiled).
 * Passage: [CK] (the fused gate/up projection whose halves
 * feed silu(gate) * up) and [EP] (the static / dynamic W4A4 backends requantise it). */
MOE_API moe_status moe_swiglu_requant(const float* gateup_f32_d, int32_t rows, int32_t inter,
                              float gs_i, uint8_t* codes_d, uint8_t* sf_d, int32_t sf_layout,
                              moe_stream_t stream);

/* Grouped GEMM down: Y_g = Aq_g . W2_g^T / (gs_i * gs2_g) (W4A16: / gs2_g; dynamic
 * intermediate scale: gs_i is the one moe_grouped_gemm_gateup left in ws_d), each row
 * multiplied by its routing weight (1 for shared rows; the weight of padded row r is
 * topk_w[perm_src[r]]), written to y_d[rows_capacity][H] fp32 at the same padded row.
 * Padding rows of y may receive arbitrary values.
 * Passage: [EP] (each local expert's output, weighted by its
 * routing weight, enters the shard's partial sum). */
MOE_API moe_status moe_grouped_gemm_down(moe_handle h, const uint8_t* inter_codes_d,
                                 const uint8_t* inter_sf_d, const void* inter_bf16_d,
                                 const int32_t* expert_counts_d,
                                 const int32_t* expert_offsets_d, const int32_t* perm_src_d,
                                 const float* topk_w_d, float* y_d, int32_t T, void* ws_d,
                                 size_t ws_bytes, moe_stream_t stream);

/* Combine: out[t] = sum_{j: inv[t*k+j] >= 0} y[inv[t*k+j]]
 *                  + (add_shared ? y[expert_offsets[E_loc] + t] : 0),
 * y indexed by padded row (moe_grouped_gemm_down), summed in ascending j then the shared
 * term in fp32, rounded to bf16.
 * Passage: [EP] (the shard's output is the partial sum over its
 * local experts [T, H], which an all-reduce adds across shards). */
MOE_API moe_status moe_combine(moe_handle h, const float* y_d, const int32_t* inv_d,
                       const int32_t* expert_offsets_d, int32_t T, void* out_bf16_d,
                       moe_stream_t stream);

/* The whole layer: route, permute, gather-quantise, gate_up (fused SwiGLU+requant),
 * down, combine.  logits_in_d (nullable): given router logits [T][E] instead of x.Wr^T;
 * logit_bias_d (nullable) [E].  out_bf16_d [T][H] receives this shard's partial sum.
 * W4A16 batches of up to 256 tokens run gate_up and down as one cooperative launch that
 * forms the fp16 activation rows from x itself (no gather launch); the results are those
 * of the staged calls up to the fp32 summation order of the expert rows.
 * Unlike the staged calls, the W4A4 modes keep the weighted expert rows between down and
 * combine as fp16 values of y x 2^e (e per local expert, from a bound on |y| that rules out
 * overflow; see moe_forward_buffers), each with 11 significant bits; the combine multiplies
 * by 2^-e and sums in the same fixed order in fp32.
 * Passage: [OV] (the layer: 320 routed + 1 shared experts, top-8)
 * and [EP] (local_expert_offset, the partial-sum output; the static W4A4, dynamic W4A4
 * and W4A16 fused-MoE backends). */
MOE_API moe_status moe_forward(moe_handle h, const void* x_bf16_d, const float* logits_in_d,
                       const float* logit_bias_d, int32_t T, void* out_bf16_d, void* ws_d,
                       size_t ws_bytes, moe_stream_t stream);

/* The whole layer on host buffers: x_bf16_h [T][H] is copied to the device, the layer runs
 * as moe_forward, and out_bf16_h [T][H] is copied back, all ordered on the stream -- the
 * call returns before the copies finish (pinned host memory; with pageable memory the
 * copies are synchronous): synchronise the stream before reading out_bf16_h.  The device
 * copies of x and out live at the end of the workspace, which must hold
 * moe_workspace_size_host(cfg, T) bytes.  logits_in_d / logit_bias_d as for moe_forward
 * (device pointers).
 * Passage: [OV] and [EP], as moe_forward. */
MOE_API moe_status moe_forward_host(moe_handle h, const void* x_bf16_h, const float* logits_in_d,
                                    const float* logit_bias_d, int32_t T, void* out_bf16_h,
                                    void* ws_d, size_t ws_bytes, moe_stream_t stream);

/* Workspace bytes for moe_forward_host: moe_workspace_size plus room for the device copies
 * of x and out (0 for an invalid cfg).
 * Passage: none; buffer sizing of this library (the pages have no counterpart). */
MOE_API size_t moe_workspace_size_host(const moe_config* cfg, int32_t T);

/* Where moe_forward keeps its intermediates inside the workspace (device pointers into
 * ws_d), so callers can inspect them after a forward.  Any pointer may be NULL.  Unlike
 * moe_permute's, the forward's perm_src leaves padding rows unmarked (stale).  W4A16
 * forwards of up to 256 tokens write no a_bf16 rows (the fused GEMV forms them while
 * staging), and with one or a few tokens, where it splits each gate_up tile's contraction,
 * no inter_bf16 rows either.  inter_gs:
 * the dynamic intermediate scale of the last forward (set only in that mode).  y: the
 * weighted expert outputs by padded row -- fp32 in W4A16 mode; in the W4A4 modes fp16 rows
 * of y x 2^e (e per local expert, chosen from a bound on |y| so that no value overflows)
 * with y_scale[row] = 2^-e (float, per padded row), which the combine multiplies back.
 * Passage: none; inspection of moe_forward's intermediates (the pages have no counterpart). */
MOE_API moe_status moe_forward_buffers(moe_handle h, void* ws_d, int32_t T, int32_t** topk_ids,
                               float** topk_w, int32_t** expert_counts,
                               int32_t** expert_offsets, int32_t** perm_src, int32_t** inv,
                               float** gs_a, uint8_t** a_codes, uint8_t** a_sf,
                               void** a_bf16, uint8_t** inter_codes, uint8_t** inter_sf,
                               void** inter_bf16, float** y, float** inter_gs,
                               float** y_scale);

/* Reads the device status word of ws (synchronises the stream) into *bits (nullable) and
 * clears it.  Returns MOE_OK, MOE_ERR_TIMEOUT (MOE_DEV_WAIT_TIMEOUT set) or
 * MOE_ERR_DEVICE_STATUS (other bits set).
 * Passage: none; the device status word of this library (the pages have no counterpart). */
MOE_API moe_status moe_get_status(moe_handle h, void* ws_d, moe_stream_t stream, uint32_t* bits);

/* Self-test of the failure path of the pipelines' bounded waits: one thread waits, with the
 * same bounded wait the kernels use, on an mbarrier phase that nothing completes, so the
 * wait runs out after limit_ns (1 ns .. 2 s) and sets MOE_DEV_WAIT_TIMEOUT in *status_d (a
 * caller-owned device word, cleared first), as a pipeline role would; no trap, the context
 * stays usable.  Synchronises the stream.  Returns MOE_ERR_TIMEOUT (the expected outcome),
 * MOE_OK (the wait completed: a broken wait), MOE_ERR_INVALID or MOE_ERR_CUDA.
 * Passage: none; a self-test of this library's bounded waits (the pages have no
 * counterpart). */
MOE_API moe_status moe_selftest_bounded_wait(uint32_t* status_d, uint64_t limit_ns,
                                             moe_stream_t stream);

/* Passage: none; error text of this library (the pages have no counterpart). */
MOE_API const char* moe_status_string(moe_status s);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4MOE_H */
