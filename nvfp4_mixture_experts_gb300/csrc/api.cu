// C ABI of the NVFP4 fused mixture-of-experts layer: argument checks, the workspace plan,
// tensor-map encoding and the launch sequence of the forward.  Every step of the forward
// runs in this library's kernels; there is no host or library fallback.
#include <cuda.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <cstdio>
#include <cmath>
#include <cstring>
#include <mutex>
#include <new>

#include "kernels.cuh"

using namespace moe;

namespace {

// ---------------------------------------------------------------- NVTX ranges
// Every C-ABI call that launches work opens a range named after itself in the "nvfp4moe"
// domain (host-side; a profiler attributes the call's launches to it).  With no tool
// attached an NVTX call returns at once.
struct NvtxRange {
    explicit NvtxRange(const char* name)
    {
        static const nvtxDomainHandle_t domain = nvtxDomainCreateA("nvfp4moe");
        nvtxEventAttributes_t a = {};
        a.version = NVTX_VERSION;
        a.size = NVTX_EVENT_ATTRIB_STRUCT_SIZE;
        a.messageType = NVTX_MESSAGE_TYPE_ASCII;
        a.message.ascii = name;
        nvtxDomainRangePushEx(domain, &a);
        dom = domain;
    }
    ~NvtxRange() { nvtxDomainRangePop(dom); }
    nvtxDomainHandle_t dom;
};

// ---------------------------------------------------------------- driver entry point
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// 2-D tensor map over rows of row_bytes (dims in elements of dtype).
bool make_tmap(CUtensorMap* m, const void* base, CUtensorMapDataType dtype, uint64_t inner,
               uint64_t rows, uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows,
               CUtensorMapSwizzle swz)
{
    EncodeTiledFn enc = encode_fn();
    if (!enc || rows == 0) return false;
    const cuuint64_t dims[2] = {inner, rows};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_inner, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

int ceil_div(int a, int b) { return (a + b - 1) / b; }

// ---------------------------------------------------------------- workspace plan
struct Plan {
    int T, k, E, El, G, H, I, cap, nblk, Tk;
    int gv_list_cap;  // W4A16 grouped GEMV: chunks of up to kGvChunk rows at most
    size_t status, amax, gs_a, gs_i, ids, w, logits, hist, blkoff, counts, offsets, mb_start,
        perm_src, inv, a_codes, a_sf, a_bf16, i_codes, i_sf, i_bf16, s_f32, y, y_scale, gv_sync,
        gv_part, total;
    // amax holds two words: the activation amax, then the intermediate amax (dynamic gs_i);
    // gv_sync: the fused GEMV's ready counts [gv_list_cap]; gv_part: its split partial sums
};

// W4A16 batches of at most this many tokens (and at most 2 x 8 expected rows per local
// expert) take the grouped GEMV (gemv_w4a16.cu), which reads each weight once per chunk of
// 8 rows of a group instead of padding every group to the tensor-core kernel's 128-row MMA.
constexpr int kGemvMaxTokens = 256;

// W4A4 with inter_global_scale == 0: the intermediate scale is computed per call.
bool dynamic_inter(const moe_config& c)
{
    return c.act_mode != MOE_W4A16 && c.inter_global_scale == 0.0f;
}

int rows_cap(const moe_config& c, int T)
{
    if (T <= 0) return 0;
    const int64_t P = (int64_t)T * c.top_k;
    const int64_t routed =
        128 * ((P + 127) / 128 + (int64_t)std::min<int64_t>(c.num_local_experts, P));
    const int64_t shared = (c.has_shared && c.add_shared) ? ((int64_t)T + 127) / 128 * 128 : 0;
    const int64_t cap = routed + shared;
    return cap > 0x7fffffff ? -1 : (int)cap;
}

Plan plan(const moe_config& c, int T)
{
    Plan p;
    p.T = T;
    p.k = c.top_k;
    p.E = c.num_experts;
    p.El = c.num_local_experts;
    p.G = p.El + 1;
    p.H = c.hidden;
    p.I = c.inter;
    p.cap = rows_cap(c, T);
    p.Tk = T * c.top_k;
    p.nblk = std::max(1, ceil_div(p.Tk, kPairsPerBlock));
    const bool a16 = c.act_mode == MOE_W4A16;
    size_t o = 0;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o += align256(bytes);
        return at;
    };
    p.status = take(4);
    p.amax = take(8);
    p.gs_a = take(4);
    p.gs_i = take(4);
    p.ids = take((size_t)p.Tk * 4);
    p.w = take((size_t)p.Tk * 4);
    // router partial sums: one plane per k-split (the split count never exceeds the one
    // for a 1024-SM device)
    p.logits = take((size_t)router_splits(std::max(T, 1), p.E, p.H, 1024) * T * p.E * 4);
    p.hist = take((size_t)p.nblk * p.El * 4);
    p.blkoff = take((size_t)p.nblk * p.El * 4);
    p.counts = take((size_t)p.G * 4);
    p.offsets = take((size_t)(p.G + 1) * 4);
    p.mb_start = take((size_t)(p.G + 1) * 4);
    p.perm_src = take((size_t)p.cap * 4);
    p.inv = take((size_t)p.Tk * 4);
    p.a_codes = take(a16 ? 0 : (size_t)p.cap * codes_pitch(p.H));
    p.a_sf = take(a16 ? 0 : (size_t)p.cap * (p.H / 16));
    p.a_bf16 = take(a16 ? (size_t)p.cap * p.H * 2 : 0);
    p.i_codes = take(a16 ? 0 : (size_t)p.cap * codes_pitch(p.I));
    p.i_sf = take(a16 ? 0 : (size_t)p.cap * (p.I / 16));
    p.i_bf16 = take(a16 ? (size_t)p.cap * p.I * 2 : 0);
    p.s_f32 = take(dynamic_inter(c) ? (size_t)p.cap * p.I * 4 : 0);
    p.y = take((size_t)p.cap * p.H * 4);  // fp32 (staged calls) or fp16 (W4A4 forward)
    p.y_scale = take((size_t)p.cap * 4);
    const int64_t rows = (int64_t)T * p.k + ((c.has_shared && c.add_shared) ? T : 0);
    p.gv_list_cap = (int)std::min<int64_t>(0x7fffffff, p.G + (rows + kGvChunk - 1) / kGvChunk);
    const bool gemv = a16 && T <= kGemvMaxTokens;
    p.gv_sync = take(gemv ? (size_t)p.gv_list_cap * 4 : 0);
    p.gv_part = take(gemv ? (size_t)kGvSplitItems * 128 * kGvChunk * 4 : 0);
    p.total = o;
    return p;
}

template <typename T>
T* at(void* ws, size_t off)
{
    return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

moe_status check_launch()
{
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// Launches a kernel, with programmatic dependent launch when pdl is set (the forward's
// chain: each kernel may start while its predecessor finishes; see pdl_wait()).
template <typename... KArgs, typename... Args>
moe_status launch(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                  bool pdl, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...) == cudaSuccess
               ? MOE_OK
               : MOE_ERR_CUDA;
}

// As launch, for a kernel whose blocks run as clusters of two (CTA pairs).
// A launch whose blocks wait on one another (the fused W4A16 GEMV's down items wait for gate_up
// tiles of other blocks): cooperative, so that every block is resident at once or the launch
// fails.
template <typename... KArgs, typename... Args>
moe_status launch_coop(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, bool pdl, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...) == cudaSuccess
               ? MOE_OK
               : MOE_ERR_CUDA;
}

template <typename... KArgs, typename... Args>
moe_status launch_pairs(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                        bool pdl, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...) == cudaSuccess
               ? MOE_OK
               : MOE_ERR_CUDA;
}

}  // namespace

// ---------------------------------------------------------------- the handle
struct moe_layer {
    moe_config cfg;
    int device = 0, num_sms = 0;
    uint16_t* router_w = nullptr;              // [E][H] bf16
    uint8_t* w13 = nullptr;                    // weight blobs, G slots (repack_tiles_kernel)
    uint8_t* w2 = nullptr;
    float *gs13 = nullptr, *gs2 = nullptr;     // [G]
    float* act_gs = nullptr;                   // static activation scale (device copy)
    CUtensorMap tm_router;                     // Wr [E][H] bf16, 64 x 64 boxes
    CUtensorMap tm_router160;                  // Wr [E][H] bf16, 64 x 160 boxes
    int max_pairs = 0;                         // CTA pairs that can be resident at once
};

namespace {

bool set_w4a16_smem_limits()
{
    for (bool gateup : {false, true})
        if (cudaFuncSetAttribute(gemv_w4a16_kernel_for(gateup),
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kSmemLimit) != cudaSuccess)
            return false;
    if (cudaFuncSetAttribute(gemv_w4a16_fused_kernel_ptr(),
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit) != cudaSuccess)
        return false;
    for (int bn : {16, 32, 64})
        for (bool f16 : {false, true})
            if (cudaFuncSetAttribute(w4a16_kernel(bn, f16),
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kSmemLimit) != cudaSuccess)
                return false;
    return true;
}

// Every top-k instantiation may take up to 16 rows of kMaxExperts floats of shared memory.
bool set_topk_smem_limits()
{
    for (int E : {128, 256, 384, 512, kMaxExperts})
        if (cudaFuncSetAttribute(topk_kernel_for(E), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)topk_smem(1, kMaxExperts)) != cudaSuccess)
            return false;
    return true;
}

// Bytes of the weight blobs of one expert slot for an N x K matrix.
size_t blob_bytes(int N, int K)
{
    return (size_t)(N / 128) * ((K + 255) / 256) * kNvf4TileBytes;
}

}  // namespace

namespace {

bool valid_cfg(const moe_config* c, moe_status* why)
{
    *why = MOE_ERR_INVALID;
    if (!c) return false;
    if (c->hidden <= 0 || c->inter <= 0 || c->num_experts <= 0 || c->top_k <= 0) return false;
    if (c->num_local_experts < 0 || c->local_expert_offset < 0) return false;
    if (c->local_expert_offset + c->num_local_experts > c->num_experts) return false;
    if (c->top_k > c->num_experts) return false;
    if (c->max_tokens < 0) return false;
    if (c->act_mode < 0 || c->act_mode > 2) return false;
    if (c->act_mode == MOE_W4A4_STATIC && !(c->act_global_scale > 0.0f)) return false;
    if (c->act_mode != MOE_W4A16 && !(c->inter_global_scale >= 0.0f)) return false;
    if (c->gemm_tiling < 0 || c->gemm_tiling > 4) return false;
    *why = MOE_ERR_UNSUPPORTED;
    if (c->hidden % 128 || c->inter % 64) return false;
    if (c->num_experts > kMaxExperts || c->top_k > kMaxTopK) return false;
    if (c->has_shared && c->shared_inter != c->inter) return false;
    if (rows_cap(*c, c->max_tokens) < 0) return false;
    *why = MOE_OK;
    return true;
}

moe_status check_ws(const moe_layer* h, int T, void* ws, size_t ws_bytes)
{
    if (!ws) return MOE_ERR_INVALID;
    if ((reinterpret_cast<uintptr_t>(ws) & 255) != 0) return MOE_ERR_INVALID;
    if (ws_bytes < plan(h->cfg, T).total) return MOE_ERR_WORKSPACE;
    return MOE_OK;
}

bool t_ok(const moe_layer* h, int T) { return T >= 0 && T <= h->cfg.max_tokens; }

int grid_for(int64_t threads, int block) { return (int)std::max<int64_t>(1, (threads + block - 1) / block); }

// W4A4 grouped GEMM form: row blocks (gemm.cu) unless the configuration asks for token
// tiles (gemm_swap.cu).  Measured on the prefill chunk (8192 tokens, ~205 rows per expert):
// row blocks 1.375 ms per forward (gate_up 690 us, down 440 us), token tiles of up to 208 /
// 160 / 128 rows 1.63 / 1.84 / 1.91 ms (gate_up 843 / 980 / 1027 us); at decode both forms
// stream the weights.  So the automatic choice is row blocks at every size.
constexpr int kTokenTileRows = 208;  // token rows per tile at most (gemm_swap.cu)

bool use_token_tiles(const moe_layer* h, int /*T*/) { return h->cfg.gemm_tiling == 2; }

// Row blocks on CTA pairs (gemm_nvf4_pair_kernel): each CTA streams half of every weight tile.
bool use_pairs(const moe_layer* h, int /*T*/) { return h->cfg.gemm_tiling == 3; }

// Row blocks x 256 weight rows per MMA (gemm_nvf4_wide_kernel), for weight matrices of a
// multiple of 256 rows.
bool use_wide(const moe_layer* h, int /*T*/, int N)
{
    return h->cfg.gemm_tiling == 4 && N % 256 == 0;
}

// Persistent grid: one CTA per SM, or fewer when the tile list (bounded above from the
// pair count, with row blocks of `rows` rows) is shorter.

int gemm_grid(const moe_layer* h, int T, int N, int rows)
{
    const int64_t P = (int64_t)T * h->cfg.top_k;
    int64_t mb = (P + rows - 1) / rows + std::min<int64_t>(h->cfg.num_local_experts, P);
    if (h->cfg.has_shared && h->cfg.add_shared) mb += (T + rows - 1) / rows;
    const int64_t tiles = mb * (N / 128);
    return (int)std::max<int64_t>(1, std::min<int64_t>(tiles, h->num_sms));
}

int shared_rows(const moe_layer* h, int T)
{
    return (h->cfg.has_shared && h->cfg.add_shared) ? T : 0;
}

// ---- launch pieces (no argument checks; callers validated)

// amax_out: the top-k kernel also folds max |x| into *amax_out (cleared by the router, or
// by the single top-k block when logits are given); returns in *amax_done whether it did.
// zero_words: nzero words the top-k kernel sets to zero (after its wait).
moe_status launch_route(const moe_layer* h, const void* x, const float* logits_in,
                        const float* bias, int T, int32_t* ids, float* w, float* logits_out,
                        float* logits_scratch, uint32_t* status, uint32_t* clear0,
                        uint32_t* clear1, bool pdl, cudaStream_t s, uint32_t* amax_out = nullptr,
                        bool* amax_done = nullptr, int32_t* zero_words = nullptr,
                        int nzero = 0)
{
    const moe_config& c = h->cfg;
    const float* src = logits_in;
    int nsplit = 1;
    if (!logits_in) {
        nsplit = router_splits(T, c.num_experts, c.hidden, h->num_sms);
        CUtensorMap tmX;
        if (!make_tmap(&tmX, x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, c.hidden, T,
                       (uint64_t)c.hidden * 2, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B))
            return MOE_ERR_CUDA;
        const int bn = router_bn(T, c.num_experts);
        dim3 grid(ceil_div(T, 128), ceil_div(c.num_experts, bn), nsplit);
        const moe_status r = launch(router_gemm_kernel, grid, dim3(192), kRouterSmem, s, pdl,
                                    tmX, bn == 160 ? h->tm_router160 : h->tm_router, T,
                                    c.num_experts, c.hidden, c.hidden / nsplit, bn,
                                    logits_scratch, status, clear0, clear1);
        if (r != MOE_OK) return r;
        src = logits_scratch;
        clear0 = clear1 = nullptr;  // done by the router
    } else if (ceil_div(T, topk_tokens_per_block(1)) > 1) {
        // given logits and several top-k blocks: nothing would clear the word before the
        // other blocks fold into it (a single block clears it first itself)
        amax_out = nullptr;
    }
    if (amax_done) *amax_done = amax_out != nullptr;
    // with given logits the top-k kernel is the first of the chain and reads the inputs (x,
    // the logits) before its wait: it starts only when the work before it on the stream is
    // complete (no programmatic launch), so an input written by a kernel that let its
    // dependents start early (a chained forward's combine) is never read too soon
    return launch(topk_kernel_for(c.num_experts), dim3(ceil_div(T, topk_tokens_per_block(nsplit))),
                  dim3(kTopkThreads), topk_smem(nsplit, c.num_experts), s,
                  pdl && !logits_in, src, nsplit,
                  bias, T, c.num_experts, c.top_k, ids, w, logits_out, clear0, clear1,
                  static_cast<const uint16_t*>(x), c.hidden, amax_out, zero_words, nzero);
}

// write_padding: mark padding rows of perm_src with -1 (the staged call's contract; the
// forward's own kernels never read them, so it skips the writes where it can).
moe_status launch_permute(const moe_layer* h, const Plan& p, const int32_t* ids, int T,
                          int32_t* counts, int32_t* offsets, int32_t* perm_src, int32_t* inv,
                          void* ws, bool pdl, cudaStream_t s, bool write_padding = true)
{
    const moe_config& c = h->cfg;
    uint32_t* status = at<uint32_t>(ws, p.status);
    int32_t* hist = at<int32_t>(ws, p.hist);
    int32_t* blkoff = at<int32_t>(ws, p.blkoff);
    int32_t* mb_start = at<int32_t>(ws, p.mb_start);
    if (p.nblk == 1)  // every pair fits one block: the whole grouping in one CTA
        return launch(perm_small_kernel, dim3(1), dim3(1024), perm_small_smem(p.G), s, pdl, ids,
                      p.Tk, c.num_experts, c.local_expert_offset, p.El, T, c.top_k,
                      shared_rows(h, T), p.cap, write_padding ? 1 : 0, counts, offsets,
                      mb_start, perm_src, inv, status);
    moe_status r = launch(perm_hist_kernel, dim3(p.nblk), dim3(256), 0, s, pdl, ids, p.Tk,
                          c.num_experts, c.local_expert_offset, p.El, hist, status);
    if (r == MOE_OK)
        r = launch(perm_scan_kernel, dim3(1), dim3(1024), 0, s, pdl, (const int32_t*)hist,
                   p.nblk, p.El, T, c.top_k, shared_rows(h, T), p.cap, blkoff, counts, offsets,
                   mb_start, perm_src, status);
    if (r == MOE_OK)
        r = launch(perm_scatter_kernel, dim3(p.nblk), dim3(kPairsPerBlock),
                   perm_small_smem(p.El), s, pdl, ids, p.Tk,
                   c.num_experts, c.local_expert_offset, p.El, (const int32_t*)blkoff,
                   (const int32_t*)offsets, p.cap, perm_src, inv);
    return r;
}

// max |x| over the T x H input into the (zeroed) amax word.
moe_status launch_amax(const moe_layer* h, const void* x, int T, uint32_t* amax, bool pdl,
                       cudaStream_t s)
{
    const int64_t n = (int64_t)T * h->cfg.hidden;
    const int blocks = (int)std::min<int64_t>(2 * h->num_sms, std::max<int64_t>(1, n / 2048));
    return launch(amax_bf16_kernel, dim3(blocks), dim3(256), 0, s, pdl,
                  static_cast<const uint16_t*>(x), n, amax);
}

// amax_zeroed: the amax word is zero (no memset); amax_ready: it already holds max |x|
// (folded by the top-k kernel), so no amax pass runs.
moe_status launch_gather(const moe_layer* h, const Plan& p, const void* x, int T,
                         const int32_t* inv, const int32_t* offsets, uint8_t* a_codes,
                         uint8_t* a_sf, void* a_bf16, float* gs_out, void* ws, bool pdl,
                         bool amax_zeroed, cudaStream_t s, bool amax_ready = false)
{
    const moe_config& c = h->cfg;
    const uint16_t* xb = static_cast<const uint16_t*>(x);
    const int add = shared_rows(h, T) > 0 ? 1 : 0;
    // a lane per 64-element k-step for large batches (1 KB pieces per destination row), per
    // 16-element block for small ones (more threads on a latency-bound step)
    const int bpl = T >= 1024 ? 4 : 1;
    const dim3 grid(grid_for((int64_t)T * ((c.hidden / 16 + 32 * bpl - 1) / (32 * bpl)) * 32, 256));
    uint32_t* amax = at<uint32_t>(ws, p.amax);
    const float* gs_static = nullptr;
    if (c.act_mode != MOE_W4A4_STATIC && !amax_ready) {
        if (!amax_zeroed && cudaMemsetAsync(amax, 0, 4, s) != cudaSuccess) return MOE_ERR_CUDA;
        const moe_status r = launch_amax(h, x, T, amax, pdl, s);
        if (r != MOE_OK) return r;
    } else if (c.act_mode == MOE_W4A4_STATIC) {
        gs_static = h->act_gs;  // the handle's device copy of act_global_scale
    }
    if (c.act_mode == MOE_W4A16)
        return launch(gather_f16_kernel,
                      dim3(grid_for((int64_t)T * ((c.hidden + 255) / 256) * 32, 256)), dim3(256),
                      0, s, pdl, xb, T, c.hidden, c.top_k, inv, offsets, p.El, add,
                      (const uint32_t*)amax, static_cast<uint16_t*>(a_bf16), gs_out,
                      (int64_t)p.cap, at<uint32_t>(ws, p.status));
    return launch(gather_quant_kernel_for(bpl), grid, dim3(256), 0, s, pdl, xb, T, c.hidden,
                  c.top_k, inv, offsets, p.El, add, gs_static, (const uint32_t*)amax, a_codes,
                  a_sf, gs_out, (int64_t)p.cap, at<uint32_t>(ws, p.status));
}

// The grouped GEMV takes a W4A16 GEMM when the batch is small and the groups' expected rows
// fit about two chunks (with more rows per group it would decode every weight once per
// further chunk, while the tensor-core kernel's cost does not grow).
bool gemv_shape(const moe_layer* h, const Plan& p)
{
    return p.T <= kGemvMaxTokens &&
           (int64_t)p.T * h->cfg.top_k <= 2LL * kGvChunk * std::max(1, p.El);
}

moe_status launch_gemm(const moe_layer* h, const Plan& p, bool gateup, int epilogue,
                       const uint8_t* a_codes, const uint8_t* a_sf, const float* gs_a,
                       const void* a_bf16, const int32_t* counts, const int32_t* offsets,
                       float* out_f32, uint8_t* out_codes, uint8_t* out_sf, void* out_bf16,
                       const int32_t* perm_src, const float* topk_w, void* ws, bool pdl,
                       cudaStream_t s)
{
    const moe_config& c = h->cfg;
    const bool a16 = c.act_mode == MOE_W4A16;
    const int K = gateup ? c.hidden : c.inter;
    const int N = gateup ? 2 * c.inter : c.hidden;
    GemmArgs args;
    memset(&args, 0, sizeof(args));
    args.a_sf = a_sf;
    args.b_tiles = gateup ? h->w13 : h->w2;
    args.gs_a = gs_a;
    args.gs_w = gateup ? h->gs13 : h->gs2;
    args.counts = counts;
    args.offsets = offsets;
    args.mb_start = at<int32_t>(ws, p.mb_start);
    args.G = p.G;
    args.N = N;
    args.K = K;
    args.epilogue = epilogue;
    args.gs_i = c.inter_global_scale;
    args.out_f32 = out_f32;
    args.out_codes = out_codes;
    args.out_sf = out_sf;
    args.out_bf16 = static_cast<uint16_t*>(out_bf16);
    args.perm_src = perm_src;
    args.topk_w = topk_w;
    args.Tk = p.Tk;
    args.inter_amax = at<uint32_t>(ws, p.amax) + 1;
    args.gs_i_dev = (is_down(epilogue) && dynamic_inter(c)) ? at<float>(ws, p.gs_i) : nullptr;
    if (epilogue == kEpiDownF16) {  // the y buffer holds fp16 rows; their scales beside it
        args.out_bf16 = reinterpret_cast<uint16_t*>(out_f32);
        args.out_f32 = nullptr;
        args.y_scale = at<float>(ws, p.y_scale);
    }
    args.status = at<uint32_t>(ws, p.status);
    if (a16) {
        // Few token rows per group: the CUDA-core GEMV reads each weight once per chunk of
        // kGvChunk rows, where a 128-row MMA per 16 k would be mostly padding.
        const int list_cap = p.gv_list_cap;
        const int slots = gemv_w4a16_slots(K, list_cap);
        if (gemv_shape(h, p) && epilogue != kEpiGateUpSwigluF32 && slots >= 4) {
            const size_t gsm = gemv_w4a16_smem(K, slots, list_cap);
            const int64_t items = (int64_t)list_cap * (N / 128);
            const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(h->num_sms, items));
            return launch(gemv_w4a16_kernel_for(gateup), dim3(grid), dim3(kGvThreads), gsm, s,
                          pdl, args, static_cast<const uint16_t*>(a_bf16), list_cap, slots);
        }
        // Token rows per tile from the expected rows per local expert: narrow tiles keep the
        // token tile (re-read for every weight tile) small when experts see few tokens.
        const int64_t local_rows = (int64_t)p.T * c.top_k / std::max(1, c.num_local_experts);
        const int bn = local_rows <= 16 ? 16 : local_rows <= 32 ? 32 : 64;
        // shared memory split between raw weight blobs and token tiles, both rings kept
        // at least 4 blobs deep
        args.raw_slots = kW16MaxRaw;
        args.stages = kW16MaxB;
        while (w4a16_smem_bytes(args.raw_slots, args.stages, bn, p.G) > kSmemLimit &&
               (args.raw_slots > 4 || args.stages > 4)) {
            if (args.stages * 4 * bn * 128 >= args.raw_slots * kNvf4TileBytes && args.stages > 4)
                --args.stages;
            else if (args.raw_slots > 4)
                --args.raw_slots;
            else
                --args.stages;
        }
        const int smem = w4a16_smem_bytes(args.raw_slots, args.stages, bn, p.G);
        if (smem > kSmemLimit) return MOE_ERR_UNSUPPORTED;
        // gate_up reads the fp16 activation rows (x * gs_a), down the bf16 intermediate
        CUtensorMap tmB;
        if (!make_tmap(&tmB, a_bf16,
                       gateup ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                       K, p.cap, (uint64_t)K * 2, 64, bn, CU_TENSOR_MAP_SWIZZLE_128B))
            return MOE_ERR_CUDA;
        return launch(w4a16_kernel(bn, gateup), dim3(gemm_grid(h, p.T, N, bn)),
                      dim3(kW16Threads), smem, s, pdl, tmB, args);
    }
    CUtensorMap tmA, tmA16, tmY;
    memset(&tmY, 0, sizeof(tmY));
    const int grid = gemm_grid(h, p.T, N, 128);
    const int pitch = codes_pitch(K);
    if (use_token_tiles(h, p.T)) {
        args.rb_cap = p.cap / 128;
        args.tile_n = kTokenTileRows;
        args.stages = kMaxStages;
        while (args.stages > 2 &&
               gemm_swap_smem_bytes(args.stages, args.tile_n, p.G) > kSmemLimit)
            --args.stages;
        const int smem = gemm_swap_smem_bytes(args.stages, args.tile_n, p.G);
        if (smem > kSmemLimit) return MOE_ERR_UNSUPPORTED;
        if (!make_tmap(&tmA, a_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, pitch, p.cap, pitch, 128,
                       128, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !make_tmap(&tmA16, a_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, pitch, p.cap, pitch, 128,
                       16, CU_TENSOR_MAP_SWIZZLE_128B))
            return MOE_ERR_CUDA;
        // kEpiDownF16 stores y in 32 x 32 fp16 boxes (64-byte rows, 64-byte swizzle)
        if (epilogue == kEpiDownF16 &&
            !make_tmap(&tmY, out_f32, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, N, p.cap, (uint64_t)N * 2,
                       32, 32, CU_TENSOR_MAP_SWIZZLE_64B))
            return MOE_ERR_CUDA;
        return launch(gemm_nvf4_swap_kernel, dim3(grid), dim3(kSwThreads), smem, s, pdl, tmA,
                      tmA16, tmY, args);
    }
    const int stage_bytes = kNvf4StageBytes;
    // Kernel configuration from the expected LOCAL load (rows per local expert), as the
    // pages' backend choice is re-tuned on the local rather than the global workload: with
    // few rows per 128-row block the down epilogue stores directly and the shared memory
    // goes to one more pipeline stage; with many it stages TMA stores.
    const int64_t local_rows = (int64_t)p.T * c.top_k / std::max(1, c.num_local_experts);
    args.staging = (is_down(epilogue) && local_rows >= 16) ? kDownStaging : 0;
    args.rb_cap = p.cap / 128;
    if (epilogue == kEpiDown &&
        !make_tmap(&tmY, out_f32, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, N, p.cap, (uint64_t)N * 4, 32,
                   32, CU_TENSOR_MAP_SWIZZLE_128B))
        return MOE_ERR_CUDA;
    if (epilogue == kEpiDownF16 &&
        !make_tmap(&tmY, out_f32, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, N, p.cap, (uint64_t)N * 2, 32,
                   32, CU_TENSOR_MAP_SWIZZLE_64B))
        return MOE_ERR_CUDA;
    if (use_wide(h, p.T, N)) {
        // fp16 y is staged through shared memory (2 KB boxes); fp32 y is stored directly
        args.staging = (epilogue == kEpiDownF16 && local_rows >= 16) ? kWideDownStaging : 0;
        args.stages = gemm_stages(5, kWideStageBytes, args.staging, p.G, args.rb_cap);
        const int smem =
            gemm_smem_bytes(args.stages, kWideStageBytes, args.staging, p.G, args.rb_cap);
        if (smem > kSmemLimit) return MOE_ERR_UNSUPPORTED;
        if (!make_tmap(&tmA, a_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, pitch, p.cap, pitch, 128,
                       128, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !make_tmap(&tmA16, a_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, pitch, p.cap, pitch, 128,
                       16, CU_TENSOR_MAP_SWIZZLE_128B))
            return MOE_ERR_CUDA;
        return launch(gemm_nvf4_wide_kernel, dim3(gemm_grid(h, p.T, N / 2, 128)),
                      dim3(kWideThreads), smem, s, pdl, tmA, tmA16, tmY, args);
    }
    if (use_pairs(h, p.T)) {
        args.stages = kMaxStages;
        while (args.stages > 2 && gemm_pair_smem_bytes(args.stages, args.staging, p.G,
                                                       args.rb_cap) > kSmemLimit)
            --args.stages;
        const int smem = gemm_pair_smem_bytes(args.stages, args.staging, p.G, args.rb_cap);
        if (smem > kSmemLimit) return MOE_ERR_UNSUPPORTED;
        if (!make_tmap(&tmA, a_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, pitch, p.cap, pitch, 128,
                       128, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !make_tmap(&tmA16, a_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, pitch, p.cap, pitch, 128,
                       16, CU_TENSOR_MAP_SWIZZLE_128B))
            return MOE_ERR_CUDA;
        const int pairs = std::max(1, std::min(std::min(grid, h->num_sms) / 2, h->max_pairs));
        return launch_pairs(gemm_nvf4_pair_kernel, dim3(2 * pairs), dim3(kNvf4Threads), smem, s,
                            pdl, tmA, tmA16, tmY, args);
    }
    args.stages = gemm_stages(6, stage_bytes, args.staging, p.G, args.rb_cap);
    const int smem = gemm_smem_bytes(args.stages, stage_bytes, args.staging, p.G, args.rb_cap);
    if (smem > kSmemLimit) return MOE_ERR_UNSUPPORTED;
    if (!make_tmap(&tmA, a_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, pitch, p.cap, pitch, 128, 128,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tmap(&tmA16, a_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, pitch, p.cap, pitch, 128, 16,
                   CU_TENSOR_MAP_SWIZZLE_128B))
        return MOE_ERR_CUDA;
    return launch(gemm_nvf4_kernel, dim3(grid), dim3(kNvf4Threads), smem, s, pdl, tmA, tmA16,
                  tmY, args);
}

// Ring slots of the fused W4A16 GEMV (gemv_w4a16_fused_kernel: the forward's gate_up and
// down in one launch) for this forward, or 0 when the forward runs them as separate kernels.
int fused_gemv_slots(const moe_layer* h, const Plan& p)
{
    const moe_config& c = h->cfg;
    if (c.act_mode != MOE_W4A16 || p.T < 1 || !gemv_shape(h, p)) return 0;
    const int slots = gemv_w4a16_fused_slots(c.hidden, std::min(kGvChunk, p.T), p.gv_list_cap);
    return slots >= 4 ? slots : 0;
}

// The fused W4A16 GEMV: activation rows from x (prescaled by max |x| in the workspace), the
// intermediate into i_bf16, the weighted expert outputs into y (fp32 rows).  The ready counts
// (gv_sync) were zeroed by the routing kernel of the same forward.
// one_block_pred: the kernel before it is the one-block grouping kernel; the grid then leaves
// one SM free for it, so that no block of this launch starts after it (one token: 41.3 vs
// 42.4 us a forward; with more blocks before it, all SMs: 256 tokens 702 vs 704 us).
moe_status launch_gemv_fused(const moe_layer* h, const Plan& p, const void* x, void* ws,
                             int slots, bool one_block_pred, bool pdl, cudaStream_t s)
{
    const moe_config& c = h->cfg;
    GvFusedArgs f;
    memset(&f, 0, sizeof(f));
    for (GemmArgs* a : {&f.gu, &f.dn}) {
        a->counts = at<int32_t>(ws, p.counts);
        a->offsets = at<int32_t>(ws, p.offsets);
        a->G = p.G;
        a->perm_src = at<int32_t>(ws, p.perm_src);
        a->Tk = p.Tk;
        a->status = at<uint32_t>(ws, p.status);
    }
    f.gu.b_tiles = h->w13;
    f.gu.gs_w = h->gs13;
    f.gu.N = 2 * c.inter;
    f.gu.K = c.hidden;
    f.gu.epilogue = kEpiGateUpSwiglu;
    f.gu.out_bf16 = at<uint16_t>(ws, p.i_bf16);
    f.dn.b_tiles = h->w2;
    f.dn.gs_w = h->gs2;
    f.dn.N = c.hidden;
    f.dn.K = c.inter;
    f.dn.epilogue = kEpiDown;
    f.dn.out_f32 = at<float>(ws, p.y);
    f.dn.topk_w = at<float>(ws, p.w);
    f.ids = at<int32_t>(ws, p.ids);
    f.E = c.num_experts;
    f.off = c.local_expert_offset;
    f.shared_rows = shared_rows(h, p.T);
    f.x = static_cast<const uint16_t*>(x);
    f.amax = at<uint32_t>(ws, p.amax);
    f.gs_out = at<float>(ws, p.gs_a);
    f.T = p.T;
    f.k = p.k;
    f.tok_rows = std::min(kGvChunk, p.T);
    f.ready = at<int32_t>(ws, p.gv_sync);
    f.part = at<float>(ws, p.gv_part);
    const int64_t items =
        (int64_t)p.gv_list_cap * ((2 * c.inter / 128) * kGvMaxSplit + c.hidden / 128);
    const int sms = one_block_pred && h->num_sms > 1 ? h->num_sms - 1 : h->num_sms;
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(sms, items));
    return launch_coop(gemv_w4a16_fused_kernel_ptr(), dim3(grid), dim3(kGvFusedThreads),
                  gemv_w4a16_fused_smem(c.hidden, f.tok_rows, slots, p.gv_list_cap), s, pdl, f,
                  p.gv_list_cap, slots);
}

}  // namespace

namespace {

// gate_up with the fused SwiGLU epilogue.  Static intermediate scale: one pass that writes
// the NVFP4 intermediate.  Dynamic: the epilogue writes the fp32 intermediate and folds
// amax |s| into the workspace (the caller zeroed it), then quant_inter_kernel quantises it
// with 2688 / amax and stores gs_i for the down GEMM.
moe_status launch_gateup_fused(const moe_layer* h, const Plan& p, const uint8_t* a_codes,
                               const uint8_t* a_sf, const float* gs_a, const void* a_bf16,
                               const int32_t* counts, const int32_t* offsets, uint8_t* i_codes,
                               uint8_t* i_sf, void* i_bf16, void* ws, bool pdl, cudaStream_t s)
{
    if (!dynamic_inter(h->cfg))
        return launch_gemm(h, p, true, kEpiGateUpSwiglu, a_codes, a_sf, gs_a, a_bf16, counts,
                           offsets, nullptr, i_codes, i_sf, i_bf16, nullptr, nullptr, ws, pdl, s);
    float* sbuf = at<float>(ws, p.s_f32);
    const moe_status r = launch_gemm(h, p, true, kEpiGateUpSwigluF32, a_codes, a_sf, gs_a,
                                     a_bf16, counts, offsets, sbuf, nullptr, nullptr, nullptr,
                                     nullptr, nullptr, ws, pdl, s);
    if (r != MOE_OK) return r;
    // upper bound on the 128-row blocks (the exact count is on the device)
    const int64_t P = (int64_t)p.T * p.k;
    const int64_t blocks = (P + 127) / 128 + std::min<int64_t>(p.El, P) +
                           ((int64_t)shared_rows(h, p.T) + 127) / 128;
    return launch(quant_inter_kernel, dim3((unsigned)std::max<int64_t>(1, blocks)), dim3(256), 0,
                  s, pdl, (const float*)sbuf, counts, offsets,
                  (const int32_t*)at<int32_t>(ws, p.mb_start), p.G, p.I,
                  (const uint32_t*)(at<uint32_t>(ws, p.amax) + 1), i_codes, i_sf,
                  at<float>(ws, p.gs_i));
}

// Large batches move the y rows with bulk copies (combine_tma_kernel): pieces of cw columns,
// the widest of 2048 / 1024 / 512 that divides H and lets two ring slots fit (wide pieces
// stream better than deep rings of narrow ones: 8 KB pieces in 2 slots took 290 us for the
// prefill combine, 4 KB pieces in 5 slots 411 us); the sums are the same as combine_kernel's.
constexpr int kCombineTmaMinTokens = 1024;
constexpr size_t kCombineSmemBudget = 220 * 1024;

// y: fp32 rows, or (y_scale non-null) fp16 rows each times y_scale[row].
moe_status launch_combine(const moe_layer* h, const void* y, const int32_t* inv,
                          const int32_t* offsets, int T, void* out, bool pdl, cudaStream_t s,
                          uint32_t* status = nullptr, const float* y_scale = nullptr)
{
    const moe_config& c = h->cfg;
    const int add = shared_rows(h, T) > 0 ? 1 : 0;
    const int nrows = c.top_k + add;
    const size_t es = y_scale ? 2 : 4;  // bytes per element of y
    if (T >= kCombineTmaMinTokens && nrows > 0 &&
        (reinterpret_cast<uintptr_t>(y) & 15) == 0 && (reinterpret_cast<uintptr_t>(out) & 7) == 0) {
        int cw = 0;  // pieces of at most 8 KB (the measured best), two slots at least
        for (int w : {4096, 2048, 1024, 512})
            if (c.hidden % w == 0 && w * es <= 8192 &&
                2 * (size_t)nrows * w * es <= kCombineSmemBudget) {
                cw = w;
                break;
            }
        if (cw) {
            const int nslots = (int)std::min<size_t>(
                kCombineMaxSlots, kCombineSmemBudget / ((size_t)nrows * cw * es));
            const int64_t units = (int64_t)T * (c.hidden / cw);
            return launch(combine_tma_kernel,
                          dim3((unsigned)std::min<int64_t>(units, h->num_sms)),
                          dim3(kCombineTmaThreads), combine_tma_smem(nrows, cw, nslots, (int)es),
                          s, pdl, y, y_scale, inv, offsets, c.num_local_experts, T, c.hidden,
                          c.top_k, add, cw, nslots, static_cast<uint16_t*>(out), status,
                          (int64_t)rows_cap(c, T));
        }
    }
    return launch(combine_kernel, dim3(grid_for((int64_t)T * (c.hidden / 8), 256)), dim3(256), 0,
                  s, pdl, y, y_scale, inv, offsets, c.num_local_experts, T, c.hidden, c.top_k,
                  shared_rows(h, T) > 0 ? 1 : 0, static_cast<uint16_t*>(out),
                  (int64_t)rows_cap(c, T), status);
}

}  // namespace

// ================================================================ routing without allocation
//
// Scratch for moe_route_topk_noalloc: the router's partial-sum logit planes live in this
// file-scope device array instead of a caller workspace, and its last 256 bytes hold the
// call's status word (set by the router when a bounded wait runs out).  Every device that
// loads the library holds it (8 MiB) until the process exits.  Host code may not pass the
// symbol itself to a kernel (on the host it only names a stand-in); the device address is
// looked up with cudaGetSymbolAddress, with that device current, once per device and
// context.
constexpr size_t kRouteScratchBytes = size_t(8) << 20;
constexpr size_t kRouteStatusBytes = 256;
constexpr size_t kRoutePlaneFloats = (kRouteScratchBytes - kRouteStatusBytes) / sizeof(float);
static __device__ __align__(256) float g_route_scratch[kRouteScratchBytes / sizeof(float)];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_route_scratch_mu;
float* g_route_scratch_ptr[kMaxDevices] = {};
void* g_route_scratch_ctx[kMaxDevices] = {};

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

// The current driver context (nullptr if it cannot be read): the cached symbol address is
// valid only for the context it was looked up in (a cudaDeviceReset makes a new one).
void* current_context()
{
    static CtxGetCurrentFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetCurrentFn>(p);
    });
    CUcontext c = nullptr;
    if (!fn || fn(&c) != CUDA_SUCCESS) return nullptr;
    return c;
}

// Device address of g_route_scratch on the current device and context (looked up on the
// first use in each).
moe_status route_scratch_address(float** out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
    void* ctx = current_context();
    std::lock_guard<std::mutex> lock(g_route_scratch_mu);
    if (!g_route_scratch_ptr[dev] || !ctx || ctx != g_route_scratch_ctx[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            g_route_scratch_ptr[dev] = nullptr;
            return MOE_ERR_CUDA;
        }
        g_route_scratch_ptr[dev] = static_cast<float*>(p);
        g_route_scratch_ctx[dev] = ctx;
    }
    *out = g_route_scratch_ptr[dev];
    return MOE_OK;
}

}  // namespace

namespace moe {

// After the top-k: if the router flagged a wait that ran out, its planes are incomplete,
// so every id becomes -1 (a pair every later step drops) and every weight 0.
__global__ void route_invalidate_kernel(const uint32_t* status, int n, int32_t* ids, float* w)
{
    if (*status == 0u) return;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
        ids[i] = -1;
        w[i] = 0.0f;
    }
}

}  // namespace moe

// ================================================================ C ABI

extern "C" {

const char* moe_status_string(moe_status s)
{
    switch (s) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID: return "invalid argument";
        case MOE_ERR_UNSUPPORTED: return "unsupported shape or mode";
        case MOE_ERR_CUDA: return "CUDA error";
        case MOE_ERR_WORKSPACE: return "workspace too small";
        case MOE_ERR_TIMEOUT: return "device wait timed out";
        case MOE_ERR_DEVICE_STATUS: return "device flagged bad data";
    }
    return "unknown status";
}

int32_t moe_rows_capacity(const moe_config* cfg, int32_t T)
{
    if (!cfg || T < 0) return -1;
    return rows_cap(*cfg, T);
}

size_t moe_workspace_size(const moe_config* cfg, int32_t T)
{
    moe_status why;
    if (!valid_cfg(cfg, &why) || T < 0) return 0;
    return plan(*cfg, T).total;
}

void moe_destroy(moe_handle h)
{
    if (!h) return;
    cudaFree(h->router_w);
    cudaFree(h->w13);
    cudaFree(h->w2);
    cudaFree(h->gs13);
    cudaFree(h->gs2);
    cudaFree(h->act_gs);
    delete h;
}

moe_status moe_create(const moe_config* cfg, const moe_weights* w, moe_stream_t stream,
                      moe_handle* out)
{
    const NvtxRange nvtx_range("moe_create");
    if (!out) return MOE_ERR_INVALID;
    *out = nullptr;
    moe_status why;
    if (!valid_cfg(cfg, &why)) return why;
    if (!w || !w->router_w_d) return MOE_ERR_INVALID;
    const int El = cfg->num_local_experts, H = cfg->hidden, I = cfg->inter;
    if (El > 0 && (!w->w13_d || !w->w13_sf_d || !w->w13_gs_d || !w->w2_d || !w->w2_sf_d ||
                   !w->w2_gs_d))
        return MOE_ERR_INVALID;
    if (cfg->has_shared && (!w->sh13_d || !w->sh13_sf_d || !w->sh13_gs_d || !w->sh2_d ||
                            !w->sh2_sf_d || !w->sh2_gs_d))
        return MOE_ERR_INVALID;
    if (!encode_fn()) return MOE_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    moe_layer* h = new (std::nothrow) moe_layer();
    if (!h) return MOE_ERR_CUDA;
    h->cfg = *cfg;
    if (cudaGetDevice(&h->device) != cudaSuccess ||
        cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device) !=
            cudaSuccess) {
        delete h;
        return MOE_ERR_CUDA;
    }
    const int G = El + 1;
    const int pairs = cfg->act_mode == MOE_W4A16 ? 1 : 0;  // W4A16 down: nibble order
    const size_t b13 = blob_bytes(2 * I, H), b2 = blob_bytes(H, I);
    bool ok = cudaMalloc(&h->router_w, (size_t)cfg->num_experts * H * 2) == cudaSuccess &&
              cudaMalloc(&h->w13, G * b13) == cudaSuccess &&
              cudaMalloc(&h->w2, G * b2) == cudaSuccess &&
              cudaMalloc(&h->gs13, G * 4) == cudaSuccess &&
              cudaMalloc(&h->gs2, G * 4) == cudaSuccess &&
              cudaMalloc(&h->act_gs, 4) == cudaSuccess &&
              cudaMemcpy(h->act_gs, &cfg->act_global_scale, 4, cudaMemcpyHostToDevice) ==
                  cudaSuccess;
    ok = ok && cudaMemsetAsync(h->w13, 0, G * b13, s) == cudaSuccess &&
         cudaMemsetAsync(h->w2, 0, G * b2, s) == cudaSuccess &&
         cudaMemsetAsync(h->gs13, 0, G * 4, s) == cudaSuccess &&
         cudaMemsetAsync(h->gs2, 0, G * 4, s) == cudaSuccess;
    ok = ok && cudaMemcpyAsync(h->router_w, w->router_w_d, (size_t)cfg->num_experts * H * 2,
                               cudaMemcpyDeviceToDevice, s) == cudaSuccess;
    const int blocks = 8 * h->num_sms;
    if (ok && El > 0) {
        repack_tiles_kernel<<<blocks, 256, 0, s>>>(w->w13_d, w->w13_sf_d, El, 2 * I, H, 1, 0,
                                                   h->w13);
        repack_tiles_kernel<<<blocks, 256, 0, s>>>(w->w2_d, w->w2_sf_d, El, H, I, 0, pairs, h->w2);
        ok = cudaMemcpyAsync(h->gs13, w->w13_gs_d, El * 4, cudaMemcpyDeviceToDevice, s) ==
                 cudaSuccess &&
             cudaMemcpyAsync(h->gs2, w->w2_gs_d, El * 4, cudaMemcpyDeviceToDevice, s) ==
                 cudaSuccess;
    }
    if (ok && cfg->has_shared) {
        repack_tiles_kernel<<<blocks, 256, 0, s>>>(w->sh13_d, w->sh13_sf_d, 1, 2 * I, H, 1, 0,
                                                   h->w13 + (size_t)El * b13);
        repack_tiles_kernel<<<blocks, 256, 0, s>>>(w->sh2_d, w->sh2_sf_d, 1, H, I, 0, pairs,
                                                   h->w2 + (size_t)El * b2);
        ok = cudaMemcpyAsync(h->gs13 + El, w->sh13_gs_d, 4, cudaMemcpyDeviceToDevice, s) ==
                 cudaSuccess &&
             cudaMemcpyAsync(h->gs2 + El, w->sh2_gs_d, 4, cudaMemcpyDeviceToDevice, s) ==
                 cudaSuccess;
    }
    ok = ok && cudaGetLastError() == cudaSuccess && cudaStreamSynchronize(s) == cudaSuccess;
    ok = ok && make_tmap(&h->tm_router, h->router_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, H,
                         cfg->num_experts, (uint64_t)H * 2, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B) &&
         make_tmap(&h->tm_router160, h->router_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, H,
                   cfg->num_experts, (uint64_t)H * 2, 64, 160, CU_TENSOR_MAP_SWIZZLE_128B);
    ok = ok &&
         cudaFuncSetAttribute(router_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kRouterSmem) == cudaSuccess &&
         cudaFuncSetAttribute(perm_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              perm_small_smem(kMaxExperts + 1)) == cudaSuccess &&
         cudaFuncSetAttribute(perm_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              perm_small_smem(kMaxExperts)) == cudaSuccess &&
         cudaFuncSetAttribute(combine_tma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)combine_tma_smem(1, (int)(kCombineSmemBudget / 4), 1)) ==
             cudaSuccess &&
         set_topk_smem_limits() &&
         cudaFuncSetAttribute(gemm_nvf4_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kSmemLimit) == cudaSuccess &&
         cudaFuncSetAttribute(gemm_nvf4_swap_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kSmemLimit) == cudaSuccess &&
         cudaFuncSetAttribute(gemm_nvf4_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kSmemLimit) == cudaSuccess &&
         cudaFuncSetAttribute(gemm_nvf4_wide_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kSmemLimit) == cudaSuccess &&
         set_w4a16_smem_limits();
    if (ok) {  // how many CTA pairs of the pair kernel fit the GPU at once (its grid)
        cudaLaunchConfig_t lc = {};
        lc.gridDim = dim3(2 * (h->num_sms / 2));
        lc.blockDim = dim3(kNvf4Threads);
        lc.dynamicSmemBytes = kSmemLimit;
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = 2;
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = 1;
        lc.attrs = at;
        lc.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, gemm_nvf4_pair_kernel, &lc) != cudaSuccess || n <= 0) {
            cudaGetLastError();
            n = h->num_sms / 2;
        }
        h->max_pairs = n;
    }
    if (!ok) {
        cudaGetLastError();
        moe_destroy(h);
        return MOE_ERR_CUDA;
    }
    *out = h;
    return MOE_OK;
}

moe_status moe_route_topk(moe_handle h, const void* x_bf16_d, const float* logits_in_d,
                          const float* logit_bias_d, int32_t T, int32_t* topk_ids_d,
                          float* topk_w_d, float* logits_out_d, void* ws_d, size_t ws_bytes,
                          moe_stream_t stream)
{
    const NvtxRange nvtx_range("moe_route_topk");
    if (!h || !t_ok(h, T) || !topk_ids_d || !topk_w_d) return MOE_ERR_INVALID;
    if (!logits_in_d && !x_bf16_d) return MOE_ERR_INVALID;
    if (T == 0) return MOE_OK;
    float* scratch = nullptr;
    uint32_t* status = nullptr;
    if (!logits_in_d) {
        if (reinterpret_cast<uintptr_t>(x_bf16_d) & 15) return MOE_ERR_INVALID;
        const moe_status st = check_ws(h, T, ws_d, ws_bytes);
        if (st != MOE_OK) return st;
        const Plan p = plan(h->cfg, T);
        scratch = at<float>(ws_d, p.logits);
        status = at<uint32_t>(ws_d, p.status);
    }
    return launch_route(h, x_bf16_d, logits_in_d, logit_bias_d, T, topk_ids_d, topk_w_d,
                        logits_out_d, scratch, status, nullptr, nullptr, false,
                        reinterpret_cast<cudaStream_t>(stream));
}

moe_status moe_permute(moe_handle h, const int32_t* topk_ids_d, int32_t T,
                       int32_t* expert_counts_d, int32_t* expert_offsets_d,
                       int32_t* perm_src_d, int32_t* inv_d, void* ws_d, size_t ws_bytes,
                       moe_stream_t stream)
{
    const NvtxRange nvtx_range("moe_permute");
    if (!h || !t_ok(h, T) || !topk_ids_d || !expert_counts_d || !expert_offsets_d ||
        !perm_src_d || !inv_d)
        return MOE_ERR_INVALID;
    if (T == 0) return MOE_OK;  // nothing to do: no workspace needed
    const moe_status st = check_ws(h, T, ws_d, ws_bytes);
    if (st != MOE_OK) return st;
    const Plan p = plan(h->cfg, T);
    return launch_permute(h, p, topk_ids_d, T, expert_counts_d, expert_offsets_d, perm_src_d,
                          inv_d, ws_d, false, reinterpret_cast<cudaStream_t>(stream));
}

moe_status moe_quant_nvfp4(const void* x_bf16_d, int32_t rows, int32_t cols,
                           const float* gs_in_d, float* gs_out_d, uint8_t* codes_d,
                           uint8_t* sf_d, int32_t sf_layout, void* ws_d, size_t ws_bytes,
                           moe_stream_t stream)
{
    const NvtxRange nvtx_range("moe_quant_nvfp4");
    if (!x_bf16_d || !codes_d || !sf_d || rows < 0 || cols <= 0) return MOE_ERR_INVALID;
    if (sf_layout != 0 && sf_layout != 1) return MOE_ERR_INVALID;
    if (cols % 64) return MOE_ERR_UNSUPPORTED;
    if (!gs_in_d && (!ws_d || ws_bytes < 4)) return MOE_ERR_WORKSPACE;
    if (rows == 0) return MOE_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const uint16_t* x = static_cast<const uint16_t*>(x_bf16_d);
    uint32_t* amax = static_cast<uint32_t*>(ws_d);
    if (!gs_in_d) {
        if (cudaMemsetAsync(amax, 0, 4, s) != cudaSuccess) return MOE_ERR_CUDA;
        int dev = 0, sms = 148;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        const int64_t n = (int64_t)rows * cols;
        const int blocks = (int)std::min<int64_t>(2 * sms, std::max<int64_t>(1, n / 2048));
        amax_bf16_kernel<<<blocks, 256, 0, s>>>(x, n, amax);
    }
    quant_rows_kernel<<<grid_for((int64_t)rows * 32, 256), 256, 0, s>>>(
        x, rows, cols, gs_in_d, gs_in_d ? nullptr : amax, codes_d, sf_d, sf_layout, gs_out_d);
    return check_launch();
}

moe_status moe_gather_activations(moe_handle h, const void* x_bf16_d, int32_t T,
                                  const int32_t* inv_d, const int32_t* expert_offsets_d,
                                  uint8_t* a_codes_d, uint8_t* a_sf_d, void* a_bf16_d,
                                  float* gs_out_d, void* ws_d, size_t ws_bytes,
                                  moe_stream_t stream)
{
    const NvtxRange nvtx_range("moe_gather_activations");
    if (!h || !t_ok(h, T) || !x_bf16_d || !inv_d || !expert_offsets_d) return MOE_ERR_INVALID;
    if (h->cfg.act_mode == MOE_W4A16 ? !a_bf16_d : (!a_codes_d || !a_sf_d || !gs_out_d))
        return MOE_ERR_INVALID;
    if (T == 0) return MOE_OK;  // nothing to do: no workspace needed
    const moe_status st = check_ws(h, T, ws_d, ws_bytes);
    if (st != MOE_OK) return st;
    const Plan p = plan(h->cfg, T);
    return launch_gather(h, p, x_bf16_d, T, inv_d, expert_offsets_d, a_codes_d, a_sf_d,
                         a_bf16_d, gs_out_d, ws_d, false, false,
                         reinterpret_cast<cudaStream_t>(stream));
}

moe_status moe_grouped_gemm_gateup(moe_handle h, const uint8_t* a_codes_d,
                                   const uint8_t* a_sf_d, const float* gs_a_d,
                                   const void* a_bf16_d, const int32_t* expert_counts_d,
                                   const int32_t* expert_offsets_d, int32_t fuse_epilogue,
                                   float* gateup_f32_d, uint8_t* inter_codes_d,
                                   uint8_t* inter_sf_d, void* inter_bf16_d, int32_t T,
                                   void* ws_d, size_t ws_bytes, moe_stream_t stream)
{
    const NvtxRange nvtx_range("moe_grouped_gemm_gateup");
    if (!h || !t_ok(h, T) || !expert_counts_d || !expert_offsets_d) return MOE_ERR_INVALID;
    const bool a16 = h->cfg.act_mode == MOE_W4A16;
    // gs_a: the activation global scale (W4A4) or the fp16 prescale (W4A16); both modes
    // read it on the device
    if (!gs_a_d || (a16 ? !a_bf16_d : (!a_codes_d || !a_sf_d))) return MOE_ERR_INVALID;
    if (fuse_epilogue) {
        if (a16 ? !inter_bf16_d : (!inter_codes_d || !inter_sf_d)) return MOE_ERR_INVALID;
    } else if (!gateup_f32_d) {
        return MOE_ERR_INVALID;
    }
    if (T == 0) return MOE_OK;  // nothing to do: no workspace needed
    const moe_status st = check_ws(h, T, ws_d, ws_bytes);
    if (st != MOE_OK) return st;
    const Plan p = plan(h->cfg, T);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (!fuse_epilogue)
        return launch_gemm(h, p, true, kEpiGateUpF32, a_codes_d, a_sf_d, gs_a_d, a_bf16_d,
                           expert_counts_d, expert_offsets_d, gateup_f32_d, nullptr, nullptr,
                           nullptr, nullptr, nullptr, ws_d, false, s);
    if (dynamic_inter(h->cfg) &&
        cudaMemsetAsync(at<uint32_t>(ws_d, p.amax) + 1, 0, 4, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    return launch_gateup_fused(h, p, a_codes_d, a_sf_d, gs_a_d, a_bf16_d, expert_counts_d,
                               expert_offsets_d, inter_codes_d, inter_sf_d, inter_bf16_d, ws_d,
                               false, s);
}

moe_status moe_prepare_weights(const uint8_t* codes_d, const uint8_t* sf_d, const float* glob_d,
                               int32_t num_experts, int32_t N, int32_t K, int32_t convention,
                               float fold_target, int32_t swap_halves, int32_t off,
                               int32_t count, uint8_t* codes_out_d, uint8_t* sf_out_d,
                               float* gs_out_d, moe_stream_t stream)
{
    const NvtxRange nvtx_range("moe_prepare_weights");
    if (N <= 0 || K <= 0 || num_experts < 0 || off < 0 || count < 0 ||
        (int64_t)off + count > num_experts)
        return MOE_ERR_INVALID;
    if ((convention != MOE_GS_ENCODE && convention != MOE_GS_DEQUANT) ||
        !(fold_target >= 0.0f) || isinf(fold_target) || (swap_halves && (N & 1)))
        return MOE_ERR_INVALID;
    if (K % 64) return MOE_ERR_UNSUPPORTED;
    if (count == 0) return MOE_OK;  // an empty slice: nothing to read or write
    if (!codes_d || !sf_d || !glob_d || !codes_out_d || !sf_out_d || !gs_out_d)
        return MOE_ERR_INVALID;
    if ((reinterpret_cast<uintptr_t>(codes_d) | reinterpret_cast<uintptr_t>(codes_out_d)) & 15)
        return MOE_ERR_INVALID;
    // a warp per output row, 8 rows per block, up to 16 blocks per SM (grid-stride)
    const int64_t blocks = ((int64_t)count * N + 7) / 8;
    prepare_weights_kernel<<<(unsigned)std::min<int64_t>(blocks, 152 * 16), 256, 0,
                             reinterpret_cast<cudaStream_t>(stream)>>>(
        codes_d, sf_d, glob_d, N, K, convention, fold_target, swap_halves ? 1 : 0, off, count,
        codes_out_d, sf_out_d, gs_out_d);
    return check_launch();
}

moe_status moe_swiglu_requant(const float* gateup_f32_d, int32_t rows, int32_t inter,
                              float gs_i, uint8_t* codes_d, uint8_t* sf_d, int32_t sf_layout,
                              moe_stream_t stream)
{
    const NvtxRange nvtx_range("moe_swiglu_requant");
    if (!gateup_f32_d || !codes_d || !sf_d || rows < 0 || inter <= 0 || !(gs_i > 0.0f))
        return MOE_ERR_INVALID;
    if (sf_layout != 0 && sf_layout != 1) return MOE_ERR_INVALID;
    if (inter % 64) return MOE_ERR_UNSUPPORTED;
    if (rows == 0) return MOE_OK;
    swiglu_requant_kernel<<<grid_for((int64_t)rows * 32, 256), 256, 0,
                            reinterpret_cast<cudaStream_t>(stream)>>>(
        gateup_f32_d, rows, inter, gs_i, codes_d, sf_d, sf_layout);
    return check_launch();
}

moe_status moe_grouped_gemm_down(moe_handle h, const uint8_t* inter_codes_d,
                                 const uint8_t* inter_sf_d, const void* inter_bf16_d,
                                 const int32_t* expert_counts_d,
                                 const int32_t* expert_offsets_d, const int32_t* perm_src_d,
                                 const float* topk_w_d, float* y_d, int32_t T, void* ws_d,
                                 size_t ws_bytes, moe_stream_t stream)
{
    const NvtxRange nvtx_range("moe_grouped_gemm_down");
    if (!h || !t_ok(h, T) || !expert_counts_d || !expert_offsets_d || !perm_src_d ||
        !topk_w_d || !y_d)
        return MOE_ERR_INVALID;
    const bool a16 = h->cfg.act_mode == MOE_W4A16;
    if (a16 ? !inter_bf16_d : (!inter_codes_d || !inter_sf_d)) return MOE_ERR_INVALID;
    if (T == 0) return MOE_OK;  // nothing to do: no workspace needed
    const moe_status st = check_ws(h, T, ws_d, ws_bytes);
    if (st != MOE_OK) return st;
    const Plan p = plan(h->cfg, T);
    return launch_gemm(h, p, false, kEpiDown, inter_codes_d, inter_sf_d, nullptr, inter_bf16_d,
                       expert_counts_d, expert_offsets_d, y_d, nullptr, nullptr, nullptr,
                       perm_src_d, topk_w_d, ws_d, false, reinterpret_cast<cudaStream_t>(stream));
}

moe_status moe_combine(moe_handle h, const float* y_d, const int32_t* inv_d,
                       const int32_t* expert_offsets_d, int32_t T, void* out_bf16_d,
                       moe_stream_t stream)
{
    const NvtxRange nvtx_range("moe_combine");
    if (!h || !t_ok(h, T) || !y_d || !inv_d || !expert_offsets_d || !out_bf16_d)
        return MOE_ERR_INVALID;
    if (T == 0) return MOE_OK;
    return launch_combine(h, y_d, inv_d, expert_offsets_d, T, out_bf16_d, false,
                          reinterpret_cast<cudaStream_t>(stream));
}

moe_status moe_forward(moe_handle h, const void* x_bf16_d, const float* logits_in_d,
                       const float* logit_bias_d, int32_t T, void* out_bf16_d, void* ws_d,
                       size_t ws_bytes, moe_stream_t stream)
{
    const NvtxRange nvtx_range("moe_forward");
    if (!h || !t_ok(h, T) || !x_bf16_d || !out_bf16_d) return MOE_ERR_INVALID;
    if (reinterpret_cast<uintptr_t>(x_bf16_d) & 15) return MOE_ERR_INVALID;
    if (T == 0) return MOE_OK;  // nothing to do: no workspace needed
    const moe_status st = check_ws(h, T, ws_d, ws_bytes);
    if (st != MOE_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const Plan p = plan(h->cfg, T);
    void* ws = ws_d;
    int32_t* ids = at<int32_t>(ws, p.ids);
    float* w = at<float>(ws, p.w);
    int32_t* counts = at<int32_t>(ws, p.counts);
    int32_t* offsets = at<int32_t>(ws, p.offsets);
    int32_t* perm_src = at<int32_t>(ws, p.perm_src);
    int32_t* inv = at<int32_t>(ws, p.inv);
    float* gs_a = at<float>(ws, p.gs_a);
    uint8_t* a_codes = at<uint8_t>(ws, p.a_codes);
    uint8_t* a_sf = at<uint8_t>(ws, p.a_sf);
    void* a_bf16 = at<void>(ws, p.a_bf16);
    uint8_t* i_codes = at<uint8_t>(ws, p.i_codes);
    uint8_t* i_sf = at<uint8_t>(ws, p.i_sf);
    void* i_bf16 = at<void>(ws, p.i_bf16);
    float* y = at<float>(ws, p.y);
    // one chain of kernels with programmatic dependent launch; the first kernel clears the
    // status word and the two amax accumulators of this forward
    uint32_t* status = at<uint32_t>(ws, p.status);
    uint32_t* amax = at<uint32_t>(ws, p.amax);
    const bool need_amax = h->cfg.act_mode != MOE_W4A4_STATIC;
    bool amax_done = false;
    // W4A16 batches of a few tokens: gate_up and down in one GEMV launch that takes the
    // activation rows from x itself (no gather); the routing kernel zeroes its counters
    const int fused_slots = fused_gemv_slots(h, p);
    moe_status r = launch_route(h, x_bf16_d, logits_in_d, logit_bias_d, T, ids, w, nullptr,
                                at<float>(ws, p.logits), status, status, amax, true, s,
                                need_amax ? amax : nullptr, &amax_done,
                                fused_slots ? at<int32_t>(ws, p.gv_sync) : nullptr,
                                fused_slots ? p.gv_list_cap : 0);
    if (r == MOE_OK)
        r = launch_permute(h, p, ids, T, counts, offsets, perm_src, inv, ws, true, s, false);
    if (fused_slots) {
        if (r == MOE_OK && !amax_done) r = launch_amax(h, x_bf16_d, T, amax, true, s);
        if (r == MOE_OK)
            r = launch_gemv_fused(h, p, x_bf16_d, ws, fused_slots, p.nblk == 1 && amax_done,
                                  true, s);
        if (r == MOE_OK) r = launch_combine(h, y, inv, offsets, T, out_bf16_d, true, s, status);
        return r;
    }
    if (r == MOE_OK)
        r = launch_gather(h, p, x_bf16_d, T, inv, offsets, a_codes, a_sf, a_bf16, gs_a, ws, true,
                          true, s, amax_done);
    if (r == MOE_OK)
        r = launch_gateup_fused(h, p, a_codes, a_sf, gs_a, a_bf16, counts, offsets, i_codes,
                                i_sf, i_bf16, ws, true, s);
    // W4A4: y as fp16 rows times a per-expert power of two (half the bytes of the y round
    // trip); W4A16 (its bf16 intermediate has no a-priori bound) keeps fp32 y
    const bool y16 = h->cfg.act_mode != MOE_W4A16;
    if (r == MOE_OK)
        r = launch_gemm(h, p, false, y16 ? kEpiDownF16 : kEpiDown, i_codes, i_sf, nullptr,
                        i_bf16, counts, offsets, y, nullptr, nullptr, nullptr, perm_src, w, ws,
                        true, s);
    if (r == MOE_OK)
        r = launch_combine(h, y, inv, offsets, T, out_bf16_d, true, s, status,
                           y16 ? at<float>(ws, p.y_scale) : nullptr);
    return r;
}

size_t moe_workspace_size_host(const moe_config* cfg, int32_t T)
{
    const size_t base = moe_workspace_size(cfg, T);
    if (!base) return 0;
    return base + 2 * align256((size_t)T * cfg->hidden * 2);
}

moe_status moe_forward_host(moe_handle h, const void* x_bf16_h, const float* logits_in_d,
                            const float* logit_bias_d, int32_t T, void* out_bf16_h, void* ws_d,
                            size_t ws_bytes, moe_stream_t stream)
{
    const NvtxRange nvtx_range("moe_forward_host");
    if (!h || !t_ok(h, T) || !x_bf16_h || !out_bf16_h) return MOE_ERR_INVALID;
    if (T == 0) return MOE_OK;  // nothing to do: no workspace needed
    const size_t base = plan(h->cfg, T).total;
    const size_t xb = (size_t)T * h->cfg.hidden * 2;
    moe_status st = check_ws(h, T, ws_d, ws_bytes);
    if (st != MOE_OK) return st;
    if (ws_bytes < base + 2 * align256(xb)) return MOE_ERR_WORKSPACE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint8_t* xd = static_cast<uint8_t*>(ws_d) + base;
    uint8_t* od = xd + align256(xb);
    if (cudaMemcpyAsync(xd, x_bf16_h, xb, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    st = moe_forward(h, xd, logits_in_d, logit_bias_d, T, od, ws_d, base, stream);
    if (st != MOE_OK) return st;
    return cudaMemcpyAsync(out_bf16_h, od, xb, cudaMemcpyDeviceToHost, s) == cudaSuccess
               ? MOE_OK
               : MOE_ERR_CUDA;
}

moe_status moe_forward_buffers(moe_handle h, void* ws_d, int32_t T, int32_t** topk_ids,
                               float** topk_w, int32_t** expert_counts,
                               int32_t** expert_offsets, int32_t** perm_src, int32_t** inv,
                               float** gs_a, uint8_t** a_codes, uint8_t** a_sf,
                               void** a_bf16, uint8_t** inter_codes, uint8_t** inter_sf,
                               void** inter_bf16, float** y, float** inter_gs,
                               float** y_scale)
{
    if (!h || !ws_d || !t_ok(h, T)) return MOE_ERR_INVALID;
    const Plan p = plan(h->cfg, T);
    if (topk_ids) *topk_ids = at<int32_t>(ws_d, p.ids);
    if (topk_w) *topk_w = at<float>(ws_d, p.w);
    if (expert_counts) *expert_counts = at<int32_t>(ws_d, p.counts);
    if (expert_offsets) *expert_offsets = at<int32_t>(ws_d, p.offsets);
    if (perm_src) *perm_src = at<int32_t>(ws_d, p.perm_src);
    if (inv) *inv = at<int32_t>(ws_d, p.inv);
    if (gs_a) *gs_a = at<float>(ws_d, p.gs_a);
    if (a_codes) *a_codes = at<uint8_t>(ws_d, p.a_codes);
    if (a_sf) *a_sf = at<uint8_t>(ws_d, p.a_sf);
    if (a_bf16) *a_bf16 = at<void>(ws_d, p.a_bf16);
    if (inter_codes) *inter_codes = at<uint8_t>(ws_d, p.i_codes);
    if (inter_bf16) *inter_bf16 = at<void>(ws_d, p.i_bf16);
    if (inter_sf) *inter_sf = at<uint8_t>(ws_d, p.i_sf);
    if (y) *y = at<float>(ws_d, p.y);
    if (inter_gs) *inter_gs = at<float>(ws_d, p.gs_i);
    if (y_scale) *y_scale = at<float>(ws_d, p.y_scale);
    return MOE_OK;
}

moe_status moe_route_topk_noalloc(moe_handle h, const void* x_bf16_d,
                                  const float* logits_in_d, const float* logit_bias_d,
                                  int32_t T, int32_t* topk_ids_d, float* topk_w_d,
                                  float* logits_out_d, moe_stream_t stream)
{
    const NvtxRange nvtx_range("moe_route_topk_noalloc");
    if (!h || !t_ok(h, T) || !topk_ids_d || !topk_w_d) return MOE_ERR_INVALID;
    if (!logits_in_d && !x_bf16_d) return MOE_ERR_INVALID;
    if (T == 0) return MOE_OK;
    const moe_config& c = h->cfg;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const float* src = logits_in_d;
    uint32_t* status = nullptr;
    int nsplit = 1;
    if (!logits_in_d) {
        if (reinterpret_cast<uintptr_t>(x_bf16_d) & 15) return MOE_ERR_INVALID;
        const size_t plane = (size_t)T * c.num_experts;          // floats per partial plane
        if (plane > kRoutePlaneFloats) return MOE_ERR_WORKSPACE;  // T * E beyond the scratch
        int dev = -1;
        if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
        if (dev != h->device) return MOE_ERR_INVALID;
        float* scratch = nullptr;
        const moe_status st = route_scratch_address(&scratch);
        if (st != MOE_OK) return st;
        status = reinterpret_cast<uint32_t*>(scratch + kRoutePlaneFloats);
        nsplit = router_splits(T, c.num_experts, c.hidden, h->num_sms);
        while (nsplit > 1 && plane * nsplit > kRoutePlaneFloats) nsplit /= 2;
        CUtensorMap tmX;
        if (!make_tmap(&tmX, x_bf16_d, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, c.hidden, T,
                       (uint64_t)c.hidden * 2, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B))
            return MOE_ERR_CUDA;
        if (cudaMemsetAsync(status, 0, 4, s) != cudaSuccess) return MOE_ERR_CUDA;
        const int bn = router_bn(T, c.num_experts);
        dim3 grid(ceil_div(T, 128), ceil_div(c.num_experts, bn), nsplit);
        const moe_status r = launch(router_gemm_kernel, grid, dim3(192), kRouterSmem, s, false,
                                    tmX, bn == 160 ? h->tm_router160 : h->tm_router, (int)T,
                                    c.num_experts, c.hidden, c.hidden / nsplit, bn, scratch,
                                    status, (uint32_t*)nullptr, (uint32_t*)nullptr);
        if (r != MOE_OK) return r;
        src = scratch;
    }
    moe_status r = launch(topk_kernel_for(c.num_experts),
                          dim3(ceil_div(T, topk_tokens_per_block(nsplit))), dim3(kTopkThreads),
                          topk_smem(nsplit, c.num_experts), s, false, src, nsplit, logit_bias_d,
                          (int)T, c.num_experts, c.top_k, topk_ids_d, topk_w_d, logits_out_d,
                          (uint32_t*)nullptr, (uint32_t*)nullptr, (const uint16_t*)nullptr, 0,
                          (uint32_t*)nullptr, (int32_t*)nullptr, 0);
    if (r == MOE_OK && status) {
        const int n = T * c.top_k;
        r = launch(route_invalidate_kernel, dim3(std::min(grid_for(n, 256), 4 * h->num_sms)),
                   dim3(256), 0, s, false, (const uint32_t*)status, n, topk_ids_d, topk_w_d);
    }
    return r;
}

namespace moe {
namespace {

// One thread waits, with the pipelines' own bounded wait, on a phase of an mbarrier that
// nothing arrives on; when the limit runs out it sets MOE_DEV_WAIT_TIMEOUT, as a pipeline
// role would, and returns.
__global__ void bounded_wait_probe_kernel(uint32_t* status, uint64_t limit_ns)
{
    __shared__ uint64_t bar;
    __shared__ int zero;
    if (threadIdx.x != 0) return;
    mbar_init(&bar, 1);
    zero = 0;
    fence_barrier_init();
    if (!mbar_wait(&bar, 0, &zero, limit_ns)) set_status(status, MOE_DEV_WAIT_TIMEOUT);
}

}  // namespace
}  // namespace moe

moe_status moe_selftest_bounded_wait(uint32_t* status_d, uint64_t limit_ns, moe_stream_t stream)
{
    const NvtxRange nvtx_range("moe_selftest_bounded_wait");
    if (!status_d || limit_ns == 0 || limit_ns > moe::kWaitLimitNs) return MOE_ERR_INVALID;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint32_t bits = 0;
    if (cudaMemsetAsync(status_d, 0, 4, s) != cudaSuccess) return MOE_ERR_CUDA;
    moe::bounded_wait_probe_kernel<<<1, 32, 0, s>>>(status_d, limit_ns);
    if (cudaGetLastError() != cudaSuccess ||
        cudaMemcpyAsync(&bits, status_d, 4, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return MOE_ERR_CUDA;
    return (bits & MOE_DEV_WAIT_TIMEOUT) ? MOE_ERR_TIMEOUT : MOE_OK;
}

moe_status moe_get_status(moe_handle h, void* ws_d, moe_stream_t stream, uint32_t* bits)
{
    const NvtxRange nvtx_range("moe_get_status");
    if (!h || !ws_d) return MOE_ERR_INVALID;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint32_t v = 0;
    // the status word is the first entry of every workspace plan
    if (cudaMemcpyAsync(&v, ws_d, 4, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess || cudaMemsetAsync(ws_d, 0, 4, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (bits) *bits = v;
    if (v & MOE_DEV_WAIT_TIMEOUT) return MOE_ERR_TIMEOUT;
    return v ? MOE_ERR_DEVICE_STATUS : MOE_OK;
}

}  // extern "C"
