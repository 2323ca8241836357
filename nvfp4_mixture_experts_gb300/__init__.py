"""Python binding of libnvfp4moe.so, the NVFP4 fused mixture-of-experts layer forward.

Argument marshalling only: every function forwards to the C entry point of the same name
(declared in include/nvfp4moe.h).  Tensors are torch tensors on the GPU (torch provides
device memory and streams); every step of the computation runs in the library's CUDA
kernels.  Importing raises if the compiled library is missing -- there is no fallback.
"""
import ctypes as C
import os

from . import build as _build

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = _build.LIB

MOE_OK, MOE_ERR_INVALID, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA, MOE_ERR_WORKSPACE, \
    MOE_ERR_TIMEOUT, MOE_ERR_DEVICE_STATUS = range(7)
MOE_W4A4_DYNAMIC, MOE_W4A4_STATIC, MOE_W4A16 = 0, 1, 2
MOE_GS_ENCODE, MOE_GS_DEQUANT = 0, 1
MOE_TILING_AUTO, MOE_TILING_ROWS, MOE_TILING_TOKENS, MOE_TILING_PAIRS, MOE_TILING_WIDE = \
    0, 1, 2, 3, 4
MOE_DEV_BAD_EXPERT_ID, MOE_DEV_WAIT_TIMEOUT, MOE_DEV_ROWS_OVERFLOW = 1, 2, 4
MOE_DEV_BAD_INDEX = 8


class moe_config(C.Structure):
    _fields_ = [("hidden", C.c_int32), ("inter", C.c_int32), ("num_experts", C.c_int32),
                ("top_k", C.c_int32), ("num_local_experts", C.c_int32),
                ("local_expert_offset", C.c_int32), ("has_shared", C.c_int32),
                ("shared_inter", C.c_int32), ("add_shared", C.c_int32),
                ("act_mode", C.c_int32), ("act_global_scale", C.c_float),
                ("inter_global_scale", C.c_float), ("max_tokens", C.c_int32),
                ("gemm_tiling", C.c_int32)]


class moe_weights(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in (
        "router_w_d", "w13_d", "w13_sf_d", "w13_gs_d", "w2_d", "w2_sf_d", "w2_gs_d",
        "sh13_d", "sh13_sf_d", "sh13_gs_d", "sh2_d", "sh2_sf_d", "sh2_gs_d")]


_V = C.c_void_p
_I = C.c_int32
_SZ = C.c_size_t

# name -> (restype, argtypes); the list mirrors include/nvfp4moe.h
SIGNATURES = {
    "moe_create": (C.c_int, [C.POINTER(moe_config), C.POINTER(moe_weights), _V, C.POINTER(_V)]),
    "moe_destroy": (None, [_V]),
    "moe_workspace_size": (_SZ, [C.POINTER(moe_config), _I]),
    "moe_rows_capacity": (_I, [C.POINTER(moe_config), _I]),
    "moe_route_topk": (C.c_int, [_V, _V, _V, _V, _I, _V, _V, _V, _V, _SZ, _V]),
    "moe_route_topk_noalloc": (C.c_int, [_V, _V, _V, _V, _I, _V, _V, _V, _V]),
    "moe_permute": (C.c_int, [_V, _V, _I, _V, _V, _V, _V, _V, _SZ, _V]),
    "moe_quant_nvfp4": (C.c_int, [_V, _I, _I, _V, _V, _V, _V, _I, _V, _SZ, _V]),
    "moe_gather_activations": (C.c_int, [_V, _V, _I, _V, _V, _V, _V, _V, _V, _V, _SZ, _V]),
    "moe_grouped_gemm_gateup": (C.c_int, [_V, _V, _V, _V, _V, _V, _V, _I, _V, _V, _V, _V, _I,
                                          _V, _SZ, _V]),
    "moe_swiglu_requant": (C.c_int, [_V, _I, _I, C.c_float, _V, _V, _I, _V]),
    "moe_prepare_weights": (C.c_int, [_V, _V, _V, _I, _I, _I, _I, C.c_float, _I, _I, _I, _V,
                                      _V, _V, _V]),
    "moe_grouped_gemm_down": (C.c_int, [_V, _V, _V, _V, _V, _V, _V, _V, _V, _I, _V, _SZ, _V]),
    "moe_combine": (C.c_int, [_V, _V, _V, _V, _I, _V, _V]),
    "moe_forward": (C.c_int, [_V, _V, _V, _V, _I, _V, _V, _SZ, _V]),
    "moe_forward_host": (C.c_int, [_V, _V, _V, _V, _I, _V, _V, _SZ, _V]),
    "moe_workspace_size_host": (_SZ, [C.POINTER(moe_config), _I]),
    "moe_forward_buffers": (C.c_int, [_V, _V, _I] + [C.POINTER(_V)] * 16),
    "moe_get_status": (C.c_int, [_V, _V, _V, C.POINTER(C.c_uint32)]),
    "moe_status_string": (C.c_char_p, [C.c_int]),
    "moe_selftest_bounded_wait": (C.c_int, [_V, C.c_uint64, _V]),
}

_lib = None
_lib_debug = None


def _open(p):
    if not os.path.exists(p):
        raise OSError("%s not built: run __graft_entry__.build()" % p)
    lib = C.CDLL(p)
    for name, (res, args) in SIGNATURES.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib


def load(path=None):
    """Loads the compiled library (raises OSError if it is not there)."""
    global _lib
    if _lib is None:
        _lib = _open(path or LIB_PATH)
    return _lib


def load_debug():
    """The MOE_DEBUG flavour of the library (same entry points; every index read from a
    buffer is bounds-checked on the device and a bad one flags MOE_DEV_BAD_INDEX).  Handles
    of one flavour are used with that flavour's calls only."""
    global _lib_debug
    if _lib_debug is None:
        _lib_debug = _open(_build.LIB_DEBUG)
    return _lib_debug


class MoEError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        msg = load().moe_status_string(status).decode()
        super().__init__("%s: %s (%d)" % (where, msg, status))


def _check(status, where):
    if status != MOE_OK:
        raise MoEError(status, where)


def _p(t):
    """Device pointer of a torch tensor (or None)."""
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    return C.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


# ---------------------------------------------------------------- C entry points

def moe_create(cfg, weights, stream=None):
    h = C.c_void_p()
    _check(load().moe_create(C.byref(cfg), C.byref(weights), _stream(stream), C.byref(h)),
           "moe_create")
    return h


def moe_destroy(h):
    load().moe_destroy(h)


def moe_workspace_size(cfg, T):
    return load().moe_workspace_size(C.byref(cfg), T)


def moe_rows_capacity(cfg, T):
    return load().moe_rows_capacity(C.byref(cfg), T)


def moe_route_topk(h, x, logits_in, logit_bias, T, topk_ids, topk_w, logits_out, ws,
                   stream=None):
    _check(load().moe_route_topk(h, _p(x), _p(logits_in), _p(logit_bias), T, _p(topk_ids),
                                 _p(topk_w), _p(logits_out), _p(ws),
                                 0 if ws is None else ws.numel() * ws.element_size(),
                                 _stream(stream)), "moe_route_topk")


def moe_route_topk_noalloc(h, x, logits_in, logit_bias, T, topk_ids, topk_w, logits_out,
                           stream=None):
    """moe_route_topk without a workspace: the scratch is a static device array of the
    library (see include/nvfp4moe.h for its size limit and sharing rules)."""
    _check(load().moe_route_topk_noalloc(h, _p(x), _p(logits_in), _p(logit_bias), T,
                                         _p(topk_ids), _p(topk_w), _p(logits_out),
                                         _stream(stream)), "moe_route_topk_noalloc")


def moe_permute(h, topk_ids, T, counts, offsets, perm_src, inv, ws, stream=None):
    _check(load().moe_permute(h, _p(topk_ids), T, _p(counts), _p(offsets), _p(perm_src),
                              _p(inv), _p(ws), ws.numel() * ws.element_size(),
                              _stream(stream)), "moe_permute")


def moe_quant_nvfp4(x, rows, cols, gs_in, gs_out, codes, sf, sf_layout, ws, stream=None):
    _check(load().moe_quant_nvfp4(_p(x), rows, cols, _p(gs_in), _p(gs_out), _p(codes), _p(sf),
                                  sf_layout, _p(ws),
                                  0 if ws is None else ws.numel() * ws.element_size(),
                                  _stream(stream)), "moe_quant_nvfp4")


def moe_gather_activations(h, x, T, inv, offsets, a_codes, a_sf, a_bf16, gs_out, ws,
                           stream=None):
    _check(load().moe_gather_activations(h, _p(x), T, _p(inv), _p(offsets), _p(a_codes),
                                         _p(a_sf), _p(a_bf16), _p(gs_out), _p(ws),
                                         ws.numel() * ws.element_size(), _stream(stream)),
           "moe_gather_activations")


def moe_grouped_gemm_gateup(h, a_codes, a_sf, gs_a, a_bf16, counts, offsets, fuse_epilogue,
                            gateup_f32, inter_codes, inter_sf, inter_bf16, T, ws, stream=None):
    _check(load().moe_grouped_gemm_gateup(h, _p(a_codes), _p(a_sf), _p(gs_a), _p(a_bf16),
                                          _p(counts), _p(offsets), int(fuse_epilogue),
                                          _p(gateup_f32), _p(inter_codes), _p(inter_sf),
                                          _p(inter_bf16), T, _p(ws),
                                          ws.numel() * ws.element_size(), _stream(stream)),
           "moe_grouped_gemm_gateup")


def moe_swiglu_requant(gateup_f32, rows, inter, gs_i, codes, sf, sf_layout, stream=None):
    _check(load().moe_swiglu_requant(_p(gateup_f32), rows, inter, float(gs_i), _p(codes),
                                     _p(sf), sf_layout, _stream(stream)), "moe_swiglu_requant")


def moe_prepare_weights(codes, sf, glob, N, K, convention, fold_target, swap_halves, off, count,
                        codes_out, sf_out, gs_out, stream=None):
    _check(load().moe_prepare_weights(_p(codes), _p(sf), _p(glob), int(glob.numel()), N, K,
                                      convention, float(fold_target), int(bool(swap_halves)),
                                      off, count, _p(codes_out), _p(sf_out), _p(gs_out),
                                      _stream(stream)), "moe_prepare_weights")


def moe_grouped_gemm_down(h, inter_codes, inter_sf, inter_bf16, counts, offsets, perm_src,
                          topk_w, y, T, ws, stream=None):
    _check(load().moe_grouped_gemm_down(h, _p(inter_codes), _p(inter_sf), _p(inter_bf16),
                                        _p(counts), _p(offsets), _p(perm_src), _p(topk_w),
                                        _p(y), T, _p(ws), ws.numel() * ws.element_size(),
                                        _stream(stream)), "moe_grouped_gemm_down")


def moe_combine(h, y, inv, offsets, T, out, stream=None):
    _check(load().moe_combine(h, _p(y), _p(inv), _p(offsets), T, _p(out), _stream(stream)),
           "moe_combine")


def moe_forward(h, x, logits_in, logit_bias, T, out, ws, stream=None):
    _check(load().moe_forward(h, _p(x), _p(logits_in), _p(logit_bias), T, _p(out), _p(ws),
                              ws.numel() * ws.element_size(), _stream(stream)), "moe_forward")


def moe_forward_host(h, x_host, logits_in, logit_bias, T, out_host, ws, stream=None):
    """x_host / out_host: CPU tensors (pinned for asynchronous copies); ws: a device workspace
    of moe_workspace_size_host bytes."""
    _check(load().moe_forward_host(h, _p(x_host), _p(logits_in), _p(logit_bias), T,
                                   _p(out_host), _p(ws), ws.numel() * ws.element_size(),
                                   _stream(stream)), "moe_forward_host")


def moe_workspace_size_host(cfg, T):
    return load().moe_workspace_size_host(C.byref(cfg), T)


FORWARD_BUFFERS = ("topk_ids", "topk_w", "expert_counts", "expert_offsets", "perm_src", "inv",
                   "gs_a", "a_codes", "a_sf", "a_bf16", "inter_codes", "inter_sf", "inter_bf16",
                   "y", "inter_gs", "y_scale")


def moe_forward_buffers(h, ws, T):
    """Device addresses (ints) of moe_forward's intermediates inside ws."""
    ptrs = [C.c_void_p() for _ in FORWARD_BUFFERS]
    _check(load().moe_forward_buffers(h, _p(ws), T, *[C.byref(p) for p in ptrs]),
           "moe_forward_buffers")
    return {n: p.value for n, p in zip(FORWARD_BUFFERS, ptrs)}


def moe_selftest_bounded_wait(status_word, limit_ns, stream=None):
    """Runs the bounded-wait failure self-test (status_word: a device tensor of >= 4 bytes);
    returns the status code (MOE_ERR_TIMEOUT expected)."""
    return load().moe_selftest_bounded_wait(_p(status_word), int(limit_ns), _stream(stream))


def moe_get_status(h, ws, stream=None):
    bits = C.c_uint32(0)
    st = load().moe_get_status(h, _p(ws), _stream(stream), C.byref(bits))
    return st, bits.value


from .layer import MoELayer, make_config  # noqa: E402,F401
