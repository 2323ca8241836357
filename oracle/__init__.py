"""Python shim over the oracle (plain C, fp64 accumulation) -- TEST INFRASTRUCTURE ONLY.

Only the tests, the smoke check and the CPU-baseline leg of the benchmark import this
package.  It shares no code with the CUDA library or its binding; the two meet only in
the seeded input generators of the separate ``synth`` package.

Every function here marshals numpy arrays into the C oracle (``moe_oracle.c``), whose
header comment states what is computed and which passage of the pages each step follows.
"""
import ctypes as C
import os

import numpy as np

from . import build as _build

_lib = None


def load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = C.CDLL(path)
        lib.orc_e2m1_value.restype = C.c_double
        lib.orc_e2m1_value.argtypes = [C.c_int]
        lib.orc_e4m3_value.restype = C.c_double
        lib.orc_e4m3_value.argtypes = [C.c_int]
        lib.orc_e2m1_encode.restype = C.c_int
        lib.orc_e2m1_encode.argtypes = [C.c_float]
        lib.orc_e4m3_encode.restype = C.c_int
        lib.orc_e4m3_encode.argtypes = [C.c_float]
        lib.orc_bf16_round.restype = C.c_uint16
        lib.orc_bf16_round.argtypes = [C.c_double]
        lib.orc_bf16_value.restype = C.c_double
        lib.orc_bf16_value.argtypes = [C.c_uint16]
        lib.orc_dynamic_global_scale.restype = C.c_float
        lib.orc_dynamic_global_scale.argtypes = [C.c_void_p, C.c_long]
        lib.orc_quant_nvfp4.restype = None
        lib.orc_quant_nvfp4.argtypes = [C.c_void_p, C.c_long, C.c_int, C.c_int,
                                        C.POINTER(C.c_float), C.c_void_p, C.c_void_p]
        lib.orc_dequant_nvfp4.restype = None
        lib.orc_dequant_nvfp4.argtypes = [C.c_void_p, C.c_void_p, C.c_float, C.c_long,
                                          C.c_int, C.c_void_p]
        lib.orc_router_logits.restype = None
        lib.orc_router_logits.argtypes = [C.c_void_p, C.c_void_p, C.c_void_p, C.c_long,
                                          C.c_int, C.c_int, C.c_void_p]
        lib.orc_topk.restype = None
        lib.orc_topk.argtypes = [C.c_void_p, C.c_long, C.c_int, C.c_int, C.c_void_p,
                                 C.c_void_p]
        lib.orc_permute.restype = C.c_long
        lib.orc_permute.argtypes = [C.c_void_p, C.c_long, C.c_int, C.c_int, C.c_int,
                                    C.c_void_p, C.c_void_p]
        lib.orc_expert_rows.restype = None
        lib.orc_expert_rows.argtypes = [C.POINTER(Cfg), C.POINTER(Expert), C.c_void_p,
                                        C.c_void_p, C.c_void_p, C.c_float, C.c_void_p,
                                        C.c_long, C.c_void_p, C.c_void_p, C.c_void_p,
                                        C.c_void_p]
        lib.orc_swiglu_requant.restype = None
        lib.orc_swiglu_requant.argtypes = [C.c_void_p, C.c_long, C.c_int, C.c_float,
                                           C.c_void_p, C.c_void_p, C.c_void_p]
        lib.orc_moe_forward.restype = C.c_int
        lib.orc_moe_forward.argtypes = [C.POINTER(Cfg), C.c_void_p, C.c_void_p, C.c_void_p,
                                        C.c_void_p, C.POINTER(Expert), C.c_void_p, C.c_long,
                                        C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                        C.c_void_p, C.POINTER(C.c_long), C.c_void_p,
                                        C.c_void_p, C.POINTER(C.c_float),
                                        C.POINTER(C.c_float), C.c_void_p, C.c_void_p]
        lib.orc_prepare_weights.restype = None
        lib.orc_prepare_weights.argtypes = [C.c_void_p, C.c_void_p, C.c_void_p, C.c_int,
                                            C.c_int, C.c_int, C.c_float, C.c_int, C.c_int,
                                            C.c_int, C.c_void_p, C.c_void_p, C.c_void_p]
        lib.orc_num_threads.restype = C.c_int
        lib.orc_set_num_threads.argtypes = [C.c_int]
        _lib = lib
    return _lib


class Cfg(C.Structure):
    _fields_ = [("T", C.c_int), ("H", C.c_int), ("I", C.c_int), ("E", C.c_int),
                ("k", C.c_int), ("E_loc", C.c_int), ("off", C.c_int),
                ("has_shared", C.c_int), ("add_shared", C.c_int), ("act_mode", C.c_int),
                ("act_gs", C.c_float), ("inter_gs", C.c_float)]


class Expert(C.Structure):
    _fields_ = [("w13", C.c_void_p), ("w13_sf", C.c_void_p), ("w2", C.c_void_p),
                ("w2_sf", C.c_void_p), ("gs13", C.c_float), ("gs2", C.c_float)]


ACT_W4A4_DYNAMIC, ACT_W4A4_STATIC, ACT_W4A16 = 0, 1, 2


def _p(a):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


# ---------------------------------------------------------------- formats

def e2m1_value(code):
    return load().orc_e2m1_value(int(code))


def e4m3_value(code):
    return load().orc_e4m3_value(int(code))


def e2m1_encode(x):
    return load().orc_e2m1_encode(float(x))


def e4m3_encode(x):
    return load().orc_e4m3_encode(float(x))


def bf16_round(d):
    return load().orc_bf16_round(float(d))


def set_num_threads(n):
    load().orc_set_num_threads(int(n))


def num_threads():
    return load().orc_num_threads()


# ---------------------------------------------------------------- quantiser

def quant_nvfp4(X, gs=None):
    """NVFP4-quantise fp32 X[R, K]; gs=None -> dynamic global scale.
    Returns (codes u8 [R, K/2], sf u8 [R, K/16], gs float)."""
    X = _c(X, np.float32)
    R, K = X.shape
    codes = np.empty((R, K // 2), np.uint8)
    sf = np.empty((R, K // 16), np.uint8)
    g = C.c_float(1.0 if gs is None else gs)
    load().orc_quant_nvfp4(_p(X), R, K, 1 if gs is None else 0, C.byref(g), _p(codes), _p(sf))
    return codes, sf, g.value


def dequant_nvfp4(codes, sf, gs):
    codes = _c(codes, np.uint8)
    sf = _c(sf, np.uint8)
    R = codes.shape[0]
    K = codes.shape[1] * 2
    out = np.empty((R, K), np.float64)
    load().orc_dequant_nvfp4(_p(codes), _p(sf), gs, R, K, _p(out))
    return out


def dynamic_global_scale(X):
    X = _c(X, np.float32)
    return load().orc_dynamic_global_scale(_p(X), X.size)


# ---------------------------------------------------------------- routing

def router_logits(x_bf16, wr_bf16, bias=None):
    x = _c(x_bf16, np.uint16)
    wr = _c(wr_bf16, np.uint16)
    b = _c(bias, np.float32)
    T, H = x.shape
    E = wr.shape[0]
    out = np.empty((T, E), np.float64)
    load().orc_router_logits(_p(x), _p(wr), _p(b), T, H, E, _p(out))
    return out


def topk(logits, k):
    lg = _c(logits, np.float64)
    T, E = lg.shape
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    load().orc_topk(_p(lg), T, E, k, _p(ids), _p(w))
    return ids, w


def permute(ids, E_loc, off):
    ids = _c(ids, np.int32)
    T, k = ids.shape
    counts = np.empty(E_loc, np.int32)
    pairs = np.empty(T * k, np.int32)
    n = load().orc_permute(_p(ids), T, k, E_loc, off, _p(counts), _p(pairs))
    return counts, pairs[:n].copy()


# ---------------------------------------------------------------- layer

class Layer:
    """Quantised weights of a layer (or shard): canonical layouts.

    w13 [El, 2I, H/2] u8, w13_sf [El, 2I, H/16] u8, w13_gs [El] f32
    w2  [El, H, I/2]  u8, w2_sf  [El, H, I/16]  u8, w2_gs  [El] f32
    shared (optional): sh13, sh13_sf, sh13_gs (scalar), sh2, sh2_sf, sh2_gs."""

    def __init__(self, w13, w13_sf, w13_gs, w2, w2_sf, w2_gs,
                 sh13=None, sh13_sf=None, sh13_gs=1.0, sh2=None, sh2_sf=None, sh2_gs=1.0):
        self.w13 = _c(w13, np.uint8)
        self.w13_sf = _c(w13_sf, np.uint8)
        self.w13_gs = _c(w13_gs, np.float32)
        self.w2 = _c(w2, np.uint8)
        self.w2_sf = _c(w2_sf, np.uint8)
        self.w2_gs = _c(w2_gs, np.float32)
        self.sh13 = _c(sh13, np.uint8)
        self.sh13_sf = _c(sh13_sf, np.uint8)
        self.sh13_gs = float(sh13_gs)
        self.sh2 = _c(sh2, np.uint8)
        self.sh2_sf = _c(sh2_sf, np.uint8)
        self.sh2_gs = float(sh2_gs)

    def experts(self):
        El = self.w13.shape[0]
        arr = (Expert * (El + 1))()
        for e in range(El):
            arr[e] = Expert(self.w13[e].ctypes.data, self.w13_sf[e].ctypes.data,
                            self.w2[e].ctypes.data, self.w2_sf[e].ctypes.data,
                            float(self.w13_gs[e]), float(self.w2_gs[e]))
        if self.sh13 is not None:
            arr[El] = Expert(_p(self.sh13), _p(self.sh13_sf), _p(self.sh2), _p(self.sh2_sf),
                             self.sh13_gs, self.sh2_gs)
        return arr

    def expert(self, e):
        """Expert struct for local expert e, or the shared expert for e == 'shared'."""
        if e == "shared":
            return Expert(_p(self.sh13), _p(self.sh13_sf), _p(self.sh2), _p(self.sh2_sf),
                          self.sh13_gs, self.sh2_gs)
        return Expert(self.w13[e].ctypes.data, self.w13_sf[e].ctypes.data,
                      self.w2[e].ctypes.data, self.w2_sf[e].ctypes.data,
                      float(self.w13_gs[e]), float(self.w2_gs[e]))


def make_cfg(T, H, I, E, k, E_loc=None, off=0, has_shared=1, add_shared=1,
             act_mode=ACT_W4A4_DYNAMIC, act_gs=1.0, inter_gs=1.0):
    return Cfg(T, H, I, E, k, E if E_loc is None else E_loc, off, has_shared, add_shared,
               act_mode, act_gs, inter_gs)


def expert_rows(cfg, layer, e, x_bf16, x_codes, x_sf, gs_a, tokens):
    """Expert MLP of expert e ('shared' for the shared expert) on the listed tokens.
    Returns (G [n, 2I] fp64, inter_codes [n, I/2], inter_sf [n, I/16], Y [n, H] fp64)."""
    tok = _c(tokens, np.int32)
    n = tok.shape[0]
    G = np.empty((n, 2 * cfg.I), np.float64)
    ic = np.empty((n, cfg.I // 2), np.uint8)
    isf = np.empty((n, cfg.I // 16), np.uint8)
    Y = np.empty((n, cfg.H), np.float64)
    ex = layer.expert(e)
    load().orc_expert_rows(C.byref(cfg), C.byref(ex), _p(_c(x_bf16, np.uint16)),
                           _p(_c(x_codes, np.uint8)), _p(_c(x_sf, np.uint8)), gs_a,
                           _p(tok), n, _p(G), _p(ic), _p(isf), _p(Y))
    return G, ic, isf, Y


def swiglu_requant(gu, I, gs_i):
    """SwiGLU then NVFP4 with static scale gs_i of fp32 gate/up rows [R, 2I]."""
    gu = _c(gu, np.float32)
    R = gu.shape[0]
    codes = np.empty((R, I // 2), np.uint8)
    sf = np.empty((R, I // 16), np.uint8)
    s = np.empty((R, I), np.float64)
    load().orc_swiglu_requant(_p(gu), R, I, gs_i, _p(codes), _p(sf), _p(s))
    return codes, sf, s


class Forward:
    """Result of ``moe_forward``."""


def moe_forward(cfg, x_bf16, layer, router_w=None, logit_bias=None, logits_in=None,
                tokens=None):
    """Oracle forward of the layer / shard.  ``tokens`` restricts the expert MLPs and the
    output to a subset of tokens (routing and quantisation always cover all tokens)."""
    x = _c(x_bf16, np.uint16)
    T, k, E, El, H = cfg.T, cfg.k, cfg.E, cfg.E_loc, cfg.H
    tok = _c(tokens, np.int32)
    nt = T if tok is None else tok.shape[0]
    r = Forward()
    r.logits = np.empty((T, E), np.float64)
    r.ids = np.empty((T, k), np.int32)
    r.w = np.empty((T, k), np.float64)
    r.counts = np.empty(El, np.int32)
    pairs = np.empty(T * k, np.int32)
    n_local = C.c_long(0)
    if cfg.act_mode != ACT_W4A16:
        r.x_codes = np.empty((T, H // 2), np.uint8)
        r.x_sf = np.empty((T, H // 16), np.uint8)
    else:
        r.x_codes = r.x_sf = None
    gs = C.c_float(0.0)
    gs_i = C.c_float(0.0)
    r.out = np.empty((nt, H), np.float64)
    r.out_bf16 = np.empty((nt, H), np.uint16)
    experts = layer.experts()
    load().orc_moe_forward(C.byref(cfg), _p(x), _p(_c(router_w, np.uint16)),
                           _p(_c(logit_bias, np.float32)), _p(_c(logits_in, np.float32)),
                           experts, _p(tok), nt, _p(r.logits), _p(r.ids), _p(r.w),
                           _p(r.counts), _p(pairs), C.byref(n_local), _p(r.x_codes),
                           _p(r.x_sf), C.byref(gs), C.byref(gs_i), _p(r.out), _p(r.out_bf16))
    r.pairs = pairs[:n_local.value].copy()
    r.gs_a = gs.value
    r.gs_i = gs_i.value
    r.tokens = np.arange(T, dtype=np.int32) if tok is None else tok
    return r


GS_ENCODE, GS_DEQUANT = 0, 1   # global-scale conventions of a checkpoint


def prepare_weights(codes, sf, glob, convention=GS_ENCODE, fold_target=0.0, swap_halves=False,
                    off=0, count=None):
    """Checkpoint-convention weights [E][N][K/2] codes, [E][N][K/16] E4M3 scales, [E]
    globals -> the library's codes / scales / encode scales for experts off..off+count-1
    (see orc_prepare_weights)."""
    codes = _c(codes, np.uint8)
    sf = _c(sf, np.uint8)
    glob = _c(glob, np.float32)
    E, N, K2 = codes.shape
    K = 2 * K2
    count = E - off if count is None else count
    co = np.empty((count, N, K // 2), np.uint8)
    so = np.empty((count, N, K // 16), np.uint8)
    go = np.empty(count, np.float32)
    load().orc_prepare_weights(_p(codes), _p(sf), _p(glob), N, K, convention, fold_target,
                               int(bool(swap_halves)), off, count, _p(co), _p(so), _p(go))
    return co, so, go
