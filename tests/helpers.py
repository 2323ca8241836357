"""Test helpers: build oracle-quantised layers from the seeded synthetic masters."""
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

import oracle
import synth


def e2m1_table():
    vals = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    return np.array(vals + [-v for v in vals])


def dequant_independent(codes, sf, gs):
    """NVFP4 -> fp64 with a table lookup and torch's E4M3 decode (no oracle code)."""
    R, Kh = codes.shape
    K = 2 * Kh
    c = np.empty((R, K), np.int64)
    c[:, 0::2] = codes & 15
    c[:, 1::2] = codes >> 4
    s = torch.from_numpy(np.ascontiguousarray(sf)).view(torch.float8_e4m3fn).double().numpy()
    return e2m1_table()[c] * np.repeat(s, 16, axis=1) / np.float64(gs)


def quantize_expert(w13, w2):
    c13, s13, g13 = oracle.quant_nvfp4(w13)
    c2, s2, g2 = oracle.quant_nvfp4(w2)
    return c13, s13, g13, c2, s2, g2


def build_layer(seed, H, I, E, experts=None, shared=True):
    """Quantise (with the oracle) the masters of the listed global experts (default all)
    and of the shared expert.  Returns an oracle.Layer whose local expert i is
    experts[i]."""
    experts = list(range(E)) if experts is None else list(experts)
    El = len(experts)
    w13 = np.empty((El, 2 * I, H // 2), np.uint8)
    w13_sf = np.empty((El, 2 * I, H // 16), np.uint8)
    w13_gs = np.empty(El, np.float32)
    w2 = np.empty((El, H, I // 2), np.uint8)
    w2_sf = np.empty((El, H, I // 16), np.uint8)
    w2_gs = np.empty(El, np.float32)
    with ThreadPoolExecutor(4) as pool:
        masters = pool.map(lambda e: synth.expert_master(seed, e, H, I), experts)
        for i, (m13, m2) in enumerate(masters):
            w13[i], w13_sf[i], w13_gs[i], w2[i], w2_sf[i], w2_gs[i] = quantize_expert(m13, m2)
    kw = {}
    if shared:
        m13, m2 = synth.shared_master(seed, H, I)
        c13, s13, g13, c2, s2, g2 = quantize_expert(m13, m2)
        kw = dict(sh13=c13, sh13_sf=s13, sh13_gs=g13, sh2=c2, sh2_sf=s2, sh2_gs=g2)
    return oracle.Layer(w13, w13_sf, w13_gs, w2, w2_sf, w2_gs, **kw)


def slice_layer(layer, lo, hi):
    """Local experts lo..hi-1 of a full layer (shared expert kept)."""
    return oracle.Layer(layer.w13[lo:hi], layer.w13_sf[lo:hi], layer.w13_gs[lo:hi],
                        layer.w2[lo:hi], layer.w2_sf[lo:hi], layer.w2_gs[lo:hi],
                        layer.sh13, layer.sh13_sf, layer.sh13_gs,
                        layer.sh2, layer.sh2_sf, layer.sh2_gs)


def rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def within_layer_tolerance(got, ref):
    """Whole-layer bar: relative L2 <= 1e-2 and max |err| <= 5e-2 * rms(ref)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    rms = float(np.sqrt(np.mean(ref ** 2)))
    return rel_l2(got, ref), float(np.max(np.abs(got - ref))) / max(rms, 1e-300)
