"""GPU-test helpers: upload oracle-quantised layers, convert the tiled layouts back to the
canonical ones for comparison, and compare quantisation decisions near rounding
boundaries."""
import numpy as np
import torch

import nvfp4_mixture_experts_gb300 as moe
import oracle
import synth


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    return t.cpu().numpy()


def bits16(a):
    """numpy uint16 bf16 bits -> torch int16 on the GPU."""
    return dev(np.ascontiguousarray(a).view(np.int16))


def upload_weights(layer, router_w_bits):
    w = dict(router_w=bits16(router_w_bits))
    if layer.w13.shape[0] > 0:
        w.update(w13=dev(layer.w13), w13_sf=dev(layer.w13_sf), w13_gs=dev(layer.w13_gs),
                 w2=dev(layer.w2), w2_sf=dev(layer.w2_sf), w2_gs=dev(layer.w2_gs))
    if layer.sh13 is not None:
        w.update(sh13=dev(layer.sh13), sh13_sf=dev(layer.sh13_sf),
                 sh13_gs=dev(np.array([layer.sh13_gs], np.float32)),
                 sh2=dev(layer.sh2), sh2_sf=dev(layer.sh2_sf),
                 sh2_gs=dev(np.array([layer.sh2_gs], np.float32)))
    return w


def make_layer(layer, router_w_bits, H, I, E, k, E_loc=None, off=0, add_shared=1,
               act_mode=0, inter_gs=1.0, act_gs=0.0, max_tokens=8192, has_shared=1,
               gemm_tiling=0):
    cfg = moe.make_config(H, I, E, k, E_loc=E_loc, off=off, has_shared=has_shared,
                          add_shared=add_shared, act_mode=act_mode, act_gs=act_gs,
                          inter_gs=inter_gs, max_tokens=max_tokens, gemm_tiling=gemm_tiling)
    return moe.MoELayer(cfg, upload_weights(layer, router_w_bits))


def codes_pitch(K):
    return (K // 2 + 127) // 128 * 128


def sf_atom_index(rows, K):
    """Byte index of scale (r, b) in the tiled atom layout, for r < rows, b < K/16."""
    r = np.arange(rows)[:, None]
    b = np.arange(K // 16)[None, :]
    rb, m = r >> 7, r & 127
    s, kk = b >> 2, b & 3
    return (rb * (K // 64) + s) * 512 + (m & 31) * 16 + (m >> 5) * 4 + kk


def tiled_to_canonical(codes_tiled, sf_tiled, rows, K):
    codes = np.asarray(codes_tiled).reshape(-1, codes_pitch(K))[:rows, :K // 2]
    sf = np.asarray(sf_tiled).reshape(-1)[sf_atom_index(rows, K)]
    return codes, sf


def canonical_to_tiled(codes, sf, rows_total, K):
    """Canonical rows -> tiled buffers with rows_total rows (missing rows zero)."""
    R = codes.shape[0]
    ct = np.zeros((rows_total, codes_pitch(K)), np.uint8)
    ct[:R, :K // 2] = codes
    st = np.zeros(((rows_total + 127) // 128) * 128 * (K // 16), np.uint8)
    st[sf_atom_index(R, K)] = sf
    return ct, st


E2M1_MAG = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def e4m3_values(codes):
    return torch.from_numpy(np.ascontiguousarray(codes, np.uint8)).view(
        torch.float8_e4m3fn).double().numpy()


def quant_decisions_near_boundary(s, gs, sf_a, sf_b, codes_a, codes_b, rel=2e-6):
    """For NVFP4 rows quantised from (almost) the same values s [R, K] (fp64) with scale gs,
    returns a boolean [R, K/16] mask of blocks whose differing decisions are explained by s
    lying within `rel` of a rounding boundary (block scale or element code)."""
    R, K = s.shape
    nb = K // 16
    blk = s.reshape(R, nb, 16)
    m = np.abs(blk).max(-1)
    q = m * gs / 6.0
    pts = np.array([oracle.e4m3_value(c) for c in range(127)])
    mids = (pts[1:] + pts[:-1]) / 2
    near_sf = np.min(np.abs(q[..., None] - mids[None, None, :]) /
                     np.maximum(q[..., None], 1e-30), -1) < rel
    ok = np.ones((R, nb), bool)
    diff_sf = sf_a != sf_b
    ok &= ~diff_sf | near_sf
    # same scale, different element code: the scaled value sits on a code midpoint
    sv = e4m3_values(sf_a)
    r = np.where(sv > 0, gs / np.where(sv > 0, sv, 1), 0)
    scaled = np.abs(blk * r[..., None])
    emids = (E2M1_MAG[1:] + E2M1_MAG[:-1]) / 2
    near_c = np.min(np.abs(scaled[..., None] - emids) / np.maximum(scaled[..., None], 1e-30),
                    -1) < rel
    ca = np.stack([codes_a & 15, codes_a >> 4], -1).reshape(R, nb, 16)
    cb = np.stack([codes_b & 15, codes_b >> 4], -1).reshape(R, nb, 16)
    # +0 and -0 decode alike
    same = (ca == cb) | (((ca & 7) == 0) & ((cb & 7) == 0))
    elem_ok = same | near_c
    ok &= diff_sf | elem_ok.all(-1)
    return ok


def bf16_rn_from_f64(v):
    """fp64 array -> bf16 bit patterns, one rounding to nearest even (no fp32 step).  The
    truncation of fp32(v) is the bf16 value at or below |v| (every bf16 value is an fp32
    value, so the fp32 rounding never crosses one); of it and the next bf16 value up the
    nearer wins, a tie going to the even pattern."""
    v = np.asarray(v, np.float64)
    lo = (np.abs(v).astype(np.float32).view(np.uint32) >> 16).astype(np.uint32)
    hi = lo + 1
    f = lambda b: (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    a = np.abs(v)
    dl, dh = a - f(lo), f(hi) - a
    pick = np.where(dl < dh, lo, np.where(dh < dl, hi, np.where(lo & 1, hi, lo)))
    sign = np.signbit(v).astype(np.uint32) << 15
    return (pick | sign).astype(np.uint16)


def bf16_adjacent_near_midpoint(got, ref64, rel):
    """Mask of elements where the bf16 patterns got and bf16_rn(ref64) agree, or are adjacent
    values with ref64 near the midpoint between them (an fp32-accumulated value can round to
    either side there): within rel of max(|ref64|, 1e-2 x its row's largest magnitude), since
    the accumulation error of a value that cancels scales with its row, not with itself."""
    want = bf16_rn_from_f64(ref64)
    same = got == want
    g = np.asarray(got, np.uint16).astype(np.int64)
    w = want.astype(np.int64)
    adjacent = (np.abs(g - w) == 1) & ((g >> 15) == (w >> 15))
    gv = (g.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    wv = (w.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    mid = (gv + wv) / 2
    ref64 = np.asarray(ref64, np.float64)
    row = np.max(np.abs(ref64), axis=-1, keepdims=True)
    near = np.abs(ref64 - mid) <= rel * np.maximum(np.maximum(np.abs(ref64), 1e-2 * row), 1e-300)
    return same | (adjacent & near)
