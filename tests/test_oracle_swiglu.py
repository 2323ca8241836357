"""Pins of the oracle's SwiGLU + NVFP4 requantisation (``oracle.swiglu_requant``), the
checker of the GPU's standalone ``moe_swiglu_requant`` and of the fused gate_up epilogue.

The operation ("Serving Solar Open 2 (NVFP4) on DGX Spark", section on reading real NVFP4
checkpoints: the fused gate/up projection, FP8 block scales clamped at 448; the layer's
SwiGLU with gate = the first I columns): for fp32 gate/up rows [R][2I], s = silu(g) * u,
rounded to fp32, then NVFP4 with the static global scale gs_i (E4M3 scale per 16 elements,
E2M1 codes, round to nearest even, saturating).

Pinned against things other than the oracle itself:
  * an independent restatement of the quantiser built on torch's float8_e4m3fn cast and a
    brute-force nearest-E2M1 search, fed with numpy's fp64 SwiGLU;
  * exact round trips: blocks whose silu(g) * u is built on the NVFP4 grid of a
    power-of-two gs_i (g = 64, where silu(g) == g in fp64) come back exactly;
  * gate and up swapped give different codes; a zero row gives all-zero codes and scales.
"""
import numpy as np
import torch

import oracle
from helpers import dequant_independent

E2M1_MAG = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def swiglu_f64(gu, I):
    g = gu[:, :I].astype(np.float64)
    u = gu[:, I:].astype(np.float64)
    return g / (1.0 + np.exp(-g)) * u


def nvfp4_independent(s32, gs):
    """NVFP4 of fp32 rows [R, K] with scale gs, restated from the format definitions:
    sf = E4M3(max|block| * gs / 6) (torch's RNE cast after clamping at 448), r = gs / sf,
    code = nearest E2M1 magnitude of |s * r| (ties to the even code), sign bit kept; a zero
    scale gives all-zero codes.  Every step in fp32."""
    R, K = s32.shape
    blk = s32.reshape(R, K // 16, 16).astype(np.float32)
    m = np.abs(blk).max(-1)
    q = (m * np.float32(gs)).astype(np.float32) / np.float32(6.0)
    q = np.minimum(q.astype(np.float32), np.float32(448.0))
    sf = torch.from_numpy(np.ascontiguousarray(q)).to(torch.float8_e4m3fn)
    sf_bytes = sf.view(torch.uint8).numpy().copy()
    sfv = sf.float().numpy()
    r = np.where(sfv > 0, np.float32(gs) / np.where(sfv > 0, sfv, np.float32(1)), 0)
    y = (blk * r.astype(np.float32)[..., None]).astype(np.float32)
    a = np.minimum(np.abs(y).astype(np.float64), 6.0)
    d = np.abs(a[..., None] - E2M1_MAG)
    best = d.min(-1, keepdims=True)
    tie = (d == best)
    # among equally near magnitudes take the even code index (round to nearest even)
    idx = np.where(tie[..., ::1] & (np.arange(8) % 2 == 0), np.arange(8), 99).min(-1)
    idx = np.where(tie.sum(-1) > 1, idx, d.argmin(-1))
    sign = np.signbit(y).astype(np.int64)
    code = (sign << 3) | idx
    code = np.where((sf_bytes == 0)[..., None], 0, code).reshape(R, K)
    packed = (code[:, 0::2] | (code[:, 1::2] << 4)).astype(np.uint8)
    return packed, sf_bytes.reshape(R, K // 16)


def test_swiglu_requant_matches_an_independent_restatement():
    rng = np.random.default_rng([21, 1])
    R, I, gs = 37, 192, 64.0
    gu = (rng.standard_normal((R, 2 * I)) * 3).astype(np.float32)
    gu[3] *= 40          # saturating blocks
    gu[5, :I] = 0.0      # a row whose gate is zero: s == 0 everywhere
    codes, sf, s = oracle.swiglu_requant(gu, I, gs)
    ref_s = swiglu_f64(gu, I)
    assert np.max(np.abs(s - ref_s) / np.maximum(np.abs(ref_s), 1e-300)) <= 1e-15
    s32 = ref_s.astype(np.float32)
    assert np.array_equal(s.astype(np.float32), s32)
    rc, rs = nvfp4_independent(s32, gs)
    assert np.array_equal(sf, rs)
    assert np.array_equal(codes, rc)
    assert np.all(codes[5] == 0) and np.all(sf[5] == 0)


def test_swiglu_requant_round_trips_values_on_the_grid():
    """gate = 64 (silu(64) == 64 in fp64, so s = 64 u exactly) and up = v / 64 with v on the
    NVFP4 grid of the power-of-two scale gs_i: every block has a maximum of 6 * S / gs_i for an
    E4M3 value S, so the codes and scales reproduce v exactly."""
    rng = np.random.default_rng([21, 2])
    R, I, gs = 8, 128, 16.0
    S = torch.tensor([2.0 ** -3, 0.625, 1.0, 1.75, 3.0, 40.0, 240.0, 448.0])
    v = np.empty((R, I), np.float64)
    for r in range(R):
        mags = E2M1_MAG[rng.integers(0, 8, size=I)]
        mags.reshape(-1, 16)[:, 0] = 6.0  # each block's maximum
        signs = np.where(rng.random(I) < 0.5, -1.0, 1.0)
        v[r] = signs * mags * float(S[r]) / gs
    gu = np.empty((R, 2 * I), np.float32)
    gu[:, :I] = 64.0
    gu[:, I:] = (v / 64.0).astype(np.float32)
    assert np.array_equal(gu[:, I:].astype(np.float64) * 64.0, v)  # exact in fp32
    codes, sf, s = oracle.swiglu_requant(gu, I, gs)
    assert np.array_equal(s, v)
    assert np.array_equal(dequant_independent(codes, sf, gs), v)
    # gate and up exchanged: s = silu(v / 64) * 64, not v
    swapped = np.concatenate([gu[:, I:], gu[:, :I]], axis=1)
    c2, s2, _ = oracle.swiglu_requant(swapped, I, gs)
    assert not np.array_equal(c2, codes)


def test_swiglu_requant_zero_rows_and_row_pitch():
    """A zero row gives zero codes and scales; rows are 2I apart (each row's gate and up are
    its own: rows built with distinct magnitudes keep them)."""
    R, I, gs = 5, 64, 8.0
    gu = np.zeros((R, 2 * I), np.float32)
    for r in range(1, R):
        gu[r, :I] = 64.0
        gu[r, I:] = np.float32(6.0 * 2.0 ** r / gs / 64.0)  # s = 6 * 2^r / gs in every element
    codes, sf, s = oracle.swiglu_requant(gu, I, gs)
    assert np.all(codes[0] == 0) and np.all(sf[0] == 0) and np.all(s[0] == 0)
    deq = dequant_independent(codes, sf, gs)
    for r in range(1, R):
        assert np.all(deq[r] == 6.0 * 2.0 ** r / gs)


def test_swiglu_requant_quantises_the_fp32_rounding_of_s():
    """s is rounded to fp32 before it is quantised.  gate = 64 + 2^-17 (silu == gate in fp64)
    times up = 2^-12 (1 - 2^-24) is s = 2^-6 (1 + 2^-24 - 2^-47) exactly in fp64, just above
    the E2M1 midpoint 0.25 / r (r = 16 here, set by a block maximum of 6 / 16); its fp32
    rounding is the midpoint itself, which rounds to the even code 0 -- while the fp64 value
    would round up to code 1 (0.5)."""
    I, gs = 64, 16.0
    gu = np.zeros((1, 2 * I), np.float32)
    gu[0, :I] = 64.0
    gu[0, I:] = np.float32(6.0 / 16.0 / 64.0)          # s = 0.375: the block maximum
    gu[0, 3] = np.float32(64.0 + 2.0 ** -17)
    gu[0, I + 3] = np.float32(2.0 ** -12 * (1.0 - 2.0 ** -24))
    assert float(gu[0, I + 3]) == 2.0 ** -12 * (1.0 - 2.0 ** -24)
    codes, sf, s = oracle.swiglu_requant(gu, I, gs)
    assert s[0, 3] > 2.0 ** -6 and np.float32(s[0, 3]) == np.float32(2.0 ** -6)
    assert sf[0, 0] == 0x38                              # E4M3 1.0
    nib = (codes[0, 1] >> 4) & 15                        # element 3: high nibble of byte 1
    assert nib == 0
    rc, rs = nvfp4_independent(s.astype(np.float32), gs)
    assert np.array_equal(codes, rc) and np.array_equal(sf, rs)
