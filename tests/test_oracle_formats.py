"""Pins of the oracle's NVFP4 formats and quantiser against things other than itself:
the published E2M1/E4M3 value tables (tests/golden), torch's float8_e4m3fn conversion (a
library routine), brute-force nearest-point searches, and closed-form round trips."""
import os

import numpy as np
import pytest
import torch

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _e2m1_table():
    vals = {}
    for line in open(os.path.join(GOLD, "e2m1_values.txt")):
        if line.startswith("#") or not line.strip():
            continue
        c, v = line.split()
        vals[int(c)] = float(v)
    return vals


E2M1 = _e2m1_table()
E2M1_MAG = np.array([E2M1[c] for c in range(8)])


def _torch_e4m3_value(code):
    return float(torch.tensor([code], dtype=torch.uint8).view(torch.float8_e4m3fn).float()[0])


def test_e2m1_values_match_published_table():
    for c in range(16):
        v = oracle.e2m1_value(c)
        assert v == E2M1[c]
        assert np.signbit(v) == (c >= 8)


def test_e4m3_values_match_published_points_and_torch():
    for line in open(os.path.join(GOLD, "e4m3_points.txt")):
        if line.startswith("#") or not line.strip():
            continue
        c, v = line.split()
        got = oracle.e4m3_value(int(c, 16))
        if v == "nan":
            assert np.isnan(got)
        else:
            assert got == float(v) and np.signbit(got) == np.signbit(float(v))
    for c in range(256):
        ref = _torch_e4m3_value(c)
        got = oracle.e4m3_value(c)
        if np.isnan(ref):
            assert np.isnan(got), c
        else:
            assert got == ref, (c, got, ref)


def test_e2m1_encode_is_nearest_with_ties_to_even():
    # every midpoint between neighbouring points goes to the even code
    mids = {0.25: 0, 0.75: 2, 1.25: 2, 1.75: 4, 2.5: 4, 3.5: 6, 5.0: 6}
    for m, code in mids.items():
        assert oracle.e2m1_encode(m) == code, m
        assert oracle.e2m1_encode(-m) == code | 8, m
    # brute force: the chosen point is a nearest point of the published table
    rng = np.random.default_rng(7)
    xs = np.concatenate([rng.uniform(-8, 8, 3000), rng.uniform(-1, 1, 1000)]).astype(np.float32)
    for x in xs:
        c = oracle.e2m1_encode(float(x))
        a = min(abs(float(x)), 6.0)
        d = np.abs(E2M1_MAG - a)
        assert abs(E2M1_MAG[c & 7] - a) == d.min()
        assert (c >= 8) == bool(np.signbit(x))
    # saturation and signed zero
    assert oracle.e2m1_encode(1e30) == 7
    assert oracle.e2m1_encode(-7.0) == 15
    assert oracle.e2m1_encode(-0.1) == 8


def test_e4m3_encode_matches_torch_rne_in_range():
    rng = np.random.default_rng(11)
    xs = np.concatenate([
        rng.uniform(0, 448, 20000),
        np.exp(rng.uniform(np.log(2.0 ** -12), np.log(448.0), 20000)),
    ]).astype(np.float32)
    # every exact midpoint between consecutive positive codes as well
    pts = [oracle.e4m3_value(c) for c in range(127)]
    mids = np.array([(pts[i] + pts[i + 1]) / 2 for i in range(126)], np.float32)
    xs = np.concatenate([xs, mids])
    ref = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(float(x)) for x in xs], np.uint8)
    assert np.array_equal(got, ref)


def test_e4m3_encode_saturates_at_448():
    for x in (448.0, 449.0, 463.9, 464.0, 480.0, 1e6, 3e38):
        assert oracle.e4m3_encode(x) == 0x7E
    assert oracle.e4m3_encode(-1e6) == 0xFE


def test_bf16_round_matches_torch_on_fp32_values_and_ties():
    rng = np.random.default_rng(3)
    xs = (rng.standard_normal(5000) * np.exp(rng.uniform(-30, 30, 5000))).astype(np.float32)
    ref = torch.from_numpy(xs).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    got = np.array([oracle.bf16_round(float(x)) for x in xs], np.uint16)
    assert np.array_equal(got, ref)
    # ties to even: 1 + 2^-8 is halfway between 1 and 1 + 2^-7
    assert oracle.bf16_round(1.0 + 2.0 ** -8) == 0x3F80
    assert oracle.bf16_round(1.0 + 3 * 2.0 ** -8) == 0x3F82
    # fp64 input rounded once (no double rounding through fp32)
    assert oracle.bf16_round(1.0 + 2.0 ** -8 + 2.0 ** -40) == 0x3F81


# ------------------------------------------------------------------ quantiser

def _dequant_independent(codes, sf, gs, K):
    """Dequantise with the published E2M1 table and torch's E4M3 decode."""
    c = np.empty((codes.shape[0], K), np.int64)
    c[:, 0::2] = codes & 15
    c[:, 1::2] = codes >> 4
    e2 = np.array([E2M1[i] for i in range(16)])[c]
    s = torch.from_numpy(np.ascontiguousarray(sf)).view(torch.float8_e4m3fn).double().numpy()
    return e2 * np.repeat(s, 16, axis=1) / np.float64(gs)


def test_quant_round_trip_on_grid_values():
    """Blocks built exactly on the grid (one element at 6 * sf / gs, gs a power of two)
    quantise back to the same codes and scales."""
    rng = np.random.default_rng(5)
    R, K = 64, 256
    gs = np.float32(2.0 ** 7)
    sf = rng.integers(0x20, 0x70, size=(R, K // 16)).astype(np.uint8)
    codes = rng.integers(0, 16, size=(R, K)).astype(np.uint8)
    codes[:, ::16] = np.where(rng.random((R, K // 16)) < 0.5, 7, 15)  # a +-6 in each block
    s_val = torch.from_numpy(sf).view(torch.float8_e4m3fn).double().numpy()
    x = np.array([[E2M1[int(c)] for c in row] for row in codes]) * np.repeat(s_val, 16, 1) / float(gs)
    got_c, got_sf, g = oracle.quant_nvfp4(x.astype(np.float32), gs=float(gs))
    assert g == float(gs)
    assert np.array_equal(got_sf, sf)
    want = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    # -0 and +0 both decode to 0; the quantiser keeps the sign of its input
    zero_lo = (codes[:, 0::2] & 7) == 0
    zero_hi = (codes[:, 1::2] & 7) == 0
    gl, gh = got_c & 15, got_c >> 4
    assert np.array_equal(np.where(zero_lo, gl & 7, gl), np.where(zero_lo, 0, codes[:, 0::2]))
    assert np.array_equal(np.where(zero_hi, gh & 7, gh), np.where(zero_hi, 0, codes[:, 1::2]))
    assert np.array_equal(got_c[~(zero_lo | zero_hi)], want[~(zero_lo | zero_hi)])


def test_quant_dynamic_scale_and_nearest_codes():
    rng = np.random.default_rng(9)
    R, K = 48, 512
    x = rng.standard_normal((R, K)).astype(np.float32)
    x[3, 17] = 37.5  # amax
    codes, sf, gs = oracle.quant_nvfp4(x)
    assert gs == float(np.float32(2688.0) / np.float32(37.5))
    # block scales: E4M3 of (m*gs)/6 in fp32, checked with torch's E4M3 rounding
    m = np.abs(x).reshape(R, K // 16, 16).max(-1).astype(np.float32)
    q = ((m * np.float32(gs)).astype(np.float32) / np.float32(6)).astype(np.float32)
    ref_sf = torch.from_numpy(q).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(sf, ref_sf)
    # every code is a nearest E2M1 point of x * (gs / sf) in fp32
    s_val = torch.from_numpy(sf).view(torch.float8_e4m3fn).float().numpy()
    r = (np.float32(gs) / s_val).astype(np.float32)
    scaled = (x * np.repeat(r, 16, 1)).astype(np.float32)
    c = np.empty((R, K), np.int64)
    c[:, 0::2] = codes & 15
    c[:, 1::2] = codes >> 4
    chosen = E2M1_MAG[c & 7]
    a = np.minimum(np.abs(scaled.astype(np.float64)), 6.0)
    best = np.abs(E2M1_MAG[None, None, :] - a[..., None]).min(-1)
    assert np.array_equal(np.abs(chosen - a), best)
    assert np.array_equal(c >= 8, np.signbit(scaled))
    # the largest element maps to the top of both ranges: 448 scale, code 6
    assert sf[3, 1] == 0x7E and (c[3, 17] & 7) == 7


def test_quant_zero_block_and_zero_tensor():
    x = np.zeros((2, 32), np.float32)
    x[1, 20] = 1.0
    codes, sf, gs = oracle.quant_nvfp4(x)
    assert sf[0].tolist() == [0, 0] and sf[1, 0] == 0 and sf[1, 1] == 0x7E
    assert not codes[0].any() and not codes[1, :8].any()
    c0, s0, g0 = oracle.quant_nvfp4(np.zeros((1, 16), np.float32))
    assert g0 == 1.0 and s0[0, 0] == 0 and c0[0].tolist() == [0] * 8


def test_quant_error_bound():
    """|x - dequant| <= half the E2M1 step at that magnitude, times sf / gs (plus the
    saturated top), with the dequantisation done independently of the oracle."""
    rng = np.random.default_rng(13)
    x = (rng.standard_normal((32, 1024)) * 3).astype(np.float32)
    codes, sf, gs = oracle.quant_nvfp4(x)
    deq = _dequant_independent(codes, sf, gs, 1024)
    s = torch.from_numpy(sf).view(torch.float8_e4m3fn).double().numpy()
    unit = np.repeat(s, 16, 1) / gs          # value of one E2M1 unit in this block
    err = np.abs(deq - x.astype(np.float64))
    # largest step between E2M1 points is 2 (4 -> 6): half of it bounds the error
    # as long as x*r <= 6 (+ the slack of the E4M3 rounding of the scale, <= 1/16)
    assert np.all(err <= unit * 1.0 * (1 + 1.0 / 16) + 1e-12)
    rel = np.linalg.norm(deq - x) / np.linalg.norm(x)
    assert rel < 0.12


def test_dequant_matches_independent_decode():
    rng = np.random.default_rng(17)
    x = rng.standard_normal((8, 128)).astype(np.float32)
    codes, sf, gs = oracle.quant_nvfp4(x)
    assert np.array_equal(oracle.dequant_nvfp4(codes, sf, gs), _dequant_independent(codes, sf, gs, 128))
