"""Pins of the oracle's checkpoint-convention weight preparation (the packed-weights
section of the pages: reciprocal global scale inverted and folded into the FP8 block
scales with re-rounding and the 448 clamp, gate/up row order, per-shard slicing):
re-rounding against a brute-force nearest-even search over torch's own E4M3 value table,
identity and convention-equivalence cases, the folding error bound, slicing and order."""
import numpy as np
import pytest
import torch

import oracle

E4M3 = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn) \
    .to(torch.float64).numpy()
POS = np.arange(127)  # the non-negative finite codes, increasing in value


def _brute_e4m3(x):
    """Nearest non-negative E4M3 code to x >= 0 by exhaustive search; exact ties go to the
    code with an even mantissa; 448 and above give 448."""
    x = float(x)
    if x >= E4M3[126]:
        return 126
    d = np.abs(E4M3[POS] - x)
    best = np.flatnonzero(d == d.min())
    if len(best) == 1:
        return int(best[0])
    return int(best[0] if best[0] % 2 == 0 else best[1])


def _one(sf_codes, gs, **kw):
    """prepare_weights on one expert whose block scales are sf_codes (1 row)."""
    sf = np.asarray(sf_codes, np.uint8).reshape(1, 1, -1)
    K = 16 * sf.shape[2]
    codes = np.zeros((1, 1, K // 2), np.uint8)
    return oracle.prepare_weights(codes, sf, np.array([gs], np.float32), **kw)


@pytest.mark.parametrize("gs,target", [(2688.0, 1.0), (300.0, 2688.0), (96.5, 96.5 * 3),
                                       (1e4, 1.0 / 7), (5.0, 640.0), (2.0 ** 20, 2.0 ** 8)])
def test_fold_rerounds_every_scale_code_to_the_nearest_even(gs, target):
    co, so, go = _one(POS, gs, fold_target=target)
    assert go[0] == np.float32(target)
    r = np.float32(target) / np.float32(gs)
    want = [_brute_e4m3(np.float32(E4M3[c]) * r) for c in POS]
    assert np.array_equal(so[0, 0], np.array(want, np.uint8))


def test_fold_with_ratio_one_is_the_identity_and_no_fold_copies():
    for gs in (1.0, 2688.0, 37.25):
        assert np.array_equal(_one(POS, gs, fold_target=gs)[1][0, 0], POS.astype(np.uint8))
        co, so, go = _one(POS, gs)
        assert np.array_equal(so[0, 0], POS.astype(np.uint8)) and go[0] == np.float32(gs)


def test_dequant_multiplier_convention_is_the_reciprocal():
    rng = np.random.default_rng(4)
    codes = rng.integers(0, 256, (4, 8, 32), dtype=np.uint8)
    sf = rng.integers(0, 127, (4, 8, 4), dtype=np.uint8)
    gs = np.float32(2.0) ** rng.integers(-10, 14, 4).astype(np.float32)   # exact reciprocals
    a = oracle.prepare_weights(codes, sf, gs, fold_target=64.0)
    b = oracle.prepare_weights(codes, sf, (1.0 / gs).astype(np.float32),
                               convention=oracle.GS_DEQUANT, fold_target=64.0)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
    m = np.array([3.0e-4, 0.7], np.float32)
    _, _, g = oracle.prepare_weights(codes[:2], sf[:2], m, convention=oracle.GS_DEQUANT)
    assert np.array_equal(g, (np.float32(1.0) / m).astype(np.float32))


def test_folded_value_error_is_within_half_an_e4m3_step():
    rng = np.random.default_rng(5)
    sf = rng.integers(1, 127, 4096).astype(np.uint8)
    gs, target = np.float32(1700.0), np.float32(900.0)
    _, so, _ = _one(sf, gs, fold_target=target)
    before = E4M3[sf] / gs
    after = E4M3[so[0, 0]] / target
    rel = np.abs(after - before) / before
    normal = E4M3[sf] * (target / gs) >= 2.0 ** -6      # E4M3 normal range after the fold
    assert rel[normal].max() <= 2.0 ** -4 * (1 + 1e-6)  # half a step of a 3-bit mantissa


def test_fold_saturates_at_448():
    _, so, _ = _one([126, 120, 119], 100.0, fold_target=400.0)   # x4: 448*4, 256*4, 240*4
    assert np.array_equal(so[0, 0], np.array([126, 126, 126], np.uint8))


def test_shard_slicing_and_gate_up_order():
    rng = np.random.default_rng(6)
    E, N, K = 6, 12, 64
    codes = rng.integers(0, 256, (E, N, K // 2), dtype=np.uint8)
    sf = rng.integers(0, 127, (E, N, K // 16), dtype=np.uint8)
    gs = rng.uniform(10, 3000, E).astype(np.float32)
    co, so, go = oracle.prepare_weights(codes, sf, gs, swap_halves=True, off=2, count=3)
    order = np.r_[np.arange(N // 2, N), np.arange(N // 2)]
    assert np.array_equal(co, codes[2:5][:, order])
    assert np.array_equal(so, sf[2:5][:, order])
    assert np.array_equal(go, gs[2:5])
