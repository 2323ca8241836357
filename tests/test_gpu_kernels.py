"""GPU parity of each C-ABI call against the oracle, on seeded inputs that span several
tiles and k-stages with ragged tails.  Integer work (top-k ids, grouping, NVFP4 codes and
scales) is compared bit for bit; contractions within fp32-accumulation tolerances."""
import numpy as np
import pytest
import torch

import nvfp4_mixture_experts_gb300 as moe
import oracle
import synth
from gpu_util import (bf16_adjacent_near_midpoint, bf16_rn_from_f64, bits16,
                      canonical_to_tiled, dev, host, make_layer,
                      quant_decisions_near_boundary, tiled_to_canonical)
from helpers import build_layer, within_layer_tolerance

pytestmark = pytest.mark.gpu


def _ws(nbytes):
    return torch.zeros(max(nbytes, 256), dtype=torch.uint8, device="cuda")


# ---------------------------------------------------------------- failure path of the waits

def test_bounded_wait_runs_out_sets_status_and_leaves_the_context_usable():
    """A wait on an mbarrier phase that nothing completes gives up after its limit, reports
    MOE_DEV_WAIT_TIMEOUT through the status word, and returns (no trap); the GPU then runs
    the quantiser bit-exactly as before."""
    import time
    word = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert moe.moe_selftest_bounded_wait(word, 0) == moe.MOE_ERR_INVALID
    assert moe.moe_selftest_bounded_wait(word, 3 * 10 ** 9) == moe.MOE_ERR_INVALID
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    st = moe.moe_selftest_bounded_wait(word, 2 * 10 ** 6)  # 2 ms
    dt = time.perf_counter() - t0
    assert st == moe.MOE_ERR_TIMEOUT
    assert int(host(word)[0]) & moe.MOE_DEV_WAIT_TIMEOUT
    assert dt >= 2e-3
    test_quant_nvfp4_dynamic_bit_exact(300, 512, 1)


# ---------------------------------------------------------------- quantiser

@pytest.mark.parametrize("R,K,layout", [(300, 512, 0), (300, 512, 1), (1, 64, 0), (129, 4096, 1),
                                        (64, 1280, 1)])
def test_quant_nvfp4_dynamic_bit_exact(R, K, layout):
    x = synth.activations(3, R, K, outlier_frac=0.02)
    xd = bits16(x)
    codes = torch.zeros((((R + 127) // 128) * 128 if layout else R) * (
        (K // 2 + 127) // 128 * 128 if layout else K // 2), dtype=torch.uint8, device="cuda")
    sf = torch.zeros((((R + 127) // 128) * 128 if layout else R) * (K // 16),
                     dtype=torch.uint8, device="cuda")
    gs = torch.zeros(1, dtype=torch.float32, device="cuda")
    moe.moe_quant_nvfp4(xd, R, K, None, gs, codes, sf, layout, _ws(256))
    torch.cuda.synchronize()
    rc, rs, rg = oracle.quant_nvfp4(synth.bf16_to_f32(x))
    assert float(host(gs)[0]) == rg
    if layout:
        c, s = tiled_to_canonical(host(codes), host(sf), R, K)
    else:
        c, s = host(codes).reshape(R, K // 2), host(sf).reshape(R, K // 16)
    assert np.array_equal(s, rs)
    assert np.array_equal(c, rc)


def test_quant_nvfp4_static_scale_and_zero_rows():
    R, K = 40, 256
    x = synth.activations(4, R, K)
    x[5] = 0  # a zero row: every scale 0, every code +0
    gsv = np.float32(96.0)
    codes = torch.zeros(R * K // 2, dtype=torch.uint8, device="cuda")
    sf = torch.zeros(R * K // 16, dtype=torch.uint8, device="cuda")
    moe.moe_quant_nvfp4(bits16(x), R, K, dev(np.array([gsv])), None, codes, sf, 0, None)
    rc, rs, _ = oracle.quant_nvfp4(synth.bf16_to_f32(x), gs=float(gsv))
    assert np.array_equal(host(sf).reshape(R, -1), rs)
    assert np.array_equal(host(codes).reshape(R, -1), rc)
    assert not host(codes).reshape(R, -1)[5].any()


def test_swiglu_requant_matches_oracle_up_to_boundaries():
    R, I, gs_i = 150, 256, 64.0
    rng = np.random.default_rng(8)
    gu = (rng.standard_normal((R, 2 * I)) * 1.5).astype(np.float32)
    codes = torch.zeros(R * I // 2, dtype=torch.uint8, device="cuda")
    sf = torch.zeros(R * I // 16, dtype=torch.uint8, device="cuda")
    moe.moe_swiglu_requant(dev(gu), R, I, gs_i, codes, sf, 0)
    rc, rs, s = oracle.swiglu_requant(gu, I, gs_i)
    gc, gsf = host(codes).reshape(R, -1), host(sf).reshape(R, -1)
    ok = quant_decisions_near_boundary(s, gs_i, rs, gsf, rc, gc)
    assert ok.all(), np.argwhere(~ok)[:5]
    assert (gsf == rs).mean() > 0.999


# ---------------------------------------------------------------- routing

def zero_layer(H, I, El):
    """All-zero NVFP4 experts (valid weights for calls that do not read them)."""
    z = lambda *shape: np.zeros(shape, np.uint8)
    one = lambda n: np.ones(n, np.float32)
    return oracle.Layer(z(El, 2 * I, H // 2), z(El, 2 * I, H // 16), one(El),
                        z(El, H, I // 2), z(El, H, I // 16), one(El),
                        z(2 * I, H // 2), z(2 * I, H // 16), 1.0, z(H, I // 2), z(H, I // 16), 1.0)


def _tiny_layer_handle(E=320, H=256, I=64, k=8, E_loc=None, **kw):
    El = E if E_loc is None else E_loc
    wr = synth.router_weight(0, E, H)
    return make_layer(zero_layer(H, I, El), wr, H, I, E, k, E_loc=El, inter_gs=64.0, **kw), wr


def test_topk_from_given_logits_bit_exact():
    T, E, k = 300, 320, 8
    h, _ = _tiny_layer_handle(E=E, k=k)
    lg = synth.logits_normal(5, T, E)
    lg[:50] = np.round(lg[:50] * 4) / 4  # exact ties -> lower id first
    ids = torch.zeros((T, k), dtype=torch.int32, device="cuda")
    w = torch.zeros((T, k), dtype=torch.float32, device="cuda")
    moe.moe_route_topk(h.handle, None, dev(lg), None, T, ids, w, None, None)
    rid, rw = oracle.topk(lg.astype(np.float64), k)
    assert np.array_equal(host(ids), rid)
    assert np.max(np.abs(host(w) - rw)) <= 1e-6
    # a bias whose sums are exact in fp32 and fp64 alike
    bias = (np.arange(E) % 7 * 0.25).astype(np.float32)
    lgq = (np.round(lg * 1024) / 1024).astype(np.float32)
    moe.moe_route_topk(h.handle, None, dev(lgq), dev(bias), T, ids, w, None, None)
    rid, rw = oracle.topk(lgq.astype(np.float64) + bias, k)
    assert np.array_equal(host(ids), rid)


@pytest.mark.parametrize("E,k,T,offset", [(37, 5, 70, 0), (320, 32, 33, 1), (1023, 32, 17, 0),
                                          (64, 1, 129, 1), (200, 8, 40, 0), (500, 8, 20, 1)])
def test_topk_edge_shapes_signed_zeros_and_unaligned_logits(E, k, T, offset):
    """E not a multiple of 4 and logits 4 bytes off a 16-byte boundary take the scalar load
    path; k up to 32; +0 and -0 rank as equal values (lower id first); blocks of 16 tokens
    with a ragged last block."""
    h, _ = _tiny_layer_handle(E=E, k=k)
    rng = np.random.default_rng(E + k)
    lg = np.round(rng.standard_normal((T, E)) * 2).astype(np.float32) / 2
    lg[:, ::5] = 0.0
    lg[:, 1::7] = -0.0
    lg[T // 2:, :] = np.abs(lg[T // 2:, :]) * -1.0  # all-negative rows (with -0 maxima)
    buf = torch.zeros(T * E + 4, dtype=torch.float32, device="cuda")
    buf[offset:offset + T * E] = torch.from_numpy(lg.reshape(-1)).cuda()
    ids = torch.zeros((T, k), dtype=torch.int32, device="cuda")
    w = torch.zeros((T, k), dtype=torch.float32, device="cuda")
    moe.moe_route_topk(h.handle, None, buf[offset:], None, T, ids, w, None, None)
    rid, rw = oracle.topk(lg.astype(np.float64), k)
    assert np.array_equal(host(ids), rid)
    assert np.max(np.abs(host(w) - rw)) <= 1e-6


def test_topk_nan_logits_rank_below_every_number():
    T, E, k = 20, 64, 8
    h, _ = _tiny_layer_handle(E=E, k=k)
    lg = synth.logits_normal(9, T, E)
    lg[::2, ::3] = np.nan
    ids = torch.zeros((T, k), dtype=torch.int32, device="cuda")
    w = torch.zeros((T, k), dtype=torch.float32, device="cuda")
    moe.moe_route_topk(h.handle, None, dev(lg), None, T, ids, w, None, None)
    rid, rw = oracle.topk(np.where(np.isnan(lg), -np.inf, lg).astype(np.float64), k)
    assert np.array_equal(host(ids), rid)
    assert np.max(np.abs(host(w) - rw)) <= 1e-6


@pytest.mark.parametrize("T", [200, 1100])  # 64-expert tiles; 160-expert tiles, ragged rows
def test_router_logits_and_topk_from_x(T):
    E, H, k = 320, 4096, 8
    h, wr = _tiny_layer_handle(E=E, H=H, k=k, max_tokens=max(T, 256))
    x = synth.activations(6, T, H)
    ids = torch.zeros((T, k), dtype=torch.int32, device="cuda")
    w = torch.zeros((T, k), dtype=torch.float32, device="cuda")
    lo = torch.zeros((T, E), dtype=torch.float32, device="cuda")
    moe.moe_route_topk(h.handle, bits16(x), None, None, T, ids, w, lo,
                       _ws(h.workspace_bytes(T)))
    ref = oracle.router_logits(x, wr)
    got = host(lo).astype(np.float64)
    # fp32 accumulation of 4096 exact products: error << 1e-4 of the sum of |terms|
    mag = np.abs(synth.bf16_to_f32(x).astype(np.float64)) @ np.abs(
        synth.bf16_to_f32(wr).astype(np.float64)).T
    assert np.all(np.abs(got - ref) <= 1e-5 * mag + 1e-6)
    rid, rw = oracle.topk(ref, k)
    srt = -np.sort(-ref, axis=1)
    thr = 2e-5 * mag.max(1)
    set_ok = srt[:, k - 1] - srt[:, k] > thr          # the selected set is unique
    ord_ok = (np.diff(-srt[:, :k + 1], axis=1) > thr[:, None]).all(1)  # and its order
    assert set_ok.mean() > 0.95
    assert np.array_equal(np.sort(host(ids)[set_ok], 1), np.sort(rid[set_ok], 1))
    assert np.array_equal(host(ids)[ord_ok], rid[ord_ok])
    assert np.max(np.abs(host(w)[ord_ok] - rw[ord_ok])) <= 1e-5


# ---------------------------------------------------------------- grouping

@pytest.mark.parametrize("T,E_loc,off,add_shared", [(1, 320, 0, 1), (64, 320, 0, 1),
                                                    (300, 160, 160, 0), (2000, 160, 0, 1),
                                                    (2000, 37, 100, 0), (9000, 320, 0, 1)])
def test_permute_bit_exact(T, E_loc, off, add_shared):
    E, k = 320, 8
    h, _ = _tiny_layer_handle(E=E, k=k, E_loc=E_loc, off=off, add_shared=add_shared,
                              max_tokens=max(T, 8192))
    rng = np.random.default_rng(T + E_loc)
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    cap = h.rows_capacity(T)
    counts = torch.zeros(E_loc + 1, dtype=torch.int32, device="cuda")
    offsets = torch.zeros(E_loc + 2, dtype=torch.int32, device="cuda")
    perm = torch.full((cap,), -7, dtype=torch.int32, device="cuda")
    inv = torch.zeros(T * k, dtype=torch.int32, device="cuda")
    ws = _ws(h.workspace_bytes(T))
    rc, rp = oracle.permute(ids, E_loc, off)
    for rep in range(4):  # repeated: a race between the kernel's phases would show up here
        perm.fill_(-7)
        moe.moe_permute(h.handle, dev(ids), T, counts, offsets, perm, inv, ws)
        _check_grouping(host(counts), host(offsets), host(perm), host(inv), rc, rp, T, k,
                        E_loc, add_shared)
    assert moe.moe_get_status(h.handle, ws) == (moe.MOE_OK, 0)


def _check_grouping(c, o, p, iv, rc, rp, T, k, E_loc, add_shared):
    assert np.array_equal(c[:E_loc], rc)
    assert c[E_loc] == (T if add_shared else 0)
    pad = (c + 127) // 128 * 128
    assert np.array_equal(o, np.concatenate([[0], np.cumsum(pad)]))
    got_pairs = np.concatenate([p[o[e]:o[e] + c[e]] for e in range(E_loc)]) if E_loc else []
    assert np.array_equal(got_pairs, rp)
    for g in range(E_loc + 1):
        assert np.all(p[o[g] + c[g]:o[g + 1]] == -1)
    assert np.array_equal(p[o[E_loc]:o[E_loc] + c[E_loc]], T * k + np.arange(c[E_loc]))
    want_inv = np.full(T * k, -1)
    rows = np.concatenate([np.arange(o[e], o[e] + c[e]) for e in range(E_loc)]) if E_loc else []
    want_inv[rp] = rows
    assert np.array_equal(iv, want_inv)


def test_permute_drops_and_flags_bad_ids():
    E, k, T = 320, 8, 10
    h, _ = _tiny_layer_handle(E=E, k=k)
    ids = np.stack([np.arange(k) + 10 * t for t in range(T)]).astype(np.int32)
    ids[3, 2] = 400   # >= E
    ids[7, 0] = -5
    cap = h.rows_capacity(T)
    counts = torch.zeros(E + 1, dtype=torch.int32, device="cuda")
    offsets = torch.zeros(E + 2, dtype=torch.int32, device="cuda")
    perm = torch.zeros(cap, dtype=torch.int32, device="cuda")
    inv = torch.zeros(T * k, dtype=torch.int32, device="cuda")
    ws = _ws(h.workspace_bytes(T))
    moe.moe_permute(h.handle, dev(ids), T, counts, offsets, perm, inv, ws)
    iv = host(inv)
    assert iv[3 * k + 2] == -1 and iv[7 * k] == -1
    assert host(counts)[:E].sum() == T * k - 2
    st, bits = moe.moe_get_status(h.handle, ws)
    assert st == moe.MOE_ERR_DEVICE_STATUS and bits & moe.MOE_DEV_BAD_EXPERT_ID
    assert moe.moe_get_status(h.handle, ws) == (moe.MOE_OK, 0)  # cleared


# ---------------------------------------------------------------- grouped GEMMs

class Staged:
    """Runs the staged calls of one layer up to the grouped GEMMs."""

    def __init__(self, h, x_bits, T, k, logits):
        self.h, self.T, self.k = h, T, k
        cfg = h.cfg
        El = cfg.num_local_experts
        self.cap = cap = h.rows_capacity(T)
        self.ws = _ws(h.workspace_bytes(T))
        self.ids = torch.zeros((T, k), dtype=torch.int32, device="cuda")
        self.w = torch.zeros((T, k), dtype=torch.float32, device="cuda")
        moe.moe_route_topk(h.handle, None, dev(logits), None, T, self.ids, self.w, None, None)
        self.counts = torch.zeros(El + 1, dtype=torch.int32, device="cuda")
        self.offsets = torch.zeros(El + 2, dtype=torch.int32, device="cuda")
        self.perm = torch.zeros(cap, dtype=torch.int32, device="cuda")
        self.inv = torch.zeros(T * k, dtype=torch.int32, device="cuda")
        moe.moe_permute(h.handle, self.ids, T, self.counts, self.offsets, self.perm, self.inv,
                        self.ws)
        H = cfg.hidden
        self.a_codes = torch.zeros(cap * ((H // 2 + 127) // 128 * 128), dtype=torch.uint8,
                                   device="cuda")
        self.a_sf = torch.zeros(cap * H // 16, dtype=torch.uint8, device="cuda")
        self.a_bf16 = torch.zeros(cap * H, dtype=torch.int16, device="cuda")
        self.gs = torch.zeros(1, dtype=torch.float32, device="cuda")
        moe.moe_gather_activations(h.handle, x_bits, T, self.inv, self.offsets, self.a_codes,
                                   self.a_sf, self.a_bf16, self.gs, self.ws)
        torch.cuda.synchronize()

    def rows(self):
        """(padded row, token, group) of every valid row."""
        c, o, p = host(self.counts), host(self.offsets), host(self.perm)
        out = []
        for g in range(len(c)):
            for i in range(c[g]):
                r = o[g] + i
                pair = p[r]
                tok = pair // self.k if pair < self.T * self.k else pair - self.T * self.k
                out.append((r, tok, g))
        return np.array(out, dtype=np.int64).reshape(-1, 3)


def _mid_problem(act_mode, T=200, tiling=0):
    H, I, E, k = 512, 256, 8, 2
    layer = build_layer(12, H, I, E)
    wr = synth.router_weight(12, E, H)
    x = synth.activations(12, T, H, outlier_frac=0.01)
    lg = synth.logits_normal(12, T, E)
    lg[:, 3] += 2.5   # one popular expert: > 128 rows at T=200 (> 208 at T=600)
    h = make_layer(layer, wr, H, I, E, k, act_mode=act_mode, inter_gs=32.0,
                   gemm_tiling=tiling)
    return layer, wr, x, lg, h, (H, I, E, k, T)


def _f16_prescale(x_bits):
    """The W4A16 activation prescale as the header states it: 2^(141 - e) for e the fp32
    exponent field of amax|x|, clamped to 2^[-126, 127] (1 for an all-zero x)."""
    amax = np.max(np.abs(synth.bf16_to_f32(x_bits).astype(np.float32)))
    if amax == 0:
        return np.float32(1.0)
    e = int(np.float32(amax).view(np.uint32) >> 23) & 0xFF
    return np.float32(2.0) ** np.float32(min(127, max(-126, 141 - e)))


@pytest.mark.parametrize("T,H", [(60, 512), (1100, 512), (1030, 1280)])
def test_gather_w4a4_rows_bit_exact(T, H):
    """Every valid padded row holds its token's NVFP4 codes and scales, bit for bit: a lane
    per 16-element block below 1024 tokens, a lane per 64-element k-step from 1024 on
    (H = 1280: 20 k-steps, a partly idle warp per token)."""
    E, k = 8, 2
    h, _ = _tiny_layer_handle(E=E, H=H, I=64, k=k, max_tokens=max(T, 8192))
    x = synth.activations(21, T, H, outlier_frac=0.01)
    st = Staged(h, bits16(x), T, k, synth.logits_normal(21, T, E))
    rc, rs, rg = oracle.quant_nvfp4(synth.bf16_to_f32(x))
    assert float(host(st.gs)[0]) == rg
    c, s = tiled_to_canonical(host(st.a_codes), host(st.a_sf), st.cap, H)
    rows = st.rows()
    assert len(rows) == T * (k + 1)
    assert np.array_equal(c[rows[:, 0]], rc[rows[:, 1]])
    assert np.array_equal(s[rows[:, 0]], rs[rows[:, 1]])


@pytest.mark.parametrize("scale", [1.0, 3e-6, 5e4])
def test_gather_w4a16_rows_are_exact_fp16_copies(scale):
    layer, wr, x, lg, h, (H, I, E, k, T) = _mid_problem(2, 60)
    xs = synth.bf16_bits(synth.bf16_to_f32(x).astype(np.float64) * scale)
    st = Staged(h, bits16(xs), T, k, lg)
    gs = _f16_prescale(xs)
    assert host(st.gs)[0] == gs
    rows = st.rows()
    got = host(st.a_bf16).view(np.uint16).reshape(st.cap, H)[rows[:, 0]]
    want = (synth.bf16_to_f32(xs)[rows[:, 1]].astype(np.float32) * gs).astype(np.float16)
    assert np.array_equal(got, want.view(np.uint16))
    assert np.max(np.abs(want.astype(np.float32))) <= 2.0 ** 15


# W4A16 runs batches of up to 256 tokens with at most 16 expected rows per expert on the
# grouped GEMV (T = 60 here: 15 rows per expert) and the others on the tensor-core kernel
# (T = 100, 200, 300: 32, 64, 64 token rows per tile from T * k / E = 25, 50, 75).
# W4A4 runs both GEMM forms (tiling 1: 128-row blocks, activation slots of 32 rows at T=30,
# 64 at T=60, 128 at T=200; tiling 2: token tiles of up to 208 rows -- one tile with two
# scale row blocks for the > 128-row group at T=200, three tiles (128 + 128 + rest) for the
# > 256-row group at T=600; tiling 3: row blocks on CTA pairs, a group's blocks two at a time,
# the second CTA of an odd group's last pair empty; tiling 4: row blocks x 256 weight rows
# per MMA)
W4A4_CASES = [(0, 30, 1), (0, 30, 2), (0, 30, 3), (0, 30, 4), (0, 60, 1), (0, 60, 2),
              (0, 200, 1), (0, 200, 2), (0, 200, 3), (0, 200, 4), (0, 600, 2), (0, 600, 3),
              (0, 600, 4)]
W4A16_CASES = [(2, 60, 0), (2, 100, 0), (2, 200, 0), (2, 300, 0)]


@pytest.mark.parametrize("act_mode,T,tiling", W4A4_CASES + W4A16_CASES)
def test_grouped_gemm_gateup_unfused_matches_oracle(act_mode, T, tiling):
    layer, wr, x, lg, h, (H, I, E, k, T) = _mid_problem(act_mode, T, tiling)
    st = Staged(h, bits16(x), T, k, lg)
    rows = st.rows()
    if T == 200:
        assert (np.bincount(rows[:, 2], minlength=E + 1) > 128).any()
    if T == 600:
        assert (np.bincount(rows[:, 2], minlength=E + 1) > 256).any()
    G = torch.zeros((st.cap, 2 * I), dtype=torch.float32, device="cuda")
    moe.moe_grouped_gemm_gateup(h.handle, st.a_codes, st.a_sf, st.gs, st.a_bf16, st.counts,
                                st.offsets, 0, G, None, None, None, T, st.ws)
    Gg = host(G)
    cfg = oracle.make_cfg(T, H, I, E, k, act_mode=act_mode, inter_gs=32.0)
    xf = synth.bf16_to_f32(x)
    xc, xsf, gs_a = oracle.quant_nvfp4(xf) if act_mode != 2 else (None, None, 1.0)
    if act_mode != 2:
        assert float(host(st.gs)[0]) == gs_a
    for g in range(E + 1):
        sel = rows[rows[:, 2] == g]
        if len(sel) == 0:
            continue
        e = "shared" if g == E else g
        Go = oracle.expert_rows(cfg, layer, e, x, xc, xsf, gs_a, sel[:, 1].astype(np.int32))[0]
        got = Gg[sel[:, 0]]
        err = np.abs(got - Go)
        scale = np.sqrt(np.mean(Go ** 2))
        assert np.max(err) <= 2e-5 * scale * np.sqrt(H / 64), (g, np.max(err), scale)


@pytest.mark.parametrize("act_mode,T,tiling", [(0, 200, 1), (0, 200, 2), (0, 200, 3),
                                               (0, 200, 4), (0, 600, 2), (0, 600, 3),
                                               (0, 600, 4)] + W4A16_CASES)
def test_grouped_gemm_fused_and_down_match_oracle(act_mode, T, tiling):
    layer, wr, x, lg, h, (H, I, E, k, T) = _mid_problem(act_mode, T, tiling)
    st = Staged(h, bits16(x), T, k, lg)
    rows = st.rows()
    ic = torch.zeros(st.cap * ((I // 2 + 127) // 128 * 128), dtype=torch.uint8, device="cuda")
    isf = torch.zeros(st.cap * I // 16, dtype=torch.uint8, device="cuda")
    ib = torch.zeros(st.cap * I, dtype=torch.int16, device="cuda")
    moe.moe_grouped_gemm_gateup(h.handle, st.a_codes, st.a_sf, st.gs, st.a_bf16, st.counts,
                                st.offsets, 1, None, ic, isf, ib, T, st.ws)
    cfg = oracle.make_cfg(T, H, I, E, k, act_mode=act_mode, inter_gs=32.0)
    xf = synth.bf16_to_f32(x)
    xc, xsf, gs_a = oracle.quant_nvfp4(xf) if act_mode != 2 else (None, None, 1.0)
    n = len(rows)
    ref_ic = np.zeros((n, I // 2), np.uint8)
    ref_isf = np.zeros((n, I // 16), np.uint8)
    ref_Y = np.zeros((n, H))
    ref_s = np.zeros((n, I))
    for g in range(E + 1):
        idx = np.nonzero(rows[:, 2] == g)[0]
        if len(idx) == 0:
            continue
        e = "shared" if g == E else g
        G, c_, s_, Y = oracle.expert_rows(cfg, layer, e, x, xc, xsf, gs_a,
                                          rows[idx, 1].astype(np.int32))
        ref_ic[idx], ref_isf[idx], ref_Y[idx] = c_, s_, Y
        ref_s[idx] = G[:, :I] / (1 + np.exp(-G[:, :I])) * G[:, I:]
    if act_mode != 2:
        gc, gsf = tiled_to_canonical(host(ic), host(isf), st.cap, I)
        gc, gsf = gc[rows[:, 0]], gsf[rows[:, 0]]
        # fp32 accumulation vs fp64: decisions may differ only next to a boundary
        same = (gsf == ref_isf)
        assert same.mean() > 0.995
        near = quant_decisions_near_boundary(ref_s, 32.0, ref_isf, gsf, ref_ic, gc, rel=5e-5)
        assert near.mean() > 0.999
        # the down GEMM alone, fed the oracle's intermediate (tiled as the library expects)
        full_c = np.zeros((st.cap, I // 2), np.uint8)
        full_s = np.zeros((st.cap, I // 16), np.uint8)
        full_c[rows[:, 0]] = ref_ic
        full_s[rows[:, 0]] = ref_isf
        ct, stl = canonical_to_tiled(full_c, full_s, st.cap, I)
        dic, disf = dev(ct.reshape(-1)), dev(stl)
        dib = None
    else:
        gb = host(ib).reshape(st.cap, I)[rows[:, 0]].view(np.uint16)
        # every row: the bf16 intermediate equals the oracle's rounding of fp64 s, except
        # adjacent values where s sits next to the midpoint between them (fp32 accumulation)
        assert np.mean(gb == bf16_rn_from_f64(ref_s)) > 0.99
        ok = bf16_adjacent_near_midpoint(gb, ref_s, 1e-4)
        assert ok.all(), np.argwhere(~ok)[:5]
        full = np.zeros((st.cap, I), np.uint16)
        full[rows[:, 0]] = bf16_rn_from_f64(ref_s)
        dic = disf = None
        dib = bits16(full.reshape(-1))
    y = torch.zeros((st.cap, H), dtype=torch.float32, device="cuda")
    moe.moe_grouped_gemm_down(h.handle, dic, disf, dib, st.counts, st.offsets, st.perm, st.w,
                              y, T, st.ws)
    yg = host(y)
    perm = host(st.perm)
    wts = host(st.w).reshape(-1)
    for j, (r, tok, g) in enumerate(rows):
        pair = perm[r]
        wt = wts[pair] if pair < T * k else 1.0
        want = ref_Y[j] * wt
        got = yg[r]  # y is indexed by padded row
        assert np.max(np.abs(got - want)) <= 1e-4 * np.sqrt(np.mean(want ** 2)) * np.sqrt(I / 64) + 1e-9, (j, g)


@pytest.mark.parametrize("T,H,k", [(33, 256, 8), (1500, 4096, 8), (1100, 1536, 8),
                                   (1200, 4096, 2)])
def test_combine_sums_pairs_and_shared(T, H, k):
    """out[t] = bf16(fp32 sum of the token's pair rows in top-k order, then its shared row),
    bit for bit, for the load-based combine (small T) and the bulk-copy combine (T >= 1024;
    2048-column pieces in 3 or 6 slots, 512-column pieces)."""
    El = 320
    h, _ = _tiny_layer_handle(E=El, k=k, H=H, max_tokens=max(T, 8192))
    rng = np.random.default_rng(T)
    n_pair_rows = T * k + 17
    shared0 = n_pair_rows + 5
    R = shared0 + T
    y = rng.standard_normal((R, H)).astype(np.float32)
    # pairs point at distinct padded rows (or -1: not local); shared rows start at shared0
    rows = rng.permutation(n_pair_rows)[:T * k].astype(np.int32)
    inv = np.where(rng.random(T * k) < 0.7, rows, -1).astype(np.int32)
    inv[:k] = -1  # a token with no local pair: its shared row alone
    offsets = np.zeros(El + 2, np.int32)
    offsets[El] = shared0
    out = torch.zeros((T, H), dtype=torch.int16, device="cuda")
    moe.moe_combine(h.handle, dev(y), dev(inv), dev(offsets), T, out)
    want = np.zeros((T, H), np.float32)
    for j in range(k):
        r = inv[j::k]
        sel = r >= 0
        want[sel] = want[sel] + y[r[sel]]
    want = want + y[shared0:shared0 + T]
    want_bits = torch.from_numpy(want).to(torch.bfloat16).view(torch.int16).numpy()
    assert np.array_equal(host(out), want_bits)


@pytest.mark.parametrize("tiling", [1, 2, 3, 4])
def test_grouped_gemms_with_the_dynamic_intermediate_scale(tiling):
    """Staged gate_up (both passes) and down with inter_global_scale 0: gs_i is 2688 / amax
    of the fp32 intermediate of the computed rows, and the down output matches the oracle's
    expert MLP quantising the intermediate with that scale (both GEMM forms)."""
    H, I, E, k, T = 512, 256, 8, 2, 200
    layer = build_layer(12, H, I, E)
    wr = synth.router_weight(12, E, H)
    x = synth.activations(12, T, H, outlier_frac=0.01)
    lg = synth.logits_normal(12, T, E)
    h = make_layer(layer, wr, H, I, E, k, act_mode=0, inter_gs=0.0, gemm_tiling=tiling)
    st = Staged(h, bits16(x), T, k, lg)
    rows = st.rows()
    ic = torch.zeros(st.cap * ((I // 2 + 127) // 128 * 128), dtype=torch.uint8, device="cuda")
    isf = torch.zeros(st.cap * I // 16, dtype=torch.uint8, device="cuda")
    moe.moe_grouped_gemm_gateup(h.handle, st.a_codes, st.a_sf, st.gs, st.a_bf16, st.counts,
                                st.offsets, 1, None, ic, isf, None, T, st.ws)
    y = torch.zeros((st.cap, H), dtype=torch.float32, device="cuda")
    moe.moe_grouped_gemm_down(h.handle, ic, isf, None, st.counts, st.offsets, st.perm, st.w,
                              y, T, st.ws)
    torch.cuda.synchronize()
    ptr = moe.moe_forward_buffers(h.handle, st.ws, T)["inter_gs"]
    gs_gpu = float(st.ws[ptr - st.ws.data_ptr():][:4].cpu().numpy().view(np.float32)[0])
    ora = oracle.moe_forward(oracle.make_cfg(T, H, I, E, k, act_mode=0, inter_gs=0.0), x, layer,
                             logits_in=lg, tokens=np.zeros(0, np.int32))
    assert abs(gs_gpu - ora.gs_i) <= 1e-5 * ora.gs_i, (gs_gpu, ora.gs_i)
    cfg = oracle.make_cfg(T, H, I, E, k, act_mode=0, inter_gs=gs_gpu)
    xc, xsf, gs_a = oracle.quant_nvfp4(synth.bf16_to_f32(x))
    wts = host(st.w).reshape(-1)
    Yg = host(y)
    for g in range(E + 1):
        sel = rows[rows[:, 2] == g]
        if len(sel) == 0:
            continue
        e = "shared" if g == E else g
        Y = oracle.expert_rows(cfg, layer, e, x, xc, xsf, gs_a, sel[:, 1].astype(np.int32))[3]
        pair = host(st.perm)[sel[:, 0]]
        w = np.where(pair < T * k, wts[np.minimum(pair, T * k - 1)], 1.0)
        rel, mx = within_layer_tolerance(Yg[sel[:, 0]], Y * w[:, None])
        assert rel <= 1e-2 and mx <= 5e-2, (g, rel, mx)


@pytest.mark.parametrize("act_mode", [0, 2])
def test_gateup_refuses_a_missing_activation_scale(act_mode):
    """gs_a is read on the device in both modes (W4A4: the activation global scale; W4A16:
    the fp16 prescale), so a null gs_a is refused before anything is launched."""
    layer, wr, x, lg, h, (H, I, E, k, T) = _mid_problem(act_mode, 60)
    st = Staged(h, bits16(x), T, k, lg)
    G = torch.zeros((st.cap, 2 * I), dtype=torch.float32, device="cuda")
    with pytest.raises(moe.MoEError) as err:
        moe.moe_grouped_gemm_gateup(h.handle, st.a_codes, st.a_sf, None, st.a_bf16, st.counts,
                                    st.offsets, 0, G, None, None, None, T, st.ws)
    assert err.value.status == moe.MOE_ERR_INVALID
