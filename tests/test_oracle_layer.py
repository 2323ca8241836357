"""Pins of the oracle's routing, grouping, expert MLP and whole-layer forward against
independent formulations: numpy fp64 matmuls over independently dequantised weights,
brute-force sorts, a dense (all-experts) mixture, and the structural facts of the pages
(shard partials add up to the full layer; 320 routed + 1 shared, top-8)."""
import json
import os

import numpy as np
import pytest
from scipy.special import expit

import oracle
import synth
from helpers import build_layer, dequant_independent, slice_layer

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _lexsort_topk(logits, k):
    T, E = logits.shape
    ids = np.empty((T, k), np.int64)
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-logits[t, e], e))
        ids[t] = order[:k]
    return ids


def test_router_logits_match_numpy_matmul():
    T, H, E = 8, 256, 16
    x = synth.activations(1, T, H)
    wr = synth.router_weight(1, E, H)
    bias = synth.zipf_bias(1, E)
    got = oracle.router_logits(x, wr, bias)
    ref = synth.bf16_to_f32(x).astype(np.float64) @ synth.bf16_to_f32(wr).astype(np.float64).T
    ref += bias.astype(np.float64)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_topk_bruteforce_ties_and_weights():
    rng = np.random.default_rng(2)
    T, E, k = 40, 12, 4
    lg = np.round(rng.standard_normal((T, E)) * 2) / 2  # many exact ties
    ids, w = oracle.topk(lg, k)
    ref = _lexsort_topk(lg, k)
    assert np.array_equal(ids, ref)
    for t in range(T):
        sel = lg[t, ref[t]]
        z = np.exp(sel - sel.max())
        np.testing.assert_allclose(w[t], z / z.sum(), rtol=1e-14)
        # equal to softmax over all E renormalised over the selected k
        full = np.exp(lg[t] - lg[t].max())
        full /= full.sum()
        np.testing.assert_allclose(w[t], full[ref[t]] / full[ref[t]].sum(), rtol=1e-12)


def test_topk_special_cases():
    # all logits equal -> the k lowest ids, uniform weights
    ids, w = oracle.topk(np.zeros((1, 10)), 3)
    assert ids.tolist() == [[0, 1, 2]] and np.allclose(w, 1 / 3)
    # k = 1 -> weight exactly 1
    ids, w = oracle.topk(np.random.default_rng(0).standard_normal((5, 7)), 1)
    assert np.all(w == 1.0)
    # one-hot logits route to the hot expert first
    lg = np.full((3, 8), -50.0)
    lg[0, 5] = lg[1, 0] = lg[2, 7] = 10.0
    ids, w = oracle.topk(lg, 2)
    assert ids[:, 0].tolist() == [5, 0, 7] and np.all(w[:, 0] >= 1 - 1e-12)


def test_permute_bruteforce():
    rng = np.random.default_rng(4)
    T, k, E = 50, 3, 10
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    for E_loc, off in [(10, 0), (5, 0), (5, 5), (3, 4), (1, 9)]:
        counts, pairs = oracle.permute(ids, E_loc, off)
        want = sorted([(int(ids.flat[p]) - off, p) for p in range(T * k)
                       if 0 <= ids.flat[p] - off < E_loc])
        assert pairs.tolist() == [p for _, p in want]
        assert counts.tolist() == [sum(1 for le, _ in want if le == e) for e in range(E_loc)]


def _inter_gs_for(G, I):
    s = G[:, :I] * expit(G[:, :I]) * G[:, I:]
    return float(2.0 ** np.floor(np.log2(2688.0 / (2 * np.abs(s).max()))))


def _numpy_expert(a, gs_a, w13d, w2d, inter_gs, I, act_mode):
    """Expert MLP with numpy: a [n, H] fp64 input values (without gs_a), w13d/w2d
    independently dequantised (with their global scales)."""
    G = (a @ w13d.T) / gs_a
    s = G[:, :I] * expit(G[:, :I]) * G[:, I:]
    if act_mode == 2:
        import torch
        sq = torch.from_numpy(s).to(torch.bfloat16).double().numpy()
        return G, sq @ w2d.T
    codes, sf, _ = oracle.quant_nvfp4(s.astype(np.float32), gs=inter_gs)
    aq = dequant_independent(codes, sf, inter_gs)
    return G, aq @ w2d.T


@pytest.mark.parametrize("act_mode", [0, 2])
def test_expert_rows_match_numpy(act_mode):
    H, I, E, T = 128, 64, 3, 6
    layer = build_layer(21, H, I, E)
    x = synth.activations(21, T, H)
    xf = synth.bf16_to_f32(x).astype(np.float64)
    if act_mode == 0:
        xc, xsf, gs_a = oracle.quant_nvfp4(synth.bf16_to_f32(x))
        a = dequant_independent(xc, xsf, 1.0)
    else:
        xc = xsf = None
        gs_a = 1.0
        a = xf
    w13d = dequant_independent(layer.w13[1], layer.w13_sf[1], layer.w13_gs[1])
    w2d = dequant_independent(layer.w2[1], layer.w2_sf[1], layer.w2_gs[1])
    G0 = (a @ w13d.T) / gs_a
    inter_gs = _inter_gs_for(G0, I)
    cfg = oracle.make_cfg(T, H, I, E, 2, act_mode=act_mode, inter_gs=inter_gs)
    tok = np.array([0, 3, 5, 5], np.int32)
    G, ic, isf, Y = oracle.expert_rows(cfg, layer, 1, x, xc, xsf, gs_a, tok)
    Gr, Yr = _numpy_expert(a[tok], gs_a, w13d, w2d, inter_gs, I, act_mode)
    np.testing.assert_allclose(G, Gr, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(Y, Yr, rtol=1e-10, atol=1e-12)


def _dense_mixture(cfg, x, wr, layer, inter_gs, bias=None, logits_in=None):
    """out[t] = sum over ALL local experts of gate[t, e] * MLP_e(x_t) + shared, where gate is
    the renormalised top-k softmax (0 for unselected) -- no grouping, no permutation."""
    T, H, I, E, k = cfg.T, cfg.H, cfg.I, cfg.E, cfg.k
    xf = synth.bf16_to_f32(x).astype(np.float64)
    if logits_in is None:
        lg = xf @ synth.bf16_to_f32(wr).astype(np.float64).T
    else:
        lg = logits_in.astype(np.float64)
    if bias is not None:
        lg = lg + bias.astype(np.float64)
    ids = _lexsort_topk(lg, k)
    gate = np.zeros((T, E))
    for t in range(T):
        z = np.exp(lg[t, ids[t]] - lg[t, ids[t]].max())
        gate[t, ids[t]] = z / z.sum()
    if cfg.act_mode == 2:
        a, gs_a = xf, 1.0
    else:
        xc, xsf, gs_a = oracle.quant_nvfp4(synth.bf16_to_f32(x))
        a = dequant_independent(xc, xsf, 1.0)
    out = np.zeros((T, H))
    for le in range(cfg.E_loc):
        w13d = dequant_independent(layer.w13[le], layer.w13_sf[le], layer.w13_gs[le])
        w2d = dequant_independent(layer.w2[le], layer.w2_sf[le], layer.w2_gs[le])
        _, Y = _numpy_expert(a, gs_a, w13d, w2d, inter_gs, I, cfg.act_mode)
        out += gate[:, cfg.off + le, None] * Y
    if cfg.has_shared and cfg.add_shared:
        w13d = dequant_independent(layer.sh13, layer.sh13_sf, layer.sh13_gs)
        w2d = dequant_independent(layer.sh2, layer.sh2_sf, layer.sh2_gs)
        out += _numpy_expert(a, gs_a, w13d, w2d, inter_gs, I, cfg.act_mode)[1]
    return out, ids


@pytest.mark.parametrize("act_mode,k,E", [(0, 2, 4), (0, 1, 4), (2, 2, 4), (0, 4, 4)])
def test_layer_matches_dense_mixture_bruteforce(act_mode, k, E):
    T, H, I = 4, 64, 32
    layer = build_layer(31, H, I, E)
    x = synth.activations(31, T, H)
    wr = synth.router_weight(31, E, H, std=0.3)
    cfg = oracle.make_cfg(T, H, I, E, k, act_mode=act_mode, inter_gs=64.0)
    r = oracle.moe_forward(cfg, x, layer, router_w=wr)
    ref, ids = _dense_mixture(cfg, x, wr, layer, 64.0)
    assert np.array_equal(r.ids, ids)
    np.testing.assert_allclose(r.out, ref, rtol=1e-9, atol=1e-12)


def test_shards_add_up_to_full_layer():
    """Contiguous shards [0, E/2) and [E/2, E), the shared expert added by one of them,
    sum to the full layer; the union of their local pairs is the full pair set."""
    c = synth.CONFIGS["tiny"]
    T, H, I, E, k = c["T"], c["H"], c["I"], c["E"], c["k"]
    layer = build_layer(0, H, I, E)
    x = synth.activations(0, T, H)
    wr = synth.router_weight(0, E, H)
    bias = synth.zipf_bias(0, E)
    full = oracle.moe_forward(oracle.make_cfg(T, H, I, E, k, inter_gs=32.0), x, layer,
                              router_w=wr, logit_bias=bias)
    h = E // 2
    s0 = oracle.moe_forward(oracle.make_cfg(T, H, I, E, k, E_loc=h, off=0, add_shared=1,
                                            inter_gs=32.0), x, slice_layer(layer, 0, h),
                            router_w=wr, logit_bias=bias)
    s1 = oracle.moe_forward(oracle.make_cfg(T, H, I, E, k, E_loc=E - h, off=h, add_shared=0,
                                            inter_gs=32.0), x, slice_layer(layer, h, E),
                            router_w=wr, logit_bias=bias)
    np.testing.assert_allclose(s0.out + s1.out, full.out, rtol=1e-12, atol=1e-12)
    assert sorted(s0.pairs.tolist() + s1.pairs.tolist()) == sorted(full.pairs.tolist())
    assert len(full.pairs) == T * k
    # the identity shard (offset 0, all experts local) is the full layer
    ident = oracle.moe_forward(oracle.make_cfg(T, H, I, E, k, E_loc=E, off=0, inter_gs=32.0),
                               x, layer, router_w=wr, logit_bias=bias)
    assert np.array_equal(ident.out, full.out)


def test_token_subset_matches_full_run():
    c = synth.CONFIGS["tiny"]
    T, H, I, E, k = c["T"], c["H"], c["I"], c["E"], c["k"]
    layer = build_layer(0, H, I, E)
    x = synth.activations(0, T, H)
    wr = synth.router_weight(0, E, H)
    cfg = oracle.make_cfg(T, H, I, E, k, inter_gs=32.0)
    full = oracle.moe_forward(cfg, x, layer, router_w=wr)
    sub = oracle.moe_forward(cfg, x, layer, router_w=wr, tokens=np.array([3, 0, 11], np.int32))
    assert np.array_equal(sub.out, full.out[[3, 0, 11]])
    assert np.array_equal(sub.out_bf16, full.out_bf16[[3, 0, 11]])


def test_k_equals_E_is_the_dense_softmax_mixture():
    T, H, I, E = 3, 64, 32, 4
    layer = build_layer(41, H, I, E, shared=False)
    x = synth.activations(41, T, H)
    lg = synth.logits_normal(41, T, E)
    cfg = oracle.make_cfg(T, H, I, E, E, has_shared=0, add_shared=0, inter_gs=64.0)
    r = oracle.moe_forward(cfg, x, layer, logits_in=lg)
    p = np.exp(lg.astype(np.float64) - lg.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    for t in range(T):
        np.testing.assert_allclose(np.sort(r.w[t]), np.sort(p[t]), rtol=1e-12)


def test_layer_facts_of_the_pages():
    facts = json.load(open(os.path.join(GOLD, "layer_facts.json")))
    for name in ("decode", "prefill", "shard", "w4a16"):
        c = synth.CONFIGS[name]
        assert c["E"] == facts["routed_experts"] and c["k"] == facts["top_k"]
    lo, hi = facts["shards"][1]
    assert synth.CONFIGS["shard"]["off"] == lo and synth.CONFIGS["shard"]["E_loc"] == hi - lo + 1


def _numpy_dynamic_inter_scale(cfg, x, wr, layer):
    """2688 / amax|fp32(s)| over every row a shard computes (its local pairs of all tokens,
    plus the shared rows when it adds the shared expert), from numpy matmuls over
    independently dequantised weights; 1 when there is no such row (or amax is 0)."""
    T, I, k = cfg.T, cfg.I, cfg.k
    lg = synth.bf16_to_f32(x).astype(np.float64) @ synth.bf16_to_f32(wr).astype(np.float64).T
    ids = _lexsort_topk(lg, k)
    xc, xsf, gs_a = oracle.quant_nvfp4(synth.bf16_to_f32(x))
    a = dequant_independent(xc, xsf, 1.0)
    amax = np.float32(0.0)
    for le in range(cfg.E_loc):
        rows = [t for t in range(T) for j in range(k) if ids[t, j] - cfg.off == le]
        if not rows:
            continue
        w13d = dequant_independent(layer.w13[le], layer.w13_sf[le], layer.w13_gs[le])
        G = (a[rows] @ w13d.T) / gs_a
        s = (G[:, :I] * expit(G[:, :I]) * G[:, I:]).astype(np.float32)
        amax = max(amax, np.abs(s).max())
    if cfg.has_shared and cfg.add_shared:
        w13d = dequant_independent(layer.sh13, layer.sh13_sf, layer.sh13_gs)
        G = (a @ w13d.T) / gs_a
        s = (G[:, :I] * expit(G[:, :I]) * G[:, I:]).astype(np.float32)
        amax = max(amax, np.abs(s).max())
    return np.float32(1.0) if amax == 0 else np.float32(2688.0) / np.float32(amax)


@pytest.mark.parametrize("E_loc,off,add_shared", [(6, 0, 1), (3, 3, 0), (3, 0, 1)])
def test_dynamic_intermediate_scale_is_the_amax_of_the_shards_rows(E_loc, off, add_shared):
    """inter_gs <= 0 (dynamic): the scale is 2688 / amax of the fp32 intermediate over the
    shard's own rows, and the forward equals the static forward at that scale."""
    H, I, E, k, T = 128, 64, 6, 2, 10
    full = build_layer(31, H, I, E)
    layer = slice_layer(full, off, off + E_loc)
    wr = synth.router_weight(31, E, H)
    x = synth.activations(31, T, H)
    cfg = oracle.make_cfg(T, H, I, E, k, E_loc=E_loc, off=off, add_shared=add_shared,
                          inter_gs=0.0)
    dyn = oracle.moe_forward(cfg, x, layer, router_w=wr)
    want = _numpy_dynamic_inter_scale(cfg, x, wr, layer)
    assert abs(dyn.gs_i - float(want)) <= 1e-6 * float(want)
    cfg_s = oracle.make_cfg(T, H, I, E, k, E_loc=E_loc, off=off, add_shared=add_shared,
                            inter_gs=dyn.gs_i)
    sta = oracle.moe_forward(cfg_s, x, layer, router_w=wr)
    assert sta.gs_i == dyn.gs_i
    assert np.array_equal(sta.out, dyn.out)


def test_dynamic_intermediate_scale_matches_dense_mixture():
    """Whole layer with the dynamic intermediate scale against the dense all-experts
    mixture (numpy) quantising the intermediate with the numpy-derived scale."""
    H, I, E, k, T = 128, 64, 4, 2, 8
    layer = build_layer(32, H, I, E)
    wr = synth.router_weight(32, E, H)
    x = synth.activations(32, T, H)
    cfg = oracle.make_cfg(T, H, I, E, k, inter_gs=0.0)
    got = oracle.moe_forward(cfg, x, layer, router_w=wr)
    gs_i = float(_numpy_dynamic_inter_scale(cfg, x, wr, layer))
    ref, ids = _dense_mixture(cfg, x, wr, layer, gs_i)
    assert np.array_equal(np.sort(got.ids, 1), np.sort(ids, 1))
    np.testing.assert_allclose(got.out, ref, rtol=1e-9, atol=1e-9 * np.abs(ref).max())
