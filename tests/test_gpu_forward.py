"""Whole-layer GPU parity against the oracle on every workload: the tiny layer, the
320-expert decode layer, the prefill chunk (sampled tokens), the expert shard 160-319
with Zipf popularity (and shard 0-159 + shard 160-319 == full layer), and the W4A16
decode sweep.  Bar: relative L2 <= 1e-2 and max |err| <= 5e-2 * rms(ref) against the
oracle's fp64 accumulation; routing ids, grouping and activation codes bit-exact."""
import json
import os

import numpy as np
import pytest
import torch

import nvfp4_mixture_experts_gb300 as moe
import oracle
import synth
from gpu_util import bits16, dev, host, make_layer, tiled_to_canonical
from helpers import build_layer, slice_layer, within_layer_tolerance

pytestmark = pytest.mark.gpu

GOLD = os.path.join(os.path.dirname(__file__), "golden")
INTER = json.load(open(os.path.join(GOLD, "inter_scale.json")))


@pytest.fixture(scope="module")
def big_layer():
    c = synth.CONFIGS["decode"]
    return build_layer(0, c["H"], c["I"], c["E"])


def _routing_clear(x, wr, bias, k, logits_in=None, order=False):
    """Tokens whose selected set (order=False: the k-th / (k+1)-th logit gap) or whose whole
    ranking of the first k+1 logits (order=True) is far above the fp32 logit error, so the
    top-k is unique."""
    if logits_in is not None:
        lg = logits_in.astype(np.float64) + (0 if bias is None else bias)
        return np.ones(lg.shape[0], bool), lg
    lg = oracle.router_logits(x, wr, bias)
    mag = np.abs(synth.bf16_to_f32(x).astype(np.float64)) @ np.abs(
        synth.bf16_to_f32(wr).astype(np.float64)).T
    srt = -np.sort(-lg, axis=1)
    thr = 2e-5 * mag.max(1)
    if order:
        return (np.diff(-srt[:, :k + 1], axis=1) > thr[:, None]).all(1), lg
    return srt[:, k - 1] - srt[:, k] > thr, lg


def _same_routing(ids, ref_ids, x, wr, bias, k):
    """Selected sets equal wherever they are unique, and the order wherever it is."""
    set_ok, _ = _routing_clear(x, wr, bias, k)
    ord_ok, _ = _routing_clear(x, wr, bias, k, order=True)
    assert np.array_equal(np.sort(ids[set_ok], 1), np.sort(ref_ids[set_ok], 1))
    assert np.array_equal(ids[ord_ok], ref_ids[ord_ok])
    assert set_ok.mean() > 0.95


def _forward(h, x, T, logits_in=None, bias=None):
    out = torch.zeros((T, h.cfg.hidden), dtype=torch.int16, device="cuda")
    h.forward(bits16(x), out=out, logits_in=None if logits_in is None else dev(logits_in),
              logit_bias=None if bias is None else dev(bias))
    torch.cuda.synchronize()
    st, bits = moe.moe_get_status(h.handle, h.ws)
    assert st == moe.MOE_OK, bits
    return synth.bf16_to_f32(host(out).view(np.uint16)).astype(np.float64)


def _check(got, ref, what):
    rel, mx = within_layer_tolerance(got, ref)
    assert rel <= 1e-2 and mx <= 5e-2, (what, rel, mx)
    return rel, mx


def _read_ws(layer, ptr, n, dtype):
    """n elements of dtype at device address ptr inside layer.ws (a forward intermediate)."""
    off = ptr - layer.ws.data_ptr()
    nbytes = n * np.dtype(dtype).itemsize
    assert 0 <= off and off + nbytes <= layer.ws.numel()
    return layer.ws[off:off + nbytes].cpu().numpy().view(dtype)


def _forward_buffers_check(h, T, ora, clear, x, wr, bias=None):
    """ids, grouping and activation codes of the forward equal the oracle's."""
    k = h.cfg.top_k
    b = moe.moe_forward_buffers(h.handle, h.ws, T)
    ids = _read_ws(h, b["topk_ids"], T * k, np.int32).reshape(T, k)
    _same_routing(ids, ora.ids, x, wr, bias, k)
    clear = clear & _routing_clear(x, wr, bias, k, order=True)[0]
    El = h.cfg.num_local_experts
    counts = _read_ws(h, b["expert_counts"], El + 1, np.int32)
    offsets = _read_ws(h, b["expert_offsets"], El + 2, np.int32)
    perm = _read_ws(h, b["perm_src"], int(offsets[-1]), np.int32)
    if clear.all():
        assert np.array_equal(counts[:El], ora.counts)
        got = np.concatenate([perm[offsets[e]:offsets[e] + counts[e]] for e in range(El)])
        assert np.array_equal(got, ora.pairs)
    if h.cfg.act_mode != moe.MOE_W4A16:
        H = h.cfg.hidden
        gs = _read_ws(h, b["gs_a"], 1, np.float32)[0]
        assert gs == np.float32(ora.gs_a)
        rows = int(offsets[-1])
        pitch = (H // 2 + 127) // 128 * 128
        ac = _read_ws(h, b["a_codes"], rows * pitch, np.uint8)
        asf = _read_ws(h, b["a_sf"], rows * H // 16, np.uint8)
        c, s = tiled_to_canonical(ac, asf, rows, H)
        # the forward's padding rows are not marked: valid rows from counts and offsets
        valid = np.concatenate([np.arange(offsets[g], offsets[g] + counts[g])
                                for g in range(El + 1)]).astype(np.int64)
        tok = np.where(perm[valid] < T * k, perm[valid] // k, perm[valid] - T * k)
        assert np.array_equal(c[valid], ora.x_codes[tok])
        assert np.array_equal(s[valid], ora.x_sf[tok])


@pytest.mark.parametrize("tiling", [0, 2, 3, 4])
def test_tiny_layer_full_parity(tiling):
    c = synth.CONFIGS["tiny"]
    T, H, I, E, k = c["T"], c["H"], c["I"], c["E"], c["k"]
    gs_i = INTER["tiny"]["inter_global_scale"]
    layer = build_layer(0, H, I, E)
    wr = synth.router_weight(0, E, H)
    x = synth.activations(0, T, H)
    h = make_layer(layer, wr, H, I, E, k, inter_gs=gs_i, max_tokens=T, gemm_tiling=tiling)
    got = _forward(h, x, T)
    ora = oracle.moe_forward(oracle.make_cfg(T, H, I, E, k, inter_gs=gs_i), x, layer, router_w=wr)
    clear, _ = _routing_clear(x, wr, None, k)
    assert clear.all()
    _check(got, ora.out, "tiny")
    _forward_buffers_check(h, T, ora, clear, x, wr)


def test_empty_batch_is_a_no_op():
    c = synth.CONFIGS["tiny"]
    H, I, E, k = c["H"], c["I"], c["E"], c["k"]
    layer = build_layer(0, H, I, E)
    h = make_layer(layer, synth.router_weight(0, E, H), H, I, E, k, inter_gs=64.0, max_tokens=4)
    out = torch.zeros((1, H), dtype=torch.int16, device="cuda")
    ws = torch.empty(1024, dtype=torch.uint8, device="cuda")
    moe.moe_forward(h.handle, out, None, None, 0, out, ws)
    torch.cuda.synchronize()


@pytest.mark.parametrize("tiling", [0, 2, 3, 4])
def test_decode_layer_full_parity(big_layer, tiling):
    c = synth.CONFIGS["decode"]
    T, H, I, E, k = c["T"], c["H"], c["I"], c["E"], c["k"]
    gs_i = INTER["decode"]["inter_global_scale"]
    wr = synth.router_weight(0, E, H)
    x = synth.activations(0, T, H)
    h = make_layer(big_layer, wr, H, I, E, k, inter_gs=gs_i, max_tokens=T, gemm_tiling=tiling)
    got = _forward(h, x, T)
    clear, _ = _routing_clear(x, wr, None, k)
    ora = oracle.moe_forward(oracle.make_cfg(T, H, I, E, k, inter_gs=gs_i), x, big_layer,
                             router_w=wr)
    _check(got[clear], ora.out[clear], "decode")
    _forward_buffers_check(h, T, ora, clear, x, wr)


def test_shard_partials_and_union(big_layer):
    c = synth.CONFIGS["shard"]
    T, H, I, E, k = c["T"], c["H"], c["I"], c["E"], c["k"]
    gs_i = INTER["shard"]["inter_global_scale"]
    wr = synth.router_weight(0, E, H)
    x = synth.activations(0, T, H)
    bias = synth.zipf_bias(0, E)
    full = make_layer(big_layer, wr, H, I, E, k, inter_gs=gs_i, max_tokens=T)
    s0 = make_layer(slice_layer(big_layer, 0, 160), wr, H, I, E, k, E_loc=160, off=0,
                    add_shared=1, inter_gs=gs_i, max_tokens=T)
    s1 = make_layer(slice_layer(big_layer, 160, 320), wr, H, I, E, k, E_loc=160, off=160,
                    add_shared=0, inter_gs=gs_i, max_tokens=T)
    of = _forward(full, x, T, bias=bias)
    o0 = _forward(s0, x, T, bias=bias)
    o1 = _forward(s1, x, T, bias=bias)
    # the two partial sums add up to the full layer (each partial rounded to bf16)
    _check(o0 + o1, of, "shard 0-159 + shard 160-319 vs full")
    # the local pair sets are disjoint and cover every pair
    inv0 = _read_ws(s0, moe.moe_forward_buffers(s0.handle, s0.ws, T)["inv"], T * k, np.int32)
    inv1 = _read_ws(s1, moe.moe_forward_buffers(s1.handle, s1.ws, T)["inv"], T * k, np.int32)
    assert np.all((inv0 >= 0) ^ (inv1 >= 0))
    # shard 160..319 against the oracle's shard on sampled tokens
    clear, _ = _routing_clear(x, wr, bias, k)
    tok = np.sort(np.random.default_rng(0).choice(T, 48, replace=False)).astype(np.int32)
    tok = tok[clear[tok]]
    ora = oracle.moe_forward(oracle.make_cfg(T, H, I, E, k, E_loc=160, off=160, add_shared=0,
                                             inter_gs=gs_i),
                             x, slice_layer(big_layer, 160, 320), router_w=wr, logit_bias=bias,
                             tokens=tok)
    _check(o1[tok], ora.out, "shard 160-319")
    counts = np.bincount(ora.ids.ravel(), minlength=E)
    assert counts.max() > 4 * counts.mean()  # Zipf popularity: a few hot experts


@pytest.mark.parametrize("T", synth.CONFIGS["w4a16"]["sweep"])
def test_w4a16_decode_sweep(big_layer, T):
    c = synth.CONFIGS["w4a16"]
    H, I, E, k = c["H"], c["I"], c["E"], c["k"]
    wr = synth.router_weight(0, E, H)
    x = synth.activations(0, T, H)
    lg = synth.logits_normal(0, T, E)
    h = make_layer(big_layer, wr, H, I, E, k, act_mode=moe.MOE_W4A16, max_tokens=T)
    got = _forward(h, x, T, logits_in=lg)
    tok = np.arange(T, dtype=np.int32) if T <= 32 else np.sort(
        np.random.default_rng(T).choice(T, 32, replace=False)).astype(np.int32)
    ora = oracle.moe_forward(oracle.make_cfg(T, H, I, E, k, act_mode=2), x, big_layer,
                             logits_in=lg, tokens=tok)
    _check(got[tok], ora.out, "w4a16 T=%d" % T)


@pytest.mark.parametrize("act_mode", [0, moe.MOE_W4A16])
def test_chained_forwards_read_complete_inputs(act_mode):
    """Two forwards chained on one stream, the first one's output the second one's input,
    with given logits and no synchronisation between them.  The second forward's first
    kernel reads its input before its dependency wait, so it may start only when the first
    forward (whose last kernel lets its dependents start early) is complete: the second
    output equals the same forward run after a synchronisation, bit for bit."""
    c = synth.CONFIGS["tiny"]
    T, H, I, E, k = c["T"], c["H"], c["I"], c["E"], c["k"]
    layer = build_layer(0, H, I, E)
    wr = synth.router_weight(0, E, H)
    h = make_layer(layer, wr, H, I, E, k, act_mode=act_mode, inter_gs=1024.0, max_tokens=T)
    x = bits16(synth.activations(4, T, H))
    lg = dev(synth.logits_normal(4, T, E))
    for _ in range(3):
        out1 = h.forward(x, logits_in=lg)
        out2 = h.forward(out1, logits_in=lg)
        torch.cuda.synchronize()
        st, bits = moe.moe_get_status(h.handle, h.ws)
        assert st == moe.MOE_OK, bits
        ref = h.forward(out1.clone(), logits_in=lg)
        torch.cuda.synchronize()
        assert torch.equal(out2, ref)


@pytest.mark.parametrize("T", [1, 3])
def test_w4a16_small_batch_forward_is_deterministic(big_layer, T):
    """Small W4A16 batches run gate_up and down in one GEMV launch that cuts each gate_up
    tile's contraction into parts when there are few tiles (one token: 180 tiles on the
    SMs); the part that arrives last adds all parts' sums in k order, so the result does not
    depend on which part came last: repeated forwards give the same bits (and the oracle's
    result within the bar)."""
    c = synth.CONFIGS["w4a16"]
    H, I, E, k = c["H"], c["I"], c["E"], c["k"]
    wr = synth.router_weight(0, E, H)
    x = synth.activations(5, T, H)
    lg = synth.logits_normal(5, T, E)
    h = make_layer(big_layer, wr, H, I, E, k, act_mode=moe.MOE_W4A16, max_tokens=T)
    first = _forward(h, x, T, logits_in=lg)
    for _ in range(4):
        assert np.array_equal(_forward(h, x, T, logits_in=lg), first)
    ora = oracle.moe_forward(oracle.make_cfg(T, H, I, E, k, act_mode=2), x, big_layer,
                             logits_in=lg)
    _check(first, ora.out, "w4a16 T=%d repeated" % T)


# W4A16 at up to 256 tokens (and at most 16 expected rows per expert: T*k/E <= 16) runs on
# the grouped GEMV, otherwise on the tensor-core kernel; here E=24 (or 8 local), k=4.
# H = 384 and I = 320 leave the last 256-element k-block of each GEMM partly empty; the
# shard (experts 8..15 of 24, no shared rows added) leaves most groups empty; has_shared=0
# drops the shared slot; T = 96 gives the shared slot 12 chunks of 8 rows on the GEMV;
# T = 40 on the shard and T >= 128 run on the tensor-core kernel.
@pytest.mark.parametrize("T,E_loc,off,add_shared,has_shared", [
    (1, None, 0, 1, 1), (7, None, 0, 1, 1), (64, None, 0, 1, 1), (65, None, 0, 1, 1),
    (96, None, 0, 1, 1), (5, 8, 8, 0, 1), (40, 8, 8, 1, 1), (9, None, 0, 1, 0),
    (256, None, 0, 1, 1), (257, None, 0, 1, 1), (300, 8, 8, 1, 1)])
def test_w4a16_forward_ragged_k(T, E_loc, off, add_shared, has_shared):
    H, I, E, k = 384, 320, 24, 4
    layer = build_layer(21, H, I, E)
    wr = synth.router_weight(21, E, H)
    x = synth.activations(21, T, H, outlier_frac=0.01)
    lg = synth.logits_normal(21 + T, T, E)
    sub = layer if E_loc is None else slice_layer(layer, off, off + E_loc)
    h = make_layer(sub, wr, H, I, E, k, E_loc=E_loc, off=off, add_shared=add_shared,
                   act_mode=moe.MOE_W4A16, max_tokens=T, has_shared=has_shared)
    got = _forward(h, x, T, logits_in=lg)
    ora = oracle.moe_forward(oracle.make_cfg(T, H, I, E, k, E_loc=E_loc, off=off,
                                             has_shared=has_shared, add_shared=add_shared,
                                             act_mode=2),
                             x, sub, logits_in=lg)
    if not np.any(ora.out):
        assert not np.any(got)
        return
    _check(got, ora.out, "w4a16 T=%d E_loc=%s" % (T, E_loc))


def test_w4a16_tiny_layer_short_k():
    """The tiny layer in W4A16 mode: down's K = I = 128 is half of one 256-element k-block,
    gate_up's K = H = 256 exactly one."""
    c = synth.CONFIGS["tiny"]
    T, H, I, E, k = c["T"], c["H"], c["I"], c["E"], c["k"]
    layer = build_layer(0, H, I, E)
    wr = synth.router_weight(0, E, H)
    x = synth.activations(0, T, H)
    lg = synth.logits_normal(3, T, E)
    h = make_layer(layer, wr, H, I, E, k, act_mode=moe.MOE_W4A16, max_tokens=T)
    got = _forward(h, x, T, logits_in=lg)
    ora = oracle.moe_forward(oracle.make_cfg(T, H, I, E, k, act_mode=2), x, layer,
                             logits_in=lg)
    _check(got, ora.out, "w4a16 tiny")


@pytest.mark.parametrize("T,tiling", [(64, 0), (1100, 0), (1100, 2), (1100, 3), (1100, 4)])
def test_forward_combine_of_fp16_y_is_exact(big_layer, T, tiling):
    """The W4A4 forward's combine (the load-based kernel below 1024 tokens, the bulk-copy one
    from 1024) against a numpy replay from the forward's own fp16 y rows and row scales:
    out[t] = bf16(sum over the token's rows, pairs in top-k order then the shared row, of
    fp32(y16[row]) * y_scale[row], added in fp32 in that order), bit for bit; the scales
    are powers of two."""
    c = synth.CONFIGS["decode"]
    H, I, E, k = c["H"], c["I"], c["E"], c["k"]
    gs_i = INTER["decode"]["inter_global_scale"]
    wr = synth.router_weight(0, E, H)
    x = synth.activations(5, T, H)
    h = make_layer(big_layer, wr, H, I, E, k, inter_gs=gs_i, max_tokens=T, gemm_tiling=tiling)
    out = torch.zeros((T, H), dtype=torch.int16, device="cuda")
    h.forward(bits16(x), out=out)
    torch.cuda.synchronize()
    assert moe.moe_get_status(h.handle, h.ws)[0] == moe.MOE_OK
    b = moe.moe_forward_buffers(h.handle, h.ws, T)
    offs = _read_ws(h, b["expert_offsets"], E + 2, np.int32)
    rows_total = int(offs[-1])
    inv = _read_ws(h, b["inv"], T * k, np.int32).reshape(T, k)
    y16 = _read_ws(h, b["y"], rows_total * H, np.float16).reshape(rows_total, H)
    ysc = _read_ws(h, b["y_scale"], rows_total, np.float32)
    rows = np.concatenate([inv, (offs[E] + np.arange(T, dtype=np.int32))[:, None]], 1)
    used = ysc[rows.ravel()]
    assert np.all(used > 0) and np.all(np.frexp(used)[0] == 0.5)  # powers of two
    acc = np.zeros((T, H), np.float32)
    for j in range(k + 1):
        r = rows[:, j]
        acc = acc + y16[r].astype(np.float32) * ysc[r][:, None]
    want = torch.from_numpy(acc).to(torch.bfloat16).view(torch.int16).numpy()
    assert np.array_equal(host(out), want)


@pytest.mark.parametrize("tiling", [0, 2, 3, 4])
def test_prefill_chunk_sampled_parity(big_layer, tiling):
    """The prefill chunk (the default, token tiles, row blocks on CTA pairs, 256-column
    tiles), on sampled tokens."""
    c = synth.CONFIGS["prefill"]
    T, H, I, E, k = c["T"], c["H"], c["I"], c["E"], c["k"]
    gs_i = INTER["prefill"]["inter_global_scale"]
    wr = synth.router_weight(0, E, H)
    x = synth.activations(0, T, H, outlier_frac=c["outlier_frac"])
    h = make_layer(big_layer, wr, H, I, E, k, inter_gs=gs_i, max_tokens=T, gemm_tiling=tiling)
    got = _forward(h, x, T)
    clear, _ = _routing_clear(x, wr, None, k)
    tok = np.sort(np.random.default_rng(1).choice(T, 96, replace=False)).astype(np.int32)
    tok = tok[clear[tok]]
    ora = oracle.moe_forward(oracle.make_cfg(T, H, I, E, k, inter_gs=gs_i), x, big_layer,
                             router_w=wr, tokens=tok)
    _check(got[tok], ora.out, "prefill")
    # routing over every token, bit-exact where the fp64 gap is clear
    ids = _read_ws(h, moe.moe_forward_buffers(h.handle, h.ws, T)["topk_ids"], T * k,
                   np.int32).reshape(T, k)
    _same_routing(ids, ora.ids, x, wr, None, k)
    counts = np.bincount(ora.ids.ravel(), minlength=E)
    assert 150 < counts.mean() < 260  # ~205 tokens per expert


def _dyn_scale_check(h, T, ora):
    gs = _read_ws(h, moe.moe_forward_buffers(h.handle, h.ws, T)["inter_gs"], 1, np.float32)[0]
    # fp32 tensor-core gate/up vs the oracle's fp64: the amax element agrees to ~1e-6
    assert abs(float(gs) - ora.gs_i) <= 1e-5 * ora.gs_i, (gs, ora.gs_i)


@pytest.mark.parametrize("tiling", [0, 2, 3, 4])
def test_tiny_layer_dynamic_intermediate_scale(tiling):
    c = synth.CONFIGS["tiny"]
    T, H, I, E, k = c["T"], c["H"], c["I"], c["E"], c["k"]
    layer = build_layer(0, H, I, E)
    wr = synth.router_weight(0, E, H)
    x = synth.activations(0, T, H)
    h = make_layer(layer, wr, H, I, E, k, inter_gs=0.0, max_tokens=T, gemm_tiling=tiling)
    got = _forward(h, x, T)
    ora = oracle.moe_forward(oracle.make_cfg(T, H, I, E, k, inter_gs=0.0), x, layer, router_w=wr)
    _dyn_scale_check(h, T, ora)
    _check(got, ora.out, "tiny dynamic intermediate scale")
    # twice in a row: the forward clears its amax accumulators itself
    got2 = _forward(h, x, T)
    assert np.array_equal(got, got2)


def test_decode_layer_dynamic_intermediate_scale(big_layer):
    c = synth.CONFIGS["decode"]
    T, H, I, E, k = c["T"], c["H"], c["I"], c["E"], c["k"]
    wr = synth.router_weight(0, E, H)
    x = synth.activations(0, T, H)
    h = make_layer(big_layer, wr, H, I, E, k, inter_gs=0.0, max_tokens=T)
    got = _forward(h, x, T)
    clear, _ = _routing_clear(x, wr, None, k)
    ora = oracle.moe_forward(oracle.make_cfg(T, H, I, E, k, inter_gs=0.0), x, big_layer,
                             router_w=wr)
    _dyn_scale_check(h, T, ora)
    _check(got[clear], ora.out[clear], "decode dynamic intermediate scale")


def test_decode_layer_static_activation_scale(big_layer):
    """W4A4 with the calibrated static activation scale: activation codes bit-exact with
    the oracle's (same scale), the layer within the bar."""
    c = synth.CONFIGS["decode_static"]
    T, H, I, E, k = c["T"], c["H"], c["I"], c["E"], c["k"]
    gs_i = INTER["decode_static"]["inter_global_scale"]
    gs_a = INTER["decode_static"]["act_global_scale"]
    wr = synth.router_weight(0, E, H)
    x = synth.activations(0, T, H)
    h = make_layer(big_layer, wr, H, I, E, k, act_mode=moe.MOE_W4A4_STATIC, act_gs=gs_a,
                   inter_gs=gs_i, max_tokens=T)
    got = _forward(h, x, T)
    clear, _ = _routing_clear(x, wr, None, k)
    ora = oracle.moe_forward(oracle.make_cfg(T, H, I, E, k, act_mode=1, act_gs=gs_a,
                                             inter_gs=gs_i), x, big_layer, router_w=wr)
    assert ora.gs_a == np.float32(gs_a)
    _check(got[clear], ora.out[clear], "decode static activation scale")
    _forward_buffers_check(h, T, ora, clear, x, wr)


@pytest.mark.parametrize("tiling", [1, 2, 3, 4])
def test_fp16_y_envelope_heavy_tails_and_small_tokens(big_layer, tiling):
    """The W4A4 forward keeps the expert outputs y as fp16 rows of y x 2^e_g, 2^e_g from the
    bound K x 2688^2 / (gs_i gs_w) on |y|.  Heavy tails (1 % of the input channels x200) and
    tokens whose input is 2^-2, 2^-4 and 2^-6 of the others' (their y rows down to ~2^-26 of
    the bound: s is about quadratic in the input's scale) stay within the whole-layer bar,
    each small token also against its own rms."""
    c = synth.CONFIGS["decode"]
    T, H, I, E, k = 64, c["H"], c["I"], c["E"], c["k"]
    gs_i = INTER["decode"]["inter_global_scale"]
    wr = synth.router_weight(0, E, H)
    xf = synth.bf16_to_f32(synth.activations(13, T, H, outlier_frac=0.01,
                                              outlier_scale=200.0)).astype(np.float32)
    small = {5: 2.0 ** -2, 6: 2.0 ** -4, 7: 2.0 ** -6}
    for t, f in small.items():
        xf[t] *= np.float32(f)
    x = synth.bf16_bits(xf)
    h = make_layer(big_layer, wr, H, I, E, k, inter_gs=gs_i, max_tokens=T, gemm_tiling=tiling)
    got = _forward(h, x, T)
    clear, _ = _routing_clear(x, wr, None, k)
    ora = oracle.moe_forward(oracle.make_cfg(T, H, I, E, k, inter_gs=gs_i), x, big_layer,
                             router_w=wr)
    _check(got[clear], ora.out[clear], "heavy-tailed input")
    for t in small:
        if clear[t]:
            _check(got[t:t + 1], ora.out[t:t + 1], "token scaled by %g" % small[t])


def test_forward_on_host_buffers_matches_the_device_call():
    """moe_forward_host (x and out in pinned host memory, copies ordered on the stream)
    gives the device call's output bit for bit; a workspace without room for the copies is
    refused before anything runs."""
    c = synth.CONFIGS["tiny"]
    T, H, I, E, k = c["T"], c["H"], c["I"], c["E"], c["k"]
    gs_i = INTER["tiny"]["inter_global_scale"]
    layer = build_layer(0, H, I, E)
    wr = synth.router_weight(0, E, H)
    x = synth.activations(0, T, H)
    h = make_layer(layer, wr, H, I, E, k, inter_gs=gs_i, max_tokens=T)
    want = host(h.forward(bits16(x)))
    torch.cuda.synchronize()
    ws = torch.zeros(moe.moe_workspace_size_host(h.cfg, T), dtype=torch.uint8, device="cuda")
    assert ws.numel() >= h.workspace_bytes(T) + 2 * T * H * 2
    xh = torch.from_numpy(x.view(np.int16).copy()).pin_memory()
    oh = torch.zeros((T, H), dtype=torch.int16).pin_memory()
    for _ in range(2):
        moe.moe_forward_host(h.handle, xh, None, None, T, oh, ws)
        torch.cuda.synchronize()
        assert np.array_equal(oh.numpy(), want)
    small = ws[:h.workspace_bytes(T)]
    with pytest.raises(moe.MoEError) as err:
        moe.moe_forward_host(h.handle, xh, None, None, T, oh, small)
    assert err.value.status == moe.MOE_ERR_WORKSPACE


@pytest.mark.parametrize("T", [16, 17])
def test_given_logits_forward_folds_the_activation_amax(T):
    """W4A4 with router logits given: at up to 16 tokens one top-k block clears the activation
    amax word and folds max |x| into it (no separate amax pass); from 17 on a separate pass
    runs.  Both give the oracle's activation scale exactly and the layer within the bar."""
    c = synth.CONFIGS["tiny"]
    H, I, E, k = c["H"], c["I"], c["E"], c["k"]
    gs_i = INTER["tiny"]["inter_global_scale"]
    layer = build_layer(0, H, I, E)
    wr = synth.router_weight(0, E, H)
    x = synth.activations(2, T, H, outlier_frac=0.02)
    lg = synth.logits_normal(2, T, E)
    h = make_layer(layer, wr, H, I, E, k, inter_gs=gs_i, max_tokens=T)
    for _ in range(2):  # twice: the word is cleared by each forward
        got = _forward(h, x, T, logits_in=lg)
    ora = oracle.moe_forward(oracle.make_cfg(T, H, I, E, k, inter_gs=gs_i), x, layer,
                             logits_in=lg)
    gs = _read_ws(h, moe.moe_forward_buffers(h.handle, h.ws, T)["gs_a"], 1, np.float32)[0]
    assert float(gs) == ora.gs_a
    _check(got, ora.out, "given logits, T=%d" % T)
