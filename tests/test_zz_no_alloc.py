"""moe_route_topk_noalloc: routing for callers that cannot allocate device memory during a
call and have no workspace to lend (its scratch is a static device array of the library).
Checked through the C ABI against moe_route_topk (which uses a caller workspace), on two
calls in a row; at sizes where it sums fewer router k-splits than moe_route_topk (T = 4096,
and T = 6553, the largest that fits at E = 320), its ids against the oracle's top-k of the
logits it returns; and its size limit is checked to fail cleanly.

This file is collected last on purpose, and builds everything it needs itself, so it runs
the same alone in a fresh process or after the other tests."""
import numpy as np
import pytest
import torch

import nvfp4_mixture_experts_gb300 as moe
import oracle
import synth
from gpu_util import bits16, dev, host, make_layer

pytestmark = pytest.mark.gpu


def _routing_handle(E=320, H=4096, I=64, k=8, max_tokens=8192):
    z = lambda *shape: np.zeros(shape, np.uint8)
    one = lambda n: np.ones(n, np.float32)
    layer = oracle.Layer(z(E, 2 * I, H // 2), z(E, 2 * I, H // 16), one(E), z(E, H, I // 2),
                         z(E, H, I // 16), one(E), z(2 * I, H // 2), z(2 * I, H // 16), 1.0,
                         z(H, I // 2), z(H, I // 16), 1.0)
    wr = synth.router_weight(7, E, H)
    return make_layer(layer, wr, H, I, E, k, inter_gs=64.0, max_tokens=max_tokens)


@pytest.mark.parametrize("T", [64, 700])
def test_noalloc_routing_matches_workspace_routing(T):
    E, H, k = 320, 4096, 8
    h = _routing_handle(E=E, H=H, k=k)
    x = bits16(synth.activations(9, T, H))
    ws = torch.zeros(h.workspace_bytes(T), dtype=torch.uint8, device="cuda")
    ids = torch.zeros((T, k), dtype=torch.int32, device="cuda")
    w = torch.zeros((T, k), dtype=torch.float32, device="cuda")
    lo = torch.zeros((T, E), dtype=torch.float32, device="cuda")
    moe.moe_route_topk(h.handle, x, None, None, T, ids, w, lo, ws)
    torch.cuda.synchronize()
    for _ in range(2):  # the shared scratch keeps the previous call's contents
        ids2 = torch.full((T, k), -1, dtype=torch.int32, device="cuda")
        w2 = torch.zeros((T, k), dtype=torch.float32, device="cuda")
        lo2 = torch.zeros((T, E), dtype=torch.float32, device="cuda")
        moe.moe_route_topk_noalloc(h.handle, x, None, None, T, ids2, w2, lo2)
        torch.cuda.synchronize()
        ref_lo = host(lo).astype(np.float64)
        assert np.max(np.abs(host(lo2) - ref_lo)) <= 1e-5 * np.max(np.abs(ref_lo))
        assert np.array_equal(host(ids2), host(ids))
        assert np.max(np.abs(host(w2) - host(w))) <= 1e-6


@pytest.mark.parametrize("T", [4096, 6553])
def test_noalloc_routing_at_large_batches_selects_the_topk_of_its_logits(T):
    """Beyond 1638 tokens (E = 320) the scratch holds fewer partial planes than the
    workspace call uses, so the logits are summed in another fp32 order: they agree with
    moe_route_topk's to fp32 rounding, and the ids are exactly the top-k of the logits this
    call returns (6553 x 320 fills the scratch up to its status word)."""
    E, H, k = 320, 4096, 8
    h = _routing_handle(E=E, H=H, k=k)
    x = bits16(synth.activations(11, T, H))
    ws = torch.zeros(h.workspace_bytes(T), dtype=torch.uint8, device="cuda")
    lo = torch.zeros((T, E), dtype=torch.float32, device="cuda")
    ids = torch.zeros((T, k), dtype=torch.int32, device="cuda")
    w = torch.zeros((T, k), dtype=torch.float32, device="cuda")
    moe.moe_route_topk(h.handle, x, None, None, T, ids, w, lo, ws)
    for _ in range(2):
        ids2 = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
        w2 = torch.zeros((T, k), dtype=torch.float32, device="cuda")
        lo2 = torch.zeros((T, E), dtype=torch.float32, device="cuda")
        moe.moe_route_topk_noalloc(h.handle, x, None, None, T, ids2, w2, lo2)
        torch.cuda.synchronize()
        l2 = host(lo2).astype(np.float64)
        ref = host(lo).astype(np.float64)
        assert np.max(np.abs(l2 - ref)) <= 1e-5 * np.max(np.abs(ref))
        rid, rw = oracle.topk(l2, k)
        assert np.array_equal(host(ids2), rid)
        assert np.max(np.abs(host(w2) - rw)) <= 1e-6


def test_noalloc_routing_with_given_logits_and_the_size_limit():
    E, k = 320, 8
    h = _routing_handle(E=E, k=k)
    T = 100
    lg = synth.logits_normal(3, T, E)
    ids = torch.zeros((T, k), dtype=torch.int32, device="cuda")
    w = torch.zeros((T, k), dtype=torch.float32, device="cuda")
    moe.moe_route_topk_noalloc(h.handle, None, dev(lg), None, T, ids, w, None)
    rid, rw = oracle.topk(lg.astype(np.float64), k)
    assert np.array_equal(host(ids), rid)
    assert np.max(np.abs(host(w) - rw)) <= 1e-6
    # T * E beyond the 8 MiB scratch (less its status word): a clean error, nothing launched
    T_big = (2 ** 21 - 64) // E + 1
    x = torch.zeros((T_big, 4096), dtype=torch.int16, device="cuda")
    ids = torch.zeros((T_big, k), dtype=torch.int32, device="cuda")
    w = torch.zeros((T_big, k), dtype=torch.float32, device="cuda")
    with pytest.raises(moe.MoEError) as err:
        moe.moe_route_topk_noalloc(h.handle, x, None, None, T_big, ids, w, None)
    assert err.value.status == moe.MOE_ERR_WORKSPACE
