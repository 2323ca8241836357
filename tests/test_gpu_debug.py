"""The MOE_DEBUG flavour of the library on the GPU: indices read from caller buffers that
are out of range are caught on the device, recorded as MOE_DEV_BAD_INDEX in the workspace
status word, and their accesses skipped -- no trap, the other rows computed as usual.

Only the debug flavour is given corrupted indices (its checks cover every access made with
them); the release library never sees them."""
import ctypes as C

import numpy as np
import pytest
import torch

import nvfp4_mixture_experts_gb300 as moe
import oracle
import synth
from gpu_util import bits16, dev, host, tiled_to_canonical, upload_weights
from helpers import build_layer

pytestmark = pytest.mark.gpu

H, I, E, k, T = 256, 128, 16, 2, 40


def _p(t):
    return None if t is None else C.c_void_p(t.data_ptr())


@pytest.fixture(scope="module")
def dbg():
    return moe.load_debug()


def _handle(lib, tiling):
    layer = build_layer(3, H, I, E)
    wr = synth.router_weight(3, E, H)
    wd = upload_weights(layer, wr)
    cfg = moe.make_config(H, I, E, k, inter_gs=64.0, max_tokens=T, gemm_tiling=tiling)
    w = moe.moe_weights(*[_p(wd.get(n)) for n in (
        "router_w", "w13", "w13_sf", "w13_gs", "w2", "w2_sf", "w2_gs",
        "sh13", "sh13_sf", "sh13_gs", "sh2", "sh2_sf", "sh2_gs")])
    h = C.c_void_p()
    s = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.moe_create(C.byref(cfg), C.byref(w), s, C.byref(h)) == moe.MOE_OK
    return h, cfg, layer, s


def _status(lib, h, ws, s):
    bits = C.c_uint32()
    st = lib.moe_get_status(h, _p(ws), s, C.byref(bits))
    return st, bits.value


@pytest.mark.parametrize("tiling", [1, 2, 3, 4])
def test_debug_build_flags_bad_indices_without_a_trap(dbg, tiling):
    h, cfg, layer, s = _handle(dbg, tiling)
    try:
        cap = dbg.moe_rows_capacity(C.byref(cfg), T)
        ws = torch.zeros(dbg.moe_workspace_size(C.byref(cfg), T), dtype=torch.uint8,
                         device="cuda")
        nbytes = ws.numel()
        lg = synth.logits_normal(4, T, E)
        ids = torch.zeros((T, k), dtype=torch.int32, device="cuda")
        w = torch.zeros((T, k), dtype=torch.float32, device="cuda")
        assert dbg.moe_route_topk(h, None, _p(dev(lg)), None, T, _p(ids), _p(w), None, None, 0,
                                  s) == moe.MOE_OK
        counts = torch.zeros(E + 1, dtype=torch.int32, device="cuda")
        offsets = torch.zeros(E + 2, dtype=torch.int32, device="cuda")
        perm = torch.zeros(cap, dtype=torch.int32, device="cuda")
        inv = torch.zeros(T * k, dtype=torch.int32, device="cuda")
        assert dbg.moe_permute(h, _p(ids), T, _p(counts), _p(offsets), _p(perm), _p(inv),
                               _p(ws), nbytes, s) == moe.MOE_OK
        torch.cuda.synchronize()
        assert _status(dbg, h, ws, s) == (moe.MOE_OK, 0)
        x = synth.activations(4, T, H)
        pitch = (H // 2 + 127) // 128 * 128
        a_codes = torch.zeros(cap * pitch, dtype=torch.uint8, device="cuda")
        a_sf = torch.zeros(cap * H // 16, dtype=torch.uint8, device="cuda")
        gs = torch.zeros(1, dtype=torch.float32, device="cuda")
        # three pairs point outside the padded rows (past the capacity, far past it, below -1)
        bad = inv.clone()
        bad_pairs = [3, 17, 30]
        bad[3], bad[17], bad[30] = cap + 5, 1 << 30, -5
        assert dbg.moe_gather_activations(h, _p(bits16(x)), T, _p(bad), _p(offsets),
                                          _p(a_codes), _p(a_sf), None, _p(gs), _p(ws), nbytes,
                                          s) == moe.MOE_OK
        torch.cuda.synchronize()
        st, bits = _status(dbg, h, ws, s)
        assert st == moe.MOE_ERR_DEVICE_STATUS and bits & moe.MOE_DEV_BAD_INDEX, (st, bits)
        # every other pair's row holds its token's NVFP4 codes and scales
        rc, rs, _ = oracle.quant_nvfp4(synth.bf16_to_f32(x))
        c, sc = tiled_to_canonical(host(a_codes), host(a_sf), cap, H)
        invh = host(inv)
        for p in range(T * k):
            if p in bad_pairs or invh[p] < 0:
                continue
            assert np.array_equal(c[invh[p]], rc[p // k]) and np.array_equal(sc[invh[p]], rs[p // k])
        # the down GEMM with a corrupted pair index: flagged, that row's weight taken as 0
        ic = torch.zeros(cap * ((I // 2 + 127) // 128 * 128), dtype=torch.uint8, device="cuda")
        isf = torch.zeros(cap * I // 16, dtype=torch.uint8, device="cuda")
        assert dbg.moe_grouped_gemm_gateup(h, _p(a_codes), _p(a_sf), _p(gs), None, _p(counts),
                                           _p(offsets), 1, None, _p(ic), _p(isf), None, T,
                                           _p(ws), nbytes, s) == moe.MOE_OK
        perm_bad = perm.clone()
        perm_bad[int(invh[0])] = -9
        y = torch.zeros((cap, H), dtype=torch.float32, device="cuda")
        assert dbg.moe_grouped_gemm_down(h, _p(ic), _p(isf), None, _p(counts), _p(offsets),
                                         _p(perm_bad), _p(w), _p(y), T, _p(ws), nbytes,
                                         s) == moe.MOE_OK
        torch.cuda.synchronize()
        st, bits = _status(dbg, h, ws, s)
        assert st == moe.MOE_ERR_DEVICE_STATUS and bits == moe.MOE_DEV_BAD_INDEX, (st, bits)
        assert not host(y)[int(invh[0])].any()
        # the same calls with intact indices raise nothing
        assert dbg.moe_grouped_gemm_down(h, _p(ic), _p(isf), None, _p(counts), _p(offsets),
                                         _p(perm), _p(w), _p(y), T, _p(ws), nbytes,
                                         s) == moe.MOE_OK
        torch.cuda.synchronize()
        assert _status(dbg, h, ws, s) == (moe.MOE_OK, 0)
    finally:
        dbg.moe_destroy(h)
