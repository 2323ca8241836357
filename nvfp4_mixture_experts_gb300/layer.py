"""MoELayer: owns a handle and a workspace; marshals torch tensors into the C calls."""
import torch

from . import (MOE_W4A4_DYNAMIC, moe_config, moe_create, moe_destroy, moe_forward,
               moe_rows_capacity, moe_weights, moe_workspace_size)


def make_config(H, I, E, k, E_loc=None, off=0, has_shared=1, add_shared=1,
                act_mode=MOE_W4A4_DYNAMIC, act_gs=0.0, inter_gs=1.0, max_tokens=8192,
                gemm_tiling=0):
    return moe_config(H, I, E, k, E if E_loc is None else E_loc, off, has_shared, I,
                      add_shared, act_mode, act_gs, inter_gs, max_tokens, gemm_tiling)


def _ptr(t):
    return None if t is None else t.data_ptr()


class MoELayer:
    """One layer (or expert shard) on the current CUDA device.

    weights: dict of device tensors in the canonical layouts of include/nvfp4moe.h:
      router_w bf16 bits (int16/uint16) [E, H]; w13 uint8 [El, 2I, H/2]; w13_sf uint8
      [El, 2I, H/16]; w13_gs float32 [El]; w2, w2_sf, w2_gs likewise; optional shared
      sh13, sh13_sf, sh13_gs [1], sh2, sh2_sf, sh2_gs [1].
    The library copies them; the tensors may be freed afterwards."""

    def __init__(self, cfg, weights, stream=None, workspace=None):
        self.cfg = cfg
        w = moe_weights(*[_ptr(weights.get(n)) for n in (
            "router_w", "w13", "w13_sf", "w13_gs", "w2", "w2_sf", "w2_gs",
            "sh13", "sh13_sf", "sh13_gs", "sh2", "sh2_sf", "sh2_gs")])
        self.handle = moe_create(cfg, w, stream)
        self.ws = workspace

    def workspace_bytes(self, T):
        return moe_workspace_size(self.cfg, T)

    def rows_capacity(self, T):
        return moe_rows_capacity(self.cfg, T)

    def ensure_workspace(self, T, device="cuda"):
        need = self.workspace_bytes(T)
        if self.ws is None or self.ws.numel() < need:
            self.ws = torch.zeros(need, dtype=torch.uint8, device=device)
        return self.ws

    def forward(self, x, out=None, logits_in=None, logit_bias=None, stream=None):
        T = x.shape[0]
        if out is None:
            out = torch.empty((T, self.cfg.hidden), dtype=torch.int16, device=x.device)
        ws = self.ensure_workspace(T, x.device)
        moe_forward(self.handle, x, logits_in, logit_bias, T, out, ws, stream)
        return out

    def close(self):
        if self.handle is not None:
            moe_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
