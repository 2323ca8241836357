"""Writes inter_scale.json: the static global scale of the intermediate (post-SwiGLU)
activation for each workload, calibrated with the ORACLE only.

Rule: run a calibration batch (activations from seed 1, the layer's weights from seed 0)
through routing and the experts' gate/up projections, take amax of silu(gate) * up over
every routed and shared pair, and set gs_i = 2^floor(log2(2688 / (2 * amax))): a power
of two (so the scale itself introduces no rounding) with at least 2x headroom before the
E4M3 block scale saturates at 448.  A workload with the dynamic intermediate scale gets 0.
A workload with a static activation scale gets act_global_scale by the same rule from
amax |x| of the calibration batch.

Usage: python tests/golden/make_inter_scale.py
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)
sys.path.insert(0, os.path.join(ROOT, "tests"))

import oracle  # noqa: E402
import synth  # noqa: E402
from helpers import build_layer  # noqa: E402

CAL_TOKENS = 64


def calibrate(name):
    c = synth.CONFIGS[name]
    H, I, E, k = c["H"], c["I"], c["E"], c["k"]
    T = min(c["T"], CAL_TOKENS)
    x = synth.activations(1, T, H, outlier_frac=c["outlier_frac"])
    bias = synth.zipf_bias(0, E) if c["bias"] else None
    if c["logits"]:
        lg = synth.logits_normal(1, T, E).astype(np.float64)
    else:
        lg = oracle.router_logits(x, synth.router_weight(0, E, H), bias)
    ids, _ = oracle.topk(lg, k)
    used = sorted(set(ids.ravel().tolist()))
    layer = build_layer(0, H, I, E, experts=used)
    cfg = oracle.make_cfg(T, H, I, E, k, E_loc=len(used), act_mode=0)
    xc, xsf, gs_a = oracle.quant_nvfp4(synth.bf16_to_f32(x))
    amax = 0.0
    for li, e in enumerate(used + ["shared"]):
        tok = np.arange(T, dtype=np.int32) if e == "shared" else \
            np.nonzero((ids == e).any(1))[0].astype(np.int32)
        G = oracle.expert_rows(cfg, layer, li if e != "shared" else "shared",
                               x, xc, xsf, gs_a, tok)[0]
        g, u = G[:, :I], G[:, I:]
        s = g / (1.0 + np.exp(-g)) * u
        amax = max(amax, float(np.abs(s).max()))
    gs = float(2.0 ** np.floor(np.log2(2688.0 / (2.0 * amax))))
    out = dict(inter_global_scale=0.0 if c.get("inter") == "dynamic" else gs, amax=amax,
               cal_tokens=T)
    if c["act_mode"] == 1:
        xa = float(np.abs(synth.bf16_to_f32(x)).max())
        out["act_global_scale"] = float(2.0 ** np.floor(np.log2(2688.0 / (2.0 * xa))))
        out["act_amax"] = xa
    return out


def main():
    out = {"_rule": __doc__.strip().splitlines()[2:11]}
    for name in synth.CONFIGS:
        out[name] = calibrate(name)
        print(name, out[name], flush=True)
    with open(os.path.join(HERE, "inter_scale.json"), "w") as f:
        json.dump(out, f, indent=1)


if __name__ == "__main__":
    main()
