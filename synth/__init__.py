"""Seeded synthetic inputs for the NVFP4 mixture-of-experts layer.

Shared by the tests, the oracle runs and the benchmark.  This module only draws random
numbers and rounds them to the layer's bf16 input format; it holds none of the layer's
arithmetic (no quantisation, routing or contraction).

Recipe (every stream is an independent numpy PCG64 generator keyed by a list):
  x        [T, H]  ~ N(0, 1), rounded to bf16            key [seed, 0]
           optional outlier channels: a fraction of the H columns, chosen without
           replacement with key [seed, 4], multiplied by a factor before rounding
  Wr       [E, H]  ~ N(0, 0.02), rounded to bf16         key [seed, 1]
  expert e w13 [2I, H], w2 [H, I] fp32 ~ N(0, 0.02)      key [seed, 2, e]
  shared   w13 [2I, H], w2 [H, I] fp32 ~ N(0, 0.02)      key [seed, 3]
  bias     [E] = -s * ln(rank_e), rank a permutation of 1..E   key [seed, 5]
           (a softmax prior proportional to rank^-s: Zipf popularity)
  logits   [T, E]  ~ N(0, 1) fp32 (router logits given directly)   key [seed, 6]
"""
from concurrent.futures import ThreadPoolExecutor
import os

import numpy as np


def _rng(*key):
    return np.random.default_rng(list(key))


def bf16_bits(f32):
    """fp32 array -> bf16 bit patterns (uint16), round to nearest even (inputs finite)."""
    u = np.ascontiguousarray(f32, dtype=np.float32).view(np.uint32)
    rounding = ((u >> 16) & 1) + np.uint32(0x7FFF)
    return ((u + rounding) >> 16).astype(np.uint16)


def bf16_to_f32(bits):
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def activations(seed, T, H, outlier_frac=0.0, outlier_scale=20.0):
    x = _rng(seed, 0).standard_normal((T, H), dtype=np.float32)
    if outlier_frac > 0:
        n = int(round(outlier_frac * H))
        cols = np.sort(_rng(seed, 4).choice(H, size=n, replace=False))
        x[:, cols] *= np.float32(outlier_scale)
    return bf16_bits(x)


def outlier_channels(seed, H, outlier_frac):
    n = int(round(outlier_frac * H))
    return np.sort(_rng(seed, 4).choice(H, size=n, replace=False))


def router_weight(seed, E, H, std=0.02):
    return bf16_bits(_rng(seed, 1).standard_normal((E, H), dtype=np.float32) * np.float32(std))


def expert_master(seed, e, H, I, std=0.02):
    """fp32 masters of routed expert e: (w13 [2I, H] rows gate then up, w2 [H, I])."""
    g = _rng(seed, 2, e)
    w13 = g.standard_normal((2 * I, H), dtype=np.float32) * np.float32(std)
    w2 = g.standard_normal((H, I), dtype=np.float32) * np.float32(std)
    return w13, w2


def shared_master(seed, H, I, std=0.02):
    g = _rng(seed, 3)
    w13 = g.standard_normal((2 * I, H), dtype=np.float32) * np.float32(std)
    w2 = g.standard_normal((H, I), dtype=np.float32) * np.float32(std)
    return w13, w2


def zipf_bias(seed, E, s=1.1):
    rank = _rng(seed, 5).permutation(E).astype(np.float64) + 1.0
    return (-s * np.log(rank)).astype(np.float32)


def logits_normal(seed, T, E):
    return _rng(seed, 6).standard_normal((T, E), dtype=np.float32)


def map_experts(fn, experts, workers=None):
    """Apply fn(e) over expert ids with a thread pool (numpy's generators release the GIL)."""
    workers = workers or min(16, os.cpu_count() or 1)
    with ThreadPoolExecutor(workers) as ex:
        return list(ex.map(fn, experts))


# Layer configurations: dimensions and input recipe of each workload.
CONFIGS = {
    # tiny layer: 16 routed experts top-2 + 1 shared, hidden 256, intermediate 128
    "tiny": dict(T=16, H=256, I=128, E=16, k=2, E_loc=16, off=0, add_shared=1,
                 act_mode=0, outlier_frac=0.0, bias=False, logits=False),
    # decode-shaped layer: 320 routed top-8 + 1 shared, hidden 4096, intermediate 1280
    "decode": dict(T=64, H=4096, I=1280, E=320, k=8, E_loc=320, off=0, add_shared=1,
                   act_mode=0, outlier_frac=0.0, bias=False, logits=False),
    # prefill chunk: same layer, 8192 tokens, 1% outlier channels x20
    "prefill": dict(T=8192, H=4096, I=1280, E=320, k=8, E_loc=320, off=0, add_shared=1,
                    act_mode=0, outlier_frac=0.01, bias=False, logits=False),
    # expert shard 160..319 of the decode layer, Zipf(1.1) popularity, 2048 tokens
    "shard": dict(T=2048, H=4096, I=1280, E=320, k=8, E_loc=160, off=160, add_shared=0,
                  act_mode=0, outlier_frac=0.0, bias=True, logits=False),
    # the decode layer with a static activation scale (calibrated once, power of two)
    "decode_static": dict(T=64, H=4096, I=1280, E=320, k=8, E_loc=320, off=0, add_shared=1,
                          act_mode=1, outlier_frac=0.0, bias=False, logits=False),
    # the decode layer with the dynamic (per-call, two-pass) intermediate scale
    "decode_dyninter": dict(T=64, H=4096, I=1280, E=320, k=8, E_loc=320, off=0, add_shared=1,
                            act_mode=0, outlier_frac=0.0, bias=False, logits=False,
                            inter="dynamic"),
    # W4A16: bf16 activations x NVFP4 weights, router logits ~ N(0,1), decode sweep
    "w4a16": dict(T=256, H=4096, I=1280, E=320, k=8, E_loc=320, off=0, add_shared=1,
                  act_mode=2, outlier_frac=0.0, bias=False, logits=True,
                  sweep=(1, 8, 32, 128, 256)),
}
