"""The C-ABI library builds, loads and exports every symbol include/nvfp4moe.h declares;
host-side argument checks answer without a GPU (no compute call is made here)."""
import ctypes as C
import os
import re

import pytest

import nvfp4_mixture_experts_gb300 as moe
from nvfp4_mixture_experts_gb300 import build as moe_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "nvfp4moe.h")


@pytest.fixture(scope="module")
def lib():
    moe_build.build()
    return moe.load()


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_0-9]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = _declared_functions()
    for n in ("moe_create", "moe_route_topk", "moe_permute", "moe_quant_nvfp4",
              "moe_grouped_gemm_gateup", "moe_swiglu_requant", "moe_grouped_gemm_down",
              "moe_combine", "moe_forward"):
        assert n in names
    assert set(names) == set(moe.SIGNATURES), "binding and header disagree"


def test_every_declared_symbol_is_exported(lib):
    for n in _declared_functions():
        assert hasattr(lib, n), n
        assert C.cast(getattr(lib, n), C.c_void_p).value


def test_status_strings(lib):
    for s in range(7):
        assert lib.moe_status_string(s)


def _cfg(**kw):
    d = dict(H=256, I=128, E=16, k=2)
    d.update(kw)
    return moe.make_config(d.pop("H"), d.pop("I"), d.pop("E"), d.pop("k"), **d)


def test_workspace_and_capacity_host_logic(lib):
    cfg = _cfg(max_tokens=64)
    T = 16
    cap = moe.moe_rows_capacity(cfg, T)
    # routed: 128 * (ceil(T*k/128) + min(E_loc, T*k)), shared: round_up(T, 128)
    assert cap == 128 * (1 + 16) + 128
    assert moe.moe_workspace_size(cfg, T) > cap * (256 // 2)
    assert moe.moe_rows_capacity(cfg, 0) == 0
    assert moe.moe_rows_capacity(_cfg(add_shared=0), 4) == 128 * (1 + 8)
    # the dynamic intermediate scale keeps the fp32 intermediate [rows][I] in the workspace
    dyn = _cfg(max_tokens=64, inter_gs=0.0)
    assert moe.moe_workspace_size(dyn, T) >= moe.moe_workspace_size(cfg, T) + cap * dyn.inter * 4


def test_invalid_configs_are_rejected_before_any_launch(lib):
    bad = [
        _cfg(H=200),                   # H % 128
        _cfg(I=96),                    # I % 64
        _cfg(k=17),                    # k > E
        _cfg(E_loc=10, off=8),         # shard past E
        _cfg(inter_gs=-1.0),           # W4A4: a static scale > 0, or 0 for the dynamic one
        _cfg(act_mode=moe.MOE_W4A4_STATIC, act_gs=0.0),
    ]
    for cfg in bad:
        assert moe.moe_workspace_size(cfg, 4) == 0
        h = C.c_void_p()
        st = lib.moe_create(C.byref(cfg), C.byref(moe.moe_weights()), None, C.byref(h))
        assert st in (moe.MOE_ERR_INVALID, moe.MOE_ERR_UNSUPPORTED) and not h.value


def test_null_arguments(lib):
    cfg = _cfg()
    h = C.c_void_p()
    assert lib.moe_create(C.byref(cfg), None, None, C.byref(h)) == moe.MOE_ERR_INVALID
    assert lib.moe_create(None, None, None, C.byref(h)) == moe.MOE_ERR_INVALID
    assert lib.moe_forward(None, None, None, None, 1, None, None, 0, None) == moe.MOE_ERR_INVALID
    assert lib.moe_quant_nvfp4(None, 1, 64, None, None, None, None, 0, None, 0, None) == \
        moe.MOE_ERR_INVALID
    # cols not a multiple of 64 -> unsupported, before anything runs
    dummy = C.c_void_p(256)
    assert lib.moe_quant_nvfp4(dummy, 1, 48, dummy, None, dummy, dummy, 0, None, 0, None) == \
        moe.MOE_ERR_UNSUPPORTED
    assert lib.moe_swiglu_requant(dummy, 1, 96, C.c_float(1.0), dummy, dummy, 0, None) == \
        moe.MOE_ERR_UNSUPPORTED
    assert lib.moe_swiglu_requant(dummy, 1, 128, C.c_float(0.0), dummy, dummy, 0, None) == \
        moe.MOE_ERR_INVALID


def test_every_declaration_cites_its_passage():
    """Each MOE_API declaration is preceded by a comment that names the passage of the pages
    defining the operation ([OV], [EP], [CK]) or says it has none (library plumbing)."""
    lines = open(HEADER).read().split("\n")
    for i, ln in enumerate(lines):
        m = re.match(r"MOE_API [^(]*\b(moe_[a-z_0-9]+)\s*\(", ln)
        if not m:
            continue
        j = i - 1
        assert lines[j].rstrip().endswith("*/"), m.group(1)
        block = []
        while True:
            block.insert(0, lines[j])
            if lines[j].lstrip().startswith("/*"):
                break
            j -= 1
        text = " ".join(block)
        assert re.search(r"Passage: (\[(OV|EP|CK)\]|none)", text), m.group(1)


def test_debug_flavour_builds_and_exports_the_same_symbols():
    """The MOE_DEBUG flavour (device bounds checks on indices read from buffers) compiles
    from the same sources and exports every declared call."""
    path = moe_build.build(debug=True)
    assert path == moe_build.LIB_DEBUG and os.path.exists(path)
    dbg = moe.load_debug()
    for n in _declared_functions():
        assert C.cast(getattr(dbg, n), C.c_void_p).value, n

