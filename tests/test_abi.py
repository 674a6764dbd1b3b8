"""The C-ABI library builds, loads and exports every entry point the header
declares; host-side config validation needs no GPU."""

import ctypes
import os
import re

import pytest

from moe_decode_layer_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    inc = os.path.join(ROOT, "include")
    for f in os.listdir(inc):
        if f.endswith(".h"):
            src = open(os.path.join(inc, f)).read()
            names |= set(re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(moe_decode_\w+)\s*\(", src, re.M))
    return names


def test_every_declared_symbol_is_exported():
    lib = _lib.load()
    declared = _declared()
    assert {"moe_decode_create", "moe_decode_run", "moe_decode_destroy"} <= declared
    for name in declared:
        assert hasattr(lib, name), name
    assert set(_lib.EXPORTS) == declared


def test_abi_version_and_strings():
    lib = _lib.load()
    assert lib.moe_decode_abi_version() == 3
    for s in range(6):
        assert _lib.status_string(s)
    assert _lib.status_string(0) == "ok"
    assert "unknown" in _lib.status_string(99)


def _cfg(**kw):
    base = dict(hidden=2560, inter=768, num_experts=512, top_k=8, num_shared=1, max_rows=6,
                wdtype=0, score=0, routed_scale=1.0, pre_rmsnorm=0, rms_eps=1e-6, sched=0)
    base.update(kw)
    return _lib.Config(**base)


def _check(**kw):
    c = _cfg(**kw)
    return _lib.load().moe_decode_config_check(ctypes.byref(c))


def test_supported_configs():
    assert _check() == 0
    assert _check(hidden=256, inter=128, num_experts=16, top_k=2, max_rows=1) == 0
    assert _check(hidden=4096, inter=1024, num_experts=256, top_k=8, num_shared=0, wdtype=1) == 0
    assert _check(wdtype=2) == 0  # FP8 block-quantised Ling shape
    assert _check(wdtype=2, hidden=256, inter=128, max_rows=16) == 0
    assert _check(pre_rmsnorm=1, rms_eps=1e-6) == 0
    assert _check(sched=1) == 0 and _check(sched=2) == 0
    assert _check(top_k=16, num_experts=16) == 0
    assert _check(inter=64) == 0  # 8 threads per down group


@pytest.mark.parametrize("kw,status", [
    (dict(num_experts=513), _lib.MOE_ERR_UNSUPPORTED),
    (dict(num_experts=2048), _lib.MOE_ERR_UNSUPPORTED),
    (dict(top_k=17), _lib.MOE_ERR_UNSUPPORTED),
    (dict(top_k=9, num_experts=8), _lib.MOE_ERR_UNSUPPORTED),
    (dict(max_rows=17), _lib.MOE_ERR_UNSUPPORTED),
    (dict(max_rows=0), _lib.MOE_ERR_INVALID_ARG),
    (dict(hidden=2564), _lib.MOE_ERR_UNSUPPORTED),
    (dict(hidden=8192), _lib.MOE_ERR_UNSUPPORTED),
    (dict(inter=776), _lib.MOE_ERR_UNSUPPORTED),      # 97 threads per group
    (dict(inter=4096), _lib.MOE_ERR_UNSUPPORTED),     # more than one CTA's consumers
    (dict(wdtype=1, hidden=2176), _lib.MOE_ERR_UNSUPPORTED),  # not a multiple of 256
    (dict(wdtype=3), _lib.MOE_ERR_UNSUPPORTED),
    (dict(wdtype=2, hidden=2496), _lib.MOE_ERR_UNSUPPORTED),  # FP8: not a multiple of 128
    (dict(wdtype=2, inter=640), _lib.MOE_ERR_UNSUPPORTED),    # FP8: not a multiple of 128
    (dict(wdtype=2, inter=384), _lib.MOE_ERR_UNSUPPORTED),    # FP8: 48 threads per down row
    (dict(score=2), _lib.MOE_ERR_UNSUPPORTED),
    (dict(sched=3), _lib.MOE_ERR_UNSUPPORTED),
    (dict(num_shared=5), _lib.MOE_ERR_UNSUPPORTED),
    (dict(num_shared=-1), _lib.MOE_ERR_INVALID_ARG),
    (dict(pre_rmsnorm=1, rms_eps=0.0), _lib.MOE_ERR_INVALID_ARG),
    (dict(routed_scale=float("inf")), _lib.MOE_ERR_INVALID_ARG),
])
def test_rejected_configs(kw, status):
    assert _check(**kw) == status


def test_null_config():
    assert _lib.load().moe_decode_config_check(None) == _lib.MOE_ERR_INVALID_ARG
