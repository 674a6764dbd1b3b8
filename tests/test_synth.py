"""Synthetic inputs: determinism, shapes, and the top-k margin guarantee."""

import math

import numpy as np
import pytest
import torch

import oracle

from moe_decode_layer_gb300 import synth
from tests import helpers


def test_tiny_layer_shapes_and_determinism():
    a = synth.make_layer(synth.TINY, seed=0)
    b = synth.make_layer(synth.TINY, seed=0)
    c = synth.make_layer(synth.TINY, seed=1)
    assert a["w13"].shape == (16, 256, 256) and a["w2"].shape == (16, 256, 128)
    assert a["sh_w13"].shape == (1, 256, 256) and a["router_w"].shape == (16, 256)
    assert a["w2_layout"] == "h_i"
    for k in a:
        if k != "w2_layout":
            assert torch.equal(a[k], b[k])
    assert not torch.equal(a["w13"], c["w13"])
    std = a["w13"].float().std().item()
    assert abs(std - 0.02) < 0.001


def test_margin_rows_checked_with_plain_loops():
    """Pin of the margin draw: recompute each row's logits with Python loops."""
    layer = synth.make_layer(synth.TINY, seed=0)
    x = helpers.hidden_with_margin(layer["router_w"], 4, 2, seed=3, rho=0.5)
    rw = helpers.f64(layer["router_w"]).tolist()
    xs = helpers.f64(x).tolist()
    for row in xs:
        logits = sorted((sum(a * b for a, b in zip(row, wr)) for wr in rw), reverse=True)
        assert logits[1] - logits[2] >= 0.05


def test_correlated_rows():
    x = synth.hidden_rows(6, 4096, seed=0, rho=0.5).float().numpy()
    c = np.corrcoef(x)
    off = c[~np.eye(6, dtype=bool)]
    assert abs(off.mean() - 0.5) < 0.05
    assert abs(x.std() - 1.0) < 0.05


def test_nvfp4_layer_shapes():
    shape = synth.LayerShape(hidden=256, inter=256, num_experts=4, top_k=2, num_shared=1, wdtype="nvfp4")
    layer = synth.make_layer(shape, seed=0)
    assert layer["w13_q"].shape == (4, 512, 128) and layer["w13_s"].shape == (4, 512, 16)
    assert layer["w2_q"].shape == (4, 256, 128) and layer["w2_s"].shape == (4, 256, 16)
    assert layer["w13_gs"].shape == (4, 2) and layer["sh_w2_gs"].shape == (1,)
    # dequantised weights track the float draw's spread
    ex = helpers.expert_accessor(shape, layer)(0)
    w13 = np.vstack([oracle.dequant_nvfp4_rows(ex.q13[:256], ex.s13[:256], float(ex.gs13[0])),
                     oracle.dequant_nvfp4_rows(ex.q13[256:], ex.s13[256:], float(ex.gs13[1]))])
    w2 = oracle.dequant_nvfp4_rows(ex.q2, ex.s2, float(ex.gs2))
    assert abs(w13.std() - 0.02) < 0.003 and abs(w2.std() - 0.02) < 0.003


def test_algorithmic_bytes_ling():
    # 8 routed + 1 shared expert of 3*2560*768*2 B plus the 512x2560 bf16 router
    assert synth.algorithmic_bytes(synth.LING, 8) == 9 * 11_796_480 + 2_621_440
    assert synth.algorithmic_bytes(synth.MUSE_NVFP4, 8) == 8 * 7_077_888 + 2_097_152


@pytest.mark.parametrize("shape", [synth.TINY, synth.LayerShape(hidden=256, inter=128, num_experts=4, top_k=2,
                                                                num_shared=1, wdtype="fp8")], ids=["bf16", "fp8"])
def test_transposed_down_layout_holds_the_same_weights(shape):
    """w2_layout "i_h" stores each down matrix (and FP8 scale grid) transposed;
    the values are the same as in the default layout for the same seed."""
    a = synth.make_layer(shape, seed=3)
    b = synth.make_layer(shape, seed=3, w2_layout="i_h")
    assert b["w2_layout"] == "i_h"
    names = ("w2", "sh_w2") if shape.wdtype == "bf16" else ("w2_q", "w2_s", "sh_w2_q", "sh_w2_s")
    for n in names:
        assert b[n].shape == (a[n].shape[0], a[n].shape[2], a[n].shape[1])
        assert torch.equal(b[n], a[n].transpose(1, 2))
        assert b[n].is_contiguous()
    with pytest.raises(ValueError):
        synth.make_layer(synth.LayerShape(hidden=256, inter=256, num_experts=4, top_k=2, num_shared=0,
                                          wdtype="nvfp4"), seed=1, w2_layout="i_h")
