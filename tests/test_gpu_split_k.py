"""GPU parity of the split-K kernel (down matrices stored transposed, w2_layout
"i_h"): each CTA applies the down projection to the h rows it computed, and the
output is a fixed-order sum of every CTA's partial sums ("Muse Spark Open
Ultrafast", section "A new tensor parallelism": the second expert GEMM split on
the intermediate dimension, one reduction at the end). Same layer, same oracle
and tolerances as the row-block kernels; the weights hold the same values in
both layouts for one seed.
"""

import numpy as np
import pytest
import torch

from moe_decode_layer_gb300 import _lib, synth
from moe_decode_layer_gb300.layer import MoEDecodeLayer
from tests import helpers

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _needs_cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _run(shape, layer, x, residual=None, out=None, max_rows=None, score=0, **kw):
    m = x.shape[0]
    mod = MoEDecodeLayer(shape, layer, max_rows or m, score=score, **kw)
    assert mod.info(_lib.MOE_INFO_SPLIT_K) == 1
    xd = x.cuda()
    rd = xd if residual is None else residual.cuda()
    idx = torch.empty((m, shape.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((m, shape.top_k), dtype=torch.float32, device="cuda")
    o = mod.run(xd, rd, out, idx, w)
    assert mod.status() == _lib.MOE_OK
    return mod, o, idx, w


SMALL = [
    synth.LayerShape(hidden=256, inter=128, num_experts=16, top_k=2, num_shared=1),
    synth.LayerShape(hidden=512, inter=256, num_experts=40, top_k=6, num_shared=2),
    synth.LayerShape(hidden=64, inter=96, num_experts=8, top_k=3, num_shared=0),
    synth.LayerShape(hidden=384, inter=128, num_experts=16, top_k=4, num_shared=1, wdtype="fp8"),
]


@pytest.mark.parametrize("shape", SMALL, ids=["tiny", "h512_s2", "h64_s0_fewer_rows_than_ctas", "fp8"])
def test_small_shapes_all_row_counts(shape):
    """Row counts 1..16 (above 8: row groups), including a hidden size below the
    CTA count (CTAs without output rows) and an expert count that is not a
    multiple of 32; every result repeats bit for bit."""
    layer = synth.make_layer(shape, seed=31, device="cuda", w2_layout="i_h")
    for m in (1, 2, 5, 8, 11, 16):
        x = helpers.hidden_with_margin(layer["router_w"], m, shape.top_k, seed=300 + m, rho=0.5)
        mod, out, idx, w = _run(shape, layer, x, max_rows=16)
        ref, ridx, rw = helpers.oracle_layer(shape, layer, x, x)
        helpers.assert_routing(idx.cpu(), w.cpu(), ridx, rw)
        helpers.assert_close(out.cpu(), ref, what=f"m={m}")
        again = mod.run(x.cuda(), x.cuda())
        assert mod.status() == _lib.MOE_OK
        assert torch.equal(out, again)


@pytest.mark.parametrize("m", [1, 6])
@pytest.mark.parametrize("wdtype", ["bf16", "fp8"])
def test_ling_shape(m, wdtype):
    shape = synth.LING if wdtype == "bf16" else synth.LING_FP8
    layer = synth.make_layer(shape, seed=33, device="cuda", w2_layout="i_h")
    x = helpers.hidden_with_margin(layer["router_w"], m, shape.top_k, seed=330 + m, rho=0.5)
    _, out, idx, w = _run(shape, layer, x)
    ref, ridx, rw = helpers.oracle_layer(shape, layer, x, x)
    helpers.assert_routing(idx.cpu(), w.cpu(), ridx, rw)
    helpers.assert_close(out.cpu(), ref)
    # the MoE part alone (zero residual)
    z = torch.zeros_like(x)
    _, out2, _, _ = _run(shape, layer, x, residual=z)
    ref2, _, _ = helpers.oracle_layer(shape, layer, x, z)
    helpers.assert_close(out2.cpu(), ref2)
    del layer
    torch.cuda.empty_cache()


def test_same_layer_as_row_block_layout():
    """The default layout and the transposed one hold the same weights for one
    seed: both kernels meet the oracle on the same input, and their outputs
    differ by no more than the summation order allows."""
    shape = synth.LayerShape(hidden=512, inter=256, num_experts=32, top_k=4, num_shared=1)
    a = synth.make_layer(shape, seed=35, device="cuda")
    b = synth.make_layer(shape, seed=35, device="cuda", w2_layout="i_h")
    x = helpers.hidden_with_margin(a["router_w"], 3, shape.top_k, seed=350)
    ma = MoEDecodeLayer(shape, a, 3)
    oa = ma.run(x.cuda(), x.cuda())
    _, ob, _, _ = _run(shape, b, x)
    ref, _, _ = helpers.oracle_layer(shape, a, x, x)
    helpers.assert_close(oa.cpu(), ref)
    helpers.assert_close(ob.cpu(), ref)
    d = (helpers.f64(oa.cpu()) - helpers.f64(ob.cpu()))
    assert np.abs(d).max() <= 2.0 ** -6 * np.abs(ref).max()


def test_in_place_and_sigmoid_bias():
    """out == x == residual (the output overwrites the input rows after every CTA
    has read them), under the bias-corrected sigmoid rule with routed scale 2.5."""
    shape = synth.LayerShape(hidden=256, inter=128, num_experts=32, top_k=4, num_shared=1)
    layer = synth.make_layer(shape, seed=37, device="cuda", w2_layout="i_h")
    bias = synth.router_bias(shape.num_experts, seed=37, device="cuda", std=0.2)
    lay = dict(layer, router_bias=bias)
    x = helpers.hidden_with_margin(layer["router_w"], 4, shape.top_k, seed=370, rho=0.5, margin=1e-3,
                                   score=1, bias=bias)
    ref, ridx, rw = helpers.oracle_layer(shape, lay, x, x, routed_scale=2.5, score=1, bias=bias)
    mod = MoEDecodeLayer(shape, lay, 4, score=1, routed_scale=2.5)
    xd = x.cuda().clone()
    idx = torch.empty((4, shape.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((4, shape.top_k), dtype=torch.float32, device="cuda")
    mod.run(xd, xd, xd, idx, w)
    assert mod.status() == _lib.MOE_OK
    helpers.assert_routing(idx.cpu(), w.cpu(), ridx, rw, by_weight=False)
    helpers.assert_close(xd.cpu(), ref)


def test_zero_rows():
    shape = synth.LayerShape(hidden=256, inter=128, num_experts=16, top_k=2, num_shared=1)
    layer = synth.make_layer(shape, seed=39, device="cuda", w2_layout="i_h")
    x = torch.zeros((3, shape.hidden), dtype=torch.bfloat16)
    _, out, idx, _ = _run(shape, layer, x)
    assert torch.count_nonzero(out.float()) == 0
    assert idx.cpu().tolist() == [[0, 1]] * 3


def test_chain_schedules_refused():
    shape = synth.LayerShape(hidden=256, inter=128, num_experts=16, top_k=2, num_shared=1)
    layer = synth.make_layer(shape, seed=41, device="cuda", w2_layout="i_h")
    with pytest.raises(_lib.MoEDecodeError):
        MoEDecodeLayer(shape, layer, 2, sched="pdl_chain")
    mod = MoEDecodeLayer(shape, layer, 2)
    with pytest.raises(_lib.MoEDecodeError):
        mod.set_option(_lib.MOE_OPT_SCHED, _lib.MOE_SCHED_CHAIN)
