"""GPU (CUDA path through the C ABI) against the float64 oracle.

Expert index sets must match exactly (inputs are drawn with a top-k logit gap of
at least 0.05), routing weights within 1e-5, outputs within max-abs 2e-2 and
relative L2 5e-3 of the oracle. Cases span the tiny layer, the Ling-shaped layer
at full size (M = 1 and M = 6 correlated rows) in the launch configuration the
bench times, ragged and degenerate shapes, all three schedules (which must agree
bit for bit), in-place outputs, repeated runs, graph capture and the host-buffer
entry point. The expert-range kernel ("flat") sums each output over the experts in
another order (per expert, then over experts), so it is held to the oracle and to
bitwise repeatability rather than to bit equality with the others.
"""

import numpy as np
import pytest
import torch

from oracle import cpp
from moe_decode_layer_gb300 import _lib, synth
from moe_decode_layer_gb300.layer import MoEDecodeLayer
from tests import helpers

pytestmark = pytest.mark.gpu

SCHEDS = ["persistent", "phased", "interleaved", "flat", "pdl_chain", "chain"]
# schedules that sum every output in the same order (bit-identical results)
SAME_ORDER = ["phased", "interleaved", "pdl_chain", "chain"]


@pytest.fixture(scope="module", autouse=True)
def _needs_cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.fixture(scope="module")
def tiny():
    return synth.make_layer(synth.TINY, seed=0, device="cuda")


@pytest.fixture(scope="module")
def ling():
    layer = synth.make_layer(synth.LING, seed=1, device="cuda")
    yield layer
    del layer
    torch.cuda.empty_cache()


def _run(shape, layer, x, residual=None, sched="persistent", max_rows=None, **kw):
    m = x.shape[0]
    mod = MoEDecodeLayer(shape, layer, max_rows or m, sched=sched, **kw)
    xd = x.cuda()
    rd = xd if residual is None else residual.cuda()
    out = torch.empty_like(xd)
    idx = torch.full((m, shape.top_k), -1, dtype=torch.int32, device="cuda")
    w = torch.zeros((m, shape.top_k), dtype=torch.float32, device="cuda")
    mod.run(xd, rd, out, idx, w)
    assert mod.status() == _lib.MOE_OK
    torch.cuda.synchronize()
    return mod, out.cpu(), idx.cpu(), w.cpu()


def _check(shape, layer, x, out, idx, w, residual=None):
    ref, ridx, rw = helpers.oracle_layer(shape, layer, x, x if residual is None else residual)
    helpers.assert_routing(idx, w, ridx, rw)
    return helpers.assert_close(out, ref)


# ----------------------------------------------------------------------------- tiny layer


@pytest.mark.parametrize("sched", SCHEDS)
def test_tiny_m1(tiny, sched):
    x = helpers.hidden_with_margin(tiny["router_w"], 1, synth.TINY.top_k, seed=0)
    _, out, idx, w = _run(synth.TINY, tiny, x, sched=sched)
    _check(synth.TINY, tiny, x, out, idx, w)


@pytest.mark.parametrize("sched", SCHEDS)
@pytest.mark.parametrize("m", [2, 6, 8])
def test_tiny_multi_row(tiny, sched, m):
    x = helpers.hidden_with_margin(tiny["router_w"], m, synth.TINY.top_k, seed=m, rho=0.5)
    _, out, idx, w = _run(synth.TINY, tiny, x, sched=sched, max_rows=8)
    _check(synth.TINY, tiny, x, out, idx, w)


def test_tiny_moe_part_alone(tiny):
    """Zero residual: the bf16 output is the MoE sum itself, so the tolerance
    bites on the expert arithmetic rather than on the residual's rounding."""
    x = helpers.hidden_with_margin(tiny["router_w"], 3, synth.TINY.top_k, seed=5, rho=0.5)
    r = torch.zeros_like(x)
    _, out, idx, w = _run(synth.TINY, tiny, x, residual=r)
    ref, _, _ = helpers.oracle_layer(synth.TINY, tiny, x, r)
    helpers.assert_close(out, ref)
    # tighter than the contract: bf16 rounding of the sum only
    g = helpers.f64(out)
    assert np.linalg.norm(g - ref) / np.linalg.norm(ref) < 3e-3


@pytest.mark.parametrize("m", [1, 4])
def test_schedules_bitwise_identical(tiny, m):
    x = helpers.hidden_with_margin(tiny["router_w"], m, synth.TINY.top_k, seed=9, rho=0.5)
    outs = [_run(synth.TINY, tiny, x, sched=s)[1] for s in SAME_ORDER]
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))


@pytest.mark.parametrize("m", [1, 3, 8])
def test_flat_kernel_repeatable_and_inplace(tiny, m):
    """The expert-range kernel: the same bits on every run (the block that finishes
    last sums its slots in a fixed order), in place as well."""
    x = helpers.hidden_with_margin(tiny["router_w"], m, synth.TINY.top_k, seed=40 + m, rho=0.5)
    mod = MoEDecodeLayer(synth.TINY, tiny, 8, sched="flat")
    assert mod.info(_lib.MOE_INFO_FLAT_ROWS) >> (m - 1) & 1
    xd = x.cuda()
    first = mod.run(xd, xd).clone()
    for _ in range(30):
        assert torch.equal(mod.run(xd, xd), first)
    buf = xd.clone()
    mod.run(buf, buf, buf)
    assert mod.status() == _lib.MOE_OK
    assert torch.equal(buf, first)
    ref, _, _ = helpers.oracle_layer(synth.TINY, tiny, x, x)
    helpers.assert_close(first.cpu(), ref)


def test_repeated_runs_and_inplace(tiny):
    x = helpers.hidden_with_margin(tiny["router_w"], 2, synth.TINY.top_k, seed=11)
    mod = MoEDecodeLayer(synth.TINY, tiny, 2)
    xd = x.cuda()
    first = mod.run(xd, xd).clone()
    for _ in range(50):
        again = mod.run(xd, xd)
        assert torch.equal(again, first)
    # in place: x, residual and out are one buffer
    buf = xd.clone()
    mod.run(buf, buf, buf)
    assert mod.status() == _lib.MOE_OK
    assert torch.equal(buf, first)


@pytest.mark.parametrize("sched", SCHEDS)
def test_zero_rows_give_zero(tiny, sched):
    """Zero rows: all logits tie at 0, so the tie rule (lower expert id first)
    decides the whole selection -- experts 0..k-1 in that order, equal weights --
    and silu(0) * 0 makes the output exactly zero."""
    x = torch.zeros((3, synth.TINY.hidden), dtype=torch.bfloat16)
    _, out, idx, w = _run(synth.TINY, tiny, x, sched=sched)
    assert torch.count_nonzero(out.float()) == 0
    np.testing.assert_allclose(w.numpy(), 1.0 / synth.TINY.top_k, rtol=0, atol=1e-7)
    assert idx.tolist() == [list(range(synth.TINY.top_k))] * 3
    _, ridx, _ = helpers.oracle_layer(synth.TINY, tiny, x, x)
    assert ridx.tolist() == idx.tolist()


def test_run_host_matches_device(tiny):
    x = helpers.hidden_with_margin(tiny["router_w"], 2, synth.TINY.top_k, seed=13)
    mod, out_dev, idx_dev, w_dev = _run(synth.TINY, tiny, x)
    out = torch.empty_like(x)
    idx = torch.empty((2, synth.TINY.top_k), dtype=torch.int32)
    w = torch.empty((2, synth.TINY.top_k), dtype=torch.float32)
    mod.run_host(x.contiguous(), x.contiguous(), out, idx, w)
    assert torch.equal(out, out_dev) and torch.equal(idx, idx_dev) and torch.equal(w, w_dev)


def test_graph_capture_replays(tiny):
    x = helpers.hidden_with_margin(tiny["router_w"], 2, synth.TINY.top_k, seed=17)
    for sched in SCHEDS:
        mod = MoEDecodeLayer(synth.TINY, tiny, 2, sched=sched)
        xd = x.cuda()
        out = torch.empty_like(xd)
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            mod.run(xd, xd, out, stream=s)  # warm-up outside capture
        torch.cuda.synchronize()
        ref = out.clone()
        out.zero_()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            mod.run(xd, xd, out, stream=s)
        for _ in range(3):
            out.zero_()
            g.replay()
            torch.cuda.synchronize()
            assert torch.equal(out, ref), sched
        assert mod.status() == _lib.MOE_OK


@pytest.mark.parametrize("cfg", [
    dict(hidden=256, inter=128, num_experts=16, top_k=16, num_shared=1),   # k = E
    dict(hidden=256, inter=128, num_experts=16, top_k=2, num_shared=0),    # no shared expert
    dict(hidden=256, inter=128, num_experts=16, top_k=4, num_shared=2),    # two shared experts
    dict(hidden=200, inter=64, num_experts=10, top_k=3, num_shared=1),     # ragged chunks
    dict(hidden=512, inter=256, num_experts=64, top_k=1, num_shared=1),    # top-1
    dict(hidden=1024, inter=768, num_experts=2, top_k=1, num_shared=1),    # E = 2, 96-thread groups
])
@pytest.mark.parametrize("m", [1, 5, 8])  # k = E = 16 at m = 8: 128 (row, expert) pairs, the most a launch has
def test_shapes(cfg, m):
    shape = synth.LayerShape(**cfg)
    layer = synth.make_layer(shape, seed=3, device="cuda")
    margin = 0.05 if cfg["top_k"] < cfg["num_experts"] else 0.0
    x = helpers.hidden_with_margin(layer["router_w"], m, shape.top_k, seed=21, rho=0.5, margin=margin)
    outs = {}
    for sched in SCHEDS:
        _, out, idx, w = _run(shape, layer, x, sched=sched, max_rows=8)
        if cfg["top_k"] < cfg["num_experts"]:
            _check(shape, layer, x, out, idx, w)
        else:
            ref, _, _ = helpers.oracle_layer(shape, layer, x, x)
            helpers.assert_close(out, ref)
        outs[sched] = out
    for s in SAME_ORDER[1:]:
        assert torch.equal(outs[SAME_ORDER[0]], outs[s]), s


# ----------------------------------------------------------------------------- bias-corrected sigmoid rule


def _sigmoid_case(shape, layer, m, seed, sched, bias, routed_scale=2.5, max_rows=8):
    lay = dict(layer, router_bias=bias)
    x = helpers.hidden_with_margin(layer["router_w"], m, shape.top_k, seed=seed, rho=0.5, margin=1e-3,
                                   score=1, bias=bias)
    mod = MoEDecodeLayer(shape, lay, max(m, max_rows), sched=sched, routed_scale=routed_scale, score=1)
    xd = x.cuda()
    out = torch.empty_like(xd)
    idx = torch.empty((m, shape.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((m, shape.top_k), dtype=torch.float32, device="cuda")
    mod.run(xd, xd, out, idx, w)
    assert mod.status() == _lib.MOE_OK
    ref, ridx, rw = helpers.oracle_layer(shape, lay, x, x, routed_scale=routed_scale, score=1, bias=bias)
    helpers.assert_routing(idx.cpu(), w.cpu(), ridx, rw, by_weight=False)
    helpers.assert_close(out.cpu(), ref)
    return x, ridx


@pytest.mark.parametrize("sched", SCHEDS)
@pytest.mark.parametrize("m", [1, 5])
def test_tiny_sigmoid_bias(tiny, sched, m):
    """Selection by sigmoid(logit) + bias, weights sigmoid(logit) / sum, routed
    scale 2.5; the bias is large enough that it changes some row's choice."""
    bias = synth.router_bias(synth.TINY.num_experts, seed=3, device="cuda", std=0.2)
    x, ridx = _sigmoid_case(synth.TINY, tiny, m, 90 + m, sched, bias)
    if m == 5:
        plain = cpp.route(helpers.f64(x), helpers.bits(tiny["router_w"]), synth.TINY.top_k, 1,
                          np.zeros(synth.TINY.num_experts))[1]
        assert any(sorted(a) != sorted(b) for a, b in zip(plain.tolist(), ridx.tolist()))


@pytest.mark.parametrize("sched", ["persistent", "flat", "pdl_chain"])
@pytest.mark.parametrize("m", [1, 6])
def test_ling_sigmoid_bias(ling, sched, m):
    bias = synth.router_bias(synth.LING.num_experts, seed=5, device="cuda")
    _sigmoid_case(synth.LING, ling, m, 120 + m, sched, bias, max_rows=m)


# ----------------------------------------------------------------------------- Ling-shaped layer


@pytest.mark.parametrize("sched", SCHEDS)
def test_ling_m1(ling, sched):
    x = helpers.hidden_with_margin(ling["router_w"], 1, synth.LING.top_k, seed=0)
    _, out, idx, w = _run(synth.LING, ling, x, sched=sched)
    _check(synth.LING, ling, x, out, idx, w)


@pytest.mark.parametrize("sched", ["persistent", "phased", "interleaved", "flat", "pdl_chain"])
def test_ling_m6_correlated(ling, sched):
    x = helpers.hidden_with_margin(ling["router_w"], 6, synth.LING.top_k, seed=1, rho=0.5)
    _, out, idx, w = _run(synth.LING, ling, x, sched=sched)
    _check(synth.LING, ling, x, out, idx, w)
    distinct = len(set(idx.flatten().tolist()))
    assert 8 <= distinct <= 48


@pytest.mark.parametrize("sched", ["persistent", "flat", "pdl_chain"])
@pytest.mark.parametrize("m", [9, 16])
def test_wide_verify_rows(tiny, ling, sched, m):
    """More than 8 rows (the 16-token verify batch): row groups of at most 8 run
    one after another; every row is checked against the oracle, in place too."""
    for shape, layer in ((synth.TINY, tiny), (synth.LING, ling)):
        x = helpers.hidden_with_margin(layer["router_w"], m, shape.top_k, seed=130 + m, rho=0.5)
        _, out, idx, w = _run(shape, layer, x, sched=sched)
        _check(shape, layer, x, out, idx, w)
        mod = MoEDecodeLayer(shape, layer, m, sched=sched)
        buf = x.cuda()
        mod.run(buf, buf, buf)
        assert mod.status() == _lib.MOE_OK
        assert torch.equal(buf.cpu(), out)


def test_ling_interleave_modes(ling):
    """The Ling-shaped layer fits the slot-interleaved layout at M = 1 and M = 6:
    the default mode (1) uses it for single-row runs, "interleaved" forces it (2),
    "phased" switches it off (0)."""
    for m in (1, 6):
        assert MoEDecodeLayer(synth.LING, ling, m).info(_lib.MOE_OPT_INTERLEAVE) == 1
        assert MoEDecodeLayer(synth.LING, ling, m, sched="interleaved").info(_lib.MOE_OPT_INTERLEAVE) == 2
        assert MoEDecodeLayer(synth.LING, ling, m, sched="phased").info(_lib.MOE_OPT_INTERLEAVE) == 0
    dflt = MoEDecodeLayer(synth.LING, ling, 6)
    flat_rows = dflt.info(_lib.MOE_INFO_FLAT_ROWS)
    assert dflt.info(_lib.MOE_INFO_INTERLEAVED_ROWS) == 0b1 & ~flat_rows
    assert MoEDecodeLayer(synth.LING, ling, 6, sched="interleaved").info(_lib.MOE_INFO_INTERLEAVED_ROWS) == 0b111111
    assert MoEDecodeLayer(synth.LING, ling, 6, sched="interleaved").info(_lib.MOE_INFO_FLAT_ROWS) == 0
    assert MoEDecodeLayer(synth.LING, ling, 6, sched="phased").info(_lib.MOE_INFO_INTERLEAVED_ROWS) == 0
    assert MoEDecodeLayer(synth.LING, ling, 6, sched="phased").info(_lib.MOE_INFO_FLAT_ROWS) == 0
    fl = MoEDecodeLayer(synth.LING, ling, 6, sched="flat")
    assert fl.info(_lib.MOE_INFO_FLAT_ROWS) == 0b111111 and fl.info(_lib.MOE_INFO_INTERLEAVED_ROWS) == 0
    assert fl.info(_lib.MOE_OPT_FLAT) == 2
    assert MoEDecodeLayer(synth.LING, ling, 1).info(_lib.MOE_INFO_THREADS) == 480
    assert MoEDecodeLayer(synth.LING, ling, 1, sched="phased").info(_lib.MOE_INFO_THREADS) == 416


@pytest.mark.parametrize("m", [1, 6])
def test_ling_flat_inplace_repeat(ling, m):
    """The expert-range kernel at full Ling size, in place (x, residual and output
    one buffer), run twice on fresh copies: identical bits, within the oracle's
    tolerance."""
    x = helpers.hidden_with_margin(ling["router_w"], m, synth.LING.top_k, seed=70 + m, rho=0.5)
    mod = MoEDecodeLayer(synth.LING, ling, m, sched="flat")
    outs = []
    for _ in range(2):
        buf = x.cuda()
        mod.run(buf, buf, buf)
        assert mod.status() == _lib.MOE_OK
        outs.append(buf.cpu())
    assert torch.equal(outs[0], outs[1])
    ref, _, _ = helpers.oracle_layer(synth.LING, ling, x, x)
    helpers.assert_close(outs[0], ref)


def test_ling_moe_part_alone(ling):
    x = helpers.hidden_with_margin(ling["router_w"], 2, synth.LING.top_k, seed=4)
    r = torch.zeros_like(x)
    _, out, idx, w = _run(synth.LING, ling, x, residual=r)
    ref, _, _ = helpers.oracle_layer(synth.LING, ling, x, r)
    helpers.assert_close(out, ref)


@pytest.mark.parametrize("slots", [2, 3, 5])
@pytest.mark.parametrize("sched", SCHEDS)
def test_small_ring_wraps(tiny, slots, sched):
    """Few ring slots force every phase to wrap the shared-memory ring many times;
    results must not change by a bit."""
    x = helpers.hidden_with_margin(tiny["router_w"], 6, synth.TINY.top_k, seed=31, rho=0.5)
    _, ref_out, _, _ = _run(synth.TINY, tiny, x, sched=sched, max_rows=8)
    mod = MoEDecodeLayer(synth.TINY, tiny, 8, sched=sched)
    mod.set_option(_lib.MOE_OPT_RING_SLOTS, slots)
    assert mod.info(_lib.MOE_OPT_RING_SLOTS) == (max(slots, 3) if sched == "flat" else slots)
    xd = x.cuda()
    for _ in range(3):
        out = mod.run(xd, xd)
        assert mod.status() == _lib.MOE_OK
        assert torch.equal(out.cpu(), ref_out)
