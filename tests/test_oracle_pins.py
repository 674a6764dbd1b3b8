"""Pins of the CPU oracle against facts fixed outside the oracle itself.

Each pin is something the pages or the mathematics decide: a hand-worked example,
a textbook reduction (uniform routing over all experts is a dense mean of SwiGLU
MLPs, written here with plain Python loops), invariants (weights sum to one,
joint permutation of experts, zero in -> zero out), closed forms (softmax over
all experts then top-k then renormalise; the bias-corrected sigmoid rule worked
by hand), brute force on tiny inputs, and library routines for the number
formats.

Every pin runs against both restatements of the oracle: the C++ oracle proper
(``oracle/moe_oracle_ref.cpp``) and the numpy one. The two are also cross-checked
on random layers in every storage format. Planted mistakes -- monkeypatched into
the numpy restatement, compiled into the C++ one (``-DORACLE_MUTANT=n``) -- must
each trip at least one pin.
"""

import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import cpp, moe_oracle, nvfp4
from moe_decode_layer_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


class CppOracle:
    """The C++ oracle (optionally a planted-mistake build) behind the numpy API."""

    def __init__(self, mutant: int = 0):
        self.lib = cpp.load(mutant)

    def moe_layer(self, *a, **k):
        return cpp.moe_layer(*a, lib=self.lib, **k)

    def router_logits(self, x, rw):
        return cpp.router_logits(x, rw, lib=self.lib)

    def topk_renorm(self, l, k):
        return cpp.topk_renorm(l, k, lib=self.lib)

    def select(self, l, k, score=0, bias=None):
        return cpp.select(l, k, score, bias, lib=self.lib)

    def silu(self, g):
        return cpp.silu(g, lib=self.lib)

    def bf16_bits_to_f64(self, b):
        return cpp.bf16_bits_to_f64(b, lib=self.lib)

    def f64_to_bf16_bits(self, v):
        return cpp.f64_to_bf16_bits(v, lib=self.lib)

    def e2m1_value(self, c):
        return cpp.e2m1_value(c, lib=self.lib)

    def e4m3_value(self, b):
        return cpp.e4m3_value(b, lib=self.lib)


IMPLS = {"cpp": lambda: CppOracle(), "numpy": lambda: oracle}


@pytest.fixture(params=sorted(IMPLS))
def o(request):
    return IMPLS[request.param]()


# ---------------------------------------------------------------------------
# independent helpers (plain Python, no numpy linear algebra, no oracle code)
# ---------------------------------------------------------------------------


def _py_dense_swiglu(x, gate, up, down):
    """W2 (silu(Wg x) * (Wu x)) with explicit loops and math.exp."""
    inter = len(gate)
    h = []
    for j in range(inter):
        g = sum(gate[j][i] * x[i] for i in range(len(x)))
        u = sum(up[j][i] * x[i] for i in range(len(x)))
        h.append(g * (1.0 / (1.0 + math.exp(-g))) * u)
    return [sum(down[o][j] * h[j] for j in range(inter)) for o in range(len(down))]


def _sig(v):
    return 1.0 / (1.0 + math.exp(-v))


def _example_experts(ex):
    return [(np.array([e["gate"], e["up"]], float), np.array(e["down"], float))
            for e in ex["experts"]]


def _run_example(o, k, with_shared, **kw):
    ex = _golden("two_expert_example.json")
    experts = _example_experts(ex)
    shared = []
    if with_shared:
        s = ex["shared"]
        shared = [(np.array([s["gate"], s["up"]], float), np.array(s["down"], float))]
    out, idx, w = o.moe_layer(np.array([ex["x"]]), np.array([ex["residual"]]),
                              np.array(ex["router_w"], float), lambda e: experts[e], shared, k, **kw)
    return ex, out[0], idx[0], w[0]


def _rand_layer(rng, h=6, i=3, e=5, s=1):
    return (rng.standard_normal((e, h)),
            [(rng.standard_normal((2 * i, h)), rng.standard_normal((h, i))) for _ in range(e)],
            [(rng.standard_normal((2 * i, h)), rng.standard_normal((h, i))) for _ in range(s)])


# ---------------------------------------------------------------------------
# the pins, each a function of the implementation so the planted-mistake
# tests can rerun them
# ---------------------------------------------------------------------------


def pin_two_expert_k2(o):
    ex, out, idx, w = _run_example(o, 2, False)
    np.testing.assert_allclose(o.router_logits(np.array([ex["x"]]), np.array(ex["router_w"], float))[0],
                               ex["logits"], rtol=0, atol=1e-15)
    assert list(idx) == ex["k2"]["idx"]
    np.testing.assert_allclose(w, ex["k2"]["w"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(out, ex["k2"]["out"], rtol=0, atol=1e-13)


def pin_two_expert_k1(o):
    ex, out, idx, w = _run_example(o, 1, False)
    assert list(idx) == ex["k1"]["idx"]
    np.testing.assert_allclose(w, ex["k1"]["w"], rtol=0, atol=1e-15)
    np.testing.assert_allclose(out, ex["k1"]["out"], rtol=0, atol=1e-13)


def pin_two_expert_shared(o):
    ex, out, _, _ = _run_example(o, 2, True)
    np.testing.assert_allclose(out, ex["k2_shared"]["out"], rtol=0, atol=1e-13)


def pin_routed_scale_scales_only_the_routed_sum(o):
    """The two-expert example with a shared expert and routed_scale 2.5, worked by
    hand: out = r + 2.5 * (w0 h0 e_0 + w1 h1 e_1) + s (1, 1)."""
    ex, out, _, _ = _run_example(o, 2, True, routed_scale=2.5)
    w0, w1 = 1 / (1 + math.e), math.e / (1 + math.e)
    h0, h1 = 2 * _sig(1.0), 2 * _sig(2.0)  # silu(1) * 2, silu(2) * 1
    s = -3 * _sig(3.0)
    np.testing.assert_allclose(out, [1 + 2.5 * w0 * h0 + s, 2 + 2.5 * w1 * h1 + s], rtol=0, atol=1e-13)


def pin_sigmoid_bias_two_expert(o):
    """Bias-corrected sigmoid rule on the two-expert example, worked by hand.

    Logits [1, 2]; bias [0.3, 0]: keys sig(1) + 0.3 = 1.031 > sig(2) = 0.881, so
    with k = 1 the bias flips the choice to expert 0 with weight 1, and with k = 2
    the order is [0, 1] with weights sig(l_j) / (sig(1) + sig(2)) -- the bias does
    not enter the weights.
    """
    bias = np.array([0.3, 0.0])
    ex, out, idx, w = _run_example(o, 1, False, score=1, bias=bias, routed_scale=2.5)
    h0, h1 = 2 * _sig(1.0), 2 * _sig(2.0)  # silu(1) * 2, silu(2) * 1
    assert list(idx) == [0]
    np.testing.assert_allclose(w, [1.0], rtol=0, atol=1e-15)
    np.testing.assert_allclose(out, [1 + 2.5 * h0, 2.0], rtol=0, atol=1e-13)
    ex, out, idx, w = _run_example(o, 2, False, score=1, bias=bias)
    z = _sig(1.0) + _sig(2.0)
    assert list(idx) == [0, 1]
    np.testing.assert_allclose(w, [_sig(1.0) / z, _sig(2.0) / z], rtol=0, atol=1e-15)
    np.testing.assert_allclose(out, [1 + _sig(1.0) / z * h0, 2 + _sig(2.0) / z * h1], rtol=0, atol=1e-13)


def pin_sigmoid_bias_invariants(o):
    """Zero bias selects what softmax selects (both monotone in the logit); a
    common shift of every bias changes nothing; a bias far above the others forces
    that expert in; the weights sum to one."""
    rng = np.random.default_rng(19)
    for trial in range(30):
        e, k = 24, 1 + trial % 8
        logits = rng.standard_normal(e) * 2
        i0, _ = o.select(logits, k, 1, np.zeros(e))
        i1, _ = o.topk_renorm(logits, k)
        assert i0.tolist() == i1.tolist()
        bias = rng.standard_normal(e) * 0.1
        a_idx, a_w = o.select(logits, k, 1, bias)
        b_idx, b_w = o.select(logits, k, 1, bias + 0.75)
        assert a_idx.tolist() == b_idx.tolist()
        np.testing.assert_allclose(a_w, b_w, rtol=0, atol=1e-15)
        assert abs(a_w.sum() - 1.0) < 1e-12
        low = int(np.argmin(logits))
        forced = bias.copy()
        forced[low] = 5.0
        f_idx, _ = o.select(logits, k, 1, forced)
        assert f_idx[0] == low


def pin_sigmoid_bias_brute_force_with_ties(o):
    """Tiny E with exactly tied keys: the set beats every other k-subset in
    (key, lower id) order, keys computed here with math.exp."""
    rng = np.random.default_rng(23)
    for _ in range(40):
        e, k = 6, int(rng.integers(1, 6))
        logits = rng.integers(-2, 3, e).astype(float)
        bias = np.zeros(e)
        keys = [_sig(v) for v in logits]
        best = None
        for sub in itertools.combinations(range(e), k):
            key = sorted(((-keys[i], i) for i in sub))
            if best is None or key < best:
                best = key
        idx, w = o.select(logits, k, 1, bias)
        assert idx.tolist() == [i for _, i in best]
        z = sum(keys[i] for i in idx)
        np.testing.assert_allclose(w, [keys[i] / z for i in idx], rtol=1e-14, atol=0)


def pin_uniform_routing_is_dense_mean(o):
    """k = E and a zero router: every expert gets weight 1/E (textbook dense MoE)."""
    rng = np.random.default_rng(11)
    hdim, e = 6, 4
    _, experts, shared = _rand_layer(rng, h=hdim, i=3, e=e, s=1)
    x = rng.standard_normal((2, hdim))
    r = rng.standard_normal((2, hdim))
    out, idx, w = o.moe_layer(x, r, np.zeros((e, hdim)), lambda j: experts[j], shared, e)
    for m in range(2):
        ref = list(r[m])
        xs = list(x[m])
        for w13, w2 in experts:
            y = _py_dense_swiglu(xs, w13[:3].tolist(), w13[3:].tolist(), w2.tolist())
            ref = [a + b / e for a, b in zip(ref, y)]
        w13, w2 = shared[0]
        y = _py_dense_swiglu(xs, w13[:3].tolist(), w13[3:].tolist(), w2.tolist())
        ref = [a + b for a, b in zip(ref, y)]
        np.testing.assert_allclose(out[m], ref, rtol=1e-12, atol=1e-12)
        assert sorted(idx[m].tolist()) == list(range(e))
        np.testing.assert_allclose(w[m], np.full(e, 1.0 / e), rtol=0, atol=1e-15)


def pin_weights_sum_to_one(o):
    rng = np.random.default_rng(3)
    for _ in range(50):
        logits = rng.standard_normal(37) * 3
        _, w = o.topk_renorm(logits, 5)
        assert abs(w.sum() - 1.0) < 1e-12
        assert np.all(w > 0) and np.all(np.diff(w) <= 0)


def pin_softmax_topk_renorm_closed_form(o):
    """Full softmax over E, keep the top k, renormalise: plain Python."""
    rng = np.random.default_rng(5)
    for trial in range(30):
        e, k = 12, 1 + trial % 6
        logits = (rng.standard_normal(e) * 2).tolist()
        z = sum(math.exp(v) for v in logits)
        p = [math.exp(v) / z for v in logits]
        order = sorted(range(e), key=lambda i: (-logits[i], i))[:k]
        ref_w = [p[i] / sum(p[j] for j in order) for i in order]
        idx, w = o.topk_renorm(np.array(logits), k)
        assert idx.tolist() == order
        np.testing.assert_allclose(w, ref_w, rtol=1e-12, atol=0)


def pin_topk_brute_force_with_ties(o):
    """Tiny E with many ties: the chosen set beats every other k-subset in
    (logit, lower id) order, found by enumerating all subsets."""
    rng = np.random.default_rng(7)
    for _ in range(40):
        e, k = 6, int(rng.integers(1, 6))
        logits = rng.integers(-2, 3, e).astype(float)
        best = None
        for sub in itertools.combinations(range(e), k):
            key = sorted(((-logits[i], i) for i in sub))
            if best is None or key < best:
                best = key
        idx, _ = o.topk_renorm(logits, k)
        assert idx.tolist() == [i for _, i in best]


def pin_joint_permutation(o):
    rng = np.random.default_rng(13)
    router, experts, shared = _rand_layer(rng, h=8, i=4, e=7, s=1)
    x = rng.standard_normal((3, 8))
    r = rng.standard_normal((3, 8))
    perm = rng.permutation(7)  # new expert p holds old expert perm[p]
    out_a, idx_a, w_a = o.moe_layer(x, r, router, lambda j: experts[j], shared, 3)
    out_b, idx_b, w_b = o.moe_layer(x, r, router[perm], lambda j: experts[perm[j]], shared, 3)
    np.testing.assert_allclose(out_a, out_b, rtol=1e-13, atol=1e-13)
    np.testing.assert_array_equal(idx_a, perm[idx_b])
    np.testing.assert_allclose(w_a, w_b, rtol=1e-14, atol=1e-15)


def pin_zero_row_zero_output(o):
    rng = np.random.default_rng(17)
    router, experts, shared = _rand_layer(rng)
    out, _, _ = o.moe_layer(np.zeros((2, 6)), np.zeros((2, 6)), router, lambda j: experts[j], shared, 2)
    assert np.all(out == 0.0)


def pin_silu_identities(o):
    g = np.linspace(-30, 30, 601)
    s = o.silu(g)
    np.testing.assert_allclose(s - o.silu(-g), g, rtol=0, atol=1e-12)  # g*sig(g) + g*sig(-g) = g
    assert o.silu(np.array([0.0]))[0] == 0.0
    assert abs(o.silu(np.array([800.0]))[0] - 800.0) < 1e-9
    assert o.silu(np.array([-800.0]))[0] == 0.0
    np.testing.assert_allclose(o.silu(np.array([1.0]))[0] * (1 + math.exp(-1)), 1.0, rtol=1e-15)


def pin_bf16_rounding(o):
    """Round to nearest, ties to even, checked against torch's float32 -> bf16
    conversion and hand-picked halfway cases."""
    rng = np.random.default_rng(0)
    v32 = (rng.standard_normal(20000) * np.exp(rng.uniform(-20, 20, 20000))).astype(np.float32)
    ref = torch.from_numpy(v32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(o.f64_to_bf16_bits(v32.astype(np.float64)), ref)
    vals = np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 2 ** -130 * 1.5])
    got = o.bf16_bits_to_f64(o.f64_to_bf16_bits(vals))
    np.testing.assert_array_equal(got, [1.0, 1 + 2 ** -6, -1.0, 2 ** -130 * 1.5])


def pin_number_formats(o):
    """e2m1 against the published table, e4m3 against torch's float8_e4m3fn."""
    ref = _golden("nvfp4_codes.json")["e2m1"]
    assert [o.e2m1_value(c) for c in range(16)] == ref
    bits = np.arange(256, dtype=np.uint8)
    ref8 = torch.from_numpy(bits).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([o.e4m3_value(b) for b in range(256)])
    assert (np.isnan(ref8) == np.isnan(got)).all()
    np.testing.assert_array_equal(got[~np.isnan(ref8)], ref8[~np.isnan(ref8)])


ALL_PINS = [pin_two_expert_k2, pin_two_expert_k1, pin_two_expert_shared,
            pin_routed_scale_scales_only_the_routed_sum, pin_sigmoid_bias_two_expert,
            pin_sigmoid_bias_invariants, pin_sigmoid_bias_brute_force_with_ties,
            pin_uniform_routing_is_dense_mean, pin_weights_sum_to_one,
            pin_softmax_topk_renorm_closed_form, pin_topk_brute_force_with_ties,
            pin_joint_permutation, pin_zero_row_zero_output, pin_silu_identities,
            pin_bf16_rounding, pin_number_formats]


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin, o):
    pin(o)


# ---------------------------------------------------------------------------
# the C++ oracle: NVFP4 storage, cross-check with the numpy restatement,
# independence of the thread count
# ---------------------------------------------------------------------------


def _nvfp4_expert(rng, hdim, inter):
    w13 = torch.from_numpy(rng.standard_normal((2 * inter, hdim)).astype(np.float32)) * 0.05
    w2 = torch.from_numpy(rng.standard_normal((hdim, inter)).astype(np.float32)) * 0.05
    qg, sg, tg = synth.quantize_nvfp4(w13[:inter])
    qu, su, tu = synth.quantize_nvfp4(w13[inter:])
    q2, s2, t2 = synth.quantize_nvfp4(w2)
    return cpp.NVFP4Expert(torch.cat([qg, qu]).numpy(), torch.cat([sg, su]).numpy(),
                           np.array([float(tg), float(tu)], np.float32), q2.numpy(), s2.numpy(), np.float32(t2))


def _nvfp4_as_f64(ex):
    i = ex.q13.shape[0] // 2
    gate = nvfp4.dequant_nvfp4_rows(ex.q13[:i], ex.s13[:i], float(ex.gs13[0]))
    up = nvfp4.dequant_nvfp4_rows(ex.q13[i:], ex.s13[i:], float(ex.gs13[1]))
    return np.vstack([gate, up]), nvfp4.dequant_nvfp4_rows(ex.q2, ex.s2, float(ex.gs2))


def test_nvfp4_layout_by_hand_cpp():
    """A one-expert NVFP4 layer whose codes are placed by hand equals the same
    layer with the hand-decoded float64 weights (bytes 0x21 -> 0.5, 1.0; 0xF8 ->
    -0.0, -6.0; scale 0x40 = 2.0; tensor scales 0.5 and 0.25)."""
    hdim, inter = 16, 16
    q13 = np.zeros((2 * inter, hdim // 2), np.uint8)
    q13[:, 0], q13[:, 1] = 0x21, 0xF8
    s13 = np.full((2 * inter, 1), 0x40, np.uint8)
    q2 = np.zeros((hdim, inter // 2), np.uint8)
    q2[:, 0] = 0x21
    s2 = np.full((hdim, 1), 0x40, np.uint8)
    ex = cpp.NVFP4Expert(q13, s13, np.array([0.5, 0.25], np.float32), q2, s2, np.float32(0.5))
    row = np.zeros(hdim)
    row[:4] = [0.5, 1.0, -0.0, -6.0]
    w13 = np.vstack([np.tile(row * 2.0 * 0.5, (inter, 1)), np.tile(row * 2.0 * 0.25, (inter, 1))])
    drow = np.zeros(inter)
    drow[:2] = [0.5 * 2.0 * 0.5, 1.0 * 2.0 * 0.5]
    w2 = np.tile(drow, (hdim, 1))
    x = np.linspace(-1, 1, hdim)[None, :]
    router = np.ones((1, hdim))
    a = cpp.moe_layer(x, x, router, lambda e: ex, [], 1)
    b = cpp.moe_layer(x, x, router, lambda e: (w13, w2), [], 1)
    np.testing.assert_array_equal(a[0], b[0])


def _fp8_expert(rng, hdim, inter):
    w13 = torch.from_numpy(rng.standard_normal((2 * inter, hdim)).astype(np.float32)) * 0.05
    w2 = torch.from_numpy(rng.standard_normal((hdim, inter)).astype(np.float32)) * 0.05
    q13, s13 = synth.quantize_fp8_block(w13)
    q2, s2 = synth.quantize_fp8_block(w2)
    return cpp.FP8Expert(q13.numpy(), s13.numpy(), q2.numpy(), s2.numpy())


def _fp8_as_f64(ex):
    return nvfp4.dequant_fp8_block(ex.q13, ex.s13), nvfp4.dequant_fp8_block(ex.q2, ex.s2)


def test_fp8_layout_by_hand_cpp():
    """A one-expert FP8 layer whose codes and block scales are placed by hand equals
    the same layer with the hand-decoded float64 weights: e4m3 0x38 = 1.0, 0xC4 =
    -3.0 (sign, exponent 8, mantissa 4: -1.5 * 2); each 128 x 128 tile of the
    [256, 256] gate/up matrix and the [128, 256] down matrix has its own scale."""
    hdim, inter = 128, 128
    q13 = np.zeros((2 * inter, hdim), np.uint8)
    q13[:, 0], q13[:, 5] = 0x38, 0xC4
    s13 = np.array([[0.5], [0.25]], np.float32)  # gate rows, up rows
    q2 = np.zeros((hdim, inter), np.uint8)
    q2[:, 3] = 0x38
    s2 = np.array([[2.0]], np.float32)
    ex = cpp.FP8Expert(q13, s13, q2, s2)
    row = np.zeros(hdim)
    row[0], row[5] = 1.0, -3.0
    w13 = np.vstack([np.tile(row * 0.5, (inter, 1)), np.tile(row * 0.25, (inter, 1))])
    w2 = np.zeros((hdim, inter))
    w2[:, 3] = 2.0
    x = np.linspace(-1, 1, hdim)[None, :]
    router = np.ones((1, hdim))
    a = cpp.moe_layer(x, x, router, lambda e: ex, [], 1)
    b = cpp.moe_layer(x, x, router, lambda e: (w13, w2), [], 1)
    np.testing.assert_array_equal(a[0], b[0])
    # a rectangular scale grid: down [256, 128] with scales [2, 1]
    q2b = np.zeros((256, 128), np.uint8)
    q2b[:, 1] = 0x38
    s2b = np.array([[3.0], [5.0]], np.float32)
    w2b = np.zeros((256, 128))
    w2b[:128, 1], w2b[128:, 1] = 3.0, 5.0
    q13b = np.zeros((256, 256), np.uint8)
    q13b[:, 7] = 0x38
    s13b = np.array([[1.0, 2.0], [4.0, 8.0]], np.float32)
    w13b = np.zeros((256, 256))
    w13b[:128, 7], w13b[128:, 7] = 1.0, 4.0
    x2 = np.linspace(-1, 1, 256)[None, :]
    a = cpp.moe_layer(x2, x2, np.ones((1, 256)), lambda e: cpp.FP8Expert(q13b, s13b, q2b, s2b), [], 1)
    b = cpp.moe_layer(x2, x2, np.ones((1, 256)), lambda e: (w13b, w2b), [], 1)
    np.testing.assert_array_equal(a[0], b[0])


def test_fp8_quantiser_roundtrip():
    """The synthetic FP8 quantiser and the oracle's decoder are independent: a tile
    whose values are e4m3 grid points times amax / 448 comes back exactly, and the
    tile maximum maps to code 448 (0x7E)."""
    grid = np.array([nvfp4.e4m3_value(b) for b in range(0x7F)], np.float64)  # 0 .. 448
    rng = np.random.default_rng(4)
    vals = rng.choice(grid, size=(128, 128)) * rng.choice([-1.0, 1.0], size=(128, 128))
    vals[0, 0] = 448.0
    w = torch.from_numpy((vals * 2.0 ** -9).astype(np.float32))  # scale 2^-9: exact
    q, sc = synth.quantize_fp8_block(w)
    assert float(sc[0, 0]) == 2.0 ** -9 and int(q[0, 0]) == 0x7E
    np.testing.assert_array_equal(nvfp4.dequant_fp8_block(q.numpy(), sc.numpy()), vals * 2.0 ** -9)


@pytest.mark.parametrize("fmt", ["f64", "bf16", "nvfp4", "fp8"])
@pytest.mark.parametrize("score", [0, 1])
def test_cpp_matches_numpy_restatement(fmt, score):
    rng = np.random.default_rng(41 + score)
    hdim, inter, e, k, s, m = 64, 32, 12, 3, 1, 4
    router = rng.standard_normal((e, hdim)) * 0.2
    bias = rng.standard_normal(e) * 0.05 if score else None
    if fmt == "nvfp4":
        raw = [_nvfp4_expert(rng, hdim, inter) for _ in range(e + s)]
        f64 = [_nvfp4_as_f64(w) for w in raw]
    elif fmt == "fp8":
        hdim, inter = 256, 128
        router = rng.standard_normal((e, hdim)) * 0.2
        raw = [_fp8_expert(rng, hdim, inter) for _ in range(e + s)]
        f64 = [_fp8_as_f64(w) for w in raw]
    else:
        f64 = [(rng.standard_normal((2 * inter, hdim)) * 0.2, rng.standard_normal((hdim, inter)) * 0.2)
               for _ in range(e + s)]
        if fmt == "bf16":
            raw = [(oracle.f64_to_bf16_bits(a), oracle.f64_to_bf16_bits(b)) for a, b in f64]
            f64 = [(oracle.bf16_bits_to_f64(a), oracle.bf16_bits_to_f64(b)) for a, b in raw]
            router_bits = oracle.f64_to_bf16_bits(router)
            router = oracle.bf16_bits_to_f64(router_bits)
        else:
            raw = f64
    x = rng.standard_normal((m, hdim))
    r = rng.standard_normal((m, hdim))
    ref = moe_oracle.moe_layer(x, r, router, lambda j: f64[j], f64[e:], k, 1.5, score, bias)
    got = cpp.moe_layer(x, r, router_bits if fmt == "bf16" else router, lambda j: raw[j], raw[e:], k, 1.5,
                        score, bias)
    np.testing.assert_array_equal(got[1], ref[1])
    np.testing.assert_allclose(got[2], ref[2], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(got[0], ref[0], rtol=1e-12, atol=1e-12)


def test_cpp_result_does_not_depend_on_thread_count():
    rng = np.random.default_rng(5)
    router, experts, shared = _rand_layer(rng, h=96, i=40, e=9, s=2)
    x = rng.standard_normal((3, 96))
    outs = [cpp.moe_layer(x, x, router, lambda j: experts[j], shared, 4, threads=t)[0] for t in (1, 3, 7)]
    for a in outs[1:]:
        np.testing.assert_array_equal(a, outs[0])


def test_cpp_reports_missing_experts():
    rng = np.random.default_rng(6)
    router, experts, shared = _rand_layer(rng)
    table = cpp._ExpertTable(5, {})
    shape = cpp._Shape(6, 3, 5, 2, 0, 1, 0, 0, 1.0, 1)
    x = rng.standard_normal((1, 6))
    out, idx, w = np.empty((1, 6)), np.empty((1, 2), np.int64), np.empty((1, 2))
    import ctypes
    st = cpp.load().moe_oracle_layer(ctypes.byref(shape), cpp._ptr(x), cpp._ptr(x), cpp._ptr(router), None,
                                     ctypes.byref(table.struct), ctypes.byref(table.struct), cpp._ptr(out),
                                     cpp._ptr(idx), cpp._ptr(w), None)
    assert st == 2  # a selected expert's weights are missing


def test_stack_input_matches_numpy_restatement():
    rng = np.random.default_rng(8)
    h = oracle.f64_to_bf16_bits(rng.standard_normal((6, 256)) * 3)
    np.testing.assert_array_equal(cpp.stack_layer_input(h), oracle.stack_layer_input(h))


# ---------------------------------------------------------------------------
# planted mistakes: every plausible slip must trip at least one pin
# ---------------------------------------------------------------------------


def _mutant_swap_gate_up(x_row, w13, w2):
    i = w13.shape[0] // 2
    return w2 @ (moe_oracle.silu(w13[i:] @ x_row) * (w13[:i] @ x_row))


def _mutant_sigmoid_not_silu(g):
    return 1.0 / (1.0 + np.exp(-np.asarray(g, float)))


def _mutant_silu_sign(g):
    g = np.asarray(g, float)
    return g / (1.0 + np.exp(g))


def _mutant_no_renorm(logits_row, k):
    l = np.asarray(logits_row, float)
    idx = np.argsort(-l, kind="stable")[:k]
    p = np.exp(l - l.max())
    return idx, (p / p.sum())[idx]


def _mutant_ties_to_higher(logits_row, k):
    l = np.asarray(logits_row, float)
    order = sorted(range(l.size), key=lambda i: (-l[i], -i))[:k]
    e = np.exp(l[order] - l[order].max())
    return np.array(order), e / e.sum()


def _mutant_router_rows_reversed(x, router_w):
    return np.asarray(x, float) @ np.asarray(router_w, float)[::-1].T


def _mutant_bottom_k(logits_row, k):
    l = np.asarray(logits_row, float)
    idx = np.argsort(l, kind="stable")[:k]  # smallest instead of largest
    e = np.exp(l[idx] - l[idx].max())
    return idx, e / e.sum()


def _mutant_bias_in_weights(logits_row, k, bias):
    l = np.asarray(logits_row, float)
    key = 1.0 / (1.0 + np.exp(-l)) + np.asarray(bias, float)
    idx = np.argsort(-key, kind="stable")[:k]
    return idx, key[idx] / key[idx].sum()


MUTANTS = {
    "swap_gate_up": ("expert_swiglu", _mutant_swap_gate_up),
    "sigmoid_not_silu": ("silu", _mutant_sigmoid_not_silu),
    "silu_sign": ("silu", _mutant_silu_sign),
    "no_renorm": ("topk_renorm", _mutant_no_renorm),
    "ties_to_higher_id": ("topk_renorm", _mutant_ties_to_higher),
    "router_rows_reversed": ("router_logits", _mutant_router_rows_reversed),
    "bottom_k": ("topk_renorm", _mutant_bottom_k),
    "bias_in_weights": ("sigmoid_bias_select", _mutant_bias_in_weights),
}


def _failures(impl):
    failures = 0
    for pin in ALL_PINS:
        try:
            pin(impl)
        except AssertionError:
            failures += 1
    return failures


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistakes_numpy(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setattr(moe_oracle, attr, fn)
    monkeypatch.setattr(oracle, attr, fn)
    assert _failures(oracle) > 0, f"no pin caught the planted mistake {name}"


def test_pins_catch_dropped_shared_expert_numpy(monkeypatch):
    real = moe_oracle.moe_layer

    def dropped(x, r, rw, ew, shared, k, routed_scale=1.0, score=0, bias=None):
        return real(x, r, rw, ew, [], k, routed_scale, score, bias)

    monkeypatch.setattr(oracle, "moe_layer", dropped)
    with pytest.raises(AssertionError):
        pin_two_expert_shared(oracle)


def test_pins_catch_dropped_residual_numpy(monkeypatch):
    real = moe_oracle.moe_layer

    def dropped(x, r, rw, ew, shared, k, routed_scale=1.0, score=0, bias=None):
        return real(x, np.zeros_like(np.asarray(r, float)), rw, ew, shared, k, routed_scale, score, bias)

    monkeypatch.setattr(oracle, "moe_layer", dropped)
    with pytest.raises(AssertionError):
        pin_two_expert_k2(oracle)


# The planted mistakes compiled into the C++ oracle (ORACLE_MUTANT in
# moe_oracle_ref.cpp); the NVFP4 ones are caught by the layout and cross-check
# tests rather than by a pin, so those tests are rerun against them.
CPP_MUTANTS = {1: "swap_gate_up", 2: "sigmoid_not_silu", 3: "silu_sign", 4: "no_renorm",
               5: "ties_to_higher_id", 6: "router_rows_reversed", 7: "bottom_k", 8: "drop_shared",
               9: "drop_residual", 10: "bias_in_weights", 11: "bf16_truncates", 12: "nibble_order",
               13: "e4m3_bias", 14: "no_routed_scale", 15: "fp8_scale_transposed"}


@pytest.mark.parametrize("mutant", sorted(CPP_MUTANTS), ids=lambda n: CPP_MUTANTS[n])
def test_pins_catch_planted_mistakes_cpp(mutant, monkeypatch):
    impl = CppOracle(mutant)
    failures = _failures(impl)
    if CPP_MUTANTS[mutant] == "fp8_scale_transposed":
        monkeypatch.setattr(cpp, "load", lambda m=0: impl.lib)
        with pytest.raises(AssertionError):
            test_fp8_layout_by_hand_cpp()
        failures += 1
    if CPP_MUTANTS[mutant] == "nibble_order":
        monkeypatch.setattr(cpp, "load", lambda m=0: impl.lib)
        with pytest.raises(AssertionError):
            test_nvfp4_layout_by_hand_cpp()
        failures += 1
    assert failures > 0, f"no pin caught the planted mistake {CPP_MUTANTS[mutant]}"


# ---------------------------------------------------------------------------
# number formats of the numpy restatement: library routines and published tables
# ---------------------------------------------------------------------------


@pytest.mark.parametrize("impl", sorted(IMPLS))
def test_bf16_widening_matches_torch_for_every_pattern(impl):
    o = IMPLS[impl]()
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = o.bf16_bits_to_f64(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    finite = np.isfinite(ref)
    np.testing.assert_array_equal(ours[finite], ref[finite])
    assert np.all(np.isnan(ours[np.isnan(ref)]))


def test_bf16_narrowing_matches_torch_on_float32_values():
    rng = np.random.default_rng(0)
    v32 = (rng.standard_normal(200000) * np.exp(rng.uniform(-20, 20, 200000))).astype(np.float32)
    ref = torch.from_numpy(v32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(oracle.f64_to_bf16_bits(v32.astype(np.float64)), ref)
    np.testing.assert_array_equal(cpp.f64_to_bf16_bits(v32.astype(np.float64)), ref)


def test_cpp_bf16_overflow_and_specials():
    big = np.array([3.5e38, -3.5e38, np.inf, -np.inf, 0.0, -0.0])
    bits = cpp.f64_to_bf16_bits(big)
    ref = torch.tensor(big, dtype=torch.float64).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(bits, ref)
    assert np.isnan(cpp.bf16_bits_to_f64(cpp.f64_to_bf16_bits(np.array([np.nan]))))[0]


def test_e4m3_points_and_nans():
    g = _golden("nvfp4_codes.json")
    for k, v in g["e4m3_points"].items():
        assert nvfp4.e4m3_value(int(k, 16)) == v
        assert cpp.e4m3_value(int(k, 16)) == v
    for k in g["e4m3_nan"]:
        assert math.isnan(nvfp4.e4m3_value(int(k, 16)))
        assert math.isnan(cpp.e4m3_value(int(k, 16)))
    e2 = g["e2m1"]
    got = [nvfp4.e2m1_value(c) for c in range(16)]
    assert [math.copysign(1, v) for v in got] == [math.copysign(1, v) for v in e2]


def test_nvfp4_dequant_layout_by_hand():
    # byte 0x21: element 0 = code 1 (0.5, low nibble), element 1 = code 2 (1.0);
    # byte 0xF8: element 2 = code 8 (-0.0), element 3 = code 15 (-6.0).
    codes = np.array([[0x21, 0xF8] + [0] * 6], np.uint8)  # K = 16: one block
    scales = np.array([[0x40]], np.uint8)  # 2.0
    out = nvfp4.dequant_nvfp4_rows(codes, scales, 0.5)
    np.testing.assert_array_equal(out[0, :4], [0.5, 1.0, -0.0, -6.0])
    assert np.all(out[0, 4:] == 0)


def test_nvfp4_quantiser_roundtrip_and_ties():
    """The synthetic quantiser (encoder) and the oracle decoder are independent;
    grid values survive a round trip exactly and midpoints round to even codes.

    Values are scaled by 1.75 so that amax = 10.5 gives an exact tensor scale
    10.5 / (6 * 448) = 2**-8 and an exact block scale 448; the codes then see the
    unscaled numbers.
    """
    grid = torch.tensor([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    row = (torch.cat([grid, -grid]) * 1.75).reshape(1, 16)
    codes, scales, ts = synth.quantize_nvfp4(row)
    assert float(ts) == 2.0 ** -8 and int(scales[0, 0]) == 0x7E
    back = nvfp4.dequant_nvfp4_rows(codes.numpy(), scales.numpy(), float(ts))
    np.testing.assert_array_equal(back, row.numpy().astype(np.float64))
    # midpoints between grid values round to the even code; 7 saturates at 6
    mids = torch.tensor([[0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0, 5.9, 0.3, 0.0, 0.0,
                          0.0, 0.0, 0.0, 0.0]]) * 1.75
    q, s, t = synth.quantize_nvfp4(mids)
    assert float(t) == 2.0 ** -8
    got = nvfp4.dequant_nvfp4_rows(q.numpy(), s.numpy(), float(t))[0, :10] / 1.75
    np.testing.assert_array_equal(got, [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0, 6.0, 6.0, 0.5])


def test_rmsnorm_identities():
    rng = np.random.default_rng(2)
    h = rng.standard_normal((3, 64)) * 5
    y = oracle.rmsnorm(h, 1e-6)
    ms = np.mean(h * h, axis=1)
    np.testing.assert_allclose(np.mean(y * y, axis=1), ms / (ms + 1e-6), rtol=1e-13)
    np.testing.assert_allclose(y / h, (1 / np.sqrt(ms + 1e-6))[:, None] * np.ones_like(h), rtol=1e-13)
    c = oracle.rmsnorm(np.full((1, 8), -0.5), 1e-6)
    np.testing.assert_allclose(c, -0.5 / math.sqrt(0.25 + 1e-6), rtol=1e-15)
    # the C++ stack input: a constant row normalises to -1 (exact in bf16 after rounding)
    bits = oracle.f64_to_bf16_bits(np.full((1, 8), -0.5))
    np.testing.assert_allclose(cpp.bf16_bits_to_f64(cpp.stack_layer_input(bits, 1e-6)), -1.0, atol=2 ** -8)


def test_expert_union_masks():
    idx = np.array([[5, 1], [1, 9], [7, 5]])
    experts, masks = oracle.expert_union(idx)
    assert experts.tolist() == [1, 5, 7, 9]
    assert masks.tolist() == [0b011, 0b101, 0b100, 0b010]
