"""Pins of the CPU oracle against facts fixed outside the oracle itself.

Each pin is something the pages or the mathematics decide: a hand-worked example,
a textbook reduction (uniform routing over all experts is a dense mean of SwiGLU
MLPs, written here with plain Python loops), invariants (weights sum to one,
joint permutation of experts, zero in -> zero out), a closed form (softmax over
all experts then top-k then renormalise), brute force on tiny inputs, and library
routines for the number formats. ``test_pins_catch_planted_mistakes`` plants
plausible mistakes in the oracle and checks that some pin fails for each.
"""

import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import moe_oracle, nvfp4
from moe_decode_layer_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


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


def _example_experts(ex):
    return [(np.array([e["gate"], e["up"]], float), np.array(e["down"], float))
            for e in ex["experts"]]


def _run_example(k, with_shared):
    ex = _golden("two_expert_example.json")
    experts = _example_experts(ex)
    shared = []
    if with_shared:
        s = ex["shared"]
        shared = [(np.array([s["gate"], s["up"]], float), np.array(s["down"], float))]
    out, idx, w = oracle.moe_layer(np.array([ex["x"]]), np.array([ex["residual"]]),
                                   np.array(ex["router_w"], float), lambda e: experts[e],
                                   shared, k)
    return ex, out[0], idx[0], w[0]


def _rand_layer(rng, h=6, i=3, e=5, s=1):
    return (rng.standard_normal((e, h)),
            [(rng.standard_normal((2 * i, h)), rng.standard_normal((h, i))) for _ in range(e)],
            [(rng.standard_normal((2 * i, h)), rng.standard_normal((h, i))) for _ in range(s)])


# ---------------------------------------------------------------------------
# the pins, each a function so the planted-mistake test can rerun them
# ---------------------------------------------------------------------------


def pin_two_expert_k2():
    ex, out, idx, w = _run_example(2, False)
    np.testing.assert_allclose(oracle.router_logits(np.array([ex["x"]]), np.array(ex["router_w"]))[0],
                               ex["logits"], rtol=0, atol=1e-15)
    assert list(idx) == ex["k2"]["idx"]
    np.testing.assert_allclose(w, ex["k2"]["w"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(out, ex["k2"]["out"], rtol=0, atol=1e-13)


def pin_two_expert_k1():
    ex, out, idx, w = _run_example(1, False)
    assert list(idx) == ex["k1"]["idx"]
    np.testing.assert_allclose(w, ex["k1"]["w"], rtol=0, atol=1e-15)
    np.testing.assert_allclose(out, ex["k1"]["out"], rtol=0, atol=1e-13)


def pin_two_expert_shared():
    ex, out, _, _ = _run_example(2, True)
    np.testing.assert_allclose(out, ex["k2_shared"]["out"], rtol=0, atol=1e-13)


def pin_uniform_routing_is_dense_mean():
    """k = E and a zero router: every expert gets weight 1/E (textbook dense MoE)."""
    rng = np.random.default_rng(11)
    hdim, e = 6, 4
    _, experts, shared = _rand_layer(rng, h=hdim, i=3, e=e, s=1)
    x = rng.standard_normal((2, hdim))
    r = rng.standard_normal((2, hdim))
    out, idx, w = oracle.moe_layer(x, r, np.zeros((e, hdim)), lambda j: experts[j], shared, e)
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


def pin_weights_sum_to_one():
    rng = np.random.default_rng(3)
    for _ in range(50):
        logits = rng.standard_normal(37) * 3
        _, w = oracle.topk_renorm(logits, 5)
        assert abs(w.sum() - 1.0) < 1e-12
        assert np.all(w > 0) and np.all(np.diff(w) <= 0)


def pin_softmax_topk_renorm_closed_form():
    """Full softmax over E, keep the top k, renormalise: plain Python."""
    rng = np.random.default_rng(5)
    for trial in range(30):
        e, k = 12, 1 + trial % 6
        logits = (rng.standard_normal(e) * 2).tolist()
        z = sum(math.exp(v) for v in logits)
        p = [math.exp(v) / z for v in logits]
        order = sorted(range(e), key=lambda i: (-logits[i], i))[:k]
        ref_w = [p[i] / sum(p[j] for j in order) for i in order]
        idx, w = oracle.topk_renorm(np.array(logits), k)
        assert idx.tolist() == order
        np.testing.assert_allclose(w, ref_w, rtol=1e-12, atol=0)


def pin_topk_brute_force_with_ties():
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
        idx, _ = oracle.topk_renorm(logits, k)
        assert idx.tolist() == [i for _, i in best]


def pin_joint_permutation():
    rng = np.random.default_rng(13)
    router, experts, shared = _rand_layer(rng, h=8, i=4, e=7, s=1)
    x = rng.standard_normal((3, 8))
    r = rng.standard_normal((3, 8))
    perm = rng.permutation(7)  # new expert p holds old expert perm[p]
    out_a, idx_a, w_a = oracle.moe_layer(x, r, router, lambda j: experts[j], shared, 3)
    out_b, idx_b, w_b = oracle.moe_layer(x, r, router[perm], lambda j: experts[perm[j]], shared, 3)
    np.testing.assert_allclose(out_a, out_b, rtol=1e-13, atol=1e-13)
    np.testing.assert_array_equal(idx_a, perm[idx_b])
    np.testing.assert_allclose(w_a, w_b, rtol=1e-14, atol=1e-15)


def pin_zero_row_zero_output():
    rng = np.random.default_rng(17)
    router, experts, shared = _rand_layer(rng)
    out, _, _ = oracle.moe_layer(np.zeros((2, 6)), np.zeros((2, 6)), router,
                                 lambda j: experts[j], shared, 2)
    assert np.all(out == 0.0)


def pin_silu_identities():
    g = np.linspace(-30, 30, 601)
    s = oracle.silu(g)
    np.testing.assert_allclose(s - oracle.silu(-g), g, rtol=0, atol=1e-12)  # g*sig(g) + g*sig(-g) = g
    assert oracle.silu(np.array([0.0]))[0] == 0.0
    assert abs(oracle.silu(np.array([800.0]))[0] - 800.0) < 1e-9
    assert oracle.silu(np.array([-800.0]))[0] == 0.0
    np.testing.assert_allclose(oracle.silu(np.array([1.0]))[0] * (1 + math.exp(-1)), 1.0, rtol=1e-15)


ALL_PINS = [pin_two_expert_k2, pin_two_expert_k1, pin_two_expert_shared,
            pin_uniform_routing_is_dense_mean, pin_weights_sum_to_one,
            pin_softmax_topk_renorm_closed_form, pin_topk_brute_force_with_ties,
            pin_joint_permutation, pin_zero_row_zero_output, pin_silu_identities]


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin()


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


MUTANTS = {
    "swap_gate_up": ("expert_swiglu", _mutant_swap_gate_up),
    "sigmoid_not_silu": ("silu", _mutant_sigmoid_not_silu),
    "silu_sign": ("silu", _mutant_silu_sign),
    "no_renorm": ("topk_renorm", _mutant_no_renorm),
    "ties_to_higher_id": ("topk_renorm", _mutant_ties_to_higher),
    "router_rows_reversed": ("router_logits", _mutant_router_rows_reversed),
    "bottom_k": ("topk_renorm", _mutant_bottom_k),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistakes(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setattr(moe_oracle, attr, fn)
    monkeypatch.setattr(oracle, attr, fn)
    failures = 0
    for pin in ALL_PINS:
        try:
            pin()
        except AssertionError:
            failures += 1
    assert failures > 0, f"no pin caught the planted mistake {name}"


def test_pins_catch_dropped_shared_expert(monkeypatch):
    real = moe_oracle.moe_layer

    def dropped(x, r, rw, ew, shared, k, routed_scale=1.0):
        return real(x, r, rw, ew, [], k, routed_scale)

    monkeypatch.setattr(oracle, "moe_layer", dropped)
    with pytest.raises(AssertionError):
        pin_two_expert_shared()


def test_pins_catch_dropped_residual(monkeypatch):
    real = moe_oracle.moe_layer

    def dropped(x, r, rw, ew, shared, k, routed_scale=1.0):
        return real(x, np.zeros_like(np.asarray(r, float)), rw, ew, shared, k, routed_scale)

    monkeypatch.setattr(oracle, "moe_layer", dropped)
    with pytest.raises(AssertionError):
        pin_two_expert_k2()


# ---------------------------------------------------------------------------
# number formats: library routines and published tables
# ---------------------------------------------------------------------------


def test_bf16_widening_matches_torch_for_every_pattern():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.bf16_bits_to_f64(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    finite = np.isfinite(ref)
    np.testing.assert_array_equal(ours[finite], ref[finite])
    assert np.all(np.isnan(ours[np.isnan(ref)]))


def test_bf16_narrowing_matches_torch_on_float32_values():
    rng = np.random.default_rng(0)
    v32 = (rng.standard_normal(200000) * np.exp(rng.uniform(-20, 20, 200000))).astype(np.float32)
    ref = torch.from_numpy(v32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(oracle.f64_to_bf16_bits(v32.astype(np.float64)), ref)


def test_bf16_narrowing_ties_to_even():
    # 1 + 2^-8 lies halfway between 1 and 1 + 2^-7: even mantissa (1.0) wins;
    # 1 + 3*2^-8 lies between 1 + 2^-7 (odd) and 1 + 2^-6 (even): rounds up.
    vals = np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 2 ** -130 * 1.5])
    got = oracle.bf16_bits_to_f64(oracle.f64_to_bf16_bits(vals))
    np.testing.assert_array_equal(got, [1.0, 1 + 2 ** -6, -1.0, 2 ** -130 * 1.5])


def test_e2m1_table():
    ref = _golden("nvfp4_codes.json")["e2m1"]
    got = [nvfp4.e2m1_value(c) for c in range(16)]
    assert got == ref
    assert [math.copysign(1, v) for v in got] == [math.copysign(1, v) for v in ref]


def test_e4m3_matches_torch_float8_for_every_byte():
    bits = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(bits).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([nvfp4.e4m3_value(b) for b in range(256)])
    same = np.isnan(ref) == np.isnan(got)
    assert same.all()
    np.testing.assert_array_equal(got[~np.isnan(ref)], ref[~np.isnan(ref)])
    g = _golden("nvfp4_codes.json")
    for k, v in g["e4m3_points"].items():
        assert nvfp4.e4m3_value(int(k, 16)) == v
    for k in g["e4m3_nan"]:
        assert math.isnan(nvfp4.e4m3_value(int(k, 16)))


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


def test_expert_union_masks():
    idx = np.array([[5, 1], [1, 9], [7, 5]])
    experts, masks = oracle.expert_union(idx)
    assert experts.tolist() == [1, 5, 7, 9]
    assert masks.tolist() == [0b011, 0b101, 0b100, 0b010]
