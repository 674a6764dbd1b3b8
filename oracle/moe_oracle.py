"""Plain float64 reference of one small-batch MoE decode layer step.

TEST INFRASTRUCTURE ONLY (see the package docstring). Slow and obvious on purpose:
each function is the textbook definition, with a numpy matmul as the only library
primitive.

What the step computes, per token row m (M = 1..8 rows):

  1. router logits     l[m, e] = sum_h x[m, h] * Wr[e, h]
       Ling-3.0-flash batch-1 decode blog, section "PDL: stacking the latency
       floors of small kernels" (router chain: norm -> gate matvec -> top-k) and
       section "bf16 router gate and lm_head" (the gate is a bf16 matvec).
  2. top-k + renormalised weights
       idx = the k largest logits (ties go to the lower expert id),
       w_j = exp(l_j - l_max) / sum_{i in idx} exp(l_i - l_max).
       This is softmax over all experts, then top-k, then renormalise: the full
       softmax denominator cancels. The pages name a top-k kernel but never its
       scoring rule; softmax -> top-k -> renormalise is the documented reading.
  3. routed experts    g = Wg_e x, u = Wu_e x, h = silu(g) * u, y_e = Wd_e h
       with W13_e = [Wg_e; Wu_e] of shape [2I, H] and W2_e = Wd_e of shape [H, I].
       Same blog, section "Two fusions and a retune" (silu(gate) * up folded into
       the up-GEMM epilogue; w13 holds gate and up).
  4. shared expert     s = the same SwiGLU MLP with the shared weights, weight 1.
       Ling model table (Chinese translation of the blog, section "模型"):
       512 routed experts + 1 shared expert, top-8(+1), moe_intermediate 768,
       hidden 2560.
  5. combine           out = r + routed_scale * sum_j w_j y_{idx_j} + s
       Same blog, section "PDL: ..." (the small-M combine is one fp32 sum times a
       scale with a single final cast). The oracle keeps float64 and does not round.

Readings where the pages are silent (each is listed in the design notes):
  * routed_scale defaults to 1.0 (never mentioned);
  * the residual r is a separate input; single-layer cases use r = x;
  * the shared expert has the routed intermediate size and weight 1;
  * RMSNorm (between stacked layers) is gamma = 1, eps = 1e-6, pre-norm.
"""

from __future__ import annotations

import numpy as np

# ----------------------------------------------------------------------------
# bf16 <-> float64 (exact widening, round-to-nearest-even narrowing)
# ----------------------------------------------------------------------------


def bf16_bits_to_f64(bits) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to float64 exactly.

    A bf16 value is the top half of the float32 with the same bits, so the
    widening shifts the pattern into the high half of a uint32 and reads that as
    float32, which float64 represents exactly.
    """
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    with np.errstate(invalid="ignore"):  # NaN patterns stay NaN
        return b.view(np.float32).astype(np.float64)


def f64_to_bf16_bits(v) -> np.ndarray:
    """Round float64 values to the nearest bf16 (ties to even), return uint16 bits.

    bf16 keeps 8 significant bits. For v = m * 2**e with 0.5 <= |m| < 1 the spacing
    of bf16 values near v is 2**(e - 8); below the smallest normal (2**-126) the
    spacing stays 2**-133. ``np.rint`` rounds halves to even. Finite inputs only.
    """
    v = np.asarray(v, dtype=np.float64)
    _, e = np.frexp(v)
    quantum = np.ldexp(1.0, np.maximum(e, -125) - 8)
    r = np.rint(v / quantum) * quantum
    r32 = r.astype(np.float32)  # exact: r has at most 8 significant bits
    return (r32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


# ----------------------------------------------------------------------------
# Steps 1-2: router and top-k with renormalised weights
# ----------------------------------------------------------------------------


def router_logits(x: np.ndarray, router_w: np.ndarray) -> np.ndarray:
    """l[m, e] = sum_h x[m, h] * Wr[e, h]; x [M, H], Wr [E, H] -> [M, E]."""
    return np.asarray(x, np.float64) @ np.asarray(router_w, np.float64).T


def topk_renorm(logits_row: np.ndarray, k: int):
    """Top-k of one row of logits and the renormalised softmax weights.

    Returns (idx, w): idx int64 [k] in descending logit order (equal logits keep
    ascending expert id), w float64 [k] = exp(l_j - l_max) / sum over the selected.
    """
    l = np.asarray(logits_row, np.float64)
    order = np.argsort(-l, kind="stable")  # stable: the lower id wins a tie
    idx = order[:k]
    sel = l[idx]
    e = np.exp(sel - sel.max())
    return idx.astype(np.int64), e / e.sum()


SCORE_SOFTMAX = 0
SCORE_SIGMOID_BIAS = 1


def sigmoid_bias_select(logits_row: np.ndarray, k: int, bias: np.ndarray):
    """Bias-corrected sigmoid selection of one row.

    s_e = 1 / (1 + exp(-l_e)); the k largest s_e + b_e are selected (equal keys:
    the lower expert id first); w_j = s_j / sum over the selected of s_i, so the
    bias steers which experts are chosen but not their weights. The Ling blog's
    router top-k "prefetches its bias" (section "PDL: stacking the latency floors
    of small kernels"); the pages give no more of the rule, so this is the plainest
    reading of a bias-corrected sigmoid router.
    """
    l = np.asarray(logits_row, np.float64)
    s = 1.0 / (1.0 + np.exp(-l))
    key = s + np.asarray(bias, np.float64)
    idx = np.argsort(-key, kind="stable")[:k]
    return idx.astype(np.int64), s[idx] / s[idx].sum()


def select(logits_row: np.ndarray, k: int, score: int = SCORE_SOFTMAX, bias=None):
    """Selection and weights of one row under a scoring rule (0 softmax, 1 sigmoid + bias)."""
    if score == SCORE_SOFTMAX:
        return topk_renorm(logits_row, k)
    if score == SCORE_SIGMOID_BIAS:
        return sigmoid_bias_select(logits_row, k, bias)
    raise ValueError(f"unknown scoring rule {score}")


def route(x: np.ndarray, router_w: np.ndarray, k: int, score: int = SCORE_SOFTMAX, bias=None):
    """Per-row routing: (logits [M, E], idx [M, k], w [M, k])."""
    logits = router_logits(x, router_w)
    idx = np.zeros((logits.shape[0], k), np.int64)
    w = np.zeros((logits.shape[0], k), np.float64)
    for m in range(logits.shape[0]):
        if score == SCORE_SOFTMAX:  # looked up by name so that planted mistakes reach it
            idx[m], w[m] = topk_renorm(logits[m], k)
        else:
            idx[m], w[m] = select(logits[m], k, score, bias)
    return logits, idx, w


def topk_margin(logits_row: np.ndarray, k: int) -> float:
    """Gap between the k-th and (k+1)-th largest logit (inf when k = E)."""
    s = np.sort(np.asarray(logits_row, np.float64))[::-1]
    return float("inf") if k >= s.size else float(s[k - 1] - s[k])


def expert_union(idx: np.ndarray):
    """Distinct experts chosen by any row (ascending id) and their row masks.

    SGLang Low-Latency Mode page, section "Low-Latency-Specific Optimizations",
    item 3: with at most eight rows every expert's rows fit one eight-row tile,
    placed by a bitmap and population counts. Returns (experts [U], masks [U])
    where bit m of masks[u] says row m chose experts[u].
    """
    idx = np.asarray(idx)
    experts = sorted(set(int(e) for e in idx.ravel()))
    masks = []
    for e in experts:
        mk = 0
        for m in range(idx.shape[0]):
            if e in set(int(v) for v in idx[m]):
                mk |= 1 << m
        masks.append(mk)
    return np.array(experts, np.int64), np.array(masks, np.int64)


# ----------------------------------------------------------------------------
# Steps 3-5: SwiGLU experts, shared expert, combine into the residual
# ----------------------------------------------------------------------------


def silu(g):
    """silu(g) = g / (1 + exp(-g)), in float64."""
    g = np.asarray(g, np.float64)
    with np.errstate(over="ignore"):
        return g / (1.0 + np.exp(-g))


def expert_swiglu(x_row: np.ndarray, w13: np.ndarray, w2: np.ndarray) -> np.ndarray:
    """One SwiGLU expert on one row: W2 (silu(Wg x) * (Wu x)).

    w13 [2I, H] holds the gate rows 0..I-1 then the up rows I..2I-1; w2 is [H, I].
    """
    w13 = np.asarray(w13, np.float64)
    inter = w13.shape[0] // 2
    g = w13[:inter] @ x_row
    u = w13[inter:] @ x_row
    return np.asarray(w2, np.float64) @ (silu(g) * u)


def moe_layer(x, residual, router_w, expert_weights, shared_weights, top_k,
              routed_scale: float = 1.0, score: int = SCORE_SOFTMAX, bias=None):
    """One MoE decode layer step for M rows, float64 throughout.

    x, residual : float64 [M, H] (the exact values of the bf16 inputs)
    router_w    : float64 [E, H]
    expert_weights(e) -> (w13 [2I, H], w2 [H, I]) for routed expert e; called only
                  for the experts some row selects, so callers can hand over just
                  those experts' weights
    shared_weights : list of (w13, w2), each added with weight 1
    score, bias : the scoring rule (see ``select``) and the per-expert bias [E]
    Returns (out float64 [M, H], idx int64 [M, k], w float64 [M, k]).
    """
    x = np.asarray(x, np.float64)
    out = np.array(residual, np.float64, copy=True)
    _, idx, w = route(x, router_w, top_k, score, bias)
    cache = {}
    for m in range(x.shape[0]):
        routed = np.zeros(x.shape[1])
        for j in range(top_k):
            e = int(idx[m, j])
            if e not in cache:
                cache[e] = expert_weights(e)
            w13, w2 = cache[e]
            routed += w[m, j] * expert_swiglu(x[m], w13, w2)
        out[m] += routed_scale * routed
        for w13, w2 in shared_weights:
            out[m] += expert_swiglu(x[m], w13, w2)
    return out, idx, w


# ----------------------------------------------------------------------------
# RMSNorm between stacked layers
# ----------------------------------------------------------------------------


def rmsnorm(h: np.ndarray, eps: float = 1e-6) -> np.ndarray:
    """h / sqrt(mean(h^2) + eps) per row, gamma = 1 (router chain "norm" step)."""
    h = np.asarray(h, np.float64)
    return h / np.sqrt(np.mean(h * h, axis=-1, keepdims=True) + eps)


def stack_layer_input(hidden_bits: np.ndarray, eps: float = 1e-6) -> np.ndarray:
    """bf16 bits of the next layer's MoE input: bf16(RMSNorm(hidden)).

    The stacked step is pre-norm: hidden_{l+1} = hidden_l + MoE_l(RMSNorm(hidden_l)),
    the normalised input rounded once to bf16 because the router and expert
    matvecs consume bf16 activations.
    """
    return f64_to_bf16_bits(rmsnorm(bf16_bits_to_f64(hidden_bits), eps))
