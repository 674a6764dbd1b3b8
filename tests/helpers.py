"""Test-side glue between the synthetic inputs, the oracle and the GPU library.

Lives under tests/ because it calls the oracle (test infrastructure). The GPU
parity tests compare against the C++ float64 oracle (``oracle.cpp``), which reads
the exact bf16 / NVFP4 bit patterns the kernels read.
"""

from __future__ import annotations

import numpy as np
import torch

import oracle
from oracle import cpp
from moe_decode_layer_gb300 import synth

MAX_ABS = 2e-2     # output tolerance against the float64 oracle (bf16 weights)
REL_L2 = 5e-3
W_ABS = 1e-5       # routing weights


def bits(t: torch.Tensor) -> np.ndarray:
    """Raw bit patterns of a bf16 / uint8 tensor as numpy (uint16 / uint8)."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def f64(t: torch.Tensor) -> np.ndarray:
    return oracle.bf16_bits_to_f64(bits(t))


def hidden_with_margin(router_w: torch.Tensor, m_rows: int, top_k: int, seed: int,
                       rho: float = 0.0, margin: float = 0.05, max_tries: int = 200, score: int = 0,
                       bias=None):
    """bf16 [M, H] rows whose float64 selection keys have a top-k gap >= margin
    (router logits for softmax scoring; sigmoid(logit) + bias for the
    bias-corrected sigmoid rule).

    Each row that misses the margin is redrawn alone (its own stream), so the
    selected expert set is decided by a gap far above fp32 rounding.
    """
    rw = bits(router_w)
    b = None if bias is None else bias.detach().cpu().double().numpy()
    attempts = [0] * m_rows
    for _ in range(max_tries):
        x = synth.hidden_rows(m_rows, rw.shape[1], seed, rho, attempts)
        logits = cpp.router_logits(f64(x), rw)
        bad = [m for m in range(m_rows) if selection_margin(logits[m], top_k, score, b) < margin]
        if not bad:
            return x
        for m in bad:
            attempts[m] += 1
    raise RuntimeError("could not draw rows with the requested top-k margin")


def expert_accessor(shape: synth.LayerShape, layer: dict, prefix: str = ""):
    """e -> the raw weights of expert e for the C++ oracle, copied from the layer
    tensors on demand: bf16 bit patterns (w13 [2I, H], w2 [H, I]) or an NVFP4
    expert (codes, e4m3 scale bytes, tensor scales). Down matrices stored
    transposed (w2_layout "i_h") are handed over in the [H, I] orientation."""
    t = layer.get("w2_layout", "h_i") == "i_h"

    def down(name, e):
        w = layer[prefix + name][e]
        return w.transpose(0, 1).contiguous() if t else w

    def get(e):
        if shape.wdtype == "bf16":
            return bits(layer[prefix + "w13"][e]), bits(down("w2", e))
        if shape.wdtype == "fp8":
            return cpp.FP8Expert(bits(layer[prefix + "w13_q"][e]), layer[prefix + "w13_s"][e].cpu().numpy(),
                                 bits(down("w2_q", e)), down("w2_s", e).cpu().numpy())
        return cpp.NVFP4Expert(bits(layer[prefix + "w13_q"][e]), bits(layer[prefix + "w13_s"][e]),
                               layer[prefix + "w13_gs"][e].cpu().numpy(), bits(layer[prefix + "w2_q"][e]),
                               bits(layer[prefix + "w2_s"][e]), np.float32(layer[prefix + "w2_gs"][e].cpu()))
    return get


def oracle_layer(shape: synth.LayerShape, layer: dict, x: torch.Tensor, residual: torch.Tensor,
                 routed_scale: float = 1.0, score: int = 0, bias=None):
    """Run the C++ oracle on the exact values of the given tensors (copied to host).

    Returns (out float64 [M, H], idx int64 [M, k], w float64 [M, k])."""
    shared_get = expert_accessor(shape, layer, "sh_")
    shared = [shared_get(s) for s in range(shape.num_shared)]
    b = None if bias is None else bias.detach().cpu().double().numpy()
    return cpp.moe_layer(f64(x), f64(residual), bits(layer["router_w"]), expert_accessor(shape, layer), shared,
                         shape.top_k, routed_scale, score, b)


def selection_margin(logits_row: np.ndarray, k: int, score: int = 0, bias=None) -> float:
    """Gap between the k-th and (k+1)-th selection key of one row (float64)."""
    key = np.asarray(logits_row, np.float64)
    if score == 1:
        key = 1.0 / (1.0 + np.exp(-key)) + np.asarray(bias, np.float64)
    return oracle.topk_margin(key, k)


def assert_close(got_bf16: torch.Tensor, ref: np.ndarray, max_abs=MAX_ABS, rel_l2=REL_L2, what="out"):
    g = f64(got_bf16)
    err = np.abs(g - ref)
    rl2 = np.linalg.norm(g - ref) / max(np.linalg.norm(ref), 1e-30)
    assert np.all(np.isfinite(g)), f"{what}: non-finite values"
    assert err.max() <= max_abs, f"{what}: max abs err {err.max():.3e} > {max_abs}"
    assert rl2 <= rel_l2, f"{what}: rel L2 {rl2:.3e} > {rel_l2}"
    return float(err.max()), float(rl2)


def assert_routing(idx_gpu: torch.Tensor, w_gpu: torch.Tensor, idx_ref: np.ndarray, w_ref: np.ndarray,
                   by_weight: bool = True):
    """Index sets bit-exact; weights within W_ABS matched by expert id. The GPU
    lists experts by descending selection key, which is the weight's order under
    softmax scoring (by_weight) but not under the bias-corrected sigmoid rule."""
    ig = idx_gpu.cpu().numpy()
    wg = w_gpu.cpu().numpy().astype(np.float64)
    for m in range(idx_ref.shape[0]):
        assert sorted(ig[m].tolist()) == sorted(idx_ref[m].tolist()), f"row {m}: expert sets differ"
        ref = dict(zip(idx_ref[m].tolist(), w_ref[m].tolist()))
        for e, w in zip(ig[m].tolist(), wg[m].tolist()):
            assert abs(w - ref[e]) <= W_ABS, f"row {m} expert {e}: weight {w} vs {ref[e]}"
        if by_weight:
            assert np.all(np.diff(wg[m]) <= 1e-7)
