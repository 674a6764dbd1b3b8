"""Seeded synthetic inputs for the MoE decode layer step.

Shared by the tests, the bench and the smoke check. This module only draws and
encodes inputs (normal draws, bf16 rounding, NVFP4 quantisation); it holds none of
the layer's arithmetic, and no expected value is ever computed here.

Recipe (the pages publish no weights, so all inputs are synthetic):
  * weights ~ N(0, 0.02^2), rounded to bf16 (torch RNG on the target device,
    drawn in chunks of experts so a 6 GB layer needs no 24 GB float32 temporary);
  * hidden rows ~ N(0, 1) as float32, rounded to bf16. With rho > 0 the rows are
    correlated: x_m = sqrt(rho) z_0 + sqrt(1 - rho) z_m, with z_0 shared, so the
    rows of a speculative verify chain route to partly overlapping experts;
  * every row draws its z_m from its own stream keyed (seed, row, attempt), so a
    caller that needs a top-k margin can redraw one row alone;
  * NVFP4 weights come from the same bf16-free N(0, 0.02^2) float32 draws,
    quantised with tensor scale amax / (6 * 448), e4m3 block scales
    amax_block / (6 * tensor_scale) and e2m1 codes rounded to nearest-even;
  * FP8 weights from the same draws: one fp32 scale per 128 x 128 block,
    amax_block / 448, and e4m3 codes rounded to nearest-even (torch's cast).
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np
import torch


@dataclass(frozen=True)
class LayerShape:
    """Sizes of one MoE layer: H hidden, I expert intermediate, E routed experts."""

    hidden: int
    inter: int
    num_experts: int
    top_k: int
    num_shared: int = 1
    wdtype: str = "bf16"  # "bf16", "nvfp4" or "fp8"

    def expert_bytes(self) -> int:
        """HBM bytes of one expert's gate/up/down weights (codes + block scales)."""
        h, i = self.hidden, self.inter
        if self.wdtype == "bf16":
            return 3 * h * i * 2
        if self.wdtype == "fp8":
            return 3 * h * i + 3 * (h // 128) * (i // 128) * 4
        return 3 * h * i // 2 + 3 * h * i // 16

    def router_bytes(self) -> int:
        return self.num_experts * self.hidden * 2


# The layer shapes the pages describe (model tables of the Ling-3.0-flash and
# Muse Spark posts) plus a tiny one for fast checks.
TINY = LayerShape(hidden=256, inter=128, num_experts=16, top_k=2, num_shared=1)
LING = LayerShape(hidden=2560, inter=768, num_experts=512, top_k=8, num_shared=1)
MUSE_NVFP4 = LayerShape(hidden=4096, inter=1024, num_experts=256, top_k=8,
                        num_shared=0, wdtype="nvfp4")
LING_E64 = LayerShape(hidden=2560, inter=768, num_experts=64, top_k=8, num_shared=1)
LING_FP8 = LayerShape(hidden=2560, inter=768, num_experts=512, top_k=8, num_shared=1, wdtype="fp8")


# Workloads of the bench and the profiling tools: layer shape, rows, row
# correlation, layers per step.
WORKLOADS = {
    "ling_m1": dict(shape="LING", m=1, rho=0.0, layers=1,
                    desc="Ling-3.0-flash-shaped MoE layer, H=2560, E=512 top-8 + 1 shared, I=768, M=1"),
    "ling_m6": dict(shape="LING", m=6, rho=0.5, layers=1,
                    desc="Ling-3.0-flash-shaped MoE layer, H=2560, E=512 top-8 + 1 shared, I=768, "
                         "M=6 verify rows correlated rho=0.5"),
    "ling_m16": dict(shape="LING", m=16, rho=0.5, layers=1,
                     desc="Ling-3.0-flash-shaped MoE layer, M=16 verify rows correlated rho=0.5 "
                          "(two launches of 8 rows)"),
    "stack_m6": dict(shape="LING", m=6, rho=0.5, layers=12,
                     desc="12 distinct Ling-shaped MoE layers back to back, RMSNorm(1e-6) + residual "
                          "between layers, M=6 rho=0.5"),
    "nvfp4_m1": dict(shape="MUSE_NVFP4", m=1, rho=0.0, layers=1,
                     desc="NVFP4 experts (e2m1, e4m3 block-16 scales, fp32 tensor scale), H=4096, "
                          "E=256 top-8, I=1024, no shared expert, M=1"),
    "nvfp4_m6": dict(shape="MUSE_NVFP4", m=6, rho=0.5, layers=1,
                     desc="NVFP4 experts, H=4096, E=256 top-8, I=1024, M=6 rho=0.5"),
    "ling_fp8_m1": dict(shape="LING_FP8", m=1, rho=0.0, layers=1,
                        desc="Ling-shaped MoE layer with FP8 experts (e4m3, fp32 scale per 128 x 128 "
                             "block), H=2560, E=512 top-8 + 1 shared, I=768, M=1"),
    "ling_fp8_m6": dict(shape="LING_FP8", m=6, rho=0.5, layers=1,
                        desc="Ling-shaped MoE layer with FP8 experts, M=6 verify rows correlated rho=0.5"),
    # decode sequences: each layer copy sees successive steps whose hidden rows
    # follow x_t = sqrt(0.8) x_{t-1} + sqrt(0.2) z_t (about half of the top-8
    # experts repeat from one step to the next), with and without the
    # speculative prefetch of the previous step's most-used experts
    "ling_m1_seq": dict(shape="LING", m=1, rho=0.0, layers=1, seq_rho=0.8, prefetch=4,
                        desc="Ling-shaped layer, M=1, successive decode steps correlated 0.8, "
                             "4 experts of the previous step prefetched into L2 while routing"),
    "ling_m1_seq_off": dict(shape="LING", m=1, rho=0.0, layers=1, seq_rho=0.8, prefetch=0,
                            desc="the same decode sequence without the prefetch"),
    "ling_m6_seq": dict(shape="LING", m=6, rho=0.5, layers=1, seq_rho=0.8, prefetch=4,
                        desc="Ling-shaped layer, M=6 rho=0.5, successive decode steps correlated 0.8, "
                             "4 most-used experts of the previous step prefetched into L2 while routing"),
    "ling_m6_seq_off": dict(shape="LING", m=6, rho=0.5, layers=1, seq_rho=0.8, prefetch=0,
                            desc="the same decode sequence without the prefetch"),
    "tiny_m1": dict(shape="TINY", m=1, rho=0.0, layers=1,
                    desc="tiny MoE layer H=256, E=16 top-2 + 1 shared, I=128, M=1"),
    # profiling case: Ling-shaped experts, 64 of them (0.76 GB per copy), same
    # bytes per step as Ling M=1 but for the smaller router
    "ling_e64_m1": dict(shape="LING_E64", m=1, rho=0.0, layers=1,
                        desc="Ling-shaped experts with E=64 top-8 + 1 shared (profiling case), M=1"),
    "ling_e64_m6": dict(shape="LING_E64", m=6, rho=0.5, layers=1,
                        desc="Ling-shaped experts with E=64 top-8 + 1 shared (profiling case), M=6"),
}


def workload_shape(name: str) -> LayerShape:
    return globals()[WORKLOADS[name]["shape"]]


def algorithmic_bytes(shape: LayerShape, distinct_routed: int) -> int:
    """Bytes one layer step must read: router + each distinct routed expert + shared."""
    return shape.router_bytes() + (distinct_routed + shape.num_shared) * shape.expert_bytes()


# ----------------------------------------------------------------------------
# hidden rows
# ----------------------------------------------------------------------------


def decode_sequence(steps: int, m_rows: int, hidden: int, seed: int, rho: float = 0.0,
                    seq_rho: float = 0.8) -> list:
    """bf16 [M, H] rows of `steps` successive decode steps: step 0 as
    hidden_rows, then x_t = sqrt(seq_rho) x_{t-1} + sqrt(1 - seq_rho) z_t, with z_t
    drawn as hidden_rows (its own seed per step), in float32, rounded to bf16."""
    x = hidden_rows(m_rows, hidden, seed=seed, rho=rho).float()
    out = [x.to(torch.bfloat16)]
    for t in range(1, steps):
        z = hidden_rows(m_rows, hidden, seed=seed * 1000 + t, rho=rho).float()
        x = math.sqrt(seq_rho) * x + math.sqrt(1.0 - seq_rho) * z
        out.append(x.to(torch.bfloat16))
    return out


def hidden_rows(m_rows: int, hidden: int, seed: int, rho: float = 0.0,
                attempts=None) -> torch.Tensor:
    """bf16 [M, H] hidden rows on the CPU (see the module recipe)."""
    rng0 = np.random.default_rng([seed, 0x5EED, 0])
    z0 = rng0.standard_normal(hidden)
    rows = np.empty((m_rows, hidden), np.float64)
    for m in range(m_rows):
        a = 0 if attempts is None else int(attempts[m])
        zm = np.random.default_rng([seed, 0x5EED, 1 + m, a]).standard_normal(hidden)
        rows[m] = math.sqrt(rho) * z0 + math.sqrt(1.0 - rho) * zm
    return torch.from_numpy(rows.astype(np.float32)).to(torch.bfloat16)


# ----------------------------------------------------------------------------
# weights
# ----------------------------------------------------------------------------


def _normal(shape, gen, device, std):
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32) * std


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _bf16_experts(n, rows, cols, seed, device, std, chunk_bytes=1 << 29):
    out = torch.empty((n, rows, cols), dtype=torch.bfloat16, device=device)
    per = max(1, chunk_bytes // (rows * cols * 4))
    for s in range(0, n, per):
        e = min(n, s + per)
        g = _gen(seed * 1000003 + s, device)
        out[s:e] = _normal((e - s, rows, cols), g, device, std).to(torch.bfloat16)
    return out


def _e2m1_codes(q: torch.Tensor) -> torch.Tensor:
    """Round float32 values to e2m1 (nearest, ties to even code), saturating at 6."""
    mag = q.abs()
    code = torch.zeros_like(mag, dtype=torch.uint8)
    # (lower bound, inclusive?) -> code; the tie at each midpoint goes to the even code
    code = torch.where(mag > 0.25, 1, code)
    code = torch.where(mag >= 0.75, 2, code)
    code = torch.where(mag > 1.25, 3, code)
    code = torch.where(mag >= 1.75, 4, code)
    code = torch.where(mag > 2.5, 5, code)
    code = torch.where(mag >= 3.5, 6, code)
    code = torch.where(mag > 5.0, 7, code).to(torch.uint8)
    sign = ((q < 0) & (code != 0)).to(torch.uint8) << 3
    return code | sign


def quantize_nvfp4(w: torch.Tensor):
    """Quantise float32 [..., R, K] to NVFP4 with one tensor scale over the last two dims.

    Returns (codes uint8 [..., R, K/2], scales uint8 [..., R, K/16], tensor_scale
    float32 [...]).
    """
    *lead, r, k = w.shape
    amax = w.abs().amax(dim=(-2, -1))
    ts = (amax / (6.0 * 448.0)).to(torch.float32)
    ts = torch.where(ts > 0, ts, torch.ones_like(ts))
    tsx = ts[..., None, None]
    blocks = w.reshape(*lead, r, k // 16, 16)
    bmax = blocks.abs().amax(dim=-1)
    sb = (bmax / (6.0 * tsx)).clamp(max=448.0).to(torch.float8_e4m3fn)
    sbv = sb.to(torch.float32)
    denom = (sbv * tsx)[..., None]
    q = torch.where(denom > 0, blocks / torch.where(denom > 0, denom, torch.ones_like(denom)),
                    torch.zeros_like(blocks))
    codes = _e2m1_codes(q).reshape(*lead, r, k)
    packed = codes[..., 0::2] | (codes[..., 1::2] << 4)
    return packed.contiguous(), sb.view(torch.uint8).contiguous(), ts


def _nvfp4_experts(n, inter, hidden, seed, device, std):
    """NVFP4 gate/up [n, 2I, H] and down [n, H, I] with per-projection tensor scales."""
    w13q = torch.empty((n, 2 * inter, hidden // 2), dtype=torch.uint8, device=device)
    w13s = torch.empty((n, 2 * inter, hidden // 16), dtype=torch.uint8, device=device)
    w13g = torch.empty((n, 2), dtype=torch.float32, device=device)
    w2q = torch.empty((n, hidden, inter // 2), dtype=torch.uint8, device=device)
    w2s = torch.empty((n, hidden, inter // 16), dtype=torch.uint8, device=device)
    w2g = torch.empty((n,), dtype=torch.float32, device=device)
    per = max(1, (1 << 29) // (3 * hidden * inter * 4))
    for s in range(0, n, per):
        e = min(n, s + per)
        g = _gen(seed * 1000003 + s, device)
        w13 = _normal((e - s, 2 * inter, hidden), g, device, std)
        w2 = _normal((e - s, hidden, inter), g, device, std)
        for p in range(2):  # gate rows, then up rows: one tensor scale each
            q, sc, ts = quantize_nvfp4(w13[:, p * inter:(p + 1) * inter])
            w13q[s:e, p * inter:(p + 1) * inter] = q
            w13s[s:e, p * inter:(p + 1) * inter] = sc
            w13g[s:e, p] = ts
        q, sc, ts = quantize_nvfp4(w2)
        w2q[s:e], w2s[s:e], w2g[s:e] = q, sc, ts
    return w13q, w13s, w13g, w2q, w2s, w2g


def router_bias(num_experts: int, seed: int, device="cpu", std: float = 0.05) -> torch.Tensor:
    """fp32 [E] selection bias for the bias-corrected sigmoid rule, ~N(0, std^2)
    (of the order of the gaps between the top sigmoid scores, so the bias changes
    which experts are chosen)."""
    return _normal((num_experts,), _gen(seed * 7919 + 11, device), device, std)


def quantize_fp8_block(w: torch.Tensor, block: int = 128):
    """Quantise float32 [..., R, K] to e4m3 codes with one fp32 scale per block x block
    tile: scale = amax_tile / 448 (1 for an all-zero tile), codes = the e4m3
    nearest-even rounding of w / scale. Returns (codes uint8 [..., R, K], scales
    float32 [..., R / block, K / block])."""
    *lead, r, k = w.shape
    t = w.reshape(*lead, r // block, block, k // block, block)
    amax = t.abs().amax(dim=(-3, -1))
    sc = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax)).to(torch.float32)
    q = (t / sc[..., :, None, :, None]).clamp(-448.0, 448.0).to(torch.float8_e4m3fn)
    return q.reshape(*lead, r, k).view(torch.uint8).contiguous(), sc.contiguous()


def _fp8_experts(n, inter, hidden, seed, device, std):
    """FP8 gate/up [n, 2I, H] and down [n, H, I] with their 128 x 128 block scales."""
    w13q = torch.empty((n, 2 * inter, hidden), dtype=torch.uint8, device=device)
    w13s = torch.empty((n, 2 * inter // 128, hidden // 128), dtype=torch.float32, device=device)
    w2q = torch.empty((n, hidden, inter), dtype=torch.uint8, device=device)
    w2s = torch.empty((n, hidden // 128, inter // 128), dtype=torch.float32, device=device)
    per = max(1, (1 << 29) // (3 * hidden * inter * 4))
    for s in range(0, n, per):
        e = min(n, s + per)
        g = _gen(seed * 1000003 + s, device)
        w13q[s:e], w13s[s:e] = quantize_fp8_block(_normal((e - s, 2 * inter, hidden), g, device, std))
        w2q[s:e], w2s[s:e] = quantize_fp8_block(_normal((e - s, hidden, inter), g, device, std))
    return w13q, w13s, w2q, w2s


def _transpose_experts(w: torch.Tensor, chunk_bytes=1 << 29) -> torch.Tensor:
    """[n, a, b] -> [n, b, a] contiguous, a few experts at a time."""
    n, a, b = w.shape
    out = torch.empty((n, b, a), dtype=w.dtype, device=w.device)
    per = max(1, chunk_bytes // max(1, a * b * w.element_size()))
    for s in range(0, n, per):
        out[s:s + per] = w[s:s + per].transpose(1, 2)
    return out


def make_layer(shape: LayerShape, seed: int, device="cpu", std: float = 0.02, w2_layout: str = "h_i") -> dict:
    """All weights of one layer as torch tensors on ``device``.

    ``w2_layout`` "i_h" stores the down matrices (and FP8 down scales) transposed,
    [E, I, H] ([E, I/128, H/128]), for the split-K kernel; the weight values are
    the same as with "h_i" for the same seed. The dict records the layout under
    "w2_layout".

    bf16:  router_w [E, H], w13 [E, 2I, H], w2 [E, H, I], sh_w13 [S, 2I, H], sh_w2 [S, H, I]
    nvfp4: router_w bf16 [E, H]; w13_q uint8 [E, 2I, H/2], w13_s uint8 [E, 2I, H/16],
           w13_gs f32 [E, 2], w2_q uint8 [E, H, I/2], w2_s uint8 [E, H, I/16],
           w2_gs f32 [E]; the same with an ``sh_`` prefix for the S shared experts.
    fp8:   router_w bf16 [E, H]; w13_q uint8 e4m3 [E, 2I, H], w13_s f32 [E, 2I/128, H/128],
           w2_q uint8 e4m3 [E, H, I], w2_s f32 [E, H/128, I/128]; ``sh_`` the same.
    """
    h, i, e, s = shape.hidden, shape.inter, shape.num_experts, shape.num_shared
    g = _gen(seed * 7919 + 1, device)
    layer = {"router_w": _normal((e, h), g, device, std).to(torch.bfloat16)}
    if shape.wdtype == "bf16":
        layer["w13"] = _bf16_experts(e, 2 * i, h, seed * 7919 + 2, device, std)
        layer["w2"] = _bf16_experts(e, h, i, seed * 7919 + 3, device, std)
        layer["sh_w13"] = _bf16_experts(s, 2 * i, h, seed * 7919 + 4, device, std)
        layer["sh_w2"] = _bf16_experts(s, h, i, seed * 7919 + 5, device, std)
    elif shape.wdtype == "nvfp4":
        names = ("w13_q", "w13_s", "w13_gs", "w2_q", "w2_s", "w2_gs")
        for n, t in zip(names, _nvfp4_experts(e, i, h, seed * 7919 + 2, device, std)):
            layer[n] = t
        for n, t in zip(names, _nvfp4_experts(s, i, h, seed * 7919 + 4, device, std)):
            layer["sh_" + n] = t
    elif shape.wdtype == "fp8":
        names = ("w13_q", "w13_s", "w2_q", "w2_s")
        for n, t in zip(names, _fp8_experts(e, i, h, seed * 7919 + 2, device, std)):
            layer[n] = t
        for n, t in zip(names, _fp8_experts(s, i, h, seed * 7919 + 4, device, std)):
            layer["sh_" + n] = t
    else:
        raise ValueError(f"unknown weight dtype {shape.wdtype!r}")
    if w2_layout == "i_h":
        if shape.wdtype == "nvfp4":
            raise ValueError("transposed down matrices are bf16 or fp8 only")
        for n in (("w2", "sh_w2") if shape.wdtype == "bf16" else ("w2_q", "w2_s", "sh_w2_q", "sh_w2_s")):
            layer[n] = _transpose_experts(layer[n])
    elif w2_layout != "h_i":
        raise ValueError(f"unknown down-matrix layout {w2_layout!r}")
    layer["w2_layout"] = w2_layout
    return layer
