"""Python handle over the C ABI: marshals torch tensors into pointers and calls
moe_decode_create / moe_decode_run. No arithmetic happens here.
"""

from __future__ import annotations

import ctypes

import torch

from . import _lib
from .synth import LayerShape


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_ptr(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


class MoEDecodeLayer:
    """One MoE layer's decode step on the current CUDA device.

    ``weights`` is the dict layout of :func:`synth.make_layer` (device tensors);
    ``score`` 1 selects the bias-corrected sigmoid rule, whose fp32 [E] bias is
    ``weights["router_bias"]``.
    The tensors are borrowed: this object keeps references so they outlive the
    C handle. ``sched``: "persistent" (one kernel; the expert-range or
    slot-interleaved kernel where that measured faster), "phased" (one kernel,
    phases in order), "interleaved" (one kernel, slot-interleaved whenever its
    layout fits), "flat" (the expert-range kernel whenever its layout fits),
    "pdl_chain" or "chain" (three kernels). Weights whose ``w2_layout`` is "i_h"
    (down matrices transposed) run the split-K kernel, under "persistent" only.
    """

    def __init__(self, shape: LayerShape, weights: dict, max_rows: int, sched: str = "persistent",
                 pre_rmsnorm: bool = False, rms_eps: float = 1e-6, routed_scale: float = 1.0,
                 score: int = 0):
        self.lib = _lib.load()
        self.shape = shape
        self.max_rows = max_rows
        self._weights = weights
        cfg = _lib.Config(hidden=shape.hidden, inter=shape.inter, num_experts=shape.num_experts,
                          top_k=shape.top_k, num_shared=shape.num_shared, max_rows=max_rows,
                          wdtype=_lib.WDTYPE[shape.wdtype],
                          score=score, routed_scale=routed_scale,
                          pre_rmsnorm=int(pre_rmsnorm), rms_eps=rms_eps,
                          sched=_lib.SCHED_NAMES["persistent" if sched in ("phased", "interleaved", "flat")
                                                  else sched],
                          w2_layout=_lib.W2_LAYOUT[weights.get("w2_layout", "h_i")])
        w = _lib.Weights()
        g = weights.get
        w.router_w = _ptr(g("router_w"))
        w.router_bias = _ptr(g("router_bias"))
        if shape.wdtype == "bf16":
            w.w13, w.w2 = _ptr(g("w13")), _ptr(g("w2"))
            if shape.num_shared:
                w.sh_w13, w.sh_w2 = _ptr(g("sh_w13")), _ptr(g("sh_w2"))
        elif shape.wdtype == "fp8":
            w.w13, w.w13_scale = _ptr(g("w13_q")), _ptr(g("w13_s"))
            w.w2, w.w2_scale = _ptr(g("w2_q")), _ptr(g("w2_s"))
            if shape.num_shared:
                w.sh_w13, w.sh_w13_scale = _ptr(g("sh_w13_q")), _ptr(g("sh_w13_s"))
                w.sh_w2, w.sh_w2_scale = _ptr(g("sh_w2_q")), _ptr(g("sh_w2_s"))
        else:
            w.w13, w.w13_scale, w.w13_gscale = _ptr(g("w13_q")), _ptr(g("w13_s")), _ptr(g("w13_gs"))
            w.w2, w.w2_scale, w.w2_gscale = _ptr(g("w2_q")), _ptr(g("w2_s")), _ptr(g("w2_gs"))
            if shape.num_shared:
                w.sh_w13, w.sh_w13_scale, w.sh_w13_gscale = (_ptr(g("sh_w13_q")), _ptr(g("sh_w13_s")),
                                                             _ptr(g("sh_w13_gs")))
                w.sh_w2, w.sh_w2_scale, w.sh_w2_gscale = (_ptr(g("sh_w2_q")), _ptr(g("sh_w2_s")),
                                                          _ptr(g("sh_w2_gs")))
        self._cfg = cfg
        h = ctypes.c_void_p()
        _lib.check(self.lib.moe_decode_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(h)),
                   "moe_decode_create")
        self.handle = h
        if sched in ("phased", "interleaved"):  # the single kernel in phase order / always interleaved
            self.set_option(_lib.MOE_OPT_FLAT, 0)
            self.set_option(_lib.MOE_OPT_INTERLEAVE, 0 if sched == "phased" else 2)
        elif sched == "flat":  # the expert-range kernel whenever it fits
            self.set_option(_lib.MOE_OPT_FLAT, 2)

    # ------------------------------------------------------------------ runs
    def run(self, x: torch.Tensor, residual: torch.Tensor | None = None, out: torch.Tensor | None = None,
            topk_idx: torch.Tensor | None = None, topk_w: torch.Tensor | None = None, stream=None):
        """Enqueue one step; returns ``out`` (allocated when not given)."""
        residual = x if residual is None else residual
        if out is None:
            out = torch.empty_like(x)
        for t in (x, residual, out):
            if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
                raise ValueError("x, residual and out must be contiguous bf16 CUDA tensors")
        m = x.shape[0]
        _lib.check(self.lib.moe_decode_run(self.handle, _ptr(x), _ptr(residual), _ptr(out), m,
                                           _ptr(topk_idx), _ptr(topk_w), _stream_ptr(stream)),
                   "moe_decode_run")
        return out

    def run_host(self, x: torch.Tensor, residual: torch.Tensor, out: torch.Tensor,
                 topk_idx: torch.Tensor | None = None, topk_w: torch.Tensor | None = None, stream=None):
        """One step from host (CPU) tensors, copies included; synchronises."""
        for t in (x, residual, out):
            if t.dtype != torch.bfloat16 or t.is_cuda or not t.is_contiguous():
                raise ValueError("run_host takes contiguous bf16 CPU tensors")
        _lib.check(self.lib.moe_decode_run_host(self.handle, _ptr(x), _ptr(residual), _ptr(out), x.shape[0],
                                                _ptr(topk_idx), _ptr(topk_w), _stream_ptr(stream)),
                   "moe_decode_run_host")
        return out

    def host_copy_bytes(self, m: int) -> tuple[int, int]:
        """Bytes run_host copies per call with m rows and x as the residual: (in, out).
        Out is one block from the status words to the m-th output row: the rest of the
        CTRL_WORDS control words, topk_idx and topk_w for max_rows rows (each padded
        to 16 bytes), then the output rows."""
        pad16 = lambda v: (v + 15) // 16 * 16  # noqa: E731
        k = self.shape.top_k
        out = _lib.CTRL_WORDS * 4 - 8 + 2 * pad16(self.max_rows * k * 4) + m * self.shape.hidden * 2
        return m * self.shape.hidden * 2, out

    def status(self, stream=None) -> int:
        """Synchronise and return (and clear) the device status code."""
        return self.lib.moe_decode_get_status(self.handle, _stream_ptr(stream))

    def set_option(self, option: int, value: int) -> None:
        _lib.check(self.lib.moe_decode_set_option(self.handle, option, value), "moe_decode_set_option")

    def info(self, what: int) -> int:
        v = ctypes.c_int64()
        _lib.check(self.lib.moe_decode_get_info(self.handle, what, ctypes.byref(v)), "moe_decode_get_info")
        return v.value

    def close(self) -> None:
        if getattr(self, "handle", None):
            self.lib.moe_decode_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
