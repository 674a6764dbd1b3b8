"""moe_decode_run_static, the entry point that allocates nothing (its scratch is
a fixed array of device memory defined in the library), on two calls in a row
with different inputs: against the C++ float64 oracle within the layer
tolerances, and bit for bit against the handle-based moe_decode_run on the same
weights and inputs (same kernel, same plan, so any difference would be state
left over in the shared array). Kept in a file of its own that pytest collects
last."""

import ctypes

import pytest
import torch

from moe_decode_layer_gb300 import _lib, synth
from moe_decode_layer_gb300.layer import MoEDecodeLayer
from tests import helpers

pytestmark = pytest.mark.gpu


def _cfg(shape, max_rows):
    return _lib.Config(hidden=shape.hidden, inter=shape.inter, num_experts=shape.num_experts,
                       top_k=shape.top_k, num_shared=shape.num_shared, max_rows=max_rows,
                       wdtype=_lib.MOE_W_BF16 if shape.wdtype == "bf16" else _lib.MOE_W_NVFP4,
                       score=0, routed_scale=1.0, pre_rmsnorm=0, rms_eps=1e-6, sched=0)


def _weights(shape, layer):
    w = _lib.Weights()
    p = lambda k: layer[k].data_ptr() if k in layer else None  # noqa: E731
    w.router_w = p("router_w")
    if shape.wdtype == "bf16":
        w.w13, w.w2, w.sh_w13, w.sh_w2 = p("w13"), p("w2"), p("sh_w13"), p("sh_w2")
    else:
        w.w13, w.w13_scale, w.w13_gscale = p("w13_q"), p("w13_s"), p("w13_gs")
        w.w2, w.w2_scale, w.w2_gscale = p("w2_q"), p("w2_s"), p("w2_gs")
        if shape.num_shared:
            w.sh_w13, w.sh_w13_scale, w.sh_w13_gscale = p("sh_w13_q"), p("sh_w13_s"), p("sh_w13_gs")
            w.sh_w2, w.sh_w2_scale, w.sh_w2_gscale = p("sh_w2_q"), p("sh_w2_s"), p("sh_w2_gs")
    return w


def _run_static(lib, cfg, w, x, m, k):
    out = torch.empty_like(x)
    idx = torch.empty((m, k), dtype=torch.int32, device="cuda")
    wt = torch.empty((m, k), dtype=torch.float32, device="cuda")
    vp = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    st = lib.moe_decode_run_static(ctypes.byref(cfg), ctypes.byref(w), vp(x), vp(x), vp(out), m, vp(idx), vp(wt),
                                   ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == _lib.MOE_OK, _lib.status_string(st)
    return out, idx, wt


@pytest.mark.parametrize("case", ["tiny_m2", "ling_e64_m1", "ling_e64_m6", "nvfp4_small_m3"])
def test_static_entry_matches_handle_entry(case):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = _lib.load()
    shape, m = {
        "tiny_m2": (synth.TINY, 2),
        "ling_e64_m1": (synth.LING_E64, 1),  # bf16, one row: the slot-interleaved kernel
        "ling_e64_m6": (synth.LING_E64, 6),
        "nvfp4_small_m3": (synth.LayerShape(hidden=512, inter=256, num_experts=32, top_k=4, num_shared=1,
                                            wdtype="nvfp4"), 3),
    }[case]
    layer = synth.make_layer(shape, seed=23, device="cuda")
    mod = MoEDecodeLayer(shape, layer, m)
    cfg, w = _cfg(shape, m), _weights(shape, layer)
    for call, seed in enumerate((101, 202)):  # two calls in a row, different inputs
        x = helpers.hidden_with_margin(layer["router_w"], m, shape.top_k, seed=seed, rho=0.5).cuda()
        ref_idx = torch.empty((m, shape.top_k), dtype=torch.int32, device="cuda")
        ref_w = torch.empty((m, shape.top_k), dtype=torch.float32, device="cuda")
        ref = mod.run(x, x, None, ref_idx, ref_w)
        assert mod.status() == _lib.MOE_OK
        out, idx, wt = _run_static(lib, cfg, w, x, m, shape.top_k)
        oref, oidx, ow = helpers.oracle_layer(shape, layer, x.cpu(), x.cpu())
        helpers.assert_routing(idx.cpu(), wt.cpu(), oidx, ow)
        helpers.assert_close(out.cpu(), oref, what=f"{case} call {call}")
        assert torch.equal(out, ref), f"{case} call {call}: differs from the handle entry"
        assert torch.equal(idx, ref_idx) and torch.equal(wt, ref_w)
    mod.close()


def test_static_entry_rejects_oversized_scratch():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = _lib.load()
    # 8 rows x (16 routed + 1 shared) experts x 3072 fp32 h values in 4 copies: 6.7 MB,
    # more than the array holds; the layout itself fits in shared memory
    big = _lib.Config(hidden=1024, inter=3072, num_experts=1024, top_k=16, num_shared=1, max_rows=8,
                      wdtype=0, score=0, routed_scale=1.0, pre_rmsnorm=0, rms_eps=1e-6, sched=0)
    w = _lib.Weights()
    x = torch.zeros((1, 1024), dtype=torch.bfloat16, device="cuda")
    vp = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    st = lib.moe_decode_run_static(ctypes.byref(big), ctypes.byref(w), vp(x), vp(x), vp(x), 1, None, None,
                                   ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == _lib.MOE_ERR_UNSUPPORTED


def test_static_entry_refuses_stream_capture():
    """The call waits for its step, which a stream under capture cannot do: it
    must refuse before any device work and leave the capture intact."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = _lib.load()
    shape = synth.TINY
    layer = synth.make_layer(shape, seed=29, device="cuda")
    cfg, w = _cfg(shape, 1), _weights(shape, layer)
    x = helpers.hidden_with_margin(layer["router_w"], 1, shape.top_k, seed=5).cuda()
    out = torch.empty_like(x)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    vp = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    with torch.cuda.graph(g, stream=s):
        st = lib.moe_decode_run_static(ctypes.byref(cfg), ctypes.byref(w), vp(x), vp(x), vp(out), 1, None, None,
                                       ctypes.c_void_p(s.cuda_stream))
    assert st == _lib.MOE_ERR_INVALID_ARG
    # outside capture the same call works
    ref = _run_static(lib, cfg, w, x, 1, shape.top_k)[0]
    oref, _, _ = helpers.oracle_layer(shape, layer, x.cpu(), x.cpu())
    helpers.assert_close(ref.cpu(), oref)
