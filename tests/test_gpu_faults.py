"""Failure paths on the GPU without faulting it: argument errors are caught on the
host before any launch, and a device-side wait that can never be satisfied (the
router results are withheld by a test flag) gives up after the wait limit,
reports MOE_ERR_DEVICE_TIMEOUT through the status word and leaves the context
usable for the next run."""

import ctypes
import time

import pytest
import torch

from moe_decode_layer_gb300 import _lib, synth
from moe_decode_layer_gb300.layer import MoEDecodeLayer
from tests import helpers

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tiny():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return synth.make_layer(synth.TINY, seed=0, device="cuda")


@pytest.mark.parametrize("sched", ["persistent", "phased", "interleaved", "flat", "pdl_chain", "chain", "split_k"])
@pytest.mark.parametrize("m", [1, 2])
def test_withheld_router_results_time_out(tiny, sched, m):
    layer = tiny
    if sched == "split_k":  # down matrices transposed: the split-K kernel
        layer = synth.make_layer(synth.TINY, seed=0, device="cuda", w2_layout="i_h")
        sched = "persistent"
    x = helpers.hidden_with_margin(tiny["router_w"], m, synth.TINY.top_k, seed=3)
    mod = MoEDecodeLayer(synth.TINY, layer, 2, sched=sched)
    xd = x.cuda()
    good = mod.run(xd, xd).clone()
    assert mod.status() == _lib.MOE_OK
    mod.set_option(_lib.MOE_OPT_WAIT_TIMEOUT_NS, 20_000_000)  # 20 ms
    mod.set_option(_lib.MOE_OPT_TEST_FLAGS, 1)
    t = time.time()
    mod.run(xd, xd)
    assert mod.status() == _lib.MOE_ERR_DEVICE_TIMEOUT
    assert time.time() - t < 5.0
    # the status word was cleared and the next normal run is correct
    mod.set_option(_lib.MOE_OPT_TEST_FLAGS, 0)
    out = mod.run(xd, xd)
    assert mod.status() == _lib.MOE_OK
    assert torch.equal(out, good)


def test_argument_errors(tiny):
    mod = MoEDecodeLayer(synth.TINY, tiny, 2)
    lib = mod.lib
    x = torch.zeros((2, synth.TINY.hidden), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(x)
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    run = lib.moe_decode_run
    assert run(mod.handle, p(x), p(x), p(out), 0, None, None, s) == _lib.MOE_ERR_INVALID_ARG
    assert run(mod.handle, p(x), p(x), p(out), 3, None, None, s) == _lib.MOE_ERR_INVALID_ARG
    assert run(mod.handle, None, p(x), p(out), 1, None, None, s) == _lib.MOE_ERR_INVALID_ARG
    mis = ctypes.c_void_p(x.data_ptr() + 2)
    assert run(mod.handle, mis, p(x), p(out), 1, None, None, s) == _lib.MOE_ERR_INVALID_ARG
    assert run(None, p(x), p(x), p(out), 1, None, None, s) == _lib.MOE_ERR_INVALID_ARG
    assert lib.moe_decode_set_option(mod.handle, _lib.MOE_OPT_SCHED, 7) == _lib.MOE_ERR_INVALID_ARG
    assert lib.moe_decode_set_option(mod.handle, _lib.MOE_OPT_RING_SLOTS, 1) == _lib.MOE_ERR_INVALID_ARG
    assert lib.moe_decode_set_option(mod.handle, 999, 0) == _lib.MOE_ERR_INVALID_ARG
    assert mod.status() == _lib.MOE_OK


def test_create_rejects_bad_weights(tiny):
    lib = _lib.load()
    cfg = _lib.Config(hidden=256, inter=128, num_experts=16, top_k=2, num_shared=1, max_rows=1,
                      wdtype=0, score=0, routed_scale=1.0, pre_rmsnorm=0, rms_eps=1e-6, sched=0)
    w = _lib.Weights()
    w.router_w = tiny["router_w"].data_ptr()
    w.w13 = tiny["w13"].data_ptr()
    w.w2 = tiny["w2"].data_ptr()
    h = ctypes.c_void_p()
    # shared expert weights missing
    assert lib.moe_decode_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(h)) == _lib.MOE_ERR_INVALID_ARG
    assert not h.value
    w.sh_w13 = tiny["sh_w13"].data_ptr()
    w.sh_w2 = tiny["sh_w2"].data_ptr() + 8  # misaligned
    assert lib.moe_decode_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(h)) == _lib.MOE_ERR_INVALID_ARG
    w.sh_w2 = tiny["sh_w2"].data_ptr()
    assert lib.moe_decode_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(h)) == _lib.MOE_OK
    assert lib.moe_decode_destroy(h) == _lib.MOE_OK
    assert lib.moe_decode_destroy(None) == _lib.MOE_OK
