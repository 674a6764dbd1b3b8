"""Speculative expert prefetch ("Muse Spark Open Ultrafast", section "Speculative
expert prefetching"): while a run routes, its producers pull into L2 the experts
the handle's previous run used most. The results must not change, and the list
each run leaves for the next is checked against the routing the run reported.
"""

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


def _predicted(mod):
    return [mod.info(_lib.MOE_INFO_PREDICTED + i) for i in range(16)]


def _expected(idx: torch.Tensor, p: int):
    """Most token rows first, ties to the lower id; one row: selection order."""
    if idx.shape[0] == 1:
        sel = idx[0].tolist()[:p]
    else:
        count = {}
        for e in idx.flatten().tolist():
            count[e] = count.get(e, 0) + 1
        sel = sorted(count, key=lambda e: (-count[e], e))[:p]
    return sel + [-1] * (16 - len(sel))


CASES = [("tiny", "persistent", 1), ("tiny", "persistent", 6), ("tiny", "pdl_chain", 3),
         ("tiny", "split_k", 1), ("tiny", "split_k", 5), ("ling", "persistent", 1), ("ling", "persistent", 6)]


@pytest.mark.parametrize("name,sched,m", CASES)
def test_prefetch_keeps_results_and_predicts_from_the_previous_run(name, sched, m):
    shape = synth.TINY if name == "tiny" else synth.LING
    layout = "i_h" if sched == "split_k" else "h_i"
    layer = synth.make_layer(shape, seed=61, device="cuda", w2_layout=layout)
    s = "persistent" if sched == "split_k" else sched
    plain = MoEDecodeLayer(shape, layer, m, sched=s)
    pf = MoEDecodeLayer(shape, layer, m, sched=s)
    p = min(4, shape.num_experts)
    pf.set_option(_lib.MOE_OPT_PREFETCH_EXPERTS, p)
    assert pf.info(_lib.MOE_OPT_PREFETCH_EXPERTS) == p
    assert _predicted(pf) == [-1] * 16  # nothing routed yet
    for step in range(3):
        x = helpers.hidden_with_margin(layer["router_w"], m, shape.top_k, seed=610 + 10 * step + m, rho=0.5)
        xd = x.cuda()
        a = plain.run(xd, xd)
        idx = torch.empty((m, shape.top_k), dtype=torch.int32, device="cuda")
        b = pf.run(xd, xd, None, idx)
        assert pf.status() == _lib.MOE_OK and plain.status() == _lib.MOE_OK
        assert torch.equal(a, b)
        assert _predicted(pf) == _expected(idx.cpu(), p)
    if name == "tiny":
        ref, _, _ = helpers.oracle_layer(shape, layer, x, x)
        helpers.assert_close(b.cpu(), ref)
    del plain, pf, layer
    torch.cuda.empty_cache()


def test_prefetch_option_range():
    layer = synth.make_layer(synth.TINY, seed=63, device="cuda")
    mod = MoEDecodeLayer(synth.TINY, layer, 2)
    for bad in (-1, 17):
        with pytest.raises(_lib.MoEDecodeError):
            mod.set_option(_lib.MOE_OPT_PREFETCH_EXPERTS, bad)
    mod.set_option(_lib.MOE_OPT_PREFETCH_EXPERTS, 16)
    assert mod.info(_lib.MOE_OPT_PREFETCH_EXPERTS) == 16
