"""Launch planning on the host (no GPU): for a sweep of supported configs and device
sizes, the planned shared-memory layout of both single-kernel schedules fits the device,
every stage fits its ring slot, and the barrier and counter index ranges stay inside their
arrays. moe_decode_plan is the library's own planner, called through the C ABI."""

import ctypes
import itertools

import numpy as np
import pytest

from moe_decode_layer_gb300 import _lib

K_MAX_SLOTS = 64        # full / empty barrier arrays
K_HSLOT_BAR = 32        # per-slot h barriers start at this full-barrier index
K_SLOT_COUNTERS = 160   # per-slot counters in the control words
K_NC = 12               # consumer warps


def _cfg(h, i, e, k, s, m, fp4):
    return _lib.Config(hidden=h, inter=i, num_experts=e, top_k=k, num_shared=s, max_rows=m,
                       wdtype=_lib.MOE_W_NVFP4 if fp4 else _lib.MOE_W_BF16, score=0, routed_scale=1.0,
                       pre_rmsnorm=0, rms_eps=1e-6, sched=0)


def _plan(lib, cfg, sms, optin, ilv):
    info = _lib.PlanInfo()
    st = lib.moe_decode_plan(ctypes.byref(cfg), sms, optin, ilv, ctypes.byref(info))
    return st, info


def _sweep():
    for fp4, h, i, e, k, s, m in itertools.product(
            (False, True), (256, 1024, 2560, 4096), (64, 128, 256, 768, 1024, 3072), (16, 64, 512, 1024),
            (1, 2, 8, 16), (0, 1, 4), (1, 6, 8)):
        if k > e:
            continue
        yield fp4, h, i, e, k, s, m


@pytest.mark.parametrize("sms,optin", [(152, 232448), (148, 232448), (132, 232448), (152, 166912)])
def test_planned_layouts_fit(sms, optin):
    lib = _lib.load()
    n_checked = n_ilv = n_unfit = 0
    for fp4, h, i, e, k, s, m in _sweep():
        cfg = _cfg(h, i, e, k, s, m, fp4)
        if lib.moe_decode_config_check(ctypes.byref(cfg)) != _lib.MOE_OK:
            continue
        pair = 2 * (h // 2 + h // 16) if fp4 else 4 * h
        down_row = (i // 2 + i // 16) if fp4 else 2 * i
        for ilv in (0, 1):
            st, p = _plan(lib, cfg, sms, optin, ilv)
            if st != _lib.MOE_OK:
                assert st == _lib.MOE_ERR_UNSUPPORTED, (cfg, ilv, st)
                if not ilv:
                    # on a GB300 only the largest rows at many token rows outgrow the
                    # shared memory (with less shared memory, more do)
                    if optin >= 232448:
                        assert m >= 6 and h * i >= 2560 * 3072, (h, i, e, k, s, m, fp4, sms, optin)
                    else:
                        assert m >= 6, (h, i, e, k, s, m, fp4, sms, optin)
                    n_unfit += 1
                continue
            what = f"{'nvfp4' if fp4 else 'bf16'} H={h} I={i} E={e} k={k} S={s} M={m} ilv={ilv} sms={sms}"
            assert p.smem_bytes <= optin, what
            assert p.slot_bytes % 128 == 0, what
            assert p.ring_slots >= (3 if ilv else 2), what
            assert p.ring_slots + max(p.extra_slots, p.down_slot_in_x) <= K_MAX_SLOTS, what
            assert 1 <= p.pairs_per_stage <= K_NC and p.pairs_per_stage * pair <= p.slot_bytes, what
            assert 1 <= p.router_pairs_per_stage <= K_NC // 2, what
            assert p.router_pairs_per_stage * 4 * h <= p.slot_bytes, what
            assert p.slots_max == s + min(e, m * k) and p.pairs_max == s * m + m * k, what
            if p.h_per_slot:
                assert p.ring_slots + max(p.extra_slots, p.down_slot_in_x) <= K_HSLOT_BAR, what
                assert p.slots_max <= K_MAX_SLOTS - K_HSLOT_BAR, what
            if ilv:
                n_ilv += 1
                rows = -(-h // sms)
                assert p.down_rows_per_stage == rows, what
                assert p.down_h_offset % 16 == 0 and p.down_h_offset >= rows * down_row, what
                assert p.down_h_offset + m * i * 4 <= p.slot_bytes, what
                assert p.slots_max <= K_SLOT_COUNTERS and p.lag >= 1 and p.threads == 480, what
                assert p.h_pairs == 0 and p.extra_slots == 0 and p.down_slot_in_x == 0, what
            else:
                assert p.down_rows_per_stage * down_row <= p.slot_bytes, what
                assert p.h_buffers in (1, 2) and p.h_pairs >= m, what
                if p.h_buffers == 2:
                    assert p.h_pairs < p.pairs_max, what
                assert p.threads == 416, what
            n_checked += 1
    assert n_checked > 500 and n_ilv > 100 and n_unfit < n_checked // 10


def _fp8_cfg(h, i, e, k, s, m):
    return _lib.Config(hidden=h, inter=i, num_experts=e, top_k=k, num_shared=s, max_rows=m,
                       wdtype=_lib.MOE_W_FP8_BLOCK, score=0, routed_scale=1.0, pre_rmsnorm=0, rms_eps=1e-6,
                       sched=0)


def _staged(nbytes):
    """Scale bytes that ride behind an FP8 stage: whole 16-byte multiples up to 4 KB."""
    return nbytes if nbytes % 16 == 0 and nbytes <= 4096 else 0


@pytest.mark.parametrize("sms,optin", [(152, 232448), (132, 232448)])
def test_planned_fp8_layouts_fit(sms, optin):
    """FP8 weights: each expert's block-scale matrix may ride behind its gate/up and
    down stages, so a stage is its rows plus those bytes. Every planned stage, with
    its scales, fits its ring slot; the interleaved kernel's h rows start after the
    staged down scales; the x area takes a down-phase slot only when a down stage
    (rows and scales) fits it."""
    lib = _lib.load()
    n_checked = 0
    for h, i, e, k, s, m in itertools.product((1024, 2560, 4096), (128, 768, 1024, 3072), (64, 512),
                                               (2, 8), (0, 1), (1, 6, 8)):
        cfg = _fp8_cfg(h, i, e, k, s, m)
        if lib.moe_decode_config_check(ctypes.byref(cfg)) != _lib.MOE_OK:
            continue
        s13 = _staged((2 * i // 128) * (h // 128) * 4)
        s2 = _staged((h // 128) * (i // 128) * 4)
        for ilv in (0, 1):
            st, p = _plan(lib, cfg, sms, optin, ilv)
            if st != _lib.MOE_OK:
                assert st == _lib.MOE_ERR_UNSUPPORTED
                continue
            what = f"fp8 H={h} I={i} E={e} k={k} S={s} M={m} ilv={ilv} sms={sms}"
            assert p.smem_bytes <= optin and p.slot_bytes % 128 == 0, what
            assert p.pairs_per_stage * 2 * h + s13 <= p.slot_bytes, what
            rows_bytes = -(-p.down_rows_per_stage * i // 16) * 16
            if ilv:
                assert p.down_h_offset % 16 == 0 and p.down_h_offset >= rows_bytes + s2, what
                assert p.down_h_offset + m * i * 4 <= p.slot_bytes, what
            else:
                assert rows_bytes + s2 <= p.slot_bytes, what
                if p.down_slot_in_x:
                    assert m * h * 2 >= rows_bytes + s2, what
            n_checked += 1
    assert n_checked > 50


def test_fp8_ling_layer_stages_its_scales():
    """The Ling-shaped FP8 layer: 960 B of gate/up and 480 B of down scales per expert
    ride with the stages, and six gate/up pairs still fit a slot."""
    lib = _lib.load()
    for m in (1, 6):
        st, p = _plan(lib, _fp8_cfg(2560, 768, 512, 8, 1, m), 152, 232448, 0)
        assert st == _lib.MOE_OK and p.pairs_per_stage == 6
        assert 6 * 2 * 2560 + 960 <= p.slot_bytes and 17 * 768 + 480 <= p.slot_bytes
        st, q = _plan(lib, _fp8_cfg(2560, 768, 512, 8, 1, m), 152, 232448, 1)
        assert st == _lib.MOE_OK and q.down_h_offset == 17 * 768 + 480


@pytest.mark.parametrize("sms,optin", [(152, 232448), (132, 232448), (152, 166912)])
def test_planned_flat_layouts_fit(sms, optin):
    """The expert-range kernel's layout: bf16 weights, at most one shared expert,
    no more routed slots than CTAs, I <= 1024; then it fits shared memory, every
    stage fits a ring slot and the slot counters stay inside the control words."""
    lib = _lib.load()
    n_flat = 0
    for fp4, h, i, e, k, s, m in _sweep():
        cfg = _cfg(h, i, e, k, s, m, fp4)
        if lib.moe_decode_config_check(ctypes.byref(cfg)) != _lib.MOE_OK:
            continue
        st, p = _plan(lib, cfg, sms, optin, 2)
        what = f"H={h} I={i} E={e} k={k} S={s} M={m} fp4={fp4} sms={sms}"
        covered = not fp4 and s <= 1 and min(e, m * k) <= sms and i <= 1024
        if st != _lib.MOE_OK:
            assert st == _lib.MOE_ERR_UNSUPPORTED, what
            # on a GB300's shared memory only the kernel's coverage, a base layout that
            # does not fit either, or three large h buffers (M x I >= 6144) rule it out
            base, _ = _plan(lib, cfg, sms, optin, 0)
            assert base != _lib.MOE_OK or not covered or optin < 232448 or m * i >= 6144 or m * h >= 16384, what
            continue
        assert covered, what
        n_flat += 1
        assert p.smem_bytes <= optin and p.slot_bytes % 128 == 0, what
        assert 3 <= p.ring_slots <= K_MAX_SLOTS, what
        assert 1 <= p.pairs_per_stage <= K_NC and p.pairs_per_stage * 4 * h <= p.slot_bytes, what
        assert p.router_pairs_per_stage * 4 * h <= p.slot_bytes, what
        assert p.down_rows_per_stage >= 1 and p.down_rows_per_stage * 2 * i <= p.slot_bytes, what
        assert p.slots_max <= K_SLOT_COUNTERS and p.threads == 480 and p.lag == 0, what
    assert n_flat > 200


def test_plan_of_the_benchmarked_layers():
    """The Ling-shaped layer on 152 SMs: both single-kernel layouts fit, with the
    numbers the kernels were measured with."""
    lib = _lib.load()
    for m in (1, 6):
        cfg = _cfg(2560, 768, 512, 8, 1, m, False)
        st, p = _plan(lib, cfg, 152, 232448, 0)
        assert st == _lib.MOE_OK and p.slot_bytes == 30720 and p.pairs_per_stage == 3
        assert p.down_rows_per_stage == 17
        st, q = _plan(lib, cfg, 152, 232448, 1)
        assert st == _lib.MOE_OK and q.lag == 5 and q.down_rows_per_stage == 17
    st, p = _plan(lib, _cfg(2560, 768, 512, 8, 1, 1, False), 152, 232448, 0)
    assert p.ring_slots == 6 and p.h_pairs == 9 and p.h_buffers == 1
    # the expert-range kernel: 30 KB stages of 3 gate/up pairs or 20 down rows
    for m, slots in ((1, 6), (6, 4)):
        st, f = _plan(lib, _cfg(2560, 768, 512, 8, 1, m, False), 152, 232448, 2)
        assert st == _lib.MOE_OK and f.slot_bytes == 30720 and f.pairs_per_stage == 3
        assert f.down_rows_per_stage == 20 and f.ring_slots == slots, (m, f.ring_slots)


def test_plan_rejects_bad_arguments():
    lib = _lib.load()
    cfg = _cfg(2560, 768, 512, 8, 1, 1, False)
    info = _lib.PlanInfo()
    assert lib.moe_decode_plan(ctypes.byref(cfg), 0, 232448, 0, ctypes.byref(info)) == _lib.MOE_ERR_INVALID_ARG
    assert lib.moe_decode_plan(ctypes.byref(cfg), 152, 232448, 3, ctypes.byref(info)) == _lib.MOE_ERR_INVALID_ARG
    assert lib.moe_decode_plan(ctypes.byref(cfg), 152, 232448, 0, None) == _lib.MOE_ERR_INVALID_ARG
    bad = _cfg(2560, 776, 512, 8, 1, 1, False)  # 97 threads per down group
    assert lib.moe_decode_plan(ctypes.byref(bad), 152, 232448, 0, ctypes.byref(info)) == _lib.MOE_ERR_UNSUPPORTED


# ---------------------------------------------------------------------------
# split-K kernel (down matrices transposed)
# ---------------------------------------------------------------------------


def _sk_cfg(**kw):
    base = dict(hidden=2560, inter=768, num_experts=512, top_k=8, num_shared=1, max_rows=8, wdtype=0, score=0,
                routed_scale=1.0, pre_rmsnorm=0, rms_eps=1e-6, sched=0, w2_layout=_lib.MOE_W2_I_H)
    base.update(kw)
    return _lib.Config(**base)


def _split_rows(costs, grid):
    """Rows (items) of each CTA under the routed cost split: the item boundaries
    of CTA b are the first items at or after b / grid and (b + 1) / grid of the
    total cost (the rule the union applies on the device)."""
    cum = np.concatenate([[0], np.cumsum(costs)])
    total = int(cum[-1])
    bounds = [int(np.searchsorted(cum, total * b // grid, side="left")) for b in range(grid + 1)]
    return [bounds[b + 1] - bounds[b] for b in range(grid)]


@pytest.mark.parametrize("maxm", [1, 6, 8])
def test_split_k_h_rows_bound_covers_the_cost_split(maxm):
    """The planner's h-row bound holds for the shared share plus the largest
    routed share the cost split can give: items whose row counts are all 1 next
    to items with maxm rows (the most rows per unit of cost), at several expert
    counts."""
    lib = _lib.load()
    info = _lib.PlanInfo()
    assert lib.moe_decode_plan(ctypes.byref(_sk_cfg(max_rows=maxm)), 152, 232448, 0, ctypes.byref(info)) == 0
    assert info.h_rows_max > 0 and info.down_t_rows_per_stage > 0
    I, S, grid, base = 768, 1, 152, 6
    shared = -(-S * I // grid)
    rng = np.random.default_rng(maxm)
    worst = 0
    for n_slots in (1, 7, 8 * maxm // 2, 8 * maxm):
        for trial in range(4):
            rows = rng.integers(1, maxm + 1, size=n_slots)
            if trial == 0:
                rows[:] = 1
            if trial == 1:
                rows[: n_slots // 2] = maxm
            costs = np.repeat(base + rows, I)
            worst = max(worst, max(_split_rows(costs, grid)))
    assert shared + worst <= info.h_rows_max


def test_split_k_plan_fits_and_refuses():
    lib = _lib.load()
    info = _lib.PlanInfo()
    for m in (1, 6, 8):
        assert lib.moe_decode_plan(ctypes.byref(_sk_cfg(max_rows=m)), 152, 232448, 0, ctypes.byref(info)) == 0
        assert info.smem_bytes <= 232448 and info.ring_slots >= 3 and info.threads == 416
    # one layout for transposed down rows: no interleaved / expert-range variant
    assert lib.moe_decode_plan(ctypes.byref(_sk_cfg()), 152, 232448, 1, ctypes.byref(info)) == _lib.MOE_ERR_UNSUPPORTED
    for kw in (dict(wdtype=1), dict(hidden=4096), dict(sched=1), dict(w2_layout=2), dict(wdtype=2, inter=704)):
        assert lib.moe_decode_config_check(ctypes.byref(_sk_cfg(**kw))) == _lib.MOE_ERR_UNSUPPORTED
    assert lib.moe_decode_config_check(ctypes.byref(_sk_cfg(wdtype=2))) == 0
    assert lib.moe_decode_config_check(ctypes.byref(_sk_cfg(hidden=3072, inter=1000))) == 0
