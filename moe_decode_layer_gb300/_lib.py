"""ctypes view of the C ABI in include/moe_decode.h (libmoe_decode.so).

Loading fails loudly when the library cannot be built or opened: there is no
fallback implementation behind these names.
"""

from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_CUDA = 3
MOE_ERR_DEVICE_TIMEOUT = 4
MOE_ERR_OOM = 5

MOE_W_BF16 = 0
MOE_W_NVFP4 = 1
MOE_W_FP8_BLOCK = 2
WDTYPE = {"bf16": MOE_W_BF16, "nvfp4": MOE_W_NVFP4, "fp8": MOE_W_FP8_BLOCK}
MOE_SCORE_SOFTMAX_TOPK_RENORM = 0
MOE_SCORE_SIGMOID_BIAS = 1
MOE_W2_H_I = 0
MOE_W2_I_H = 1
W2_LAYOUT = {"h_i": MOE_W2_H_I, "i_h": MOE_W2_I_H}
MOE_SCHED_PERSISTENT = 0
MOE_SCHED_PDL_CHAIN = 1
MOE_SCHED_CHAIN = 2
SCHED_NAMES = {"persistent": MOE_SCHED_PERSISTENT, "pdl_chain": MOE_SCHED_PDL_CHAIN,
               "chain": MOE_SCHED_CHAIN}

MOE_OPT_SCHED = 1
MOE_OPT_WAIT_TIMEOUT_NS = 2
MOE_OPT_TEST_FLAGS = 3
MOE_OPT_RING_SLOTS = 4
MOE_OPT_STAMPS = 5
MOE_OPT_INTERLEAVE = 6
MOE_OPT_FLAT = 7
MOE_OPT_PREFETCH_EXPERTS = 8
STAMP_NAMES = {0: "start", 1: "x_loaded", 2: "R_done", 3: "routed", 4: "U_done", 5: "D_first",
               6: "D_done", 8: "prod_R_issued", 9: "prod_route", 10: "prod_U_issued",
               11: "prod_D_issued", 12: "logits_seen", 13: "topk_row0", 14: "ucount_full",
               16: "logits_stored", 17: "U_first_data",
               19: "D_summed"}
STAMP_COUNTS = {7: "D_hwait_us(t0)", 20: "D_math_us(t0)", 21: "D_bar_us(t0)", 22: "D_wait_us(warp0)",
                23: "sm_clock_mhz"}
STAMP_SLOTS = 24
CTRL_WORDS = 176  # control words at the start of a handle's scratch
MOE_INFO_GRID = 16
MOE_INFO_THREADS = 17
MOE_INFO_SMEM = 18
MOE_INFO_RING_SLOTS = 19
MOE_INFO_SLOT_BYTES = 20
MOE_INFO_KERNELS_PER_RUN = 21
MOE_INFO_SCRATCH_BYTES = 22
MOE_INFO_INTERLEAVED_ROWS = 23
MOE_INFO_FLAT_ROWS = 24
MOE_INFO_SPLIT_K = 25
MOE_INFO_PREDICTED = 32
STATIC_SCRATCH_BYTES = 4 << 20

EXPORTS = ("moe_decode_config_check", "moe_decode_plan", "moe_decode_create", "moe_decode_run", "moe_decode_run_host",
           "moe_decode_run_static",
           "moe_decode_get_status", "moe_decode_set_option", "moe_decode_get_info",
           "moe_decode_destroy", "moe_decode_status_string", "moe_decode_abi_version")


class Config(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("inter", ctypes.c_int32),
                ("num_experts", ctypes.c_int32), ("top_k", ctypes.c_int32),
                ("num_shared", ctypes.c_int32), ("max_rows", ctypes.c_int32),
                ("wdtype", ctypes.c_int32), ("score", ctypes.c_int32),
                ("routed_scale", ctypes.c_float), ("pre_rmsnorm", ctypes.c_int32),
                ("rms_eps", ctypes.c_float), ("sched", ctypes.c_int32),
                ("w2_layout", ctypes.c_int32)]


class Weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "router_w", "w13", "w2", "w13_scale", "w2_scale", "w13_gscale", "w2_gscale",
        "sh_w13", "sh_w2", "sh_w13_scale", "sh_w2_scale", "sh_w13_gscale", "sh_w2_gscale", "router_bias")]


class PlanInfo(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "smem_bytes", "ring_slots", "slot_bytes", "extra_slots", "down_slot_in_x", "pairs_per_stage",
        "router_pairs_per_stage", "down_rows_per_stage", "h_pairs", "h_buffers", "h_per_slot", "slots_max",
        "pairs_max", "lag", "down_h_offset", "threads", "h_rows_max", "down_t_rows_per_stage")]


class MoEDecodeError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


_lock = threading.Lock()
_lib = None


def load(build_if_stale: bool = True) -> ctypes.CDLL:
    """Open libmoe_decode.so (building it first if sources are newer)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if build_if_stale and not _build.up_to_date():
            _build.build()
        if not os.path.exists(_build.LIB):
            raise RuntimeError(f"{_build.LIB} is missing: build the CUDA library first "
                               "(python -m moe_decode_layer_gb300.build)")
        lib = ctypes.CDLL(_build.LIB)
        vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        lib.moe_decode_config_check.argtypes = [ctypes.POINTER(Config)]
        lib.moe_decode_plan.argtypes = [ctypes.POINTER(Config), i32, i32, i32, ctypes.POINTER(PlanInfo)]
        lib.moe_decode_create.argtypes = [ctypes.POINTER(Config), ctypes.POINTER(Weights),
                                          ctypes.POINTER(vp)]
        lib.moe_decode_run.argtypes = [vp, vp, vp, vp, i32, vp, vp, vp]
        lib.moe_decode_run_host.argtypes = [vp, vp, vp, vp, i32, vp, vp, vp]
        lib.moe_decode_run_static.argtypes = [ctypes.POINTER(Config), ctypes.POINTER(Weights), vp, vp, vp, i32,
                                              vp, vp, vp]
        lib.moe_decode_get_status.argtypes = [vp, vp]
        lib.moe_decode_set_option.argtypes = [vp, i32, i64]
        lib.moe_decode_get_info.argtypes = [vp, i32, ctypes.POINTER(i64)]
        lib.moe_decode_destroy.argtypes = [vp]
        lib.moe_decode_status_string.argtypes = [i32]
        lib.moe_decode_status_string.restype = ctypes.c_char_p
        lib.moe_decode_abi_version.argtypes = []
        for name in EXPORTS:
            if name != "moe_decode_status_string":
                getattr(lib, name).restype = i32
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return load().moe_decode_status_string(status).decode()


def check(status: int, what: str) -> None:
    if status != MOE_OK:
        raise MoEDecodeError(status, what)
