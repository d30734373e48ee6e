"""ctypes view of include/e0.h: structures and prototypes of libe0.so.

The library is required: there is no fallback.  Loading fails loudly if libe0.so has
not been built (``python -c "import __graft_entry__ as g; g.build()"``).
"""
from __future__ import annotations

import ctypes as C
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libe0.so")

vp = C.c_void_p
i32 = C.c_int32
i64 = C.c_int64
u32 = C.c_uint32
u64 = C.c_uint64
f32 = C.c_float
f64 = C.c_double
sz = C.c_size_t

E0_OK = 0
E0_ERR_INVALID = -1
E0_ERR_SHAPE = -2
E0_ERR_CUDA = -3
E0_ERR_UNSUPPORTED = -6
E0_ROUTE_SOFTMAX_TOPK = 0
E0_ROUTE_SIGMOID_GROUP = 1
E0_LAYOUT_ROWS = 0
E0_LAYOUT_COLSLAB = 1
E0_DEV_TIMEOUT = 1
E0_DEV_BAD_ID = 2
E0_DEV_NOT_RESIDENT = 4
E0_DEV_ABORTED = 8
STATUS_NAMES = {0: "E0_OK", -1: "E0_ERR_INVALID", -2: "E0_ERR_SHAPE", -3: "E0_ERR_CUDA", -4: "E0_ERR_TIMEOUT",
                -5: "E0_ERR_NOMEM", -6: "E0_ERR_UNSUPPORTED", -7: "E0_ERR_DEVICE"}


class e0_q4(C.Structure):
    _fields_ = [("q", vp), ("scale", vp), ("bias", vp)]


class e0_experts(C.Structure):
    _fields_ = [("gate_up", e0_q4), ("down", e0_q4), ("n", i32), ("slot_of", vp), ("stride", i64), ("ready", vp)]


class e0_qlora(C.Structure):
    _fields_ = [("w", e0_q4), ("a", vp), ("bt", vp), ("out", i32), ("r", i32), ("alpha", f32)]


class e0_prerouter(C.Structure):
    _fields_ = [("H", i32), ("w1h", vp), ("w1c_t", vp), ("w1p_t", vp), ("b1", vp), ("w2t", vp), ("b2", vp),
                ("lres", vp)]


class e0_dims(C.Structure):
    _fields_ = [("d", i32), ("E", i32), ("F", i32), ("K", i32), ("route", i32), ("n_group", i32),
                ("topk_group", i32), ("route_scale", f32), ("score_bias", vp)]


class e0_stage_stats(C.Structure):
    _fields_ = [("hits", i32), ("misses", i32), ("evictions", i32), ("h2d_bytes", i64)]


class e0_layer(C.Structure):
    _fields_ = [("routed", e0_experts), ("shared", e0_experts), ("lora", e0_qlora), ("head", e0_prerouter),
                ("router", vp), ("score_bias", vp)]


class e0_stack_outputs(C.Structure):
    _fields_ = [("ids", vp), ("weights", vp), ("h_trace", vp), ("delta", vp), ("logits", vp), ("next_ids", vp),
                ("commit_box", vp)]


P = C.POINTER

PROTOTYPES = {
    "e0_last_error": (C.c_char_p, []),
    "e0_version": (C.c_char_p, []),
    "e0_pack_int4": (i32, [vp, i64, i64, i64, i32, i32, vp, vp, vp, vp]),
    "e0_workspace_size": (sz, [P(e0_dims), i32]),
    "e0_workspace_reset": (i32, [vp, sz, vp]),
    "e0_get_device_status": (i32, [vp, P(u32), vp]),
    "e0_prerouter_forward": (i32, [P(e0_prerouter), i32, i32, vp, vp, vp, i32, i32, vp, vp, vp, vp, vp, sz, vp]),
    "e0_qlinear_lora": (i32, [P(e0_qlora), i32, vp, i32, i32, vp, vp, vp, sz, vp]),
    "e0_moe_decode_layer": (i32, [P(e0_dims), P(e0_experts), P(e0_experts), P(e0_qlora), P(e0_prerouter), vp, vp,
                                  vp, vp, i32, vp, vp, vp, vp, vp, vp, sz, vp]),
    "e0_moe_decode_layer_noalloc": (i32, [P(e0_dims), P(e0_experts), P(e0_experts), P(e0_qlora), P(e0_prerouter),
                                          vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]),
    "e0_prefill_workspace_size": (sz, [P(e0_dims), i32, i32]),
    "e0_decode_workspace_size": (sz, [P(e0_dims), i32, i32, i32]),
    "e0_moe_prefill_layer": (i32, [P(e0_dims), P(e0_experts), P(e0_experts), P(e0_qlora), vp, vp, i32, vp, vp, vp,
                                   vp, vp, sz, vp]),
    "e0_expert_bundle_bytes": (sz, [P(e0_dims), vp]),
    "e0_slot_pool_create": (i32, [P(vp), P(e0_dims), i32, i32, vp, sz]),
    "e0_slot_pool_destroy": (None, [vp]),
    "e0_slot_pool_view": (i32, [vp, i32, P(e0_experts)]),
    "e0_stage_slots": (i32, [vp, vp, i32, vp, vp, i32, u32, vp, vp, P(e0_stage_stats)]),
    "e0_stage_slots_host": (i32, [vp, vp, i32, vp, i32, u32, vp, vp, P(e0_stage_stats)]),
    "e0_slot_pool_resident": (i32, [vp, i32, vp]),
    "e0_commit_box_create": (i32, [P(vp), i32]),
    "e0_commit_box_destroy": (None, [vp]),
    "e0_commit_box_device": (vp, [vp]),
    "e0_stage_slots_committed": (i32, [vp, vp, vp, vp, i32, i32, u32, vp, u64, P(e0_stage_stats)]),
    "e0_debug_fail_copies": (i32, [vp, i32]),
    "e0_stack_create": (i32, [P(vp), P(e0_dims), P(e0_layer), i32, vp]),
    "e0_stack_destroy": (None, [vp]),
    "e0_stack_workspace_size": (sz, [vp]),
    "e0_stack_step": (i32, [vp, i32, vp, vp, vp, P(e0_stack_outputs), vp, vp, sz, vp]),
    "e0_synth_normal": (i32, [vp, i64, u64, u32, i64, f64, i32, vp]),
    "e0_debug_inject_stall": (i32, [vp, u64, vp]),
    "e0_debug_trace": (i32, [vp, sz]),
    "e0_debug_plan": (i32, [i32, i32, i32, i32, i32, i32, i32, i32, vp, vp, vp]),
}

_lib = None


def lib():
    """Load libe0.so (once) and attach prototypes.  Raises if the library is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libe0.so is not built ({LIB_PATH}); run __graft_entry__.build() first")
        h = C.CDLL(LIB_PATH)
        for name, (res, args) in PROTOTYPES.items():
            fn = getattr(h, name)
            fn.restype = res
            fn.argtypes = args
        _lib = h
    return _lib


class E0Error(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


def check(status: int) -> None:
    if status != E0_OK:
        raise E0Error(status, lib().e0_last_error().decode())
