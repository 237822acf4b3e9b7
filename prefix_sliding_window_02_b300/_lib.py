"""ctypes view of libps.so (declarations in include/ps.h).

Loads the in-tree library built by ``prefix_sliding_window_02_b300.build``.
There is no fallback: if the library is missing, importing this module raises.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libps.so")

PS_OK = 0
PS_PE_CONTINUE = 0
PS_PE_RESET = 1
PS_DEV_BAD_PREFIX = 0x1
PS_DEV_BAD_POS = 0x2
PS_DEV_BAD_SLOT = 0x4
PS_DEV_TIMEOUT = 0x8
PS_DEV_BAD_RUN = 0x10
PS_DEV_BAD_SEQ = 0x20

EXPORTS = (
    "ps_status_string", "ps_ring_slots", "ps_kv_append", "ps_decode_workspace_size",
    "ps_decode", "ps_decode_partial", "ps_decode_combine", "ps_decode_noalloc", "ps_decode_append",
    "ps_prefill_workspace_size", "ps_prefill", "ps_prefill_tile_grid", "ps_prefill_tile_classes",
    "ps_prefill_backward_workspace_size", "ps_prefill_backward",
    "ps_check_device_status", "ps_device_code_version", "ps_test_force_wait_timeout",
    "ps_decode_step_layout_get", "ps_decode_graph_create", "ps_decode_graph_step",
    "ps_decode_graph_destroy",
)


class CacheDesc(ctypes.Structure):
    """Mirror of ``ps_cache_desc``."""
    _fields_ = [
        ("k_pool", ctypes.c_void_p),
        ("v_pool", ctypes.c_void_p),
        ("slot_base", ctypes.c_void_p),
        ("prefix_len", ctypes.c_void_p),
        ("status", ctypes.c_void_p),
        ("total_slots", ctypes.c_int64),
        ("nseq", ctypes.c_int32),
        ("n_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("window", ctypes.c_int32),
        ("capacity", ctypes.c_int32),
        ("prefix_max", ctypes.c_int32),
        ("rope_theta", ctypes.c_double),
        ("block_table", ctypes.c_void_p),
        ("block_size", ctypes.c_int32),
        ("blocks_per_seq", ctypes.c_int32),
        ("pe_mode", ctypes.c_int32),
    ]


class StepLayout(ctypes.Structure):
    """Mirror of ``ps_decode_step_layout``."""
    _fields_ = [(name, ctypes.c_size_t) for name in
                ("q_off", "k_off", "v_off", "pos_off", "in_bytes", "out_off", "lse_off",
                 "res_bytes")]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libps.so not built at {LIB_PATH}; run __graft_entry__.build()")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    f32, f64 = ctypes.c_float, ctypes.c_double
    pdesc = ctypes.POINTER(CacheDesc)
    sig = {
        "ps_status_string": (ctypes.c_char_p, [ctypes.c_int]),
        "ps_ring_slots": (ctypes.c_int, [vp, vp, i32, vp, i64, vp]),
        "ps_kv_append": (ctypes.c_int, [pdesc, vp, vp, vp, i32, vp, vp, i64, vp]),
        "ps_decode_workspace_size": (ctypes.c_int, [i32, i32, i32, i32, ctypes.POINTER(sz)]),
        "ps_decode": (ctypes.c_int, [pdesc, vp, vp, i32, f32, vp, vp, vp, sz, vp]),
        "ps_decode_partial": (ctypes.c_int, [pdesc, vp, vp, i32, f32, vp, sz, vp]),
        "ps_decode_combine": (ctypes.c_int, [pdesc, i32, vp, vp, vp, sz, vp]),
        "ps_decode_noalloc": (ctypes.c_int, [pdesc, vp, vp, i32, f32, vp, vp, vp]),
        "ps_decode_append": (ctypes.c_int, [pdesc, vp, vp, vp, vp, i32, f32, vp, vp, vp, sz, vp]),
        "ps_prefill_workspace_size": (ctypes.c_int, [i32, i32, i32, i32, i32, i32, i32,
                                                     ctypes.POINTER(sz)]),
        "ps_prefill": (ctypes.c_int, [vp, vp, vp, i32, i32, vp, vp, i32, i32, i32, i32, f32, f64,
                                      i32, pdesc, vp, vp, vp, vp, sz, vp, vp]),
        "ps_prefill_tile_grid": (ctypes.c_int, [i32, i32, i32, i32, i32, i32, i32,
                                                ctypes.POINTER(i32), ctypes.POINTER(i32)]),
        "ps_prefill_tile_classes": (ctypes.c_int, [i32, i32, i32, i32, i32, i32, i32, vp, vp]),
        "ps_check_device_status": (ctypes.c_int, [vp, ctypes.POINTER(i32)]),
        "ps_device_code_version": (ctypes.c_int, [ctypes.POINTER(i32)]),
        "ps_test_force_wait_timeout": (ctypes.c_int, [i32, i64]),
        "ps_decode_step_layout_get": (ctypes.c_int, [i32, i32, i32, i32,
                                                     ctypes.POINTER(StepLayout)]),
        "ps_decode_graph_create": (ctypes.c_int, [pdesc, i32, f32, vp, vp, vp, sz,
                                                  ctypes.POINTER(vp)]),
        "ps_decode_graph_step": (ctypes.c_int, [vp, vp, vp, i32, vp]),
        "ps_decode_graph_destroy": (ctypes.c_int, [vp]),
        "ps_prefill_backward_workspace_size": (ctypes.c_int, [i32, i32, i32, i32, i32,
                                                              ctypes.POINTER(sz)]),
        "ps_prefill_backward": (ctypes.c_int, [vp, vp, vp, vp, vp, vp, i32, i32, vp, vp, i32, i32,
                                               i32, i32, f32, f64, vp, vp, vp, vp, vp, sz, vp,
                                               vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()


class PsError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {lib.ps_status_string(code).decode()} ({code})")


def check(code: int, where: str) -> None:
    if code != PS_OK:
        raise PsError(code, where)
