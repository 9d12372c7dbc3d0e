"""ctypes loader for librssm.so (argument marshalling only)."""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "librssm.so")
_lock = threading.Lock()
_lib = None


class RssmCacheStruct(ctypes.Structure):
    """Mirror of `rssm_cache` in include/rssm.h."""

    _fields_ = [
        ("num_slots", ctypes.c_int32), ("nheads", ctypes.c_int32), ("ngroups", ctypes.c_int32),
        ("dim", ctypes.c_int32), ("dstate", ctypes.c_int32), ("max_window", ctypes.c_int32),
        ("npredicted", ctypes.c_int32), ("state_dtype", ctypes.c_int32), ("rounding", ctypes.c_int32),
        ("state", ctypes.c_void_p), ("state_slot_stride", ctypes.c_int64),
        ("scale", ctypes.c_void_p), ("scale_slot_stride", ctypes.c_int64),
        ("x_cache", ctypes.c_void_p), ("x_slot_stride", ctypes.c_int64),
        ("B_cache", ctypes.c_void_p), ("B_slot_stride", ctypes.c_int64),
        ("dt_cache", ctypes.c_void_p), ("dt_slot_stride", ctypes.c_int64),
        ("ring_start", ctypes.c_void_p), ("flush_epoch", ctypes.c_void_p), ("error_word", ctypes.c_void_p),
        ("read_state", ctypes.c_void_p), ("read_slot_stride", ctypes.c_int64),
        ("read_scale", ctypes.c_void_p), ("read_scale_slot_stride", ctypes.c_int64),
        ("read_dtype", ctypes.c_int32),
        ("read_sf", ctypes.c_void_p), ("read_sf_slot_stride", ctypes.c_int64),
        ("read_gs", ctypes.c_void_p),
    ]


EXPORTS = ("rssm_scratch_bytes", "rssm_init_state", "rssm_flush", "rssm_step", "rssm_step_precompute",
           "rssm_step_readout", "rssm_step_gated", "rssm_step_readout_gated", "rssm_flush_step", "rssm_flush_step_classify", "rssm_flush_step_main", "rssm_accept", "rssm_accept_flush", "rssm_eval_spec_math", "rssm_selftest_wait_timeout",
           "rssm_status_string")


def load(path: str | None = None):
    """Load librssm.so; raises if it has not been built (no fallback exists)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"librssm.so not found at {p}: build it with `python -c 'import __graft_entry__ as g; "
                               "g.build()'` (needs nvcc); there is no CPU fallback")
        lib = ctypes.CDLL(p)
        vp, i32, i64, u64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64, ctypes.c_size_t
        cp = ctypes.POINTER(RssmCacheStruct)
        lib.rssm_scratch_bytes.restype = sz
        lib.rssm_scratch_bytes.argtypes = [cp, i32, i32]
        lib.rssm_init_state.restype = ctypes.c_int
        lib.rssm_init_state.argtypes = [cp, vp, vp, i32, u64, vp]
        lib.rssm_flush.restype = ctypes.c_int
        lib.rssm_flush.argtypes = [cp, vp, vp, vp, vp, i32, i32, i32, u64, vp, sz, vp]
        step_args = [cp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, vp, vp, sz, vp]
        for name in ("rssm_step", "rssm_step_precompute", "rssm_step_readout"):
            getattr(lib, name).restype = ctypes.c_int
            getattr(lib, name).argtypes = step_args
        gated_args = step_args[:13] + [vp] + step_args[13:]  # z before out
        for name in ("rssm_step_gated", "rssm_step_readout_gated"):
            getattr(lib, name).restype = ctypes.c_int
            getattr(lib, name).argtypes = gated_args
        for name in ("rssm_flush_step", "rssm_flush_step_classify", "rssm_flush_step_main"):
            getattr(lib, name).restype = ctypes.c_int
            getattr(lib, name).argtypes = [cp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, u64, vp, vp, sz, vp]
        lib.rssm_accept.restype = ctypes.c_int
        lib.rssm_accept.argtypes = [cp, vp, vp, vp, vp, i32, i32, vp]
        lib.rssm_accept_flush.restype = ctypes.c_int
        lib.rssm_accept_flush.argtypes = [cp, vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, u64, vp, sz, vp]
        lib.rssm_eval_spec_math.restype = ctypes.c_int
        lib.rssm_eval_spec_math.argtypes = [vp, vp, vp, i64, vp]
        lib.rssm_selftest_wait_timeout.restype = ctypes.c_int
        lib.rssm_selftest_wait_timeout.argtypes = [vp, i32, vp]
        lib.rssm_status_string.restype = ctypes.c_char_p
        lib.rssm_status_string.argtypes = [ctypes.c_int]
        _lib = lib
        return lib
