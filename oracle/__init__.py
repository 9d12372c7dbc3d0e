"""CPU oracle for the ReplaySSM checkpointing selective-state-update.

TEST INFRASTRUCTURE ONLY.  The arithmetic lives in ``rssm_oracle.c`` (plain C,
built with ``-ffp-contract=off``); this module only compiles it and marshals
numpy arrays through ctypes.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline / reference leg may import it.  It shares no code
with the CUDA library and the CUDA library never calls it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rssm_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle_rssm.so")
_lock = threading.Lock()
_lib = None

F32, BF16, F16, I8, E4M3, NVFP4 = 0, 1, 2, 3, 4, 5
NEAREST, STOCHASTIC = 0, 1
ERR_PNAT, ERR_SEQLEN, ERR_ACCEPT = 1, 2, 4
P_DIM, N_DIM = 64, 128


def build(force: bool = False) -> str:
    """Compile the oracle into a shared library next to its source."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    base = ["gcc", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-std=gnu11", _SRC, "-o", _LIB_PATH + ".tmp"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:] + ["-lm"], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base + ["-lm"], check=True, capture_output=True)
    os.replace(_LIB_PATH + ".tmp", _LIB_PATH)
    return _LIB_PATH


class OrcCache(ctypes.Structure):
    _fields_ = [
        ("num_slots", ctypes.c_int32), ("nheads", ctypes.c_int32), ("ngroups", ctypes.c_int32),
        ("max_window", ctypes.c_int32), ("npredicted", ctypes.c_int32),
        ("state_dtype", ctypes.c_int32), ("rounding", ctypes.c_int32),
        ("state", ctypes.c_void_p), ("state_slot_stride", ctypes.c_int64),
        ("scale", ctypes.c_void_p), ("scale_slot_stride", ctypes.c_int64),
        ("x_cache", ctypes.c_void_p), ("x_slot_stride", ctypes.c_int64),
        ("B_cache", ctypes.c_void_p), ("B_slot_stride", ctypes.c_int64),
        ("dt_cache", ctypes.c_void_p), ("dt_slot_stride", ctypes.c_int64),
        ("ring_start", ctypes.c_void_p), ("flush_epoch", ctypes.c_void_p), ("error_word", ctypes.c_void_p),
        ("read_state", ctypes.c_void_p), ("read_slot_stride", ctypes.c_int64),
        ("read_scale", ctypes.c_void_p), ("read_scale_stride", ctypes.c_int64),
        ("read_dtype", ctypes.c_int32),
        ("read_sf", ctypes.c_void_p), ("read_sf_stride", ctypes.c_int64),
        ("read_gs", ctypes.c_void_p),
    ]


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = ctypes.CDLL(build())
            vp, i32, i64, u32, u64, f32 = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32,
                                           ctypes.c_uint64, ctypes.c_float)
            for name in ("orc_spec_exp", "orc_spec_log1p", "orc_spec_softplus"):
                getattr(_lib, name).restype = f32
                getattr(_lib, name).argtypes = [f32]
            for name in ("orc_spec_exp_n", "orc_spec_log1p_n", "orc_spec_softplus_n", "orc_f32_to_bf16_n",
                         "orc_f32_to_f16_n", "orc_f32_to_e4m3_n", "orc_f16_decode_n", "orc_e4m3_decode_n",
                         "orc_f32_to_e2m1_n", "orc_e2m1_decode_n"):
                getattr(_lib, name).restype = None
                getattr(_lib, name).argtypes = [vp, vp, ctypes.c_long]
            _lib.orc_philox4x32.argtypes = [u32, vp, vp, vp]
            _lib.orc_philox4x64.argtypes = [u32, vp, vp, vp]
            _lib.orc_sr_word.restype = u32
            _lib.orc_sr_word.argtypes = [u64, u32, u32, u32, u32]
            _lib.orc_quantize_rows.argtypes = [ctypes.c_int, ctypes.c_int, vp, ctypes.c_int, u32, u32, u32, u32,
                                               u64, vp, vp]
            _lib.orc_init_state.restype = ctypes.c_int
            _lib.orc_init_state.argtypes = [ctypes.POINTER(OrcCache), vp, vp, i32, u64]
            _lib.orc_flush.restype = ctypes.c_int
            _lib.orc_flush.argtypes = [ctypes.POINTER(OrcCache), vp, vp, vp, vp, i32, i32, i32, u64, ctypes.c_int]
            _lib.orc_step.restype = ctypes.c_int
            _lib.orc_step.argtypes = [ctypes.POINTER(OrcCache), vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32,
                                      vp, vp, vp, ctypes.c_int]
            _lib.orc_accept.restype = ctypes.c_int
            _lib.orc_accept.argtypes = [ctypes.POINTER(OrcCache), vp, vp, vp, vp, i32, i32]
            _lib.orc_quantize_rows_nvfp4.argtypes = [vp, ctypes.c_int, f32, vp, vp]
            _lib.orc_nvfp4_global_scale.restype = f32
            _lib.orc_nvfp4_global_scale.argtypes = [vp, ctypes.c_long]
            _lib.orc_have_openmp.restype = ctypes.c_int
            del i64
        return _lib


def openmp_threads() -> int:
    """Threads the oracle's OpenMP loops use by default (0: built without OpenMP)."""
    return int(lib().orc_have_openmp())


# --------------------------------------------------------------------------- #
# elementwise helpers (vectorised over numpy arrays)
# --------------------------------------------------------------------------- #
def _map(name, x, out_dtype):
    x = np.ascontiguousarray(x)
    y = np.empty(x.shape, dtype=out_dtype)
    getattr(lib(), name)(_p(x), _p(y), x.size)
    return y


def spec_exp(x):
    return _map("orc_spec_exp_n", np.asarray(x, np.float32), np.float32)


def spec_log1p(x):
    return _map("orc_spec_log1p_n", np.asarray(x, np.float32), np.float32)


def spec_softplus(x):
    return _map("orc_spec_softplus_n", np.asarray(x, np.float32), np.float32)


def f32_to_bf16_bits(x):
    return _map("orc_f32_to_bf16_n", np.asarray(x, np.float32), np.uint16)


def f32_to_f16_bits(x):
    return _map("orc_f32_to_f16_n", np.asarray(x, np.float32), np.uint16)


def f32_to_e4m3_bits(x):
    return _map("orc_f32_to_e4m3_n", np.asarray(x, np.float32), np.uint8)


def f32_to_e2m1_bits(x):
    return _map("orc_f32_to_e2m1_n", np.asarray(x, np.float32), np.uint8)


def e2m1_decode(bits):
    return _map("orc_e2m1_decode_n", np.asarray(bits, np.uint8), np.float32)


def quantize_rows_nvfp4(acc, gs):
    """NVFP4-encode rows x 128 fp32 values with global scale gs; returns
    (codes [rows][64] bytes, two per byte, even element low; block scales
    [rows][8] e4m3 bytes)."""
    acc = np.ascontiguousarray(acc, dtype=np.float32).reshape(-1, N_DIM)
    codes = np.zeros((acc.shape[0], N_DIM // 2), np.uint8)
    sf = np.zeros((acc.shape[0], N_DIM // 16), np.uint8)
    lib().orc_quantize_rows_nvfp4(_p(acc), acc.shape[0], np.float32(gs), _p(codes), _p(sf))
    return codes, sf


def nvfp4_global_scale(state):
    st = np.ascontiguousarray(state, dtype=np.float32)
    return float(lib().orc_nvfp4_global_scale(_p(st), st.size))


def f16_decode(bits):
    return _map("orc_f16_decode_n", np.asarray(bits, np.uint16), np.float32)


def e4m3_decode(bits):
    return _map("orc_e4m3_decode_n", np.asarray(bits, np.uint8), np.float32)


def bf16_decode(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def philox4x32(rounds, ctr, key):
    c = np.ascontiguousarray(ctr, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    o = np.zeros(4, np.uint32)
    lib().orc_philox4x32(rounds, _p(c), _p(k), _p(o))
    return o


def philox4x64(rounds, ctr, key):
    c = np.ascontiguousarray(ctr, dtype=np.uint64)
    k = np.ascontiguousarray(key, dtype=np.uint64)
    o = np.zeros(4, np.uint64)
    lib().orc_philox4x64(rounds, _p(c), _p(k), _p(o))
    return o


def sr_word(seed, elem, h, s, epoch):
    return int(lib().orc_sr_word(seed, elem, h, s, epoch))


STATE_NP = {F32: np.float32, BF16: np.uint16, F16: np.uint16, I8: np.int8, E4M3: np.uint8}


def quantize_rows(dtype, rounding, acc, d0=0, h=0, s=0, epoch=0, seed=0):
    """Quantise rows x 128 fp32 accumulators; returns (codes, scales)."""
    acc = np.ascontiguousarray(acc, dtype=np.float32).reshape(-1, N_DIM)
    codes = np.zeros(acc.shape, dtype=STATE_NP[dtype])
    scales = np.zeros(acc.shape[0], dtype=np.float32)
    lib().orc_quantize_rows(dtype, rounding, _p(acc), acc.shape[0], d0, h, s, epoch, seed, _p(codes),
                            _p(scales))
    return codes, scales


# --------------------------------------------------------------------------- #
# cache + operations
# --------------------------------------------------------------------------- #
class OracleCache:
    """numpy-backed cache with the same layout as the library's.

    Arrays are 2-D [slot, slot_stride] so a slot may carry padding at its end.
    """

    def __init__(self, num_slots, nheads, ngroups, max_window, npredicted, state_dtype, rounding=NEAREST,
                 slot_pad_bytes=0, read_dtype=None):
        """read_dtype (I8, E4M3 or NVFP4): keep a separate read checkpoint,
        nearest-encoded from the recurrence's fp32 values at init and at every
        flush, which the step reads S0 from (None: the step reads the
        recurrence state).  NVFP4: E2M1 codes (two per byte), one E4M3 scale
        per 16 dstate values, one FP32 global scale per slot."""
        self.S, self.H, self.G = num_slots, nheads, ngroups
        self.W, self.Tmax = max_window, npredicted
        self.L = max_window + npredicted
        self.state_dtype, self.rounding = state_dtype, rounding
        sd = STATE_NP[state_dtype]
        esz = np.dtype(sd).itemsize

        def stride(n_elem, itemsize):
            return n_elem + slot_pad_bytes // itemsize

        self.state = np.zeros((num_slots, stride(nheads * P_DIM * N_DIM, esz)), sd)
        self.scale = np.ones((num_slots, stride(nheads * P_DIM, 4)), np.float32)
        self.x_cache = np.zeros((num_slots, stride(nheads * self.L * P_DIM, 2)), np.uint16)
        self.B_cache = np.zeros((num_slots, stride(ngroups * self.L * N_DIM, 2)), np.uint16)
        self.dt_cache = np.zeros((num_slots, stride(nheads * self.L, 4)), np.float32)
        self.ring_start = np.zeros(num_slots, np.int32)
        self.flush_epoch = np.zeros(num_slots, np.uint32)
        self.error_word = np.zeros(1, np.uint32)
        self.read_dtype = read_dtype
        self.read_state = self.read_scale = self.read_sf = self.read_gs = None
        if read_dtype == NVFP4:
            self.read_state = np.zeros((num_slots, stride(nheads * P_DIM * N_DIM // 2, 1)), np.uint8)
            self.read_sf = np.zeros((num_slots, stride(nheads * P_DIM * N_DIM // 16, 1)), np.uint8)
            self.read_gs = np.ones(num_slots, np.float32)
        elif read_dtype is not None:
            self.read_state = np.zeros((num_slots, stride(nheads * P_DIM * N_DIM, 1)), np.uint8)
            self.read_scale = np.ones((num_slots, stride(nheads * P_DIM, 4)), np.float32)

    def read_state_view(self):
        if self.read_dtype == NVFP4:
            return self.read_state[:, : self.H * P_DIM * N_DIM // 2].reshape(self.S, self.H, P_DIM, N_DIM // 2)
        return self.read_state[:, : self.H * P_DIM * N_DIM].reshape(self.S, self.H, P_DIM, N_DIM)

    def read_sf_view(self):
        return self.read_sf[:, : self.H * P_DIM * N_DIM // 16].reshape(self.S, self.H, P_DIM, N_DIM // 16)

    def read_scale_view(self):
        return self.read_scale[:, : self.H * P_DIM].reshape(self.S, self.H, P_DIM)

    # logical views (no padding)
    def state_view(self):
        return self.state[:, : self.H * P_DIM * N_DIM].reshape(self.S, self.H, P_DIM, N_DIM)

    def scale_view(self):
        return self.scale[:, : self.H * P_DIM].reshape(self.S, self.H, P_DIM)

    def x_view(self):
        return self.x_cache[:, : self.H * self.L * P_DIM].reshape(self.S, self.H, self.L, P_DIM)

    def B_view(self):
        return self.B_cache[:, : self.G * self.L * N_DIM].reshape(self.S, self.G, self.L, N_DIM)

    def dt_view(self):
        return self.dt_cache[:, : self.H * self.L].reshape(self.S, self.H, self.L)

    def copy(self):
        o = OracleCache.__new__(OracleCache)
        o.__dict__.update({k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in self.__dict__.items()})
        return o

    def struct(self):
        c = OrcCache()
        c.num_slots, c.nheads, c.ngroups = self.S, self.H, self.G
        c.max_window, c.npredicted = self.W, self.Tmax
        c.state_dtype, c.rounding = self.state_dtype, self.rounding
        c.state, c.state_slot_stride = _p(self.state), self.state.shape[1]
        c.scale, c.scale_slot_stride = _p(self.scale), self.scale.shape[1]
        c.x_cache, c.x_slot_stride = _p(self.x_cache), self.x_cache.shape[1]
        c.B_cache, c.B_slot_stride = _p(self.B_cache), self.B_cache.shape[1]
        c.dt_cache, c.dt_slot_stride = _p(self.dt_cache), self.dt_cache.shape[1]
        c.ring_start, c.flush_epoch, c.error_word = _p(self.ring_start), _p(self.flush_epoch), _p(self.error_word)
        rd = getattr(self, "read_state", None)
        if rd is not None:
            c.read_state, c.read_slot_stride = _p(rd), rd.shape[1]
            c.read_dtype = self.read_dtype
            if self.read_dtype == NVFP4:
                c.read_sf, c.read_sf_stride = _p(self.read_sf), self.read_sf.shape[1]
                c.read_gs = _p(self.read_gs)
            else:
                c.read_scale, c.read_scale_stride = _p(self.read_scale), self.read_scale.shape[1]
        return c

    def init_state(self, states, ids, seed=0):
        states = np.ascontiguousarray(states, np.float32)
        ids = np.ascontiguousarray(ids, np.int32)
        st = self.struct()
        rc = lib().orc_init_state(ctypes.byref(st), _p(states), _p(ids), ids.size, seed)
        assert rc == 0

    def flush(self, A, slot_idx, pnat, T, cu_seqlens=None, force=0, seed=0, nthreads=0):
        """pnat is updated in place (flushed rows -> 0)."""
        A = np.ascontiguousarray(A, np.float32)
        slot_idx = np.ascontiguousarray(slot_idx, np.int32)
        assert pnat.dtype == np.int32 and pnat.flags.c_contiguous
        cu = None if cu_seqlens is None else np.ascontiguousarray(cu_seqlens, np.int32)
        st = self.struct()
        rc = lib().orc_flush(ctypes.byref(st), _p(A), _p(slot_idx), _p(pnat), _p(cu), slot_idx.size, T, force,
                             seed, nthreads)
        assert rc == 0

    def step(self, x, dt, A, B, C, D, dt_bias, slot_idx, pnat, T, cu_seqlens=None, want_f64=False, nthreads=0,
             z=None):
        """Returns y (bf16 bits, [tok][H][64]) and optionally y in float64.
        `z` (bf16 bits, [tok][H][64]): output gate, y * silu(z) before rounding."""
        x = np.ascontiguousarray(x, np.uint16)
        B = np.ascontiguousarray(B, np.uint16)
        C = np.ascontiguousarray(C, np.uint16)
        dt = np.ascontiguousarray(dt, np.float32)
        A = np.ascontiguousarray(A, np.float32)
        D = np.ascontiguousarray(D, np.float32)
        dt_bias = np.ascontiguousarray(dt_bias, np.float32)
        slot_idx = np.ascontiguousarray(slot_idx, np.int32)
        pnat = np.ascontiguousarray(pnat, np.int32)
        cu = None if cu_seqlens is None else np.ascontiguousarray(cu_seqlens, np.int32)
        ntok = x.shape[0]
        out = np.zeros((ntok, self.H, P_DIM), np.uint16)
        out64 = np.zeros((ntok, self.H, P_DIM), np.float64) if want_f64 else None
        st = self.struct()
        zz = None if z is None else np.ascontiguousarray(z, np.uint16)
        assert zz is None or zz.shape == out.shape
        rc = lib().orc_step(ctypes.byref(st), _p(x), _p(dt), _p(A), _p(B), _p(C), _p(D), _p(dt_bias),
                            _p(slot_idx), _p(pnat), _p(cu), slot_idx.size, T, _p(zz), _p(out), _p(out64), nthreads)
        assert rc == 0
        return (out, out64) if want_f64 else out

    def accept(self, slot_idx, pnat, accepted, T, cu_seqlens=None):
        slot_idx = np.ascontiguousarray(slot_idx, np.int32)
        accepted = np.ascontiguousarray(accepted, np.int32)
        assert pnat.dtype == np.int32 and pnat.flags.c_contiguous
        cu = None if cu_seqlens is None else np.ascontiguousarray(cu_seqlens, np.int32)
        st = self.struct()
        rc = lib().orc_accept(ctypes.byref(st), _p(slot_idx), _p(pnat), _p(accepted), _p(cu), slot_idx.size, T)
        assert rc == 0
