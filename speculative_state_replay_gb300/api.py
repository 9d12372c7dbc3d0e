"""Python binding of librssm: the C ABI entry points with torch tensors.

Every function marshals tensor pointers, sizes and the current CUDA stream
into the C call of the same name and raises on a non-OK status.  All work
runs in the library's CUDA kernels; nothing here computes any part of the op.
Layouts and semantics are those of include/rssm.h.
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib

F32, BF16, F16, I8, E4M3, NVFP4 = 0, 1, 2, 3, 4, 5
NEAREST, STOCHASTIC = 0, 1
ERRBIT_PNAT, ERRBIT_SEQLEN, ERRBIT_ACCEPT, ERRBIT_TIMEOUT = 1, 2, 4, 8
DIM, DSTATE = 64, 128
STATE_TORCH = {F32: torch.float32, BF16: torch.int16, F16: torch.int16, I8: torch.int8, E4M3: torch.uint8,
               NVFP4: torch.uint8}


class RssmError(RuntimeError):
    def __init__(self, fn: str, status: int):
        msg = _lib.load().rssm_status_string(status).decode()
        super().__init__(f"{fn} failed: {msg} (status {status})")
        self.status = status


def _ptr(t):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(fn, status):
    if status != 0:
        raise RssmError(fn, status)


def _check_tokens(fn, cache, slot_idx, T, cu_seqlens, **per_token):
    """Host-side size check of the per-token tensors (no device read).

    Without cu_seqlens the kernels address batch * T tokens in every per-token
    tensor (x, dt, B, C, z, out), so each must hold at least that many token
    rows of its row size; with cu_seqlens the token count lives on the device
    and the caller sizes the tensors (include/rssm.h)."""
    if cu_seqlens is not None:
        return
    need = slot_idx.numel() * T
    row = {"x": cache.H * DIM, "out": cache.H * DIM, "z": cache.H * DIM, "dt": cache.H,
           "B": cache.G * DSTATE, "C": cache.G * DSTATE}
    for name, t in per_token.items():
        if t is None or need == 0:
            continue
        if t.numel() < need * row[name]:
            raise ValueError(f"{fn}: {name} holds {t.numel()} elements, fewer than batch * T = {need} tokens of "
                             f"{row[name]} (pass cu_seqlens for variable-length rows)")


class RssmCache:
    """Cache of all slots on one device: checkpoints, rings, bookkeeping.

    Every tensor is 2-D [slot, slot_stride]; `slot_pad_bytes` adds padding
    after each slot's page.  bf16/f16 data is held as raw 16-bit words.
    `read_dtype` (I8 or E4M3) adds a separate 8-bit read checkpoint
    (`read_state`, `read_scale`) that the step's readout reads S0 from;
    NVFP4 adds an NVFP4 one (`read_state` codes two per byte, `read_sf` block
    scales, `read_gs` per-slot global scales).
    """

    def __init__(self, num_slots, nheads, ngroups, max_window, npredicted, state_dtype, rounding=NEAREST,
                 device="cuda", slot_pad_bytes=0, read_dtype=None):
        self.S, self.H, self.G = num_slots, nheads, ngroups
        self.W, self.Tmax = max_window, npredicted
        self.L = max_window + npredicted
        self.state_dtype, self.rounding = state_dtype, rounding
        dev = torch.device(device)
        sd = STATE_TORCH[state_dtype]
        esz = torch.empty(0, dtype=sd).element_size()

        def stride(n, itemsize):
            return n + slot_pad_bytes // itemsize

        z = lambda shape, dt: torch.zeros(shape, dtype=dt, device=dev)  # noqa: E731
        self.state = z((num_slots, stride(nheads * DIM * DSTATE, esz)), sd)
        self.scale = torch.ones((num_slots, stride(nheads * DIM, 4)), dtype=torch.float32, device=dev)
        self.x_cache = z((num_slots, stride(nheads * self.L * DIM, 2)), torch.int16)
        self.B_cache = z((num_slots, stride(ngroups * self.L * DSTATE, 2)), torch.int16)
        self.dt_cache = z((num_slots, stride(nheads * self.L, 4)), torch.float32)
        self.ring_start = z((num_slots,), torch.int32)
        self.flush_epoch = z((num_slots,), torch.int32)
        self.error_word = z((1,), torch.int32)
        self.read_dtype = read_dtype
        self.read_state = self.read_scale = self.read_sf = self.read_gs = None
        if read_dtype == NVFP4:
            self.read_state = z((num_slots, stride(nheads * DIM * DSTATE // 2, 1)), torch.uint8)
            self.read_sf = z((num_slots, stride(nheads * DIM * DSTATE // 16, 1)), torch.uint8)
            self.read_gs = torch.ones((num_slots,), dtype=torch.float32, device=dev)
        elif read_dtype is not None:
            self.read_state = z((num_slots, stride(nheads * DIM * DSTATE, 1)), STATE_TORCH[read_dtype])
            self.read_scale = torch.ones((num_slots, stride(nheads * DIM, 4)), dtype=torch.float32, device=dev)
        self._struct = None

    def struct(self):
        if self._struct is None:
            c = _lib.RssmCacheStruct()
            c.num_slots, c.nheads, c.ngroups = self.S, self.H, self.G
            c.dim, c.dstate = DIM, DSTATE
            c.max_window, c.npredicted = self.W, self.Tmax
            c.state_dtype, c.rounding = self.state_dtype, self.rounding
            c.state, c.state_slot_stride = self.state.data_ptr(), self.state.shape[1]
            c.scale, c.scale_slot_stride = self.scale.data_ptr(), self.scale.shape[1]
            c.x_cache, c.x_slot_stride = self.x_cache.data_ptr(), self.x_cache.shape[1]
            c.B_cache, c.B_slot_stride = self.B_cache.data_ptr(), self.B_cache.shape[1]
            c.dt_cache, c.dt_slot_stride = self.dt_cache.data_ptr(), self.dt_cache.shape[1]
            c.ring_start = self.ring_start.data_ptr()
            c.flush_epoch = self.flush_epoch.data_ptr()
            c.error_word = self.error_word.data_ptr()
            if self.read_state is not None:
                c.read_state, c.read_slot_stride = self.read_state.data_ptr(), self.read_state.shape[1]
                c.read_dtype = self.read_dtype
                if self.read_dtype == NVFP4:
                    c.read_sf, c.read_sf_slot_stride = self.read_sf.data_ptr(), self.read_sf.shape[1]
                    c.read_gs = self.read_gs.data_ptr()
                else:
                    c.read_scale, c.read_scale_slot_stride = self.read_scale.data_ptr(), self.read_scale.shape[1]
            self._struct = c
        return ctypes.byref(self._struct)

    # logical views (without the slot padding)
    def state_view(self):
        return self.state[:, : self.H * DIM * DSTATE].view(self.S, self.H, DIM, DSTATE)

    def scale_view(self):
        return self.scale[:, : self.H * DIM].view(self.S, self.H, DIM)

    def x_view(self):
        return self.x_cache[:, : self.H * self.L * DIM].view(self.S, self.H, self.L, DIM)

    def B_view(self):
        return self.B_cache[:, : self.G * self.L * DSTATE].view(self.S, self.G, self.L, DSTATE)

    def dt_view(self):
        return self.dt_cache[:, : self.H * self.L].view(self.S, self.H, self.L)


def rssm_scratch_bytes(cache: RssmCache, batch: int, T: int) -> int:
    return int(_lib.load().rssm_scratch_bytes(cache.struct(), batch, T))


def alloc_scratch(cache: RssmCache, batch: int, T: int) -> torch.Tensor:
    n = rssm_scratch_bytes(cache, batch, T)
    if n == 0:
        raise RssmError("rssm_scratch_bytes", 1)
    # zero-filled: rssm_flush keeps a counter in the first word, which must start
    # at zero (every call leaves it at zero)
    return torch.zeros(n, dtype=torch.uint8, device=cache.state.device)


def rssm_init_state(cache, states, slot_idx, seed=0, stream=None):
    _check("rssm_init_state", _lib.load().rssm_init_state(cache.struct(), _ptr(states), _ptr(slot_idx),
                                                          slot_idx.numel(), seed, _stream(stream)))


def rssm_flush(cache, A, slot_idx, pnat, T, scratch, cu_seqlens=None, force=0, seed=0, stream=None):
    _check("rssm_flush", _lib.load().rssm_flush(cache.struct(), _ptr(A), _ptr(slot_idx), _ptr(pnat),
                                                _ptr(cu_seqlens), slot_idx.numel(), T, force, seed,
                                                _ptr(scratch), scratch.numel(), _stream(stream)))


def rssm_accept_flush(cache, A, slot_idx, pnat, accepted, accept_T, T, scratch, accept_cu_seqlens=None,
                      cu_seqlens=None, force=0, seed=0, stream=None):
    """rssm_accept(accepted, accept_cu_seqlens, accept_T) then rssm_flush(...), one launch."""
    _check("rssm_accept_flush", _lib.load().rssm_accept_flush(
        cache.struct(), _ptr(A), _ptr(slot_idx), _ptr(pnat), _ptr(accepted), _ptr(accept_cu_seqlens), accept_T,
        _ptr(cu_seqlens), slot_idx.numel(), T, force, seed, _ptr(scratch), scratch.numel(), _stream(stream)))


def _step(fn, cache, x, dt, A, B, C, D, dt_bias, slot_idx, pnat, T, out, scratch, cu_seqlens, stream):
    _check_tokens(fn, cache, slot_idx, T, cu_seqlens, x=x, dt=dt, B=B, C=C, out=out)
    f = getattr(_lib.load(), fn)
    _check(fn, f(cache.struct(), _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(dt_bias),
                 _ptr(slot_idx), _ptr(pnat), _ptr(cu_seqlens), slot_idx.numel(), T, _ptr(out), _ptr(scratch),
                 scratch.numel(), _stream(stream)))


def _step_gated(fn, cache, x, dt, A, B, C, D, dt_bias, slot_idx, pnat, T, z, out, scratch, cu_seqlens, stream):
    _check_tokens(fn, cache, slot_idx, T, cu_seqlens, x=x, dt=dt, B=B, C=C, z=z, out=out)
    f = getattr(_lib.load(), fn)
    _check(fn, f(cache.struct(), _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(dt_bias),
                 _ptr(slot_idx), _ptr(pnat), _ptr(cu_seqlens), slot_idx.numel(), T, _ptr(z), _ptr(out),
                 _ptr(scratch), scratch.numel(), _stream(stream)))


def rssm_step(cache, x, dt, A, B, C, D, dt_bias, slot_idx, pnat, T, out, scratch, cu_seqlens=None, stream=None,
              z=None):
    """`z`: optional output gate (bf16 bits [tok][H][64]): y * silu(z)."""
    if z is None:
        _step("rssm_step", cache, x, dt, A, B, C, D, dt_bias, slot_idx, pnat, T, out, scratch, cu_seqlens, stream)
    else:
        _step_gated("rssm_step_gated", cache, x, dt, A, B, C, D, dt_bias, slot_idx, pnat, T, z, out, scratch,
                    cu_seqlens, stream)


def rssm_step_precompute(cache, x, dt, A, B, C, D, dt_bias, slot_idx, pnat, T, out, scratch, cu_seqlens=None,
                         stream=None):
    _step("rssm_step_precompute", cache, x, dt, A, B, C, D, dt_bias, slot_idx, pnat, T, out, scratch, cu_seqlens,
          stream)


def rssm_step_readout(cache, x, dt, A, B, C, D, dt_bias, slot_idx, pnat, T, out, scratch, cu_seqlens=None,
                      stream=None, z=None):
    if z is None:
        _step("rssm_step_readout", cache, x, dt, A, B, C, D, dt_bias, slot_idx, pnat, T, out, scratch, cu_seqlens,
              stream)
    else:
        _step_gated("rssm_step_readout_gated", cache, x, dt, A, B, C, D, dt_bias, slot_idx, pnat, T, z, out,
                    scratch, cu_seqlens, stream)


def _flush_step(fn, cache, x, dt, A, B, C, D, dt_bias, slot_idx, pnat, T, out, scratch, cu_seqlens, force, seed,
                stream):
    _check_tokens(fn, cache, slot_idx, T, cu_seqlens, x=x, dt=dt, B=B, C=C, out=out)
    f = getattr(_lib.load(), fn)
    _check(fn, f(cache.struct(), _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(dt_bias),
                 _ptr(slot_idx), _ptr(pnat), _ptr(cu_seqlens), slot_idx.numel(), T, force, seed, _ptr(out),
                 _ptr(scratch), scratch.numel(), _stream(stream)))


def rssm_flush_step(cache, x, dt, A, B, C, D, dt_bias, slot_idx, pnat, T, out, scratch, cu_seqlens=None, force=0,
                    seed=0, stream=None):
    _flush_step("rssm_flush_step", cache, x, dt, A, B, C, D, dt_bias, slot_idx, pnat, T, out, scratch, cu_seqlens,
                force, seed, stream)


def rssm_flush_step_classify(cache, x, dt, A, B, C, D, dt_bias, slot_idx, pnat, T, out, scratch, cu_seqlens=None,
                               force=0, seed=0, stream=None):
    _flush_step("rssm_flush_step_classify", cache, x, dt, A, B, C, D, dt_bias, slot_idx, pnat, T, out, scratch,
                cu_seqlens, force, seed, stream)


def rssm_flush_step_main(cache, x, dt, A, B, C, D, dt_bias, slot_idx, pnat, T, out, scratch, cu_seqlens=None,
                            force=0, seed=0, stream=None):
    _flush_step("rssm_flush_step_main", cache, x, dt, A, B, C, D, dt_bias, slot_idx, pnat, T, out, scratch,
                cu_seqlens, force, seed, stream)


def rssm_accept(cache, slot_idx, pnat, accepted, T, cu_seqlens=None, stream=None):
    _check("rssm_accept", _lib.load().rssm_accept(cache.struct(), _ptr(slot_idx), _ptr(pnat), _ptr(accepted),
                                                  _ptr(cu_seqlens), slot_idx.numel(), T, _stream(stream)))


def rssm_eval_spec_math(x, out_exp=None, out_softplus=None, stream=None):
    _check("rssm_eval_spec_math", _lib.load().rssm_eval_spec_math(_ptr(x), _ptr(out_exp), _ptr(out_softplus),
                                                                  x.numel(), _stream(stream)))


def rssm_selftest_wait_timeout(error_word, wait_ms=50, stream=None):
    """Diagnostics: one bounded mbarrier wait that runs out (sets ERRBIT_TIMEOUT)."""
    _check("rssm_selftest_wait_timeout", _lib.load().rssm_selftest_wait_timeout(_ptr(error_word), wait_ms,
                                                                                _stream(stream)))
