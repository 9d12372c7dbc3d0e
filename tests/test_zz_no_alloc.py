"""rssm_step_static_scratch: the step for callers that cannot allocate.

Engines whose allocator owns all device memory, or FFI hosts without a device
allocator, cannot hand rssm_step a scratch buffer; this entry point uses an
array compiled into the library instead.  Called through the C ABI it runs
the same kernels on the same inputs as rssm_step with a caller scratch, so it
must give the same output bits and cache updates, on consecutive calls (the
array keeps the previous call's contents: a smaller call with empty and
padding rows follows a larger one), and must refuse a step larger than the
array.  Needs a GPU; collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

from speculative_state_replay_gb300 import _lib, api
from speculative_state_replay_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _entry():
    from speculative_state_replay_gb300 import build

    build.build()
    lib = _lib.load()
    f = lib.rssm_step_static_scratch
    vp, i32 = ctypes.c_void_p, ctypes.c_int32
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.POINTER(_lib.RssmCacheStruct)] + [vp] * 10 + [i32, i32, vp, vp]
    return f


def _cache(wl, gen, dev):
    gc = api.RssmCache(wl.num_slots, wl.nheads, wl.ngroups, wl.max_window, wl.npredicted, wl.state_dtype,
                       device=dev)
    ids = gen.slot_idx()
    act = ids[ids > 0]
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
    api.rssm_init_state(gc, t(gen.init_states(0, act.size)), t(act.astype(np.int32)))
    return gc, ids


def test_static_scratch_step_matches_rssm_step_twice():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    f = _entry()
    dev = torch.device("cuda:0")
    wl = W.config("mamba2_decode", batch=16)
    gen = W.Generator(wl)
    A, D, dtb = gen.params()
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
    gA, gD, gb = t(A), t(D), t(dtb)
    ref, ids = _cache(wl, gen, dev)
    sut, _ = _cache(wl, gen, dev)
    gids = t(ids)
    p_ref = torch.zeros(ids.size, dtype=torch.int32, device=dev)
    p_sut = p_ref.clone()
    scratch = api.alloc_scratch(ref, ids.size, wl.T)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    ptr = lambda x: ctypes.c_void_p(x.data_ptr())  # noqa: E731
    for k in range(3):
        inp = gen.step(k)
        rows, cu = ids.size, None
        if k == 2:
            # a smaller varlen call right after the larger ones: 6 rows, two of
            # them with no tokens and one on the padding slot, so the array still
            # holds records and coefficient blocks of the previous call
            rows = 6
            lens = np.array([3, 0, 4, 1, 0, 2], np.int32)
            cu_h = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
            cu = t(cu_h)
        n = int(cu_h[-1]) if k == 2 else inp.ntok
        x, dt, B, C = (t(inp.x[:n].view(np.int16)), t(inp.dt[:n]), t(inp.B[:n].view(np.int16)),
                       t(inp.C[:n].view(np.int16)))
        sid = gids[:rows].clone()
        if k == 2:
            sid[3] = 0  # padding row
        y_ref = torch.full((n, wl.nheads, 64), 0x7FC0, dtype=torch.int16, device=dev)
        y_sut = y_ref.clone()
        api.rssm_step(ref, x, dt, gA, B, C, gD, gb, sid, p_ref[:rows], wl.T, y_ref, scratch, cu_seqlens=cu)
        rc = f(sut.struct(), ptr(x), ptr(dt), ptr(gA), ptr(B), ptr(C), ptr(gD), ptr(gb), ptr(sid), ptr(p_sut),
               None if cu is None else ptr(cu), rows, wl.T, ptr(y_sut), stream)
        assert rc == 0
        torch.cuda.synchronize()
        assert torch.equal(y_sut, y_ref), k
        for name in ("x_cache", "B_cache", "dt_cache", "state", "ring_start", "error_word"):
            assert torch.equal(getattr(sut, name), getattr(ref, name)), (k, name)
        if k < 2:
            acc = t(inp.accepted)
            api.rssm_accept(ref, gids, p_ref, acc, wl.T)
            api.rssm_accept(sut, gids, p_sut, acc, wl.T)
    torch.cuda.synchronize()
    assert torch.equal(p_ref, p_sut)
    assert int(ref.error_word.item()) == 0


def test_static_scratch_refuses_steps_larger_than_the_array():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    f = _entry()
    dev = torch.device("cuda:0")
    wl = W.config("large_batch", batch=512, num_slots=2)  # needs ~43 MB of scratch
    c = api.RssmCache(wl.num_slots, wl.nheads, wl.ngroups, wl.max_window, wl.npredicted, wl.state_dtype,
                      device=dev)
    assert api.rssm_scratch_bytes(c, wl.batch, wl.T) > (16 << 20)
    buf = torch.zeros(1 << 20, dtype=torch.int32, device=dev)
    p = ctypes.c_void_p(buf.data_ptr())
    out = torch.full((8,), 7, dtype=torch.int32, device=dev)
    rc = f(c.struct(), p, p, p, p, p, p, p, p, p, None, wl.batch, wl.T, ctypes.c_void_p(out.data_ptr()),
           ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 3  # RSSM_ERR_SCRATCH_TOO_SMALL, nothing launched
    torch.cuda.synchronize()
    assert (out == 7).all()
