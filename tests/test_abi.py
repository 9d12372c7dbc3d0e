"""The C ABI library (CPU only): it builds, loads, exports every function the
header declares, and rejects bad arguments before touching the GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from speculative_state_replay_gb300 import _lib, build

    try:
        build.nvcc()
    except RuntimeError:
        pytest.skip("nvcc not available")
    build.build()
    return _lib.load()


def header_functions():
    text = open(os.path.join(ROOT, "include", "rssm.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(rssm_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_entry_points():
    names = header_functions()
    for n in ("rssm_init_state", "rssm_flush", "rssm_step", "rssm_accept", "rssm_scratch_bytes",
              "rssm_status_string", "rssm_step_precompute", "rssm_step_readout", "rssm_step_gated",
              "rssm_step_readout_gated"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in header_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_binding_exports_match_header():
    from speculative_state_replay_gb300 import _lib

    assert set(_lib.EXPORTS) <= set(header_functions())


def _cache(**kw):
    from speculative_state_replay_gb300 import _lib

    c = _lib.RssmCacheStruct()
    c.num_slots, c.nheads, c.ngroups, c.dim, c.dstate = 5, 8, 1, 64, 128
    c.max_window, c.npredicted, c.state_dtype, c.rounding = 16, 4, 1, 0
    base = 1 << 20  # fake, aligned, never dereferenced on these paths
    c.state, c.state_slot_stride = base, 8 * 64 * 128
    c.scale, c.scale_slot_stride = base, 8 * 64
    c.x_cache, c.x_slot_stride = base, 8 * 20 * 64
    c.B_cache, c.B_slot_stride = base, 1 * 20 * 128
    c.dt_cache, c.dt_slot_stride = base, 8 * 20
    c.ring_start = c.flush_epoch = c.error_word = base
    for k, v in kw.items():
        setattr(c, k, v)
    return c


def test_scratch_bytes_and_shape_validation(lib):
    good = _cache()
    n = lib.rssm_scratch_bytes(ctypes.byref(good), 64, 4)
    assert n >= 64 * 32
    assert lib.rssm_scratch_bytes(ctypes.byref(_cache(dim=32)), 64, 4) == 0
    assert lib.rssm_scratch_bytes(ctypes.byref(_cache(ngroups=3)), 64, 4) == 0
    assert lib.rssm_scratch_bytes(ctypes.byref(_cache(npredicted=20)), 64, 4) == 0  # L > 32
    assert lib.rssm_scratch_bytes(ctypes.byref(_cache(x_slot_stride=10)), 64, 4) == 0
    assert lib.rssm_scratch_bytes(ctypes.byref(_cache(state=(1 << 20) + 8)), 64, 4) == 0  # misaligned
    assert lib.rssm_scratch_bytes(ctypes.byref(good), 64, 9) == 0


def test_entry_points_reject_bad_arguments_before_launching(lib):
    c = ctypes.byref(_cache())
    nul = None
    assert lib.rssm_step(None, *([nul] * 10), 4, 4, nul, nul, 0, nul) == 1
    assert lib.rssm_step(c, *([nul] * 10), 4, 4, nul, nul, 0, nul) == 1  # null inputs
    assert lib.rssm_step(ctypes.byref(_cache(dim=32)), *([nul] * 10), 4, 4, nul, nul, 0, nul) == 2
    p = ctypes.c_void_p(1 << 20)
    args = [p] * 10
    assert lib.rssm_step(c, *args, 4, 5, p, p, 1 << 30, nul) == 2  # T > npredicted
    assert lib.rssm_step(c, *args, 4, 4, p, p, 16, nul) == 3  # scratch too small
    assert lib.rssm_flush(c, p, p, p, nul, 4, 4, 2, 0, p, 1 << 20, nul) == 1  # force not 0/1
    assert lib.rssm_flush(c, p, p, p, nul, 4, 4, 0, 0, p, 8, nul) == 3
    assert lib.rssm_init_state(c, ctypes.c_void_p((1 << 20) + 4), p, 2, 0, nul) == 1  # misaligned states
    assert lib.rssm_accept(c, nul, nul, nul, nul, 4, 4, nul) == 1
    # rssm_accept_flush(cache, A, slot_idx, pnat, accepted, accept_cu, accept_T, cu, batch, T, force, seed, ...)
    assert lib.rssm_accept_flush(c, p, p, p, nul, nul, 4, nul, 4, 4, 0, 0, p, 1 << 20, nul) == 1  # no accepted
    assert lib.rssm_accept_flush(c, p, p, p, p, nul, -1, nul, 4, 4, 0, 0, p, 1 << 20, nul) == 1  # accept_T < 0
    assert lib.rssm_accept_flush(c, p, p, p, p, nul, 4, nul, 4, 4, 2, 0, p, 1 << 20, nul) == 1  # force not 0/1
    assert lib.rssm_accept_flush(c, p, p, p, p, nul, 4, nul, 4, 4, 0, 0, p, 8, nul) == 3
    assert lib.rssm_accept_flush(c, p, p, p, nul, nul, 4, nul, 0, 4, 0, 0, p, 0, nul) == 0  # empty batch
    # empty batches are a no-op
    assert lib.rssm_step(c, *args, 0, 4, p, p, 0, nul) == 0
    assert lib.rssm_flush(c, p, p, p, nul, 0, 4, 0, 0, p, 0, nul) == 0
    for s, text in [(0, b"ok"), (3, b"scratch buffer too small")]:
        assert lib.rssm_status_string(s) == text


def test_gated_entry_points_reject_bad_arguments_before_launching(lib):
    """rssm_step_gated / rssm_step_readout_gated: the gate pointer is checked
    (16-byte aligned) with everything else before any launch; z = NULL and an
    empty batch behave as the ungated calls."""
    c = ctypes.byref(_cache())
    nul = None
    p = ctypes.c_void_p(1 << 20)
    z_bad = ctypes.c_void_p((1 << 20) + 4)
    args = [p] * 10
    for fn in (lib.rssm_step_gated, lib.rssm_step_readout_gated):
        assert fn(None, *([nul] * 10), 4, 4, p, nul, nul, 0, nul) == 1
        assert fn(c, *args, 4, 4, z_bad, p, p, 1 << 30, nul) == 1  # misaligned z
        assert fn(c, *args, 4, 5, p, p, p, 1 << 30, nul) == 2  # T > npredicted
        assert fn(c, *args, 4, 4, p, p, p, 16, nul) == 3  # scratch too small
        assert fn(c, *args, 0, 4, z_bad, p, p, 0, nul) == 0  # empty batch: no-op


def test_binding_refuses_token_tensors_shorter_than_batch_times_T():
    """Without cu_seqlens the kernels address batch * T tokens in every
    per-token tensor: the binding checks the sizes on the host (no device read)
    and raises before calling the library."""
    import torch

    from speculative_state_replay_gb300 import api

    c = api.RssmCache(5, 8, 1, 16, 4, api.BF16, device="cpu")
    batch, T = 3, 4
    ids = torch.zeros(batch, dtype=torch.int32)
    f = torch.zeros(8)
    x = torch.zeros((batch * T - 1, 8, 64), dtype=torch.int16)  # one token short
    dt = torch.zeros((batch * T, 8))
    B = torch.zeros((batch * T, 1, 128), dtype=torch.int16)
    out = torch.zeros((batch * T, 8, 64), dtype=torch.int16)
    scratch = torch.zeros(1 << 16, dtype=torch.uint8)
    for fn in (api.rssm_step, api.rssm_step_precompute, api.rssm_step_readout, api.rssm_flush_step):
        with pytest.raises(ValueError, match="x holds"):
            fn(c, x, dt, f, B, B, f, f, ids, ids, T, out, scratch)
    with pytest.raises(ValueError, match="out holds"):
        api.rssm_step(c, out, dt, f, B, B, f, f, ids, ids, T, x, scratch)
    with pytest.raises(ValueError, match="z holds"):
        api.rssm_step(c, out, dt, f, B, B, f, f, ids, ids, T, out, scratch, z=x)


def test_wait_selftest_rejects_bad_arguments(lib):
    assert lib.rssm_selftest_wait_timeout(None, 50, None) == 1
    p = ctypes.c_void_p(1 << 20)
    assert lib.rssm_selftest_wait_timeout(p, 0, None) == 1
    assert lib.rssm_selftest_wait_timeout(p, 20000, None) == 1
    assert lib.rssm_selftest_wait_timeout(ctypes.c_void_p((1 << 20) + 2), 50, None) == 1


def test_read_checkpoint_fields_are_validated(lib):
    """A read checkpoint's format, pointers and strides are checked before any
    launch; NVFP4 is a read format only."""
    base = 1 << 20
    ok8 = _cache(read_state=base, read_slot_stride=8 * 64 * 128, read_scale=base, read_scale_slot_stride=8 * 64,
                 read_dtype=4)
    assert lib.rssm_scratch_bytes(ctypes.byref(ok8), 4, 4) > 0
    ok4 = _cache(read_state=base, read_slot_stride=8 * 64 * 64, read_sf=base, read_sf_slot_stride=8 * 64 * 8,
                 read_gs=base, read_dtype=5)
    assert lib.rssm_scratch_bytes(ctypes.byref(ok4), 4, 4) > 0
    bad = [
        _cache(read_state=base, read_slot_stride=8 * 64 * 128, read_scale=base, read_scale_slot_stride=8 * 64,
               read_dtype=2),                                     # not a read format
        _cache(read_state=base, read_slot_stride=8 * 64 * 128, read_dtype=3),  # 8-bit without scales
        _cache(read_state=base, read_slot_stride=8 * 64 * 64, read_gs=base, read_dtype=5),  # NVFP4 without block scales
        _cache(read_state=base, read_slot_stride=8 * 64 * 64, read_sf=base, read_sf_slot_stride=8 * 64 * 8,
               read_dtype=5),                                     # NVFP4 without global scales
        _cache(read_state=base, read_slot_stride=8 * 64 * 32, read_sf=base, read_sf_slot_stride=8 * 64 * 8,
               read_gs=base, read_dtype=5),                       # codes stride too small
        _cache(state_dtype=5),                                    # NVFP4 recurrence state
    ]
    for c in bad:
        assert lib.rssm_scratch_bytes(ctypes.byref(c), 4, 4) == 0
