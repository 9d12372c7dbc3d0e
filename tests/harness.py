"""Shared test drivers: build a cache from a workload and run decode steps.

Only input plumbing lives here; the arithmetic is in the oracle (CPU) or the
CUDA library (GPU).
"""
import numpy as np

from speculative_state_replay_gb300 import workloads as W


def oracle_cache(orc, wl, gen, slot_pad_bytes=None, ring_start=None):
    """Oracle cache initialised like a fresh decode batch of `wl`."""
    pad = wl.slot_pad_bytes if slot_pad_bytes is None else slot_pad_bytes
    c = orc.OracleCache(wl.num_slots, wl.nheads, wl.ngroups, wl.max_window, wl.npredicted, wl.state_dtype,
                        wl.rounding, slot_pad_bytes=pad, read_dtype=wl.read_dtype)
    ids = gen.slot_idx()
    active = ids[ids > 0]
    states = gen.init_states(0, active.size)
    c.init_state(states, active, seed=wl.sr_seed)
    pnat = np.zeros(ids.size, np.int32)
    if wl.prefill_live:
        for b, s in enumerate(ids):
            if s <= 0:
                continue
            x, B, dtp, live = gen.ring_prefill(int(s))
            c.x_view()[s] = x
            c.B_view()[s] = B
            c.dt_view()[s] = dtp
            pnat[b] = live
    rs = gen.ring_start() if ring_start is None else ring_start
    c.ring_start[:] = rs
    return c, ids, pnat


def run_oracle_step(c, wl, params, ids, pnat, inp, seed=None):
    """flush -> step -> accept on the oracle; returns y bits [tok][H][64]."""
    A, D, dt_bias = params
    seed = wl.sr_seed if seed is None else seed
    c.flush(A, ids, pnat, wl.T, cu_seqlens=inp.cu_seqlens, seed=seed)
    y = c.step(inp.x, inp.dt, A, inp.B, inp.C, D, dt_bias, ids, pnat, wl.T, cu_seqlens=inp.cu_seqlens)
    c.accept(ids, pnat, inp.accepted, wl.T, cu_seqlens=inp.cu_seqlens)
    return y


def logical_ring(c, s, arr_view):
    """Ring rows of slot s in logical order (live token 0 first)."""
    return np.roll(arr_view[s], -int(c.ring_start[s]), axis=-2 if arr_view.ndim == 4 else -1)


def tiny(**kw):
    return W.config("tiny", **kw)
