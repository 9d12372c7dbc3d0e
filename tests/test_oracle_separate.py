"""The oracle's separate read checkpoint (CPU only).

vLLM PR #65660 ("separate CuTeDSL ReplaySSM checkpoints", Overview and
Claims): the recurrence checkpoint (FP16 with stochastic rounding there) takes
the FP32 flush work, and an 8-bit read checkpoint, encoded to nearest, is what
the readout reads.  Reading taken: both are rounded from the same fp32 values
(the prefill states at init, the fold's accumulators at every flush).

Pins:
  * at init the read checkpoint is the pinned quantiser's nearest encoding of
    the FP32 states, bit for bit
  * after a flush it is the quantiser's nearest encoding of the fold's fp32
    result, bit for bit (an f32 recurrence holds that result exactly)
  * the step's outputs are the float64 brute-force recurrence started from the
    decoded read checkpoint
  * the recurrence state, rings and bookkeeping do not depend on the read
    checkpoint
"""
import numpy as np
import pytest

from speculative_state_replay_gb300 import workloads as W
from tests import brute


def _caches(orc, wl, gen, read_dtype, state_dtype=None, rounding=None):
    """The same fresh decode batch twice: with and without a read checkpoint."""
    sd = wl.state_dtype if state_dtype is None else state_dtype
    rnd = wl.rounding if rounding is None else rounding
    out = []
    ids = gen.slot_idx()
    active = ids[ids > 0]
    states = gen.init_states(0, active.size)
    for rd in (read_dtype, None):
        c = orc.OracleCache(wl.num_slots, wl.nheads, wl.ngroups, wl.max_window, wl.npredicted, sd, rnd,
                            read_dtype=rd)
        c.init_state(states, active, seed=7)
        for s in active:
            x, B, dtp, live = gen.ring_prefill(int(s))
            c.x_view()[s], c.B_view()[s], c.dt_view()[s] = x, B, dtp
        c.ring_start[:] = gen.ring_start()
        out.append(c)
    pnat = np.array([gen.ring_prefill(int(s))[3] if s > 0 else 0 for s in ids], np.int32)
    return out[0], out[1], ids, active, states, pnat


@pytest.mark.parametrize("read_dtype", [W.I8, W.E4M3])
def test_read_checkpoint_at_init_is_the_nearest_encoding(orc, read_dtype):
    wl = W.config("tiny", state_dtype=W.F16, rounding=W.STOCHASTIC, prefill_live=12)
    gen = W.Generator(wl)
    c, _, ids, active, states, _ = _caches(orc, wl, gen, read_dtype)
    for i, s in enumerate(active):
        for h in range(wl.nheads):
            codes, scales = orc.quantize_rows(read_dtype, W.NEAREST, states[i, h], h=h, s=int(s))
            assert np.array_equal(c.read_state_view()[s, h].view(codes.dtype), codes)
            assert np.array_equal(c.read_scale_view()[s, h], scales)


@pytest.mark.parametrize("read_dtype", [W.I8, W.E4M3])
def test_read_checkpoint_after_a_flush_is_the_nearest_encoding_of_the_fold(orc, read_dtype):
    """With an f32 recurrence the recurrence state holds the fold's fp32
    result exactly; the read checkpoint must be its nearest encoding."""
    wl = W.config("tiny", prefill_live=14)
    gen = W.Generator(wl)
    A, D, dtb = gen.params()
    c, _, ids, active, _, pnat = _caches(orc, wl, gen, read_dtype, state_dtype=W.F32, rounding=W.NEAREST)
    p0 = pnat.copy()
    c.flush(A, ids, pnat, wl.T, force=1, seed=7)
    assert (c.flush_epoch[active] == 1).all()
    for b, s in enumerate(ids):
        if s <= 0:
            continue
        for h in range(wl.nheads):
            acc = c.state_view()[s, h]
            codes, scales = orc.quantize_rows(read_dtype, W.NEAREST, acc, h=h, s=int(s), epoch=1)
            assert np.array_equal(c.read_state_view()[s, h].view(codes.dtype), codes), (b, h, int(p0[b]))
            assert np.array_equal(c.read_scale_view()[s, h], scales)


def test_step_reads_s0_from_the_read_checkpoint(orc):
    """y = the float64 recurrence started from the decoded read checkpoint
    (int8 read checkpoint of an FP16 stochastically rounded recurrence)."""
    wl = W.config("tiny", state_dtype=W.F16, rounding=W.STOCHASTIC, prefill_live=12, ring_start_random=True)
    gen = W.Generator(wl)
    A, D, dtb = gen.params()
    c, _, ids, active, _, pnat = _caches(orc, wl, gen, W.I8)
    inp = gen.step(0)
    _, y64 = c.copy().step(inp.x, inp.dt, A, inp.B, inp.C, D, dtb, ids, pnat, wl.T, want_f64=True)
    L = wl.L
    worst = 0.0
    for b, s in enumerate(ids):
        tok0, Tb = b * wl.T, wl.T
        if s <= 0:
            continue
        r, p = int(c.ring_start[s]), int(pnat[b])
        for h in range(wl.nheads):
            g = h // wl.hpg
            S0 = c.read_state_view()[s, h].view(np.int8).astype(np.float64) * \
                c.read_scale_view()[s, h].astype(np.float64)[:, None]
            live = [(brute.bf16_to_f64(c.x_view()[s, h, (r + k) % L]), brute.bf16_to_f64(c.B_view()[s, g, (r + k) % L]),
                     float(c.dt_view()[s, h, (r + k) % L])) for k in range(p)]
            new = []
            for t in range(Tb):
                tok = tok0 + t
                v = np.float32(inp.dt[tok, h]) + np.float32(dtb[h])
                new.append((brute.bf16_to_f64(inp.x[tok, h]), brute.bf16_to_f64(inp.B[tok, g]),
                            float(brute.softplus64(np.float64(v))), brute.bf16_to_f64(inp.C[tok, g])))
            ys, _, _ = brute.recurrence(S0, live, new, float(A[h]), float(D[h]))
            got = y64[tok0:tok0 + Tb, h]
            worst = max(worst, float(np.abs(got - ys).max() / (np.abs(ys).max() + 1e-30)))
    assert worst < 2e-5, worst


def test_recurrence_does_not_depend_on_the_read_checkpoint(orc):
    """Several flush -> step -> accept iterations: the recurrence state, rings,
    ring_start, pnat and epochs equal those of the oracle without a read
    checkpoint bit for bit (only the outputs read S0 from the read copy)."""
    wl = W.config("tiny", state_dtype=W.F16, rounding=W.STOCHASTIC, prefill_live=12, ring_start_random=True)
    gen = W.Generator(wl)
    A, D, dtb = gen.params()
    sep, one, ids, _, _, pnat = _caches(orc, wl, gen, W.E4M3)
    p_sep, p_one = pnat.copy(), pnat.copy()
    for k in range(wl.steps):
        inp = gen.step(k)
        for c, pn in ((sep, p_sep), (one, p_one)):
            c.flush(A, ids, pn, wl.T, seed=7)
            c.step(inp.x, inp.dt, A, inp.B, inp.C, D, dtb, ids, pn, wl.T)
            c.accept(ids, pn, inp.accepted, wl.T)
        assert np.array_equal(p_sep, p_one)
        for name in ("state", "x_cache", "B_cache", "dt_cache", "ring_start", "flush_epoch", "error_word"):
            assert np.array_equal(getattr(sep, name), getattr(one, name)), (k, name)
    assert sep.flush_epoch.max() >= 1
