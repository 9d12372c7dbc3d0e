"""The oracle's NVFP4 read checkpoint (CPU only).

Source: vLLM API docs, replayssm_cutedsl, initialize_replayssm_state (NVFP4
branch: the group maxima of each state, their maximum divided by 6 * 448 as
the global scale, 1 where that maximum is 0) and the NVFP4 kernels' state_lo /
sf_lo / sg_meta arguments; vLLM PR #65660, Claims: read checkpoints use
nearest encoding.  Reading: FP4 E2M1 codes, one E4M3 scale per 16 consecutive
dstate values, one FP32 global scale per slot, set at init and kept by the
slot's flushes.

Pins (each against something other than the oracle's own code):
  * the 16 E2M1 codes decode to the format's published value table
  * E2M1 nearest rounding equals a brute-force nearest search over that table
    with ties to the even code
  * block scales are the E4M3 nearest encoding of block max / (6 gs), by
    PyTorch's float8_e4m3fn cast
  * every decoded value is the nearest point of its block's scaled grid
  * the global scale is max|state| / 2688 (1 for a zero state)
  * init and flush write the nearest encoding of the fp32 values; the step's
    outputs are the float64 brute-force recurrence from the decoded checkpoint;
    the recurrence state does not depend on the read checkpoint
"""
import numpy as np
import pytest
import torch

from speculative_state_replay_gb300 import workloads as W
from tests import brute

NVFP4 = 5
# OCP Microscaling Formats (MX) v1.0, FP4 E2M1: the 8 magnitudes of codes 0..7
E2M1_TABLE = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def e4m3_value(bits):
    return torch.from_numpy(np.asarray(bits, np.uint8).copy()).view(torch.float8_e4m3fn).float().numpy()


def e2m1_value(code):
    code = np.asarray(code, np.int64)
    mag = np.array(E2M1_TABLE)[code & 7]
    return np.where(code & 8, -mag, mag)


def test_e2m1_codes_decode_to_the_published_table(orc):
    got = orc.e2m1_decode(np.arange(16, dtype=np.uint8))
    assert np.array_equal(got[:8], np.float32(E2M1_TABLE))
    assert np.array_equal(got[8:], -np.float32(E2M1_TABLE))
    assert np.signbit(got[8]) and not np.signbit(got[0])


def test_e2m1_nearest_is_the_brute_force_nearest_with_ties_to_even(orc):
    rng = np.random.default_rng(3)
    mids = np.array([(a + b) / 2 for a, b in zip(E2M1_TABLE, E2M1_TABLE[1:])])
    v = np.concatenate([rng.uniform(-8, 8, 20000), mids, -mids, E2M1_TABLE, [6.5, 7.0, 100.0, -9.0, 1e-9, -1e-9]])
    v = v.astype(np.float32)
    got = orc.f32_to_e2m1_bits(v)
    mags = np.array(E2M1_TABLE)
    for x, c in zip(v.astype(np.float64), got):
        a = min(abs(x), 6.0)
        d = np.abs(mags - a)
        best = np.nonzero(d == d.min())[0]
        m = best[0] if best.size == 1 else [k for k in best if k % 2 == 0][0]  # tie: the even code
        assert (c & 7) == m, (x, c)
        assert bool(c & 8) == bool(np.signbit(np.float32(x))), (x, c)


def _rows(seed, n=24):
    rng = np.random.default_rng(seed)
    a = (rng.standard_normal((n, 128)) * 0.1).astype(np.float32)
    a[3] = 0.0                  # an all-zero row
    a[5, 17] = 0.9              # one large value in a block
    a[7, :16] = 1e-12           # a block too small for its scale (codes 0)
    return a


def test_block_scales_are_the_e4m3_nearest_of_block_max(orc):
    a = _rows(1)
    gs = orc.nvfp4_global_scale(a)
    _, sf = orc.quantize_rows_nvfp4(a, gs)
    bmax = np.abs(a.reshape(-1, 8, 16)).max(axis=2)
    want = torch.from_numpy(bmax / (np.float32(6.0) * np.float32(gs))).to(torch.float8_e4m3fn)
    assert np.array_equal(sf, want.view(torch.uint8).numpy())


def test_codes_are_the_nearest_points_of_their_block_grid(orc):
    a = _rows(2)
    gs = np.float32(orc.nvfp4_global_scale(a))
    codes, sf = orc.quantize_rows_nvfp4(a, gs)
    lo, hi = codes & 0xF, codes >> 4
    c = np.stack([lo, hi], axis=-1).reshape(a.shape)
    q = (e4m3_value(sf).astype(np.float32) * gs).astype(np.float64)  # [rows][8]
    qe = np.repeat(q, 16, axis=1)
    dec = e2m1_value(c) * qe
    grid = np.array(E2M1_TABLE)
    for i in range(a.shape[0]):
        for n in range(128):
            v, qq = float(a[i, n]), qe[i, n]
            if qq == 0:
                assert dec[i, n] == 0
                continue
            d = np.abs(np.abs(v) - grid * qq)
            if np.sort(d)[1] - d.min() < 1e-6 * qq:
                continue  # an exact tie (decided by the even code)
            assert abs(abs(dec[i, n]) - grid[d.argmin()] * qq) <= 1e-12, (i, n)
    # error bound: half a grid step of the block (at most 1 q) inside the range
    assert np.all(np.abs(dec - a) <= qe + 1e-12)


def test_global_scale(orc):
    a = _rows(4)
    assert orc.nvfp4_global_scale(a) == np.float32(np.abs(a).max()) / np.float32(2688.0)
    assert orc.nvfp4_global_scale(np.zeros((3, 128), np.float32)) == 1.0


def _caches(orc, wl, gen, state_dtype, rounding):
    out = []
    ids = gen.slot_idx()
    active = ids[ids > 0]
    states = gen.init_states(0, active.size)
    for rd in (NVFP4, None):
        c = orc.OracleCache(wl.num_slots, wl.nheads, wl.ngroups, wl.max_window, wl.npredicted, state_dtype, rounding,
                            read_dtype=rd)
        c.init_state(states, active, seed=7)
        for s in active:
            x, B, dtp, live = gen.ring_prefill(int(s))
            c.x_view()[s], c.B_view()[s], c.dt_view()[s] = x, B, dtp
        c.ring_start[:] = gen.ring_start()
        out.append(c)
    pnat = np.array([gen.ring_prefill(int(s))[3] if s > 0 else 0 for s in ids], np.int32)
    return out[0], out[1], ids, active, states, pnat


def test_init_writes_the_nearest_encoding_with_the_slot_global_scale(orc):
    wl = W.config("tiny", prefill_live=12)
    gen = W.Generator(wl)
    c, _, ids, active, states, _ = _caches(orc, wl, gen, W.F16, W.STOCHASTIC)
    for i, s in enumerate(active):
        gs = orc.nvfp4_global_scale(states[i])
        assert c.read_gs[s] == np.float32(gs)
        for h in range(wl.nheads):
            codes, sf = orc.quantize_rows_nvfp4(states[i, h], gs)
            assert np.array_equal(c.read_state_view()[s, h], codes)
            assert np.array_equal(c.read_sf_view()[s, h], sf)


def test_flush_writes_the_nearest_encoding_of_the_fold(orc):
    """With an f32 recurrence the recurrence state holds the fold's fp32 result
    exactly; the NVFP4 read copy is its encoding with the slot's init scale."""
    wl = W.config("tiny", prefill_live=14)
    gen = W.Generator(wl)
    A, _, _ = gen.params()
    c, _, ids, active, states, pnat = _caches(orc, wl, gen, W.F32, W.NEAREST)
    gs0 = c.read_gs.copy()
    c.flush(A, ids, pnat, wl.T, force=1, seed=7)
    assert np.array_equal(c.read_gs, gs0)
    for s in active:
        for h in range(wl.nheads):
            codes, sf = orc.quantize_rows_nvfp4(c.state_view()[s, h], c.read_gs[s])
            assert np.array_equal(c.read_state_view()[s, h], codes)
            assert np.array_equal(c.read_sf_view()[s, h], sf)


def test_step_reads_s0_from_the_nvfp4_checkpoint(orc):
    wl = W.config("tiny", prefill_live=12, ring_start_random=True)
    gen = W.Generator(wl)
    A, D, dtb = gen.params()
    c, _, ids, active, _, pnat = _caches(orc, wl, gen, W.F16, W.STOCHASTIC)
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
            codes = c.read_state_view()[s, h]
            cc = np.stack([codes & 0xF, codes >> 4], axis=-1).reshape(64, 128)
            q = np.repeat(e4m3_value(c.read_sf_view()[s, h]).astype(np.float64), 16, axis=1)
            S0 = e2m1_value(cc) * q * float(c.read_gs[s])
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


def test_recurrence_does_not_depend_on_the_nvfp4_checkpoint(orc):
    wl = W.config("tiny", prefill_live=12, ring_start_random=True)
    gen = W.Generator(wl)
    A, D, dtb = gen.params()
    sep, one, ids, _, _, pnat = _caches(orc, wl, gen, W.F16, W.STOCHASTIC)
    p_sep, p_one = pnat.copy(), pnat.copy()
    for k in range(wl.steps):
        inp = gen.step(k)
        for c, pn in ((sep, p_sep), (one, p_one)):
            c.flush(A, ids, pn, wl.T, seed=7)
            c.step(inp.x, inp.dt, A, inp.B, inp.C, D, dtb, ids, pn, wl.T)
            c.accept(ids, pn, inp.accepted, wl.T)
        for name in ("state", "x_cache", "B_cache", "dt_cache", "ring_start", "flush_epoch"):
            assert np.array_equal(getattr(sep, name), getattr(one, name)), (k, name)
    assert sep.flush_epoch.max() >= 1
