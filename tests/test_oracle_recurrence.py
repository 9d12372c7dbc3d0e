"""The oracle against the brute-force recurrence and the invariants the pages
state (CPU only).

Pins:
  * checkpoint + replay (oracle) == token-by-token recurrence (float64)
  * flush result == recurrence state after the accepted prefix
  * flush-then-step output == step-without-flush output (f32 state)
  * p = 0, T = 1 is the single-step selective_state_update; C = 0 gives D x
  * rejected drafts never change the checkpoint (vLLM PR #65660, Details)
  * outputs and logical rings do not depend on the initial ring_start
    (FlashInfer PR #3975, Description item 2: positions are taken mod L)
  * ring bookkeeping equals a plain list model
  * packed cu_seqlens == separate per-request calls; padded slot pages ==
    contiguous pages; init ignores ids <= 0 or >= S
  * output gate: y * silu(z) == torch's silu on the float64 recurrence; z = 0
    gives zeros, z = 40 gives z * y exactly
"""
import numpy as np
import pytest

from speculative_state_replay_gb300 import workloads as W
from tests import brute
from tests.harness import logical_ring, oracle_cache, run_oracle_step


def _row_tokens(inp, b, T):
    if inp.cu_seqlens is None:
        return b * T, T
    return int(inp.cu_seqlens[b]), int(inp.cu_seqlens[b + 1] - inp.cu_seqlens[b])


def _state_f64(c, s, h):
    st = c.state_view()[s, h]
    if c.state_dtype == W.F32:
        return st.astype(np.float64)
    if c.state_dtype == W.BF16:
        return brute.bf16_to_f64(st)
    if c.state_dtype == W.F16:
        return st.view(np.float16).astype(np.float64)
    raise NotImplementedError


def _bruteforce_row(c, wl, params, s, p, h, inp, tok0, Tb):
    A, D, dt_bias = params
    g = h // wl.hpg
    r, L = int(c.ring_start[s]), wl.L
    live = []
    for k in range(p):
        pos = (r + k) % L
        live.append((brute.bf16_to_f64(c.x_view()[s, h, pos]), brute.bf16_to_f64(c.B_view()[s, g, pos]),
                     float(c.dt_view()[s, h, pos])))
    new = []
    for t in range(Tb):
        tok = tok0 + t
        v = np.float32(inp.dt[tok, h]) + np.float32(dt_bias[h])
        new.append((brute.bf16_to_f64(inp.x[tok, h]), brute.bf16_to_f64(inp.B[tok, g]),
                    float(brute.softplus64(np.float64(v))), brute.bf16_to_f64(inp.C[tok, g])))
    return brute.recurrence(_state_f64(c, s, h), live, new, float(A[h]), float(D[h]))


@pytest.mark.parametrize("varlen", [False, True])
def test_step_equals_bruteforce_recurrence(orc, varlen):
    wl = W.config("tiny", prefill_live=12, ring_start_random=True, varlen=varlen)
    gen = W.Generator(wl)
    params = gen.params()
    c, ids, pnat = oracle_cache(orc, wl, gen)
    inp = gen.step(0)
    y_bits, y64 = c.copy().step(inp.x, inp.dt, *params[:1], inp.B, inp.C, params[1], params[2], ids, pnat, wl.T,
                                cu_seqlens=inp.cu_seqlens, want_f64=True)
    worst = 0.0
    for b, s in enumerate(ids):
        tok0, Tb = _row_tokens(inp, b, wl.T)
        if s <= 0:
            assert not y64[tok0:tok0 + Tb].any()
            continue
        for h in range(wl.nheads):
            ys, _, _ = _bruteforce_row(c, wl, params, int(s), int(pnat[b]), h, inp, tok0, Tb)
            got = y64[tok0:tok0 + Tb, h]
            scale = np.abs(ys).max() + 1e-30
            worst = max(worst, float(np.abs(got - ys).max() / scale))
    assert worst < 2e-5, worst
    # the bf16 output is the float64 value rounded once
    assert np.array_equal(y_bits, orc.f32_to_bf16_bits(y64.astype(np.float32)))


def test_flush_equals_bruteforce_state(orc):
    wl = W.config("tiny", prefill_live=16, ring_start_random=True)
    gen = W.Generator(wl)
    A, D, dt_bias = gen.params()
    c, ids, pnat = oracle_cache(orc, wl, gen)
    before = c.copy()
    p0 = pnat.copy()
    c.flush(A, ids, pnat, wl.T, force=1)
    for b, s in enumerate(ids):
        if s <= 0:
            continue
        assert pnat[b] == 0
        assert c.ring_start[s] == (before.ring_start[s] + p0[b]) % wl.L
        assert c.flush_epoch[s] == 1
        for h in range(wl.nheads):
            inp_none = W.StepInputs(x=None, dt=None, B=None, C=None, accepted=None, cu_seqlens=None, ntok=0)
            _, S_live, _ = _bruteforce_row(before, wl, (A, D, dt_bias), int(s), int(p0[b]), h, inp_none, 0, 0)
            got = c.state_view()[s, h].astype(np.float64)
            assert np.abs(got - S_live).max() <= 1e-5 * (np.abs(S_live).max() + 1e-30)


def test_flush_then_step_equals_step_without_flush(orc):
    wl = W.config("tiny", prefill_live=16, ring_start_random=True)
    gen = W.Generator(wl)
    A, D, dt_bias = gen.params()
    c, ids, pnat = oracle_cache(orc, wl, gen)
    inp = gen.step(3)
    # keep p + T within the ring for the no-flush path
    pnat = np.minimum(pnat, wl.L - wl.T).astype(np.int32)
    a, pa = c.copy(), pnat.copy()
    a.flush(A, ids, pa, wl.T, force=1)
    _, ya = a.step(inp.x, inp.dt, A, inp.B, inp.C, D, dt_bias, ids, pa, wl.T, want_f64=True)
    _, yb = c.copy().step(inp.x, inp.dt, A, inp.B, inp.C, D, dt_bias, ids, pnat, wl.T, want_f64=True)
    assert np.abs(ya - yb).max() <= 1e-5 * np.abs(yb).max()


def test_single_token_from_empty_ring_is_plain_ssu(orc):
    """p = 0, T = 1: y = (e^{A dt'} S0 + dt' x (x) B) C + D x, the textbook update."""
    wl = W.config("tiny", T=1, npredicted=1)
    gen = W.Generator(wl)
    A, D, dt_bias = gen.params()
    c, ids, pnat = oracle_cache(orc, wl, gen)
    inp = gen.step(0)
    _, y64 = c.copy().step(inp.x, inp.dt, A, inp.B, inp.C, D, dt_bias, ids, pnat, 1, want_f64=True)
    for b, s in enumerate(ids):
        if s <= 0:
            continue
        for h in range(wl.nheads):
            g = h // wl.hpg
            dtp = float(brute.softplus64(np.float32(inp.dt[b, h]) + np.float32(dt_bias[h])))
            x, B, C = (brute.bf16_to_f64(inp.x[b, h]), brute.bf16_to_f64(inp.B[b, g]),
                       brute.bf16_to_f64(inp.C[b, g]))
            S1 = np.exp(A[h] * dtp) * c.state_view()[s, h].astype(np.float64) + dtp * np.outer(x, B)
            want = S1 @ C + D[h] * x
            assert np.abs(y64[b, h] - want).max() <= 1e-5 * np.abs(want).max()


def test_zero_C_gives_Dx_and_zero_inputs_give_zero(orc):
    wl = W.config("tiny", prefill_live=10)
    gen = W.Generator(wl)
    A, D, dt_bias = gen.params()
    c, ids, pnat = oracle_cache(orc, wl, gen)
    inp = gen.step(1)
    C0 = np.zeros_like(inp.C)
    y = c.copy().step(inp.x, inp.dt, A, inp.B, C0, D, dt_bias, ids, pnat, wl.T)
    xf = brute.bf16_to_f64(inp.x)
    want = orc.f32_to_bf16_bits((D[None, :, None].astype(np.float64) * xf).astype(np.float32))
    for b, s in enumerate(ids):
        sl = slice(b * wl.T, (b + 1) * wl.T)
        assert np.array_equal(y[sl], want[sl] if s > 0 else np.zeros_like(want[sl]))
    z = c.copy()
    z.state[:] = 0
    z.x_cache[:] = 0
    y = z.step(np.zeros_like(inp.x), inp.dt, A, inp.B, inp.C, D, dt_bias, ids, pnat, wl.T)
    assert not (y & 0x7FFF).any()


def test_rejected_drafts_never_reach_the_checkpoint(orc):
    wl = W.config("tiny", state_dtype=W.BF16)
    gen = W.Generator(wl)
    params = gen.params()
    a, ids, pa = oracle_cache(orc, wl, gen)
    b_, pb = a.copy(), pa.copy()
    rng = np.random.default_rng(7)
    ya_all, yb_all = [], []
    for k in range(wl.steps):
        inp = gen.step(k)
        ya_all.append(run_oracle_step(a, wl, params, ids, pa, inp))
        yb_all.append(run_oracle_step(b_, wl, params, ids, pb, inp))
        # scribble over every rejected (appended but not accepted) ring entry of copy b
        for row, s in enumerate(ids):
            if s <= 0:
                continue
            for i in range(int(inp.accepted[row]), wl.T):
                pos = (int(b_.ring_start[s]) + int(pb[row]) - int(inp.accepted[row]) + i) % wl.L
                b_.x_view()[s, :, pos] = rng.integers(0, 65535, (wl.nheads, 64), dtype=np.uint16) & 0x3FFF
                b_.B_view()[s, :, pos] = rng.integers(0, 65535, (wl.ngroups, 128), dtype=np.uint16) & 0x3FFF
                b_.dt_view()[s, :, pos] = rng.uniform(0, 5, wl.nheads)
        assert np.array_equal(a.state, b_.state), k
        assert np.array_equal(ya_all[-1], yb_all[-1]), k
    assert a.flush_epoch.max() >= 1  # the run did flush


def test_outputs_do_not_depend_on_initial_ring_start(orc):
    wl = W.config("tiny", state_dtype=W.BF16)
    gen = W.Generator(wl)
    params = gen.params()
    runs = []
    for r0 in (0, 7, wl.L - 1):
        c, ids, p = oracle_cache(orc, wl, gen, ring_start=np.full(wl.num_slots, r0, np.int32))
        ys = [run_oracle_step(c, wl, params, ids, p, gen.step(k)) for k in range(wl.steps)]
        rings = [(logical_ring(c, s, c.x_view()), logical_ring(c, s, c.B_view()), logical_ring(c, s, c.dt_view()))
                 for s in ids if s > 0]
        runs.append((ys, c.state.copy(), rings, p.copy(), c.flush_epoch.copy()))
    for other in runs[1:]:
        for ya, yb in zip(runs[0][0], other[0]):
            assert np.array_equal(ya, yb)
        assert np.array_equal(runs[0][1], other[1])
        for ra, rb in zip(runs[0][2], other[2]):
            for xa, xb in zip(ra, rb):
                assert np.array_equal(xa, xb)
        assert np.array_equal(runs[0][3], other[3]) and np.array_equal(runs[0][4], other[4])


def test_ring_bookkeeping_equals_list_model(orc):
    """ring_start / pnat / epoch / live ring contents against a list model."""
    wl = W.config("tiny", state_dtype=W.BF16, ring_start_random=True)
    gen = W.Generator(wl)
    params = gen.params()
    c, ids, p = oracle_cache(orc, wl, gen)
    model = {int(s): {"start": int(c.ring_start[s]), "live": [], "epoch": 0} for s in ids if s > 0}
    for k in range(wl.steps):
        inp = gen.step(k)
        for row, s in enumerate(ids):
            if s <= 0:
                continue
            m = model[int(s)]
            if len(m["live"]) + wl.T > wl.max_window:  # flush rule: pnat + T > max_window
                m["start"] = (m["start"] + len(m["live"])) % wl.L
                m["live"] = []
                m["epoch"] += 1
            toks = [inp.x[row * wl.T + t, 0].copy() for t in range(wl.T)]
            m["live"] += toks[: int(inp.accepted[row])]
        run_oracle_step(c, wl, params, ids, p, inp)
        for row, s in enumerate(ids):
            if s <= 0:
                continue
            m = model[int(s)]
            assert c.ring_start[s] == m["start"] and p[row] == len(m["live"]) and c.flush_epoch[s] == m["epoch"]
            for j, tok in enumerate(m["live"]):
                assert np.array_equal(c.x_view()[s, 0, (m["start"] + j) % wl.L], tok)


def test_varlen_packing_equals_separate_calls(orc):
    wl = W.config("tiny", varlen=True, state_dtype=W.BF16, prefill_live=11)
    gen = W.Generator(wl)
    A, D, dt_bias = gen.params()
    c, ids, p = oracle_cache(orc, wl, gen)
    inp = gen.step(2)
    packed = c.copy()
    pp = p.copy()
    packed.flush(A, ids, pp, wl.T, cu_seqlens=inp.cu_seqlens)
    y_packed = packed.step(inp.x, inp.dt, A, inp.B, inp.C, D, dt_bias, ids, pp, wl.T, cu_seqlens=inp.cu_seqlens)
    sep = c.copy()
    for b in range(ids.size):
        lo, hi = int(inp.cu_seqlens[b]), int(inp.cu_seqlens[b + 1])
        pb = p[b:b + 1].copy()
        sep.flush(A, ids[b:b + 1], pb, hi - lo)
        y = sep.step(inp.x[lo:hi], inp.dt[lo:hi], A, inp.B[lo:hi], inp.C[lo:hi], D, dt_bias, ids[b:b + 1], pb,
                     hi - lo)
        assert np.array_equal(y, y_packed[lo:hi])
        assert pb[0] == pp[b]
    for name in ("state", "x_cache", "B_cache", "dt_cache", "ring_start", "flush_epoch"):
        assert np.array_equal(getattr(sep, name), getattr(packed, name)), name


def test_padded_slot_pages_equal_contiguous(orc):
    wl = W.config("tiny", state_dtype=W.I8, rounding=W.STOCHASTIC, sr_seed=7)
    gen = W.Generator(wl)
    params = gen.params()
    a, ids, pa = oracle_cache(orc, wl, gen, slot_pad_bytes=0)
    b_, _, pb = oracle_cache(orc, wl, gen, slot_pad_bytes=4096)
    for k in range(wl.steps):
        inp = gen.step(k)
        assert np.array_equal(run_oracle_step(a, wl, params, ids, pa, inp),
                              run_oracle_step(b_, wl, params, ids, pb, inp))
    for v in ("state_view", "scale_view", "x_view", "B_view", "dt_view"):
        assert np.array_equal(getattr(a, v)(), getattr(b_, v)()), v


def test_init_ignores_bad_ids_and_clears_rings(orc):
    wl = W.config("tiny", state_dtype=W.E4M3)
    c = orc.OracleCache(wl.num_slots, wl.nheads, wl.ngroups, wl.max_window, wl.npredicted, wl.state_dtype)
    c.x_cache[:] = 7
    c.B_cache[:] = 7
    c.dt_cache[:] = 1.0
    c.ring_start[:] = 3
    c.flush_epoch[:] = 9
    gen = W.Generator(wl)
    states = gen.init_states(0, 4)
    c.init_state(states, np.array([0, 2, -1, 5], np.int32))  # only slot 2 is valid (S = 5)
    assert not c.x_view()[2].any() and not c.B_view()[2].any() and not c.dt_view()[2].any()
    assert c.ring_start[2] == 0 and c.flush_epoch[2] == 0
    for s in (0, 1, 3, 4):
        assert (c.x_view()[s] == 7).all() and c.ring_start[s] == 3 and c.flush_epoch[s] == 9
        assert not c.state_view()[s].any()
    codes, scales = orc.quantize_rows(W.E4M3, W.NEAREST, states[1].reshape(-1, 128), h=0, s=2)
    assert np.array_equal(c.state_view()[2].reshape(-1, 128)[:64], codes[:64])


def test_error_bits_for_bad_rows(orc):
    wl = W.config("tiny", state_dtype=W.BF16)
    gen = W.Generator(wl)
    A, D, dt_bias = gen.params()
    c, ids, p = oracle_cache(orc, wl, gen)
    inp = gen.step(0)
    bad = p.copy()
    row = int(np.nonzero(ids > 0)[0][0])
    bad[row] = wl.L - wl.T + 1  # p + T > L
    before = c.copy()
    y = c.step(inp.x, inp.dt, A, inp.B, inp.C, D, dt_bias, ids, bad, wl.T)
    assert c.error_word[0] & orc.ERR_PNAT
    assert not y[row * wl.T:(row + 1) * wl.T].any()
    s = ids[row]
    assert np.array_equal(c.x_view()[s], before.x_view()[s])
    acc = np.zeros(ids.size, np.int32)
    acc[row] = wl.T + 1
    c.error_word[:] = 0
    c.accept(ids, p, acc, wl.T)
    assert c.error_word[0] & orc.ERR_ACCEPT


def _gate_bits(shape, seed, value=None):
    """bf16 bits of an output gate z: N(0, 1) draws, or a constant."""
    if value is not None:
        return np.full(shape, np.float32(value), np.float32).view(np.uint32).__rshift__(16).astype(np.uint16)
    v = np.random.default_rng(seed).standard_normal(shape).astype(np.float32)
    return (v.view(np.uint32) >> 16).astype(np.uint16)


def test_output_gate_equals_library_silu_on_the_recurrence(orc):
    """y * silu(z): the gated oracle against torch's silu applied to the
    float64 brute-force recurrence, and rounded to bf16 once."""
    import torch

    wl = W.config("tiny", prefill_live=12, ring_start_random=True)
    gen = W.Generator(wl)
    params = gen.params()
    c, ids, pnat = oracle_cache(orc, wl, gen)
    inp = gen.step(0)
    z = _gate_bits((inp.ntok, wl.nheads, 64), 5)
    y_bits, y64 = c.copy().step(inp.x, inp.dt, params[0], inp.B, inp.C, params[1], params[2], ids, pnat, wl.T,
                                want_f64=True, z=z)
    zf = torch.nn.functional.silu(torch.from_numpy(brute.bf16_to_f64(z))).numpy()
    worst = 0.0
    for b, s in enumerate(ids):
        tok0, Tb = _row_tokens(inp, b, wl.T)
        if s <= 0:
            assert not y64[tok0:tok0 + Tb].any()
            continue
        for h in range(wl.nheads):
            ys, _, _ = _bruteforce_row(c, wl, params, int(s), int(pnat[b]), h, inp, tok0, Tb)
            want = ys * zf[tok0:tok0 + Tb, h]
            got = y64[tok0:tok0 + Tb, h]
            worst = max(worst, float(np.abs(got - want).max() / (np.abs(want).max() + 1e-30)))
    assert worst < 2e-5, worst
    assert np.array_equal(y_bits, orc.f32_to_bf16_bits(y64.astype(np.float32)))


def test_output_gate_special_values(orc):
    """z = 0 closes the gate (every output exactly zero); z = 40 makes
    silu(z) = z exactly in double, so the output is z * y rounded once."""
    wl = W.config("tiny", prefill_live=12, ring_start_random=True)
    gen = W.Generator(wl)
    params = gen.params()
    c, ids, pnat = oracle_cache(orc, wl, gen)
    inp = gen.step(0)
    shape = (inp.ntok, wl.nheads, 64)
    args = (inp.x, inp.dt, params[0], inp.B, inp.C, params[1], params[2], ids, pnat, wl.T)
    y0 = c.copy().step(*args, z=_gate_bits(shape, 0, 0.0))
    assert not (y0 & 0x7FFF).any()
    _, y64 = c.copy().step(*args, want_f64=True)
    y40 = c.copy().step(*args, z=_gate_bits(shape, 0, 40.0))
    assert np.array_equal(y40, orc.f32_to_bf16_bits((y64 * 40.0).astype(np.float32)))
