"""CUDA library vs CPU oracle on the same seeded inputs (needs a GPU).

Bar: bf16 outputs within atol 2e-2 / rtol 1e-2; f32 checkpoints within 1e-4
relative; 2-byte checkpoints within one unit in the last place of the
oracle's codes (2^-20 absolute near zero); 8-bit codes and scales, rings,
ring_start, pnat, flush epochs and error bits bit-exact.
"""
import numpy as np
import pytest
import torch

from speculative_state_replay_gb300 import api
from speculative_state_replay_gb300 import workloads as W
from tests.gpu_harness import Pair, bf16_f32, dev_of, host_of, state_close
from tests.harness import oracle_cache

pytestmark = pytest.mark.gpu

DTYPES = [W.F32, W.BF16, W.F16, W.I8, W.E4M3]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_state_replay_gb300 import _lib, build

    build.build()
    _lib.load()


def run_pair(orc, wl, steps=None, force_every=0, oracle_ids=None):
    gen = W.Generator(wl)
    oc, ids, pnat = oracle_cache(orc, wl, gen)
    pair = Pair(orc, wl, oc, ids, pnat)
    for k in range(wl.steps if steps is None else steps):
        force = 1 if force_every and k % force_every == force_every - 1 else 0
        pair.step(gen.step(k), force=force)
    return pair


def test_spec_math_bit_exact(orc):
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.uniform(-90, 90, 1 << 22), rng.normal(-2.0, 0.5, 1 << 22),
                        np.linspace(-30, 25, 1 << 20), np.float32([0.0, -0.0, 20.0, 20.000002, -87.0, 88.0])])
    x = x.astype(np.float32)
    gx = dev_of(x, "cuda")
    ge, gs = torch.empty_like(gx), torch.empty_like(gx)
    api.rssm_eval_spec_math(gx, ge, gs)
    torch.cuda.synchronize()
    assert np.array_equal(ge.cpu().numpy().view(np.uint32), orc.spec_exp(x).view(np.uint32))
    assert np.array_equal(gs.cpu().numpy().view(np.uint32), orc.spec_softplus(x).view(np.uint32))


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("rounding", [W.NEAREST, W.STOCHASTIC])
def test_init_state_bit_exact(orc, dtype, rounding):
    wl = W.config("tiny", state_dtype=dtype, rounding=rounding, sr_seed=7)
    gen = W.Generator(wl)
    states = gen.init_states(0, 4)
    states[0, 0, 3] = 0.0  # an all-zero row
    states[1, 2, 5, 7] = 1e4  # a row with a large outlier
    ids = np.array([3, 0, 1, 4], np.int32)  # slot 0 is ignored
    oc = orc.OracleCache(wl.num_slots, wl.nheads, wl.ngroups, wl.max_window, wl.npredicted, dtype, rounding)
    oc.x_cache[:] = 5
    oc.ring_start[:] = 2
    oc.init_state(states, ids, seed=wl.sr_seed)
    gc = api.RssmCache(wl.num_slots, wl.nheads, wl.ngroups, wl.max_window, wl.npredicted, dtype, rounding)
    gc.x_cache.fill_(5)
    gc.ring_start.fill_(2)
    api.rssm_init_state(gc, dev_of(states, "cuda"), dev_of(ids, "cuda"), seed=wl.sr_seed)
    torch.cuda.synchronize()
    for name in ("state", "scale", "x_cache", "ring_start", "flush_epoch"):
        o = getattr(oc, name)
        assert np.array_equal(host_of(getattr(gc, name), o), o), name


@pytest.mark.parametrize("dtype", DTYPES)
def test_tiny_all_dtypes(orc, dtype):
    wl = W.config("tiny", state_dtype=dtype, prefill_live=14, ring_start_random=True)
    pair = run_pair(orc, wl)
    assert pair.oc.flush_epoch.max() >= 1


def test_tiny_config_f32_full(orc):
    """The Tiny configuration exactly as specified: f32 state, 12 steps."""
    pair = run_pair(orc, W.config("tiny"))
    assert pair.exact_state_steps == W.config("tiny").steps


@pytest.mark.parametrize("dtype,rounding", [(W.I8, W.NEAREST), (W.I8, W.STOCHASTIC), (W.E4M3, W.NEAREST),
                                            (W.E4M3, W.STOCHASTIC), (W.F16, W.STOCHASTIC),
                                            (W.BF16, W.STOCHASTIC)])
def test_eight_bit_config_reduced(orc, dtype, rounding):
    """8-bit checkpoint configuration (accept all -> flush every 4 steps), 8 rows."""
    wl = W.config("eight_bit", batch=8, state_dtype=dtype, rounding=rounding, sr_seed=7)
    pair = run_pair(orc, wl)
    assert pair.oc.flush_epoch.max() >= 3
    assert pair.exact_state_steps == wl.steps


@pytest.mark.parametrize("dtype", [W.I8, W.E4M3])
def test_eight_bit_odd_heads_per_group(orc, dtype):
    """8-bit states with 3 heads per group: the readout takes one head per unit
    (with an even count it takes two)."""
    wl = W.Workload(name="edge", num_slots=9, nheads=12, ngroups=4, max_window=16, npredicted=4, state_dtype=dtype,
                    rounding=W.STOCHASTIC, sr_seed=5, batch=6, T=4, steps=10, pad_row=True, ring_start_random=True,
                    prefill_live=10, accept="all", config_id=9)
    pair = run_pair(orc, wl)
    assert pair.oc.flush_epoch.max() >= 1
    assert pair.exact_state_steps == wl.steps


def test_mamba2_decode_reduced(orc):
    wl = W.config("mamba2_decode", batch=12, steps=20)
    pair = run_pair(orc, wl)
    assert pair.oc.flush_epoch.max() >= 1


def test_large_batch_reduced(orc):
    """fp16 state, T = 7 drafts (L = 23), random ring starts: wraparound."""
    wl = W.config("large_batch", batch=24, steps=16)
    run_pair(orc, wl)


def test_sweep_reduced_varlen_padded(orc):
    """varlen 1..5 tokens, padded slot pages, prefilled rings, mixed pnat."""
    wl = W.config("sweep", batch=24, steps=10)
    pair = run_pair(orc, wl)
    assert pair.oc.flush_epoch.max() >= 1


@pytest.mark.parametrize("dtype", DTYPES)
def test_forced_full_window_flush(orc, dtype):
    """Every active row flushes with a full window (p = 16)."""
    wl = W.config("mamba2_decode", batch=6, state_dtype=dtype, prefill_live=16, ring_start_random=True, steps=3)
    gen = W.Generator(wl)
    oc, ids, pnat = oracle_cache(orc, wl, gen)
    pnat[:] = 16
    pair = Pair(orc, wl, oc, ids, pnat)
    for k in range(wl.steps):
        pair.step(gen.step(k), force=1)


@pytest.mark.parametrize("T,W_,G", [(1, 16, 8), (8, 24, 8), (3, 0, 128), (8, 0, 1)])
def test_shape_edges(orc, T, W_, G):
    """T = 1; the largest ring (L = 32) with T = 8; one head per group;
    max_window 0 (flush every step); one group for all heads."""
    H = 128 if G == 128 else 16
    wl = W.Workload(name="edge", num_slots=9, nheads=H, ngroups=G, max_window=W_, npredicted=T,
                    state_dtype=W.BF16, batch=6, T=T, steps=6, pad_row=True, ring_start_random=True,
                    config_id=9)
    run_pair(orc, wl)


def test_batch_beyond_one_classification_pass(orc):
    """640 rows (more than one CTA's threads, so the flush classifies the rows
    in several passes of 288 and carries the compacted positions across them),
    varlen rows, a padding row, random ring starts, live prefixes that flush in
    the first steps, and a forced flush every third step."""
    wl = W.Workload(name="edge", num_slots=700, nheads=4, ngroups=2, max_window=16, npredicted=4,
                    state_dtype=W.BF16, batch=640, T=4, steps=6, varlen=True, pad_row=True,
                    ring_start_random=True, prefill_live=14, config_id=9)
    pair = run_pair(orc, wl, force_every=3)
    assert pair.oc.flush_epoch.max() >= 2
    assert int(pair.oc.error_word[0]) == 0


@pytest.mark.parametrize("dtype", [W.F32, W.BF16, W.F16, W.I8, W.E4M3])
def test_output_gate_tiny_all_dtypes(orc, dtype):
    """rssm_step_gated: y * silu(z) against the oracle's gated step (every
    state format; 8-bit units of one head at hpg = 8 / G = 1)."""
    wl = W.config("tiny", state_dtype=dtype, prefill_live=14, ring_start_random=True)
    gen = W.Generator(wl)
    oc, ids, pnat = oracle_cache(orc, wl, gen)
    pair = Pair(orc, wl, oc, ids, pnat, gate=True)
    for k in range(wl.steps):
        pair.step(gen.step(k))
    assert pair.oc.flush_epoch.max() >= 1


@pytest.mark.parametrize("cfg,over", [("mamba2_decode", dict(batch=12, steps=10)),
                                      ("eight_bit", dict(batch=8, steps=8)),
                                      ("sweep", dict(batch=24, steps=6))])
def test_output_gate_reduced_configs(orc, cfg, over):
    """The gate on the readout's other unit shapes: two-head 8-bit units,
    varlen rows with padded slot pages."""
    wl = W.config(cfg, **over)
    gen = W.Generator(wl)
    oc, ids, pnat = oracle_cache(orc, wl, gen)
    pair = Pair(orc, wl, oc, ids, pnat, gate=True)
    for k in range(wl.steps):
        pair.step(gen.step(k))


def test_output_gate_closed_and_halves():
    """z = 0 gives zeros for every output; precompute + gated readout equals
    the gated step bit for bit; z = NULL equals the ungated step."""
    wl = W.config("mamba2_decode", batch=8, steps=1)
    gen = W.Generator(wl)
    A, D, dtb = gen.params()
    ids = gen.slot_idx()
    act = ids[ids > 0]
    g = lambda a: dev_of(a, "cuda")  # noqa: E731
    outs = []
    for mode in ("zero", "gated", "halves", "plain", "none"):
        c = api.RssmCache(wl.num_slots, wl.nheads, wl.ngroups, wl.max_window, wl.npredicted, wl.state_dtype)
        api.rssm_init_state(c, g(gen.init_states(0, act.size)), g(act.astype(np.int32)))
        pn = torch.zeros(ids.size, dtype=torch.int32, device="cuda")
        sc = api.alloc_scratch(c, ids.size, wl.T)
        inp = gen.step(0)
        out = torch.zeros((inp.ntok, wl.nheads, 64), dtype=torch.int16, device="cuda")
        zf = np.random.default_rng(3).standard_normal((inp.ntok, wl.nheads, 64)).astype(np.float32)
        z = torch.zeros_like(out) if mode == "zero" else g((zf.view(np.uint32) >> 16).astype(np.uint16))
        args = (c, g(inp.x), g(inp.dt), g(A), g(inp.B), g(inp.C), g(D), g(dtb), g(ids), pn, wl.T, out, sc)
        if mode == "halves":
            api.rssm_step_precompute(*args)
            api.rssm_step_readout(*args, z=z)
        elif mode == "plain":
            api.rssm_step(*args)
        elif mode == "none":
            api.rssm_step(*args, z=None)
        else:
            api.rssm_step(*args, z=z)
        torch.cuda.synchronize()
        outs.append(out.cpu().numpy().view(np.uint16))
    zero, gated, halves, plain, none = outs
    assert not (zero & 0x7FFF).any()
    assert np.array_equal(gated, halves)
    assert np.array_equal(plain, none)
    assert not np.array_equal(gated, plain)


def test_bad_rows_set_error_bits_and_zero_outputs(orc):
    wl = W.config("tiny", state_dtype=W.BF16)
    gen = W.Generator(wl)
    oc, ids, pnat = oracle_cache(orc, wl, gen)
    rows = np.nonzero(ids > 0)[0]
    pnat[rows[0]] = wl.L - 1  # p + T > L after no flush (force = 0 flushes it: p + T > W)
    pair = Pair(orc, wl, oc, ids, pnat)
    inp = gen.step(0)
    inp.accepted[rows[1]] = wl.T + 3  # bad accept count
    pair.step(inp)
    assert pair.oc.error_word[0] & api.ERRBIT_ACCEPT
    # a step without the flush on an overfull row: y = 0, error bit, no cache change
    p2 = pair.pnat.copy()
    p2[rows[2]] = wl.L
    gp = dev_of(p2, "cuda")
    out = torch.full((inp.ntok, wl.nheads, 64), 0x3F80, dtype=torch.int16, device="cuda")
    before = pair.gc.x_cache.clone()
    api.rssm_step(pair.gc, dev_of(inp.x, "cuda"), dev_of(inp.dt, "cuda"), pair.gA, dev_of(inp.B, "cuda"),
                  dev_of(inp.C, "cuda"), pair.gD, pair.gb, pair.gids, gp, wl.T, out, pair.scratch)
    torch.cuda.synchronize()
    r = rows[2]
    assert not out[r * wl.T:(r + 1) * wl.T].any()
    assert int(pair.gc.error_word.item()) & api.ERRBIT_PNAT
    s = int(ids[r])
    assert torch.equal(pair.gc.x_cache[s], before[s])


def test_empty_batch_is_noop():
    wl = W.config("tiny")
    gc = api.RssmCache(wl.num_slots, wl.nheads, wl.ngroups, wl.max_window, wl.npredicted, wl.state_dtype)
    z = torch.zeros(0, dtype=torch.int32, device="cuda")
    f = torch.zeros(wl.nheads, dtype=torch.float32, device="cuda")
    scratch = torch.zeros(256, dtype=torch.uint8, device="cuda")
    api.rssm_flush(gc, f, z, z, wl.T, scratch)
    e = torch.zeros(16, dtype=torch.int16, device="cuda")
    api.rssm_step(gc, e, f, f, e, e, f, f, z, z, wl.T, e, scratch)
    api.rssm_accept(gc, z, z, z, wl.T)
    torch.cuda.synchronize()
    assert int(gc.error_word.item()) == 0


@pytest.mark.parametrize("cfg,sample,steps", [
    ("mamba2_decode", [0, 17, 40, 63], 24),
    ("large_batch", [0, 1, 130, 255, 256, 401, 511], 12),
    ("sweep", [0, 1, 255, 256, 600, 777, 1022, 1023], 8),
])
def test_full_size_sampled_rows(orc, cfg, sample, steps):
    """The benchmark's launch configurations on the GPU at full size (Mamba-2
    decode 64 x 128 bf16; 512 x 64 fp16 at T = 7 with ring wraparound; the
    1024-row varlen sweep with padded slot pages and prefilled rings), cache
    initialised as bench.py does; the oracle follows a sample of rows one by
    one (rows are independent).  Outputs, checkpoints (the 2-byte bar),
    rings and bookkeeping of the sampled rows every step."""
    from tests.gpu_harness import init_gpu_cache_like_bench, oracle_cache_for_rows, token_rows

    wl = W.config(cfg)
    gen = W.Generator(wl)
    A, D, dtb = gen.params()
    ids = gen.slot_idx()
    sample = np.array(sample)
    gc, pnat0 = init_gpu_cache_like_bench(wl, gen, ids)
    oc = oracle_cache_for_rows(orc, wl, gen, ids, sample)
    g = lambda a: dev_of(a, "cuda")  # noqa: E731
    gA, gD, gb, gids, gp = g(A), g(D), g(dtb), g(ids), g(pnat0)
    scratch = api.alloc_scratch(gc, ids.size, wl.T)
    p_o = pnat0.copy()
    sid = ids[sample]
    gsid = torch.from_numpy(sid.astype(np.int64)).cuda()
    flushes = 0
    for k in range(steps):
        inp = gen.step(k)
        cu = None if inp.cu_seqlens is None else g(inp.cu_seqlens)
        out = torch.empty((inp.ntok, wl.nheads, 64), dtype=torch.int16, device="cuda")
        api.rssm_flush(gc, gA, gids, gp, wl.T, scratch, cu_seqlens=cu, seed=wl.sr_seed)
        api.rssm_step(gc, g(inp.x), g(inp.dt), gA, g(inp.B), g(inp.C), gD, gb, gids, gp, wl.T, out, scratch,
                      cu_seqlens=cu)
        api.rssm_accept(gc, gids, gp, g(inp.accepted), wl.T, cu_seqlens=cu)
        # oracle on the sampled rows only
        tok, sub_cu = token_rows(inp, sample, wl.T)
        ps = p_o[sample].copy()
        ep = oc.flush_epoch[sid].copy()
        oc.flush(A, sid, ps, wl.T, cu_seqlens=sub_cu, seed=wl.sr_seed)
        flushes += int((oc.flush_epoch[sid] != ep).sum())
        yo = oc.step(inp.x[tok], inp.dt[tok], A, inp.B[tok], inp.C[tok], D, dtb, sid, ps, wl.T, cu_seqlens=sub_cu)
        oc.accept(sid, ps, inp.accepted[sample], wl.T, cu_seqlens=sub_cu)
        p_o[sample] = ps
        torch.cuda.synchronize()
        yg = out.cpu().numpy().view(np.uint16)[tok]
        assert np.allclose(bf16_f32(yg), bf16_f32(yo), atol=2e-2, rtol=1e-2), k
        assert np.array_equal(gp.cpu().numpy()[sample], ps), k
        o = oc.state[sid]
        assert state_close(wl.state_dtype, host_of(gc.state[gsid], o), o, carried=True), (k, "state")
        for name in ("x_cache", "B_cache", "dt_cache", "ring_start", "flush_epoch"):
            o = getattr(oc, name)[sid]
            assert np.array_equal(host_of(getattr(gc, name)[gsid], o), o), (k, name)
    assert flushes >= 2
    assert int(gc.error_word.item()) == 0
