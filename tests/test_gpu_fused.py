"""rssm_flush_step (flush and step in one call) vs the oracle's flush then
step, on the same seeded inputs (needs a GPU).

The one call folds every flushed checkpoint in the flush's canonical fp32
order (for every format), from the stage its readout streams: checkpoints,
8-bit scales, rings, ring_start, pnat, flush epochs and error bits bit for bit
against the oracle.  A flushed row's outputs replay its whole live prefix
from the old checkpoint (the fold's fp32 values before their rounding), where
the oracle reads the rounded new checkpoint: bf16 outputs within atol 2e-2 /
rtol 1e-2.  Rows whose live prefix and new tokens do not fit the ring
together (pnat + T_b > L, which the decode protocol never produces when
max_window >= npredicted) are refused with RSSM_ERRBIT_PNAT.
"""
import numpy as np
import pytest
import torch

from speculative_state_replay_gb300 import api
from speculative_state_replay_gb300 import workloads as W
from tests.gpu_harness import Pair, bf16_f32, dev_of, gpu_cache_from, host_of
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


def run_fused(orc, wl, steps=None, force_every=0, pnat_override=None):
    gen = W.Generator(wl)
    oc, ids, pnat = oracle_cache(orc, wl, gen)
    if pnat_override is not None:
        pnat[:] = pnat_override
    pair = Pair(orc, wl, oc, ids, pnat, fused=True)
    for k in range(wl.steps if steps is None else steps):
        force = 1 if force_every and k % force_every == force_every - 1 else 0
        pair.step(gen.step(k), force=force)
    return pair


@pytest.mark.parametrize("dtype", DTYPES)
def test_fused_tiny_all_dtypes(orc, dtype):
    wl = W.config("tiny", state_dtype=dtype, prefill_live=14, ring_start_random=True)
    pair = run_fused(orc, wl)
    assert pair.oc.flush_epoch.max() >= 1
    assert pair.exact_state_steps == wl.steps


def test_fused_tiny_config_f32_full(orc):
    pair = run_fused(orc, W.config("tiny"))
    assert pair.exact_state_steps == W.config("tiny").steps


@pytest.mark.parametrize("dtype,rounding", [(W.I8, W.NEAREST), (W.I8, W.STOCHASTIC), (W.E4M3, W.NEAREST),
                                            (W.E4M3, W.STOCHASTIC), (W.F16, W.STOCHASTIC),
                                            (W.BF16, W.STOCHASTIC)])
def test_fused_eight_bit_config_reduced(orc, dtype, rounding):
    """Flush every 4 steps; the folded codes, scales and the outputs read from
    the freshly rounded stage must all match."""
    wl = W.config("eight_bit", batch=8, state_dtype=dtype, rounding=rounding, sr_seed=7)
    pair = run_fused(orc, wl)
    assert pair.oc.flush_epoch.max() >= 3
    assert pair.exact_state_steps == wl.steps


def test_fused_mamba2_decode_reduced(orc):
    wl = W.config("mamba2_decode", batch=12, steps=20)
    pair = run_fused(orc, wl)
    assert pair.oc.flush_epoch.max() >= 1
    assert pair.exact_state_steps == wl.steps


def test_fused_large_batch_reduced(orc):
    wl = W.config("large_batch", batch=24, steps=16)
    pair = run_fused(orc, wl)
    assert pair.exact_state_steps == wl.steps


def test_fused_sweep_reduced_varlen_padded(orc):
    wl = W.config("sweep", batch=24, steps=10)
    pair = run_fused(orc, wl)
    assert pair.oc.flush_epoch.max() >= 1


@pytest.mark.parametrize("dtype", DTYPES)
def test_fused_forced_full_window_flush(orc, dtype):
    """Every active row flushes a full window (p = 16 = W) every step."""
    wl = W.config("mamba2_decode", batch=6, state_dtype=dtype, prefill_live=16, ring_start_random=True, steps=3)
    pair = run_fused(orc, wl, force_every=1, pnat_override=16)
    assert pair.exact_state_steps == wl.steps


@pytest.mark.parametrize("T,W_,G", [(1, 16, 8), (8, 24, 8), (3, 3, 128), (8, 8, 1)])
def test_fused_shape_edges(orc, T, W_, G):
    """T = 1; the largest ring (L = 32) with T = 8; one head per group with
    max_window = T (a row flushes about every other step); one group for all
    heads."""
    H = 128 if G == 128 else 16
    wl = W.Workload(name="edge", num_slots=9, nheads=H, ngroups=G, max_window=W_, npredicted=T,
                    state_dtype=W.BF16, batch=6, T=T, steps=6, pad_row=True, ring_start_random=True,
                    config_id=9)
    pair = run_fused(orc, wl)
    assert pair.exact_state_steps == wl.steps


@pytest.mark.parametrize("dtype", [W.BF16, W.I8])
def test_fused_refuses_rows_that_overflow_the_ring(orc, dtype):
    """A row whose live prefix and new tokens do not fit the ring together
    (pnat + T_b > L: the new tokens would land on live slots the fold reads) is
    refused: RSSM_ERRBIT_PNAT, zero outputs, its caches untouched; the other
    rows are computed as usual.  (rssm_flush + rssm_step folds such a row
    first; the decode protocol never produces one when max_window >=
    npredicted.)"""
    wl = W.config("tiny", state_dtype=dtype, prefill_live=14, ring_start_random=True, steps=1)
    gen = W.Generator(wl)
    oc, ids, pnat = oracle_cache(orc, wl, gen)
    rows = np.nonzero(ids > 0)[0]
    bad = rows[0]
    pnat[bad] = wl.L - 1
    gc = gpu_cache_from(oc)
    A, D, dtb = gen.params()
    g = lambda a: dev_of(a, "cuda")  # noqa: E731
    gp = g(pnat)
    inp = gen.step(0)
    out = torch.full((inp.ntok, wl.nheads, 64), 0x3F80, dtype=torch.int16, device="cuda")
    before = {n: getattr(gc, n).clone() for n in ("state", "x_cache", "ring_start", "flush_epoch")}
    sc = api.alloc_scratch(gc, ids.size, wl.T)
    api.rssm_flush_step(gc, g(inp.x), g(inp.dt), g(A), g(inp.B), g(inp.C), g(D), g(dtb), g(ids), gp, wl.T, out, sc)
    torch.cuda.synchronize()
    assert int(gc.error_word.item()) & api.ERRBIT_PNAT
    assert not out[bad * wl.T:(bad + 1) * wl.T].any()
    s = int(ids[bad])
    for n, v in before.items():
        assert torch.equal(getattr(gc, n)[s], v[s]), n
    assert int(gp[bad].item()) == wl.L - 1
    # the other rows match the oracle (the bad row left out on both sides)
    good = np.array([b for b in range(ids.size) if b != bad])
    ps = pnat[good].copy()
    tok = (good[:, None] * wl.T + np.arange(wl.T)[None]).reshape(-1)
    oc.flush(A, ids[good], ps, wl.T)
    yo = oc.step(inp.x[tok], inp.dt[tok], A, inp.B[tok], inp.C[tok], D, dtb, ids[good], ps, wl.T)
    yg = out.cpu().numpy().view(np.uint16)[tok]
    assert np.allclose(bf16_f32(yg), bf16_f32(yo), atol=2e-2, rtol=1e-2)
    assert np.array_equal(gp.cpu().numpy()[good], ps)


def test_fused_batch_beyond_one_cta(orc):
    """640 varlen rows with a padding row, random ring starts and flushes in
    the first steps, through rssm_flush_step."""
    wl = W.Workload(name="edge", num_slots=700, nheads=4, ngroups=2, max_window=16, npredicted=4,
                    state_dtype=W.BF16, batch=640, T=4, steps=6, varlen=True, pad_row=True,
                    ring_start_random=True, prefill_live=14, config_id=9)
    pair = run_fused(orc, wl, force_every=3)
    assert pair.oc.flush_epoch.max() >= 2


def test_fused_matches_two_calls_bit_for_bit():
    """rssm_flush_step and rssm_flush + rssm_step on twin GPU caches: the same
    checkpoint bits, rings and bookkeeping, step after step (outputs within
    the bf16 tolerance: a flushed row's outputs come from the fold's values
    before their rounding)."""
    wl = W.config("eight_bit", batch=16, state_dtype=W.E4M3, rounding=W.STOCHASTIC, sr_seed=11, steps=8)
    gen = W.Generator(wl)
    A, D, dtb = gen.params()
    ids = gen.slot_idx()
    act = ids[ids > 0]
    g = lambda a: dev_of(a, "cuda")  # noqa: E731
    caches = []
    for _ in range(2):
        c = api.RssmCache(wl.num_slots, wl.nheads, wl.ngroups, wl.max_window, wl.npredicted, wl.state_dtype,
                          wl.rounding)
        api.rssm_init_state(c, g(gen.init_states(0, act.size)), g(act.astype(np.int32)), seed=wl.sr_seed)
        caches.append(c)
    two, one = caches
    gA, gD, gb, gids = g(A), g(D), g(dtb), g(ids)
    p2 = torch.zeros(ids.size, dtype=torch.int32, device="cuda")
    p1 = p2.clone()
    s2, s1 = api.alloc_scratch(two, ids.size, wl.T), api.alloc_scratch(one, ids.size, wl.T)
    for k in range(wl.steps):
        inp = gen.step(k)
        x, dt, B, C, acc = g(inp.x), g(inp.dt), g(inp.B), g(inp.C), g(inp.accepted)
        o2 = torch.zeros((inp.ntok, wl.nheads, 64), dtype=torch.int16, device="cuda")
        o1 = o2.clone()
        api.rssm_flush(two, gA, gids, p2, wl.T, s2, seed=wl.sr_seed)
        api.rssm_step(two, x, dt, gA, B, C, gD, gb, gids, p2, wl.T, o2, s2)
        api.rssm_accept(two, gids, p2, acc, wl.T)
        api.rssm_flush_step(one, x, dt, gA, B, C, gD, gb, gids, p1, wl.T, o1, s1, seed=wl.sr_seed)
        api.rssm_accept(one, gids, p1, acc, wl.T)
        torch.cuda.synchronize()
        for name in ("state", "scale", "x_cache", "B_cache", "dt_cache", "ring_start", "flush_epoch", "error_word"):
            assert torch.equal(getattr(one, name), getattr(two, name)), (k, name)
        assert torch.equal(p1, p2), k
        a1, a2 = bf16_f32(o1.cpu().numpy().view(np.uint16)), bf16_f32(o2.cpu().numpy().view(np.uint16))
        assert np.allclose(a1, a2, atol=2e-2, rtol=1e-2), k
    assert int(one.flush_epoch.max().item()) >= 1


def test_fused_full_size_mamba2_decode_sampled_rows(orc):
    """The benchmark's launch configuration (64 rows x 128 heads, bf16)
    through rssm_flush_step; the oracle recomputes a sample of rows."""
    wl = W.config("mamba2_decode")
    gen = W.Generator(wl)
    oc_full, ids, pnat = oracle_cache(orc, wl, gen)
    A, D, dtb = gen.params()
    gc = gpu_cache_from(oc_full)
    g = lambda a: dev_of(a, "cuda")  # noqa: E731
    gA, gD, gb, gids, gp = g(A), g(D), g(dtb), g(ids), g(pnat)
    scratch = api.alloc_scratch(gc, ids.size, wl.T)
    sample = np.array([0, 17, 40, 63])
    p_o = pnat.copy()
    flushed = 0
    for k in range(24):
        inp = gen.step(k)
        out = torch.empty((inp.ntok, wl.nheads, 64), dtype=torch.int16, device="cuda")
        api.rssm_flush_step(gc, g(inp.x), g(inp.dt), gA, g(inp.B), g(inp.C), gD, gb, gids, gp, wl.T, out, scratch)
        api.rssm_accept(gc, gids, gp, g(inp.accepted), wl.T)
        sid = ids[sample]
        ps = p_o[sample].copy()
        e0 = oc_full.flush_epoch[sid].copy()
        tok = (sample[:, None] * wl.T + np.arange(wl.T)[None]).reshape(-1)
        oc_full.flush(A, sid, ps, wl.T)
        flushed += int((oc_full.flush_epoch[sid] != e0).sum())
        yo = oc_full.step(inp.x[tok], inp.dt[tok], A, inp.B[tok], inp.C[tok], D, dtb, sid, ps, wl.T)
        oc_full.accept(sid, ps, inp.accepted[sample], wl.T)
        p_o[sample] = ps
        torch.cuda.synchronize()
        yg = out.cpu().numpy().view(np.uint16)[tok]
        assert np.allclose(bf16_f32(yg), bf16_f32(yo), atol=2e-2, rtol=1e-2), k
        assert np.array_equal(gp.cpu().numpy()[sample], ps)
        gsid = torch.from_numpy(sid.astype(np.int64)).cuda()
        for name in ("state", "x_cache", "B_cache", "dt_cache", "ring_start", "flush_epoch"):
            o = getattr(oc_full, name)[sid]
            assert np.array_equal(host_of(getattr(gc, name)[gsid], o), o), (k, name)
    assert flushed >= 4
    assert int(gc.error_word.item()) == 0
