"""rssm_accept_flush: the previous step's acceptance and this step's flush
in one launch (needs a GPU).

* Against the library's own two calls: a cache driven by rssm_flush ->
  rssm_step -> rssm_accept and one driven by rssm_accept_flush (the previous
  step's accepted counts and sequence bounds) -> rssm_step hold the same bits
  after every step -- outputs, checkpoints, 8-bit scales, rings, ring starts,
  flush epochs -- and the same pnat and error bits once the last acceptance
  is applied, through forced flushes and acceptances that fail their checks.
* Against the oracle's flush, step and accept (FlashInfer PR #3975, commit
  notes: the write decision prev_k + T > max_window per slot; vLLM PR #65660,
  Details: only accepted tokens enter the checkpoint), through the parity
  harness with the acceptance deferred to the next call.
"""
import numpy as np
import pytest
import torch

from speculative_state_replay_gb300 import api
from speculative_state_replay_gb300 import workloads as W
from tests.gpu_harness import Pair, dev_of, gpu_cache_from
from tests.harness import oracle_cache

pytestmark = pytest.mark.gpu

ARRAYS = ("state", "scale", "x_cache", "B_cache", "dt_cache", "ring_start", "flush_epoch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_state_replay_gb300 import _lib, build

    build.build()
    _lib.load()


@pytest.mark.parametrize("cfg,over", [
    ("mamba2_decode", dict(batch=16, prefill_live=14, ring_start_random=True)),  # bf16, tensor-core folds
    ("sweep", dict(batch=24)),                                                   # varlen, padded pages
    ("eight_bit", dict(batch=8, state_dtype=W.E4M3, rounding=W.STOCHASTIC, sr_seed=7)),
    ("tiny", dict(prefill_live=14, ring_start_random=True)),                    # f32
    ("large_batch", dict(batch=8, prefill_live=14)),                           # fp16, T = 7
])
def test_accept_flush_is_accept_then_flush(orc, cfg, over):
    wl = W.config(cfg, steps=12, **over)
    gen = W.Generator(wl)
    A, D, dtb = gen.params()
    oc, ids, pnat = oracle_cache(orc, wl, gen)
    g = lambda a: None if a is None else dev_of(a, "cuda")  # noqa: E731
    ca, cb = gpu_cache_from(oc), gpu_cache_from(oc)
    gA, gD, gdtb, gids = g(A), g(D), g(dtb), g(ids)
    pa, pb = g(pnat), g(pnat)
    sa, sb = api.alloc_scratch(ca, ids.size, wl.T), api.alloc_scratch(cb, ids.size, wl.T)
    prev = None
    active = np.nonzero(ids > 0)[0]
    for k in range(wl.steps):
        inp = gen.step(k)
        acc = inp.accepted.copy()
        if k == 5:  # acceptances that fail rssm_accept's checks: the rows keep their pnat
            acc[active[0]] = wl.T + 3
            acc[active[-1]] = -1
        force = 1 if k == 7 else 0
        cu = g(inp.cu_seqlens)
        x, dt, B, C = g(inp.x), g(inp.dt), g(inp.B), g(inp.C)
        outs = []
        for cache, pn, sc, fused in ((ca, pa, sa, False), (cb, pb, sb, True)):
            if fused and prev is not None:
                api.rssm_accept_flush(cache, gA, gids, pn, prev[0], wl.T, wl.T, sc, accept_cu_seqlens=prev[1],
                                      cu_seqlens=cu, force=force, seed=wl.sr_seed)
            else:
                api.rssm_flush(cache, gA, gids, pn, wl.T, sc, cu_seqlens=cu, force=force, seed=wl.sr_seed)
            out = torch.full((max(inp.ntok, 1), wl.nheads, 64), 0x7FC0, dtype=torch.int16, device="cuda")
            api.rssm_step(cache, x, dt, gA, B, C, gD, gdtb, gids, pn, wl.T, out, sc, cu_seqlens=cu)
            outs.append(out)
        api.rssm_accept(ca, gids, pa, g(acc), wl.T, cu_seqlens=cu)
        prev = (g(acc), cu)
        torch.cuda.synchronize()
        assert torch.equal(outs[0], outs[1]), k
        for name in ARRAYS:
            assert torch.equal(getattr(ca, name), getattr(cb, name)), (k, name)
    api.rssm_accept(cb, gids, pb, prev[0], wl.T, cu_seqlens=prev[1])
    torch.cuda.synchronize()
    assert torch.equal(pa, pb)
    assert torch.equal(ca.error_word, cb.error_word)
    assert int(ca.error_word.cpu()[0]) != 0  # the failed acceptances were seen
    assert int(ca.flush_epoch.max()) >= 2


@pytest.mark.parametrize("cfg,over", [
    ("mamba2_decode", dict(batch=16, prefill_live=14, ring_start_random=True)),
    ("sweep", dict(batch=16)),
    ("eight_bit", dict(batch=8)),
])
def test_accept_flush_against_oracle(orc, cfg, over):
    wl = W.config(cfg, steps=10, **over)
    gen = W.Generator(wl)
    oc, ids, pnat = oracle_cache(orc, wl, gen)
    pair = Pair(orc, wl, oc, ids, pnat, accept_flush=True)
    for k in range(wl.steps):
        pair.step(gen.step(k), force=1 if k == 6 else 0)
    assert pair.oc.flush_epoch.max() >= 2
