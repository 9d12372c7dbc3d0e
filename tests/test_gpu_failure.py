"""Failure detection on the GPU without a fault (needs a GPU).

Every wait in the pipeline kernels is bounded: a wait that runs out sets
RSSM_ERRBIT_TIMEOUT and the kernel returns.  rssm_selftest_wait_timeout makes
one such wait run out -- an mbarrier told to expect bytes no copy brings --
with a short limit; the call returns, the bit is set, and the same process
then runs decode steps that match the oracle.
"""
import time

import numpy as np
import pytest
import torch

from speculative_state_replay_gb300 import api
from speculative_state_replay_gb300 import workloads as W
from tests.gpu_harness import Pair
from tests.harness import oracle_cache

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_state_replay_gb300 import _lib, build

    build.build()
    _lib.load()


def test_bounded_wait_runs_out_and_the_context_stays_usable(orc):
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    api.rssm_selftest_wait_timeout(err, wait_ms=30)
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 < 20.0
    assert int(err.item()) & api.ERRBIT_TIMEOUT
    # a second time on the same word: still bounded, the bit stays (sticky)
    api.rssm_selftest_wait_timeout(err, wait_ms=5)
    torch.cuda.synchronize()
    assert int(err.item()) == api.ERRBIT_TIMEOUT
    # the context is intact: decode steps on a fresh cache match the oracle
    wl = W.config("tiny", state_dtype=W.E4M3, rounding=W.STOCHASTIC, sr_seed=3, steps=6, prefill_live=14)
    gen = W.Generator(wl)
    oc, ids, pnat = oracle_cache(orc, wl, gen)
    pair = Pair(orc, wl, oc, ids, pnat)
    for k in range(wl.steps):
        pair.step(gen.step(k))
    assert pair.exact_state_steps == wl.steps
    assert int(pair.gc.error_word.item()) == 0
    assert np.all(pair.oc.error_word == 0)
