"""Separate read checkpoints on the GPU vs the oracle (needs a GPU).

vLLM PR #65660 (Overview) keeps an FP16 recurrence checkpoint with stochastic
rounding, does the flush work in FP32 and re-encodes an FP8 read checkpoint
that the readout streams; its Claims: read checkpoints use nearest encoding.
Here: the recurrence state and the 8-bit read copy (codes + FP32 row scales)
are both rounded from the same fp32 values at init and at every flush; the
step reads S0 from the read copy.  Bar: read codes and scales bit for bit,
the recurrence checkpoint bit for bit (every fold with a read copy takes the
canonical fp32 order), outputs at the bf16 tolerance, rings and bookkeeping
bit for bit.
"""
import numpy as np
import pytest
import torch

from speculative_state_replay_gb300 import api
from speculative_state_replay_gb300 import workloads as W
from tests.gpu_harness import Pair, dev_of, host_of
from tests.harness import oracle_cache

pytestmark = pytest.mark.gpu

PAIRS = [(W.F16, W.STOCHASTIC, W.E4M3), (W.F16, W.STOCHASTIC, W.I8), (W.BF16, W.NEAREST, W.E4M3),
         (W.F32, W.NEAREST, W.I8), (W.BF16, W.STOCHASTIC, W.E4M3), (W.F16, W.STOCHASTIC, W.NVFP4),
         (W.F32, W.NEAREST, W.NVFP4), (W.BF16, W.NEAREST, W.NVFP4)]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_state_replay_gb300 import _lib, build

    build.build()
    _lib.load()


@pytest.mark.parametrize("dtype,rounding,read", PAIRS)
def test_init_writes_both_checkpoints_bit_exact(orc, dtype, rounding, read):
    wl = W.config("tiny", state_dtype=dtype, rounding=rounding, sr_seed=7, read_dtype=read)
    gen = W.Generator(wl)
    states = gen.init_states(0, 4)
    states[0, 0, 3] = 0.0     # an all-zero row (scale 1)
    states[1, 2, 5, 7] = 1e4  # a row with a large outlier
    ids = np.array([3, 0, 1, 4], np.int32)
    oc = orc.OracleCache(wl.num_slots, wl.nheads, wl.ngroups, wl.max_window, wl.npredicted, dtype, rounding,
                         read_dtype=read)
    oc.init_state(states, ids, seed=wl.sr_seed)
    gc = api.RssmCache(wl.num_slots, wl.nheads, wl.ngroups, wl.max_window, wl.npredicted, dtype, rounding,
                       read_dtype=read)
    api.rssm_init_state(gc, dev_of(states, "cuda"), dev_of(ids, "cuda"), seed=wl.sr_seed)
    torch.cuda.synchronize()
    from tests.gpu_harness import cache_arrays

    for name in cache_arrays(oc):
        if name == "error_word":
            continue
        o = getattr(oc, name)
        assert np.array_equal(host_of(getattr(gc, name), o), o), name


@pytest.mark.parametrize("dtype,rounding,read", PAIRS)
def test_decode_steps_with_a_read_checkpoint(orc, dtype, rounding, read):
    """Mamba-2 decode reduced, prefilled rings (folds of up to 16 tokens from
    the first step), random ring starts, a forced flush every fifth step."""
    wl = W.config("mamba2_decode", batch=12, steps=15, state_dtype=dtype, rounding=rounding, sr_seed=7,
                  read_dtype=read, prefill_live=14, ring_start_random=True)
    gen = W.Generator(wl)
    oc, ids, pnat = oracle_cache(orc, wl, gen)
    pair = Pair(orc, wl, oc, ids, pnat)
    for k in range(wl.steps):
        pair.step(gen.step(k), force=1 if k % 5 == 4 else 0)
    assert pair.oc.flush_epoch.max() >= 3
    assert pair.exact_state_steps == wl.steps


@pytest.mark.parametrize("read", [W.E4M3, W.I8, W.NVFP4])
def test_separate_sweep_without_resync(orc, read):
    """The separate-checkpoint benchmark workload reduced (varlen rows, padded
    slot pages, fp16 recurrence with stochastic rounding), 16 steps with each
    side carrying its own caches."""
    wl = W.config("separate", batch=20, steps=16, read_dtype=read)
    gen = W.Generator(wl)
    oc, ids, pnat = oracle_cache(orc, wl, gen)
    pair = Pair(orc, wl, oc, ids, pnat, resync=False)
    for k in range(wl.steps):
        pair.step(gen.step(k))
    assert pair.oc.flush_epoch.max() >= 2
    assert pair.exact_state_steps == wl.steps


def test_read_checkpoint_is_what_the_step_reads(orc):
    """Scribbling over the recurrence state between a flush and a step leaves
    the step's outputs unchanged (the readout reads the read copy); scribbling
    over the read copy changes them."""
    wl = W.config("mamba2_decode", batch=6, steps=1, state_dtype=W.F16, rounding=W.STOCHASTIC, sr_seed=7,
                  read_dtype=W.E4M3)
    gen = W.Generator(wl)
    A, D, dtb = gen.params()
    oc, ids, pnat = oracle_cache(orc, wl, gen)
    from tests.gpu_harness import gpu_cache_from

    inp = gen.step(0)
    g = lambda a: dev_of(a, "cuda")  # noqa: E731
    outs = []
    for scribble in (None, "state", "read_state"):
        gc = gpu_cache_from(oc)
        if scribble:
            getattr(gc, scribble).view(torch.uint8).fill_(0x3A)
        out = torch.zeros((inp.ntok, wl.nheads, 64), dtype=torch.int16, device="cuda")
        sc = api.alloc_scratch(gc, ids.size, wl.T)
        api.rssm_step(gc, g(inp.x), g(inp.dt), g(A), g(inp.B), g(inp.C), g(D), g(dtb), g(ids), g(pnat), wl.T, out,
                      sc)
        torch.cuda.synchronize()
        outs.append(out.cpu())
    assert torch.equal(outs[0], outs[1])
    assert not torch.equal(outs[0], outs[2])


def test_one_call_path_refuses_a_read_checkpoint():
    wl = W.config("tiny", state_dtype=W.F16, read_dtype=W.E4M3)
    gc = api.RssmCache(wl.num_slots, wl.nheads, wl.ngroups, wl.max_window, wl.npredicted, wl.state_dtype,
                       read_dtype=W.E4M3)
    z = torch.zeros(4096, dtype=torch.int32, device="cuda")
    with pytest.raises(api.RssmError) as e:
        api.rssm_flush_step(gc, z, z, z, z, z, z, z, z[:1], z[:1], 1, z, torch.zeros(1 << 20, dtype=torch.uint8,
                                                                                       device="cuda"))
    assert e.value.status == 2
