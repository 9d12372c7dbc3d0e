"""The 2-byte checkpoint bar of the GPU parity tests can fail (CPU only).

The GPU tests accept a bf16/f16 checkpoint code within one unit in the last
place of the oracle's (2^-20 absolute near zero).  Mistakes are planted here
in the oracle's inputs, on the CPU: a fold that dropped one live token, or
weighted it wrongly, must be rejected; a checkpoint off by one unit in the
last place everywhere must pass, and one off by two must not.
"""
import numpy as np
import pytest

from speculative_state_replay_gb300 import workloads as W
from tests.gpu_harness import code_distance, half_state_close, state_close
from tests.harness import oracle_cache


def _flushed_pair(orc, dtype, mutate, token=13):
    """(reference checkpoint, checkpoint after a fold of 14 live tokens whose
    inputs `mutate` changed at live token `token`)."""
    wl = W.config("mamba2_decode", batch=6, state_dtype=dtype, prefill_live=16, ring_start_random=True)
    gen = W.Generator(wl)
    oc, ids, pnat = oracle_cache(orc, wl, gen)
    A, _, _ = gen.params()
    pnat[ids > 0] = 14
    ref, bad = oc.copy(), oc.copy()
    for b, s in enumerate(ids):
        if s > 0:
            pos = (int(oc.ring_start[s]) + token) % wl.L
            mutate(bad, s, pos)
    ref.flush(A, ids, pnat.copy(), wl.T, force=1)
    bad.flush(A, ids, pnat.copy(), wl.T, force=1)
    active = ids[ids > 0]
    return ref.state[active], bad.state[active]


def _drop(c, s, pos):
    c.x_view()[s][:, pos] = 0  # the token's contribution u_j = w_j x_j vanishes


def _misweight(c, s, pos):
    x = (c.x_view()[s][:, pos].astype(np.uint32) << 16).view(np.float32) * np.float32(1.25)
    c.x_view()[s][:, pos] = (x.view(np.uint32) >> 16).astype(np.uint16)


@pytest.mark.parametrize("dtype", [W.BF16, W.F16])
@pytest.mark.parametrize("mutate", [_drop, _misweight])
@pytest.mark.parametrize("token", [13, 5, 0])
def test_bar_rejects_a_wrong_token_in_the_fold(orc, dtype, mutate, token):
    """The newest live token (13) enters with weight dt', older ones decayed by
    e^{c_end - c_j}: a wrong newest token moves most elements past the bar; a
    wrong older one still moves some (tokens whose decayed weight is below one
    unit in the last place are invisible at the checkpoint's precision, to the
    oracle's own rounding as much as to the bar)."""
    ref, bad = _flushed_pair(orc, dtype, mutate, token)
    assert state_close(dtype, ref, ref)
    assert not state_close(dtype, bad, ref)
    far = (code_distance(bad.view(np.uint16), ref.view(np.uint16)) > 1).mean()
    if token == 13:
        assert far > 0.3, far
        # the newest token also fails the bar for checkpoints carried through
        # several folds (two units of each row's largest magnitude)
        assert not state_close(dtype, bad, ref, carried=True)
        assert state_close(dtype, ref, ref, carried=True)


@pytest.mark.parametrize("dtype", [W.BF16, W.F16])
def test_bar_admits_one_unit_in_the_last_place(orc, dtype):
    ref, _ = _flushed_pair(orc, dtype, lambda c, s, pos: None)
    bits = ref.view(np.uint16)
    mag = bits & 0x7FFF
    finite = mag < (0x7F7F if dtype == W.BF16 else 0x7BFF) - 2
    up1 = np.where(finite, bits + 1, bits).astype(np.uint16)   # one unit away from zero
    up2 = np.where(finite, bits + 2, bits).astype(np.uint16)
    assert half_state_close(dtype, up1, bits)
    assert not half_state_close(dtype, up2, bits)
    assert state_close(dtype, up1, bits, carried=True)  # one unit of a value <= two of its row maximum
    # the near-zero slack: +0 against the smallest codes of either sign
    tiny = np.array([0x0001, 0x8003, 0x0000], np.uint16)
    assert half_state_close(dtype, tiny, np.zeros(3, np.uint16))
