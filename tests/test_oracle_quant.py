"""Pins for the oracle's checkpoint quantiser (CPU only).

Per-row FP32 scales (vLLM PR #65660 commit notes; one row = 128 dstate values
of one (slot, head, d)), nearest encoding for read checkpoints (same PR,
Claims) and Philox-driven stochastic rounding (FlashInfer PR #3975 commit
notes).  Checked against the format definitions, exact ties, saturation,
error bounds and the unbiasedness of stochastic rounding.
"""
import numpy as np
import pytest

from speculative_state_replay_gb300 import workloads as W


def test_int8_nearest_ties_to_even_and_scale():
    import oracle as orc

    row = np.zeros(128, np.float32)
    row[:9] = [127.0, 0.5, 1.5, 2.5, -0.5, -1.5, -2.5, 126.5, -127.0]
    codes, scales = orc.quantize_rows(W.I8, W.NEAREST, row)
    assert scales[0] == 1.0  # amax / 127 = 1
    assert list(codes[0, :9]) == [127, 0, 2, 2, 0, -2, -2, 126, -127]


def test_zero_and_tiny_rows_get_unit_scale():
    import oracle as orc

    rows = np.zeros((2, 128), np.float32)
    rows[1, 5] = 2.0 ** -110
    for dt in (W.I8, W.E4M3):
        codes, scales = orc.quantize_rows(dt, W.NEAREST, rows)
        assert list(scales) == [1.0, 1.0]
        assert not (codes.view(np.uint8) & 0x7F).any()


def test_e4m3_row_with_amax_448_is_plain_rne():
    import oracle as orc

    rng = np.random.default_rng(11)
    row = rng.uniform(-448, 448, 128).astype(np.float32)
    row[0] = 448.0
    codes, scales = orc.quantize_rows(W.E4M3, W.NEAREST, row)
    assert scales[0] == 1.0
    assert np.array_equal(codes[0], orc.f32_to_e4m3_bits(row))


@pytest.mark.parametrize("dt", [W.I8, W.E4M3])
def test_nearest_error_bound(dt):
    import oracle as orc

    rng = np.random.default_rng(12)
    acc = (rng.standard_normal((64, 128)) * rng.uniform(0.01, 10, (64, 1))).astype(np.float32)
    codes, scales = orc.quantize_rows(dt, W.NEAREST, acc)
    dec = codes.astype(np.float64) if dt == W.I8 else orc.e4m3_decode(codes).astype(np.float64)
    v = acc.astype(np.float64) / scales[:, None]
    if dt == W.I8:
        half = 0.5
    else:  # half the local grid spacing
        half = np.where(np.abs(dec) < 2.0 ** -6, 2.0 ** -10, 2.0 ** (np.floor(np.log2(np.maximum(np.abs(dec), 1e-30))) - 4))
    assert (np.abs(dec - v) <= half * (1 + 1e-6) + 1e-6).all()
    amax = np.abs(acc).max(axis=1)
    assert np.allclose(scales, amax / (127.0 if dt == W.I8 else 448.0), rtol=1e-7)


@pytest.mark.parametrize("dt", [W.I8, W.E4M3, W.BF16, W.F16])
def test_stochastic_rounding_brackets_and_is_unbiased(dt):
    import oracle as orc

    rng = np.random.default_rng(13)
    acc = (rng.standard_normal(128) * 3.0).astype(np.float32)
    acc[0] = 11.0 if dt == W.I8 else acc[0]
    nseeds = 4096
    vals = np.empty((nseeds, 128), np.float64)
    for k in range(nseeds):
        codes, sc = orc.quantize_rows(dt, W.STOCHASTIC, acc, h=3, s=2, epoch=1, seed=k * 7919 + 1)
        if dt == W.I8:
            vals[k] = codes[0].astype(np.float64) * sc[0]
        elif dt == W.E4M3:
            vals[k] = orc.e4m3_decode(codes[0]).astype(np.float64) * sc[0]
        elif dt == W.BF16:
            vals[k] = orc.bf16_decode(codes[0])
        else:
            vals[k] = orc.f16_decode(codes[0])
    lo, hi = vals.min(axis=0), vals.max(axis=0)
    # every outcome is one of the two grid neighbours of the exact value
    for j in range(128):
        assert len(np.unique(vals[:, j])) <= 2
    target = acc.astype(np.float64)
    if dt in (W.I8, W.E4M3):
        target = acc.astype(np.float64)  # scale * v reproduces acc up to rounding of v
    assert (lo <= target + 1e-6 * np.abs(target) + 1e-12).all() and (hi >= target - 1e-6 * np.abs(target) - 1e-12).all()
    mean = vals.mean(axis=0)
    sigma = (hi - lo) / 2 / np.sqrt(nseeds) + 1e-12
    assert (np.abs(mean - target) <= 4.5 * sigma + 1e-6 * np.abs(target)).all()


def test_stochastic_rounding_is_deterministic_and_epoch_dependent():
    import oracle as orc

    rng = np.random.default_rng(14)
    acc = rng.standard_normal((64, 128)).astype(np.float32)
    a, sa = orc.quantize_rows(W.E4M3, W.STOCHASTIC, acc, h=1, s=4, epoch=2, seed=7)
    b, sb = orc.quantize_rows(W.E4M3, W.STOCHASTIC, acc, h=1, s=4, epoch=2, seed=7)
    c, _ = orc.quantize_rows(W.E4M3, W.STOCHASTIC, acc, h=1, s=4, epoch=3, seed=7)
    assert np.array_equal(a, b) and np.array_equal(sa, sb)
    assert not np.array_equal(a, c)
