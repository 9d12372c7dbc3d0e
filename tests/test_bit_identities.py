"""The exact fp32 bit identities the flush kernel's int8 paths use in place
of conversion instructions, checked exhaustively (no GPU needed): int8 code ->
fp32 by placing (q + 128) in the fraction of 2^23 and subtracting 2^23 + 128;
round-to-nearest-even onto -127..127 by adding 1.5 * 2^23 to the clamped value
and taking the low byte of the sum.  Same operations and rounding (IEEE fp32, round to nearest
even) as the device code."""
import numpy as np


def test_int8_code_to_f32():
    q = np.arange(-128, 128)
    bits = (0x4B000000 | ((q & 0xFF) ^ 0x80)).astype(np.uint32)
    f = bits.view(np.float32) - np.float32(8388736.0)
    assert np.array_equal(f.astype(np.int64), q)


def test_int8_round_nearest_even():
    rng = np.random.default_rng(0)
    v = np.concatenate([rng.uniform(-130, 130, 200000), np.arange(-130, 131) + 0.5,
                        np.arange(-130, 131).astype(float)]).astype(np.float32)
    t = (np.clip(v, -127, 127).astype(np.float32) + np.float32(12582912.0)).astype(np.float32)
    code = (t.view(np.uint32) & 0xFF).astype(np.int64)
    ref = np.clip(np.rint(v.astype(np.float64)), -127, 127).astype(np.int64) & 0xFF
    assert np.array_equal(code, ref)
