"""Pins for the oracle's scalar building blocks (CPU only).

Each check compares the oracle against something other than itself: float64
libm through numpy, numpy's and PyTorch's format conversions, cuRAND's host
Philox4_32_10 generator and numpy's Philox4x64-10 bit generator, and closed
forms of the Philox Weyl constants.
"""
import ctypes
import decimal
import math
import os

import numpy as np
import pytest
import torch


def ulp_err(got32, ref64):
    """Error in units of the float32 ulp at the reference."""
    ref32 = ref64.astype(np.float32)
    spacing = np.spacing(np.abs(ref32)).astype(np.float64)
    return np.abs(got32.astype(np.float64) - ref64) / spacing


def test_spec_exp_within_2ulp(orc):
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.uniform(-87.0, 88.0, 200000), rng.uniform(-1, 1, 50000),
                        np.linspace(-87.0, 0.0, 20001)]).astype(np.float32)
    y = orc.spec_exp(x)
    ref = np.exp(x.astype(np.float64))
    keep = ref >= 2.0 ** -126  # normal results
    assert ulp_err(y[keep], ref[keep]).max() <= 2.0
    assert orc.spec_exp(np.float32([0.0]))[0] == 1.0
    assert orc.spec_exp(np.float32([-100.0]))[0] == 0.0
    assert np.isinf(orc.spec_exp(np.float32([100.0]))[0])


def test_spec_log1p_within_2p5ulp(orc):
    rng = np.random.default_rng(2)
    z = np.concatenate([rng.uniform(0, 0.25, 100000), rng.uniform(0.25, 4, 100000),
                        np.exp(rng.uniform(-40, 20, 100000)), np.float32([0.25, 0.2499999, 1.0, 3.0])])
    z = z.astype(np.float32)
    y = orc.spec_log1p(z)
    ref = np.log1p(z.astype(np.float64))
    assert ulp_err(y[ref > 0], ref[ref > 0]).max() <= 2.5
    assert orc.spec_log1p(np.float32([0.0]))[0] == 0.0


def test_spec_softplus_matches_definition(orc):
    rng = np.random.default_rng(3)
    v = np.concatenate([rng.normal(-2.0, 0.5, 200000), rng.uniform(-30, 25, 100000)]).astype(np.float32)
    y = orc.spec_softplus(v)
    v64 = v.astype(np.float64)
    ref = np.where(v64 > 20, v64, np.log1p(np.exp(v64)))
    keep = ref > 2.0 ** -126
    assert ulp_err(y[keep], ref[keep]).max() <= 3.0
    big = np.float32([20.5, 30.0])
    assert np.array_equal(orc.spec_softplus(big), big)


def _frac_weyl(bits, expr):
    decimal.getcontext().prec = 80
    return int((decimal.Decimal(2) ** bits) * expr)


def test_philox_weyl_constants_are_closed_forms():
    decimal.getcontext().prec = 80
    phi_m1 = (decimal.Decimal(5).sqrt() - 1) / 2
    sqrt3_m1 = decimal.Decimal(3).sqrt() - 1
    assert _frac_weyl(32, phi_m1) == 0x9E3779B9
    assert _frac_weyl(32, sqrt3_m1) == 0xBB67AE85
    assert _frac_weyl(64, phi_m1) == 0x9E3779B97F4A7C15
    assert _frac_weyl(64, sqrt3_m1) == 0xBB67AE8584CAA73B


def test_philox4x64_10_matches_numpy(orc):
    for key, ctr in [((1, 2), (5, 0, 0, 0)), ((0xDEADBEEF12345678, 0x0F0F0F0F), (2**64 - 3, 7, 9, 11))]:
        bg = np.random.Philox(key=np.array(key, np.uint64), counter=np.array(ctr, np.uint64))
        got = bg.random_raw(4)
        # numpy advances the 256-bit counter before producing a block
        c = list(ctr)
        c[0] = (c[0] + 1) % 2**64
        if c[0] == 0:
            c[1] += 1
        want = orc.philox4x64(10, c, key)
        assert np.array_equal(got, want)


def _curand():
    for p in (os.environ.get("CUDA_HOME", "/usr/local/cuda") + "/lib64/libcurand.so", "libcurand.so.10",
              "libcurand.so"):
        try:
            return ctypes.CDLL(p)
        except OSError:
            continue
    return None


def test_philox4x32_10_matches_curand_host_generator(orc):
    cr = _curand()
    if cr is None:
        pytest.skip("cuRAND host library not available")
    gen = ctypes.c_void_p()
    if cr.curandCreateGeneratorHost(ctypes.byref(gen), 161) != 0:  # CURAND_RNG_PSEUDO_PHILOX4_32_10
        pytest.skip("cuRAND host generator unavailable")
    try:
        for seed in (0x123456789ABCDEF, 20261202):
            assert cr.curandSetPseudoRandomGeneratorSeed(gen, ctypes.c_ulonglong(seed)) == 0
            assert cr.curandSetGeneratorOffset(gen, ctypes.c_ulonglong(0)) == 0
            out = np.zeros(4096, np.uint32)
            assert cr.curandGenerate(gen, out.ctypes.data_as(ctypes.c_void_p), ctypes.c_size_t(out.size)) == 0
            key = (seed & 0xFFFFFFFF, seed >> 32)
            # the host generator emits the first block of subsequence i as words 4i..4i+3;
            # Philox4x32 puts the subsequence in counter word 2
            for i in range(out.size // 4):
                assert np.array_equal(out[4 * i:4 * i + 4], orc.philox4x32(10, (0, 0, i, 0), key)), i
    finally:
        cr.curandDestroyGenerator(gen)


def test_sr_word_uses_7_rounds_and_counter_layout(orc):
    seed = 0x0000000700000003
    blk = orc.philox4x32(7, (123 >> 2, 5, 9, 2), (3, 7))
    assert orc.sr_word(seed, 123, 5, 9, 2) == blk[123 & 3]
    # uniformity of the top 24 bits (chi-square over 64 bins)
    u = np.array([orc.sr_word(7, e, 1, 1, 1) >> 26 for e in range(20000)])
    counts = np.bincount(u, minlength=64)
    chi2 = ((counts - 20000 / 64) ** 2 / (20000 / 64)).sum()
    assert chi2 < 120  # 63 dof, p ~ 1e-5


def test_bf16_nearest_matches_torch(orc):
    rng = np.random.default_rng(4)
    x = np.concatenate([rng.standard_normal(100000) * 10.0 ** rng.integers(-30, 30, 100000),
                        np.float32([1.00390625, 1.01171875, -1.00390625, 0.0, -0.0])]).astype(np.float32)
    # exact ties: midpoints between bf16 neighbours
    mids = ((rng.integers(0x3F80, 0x4F00, 10000).astype(np.uint32) << 16) | 0x8000).view(np.float32)
    x = np.concatenate([x, mids, -mids])
    got = orc.f32_to_bf16_bits(x)
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want)


def test_f16_nearest_matches_numpy_and_saturates(orc):
    rng = np.random.default_rng(5)
    x = (rng.standard_normal(200000) * 10.0 ** rng.uniform(-9, 4.7, 200000)).astype(np.float32)
    x = x[np.abs(x) < 65504]
    mids = (np.arange(1, 60000, 7, dtype=np.float64) + 0.5).astype(np.float32)  # ties at integer spacing
    x = np.concatenate([x, mids, -mids, np.float32([2.0 ** -25, 3 * 2.0 ** -26, 2.0 ** -24])])
    got = orc.f32_to_f16_bits(x)
    want = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, want)
    sat = orc.f32_to_f16_bits(np.float32([65519.0, 65520.0, 1e6, -1e30]))
    assert list(sat) == [0x7BFF, 0x7BFF, 0x7BFF, 0xFBFF]
    codes = np.arange(65536, dtype=np.uint16)
    finite = (codes & 0x7C00) != 0x7C00
    assert np.array_equal(orc.f16_decode(codes[finite]), codes[finite].view(np.float16).astype(np.float32))


def test_e4m3_decode_table_matches_torch_and_definition(orc):
    codes = np.arange(256, dtype=np.uint8)
    got = orc.e4m3_decode(codes)
    want = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    nan = (codes & 0x7F) == 0x7F
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    # definition: exponent field e (bias 7), fraction m; subnormal m * 2^-9; max 448
    for c in range(256):
        if (c & 0x7F) == 0x7F:
            continue
        e, m = (c >> 3) & 15, c & 7
        v = m * 2.0 ** -9 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7)
        assert got[c] == (-v if c & 0x80 else v)
    assert np.nanmax(got) == 448.0


def test_e4m3_nearest_matches_torch_in_range_and_saturates(orc):
    rng = np.random.default_rng(6)
    x = (rng.standard_normal(200000) * 10.0 ** rng.uniform(-4, 2.6, 200000)).astype(np.float32)
    x = x[np.abs(x) < 448]
    grid = orc.e4m3_decode(np.arange(0, 0x7E, dtype=np.uint8)).astype(np.float64)
    mids = ((grid[:-1] + grid[1:]) / 2).astype(np.float32)  # exact ties
    x = np.concatenate([x, mids, -mids])
    got = orc.f32_to_e4m3_bits(x)
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, want)
    sat = orc.f32_to_e4m3_bits(np.float32([448.0, 463.9, 464.0, 500.0, 1e9, -1e9]))
    assert list(sat) == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE]
