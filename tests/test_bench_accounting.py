"""The benchmark's algorithmic-byte accounting (CPU only): the per-unit
figures the roofline fractions are computed from.

Readout, per active (row, head): S0 (64 x 128 state elements, plus 64 fp32 row
scales for 8-bit states), the head's share of the group's C rows (T_b x 128
bf16 / heads per group) and y (T_b x 64 bf16).  Flush, per flushed (row,
head): S0 read and written (plus scales), the live x rows (p x 64 bf16), the
head's share of the live B rows (p x 128 bf16 / heads per group) and dt'
(p x f32).
"""
import importlib.util
import os

import pytest

from speculative_state_replay_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_readout_bytes_of_the_mamba2_decode_launch(bench):
    """bf16, 128 heads in 8 groups, T = 4: 16 960 bytes per (row, head), so a
    launch over 64 active rows is 138 936 320 bytes."""
    wl = W.config("mamba2_decode")
    row = (1, 0, 0, 4, 0, 1)  # (slot, ring start, p, T_b, tok0, flags: active)
    assert bench.algorithmic_bytes(wl, [row], None, 2) == 128 * (8192 * 2 + 4 * 256 / 16 + 4 * 128)
    assert bench.algorithmic_bytes(wl, [row] * 64, None, 2) == 138936320


def test_readout_bytes_of_8bit_and_inactive_rows(bench):
    wl = W.config("eight_bit")
    active = (1, 0, 3, 4, 0, 1)
    padding = (0, 0, 0, 4, 4, 0)  # a padding row only writes its zero outputs
    got = bench.algorithmic_bytes(wl, [active, padding], None, 1)
    assert got == 128 * (8192 + 256 + 4 * 256 / 16 + 4 * 128) + 128 * 4 * 128


def test_flush_bytes_of_a_full_window(bench):
    """bf16, p = 16: 35 136 bytes per (row, head); the full-window Mamba-2
    decode flush (64 rows x 128 heads) is 287 834 112 bytes."""
    wl = W.config("mamba2_decode")
    assert bench.flush_bytes(wl, [16], 2) == 128 * (2 * 16384 + 16 * 128 + 16 * 256 / 16 + 16 * 4)
    assert bench.flush_bytes(wl, [16] * 64, 2) == 287834112
    # 8-bit states add the 64 row scales read and written
    assert bench.flush_bytes(W.config("eight_bit"), [0], 1) == 128 * (2 * 8192 + 512)


def test_bytes_with_a_separate_read_checkpoint(bench):
    """The separate-checkpoint workload (fp16 recurrence, e4m3 read copy): the
    readout streams 8192 codes + 64 row scales per (row, head) -- about half of
    a 2-byte checkpoint -- and a fold also writes the read copy."""
    wl = W.config("separate")
    row = (1, 0, 0, 5, 0, 1)
    assert bench.algorithmic_bytes(wl, [row], None, 1) == 128 * (8192 + 256 + 5 * 256 / 16 + 5 * 128)
    assert bench.flush_bytes(wl, [16], 2) == 128 * (2 * 16384 + 16 * 132 + 16 * 256 / 16 + 8192 + 256)


def test_bytes_with_an_nvfp4_read_checkpoint(bench):
    """NVFP4 read copy: 4096 bytes of codes + 512 of block scales per (row,
    head) for the readout; a fold also writes them."""
    wl = W.config("separate_nvfp4")
    row = (1, 0, 0, 5, 0, 1)
    assert bench.algorithmic_bytes(wl, [row], None, 0.5) == 128 * (4096 + 512 + 5 * 256 / 16 + 5 * 128)
    assert bench.flush_bytes(wl, [16], 2) == 128 * (2 * 16384 + 16 * 132 + 16 * 256 / 16 + 4096 + 512)
