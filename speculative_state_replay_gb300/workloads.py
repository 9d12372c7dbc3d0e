"""Seeded synthetic decode workloads (inputs only, no arithmetic of the op).

The same generator feeds the CUDA library and the CPU oracle so both see
identical bytes.  Nothing here computes any part of the selective-state-update:
it only draws random numbers with fixed seeds and lays them out in the shapes
the op takes.  bf16 values are drawn in fp32 and truncated to their top 16 bits
(a distribution choice, not the op's rounding).

Shapes follow the ring-buffer cache contract of FlashInfer PR #3975 ("mamba
checkpointing SSU: two-kernel split + ring-buffer cache", Description item 2):
x_cache [slot][H][L][64], B_cache [slot][G][L][128], dt_cache [slot][H][L],
L = max_window + npredicted; slot 0 is a padding slot (vLLM replayssm_cutedsl
API docs, module docstring).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

F32, BF16, F16, I8, E4M3, NVFP4 = 0, 1, 2, 3, 4, 5
NEAREST, STOCHASTIC = 0, 1
DTYPE_NAMES = {F32: "f32", BF16: "bf16", F16: "f16", I8: "int8", E4M3: "e4m3", NVFP4: "nvfp4"}
DTYPE_BYTES = {F32: 4, BF16: 2, F16: 2, I8: 1, E4M3: 1, NVFP4: 0.5}
P_DIM, N_DIM = 64, 128
BASE_SEED = 20261202


@dataclasses.dataclass
class Workload:
    name: str
    num_slots: int
    nheads: int
    ngroups: int
    max_window: int
    npredicted: int
    state_dtype: int
    batch: int
    T: int                       # tokens per row (max tokens per row when varlen)
    steps: int
    rounding: int = NEAREST
    sr_seed: int = 0
    varlen: bool = False         # rows carry 1..T tokens through cu_seqlens
    accept: str = "uniform"      # "uniform": a ~ U{0..T_b}; "all": a = T_b
    ring_start_random: bool = False
    prefill_live: int = 0        # initial live tokens ~ U{0..prefill_live} with random rings
    slot_pad_bytes: int = 0      # padding after each slot in every cache tensor
    pad_row: bool = False        # one extra row that points at padding slot 0
    config_id: int = 0
    read_dtype: int | None = None  # separate 8-bit read checkpoint (I8 / E4M3), nearest-encoded

    @property
    def L(self) -> int:
        return self.max_window + self.npredicted

    @property
    def hpg(self) -> int:
        return self.nheads // self.ngroups

    @property
    def seed(self) -> int:
        return BASE_SEED + self.config_id

    def describe(self) -> dict:
        return {
            "workload": self.name, "batch": self.batch, "num_slots": self.num_slots, "nheads": self.nheads,
            "ngroups": self.ngroups, "dim": P_DIM, "dstate": N_DIM, "state_dtype": DTYPE_NAMES[self.state_dtype],
            "rounding": "stochastic" if self.rounding == STOCHASTIC else "nearest", "max_window": self.max_window,
            "T": self.T, "L": self.L, "varlen": self.varlen,
            "read_checkpoint": None if self.read_dtype is None else DTYPE_NAMES[self.read_dtype],
        }


def config(name: str, **overrides) -> Workload:
    """The five decode configurations (sizes of the benchmark definitions),
    and "separate" / "separate_nvfp4": the sweep's largest batch with the
    separate checkpoints of vLLM PR #65660 (Overview: an FP16 recurrence
    checkpoint with stochastic rounding, an FP8 or NVFP4 read checkpoint the
    readout streams)."""
    base = {
        "tiny": dict(num_slots=5, nheads=8, ngroups=1, max_window=16, npredicted=4, state_dtype=F32, batch=4,
                     T=4, steps=12, pad_row=True, config_id=1),
        "mamba2_decode": dict(num_slots=256, nheads=128, ngroups=8, max_window=16, npredicted=4,
                              state_dtype=BF16, batch=64, T=4, steps=64, config_id=2),
        "large_batch": dict(num_slots=1024, nheads=64, ngroups=8, max_window=16, npredicted=7, state_dtype=F16,
                            batch=512, T=7, steps=64, ring_start_random=True, config_id=3),
        "eight_bit": dict(num_slots=257, nheads=128, ngroups=8, max_window=16, npredicted=4, state_dtype=I8,
                          batch=128, T=4, steps=16, accept="all", config_id=4),
        "sweep": dict(num_slots=2 * 1024 + 1, nheads=128, ngroups=8, max_window=16, npredicted=5,
                      state_dtype=BF16, batch=1024, T=5, steps=32, varlen=True, ring_start_random=True,
                      prefill_live=16, slot_pad_bytes=4096, config_id=5),
        "separate": dict(num_slots=2 * 1024 + 1, nheads=128, ngroups=8, max_window=16, npredicted=5,
                         state_dtype=F16, rounding=STOCHASTIC, sr_seed=7, read_dtype=E4M3, batch=1024, T=5,
                         steps=32, varlen=True, ring_start_random=True, prefill_live=16, slot_pad_bytes=4096,
                         config_id=6),
        "separate_nvfp4": dict(num_slots=2 * 1024 + 1, nheads=128, ngroups=8, max_window=16, npredicted=5,
                               state_dtype=F16, rounding=STOCHASTIC, sr_seed=7, read_dtype=NVFP4, batch=1024, T=5,
                               steps=32, varlen=True, ring_start_random=True, prefill_live=16, slot_pad_bytes=4096,
                               config_id=7),
    }[name]
    base.update(overrides)
    if name in ("sweep", "separate", "separate_nvfp4") and "batch" in overrides and "num_slots" not in overrides:
        base["num_slots"] = 2 * overrides["batch"] + 1
    return Workload(name=name, **base)


def _bf16_bits(a: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(a, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


@dataclasses.dataclass
class StepInputs:
    x: np.ndarray            # bf16 bits [tok][H][64]
    dt: np.ndarray           # f32 [tok][H]
    B: np.ndarray            # bf16 bits [tok][G][128]
    C: np.ndarray            # bf16 bits [tok][G][128]
    accepted: np.ndarray     # i32 [batch]
    cu_seqlens: np.ndarray | None  # i32 [batch+1]
    ntok: int


class Generator:
    """Deterministic draws for one workload.  Each draw has its own stream."""

    def __init__(self, wl: Workload, seed: int | None = None):
        self.wl = wl
        self.seed = wl.seed if seed is None else seed

    def _rng(self, *tag) -> np.random.Generator:
        return np.random.default_rng([self.seed, *tag])

    # ------------------------------------------------------------------ #
    def params(self):
        """A [H] = -exp(U(0, ln 16)), D [H] ~ N(0,1), dt_bias [H] ~ U(-0.5, 0.5)."""
        wl, r = self.wl, self._rng(1)
        A = (-np.exp(r.uniform(0.0, math.log(16.0), wl.nheads))).astype(np.float32)
        D = r.standard_normal(wl.nheads).astype(np.float32)
        dt_bias = r.uniform(-0.5, 0.5, wl.nheads).astype(np.float32)
        return A, D, dt_bias

    def slot_idx(self) -> np.ndarray:
        """Unique active slot ids in [1, S); with pad_row one extra row uses slot 0."""
        wl, r = self.wl, self._rng(2)
        ids = r.choice(np.arange(1, wl.num_slots), size=wl.batch, replace=False).astype(np.int32)
        if wl.pad_row:
            pos = int(r.integers(0, wl.batch + 1))
            ids = np.insert(ids, pos, 0).astype(np.int32)
        return ids

    @property
    def rows(self) -> int:
        return self.wl.batch + (1 if self.wl.pad_row else 0)

    def init_states(self, first: int, count: int) -> np.ndarray:
        """FP32 prefill states for rows first..first+count-1: N(0, 0.1), [n][H][64][128]."""
        wl = self.wl
        out = np.empty((count, wl.nheads, P_DIM, N_DIM), np.float32)
        for i in range(count):
            r = self._rng(3, first + i)
            out[i] = (r.standard_normal((wl.nheads, P_DIM, N_DIM), dtype=np.float32) * np.float32(0.1))
        return out

    def ring_prefill(self, slot: int):
        """Random ring contents and live count for one slot (prefill_live > 0).

        x and B ring rows as for step inputs; dt' ring entries log-uniform in
        [0.01, 0.6] (a positive spread like the post-softplus step values).
        """
        wl, r = self.wl, self._rng(4, slot)
        L = wl.L
        x = _bf16_bits(r.standard_normal((wl.nheads, L, P_DIM), dtype=np.float32))
        B = _bf16_bits(r.standard_normal((wl.ngroups, L, N_DIM), dtype=np.float32) / np.float32(math.sqrt(N_DIM)))
        dtp = np.exp(r.uniform(math.log(0.01), math.log(0.6), (wl.nheads, L))).astype(np.float32)
        live = int(r.integers(0, wl.prefill_live + 1))
        return x, B, dtp, live

    def ring_start(self) -> np.ndarray:
        wl = self.wl
        if not wl.ring_start_random:
            return np.zeros(wl.num_slots, np.int32)
        return self._rng(5).integers(0, wl.L, wl.num_slots).astype(np.int32)

    def step(self, k: int) -> StepInputs:
        """Inputs of decode step k: x ~ N(0,1); B, C ~ N(0,1)/sqrt(128) (bf16);
        dt ~ N(-2, 0.5); tokens per row T (or U{1..T} when varlen); accepted
        drafts ~ U{0..T_b} (or all T_b)."""
        wl, r = self.wl, self._rng(6, k)
        rows = self.rows
        if wl.varlen:
            lens = r.integers(1, wl.T + 1, rows).astype(np.int32)
            cu = np.zeros(rows + 1, np.int32)
            cu[1:] = np.cumsum(lens)
        else:
            lens = np.full(rows, wl.T, np.int32)
            cu = None
        ntok = int(lens.sum())
        x = _bf16_bits(r.standard_normal((ntok, wl.nheads, P_DIM), dtype=np.float32))
        inv = np.float32(1.0 / math.sqrt(N_DIM))
        B = _bf16_bits(r.standard_normal((ntok, wl.ngroups, N_DIM), dtype=np.float32) * inv)
        C = _bf16_bits(r.standard_normal((ntok, wl.ngroups, N_DIM), dtype=np.float32) * inv)
        dt = (r.standard_normal((ntok, wl.nheads), dtype=np.float32) * np.float32(0.5) - np.float32(2.0))
        if wl.accept == "all":
            acc = lens.copy()
        else:
            acc = np.array([r.integers(0, int(t) + 1) for t in lens], np.int32)
        return StepInputs(x=x, dt=dt.astype(np.float32), B=B, C=C, accepted=acc.astype(np.int32), cu_seqlens=cu,
                          ntok=ntok)
