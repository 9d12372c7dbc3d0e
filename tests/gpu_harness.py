"""Drive the CUDA library and the oracle on the same inputs (test-only).

The GPU cache is a byte copy of the oracle cache; every step both run flush ->
step -> accept on identical inputs and the results are compared.  By default
the GPU cache is then overwritten with the oracle's, so each step is checked
from identical state; with resync=False both sides carry their own state on.
"""
import numpy as np
import torch

from speculative_state_replay_gb300 import api
from speculative_state_replay_gb300 import workloads as W

Y_ATOL, Y_RTOL = 2e-2, 1e-2          # bf16 outputs
F32_STATE_RTOL, F32_STATE_ATOL = 1e-4, 1e-6
# 2-byte checkpoints: at most one unit in the last place of the oracle's code
# (the GPU's tensor-core fold differs from the oracle's fp32 chain by
# summation order only, which can move a value across one rounding boundary),
# or within 2^-20 of it: near zero, where the fold's terms cancel, the fp32
# accumulators of the two orders still agree to ~1e-7 absolute while one unit
# of the code is smaller than that.  The slack only matters below |v| = 2^-12
# (bf16) or 2^-9 (f16).  One folded token changes a checkpoint by ~1e-2.
HALF_STATE_ULPS = 1
HALF_STATE_ABS = 2.0 ** -20


def dev_of(a, device):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    elif a.dtype == np.uint32:
        a = a.view(np.int32)
    return torch.from_numpy(a).to(device)


def host_of(t, like):
    a = t.detach().cpu().numpy()
    return a.view(like.dtype) if a.dtype.itemsize == np.dtype(like.dtype).itemsize else a.astype(like.dtype)


def bf16_f32(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


CACHE_ARRAYS = ("state", "scale", "x_cache", "B_cache", "dt_cache", "ring_start", "flush_epoch", "error_word")


def gpu_cache_from(oc, device="cuda"):
    pad = (oc.state.shape[1] - oc.H * 64 * 128) * oc.state.dtype.itemsize
    gc = api.RssmCache(oc.S, oc.H, oc.G, oc.W, oc.Tmax, oc.state_dtype, oc.rounding, device=device,
                       slot_pad_bytes=pad, read_dtype=getattr(oc, "read_dtype", None))
    sync_gpu_from(gc, oc)
    return gc


def cache_arrays(oc):
    rd = getattr(oc, "read_dtype", None)
    if rd is None:
        return CACHE_ARRAYS
    return CACHE_ARRAYS + (("read_state", "read_sf", "read_gs") if rd == W.NVFP4 else ("read_state", "read_scale"))


def sync_gpu_from(gc, oc):
    for name in cache_arrays(oc):
        src = getattr(oc, name)
        dst = getattr(gc, name)
        assert tuple(dst.shape) == src.shape, (name, tuple(dst.shape), src.shape)
        dst.copy_(dev_of(src, dst.device).view(dst.dtype))


def half_decode(dtype, bits):
    b = np.asarray(bits, np.uint16)
    return bf16_f32(b) if dtype == W.BF16 else b.view(np.float16).astype(np.float32)


def code_distance(bits_a, bits_b):
    """Distance in units in the last place between two 16-bit sign-magnitude
    codes (bf16 or f16), through the order-preserving map code -> integer
    (+0 and -0 both map to 0)."""
    def ordinal(b):
        b = np.asarray(b, np.uint16).astype(np.int64)
        mag = b & 0x7FFF
        return np.where(b & 0x8000, -mag, mag)

    return np.abs(ordinal(bits_a) - ordinal(bits_b))


def half_state_close(dtype, g, o, ulps=HALF_STATE_ULPS, abs_slack=HALF_STATE_ABS):
    """Per element: code distance <= ulps, or decoded difference <= abs_slack."""
    g = np.asarray(g).view(np.uint16)
    o = np.asarray(o).view(np.uint16)
    near = code_distance(g, o) <= ulps
    if near.all():
        return True
    diff = np.abs(half_decode(dtype, g).astype(np.float64) - half_decode(dtype, o).astype(np.float64))
    return bool(np.all(near | (diff <= abs_slack)))


def half_state_close_carried(dtype, g, o, row_ulps=2, abs_slack=HALF_STATE_ABS):
    """The bar for 2-byte checkpoints that have gone through several folds on
    each side without being re-synchronised: every element within `row_ulps`
    units in the last place of its row's largest magnitude (rows of 128
    dstate values).  A one-unit difference left by an earlier fold enters the
    next fold in absolute terms, scaled by its decay e^{c_end} < 1, next to the
    new fold's own rounding; where the new terms cancel to a small value that
    carried difference is many units of the new code but stays below one unit
    of the row's scale, and decays at every later fold."""
    g = np.asarray(g).view(np.uint16)
    o = np.asarray(o).view(np.uint16)
    n = g.size // 128 * 128
    gv = half_decode(dtype, g.reshape(-1)[:n]).astype(np.float64).reshape(-1, 128)
    ov = half_decode(dtype, o.reshape(-1)[:n]).astype(np.float64).reshape(-1, 128)
    if not np.array_equal(g.reshape(-1)[n:], o.reshape(-1)[n:]):
        return False
    m = np.abs(ov).max(axis=1, keepdims=True)
    mant = 7 if dtype == W.BF16 else 10
    _, e = np.frexp(m)  # m = f 2^e, f in [0.5, 1): the binade of m starts at 2^(e-1)
    ulp = np.where(m > 0, np.ldexp(1.0, e - 1 - mant), 0.0)
    if dtype == W.F16:
        ulp = np.maximum(ulp, 2.0 ** -24)
    return bool(np.all(np.abs(gv - ov) <= row_ulps * ulp + abs_slack))


def state_close(dtype, g, o, ulps=HALF_STATE_ULPS, carried=False):
    """Checkpoint comparison: bit-exact for 8-bit codes, 1e-4 relative for f32;
    bf16/f16: `ulps` units in the last place (with the near-zero slack) after
    one fold from identical state, or the carried-difference bar
    (half_state_close_carried) when both sides have folded on their own."""
    if dtype in (W.I8, W.E4M3):
        return np.array_equal(g, o)
    if dtype == W.F32:
        return bool(np.all(np.abs(g - o) <= F32_STATE_RTOL * np.abs(o) + F32_STATE_ATOL))
    if carried:
        return half_state_close_carried(dtype, g, o)
    return half_state_close(dtype, g, o, ulps=ulps)


class Pair:
    """Oracle + GPU replicas of one workload."""

    def __init__(self, orc, wl, oc, ids, pnat, device="cuda", seed=None, fused=False, gate=False, resync=True,
                 accept_flush=False):
        self.fused = fused  # GPU side through rssm_flush_step instead of rssm_flush + rssm_step
        # accept_flush: the GPU side applies each step's acceptance in the next
        # step's rssm_accept_flush (the oracle: flush, step, accept); between
        # steps the GPU's pnat lacks the pending acceptance
        self.accept_flush = accept_flush
        self.pending = None
        assert not (fused and accept_flush)
        self.gate = gate    # output gate z (seeded N(0, 1), bf16) on both sides, split path only
        # resync: after each comparison the GPU cache is overwritten with the
        # oracle's; without it both sides carry their own checkpoints on (2-byte
        # checkpoints folded on the tensor cores are then held to the
        # carried-difference bar)
        self.resync = resync
        assert not (fused and gate)
        self.orc, self.wl, self.oc = orc, wl, oc
        self.ids, self.pnat = ids, pnat.copy()
        self.device = device
        self.seed = wl.sr_seed if seed is None else seed
        self.gen = W.Generator(wl)
        self.A, self.D, self.dt_bias = self.gen.params()
        self.gc = gpu_cache_from(oc, device)
        d = lambda a: dev_of(a, device)  # noqa: E731
        self.gA, self.gD, self.gb = d(self.A), d(self.D), d(self.dt_bias)
        self.gids = d(ids)
        self.gpnat = d(self.pnat)
        self.scratch = api.alloc_scratch(self.gc, ids.size, wl.T)
        self.exact_state_steps = 0

    def step(self, inp, force=0, check=True):
        wl, oc, gc = self.wl, self.oc, self.gc
        d = lambda a: None if a is None else dev_of(a, self.device)  # noqa: E731
        cu = d(inp.cu_seqlens)
        z = None
        if self.gate:
            zf = np.random.default_rng(1000 + self.exact_state_steps + 7919 * inp.ntok).standard_normal(
                (max(inp.ntok, 1), wl.nheads, 64)).astype(np.float32)
            z = (zf.view(np.uint32) >> 16).astype(np.uint16)
        # oracle
        oc.flush(self.A, self.ids, self.pnat, wl.T, cu_seqlens=inp.cu_seqlens, force=force, seed=self.seed)
        y_o = oc.step(inp.x, inp.dt, self.A, inp.B, inp.C, self.D, self.dt_bias, self.ids, self.pnat, wl.T,
                      cu_seqlens=inp.cu_seqlens, z=None if z is None else z[:inp.ntok])
        oc.accept(self.ids, self.pnat, inp.accepted, wl.T, cu_seqlens=inp.cu_seqlens)
        # gpu
        out = torch.full((max(inp.ntok, 1), wl.nheads, 64), 0x7FC0, dtype=torch.int16, device=self.device)
        if self.fused:
            api.rssm_flush_step(gc, d(inp.x), d(inp.dt), self.gA, d(inp.B), d(inp.C), self.gD, self.gb, self.gids,
                                self.gpnat, wl.T, out, self.scratch, cu_seqlens=cu, force=force, seed=self.seed)
        else:
            if self.accept_flush and self.pending is not None:
                acc_prev, cu_prev = self.pending
                api.rssm_accept_flush(gc, self.gA, self.gids, self.gpnat, acc_prev, wl.T, wl.T, self.scratch,
                                      accept_cu_seqlens=cu_prev, cu_seqlens=cu, force=force, seed=self.seed)
            else:
                api.rssm_flush(gc, self.gA, self.gids, self.gpnat, wl.T, self.scratch, cu_seqlens=cu, force=force,
                               seed=self.seed)
            api.rssm_step(gc, d(inp.x), d(inp.dt), self.gA, d(inp.B), d(inp.C), self.gD, self.gb, self.gids,
                          self.gpnat, wl.T, out, self.scratch, cu_seqlens=cu, z=None if z is None else d(z))
        if self.accept_flush:
            self.pending = (d(inp.accepted), cu)
            self.pending_host = np.where(self.ids > 0, inp.accepted, 0).astype(np.int32)
        else:
            api.rssm_accept(gc, self.gids, self.gpnat, d(inp.accepted), wl.T, cu_seqlens=cu)
        torch.cuda.synchronize()
        y_g = out[: inp.ntok].cpu().numpy().view(np.uint16)
        if check:
            self.compare(y_g, y_o)
        return y_g, y_o

    def compare(self, y_g, y_o):
        oc, gc, wl = self.oc, self.gc, self.wl
        yg, yo = bf16_f32(y_g), bf16_f32(y_o)
        bad = ~(np.abs(yg - yo) <= Y_ATOL + Y_RTOL * np.abs(yo))
        assert not bad.any(), f"y mismatch at {np.argwhere(bad)[:5].tolist()}: gpu {yg[bad][:5]} oracle {yo[bad][:5]}"
        gp = self.gpnat.cpu().numpy()
        if self.accept_flush:  # the acceptance the next step applies
            gp = gp + self.pending_host
        assert np.array_equal(gp, self.pnat), "pnat"
        for name in ("ring_start", "flush_epoch", "error_word"):
            assert np.array_equal(host_of(getattr(gc, name), getattr(oc, name)), getattr(oc, name)), name
        for name in ("x_cache", "B_cache", "dt_cache"):
            g = host_of(getattr(gc, name), getattr(oc, name))
            assert np.array_equal(g, getattr(oc, name)), name
        gs = host_of(gc.state, oc.state)
        assert state_close(oc.state_dtype, gs, oc.state, carried=not self.resync), "checkpoint"
        if oc.state_dtype in (W.I8, W.E4M3):
            assert np.array_equal(host_of(gc.scale, oc.scale), oc.scale), "scales"
        if getattr(oc, "read_dtype", None) is not None:  # the read checkpoint: nearest codes, bit for bit
            for name in cache_arrays(oc)[len(CACHE_ARRAYS):]:
                o = getattr(oc, name)
                assert np.array_equal(host_of(getattr(gc, name), o), o), name
        if np.array_equal(gs, oc.state):
            self.exact_state_steps += 1
        if self.resync:  # continue from identical state
            sync_gpu_from(gc, oc)
            pn = self.pnat - self.pending_host if self.accept_flush else self.pnat
            self.gpnat.copy_(dev_of(np.ascontiguousarray(pn, np.int32), self.device))


def init_gpu_cache_like_bench(wl, gen, ids, device="cuda"):
    """A full-size GPU cache initialised the way bench.py initialises it:
    every active row's FP32 state through rssm_init_state (16 rows a call),
    prefilled rings, the workload's ring starts.  Returns (cache, pnat0)."""
    gc = api.RssmCache(wl.num_slots, wl.nheads, wl.ngroups, wl.max_window, wl.npredicted, wl.state_dtype,
                       wl.rounding, device=device, slot_pad_bytes=wl.slot_pad_bytes, read_dtype=wl.read_dtype)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(device)  # noqa: E731
    active = ids[ids > 0]
    for i in range(0, active.size, 16):
        sl = active[i:i + 16]
        api.rssm_init_state(gc, t(gen.init_states(i, sl.size)), t(sl.astype(np.int32)), seed=wl.sr_seed)
    pnat0 = np.zeros(ids.size, np.int32)
    if wl.prefill_live:
        for b, s in enumerate(ids):
            if s > 0:
                x, B, dtp, live = gen.ring_prefill(int(s))
                gc.x_view()[s] = t(x.view(np.int16))
                gc.B_view()[s] = t(B.view(np.int16))
                gc.dt_view()[s] = t(dtp)
                pnat0[b] = live
    gc.ring_start.copy_(t(gen.ring_start()))
    torch.cuda.synchronize()
    return gc, pnat0


def oracle_cache_for_rows(orc, wl, gen, ids, rows):
    """An oracle cache holding only the given rows of a full-size workload,
    initialised exactly as init_gpu_cache_like_bench initialises them (rows
    are independent, so the oracle can follow a sample of them)."""
    oc = orc.OracleCache(wl.num_slots, wl.nheads, wl.ngroups, wl.max_window, wl.npredicted, wl.state_dtype,
                         wl.rounding, slot_pad_bytes=wl.slot_pad_bytes, read_dtype=wl.read_dtype)
    act_pos = np.cumsum(ids > 0) - 1  # index of each row among the active rows
    for b in rows:
        s = int(ids[b])
        if s <= 0:
            continue
        oc.init_state(gen.init_states(int(act_pos[b]), 1), np.array([s], np.int32), seed=wl.sr_seed)
        if wl.prefill_live:
            x, B, dtp, _ = gen.ring_prefill(s)
            oc.x_view()[s] = x
            oc.B_view()[s] = B
            oc.dt_view()[s] = dtp
    oc.ring_start[:] = gen.ring_start()
    return oc


def token_rows(inp, rows, T):
    """Token indices of `rows` in a step's packed inputs and the cu_seqlens of
    those rows packed alone (None without varlen)."""
    if inp.cu_seqlens is None:
        tok = (np.asarray(rows)[:, None] * T + np.arange(T)[None]).reshape(-1)
        return tok, None
    cu = inp.cu_seqlens
    parts = [np.arange(cu[b], cu[b + 1]) for b in rows]
    lens = np.array([p.size for p in parts], np.int32)
    sub = np.zeros(len(rows) + 1, np.int32)
    sub[1:] = np.cumsum(lens)
    return np.concatenate(parts).astype(np.int64), sub
