"""Drive the CUDA library and the oracle on the same inputs (test-only).

The GPU cache is a byte copy of the oracle cache; every step both run flush ->
step -> accept on identical inputs and the results are compared.  After the
comparison the GPU cache is overwritten with the oracle's, so each step is
checked from identical state.
"""
import numpy as np
import torch

from speculative_state_replay_gb300 import api
from speculative_state_replay_gb300 import workloads as W

Y_ATOL, Y_RTOL = 2e-2, 1e-2          # bf16 outputs
F32_STATE_RTOL, F32_STATE_ATOL = 1e-4, 1e-6
HALF_STATE_ATOL, HALF_STATE_RTOL = 2e-2, 1e-2


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
                       slot_pad_bytes=pad)
    sync_gpu_from(gc, oc)
    return gc


def sync_gpu_from(gc, oc):
    for name in CACHE_ARRAYS:
        src = getattr(oc, name)
        dst = getattr(gc, name)
        assert tuple(dst.shape) == src.shape, (name, tuple(dst.shape), src.shape)
        dst.copy_(dev_of(src, dst.device).view(dst.dtype))


def state_close(dtype, g, o):
    """Checkpoint comparison: bit-exact for 8-bit codes, tolerance otherwise."""
    if dtype in (W.I8, W.E4M3):
        return np.array_equal(g, o)
    if dtype == W.F32:
        return bool(np.all(np.abs(g - o) <= F32_STATE_RTOL * np.abs(o) + F32_STATE_ATOL))
    f = bf16_f32 if dtype == W.BF16 else (lambda b: np.asarray(b, np.uint16).view(np.float16).astype(np.float32))
    return bool(np.allclose(f(g), f(o), atol=HALF_STATE_ATOL, rtol=HALF_STATE_RTOL))


class Pair:
    """Oracle + GPU replicas of one workload."""

    def __init__(self, orc, wl, oc, ids, pnat, device="cuda", seed=None, fused=False, gate=False):
        self.fused = fused  # GPU side through rssm_flush_step instead of rssm_flush + rssm_step
        self.gate = gate    # output gate z (seeded N(0, 1), bf16) on both sides, split path only
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
            api.rssm_flush(gc, self.gA, self.gids, self.gpnat, wl.T, self.scratch, cu_seqlens=cu, force=force,
                           seed=self.seed)
            api.rssm_step(gc, d(inp.x), d(inp.dt), self.gA, d(inp.B), d(inp.C), self.gD, self.gb, self.gids,
                          self.gpnat, wl.T, out, self.scratch, cu_seqlens=cu, z=None if z is None else d(z))
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
        assert np.array_equal(self.gpnat.cpu().numpy(), self.pnat), "pnat"
        for name in ("ring_start", "flush_epoch", "error_word"):
            assert np.array_equal(host_of(getattr(gc, name), getattr(oc, name)), getattr(oc, name)), name
        for name in ("x_cache", "B_cache", "dt_cache"):
            g = host_of(getattr(gc, name), getattr(oc, name))
            assert np.array_equal(g, getattr(oc, name)), name
        gs = host_of(gc.state, oc.state)
        assert state_close(oc.state_dtype, gs, oc.state), "checkpoint"
        if oc.state_dtype in (W.I8, W.E4M3):
            assert np.array_equal(host_of(gc.scale, oc.scale), oc.scale), "scales"
        if np.array_equal(gs, oc.state):
            self.exact_state_steps += 1
        # continue from identical state
        sync_gpu_from(gc, oc)
        self.gpnat.copy_(dev_of(self.pnat, self.device))
