"""Benchmark: one decode step of the ReplaySSM checkpointing SSU on GB300.

A step = accept + flush + step over one batch of synthetic decode inputs:
by default (--path split) rssm_accept_flush (the previous step's accepted
drafts, then classify + fold + bookkeeping) -> rssm_step (precompute +
readout); with --path fused, rssm_flush_step (flush decision + precompute,
then the fused fold + readout) -> rssm_accept.
Default workload: the largest batch of the decode sweep -- 1024 rows of 2049
slots, 128 heads in 8 groups, bf16 checkpoints, window 16, 1..5 draft tokens
per row through cu_seqlens, padded slot pages, prefilled rings.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]
                    [--config NAME] [--batch B] [--path fused|split] [--force-flush]
                    [--full-window] [--no-full-window-leg] [--no-e2e] [--no-cpu-baseline]

Timing: W untimed warm-up steps, then K steps, each one CUDA graph (the
library's kernels chained by programmatic dependent launch) bracketed by CUDA
events on the launching stream -> `value`.  A second pass replays the same
steps as one graph per launch group with events between the groups -> the
per-kernel durations behind `roofline`.  A last leg flushes every active row
with a full window (pnat = max_window, set outside the events) -> the flush
roofline.  Between steps (outside the events) a 1 GiB buffer is written and a
512 MiB buffer read, so every step starts with a cold L2 that holds no dirty
lines.  Under torchrun (N > 1) every rank runs an independent replica (weak
scaling, no data-path collective); the time is the max over ranks.  Prints one
JSON line on rank 0.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import tempfile
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from speculative_state_replay_gb300 import workloads as W  # noqa: E402

METRIC = "slot-head SSU updates/s and achieved HBM GB/s vs GB300 roofline (1 GPU)"
UNIT = "slot-head updates/s"
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=32)
    ap.add_argument("--warmup", type=int, default=4)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--config", default="sweep")
    ap.add_argument("--batch", type=int, default=None, help="override the workload's batch")
    ap.add_argument("--force-flush", action="store_true", help="flush every active row every step")
    ap.add_argument("--full-window", action="store_true",
                    help="before every step (outside the timed region) give every active row a full window of "
                         "live tokens (pnat = max_window) and flush them all: the flush roofline run")
    ap.add_argument("--path", default="split", choices=["fused", "split"],
                    help="fused: rssm_flush_step; split: rssm_flush then rssm_step")
    ap.add_argument("--no-full-window-leg", action="store_true",
                    help="skip the full-window flush leg (split path only) at the end of the run")
    ap.add_argument("--full-window-reps", type=int, default=8)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="CPU budget of the oracle baseline sample")
    args = ap.parse_args()
    if args.full_window:  # the refill runs between steps, so there is no back-to-back leg or oracle sample
        args.no_e2e = True
        args.no_cpu_baseline = True
        args.no_full_window_leg = True
    if args.path == "fused":
        args.no_full_window_leg = True
    return args


def workload(args):
    kw = {}
    if args.batch is not None:
        kw["batch"] = args.batch
    return W.config(args.config, **kw)


L2_BYTES = 129e6  # GB300 L2 capacity


def profiled_traffic(kernel, workload_name, units_per_launch=None):
    """DRAM bytes per launch (dram__bytes_read + dram__bytes_write) from the
    committed ncu summary of `kernel` on this workload, if the kernel's sources
    still hash as they did when the counters were taken; else None.  A summary
    taken on a smaller launch of the same workload gives its traffic per
    (row, head) unit, scaled here to the launch's units."""
    import hashlib
    import re

    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload_name}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    fields = dict(re.findall(r"^\s+(traffic_bytes_per_launch|traffic_bytes_per_unit|workload|sources|sources_sha256): "
                             r"(.+)$", text, re.M))
    if fields.get("workload") != workload_name or "sources" not in fields:
        return None
    h = hashlib.sha256()
    for src in fields["sources"].split():
        fp = os.path.join(ROOT, src)
        if not os.path.exists(fp):
            return None
        h.update(open(fp, "rb").read())
    if h.hexdigest() != fields.get("sources_sha256"):
        return None
    if "traffic_bytes_per_launch" in fields:
        return float(fields["traffic_bytes_per_launch"])
    if "traffic_bytes_per_unit" in fields and units_per_launch:
        return float(fields["traffic_bytes_per_unit"]) * units_per_launch
    return None


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            return float(d["hbm_gbs"]), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback"


# --------------------------------------------------------------------------- #
# distributed plumbing (timing only)
# --------------------------------------------------------------------------- #
def dist_setup():
    import torch

    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return rank, ws, local


def max_over_ranks(value: float, ws: int, device=None) -> float:
    if ws <= 1:
        return value
    import torch
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(value: float, ws: int, device=None) -> float:
    if ws <= 1:
        return value
    import torch
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist

        dist.barrier()


# --------------------------------------------------------------------------- #
# clocks
# --------------------------------------------------------------------------- #
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        # raw samples: a temporary file unless RSSM_BENCH_OUT names a folder to keep them in
        out_dir = os.environ.get("RSSM_BENCH_OUT") or tempfile.gettempdir()
        self.path = os.path.join(out_dir, f"rssm_clocks_gpu{gpu_index}_{os.getpid()}.csv")
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "100", "-i", str(gpu_index)], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------------------- #
# GPU arm
# --------------------------------------------------------------------------- #
def algorithmic_bytes(wl, rows_rec, ntok_b, esz):
    """Algorithmic HBM bytes of one readout launch from its per-row records:
    S0 (+ scales) once per (row, head), the group's C rows shared by its heads,
    and y; inactive rows only write zero outputs.  (The live x rows, the ring
    term and the appends are the precompute's.)"""
    total = 0
    hpg = wl.hpg
    for (s, r, p, Tb, tok0, flags) in rows_rec:
        if (flags & 1) and Tb > 0:
            # 8-bit: 64 row scales; NVFP4 (0.5 bytes an element): 64 x 8 block scales
            per_head = 64 * 128 * esz + {1: 256, 0.5: 512}.get(esz, 0) + Tb * 256 / hpg + Tb * 128
            total += per_head * wl.nheads
        elif Tb > 0:
            total += Tb * 128 * wl.nheads
    return total


def fused_bytes(wl, rows_rec, esz):
    """Algorithmic HBM bytes of one readout-with-fold launch (the main half of
    rssm_flush_step) from its per-row records (s, r, p, Tb, tok0, flags,
    epoch, gs), per (row, head): S0 (+ scales) read once if the row is read out or
    folded; for a folded row the new S0 (+ scales) written and its live x rows
    and (the group's share of) B rows read; for a row read out the group's
    share of its C rows and y written; rows without outputs write zero y.
    (dt', the replay terms and the ring appends are the precompute's.)"""
    total = 0
    hpg = wl.hpg
    s0 = 64 * 128 * esz + (256 if esz == 1 else 0)
    for (s, r, p, Tb, tok0, flags, ep, gs) in rows_rec:
        out_ok, fo = (flags & 1) and Tb > 0, flags & 2
        p_old = p  # the prefix a fold folds is the live prefix the outputs replay
        per_head = 0
        if out_ok or fo:
            per_head += s0
        if fo:
            per_head += s0 + p_old * 128 + p_old * 256 / hpg
        if out_ok:
            per_head += Tb * 256 / hpg + Tb * 128
        elif Tb > 0:
            per_head += Tb * 128
        total += per_head * wl.nheads
    return total


def flush_bytes(wl, recs, esz):
    """Algorithmic bytes of one fold launch: S0 read + write (+ scales), live x
    and B rows per flagged (row, head); with a separate read checkpoint also
    its 8-bit codes and row scales written."""
    total = 0
    rd = 0
    if wl.read_dtype == W.NVFP4:
        rd = 64 * 128 // 2 + 512
    elif wl.read_dtype is not None:
        rd = 64 * 128 + 256
    for p in recs:
        total += wl.nheads * (2 * 64 * 128 * esz + (512 if esz == 1 else 0) + p * 128 + p * 256 / wl.hpg + p * 4
                              + rd)
    return total


def run_gpu(args, rank, ws, local):
    import torch

    from speculative_state_replay_gb300 import api, build

    build.build()
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    wl = workload(args)
    gen = W.Generator(wl)
    A, D, dt_bias = gen.params()
    ids = gen.slot_idx()
    esz = W.DTYPE_BYTES[wl.state_dtype]
    # the readout streams the read checkpoint when there is one
    read_esz = esz if wl.read_dtype is None else W.DTYPE_BYTES[wl.read_dtype]

    gc = api.RssmCache(wl.num_slots, wl.nheads, wl.ngroups, wl.max_window, wl.npredicted, wl.state_dtype,
                       wl.rounding, device=dev, slot_pad_bytes=wl.slot_pad_bytes, read_dtype=wl.read_dtype)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
    active = ids[ids > 0]
    chunk = 16
    for i in range(0, active.size, chunk):
        sl = active[i:i + chunk]
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

    gA, gD, gb, gids = t(A), t(D), t(dt_bias), t(ids)
    pnat = t(pnat0)
    nsteps = args.warmup + args.steps
    host = [gen.step(k) for k in range(nsteps)]
    max_tok = max(i.ntok for i in host)
    # fixed device input buffers: each step's inputs are copied in before its
    # timed region (the kernels read them from HBM, as in a graph-replayed decode)
    # one allocation holding every per-step input (256-byte aligned regions), so
    # a step's inputs move host -> device in a single copy
    shapes = dict(x=((max_tok, wl.nheads, 64), torch.int16), dt=((max_tok, wl.nheads), torch.float32),
                  B=((max_tok, wl.ngroups, 128), torch.int16), C=((max_tok, wl.ngroups, 128), torch.int16),
                  acc=((ids.size,), torch.int32))
    fused = args.path == "fused"
    if wl.varlen:
        shapes["cu"] = ((ids.size + 1,), torch.int32)
        if not fused:  # the sequence bounds of the acceptance the step's rssm_accept_flush applies
            shapes["pcu"] = ((ids.size + 1,), torch.int32)
    esize = {torch.int16: 2, torch.int32: 4, torch.float32: 4}
    offs, total = {}, 0
    for key, (shp, dtp) in shapes.items():
        offs[key] = total
        total += (int(np.prod(shp)) * esize[dtp] + 255) // 256 * 256

    def views(raw):
        v = {key: raw[offs[key]: offs[key] + int(np.prod(shp)) * esize[dtp]].view(dtp).view(shp)
             for key, (shp, dtp) in shapes.items()}
        v.setdefault("cu", None)
        v.setdefault("pcu", None)
        return v

    dbuf = torch.zeros(total, dtype=torch.uint8, device=dev)
    buf = views(dbuf)
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a))  # noqa: E731  (host copies of the inputs)
    # the acceptance a step's launches apply: with --path fused this step's
    # (rssm_accept after the step); otherwise the previous step's, applied by
    # this step's rssm_accept_flush (none before the first step, and none under
    # --full-window, whose rows fold exactly max_window tokens)
    hin = []
    for k, i in enumerate(host):
        if fused:
            acc, pcu = i.accepted, None
        else:
            prev = host[k - 1] if k > 0 and not args.full_window else None
            acc = prev.accepted if prev is not None else np.zeros_like(i.accepted)
            pcu = None if i.cu_seqlens is None else (prev.cu_seqlens if prev is not None else i.cu_seqlens)
        hin.append(dict(x=pin(i.x.view(np.int16)), dt=pin(i.dt), B=pin(i.B.view(np.int16)), C=pin(i.C.view(np.int16)),
                        acc=pin(acc), cu=None if i.cu_seqlens is None else pin(i.cu_seqlens),
                        pcu=None if pcu is None else pin(pcu), ntok=i.ntok))
    dev_inp = [{k: (v.to(dev) if torch.is_tensor(v) else v) for k, v in hi.items()} for hi in hin]
    out = torch.zeros((max_tok, wl.nheads, 64), dtype=torch.int16, device=dev)
    scr_flush = api.alloc_scratch(gc, ids.size, wl.T)
    scr_step = api.alloc_scratch(gc, ids.size, wl.T)
    l2 = torch.empty(1 << 30, dtype=torch.uint8, device=dev)
    l2r = torch.ones(1 << 27, dtype=torch.int32, device=dev)

    def cold_l2():
        """Write 1 GiB, then read 512 MiB: afterwards the L2 holds neither step
        data nor dirty lines whose write-back the next step would pay for."""
        l2.zero_()
        l2r.max()

    force = 1 if (args.force_flush or args.full_window) else 0
    full_p = min(wl.max_window, wl.L - wl.T)  # a full window that still leaves room for the step's tokens

    def refill():
        """Full-window runs: every active row gets pnat = max_window live tokens
        (the rings hold earlier appends); untimed."""
        if args.full_window:
            pnat.masked_fill_(gids > 0, full_p)
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    cu = buf["cu"]

    def load_inputs(src, non_blocking=False):
        n = src["ntok"]
        for key in ("x", "dt", "B", "C"):
            buf[key][:n].copy_(src[key], non_blocking=non_blocking)
        buf["acc"].copy_(src["acc"], non_blocking=non_blocking)
        if cu is not None:
            cu.copy_(src["cu"], non_blocking=non_blocking)
        if buf["pcu"] is not None:
            buf["pcu"].copy_(src["pcu"], non_blocking=non_blocking)

    def step_groups(bv, yv):
        """The launch groups of one step on input buffers `bv` and output `yv`."""
        cuv = bv["cu"]

        def g_flush():
            api.rssm_accept_flush(gc, gA, gids, pnat, bv["acc"], wl.T, wl.T, scr_flush, accept_cu_seqlens=bv["pcu"],
                                  cu_seqlens=cuv, force=force, seed=wl.sr_seed)

        def g_pre():
            api.rssm_step_precompute(gc, bv["x"], bv["dt"], gA, bv["B"], bv["C"], gD, gb, gids, pnat, wl.T, yv,
                                     scr_step, cu_seqlens=cuv)

        def g_read():
            api.rssm_step_readout(gc, bv["x"], bv["dt"], gA, bv["B"], bv["C"], gD, gb, gids, pnat, wl.T, yv,
                                  scr_step, cu_seqlens=cuv)

        def g_acc():
            api.rssm_accept(gc, gids, pnat, bv["acc"], wl.T, cu_seqlens=cuv)

        def g_fpre():
            api.rssm_flush_step_classify(gc, bv["x"], bv["dt"], gA, bv["B"], bv["C"], gD, gb, gids, pnat, wl.T, yv,
                                         scr_step, cu_seqlens=cuv, force=force, seed=wl.sr_seed)

        def g_fread():
            api.rssm_flush_step_main(gc, bv["x"], bv["dt"], gA, bv["B"], bv["C"], gD, gb, gids, pnat, wl.T, yv,
                                     scr_step, cu_seqlens=cuv, force=force, seed=wl.sr_seed)

        return [g_fpre, g_fread, g_acc] if fused else [g_flush, g_pre, g_read]

    # the launch groups of one step; `rg` is the dominant kernel's group
    groups = step_groups(buf, out)
    if fused:
        names, rg = ["precompute", "readout_fold", "accept"], 1
    else:
        names, rg = ["accept_flush", "precompute", "readout"], 2
    # a second set of device inputs and output: the end-to-end leg alternates
    # between the two so one step's copies overlap the neighbouring steps' work
    dbuf_b = torch.zeros(total, dtype=torch.uint8, device=dev) if not args.no_e2e else None
    out_b = torch.zeros((max_tok, wl.nheads, 64), dtype=torch.int16, device=dev) if not args.no_e2e else None
    # one eager step (sets kernel attributes), then capture on a snapshot of the
    # cache that is restored afterwards so capture has no side effects
    load_inputs(dev_inp[0])
    for f in groups:
        f()
    torch.cuda.synchronize()
    graphs = []
    side = torch.cuda.Stream(device=dev)
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for f in groups:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side, capture_error_mode="thread_local"):
                f()
            graphs.append(g)
        # the whole step as one graph (kernels chained by programmatic launch)
        g_step = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_step, stream=side, capture_error_mode="thread_local"):
            for f in groups:
                f()
        g_b = None
        if dbuf_b is not None:
            g_b = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_b, stream=side, capture_error_mode="thread_local"):
                for f in step_groups(views(dbuf_b), out_b):
                    f()
        # the full-window flush leg: every active row flushed (force = 1)
        g_fw = None
        if not args.no_full_window_leg:
            g_fw = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_fw, stream=side, capture_error_mode="thread_local"):
                api.rssm_flush(gc, gA, gids, pnat, wl.T, scr_flush, cu_seqlens=cu, force=1, seed=wl.sr_seed)
    torch.cuda.synchronize()
    # restart the workload from its initial state
    for i in range(0, active.size, chunk):
        sl = active[i:i + chunk]
        api.rssm_init_state(gc, t(gen.init_states(i, sl.size)), t(sl.astype(np.int32)), seed=wl.sr_seed)
    gc.ring_start.copy_(t(gen.ring_start()))
    pnat.copy_(t(pnat0))
    if wl.prefill_live:
        for b, s in enumerate(ids):
            if s > 0:
                x, B, dtp, live = gen.ring_prefill(int(s))
                gc.x_view()[s] = t(x.view(np.int16))
                gc.B_view()[s] = t(B.view(np.int16))
                gc.dt_view()[s] = t(dtp)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()

    def step_units():
        rr = scr_step[256: 256 + ids.size * 32].view(torch.int32).view(ids.size, 8).cpu().numpy()
        return rr, int((((rr[:, 5] & 1) == 1) & (rr[:, 3] > 0)).sum()) * wl.nheads

    def host_units(k):
        """(slot, head) updates of step k from its inputs: active rows with at
        least one token (what the step's row records count)."""
        tb = np.diff(host[k].cu_seqlens) if host[k].cu_seqlens is not None else np.full(ids.size, wl.T)
        return int(((ids > 0) & (tb > 0)).sum()) * wl.nheads

    for k in range(args.warmup):
        refill()
        load_inputs(dev_inp[k])
        cold_l2()
        g_step.replay()
    torch.cuda.synchronize()

    # timed pass 1: whole steps (one graph each) -> value
    step_ms, units = [], 0
    barrier(ws)
    torch.cuda.synchronize()
    # clocks are sampled across every timed leg (whole steps, per-kernel pass,
    # end to end, full-window flush)
    clocks = ClockSampler(torch.cuda.current_device())
    for k in range(args.warmup, nsteps):
        refill()
        load_inputs(dev_inp[k])
        cold_l2()
        e0 = ev()
        e0.record(stream)
        g_step.replay()
        e1 = ev()
        e1.record(stream)
        torch.cuda.synchronize()
        step_ms.append(e0.elapsed_time(e1))
        u_dev = step_units()[1]
        if u_dev != host_units(k):
            raise RuntimeError(f"step {k}: {u_dev} updates on the device, {host_units(k)} from the inputs")
        units += u_dev
    barrier(ws)
    torch.cuda.synchronize()

    # timed pass 2: the same steps launched group by group with events between
    # the groups -> per-kernel durations for the roofline
    grp_ms = [[] for _ in groups]
    read_bytes, fold_bytes, fold_units = 0.0, 0.0, 0
    for k in range(args.warmup, nsteps):
        refill()
        load_inputs(dev_inp[k])
        cold_l2()
        evs = [ev()]
        evs[0].record(stream)
        for g in graphs:
            g.replay()
            e = ev()
            e.record(stream)
            evs.append(e)
        torch.cuda.synchronize()
        for j in range(len(groups)):
            grp_ms[j].append(evs[j].elapsed_time(evs[j + 1]))
        rr, _ = step_units()
        if fused:
            read_bytes += fused_bytes(wl, [tuple(int(v) for v in r) for r in rr], esz)
            fold_units += int(((rr[:, 5] & 2) != 0).sum()) * wl.nheads
        else:
            read_bytes += algorithmic_bytes(wl, [tuple(r[:6]) for r in rr], None, read_esz)
            cnt = int(scr_flush[4:8].view(torch.int32).item())
            recs = (scr_flush[256: 256 + cnt * 32].view(torch.int32).view(cnt, 8).cpu().numpy() if cnt
                    else np.zeros((0, 8)))
            fold_bytes += flush_bytes(wl, [int(r[3]) for r in recs], esz)
            fold_units += cnt * wl.nheads
    read_ms = grp_ms[rg]
    flush_ms = grp_ms[0] if not fused else []
    torch.cuda.synchronize()
    err = int(gc.error_word.item())
    if err:
        raise RuntimeError(f"device error bits set: {err:#x}")

    total_ms = sum(step_ms)
    t_max = max_over_ranks(total_ms, ws, dev)
    units_all = sum_over_ranks(units, ws, dev)
    value = units_all / (t_max / 1e3)

    # end to end through the public calls: every step's inputs are copied in
    # from pinned host memory and its y is copied back, inside the timed region
    e2e = None
    if not args.no_e2e:
        n_e2e = nsteps - args.warmup
        # pinned staging laid out like the device inputs, filled before the
        # timed region (the host's part of a serving loop); at most 4 buffers:
        # the timed steps take the inputs of the first n_stage timed steps in turn
        n_stage = min(n_e2e, 4)
        stage = [torch.empty(total, dtype=torch.uint8, pin_memory=True) for _ in range(n_stage)]
        ks = [args.warmup + i % n_stage for i in range(n_e2e)]  # the inputs each e2e step takes
        for j in range(n_stage):
            hv, hi = views(stage[j]), hin[args.warmup + j]
            n = hi["ntok"]
            for key in ("x", "dt", "B", "C"):
                hv[key][:n].copy_(hi[key])
            hv["acc"].copy_(hi["acc"])
            if cu is not None:
                hv["cu"].copy_(hi["cu"])
            if hv["pcu"] is not None:
                hv["pcu"].copy_(hi["pcu"])
        yh = [torch.empty((max_tok, wl.nheads, 64), dtype=torch.int16, pin_memory=True) for _ in range(2)]
        e2e_units = sum(host_units(k) for k in ks)
        d2h_sum = sum(hin[k]["ntok"] for k in ks) * wl.nheads * 64 * 2

        # (a) serial: H2D copy -> step -> D2H copy of y, one step at a time
        ser_ms = []
        parts = {"h2d": [], "step": [], "d2h": []}
        for i, k in enumerate(ks):
            n = hin[k]["ntok"]
            cold_l2()
            e0 = ev()
            e0.record(stream)
            dbuf.copy_(stage[i % n_stage], non_blocking=True)
            e_h = ev()
            e_h.record(stream)
            g_step.replay()
            e_g = ev()
            e_g.record(stream)
            yh[0][:n].copy_(out[:n], non_blocking=True)
            e1 = ev()
            e1.record(stream)
            torch.cuda.synchronize()
            ser_ms.append(e0.elapsed_time(e1))
            parts["h2d"].append(e0.elapsed_time(e_h))
            parts["step"].append(e_h.elapsed_time(e_g))
            parts["d2h"].append(e_g.elapsed_time(e1))
        t_ser = max_over_ranks(sum(ser_ms), ws, dev)
        serial = {"value": sum_over_ranks(e2e_units, ws, dev) / (t_ser / 1e3), "unit": UNIT,
                  "ms_per_step": t_ser / n_e2e,
                  "breakdown_us": {key: 1e3 * statistics.median(v) for key, v in parts.items()},
                  "l2": "cleared before each step (untimed)"}

        # (b) pipelined: the steps back to back on the compute stream, alternating
        # between two device input/output sets; step k's H2D copy (copy stream)
        # overlaps step k-1's kernels and its D2H copy (a third stream) step k+1's
        dbufs, outs, gs = [dbuf, dbuf_b], [out, out_b], [g_step, g_b]
        s_h2d, s_d2h = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        sev = lambda: torch.cuda.Event()  # noqa: E731
        h_done, c_done, d_done = [sev() for _ in range(n_e2e)], [sev() for _ in range(n_e2e)], \
            [sev() for _ in range(n_e2e)]
        torch.cuda.synchronize()
        barrier(ws)
        torch.cuda.synchronize()
        e_start, e_end = ev(), ev()
        e_start.record(s_h2d)
        for i in range(n_e2e):
            k, par = ks[i], i % 2
            n = hin[k]["ntok"]
            with torch.cuda.stream(s_h2d):
                if i >= 2:
                    s_h2d.wait_event(c_done[i - 2])  # step i-2 is done with this input set
                dbufs[par].copy_(stage[i % n_stage], non_blocking=True)
                h_done[i].record(s_h2d)
            with torch.cuda.stream(stream):
                stream.wait_event(h_done[i])
                if i >= 2:
                    stream.wait_event(d_done[i - 2])  # y of step i-2 has left this output
                gs[par].replay()
                c_done[i].record(stream)
            with torch.cuda.stream(s_d2h):
                s_d2h.wait_event(c_done[i])
                yh[par][:n].copy_(outs[par][:n], non_blocking=True)
                d_done[i].record(s_d2h)
        e_end.record(s_d2h)
        torch.cuda.synchronize()
        t_e2e = max_over_ranks(e_start.elapsed_time(e_end), ws, dev)
        e2e = {"value": sum_over_ranks(e2e_units, ws, dev) / (t_e2e / 1e3), "unit": UNIT,
               "h2d_bytes_per_step": int(total), "d2h_bytes_per_step": int(d2h_sum // n_e2e),
               "ms_per_step": t_e2e / n_e2e,
               "mode": ("rssm_flush_step -> rssm_accept" if fused else "rssm_accept_flush -> rssm_step") +
                       " on a compute stream, every step's inputs copied in "
                       "from pinned host memory (one H2D copy per step) and its y copied back (one D2H copy), "
                       "copies on two other streams overlapping the neighbouring steps' kernels; two device "
                       f"input/output sets alternate; {n_stage} pinned input sets (the inputs of the first "
                       f"{n_stage} timed steps) taken in turn",
               "l2": ("not cleared (back-to-back steps); " +
                      (f"each step's readout alone streams {read_bytes / args.steps / 1e6:.0f} MB, more than the "
                       "129 MB L2" if read_bytes / args.steps > L2_BYTES else
                       f"the step's working set ({read_bytes / args.steps / 1e6:.0f} MB read by the readout) fits in "
                       "the L2, so this leg runs warm")),
               "serial": serial}

    # full-window flush: every active row holds a full window of live tokens
    # (pnat set outside the events; the rings hold earlier appends) and flushes
    fw = None
    if g_fw is not None:
        fw_ms, fw_bytes, fw_units = [], 0.0, 0
        for r in range(args.full_window_reps):
            pnat.masked_fill_(gids > 0, full_p)
            cold_l2()
            e0 = ev()
            e0.record(stream)
            g_fw.replay()
            e1 = ev()
            e1.record(stream)
            torch.cuda.synchronize()
            fw_ms.append(e0.elapsed_time(e1))
            cnt = int(scr_flush[4:8].view(torch.int32).item())
            recs = (scr_flush[256: 256 + cnt * 32].view(torch.int32).view(cnt, 8).cpu().numpy() if cnt
                    else np.zeros((0, 8)))
            fw_bytes += flush_bytes(wl, [int(v[3]) for v in recs], esz)
            fw_units += cnt * wl.nheads
        fw = dict(ms=fw_ms, bytes=fw_bytes, units=fw_units)
    clk = clocks.stop()
    err = int(gc.error_word.item())
    if err:
        raise RuntimeError(f"device error bits set: {err:#x}")

    peak, peak_kind = measured_peaks()
    achieved = read_bytes / (sum(read_ms) / 1e3) / 1e9
    fold_achieved = fold_bytes / (sum(flush_ms) / 1e3) / 1e9 if sum(flush_ms) > 0 else 0.0
    flush_roofline = None
    if not fused:
        flush_roofline = {"bound": "hbm", "kernel": "flush_kernel (rssm_accept_flush)", "achieved": fold_achieved,
                          "peak": peak, "unit": "GB/s", "frac": fold_achieved / peak,
                          "avg_us": 1e3 * statistics.mean(flush_ms),
                          "algorithmic_bytes_per_step": fold_bytes / args.steps}
    fw_roofline = None
    if fw is not None:
        fw_achieved = fw["bytes"] / (sum(fw["ms"]) / 1e3) / 1e9
        fw_roofline = {"bound": "hbm", "kernel": "flush_kernel", "achieved": fw_achieved, "peak": peak,
                       "unit": "GB/s", "frac": fw_achieved / peak, "avg_us": 1e3 * statistics.mean(fw["ms"]),
                       "launches": len(fw["ms"]), "live_tokens_per_row": full_p,
                       "units_per_launch": fw["units"] / len(fw["ms"]),
                       "algorithmic_bytes_per_launch": fw["bytes"] / len(fw["ms"]),
                       "mode": "rssm_flush with force = 1 after every active row's pnat is set to max_window "
                               "(outside the events), one CUDA graph per launch, cold L2"}
    units_per_read = sum(host_units(k) for k in range(args.warmup, nsteps)) / args.steps
    res = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": t_max / args.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": dict(wl.describe(), parallelism=f"replicas{ws}", l2="1 GiB written then 512 MiB read between steps (cold, clean L2)",
                       launch="one CUDA graph per step (kernels chained by programmatic dependent launch); kernel times from a second pass with one graph per launch group",
                       force_flush=bool(args.force_flush or args.full_window),
                       full_window=bool(args.full_window), path=args.path),
        "roofline": {"bound": "hbm", "kernel": "readout_kernel (fold variant)" if fused else "readout_kernel",
                     "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": None if fused or args.batch is not None else profiled_traffic(
                         "readout_kernel", wl.name, units_per_read),
                     "traffic_unit": "bytes per launch (ncu dram__bytes_read.sum + dram__bytes_write.sum)",
                     "peak_source": peak_kind, "avg_launch_us": 1e3 * statistics.mean(read_ms),
                     "algorithmic_bytes_per_launch": read_bytes / args.steps,
                     "folded_units_per_launch": fold_units / args.steps},
        "flush_roofline": flush_roofline,
        "flush_roofline_full_window": fw_roofline,
        "e2e": e2e,
        # per timed step: precompute, readout with fold, accept (split: accept + flush, precompute, readout)
        "gpu_launches": 3 * args.steps,
        "clocks": clk,
        "device_time_ms": dict({"step": statistics.mean(step_ms)},
                               **{n: statistics.mean(v) for n, v in zip(names, grp_ms)}),
    }
    return res, wl


# --------------------------------------------------------------------------- #
# CPU oracle (baseline leg and reference arm)
# --------------------------------------------------------------------------- #
class OracleRun:
    """The oracle as it stands on the workload, restricted to the first `rows`
    rows (rows are independent); one decode step = flush + step + accept."""

    def __init__(self, wl, rows=None):
        import oracle

        oracle.build()
        self.oracle, self.wl = oracle, wl
        self.gen = W.Generator(wl)
        self.A, self.D, self.dtb = self.gen.params()
        ids = self.gen.slot_idx()
        self.ids = ids[:rows] if rows is not None and rows < ids.size else ids
        self.oc = oracle.OracleCache(wl.num_slots, wl.nheads, wl.ngroups, wl.max_window, wl.npredicted,
                                     wl.state_dtype, wl.rounding, slot_pad_bytes=wl.slot_pad_bytes,
                                     read_dtype=wl.read_dtype)
        act = self.ids[self.ids > 0]
        self.oc.init_state(self.gen.init_states(0, act.size), act, seed=wl.sr_seed)
        self.pnat = np.zeros(self.ids.size, np.int32)
        if wl.prefill_live:  # prefilled rings, as the GPU run starts
            for b, s in enumerate(self.ids):
                if s > 0:
                    x, B, dtp, live = self.gen.ring_prefill(int(s))
                    self.oc.x_view()[s] = x
                    self.oc.B_view()[s] = B
                    self.oc.dt_view()[s] = dtp
                    self.pnat[b] = live
        self.oc.ring_start[:] = self.gen.ring_start()
        self.k = 0

    def step(self):
        """Runs one decode step; returns (units, seconds)."""
        wl, ids, T = self.wl, self.ids, self.wl.T
        inp = self.gen.step(self.k)
        self.k += 1
        if inp.cu_seqlens is None:
            tok, cu = np.arange(ids.size * T), None
        else:
            cu = inp.cu_seqlens[: ids.size + 1].copy()
            tok = np.arange(int(cu[-1]))
        x, dt, B, C = inp.x[tok], inp.dt[tok], inp.B[tok], inp.C[tok]
        t0 = time.perf_counter()
        self.oc.flush(self.A, ids, self.pnat, T, cu_seqlens=cu, seed=wl.sr_seed)
        self.oc.step(x, dt, self.A, B, C, self.D, self.dtb, ids, self.pnat, T, cu_seqlens=cu)
        self.oc.accept(ids, self.pnat, inp.accepted[: ids.size], T, cu_seqlens=cu)
        return int((ids > 0).sum()) * wl.nheads, time.perf_counter() - t0

    @property
    def threads(self):
        return self.oracle.openmp_threads() or 1


def cpu_baseline(wl, seconds):
    run = OracleRun(wl, rows=min(wl.batch, 128))
    units, secs, steps = 0, 0.0, 0
    while secs < seconds and steps < 64:
        u, dt = run.step()
        units, secs, steps = units + u, secs + dt, steps + 1
    return {"value": units / secs, "unit": UNIT, "cores": run.threads, "kind": "oracle",
            "sample": f"{steps} consecutive decode steps x {run.ids.size} rows x {wl.nheads} heads of {wl.name} "
                      f"(flush+step+accept, {secs:.1f} s of CPU wall time, OpenMP over (row, head))"}


def run_reference(args, rank, ws):
    if rank != 0:
        return None
    wl = workload(args)
    run = OracleRun(wl, rows=min(16, wl.batch))
    vals = []
    for k in range(args.warmup + args.steps):
        u, secs = run.step()
        if k >= args.warmup:
            vals.append((u, secs))
    value = sum(u for u, _ in vals) / sum(s for _, s in vals)
    sample = (f"each step: one decode step (flush+step+accept) of the first {run.ids.size} rows x {wl.nheads} heads "
              f"of {wl.name} on the CPU oracle, consecutive steps on one cache")
    cb = {"value": value, "unit": UNIT, "cores": run.threads, "kind": "oracle", "sample": sample}
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * statistics.mean(s for _, s in vals),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": dict(wl.describe(), parallelism=f"replicas{ws}"), "cpu_baseline": cb,
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    args = parse()
    rank, ws, local = dist_setup()
    if args.impl == "reference":
        res = run_reference(args, rank, ws)
        if rank == 0:
            print(json.dumps(res))
        return
    res, wl = run_gpu(args, rank, ws, local)
    if rank == 0:
        if not args.no_cpu_baseline and ws == 1:
            res["cpu_baseline"] = cpu_baseline(wl, args.cpu_seconds)
        else:
            res["cpu_baseline"] = None
        print(json.dumps(res))


if __name__ == "__main__":
    main()
