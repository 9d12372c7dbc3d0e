"""Golden fixtures taken from statements on the pages (CPU only)."""
import os

import numpy as np
import pytest

from speculative_state_replay_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _cases():
    out = []
    for line in open(os.path.join(GOLDEN, "ring_contract.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        head, live, app, flush = [p.strip() for p in line.split("|")]
        Wn, npred, r, p, T = map(int, head.split())
        live = [] if live == "-" else list(map(int, live.split()))
        out.append((Wn, npred, r, p, T, live, list(map(int, app.split())), int(flush)))
    return out


@pytest.mark.parametrize("case", _cases())
def test_ring_contract_positions_and_flush_rule(orc, case):
    Wn, npred, r, p, T, live, app, flush = case
    L = Wn + npred
    assert len(live) == p and len(app) == T
    c = orc.OracleCache(3, 2, 1, Wn, npred, W.F32)
    rng = np.random.default_rng(0)
    c.state_view()[1] = rng.standard_normal((2, 64, 128)).astype(np.float32)
    c.ring_start[1] = r
    # distinctive ring contents: position pos holds the value 1 + pos / 64 everywhere
    for pos in range(L):
        c.x_view()[1, :, pos] = ((np.float32(1 + pos / 64)).view(np.uint32) >> 16)
        c.B_view()[1, :, pos] = ((np.float32(0.1)).view(np.uint32) >> 16)
        c.dt_view()[1, :, pos] = 0.05
    ids = np.array([1], np.int32)
    A, D, dtb = np.float32([-1.0, -2.0]), np.float32([0.5, 0.5]), np.float32([0.0, 0.0])
    x = np.full((T, 2, 64), 0x4100, np.uint16)  # 8.0
    x += np.arange(T, dtype=np.uint16)[:, None, None]
    Bn = np.full((T, 1, 128), 0x3DCC, np.uint16)
    C = np.full((T, 1, 128), 0x3DCC, np.uint16)
    dt = np.full((T, 2), -2.0, np.float32)

    def y_of(cache, pn):
        return cache.copy().step(x, dt, A, Bn, C, D, dtb, ids, np.array([pn], np.int32), T)

    # only the listed live positions enter the output (a step without a flush
    # needs p + T <= L)
    base = y_of(c, p)
    for pos in range(L if p + T <= L else 0):
        d = c.copy()
        d.x_view()[1, :, pos] = 0x4200  # 32.0
        changed = not np.array_equal(y_of(d, p), base)
        assert changed == (pos in live), pos
    # appends land at the listed positions
    pn = np.array([p], np.int32)
    e = c.copy()
    e.flush(A, ids, pn, T)
    assert int(e.flush_epoch[1]) == flush
    e.step(x, dt, A, Bn, C, D, dtb, ids, pn, T)
    for i, pos in enumerate(app):
        assert (e.x_view()[1, :, pos] == 0x4100 + i).all()
