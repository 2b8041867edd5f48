"""Parity rules between the CUDA path and the oracle (test infrastructure).

* Index sets: bit-exact, except that a block may differ when the oracle's
  score of it lies within TIE_WINDOW of the oracle's K_b-th score (the
  selection boundary), i.e. where the K_b-th and (K_b+1)-th scores are
  closer than the window.
* Compressed keys / query prep / attention output (bf16): |gpu - oracle| <=
  ATOL + RTOL * |oracle|.
* e4m3 values: the oracle rounds a float64 value once, the kernel an fp32
  value once; the two unrounded values differ by ~1e-6 relative, so a code
  can differ only when the value sits within that distance of a rounding
  midpoint: at most one e4m3 step apart, and on a tiny fraction of entries.
"""

from __future__ import annotations

import numpy as np

from oracle import qsa_oracle as O

TIE_WINDOW = 1e-3
ATOL = 2e-2
RTOL = 1e-2
E4M3_FLIP_FRACTION = 1e-3


def close_bf16(got, want, atol=ATOL, rtol=RTOL):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    err = np.abs(got - want)
    ok = err <= atol + rtol * np.abs(want)
    return bool(ok.all()), float(err.max(initial=0.0))


def close_e4m3(got, want):
    """At most one e4m3 step apart everywhere, and rarely apart at all."""
    got = np.asarray(got, dtype=np.float64).ravel()
    want = np.asarray(want, dtype=np.float64).ravel()
    table = O.e4m3_decode_table()
    vals = np.unique(table[~np.isnan(table)])
    ig = np.searchsorted(vals, got)
    iw = np.searchsorted(vals, want)
    if not (np.isin(got, vals).all() and np.isin(want, vals).all()):
        return False, 1.0
    steps = np.abs(ig - iw)
    frac = float((steps > 0).mean()) if len(steps) else 0.0
    return bool(steps.max(initial=0) <= 1 and frac <= E4M3_FLIP_FRACTION), frac


def selection_ok(cfg: O.QsaConfig, gpu_row, oracle_row, oracle_scores, p: int):
    """Compare a packed selection row of the CUDA path with the oracle's.

    Returns (ok, number of differing blocks)."""
    gpu_row = np.asarray(gpu_row)
    oracle_row = np.asarray(oracle_row)
    n = int(oracle_row[-1])
    if int(gpu_row[-1]) != n:
        return False, -1
    if not (gpu_row[n:-1] == -1).all():
        return False, -1
    g = set(gpu_row[:n].tolist())
    o = set(oracle_row[:n].tolist())
    if len(g) != n:
        return False, -1
    if g == o:
        return True, 0
    r = cfg.compress_ratio
    V = O.visible_blocks(p, r)
    gb = {t // r for t in g if t < V * r}
    ob = {t // r for t in o if t < V * r}
    if {t for t in g if t >= V * r} != {t for t in o if t >= V * r}:
        return False, -1
    diff = gb ^ ob
    s = np.asarray(oracle_scores, dtype=np.float64)
    kth = np.sort(s)[::-1][cfg.block_topk - 1]
    ok = all(abs(s[b] - kth) <= TIE_WINDOW for b in diff if 0 <= b < V)
    return ok, len(diff)
