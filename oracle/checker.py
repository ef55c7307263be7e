"""Parity checker: indexer ids against the oracle, modulo score ties.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

The GPU path computes page scores S' in fp32 with |S' - S| <= eps = RTOL * A
(S exact, A = max_t sum_d |q_d k_td|; RTOL = 1e-5) and then selects exactly
under S'.  An id row is therefore accepted iff it is the exact top-m of SOME
score vector inside that band.  That gives, per (row, head), with
m = min(15, L):
  1. structure: ids[:m] are distinct history pages (0 <= id < L), ids[m] is
     the local page L, ids[m+1:] are -1; a row with no valid page is all -1;
  2. order: consecutive ranked ids satisfy S[a] + eps[a] >= S[b] - eps[b];
  3. boundary: every selected id beats every unselected history page up to
     the band: min_sel (S + eps) >= max_unsel (S - eps).
With no scores within the band of each other this is bit-exact equality with
the oracle's ids; the report counts rows that differ at all.
Rows of a request with an unreadable page must be all -1 (the GPU also
raises its status flag).
"""
from __future__ import annotations

import numpy as np

RTOL = 1e-5
TOPK = 16
HIST_TOPK = 15


def check_ids(gpu_out: np.ndarray, ref, rtol: float = RTOL, max_report: int = 8) -> dict:
    gpu_out = np.asarray(gpu_out)
    rows, H, k = gpu_out.shape
    assert k == TOPK and rows == ref.out.shape[0] and H == ref.out.shape[1]
    fails = []
    n_diff = 0
    for r in range(rows):
        Lr = int(ref.L[r])
        for h in range(H):
            g = gpu_out[r, h]
            if not np.array_equal(g, ref.out[r, h]):
                n_diff += 1
            if ref.bad[r] or Lr < 0:
                if np.any(g != -1):
                    fails.append((r, h, "expected all -1", g.tolist()))
                continue
            m = min(HIST_TOPK, Lr)
            sel = g[:m]
            if g[m] != Lr or np.any(g[m + 1:] != -1):
                fails.append((r, h, f"local page {Lr} / -1 tail", g.tolist()))
                continue
            if np.any(sel < 0) or np.any(sel >= Lr) or len(set(sel.tolist())) != m:
                fails.append((r, h, "ids not distinct history pages", g.tolist()))
                continue
            S = ref.S[r, h, :Lr]
            eps = rtol * ref.A[r, h, :Lr]
            ss, es = S[sel], eps[sel]
            if m > 1 and np.any(ss[:-1] + es[:-1] < ss[1:] - es[1:]):
                fails.append((r, h, "ranked ids out of score order", g.tolist()))
                continue
            if m < Lr:
                mask = np.ones(Lr, dtype=bool)
                mask[sel] = False
                worst_sel = np.min(ss + es)
                best_uns = np.max(S[mask] - eps[mask])
                if worst_sel < best_uns:
                    fails.append((r, h, f"unselected page beats a selected one "
                                        f"({best_uns:.6g} > {worst_sel:.6g})", g.tolist()))
    return dict(rows=rows * H, differ=n_diff, fails=len(fails), examples=fails[:max_report])


def check_scores(gpu_scores: np.ndarray, ref, rtol: float = RTOL) -> dict:
    """Debug scores: |S_gpu - S| <= rtol * A on every history page."""
    gpu_scores = np.asarray(gpu_scores, dtype=np.float64)
    W = ref.S.shape[2]
    g = gpu_scores[:, :, :W]
    valid = ~np.isnan(ref.S)
    err = np.abs(g - np.nan_to_num(ref.S))
    lim = rtol * np.nan_to_num(ref.A)
    bad = valid & ~(err <= lim)
    rel = np.where(valid & (ref.A > 0), err / np.where(ref.A > 0, ref.A, 1), 0)
    return dict(checked=int(valid.sum()), fails=int(bad.sum()),
                max_rel_err=float(np.nanmax(rel)) if valid.any() else 0.0)
