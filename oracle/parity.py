"""Comparison rules between the GPU library and the oracle (test infrastructure only).

Acceptance (the method's own tolerance statement for this build):
* index sets (R, C, P and each step's selection) must match exactly, except for
  channels whose oracle score lies within FLAG_REL (1e-4) relative of the
  cut-off score; those are flagged and counted, not failed;
* FFN outputs: relative L2 error <= 5e-3 and max abs error <= 2e-2 against the
  oracle on the same bf16 inputs. Every output is held to this, the prefill's
  included. When a flagged near-tie went the other way, the GPU's output is
  checked against the FFN over the set the GPU kept (``y_on_set``), so that no
  step goes unchecked.
"""
from __future__ import annotations

import numpy as np

from . import down_projection, ffn_activations

FLAG_REL = 1e-4
Y_REL_L2 = 5e-3
Y_MAX_ABS = 2e-2


def rel_l2(a, ref) -> float:
    a = np.asarray(a, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(a - ref) / (den if den > 0 else 1.0))


def max_abs(a, ref) -> float:
    a = np.asarray(a, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.max(np.abs(a - ref))) if a.size else 0.0


def check_y(y, y_ref, what="y"):
    e2, ea = rel_l2(y, y_ref), max_abs(y, y_ref)
    assert e2 <= Y_REL_L2 and ea <= Y_MAX_ABS, \
        f"{what}: rel-L2 {e2:.3e} (<= {Y_REL_L2}), max-abs {ea:.3e} (<= {Y_MAX_ABS})"
    return e2, ea


def near_cutoff(scores, cut_values, rel=FLAG_REL) -> np.ndarray:
    """Boolean mask of entries whose score is within `rel` relative of any cut-off value."""
    s = np.asarray(scores, dtype=np.float64)
    m = np.zeros(s.shape, dtype=bool)
    for v in cut_values:
        m |= np.abs(s - v) <= rel * max(abs(v), 1e-30)
    return m


def partition_cut_values(I, counts):
    """Oracle importance values at the two cut-offs (the n_P-th smallest and the n_R-th largest)."""
    I = np.asarray(I, dtype=np.float64)
    order = np.sort(I)
    cuts = []
    if counts.n_P > 0:
        cuts.append(order[counts.n_P - 1])
    if counts.n_R > 0:
        cuts.append(order[len(I) - counts.n_R])
    return cuts


def compare_partition(gpu, ref, I_ref, counts):
    """(unflagged mismatching channels, flagged count, differing count); gpu/ref are (R, C, P)."""
    N = len(I_ref)
    cls_g = np.full(N, -1)
    cls_r = np.full(N, -1)
    for c, (a, b) in enumerate(zip(gpu, ref)):
        cls_g[np.asarray(a, dtype=np.int64)] = c
        cls_r[np.asarray(b, dtype=np.int64)] = c
    flagged = near_cutoff(I_ref, partition_cut_values(I_ref, counts))
    bad = np.nonzero((cls_g != cls_r) & ~flagged)[0]
    return bad, int(flagged.sum()), int(np.sum(cls_g != cls_r))


def selection_cut_value(scores, k):
    s = np.sort(np.asarray(scores, dtype=np.float64))[::-1]
    return [s[k - 1]] if 0 < k <= len(s) else []


def compare_selection(S_gpu, S_ref, C, scores_ref, k):
    """Selected channel sets: (unflagged differences, flagged count, differing count)."""
    S_gpu = set(np.asarray(S_gpu).tolist())
    S_ref = set(np.asarray(S_ref).tolist())
    diff = sorted(S_gpu ^ S_ref)
    flagged = near_cutoff(scores_ref, selection_cut_value(scores_ref, k))
    pos = {ch: p for p, ch in enumerate(np.asarray(C).tolist())}
    bad = [ch for ch in diff if ch not in pos or not flagged[pos[ch]]]
    return bad, int(flagged.sum()), len(diff)


def y_on_set(Wg, W1, W2, channels, x):
    """The FFN output over a fixed kept set of channels ("Overall framework": the final FFN runs
    on R plus the selected candidates), for a step whose set differs from the oracle's own only
    by flagged near-ties."""
    keep = np.sort(np.asarray(channels, dtype=np.int64))
    Z = ffn_activations(Wg[keep], W1[keep], x)
    return down_projection(W2[:, keep], Z)
