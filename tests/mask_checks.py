"""Checks of one predicted mask row against the float64 oracle when the GPU's rounding may move
its top-k cut.  Test helpers only (no GPU needed; the CPU tests in test_mask_checks.py plant
mistakes in oracle rows and check that these helpers catch them).

The slack is derived from the arithmetic of the library's pooled scores, not fitted:

- scores: each block mean is split into bf16 hi + lo parts and S = scale (hi.hi + hi.lo + lo.hi)
  is accumulated in fp32 on the tensor cores.  hi keeps 8 significant bits of a mean and lo 8 of
  what is left, so per element the dropped lo.lo term and the residual of the split are below
  2^-16 |muq_e muk_e|; the score of block j is off by at most
  E_j = 2^-16 scale sum_e |muq_e| |muk_e|  (+ 2^-22 |S_j| for the fp32 accumulation);
- probabilities: p_j = exp(S_j - logZ) moves by a factor exp(delta_j - delta_logZ) with
  |delta_logZ| <= max_j E_j, so its relative error is below eps_rel = 2 max_j E_j + 2^-20 (the
  fp32 exponential);
- cumulative mass: a prefix sum of those probabilities is off by at most eps_rel of itself
  plus its fp32 summation error (a lane sums at most 64 values in sequence and the lanes and
  bins are combined in trees: under 80 roundings of 2^-24), eps_mass = eps_rel + 1e-5;
- similarities: fp32 sums of 128 or 64 unit vectors, eps_sim = 1e-5.

The GPU tests check the first and last of these directly on the rows they sample (the
library's S, sQ and sK from its workspace against the oracle's)."""
from __future__ import annotations

import numpy as np

import oracle

SPLIT_REL = 2.0 ** -16   # bf16 hi/lo split of the pooled means
ACC_REL = 2.0 ** -22     # fp32 accumulation of a score
EXP_REL = 2.0 ** -20     # fp32 exponential
SUM_ABS = 1e-5           # fp32 summation of a row's probabilities
EPS_SIM = 1e-5           # fp32 similarity


def score_error_bound(muq: np.ndarray, muk: np.ndarray, S: np.ndarray, valid: np.ndarray, scale: float) -> np.ndarray:
    """Per-block bound E_j of |S_gpu - S| for one row: muq (d,), muk (nkb, d), S (nkb,) the
    oracle's scaled scores; 0 on invalid blocks."""
    E = SPLIT_REL * scale * (np.abs(muk) @ np.abs(muq)) + ACC_REL * np.where(valid, np.abs(S), 0.0)
    return np.where(valid, E, 0.0)


def slack(E: np.ndarray):
    """(eps_rel, eps_mass) from the per-block score bounds of a row."""
    eps_rel = 2.0 * float(E.max(initial=0.0)) + EXP_REL
    return eps_rel, eps_rel + SUM_ABS


def decisive(pr, topk: float, theta: float, eps_rel: float, eps_mass: float, eps_sim: float = EPS_SIM,
             mode: str = "cdf") -> bool:
    """Whether no rounding within the slack can change the row: pr is an oracle
    predict_mask_row result.  The similarities must be farther than eps_sim from theta (a row
    with s_Q below theta keeps all its blocks and is then decisive); the probabilities at the
    cut must differ by more than eps_rel of their sum, and (cumulative reading) the mass through
    the cut and through the block before it must be farther than eps_mass from topk."""
    valid, p, sk, sq = pr["valid"], pr["P"], pr["sK"], pr["sQ"]
    if abs(sq - theta) <= eps_sim:
        return False
    if sq < theta:
        return True
    if not np.all(np.abs(sk[valid] - theta) > eps_sim):
        return False
    if topk >= 1.0:
        return True
    m = oracle.cut_margins(p, valid, topk, mode)
    if m["gap"] <= eps_rel * (m["p_cut"] + m["p_next"]):
        return False
    if mode == "count":
        return True
    return abs(m["c_at"] - topk) > eps_mass and abs(topk - m["c_before"]) > eps_mass


def cut_violations(pr, row: np.ndarray, topk: float, theta: float, eps_rel: float, eps_mass: float,
                   eps_sim: float = EPS_SIM):
    """What is wrong with a GPU mask row (cumulative reading of topk) for the oracle row pr,
    allowing every change that rounding within the slack can make; [] if nothing.

    In the oracle's (probability desc, index asc) order, the blocks the row keeps for their
    probability (kept and not always-kept by a key similarity) must end at some position L - 1
    such that: the dropped blocks before it are near-ties of the block at L - 1 (only rounding
    can swap them), the kept mass up to there (with the always-kept blocks that continue the
    run) reaches topk - eps_mass, and without the block at L - 1 it stays below
    topk + eps_mass (the kept prefix is the shortest one).  A row that keeps every valid block
    (unless its s_Q is below theta) fails the last condition, as does any row with an extra
    block beyond the cut."""
    valid, p, sk, sq = pr["valid"], pr["P"], pr["sK"], pr["sQ"]
    kept = row.astype(bool)
    out = []
    if (kept & ~valid).any():
        out.append("kept blocks outside the valid range")
    if sq < theta - eps_sim:
        if not kept[valid].all():
            out.append("s_Q < theta but the row is not kept whole")
        return out
    if abs(sq - theta) <= eps_sim and kept[valid].all():
        return out  # the row may legitimately be kept whole
    a_sure = valid & (sk < theta - eps_sim)
    a_maybe = valid & (np.abs(sk - theta) <= eps_sim)
    if not kept[a_sure].all():
        out.append("an always-keep column is dropped")
    if topk >= 1.0:
        if not kept[valid].all():
            out.append("topk >= 1 but a valid block is dropped")
        return out
    m = oracle.cut_margins(p, valid, topk)
    order = m["order"]
    ko = kept[order]
    by_p = ko & ~(a_sure | a_maybe)[order]  # kept for their probability alone
    L = int(np.nonzero(by_p)[0].max()) + 1 if by_p.any() else 0
    Lrun = L
    while Lrun < order.size and ko[Lrun]:
        Lrun += 1
    ps = p[order]
    mass_run = float(ps[:Lrun][ko[:Lrun]].sum())
    if mass_run < topk - eps_mass:
        out.append("kept prefix mass %.6g < topk - %.2g" % (mass_run, eps_mass))
    if L > 0:
        p_last = float(ps[L - 1])
        dropped = ~ko[:L]
        if dropped.any():
            worst = float(ps[:L][dropped].max())
            if worst - p_last > eps_rel * (worst + p_last):
                out.append("a block of probability %.6g is dropped before the cut (%.6g)" % (worst, p_last))
        mass_L = float(ps[:L][ko[:L]].sum())
        if mass_L - p_last >= topk + eps_mass:
            out.append("the kept prefix is not the shortest: %.6g without its last block" % (mass_L - p_last))
    return out
