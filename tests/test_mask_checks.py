"""CPU checks of the full-size mask comparison (tests/mask_checks.py): on oracle rows of a
Llama-like workload with long rows, the oracle's own masks pass, and masks with a planted
mistake (every block kept, the most probable block dropped, an extra block past the cut, the
cut block dropped) are caught on every row where the slack leaves the cut in place."""
import math

import numpy as np
import pytest

import oracle
import workloads as W
from mask_checks import EPS_SIM, cut_violations, decisive, score_error_bound, slack


@pytest.fixture(scope="module")
def rows():
    w = W.make_config("llama32k", Hq=1, Hkv=1, N=16384 + 77)
    q, k = W.bf16_to_f64(w.q[0, 0]), W.bf16_to_f64(w.k[0, 0])
    kp = oracle.pool_key_head(k)
    scale = oracle.default_scale(w.d)
    out = []
    for i in range(0, w.nqb, 3):
        pr = oracle.predict_mask_row(q[i * 128:(i + 1) * 128], k, i, w.topk, w.theta, w.causal, k_pool=kp)
        E = score_error_bound(pr["muQ"], kp[0], pr["S"], pr["valid"], scale)
        out.append((pr,) + slack(E))
    return w, out


def test_oracle_rows_pass_and_most_are_decisive(rows):
    w, rs = rows
    n_dec = 0
    for pr, er, em in rs:
        assert cut_violations(pr, pr["mask"], w.topk, w.theta, er, em) == []
        n_dec += decisive(pr, w.topk, w.theta, er, em)
    assert n_dec >= len(rs) // 2, (n_dec, len(rs))


def _planted(pr, topk, theta, eps_sim):
    """Masks with one mistake each, for a row whose s_Q is above theta."""
    valid, p, sk = pr["valid"], pr["P"], pr["sK"]
    base = pr["mask"].astype(bool)
    m = oracle.cut_margins(p, valid, topk)
    order = m["order"]
    always = valid & (sk < theta + eps_sim)
    by_p = [j for j in order[:m["kstar"]] if not always[j]]
    out = {}
    allk = base.copy()
    allk[valid] = True
    if not np.array_equal(allk, base):
        out["keep all"] = allk
    if by_p:
        top = base.copy()
        top[by_p[0]] = False
        out["most probable dropped"] = top
        cut = base.copy()
        cut[order[m["kstar"] - 1]] = False
        if not always[order[m["kstar"] - 1]]:
            out["cut block dropped"] = cut
    extra = [j for j in order[m["kstar"]:] if not base[j]]
    if extra:
        e = base.copy()
        e[extra[len(extra) // 2]] = True
        out["extra block past the cut"] = e
    return out


def test_planted_mistakes_are_caught_on_decisive_rows(rows):
    w, rs = rows
    n_checked = 0
    for pr, er, em in rs:
        if pr["sQ"] < w.theta + EPS_SIM or not decisive(pr, w.topk, w.theta, er, em):
            continue
        for what, bad in _planted(pr, w.topk, w.theta, EPS_SIM).items():
            assert cut_violations(pr, bad.astype(np.uint8), w.topk, w.theta, er, em), what
            n_checked += 1
    assert n_checked >= 40, n_checked


def test_keep_all_rows_fail_even_where_not_decisive(rows):
    """A row that keeps every valid block passes only where s_Q puts it near or below theta."""
    w, rs = rows
    for pr, er, em in rs:
        if pr["sQ"] < w.theta + EPS_SIM:
            continue
        allk = pr["valid"].astype(np.uint8)
        if not np.array_equal(allk, pr["mask"]):
            assert cut_violations(pr, allk, w.topk, w.theta, er, em)
