"""Pins of the oracle's draft-side sampler (sample_row) that do not come from
the oracle itself.

- golden rows with hand-derived tokens (tests/golden/sample_rows.txt);
- the exact law of sample_row over the uniform u: on every cell of [0, 1)
  between consecutive prefix sums of the filtered distribution (restated per
  element, with no sort or cumulative sum, and with the tie key of an EAGLE3
  compact row when one is given) the draw is the cell's token, so the token
  law equals that distribution; a sampler that drew from the unfiltered
  softmax, or ranked ties by the compact index instead of the target id,
  fails these checks;
- T = 0: the argmax with the lowest id on ties, by a plain scan.

Source: "LLM inference acceleration in practice: draft models and speculative
sampling explained" (mlqm.cn) §3.1 (drafting) and §4.2 (the draft loop:
/ T, _apply_top_p, softmax, multinomial).
"""
import math
import os

import numpy as np
import pytest

from oracle import sv_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _eval(tok):
    env = {"log": math.log, "inf": math.inf}
    return float(eval(tok.strip(), {"__builtins__": {}}, env))


def _golden():
    rows = []
    with open(os.path.join(GOLDEN, "sample_rows.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append([p.strip() for p in line.split("|")])
    return rows


@pytest.mark.parametrize("row", _golden())
def test_golden_sample_rows(row):
    logits = np.array([_eval(t) for t in row[0].split(",")])
    tok, _ = O.sample_row(logits, float(row[1]), float(row[2]), float(row[3]))
    assert tok == int(row[4])


def _filtered(logits, T, top_p, tie):
    """softmax(top_p_filter(logits / T)) restated per element: token j is
    kept iff the softmax mass of every token ranked before it (higher logit,
    or equal logit and lower tie key) is at most top_p.  Returns the
    probabilities and the distance of the closest kept/dropped decision from
    top_p."""
    V = len(logits)
    finite = [l for l in logits if l != -math.inf]
    m = max(finite) / T
    e = [0.0 if l == -math.inf else math.exp(l / T - m) for l in logits]
    s = sum(e)
    pi = [v / s for v in e]
    if top_p >= 1.0:
        return pi, math.inf
    kept, margin = [], math.inf
    for j in range(V):
        before = sum(pi[k] for k in range(V)
                     if logits[k] > logits[j] or (logits[k] == logits[j] and tie[k] < tie[j]))
        kept.append(before <= top_p)
        margin = min(margin, abs(before - top_p))
    z = sum(p for p, k in zip(pi, kept) if k)
    return [p / z if k else 0.0 for p, k in zip(pi, kept)], margin


def _check_law(logits, T, top_p, tie_index=None):
    """For every token j with probability p_j > 0, every u in the cell
    [P_{j-1}, P_j) (prefix sums in ascending id order, P_{-1} = 0) draws j.
    The cells cover [0, 1) and have lengths p_j: the law of the draw is p."""
    V = len(logits)
    tie = list(range(V)) if tie_index is None else list(tie_index)
    p, margin = _filtered(list(logits), T, top_p, tie)
    if margin < 1e-9:
        pytest.skip("a top-p decision within rounding of top_p")
    lo = 0.0
    checked = 0
    for j in range(V):
        if p[j] == 0.0:
            continue
        hi = lo + p[j]
        for f in (1e-9, 0.25, 0.5, 0.75, 1.0 - 1e-9):
            u = lo + f * (hi - lo)
            if u >= 1.0 or min(u - lo, hi - u) < 1e-11:
                continue
            tok, _ = O.sample_row(logits, T, top_p, u, tie_index=tie_index)
            assert tok == j, (j, u, tok, p)
            checked += 1
        lo = hi
    assert checked > 0 and abs(lo - 1.0) < 1e-12


@pytest.mark.parametrize("seed", range(40))
def test_law_equals_filtered_distribution(seed):
    g = np.random.default_rng(500 + seed)
    V = int(g.choice([2, 3, 5, 8, 13]))
    logits = g.normal(0, 2, V)
    if seed % 4 == 0:
        logits = np.round(logits)              # ties
    if seed % 5 == 1 and V > 2:
        logits[g.integers(V)] = -math.inf      # an impossible token
    T = float(g.choice([0.4, 0.8, 1.0, 1.5]))
    top_p = float(g.choice([0.2, 0.5, 0.8, 0.95, 1.0]))
    _check_law(logits, T, top_p)


@pytest.mark.parametrize("seed", range(20))
def test_law_on_compact_rows_with_target_tie_keys(seed):
    """EAGLE3 compact draft rows: ties in the top-p ranking follow the
    target ids given as tie_index (a permuted map here), and the draw is
    over compact ids."""
    g = np.random.default_rng(900 + seed)
    V = int(g.choice([4, 6, 9]))
    logits = np.round(g.normal(0, 1.5, V))   # many ties, so the tie key matters
    tie_index = g.permutation(40)[:V]
    T = float(g.choice([0.7, 1.0]))
    top_p = float(g.choice([0.3, 0.6, 0.9]))
    _check_law(logits, T, top_p, tie_index=tie_index)


def test_unfiltered_sampler_would_fail():
    """The cell check tells the filtered law from the unfiltered one on a
    row where they differ."""
    logits = np.log(np.array([0.1, 0.3, 0.2, 0.4]))
    p_f, _ = _filtered(list(logits), 1.0, 0.6, [0, 1, 2, 3])
    p_u, _ = _filtered(list(logits), 1.0, 1.0, [0, 1, 2, 3])
    assert not np.allclose(p_f, p_u)
    # u = .45 lies in token 3's filtered cell [3/7, 1) but in token 2's
    # unfiltered cell [.4, .6)
    assert O.sample_row(logits, 1.0, 0.6, 0.45)[0] == 3
    assert O.sample_row(logits, 1.0, 1.0, 0.45)[0] == 2


@pytest.mark.parametrize("seed", range(10))
def test_greedy_is_lowest_argmax(seed):
    g = np.random.default_rng(seed)
    logits = np.round(g.normal(0, 1, 9))
    best = 0
    for j in range(1, 9):
        if logits[j] > logits[best]:
            best = j
    assert O.sample_row(logits, 0.0, 0.9, 0.3)[0] == best


def test_compact_row_ties_follow_the_target_ids():
    """Three equal logits whose target ids are 30, 10, 20: top_p = 0.3 keeps
    only the lowest target id (compact id 1), whatever u is; with the compact
    index as the tie key compact id 0 would be drawn instead."""
    logits = np.zeros(3)
    tie_index = np.array([30, 10, 20])
    for u in (0.0, 0.3, 0.7, 0.999):
        assert O.sample_row(logits, 1.0, 0.3, u, tie_index=tie_index)[0] == 1
    assert O.sample_row(logits, 1.0, 0.3, 0.5)[0] == 0


def test_sample_row_lists_the_draws_of_admissible_cuts():
    """Masses 0.5, 0.3, 0.15, 0.05 (cum 0.5, 0.8, 0.95, 1.0) and top_p 1e-9
    above 0.8: the cut keeps three ids, or two.  u = 0.55 draws id 1 under
    the own cut (its interval [0.5/0.95, 0.8/0.95]) and id 0 under the
    shorter one ([0, 0.625]); the margin is the smaller distance to an edge."""
    row = np.log(np.array([0.5, 0.3, 0.15, 0.05]))
    alts = []
    tok, mg = O.sample_row(row, 1.0, 0.8 + 1e-9, 0.55, alts=alts)
    assert tok == 1
    assert [a[0] for a in alts] == [1, 0]
    assert alts[0][1] == pytest.approx(0.3 / 0.95, rel=1e-12) and alts[1][1] == pytest.approx(0.625, rel=1e-12)
    assert mg == pytest.approx(0.55 - 0.5 / 0.95, rel=1e-12)
    # without the list, the cut's own margin (1e-9) decides
    assert O.sample_row(row, 1.0, 0.8 + 1e-9, 0.55)[1] < 1e-8
    # far from any cut: one admissible draw
    alts = []
    O.sample_row(row, 1.0, 0.9, 0.55, alts=alts)
    assert len(alts) == 1
