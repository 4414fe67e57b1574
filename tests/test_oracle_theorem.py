"""Exact enumeration of the speculative-sampling theorem on the oracle.

Source: "LLM inference acceleration in practice: draft models and speculative
sampling explained" (mlqm.cn) §3.1: accepting each draft with min(1, p/q),
resampling from norm(max(0, p - q)) at the first rejection and drawing the
bonus from p leaves the output distributed as the target's.

For tiny vocabularies every draft sequence (weighted by its draft
probability) and every cell of the uniforms on which the oracle's output is
constant is visited; the oracle's verify function itself runs at each cell
midpoint.  The checks are the theorem's closed forms:
  * conditioned on the first i drafts surviving, the token at position i is
    distributed as p_i;
  * P(draft i survives | drafts < i survived) = sum_x min(p_i(x), q_i(x)).
"""
import itertools

import numpy as np
import pytest

from oracle import sv_oracle as O


def _cells_accept(ratio):
    """Cells of u for the test u*q < p, i.e. u < ratio."""
    if ratio >= 1.0:
        return [(0.5, 1.0)]
    if ratio <= 0.0:
        return [(0.5, 1.0)]
    return [(ratio / 2, ratio), ((1 + ratio) / 2, 1 - ratio)]


def _cells_resample(dists):
    """Cells of u on which every candidate inverse CDF is constant."""
    pts = {0.0, 1.0}
    for w in dists:
        c = np.cumsum(w)
        if c[-1] > 0:
            pts.update(float(v) for v in c / c[-1])
    pts = sorted(p for p in pts if 0.0 <= p <= 1.0)
    return [((a + b) / 2, b - a) for a, b in zip(pts, pts[1:]) if b - a > 1e-15]


def _enumerate(target, draft, T, top_p):
    gamma, V = draft.shape
    p = [O.dist(target[i], T, top_p)[0] for i in range(gamma + 1)]
    q = [O.dist(draft[i], T, top_p)[0] for i in range(gamma)]
    cand = [np.maximum(0.0, p[i] - q[i]) for i in range(gamma)] + p
    res_cells = _cells_resample(cand)
    reach = np.zeros(gamma + 1)
    emitted = np.zeros((gamma + 1, V))
    for ids in itertools.product(range(V), repeat=gamma):
        wd = float(np.prod([q[i][ids[i]] for i in range(gamma)]))
        if wd == 0.0:
            continue
        per_pos = [_cells_accept(p[i][ids[i]] / q[i][ids[i]]) for i in range(gamma)]
        for combo in itertools.product(*per_pos):
            u_acc = np.array([c[0] for c in combo])
            w_acc = float(np.prod([c[1] for c in combo]))
            for u_res, w_res in res_cells:
                r = O.verify_chain_row(target, draft, np.array(ids), u_acc, u_res, T, top_p)
                w = wd * w_acc * w_res
                for i in range(r["k"] + 1):
                    reach[i] += w
                    emitted[i, r["tokens"][i]] += w
    return p, q, reach, emitted


CASES = [(2, 1), (3, 1), (4, 1), (2, 2), (3, 2), (4, 2), (2, 3), (3, 3)]


@pytest.mark.parametrize("V,gamma", CASES)
@pytest.mark.parametrize("T,top_p", [(1.0, 1.0), (0.7, 0.8)])
def test_speculative_sampling_theorem(V, gamma, T, top_p):
    g = np.random.default_rng(V * 100 + gamma * 10 + int(top_p * 7))
    target = g.normal(0, 1.5, (gamma + 1, V))
    draft = target[:gamma] + g.normal(0, 1.0, (gamma, V))
    p, q, reach, emitted = _enumerate(target, draft, T, top_p)
    assert abs(reach[0] - 1.0) < 1e-12
    for i in range(gamma + 1):
        if reach[i] < 1e-9:
            continue
        np.testing.assert_allclose(emitted[i] / reach[i], p[i], rtol=0, atol=1e-12)
    for i in range(gamma):
        beta = float(np.minimum(p[i], q[i]).sum())
        assert abs(reach[i + 1] / reach[i] - beta) < 1e-12


def test_theorem_with_sparse_supports():
    """Supports that differ (q puts mass where p has none and vice versa)."""
    target = np.log(np.array([[0.6, 0.4, 1e-300, 1e-300], [0.1, 0.2, 0.3, 0.4]]))
    target[0, 2:] = -np.inf
    draft = np.log(np.array([[0.2, 1e-300, 0.5, 0.3]]))
    draft[0, 1] = -np.inf
    p, q, reach, emitted = _enumerate(target, draft, 1.0, 1.0)
    np.testing.assert_allclose(emitted[0] / reach[0], p[0], atol=1e-12)
    np.testing.assert_allclose(emitted[1] / reach[1], p[1], atol=1e-12)
    assert abs(reach[1] - np.minimum(p[0], q[0]).sum()) < 1e-12
