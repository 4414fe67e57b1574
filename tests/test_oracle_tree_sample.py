"""Pins of the tree speculative-sampling oracle (verify_tree_sample_row).

The pages fix only the one-draft rule ("LLM inference acceleration in
practice ..." §3.1) and the tree's shape ("A 2.16x speculative-decoding
speedup ..." §5); the tree rule is a reading (sequential per-child rejection
with a residual update).  What pins it is the property that reading must
have: when every node's children are independent draws from that node's
draft distribution, the emitted tokens follow the target.  The theorem test
enumerates every token assignment of small trees and every accept/reject
history exactly (the thresholds come from the oracle's trace and are checked
against its decisions; the last draw is checked against its CDF), and
compares the distribution of the first two emitted tokens with the target's.
Further pins: a one-child-per-node tree is the chain verify (pinned on its
own), q == p accepts every first child, hand-derived small cases, the
zero-residual fallback and invalid trees.
"""
import itertools

import numpy as np
import pytest

from oracle import sv_oracle as O


def _emit_distribution(rows_of, parents, V, temperature, top_p, max_depth):
    """Exact law of (first token, second token or None) over every token
    assignment of the tree (children drawn from their parent's q) and every
    accept/reject history."""
    N = len(parents)
    first = np.zeros(V)
    pair = np.zeros((V, V))
    first_accepted = np.zeros(V)
    for assign in itertools.product(range(V), repeat=N - 1):
        tokens = np.array((0,) + assign)
        # token path of every node -> its target and draft rows
        paths = [()]
        for n in range(1, N):
            paths.append(paths[parents[n]] + (int(tokens[n]),))
        t_rows = np.array([rows_of(pth)[0] for pth in paths])
        d_rows = np.array([rows_of(pth)[1] for pth in paths])
        w = 1.0
        for n in range(1, N):
            q, _ = O.dist(d_rows[parents[n]], temperature, top_p)
            w *= q[tokens[n]]
        if w == 0.0:
            continue
        for prob, seq, acc in _histories(t_rows, d_rows, parents, tokens, temperature, top_p, max_depth):
            first[seq[0]] += w * prob
            if len(seq) > 1:
                pair[seq[0], seq[1]] += w * prob
                first_accepted[seq[0]] += w * prob
            else:
                assert acc == 0
    return first, pair, first_accepted


def _histories(t_rows, d_rows, parents, tokens, temperature, top_p, max_depth):
    N = len(parents)
    out = []

    def run(fixed, u_final=0.5):
        u = np.zeros(N)
        for n, (acc, th) in fixed.items():
            u[n] = th / 2 if acc else (1 + th) / 2
        tr = []
        res = O.verify_tree_sample_row(t_rows, d_rows, parents, tokens, u, u_final, temperature, top_p,
                                       max_depth, trace=tr)
        assert res["status"] == 0
        return res, tr

    def explore(fixed, prob):
        res, tr = run(fixed)
        tests = [e for e in tr if "node" in e]
        for e in tests:
            n = e["node"]
            if n in fixed:
                assert e["accepted"] == fixed[n][0]      # the oracle honours its own threshold
                continue
            th = e["threshold"]
            assert 0.0 <= th <= 1.0
            if th > 0.0:
                explore({**fixed, n: (True, th)}, prob * th)
            if th < 1.0:
                explore({**fixed, n: (False, th)}, prob * (1.0 - th))
            return
        w = tr[-1]["weights"]
        d = res["accept_len"]
        path_tokens = tuple(int(x) for x in res["out_tokens"][:d])
        cdf = np.cumsum(w)
        for x in range(len(w)):
            if w[x] <= 0.0:
                continue
            mid = (cdf[x] - w[x] / 2) / cdf[-1]
            r2, _ = run(fixed, u_final=mid)
            assert r2["out_tokens"][d] == x                   # the draw follows the reported weights
            out.append((prob * w[x], path_tokens + (x,), d))

    explore({}, 1.0)
    return out


def _rows_table(seed, V):
    g = np.random.default_rng(seed)
    cache = {}

    def rows_of(path):
        if path not in cache:
            cache[path] = (g.normal(0, 1.5, V), g.normal(0, 1.5, V))
        return cache[path]
    return rows_of


@pytest.mark.parametrize("parents,V,T,top_p,seed", [
    ([-1, 0, 0, 0], 5, 1.0, 1.0, 1),           # three children of the root
    ([-1, 0, 0, 0, 1], 4, 0.8, 1.0, 2),        # three children, one grandchild
    ([-1, 0, 0, 1, 1], 4, 1.3, 1.0, 3),        # depth 2, two children per node
    ([-1, 0, 0, 0, 2], 4, 1.0, 0.8, 6),        # top-p on p and q (children of q = 0 never drawn)
    ([-1, 0, 0, 1, 2], 3, 1.0, 0.7, 6),
])
def test_emitted_tokens_follow_the_target(parents, V, T, top_p, seed):
    """Exact to 1e-12.  With three or more tokens and three siblings, a
    residual taken from p instead of r, or left unnormalised, moves the first
    token's law by 2e-3 to 1e-1 on these cases; the sibling order is free
    here (siblings are exchangeable) and is pinned by the hand-derived case."""
    rows_of = _rows_table(seed, V)
    rows_of(())
    first, pair, first_acc = _emit_distribution(rows_of, np.array(parents), V, T, top_p, max_depth=3)
    p_root, _ = O.dist(rows_of(())[0], T, top_p)
    np.testing.assert_allclose(first, p_root, rtol=0, atol=1e-12)
    for x1 in range(V):
        p1, _ = O.dist(rows_of((x1,))[0], T, top_p)
        np.testing.assert_allclose(pair[x1], first_acc[x1] * p1, rtol=0, atol=1e-12)
    assert first_acc.sum() > 0.05                 # the second-token check is not vacuous


def test_chain_shaped_tree_is_the_chain_verify():
    g = np.random.default_rng(7)
    V, gamma = 40, 5
    for trial in range(30):
        t = g.normal(0, 2, (gamma + 1, V))
        d = t + g.normal(0, 0.7, (gamma + 1, V))
        ids = g.integers(0, V, gamma)
        ua, uf = g.random(gamma), float(g.random())
        T, top_p = (1.0, 1.0) if trial % 2 else (0.7, 0.9)
        chain = O.verify_chain_row(t, d[:gamma], ids, ua, uf, T, top_p)
        parents = np.arange(-1, gamma)
        tokens = np.concatenate([[0], ids])
        u_tree = np.concatenate([[0.0], ua])
        tree = O.verify_tree_sample_row(t, d, parents, tokens, u_tree, uf, T, top_p, gamma)
        assert tree["accept_len"] == chain["k"]
        assert tree["out_tokens"].tolist() == chain["tokens"].tolist()


def test_q_equal_p_accepts_every_first_child():
    g = np.random.default_rng(8)
    V = 30
    parents = np.array([-1, 0, 0, 1, 1, 3, 2])
    tokens = np.array([0, 4, 9, 4, 4, 7, 1])
    t = g.normal(0, 1, (7, V))
    u = g.random(7) * 0.999
    r = O.verify_tree_sample_row(t, t, parents, tokens, u, 0.37, 1.0, 1.0, 4)
    assert r["path"].tolist() == [0, 1, 3, 5, -1]
    p5, _ = O.dist(t[5], 1.0, 1.0)
    assert r["out_tokens"].tolist() == [4, 4, 7, O.inverse_cdf(p5, 0.37)[0], -1]


def test_hand_derived_residual_updates():
    """p = (1/2, 1/2) and q = (0.9, 0.1) at the root (T = 1, no top-p)."""
    t = np.log(np.array([[0.5, 0.5]] * 3))
    d = np.log(np.array([[0.9, 0.1]] * 3))
    parents = np.array([-1, 0, 0])
    # Both children token 0.  Child 1: 0.9 * 0.9 = 0.81 >= 0.5, rejected;
    # r = norm(max(0, p - q)) = (0, 1).  Child 2: 0.1 * 0.9 >= r(0) = 0,
    # rejected; r = norm(max(0, (0, 1) - q)) = (0, 1).  Last token: 1.
    r = O.verify_tree_sample_row(t, d, parents, np.array([0, 0, 0]), np.array([0, 0.9, 0.1]), 0.01, 1.0, 1.0, 1)
    assert (r["accept_len"], r["out_tokens"].tolist()) == (0, [1, -1])
    # Tokens 0 then 1: child 1 rejected as above; child 2 has r(1) = 1 > u * 0.1
    # for every u < 1, so it is accepted; its row has no children and the bonus
    # comes from p = (1/2, 1/2): u = 0.7 -> token 1, u = 0.2 -> token 0.
    for uf, bonus in ((0.7, 1), (0.2, 0)):
        r = O.verify_tree_sample_row(t, d, parents, np.array([0, 0, 1]), np.array([0, 0.9, 0.999]), uf, 1.0, 1.0, 1)
        assert (r["accept_len"], r["path"].tolist(), r["out_tokens"].tolist()) == (1, [0, 2], [1, bonus])
    # Child 1 with u = 0.5: 0.5 * 0.9 = 0.45 < 0.5, accepted.
    r = O.verify_tree_sample_row(t, d, parents, np.array([0, 0, 1]), np.array([0, 0.5, 0.0]), 0.7, 1.0, 1.0, 1)
    assert r["path"].tolist() == [0, 1]


def test_zero_residual_fallback():
    """q == p, and top-p removes the child's token from both: r(x) = q(x) = 0,
    the child is rejected and max(0, r - q) has no mass; r stays p."""
    V = 6
    row = np.array([3.0, 2.5, 0.0, -1.0, -2.0, -3.0])
    t = np.stack([row, row])
    r = O.verify_tree_sample_row(t, t, np.array([-1, 0]), np.array([0, 5]), np.array([0, 0.5]), 0.6, 1.0, 0.5, 1)
    p, _ = O.dist(row, 1.0, 0.5)
    assert p[5] == 0.0 and r["resample_fallback"] and r["accept_len"] == 0
    assert r["out_tokens"][0] == O.inverse_cdf(p, 0.6)[0]


def test_invalid_trees_emit_nothing():
    g = np.random.default_rng(9)
    t = g.normal(size=(4, 8))
    u = np.full(4, 0.5)
    cases = [(np.array([-1, 0, 3, 1]), np.array([0, 1, 2, 3]), O.STATUS_BAD_PARENT),
             (np.array([-1, 0, 1, 2]), np.array([0, 1, 8, 3]), O.STATUS_BAD_TOKEN),
             (np.array([-1, 0, 1, 2]), np.array([0, 1, 2, 3]), O.STATUS_DEPTH_EXCEEDED)]
    for parents, tokens, bit in cases:
        r = O.verify_tree_sample_row(t, t, parents, tokens, u, 0.5, 1.0, 1.0, 2)
        assert r["status"] & bit and r["accept_len"] == 0 and np.all(r["out_tokens"] == -1)
    bad = t.copy()
    bad[2] = -np.inf
    r = O.verify_tree_sample_row(t, bad, np.array([-1, 0, 0, 1]), np.array([0, 1, 2, 3]), u, 0.5, 1.0, 1.0, 3)
    assert r["status"] & O.STATUS_EMPTY_ROW


def test_decisions_under_admissible_cuts():
    """Rows (0.5, 0.3, 0.15, 0.05) with top_p 1e-9 above cum[1] = 0.8: id 2 is
    kept, or not (the one-rank-shorter cut, (0.625, 0.375, 0, 0))."""
    row = np.log(np.array([0.5, 0.3, 0.15, 0.05]))
    top_p = 0.8 + 1e-9
    rows = np.stack([row, row])
    # Root with one child of token 2, u = 0.25: accepted under the oracle's own
    # cuts (r = p, q(2) = p(2)), rejected once the target's cut drops id 2.
    r = O.verify_tree_sample_row(rows, rows, np.array([-1, 0]), np.array([0, 2]), np.array([0.0, 0.25]),
                                 0.3, 1.0, top_p, 1)
    assert r["accept_len"] == 1 and r["margin"] == 0.0
    # A root alone: the bonus draw from p with u = 0.55 gives id 1 under the
    # own cut (CDF interval [0.5/0.95, 0.8/0.95]) and id 0 under the shorter
    # one ([0, 0.625]); margin the smaller distance to an interval edge.
    r = O.verify_tree_sample_row(rows[:1], rows[:1], np.array([-1]), np.array([0]), np.array([0.0]),
                                 0.55, 1.0, top_p, 1)
    assert r["out_tokens"].tolist() == [1, -1]
    assert r["final_alts"].tolist() == [1, 0] + [-1] * 7
    assert r["margin"] == pytest.approx(0.55 - 0.5 / 0.95, rel=1e-12)
    # Far from any cut: one admissible token, the oracle's own.
    r = O.verify_tree_sample_row(rows[:1], rows[:1], np.array([-1]), np.array([0]), np.array([0.0]),
                                 0.55, 1.0, 0.9, 1)
    assert r["final_alts"].tolist() == [int(r["out_tokens"][0])] + [-1] * 8
