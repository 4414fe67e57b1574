"""Pins of the fp64 oracle against facts that do not come from the oracle itself.

- golden closed-form rows (tests/golden/*.txt)
- top-p restated per element, O(V^2), with no sort or cumulative sum
- q == p: every draft with q > 0 is accepted, for every u < 1
- greedy chain == autoregressive greedy on a prefix-conditioned toy model
  (the Eaglet1 page's "Match = True": speculative greedy output equals plain
  greedy decoding)
- greedy tree == autoregressive greedy, deepest consistent node
- compact draft row + d2t == scattered draft row (EAGLE3 section of the SSD page)
- top-k node expansion == repeated selection of the largest remaining logit
"""
import itertools
import math
import os

import numpy as np
import pytest

from oracle import sv_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _eval(tok):
    tok = tok.strip()
    env = {"log": math.log, "sqrt": math.sqrt, "inf": math.inf}
    return float(eval(tok, {"__builtins__": {}}, env))


def _golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append([part.strip() for part in line.split("|")])
    return rows


@pytest.mark.parametrize("row", _golden("top_p_rows.txt"))
def test_golden_top_p_rows(row):
    logits = np.array([_eval(t) for t in row[0].split(",")])
    T, top_p = float(row[1]), float(row[2])
    want = np.array([_eval(t) for t in row[3].split(",")])
    got, _ = O.dist(logits, T, top_p)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-15)


@pytest.mark.parametrize("row", _golden("inverse_cdf.txt"))
def test_golden_inverse_cdf(row):
    w = np.array([float(t) for t in row[0].split(",")])
    tok, _ = O.inverse_cdf(w, float(row[1]))
    assert tok == int(row[2])


def _kept_per_element(logits, T, top_p):
    """Top-p membership restated without sorting: token j survives iff the
    softmax mass of every token ranked before it (higher logit, or equal
    logit and lower index) is at most top_p."""
    V = len(logits)
    z = [l / T for l in logits]
    m = max(z)
    e = [math.exp(v - m) for v in z]
    s = sum(e)
    pi = [v / s for v in e]
    kept = []
    margins = []
    for j in range(V):
        before = sum(pi[s_] for s_ in range(V)
                     if logits[s_] > logits[j] or (logits[s_] == logits[j] and s_ < j))
        kept.append(before <= top_p)
        margins.append(abs(before - top_p))
    return kept, pi, min(margins)


@pytest.mark.parametrize("seed", range(60))
def test_top_p_matches_per_element_definition(seed):
    g = np.random.default_rng(seed)
    V = int(g.choice([1, 2, 3, 5, 7, 16, 31]))
    if seed % 3 == 0:
        logits = g.integers(-3, 3, V).astype(float)   # many ties
    else:
        logits = g.normal(0, 2, V)
    T = float(g.choice([0.3, 0.8, 1.0, 1.7]))
    top_p = float(g.choice([0.05, 0.3, 0.5, 0.9, 0.95, 0.999]))
    kept, pi, margin = _kept_per_element(list(logits), T, top_p)
    if margin < 1e-9:
        pytest.skip("boundary within rounding of top_p")
    got, _ = O.dist(logits, T, top_p)
    z = sum(p for p, k in zip(pi, kept) if k)
    want = np.array([p / z if k else 0.0 for p, k in zip(pi, kept)])
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-300)
    assert np.array_equal(got > 0, np.array(kept))


def test_top_p_one_keeps_everything():
    g = np.random.default_rng(5)
    logits = g.normal(0, 3, 4000)
    p, margin = O.dist(logits, 1.0, 1.0)
    assert np.all(p > 0) and margin == np.inf


def test_inverse_cdf_never_picks_zero_weight():
    g = np.random.default_rng(9)
    for _ in range(200):
        w = g.random(12) * (g.random(12) < 0.5)
        if w.sum() == 0:
            continue
        for u in (0.0, 0.5, 1.0 - 2 ** -53, g.random()):
            j, _ = O.inverse_cdf(w, u)
            assert w[j] > 0


@pytest.mark.parametrize("seed", range(8))
def test_q_equal_p_accepts_all(seed):
    g = np.random.default_rng(100 + seed)
    gamma, V = 4, 50
    T, top_p = float(g.choice([0.7, 1.0])), float(g.choice([0.8, 1.0]))
    target = g.normal(0, 2, (gamma + 1, V))
    draft = target[:gamma].copy()
    for _ in range(20):
        ids = []
        for i in range(gamma):   # ids with q > 0
            q, _ = O.dist(draft[i], T, top_p)
            ids.append(int(g.choice(np.nonzero(q > 0)[0])))
        u = g.random(gamma) * (1 - 1e-12)
        r = O.verify_chain_row(target, draft, np.array(ids), u, float(g.random()), T, top_p)
        assert r["k"] == gamma
        assert list(r["tokens"][:gamma]) == ids
        p_g, _ = O.dist(target[gamma], T, top_p)
        assert p_g[r["tokens"][gamma]] > 0


def _first_max(row):
    best = 0
    for j in range(1, len(row)):
        if row[j] > row[best]:
            best = j
    return best


def _toy_logits(prefix, V, seed):
    """Prefix-conditioned toy 'target model': quantised logits (frequent ties)."""
    g = np.random.default_rng([seed, len(prefix)] + [int(t) for t in prefix])
    return g.integers(0, 4, V).astype(float)


@pytest.mark.parametrize("seed", range(40))
def test_greedy_chain_equals_autoregressive(seed):
    g = np.random.default_rng(seed)
    V = int(g.choice([3, 5, 8]))
    gamma = int(g.integers(1, 7))
    prefix = tuple(int(t) for t in g.integers(0, V, 3))
    drafts = []
    for i in range(gamma):
        a = _first_max(_toy_logits(prefix + tuple(drafts), V, seed))
        drafts.append(a if g.random() < 0.7 else int(g.integers(V)))
    rows = np.stack([_toy_logits(prefix + tuple(drafts[:i]), V, seed) for i in range(gamma + 1)])
    ar, ctx = [], prefix
    for _ in range(gamma + 1):
        t = _first_max(_toy_logits(ctx, V, seed))
        ar.append(t)
        ctx = ctx + (t,)
    r = O.verify_chain_row(rows, None, np.array(drafts), None, None, 0.0, 0.9)
    k = r["k"]
    assert list(r["tokens"][: k + 1]) == ar[: k + 1]
    assert k == gamma or drafts[k] != ar[k]
    assert all(t == -1 for t in r["tokens"][k + 1:])


def _random_tree(g, N, max_depth, max_children, V):
    parents, depth, nchild = [-1], [0], [0]
    tokens = [int(g.integers(V))]
    for n in range(1, N):
        cand = [m for m in range(n) if depth[m] < max_depth and nchild[m] < max_children]
        if not cand:
            break
        p = int(cand[g.integers(len(cand))])
        parents.append(p)
        depth.append(depth[p] + 1)
        nchild[p] += 1
        nchild.append(0)
        tokens.append(int(g.integers(V)))
    return np.array(parents), np.array(tokens), depth


@pytest.mark.parametrize("seed", range(40))
def test_greedy_tree_equals_autoregressive(seed):
    g = np.random.default_rng(1000 + seed)
    V = int(g.choice([2, 3, 4]))
    N = int(g.integers(1, 14))
    max_depth = int(g.integers(1, 6))
    parents, tokens, depth = _random_tree(g, N, max_depth, 3, V)
    N = len(parents)
    prefix = (7,)

    def path_tokens(n):
        out = []
        while n > 0:
            out.append(int(tokens[n]))
            n = int(parents[n])
        return tuple(reversed(out))

    logits = np.stack([_toy_logits(prefix + path_tokens(n), V, seed) for n in range(N)])
    ar, ctx = [], prefix
    for _ in range(max_depth + 1):
        t = _first_max(_toy_logits(ctx, V, seed))
        ar.append(t)
        ctx = ctx + (t,)
    consistent = [n for n in range(N) if list(path_tokens(n)) == ar[: depth[n]]]
    L = max(depth[n] for n in consistent)

    r = O.verify_tree_row(logits, parents, tokens, max_depth)
    assert r["status"] == 0
    assert r["accept_len"] == L
    assert list(r["out_tokens"][: L + 1]) == ar[: L + 1]
    path = list(r["path"][: L + 1])
    assert path[0] == 0 and all(int(parents[path[i + 1]]) == path[i] for i in range(L))
    assert path[-1] in consistent
    # deepest consistent node, lowest id among equals
    assert path[-1] == min(n for n in consistent if depth[n] == L)


def test_tree_status_bits():
    logits = np.zeros((4, 5))
    ok_par, toks = np.array([-1, 0, 1, 2]), np.array([0, 1, 2, 3])
    assert O.verify_tree_row(logits, ok_par, toks, 3)["status"] == 0
    assert O.verify_tree_row(logits, np.array([-1, 0, 5, 1]), toks, 3)["status"] & O.STATUS_BAD_PARENT
    assert O.verify_tree_row(logits, np.array([0, 0, 1, 1]), toks, 3)["status"] & O.STATUS_BAD_PARENT
    assert O.verify_tree_row(logits, ok_par, toks, 2)["status"] & O.STATUS_DEPTH_EXCEEDED
    assert O.verify_tree_row(logits, ok_par, np.array([0, 1, 9, 3]), 3)["status"] & O.STATUS_BAD_TOKEN


def test_chain_bad_draft_id_flagged():
    t = np.zeros((3, 4))
    r = O.verify_chain_row(t, np.zeros((2, 4)), np.array([1, 4]), np.array([.5, .5]), .5, 1.0, 1.0)
    assert r["status"] == O.STATUS_BAD_DRAFT_ID and r["k"] == 0
    assert np.all(r["tokens"] == -1)


@pytest.mark.parametrize("shuffled", [False, True])
@pytest.mark.parametrize("top_p", [1.0, 0.9, 0.5])
def test_d2t_compact_equals_scattered(shuffled, top_p):
    g = np.random.default_rng(3)
    V, Vd = 300, 60
    d2t = np.sort(g.choice(V, Vd, replace=False))
    if shuffled:
        d2t = d2t[g.permutation(Vd)]
    for rep in range(10):
        row = g.integers(-4, 4, Vd).astype(float) if rep % 2 else g.normal(0, 2, Vd)
        a, _ = O.dist(O.d2t_scatter(row, d2t, V)[0], 0.9, top_p)
        b, _ = O.dist_compact(row, d2t, V, 0.9, top_p)
        np.testing.assert_allclose(a, b, rtol=1e-14, atol=0)
        assert np.array_equal(a > 0, b > 0)


def test_build_t2d_inverse_and_errors():
    d2t = np.array([5, 0, 9, 3])
    t2d = O.build_t2d(d2t, 10)
    assert all(t2d[d2t[j]] == j for j in range(4))
    assert sorted(np.nonzero(t2d < 0)[0]) == [1, 2, 4, 6, 7, 8]
    with pytest.raises(ValueError):
        O.build_t2d(np.array([1, 1]), 4)
    with pytest.raises(ValueError):
        O.build_t2d(np.array([1, 4]), 4)


def test_scatter_fill_and_values():
    out = O.d2t_scatter(np.array([[1.0, 2.0]]), np.array([3, 0]), 5, fill=-7.0)
    assert out.tolist() == [[2.0, -7.0, -7.0, 1.0, -7.0]]


def test_bf16_generator_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    from synth import to_bf16_bits, bf16_bits_to_f32
    g = np.random.default_rng(0)
    x = (g.normal(0, 3, 10000) * g.choice([1e-3, 1, 1e3], 10000)).astype(np.float32)
    x[:4] = [0.0, -0.0, 1.0, -1.0]
    want = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    np.testing.assert_array_equal(bf16_bits_to_f32(to_bf16_bits(x)), want)


# --- top-k node expansion ("A 2.16x speculative-decoding speedup ..." §5) ---

def _top_k_rows():
    rows = []
    for ln in open(os.path.join(GOLDEN, "top_k_rows.txt")):
        if ln.startswith("#") or not ln.strip():
            continue
        k, lg, ids = [c.strip() for c in ln.split("|")]
        rows.append((int(k), np.array([float(x) for x in lg.split()]), [int(x) for x in ids.split()]))
    return rows


@pytest.mark.parametrize("row", _top_k_rows())
def test_golden_top_k_rows(row):
    k, logits, ids = row
    assert O.top_k(logits, k).tolist() == ids


@pytest.mark.parametrize("seed", range(20))
def test_top_k_equals_repeated_selection(seed):
    """Brute force: take the largest remaining logit k times (lowest id among
    equal ones) -- no sort involved."""
    g = np.random.default_rng(seed)
    V = int(g.integers(1, 60))
    x = np.round(g.normal(0, 2, V))            # many ties
    if seed % 4 == 0:
        x[g.integers(0, V, size=max(1, V // 3))] = -np.inf
    k = int(g.integers(1, V + 1))
    left = list(range(V))
    want = []
    for _ in range(k):
        best = left[0]
        for j in left[1:]:
            if x[j] > x[best]:
                best = j
        want.append(best)
        left.remove(best)
    assert O.top_k(x, k).tolist() == want


# ---------------------------------------------------------------------------
# Top-p cuts within NEAR of top_p (reporting only: no result depends on it):
# the alternative cuts one rank shorter or longer, and chain decisions taken
# under every admissible pair of cuts, on rows whose cumulative masses are
# known in closed form: cum = 0.5, 0.8, 0.95, 1.0.

PROBS = [0.5, 0.3, 0.15, 0.05]


def _row_of(probs):
    return np.log(np.asarray(probs, dtype=np.float64))


def test_cut_alternative_one_rank_shorter():
    # top_p just above 0.8: rank 2 is kept because cum[1] = 0.8 <= top_p, a
    # comparison 1e-9 from flipping; the alternative keeps ranks 0 and 1.
    cut = {}
    p, mg = O.dist(_row_of(PROBS), 1.0, 0.8 + 1e-9, cut=cut)
    assert p[3] == 0.0 and p[2] > 0.0 and mg < 1e-8
    assert len(cut["alts"]) == 1
    np.testing.assert_allclose(cut["alts"][0], [0.625, 0.375, 0.0, 0.0], rtol=1e-12)


def test_cut_alternative_one_rank_longer():
    # top_p just below 0.95: rank 3 is removed because cum[2] = 0.95 > top_p;
    # the alternative keeps every id.
    cut = {}
    p, mg = O.dist(_row_of(PROBS), 1.0, 0.95 - 1e-9, cut=cut)
    assert p[3] == 0.0 and p[2] > 0.0
    assert len(cut["alts"]) == 1
    np.testing.assert_allclose(cut["alts"][0], PROBS, rtol=1e-12)


def test_cut_far_from_top_p_has_no_alternative():
    for top_p in (0.9, 1.0):
        cut = {}
        O.dist(_row_of(PROBS), 1.0, top_p, cut=cut)
        assert cut["alts"] == []


def test_chain_decisions_under_admissible_cuts():
    """A one-draft chain whose target and draft rows all have a cut 1e-9 from
    top_p = 0.8 (id 2 kept, or not)."""
    t = np.stack([_row_of(PROBS)] * 2)
    d = _row_of(PROBS)[None, :]
    top_p = 0.8 + 1e-9
    # Draft id 2: p = q = 0.15/0.95 accepts, but with the target's shorter
    # cut p(2) = 0 rejects: the outcome depends on the cut, margin 0.
    r = O.verify_chain_row(t, d, np.array([2]), np.array([0.25]), 0.5, 1.0, top_p)
    assert r["margin"] == 0.0 and r["near_from"] == 0
    np.testing.assert_allclose(r["p_alts"][0, :2], [0.15 / 0.95, 0.0], rtol=1e-12)
    np.testing.assert_allclose(r["q_alts"][0, :2], [0.15 / 0.95, 0.0], rtol=1e-12)
    assert np.isnan(r["p_alts"][0, 2])
    # Draft id 0: p, q in {0.5/0.95, 0.625}, so p/q is 1, 0.5/0.95/0.625 or
    # its inverse: accepted under every pair, margin 0.5/0.95/0.625 - 0.25.
    # The bonus draw from p_1 with u = 0.3 gives id 0 under both cuts, with
    # margins 0.5/0.95 - 0.3 and 0.625 - 0.3.
    r = O.verify_chain_row(t, d, np.array([0]), np.array([0.25]), 0.3, 1.0, top_p)
    assert r["k"] == 1 and r["tokens"].tolist() == [0, 0] and r["near_from"] == 2
    assert r["final_alts"].tolist() == [0] + [-1] * 8
    assert r["margin"] == pytest.approx(min(0.5 / 0.95 / 0.625 - 0.25, 0.5 / 0.95 - 0.3), rel=1e-12)
    # u = 0.55 for the bonus draw: id 1 under the oracle's own cut (its CDF
    # interval is [0.5/0.95, 0.8/0.95]), id 0 under the shorter one ([0, 0.625]).
    r = O.verify_chain_row(t, d, np.array([0]), np.array([0.25]), 0.55, 1.0, top_p)
    assert r["tokens"].tolist() == [0, 1]
    assert r["final_alts"].tolist() == [1, 0] + [-1] * 7
    assert r["margin"] == pytest.approx(0.55 - 0.5 / 0.95, rel=1e-12)
    assert r["near_from"] == 2


def test_chain_residual_draw_under_admissible_cuts():
    """Rejection at 0 with q concentrated on the draft id: the residual
    max(0, p - q) under each pair of cuts, closed form.  Target cut 1e-9 from
    0.8 (p = (0.5, 0.3, 0.15, 0)/0.95, or (0.625, 0.375, 0, 0)); draft row
    (0.97, 0.01, 0.01, 0.01) with top_p 0.8 keeps id 0 only."""
    t = np.stack([_row_of(PROBS)] * 2)
    d = _row_of([0.97, 0.01, 0.01, 0.01])[None, :]
    top_p = 0.8 + 1e-9
    # q = (1, 0, 0, 0): p/q = 0.5/0.95 or 0.625 at id 0; u = 0.9 rejects both.
    # Residual (0, 0.3, 0.15, 0)/0.95 -> ids 1, 2 with weights 2/3, 1/3; or
    # (0, 0.375, 0, 0) -> id 1 alone.  u = 0.7 draws id 2 from the first
    # (margin 0.7 - 2/3), id 1 from the second (margin 0.3).
    r = O.verify_chain_row(t, d, np.array([0]), np.array([0.9]), 0.7, 1.0, top_p)
    assert r["k"] == 0 and r["tokens"].tolist() == [2, -1]
    assert r["final_alts"].tolist() == [2, 1] + [-1] * 7
    assert r["margin"] == pytest.approx(min(0.9 - 0.625, 0.7 - 2 / 3), rel=1e-12)
    assert not r["resample_fallback"]


def test_greedy_row_lists_its_one_final_token():
    t = np.stack([_row_of(PROBS)] * 3)
    r = O.verify_chain_row(t, None, np.array([0, 1]), None, None, 0.0, 1.0)
    assert r["k"] == 1 and r["tokens"].tolist() == [0, 0, -1]
    assert r["final_alts"].tolist() == [0] + [-1] * 8
