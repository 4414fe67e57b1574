"""fp64 CPU oracle for the speculative-decoding verify step.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import this module:
only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` use it.  It shares no code with the
CUDA library (no kernels, headers, tables or helpers); the only thing both
sides consume is the seeded input generator in ``synth/``.

Everything here is plain numpy in float64, one row at a time, written to be
checked against the pages by eye rather than to be fast.  Sources:

[P3] "LLM inference acceleration in practice: draft models and speculative
     sampling explained" (mlqm.cn/news/1205650):
     §3.1 (the algorithm: draft, verify, accept with min(1, p/q), resample
     from norm(max(0, p - q)), bonus token from p when all drafts survive),
     §4.2 (``SpeculativeDecoder.generate`` and ``_apply_top_p``),
     §6.2 (batched verify; draft and target share temperature and top_p).
[P2] "A 2.16x speculative-decoding speedup from a 1-layer Llama draft"
     (blog.bruce.linkpc.net, Eagle-2.16x-acceleration-in-5-minutes):
     the headline table (greedy output "Match = True"), §5 (draft token tree:
     total_token 32, depth 5, top_k 8).
[P1] "SSD: extending the engine with new models and an EAGLE3 draft"
     (lpnh.cn/news/2716086): §六 (EAGLE3 ``lm_head`` over a small draft
     vocabulary, ``d2t``/``t2d`` scatter back into the target vocabulary),
     §七 (``--temp 0`` greedy benchmarking).

Readings where the pages are silent or garbled (their punctuation was lost in
extraction) are marked READING and listed in the design notes.

Status bits follow the library's public convention so tests can compare them;
they are restated here, not imported.

Parity pins (tests/test_oracle_*.py): the speculative-sampling theorem by
exact enumeration (for the chain and for the sampled tree), q == p
acceptance, greedy == autoregressive greedy on a prefix-conditioned toy
model, an O(V^2) per-element statement of top-p, closed-form golden rows,
compact-vs-scattered d2t, brute-force tree paths, a one-child-per-node tree
against the chain, and repeated-argmax top-k.  No function here is "parity
unpinned".
"""
from __future__ import annotations

import numpy as np

# Row status bits (restated from the public header's documentation).
STATUS_BAD_DRAFT_ID = 1    # a draft id outside [0, V)
STATUS_BAD_PARENT = 2      # tree: parents[0] != -1 or parents[n] not in [0, n)
STATUS_DEPTH_EXCEEDED = 4  # tree: a node deeper than max_depth
STATUS_BAD_TOKEN = 8       # tree: a node token outside [0, V)
STATUS_EMPTY_ROW = 16      # a row whose logits are all -inf (no distribution)

NEAR = 1e-6  # decisions closer than this to their threshold may legitimately differ
ALTS = 3     # a top-p cut, and the one rank shorter and longer that NEAR admits


# ---------------------------------------------------------------------------
# One row: temperature, top-p, softmax  ([P3] §4.2 generate(), _apply_top_p)
# ---------------------------------------------------------------------------

def softmax(z: np.ndarray) -> np.ndarray:
    """Plain softmax in float64; -inf entries get probability 0."""
    z = np.asarray(z, dtype=np.float64)
    m = np.max(z)
    e = np.exp(z - m)
    return e / e.sum()


def nucleus_order(logits: np.ndarray, tie_index: np.ndarray | None = None) -> np.ndarray:
    """Indices of the row sorted by logit descending, ties by index ascending.

    [P3] §4.2 ``_apply_top_p`` sorts descending with ``torch.sort``, whose tie
    order is unspecified.  READING: equal logits are ranked lower index first,
    and ranking is on the logit itself (dividing by T > 0 keeps the order).
    ``tie_index`` replaces the position as the tie key (used when a compact
    draft row stands for a scattered one: ties follow target-vocab ids).
    """
    logits = np.asarray(logits, dtype=np.float64)
    idx = np.arange(logits.size) if tie_index is None else np.asarray(tie_index)
    # +0.0 makes -0.0 and +0.0 the same sort key (they are equal logits).
    return np.lexsort((idx, -(logits + 0.0)))


def top_p_filter(z: np.ndarray, top_p: float, order: np.ndarray, cut: dict | None = None):
    """[P3] §4.2 ``_apply_top_p`` on temperature-scaled logits ``z``.

    Steps as the page gives them: sort descending, softmax of the sorted
    logits, cumulative sum, mark for removal where the cumulative probability
    exceeds top_p, shift the mark right by one so the first token past the
    threshold survives, never remove the top token, then set removed logits
    to -inf.

    READING (comparator lost in extraction): "remove if cumulative > top_p",
    i.e. rank r is kept iff r == 0 or cum[r-1] <= top_p.  READING: top_p >= 1
    filters nothing (rounding of the cumulative sum must not drop the tail).

    Returns (filtered z, boundary margin).  The margin is the distance of
    top_p from the nearest cumulative value that decides the cut; inf when
    no filtering happens.  When ``cut`` is a dict it also receives (for
    reporting only) "alts": the filtered z of every other cut whose
    keep-or-drop comparison lies within NEAR of top_p -- one rank fewer when
    the last kept rank's comparison is that close, one rank more when the
    first removed rank's is -- so that a caller can take each decision under
    every cut that rounding could produce.
    """
    z = np.asarray(z, dtype=np.float64)
    if top_p >= 1.0:
        return z.copy(), np.inf
    sorted_probs = softmax(z[order])
    cum = np.cumsum(sorted_probs)
    remove = cum > top_p
    remove[1:] = remove[:-1].copy()
    remove[0] = False
    out = z.copy()
    out[order[remove]] = -np.inf
    kept = int(np.count_nonzero(~remove))  # ranks 0..kept-1 survive
    margin = np.inf
    if kept >= 1 and kept - 1 < cum.size:
        margin = min(margin, abs(cum[kept - 1] - top_p))   # first cum above top_p
    if kept >= 2:
        margin = min(margin, abs(cum[kept - 2] - top_p))   # last cum at or below
    if cut is not None:
        alt_kept = []
        if kept < cum.size and abs(cum[kept - 1] - top_p) < NEAR:
            alt_kept.append(kept + 1)   # the first removed rank kept as well
        if kept >= 2 and abs(cum[kept - 2] - top_p) < NEAR:
            alt_kept.append(kept - 1)   # the last kept rank removed
        for n in alt_kept:
            alt = z.copy()
            alt[order[n:]] = -np.inf
            cut["alts"].append(alt)
    return out, margin


def dist(logits: np.ndarray, temperature: float, top_p: float,
         tie_index: np.ndarray | None = None, cut: dict | None = None):
    """Distribution of one position: softmax(top_p_filter(logits / T)).

    [P3] §4.2: ``logits / temperature`` -> ``_apply_top_p`` -> ``F.softmax``.
    Returns (probabilities float64[V], top-p boundary margin).  When ``cut``
    is a dict it receives "alts": the distributions of the other cuts within
    NEAR of top_p (see top_p_filter), empty when there are none.
    """
    logits = np.asarray(logits, dtype=np.float64)
    if not np.any(np.isfinite(logits)):
        raise ValueError("row has no finite logit")
    z = logits / float(temperature)
    order = nucleus_order(logits, tie_index) if top_p < 1.0 else None
    if cut is not None:
        cut["alts"] = []
    filtered, margin = top_p_filter(z, top_p, order, cut)
    if cut is not None:
        cut["alts"] = [softmax(a) for a in cut["alts"]]
    return softmax(filtered), margin


def inverse_cdf(weights: np.ndarray, u: float):
    """Draw one index from non-negative ``weights`` with the uniform ``u``.

    READING ([P3] §4.2 uses ``torch.multinomial``): the sample is the smallest
    index j whose inclusive prefix sum exceeds u * total, scanning ascending
    token ids.  Zero-weight ids are never chosen; if rounding leaves u * total
    at or above the final prefix, the last positive-weight id is taken.
    Returns (index, margin in u units: distance of u to the nearest edge of
    the chosen index's CDF interval).
    """
    w = np.asarray(weights, dtype=np.float64)
    c = np.cumsum(w)
    total = c[-1]
    if not total > 0.0:
        raise ValueError("no positive weight")
    target = u * total
    hit = np.nonzero(c > target)[0]
    if hit.size:
        j = int(hit[0])
        if w[j] == 0.0:  # cannot happen for a first crossing, kept for clarity
            j = int(np.nonzero(w > 0)[0][-1])
    else:
        j = int(np.nonzero(w > 0)[0][-1])
    lo = c[j - 1] if j > 0 else 0.0
    margin = min(abs(u - lo / total), abs(c[j] / total - u))
    return j, margin


# ---------------------------------------------------------------------------
# EAGLE3 small-vocabulary mapping  ([P1] §六)
# ---------------------------------------------------------------------------

def build_t2d(d2t: np.ndarray, vocab: int) -> np.ndarray:
    """Inverse of d2t: t2d[d2t[j]] = j, every other target id -> -1.

    READING ([P1] §六 only names d2t/t2d): d2t[j] is the absolute target id
    of draft id j, and the map is injective.
    """
    d2t = np.asarray(d2t, dtype=np.int64)
    if d2t.size and (d2t.min() < 0 or d2t.max() >= vocab):
        raise ValueError("d2t entry outside the target vocabulary")
    if np.unique(d2t).size != d2t.size:
        raise ValueError("d2t is not injective")
    t2d = np.full(vocab, -1, dtype=np.int64)
    t2d[d2t] = np.arange(d2t.size)
    return t2d


def d2t_scatter(draft_rows: np.ndarray, d2t: np.ndarray, vocab: int,
                fill: float = -np.inf) -> np.ndarray:
    """[P1] §六: scatter small-vocab draft logits back into the full vocab.

    out[r, d2t[j]] = draft_rows[r, j]; every unmapped target id holds ``fill``
    (-inf: probability 0 after softmax).
    """
    draft_rows = np.atleast_2d(np.asarray(draft_rows, dtype=np.float64))
    out = np.full((draft_rows.shape[0], vocab), fill, dtype=np.float64)
    out[:, np.asarray(d2t, dtype=np.int64)] = draft_rows
    return out


def dist_compact(compact_logits: np.ndarray, d2t: np.ndarray, vocab: int,
                 temperature: float, top_p: float):
    """Draft distribution over the target vocab computed on the compact row.

    Same result as ``dist(d2t_scatter(row))``: the filter runs on the V_d
    compact logits with target ids as the tie key, then the probabilities
    are placed at their target ids.  The tests check the two agree exactly.
    """
    pc, margin = dist(compact_logits, temperature, top_p, tie_index=np.asarray(d2t))
    out = np.zeros(vocab, dtype=np.float64)
    out[np.asarray(d2t, dtype=np.int64)] = pc
    return out, margin


# ---------------------------------------------------------------------------
# Chain verify  ([P3] §3.1 and §4.2, steps 3-5 of generate())
# ---------------------------------------------------------------------------

def verify_chain_row(target_logits: np.ndarray, draft_logits: np.ndarray | None,
                     draft_ids: np.ndarray, u_accept: np.ndarray | None,
                     u_resample: float | None, temperature: float, top_p: float,
                     d2t: np.ndarray | None = None) -> dict:
    """Verify one batch row of a γ-token draft chain.

    target_logits: [γ+1, V] target logits at the γ draft positions plus the
        one after them ([P3] §3.1 "one extra position").
    draft_logits: [γ, V] (or [γ, V_d] with ``d2t``); unused when T == 0.
    draft_ids: [γ] draft tokens as target-vocab ids.
    u_accept: [γ] uniforms for the accept tests; u_resample: one uniform used
        by whichever of the residual resample or the bonus draw happens
        (READING: one per row).

    T > 0 ([P3] §3.1, §4.2):
      p_i = dist(target row i), q_i = dist(draft row i) with the same T and
      top_p ([P3] §6.2).  For i = 0..γ-1, draft x = d_i is accepted iff
      u_i * q_i(x) < p_i(x)  (READING of ``rand < min(1, p/(q + 1e-10))``:
      strict, and the epsilon replaced by the exact product form, which
      accepts q = 0 < p and rejects p = 0).  At the first rejection k the
      token is drawn from max(0, p_k - q_k) (if that mass is 0 -- impossible
      in exact arithmetic -- from p_k); when all γ survive the bonus token is
      drawn from p_γ.
    T == 0 ([P1] §七 ``--temp 0``, [P2] "Match = True"): g_i = argmax of target
      row i (lowest index on ties); accept iff d_i == g_i; the token after the
      accepted prefix is g_k.  Draft logits and uniforms are not used; top_p
      never removes the argmax, so it is ignored.

    Returns dict(tokens [γ+1] int64 (-1 padded), k, p_draft [γ], q_draft [γ],
    margin (smallest decision margin on the path that produced the output),
    near_from (the first output position decided by a decision whose margin
    is below NEAR -- the accept test of draft i decides position i, the draw
    decides position k --; γ+1 when none), pq_margin [γ+1, 2] (top-p margins
    of target row i and draft row i, for every row whose distribution was
    computed; inf otherwise), p_alts / q_alts [γ, ALTS] (p_i(d_i) and
    q_i(d_i) under every admissible cut, the oracle's own first; NaN padded),
    final_alts [ALTS^2] (every token the draw at k gives under the admissible
    cuts of rows k, the oracle's own first; at T == 0 the argmax g_k alone;
    -1 padded), status,
    resample_fallback (bool: residual mass was 0)).

    Margins and alternatives (reporting only; no result depends on them).  A
    top-p cut whose deciding cumulative sum lies within NEAR of top_p could
    come out one rank shorter or longer under rounding (top_p_filter's
    "alts"); every accept test and the draw are taken under each admissible
    pair (target cut, draft cut) of their row.  An accept test whose outcome
    differs between pairs has margin 0; otherwise its margin is the smallest
    |u - p/q| over the pairs.  The draw's margin is the smallest over the
    pairs, and the tokens it gives are listed in final_alts.
    """
    target_logits = np.asarray(target_logits, dtype=np.float64)
    gamma = target_logits.shape[0] - 1
    vocab = target_logits.shape[1]
    ids = np.asarray(draft_ids, dtype=np.int64)
    tokens = np.full(gamma + 1, -1, dtype=np.int64)
    res = dict(tokens=tokens, k=0, p_draft=np.zeros(gamma), q_draft=np.zeros(gamma),
               margin=np.inf, near_from=gamma + 1, pq_margin=np.full((gamma + 1, 2), np.inf),
               p_alts=np.full((gamma, ALTS), np.nan), q_alts=np.full((gamma, ALTS), np.nan),
               final_alts=np.full(ALTS * ALTS, -1, np.int64), status=0, resample_fallback=False)

    if np.any((ids < 0) | (ids >= vocab)):
        res["status"] = STATUS_BAD_DRAFT_ID
        return res
    if not np.all(np.any(np.isfinite(target_logits), axis=1)):
        res["status"] = STATUS_EMPTY_ROW
        return res

    if temperature == 0.0:
        g = np.argmax(target_logits, axis=1)  # first maximum: lowest index on ties
        k = gamma
        for i in range(gamma):
            if ids[i] != g[i]:
                k = i
                break
        tokens[:k] = ids[:k]
        tokens[k] = g[k]
        res["final_alts"][0] = g[k]
        res["k"] = k
        return res

    draft_logits = np.asarray(draft_logits, dtype=np.float64)
    if not np.all(np.any(np.isfinite(draft_logits), axis=1)):
        res["status"] = STATUS_EMPTY_ROW
        return res
    margins = []   # margin of every decision on the output's path
    decides = []   # the output position each of those decisions decides
    cands = {}     # (i, 0 target / 1 draft) -> [own distribution, admissible alternatives]

    def p_row(i):
        cut = {}
        p, mg = dist(target_logits[i], temperature, top_p, cut=cut)
        cands[(i, 0)] = [p] + cut["alts"]
        res["pq_margin"][i, 0] = mg
        return p

    def q_row(i):
        cut = {}
        if d2t is None:
            q, mg = dist(draft_logits[i], temperature, top_p, cut=cut)
        else:
            scattered = d2t_scatter(draft_logits[i], d2t, vocab)[0]
            q, mg = dist(scattered, temperature, top_p, cut=cut)
        cands[(i, 1)] = [q] + cut["alts"]
        res["pq_margin"][i, 1] = mg
        return q

    def record(i, x):
        """p_i(x), q_i(x) under the row's own and admissible cuts."""
        for key, col in (("p", 0), ("q", 1)):
            vals = [d[x] for d in cands[(i, col)]]
            res[key + "_draft"][i] = vals[0]
            res[key + "_alts"][i, :len(vals)] = vals

    k = gamma
    p_k = q_k = None
    for i in range(gamma):
        p_i, q_i = p_row(i), q_row(i)
        x = ids[i]
        record(i, x)
        accept = u_accept[i] * q_i[x] < p_i[x]
        outcomes, mg = set(), np.inf
        for p in cands[(i, 0)]:
            for q in cands[(i, 1)]:
                outcomes.add(bool(u_accept[i] * q[x] < p[x]))
                if q[x] > 0.0:
                    mg = min(mg, abs(float(u_accept[i]) - p[x] / q[x]))
        margins.append(0.0 if len(outcomes) > 1 else mg)
        decides.append(i)
        if not accept:
            k = i
            p_k, q_k = p_i, q_i
            break

    def draw(p, q):
        """(token, margin, fallback) of the draw at k under one pair of cuts."""
        if q is None:                           # bonus token from p_γ, [P3] §3.1
            return inverse_cdf(p, float(u_resample)) + (False,)
        residual = np.maximum(0.0, p - q)       # norm(max(0, p - q)), [P3] §3.1
        if residual.sum() > 0.0:
            return inverse_cdf(residual, float(u_resample)) + (False,)
        return inverse_cdf(p, float(u_resample)) + (True,)

    if k < gamma:
        # The remaining positions are still scored by the target ([P3] §4.2
        # computes every position before deciding); record p/q for them.
        for i in range(k + 1, gamma):
            p_row(i), q_row(i)
            record(i, ids[i])
        pairs = [(p, q) for p in cands[(k, 0)] for q in cands[(k, 1)]]
    else:
        p_row(gamma)
        pairs = [(p, None) for p in cands[(gamma, 0)]]
    finals = [draw(p, q) for p, q in pairs]
    tok, _, res["resample_fallback"] = finals[0]
    margins.append(min(f[1] for f in finals))
    decides.append(k)
    alts = list(dict.fromkeys(f[0] for f in finals))
    res["final_alts"][:len(alts)] = alts
    tokens[:k] = ids[:k]
    tokens[k] = tok
    res["k"] = k
    res["margin"] = float(min(margins)) if margins else np.inf
    near = [pos for mg_, pos in zip(margins, decides) if mg_ < NEAR]
    res["near_from"] = min(near) if near else gamma + 1
    return res


def verify_chain(target_logits, draft_logits, draft_ids, u_accept, u_resample,
                 temperature, top_p, d2t=None, rows=None) -> dict:
    """Batched verify ([P3] §6.2: each row stops at its own first rejection).

    Shapes: target [B, γ+1, V]; draft [B, γ, V or V_d]; draft_ids [B, γ];
    u_accept [B, γ]; u_resample [B].  ``rows`` restricts the work to a list of
    batch rows (the others are left at -1 / 0).
    """
    target_logits = np.asarray(target_logits)
    B, gp1, _ = target_logits.shape
    gamma = gp1 - 1
    rows = range(B) if rows is None else rows
    out = dict(tokens=np.full((B, gp1), -1, np.int64), num_accepted=np.zeros(B, np.int64),
               p_draft=np.zeros((B, gamma)), q_draft=np.zeros((B, gamma)),
               margin=np.full(B, np.inf), near_from=np.full(B, gp1, np.int64),
               pq_margin=np.full((B, gp1, 2), np.inf), p_alts=np.full((B, gamma, ALTS), np.nan),
               q_alts=np.full((B, gamma, ALTS), np.nan), final_alts=np.full((B, ALTS * ALTS), -1, np.int64),
               status=np.zeros(B, np.int64),
               resample_fallback=np.zeros(B, bool))
    for b in rows:
        r = verify_chain_row(
            target_logits[b], None if draft_logits is None else np.asarray(draft_logits[b]),
            np.asarray(draft_ids)[b], None if u_accept is None else np.asarray(u_accept)[b],
            None if u_resample is None else float(np.asarray(u_resample)[b]),
            temperature, top_p, d2t)
        out["tokens"][b] = r["tokens"]
        out["num_accepted"][b] = r["k"]
        out["p_draft"][b] = r["p_draft"]
        out["q_draft"][b] = r["q_draft"]
        out["margin"][b] = r["margin"]
        out["near_from"][b] = r["near_from"]
        out["pq_margin"][b] = r["pq_margin"]
        out["p_alts"][b] = r["p_alts"]
        out["q_alts"][b] = r["q_alts"]
        out["final_alts"][b] = r["final_alts"]
        out["status"][b] = r["status"]
        out["resample_fallback"][b] = r["resample_fallback"]
    return out


# ---------------------------------------------------------------------------
# Draft-side sampling of one position ([P3] §3.1 drafting, §4.2 draft loop)
# ---------------------------------------------------------------------------

def sample_row(logits: np.ndarray, temperature: float, top_p: float, u: float,
               tie_index: np.ndarray | None = None, alts: list | None = None):
    """One token from dist(logits, T, top_p) with the uniform u.

    [P3] §4.2 draft loop: ``/ temperature`` -> ``_apply_top_p`` -> softmax ->
    ``multinomial``; T == 0 is the argmax (lowest index on ties).
    Returns (token, margin); the margin includes the top-p cut's own.

    When ``alts`` is a list (reporting only, as for the chain verify's
    final_alts) it receives (token, its probability) for the oracle's own cut
    and for every other cut within NEAR of top_p (top_p_filter's "alts"), and
    the margin returned is the draw's smallest margin over those cuts, without
    the cut's own.
    """
    logits = np.asarray(logits, dtype=np.float64)
    if temperature == 0.0:
        tok = int(np.argmax(logits))
        if alts is not None:
            alts.append((tok, 1.0))
        return tok, np.inf
    cut = {} if alts is not None else None
    p, mg_top = dist(logits, temperature, top_p, tie_index, cut=cut)
    tok, mg = inverse_cdf(p, u)
    if alts is None:
        return tok, min(mg, mg_top)
    alts.append((tok, float(p[tok])))
    for q in cut["alts"]:
        t2, m2 = inverse_cdf(q, u)
        alts.append((t2, float(q[t2])))
        mg = min(mg, m2)
    return tok, mg


# ---------------------------------------------------------------------------
# Greedy token-tree verify ([P2] §5 draft tree; headline "Match = True")
# ---------------------------------------------------------------------------

def verify_tree_row(logits: np.ndarray, parents: np.ndarray, tokens: np.ndarray,
                    max_depth: int) -> dict:
    """Greedy verify of one draft tree.

    logits [N, V]: target logits at every node; the row of node n predicts the
    token after n's root path.  parents [N]: parents[0] = -1 (node 0 is the
    root, the last committed token, not itself verified), parents[n] < n.
    tokens [N]: node tokens (tokens[0] unused).

    READING of [P2] §5 and the greedy benchmark: a node is accepted when its
    parent is accepted and its token equals the argmax of the parent's row
    (lowest index on argmax ties).  The output is the deepest accepted node
    (lowest node id among equally deep ones), its root path, and the bonus
    token argmax(row of that node).  With distinct sibling tokens at most
    one child matches at each step, so this is the unique accepted chain.

    Returns dict(accept_len, path [max_depth+1] node ids from the root (-1
    padded), out_tokens [max_depth+1] (path tokens then bonus, -1 padded),
    status).
    """
    logits = np.asarray(logits, dtype=np.float64)
    parents = np.asarray(parents, dtype=np.int64)
    tokens = np.asarray(tokens, dtype=np.int64)
    N, V = logits.shape
    L = max_depth + 1
    res = dict(accept_len=0, path=np.full(L, -1, np.int64),
               out_tokens=np.full(L, -1, np.int64), status=0)
    status = 0
    if parents[0] != -1:
        status |= STATUS_BAD_PARENT
    for n in range(1, N):
        if not (0 <= parents[n] < n):
            status |= STATUS_BAD_PARENT
        if not (0 <= tokens[n] < V):
            status |= STATUS_BAD_TOKEN
    depth = np.zeros(N, np.int64)
    if not status & STATUS_BAD_PARENT:
        for n in range(1, N):
            depth[n] = depth[parents[n]] + 1
        if depth.max() > max_depth:
            status |= STATUS_DEPTH_EXCEEDED
    if not np.all(np.any(np.isfinite(logits), axis=1)):
        status |= STATUS_EMPTY_ROW
    if status:
        res["status"] = status
        return res
    g = np.argmax(logits, axis=1)
    accepted = np.zeros(N, bool)
    accepted[0] = True
    for n in range(1, N):
        accepted[n] = accepted[parents[n]] and tokens[n] == g[parents[n]]
    best = 0
    for n in range(N):
        if accepted[n] and depth[n] > depth[best]:
            best = n
    chain = []
    n = best
    while n != -1:
        chain.append(n)
        n = parents[n]
    chain.reverse()
    d = depth[best]
    res["accept_len"] = int(d)
    res["path"][: d + 1] = chain
    res["out_tokens"][:d] = tokens[chain[1:]]
    res["out_tokens"][d] = g[best]
    return res


def verify_tree(logits, parents, tokens, max_depth, rows=None) -> dict:
    """Batched greedy tree verify: logits [B, N, V], parents/tokens [B, N]."""
    logits = np.asarray(logits)
    B = logits.shape[0]
    L = max_depth + 1
    out = dict(accept_len=np.zeros(B, np.int64), path=np.full((B, L), -1, np.int64),
               out_tokens=np.full((B, L), -1, np.int64), status=np.zeros(B, np.int64))
    for b in (range(B) if rows is None else rows):
        r = verify_tree_row(logits[b], np.asarray(parents)[b], np.asarray(tokens)[b], max_depth)
        out["accept_len"][b] = r["accept_len"]
        out["path"][b] = r["path"]
        out["out_tokens"][b] = r["out_tokens"]
        out["status"][b] = r["status"]
    return out


# ---------------------------------------------------------------------------
# Token-tree speculative sampling verify (T > 0) over the [P2] §5 tree shape
# ---------------------------------------------------------------------------

def _tree_checks(parents: np.ndarray, tokens: np.ndarray, vocab: int, max_depth: int):
    """Status bits of a tree's shape and tokens, and node depths."""
    N = parents.shape[0]
    status = 0
    if parents[0] != -1:
        status |= STATUS_BAD_PARENT
    for n in range(1, N):
        if not (0 <= parents[n] < n):
            status |= STATUS_BAD_PARENT
        if not (0 <= tokens[n] < vocab):
            status |= STATUS_BAD_TOKEN
    depth = np.zeros(N, np.int64)
    if not status & STATUS_BAD_PARENT:
        for n in range(1, N):
            depth[n] = depth[parents[n]] + 1
        if depth.max() > max_depth:
            status |= STATUS_DEPTH_EXCEEDED
    return status, depth


def verify_tree_sample_row(target_logits: np.ndarray, draft_logits: np.ndarray,
                           parents: np.ndarray, tokens: np.ndarray,
                           u_accept: np.ndarray, u_final: float,
                           temperature: float, top_p: float, max_depth: int,
                           trace: list | None = None) -> dict:
    """Speculative-sampling verify of one draft token tree.

    target_logits [N, V]: the target's logits at every node (row n predicts
    the token after n's root path, as in the greedy tree).  draft_logits
    [N, V]: the draft's logits at every node; n's children are the draft's
    samples from dist(draft row n).  parents/tokens as for the greedy tree.
    u_accept [N]: the uniform of each node's accept test (entry 0 unused).
    u_final: one uniform for the token drawn after the accepted path.

    READING (the pages give the tree's shape, [P2] §5, and the rule for one
    draft per position, [P3] §3.1, but no rule for several drafts at one
    position): sequential per-child rejection with a residual update.  At an
    accepted node with p = dist(target row), q = dist(draft row) (same T and
    top_p, [P3] §6.2) the residual starts as r = p.  The children are tested
    in increasing node order: a child with token x is accepted iff
    u * q(x) < r(x) (the chain's rule with p replaced by r); a rejection
    replaces r by norm(max(0, r - q)) (if that has no mass -- impossible in
    exact arithmetic for a child the draft could have drawn -- r is kept and
    the fallback bit is set).  The first accepted child becomes the current
    node.  When every child is rejected the last token is drawn from r; at a
    node without children it is the bonus token drawn from p.  Every test is
    one-draft speculative sampling against the current residual, so the
    emitted tokens follow the target whenever each node's children are
    independent draws from that node's q.

    ``trace`` (optional list) receives one dict per accept test (node,
    token, threshold = min(1, r(x)/q(x)) -- 1 when q(x) = 0 < r(x) --,
    accepted) and a final dict(final=True, weights) with the distribution
    the last token was drawn from.

    Returns dict(accept_len, path [max_depth+1], out_tokens [max_depth+1]
    (-1 padded), status, margin, resample_fallback, final_alts [ALTS^2]
    (every token the final draw gives under the admissible cuts, the
    oracle's own first; -1 padded)).

    Margins and alternatives (reporting only; no result depends on them), as
    for the chain: a top-p cut within NEAR of top_p could come out one rank
    shorter or longer (top_p_filter's "alts"), and each node's children are
    tested under every admissible pair (target cut, draft cut) of the node.
    When the pairs accept different children (or one accepts and another
    none) the node's margin is 0; otherwise the margin is the smallest
    |u - r(x)/q(x)| over the pairs' tests, and the final draw's the smallest
    over the pairs, whose tokens are listed in final_alts.
    """
    target_logits = np.asarray(target_logits, dtype=np.float64)
    draft_logits = np.asarray(draft_logits, dtype=np.float64)
    parents = np.asarray(parents, dtype=np.int64)
    tokens = np.asarray(tokens, dtype=np.int64)
    N, V = target_logits.shape
    L = max_depth + 1
    res = dict(accept_len=0, path=np.full(L, -1, np.int64), out_tokens=np.full(L, -1, np.int64),
               status=0, margin=np.inf, resample_fallback=False, final_alts=np.full(ALTS * ALTS, -1, np.int64))
    status, _ = _tree_checks(parents, tokens, V, max_depth)
    if not (np.all(np.any(np.isfinite(target_logits), axis=1))
            and np.all(np.any(np.isfinite(draft_logits), axis=1))):
        status |= STATUS_EMPTY_ROW
    if status:
        res["status"] = status
        return res

    def children_pass(node, p, q, log):
        """Test node's children against r = p under one pair of cuts.
        Returns (accepted child or None, final r, margins, fallback)."""
        r = p.copy()
        mgs, fallback = [], False
        for c in range(node + 1, N):
            if parents[c] != node:
                continue
            x = tokens[c]
            u = float(u_accept[c])
            accept = u * q[x] < r[x]
            if q[x] > 0.0:
                threshold = min(1.0, r[x] / q[x])
                mgs.append(abs(u - r[x] / q[x]))
            else:
                threshold = 1.0 if r[x] > 0.0 else 0.0
            if log is not None:
                log.append(dict(node=c, token=int(x), threshold=threshold, accepted=bool(accept)))
            if accept:
                return c, r, mgs, fallback
            residual = np.maximum(0.0, r - q)
            if residual.sum() > 0.0:
                r = residual / residual.sum()
            else:
                fallback = True
        return None, r, mgs, fallback

    margins = []
    node, chain = 0, [0]
    while True:
        cut_p, cut_q = {}, {}
        p, _ = dist(target_logits[node], temperature, top_p, cut=cut_p)
        q, _ = dist(draft_logits[node], temperature, top_p, cut=cut_q)
        passes = [children_pass(node, pp, qq, trace if (pp is p and qq is q) else None)
                  for pp in [p] + cut_p["alts"] for qq in [q] + cut_q["alts"]]
        nxt, r, _, fallback = passes[0]
        res["resample_fallback"] |= fallback
        for other in passes:
            margins += other[2]
        if any(other[0] != nxt for other in passes):
            margins.append(0.0)            # the accepted child depends on the cut
        if nxt is None:
            break
        node = nxt
        chain.append(node)
    # r is p when the node has no children, else the residual after the last rejection.
    draws = [inverse_cdf(other[1], float(u_final)) for other in passes]
    tok = draws[0][0]
    margins.append(min(mg for _, mg in draws))
    alts = list(dict.fromkeys(t for t, _ in draws))
    res["final_alts"][:len(alts)] = alts
    if trace is not None:
        trace.append(dict(final=True, weights=r / r.sum()))
    d = len(chain) - 1
    res["accept_len"] = d
    res["path"][: d + 1] = chain
    res["out_tokens"][:d] = tokens[chain[1:]]
    res["out_tokens"][d] = tok
    res["margin"] = float(min(margins))
    return res


def verify_tree_sample(target_logits, draft_logits, parents, tokens, u_accept, u_final,
                       temperature, top_p, max_depth, rows=None) -> dict:
    """Batched tree sampling verify: logits [B, N, V], parents/tokens/u_accept
    [B, N], u_final [B]."""
    target_logits = np.asarray(target_logits)
    B = target_logits.shape[0]
    L = max_depth + 1
    out = dict(accept_len=np.zeros(B, np.int64), path=np.full((B, L), -1, np.int64),
               out_tokens=np.full((B, L), -1, np.int64), status=np.zeros(B, np.int64),
               margin=np.full(B, np.inf), resample_fallback=np.zeros(B, bool),
               final_alts=np.full((B, ALTS * ALTS), -1, np.int64))
    for b in (range(B) if rows is None else rows):
        r = verify_tree_sample_row(target_logits[b], np.asarray(draft_logits)[b], np.asarray(parents)[b],
                                   np.asarray(tokens)[b], np.asarray(u_accept)[b],
                                   float(np.asarray(u_final)[b]), temperature, top_p, max_depth)
        for k in ("accept_len", "path", "out_tokens", "status", "margin", "resample_fallback", "final_alts"):
            out[k][b] = r[k]
    return out


# ---------------------------------------------------------------------------
# Top-k node expansion of a draft tree ([P2] §5: every node expanded into its
# top_k draft tokens)
# ---------------------------------------------------------------------------

def top_k(logits: np.ndarray, k: int) -> np.ndarray:
    """The ids of the k highest logits of a row, in descending logit order,
    equal logits by lower id (the same ranking as the top-p filter).  -inf
    logits rank last, by id.  Requires 1 <= k <= len(row)."""
    logits = np.asarray(logits, dtype=np.float64)
    return nucleus_order(logits)[:k].astype(np.int64)
