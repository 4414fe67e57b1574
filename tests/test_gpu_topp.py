"""The filtered distribution softmax(top_p_filter(l / T)) on the GPU against
the fp64 oracle, element by element: random rows over the pages' vocabulary
sizes, and rows built to reach every branch of the threshold search (the
common binned path, a candidate list overflow, a cut among masses below
2^-30, and a tie group of more than 64 equal logits at the cut)."""
import numpy as np
import pytest

import synth
from oracle import sv_oracle as O

from _parity import TOL, logits_tensor

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    import __graft_entry__
    __graft_entry__.build()
    import draft_token_verification_sv_gb300 as sv
    return sv


def _check(sv, rows, dtype, T, top_p, tie_index=None):
    import torch
    if dtype == "bf16":
        store = synth.to_bf16_bits(rows)
        rows = synth.bf16_bits_to_f32(store)
    else:
        store = np.ascontiguousarray(rows, dtype=np.float32)
        rows = store
    got = sv.softmax_topp(logits_tensor(store, dtype), T, top_p)
    torch.cuda.synchronize()
    got = got.cpu().numpy().astype(np.float64)
    near = 0
    for r in range(rows.shape[0]):
        cut = {}
        want, margin = O.dist(rows[r], T, top_p, cut=cut)

        def matches(w):
            same_set = ((got[r] > 0) == (w > 0)) | (w < 1e-30)
            ok = np.abs(got[r] - w) <= np.maximum(1e-12, TOL[dtype] * w)
            return bool(same_set.all() and ok.all())

        if matches(want):
            continue
        # Not the oracle's own cut: one of the cuts within 1e-6 of top_p
        # (one rank shorter or longer), exactly.
        if any(matches(w) for w in cut["alts"]):
            near += 1
            continue
        # Several ranks within 1e-6 of top_p (masses below 1e-6 at the cut):
        # the kept sets may differ at the boundary only, by at most 2e-6 of
        # unfiltered mass; the common ids agree up to the kept mass they are
        # normalised by.
        assert margin < O.NEAR, (r, margin)
        near += 1
        both = (got[r] > 0) & (want > 0)
        pi, _ = O.dist(rows[r], T, 1.0)          # unfiltered softmax
        differ = (got[r] > 0) != (want > 0)
        assert pi[differ].sum() <= 2e-6, pi[differ].sum()
        scale = got[r][both].sum() / want[both].sum()
        np.testing.assert_allclose(got[r][both], want[both] * scale, rtol=TOL[dtype], atol=1e-12)
    return near


@pytest.mark.parametrize("V,dtype,T,top_p", [
    (1, "f32", 1.0, 0.5), (7, "bf16", 0.7, 0.9), (1000, "f32", 0.8, 0.9), (4097, "bf16", 1.3, 0.5),
    (32000, "f32", 1.0, 0.95), (49152, "bf16", 0.8, 0.9), (128256, "bf16", 1.0, 0.99),
    (151936, "f32", 1.0, 0.95), (151936, "f32", 0.5, 0.1), (50257, "bf16", 1.0, 0.9),
])
def test_random_rows(sv, V, dtype, T, top_p):
    g = np.random.default_rng(V + int(top_p * 100))
    R = 12
    rows = g.normal(0, 2.5, (R, V)).astype(np.float32)
    rows[::3] *= 4.0          # some peaked rows
    rows[1::4] = np.round(rows[1::4])  # some with many ties
    _check(sv, rows, dtype, T, top_p)


def test_candidate_overflow_path(sv):
    """Nearly all logits equal: the cut bin holds far more than one block's
    candidate list, so the exact generic select runs."""
    g = np.random.default_rng(1)
    rows = np.zeros((4, 30000), np.float32)
    for r in range(4):
        rows[r, g.choice(30000, 10, replace=False)] = 1.0
    _check(sv, rows, "f32", 1.0, 0.49991)
    _check(sv, rows, "bf16", 1.0, 0.3)


def test_cut_among_tiny_masses(sv):
    """One dominant logit and a long tail below 2^-30.5 of its mass: with
    top_p close to 1 the cut falls in the open bin."""
    rows = np.full((3, 150000), -21.5, np.float32)
    rows[:, 17] = 0.0
    rows[1, 100:200] = -21.0
    _check(sv, rows, "bf16", 1.0, 0.99999)
    _check(sv, rows, "f32", 1.0, 0.99999)


def test_large_tie_group_at_cut(sv):
    """More than 64 equal logits straddle the cut: the tie group is cut by
    index."""
    g = np.random.default_rng(2)
    rows = np.full((4, 50000), -3.0, np.float32)
    for r in range(4):
        idx = g.permutation(50000)
        rows[r, idx[:100]] = 5.0
        rows[r, idx[100:1100]] = 4.0
    for top_p in (0.3, 0.6, 0.9):
        _check(sv, rows, "bf16", 1.0, top_p)
        _check(sv, rows, "f32", 1.0, top_p)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_slice_cuts_far_from_the_row_cut(sv, dtype):
    """Rows where one stretch of logits sits far above the rest: the other
    slices' own cuts lie far from the row's, so where they hold logits in the
    row's cut bin those are read by the rescan; plus rows where one slice is
    far below the rest (its bins lie under the row's window)."""
    g = np.random.default_rng(23)
    V, R = 151936, 8
    rows = g.normal(0, 1.5, (R, V)).astype(np.float32)
    rows[0, 20000:40000] += 6.0
    rows[1, :9000] += 4.0
    rows[2, 100000:] -= 30.0
    rows[3, 50000:60000] -= 80.0
    rows[4, ::3] += 2.5
    rows[5] = np.round(rows[5] * 4) / 4   # ties
    rows[6, 70000:] = -np.inf
    for T, top_p in ((1.0, 0.9), (0.6, 0.5), (2.0, 0.99)):
        _check(sv, rows, dtype, T, top_p)


def test_unaligned_rows(sv):
    """Rows whose start is not 16-byte aligned (odd row length, packed)."""
    g = np.random.default_rng(3)
    for V in (1001, 32003, 151937):
        rows = g.normal(0, 2, (5, V)).astype(np.float32)
        _check(sv, rows, "f32", 0.9, 0.9)
        _check(sv, rows, "bf16", 0.9, 0.9)


@pytest.mark.parametrize("shift,T", [(4.0e5, 1.0), (-4.0e5, 1.0), (2.0e4, 0.01), (3.0e5, 0.5)])
def test_large_logits_take_the_conversion_path(sv, shift, T):
    """Logits so large that 8 * l * log2(e) / T leaves the range where the
    bins are computed by magic-number additions (|floor| >= 4e6): those
    slices are binned by floorf and conversions.  Rows mix such slices with
    ordinary ones, and the values keep a spread of a few units (exactly
    representable in fp32 at this magnitude), so the cut still falls among
    many logits."""
    g = np.random.default_rng(int(abs(shift)) + 7)
    V = 40000
    rows = np.round(g.normal(0, 2, (4, V)) * 64) / 64
    rows = (rows + shift).astype(np.float32)
    rows[1, : V // 2] = np.round(g.normal(0, 2, V // 2) * 64) / 64   # ordinary slices in the same row
    rows[3] = np.round(rows[3])                                        # ties
    _check(sv, rows, "f32", T, 0.9)
