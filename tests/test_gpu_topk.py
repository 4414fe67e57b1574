"""Top-k node expansion (sv_topk) on the GPU against the fp64 oracle: ids
bit-exact (descending logit, equal logits by lower id), values equal to the
row's logits at those ids; rows with many ties, -inf entries, odd lengths
and rows that do not start on a 16-byte boundary."""
import numpy as np
import pytest

import synth
from oracle import sv_oracle as O

from _parity import logits_tensor

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    import __graft_entry__
    __graft_entry__.build()
    import draft_token_verification_sv_gb300 as sv
    return sv


def _check(sv, rows, dtype, k):
    import torch
    store = synth.to_bf16_bits(rows) if dtype == "bf16" else np.ascontiguousarray(rows, np.float32)
    exact = synth.bf16_bits_to_f32(store) if dtype == "bf16" else store
    ids, vals = sv.topk(logits_tensor(store, dtype), k, values=True)
    torch.cuda.synchronize()
    ids, vals = ids.cpu().numpy(), vals.cpu().numpy()
    for r in range(rows.shape[0]):
        want = O.top_k(exact[r], k)
        assert ids[r].tolist() == want.tolist(), (r, ids[r], want)
        np.testing.assert_array_equal(vals[r], exact[r][want].astype(np.float32))


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("V,k", [(1, 1), (7, 5), (1000, 8), (4097, 16), (49152, 8), (128256, 8), (151936, 10)])
def test_topk_random_rows(sv, dtype, V, k):
    g = np.random.default_rng(V + k)
    rows = g.normal(0, 3, (9, V)).astype(np.float32)
    rows[1::3] = np.round(rows[1::3])          # many ties
    rows[2, g.integers(0, V, size=max(1, V // 2))] = -np.inf
    _check(sv, rows, dtype, k)


def test_topk_all_equal_and_mostly_neg_inf(sv):
    rows = np.zeros((3, 5000), np.float32)
    rows[1] = -np.inf
    rows[1, [4999, 17, 3000]] = 1.0
    rows[2] = -np.inf
    _check(sv, rows, "f32", 16)
    _check(sv, rows, "bf16", 8)


def test_topk_unaligned_rows(sv):
    g = np.random.default_rng(5)
    for V in (1001, 32003):
        rows = g.normal(0, 2, (5, V)).astype(np.float32)
        _check(sv, rows, "f32", 8)
        _check(sv, rows, "bf16", 8)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_topk_weak_first_batch(sv, dtype):
    """The lower bound taken from the start of the row is far below the
    answer: a thousand planted winners late in the row (a long candidate
    list), a rising row and a row of one repeated value (the list
    overflows and the whole row is searched)."""
    g = np.random.default_rng(11)
    V = 128256
    rows = g.normal(0, 1, (4, V)).astype(np.float32)
    late = g.choice(np.arange(40000, V), size=1000, replace=False)
    rows[0, late] = g.uniform(5, 9, size=late.size)
    rows[1] = np.linspace(-4, 4, V, dtype=np.float32)
    rows[2] = 0.5
    rows[3, :20000] = -np.inf
    _check(sv, rows, dtype, 16)
    _check(sv, rows, dtype, 3)


def test_topk_nan_logits_never_chosen(sv):
    import torch
    rows = np.full((2, 300), np.nan, np.float32)
    rows[0, [7, 150, 299]] = [1.0, 3.0, 2.0]
    rows[1, :] = np.arange(300, dtype=np.float32)
    rows[1, 299] = np.nan
    ids, vals = sv.topk(logits_tensor(rows, "f32"), 5, values=True)
    torch.cuda.synchronize()
    ids, vals = ids.cpu().numpy(), vals.cpu().numpy()
    assert ids[0].tolist() == [150, 299, 7, -1, -1]
    assert np.all(np.isnan(vals[0, 3:])) and vals[0, :3].tolist() == [3.0, 2.0, 1.0]
    assert ids[1].tolist() == [298, 297, 296, 295, 294]
