"""Greedy tree verify along the accepted frontier (sv_verify_tree_path) on
the GPU against the fp64 oracle and against the all-node verify: the full
tree workload, small trees with ties and duplicate sibling tokens (frontiers
of several nodes), invalid trees, and rows with no finite logit on and off
the walked path."""
import numpy as np
import pytest

import synth
from oracle import sv_oracle as O

from _parity import logits_tensor, t

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    import __graft_entry__
    __graft_entry__.build()
    import draft_token_verification_sv_gb300 as sv
    return sv


def _run(sv, tr, dtype="bf16", path_walk=True):
    import torch
    logits = logits_tensor(tr["logits_store"], dtype)
    got = sv.verify_tree(logits, t(tr["parents"]), t(tr["tokens"]), tr["max_depth"], path_walk=path_walk)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in got.items()}


def _compare(got, want):
    assert np.array_equal(got["accept_len"], want["accept_len"])
    assert np.array_equal(got["out_tokens"], want["out_tokens"])
    assert np.array_equal(got["path"], want["path"])
    assert np.array_equal(got["row_status"] != 0, want["status"] != 0)


def test_path_full_workload(sv):
    """64 trees x 32 nodes, V = 128256 bf16: same result as the oracle and
    as the all-node verify."""
    tr = synth.make_tree_inputs(synth.TREE)
    got = _run(sv, tr)
    want = O.verify_tree(tr["logits"], tr["parents"], tr["tokens"], tr["max_depth"])
    _compare(got, want)
    allnode = _run(sv, tr, path_walk=False)
    for k in ("accept_len", "path", "out_tokens", "row_status"):
        assert np.array_equal(got[k], allnode[k]), k
    assert got["accept_len"].max() >= 2


@pytest.mark.parametrize("N,V,D,dtype", [(1, 5, 0, "bf16"), (2, 3, 1, "f32"), (12, 4, 4, "bf16"),
                                         (32, 7, 5, "f32"), (600, 3, 64, "bf16"), (1024, 2, 12, "f32")])
def test_path_small_with_ties(sv, N, V, D, dtype):
    """Rounded logits (ties everywhere) and many children planted on their
    parent's argmax, so sibling tokens repeat and several nodes of one
    depth are accepted at once."""
    cfg = synth.TreeConfig("t", 5, N, V, dtype, D, 8 if N <= 32 else 64, 1.0, 0.8, 0.0)
    tr = synth.make_tree_inputs(cfg, seed=N * 7 + V)
    q = np.round(tr["logits"]).astype(np.float32)
    tr["logits"] = q
    tr["logits_store"] = synth.to_bf16_bits(q) if dtype == "bf16" else q
    for b in range(tr["batch"]):
        for n in range(1, N):
            if n % 3:
                tr["tokens"][b, n] = int(np.argmax(q[b, tr["parents"][b, n]]))
    got = _run(sv, tr, dtype)
    want = O.verify_tree(tr["logits"], tr["parents"], tr["tokens"], tr["max_depth"])
    _compare(got, want)


def test_path_invalid_trees(sv):
    tr = synth.make_tree_inputs(synth.TREE, batch=4, vocab=257)
    tr["parents"][1, 5] = 9          # parent after child
    tr["parents"][2, 0] = 0          # root with a parent
    tr["tokens"][3, 4] = 257         # token out of range
    got = _run(sv, tr)
    assert got["row_status"][1] & O.STATUS_BAD_PARENT and got["row_status"][2] & O.STATUS_BAD_PARENT
    assert got["row_status"][3] & O.STATUS_BAD_TOKEN
    for b in (1, 2, 3):
        assert got["accept_len"][b] == 0 and np.all(got["out_tokens"][b] == -1) and np.all(got["path"][b] == -1)
    want = O.verify_tree(tr["logits"], tr["parents"], tr["tokens"], tr["max_depth"])
    _compare({k: v[:1] for k, v in got.items()}, {k: v[:1] for k, v in want.items()})
    cfg = synth.TreeConfig("chain", 1, 8, 50, "f32", 7, 1, 1.0, 1.0, 16.0)
    deep = synth.make_tree_inputs(cfg, seed=1)
    deep["max_depth"] = 3
    g = _run(sv, deep, "f32")
    assert g["row_status"][0] & O.STATUS_DEPTH_EXCEEDED


def test_path_rows_without_finite_logit(sv):
    """A row the walk reads with no finite logit flags the tree; one off the
    walked path is never read, and the result is the oracle's for the tree
    with that row restored."""
    tr = synth.make_tree_inputs(synth.TREE, batch=2, vocab=1000)
    want = O.verify_tree(tr["logits"], tr["parents"], tr["tokens"], tr["max_depth"])
    on, off = tr.copy(), tr.copy()
    on_logits = tr["logits"].copy()
    on_logits[0, 0] = -np.inf                            # the root row: always read
    on["logits"], on["logits_store"] = on_logits, synth.to_bf16_bits(on_logits)
    g = _run(sv, on)
    assert g["row_status"][0] & O.STATUS_EMPTY_ROW and g["accept_len"][0] == 0
    assert np.all(g["out_tokens"][0] == -1)
    walked = set(int(n) for n in want["path"][1] if n >= 0)
    spare = [n for n in range(tr["nodes"]) if n not in walked]
    off_logits = tr["logits"].copy()
    off_logits[1, spare[-1]] = -np.inf
    off["logits"], off["logits_store"] = off_logits, synth.to_bf16_bits(off_logits)
    g = _run(sv, off)
    assert g["row_status"][1] == 0
    for k in ("accept_len", "path", "out_tokens"):
        assert np.array_equal(g[k][1], want[k][1]), k
