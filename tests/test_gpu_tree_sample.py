"""Speculative-sampling tree verify (sv_verify_tree_sample) on the GPU
against the fp64 oracle: the full tree workload, top-p and T != 1, trees
with many siblings on tiny vocabularies (long runs of rejections, repeated
tokens), ragged and unaligned rows, vocabularies of more than 256 chunks,
the zero-residual fallback, and invalid trees.

The path, accept length and every emitted token must equal the oracle's,
whether a tree is walked by one thread block or by a cluster of two that
splits every residual pass.
The final token may be any that the oracle's draw gives under the top-p cuts
within 1e-6 of top_p (one rank shorter or longer).  A tree may differ
otherwise only where one of the oracle's decisions on it, under one of those
cuts, lies within NEAR = 1e-6 of its threshold (in units of the uniform), the
same margin as the chain verify.  The GPU takes each accept test in double (p(x)
and q(x) with the double-precision exp2), forms the residual max(0, p - c q)
per id with c split into two floats (so p - c q keeps the precision of p and
q where they nearly cancel), and sums it in fp32 per lane of a chunk and in
fp64 across lanes.  Such trees are counted, and must stay rare.
"""
import numpy as np
import pytest

import synth
from oracle import sv_oracle as O

from _parity import logits_tensor, t

pytestmark = pytest.mark.gpu

NEAR = O.NEAR  # 1e-6


@pytest.fixture(scope="module")
def sv():
    import __graft_entry__
    __graft_entry__.build()
    import draft_token_verification_sv_gb300 as sv
    return sv


def _run(sv, tr, T, top_p, dtype, stride_pad=0):
    import torch
    tgt = logits_tensor(tr["logits_store"], dtype)
    dft = logits_tensor(tr["draft_store"], dtype)
    if stride_pad:
        B, N, V = tgt.shape
        tb = torch.zeros((B, N, V + stride_pad), dtype=tgt.dtype, device=tgt.device)
        db = torch.zeros_like(tb)
        tb[..., :V] = tgt
        db[..., :V] = dft
        tgt, dft = tb[..., :V], db[..., :V]
    got = sv.verify_tree_sample(tgt, dft, t(tr["parents"]), t(tr["tokens"]), t(tr["u_accept"]),
                                t(tr["u_final"]), tr["max_depth"], T, top_p)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in got.items()}


def _oracle(tr, T, top_p):
    return O.verify_tree_sample(tr["logits"], tr["draft_logits"], tr["parents"], tr["tokens"], tr["u_accept"],
                                tr["u_final"], T, top_p, tr["max_depth"])


def _compare(got, want, max_near_frac=0.05):
    B = want["accept_len"].shape[0]
    near = 0
    for b in range(B):
        d = int(want["accept_len"][b])
        alts = want["final_alts"][b]
        # the final token may be any the oracle admits under top-p cuts within 1e-6 of top_p
        same = (got["accept_len"][b] == d and np.array_equal(got["path"][b], want["path"][b])
                and np.array_equal(got["out_tokens"][b, :d], want["out_tokens"][b, :d])
                and int(got["out_tokens"][b, d]) in alts[alts >= 0].tolist()
                and np.array_equal(got["out_tokens"][b, d + 1:], want["out_tokens"][b, d + 1:]))
        if not same:
            assert want["margin"][b] < NEAR, (b, got["path"][b], want["path"][b], got["out_tokens"][b],
                                              want["out_tokens"][b], want["margin"][b])
            near += 1
            continue
        assert (got["row_status"][b] != 0) == (want["status"][b] != 0 or want["resample_fallback"][b]), b
    assert near <= max(1, int(max_near_frac * B)), near
    return near


def test_full_tree_workload(sv):
    """64 trees x 32 nodes, V = 128256 bf16, T = 1."""
    tr = synth.make_tree_sample_inputs(synth.TREE)
    got = _run(sv, tr, 1.0, 1.0, "bf16")
    want = _oracle(tr, 1.0, 1.0)
    _compare(got, want)
    assert want["accept_len"].max() >= 2


@pytest.mark.parametrize("dtype,T,top_p,V", [("f32", 0.7, 0.9, 32000), ("bf16", 1.3, 0.8, 50000),
                                             ("f32", 1.0, 1.0, 4099), ("bf16", 0.5, 0.95, 2048 * 3 + 5)])
def test_top_p_and_temperature(sv, dtype, T, top_p, V):
    cfg = synth.TreeConfig("t", 9, 32, V, dtype, 5, 8, 2.0, 0.7, 6.0)
    tr = synth.make_tree_sample_inputs(cfg, seed=V, batch=12)
    _compare(_run(sv, tr, T, top_p, dtype), _oracle(tr, T, top_p))


@pytest.mark.parametrize("N,V,D,dtype,noise", [(40, 3, 3, "f32", 2.0), (200, 5, 4, "bf16", 1.0),
                                               (600, 7, 64, "f32", 3.0), (1024, 2, 12, "bf16", 0.5)])
def test_many_siblings_tiny_vocab(sv, N, V, D, dtype, noise):
    """Many children per node on a tiny vocabulary: long runs of rejections
    (one residual pass each) and repeated sibling tokens."""
    cfg = synth.TreeConfig("t", 3, N, V, dtype, D, 64, 1.0, 0.3, 1.0)
    tr = synth.make_tree_sample_inputs(cfg, seed=N + V, draft_noise=noise)
    got = _run(sv, tr, 1.0, 1.0, dtype)
    want = _oracle(tr, 1.0, 1.0)
    _compare(got, want)


def test_unaligned_rows_and_large_vocab(sv):
    """Rows that do not start on a 16-byte boundary (scalar loads), and a
    vocabulary of more than 256 chunks of 2048 ids (wider chunks)."""
    cfg = synth.TreeConfig("t", 5, 8, 1001, "bf16", 4, 4, 2.0, 0.5, 4.0)
    tr = synth.make_tree_sample_inputs(cfg, seed=3, batch=6)
    _compare(_run(sv, tr, 1.0, 1.0, "bf16", stride_pad=3), _oracle(tr, 1.0, 1.0))
    cfg = synth.TreeConfig("t", 5, 6, 600_000, "f32", 3, 3, 2.0, 0.5, 4.0)
    tr = synth.make_tree_sample_inputs(cfg, seed=4, batch=2)
    _compare(_run(sv, tr, 1.0, 1.0, "f32"), _oracle(tr, 1.0, 1.0))


def test_many_trees_one_block_each(sv):
    """More trees than half the SMs: one thread block per tree instead of a
    cluster of two (the smaller batches above take the clusters)."""
    cfg = synth.TreeConfig("t", 9, 16, 3001, "bf16", 4, 4, 2.0, 0.6, 4.0)
    tr = synth.make_tree_sample_inputs(cfg, seed=11, batch=200, draft_noise=1.5)
    _compare(_run(sv, tr, 0.9, 0.9, "bf16"), _oracle(tr, 0.9, 0.9))


def test_zero_residual_fallback(sv):
    """q == p and top-p removes the first child's token from both: the child
    is rejected and max(0, r - q) has no mass (fallback bit); r stays p."""
    V = 64
    row = np.linspace(6.0, -6.0, V).astype(np.float32)
    tr = dict(logits=np.tile(row, (1, 2, 1)), parents=np.array([[-1, 0]], np.int32),
              tokens=np.array([[0, V - 1]], np.int32), u_accept=np.array([[0.0, 0.5]], np.float32),
              u_final=np.array([0.3], np.float32), max_depth=1)
    tr["draft_logits"] = tr["logits"].copy()
    tr["logits_store"] = tr["draft_store"] = tr["logits"]
    got = _run(sv, tr, 1.0, 0.5, "f32")
    want = _oracle(tr, 1.0, 0.5)
    assert want["resample_fallback"][0]
    assert got["row_status"][0] & 32             # SV_ROW_RESAMPLE_FALLBACK
    assert got["out_tokens"][0].tolist() == want["out_tokens"][0].tolist()


def test_invalid_trees_and_empty_rows(sv):
    cfg = synth.TreeConfig("t", 5, 10, 257, "f32", 4, 4, 2.0, 0.5, 4.0)
    tr = synth.make_tree_sample_inputs(cfg, seed=5, batch=5)
    tr["parents"][1, 5] = 9
    tr["tokens"][2, 3] = 257
    tr["parents"][3] = np.arange(-1, 9)          # a chain of depth 9 > 4
    tr["logits"][4, 7] = -np.inf
    tr["logits_store"] = tr["logits"]
    got = _run(sv, tr, 1.0, 1.0, "f32")
    want = _oracle(tr, 1.0, 1.0)
    for b, bit in ((1, O.STATUS_BAD_PARENT), (2, O.STATUS_BAD_TOKEN), (3, O.STATUS_DEPTH_EXCEEDED),
                   (4, O.STATUS_EMPTY_ROW)):
        assert want["status"][b] & bit and got["row_status"][b] & bit, b
        assert got["accept_len"][b] == 0 and np.all(got["out_tokens"][b] == -1) and np.all(got["path"][b] == -1)
    _compare({k: v[:1] for k, v in got.items()}, {k: v[:1] for k, v in want.items()})
