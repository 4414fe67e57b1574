"""Tree verify, d2t scatter, t2d build and draft-side sampling on the GPU
(through the C-ABI) against the fp64 oracle."""
import math

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


def _tree_run(sv, tr, dtype="bf16"):
    import torch
    logits = logits_tensor(tr["logits_store"], dtype)
    got = sv.verify_tree(logits, t(tr["parents"]), t(tr["tokens"]), tr["max_depth"])
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in got.items()}


def _tree_compare(got, want):
    assert np.array_equal(got["accept_len"], want["accept_len"])
    assert np.array_equal(got["out_tokens"], want["out_tokens"])
    assert np.array_equal(got["path"], want["path"])
    assert np.array_equal(got["row_status"] != 0, want["status"] != 0)


def test_tree_full_workload(sv):
    """64 trees x 32 nodes, V = 128256 bf16 (the Eaglet1 tree budget)."""
    tr = synth.make_tree_inputs(synth.TREE)
    got = _tree_run(sv, tr)
    want = O.verify_tree(tr["logits"], tr["parents"], tr["tokens"], tr["max_depth"])
    _tree_compare(got, want)
    print(f"[tree] mean accepted length {got['accept_len'].mean():.2f}")
    assert got["accept_len"].max() >= 2


@pytest.mark.parametrize("N,V,D,dtype", [(1, 5, 0, "bf16"), (2, 3, 1, "f32"), (12, 4, 4, "bf16"),
                                         (32, 7, 5, "f32"), (600, 3, 64, "bf16"), (1024, 2, 12, "f32")])
def test_tree_small_with_ties(sv, N, V, D, dtype):
    cfg = synth.TreeConfig("t", 5, N, V, dtype, D, 8 if N <= 32 else 64, 1.0, 0.8, 0.0)
    tr = synth.make_tree_inputs(cfg, seed=N * 7 + V)
    q = np.round(tr["logits"]).astype(np.float32)   # ties everywhere
    tr["logits"] = q
    tr["logits_store"] = synth.to_bf16_bits(q) if dtype == "bf16" else q
    # Plant matches so paths are long: child token = parent's argmax.
    for b in range(tr["batch"]):
        for n in range(1, N):
            if n % 3:
                tr["tokens"][b, n] = int(np.argmax(q[b, tr["parents"][b, n]]))
    got = _tree_run(sv, tr, dtype)
    want = O.verify_tree(tr["logits"], tr["parents"], tr["tokens"], tr["max_depth"])
    _tree_compare(got, want)


@pytest.mark.parametrize("dtype,V", [("bf16", 128256), ("f32", 151936)])
def test_tree_one_tree_long_rows(sv, dtype, V):
    """One small tree over a large vocabulary: its rows are split over
    several blocks each."""
    cfg = synth.TreeConfig("t", 1, 6, V, dtype, 3, 8, 2.0, 0.8, 0.0)
    tr = synth.make_tree_inputs(cfg, seed=V)
    for n in range(1, 6):
        if n % 2:
            tr["tokens"][0, n] = int(np.argmax(tr["logits"][0, tr["parents"][0, n]]))
    got = _tree_run(sv, tr, dtype)
    want = O.verify_tree(tr["logits"], tr["parents"], tr["tokens"], tr["max_depth"])
    _tree_compare(got, want)


def test_tree_invalid(sv):
    tr = synth.make_tree_inputs(synth.TREE, batch=4, vocab=257)
    tr["parents"][1, 5] = 9          # parent after child
    tr["parents"][2, 0] = 0          # root with a parent
    tr["tokens"][3, 4] = 257         # token out of range
    got = _tree_run(sv, tr)
    want = O.verify_tree(tr["logits"], tr["parents"], tr["tokens"], tr["max_depth"])
    assert got["row_status"][1] & O.STATUS_BAD_PARENT and got["row_status"][2] & O.STATUS_BAD_PARENT
    assert got["row_status"][3] & O.STATUS_BAD_TOKEN
    for b in (1, 2, 3):
        assert got["accept_len"][b] == 0 and np.all(got["out_tokens"][b] == -1)
    _tree_compare({k: v[:1] for k, v in got.items()}, {k: v[:1] for k, v in want.items()})
    # A tree deeper than max_depth.
    cfg = synth.TreeConfig("chain", 1, 8, 50, "f32", 7, 1, 1.0, 1.0, 16.0)
    deep = synth.make_tree_inputs(cfg, seed=1)
    deep["max_depth"] = 3
    g = _tree_run(sv, deep, "f32")
    assert g["row_status"][0] & O.STATUS_DEPTH_EXCEEDED


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shuffled", [False, True])
@pytest.mark.parametrize("with_t2d", [False, True])
def test_d2t_scatter_matches_oracle(sv, dtype, shuffled, with_t2d):
    import torch
    V, Vd, R = 151936, 32000, 16
    d2t = synth.make_d2t(5, V, Vd, shuffled=shuffled)
    rows = np.random.default_rng(1).normal(0, 2, (R, Vd)).astype(np.float32)
    store = synth.to_bf16_bits(rows) if dtype == "bf16" else rows
    vals = synth.bf16_bits_to_f32(store) if dtype == "bf16" else rows
    x = logits_tensor(store, dtype)
    t2d = sv.build_t2d(t(d2t), V)[0] if with_t2d else None
    out = sv.d2t_scatter(x, t(d2t), V, fill=-math.inf, t2d=t2d)
    torch.cuda.synchronize()
    want = O.d2t_scatter(vals, d2t, V)
    np.testing.assert_array_equal(out.float().cpu().numpy(), want.astype(np.float32))


@pytest.mark.parametrize("with_t2d,shuffled", [(True, False), (False, False), (False, True)])
def test_d2t_scatter_full_draft_set(sv, with_t2d, shuffled):
    """Every draft row of the Qwen3/EAGLE3 workload (256 x 7 rows of 32000
    fp32 logits into 151936 ids) in one call: sampled rows equal the oracle's
    scatter, and every row is its draft row at the mapped ids and the fill
    elsewhere (checked on the device).  An increasing d2t (EAGLE3's) takes
    the tiled fill form without t2d; a shuffled one the two-phase form."""
    import torch
    V, Vd, R = 151936, 32000, 256 * 7
    d2t = synth.make_d2t(7, V, Vd, shuffled=shuffled)
    g = torch.Generator(device="cuda").manual_seed(7)
    x = torch.randn((R, Vd), generator=g, device="cuda") * 2.0
    d2t_t = t(d2t)
    t2d = sv.build_t2d(d2t_t, V)[0] if with_t2d else None
    out = sv.d2t_scatter(x, d2t_t, V, fill=-math.inf, t2d=t2d)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    sv.d2t_scatter(x, d2t_t, V, fill=-math.inf, t2d=t2d, out=out)
    end.record()
    torch.cuda.synchronize()
    ms = start.elapsed_time(end)
    form = "gather form" if with_t2d else ("fill form, shuffled d2t" if shuffled else "fill form, increasing d2t")
    print(f"[d2t scatter {form}] {R} rows: {ms * 1e3:.1f} us, "
          f"{R * (V + Vd) * 4 / (ms * 1e-3) / 1e12:.2f} TB/s (rows read once, written once)")
    rows = np.random.default_rng(3).choice(R, 8, replace=False)
    xs = x[torch.from_numpy(rows).cuda()].cpu().numpy()
    np.testing.assert_array_equal(out[torch.from_numpy(rows).cuda()].cpu().numpy(), O.d2t_scatter(xs, d2t, V))
    idx = d2t_t.long()
    assert torch.equal(out[:, idx], x)
    mask = torch.ones(V, dtype=torch.bool, device="cuda")
    mask[idx] = False
    assert bool(torch.isneginf(out[:, mask]).all())


def test_d2t_scatter_odd_sizes_and_fill(sv):
    import torch
    V, Vd, R = 1001, 37, 3
    d2t = synth.make_d2t(2, V, Vd, shuffled=True)
    rows = np.random.default_rng(2).normal(0, 1, (R, 40)).astype(np.float32)[:, :Vd]
    x = t(np.ascontiguousarray(np.pad(rows, ((0, 0), (0, 3)))))[:, :Vd]  # stride 40
    for use_t2d in (False, True):
        t2d = sv.build_t2d(t(d2t), V)[0] if use_t2d else None
        out = torch.empty((R, 1004), device="cuda")[:, :V]
        sv.d2t_scatter(x, t(d2t), V, fill=-3.5, t2d=t2d, out=out)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(out.cpu().numpy(), O.d2t_scatter(rows, d2t, V, fill=-3.5))


def test_build_t2d(sv):
    import torch
    d2t = synth.make_d2t(3, 151936, 32000, shuffled=True)
    t2d, st = sv.build_t2d(t(d2t), 151936)
    torch.cuda.synchronize()
    assert st.item() == 0
    np.testing.assert_array_equal(t2d.cpu().numpy(), O.build_t2d(d2t, 151936))
    _, st = sv.build_t2d(t(np.array([1, 2, 1], np.int32)), 5)
    assert st.item() & 2
    _, st = sv.build_t2d(t(np.array([1, 7], np.int32)), 5)
    assert st.item() & 1


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("V", [8, 2048, 4104, 65536])
def test_sample_rows_one_pass_edge_cases(sv, dtype, V):
    """The one-pass sampler (no top-p, aligned rows): logits with -inf
    entries, a row with a single finite logit, an all -inf row (token -1),
    uniforms 0 and just below 1, rows shorter than one chunk and not a
    multiple of it."""
    import torch
    R = 16
    g = np.random.default_rng(V)
    rows = g.normal(0, 2.0, (R, V)).astype(np.float32)
    rows[g.random((R, V)) < 0.3] = -np.inf
    rows[1, :] = -np.inf
    rows[1, V // 3] = 0.5            # a single finite logit
    rows[2, :] = -np.inf             # no finite logit at all
    if dtype == "bf16":
        store = synth.to_bf16_bits(rows)
        rows = synth.bf16_bits_to_f32(store)
    else:
        store = rows
    u = g.random(R).astype(np.float32)
    u[3] = 0.0
    u[4] = np.float32(1.0) - np.float32(2.0 ** -24)
    tok, prob = sv.sample(logits_tensor(store, dtype), 1.0, 1.0, t(u))
    torch.cuda.synchronize()
    tok, prob = tok.cpu().numpy(), prob.cpu().numpy()
    assert tok[2] == -1 and prob[2] == 0.0
    assert tok[1] == V // 3 and abs(prob[1] - 1.0) <= 1e-6
    for r in range(R):
        if r == 2:
            continue
        alts = []
        want, margin = O.sample_row(rows[r], 1.0, 1.0, float(u[r]), alts=alts)
        if margin < O.NEAR:
            continue
        assert int(tok[r]) == want, (r, int(tok[r]), want, margin)
        p, _ = O.dist(rows[r], 1.0, 1.0)
        assert abs(prob[r] - p[want]) <= max(1e-12, 1e-5 * p[want])


@pytest.mark.parametrize("dtype,V,top_p", [("f32", 32000, 0.95), ("bf16", 49152, 0.9), ("bf16", 128256, 1.0)])
def test_sample_rows_full_size(sv, dtype, V, top_p):
    """Draft-side sampling of 1792 rows at once (the qwen3 draft rows'
    count: 32000 fp32 at top_p 0.95; 49152 bf16 at 0.9; 128256 bf16 without
    top-p), timed; sampled rows against the oracle's admissible draws."""
    import torch
    R, T = 1792, 1.0
    g = torch.Generator(device="cuda").manual_seed(V)
    x = torch.randn((R, V), generator=g, device="cuda") * 2.5
    if dtype == "bf16":
        x = x.to(torch.bfloat16)
    u = torch.rand(R, generator=g, device="cuda")
    tok, prob = sv.sample(x, T, top_p, u)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    tok, prob = sv.sample(x, T, top_p, u)
    end.record()
    torch.cuda.synchronize()
    ms = start.elapsed_time(end)
    es = 2 if dtype == "bf16" else 4
    print(f"[sample {R} x {V} {dtype} top_p={top_p}] {ms * 1e3:.1f} us, {R * V * es / (ms * 1e-3) / 1e12:.2f} TB/s "
          "(rows read once; the draw re-reads one chunk per row)")
    rows = np.random.default_rng(V).choice(R, 8, replace=False)
    xs = x[torch.from_numpy(rows).cuda()].float().cpu().numpy()
    us = u[torch.from_numpy(rows).cuda()].cpu().numpy()
    checked = 0
    for i, r in enumerate(rows):
        alts = []
        want, margin = O.sample_row(xs[i], T, top_p, float(us[i]), alts=alts)
        if margin < O.NEAR:
            continue
        assert int(tok[r]) in [a for a, _ in alts], (r, int(tok[r]), alts)
        checked += 1
    assert checked >= 4, checked


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("V,T,top_p", [(1, 1.0, 0.9), (3, 0.5, 1.0), (1000, 0.8, 0.9), (49152, 0.8, 0.9),
                                       (32000, 1.0, 0.95), (4097, 0.0, 1.0), (128256, 1.0, 1.0)])
def test_sample_rows(sv, dtype, V, T, top_p):
    import torch
    R = 24
    g = np.random.default_rng(V)
    rows = g.normal(0, 2.5, (R, V)).astype(np.float32)
    if dtype == "bf16":
        store = synth.to_bf16_bits(rows)
        rows = synth.bf16_bits_to_f32(store)
    else:
        store = rows
    u = g.random(R, dtype=np.float32)
    tok, prob = sv.sample(logits_tensor(store, dtype), T, top_p, t(u) if T > 0 else None)
    torch.cuda.synchronize()
    tok, prob = tok.cpu().numpy(), prob.cpu().numpy()
    checked = 0
    for r in range(R):
        # every draw the top-p cuts within 1e-6 of top_p admit, with its probability
        alts = []
        want, margin = O.sample_row(rows[r], T, top_p, float(u[r]), alts=alts)
        if margin < O.NEAR:
            continue
        admitted = {a: pa for a, pa in alts}
        assert int(tok[r]) in admitted, (r, tok[r], want, alts, margin)
        if T > 0:
            pw = admitted[int(tok[r])]
            assert abs(prob[r] - pw) <= max(1e-12, 1e-5 * pw) or any(
                a == int(tok[r]) and abs(prob[r] - pa) <= max(1e-12, 1e-5 * pa) for a, pa in alts)
        checked += 1
    assert checked >= (3 * R) // 4, checked  # rows decided clear of every threshold
