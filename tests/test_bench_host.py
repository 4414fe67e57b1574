"""Host logic of bench.py that needs no GPU: every workload's byte count
and config line, the oracle arm on small copies of each workload (including
tree sampling), and the seeded inputs being reproducible."""
import dataclasses
import os
import sys

import numpy as np
import pytest

import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_every_workload_has_bytes_and_a_config_line():
    for name, cfg in bench.WORKLOADS.items():
        b = bench.step_bytes(cfg)
        assert b > 0
        c = bench.config_of(cfg, name, bench.n_sets_for(cfg), 1)
        assert c["workload"] == name and c["batch"] == cfg.batch and c["vocab"] == cfg.vocab
        assert bench.n_sets_for(cfg) * b > 4 * bench.L2_BYTES      # rotation exceeds 4x L2


def test_tree_sample_counts_target_and_draft_rows():
    s, t = synth.TREE_SAMPLE, synth.TREE
    assert s.algorithmic_bytes() == 2 * t.algorithmic_bytes() == 2 * 64 * 32 * 128256 * 2
    c = bench.config_of(s, "tree-sample", 2, 1)
    assert (c["temperature"], c["top_p"], c["nodes"], c["max_depth"]) == (1.0, 1.0, 32, 5)
    assert bench.config_of(t, "tree", 2, 1)["temperature"] == 0.0


def test_tree_sample_inputs_are_seeded():
    small = dataclasses.replace(synth.TREE_SAMPLE, batch=2, vocab=300)
    a = synth.make_tree_sample_inputs(small)
    b = synth.make_tree_sample_inputs(small)
    for k in ("logits", "draft_logits", "parents", "tokens", "u_accept", "u_final"):
        assert np.array_equal(a[k], b[k]), k
    assert not np.array_equal(a["logits"], a["draft_logits"])
    assert a["u_accept"].dtype == np.float32 and (0 <= a["u_accept"]).all() and (a["u_accept"] < 1).all()
    # the same target logits as the greedy tree workload of that shape
    g = synth.make_tree_inputs(dataclasses.replace(synth.TREE, batch=2, vocab=300))
    assert np.array_equal(a["logits"], g["logits"]) and np.array_equal(a["tokens"], g["tokens"])


@pytest.mark.parametrize("name", ["tree", "tree-sample"])
def test_oracle_arm_on_small_trees(name):
    cfg = dataclasses.replace(bench.WORKLOADS[name], batch=3, vocab=500)
    host = synth.make_tree_sample_inputs(cfg) if isinstance(cfg, synth.TreeSampleConfig) \
        else synth.make_tree_inputs(cfg)
    out = bench.oracle_rows(cfg, host, [0, 2])
    assert out["accept_len"][1] == 0 and np.all(out["out_tokens"][1] == -1)   # row 1 not computed
    for b in (0, 2):
        d = out["accept_len"][b]
        assert 0 <= d <= cfg.max_depth and out["out_tokens"][b][d] >= 0
    assert bench.units_per_batch_row(cfg) == cfg.nodes


@pytest.mark.parametrize("name", ["tiny", "tree", "tree-sample"])
def test_parity_sample_counts_mismatches(name):
    cfg = bench.WORKLOADS[name]
    if isinstance(cfg, synth.TreeConfig):
        cfg = dataclasses.replace(cfg, batch=4, vocab=400)
        host = synth.make_tree_sample_inputs(cfg) if isinstance(cfg, synth.TreeSampleConfig) \
            else synth.make_tree_inputs(cfg)
        key = "out_tokens"
    else:
        host = synth.make_chain_inputs(cfg, batch=4)
        bench.oracle_draft_ids(cfg, host, range(4))
        key = "tokens"
    sampled = []
    inputs = {"host": host}
    cfg_b = dataclasses.replace(cfg, batch=4)
    base = bench.cpu_baseline(cfg_b, inputs, 0.0, sink=sampled, cores=2)
    assert base["kind"] == "oracle" and base["cores"] == 2 and len(sampled) >= 1
    # the workers' rows are the oracle's own rows
    rows = [b for b, _, _, _ in sampled]
    direct = bench.oracle_rows(cfg_b, host, rows)
    for b, tok, margin, others in sampled:
        assert np.array_equal(tok, direct[key][b])
    got = np.full((4, sampled[0][1].size), -1, np.int64)
    for b, tok, _, _ in sampled:
        got[b] = tok
    assert bench.parity_sample(cfg_b, sampled, got) == {"rows": len(sampled), "mismatch": 0,
                                                        "near_threshold": 0}
    b0 = sampled[0][0]
    got[b0, 0] = got[b0, 0] + 1
    r = bench.parity_sample(cfg_b, sampled, got)
    assert r["mismatch"] == 1 and r["near_threshold"] in (0, 1)


def test_host_cores_is_positive():
    assert bench.host_cores() >= 1
