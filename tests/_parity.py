"""Helpers shared by the GPU parity tests (CUDA library vs fp64 oracle)."""
from __future__ import annotations

import numpy as np

from oracle import sv_oracle as O

# Probability tolerances (relative), per input dtype: the stated contract.
TOL = {"f32": 1e-5, "bf16": 2e-3}
ATOL = 1e-12


def torch_mod():
    import torch
    return torch


def dev():
    return torch_mod().device("cuda:0")


def t(a):
    torch = torch_mod()
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev())


def logits_tensor(store: np.ndarray, dtype: str):
    torch = torch_mod()
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(store).view(np.int16)).to(dev()).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(store, dtype=np.float32)).to(dev())


def oracle_draft_ids(x: dict) -> np.ndarray:
    """Draft ids drawn by the oracle from q_i with the seeded uniforms u_draft
    (argmax at T = 0); target-vocabulary ids."""
    cfg = x["cfg"]
    B, G = x["batch"], x["gamma"]
    T, top_p = cfg.temperature, cfg.top_p
    d2t = x["d2t"]
    ids = np.zeros((B, G), np.int32)
    for b in range(B):
        for i in range(G):
            row = x["draft"][b, i]
            tok, _ = O.sample_row(row, T, top_p, float(x["u_draft"][b, i]), tie_index=d2t)
            ids[b, i] = d2t[tok] if d2t is not None else tok
    return ids


def run_chain(sv, x: dict, ids: np.ndarray, *, temperature=None, top_p=None, t2d_dev=None):
    cfg = x["cfg"]
    T = cfg.temperature if temperature is None else temperature
    P = cfg.top_p if top_p is None else top_p
    target = logits_tensor(x["target_store"], cfg.dtype)
    draft = logits_tensor(x["draft_store"], cfg.dtype) if T > 0 else None
    d2t = t(x["d2t"]) if (x["d2t"] is not None and T > 0) else None
    t2d = None
    if d2t is not None:
        t2d = t2d_dev if t2d_dev is not None else sv.build_t2d(d2t, x["vocab"])[0]
    got = sv.verify_chain(target, draft, t(ids), t(x["u_accept"]) if T > 0 else None,
                          t(x["u_resample"]) if T > 0 else None, T, P, d2t=d2t, t2d=t2d)
    torch_mod().cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in got.items()}


def oracle_chain(x: dict, ids: np.ndarray, rows=None, *, temperature=None, top_p=None):
    cfg = x["cfg"]
    T = cfg.temperature if temperature is None else temperature
    P = cfg.top_p if top_p is None else top_p
    return O.verify_chain(x["target"], x["draft"] if T > 0 else None, ids,
                          x["u_accept"] if T > 0 else None, x["u_resample"] if T > 0 else None,
                          T, P, d2t=x["d2t"], rows=rows)


def compare_chain(got: dict, want: dict, ids: np.ndarray, dtype: str, rows=None, check_probs=True):
    """Ids/counts equal to the oracle's, the drawn token being any of the
    oracle's final_alts (the draw under every top-p cut that lies within
    1e-6 of top_p), except from the first output position that an oracle
    decision within 1e-6 of its threshold decides (the oracle's near_from):
    the positions before it must match on every row.  The draft's p/q within
    the dtype's tolerance of the oracle's value under one of the admissible
    cuts.  Returns (n_rows, n_near, n_near_mismatch, max_rel_err)."""
    B, gp1 = got["tokens"].shape
    rows = list(range(B)) if rows is None else list(rows)
    near = want["margin"] < O.NEAR
    n_near = n_near_mis = 0
    max_rel = 0.0
    for b in rows:
        k = int(want["num_accepted"][b])
        alts = want["final_alts"][b] if "final_alts" in want else want["tokens"][b, k:k + 1]
        alts = alts[alts >= 0] if np.any(alts >= 0) else want["tokens"][b, k:k + 1]  # greedy and status rows
        same = (got["num_accepted"][b] == k and np.array_equal(got["tokens"][b, :k], want["tokens"][b, :k])
                and int(got["tokens"][b, k]) in alts.tolist()
                and np.array_equal(got["tokens"][b, k + 1:], want["tokens"][b, k + 1:]))
        st_got = int(got["row_status"][b]) & ~32
        st_want = int(want["status"][b])
        assert (st_got != 0) == (st_want != 0), (b, st_got, st_want)
        if near[b]:
            n_near += 1
            n_near_mis += int(not same)
            nf = int(want["near_from"][b]) if "near_from" in want else 0
            # Everything decided before the near decision still matches.
            assert np.array_equal(got["tokens"][b, :nf], want["tokens"][b, :nf]), (b, nf)
            assert min(int(got["num_accepted"][b]), nf) == min(k, nf), (b, nf)
        else:
            assert same, (f"row {b}: tokens {got['tokens'][b]} k={got['num_accepted'][b]} vs oracle "
                          f"{want['tokens'][b]} k={k} (or {alts}) margin={want['margin'][b]:.3g}")
        if check_probs and "p_draft" in got and st_want == 0:
            G = got["p_draft"].shape[1]
            for key in ("p", "q"):
                g = got[key + "_draft"][b].astype(np.float64)
                w = want[key + "_alts"][b] if key + "_alts" in want else want[key + "_draft"][b][:, None]
                w = w[:G]
                err = np.abs(g[:, None] - w) / np.maximum(np.abs(w), 1e-300)
                hit = (np.abs(g[:, None] - w) <= ATOL) | (err <= TOL[dtype])   # NaN pads never hit
                assert hit.any(axis=1).all(), (b, key, g, w)
                # relative error against the closest admissible value (0 where an
                # absolute match within ATOL), over positions with a non-tiny value
                ea = np.where(np.abs(g[:, None] - w) <= ATOL, 0.0, err)
                e = np.where(np.isnan(ea), np.inf, ea).min(axis=1)
                e = e[np.isfinite(e) & (np.nanmax(np.abs(w), axis=1) > 1e-9)]
                if e.size:
                    max_rel = max(max_rel, float(e.max()))
    return len(rows), n_near, n_near_mis, max_rel


def chain_properties(got: dict, ids: np.ndarray, vocab: int):
    """Properties every output row satisfies, whatever the oracle says."""
    B, gp1 = got["tokens"].shape
    G = gp1 - 1
    for b in range(B):
        k = int(got["num_accepted"][b])
        assert 0 <= k <= G
        assert int(got["row_status"][b]) & ~32 == 0
        assert np.array_equal(got["tokens"][b, :k], ids[b, :k])
        assert 0 <= got["tokens"][b, k] < vocab
        assert np.all(got["tokens"][b, k + 1:] == -1)
