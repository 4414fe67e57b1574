"""sv_verify_chain_static, the entry point for callers that cannot allocate
device memory (it uses scratch built into the library instead of a
caller-provided workspace), must give the same results as sv_verify_chain.

Both are called through the C-ABI on the same inputs, twice in a row (the
built-in scratch keeps the previous call's contents), for a top-p sampling
workload, an EAGLE3 small-vocabulary workload and a greedy one.  The file is
named to be collected last."""
import ctypes

import numpy as np
import pytest

import synth

from _parity import TOL, logits_tensor, oracle_draft_ids, t

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    import __graft_entry__
    __graft_entry__.build()
    import draft_token_verification_sv_gb300 as sv
    return sv


def _static_call(sv, target, draft, ids, ua, ur, T, top_p, d2t=None, t2d=None):
    import torch
    from draft_token_verification_sv_gb300 import _native as N
    from draft_token_verification_sv_gb300.verify import chain_desc
    B, gp1, _ = target.shape
    d = chain_desc(target, draft, T, top_p, d2t)
    out = dict(tokens=torch.full((B, gp1), -7, dtype=torch.int32, device="cuda"),
               num_accepted=torch.full((B,), -7, dtype=torch.int32, device="cuda"),
               p_draft=torch.full((B, gp1 - 1), -7.0, device="cuda"),
               q_draft=torch.full((B, gp1 - 1), -7.0, device="cuda"),
               row_status=torch.full((B,), -7, dtype=torch.int32, device="cuda"))
    p = lambda x: None if x is None else ctypes.c_void_p(x.data_ptr())
    st = N.lib().sv_verify_chain_static(
        ctypes.byref(d), p(target), p(draft), p(d2t), p(t2d), p(ids), p(ua), p(ur), p(out["tokens"]),
        p(out["num_accepted"]), p(out["p_draft"]), p(out["q_draft"]), p(out["row_status"]),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, N.lib().sv_status_string(st)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


def _compare(a, b, dtype):
    for k in ("tokens", "num_accepted", "row_status"):
        assert np.array_equal(a[k], b[k]), k
    for k in ("p_draft", "q_draft"):
        np.testing.assert_allclose(a[k], b[k], rtol=TOL[dtype], atol=1e-12)


@pytest.mark.parametrize("case", ["topp", "d2t", "greedy"])
def test_static_matches_workspace_entry(sv, case):
    import torch
    if case == "topp":
        cfg = synth.ChainConfig("c", 8, 5, 49152, "bf16", 0.8, 0.9, 3.0, 0.7, spikes=5, spike_value=8.0)
    elif case == "d2t":
        cfg = synth.ChainConfig("c", 6, 7, 151936, "f32", 1.0, 0.95, 2.0, 0.7, draft_vocab=32000)
    else:
        cfg = synth.ChainConfig("c", 16, 6, 128256, "bf16", 0.0, 1.0, 2.0, 0.5)
    x = synth.make_chain_inputs(cfg, seed=77)
    ids = oracle_draft_ids(x)
    T, P = cfg.temperature, cfg.top_p
    target = logits_tensor(x["target_store"], cfg.dtype)
    draft = logits_tensor(x["draft_store"], cfg.dtype) if T > 0 else None
    ua = t(x["u_accept"]) if T > 0 else None
    ur = t(x["u_resample"]) if T > 0 else None
    d2t = t2d = None
    if x["d2t"] is not None:
        d2t = t(x["d2t"])
        t2d = sv.build_t2d(d2t, x["vocab"])[0]
    ids_t = t(ids)
    want = sv.verify_chain(target, draft, ids_t, ua, ur, T, P, d2t=d2t, t2d=t2d)
    torch.cuda.synchronize()
    want = {k: v.cpu().numpy() for k, v in want.items()}
    for _ in range(2):  # two calls in a row share the built-in scratch
        got = _static_call(sv, target, draft, ids_t, ua, ur, T, P, d2t, t2d)
        _compare(got, want, cfg.dtype)


def test_static_rejects_oversized_requests(sv):
    from draft_token_verification_sv_gb300 import _native as N
    lib = N.lib()
    cap = lib.sv_static_scratch_bytes()
    d = N.ChainDesc()
    d.batch, d.gamma, d.vocab, d.draft_vocab = 2048, 7, 151936, 151936
    d.target_dtype = d.draft_dtype = N.SV_F32
    d.temperature, d.top_p = 1.0, 0.9
    d.target_row_stride = d.draft_row_stride = 151936
    assert lib.sv_chain_workspace_size(ctypes.byref(d)) > cap
    A = ctypes.c_void_p(0x100000)
    st = lib.sv_verify_chain_static(ctypes.byref(d), A, A, None, None, A, A, A, A, A, None, None, None, None)
    assert st == N.SV_ERR_WORKSPACE_TOO_SMALL


@pytest.mark.parametrize("temperature", [0.0, 1.0])
def test_static_empty_batch(sv, temperature):
    """An empty batch is a valid call that needs no scratch: SV_OK, as from
    sv_verify_chain, with nothing launched."""
    from draft_token_verification_sv_gb300 import _native as N
    lib = N.lib()
    d = N.ChainDesc()
    d.batch, d.gamma, d.vocab, d.draft_vocab = 0, 4, 1000, 1000
    d.target_dtype = d.draft_dtype = N.SV_F32
    d.temperature, d.top_p = temperature, 1.0
    d.target_row_stride = d.draft_row_stride = 1000
    st = lib.sv_verify_chain_static(ctypes.byref(d), None, None, None, None, None, None, None, None, None,
                                    None, None, None, None)
    assert st == N.SV_OK
    d.top_p = 0.0  # still checked: an invalid descriptor is rejected
    st = lib.sv_verify_chain_static(ctypes.byref(d), None, None, None, None, None, None, None, None, None,
                                    None, None, None, None)
    assert st == N.SV_ERR_INVALID_ARGUMENT
