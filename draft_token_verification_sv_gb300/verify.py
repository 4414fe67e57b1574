"""PyTorch-facing wrappers over the C-ABI (argument marshalling only).

Every function checks tensor placement, dtype and layout, allocates outputs,
passes raw device pointers and the current CUDA stream to the library, and
raises ``SVError`` on a non-OK status.  All arithmetic runs in the library's
CUDA kernels.
"""
from __future__ import annotations

import ctypes
import math

import torch

from . import _native as N

_WORKSPACES: dict = {}


def _code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return N.SV_BF16
    if t.dtype == torch.float32:
        return N.SV_F32
    raise TypeError(f"logits must be float32 or bfloat16, got {t.dtype}")


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _cuda(t, name):
    if t is not None and not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")


def _row_stride(t: torch.Tensor, name: str) -> int:
    """Row stride (elements) of a tensor whose last dim is contiguous and whose
    leading dims collapse into evenly spaced rows."""
    if t.stride(-1) != 1:
        raise ValueError(f"{name}: last dimension must be contiguous")
    if t.dim() == 1:
        return t.shape[0]
    rs = t.stride(-2)
    for d in range(t.dim() - 2):
        if t.shape[d] > 1 and t.stride(d) != t.shape[d + 1] * t.stride(d + 1):
            raise ValueError(f"{name}: rows are not evenly spaced")
    return rs


def _i32(t, name):
    if t is None:
        return None
    if t.dtype != torch.int32 or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous int32 tensor")
    return t


def _f32(t, name):
    if t is None:
        return None
    if t.dtype != torch.float32 or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous float32 tensor")
    return t


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def workspace(nbytes: int, device: torch.device, stream=None) -> torch.Tensor:
    """A device workspace of at least ``nbytes``, cached per device and
    stream (calls on one stream run in order, so they may share it)."""
    s = stream if stream is not None else torch.cuda.current_stream(device)
    key = (device.index, s.cuda_stream)
    ws = _WORKSPACES.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=device)
        _WORKSPACES[key] = ws
    return ws


def chain_desc(target, draft, temperature, top_p, d2t=None) -> N.ChainDesc:
    B, gp1, V = target.shape
    G = gp1 - 1
    d = N.ChainDesc()
    d.batch, d.gamma, d.vocab = B, G, V
    d.target_dtype = _code(target)
    d.target_row_stride = _row_stride(target, "target")
    d.temperature = float(temperature)
    d.top_p = float(top_p)
    if draft is not None and G > 0:
        d.draft_vocab = draft.shape[-1]
        d.draft_dtype = _code(draft)
        d.draft_row_stride = _row_stride(draft, "draft")
    else:
        d.draft_vocab = V
        d.draft_dtype = d.target_dtype
        d.draft_row_stride = d.target_row_stride
    return d


def verify_chain(target: torch.Tensor, draft: torch.Tensor | None, draft_ids: torch.Tensor | None,
                 u_accept: torch.Tensor | None, u_resample: torch.Tensor | None,
                 temperature: float, top_p: float = 1.0, d2t: torch.Tensor | None = None,
                 t2d: torch.Tensor | None = None, *, probs: bool = True, out: dict | None = None,
                 ws: torch.Tensor | None = None, stream=None) -> dict:
    """Verify B draft chains; see sv_verify_chain in include/spec_verify.h.

    target [B, γ+1, V], draft [B, γ, V or V_d] (float32 or bfloat16, CUDA),
    draft_ids [B, γ] int32, u_accept [B, γ] / u_resample [B] float32.
    Returns dict(tokens [B, γ+1], num_accepted [B], p_draft, q_draft [B, γ]
    (when ``probs``), row_status [B]).
    """
    for t, n in ((target, "target"), (draft, "draft"), (draft_ids, "draft_ids"), (u_accept, "u_accept"),
                 (u_resample, "u_resample"), (d2t, "d2t"), (t2d, "t2d")):
        _cuda(t, n)
    if target.dim() != 3:
        raise ValueError("target must be [B, gamma+1, V]")
    B, gp1, V = target.shape
    G = gp1 - 1
    d = chain_desc(target, draft, temperature, top_p, d2t)
    dev = target.device
    if out is None:
        out = dict(tokens=torch.empty((B, gp1), dtype=torch.int32, device=dev),
                   num_accepted=torch.empty(B, dtype=torch.int32, device=dev),
                   row_status=torch.empty(B, dtype=torch.int32, device=dev))
        if probs:
            out["p_draft"] = torch.empty((B, G), dtype=torch.float32, device=dev)
            out["q_draft"] = torch.empty((B, G), dtype=torch.float32, device=dev)
    need = N.lib().sv_chain_workspace_size(ctypes.byref(d))
    if ws is None:
        ws = workspace(need, dev, stream)
    st = N.lib().sv_verify_chain(
        ctypes.byref(d), _p(target), _p(draft), _p(_i32(d2t, "d2t")), _p(_i32(t2d, "t2d")),
        _p(_i32(draft_ids, "draft_ids")), _p(_f32(u_accept, "u_accept")),
        _p(_f32(u_resample, "u_resample")), _p(out["tokens"]), _p(out["num_accepted"]),
        _p(out.get("p_draft")), _p(out.get("q_draft")), _p(out.get("row_status")),
        _p(ws), ctypes.c_size_t(ws.numel()), _stream(stream))
    N.check(st, "sv_verify_chain")
    return out


def verify_tree(logits: torch.Tensor, parents: torch.Tensor, tokens: torch.Tensor, max_depth: int,
                *, out: dict | None = None, ws: torch.Tensor | None = None, stream=None,
                path_walk: bool = False) -> dict:
    """Greedy verify of B draft trees; see sv_verify_tree (path_walk:
    sv_verify_tree_path, which reads only the rows of the accepted frontier).

    logits [B, N, V], parents/tokens [B, N] int32.  Returns dict(accept_len
    [B], path [B, D+1], out_tokens [B, D+1], row_status [B]).
    """
    for t, n in ((logits, "logits"), (parents, "parents"), (tokens, "tokens")):
        _cuda(t, n)
    B, Nn, V = logits.shape
    d = N.TreeDesc()
    d.batch, d.nodes, d.vocab, d.max_depth = B, Nn, V, int(max_depth)
    d.dtype = _code(logits)
    d.row_stride = _row_stride(logits, "logits")
    dev = logits.device
    L = int(max_depth) + 1
    if out is None:
        out = dict(accept_len=torch.empty(B, dtype=torch.int32, device=dev),
                   path=torch.empty((B, L), dtype=torch.int32, device=dev),
                   out_tokens=torch.empty((B, L), dtype=torch.int32, device=dev),
                   row_status=torch.empty(B, dtype=torch.int32, device=dev))
    lib = N.lib()
    size_fn, fn, name = ((lib.sv_tree_path_workspace_size, lib.sv_verify_tree_path, "sv_verify_tree_path")
                         if path_walk else (lib.sv_tree_workspace_size, lib.sv_verify_tree, "sv_verify_tree"))
    need = size_fn(ctypes.byref(d))
    if ws is None:
        ws = workspace(need, dev, stream)
    st = fn(ctypes.byref(d), _p(logits), _p(_i32(parents, "parents")), _p(_i32(tokens, "tokens")),
            _p(out["accept_len"]), _p(out["path"]), _p(out["out_tokens"]), _p(out.get("row_status")), _p(ws),
            ctypes.c_size_t(ws.numel()), _stream(stream))
    N.check(st, name)
    return out


def verify_tree_sample(target_logits: torch.Tensor, draft_logits: torch.Tensor, parents: torch.Tensor,
                       tokens: torch.Tensor, u_accept: torch.Tensor, u_final: torch.Tensor, max_depth: int,
                       temperature: float, top_p: float = 1.0, *, out: dict | None = None,
                       ws: torch.Tensor | None = None, stream=None) -> dict:
    """Speculative-sampling verify of B draft trees (T > 0); see
    sv_verify_tree_sample.

    target_logits / draft_logits [B, N, V] (same dtype), parents/tokens [B, N]
    int32, u_accept [B, N] and u_final [B] float32.  Returns dict(accept_len
    [B], path [B, D+1], out_tokens [B, D+1], row_status [B]).
    """
    for t, n in ((target_logits, "target_logits"), (draft_logits, "draft_logits"), (parents, "parents"),
                 (tokens, "tokens"), (u_accept, "u_accept"), (u_final, "u_final")):
        _cuda(t, n)
    B, Nn, V = target_logits.shape
    if tuple(draft_logits.shape) != (B, Nn, V) or draft_logits.dtype != target_logits.dtype:
        raise ValueError("draft_logits must match target_logits in shape and dtype")
    d = N.TreeSampleDesc()
    d.batch, d.nodes, d.vocab, d.max_depth = B, Nn, V, int(max_depth)
    d.temperature, d.top_p = float(temperature), float(top_p)
    d.dtype = _code(target_logits)
    d.target_row_stride = _row_stride(target_logits, "target_logits")
    d.draft_row_stride = _row_stride(draft_logits, "draft_logits")
    dev = target_logits.device
    L = int(max_depth) + 1
    if out is None:
        out = dict(accept_len=torch.empty(B, dtype=torch.int32, device=dev),
                   path=torch.empty((B, L), dtype=torch.int32, device=dev),
                   out_tokens=torch.empty((B, L), dtype=torch.int32, device=dev),
                   row_status=torch.empty(B, dtype=torch.int32, device=dev))
    lib = N.lib()
    need = lib.sv_tree_sample_workspace_size(ctypes.byref(d))
    if need == 0:
        raise ValueError("invalid tree sampling descriptor")
    if ws is None:
        ws = workspace(need, dev, stream)
    st = lib.sv_verify_tree_sample(
        ctypes.byref(d), _p(target_logits), _p(draft_logits), _p(_i32(parents, "parents")),
        _p(_i32(tokens, "tokens")), _p(_f32(u_accept, "u_accept")), _p(_f32(u_final, "u_final")),
        _p(out["accept_len"]), _p(out["path"]), _p(out["out_tokens"]), _p(out.get("row_status")), _p(ws),
        ctypes.c_size_t(ws.numel()), _stream(stream))
    N.check(st, "sv_verify_tree_sample")
    return out


def topk(logits: torch.Tensor, k: int, *, values: bool = False, stream=None):
    """Top-k node expansion; see sv_topk.  logits [R, V] -> ids [R, k] int32
    (and their logits [R, k] float32 when ``values``)."""
    _cuda(logits, "logits")
    if logits.dim() != 2:
        raise ValueError("logits must be [rows, vocab]")
    R, V = logits.shape
    d = N.TopkDesc()
    d.rows, d.vocab, d.k = R, V, int(k)
    d.dtype = _code(logits)
    d.row_stride = _row_stride(logits, "logits")
    ids = torch.empty((R, int(k)), dtype=torch.int32, device=logits.device)
    vals = torch.empty((R, int(k)), dtype=torch.float32, device=logits.device) if values else None
    st = N.lib().sv_topk(ctypes.byref(d), _p(logits), _p(ids), _p(vals), _stream(stream))
    N.check(st, "sv_topk")
    return (ids, vals) if values else ids


def d2t_scatter(draft_logits: torch.Tensor, d2t: torch.Tensor, vocab: int, fill: float = -math.inf,
                t2d: torch.Tensor | None = None, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Scatter [R, V_d] draft logits into [R, vocab]; see sv_d2t_scatter."""
    _cuda(draft_logits, "draft_logits")
    _cuda(d2t, "d2t")
    _cuda(t2d, "t2d")
    x = draft_logits if draft_logits.dim() == 2 else draft_logits.reshape(-1, draft_logits.shape[-1])
    R, vd = x.shape
    if out is None:
        out = torch.empty((R, vocab), dtype=x.dtype, device=x.device)
    st = N.lib().sv_d2t_scatter(_p(x), _row_stride(x, "draft_logits"), _p(_i32(d2t, "d2t")),
                                _p(_i32(t2d, "t2d")), R, vd, int(vocab), _code(x), float(fill), _p(out),
                                _row_stride(out, "out"), _stream(stream))
    N.check(st, "sv_d2t_scatter")
    return out


def build_t2d(d2t: torch.Tensor, vocab: int, stream=None):
    """Inverse map of d2t; returns (t2d [vocab] int32, status [1] int32)."""
    _cuda(d2t, "d2t")
    t2d = torch.empty(int(vocab), dtype=torch.int32, device=d2t.device)
    status = torch.empty(1, dtype=torch.int32, device=d2t.device)
    st = N.lib().sv_build_t2d(_p(_i32(d2t, "d2t")), d2t.numel(), int(vocab), _p(t2d), _p(status),
                              _stream(stream))
    N.check(st, "sv_build_t2d")
    return t2d, status


def sample(logits: torch.Tensor, temperature: float, top_p: float = 1.0, u: torch.Tensor | None = None,
           *, ws: torch.Tensor | None = None, stream=None):
    """One token per row from softmax(top_p(logits / T)); see sv_sample.

    Returns (tokens [R] int32, probs [R] float32)."""
    _cuda(logits, "logits")
    _cuda(u, "u")
    x = logits if logits.dim() == 2 else logits.reshape(-1, logits.shape[-1])
    R, V = x.shape
    d = N.SampleDesc()
    d.rows, d.vocab, d.dtype = R, V, _code(x)
    d.temperature, d.top_p = float(temperature), float(top_p)
    d.row_stride = _row_stride(x, "logits")
    tok = torch.empty(R, dtype=torch.int32, device=x.device)
    prob = torch.empty(R, dtype=torch.float32, device=x.device)
    need = N.lib().sv_sample_workspace_size(ctypes.byref(d))
    if ws is None:
        ws = workspace(need, x.device, stream)
    st = N.lib().sv_sample(ctypes.byref(d), _p(x), _p(_f32(u, "u")), _p(tok), _p(prob), _p(ws),
                           ctypes.c_size_t(ws.numel()), _stream(stream))
    N.check(st, "sv_sample")
    return tok, prob


def softmax_topp(logits: torch.Tensor, temperature: float, top_p: float = 1.0, *,
                 ws: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Filtered distribution softmax(top_p_filter(logits / T)) of every row;
    see sv_softmax_topp.  Returns float32 [R, V]."""
    _cuda(logits, "logits")
    x = logits if logits.dim() == 2 else logits.reshape(-1, logits.shape[-1])
    R, V = x.shape
    d = N.SampleDesc()
    d.rows, d.vocab, d.dtype = R, V, _code(x)
    d.temperature, d.top_p = float(temperature), float(top_p)
    d.row_stride = _row_stride(x, "logits")
    out = torch.empty((R, V), dtype=torch.float32, device=x.device)
    need = N.lib().sv_sample_workspace_size(ctypes.byref(d))
    if ws is None:
        ws = workspace(need, x.device, stream)
    st = N.lib().sv_softmax_topp(ctypes.byref(d), _p(x), _p(out), V, _p(ws), ctypes.c_size_t(ws.numel()),
                                 _stream(stream))
    N.check(st, "sv_softmax_topp")
    return out
