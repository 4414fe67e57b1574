"""The C-ABI library on the host: it loads, exports every function the header
declares, its descriptor structs match the ctypes layout, and bad arguments
are rejected before anything is launched (no GPU needed: nothing here reaches
a CUDA call)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "spec_verify.h")


@pytest.fixture(scope="module")
def N():
    from draft_token_verification_sv_gb300 import build as b
    b.build()
    from draft_token_verification_sv_gb300 import _native
    _native.lib()
    return _native


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    return sorted(set(re.findall(r"\b(sv_\w+)\s*\(", src)))


def test_exports_every_declared_function(N):
    names = _declared_functions()
    assert len(names) >= 10
    lib = N.lib()
    for name in names:
        assert hasattr(lib, name), name
        assert name in N.SIGNATURES, f"binding lacks {name}"


def test_version_and_status_strings(N):
    lib = N.lib()
    assert lib.sv_version() >= 100
    for s in range(5):
        assert lib.sv_status_string(s)
    assert lib.sv_status_string(1) == b"invalid argument"


def test_struct_layout_matches_c(N, tmp_path):
    """Compile the header with gcc and compare sizes/offsets with ctypes."""
    prog = tmp_path / "layout.c"
    prog.write_text("""
#include <stdio.h>
#include <stddef.h>
#include "spec_verify.h"
int main(void) {
  printf("%zu %zu %zu %zu\\n", sizeof(sv_chain_desc), offsetof(sv_chain_desc, temperature),
         offsetof(sv_chain_desc, target_row_stride), offsetof(sv_chain_desc, draft_row_stride));
  printf("%zu %zu\\n", sizeof(sv_tree_desc), offsetof(sv_tree_desc, row_stride));
  printf("%zu %zu %zu\\n", sizeof(sv_sample_desc), offsetof(sv_sample_desc, temperature),
         offsetof(sv_sample_desc, row_stride));
  printf("%d %d %d %d %d %d\\n", SV_ROW_BAD_DRAFT_ID, SV_ROW_BAD_PARENT, SV_ROW_DEPTH_EXCEEDED,
         SV_ROW_BAD_TOKEN, SV_ROW_EMPTY, SV_ROW_RESAMPLE_FALLBACK);
  printf("%d %d %d %d\\n", SV_MAX_GAMMA, SV_MAX_VOCAB, SV_MAX_TREE_NODES, SV_MAX_TREE_DEPTH);
  return 0;
}
""")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c99", "-I", os.path.join(ROOT, "include"), str(prog), "-o", str(exe)],
                   check=True)
    lines = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")
    c = N.ChainDesc
    assert lines[0].split() == [str(ctypes.sizeof(c)), str(c.temperature.offset),
                                str(c.target_row_stride.offset), str(c.draft_row_stride.offset)]
    assert lines[1].split() == [str(ctypes.sizeof(N.TreeDesc)), str(N.TreeDesc.row_stride.offset)]
    assert lines[2].split() == [str(ctypes.sizeof(N.SampleDesc)), str(N.SampleDesc.temperature.offset),
                                str(N.SampleDesc.row_stride.offset)]
    assert [int(v) for v in lines[3].split()] == [N.SV_ROW_BAD_DRAFT_ID, N.SV_ROW_BAD_PARENT,
                                                  N.SV_ROW_DEPTH_EXCEEDED, N.SV_ROW_BAD_TOKEN,
                                                  N.SV_ROW_EMPTY, N.SV_ROW_RESAMPLE_FALLBACK]
    assert [int(v) for v in lines[4].split()] == [N.SV_MAX_GAMMA, N.SV_MAX_VOCAB, N.SV_MAX_TREE_NODES,
                                                  N.SV_MAX_TREE_DEPTH]


# Fake, 16-byte aligned "device" addresses: validation must reject the call
# before anything could dereference them.
A = ctypes.c_void_p(0x100000)
MIS = ctypes.c_void_p(0x100001)  # not even 2-byte aligned


def _chain(N, **kw):
    d = N.ChainDesc()
    d.batch, d.gamma, d.vocab, d.draft_vocab = 4, 3, 1000, 1000
    d.target_dtype = d.draft_dtype = N.SV_F32
    d.temperature, d.top_p = 1.0, 0.9
    d.target_row_stride = d.draft_row_stride = 1000
    for k, v in kw.items():
        setattr(d, k, v)
    return d


def _call_chain(N, d, ws_bytes=1 << 30, **ptr):
    p = dict(target=A, draft=A, d2t=None, t2d=None, ids=A, ua=A, ur=A, out=A, k=A, pd=None, qd=None,
             rs=None, ws=A)
    p.update(ptr)
    return N.lib().sv_verify_chain(ctypes.byref(d), p["target"], p["draft"], p["d2t"], p["t2d"],
                                   p["ids"], p["ua"], p["ur"], p["out"], p["k"], p["pd"], p["qd"],
                                   p["rs"], p["ws"], ctypes.c_size_t(ws_bytes), None)


@pytest.mark.parametrize("field,value", [
    ("gamma", 65), ("gamma", -1), ("batch", -1), ("vocab", 0), ("vocab", (1 << 24) + 1),
    ("top_p", 0.0), ("top_p", 1.5), ("top_p", float("nan")), ("temperature", -0.5),
    ("temperature", float("inf")), ("target_row_stride", 999), ("target_row_stride", -4),
    ("draft_row_stride", 999), ("target_dtype", 7), ("draft_vocab", 999),
])
def test_chain_rejects_bad_descriptor(N, field, value):
    assert _call_chain(N, _chain(N, **{field: value})) == N.SV_ERR_INVALID_ARGUMENT
    if field != "draft_vocab":  # the size query cannot tell whether a d2t map will be passed
        assert N.lib().sv_chain_workspace_size(ctypes.byref(_chain(N, **{field: value}))) == 0


def test_chain_rejects_bad_pointers(N):
    d = _chain(N)
    E = N.SV_ERR_INVALID_ARGUMENT
    assert _call_chain(N, d, target=None) == E
    assert _call_chain(N, d, target=MIS) == E
    assert _call_chain(N, d, draft=None) == E
    assert _call_chain(N, d, draft=MIS) == E
    assert _call_chain(N, d, ids=None) == E
    assert _call_chain(N, d, ua=None) == E
    assert _call_chain(N, d, ur=None) == E
    assert _call_chain(N, d, out=None) == E
    assert _call_chain(N, d, k=None) == E
    assert _call_chain(N, d, ws=None) == E
    assert _call_chain(N, d, d2t=A) == E  # d2t without t2d
    assert N.lib().sv_verify_chain(None, A, A, None, None, A, A, A, A, A, None, None, None, A,
                                   ctypes.c_size_t(1 << 30), None) == E


def test_chain_workspace_checks(N):
    d = _chain(N)
    need = N.lib().sv_chain_workspace_size(ctypes.byref(d))
    assert need > 0
    assert _call_chain(N, d, ws_bytes=need - 1) == N.SV_ERR_WORKSPACE_TOO_SMALL


def test_chain_empty_batch_is_a_noop(N):
    d = _chain(N, batch=0)
    assert _call_chain(N, d, target=None, draft=None, ids=None, out=None, k=None, ws=None) == N.SV_OK


def test_d2t_descriptor_rules(N):
    d = _chain(N, draft_vocab=300, draft_row_stride=300)
    assert N.lib().sv_chain_workspace_size(ctypes.byref(d)) > 0
    assert _call_chain(N, d, d2t=A, t2d=None) == N.SV_ERR_INVALID_ARGUMENT
    d = _chain(N, draft_vocab=1200, draft_row_stride=1200)
    assert _call_chain(N, d, d2t=A, t2d=A) == N.SV_ERR_INVALID_ARGUMENT


def test_greedy_needs_no_draft_logits(N):
    d = _chain(N, temperature=0.0)
    # Greedy ignores draft pointers: only the workspace check fails here.
    assert _call_chain(N, d, draft=None, ua=None, ur=None, ws_bytes=1) == N.SV_ERR_WORKSPACE_TOO_SMALL


def _tree(N, **kw):
    d = N.TreeDesc()
    d.batch, d.nodes, d.vocab, d.max_depth, d.dtype, d.row_stride = 2, 32, 1000, 5, N.SV_BF16, 1000
    for k, v in kw.items():
        setattr(d, k, v)
    return d


@pytest.mark.parametrize("field,value", [("nodes", 0), ("nodes", 1025), ("max_depth", -1),
                                         ("max_depth", 65), ("row_stride", 999), ("vocab", 0)])
def test_tree_rejects_bad_descriptor(N, field, value):
    d = _tree(N, **{field: value})
    assert N.lib().sv_verify_tree(ctypes.byref(d), A, A, A, A, A, A, None, A, ctypes.c_size_t(1 << 30),
                                  None) == N.SV_ERR_INVALID_ARGUMENT


def test_tree_pointer_and_workspace_checks(N):
    d = _tree(N)
    need = N.lib().sv_tree_workspace_size(ctypes.byref(d))
    assert need >= 2 * 32 * 4
    f = N.lib().sv_verify_tree
    assert f(ctypes.byref(d), None, A, A, A, A, A, None, A, ctypes.c_size_t(need), None) == 1
    assert f(ctypes.byref(d), MIS, A, A, A, A, A, None, A, ctypes.c_size_t(need), None) == 1
    assert f(ctypes.byref(d), A, A, A, A, A, A, None, A, ctypes.c_size_t(need - 1), None) == 4


def test_scatter_and_t2d_checks(N):
    f = N.lib().sv_d2t_scatter
    E = N.SV_ERR_INVALID_ARGUMENT
    assert f(A, 32, A, None, 2, 32, 16, N.SV_F32, -1.0, A, 16, None) == E   # draft_vocab > vocab
    assert f(A, 30, A, None, 2, 32, 64, N.SV_F32, -1.0, A, 64, None) == E   # in stride < draft_vocab
    assert f(A, 32, A, None, 2, 32, 64, N.SV_F32, -1.0, A, 60, None) == E   # out stride < vocab
    assert f(A, 32, None, None, 2, 32, 64, N.SV_F32, -1.0, A, 64, None) == E
    assert f(MIS, 32, A, None, 2, 32, 64, N.SV_F32, -1.0, A, 64, None) == E
    assert f(A, 32, A, None, 0, 32, 64, N.SV_F32, -1.0, A, 64, None) == N.SV_OK  # no rows
    g = N.lib().sv_build_t2d
    assert g(A, 10, 5, A, None, None) == E
    assert g(None, 3, 5, A, None, None) == E
    assert g(A, 3, 5, None, None, None) == E


def test_sample_checks(N):
    d = N.SampleDesc()
    d.rows, d.vocab, d.dtype, d.temperature, d.top_p, d.row_stride = 3, 100, N.SV_F32, 1.0, 0.9, 100
    f = N.lib().sv_sample
    need = N.lib().sv_sample_workspace_size(ctypes.byref(d))
    assert need >= 3 * 32
    assert f(ctypes.byref(d), A, None, A, None, A, ctypes.c_size_t(need), None) == 1  # no uniforms
    assert f(ctypes.byref(d), A, A, A, None, A, ctypes.c_size_t(need - 1), None) == 4
    d.top_p = 0.0
    assert f(ctypes.byref(d), A, A, A, None, A, ctypes.c_size_t(need), None) == 1


def test_missing_library_fails_loudly(N, tmp_path, monkeypatch):
    monkeypatch.setattr(N, "LIB_PATH", str(tmp_path / "nope.so"))
    monkeypatch.setattr(N, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        N.lib()


def _topk(N, **kw):
    d = N.TopkDesc()
    d.rows, d.vocab, d.k, d.dtype, d.row_stride = 4, 1000, 8, N.SV_BF16, 1000
    for k, v in kw.items():
        setattr(d, k, v)
    return d


@pytest.mark.parametrize("field,value", [("k", 0), ("k", 17), ("vocab", 0), ("rows", -1), ("row_stride", 999)])
def test_topk_rejects_bad_descriptor(N, field, value):
    d = _topk(N, **{field: value})
    assert N.lib().sv_topk(ctypes.byref(d), A, A, None, None) == N.SV_ERR_INVALID_ARGUMENT


def test_topk_k_above_vocab_and_pointers(N):
    f = N.lib().sv_topk
    E = N.SV_ERR_INVALID_ARGUMENT
    assert f(ctypes.byref(_topk(N, vocab=5, row_stride=5, k=6)), A, A, None, None) == E
    assert f(ctypes.byref(_topk(N)), None, A, None, None) == E
    assert f(ctypes.byref(_topk(N)), MIS, A, None, None) == E
    assert f(ctypes.byref(_topk(N)), A, None, None, None) == E


def test_tree_path_pointer_and_workspace_checks(N):
    d = _tree(N)
    need = N.lib().sv_tree_path_workspace_size(ctypes.byref(d))
    assert need >= 2 * 32 * (4 + 8)
    f = N.lib().sv_verify_tree_path
    assert f(ctypes.byref(d), None, A, A, A, A, A, None, A, ctypes.c_size_t(need), None) == 1
    assert f(ctypes.byref(d), A, A, A, A, A, A, None, A, ctypes.c_size_t(need - 1), None) == 4
    assert f(ctypes.byref(_tree(N, nodes=0)), A, A, A, A, A, A, None, A, ctypes.c_size_t(need), None) == 1


def _tsample(N, **kw):
    d = N.TreeSampleDesc()
    d.batch, d.nodes, d.vocab, d.max_depth = 2, 32, 1000, 5
    d.temperature, d.top_p, d.dtype = 1.0, 1.0, N.SV_BF16
    d.target_row_stride, d.draft_row_stride = 1000, 1000
    for k, v in kw.items():
        setattr(d, k, v)
    return d


@pytest.mark.parametrize("field,value", [("temperature", 0.0), ("temperature", -1.0), ("top_p", 0.0),
                                         ("top_p", 1.5), ("nodes", 0), ("nodes", 1025), ("max_depth", 65),
                                         ("draft_row_stride", 999), ("vocab", 0)])
def test_tree_sample_rejects_bad_descriptor(N, field, value):
    d = _tsample(N, **{field: value})
    assert N.lib().sv_tree_sample_workspace_size(ctypes.byref(d)) == 0
    f = N.lib().sv_verify_tree_sample
    assert f(ctypes.byref(d), A, A, A, A, A, A, A, A, A, None, A, ctypes.c_size_t(1 << 30), None) == 1


def test_tree_sample_pointer_and_workspace_checks(N):
    d = _tsample(N)
    need = N.lib().sv_tree_sample_workspace_size(ctypes.byref(d))
    assert need >= 2 * 2 * 32 * 32                      # target and draft row statistics
    assert N.lib().sv_tree_sample_workspace_size(ctypes.byref(_tsample(N, top_p=0.9))) > need
    f = N.lib().sv_verify_tree_sample
    sz = ctypes.c_size_t(need)
    assert f(ctypes.byref(d), None, A, A, A, A, A, A, A, A, None, A, sz, None) == 1
    assert f(ctypes.byref(d), A, MIS, A, A, A, A, A, A, A, None, A, sz, None) == 1
    assert f(ctypes.byref(d), A, A, A, A, None, A, A, A, A, None, A, sz, None) == 1
    assert f(ctypes.byref(d), A, A, A, A, A, A, A, A, A, None, A, ctypes.c_size_t(need - 1), None) == 4
    assert f(ctypes.byref(_tsample(N, batch=0)), None, None, None, None, None, None, None, None, None, None,
             None, ctypes.c_size_t(0), None) == 0
