"""The bounds-checked debug build (-DSV_DEBUG, libspec_verify_debug.so).

Every computed or data-dependent index of the kernels is checked there
before the access, and a failed check raises a flag that sv_debug_flags
returns (it never traps).  This test builds that library and runs the
small, odd-shaped parity cases of every entry point through it in a child
pytest (same oracle comparisons as the release build), with a fixture that
asserts after each case that no check failed.  The release library's
sv_debug_flags is always 0."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (file, -k expression): the small and malformed cases, not the full-size workloads.
CASES = [
    ("test_gpu_chain.py", "not full and not qwen3 and not llama3"),
    ("test_gpu_topp.py", "not 151936 and not 128256"),
    ("test_gpu_topk.py", "not 151936 and not 128256"),
    ("test_gpu_tree_path.py", "not full"),
    ("test_gpu_tree_sample.py", "not full"),
    ("test_gpu_tree_d2t_sample.py", "not full"),
]


def test_debug_build_runs_the_small_parity_cases():
    from draft_token_verification_sv_gb300 import build as b
    lib = b.build(debug=True)
    env = dict(os.environ, SPEC_VERIFY_LIBRARY=lib)
    failed = []
    for fname, expr in CASES:
        cmd = [sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider", "-k", expr,
               os.path.join(ROOT, "tests", fname)]
        r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=1200)
        tail = "\n".join(r.stdout.splitlines()[-15:])
        print(f"[debug build] {fname}: rc={r.returncode}\n{tail}")
        if r.returncode != 0 or " passed" not in r.stdout:
            failed.append((fname, r.returncode, tail + r.stderr[-2000:]))
    assert not failed, failed


def test_debug_flags_api():
    """The release library reports no flags; the debug library starts clean."""
    import draft_token_verification_sv_gb300 as sv
    from draft_token_verification_sv_gb300 import _native as N
    import __graft_entry__
    __graft_entry__.build()
    assert sv.lib().sv_debug_flags(0) == 0
    code = ("import ctypes, torch; torch.zeros(1, device='cuda'); "
            f"L = ctypes.CDLL({N.DEBUG_LIB_PATH!r}); L.sv_debug_flags.restype = ctypes.c_uint32; "
            "print(L.sv_debug_flags(1), L.sv_debug_flags(0))")
    from draft_token_verification_sv_gb300 import build as b
    b.build(debug=True)
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.split() == ["0", "0"], r.stdout
