"""The multi-process host logic of bench.py on CPU: two gloo ranks (the
rendezvous on 127.0.0.1) reduce their timings and units the way the GPU run
does -- the slowest rank's time, the sum of the units -- and the reference
arm runs on rank 0 alone, the other ranks leaving without output."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

WORKER = r"""
import json, os, sys
sys.path.insert(0, os.environ["SV_ROOT"])
import bench
d = bench.Dist()
d.init(False)
rank = d.rank
ms = [3.0, 5.0][rank]
units = [100.0, 300.0][rank]
t_max = d.max(ms)
u_sum = d.sum(units)
d.barrier()
d.close()
print(json.dumps({"rank": rank, "t_max": t_max, "u_sum": u_sum}))
"""


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _launch(code_or_args, world=2, extra_env=None):
    port = _free_port()
    procs = []
    for r in range(world):
        env = dict(os.environ, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(r),
                   LOCAL_RANK=str(r), WORLD_SIZE=str(world), SV_ROOT=ROOT, CUDA_VISIBLE_DEVICES="")
        env.update(extra_env or {})
        cmd = [sys.executable, "-c", code_or_args] if isinstance(code_or_args, str) else \
            [sys.executable] + code_or_args
        procs.append(subprocess.Popen(cmd, env=env, cwd=ROOT, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        try:
            out, err = p.communicate(timeout=180)
        except subprocess.TimeoutExpired:
            p.kill()
            out, err = p.communicate()
        outs.append((p.returncode, out, err))
    return outs


def test_two_gloo_ranks_reduce_like_the_gpu_run():
    pytest.importorskip("torch.distributed")
    outs = _launch(WORKER)
    for rc, out, err in outs:
        assert rc == 0, err[-2000:]
    res = [json.loads(out.strip().splitlines()[-1]) for _, out, _ in outs]
    for r in res:
        assert r["t_max"] == 5.0          # the slowest rank's time
        assert r["u_sum"] == 400.0        # every rank's units
    sys.path.insert(0, ROOT)
    import bench
    value, t = bench.aggregate([3.0, 5.0], [100.0, 300.0])
    assert t == 5.0 and value == pytest.approx(400.0 / 5e-3)


def test_reference_arm_runs_on_rank_zero_only():
    outs = _launch(["bench.py", "--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "1",
                    "--reference-seconds", "5"])
    (rc0, out0, err0), (rc1, out1, err1) = outs
    assert rc0 == 0, err0[-2000:]
    assert rc1 == 0, err1[-2000:]
    assert out1.strip() == ""
    line = json.loads(out0.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "rows/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0
