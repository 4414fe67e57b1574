#!/usr/bin/env python
"""Throughput of the speculative-decoding verify step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one full verify call (every kernel of the path) over one batch of
synthetic logits already resident in HBM.  The default workload is the
largest single-GPU setting: Qwen3-vocabulary chain verify with an EAGLE3
draft vocabulary (B=256, γ=7, V=151936 fp32 target rows, 32000-id fp32 draft
rows mapped through d2t, T=1, top_p=0.95); --workload selects another of the
pages' settings.  Rank 0 prints one JSON
line.  Under torchrun every rank verifies its own batch (weak scaling, no
data-path collective); timing is the max over ranks.

The timed region replays the K steps from a CUDA graph (no host launch gaps)
and rotates over enough copies of the inputs that they exceed 4x the L2
cache, so every step reads its logits from HBM; the graph is replayed
--repeats times and the median replay is reported, with the spread.  A
second, instrumented graph records CUDA events around each kernel (on the
kernels' stream); the dominant kernel's time per step for the roofline is
the smaller of its median event-timed duration and the median step time
(both bound it from above).
"e2e" is the same metric through the public Python call with the step's
inputs copied from pinned host memory and its outputs copied back, every
step; the copy of step i+1's inputs (on a copy stream, into a second device
buffer) overlaps the verify of step i.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0
WORKLOADS = {
    "tiny": synth.TINY,
    "smollm2": synth.SMOLLM2,
    "llama3-greedy": synth.LLAMA3_GREEDY,
    "llama3-sample": synth.LLAMA3_SAMPLE,
    "qwen3-d2t": synth.QWEN3_D2T,
    "tree": synth.TREE,
    "tree-path": synth.TREE,
    "tree-topk": synth.TREE,
    "tree-sample": synth.TREE_SAMPLE,
}
# Top-k node expansion (sv_topk, k = 8) over the tree workload's node rows.
TOPK = {"tree-topk": 8}
# Workloads verified by the path walk (sv_verify_tree_path): only the rows of
# the accepted frontier are read.
PATH_WALK = {"tree-path"}
DEFAULT_WORKLOAD = "qwen3-d2t"


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="CPU budget of the oracle baseline sample")
    ap.add_argument("--reference-seconds", type=float, default=150.0,
                    help="wall budget of the whole --impl reference run")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--repeats", type=int, default=11,
                    help="replays of the K-step graph; the median replay is reported")
    return ap.parse_args(argv)


# ------------------------------------------------------------ distributed ----

class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None

    def init(self, device_ok: bool):
        if self.world > 1:
            import torch.distributed as dist
            dist.init_process_group("nccl" if device_ok else "gloo")
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x: float) -> float:
        return self._reduce(x, "max")

    def sum(self, x: float) -> float:
        return self._reduce(x, "sum")

    def _reduce(self, x: float, op: str) -> float:
        if not self.pg:
            return x
        import torch
        dev = torch.device("cuda", self.local_rank) if torch.cuda.is_available() else torch.device("cpu")
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX if op == "max" else self.pg.ReduceOp.SUM)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


def aggregate(times_ms: list[float], units: list[float]) -> tuple[float, float]:
    """Whole-job throughput from per-rank (elapsed ms, units): units summed,
    time = the slowest rank.  Returns (units per second, max ms)."""
    t = max(times_ms)
    return sum(units) / (t / 1e3), t


# ------------------------------------------------------------------ peaks ----

def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def ncu_traffic(workload: str, kernel: str):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    summary is missing or was taken on different kernel sources."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.md")
    try:
        lines = open(path).read().splitlines()
    except OSError:
        return None
    src = source_hash(kernel)
    for ln in lines:
        cells = [c.strip() for c in ln.strip().strip("|").split("|")]
        if len(cells) >= 4 and cells[0] == workload and cells[1] == kernel:
            try:
                traffic, h = float(cells[2]), cells[3]
            except ValueError:
                continue
            return traffic if h == src else None
    return None


KERNEL_SOURCES = {
    "topp_slice_kernel": "sv_topp.cu",
    "stats_stream_kernel": "sv_chain.cu",
    "decide_kernel": "sv_decide.cu",
    "greedy_kernel(chain)": "sv_greedy.cu",
    "greedy_kernel(tree)": "sv_greedy.cu",
    "topk_kernel": "sv_topk.cu",
    "tree_sample_kernel": "sv_tree_sample.cu",
    "walk_level_kernel (all levels)": "sv_tree_walk.cu",
}


def source_hash(kernel: str | None = None) -> str:
    """Hash of the sources a kernel is built from: its .cu file and the
    shared headers (every source when the kernel is not listed)."""
    d = os.path.join(ROOT, "draft_token_verification_sv_gb300", "csrc")
    own = KERNEL_SOURCES.get(kernel) if kernel else None
    h = hashlib.sha256()
    for name in sorted(os.listdir(d)):
        if name.endswith((".cuh", ".h")) or (name.endswith(".cu") and (own is None or name == own)):
            h.update(name.encode())
            h.update(open(os.path.join(d, name), "rb").read())
    return h.hexdigest()[:12]


# ----------------------------------------------------------------- clocks ----

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.proc = None
        self.out = None

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"]
        if self.uuid:
            cmd += ["-i", self.uuid]
        try:
            self.out = tempfile.TemporaryFile(mode="w+")
            self.proc = subprocess.Popen(cmd, stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self) -> dict | None:
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            self.proc.wait()
        self.out.seek(0)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.out.read().splitlines():
            cells = [c.strip() for c in ln.split(",")]
            if len(cells) < 7:
                continue
            try:
                sm.append(float(cells[0]))
                mx.append(float(cells[1]))
            except ValueError:
                continue
            for n, c in zip(names, cells[3:7]):
                if c.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------- workloads ----

def make_inputs(cfg, dev, sv):
    """Seeded inputs on the device, plus draft ids drawn by the library's
    draft sampler from the uniforms (outside any timed region)."""
    import torch
    if isinstance(cfg, synth.TreeSampleConfig):
        x = synth.make_tree_sample_inputs(cfg)

        def as_t(store):
            t = torch.from_numpy(np.ascontiguousarray(store).view(np.int16)).view(torch.bfloat16) \
                if cfg.dtype == "bf16" else torch.from_numpy(store)
            return t.to(dev)
        return dict(host=x, logits=as_t(x["logits_store"]), draft=as_t(x["draft_store"]),
                    parents=torch.from_numpy(x["parents"]).to(dev), tokens=torch.from_numpy(x["tokens"]).to(dev),
                    u_accept=torch.from_numpy(x["u_accept"]).to(dev), u_final=torch.from_numpy(x["u_final"]).to(dev))
    if isinstance(cfg, synth.TreeConfig):
        x = synth.make_tree_inputs(cfg)
        store = x["logits_store"]
        logits = torch.from_numpy(store.view(np.int16)).view(torch.bfloat16) if cfg.dtype == "bf16" \
            else torch.from_numpy(store)
        return dict(host=x, logits=logits.to(dev), parents=torch.from_numpy(x["parents"]).to(dev),
                    tokens=torch.from_numpy(x["tokens"]).to(dev))
    x = synth.make_chain_inputs(cfg)

    def as_t(store):
        if cfg.dtype == "bf16":
            return torch.from_numpy(np.ascontiguousarray(store).view(np.int16)).view(torch.bfloat16).to(dev)
        return torch.from_numpy(np.ascontiguousarray(store)).to(dev)

    target, draft = as_t(x["target_store"]), as_t(x["draft_store"])
    B, G = x["batch"], x["gamma"]
    u_draft = torch.from_numpy(x["u_draft"]).to(dev)
    tok, _ = sv.sample(draft.reshape(B * G, -1), cfg.temperature, cfg.top_p,
                       u_draft.reshape(-1) if cfg.temperature > 0 else None)
    d2t = t2d = None
    if x["d2t"] is not None:
        d2t = torch.from_numpy(x["d2t"]).to(dev)
        t2d = sv.build_t2d(d2t, x["vocab"])[0]
        tok = d2t[tok.long()]
    ids = tok.reshape(B, G).to(torch.int32).contiguous()
    torch.cuda.synchronize()
    x["draft_ids"] = ids.cpu().numpy()
    return dict(host=x, target=target, draft=draft, ids=ids, d2t=d2t, t2d=t2d,
                u_accept=torch.from_numpy(x["u_accept"]).to(dev),
                u_resample=torch.from_numpy(x["u_resample"]).to(dev))


def step_bytes(cfg) -> int:
    return cfg.algorithmic_bytes()


class Runner:
    """Pre-marshalled C-ABI calls, one per rotating input set."""

    def __init__(self, sv, cfg, inputs, nsets, dev, path_walk=False, topk=0):
        import torch
        from draft_token_verification_sv_gb300 import _native as N
        from draft_token_verification_sv_gb300.verify import chain_desc
        self.N = N
        self.lib = N.lib()
        self.cfg = cfg
        self.tree = isinstance(cfg, synth.TreeConfig)
        self.sample = isinstance(cfg, synth.TreeSampleConfig)
        self.sets = []
        self.keep = []
        vp = lambda t: ctypes.c_void_p(t.data_ptr()) if t is not None else None
        if self.sample:
            d = N.TreeSampleDesc()
            d.batch, d.nodes, d.vocab, d.max_depth = cfg.batch, cfg.nodes, cfg.vocab, cfg.max_depth
            d.temperature, d.top_p = cfg.temperature, cfg.top_p
            d.dtype = N.SV_BF16 if cfg.dtype == "bf16" else N.SV_F32
            d.target_row_stride = d.draft_row_stride = cfg.vocab
            self.desc = d
            ws_need = self.lib.sv_tree_sample_workspace_size(ctypes.byref(d))
        elif self.tree:
            B, Nn = cfg.batch, cfg.nodes
            d = N.TreeDesc()
            d.batch, d.nodes, d.vocab, d.max_depth = B, Nn, cfg.vocab, cfg.max_depth
            d.dtype = N.SV_BF16 if cfg.dtype == "bf16" else N.SV_F32
            d.row_stride = cfg.vocab
            self.desc = d
            ws_need = (self.lib.sv_tree_path_workspace_size if path_walk else
                       self.lib.sv_tree_workspace_size)(ctypes.byref(d))
        else:
            d = chain_desc(inputs["target"], inputs["draft"], cfg.temperature, cfg.top_p, inputs["d2t"])
            self.desc = d
            ws_need = self.lib.sv_chain_workspace_size(ctypes.byref(d))
        self.ws = torch.zeros(ws_need, dtype=torch.uint8, device=dev)
        L = cfg.max_depth + 1 if self.tree else cfg.gamma + 1
        B = cfg.batch
        self.out = dict(tokens=torch.empty((B, L), dtype=torch.int32, device=dev),
                        k=torch.empty(B, dtype=torch.int32, device=dev),
                        status=torch.empty(B, dtype=torch.int32, device=dev),
                        path=torch.empty((B, L), dtype=torch.int32, device=dev))
        o = self.out
        for s in range(nsets):
            if self.sample:
                lg = inputs["logits"] if s == 0 else inputs["logits"].clone()
                dr = inputs["draft"] if s == 0 else inputs["draft"].clone()
                self.keep += [lg, dr]
                args = (ctypes.byref(self.desc), vp(lg), vp(dr), vp(inputs["parents"]), vp(inputs["tokens"]),
                        vp(inputs["u_accept"]), vp(inputs["u_final"]), vp(o["k"]), vp(o["path"]), vp(o["tokens"]),
                        vp(o["status"]), vp(self.ws), ctypes.c_size_t(self.ws.numel()))
            elif self.tree:
                lg = inputs["logits"] if s == 0 else inputs["logits"].clone()
                self.keep.append(lg)
                args = (ctypes.byref(self.desc), vp(lg), vp(inputs["parents"]), vp(inputs["tokens"]),
                        vp(o["k"]), vp(o["path"]), vp(o["tokens"]), vp(o["status"]), vp(self.ws),
                        ctypes.c_size_t(self.ws.numel()))
            else:
                tg = inputs["target"] if s == 0 else inputs["target"].clone()
                dr = None
                if cfg.temperature > 0:
                    dr = inputs["draft"] if s == 0 else inputs["draft"].clone()
                self.keep += [tg, dr]
                args = (ctypes.byref(self.desc), vp(tg), vp(dr), vp(inputs["d2t"]), vp(inputs["t2d"]),
                        vp(inputs["ids"]), vp(inputs["u_accept"]), vp(inputs["u_resample"]),
                        vp(o["tokens"]), vp(o["k"]), None, None, vp(o["status"]), vp(self.ws),
                        ctypes.c_size_t(self.ws.numel()))
            self.sets.append(args)
        self.fn = (self.lib.sv_verify_tree_path if path_walk else self.lib.sv_verify_tree) if self.tree \
            else self.lib.sv_verify_chain
        if self.sample:
            self.fn = self.lib.sv_verify_tree_sample
        if topk:
            # Every node row of every tree: R = B*N rows, k ids each.
            kd = N.TopkDesc()
            kd.rows, kd.vocab, kd.k = cfg.batch * cfg.nodes, cfg.vocab, topk
            kd.dtype, kd.row_stride = self.desc.dtype, cfg.vocab
            self.kdesc = kd
            self.out["ids"] = torch.empty((cfg.batch * cfg.nodes, topk), dtype=torch.int32, device=dev)
            self.sets = [(ctypes.byref(kd), a[1], vp(self.out["ids"]), None) for a in self.sets]
            self.fn = self.lib.sv_topk

    def step(self, s: int, stream_handle):
        st = self.fn(*self.sets[s % len(self.sets)], stream_handle)
        if st != 0:
            raise RuntimeError(f"verify call failed with status {st}")


def n_sets_for(cfg) -> int:
    per = step_bytes(cfg)
    return max(2, math.ceil(4 * L2_BYTES / per))


# ------------------------------------------------------------- our arm ----

def run_ours(args, dist: Dist):
    import torch
    import draft_token_verification_sv_gb300 as sv
    from draft_token_verification_sv_gb300 import build as b
    b.build()
    assert torch.cuda.is_available(), "bench needs a CUDA device"
    dev = torch.device("cuda", dist.local_rank)
    torch.cuda.set_device(dev)
    dist.init(True)
    cfg = WORKLOADS[args.workload]
    inputs = make_inputs(cfg, dev, sv)
    nsets = n_sets_for(cfg)
    if args.workload in PATH_WALK:
        nsets = max(nsets, 4)  # the walk reads a fifth of the rows: rotate further
    walk = args.workload in PATH_WALK
    R = Runner(sv, cfg, inputs, nsets, dev, path_walk=walk, topk=TOPK.get(args.workload, 0))
    lib = R.lib
    stream = torch.cuda.Stream(device=dev)
    sh = ctypes.c_void_p(stream.cuda_stream)
    K, W = args.steps, args.warmup

    # Warm-up (also sets kernel attributes before any capture).
    with torch.cuda.stream(stream):
        for s in range(max(W, 3)):
            R.step(s, sh)
    stream.synchronize()

    # Pure graph of K steps.
    launches0 = lib.sv_launch_count()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for s in range(K):
            R.step(s, sh)
    launches = int(lib.sv_launch_count() - launches0)
    per_step_launches = launches // K

    # Instrumented graph: events around every kernel of every step.
    nph = per_step_launches + 1
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(nph)] for _ in range(K)]
    with torch.cuda.stream(stream):
        for row in events:
            for e in row:
                e.record(stream)
    stream.synchronize()
    handles = [(ctypes.c_void_p * nph)(*[ctypes.c_void_p(e.cuda_event) for e in row]) for row in events]
    gi = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gi, stream=stream):
        for s in range(K):
            lib.sv_set_phase_events(handles[s], nph)
            R.step(s, sh)

    # Clock samples over a load window that ends with the timed region.
    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
        uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        uuid = None
    sampler = ClockSampler(uuid)
    sampler.start()
    t_end = time.time() + 1.5
    with torch.cuda.stream(stream):
        while time.time() < t_end:
            g.replay()
            stream.synchronize()

    # The timed region: R replays of the K-step graph, each bracketed by a
    # barrier and a synchronize; the median replay is reported.
    reps = max(1, args.repeats)
    rep_ms = []
    for _ in range(reps):
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        dist.barrier()
        with torch.cuda.stream(stream):
            start.record(stream)
            g.replay()
            end.record(stream)
        torch.cuda.synchronize()
        dist.barrier()
        rep_ms.append(start.elapsed_time(end))
    clocks = sampler.stop()
    elapsed = statistics.median(rep_ms)

    # Instrumented replays: per-kernel durations (events around every kernel
    # of every step; medians over steps and replays).
    phase_all = [[] for _ in range(nph - 1)]
    for _ in range(min(reps, 5)):
        with torch.cuda.stream(stream):
            gi.replay()
        torch.cuda.synchronize()
        for row in events:
            for i in range(nph - 1):
                phase_all[i].append(row[i].elapsed_time(row[i + 1]))
    avg_phase = [statistics.median(p) for p in phase_all]

    units = cfg.rows_metric * K
    t_max = dist.max(elapsed)
    tot_units = dist.sum(units)
    value = tot_units / (t_max / 1e3)

    # End to end through the public call, pinned host inputs each step.
    e2e = run_e2e(cfg, inputs, sv, dev, stream, K, dist, path_walk=walk, topk=TOPK.get(args.workload, 0))

    peak, peak_kind = hbm_peak()
    dom = 0
    dom_name = {True: "greedy_kernel(tree)", False: None}[R.tree]
    if args.workload in TOPK:
        dom_name = "topk_kernel"
    if R.sample:
        # The statistics pass over every target and draft row; the walk reads
        # only the visited nodes' rows after it.
        dom_name = "topp_slice_kernel" if cfg.top_p < 1 else "stats_stream_kernel"
    if not R.tree:
        dom_name = "greedy_kernel(chain)" if cfg.temperature == 0 else (
            "topp_slice_kernel" if cfg.top_p < 1 else "stats_stream_kernel")
    bytes_dom, dom_phases = step_bytes(cfg), [dom]
    if walk:
        # Rows read: (accept_len + 1) per tree (distinct sibling tokens), over
        # every level launch (phase 0 is the validation launch).
        acc = R.out["k"].cpu().numpy().astype(np.int64)
        bytes_dom = int((acc + 1).sum()) * cfg.vocab * (2 if cfg.dtype == "bf16" else 4)
        dom_phases = list(range(1, nph - 1))
        dom_name = "walk_level_kernel (all levels)"
    # The dominant kernel's time per step: its median event-timed duration
    # (an event pair around a kernel inside a graph adds the gap of the event
    # records, a microsecond or two) or the median step time, whichever is
    # smaller.  Both bound the kernel's own duration from above, so the
    # fraction of the roofline below is a lower bound.
    ms_step = t_max / K
    ms_event = sum(avg_phase[i] for i in dom_phases)
    ms_dom = min(ms_event, ms_step)
    achieved = bytes_dom / (ms_dom / 1e3) / 1e9
    traffic = ncu_traffic(args.workload, dom_name)
    res = {
        "metric": "verify rows/s (B*(2*gamma+1) rows per chain step, B*N per tree step)",
        "value": value,
        "unit": "rows/s",
        "n_gpus": dist.world,
        "steps": K,
        "warmup": W,
        "ms_per_step": ms_step,
        "ms_per_step_spread": [min(rep_ms) / K, max(rep_ms) / K],
        "repeats": reps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if cfg.dtype == "bf16" else "f32",
        "data": "synthetic (seeded, shapes and value recipe of the pages' settings)",
        "config": config_of(cfg, args.workload, nsets, dist.world),
        "hbm_gbs_algorithmic": (bytes_dom if walk else step_bytes(cfg)) * K / (elapsed / 1e3) / 1e9,
        "roofline": {"bound": "hbm", "kernel": dom_name, "achieved": achieved, "peak": peak,
                     "peak_source": f"hbm_gbs of {peak_kind}", "unit": "GB/s", "frac": achieved / peak,
                     "traffic": traffic, "bytes_per_launch": bytes_dom,
                     "avg_launch_ms": ms_dom, "event_ms": ms_event,
                     "timing": "the smaller of the kernel's median event-timed duration and the median step time"},
        "phase_ms": avg_phase,
        "gpu_launches": launches,
        "e2e": e2e,
        "clocks": clocks,
    }
    if args.workload not in TOPK:
        # Accepted drafts per batch row in the last replayed step.
        try:
            res["mean_accepted"] = float(R.out["k"].float().mean().item())
        except Exception:
            res["mean_accepted"] = None
    if dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline:
        sampled = []
        res["cpu_baseline"] = cpu_baseline(cfg, inputs, args.cpu_seconds, sink=sampled)
        if args.workload not in TOPK:
            try:
                res["parity_sample"] = parity_sample(cfg, sampled, R.out["tokens"].cpu().numpy())
            except Exception as e:  # never let the cross-check cost the measurement
                res["parity_sample"] = {"error": str(e)[:200]}
    dist.close()
    return res


def config_of(cfg, workload, nsets, world):
    l2 = f"{nsets} rotating input copies ({nsets * step_bytes(cfg) / 1e6:.0f} MB > 4x L2)" if nsets else \
        "not applicable (CPU oracle)"
    c = {"workload": workload, "batch": cfg.batch, "vocab": cfg.vocab, "dtype": cfg.dtype, "l2": l2,
         "parallelism": f"replicas x{world} (batch rows independent)"}
    if isinstance(cfg, synth.TreeSampleConfig):
        c.update(nodes=cfg.nodes, max_depth=cfg.max_depth, temperature=cfg.temperature, top_p=cfg.top_p)
    elif isinstance(cfg, synth.TreeConfig):
        c.update(nodes=cfg.nodes, max_depth=cfg.max_depth, temperature=0.0)
    else:
        c.update(gamma=cfg.gamma, temperature=cfg.temperature, top_p=cfg.top_p,
                 draft_vocab=cfg.draft_vocab or cfg.vocab)
    return c


def run_e2e(cfg, inputs, sv, dev, stream, K, dist, path_walk=False, topk=0):
    import torch
    tree = isinstance(cfg, synth.TreeConfig)
    sample = isinstance(cfg, synth.TreeSampleConfig)
    names = ["logits", "parents", "tokens"] if tree else \
        ["target", "draft", "ids", "u_accept", "u_resample"]
    if sample:
        names = ["logits", "draft", "parents", "tokens", "u_accept", "u_final"]
    if topk:
        names = ["logits"]
    if not tree and cfg.temperature == 0:
        names = ["target", "ids"]
    host = {n: inputs[n].cpu().pin_memory() for n in names}
    # Two device copies of the inputs: step i+1's inputs are copied (on a copy
    # stream) while step i is verified; events order each buffer's reuse.
    bufs = [{n: torch.empty_like(inputs[n]) for n in names} for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    L = cfg.max_depth + 1 if tree else cfg.gamma + 1
    if topk:
        L = cfg.nodes * topk
    out_host = torch.empty((cfg.batch, L), dtype=torch.int32).pin_memory()
    k_host = torch.empty(cfg.batch, dtype=torch.int32).pin_memory()
    d2h = out_host.numel() * 4 + (0 if topk else k_host.numel() * 4)

    copy_stream = torch.cuda.Stream(device=dev)
    ready = [torch.cuda.Event() for _ in range(2)]
    free = [torch.cuda.Event() for _ in range(2)]
    for e in free:
        e.record(stream)

    def one(i):
        devb = bufs[i % 2]
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_event(free[i % 2])
            for n in names:
                devb[n].copy_(host[n], non_blocking=True)
            ready[i % 2].record(copy_stream)
        stream.wait_event(ready[i % 2])
        if topk:
            ids = sv.topk(devb["logits"].reshape(cfg.batch * cfg.nodes, cfg.vocab), topk)
            out_host.copy_(ids.reshape(cfg.batch, -1), non_blocking=True)
        elif sample:
            o = sv.verify_tree_sample(devb["logits"], devb["draft"], devb["parents"], devb["tokens"],
                                      devb["u_accept"], devb["u_final"], cfg.max_depth, cfg.temperature, cfg.top_p)
            out_host.copy_(o["out_tokens"], non_blocking=True)
            k_host.copy_(o["accept_len"], non_blocking=True)
        elif tree:
            o = sv.verify_tree(devb["logits"], devb["parents"], devb["tokens"], cfg.max_depth, path_walk=path_walk)
            out_host.copy_(o["out_tokens"], non_blocking=True)
            k_host.copy_(o["accept_len"], non_blocking=True)
        else:
            o = sv.verify_chain(devb["target"], devb.get("draft"), devb["ids"], devb.get("u_accept"),
                                devb.get("u_resample"), cfg.temperature, cfg.top_p, d2t=inputs["d2t"],
                                t2d=inputs["t2d"], probs=False)
            out_host.copy_(o["tokens"], non_blocking=True)
            k_host.copy_(o["num_accepted"], non_blocking=True)
        free[i % 2].record(stream)

    with torch.cuda.stream(stream):
        for i in range(3):
            one(i)
        torch.cuda.synchronize()
        dist.barrier()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        copy_stream.wait_event(start)
        for i in range(K):
            one(i)
        end.record(stream)
    torch.cuda.synchronize()
    dist.barrier()
    ms = dist.max(start.elapsed_time(end))
    units = dist.sum(cfg.rows_metric * K)
    return {"value": units / (ms / 1e3), "unit": "rows/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": ms / K}


# ------------------------------------------------------ oracle baselines ----

def oracle_rows(cfg, host, rows):
    from oracle import sv_oracle as O
    if isinstance(cfg, synth.TreeSampleConfig):
        return O.verify_tree_sample(host["logits"], host["draft_logits"], host["parents"], host["tokens"],
                                    host["u_accept"], host["u_final"], cfg.temperature, cfg.top_p,
                                    host["max_depth"], rows=rows)
    if isinstance(cfg, synth.TreeConfig):
        return O.verify_tree(host["logits"], host["parents"], host["tokens"], host["max_depth"], rows=rows)
    return O.verify_chain(host["target"], host["draft"] if cfg.temperature > 0 else None,
                          host["draft_ids"], host["u_accept"], host["u_resample"], cfg.temperature,
                          cfg.top_p, d2t=host["d2t"], rows=rows)


def units_per_batch_row(cfg) -> int:
    return cfg.nodes if isinstance(cfg, synth.TreeConfig) else 2 * cfg.gamma + 1


def host_cores() -> int:
    """Host cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


# The oracle runs one batch row per task in worker processes (started with
# "spawn": a forked child of a process that has used CUDA can hang).  The
# inputs reach the workers through shared memory, not through pickling.
_WORKER = {}


def _share_host(host):
    """Copy the host input arrays into shared memory; returns (spec, blocks)."""
    from multiprocessing import shared_memory
    spec, blocks = {}, []
    for k, v in host.items():
        if isinstance(v, np.ndarray):
            shm = shared_memory.SharedMemory(create=True, size=max(1, v.nbytes))
            np.ndarray(v.shape, v.dtype, buffer=shm.buf)[...] = v
            spec[k] = ("shm", shm.name, v.shape, v.dtype.str)
            blocks.append(shm)
        elif k != "cfg":
            spec[k] = ("val", v)
    return spec, blocks


def _worker_init(cfg, spec):
    from multiprocessing import shared_memory
    host, keep = {}, []
    for k, sp in spec.items():
        if sp[0] == "shm":
            # The parent owns and unlinks the block; attaching registers the
            # same name with the shared resource tracker again, which the
            # parent's unlink then removes once.
            shm = shared_memory.SharedMemory(name=sp[1])
            keep.append(shm)
            host[k] = np.ndarray(sp[2], np.dtype(sp[3]), buffer=shm.buf)
        else:
            host[k] = sp[1]
    _WORKER.update(cfg=cfg, host=host, keep=keep)


def _worker_row(b):
    """Oracle output of batch row b: (b, token row, margin, the other token
    rows admissible under top-p cuts within 1e-6 of top_p)."""
    cfg, host = _WORKER["cfg"], _WORKER["host"]
    out = oracle_rows(cfg, host, [b])
    tree = isinstance(cfg, synth.TreeConfig)
    tokens = np.asarray(out["out_tokens"][b] if tree else out["tokens"][b], dtype=np.int64)
    margin = out.get("margin")
    others = []
    if "final_alts" in out:
        k = int(out["accept_len"][b] if tree else out["num_accepted"][b])
        for tok in out["final_alts"][b][1:]:
            if tok >= 0:
                alt = tokens.copy()
                alt[k] = tok
                others.append(alt)
    return b, tokens, (float(margin[b]) if margin is not None else float("inf")), others


class OraclePool:
    """The fp64 oracle over batch rows on every host core."""

    def __init__(self, cfg, host, cores=None):
        import multiprocessing as mp
        self.cores = cores or host_cores()
        self.spec, self.blocks = _share_host(host)
        ctx = mp.get_context("spawn")
        self.pool = ctx.Pool(self.cores, initializer=_worker_init, initargs=(cfg, self.spec))

    def rows(self, rows, budget_s=None):
        """Oracle outputs of ``rows`` (all of them, or as many as finish
        within ``budget_s`` seconds of wall time, at least one)."""
        t0 = time.perf_counter()
        done = []
        it = self.pool.imap_unordered(_worker_row, list(rows))
        for r in it:
            done.append(r)
            if budget_s is not None and time.perf_counter() - t0 > budget_s:
                break
        return done, time.perf_counter() - t0

    def close(self):
        self.pool.terminate()
        self.pool.join()
        for shm in self.blocks:
            shm.close()
            shm.unlink()


def cpu_baseline(cfg, inputs, seconds, sink=None, cores=None):
    """The fp64 oracle as it stands, one batch row per task on every host
    core, over batch rows of the same workload until about ``seconds`` of
    wall time is spent (at least one row per core).  Each finished row's
    (row, oracle tokens, margin, other admissible token rows) is appended to
    ``sink``."""
    host = inputs["host"]
    B = cfg.batch
    pool = OraclePool(cfg, host, cores)
    try:
        pool.rows(range(min(B, pool.cores)))  # start-up of the workers, untimed
        done, dt = pool.rows(range(B), budget_s=seconds)
    finally:
        pool.close()
    if sink is not None:
        sink.extend(done)
    return {"value": len(done) * units_per_batch_row(cfg) / dt, "unit": "rows/s", "cores": pool.cores,
            "kind": "oracle",
            "sample": f"{len(done)} of {B} batch rows of the {cfg.name} workload, fp64 numpy, "
                      f"one batch row per task on {pool.cores} worker processes"}


def parity_sample(cfg, sampled, got_tokens) -> dict:
    """The batch rows the oracle computed for the CPU baseline against the
    library's tokens for the same rows of the timed workload: how many rows
    differ from every token row the oracle admits, and how many of those
    have an oracle decision within the near-threshold margin (1e-6 in the
    uniform's units)."""
    from oracle import sv_oracle as O
    tol = O.NEAR
    mismatch = near = 0
    for b, want, margin, others in sampled:
        got = np.asarray(got_tokens[b], dtype=np.int64)
        if not any(np.array_equal(got, w) for w in [want] + list(others)):
            mismatch += 1
            if margin < tol:
                near += 1
    return {"rows": len(sampled), "mismatch": mismatch, "near_threshold": near}


def oracle_draft_ids(cfg, host, rows):
    """Draft ids of the given batch rows, drawn by the oracle from q with the
    seeded uniforms (argmax at T = 0)."""
    from oracle import sv_oracle as O
    G = host["gamma"]
    ids = host.setdefault("draft_ids", np.zeros((host["batch"], G), np.int32))
    d2t = host["d2t"]
    for b in rows:
        for i in range(G):
            tok, _ = O.sample_row(host["draft"][b, i], cfg.temperature, cfg.top_p,
                                  float(host["u_draft"][b, i]), tie_index=d2t)
            ids[b, i] = d2t[tok] if d2t is not None else tok


def run_reference(args, dist: Dist):
    """The oracle timed as the reference arm: K steps, each a bounded sample
    of batch rows of the same workload, one batch row per task on every host
    core."""
    cfg = WORKLOADS[args.workload]
    chain = not isinstance(cfg, synth.TreeConfig)
    host = synth.make_chain_inputs(cfg) if chain else (
        synth.make_tree_sample_inputs(cfg) if isinstance(cfg, synth.TreeSampleConfig) else synth.make_tree_inputs(cfg))
    if chain:
        oracle_draft_ids(cfg, host, [0])
    t0 = time.perf_counter()
    oracle_rows(cfg, host, [0])
    t_row = max(time.perf_counter() - t0, 1e-3)
    K, W = args.steps, args.warmup
    cores = host_cores()
    # Rows per step: whole rounds of one row per core, within the wall budget.
    rounds = max(1, int(args.reference_seconds / (K + W) / t_row))
    per_step = max(1, min(cfg.batch, rounds * cores))
    rows = list(range(per_step))
    if chain:
        oracle_draft_ids(cfg, host, rows[1:])
    pool = OraclePool(cfg, host, cores)
    try:
        for _ in range(W):
            pool.rows(rows[:cores])
        times = []
        for _ in range(K):
            _, dt = pool.rows(rows)
            times.append(dt)
    finally:
        pool.close()
    total = sum(times)
    value = K * per_step * units_per_batch_row(cfg) / total
    return {"impl": "reference", "metric": "verify rows/s (B*(2*gamma+1) rows per chain step, B*N per tree step)",
            "value": value, "unit": "rows/s", "n_gpus": dist.world, "steps": K, "warmup": W,
            "ms_per_step": 1e3 * total / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic (seeded)", "config": config_of(cfg, args.workload, 0, 1),
            "cpu_baseline": {"value": value, "unit": "rows/s", "cores": cores, "kind": "oracle",
                             "sample": f"{per_step} batch rows of the {cfg.name} workload per step, "
                                       f"one batch row per task on {cores} worker processes"},
            "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main(argv=None):
    args = parse_args(argv)
    dist = Dist()
    if args.impl == "reference":
        if dist.rank != 0:
            return 0
        print(json.dumps(run_reference(args, dist)), flush=True)
        return 0
    res = run_ours(args, dist)
    if dist.rank == 0:
        print(json.dumps(res), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
