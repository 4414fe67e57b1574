"""Seeded synthetic inputs for the verify step (shared by tests and bench).

This module only draws random numbers and lays them out; it computes none of
the verify arithmetic (no softmax, filtering, argmax, acceptance or sampling).
Draft token ids are NOT made here: a test draws them with the oracle's own
sampler and the benchmark with the library's draft sampler, both from the
uniforms ``u_draft`` generated here.

Workloads restate the shapes of the pages' settings:
  tiny      B=1,   γ=3, V=1000   fp32, T=0.8, top_p=0.9  (page defaults of
            ``generate(prompt, temperature=0.8, top_p=0.9)``)
  smollm2   B=64,  γ=5, V=49152  bf16, T=0.8, top_p=0.9, 5 spiked ids per row
            (SmolLM2-360M vocabulary of the Eaglet1 page)
  llama3    B=128, γ=6, V=128256 bf16, greedy (T=0) or T=1, top_p=1
            (Llama-3 vocabulary; ``--k 6 --temp 0`` benchmark)
  qwen3     B=256, γ=7, V=151936 fp32 target, V_d=32000 fp32 EAGLE3 draft
            vocabulary scattered through d2t, T=1, top_p=0.95
  tree      B=64 trees of 32 nodes, depth <= 5, <= 8 children, V=128256 bf16
            (total_token 32 / depth 5 / top_k 8 of the Eaglet1 page)

N(0, s) below means mean 0 and standard deviation s.  Logits are drawn in
fp32 and, for bf16 workloads, rounded to bf16 (round to nearest even); the
rounded values are the ground truth for both sides.
"""
from __future__ import annotations

import dataclasses

import numpy as np

BASE_SEED = 20260000


@dataclasses.dataclass(frozen=True)
class ChainConfig:
    name: str
    batch: int
    gamma: int
    vocab: int
    dtype: str                 # "f32" or "bf16"
    temperature: float
    top_p: float
    target_sigma: float
    draft_sigma: float
    draft_vocab: int = 0       # > 0: EAGLE3 small draft vocabulary through d2t
    spikes: int = 0            # spiked ids per target row
    spike_value: float = 0.0
    number: int = 0            # workload number (seed offset)

    @property
    def rows_metric(self) -> int:
        """Verify rows per step: B * (2γ + 1)."""
        return self.batch * (2 * self.gamma + 1)

    def esize(self) -> int:
        return 2 if self.dtype == "bf16" else 4

    def algorithmic_bytes(self) -> int:
        """Logit bytes read once: B*[(γ+1)*V*e + γ*V_d*e]; greedy reads target rows only."""
        e = self.esize()
        t = self.batch * (self.gamma + 1) * self.vocab * e
        if self.temperature == 0.0:
            return t
        vd = self.draft_vocab or self.vocab
        return t + self.batch * self.gamma * vd * e


@dataclasses.dataclass(frozen=True)
class TreeConfig:
    name: str
    batch: int
    nodes: int
    vocab: int
    dtype: str
    max_depth: int
    max_children: int
    sigma: float
    plant_prob: float
    plant_spike: float
    number: int = 0

    @property
    def rows_metric(self) -> int:
        return self.batch * self.nodes

    def esize(self) -> int:
        return 2 if self.dtype == "bf16" else 4

    def algorithmic_bytes(self) -> int:
        return self.batch * self.nodes * self.vocab * self.esize()


@dataclasses.dataclass(frozen=True)
class TreeSampleConfig(TreeConfig):
    """A tree workload verified by speculative sampling at temperature T and
    top_p: target and draft logits at every node."""
    temperature: float = 1.0
    top_p: float = 1.0

    def algorithmic_bytes(self) -> int:
        return 2 * super().algorithmic_bytes()  # target and draft rows


TINY = ChainConfig("tiny", 1, 3, 1000, "f32", 0.8, 0.9, 2.0, 0.5, number=1)
SMOLLM2 = ChainConfig("smollm2", 64, 5, 49152, "bf16", 0.8, 0.9, 3.0, 0.7,
                      spikes=5, spike_value=8.0, number=2)
LLAMA3_GREEDY = ChainConfig("llama3-greedy", 128, 6, 128256, "bf16", 0.0, 1.0, 2.0, 0.5, number=3)
LLAMA3_SAMPLE = ChainConfig("llama3-sample", 128, 6, 128256, "bf16", 1.0, 1.0, 2.0, 0.5, number=3)
QWEN3_D2T = ChainConfig("qwen3-d2t", 256, 7, 151936, "f32", 1.0, 0.95, 2.0, 0.7,
                        draft_vocab=32000, number=4)
TREE = TreeConfig("tree", 64, 32, 128256, "bf16", 5, 8, 2.0, 0.7, 16.0, number=5)
TREE_SAMPLE = TreeSampleConfig("tree-sample", 64, 32, 128256, "bf16", 5, 8, 2.0, 0.7, 16.0, number=5,
                               temperature=1.0, top_p=1.0)

CHAIN_CONFIGS = {c.name: c for c in (TINY, SMOLLM2, LLAMA3_GREEDY, LLAMA3_SAMPLE, QWEN3_D2T)}
ALL_CONFIGS = dict(CHAIN_CONFIGS, tree=TREE)


def rng(seed: int, stream: int) -> np.random.Generator:
    """Independent Philox stream ``stream`` of ``seed``."""
    return np.random.Generator(np.random.Philox(np.random.SeedSequence([seed, stream])))


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest even (finite inputs)."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return b.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> the exact fp32 values they denote."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _finish(x: np.ndarray, dtype: str):
    """Return (values as fp32, storage array: fp32 or bf16 bits)."""
    if dtype == "bf16":
        bits = to_bf16_bits(x)
        return bf16_bits_to_f32(bits), bits
    x = np.ascontiguousarray(x, dtype=np.float32)
    return x, x


def make_d2t(seed: int, vocab: int, draft_vocab: int, shuffled: bool = False) -> np.ndarray:
    """Injective draft->target id map: a random draft_vocab-subset of [0, vocab).

    Sorted ascending by default; ``shuffled`` permutes the draft ids so the map
    is not monotone.
    """
    g = rng(seed, 7)
    d2t = np.sort(g.choice(vocab, size=draft_vocab, replace=False)).astype(np.int32)
    if shuffled:
        d2t = d2t[g.permutation(draft_vocab)]
    return d2t


def make_chain_inputs(cfg: ChainConfig, seed: int | None = None, *, batch: int | None = None,
                      vocab: int | None = None, shuffled_d2t: bool = False) -> dict:
    """Seeded inputs for one chain-verify workload.

    Returns a dict with
      target, draft        fp32 values [B, γ+1, V] and [B, γ, V or V_d]
      target_store, draft_store   what the device receives (fp32 or bf16 bits)
      d2t                  int32 [V_d] or None
      u_accept [B, γ], u_resample [B], u_draft [B, γ]   fp32 in [0, 1)
    ``batch``/``vocab`` override the sizes for small parity cases.
    """
    seed = BASE_SEED + cfg.number if seed is None else seed
    B = cfg.batch if batch is None else batch
    V = cfg.vocab if vocab is None else vocab
    vd = min(cfg.draft_vocab, V) if cfg.draft_vocab else 0
    G = cfg.gamma
    g_t, g_d, g_u = rng(seed, 1), rng(seed, 2), rng(seed, 3)

    target = g_t.normal(0.0, cfg.target_sigma, size=(B, G + 1, V)).astype(np.float32)
    if cfg.spikes:
        for b in range(B):
            for i in range(G + 1):
                ids = g_t.choice(V, size=min(cfg.spikes, V), replace=False)
                target[b, i, ids] += np.float32(cfg.spike_value)
    d2t = None
    if vd:
        d2t = make_d2t(seed, V, vd, shuffled=shuffled_d2t)
        base = target[:, :G, :][:, :, d2t]
    else:
        base = target[:, :G, :]
    draft = (base + g_d.normal(0.0, cfg.draft_sigma, size=base.shape)).astype(np.float32)

    target_v, target_s = _finish(target, cfg.dtype)
    draft_v, draft_s = _finish(draft, cfg.dtype)
    return dict(
        cfg=cfg, seed=seed, batch=B, gamma=G, vocab=V, draft_vocab=vd or V,
        target=target_v, draft=draft_v, target_store=target_s, draft_store=draft_s,
        d2t=d2t,
        u_accept=g_u.random((B, G), dtype=np.float32),
        u_resample=g_u.random(B, dtype=np.float32),
        u_draft=g_u.random((B, G), dtype=np.float32),
    )


def make_tree_inputs(cfg: TreeConfig, seed: int | None = None, *, batch: int | None = None,
                     vocab: int | None = None, nodes: int | None = None) -> dict:
    """Seeded draft trees with target logits at every node.

    Node 0 is the root.  Node n = 1..N-1 picks its parent uniformly among the
    earlier nodes that are shallower than max_depth and have fewer than
    max_children children.  A node's first child is "planted" with
    probability plant_prob: its token t is random and the parent's row gets
    +plant_spike at t, so t is almost surely the parent's argmax (otherwise
    almost every tree would accept nothing).  Other children get distinct
    random tokens different from the planted one.
    """
    seed = BASE_SEED + cfg.number if seed is None else seed
    B = cfg.batch if batch is None else batch
    V = cfg.vocab if vocab is None else vocab
    N = cfg.nodes if nodes is None else nodes
    g_l, g_t = rng(seed, 1), rng(seed, 4)
    logits = g_l.normal(0.0, cfg.sigma, size=(B, N, V)).astype(np.float32)
    parents = np.full((B, N), -1, np.int32)
    tokens = np.zeros((B, N), np.int32)
    for b in range(B):
        depth = [0]
        nchild = [0]
        used = [set() for _ in range(N)]
        planted = [None] * N
        tokens[b, 0] = g_t.integers(V)
        for n in range(1, N):
            cand = [m for m in range(n) if depth[m] < cfg.max_depth and nchild[m] < cfg.max_children]
            par = int(cand[g_t.integers(len(cand))])
            parents[b, n] = par
            if nchild[par] == 0 and g_t.random() < cfg.plant_prob:
                t = int(g_t.integers(V))
                planted[par] = t
                logits[b, par, t] += np.float32(cfg.plant_spike)
            else:
                # Distinct sibling tokens while the vocabulary allows it (a few
                # tries); tiny vocabularies fall back to a repeated token.
                for _ in range(64):
                    t = int(g_t.integers(V))
                    if t not in used[par] and t != planted[par]:
                        break
            used[par].add(t)
            tokens[b, n] = t
            nchild[par] += 1
            depth.append(depth[par] + 1)
            nchild.append(0)
    values, store = _finish(logits, cfg.dtype)
    return dict(cfg=cfg, seed=seed, batch=B, nodes=N, vocab=V, logits=values,
                logits_store=store, parents=parents, tokens=tokens, max_depth=cfg.max_depth)


def make_tree_sample_inputs(cfg: TreeConfig, seed: int | None = None, *, batch: int | None = None,
                            vocab: int | None = None, nodes: int | None = None,
                            draft_noise: float = 1.0) -> dict:
    """The tree workload plus what sampling verify needs.

    draft_logits [B, N, V]: the target logits plus seeded Gaussian noise of
    scale ``draft_noise`` (a draft that shares the target's planted peaks and
    differs from it everywhere else); u_accept [B, N] and u_final [B] fp32
    uniforms in [0, 1).  The children are the tree workload's tokens (the
    planted child first), not draws from the draft.
    """
    tr = make_tree_inputs(cfg, seed, batch=batch, vocab=vocab, nodes=nodes)
    g_d, g_u = rng(tr["seed"], 7), rng(tr["seed"], 8)
    draft = tr["logits"] + g_d.normal(0.0, draft_noise, size=tr["logits"].shape).astype(np.float32)
    dvals, dstore = _finish(draft, cfg.dtype)
    B, N = tr["batch"], tr["nodes"]
    tr.update(draft_logits=dvals, draft_store=dstore,
              u_accept=g_u.random((B, N), dtype=np.float32), u_final=g_u.random(B, dtype=np.float32))
    return tr
