"""Seeded synthetic inputs for the tree-verify round (shared by the CUDA tests,
the oracle tests, the smoke check and the benchmark).

This module holds no arithmetic of the method itself: only random draws with
the shapes and distributions of the workloads.  Both sides (the CUDA library
and the fp64 oracle) receive exactly the same tensors from here.

Workloads (sizes from the model the pages describe -- Qwen3.8-27B: 16
full-attention layers, vocabulary 248,320, 262,144-token native context, an
8-row draft tree / 16-row verify block; head shapes 24 Q heads, 4 KV heads,
head_dim 256):

- ``tiny``: 1 layer, context 1,024, a 16-node random tree of depth <= 8.
- ``chain``: 1 layer, context 8,192, an 8-node chain (root + 7 drafts).
- ``tree32k``: 16 layers, context 32,768, 16-node tree, pages permuted.
- ``long262k``: 16 layers, context 262,144, 16-node tree; acceptance
  probability swept over {0, 0.5, 1}.
- ``ragged``: 8 requests with contexts 1K..128K in one shared page pool,
  16 layers, per-request trees.

Distributions: Q, K, V are fp16 draws of N(0, 1); K is multiplied by 8 on
4 seeded outlier channels per (layer, KV head), the same channels for every
token.  Tree: parent[i] uniform over the earlier nodes whose depth is below
the depth limit.  Target argmax ids are uniform over the vocabulary; node
c >= 1 drafts argmax[parent[c]] with probability p, else a uniform id that
differs from it.  Page tables are a seeded random permutation of the pool.
Seeds: workload index k gives seed 1000 + k; layer l adds 17 * l.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

HQ, HKV, HEAD_DIM = 24, 4, 256
PAGE_TOKENS = 256
VOCAB = 248_320
OUTLIER_CHANNELS = 4
OUTLIER_GAIN = 8.0


@dataclass(frozen=True)
class Workload:
    name: str
    index: int
    ctx: tuple
    t_nodes: int
    layers: int
    tree: str = "random"  # "random" or "chain"
    max_depth: int = 8
    p_accept: tuple = (0.7,)
    hq: int = HQ
    hkv: int = HKV

    @property
    def seed(self) -> int:
        return 1000 + self.index

    @property
    def n_seqs(self) -> int:
        return len(self.ctx)


WORKLOADS = {
    "tiny": Workload("tiny", 0, (1024,), 16, 1),
    "chain": Workload("chain", 1, (8192,), 8, 1, tree="chain"),
    "tree32k": Workload("tree32k", 2, (32768,), 16, 16),
    "long262k": Workload("long262k", 3, (262144,), 16, 16, p_accept=(0.0, 0.5, 1.0)),
    "ragged": Workload("ragged", 4, tuple(1024 << i for i in range(8)), 16, 16),
}


def layer_seed(w: Workload, layer: int) -> int:
    return w.seed + 17 * layer


# --------------------------------------------------------------------------
# Trees and token ids (small, numpy)
# --------------------------------------------------------------------------

def random_tree(rng: np.random.Generator, t: int, max_depth: int) -> np.ndarray:
    """parent[0] = -1; parent[i] uniform over {j < i : depth[j] < max_depth}."""
    parent = np.full(t, -1, np.int32)
    depth = np.zeros(t, np.int32)
    for i in range(1, t):
        cand = [j for j in range(i) if depth[j] < max_depth]
        parent[i] = cand[rng.integers(len(cand))]
        depth[i] = depth[parent[i]] + 1
    return parent


def chain_tree(t: int) -> np.ndarray:
    return np.arange(-1, t - 1, dtype=np.int32)


def tree_for(w: Workload, rng: np.random.Generator) -> np.ndarray:
    if w.tree == "chain":
        return chain_tree(w.t_nodes)
    return random_tree(rng, w.t_nodes, w.max_depth)


def draft_and_argmax(rng: np.random.Generator, parent: np.ndarray, p: float, vocab: int = VOCAB):
    """Target argmax ids and draft ids for one tree.

    argmax[i] ~ U[0, vocab).  draft[0] (the root, already emitted) ~ U.
    For c >= 1: draft[c] = argmax[parent[c]] with probability p, else a
    uniform id different from it.
    """
    t = len(parent)
    argmax = rng.integers(0, vocab, size=t, dtype=np.int64).astype(np.int32)
    draft = np.zeros(t, np.int32)
    draft[0] = rng.integers(0, vocab)
    for c in range(1, t):
        want = int(argmax[parent[c]])
        if rng.random() < p:
            draft[c] = want
        else:
            x = int(rng.integers(0, vocab - 1))
            draft[c] = x if x < want else x + 1
    return draft, argmax


def all_parent_arrays(t: int):
    """Every parent array with parent[0] = -1 and 0 <= parent[i] < i ((t-1)! of them)."""
    def rec(prefix):
        i = len(prefix)
        if i == t:
            yield np.asarray(prefix, np.int32)
            return
        for p in range(i):
            yield from rec(prefix + [p])
    yield from rec([-1])


# --------------------------------------------------------------------------
# Page tables
# --------------------------------------------------------------------------

def pages_needed(ctx: int, t_nodes: int) -> int:
    return -(-(ctx + t_nodes) // PAGE_TOKENS)


def page_tables_for(w: Workload, seed: int | None = None):
    """(pool_pages, [page table per sequence]) from one seeded permutation."""
    need = [pages_needed(c, w.t_nodes) for c in w.ctx]
    pool_pages = int(sum(need))
    rng = np.random.default_rng(w.seed if seed is None else seed)
    perm = rng.permutation(pool_pages).astype(np.int32)
    tables, at = [], 0
    for n in need:
        tables.append(perm[at:at + n].copy())
        at += n
    return pool_pages, tables


# --------------------------------------------------------------------------
# fp16 activations (torch, on any device)
# --------------------------------------------------------------------------

def outlier_channels(seed: int, hkv: int = HKV) -> np.ndarray:
    rng = np.random.default_rng(seed + 424242)
    return np.stack([rng.choice(HEAD_DIM, OUTLIER_CHANNELS, replace=False) for _ in range(hkv)])


def _gen(torch, device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def kv_rows(seed: int, n_rows: int, hkv: int = HKV, device="cpu", stream_id: int = 0):
    """K, V fp16 [n_rows][hkv][256]: N(0,1), K x8 on the outlier channels."""
    import torch

    g = _gen(torch, device, seed * 1_000_003 + 2 * stream_id + 1)
    k = torch.randn((n_rows, hkv, HEAD_DIM), generator=g, device=device, dtype=torch.float32)
    v = torch.randn((n_rows, hkv, HEAD_DIM), generator=g, device=device, dtype=torch.float32)
    out = outlier_channels(seed, hkv)
    gain = torch.ones((hkv, HEAD_DIM), device=device, dtype=torch.float32)
    for h in range(hkv):
        gain[h, torch.as_tensor(out[h], device=device)] = OUTLIER_GAIN
    k = k * gain
    return k.to(torch.float16), v.to(torch.float16)


def q_rows(seed: int, n_seqs: int, t_nodes: int, hq: int = HQ, device="cpu"):
    """Q fp16 [n_seqs][t_nodes][hq][256] ~ N(0, 1)."""
    import torch

    g = _gen(torch, device, seed * 1_000_003 + 777)
    return torch.randn((n_seqs, t_nodes, hq, HEAD_DIM), generator=g, device=device,
                       dtype=torch.float32).to(torch.float16)


@dataclass
class RoundInputs:
    """Everything one layer's verify round consumes (besides the cache)."""
    parent: np.ndarray       # [n_seqs][T] int32
    draft: np.ndarray        # [n_seqs][T] int32
    argmax: np.ndarray       # [n_seqs][T] int32
    extra: dict = field(default_factory=dict)


def round_trees(w: Workload, p: float | None = None) -> RoundInputs:
    rng = np.random.default_rng(w.seed + 99)
    p = w.p_accept[0] if p is None else p
    par, dr, am = [], [], []
    for _ in range(w.n_seqs):
        parent = tree_for(w, rng)
        d, a = draft_and_argmax(rng, parent, p)
        par.append(parent)
        dr.append(d)
        am.append(a)
    return RoundInputs(np.stack(par), np.stack(dr), np.stack(am))


def token_history(seed: int, n: int, p_copy: float = 0.7, tail: int = 64, alphabet: int = VOCAB) -> np.ndarray:
    """Seeded synthetic token history of n ids for lookup drafting: uniform
    ids over `alphabet`; with probability p_copy its last `tail` tokens repeat
    an earlier span, as when an answer quotes its prompt ("reproduce every
    command" work).  Random draws only."""
    rng = np.random.default_rng(seed)
    h = rng.integers(0, alphabet, n, dtype=np.int64).astype(np.int32)
    if n > 2 * tail and rng.random() < p_copy:
        a = int(rng.integers(0, n - 2 * tail))
        h[n - tail:] = h[a:a + tail]
    return h


def lookup_histories(w: Workload, p_copy: float = 0.7):
    """One history per request of the workload, as long as its context."""
    return [token_history(1000 + 31 * s + w.ctx[s] % 997, c, p_copy) for s, c in enumerate(w.ctx)]
