"""Test kit: one layer's verify round built twice from the same seeded inputs
-- on the GPU through the C ABI, and on the CPU through the fp64 oracle."""
from __future__ import annotations

import os

import numpy as np
import torch

import oracle
import speculative_tree_verify_bit_gb300 as stv
import workloads

REL_L2_TOL = 1e-3   # per head: (sequence, Q head) block of T rows, relative L2
MAX_ABS_TOL = 4e-3  # per head, max absolute error
CPU_THREADS = os.cpu_count() or 4


class Round:
    """Inputs of one layer's round: contexts, trees, fp16 K/V/Q, page tables."""

    def __init__(self, ctx, t_nodes, seed, hq=24, hkv=4, tree="random", p_accept=0.7, max_depth=8,
                 device="cuda", extra_pages=1, parents=None, group=32, kind=None):
        self.ctx = list(ctx)
        self.n_seqs = len(self.ctx)
        self.T, self.hq, self.hkv = t_nodes, hq, hkv
        self.device = device
        rng = np.random.default_rng(seed + 99)
        need = [workloads.pages_needed(c, t_nodes) for c in self.ctx]
        self.pool_pages = int(sum(need)) + extra_pages
        perm = np.random.default_rng(seed).permutation(self.pool_pages).astype(np.int32)
        self.tables, at = [], 0
        for n in need:
            self.tables.append(perm[at:at + n].copy())
            at += n
        par, dr, am = [], [], []
        for s in range(self.n_seqs):
            if parents is not None:
                p = np.asarray(parents[s], np.int32)
            elif tree == "chain":
                p = workloads.chain_tree(t_nodes)
            else:
                p = workloads.random_tree(rng, t_nodes, max_depth)
            if parents is not None and not oracle.check_tree(p):  # deliberately invalid tree
                d = rng.integers(0, workloads.VOCAB, t_nodes).astype(np.int32)
                a = rng.integers(0, workloads.VOCAB, t_nodes).astype(np.int32)
            else:
                d, a = workloads.draft_and_argmax(rng, p, p_accept)
            par.append(p); dr.append(d); am.append(a)
        self.parent = np.stack(par)
        self.draft = np.stack(dr)
        self.argmax = np.stack(am)
        # rows of every sequence: context rows then tree rows, positions 0..ctx+T-1
        ks, vs = [], []
        for s, c in enumerate(self.ctx):
            k, v = workloads.kv_rows(seed + 7919 * s, c + t_nodes, hkv, device=device)
            ks.append(k); vs.append(v)
        self.k = torch.cat(ks).contiguous()
        self.v = torch.cat(vs).contiguous()
        self.row_seq = np.concatenate([np.full(c + t_nodes, s, np.int32) for s, c in enumerate(self.ctx)])
        self.row_pos = np.concatenate([np.arange(c + t_nodes, dtype=np.int32) for c in self.ctx])
        self.q = workloads.q_rows(seed, self.n_seqs, t_nodes, hq, device=device).contiguous()
        self.group = group  # 32: the 3-bit cache; 256: the int4 per-token-head cache
        self.kind = kind    # "k4v2": the K 4 / V 2-bit cache (group 32)
        self.shape = stv.make_shape(hq, hkv, group, stv.STV_KV_K4V2 if kind == "k4v2" else stv.STV_KV_BY_GROUP)

    # ---------------- GPU side ----------------
    def gpu_cache(self):
        layer = stv.LayerCache.empty(self.pool_pages, self.hkv, device=self.device, group=self.group)
        self.seqs = [stv.Seq(torch.as_tensor(t, device=self.device), c) for t, c in zip(self.tables, self.ctx)]
        status = torch.zeros(1, dtype=torch.int32, device=self.device)
        stv.stv_kv_append_pack(self.shape, layer, self.seqs, self.k, self.v,
                               torch.as_tensor(self.row_seq, device=self.device),
                               torch.as_tensor(self.row_pos, device=self.device), dev_status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        self.layer = layer
        return layer

    def gpu_verify(self, path, layer=None):
        layer = layer or self.layer
        ws_bytes = stv.stv_verify_workspace_bytes(self.shape, self.seqs, self.T)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=self.device)
        o = torch.empty((self.n_seqs, self.T, self.hq, 256), dtype=torch.float16, device=self.device)
        status = torch.zeros(1, dtype=torch.int32, device=self.device)
        parent = torch.as_tensor(self.parent, device=self.device)
        stv.stv_verify_attn(self.shape, layer, self.seqs, self.q, parent, self.T, path, ws, dev_status=status)
        stv.stv_split_combine(self.shape, self.seqs, self.T, ws, o)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        return o

    # ---------------- oracle side ----------------
    def oracle_cache(self):
        cache = oracle.Cache(self.hkv, self.pool_pages, bits=4 if self.group == 256 else 3, kind=self.kind)
        oracle.kv_append(cache, self.tables, self.k.cpu().numpy(), self.v.cpu().numpy(), self.row_seq, self.row_pos)
        self.ocache = cache
        return cache

    def oracle_attention(self, path, rows=None):
        return oracle.attention(self.ocache, self.tables, self.ctx, self.q.cpu().numpy(), self.parent, self.hq, path,
                                rows=rows, n_threads=CPU_THREADS)


def head_errors(got: np.ndarray, want: np.ndarray):
    """Errors per head: arrays [n_seqs][T][hq][256] (or [n_heads][T][256]
    blocks); each (sequence, Q head) block of T rows is one head.  Returns
    relative L2 error and max abs error per head."""
    g = np.asarray(got, np.float64)
    w = np.asarray(want, np.float64)
    if g.ndim == 4:  # [n_seqs][T][hq][256] -> [n_seqs*hq][T*256]
        g = g.transpose(0, 2, 1, 3)
        w = w.transpose(0, 2, 1, 3)
    g = g.reshape(-1, g.shape[-2] * g.shape[-1])
    w = w.reshape(-1, w.shape[-2] * w.shape[-1])
    rel = np.linalg.norm(g - w, axis=1) / np.maximum(np.linalg.norm(w, axis=1), 1e-30)
    mab = np.abs(g - w).max(axis=1)
    return rel, mab


# Worst errors seen by assert_attention_close in this session, per check:
# (what, worst head rel-L2, worst head max-abs, worst row rel-L2, worst row
# max-abs).  conftest prints them at the end of the run.
ERROR_LOG: list = []


def row_errors(got: np.ndarray, want: np.ndarray):
    """Errors per single row (one node of one Q head, 256 values): relative
    L2 and max abs."""
    g = np.asarray(got, np.float64).reshape(-1, 256)
    w = np.asarray(want, np.float64).reshape(-1, 256)
    rel = np.linalg.norm(g - w, axis=1) / np.maximum(np.linalg.norm(w, axis=1), 1e-30)
    return rel, np.abs(g - w).max(axis=1)


def assert_attention_close(got, want, what=""):
    """Tolerance per head: relative L2 <= 1e-3 and max abs <= 4e-3.  The
    per-row maxima are computed too and logged (not asserted: a single row
    carries one node's fp16 rounding of P and of the output without the
    averaging over a head's T rows)."""
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    rel, mab = head_errors(got, want)
    rrel, rmab = row_errors(got, want)
    ERROR_LOG.append((what, float(rel.max()), float(mab.max()), float(rrel.max()), float(rmab.max())))
    assert rel.max() <= REL_L2_TOL, f"{what}: max rel-L2 {rel.max():.3e} (head {rel.argmax()}); worst row {rrel.max():.3e}"
    assert mab.max() <= MAX_ABS_TOL, f"{what}: max abs {mab.max():.3e} (head {mab.argmax()}); worst row {rmab.max():.3e}"
    return rel.max(), mab.max()


def head_rows(seqs, heads, t):
    """All T nodes of the given (sequence, Q head) pairs, as oracle rows."""
    return [(s, n, h) for s in seqs for h in heads for n in range(t)]


def gather_heads(got, seqs, heads, t):
    """[len(seqs)*len(heads)][T][256] blocks of a [n_seqs][T][hq][256] output."""
    return np.stack([got[s, :, h] for s in seqs for h in heads])
