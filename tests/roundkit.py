"""Test kit: one layer's verify round built twice from the same seeded inputs
-- on the GPU through the C ABI, and on the CPU through the fp64 oracle."""
from __future__ import annotations

import os

import numpy as np
import torch

import oracle
import speculative_tree_verify_bit_gb300 as stv
import workloads

REL_L2_TOL = 1e-3   # per (node, Q head) row, relative L2 error
MAX_ABS_TOL = 4e-3  # per (node, Q head) row, max absolute error
CPU_THREADS = os.cpu_count() or 4


class Round:
    """Inputs of one layer's round: contexts, trees, fp16 K/V/Q, page tables."""

    def __init__(self, ctx, t_nodes, seed, hq=24, hkv=4, tree="random", p_accept=0.7, max_depth=8,
                 device="cuda", extra_pages=1, parents=None):
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
        self.shape = stv.make_shape(hq, hkv)

    # ---------------- GPU side ----------------
    def gpu_cache(self):
        layer = stv.LayerCache.empty(self.pool_pages, self.hkv, device=self.device)
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
        cache = oracle.Cache(self.hkv, self.pool_pages)
        oracle.kv_append(cache, self.tables, self.k.cpu().numpy(), self.v.cpu().numpy(), self.row_seq, self.row_pos)
        self.ocache = cache
        return cache

    def oracle_attention(self, path, rows=None):
        return oracle.attention(self.ocache, self.tables, self.ctx, self.q.cpu().numpy(), self.parent, self.hq, path,
                                rows=rows, n_threads=CPU_THREADS)


def row_errors(got: np.ndarray, want: np.ndarray):
    """Per-row relative L2 and max-abs errors (rows = leading axes flattened)."""
    g = got.reshape(-1, 256).astype(np.float64)
    w = want.reshape(-1, 256)
    rel = np.linalg.norm(g - w, axis=1) / np.maximum(np.linalg.norm(w, axis=1), 1e-30)
    mab = np.abs(g - w).max(axis=1)
    return rel, mab


def assert_attention_close(got, want, what=""):
    rel, mab = row_errors(got, want)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    assert rel.max() <= REL_L2_TOL, f"{what}: max rel-L2 {rel.max():.3e} (row {rel.argmax()})"
    assert mab.max() <= MAX_ABS_TOL, f"{what}: max abs {mab.max():.3e} (row {mab.argmax()})"
    return rel.max(), mab.max()
