"""a6 tree_accept and a7 kv_commit on the GPU: bit-exact against the oracle.

Sources: "elpis" README, "Why fast" (commit the longest matching path + 1);
"elpis-lossless" README, "How" (best-first nodes), "Lossless" (exact id
comparison), "Proofs and tests" (all 5,040 tree shapes)."""
import numpy as np
import pytest
import torch

import oracle
import speculative_tree_verify_bit_gb300 as stv
import workloads
from roundkit import Round

pytestmark = pytest.mark.gpu


def run_accept(gpu, parent, draft, argmax):
    n, t = parent.shape
    P = lambda a: torch.as_tensor(np.ascontiguousarray(a, np.int32), device=gpu)
    nc = torch.full((n,), -7, dtype=torch.int32, device=gpu)
    path = torch.full((n, t), -7, dtype=torch.int32, device=gpu)
    out = torch.full((n, t), -7, dtype=torch.int32, device=gpu)
    status = torch.zeros(1, dtype=torch.int32, device=gpu)
    stv.stv_tree_accept(P(parent), P(draft), P(argmax), nc, path, out, dev_status=status)
    torch.cuda.synchronize()
    return nc.cpu().numpy(), path.cpu().numpy(), out.cpu().numpy(), int(status.item())


def test_accept_all_5040_shapes_three_draft_modes(gpu):
    rng = np.random.default_rng(2024)
    parents, drafts, argmaxes = [], [], []
    for parent in workloads.all_parent_arrays(8):
        for p, vocab in ((0.0, workloads.VOCAB), (1.0, workloads.VOCAB), (0.6, 5)):
            d, a = workloads.draft_and_argmax(rng, parent, p, vocab=vocab)
            parents.append(parent); drafts.append(d); argmaxes.append(a)
    parents, drafts, argmaxes = np.stack(parents), np.stack(drafts), np.stack(argmaxes)
    nc, path, out, st = run_accept(gpu, parents, drafts, argmaxes)
    assert st == 0
    for i in range(len(parents)):
        n, pth, ids = oracle.tree_accept(parents[i], drafts[i], argmaxes[i])
        assert nc[i] == n
        assert path[i, :n].tolist() == pth.tolist() and (path[i, n:] == -1).all()
        assert out[i, :n].tolist() == ids.tolist() and (out[i, n:] == -1).all()


@pytest.mark.parametrize("t", [1, 16, 32])
def test_accept_random_trees(gpu, t):
    rng = np.random.default_rng(t)
    parents, drafts, argmaxes = [], [], []
    for _ in range(500):
        parent = workloads.random_tree(rng, t, 8 if t > 1 else 1)
        d, a = workloads.draft_and_argmax(rng, parent, rng.random(), vocab=int(rng.choice([3, 50, workloads.VOCAB])))
        parents.append(parent); drafts.append(d); argmaxes.append(a)
    parents, drafts, argmaxes = np.stack(parents), np.stack(drafts), np.stack(argmaxes)
    nc, path, out, st = run_accept(gpu, parents, drafts, argmaxes)
    for i in range(len(parents)):
        n, pth, ids = oracle.tree_accept(parents[i], drafts[i], argmaxes[i])
        assert nc[i] == n and path[i, :n].tolist() == pth.tolist() and out[i, :n].tolist() == ids.tolist()


def test_accept_bad_tree_flagged(gpu):
    parent = np.array([[-1, 0, 1], [-1, 2, 0]], np.int32)
    nc, path, out, st = run_accept(gpu, parent, np.zeros_like(parent), np.zeros_like(parent))
    assert st & stv.STV_DEV_BAD_TREE
    assert nc[1] == 0 and (path[1] == -1).all()
    assert nc[0] == 3


@pytest.mark.parametrize("ctx,p", [([1024], 0.7), ([250, 13, 4000], 1.0), ([100], 0.0), ([255, 511], 0.8)])
def test_commit_bytes_bit_exact(gpu, ctx, p):
    """Three layers, several sequences (one whose tree straddles a page):
    accept on the GPU, commit on the GPU; the pools equal the oracle's after
    the oracle's own accept and commit, and ctx_dev advances by n_commit."""
    t = 16
    layers, ocaches = [], []
    base = None
    for l in range(3):
        r = Round(ctx, t, seed=300 + 11 * l, p_accept=p)
        if base is None:
            base = r
        else:  # same trees and tables for every layer
            r.parent, r.draft, r.argmax, r.tables = base.parent, base.draft, base.argmax, base.tables
        layers.append(r.gpu_cache())
        ocaches.append(r.oracle_cache())
    r = base
    nc, path, out, st = run_accept(gpu, r.parent, r.draft, r.argmax)
    assert st == 0
    ctx_dev = torch.as_tensor(np.array(ctx, np.int32), device=gpu)
    status = torch.zeros(1, dtype=torch.int32, device=gpu)
    stv.stv_kv_commit(r.shape, layers, r.seqs, t, torch.as_tensor(nc, device=gpu), torch.as_tensor(path, device=gpu),
                      ctx_dev=ctx_dev, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert ctx_dev.cpu().numpy().tolist() == [c + int(n) for c, n in zip(ctx, nc)]
    for s in range(len(ctx)):
        n, pth, _ = oracle.tree_accept(r.parent[s], r.draft[s], r.argmax[s])
        assert n == nc[s]
    full = np.where(path >= 0, path, 0).astype(np.int32)
    for l in range(3):
        oracle.kv_commit(ocaches[l], r.tables, ctx, nc, full, t)
        assert np.array_equal(layers[l].pool.cpu().numpy(), ocaches[l].pool), l


def test_commit_rejects_bad_counts_without_writing(gpu):
    r = Round([300], 8, seed=9)
    layer = r.gpu_cache()
    before = layer.pool.clone()
    status = torch.zeros(1, dtype=torch.int32, device=gpu)
    bad_path = torch.tensor([[0, 3, 2, -1, -1, -1, -1, -1]], dtype=torch.int32, device=gpu)
    for nc in ([0], [9], [3]):
        stv.stv_kv_commit(r.shape, [layer], r.seqs, 8, torch.tensor(nc, dtype=torch.int32, device=gpu), bad_path,
                          dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & stv.STV_DEV_BAD_COMMIT
    assert torch.equal(before, layer.pool)


def test_commit_all_or_nothing_on_bad_page(gpu):
    """A destination page outside one layer's pool: no layer is written and
    ctx_dev stays put (STV_DEV_BAD_PAGE); with pages inside every pool the
    same call commits every layer and advances ctx_dev."""
    shape = stv.make_shape(24, 4)
    g = torch.Generator(device="cpu").manual_seed(11)
    big = stv.LayerCache(torch.randint(0, 256, (6 * 4 * stv.HEAD_BLOCK_BYTES,), generator=g, dtype=torch.uint8).to(gpu), 4)
    small = stv.LayerCache(torch.randint(0, 256, (3 * 4 * stv.HEAD_BLOCK_BYTES,), generator=g, dtype=torch.uint8).to(gpu), 4)
    n_commit = torch.tensor([3], dtype=torch.int32, device=gpu)
    path = torch.tensor([[0, 2, 5, -1, -1, -1, -1, -1]], dtype=torch.int32, device=gpu)
    for table, bad in (([0, 5], True), ([0, 2], False)):
        seqs = [stv.Seq(torch.tensor(table, dtype=torch.int32, device=gpu), 300)]  # rows 300.. sit in logical page 1
        before = [big.pool.clone(), small.pool.clone()]
        ctx_dev = torch.tensor([300], dtype=torch.int32, device=gpu)
        status = torch.zeros(1, dtype=torch.int32, device=gpu)
        stv.stv_kv_commit(shape, [big, small], seqs, 8, n_commit, path, ctx_dev=ctx_dev, dev_status=status)
        torch.cuda.synchronize()
        if bad:
            assert int(status.item()) & stv.STV_DEV_BAD_PAGE
            assert torch.equal(before[0], big.pool) and torch.equal(before[1], small.pool)
            assert int(ctx_dev.item()) == 300
        else:
            assert int(status.item()) == 0
            assert not torch.equal(before[0], big.pool) and not torch.equal(before[1], small.pool)
            assert int(ctx_dev.item()) == 303
