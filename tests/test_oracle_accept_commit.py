"""Pins for the oracle's greedy tree acceptance and KV commit.

Acceptance ("elpis" README, "Why fast": commit the longest matching path + 1;
"elpis-lossless" README, "How": 7 nodes ranked best first; "Lossless": token
ids compared exactly) is checked against brute-force enumeration of every
root path, on all 5,040 eight-row parent arrays (the shape sweep the
"elpis-lossless" "Proofs and tests" table runs), with all-rejected,
all-accepted and random drafts.  Commit is checked against re-packing the
committed rows' fp16 K/V at their new positions."""
import numpy as np
import pytest

import oracle
import workloads


def brute_accept(parent, draft, argmax):
    t = len(parent)
    paths = []
    for end in range(t):
        p, n = [], end
        while n >= 0:
            p.append(n)
            n = parent[n]
        p.reverse()
        if all(draft[c] == argmax[a] for a, c in zip(p, p[1:])):
            paths.append(p)
    best = sorted(paths, key=lambda p: (-len(p), p))[0]
    out = [int(draft[c]) for c in best[1:]] + [int(argmax[best[-1]])]
    return len(best), best, out


def depth_of(parent):
    d = [0] * len(parent)
    for i in range(1, len(parent)):
        d[i] = d[parent[i]] + 1
    return d


def test_acceptance_all_5040_shapes():
    rng = np.random.default_rng(123)
    n_shapes = 0
    for parent in workloads.all_parent_arrays(8):
        n_shapes += 1
        for p in (0.0, 1.0, 0.6):
            # small vocabulary in the random case so equal sibling drafts occur
            vocab = 5 if p == 0.6 else workloads.VOCAB
            draft, argmax = workloads.draft_and_argmax(rng, parent, p, vocab=vocab)
            n, path, out = oracle.tree_accept(parent, draft, argmax)
            bn, bpath, bout = brute_accept(parent, draft, argmax)
            assert n == bn and path.tolist() == bpath and out.tolist() == bout
            if p == 0.0:
                assert n == 1 and out.tolist() == [int(argmax[0])]
            if p == 1.0:
                assert n == max(depth_of(parent)) + 1
    assert n_shapes == 5040


def test_acceptance_tie_break_prefers_lower_indices():
    # two matching children of the root (equal drafts): [0,1,3] vs [0,2,4]
    parent = np.array([-1, 0, 0, 1, 2], np.int32)
    argmax = np.array([7, 8, 8, 1, 1], np.int32)
    draft = np.array([0, 7, 7, 8, 8], np.int32)
    n, path, out = oracle.tree_accept(parent, draft, argmax)
    assert n == 3 and path.tolist() == [0, 1, 3] and out.tolist() == [7, 8, 1]


@pytest.mark.parametrize("bad", [[0, 0, 1], [-1, 1, 0], [-1, 0, 3], [-1, -1, 0]])
def test_invalid_trees_rejected(bad):
    assert not oracle.check_tree(bad)
    with pytest.raises(oracle.OracleError):
        oracle.tree_accept(bad, [0] * len(bad), [0] * len(bad))


def packed_token(cache, tables, seq, tok, h):
    """One token's packed row, read straight from the page bytes using the
    layout statement (K codes/scales by token, V codes channel-major)."""
    page = tables[seq][tok // 256]
    slot = tok % 256
    base = page * cache.page_bytes + h * oracle.HEAD_BYTES
    pool = cache.pool
    kc = pool[base + slot * 96: base + slot * 96 + 96].copy()
    ks = pool[base + 24576 + slot * 16: base + 24576 + slot * 16 + 16].copy()
    vs, vc = [], []
    tile, within = slot // 64, slot % 64
    for g in range(8):
        o = base + 53248 + tile * 1024 + g * 128 + within * 2
        vs.append(pool[o:o + 2].copy())
    for ch in range(256):
        o = base + 28672 + tile * 6144 + ch * 24 + (within // 32) * 12
        w = pool[o:o + 12].view(np.uint32)
        vc.append(oracle.block_code(w, within % 32))
    return kc, ks, np.concatenate(vs), np.array(vc, np.uint8)


def test_commit_equals_repacking_committed_rows():
    rng = np.random.default_rng(55)
    hkv, t = 2, 12
    ctxs = [250, 13]  # the first sequence's tree straddles a page boundary
    need = [-(-(c + t) // 256) for c in ctxs]
    pool_pages = sum(need) + 2
    perm = rng.permutation(pool_pages).astype(np.int32)
    tables = [perm[:need[0]], perm[need[0]:need[0] + need[1]]]
    k = [rng.standard_normal((c + t, hkv, 256)).astype(np.float16) for c in ctxs]
    v = [rng.standard_normal((c + t, hkv, 256)).astype(np.float16) for c in ctxs]
    cache = oracle.Cache(hkv, pool_pages)
    for s, c in enumerate(ctxs):
        oracle.kv_append(cache, tables, k[s], v[s], [s] * (c + t), list(range(c + t)))
    parents, ncs, paths = [], [], []
    for s in range(2):
        parent = workloads.random_tree(rng, t, 8)
        draft, argmax = workloads.draft_and_argmax(rng, parent, 1.0)
        n, path, _ = oracle.tree_accept(parent, draft, argmax)
        assert n >= 2
        parents.append(parent)
        ncs.append(n)
        full = np.zeros(t, np.int32)
        full[:n] = path
        paths.append(full)
    oracle.kv_commit(cache, tables, ctxs, ncs, np.stack(paths), t)

    ref = oracle.Cache(hkv, pool_pages)
    for s, c in enumerate(ctxs):
        oracle.kv_append(ref, tables, k[s][:c], v[s][:c], [s] * c, list(range(c)))
        rows = [c + int(paths[s][i]) for i in range(ncs[s])]
        oracle.kv_append(ref, tables, k[s][rows], v[s][rows], [s] * ncs[s], [c + i for i in range(ncs[s])])
    for s, c in enumerate(ctxs):
        for tok in list(range(max(0, c - 3), c + ncs[s])):
            for h in range(hkv):
                a = packed_token(cache, tables, s, tok, h)
                b = packed_token(ref, tables, s, tok, h)
                for x, y in zip(a, b):
                    assert np.array_equal(x, y), (s, tok, h)
