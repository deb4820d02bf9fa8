"""Pins for the oracle's tree-masked attention (exact and int8 definitions).

The oracle quantizes, packs, decodes and runs a two-pass softmax over a
visible-key list.  Here it is checked against (1) a dense fp64 attention with
an explicit node-by-key mask matrix built from a parent walk, on K/V that the
3-bit format represents exactly; (2) closed forms; (3) the invariant that a
chain tree equals sequential one-row decoding ("elpis" README, Bend table:
the tree verify emits the sequential round's tokens)."""
from fractions import Fraction

import numpy as np
import pytest
import scipy.special

import oracle

D = 256


def representable_rows(rng, n_rows, hkv, zero=False):
    """fp16 rows whose 32-channel groups are exactly s*(c-4), s a power of two,
    with one code 0 per group so that max|x| = 4s fixes the scale to s."""
    x = np.zeros((n_rows, hkv, D), np.float64)
    if zero:
        return x.astype(np.float16), x
    for r in range(n_rows):
        for h in range(hkv):
            for g in range(8):
                s = 2.0 ** int(rng.integers(-3, 3))
                codes = rng.integers(0, 8, 32)
                codes[rng.integers(32)] = 0
                x[r, h, 32 * g:32 * g + 32] = s * (codes - 4)
    x16 = x.astype(np.float16)
    assert np.array_equal(x16.astype(np.float64), x)
    return x16, x


def ancestors_by_walk(parent, i):
    out, n = [], i
    while n >= 0:
        out.append(n)
        n = parent[n]
    return set(out)


def build_cache(rng, ctx, parent_list, hkv, k_ctx, v_ctx, k_tree, v_tree):
    """One layer, n_seqs sequences, contiguous pages per sequence."""
    n_seqs = len(ctx)
    t = len(parent_list[0])
    need = [-(-(c + t) // 256) for c in ctx]
    pool_pages = sum(need) + 1
    perm = rng.permutation(pool_pages)
    tables, at = [], 0
    for n in need:
        tables.append(perm[at:at + n].astype(np.int32))
        at += n
    cache = oracle.Cache(hkv, pool_pages)
    for s in range(n_seqs):
        if ctx[s]:
            oracle.kv_append(cache, tables, k_ctx[s], v_ctx[s], [s] * ctx[s], list(range(ctx[s])))
        oracle.kv_append(cache, tables, k_tree[s], v_tree[s], [s] * t, [ctx[s] + i for i in range(t)])
    return cache, tables


def dense_attention(q, kfull, vfull, parent, ctx, hq, hkv, int8=False):
    """Dense fp64 reference: explicit mask matrix, no quantization."""
    t = len(parent)
    G = hq // hkv
    n_keys = ctx + t
    mask = np.zeros((t, n_keys), bool)
    for i in range(t):
        mask[i, :ctx] = True
        for a in ancestors_by_walk(parent, i):
            mask[i, ctx + a] = True
    out = np.zeros((t, hq, D))
    for qh in range(hq):
        h = qh // G
        qm = q[:, qh, :].astype(np.float64)
        if int8:
            rows = []
            for i in range(t):
                qs = [Fraction(float(v)) for v in qm[i]]
                m = max(abs(v) for v in qs)
                qi = np.array([round(Fraction(127) * v / m) if m else 0 for v in qs], np.float64)
                sq = float(np.float32(float(m) / 127.0))
                rows.append(sq * qi)
            qm = np.stack(rows)
        s = qm @ kfull[:, h, :].T / 16.0
        s = np.where(mask, s, -np.inf)
        p = scipy.special.softmax(s, axis=1)
        out[:, qh, :] = p @ vfull[:, h, :]
    return out


@pytest.mark.parametrize("path", ["exact", "int8"])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_attention_matches_dense_bruteforce(path, seed):
    rng = np.random.default_rng(seed)
    hkv, hq, t = 2, 4, 6
    ctxs = [int(rng.integers(0, 40)), int(rng.integers(1, 70))]
    parents = []
    for _ in ctxs:
        p = np.full(t, -1, np.int32)
        for i in range(1, t):
            p[i] = rng.integers(0, i)
        parents.append(p)
    kc, vc, kt, vt, kx, vx = [], [], [], [], [], []
    for c in ctxs:
        k16, k64 = representable_rows(rng, c + t, hkv)
        v16, v64 = representable_rows(rng, c + t, hkv)
        kc.append(k16[:c]); vc.append(v16[:c]); kt.append(k16[c:]); vt.append(v16[c:])
        kx.append(k64); vx.append(v64)
    cache, tables = build_cache(rng, ctxs, parents, hkv, kc, vc, kt, vt)
    q = (rng.standard_normal((len(ctxs), t, hq, D))).astype(np.float16)
    got = oracle.attention(cache, tables, ctxs, q, np.stack(parents), hq, path)
    for s, c in enumerate(ctxs):
        want = dense_attention(q[s], kx[s], vx[s], parents[s], c, hq, hkv, int8=(path == "int8"))
        np.testing.assert_allclose(got[s], want, rtol=1e-12, atol=1e-13)


def test_decode_reproduces_representable_values():
    rng = np.random.default_rng(4)
    k16, k64 = representable_rows(rng, 300, 2)
    v16, v64 = representable_rows(rng, 300, 2)
    cache = oracle.Cache(2, 3)
    tables = [np.array([2, 0], np.int32)]
    oracle.kv_append(cache, tables, k16, v16, [0] * 300, list(range(300)))
    assert np.array_equal(oracle.decode(cache, tables, 0, 0, 300, "k"), k64)
    assert np.array_equal(oracle.decode(cache, tables, 0, 0, 300, "v"), v64)


def test_closed_form_zero_keys_give_mean_of_visible_values():
    rng = np.random.default_rng(8)
    hkv, hq, t, ctx = 1, 2, 5, 33
    parent = np.array([-1, 0, 1, 0, 3], np.int32)
    kz16, _ = representable_rows(rng, ctx + t, hkv, zero=True)
    v16, v64 = representable_rows(rng, ctx + t, hkv)
    cache, tables = build_cache(rng, [ctx], [parent], hkv, [kz16[:ctx]], [v16[:ctx]], [kz16[ctx:]], [v16[ctx:]])
    q = rng.standard_normal((1, t, hq, D)).astype(np.float16)
    got = oracle.attention(cache, tables, [ctx], q, parent[None], hq, "exact")
    for i in range(t):
        vis = list(range(ctx)) + [ctx + a for a in sorted(ancestors_by_walk(parent, i))]
        want = v64[vis, 0, :].mean(axis=0)
        for qh in range(hq):
            np.testing.assert_allclose(got[0, i, qh], want, rtol=1e-13, atol=1e-14)


def test_closed_form_root_with_empty_context_is_its_own_value():
    rng = np.random.default_rng(9)
    t = 4
    parent = np.array([-1, 0, 0, 2], np.int32)
    k16 = rng.standard_normal((t, 1, D)).astype(np.float16)
    v16, v64 = representable_rows(rng, t, 1)
    cache, tables = build_cache(rng, [0], [parent], 1, [k16[:0]], [v16[:0]], [k16], [v16])
    q = rng.standard_normal((1, t, 1, D)).astype(np.float16)
    got = oracle.attention(cache, tables, [0], q, parent[None], 1, "exact")
    assert np.array_equal(got[0, 0, 0], v64[0, 0])


def test_closed_form_dominant_key():
    rng = np.random.default_rng(10)
    hkv, hq, t, ctx, j = 1, 1, 2, 50, 17
    parent = np.array([-1, 0], np.int32)
    k16 = (rng.standard_normal((ctx + t, hkv, D)) * 0.01).astype(np.float16)
    k16[j] = np.float16(-16.0)  # all codes 0 with s = 4: exact
    v16, v64 = representable_rows(rng, ctx + t, hkv)
    q = np.full((1, t, hq, D), -1.0, np.float16)  # S_j = 256 * 16 / 16 = 256
    cache, tables = build_cache(rng, [ctx], [parent], hkv, [k16[:ctx]], [v16[:ctx]], [k16[ctx:]], [v16[ctx:]])
    got = oracle.attention(cache, tables, [ctx], q, parent[None], hq, "exact")
    for i in range(t):
        np.testing.assert_allclose(got[0, i, 0], v64[j, 0], rtol=1e-15, atol=1e-15)


@pytest.mark.parametrize("path", ["exact", "int8"])
def test_chain_tree_equals_sequential_single_row_decodes(path):
    """A chain of 8 verified in one round == 8 one-row decode steps, each of
    which appends its row and then attends (bit-identical in fp64)."""
    rng = np.random.default_rng(21)
    hkv, hq, t, ctx = 2, 6, 8, 77
    k16 = rng.standard_normal((ctx + t, hkv, D)).astype(np.float16)
    v16 = rng.standard_normal((ctx + t, hkv, D)).astype(np.float16)
    q = rng.standard_normal((1, t, hq, D)).astype(np.float16)
    chain = np.arange(-1, t - 1, dtype=np.int32)
    cache, tables = build_cache(rng, [ctx], [chain], hkv, [k16[:ctx]], [v16[:ctx]], [k16[ctx:]], [v16[ctx:]])
    tree_out = oracle.attention(cache, tables, [ctx], q, chain[None], hq, path)

    seq_cache = oracle.Cache(hkv, cache.pool_pages)
    oracle.kv_append(seq_cache, tables, k16[:ctx], v16[:ctx], [0] * ctx, list(range(ctx)))
    for i in range(t):
        oracle.kv_append(seq_cache, tables, k16[ctx + i:ctx + i + 1], v16[ctx + i:ctx + i + 1], [0], [ctx + i])
        step = oracle.attention(seq_cache, tables, [ctx + i], q[:, i:i + 1], np.array([[-1]], np.int32), hq, path)
        assert np.array_equal(step[0, 0], tree_out[0, i]), i


def test_int8_dots_match_big_integer_recomputation():
    rng = np.random.default_rng(31)
    hkv, hq, n = 2, 4, 40
    kx16 = np.zeros((n, hkv, D), np.float16)
    codes = np.zeros((n, hkv, D), np.int64)
    for r in range(n):
        for h in range(hkv):
            for g in range(8):
                s = 2.0 ** int(rng.integers(-2, 2))
                c = rng.integers(0, 8, 32)
                c[rng.integers(32)] = 0
                codes[r, h, 32 * g:32 * g + 32] = c
                kx16[r, h, 32 * g:32 * g + 32] = (s * (c - 4)).astype(np.float16)
    v16 = np.zeros_like(kx16)
    cache = oracle.Cache(hkv, 1)
    tables = [np.array([0], np.int32)]
    oracle.kv_append(cache, tables, kx16, v16, [0] * n, list(range(n)))
    q = (rng.standard_normal(D) * 3).astype(np.float16)
    for qh in range(hq):
        got = oracle.int8_dots(cache, tables, 0, q, qh, hq, 0, n)
        qs = [Fraction(float(v)) for v in q.astype(np.float64)]
        m = max(abs(v) for v in qs)
        qi = [round(Fraction(127) * v / m) for v in qs]
        h = qh // (hq // hkv)
        for j in range(n):
            for g in range(8):
                want = sum(qi[32 * g + i] * (int(codes[j, h, 32 * g + i]) - 4) for i in range(32))
                assert got[j, g] == want


def test_closed_form_huge_scores_stay_finite():
    """Scores far beyond exp()'s range (S_j = 4096): the softmax must still
    return the dominant key's value, not inf/inf."""
    rng = np.random.default_rng(12)
    hkv, hq, t, ctx, j = 1, 1, 1, 20, 5
    parent = np.array([-1], np.int32)
    k16 = (rng.standard_normal((ctx + t, hkv, D)) * 0.01).astype(np.float16)
    k16[j] = np.float16(-256.0)  # all codes 0 with s = 64: exact
    v16, v64 = representable_rows(rng, ctx + t, hkv)
    q = np.full((1, t, hq, D), -1.0, np.float16)
    cache, tables = build_cache(rng, [ctx], [parent], hkv, [k16[:ctx]], [v16[:ctx]], [k16[ctx:]], [v16[ctx:]])
    for path in ("exact", "int8"):
        got = oracle.attention(cache, tables, [ctx], q, parent[None], hq, path)
        assert np.all(np.isfinite(got))
        np.testing.assert_allclose(got[0, 0, 0], v64[j, 0], rtol=1e-15, atol=1e-15)
