"""Pins for the oracle's second cache format (next row f3): int4 codes with one
fp16 scale per token and KV head (syv-ai README (mirror), int4 KV section:
the stock int4_per_token_head cache).  Reading: s = fp16(max|x| / 7),
c = clamp(rne(x / s), -8, 7), stored as c + 8; decoded s * c.

Checked against closed forms for the scale, a brute-force nearest-code search
for the codes, a hand-derived word of the nibble layout, exact decoding of
representable rows, dense fp64 attention with an explicit mask, and commit ==
re-packing the committed rows."""
import numpy as np
import pytest

import oracle
from test_oracle_attention import build_cache, dense_attention  # noqa: F401 (dense reference)

D = 256


@pytest.mark.parametrize("m,s", [(7.0, 1.0), (3.5, 0.5), (896.0, 128.0), (7 * 2.0 ** -10, 2.0 ** -10)])
def test_scale_closed_forms(m, s):
    row = np.zeros(D, np.float16)
    row[3] = np.float16(-m)
    got, _ = oracle.quantize_row_i4(row)
    assert float(np.uint16(got).view(np.float16)) == s


def nearest_codes(x, s):
    """argmin over c in -8..7 of |x - s c|, ties to the even c, clamped."""
    cs = np.arange(-8, 8, dtype=np.float64)
    out = np.zeros(len(x), np.int64)
    for i, v in enumerate(x.astype(np.float64)):
        err = np.abs(v - s * cs)
        best = np.flatnonzero(err == err.min())
        out[i] = int(cs[best[0]]) if len(best) == 1 else int(cs[best[np.argmin(np.abs(cs[best]) % 2)]])
    return out


@pytest.mark.parametrize("m", [7.0, 1.0, 0.37, 1000.0, 5e-5, 3 * 2.0 ** -24, 11 * 2.0 ** -24])
def test_codes_are_the_nearest_representable_value(m):
    h = np.arange(65536, dtype=np.uint16).view(np.float16)
    vals = h[np.isfinite(h) & (np.abs(h.astype(np.float64)) <= np.float16(m))]
    for start in range(0, len(vals), 255):
        row = np.zeros(D, np.float16)
        row[0] = np.float16(m)
        chunk = vals[start:start + 255]
        row[1:1 + len(chunk)] = chunk
        sbits, u = oracle.quantize_row_i4(row)
        s = float(np.uint16(sbits).view(np.float16))
        if s == 0.0:
            assert np.all(u == 8)
            continue
        want = nearest_codes(row, s) + 8
        assert np.array_equal(u.astype(np.int64), want), (m, start)


def test_word_layout_hand_derived():
    """Codes u = 1..8 for elements 0..7 of a word: even elements fill bits
    0-15 (4 bits each, in order), odd ones bits 16-31, so the word is
    0x86427531.  K: channels 0..7 of token 0; V: channel 0, tokens 0..7."""
    row = np.zeros(D, np.float16)
    row[:8] = np.arange(-7, 1, dtype=np.float16)  # u = c + 8 = 1..8, and max |x| = 7 gives s = 1
    rows = np.repeat(row[None, None, :], 8, axis=0)  # 8 tokens, one KV head
    vrows = np.zeros((8, 1, D), np.float16)
    for tok in range(8):
        vrows[tok, 0, :] = np.float16(tok - 7)  # channel 0 of token tok: c = tok - 7, u = tok + 1
        vrows[tok, 0, 1] = np.float16(7.0)      # max |x| = 7: s = 1 for every token
    cache = oracle.Cache(1, 1, bits=4)
    table = [np.zeros(1, np.int32)]
    oracle.kv_append(cache, table, rows, vrows, [0] * 8, list(range(8)))
    k_word0 = int(cache.pool[0:4].view(np.uint32)[0])
    v_off = 32768 + 512  # V codes of tile 0, channel 0, tokens 0..7
    v_word0 = int(cache.pool[v_off:v_off + 4].view(np.uint32)[0])
    assert k_word0 == 0x86427531
    assert v_word0 == 0x86427531


def representable_rows_i4(rng, n_rows, hkv):
    """fp16 rows exactly s * c, s a power of two, c in -7..7 with one |c| = 7
    per (token, head), so max |x| = 7 s fixes the scale to s."""
    x = np.zeros((n_rows, hkv, D), np.float64)
    for r in range(n_rows):
        for h in range(hkv):
            s = 2.0 ** int(rng.integers(-3, 3))
            c = rng.integers(-7, 8, D)
            c[rng.integers(D)] = 7 * (1 if rng.random() < 0.5 else -1)
            x[r, h] = s * c
    x16 = x.astype(np.float16)
    assert np.array_equal(x16.astype(np.float64), x)
    return x16, x


def test_decode_reproduces_representable_values():
    rng = np.random.default_rng(41)
    k16, k64 = representable_rows_i4(rng, 300, 2)
    v16, v64 = representable_rows_i4(rng, 300, 2)
    cache = oracle.Cache(2, 3, bits=4)
    tables = [np.array([2, 0, 1], np.int32)]
    oracle.kv_append(cache, tables, k16, v16, [0] * 300, list(range(300)))
    assert np.array_equal(oracle.decode(cache, tables, 0, 0, 300, "k"), k64)
    assert np.array_equal(oracle.decode(cache, tables, 0, 0, 300, "v"), v64)


def build_cache_i4(rng, ctx, parent_list, hkv, k_ctx, v_ctx, k_tree, v_tree):
    n_seqs, t = len(ctx), len(parent_list[0])
    need = [-(-(c + t) // 256) for c in ctx]
    pool_pages = sum(need) + 1
    perm = rng.permutation(pool_pages)
    tables, at = [], 0
    for n in need:
        tables.append(perm[at:at + n].astype(np.int32))
        at += n
    cache = oracle.Cache(hkv, pool_pages, bits=4)
    for s in range(n_seqs):
        if ctx[s]:
            oracle.kv_append(cache, tables, k_ctx[s], v_ctx[s], [s] * ctx[s], list(range(ctx[s])))
        oracle.kv_append(cache, tables, k_tree[s], v_tree[s], [s] * t, [ctx[s] + i for i in range(t)])
    return cache, tables


@pytest.mark.parametrize("path", ["exact", "int8"])
@pytest.mark.parametrize("seed", [0, 1])
def test_attention_matches_dense_bruteforce(path, seed):
    rng = np.random.default_rng(500 + seed)
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
        k16, k64 = representable_rows_i4(rng, c + t, hkv)
        v16, v64 = representable_rows_i4(rng, c + t, hkv)
        kc.append(k16[:c]); vc.append(v16[:c]); kt.append(k16[c:]); vt.append(v16[c:])
        kx.append(k64); vx.append(v64)
    cache, tables = build_cache_i4(rng, ctxs, parents, hkv, kc, vc, kt, vt)
    q = (rng.standard_normal((len(ctxs), t, hq, D))).astype(np.float16)
    got = oracle.attention(cache, tables, ctxs, q, np.stack(parents), hq, path)
    for s, c in enumerate(ctxs):
        want = dense_attention(q[s], kx[s], vx[s], parents[s], c, hq, hkv, int8=(path == "int8"))
        np.testing.assert_allclose(got[s], want, rtol=1e-12, atol=1e-13)


def test_commit_equals_repacking_committed_rows():
    rng = np.random.default_rng(61)
    hkv, t, ctx = 2, 5, 250  # the tree rows straddle a page and a 64-token tile
    k = rng.standard_normal((ctx + t, hkv, D)).astype(np.float16)
    v = rng.standard_normal((ctx + t, hkv, D)).astype(np.float16)
    tables = [np.array([1, 0, 2], np.int32)]
    cache = oracle.Cache(hkv, 3, bits=4)
    oracle.kv_append(cache, tables, k, v, [0] * (ctx + t), list(range(ctx + t)))
    path = np.array([[0, 2, 3, 0, 0]], np.int32)
    oracle.kv_commit(cache, tables, [ctx], [3], path, t)
    ref = oracle.Cache(hkv, 3, bits=4)
    rows = [ctx + i for i in (0, 2, 3)] + [ctx + 3, ctx + 4]  # slots past the commit keep their old rows
    oracle.kv_append(ref, tables, k[:ctx], v[:ctx], [0] * ctx, list(range(ctx)))
    oracle.kv_append(ref, tables, k[rows], v[rows], [0] * len(rows), list(range(ctx, ctx + len(rows))))
    assert np.array_equal(cache.pool, ref.pool)
