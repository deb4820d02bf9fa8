"""Pins for the oracle's third cache format (next row f3): the KVarN-style
4/2-bit cache (Reddit posts (u/iamMess), "Now added" list: KVarN 4/2-bit KV
cache; syv-ai README (mirror), DFlash2 at 240k: CTX=huge).  The pages give
its name and cost, not its quantizer.  Reading: the 3-bit cache's quantizer
at other widths, per (token, KV head, 32-channel group): at b bits, h =
2^(b-1), s = fp16(max|x| / h), c = clamp(rne(x / s), -h, h - 1), stored as
c + h; K at 4 bits, V at 2 bits; decoded s * c.

Checked against: the 3-bit quantizer it generalises (b = 3), closed forms for
the scale, a brute-force nearest-code search, hand-derived words and byte
positions of the layout, exact decoding of representable rows, dense fp64
attention with an explicit mask (both paths), and commit == re-packing the
committed rows."""
import numpy as np
import pytest

import oracle
from test_oracle_attention import dense_attention
from test_oracle_int4 import nearest_codes as _nearest_i4  # noqa: F401 (same search, other range below)

D = 256


def nearest(x, s, lo, hi):
    """argmin over c in lo..hi of |x - s c|, ties to the even c."""
    cs = np.arange(lo, hi + 1, dtype=np.float64)
    out = np.zeros(len(x), np.int64)
    for i, v in enumerate(np.asarray(x, np.float64)):
        err = np.abs(v - s * cs)
        best = np.flatnonzero(err == err.min())
        out[i] = int(cs[best[0]]) if len(best) == 1 else int(cs[best[np.argmin(np.abs(cs[best]) % 2)]])
    return out


def test_three_bits_is_the_three_bit_cache_quantizer():
    """At b = 3 the generalised quantizer is the 3-bit cache's (whose code is
    already c + 4), on random groups and groups with ties and clamps."""
    rng = np.random.default_rng(7)
    for trial in range(400):
        x = (rng.standard_normal(32) * 10.0 ** rng.integers(-3, 3)).astype(np.float16)
        if trial % 4 == 0:  # exact halves between codes: ties
            s = np.float16(2.0 ** rng.integers(-3, 3))
            x = (s * (rng.integers(-8, 8, 32) / 2.0)).astype(np.float16)
            x[0] = np.float16(4 * s)
        s3, c3 = oracle.quantize_group(x)
        sb, cb = oracle.quantize_group_bits(x, 3)
        assert s3 == sb and np.array_equal(c3, cb), trial


@pytest.mark.parametrize("bits,m,s", [(4, 8.0, 1.0), (4, 3.0, 0.375), (4, 896.0, 112.0), (2, 2.0, 1.0),
                                      (2, 0.75, 0.375), (2, 2.0 ** -23, 2.0 ** -24)])
def test_scale_closed_forms(bits, m, s):
    x = np.zeros(32, np.float16)
    x[5] = np.float16(-m)
    got, _ = oracle.quantize_group_bits(x, bits)
    assert float(np.uint16(got).view(np.float16)) == s


@pytest.mark.parametrize("bits", [4, 2])
@pytest.mark.parametrize("m", [8.0, 1.0, 0.37, 900.0, 5e-5, 3 * 2.0 ** -24])
def test_codes_are_the_nearest_representable_value(bits, m):
    """Every finite fp16 value in [-m, m] (groups whose maximum is m): the
    code is the nearest of -h..h-1 to x / s, ties to even."""
    h = 1 << (bits - 1)
    allh = np.arange(65536, dtype=np.uint16).view(np.float16)
    vals = allh[np.isfinite(allh) & (np.abs(allh.astype(np.float64)) <= np.float16(m))]
    for start in range(0, len(vals), 31):
        x = np.zeros(32, np.float16)
        x[0] = np.float16(m)
        chunk = vals[start:start + 31]
        x[1:1 + len(chunk)] = chunk
        sbits, u = oracle.quantize_group_bits(x, bits)
        s = float(np.uint16(sbits).view(np.float16))
        if s == 0.0:
            assert np.all(u == h)
            continue
        assert np.array_equal(u.astype(np.int64), nearest(x, s, -h, h - 1) + h), (bits, m, start)


def test_words_hand_derived():
    """K: codes u = 1..8 on channels 0..7 of group 0 -> word 0x86427531 (even
    elements in bits 0-15, 4 bits each in order, odd ones in bits 16-31).
    V: channel 0 of tokens 0..15 with u = t mod 4 -> even tokens fill bits
    0-15 (2 bits each), odd ones bits 16-31: 0xDDDD8888."""
    k = np.zeros((16, 1, D), np.float16)
    k[0, 0, :8] = np.arange(-7, 1, dtype=np.float16)  # c = -7..0, u = 1..8
    k[0, 0, 8] = np.float16(-8.0)                       # max |x| = 8: s = 1
    v = np.zeros((16, 1, D), np.float16)
    for t in range(16):
        v[t, 0, 0] = np.float16(t % 4 - 2)  # c = t mod 4 - 2, u = t mod 4
        v[t, 0, 1] = np.float16(-2.0)       # max |x| = 2: s = 1
    cache = oracle.Cache(1, 1, kind="k4v2")
    oracle.kv_append(cache, [np.zeros(1, np.int32)], k, v, [0] * 16, list(range(16)))
    assert int(cache.pool[0:4].view(np.uint32)[0]) == 0x86427531
    assert int(cache.pool[36864:36868].view(np.uint32)[0]) == 0xDDDD8888


def test_byte_positions_hand_derived():
    """One K and one V entry of token 600 (page table [2, 0, 3, 1]: logical
    page 2 -> pool page 3, slot 88, tile 1, within 24), KV head 3 of 4, in
    channel 77 (group 2, element 13 of the group): worked out by hand from
    the layout.
      K word: 3*229376 + 3*57344 + slot 88 * 128 + group 2 * 16 + (13 // 8) * 4
              = 688128 + 172032 + 11264 + 32 + 4 = 871460, element 13 % 8 = 5
              at bit 4*2 + 16 = 24.
      K scale: 688128 + 172032 + 32768 + 88*16 + 2*2 = 894340.
      V word: 688128 + 172032 + 36864 + tile 1 * 4096 + 77*16 + (24 // 16)*4
              = 688128 + 172032 + 36864 + 4096 + 1232 + 4 = 902356, token
              24 % 16 = 8 at bit 2*4 + 0 = 8.
      V scale: 688128 + 172032 + 53248 + 1*1024 + 2*128 + 24*2 = 914736."""
    k = np.zeros((1, 4, D), np.float16)
    v = np.zeros((1, 4, D), np.float16)
    k[0, 3, 64] = np.float16(4.0)   # group 2's maximum: s = 0.5
    k[0, 3, 77] = np.float16(-2.5)  # c = -5 -> u = 3
    v[0, 3, 64] = np.float16(3.0)   # s = 1.5
    v[0, 3, 77] = np.float16(1.5)   # c = 1 -> u = 3
    cache = oracle.Cache(4, 4, kind="k4v2")
    oracle.kv_append(cache, [np.array([2, 0, 3, 1], np.int32)], k, v, [0], [600])
    pool = cache.pool
    assert (int(pool[871460:871464].view(np.uint32)[0]) >> 24) & 15 == 3
    assert int(pool[894340:894342].view(np.uint16)[0]) == 0x3800  # 0.5
    assert (int(pool[902356:902360].view(np.uint32)[0]) >> 8) & 3 == 3
    assert int(pool[914736:914738].view(np.uint16)[0]) == 0x3E00  # 1.5


def representable_rows_k4v2(rng, n_rows, hkv, bits):
    """fp16 rows exactly s * c per 32-channel group, s a power of two, c in
    -h..h-1 with one c = -h per group (max |x| = h s fixes the scale)."""
    h = 1 << (bits - 1)
    x = np.zeros((n_rows, hkv, D), np.float64)
    for r in range(n_rows):
        for kh in range(hkv):
            for g in range(D // 32):
                s = 2.0 ** int(rng.integers(-3, 3))
                c = rng.integers(-h, h, 32)
                c[rng.integers(32)] = -h
                x[r, kh, 32 * g:32 * g + 32] = s * c
    x16 = x.astype(np.float16)
    assert np.array_equal(x16.astype(np.float64), x)
    return x16, x


def test_decode_reproduces_representable_values():
    rng = np.random.default_rng(43)
    k16, k64 = representable_rows_k4v2(rng, 300, 2, 4)
    v16, v64 = representable_rows_k4v2(rng, 300, 2, 2)
    cache = oracle.Cache(2, 3, kind="k4v2")
    tables = [np.array([2, 0, 1], np.int32)]
    oracle.kv_append(cache, tables, k16, v16, [0] * 300, list(range(300)))
    assert np.array_equal(oracle.decode(cache, tables, 0, 0, 300, "k"), k64)
    assert np.array_equal(oracle.decode(cache, tables, 0, 0, 300, "v"), v64)


@pytest.mark.parametrize("path", ["exact", "int8"])
@pytest.mark.parametrize("seed", [0, 1])
def test_attention_matches_dense_bruteforce(path, seed):
    rng = np.random.default_rng(700 + seed)
    hkv, hq, t = 2, 4, 6
    ctxs = [int(rng.integers(0, 40)), int(rng.integers(1, 70))]
    parents = []
    for _ in ctxs:
        p = np.full(t, -1, np.int32)
        for i in range(1, t):
            p[i] = rng.integers(0, i)
        parents.append(p)
    need = [-(-(c + t) // 256) for c in ctxs]
    pool_pages = sum(need) + 1
    perm = rng.permutation(pool_pages)
    tables, at = [], 0
    for n in need:
        tables.append(perm[at:at + n].astype(np.int32))
        at += n
    cache = oracle.Cache(hkv, pool_pages, kind="k4v2")
    kx, vx = [], []
    for s, c in enumerate(ctxs):
        k16, k64 = representable_rows_k4v2(rng, c + t, hkv, 4)
        v16, v64 = representable_rows_k4v2(rng, c + t, hkv, 2)
        oracle.kv_append(cache, tables, k16, v16, [s] * (c + t), list(range(c + t)))
        kx.append(k64)
        vx.append(v64)
    q = rng.standard_normal((len(ctxs), t, hq, D)).astype(np.float16)
    got = oracle.attention(cache, tables, ctxs, q, np.stack(parents), hq, path)
    for s, c in enumerate(ctxs):
        want = dense_attention(q[s], kx[s], vx[s], parents[s], c, hq, hkv, int8=(path == "int8"))
        np.testing.assert_allclose(got[s], want, rtol=1e-12, atol=1e-13)


def test_commit_equals_repacking_committed_rows():
    rng = np.random.default_rng(63)
    hkv, t, ctx = 2, 5, 250  # the tree rows straddle a page and a 64-token tile
    k = rng.standard_normal((ctx + t, hkv, D)).astype(np.float16)
    v = rng.standard_normal((ctx + t, hkv, D)).astype(np.float16)
    tables = [np.array([1, 0, 2], np.int32)]
    cache = oracle.Cache(hkv, 3, kind="k4v2")
    oracle.kv_append(cache, tables, k, v, [0] * (ctx + t), list(range(ctx + t)))
    path = np.array([[0, 2, 3, 0, 0]], np.int32)
    oracle.kv_commit(cache, tables, [ctx], [3], path, t)
    ref = oracle.Cache(hkv, 3, kind="k4v2")
    rows = [ctx + i for i in (0, 2, 3)] + [ctx + 3, ctx + 4]  # slots past the commit keep their old rows
    oracle.kv_append(ref, tables, k[:ctx], v[:ctx], [0] * ctx, list(range(ctx)))
    oracle.kv_append(ref, tables, k[rows], v[rows], [0] * len(rows), list(range(ctx, ctx + len(rows))))
    assert np.array_equal(cache.pool, ref.pool)
