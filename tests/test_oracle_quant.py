"""Pins for the oracle's fp16 conversion, 3-bit quantizer, block layout and
int8 Q quantizer -- each checked against something other than the oracle:
numpy's IEEE binary16 conversion, brute-force nearest-code search, exact
rational arithmetic (fractions.Fraction) and hand-derived bit layouts."""
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def f16(bits: int) -> float:
    return float(np.array([bits], np.uint16).view(np.float16)[0])


def test_half_to_double_matches_numpy_all_patterns():
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    for b in range(0, 65536, 1):
        got = oracle.half_to_double(b)
        r = ref[b]
        if np.isnan(r):
            assert np.isnan(got)
        else:
            assert got == r, b


def test_double_to_half_matches_numpy_rounding():
    rng = np.random.default_rng(5)
    xs = np.concatenate([
        rng.standard_normal(4000) * 10.0 ** rng.integers(-9, 5, 4000),
        # exact midpoints between neighbouring halves (ties to even)
        (np.arange(0, 65000, 7).astype(np.uint16).view(np.float16).astype(np.float64)
         + np.arange(1, 65001, 7).astype(np.uint16).view(np.float16).astype(np.float64)) / 2,
        [0.0, -0.0, 65504.0, 65519.99, 65520.0, 1e-8, 2.0 ** -25, 3 * 2.0 ** -26, 2.0 ** -24],
    ])
    xs = xs[np.isfinite(xs)]
    for x in xs:
        want = int(np.array([x], np.float64).astype(np.float16).view(np.uint16)[0])
        assert oracle.double_to_half(float(x)) == want, x


def brute_code(x: float, s: float) -> int:
    """Nearest of s*(c-4), c = 0..7; ties go to the even code."""
    best, bestd = None, None
    for c in range(8):
        d = abs(Fraction(x) - Fraction(s) * (c - 4))
        if bestd is None or d < bestd or (d == bestd and c % 2 == 0):
            best, bestd = c, d
    return best


@pytest.mark.parametrize("s_bits", [0x3C00, 0x2E66, 0x4A12, 0x0400, 0x0013, 0x57FF])
def test_quantizer_exhaustive_against_brute_force(s_bits):
    """Every fp16 x in [-4s, 4s] for a fixed scale s: the code must be the
    nearest representable level (ties to even), as a brute-force search
    over the 8 codes finds it.  The group's first element is -4s, so that
    max|x| = 4s and the group scale is exactly s."""
    s = f16(s_bits)
    lead = np.float16(-4 * s)
    assert float(lead) == -4 * s
    allv = np.arange(65536, dtype=np.uint16).view(np.float16)
    allv = allv[np.isfinite(allv)]
    vals = allv[np.abs(allv.astype(np.float64)) <= 4 * s]
    # A sample when the range is huge keeps the test fast but still hits
    # every exact tie x = s*(k + 1/2).
    ties = np.array([s * (k + 0.5) for k in range(-5, 4)], np.float64)
    ties = ties[np.abs(ties) <= 4 * s]
    ties16 = ties.astype(np.float16)
    ties16 = ties16[ties16.astype(np.float64) == ties]
    if len(vals) > 8000:
        rng = np.random.default_rng(s_bits)
        vals = np.concatenate([rng.choice(vals, 8000, replace=False), ties16])
    else:
        vals = np.concatenate([vals, ties16])
    for start in range(0, len(vals), 31):
        chunk = vals[start:start + 31]
        grp = np.concatenate([[lead], chunk, np.zeros(31 - len(chunk), np.float16)]).astype(np.float16)
        sb, codes = oracle.quantize_group(grp)
        assert sb == s_bits
        assert codes[0] == 0
        for i, x in enumerate(chunk):
            assert codes[i + 1] == brute_code(float(x), s), (float(x), s)


def test_quantizer_scale_is_fp16_of_quarter_max():
    rng = np.random.default_rng(11)
    for _ in range(300):
        x = (rng.standard_normal(32) * 10.0 ** rng.integers(-6, 4)).astype(np.float16)
        sb, codes = oracle.quantize_group(x)
        m = np.max(np.abs(x.astype(np.float64)))
        assert sb == int(np.array([m / 4], np.float64).astype(np.float16).view(np.uint16)[0])
        s = f16(sb)
        for xi, c in zip(x.astype(np.float64), codes):
            assert 0 <= c <= 7
            if s > 0 and xi <= 3.5 * s:
                # not clamped: within half a step of the decoded level
                assert abs(xi - s * (int(c) - 4)) <= s / 2 + 1e-300


def test_quantizer_zero_scale_gives_code_four():
    assert oracle.quantize_group(np.zeros(32, np.float16))[1].tolist() == [4] * 32
    # max|x| = 2^-23: m/4 = 2^-25 rounds (tie, to even) to scale 0
    x = np.zeros(32, np.float16)
    x[3] = np.float16(2.0 ** -23)
    sb, codes = oracle.quantize_group(x)
    assert sb == 0 and codes.tolist() == [4] * 32


def test_block_layout_against_hand_derived_words():
    path = os.path.join(GOLDEN, "block_layout.txt")
    n = 0
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        spec, *words = line.split()
        codes = np.zeros(32, np.uint8)
        for kv in spec.split(","):
            i, c = kv.split("=")
            codes[int(i)] = int(c)
        want = [int(w, 16) for w in words]
        assert oracle.pack_block(codes).tolist() == want, spec
        for i in range(32):
            assert oracle.block_code(np.asarray(want, np.uint32), i) == codes[i]
        n += 1
    assert n >= 10


def test_block_round_trip_random():
    rng = np.random.default_rng(3)
    for _ in range(2000):
        codes = rng.integers(0, 8, 32).astype(np.uint8)
        w = oracle.pack_block(codes)
        assert [oracle.block_code(w, i) for i in range(32)] == codes.tolist()
    # 96 bits, each code bit lands on a distinct bit
    seen = set()
    for i in range(32):
        for b in range(3):
            c = np.zeros(32, np.uint8)
            c[i] = 1 << b
            w = oracle.pack_block(c)
            assert sum(bin(int(x)).count("1") for x in w) == 1
            seen.add(tuple(int(x) for x in w))
    assert len(seen) == 96


def exact_qi(q: np.ndarray):
    qs = [Fraction(float(v)) for v in q.astype(np.float64)]
    m = max(abs(v) for v in qs)
    if m == 0:
        return [0] * len(qs), 0.0
    return [round(Fraction(127) * v / m) for v in qs], float(np.float32(float(m) / 127.0))


def test_int8_q_quantizer_exact():
    rng = np.random.default_rng(17)
    for trial in range(200):
        q = (rng.standard_normal(256) * 10.0 ** rng.integers(-3, 3)).astype(np.float16)
        qi, sq = oracle.quantize_q_int8(q)
        want, wsq = exact_qi(q)
        assert qi.tolist() == want
        assert np.float32(sq) == np.float32(wsq)
        amax = int(np.argmax(np.abs(q.astype(np.float64))))
        assert abs(int(qi[amax])) == 127


def test_int8_q_quantizer_ties_to_even():
    # m = 127 exactly, so 127*q/m = q: q = k + 1/2 is an exact tie.
    q = np.zeros(256, np.float16)
    q[0] = 127
    q[1:9] = [0.5, 1.5, 2.5, -2.5, 3.5, -0.5, 126.5, -1.5]
    qi, sq = oracle.quantize_q_int8(q)
    assert qi[:9].tolist() == [127, 0, 2, 2, -2, 4, 0, 126, -2]
    assert sq == pytest.approx(1.0, abs=0)
    qz, sz = oracle.quantize_q_int8(np.zeros(256, np.float16))
    assert qz.tolist() == [0] * 256 and sz == 0.0


def test_v_layout_against_hand_derived_positions():
    """The V half of the page layout: one V entry's code bits and its group
    scale land at byte positions worked out by hand (tests/golden/v_layout.txt)
    from the layout statement, for tokens in different pages, tiles, 32-token
    blocks, KV heads and channel groups (the code-31 case spreads its bits
    over all three words)."""
    rows = []
    for line in open(os.path.join(GOLDEN, "v_layout.txt")):
        line = line.strip()
        if line and not line.startswith("#"):
            rows.append(line.split())
    assert len(rows) == 4
    table = np.array([2, 0, 3, 1], np.int32)
    for pos, head, ch, val, mch, gmax, code, word_off, shift, scale_off, scale_bits in rows:
        cache = oracle.Cache(4, 4)
        k = np.zeros((1, 4, 256), np.float16)
        v = np.zeros((1, 4, 256), np.float16)
        v[0, int(head), int(mch)] = float(gmax)
        v[0, int(head), int(ch)] = float(val)
        oracle.kv_append(cache, [table], k, v, np.zeros(1, np.int32), np.array([int(pos)], np.int32))
        pool = cache.pool
        words = pool[int(word_off):int(word_off) + 12].view(np.uint32)
        if int(shift) == 31:  # code 31: bit b in bit 31 of word b
            got = sum(((int(words[b]) >> 31) & 1) << b for b in range(3))
        else:
            got = (int(words[0]) >> int(shift)) & 7
        assert got == int(code), (pos, got)
        assert int(pool[int(scale_off):int(scale_off) + 2].view(np.uint16)[0]) == int(scale_bits, 16), pos
