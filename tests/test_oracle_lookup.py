"""Pins for the lookup-drafting oracle (Reddit posts (u/iamMess), "Now added"
list, lookup-augmented drafting: draft tokens copied from where the request's
trailing six to twelve tokens last appeared earlier in it).

The oracle tries every length from longest to shortest and every start, token
by token.  Here it is checked against hand-worked cases and against a search
written differently: tokens encoded as fixed-width bytes and found with
bytes.rfind, on random histories over tiny alphabets (many repeats at every
length)."""
import numpy as np
import pytest

import oracle


def rfind_reference(h, min_len, max_len, k):
    """Longest suffix length first, latest earlier start, via bytes.rfind."""
    h = [int(x) for x in h]
    n = len(h)
    enc = b"".join(x.to_bytes(4, "little", signed=True) for x in h)
    for L in range(max_len, min_len - 1, -1):
        if L >= n:
            continue
        suffix = enc[4 * (n - L):]
        end = 4 * (n - 1)  # an occurrence must start before n - L, so end before byte 4(n-1)
        while True:
            at = enc.rfind(suffix, 0, end)
            if at < 0:
                break
            if at % 4 == 0:  # aligned to a token boundary
                p = at // 4
                return h[p + L:p + L + k], L, p
            end = at + len(suffix) - 1  # retry left of this unaligned hit
    return [], 0, -1


@pytest.mark.parametrize("h,min_len,max_len,k,want", [
    # suffix 1..6 (length 6) occurs at 0; the longer suffixes 9,1..6 etc. never
    # occurred; propose what followed: 7 8 9 1 2
    (list(range(1, 10)) + list(range(1, 7)), 6, 12, 5, ([7, 8, 9, 1, 2], 6, 0)),
    # eight equal tokens: lengths 12..8 are too long for an earlier start; the
    # length-7 suffix occurs at 0 (overlapping itself); one token follows it
    ([5] * 8, 6, 12, 4, ([5], 7, 0)),
    # no repeated window at all
    (list(range(20)), 6, 12, 4, ([], 0, -1)),
    # the suffix 3 4 5 6 7 8 occurs at 2 and at 12; the later start (12) wins
    ([1, 2, 3, 4, 5, 6, 7, 8, 100, 101, 102, 103, 3, 4, 5, 6, 7, 8, 200, 3, 4, 5, 6, 7, 8], 6, 12, 3,
     ([200, 3, 4], 6, 12)),
    # a 7-token suffix occurs early (start 0) and a 6-token one later (start
    # 9, where 99 precedes it): the longer match wins even though it is older
    ([10, 11, 12, 13, 14, 15, 16, 50, 99, 11, 12, 13, 14, 15, 16, 60, 10, 11, 12, 13, 14, 15, 16], 6, 12, 2,
     ([50, 99], 7, 0)),
    # history shorter than the shortest length + 1
    ([1, 2, 3, 1, 2, 3], 6, 12, 4, ([], 0, -1)),
])
def test_hand_worked_cases(h, min_len, max_len, k, want):
    prop, mlen, mpos = oracle.lookup_draft(h, min_len, max_len, k)
    assert (list(prop), mlen, mpos) == want


@pytest.mark.parametrize("alphabet,n", [(2, 40), (3, 60), (4, 200), (2, 300), (16, 500)])
def test_against_byte_string_search(alphabet, n):
    rng = np.random.default_rng(1000 * alphabet + n)
    for trial in range(60):
        h = rng.integers(0, alphabet, rng.integers(1, n + 1)).astype(np.int32)
        if trial % 3 == 0:  # plant a copied span so long matches are common
            m = len(h)
            if m > 30:
                a = rng.integers(0, m - 20)
                h = np.concatenate([h, h[a:a + rng.integers(6, 20)]])
        for min_len, max_len, k in ((6, 12, 15), (1, 3, 4), (2, 32, 7), (6, 6, 1)):
            got = oracle.lookup_draft(h, min_len, max_len, k)
            want = rfind_reference(h, min_len, max_len, k)
            assert (list(got[0]), got[1], got[2]) == (list(want[0]), want[1], want[2]), (h.tolist(), min_len, max_len)


def test_rejects_bad_lengths():
    with pytest.raises(ValueError):
        oracle.lookup_draft([1, 2, 3], 0, 4, 2)
    with pytest.raises(ValueError):
        oracle.lookup_draft([1, 2, 3], 5, 4, 2)
