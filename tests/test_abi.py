"""The C-ABI library loads and exports every symbol include/stv.h declares;
host-side validation and workspace sizing work without a GPU (no compute
calls here)."""
import ctypes
import os
import re

import pytest

import speculative_tree_verify_bit_gb300 as stv
from speculative_tree_verify_bit_gb300 import build as stv_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    stv_build.build()
    return stv.load()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "stv.h")).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(stv_\w+)\(", text, re.M)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_symbols()
    assert len(names) >= 10
    assert set(names) == set(stv.EXPORTS)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    assert stv.status_string(0) == "STV_OK"
    assert stv.status_string(-3) == "STV_ERR_WORKSPACE_TOO_SMALL"
    assert stv.status_string(-99) == "STV_ERR_UNKNOWN"


def test_page_bytes_and_shape_validation(lib):
    assert stv.stv_page_bytes(stv.make_shape(24, 4)) == 229376
    # the int4 per-token-head format (group 256): 4 heads x 66,560 B
    assert stv.stv_page_bytes(stv.make_shape(24, 4, stv.GROUP_INT4)) == 4 * stv.HEAD_BLOCK_BYTES_INT4 == 266240
    for bad in (stv.stv_shape(24, 4, 128, 32, 256), stv.stv_shape(24, 5, 256, 32, 256),
                stv.stv_shape(24, 4, 256, 16, 256), stv.stv_shape(24, 4, 256, 32, 128)):
        with pytest.raises(stv.StvError) as e:
            stv.stv_page_bytes(bad)
        assert e.value.status == stv.STV_ERR_SHAPE_UNSUPPORTED


def _seqs(ctxs, pages):
    arr = (stv.stv_seq * len(ctxs))()
    for i, (c, p) in enumerate(zip(ctxs, pages)):
        arr[i] = stv.stv_seq(0x1000, p, c)  # a dummy device address: never dereferenced here
    return arr


def _ws(shape, ctxs, pages, t, sm):
    out = ctypes.c_size_t()
    rc = stv.load().stv_verify_workspace_bytes(ctypes.byref(shape), _seqs(ctxs, pages), len(ctxs), t, sm,
                                               ctypes.byref(out))
    return rc, out.value


def test_workspace_bytes_long_context_plan(lib):
    # 262,144 + 16 keys = 4,097 tiles of 64 per KV head; 4 heads on 152 SMs
    # -> 108 tiles per split, 38 splits per head, 152 work units.
    rc, nbytes = _ws(stv.make_shape(), [262144], [1025], 16, 152)
    assert rc == 0
    qi = 16 * 24 * 256
    sq = 16 * 24 * 4
    opart = 152 * 96 * 256 * 4
    ml = 152 * 96 * 2 * 4
    cnt = (2 + 64 * 4) * 4  # stv_append_verify_combine's counters, first: 2 + STV_MAX_SEQS * hkv words
    a = lambda x: (x + 255) // 256 * 256
    assert nbytes == a(a(a(a(cnt) + qi) + sq) + opart) + ml


def test_workspace_units_never_exceed_sm_count(lib):
    for ctxs in ([1024], [1 << 20], [1024 << i for i in range(8)], [0] * 64, [7] * 3):
        pages = [-(-(c + 16) // 256) for c in ctxs]
        rc1, small = _ws(stv.make_shape(), ctxs, pages, 16, 152)
        rc2, big = _ws(stv.make_shape(), ctxs, pages, 16, 10_000)
        assert rc1 == 0 and rc2 == 0 and big >= small


def _balanced_units(ctxs, t, hkv, sm, rows):
    """The split plan for several sequences on the 3-bit cache, restated: the
    one-unit-per-SM split k0, then the split k in [k0 / 4, k0) whose units,
    dealt longest first in snake order to min(SMs, units) CTAs at (tiles + 3)
    each, finish first (ties to the larger k), within 640 units and 24 MiB of
    partials."""
    tiles = [-(-(c + t) // 64) for c in ctxs]
    total = hkv * sum(tiles)
    k_min = max([1] + [-(-x // 256) for x in tiles])
    k0 = max(-(-total // sm), k_min)
    while sum(hkv * -(-x // k0) for x in tiles) > max(sm, len(tiles) * hkv):
        k0 += 1

    def lengths(k):
        return [min(k, x - j * k) for x in tiles for _ in range(hkv) for j in range(-(-x // k))]

    def makespan(lens):
        n = min(sm, len(lens))
        load = [0] * n
        for w, ln in enumerate(sorted(lens, reverse=True)):
            kk, b = divmod(w, n)
            load[n - 1 - b if kk % 2 else b] += ln + 3
        return max(load)

    best_k, best = k0, makespan(lengths(k0))
    for k in range(k0 - 1, max(k_min, k0 // 4) - 1, -1):
        lens = lengths(k)
        if len(lens) > 640 or len(lens) * rows * 1024 > 24 << 20:
            break
        c = makespan(lens)
        if c < best:
            best_k, best = k, c
    return sum(hkv * -(-x // best_k) for x in tiles)


@pytest.mark.parametrize("ctxs", [[1024 << i for i in range(8)], [300, 0, 1000, 2047], [131072, 131072],
                                  [100000, 20000, 5000], [40000] + [500] * 20])
def test_balanced_plan_for_several_sequences(lib, ctxs):
    """Several sequences on the 3-bit cache: the plan may hold more units
    than SMs (the persistent verify kernel deals them longest first); the
    workspace holds that plan's partials."""
    units = _balanced_units(ctxs, 16, 4, 152, 96)
    pages = [-(-(c + 16) // 256) for c in ctxs]
    rc, nbytes = _ws(stv.make_shape(), ctxs, pages, 16, 152)
    assert rc == 0
    n = len(ctxs)
    a = lambda x: (x + 255) // 256 * 256
    cnt = (2 + 64 * 4) * 4
    assert nbytes == a(a(a(a(cnt) + n * 16 * 24 * 256) + n * 16 * 24 * 4) + units * 96 * 256 * 4) + units * 96 * 2 * 4
    if ctxs[0] == 1024:
        assert units == 168  # 109 tiles per split: 152 long units and 16 short ones


def test_balanced_plan_is_for_the_three_bit_cache_only(lib):
    """The int4 cache keeps one unit per SM (its kernel is not persistent)."""
    ctxs = [1024 << i for i in range(8)]
    pages = [-(-(c + 16) // 256) for c in ctxs]
    rc, nbytes = _ws(stv.make_shape(group=256), ctxs, pages, 16, 152)
    assert rc == 0
    a = lambda x: (x + 255) // 256 * 256
    units = 4 * sum(-(-(-(-(c + 16) // 64)) // 129) for c in ctxs)  # 129 tiles per split
    assert units == 136
    cnt = (2 + 64 * 4) * 4
    assert nbytes == a(a(a(a(cnt) + 8 * 16 * 24 * 256) + 8 * 16 * 24 * 4) + units * 96 * 256 * 4) + units * 96 * 2 * 4


def test_split_plan_caps_splits_per_head(lib):
    # 2^20 + 16 keys = 16,385 tiles per KV head.  Planned for 10,000 SMs the
    # plan would cut them finer than the 256 splits split_combine accepts, so
    # it takes ceil(16,385 / 256) = 65 tiles per split: 253 splits per head,
    # 1,012 work units.
    ctx = 1 << 20
    rc, nbytes = _ws(stv.make_shape(), [ctx], [-(-(ctx + 16) // 256)], 16, 10_000)
    assert rc == 0
    units = 4 * -(-16385 // 65)
    a = lambda x: (x + 255) // 256 * 256
    assert units == 1012
    cnt = (2 + 64 * 4) * 4
    assert nbytes == a(a(a(a(cnt) + 16 * 24 * 256) + 16 * 24 * 4) + units * 96 * 256 * 4) + units * 96 * 2 * 4


@pytest.mark.parametrize("ctxs,pages,t,rc", [
    ([100], [1], 16, stv.STV_OK),
    ([250], [1], 16, stv.STV_ERR_INVALID_ARG),    # ctx + T past the pages
    ([-1], [1], 16, stv.STV_ERR_INVALID_ARG),
    ([100], [1], 0, stv.STV_ERR_SHAPE_UNSUPPORTED),
    ([100], [1], 33, stv.STV_ERR_SHAPE_UNSUPPORTED),
    ([100] * 65, [1] * 65, 16, stv.STV_ERR_INVALID_ARG),
])
def test_host_validation(lib, ctxs, pages, t, rc):
    assert _ws(stv.make_shape(), ctxs, pages, t, 152)[0] == rc


def test_rows_per_kv_head_limit(lib):
    # T * G must stay <= 128: 32 nodes x 6 heads is rejected, 32 x 4 accepted
    assert _ws(stv.make_shape(24, 4), [10], [1], 32, 152)[0] == stv.STV_ERR_SHAPE_UNSUPPORTED
    assert _ws(stv.make_shape(16, 4), [10], [1], 32, 152)[0] == stv.STV_OK


def test_int4_format_plans_like_the_3bit_cache(lib):
    """The workspace and the split plan depend on the shape and the key
    ranges, not on the cache format: group 256 sizes exactly as group 32, and
    the host checks (T limit, pages) are the same."""
    for ctxs, t in (([262144], 16), ([1024, 77, 4000], 7), ([0], 16)):
        pages = [-(-(c + t) // 256) for c in ctxs]
        rc3, b3 = _ws(stv.make_shape(24, 4), ctxs, pages, t, 152)
        rc4, b4 = _ws(stv.make_shape(24, 4, stv.GROUP_INT4), ctxs, pages, t, 152)
        assert rc3 == rc4 == 0 and b3 == b4
    assert _ws(stv.make_shape(24, 4, stv.GROUP_INT4), [250], [1], 16, 152)[0] == stv.STV_ERR_INVALID_ARG
    assert _ws(stv.make_shape(24, 4, stv.GROUP_INT4), [10], [1], 33, 152)[0] == stv.STV_ERR_SHAPE_UNSUPPORTED
