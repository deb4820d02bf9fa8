"""fp64 CPU oracle for the tree-verify round over a 3-bit KV cache.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package.  It shares no code with
the CUDA library (``speculative_tree_verify_bit_gb300``) and imports nothing
from it; the two meet only in the seeded input generators (``workloads``).

The arithmetic lives in ``stv_oracle.c`` (plain C, fp64, plain loops); this
module compiles it with gcc on first use and wraps it with numpy + ctypes.
Every function cites the passage it follows in the C source.

Parity pins: every function here is pinned by ``tests/test_oracle_*.py``
against brute force, closed forms, invariants or library routines.  The
pages print no worked numeric example, so nothing is pinned to a printed
value, and the oracle's fp64 values for real-model activations are
"parity unpinned" (no captured tensors exist).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "stv_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

HEAD_DIM = 256
GROUP = 32
PAGE_TOKENS = 256
HEAD_BYTES = 57344
HEAD_BYTES_I4 = 66560  # int4 per token and head (next row f3)
FORMATS = {"bit3": 0, "int4": 1, "k4v2": 2}  # cache formats (stv_oracle.c): 3-bit; int4 per token-head; K 4 / V 2 bits


def compile_c(src: str, out: str) -> None:
    """gcc, -O2, portable C11 (no flag that changes float semantics)."""
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", out, src, "-lm", "-lpthread"])


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/liboracle.so``."""
    stale = (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        compile_c(_SRC, tmp)
        os.replace(tmp, _LIB)
    return _LIB


def bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    """Declare the argument and result types of the oracle's C functions on a
    loaded library (the oracle's own build, or a test's copy of it)."""
    P = ctypes.c_void_p
    I = ctypes.c_int
    I32 = ctypes.c_int32
    I64 = ctypes.c_int64
    lib.orc_half_to_double.restype = ctypes.c_double
    lib.orc_half_to_double.argtypes = [ctypes.c_uint16]
    lib.orc_double_to_half.restype = ctypes.c_uint16
    lib.orc_double_to_half.argtypes = [ctypes.c_double]
    lib.orc_quantize_group.argtypes = [P, P, P]
    lib.orc_pack_block.argtypes = [P, P]
    lib.orc_block_code.restype = ctypes.c_uint8
    lib.orc_block_code.argtypes = [P, I]
    lib.orc_kv_append.restype = I
    lib.orc_kv_append.argtypes = [P, I64, I32, I32, P, P, I, P, P, P, P, I, I]
    lib.orc_check_tree.restype = I
    lib.orc_check_tree.argtypes = [P, I]
    lib.orc_ancestors.restype = I
    lib.orc_ancestors.argtypes = [P, I, P]
    lib.orc_quantize_q_int8.argtypes = [P, P, P]
    lib.orc_attention.restype = I
    lib.orc_attention.argtypes = [P, I64, I32, I32, I32, P, P, P, I, P, P, I, I, P, I, P, I, I]
    lib.orc_int8_dots.restype = I
    lib.orc_int8_dots.argtypes = [P, I64, I32, I32, I32, P, P, I, P, I, I64, I64, P, I]
    lib.orc_tree_accept.restype = I
    lib.orc_tree_accept.argtypes = [P, P, P, I, P, P, P]
    lib.orc_kv_commit.restype = I
    lib.orc_kv_commit.argtypes = [P, I64, I32, I32, P, P, P, I, P, P, I, I]
    lib.orc_decode_rows.restype = I
    lib.orc_decode_rows.argtypes = [P, I64, I32, I32, P, P, I, I64, I64, I, P, I]
    lib.orc_quantize_row_i4.restype = None
    lib.orc_quantize_row_i4.argtypes = [P, P, P]
    lib.orc_quantize_group_bits.restype = None
    lib.orc_quantize_group_bits.argtypes = [P, I, P, P]
    lib.orc_lookup_draft.restype = I
    lib.orc_lookup_draft.argtypes = [P, I64, I, I, I, P, P, P, P]
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = bind(ctypes.CDLL(_LIB))
    return _lib


def _p(a: np.ndarray) -> ctypes.c_void_p:
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return ctypes.c_void_p(a.ctypes.data)


def _u16(a) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype == np.float16:
        a = a.view(np.uint16)
    return np.ascontiguousarray(a, dtype=np.uint16)


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


class OracleError(RuntimeError):
    pass


def _check(rc: int, what: str):
    if rc != 0:
        raise OracleError(f"oracle {what} failed with status {rc}")


# --------------------------------------------------------------------------
# Scalars and the quantizer
# --------------------------------------------------------------------------

def half_to_double(h: int) -> float:
    return _load().orc_half_to_double(int(h) & 0xFFFF)


def double_to_half(x: float) -> int:
    return int(_load().orc_double_to_half(float(x)))


def quantize_group(x16) -> tuple[int, np.ndarray]:
    """32 fp16 values -> (fp16 scale bits, codes uint8[32])."""
    x = _u16(x16).reshape(32)
    s = np.zeros(1, np.uint16)
    codes = np.zeros(32, np.uint8)
    _load().orc_quantize_group(_p(x), _p(s), _p(codes))
    return int(s[0]), codes


def pack_block(codes) -> np.ndarray:
    c = np.ascontiguousarray(np.asarray(codes, np.uint8).reshape(32))
    w = np.zeros(3, np.uint32)
    _load().orc_pack_block(_p(c), _p(w))
    return w


def block_code(words, i: int) -> int:
    w = np.ascontiguousarray(np.asarray(words, np.uint32).reshape(3))
    return int(_load().orc_block_code(_p(w), int(i)))


def quantize_q_int8(q16) -> tuple[np.ndarray, float]:
    q = _u16(q16).reshape(HEAD_DIM)
    qi = np.zeros(HEAD_DIM, np.int8)
    sq = np.zeros(1, np.float32)
    _load().orc_quantize_q_int8(_p(q), _p(qi), _p(sq))
    return qi, float(sq[0])


def ancestors(parent) -> np.ndarray:
    p = _i32(parent)
    anc = np.zeros(len(p), np.uint32)
    _check(_load().orc_ancestors(_p(p), len(p), _p(anc)), "ancestors")
    return anc


def check_tree(parent) -> bool:
    p = _i32(parent)
    return _load().orc_check_tree(_p(p), len(p)) == 0


# --------------------------------------------------------------------------
# The paged cache
# --------------------------------------------------------------------------

class Cache:
    """A host-side paged cache for one layer (bytes as uint8): the 3-bit cache
    (bits=3), the int4 per-token-head cache (bits=4) or the K 4 / V 2-bit
    cache (kind="k4v2"); every call names the format to the C side."""

    def __init__(self, hkv: int, pool_pages: int, pool: np.ndarray | None = None, bits: int = 3,
                 kind: str | None = None):
        self.hkv = int(hkv)
        self.bits = int(bits)
        self.kind = kind or ("bit3" if bits == 3 else "int4")
        self.fmt = FORMATS[self.kind]
        self.page_bytes = self.hkv * (HEAD_BYTES_I4 if self.kind == "int4" else HEAD_BYTES)
        self.pool_pages = int(pool_pages)
        if pool is None:
            pool = np.zeros(self.page_bytes * self.pool_pages, np.uint8)
        assert pool.dtype == np.uint8 and pool.size == self.page_bytes * self.pool_pages
        self.pool = np.ascontiguousarray(pool)


def _tables(page_tables):
    offs = np.zeros(len(page_tables) + 1, np.int32)
    for i, t in enumerate(page_tables):
        offs[i + 1] = offs[i] + len(t)
    flat = _i32(np.concatenate([np.asarray(t, np.int32) for t in page_tables]) if page_tables else [])
    return flat, offs


def kv_append(cache: Cache, page_tables, k16, v16, row_seq, row_pos):
    """Quantize fp16 K/V rows [n_rows][hkv][256] into ``cache`` in place."""
    flat, offs = _tables(page_tables)
    k = _u16(k16)
    v = _u16(v16)
    rs = _i32(row_seq)
    rp = _i32(row_pos)
    n = len(rs)
    assert k.size == n * cache.hkv * HEAD_DIM and v.size == k.size
    _check(
        _load().orc_kv_append(_p(cache.pool), cache.page_bytes, cache.pool_pages, cache.hkv, _p(flat),
                              _p(offs), len(page_tables), _p(k), _p(v), _p(rs), _p(rp), n, cache.fmt),
        "kv_append",
    )


def decode(cache: Cache, page_tables, seq: int, tok_begin: int, tok_end: int, which: str) -> np.ndarray:
    """Decoded K or V values (fp64) [n_tok][hkv][256]."""
    flat, offs = _tables(page_tables)
    out = np.zeros((tok_end - tok_begin, cache.hkv, HEAD_DIM), np.float64)
    _check(
        _load().orc_decode_rows(_p(cache.pool), cache.page_bytes, cache.pool_pages, cache.hkv, _p(flat), _p(offs),
                                int(seq), int(tok_begin), int(tok_end), 0 if which == "k" else 1, _p(out), cache.fmt),
        "decode",
    )
    return out


def attention(cache: Cache, page_tables, ctx, q16, parent, hq: int, path: str, rows=None,
              n_threads: int = 1) -> np.ndarray:
    """Attention output (fp64) of the verify round.

    q16: [n_seqs][T][hq][256] fp16; parent: [n_seqs][T]; ctx: [n_seqs].
    rows: list of (seq, node, q head); default every row.  Returns
    [len(rows)][256], or [n_seqs][T][hq][256] when rows is None.
    """
    flat, offs = _tables(page_tables)
    q = _u16(q16)
    par = _i32(parent)
    n_seqs, t = par.shape
    ctx_a = _i32(ctx)
    full = rows is None
    if full:
        rows = [(s, i, h) for s in range(n_seqs) for i in range(t) for h in range(hq)]
    r = _i32(np.asarray(rows, np.int32).reshape(-1, 3))
    out = np.zeros((len(r), HEAD_DIM), np.float64)
    _check(
        _load().orc_attention(_p(cache.pool), cache.page_bytes, cache.pool_pages, int(hq), cache.hkv, _p(flat),
                              _p(offs), _p(ctx_a), n_seqs, _p(q), _p(par), t, 0 if path == "exact" else 1,
                              _p(r), len(r), _p(out), int(n_threads), cache.fmt),
        "attention",
    )
    if full:
        return out.reshape(n_seqs, t, hq, HEAD_DIM)
    return out


def int8_dots(cache: Cache, page_tables, seq: int, q_row16, qhead: int, hq: int, tok_begin: int,
              tok_end: int) -> np.ndarray:
    """Integer per-group dots I_g [n_tok][8] of one Q row against keys."""
    flat, offs = _tables(page_tables)
    q = _u16(q_row16).reshape(HEAD_DIM)
    out = np.zeros((tok_end - tok_begin, 8), np.int32)
    _check(
        _load().orc_int8_dots(_p(cache.pool), cache.page_bytes, cache.pool_pages, int(hq), cache.hkv, _p(flat),
                              _p(offs), int(seq), _p(q), int(qhead), int(tok_begin), int(tok_end), _p(out), cache.fmt),
        "int8_dots",
    )
    return out


def tree_accept(parent, draft, argmax):
    """Greedy acceptance of one tree -> (n_commit, path, out_ids)."""
    p = _i32(parent)
    d = _i32(draft)
    a = _i32(argmax)
    t = len(p)
    n = np.zeros(1, np.int32)
    path = np.zeros(t, np.int32)
    out = np.zeros(t, np.int32)
    _check(_load().orc_tree_accept(_p(p), _p(d), _p(a), t, _p(n), _p(path), _p(out)), "tree_accept")
    k = int(n[0])
    return k, path[:k].copy(), out[:k].copy()


def kv_commit(cache: Cache, page_tables, ctx, n_commit, path, t: int):
    """Compact accepted rows in place.  path: [n_seqs][t] (first n_commit used)."""
    flat, offs = _tables(page_tables)
    c = _i32(ctx)
    n = _i32(n_commit)
    pth = _i32(path).reshape(len(c), t)
    _check(
        _load().orc_kv_commit(_p(cache.pool), cache.page_bytes, cache.pool_pages, cache.hkv, _p(flat), _p(offs),
                              _p(c), len(c), _p(n), _p(pth), int(t), cache.fmt),
        "kv_commit",
    )


def lookup_draft(history, min_len: int = 6, max_len: int = 12, k: int = 15):
    """Lookup drafting (stv_oracle.c, orc_lookup_draft): propose the up to k
    tokens that followed the latest earlier occurrence of the history's
    longest suffix of length max_len .. min_len.  Returns
    (proposal int32 array, match_len, match_pos); match_len 0 and match_pos -1
    when no suffix of those lengths occurs earlier."""
    h = np.ascontiguousarray(history, dtype=np.int32)
    prop = np.zeros(max(k, 1), np.int32)
    n_prop, mlen, mpos = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int64()
    rc = _load().orc_lookup_draft(_p(h), len(h), int(min_len), int(max_len), int(k), ctypes.byref(n_prop), _p(prop),
                                  ctypes.byref(mlen), ctypes.byref(mpos))
    if rc != 0:
        raise ValueError("orc_lookup_draft: bad lengths")
    return prop[:n_prop.value].copy(), mlen.value, mpos.value


def quantize_row_i4(x):
    """int4 per-token-head quantizer (stv_oracle.c, orc_quantize_row_i4):
    256 fp16 values -> (fp16 scale bits, codes u = c + 8 in 0..15)."""
    xh = np.ascontiguousarray(np.asarray(x, np.float16).view(np.uint16))
    assert xh.size == HEAD_DIM
    s = np.zeros(1, np.uint16)
    u = np.zeros(HEAD_DIM, np.uint8)
    _load().orc_quantize_row_i4(_p(xh), _p(s), _p(u))
    return s[0], u


def quantize_group_bits(x, bits: int):
    """The b-bit group quantizer (stv_oracle.c, orc_quantize_group_bits): 32
    fp16 values -> (fp16 scale bits, codes u = c + 2^(b-1))."""
    xh = np.ascontiguousarray(np.asarray(x, np.float16).view(np.uint16))
    assert xh.size == GROUP
    s = np.zeros(1, np.uint16)
    u = np.zeros(GROUP, np.uint8)
    _load().orc_quantize_group_bits(_p(xh), int(bits), _p(s), _p(u))
    return s[0], u
