"""Python binding of libstv.so -- the GB300 (sm_103a) tree-verify library.

Argument marshalling only: every function has the name of the C entry point
it calls (include/stv.h), takes torch CUDA tensors for the device pointers
and raises ``StvError`` on a negative status.  Every step of the round runs
in the library's CUDA kernels; there is no other implementation behind these
names, and importing a function fails loudly when the library is not built
(``python -m speculative_tree_verify_bit_gb300.build``).
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libstv.so")

STV_OK = 0
STV_ERR_INVALID_ARG = -1
STV_ERR_SHAPE_UNSUPPORTED = -2
STV_ERR_WORKSPACE_TOO_SMALL = -3
STV_ERR_CUDA = -4
STV_ERR_UNIMPLEMENTED = -5

STV_DEV_BAD_PAGE = 1
STV_DEV_BAD_TREE = 2
STV_DEV_BAD_ROW = 4
STV_DEV_BAD_COMMIT = 8
STV_DEV_TIMEOUT = 16

STV_KV_BY_GROUP = 0  # group 32: the 3-bit cache; group 256: the int4 per-token-head cache
STV_KV_K4V2 = 2      # the K 4 / V 2-bit cache (group 32)

STV_PATH_EXACT = 0
STV_PATH_INT8 = 1
PATHS = {"exact": STV_PATH_EXACT, "int8": STV_PATH_INT8}

STV_MAX_SEQS = 64
HEAD_DIM = 256
GROUP = 32
PAGE_TOKENS = 256
HEAD_BLOCK_BYTES = 57344
GROUP_INT4 = 256                # the int4 per-token-head cache (include/stv.h)
HEAD_BLOCK_BYTES_INT4 = 66560

# Every symbol include/stv.h declares.
EXPORTS = (
    "stv_status_string", "stv_version", "stv_page_bytes", "stv_kv_append_pack", "stv_verify_workspace_bytes",
    "stv_verify_attn", "stv_split_combine", "stv_tree_accept", "stv_kv_commit", "stv_int8_qk_dots",
    "stv_verify_attn_no_alloc", "stv_append_verify_attn", "stv_lookup_workspace_bytes", "stv_lookup_draft",
    "stv_prefill_workspace_bytes", "stv_prefill_attn", "stv_verify_attn_timeout_test",
    "stv_prefill_attn_timeout_test", "stv_append_verify_combine",
)


class StvError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {status_string(status)} ({status})")


class stv_shape(ctypes.Structure):
    _fields_ = [("hq", ctypes.c_int32), ("hkv", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("group", ctypes.c_int32), ("page_tokens", ctypes.c_int32), ("kv_format", ctypes.c_int32)]


class stv_layer_cache(ctypes.Structure):
    _fields_ = [("pool", ctypes.c_void_p), ("page_bytes", ctypes.c_int64), ("n_pages", ctypes.c_int32)]


class stv_history(ctypes.Structure):
    _fields_ = [("tokens", ctypes.c_void_p), ("n", ctypes.c_int64)]


class stv_seq(ctypes.Structure):
    _fields_ = [("page_table", ctypes.c_void_p), ("n_pages", ctypes.c_int32), ("ctx", ctypes.c_int32)]


_lib = None


def load() -> ctypes.CDLL:
    """Load libstv.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m speculative_tree_verify_bit_gb300.build` (no fallback exists)")
        lib = ctypes.CDLL(LIB_PATH)
        P, I, I32, I64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int32, ctypes.c_int64
        lib.stv_status_string.restype = ctypes.c_char_p
        lib.stv_status_string.argtypes = [I]
        lib.stv_version.restype = I
        lib.stv_page_bytes.restype = I
        lib.stv_page_bytes.argtypes = [P, P]
        lib.stv_kv_append_pack.restype = I
        lib.stv_kv_append_pack.argtypes = [P, P, P, I, P, P, P, P, I, P, P]
        lib.stv_verify_workspace_bytes.restype = I
        lib.stv_verify_workspace_bytes.argtypes = [P, P, I, I, I, P]
        lib.stv_verify_attn.restype = I
        lib.stv_verify_attn.argtypes = [P, P, P, I, P, P, I, I, P, ctypes.c_size_t, P, P]
        lib.stv_split_combine.restype = I
        lib.stv_split_combine.argtypes = [P, P, I, I, P, ctypes.c_size_t, P, P]
        lib.stv_tree_accept.restype = I
        lib.stv_tree_accept.argtypes = [P, P, P, I, I, P, P, P, P, P]
        lib.stv_kv_commit.restype = I
        lib.stv_kv_commit.argtypes = [P, P, I, P, I, I, P, P, P, P, P]
        lib.stv_int8_qk_dots.restype = I
        lib.stv_int8_qk_dots.argtypes = [P, P, P, P, P, I, P, ctypes.c_size_t, P, P, P]
        lib.stv_prefill_workspace_bytes.restype = I
        lib.stv_prefill_workspace_bytes.argtypes = [P, P, I, P]
        lib.stv_prefill_attn.restype = I
        lib.stv_prefill_attn.argtypes = [P, P, P, P, I, I, P, ctypes.c_size_t, P, P, P]
        lib.stv_lookup_workspace_bytes.restype = I
        lib.stv_lookup_workspace_bytes.argtypes = [I, P]
        lib.stv_lookup_draft.restype = I
        lib.stv_lookup_draft.argtypes = [P, I, I, I, I, P, P, P, P, P, ctypes.c_size_t, P]
        lib.stv_append_verify_attn.restype = I
        lib.stv_append_verify_attn.argtypes = [P, P, P, I, P, P, P, P, I, I, P, ctypes.c_size_t, P, P]
        lib.stv_append_verify_combine.restype = I
        lib.stv_append_verify_combine.argtypes = [P, P, P, I, P, P, P, P, I, I, P, ctypes.c_size_t, P, P, P]
        lib.stv_verify_attn_no_alloc.restype = I
        lib.stv_verify_attn_no_alloc.argtypes = [P, P, P, I, P, P, I, I, P, P, P]
        lib.stv_verify_attn_timeout_test.restype = I
        lib.stv_verify_attn_timeout_test.argtypes = [P, P, P, I, P, P, I, I, P, ctypes.c_size_t, P, P]
        _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load().stv_status_string(int(status)).decode()


def _check(fn: str, rc: int):
    if rc != STV_OK:
        raise StvError(fn, rc)


# --------------------------------------------------------------------------
# marshalling helpers
# --------------------------------------------------------------------------

def _ptr(t, dtype=None, name="tensor"):
    if t is None:
        return None
    import torch

    if not isinstance(t, torch.Tensor) or t.device.type != "cuda":
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def make_shape(hq: int = 24, hkv: int = 4, group: int = GROUP, kv_format: int = STV_KV_BY_GROUP) -> stv_shape:
    """group 32: the 3-bit cache; group 256 (GROUP_INT4): the int4
    per-token-head cache; kv_format STV_KV_K4V2 (group 32): the K 4 / V 2-bit
    cache (include/stv.h)."""
    return stv_shape(hq, hkv, HEAD_DIM, group, PAGE_TOKENS, kv_format)


def head_block_bytes(group: int = GROUP) -> int:
    return HEAD_BLOCK_BYTES_INT4 if group == GROUP_INT4 else HEAD_BLOCK_BYTES


class LayerCache:
    """One layer's paged pool: a uint8 CUDA tensor of n_pages * page_bytes."""

    def __init__(self, pool, hkv: int, group: int = GROUP):
        import torch

        self.hkv = hkv
        self.group = group
        self.page_bytes = hkv * head_block_bytes(group)
        assert pool.dtype == torch.uint8 and pool.numel() % self.page_bytes == 0
        self.pool = pool
        self.n_pages = pool.numel() // self.page_bytes

    @classmethod
    def empty(cls, n_pages: int, hkv: int = 4, device="cuda", group: int = GROUP):
        import torch

        return cls(torch.zeros(n_pages * hkv * head_block_bytes(group), dtype=torch.uint8, device=device), hkv, group)

    def c(self) -> stv_layer_cache:
        return stv_layer_cache(_ptr(self.pool, name="pool").value, self.page_bytes, self.n_pages)


class Seq:
    """A sequence: its device page table (int32) and its context length."""

    def __init__(self, page_table, ctx: int):
        self.page_table = page_table
        self.ctx = int(ctx)

    def c(self) -> stv_seq:
        import torch

        return stv_seq(_ptr(self.page_table, torch.int32, "page_table").value, self.page_table.numel(), self.ctx)


def _seq_array(seqs):
    arr = (stv_seq * len(seqs))()
    for i, s in enumerate(seqs):
        arr[i] = s.c()
    return arr


# --------------------------------------------------------------------------
# entry points (same names as include/stv.h)
# --------------------------------------------------------------------------

def stv_version() -> int:
    return load().stv_version()


def stv_page_bytes(shape: stv_shape) -> int:
    out = ctypes.c_int64()
    _check("stv_page_bytes", load().stv_page_bytes(ctypes.byref(shape), ctypes.byref(out)))
    return out.value


def stv_kv_append_pack(shape, layer: LayerCache, seqs, k, v, row_seq, row_pos, dev_status=None, stream=None):
    import torch

    lc = layer.c()
    arr = _seq_array(seqs)
    _check("stv_kv_append_pack", load().stv_kv_append_pack(
        ctypes.byref(shape), ctypes.byref(lc), arr, len(seqs), _ptr(k, torch.float16, "k"), _ptr(v, torch.float16, "v"),
        _ptr(row_seq, torch.int32, "row_seq"), _ptr(row_pos, torch.int32, "row_pos"), row_seq.numel(),
        _ptr(dev_status, torch.int32, "dev_status"), _stream(stream)))


def stv_verify_workspace_bytes(shape, seqs, t_nodes: int, sm_count: int = 0) -> int:
    out = ctypes.c_size_t()
    arr = _seq_array(seqs)
    _check("stv_verify_workspace_bytes", load().stv_verify_workspace_bytes(
        ctypes.byref(shape), arr, len(seqs), int(t_nodes), int(sm_count), ctypes.byref(out)))
    return out.value


def stv_verify_attn(shape, layer: LayerCache, seqs, q, parent, t_nodes: int, path, workspace, dev_status=None,
                    stream=None):
    import torch

    lc = layer.c()
    arr = _seq_array(seqs)
    path = PATHS.get(path, path)
    _check("stv_verify_attn", load().stv_verify_attn(
        ctypes.byref(shape), ctypes.byref(lc), arr, len(seqs), _ptr(q, torch.float16, "q"),
        _ptr(parent, torch.int32, "parent"), int(t_nodes), int(path), _ptr(workspace, name="workspace"),
        workspace.numel() * workspace.element_size(), _ptr(dev_status, torch.int32, "dev_status"), _stream(stream)))


def stv_append_verify_attn(shape, layer: LayerCache, seqs, k_tree, v_tree, q, parent, t_nodes: int, path, workspace,
                           dev_status=None, stream=None):
    """stv_kv_append_pack of the round's tree rows (k_tree, v_tree: fp16
    [n_seqs][T][hkv][256], row i of sequence s at ctx_s + i) fused into
    stv_verify_attn: one launch.  The workspace must be zero-filled before
    its first use here (arrival counters of the exact path's packing warp);
    each completed call leaves them zero."""
    import torch

    lc = layer.c()
    arr = _seq_array(seqs)
    path = PATHS.get(path, path)
    _check("stv_append_verify_attn", load().stv_append_verify_attn(
        ctypes.byref(shape), ctypes.byref(lc), arr, len(seqs), _ptr(k_tree, torch.float16, "k_tree"),
        _ptr(v_tree, torch.float16, "v_tree"), _ptr(q, torch.float16, "q"), _ptr(parent, torch.int32, "parent"),
        int(t_nodes), int(path), _ptr(workspace, name="workspace"), workspace.numel() * workspace.element_size(),
        _ptr(dev_status, torch.int32, "dev_status"), _stream(stream)))


def stv_append_verify_combine(shape, layer: LayerCache, seqs, k_tree, v_tree, q, parent, t_nodes: int, path,
                              workspace, o, dev_status=None, stream=None):
    """stv_kv_append_pack of the round's tree rows + stv_verify_attn +
    stv_split_combine in one cooperative launch.  The workspace (the size
    stv_verify_workspace_bytes gives) must be zero-filled before its first
    use here; each completed call leaves its counters zero."""
    import torch

    lc = layer.c()
    arr = _seq_array(seqs)
    path = PATHS.get(path, path)
    _check("stv_append_verify_combine", load().stv_append_verify_combine(
        ctypes.byref(shape), ctypes.byref(lc), arr, len(seqs), _ptr(k_tree, torch.float16, "k_tree"),
        _ptr(v_tree, torch.float16, "v_tree"), _ptr(q, torch.float16, "q"), _ptr(parent, torch.int32, "parent"),
        int(t_nodes), int(path), _ptr(workspace, name="workspace"), workspace.numel() * workspace.element_size(),
        _ptr(o, torch.float16, "o"), _ptr(dev_status, torch.int32, "dev_status"), _stream(stream)))


def stv_split_combine(shape, seqs, t_nodes: int, workspace, o, stream=None):
    import torch

    arr = _seq_array(seqs)
    _check("stv_split_combine", load().stv_split_combine(
        ctypes.byref(shape), arr, len(seqs), int(t_nodes), _ptr(workspace, name="workspace"),
        workspace.numel() * workspace.element_size(), _ptr(o, torch.float16, "o"), _stream(stream)))


def stv_tree_accept(parent, draft_ids, target_argmax, n_commit, path, out_ids, dev_status=None, stream=None):
    import torch

    n_seqs, t = parent.shape
    _check("stv_tree_accept", load().stv_tree_accept(
        _ptr(parent, torch.int32, "parent"), _ptr(draft_ids, torch.int32, "draft_ids"),
        _ptr(target_argmax, torch.int32, "target_argmax"), int(t), int(n_seqs), _ptr(n_commit, torch.int32, "n_commit"),
        _ptr(path, torch.int32, "path"), _ptr(out_ids, torch.int32, "out_ids"),
        _ptr(dev_status, torch.int32, "dev_status"), _stream(stream)))


def stv_kv_commit(shape, layers, seqs, t_nodes: int, n_commit, path, ctx_dev=None, dev_status=None, stream=None):
    import torch

    larr = (stv_layer_cache * len(layers))()
    for i, l in enumerate(layers):
        larr[i] = l.c()
    arr = _seq_array(seqs)
    _check("stv_kv_commit", load().stv_kv_commit(
        ctypes.byref(shape), larr, len(layers), arr, len(seqs), int(t_nodes), _ptr(n_commit, torch.int32, "n_commit"),
        _ptr(path, torch.int32, "path"), _ptr(ctx_dev, torch.int32, "ctx_dev"),
        _ptr(dev_status, torch.int32, "dev_status"), _stream(stream)))


def stv_int8_qk_dots(shape, layer: LayerCache, seq: Seq, q, parent, t_nodes: int, workspace, dots, dev_status=None,
                     stream=None):
    """The int8 verify of one sequence, also writing the kernel's own
    per-group integer dots: dots int32 [hkv][T*G][ctx+T][8]."""
    import torch

    lc = layer.c()
    arr = _seq_array([seq])
    _check("stv_int8_qk_dots", load().stv_int8_qk_dots(
        ctypes.byref(shape), ctypes.byref(lc), arr, _ptr(q, torch.float16, "q"), _ptr(parent, torch.int32, "parent"),
        int(t_nodes), _ptr(workspace, name="workspace"), workspace.numel() * workspace.element_size(),
        _ptr(dots, torch.int32, "dots"), _ptr(dev_status, torch.int32, "dev_status"), _stream(stream)))


def stv_verify_attn_timeout_test(shape, layer: LayerCache, seqs, q, parent, t_nodes: int, path, workspace,
                                 dev_status=None, stream=None):
    """stv_verify_attn with the kernel's copies withheld: every wait runs out
    and the kernel reports STV_DEV_TIMEOUT (failure-path test)."""
    import torch

    lc = layer.c()
    arr = _seq_array(seqs)
    path = PATHS.get(path, path)
    _check("stv_verify_attn_timeout_test", load().stv_verify_attn_timeout_test(
        ctypes.byref(shape), ctypes.byref(lc), arr, len(seqs), _ptr(q, torch.float16, "q"),
        _ptr(parent, torch.int32, "parent"), int(t_nodes), int(path), _ptr(workspace, name="workspace"),
        workspace.numel() * workspace.element_size(), _ptr(dev_status, torch.int32, "dev_status"), _stream(stream)))


def stv_verify_attn_no_alloc(shape, layer: LayerCache, seqs, q, parent, t_nodes: int, path, o, dev_status=None,
                             stream=None):
    """Verify attention + split merge with the library's own fixed scratch
    (for callers that cannot allocate device memory; see include/stv.h)."""
    import torch

    lc = layer.c()
    arr = _seq_array(seqs)
    path = PATHS.get(path, path)
    _check("stv_verify_attn_no_alloc", load().stv_verify_attn_no_alloc(
        ctypes.byref(shape), ctypes.byref(lc), arr, len(seqs), _ptr(q, torch.float16, "q"),
        _ptr(parent, torch.int32, "parent"), int(t_nodes), int(path), _ptr(o, torch.float16, "o"),
        _ptr(dev_status, torch.int32, "dev_status"), _stream(stream)))


def stv_lookup_workspace_bytes(n_seqs: int) -> int:
    out = ctypes.c_size_t()
    _check("stv_lookup_workspace_bytes", load().stv_lookup_workspace_bytes(int(n_seqs), ctypes.byref(out)))
    return out.value


def stv_lookup_draft(histories, min_len: int, max_len: int, k: int, n_prop, prop, match_len, match_pos, workspace,
                     stream=None):
    """Lookup drafting over each history (int32 CUDA tensors): the up to k
    tokens that followed the latest earlier occurrence of the longest suffix
    of length max_len .. min_len (include/stv.h).  The workspace must be zero
    before its first use; each call leaves it zero."""
    import torch

    arr = (stv_history * len(histories))()
    for i, t in enumerate(histories):
        arr[i].tokens = _ptr(t, torch.int32, "history").value if t.numel() else None
        arr[i].n = t.numel()
    _check("stv_lookup_draft", load().stv_lookup_draft(
        arr, len(histories), int(min_len), int(max_len), int(k), _ptr(n_prop, torch.int32, "n_prop"),
        _ptr(prop, torch.int32, "prop"), _ptr(match_len, torch.int32, "match_len"),
        _ptr(match_pos, torch.int64, "match_pos"), _ptr(workspace, name="workspace"),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def stv_prefill_workspace_bytes(shape, seq, n_tokens: int) -> int:
    arr = _seq_array([seq])
    out = ctypes.c_size_t()
    _check("stv_prefill_workspace_bytes", load().stv_prefill_workspace_bytes(
        ctypes.byref(shape), arr, int(n_tokens), ctypes.byref(out)))
    return out.value


def stv_prefill_attn(shape, layer: LayerCache, seq, q, n_tokens: int, path, workspace, o, dev_status=None,
                     stream=None):
    """Prefill attention over the 3-bit cache (include/stv.h): q and o are
    fp16 [n_tokens][hq][256]; the prompt's rows are already in the cache at
    seq.ctx .. seq.ctx + n_tokens - 1."""
    import torch

    lc = layer.c()
    arr = _seq_array([seq])
    path = PATHS.get(path, path)
    _check("stv_prefill_attn", load().stv_prefill_attn(
        ctypes.byref(shape), ctypes.byref(lc), arr, _ptr(q, torch.float16, "q"), int(n_tokens), int(path),
        _ptr(workspace, name="workspace"), workspace.numel() * workspace.element_size(),
        _ptr(o, torch.float16, "o"), _ptr(dev_status, torch.int32, "dev_status"), _stream(stream)))


def stv_prefill_attn_timeout_test(shape, layer: LayerCache, seq, q, n_tokens: int, path, workspace, o,
                                  dev_status=None, stream=None):
    """stv_prefill_attn with the persistent kernel's copies withheld: every
    wait runs out and the kernel reports STV_DEV_TIMEOUT (failure-path test)."""
    import torch

    lc = layer.c()
    arr = _seq_array([seq])
    path = PATHS.get(path, path)
    _check("stv_prefill_attn_timeout_test", load().stv_prefill_attn_timeout_test(
        ctypes.byref(shape), ctypes.byref(lc), arr, _ptr(q, torch.float16, "q"), int(n_tokens), int(path),
        _ptr(workspace, name="workspace"), workspace.numel() * workspace.element_size(),
        _ptr(o, torch.float16, "o"), _ptr(dev_status, torch.int32, "dev_status"), _stream(stream)))
