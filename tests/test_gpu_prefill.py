"""stv_prefill_attn (prefill attention over the 3-bit cache) against the
oracle.  "elpis" README, "Why fast": prefill int8 Q.K^T (3021c), prefill K/V
double-buffered ring (3022).

The GPU splits the prompt into chain-tree chunks; the oracle side does not:
each sampled prompt token t is its own one-node sequence whose context is
ctx + t, so it sees exactly the cached tokens and the prompt tokens up to
itself.  Sampled tokens include every chunk boundary region, the boundary
between launches of the chunked path (64 chunks), the ragged tail and the
last chunks (the longest units, which the persistent exact-path kernel takes
first)."""
import numpy as np
import pytest
import torch

import oracle
import speculative_tree_verify_bit_gb300 as stv
import workloads
from roundkit import CPU_THREADS, assert_attention_close

pytestmark = pytest.mark.gpu


def prefill_case(ctx0, n, hq, hkv, seed):
    dev = "cuda"
    total = ctx0 + n
    pages = workloads.pages_needed(total, 0) + 1
    table = np.random.default_rng(seed).permutation(pages).astype(np.int32)
    k, v = workloads.kv_rows(seed + 1, total, hkv, device=dev)
    q = workloads.q_rows(seed + 2, 1, n, hq, device=dev)[0].contiguous()  # [n][hq][256]
    layer = stv.LayerCache.empty(pages, hkv, device=dev)
    seq = stv.Seq(torch.as_tensor(table, device=dev), ctx0)
    pos = np.arange(total, dtype=np.int32)
    shape = stv.make_shape(hq, hkv)
    stv.stv_kv_append_pack(shape, layer, [stv.Seq(seq.page_table, 0)], k.contiguous(), v.contiguous(),
                           torch.zeros(total, dtype=torch.int32, device=dev), torch.as_tensor(pos, device=dev))
    cache = oracle.Cache(hkv, pages)
    oracle.kv_append(cache, [table], k.cpu().numpy(), v.cpu().numpy(), np.zeros(total, np.int32), pos)
    return shape, layer, seq, q, table, cache


def gpu_prefill(shape, layer, seq, q, n, path):
    ws = torch.empty(stv.stv_prefill_workspace_bytes(shape, seq, n), dtype=torch.uint8, device="cuda")
    o = torch.full((n, shape.hq, 256), float("nan"), dtype=torch.float16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stv.stv_prefill_attn(shape, layer, seq, q, n, path, ws, o, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return o.float().cpu().numpy()


def sampled_tokens(n, c, rng):
    ts = {0, n - 1}
    for b in range(c, n, c):  # chunk boundaries: the last token of a chunk and the first of the next
        if b % (64 * c) == 0 or len(ts) < 24:
            ts.update({b - 1, b})
    ts.update(rng.integers(0, n, 8).tolist())
    ts.update(range(max(0, n - 2 * c - 1), n, max(1, c // 3)))  # the last two chunks
    return sorted(t for t in ts if 0 <= t < n)


@pytest.mark.parametrize("path", ["exact", "int8"])
@pytest.mark.parametrize("ctx0,n,hq,hkv", [
    (0, 1, 24, 4),          # a one-token prompt on an empty cache
    (300, 20, 24, 4),       # under one chunk (21 tokens at G = 6)
    (1000, 64, 24, 4),      # three chunks and a tail
    (0, 1400, 24, 4),       # 66 chunks: two launches (64 chunks each at most) and a tail
    (5000, 500, 8, 4),      # G = 2: chunks of 32 tokens
])
def test_prefill_matches_per_token_oracle(gpu, path, ctx0, n, hq, hkv):
    check_prefill(path, ctx0, n, hq, hkv)


@pytest.mark.parametrize("ctx0,n,hq,hkv", [
    (700, 3000, 24, 4),     # 143 chunks x 4 heads = 572 units: several per CTA; tail of 18 tokens
    (0, 2048, 32, 4),       # G = 8: chunks of 16 tokens, 128 rows
    (64, 1100, 24, 1),      # one KV head, G = 24: chunks of 5 tokens (120 rows)
    (255, 97, 8, 4),        # G = 2: three full chunks of 32 and one token
])
def test_prefill_persistent_exact_path(gpu, ctx0, n, hq, hkv):
    """The exact path's persistent kernel over many (chunk, KV head) units."""
    check_prefill("exact", ctx0, n, hq, hkv)


def check_prefill(path, ctx0, n, hq, hkv):
    seed = 9100 + ctx0 + n + hq
    shape, layer, seq, q, table, cache = prefill_case(ctx0, n, hq, hkv, seed)
    got = gpu_prefill(shape, layer, seq, q, n, path)
    assert np.all(np.isfinite(got))
    c = min(32, 128 // (hq // hkv))
    ts = sampled_tokens(n, c, np.random.default_rng(seed))
    heads = (0, hq - 1)
    qn = q.cpu().numpy()
    want = oracle.attention(cache, [table] * len(ts), [ctx0 + t for t in ts], qn[ts][:, None],
                            -np.ones((len(ts), 1), np.int32), hq, path,
                            rows=[(i, 0, h) for h in heads for i in range(len(ts))], n_threads=CPU_THREADS)
    want = np.asarray(want).reshape(len(heads), len(ts), 256)
    got_rows = np.stack([got[ts, h] for h in heads])
    assert_attention_close(got_rows, want, f"prefill ctx0={ctx0} n={n} {path}")


def test_prefill_reports_bad_page(gpu):
    """A page-table entry outside the pool: the kernel reads a valid page in
    its place, finishes, and reports STV_DEV_BAD_PAGE."""
    shape, layer, seq, q, table, cache = prefill_case(300, 200, 24, 4, 17)
    bad = seq.page_table.clone()
    bad[0] = layer.n_pages + 5
    ws = torch.empty(stv.stv_prefill_workspace_bytes(shape, seq, 200), dtype=torch.uint8, device="cuda")
    o = torch.empty((200, 24, 256), dtype=torch.float16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stv.stv_prefill_attn(shape, layer, stv.Seq(bad, 300), q, 200, "exact", ws, o, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & stv.STV_DEV_BAD_PAGE
    # the context is still usable
    assert np.all(np.isfinite(gpu_prefill(shape, layer, seq, q, 200, "exact")))


def test_prefill_timeout_reported_and_context_usable(gpu):
    """Failure detection without a GPU fault: the persistent prefill kernel
    with its copies withheld (stv_prefill_attn_timeout_test) has every
    consumer's wait run out; the launch returns within seconds with
    STV_DEV_TIMEOUT, and a normal prefill right after it matches the oracle.
    The int8 path, which runs the chunked verify launches, refuses it."""
    import time

    shape, layer, seq, q, table, cache = prefill_case(200, 300, 24, 4, 23)
    ws = torch.empty(stv.stv_prefill_workspace_bytes(shape, seq, 300), dtype=torch.uint8, device="cuda")
    o = torch.empty((300, 24, 256), dtype=torch.float16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.monotonic()
    stv.stv_prefill_attn_timeout_test(shape, layer, seq, q, 300, "exact", ws, o, dev_status=status)
    torch.cuda.synchronize()
    assert time.monotonic() - t0 < 30.0
    assert int(status.item()) & stv.STV_DEV_TIMEOUT
    with pytest.raises(stv.StvError) as e:
        stv.stv_prefill_attn_timeout_test(shape, layer, seq, q, 300, "int8", ws, o)
    assert e.value.status == stv.STV_ERR_UNIMPLEMENTED
    check_prefill("exact", 200, 300, 24, 4)


def test_prefill_deterministic_and_rejects_bad_args(gpu):
    shape, layer, seq, q, table, cache = prefill_case(100, 50, 24, 4, 9)
    a = gpu_prefill(shape, layer, seq, q, 50, "exact")
    b = gpu_prefill(shape, layer, seq, q, 50, "exact")
    assert np.array_equal(a, b)
    with pytest.raises(stv.StvError) as e:
        stv.stv_prefill_workspace_bytes(shape, seq, 0)
    assert e.value.status == stv.STV_ERR_INVALID_ARG
    far = stv.Seq(seq.page_table, 100 + 10_000)  # prompt past the sequence's pages
    with pytest.raises(stv.StvError):
        stv.stv_prefill_workspace_bytes(shape, far, 50)
