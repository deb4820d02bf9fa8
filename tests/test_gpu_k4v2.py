"""The KVarN-style 4/2-bit cache (STV_KV_K4V2; next row f3) on the GPU against
the oracle: append and commit bytes bit-exact, exact-path verify within the
attention tolerance (the verify pipeline of the 3-bit cache with a 4-bit K
and a 2-bit V unpack), prefill, and the entry points that refuse this format.
Sources: Reddit posts (u/iamMess), "Now added" list (KVarN 4/2-bit KV cache);
syv-ai README (mirror), DFlash2 at 240k (CTX=huge); the quantizer and layout
are the readings stated in include/stv.h."""
import numpy as np
import pytest
import torch

import oracle
import speculative_tree_verify_bit_gb300 as stv
import workloads
from roundkit import CPU_THREADS, Round, assert_attention_close, gather_heads, head_rows

pytestmark = pytest.mark.gpu
KV2 = "k4v2"


def shape(hq=24, hkv=4):
    return stv.make_shape(hq, hkv, stv.GROUP, stv.STV_KV_K4V2)


@pytest.mark.parametrize("ctx,t", [([1024], 16), ([0, 250, 777], 5), ([63, 64, 65], 32)])
def test_append_bytes_bit_exact(gpu, ctx, t):
    r = Round(ctx, t, seed=6000 + sum(ctx) + t, hq=16 if t > 16 else 24, hkv=4, kind=KV2)
    layer = r.gpu_cache()
    assert np.array_equal(layer.pool.cpu().numpy(), r.oracle_cache().pool)


@pytest.mark.parametrize("m", [8.0, 2.0, 0.37, 1000.0, 65504.0, 5e-5, 10 * 2.0 ** -24])
def test_append_quantizer_every_fp16_value(gpu, m):
    """Every finite fp16 value in [-m, m], in groups of 32 channels whose
    maximum is m (the group's first channel), as K (4 bits) and, negated, as
    V (2 bits), one KV head: bytes equal the oracle's."""
    h = np.arange(65536, dtype=np.uint16).view(np.float16)
    vals = h[np.isfinite(h) & (np.abs(h.astype(np.float64)) <= np.float16(m))]
    per_row = 8 * 31
    n_rows = -(-len(vals) // per_row)
    rows = np.zeros((n_rows, 8, 32), np.float16)
    rows[:, :, 0] = np.float16(m)
    flat = rows[:, :, 1:].reshape(-1)
    flat[:len(vals)] = vals
    rows[:, :, 1:] = flat.reshape(n_rows, 8, 31)
    rows = rows.reshape(n_rows, 1, 256)
    vrows = (-rows).copy()
    pages = -(-n_rows // 256)
    table = np.arange(pages, dtype=np.int32)
    pos = np.arange(n_rows, dtype=np.int32)
    layer = stv.LayerCache.empty(pages, 1, device=gpu)
    stv.stv_kv_append_pack(shape(1, 1), layer, [stv.Seq(torch.as_tensor(table, device=gpu), 0)],
                           torch.as_tensor(rows, device=gpu), torch.as_tensor(vrows, device=gpu),
                           torch.zeros(n_rows, dtype=torch.int32, device=gpu), torch.as_tensor(pos, device=gpu))
    cache = oracle.Cache(1, pages, kind=KV2)
    oracle.kv_append(cache, [table], rows, vrows, np.zeros(n_rows, np.int32), pos)
    assert np.array_equal(layer.pool.cpu().numpy(), cache.pool)


@pytest.mark.parametrize("ctx,t,hq,hkv", [
    ([1024], 16, 24, 4),
    ([0], 16, 24, 4),
    ([300, 0, 1000], 7, 24, 4),
    ([511], 32, 16, 4),
    ([2000], 16, 8, 1),
])
def test_verify_matches_oracle(gpu, ctx, t, hq, hkv):
    r = Round(ctx, t, seed=6200 + t + sum(ctx), hq=hq, hkv=hkv, kind=KV2)
    r.gpu_cache()
    r.oracle_cache()
    assert_attention_close(r.gpu_verify("exact").float().cpu().numpy(), r.oracle_attention("exact"),
                           f"k4v2 {ctx}/{t}")


def test_verify_full_size_long_context(gpu):
    """262,144-token context, one layer, exact path: whole sampled heads."""
    w = workloads.WORKLOADS["long262k"]
    r = Round(list(w.ctx), w.t_nodes, seed=workloads.layer_seed(w, 0), kind=KV2)
    r.gpu_cache()
    r.oracle_cache()
    got = r.gpu_verify("exact").float().cpu().numpy()
    heads = (0, 11, 23)
    want = r.oracle_attention("exact", rows=head_rows((0,), heads, r.T)).reshape(-1, r.T, 256)
    assert_attention_close(gather_heads(got, (0,), heads, r.T), want, "k4v2 262K")


@pytest.mark.parametrize("ctx", [[1024], [250, 13, 4000]])
def test_commit_bytes_bit_exact(gpu, ctx):
    t = 16
    r = Round(ctx, t, seed=6400 + sum(ctx), p_accept=0.8, kind=KV2)
    layer = r.gpu_cache()
    cache = r.oracle_cache()
    P = lambda a: torch.as_tensor(np.ascontiguousarray(a, np.int32), device=gpu)
    n = len(ctx)
    nc = torch.zeros(n, dtype=torch.int32, device=gpu)
    path = torch.zeros((n, t), dtype=torch.int32, device=gpu)
    out = torch.zeros((n, t), dtype=torch.int32, device=gpu)
    status = torch.zeros(1, dtype=torch.int32, device=gpu)
    stv.stv_tree_accept(P(r.parent), P(r.draft), P(r.argmax), nc, path, out, dev_status=status)
    stv.stv_kv_commit(r.shape, [layer], r.seqs, t, nc, path, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ncn, pathn = nc.cpu().numpy(), path.cpu().numpy()
    oracle.kv_commit(cache, r.tables, ctx, ncn, np.where(pathn >= 0, pathn, 0).astype(np.int32), t)
    assert np.array_equal(layer.pool.cpu().numpy(), cache.pool)


def test_prefill_on_k4v2_cache(gpu):
    ctx0, n, hq, hkv = 300, 100, 24, 4
    total = ctx0 + n
    pages = workloads.pages_needed(total, 0) + 1
    table = np.random.default_rng(4).permutation(pages).astype(np.int32)
    k, v = workloads.kv_rows(87, total, hkv, device=gpu)
    q = workloads.q_rows(88, 1, n, hq, device=gpu)[0].contiguous()
    sh = shape(hq, hkv)
    layer = stv.LayerCache.empty(pages, hkv, device=gpu)
    seq = stv.Seq(torch.as_tensor(table, device=gpu), ctx0)
    pos = np.arange(total, dtype=np.int32)
    stv.stv_kv_append_pack(sh, layer, [stv.Seq(seq.page_table, 0)], k.contiguous(), v.contiguous(),
                           torch.zeros(total, dtype=torch.int32, device=gpu), torch.as_tensor(pos, device=gpu))
    ws = torch.empty(stv.stv_prefill_workspace_bytes(sh, seq, n), dtype=torch.uint8, device=gpu)
    o = torch.empty((n, hq, 256), dtype=torch.float16, device=gpu)
    stv.stv_prefill_attn(sh, layer, seq, q, n, "exact", ws, o)
    torch.cuda.synchronize()
    cache = oracle.Cache(hkv, pages, kind=KV2)
    oracle.kv_append(cache, [table], k.cpu().numpy(), v.cpu().numpy(), np.zeros(total, np.int32), pos)
    ts = [0, 20, 21, 63, 99]
    heads = (0, 23)
    want = oracle.attention(cache, [table] * len(ts), [ctx0 + t for t in ts], q.cpu().numpy()[ts][:, None],
                            -np.ones((len(ts), 1), np.int32), hq, "exact",
                            rows=[(i, 0, h) for h in heads for i in range(len(ts))], n_threads=CPU_THREADS)
    got = o.float().cpu().numpy()
    assert_attention_close(np.stack([got[ts, h] for h in heads]), np.asarray(want).reshape(2, len(ts), 256),
                           "k4v2 prefill")


def test_refused_entry_points(gpu):
    r = Round([100], 4, seed=6600, kind=KV2)
    r.gpu_cache()
    ws = torch.empty(stv.stv_verify_workspace_bytes(r.shape, r.seqs, 4), dtype=torch.uint8, device=gpu)
    parent = torch.as_tensor(r.parent, device=gpu)
    with pytest.raises(stv.StvError) as e:
        stv.stv_verify_attn(r.shape, r.layer, r.seqs, r.q, parent, 4, "int8", ws)
    assert e.value.status == stv.STV_ERR_UNIMPLEMENTED
    kt = torch.zeros((1, 4, 4, 256), dtype=torch.float16, device=gpu)
    with pytest.raises(stv.StvError) as e:
        stv.stv_append_verify_attn(r.shape, r.layer, r.seqs, kt, kt, r.q, parent, 4, "exact", ws)
    assert e.value.status == stv.STV_ERR_UNIMPLEMENTED
    dots = torch.zeros((4, 24, 104, 8), dtype=torch.int32, device=gpu)
    with pytest.raises(stv.StvError) as e:
        stv.stv_int8_qk_dots(r.shape, r.layer, r.seqs[0], r.q, parent, 4, ws, dots)
    assert e.value.status == stv.STV_ERR_UNIMPLEMENTED
