"""stv_append_verify_attn: the round's tree-row append fused into the verify
launch.  It must leave the cache byte for byte as stv_kv_append_pack of the
same rows would, and give exactly the output of the separate append + verify
(and so the oracle's, within the attention tolerance).

Sources: "elpis" README, "Why fast" (tree verify pipe: host check after the
launch); syv-ai README (mirror), CUDA graph notes (an uncaptured verify step
is launch-bound)."""
import numpy as np
import pytest
import torch

import speculative_tree_verify_bit_gb300 as stv
import workloads
from roundkit import Round, assert_attention_close, gather_heads, head_rows

pytestmark = pytest.mark.gpu


def context_only_cache(r: Round):
    """The round's cache with the context rows packed and the tree rows not."""
    dev = r.device
    layer = stv.LayerCache.empty(r.pool_pages, r.hkv, device=dev)
    r.seqs = [stv.Seq(torch.as_tensor(t, device=dev), c) for t, c in zip(r.tables, r.ctx)]
    ctx_rows = np.nonzero(r.row_pos < np.repeat(np.array(r.ctx), [c + r.T for c in r.ctx]))[0]
    if len(ctx_rows):
        idx = torch.as_tensor(ctx_rows, device=dev)
        stv.stv_kv_append_pack(r.shape, layer, r.seqs, r.k[idx].contiguous(), r.v[idx].contiguous(),
                               torch.as_tensor(r.row_seq[ctx_rows], device=dev),
                               torch.as_tensor(r.row_pos[ctx_rows], device=dev))
    return layer


def tree_rows(r: Round):
    """k, v of the tree rows as [n_seqs][T][hkv][256]."""
    tree = np.nonzero(r.row_pos >= np.repeat(np.array(r.ctx), [c + r.T for c in r.ctx]))[0]
    idx = torch.as_tensor(tree, device=r.device)
    shape = (r.n_seqs, r.T, r.hkv, 256)
    return r.k[idx].reshape(shape).contiguous(), r.v[idx].reshape(shape).contiguous()


def fused_verify(r: Round, layer, path):
    kt, vt = tree_rows(r)
    ws = torch.zeros(stv.stv_verify_workspace_bytes(r.shape, r.seqs, r.T), dtype=torch.uint8, device=r.device)
    o = torch.empty((r.n_seqs, r.T, r.hq, 256), dtype=torch.float16, device=r.device)
    status = torch.zeros(1, dtype=torch.int32, device=r.device)
    stv.stv_append_verify_attn(r.shape, layer, r.seqs, kt, vt, r.q, torch.as_tensor(r.parent, device=r.device), r.T,
                               path, ws, dev_status=status)
    stv.stv_split_combine(r.shape, r.seqs, r.T, ws, o)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return o


@pytest.mark.parametrize("path", ["exact", "int8"])
@pytest.mark.parametrize("ctx,t,hq", [
    ([1024], 16, 24),                 # tree rows open a fresh 64-key tile
    ([0], 16, 24),                    # tree rows only
    ([60], 16, 24),                   # tree rows straddle a tile and a split boundary
    ([250], 16, 24),                  # tree rows straddle a page boundary
    ([300, 0, 1000, 2047], 7, 24),    # ragged batch
    ([8192], 8, 24),                  # chain-sized round
    ([511], 32, 16),                  # T = 32 (128 rows per KV head)
])
def test_fused_append_equals_separate_append(gpu, path, ctx, t, hq):
    r = Round(ctx, t, seed=7100 + sum(ctx) + t, hq=hq)
    want_layer = r.gpu_cache()                 # every row appended by stv_kv_append_pack
    want = r.gpu_verify(path, want_layer)
    layer = context_only_cache(r)
    got = fused_verify(r, layer, path)
    assert np.array_equal(layer.pool.cpu().numpy(), want_layer.pool.cpu().numpy())
    assert torch.equal(got, want)
    r.oracle_cache()
    assert_attention_close(got.float().cpu().numpy(), r.oracle_attention(path), f"fused {ctx}/{t}/{path}")


def test_fused_append_full_size_long_context(gpu):
    """262,144-token context, one layer, the benchmark's launch configuration:
    cache bytes and output identical to the separate path; sampled heads
    against the oracle."""
    w = workloads.WORKLOADS["long262k"]
    r = Round(list(w.ctx), w.t_nodes, seed=workloads.layer_seed(w, 0))
    want_layer = r.gpu_cache()
    outs = {}
    for path in ("exact", "int8"):
        want = r.gpu_verify(path, want_layer)
        layer = context_only_cache(r)
        outs[path] = fused_verify(r, layer, path)
        assert np.array_equal(layer.pool.cpu().numpy(), want_layer.pool.cpu().numpy())
        assert torch.equal(outs[path], want)
        del layer
    r.oracle_cache()
    heads = (0, 23)
    for path in ("exact", "int8"):
        want = r.oracle_attention(path, rows=head_rows((0,), heads, r.T)).reshape(-1, r.T, 256)
        got = gather_heads(outs[path].float().cpu().numpy(), (0,), heads, r.T)
        assert_attention_close(got, want, f"fused 262K {path}")


def test_fused_append_rejects_missing_rows(gpu):
    r = Round([100], 4, seed=71)
    layer = context_only_cache(r)
    ws = torch.zeros(stv.stv_verify_workspace_bytes(r.shape, r.seqs, 4), dtype=torch.uint8, device=gpu)
    kt, _ = tree_rows(r)
    with pytest.raises(stv.StvError) as e:
        stv.stv_append_verify_attn(r.shape, layer, r.seqs, kt, None, r.q, torch.as_tensor(r.parent, device=gpu), 4,
                                   "exact", ws)
    assert e.value.status == stv.STV_ERR_INVALID_ARG
