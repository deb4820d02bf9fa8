"""stv_append_verify_combine: one layer of a verify round (append of the tree
rows, tree-masked split-KV attention, merge of the splits) in one cooperative
launch.  It must leave the cache byte for byte as stv_kv_append_pack of the
same rows would, give exactly the output of the three separate launches (and
so the oracle's, within the attention tolerance), and leave its workspace
counters zero for the next call.

Sources: "elpis" README, "Why fast" (tree verify pipe); Reddit posts
(u/iamMess), second post (split-KV verify attention, then a merge)."""
import numpy as np
import pytest
import torch

import speculative_tree_verify_bit_gb300 as stv
import workloads
from roundkit import Round, assert_attention_close, gather_heads, head_rows
from test_gpu_fused_append import context_only_cache, tree_rows

pytestmark = pytest.mark.gpu


def counter_bytes(r: Round) -> int:
    """Size of the counter block at the start of the workspace (256-aligned):
    2 + STV_MAX_SEQS * hkv words."""
    return -(-(2 + 64 * r.hkv) * 4 // 256) * 256


def fused_round(r: Round, layer, ws=None):
    kt, vt = tree_rows(r)
    if ws is None:
        ws = torch.zeros(stv.stv_verify_workspace_bytes(r.shape, r.seqs, r.T), dtype=torch.uint8, device=r.device)
    o = torch.empty((r.n_seqs, r.T, r.hq, 256), dtype=torch.float16, device=r.device)
    status = torch.zeros(1, dtype=torch.int32, device=r.device)
    stv.stv_append_verify_combine(r.shape, layer, r.seqs, kt, vt, r.q, torch.as_tensor(r.parent, device=r.device),
                                  r.T, "exact", ws, o, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert int(ws[:counter_bytes(r)].count_nonzero().item()) == 0, "counters not left zero"
    return o, ws


@pytest.mark.parametrize("ctx,t,hq", [
    ([1024], 16, 24),                 # tree rows open a fresh 64-key tile
    ([0], 16, 24),                    # tree rows only: every unit's first tile waits for the packing
    ([60], 16, 24),                   # tree rows straddle a tile and a split boundary
    ([250], 16, 24),                  # tree rows straddle a page boundary
    ([300, 0, 1000, 2047], 7, 24),    # ragged batch
    ([8192], 8, 24),                  # chain-sized round
    ([511], 32, 16),                  # T = 32 (128 rows per KV head)
    ([40000], 16, 24),                # 64-deep merge (more than 32 splits per head)
])
def test_fused_round_equals_three_launches(gpu, ctx, t, hq):
    r = Round(ctx, t, seed=7300 + sum(ctx) + t, hq=hq)
    want_layer = r.gpu_cache()
    want = r.gpu_verify("exact", want_layer)
    layer = context_only_cache(r)
    got, ws = fused_round(r, layer)
    assert np.array_equal(layer.pool.cpu().numpy(), want_layer.pool.cpu().numpy())
    assert torch.equal(got, want)
    # the same workspace again (its counters were reset by the first call)
    again, _ = fused_round(r, layer, ws)
    assert torch.equal(again, want)
    if sum(ctx) <= 10000:
        r.oracle_cache()
        assert_attention_close(got.float().cpu().numpy(), r.oracle_attention("exact"), f"fused round {ctx}/{t}")


def test_fused_round_eight_requests(gpu):
    """Eight requests, 1K..128K.  The one-launch layer plans one unit per SM;
    the separate launches plan more units than SMs for this batch (their
    persistent verify kernel), so the splits, and the last bits of the sums,
    differ: cache bytes equal, sampled heads against the oracle."""
    r = Round([1024 << i for i in range(8)], 16, seed=7390)
    want_layer = r.gpu_cache()
    layer = context_only_cache(r)
    got, _ = fused_round(r, layer)
    assert np.array_equal(layer.pool.cpu().numpy(), want_layer.pool.cpu().numpy())
    del layer, want_layer
    r.oracle_cache()
    seqs, heads = (0, 5, 7), (0, 23)
    want = r.oracle_attention("exact", rows=head_rows(seqs, heads, r.T)).reshape(-1, r.T, 256)
    assert_attention_close(gather_heads(got.float().cpu().numpy(), seqs, heads, r.T), want, "fused round ragged")


def test_fused_round_full_size_long_context(gpu):
    """262,144-token context, one layer: cache bytes and output identical to
    the three separate launches; sampled heads against the oracle."""
    w = workloads.WORKLOADS["long262k"]
    r = Round(list(w.ctx), w.t_nodes, seed=workloads.layer_seed(w, 0))
    want_layer = r.gpu_cache()
    want = r.gpu_verify("exact", want_layer)
    layer = context_only_cache(r)
    got, _ = fused_round(r, layer)
    assert np.array_equal(layer.pool.cpu().numpy(), want_layer.pool.cpu().numpy())
    assert torch.equal(got, want)
    del layer, want_layer
    r.oracle_cache()
    heads = (0, 23)
    want_o = r.oracle_attention("exact", rows=head_rows((0,), heads, r.T)).reshape(-1, r.T, 256)
    assert_attention_close(gather_heads(got.float().cpu().numpy(), (0,), heads, r.T), want_o, "fused round 262K")


def test_fused_round_in_a_cuda_graph(gpu):
    """Two layers' fused launches captured in one CUDA graph and replayed
    twice: the same output as the eager calls, counters zero after each."""
    rounds = [Round([5000 + 3000 * l], 16, seed=7400 + l) for l in range(2)]
    layers, wants, kts = [], [], []
    for r in rounds:
        want_layer = r.gpu_cache()
        wants.append(r.gpu_verify("exact", want_layer))
        layers.append(context_only_cache(r))
        kts.append(tree_rows(r))
    ws = torch.zeros(max(stv.stv_verify_workspace_bytes(r.shape, r.seqs, r.T) for r in rounds), dtype=torch.uint8,
                     device=gpu)
    outs = [torch.empty_like(w) for w in wants]
    parents = [torch.as_tensor(r.parent, device=gpu) for r in rounds]
    status = torch.zeros(1, dtype=torch.int32, device=gpu)
    stream = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            for r, layer, (kt, vt), par, o in zip(rounds, layers, kts, parents, outs):
                stv.stv_append_verify_combine(r.shape, layer, r.seqs, kt, vt, r.q, par, r.T, "exact", ws, o,
                                              dev_status=status, stream=stream)
    for _ in range(2):
        for o in outs:
            o.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert int(ws[:counter_bytes(rounds[0])].count_nonzero().item()) == 0
        for o, want in zip(outs, wants):
            assert torch.equal(o, want)


def test_fused_round_rejects(gpu):
    r = Round([100], 4, seed=73)
    layer = context_only_cache(r)
    ws = torch.zeros(stv.stv_verify_workspace_bytes(r.shape, r.seqs, 4), dtype=torch.uint8, device=gpu)
    kt, vt = tree_rows(r)
    o = torch.empty((1, 4, r.hq, 256), dtype=torch.float16, device=gpu)
    par = torch.as_tensor(r.parent, device=gpu)
    with pytest.raises(stv.StvError) as e:
        stv.stv_append_verify_combine(r.shape, layer, r.seqs, kt, vt, r.q, par, 4, "int8", ws, o)
    assert e.value.status == stv.STV_ERR_UNIMPLEMENTED
    with pytest.raises(stv.StvError) as e:
        stv.stv_append_verify_combine(r.shape, layer, r.seqs, kt, vt, r.q, par, 4, "exact", ws, None)
    assert e.value.status == stv.STV_ERR_INVALID_ARG
