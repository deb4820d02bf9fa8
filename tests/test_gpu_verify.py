"""a2..a5 verify_attn + split_combine on the GPU against the fp64 oracle.

Sources: "elpis" README, "Why fast" (8-row token tree verified in one pass;
decode verify with 3-bit K codes as exact int8); Reddit posts (u/iamMess),
second post (split-KV verify attention).  Tolerance per head (one sequence's
Q head over all T nodes): relative L2 <= 1e-3 and max abs <= 4e-3; int8 dots
bit-exact."""
import numpy as np
import pytest
import torch

import oracle
import speculative_tree_verify_bit_gb300 as stv
import workloads
from roundkit import Round, assert_attention_close, gather_heads, head_rows

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("path", ["exact", "int8"])
def test_tiny_workload_all_rows(gpu, path):
    """1 layer, context 1,024, 16-node tree of depth <= 8, 24/4 heads: every
    output row against the oracle."""
    w = workloads.WORKLOADS["tiny"]
    r = Round(list(w.ctx), w.t_nodes, seed=workloads.layer_seed(w, 0))
    r.gpu_cache()
    r.oracle_cache()
    got = r.gpu_verify(path).float().cpu().numpy()
    want = r.oracle_attention(path)
    assert_attention_close(got, want, f"tiny/{path}")


@pytest.mark.parametrize("path", ["exact", "int8"])
def test_chain_workload_all_rows_and_sequential_decode(gpu, path):
    """Context 8,192, an 8-node chain: all rows against the oracle, and each
    node against a one-row decode on the GPU at context ctx + i (the chain
    verify must equal eight sequential decode steps)."""
    w = workloads.WORKLOADS["chain"]
    r = Round(list(w.ctx), w.t_nodes, seed=workloads.layer_seed(w, 0), tree="chain")
    layer = r.gpu_cache()
    r.oracle_cache()
    got = r.gpu_verify(path).float().cpu().numpy()
    assert_attention_close(got, r.oracle_attention(path), f"chain/{path}")
    ctx = w.ctx[0]
    for i in range(w.t_nodes):
        seqs = [stv.Seq(r.seqs[0].page_table, ctx + i)]
        ws = torch.empty(stv.stv_verify_workspace_bytes(r.shape, seqs, 1), dtype=torch.uint8, device=gpu)
        o = torch.empty((1, 1, r.hq, 256), dtype=torch.float16, device=gpu)
        q = r.q[:, i:i + 1].contiguous()
        stv.stv_verify_attn(r.shape, layer, seqs, q, torch.tensor([[-1]], dtype=torch.int32, device=gpu), 1, path, ws)
        stv.stv_split_combine(r.shape, seqs, 1, ws, o)
        step = o.float().cpu().numpy()[0, 0]
        assert_attention_close(got[0, i][:, None, :], step[:, None, :], f"chain step {i}")
        # Both launches cut keys [0, 8200) and [0, 8193 + i) into the same
        # splits (129 tiles of 64 per KV head, 4 tiles per split, 132 work
        # units), and every row's arithmetic is its own: node i of the chain
        # equals the one-row decode bit for bit.
        assert np.array_equal(got[0, i], step), f"chain node {i} differs from its sequential decode"


@pytest.mark.parametrize("path", ["exact", "int8"])
@pytest.mark.parametrize("ctx,t,hq,hkv", [
    ([0], 16, 24, 4),                 # tree rows only
    ([1], 1, 24, 4),                  # one-row decode
    ([300, 0, 1000], 7, 24, 4),       # ragged batch, ragged tails
    ([511], 32, 16, 4),               # T = 32, 128 rows per KV head
    ([2000], 16, 8, 1),               # one KV head, G = 8
])
def test_edge_shapes(gpu, path, ctx, t, hq, hkv):
    r = Round(ctx, t, seed=4242 + t + sum(ctx), hq=hq, hkv=hkv)
    r.gpu_cache()
    r.oracle_cache()
    got = r.gpu_verify(path).float().cpu().numpy()
    assert_attention_close(got, r.oracle_attention(path), f"{ctx}/{t}/{path}")


def test_ragged_batch_small(gpu):
    """The ragged workload's structure (8 requests, contexts doubling from
    1K, one launch, shared pool with a random page assignment) at contexts
    1K..8K, three whole heads per request."""
    ctx = [1024 << (i % 4) for i in range(8)]
    r = Round(ctx, 16, seed=1004)
    r.gpu_cache()
    r.oracle_cache()
    got = r.gpu_verify("exact").float().cpu().numpy()
    seqs, heads = range(8), (0, 13, 23)
    want = r.oracle_attention("exact", rows=head_rows(seqs, heads, 16)).reshape(-1, 16, 256)
    assert_attention_close(gather_heads(got, seqs, heads, 16), want, "ragged-small")


@pytest.mark.parametrize("name", ["tree32k", "long262k", "ragged"])
def test_full_size_sampled_rows(gpu, name):
    """Full-size workloads, one layer, in the benchmark's launch configuration:
    whole sampled heads (all T nodes) against the oracle."""
    w = workloads.WORKLOADS[name]
    r = Round(list(w.ctx), w.t_nodes, seed=workloads.layer_seed(w, 0))
    r.gpu_cache()
    r.oracle_cache()
    for path in ("exact", "int8"):
        got = r.gpu_verify(path).float().cpu().numpy()
        seqs = (0, 5, 7) if name == "ragged" else (0,)
        heads = (0, 23) if name == "ragged" else (0, 11, 23)
        want = r.oracle_attention(path, rows=head_rows(seqs, heads, r.T)).reshape(-1, r.T, 256)
        assert_attention_close(gather_heads(got, seqs, heads, r.T), want, f"{name}/{path}")


@pytest.mark.parametrize("name,layers", [("tree32k", tuple(range(1, 16))), ("long262k", (7, 15))])
def test_full_size_other_layers(gpu, name, layers):
    """The other layers of the full-size workloads (layer 0 is above): every
    layer at 32K and layers 7 and 15 at 262K, exact path, the first and last
    Q head of each layer (all T nodes) against the oracle."""
    w = workloads.WORKLOADS[name]
    for layer in layers:
        r = Round(list(w.ctx), w.t_nodes, seed=workloads.layer_seed(w, layer))
        r.gpu_cache()
        r.oracle_cache()
        got = r.gpu_verify("exact").float().cpu().numpy()
        heads = (0, r.hq - 1)
        want = r.oracle_attention("exact", rows=head_rows((0,), heads, r.T)).reshape(-1, r.T, 256)
        assert_attention_close(gather_heads(got, (0,), heads, r.T), want, f"{name} layer {layer}")
        del r


@pytest.mark.parametrize("ctx,t,hq,hkv", [
    ([700], 16, 24, 4),    # 716 keys: ragged last tile, one split per head
    ([3000], 5, 24, 4),    # several splits per head, 30 rows
    ([511], 32, 16, 4),    # 128 rows per KV head: one group per QK round
])
def test_int8_dots_bit_exact(gpu, ctx, t, hq, hkv):
    """The int8 path's per-group integer dots I_g, as the verify kernel forms
    them on the tensor cores (every row, every key of [0, ctx + T), every
    group), equal the oracle's exact integers bit for bit; the same launch's
    attention output stays within the tolerance."""
    r = Round(ctx, t, seed=77 + t, hq=hq, hkv=hkv)
    layer = r.gpu_cache()
    r.oracle_cache()
    G, n = hq // hkv, ctx[0] + t
    ws = torch.empty(stv.stv_verify_workspace_bytes(r.shape, r.seqs, t), dtype=torch.uint8, device=gpu)
    dots = torch.full((hkv, t * G, n, 8), -(2 ** 31), dtype=torch.int32, device=gpu)
    parent = torch.as_tensor(r.parent, device=gpu)
    stv.stv_int8_qk_dots(r.shape, layer, r.seqs[0], r.q, parent, t, ws, dots)
    o = torch.empty((1, t, hq, 256), dtype=torch.float16, device=gpu)
    stv.stv_split_combine(r.shape, r.seqs, t, ws, o)
    torch.cuda.synchronize()
    got = dots.cpu().numpy()
    qn = r.q.cpu().numpy()
    for h in range(hkv):
        for row in range(t * G):
            node, qh = row // G, h * G + row % G
            want = oracle.int8_dots(r.ocache, r.tables, 0, qn[0, node, qh], qh, r.hq, 0, n)
            assert np.array_equal(got[h, row], want), f"KV head {h} row {row}"
    assert_attention_close(o.float().cpu().numpy(), r.oracle_attention("int8"), f"{ctx}/{t}/int8 (dump launch)")


def test_deterministic_run_to_run(gpu):
    r = Round([5000, 3000], 16, seed=5)
    r.gpu_cache()
    a = r.gpu_verify("exact")
    b = r.gpu_verify("exact")
    assert torch.equal(a, b)


def test_bad_tree_flagged(gpu):
    r = Round([100], 4, seed=6, parents=[[-1, 0, 5, 1]])
    r.gpu_cache()
    ws = torch.empty(stv.stv_verify_workspace_bytes(r.shape, r.seqs, 4), dtype=torch.uint8, device=gpu)
    status = torch.zeros(1, dtype=torch.int32, device=gpu)
    stv.stv_verify_attn(r.shape, r.layer, r.seqs, r.q, torch.as_tensor(r.parent, device=gpu), 4, "exact", ws,
                        dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & stv.STV_DEV_BAD_TREE


def test_bad_tree_flagged_batch(gpu):
    """The same check in a batch of several sequences (the persistent kernel)."""
    r = Round([3000, 100], 4, seed=8, parents=[[-1, 0, 1, 2], [-1, 0, 5, 1]])
    r.gpu_cache()
    ws = torch.empty(stv.stv_verify_workspace_bytes(r.shape, r.seqs, 4), dtype=torch.uint8, device=gpu)
    status = torch.zeros(1, dtype=torch.int32, device=gpu)
    stv.stv_verify_attn(r.shape, r.layer, r.seqs, r.q, torch.as_tensor(r.parent, device=gpu), 4, "exact", ws,
                        dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & stv.STV_DEV_BAD_TREE


@pytest.mark.parametrize("path", ["exact", "int8"])
def test_sixty_four_sequences(gpu, path):
    """The largest batch: 64 sequences of 0..3,000 cached tokens.  Every
    (sequence, KV head) takes at least one work unit, so the plan holds more
    units than SMs: the exact path's persistent kernel takes two or more per
    CTA, the int8 kernel runs them as waves.  Whole heads of every eighth
    sequence against the oracle."""
    rng = np.random.default_rng(64)
    ctx = [int(c) for c in rng.integers(0, 3000, 64)]
    r = Round(ctx, 16, seed=6464)
    r.gpu_cache()
    r.oracle_cache()
    got = r.gpu_verify(path).float().cpu().numpy()
    seqs, heads = range(0, 64, 8), (0, 23)
    want = r.oracle_attention(path, rows=head_rows(seqs, heads, 16)).reshape(-1, 16, 256)
    assert_attention_close(gather_heads(got, seqs, heads, 16), want, f"64 sequences/{path}")


def test_ragged_full_size_deterministic(gpu):
    """Eight requests, 1K..128K: the balanced plan (more units than SMs, the
    persistent kernel dealing them longest first) gives the same bytes on
    every run."""
    w = workloads.WORKLOADS["ragged"]
    r = Round(list(w.ctx), w.t_nodes, seed=workloads.layer_seed(w, 3))
    r.gpu_cache()
    a = r.gpu_verify("exact")
    b = r.gpu_verify("exact")
    assert torch.equal(a, b)


def test_workspace_too_small_rejected(gpu):
    r = Round([100], 4, seed=7)
    r.gpu_cache()
    need = stv.stv_verify_workspace_bytes(r.shape, r.seqs, 4)
    ws = torch.empty(need - 256, dtype=torch.uint8, device=gpu)
    with pytest.raises(stv.StvError) as e:
        stv.stv_verify_attn(r.shape, r.layer, r.seqs, r.q, torch.as_tensor(r.parent, device=gpu), 4, "exact", ws)
    assert e.value.status == stv.STV_ERR_WORKSPACE_TOO_SMALL


@pytest.mark.parametrize("path", ["exact", "int8"])
def test_graph_replay_deterministic(gpu, path):
    """A round's verify, split merge and acceptance captured once in a CUDA
    graph and replayed twice give bit-identical outputs, equal to the eager
    launches' (fixed split order, no float atomics, no data-dependent
    scheduling)."""
    r = Round([5000, 300, 12000], 16, seed=61)
    r.gpu_cache()
    eager = r.gpu_verify(path)
    parent = torch.as_tensor(r.parent, device=gpu)
    draft = torch.as_tensor(r.draft, device=gpu)
    argmax = torch.as_tensor(r.argmax, device=gpu)
    ws = torch.empty(stv.stv_verify_workspace_bytes(r.shape, r.seqs, r.T), dtype=torch.uint8, device=gpu)
    o = torch.empty_like(eager)
    n_commit = torch.zeros(r.n_seqs, dtype=torch.int32, device=gpu)
    acc_path = torch.zeros((r.n_seqs, r.T), dtype=torch.int32, device=gpu)
    out_ids = torch.zeros((r.n_seqs, r.T), dtype=torch.int32, device=gpu)

    def launches():
        stv.stv_verify_attn(r.shape, r.layer, r.seqs, r.q, parent, r.T, path, ws)
        stv.stv_split_combine(r.shape, r.seqs, r.T, ws, o)
        stv.stv_tree_accept(parent, draft, argmax, n_commit, acc_path, out_ids)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        launches()  # warm-up off the capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        launches()
    outs = []
    for _ in range(2):
        o.fill_(float("nan"))
        n_commit.zero_()
        graph.replay()
        torch.cuda.synchronize()
        outs.append((o.clone(), n_commit.clone(), acc_path.clone(), out_ids.clone()))
    for a, b in zip(outs[0], outs[1]):
        assert torch.equal(a, b)
    assert torch.equal(outs[0][0], eager)


@pytest.mark.parametrize("path", ["exact", "int8"])
def test_wait_timeout_reported_and_context_usable(gpu, path):
    """Failure detection without a GPU fault: the verify kernel with its
    copies withheld (stv_verify_attn_timeout_test) has every consumer's wait
    run out; the launch returns within seconds with STV_DEV_TIMEOUT, and a
    normal verify right after it on the same context still matches the
    oracle."""
    import time

    r = Round([300], 4, seed=303)
    r.gpu_cache()
    r.oracle_cache()
    ws = torch.empty(stv.stv_verify_workspace_bytes(r.shape, r.seqs, r.T), dtype=torch.uint8, device=gpu)
    status = torch.zeros(1, dtype=torch.int32, device=gpu)
    parent = torch.as_tensor(r.parent, device=gpu)
    torch.cuda.synchronize()
    t0 = time.monotonic()
    stv.stv_verify_attn_timeout_test(r.shape, r.layer, r.seqs, r.q, parent, r.T, path, ws, dev_status=status)
    torch.cuda.synchronize()
    elapsed = time.monotonic() - t0
    assert int(status.item()) & stv.STV_DEV_TIMEOUT
    assert elapsed < 30.0, elapsed
    got = r.gpu_verify(path).float().cpu().numpy()
    assert_attention_close(got, r.oracle_attention(path), f"verify after a timed-out launch ({path})")
