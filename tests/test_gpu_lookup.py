"""stv_lookup_draft on the GPU against the lookup-drafting oracle, exactly:
proposal, its length, the match length and the match start (Reddit posts
(u/iamMess), "Now added" list, lookup-augmented drafting)."""
import numpy as np
import pytest
import torch

import oracle
import speculative_tree_verify_bit_gb300 as stv
import workloads

pytestmark = pytest.mark.gpu


def gpu_lookup(histories, min_len=6, max_len=12, k=15, ws=None):
    dev = "cuda"
    n = len(histories)
    hs = [torch.as_tensor(np.asarray(h, np.int32), device=dev) for h in histories]
    n_prop = torch.full((n,), -7, dtype=torch.int32, device=dev)
    prop = torch.full((n, max(k, 1)), -7, dtype=torch.int32, device=dev)
    mlen = torch.full((n,), -7, dtype=torch.int32, device=dev)
    mpos = torch.full((n,), -7, dtype=torch.int64, device=dev)
    if ws is None:
        ws = torch.zeros(stv.stv_lookup_workspace_bytes(n), dtype=torch.uint8, device=dev)
    stv.stv_lookup_draft(hs, min_len, max_len, k, n_prop, prop, mlen, mpos, ws)
    torch.cuda.synchronize()
    assert int(ws.count_nonzero().item()) == 0, "workspace not left zero"
    return n_prop.cpu().numpy(), prop.cpu().numpy(), mlen.cpu().numpy(), mpos.cpu().numpy()


def assert_matches_oracle(histories, min_len=6, max_len=12, k=15, ws=None):
    n_prop, prop, mlen, mpos = gpu_lookup(histories, min_len, max_len, k, ws)
    for s, h in enumerate(histories):
        want, wl, wp = oracle.lookup_draft(h, min_len, max_len, k)
        assert n_prop[s] == len(want), (s, len(h))
        assert list(prop[s, :len(want)]) == list(want), s
        assert not prop[s, len(want):k].any(), s  # zero beyond the proposal
        assert (mlen[s], mpos[s]) == (wl, wp), (s, len(h))


@pytest.mark.parametrize("alphabet,n", [(2, 100), (3, 3000), (4, 10_000), (8, 50_000), (2, 6000)])
def test_small_alphabets_many_matches(gpu, alphabet, n):
    """Tiny alphabets: matches of every length and many tied candidates, far
    apart and across the 2,048-position chunk boundaries of the scan."""
    rng = np.random.default_rng(alphabet * 7 + n)
    hs = [rng.integers(0, alphabet, int(rng.integers(1, n + 1))).astype(np.int32) for _ in range(12)]
    for min_len, max_len, k in ((6, 12, 15), (1, 4, 3), (2, 32, 64), (6, 6, 1), (12, 12, 0)):
        assert_matches_oracle(hs, min_len, max_len, k)


def test_edge_histories(gpu):
    hs = [np.zeros(0, np.int32), np.array([5], np.int32), np.arange(6, dtype=np.int32),   # empty, 1, too short
          np.full(7, 9, np.int32), np.full(100, 9, np.int32),                               # self-overlapping suffix
          np.arange(5000, dtype=np.int32),                                                  # no repeat
          np.concatenate([np.arange(3000), np.arange(2990, 3000)]).astype(np.int32),       # match ends at n-11
          np.array([2**31 - 1, -2**31, 0, 7] * 40, np.int32)]                              # extreme ids
    assert_matches_oracle(hs)
    assert_matches_oracle(hs, 1, 32, 64)


def test_ragged_and_long_workload_histories(gpu):
    """The ragged workload's 8 requests (1K..128K tokens) and the long
    workload's 262,144-token history, with quoted spans."""
    for name in ("ragged", "long262k", "tree32k"):
        w = workloads.WORKLOADS[name]
        for p_copy in (1.0, 0.0):
            assert_matches_oracle(workloads.lookup_histories(w, p_copy))


def test_workspace_zeroed_once_serves_every_call(gpu):
    """One workspace, zeroed once, for calls with 8, 1, 3 and 8 sequences
    (the counters' offsets move with the count): each call leaves it zero and
    matches the oracle."""
    rng = np.random.default_rng(91)
    ws = torch.zeros(stv.stv_lookup_workspace_bytes(8), dtype=torch.uint8, device=gpu)
    for n in (8, 1, 3, 8):
        hs = [rng.integers(0, 3, int(rng.integers(1, 9000))).astype(np.int32) for _ in range(n)]
        assert_matches_oracle(hs, 2, 12, 15, ws=ws)


def test_rejects_bad_arguments(gpu):
    h = [torch.arange(10, dtype=torch.int32, device=gpu)]
    ws = torch.empty(stv.stv_lookup_workspace_bytes(1), dtype=torch.uint8, device=gpu)
    outs = (torch.zeros(1, dtype=torch.int32, device=gpu), torch.zeros((1, 4), dtype=torch.int32, device=gpu),
            torch.zeros(1, dtype=torch.int32, device=gpu), torch.zeros(1, dtype=torch.int64, device=gpu))
    for min_len, max_len, k in ((0, 4, 4), (5, 4, 4), (1, 33, 4), (1, 4, 65)):
        with pytest.raises(stv.StvError) as e:
            stv.stv_lookup_draft(h, min_len, max_len, k, *outs, ws)
        assert e.value.status == stv.STV_ERR_INVALID_ARG
    with pytest.raises(stv.StvError) as e:
        stv.stv_lookup_draft(h, 1, 4, 4, *outs, ws[:4])
    assert e.value.status == stv.STV_ERR_WORKSPACE_TOO_SMALL
