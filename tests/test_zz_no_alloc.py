"""stv_verify_attn_no_alloc: the verify + merge entry point for callers that
cannot allocate device memory (a serving engine whose allocator already owns
the device memory, or a plain C host without a device allocator).  It must
give the workspace path's results, call after call, and refuse rounds whose
scratch would not fit its fixed array.

This file is named so that pytest collects it last."""
import numpy as np
import pytest
import torch

import speculative_tree_verify_bit_gb300 as stv
from roundkit import Round

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("path", ["exact", "int8"])
def test_no_alloc_matches_workspace_path_on_consecutive_calls(gpu, path):
    """Bit for bit the workspace path's output (the same kernels and split
    plan run on the same inputs), on two calls in a row.  A larger round goes
    through the library's array first, so the calls under test find its
    contents stale: nothing they read may depend on them."""
    big = Round([20000, 9000], 32, seed=8081, hq=16, hkv=4)
    big.gpu_cache()
    o_big = torch.empty((big.n_seqs, big.T, big.hq, 256), dtype=torch.float16, device=gpu)
    stv.stv_verify_attn_no_alloc(big.shape, big.layer, big.seqs, big.q, torch.as_tensor(big.parent, device=gpu), big.T,
                                 path, o_big)
    r = Round([1500, 300, 4000], 16, seed=8080)
    r.gpu_cache()
    want = r.gpu_verify(path)  # workspace path
    parent = torch.as_tensor(r.parent, device=gpu)
    for call in range(2):
        o = torch.full((r.n_seqs, r.T, r.hq, 256), float("nan"), dtype=torch.float16, device=gpu)
        status = torch.zeros(1, dtype=torch.int32, device=gpu)
        stv.stv_verify_attn_no_alloc(r.shape, r.layer, r.seqs, r.q, parent, r.T, path, o, dev_status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.equal(o, want), f"no-alloc call {call} differs from the workspace path"


def test_no_alloc_rejects_rounds_beyond_its_scratch(gpu):
    # 64 sequences x 4 KV heads x 128 rows of fp32 partials exceed 32 MiB.
    n, t, hq, hkv = 64, 32, 16, 4
    layer = stv.LayerCache.empty(n, hkv, device=gpu)
    seqs = [stv.Seq(torch.tensor([i], dtype=torch.int32, device=gpu), 0) for i in range(n)]
    q = torch.zeros((n, t, hq, 256), dtype=torch.float16, device=gpu)
    parent = torch.as_tensor(np.tile(np.arange(-1, t - 1, dtype=np.int32), (n, 1)), device=gpu)
    o = torch.zeros_like(q)
    shape = stv.make_shape(hq, hkv)
    assert stv.stv_verify_workspace_bytes(shape, seqs, t) > (32 << 20)
    with pytest.raises(stv.StvError) as e:
        stv.stv_verify_attn_no_alloc(shape, layer, seqs, q, parent, t, "exact", o)
    assert e.value.status == stv.STV_ERR_WORKSPACE_TOO_SMALL
