"""a1 kv_append_pack on the GPU: cache bytes bit-exact against the oracle.

Source: "elpis" README, header table (3-bit KV cache, 12 KiB per token over
16 layers); quantizer, bit layout and page layout as stated in include/stv.h."""
import numpy as np
import pytest
import torch

import oracle
import speculative_tree_verify_bit_gb300 as stv
import workloads
from roundkit import Round

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("ctx,t", [([1024], 16), ([8192], 8), ([0, 250, 777], 5), ([63, 64, 65], 32)])
def test_pack_bytes_bit_exact(gpu, ctx, t):
    r = Round(ctx, t, seed=1000 + sum(ctx) + t, hq=4 * 6 if t <= 16 else 16, hkv=4)
    layer = r.gpu_cache()
    cache = r.oracle_cache()
    got = layer.pool.cpu().numpy()
    assert np.array_equal(got, cache.pool)


def test_pack_full_size_long_context_layer(gpu):
    """262,144-token context of one layer (the long workload's size), packed in
    one launch: every byte of the pool equals the oracle's."""
    w = workloads.WORKLOADS["long262k"]
    r = Round(list(w.ctx), w.t_nodes, seed=workloads.layer_seed(w, 0))
    layer = r.gpu_cache()
    cache = r.oracle_cache()
    assert np.array_equal(layer.pool.cpu().numpy(), cache.pool)


def test_pack_special_values(gpu):
    """Zero groups (scale 0, codes 4), tiny subnormal groups, max-magnitude
    values, exact quantization ties."""
    rows = np.zeros((6, 1, 256), np.float16)
    rows[1, 0, :] = np.float16(2.0 ** -24)            # m/4 rounds to 0
    rows[2, 0, :] = np.float16(65504.0)
    rows[2, 0, ::3] = np.float16(-65504.0)
    s = 0.5
    rows[3, 0, :32] = np.array([-4 * s] + [s * (k + 0.5) for k in range(-4, 3)] * 4 + [s * 3] * 3,
                               np.float64)[:32].astype(np.float16)
    rows[4, 0, :] = (np.arange(256) - 128).astype(np.float16) * np.float16(1e-3)
    rows[5, 0, :] = np.float16(-3.0)
    k = torch.as_tensor(rows, device=gpu)
    v = torch.as_tensor(rows[::-1].copy(), device=gpu)
    table = np.array([1, 0], np.int32)
    pos = np.array([0, 31, 32, 63, 64, 300], np.int32)
    layer = stv.LayerCache.empty(2, 1, device=gpu)
    seqs = [stv.Seq(torch.as_tensor(table, device=gpu), 0)]
    stv.stv_kv_append_pack(stv.make_shape(1, 1), layer, seqs, k, v, torch.zeros(6, dtype=torch.int32, device=gpu),
                           torch.as_tensor(pos, device=gpu))
    cache = oracle.Cache(1, 2)
    oracle.kv_append(cache, [table], rows, rows[::-1].copy(), np.zeros(6, np.int32), pos)
    assert np.array_equal(layer.pool.cpu().numpy(), cache.pool)


def test_pack_bad_rows_and_pages_flagged_not_written(gpu):
    layer = stv.LayerCache.empty(2, 1, device=gpu)
    table = torch.tensor([0, 7], dtype=torch.int32, device=gpu)  # page 7 is outside the 2-page pool
    seqs = [stv.Seq(table, 0)]
    k = torch.ones((3, 1, 256), dtype=torch.float16, device=gpu)
    status = torch.zeros(1, dtype=torch.int32, device=gpu)
    stv.stv_kv_append_pack(stv.make_shape(1, 1), layer, seqs, k, k, torch.tensor([0, 5, 0], dtype=torch.int32,
                           device=gpu), torch.tensor([300, 1, 600], dtype=torch.int32, device=gpu), dev_status=status)
    torch.cuda.synchronize()
    st = int(status.item())
    assert st & stv.STV_DEV_BAD_PAGE and st & stv.STV_DEV_BAD_ROW
    assert int(layer.pool.sum().item()) == 0


def test_host_validation_rejects_before_launch(gpu):
    layer = stv.LayerCache.empty(1, 4, device=gpu)
    seqs = [stv.Seq(torch.zeros(1, dtype=torch.int32, device=gpu), 0)]
    k = torch.zeros((1, 4, 256), dtype=torch.float16, device=gpu)
    idx = torch.zeros(1, dtype=torch.int32, device=gpu)
    bad = stv.stv_shape(24, 4, 128, 32, 256)
    with pytest.raises(stv.StvError) as e:
        stv.stv_kv_append_pack(bad, layer, seqs, k, k, idx, idx)
    assert e.value.status == stv.STV_ERR_SHAPE_UNSUPPORTED
    with pytest.raises(stv.StvError) as e:
        stv.stv_kv_append_pack(stv.make_shape(24, 4), stv.LayerCache.empty(1, 2, device=gpu), seqs, k, k, idx, idx)
    assert e.value.status == stv.STV_ERR_SHAPE_UNSUPPORTED


@pytest.mark.parametrize("m", [4.0, 3.0, 0.37, 1000.0, 65504.0, 6.0e-5, 5 * 2.0 ** -24, 7 * 2.0 ** -24])
def test_pack_quantizer_every_fp16_value(gpu, m):
    """Every finite fp16 value in [-m, m] quantized in a group whose maximum
    is m (channel 0 of each group holds m), as K and as V: the cache bytes
    equal the oracle's.  The scales include fp16-subnormal ones (the last two
    maxima give s = 2^-24 and 2^-23, where x / s reaches 5 and 3.5)."""
    h = np.arange(65536, dtype=np.uint16).view(np.float16)
    vals = h[np.isfinite(h) & (np.abs(h.astype(np.float64)) <= np.float16(m))]
    n_groups = -(-len(vals) // 31)
    groups = np.zeros((n_groups, 32), np.float16)
    groups[:, 0] = np.float16(m)
    flat = groups[:, 1:].reshape(-1)
    flat[:len(vals)] = vals
    groups[:, 1:] = flat.reshape(n_groups, 31)
    n_rows = -(-n_groups // 8)
    rows = np.zeros((n_rows * 8, 32), np.float16)
    rows[:n_groups] = groups
    rows = rows.reshape(n_rows, 1, 256)
    pages = -(-n_rows // 256)
    table = np.arange(pages, dtype=np.int32)
    pos = np.arange(n_rows, dtype=np.int32)
    vrows = (-rows).copy()
    layer = stv.LayerCache.empty(pages, 1, device=gpu)
    seqs = [stv.Seq(torch.as_tensor(table, device=gpu), 0)]
    stv.stv_kv_append_pack(stv.make_shape(1, 1), layer, seqs, torch.as_tensor(rows, device=gpu),
                           torch.as_tensor(vrows, device=gpu), torch.zeros(n_rows, dtype=torch.int32, device=gpu),
                           torch.as_tensor(pos, device=gpu))
    cache = oracle.Cache(1, pages)
    oracle.kv_append(cache, [table], rows, vrows, np.zeros(n_rows, np.int32), pos)
    assert np.array_equal(layer.pool.cpu().numpy(), cache.pool)
