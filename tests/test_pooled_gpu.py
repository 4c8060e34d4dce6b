"""Layers whose adapters are stored at their true rank in a row pool
(lora_layer_create_pooled), against the oracle: every kernel path reads a slot from its
first pool row -- the decode BGMV (slot widths 16, 32 and 64), the tensor-core SGMV shrink
and expand of large batches, the fp32 tile kernel and GEMM, compositions -- and the row
allocator: reloads at another rank, unloads, a full or fragmented pool.
"""
import numpy as np
import pytest
import torch

import oracle
from segmented_rank_gemm_gb300 import workloads
from gpu_helpers import assert_parity, oracle_rows

pytestmark = pytest.mark.gpu
BF16, F32 = torch.bfloat16, torch.float32


def _rows(r):
    return (r + 7) // 8 * 8


def _pooled(wl, max_rank, pool_rows, T=None):
    from segmented_rank_gemm_gb300.lora import LoraLayer
    layer = LoraLayer(wl.W.cuda(), wl.S, max_rank, T or wl.T, pool_rows=pool_rows)
    for s, ad in enumerate(wl.adapters):
        if ad is not None:
            layer.load(s, ad[0].cuda(), ad[1].cuda(), ad[2])
    return layer


def _run(layer, wl):
    y = layer(wl.x.cuda(), wl.token_slot.cuda())
    torch.cuda.synchronize()
    return y


@pytest.mark.parametrize("T", [300, 700])
@pytest.mark.parametrize("max_rank,ranks", [(16, [1, 7, 16, 3, 12, 5]),
                                            (32, [32, 1, 20, 9, 17, 8]),
                                            (64, [1, 40, 64, 9, 33, 17])])
def test_pooled_parity_bf16(T, max_rank, ranks):
    wl = workloads.synthetic(600 + T + max_rank, T, 256, 200, S=len(ranks), ranks=ranks,
                             R=max_rank, base_frac=0.1)
    need = sum(_rows(r) for r in ranks)
    layer = _pooled(wl, max_rank, need)  # exactly full
    assert layer.pool_usage() == (need, need)
    assert need < len(ranks) * _rows(max_rank)
    y = _run(layer, wl)
    assert layer.status() == 0
    assert_parity(y, oracle_rows(wl), BF16, what="pooled T=%d R=%d" % (T, max_rank))
    layer.close()


def test_pooled_parity_fp32():
    wl = workloads.synthetic(650, 150, 72, 40, S=4, ranks=[1, 16, 5, 9], R=16, dtype=F32)
    layer = _pooled(wl, 16, 48)
    y = _run(layer, wl)
    assert_parity(y, oracle_rows(wl), F32, what="pooled fp32")
    layer.close()


@pytest.mark.parametrize("T", [200, 600])
def test_pooled_compositions(T):
    from segmented_rank_gemm_gb300.lora import LoraLayer
    g = torch.Generator().manual_seed(T)
    K, N = 256, 128
    W = (torch.randn(K, N, generator=g) * 0.02).to(BF16)
    x = torch.randn(T, K, generator=g).to(BF16)

    def m(r, w):
        return ((torch.randn(K, r, generator=g) * 0.02).to(BF16),
                (torch.randn(r, N, generator=g) * 0.02).to(BF16), 2.0 * r, w)

    comps = [[m(3, 0.5), m(5, -1.0)], [m(16, 1.0)], [m(1, 2.0), m(2, 1.0), m(4, 0.25)]]
    layer = LoraLayer(W.cuda(), 3, 16, T, pool_rows=8 + 16 + 8)
    for s, c in enumerate(comps):
        layer.load_composed(s, [(A.cuda(), B.cuda(), al, w) for A, B, al, w in c])
    ids = torch.tensor(np.random.default_rng(T).integers(-1, 3, size=T), dtype=torch.int32)
    y = layer(x.cuda(), ids.cuda())
    torch.cuda.synchronize()
    assert_parity(y, oracle.forward_composed(x, W, comps, ids), BF16, what="pooled compositions")
    layer.close()


def test_row_allocator():
    from segmented_rank_gemm_gb300.lora import LoraError
    wl = workloads.synthetic(660, 256, 256, 136, S=4, ranks=[8, 16, 8, 8], R=16, base_frac=0.0)
    layer = _pooled(wl, 16, 48)  # rows: slot 0 [0, 8), 1 [8, 24), 2 [24, 32), 3 [32, 40)
    assert layer.pool_usage() == (40, 48)
    g = torch.Generator().manual_seed(1)

    def adapter(r):
        return ((torch.randn(wl.K, r, generator=g) * 0.02).to(BF16),
                (torch.randn(r, wl.N, generator=g) * 0.02).to(BF16), 2.0 * r)

    # a rank-16 adapter does not fit in the 8 free rows: refused, slot 2 unchanged
    big = adapter(16)
    with pytest.raises(LoraError) as e:
        layer.load(2, big[0].cuda(), big[1].cuda(), big[2])
    assert e.value.code == -6  # LORA_ENOMEM
    assert layer.pool_usage() == (40, 48)
    assert_parity(_run(layer, wl), oracle_rows(wl), BF16, what="after a refused load")
    # unloading slot 1 frees 16 rows in the middle: the rank-16 adapter fits there
    layer.unload(1)
    assert layer.pool_usage() == (24, 48)
    layer.load(0, big[0].cuda(), big[1].cuda(), big[2])  # slot 0 moves: 8 rows -> 16
    wl.adapters[0] = big
    assert layer.pool_usage() == (32, 48)
    # slot 1 back at rank 5 (8 rows), slot 3 at rank 9 (16 rows, after its 8 are returned)
    for s, r in ((1, 5), (3, 9)):
        ad = adapter(r)
        layer.load(s, ad[0].cuda(), ad[1].cuda(), ad[2])
        wl.adapters[s] = ad
    assert layer.pool_usage() == (48, 48)
    y = _run(layer, wl)
    assert layer.status() == 0
    assert_parity(y, oracle_rows(wl), BF16, what="after moves and reloads")
    layer.close()
