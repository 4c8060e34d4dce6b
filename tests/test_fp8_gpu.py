"""The e4m3-base layer (lora_layer_create_fp8) on the GPU against the oracle's definition:
y = sx sw (xq wq) + the low-rank term of the bf16 x, with the quantisation of x (per row,
every forward) and W (per column, at creation) decided exactly as the oracle decides it.
Ragged shapes, inputs already on the e4m3 grid (quantisation is the identity: the plain
product), every tiling of the decode-mode GEMM, and the decode workload's full shape.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import fp8
from segmented_rank_gemm_gb300 import workloads
from gpu_helpers import assert_parity

pytestmark = pytest.mark.gpu
BF16 = torch.bfloat16


def _ref(wl, rows=None):
    x = wl.x.float().numpy()
    table = oracle.SlotTable(wl.adapters, wl.K, wl.N)
    delta = oracle.forward_rows(wl.x, torch.zeros(wl.K, wl.N, dtype=torch.float64), table,
                                wl.token_slot, rows=rows)
    base = fp8.base_w8a8(x if rows is None else x[rows], wl.W.float().numpy())
    return base + delta


def _layer(wl):
    from segmented_rank_gemm_gb300.lora import LoraLayer
    layer = LoraLayer(wl.W.cuda(), wl.S, wl.R, max(wl.T, 1), fp8_base=True)
    for s, ad in enumerate(wl.adapters):
        if ad is not None:
            layer.load(s, ad[0].cuda(), ad[1].cuda(), ad[2])
    return layer


@pytest.mark.parametrize("T,K,N", [(256, 512, 320), (300, 1024, 264), (1, 64, 72),
                                   (129, 256, 1040)])
def test_fp8_base_parity(T, K, N):
    wl = workloads.synthetic(700 + T, T, K, N, S=6, ranks=[1, 16, 8, 3, 12, 2], R=16,
                             base_frac=0.15, empty_slots=(4,))
    layer = _layer(wl)
    y = layer(wl.x.cuda(), wl.token_slot.cuda())
    torch.cuda.synchronize()
    assert layer.status() == (-4 if (wl.token_slot == 4).any() else 0)
    assert_parity(y, _ref(wl), BF16, what="fp8 base T=%d K=%d N=%d" % (T, K, N))
    layer.close()


def test_fp8_on_grid_inputs_equal_the_plain_product():
    rng = np.random.default_rng(3)
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F])
    grid = np.unique([float(fp8.e4m3_round(v)) for v in
                      [(-1) ** (c >> 7) * (2.0 ** ((c >> 3 & 15) - 7) * (1 + (c & 7) / 8)
                                           if (c >> 3 & 15) else (c & 7) * 2.0 ** -9)
                       for c in codes]])
    T, K, N = 64, 128, 96
    x = rng.choice(grid, size=(T, K)) / 64.0  # on the grid, row max set to 448 / 64 below
    x[:, 5] = 448.0 / 64.0
    W = rng.choice(grid, size=(K, N)) / 4096.0
    W[7, :] = 448.0 / 4096.0
    wl = workloads.synthetic(720, T, K, N, S=2, ranks=[4, 8], R=8, base_frac=0.3)
    wl.x = torch.tensor(x, dtype=BF16)
    wl.W = torch.tensor(W, dtype=BF16)
    assert np.array_equal(wl.x.double().numpy(), x) and np.array_equal(wl.W.double().numpy(), W)
    layer = _layer(wl)
    y = layer(wl.x.cuda(), wl.token_slot.cuda())
    torch.cuda.synchronize()
    plain = oracle.forward_rows(wl.x, wl.W, oracle.SlotTable(wl.adapters, K, N), wl.token_slot)
    assert np.allclose(_ref(wl), plain, rtol=0, atol=1e-12)  # quantisation is the identity
    assert_parity(y, plain, BF16, what="fp8 base, inputs on the e4m3 grid")
    layer.close()


def test_fp8_every_decode_plan():
    wl = workloads.synthetic(730, 300, 1024, 520, S=5, ranks=16, R=16, base_frac=0.1)
    ref = _ref(wl)
    layer = _layer(wl)
    for bn in (64, 128, 256):
        for ks in (1, 2, 4):
            for pair in (0, 1):
                if bn // ks < 32 or (pair and bn < 128):
                    continue
                layer.set_gemm_plan(bn, ks, pair)
                y = layer(wl.x.cuda(), wl.token_slot.cuda())
                torch.cuda.synchronize()
                assert layer.status() == 0
                assert_parity(y, ref, BF16, what="fp8 plan (%d, %d, %d)" % (bn, ks, pair))
    layer.close()


def test_fp8_decode_workload_full_shape():
    wl = workloads.decode_bgmv(seed=1002, device="cpu")
    layer = _layer(wl)
    y = layer(wl.x.cuda(), wl.token_slot.cuda())
    torch.cuda.synchronize()
    assert layer.status() == 0
    assert_parity(y, _ref(wl), BF16, what="fp8 base, decode workload, every row")
    layer.close()


def test_fp8_limits():
    from segmented_rank_gemm_gb300.lora import LoraError, LoraLayer
    W = torch.zeros(72, 64, dtype=BF16, device="cuda")  # K = 72: not a multiple of 16
    with pytest.raises(LoraError):
        LoraLayer(W, 2, 8, 16, fp8_base=True)
    # a K split is refused for batches beyond 512 rows (their expand blocks follow the base
    # blocks in one accumulation per tile)
    wl = workloads.synthetic(790, 600, 128, 256, S=2, ranks=[8, 4], R=8, base_frac=0.1)
    layer = _layer(wl)
    try:
        layer.set_gemm_plan(256, 2, 0)
        y = layer(wl.x.cuda(), wl.token_slot.cuda())  # (v mode runs the plan unsplit)
        torch.cuda.synchronize()
        assert layer.status() == 0
        assert_parity(y, _ref(wl), BF16, what="fp8 prefill, a split plan run unsplit")
    finally:
        layer.close()


# ---- batches of more than 512 rows: the SGMV path; the e4m3 base product is scaled in TMEM
# before the expand blocks' bf16 MMAs add to the same accumulator ----

@pytest.mark.parametrize("T,K,N,layout", [(700, 1024, 1040, "runs"), (1300, 512, 264, "random"),
                                          (513, 2048, 4096, "runs")])
def test_fp8_prefill_parity(T, K, N, layout):
    wl = workloads.synthetic(800 + T, T, K, N, S=9, ranks=[16, 1, 8, 16, 3, 12, 16, 5, 2], R=16,
                             base_frac=0.1, layout=layout, empty_slots=(6,))
    layer = _layer(wl)
    try:
        for rep in range(2):
            y = layer(wl.x.cuda(), wl.token_slot.cuda())
            torch.cuda.synchronize()
            assert layer.status() == (-4 if (wl.token_slot == 6).any() else 0)
            assert_parity(y, _ref(wl), BF16, what="fp8 prefill T=%d K=%d N=%d (%d)" % (T, K, N, rep))
    finally:
        layer.close()


def test_fp8_prefill_every_plan():
    # 700 rows (5.5 row tiles; pairs: the last CTA partial), 8 e4m3 K blocks, N = 1000
    wl = workloads.synthetic(830, 700, 1024, 1000, S=24, ranks=16, R=16, base_frac=0.1,
                             layout="runs")
    ref = _ref(wl)
    layer = _layer(wl)
    try:
        for bn, pair in ((64, 0), (128, 0), (128, 1), (256, 0), (256, 1)):
            layer.set_gemm_plan(bn, 1, pair)
            y = layer(wl.x.cuda(), wl.token_slot.cuda())
            torch.cuda.synchronize()
            assert layer.status() == 0
            assert_parity(y, ref, BF16, what="fp8 prefill plan (%d, 1, %d)" % (bn, pair))
    finally:
        layer.close()


def test_fp8_prefill_stream_k_tail_and_wide_rank():
    # more tiles than resident CTAs with a short last round (its tiles cut in two, the
    # tail's partial added to the head's base accumulator before the scales), and rank 64
    # (two expand blocks per slot and half)
    for wl in (workloads.synthetic(840, 2600, 1024, 2048, S=24, ranks=16, R=16, base_frac=0.1,
                                   layout="runs"),
               workloads.synthetic(841, 900, 512, 512, S=10,
                                   ranks=[64, 40, 8, 64, 17, 64, 1, 33, 64, 2], R=64,
                                   base_frac=0.05, layout="random")):
        layer = _layer(wl)
        try:
            y = layer(wl.x.cuda(), wl.token_slot.cuda())
            torch.cuda.synchronize()
            assert layer.status() == 0
            assert_parity(y, _ref(wl), BF16, what="fp8 prefill " + wl.name)
        finally:
            layer.close()


def test_fp8_prefill_base_only_tiles_and_stream_k_heads():
    # The base product is scaled in TMEM before a tile's expand blocks add to it; a tile
    # with no adapted row has no expand block and is scaled as it drains.  Rows 0-255 and
    # 1024-1535 are base-only, so whole row tiles of each kind run in the full rounds and
    # among the stream-K heads of the short last round (whose tails' partials are added
    # before or after the scales), on the automatic plan, 128-wide tiles and CTA pairs.
    wl = workloads.synthetic(850, 2600, 1024, 2048, S=24, ranks=16, R=16, base_frac=0.1,
                             layout="runs")
    wl.token_slot[0:256] = -1
    wl.token_slot[1024:1536] = -1
    ref = _ref(wl)
    layer = _layer(wl)
    try:
        for plan in ((0, 1, 0), (128, 1, 0), (256, 1, 1)):
            layer.set_gemm_plan(*plan)
            y = layer(wl.x.cuda(), wl.token_slot.cuda())
            torch.cuda.synchronize()
            assert layer.status() == 0
            assert_parity(y, ref, BF16, what="fp8 prefill, base-only tiles, plan %s" % (plan,))
    finally:
        layer.close()


@pytest.mark.parametrize("K", [128, 192])
def test_fp8_prefill_short_k_range(K):
    # one e4m3 K block (K = 128) is never cut between a stream-K head and tail; two (the
    # second ragged, K = 192) are cut one and one
    wl = workloads.synthetic(860 + K, 2600, K, 2048, S=24, ranks=16, R=16, base_frac=0.1,
                             layout="runs")
    layer = _layer(wl)
    try:
        y = layer(wl.x.cuda(), wl.token_slot.cuda())
        torch.cuda.synchronize()
        assert layer.status() == 0
        assert_parity(y, _ref(wl), BF16, what="fp8 prefill, K = %d" % K)
    finally:
        layer.close()


def test_fp8_prefill_workload_full_shape():
    wl = workloads.prefill_sgmv(seed=1003, device="cpu")
    layer = _layer(wl)
    try:
        y = layer(wl.x.cuda(), wl.token_slot.cuda())
        torch.cuda.synchronize()
        assert layer.status() == 0
        # every row (the e4m3 base product is one fp64 matrix product on the host; the
        # low-rank term comes from the C oracle)
        assert_parity(y, _ref(wl), BF16, what="fp8 base, prefill workload, every row")
    finally:
        layer.close()


def test_fp8_mixed_workload_full_shape():
    # the continuous batch: 8 prefill requests of 448 rows and 512 one-row decode requests
    # over 100 slots (K = 14336, N = 4096), so most row tiles carry many expand blocks
    wl = workloads.mixed_continuous(seed=1004, device="cpu")
    layer = _layer(wl)
    try:
        y = layer(wl.x.cuda(), wl.token_slot.cuda())
        torch.cuda.synchronize()
        assert layer.status() == 0
        assert_parity(y, _ref(wl), BF16, what="fp8 base, mixed workload, every row")
    finally:
        layer.close()


def test_fp8_back_to_back_forwards_and_split_batches():
    # The BGMV kernel quantises x's rows as it starts and counts them; the GEMM's loads wait
    # for the count, and the last CTA of the batch's last GEMM launch resets it.  Several
    # forwards in a row on one stream, each with new x, on shapes whose automatic plan runs
    # the GEMM as one launch and as two (a last round at most half full: N = 14336).
    for T, K, N in [(512, 4096, 14336), (300, 1024, 4104), (37, 512, 264)]:
        wl = workloads.synthetic(740 + T, T, K, N, S=7, ranks=[16, 4, 8, 16, 1, 12, 16], R=16,
                                 base_frac=0.1)
        layer = _layer(wl)
        rows = np.arange(0, T, 7)
        try:
            for rep in range(3):
                g = torch.Generator().manual_seed(9000 + 31 * T + rep)
                wl.x = (torch.randn(T, K, generator=g) * (0.5 + rep)).to(BF16)
                y = layer(wl.x.cuda(), wl.token_slot.cuda())
                torch.cuda.synchronize()
                assert layer.status() == 0, (T, K, N, rep)
                assert_parity(y[rows], _ref(wl, rows), BF16,
                              what="fp8 T=%d K=%d N=%d forward %d" % (T, K, N, rep))
        finally:
            layer.close()


def test_fp8_wide_rank_quantises_in_its_own_launch():
    # rank width 64: the decode BGMV runs row-major, and x is quantised by a launch of its
    # own before it (counted the same way)
    wl = workloads.synthetic(760, 200, 1024, 520, S=5, ranks=[64, 33, 8, 64, 1], R=64,
                             base_frac=0.1)
    layer = _layer(wl)
    try:
        for rep in range(2):
            y = layer(wl.x.cuda(), wl.token_slot.cuda())
            torch.cuda.synchronize()
            assert layer.status() == 0
            assert_parity(y, _ref(wl), BF16, what="fp8 rank width 64, forward %d" % rep)
    finally:
        layer.close()


def test_fp8_forward_after_a_failed_launch():
    # a GEMM plan refused at launch time (an empty K range) fails the forward after the BGMV
    # kernel counted its rows; the next forward clears the count and is exact
    from segmented_rank_gemm_gb300.lora import LoraError
    wl = workloads.synthetic(770, 64, 128, 200, S=3, ranks=[8, 4, 16], R=16, base_frac=0.2)
    layer = _layer(wl)
    try:
        layer.set_gemm_plan(128, 4, 0)  # K = 128 e4m3 elements: one K block, no 4-way split
        with pytest.raises(LoraError):
            layer(wl.x.cuda(), wl.token_slot.cuda())
        layer.set_gemm_plan(0)
        y = layer(wl.x.cuda(), wl.token_slot.cuda())
        torch.cuda.synchronize()
        assert layer.status() == 0
        assert_parity(y, _ref(wl), BF16, what="fp8 forward after a refused plan")
    finally:
        layer.close()
