"""The layer on the GPU (through the C ABI) against the CPU oracle, element by element:
small shapes that span several tiles with ragged tails, the pages' two worked examples,
and the edge cases (empty batch, one row, base-only, one slot, rank 1 and full rank,
empty slots, reloads, fp32)."""
import numpy as np
import pytest
import torch

import oracle
from segmented_rank_gemm_gb300 import workloads
from gpu_helpers import TOL, assert_parity, build_layer, oracle_rows, run_layer

pytestmark = pytest.mark.gpu
BF16, F32 = torch.bfloat16, torch.float32


def _check(wl, **kw):
    layer = build_layer(wl, **kw)
    y = run_layer(layer, wl)
    assert layer.status() == 0, layer
    ref = oracle_rows(wl)
    assert_parity(y, ref, wl.dtype, what=wl.name)
    layer.close()
    return y


def test_worked_example_fp32():
    _check(workloads.worked_example())


def test_handbook_toy_fp32():
    _check(workloads.handbook_toy())


def test_handbook_toy_bf16():
    wl = workloads.handbook_toy()
    wl.x, wl.W = wl.x.to(BF16), wl.W.to(BF16)
    wl.adapters = [(A.to(BF16), B.to(BF16), a) for A, B, a in wl.adapters]
    _check(wl)


@pytest.mark.parametrize("T,K,N", [(300, 520, 328), (129, 64, 64), (128, 128, 256),
                                   (1, 8, 8), (257, 1032, 1040), (640, 256, 8)])
def test_ragged_shapes_bf16(T, K, N):
    wl = workloads.synthetic(100 + T, T, K, N, S=7, ranks=[1, 16, 8, 3, 16, 2, 12], R=16,
                             base_frac=0.2)
    _check(wl)


@pytest.mark.parametrize("layout", ["random", "sorted", "runs"])
def test_layouts_bf16(layout):
    wl = workloads.synthetic(200, 700, 384, 520, S=12, ranks=8, R=8, base_frac=0.15,
                             layout=layout)
    _check(wl)


def test_all_base_only_and_one_slot():
    wl = workloads.synthetic(300, 200, 256, 256, S=3, ranks=16, R=16, base_frac=1.0)
    assert (wl.token_slot == -1).all()
    _check(wl)
    wl = workloads.synthetic(301, 200, 256, 256, S=3, ranks=16, R=16, base_frac=0.0)
    wl.token_slot[:] = 1
    _check(wl)


def test_rank_extremes_and_wide_slots():
    # rank 1 and rank = slot width 128, mixed with padded slots
    wl = workloads.synthetic(302, 300, 512, 384, S=4, ranks=[1, 128, 64, 7], R=128,
                             base_frac=0.1)
    _check(wl)


def test_empty_slot_rows_are_base_only():
    wl = workloads.synthetic(303, 150, 256, 256, S=5, ranks=8, R=8, base_frac=0.1,
                             empty_slots=(2,))
    wl.token_slot[::7] = 2  # rows naming the empty slot
    layer = build_layer(wl)
    y = run_layer(layer, wl)
    assert layer.status() == -4  # LORA_EID, flagged
    ids = wl.token_slot.clone()
    ids[ids == 2] = -1
    table = oracle.SlotTable(wl.adapters, wl.K, wl.N)
    ref = oracle.forward_rows(wl.x, wl.W, table, ids)
    assert_parity(y, ref, BF16, what="empty slot")
    layer.close()


def test_empty_batch_and_single_row():
    wl = workloads.synthetic(304, 1, 256, 128, S=2, ranks=4, R=4, base_frac=0.0)
    _check(wl)
    layer = build_layer(wl)
    layer.set_batch(torch.zeros(0, dtype=torch.int32, device="cuda"))
    x = torch.zeros(0, wl.K, dtype=BF16, device="cuda")
    y = layer.forward(x)
    torch.cuda.synchronize()
    assert y.shape == (0, wl.N) and layer.status() == 0
    layer.close()


def test_reload_and_unload_slot():
    wl = workloads.synthetic(305, 256, 256, 256, S=4, ranks=8, R=16, base_frac=0.0)
    layer = build_layer(wl)
    y0 = run_layer(layer, wl)
    assert_parity(y0, oracle_rows(wl), BF16, what="before reload")
    # replace slot 1 by a new rank-16 adapter, twice (in-flight ordering)
    g = torch.Generator().manual_seed(9)
    for _ in range(2):
        A = (torch.randn(wl.K, 16, generator=g) * 0.02).to(BF16)
        B = (torch.randn(16, wl.N, generator=g) * 0.02).to(BF16)
        layer.load(1, A.cuda(), B.cuda(), 48.0)
        wl.adapters[1] = (A, B, 48.0)
        y1 = run_layer(layer, wl)
    assert_parity(y1, oracle_rows(wl), BF16, what="after reload")
    layer.unload(3)
    y2 = run_layer(layer, wl)
    assert layer.status() == -4
    ids = wl.token_slot.clone()
    ids[ids == 3] = -1
    table = oracle.SlotTable(wl.adapters, wl.K, wl.N)
    assert_parity(y2, oracle.forward_rows(wl.x, wl.W, table, ids), BF16, what="after unload")
    layer.close()


def test_fp32_ragged():
    wl = workloads.synthetic(306, 150, 37, 29, S=3, ranks=[2, 5, 1], R=8, dtype=F32,
                             base_frac=0.2, w_std=0.5)
    _check(wl)
    wl = workloads.synthetic(307, 200, 300, 130, S=5, ranks=16, R=16, dtype=F32,
                             base_frac=0.1, w_std=0.05)
    _check(wl)


def test_deterministic():
    wl = workloads.synthetic(308, 500, 512, 512, S=9, ranks=16, R=16)
    layer = build_layer(wl)
    a = run_layer(layer, wl).clone()
    b = run_layer(layer, wl).clone()
    assert torch.equal(a, b)
    layer.close()


def test_host_buffer_entry_point():
    wl = workloads.synthetic(309, 300, 256, 264, S=5, ranks=8, R=8)
    layer = build_layer(wl)
    x_h = wl.x.clone().pin_memory()
    ids_h = wl.token_slot.clone().pin_memory()
    y_h = torch.empty(wl.T, wl.N, dtype=BF16).pin_memory()
    layer.forward_host(x_h, ids_h, y_h)
    torch.cuda.synchronize()
    assert layer.status() == 0
    assert_parity(y_h, oracle_rows(wl), BF16, what="host entry")
    layer.close()


def test_host_entry_point_concurrent_streams():
    # four layers on four streams, each called several times in turn (as a serving loop
    # rotating independent batches over streams): every call's copies and kernels overlap
    # other layers' work, and every result must still be its own
    streams = [torch.cuda.Stream() for _ in range(4)]
    cases = []
    for i, (T, mode_rows) in enumerate([(200, 8), (700, 16), (64, 8), (1100, 16)]):
        wl = workloads.synthetic(320 + i, T, 264, 392, S=6, ranks=mode_rows, R=16,
                                 base_frac=0.1, layout="runs" if T > 512 else "random")
        layer = build_layer(wl)
        x_h = wl.x.clone().pin_memory()
        ids_h = wl.token_slot.clone().pin_memory()
        outs = [torch.empty(wl.T, wl.N, dtype=BF16).pin_memory() for _ in range(3)]
        cases.append((wl, layer, x_h, ids_h, outs))
    for rep in range(3):
        for (wl, layer, x_h, ids_h, outs), st in zip(cases, streams):
            with torch.cuda.stream(st):
                layer.forward_host(x_h, ids_h, outs[rep], st)
    torch.cuda.synchronize()
    for wl, layer, x_h, ids_h, outs in cases:
        assert layer.status() == 0
        ref = oracle_rows(wl)
        for y_h in outs:
            assert_parity(y_h, ref, BF16, what="concurrent host entry T=%d" % wl.T)
        layer.close()


def test_argument_errors():
    from segmented_rank_gemm_gb300.lora import LoraError, LoraLayer
    wl = workloads.synthetic(310, 64, 64, 64, S=2, ranks=4, R=4)
    layer = LoraLayer(wl.W.cuda(), 2, 4, 64)
    A, B, alpha = wl.adapters[0]
    with pytest.raises(LoraError) as e:
        layer.forward(wl.x.cuda())
    assert e.value.code == -7  # LORA_ESTATE: no batch set
    with pytest.raises(LoraError) as e:
        layer.set_batch(torch.zeros(65, dtype=torch.int32, device="cuda"))
    assert e.value.code == -1  # above max_tokens
    from segmented_rank_gemm_gb300 import lora
    with pytest.raises(LoraError) as e:
        lora.load_adapter_slot(layer.handle, 2, A.cuda(), B.cuda(), 4, alpha)
    assert e.value.code == -2
    with pytest.raises(LoraError) as e:
        lora.load_adapter_slot(layer.handle, 0, A.cuda(), B.cuda(), 5, alpha)
    assert e.value.code == -3
    layer.set_batch(torch.zeros(64, dtype=torch.int32, device="cuda"))
    with pytest.raises(LoraError) as e:
        layer.forward(wl.x.cuda()[:32])
    assert e.value.code == -7  # T differs from the batch
    x = torch.zeros(64 * 64 + 8, dtype=BF16, device="cuda")[1:].view(-1)[: 64 * 64].view(64, 64)
    with pytest.raises(LoraError) as e:
        layer.forward(x)
    assert e.value.code == -1  # misaligned x
    layer.close()


def test_launch_count():
    # the kernels a batch launches, as the layer counts them (the bench's gpu_launches):
    # decode bf16: BGMV + GEMM; prefill: builder + shrink + GEMM; fp32: builder + tile + GEMM;
    # e4m3 decode: + the row quantiser
    from segmented_rank_gemm_gb300.lora import LoraLayer
    cases = [(workloads.synthetic(5101, 64, 256, 256, S=3, ranks=8, R=8), False, 2),
             (workloads.synthetic(5102, 600, 256, 256, S=3, ranks=8, R=8), False, 3),
             (workloads.synthetic(5103, 40, 64, 48, S=3, ranks=4, R=8, dtype=torch.float32),
              False, 3),
             (workloads.synthetic(5104, 64, 256, 256, S=3, ranks=8, R=8), True, 3)]
    for wl, fp8, want in cases:
        if fp8:
            layer = LoraLayer(wl.W.cuda(), wl.S, wl.R, wl.T, fp8_base=True)
            for s, ad in enumerate(wl.adapters):
                layer.load(s, ad[0].cuda(), ad[1].cuda(), ad[2])
        else:
            layer = build_layer(wl)
        try:
            run_layer(layer, wl)
            torch.cuda.synchronize()
            assert layer.status() == 0
            assert layer.launch_count() == want, (wl.name, fp8, layer.launch_count())
        finally:
            layer.close()
