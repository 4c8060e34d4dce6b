"""Ordering and failure handling on the GPU, without faulting it.

- A slot reloaded right after a forward that reads it was enqueued (no host
  synchronisation in between): the forward must see the old adapter, the next forward the
  new one -- the reload waits for the forward ("Multi-LoRA Serving 与 Adapter 隔离",
  failure modes: an adapter evicted while an in-flight kernel still uses its storage).
- A layer destroyed with forwards still in flight: destruction synchronises first, so the
  outputs are complete and correct.
- The bounded waits: a flag nothing sets and an mbarrier phase nobody completes both give
  up after their bound and report LORA_ETIMEOUT, and the context stays usable.
"""
import pytest
import torch

from segmented_rank_gemm_gb300 import workloads
from gpu_helpers import assert_parity, oracle_rows

pytestmark = pytest.mark.gpu
BF16 = torch.bfloat16


def _layer(wl):
    from segmented_rank_gemm_gb300.lora import LoraLayer
    layer = LoraLayer(wl.W.cuda(), wl.S, wl.R, wl.T)
    for s, (A, B, alpha) in enumerate(wl.adapters):
        layer.load(s, A.cuda(), B.cuda(), alpha)
    torch.cuda.synchronize()
    return layer


@pytest.mark.parametrize("T", [256, 1024])  # decode (delta) and prefill (v mode)
def test_reload_behind_an_inflight_forward(T):
    wl = workloads.synthetic(400 + T, T, 2048, 2048, S=3, ranks=16, R=16, base_frac=0.0)
    layer = _layer(wl)
    stream = torch.cuda.Stream()
    g = torch.Generator().manual_seed(T)
    new = [((torch.randn(wl.K, 16, generator=g) * 0.02).to(BF16),
            (torch.randn(16, wl.N, generator=g) * 0.02).to(BF16), 40.0) for _ in range(2)]
    side = torch.cuda.Stream()
    new_dev = [(A.cuda(), B.cuda(), alpha) for A, B, alpha in new]
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        x, ids = wl.x.cuda(), wl.token_slot.cuda()
        y_old = layer(x, ids, stream=stream)
    # reload slots 0 and 1 on another stream right away, no host wait
    for s in (0, 1):
        layer.load(s, new_dev[s][0], new_dev[s][1], new_dev[s][2], side_stream=side)
    with torch.cuda.stream(stream):
        y_new = layer(x, ids, stream=stream)
    torch.cuda.synchronize()
    assert layer.status(stream) == 0
    assert_parity(y_old, oracle_rows(wl), BF16, what="forward enqueued before the reload")
    wl.adapters[0], wl.adapters[1] = new[0], new[1]
    assert_parity(y_new, oracle_rows(wl), BF16, what="forward after the reload")
    layer.close()


def test_destroy_with_forwards_in_flight():
    wl = workloads.synthetic(410, 512, 2048, 4096, S=8, ranks=16, R=16)
    layer = _layer(wl)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        x, ids = wl.x.cuda(), wl.token_slot.cuda()
        ys = [layer(x, ids, stream=stream) for _ in range(4)]
    layer.close()  # no host synchronisation before: destroy waits for the forwards
    for y in ys:
        assert_parity(y, oracle_rows(wl), BF16, what="output of a forward in flight at destroy")


@pytest.mark.parametrize("which", [0, 1])  # a global flag / an mbarrier phase
def test_bounded_wait_gives_up_and_context_stays_usable(which):
    from segmented_rank_gemm_gb300.lora import LORA_ETIMEOUT, lora_wait_selftest
    assert lora_wait_selftest(which) == LORA_ETIMEOUT
    wl = workloads.synthetic(420, 200, 256, 192, S=4, ranks=8, R=8)
    layer = _layer(wl)
    y = layer(wl.x.cuda(), wl.token_slot.cuda())
    torch.cuda.synchronize()
    assert layer.status() == 0
    assert_parity(y, oracle_rows(wl), BF16, what="forward after a timed-out wait")
    layer.close()
