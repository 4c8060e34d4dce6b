"""Shared helpers of the GPU parity tests: drive the layer through the C ABI binding and
compare with the CPU oracle element by element."""
from __future__ import annotations

import numpy as np
import torch

import oracle

# Tolerances of the parity bar: max |err| <= tol * (1 + |ref|)
TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}


def build_layer(wl, device="cuda", max_tokens=None, max_rank=None, num_slots=None):
    from segmented_rank_gemm_gb300.lora import LoraLayer
    layer = LoraLayer(wl.W.to(device), num_slots or wl.S, max_rank or wl.R,
                      max_tokens or max(wl.T, 1))
    for s, ad in enumerate(wl.adapters):
        if ad is None:
            continue
        A, B, alpha = ad
        layer.load(s, A.to(device), B.to(device), alpha)
    return layer


def run_layer(layer, wl, device="cuda"):
    x = wl.x.to(device)
    ids = wl.token_slot.to(device)
    y = layer(x, ids)
    torch.cuda.synchronize()
    return y


def oracle_rows(wl, rows=None):
    table = oracle.SlotTable(wl.adapters, wl.K, wl.N)
    return oracle.forward_rows(wl.x, wl.W, table, wl.token_slot, rows=rows)


def assert_parity(y_gpu, ref, dtype, strict=True, what=""):
    """The bar: |y - ref| <= tol (1 + |ref|) everywhere.  ``strict`` adds a tighter check
    that holds for a correct kernel (one rounding of the fp32 result to the output dtype
    plus fp32 accumulation error) and catches small systematic mistakes."""
    y = y_gpu.detach().float().cpu().double().numpy() if hasattr(y_gpu, "detach") else y_gpu
    ref = np.asarray(ref, dtype=np.float64)
    assert y.shape == ref.shape, (y.shape, ref.shape)
    assert np.all(np.isfinite(y)), what + ": non-finite output"
    tol = TOL[dtype]
    err = np.abs(y - ref)
    bar = tol * (1.0 + np.abs(ref))
    worst = float((err / (1.0 + np.abs(ref))).max()) if err.size else 0.0
    assert np.all(err <= bar), "%s: parity bar broken, max err/(1+|ref|) = %.3g > %g" % (
        what, worst, tol)
    if strict:
        if dtype == torch.bfloat16:
            lim = 2.0 ** -8 * np.abs(ref) + 2e-3
        else:
            lim = 2e-6 * (1.0 + np.abs(ref))
        bad = int((err > lim).sum())
        assert bad == 0, "%s: %d elements beyond one rounding (worst %.3g)" % (
            what, bad, float((err - lim).max()))
    return worst
