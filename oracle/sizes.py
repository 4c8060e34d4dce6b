"""Adapter size and compute-share arithmetic, as the pages state it.

TEST INFRASTRUCTURE (part of the oracle package).

- "Multi-LoRA Serving: Architecture for Thousands of Adapters", section "Context and
  Background": one adapted d x k matrix carries r * (d + k) parameters; section "A worked
  memory example" prices rank 16 on four 4096 x 4096 projections over 32 layers.
- "LoRAX, in depth", section "Worked example: how many adapters fit": each projection adds
  r times (d_in + d_out) parameters (the formula after the colon was lost in extraction;
  this is the reading that reproduces the page's printed totals).
- "Multi-LoRA Serving 与 Adapter 隔离", grouped-batch experiment: per-adapter delta
  elements K*r + r*N against K*N full-weight elements.
- "Serving multiple LoRAs ...", section "Not merging the weights, computing in batches":
  rank-16 LoRA costs about 0.5% of the base compute.
"""
from __future__ import annotations

# The 8B-class projection shapes (d_in, d_out) used by the pages' sizing examples:
# hidden 4096, 8 KV heads of dimension 128 (k/v output 1024), MLP width 14336.
LLAMA8B_PROJECTIONS = {
    "q": (4096, 4096),
    "k": (4096, 1024),
    "v": (4096, 1024),
    "o": (4096, 4096),
    "gate": (4096, 14336),
    "up": (4096, 14336),
    "down": (14336, 4096),
}


def adapter_params(shapes, rank: int, layers: int = 1) -> int:
    """Parameters of one adapter: sum over adapted projections of r * (d_in + d_out)."""
    return layers * sum(rank * (d_in + d_out) for d_in, d_out in shapes)


def adapter_bytes(shapes, rank: int, layers: int = 1, bytes_per_param: int = 2) -> int:
    return adapter_params(shapes, rank, layers) * bytes_per_param


def lora_flop_share(shapes, rank: int) -> float:
    """LoRA multiply-adds per token relative to the base multiply-adds per token."""
    lora = sum(rank * (d_in + d_out) for d_in, d_out in shapes)
    base = sum(d_in * d_out for d_in, d_out in shapes)
    return lora / base
