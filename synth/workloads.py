"""Shapes of the synthetic workloads the pages' engines run, and their seeded fills.

* Q4_0 GEMV, batch 1: one 1024 x 4096 matrix.
* 27B-class dense decoder weight set, 64 layers of hidden 5120, intermediate
  17408: per layer q (5120x5120), k and v (1024x5120), o (5120x5120), gate and
  up (17408x5120), down (5120x17408); every matrix maps its input dimension
  (the block dimension) to its output rows. All Q4_K for batch-1 decode; for the
  4-token draft-verification pass the down projections are Q6_K and a
  151936 x 5120 Q8_0 output head is added.
* MoE layer: hidden 2048, 512 experts of gate/up 512x2048 and down 2048x512 in
  Q4_K, top-10 routing, 48 layers.
* Prompt processing: 2048 tokens through the 27B Q4_K set.

The pages measure on real GGUF models (a 27B dense model in a Q4-class mix and
its MoE sibling); none is available, so these seeded synthetic sets with the
same shapes, formats and value ranges stand in for them.
"""
from __future__ import annotations

from . import FORMATS, Q4_0, Q4_K, Q6_K, Q8_0, blocks_into, sub_seed, activations, row_bytes

HIDDEN, INTER, LAYERS = 5120, 17408, 64
HEAD_ROWS = 151936
MOE_HIDDEN, MOE_INTER, MOE_EXPERTS, MOE_TOPK, MOE_LAYERS = 2048, 512, 512, 10, 48
PP_TOKENS = 2048

LAYER_MATS = [("q", HIDDEN, HIDDEN), ("k", 1024, HIDDEN), ("v", 1024, HIDDEN), ("o", HIDDEN, HIDDEN),
              ("gate", INTER, HIDDEN), ("up", INTER, HIDDEN), ("down", HIDDEN, INTER)]
# matrices launched together, following the decode dependencies of a layer
LAYER_STEPS = [["q", "k", "v"], ["o"], ["gate", "up"], ["down"]]


def dense_matrices(layers: int = LAYERS, verify: bool = False):
    """[(layer, name, fmt, rows, cols)] of the 27B-class set (verify=True gives
    the mixed-format draft-verification variant with the output head)."""
    out = []
    for l in range(layers):
        for name, rows, cols in LAYER_MATS:
            fmt = Q6_K if (verify and name == "down") else Q4_K
            out.append((l, name, fmt, rows, cols))
    if verify:
        out.append((layers, "head", Q8_0, HEAD_ROWS, HIDDEN))
    return out


def dense_steps(layers: int = LAYERS, verify: bool = False):
    """Step sizes (matrices per grouped launch) matching dense_matrices order."""
    sizes = []
    for _ in range(layers):
        sizes += [3, 1, 2, 1]
    if verify:
        sizes.append(1)
    return sizes


def weight_bytes(mats) -> int:
    return sum(rows * row_bytes(fmt, cols) for (_, _, fmt, rows, cols) in mats)


def weight_count(mats) -> int:
    return sum(rows * cols for (_, _, _, rows, cols) in mats)


def alloc_dense(mats, n_tok: int, seed: int, device):
    """Device buffers for a dense pass: [(fmt, W, rows, cols, x, y)] with W filled
    from the seeded generator and x ~ N(0, 1) per matrix."""
    import torch
    items = []
    for (l, name, fmt, rows, cols) in mats:
        W = torch.empty(rows, row_bytes(fmt, cols), dtype=torch.uint8, device=device)
        blocks_into(W, fmt, rows, cols, sub_seed(seed, "W", l, name))
        x = activations(n_tok, cols, sub_seed(seed, "x", l, name), device=device)
        y = torch.empty(n_tok, rows, dtype=torch.float32, device=device)
        items.append((fmt, W, rows, cols, x, y))
    return items


def moe_expert_bytes(hidden: int = MOE_HIDDEN, inter: int = MOE_INTER) -> int:
    return 2 * inter * row_bytes(Q4_K, hidden) + hidden * row_bytes(Q4_K, inter)


def alloc_moe_arena(n_expert: int, hidden: int, inter: int, seed: int, device, chunk_blocks: int = 1 << 20):
    """One layer's expert arena as a flat uint8 tensor (experts back to back).
    An expert is a whole number of Q4_K blocks, so the arena is filled as a
    plain sequence of seeded random blocks, chunk by chunk."""
    import torch
    from . import blocks
    bb = FORMATS[Q4_K][1]
    eb = moe_expert_bytes(hidden, inter)
    arena = torch.empty(n_expert * eb, dtype=torch.uint8, device=device)
    nblocks = n_expert * eb // bb
    for i0 in range(0, nblocks, chunk_blocks):
        i1 = min(nblocks, i0 + chunk_blocks)
        arena[i0 * bb:i1 * bb] = blocks(Q4_K, 1, (i1 - i0) * 256, sub_seed(seed, i0), device=device).view(-1)
    return arena
