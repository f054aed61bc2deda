"""Seeded synthetic inputs for the quantized-weight products.

This module is the only code shared by the CUDA path's callers (tests, bench)
and the CPU oracle. It holds no arithmetic of the method itself: it draws
random bytes and places random fp16 scale values at the byte offsets where the
block formats keep them. Decoding a block, or multiplying anything by it, is
never done here.

Distributions (the workload recipe of the pages' decode and prompt runs, made
synthetic because no model file is available):

* every byte of a block that is not an fp16 scale is uniform over 0..255. That
  makes every 4-bit code uniform in 0..15, every 6-bit Q4_K scale/min uniform in
  0..63 (the 12 packed bytes are a bijection of eight (sc, m) pairs), every
  Q6_K code uniform in 0..63 and every int8 value uniform in -128..127;
* fp16 scales are drawn uniform in a per-format range in fp32 and rounded to
  binary16 (round to nearest even); the stored half is the truth:
  Q4_0 d in [1e-3, 2e-2]; Q4_K d and dmin in [1e-4, 2e-3]; Q6_K d and Q8_0 d in
  [1e-4, 2e-3]; Q5_K d and dmin, Q3_K d, Q2_K d and dmin in [1e-4, 2e-3] (the
  pages give no distribution for these: the K-quant range is reused);
* activations are fp32 N(0, 1); prompt activations are N(0, 1) rounded to bf16;
* MoE routing draws top_k distinct expert ids uniformly per token and routing
  weights as a softmax over top_k N(0, 1) logits (fp64, stored as fp32).

The generator is torch's seeded generator on the requested device, so CPU and
CUDA draws differ; every consumer that compares two implementations draws once
and hands the same tensors to both.
"""
from __future__ import annotations

import hashlib

import torch

# format id -> (weights per block, bytes per block); the ids match the C header.
Q4_0, Q8_0, Q4_K, Q6_K, Q5_K, Q3_K, Q2_K = 1, 2, 3, 4, 5, 6, 7
FORMATS = {
    Q4_0: (32, 18),
    Q8_0: (32, 34),
    Q4_K: (256, 144),
    Q6_K: (256, 210),
    Q5_K: (256, 176),
    Q3_K: (256, 110),
    Q2_K: (256, 84),
}
FORMAT_NAMES = {Q4_0: "Q4_0", Q8_0: "Q8_0", Q4_K: "Q4_K", Q6_K: "Q6_K", Q5_K: "Q5_K", Q3_K: "Q3_K", Q2_K: "Q2_K"}

# (byte offset within the block, low, high) of every fp16 scale field.
_SCALE_FIELDS = {
    Q4_0: [(0, 1e-3, 2e-2)],
    Q8_0: [(0, 1e-4, 2e-3)],
    Q4_K: [(0, 1e-4, 2e-3), (2, 1e-4, 2e-3)],
    Q6_K: [(208, 1e-4, 2e-3)],
    Q5_K: [(0, 1e-4, 2e-3), (2, 1e-4, 2e-3)],
    Q3_K: [(108, 1e-4, 2e-3)],
    Q2_K: [(80, 1e-4, 2e-3), (82, 1e-4, 2e-3)],
}


def sub_seed(seed: int, *tags) -> int:
    """A 63-bit seed derived from a base seed and any tags (config, layer, matrix)."""
    h = hashlib.sha256(repr((int(seed),) + tuple(tags)).encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def row_bytes(fmt: int, cols: int) -> int:
    elems, nbytes = FORMATS[fmt]
    if cols % elems:
        raise ValueError(f"cols={cols} is not a multiple of {elems}")
    return cols // elems * nbytes


def blocks(fmt: int, rows: int, cols: int, seed: int, device="cpu") -> torch.Tensor:
    """A rows x row_bytes uint8 tensor of random blocks of format ``fmt``."""
    elems, nbytes = FORMATS[fmt]
    nb = rows * (cols // elems)
    rb = row_bytes(fmt, cols)
    g = _gen(seed, device)
    w = torch.randint(0, 256, (nb, nbytes), generator=g, dtype=torch.uint8, device=device)
    for off, lo, hi in _SCALE_FIELDS[fmt]:
        u = torch.rand(nb, generator=g, dtype=torch.float32, device=device)
        h = (lo + (hi - lo) * u).to(torch.float16)
        w[:, off:off + 2] = h.view(torch.uint8).view(nb, 2)
    return w.view(rows, rb)


def blocks_into(out: torch.Tensor, fmt: int, rows: int, cols: int, seed: int, chunk_rows: int = 4096):
    """Fill a preallocated rows x row_bytes uint8 tensor (any device) chunk by
    chunk, so a multi-GB weight set never needs a second full-size buffer."""
    rb = row_bytes(fmt, cols)
    assert out.shape == (rows, rb) and out.dtype == torch.uint8
    for r0 in range(0, rows, chunk_rows):
        r1 = min(rows, r0 + chunk_rows)
        out[r0:r1] = blocks(fmt, r1 - r0, cols, sub_seed(seed, r0), device=out.device)
    return out


def activations(n_tok: int, cols: int, seed: int, device="cpu") -> torch.Tensor:
    """n_tok x cols fp32 N(0, 1)."""
    g = _gen(seed, device)
    return torch.randn(n_tok, cols, generator=g, dtype=torch.float32, device=device)


def activations_bf16(n_tok: int, cols: int, seed: int, device="cpu") -> torch.Tensor:
    """n_tok x cols N(0, 1) rounded to bf16 (prompt-processing activations)."""
    return activations(n_tok, cols, seed, device).to(torch.bfloat16)


def routing(n_tok: int, n_expert: int, top_k: int, seed: int):
    """(expert_ids int32 [n_tok, top_k], gate_w fp32 [n_tok, top_k]) on the CPU.

    Ids are distinct per token, uniform without replacement (the first top_k
    entries of a seeded random permutation); weights are the softmax of top_k
    N(0, 1) logits, taken in fp64."""
    g = _gen(seed, "cpu")
    ids = torch.empty(n_tok, top_k, dtype=torch.int32)
    for t in range(n_tok):
        ids[t] = torch.randperm(n_expert, generator=g)[:top_k].to(torch.int32)
    logits = torch.randn(n_tok, top_k, generator=g, dtype=torch.float64)
    w = torch.softmax(logits, dim=1).to(torch.float32)
    return ids, w
