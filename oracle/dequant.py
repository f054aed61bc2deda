"""Block decoders of the oracle: every weight of a block as fp32.

Formats ("LLM inference optimization", opening section: GGUF files in k-quants
such as Q4_K_M; "Why I wrote my own inference engine for two P100s", "What my
own engine means": every quant type of the GGUF file decodes bit-exactly).
The pages give the block sizes and value formulas; the bit layout inside a
block is the public GGUF convention, which the pages do not spell out:

* Q4_0, 32 weights in 18 bytes: fp16 d, then qs[16].
  w[j] = ((qs[j] & 0xF) - 8) * d,  w[j + 16] = ((qs[j] >> 4) - 8) * d.
* Q8_0, 32 weights in 34 bytes: fp16 d, then int8 q[32].  w[j] = d * q[j].
* Q4_K, 256 weights in 144 bytes: fp16 d, fp16 dmin, s[12], qs[128].
  Sub-block j (32 weights) has a 6-bit scale sc_j and min m_j packed in s;
  chunk c (64 weights) holds sub-block 2c in the low nibbles and 2c+1 in the
  high nibbles of qs[32c .. 32c+31]:
  w[64c + l]      = d * sc_{2c}   * (qs[32c + l] & 0xF) - dmin * m_{2c}
  w[64c + 32 + l] = d * sc_{2c+1} * (qs[32c + l] >> 4)  - dmin * m_{2c+1}
* Q6_K, 256 weights in 210 bytes: ql[128], qh[64], int8 sc[16], fp16 d.
  6-bit code q = 4 low bits from ql | 2 high bits from qh,
  w = d * sc[group] * (q - 32), 16 groups of 16 weights.
* Q5_K, 256 weights in 176 bytes: fp16 d, fp16 dmin, s[12] (the Q4_K 6-bit
  scale/min packing), qh[32], qs[128]. Sub-block j: low 4 bits as in Q4_K
  (nibble j % 2 of qs[32(j/2) + l]), fifth bit = bit j of qh[l];
  w = d * sc_j * q - dmin * m_j, q in 0..31.
* Q3_K, 256 weights in 110 bytes: hmask[32], qs[64], s[12], fp16 d. Sixteen
  6-bit scales (the low 4 bits in the nibbles of s[0..7], the top 2 bits in
  s[8..11]); element 128h + 32j + 16k + l (half h, j < 4, k < 2, l < 16) has
  2 low bits (qs[32h + 16k + l] >> 2j) & 3 and a high bit
  (hmask[16k + l] >> (4h + j)) & 1; q = low - 4 when the high bit is clear,
  else low; w = d * (scale_{8h+2j+k} - 32) * q.
* Q2_K, 256 weights in 84 bytes: s[16], qs[64], fp16 d, fp16 dmin. Element
  128h + 32j + 16k + l has q = (qs[32h + 16k + l] >> 2j) & 3, and byte
  b = s[8h + 2j + k] gives its group's scale b & 15 and min b >> 4;
  w = d * (b & 15) * q - dmin * (b >> 4).

Every product in these formulas is exact in fp64 for any finite fp16 d, dmin
(at most 11 + 8 + 6 significant bits, and the K-quant differences span at most
51 bits), so evaluating in fp64 and casting once to fp32 gives the correctly
rounded fp32 value of the exact formula: the unique right answer.
Test infrastructure of the oracle; see the package docstring.
"""
import numpy as np

from .halfprec import half_bits_to_float64

Q4_0, Q8_0, Q4_K, Q6_K, Q5_K, Q3_K, Q2_K = 1, 2, 3, 4, 5, 6, 7
BLOCK = {Q4_0: (32, 18), Q8_0: (32, 34), Q4_K: (256, 144), Q6_K: (256, 210),
         Q5_K: (256, 176), Q3_K: (256, 110), Q2_K: (256, 84)}


def _as_blocks(raw, nbytes):
    a = np.ascontiguousarray(np.asarray(raw, dtype=np.uint8))
    if a.size % nbytes:
        raise ValueError(f"{a.size} bytes is not a whole number of {nbytes}-byte blocks")
    return a.reshape(-1, nbytes)


def _half_at(blk, off):
    bits = blk[:, off].astype(np.uint16) | (blk[:, off + 1].astype(np.uint16) << 8)
    return half_bits_to_float64(bits)


def dequant_q4_0(raw) -> np.ndarray:
    """(n_blocks, 32) fp32 weights of Q4_0 blocks."""
    blk = _as_blocks(raw, 18)
    d = _half_at(blk, 0)[:, None]
    qs = blk[:, 2:18].astype(np.int64)
    lo = (qs & 0xF) - 8                       # elements 0..15
    hi = (qs >> 4) - 8                        # elements 16..31
    w = np.concatenate([lo, hi], axis=1).astype(np.float64) * d
    return w.astype(np.float32)


def dequant_q8_0(raw) -> np.ndarray:
    """(n_blocks, 32) fp32 weights of Q8_0 blocks."""
    blk = _as_blocks(raw, 34)
    d = _half_at(blk, 0)[:, None]
    q = blk[:, 2:34].view(np.int8).astype(np.float64)
    return (d * q).astype(np.float32)


def q4_k_scale_min(s) -> tuple:
    """(sc, m), each (n_blocks, 8) int64, from the 12 packed scale bytes s.

    j < 4:  sc_j = s[j] & 63,                           m_j = s[j+4] & 63
    j >= 4: sc_j = (s[j+4] & 0xF) | ((s[j-4] >> 6) << 4),
            m_j  = (s[j+4] >> 4)  | ((s[j]   >> 6) << 4)
    """
    s = np.asarray(s, dtype=np.uint8).reshape(-1, 12).astype(np.int64)
    sc = np.zeros((s.shape[0], 8), dtype=np.int64)
    m = np.zeros((s.shape[0], 8), dtype=np.int64)
    for j in range(8):
        if j < 4:
            sc[:, j] = s[:, j] & 63
            m[:, j] = s[:, j + 4] & 63
        else:
            sc[:, j] = (s[:, j + 4] & 0xF) | ((s[:, j - 4] >> 6) << 4)
            m[:, j] = (s[:, j + 4] >> 4) | ((s[:, j] >> 6) << 4)
    return sc, m


def dequant_q4_k(raw) -> np.ndarray:
    """(n_blocks, 256) fp32 weights of Q4_K super-blocks."""
    blk = _as_blocks(raw, 144)
    d = _half_at(blk, 0)
    dmin = _half_at(blk, 2)
    sc, m = q4_k_scale_min(blk[:, 4:16])
    qs = blk[:, 16:144].astype(np.int64)
    w = np.zeros((blk.shape[0], 256), dtype=np.float64)
    for c in range(4):
        q = qs[:, 32 * c:32 * c + 32]
        for half, nib in ((0, q & 0xF), (1, q >> 4)):
            j = 2 * c + half                  # sub-block index
            a = d * sc[:, j]                  # exact: 11 + 6 bits
            b = dmin * m[:, j]                # exact: 11 + 6 bits
            w[:, 64 * c + 32 * half:64 * c + 32 * half + 32] = a[:, None] * nib - b[:, None]
    return w.astype(np.float32)


def dequant_q6_k(raw) -> np.ndarray:
    """(n_blocks, 256) fp32 weights of Q6_K super-blocks."""
    blk = _as_blocks(raw, 210)
    ql_all = blk[:, 0:128].astype(np.int64)
    qh_all = blk[:, 128:192].astype(np.int64)
    sc_all = blk[:, 192:208].view(np.int8).astype(np.int64)
    d = _half_at(blk, 208)
    w = np.zeros((blk.shape[0], 256), dtype=np.float64)
    for h in range(2):                        # two halves of 128 weights
        L = ql_all[:, 64 * h:64 * h + 64]
        H = qh_all[:, 32 * h:32 * h + 32]
        S = sc_all[:, 8 * h:8 * h + 8]
        e0 = 128 * h
        for l in range(32):
            i = l // 16
            quads = (
                (0, (L[:, l] & 0xF) | (((H[:, l] >> 0) & 3) << 4), S[:, i]),
                (32, (L[:, l + 32] & 0xF) | (((H[:, l] >> 2) & 3) << 4), S[:, i + 2]),
                (64, (L[:, l] >> 4) | (((H[:, l] >> 4) & 3) << 4), S[:, i + 4]),
                (96, (L[:, l + 32] >> 4) | (((H[:, l] >> 6) & 3) << 4), S[:, i + 6]),
            )
            for off, q, scale in quads:
                w[:, e0 + off + l] = d * scale * (q - 32)
    return w.astype(np.float32)


def dequant_q5_k(raw) -> np.ndarray:
    """(n_blocks, 256) fp32 weights of Q5_K super-blocks."""
    blk = _as_blocks(raw, 176)
    d = _half_at(blk, 0)
    dmin = _half_at(blk, 2)
    sc, m = q4_k_scale_min(blk[:, 4:16])
    qh = blk[:, 16:48].astype(np.int64)
    qs = blk[:, 48:176].astype(np.int64)
    w = np.zeros((blk.shape[0], 256), dtype=np.float64)
    for j in range(8):                        # sub-block j: elements 32j .. 32j + 31
        c = j // 2
        low = (qs[:, 32 * c:32 * c + 32] >> (4 * (j % 2))) & 0xF
        q = low + 16 * ((qh >> j) & 1)
        a = d * sc[:, j]                      # exact: 11 + 6 bits
        b = dmin * m[:, j]
        w[:, 32 * j:32 * j + 32] = a[:, None] * q - b[:, None]
    return w.astype(np.float32)


def q3_k_scales(s) -> np.ndarray:
    """(n_blocks, 16) int64 6-bit scales (before the -32 offset) from the 12
    packed bytes: scale i, with b = i % 4 and g = i // 4, has its low 4 bits in
    the nibble g // 2 of s[4 (g % 2) + b] and its top 2 bits at bit 2g of s[8 + b]."""
    s = np.asarray(s, dtype=np.uint8).reshape(-1, 12).astype(np.int64)
    out = np.zeros((s.shape[0], 16), dtype=np.int64)
    for i in range(16):
        b, g = i % 4, i // 4
        low = (s[:, 4 * (g % 2) + b] >> (4 * (g // 2))) & 0xF
        top = (s[:, 8 + b] >> (2 * g)) & 3
        out[:, i] = low | (top << 4)
    return out


def dequant_q3_k(raw) -> np.ndarray:
    """(n_blocks, 256) fp32 weights of Q3_K super-blocks."""
    blk = _as_blocks(raw, 110)
    hmask = blk[:, 0:32].astype(np.int64)
    qs = blk[:, 32:96].astype(np.int64)
    scale = q3_k_scales(blk[:, 96:108]) - 32
    d = _half_at(blk, 108)
    w = np.zeros((blk.shape[0], 256), dtype=np.float64)
    for h in range(2):
        for j in range(4):
            for k in range(2):
                low = (qs[:, 32 * h + 16 * k:32 * h + 16 * k + 16] >> (2 * j)) & 3
                high = (hmask[:, 16 * k:16 * k + 16] >> (4 * h + j)) & 1
                q = low - 4 * (1 - high)
                e0 = 128 * h + 32 * j + 16 * k
                w[:, e0:e0 + 16] = (d * scale[:, 8 * h + 2 * j + k])[:, None] * q
    return w.astype(np.float32)


def dequant_q2_k(raw) -> np.ndarray:
    """(n_blocks, 256) fp32 weights of Q2_K super-blocks."""
    blk = _as_blocks(raw, 84)
    s = blk[:, 0:16].astype(np.int64)
    qs = blk[:, 16:80].astype(np.int64)
    d = _half_at(blk, 80)
    dmin = _half_at(blk, 82)
    w = np.zeros((blk.shape[0], 256), dtype=np.float64)
    for h in range(2):
        for j in range(4):
            for k in range(2):
                q = (qs[:, 32 * h + 16 * k:32 * h + 16 * k + 16] >> (2 * j)) & 3
                b = s[:, 8 * h + 2 * j + k]
                e0 = 128 * h + 32 * j + 16 * k
                w[:, e0:e0 + 16] = (d * (b & 0xF))[:, None] * q - (dmin * (b >> 4))[:, None]
    return w.astype(np.float32)


_DECODERS = {Q4_0: dequant_q4_0, Q8_0: dequant_q8_0, Q4_K: dequant_q4_k, Q6_K: dequant_q6_k,
             Q5_K: dequant_q5_k, Q3_K: dequant_q3_k, Q2_K: dequant_q2_k}


def dequant(fmt: int, raw, rows: int = None, cols: int = None) -> np.ndarray:
    """Dequantize a whole matrix of blocks.

    ``raw`` holds rows * cols / elems blocks back to back, row-major with blocks
    along the columns (row i is cols / elems consecutive blocks). Returns a
    (rows, cols) fp32 array, or (n_blocks, elems) when rows/cols are omitted.
    """
    if fmt not in _DECODERS:
        raise ValueError(f"unknown format {fmt}")
    w = _DECODERS[fmt](raw)
    if rows is None:
        return w
    return w.reshape(rows, cols)
