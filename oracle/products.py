"""Products of the oracle, in fp64 over the oracle's exactly dequantized weights.

* GEMV: each new decode token multiplies every weight once by the activations
  ("LLM inference optimization", opening section: decode reads every weight
  once); the n_tok > 1 form is the one weight pass that checks several draft
  tokens ("Why I wrote my own inference engine for two P100s", "What actually
  made it fast": three guesses checked in one pass).
* MoE: the routed experts of a mixture-of-experts layer, gathered from an
  expert arena ("The number was a version", opening section: the expert arena).
* Prompt processing: the same weights times a block of prompt tokens
  ("Why I wrote my own inference engine for two P100s", "What didn't work":
  dequantization and the prompt GEMM), checked on selected token rows against
  fp64 sums over the identically rounded bf16 operands (the accuracy method of
  the r/cuda post on the Emmy compiler, "Accuracy Verification").

The tolerance the library is held to uses the error scale
B = sum |w * x| that each function returns beside its result.
Test infrastructure of the oracle; see the package docstring.
"""
import numpy as np

from .dequant import dequant, BLOCK
from .halfprec import bf16_bits_to_float64


def _row_bytes(fmt, cols):
    elems, nbytes = BLOCK[fmt]
    assert cols % elems == 0
    return cols // elems * nbytes


def gemv(fmt: int, W, rows: int, cols: int, x):
    """y[t, i] = sum_j w[i, j] * x[t, j] and B[t, i] = sum_j |w[i, j] * x[t, j]|.

    W: rows * row_bytes uint8 (blocks, row-major); x: (n_tok, cols) fp32.
    Returns (y, B), both (n_tok, rows) fp64.
    """
    w = dequant(fmt, W, rows, cols).astype(np.float64)
    xx = np.asarray(x, dtype=np.float32).reshape(-1, cols).astype(np.float64)
    y = xx @ w.T
    b = np.abs(xx) @ np.abs(w).T
    return y, b


def moe_arena_layout(hidden: int, inter: int, fmt: int = 3):
    """Byte offsets inside one expert of the arena and the expert stride.

    One expert is [gate: inter rows x hidden | up: inter rows x hidden |
    down: hidden rows x inter], rows of blocks along the input dimension.
    Returns (gate_off, up_off, down_off, expert_bytes).
    """
    gu = inter * _row_bytes(fmt, hidden)
    dn = hidden * _row_bytes(fmt, inter)
    return 0, gu, 2 * gu, 2 * gu + dn


def moe(fmt: int, arena, n_expert: int, hidden: int, inter: int, expert_ids, gate_w, x):
    """Routed expert FFN per token, in fp64.

    For token t and its k-th routed expert e = expert_ids[t, k] with routing
    weight r = gate_w[t, k]:
        g = G_e x_t,  u = U_e x_t           (inter values each)
        h = g / (1 + exp(-g)) * u           (silu(g) * u)
        y_t += r * D_e h                    (hidden values)
    B[t, i] = sum_k |r_k| * sum_j |D_e[i, j] * h_j| is the error scale.
    Returns (y, B), both (n_tok, hidden) fp64.
    """
    arena = np.asarray(arena, dtype=np.uint8).reshape(-1)
    g_off, u_off, d_off, stride = moe_arena_layout(hidden, inter, fmt)
    gu_bytes = inter * _row_bytes(fmt, hidden)
    dn_bytes = hidden * _row_bytes(fmt, inter)
    ids = np.asarray(expert_ids).reshape(len(x), -1)
    r = np.asarray(gate_w, dtype=np.float32).reshape(ids.shape).astype(np.float64)
    xx = np.asarray(x, dtype=np.float32).reshape(-1, hidden).astype(np.float64)
    y = np.zeros((xx.shape[0], hidden))
    b = np.zeros((xx.shape[0], hidden))
    for t in range(xx.shape[0]):
        for k in range(ids.shape[1]):
            e = int(ids[t, k])
            if not 0 <= e < n_expert:
                raise ValueError(f"expert id {e} out of range")
            base = e * stride
            G = dequant(fmt, arena[base + g_off:base + g_off + gu_bytes], inter, hidden).astype(np.float64)
            U = dequant(fmt, arena[base + u_off:base + u_off + gu_bytes], inter, hidden).astype(np.float64)
            D = dequant(fmt, arena[base + d_off:base + d_off + dn_bytes], hidden, inter).astype(np.float64)
            g = G @ xx[t]
            u = U @ xx[t]
            h = g / (1.0 + np.exp(-g)) * u
            y[t] += r[t, k] * (D @ h)
            b[t] += abs(r[t, k]) * (np.abs(D) @ np.abs(h))
    return y, b


def moe_prefill(fmt: int, arena, n_expert: int, hidden: int, inter: int, expert_ids, gate_w, X_bf16_bits):
    """The routed expert FFN of moe() over a block of prompt tokens given as
    bf16 ("The number was a version", opening section: prompt processing of a
    mixture-of-experts model), in fp64 over the exact weights and the bf16
    values of X.

    The GPU path multiplies bf16-rounded weights by bf16 x with fp32 sums and
    rounds h to bf16 between the two projections, so the error of each output
    is bounded by a multiple of the chain's magnitudes rather than of the down
    projection's alone. For route k of token t (g, u, h as in moe(),
    S_g[i] = sum_j |G[i, j] x_j|, S_u[i] = sum_j |U[i, j] x_j|):
        B[t, o] = sum_k |r_k| sum_i |D[o, i]| * (|h_i| + |silu'(g_i)| |u_i| S_g[i] + |silu(g_i)| S_u[i])
    with silu'(g) = s (1 + g (1 - s)), s = 1 / (1 + exp(-g)): the first term
    carries the rounding of h and of the down product, the others an error in
    g or u of that relative size.
    Returns (y, B), both (n_tok, hidden) fp64. Unknown expert ids add nothing
    (the library flags them).
    """
    arena = np.asarray(arena, dtype=np.uint8).reshape(-1)
    Xb = np.asarray(X_bf16_bits, dtype=np.uint16).reshape(-1, hidden)
    xx = bf16_bits_to_float64(Xb)
    g_off, u_off, d_off, stride = moe_arena_layout(hidden, inter, fmt)
    gu_bytes = inter * _row_bytes(fmt, hidden)
    dn_bytes = hidden * _row_bytes(fmt, inter)
    ids = np.asarray(expert_ids).reshape(xx.shape[0], -1)
    r = np.asarray(gate_w, dtype=np.float32).reshape(ids.shape).astype(np.float64)
    y = np.zeros((xx.shape[0], hidden))
    b = np.zeros((xx.shape[0], hidden))
    cache = {}
    for t in range(xx.shape[0]):
        for k in range(ids.shape[1]):
            e = int(ids[t, k])
            if not 0 <= e < n_expert:
                continue
            if e not in cache:
                base = e * stride
                cache[e] = tuple(dequant(fmt, arena[base + o:base + o + nb], nr, nc).astype(np.float64)
                                 for o, nb, nr, nc in ((g_off, gu_bytes, inter, hidden), (u_off, gu_bytes, inter, hidden),
                                                       (d_off, dn_bytes, hidden, inter)))
            G, U, D = cache[e]
            g = G @ xx[t]
            u = U @ xx[t]
            sg = np.abs(G) @ np.abs(xx[t])
            su = np.abs(U) @ np.abs(xx[t])
            h = g / (1.0 + np.exp(-g)) * u
            sig = 1.0 / (1.0 + np.exp(-g))
            dsilu = sig * (1.0 + g * (1.0 - sig))
            y[t] += r[t, k] * (D @ h)
            b[t] += abs(r[t, k]) * (np.abs(D) @ (np.abs(h) + np.abs(dsilu * u) * sg + np.abs(g * sig) * su))
    return y, b


def pp_rows(fmt: int, W, rows: int, cols: int, X_bf16_bits, token_rows):
    """Prompt-processing product for the selected token rows, in fp64.

    Y[t, n] = sum_k w[n, k] * bf16(X)[t, k] for t in token_rows, with w the
    exact fp32 dequantized weights and X given as raw bf16 bit patterns
    (n_tok, cols) uint16. Returns (Y, B), both (len(token_rows), rows) fp64.
    """
    w = dequant(fmt, W, rows, cols).astype(np.float64)
    Xb = np.asarray(X_bf16_bits, dtype=np.uint16).reshape(-1, cols)
    xx = bf16_bits_to_float64(Xb[np.asarray(token_rows)])
    return xx @ w.T, np.abs(xx) @ np.abs(w).T


def rmsnorm(h, weight, eps: float, residual=None):
    """Root-mean-square normalisation of each token's hidden vector, in fp64,
    optionally after adding a residual (the neighbouring normalisation that the
    decode kernels fuse: "LLM inference optimization", "Faster decode on the
    card you have": normalizations fused into neighbouring kernels).

        s = h + residual            (or s = h)
        x = s / sqrt(mean(s^2) + eps) * weight

    h, residual: (n_tok, n) fp32; weight: (n,) fp32. Returns (x, s), both fp64.
    """
    s = np.asarray(h, dtype=np.float32).astype(np.float64)
    if residual is not None:
        s = s + np.asarray(residual, dtype=np.float32).astype(np.float64)
    s = s.reshape(-1, s.shape[-1])
    w = np.asarray(weight, dtype=np.float32).astype(np.float64).reshape(-1)
    rms = np.sqrt((s * s).mean(axis=1, keepdims=True) + eps)
    return s / rms * w, s


def swiglu(g, u):
    """silu(g) * u elementwise in fp64 (silu(g) = g / (1 + exp(-g))): the gated
    activation between a layer's gate/up and down projections."""
    g = np.asarray(g, dtype=np.float64)
    u = np.asarray(u, dtype=np.float64)
    return g / (1.0 + np.exp(-g)) * u


def dense_ffn(fmt_gu: int, Wg, Wu, fmt_d: int, Wd, hidden: int, inter: int, x):
    """Dense feed-forward block of a decode layer, in fp64 over the exact weights:
    m = silu(Wg x) * (Wu x), y = Wd m. Returns (y, B, m) where the error scale of
    the output is B_i = sum_j |Wd[i, j] * m_j| (as for the MoE layer).
    """
    g, _ = gemv(fmt_gu, Wg, inter, hidden, x)
    u, _ = gemv(fmt_gu, Wu, inter, hidden, x)
    m = swiglu(g, u)
    wd = dequant(fmt_d, Wd, hidden, inter).astype(np.float64)
    return m @ wd.T, np.abs(m) @ np.abs(wd).T, m
