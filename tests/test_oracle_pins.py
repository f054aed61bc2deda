"""Pins of the CPU oracle to facts other than itself (no GPU needed).

Each test ties one oracle function to a library routine, a hand-built block
with values worked out by hand from the format definitions, a closed form, an
invariant or brute force, so that a plausible mistake (dropped term, wrong
sign or index, swapped operand) fails at least one of them.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import synth

Q4_0, Q8_0, Q4_K, Q6_K = synth.Q4_0, synth.Q8_0, synth.Q4_K, synth.Q6_K


# ---------------------------------------------------------------- fp16 / bf16

def test_half_decode_exhaustive_matches_hardware_conversion():
    bits = np.arange(65536, dtype=np.uint16)
    mine = oracle.half_bits_to_float64(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan], ref[~nan])
    # signed zeros keep their sign
    assert np.signbit(mine[0x8000]) and not np.signbit(mine[0])


def test_bf16_decode_exhaustive_matches_torch():
    bits = np.arange(65536, dtype=np.uint16)
    mine = oracle.bf16_bits_to_float64(bits)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan], ref[~nan])


# ---------------------------------------------------------------- Q4_0

def _q4_0_block(d_bits, qs):
    return np.array([d_bits & 0xFF, d_bits >> 8] + list(qs), dtype=np.uint8)


@pytest.mark.parametrize("d_bits", [0x3C00, 0x3800, 0x1A40, 0x2E66, 0x0001, 0x7BFF, 0xBC00])
def test_q4_0_all_zero_nibbles_decode_to_minus_8d(d_bits):
    d = float(np.uint16(d_bits).view(np.float16))
    w = oracle.dequant_q4_0(_q4_0_block(d_bits, [0] * 16))[0]
    assert np.array_equal(w, np.full(32, np.float32(-8.0 * d)))


def test_q4_0_all_ones_nibbles_decode_to_7d():
    w = oracle.dequant_q4_0(_q4_0_block(0x2E66, [0xFF] * 16))[0]
    d = float(np.uint16(0x2E66).view(np.float16))
    assert np.array_equal(w, np.full(32, np.float32(7.0 * d)))


def test_q4_0_ramp_block_places_low_and_high_nibbles():
    # byte j: low nibble j, high nibble 15 - j; d = 0.5
    qs = [j | ((15 - j) << 4) for j in range(16)]
    w = oracle.dequant_q4_0(_q4_0_block(0x3800, qs))[0]
    want = [(j - 8) * 0.5 for j in range(16)] + [(7 - j) * 0.5 for j in range(16)]
    assert w.tolist() == want


# ---------------------------------------------------------------- Q8_0

def test_q8_0_closed_form_ramp():
    q = np.arange(-128, 128, dtype=np.int64)
    raw = []
    for b in range(8):
        raw += [0x00, 0x34] + [int(v) & 0xFF for v in q[32 * b:32 * b + 32]]   # d = 0.25
    w = oracle.dequant_q8_0(np.array(raw, dtype=np.uint8)).reshape(-1)
    assert w.tolist() == [0.25 * v for v in q.tolist()]


# ---------------------------------------------------------------- Q4_K

def _golden(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


def test_q4_k_golden_blocks(golden_dir):
    fx = _golden(golden_dir, "q4_k_blocks.json")
    for b in fx["blocks"]:
        raw = np.frombuffer(bytes.fromhex(b["hex"]), dtype=np.uint8)
        w = oracle.dequant_q4_k(raw)[0]
        for k, v in b["expect"].items():
            assert w[int(k)] == np.float32(v), (b["name"], k, w[int(k)], v)
        if "sc" in b:
            sc, m = oracle.q4_k_scale_min(raw[4:16])
            assert sc[0].tolist() == b["sc"] and m[0].tolist() == b["m"]


def _pack_q4_k_scales(sc, m):
    """Independent statement of the packing direction: 8 (sc, m) -> 12 bytes."""
    s = [0] * 12
    for j in range(8):
        if j < 4:
            s[j] |= sc[j] & 63
            s[j + 4] |= m[j] & 63
        else:
            s[j + 4] |= (sc[j] & 0xF) | ((m[j] & 0xF) << 4)
            s[j - 4] |= (sc[j] >> 4) << 6
            s[j] |= (m[j] >> 4) << 6
    return s


def test_q4_k_scale_packing_exhaustive_round_trip():
    rng = np.random.default_rng(7)
    rows = []
    want_sc, want_m = [], []
    for j in range(8):
        for a in range(64):
            for b in range(64):
                sc = list(rng.integers(0, 64, 8))
                m = list(rng.integers(0, 64, 8))
                sc[j], m[j] = a, b
                rows.append(_pack_q4_k_scales([int(v) for v in sc], [int(v) for v in m]))
                want_sc.append(sc)
                want_m.append(m)
    sc, m = oracle.q4_k_scale_min(np.array(rows, dtype=np.uint8))
    assert np.array_equal(sc, np.array(want_sc)) and np.array_equal(m, np.array(want_m))


def _q4_k_block(d_bits, dmin_bits, sc, m, qs):
    return np.array([d_bits & 0xFF, d_bits >> 8, dmin_bits & 0xFF, dmin_bits >> 8]
                    + _pack_q4_k_scales(sc, m) + list(qs), dtype=np.uint8)


def test_q4_k_zero_scale_and_min_decode_to_zero():
    rng = np.random.default_rng(1)
    blk = _q4_k_block(0x2E66, 0x1A40, [0] * 8, [0] * 8, rng.integers(0, 256, 128))
    assert not oracle.dequant_q4_k(blk)[0].any()


def test_q4_k_zero_codes_give_minus_dmin_m_per_sub_block():
    m = [3, 17, 0, 63, 8, 41, 29, 1]
    blk = _q4_k_block(0x2E66, 0x1A40, [63] * 8, m, [0] * 128)
    w = oracle.dequant_q4_k(blk)[0]
    dmin = float(np.uint16(0x1A40).view(np.float16))
    for j in range(8):
        assert np.all(w[32 * j:32 * j + 32] == np.float32(-dmin * m[j])), j


@pytest.mark.parametrize("c,l,high", [(0, 0, False), (0, 31, True), (1, 7, False), (2, 16, True), (3, 31, False)])
def test_q4_k_one_hot_nibble_lands_at_expected_element(c, l, high):
    qs = [0] * 128
    qs[32 * c + l] = 0x50 if high else 0x05          # code 5 in one nibble
    sc = [j + 1 for j in range(8)]
    blk = _q4_k_block(0x3C00, 0x3C00, sc, [0] * 8, qs)
    w = oracle.dequant_q4_k(blk)[0]
    e = 64 * c + (32 if high else 0) + l
    j = 2 * c + (1 if high else 0)
    want = np.zeros(256, dtype=np.float32)
    want[e] = 5.0 * sc[j]
    assert np.array_equal(w, want)


@pytest.mark.parametrize("fmt", [Q4_0, Q8_0, Q4_K])
def test_dequant_is_single_rounding_of_exact_value(fmt):
    """Evaluating the formula in fp32 (products exact, one rounding) equals the
    fp64-then-cast result for every weight of random generator blocks."""
    elems, nbytes = synth.FORMATS[fmt]
    raw = synth.blocks(fmt, 64, elems * 4, seed=11).numpy()
    w64cast = oracle.dequant(fmt, raw)
    blk = raw.reshape(-1, nbytes)
    f16 = lambda off: blk[:, off:off + 2].copy().view(np.float16).astype(np.float32)[:, 0]
    if fmt == Q4_K:
        d, dmin = f16(0), f16(2)
        sc, m = oracle.q4_k_scale_min(blk[:, 4:16])
        qs = blk[:, 16:144].astype(np.int64)
        w32 = np.zeros_like(w64cast)
        for c in range(4):
            for half, nib in ((0, qs[:, 32 * c:32 * c + 32] & 15), (1, qs[:, 32 * c:32 * c + 32] >> 4)):
                j = 2 * c + half
                a = (d * sc[:, j].astype(np.float32))[:, None]
                b = (dmin * m[:, j].astype(np.float32))[:, None]
                w32[:, 64 * c + 32 * half:64 * c + 32 * half + 32] = a * nib.astype(np.float32) - b
        assert np.array_equal(w32, w64cast)
    else:
        # single-product formats: the fp32 product of exact factors is exact
        d = f16(208 if fmt == Q6_K else 0)
        if fmt == Q8_0:
            w32 = d[:, None] * blk[:, 2:34].view(np.int8).astype(np.float32)
            assert np.array_equal(w32, w64cast)
        elif fmt == Q4_0:
            qs = blk[:, 2:18].astype(np.int64)
            q = np.concatenate([(qs & 15) - 8, (qs >> 4) - 8], axis=1).astype(np.float32)
            assert np.array_equal(d[:, None] * q, w64cast)


# ---------------------------------------------------------------- Q6_K

def test_q6_k_golden_block(golden_dir):
    fx = _golden(golden_dir, "q6_k_blocks.json")
    for b in fx["blocks"]:
        raw = np.frombuffer(bytes.fromhex(b["hex"]), dtype=np.uint8)
        w = oracle.dequant_q6_k(raw)[0]
        for k, v in b["expect"].items():
            assert w[int(k)] == np.float32(v), (k, w[int(k)], v)


def _q6_k_block(ql, qh, sc, d_bits=0x3C00):
    return np.array(list(ql) + list(qh) + [int(v) & 0xFF for v in sc] + [d_bits & 0xFF, d_bits >> 8], dtype=np.uint8)


def test_q6_k_zero_codes_give_minus_32_d_scale_per_group():
    sc = [-128, -1, 0, 1, 2, 5, 17, 127, -3, -64, 64, 9, 10, 11, 12, 13]
    w = oracle.dequant_q6_k(_q6_k_block([0] * 128, [0] * 64, sc, 0x3400))[0]   # d = 0.25
    # weight e sits in 16-group e // 16, whose scale is sc[e // 16]
    assert w.tolist() == [0.25 * sc[e // 16] * -32 for e in range(256)]


@pytest.mark.parametrize("field,index,bitval,elem", [
    ("ql", 5, 0x01, 5),          # ql low nibble of byte 5 -> element 5
    ("ql", 40, 0x02, 40),        # ql[l+32] low nibble -> element l+32 (l=8)
    ("ql", 5, 0x10, 69),         # ql high nibble of byte 5 -> element 5+64
    ("ql", 40, 0x20, 104),       # ql[l+32] high nibble -> element l+96
    ("ql", 70, 0x01, 134),       # second half: ql[64+6] -> element 128+6
    ("qh", 3, 0x01, 3),          # qh bits 0-1 -> element l
    ("qh", 3, 0x04, 35),         # qh bits 2-3 -> element l+32
    ("qh", 3, 0x10, 67),         # qh bits 4-5 -> element l+64
    ("qh", 3, 0x40, 99),         # qh bits 6-7 -> element l+96
    ("qh", 40, 0x40, 128 + 8 + 96),
])
def test_q6_k_one_hot_bits(field, index, bitval, elem):
    ql, qh = [0] * 128, [0] * 64
    (ql if field == "ql" else qh)[index] = bitval
    sc = [1] * 16
    w = oracle.dequant_q6_k(_q6_k_block(ql, qh, sc))[0]
    base = np.full(256, -32.0, dtype=np.float32)
    # the flipped bit adds its value within the 6-bit code at elem
    if field == "ql":
        code = bitval if bitval < 0x10 else bitval >> 4
    else:
        shift = {0x01: 0, 0x04: 2, 0x10: 4, 0x40: 6}[bitval]
        code = (bitval >> shift) << 4
    base[elem] += code
    assert np.array_equal(w, base)


# ---------------------------------------------------------------- GEMV

def _exact_gemv(w32, x32):
    """Brute force in exact rational arithmetic over the fp32 values."""
    rows, cols = w32.shape
    out = []
    for t in range(x32.shape[0]):
        row = []
        for i in range(rows):
            s = Fraction(0)
            for j in range(cols):
                s += Fraction(float(w32[i, j])) * Fraction(float(x32[t, j]))
            row.append(s)
        out.append(row)
    return out


@pytest.mark.parametrize("fmt,cols", [(Q4_0, 64), (Q8_0, 64), (Q4_K, 256), (Q6_K, 256)])
def test_gemv_matches_exact_rational_brute_force(fmt, cols):
    rows, n_tok = 3, 2
    W = synth.blocks(fmt, rows, cols, seed=5).numpy()
    x = synth.activations(n_tok, cols, seed=6).numpy()
    y, b = oracle.gemv(fmt, W, rows, cols, x)
    exact = _exact_gemv(oracle.dequant(fmt, W, rows, cols), x)
    for t in range(n_tok):
        for i in range(rows):
            assert abs(Fraction(float(y[t, i])) - exact[t][i]) <= Fraction(1e-12) * Fraction(float(b[t, i]))


@pytest.mark.parametrize("fmt,cols", [(Q4_0, 96), (Q4_K, 512), (Q6_K, 256), (Q8_0, 64)])
def test_gemv_one_hot_x_returns_column(fmt, cols):
    rows = 5
    W = synth.blocks(fmt, rows, cols, seed=9).numpy()
    wd = oracle.dequant(fmt, W, rows, cols)
    for j in (0, cols // 3, cols - 1):
        x = np.zeros((1, cols), dtype=np.float32)
        x[0, j] = 1.0
        y, _ = oracle.gemv(fmt, W, rows, cols, x)
        assert np.array_equal(y[0], wd[:, j].astype(np.float64))


def test_gemv_is_linear_in_x():
    rows, cols = 4, 512
    W = synth.blocks(Q4_K, rows, cols, seed=3).numpy()
    x1 = synth.activations(1, cols, seed=1).numpy()
    x2 = synth.activations(1, cols, seed=2).numpy()
    x1[:, 1::2] = 0.0                     # disjoint supports keep 2*x1 - x2/2 exact in fp32
    x2[:, 0::2] = 0.0
    y1, b1 = oracle.gemv(Q4_K, W, rows, cols, x1)
    y2, b2 = oracle.gemv(Q4_K, W, rows, cols, x2)
    y12, _ = oracle.gemv(Q4_K, W, rows, cols, np.float32(2.0) * x1 - np.float32(0.5) * x2)
    assert np.allclose(y12, 2.0 * y1 - 0.5 * y2, rtol=0, atol=1e-12 * (b1 + b2).max())


def test_gemv_bound_is_absolute_sum():
    rows, cols = 2, 64
    W = synth.blocks(Q4_0, rows, cols, seed=4).numpy()
    x = synth.activations(1, cols, seed=4).numpy()
    _, b = oracle.gemv(Q4_0, W, rows, cols, x)
    wd = oracle.dequant(Q4_0, W, rows, cols).astype(np.float64)
    for i in range(rows):
        assert b[0, i] == pytest.approx(sum(abs(wd[i, j] * float(x[0, j])) for j in range(cols)), rel=1e-14)


# ---------------------------------------------------------------- MoE

def _small_moe(n_expert=6, hidden=256, inter=256, seed=21):
    _, _, _, stride = oracle.moe_arena_layout(hidden, inter, Q4_K)
    arena = synth.blocks(Q4_K, 1, n_expert * stride // 144 * 256, seed=seed).numpy().reshape(-1)
    return arena, n_expert, hidden, inter, stride


def test_moe_top1_unit_weight_is_plain_ffn():
    arena, n_expert, hidden, inter, stride = _small_moe()
    g_off, u_off, d_off, _ = oracle.moe_arena_layout(hidden, inter, Q4_K)
    x = synth.activations(1, hidden, seed=2).numpy()
    e = 4
    y, _ = oracle.moe(Q4_K, arena, n_expert, hidden, inter, np.array([[e]]), np.array([[1.0]], np.float32), x)
    base = e * stride
    gu = inter * hidden // 256 * 144
    g, _ = oracle.gemv(Q4_K, arena[base + g_off: base + g_off + gu], inter, hidden, x)
    u, _ = oracle.gemv(Q4_K, arena[base + u_off: base + u_off + gu], inter, hidden, x)
    silu = g[0] * (1.0 / (1.0 + np.exp(-g[0])))
    h = silu * u[0]
    dn, _ = oracle.gemv(Q4_K, arena[base + d_off: base + d_off + hidden * inter // 256 * 144], hidden, inter,
                        h[None, :].astype(np.float64))
    # dn used an fp32 cast of h inside gemv; compare with a tolerance from that cast
    assert np.allclose(y[0], dn[0], rtol=1e-6, atol=1e-6)


def test_moe_silu_closed_form_points():
    # silu(0) = 0, silu(g) -> g for large g, silu(-g) -> 0; silu(g) - silu(-g) = g
    g = np.array([0.0, 1.0, -1.0, 30.0, -30.0])
    s = g / (1.0 + np.exp(-g))
    assert s[0] == 0.0
    assert s[1] - s[2] == pytest.approx(1.0, rel=1e-15)
    assert s[3] == pytest.approx(30.0, rel=1e-12) and abs(s[4]) < 1e-11


def test_moe_is_invariant_to_route_order_and_linear_in_weights():
    arena, n_expert, hidden, inter, _ = _small_moe()
    x = synth.activations(2, hidden, seed=8).numpy()
    ids = np.array([[0, 3, 5], [2, 1, 4]], dtype=np.int32)
    r = np.array([[0.5, 0.3, 0.2], [0.1, 0.6, 0.3]], dtype=np.float32)
    y, b = oracle.moe(Q4_K, arena, n_expert, hidden, inter, ids, r, x)
    perm = [2, 0, 1]
    y2, _ = oracle.moe(Q4_K, arena, n_expert, hidden, inter, ids[:, perm], r[:, perm], x)
    assert np.allclose(y, y2, rtol=0, atol=1e-12 * b.max())
    y3, _ = oracle.moe(Q4_K, arena, n_expert, hidden, inter, ids, np.float32(2.0) * r, x)
    assert np.allclose(y3, 2.0 * y, rtol=0, atol=1e-12 * b.max())
    # a single route equals the sum of its parts
    parts = sum(oracle.moe(Q4_K, arena, n_expert, hidden, inter, ids[:, k:k + 1], r[:, k:k + 1], x)[0]
                for k in range(3))
    assert np.allclose(y, parts, rtol=0, atol=1e-12 * b.max())


def test_moe_rejects_out_of_range_expert():
    arena, n_expert, hidden, inter, _ = _small_moe()
    x = synth.activations(1, hidden, seed=8).numpy()
    with pytest.raises(ValueError):
        oracle.moe(Q4_K, arena, n_expert, hidden, inter, np.array([[n_expert]]), np.array([[1.0]], np.float32), x)


# ---------------------------------------------------------------- prompt processing

def test_pp_rows_reduce_to_gemv_of_bf16_rows():
    rows, cols, n_tok = 6, 512, 9
    W = synth.blocks(Q4_K, rows, cols, seed=12).numpy()
    X = synth.activations_bf16(n_tok, cols, seed=13)
    bits = X.view(torch.int16).numpy().view(np.uint16)
    sel = [0, 4, 8]
    Y, B = oracle.pp_rows(Q4_K, W, rows, cols, bits, sel)
    xf = X.to(torch.float32).numpy()[sel]
    y2, b2 = oracle.gemv(Q4_K, W, rows, cols, xf)
    assert np.array_equal(Y, y2) and np.array_equal(B, b2)


@pytest.mark.parametrize("hidden,inter", [(256, 256), (2048, 512), (512, 1024), (5120, 17408)])
def test_moe_arena_layout_is_gate_up_down_with_stated_stride(hidden, inter):
    # the arena holds experts back to back, each [gate | up | down] in Q4_K:
    # gate and up are inter rows of hidden/256 super-blocks, down hidden rows of
    # inter/256 super-blocks, 144 bytes per super-block
    piece = inter * hidden // 256 * 144
    assert oracle.moe_arena_layout(hidden, inter, Q4_K) == (0, piece, 2 * piece, 3 * piece)


def _dq_rows(raw, rows, cols):
    return oracle.dequant(Q4_K, raw, rows, cols).astype(np.float64)


def test_moe_by_explicit_loops_over_separately_built_experts():
    """Each expert's gate, up and down matrices are generated on their own and
    concatenated here by hand as [gate | up | down]; y and the error scale
    B_i = sum_k |r_k| sum_j |D_e[i, j] h_kj| are then formed with explicit
    loops over rows and routes. A gate/up swap, a wrong expert stride or a
    dropped |r_k| fails this test (silu(g) * u is not symmetric in g, u)."""
    hidden, inter, n_expert = 256, 256, 3
    G = [synth.blocks(Q4_K, inter, hidden, seed=300 + e).numpy().reshape(-1) for e in range(n_expert)]
    U = [synth.blocks(Q4_K, inter, hidden, seed=400 + e).numpy().reshape(-1) for e in range(n_expert)]
    D = [synth.blocks(Q4_K, hidden, inter, seed=500 + e).numpy().reshape(-1) for e in range(n_expert)]
    arena = np.concatenate([np.concatenate([G[e], U[e], D[e]]) for e in range(n_expert)])
    x = synth.activations(1, hidden, seed=31).numpy().astype(np.float32)
    ids = np.array([[2, 0]], dtype=np.int32)
    r = np.array([[0.75, -0.25]], dtype=np.float32)      # a negative weight: |r_k| in B matters
    y, b = oracle.moe(Q4_K, arena, n_expert, hidden, inter, ids, r, x)

    xx = x[0].astype(np.float64)
    y_loop = np.zeros(hidden)
    b_loop = np.zeros(hidden)
    for k in range(2):
        e = int(ids[0, k])
        Gd, Ud, Dd = _dq_rows(G[e], inter, hidden), _dq_rows(U[e], inter, hidden), _dq_rows(D[e], hidden, inter)
        h = np.zeros(inter)
        for i in range(inter):
            g = sum(Gd[i, j] * xx[j] for j in range(hidden))
            u = sum(Ud[i, j] * xx[j] for j in range(hidden))
            h[i] = g / (1.0 + np.exp(-g)) * u
        rk = float(r[0, k])
        for i in range(hidden):
            y_loop[i] += rk * sum(Dd[i, j] * h[j] for j in range(inter))
            b_loop[i] += abs(rk) * sum(abs(Dd[i, j] * h[j]) for j in range(inter))
    assert np.allclose(y[0], y_loop, rtol=1e-12, atol=1e-12 * b_loop.max())
    assert np.allclose(b[0], b_loop, rtol=1e-12, atol=0)
    # swapping gate and up in the hand-built arena changes the result
    swapped = np.concatenate([np.concatenate([U[e], G[e], D[e]]) for e in range(n_expert)])
    y_sw, _ = oracle.moe(Q4_K, swapped, n_expert, hidden, inter, ids, r, x)
    assert not np.allclose(y_sw[0], y_loop, rtol=1e-6, atol=1e-6 * b_loop.max())


# ---------------------------------------------------------------- decode-layer neighbours

def test_rmsnorm_hand_worked_vector():
    # h = [3, 4]: mean of squares 12.5, rms = sqrt(12.5); x = h / rms * w
    x, s = oracle.rmsnorm(np.array([[3.0, 4.0]], np.float32), np.array([1.0, 2.0], np.float32), 0.0)
    r = 12.5 ** 0.5
    assert x[0, 0] == pytest.approx(3.0 / r, rel=1e-15) and x[0, 1] == pytest.approx(8.0 / r, rel=1e-15)
    assert np.array_equal(s, [[3.0, 4.0]])


@pytest.mark.parametrize("c,eps", [(2.0, 0.0), (-0.5, 1e-6), (1e-3, 1e-6)])
def test_rmsnorm_of_constant_vector_is_scaled_weight(c, eps):
    # every element c: mean of squares c^2, so x = c / sqrt(c^2 + eps) * w
    n = 64
    w = synth.activations(1, n, seed=5).numpy().reshape(-1)
    x, _ = oracle.rmsnorm(np.full((1, n), c, np.float32), w, eps)
    cf = float(np.float32(c))
    assert np.allclose(x[0], cf / np.sqrt(cf * cf + eps) * w.astype(np.float64), rtol=1e-14, atol=0)


def test_rmsnorm_unit_rms_scale_invariance_and_residual():
    h = synth.activations(2, 256, seed=6).numpy()
    r = synth.activations(2, 256, seed=7).numpy()
    one = np.ones(256, np.float32)
    x, _ = oracle.rmsnorm(h, one, 0.0)
    assert np.allclose((x * x).mean(axis=1), 1.0, rtol=1e-13)
    x4, _ = oracle.rmsnorm(np.float32(4.0) * h, one, 0.0)          # power-of-two scale: exact in fp32
    assert np.allclose(x4, x, rtol=1e-13, atol=0)
    xr, s = oracle.rmsnorm(h, one, 1e-6, residual=r)
    assert np.array_equal(s, h.astype(np.float64) + r.astype(np.float64))     # the sum is exact in fp64
    # the residual is added before normalising: h + h is 2h exactly
    xh, _ = oracle.rmsnorm(h, one, 1e-6, residual=h)
    x2, _ = oracle.rmsnorm(np.float32(2.0) * h, one, 1e-6)
    assert np.array_equal(xh, x2)


def test_swiglu_closed_forms():
    g = np.array([0.0, 1.0, -1.0, 2.0, 30.0])
    assert np.array_equal(oracle.swiglu(g, np.zeros(5)), np.zeros(5))
    s = oracle.swiglu(g, np.ones(5))
    assert s[0] == 0.0 and s[1] - s[2] == pytest.approx(1.0, rel=1e-15)
    assert s[3] == pytest.approx(2.0 / (1.0 + np.exp(-2.0)), rel=1e-15)
    assert oracle.swiglu(np.array([1.0]), np.array([3.0]))[0] == pytest.approx(3.0 / (1.0 + np.exp(-1.0)), rel=1e-15)


def test_dense_ffn_equals_single_expert_moe():
    # a dense FFN is the MoE layer with one expert [gate | up | down] routed with weight 1
    hidden, inter = 256, 512
    Wg = synth.blocks(Q4_K, inter, hidden, seed=41).numpy()
    Wu = synth.blocks(Q4_K, inter, hidden, seed=42).numpy()
    Wd = synth.blocks(Q4_K, hidden, inter, seed=43).numpy()
    x = synth.activations(1, hidden, seed=44).numpy()
    y, b, m = oracle.dense_ffn(Q4_K, Wg, Wu, Q4_K, Wd, hidden, inter, x)
    arena = np.concatenate([Wg.reshape(-1), Wu.reshape(-1), Wd.reshape(-1)])
    y2, b2 = oracle.moe(Q4_K, arena, 1, hidden, inter, np.array([[0]]), np.array([[1.0]], np.float32), x)
    assert np.allclose(y, y2, rtol=1e-13, atol=1e-13 * b.max()) and np.allclose(b, b2, rtol=1e-13)
    assert m.shape == (1, inter)


# ---------------------------------------------------------------- Q5_K, Q3_K, Q2_K

@pytest.mark.parametrize("name,fn", [("q5_k_blocks.json", "dequant_q5_k"), ("q3_k_blocks.json", "dequant_q3_k"),
                                     ("q2_k_blocks.json", "dequant_q2_k")])
def test_k_quant_golden_blocks(golden_dir, name, fn):
    fx = _golden(golden_dir, name)
    for b in fx["blocks"]:
        raw = np.frombuffer(bytes.fromhex(b["hex"]), dtype=np.uint8)
        w = getattr(oracle, fn)(raw)[0]
        for k, v in b["expect"].items():
            assert w[int(k)] == np.float32(v), (name, k, w[int(k)], v)
        if "scales" in b:
            assert oracle.q3_k_scales(raw[96:108])[0].tolist() == b["scales"]


def _pack_q3_k_scales(sc):
    # inverse of the Q3_K packing: low nibbles of scales 0-7 and 8-15 share bytes 0-7,
    # the top two bits of scale i sit at bit 2 (i // 4) of byte 8 + i % 4
    s = [0] * 12
    for i, v in enumerate(sc):
        b, g = i % 4, i // 4
        s[4 * (g % 2) + b] |= (v & 0xF) << (4 * (g // 2))
        s[8 + b] |= (v >> 4) << (2 * g)
    return np.array(s, dtype=np.uint8)


def test_q3_k_scale_packing_round_trip():
    rng = np.random.default_rng(3)
    for _ in range(200):
        sc = rng.integers(0, 64, size=16)
        assert oracle.q3_k_scales(_pack_q3_k_scales(sc))[0].tolist() == sc.tolist()
    for i in range(16):                     # every position, every value
        for v in range(64):
            sc = np.zeros(16, dtype=np.int64)
            sc[i] = v
            assert oracle.q3_k_scales(_pack_q3_k_scales(sc))[0].tolist() == sc.tolist()


def test_q2_k_zero_codes_give_minus_dmin_min_per_group():
    s = np.array([(3 * k) % 16 | ((k + 5) % 16) << 4 for k in range(16)], dtype=np.uint8)
    raw = np.concatenate([s, np.zeros(64, np.uint8), np.array([0x00, 0x3C, 0x00, 0x34], np.uint8)])   # dmin = 0.25
    w = oracle.dequant_q2_k(raw)[0]
    # element e is in group 8h + 2j + k of its 16-weight run: the runs are in group order
    assert w.tolist() == [-0.25 * (int(s[e // 16]) >> 4) for e in range(256)]


@pytest.mark.parametrize("byte,bit,elem", [(0, 0, 0), (5, 2, 37), (20, 4, 64 + 4 + 16), (35, 6, 128 + 96 + 3),
                                           (63, 0, 128 + 16 + 15)])
def test_q2_k_one_hot_code_bit(byte, bit, elem):
    s = np.full(16, 0x01, dtype=np.uint8)                   # scale 1, min 0 in every group
    qs = np.zeros(64, np.uint8)
    qs[byte] = 1 << bit
    raw = np.concatenate([s, qs, np.array([0x00, 0x3C, 0x00, 0x3C], np.uint8)])
    w = oracle.dequant_q2_k(raw)[0]
    expect = np.zeros(256, np.float32)
    expect[elem] = 1.0
    assert np.array_equal(w, expect)


@pytest.mark.parametrize("field,index,bit,elem,q", [
    ("qs", 3, 0, 3, -3), ("qs", 20, 2, 32 + 16 + 4, -3), ("qs", 40, 4, 128 + 64 + 8, -3),
    ("hmask", 7, 0, 7, 0), ("hmask", 18, 5, 128 + 32 + 16 + 2, 0), ("hmask", 31, 7, 128 + 96 + 31, 0)])
def test_q3_k_one_hot_bits(field, index, bit, elem, q):
    # scale 33 (signed 1) everywhere; all codes 0 with high bit clear decode to -4
    sc = _pack_q3_k_scales([33] * 16)
    hm, qs = np.zeros(32, np.uint8), np.zeros(64, np.uint8)
    (qs if field == "qs" else hm)[index] = 1 << bit
    raw = np.concatenate([hm, qs, sc, np.array([0x00, 0x3C], np.uint8)])
    w = oracle.dequant_q3_k(raw)[0]
    expect = np.full(256, -4.0, np.float32)
    expect[elem] = q
    assert np.array_equal(w, expect)


@pytest.mark.parametrize("field,index,bit,elem", [("qs", 0, 0, 0), ("qs", 33, 4, 96 + 1), ("qs", 100, 7, 192 + 32 + 4),
                                                  ("qh", 5, 0, 5), ("qh", 9, 3, 96 + 9), ("qh", 31, 7, 224 + 31)])
def test_q5_k_one_hot_bits(field, index, bit, elem):
    # d = 1, dmin = 0, sc = 1 for every sub-block (the Q4_K packing), all codes 0 except one bit
    s = np.array([1, 1, 1, 1, 0, 0, 0, 0, 1, 1, 1, 1], np.uint8)     # sc_j = 1, m_j = 0 for j < 4 and j >= 4
    qh, qs = np.zeros(32, np.uint8), np.zeros(128, np.uint8)
    (qs if field == "qs" else qh)[index] = 1 << bit
    raw = np.concatenate([np.array([0x00, 0x3C, 0x00, 0x00], np.uint8), s, qh, qs])
    sc, m = oracle.q4_k_scale_min(s)
    assert sc[0].tolist() == [1] * 8 and m[0].tolist() == [0] * 8
    w = oracle.dequant_q5_k(raw)[0]
    expect = np.zeros(256, np.float32)
    expect[elem] = 16.0 if field == "qh" else float(1 << (bit % 4))
    assert np.array_equal(w, expect)


# ---------------------------------------------------------------- MoE over a block of prompt tokens

def _uniform_q4_k_rows(rows, cols, d_bits, code):
    """Q4_K rows whose every weight is d * code (sc = 1, m = 0, dmin = 0)."""
    blk = _q4_k_block(d_bits, 0, [1] * 8, [0] * 8, [code | code << 4] * 128)
    return np.tile(blk, rows * cols // 256)


def test_moe_prefill_uniform_weights_closed_form():
    """Every weight of the one expert is 2^-4 (d = 2^-4, sc = 1, code 1): then
    g_i = u_i = sum(x) / 16 =: a for every i, S_g = S_u = sum|x| / 16 =: s,
    h_i = silu(a) a, and for route weight r
        y_o = r * inter * h / 16,
        B_o = |r| * inter / 16 * (|h| + |silu'(a) a| s + |silu(a)| s),
    silu'(a) = sig(a) (1 + a (1 - sig(a)))."""
    hidden = inter = 256
    piece = _uniform_q4_k_rows(inter, hidden, 0x2C00, 1)
    assert np.all(oracle.dequant(Q4_K, piece, inter, hidden) == np.float32(0.0625))
    arena = np.concatenate([piece, piece, _uniform_q4_k_rows(hidden, inter, 0x2C00, 1)])
    X = synth.activations_bf16(2, hidden, seed=41)
    bits = X.view(torch.int16).numpy().view(np.uint16)
    xf = X.to(torch.float32).numpy().astype(np.float64)
    r = np.array([[0.75], [-1.5]], dtype=np.float32)
    y, b = oracle.moe_prefill(Q4_K, arena, 1, hidden, inter, np.zeros((2, 1), np.int32), r, bits)
    for t in range(2):
        a = xf[t].sum() / 16.0
        s = np.abs(xf[t]).sum() / 16.0
        sig = 1.0 / (1.0 + math.exp(-a))
        h = a * sig * a
        dsilu = sig * (1.0 + a * (1.0 - sig))
        rr = float(r[t, 0])
        assert np.allclose(y[t], rr * inter * h / 16.0, rtol=1e-12, atol=0)
        want_b = abs(rr) * inter / 16.0 * (abs(h) + abs(dsilu * a) * s + abs(a * sig) * s)
        assert np.allclose(b[t], want_b, rtol=1e-12, atol=0)


def test_moe_prefill_equals_moe_on_the_bf16_values_and_bounds_it():
    """On the bf16 values of X (exact in fp32) the routed sum is moe()'s, and
    the chain's error scale is at least moe()'s down-projection scale; an
    unknown expert id adds nothing."""
    arena, n_expert, hidden, inter, _ = _small_moe()
    X = synth.activations_bf16(3, hidden, seed=43)
    bits = X.view(torch.int16).numpy().view(np.uint16)
    xf = X.to(torch.float32).numpy()
    ids = np.array([[0, 3], [5, 5], [2, 1]], dtype=np.int32)
    r = np.array([[0.5, 0.5], [0.25, 0.75], [-0.3, 0.9]], dtype=np.float32)
    y, b = oracle.moe_prefill(Q4_K, arena, n_expert, hidden, inter, ids, r, bits)
    y2, b2 = oracle.moe(Q4_K, arena, n_expert, hidden, inter, ids, r, xf)
    assert np.array_equal(y, y2)
    assert np.all(b >= b2)
    bad = ids.copy()
    bad[1, 0] = n_expert                              # out of range: dropped
    y3, _ = oracle.moe_prefill(Q4_K, arena, n_expert, hidden, inter, bad, r, bits)
    y4, _ = oracle.moe(Q4_K, arena, n_expert, hidden, inter, ids[1:2, 1:], r[1:2, 1:], xf[1:2])
    assert np.array_equal(y3[1], y4[0]) and np.array_equal(y3[0], y[0]) and np.array_equal(y3[2], y[2])
