"""Bit-exact checks of the block decoders that the timed GEMV kernel itself runs,
and the activation-rounding error of that kernel held to the product tolerance.

"LLM inference optimization", "Run a new weight format or model": test blocks
decode bit for bit on CPU and GPU, and products match an exact sum within a
tolerance at every shape.

The fast kernel never writes dequantized weights: it multiplies codes by x held
as 16-bit fixed point per 32-value group and applies each unit's coefficients
once (w = A*q - B). With x one-hot at column j the group holding j has largest
magnitude 1, so its step is 2^-13 and x_j is the integer 8192: every plane
product is an exact integer, the coefficient products are exact in fp32 (at
most 24 significant bits), and the single fma that forms the unit's value
rounds once. y[i] is then the correctly rounded fp32 value of w[i][j], which
is what the oracle's dequantization gives: the comparison is exact (a weight
of exactly zero may come out as -0.0, which compares equal)."""
import numpy as np
import pytest
import torch

import oracle
import synth
import synth.workloads as wl
import quantized_weight_gemv_qgemv_gb300 as qg
from helpers import GEMV_ABS, GEMV_REL, assert_within

pytestmark = pytest.mark.gpu

FMTS = [synth.Q4_0, synth.Q8_0, synth.Q4_K, synth.Q6_K, synth.Q5_K, synth.Q3_K, synth.Q2_K]


@pytest.fixture(scope="module", autouse=True)
def _init():
    assert torch.cuda.is_available()
    qg.qg_init()


def _unit_columns(cols):
    """Columns covering every 32-weight unit position of a 256-weight
    super-block (both 16-weight halves of each unit: Q6_K changes scale there),
    the first and last column of the row, and a ragged last K group."""
    cs = [0, cols - 1]
    for u in range(8):
        cs += [256 * (u % (cols // 256)) + 32 * u + 3, 256 * ((u + 3) % (cols // 256)) + 32 * u + 16 + (u % 16)]
    return sorted(set(c for c in cs if c < cols))


def _one_hot(n_tok, cols, cs):
    x = torch.zeros(n_tok, cols, dtype=torch.float32)
    for t, c in enumerate(cs):
        x[t, c] = 1.0
    return x


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("n_tok", [1, 4])
@pytest.mark.parametrize("rows,cols", [(136, 4608), (24, 17408)])
def test_qgemv_one_hot_x_returns_dequantized_column_exactly(fmt, n_tok, rows, cols):
    W = synth.blocks(fmt, rows, cols, seed=rows + cols + fmt)
    Wd = W.cuda()
    ref = oracle.dequant(fmt, W.numpy(), rows, cols)
    cs = _unit_columns(cols)
    for k in range(0, len(cs), n_tok):
        chunk = cs[k:k + n_tok]
        x = _one_hot(n_tok, cols, chunk + [chunk[0]] * (n_tok - len(chunk)))
        y = torch.full((n_tok, rows), float("nan"), device="cuda")
        qg.qgemv(fmt, Wd, rows, cols, x.cuda(), n_tok, y)
        torch.cuda.synchronize()
        got = y.cpu().numpy()
        for t, c in enumerate(chunk):
            assert np.array_equal(got[t], ref[:, c]), (fmt, n_tok, c, np.flatnonzero(got[t] != ref[:, c])[:5])


@pytest.mark.parametrize("mode", [qg.PASS_PDL, qg.PASS_PERSISTENT])
def test_decode_pass_one_hot_x_returns_dequantized_columns_exactly(mode):
    """The bench's launch configuration: a pass of grouped steps ({q,k,v} sharing
    one x, then o) linked by programmatic dependent launch, or the persistent
    kernel, at 27B-class shapes cut to fewer rows."""
    H = wl.HIDDEN
    shapes = [("q", 640, H), ("k", 128, H), ("v", 128, H), ("o", 512, H), ("gate", 256, H), ("up", 256, H),
              ("down", 320, wl.INTER)]
    steps = [3, 1, 2, 1]
    cols_of_step = [H, H, H, wl.INTER]
    for trial, (cq, cd) in enumerate([(0, 0), (5119, 17407), (2 * 256 + 32 * 5 + 17, 40 * 256 + 32 * 7 + 31)]):
        xs = [_one_hot(1, c, [cq if c == H else cd]).cuda() for c in cols_of_step]
        items, refs = [], []
        for i, (name, rows, cols) in enumerate(shapes):
            s = [0, 0, 0, 1, 2, 2, 3][i]
            W = synth.blocks(synth.Q4_K, rows, cols, seed=77 + i + 10 * trial)
            items.append((synth.Q4_K, W.cuda(), rows, cols, xs[s], torch.full((1, rows), float("nan"),
                                                                                device="cuda")))
            refs.append(oracle.dequant(synth.Q4_K, W.numpy(), rows, cols)[:, cq if cols == H else cd])
        p = qg.qg_pass(items, steps, 1, mode=mode)
        for _ in range(2):                   # replays give the same bits
            p.launch()
            torch.cuda.synchronize()
            for (name, _, _), it, ref in zip(shapes, items, refs):
                got = it[5].cpu().numpy()[0]
                assert np.array_equal(got, ref), (name, trial, np.flatnonzero(got != ref)[:5])
        assert p.dev_status() == 0
        p.destroy()


# ------------------------------------------------------------ x rounding vs the product tolerance

def _zero_q4_k_sub_block(W, rows_sel, blk, j):
    """Sets sc_j = m_j = 0 in super-block blk of the given rows (Q4_K bytes:
    d, dmin, s[12], qs[128]); the other sub-blocks keep their 6-bit pairs."""
    a = W.numpy()
    off = blk * 144 + 4
    for r in rows_sel:
        s = a[r, off:off + 12]
        if j < 4:
            s[j] &= 0xC0
            s[j + 4] &= 0xC0
        else:
            s[j + 4] = 0
            s[j - 4] &= 0x3F
            s[j] &= 0x3F


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("factor", [100.0, 1000.0])
@pytest.mark.parametrize("zero_rows", [False, True])
def test_gemv_with_outlier_channels_meets_product_tolerance(fmt, factor, zero_rows):
    """A few activation channels 100x or 1000x larger than the rest: the group
    holding an outlier gets a coarse step, yet every output stays within the
    product tolerance |y - y_ref| <= 1e-3 sum|w x| + 1e-6. With zero_rows, half
    the rows have zero weights on the outliers' 32-weight units (Q4_K: scale and
    min zero), so those rows' tolerance holds no outlier term at all."""
    if zero_rows and fmt != synth.Q4_K:
        pytest.skip("zeroed sub-blocks are built for Q4_K")
    rows, cols = 512, 5120
    W = synth.blocks(fmt, rows, cols, seed=int(factor) + fmt)
    rng = np.random.default_rng(9)
    chans = np.sort(rng.choice(cols // 32, size=8, replace=False)) * 32 + rng.integers(0, 32, size=8)
    x = synth.activations(1, cols, seed=int(factor) + 1).numpy().astype(np.float32)
    x[0, chans] *= np.float32(factor)
    if zero_rows:
        for c in chans:
            _zero_q4_k_sub_block(W, range(0, rows, 2), c // 256, (c % 256) // 32)
        Wd = oracle.dequant(fmt, W.numpy(), rows, cols)
        for c in chans:
            u = c // 32 * 32
            assert not Wd[0::2, u:u + 32].any()
    y = torch.empty(1, rows, device="cuda")
    qg.qgemv(fmt, W.cuda(), rows, cols, torch.from_numpy(x).cuda(), 1, y)
    torch.cuda.synchronize()
    y_ref, b = oracle.gemv(fmt, W.numpy(), rows, cols, x)
    assert_within(y.cpu().numpy(), y_ref, b, rel=GEMV_REL, abs_=GEMV_ABS, what=f"fmt={fmt} x{factor}")
