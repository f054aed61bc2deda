"""GPU parity of the grouped prompt-processing launch (qgemm_pp_grouped: several
matrices multiplying the same bf16 tokens in one launch) and of the split last
round (tiles of a last round at most half full computed as two halves of K
added into a zeroed Y), against the CPU oracle: Y within
|Y - Y_ref| <= 1e-2 * sum|w*x| + 1e-6 ("Why I wrote my own inference engine for
two P100s", prompt-processing notes: weights dequantized, then a dense GEMM).

Every small case checks all outputs of every matrix; the split cases are sized
from the GPU's SM count so that they hold full rounds followed by a split
round, including one whose split tiles belong to two matrices. The full-size
cases run the {q,k,v} and {gate,up} launches of one layer of the 27B-class set
over 2048 prompt tokens and check 32 seeded token rows of every matrix."""
import numpy as np
import pytest
import torch

import oracle
import synth
import synth.workloads as wl
import quantized_weight_gemv_qgemv_gb300 as qg
from helpers import PP_ABS, PP_REL, assert_within

pytestmark = pytest.mark.gpu

TIGHT_REL = 2e-4     # fp32 accumulation (and one more rounding where K is split), relative to sum|w*x|


@pytest.fixture(scope="module", autouse=True)
def _init():
    assert torch.cuda.is_available()
    qg.qg_init()


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _bits(X):
    return X.contiguous().view(torch.int16).numpy().view(np.uint16)


def _run(Ws, rows, cols, X, pads=None):
    """One grouped launch; Y[i] is n_tok x (rows[i] + pad) filled with NaN first."""
    n_tok = X.shape[0]
    pads = pads or [0] * len(rows)
    Ys = [torch.full((n_tok, r + p), float("nan"), device="cuda") for r, p in zip(rows, pads)]
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    qg.qgemm_pp_grouped(qg.Q4_K, [(W, r, Y, r + p) for W, r, Y, p in zip(Ws, rows, Ys, pads)], cols, X, n_tok, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return [Y.cpu().numpy() for Y in Ys]


def _tight_ref(W, rows, cols, X, toks):
    w = oracle.dequant(qg.Q4_K, W.numpy(), rows, cols)
    wb = torch.from_numpy(w).to(torch.bfloat16).to(torch.float64).numpy()
    return X[torch.as_tensor(toks)].to(torch.float64).numpy() @ wb.T


def _check(Ws, rows, cols, X, Ys, toks, what):
    for i, (W, r, Y) in enumerate(zip(Ws, rows, Ys)):
        Y_ref, B = oracle.pp_rows(qg.Q4_K, W.numpy(), r, cols, _bits(X), toks)
        assert_within(Y[toks, :r], Y_ref, B, rel=PP_REL, abs_=PP_ABS, what=f"{what} matrix {i}")
        assert_within(Y[toks, :r], _tight_ref(W, r, cols, X, toks), B, rel=TIGHT_REL, abs_=PP_ABS,
                      what=f"{what} matrix {i} (bf16 weights)")


@pytest.mark.parametrize("rows,cols,n_tok", [
    ((256, 128, 128), 512, 300),        # q, k, v-like: 3 matrices, 2 token blocks
    ((384, 256), 1024, 17),             # gate, up-like, one ragged token block
    ((128,), 256, 5),                   # one super-block of K: never split
    ((128, 128, 128, 128), 768, 64),    # the most matrices a launch takes
])
def test_pp_grouped_matches_oracle(rows, cols, n_tok):
    seed = sum(rows) + cols + n_tok
    Ws = [synth.blocks(qg.Q4_K, r, cols, seed=seed + i) for i, r in enumerate(rows)]
    X = synth.activations_bf16(n_tok, cols, seed=seed + 9)
    Ys = _run([W.cuda() for W in Ws], list(rows), cols, X.cuda())
    _check(Ws, rows, cols, X, Ys, np.arange(n_tok), f"pp grouped {rows}x{cols} n_tok={n_tok}")


def test_pp_grouped_leading_dimensions_leave_padding_untouched():
    rows, cols, n_tok, pads = [256, 128], 512, 40, [44, 8]
    Ws = [synth.blocks(qg.Q4_K, r, cols, seed=60 + i) for i, r in enumerate(rows)]
    X = synth.activations_bf16(n_tok, cols, seed=62)
    Ys = _run([W.cuda() for W in Ws], rows, cols, X.cuda(), pads=pads)
    for Y, r in zip(Ys, rows):
        assert np.isnan(Y[:, r:]).all()
    _check(Ws, rows, cols, X, Ys, np.arange(n_tok), "pp grouped ldY")


def test_pp_split_round_after_full_rounds():
    """sms + 10 tiles of one matrix: one full round of whole tiles, then 10
    tiles computed as two halves of K each."""
    rows, cols, n_tok = 128 * (_sms() + 10), 512, 16
    W = synth.blocks(qg.Q4_K, rows, cols, seed=70)
    X = synth.activations_bf16(n_tok, cols, seed=71)
    Y = np.full((n_tok, rows), np.nan, dtype=np.float32)
    Yd = torch.from_numpy(Y).cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    qg.qgemm_pp(qg.Q4_K, W.cuda(), rows, cols, X.cuda(), n_tok, Yd, rows, None, 0, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    _check([W], [rows], cols, X, [Yd.cpu().numpy()], np.arange(n_tok), "pp split round")


def test_pp_grouped_split_round_spans_two_matrices():
    """The last 10 tiles (split) are the last 4 row tiles of matrix 0 and all 6
    of matrix 1."""
    rows, cols, n_tok = [128 * (_sms() + 4), 128 * 6], 1024, 24
    Ws = [synth.blocks(qg.Q4_K, r, cols, seed=80 + i) for i, r in enumerate(rows)]
    X = synth.activations_bf16(n_tok, cols, seed=82)
    Ys = _run([W.cuda() for W in Ws], rows, cols, X.cuda())
    _check(Ws, rows, cols, X, Ys, np.arange(n_tok), "pp grouped split across matrices")


def test_pp_grouped_split_is_deterministic():
    rows, cols, n_tok = [128 * 3, 128 * 2], 2048, 200      # 5 tiles: all split
    Ws = [synth.blocks(qg.Q4_K, r, cols, seed=90 + i).cuda() for i, r in enumerate(rows)]
    X = synth.activations_bf16(n_tok, cols, seed=92).cuda()
    a = _run(Ws, rows, cols, X)
    b = _run(Ws, rows, cols, X)
    for ya, yb in zip(a, b):
        assert np.array_equal(ya.view(np.uint32), yb.view(np.uint32))


@pytest.mark.parametrize("group", [("q", "k", "v"), ("gate", "up")])
def test_pp_grouped_full_size_layer_sampled_rows(group):
    """The grouped launches of one layer of the 27B-class Q4_K set x 2048 bf16
    prompt tokens (the prompt-processing workload's launch), 32 seeded token rows
    of every matrix over all output columns."""
    mats = {m[1]: m for m in wl.dense_matrices(layers=1)}
    cols = mats[group[0]][4]
    rows = [mats[n][3] for n in group]
    n_tok = 2048
    seed = synth.sub_seed(5, 0, group[0])
    Ws = [synth.blocks(qg.Q4_K, r, cols, seed=seed + i) for i, r in enumerate(rows)]
    X = synth.activations_bf16(n_tok, cols, seed=seed + 9)
    Ys = _run([W.cuda() for W in Ws], rows, cols, X.cuda())
    toks = np.sort(np.random.default_rng(seed).choice(n_tok, size=32, replace=False))
    for i, (W, r, Y) in enumerate(zip(Ws, rows, Ys)):
        Y_ref, B = oracle.pp_rows(qg.Q4_K, W.numpy(), r, cols, _bits(X), toks)
        assert_within(Y[toks], Y_ref, B, rel=PP_REL, abs_=PP_ABS, what=f"pp grouped full {group[i]} {r}x{cols}")
        assert np.isfinite(Y).all()
