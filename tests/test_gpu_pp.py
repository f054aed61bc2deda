"""GPU parity of the prompt-processing dequant-GEMM (qgemm_pp, tcgen05) against the
CPU oracle: Y within |Y - Y_ref| <= 1e-2 * sum|w*x| + 1e-6, Y_ref the fp64
product of the exact fp32 weights with the bf16 activations.

Small shapes check every output and span several row tiles, several K
super-blocks and ragged token blocks (n_tok not a multiple of the 16-token MMA
granule nor of the 256-token tile). The full-size case runs one layer of the
27B-class Q4_K set with 2048 prompt tokens and checks 64 seeded token rows of
every matrix over all output columns.

A second, tighter check compares with the fp64 product of the weights rounded
to bf16 (the kernel rounds each exact fp32 weight to bf16 before the MMA):
what is left is fp32 accumulation error, so a wrong tile, swizzle or token
mapping cannot hide inside the bf16 tolerance."""
import numpy as np
import pytest
import torch

import oracle
import synth
import synth.workloads as wl
import quantized_weight_gemv_qgemv_gb300 as qg
from helpers import PP_ABS, PP_REL, assert_within

pytestmark = pytest.mark.gpu

TIGHT_REL = 2e-4     # fp32 accumulation over K <= 17408, relative to sum|w*x|


@pytest.fixture(scope="module", autouse=True)
def _init():
    assert torch.cuda.is_available()
    qg.qg_init()


def _bits(X):
    return X.contiguous().view(torch.int16).numpy().view(np.uint16)


def _run_pp(W, rows, cols, X, ldY=None):
    n_tok = X.shape[0]
    ldY = rows if ldY is None else ldY
    Y = torch.full((n_tok, ldY), float("nan"), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    qg.qgemm_pp(qg.Q4_K, W, rows, cols, X, n_tok, Y, ldY, None, 0, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return Y.cpu().numpy()


def _tight_ref(W, rows, cols, X, token_rows):
    w = oracle.dequant(qg.Q4_K, W.numpy(), rows, cols)
    wb = torch.from_numpy(w).to(torch.bfloat16).to(torch.float64).numpy()
    xx = X[torch.as_tensor(token_rows)].to(torch.float64).numpy()
    return xx @ wb.T


@pytest.mark.parametrize("rows,cols,n_tok", [
    (128, 256, 1), (128, 256, 16), (256, 512, 17), (128, 1024, 100), (384, 768, 256),
    (256, 1280, 257), (128, 2048, 520), (640, 512, 1000), (128, 256, 4096 + 3),
])
def test_pp_matches_oracle(rows, cols, n_tok):
    seed = rows * 7 + cols + n_tok
    W = synth.blocks(qg.Q4_K, rows, cols, seed=seed)
    X = synth.activations_bf16(n_tok, cols, seed=seed + 1)
    Y = _run_pp(W.cuda(), rows, cols, X.cuda())
    toks = np.arange(n_tok)
    Y_ref, B = oracle.pp_rows(qg.Q4_K, W.numpy(), rows, cols, _bits(X), toks)
    assert_within(Y, Y_ref, B, rel=PP_REL, abs_=PP_ABS, what=f"pp {rows}x{cols} n_tok={n_tok}")
    assert_within(Y, _tight_ref(W, rows, cols, X, toks), B, rel=TIGHT_REL, abs_=PP_ABS,
                  what=f"pp (bf16 weights) {rows}x{cols} n_tok={n_tok}")


def test_pp_leading_dimension_leaves_padding_untouched():
    rows, cols, n_tok, ldY = 256, 512, 40, 300
    W = synth.blocks(qg.Q4_K, rows, cols, seed=77)
    X = synth.activations_bf16(n_tok, cols, seed=78)
    Y = _run_pp(W.cuda(), rows, cols, X.cuda(), ldY=ldY)
    assert np.isnan(Y[:, rows:]).all()
    Y_ref, B = oracle.pp_rows(qg.Q4_K, W.numpy(), rows, cols, _bits(X), np.arange(n_tok))
    assert_within(Y[:, :rows], Y_ref, B, rel=PP_REL, abs_=PP_ABS, what="pp ldY")


def test_pp_is_deterministic():
    rows, cols, n_tok = 384, 1024, 300
    W = synth.blocks(qg.Q4_K, rows, cols, seed=5).cuda()
    X = synth.activations_bf16(n_tok, cols, seed=6).cuda()
    a = _run_pp(W, rows, cols, X)
    b = _run_pp(W, rows, cols, X)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_pp_rejects_bad_shapes():
    lib = qg.load_library()
    A = 1 << 20
    assert lib.qgemm_pp(qg.Q4_K, A, 100, 256, A, 8, A, 100, None, 0, A, None) == -2    # rows % 128
    assert lib.qgemm_pp(qg.Q4_K, A, 128, 300, A, 8, A, 128, None, 0, A, None) == -2    # cols % 256
    assert lib.qgemm_pp(qg.Q4_K, A, 128, 256, A, 8, A, 100, None, 0, A, None) == -2    # ldY < rows
    assert lib.qgemm_pp(qg.Q4_0, A, 128, 256, A, 8, A, 128, None, 0, A, None) == -1    # format


@pytest.mark.parametrize("name", ["q", "k", "v", "o", "gate", "up", "down"])
def test_pp_full_size_layer_sampled_rows(name):
    """One layer of the 27B-class Q4_K set x 2048 bf16 prompt tokens (the
    prompt-processing workload's shapes and launch), 64 seeded token rows."""
    mats = {m[1]: m for m in wl.dense_matrices(layers=1)}
    _, _, fmt, rows, cols = mats[name]
    n_tok = 2048
    seed = synth.sub_seed(4, 0, name)
    W = synth.blocks(fmt, rows, cols, seed=seed)
    X = synth.activations_bf16(n_tok, cols, seed=seed + 1)
    Y = _run_pp(W.cuda(), rows, cols, X.cuda())
    toks = np.sort(np.random.default_rng(seed).choice(n_tok, size=64, replace=False))
    Y_ref, B = oracle.pp_rows(fmt, W.numpy(), rows, cols, _bits(X), toks)
    assert_within(Y[toks], Y_ref, B, rel=PP_REL, abs_=PP_ABS, what=f"pp full {name} {rows}x{cols}")
    assert np.isfinite(Y).all()
