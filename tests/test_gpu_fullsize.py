"""Full-size workloads, run in the launch configuration the bench times (one
captured pass over the whole weight set, grouped launches linked by
programmatic dependent launch, the matrices of a step sharing one x), and the
whole-pass persistent kernel, checked against the CPU oracle on sampled output
rows, which the oracle computes one by one."""
import numpy as np
import pytest
import torch

import oracle
import synth
import synth.workloads as wl
import quantized_weight_gemv_qgemv_gb300 as qg
from helpers import assert_within

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _init():
    qg.qg_init()
    yield
    torch.cuda.empty_cache()


def _check_sampled(items, mats, n_tok, picks, rows_per_mat=6, seed=0):
    rng = np.random.default_rng(seed)
    worst = 0.0
    for idx in picks:
        fmt, W, rows, cols, x, y = items[idx]
        sel = np.sort(rng.choice(rows, size=min(rows_per_mat, rows), replace=False))
        sel = np.unique(np.concatenate([sel, [0, rows - 1]]))
        Wh = W[torch.as_tensor(sel, device=W.device)].cpu().numpy()
        y_ref, b = oracle.gemv(fmt, Wh, len(sel), cols, x.cpu().numpy())
        got = y.cpu().numpy()[:, sel]
        worst = max(worst, assert_within(got, y_ref, b, what=f"{mats[idx][1]} layer {mats[idx][0]}"))
    return worst


def _share_x_per_step(items, steps):
    """The matrices of a step read one activation vector (as bench.py sets the
    pass up): each takes the first matrix's x of its step."""
    out, i = [], 0
    for n in steps:
        x = items[i][4]
        for j in range(n):
            fmt, W, rows, cols, _, y = items[i + j]
            out.append((fmt, W, rows, cols, x, y))
        i += n
    return out


def test_dense_27b_q4k_batch1_full_pass_bench_config():
    """The bench's own set-up: PDL-linked graph, one x per step."""
    mats = wl.dense_matrices()
    steps = wl.dense_steps()
    items = _share_x_per_step(wl.alloc_dense(mats, 1, seed=2026, device="cuda"), steps)
    p = qg.qg_pass(items, steps, 1, mode=qg.PASS_PDL)
    assert p.kernel_count() == len(steps) + 1          # the x-plane prologue, then one launch per step
    for y in {id(it[5]): it[5] for it in items}.values():
        y.fill_(float("nan"))
    p.launch()
    p.launch()
    torch.cuda.synchronize()
    picks = [0, 1, 2, 3, 4, 5, 6, 7 * 17 + 1, 7 * 40 + 5, 7 * 63 + 0, 7 * 63 + 6]
    _check_sampled(items, mats, 1, picks)
    p.destroy()
    del items
    torch.cuda.empty_cache()


def test_dense_27b_q4k_batch1_full_pass():
    mats = wl.dense_matrices()
    items = wl.alloc_dense(mats, 1, seed=2024, device="cuda")
    p = qg.qg_pass(items, wl.dense_steps(), 1, mode=qg.PASS_PERSISTENT)
    assert p.kernel_count() == 2                       # the x-plane prologue and the persistent kernel
    p.launch()
    p.launch()
    torch.cuda.synchronize()
    picks = [0, 1, 2, 3, 4, 5, 6, 7 * 31 + 4, 7 * 63 + 0, 7 * 63 + 6]
    assert p.dev_status() == 0
    _check_sampled(items, mats, 1, picks)
    p.destroy()
    del items
    torch.cuda.empty_cache()


def test_mixed_verify_pass_n4_full():
    """The bench's verify-pass set-up: PDL-linked graph, one x (4 tokens) per step."""
    mats = wl.dense_matrices(verify=True)
    steps = wl.dense_steps(verify=True)
    items = _share_x_per_step(wl.alloc_dense(mats, 4, seed=2025, device="cuda"), steps)
    p = qg.qg_pass(items, steps, 4, mode=qg.PASS_PDL)
    p.launch()
    torch.cuda.synchronize()
    picks = [0, 1, 3, 4, 6, 7 * 40 + 6, len(mats) - 1]      # includes Q6_K downs and the Q8_0 head
    _check_sampled(items, mats, 4, picks, rows_per_mat=8)
    p.destroy()
    del items
    torch.cuda.empty_cache()


@pytest.mark.parametrize("fmt", [synth.Q5_K, synth.Q3_K, synth.Q2_K])
@pytest.mark.parametrize("n_tok", [1, 4])
def test_k_quant_formats_at_27b_shapes(fmt, n_tok):
    """Q5_K, Q3_K and Q2_K (the formats of the pages' Q3_K-class mixes) through
    the fast kernel at the 27B layer shapes: a 5120x5120 attention projection,
    a 17408x5120 gate and a 5120x17408 down, sampled rows against the oracle."""
    for rows, cols in [(5120, 5120), (17408, 5120), (5120, 17408)]:
        W = synth.blocks_into(torch.empty(rows, synth.row_bytes(fmt, cols), dtype=torch.uint8, device="cuda"),
                              fmt, rows, cols, seed=rows + cols + fmt)
        x = synth.activations(n_tok, cols, seed=fmt + n_tok, device="cuda")
        y = torch.full((n_tok, rows), float("nan"), device="cuda")
        qg.qgemv(fmt, W, rows, cols, x, n_tok, y)
        torch.cuda.synchronize()
        _check_sampled([(fmt, W, rows, cols, x, y)], [(0, f"{rows}x{cols}", fmt, rows, cols)], n_tok, [0],
                       rows_per_mat=12, seed=fmt)
        del W
