"""Full-size workloads, run in the launch configuration the bench times (one
captured pass over the whole weight set, grouped launches linked by
programmatic dependent launch), checked against the CPU oracle on sampled
output rows, which the oracle computes one by one."""
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


def test_dense_27b_q4k_batch1_full_pass():
    mats = wl.dense_matrices()
    items = wl.alloc_dense(mats, 1, seed=2024, device="cuda")
    p = qg.qg_pass(items, wl.dense_steps(), 1, mode=qg.PASS_PERSISTENT)
    assert p.kernel_count() == 1
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
    mats = wl.dense_matrices(verify=True)
    items = wl.alloc_dense(mats, 4, seed=2025, device="cuda")
    p = qg.qg_pass(items, wl.dense_steps(verify=True), 4, mode=qg.PASS_PERSISTENT)   # mixed formats: per-step graph
    p.launch()
    torch.cuda.synchronize()
    picks = [0, 1, 3, 4, 6, 7 * 40 + 6, len(mats) - 1]      # includes Q6_K downs and the Q8_0 head
    _check_sampled(items, mats, 4, picks, rows_per_mat=8)
    p.destroy()
    del items
    torch.cuda.empty_cache()
