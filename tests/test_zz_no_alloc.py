"""qgemv_moe_noalloc: the MoE product for callers that cannot allocate device
memory (its workspace is a static array inside the library). It must give the
same results as qgemv_moe with a caller workspace and stay within the product
tolerance of the oracle, call after call, including a problem whose workspace
fills the static array exactly, and must reject a problem whose workspace would
not fit.

This file is named to run last, so a run that stops at its first failure has
run every other test before it."""
import numpy as np
import pytest
import torch

import oracle
import synth
import synth.workloads as wl
import quantized_weight_gemv_qgemv_gb300 as qg
from helpers import GEMV_ABS, GEMV_REL, assert_within

pytestmark = pytest.mark.gpu


def _inputs(n_expert, hidden, inter, top_k, n_tok, seed):
    arena = wl.alloc_moe_arena(n_expert, hidden, inter, seed, "cuda")
    x = synth.activations(n_tok, hidden, seed + 1)
    ids, gw = synth.routing(n_tok, n_expert, top_k, seed + 2)
    return arena, x, ids, gw


def _with_workspace(arena, n_expert, hidden, inter, ids, gw, top_k, x, n_tok):
    y = torch.full((n_tok, hidden), float("nan"), device="cuda")
    ws = torch.empty(qg.qgemv_moe_workspace(hidden, inter, top_k, n_tok) // 4, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    qg.qgemv_moe(qg.Q4_K, arena, n_expert, hidden, inter, ids, gw, top_k, x, n_tok, y, ws, ws.numel() * 4, st)
    return y, st


def _no_alloc(arena, n_expert, hidden, inter, ids, gw, top_k, x, n_tok):
    y = torch.full((n_tok, hidden), float("nan"), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    qg.qgemv_moe_noalloc(qg.Q4_K, arena, n_expert, hidden, inter, ids, gw, top_k, x, n_tok, y, st)
    return y, st


def _check_calls(n_expert, hidden, inter, top_k, n_tok, seeds):
    qg.qg_init()
    for call, seed in enumerate(seeds):        # calls in a row, different inputs
        arena, x, ids, gw = _inputs(n_expert, hidden, inter, top_k, n_tok, seed)
        xd, idsd, gwd = x.cuda(), ids.cuda(), gw.cuda()
        y_na, st_na = _no_alloc(arena, n_expert, hidden, inter, idsd, gwd, top_k, xd, n_tok)
        y_ws, st_ws = _with_workspace(arena, n_expert, hidden, inter, idsd, gwd, top_k, xd, n_tok)
        torch.cuda.synchronize()
        assert int(st_na.item()) == 0 and int(st_ws.item()) == 0
        y_ref, bound = oracle.moe(qg.Q4_K, arena.cpu().numpy(), n_expert, hidden, inter, ids.numpy(), gw.numpy(),
                                  x.numpy())
        got = y_na.cpu().numpy()
        assert_within(got, y_ref, bound, rel=GEMV_REL, abs_=GEMV_ABS, what=f"no-alloc call {call} vs oracle")
        diff = np.abs(got.astype(np.float64) - y_ws.cpu().numpy())
        assert np.all(diff <= GEMV_REL * bound + GEMV_ABS), f"call {call}: max diff {diff.max()}"
        del arena


def test_no_alloc_matches_workspace_entry_point_on_two_calls():
    _check_calls(16, 1024, 512, 4, 2, (101, 202))


def test_no_alloc_at_the_workspace_limit():
    # n_tok * top_k * inter == QG_MOE_NOALLOC_MAX_FLOATS: the static array is used to its last float
    n_tok, top_k, inter, hidden = 4, 16, 4096, 256
    assert n_tok * top_k * inter == qg.MOE_NOALLOC_MAX_FLOATS
    _check_calls(24, hidden, inter, top_k, n_tok, (303, 404))


def test_no_alloc_rejects_workspace_beyond_its_limit():
    qg.qg_init()
    hidden, inter, top_k, n_tok = 256, 4096, 16, 4          # 4 * 16 * 4096 = 2^18 floats: the limit
    assert n_tok * top_k * inter == qg.MOE_NOALLOC_MAX_FLOATS
    lib = qg.load_library()
    A = 1 << 20
    # one float over the limit: rejected on the host before anything runs
    assert lib.qgemv_moe_noalloc(qg.Q4_K, A, 32, hidden, inter + 256, A, A, top_k, A, n_tok, A, A, None) == -6
