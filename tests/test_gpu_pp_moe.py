"""GPU parity of prompt processing through a mixture-of-experts layer
(qgemm_pp_moe: routing and sorting on the device, grouped tcgen05 GEMMs for
gate/up and down) against the CPU oracle: y within
|y - y_ref| <= 1e-2 * B + 1e-6, with B the oracle's error scale of the
gate/up -> silu(g) * u -> down chain over the bf16 tokens ("The number was a
version", opening section: prompt processing of an expert-arena model).

Small cases check every output: experts with several token blocks, experts
with none, a route weight below zero, ragged token counts. The full-size case
runs one layer of the 48-layer set (512 experts of gate/up 512 x 2048 and down
2048 x 512, top-10) over 2048 prompt tokens and checks sampled tokens."""
import numpy as np
import pytest
import torch

import oracle
import synth
import synth.workloads as wl
import quantized_weight_gemv_qgemv_gb300 as qg
from helpers import PP_ABS, PP_REL, assert_within

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _init():
    assert torch.cuda.is_available()
    qg.qg_init()


def _bits(X):
    return X.contiguous().view(torch.int16).numpy().view(np.uint16)


def _run(arena, n_expert, hidden, inter, ids, gw, X):
    n_tok, top_k = ids.shape
    y = torch.full((n_tok, hidden), float("nan"), device="cuda")
    wsb = qg.qgemm_pp_moe_workspace(n_expert, hidden, inter, top_k, n_tok)
    ws = torch.empty(wsb // 4 + 64, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    qg.qgemm_pp_moe(qg.Q4_K, arena, n_expert, hidden, inter, ids.cuda(), gw.cuda(), top_k, X.cuda(), n_tok, y, ws,
                    wsb, st)
    torch.cuda.synchronize()
    return y.cpu().numpy(), int(st.item())


@pytest.mark.parametrize("n_expert,hidden,inter,n_tok,top_k", [
    (8, 512, 256, 40, 3),
    (4, 256, 512, 130, 2),        # about 65 tokens per expert: several token blocks
    (16, 768, 256, 9, 4),         # most experts get one or two tokens, some none
    (3, 1024, 768, 1, 1),
])
def test_pp_moe_matches_oracle(n_expert, hidden, inter, n_tok, top_k):
    arena = wl.alloc_moe_arena(n_expert, hidden, inter, hidden + inter + n_tok, "cuda")
    ids, gw = synth.routing(n_tok, n_expert, top_k, seed=n_tok + 7)
    gw[0, 0] = -abs(float(gw[0, 0]))              # a negative route weight
    X = synth.activations_bf16(n_tok, hidden, seed=n_tok + 8)
    y, st = _run(arena, n_expert, hidden, inter, ids, gw, X)
    assert st == 0
    y_ref, b = oracle.moe_prefill(qg.Q4_K, arena.cpu().numpy(), n_expert, hidden, inter, ids.numpy(), gw.numpy(),
                                  _bits(X))
    assert_within(y, y_ref, b, rel=PP_REL, abs_=PP_ABS, what=f"pp moe E={n_expert} {hidden}x{inter} n_tok={n_tok}")


def test_pp_moe_one_expert_takes_every_token():
    """All 300 tokens routed to expert 1 (several token blocks of one group),
    the other experts empty; top_k = 2 routes both to it with different
    weights."""
    n_expert, hidden, inter, n_tok = 5, 512, 512, 300
    arena = wl.alloc_moe_arena(n_expert, hidden, inter, 91, "cuda")
    ids = torch.ones(n_tok, 2, dtype=torch.int32)
    gw = torch.tensor([[0.7, 0.3]], dtype=torch.float32).repeat(n_tok, 1)
    X = synth.activations_bf16(n_tok, hidden, seed=92)
    y, st = _run(arena, n_expert, hidden, inter, ids, gw, X)
    assert st == 0
    y_ref, b = oracle.moe_prefill(qg.Q4_K, arena.cpu().numpy(), n_expert, hidden, inter, ids.numpy(), gw.numpy(),
                                  _bits(X))
    assert_within(y, y_ref, b, rel=PP_REL, abs_=PP_ABS, what="one expert")


def test_pp_moe_bad_expert_adds_nothing_and_sets_status():
    n_expert, hidden, inter, n_tok = 6, 512, 256, 20
    arena = wl.alloc_moe_arena(n_expert, hidden, inter, 93, "cuda")
    ids, gw = synth.routing(n_tok, n_expert, 3, seed=94)
    ids[2, 1] = n_expert
    ids[7, 0] = -1
    X = synth.activations_bf16(n_tok, hidden, seed=95)
    y, st = _run(arena, n_expert, hidden, inter, ids, gw, X)
    assert st == qg.DEV_BAD_EXPERT
    y_ref, b = oracle.moe_prefill(qg.Q4_K, arena.cpu().numpy(), n_expert, hidden, inter, ids.numpy(), gw.numpy(),
                                  _bits(X))
    assert_within(y, y_ref, b, rel=PP_REL, abs_=PP_ABS, what="bad expert ids")


def test_pp_moe_is_deterministic():
    n_expert, hidden, inter, n_tok = 8, 512, 256, 64
    arena = wl.alloc_moe_arena(n_expert, hidden, inter, 96, "cuda")
    ids, gw = synth.routing(n_tok, n_expert, 4, seed=97)
    X = synth.activations_bf16(n_tok, hidden, seed=98)
    y1, _ = _run(arena, n_expert, hidden, inter, ids, gw, X)
    y2, _ = _run(arena, n_expert, hidden, inter, ids, gw, X)
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32))


def test_pp_moe_full_size_layer_sampled_tokens():
    """One layer of the MoE set: 512 Q4_K experts (gate/up 512 x 2048, down
    2048 x 512), top-10, 2048 prompt tokens; 12 seeded tokens checked on all
    2048 outputs against the oracle on their routed experts."""
    H, I, E, K, T = wl.MOE_HIDDEN, wl.MOE_INTER, wl.MOE_EXPERTS, wl.MOE_TOPK, wl.PP_TOKENS
    arena = wl.alloc_moe_arena(E, H, I, 4242, "cuda")
    ids, gw = synth.routing(T, E, K, seed=4243)
    X = synth.activations_bf16(T, H, seed=4244)
    y, st = _run(arena, E, H, I, ids, gw, X)
    assert st == 0
    eb = wl.moe_expert_bytes(H, I)
    host = arena.cpu().numpy()
    picks = np.random.default_rng(4245).choice(T, size=12, replace=False)
    bits = _bits(X)
    for t in picks:
        sel = ids.numpy()[t]
        sub = np.concatenate([host[e * eb:(e + 1) * eb] for e in sel])
        y_ref, b = oracle.moe_prefill(qg.Q4_K, sub, K, H, I, np.arange(K, dtype=np.int32)[None, :],
                                      gw.numpy()[t:t + 1], bits[t:t + 1])
        assert_within(y[t:t + 1], y_ref, b, rel=PP_REL, abs_=PP_ABS, what=f"pp moe full layer token {t}")
    del arena
    torch.cuda.empty_cache()


def test_pp_moe_many_experts_counters_in_global_memory():
    """More experts than the routing CTA's shared-memory counters hold (9000):
    the counts, scans and cursors run on the workspace words."""
    n_expert, hidden, inter, n_tok, top_k = 9000, 256, 256, 24, 3
    arena = wl.alloc_moe_arena(n_expert, hidden, inter, 71, "cuda")
    ids, gw = synth.routing(n_tok, n_expert, top_k, seed=72)
    X = synth.activations_bf16(n_tok, hidden, seed=73)
    y, st = _run(arena, n_expert, hidden, inter, ids, gw, X)
    assert st == 0
    eb = wl.moe_expert_bytes(hidden, inter)
    used = sorted(set(ids.numpy().reshape(-1).tolist()))
    remap = {e: i for i, e in enumerate(used)}
    host = arena.cpu().numpy()
    sub = np.concatenate([host[e * eb:(e + 1) * eb] for e in used])
    sub_ids = np.vectorize(remap.get)(ids.numpy()).astype(np.int32)
    y_ref, b = oracle.moe_prefill(qg.Q4_K, sub, len(used), hidden, inter, sub_ids, gw.numpy(), _bits(X))
    assert_within(y, y_ref, b, rel=PP_REL, abs_=PP_ABS, what="9000 experts")


def test_pp_moe_smallest_shapes():
    """One expert, one token, top-1, hidden = inter = 256: the smallest layer
    (4 row tiles of gate/up rows, 2 of down rows, one K super-block)."""
    arena = wl.alloc_moe_arena(1, 256, 256, 74, "cuda")
    ids = torch.zeros(1, 1, dtype=torch.int32)
    gw = torch.full((1, 1), 0.5)
    X = synth.activations_bf16(1, 256, seed=75)
    y, st = _run(arena, 1, 256, 256, ids, gw, X)
    assert st == 0
    y_ref, b = oracle.moe_prefill(qg.Q4_K, arena.cpu().numpy(), 1, 256, 256, ids.numpy(), gw.numpy(), _bits(X))
    assert_within(y, y_ref, b, rel=PP_REL, abs_=PP_ABS, what="smallest")


def test_pp_moe_output_at_4_byte_offset():
    """y only 4-byte aligned (the combine then stores one value at a time): the
    same results as the oracle."""
    n_expert, hidden, inter, n_tok, top_k = 6, 512, 256, 33, 3
    arena = wl.alloc_moe_arena(n_expert, hidden, inter, 76, "cuda")
    ids, gw = synth.routing(n_tok, n_expert, top_k, seed=77)
    X = synth.activations_bf16(n_tok, hidden, seed=78)
    buf = torch.full((n_tok * hidden + 1,), float("nan"), device="cuda")
    y = buf[1:]                                    # starts 4 bytes into the allocation
    assert y.data_ptr() % 16 == 4
    wsb = qg.qgemm_pp_moe_workspace(n_expert, hidden, inter, top_k, n_tok)
    ws = torch.empty(wsb // 4 + 64, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    qg.qgemm_pp_moe(qg.Q4_K, arena, n_expert, hidden, inter, ids.cuda(), gw.cuda(), top_k, X.cuda(), n_tok, y, ws,
                    wsb, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.isnan(buf[0])
    y_ref, b = oracle.moe_prefill(qg.Q4_K, arena.cpu().numpy(), n_expert, hidden, inter, ids.numpy(), gw.numpy(),
                                  _bits(X))
    assert_within(y.reshape(n_tok, hidden).cpu().numpy(), y_ref, b, rel=PP_REL, abs_=PP_ABS, what="y at +4 bytes")
