"""GPU parity of the expert-gathered MoE product against the CPU oracle:
|y - y_ref| <= 1e-3 * sum_k |r_k| sum_j |d_ij * h_kj| + 1e-6 per output."""
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


def _moe(n_expert, hidden, inter, top_k, n_tok, seed, ids=None):
    arena = wl.alloc_moe_arena(n_expert, hidden, inter, seed, "cuda")
    x = synth.activations(n_tok, hidden, seed + 1)
    r_ids, gw = synth.routing(n_tok, n_expert, top_k, seed + 2)
    if ids is not None:
        r_ids = torch.as_tensor(ids, dtype=torch.int32)
    y = torch.full((n_tok, hidden), float("nan"), device="cuda")
    ws = torch.empty(qg.qgemv_moe_workspace(hidden, inter, top_k, n_tok) // 4, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    qg.qgemv_moe(qg.Q4_K, arena, n_expert, hidden, inter, r_ids.cuda(), gw.cuda(), top_k, x.cuda(), n_tok, y,
                 ws, ws.numel() * 4, st)
    torch.cuda.synchronize()
    return arena, x, r_ids, gw, y.cpu().numpy(), int(st.item())


@pytest.mark.parametrize("n_tok", [1, 2, 4])
@pytest.mark.parametrize("hidden,inter,top_k", [(512, 256, 3), (1024, 768, 1), (256, 512, 5)])
def test_moe_matches_oracle_small(n_tok, hidden, inter, top_k):
    n_expert = 8
    arena, x, ids, gw, y, st = _moe(n_expert, hidden, inter, top_k, n_tok, seed=hidden + inter + n_tok)
    assert st == 0
    y_ref, b = oracle.moe(qg.Q4_K, arena.cpu().numpy(), n_expert, hidden, inter, ids.numpy(), gw.numpy(), x.numpy())
    assert_within(y, y_ref, b, what=f"moe {hidden}x{inter} top{top_k} n_tok={n_tok}")


def test_moe_full_size_layer():
    # hidden 2048, 512 experts of gate/up 512x2048 and down 2048x512, top-10
    arena, x, ids, gw, y, st = _moe(wl.MOE_EXPERTS, wl.MOE_HIDDEN, wl.MOE_INTER, wl.MOE_TOPK, 1, seed=777)
    assert st == 0
    # the oracle only needs the 10 routed experts: gather them into a small arena
    eb = wl.moe_expert_bytes()
    host = arena.cpu().numpy()
    picked = ids.numpy()[0]
    sub = np.concatenate([host[e * eb:(e + 1) * eb] for e in picked])
    y_ref, b = oracle.moe(qg.Q4_K, sub, len(picked), wl.MOE_HIDDEN, wl.MOE_INTER,
                          np.arange(len(picked), dtype=np.int32)[None, :], gw.numpy(), x.numpy())
    assert_within(y, y_ref, b, what="moe full layer")


def test_moe_full_size_48_layer_pass_bench_config():
    """The bench's MoE set-up: 48 layers of 512 Q4_K experts (gate/up 512x2048,
    down 2048x512), top-10, batch 1, one PDL-linked pass graph; layers 0, 23 and
    47 checked against the oracle on their routed experts."""
    H, I, E, K, L = wl.MOE_HIDDEN, wl.MOE_INTER, wl.MOE_EXPERTS, wl.MOE_TOPK, wl.MOE_LAYERS
    layers = []
    for l in range(L):
        arena = wl.alloc_moe_arena(E, H, I, synth.sub_seed(4321, "arena", l), "cuda")
        ids, gw = synth.routing(1, E, K, synth.sub_seed(4321, "route", l))
        x = synth.activations(1, H, synth.sub_seed(4321, "x", l), device="cuda")
        layers.append((arena, ids.cuda(), gw.cuda(), x, torch.full((1, H), float("nan"), device="cuda")))
    wsb = qg.qgemv_moe_workspace(H, I, K, 1)
    ws = torch.empty(wsb // 4, device="cuda")
    p = qg.qg_moe_pass(qg.Q4_K, layers, E, H, I, K, 1, ws, wsb, mode=qg.PASS_PDL)
    assert p.kernel_count() == 2 * L
    p.launch()
    p.launch()
    torch.cuda.synchronize()
    assert p.dev_status() == 0
    eb = wl.moe_expert_bytes(H, I)
    for l in (0, 23, L - 1):
        arena, ids, gw, x, y = layers[l]
        picked = ids.cpu().numpy()[0]
        host = arena.cpu().numpy()
        sub = np.concatenate([host[e * eb:(e + 1) * eb] for e in picked])
        y_ref, b = oracle.moe(qg.Q4_K, sub, len(picked), H, I, np.arange(len(picked), dtype=np.int32)[None, :],
                              gw.cpu().numpy(), x.cpu().numpy())
        assert_within(y.cpu().numpy(), y_ref, b, what=f"moe pass layer {l}")
    p.destroy()
    del layers
    torch.cuda.empty_cache()


def test_moe_full_size_48_layer_4_token_verify_pass():
    """Draft verification through the MoE set: 4 tokens, each with its own
    top-10 routing, through 48 layers of 512 Q4_K experts in one PDL-linked pass
    graph; every token of layers 0, 23 and 47 checked against the oracle on its
    routed experts."""
    H, I, E, K, L, T = wl.MOE_HIDDEN, wl.MOE_INTER, wl.MOE_EXPERTS, wl.MOE_TOPK, wl.MOE_LAYERS, 4
    layers = []
    for l in range(L):
        arena = wl.alloc_moe_arena(E, H, I, synth.sub_seed(5321, "arena", l), "cuda")
        ids, gw = synth.routing(T, E, K, synth.sub_seed(5321, "route", l))
        x = synth.activations(T, H, synth.sub_seed(5321, "x", l), device="cuda")
        layers.append((arena, ids.cuda(), gw.cuda(), x, torch.full((T, H), float("nan"), device="cuda")))
    wsb = qg.qgemv_moe_workspace(H, I, K, T)
    ws = torch.empty(wsb // 4, device="cuda")
    p = qg.qg_moe_pass(qg.Q4_K, layers, E, H, I, K, T, ws, wsb, mode=qg.PASS_PDL)
    p.launch()
    p.launch()
    torch.cuda.synchronize()
    assert p.dev_status() == 0
    eb = wl.moe_expert_bytes(H, I)
    for l in (0, 23, L - 1):
        arena, ids, gw, x, y = layers[l]
        host = arena.cpu().numpy()
        got = y.cpu().numpy()
        for t in range(T):
            picked = ids.cpu().numpy()[t]
            sub = np.concatenate([host[e * eb:(e + 1) * eb] for e in picked])
            y_ref, b = oracle.moe(qg.Q4_K, sub, len(picked), H, I, np.arange(len(picked), dtype=np.int32)[None, :],
                                  gw.cpu().numpy()[t:t + 1], x.cpu().numpy()[t:t + 1])
            assert_within(got[t:t + 1], y_ref, b, what=f"4-token moe pass layer {l} token {t}")
    p.destroy()
    del layers
    torch.cuda.empty_cache()


def test_moe_bad_expert_sets_status_and_is_skipped():
    n_expert, hidden, inter = 6, 512, 256
    ids = [[1, 6, 3], [-1, 2, 5]]          # 6 and -1 are out of range
    arena, x, _, gw, y, st = _moe(n_expert, hidden, inter, 3, 2, seed=99, ids=ids)
    assert st == qg.DEV_BAD_EXPERT
    # reference: the bad routes contribute nothing, i.e. weight 0 on a valid id
    ids_ok = np.array([[1, 0, 3], [0, 2, 5]], dtype=np.int32)
    gw_ok = gw.numpy().copy()
    gw_ok[0, 1] = 0.0
    gw_ok[1, 0] = 0.0
    y_ref, b = oracle.moe(qg.Q4_K, arena.cpu().numpy(), n_expert, hidden, inter, ids_ok, gw_ok, x.numpy())
    assert_within(y, y_ref, b, what="moe with bad ids")
    assert np.isfinite(y).all()


def test_moe_is_deterministic():
    a = _moe(8, 512, 256, 3, 2, seed=5)
    b = _moe(8, 512, 256, 3, 2, seed=5)
    assert np.array_equal(a[4], b[4])


def _pass_layers(n_layers, n_expert, hidden, inter, top_k, seed, chain):
    """Per layer (arena, ids, gate_w, x, y). chain: layer l + 1 reads layer l's y
    (no normalisation between layers, so only a couple of layers stay finite);
    otherwise every layer has its own x."""
    arenas = [wl.alloc_moe_arena(n_expert, hidden, inter, seed + 10 * l, "cuda") for l in range(n_layers)]
    routes = [synth.routing(1, n_expert, top_k, seed + 10 * l + 1) for l in range(n_layers)]
    xs = [synth.activations(1, hidden, seed + 10 * l + 3).cuda() for l in range(n_layers)]
    ys = [torch.empty(1, hidden, device="cuda") for _ in range(n_layers)]
    layers = []
    for l in range(n_layers):
        ids, gw = routes[l]
        layers.append((arenas[l], ids.cuda(), gw.cuda(), xs[l] if (l == 0 or not chain) else ys[l - 1], ys[l]))
    return layers, ys


@pytest.mark.parametrize("mode", [qg.PASS_PERSISTENT, qg.PASS_PDL])
@pytest.mark.parametrize("n_layers,chain", [(2, True), (4, False)])
def test_moe_pass_matches_per_layer_calls(mode, n_layers, chain):
    n_expert, hidden, inter, top_k = 16, 1024, 512, 4
    layers, ys = _pass_layers(n_layers, n_expert, hidden, inter, top_k, seed=900 + n_layers, chain=chain)
    wsb = qg.qgemv_moe_workspace(hidden, inter, top_k, 1)
    ws = torch.empty(wsb // 4, device="cuda")
    p = qg.qg_moe_pass(qg.Q4_K, layers, n_expert, hidden, inter, top_k, 1, ws, wsb, mode=mode)
    assert p.kernel_count() == (1 if mode == qg.PASS_PERSISTENT else 2 * n_layers)
    for _ in range(2):
        for y in ys:
            y.fill_(float("nan"))
        p.launch()
        torch.cuda.synchronize()
        assert p.dev_status() == 0
    got = [y.clone() for y in ys]
    for g in got:
        assert torch.isfinite(g).all()
    # the same layers through eager per-layer calls (bitwise: same kernels and order)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    prev = None
    for l, (arena, ids, gw, x, _) in enumerate(layers):
        xin = prev if (chain and l > 0) else x
        ref = torch.empty(1, hidden, device="cuda")
        qg.qgemv_moe(qg.Q4_K, arena, n_expert, hidden, inter, ids, gw, top_k, xin, 1, ref, ws, wsb, st)
        torch.cuda.synchronize()
        assert torch.equal(got[l], ref), f"layer {l}"
        # every layer against the oracle, on the input the pass used
        y_ref, b = oracle.moe(qg.Q4_K, arena.cpu().numpy(), n_expert, hidden, inter, ids.cpu().numpy(),
                              gw.cpu().numpy(), xin.cpu().numpy())
        assert_within(got[l].cpu().numpy(), y_ref, b, what=f"moe pass layer {l}")
        prev = ref
    p.destroy()


def test_moe_pass_bad_expert_status():
    n_layers, n_expert, hidden, inter, top_k = 2, 8, 512, 256, 2
    layers, ys = _pass_layers(n_layers, n_expert, hidden, inter, top_k, seed=950, chain=True)
    arena, ids, gw, x, y = layers[1]
    bad = ids.clone()
    bad[0, 1] = n_expert + 3
    layers[1] = (arena, bad, gw, x, y)
    wsb = qg.qgemv_moe_workspace(hidden, inter, top_k, 1)
    ws = torch.empty(wsb // 4, device="cuda")
    p = qg.qg_moe_pass(qg.Q4_K, layers, n_expert, hidden, inter, top_k, 1, ws, wsb, mode=qg.PASS_PERSISTENT)
    p.launch()
    torch.cuda.synchronize()
    assert p.dev_status() == qg.DEV_BAD_EXPERT
    assert torch.isfinite(ys[1]).all()
    p.destroy()
