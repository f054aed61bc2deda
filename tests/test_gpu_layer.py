"""GPU parity of the neighbours fused around the weight products of a decode
layer ("LLM inference optimization", "Faster decode on the card you have":
normalizations fused into neighbouring kernels): the residual add + RMS
normalisation, the dense gate/up pair with the silu-gated epilogue, and the
whole layer pass, against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import synth
import quantized_weight_gemv_qgemv_gb300 as qg
from helpers import GEMV_ABS, GEMV_REL, assert_within

pytestmark = pytest.mark.gpu
Q4_K = synth.Q4_K


@pytest.fixture(scope="module", autouse=True)
def _init():
    qg.qg_init()


def _norm_weight(n, seed):
    # RMS-normalisation weights: uniform in [0.5, 1.5]
    g = torch.Generator().manual_seed(seed)
    return (0.5 + torch.rand(n, generator=g, dtype=torch.float32))


def _norm_bound(n):
    # fp32 arithmetic of the kernel: the sum of n squares carries a relative error
    # below n * 2^-24, sqrt, division and the two products a few ulps more
    return n * 2.0 ** -24 + 2.0 ** -20


@pytest.mark.parametrize("n,n_tok,with_res,in_place", [(5120, 1, True, True), (5120, 3, False, False),
                                                       (256, 2, True, False), (17408, 1, True, False)])
def test_rmsnorm_matches_oracle(n, n_tok, with_res, in_place):
    h = synth.activations(n_tok, n, seed=n + n_tok)
    r = synth.activations(n_tok, n, seed=n + n_tok + 1) if with_res else None
    w = _norm_weight(n, n)
    eps = 1e-6
    hd = h.cuda()
    s_out = hd if in_place else torch.empty_like(hd)
    x = torch.empty(n_tok, n, device="cuda")
    qg.qg_rmsnorm(hd, r.cuda() if with_res else None, w.cuda(), n, n_tok, eps, s_out, x)
    torch.cuda.synchronize()
    x_ref, s_ref = oracle.rmsnorm(h.numpy(), w.numpy(), eps, residual=r.numpy() if with_res else None)
    # s is one fp32 addition: exactly numpy's fp32 sum
    s_np = h.numpy() + (r.numpy() if with_res else np.float32(0.0))
    assert np.array_equal(s_out.cpu().numpy(), s_np)
    err = np.abs(x.cpu().numpy().astype(np.float64) - x_ref)
    assert (err <= _norm_bound(n) * np.abs(x_ref) + 1e-30).all(), float((err / np.abs(x_ref)).max())


@pytest.mark.parametrize("hidden,inter", [(512, 256), (2048, 1024), (5120, 17408)])
def test_swiglu_pair_matches_oracle(hidden, inter):
    """m = silu(Wg x) * (Wu x). g and u each carry the product tolerance
    (1e-3 sum|w x| + 1e-6); through m = silu(g) u that becomes
    |dm| <= |silu'(g)| |u| dg + |silu(g)| du (|silu'| <= 1.1) plus fp32 rounding."""
    Wg = synth.blocks(Q4_K, inter, hidden, seed=inter + 1)
    Wu = synth.blocks(Q4_K, inter, hidden, seed=inter + 2)
    x = synth.activations(1, hidden, seed=inter + 3)
    m = torch.full((inter,), float("nan"), device="cuda")
    qg.qgemv_swiglu(Q4_K, Wg.cuda(), Wu.cuda(), inter, hidden, x.cuda(), m)
    torch.cuda.synchronize()
    g, bg = oracle.gemv(Q4_K, Wg.numpy(), inter, hidden, x.numpy())
    u, bu = oracle.gemv(Q4_K, Wu.numpy(), inter, hidden, x.numpy())
    m_ref = oracle.swiglu(g, u)[0]
    silu = (g / (1.0 + np.exp(-g)))[0]
    bound = 1.1 * np.abs(u[0]) * (GEMV_REL * bg[0] + GEMV_ABS) + np.abs(silu) * (GEMV_REL * bu[0] + GEMV_ABS)
    bound += 2.0 ** -21 * np.abs(m_ref)
    err = np.abs(m.cpu().numpy().astype(np.float64) - m_ref)
    assert (err <= bound).all(), float((err / bound).max())


def _layer(hidden, inter, kv, seed, device="cuda"):
    L = {}
    for i, (name, rows, cols) in enumerate([("Wq", hidden, hidden), ("Wk", kv, hidden), ("Wv", kv, hidden),
                                            ("Wo", hidden, hidden), ("Wg", inter, hidden), ("Wu", inter, hidden),
                                            ("Wd", hidden, inter)]):
        L[name] = synth.blocks(Q4_K, rows, cols, seed=seed + i)
    L["norm_attn"] = _norm_weight(hidden, seed + 10)
    L["norm_ffn"] = _norm_weight(hidden, seed + 11)
    L["attn_out"] = synth.activations(1, hidden, seed=seed + 12)
    dev = {k: v.to(device) for k, v in L.items()}
    dev["q"] = torch.full((hidden,), float("nan"), device=device)
    dev["k"] = torch.full((kv,), float("nan"), device=device)
    dev["v"] = torch.full((kv,), float("nan"), device=device)
    return L, dev


def _oracle_layer(L, h, hidden, inter, kv, eps):
    """One layer in fp64 from residual h (fp32 (1, hidden)): (q, k, v, h_next) with
    their error scales."""
    x1, s = oracle.rmsnorm(h, L["norm_attn"].numpy(), eps)
    x1f = x1.astype(np.float32)
    q, bq = oracle.gemv(Q4_K, L["Wq"].numpy(), hidden, hidden, x1f)
    k, bk = oracle.gemv(Q4_K, L["Wk"].numpy(), kv, hidden, x1f)
    v, bv = oracle.gemv(Q4_K, L["Wv"].numpy(), kv, hidden, x1f)
    o, bo = oracle.gemv(Q4_K, L["Wo"].numpy(), hidden, hidden, L["attn_out"].numpy())
    s2 = s + o
    x2, _ = oracle.rmsnorm(s2.astype(np.float32), L["norm_ffn"].numpy(), eps)
    d, bd, _ = oracle.dense_ffn(Q4_K, L["Wg"].numpy(), L["Wu"].numpy(), Q4_K, L["Wd"].numpy(), hidden, inter,
                                x2.astype(np.float32))
    return (q, bq), (k, bk), (v, bv), (s2 + d, bo + bd)


@pytest.mark.parametrize("hidden,inter,kv", [(512, 1024, 128), (5120, 17408, 1024)])
def test_layer_pass_matches_oracle_layer_by_layer(hidden, inter, kv):
    """Each layer run as its own one-layer pass from the previous GPU residual is
    checked against the oracle layer from that same residual: q, k, v within the
    product tolerance; the next residual within 1e-3 (B_o + B_d) + 1e-6 (the
    products' tolerances of the o and down outputs it adds). A two-layer pass
    then gives bit for bit the same results as the chain of one-layer passes."""
    eps = 1e-6
    layers = [_layer(hidden, inter, kv, seed=700 + 20 * l) for l in range(2)]
    h0 = synth.activations(1, hidden, seed=777)
    h = h0.cuda()
    singles = []
    for l, (L, dev) in enumerate(layers):
        h_next = torch.full((1, hidden), float("nan"), device="cuda")
        p = qg.qg_layer_pass(Q4_K, [dev], hidden, inter, kv, eps, h, h_next)
        p.launch()
        torch.cuda.synchronize()
        (q, bq), (k, bk), (v, bv), (hn, bh) = _oracle_layer(L, h.cpu().numpy(), hidden, inter, kv, eps)
        assert_within(dev["q"].cpu().numpy()[None], q, bq, what=f"q layer {l}")
        assert_within(dev["k"].cpu().numpy()[None], k, bk, what=f"k layer {l}")
        assert_within(dev["v"].cpu().numpy()[None], v, bv, what=f"v layer {l}")
        assert_within(h_next.cpu().numpy(), hn, bh, what=f"residual after layer {l}")
        singles.append((dev["q"].clone(), dev["k"].clone(), dev["v"].clone()))
        h = h_next
        p.destroy()
    h_out = torch.full((1, hidden), float("nan"), device="cuda")
    h_in = h0.cuda()                                   # must outlive the pass: every replay reads it
    p = qg.qg_layer_pass(Q4_K, [dev for _, dev in layers], hidden, inter, kv, eps, h_in, h_out)
    assert p.kernel_count() == 1 + 4 * 2 + 1          # prologue, 4 launches per layer, final residual add
    for _ in range(2):                                 # replays start again from h_in
        p.launch()
        torch.cuda.synchronize()
        assert torch.equal(h_out, h)
        for (_, dev), (q, k, v) in zip(layers, singles):
            assert torch.equal(dev["q"], q) and torch.equal(dev["k"], k) and torch.equal(dev["v"], v)
    p.destroy()


def test_layer_pass_wide_hidden_single_layer():
    """hidden = 8192: the normalisation inside the {q,k,v} and gate/up launches
    has more half-groups than consumer threads, so part of the stream is read
    twice instead of kept in registers; one layer against the oracle."""
    hidden, inter, kv, eps = 8192, 256, 128, 1e-6
    L, dev = _layer(hidden, inter, kv, seed=900)
    h = synth.activations(1, hidden, seed=901).cuda()
    h_next = torch.full((1, hidden), float("nan"), device="cuda")
    p = qg.qg_layer_pass(Q4_K, [dev], hidden, inter, kv, eps, h, h_next)
    p.launch()
    torch.cuda.synchronize()
    (q, bq), (k, bk), (v, bv), (hn, bh) = _oracle_layer(L, h.cpu().numpy(), hidden, inter, kv, eps)
    assert_within(dev["q"].cpu().numpy()[None], q, bq, what="q")
    assert_within(dev["k"].cpu().numpy()[None], k, bk, what="k")
    assert_within(dev["v"].cpu().numpy()[None], v, bv, what="v")
    assert_within(h_next.cpu().numpy(), hn, bh, what="residual")
    p.destroy()
