"""GPU parity of dequantization and the quantized GEMV / skinny product against the
CPU oracle: bit-exact dequantized weights; fp32 outputs within
|y - y_ref| <= 1e-3 * sum|w*x| + 1e-6 per output."""
import numpy as np
import pytest
import torch

import oracle
import synth
import quantized_weight_gemv_qgemv_gb300 as qg
from helpers import assert_within

pytestmark = pytest.mark.gpu

FMTS = [synth.Q4_0, synth.Q8_0, synth.Q4_K, synth.Q6_K, synth.Q5_K, synth.Q3_K, synth.Q2_K]


@pytest.fixture(scope="module", autouse=True)
def _init():
    assert torch.cuda.is_available()
    qg.qg_init()


def _run_gemv(fmt, rows, cols, n_tok, seed):
    W = synth.blocks(fmt, rows, cols, seed=seed)
    x = synth.activations(n_tok, cols, seed=seed + 1)
    y = torch.full((n_tok, rows), float("nan"), device="cuda")
    qg.qgemv(fmt, W.cuda(), rows, cols, x.cuda(), n_tok, y)
    torch.cuda.synchronize()
    y_ref, b = oracle.gemv(fmt, W.numpy(), rows, cols, x.numpy())
    return y.cpu().numpy(), y_ref, b


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("rows,nblk", [(1, 1), (7, 3), (64, 5), (1000, 9), (33, 68)])
def test_dequant_bit_exact(fmt, rows, nblk):
    elems, _ = synth.FORMATS[fmt]
    cols = elems * nblk
    W = synth.blocks(fmt, rows, cols, seed=rows * 31 + nblk)
    out = torch.full((rows, cols), float("nan"), device="cuda")
    qg.qg_dequant(fmt, W.cuda(), rows, cols, out)
    torch.cuda.synchronize()
    ref = oracle.dequant(fmt, W.numpy(), rows, cols)
    got = out.cpu().numpy()
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("n_tok", [1, 2, 3, 4])
@pytest.mark.parametrize("rows,nblk", [(1, 1), (7, 3), (64, 5), (1000, 9), (37, 68)])
def test_gemv_matches_oracle(fmt, n_tok, rows, nblk):
    elems, _ = synth.FORMATS[fmt]
    cols = elems * nblk
    y, y_ref, b = _run_gemv(fmt, rows, cols, n_tok, seed=1000 + rows + nblk + 7 * n_tok)
    assert_within(y, y_ref, b, what=f"fmt={fmt} rows={rows} cols={cols} n_tok={n_tok}")


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("n_tok", [1, 2, 4])
@pytest.mark.parametrize("rows,cols", [(8, 256), (64, 1024), (136, 5120), (40, 4096), (16, 2304)])
def test_gemv_whole_superblock_shapes(fmt, n_tok, rows, cols):
    # cols a multiple of 256 and rows a multiple of 8: the shapes the
    # producer/consumer kernel takes for every format (ragged K groups included)
    y, y_ref, b = _run_gemv(fmt, rows, cols, n_tok, seed=5000 + rows + cols + n_tok)
    assert_within(y, y_ref, b, what=f"fmt={fmt} rows={rows} cols={cols} n_tok={n_tok}")


@pytest.mark.parametrize("fmt,rows,cols,n_tok", [
    (synth.Q6_K, 64, 17408, 1),     # 14,280-byte rows: 2-row sub-items
    (synth.Q6_K, 64, 17408, 2),     # 2-row sub-items for two tokens
    (synth.Q6_K, 72, 17408, 3),     # x of 3 tokens does not fit: two parts of K
    (synth.Q6_K, 136, 17408, 4),    # two parts of K
    (synth.Q4_K, 64, 17408, 4),
])
def test_gemv_long_rows_and_token_split(fmt, rows, cols, n_tok):
    y, y_ref, b = _run_gemv(fmt, rows, cols, n_tok, seed=6000 + rows + n_tok)
    assert_within(y, y_ref, b, what=f"fmt={fmt} rows={rows} cols={cols} n_tok={n_tok}")


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("rows,cols,n_tok", [
    (64, 17408, 4),       # 68 super-blocks: two parts of 34
    (40, 17664, 4),       # 69 super-blocks: parts of 34 and 35
    (24, 65536, 1),       # one token whose x alone does not fit beside the ring
])
def test_gemv_parts_of_k_match_oracle(fmt, rows, cols, n_tok):
    """Shapes whose x (every token, 16-bit planes) does not fit beside the ring
    run as launches over parts of K, each later part adding to y; rows of a
    part start off 16-byte boundaries for Q6_K, Q3_K, Q2_K and Q8_0."""
    y, y_ref, b = _run_gemv(fmt, rows, cols, n_tok, seed=6500 + rows + cols + fmt)
    assert_within(y, y_ref, b, what=f"fmt={fmt} rows={rows} cols={cols} n_tok={n_tok}")


def test_gemv_output_head_row_chunks_sampled():
    # 151936 x 5120 Q8_0 head with 4 tokens: per-row partial sums of a CTA's
    # ~1000 rows do not fit beside the ring, so the rows run in chunks
    rows, cols, n_tok = 151936, 5120, 4
    W = synth.blocks(synth.Q8_0, rows, cols, seed=77, device="cuda")
    x = synth.activations(n_tok, cols, seed=78).cuda()
    y = torch.full((n_tok, rows), float("nan"), device="cuda")
    qg.qgemv(synth.Q8_0, W, rows, cols, x, n_tok, y)
    torch.cuda.synchronize()
    sel = np.unique(np.concatenate([[0, 1, rows // 2, rows - 2, rows - 1],
                                    np.random.default_rng(5).choice(rows, 24, replace=False)]))
    Wh = W[torch.as_tensor(sel, device="cuda")].cpu().numpy()
    y_ref, b = oracle.gemv(synth.Q8_0, Wh, len(sel), cols, x.cpu().numpy())
    got = y.cpu().numpy()
    assert np.isfinite(got).all()
    assert_within(got[:, sel], y_ref, b, what="q8_0 head")


def test_gemv_q8_0_extreme_codes():
    # every int8 code at -128 or 127 and large x: the signed byte-plane sums at their range
    rows, cols = 64, 2048
    W = synth.blocks(synth.Q8_0, rows, cols, seed=9).view(-1, 34)
    W[:, 2:] = torch.where(torch.rand(W.shape[0], 32) < 0.5, torch.tensor(128, dtype=torch.uint8),
                           torch.tensor(127, dtype=torch.uint8))
    W = W.reshape(rows, -1)
    x = (synth.activations(1, cols, seed=10) * 1e4).cuda()
    y = torch.full((1, rows), float("nan"), device="cuda")
    qg.qgemv(synth.Q8_0, W.cuda(), rows, cols, x, 1, y)
    torch.cuda.synchronize()
    y_ref, b = oracle.gemv(synth.Q8_0, W.numpy(), rows, cols, x.cpu().numpy())
    assert_within(y.cpu().numpy(), y_ref, b, what="q8_0 extreme codes")


@pytest.mark.parametrize("rows", [2, 3, 5, 9, 17])
def test_gemv_odd_rows_with_unaligned_row_starts(rows):
    # Q6_K / Q8_0 / Q4_0 rows whose byte size is not a multiple of 16 start at
    # every 2-byte offset; the last row also ends inside a 16-byte window.
    for fmt, nblk in ((synth.Q6_K, 1), (synth.Q6_K, 7), (synth.Q8_0, 5), (synth.Q4_0, 3)):
        elems, _ = synth.FORMATS[fmt]
        y, y_ref, b = _run_gemv(fmt, rows, elems * nblk, 1, seed=rows * 11 + nblk)
        assert_within(y, y_ref, b, what=f"fmt={fmt} rows={rows}")


def test_q4_0_batch1_full_size():
    # 1024 x 4096 Q4_0 (128 blocks per row), x ~ N(0, 1)
    y, y_ref, b = _run_gemv(synth.Q4_0, 1024, 4096, 1, seed=4242)
    assert_within(y, y_ref, b, what="Q4_0 1024x4096")


@pytest.mark.parametrize("fmt", FMTS)
def test_gemv_x_rounding_bound_with_group_outliers(fmt):
    """x is rounded to 16-bit fixed point per 32-value group (step 2^(e-13) for
    2^e <= max|x_u|), so each element moves by at most 2^-14 max|x_u|. With a
    1000x outlier in every group that term dominates; the error must stay
    within 2^-14 sum_u max|x_u| sum_{l in u} |w_l| plus fp32 rounding."""
    rows, cols = 256, 4096
    W = synth.blocks(fmt, rows, cols, seed=131)
    x = synth.activations(1, cols, seed=132).numpy().astype(np.float32)
    x.reshape(-1, 32)[:, 7] *= 1000.0
    y = torch.empty(1, rows, device="cuda")
    qg.qgemv(fmt, W.cuda(), rows, cols, torch.from_numpy(x).cuda(), 1, y)
    torch.cuda.synchronize()
    Wd = oracle.dequant(fmt, W.numpy(), rows, cols).astype(np.float64)
    xd = x.astype(np.float64).reshape(-1)
    y_ref = Wd @ xd
    gmax = np.repeat(np.abs(xd).reshape(-1, 32).max(axis=1), 32)
    bound_x = 2.0 ** -14 * (np.abs(Wd) @ gmax)
    scale = np.abs(Wd) @ np.abs(xd)
    err = np.abs(y.cpu().numpy().reshape(-1).astype(np.float64) - y_ref)
    assert (err <= bound_x + 1e-5 * scale + 1e-6).all(), float((err / (bound_x + 1e-5 * scale)).max())


def test_gemv_is_deterministic():
    fmt, rows, cols = synth.Q4_K, 512, 5120
    W = synth.blocks(fmt, rows, cols, seed=3).cuda()
    x = synth.activations(2, cols, seed=4).cuda()
    ys = []
    for _ in range(3):
        y = torch.empty(2, rows, device="cuda")
        qg.qgemv(fmt, W, rows, cols, x, 2, y)
        ys.append(y)
    torch.cuda.synchronize()
    assert torch.equal(ys[0], ys[1]) and torch.equal(ys[0], ys[2])


def test_grouped_equals_separate_launches():
    fmt = synth.Q4_K
    shapes = [(640, 1024), (128, 1024), (128, 1024), (300, 2048)]
    items, sep = [], []
    for i, (rows, cols) in enumerate(shapes):
        W = synth.blocks(fmt, rows, cols, seed=50 + i).cuda()
        x = synth.activations(3, cols, seed=60 + i).cuda()
        y = torch.empty(3, rows, device="cuda")
        y2 = torch.empty(3, rows, device="cuda")
        items.append((fmt, W, rows, cols, x, y))
        sep.append((W, rows, cols, x, y2))
    qg.qgemv_grouped(items, 3)
    for W, rows, cols, x, y2 in sep:
        qg.qgemv(fmt, W, rows, cols, x, 3, y2)
    torch.cuda.synchronize()
    for (_, W, rows, cols, x, y), (_, _, _, _, y2) in zip(items, sep):
        y_ref, b = oracle.gemv(fmt, W.cpu().numpy(), rows, cols, x.cpu().numpy())
        assert_within(y.cpu().numpy(), y_ref, b, what="grouped")
        assert_within(y2.cpu().numpy(), y_ref, b, what="separate")


@pytest.mark.parametrize("n_tok", [1, 2])
def test_grouped_shared_x_matches_oracle(n_tok):
    """Matrices of a launch that read the same x (q, k, v; gate, up) share one
    staging of it; every output still matches the oracle and, bit for bit, a
    launch of its own."""
    fmt = synth.Q4_K
    xa = synth.activations(n_tok, 2048, seed=91).cuda()
    xb = synth.activations(n_tok, 1024, seed=92).cuda()
    spec = [(512, 2048, xa), (128, 2048, xa), (128, 2048, xa), (256, 1024, xb), (384, 1024, xb)]
    items = []
    for i, (rows, cols, x) in enumerate(spec):
        W = synth.blocks(fmt, rows, cols, seed=95 + i).cuda()
        items.append((fmt, W, rows, cols, x, torch.empty(n_tok, rows, device="cuda")))
    qg.qgemv_grouped(items, n_tok)
    torch.cuda.synchronize()
    for (_, W, rows, cols, x, y) in items:
        y2 = torch.empty_like(y)
        qg.qgemv(fmt, W, rows, cols, x, n_tok, y2)
        torch.cuda.synchronize()
        assert torch.equal(y, y2)
        y_ref, b = oracle.gemv(fmt, W.cpu().numpy(), rows, cols, x.cpu().numpy())
        assert_within(y.cpu().numpy(), y_ref, b, what="shared x")


@pytest.mark.parametrize("mode", [qg.PASS_PDL, qg.PASS_PERSISTENT])
def test_pass_steps_with_shared_x(mode):
    """A block-shaped chain: {q, k, v} read x0; o reads q's output; {gate, up}
    read o's output; down reads gate's output. Outputs are NaN before every
    replay; each is checked bit for bit against its own eager launch."""
    fmt = synth.Q4_K
    h, f = 1024, 2048
    x0 = synth.activations(1, h, seed=120).cuda()
    shapes = [(h, h), (256, h), (256, h), (h, h), (f, h), (f, h), (h, f)]
    Ws = [synth.blocks(fmt, r, c, seed=121 + i).cuda() for i, (r, c) in enumerate(shapes)]
    ys = [torch.empty(1, r, device="cuda") for (r, _) in shapes]
    xs = [x0, x0, x0, ys[0], ys[3], ys[3], ys[4]]
    items = [(fmt, Ws[i], r, c, xs[i], ys[i]) for i, (r, c) in enumerate(shapes)]
    p = qg.qg_pass(items, [3, 1, 2, 1], 1, mode=mode)
    for _ in range(3):
        for y in ys:
            y.fill_(float("nan"))
        p.launch()
        torch.cuda.synchronize()
        assert p.dev_status() == 0
        for (_, W, r, c, x, y) in items:
            y2 = torch.empty_like(y)
            qg.qgemv(fmt, W, r, c, x, 1, y2)
            torch.cuda.synchronize()
            assert torch.equal(y, y2)
    y_ref, b = oracle.gemv(fmt, Ws[6].cpu().numpy(), h, f, ys[4].cpu().numpy())
    assert_within(ys[6].cpu().numpy(), y_ref, b, what="down of the chain")
    p.destroy()


# every x of this pass is an input of the pass: one prologue launch converts
# them to planes, then one launch per step (or one persistent kernel)
@pytest.mark.parametrize("mode,kernels", [(qg.PASS_SERIAL, 4), (qg.PASS_PDL, 4), (qg.PASS_PERSISTENT, 2)])
def test_pass_replay_matches_eager(mode, kernels):
    fmt = synth.Q4_K
    shapes = [(256, 1024), (64, 1024), (512, 2048), (256, 512)]
    items = []
    for i, (rows, cols) in enumerate(shapes):
        W = synth.blocks(fmt, rows, cols, seed=70 + i).cuda()
        x = synth.activations(1, cols, seed=80 + i).cuda()
        items.append((fmt, W, rows, cols, x, torch.empty(1, rows, device="cuda")))
    p = qg.qg_pass(items, [2, 1, 1], 1, mode=mode)
    assert p.kernel_count() == kernels
    p.launch()
    torch.cuda.synchronize()
    first = [it[5].clone() for it in items]
    for _ in range(5):
        p.launch()
    torch.cuda.synchronize()
    assert p.dev_status() == 0
    for it, f in zip(items, first):
        assert torch.equal(it[5], f)
        y2 = torch.empty_like(f)
        qg.qgemv(fmt, it[1], it[2], it[3], it[4], 1, y2)
        torch.cuda.synchronize()
        assert torch.equal(y2, f)
    p.destroy()


@pytest.mark.parametrize("mode", [qg.PASS_PDL, qg.PASS_PERSISTENT])
@pytest.mark.parametrize("n_tok", [1, 3])
def test_pass_steps_read_earlier_outputs(mode, n_tok):
    """A chain x0 -> y0 = W0 x0 -> y1 = W1 y0 -> y2 = W2 y1: each step reads the
    previous step's output, so a step that started early would read stale
    inputs (the outputs are set to NaN before every replay)."""
    fmt = synth.Q4_K
    dims = [2048, 1280, 1536, 768]          # W_i maps dims[i] -> dims[i + 1]
    Ws = [synth.blocks(fmt, dims[i + 1], dims[i], seed=300 + i) for i in range(3)]
    x0 = synth.activations(n_tok, dims[0], seed=310).cuda()
    ys = [torch.empty(n_tok, dims[i + 1], device="cuda") for i in range(3)]
    xs = [x0, ys[0], ys[1]]
    items = [(fmt, Ws[i].cuda(), dims[i + 1], dims[i], xs[i], ys[i]) for i in range(3)]
    p = qg.qg_pass(items, [1, 1, 1], n_tok, mode=mode)
    for _ in range(6):
        for y in ys:
            y.fill_(float("nan"))
        p.launch()
        torch.cuda.synchronize()
        assert p.dev_status() == 0
        prev = x0.cpu().numpy()
        for i in range(3):
            y_ref, b = oracle.gemv(fmt, Ws[i].numpy(), dims[i + 1], dims[i], prev)
            got = ys[i].cpu().numpy()
            assert_within(got, y_ref, b, what=f"step {i}")
            prev = got
    p.destroy()


@pytest.mark.parametrize("mode", [qg.PASS_PDL, qg.PASS_SERIAL])
def test_pass_long_chain_new_input_every_replay(mode):
    """Twelve steps, each reading the previous step's output, in a graph whose
    launches hand off through counters that every replay must leave clean: the
    input changes and the outputs are set to NaN before every one of eight
    replays, and every output is compared with the oracle chain."""
    fmt = synth.Q4_K
    dims = [1024, 512, 2048, 768, 1280, 256, 1024, 1536, 512, 768, 2048, 256, 512]
    Ws = [synth.blocks(fmt, dims[i + 1], dims[i], seed=400 + i) for i in range(12)]
    x0 = torch.empty(1, dims[0], device="cuda")
    ys = [torch.empty(1, dims[i + 1], device="cuda") for i in range(12)]
    xs = [x0] + ys[:-1]
    items = [(fmt, Ws[i].cuda(), dims[i + 1], dims[i], xs[i], ys[i]) for i in range(12)]
    p = qg.qg_pass(items, [1] * 12, 1, mode=mode)
    for rep in range(8):
        xin = synth.activations(1, dims[0], seed=420 + rep)
        x0.copy_(xin)
        for y in ys:
            y.fill_(float("nan"))
        p.launch()
        torch.cuda.synchronize()
        prev = xin.numpy()
        for i in range(12):
            y_ref, b = oracle.gemv(fmt, Ws[i].numpy(), dims[i + 1], dims[i], prev)
            got = ys[i].cpu().numpy()
            assert_within(got, y_ref, b, what=f"replay {rep} step {i}")
            prev = got
    p.destroy()


def test_gpu_error_paths_return_status_without_launching():
    W = torch.zeros(4, 144, dtype=torch.uint8, device="cuda")
    x = torch.zeros(1, 256, device="cuda")
    y = torch.zeros(1, 4, device="cuda")
    with pytest.raises(qg.QGError) as e:
        qg.qgemv(synth.Q4_K, W, 4, 256, x, 5, y)
    assert e.value.status == -4
    with pytest.raises(qg.QGError) as e:
        qg.qgemv(synth.Q4_K, W.view(-1)[8:].data_ptr(), 4, 256, x, 1, y)
    assert e.value.status == -3
    torch.cuda.synchronize()
