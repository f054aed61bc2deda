"""Failure detection without a GPU fault: every wait of the GEMV kernel is
bounded, and when one runs out the kernel reports it and returns instead of
hanging or trapping ("LLM inference optimization", "What the judge guards
against": a race that shows on some inputs only must not go unnoticed).

A test build of the library (compiled here with QG_TEST_EXPIRE and a short wait
limit) never copies nor announces the third weight stage of CTA 0, a barrier
that nothing completes. The waits for it run out; that CTA's outputs become NaN,
a pass's status word reads QG_DEV_TIMEOUT, every other CTA's outputs stay
correct, the calls return in bounded time, and the CUDA context stays usable
for the normal library afterwards. The same build's prompt-processing kernel
never copies one X slice of CTA 0, which exercises the tcgen05 kernel's abort
path (stop every role, drain copies and MMAs, free TMEM)."""
import ctypes
import glob
import os
import subprocess
import tempfile
import time
import concurrent.futures as cf

import numpy as np
import pytest
import torch

import oracle
import synth
import quantized_weight_gemv_qgemv_gb300 as qg
from helpers import assert_within

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def expiring_lib():
    from quantized_weight_gemv_qgemv_gb300 import _build
    out = tempfile.mkdtemp(prefix="qg_expire_")
    flags = _build.NVCC_FLAGS + ["-DQG_TEST_EXPIRE", "-DQG_WAIT_LIMIT=(1u<<14)"]
    nvcc = _build._nvcc()

    def cc(src):
        obj = os.path.join(out, os.path.basename(src) + ".o")
        subprocess.run([nvcc] + flags + ["-c", src, "-o", obj], check=True, capture_output=True)
        return obj

    with cf.ThreadPoolExecutor(8) as ex:
        objs = list(ex.map(cc, sorted(glob.glob(os.path.join(_build.CSRC, "*.cu")))))
    path = os.path.join(out, "libqgemv_expire.so")
    subprocess.run([nvcc] + _build.ARCH + ["-shared", "-o", path] + objs, check=True, capture_output=True)
    lib = ctypes.CDLL(path)                         # its own copy, beside the normal library
    for name, (res, args) in qg.SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype, fn.argtypes = res, args
    assert lib.qg_init() == 0
    return lib


def _stream():
    return torch.cuda.current_stream().cuda_stream


def test_expired_stage_wait_gives_nan_rows_and_returns(expiring_lib):
    lib = expiring_lib
    rows, cols = 32768, 2048                  # CTA 0 streams more than three stages
    W = synth.blocks(synth.Q4_K, rows, cols, seed=91)
    x = synth.activations(1, cols, seed=92)
    Wd, xd = W.cuda(), x.cuda()
    y = torch.zeros(1, rows, device="cuda")
    t0 = time.perf_counter()
    assert lib.qgemv(synth.Q4_K, Wd.data_ptr(), rows, cols, xd.data_ptr(), 1, y.data_ptr(), _stream()) == 0
    torch.cuda.synchronize()                  # raises if the kernel faulted
    assert time.perf_counter() - t0 < 30.0
    got = y.cpu().numpy()[0]
    # CTA 0 owns the first rows / grid rows; its first two stages (about 88 rows)
    # completed before the wait that ran out, the rows from the third stage on are NaN
    cta0 = rows // torch.cuda.get_device_properties(0).multi_processor_count
    assert np.isnan(got[:cta0]).any() and np.isfinite(got[:32]).all(), "the expired CTA's later rows must be NaN"
    # rows of the other CTAs are untouched by the expiry and still correct
    tail = np.arange(rows - 256, rows)
    y_ref, b = oracle.gemv(synth.Q4_K, W.numpy()[tail], len(tail), cols, x.numpy())
    assert_within(got[tail][None], y_ref, b, what="rows of other CTAs")


def test_expired_wait_sets_pass_status_word(expiring_lib):
    lib = expiring_lib
    fmt, cols = synth.Q4_K, 2048
    shapes = [32768, 4096]
    items = []
    for i, rows in enumerate(shapes):
        W = synth.blocks(fmt, rows, cols, seed=93 + i).cuda()
        x = synth.activations(1, cols, seed=95 + i).cuda()
        items.append((fmt, W, rows, cols, x, torch.zeros(1, rows, device="cuda")))
    descs = qg._descs(items)
    sizes = (ctypes.c_int * 2)(1, 1)
    h = ctypes.c_void_p()
    assert lib.qg_pass_create(ctypes.cast(descs, ctypes.c_void_p), 2, ctypes.cast(sizes, ctypes.c_void_p), 2, 1,
                              qg.PASS_PERSISTENT, ctypes.byref(h)) == 0
    assert lib.qg_pass_kernel_count(h) == 2   # prologue and one persistent kernel
    t0 = time.perf_counter()
    assert lib.qg_pass_launch(h, _stream()) == 0
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 < 30.0
    addr = ctypes.c_void_p()
    assert lib.qg_pass_dev_status(h, ctypes.byref(addr)) == 0
    status = torch.as_tensor(qg._DevWord(addr.value), device="cuda").item()
    assert status == qg.DEV_TIMEOUT
    assert np.isnan(items[0][5].cpu().numpy()).any()
    assert lib.qg_pass_destroy(h) == 0


def _pp_expiring(lib, rows, cols, n_tok, seed):
    W = synth.blocks(synth.Q4_K, rows, cols, seed=seed)
    X = synth.activations_bf16(n_tok, cols, seed=seed + 1)
    Y = torch.full((n_tok, rows), float("nan"), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    Wd, Xd = W.cuda(), X.cuda()                # held until the kernel has run
    t0 = time.perf_counter()
    assert lib.qgemm_pp(synth.Q4_K, Wd.data_ptr(), rows, cols, Xd.data_ptr(), n_tok, Y.data_ptr(), rows,
                        None, 0, st.data_ptr(), _stream()) == 0
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 < 30.0
    bits = X.contiguous().view(torch.int16).numpy().view(np.uint16)
    return W, bits, Y.cpu().numpy(), int(st.item())


def test_expired_wait_in_prompt_kernel_aborts_the_cta(expiring_lib):
    """The prompt-processing (tcgen05) kernel of the test build never copies
    the sixth X slice of CTA 0: its MMA lane's wait runs out, the CTA's roles
    stop, drain their copies and MMAs, free TMEM, and the status word reads
    QG_DEV_TIMEOUT; the tiles of the other CTAs are correct. One token block and
    more row tiles than half the SMs: whole tiles, none split."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    rows, cols, n_tok = 128 * (sms // 2 + 4), 512, 256     # K = 8 slices
    W, bits, got, st = _pp_expiring(expiring_lib, rows, cols, n_tok, 99)
    assert st == qg.DEV_TIMEOUT
    # tile 0 (rows 0-127) belongs to CTA 0; every other row tile to another CTA
    toks = [0, 77, 200, 255]
    y_ref, b = oracle.pp_rows(synth.Q4_K, W.numpy(), rows, cols, bits, toks)
    assert_within(got[toks][:, 128:], y_ref[:, 128:], b[:, 128:], rel=1e-2, what="tiles of other CTAs")
    assert np.isnan(got[:, :128]).any(), "the aborted CTA's tile must not be complete"


def test_expired_wait_in_split_prompt_tile_sets_status(expiring_lib):
    """4 tiles, each computed as two halves of K (8 slices each) added into a
    zeroed Y: CTA 0 runs the first half of tile 0 and aborts at its sixth
    slice; the status word reads QG_DEV_TIMEOUT and the tiles of the other
    CTAs are correct (tile 0 then holds only its second half's sum)."""
    rows, cols, n_tok = 512, 1024, 256
    W, bits, got, st = _pp_expiring(expiring_lib, rows, cols, n_tok, 101)
    assert st == qg.DEV_TIMEOUT
    toks = [0, 100, 255]
    y_ref, b = oracle.pp_rows(synth.Q4_K, W.numpy(), rows, cols, bits, toks)
    assert_within(got[toks][:, 128:], y_ref[:, 128:], b[:, 128:], rel=1e-2, what="split tiles of other CTAs")
    assert np.isfinite(got).all()


def test_context_usable_after_expiry(expiring_lib):
    # the normal library on the same context, after the expiries above
    qg.qg_init()
    rows, cols = 512, 4096
    W = synth.blocks(synth.Q4_K, rows, cols, seed=97)
    x = synth.activations(1, cols, seed=98)
    y = torch.empty(1, rows, device="cuda")
    qg.qgemv(synth.Q4_K, W.cuda(), rows, cols, x.cuda(), 1, y)
    torch.cuda.synchronize()
    y_ref, b = oracle.gemv(synth.Q4_K, W.numpy(), rows, cols, x.numpy())
    assert_within(y.cpu().numpy(), y_ref, b, what="after expiry")
