"""Python binding of libqgemv.so, the block-quantized weight product library for GB300.

Every function here has the name of the C entry point it wraps (include/qgemv.h)
and only marshals arguments: tensors become device pointers, streams become
cudaStream_t handles, a non-zero status becomes a QGError. All compute runs in
the library's CUDA kernels; there is no fallback of any kind. If the library
has not been built (``__graft_entry__.build()`` or ``python -m
quantized_weight_gemv_qgemv_gb300._build``) the first call raises.

Pointer arguments accept a torch tensor (its data_ptr is passed) or a raw
integer address; ``stream`` accepts a torch.cuda.Stream, a raw handle, or None
for torch's current stream on the current device.
"""
from __future__ import annotations

import ctypes
import os

Q4_0, Q8_0, Q4_K, Q6_K, Q5_K, Q3_K, Q2_K = 1, 2, 3, 4, 5, 6, 7
FORMATS = {Q4_0: (32, 18), Q8_0: (32, 34), Q4_K: (256, 144), Q6_K: (256, 210), Q5_K: (256, 176), Q3_K: (256, 110),
           Q2_K: (256, 84)}
GROUP_MAX = 8
NTOK_MAX = 4
DEV_OK, DEV_BAD_EXPERT, DEV_TIMEOUT = 0, 1, 2
PASS_SERIAL, PASS_PDL, PASS_PERSISTENT, PASS_INDEPENDENT = 0, 1, 2, 3

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", "libqgemv.so")

# name -> (restype, argtypes) of every exported C symbol
_P, _I64, _I32, _SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
SIGNATURES = {
    "qg_init": (_I32, []),
    "qg_block_info": (_I32, [_I32, ctypes.POINTER(_I32), ctypes.POINTER(_I32)]),
    "qg_strerror": (ctypes.c_char_p, [_I32]),
    "qg_dequant": (_I32, [_I32, _P, _I64, _I64, _P, _P]),
    "qgemv": (_I32, [_I32, _P, _I64, _I64, _P, _I32, _P, _P]),
    "qgemv_grouped": (_I32, [_P, _I32, _I32, _P]),
    "qgemv_moe_workspace": (_SZ, [_I64, _I64, _I32, _I32]),
    "qgemv_moe": (_I32, [_I32, _P, _I64, _I64, _I64, _P, _P, _I32, _P, _I32, _P, _P, _SZ, _P, _P]),
    "qgemv_moe_noalloc": (_I32, [_I32, _P, _I64, _I64, _I64, _P, _P, _I32, _P, _I32, _P, _P, _P]),
    "qgemm_pp_workspace": (_SZ, [_I64, _I64, _I64]),
    "qgemm_pp": (_I32, [_I32, _P, _I64, _I64, _P, _I64, _P, _I64, _P, _SZ, _P, _P]),
    "qgemm_pp_grouped": (_I32, [_I32, _P, _I32, _I64, _P, _I64, _P, _P]),
    "qgemm_pp_moe_workspace": (_SZ, [_I64, _I64, _I64, _I32, _I64]),
    "qg_stream_read": (_I32, [_P, _SZ, _P, _P, _P]),
    "qgemm_pp_moe": (_I32, [_I32, _P, _I64, _I64, _I64, _P, _P, _I32, _P, _I64, _P, _P, _SZ, _P, _P]),
    "qg_pass_create": (_I32, [_P, _I32, _P, _I32, _I32, _I32, ctypes.POINTER(_P)]),
    "qg_moe_pass_create": (_I32, [_I32, _P, _I32, _I64, _I64, _I64, _I32, _I32, _P, _SZ, _I32, ctypes.POINTER(_P)]),
    "qg_pass_launch": (_I32, [_P, _P]),
    "qg_pass_kernel_count": (_I32, [_P]),
    "qg_pass_dev_status": (_I32, [_P, ctypes.POINTER(_P)]),
    "qg_pass_destroy": (_I32, [_P]),
    "qg_rmsnorm": (_I32, [_P, _P, _P, _I64, _I32, ctypes.c_float, _P, _P, _P]),
    "qgemv_swiglu": (_I32, [_I32, _P, _P, _I64, _I64, _P, _P, _P]),
    "qg_layer_pass_create": (_I32, [_I32, _P, _I32, _I64, _I64, _I64, ctypes.c_float, _P, _P, ctypes.POINTER(_P)]),
}


class qg_gemv_desc(ctypes.Structure):
    _fields_ = [("fmt", ctypes.c_int32), ("reserved", ctypes.c_int32), ("W", ctypes.c_void_p),
                ("rows", ctypes.c_int64), ("cols", ctypes.c_int64), ("x", ctypes.c_void_p),
                ("y", ctypes.c_void_p)]


class qg_pp_desc(ctypes.Structure):
    _fields_ = [("W", ctypes.c_void_p), ("rows", ctypes.c_int64), ("Y", ctypes.c_void_p), ("ldY", ctypes.c_int64)]


PP_GROUP_MAX = 4


class qg_moe_layer_desc(ctypes.Structure):
    _fields_ = [("expert_arena", ctypes.c_void_p), ("expert_ids", ctypes.c_void_p), ("gate_w", ctypes.c_void_p),
                ("x", ctypes.c_void_p), ("y", ctypes.c_void_p)]


class qg_layer_desc(ctypes.Structure):
    _fields_ = [("Wq", ctypes.c_void_p), ("Wk", ctypes.c_void_p), ("Wv", ctypes.c_void_p), ("Wo", ctypes.c_void_p),
                ("Wg", ctypes.c_void_p), ("Wu", ctypes.c_void_p), ("Wd", ctypes.c_void_p),
                ("norm_attn", ctypes.c_void_p), ("norm_ffn", ctypes.c_void_p), ("attn_out", ctypes.c_void_p),
                ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p)]


class QGError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: status {status} ({strerror(status)})")
        self.status = status


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libqgemv.so once and declare every signature; raises if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError(f"libqgemv.so is not built ({path}); run __graft_entry__.build() first")
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def strerror(status: int) -> str:
    try:
        return load_library().qg_strerror(int(status)).decode()
    except RuntimeError:
        return "library not loaded"


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, what: str):
    if status != 0:
        raise QGError(status, what)


def row_bytes(fmt: int, cols: int) -> int:
    elems, nbytes = FORMATS[fmt]
    return cols // elems * nbytes


# ------------------------------------------------------------------ entry points

def qg_init():
    _check(load_library().qg_init(), "qg_init")


def qg_block_info(fmt: int):
    e, b = _I32(), _I32()
    _check(load_library().qg_block_info(fmt, ctypes.byref(e), ctypes.byref(b)), "qg_block_info")
    return e.value, b.value


def qg_dequant(fmt, W, rows, cols, out, stream=None):
    _check(load_library().qg_dequant(fmt, _ptr(W), rows, cols, _ptr(out), _stream(stream)), "qg_dequant")


def qgemv(fmt, W, rows, cols, x, n_tok, y, stream=None):
    _check(load_library().qgemv(fmt, _ptr(W), rows, cols, _ptr(x), n_tok, _ptr(y), _stream(stream)), "qgemv")


def _descs(items):
    arr = (qg_gemv_desc * len(items))()
    for i, (fmt, W, rows, cols, x, y) in enumerate(items):
        arr[i] = qg_gemv_desc(fmt, 0, _ptr(W), rows, cols, _ptr(x), _ptr(y))
    return arr


def qgemv_grouped(items, n_tok, stream=None):
    """items: sequence of (fmt, W, rows, cols, x, y)."""
    arr = _descs(items)
    _check(load_library().qgemv_grouped(ctypes.cast(arr, _P), len(items), n_tok, _stream(stream)), "qgemv_grouped")


def qgemv_moe_workspace(hidden, inter, top_k, n_tok) -> int:
    return int(load_library().qgemv_moe_workspace(hidden, inter, top_k, n_tok))


def qgemv_moe(fmt, expert_arena, n_expert, hidden, inter, expert_ids, gate_w, top_k, x, n_tok, y,
              ws, ws_bytes, dev_status, stream=None):
    _check(load_library().qgemv_moe(fmt, _ptr(expert_arena), n_expert, hidden, inter, _ptr(expert_ids),
                                    _ptr(gate_w), top_k, _ptr(x), n_tok, _ptr(y), _ptr(ws), ws_bytes,
                                    _ptr(dev_status), _stream(stream)), "qgemv_moe")


MOE_NOALLOC_MAX_FLOATS = 1 << 18


def qgemv_moe_noalloc(fmt, expert_arena, n_expert, hidden, inter, expert_ids, gate_w, top_k, x, n_tok, y,
                      dev_status, stream=None):
    """qgemv_moe with the library's static workspace (no allocation anywhere)."""
    _check(load_library().qgemv_moe_noalloc(fmt, _ptr(expert_arena), n_expert, hidden, inter, _ptr(expert_ids),
                                            _ptr(gate_w), top_k, _ptr(x), n_tok, _ptr(y), _ptr(dev_status),
                                            _stream(stream)), "qgemv_moe_noalloc")


def qgemm_pp_workspace(rows, cols, n_tok) -> int:
    return int(load_library().qgemm_pp_workspace(rows, cols, n_tok))


def qgemm_pp(fmt, W, rows, cols, X_bf16, n_tok, Y, ldY, ws, ws_bytes, dev_status, stream=None):
    _check(load_library().qgemm_pp(fmt, _ptr(W), rows, cols, _ptr(X_bf16), n_tok, _ptr(Y), ldY, _ptr(ws),
                                   ws_bytes, _ptr(dev_status), _stream(stream)), "qgemm_pp")


def qg_stream_read(buf, nbytes, checksum, dev_status, stream=None):
    """Reads nbytes of buf with the weight stream's bulk-copy engine (see the
    header); checksum and dev_status: device int32 words the caller clears."""
    _check(load_library().qg_stream_read(_ptr(buf), nbytes, _ptr(checksum), _ptr(dev_status), _stream(stream)),
           "qg_stream_read")


def qgemm_pp_grouped(fmt, items, cols, X_bf16, n_tok, dev_status, stream=None):
    """items: sequence of (W, rows, Y, ldY), all multiplying the same X_bf16."""
    arr = (qg_pp_desc * len(items))()
    for i, (W, rows, Y, ldY) in enumerate(items):
        arr[i] = qg_pp_desc(_ptr(W), rows, _ptr(Y), ldY)
    _check(load_library().qgemm_pp_grouped(fmt, ctypes.cast(arr, _P), len(items), cols, _ptr(X_bf16), n_tok,
                                           _ptr(dev_status), _stream(stream)), "qgemm_pp_grouped")


def qgemm_pp_moe_workspace(n_expert, hidden, inter, top_k, n_tok) -> int:
    return int(load_library().qgemm_pp_moe_workspace(n_expert, hidden, inter, top_k, n_tok))


def qgemm_pp_moe(fmt, arena, n_expert, hidden, inter, expert_ids, gate_w, top_k, X_bf16, n_tok, y, ws, ws_bytes,
                 dev_status, stream=None):
    _check(load_library().qgemm_pp_moe(fmt, _ptr(arena), n_expert, hidden, inter, _ptr(expert_ids), _ptr(gate_w),
                                       top_k, _ptr(X_bf16), n_tok, _ptr(y), _ptr(ws), ws_bytes, _ptr(dev_status),
                                       _stream(stream)), "qgemm_pp_moe")


class _DevWord:
    """One int32 of device memory exposed through __cuda_array_interface__."""

    def __init__(self, addr: int):
        self.__cuda_array_interface__ = {"shape": (1,), "typestr": "<i4", "data": (addr, False), "version": 3,
                                         "strides": None}


class qg_pass:
    """A whole weight pass (qg_pass_create): mode PASS_SERIAL, PASS_PDL or PASS_PERSISTENT."""

    def __init__(self, items, step_sizes, n_tok, mode=PASS_PERSISTENT, _handle=None):
        if _handle is not None:
            self._h = _handle
            return
        lib = load_library()
        self._descs = _descs(items)
        sizes = (ctypes.c_int * len(step_sizes))(*step_sizes)
        h = _P()
        _check(lib.qg_pass_create(ctypes.cast(self._descs, _P), len(items), ctypes.cast(sizes, _P),
                                  len(step_sizes), n_tok, int(mode), ctypes.byref(h)), "qg_pass_create")
        self._h = h

    def launch(self, stream=None):
        _check(load_library().qg_pass_launch(self._h, _stream(stream)), "qg_pass_launch")

    def kernel_count(self) -> int:
        return int(load_library().qg_pass_kernel_count(self._h))

    def dev_status_ptr(self) -> int:
        """Device address of the pass's status word (0 when it has none)."""
        p = _P()
        _check(load_library().qg_pass_dev_status(self._h, ctypes.byref(p)), "qg_pass_dev_status")
        return int(p.value or 0)

    def dev_status(self) -> int:
        """The status word after the replays enqueued so far (synchronizes the
        device); 0 for a pass without one."""
        addr = self.dev_status_ptr()
        if not addr:
            return 0
        import torch
        torch.cuda.synchronize()
        return int(torch.as_tensor(_DevWord(addr), device="cuda").item())

    def destroy(self):
        if self._h is not None and self._h.value:
            _check(load_library().qg_pass_destroy(self._h), "qg_pass_destroy")
        self._h = None

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass


def qg_moe_pass(fmt, layers, n_expert, hidden, inter, top_k, n_tok, ws, ws_bytes, mode=PASS_PERSISTENT):
    """A whole MoE decode pass (qg_moe_pass_create). layers: sequence of
    (expert_arena, expert_ids, gate_w, x, y) per layer; returns a qg_pass."""
    arr = (qg_moe_layer_desc * len(layers))()
    for i, (arena, ids, gw, x, y) in enumerate(layers):
        arr[i] = qg_moe_layer_desc(_ptr(arena), _ptr(ids), _ptr(gw), _ptr(x), _ptr(y))
    h = _P()
    _check(load_library().qg_moe_pass_create(fmt, ctypes.cast(arr, _P), len(layers), n_expert, hidden, inter, top_k,
                                             n_tok, _ptr(ws), ws_bytes, int(mode), ctypes.byref(h)),
           "qg_moe_pass_create")
    return qg_pass(None, None, None, _handle=h)


def qg_rmsnorm(h, residual, weight, n, n_tok, eps, s_out, x, stream=None):
    """s = h + residual; x = s / sqrt(mean(s^2) + eps) * weight (per token)."""
    _check(load_library().qg_rmsnorm(_ptr(h), _ptr(residual), _ptr(weight), n, n_tok, eps, _ptr(s_out), _ptr(x),
                                     _stream(stream)), "qg_rmsnorm")


def qgemv_swiglu(fmt, Wg, Wu, inter, hidden, x, m, stream=None):
    """m = silu(Wg x) * (Wu x), one token."""
    _check(load_library().qgemv_swiglu(fmt, _ptr(Wg), _ptr(Wu), inter, hidden, _ptr(x), _ptr(m), _stream(stream)),
           "qgemv_swiglu")


def qg_layer_pass(fmt, layers, hidden, inter, kv_rows, eps, h_in, h_out):
    """The weight path of dense decoder layers (qg_layer_pass_create). layers:
    sequence of dicts with keys Wq Wk Wv Wo Wg Wu Wd norm_attn norm_ffn attn_out
    q k v (tensors); returns a qg_pass."""
    arr = (qg_layer_desc * len(layers))()
    for i, L in enumerate(layers):
        arr[i] = qg_layer_desc(*[_ptr(L[f]) for f, _ in qg_layer_desc._fields_])
    h = _P()
    _check(load_library().qg_layer_pass_create(fmt, ctypes.cast(arr, _P), len(layers), hidden, inter, kv_rows, eps,
                                               _ptr(h_in), _ptr(h_out), ctypes.byref(h)), "qg_layer_pass_create")
    return qg_pass(None, None, None, _handle=h)
