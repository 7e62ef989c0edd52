"""GB300-native k-quant batch-1 decode GEMV (q6_K / q4_K x q8) and its q8
producers, behind the C ABI of include/mq.h (libmq.so, built in-tree).

This module is a thin binding: the functions carry the C entry points' names
and only marshal arguments (torch tensors -> pointers, the current CUDA
stream).  Every step of the path runs in the library's CUDA kernels; there is
no CPU or PyTorch fallback, and a missing library raises.

Typical decode use:
    Wp  = to_device(mq_repack_q6k(gguf_rows, rows, cols))   # once, at load
    ws  = mq_gemv_workspace(rows, cols)                      # once, zeroed
    y, q8 = mq_swiglu_quant_q8(g, u)                         # producer
    out = mq_gemv_q6k_q8(Wp, q8, rows, cols, ws=ws)          # GEMV
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_PKG, "_build", "libmq.so")
_lib = None

(MQ_OK, MQ_ERR_SHAPE, MQ_ERR_ALIGN, MQ_ERR_NULL, MQ_ERR_COVERAGE, MQ_ERR_WORKSPACE, MQ_ERR_CUDA,
 MQ_ERR_ACCESS) = range(8)

# every symbol include/mq.h declares
EXPORTS = [
    "mq_strerror", "mq_version", "mq_last_error", "mq_repacked_bytes_q6k", "mq_repacked_bytes_q4k",
    "mq_repack_q6k", "mq_repack_q4k", "mq_unrepack_q6k", "mq_unrepack_q4k", "mq_q8_bytes",
    "mq_q8_unpack_host", "mq_quantize_q8", "mq_rmsnorm_quant_q8", "mq_swiglu_quant_q8",
    "mq_gemv_workspace_bytes", "mq_gemv_plan", "mq_gemv_q6k_q8", "mq_gemv_q4k_q8",
    "mq_gemv_q6k_q8_plan", "mq_gemv_q4k_q8_plan", "mq_gemv_workspace_bytes_for",
    "mq_check_coverage", "mq_gemv_plan_for", "mq_set_pdl", "mq_gemv_q6k_q8_noalloc",
    "mq_gemv_group_workspace_bytes", "mq_gemv_group_q8", "mq_gemv_group_q8_plan",
    "mq_gemv_q6k_q8_subdots",
    "mq_gemv_q4k_q8_subdots", "mq_device_sms",
    "mq_quantize_q8_batch", "mq_rmsnorm_quant_q8_batch", "mq_swiglu_quant_q8_batch",
    "mq_gemv_batch_plan", "mq_gemv_batch_plan_for", "mq_gemv_q6k_q8_batch", "mq_gemv_q4k_q8_batch", "mq_gemv_q6k_q8_batch_plan",
    "mq_gemv_q4k_q8_batch_plan", "mq_gemv_gateup_swiglu_q8", "mq_gemv_gateup_swiglu_q8_plan",
    "mq_gemv_gateup_plan_for", "mq_repacked_bytes_q5k", "mq_repack_q5k", "mq_unrepack_q5k",
    "mq_gemv_q5k_q8", "mq_gemv_q5k_q8_plan", "mq_gemv_q5k_q8_subdots", "mq_gemv_q5k_q8_batch",
    "mq_gemv_q5k_q8_batch_plan", "mq_read_floor", "mq_gemv_q6k_f32", "mq_gemv_q6k_f32_plan",
    "mq_gemv_q6k_f32_plan_of", "mq_copy", "mq_repack_device", "mq_gemv_group_q8_coverage",
    "mq_device_address", "mq_set_gemv_ring",
]


class MQGemvPart(ctypes.Structure):
    """mq_gemv_part of include/mq.h."""
    _fields_ = [("fmt", ctypes.c_int), ("rows", ctypes.c_int), ("Wp", ctypes.c_void_p),
                ("y", ctypes.c_void_p)]


MQ_MAX_GROUP = 8
MQ_MAX_TOKENS = 8


class MQError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = f"{where}: {lib().mq_strerror(status).decode()} (status {status})"
        if status == MQ_ERR_CUDA:
            msg += f": {lib().mq_last_error().decode()}"
        super().__init__(msg)


def library_path() -> str:
    return _SO


def lib():
    """Load libmq.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_SO):
        raise RuntimeError(f"{_SO} is missing: build it with "
                           "`python -m quant_quantized_gemv_gb300.build` (or __graft_entry__.build())")
    L = ctypes.CDLL(_SO)
    P, I, S, F, LL = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_float, ctypes.c_longlong
    sig = {
        "mq_strerror": ([I], ctypes.c_char_p),
        "mq_version": ([], ctypes.c_char_p),
        "mq_last_error": ([], ctypes.c_char_p),
        "mq_repacked_bytes_q6k": ([I, I], S),
        "mq_repacked_bytes_q4k": ([I, I], S),
        "mq_repack_q6k": ([P, P, I, I], I),
        "mq_repack_q4k": ([P, P, I, I], I),
        "mq_unrepack_q6k": ([P, P, I, I], I),
        "mq_unrepack_q4k": ([P, P, I, I], I),
        "mq_q8_bytes": ([I], S),
        "mq_q8_unpack_host": ([P, I, P, P, P], I),
        "mq_quantize_q8": ([P, P, I, P], I),
        "mq_rmsnorm_quant_q8": ([P, P, F, P, P, I, P], I),
        "mq_swiglu_quant_q8": ([P, P, P, P, I, P], I),
        "mq_gemv_workspace_bytes": ([I, I], S),
        "mq_gemv_plan": ([I, I, I, P, P, P], I),
        "mq_gemv_q6k_q8": ([P, P, P, I, I, P, S, P], I),
        "mq_gemv_q4k_q8": ([P, P, P, I, I, P, S, P], I),
        "mq_gemv_q6k_q8_plan": ([P, P, P, I, I, I, I, I, P, S, P], I),
        "mq_gemv_q4k_q8_plan": ([P, P, P, I, I, I, I, I, P, S, P], I),
        "mq_gemv_workspace_bytes_for": ([I, I, I, I, I], S),
        "mq_check_coverage": ([I, I, I], I),
        "mq_gemv_plan_for": ([I, I, I, I, P, P, P], I),
        "mq_set_pdl": ([I], I),
        "mq_set_gemv_ring": ([I, I], I),
        "mq_gemv_q6k_q8_noalloc": ([P, P, P, I, I, P], I),
        "mq_gemv_group_workspace_bytes": ([P, I, I, I, I, I], S),
        "mq_gemv_group_q8": ([P, I, P, I, P, S, P], I),
        "mq_gemv_group_q8_plan": ([P, I, P, I, I, I, I, P, S, P], I),
        "mq_gemv_q6k_q8_subdots": ([P, P, P, I, I, P], I),
        "mq_gemv_q4k_q8_subdots": ([P, P, P, I, I, P], I),
        "mq_device_sms": ([], I),
        "mq_quantize_q8_batch": ([P, P, I, I, P], I),
        "mq_rmsnorm_quant_q8_batch": ([P, P, F, P, P, I, I, P], I),
        "mq_swiglu_quant_q8_batch": ([P, P, P, P, I, I, P], I),
        "mq_gemv_batch_plan": ([I, I, I, P, P, P], I),
        "mq_gemv_batch_plan_for": ([I, I, I, I, I, P, P, P], I),
        "mq_gemv_q6k_q8_batch": ([P, P, I, P, I, I, P], I),
        "mq_gemv_q4k_q8_batch": ([P, P, I, P, I, I, P], I),
        "mq_gemv_q6k_q8_batch_plan": ([P, P, I, P, I, I, I, I, I, P], I),
        "mq_gemv_q4k_q8_batch_plan": ([P, P, I, P, I, I, I, I, I, P], I),
        "mq_gemv_gateup_swiglu_q8": ([I, P, P, P, I, I, P, P, P], I),
        "mq_gemv_gateup_swiglu_q8_plan": ([I, P, P, P, I, I, P, P, I, I, P], I),
        "mq_gemv_gateup_plan_for": ([I, I, I, P, P], I),
        "mq_repacked_bytes_q5k": ([I, I], S),
        "mq_repack_q5k": ([P, P, I, I], I),
        "mq_unrepack_q5k": ([P, P, I, I], I),
        "mq_gemv_q5k_q8": ([P, P, P, I, I, P, S, P], I),
        "mq_gemv_q5k_q8_plan": ([P, P, P, I, I, I, I, I, P, S, P], I),
        "mq_gemv_q5k_q8_subdots": ([P, P, P, I, I, P], I),
        "mq_gemv_q5k_q8_batch": ([P, P, I, P, I, I, P], I),
        "mq_gemv_q5k_q8_batch_plan": ([P, P, I, P, I, I, I, I, I, P], I),
        "mq_read_floor": ([P, S, P], I),
        "mq_gemv_q6k_f32": ([P, P, P, I, I, P], I),
        "mq_gemv_q6k_f32_plan": ([P, P, P, I, I, I, I, I, P], I),
        "mq_gemv_q6k_f32_plan_of": ([I, I, P, P, P], I),
        "mq_copy": ([P, P, S, P], I),
        "mq_device_address": ([P, ctypes.POINTER(ctypes.c_void_p)], I),
        "mq_repack_device": ([I, P, P, I, I, P], I),
        "mq_gemv_group_q8_coverage": ([P, I, P, I, I, I, I, P, S, P, P], I),
    }
    for name, (args, res) in sig.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = res
    _lib = L
    return L


def _check(status: int, where: str):
    if status != MQ_OK:
        raise MQError(status, where)


# ------------------------------------------------------------------ helpers
def _np_ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _dev(t, dtype=None):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError("expected a CUDA tensor (the library has no CPU path)")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"expected {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return ctypes.c_void_p(t.data_ptr())


def _act(t, dtype=None):
    """An activation input or a GEMV output: a CUDA tensor, or a pinned CPU
    tensor that the kernels reach over the host link (its device address)."""
    import torch
    if isinstance(t, torch.Tensor) and not t.is_cuda:
        if not t.is_pinned():
            raise TypeError("a CPU tensor must be pinned (the kernels address it directly)")
        if dtype is not None and t.dtype != dtype:
            raise TypeError(f"expected {dtype}, got {t.dtype}")
        if not t.is_contiguous():
            raise ValueError("expected a contiguous tensor")
        return ctypes.c_void_p(mq_device_address(t.data_ptr()))
    return _dev(t, dtype)


def mq_device_address(ptr: int) -> int:
    """The device-side address of ptr (device or pinned host memory)."""
    out = ctypes.c_void_p(0)
    _check(lib().mq_device_address(ctypes.c_void_p(ptr), ctypes.byref(out)), "mq_device_address")
    return out.value or 0


def _stream(stream=None):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


# ------------------------------------------------------------------ repack (host)
def mq_repacked_bytes_q6k(rows: int, cols: int) -> int:
    return lib().mq_repacked_bytes_q6k(rows, cols)


def mq_repacked_bytes_q4k(rows: int, cols: int) -> int:
    return lib().mq_repacked_bytes_q4k(rows, cols)


def _repack(fn, size_fn, gguf: np.ndarray, rows: int, cols: int) -> np.ndarray:
    gguf = np.ascontiguousarray(gguf, dtype=np.uint8)
    out = np.empty(size_fn(rows, cols), np.uint8)
    _check(fn(_np_ptr(gguf), _np_ptr(out), rows, cols), fn.__name__)
    return out


def mq_repack_q6k(gguf: np.ndarray, rows: int, cols: int) -> np.ndarray:
    """GGUF q6_K rows (host) -> repacked bytes (host numpy)."""
    return _repack(lib().mq_repack_q6k, mq_repacked_bytes_q6k, gguf, rows, cols)


def mq_repack_q4k(gguf: np.ndarray, rows: int, cols: int) -> np.ndarray:
    return _repack(lib().mq_repack_q4k, mq_repacked_bytes_q4k, gguf, rows, cols)


def mq_unrepack_q6k(packed: np.ndarray, rows: int, cols: int) -> np.ndarray:
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    out = np.empty(rows * (cols // 256) * 210, np.uint8)
    _check(lib().mq_unrepack_q6k(_np_ptr(packed), _np_ptr(out), rows, cols), "mq_unrepack_q6k")
    return out.reshape(rows, -1)


def mq_unrepack_q4k(packed: np.ndarray, rows: int, cols: int) -> np.ndarray:
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    out = np.empty(rows * (cols // 256) * 144, np.uint8)
    _check(lib().mq_unrepack_q4k(_np_ptr(packed), _np_ptr(out), rows, cols), "mq_unrepack_q4k")
    return out.reshape(rows, -1)


def mq_repacked_bytes_q5k(rows: int, cols: int) -> int:
    return lib().mq_repacked_bytes_q5k(rows, cols)


def mq_repack_q5k(gguf: np.ndarray, rows: int, cols: int) -> np.ndarray:
    """GGUF q5_K rows (host) -> repacked bytes (host numpy)."""
    return _repack(lib().mq_repack_q5k, mq_repacked_bytes_q5k, gguf, rows, cols)


def mq_unrepack_q5k(packed: np.ndarray, rows: int, cols: int) -> np.ndarray:
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    out = np.empty(rows * (cols // 256) * 176, np.uint8)
    _check(lib().mq_unrepack_q5k(_np_ptr(packed), _np_ptr(out), rows, cols), "mq_unrepack_q5k")
    return out.reshape(rows, -1)


FMT_CODES = {"q6k": 6, "q4k": 4, "q5k": 5}


def fmt_code(fmt: str) -> int:
    """The C ABI's format code of 'q6k', 'q4k' or 'q5k'."""
    try:
        return FMT_CODES[fmt]
    except KeyError:
        raise ValueError(f"unknown format {fmt!r}") from None


def mq_repack(fmt: str, gguf: np.ndarray, rows: int, cols: int) -> np.ndarray:
    """GGUF rows of format fmt (host) -> repacked bytes (host numpy)."""
    return {"q6k": mq_repack_q6k, "q4k": mq_repack_q4k, "q5k": mq_repack_q5k}[fmt](gguf, rows, cols)


# ------------------------------------------------------------------ q8 plane
def mq_q8_bytes(n: int) -> int:
    return lib().mq_q8_bytes(n)


def mq_q8_unpack_host(plane: np.ndarray, n: int):
    """Host copy of a q8 plane -> (d fp16 bits [n/32], qs int8 [n], sum int32 [n/32])."""
    plane = np.ascontiguousarray(plane, dtype=np.uint8)
    d = np.empty(n // 32, np.uint16)
    qs = np.empty(n, np.int8)
    s = np.empty(n // 32, np.int32)
    _check(lib().mq_q8_unpack_host(_np_ptr(plane), n, _np_ptr(d), _np_ptr(qs), _np_ptr(s)),
           "mq_q8_unpack_host")
    return d, qs, s


def _gpu_of(like):
    """Where outputs go by default: like's device, or the current CUDA device
    when like is a (pinned) host input."""
    import torch
    if not isinstance(like, torch.Tensor) or not (like.is_cuda or like.is_pinned()):
        raise TypeError("expected a CUDA tensor or a pinned CPU tensor (the library has no CPU path)")
    return like.device if like.is_cuda else torch.device("cuda", torch.cuda.current_device())


def _q8_out(n: int, like, q8):
    import torch
    if q8 is None:
        q8 = torch.empty(mq_q8_bytes(n), dtype=torch.uint8, device=_gpu_of(like))
    return q8


# ------------------------------------------------------------------ producers
def mq_quantize_q8(x, q8=None, stream=None):
    import torch
    n = x.numel()
    q8 = _q8_out(n, x, q8)
    _check(lib().mq_quantize_q8(_act(x, torch.float32), _dev(q8), n, _stream(stream)),
           "mq_quantize_q8")
    return q8


def mq_rmsnorm_quant_q8(x, gain, eps: float, y=None, q8=None, stream=None):
    import torch
    n = x.numel()
    y = torch.empty(x.shape, dtype=x.dtype, device=_gpu_of(x)) if y is None else y
    q8 = _q8_out(n, x, q8)
    _check(lib().mq_rmsnorm_quant_q8(_act(x, torch.float32), _dev(gain, torch.float32), float(eps),
                                     _dev(y, torch.float32), _dev(q8), n, _stream(stream)),
           "mq_rmsnorm_quant_q8")
    return y, q8


def mq_swiglu_quant_q8(g, u, y=None, q8=None, stream=None):
    import torch
    n = g.numel()
    y = torch.empty(g.shape, dtype=g.dtype, device=_gpu_of(g)) if y is None else y
    q8 = _q8_out(n, g, q8)
    _check(lib().mq_swiglu_quant_q8(_act(g, torch.float32), _act(u, torch.float32),
                                    _dev(y, torch.float32), _dev(q8), n, _stream(stream)),
           "mq_swiglu_quant_q8")
    return y, q8


# ------------------------------------------------------------------ producers over nt rows
def _q8_out_rows(n: int, nt: int, like, q8):
    import torch
    if q8 is None:
        q8 = torch.empty(nt * mq_q8_bytes(n), dtype=torch.uint8, device=_gpu_of(like))
    return q8


def mq_quantize_q8_batch(x, q8=None, stream=None):
    """x: [nt, n] f32 -> nt q8 planes, back to back."""
    import torch
    nt, n = x.shape[0], x.shape[1]
    q8 = _q8_out_rows(n, nt, x, q8)
    _check(lib().mq_quantize_q8_batch(_act(x, torch.float32), _dev(q8), n, nt, _stream(stream)),
           "mq_quantize_q8_batch")
    return q8


def mq_rmsnorm_quant_q8_batch(x, gain, eps: float, y=None, q8=None, stream=None):
    """x: [nt, n] f32, gain: [n] -> y [nt, n] and nt q8 planes."""
    import torch
    nt, n = x.shape[0], x.shape[1]
    y = torch.empty(x.shape, dtype=x.dtype, device=_gpu_of(x)) if y is None else y
    q8 = _q8_out_rows(n, nt, x, q8)
    _check(lib().mq_rmsnorm_quant_q8_batch(_act(x, torch.float32), _dev(gain, torch.float32),
                                           float(eps), _dev(y, torch.float32), _dev(q8), n, nt,
                                           _stream(stream)),
           "mq_rmsnorm_quant_q8_batch")
    return y, q8


def mq_swiglu_quant_q8_batch(g, u, y=None, q8=None, stream=None):
    """g, u: [nt, n] f32 -> y [nt, n] and nt q8 planes."""
    import torch
    nt, n = g.shape[0], g.shape[1]
    y = torch.empty(g.shape, dtype=g.dtype, device=_gpu_of(g)) if y is None else y
    q8 = _q8_out_rows(n, nt, g, q8)
    _check(lib().mq_swiglu_quant_q8_batch(_act(g, torch.float32), _act(u, torch.float32),
                                          _dev(y, torch.float32), _dev(q8), n, nt, _stream(stream)),
           "mq_swiglu_quant_q8_batch")
    return y, q8


# ------------------------------------------------------------------ GEMV
def mq_gemv_workspace_bytes(rows: int, cols: int) -> int:
    return lib().mq_gemv_workspace_bytes(rows, cols)


def mq_gemv_workspace_bytes_for(rows: int, cols: int, plan) -> int:
    """Workspace bytes for an explicit plan (splits, chunks_per_split, tiles_per_item)."""
    return lib().mq_gemv_workspace_bytes_for(rows, cols, *map(int, plan))


def mq_check_coverage(nchunks: int, splits: int, chunks_per_split: int) -> int:
    return lib().mq_check_coverage(nchunks, splits, chunks_per_split)


def _plan_out(fn, *args):
    s, c, t = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    _check(fn(*args, ctypes.byref(s), ctypes.byref(c), ctypes.byref(t)), fn.__name__)
    return s.value, c.value, t.value


def mq_gemv_plan(rows: int, cols: int, fmt: str = "q6k"):
    """Default (splits, chunks_per_split, tiles_per_item) on the current device."""
    return _plan_out(lib().mq_gemv_plan, rows, cols, fmt_code(fmt))


def mq_gemv_plan_for(rows: int, cols: int, sms: int, regs_per_thread: int = 128):
    """Default plan for a device with `sms` SMs and a kernel of regs_per_thread registers."""
    return _plan_out(lib().mq_gemv_plan_for, rows, cols, sms, regs_per_thread)


def mq_set_pdl(enable: bool) -> bool:
    """Programmatic dependent launch for every later launch (process-wide)."""
    return bool(lib().mq_set_pdl(1 if enable else 0))


def mq_set_gemv_ring(stages: int = -1, pre_wait: int = -1) -> int:
    """Weight-ring depth of the single-token GEMV (process-wide; -1 = default).
    Returns the previous stages setting."""
    return int(lib().mq_set_gemv_ring(int(stages), int(pre_wait)))


def mq_read_floor(buf, nbytes: int = None, stream=None):
    """One plain read of nbytes (default: all) of a device tensor: the single-launch floor."""
    nb = buf.numel() * buf.element_size() if nbytes is None else int(nbytes)
    _check(lib().mq_read_floor(_dev(buf), nb, _stream(stream)), "mq_read_floor")


def mq_repack_device(fmt: str, gguf, rows: int, cols: int, out=None, stream=None):
    """Repack GGUF rows already on the device (a uint8 CUDA tensor) into a
    new (or the given) device buffer; the bytes equal mq_repack(fmt, ...)."""
    import torch
    code = fmt_code(fmt)
    nbytes = {6: mq_repacked_bytes_q6k, 4: mq_repacked_bytes_q4k, 5: mq_repacked_bytes_q5k}[code](rows, cols)
    if nbytes == 0:
        raise MQError(MQ_ERR_SHAPE, "mq_repack_device")
    if out is None:
        out = torch.empty(nbytes, dtype=torch.uint8, device=gguf.device)
    elif out.numel() * out.element_size() < nbytes:
        raise ValueError("output smaller than the repacked size")
    _check(lib().mq_repack_device(code, _dev(gguf), _dev(out), rows, cols, _stream(stream)),
           "mq_repack_device")
    return out


def mq_copy(dst, src, nbytes: int = None, stream=None):
    """Copy nbytes (default: all of src) from src to dst with a kernel; each
    may be a CUDA tensor or a pinned CPU tensor."""
    import torch
    for t in (dst, src):
        if not isinstance(t, torch.Tensor) or not t.is_contiguous():
            raise TypeError("expected contiguous tensors")
        if not t.is_cuda and not t.is_pinned():
            raise ValueError("a CPU tensor must be pinned (the GPU reads it directly)")
    nb = src.numel() * src.element_size() if nbytes is None else int(nbytes)
    if nb > dst.numel() * dst.element_size():
        raise ValueError("destination smaller than the copy")
    _check(lib().mq_copy(ctypes.c_void_p(dst.data_ptr()), ctypes.c_void_p(src.data_ptr()), nb,
                         _stream(stream)), "mq_copy")


def mq_device_sms() -> int:
    return lib().mq_device_sms()


def mq_gemv_workspace(rows: int, cols: int, plan=None, device=None):
    """A zero-filled workspace for (rows, cols) under the default plans, or
    under an explicit plan (splits, chunks_per_split, tiles_per_item); None
    when not needed."""
    import torch
    nbytes = (mq_gemv_workspace_bytes(rows, cols) if plan is None
              else mq_gemv_workspace_bytes_for(rows, cols, plan))
    if nbytes == 0:
        return None
    return torch.zeros(nbytes, dtype=torch.uint8, device=device or "cuda")


def _ws_args(ws):
    if ws is None:
        return ctypes.c_void_p(0), 0
    return _dev(ws), ws.numel() * ws.element_size()


def _gemv(name: str, Wp, q8, rows: int, cols: int, y, ws, stream, plan=None):
    import torch
    y = torch.empty(rows, dtype=torch.float32, device=Wp.device) if y is None else y
    wsp, wsb = _ws_args(ws)
    L = lib()
    if plan is None:
        st = getattr(L, name)(_dev(Wp), _dev(q8), _act(y, torch.float32), rows, cols, wsp, wsb,
                              _stream(stream))
    else:
        st = getattr(L, name + "_plan")(_dev(Wp), _dev(q8), _act(y, torch.float32), rows, cols,
                                        int(plan[0]), int(plan[1]), int(plan[2]), wsp, wsb,
                                        _stream(stream))
    _check(st, name)
    return y


def mq_gemv_q6k_q8(Wp, q8, rows: int, cols: int, y=None, ws=None, stream=None, plan=None):
    """y = W x_hat for repacked q6_K weights Wp (device) and a q8 plane."""
    return _gemv("mq_gemv_q6k_q8", Wp, q8, rows, cols, y, ws, stream, plan)


def mq_gemv_q4k_q8(Wp, q8, rows: int, cols: int, y=None, ws=None, stream=None, plan=None):
    """y = W x_hat for repacked q4_K weights Wp (device) and a q8 plane."""
    return _gemv("mq_gemv_q4k_q8", Wp, q8, rows, cols, y, ws, stream, plan)


def mq_gemv_q5k_q8(Wp, q8, rows: int, cols: int, y=None, ws=None, stream=None, plan=None):
    """y = W x_hat for repacked q5_K weights Wp (device) and a q8 plane."""
    return _gemv("mq_gemv_q5k_q8", Wp, q8, rows, cols, y, ws, stream, plan)


def mq_gemv(fmt: str, Wp, q8, rows: int, cols: int, y=None, ws=None, stream=None, plan=None):
    """The single-token GEMV of format fmt ('q6k', 'q4k', 'q5k')."""
    return _gemv("mq_gemv_" + {6: "q6k", 4: "q4k", 5: "q5k"}[fmt_code(fmt)] + "_q8", Wp, q8, rows,
                 cols, y, ws, stream, plan)


# ------------------------------------------------------------------ f32 activations
def mq_gemv_q6k_f32_plan_of(rows: int, cols: int):
    """Default plan of the f32-activation q6_K GEMV on the current device."""
    return _plan_out(lib().mq_gemv_q6k_f32_plan_of, rows, cols)


def mq_gemv_q6k_f32(Wp, x, rows: int, cols: int, y=None, stream=None, plan=None):
    """y = W x for repacked q6_K weights Wp and an f32 activation row x (device)."""
    import torch
    y = torch.empty(rows, dtype=torch.float32, device=Wp.device) if y is None else y
    L = lib()
    if plan is None:
        st = L.mq_gemv_q6k_f32(_dev(Wp), _dev(x, torch.float32), _act(y, torch.float32), rows, cols,
                               _stream(stream))
    else:
        st = L.mq_gemv_q6k_f32_plan(_dev(Wp), _dev(x, torch.float32), _act(y, torch.float32), rows,
                                    cols, int(plan[0]), int(plan[1]), int(plan[2]), _stream(stream))
    _check(st, "mq_gemv_q6k_f32")
    return y


# ------------------------------------------------------------------ small-batch GEMV
def mq_gemv_batch_plan(rows: int, cols: int, nt: int):
    """Default plan of the nt-token GEMV on the current device."""
    return _plan_out(lib().mq_gemv_batch_plan, rows, cols, nt)


def mq_gemv_batch_plan_for(rows: int, cols: int, nt: int, sms: int, regs_per_thread: int = 168):
    """Default nt-token plan for a device with `sms` SMs (host-only model)."""
    return _plan_out(lib().mq_gemv_batch_plan_for, rows, cols, nt, sms, regs_per_thread)


def _gemv_batch(name: str, Wp, q8, nt: int, rows: int, cols: int, y, stream, plan=None):
    import torch
    y = torch.empty((nt, rows), dtype=torch.float32, device=Wp.device) if y is None else y
    L = lib()
    if plan is None:
        st = getattr(L, name)(_dev(Wp), _dev(q8), nt, _act(y, torch.float32), rows, cols,
                              _stream(stream))
    else:
        st = getattr(L, name + "_plan")(_dev(Wp), _dev(q8), nt, _act(y, torch.float32), rows, cols,
                                        int(plan[0]), int(plan[1]), int(plan[2]), _stream(stream))
    _check(st, name)
    return y


def mq_gemv_q6k_q8_batch(Wp, q8, nt: int, rows: int, cols: int, y=None, stream=None, plan=None):
    """Y[nt, rows] = W x_hat_t for nt q8 planes (back to back), one pass over W."""
    return _gemv_batch("mq_gemv_q6k_q8_batch", Wp, q8, nt, rows, cols, y, stream, plan)


def mq_gemv_q4k_q8_batch(Wp, q8, nt: int, rows: int, cols: int, y=None, stream=None, plan=None):
    """Y[nt, rows] = W x_hat_t for nt q8 planes (back to back), one pass over W."""
    return _gemv_batch("mq_gemv_q4k_q8_batch", Wp, q8, nt, rows, cols, y, stream, plan)


def mq_gemv_q5k_q8_batch(Wp, q8, nt: int, rows: int, cols: int, y=None, stream=None, plan=None):
    """Y[nt, rows] = W x_hat_t for nt q8 planes (back to back), one pass over W."""
    return _gemv_batch("mq_gemv_q5k_q8_batch", Wp, q8, nt, rows, cols, y, stream, plan)


# ------------------------------------------------------------------ gate||up + SwiGLU -> q8
def mq_gemv_gateup_swiglu_q8(fmt: str, Wg, Wu, q8, rows: int, cols: int, act=None, q8_out=None,
                             stream=None, plan=None):
    """act = silu(Wg x_hat) * (Wu x_hat) and its q8 plane, in one launch.
    plan: None (default) or (warps_per_cta, ctas).  Returns (act, q8_out)."""
    import torch
    act = torch.empty(rows, dtype=torch.float32, device=Wg.device) if act is None else act
    q8_out = _q8_out(rows, act, q8_out)
    L = lib()
    f = fmt_code(fmt)
    if plan is None:
        st = L.mq_gemv_gateup_swiglu_q8(f, _dev(Wg), _dev(Wu), _dev(q8), rows, cols,
                                        _dev(act, torch.float32), _dev(q8_out), _stream(stream))
    else:
        st = L.mq_gemv_gateup_swiglu_q8_plan(f, _dev(Wg), _dev(Wu), _dev(q8), rows, cols,
                                             _dev(act, torch.float32), _dev(q8_out), int(plan[0]),
                                             int(plan[1]), _stream(stream))
    _check(st, "mq_gemv_gateup_swiglu_q8")
    return act, q8_out


def mq_gemv_gateup_plan_for(rows: int, sms: int, regs_per_thread: int = 168):
    """Default (warps_per_cta, ctas) of the gate||up kernel (host-only model)."""
    w, c = ctypes.c_int(), ctypes.c_int()
    _check(lib().mq_gemv_gateup_plan_for(rows, sms, regs_per_thread, ctypes.byref(w), ctypes.byref(c)),
           "mq_gemv_gateup_plan_for")
    return w.value, c.value


def _parts_array(parts, ys=None):
    """parts: [(fmt 'q6k'|'q4k', Wp tensor or None, rows)] -> ctypes array."""
    arr = (MQGemvPart * len(parts))()
    for i, (fmt, Wp, rows) in enumerate(parts):
        arr[i].fmt = fmt_code(fmt)
        arr[i].rows = int(rows)
        arr[i].Wp = None if Wp is None else Wp.data_ptr()
        arr[i].y = None if ys is None else _act(ys[i]).value   # device address (pinned host too)
    return arr


def mq_gemv_group_workspace_bytes(parts, cols: int, plan=None) -> int:
    """Workspace bytes of a group (default plan, or plan = (splits, cps, tpi))."""
    s, c, t = plan if plan is not None else (0, 0, 0)
    return lib().mq_gemv_group_workspace_bytes(_parts_array(parts), len(parts), cols, s, c, t)


def mq_gemv_group_workspace(parts, cols: int, plan=None, device=None):
    import torch
    nbytes = mq_gemv_group_workspace_bytes(parts, cols, plan)
    if nbytes == 0:
        return None
    return torch.zeros(nbytes, dtype=torch.uint8, device=device or "cuda")


def mq_gemv_group_q8(parts, q8, cols: int, ys=None, ws=None, stream=None, plan=None):
    """One launch for several matrices reading the same q8 plane.

    parts: [(fmt 'q6k'|'q4k', Wp device tensor, rows)]; returns the list of y."""
    import torch
    for _, Wp, _ in parts:
        _dev(Wp)
    if ys is None:
        ys = [torch.empty(rows, dtype=torch.float32, device=q8.device) for _, _, rows in parts]
    for y in ys:
        _act(y, torch.float32)
    arr = _parts_array(parts, ys)
    wsp, wsb = _ws_args(ws)
    if plan is None:
        st = lib().mq_gemv_group_q8(arr, len(parts), _dev(q8), cols, wsp, wsb, _stream(stream))
    else:
        st = lib().mq_gemv_group_q8_plan(arr, len(parts), _dev(q8), cols, int(plan[0]), int(plan[1]),
                                         int(plan[2]), wsp, wsb, _stream(stream))
    _check(st, "mq_gemv_group_q8")
    return ys


def mq_gemv_group_q8_coverage(parts, q8, cols: int, ys=None, ws=None, stream=None, plan=None):
    """The grouped GEMV that also counts, per (global tile, chunk) unit, how
    often a warp processed it.  Returns (ys, counts) with counts a CUDA int32
    tensor [total tiles, nchunks]; every count is 1 when the plan covers the
    work exactly once."""
    import torch
    for _, Wp, _ in parts:
        _dev(Wp)
    if ys is None:
        ys = [torch.empty(rows, dtype=torch.float32, device=q8.device) for _, _, rows in parts]
    for y in ys:
        _act(y, torch.float32)
    tiles = sum(-(-rows // 8) for _, _, rows in parts)
    nch = -(-(cols // 256) // 4)
    counts = torch.zeros((tiles, nch), dtype=torch.int32, device=q8.device)
    arr = _parts_array(parts, ys)
    wsp, wsb = _ws_args(ws)
    s, c, t = (0, 0, 0) if plan is None else (int(plan[0]), int(plan[1]), int(plan[2]))
    _check(lib().mq_gemv_group_q8_coverage(arr, len(parts), _dev(q8), cols, s, c, t, wsp, wsb,
                                           _dev(counts), _stream(stream)), "mq_gemv_group_q8_coverage")
    return ys, counts


def mq_gemv_q6k_q8_noalloc(Wp, q8, rows: int, cols: int, y=None, stream=None):
    """The q6_K GEMV without a caller workspace: for callers that may not
    allocate device memory (the library keeps the split-K scratch in a
    static device array).  The first call on a device must precede any CUDA
    graph capture; calls that overlap on the GPU race on the shared array."""
    import torch
    if y is None:
        y = torch.empty(rows, dtype=torch.float32, device=Wp.device)
    _check(lib().mq_gemv_q6k_q8_noalloc(_dev(Wp), _dev(q8), _act(y, torch.float32), rows, cols,
                                        _stream(stream)), "mq_gemv_q6k_q8_noalloc")
    return y


def _subdots(name: str, per: int, Wp, q8, rows: int, cols: int, stream):
    import torch
    out = torch.empty(rows * (cols // 256) * per, dtype=torch.int32, device=Wp.device)
    _check(getattr(lib(), name)(_dev(Wp), _dev(q8), _dev(out), rows, cols, _stream(stream)), name)
    return out.view(rows, cols // 256, per)


def mq_gemv_q6k_q8_subdots(Wp, q8, rows: int, cols: int, stream=None):
    """Integer sub-block dots rows x nb x 16 (int32) through the GEMV's lane mapping."""
    return _subdots("mq_gemv_q6k_q8_subdots", 16, Wp, q8, rows, cols, stream)


def mq_gemv_q4k_q8_subdots(Wp, q8, rows: int, cols: int, stream=None):
    return _subdots("mq_gemv_q4k_q8_subdots", 8, Wp, q8, rows, cols, stream)


def mq_gemv_q5k_q8_subdots(Wp, q8, rows: int, cols: int, stream=None):
    return _subdots("mq_gemv_q5k_q8_subdots", 8, Wp, q8, rows, cols, stream)
