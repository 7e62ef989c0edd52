"""The oracle: ctypes wrapper around the plain C reference in ``mq_oracle.c``.

TEST INFRASTRUCTURE ONLY.  The tests, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` import this package; the library
(``quant_quantized_gemv_gb300``) never does, and this package imports nothing
from the library.  Inputs are numpy arrays in the GGUF block order; the oracle
knows nothing of the library's repacked layout.

Every function states the page and section of the minfer log it follows; the
C source carries the full statement of each formula.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mq_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "libmq_oracle.so")
_lock = threading.Lock()
_lib = None

Q6K_BYTES = 210
Q4K_BYTES = 144
Q5K_BYTES = 176
QK = 256


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (no fast-math, no FMA contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
                               "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _bind(L):
    P = ctypes.c_void_p
    I = ctypes.c_int
    L.mqo_f16_to_f32.argtypes = [ctypes.c_uint16]
    L.mqo_f16_to_f32.restype = ctypes.c_float
    L.mqo_f32_to_f16.argtypes = [ctypes.c_float]
    L.mqo_f32_to_f16.restype = ctypes.c_uint16
    L.mqo_quantize_q8.argtypes = [P, I, P, P, P]
    L.mqo_dequant_q6k.argtypes = [P, ctypes.c_long, P]
    L.mqo_dequant_q4k.argtypes = [P, ctypes.c_long, P]
    L.mqo_dequant_q5k.argtypes = [P, ctypes.c_long, P]
    L.mqo_q4k_scale_min.argtypes = [P, I, P, P]
    L.mqo_subdots_q6k.argtypes = [P, P, I, I, P]
    L.mqo_subdots_q4k.argtypes = [P, P, I, I, P]
    L.mqo_subdots_q5k.argtypes = [P, P, I, I, P]
    L.mqo_gemv_q6k.argtypes = [P, P, P, I, I, I, P, P]
    L.mqo_gemv_q4k.argtypes = [P, P, P, I, I, I, P, P]
    L.mqo_gemv_q5k.argtypes = [P, P, P, I, I, I, P, P]
    L.mqo_gemv_q6k_f32.argtypes = [P, P, I, I, I, P, P]
    L.mqo_rmsnorm.argtypes = [P, P, ctypes.c_float, I, P]
    L.mqo_swiglu.argtypes = [P, P, I, P]
    for f in ("mqo_quantize_q8", "mqo_dequant_q6k", "mqo_dequant_q4k", "mqo_dequant_q5k",
              "mqo_q4k_scale_min", "mqo_subdots_q6k", "mqo_subdots_q4k", "mqo_subdots_q5k",
              "mqo_gemv_q6k", "mqo_gemv_q4k", "mqo_gemv_q5k", "mqo_gemv_q6k_f32", "mqo_rmsnorm",
              "mqo_swiglu"):
        getattr(L, f).restype = None
    return L


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = _bind(ctypes.CDLL(_SO))
    return _lib


@contextlib.contextmanager
def variant(source: str, workdir: str):
    """Temporarily run every oracle function from another C source text (used
    by the mutation tests to show that the pins catch planted mistakes)."""
    global _lib
    src = os.path.join(workdir, "variant.c")
    so = os.path.join(workdir, "libvariant.so")
    with open(src, "w") as f:
        f.write(source)
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
                           "-fPIC", "-shared", "-o", so, src, "-lm"])
    saved = lib()
    with _lock:
        _lib = _bind(ctypes.CDLL(so))
    try:
        yield
    finally:
        with _lock:
            _lib = saved


def source() -> str:
    with open(_SRC) as f:
        return f.read()


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def f16_to_f32(h: int) -> float:
    """IEEE binary16 -> binary32 (exact)."""
    return float(lib().mqo_f16_to_f32(int(h)))


def f32_to_f16(x: float) -> int:
    """binary32 -> binary16, round to nearest even (as __float2half, D3-5 §3.2)."""
    return int(lib().mqo_f32_to_f16(float(np.float32(x))))


def quantize_q8(x: np.ndarray):
    """q8 quantizer of the D3-5 page, §3.2 (per 32-value block, f32 arithmetic).

    Returns (d: uint16 fp16 bits [n/32], q: int8 [n], sum: int32 [n/32]).
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    n = x.size
    assert n % 32 == 0
    d = np.zeros(n // 32, np.uint16)
    q = np.zeros(n, np.int8)
    s = np.zeros(n // 32, np.int32)
    lib().mqo_quantize_q8(_p(x), n, _p(d), _p(q), _p(s))
    return d, q, s


def dequant_q6k(blocks: np.ndarray) -> np.ndarray:
    """q6_K blocks (GGUF order, 210 B each) -> fp64 weights (D4-4 §1-§3.2)."""
    blocks = np.ascontiguousarray(blocks, dtype=np.uint8).reshape(-1)
    nblk = blocks.size // Q6K_BYTES
    w = np.zeros(nblk * QK, np.float64)
    lib().mqo_dequant_q6k(_p(blocks), nblk, _p(w))
    return w


def dequant_q4k(blocks: np.ndarray) -> np.ndarray:
    """q4_K blocks (GGUF order, 144 B each) -> fp64 weights."""
    blocks = np.ascontiguousarray(blocks, dtype=np.uint8).reshape(-1)
    nblk = blocks.size // Q4K_BYTES
    w = np.zeros(nblk * QK, np.float64)
    lib().mqo_dequant_q4k(_p(blocks), nblk, _p(w))
    return w


def dequant_q5k(blocks: np.ndarray) -> np.ndarray:
    """q5_K blocks (GGUF order, 176 B each) -> fp64 weights."""
    blocks = np.ascontiguousarray(blocks, dtype=np.uint8).reshape(-1)
    nblk = blocks.size // Q5K_BYTES
    w = np.zeros(nblk * QK, np.float64)
    lib().mqo_dequant_q5k(_p(blocks), nblk, _p(w))
    return w


def q4k_scale_min(block: np.ndarray, k: int):
    block = np.ascontiguousarray(block, dtype=np.uint8).reshape(-1)
    sc = ctypes.c_int()
    m = ctypes.c_int()
    lib().mqo_q4k_scale_min(_p(block), int(k), ctypes.byref(sc), ctypes.byref(m))
    return sc.value, m.value


def subdots(fmt: str, W: np.ndarray, q8: np.ndarray, rows: int, cols: int) -> np.ndarray:
    """Integer sub-block dots: q6_K rows x nb x 16, q4_K / q5_K rows x nb x 8 (int32)."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    q8 = np.ascontiguousarray(q8, dtype=np.int8)
    nb = cols // QK
    per = 16 if fmt == "q6k" else 8
    out = np.zeros((rows, nb, per), np.int32)
    getattr(lib(), "mqo_subdots_" + _fmt(fmt))(_p(W), _p(q8), rows, cols, _p(out))
    return out


def _fmt(fmt: str) -> str:
    if fmt not in ("q6k", "q4k", "q5k"):
        raise ValueError(f"unknown format {fmt!r}")
    return fmt


def gemv(fmt: str, W: np.ndarray, d8: np.ndarray, q8: np.ndarray, rows: int, cols: int,
         row_range=None, threads: int = 1):
    """y = W x_hat in fp64 (D4-2 §3.2 Excerpt C accumulation, integer dots).

    W is GGUF-ordered (rows x cols/256 blocks).  Returns (y, absum), both fp64
    arrays over the requested row range; absum is sum |term| per row.  With
    threads > 1 the row range is split over host threads (ctypes releases the
    GIL), each running the same single-threaded C function on its rows.
    """
    W = np.ascontiguousarray(W, dtype=np.uint8)
    d8 = np.ascontiguousarray(d8, dtype=np.uint16)
    q8 = np.ascontiguousarray(q8, dtype=np.int8)
    r0, r1 = (0, rows) if row_range is None else row_range
    y = np.zeros(rows, np.float64)
    a = np.zeros(rows, np.float64)
    fn = getattr(lib(), "mqo_gemv_" + _fmt(fmt))
    if threads <= 1 or r1 - r0 < 2 * threads:
        fn(_p(W), _p(d8), _p(q8), r0, r1, cols, _p(y), _p(a))
    else:
        edges = np.linspace(r0, r1, threads + 1).astype(int)
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(lambda i: fn(_p(W), _p(d8), _p(q8), int(edges[i]), int(edges[i + 1]),
                                     cols, _p(y), _p(a)), range(threads)))
    return y[r0:r1], a[r0:r1]


def gemv_q6k_f32(W: np.ndarray, x: np.ndarray, rows: int, cols: int, row_range=None,
                 threads: int = 1):
    """y = W x for q6_K weights and an f32 activation row, in fp64 (the
    dequantize-and-FMA "padded f32" family of the D3 page, §2.3 and §3.3).

    Returns (y, absum) over the requested row range, as gemv() does.
    """
    W = np.ascontiguousarray(W, dtype=np.uint8)
    x = np.ascontiguousarray(x, dtype=np.float32)
    assert x.size == cols
    r0, r1 = (0, rows) if row_range is None else row_range
    y = np.zeros(rows, np.float64)
    a = np.zeros(rows, np.float64)
    fn = lib().mqo_gemv_q6k_f32
    if threads <= 1 or r1 - r0 < 2 * threads:
        fn(_p(W), _p(x), r0, r1, cols, _p(y), _p(a))
    else:
        edges = np.linspace(r0, r1, threads + 1).astype(int)
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(lambda i: fn(_p(W), _p(x), int(edges[i]), int(edges[i + 1]), cols,
                                     _p(y), _p(a)), range(threads)))
    return y[r0:r1], a[r0:r1]


def rmsnorm(x: np.ndarray, gain: np.ndarray, eps: float) -> np.ndarray:
    """y = x / sqrt(mean(x^2) + eps) * gain in fp64 (the rms arm of D3-5 §3.2)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    gain = np.ascontiguousarray(gain, dtype=np.float32)
    y = np.zeros(x.size, np.float64)
    lib().mqo_rmsnorm(_p(x), _p(gain), float(eps), x.size, _p(y))
    return y


def swiglu(g: np.ndarray, u: np.ndarray) -> np.ndarray:
    """y = (g / (1 + exp(-g))) * u in fp64 (D3-5 §3.2, swiglu_quant body)."""
    g = np.ascontiguousarray(g, dtype=np.float32)
    u = np.ascontiguousarray(u, dtype=np.float32)
    y = np.zeros(g.size, np.float64)
    lib().mqo_swiglu(_p(g), _p(u), g.size, _p(y))
    return y
