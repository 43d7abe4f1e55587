"""Python access to the fp64 CPU oracle in ``oracle/vst_oracle.c``.

TEST INFRASTRUCTURE. Only the test suite, the package smoke check and the CPU-baseline leg
of the benchmark import this module. The CUDA library never imports, links or calls it, and
it imports nothing from the CUDA library.

Inputs are bf16 bit patterns held in ``numpy.uint16`` arrays (the exact values the GPU path
receives); outputs are ``float64``. The C file states what each function computes and the
passages it follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "vst_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libvst_oracle.so")
_lib = None
_lock = threading.Lock()

THETA = 1.0e6


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fused multiply-add contraction, IEEE semantics)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + ".tmp.%d" % os.getpid()
        subprocess.check_call(
            ["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
             "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _RingState(ctypes.Structure):
    _fields_ = [("n_kv", ctypes.c_longlong), ("abs_base", ctypes.c_longlong),
                ("abs_next", ctypes.c_longlong), ("n_compactions", ctypes.c_longlong)]


def _bind(lib):
    """Declare the C signatures on a loaded oracle library."""
    P = ctypes.c_void_p
    LL = ctypes.c_longlong
    I = ctypes.c_int
    D = ctypes.c_double
    lib.vst_oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
    lib.vst_oracle_bf16_to_double.restype = D
    lib.vst_oracle_bf16_to_double_n.argtypes = [P, LL, P]
    lib.vst_oracle_rope.argtypes = [P, I, D, LL, P]
    lib.vst_oracle_rope_rows.argtypes = [P, LL, I, I, D, LL, P]
    lib.vst_oracle_attend.argtypes = [P, P, P, LL, I, I, I, LL, LL, LL, P]
    lib.vst_oracle_attend_lr.argtypes = [P, P, P, LL, I, I, I, LL, LL, LL, LL, P]
    lib.vst_oracle_ring_feed.argtypes = [ctypes.POINTER(_RingState), LL, LL, LL, LL]
    for f in ("vst_oracle_bf16_to_double_n", "vst_oracle_rope", "vst_oracle_rope_rows",
              "vst_oracle_attend", "vst_oracle_attend_lr", "vst_oracle_ring_feed"):
        getattr(lib, f).restype = None
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _u16(x) -> np.ndarray:
    a = np.ascontiguousarray(x)
    if a.dtype != np.uint16:
        raise TypeError("bf16 inputs are passed as uint16 bit patterns, got %s" % a.dtype)
    return a


def bf16_to_double(bits) -> np.ndarray:
    a = _u16(bits)
    out = np.empty(a.shape, dtype=np.float64)
    _load().vst_oracle_bf16_to_double_n(_ptr(a), a.size, _ptr(out))
    return out


def rope(x, p: int, theta: float = THETA) -> np.ndarray:
    """NEOX rotation of one double vector x[D] at absolute position p."""
    a = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty_like(a)
    _load().vst_oracle_rope(_ptr(a), a.shape[-1], theta, int(p), _ptr(out))
    return out


def rope_rows(bits, pos0: int = 0, theta: float = THETA) -> np.ndarray:
    """Rotate a bf16 [T][heads][D] tensor; row r is at absolute position pos0 + r."""
    a = _u16(bits)
    T, nh, D = a.shape
    if D > 1024:
        raise ValueError("head_dim > 1024")
    out = np.empty(a.shape, dtype=np.float64)
    _load().vst_oracle_rope_rows(_ptr(a), T, nh, D, theta, int(pos0), _ptr(out))
    return out


def attend(qr: np.ndarray, kr: np.ndarray, v: np.ndarray, window: int,
           rows: tuple[int, int] | None = None, threads: int = 1) -> np.ndarray:
    """Windowed-causal attention rows of rotated double inputs.

    qr [T][H][D], kr/v [T][Hk][D]; returns out [r1-r0][H][D] for rows [r0, r1)."""
    qr = np.ascontiguousarray(qr, dtype=np.float64)
    kr = np.ascontiguousarray(kr, dtype=np.float64)
    v = np.ascontiguousarray(v, dtype=np.float64)
    T, H, D = qr.shape
    Hk = kr.shape[1]
    if kr.shape != (T, Hk, D) or v.shape != (T, Hk, D) or H % Hk:
        raise ValueError("shape mismatch")
    r0, r1 = rows if rows is not None else (0, T)
    out = np.empty((r1 - r0, H, D), dtype=np.float64)
    lib = _load()

    def run(a, b):
        sub = out[a - r0:b - r0]
        # out rows are contiguous, so a slice of out is a valid output buffer
        lib.vst_oracle_attend(_ptr(qr), _ptr(kr), _ptr(v), T, H, Hk, D, int(window), a, b,
                              sub.ctypes.data_as(ctypes.c_void_p))

    if threads <= 1 or r1 - r0 < 2 * threads:
        run(r0, r1)
    else:
        step = -(-(r1 - r0) // (4 * threads))
        spans = [(a, min(a + step, r1)) for a in range(r0, r1, step)]
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(lambda s: run(*s), spans))
    return out


def attend_lr(qr: np.ndarray, kr: np.ndarray, v: np.ndarray, left: int, right: int,
              rows: tuple[int, int] | None = None, threads: int = 1) -> np.ndarray:
    """Sliding attention with a left window and a right lookahead: row i sees key j of the
    clip iff 0 <= i - j < left or 0 < j - i < right. Arguments as `attend`."""
    qr = np.ascontiguousarray(qr, dtype=np.float64)
    kr = np.ascontiguousarray(kr, dtype=np.float64)
    v = np.ascontiguousarray(v, dtype=np.float64)
    T, H, D = qr.shape
    Hk = kr.shape[1]
    if kr.shape != (T, Hk, D) or v.shape != (T, Hk, D) or H % Hk or left < 1 or right < 0:
        raise ValueError("shape or mask mismatch")
    r0, r1 = rows if rows is not None else (0, T)
    out = np.empty((r1 - r0, H, D), dtype=np.float64)
    lib = _load()

    def run(a, b):
        sub = out[a - r0:b - r0]
        lib.vst_oracle_attend_lr(_ptr(qr), _ptr(kr), _ptr(v), T, H, Hk, D, int(left), int(right), a, b,
                                 sub.ctypes.data_as(ctypes.c_void_p))

    if threads <= 1 or r1 - r0 < 2 * threads:
        run(r0, r1)
    else:
        step = -(-(r1 - r0) // (4 * threads))
        spans = [(a, min(a + step, r1)) for a in range(r0, r1, step)]
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(lambda s: run(*s), spans))
    return out


def attention_lr(q_bits, k_bits, v_bits, left: int, right: int, pos0: int = 0, theta: float = THETA,
                 rows: tuple[int, int] | None = None, threads: int = 1) -> np.ndarray:
    """Whole-clip oracle with a (left, right) mask: RoPE at absolute positions pos0 + t,
    then `attend_lr`. q [T][H][D], k/v [T][Hk][D] as bf16 bit patterns."""
    qr = rope_rows(q_bits, pos0, theta)
    kr = rope_rows(k_bits, pos0, theta)
    vv = bf16_to_double(v_bits)
    return attend_lr(qr, kr, vv, left, right, rows, threads)


def attention(q_bits, k_bits, v_bits, window: int, pos0: int = 0, theta: float = THETA,
              rows: tuple[int, int] | None = None, threads: int = 1) -> np.ndarray:
    """Whole-clip oracle: RoPE at absolute positions pos0 + t, then windowed-causal attention.

    q [T][H][D], k/v [T][Hk][D] as bf16 bit patterns; returns double [rows][H][D]."""
    qr = rope_rows(q_bits, pos0, theta)
    kr = rope_rows(k_bits, pos0, theta)
    vv = bf16_to_double(v_bits)
    return attend(qr, kr, vv, window, rows, threads)


def attention_row(q_bits, k_bits, v_bits, i: int, window: int, theta: float = THETA) -> np.ndarray:
    """One output row (all heads) at absolute position i, from the window [i-W+1, i] alone.

    q_bits [H][D] is the query of row i; k_bits/v_bits [n][Hk][D] hold positions
    i-n+1 .. i, with n = min(W, i+1)."""
    n = k_bits.shape[0]
    if n != min(window, i + 1):
        raise ValueError("window slice has %d rows, expected %d" % (n, min(window, i + 1)))
    j0 = i - n + 1
    H, D = q_bits.shape
    qr = np.zeros((n, H, D), dtype=np.float64)
    qr[-1] = rope_rows(np.ascontiguousarray(q_bits)[None], i, theta)[0]
    kr = rope_rows(k_bits, j0, theta)
    vv = bf16_to_double(v_bits)
    return attend(qr, kr, vv, n, rows=(n - 1, n))[0]


class RingState:
    """The pages' encoder ring bookkeeping (slots [0, n_kv) hold frames abs_base...)."""

    def __init__(self):
        self._s = _RingState(0, 0, 0, 0)

    def feed(self, n_new: int, ring_slots: int = 1536, keep: int = 750, max_batch: int = 512):
        _load().vst_oracle_ring_feed(ctypes.byref(self._s), int(n_new), ring_slots, keep, max_batch)
        return self

    n_kv = property(lambda self: self._s.n_kv)
    abs_base = property(lambda self: self._s.abs_base)
    abs_next = property(lambda self: self._s.abs_next)
    n_compactions = property(lambda self: self._s.n_compactions)
