"""fp64 CPU oracle for the frame-window + reference-frame block-sparse attention.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg may import this package. The library
(``block_sparse_video_frame_gb300``) never imports it and shares no code with it.

The arithmetic lives in ``vdit_oracle.c`` (plain C, fp64, OpenMP over rows);
this module builds it with gcc on first use and wraps it with ctypes/numpy.
Every function states the plain definition it computes; see the C file for
the formulas and the passages of "HeyGen x Google Cloud: Bringing Avatar IV to
TPUs" they follow ("Deleting the Mask", Fig. 3; "Unchaining the Softmax", Fig. 4).

Parity pins (tests/test_oracle_*.py): closed-form schedule counts, brute force
on tiny inputs, dense and block-diagonal special cases against torch's float64
scaled-dot-product attention, centring and permutation invariance, bound >= max,
key statistics against numpy. No function is "parity unpinned".
tests/test_oracle_mutants.py plants mistakes in copies of the C source and
checks that these pins reject every one.

VDIT_ORACLE_LIB, when set, names an already built oracle library to load
instead of building ``vdit_oracle.c`` (the planted-mistake tests point it at
their mutated builds).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "vdit_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

_i32p = ctypes.POINTER(ctypes.c_int32)
_i64p = ctypes.POINTER(ctypes.c_int64)
_f64p = ctypes.POINTER(ctypes.c_double)
_u8p = ctypes.POINTER(ctypes.c_uint8)


GCC_FLAGS = ("-O2", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared", "-std=c11")


def compile_source(src: str, out: str) -> None:
    """gcc one oracle source file into a shared library (fp64, no fast-math, no
    FMA contraction)."""
    subprocess.run(["gcc", *GCC_FLAGS, "-o", out, src, "-lm"], check=True)


def build(force: bool = False) -> str:
    """Compile the oracle (vdit_oracle.c) into oracle/_build/liboracle.so."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        compile_source(_SRC, tmp)
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(os.environ.get("VDIT_ORACLE_LIB") or build())
        lib.vo_set_threads.argtypes = [ctypes.c_int]
        lib.vo_set_threads.restype = ctypes.c_int
        lib.vo_mask.argtypes = [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                ctypes.c_int64, ctypes.c_int64]
        lib.vo_mask.restype = ctypes.c_int
        lib.vo_block_census.argtypes = [ctypes.c_int32] * 5 + [_i64p] * 3
        lib.vo_block_census.restype = None
        lib.vo_schedule.argtypes = [ctypes.c_int32] * 5 + [_i32p, _i32p, ctypes.c_int64, _i64p,
                                                          _i32p, _i64p]
        lib.vo_schedule.restype = ctypes.c_int
        lib.vo_key_stats.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                     ctypes.c_int32, ctypes.c_int32, ctypes.c_int64,
                                     ctypes.c_int32, _i64p, _i64p, ctypes.c_double,
                                     ctypes.c_double, _f64p, _f64p, _f64p, _f64p, _u8p]
        lib.vo_key_stats.restype = None
        lib.vo_row_bounds.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int32,
                                      ctypes.c_int64, ctypes.c_int32, _i64p, _f64p, _f64p,
                                      ctypes.c_double, ctypes.c_int64, _i64p, _f64p]
        lib.vo_row_bounds.restype = None
        lib.vo_attention_rows.argtypes = [ctypes.c_void_p] * 3 + [
            ctypes.c_int, ctypes.c_int32, ctypes.c_int64, ctypes.c_int32, _i64p, _i64p, _i64p,
            ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_double, ctypes.c_int64,
            _i64p, _f64p, _f64p, _f64p]
        lib.vo_attention_rows.restype = None
        lib.vo_frame_stats.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                       ctypes.c_int32, ctypes.c_int32, ctypes.c_int64,
                                       ctypes.c_int32, _i64p, _i64p, ctypes.c_int32,
                                       ctypes.c_int32, ctypes.c_int32, ctypes.c_double,
                                       ctypes.c_double, _f64p, _f64p, _f64p, _u8p]
        lib.vo_frame_stats.restype = None
        lib.vo_row_bounds_frames.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int32,
                                             ctypes.c_int64, ctypes.c_int32, _i64p, _f64p,
                                             _f64p, ctypes.c_int32, ctypes.c_double,
                                             ctypes.c_int64, _i64p, _f64p]
        lib.vo_row_bounds_frames.restype = None
        lib.vo_qkv_prologue.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                        ctypes.c_int32, ctypes.c_int64, ctypes.c_int32, _i64p,
                                        _f64p, ctypes.c_int32, ctypes.c_int32, ctypes.c_double,
                                        ctypes.c_double, ctypes.c_int64, _i64p, _f64p, _f64p,
                                        _f64p]
        lib.vo_qkv_prologue.restype = None
        _lib = lib
        return lib


def _ptr(a, t):
    return a.ctypes.data_as(t)


def _as_input(x):
    """Accept a torch bf16/float64 tensor or a numpy uint16(bf16 bits)/float64 array of
    shape [B, H, N, D] with contiguous last dim. Returns (array, dtype code, strides)."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            if x.dtype == torch.bfloat16:
                x = x.contiguous().view(torch.int16).numpy().view(np.uint16)
            elif x.dtype == torch.float64:
                x = x.contiguous().numpy()
            else:
                raise TypeError(f"oracle input must be bf16 or float64, got {x.dtype}")
    except ImportError:  # pragma: no cover
        pass
    x = np.asarray(x)
    if x.dtype == np.uint16:
        code = 0
    elif x.dtype == np.float64:
        code = 1
    else:
        raise TypeError(f"oracle input must be bf16 bits (uint16) or float64, got {x.dtype}")
    if x.ndim != 4 or x.strides[3] != x.itemsize:
        x = np.ascontiguousarray(x)
    strides = np.array([s // x.itemsize for s in x.strides[:3]], dtype=np.int64)
    return x, code, strides


def set_threads(n: int = 0) -> int:
    """Set (n > 0) and return the number of OpenMP threads the oracle uses."""
    return _load().vo_set_threads(int(n))


def mask(T: int, W: int, ref: int, i: int, j: int) -> bool:
    return bool(_load().vo_mask(T, W, ref, i, j))


def block_census(F, T, W, ref, bs):
    """(fully live, partially live, dead) counts of bs x bs blocks."""
    out = [ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()]
    _load().vo_block_census(F, T, W, ref, bs, *[ctypes.byref(o) for o in out])
    return tuple(int(o.value) for o in out)


class Schedule:
    def __init__(self, row_ptr, col_idx, runs, live_pairs):
        self.row_ptr = row_ptr
        self.col_idx = col_idx
        self.runs = runs
        self.live_pairs = live_pairs


def schedule(F, T, W, ref, bs) -> Schedule:
    """Block schedule built by testing every token pair of every block (see C)."""
    N = F * T
    nb = (N + bs - 1) // bs
    row_ptr = np.zeros(nb + 1, dtype=np.int32)
    runs = np.zeros(4 * F, dtype=np.int32)
    cap = nb * nb
    col_idx = np.zeros(max(cap, 1), dtype=np.int32)
    nnz = ctypes.c_int64()
    pairs = ctypes.c_int64()
    rc = _load().vo_schedule(F, T, W, ref, bs, _ptr(row_ptr, _i32p), _ptr(col_idx, _i32p),
                             cap, ctypes.byref(nnz), _ptr(runs, _i32p), ctypes.byref(pairs))
    if rc == -1:
        raise ValueError("partially live block: block size does not align with frames")
    if rc != 0:
        raise RuntimeError(f"vo_schedule failed with {rc}")
    return Schedule(row_ptr, col_idx[: nnz.value].copy(), runs.reshape(F, 4), int(pairs.value))


def key_stats(q, k, scale: float, tau: float):
    """Returns dict(c=[B,H,D], R=[B,H], qmax=[B,H], G=[B,H], elig=[B,H] uint8), fp64."""
    qa, qc, qs = _as_input(q)
    ka, kc, ks = _as_input(k)
    if qc != kc:
        raise TypeError("q and k must have the same element type")
    B, H, N, D = ka.shape
    c = np.zeros((B, H, D))
    R = np.zeros((B, H))
    qmax = np.zeros((B, H))
    G = np.zeros((B, H))
    elig = np.zeros((B, H), dtype=np.uint8)
    _load().vo_key_stats(qa.ctypes.data, ka.ctypes.data, kc, B, H, N, D, _ptr(qs, _i64p),
                         _ptr(ks, _i64p), float(scale), float(tau), _ptr(c, _f64p),
                         _ptr(R, _f64p), _ptr(qmax, _f64p), _ptr(G, _f64p), _ptr(elig, _u8p))
    return dict(c=c, R=R, qmax=qmax, G=G, elig=elig)


def frame_stats(q, k, T: int, W: int, ref: int, scale: float, tau: float):
    """Per query frame: R_f (largest centred norm over the keys the frame sees),
    Qmax_f, G_f and eligibility. Returns dict of [B, H, F] arrays."""
    qa, qc, qs = _as_input(q)
    ka, kc, ks = _as_input(k)
    if qc != kc:
        raise TypeError("q and k must have the same element type")
    B, H, N, D = ka.shape
    F = N // T
    R = np.zeros((B, H, F))
    qmax = np.zeros((B, H, F))
    G = np.zeros((B, H, F))
    elig = np.zeros((B, H, F), dtype=np.uint8)
    _load().vo_frame_stats(qa.ctypes.data, ka.ctypes.data, kc, B, H, N, D, _ptr(qs, _i64p),
                           _ptr(ks, _i64p), T, W, ref, float(scale), float(tau), _ptr(R, _f64p),
                           _ptr(qmax, _f64p), _ptr(G, _f64p), _ptr(elig, _u8p))
    return dict(R=R, qmax=qmax, G=G, elig=elig)


def row_bounds_frames(q, c, Rf, T: int, scale: float, rows=None):
    """m_i = scale * (q_i . c_h + |q_i| R_{h, f(i)}) with per-query-frame R."""
    qa, qc, qs = _as_input(q)
    B, H, N, D = qa.shape
    rows = _rows_arg(rows, B * H, N)
    c = np.ascontiguousarray(np.asarray(c, dtype=np.float64))
    Rf = np.ascontiguousarray(np.asarray(Rf, dtype=np.float64))
    m = np.zeros(len(rows))
    _load().vo_row_bounds_frames(qa.ctypes.data, qc, H, N, D, _ptr(qs, _i64p), _ptr(c, _f64p),
                                 _ptr(Rf, _f64p), T, float(scale), len(rows), _ptr(rows, _i64p),
                                 _ptr(m, _f64p))
    return m


def _as_matrix(x, ndim):
    """bf16 torch / uint16 numpy (bf16 bits) / float64 -> (array, dtype code)."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            if x.dtype == torch.bfloat16:
                x = x.contiguous().view(torch.int16).numpy().view(np.uint16)
            elif x.dtype == torch.float64:
                x = x.contiguous().numpy()
            else:
                raise TypeError(f"oracle input must be bf16 or float64, got {x.dtype}")
    except ImportError:  # pragma: no cover
        pass
    x = np.ascontiguousarray(np.asarray(x))
    if x.ndim != ndim:
        raise ValueError(f"expected {ndim} dimensions, got {x.ndim}")
    if x.dtype == np.uint16:
        return x, 0
    if x.dtype == np.float64:
        return x, 1
    raise TypeError(f"oracle input must be bf16 bits or float64, got {x.dtype}")


def qkv_prologue(x, w, gamma, H: int, D: int, eps: float, base: float, rows=None):
    """RMSNorm -> QKV projection -> rotary embedding on q, k (pairs i, i + D/2,
    position = token index) -> per-head outputs. x: [B, N, C]; w: [3*H*D, C]
    (q rows, then k, then v, head-major); gamma: [C]. Returns (q, k, v), each
    [nrows, H, D] float64, for flattened rows b*N + n (all rows by default)."""
    xa, xc = _as_matrix(x, 3)
    wa, wc = _as_matrix(w, 2)
    if xc != wc:
        raise TypeError("x and w must have the same element type")
    B, N, C = xa.shape
    if wa.shape != (3 * H * D, C):
        raise ValueError(f"w must be [{3 * H * D}, {C}], got {wa.shape}")
    g = np.ascontiguousarray(np.asarray(gamma, dtype=np.float64))
    rows = np.ascontiguousarray(np.arange(B * N, dtype=np.int64) if rows is None
                                else np.asarray(rows, dtype=np.int64))
    xs = np.array([N * C, C], dtype=np.int64)
    out = [np.zeros((len(rows), H, D)) for _ in range(3)]
    _load().vo_qkv_prologue(xa.ctypes.data, wa.ctypes.data, xc, B, N, C, _ptr(xs, _i64p),
                            _ptr(g, _f64p), H, D, float(eps), float(base), len(rows),
                            _ptr(rows, _i64p), *[_ptr(o, _f64p) for o in out])
    return tuple(out)


def _rows_arg(rows, BH, N):
    if rows is None:
        rows = np.arange(BH * N, dtype=np.int64)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    return rows


def row_bounds(q, c, R, scale: float, rows=None):
    """m_i = scale * (q_i . c_h + |q_i| R_h) for the given flattened rows."""
    qa, qc, qs = _as_input(q)
    B, H, N, D = qa.shape
    rows = _rows_arg(rows, B * H, N)
    c = np.ascontiguousarray(np.asarray(c, dtype=np.float64))
    R = np.ascontiguousarray(np.asarray(R, dtype=np.float64))
    m = np.zeros(len(rows))
    _load().vo_row_bounds(qa.ctypes.data, qc, H, N, D, _ptr(qs, _i64p), _ptr(c, _f64p),
                          _ptr(R, _f64p), float(scale), len(rows), _ptr(rows, _i64p),
                          _ptr(m, _f64p))
    return m


def attention_rows(q, k, v, T: int, W: int, ref: int, scale: float, rows=None):
    """fp64 masked attention for flattened rows ((b*H + h)*N + i).
    Returns (o [nrows, D], lse [nrows], rowmax [nrows])."""
    qa, qc, qs = _as_input(q)
    ka, kc, ks = _as_input(k)
    va, vc, vs = _as_input(v)
    if not (qc == kc == vc):
        raise TypeError("q, k, v must have the same element type")
    B, H, N, D = qa.shape
    rows = _rows_arg(rows, B * H, N)
    o = np.zeros((len(rows), D))
    lse = np.zeros(len(rows))
    mx = np.zeros(len(rows))
    _load().vo_attention_rows(qa.ctypes.data, ka.ctypes.data, va.ctypes.data, qc, H, N, D,
                              _ptr(qs, _i64p), _ptr(ks, _i64p), _ptr(vs, _i64p), T, W, ref,
                              float(scale), len(rows), _ptr(rows, _i64p), _ptr(o, _f64p),
                              _ptr(lse, _f64p), _ptr(mx, _f64p))
    return o, lse, mx
