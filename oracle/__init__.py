"""Oracle for the fused attention forward: plain, slow, fp64, CPU only.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU
baseline (and its ``--impl reference`` arm) may import this package. The CUDA library never
calls it and shares no code with it; the only thing both sides use is the seeded input
generator, which holds none of the method's arithmetic.

Contents
--------
``attention`` / ``attention_rows``
    The plain definition of attention (C, fp64, OpenMP over rows) in ``attn_oracle.c``:
    S = scale * Q K^T, three-pass softmax, O = P V, LSE = m + ln l ("FlashAttention
    优化原理与实现要点解析" §1, §2, §4.1; causal rule §7; the kept statistics m, l from
    "FlashAttention V2 核心原理与架构设计" §2.3).
``decode``
    Exact value of bf16 / fp16 bit patterns as float64.
``softmax_three_pass``, ``online_softmax``, ``online_softmax_stream``, ``blockwise_attention``
    The method's own algorithm in fp64 numpy, in the pages' order and notation, used to show
    that tiling with online softmax reaches the plain definition (see ``softmax.py``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from .softmax import (blockwise_attention, online_softmax, online_softmax_stream,
                      softmax_three_pass)

__all__ = [
    "build", "load", "decode", "attention", "attention_rows", "attention_bwd", "max_threads",
    "softmax_three_pass", "online_softmax", "online_softmax_stream", "blockwise_attention",
    "KIND_F64", "KIND_BF16", "KIND_FP16",
]

KIND_F64, KIND_BF16, KIND_FP16 = 0, 1, 2
_DTYPE_KIND = {"bf16": KIND_BF16, "fp16": KIND_FP16}

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "attn_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

_lock = threading.Lock()
_lib = None


def compile_library(source: str, out_path: str) -> str:
    """Compile an oracle C source into a shared library with gcc (-O2, IEEE maths, OpenMP)."""
    os.makedirs(os.path.dirname(out_path), exist_ok=True)
    tmp = out_path + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math",
           source, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out_path)
    return out_path


def build(force: bool = False) -> str:
    """Compile ``attn_oracle.c`` into ``oracle/_build/liboracle.so`` when stale."""
    with _lock:
        stale = (not os.path.exists(_LIB_PATH)
                 or os.path.getmtime(_LIB_PATH) < os.path.getmtime(SOURCE))
        if force or stale:
            compile_library(SOURCE, _LIB_PATH)
    return _LIB_PATH


def _bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    vp, i64, i32, dbl = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_double
    lib.oracle_decode.argtypes = [vp, i64, i32, vp]
    lib.oracle_attention.argtypes = [vp, vp, vp, i32, i64, i64, i64, i64, i32, dbl, vp, vp]
    lib.oracle_attention_rows.argtypes = [vp, vp, vp, i32, i64, i64, i64, i64, i32, dbl, vp,
                                          i64, vp, vp]
    lib.oracle_attention_masked.argtypes = [vp, vp, vp, i32, i64, i64, i64, i64, i32, i64, i64,
                                            vp, dbl, vp, vp]
    lib.oracle_attention_rows_masked.argtypes = [vp, vp, vp, i32, i64, i64, i64, i64, i32, i64,
                                                 i64, vp, dbl, vp, i64, vp, vp]
    lib.oracle_attention_qk.argtypes = [vp, vp, vp, i32, i64, i64, i64, i64, i64, i32, i64, i64,
                                        vp, dbl, vp, vp]
    lib.oracle_attention_rows_qk.argtypes = [vp, vp, vp, i32, i64, i64, i64, i64, i64, i32, i64,
                                             i64, vp, dbl, vp, i64, vp, vp]
    lib.oracle_attention_bwd.argtypes = [vp, vp, vp, vp, i32, i64, i64, i64, i64, i32, i64, i64,
                                         vp, dbl, vp, vp, vp]
    lib.oracle_attention_bwd.restype = i32
    lib.oracle_attention_bwd_sampled.argtypes = [vp, vp, vp, vp, i32, i64, i64, i64, i64, i32,
                                                 i64, i64, vp, dbl, vp, i64, vp, i64, vp, i64,
                                                 vp, vp, vp]
    lib.oracle_attention_bwd_sampled.restype = i32
    for fn in (lib.oracle_decode, lib.oracle_attention, lib.oracle_attention_rows,
               lib.oracle_attention_masked, lib.oracle_attention_rows_masked,
               lib.oracle_attention_qk, lib.oracle_attention_rows_qk, lib.oracle_max_threads):
        fn.restype = i32
    lib.oracle_max_threads.argtypes = []
    return lib


def load(path: str | None = None) -> ctypes.CDLL:
    """Load the compiled oracle (building it first if needed). ``path`` loads another build."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    if _lib is None:
        _lib = _bind(ctypes.CDLL(build()))
    return _lib


def max_threads(lib: ctypes.CDLL | None = None) -> int:
    """Number of OpenMP threads the oracle uses."""
    return int((lib or load()).oracle_max_threads())


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _kind_and_arrays(q, k, v, dtype):
    if dtype is None:
        arrs = [np.ascontiguousarray(x, dtype=np.float64) for x in (q, k, v)]
        return KIND_F64, arrs
    kind = _DTYPE_KIND[dtype]
    arrs = []
    for x in (q, k, v):
        x = np.asarray(x)
        if x.dtype != np.uint16:
            raise TypeError("bf16/fp16 inputs are passed as their uint16 bit patterns")
        arrs.append(np.ascontiguousarray(x))
    return kind, arrs


def decode(bits: np.ndarray, dtype: str, lib: ctypes.CDLL | None = None) -> np.ndarray:
    """Exact float64 values of a bf16 or fp16 bit-pattern array (any shape)."""
    lib = lib or load()
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(bits.shape, dtype=np.float64)
    rc = lib.oracle_decode(_ptr(bits), bits.size, _DTYPE_KIND[dtype], _ptr(out))
    if rc:
        raise RuntimeError("oracle_decode failed: %d" % rc)
    return out


def _shapes(q, k, v):
    if q.ndim != 4 or k.ndim != 4 or k.shape != v.shape:
        raise ValueError("q must be [B, Nq, H, d] and k, v one [B, Nk, H, d] shape")
    B, Nq, H, d = q.shape
    if k.shape[0] != B or k.shape[2] != H or k.shape[3] != d or k.shape[1] < Nq:
        raise ValueError("k, v must be [B, Nk, H, d] with Nk >= Nq")
    return B, Nq, k.shape[1], H, d


def _lengths(seqlens_k, B):
    if seqlens_k is None:
        return None, None
    arr = np.ascontiguousarray(np.asarray(seqlens_k, dtype=np.int32).reshape(-1))
    if arr.size != B:
        raise ValueError("seqlens_k must have one entry per batch")
    return arr, _ptr(arr)


def attention(q, k, v, causal: bool, scale: float, dtype: str | None = None,
              lib: ctypes.CDLL | None = None, window=(-1, -1), seqlens_k=None):
    """Plain fp64 attention over [B, N, H, d] inputs.

    ``dtype`` None: q, k, v are real arrays (converted to float64). ``dtype`` "bf16"/"fp16":
    they are uint16 bit patterns of that type. q is [B, Nq, H, d], k and v [B, Nk, H, d] with
    Nk >= Nq; the queries are the last Nq positions (query i sits at position i + Nk - Nq).
    ``window`` = (left, right): key j is allowed for the query at position p only if
    j >= p - left (left >= 0) and j <= p + right (right >= 0); -1 means no bound; causal means
    j <= p. ``seqlens_k``: optional per-batch key lengths (keys at or past the length do not
    exist). Rows with no allowed key get O = 0 and LSE = -inf. Returns (o [B,Nq,H,d] float64,
    lse [B,H,Nq] float64). ``scale`` is used exactly as given.
    """
    lib = lib or load()
    kind, (q, k, v) = _kind_and_arrays(q, k, v, dtype)
    B, Nq, Nk, H, d = _shapes(q, k, v)
    lens, lens_ptr = _lengths(seqlens_k, B)
    o = np.empty((B, Nq, H, d), dtype=np.float64)
    lse = np.empty((B, H, Nq), dtype=np.float64)
    rc = lib.oracle_attention_qk(_ptr(q), _ptr(k), _ptr(v), kind, B, H, Nq, Nk, d,
                                 int(bool(causal)), int(window[0]), int(window[1]), lens_ptr,
                                 float(scale), _ptr(o), _ptr(lse))
    if rc:
        raise RuntimeError("oracle_attention_qk failed: %d" % rc)
    return o, lse


def attention_rows(q, k, v, rows, causal: bool, scale: float, dtype: str | None = None,
                   lib: ctypes.CDLL | None = None, window=(-1, -1), seqlens_k=None):
    """Selected output rows of the same attention. ``rows`` is an int array of (b, h, i)
    triples, shape [R, 3]. Returns (o_rows [R, d], lse_rows [R])."""
    lib = lib or load()
    kind, (q, k, v) = _kind_and_arrays(q, k, v, dtype)
    B, Nq, Nk, H, d = _shapes(q, k, v)
    lens, lens_ptr = _lengths(seqlens_k, B)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 3))
    o = np.empty((rows.shape[0], d), dtype=np.float64)
    lse = np.empty((rows.shape[0],), dtype=np.float64)
    rc = lib.oracle_attention_rows_qk(_ptr(q), _ptr(k), _ptr(v), kind, B, H, Nq, Nk, d,
                                      int(bool(causal)), int(window[0]), int(window[1]),
                                      lens_ptr, float(scale), _ptr(rows), rows.shape[0],
                                      _ptr(o), _ptr(lse))
    if rc:
        raise RuntimeError("oracle_attention_rows_qk failed: %d" % rc)
    return o, lse


def attention_bwd(q, k, v, dout, causal: bool, scale: float, dtype: str | None = None,
                  lib: ctypes.CDLL | None = None, window=(-1, -1), seqlens_k=None):
    """Gradients (dq, dk, dv), float64 [B, N, H, d], of L = sum(dout * O) for the attention
    ``attention(q, k, v, causal, scale, ...)`` (queries and keys share N). ``dout`` has q's
    shape and, like q, k, v, is a real array (dtype None) or uint16 bit patterns of ``dtype``.
    """
    lib = lib or load()
    kind, (q, k, v) = _kind_and_arrays(q, k, v, dtype)
    _, (dout, _, _) = _kind_and_arrays(dout, dout, dout, dtype)
    B, Nq, Nk, H, d = _shapes(q, k, v)
    if Nq != Nk or dout.shape != q.shape:
        raise ValueError("the backward takes one length N and dout shaped like q")
    lens, lens_ptr = _lengths(seqlens_k, B)
    dq, dk, dv = (np.empty((B, Nq, H, d), dtype=np.float64) for _ in range(3))
    rc = lib.oracle_attention_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), kind, B, H, Nq, d,
                                  int(bool(causal)), int(window[0]), int(window[1]), lens_ptr,
                                  float(scale), _ptr(dq), _ptr(dk), _ptr(dv))
    if rc:
        raise RuntimeError("oracle_attention_bwd failed: %d" % rc)
    return dq, dk, dv


def attention_bwd_sampled(q, k, v, dout, causal: bool, scale: float, heads, keys, queries,
                          dtype: str | None = None, lib: ctypes.CDLL | None = None,
                          window=(-1, -1), seqlens_k=None):
    """The gradients of ``attention_bwd`` on sampled outputs only, without N x N storage:
    for each (b, h) in ``heads``, dK and dV at the key positions ``keys`` and dQ at the query
    positions ``queries``. Returns float64 arrays dq [len(heads), len(queries), d] and dk, dv
    [len(heads), len(keys), d]. The masks of ``attention`` (causal, window, key lengths);
    queries and keys share N."""
    lib = lib or load()
    kind, (q, k, v) = _kind_and_arrays(q, k, v, dtype)
    _, (dout, _, _) = _kind_and_arrays(dout, dout, dout, dtype)
    B, Nq, Nk, H, d = _shapes(q, k, v)
    if Nq != Nk or dout.shape != q.shape:
        raise ValueError("the backward takes one length N and dout shaped like q")
    hs = np.ascontiguousarray(np.asarray(heads, dtype=np.int64).reshape(-1, 2))
    ks = np.ascontiguousarray(np.asarray(keys, dtype=np.int64).ravel())
    qs = np.ascontiguousarray(np.asarray(queries, dtype=np.int64).ravel())
    dq = np.empty((len(hs), len(qs), d), dtype=np.float64)
    dk = np.empty((len(hs), len(ks), d), dtype=np.float64)
    dv = np.empty((len(hs), len(ks), d), dtype=np.float64)
    lens, lens_ptr = _lengths(seqlens_k, B)
    rc = lib.oracle_attention_bwd_sampled(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), kind, B, H, Nq,
                                          d, int(bool(causal)), int(window[0]), int(window[1]),
                                          lens_ptr, float(scale), _ptr(hs), len(hs), _ptr(ks),
                                          len(ks), _ptr(qs), len(qs), _ptr(dq), _ptr(dk),
                                          _ptr(dv))
    if rc:
        raise RuntimeError("oracle_attention_bwd_sampled failed: %d" % rc)
    return dq, dk, dv
