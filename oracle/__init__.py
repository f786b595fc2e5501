"""CPU fp64 oracle for Hybrid Tree Attention.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package; the product path
(the CUDA library and its Python binding) never does. The arithmetic lives in
``hta_oracle.c`` (plain C, fp64, OpenMP over query rows); this module only
compiles it with gcc and marshals numpy arrays through ctypes.

Definitions followed (page titles and sections):
  * "LongSpec: Long-Context Lossless Speculative Decoding with Efficient
    Drafting and Verification", Korean summary section 2.C "Fast Tree
    Attention", Dutch summary Methodologie section 3: the verification
    attention equals one softmax over [cached prefix || visible tree keys];
    the split-and-merge method reproduces it exactly.
  * "LogitSpec: Accelerating Retrieval-based Speculative Decoding via Next
    Next Token Speculation", section 2, workflow step 2: the tree mask lets
    the target check every branch at once (read here as ancestor-or-self).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "hta_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libhta_oracle.so")
_lock = threading.Lock()
_lib = None


class _Dims(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int32),
        ("T", ctypes.c_int32),
        ("Hq", ctypes.c_int32),
        ("Hkv", ctypes.c_int32),
        ("d", ctypes.c_int32),
        ("Lmax", ctypes.c_int64),
        ("scale", ctypes.c_double),
    ]


def build(force: bool = False) -> str:
    """Compile hta_oracle.c into a shared library next to it (gcc, -O2, OpenMP)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)) or (
        os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-shared", "-fPIC",
               _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.oracle_build_mask.restype = ctypes.c_int
            lib.oracle_build_mask.argtypes = [ctypes.c_void_p, ctypes.c_int32,
                                              ctypes.c_int32, ctypes.c_void_p]
            lib.oracle_attention.restype = None
            lib.oracle_attention.argtypes = [ctypes.POINTER(_Dims)] + [ctypes.c_void_p] * 7 + [
                ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p]
            lib.oracle_num_threads.restype = ctypes.c_int
            lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
            _lib = lib
    return _lib


def mask_words(T: int) -> int:
    return (T + 31) // 32


def build_mask(parents: np.ndarray) -> tuple[np.ndarray, int]:
    """Ancestor-or-self bit mask [B][T][W] uint32 from parents [B][T] int32.

    Returns (mask, number_of_invalid_trees); rows of invalid trees are zero.
    """
    par = np.ascontiguousarray(parents, dtype=np.int32)
    if par.ndim == 1:
        par = par[None]
    B, T = par.shape
    mask = np.zeros((B, T, mask_words(T)), dtype=np.uint32)
    bad = _load().oracle_build_mask(par.ctypes.data, B, T, mask.ctypes.data)
    return mask, int(bad)


def _u16(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"bf16 tensors are passed as uint16 bit patterns, got {a.dtype}")
    return a


def attention(q, k_cache, v_cache, cache_lens, k_spec, v_spec, mask,
              rows=None, scale: float = 0.0):
    """Monolithic fp64 masked attention over [prefix || visible tree keys].

    q [B][T][Hq][d], k/v_cache [B][Hkv][Lmax][d], k/v_spec [B][Hkv][T][d]
    (all uint16 bf16 bits), cache_lens [B] int32, mask [B][T][W] uint32.
    rows: optional int64 array of flat row ids (b*T + t)*Hq + hq.
    Returns (o [n_rows][d] float64, lse [n_rows] float64); with rows=None the
    result is reshaped to [B][T][Hq][d] and [B][T][Hq].
    """
    q, k_cache, v_cache = _u16(q), _u16(k_cache), _u16(v_cache)
    k_spec, v_spec = _u16(k_spec), _u16(v_spec)
    lens = np.ascontiguousarray(cache_lens, dtype=np.int32)
    mask = np.ascontiguousarray(mask, dtype=np.uint32)
    B, T, Hq, d = q.shape
    _, Hkv, Lmax, d2 = k_cache.shape
    if d2 != d or Hq % Hkv or k_spec.shape != (B, Hkv, T, d) or mask.shape[:2] != (B, T):
        raise ValueError("inconsistent shapes")
    if (lens < 0).any() or (lens > Lmax).any():
        raise ValueError("cache_lens out of range")
    dims = _Dims(B, T, Hq, Hkv, d, Lmax, float(scale))
    if rows is None:
        n = B * T * Hq
        rows_arr = None
        rows_ptr = None
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
        n = rows_arr.size
        rows_ptr = rows_arr.ctypes.data
    o = np.zeros((n, d), dtype=np.float64)
    lse = np.zeros((n,), dtype=np.float64)
    _load().oracle_attention(ctypes.byref(dims), q.ctypes.data, k_cache.ctypes.data,
                             v_cache.ctypes.data, lens.ctypes.data, k_spec.ctypes.data,
                             v_spec.ctypes.data, mask.ctypes.data, rows_ptr, n,
                             o.ctypes.data, lse.ctypes.data)
    if rows is None:
        return o.reshape(B, T, Hq, d), lse.reshape(B, T, Hq)
    return o, lse


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))
