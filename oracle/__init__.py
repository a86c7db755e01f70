"""CPU oracle for the QSA indexer step (score + exact top-k).

TEST INFRASTRUCTURE ONLY: only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import this package.  The
product path (the CUDA library and its binding) never imports, links or calls
it, and it imports nothing from the product package.

The arithmetic lives in ``qsa_oracle.c`` (plain C, binary32 multiply-then-add
in a fixed order, compiled with ``-ffp-contract=off``); this module only builds
that file with gcc and marshals numpy arrays into it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qsa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle_qsa.so")
_lock = threading.Lock()
_lib = None

_i32p = ctypes.POINTER(ctypes.c_int32)
_f32p = ctypes.POINTER(ctypes.c_float)
_u16p = ctypes.POINTER(ctypes.c_uint16)


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP over rows) into liboracle_qsa.so."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
           "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        lib.oracle_half_to_float.restype = ctypes.c_float
        lib.oracle_half_to_float.argtypes = [ctypes.c_uint16]
        lib.oracle_visible_positions.restype = ctypes.c_int64
        lib.oracle_visible_positions.argtypes = [ctypes.c_int64, ctypes.c_int32]
        lib.oracle_score.restype = None
        lib.oracle_score.argtypes = [_u16p, _f32p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                     _u16p, ctypes.c_int32, ctypes.c_int32, _i32p, ctypes.c_int32,
                                     _i32p, _i32p, _f32p, ctypes.c_int64, ctypes.c_int32]
        lib.oracle_select.restype = None
        lib.oracle_select.argtypes = [_f32p, ctypes.c_int64, ctypes.c_int32, _i32p, ctypes.c_int32,
                                      _i32p, _f32p, ctypes.c_int32]
        lib.oracle_select_bruteforce.restype = None
        lib.oracle_select_bruteforce.argtypes = [_f32p, ctypes.c_int64, ctypes.c_int32, _i32p,
                                                 ctypes.c_int32, _i32p, _f32p]
        lib.oracle_max_threads.restype = ctypes.c_int32
        lib.oracle_max_threads.argtypes = []
        _lib = lib
        return lib


def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def half_to_float(bits: int) -> float:
    """binary16 bit pattern -> float, by the format's definition."""
    return float(_load().oracle_half_to_float(int(bits) & 0xFFFF))


def visible_positions(t: int, ratio: int = 4) -> int:
    """Compressed positions visible to a query at 0-based token position t."""
    return int(_load().oracle_visible_positions(int(t), int(ratio)))


def score(q: np.ndarray, w: np.ndarray, k_cache: np.ndarray, block_table: np.ndarray,
          row_req: np.ndarray, row_visible: np.ndarray, ld: int, nthreads: int = 0) -> np.ndarray:
    """Logits [R, ld] float32 (-inf at j >= V_r).

    q: float16 [R, H, D]; w: float32 [R, H]; k_cache: float16 [num_pages, P, D];
    block_table: int32 [num_reqs, max_pages]; row_req, row_visible: int32 [R].
    """
    lib = _load()
    q = _c(q, np.float16)
    R, H, D = q.shape
    w = _c(w, np.float32).reshape(R, H)
    k_cache = _c(k_cache, np.float16)
    num_pages, P, D2 = k_cache.shape
    assert D2 == D
    bt = _c(block_table, np.int32)
    if bt.ndim == 1:
        bt = bt.reshape(1, -1)
    rr = _c(row_req, np.int32)
    rv = _c(row_visible, np.int32)
    out = np.empty((R, int(ld)), dtype=np.float32)
    lib.oracle_score(_ptr(q.view(np.uint16), ctypes.c_uint16), _ptr(w, ctypes.c_float),
                     R, H, D, _ptr(k_cache.view(np.uint16), ctypes.c_uint16), num_pages, P,
                     _ptr(bt, ctypes.c_int32), bt.shape[1], _ptr(rr, ctypes.c_int32),
                     _ptr(rv, ctypes.c_int32), _ptr(out, ctypes.c_float), int(ld), int(nthreads))
    return out


def select(logits: np.ndarray, row_visible: np.ndarray, k: int, nthreads: int = 0):
    """Exact top-k by (score desc, index asc); returns (idx int32 [R,k], val float32 [R,k])."""
    lib = _load()
    lg = _c(logits, np.float32)
    R, ld = lg.shape
    rv = _c(row_visible, np.int32)
    idx = np.empty((R, int(k)), dtype=np.int32)
    val = np.empty((R, int(k)), dtype=np.float32)
    lib.oracle_select(_ptr(lg, ctypes.c_float), ld, R, _ptr(rv, ctypes.c_int32), int(k),
                      _ptr(idx, ctypes.c_int32), _ptr(val, ctypes.c_float), int(nthreads))
    return idx, val


def select_bruteforce(logits: np.ndarray, row_visible: np.ndarray, k: int):
    """Repeated-argmax top-k (tiny inputs only); same output convention as select()."""
    lib = _load()
    lg = _c(logits, np.float32)
    R, ld = lg.shape
    rv = _c(row_visible, np.int32)
    idx = np.empty((R, int(k)), dtype=np.int32)
    val = np.empty((R, int(k)), dtype=np.float32)
    lib.oracle_select_bruteforce(_ptr(lg, ctypes.c_float), ld, R, _ptr(rv, ctypes.c_int32),
                                 int(k), _ptr(idx, ctypes.c_int32), _ptr(val, ctypes.c_float))
    return idx, val


def select_paged_tokens(q, w, k_cache, block_table, row_req, row_visible, k, ld=None,
                        nthreads: int = 0):
    """Score then select: the whole step, as plainly as it can be written."""
    if ld is None:
        ld = max(1, int(np.max(row_visible)) if len(row_visible) else 1)
    lg = score(q, w, k_cache, block_table, row_req, row_visible, ld, nthreads)
    idx, val = select(lg, row_visible, k, nthreads)
    return idx, val, lg
