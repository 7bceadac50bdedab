"""CPU oracle for the ragged per-row top-K (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package. The product
library (``sparse_attention_row_gb300``) never imports, links or calls it.

The oracle itself is plain C (``topk_oracle.c``): for each row it sorts the
valid prefix by (value desc, index asc) and keeps the first ``topk`` indices,
padding with -1. This module compiles it with gcc into ``liboracle.so`` next to
the source and wraps it with ctypes. ``build(mutant=n)`` compiles a copy with a
deliberately planted bug, used by the tests that show the pins catch mistakes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "topk_oracle.c")
_LOCK = threading.Lock()
_LIBS: dict[int, ctypes.CDLL] = {}

STATUS_LENGTH_CLAMPED = 1


def lib_path(mutant: int = 0) -> str:
    name = "liboracle.so" if mutant == 0 else f"liboracle_mutant{mutant}.so"
    return os.path.join(_HERE, name)


def build(mutant: int = 0, force: bool = False) -> str:
    """Compiles the oracle (or one planted-bug variant) with gcc; returns the .so path."""
    out = lib_path(mutant)
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(_SRC):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-pthread",
           f"-DORACLE_MUTANT={int(mutant)}", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _load(mutant: int = 0) -> ctypes.CDLL:
    with _LOCK:
        if mutant not in _LIBS:
            lib = ctypes.CDLL(build(mutant))
            fn = lib.oracle_topk_ragged
            fn.restype = ctypes.c_uint
            fn.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64,
                           ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_int]
            _LIBS[mutant] = lib
        return _LIBS[mutant]


def topk_ragged(logits: np.ndarray, lengths: np.ndarray, topk: int, next_n: int = 1,
                nthreads: int | None = None, mutant: int = 0) -> tuple[np.ndarray, int]:
    """Runs the oracle on host arrays.

    logits:  float32 array of shape [num_rows, row_stride] (C-contiguous).
    lengths: int32 array of shape [num_rows] (or [num_rows // next_n, next_n]).
    Returns (indices int32 [num_rows, topk] in (value desc, index asc) order with
    -1 padding, status word; bit 0 = some length was clamped into [0, row_stride]).
    """
    x = np.ascontiguousarray(logits, dtype=np.float32)
    if x.ndim != 2:
        raise ValueError("logits must be 2-D [num_rows, row_stride]")
    ln = np.ascontiguousarray(lengths, dtype=np.int32).reshape(-1)
    num_rows, row_stride = x.shape
    if ln.shape[0] != num_rows:
        raise ValueError("one length per row is required")
    out = np.empty((num_rows, topk), dtype=np.int32)
    if nthreads is None:
        nthreads = os.cpu_count() or 1
    st = _load(mutant).oracle_topk_ragged(
        x.ctypes.data, row_stride, ln.ctypes.data, num_rows, int(next_n), int(topk),
        out.ctypes.data, int(nthreads))
    if st == 0xFFFFFFFE:
        raise ValueError("oracle rejected its arguments")
    if st & 0x80000000:
        raise MemoryError("oracle ran out of host memory")
    return out, int(st)
