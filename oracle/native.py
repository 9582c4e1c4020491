"""Loader for the oracle's C part (``cache_write.c``) — test infrastructure only.

The shared object is built with gcc into ``oracle/_build/`` on first use (or by
the package's ``build()``).  It is never linked into the CUDA library.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "cache_write.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle_cw.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle's C code (plain IEEE binary32/binary64, no contraction)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
           "-fopenmp", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            _lib = ctypes.CDLL(build())
            _declare(_lib)
    return _lib


_P = ctypes.c_void_p
_I64 = ctypes.c_int64


def _declare(L: ctypes.CDLL) -> None:
    L.oracle_e2m1_encode.restype = ctypes.c_uint8
    L.oracle_e2m1_encode.argtypes = [ctypes.c_float]
    L.oracle_e2m1_decode.restype = ctypes.c_double
    L.oracle_e2m1_decode.argtypes = [ctypes.c_uint8]
    L.oracle_e4m3_encode.restype = ctypes.c_uint8
    L.oracle_e4m3_encode.argtypes = [ctypes.c_float]
    L.oracle_e4m3_decode.restype = ctypes.c_double
    L.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
    L.oracle_fp4_group_quantize.restype = None
    L.oracle_fp4_group_quantize.argtypes = [_P, _P, _P]
    L.oracle_e4m3_encode_rows.restype = None
    L.oracle_e4m3_encode_rows.argtypes = [_P, _I64, _P]
    L.oracle_mxfp4_block_quantize.restype = None
    L.oracle_mxfp4_block_quantize.argtypes = [_P, _P, _P]
    L.oracle_mxfp4_rows.restype = None
    L.oracle_mxfp4_rows.argtypes = [_P, _I64, _P, _P]
    L.oracle_compress.restype = None
    L.oracle_compress.argtypes = [_P, _P, _P, _P, ctypes.c_int, _P]
    L.oracle_rmsnorm.restype = None
    L.oracle_rmsnorm.argtypes = [_P, _P]
    L.oracle_rope_table.restype = None
    L.oracle_rope_table.argtypes = [_I64, ctypes.c_double, _P]
    L.oracle_rope_apply.restype = None
    L.oracle_rope_apply.argtypes = [_P, _P]
    L.oracle_project.restype = None
    L.oracle_project.argtypes = [_P, _P, _P]
    L.oracle_main_entry.restype = None
    L.oracle_main_entry.argtypes = [_P, _P]
    L.oracle_compress_quantize.restype = None
    L.oracle_compress_quantize.argtypes = [_P, _I64, ctypes.c_int, _P, _P, _P, _I64,
                                           _P, _P, _P, _P]
    L.oracle_entry_stages.restype = None
    L.oracle_entry_stages.argtypes = [_P, _P, ctypes.c_int, _P, _P, _P, _P,
                                      _P, _P, _P, _P]


def ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data
