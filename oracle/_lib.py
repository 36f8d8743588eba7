"""Loader and build step for the oracle's C part (``formats.c`` -> ``liboracle.so``).

The oracle is TEST INFRASTRUCTURE: only the tests, ``__graft_entry__.smoke()``
and bench.py's CPU-baseline leg may load it.  It shares no code with the CUDA
path.  Building the checker is not using it: ``__graft_entry__.build()`` calls
:func:`build` so the library exists on a fresh machine.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "formats.c")
LIB = os.path.join(HERE, "liboracle.so")


def build(force: bool = False) -> str:
    """Compile formats.c with gcc (IEEE arithmetic, no FMA contraction, OpenMP)."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
           "-fopenmp", "-std=c11", SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


_lib = None

_i64 = ctypes.c_int64
_p = ctypes.c_void_p


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(LIB)
        sig = {
            "orc_bf16_to_double": (ctypes.c_double, [ctypes.c_uint16]),
            "orc_bf16_from_double": (ctypes.c_uint16, [ctypes.c_double]),
            "orc_bf16_from_double_array": (None, [_p, _i64, _p]),
            "orc_bf16_to_double_array": (None, [_p, _i64, _p]),
            "orc_e4m3_decode": (ctypes.c_double, [ctypes.c_uint8]),
            "orc_e4m3_encode": (ctypes.c_uint8, [ctypes.c_double]),
            "orc_e2m1_decode": (ctypes.c_double, [ctypes.c_uint8]),
            "orc_e2m1_encode": (ctypes.c_uint8, [ctypes.c_double]),
            "orc_mxfp8_scale_exponent": (ctypes.c_int, [ctypes.c_double]),
            "orc_mxfp8_quantize_rows": (None, [_p, _i64, _i64, _p, _p]),
            "orc_mxfp8_dequant_rows": (None, [_p, _p, _i64, _i64, _p]),
            "orc_nvfp4_global_scale": (ctypes.c_float, [ctypes.c_float]),
            "orc_nvfp4_quantize_block": (None, [_p, ctypes.c_float, _p, _p]),
            "orc_nvfp4_quantize_rows": (None, [_p, _i64, _i64, ctypes.c_float, _p, _p]),
            "orc_nvfp4_dequant_rows": (None, [_p, _p, _i64, _i64, ctypes.c_float, _p]),
            "orc_rht16": (None, [_p, ctypes.c_uint32, _p]),
            "orc_group_hadamard_amax": (None, [_p, _i64, _i64, _p, ctypes.c_int, ctypes.c_uint32, _p, _p]),
            "orc_group_quantize_col": (None, [_p, _i64, _i64, _p, ctypes.c_int, ctypes.c_int,
                                              ctypes.c_uint32, _p, _p, _p]),
            "orc_amax_bf16": (ctypes.c_float, [_p, _i64]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def ptr(a) -> int:
    """Address of a C-contiguous numpy array."""
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data
