"""ctypes front of the seeded input generator (`synth.c`).

Holds no arithmetic of the MoE layer; see `synth.c` for the generator's
definition.  The shared library is built in-tree by `build_synth()`.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = os.path.join(_HERE, "libmoe_synth.so")
_lib = None


def build_synth(force: bool = False) -> str:
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared",
                               "-o", _LIB, _SRC, "-lm"])
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build_synth()
        lib = ctypes.CDLL(_LIB)
        u64, i64, dbl, vp = ctypes.c_uint64, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
        for fn in (lib.synth_normal_f32, lib.synth_normal_bf16):
            fn.argtypes = [u64, u64, u64, i64, i64, dbl, vp]
            fn.restype = None
        lib.synth_raw_u64.argtypes = [u64, u64, u64, i64, i64, vp]
        lib.synth_raw_u64.restype = None
        lib.synth_splitmix64.argtypes = [u64]
        lib.synth_splitmix64.restype = u64
        _lib = lib
    return _lib


def fill_normal(out: torch.Tensor, seed: int, tid: int, attempt: int, start: int,
                scale: float) -> None:
    """Write elements [start, start + out.numel()) of stream (seed, tid, attempt) into `out`."""
    if not out.is_contiguous() or out.device.type != "cpu":
        raise ValueError("fill_normal needs a contiguous host tensor")
    lib = _load()
    if out.dtype == torch.float32:
        lib.synth_normal_f32(seed, tid, attempt, start, out.numel(), scale, out.data_ptr())
    elif out.dtype == torch.bfloat16:
        lib.synth_normal_bf16(seed, tid, attempt, start, out.numel(), scale, out.data_ptr())
    else:
        raise ValueError(f"unsupported dtype {out.dtype}")


def raw_u64(seed: int, tid: int, attempt: int, start: int, count: int) -> list[int]:
    lib = _load()
    buf = (ctypes.c_uint64 * count)()
    lib.synth_raw_u64(seed, tid, attempt, start, count, ctypes.addressof(buf))
    return list(buf)


def splitmix64(z: int) -> int:
    return _load().synth_splitmix64(z)
