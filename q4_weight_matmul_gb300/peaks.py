"""Tensor-core rate probes (libq4k_peaks.so) used by the benchmark as the
prefill GEMM's roofline denominators: the dense int8 rate of mma.sync
m16n8k32 s8 and the dense fp16 rate of tcgen05.mma kind::f16."""
from __future__ import annotations

import ctypes
import os

from .build import PEAKS_LIB, build

_lib = None


def _load():
    global _lib
    if _lib is None:
        if not os.path.exists(PEAKS_LIB):
            build()
        lib = ctypes.CDLL(PEAKS_LIB)
        for name in ("q4kp_mma_s8_tops", "q4kp_tc_f16_tflops"):
            fn = getattr(lib, name)
            fn.restype = ctypes.c_int
            fn.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_double)]
        _lib = lib
    return _lib


def mma_s8_tops(iters: int = 4000) -> float:
    """Dense int8 TOPS of mma.sync m16n8k32 s8 on the current device."""
    out = ctypes.c_double()
    st = _load().q4kp_mma_s8_tops(iters, ctypes.byref(out))
    if st != 0:
        raise RuntimeError(f"q4kp_mma_s8_tops failed with status {st}")
    return out.value


def tc_f16_tflops(groups: int = 256) -> float:
    """Dense fp16 TFLOP/s of tcgen05.mma kind::f16 (M=128, N=256) on the current device."""
    out = ctypes.c_double()
    st = _load().q4kp_tc_f16_tflops(groups, ctypes.byref(out))
    if st != 0:
        raise RuntimeError(f"q4kp_tc_f16_tflops failed with status {st}")
    return out.value
