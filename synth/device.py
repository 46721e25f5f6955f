"""ctypes front end of the device twin of the input generator (synth.cu)."""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

from . import weight_scale

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.cu")
_OUT = os.path.join(_HERE, "_build", "libcssynth.so")
_lock = threading.Lock()
_lib = None

NVCC_ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def build(force: bool = False) -> str:
    os.makedirs(os.path.dirname(_OUT), exist_ok=True)
    if not force and os.path.exists(_OUT) and os.path.getmtime(_OUT) >= os.path.getmtime(_SRC):
        return _OUT
    tmp = _OUT + f".tmp{os.getpid()}"
    cmd = ["nvcc", *NVCC_ARCH, "-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-shared",
           "-cudart", "shared", _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _OUT)
    return _OUT


def lib():
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_OUT):
                raise RuntimeError(f"{_OUT} is missing: build it with synth.device.build()")
            L = C.CDLL(_OUT)
            L.synth_fill_normal.argtypes = [C.c_void_p, C.c_int, C.c_longlong, C.c_longlong,
                                            C.c_longlong, C.c_ulonglong, C.c_ulonglong, C.c_float,
                                            C.c_void_p]
            L.synth_fill_normal.restype = C.c_int
            L.synth_stream_key.argtypes = [C.c_ulonglong, C.c_ulonglong]
            L.synth_stream_key.restype = C.c_ulonglong
            _lib = L
    return _lib


def fill_normal(t, seed: int, tid: int, std: float, cols: int | None = None, dtype: int | None = None,
                stream=None) -> None:
    """Fill a CUDA tensor [rows, ld] in place (columns >= cols are zero)."""
    import torch
    rows, ld = t.shape
    cols = ld if cols is None else cols
    if dtype is None:
        dtype = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}[t.dtype]
    s = stream if stream is not None else torch.cuda.current_stream().cuda_stream
    rc = lib().synth_fill_normal(t.data_ptr(), dtype, rows, cols, ld, seed, tid,
                                 float(weight_scale(std)), s)
    if rc != 0:
        raise RuntimeError(f"synth_fill_normal failed ({rc})")
