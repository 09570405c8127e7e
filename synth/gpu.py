"""Device side of the seeded input generator (``synth_gpu.cu``).

Fills torch CUDA tensors with the same values ``synth.normal_f32`` produces on
the host, so large inputs (tens of GB of expert weights) never cross PCIe.
"""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth_gpu.cu")
_LIB = os.path.join(_HERE, "libsynth.so")
_lib = None


def build(force: bool = False) -> str:
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
        tmp = _LIB + ".tmp.%d" % os.getpid()
        subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                        "-Xcompiler", "-fPIC", "-shared", _SRC, "-o", tmp], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB):
            build()
        L = ctypes.CDLL(_LIB)
        i64 = ctypes.c_int64
        L.synth_fill_normal.argtypes = [ctypes.c_void_p, i64, i64, i64, i64, i64, i64, i64,
                                        ctypes.c_uint64, ctypes.c_uint32, ctypes.c_float,
                                        ctypes.c_int, ctypes.c_void_p]
        L.synth_fill_normal.restype = ctypes.c_int
        _lib = L
    return _lib


def fill(t, seed: int, stream_id: int, std: float, index0: int = 0, dims=None, strides=None) -> None:
    """Fill CUDA tensor ``t`` (bf16 or fp32, contiguous) with generator values.

    Element (a,b,c) of the 3-D view ``dims`` takes counter index
    ``index0 + a*s0 + b*s1 + c*s2``. The default is the identity layout."""
    import torch
    assert t.is_cuda and t.is_contiguous() and t.dtype in (torch.bfloat16, torch.float32)
    n = t.numel()
    if dims is None:
        dims, strides = (1, 1, n), (0, 0, 1)
    assert dims[0] * dims[1] * dims[2] == n
    rc = lib().synth_fill_normal(t.data_ptr(), dims[0], dims[1], dims[2], strides[0], strides[1],
                                 strides[2], index0, seed, stream_id, float(std),
                                 int(t.dtype == torch.bfloat16),
                                 torch.cuda.current_stream(t.device).cuda_stream)
    if rc != 0:
        raise RuntimeError("synth_fill_normal failed: %d" % rc)
