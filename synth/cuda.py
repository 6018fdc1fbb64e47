"""Device-side draws of the same seeded inputs as ``synth`` (for tensors too large to
draw on the host).  Built from synth/gen.cu by ``synth.cuda.build()``; the values are
bit-identical to the numpy definition (checked by a GPU test)."""
from __future__ import annotations

import ctypes
import os
import subprocess

from synth import STREAM_LSE, STREAM_LSE_DROP, STREAM_ROW_DROP

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB = os.path.join(_HERE, "_build", "libsynth.so")
_L = None
_CODES = {"f16": 0, "bf16": 1, "f32": 2}


def build() -> str:
    os.makedirs(os.path.dirname(LIB), exist_ok=True)
    nvcc = os.environ.get("NVCC", "nvcc")
    cmd = [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-Xcompiler", "-fPIC", "-shared",
           os.path.join(_HERE, "gen.cu"), "-o", LIB + ".tmp"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on synth/gen.cu:\n{r.stdout}\n{r.stderr}")
    os.replace(LIB + ".tmp", LIB)
    return LIB


def _lib():
    global _L
    if _L is None:
        if not os.path.exists(LIB):
            raise ImportError(f"{LIB} missing: run synth.cuda.build()")
        L = ctypes.CDLL(LIB)
        vp, ll, u, f, i = ctypes.c_void_p, ctypes.c_longlong, ctypes.c_uint, ctypes.c_float, ctypes.c_int
        L.synth_fill_normal.argtypes = [vp, ll, ll, u, u, f, f, i, vp]
        L.synth_fill_lse.argtypes = [vp, i, ll, u, u, u, u, f, f, u, u, vp]
        L.synth_fill_normal.restype = i
        L.synth_fill_lse.restype = i
        _L = L
    return _L


def fill_normal(t, seed: int, stream: int, dtype: str, start: int = 0, mu: float = 0.0, sigma: float = 1.0):
    """Fill a contiguous CUDA tensor with elements [start, start+numel) of (seed, stream)."""
    import torch
    assert t.is_cuda and t.is_contiguous()
    r = _lib().synth_fill_normal(ctypes.c_void_p(t.data_ptr()), t.numel(), start, seed, stream, mu, sigma,
                                 _CODES[dtype], ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    if r != 0:
        raise RuntimeError(f"synth_fill_normal failed with CUDA error {r}")
    return t


def fill_lse(t, seed: int, mu: float = 10.0, sigma: float = 2.0, drop: float = 0.05, row_drop: float = 0.001):
    """Fill a float32 [P, RH] CUDA tensor like synth.lse_partials."""
    import math
    import torch
    P, RH = t.shape
    r = _lib().synth_fill_lse(ctypes.c_void_p(t.data_ptr()), P, RH, seed, STREAM_LSE, STREAM_LSE_DROP,
                              STREAM_ROW_DROP, mu, sigma, int(math.floor(drop * 2**32)),
                              int(math.floor(row_drop * 2**32)),
                              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    if r != 0:
        raise RuntimeError(f"synth_fill_lse failed with CUDA error {r}")
    return t
