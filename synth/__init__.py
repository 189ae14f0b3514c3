"""Seeded synthetic inputs for the optimizer step (no method arithmetic here).

Both the parity oracle and the CUDA library consume the arrays this module
produces; it is the only code the two sides share.  Values are counter-based,
so any slice of a large virtual buffer can be generated on its own, on the CPU
(numpy) or on the GPU (the small CUDA kernel in ``synth_gen.cu``), with
bit-identical results.

Definition
----------
``mix64`` is the SplitMix64 output function (Steele, Lea & Flood, "Fast
splittable pseudorandom number generators", OOPSLA 2014).  For a buffer with
key ``key(seed, stream) = mix64(mix64(seed) ^ stream)`` the i-th 64-bit draw is
``mix64(key + (i + 1) * 0x9E3779B97F4A7C15)`` (all arithmetic mod 2**64).

Element j of an approximately normal buffer is the Irwin-Hall sum of twelve
24-bit uniforms: ``n = sum_{u<12} (draw(12*j + u) >> 40)``, an integer in
[0, 12 * 2**24); ``z = n - 6 * 2**24`` lies in [-6 * 2**24, 6 * 2**24) and has
unit variance in units of 2**-24.  The value is ``(z * 2**-24) * sigma`` in
binary64 (one rounding), then rounded to binary32, then (for 16-bit buffers)
rounded to fp16 or bf16, each rounding to nearest-even.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile

import numpy as np

GAMMA = 0x9E3779B97F4A7C15
M1 = 0xBF58476D1CE4E5B9
M2 = 0x94D049BB133111EB
_MASK = (1 << 64) - 1

# Kinds of output buffer.
F32 = 0
F16 = 1
BF16 = 2

_HERE = os.path.dirname(os.path.abspath(__file__))
_CU = os.path.join(_HERE, "synth_gen.cu")
_SO = os.path.join(_HERE, "libsynth.so")
_lib = None


def mix64_int(z: int) -> int:
    z &= _MASK
    z = ((z ^ (z >> 30)) * M1) & _MASK
    z = ((z ^ (z >> 27)) * M2) & _MASK
    return z ^ (z >> 31)


def key(seed: int, stream: int) -> int:
    return mix64_int(mix64_int(seed) ^ (stream & _MASK))


def _mix64_np(z: np.ndarray) -> np.ndarray:
    z = z ^ (z >> np.uint64(30))
    z = z * np.uint64(M1)
    z = z ^ (z >> np.uint64(27))
    z = z * np.uint64(M2)
    return z ^ (z >> np.uint64(31))


def normal_f64_np(seed: int, stream: int, offset: int, n: int, sigma: float,
                  chunk: int = 1 << 20) -> np.ndarray:
    """Binary64 values (z * 2**-24) * sigma for elements [offset, offset+n)."""
    k = np.uint64(key(seed, stream))
    out = np.empty(n, dtype=np.float64)
    with np.errstate(over="ignore"):
        for c0 in range(0, n, chunk):
            c1 = min(n, c0 + chunk)
            j = np.arange(offset + c0, offset + c1, dtype=np.uint64)
            acc = np.zeros(c1 - c0, dtype=np.int64)
            for u in range(12):
                ctr = j * np.uint64(12) + np.uint64(u + 1)
                d = _mix64_np(k + ctr * np.uint64(GAMMA))
                acc += (d >> np.uint64(40)).astype(np.int64)
            z = acc - 6 * (1 << 24)
            out[c0:c1] = (z.astype(np.float64) * 2.0 ** -24) * sigma
    return out


def _f32_to_bf16_bits(x32: np.ndarray) -> np.ndarray:
    import torch
    return (torch.from_numpy(np.ascontiguousarray(x32)).to(torch.bfloat16)
            .view(torch.int16).numpy().view(np.uint16))


def normal_np(seed: int, stream: int, offset: int, n: int, sigma: float,
              kind: int) -> np.ndarray:
    """CPU generator: float32 array (kind F32) or uint16 bit patterns."""
    x32 = normal_f64_np(seed, stream, offset, n, sigma).astype(np.float32)
    if kind == F32:
        return x32
    if kind == F16:
        with np.errstate(over="ignore"):
            return x32.astype(np.float16).view(np.uint16)
    if kind == BF16:
        return _f32_to_bf16_bits(x32)
    raise ValueError(kind)


# ---------------------------------------------------------------- GPU side

def build(force: bool = False, nvcc: str = "nvcc") -> str:
    if (not force and os.path.exists(_SO)
            and os.path.getmtime(_SO) >= os.path.getmtime(_CU)):
        return _SO
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_HERE)
    os.close(fd)
    cmd = [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3",
           "-lineinfo", "-Xcompiler", "-fPIC", "-shared", "-o", tmp, _CU]
    try:
        subprocess.run(cmd, check=True, capture_output=True, text=True)
        os.replace(tmp, _SO)
    except subprocess.CalledProcessError as e:
        os.unlink(tmp)
        raise RuntimeError("synth build failed:\n" + e.stderr) from e
    return _SO


def _gpu_lib():
    global _lib
    if _lib is None:
        if not os.path.exists(_SO):
            raise RuntimeError("synth/libsynth.so is not built; run build()")
        L = ctypes.CDLL(_SO)
        L.synth_normal.argtypes = [ctypes.c_uint64, ctypes.c_int64, ctypes.c_int64,
                                   ctypes.c_double, ctypes.c_int32,
                                   ctypes.c_void_p, ctypes.c_void_p]
        L.synth_normal.restype = ctypes.c_int
        _lib = L
    return _lib


def fill_gpu(t, seed: int, stream: int, offset: int, sigma: float, kind: int,
             cuda_stream=None) -> None:
    """Fill the contiguous CUDA tensor ``t`` with elements [offset, offset+numel)."""
    import torch
    assert t.is_cuda and t.is_contiguous()
    expect = {F32: torch.float32, F16: torch.float16, BF16: torch.bfloat16}[kind]
    assert t.dtype == expect, (t.dtype, kind)
    if cuda_stream is None:
        cuda_stream = torch.cuda.current_stream(t.device).cuda_stream
    rc = _gpu_lib().synth_normal(key(seed, stream), offset, t.numel(), sigma,
                                 kind, ctypes.c_void_p(t.data_ptr()),
                                 ctypes.c_void_p(cuda_stream))
    if rc != 0:
        raise RuntimeError(f"synth_normal failed with CUDA error {rc}")


def normal_torch(seed: int, stream: int, n: int, sigma: float, kind: int,
                 device="cpu", offset: int = 0):
    """A torch tensor of the synthetic values on ``device``."""
    import torch
    dt = {F32: torch.float32, F16: torch.float16, BF16: torch.bfloat16}[kind]
    if str(device).startswith("cuda"):
        t = torch.empty(n, dtype=dt, device=device)
        if n:
            fill_gpu(t, seed, stream, offset, sigma, kind)
        return t
    a = normal_np(seed, stream, offset, n, sigma, kind)
    if kind == F32:
        return torch.from_numpy(a)
    return torch.from_numpy(a.view(np.int16)).view(dt)


def seeded_indices(seed: int, stream: int, count: int, low: int, high: int):
    """`count` integers in [low, high) from the same counter generator."""
    k = key(seed, stream)
    out = []
    for i in range(count):
        d = mix64_int(k + (i + 1) * GAMMA)
        out.append(low + d % (high - low))
    return out
