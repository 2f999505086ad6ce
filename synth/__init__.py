"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the CPU oracle.

This module only draws numbers; it holds none of the FSDP step's arithmetic.
The same counter-based generator is implemented twice, once here (numpy, for
any subset of positions) and once in ``synth/csrc/synth.cu`` (a fill kernel
for whole device buffers), and the two agree bit for bit, so a test can fill
a multi-GB buffer on the device and regenerate any sampled position on the
host.

Definition (per element at flat position ``i`` of a stream with 64-bit key ``K``):

* splitmix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014; the public-domain ``splitmix64`` finaliser):
  ``z_d = mix64(K + (6*i + d + 1) * GAMMA)`` for ``d = 0..5`` (mod 2**64);
* twelve 24-bit uniforms, two per draw: ``z_d >> 40`` and ``(z_d >> 16) & 0xFFFFFF``;
* Irwin-Hall: ``c = sum(u) - 6 * 2**24`` (an integer, variance 2**48, tails cut at 6 sigma);
* ``x = float32(c) * float32(sigma * 2**-24)``, both steps IEEE round-to-nearest;
* bf16 streams round ``x`` to bfloat16 with the library conversion (RNE);
* ``abs`` streams take ``|x|``;
* positions ``i >= n_valid`` (FlatParameter padding) are exactly zero.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Iterable

import numpy as np

GAMMA = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB
_MASK64 = (1 << 64) - 1

# stream kinds: what a buffer holds (part of the stream key)
KIND_MASTER = 1   # fp32 master parameters
KIND_EXP_AVG = 2  # Adam first moment m
KIND_EXP_AVG_SQ = 3  # Adam second moment v
KIND_GRAD = 4     # a rank's bf16 full gradient
KIND_SHARD = 5    # another rank's bf16 parameter shard (all-gather input)
KIND_TENSOR = 6   # an unflattened parameter tensor


def _mix64_int(z: int) -> int:
    z &= _MASK64
    z = ((z ^ (z >> 30)) * _M1) & _MASK64
    z = ((z ^ (z >> 27)) * _M2) & _MASK64
    return z ^ (z >> 31)


def stream_key(seed: int, *fields: int) -> int:
    """64-bit key of one stream, derived from the seed and integer fields."""
    k = _mix64_int(seed + GAMMA)
    for f in fields:
        k = _mix64_int(k ^ _mix64_int((int(f) + 1) * GAMMA))
    return k


def _mix64(z: np.ndarray) -> np.ndarray:
    z = z ^ (z >> np.uint64(30))
    z = z * np.uint64(_M1)
    z = z ^ (z >> np.uint64(27))
    z = z * np.uint64(_M2)
    return z ^ (z >> np.uint64(31))


def scale_of(sigma: float) -> np.float32:
    """fp32 factor that maps the Irwin-Hall integer to a draw of std ``sigma``."""
    return np.float32(sigma) * np.float32(2.0 ** -24)


def normal_f32_at(key: int, idx: np.ndarray, sigma: float, absval: bool = False,
                  n_valid: int | None = None) -> np.ndarray:
    """fp32 draws at the given flat positions (any order, any subset)."""
    idx = np.asarray(idx, dtype=np.uint64)
    out = np.empty(idx.shape, dtype=np.float32)
    flat_i = idx.reshape(-1)
    flat_o = out.reshape(-1)
    step = 1 << 20
    k = np.uint64(key)
    g = np.uint64(GAMMA)
    sc = scale_of(sigma)
    with np.errstate(over="ignore"):
        for a in range(0, flat_i.size, step):
            ii = flat_i[a:a + step]
            base = ii * np.uint64(6)
            s = np.zeros(ii.shape, dtype=np.int64)
            for d in range(6):
                z = _mix64(k + (base + np.uint64(d + 1)) * g)
                s += (z >> np.uint64(40)).astype(np.int64)
                s += ((z >> np.uint64(16)) & np.uint64(0xFFFFFF)).astype(np.int64)
            c = s - np.int64(6 << 24)
            x = c.astype(np.float32) * sc
            if absval:
                x = np.abs(x)
            if n_valid is not None:
                x[ii >= np.uint64(n_valid)] = np.float32(0.0)
            flat_o[a:a + step] = x
    return out


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bfloat16 with torch's CPU conversion; return the uint16 bits."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def normal_bf16_at(key: int, idx: np.ndarray, sigma: float, absval: bool = False,
                   n_valid: int | None = None) -> np.ndarray:
    return to_bf16_bits(normal_f32_at(key, idx, sigma, absval, n_valid))


def normal_f32(key: int, n: int, sigma: float, idx0: int = 0, absval: bool = False,
               n_valid: int | None = None) -> np.ndarray:
    """fp32 draws for the contiguous positions ``idx0 .. idx0+n-1``."""
    idx = np.arange(idx0, idx0 + n, dtype=np.uint64)
    return normal_f32_at(key, idx, sigma, absval, n_valid)


def normal_bf16(key: int, n: int, sigma: float, idx0: int = 0, absval: bool = False,
                n_valid: int | None = None) -> np.ndarray:
    return to_bf16_bits(normal_f32(key, n, sigma, idx0, absval, n_valid))


# ---------------------------------------------------------------- device side

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "_build", "libfsdp_synth.so")
_SRC = os.path.join(_HERE, "csrc", "synth.cu")
_lib = None


def build(force: bool = False) -> str:
    """Compile the device fill kernels for sm_103a into ``synth/_build``."""
    os.makedirs(os.path.dirname(_SO), exist_ok=True)
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(_SRC):
        return _SO
    nvcc = os.environ.get("NVCC", "nvcc")
    tmp = _SO + ".tmp%d" % os.getpid()
    cmd = [nvcc, "-O3", "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a",
           "-lineinfo", "-shared", "-Xcompiler", "-fPIC", "-o", tmp, _SRC]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    if _lib is None:
        if not os.path.exists(_SO):
            raise RuntimeError("synth device library not built: run synth.build()")
        lib = ctypes.CDLL(_SO)
        for name in ("synth_fill_f32", "synth_fill_bf16"):
            fn = getattr(lib, name)
            fn.restype = ctypes.c_int
            fn.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                           ctypes.c_uint64, ctypes.c_float, ctypes.c_int, ctypes.c_void_p]
        _lib = lib
    return _lib


def _stream_ptr(stream) -> int:
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def fill_(t, key: int, sigma: float, idx0: int = 0, absval: bool = False,
          n_valid: int | None = None, stream=None):
    """Fill a contiguous CUDA tensor (fp32, or bf16/int16/uint16 bits) in place.

    Element ``i`` of ``t`` receives the draw at flat position ``idx0 + i``;
    positions ``>= n_valid`` receive zero.
    """
    import torch
    assert t.is_cuda and t.is_contiguous()
    lib = _load()
    n = t.numel()
    nv = (1 << 62) if n_valid is None else int(n_valid)
    if t.dtype == torch.float32:
        fn = lib.synth_fill_f32
    elif t.dtype in (torch.bfloat16, torch.int16, torch.uint16):
        fn = lib.synth_fill_bf16
    else:
        raise TypeError("fill_: unsupported dtype %s" % t.dtype)
    rc = fn(t.data_ptr(), n, idx0, nv, key & _MASK64, float(scale_of(sigma)),
            1 if absval else 0, _stream_ptr(stream))
    if rc != 0:
        raise RuntimeError("synth fill failed (cuda error %d)" % rc)
    return t


def keys(seed: int, fields: Iterable[int]) -> int:
    return stream_key(seed, *fields)
