"""Seeded synthetic inputs shared by the oracle and the CUDA path.

This package holds no attention arithmetic: it only turns (seed, tensor tag, flat index)
into bf16 bit patterns (SplitMix64 + Box-Muller, defined in ``synth.c``) and names the
benchmark workloads' shapes. Both sides of every parity test read their inputs from here,
so the GPU receives exactly the bits the oracle computes from.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile

import numpy as np

from .configs import CONFIGS, LAYOUT_IDS, LAYOUT_NAMES, ORDER, Workload, workload  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_OUT = os.path.join(_HERE, "_build", "libsynth.so")
_lib = None

TAG_Q, TAG_K, TAG_V = 1, 2, 3


def build(force: bool = False) -> str:
    """Compile synth.c into a shared library next to it (host C only, any CPU)."""
    if not force and os.path.exists(_OUT) and os.path.getmtime(_OUT) >= os.path.getmtime(_SRC):
        return _OUT
    os.makedirs(os.path.dirname(_OUT), exist_ok=True)
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=os.path.dirname(_OUT))
    os.close(fd)
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _OUT)
    return _OUT


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        lib.synth_normal_bf16.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint64,
                                          ctypes.c_uint64, ctypes.c_double, ctypes.c_void_p]
        lib.synth_normal_bf16.restype = None
        lib.synth_normal_bf16_one.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint64,
                                              ctypes.c_double]
        lib.synth_normal_bf16_one.restype = ctypes.c_uint16
        lib.synth_splitmix64.argtypes = [ctypes.c_uint64]
        lib.synth_splitmix64.restype = ctypes.c_uint64
        _lib = lib
    return _lib


def normal_bf16(seed: int, tag: int, shape, mult: float = 1.0, out: np.ndarray | None = None) -> np.ndarray:
    """bf16 bit patterns (uint16) of N(0,1)*mult, element i of the flat tensor from (seed, tag, i)."""
    count = int(np.prod(shape))
    if out is None:
        out = np.empty(count, dtype=np.uint16)
    else:
        assert out.dtype == np.uint16 and out.size == count and out.flags.c_contiguous
    _load().synth_normal_bf16(seed, tag, 0, count, float(mult), out.ctypes.data)
    return out.reshape(shape)


def normal_bf16_at(seed: int, tag: int, index: int, mult: float = 1.0) -> int:
    """The single element with flat index ``index`` (for spot checks)."""
    return int(_load().synth_normal_bf16_one(seed, tag, index, float(mult)))


def splitmix64(x: int) -> int:
    return int(_load().synth_splitmix64(x & 0xFFFFFFFFFFFFFFFF))


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    return (bits.astype(np.uint32) << 16).view(np.float32)


def make_qkv(w: "Workload", B: int | None = None, T: int | None = None):
    """Q [B,T,h,d], K and V [B,T,n_kv,d] as bf16 bit arrays (uint16) for workload ``w``."""
    B = w.B if B is None else B
    T = w.T if T is None else T
    q = normal_bf16(w.seed, TAG_Q, (B, T, w.h, w.d))
    k = normal_bf16(w.seed, TAG_K, (B, T, w.n_kv, w.d), mult=w.k_mult)
    v = normal_bf16(w.seed, TAG_V, (B, T, w.n_kv, w.d))
    return q, k, v


def sample_rows(T: int, n_cp: int, count: int, seed: int) -> np.ndarray:
    """Sorted natural token ids for sampled-row checks: t = 0, t = T-1, the first and last
    token of each of the 2*n_cp equal natural chunks (every contiguous and zigzag chunk
    boundary), then uniform draws without replacement from ``seed`` up to ``count``."""
    m = T // (2 * n_cp)
    must = {0, T - 1}
    for c in range(2 * n_cp):
        must.update((c * m, c * m + m - 1))
    must = sorted(t for t in must if 0 <= t < T)
    rest = np.setdiff1d(np.arange(T), np.array(must))
    extra = max(0, min(count - len(must), rest.size))
    pick = np.random.default_rng(seed).choice(rest, size=extra, replace=False) if extra else np.array([], int)
    return np.sort(np.concatenate([np.array(must, dtype=np.int64), pick.astype(np.int64)]))
