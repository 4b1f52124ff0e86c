"""Seeded synthetic inputs shared by the CUDA path's harness and by the oracle.

Nothing here computes any part of a training step. The module turns
(seed, stream, index) into initial weights and token/label ids with a
counter-based SplitMix64 generator (definition in ``gen.c``), so that the
product and the oracle read bit-identical inputs without sharing code.

Workload recipe (the benchmark configurations' synthetic inputs):
  * weight matrices and the embedding: N(0, 0.02^2), stored as bfloat16;
  * RMSNorm gains: 1.0;
  * Adam moments and gradients: zero;
  * tokens and labels: i.i.d. uniform in [0, vocab).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

WEIGHT_SEED = 1234
TOKEN_SEED = 5678
LABEL_SEED = 9012
INIT_STD = 0.02

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_LIB = os.path.join(_HERE, "_libsynth.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile ``gen.c`` into ``_libsynth.so`` (gcc, OpenMP, no fast-math, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(
            ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
        )
        os.replace(tmp, _LIB)
    return _LIB


def _get():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        u64, i64, u32, dbl, vp = (ctypes.c_uint64, ctypes.c_int64, ctypes.c_uint32,
                                  ctypes.c_double, ctypes.c_void_p)
        lib.synth_normal_bf16.argtypes = [u64, u64, dbl, vp, i64]
        lib.synth_const_bf16.argtypes = [dbl, vp, i64]
        lib.synth_uniform_i32.argtypes = [u64, u64, u32, vp, i64]
        lib.synth_zero.argtypes = [vp, i64]
        for f in (lib.synth_normal_bf16, lib.synth_const_bf16, lib.synth_uniform_i32, lib.synth_zero):
            f.restype = None
        _lib = lib
    return _lib


def weight_stream(block: int, tensor: int) -> int:
    """Stream id of tensor ``tensor`` of block ``block`` (block 0 = embedding)."""
    return block * 64 + tensor


def normal_bf16_into(ptr: int, n: int, seed: int, stream: int, std: float = INIT_STD) -> None:
    _get().synth_normal_bf16(seed, stream, std, ctypes.c_void_p(ptr), n)


def const_bf16_into(ptr: int, n: int, value: float) -> None:
    _get().synth_const_bf16(value, ctypes.c_void_p(ptr), n)


def zero_into(ptr: int, nbytes: int) -> None:
    _get().synth_zero(ctypes.c_void_p(ptr), nbytes)


def normal_bf16(n: int, seed: int, stream: int, std: float = INIT_STD) -> np.ndarray:
    """bfloat16 bit patterns (uint16) of N(0, std^2) values."""
    out = np.empty(n, dtype=np.uint16)
    normal_bf16_into(out.ctypes.data, n, seed, stream, std)
    return out


def const_bf16(n: int, value: float) -> np.ndarray:
    out = np.empty(n, dtype=np.uint16)
    const_bf16_into(out.ctypes.data, n, value)
    return out


def uniform_i32(n: int, vocab: int, seed: int, stream: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.int32)
    _get().synth_uniform_i32(seed, stream, vocab, ctypes.c_void_p(out.ctypes.data), n)
    return out


def tokens(n: int, vocab: int, seed: int = TOKEN_SEED) -> np.ndarray:
    return uniform_i32(n, vocab, seed)


def labels(n: int, vocab: int, seed: int = LABEL_SEED) -> np.ndarray:
    return uniform_i32(n, vocab, seed)
