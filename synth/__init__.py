"""Seeded synthetic inputs for the decode step (shared by tests and bench).

This module holds no arithmetic of the decode step. It draws reproducible
random numbers (counter-based splitmix64 keyed by a seed and a tag, normals by
Box-Muller, see synth.c) and lays them out in the shapes the workloads use:

* weights  N(0, 0.02) drawn in double, rounded to fp32 (quantised later by
  whoever consumes them); the LM head and norm gains are fp16;
* prior KV N(0, 1) rounded to fp16, laid out [L][n][Hkv][d];
* hidden inputs N(0, 1) rounded to fp16;
* agent-batch contexts log-uniform on [20, 2048];
* a seeded Fisher-Yates order of the KV block pool.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = os.path.join(_HERE, "libsynth.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile libsynth.so beside its source (gcc, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB)
            u64, i64, d, cp, vp = ctypes.c_uint64, ctypes.c_int64, ctypes.c_double, ctypes.c_char_p, ctypes.c_void_p
            L.synth_key.argtypes = [u64, cp]
            L.synth_key.restype = u64
            L.synth_draw.argtypes = [u64, u64]
            L.synth_draw.restype = u64
            L.synth_uniform_f64.argtypes = [u64, cp, i64, vp]
            L.synth_u64.argtypes = [u64, cp, i64, vp]
            for f in (L.synth_normal_f64, L.synth_normal_f32, L.synth_normal_f16):
                f.argtypes = [u64, cp, i64, i64, d, d, vp]
            L.synth_uniform_f32.argtypes = [u64, cp, i64, d, d, vp]
            _lib = L
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def normal(seed: int, tag: str, shape, std: float = 1.0, mean: float = 0.0, dtype=np.float32, offset: int = 0,
           out: np.ndarray | None = None) -> np.ndarray:
    """N(mean, std^2) in `dtype` (float64, float32 or float16), element i of stream (seed, tag) at offset+i."""
    n = int(np.prod(shape)) if not isinstance(shape, int) else shape
    dtype = np.dtype(dtype)
    if out is None:
        out = np.empty(shape, dtype=dtype)
    assert out.dtype == dtype and out.size == n
    fn = {np.dtype(np.float64): lib().synth_normal_f64, np.dtype(np.float32): lib().synth_normal_f32,
          np.dtype(np.float16): lib().synth_normal_f16}[dtype]
    fn(seed, tag.encode(), offset, n, float(mean), float(std), _ptr(out))
    return out


def uniform(seed: int, tag: str, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    lib().synth_uniform_f64(seed, tag.encode(), n, _ptr(out))
    return out


def uniform_f32(seed: int, tag: str, shape, lo: float, hi: float) -> np.ndarray:
    out = np.empty(shape, dtype=np.float32)
    lib().synth_uniform_f32(seed, tag.encode(), out.size, float(lo), float(hi), _ptr(out))
    return out


def u64(seed: int, tag: str, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.uint64)
    lib().synth_u64(seed, tag.encode(), n, _ptr(out))
    return out


# ----------------------------------------------------------------------------- workload recipes

WEIGHT_STD = 0.02


def weight_tag(layer: int, name: str) -> str:
    return f"L{layer}.{name}"


def weight_f32(seed: int, layer: int, name: str, n_rows: int, n_cols: int) -> np.ndarray:
    """A projection's dense weights [n_rows, n_cols], N(0, 0.02) rounded to fp32."""
    return normal(seed, weight_tag(layer, name), (n_rows, n_cols), std=WEIGHT_STD, dtype=np.float32)


def lm_head_f16(seed: int, vocab: int, hidden: int, row0: int = 0, n_rows: int | None = None) -> np.ndarray:
    """Rows [row0, row0+n_rows) of the fp16 LM head, N(0, 0.02)."""
    n_rows = vocab - row0 if n_rows is None else n_rows
    return normal(seed, "lm_head", (n_rows, hidden), std=WEIGHT_STD, dtype=np.float16, offset=row0 * hidden)


def norm_gain_f16(seed: int, tag: str, n: int, random_gain: bool = False) -> np.ndarray:
    """RMSNorm gain: ones (a freshly initialised norm) or, to show the gain is applied, U(0.5, 1.5)."""
    if not random_gain:
        return np.ones(n, dtype=np.float16)
    return uniform_f32(seed, "gain." + tag, n, 0.5, 1.5).astype(np.float16)


def hidden_f16(seed: int, n_tok: int, hidden: int, tag: str = "x") -> np.ndarray:
    return normal(seed, tag, (n_tok, hidden), std=1.0, dtype=np.float16)


def prior_kv_f16(seed: int, session: int, layer: int, which: str, n_tok: int, n_kv_heads: int, head_dim: int,
                 tok0: int = 0) -> np.ndarray:
    """Prior (already rotated) K or V of one session and layer: [n_tok, Hkv, d] fp16, N(0, 1)."""
    tag = f"kv.S{session}.L{layer}.{which}"
    per_tok = n_kv_heads * head_dim
    return normal(seed, tag, (n_tok, n_kv_heads, head_dim), std=1.0, dtype=np.float16, offset=tok0 * per_tok)


def agent_contexts(seed: int, n_sessions: int, lo: int = 20, hi: int = 2048) -> np.ndarray:
    """Per-session prior lengths, log-uniform on [lo, hi]: round(exp(ln lo + u (ln hi - ln lo)))."""
    u = uniform(seed, "ctx", n_sessions)
    p = np.array([int(round(math.exp(math.log(lo) + x * (math.log(hi) - math.log(lo))))) for x in u], dtype=np.int64)
    return np.clip(p, lo, hi)


def pool_order(seed: int, n_blocks: int) -> np.ndarray:
    """A seeded Fisher-Yates shuffle of block ids 0..n_blocks-1 (draw i -> j = u64 % (i+1), i from n-1 down)."""
    order = np.arange(n_blocks, dtype=np.int32)
    r = u64(seed, "pool", n_blocks)
    for k, i in enumerate(range(n_blocks - 1, 0, -1)):
        j = int(r[k] % np.uint64(i + 1))
        order[i], order[j] = order[j], order[i]
    return order
