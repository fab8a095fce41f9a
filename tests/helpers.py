"""Test-side helpers: build the oracle's model and KV stores from the seeded inputs."""
from __future__ import annotations

import numpy as np

import oracle
import synth
from synth.workloads import Shape

PROJ = ("wqkv", "wo", "wgu", "wdown")


def proj_shape(shape: Shape, name: str):
    D, F = shape.hidden, shape.ffn
    return {"wqkv": (shape.qkv_rows, D), "wo": (D, shape.n_heads * shape.head_dim), "wgu": (2 * F, D),
            "wdown": (D, F)}[name]


def model_cfg(shape: Shape, kv_dtype: int) -> oracle.ModelCfg:
    return oracle.ModelCfg(shape.n_layers, shape.hidden, shape.n_heads, shape.n_kv_heads, shape.head_dim,
                           shape.ffn, shape.vocab, shape.rms_eps, shape.rope_base, kv_dtype, 16)


def oracle_weights(shape: Shape, seed: int, random_gain: bool = False, layers=None) -> oracle.Weights:
    """Quantise the seeded fp32 projections with the oracle's quantiser."""
    w = oracle.Weights()
    for l in (range(shape.n_layers) if layers is None else layers):
        for name in PROJ:
            n, k = proj_shape(shape, name)
            p, sm = oracle.w4g32_quantize(synth.weight_f32(seed, l, name, n, k))
            getattr(w, name).append(p)
            getattr(w, "s" + name[1:]).append(sm)
        w.gamma1.append(synth.norm_gain_f16(seed, f"L{l}.g1", shape.hidden, random_gain))
        w.gamma2.append(synth.norm_gain_f16(seed, f"L{l}.g2", shape.hidden, random_gain))
    w.gamma_f = synth.norm_gain_f16(seed, "gf", shape.hidden, random_gain)
    if shape.vocab:
        w.lm_head = synth.lm_head_f16(seed, shape.vocab, shape.hidden)
    return w


def prior_kv(shape: Shape, seed: int, session: int, n_tok: int):
    """[L, n, Hkv, d] fp16 prior K and V of one session."""
    L, H, d = shape.n_layers, shape.n_kv_heads, shape.head_dim
    k = np.empty((L, n_tok, H, d), dtype=np.float16)
    v = np.empty((L, n_tok, H, d), dtype=np.float16)
    for l in range(L):
        k[l] = synth.prior_kv_f16(seed, session, l, "K", n_tok, H, d)
        v[l] = synth.prior_kv_f16(seed, session, l, "V", n_tok, H, d)
    return k, v


def rel_l2(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def max_abs(a, b) -> float:
    return float(np.max(np.abs(np.asarray(a, np.float64) - np.asarray(b, np.float64))))


# The tolerance of fp16 logits and hidden states against the oracle: both must hold.
TOL_MAX_ABS = 2e-2
TOL_REL_L2 = 1e-3
# Deep (32-layer) random models: the oracle's own logits move by about 2e-3 (rel-L2) when a single
# input value moves by one fp16 ulp, so there the rel-L2 bar is this factor times that measured
# sensitivity (max-abs stays 2e-2).
FLOOR_FACTOR = 1.25


def one_ulp_floor(run_oracle, x_f16, n=3):
    """Mean rel-L2 change of the oracle's output when one input element of every token row moves by one
    fp16 ulp (each row is an independent sequence, so each gets its own perturbation)."""
    base = run_oracle(x_f16)
    vals = []
    for i in range(n):
        x2 = np.array(x_f16, copy=True).reshape(-1, x_f16.shape[-1])
        rows = x2.view(np.uint16)
        rows[:, (977 * i + 101) % rows.shape[1]] += 1
        vals.append(rel_l2(run_oracle(x2.reshape(x_f16.shape)), base))
    return float(np.mean(vals)), base


def fp16_ulps(a, b):
    """Distance in fp16 steps between fp16 arrays (sign-magnitude bit patterns mapped onto one ordered line)."""
    ai = np.asarray(a, np.float16).view(np.uint16).astype(np.int64)
    bi = np.asarray(b, np.float16).view(np.uint16).astype(np.int64)
    ai = np.where(ai >= 0x8000, 0x8000 - ai, ai)
    bi = np.where(bi >= 0x8000, 0x8000 - bi, bi)
    return np.abs(ai - bi)


def device_bytes(ptr, nbytes):
    """A uint8 CUDA tensor copy of `nbytes` at device address `ptr` (read through the CUDA array interface)."""
    import torch

    class _Arr:
        __cuda_array_interface__ = {"shape": (nbytes,), "typestr": "|u1", "data": (ptr, False), "version": 3}
    return torch.as_tensor(_Arr(), device="cuda").clone()
