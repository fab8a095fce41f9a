"""Set up a library context with a workload's seeded inputs (used by the tests and the bench).

Only input generation and C-ABI calls: the weights are drawn as fp32 and
handed to mag_load_weights, which quantises them on the device; prior KV is
drawn as fp16 and handed to mag_kv_append.
"""
from __future__ import annotations

import numpy as np
import torch

import quantized_decode_step_gb300 as mag
from . import hidden_f16, lm_head_f16, norm_gain_f16, pool_order, prior_kv_f16, weight_f32
from .workloads import Shape, Workload

PROJ = (("wqkv", mag.W_QKV), ("wo", mag.W_O), ("wgu", mag.W_GATE_UP), ("wdown", mag.W_DOWN))


def proj_shape(shape: Shape, name: str):
    D, F = shape.hidden, shape.ffn
    return {"wqkv": (shape.qkv_rows, D), "wo": (D, shape.n_heads * shape.head_dim), "wgu": (2 * F, D),
            "wdown": (D, F)}[name]


def pool_blocks_for(workload: Workload, extra_tokens: int = 1) -> int:
    return sum(-(-(p + max(workload.chunk, extra_tokens)) // 16) for p in workload.prior)


def create(workload: Workload, seed: int, max_context: int | None = None, pool_blocks: int | None = None,
           flags: int = 0, stream: int | None = None, extra_tokens: int = 1) -> mag.Context:
    shape = workload.shape
    need_ctx = max(workload.prior) + max(workload.chunk, extra_tokens)
    P = pool_blocks if pool_blocks is not None else pool_blocks_for(workload, extra_tokens)
    order = pool_order(seed, P) if workload.scattered_pool else None
    cfg = mag.make_config(shape, kv_dtype=workload.kv_dtype, pool_blocks=P, max_sessions=max(workload.batch, 1),
                          max_batch=workload.batch, max_chunk=workload.chunk,
                          max_context=max_context or need_ctx, flags=flags, pool_order=order)
    if stream is None:
        stream = torch.cuda.current_stream().cuda_stream
    return mag.Context(cfg, stream)


def load_weights(ctx: mag.Context, shape: Shape, seed: int, random_gain: bool = False, keep_f32=None):
    """Draw every projection (fp32), norm gain and the LM head, and load them. If keep_f32 is a callable
    it is given (layer, name, fp32 numpy array) before upload (the tests quantise the same array with the
    oracle)."""
    for l in range(shape.n_layers):
        for name, tid in PROJ:
            n, k = proj_shape(shape, name)
            w = weight_f32(seed, l, name, n, k)
            if keep_f32 is not None:
                keep_f32(l, name, w)
            t = torch.from_numpy(w).cuda()
            ctx.load_weights(tid, l, t, mag.FMT_F32_DENSE, t.numel() * 4)
            torch.cuda.current_stream().synchronize()
            del t
        for tag, tid in ((f"L{l}.g1", mag.NORM_ATTN), (f"L{l}.g2", mag.NORM_FFN)):
            g = torch.from_numpy(norm_gain_f16(seed, tag, shape.hidden, random_gain)).cuda()
            ctx.load_weights(tid, l, g, mag.FMT_F16, g.numel() * 2)
            torch.cuda.current_stream().synchronize()
    g = torch.from_numpy(norm_gain_f16(seed, "gf", shape.hidden, random_gain)).cuda()
    ctx.load_weights(mag.NORM_FINAL, 0, g, mag.FMT_F16, g.numel() * 2)
    if shape.vocab:
        lm = torch.from_numpy(lm_head_f16(seed, shape.vocab, shape.hidden)).cuda()
        ctx.load_weights(mag.LM_HEAD, 0, lm, mag.FMT_F16, lm.numel() * 2)
        torch.cuda.current_stream().synchronize()
        del lm
    torch.cuda.current_stream().synchronize()


def append_prior(ctx: mag.Context, sid: int, shape: Shape, seed: int, session_index: int, n_tok: int,
                 chunk: int = 4096, keep=None):
    """Append a session's seeded prior K/V ([L][n][Hkv][d] fp16) in token chunks."""
    L, H, d = shape.n_layers, shape.n_kv_heads, shape.head_dim
    for t0 in range(0, n_tok, chunk):
        n = min(chunk, n_tok - t0)
        k = np.empty((L, n, H, d), dtype=np.float16)
        v = np.empty((L, n, H, d), dtype=np.float16)
        for l in range(L):
            k[l] = prior_kv_f16(seed, session_index, l, "K", n, H, d, tok0=t0)
            v[l] = prior_kv_f16(seed, session_index, l, "V", n, H, d, tok0=t0)
        if keep is not None:
            keep(k, v)
        kt, vt = torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda()
        ctx.kv_append(sid, n, kt, vt)
        torch.cuda.current_stream().synchronize()
        del kt, vt


def setup(workload: Workload, seed: int, **kw):
    """Context with weights and every session's prior KV; returns (ctx, session ids)."""
    ctx = create(workload, seed, **{k: v for k, v in kw.items() if k in ("max_context", "pool_blocks", "flags",
                                                                        "stream", "extra_tokens")})
    load_weights(ctx, workload.shape, seed, kw.get("random_gain", False))
    sids = []
    for i, p in enumerate(workload.prior):
        sid = ctx.session_open()
        append_prior(ctx, sid, workload.shape, seed, i, p)
        sids.append(sid)
    return ctx, sids


def step_inputs(workload: Workload, seed: int, step: int = 0) -> np.ndarray:
    """fp16 hidden inputs of one decode step: [batch, D] (or [chunk, D] for prefill)."""
    n = workload.chunk if workload.chunk else workload.batch
    return hidden_f16(seed, n, workload.shape.hidden, tag=f"x.step{step}")
