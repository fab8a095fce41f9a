"""The decode-step workloads: shapes and the recipe of their synthetic inputs.

Shapes follow the pages' 8B/GQA-8 example ("5. Core modules", section 5.4: 32
layers, 8 KV heads, head_dim 128, FP16 KV = 131072 B/token) with the rest of a
Llama-3-8B-shaped decoder, plus a one-layer tiny shape for fast parity.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

KV_FP16, KV_INT8, KV_INT4 = 0, 1, 2


@dataclass(frozen=True)
class Shape:
    name: str
    n_layers: int
    hidden: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    vocab: int
    rms_eps: float = 1e-5
    rope_base: float = 10000.0

    @property
    def qkv_rows(self) -> int:
        return (self.n_heads + 2 * self.n_kv_heads) * self.head_dim


TINY = Shape("tiny-1L-d256", n_layers=1, hidden=256, n_heads=4, n_kv_heads=2, head_dim=64, ffn=688, vocab=0,
             rope_base=10000.0)
LLAMA8B = Shape("llama3-8b-shape", n_layers=32, hidden=4096, n_heads=32, n_kv_heads=8, head_dim=128, ffn=14336,
                vocab=128256, rope_base=500000.0)


def shrink(shape: Shape, n_layers: int | None = None, vocab: int | None = None) -> Shape:
    """The same per-layer shape with fewer layers and/or a smaller vocabulary (for sampled parity)."""
    return replace(shape, name=shape.name + f"-L{n_layers}-V{vocab}",
                   n_layers=shape.n_layers if n_layers is None else n_layers,
                   vocab=shape.vocab if vocab is None else vocab)


@dataclass(frozen=True)
class Workload:
    name: str
    shape: Shape
    kv_dtype: int
    batch: int
    prior: tuple  # prior context length of each session (decode) or of the one session (prefill)
    chunk: int = 0  # >0: a prefill chunk of this many tokens instead of one decode token per session
    scattered_pool: bool = False


TINY_DECODE = Workload("tiny-decode-b1-ctx128-fp16", TINY, KV_FP16, 1, (128,))
DECODE_8B = Workload("8b-decode-b1-ctx2048-fp16", LLAMA8B, KV_FP16, 1, (2048,))
LONG_FP16 = Workload("8b-decode-b1-ctx19431-fp16", LLAMA8B, KV_FP16, 1, (19431,))
LONG_INT8 = Workload("8b-decode-b1-ctx38863-int8", LLAMA8B, KV_INT8, 1, (38863,))
LONG_INT4 = Workload("8b-decode-b1-ctx77726-int4", LLAMA8B, KV_INT4, 1, (77726,))
PREFILL_8B = Workload("8b-prefill-512-on-800-fp16", LLAMA8B, KV_FP16, 1, (800,), chunk=512)


def agent_batch(seed: int, n_sessions: int = 16) -> Workload:
    from . import agent_contexts
    ctx = tuple(int(c) for c in agent_contexts(seed, n_sessions))
    return Workload(f"8b-decode-b{n_sessions}-agent-fp16-seed{seed}", LLAMA8B, KV_FP16, n_sessions, ctx,
                    scattered_pool=True)
