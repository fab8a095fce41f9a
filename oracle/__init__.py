"""Oracle for the quantized decode step -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package. The product library never loads it and shares
no code with it. The arithmetic lives in ``oracle.c`` (plain C, built with
``-ffp-contract=off``); this module builds it, loads it with ctypes and adds
the block-pool allocator model, which is host bookkeeping only.

Pages, cited by title and section:
  [Magnitude] "Magnitude: on-device AI-agent inference engine" (0539edu.com)
  [Core]      "5. Core modules: format, runtime, scheduling, memory and routing"
  [TFLite]    "TFLite memory planner" (pwwt.cn)
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_HDR = os.path.join(_HERE, "oracle.h")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

KV_FP16, KV_INT8, KV_INT4 = 0, 1, 2


def build(force: bool = False) -> str:
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < newest:
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


class Cfg(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int), ("hidden", ctypes.c_int), ("n_heads", ctypes.c_int),
                ("n_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int), ("ffn", ctypes.c_int),
                ("vocab", ctypes.c_int), ("rms_eps", ctypes.c_float), ("rope_base", ctypes.c_float),
                ("kv_dtype", ctypes.c_int), ("block_tokens", ctypes.c_int)]


_PP = ctypes.POINTER(ctypes.c_void_p)


class _Weights(ctypes.Structure):
    _fields_ = [(n, _PP) for n in ("wqkv", "sqkv", "wo", "so", "wgu", "sgu", "wdown", "sdown", "gamma1", "gamma2")] + \
               [("gamma_f", ctypes.c_void_p), ("lm_head", ctypes.c_void_p)]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB)
            vp, i64, i32, f32, f64 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_double
            sig = {
                "orc_set_threads": ([i32], i32),
                "orc_f64_to_f16": ([f64], ctypes.c_uint16),
                "orc_f32_to_f16": ([f32], ctypes.c_uint16),
                "orc_f16_to_f32": ([ctypes.c_uint16], f32),
                "orc_f32_to_f16_array": ([vp, i64, vp], None),
                "orc_w4g32_quantize": ([vp, i64, i64, vp, vp], None),
                "orc_w4g32_dequant": ([vp, vp, i64, i64, vp], None),
                "orc_w4_gemv": ([vp, vp, i64, i64, i32, vp, vp], None),
                "orc_w4_gemv_folded": ([vp, vp, i64, i64, vp, vp], None),
                "orc_kv_quant_int8": ([vp, i32, i32, vp, vp], None),
                "orc_kv_quant_int4": ([vp, i32, i32, vp, vp], None),
                "orc_kv_block_bytes": ([i32, i32, i32, i32], i64),
                "orc_kv_offset": ([i32, i32, i32, i32, i64, i32, i64, i32, i32, i32], i64),
                "orc_kv_bytes_per_token": ([i32, i32, i32, f64], i64),
                "orc_kv_max_context": ([f64, f64, f64, f64], i64),
                "orc_arena_plan": ([i32, vp, vp, vp, i64, i32, vp], i64),
                "orc_rmsnorm": ([vp, vp, i32, f32, vp], None),
                "orc_rope_table": ([i32, i32, f32, vp, vp], None),
                "orc_rope_apply": ([vp, i32, vp, vp, vp], None),
                "orc_kv_create": ([ctypes.POINTER(Cfg), i32], vp),
                "orc_kv_destroy": ([vp], None),
                "orc_kv_len": ([vp], i32),
                "orc_kv_truncate": ([vp, i32], None),
                "orc_kv_commit": ([vp, i32], i32),
                "orc_kv_append": ([vp, i32, vp, vp], i32),
                "orc_kv_read": ([vp, i32, i32, i32, i32, vp], None),
                "orc_kv_stored": ([vp, i32, i32, i32, i32, vp, vp], i64),
                "orc_attention": ([ctypes.POINTER(Cfg), vp, i32, i32, vp, i32, vp], None),
                "orc_forward": ([ctypes.POINTER(Cfg), ctypes.POINTER(_Weights), i32, vp, vp, vp, vp, vp, i32, vp], i32),
                "orc_layer": ([ctypes.POINTER(Cfg), ctypes.POINTER(_Weights), i32, i32, vp, vp, vp, vp, vp, i32, vp],
                              i32),
                "orc_output": ([ctypes.POINTER(Cfg), ctypes.POINTER(_Weights), vp, vp], None),
            }
            for name, (args, res) in sig.items():
                fn = getattr(L, name)
                fn.argtypes = args
                fn.restype = res
            _lib = L
    return _lib


def _p(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


# ---------------------------------------------------------------------------- fp16

def set_threads(n: int) -> int:
    """Threads of the oracle's parallel loops (n < 1: every core); returns the count in use."""
    return int(lib().orc_set_threads(int(n)))


def f64_to_f16_bits(x: float) -> int:
    return int(lib().orc_f64_to_f16(float(x)))


def f32_to_f16(x) -> np.ndarray:
    """fp32 -> fp16 (as np.float16), the oracle's own round-to-nearest-even."""
    x = _c(x, np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    lib().orc_f32_to_f16_array(_p(x), x.size, _p(out))
    return out.view(np.float16)


# ---------------------------------------------------------------------------- 4-bit weights

def w4g32_quantize(w):
    """fp32 [N, K] -> (packed u8 [N, 16*G], scale/min fp16 [N, G, 2]) with G = ceil(K/32) groups."""
    w = _c(w, np.float32)
    n, k = w.shape
    g = -(-k // 32)
    packed = np.empty((n, 16 * g), dtype=np.uint8)
    sm = np.empty((n, g, 2), dtype=np.uint16)
    lib().orc_w4g32_quantize(_p(w), n, k, _p(packed), _p(sm))
    return packed, sm.view(np.float16)


def w4g32_dequant(packed, sm, n_cols=None):
    packed = _c(packed, np.uint8)
    sm = _sm16(sm)
    n, k2 = packed.shape
    k = 2 * k2 if n_cols is None else n_cols
    out = np.empty((n, k), dtype=np.float32)
    lib().orc_w4g32_dequant(_p(packed), _p(sm), n, k, _p(out))
    return out


def _sm16(sm):
    sm = np.asarray(sm)
    return _c(sm.view(np.uint16) if sm.dtype == np.float16 else sm, np.uint16)


def w4_gemv(packed, sm, x_f16):
    """y[T, N] (float64) = x[T, K] . dequant(W)[N, K]^T (K taken from x)."""
    packed = _c(packed, np.uint8)
    sm = _sm16(sm)
    x = _c(np.atleast_2d(x_f16), np.float16)
    n = packed.shape[0]
    t, k = x.shape
    assert packed.shape[1] == 16 * (-(-k // 32))
    y = np.empty((t, n), dtype=np.float64)
    lib().orc_w4_gemv(_p(packed), _p(sm), n, k, t, _p(x.view(np.uint16)), _p(y))
    return y


def w4_gemv_folded(packed, sm, x_f16):
    packed = _c(packed, np.uint8)
    sm = _sm16(sm)
    x = _c(x_f16, np.float16).reshape(-1)
    n = packed.shape[0]
    y = np.empty(n, dtype=np.float64)
    lib().orc_w4_gemv_folded(_p(packed), _p(sm), n, x.shape[0], _p(x.view(np.uint16)), _p(y))
    return y


# ---------------------------------------------------------------------------- KV quantisers

def kv_quant_int8(x_f16):
    x = _c(x_f16, np.float16)
    n, d = x.shape
    q = np.empty((n, d), dtype=np.int8)
    s = np.empty(n, dtype=np.uint16)
    lib().orc_kv_quant_int8(_p(x.view(np.uint16)), n, d, _p(q), _p(s))
    return q, s.view(np.float16)


def kv_quant_int4(x_f16):
    x = _c(x_f16, np.float16)
    n, d = x.shape
    packed = np.empty((n, d // 2), dtype=np.uint8)
    sm = np.empty((n, d // 32, 2), dtype=np.uint16)
    lib().orc_kv_quant_int4(_p(x.view(np.uint16)), n, d, _p(packed), _p(sm))
    return packed, sm.view(np.float16)


# ---------------------------------------------------------------------------- pool layout, closed forms

def kv_block_bytes(n_kv_heads, head_dim, kv_dtype, block_tokens=16) -> int:
    return int(lib().orc_kv_block_bytes(n_kv_heads, head_dim, kv_dtype, block_tokens))


def kv_offset(n_kv_heads, head_dim, kv_dtype, block_tokens, pool_blocks, layer, block, part, head, slot) -> int:
    return int(lib().orc_kv_offset(n_kv_heads, head_dim, kv_dtype, block_tokens, pool_blocks, layer, block, part,
                                   head, slot))


def kv_bytes_per_token(n_layers, n_kv_heads, head_dim, bytes_per_value) -> int:
    return int(lib().orc_kv_bytes_per_token(n_layers, n_kv_heads, head_dim, float(bytes_per_value)))


def kv_max_context(total, os_reserve, weights, bpt) -> int:
    return int(lib().orc_kv_max_context(float(total), float(os_reserve), float(weights), float(bpt)))


class PoolModel:
    """The block allocator as host bookkeeping ([Core] 5.2: a preallocated KV pool).

    Reading: the free list starts in the given order (identity by default);
    blocks are taken from its front; a sequence takes a new block when it
    stores token t with t % block_tokens == 0; token t of a sequence lives in
    (table[t // block_tokens], slot t % block_tokens); a closed sequence's
    blocks go to the back of the free list in table order."""

    def __init__(self, n_blocks: int, block_tokens: int = 16, order=None):
        self.block_tokens = block_tokens
        self.free = list(range(n_blocks)) if order is None else [int(b) for b in order]
        self.tables: dict[int, list[int]] = {}
        self.lens: dict[int, int] = {}

    def open(self, sid: int):
        self.tables[sid] = []
        self.lens[sid] = 0

    def append(self, sid: int, n: int) -> bool:
        need = 0
        for t in range(self.lens[sid], self.lens[sid] + n):
            if t % self.block_tokens == 0:
                need += 1
        if need > len(self.free):
            return False
        for t in range(self.lens[sid], self.lens[sid] + n):
            if t % self.block_tokens == 0:
                self.tables[sid].append(self.free.pop(0))
        self.lens[sid] += n
        return True

    def close(self, sid: int):
        self.free.extend(self.tables.pop(sid))
        self.lens.pop(sid)

    def locate(self, sid: int, t: int):
        return self.tables[sid][t // self.block_tokens], t % self.block_tokens


# ---------------------------------------------------------------------------- arena planner

def arena_plan(sizes, first, last, align=64, closed=True):
    """Offsets and arena size by lifetime analysis and greedy-by-size placement ([TFLite] 2.1-2.2)."""
    n = len(sizes)
    sz = _c(sizes, np.int64)
    f = _c(first, np.int32)
    l = _c(last, np.int32)
    off = np.zeros(max(n, 1), dtype=np.int64)
    arena = lib().orc_arena_plan(n, _p(sz), _p(f), _p(l), align, 1 if closed else 0, _p(off))
    return off[:n], int(arena)


# ---------------------------------------------------------------------------- layer pieces

def rmsnorm(r, gamma_f16, eps=1e-5):
    r = _c(r, np.float64)
    g = _c(gamma_f16, np.float16)
    out = np.empty(r.shape[0], dtype=np.uint16)
    lib().orc_rmsnorm(_p(r), _p(g.view(np.uint16)), r.shape[0], eps, _p(out))
    return out.view(np.float16)


def rope_table(max_pos, head_dim, base):
    c = np.empty((max_pos, head_dim // 2), dtype=np.float32)
    s = np.empty((max_pos, head_dim // 2), dtype=np.float32)
    lib().orc_rope_table(max_pos, head_dim, float(base), _p(c), _p(s))
    return c, s


def rope_apply(x_f16, cos_row, sin_row):
    x = _c(x_f16, np.float16)
    out = np.empty_like(x)
    lib().orc_rope_apply(_p(x.view(np.uint16)), x.shape[0], _p(_c(cos_row, np.float32)), _p(_c(sin_row, np.float32)),
                         _p(out.view(np.uint16)))
    return out


# ---------------------------------------------------------------------------- model + KV store + forward

@dataclass
class ModelCfg:
    n_layers: int
    hidden: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    vocab: int
    rms_eps: float = 1e-5
    rope_base: float = 10000.0
    kv_dtype: int = KV_FP16
    block_tokens: int = 16

    def c(self) -> Cfg:
        return Cfg(self.n_layers, self.hidden, self.n_heads, self.n_kv_heads, self.head_dim, self.ffn, self.vocab,
                   self.rms_eps, self.rope_base, self.kv_dtype, self.block_tokens)

    @property
    def qkv_rows(self):
        return (self.n_heads + 2 * self.n_kv_heads) * self.head_dim


@dataclass
class Weights:
    """Canonical packed W4 tensors (numpy) per layer, fp16 norm gains and LM head."""
    wqkv: list = field(default_factory=list)
    sqkv: list = field(default_factory=list)
    wo: list = field(default_factory=list)
    so: list = field(default_factory=list)
    wgu: list = field(default_factory=list)
    sgu: list = field(default_factory=list)
    wdown: list = field(default_factory=list)
    sdown: list = field(default_factory=list)
    gamma1: list = field(default_factory=list)
    gamma2: list = field(default_factory=list)
    gamma_f: np.ndarray | None = None
    lm_head: np.ndarray | None = None

    def c(self):
        keep = []

        def arr(lst, dtype):
            a = [_c(x.view(dtype) if x.dtype != dtype and x.dtype.itemsize == np.dtype(dtype).itemsize else x, dtype)
                 for x in lst]
            keep.extend(a)
            ptrs = (ctypes.c_void_p * len(a))(*[x.ctypes.data for x in a])
            keep.append(ptrs)
            return ctypes.cast(ptrs, _PP)

        w = _Weights(arr(self.wqkv, np.uint8), arr(self.sqkv, np.uint16), arr(self.wo, np.uint8),
                     arr(self.so, np.uint16), arr(self.wgu, np.uint8), arr(self.sgu, np.uint16),
                     arr(self.wdown, np.uint8), arr(self.sdown, np.uint16), arr(self.gamma1, np.uint16),
                     arr(self.gamma2, np.uint16), None, None)
        gf = _c(self.gamma_f.view(np.uint16), np.uint16)
        keep.append(gf)
        w.gamma_f = gf.ctypes.data
        if self.lm_head is not None:
            lm = _c(self.lm_head.view(np.uint16), np.uint16)
            keep.append(lm)
            w.lm_head = lm.ctypes.data
        return w, keep


class KV:
    """The oracle's logical KV store of one sequence (stored codes in token order)."""

    def __init__(self, cfg: ModelCfg, capacity: int):
        self.cfg = cfg
        self._c = cfg.c()
        self.h = lib().orc_kv_create(ctypes.byref(self._c), capacity)
        self.data_bytes = {KV_FP16: 2 * cfg.head_dim, KV_INT8: cfg.head_dim, KV_INT4: cfg.head_dim // 2}[cfg.kv_dtype]
        self.meta_bytes = {KV_FP16: 0, KV_INT8: 2, KV_INT4: (cfg.head_dim // 32) * 4}[cfg.kv_dtype]

    def __del__(self):
        if getattr(self, "h", None):
            lib().orc_kv_destroy(self.h)
            self.h = None

    def __len__(self):
        return int(lib().orc_kv_len(self.h))

    def truncate(self, n: int):
        lib().orc_kv_truncate(self.h, n)

    def commit(self, n: int):
        """Make the n tokens that layer() stored past the length part of the store."""
        if lib().orc_kv_commit(self.h, n) != 0:
            raise RuntimeError("oracle KV: commit past the capacity")

    def append(self, k_f16, v_f16):
        """k, v: fp16 [L, n, Hkv, d] (already rotated)."""
        k = _c(k_f16, np.float16)
        v = _c(v_f16, np.float16)
        rc = lib().orc_kv_append(self.h, k.shape[1], _p(k.view(np.uint16)), _p(v.view(np.uint16)))
        if rc != 0:
            raise RuntimeError("oracle KV store full")

    def read(self, layer, which, tok, head):
        out = np.empty(self.cfg.head_dim, dtype=np.float32)
        lib().orc_kv_read(self.h, layer, which, tok, head, _p(out))
        return out

    def stored(self, layer, which, tok, head):
        data = np.empty(self.data_bytes, dtype=np.uint8)
        meta = np.empty(max(self.meta_bytes, 1), dtype=np.uint8)
        lib().orc_kv_stored(self.h, layer, which, tok, head, _p(data), _p(meta))
        return data, meta[:self.meta_bytes]

    def attention(self, layer, kv_head, q_f16, n_keys):
        q = _c(q_f16, np.float16)
        out = np.empty(self.cfg.head_dim, dtype=np.uint16)
        lib().orc_attention(ctypes.byref(self._c), self.h, layer, kv_head, _p(q.view(np.uint16)), n_keys,
                            _p(out))
        return out.view(np.float16)


def forward(cfg: ModelCfg, weights: Weights, kvs, n_tok, x_f16, rope_cos, rope_sin):
    """Run the step for len(kvs) sequences; returns fp16 [n_seq, vocab or hidden] for each last token."""
    c = cfg.c()
    w, keep = weights.c()
    n_seq = len(kvs)
    hs = (ctypes.c_void_p * n_seq)(*[k.h for k in kvs])
    nt = _c(n_tok, np.int32)
    x = _c(x_f16, np.float16)
    rc_, rs_ = _c(rope_cos, np.float32), _c(rope_sin, np.float32)
    width = cfg.vocab if cfg.vocab else cfg.hidden
    out = np.empty((n_seq, width), dtype=np.uint16)
    rc = lib().orc_forward(ctypes.byref(c), ctypes.byref(w), n_seq, ctypes.cast(hs, ctypes.c_void_p), _p(nt),
                           _p(x.view(np.uint16)), _p(rc_), _p(rs_), rc_.shape[0], _p(out))
    del keep
    if rc != 0:
        raise RuntimeError("oracle forward: KV store full or RoPE table too short")
    return out.view(np.float16)


def layer(cfg: ModelCfg, weights: Weights, l: int, kvs, n_tok, r_in, rope_cos, rope_sin):
    """Layer l alone, from the residual r_in (float64 [T, hidden], the tokens of the sequences in order) to
    the residual after it (float64 [T, hidden]). The tokens' k and v are stored at layer l of each store at
    positions len .. len + n_tok - 1; the stores' lengths do not change."""
    c = cfg.c()
    w, keep = weights.c()
    n_seq = len(kvs)
    hs = (ctypes.c_void_p * n_seq)(*[k.h for k in kvs])
    nt = _c(n_tok, np.int32)
    r = _c(r_in, np.float64)
    out = np.empty_like(r)
    rc_, rs_ = _c(rope_cos, np.float32), _c(rope_sin, np.float32)
    rc = lib().orc_layer(ctypes.byref(c), ctypes.byref(w), l, n_seq, ctypes.cast(hs, ctypes.c_void_p), _p(nt),
                         _p(r), _p(rc_), _p(rs_), rc_.shape[0], _p(out))
    del keep
    if rc != 0:
        raise RuntimeError("oracle layer: KV store full or RoPE table too short")
    return out


def output(cfg: ModelCfg, weights: Weights, r):
    """The output of each row of the final residual r (float64 [n, hidden]): fp16 logits [n, vocab], or the
    fp16 hidden state [n, hidden] without an LM head."""
    c = cfg.c()
    w, keep = weights.c()
    r = _c(np.atleast_2d(r), np.float64)
    width = cfg.vocab if cfg.vocab else cfg.hidden
    out = np.empty((r.shape[0], width), dtype=np.uint16)
    for i in range(r.shape[0]):
        lib().orc_output(ctypes.byref(c), ctypes.byref(w), _p(r[i]), _p(out[i]))
    del keep
    return out.view(np.float16)
