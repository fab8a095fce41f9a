"""Python binding of libmag (the GB300 decode-step library): argument marshalling only.

Every step of the decode path runs in the library's CUDA kernels; this module
only converts Python/torch arguments into the C ABI of ``include/mag.h``. If
the shared library is missing or cannot be loaded it raises -- there is no
fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmag.so")
_lock = threading.Lock()
_lib = None

(OK, ERR_INVALID_ARG, ERR_OOM, ERR_KV_FULL, ERR_CONTEXT_FULL, ERR_NOT_LOADED, ERR_CUDA, ERR_TIMEOUT, ERR_UNSUPPORTED,
 ERR_CORRUPT) = range(10)
STATUS_NAMES = ["OK", "INVALID_ARG", "OOM", "KV_FULL", "CONTEXT_FULL", "NOT_LOADED", "CUDA", "TIMEOUT", "UNSUPPORTED",
                "CORRUPT"]
KV_FP16, KV_INT8, KV_INT4 = 0, 1, 2
W_QKV, W_O, W_GATE_UP, W_DOWN, NORM_ATTN, NORM_FFN, NORM_FINAL, LM_HEAD = range(8)
FMT_F32_DENSE, FMT_W4G32, FMT_F16 = 0, 1, 2
FLAG_NO_GRAPH, FLAG_ARENA_NO_REUSE, FLAG_NO_PDL, FLAG_ELASTIC_POOL, FLAG_STEP_TIMING = 1, 2, 4, 8, 16
FLAG_DEBUG_CANARY = 32

EXPORTED = [
    "mag_create", "mag_destroy", "mag_load_weights", "mag_load_weights_f32_noalloc", "mag_session_open", "mag_session_close", "mag_session_length",
    "mag_session_truncate", "mag_kv_append", "mag_decode_step", "mag_decode_step_host", "mag_prefill_chunk",
    "mag_verify_tokens", "mag_prefill_batch", "mag_sync",
    "mag_get_memory_stats", "mag_get_step_stats", "mag_last_error", "mag_kv_bytes_per_token", "mag_quantize_w4g32",
    "mag_debug_read_weights", "mag_debug_kv_locate", "mag_debug_pool", "mag_debug_arena_plan",
    "mag_debug_last_step_launches", "mag_debug_profile_step", "mag_debug_step_residuals", "mag_debug_timeline",
    "mag_debug_prefill_residuals", "mag_debug_set_wait_limit",
    "mag_debug_fail_allocations", "mag_debug_set_table_entry", "mag_debug_arena",
    "mag_adapt_defaults", "mag_set_adaptive", "mag_get_profile", "mag_profiler_create", "mag_profiler_destroy",
    "mag_profiler_observe", "mag_profiler_quantile", "mag_profiler_count", "mag_plan_for", "mag_hot_pool_blocks",
]
OP_NAMES = ["step_begin", "qkv", "attention", "o_proj", "gate_up", "down", "lm_head"]


def debug_fail_allocations(skip: int, count: int) -> None:
    """Process-wide: the next `skip` library allocations succeed, the `count` after them fail (0: off)."""
    lib().mag_debug_fail_allocations(int(skip), int(count))


class MagError(RuntimeError):
    def __init__(self, status: int, msg: str):
        self.status = status
        super().__init__(f"{STATUS_NAMES[status] if 0 <= status < len(STATUS_NAMES) else status}: {msg}")


class Config(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("hidden", ctypes.c_int32), ("n_heads", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("ffn", ctypes.c_int32),
                ("vocab", ctypes.c_int32), ("rms_eps", ctypes.c_float), ("rope_base", ctypes.c_float),
                ("kv_dtype", ctypes.c_int32), ("block_tokens", ctypes.c_int32), ("pool_blocks", ctypes.c_int32),
                ("max_sessions", ctypes.c_int32), ("max_batch", ctypes.c_int32), ("max_chunk", ctypes.c_int32),
                ("max_context", ctypes.c_int32), ("pool_order_host", ctypes.POINTER(ctypes.c_int32)),
                ("flags", ctypes.c_uint64)]


class MemoryStats(ctypes.Structure):
    _fields_ = [("weight_bytes", ctypes.c_uint64), ("kv_pool_bytes", ctypes.c_uint64),
                ("kv_block_bytes", ctypes.c_uint64), ("pool_blocks_total", ctypes.c_int32),
                ("pool_blocks_free", ctypes.c_int32), ("arena_bytes", ctypes.c_uint64),
                ("arena_unshared_bytes", ctypes.c_uint64), ("other_device_bytes", ctypes.c_uint64),
                ("sessions_open", ctypes.c_int32), ("prefill_weight_bytes", ctypes.c_uint64),
                ("prefill_arena_bytes", ctypes.c_uint64), ("kv_pool_mapped_bytes", ctypes.c_uint64),
                ("pool_blocks_mapped", ctypes.c_int32), ("pool_blocks_hot", ctypes.c_int32),
                ("pool_group_blocks", ctypes.c_int32)]


class StepStats(ctypes.Structure):
    _fields_ = [("steps", ctypes.c_int64), ("last_kind", ctypes.c_int32), ("last_rows", ctypes.c_int32),
                ("last_launches", ctypes.c_int32), ("last_max_keys", ctypes.c_int32),
                ("last_bytes", ctypes.c_uint64), ("last_ms", ctypes.c_double)]


class ArenaTensor(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 24), ("size", ctypes.c_uint64), ("first", ctypes.c_int32),
                ("last", ctypes.c_int32), ("offset", ctypes.c_uint64)]


class AdaptConfig(ctypes.Structure):
    _fields_ = [("enable_adaptive", ctypes.c_int32), ("adaptive_window_size", ctypes.c_int32),
                ("adaptive_sample_rate", ctypes.c_int32), ("plan_short_below", ctypes.c_int32),
                ("plan_long_above", ctypes.c_int32), ("plan_splits", ctypes.c_int32 * 3),
                ("plan_wide", ctypes.c_int32 * 3), ("force_plan", ctypes.c_int32), ("async_switch", ctypes.c_int32), ("hot_pool_slack", ctypes.c_float)]


class Profile(ctypes.Structure):
    _fields_ = [("seen", ctypes.c_int64), ("recorded", ctypes.c_int32), ("p50", ctypes.c_int32),
                ("p90", ctypes.c_int32), ("p99", ctypes.c_int32), ("plan", ctypes.c_int32),
                ("pending_plan", ctypes.c_int32), ("plan_splits", ctypes.c_int32), ("plan_wide", ctypes.c_int32),
                ("switches", ctypes.c_int32),
                ("hot_blocks", ctypes.c_int64)]


def build(force: bool = False) -> str:
    from . import _build
    return _build.build(force=force)


def lib():
    """Load libmag.so (raises if it is missing: build it with ``build()``)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: the CUDA library must be built (quantized_decode_step_gb300."
                                   "build()); there is no CPU fallback")
            L = ctypes.CDLL(LIB_PATH)
            vp, i32, i64, u64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64, ctypes.c_size_t
            P32 = ctypes.POINTER(ctypes.c_int32)
            sig = {
                "mag_create": ([ctypes.POINTER(Config), vp, ctypes.POINTER(vp)], i32),
                "mag_destroy": ([vp], None),
                "mag_load_weights": ([vp, i32, i32, vp, i32, sz], i32),
                "mag_load_weights_f32_noalloc": ([vp, i32, i32, vp, sz], i32),
                "mag_session_open": ([vp, P32], i32),
                "mag_session_close": ([vp, i32], i32),
                "mag_session_length": ([vp, i32, P32], i32),
                "mag_session_truncate": ([vp, i32, i32], i32),
                "mag_kv_append": ([vp, i32, i32, vp, vp], i32),
                "mag_decode_step": ([vp, i32, P32, vp, vp], i32),
                "mag_decode_step_host": ([vp, i32, P32, vp, vp], i32),
                "mag_prefill_chunk": ([vp, i32, i32, vp, vp], i32),
                "mag_verify_tokens": ([vp, i32, i32, vp, vp], i32),
                "mag_prefill_batch": ([vp, i32, P32, P32, vp, vp], i32),
                "mag_sync": ([vp], i32),
                "mag_get_memory_stats": ([vp, ctypes.POINTER(MemoryStats)], i32),
                "mag_get_step_stats": ([vp, ctypes.POINTER(StepStats)], i32),
                "mag_last_error": ([vp], ctypes.c_char_p),
                "mag_kv_bytes_per_token": ([ctypes.POINTER(Config)], u64),
                "mag_quantize_w4g32": ([vp, i64, i64, vp, vp, vp], i32),
                "mag_debug_read_weights": ([vp, i32, i32, vp, sz], i32),
                "mag_debug_kv_locate": ([vp, i32, i32, i32, ctypes.POINTER(ctypes.c_int64)], i32),
                "mag_debug_pool": ([vp, ctypes.POINTER(vp), ctypes.POINTER(u64)], i32),
                "mag_debug_arena_plan": ([vp, i32, ctypes.POINTER(ArenaTensor), i32, P32, ctypes.POINTER(u64)], i32),
                "mag_debug_last_step_launches": ([vp], i32),
                "mag_debug_profile_step": ([vp, i32, P32, vp, vp, P32, ctypes.POINTER(ctypes.c_float), i32, P32],
                                           i32),
                "mag_debug_step_residuals": ([vp, i32, P32, vp, vp, vp], i32),
                "mag_debug_timeline": ([vp, i32, P32, vp, vp, vp, i32, P32], i32),
                "mag_debug_prefill_residuals": ([vp, i32, i32, vp, vp, vp], i32),
                "mag_debug_set_wait_limit": ([vp, i64], i32),
                "mag_debug_fail_allocations": ([i32, i32], None),
                "mag_debug_set_table_entry": ([vp, i32, i32, i32], i32),
                "mag_debug_arena": ([vp, ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(ctypes.c_uint64)], i32),
                "mag_adapt_defaults": ([ctypes.POINTER(AdaptConfig)], None),
                "mag_set_adaptive": ([vp, ctypes.POINTER(AdaptConfig)], i32),
                "mag_get_profile": ([vp, ctypes.POINTER(Profile)], i32),
                "mag_profiler_create": ([i32, i32, ctypes.POINTER(vp)], i32),
                "mag_profiler_destroy": ([vp], None),
                "mag_profiler_observe": ([vp, i32], i32),
                "mag_profiler_quantile": ([vp, ctypes.c_double, P32], i32),
                "mag_profiler_count": ([vp], i32),
                "mag_plan_for": ([i32, i32, i32], i32),
                "mag_hot_pool_blocks": ([i32, i32, ctypes.c_float], i64),
            }
            for name, (args, res) in sig.items():
                fn = getattr(L, name)
                fn.argtypes = args
                fn.restype = res
            _lib = L
    return _lib


def _ptr(t) -> int:
    """Device or host address of a torch tensor / numpy array / int."""
    if t is None:
        return 0
    if isinstance(t, int):
        return t
    if hasattr(t, "data_ptr"):
        return t.data_ptr()
    return t.ctypes.data


def make_config(shape, kv_dtype=KV_FP16, pool_blocks=64, max_sessions=4, max_batch=1, max_chunk=0, max_context=2048,
                flags=0, pool_order=None) -> Config:
    """A Config from any object with the shape fields (n_layers, hidden, ..., rms_eps, rope_base)."""
    c = Config(shape.n_layers, shape.hidden, shape.n_heads, shape.n_kv_heads, shape.head_dim, shape.ffn, shape.vocab,
               shape.rms_eps, shape.rope_base, kv_dtype, 16, pool_blocks, max_sessions, max_batch, max_chunk,
               max_context, None, flags)
    if pool_order is not None:
        import numpy as np
        arr = np.ascontiguousarray(pool_order, dtype=np.int32)
        c._order = arr  # keep alive
        c.pool_order_host = arr.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
    return c


def kv_bytes_per_token(cfg: Config) -> int:
    return int(lib().mag_kv_bytes_per_token(ctypes.byref(cfg)))


def quantize_w4g32(src, rows, cols, codes, scale_min, stream=0):
    st = lib().mag_quantize_w4g32(_ptr(src), rows, cols, _ptr(codes), _ptr(scale_min), stream)
    if st != OK:
        raise MagError(st, "mag_quantize_w4g32")


def adapt_defaults() -> AdaptConfig:
    a = AdaptConfig()
    lib().mag_adapt_defaults(ctypes.byref(a))
    return a


class Profiler:
    """The load profile on its own (host only): sliding window, sampled, nearest-rank quantiles."""

    def __init__(self, window=64, sample_every=4):
        h = ctypes.c_void_p()
        st = lib().mag_profiler_create(window, sample_every, ctypes.byref(h))
        if st != 0:
            raise MagError(st, f"mag_profiler_create({window}, {sample_every})")
        self.h = h

    def observe(self, length) -> bool:
        return bool(lib().mag_profiler_observe(self.h, int(length)))

    def quantile(self, q) -> int:
        out = ctypes.c_int32()
        st = lib().mag_profiler_quantile(self.h, float(q), ctypes.byref(out))
        if st != 0:
            raise MagError(st, f"mag_profiler_quantile({q})")
        return out.value

    def count(self) -> int:
        return int(lib().mag_profiler_count(self.h))

    def close(self):
        if self.h:
            lib().mag_profiler_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def plan_for(p90, short_below=128, long_above=512) -> int:
    return int(lib().mag_plan_for(p90, short_below, long_above))


def hot_pool_blocks(p90, n_sessions, slack=1.2) -> int:
    return int(lib().mag_hot_pool_blocks(p90, n_sessions, slack))


class Context:
    """One mag_ctx. Methods mirror the C entry points of the same names."""

    def __init__(self, cfg: Config, stream: int = 0):
        self.cfg = cfg
        h = ctypes.c_void_p()
        st = lib().mag_create(ctypes.byref(cfg), stream, ctypes.byref(h))
        if st != OK:
            raise MagError(st, "mag_create failed (details on stderr)")
        self.h = h

    def _check(self, st, what):
        if st != OK:
            raise MagError(st, f"{what}: {lib().mag_last_error(self.h).decode()}")

    def close(self):
        if getattr(self, "h", None):
            lib().mag_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def last_error(self) -> str:
        return lib().mag_last_error(self.h).decode()

    def load_weights(self, tensor, layer, src, fmt, nbytes):
        self._check(lib().mag_load_weights(self.h, tensor, layer, _ptr(src), fmt, nbytes), "mag_load_weights")

    def load_weights_f32_noalloc(self, tensor, layer, src, nbytes):
        """fp32 projection load through the library's fixed per-device scratch (no device allocation)."""
        self._check(lib().mag_load_weights_f32_noalloc(self.h, tensor, layer, _ptr(src), nbytes),
                    "mag_load_weights_f32_noalloc")

    def session_open(self) -> int:
        sid = ctypes.c_int32()
        self._check(lib().mag_session_open(self.h, ctypes.byref(sid)), "mag_session_open")
        return sid.value

    def session_close(self, sid):
        self._check(lib().mag_session_close(self.h, sid), "mag_session_close")

    def session_length(self, sid) -> int:
        n = ctypes.c_int32()
        self._check(lib().mag_session_length(self.h, sid, ctypes.byref(n)), "mag_session_length")
        return n.value

    def session_truncate(self, sid, length):
        self._check(lib().mag_session_truncate(self.h, sid, length), "mag_session_truncate")

    def kv_append(self, sid, n_tokens, k, v):
        self._check(lib().mag_kv_append(self.h, sid, n_tokens, _ptr(k), _ptr(v)), "mag_kv_append")

    def decode_step(self, sessions, hidden_in, out):
        ids = (ctypes.c_int32 * len(sessions))(*sessions)
        self._check(lib().mag_decode_step(self.h, len(sessions), ids, _ptr(hidden_in), _ptr(out)), "mag_decode_step")

    def decode_step_host(self, sessions, hidden_in_host, out_host):
        ids = (ctypes.c_int32 * len(sessions))(*sessions)
        self._check(lib().mag_decode_step_host(self.h, len(sessions), ids, _ptr(hidden_in_host), _ptr(out_host)),
                    "mag_decode_step_host")

    def prefill_chunk(self, sid, n_tokens, hidden_in, last_out):
        self._check(lib().mag_prefill_chunk(self.h, sid, n_tokens, _ptr(hidden_in), _ptr(last_out)),
                    "mag_prefill_chunk")

    def prefill_batch(self, sessions, n_tokens, hidden_in, last_out):
        ids = (ctypes.c_int32 * len(sessions))(*sessions)
        nt = (ctypes.c_int32 * len(n_tokens))(*n_tokens)
        self._check(lib().mag_prefill_batch(self.h, len(sessions), ids, nt, _ptr(hidden_in), _ptr(last_out)),
                    "mag_prefill_batch")

    def verify_tokens(self, sid, n_tokens, hidden_in, out):
        self._check(lib().mag_verify_tokens(self.h, sid, n_tokens, _ptr(hidden_in), _ptr(out)), "mag_verify_tokens")

    def sync(self):
        self._check(lib().mag_sync(self.h), "mag_sync")

    def memory_stats(self) -> dict:
        s = MemoryStats()
        self._check(lib().mag_get_memory_stats(self.h, ctypes.byref(s)), "mag_get_memory_stats")
        return {n: getattr(s, n) for n, _ in MemoryStats._fields_}

    def step_stats(self) -> dict:
        s = StepStats()
        self._check(lib().mag_get_step_stats(self.h, ctypes.byref(s)), "mag_get_step_stats")
        return {n: getattr(s, n) for n, _ in StepStats._fields_}

    def debug_read_weights(self, tensor, layer, dst, nbytes):
        self._check(lib().mag_debug_read_weights(self.h, tensor, layer, _ptr(dst), nbytes), "mag_debug_read_weights")

    def debug_kv_locate(self, sid, layer, token):
        out = (ctypes.c_int64 * 5)()
        self._check(lib().mag_debug_kv_locate(self.h, sid, layer, token, out), "mag_debug_kv_locate")
        return list(out)

    def debug_pool(self):
        p, n = ctypes.c_void_p(), ctypes.c_uint64()
        self._check(lib().mag_debug_pool(self.h, ctypes.byref(p), ctypes.byref(n)), "mag_debug_pool")
        return p.value, n.value

    def debug_arena(self):
        p, n = ctypes.c_void_p(), ctypes.c_uint64()
        self._check(lib().mag_debug_arena(self.h, ctypes.byref(p), ctypes.byref(n)), "mag_debug_arena")
        return p.value, n.value

    def debug_arena_plan(self, phase=0):
        n, total = ctypes.c_int32(), ctypes.c_uint64()
        self._check(lib().mag_debug_arena_plan(self.h, phase, None, 0, ctypes.byref(n), ctypes.byref(total)),
                    "mag_debug_arena_plan")
        arr = (ArenaTensor * max(n.value, 1))()
        self._check(lib().mag_debug_arena_plan(self.h, phase, arr, n.value, ctypes.byref(n), ctypes.byref(total)),
                    "mag_debug_arena_plan")
        return [dict(name=a.name.decode(), size=a.size, first=a.first, last=a.last, offset=a.offset)
                for a in arr[:n.value]], total.value

    def last_step_launches(self) -> int:
        return int(lib().mag_debug_last_step_launches(self.h))

    def set_adaptive(self, enable=True, **fields):
        """Adaptive runtime from the library's defaults with the given fields replaced (plan_splits: a
        3-sequence); enable=False turns it off."""
        a = adapt_defaults()
        a.enable_adaptive = 1 if enable else 0
        for k, v in fields.items():
            if k in ("plan_splits", "plan_wide"):
                setattr(a, k, (ctypes.c_int32 * 3)(*v))
            else:
                setattr(a, k, v)
        self._check(lib().mag_set_adaptive(self.h, ctypes.byref(a)), "mag_set_adaptive")

    def profile(self) -> dict:
        p = Profile()
        self._check(lib().mag_get_profile(self.h, ctypes.byref(p)), "mag_get_profile")
        return {n: getattr(p, n) for n, _ in Profile._fields_}

    def step_residuals(self, sessions, hidden_in, out, resid):
        """Eager step that also fills resid (device fp32 [L+1, batch, hidden]) with the residual stream:
        row 0 the input, row l+1 after layer l."""
        ids = (ctypes.c_int32 * len(sessions))(*sessions)
        self._check(lib().mag_debug_step_residuals(self.h, len(sessions), ids, _ptr(hidden_in), _ptr(out),
                                                   _ptr(resid)), "mag_debug_step_residuals")

    def timeline(self, sessions, hidden_in, out, recs):
        """One step (launched one by one, as the graph holds it) whose GEMV and attention blocks stamp their
        phases into recs (device uint64 [cap, 4]: tag, block, event, ns); returns the records attempted."""
        ids = (ctypes.c_int32 * len(sessions))(*sessions)
        n = ctypes.c_int32(0)
        self._check(lib().mag_debug_timeline(self.h, len(sessions), ids, _ptr(hidden_in), _ptr(out), _ptr(recs),
                                             int(recs.shape[0]), ctypes.byref(n)), "mag_debug_timeline")
        return n.value

    def debug_set_table_entry(self, sid: int, index: int, value: int):
        """Write one block-table entry on the device only (tests of the block-id checks)."""
        self._check(lib().mag_debug_set_table_entry(self.h, sid, index, value), "mag_debug_set_table_entry")

    def set_wait_limit(self, polls: int):
        """Polls of a GEMV pipeline wait before it gives up (< 0: the built-in limit; 0: at once)."""
        self._check(lib().mag_debug_set_wait_limit(self.h, int(polls)), "mag_debug_set_wait_limit")

    def prefill_residuals(self, sid, n_tokens, hidden_in, last_out, resid):
        """Prefill chunk that also fills resid (device fp32 [L+1, n_tokens, hidden]) with the residual stream."""
        self._check(lib().mag_debug_prefill_residuals(self.h, sid, n_tokens, _ptr(hidden_in), _ptr(last_out),
                                                      _ptr(resid)), "mag_debug_prefill_residuals")

    def profile_step(self, sessions, hidden_in, out, cap=4096):
        """Instrumented step: list of (op name, device ms) per kernel launch."""
        ids = (ctypes.c_int32 * len(sessions))(*sessions)
        kinds = (ctypes.c_int32 * cap)()
        ms = (ctypes.c_float * cap)()
        n = ctypes.c_int32()
        self._check(lib().mag_debug_profile_step(self.h, len(sessions), ids, _ptr(hidden_in), _ptr(out), kinds, ms,
                                                 cap, ctypes.byref(n)), "mag_debug_profile_step")
        return [(OP_NAMES[kinds[i]], float(ms[i])) for i in range(min(n.value, cap))]
