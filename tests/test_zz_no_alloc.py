"""mag_load_weights_f32_noalloc against the ordinary fp32 load (mag_load_weights with FMT_F32_DENSE).

The no-alloc entry point quantises and tiles a projection slab by slab
through the library's fixed per-device scratch instead of a transient
allocation of the whole projection. The bytes it leaves in the context are
integer work, so the bar is bit-exact equality with the ordinary load's:
* the 8B layer (4096 / 14336 wide: several slabs per projection, QKV slabs of
  whole heads, gate-up slabs pairing gate and up rows) and the tiny layer
  (FFN 688: a ragged last group), every projection loaded by two calls in a
  row with two different weight draws, each compared after its call;
* the decode step of the tiny model with all weights loaded each way: equal
  hidden states;
* a projection whose one-head slab exceeds the scratch: INVALID_ARG naming
  the scratch, before any device work;
* that it allocates nothing: the high-water mark of the device's default
  memory pool (which the ordinary load's stream-ordered allocation raises)
  stays where it was across no-alloc loads of every 8B projection;
* a context with prefill enabled (max_chunk > 0), whose loads also refresh the
  prefill GEMM's weights: a prefill chunk then a decode step give the same
  outputs, bit for bit, as with the ordinary load, and match the oracle.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import quantized_decode_step_gb300 as mag
import synth
from synth.workloads import LLAMA8B, TINY, Shape, shrink
from tests.helpers import TOL_MAX_ABS, TOL_REL_L2, max_abs, model_cfg, oracle_weights, prior_kv, proj_shape, rel_l2

pytestmark = pytest.mark.gpu

SEED = 11
PROJ = (("wgu", mag.W_GATE_UP), ("wdown", mag.W_DOWN), ("wqkv", mag.W_QKV), ("wo", mag.W_O))


@pytest.fixture(scope="module", autouse=True)
def built():
    mag.build()
    assert torch.cuda.is_available()


def _ctx(shape):
    cfg = mag.make_config(shape, pool_blocks=4, max_sessions=1, max_batch=1, max_context=64)
    return mag.Context(cfg, torch.cuda.current_stream().cuda_stream)


def _read(ctx, tid, layer, n, k):
    out = torch.empty(n * ((k + 31) // 32) * 20, dtype=torch.uint8, device="cuda")
    ctx.debug_read_weights(tid, layer, out, out.numel())
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("shape", [shrink(LLAMA8B, n_layers=1, vocab=0), TINY], ids=["8b-layer", "tiny"])
def test_noalloc_load_matches_ordinary_load(shape):
    ref, ctx = _ctx(shape), _ctx(shape)
    for name, tid in PROJ:
        n, k = proj_shape(shape, name)
        for seed in (SEED, SEED + 1):  # two calls in a row into the same projection
            src = torch.from_numpy(synth.weight_f32(seed, 0, name, n, k)).cuda()
            ref.load_weights(tid, 0, src, mag.FMT_F32_DENSE, src.numel() * 4)
            ctx.load_weights_f32_noalloc(tid, 0, src, src.numel() * 4)
            torch.cuda.synchronize()
            assert torch.equal(_read(ctx, tid, 0, n, k), _read(ref, tid, 0, n, k)), (shape.name, name, seed)
    ref.close()
    ctx.close()


def test_noalloc_decode_matches_ordinary_load():
    shape = TINY
    outs = []
    for noalloc in (False, True):
        ctx = _ctx(shape)
        for name, tid in PROJ:
            n, k = proj_shape(shape, name)
            src = torch.from_numpy(synth.weight_f32(SEED, 0, name, n, k)).cuda()
            if noalloc:
                ctx.load_weights_f32_noalloc(tid, 0, src, src.numel() * 4)
            else:
                ctx.load_weights(tid, 0, src, mag.FMT_F32_DENSE, src.numel() * 4)
        for tag, tid in (("L0.g1", mag.NORM_ATTN), ("L0.g2", mag.NORM_FFN), ("gf", mag.NORM_FINAL)):
            g = torch.from_numpy(synth.norm_gain_f16(SEED, tag, shape.hidden, True)).cuda()
            ctx.load_weights(tid, 0, g, mag.FMT_F16, g.numel() * 2)
        sid = ctx.session_open()
        step = []
        for s in range(2):
            x = torch.from_numpy(synth.hidden_f16(SEED, 1, shape.hidden, f"x.step{s}")).cuda()
            out = torch.empty((1, shape.hidden), dtype=torch.float16, device="cuda")
            ctx.decode_step([sid], x, out)
            ctx.sync()
            step.append(out.cpu())
        outs.append(step)
        ctx.close()
    for a, b in zip(*outs):
        assert torch.isfinite(a.float()).all()
        assert torch.equal(a, b)


def test_noalloc_rejects_slab_beyond_scratch():
    # QKV slabs hold whole heads: one head of d = 128 rows of K = 53,248 values is 4.26 MB of W4G32 bytes
    shape = Shape("wide-qkv", n_layers=1, hidden=53248, n_heads=1, n_kv_heads=1, head_dim=128, ffn=8, vocab=0)
    ctx = _ctx(shape)
    n, k = proj_shape(shape, "wqkv")
    src = torch.zeros((n, k), dtype=torch.float32, device="cuda")
    with pytest.raises(mag.MagError, match="scratch") as e:
        ctx.load_weights_f32_noalloc(mag.W_QKV, 0, src, src.numel() * 4)
    assert e.value.status == mag.ERR_INVALID_ARG
    # the other projections of that model fit and load
    n, k = proj_shape(shape, "wo")
    src = torch.from_numpy(synth.weight_f32(SEED, 0, "wo", n, k)).cuda()
    ctx.load_weights_f32_noalloc(mag.W_O, 0, src, src.numel() * 4)
    torch.cuda.synchronize()
    ctx.close()


class _DefaultPool:
    """The current device's default memory pool through the driver API (the pool that stream-ordered
    allocations such as cudaMallocAsync draw from): reset and read its used-memory high-water mark."""
    USED_MEM_CURRENT, USED_MEM_HIGH = 7, 8

    def __init__(self):
        self.cu = ctypes.CDLL("libcuda.so.1")
        dev = ctypes.c_int()
        assert self.cu.cuCtxGetDevice(ctypes.byref(dev)) == 0
        self.pool = ctypes.c_void_p()
        assert self.cu.cuDeviceGetDefaultMemPool(ctypes.byref(self.pool), dev) == 0

    def get(self, attr):
        v = ctypes.c_uint64()
        assert self.cu.cuMemPoolGetAttribute(self.pool, attr, ctypes.byref(v)) == 0
        return v.value

    def reset_high(self):
        """The high-water mark restarts from the memory in use now; returns that."""
        zero = ctypes.c_uint64(0)
        assert self.cu.cuMemPoolSetAttribute(self.pool, self.USED_MEM_HIGH, ctypes.byref(zero)) == 0
        return self.get(self.USED_MEM_HIGH)


def test_noalloc_load_allocates_nothing():
    shape = shrink(LLAMA8B, n_layers=1, vocab=0)
    ctx = _ctx(shape)
    srcs = []
    for name, tid in PROJ:
        n, k = proj_shape(shape, name)
        srcs.append((tid, torch.from_numpy(synth.weight_f32(SEED, 0, name, n, k)).cuda()))
    torch.cuda.synchronize()
    pool = _DefaultPool()
    base = pool.reset_high()
    for tid, src in srcs:
        ctx.load_weights_f32_noalloc(tid, 0, src, src.numel() * 4)
    torch.cuda.synchronize()
    assert pool.get(pool.USED_MEM_HIGH) == base, "a no-alloc load drew memory from the device's pool"
    # control: the ordinary fp32 load quantises through a stream-ordered copy from that pool
    base = pool.reset_high()
    tid, src = srcs[0]
    ctx.load_weights(tid, 0, src, mag.FMT_F32_DENSE, src.numel() * 4)
    torch.cuda.synchronize()
    assert pool.get(pool.USED_MEM_HIGH) > base
    ctx.close()


def test_noalloc_load_with_prefill_enabled():
    """max_chunk > 0: the loads also refresh the prefill GEMM's copy of each projection."""
    shape, seed, p, T = TINY, SEED + 5, 40, 24
    outs = []
    for noalloc in (False, True):
        cfg = mag.make_config(shape, pool_blocks=8, max_sessions=1, max_batch=1, max_chunk=T, max_context=p + T + 2)
        ctx = mag.Context(cfg, torch.cuda.current_stream().cuda_stream)
        for name, tid in PROJ:
            n, k = proj_shape(shape, name)
            src = torch.from_numpy(synth.weight_f32(seed, 0, name, n, k)).cuda()
            if noalloc:
                ctx.load_weights_f32_noalloc(tid, 0, src, src.numel() * 4)
            else:
                ctx.load_weights(tid, 0, src, mag.FMT_F32_DENSE, src.numel() * 4)
        for tag, tid in (("L0.g1", mag.NORM_ATTN), ("L0.g2", mag.NORM_FFN), ("gf", mag.NORM_FINAL)):
            g = torch.from_numpy(synth.norm_gain_f16(seed, tag, shape.hidden)).cuda()
            ctx.load_weights(tid, 0, g, mag.FMT_F16, g.numel() * 2)
        sid = ctx.session_open()
        k, v = prior_kv(shape, seed, 0, p)
        ctx.kv_append(sid, p, torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda())
        x = torch.from_numpy(synth.hidden_f16(seed, T, shape.hidden, "chunk")).cuda()
        o1 = torch.empty(shape.hidden, dtype=torch.float16, device="cuda")
        ctx.prefill_chunk(sid, T, x, o1)
        x2 = torch.from_numpy(synth.hidden_f16(seed, 1, shape.hidden, "after")).cuda()
        o2 = torch.empty((1, shape.hidden), dtype=torch.float16, device="cuda")
        ctx.decode_step([sid], x2, o2)
        ctx.sync()
        outs.append((o1.cpu(), o2.cpu()))
        ctx.close()
    for a, b in zip(*outs):
        assert torch.equal(a, b)
    w = oracle_weights(shape, seed)
    ocfg = model_cfg(shape, 0)
    kv = oracle.KV(ocfg, p + T + 2)
    kv.append(k, v)
    c, s = oracle.rope_table(p + T + 2, shape.head_dim, shape.rope_base)
    ref1 = oracle.forward(ocfg, w, [kv], [T], synth.hidden_f16(seed, T, shape.hidden, "chunk"), c, s)[0]
    ref2 = oracle.forward(ocfg, w, [kv], [1], synth.hidden_f16(seed, 1, shape.hidden, "after"), c, s)
    for got, ref in ((outs[1][0].numpy(), ref1), (outs[1][1].numpy(), ref2)):
        assert max_abs(got, ref) <= TOL_MAX_ABS and rel_l2(got, ref) <= TOL_REL_L2
