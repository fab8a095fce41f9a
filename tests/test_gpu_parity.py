"""GPU parity: the library's kernels (through the C ABI) against the oracle on the same seeded inputs.

Bit-exact: W4 quantise/pack, KV quantise + block placement, arena offsets.
Tolerance (fp16 logits / hidden states): max-abs <= 2e-2 AND rel-L2 <= 1e-3.
"""
import numpy as np
import pytest
import torch

import oracle
import quantized_decode_step_gb300 as mag
import synth
from synth import driver
from synth.workloads import KV_FP16, KV_INT4, KV_INT8, TINY, TINY_DECODE, Workload, shrink
from tests.helpers import TOL_MAX_ABS, TOL_REL_L2, device_bytes, max_abs, model_cfg, rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    mag.build()
    assert torch.cuda.is_available()
    torch.cuda.init()


def _gpu_quantize(w):
    rows, cols = w.shape
    g = -(-cols // 32)
    src = torch.from_numpy(np.ascontiguousarray(w)).cuda()
    codes = torch.empty((rows, 16 * g), dtype=torch.uint8, device="cuda")
    sm = torch.empty((rows, g, 2), dtype=torch.float16, device="cuda")
    mag.quantize_w4g32(src, rows, cols, codes, sm, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return codes.cpu().numpy(), sm.cpu().numpy()


@pytest.mark.parametrize("rows,cols", [(64, 256), (37, 688), (16, 4096), (3, 32), (5, 48)])
def test_quantize_w4g32_bit_exact(rows, cols):
    w = synth.weight_f32(3, 0, f"q{rows}x{cols}", rows, cols)
    if rows >= 16:  # plant the hand cases' awkward values: ties, constant groups, zeros
        w[0, :32] = 0.0
        w[1, :32] = 0.3
        w[2, :32] = np.arange(32) * 0.5 - 1.5
    c_gpu, s_gpu = _gpu_quantize(w)
    c_ref, s_ref = oracle.w4g32_quantize(w)
    assert np.array_equal(c_gpu, c_ref)
    assert np.array_equal(s_gpu.view(np.uint16), s_ref.view(np.uint16))


def _oracle_model(shape, seed, random_gain=False):
    """Quantise the same fp32 draws with the oracle."""
    return oracle_weights_from(shape, seed, random_gain)


def oracle_weights_from(shape, seed, random_gain):
    from tests.helpers import oracle_weights
    return oracle_weights(shape, seed, random_gain=random_gain)


def _oracle_kvs(wl: Workload, seed):
    cfg = model_cfg(wl.shape, wl.kv_dtype)
    kvs = []
    for i, p in enumerate(wl.prior):
        kv = oracle.KV(cfg, p + 64)
        for t0 in range(0, p, 4096):
            n = min(4096, p - t0)
            L, H, d = wl.shape.n_layers, wl.shape.n_kv_heads, wl.shape.head_dim
            k = np.empty((L, n, H, d), np.float16)
            v = np.empty((L, n, H, d), np.float16)
            for l in range(L):
                k[l] = synth.prior_kv_f16(seed, i, l, "K", n, H, d, tok0=t0)
                v[l] = synth.prior_kv_f16(seed, i, l, "V", n, H, d, tok0=t0)
            kv.append(k, v)
        kvs.append(kv)
    return cfg, kvs


def _compare(out_gpu, out_ref, what):
    a = out_gpu.astype(np.float64)
    b = out_ref.astype(np.float64)
    assert np.all(np.isfinite(a)), what
    ma, rl = max_abs(a, b), rel_l2(a, b)
    assert ma <= TOL_MAX_ABS and rl <= TOL_REL_L2, f"{what}: max-abs {ma:.3e}, rel-L2 {rl:.3e}"
    return ma, rl


def _run_decode(wl: Workload, seed, n_steps=1, random_gain=False, flags=0, weights_check=False):
    ctx, sids = driver.setup(wl, seed, random_gain=random_gain, flags=flags, extra_tokens=n_steps)
    w = _oracle_model(wl.shape, seed, random_gain)
    if weights_check:
        for l in range(wl.shape.n_layers):
            for name, tid in driver.PROJ:
                p, sm = getattr(w, name)[l], getattr(w, "s" + name[1:])[l]
                buf = torch.empty(p.size + sm.size * 2, dtype=torch.uint8, device="cuda")
                ctx.debug_read_weights(tid, l, buf, buf.numel())
                torch.cuda.synchronize()
                got = buf.cpu().numpy()
                assert np.array_equal(got[:p.size], p.reshape(-1)), (l, name)
                assert np.array_equal(got[p.size:].view(np.uint16), sm.view(np.uint16).reshape(-1)), (l, name)
    cfg, kvs = _oracle_kvs(wl, seed)
    c, s = oracle.rope_table(max(wl.prior) + n_steps + 1, wl.shape.head_dim, wl.shape.rope_base)
    width = wl.shape.vocab or wl.shape.hidden
    results = []
    for step in range(n_steps):
        x = driver.step_inputs(wl, seed, step)
        xin = torch.from_numpy(x).cuda()
        out = torch.empty((wl.batch, width), dtype=torch.float16, device="cuda")
        ctx.decode_step(sids, xin, out)
        ctx.sync()
        got = out.cpu().numpy()
        ref = oracle.forward(cfg, w, kvs, [1] * wl.batch, x, c, s)
        results.append(_compare(got, ref, f"{wl.name} step {step}"))
    for sid, p in zip(sids, wl.prior):
        assert ctx.session_length(sid) == p + n_steps
    return ctx, results


@pytest.mark.parametrize("dt", [KV_FP16, KV_INT8, KV_INT4])
def test_tiny_decode_matches_oracle(dt):
    wl = Workload(f"tiny-{dt}", TINY, dt, 1, (128,))
    ctx, res = _run_decode(wl, 11, n_steps=3, random_gain=True, weights_check=True)
    assert ctx.last_step_launches() == 1 + 5 * TINY.n_layers + 1


@pytest.mark.parametrize("flags", [mag.FLAG_NO_GRAPH, mag.FLAG_NO_PDL, mag.FLAG_ARENA_NO_REUSE, mag.FLAG_DEBUG_CANARY,
                                   mag.FLAG_STEP_TIMING])
def test_tiny_decode_modes(flags):
    _run_decode(TINY_DECODE, 12, n_steps=2, flags=flags)


def test_tiny_batch_ragged_contexts():
    """Batch of 5 sessions with ragged contexts (1, 15, 16, 17, 200 tokens) in a scattered pool."""
    wl = Workload("tiny-b5", TINY, KV_INT4, 5, (1, 15, 16, 17, 200), scattered_pool=True)
    _run_decode(wl, 13, n_steps=2)


@pytest.mark.parametrize("B", [2, 3, 4])
def test_tiny_small_batches(B):
    """Batches of 2-4 sessions (the multi-token path of the one-block-per-SM GEMV), ragged contexts."""
    wl = Workload(f"tiny-b{B}", TINY, KV_INT8, B, tuple(range(5, 5 + 37 * B, 37)), scattered_pool=True)
    _run_decode(wl, 15 + B, n_steps=2)


@pytest.mark.parametrize("B", [11, 16])
def test_tiny_batch_two_token_tiles(B):
    """11 and 16 sessions: the W4 GEMVs run two 8-token MMA column tiles (at 11 the last five columns repeat
    the last session's row and are dropped); the 688-wide FFN's down projection runs as three k-windows
    whose tile sums meet in global memory."""
    wl = Workload(f"tiny-b{B}", TINY, KV_FP16, B, tuple(range(3, 3 + B * 9, 9)), scattered_pool=True)
    _run_decode(wl, 14, n_steps=2 if B == 11 else 1)


@pytest.mark.parametrize("dt", [KV_FP16, KV_INT8, KV_INT4])
def test_kv_append_bytes_and_placement_bit_exact(dt):
    shape = shrink(TINY, n_layers=2)
    wl = Workload("kv", shape, dt, 2, (37, 50), scattered_pool=True)
    P = 10
    ctx = driver.create(wl, 5, pool_blocks=P, max_context=200)
    order = synth.pool_order(5, P)
    model = oracle.PoolModel(P, 16, order)
    cfg = model_cfg(shape, dt)
    kvs = []
    for i, n in enumerate(wl.prior):
        sid = ctx.session_open()
        model.open(sid)
        kv = oracle.KV(cfg, 64)
        driver.append_prior(ctx, sid, shape, 5, i, n, chunk=20, keep=lambda k, v, kv=kv: kv.append(k, v))
        assert model.append(sid, n)
        kvs.append((sid, kv, n))
    ptr, nbytes = ctx.debug_pool()
    assert nbytes == 2 * P * oracle.kv_block_bytes(2, 64, dt)
    torch.cuda.synchronize()
    host = device_bytes(ptr, nbytes).cpu().numpy()
    H, d = 2, 64
    for sid, kv, n in kvs:
        for t in range(n):
            blk, slot = model.locate(sid, t)
            for l in range(2):
                loc = ctx.debug_kv_locate(sid, l, t)
                assert loc[4] == blk
                for h in range(H):
                    for which in (0, 1):
                        off = oracle.kv_offset(H, d, dt, 16, P, l, blk, which, h, slot)
                        data, meta = kv.stored(l, which, t, h)
                        assert off == loc[which] + h * 16 * len(data)
                        assert np.array_equal(host[off:off + len(data)], data), (sid, t, l, h, which)
                        if len(meta):
                            moff = oracle.kv_offset(H, d, dt, 16, P, l, blk, 2 + which, h, slot)
                            assert moff == loc[2 + which] + h * 16 * len(meta)
                            assert np.array_equal(host[moff:moff + len(meta)], meta), (sid, t, l, h, which)


def test_arena_plan_offsets_match_oracle():
    for flags in (0, mag.FLAG_ARENA_NO_REUSE):
        wl = Workload("arena", TINY, KV_FP16, 16, (10,) * 16)
        ctx = driver.create(wl, 1, flags=flags)
        plan, total = ctx.debug_arena_plan(0)
        sizes = [t["size"] for t in plan]
        first = [t["first"] for t in plan]
        last = [t["last"] for t in plan]
        if flags:
            # preserve-all: every tensor has its own bytes
            ends = sorted((t["offset"], t["offset"] + t["size"]) for t in plan)
            assert all(a[1] <= b[0] for a, b in zip(ends, ends[1:]))
            assert total == ctx.memory_stats()["arena_bytes"]
            continue
        off, arena = oracle.arena_plan(sizes, first, last, 64, closed=True)
        assert [t["offset"] for t in plan] == off.tolist()
        assert total == arena
        st = ctx.memory_stats()
        assert st["arena_bytes"] == total and st["arena_unshared_bytes"] == sum(sizes)


def test_host_errors_leave_state_unchanged():
    wl = Workload("err", TINY, KV_FP16, 2, (30,))
    ctx = driver.create(wl, 2, pool_blocks=3, max_context=40)
    sid = ctx.session_open()
    k = torch.zeros((1, 40, 2, 64), dtype=torch.float16, device="cuda")
    x = torch.zeros((2, 256), dtype=torch.float16, device="cuda")
    out = torch.zeros((2, 256), dtype=torch.float16, device="cuda")
    with pytest.raises(mag.MagError) as e:
        ctx.decode_step([sid], x, out)
    assert e.value.status == mag.ERR_NOT_LOADED
    driver.load_weights(ctx, TINY, 2)
    with pytest.raises(mag.MagError) as e:
        ctx.kv_append(sid, 41, k, k)
    assert e.value.status == mag.ERR_CONTEXT_FULL and ctx.session_length(sid) == 0
    ctx.kv_append(sid, 33, k, k)  # 3 blocks: the pool is now empty
    assert ctx.memory_stats()["pool_blocks_free"] == 0
    sid2 = ctx.session_open()
    with pytest.raises(mag.MagError) as e:
        ctx.kv_append(sid2, 1, k, k)
    assert e.value.status == mag.ERR_KV_FULL and ctx.session_length(sid2) == 0
    with pytest.raises(mag.MagError) as e:
        ctx.decode_step([sid, sid2], x, out)  # sid2 needs a block at token 0
    assert e.value.status == mag.ERR_KV_FULL and ctx.session_length(sid) == 33
    with pytest.raises(mag.MagError) as e:
        ctx.decode_step([sid, sid], x, out)
    assert e.value.status == mag.ERR_INVALID_ARG
    with pytest.raises(mag.MagError) as e:
        ctx.decode_step([7], x, out)
    assert e.value.status == mag.ERR_INVALID_ARG
    ctx.session_close(sid2)
    ctx.decode_step([sid], x[:1], out[:1])  # token 33 fits block 3 of the session
    ctx.sync()
    assert ctx.session_length(sid) == 34
    for _ in range(6):
        ctx.decode_step([sid], x[:1], out[:1])
    with pytest.raises(mag.MagError) as e:
        ctx.decode_step([sid], x[:1], out[:1])  # 40 tokens: at max_context
    assert e.value.status == mag.ERR_CONTEXT_FULL
    ctx.session_close(sid)
    assert ctx.memory_stats()["pool_blocks_free"] == 3


def test_decode_step_host_buffers():
    ctx, _ = _run_decode(TINY_DECODE, 15, n_steps=1)
    # a second context fed through host buffers gives the same output as the device-buffer call
    wl = TINY_DECODE
    ctx2, sids2 = driver.setup(wl, 15)
    ctx3, sids3 = driver.setup(wl, 15)
    x = driver.step_inputs(wl, 15, 0)
    out_h = np.empty((1, wl.shape.hidden), np.float16)
    ctx2.decode_step_host(sids2, x, out_h)
    out_d = torch.empty((1, wl.shape.hidden), dtype=torch.float16, device="cuda")
    ctx3.decode_step(sids3, torch.from_numpy(x).cuda(), out_d)
    ctx3.sync()
    assert np.array_equal(out_h.view(np.uint16), out_d.cpu().numpy().view(np.uint16))
