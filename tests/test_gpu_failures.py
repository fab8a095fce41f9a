"""Failure detection on the GPU without a GPU fault ("Magnitude" 5.1-5.2: the engine's error behaviour).

* A decode GEMV whose pipeline waits give up (mag_debug_set_wait_limit(0): every main-loop wait for a weight
  copy gives up at its first poll, as if the copy were stuck): the kernel sets its bit in the error word,
  waits for the copies it has in flight within the built-in bound and returns; mag_sync reports
  MAG_ERR_TIMEOUT, and with the limit restored and the step's token dropped the context decodes on
  against the oracle. Nothing waits without a bound, so nothing can hang.
* The prefill GEMM's waits give up the same way (every role: the activation and weight copies, the
  expansion, the MMA thread, the epilogue). Each copy issuer waits for its own copies to land before the
  block exits, the MMA thread for its MMAs, so the block frees its tensor memory with nothing in flight;
  the arrival counters of the split-K merges are reset after the timeout is reported. With the limit
  restored the same chunk, and a decode step after it, match the oracle.
* Allocation failures injected on the host (mag_debug_fail_allocations), never a real out-of-memory:
  - mag_create failing at each of its allocations in turn (fixed and elastic pools, prefill enabled)
    returns MAG_ERR_OOM and leaves the device memory as it found it;
  - an elastic pool that can map no new group: the append that needed it returns MAG_ERR_OOM and changes
    nothing; the same append succeeds once the failure is gone and decode matches the oracle;
  - an fp32 weight load whose scratch can not be allocated returns MAG_ERR_OOM; a step then says
    NOT_LOADED; the load succeeds on retry.
"""
import numpy as np
import pytest
import torch

import oracle
import quantized_decode_step_gb300 as mag
import synth
from synth import driver
from synth.workloads import KV_FP16, TINY, TINY_DECODE, Workload
from tests.helpers import TOL_MAX_ABS, TOL_REL_L2, max_abs, model_cfg, oracle_weights, prior_kv, proj_shape, rel_l2

pytestmark = pytest.mark.gpu

SEED = 41


@pytest.fixture(scope="module", autouse=True)
def built():
    mag.build()
    assert torch.cuda.is_available()
    yield
    mag.debug_fail_allocations(0, 0)


def _check_vs_oracle(got, ref, what):
    a, b = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    assert np.all(np.isfinite(a)), what
    ma, rl = max_abs(a, b), rel_l2(a, b)
    assert ma <= TOL_MAX_ABS and rl <= TOL_REL_L2, f"{what}: max-abs {ma:.3e}, rel-L2 {rl:.3e}"


@pytest.mark.parametrize("flags", [0, mag.FLAG_NO_GRAPH], ids=["graph", "eager"])
def test_pipeline_wait_gives_up_then_context_recovers(flags):
    wl = TINY_DECODE
    ctx, sids = driver.setup(wl, SEED, flags=flags, extra_tokens=4)
    sid, p = sids[0], wl.prior[0]
    shape = wl.shape
    out = torch.empty((1, shape.hidden), dtype=torch.float16, device="cuda")
    x0 = torch.from_numpy(driver.step_inputs(wl, SEED, 0)).cuda()
    ctx.decode_step([sid], x0, out)  # a first step under the built-in limit (its graph is captured)
    ctx.sync()
    ctx.session_truncate(sid, p)
    ctx.set_wait_limit(0)
    ctx.decode_step([sid], x0, out)
    with pytest.raises(mag.MagError) as e:
        ctx.sync()
    assert e.value.status == mag.ERR_TIMEOUT and "gave up" in str(e.value)
    ctx.sync()  # the error word was read and cleared
    # the built-in limit again; the step's token (computed from nothing) is dropped
    ctx.set_wait_limit(-1)
    ctx.session_truncate(sid, p)
    cfg = model_cfg(shape, wl.kv_dtype)
    kv = oracle.KV(cfg, p + 8)
    kv.append(*prior_kv(shape, SEED, 0, p))
    w = oracle_weights(shape, SEED)
    c, s = oracle.rope_table(p + 8, shape.head_dim, shape.rope_base)
    for step in range(2):
        x = driver.step_inputs(wl, SEED, step)
        ctx.decode_step([sid], torch.from_numpy(x).cuda(), out)
        ctx.sync()
        ref = oracle.forward(cfg, w, [kv], [1], x, c, s)
        _check_vs_oracle(out.cpu().numpy(), ref, f"step {step} after the timeout")
    ctx.close()


def test_prefill_wait_gives_up_then_context_recovers():
    wl = Workload("tiny-prefill-timeout", TINY, KV_FP16, 1, (128,), chunk=64)
    shape, T = wl.shape, 48
    ctx, sids = driver.setup(wl, SEED, extra_tokens=T + 4)
    sid, p = sids[0], wl.prior[0]
    x = synth.hidden_f16(SEED, T, shape.hidden, tag="timeout-chunk")
    out = torch.empty(shape.hidden, dtype=torch.float16, device="cuda")
    ctx.set_wait_limit(0)
    ctx.prefill_chunk(sid, T, torch.from_numpy(x).cuda(), out)
    with pytest.raises(mag.MagError) as e:
        ctx.sync()
    assert e.value.status == mag.ERR_TIMEOUT and "gave up" in str(e.value)
    ctx.sync()
    ctx.set_wait_limit(-1)
    ctx.session_truncate(sid, p)
    cfg = model_cfg(shape, wl.kv_dtype)
    kv = oracle.KV(cfg, p + T + 8)
    kv.append(*prior_kv(shape, SEED, 0, p))
    w = oracle_weights(shape, SEED)
    c, s = oracle.rope_table(p + T + 8, shape.head_dim, shape.rope_base)
    ctx.prefill_chunk(sid, T, torch.from_numpy(x).cuda(), out)
    ctx.sync()
    assert ctx.session_length(sid) == p + T
    _check_vs_oracle(out.cpu().numpy(), oracle.forward(cfg, w, [kv], [T], x, c, s)[0], "the chunk after the timeout")
    x1 = synth.hidden_f16(SEED, 1, shape.hidden, tag="timeout-after")
    out1 = torch.empty((1, shape.hidden), dtype=torch.float16, device="cuda")
    ctx.decode_step([sid], torch.from_numpy(x1).cuda(), out1)
    ctx.sync()
    _check_vs_oracle(out1.cpu().numpy(), oracle.forward(cfg, w, [kv], [1], x1, c, s), "the step after the chunk")
    ctx.close()


def _free_bytes():
    torch.cuda.synchronize()
    return torch.cuda.mem_get_info()[0]


@pytest.mark.parametrize("flags,max_chunk", [(0, 0), (0, 64), (mag.FLAG_ELASTIC_POOL, 64)],
                         ids=["fixed", "fixed-prefill", "elastic-prefill"])
def test_create_fails_cleanly_at_every_allocation(flags, max_chunk):
    cfg = mag.make_config(TINY, pool_blocks=64, max_sessions=2, max_batch=2, max_chunk=max_chunk, max_context=512,
                          flags=flags)
    stream = torch.cuda.current_stream().cuda_stream
    mag.Context(cfg, stream).close()  # warm the allocator and the library's module
    free0 = _free_bytes()
    failures = 0
    for i in range(200):
        mag.debug_fail_allocations(i, 1)
        try:
            ctx = mag.Context(cfg, stream)
        except mag.MagError as e:
            assert e.status == mag.ERR_OOM, (i, e.status)
            failures += 1
            continue
        finally:
            mag.debug_fail_allocations(0, 0)
        # allocation i was past the last one create makes: it succeeded and works
        ctx.close()
        break
    else:
        pytest.fail("mag_create made more than 200 allocations")
    assert failures >= 8, failures
    assert abs(_free_bytes() - free0) < 8 << 20, "a failed create left device memory behind"


def test_elastic_group_mapping_failure_changes_nothing():
    shape = TINY
    cfg = mag.make_config(shape, pool_blocks=1024, max_sessions=1, max_batch=1, max_context=8192,
                          flags=mag.FLAG_ELASTIC_POOL)
    ctx = mag.Context(cfg, torch.cuda.current_stream().cuda_stream)
    driver.load_weights(ctx, shape, SEED)
    G = ctx.memory_stats()["pool_group_blocks"]
    n0 = 16 * G  # exactly one group of blocks
    sid = ctx.session_open()
    driver.append_prior(ctx, sid, shape, SEED, 0, n0)
    st0 = ctx.memory_stats()
    k, v = prior_kv(shape, SEED, 1, 40)
    kt, vt = torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda()
    mag.debug_fail_allocations(0, 1)
    try:
        with pytest.raises(mag.MagError) as e:
            ctx.kv_append(sid, 40, kt, vt)
    finally:
        mag.debug_fail_allocations(0, 0)
    assert e.value.status == mag.ERR_OOM
    assert ctx.session_length(sid) == n0
    st1 = ctx.memory_stats()
    assert (st1["pool_blocks_free"], st1["pool_blocks_mapped"]) == (st0["pool_blocks_free"], st0["pool_blocks_mapped"])
    ctx.kv_append(sid, 40, kt, vt)  # now it maps the group
    assert ctx.session_length(sid) == n0 + 40
    assert ctx.memory_stats()["pool_blocks_mapped"] == 2 * G
    ocfg = model_cfg(shape, KV_FP16)
    kv = oracle.KV(ocfg, n0 + 48)
    kv.append(*prior_kv(shape, SEED, 0, n0))
    kv.append(k, v)
    w = oracle_weights(shape, SEED)
    c, s = oracle.rope_table(n0 + 48, shape.head_dim, shape.rope_base)
    x = synth.hidden_f16(SEED, 1, shape.hidden, tag="after")
    out = torch.empty((1, shape.hidden), dtype=torch.float16, device="cuda")
    ctx.decode_step([sid], torch.from_numpy(x).cuda(), out)
    ctx.sync()
    _check_vs_oracle(out.cpu().numpy(), oracle.forward(ocfg, w, [kv], [1], x, c, s), "decode across both groups")
    ctx.close()


def test_weight_load_allocation_failure():
    wl = Workload("tiny-oom-load", TINY, KV_FP16, 1, (16,))
    ctx = driver.create(wl, SEED)
    n, k = proj_shape(TINY, "wgu")
    src = torch.from_numpy(synth.weight_f32(SEED, 0, "wgu", n, k)).cuda()
    mag.debug_fail_allocations(0, 1)
    try:
        with pytest.raises(mag.MagError) as e:
            ctx.load_weights(mag.W_GATE_UP, 0, src, mag.FMT_F32_DENSE, src.numel() * 4)
    finally:
        mag.debug_fail_allocations(0, 0)
    assert e.value.status == mag.ERR_OOM
    # everything else loaded, the gate-up not: a step is refused
    for name, tid in driver.PROJ:
        if tid != mag.W_GATE_UP:
            nn, kk = proj_shape(TINY, name)
            t = torch.from_numpy(synth.weight_f32(SEED, 0, name, nn, kk)).cuda()
            ctx.load_weights(tid, 0, t, mag.FMT_F32_DENSE, t.numel() * 4)
    for tag, tid in (("L0.g1", mag.NORM_ATTN), ("L0.g2", mag.NORM_FFN), ("gf", mag.NORM_FINAL)):
        g = torch.from_numpy(synth.norm_gain_f16(SEED, tag, TINY.hidden)).cuda()
        ctx.load_weights(tid, 0, g, mag.FMT_F16, g.numel() * 2)
    sid = ctx.session_open()
    x = torch.zeros((1, TINY.hidden), dtype=torch.float16, device="cuda")
    out = torch.empty((1, TINY.hidden), dtype=torch.float16, device="cuda")
    with pytest.raises(mag.MagError) as e:
        ctx.decode_step([sid], x, out)
    assert e.value.status == mag.ERR_NOT_LOADED
    assert ctx.session_length(sid) == 0
    ctx.load_weights(mag.W_GATE_UP, 0, src, mag.FMT_F32_DENSE, src.numel() * 4)
    ctx.decode_step([sid], x, out)
    ctx.sync()
    assert torch.isfinite(out.float()).all()
    ctx.close()
