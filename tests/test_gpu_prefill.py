"""GPU parity of the chunked prefill (mag_prefill_chunk).

* Tiny layer (FFN 688: ragged K and a ragged gate-up tile; G = 2; d = 64) with
  FP16 / INT8 / INT4 KV: two chunks (37 tokens, one partial 128-row tile; 150
  tokens, two tiles) on a 128-token cache, then one decode step. The output
  of each chunk's last token and of the decode step (which reads every key the
  chunks stored) against the oracle's causal forward pass.
* A chunk on an empty cache (position 0 onwards).
* Two 8B-shaped layers with the full vocabulary: a 64-token chunk on an
  800-token FP16 / INT8 / INT4 cache against the oracle (quantised pools then
  also decode one token). With a quantised pool the chunk's own k and v go
  through the quantiser, where one fp16 ulp upstream can move a code; there
  the rel-L2 bar for the chunk and the step after it is 1.25 x the oracle's
  own change under one ulp of one input value per token (measured in the
  test), as for the 32-layer decode.
* The 8B chunked-prefill configuration's own chunk (512 tokens on an 800-token
  FP16 cache, full vocabulary) on two layers against the oracle's forward
  pass: the last token's logits, every stored key and value of the chunk at
  both layers (within the tolerance), and the prior cache bit-exact.
* The same configuration at full size (32 layers), teacher forced: the chunk's
  fp32 residuals after every layer are read back (mag_debug_prefill_residuals);
  the oracle runs sampled layers alone from the GPU's residual at their input
  (all 512 tokens, causal over the cache and the chunk) and the final norm and
  LM head from the GPU's last residual, all at the strict bar. (Each oracle
  layer of 512 tokens costs several seconds of CPU, so not all 32 run.)
* Also at full size: the chunk's last logits against the same 512 tokens
  decoded one by one on the GPU (a property of any correct prefill; bar: the
  two paths' own distance to the oracle at 32 layers, each about 2e-3).
"""
import numpy as np
import pytest
import torch

import oracle
import quantized_decode_step_gb300 as mag
import synth
from synth import driver
from synth.workloads import KV_FP16, KV_INT4, KV_INT8, LLAMA8B, PREFILL_8B, TINY, Workload, shrink
from tests.helpers import (FLOOR_FACTOR, TOL_MAX_ABS, TOL_REL_L2, device_bytes, fp16_ulps, max_abs, model_cfg,
                           one_ulp_floor, oracle_weights, prior_kv, rel_l2)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    mag.build()
    assert torch.cuda.is_available()


def _compare(got, ref, what, bar=TOL_REL_L2):
    a, b = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    assert np.all(np.isfinite(a)), what
    ma, rl = max_abs(a, b), rel_l2(a, b)
    print(f"{what}: max-abs {ma:.3e} rel-L2 {rl:.3e}")
    assert ma <= TOL_MAX_ABS and rl <= bar, f"{what}: max-abs {ma:.3e}, rel-L2 {rl:.3e}"


def _run(wl: Workload, seed: int, chunks, decode_after=1, random_gain=True, floor_check=False):
    shape = wl.shape
    total = sum(chunks) + decode_after
    ctx, sids = driver.setup(wl, seed, random_gain=random_gain, extra_tokens=total)
    sid = sids[0]
    w = oracle_weights(shape, seed, random_gain)
    cfg = model_cfg(shape, wl.kv_dtype)
    p = wl.prior[0]
    kv = oracle.KV(cfg, p + total + 8)
    if p:
        k, v = prior_kv(shape, seed, 0, p)
        kv.append(k, v)
    c, s = oracle.rope_table(p + total + 2, shape.head_dim, shape.rope_base)
    width = shape.vocab or shape.hidden
    pos = p
    bar = TOL_REL_L2
    for i, T in enumerate(chunks):
        x = synth.hidden_f16(seed, T, shape.hidden, tag=f"chunk{i}")
        out = torch.empty(width, dtype=torch.float16, device="cuda")
        ctx.prefill_chunk(sid, T, torch.from_numpy(x).cuda(), out)
        ctx.sync()
        pos += T
        assert ctx.session_length(sid) == pos
        if floor_check and i == 0:
            # a quantised pool stores the chunk's own k and v through the quantiser, so one fp16 ulp of
            # difference upstream can move a code: the bar is the oracle's own change under one ulp of one
            # input value per token, from a store holding only the prior
            def run(xx, T=T):
                kv2 = oracle.KV(cfg, p + total + 8)
                if p:
                    kv2.append(k, v)
                return oracle.forward(cfg, w, [kv2], [T], xx, c, s)[0]
            floor, _ = one_ulp_floor(run, x)
            bar = max(TOL_REL_L2, FLOOR_FACTOR * floor)
            print(f"{wl.name}: one-ulp sensitivity of the oracle {floor:.3e} -> rel-L2 bar {bar:.3e}")
        ref = oracle.forward(cfg, w, [kv], [T], x, c, s)[0]
        _compare(out.cpu().numpy(), ref, f"{wl.name} chunk {i} ({T} tokens)", bar)
    for j in range(decode_after):
        x = synth.hidden_f16(seed, 1, shape.hidden, tag=f"after{j}")
        out = torch.empty((1, width), dtype=torch.float16, device="cuda")
        ctx.decode_step([sid], torch.from_numpy(x).cuda(), out)
        ctx.sync()
        ref = oracle.forward(cfg, w, [kv], [1], x, c, s)
        # the step reads the chunk's stored keys and values: the same bar as the chunk
        _compare(out.cpu().numpy(), ref, f"{wl.name} decode after the chunks", bar)
    return ctx


@pytest.mark.parametrize("dt", [KV_FP16, KV_INT8, KV_INT4])
def test_tiny_prefill_chunks_then_decode(dt):
    wl = Workload(f"tiny-prefill-kv{dt}", TINY, dt, 1, (128,), chunk=160)
    ctx = _run(wl, 21 + dt, (37, 150))
    st = ctx.memory_stats()
    # the prefill GEMMs read the W4 tiles themselves: no weight copy
    assert st["prefill_weight_bytes"] == 0 and st["prefill_arena_bytes"] > 0


def test_tiny_prefill_on_empty_cache():
    wl = Workload("tiny-prefill-empty", TINY, KV_FP16, 1, (0,), chunk=40)
    _run(wl, 25, (40,), decode_after=2)


def test_prefill_unsupported_without_max_chunk():
    wl = Workload("tiny-no-chunk", TINY, KV_FP16, 1, (16,))
    ctx, sids = driver.setup(wl, 26)
    assert ctx.memory_stats()["prefill_weight_bytes"] == 0
    x = torch.zeros((4, TINY.hidden), dtype=torch.float16, device="cuda")
    out = torch.empty(TINY.hidden, dtype=torch.float16, device="cuda")
    with pytest.raises(mag.MagError) as e:
        ctx.prefill_chunk(sids[0], 4, x, out)
    assert e.value.status == mag.ERR_UNSUPPORTED
    assert ctx.session_length(sids[0]) == 16


@pytest.mark.slow
@pytest.mark.parametrize("dt", [KV_FP16, KV_INT8, KV_INT4])
def test_8b_two_layers_prefill_chunk(dt):
    shape = shrink(LLAMA8B, n_layers=2)
    wl = Workload(f"8b2L-prefill-64-on-800-kv{dt}", shape, dt, 1, (800,), chunk=64)
    _run(wl, 27, (64,), decode_after=1 if dt else 0, random_gain=False, floor_check=dt != KV_FP16)


def _pool_host(ctx):
    ptr, nbytes = ctx.debug_pool()
    torch.cuda.synchronize()
    return device_bytes(ptr, nbytes).cpu().numpy()


def _stored_vec(host, ctx, sid, l, t, h, which, vec_bytes):
    off = ctx.debug_kv_locate(sid, l, t)[which] + h * 16 * vec_bytes
    return host[off:off + vec_bytes]


@pytest.mark.slow
def test_8b_prefill_512_on_800_two_layers_vs_oracle():
    """The configuration's chunk (512 tokens at positions 800..1311, FP16 cache, full vocabulary) on two of
    the 32 layers: four 128-row token tiles per weight tile, the 1312-key causal attention, and the chunk's
    keys and values written into the pool ("5. Core modules" 5.2)."""
    wl0 = PREFILL_8B
    shape = shrink(wl0.shape, n_layers=2)
    wl = Workload("8b2L-prefill-512-on-800", shape, KV_FP16, 1, wl0.prior, chunk=wl0.chunk)
    seed, T, p = 29, wl.chunk, wl.prior[0]
    ctx, sids = driver.setup(wl, seed, extra_tokens=T)
    sid = sids[0]
    x = synth.hidden_f16(seed, T, shape.hidden, tag="chunk0")
    out = torch.empty(shape.vocab, dtype=torch.float16, device="cuda")
    ctx.prefill_chunk(sid, T, torch.from_numpy(x).cuda(), out)
    ctx.sync()
    assert ctx.session_length(sid) == p + T
    w = oracle_weights(shape, seed)
    cfg = model_cfg(shape, KV_FP16)
    kv = oracle.KV(cfg, p + T)
    kv.append(*prior_kv(shape, seed, 0, p))
    c, s = oracle.rope_table(p + T + 1, shape.head_dim, shape.rope_base)
    ref = oracle.forward(cfg, w, [kv], [T], x, c, s)[0]
    _compare(out.cpu().numpy(), ref, f"{wl.name} last-token logits")
    host = _pool_host(ctx)
    H, d, vb = shape.n_kv_heads, shape.head_dim, 2 * shape.head_dim
    for t in range(0, p, 37):  # the prior cache, as appended
        for l in range(2):
            for h in range(H):
                for which in (0, 1):
                    assert np.array_equal(_stored_vec(host, ctx, sid, l, t, h, which, vb),
                                          kv.stored(l, which, t, h)[0]), (t, l, h, which)
    for l in range(2):
        got = np.empty((T, H, 2, d), np.float16)
        exp = np.empty_like(got)
        for i in range(T):
            for h in range(H):
                for which in (0, 1):
                    got[i, h, which] = _stored_vec(host, ctx, sid, l, p + i, h, which, vb).view(np.float16)
                    exp[i, h, which] = kv.stored(l, which, p + i, h)[0].view(np.float16)
        assert np.all(np.isfinite(got.astype(np.float32)))
        # placement: a key or value read from the wrong block or slot would be unrelated N(0, 1)-scale
        # data; the values themselves come out of an fp32 GEMM (the oracle's is double), are rounded to
        # fp16, and keys are rotated and rounded again, so they are held to the tolerance
        u = fp16_ulps(got, exp)
        print(f"{wl.name} layer {l} stored K / V: {np.mean(u[:, :, 0] == 0):.4f} / {np.mean(u[:, :, 1] == 0):.4f} "
              f"bit-identical")
        _compare(got, exp, f"{wl.name} layer {l} stored K/V of the chunk")


@pytest.mark.slow
def test_8b_prefill_512_on_800_layerwise():
    """The configuration at full size, 32 layers, teacher forced on sampled layers (see the module note)."""
    wl = PREFILL_8B
    shape, T, p = wl.shape, wl.chunk, wl.prior[0]
    seed = 30
    sample = (1, 16, 31)
    ctx, sids = driver.setup(wl, seed, extra_tokens=T)
    sid = sids[0]
    x = synth.hidden_f16(seed, T, shape.hidden, tag="chunk0")
    out = torch.empty(shape.vocab, dtype=torch.float16, device="cuda")
    resid = torch.empty((shape.n_layers + 1, T, shape.hidden), dtype=torch.float32, device="cuda")
    ctx.prefill_residuals(sid, T, torch.from_numpy(x).cuda(), out, resid)
    R = resid.cpu().numpy().astype(np.float64)
    got = out.cpu().numpy()
    del resid
    assert np.array_equal(R[0], x.astype(np.float64))
    cfg = model_cfg(shape, KV_FP16)
    w = oracle_weights(shape, seed, layers=sample)
    # oracle weights of the sampled layers only: index them as layers 0..2 of a 3-layer model
    c, s = oracle.rope_table(p + T + 1, shape.head_dim, shape.rope_base)
    k_all, v_all = prior_kv(shape, seed, 0, p)
    sub = shrink(shape, n_layers=len(sample))
    scfg = model_cfg(sub, KV_FP16)
    kv = oracle.KV(scfg, p + T)
    kv.append(np.ascontiguousarray(k_all[list(sample)]), np.ascontiguousarray(v_all[list(sample)]))
    for j, l in enumerate(sample):
        ref = oracle.layer(scfg, w, j, [kv], [T], R[l], c, s)
        ma, rl = max_abs(R[l + 1], ref), rel_l2(R[l + 1], ref)
        dl = rel_l2(R[l + 1] - R[l], ref - R[l])
        print(f"{wl.name} layer {l}: hidden max-abs {ma:.2e} rel-L2 {rl:.2e}, layer contribution rel-L2 {dl:.2e}")
        assert ma <= TOL_MAX_ABS and rl <= TOL_REL_L2 and dl <= TOL_REL_L2, (l, ma, rl, dl)
    ref = oracle.output(model_cfg(shape, KV_FP16), w, R[shape.n_layers][-1:])[0]
    _compare(got, ref, f"{wl.name} logits from the final residual")


@pytest.mark.slow
def test_8b_prefill_512_on_800_matches_token_by_token_decode():
    wl = PREFILL_8B
    shape, T, p = wl.shape, wl.chunk, wl.prior[0]
    seed = 28
    x = synth.hidden_f16(seed, T, shape.hidden, tag="chunk0")
    width = shape.vocab
    # the chunk at once
    ctx, sids = driver.setup(wl, seed, extra_tokens=T)
    out_p = torch.empty(width, dtype=torch.float16, device="cuda")
    ctx.prefill_chunk(sids[0], T, torch.from_numpy(x).cuda(), out_p)
    ctx.sync()
    assert ctx.session_length(sids[0]) == p + T
    got_p = out_p.cpu().numpy().astype(np.float64)
    ctx.close()
    torch.cuda.empty_cache()
    # the same tokens one decode step at a time
    wl_d = Workload(wl.name + "-decode", shape, wl.kv_dtype, 1, wl.prior)
    ctx, sids = driver.setup(wl_d, seed, extra_tokens=T)
    xd = torch.from_numpy(x).cuda()
    out_d = torch.empty((1, width), dtype=torch.float16, device="cuda")
    for t in range(T):
        ctx.decode_step([sids[0]], xd[t:t + 1], out_d)
    ctx.sync()
    got_d = out_d.cpu().numpy()[0].astype(np.float64)
    ctx.close()
    assert np.all(np.isfinite(got_p)) and np.all(np.isfinite(got_d))
    ma, rl = max_abs(got_p, got_d), rel_l2(got_p, got_d)
    print(f"{wl.name}: prefill vs token-by-token decode: max-abs {ma:.3e} rel-L2 {rl:.3e}")
    assert ma <= TOL_MAX_ABS and rl <= 5e-3
    top = np.argsort(got_d)[-2:]
    if got_d[top[1]] - got_d[top[0]] > 2 * TOL_MAX_ABS:
        assert int(np.argmax(got_p)) == int(top[1])


def _run_batch(wl: Workload, seed: int, ntok, random_gain=True, decode_after=True, bar=TOL_REL_L2):
    """Several sessions' chunks in one mag_prefill_batch call, then one decode step of all of them."""
    shape = wl.shape
    ctx, sids = driver.setup(wl, seed, random_gain=random_gain, extra_tokens=max(ntok) + 2)
    w = oracle_weights(shape, seed, random_gain)
    cfg = model_cfg(shape, wl.kv_dtype)
    kvs = []
    for i, p in enumerate(wl.prior):
        kv = oracle.KV(cfg, p + max(ntok) + 8)
        if p:
            kv.append(*prior_kv(shape, seed, i, p))
        kvs.append(kv)
    c, s = oracle.rope_table(max(wl.prior) + max(ntok) + 4, shape.head_dim, shape.rope_base)
    width = shape.vocab or shape.hidden
    xs = [synth.hidden_f16(seed, n, shape.hidden, tag=f"batch{i}") for i, n in enumerate(ntok)]
    out = torch.empty((len(sids), width), dtype=torch.float16, device="cuda")
    ctx.prefill_batch(sids, list(ntok), torch.from_numpy(np.concatenate(xs)).cuda(), out)
    ctx.sync()
    got = out.cpu().numpy()
    for i, (sid, p, n) in enumerate(zip(sids, wl.prior, ntok)):
        assert ctx.session_length(sid) == p + n
        ref = oracle.forward(cfg, w, [kvs[i]], [n], xs[i], c, s)[0]
        _compare(got[i], ref, f"{wl.name} session {i} ({p} + {n} tokens)", bar)
    if decode_after:
        x = synth.hidden_f16(seed, len(sids), shape.hidden, tag="after")
        od = torch.empty((len(sids), width), dtype=torch.float16, device="cuda")
        ctx.decode_step(sids, torch.from_numpy(x).cuda(), od)
        ctx.sync()
        ref = oracle.forward(cfg, w, kvs, [1] * len(sids), x, c, s)
        _compare(od.cpu().numpy(), ref, f"{wl.name} decode of every session after the batch", bar)
    return ctx, sids


@pytest.mark.parametrize("dt", [KV_FP16, KV_INT8, KV_INT4])
def test_tiny_prefill_batch_of_sessions(dt):
    # three sessions (128-token cache, empty, 37-token cache) with 37, 20 and 64 new tokens: ragged tiles,
    # a session from position 0, one that crosses blocks
    wl = Workload(f"tiny-prefill-batch-kv{dt}", TINY, dt, 3, (128, 0, 37), chunk=160)
    _run_batch(wl, 91 + dt, (37, 20, 64))


def test_tiny_prefill_batch_errors_change_nothing():
    wl = Workload("tiny-prefill-batch-args", TINY, KV_FP16, 2, (10, 20), chunk=16)
    ctx, sids = driver.setup(wl, 95, extra_tokens=16)
    x = torch.zeros((16, TINY.hidden), dtype=torch.float16, device="cuda")
    out = torch.empty((2, TINY.hidden), dtype=torch.float16, device="cuda")
    free0 = ctx.memory_stats()["pool_blocks_free"]
    for ids, nt in (([sids[0], sids[0]], [4, 4]), (sids, [10, 7]), (sids, [4, 0]), ([sids[0], 99], [4, 4])):
        with pytest.raises(mag.MagError) as e:
            ctx.prefill_batch(ids, nt, x, out)
        assert e.value.status == mag.ERR_INVALID_ARG, (ids, nt)
    assert [ctx.session_length(s) for s in sids] == [10, 20]
    assert ctx.memory_stats()["pool_blocks_free"] == free0


@pytest.mark.slow
def test_8b_two_layers_prefill_batch():
    shape = shrink(LLAMA8B, n_layers=2)
    wl = Workload("8b2L-prefill-batch", shape, KV_FP16, 2, (800, 300), chunk=128)
    _run_batch(wl, 97, (64, 40), random_gain=False)
