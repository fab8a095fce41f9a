"""GPU parity at the 8B shape (32 layers, D 4096, 32/8 heads, d 128, F 14336, V 128256).

* 8B decode, batch 1, FP16 KV at context 2048 -- the configuration the bench
  times -- with every projection's packed bytes checked bit-exactly against
  the oracle's quantiser, and the logits of two consecutive steps against the
  oracle's full 32-layer step.
* Agent batch: 16 sessions, log-uniform contexts 20..2048, KV blocks
  scattered through a shared pool; the same with INT8 and INT4 KV on two
  layers.
* Long context, FP16 at 19,431 / INT8 at 38,863 / INT4 at 77,726 tokens (the
  capacities "5. Core modules" 5.4 prints): the full contexts, all 32 layers
  and the full vocabulary; one token with the default attention blocks, the
  next with the wide ones over two clusters per KV head.
* Layer by layer (teacher forced): the step's fp32 residual after every layer
  is read back (mag_debug_step_residuals) and the oracle runs each layer alone
  from the GPU's residual at that layer's input; every layer's output hidden
  state and its own contribution (output minus input), and the logits from the
  GPU's final residual, are held to the strict bar. The graph-replayed step
  the bench times gives the same logits, bit for bit, as that eager step.
Tolerance on fp16 logits and hidden states: max-abs <= 2e-2 and rel-L2 <= 1e-3
-- except that for the logits of the whole 32-layer step (not teacher forced)
rel-L2 is bounded by 1.25 x the oracle's own change under a one-ulp change of
one input value (measured in the test, about 2e-3): no implementation that
differs from the oracle in a single fp16 rounding can do better than that floor.
"""
import numpy as np
import pytest
import torch

import oracle
import quantized_decode_step_gb300 as mag
import synth
from synth import driver
from synth.workloads import DECODE_8B, KV_FP16, KV_INT4, KV_INT8, LLAMA8B, Workload, agent_batch, shrink
from tests.helpers import FLOOR_FACTOR, TOL_MAX_ABS, TOL_REL_L2, max_abs, model_cfg, one_ulp_floor, rel_l2

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

SEED = 7
_cache = {}


@pytest.fixture(scope="module", autouse=True)
def built():
    mag.build()
    assert torch.cuda.is_available()


def _oracle_weights_and_ctx(wl: Workload, seed=SEED, check_bytes=True, **kw):
    """Create a context, load the seeded fp32 weights through the device quantiser, and quantise the same
    draws with the oracle (cached per shape). With check_bytes every projection's device bytes are compared
    with the oracle's."""
    shape = wl.shape
    ctx = driver.create(wl, seed, **kw)
    key = (shape.name, seed)
    if key in _cache:
        w = _cache[key]
        # the oracle's bytes were shown equal to the device quantiser's in the first load: load them packed
        for l in range(shape.n_layers):
            for name, tid in driver.PROJ:
                p, sm = getattr(w, name)[l], getattr(w, "s" + name[1:])[l]
                buf = torch.from_numpy(np.concatenate([p.reshape(-1), sm.view(np.uint8).reshape(-1)])).cuda()
                ctx.load_weights(tid, l, buf, mag.FMT_W4G32, buf.numel())
                torch.cuda.synchronize()
        for l in range(shape.n_layers):
            for g, tid in ((w.gamma1[l], mag.NORM_ATTN), (w.gamma2[l], mag.NORM_FFN)):
                ctx.load_weights(tid, l, torch.from_numpy(g).cuda(), mag.FMT_F16, g.size * 2)
        ctx.load_weights(mag.NORM_FINAL, 0, torch.from_numpy(w.gamma_f).cuda(), mag.FMT_F16, w.gamma_f.size * 2)
        lm = torch.from_numpy(w.lm_head).cuda()
        ctx.load_weights(mag.LM_HEAD, 0, lm, mag.FMT_F16, lm.numel() * 2)
        torch.cuda.synchronize()
        return ctx, w
    w = oracle.Weights()
    mismatches = []

    def keep(l, name, f32):
        p, sm = oracle.w4g32_quantize(f32)
        getattr(w, name).append(p)
        getattr(w, "s" + name[1:]).append(sm)

    driver.load_weights(ctx, shape, seed, keep_f32=keep)
    for l in range(shape.n_layers):
        w.gamma1.append(synth.norm_gain_f16(seed, f"L{l}.g1", shape.hidden))
        w.gamma2.append(synth.norm_gain_f16(seed, f"L{l}.g2", shape.hidden))
        if check_bytes:
            for name, tid in driver.PROJ:
                p, sm = getattr(w, name)[l], getattr(w, "s" + name[1:])[l]
                ref = torch.from_numpy(np.concatenate([p.reshape(-1), sm.view(np.uint8).reshape(-1)])).cuda()
                got = torch.empty_like(ref)
                ctx.debug_read_weights(tid, l, got, got.numel())
                torch.cuda.synchronize()
                if not torch.equal(got, ref):
                    mismatches.append((l, name))
    w.gamma_f = synth.norm_gain_f16(seed, "gf", shape.hidden)
    w.lm_head = synth.lm_head_f16(seed, shape.vocab, shape.hidden)
    assert not mismatches, f"device W4 bytes differ from the oracle's: {mismatches[:5]}"
    _cache[key] = w
    return ctx, w


def _priors(ctx, wl: Workload, seed=SEED):
    cfg = model_cfg(wl.shape, wl.kv_dtype)
    sids, kvs = [], []
    for i, p in enumerate(wl.prior):
        sid = ctx.session_open()
        kv = oracle.KV(cfg, p + 8)
        driver.append_prior(ctx, sid, wl.shape, seed, i, p, keep=lambda k, v, kv=kv: kv.append(k, v))
        sids.append(sid)
        kvs.append(kv)
    return sids, kvs, cfg


def _clone_kvs(cfg, kvs, wl, seed=SEED):
    """Fresh oracle stores holding the same priors (for the sensitivity runs)."""
    out = []
    for i, p in enumerate(wl.prior):
        kv = oracle.KV(cfg, p + 8)
        L, H, d = wl.shape.n_layers, wl.shape.n_kv_heads, wl.shape.head_dim
        for t0 in range(0, p, 4096):
            n = min(4096, p - t0)
            k = np.empty((L, n, H, d), np.float16)
            v = np.empty((L, n, H, d), np.float16)
            for l in range(L):
                k[l] = synth.prior_kv_f16(seed, i, l, "K", n, H, d, tok0=t0)
                v[l] = synth.prior_kv_f16(seed, i, l, "V", n, H, d, tok0=t0)
            kv.append(k, v)
        out.append(kv)
    return out


def _steps(ctx, w, wl, sids, kvs, cfg, n_steps, seed=SEED, floor_check=False):
    c, s = oracle.rope_table(max(wl.prior) + n_steps + 1, wl.shape.head_dim, wl.shape.rope_base)
    res = []
    bar = TOL_REL_L2
    for step in range(n_steps):
        x = driver.step_inputs(wl, seed, step)
        out = torch.empty((wl.batch, wl.shape.vocab), dtype=torch.float16, device="cuda")
        ctx.decode_step(sids, torch.from_numpy(x).cuda(), out)
        ctx.sync()
        got = out.cpu().numpy().astype(np.float64)
        if floor_check and step == 0:
            # the oracle's sensitivity to one fp16 ulp of one input value, from stores at the same state
            def run(xx):
                return oracle.forward(cfg, w, _clone_kvs(cfg, kvs, wl, seed), [1] * wl.batch, xx, c, s)
            floor, _ = one_ulp_floor(run, x)
            bar = max(TOL_REL_L2, FLOOR_FACTOR * floor)
            print(f"{wl.name}: one-ulp sensitivity of the oracle {floor:.3e} -> rel-L2 bar {bar:.3e}")
        ref = oracle.forward(cfg, w, kvs, [1] * wl.batch, x, c, s).astype(np.float64)
        assert np.all(np.isfinite(got))
        ma, rl = max_abs(got, ref), rel_l2(got, ref)
        print(f"{wl.name} step {step}: max-abs {ma:.3e} rel-L2 {rl:.3e}")
        assert ma <= TOL_MAX_ABS and rl <= bar, (wl.name, step, ma, rl, bar)
        # the top-1 token agrees wherever the oracle's margin exceeds the tolerance
        for b in range(wl.batch):
            top = np.argsort(ref[b])[-2:]
            if ref[b, top[1]] - ref[b, top[0]] > 2 * TOL_MAX_ABS:
                assert int(np.argmax(got[b])) == int(top[1])
        res.append((ma, rl))
    return res


def _layerwise_step(ctx, w, wl, sids, kvs, cfg, step, seed=SEED, graph_check=True):
    """One decode step through mag_debug_step_residuals, checked layer by layer against the oracle fed the
    GPU's residual at each layer's input; then the logits from the GPU's final residual. With graph_check
    the sessions are cut back and the same step is replayed through the captured graph (the bench's launch
    path): its logits must equal the eager step's bit for bit."""
    shape, B = wl.shape, wl.batch
    L, D = shape.n_layers, shape.hidden
    rows = max(wl.prior) + step + 2
    c, s = oracle.rope_table(rows, shape.head_dim, shape.rope_base)
    x = driver.step_inputs(wl, seed, step)
    xt = torch.from_numpy(x).cuda()
    out = torch.empty((B, shape.vocab), dtype=torch.float16, device="cuda")
    resid = torch.empty((L + 1, B, D), dtype=torch.float32, device="cuda")
    lens = [ctx.session_length(sid) for sid in sids]
    ctx.step_residuals(sids, xt, out, resid)
    R = resid.cpu().numpy().astype(np.float64)
    got = out.cpu().numpy()
    assert np.array_equal(R[0], x.astype(np.float64)), "row 0 is the fp16 input"
    worst = [0.0, 0.0, 0.0]
    for l in range(L):
        ref = oracle.layer(cfg, w, l, kvs, [1] * B, R[l], c, s)
        ma, rl = max_abs(R[l + 1], ref), rel_l2(R[l + 1], ref)
        dl = rel_l2(R[l + 1] - R[l], ref - R[l])  # the layer's own contribution
        worst = [max(worst[0], ma), max(worst[1], rl), max(worst[2], dl)]
        assert ma <= TOL_MAX_ABS and rl <= TOL_REL_L2 and dl <= TOL_REL_L2, (wl.name, step, l, ma, rl, dl)
    for kv in kvs:
        kv.commit(1)
    ref = oracle.output(cfg, w, R[L]).astype(np.float64)
    ma, rl = max_abs(got, ref), rel_l2(got, ref)
    print(f"{wl.name} step {step} layer by layer: hidden max-abs {worst[0]:.2e} rel-L2 {worst[1]:.2e}, "
          f"layer contribution rel-L2 {worst[2]:.2e} (worst of {L}); logits max-abs {ma:.2e} rel-L2 {rl:.2e}")
    assert ma <= TOL_MAX_ABS and rl <= TOL_REL_L2, (wl.name, step, "logits", ma, rl)
    if graph_check:
        for sid, n in zip(sids, lens):
            ctx.session_truncate(sid, n)
        out2 = torch.empty_like(out)
        ctx.decode_step(sids, xt, out2)
        ctx.sync()
        assert torch.equal(out2.view(torch.int16), out.view(torch.int16)), "graph step differs from the eager step"
    return worst, (ma, rl)


def test_8b_layerwise_decode_b1_ctx2048_fp16():
    """The bench's configuration, all 32 layers, teacher forced at the strict bar; two steps."""
    wl = DECODE_8B
    ctx, w = _oracle_weights_and_ctx(wl, extra_tokens=3)
    sids, kvs, cfg = _priors(ctx, wl)
    for step in range(2):
        _layerwise_step(ctx, w, wl, sids, kvs, cfg, step)


def test_8b_layerwise_agent_batch16():
    """The agent batch (16 sessions, contexts 20..2048, scattered pool), all 32 layers, teacher forced."""
    wl = agent_batch(SEED)
    ctx, w = _oracle_weights_and_ctx(wl, extra_tokens=2)
    sids, kvs, cfg = _priors(ctx, wl)
    _layerwise_step(ctx, w, wl, sids, kvs, cfg, 0)


def test_8b_decode_b1_ctx2048_fp16():
    wl = DECODE_8B
    ctx, w = _oracle_weights_and_ctx(wl, extra_tokens=2)
    sids, kvs, cfg = _priors(ctx, wl)
    _steps(ctx, w, wl, sids, kvs, cfg, 2, floor_check=True)
    st = ctx.memory_stats()
    assert st["weight_bytes"] >= 5_413_281_792


def test_8b_agent_batch16_scattered_pool():
    wl = agent_batch(SEED)
    assert wl.batch == 16 and min(wl.prior) >= 20 and max(wl.prior) <= 2048
    ctx, w = _oracle_weights_and_ctx(wl)
    sids, kvs, cfg = _priors(ctx, wl)
    _steps(ctx, w, wl, sids, kvs, cfg, 1, floor_check=True)


@pytest.mark.parametrize("dt", [KV_INT8, KV_INT4])
def test_8b_agent_batch16_quantized_kv(dt):
    """The agent batch (16 sessions, contexts 20..2048, scattered pool) with INT8 / INT4 KV, on two of the 32
    layers with the full vocabulary (strict bar)."""
    base = agent_batch(SEED)
    wl = Workload(f"8b2L-b16-agent-kv{dt}", shrink(LLAMA8B, n_layers=2), dt, base.batch, base.prior,
                  scattered_pool=True)
    ctx, w = _oracle_weights_and_ctx(wl, check_bytes=False)
    sids, kvs, cfg = _priors(ctx, wl)
    _steps(ctx, w, wl, sids, kvs, cfg, 1)


@pytest.mark.parametrize("n", [8, 6])
def test_8b_two_layers_agent_batch_k_split(n):
    """8 and 6 sessions of the agent batch on two layers (FP16, strict bar): the W4 GEMVs with one 8-token
    column tile, the whole K of QKV / O / gate-up staged per block and the down projection as 4 k-windows of
    56 chunks; the fp16 LM head's k-split with four tiles per warp and a ragged last block."""
    base = agent_batch(SEED)
    wl = Workload(f"8b2L-b{n}-agent-fp16", shrink(LLAMA8B, n_layers=2), KV_FP16, n, base.prior[:n],
                  scattered_pool=True)
    ctx, w = _oracle_weights_and_ctx(wl, check_bytes=False)
    sids, kvs, cfg = _priors(ctx, wl)
    _steps(ctx, w, wl, sids, kvs, cfg, 1)


def test_8b_two_layers_strict():
    """Two of the 32 layers with the full vocabulary: the strict bar holds at this depth."""
    shape = shrink(LLAMA8B, n_layers=2)
    wl = Workload("8b2L-ctx2048-fp16", shape, KV_FP16, 1, (2048,))
    ctx, w = _oracle_weights_and_ctx(wl, check_bytes=False, extra_tokens=2)
    sids, kvs, cfg = _priors(ctx, wl)
    _steps(ctx, w, wl, sids, kvs, cfg, 2)


@pytest.mark.parametrize("dt,ctx_len", [(KV_FP16, 19431), (KV_INT8, 38863), (KV_INT4, 77726)])
def test_8b_long_context_kv_precision(dt, ctx_len):
    """The long-context configurations at full size (32 layers, full vocabulary), teacher forced layer by
    layer: one token with the default attention blocks, the next through the long plan's wide blocks with
    32 splits as two clusters merged by the last block to finish."""
    wl = Workload(f"8b-ctx{ctx_len}-kv{dt}", LLAMA8B, dt, 1, (ctx_len,))
    ctx, w = _oracle_weights_and_ctx(wl, check_bytes=False, extra_tokens=2)
    sids, kvs, cfg = _priors(ctx, wl)
    _layerwise_step(ctx, w, wl, sids, kvs, cfg, 0)
    ctx.set_adaptive(True, force_plan=2, plan_splits=(4, 8, 32), plan_wide=(0, 0, 1))
    assert ctx.profile()["plan_wide"] == 1 and ctx.profile()["plan_splits"] == 32
    _layerwise_step(ctx, w, wl, sids, kvs, cfg, 1)
