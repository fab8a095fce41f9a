"""GPU checks of the adaptive runtime ("Magnitude" 3.1-3.3): plans (decode-attention split counts, one
set of captured graphs each), the load profile that picks them, and the hot pool target.

* Every plan forced in turn on a 3-session ragged batch (FP16 and INT4 pools), decode and verify
  steps against the oracle: a plan changes only how attention splits the keys and how many warps a
  block has (4, or the wide blocks).
* Plans chosen by the profile (window 8, every step recorded): short-context steps switch to the short
  plan once the window is full, long-context ones to the long plan; the switch points, the profile's
  quantiles and the hot pool target agree with the oracle's window fed the same lengths; outputs
  match the oracle throughout. The same with the switch captured on a background thread.
* Argument errors of mag_set_adaptive.
"""
import time

import numpy as np
import pytest
import torch

import oracle
import quantized_decode_step_gb300 as mag
import synth
from oracle import adapt
from synth import driver
from synth.workloads import KV_FP16, KV_INT4, TINY, Workload
from tests.helpers import TOL_MAX_ABS, TOL_REL_L2, max_abs, model_cfg, oracle_weights, prior_kv, rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    mag.build()
    assert torch.cuda.is_available()


def _compare(got, ref, what):
    a, b = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    assert np.all(np.isfinite(a)), what
    ma, rl = max_abs(a, b), rel_l2(a, b)
    assert ma <= TOL_MAX_ABS and rl <= TOL_REL_L2, f"{what}: max-abs {ma:.3e}, rel-L2 {rl:.3e}"


class _Run:
    """A context and the oracle's stores of its sessions, stepped together."""

    def __init__(self, wl: Workload, seed: int, extra: int):
        self.wl, self.seed, self.shape = wl, seed, wl.shape
        self.ctx, self.sids = driver.setup(wl, seed, random_gain=True, extra_tokens=extra)
        self.w = oracle_weights(self.shape, seed, True)
        self.cfg = model_cfg(self.shape, wl.kv_dtype)
        self.kvs = []
        for i, p in enumerate(wl.prior):
            kv = oracle.KV(self.cfg, p + extra + 8)
            if p:
                kv.append(*prior_kv(self.shape, seed, i, p))
            self.kvs.append(kv)
        self.c, self.s = oracle.rope_table(max(wl.prior) + extra + 2, self.shape.head_dim, self.shape.rope_base)
        self.width = self.shape.vocab or self.shape.hidden
        self.n = 0

    def decode(self, rows, what):
        x = synth.hidden_f16(self.seed, len(rows), self.shape.hidden, tag=f"s{self.n}")
        self.n += 1
        out = torch.empty((len(rows), self.width), dtype=torch.float16, device="cuda")
        self.ctx.decode_step([self.sids[i] for i in rows], torch.from_numpy(x).cuda(), out)
        self.ctx.sync()
        ref = oracle.forward(self.cfg, self.w, [self.kvs[i] for i in rows], [1] * len(rows), x, self.c, self.s)
        _compare(out.cpu().numpy(), ref, what)

    def verify(self, i, n, what):
        x = synth.hidden_f16(self.seed, n, self.shape.hidden, tag=f"v{self.n}")
        self.n += 1
        out = torch.empty((n, self.width), dtype=torch.float16, device="cuda")
        self.ctx.verify_tokens(self.sids[i], n, torch.from_numpy(x).cuda(), out)
        self.ctx.sync()
        for j in range(n):
            ref = oracle.forward(self.cfg, self.w, [self.kvs[i]], [1], x[j:j + 1], self.c, self.s)[0]
            _compare(out[j].cpu().numpy(), ref, f"{what} draft {j}")

    def length(self, i):
        return self.ctx.session_length(self.sids[i])


@pytest.mark.parametrize("dt", [KV_FP16, KV_INT4])
def test_forced_plans_match_oracle(dt):
    wl = Workload(f"tiny-plans-kv{dt}", TINY, dt, 3, (40, 300, 1000))
    run = _Run(wl, 51 + dt, extra=20)
    # plan 2 spreads each (session, KV head) over 3 clusters of 16 (48 splits), merged by the last block
    splits, wide = (1, 3, 48), (0, 1, 1)
    for p in (0, 1, 2, 0):
        run.ctx.set_adaptive(True, force_plan=p, plan_splits=splits, plan_wide=wide)
        prof = run.ctx.profile()
        assert prof["plan"] == p and prof["plan_splits"] == splits[p]
        assert prof["plan_wide"] == wide[p]
        run.decode([0, 1, 2], f"{wl.name} plan {p} decode")
        run.verify(1, 3, f"{wl.name} plan {p} verify")
    # off again: the default plan
    run.ctx.set_adaptive(False)
    assert run.ctx.profile()["plan"] == 1
    run.decode([0, 1, 2], f"{wl.name} adaptive off")


def _profile_switching(async_switch: bool):
    wl = Workload(f"tiny-switch-async{int(async_switch)}", TINY, KV_FP16, 2, (20, 700))
    run = _Run(wl, 61 + int(async_switch), extra=40)
    splits = (2, 4, 8)
    run.ctx.set_adaptive(True, adaptive_window_size=8, adaptive_sample_rate=1, plan_splits=splits,
                         async_switch=int(async_switch))
    win = adapt.LoadWindow(8, 1)
    plan, pending = 1, None  # the oracle's view: plan in use and a switch on its way
    n_open = 2

    def settle():
        # a background capture ends by itself; the library takes its plan at the next call
        if not async_switch:
            return run.ctx.profile()
        for _ in range(500):
            prof = run.ctx.profile()
            if prof["pending_plan"] == -1:
                return prof
            time.sleep(0.01)
        raise AssertionError("background capture did not finish")

    for k, i in enumerate([0] * 10 + [1] * 10):
        run.decode([i], f"{wl.name} step {k}")
        win.observe(run.length(i))
        if win.full():
            want = adapt.plan_for(win.quantile(0.9))
            if pending is None and want != plan:
                pending = want
        prof = settle()
        if pending is not None:
            plan, pending = pending, None
        assert prof["plan"] == plan, (k, prof)
        assert prof["recorded"] == len(win.values)
        assert (prof["p50"], prof["p90"], prof["p99"]) == (win.quantile(0.5), win.quantile(0.9), win.quantile(0.99))
        if win.full():
            assert prof["hot_blocks"] == adapt.hot_pool_blocks(win.quantile(0.9), n_open, "1.2")
        assert prof["plan_splits"] == splits[plan]
    assert prof["switches"] == 2  # medium -> short (short contexts), then -> long
    assert plan == 2


def test_profile_switches_plans():
    _profile_switching(False)


def test_profile_switches_plans_async():
    _profile_switching(True)


def test_set_adaptive_argument_errors():
    wl = Workload("tiny-adapt-args", TINY, KV_FP16, 1, (10,))
    ctx, _ = driver.setup(wl, 71)
    bad = [dict(adaptive_window_size=0), dict(adaptive_sample_rate=0), dict(plan_short_below=600, plan_long_above=500),
           dict(plan_splits=(0, 65, 0)), dict(plan_splits=(-1, 0, 0)), dict(force_plan=3),
           dict(hot_pool_slack=0.5)]
    for kw in bad:
        with pytest.raises(mag.MagError) as e:
            ctx.set_adaptive(True, **kw)
        assert e.value.status == mag.ERR_INVALID_ARG, kw
    assert ctx.profile()["seen"] == 0
