"""GPU parity of the multi-token verify step (mag_verify_tokens) and of session truncation.

The verify step runs n draft tokens of one session and returns the output of every token; token j attends
causally to the session's cache and tokens 0..j. It has two engines: with n <= max_batch a decode step
whose rows are the drafts (their keys and values stored between the QKV projection and attention), else
the prefill chunk path. Its reference is the oracle fed the same tokens one at a time (each a one-token
forward on the growing store), which is the same causal computation. After a verify step the caller
keeps the accepted prefix with mag_session_truncate: a decode step then reads exactly the cache of
prior + accepted tokens, compared with the oracle on a store built from the prior and the accepted
tokens alone.

* Tiny layer (no LM head: hidden outputs), both engines, FP16 / INT8 / INT4 pools: 4 drafts on a
  126-token cache (the drafts cross into a new block), 2 or 0 accepted, one decode step after; block
  accounting across the truncation. On the decode engine also 4 drafts from a block boundary (the new
  block holds them all) and 6 drafts (the k-split GEMVs of batches above 4).
* Two 8B-shaped layers with the full vocabulary, 4 drafts on an 800-token FP16 cache, both engines.
* Argument errors: more drafts than either engine takes, truncation past the length, a closed session.
"""
import numpy as np
import pytest
import torch

import oracle
import quantized_decode_step_gb300 as mag
import synth
from synth import driver
from synth.workloads import KV_FP16, KV_INT4, KV_INT8, LLAMA8B, TINY, Workload, shrink
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
    print(f"{what}: max-abs {ma:.3e} rel-L2 {rl:.3e}")
    assert ma <= TOL_MAX_ABS and rl <= TOL_REL_L2, f"{what}: max-abs {ma:.3e}, rel-L2 {rl:.3e}"


class _Oracle:
    """The oracle's weights, RoPE tables and a store holding the session's prior."""

    def __init__(self, wl: Workload, seed: int, random_gain: bool, extra: int):
        self.shape, self.p = wl.shape, wl.prior[0]
        self.w = oracle_weights(self.shape, seed, random_gain)
        self.cfg = model_cfg(self.shape, wl.kv_dtype)
        self.cap = self.p + extra + 8
        self.k, self.v = prior_kv(self.shape, seed, 0, self.p) if self.p else (None, None)
        self.c, self.s = oracle.rope_table(self.p + extra + 2, self.shape.head_dim, self.shape.rope_base)

    def store(self):
        kv = oracle.KV(self.cfg, self.cap)
        if self.p:
            kv.append(self.k, self.v)
        return kv

    def tokens(self, kv, x):
        """Outputs of the rows of x fed one at a time to the store kv (which they extend)."""
        if x.shape[0] == 0:
            return np.empty((0, self.shape.vocab or self.shape.hidden), np.float16)
        return np.stack([oracle.forward(self.cfg, self.w, [kv], [1], x[j:j + 1], self.c, self.s)[0]
                         for j in range(x.shape[0])])


def _verify_then_accept(wl: Workload, seed: int, n_draft: int, n_keep: int, random_gain: bool, on_step: bool):
    shape = wl.shape
    ctx, sids = driver.setup(wl, seed, random_gain=random_gain, extra_tokens=n_draft + 1)
    sid, p = sids[0], wl.prior[0]
    orc = _Oracle(wl, seed, random_gain, n_draft + 1)
    width = shape.vocab or shape.hidden
    x = synth.hidden_f16(seed, n_draft, shape.hidden, tag="drafts")
    free0 = ctx.memory_stats()["pool_blocks_free"]
    out = torch.empty((n_draft, width), dtype=torch.float16, device="cuda")
    ctx.verify_tokens(sid, n_draft, torch.from_numpy(x).cuda(), out)
    ctx.sync()
    # the decode engine: step prologue, 6 kernels per layer (QKV, KV store, attention, O, gate-up, down)
    # and the LM head; the chunk engine runs 8 per layer
    assert (ctx.last_step_launches() == 2 + 6 * shape.n_layers) == on_step
    assert ctx.session_length(sid) == p + n_draft
    ref = orc.tokens(orc.store(), x)
    for j in range(n_draft):
        _compare(out[j].cpu().numpy(), ref[j], f"{wl.name} draft {j} of {n_draft}")
    # keep the first n_keep drafts, then decode the next token on the shortened cache
    ctx.session_truncate(sid, p + n_keep)
    assert ctx.session_length(sid) == p + n_keep
    blocks_used = lambda n: (n + 15) // 16  # noqa: E731
    assert ctx.memory_stats()["pool_blocks_free"] == free0 - (blocks_used(p + n_keep) - blocks_used(p))
    xd = synth.hidden_f16(seed, 1, shape.hidden, tag="after")
    od = torch.empty((1, width), dtype=torch.float16, device="cuda")
    ctx.decode_step([sid], torch.from_numpy(xd).cuda(), od)
    ctx.sync()
    kv = orc.store()
    orc.tokens(kv, x[:n_keep])
    refd = oracle.forward(orc.cfg, orc.w, [kv], [1], xd, orc.c, orc.s)
    _compare(od.cpu().numpy(), refd, f"{wl.name} decode after keeping {n_keep}")
    return ctx, sid


def _workload(name, shape, dt, prior, n_draft, on_step):
    # the decode engine takes up to max_batch drafts; the chunk engine needs max_chunk
    if on_step:
        return Workload(name + "-step", shape, dt, n_draft, (prior,))
    return Workload(name + "-chunk", shape, dt, 1, (prior,), chunk=8)


@pytest.mark.parametrize("on_step", [True, False], ids=["step", "chunk"])
@pytest.mark.parametrize("dt", [KV_FP16, KV_INT8, KV_INT4])
def test_tiny_verify_then_truncate(dt, on_step):
    # 126 prior tokens + 4 drafts cross into a ninth block, which the truncation (to 128 or 126) returns
    wl = _workload(f"tiny-verify-kv{dt}", TINY, dt, 126, 4, on_step)
    _verify_then_accept(wl, 31 + dt, 4, 2, random_gain=True, on_step=on_step)
    ctx, sid = _verify_then_accept(wl, 33 + dt, 4, 0, random_gain=True, on_step=on_step)
    ctx.session_truncate(sid, 0)
    assert ctx.session_length(sid) == 0


@pytest.mark.parametrize("dt", [KV_FP16, KV_INT4])
def test_tiny_verify_from_block_boundary(dt):
    # 128 prior tokens: the step prologue maps a new block that holds all four drafts
    wl = _workload(f"tiny-verify-boundary-kv{dt}", TINY, dt, 128, 4, True)
    _verify_then_accept(wl, 39 + dt, 4, 4, random_gain=True, on_step=True)


def test_tiny_verify_six_drafts():
    # six rows: the GEMVs of batches above four (k-split kernels)
    wl = _workload("tiny-verify-6", TINY, KV_INT8, 75, 6, True)
    _verify_then_accept(wl, 43, 6, 5, random_gain=True, on_step=True)


@pytest.mark.slow
@pytest.mark.parametrize("on_step", [True, False], ids=["step", "chunk"])
def test_8b_two_layers_verify(on_step):
    shape = shrink(LLAMA8B, n_layers=2)
    wl = _workload("8b2L-verify-4-on-800", shape, KV_FP16, 800, 4, on_step)
    _verify_then_accept(wl, 35, 4, 3, random_gain=False, on_step=on_step)


def test_verify_argument_errors():
    wl = Workload("tiny-verify-args", TINY, KV_FP16, 2, (20,), chunk=3)
    ctx, sids = driver.setup(wl, 37, extra_tokens=8)
    sid = sids[0]
    x = torch.zeros((5, TINY.hidden), dtype=torch.float16, device="cuda")
    out = torch.empty((5, TINY.hidden), dtype=torch.float16, device="cuda")
    # max_batch 2, max_chunk 3: four drafts exceed both engines
    with pytest.raises(mag.MagError) as e:
        ctx.verify_tokens(sid, 4, x, out)
    assert e.value.status == mag.ERR_INVALID_ARG
    with pytest.raises(mag.MagError) as e:
        ctx.verify_tokens(sid, 0, x, out)
    assert e.value.status == mag.ERR_INVALID_ARG
    assert ctx.session_length(sid) == 20
    with pytest.raises(mag.MagError) as e:
        ctx.session_truncate(sid, 21)
    assert e.value.status == mag.ERR_INVALID_ARG
    assert ctx.session_length(sid) == 20
    ctx.session_close(sid)
    with pytest.raises(mag.MagError) as e:
        ctx.verify_tokens(sid, 2, x, out)
    assert e.value.status == mag.ERR_INVALID_ARG
    with pytest.raises(mag.MagError) as e:
        ctx.session_truncate(sid, 0)
    assert e.value.status == mag.ERR_INVALID_ARG
