"""Debug aids of the library, on the GPU without a GPU fault.

* mag_get_step_stats: kind, rows, launches, most keys attended and the modelled bytes of the last decode,
  verify and prefill call (weights once, every row's KV, hidden states in and out), and its device time
  with MAG_FLAG_STEP_TIMING (-1 without).
* MAG_FLAG_DEBUG_CANARY: the steps still match the oracle and report nothing; a band changed from the host
  (a plain write of device memory) is reported by the next mag_sync as MAG_ERR_CORRUPT naming the tensor,
  and the steps after it are clean.
* The block-id checks: a block-table entry outside the pool, written on the device only, is not used (the
  attention kernel reads block 0 instead) and the next mag_sync returns MAG_ERR_CORRUPT; the host then
  rewrites the device tables from its own copy, and the same step again matches the oracle.
* The step timeline (mag_debug_timeline): every GEMV and attention launch of the step is there with all its
  blocks and their events in order, and the stamped step's output is the plain step's, bit for bit.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import quantized_decode_step_gb300 as mag
import synth
from synth import driver
from synth.workloads import KV_FP16, TINY, Workload
from tests.helpers import TOL_MAX_ABS, TOL_REL_L2, max_abs, model_cfg, oracle_weights, prior_kv, rel_l2

pytestmark = pytest.mark.gpu

SEED = 53


@pytest.fixture(scope="module", autouse=True)
def built():
    mag.build()
    assert torch.cuda.is_available()


def _check(got, ref, what):
    a, b = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    assert np.all(np.isfinite(a)), what
    ma, rl = max_abs(a, b), rel_l2(a, b)
    assert ma <= TOL_MAX_ABS and rl <= TOL_REL_L2, f"{what}: max-abs {ma:.3e}, rel-L2 {rl:.3e}"


def _writable(ptr, nbytes):
    """A uint8 CUDA tensor aliasing `nbytes` at device address `ptr` (host-side writes through torch)."""
    class _Arr:
        __cuda_array_interface__ = {"shape": (nbytes,), "typestr": "|u1", "data": (ptr, False), "version": 3}
    return torch.as_tensor(_Arr(), device="cuda")


@pytest.mark.parametrize("timing", [True, False])
def test_step_stats(timing):
    wl = Workload("tiny-stats", TINY, KV_FP16, 2, (37, 100), chunk=16)
    flags = mag.FLAG_STEP_TIMING if timing else 0
    ctx, sids = driver.setup(wl, SEED, flags=flags, extra_tokens=32)
    shape = wl.shape
    D = shape.hidden
    cfg = mag.make_config(shape, kv_dtype=KV_FP16)
    per_token = mag.kv_bytes_per_token(cfg)
    wbytes = ctx.memory_stats()["weight_bytes"]
    assert ctx.step_stats()["steps"] == 0
    # decode step of both sessions
    x = torch.from_numpy(synth.hidden_f16(SEED, 2, D, tag="stats0")).cuda()
    out = torch.empty((2, D), dtype=torch.float16, device="cuda")
    ctx.decode_step(sids, x, out)
    st = ctx.step_stats()
    assert (st["steps"], st["last_kind"], st["last_rows"]) == (1, 0, 2)
    assert st["last_launches"] == ctx.last_step_launches() == 1 + 5 * shape.n_layers + 1
    assert st["last_max_keys"] == 101
    assert st["last_bytes"] == wbytes + (38 + 101) * per_token + 2 * D * 2 + 2 * D * 2
    assert (st["last_ms"] > 0) if timing else (st["last_ms"] == -1)
    # verify of 2 drafts of the first session (now 38 tokens)
    xd = torch.from_numpy(synth.hidden_f16(SEED, 2, D, tag="stats1")).cuda()
    ctx.verify_tokens(sids[0], 2, xd, out)
    st = ctx.step_stats()
    assert (st["steps"], st["last_kind"], st["last_rows"], st["last_max_keys"]) == (2, 1, 2, 40)
    assert st["last_bytes"] == wbytes + (39 + 40) * per_token + 2 * D * 2 + 2 * D * 2
    # a prefill chunk of 8 tokens on the second session (now 101 tokens)
    xc = torch.from_numpy(synth.hidden_f16(SEED, 8, D, tag="stats2")).cuda()
    o1 = torch.empty(D, dtype=torch.float16, device="cuda")
    ctx.prefill_chunk(sids[1], 8, xc, o1)
    st = ctx.step_stats()
    assert (st["steps"], st["last_kind"], st["last_rows"], st["last_max_keys"]) == (3, 2, 8, 109)
    assert st["last_launches"] == ctx.last_step_launches()
    assert st["last_bytes"] == wbytes + 109 * per_token + 8 * D * 2 + 1 * D * 2
    assert (st["last_ms"] > 0) if timing else (st["last_ms"] == -1)
    ctx.sync()
    ctx.close()


def _oracle_setup(shape, p, extra):
    cfg = model_cfg(shape, KV_FP16)
    kv = oracle.KV(cfg, p + extra + 8)
    kv.append(*prior_kv(shape, SEED, 0, p))
    c, s = oracle.rope_table(p + extra + 8, shape.head_dim, shape.rope_base)
    return cfg, kv, c, s


def test_canary_bands_report_a_stray_write():
    wl = Workload("tiny-canary", TINY, KV_FP16, 1, (40,))
    shape, p = wl.shape, wl.prior[0]
    ctx, sids = driver.setup(wl, SEED, flags=mag.FLAG_DEBUG_CANARY, extra_tokens=8)
    sid = sids[0]
    cfg, kv, c, s = _oracle_setup(shape, p, 8)
    w = oracle_weights(shape, SEED)
    out = torch.empty((1, shape.hidden), dtype=torch.float16, device="cuda")

    def step(i):
        x = synth.hidden_f16(SEED, 1, shape.hidden, tag=f"canary{i}")
        ctx.decode_step([sid], torch.from_numpy(x).cuda(), out)
        return x

    x = step(0)
    ctx.sync()
    assert ctx.last_step_launches() == 1 + 5 * shape.n_layers + 1 + 1  # + the band check
    _check(out.cpu().numpy(), oracle.forward(cfg, w, [kv], [1], x, c, s), "step 0 with canaries")
    base, nbytes = ctx.debug_arena()
    plan = {t["name"]: t for t in ctx.debug_arena_plan(0)[0]}
    t = plan["qkv"]
    assert t["offset"] + t["size"] <= nbytes
    # a stray byte in the band after the qkv tensor (its last 64 bytes)
    band = _writable(base + t["offset"] + t["size"] - 64, 64)
    band[5] = 0
    torch.cuda.synchronize()
    x = step(1)
    with pytest.raises(mag.MagError) as e:
        ctx.sync()
    assert e.value.status == mag.ERR_CORRUPT and "qkv" in str(e.value)
    # the band is not the tensor: the step itself computed correctly, and its token stays
    _check(out.cpu().numpy(), oracle.forward(cfg, w, [kv], [1], x, c, s), "step 1 (reported)")
    x = step(2)
    ctx.sync()  # the bands were rewritten: clean again
    _check(out.cpu().numpy(), oracle.forward(cfg, w, [kv], [1], x, c, s), "step 2 after the report")
    ctx.close()


def test_block_id_outside_the_pool_is_not_used():
    wl = Workload("tiny-bounds", TINY, KV_FP16, 1, (40,))
    shape, p = wl.shape, wl.prior[0]
    ctx, sids = driver.setup(wl, SEED, extra_tokens=8)
    sid = sids[0]
    P = ctx.memory_stats()["pool_blocks_total"]
    cfg, kv, c, s = _oracle_setup(shape, p, 8)
    w = oracle_weights(shape, SEED)
    out = torch.empty((1, shape.hidden), dtype=torch.float16, device="cuda")
    x = synth.hidden_f16(SEED, 1, shape.hidden, tag="bounds0")
    ctx.debug_set_table_entry(sid, 0, P + 7)
    ctx.decode_step([sid], torch.from_numpy(x).cuda(), out)
    with pytest.raises(mag.MagError) as e:
        ctx.sync()
    assert e.value.status == mag.ERR_CORRUPT and "block-table entry" in str(e.value)
    # the device tables came back from the host's copy: the same step again matches the oracle
    ctx.session_truncate(sid, p)
    ctx.decode_step([sid], torch.from_numpy(x).cuda(), out)
    ctx.sync()
    _check(out.cpu().numpy(), oracle.forward(cfg, w, [kv], [1], x, c, s), "the step after the report")
    ctx.close()


@pytest.mark.parametrize("shape", [TINY, dataclasses.replace(TINY, name="tiny-2L-v512", n_layers=2, vocab=512)])
def test_timeline(shape):
    from quantized_decode_step_gb300 import timeline as tl
    wl = Workload("tiny-timeline", shape, KV_FP16, 1, (37,))
    ctx, sids = driver.setup(wl, SEED, extra_tokens=8)
    sid, p = sids[0], wl.prior[0]
    x = torch.from_numpy(synth.hidden_f16(SEED, 1, shape.hidden, tag="tl0")).cuda()
    width = shape.vocab or shape.hidden
    out1 = torch.empty((1, width), dtype=torch.float16, device="cuda")
    out2 = torch.empty_like(out1)
    ctx.decode_step([sid], x, out1)
    ctx.sync()
    ctx.session_truncate(sid, p)
    recs = torch.zeros((4096, 4), dtype=torch.int64, device="cuda")
    n = ctx.timeline([sid], x, out2, recs)
    assert ctx.session_length(sid) == p + 1
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16)), "the stamps changed the step"
    assert 0 < n <= recs.shape[0]
    R = recs[:n].cpu().numpy()
    Ls = tl.launches(R)
    kinds = [L["kind"][0] for L in Ls]
    assert kinds.count(tl.ATTN) == shape.n_layers
    assert kinds.count(tl.GEMV) == 4 * shape.n_layers + (1 if shape.vocab else 0)
    for L in Ls:
        evs = (0, 1, 2) if L["kind"][0] == tl.GEMV else (0, 1, 2, 3)
        assert all(len(L["ev"][e]) == len(L["blocks"]) for e in evs), L["kind"]
    # a block's records in time order: its events in order, once per launch of its tag (launches of one tag
    # are layers apart)
    by_block = {}
    for tag, blk, ev, t in sorted(R.tolist(), key=lambda r: (r[3], r[2])):
        by_block.setdefault((tag, blk), []).append(ev)
    n_of_tag = {}
    for L in Ls:
        n_of_tag[L["tag"]] = n_of_tag.get(L["tag"], 0) + 1
    for (tag, blk), evs in by_block.items():
        one = [0, 1, 2] if (tag >> 60) == tl.GEMV else [0, 1, 2, 3]
        assert evs == one * n_of_tag[tag], (hex(tag), blk, evs)
    rows = tl.phases(Ls)
    assert len(rows) == len(Ls) and rows[0]["entry_first"] == 0.0
    ctx.close()

