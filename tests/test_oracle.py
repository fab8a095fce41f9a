"""Pins of the oracle against what the pages and the mathematics fix (CPU only).

Each test checks the oracle against something other than itself: a value the
pages print, a closed form, an invariant, a hand-computed case, a special case
that reduces to a library routine, or brute force on tiny inputs.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import synth
from synth.workloads import TINY, shrink
from tests.helpers import fp16_ulps, model_cfg, oracle_weights, prior_kv, rel_l2

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ----------------------------------------------------------------------------- fp16

def test_fp16_matches_numpy_rounding():
    rng = np.random.default_rng(1)
    x = np.concatenate([
        rng.standard_normal(200000).astype(np.float32) * np.float32(10.0) ** rng.integers(-9, 6, 200000),
        np.array([0.0, -0.0, 65504, 65519.99, 65520, 65536, 1e9, -1e9, 2.0 ** -24, 2.0 ** -25, 2.0 ** -25 * 1.0001,
                  3 * 2.0 ** -25, 2.0 ** -14, 2.0 ** -14 * (1 - 2.0 ** -11), np.inf, -np.inf], dtype=np.float32),
        # exact ties between fp16 neighbours
        (np.arange(1, 2000, dtype=np.float32) * np.float32(2.0 ** -11) + np.float32(1.0)),
    ]).astype(np.float32)
    ours = oracle.f32_to_f16(x).view(np.uint16)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(ours, ref)
    assert oracle.f64_to_f16_bits(float("nan")) & 0x7C00 == 0x7C00
    # a double just above a tie rounds up (no double rounding through fp32)
    d = 1.0 + 2.0 ** -11 + 2.0 ** -40
    assert oracle.f64_to_f16_bits(d) == np.float16(1.0 + 2.0 ** -10).view(np.uint16)


# ----------------------------------------------------------------------------- 4-bit weights

def test_w4g32_hand_examples():
    g = golden("w4g32_hand.json")
    for case in g["cases"]:
        x = np.array(case["x"], dtype=np.float32)[None, :]
        packed, sm = oracle.w4g32_quantize(x)
        assert [f"{b:02x}" for b in packed[0]] == case["bytes"], case["name"]
        assert f"{int(sm.view(np.uint16)[0, 0, 0]):04x}" == case["scale_bits"], case["name"]
        assert f"{int(sm.view(np.uint16)[0, 0, 1]):04x}" == case["min_bits"], case["name"]


def test_w4g32_ragged_last_group():
    """A row of 48 values: a full group, then a 16-value group whose statistics cover only its own values."""
    g = golden("w4g32_hand.json")["cases"]
    x = np.array(g[0]["x"] + g[3]["x"][:16], dtype=np.float32)[None, :]
    packed, sm = oracle.w4g32_quantize(x)
    assert packed.shape == (1, 32) and sm.shape == (1, 2, 2)
    assert [f"{b:02x}" for b in packed[0, :16]] == g[0]["bytes"]
    # values -1.5 .. 6.0 step 0.5: lo -1.5, hi 6.0, s = 0.5, codes 0..15, padding codes 0
    assert [f"{b:02x}" for b in packed[0, 16:]] == ["10", "32", "54", "76", "98", "ba", "dc", "fe"] + ["00"] * 8
    assert sm.view(np.uint16)[0, 1].tolist() == [0x3800, 0xBE00]
    y = oracle.w4_gemv(packed, sm, np.ones((1, 48), np.float16))
    assert y[0, 0] == float(np.sum(x))


def test_w4g32_invariants_random():
    w = synth.weight_f32(7, 0, "inv", 96, 512)
    packed, sm = oracle.w4g32_quantize(w)
    lo = packed & 15
    hi = packed >> 4
    assert lo.max() <= 15 and hi.max() <= 15
    deq = oracle.w4g32_dequant(packed, sm)
    s = sm[..., 0].astype(np.float32).repeat(32, axis=1)
    m = sm[..., 1].astype(np.float32).repeat(32, axis=1)
    # every value inside the representable range [m, m + 15 s] is reconstructed within half a step
    inside = (w >= m) & (w <= m + 15 * s)
    err = np.abs(deq - w)
    assert np.all(err[inside] <= s[inside] * 0.5 * (1 + 1e-5) + 1e-7)
    # outside it (fp16 rounding of min and scale moves the ends) the error is bounded by the end's shift
    gmin = w.reshape(96, -1, 32).min(-1).repeat(32, axis=1)
    gmax = w.reshape(96, -1, 32).max(-1).repeat(32, axis=1)
    slack = np.abs(m - gmin) + np.abs(m + 15 * s - gmax)
    assert np.all(err <= s * 0.5 * (1 + 1e-5) + slack + 1e-7)
    # the group's extremes map to codes 0 and 15 (up to the fp16 rounding of m and s)
    q = np.stack([lo, hi], -1).reshape(96, 512)
    qg = q.reshape(96, -1, 32)
    assert np.all(qg.min(-1) <= 1) and np.all(qg.max(-1) >= 14)


def test_w4g32_round_trip_on_grid():
    rng = np.random.default_rng(3)
    rows = []
    for _ in range(64):
        s = np.float16(rng.uniform(0.001, 0.01))
        m = np.float16(rng.uniform(-0.1, 0.0))
        q = rng.integers(0, 16, 32)
        q[0], q[1] = 0, 15
        x = np.float32(s) * q.astype(np.float32) + np.float32(m)  # exact: small integers times an fp16 value
        rows.append(x)
    w = np.stack(rows).astype(np.float32)
    packed, sm = oracle.w4g32_quantize(w)
    deq = oracle.w4g32_dequant(packed, sm)
    # range/15 may round the scale to a neighbouring fp16 value; codes then still reproduce x
    # within that one-ulp scale change times 15
    s_rec = sm[:, 0, 0].astype(np.float32)[:, None]
    assert np.all(np.abs(deq - w) <= 15 * np.abs(s_rec) * 2.0 ** -10 + 1e-8)


def test_w4_gemv_matches_library_matmul_and_fold():
    w = synth.weight_f32(5, 0, "gemv", 200, 320)
    x = synth.hidden_f16(5, 3, 320)
    packed, sm = oracle.w4g32_quantize(w)
    y = oracle.w4_gemv(packed, sm, x)
    deq = oracle.w4g32_dequant(packed, sm).astype(np.float64)
    ref = x.astype(np.float64) @ deq.T  # numpy matmul over the explicitly dequantised matrix
    assert np.allclose(y, ref, rtol=0, atol=1e-12)
    for t in range(3):
        yf = oracle.w4_gemv_folded(packed, sm, x[t])
        assert np.allclose(yf, y[t], rtol=0, atol=1e-12)


# ----------------------------------------------------------------------------- KV quantisers

def test_kv_int8_hand_examples():
    g = golden("kv_int8_hand.json")
    for case in g["cases"]:
        x = np.array(case["x"], dtype=np.float16)[None, :]
        q, s = oracle.kv_quant_int8(x)
        assert q[0].tolist() == case["q"], case["name"]
        assert f"{int(s.view(np.uint16)[0]):04x}" == case["scale_bits"], case["name"]


def test_kv_int8_invariants():
    x = synth.normal(9, "int8", (500, 128), dtype=np.float16)
    q, s = oracle.kv_quant_int8(x)
    assert np.abs(q.astype(np.int32)).max() <= 127
    sf = s.astype(np.float32)[:, None]
    rec = q.astype(np.float32) * sf
    amax = np.abs(x.astype(np.float32)).max(1, keepdims=True)
    # the fp16 scale may sit a little below amax/127, in which case the top codes clip
    bound = sf * 0.5 * (1 + 1e-3) + np.maximum(amax - 127 * sf, 0)
    assert np.all(np.abs(rec - x.astype(np.float32)) <= bound)


def test_kv_int4_is_the_weight_format_along_head_dim():
    x = synth.normal(11, "int4", (40, 128), dtype=np.float16)
    p4, sm4 = oracle.kv_quant_int4(x)
    pw, smw = oracle.w4g32_quantize(x.astype(np.float32))
    assert np.array_equal(p4, pw) and np.array_equal(sm4.view(np.uint16), smw.view(np.uint16))


# ----------------------------------------------------------------------------- pool and closed forms

def test_kv_bytes_per_token_and_capacity_printed():
    g = golden("kv_capacity.json")["printed"]
    gib = 2.0 ** 30
    bpt = oracle.kv_bytes_per_token(g["layers"], g["kv_heads"], g["head_dim"], 2)
    assert bpt == g["bytes_per_token_fp16"] == 131072
    w = golden("kv_capacity.json")["weights_bytes_reading"]
    caps = {k: oracle.kv_max_context(8 * gib, 0.8 * gib, w, oracle.kv_bytes_per_token(32, 8, 128, b))
            for k, b in (("fp16", 2), ("int8", 1), ("int4", 0.5))}
    assert caps == g["capacity"]
    # with the budget read as exactly 2.37 GiB the same formula lands within 0.1% of the printed values
    for k, b in (("fp16", 2), ("int8", 1), ("int4", 0.5)):
        c = oracle.kv_max_context(g["budget_gib"] * gib, 0, 0, oracle.kv_bytes_per_token(32, 8, 128, b))
        assert abs(c - g["capacity"][k]) / g["capacity"][k] < 1e-3


def test_pool_block_bytes_and_offsets_hand():
    assert oracle.kv_block_bytes(8, 128, oracle.KV_FP16) == 2 * 8 * 16 * 128 * 2 == 65536
    assert oracle.kv_block_bytes(8, 128, oracle.KV_INT8) == 2 * 8 * 16 * 128 + 2 * 8 * 16 * 2 == 33280
    assert oracle.kv_block_bytes(8, 128, oracle.KV_INT4) == 2 * 8 * 16 * 64 + 2 * 8 * 16 * 16 == 20480
    # (layer 2, block 5, V data, head 3, slot 7) in a 100-block FP16 pool
    blk = 65536
    assert oracle.kv_offset(8, 128, 0, 16, 100, 2, 5, 1, 3, 7) == (2 * 100 + 5) * blk + 32768 + (3 * 16 + 7) * 256
    # INT8 K meta of (layer 0, block 1, head 2, slot 3)
    assert oracle.kv_offset(8, 128, 1, 16, 10, 0, 1, 2, 2, 3) == 33280 + 2 * 16384 + (2 * 16 + 3) * 2
    # INT4 V meta of (layer 1, block 0, head 7, slot 15)
    assert oracle.kv_offset(8, 128, 2, 16, 4, 1, 0, 3, 7, 15) == 4 * 20480 + 2 * 8192 + 2048 + (7 * 16 + 15) * 16


@pytest.mark.parametrize("dt", [0, 1, 2])
def test_pool_no_two_live_tokens_share_bytes(dt):
    """Brute force over every (session, layer, token, head, part) of a small scattered pool."""
    H, d, P, L = 2, 64, 24, 2
    order = synth.pool_order(3, P)
    pool = oracle.PoolModel(P, 16, order)
    lens = [37, 16, 1, 90, 15]
    for s, n in enumerate(lens):
        pool.open(s)
        assert pool.append(s, n)
    db = {0: 2 * d, 1: d, 2: d // 2}[dt]
    mb = {0: 0, 1: 2, 2: (d // 32) * 4}[dt]
    owner = np.full(L * P * oracle.kv_block_bytes(H, d, dt), -1, dtype=np.int64)
    tag = 0
    for s, n in enumerate(lens):
        for t in range(n):
            blk, slot = pool.locate(s, t)
            for l in range(L):
                for h in range(H):
                    for part in range(4):
                        size = db if part < 2 else mb
                        if size == 0:
                            continue
                        off = oracle.kv_offset(H, d, dt, 16, P, l, blk, part, h, slot)
                        assert np.all(owner[off:off + size] == -1)
                        owner[off:off + size] = tag
                        tag += 1
    # the blocks in use are exactly those handed out, each once
    used = [b for s in range(len(lens)) for b in pool.tables[s]]
    assert len(used) == len(set(used)) == sum(-(-n // 16) for n in lens)


def test_pool_model_orders():
    pool = oracle.PoolModel(6, 16, [4, 2, 0, 1, 3, 5])
    pool.open(0)
    pool.open(1)
    assert pool.append(0, 17)  # tokens 0 and 16 take blocks 4 and 2
    assert pool.append(1, 1)   # block 0
    assert pool.tables == {0: [4, 2], 1: [0]}
    assert pool.locate(0, 16) == (2, 0) and pool.locate(0, 15) == (4, 15)
    assert not pool.append(1, 16 * 4)  # needs 4 more blocks, 3 free: refused whole
    assert pool.tables[1] == [0] and pool.lens[1] == 1
    pool.close(0)
    assert pool.free == [1, 3, 5, 4, 2]


# ----------------------------------------------------------------------------- arena planner

def _max_live(sizes, first, last, closed=True):
    steps = range(min(first), max(last) + 1)
    best = 0
    for s in steps:
        live = sum(z for z, f, l in zip(sizes, first, last) if (f <= s <= l if closed else f <= s < l))
        best = max(best, live)
    return best


def test_arena_worked_example():
    g = golden("arena_worked_example.json")
    MB = g["mb"]
    names = [t["name"] for t in g["tensors"]]
    sizes = [t["mb"] * MB for t in g["tensors"]]
    first = [t["first"] for t in g["tensors"]]
    last = [t["last"] for t in g["tensors"]]
    assert sum(sizes) == g["printed_unshared_mb"] * MB
    off, arena = oracle.arena_plan(sizes, first, last, 64, closed=True)
    assert arena == g["expected_closed_mb"] * MB == _max_live(sizes, first, last, True)
    assert {n: int(o) // MB for n, o in zip(names, off)} == g["expected_closed_offsets_mb"]
    off_h, arena_h = oracle.arena_plan(sizes, first, last, 64, closed=False)
    assert arena_h == g["expected_half_open_mb"] * MB == _max_live(sizes, first, last, False)
    assert arena_h > g["printed_planned_mb"] * MB  # the printed 12 MB is below every lower bound
    tc = g["three_conv"]
    s3 = [m * MB for m in tc["tensors_mb"]]
    assert sum(s3) == tc["printed_unshared_mb"] * MB
    _, a3 = oracle.arena_plan(s3, [0, 1, 2], [1, 2, 3], 64, closed=True)
    assert a3 == tc["expected_closed_mb"] * MB


def test_arena_random_invariants():
    rng = np.random.default_rng(12)
    for trial in range(300):
        n = int(rng.integers(1, 40))
        sizes = rng.integers(1, 1 << 20, n)
        if trial % 3 == 0:
            sizes = rng.integers(1, 200, n)  # sub-alignment sizes exercise the padding
        first = rng.integers(0, 30, n)
        last = first + rng.integers(0, 10, n)
        off, arena = oracle.arena_plan(sizes, first, last, 64, closed=True)
        assert np.all(off % 64 == 0) and arena % 64 == 0
        assert arena >= _max_live(sizes.tolist(), first.tolist(), last.tolist())
        assert arena <= sum(int(-(-z // 64) * 64) for z in sizes)
        assert np.all(off + sizes <= arena)
        for i in range(n):
            for j in range(i + 1, n):
                if first[i] <= last[j] and first[j] <= last[i]:
                    assert off[i] + sizes[i] <= off[j] or off[j] + sizes[j] <= off[i], (trial, i, j)


# ----------------------------------------------------------------------------- layer pieces

def test_rmsnorm_matches_torch_rms_norm():
    r = synth.normal(4, "rms", (6, 256), dtype=np.float64) * 3.0
    g = synth.norm_gain_f16(4, "rms", 256, random_gain=True)
    for i in range(6):
        ours = oracle.rmsnorm(r[i], g, 1e-5).astype(np.float64)
        ref = torch.nn.functional.rms_norm(torch.from_numpy(r[i]), (256,), torch.from_numpy(g.astype(np.float64)),
                                           eps=1e-5).numpy()
        # one rounding to fp16 of the same real number: equal up to one fp16 ulp (ties of nearly equal doubles)
        assert np.all(np.abs(ours - ref) <= np.abs(ref) * 2.0 ** -11 + 2.0 ** -24)
    ones = np.ones(256, np.float16)
    y = oracle.rmsnorm(r[0], ones).astype(np.float64)
    assert abs(math.sqrt(np.mean(y * y)) - 1.0) < 2e-3


def test_rope_pins():
    d, base = 64, 10000.0
    c, s = oracle.rope_table(300, d, base)
    x = synth.normal(8, "rope", d, dtype=np.float16)
    # p = 0 is the identity
    assert np.array_equal(oracle.rope_apply(x, c[0], s[0]).view(np.uint16), x.view(np.uint16))
    # complex form: (x_i + i x_{i+d/2}) e^{i theta_i}, theta_i = p base^(-2i/d)  (numpy complex arithmetic)
    for p in (1, 17, 299):
        z = (x[:d // 2].astype(np.float64) + 1j * x[d // 2:].astype(np.float64)) * np.exp(
            1j * p * base ** (-2.0 * np.arange(d // 2) / d))
        ours = oracle.rope_apply(x, c[p], s[p]).astype(np.float64)
        ref = np.concatenate([z.real, z.imag])
        assert np.max(np.abs(ours - ref)) < 4e-3
        # per-pair norms kept
        n0 = x[:d // 2].astype(np.float64) ** 2 + x[d // 2:].astype(np.float64) ** 2
        n1 = ours[:d // 2] ** 2 + ours[d // 2:] ** 2
        assert np.max(np.abs(n1 - n0)) < 2e-2
    # relative position: q(p).k(p') depends only on p - p'
    q = synth.normal(8, "rq", d, dtype=np.float16)
    k = synth.normal(8, "rk", d, dtype=np.float16)
    dots = [float(oracle.rope_apply(q, c[p + 5], s[p + 5]).astype(np.float64) @
                  oracle.rope_apply(k, c[p], s[p]).astype(np.float64)) for p in (0, 40, 200)]
    assert max(dots) - min(dots) < 0.05


def _kv_with(cfg, kvec, vvec):
    kv = oracle.KV(cfg, kvec.shape[1] + 1)
    kv.append(kvec, vvec)
    return kv


@pytest.mark.parametrize("dt", [0, 1, 2])
def test_attention_matches_torch_sdpa(dt):
    cfg = oracle.ModelCfg(1, 256, 4, 2, 64, 688, 0, kv_dtype=dt)
    n = 45
    k = synth.normal(2, "ak", (1, n, 2, 64), dtype=np.float16)
    v = synth.normal(2, "av", (1, n, 2, 64), dtype=np.float16)
    kv = _kv_with(cfg, k, v)
    q = synth.normal(2, "aq", (4, 64), dtype=np.float16)
    for h in range(4):
        g = h // 2
        ours = kv.attention(0, g, q[h], n).astype(np.float64)
        K = torch.tensor(np.stack([kv.read(0, 0, t, g) for t in range(n)]), dtype=torch.float64)
        V = torch.tensor(np.stack([kv.read(0, 1, t, g) for t in range(n)]), dtype=torch.float64)
        Q = torch.tensor(q[h].astype(np.float64))[None, None, None, :]
        ref = torch.nn.functional.scaled_dot_product_attention(Q, K[None, None], V[None, None])[0, 0, 0].numpy()
        assert np.all(np.abs(ours - ref) <= np.abs(ref) * 2.0 ** -10 + 2.0 ** -24)
        if dt == 0:  # FP16 store: the dequantised key is the fp16 input itself
            assert np.array_equal(K.numpy().astype(np.float16), k[0, :, g])


def test_attention_special_cases():
    cfg = oracle.ModelCfg(1, 256, 4, 2, 64, 688, 0)
    k = synth.normal(3, "k1", (1, 9, 2, 64), dtype=np.float16)
    v = synth.normal(3, "v1", (1, 9, 2, 64), dtype=np.float16)
    kv = _kv_with(cfg, k, v)
    q = synth.normal(3, "q1", 64, dtype=np.float16)
    # one key: the output is that key's value
    assert np.array_equal(kv.attention(0, 1, q, 1).view(np.uint16), v[0, 0, 1].view(np.uint16))
    # zero query: every score is equal, the output is the mean of the values
    mean = v[0, :, 0].astype(np.float64).mean(0)
    assert np.array_equal(kv.attention(0, 0, np.zeros(64, np.float16), 9).view(np.uint16),
                          mean.astype(np.float16).view(np.uint16))


# ----------------------------------------------------------------------------- composition

def _torch_layer(shape, w, l, r, kprior, vprior, rope_c, rope_s):
    """Layer l of the decode step for one token, from the float64 residual r [D], composed from torch library
    routines (float64, fp16 cast points); kprior / vprior [p, Hkv, d] are that layer's cached keys and values.
    Returns the float64 residual after the layer (unrounded)."""
    D, Hq, Hkv, d, F = shape.hidden, shape.n_heads, shape.n_kv_heads, shape.head_dim, shape.ffn
    f16 = lambda t: t.to(torch.float16).to(torch.float64)
    deq = lambda p, sm, k: torch.from_numpy(oracle.w4g32_dequant(p, sm, k).astype(np.float64))
    Wqkv, Wo, Wgu, Wd = (deq(w.wqkv[l], w.sqkv[l], D), deq(w.wo[l], w.so[l], Hq * d), deq(w.wgu[l], w.sgu[l], D),
                         deq(w.wdown[l], w.sdown[l], F))
    g1 = torch.from_numpy(w.gamma1[l].astype(np.float64))
    g2 = torch.from_numpy(w.gamma2[l].astype(np.float64))
    p = kprior.shape[0]
    xn = f16(torch.nn.functional.rms_norm(r, (D,), g1, eps=shape.rms_eps))
    qkv = f16(Wqkv @ xn)
    q, k, v = qkv[:Hq * d].view(Hq, d), qkv[Hq * d:(Hq + Hkv) * d].view(Hkv, d), qkv[(Hq + Hkv) * d:].view(Hkv, d)
    cos = torch.from_numpy(rope_c[p].astype(np.float64))
    sin = torch.from_numpy(rope_s[p].astype(np.float64))
    rot = lambda t: f16(torch.view_as_real(torch.complex(t[:, :d // 2], t[:, d // 2:]) *
                                           torch.complex(cos, sin)).permute(0, 2, 1).reshape(t.shape[0], d))
    q, k = rot(q), rot(k)
    K = torch.cat([torch.from_numpy(kprior.astype(np.float64)), k[None]], 0)  # [p+1, Hkv, d]
    V = torch.cat([torch.from_numpy(vprior.astype(np.float64)), v[None]], 0)
    Kh = K.permute(1, 0, 2).repeat_interleave(Hq // Hkv, 0)  # contiguous grouping: head h uses KV head h // G
    Vh = V.permute(1, 0, 2).repeat_interleave(Hq // Hkv, 0)
    o = f16(torch.nn.functional.scaled_dot_product_attention(q[:, None, :], Kh, Vh)[:, 0, :]).reshape(-1)
    r = r + Wo @ o
    xn2 = f16(torch.nn.functional.rms_norm(r, (D,), g2, eps=shape.rms_eps))
    gu = Wgu @ xn2
    a = f16(torch.nn.functional.silu(gu[:F]) * gu[F:])
    return r + Wd @ a


def _torch_logits(shape, w, r):
    """Final RMSNorm (gain gamma_f, fp16) and the fp16 LM head, float64 accumulation rounded once."""
    gf = torch.from_numpy(w.gamma_f.astype(np.float64))
    xf = torch.nn.functional.rms_norm(r, (shape.hidden,), gf, eps=shape.rms_eps).to(torch.float16)
    return (torch.from_numpy(w.lm_head.astype(np.float64)) @ xf.to(torch.float64)).to(torch.float16).numpy()


def _torch_layer_reference(shape, w, x, kprior, vprior, rope_c, rope_s):
    """The tiny one-layer step composed from torch library routines: its fp16 output hidden state."""
    r = torch.from_numpy(x.astype(np.float64))[0]
    return _torch_layer(shape, w, 0, r, kprior[0], vprior[0], rope_c, rope_s).to(torch.float16).numpy()


def test_tiny_layer_composition_matches_torch_library_model():
    shape = TINY
    seed = 21
    cfg = model_cfg(shape, oracle.KV_FP16)
    w = oracle_weights(shape, seed, random_gain=True)
    kp, vp = prior_kv(shape, seed, 0, 128)
    kv = oracle.KV(cfg, 200)
    kv.append(kp, vp)
    x = synth.hidden_f16(seed, 1, shape.hidden)
    c, s = oracle.rope_table(200, shape.head_dim, shape.rope_base)
    out = oracle.forward(cfg, w, [kv], [1], x, c, s)
    ref = _torch_layer_reference(shape, w, x, kp, vp, c, s)
    assert len(kv) == 129
    assert rel_l2(out[0], ref) < 1e-4
    assert np.max(np.abs(out[0].astype(np.float64) - ref.astype(np.float64))) < 4e-3


def test_prefill_equals_token_by_token_decode():
    """A chunk of T tokens gives the same last output and the same stored KV as T single-token steps."""
    shape = TINY
    seed = 22
    cfg = model_cfg(shape, oracle.KV_INT8)
    w = oracle_weights(shape, seed)
    kp, vp = prior_kv(shape, seed, 0, 20)
    x = synth.hidden_f16(seed, 7, shape.hidden)
    c, s = oracle.rope_table(64, shape.head_dim, shape.rope_base)
    a, b = oracle.KV(cfg, 64), oracle.KV(cfg, 64)
    a.append(kp, vp)
    b.append(kp, vp)
    out_chunk = oracle.forward(cfg, w, [a], [7], x, c, s)
    for t in range(7):
        out_step = oracle.forward(cfg, w, [b], [1], x[t:t + 1], c, s)
    assert np.array_equal(out_chunk.view(np.uint16), out_step.view(np.uint16))
    for t in range(27):
        for h in range(2):
            for which in (0, 1):
                da, ma = a.stored(0, which, t, h)
                db, mb = b.stored(0, which, t, h)
                assert np.array_equal(da, db) and np.array_equal(ma, mb)


def test_two_layer_chain_matches_torch_library_model():
    """The layer loop: two layers, each with its own weights, gains and KV, against two torch layers chained
    through the float64 residual ([Core] 5.1: pre-norm decoder layers in sequence)."""
    shape = shrink(TINY, n_layers=2)
    seed = 23
    cfg = model_cfg(shape, oracle.KV_FP16)
    w = oracle_weights(shape, seed, random_gain=True)
    kp, vp = prior_kv(shape, seed, 0, 40)
    kv = oracle.KV(cfg, 64)
    kv.append(kp, vp)
    x = synth.hidden_f16(seed, 1, shape.hidden)
    c, s = oracle.rope_table(64, shape.head_dim, shape.rope_base)
    out = oracle.forward(cfg, w, [kv], [1], x, c, s)
    r = torch.from_numpy(x.astype(np.float64))[0]
    for l in range(2):
        r = _torch_layer(shape, w, l, r, kp[l], vp[l], c, s)
    ref = r.to(torch.float16).numpy()
    assert len(kv) == 41
    assert rel_l2(out[0], ref) < 1e-4
    assert np.max(np.abs(out[0].astype(np.float64) - ref.astype(np.float64))) < 4e-3
    # a layer that read another layer's weights or cache would be far off: the second layer matters
    r1 = _torch_layer(shape, w, 0, torch.from_numpy(x.astype(np.float64))[0], kp[0], vp[0], c, s)
    assert rel_l2(out[0], r1.to(torch.float16).numpy()) > 1e-2


def test_lm_head_branch_matches_torch_library_model():
    """The output branch: logits = fp16(W_lm fp16(rmsnorm(r) gamma_f)) after two layers, against torch's
    rms_norm and a float64 matmul; orc_output alone against the same on one residual."""
    shape = shrink(TINY, n_layers=2, vocab=1024)
    seed = 24
    cfg = model_cfg(shape, oracle.KV_FP16)
    w = oracle_weights(shape, seed, random_gain=True)
    assert w.lm_head.shape == (1024, shape.hidden)
    kp, vp = prior_kv(shape, seed, 0, 33)
    kv = oracle.KV(cfg, 64)
    kv.append(kp, vp)
    x = synth.hidden_f16(seed, 1, shape.hidden)
    c, s = oracle.rope_table(64, shape.head_dim, shape.rope_base)
    out = oracle.forward(cfg, w, [kv], [1], x, c, s)[0]
    r = torch.from_numpy(x.astype(np.float64))[0]
    for l in range(2):
        r = _torch_layer(shape, w, l, r, kp[l], vp[l], c, s)
    ref = _torch_logits(shape, w, r)
    assert out.shape == (1024,)
    # two chained layers differ from torch's in a few fp16 roundings (rms_norm and SDPA sum in another
    # order); those flips reach every logit, so this end-to-end bar is the tolerance's 1e-3
    assert rel_l2(out, ref) < 1e-3
    # the same final residual through orc_output: the logits agree to within one fp16 step (summation order)
    got = oracle.output(cfg, w, r.numpy()[None])[0]
    u = fp16_ulps(got, ref)
    assert u.max() <= 1 and np.mean(u == 0) > 0.99
    # the gain is applied, and row v of the LM head gives logit v
    w_plain = oracle.Weights(**{**w.__dict__, "gamma_f": np.ones(shape.hidden, np.float16)})
    assert rel_l2(oracle.output(cfg, w_plain, r.numpy()[None])[0], ref) > 1e-2
    w_rev = oracle.Weights(**{**w.__dict__, "lm_head": np.ascontiguousarray(w.lm_head[::-1])})
    assert np.array_equal(oracle.output(cfg, w_rev, r.numpy()[None])[0].view(np.uint16),
                          got[::-1].view(np.uint16))


@pytest.mark.parametrize("dt", [oracle.KV_FP16, oracle.KV_INT4])
def test_several_sequences_equal_separate_calls(dt):
    """n_seq > 1: each sequence's output row and stored KV are those of the same sequence run alone, for
    decode (one token each) and for a batched chunk (several tokens each)."""
    shape = shrink(TINY, n_layers=2, vocab=64)
    seed = 25
    cfg = model_cfg(shape, dt)
    w = oracle_weights(shape, seed)
    priors = (5, 17, 33)
    c, s = oracle.rope_table(64, shape.head_dim, shape.rope_base)
    for n_tok in ((1, 1, 1), (3, 1, 2)):
        x = synth.hidden_f16(seed, sum(n_tok), shape.hidden, tag=f"x{n_tok}")
        together, alone = [], []
        for i, p in enumerate(priors):
            kp, vp = prior_kv(shape, seed, i, p)
            for lst in (together, alone):
                kv = oracle.KV(cfg, 64)
                kv.append(kp, vp)
                lst.append(kv)
        out = oracle.forward(cfg, w, together, list(n_tok), x, c, s)
        assert out.shape == (3, 64)
        t0 = 0
        for i, n in enumerate(n_tok):
            ref = oracle.forward(cfg, w, [alone[i]], [n], x[t0:t0 + n], c, s)
            assert np.array_equal(out[i].view(np.uint16), ref[0].view(np.uint16)), (n_tok, i)
            assert len(together[i]) == len(alone[i]) == priors[i] + n
            for t in range(priors[i] + n):
                for l in range(2):
                    for which in (0, 1):
                        da, ma = together[i].stored(l, which, t, 1)
                        db, mb = alone[i].stored(l, which, t, 1)
                        assert np.array_equal(da, db) and np.array_equal(ma, mb)
            t0 += n


def test_forward_is_layers_then_output():
    """orc_forward = orc_layer for each layer in turn on the carried residual, then orc_output of the last
    token; orc_layer stores the tokens' KV at its own layer and leaves the lengths alone."""
    shape = shrink(TINY, n_layers=2, vocab=256)
    seed = 26
    cfg = model_cfg(shape, oracle.KV_INT8)
    w = oracle_weights(shape, seed, random_gain=True)
    kp, vp = prior_kv(shape, seed, 0, 19)
    a, b = oracle.KV(cfg, 64), oracle.KV(cfg, 64)
    a.append(kp, vp)
    b.append(kp, vp)
    x = synth.hidden_f16(seed, 2, shape.hidden)
    c, s = oracle.rope_table(64, shape.head_dim, shape.rope_base)
    out = oracle.forward(cfg, w, [a], [2], x, c, s)
    r = x.astype(np.float64)
    r = oracle.layer(cfg, w, 0, [b], [2], r, c, s)
    assert len(b) == 19
    d0, _ = b.stored(0, 0, 19, 0)
    d1, _ = b.stored(1, 0, 19, 0)
    r = oracle.layer(cfg, w, 1, [b], [2], r, c, s)
    got = oracle.output(cfg, w, r[-1:])
    assert np.array_equal(got.view(np.uint16), out.view(np.uint16))
    # the tokens are stored (read past the length, which was left behind)
    for t in range(21):
        for l in range(2):
            for which in (0, 1):
                da, ma = a.stored(l, which, t, 1)
                db, mb = b.stored(l, which, t, 1)
                assert np.array_equal(da, db) and np.array_equal(ma, mb)
    assert not np.array_equal(d0, d1)  # each layer stored its own keys
    # committed, the layer-by-layer store continues like the forward's
    b.commit(2)
    assert len(b) == len(a) == 21
    x1 = synth.hidden_f16(seed, 1, shape.hidden, tag="next")
    o_a = oracle.forward(cfg, w, [a], [1], x1, c, s)
    o_b = oracle.forward(cfg, w, [b], [1], x1, c, s)
    assert np.array_equal(o_a.view(np.uint16), o_b.view(np.uint16))
