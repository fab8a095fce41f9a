"""The adaptive runtime's host policies, no GPU: the oracle (oracle/adapt.py) pinned to what the page
("Magnitude" 3.1-3.3, 4.3, 6.2) and the mathematics fix, then the library's own profile and policy
functions (C ABI) against the oracle, exactly (all integers).

Pins of the oracle:
* nearest-rank quantiles = numpy's inverted-CDF percentile (a library routine) on random windows, and
  hand values;
* the window holds exactly the last `window` recorded values (a deque of the recorded stream);
  one inference in `sample_every` is recorded, so n inferences record ceil(n / sample_every);
* the page's thresholds: P90 below 128 -> short plan, above 512 -> long plan;
* the page's hot pool rule at its slack values (1.2 default, 1.05, 1.1) on hand cases.
"""
import math
import random

import numpy as np
import pytest

import quantized_decode_step_gb300 as mag
from oracle import adapt


@pytest.fixture(scope="module")
def lib():
    mag.build()
    return mag.lib()


# ---------------------------------------------------------------- oracle pins
def test_oracle_quantile_is_inverted_cdf_percentile():
    rng = np.random.default_rng(0)
    for n in (1, 2, 3, 7, 16, 63, 64, 128):
        w = adapt.LoadWindow(window=n, sample_every=1)
        vals = rng.integers(1, 5000, size=n)
        for v in vals:
            w.observe(int(v))
        for q in (0.5, 0.9, 0.99, 1.0, 0.25):
            want = int(np.percentile(vals, 100 * q, method="inverted_cdf"))
            assert w.quantile(q) == want, (n, q)


def test_oracle_quantile_hand_values():
    w = adapt.LoadWindow(window=10, sample_every=1)
    assert w.quantile(0.9) == -1
    for v in (10, 20, 30, 40, 50, 60, 70, 80, 90, 100):
        w.observe(v)
    # nearest rank: P50 is the 5th smallest, P90 the 9th, P99 the 10th
    assert (w.quantile(0.5), w.quantile(0.9), w.quantile(0.99)) == (50, 90, 100)


def test_oracle_window_and_sampling():
    rng = random.Random(1)
    for window, rate in ((64, 4), (8, 1), (5, 3), (128, 2), (32, 8)):
        w = adapt.LoadWindow(window, rate)
        recorded = []
        for i in range(1000):
            v = rng.randrange(1, 9000)
            took = w.observe(v)
            assert took == (i % rate == 0)
            if took:
                recorded.append(v)
            assert len(w.values) == min(window, math.ceil((i + 1) / rate))
            assert list(w.values) == recorded[-window:]
        assert w.full()


def test_oracle_pages_defaults_fill_after_253_inferences():
    # window 64 at rate 1/4: the 64th record is inference 253 (counts 0, 4, ..., 252)
    w = adapt.LoadWindow()
    for i in range(252):
        w.observe(100)
    assert not w.full()
    w.observe(100)
    assert w.full()


def test_oracle_plan_thresholds():
    assert [adapt.plan_for(p) for p in (1, 127, 128, 300, 512, 513, 100000)] == [0, 0, 1, 1, 1, 2, 2]


def test_oracle_hot_pool_hand_cases():
    # one session, P90 = 160 tokens = 10 blocks: 1.2 x 10 = 12; 1.05 x 10 = 10.5 -> 11; 1.1 -> 11
    assert adapt.hot_pool_blocks(160, 1, "1.2") == 12
    assert adapt.hot_pool_blocks(160, 1, "1.05") == 11
    assert adapt.hot_pool_blocks(160, 1, "1.1") == 11
    # P90 = 161 tokens is 11 blocks; three sessions 33 blocks; x 1.2 = 39.6 -> 40
    assert adapt.hot_pool_blocks(161, 3, "1.2") == 40
    assert adapt.hot_pool_blocks(0, 3) == 0 and adapt.hot_pool_blocks(50, 0) == 0


# ---------------------------------------------------------------- library vs oracle
def test_library_defaults_are_the_pages(lib):
    a = mag.adapt_defaults()
    assert (a.enable_adaptive, a.adaptive_window_size, a.adaptive_sample_rate) == (1, 64, 4)
    assert (a.plan_short_below, a.plan_long_above, a.force_plan, a.async_switch) == (128, 512, -1, 0)
    assert abs(a.hot_pool_slack - 1.2) < 1e-6
    assert list(a.plan_splits) == [4, 8, 16]  # GB300 presets of the three plans (not the page's)


@pytest.mark.parametrize("window,rate", [(64, 4), (8, 1), (5, 3), (128, 2), (32, 8), (1, 1)])
def test_library_profile_matches_oracle(lib, window, rate):
    rng = random.Random(window * 31 + rate)
    p = mag.Profiler(window, rate)
    o = adapt.LoadWindow(window, rate)
    for i in range(700):
        # a length mix with long tails, as an agent's contexts
        v = int(rng.lognormvariate(5.5, 1.0)) + 1
        assert p.observe(v) == o.observe(v)
        assert p.count() == len(o.values)
        if i % 7 == 0 or i > 650:
            for q in (0.5, 0.9, 0.99, 1.0):
                assert p.quantile(q) == o.quantile(q), (i, q)
    p.close()


def test_library_profiler_argument_errors(lib):
    with pytest.raises(mag.MagError):
        mag.Profiler(0, 4)
    with pytest.raises(mag.MagError):
        mag.Profiler(64, 0)
    p = mag.Profiler(4, 1)
    assert p.quantile(0.5) == -1
    for q in (0.0, -0.1, 1.5):
        with pytest.raises(mag.MagError):
            p.quantile(q)


def test_library_policies_match_oracle(lib):
    for p90 in list(range(0, 1200, 7)) + [127, 128, 129, 511, 512, 513]:
        for sb, la in ((128, 512), (64, 64), (100, 2000)):
            assert mag.plan_for(p90, sb, la) == adapt.plan_for(p90, sb, la)
        for n in (0, 1, 2, 5, 16):
            for slack in ("1.0", "1.05", "1.1", "1.15", "1.2", "2.5"):
                assert mag.hot_pool_blocks(p90, n, float(slack)) == adapt.hot_pool_blocks(p90, n, slack), \
                    (p90, n, slack)


# ---------------------------------------------------------------- elastic pool model
def test_elastic_model_hand_case():
    # 600 blocks in groups of 256 -> 768; sessions of 188, 1 and 125 blocks fill group 0 and start group 1
    m = adapt.ElasticPoolModel(600, 256)
    assert (m.P, m.available(), sorted(m.mapped)) == (768, 768, [0])
    a, c, b = m.alloc(188), m.alloc(1), m.alloc(125)
    assert (a[0], a[-1], c, b[0], b[-1]) == (0, 187, [188], 189, 313)
    assert sorted(m.mapped) == [0, 1]
    m.release(b)  # group 1 wholly free again: given back
    assert sorted(m.mapped) == [0] and m.available() == 768 - 189
    assert m.alloc(1000) is None and sorted(m.mapped) == [0]


def test_elastic_model_invariants_random():
    rng = random.Random(5)
    for G, n in ((4, 37), (16, 100), (256, 600)):
        m = adapt.ElasticPoolModel(n, G)
        held = []
        for _ in range(2000):
            op = rng.random()
            if op < 0.45:
                got = m.alloc(rng.randrange(1, 3 * G))
                if got is not None:
                    held.append(got)
            elif op < 0.85 and held:
                m.release(held.pop(rng.randrange(len(held))))
            else:
                m.set_hot(rng.randrange(0, m.P + 1))
            in_use = [b for h in held for b in h]
            assert len(in_use) == len(set(in_use))  # no block handed out twice
            assert not (set(in_use) & m.free)
            assert all(b // G in m.mapped for b in in_use)  # every block in use is mapped
            # mapped = the hot groups and the groups with a block in use, nothing else
            assert m.mapped == set(range(m.hot)) | {b // G for b in in_use}
            assert m.free == {b for g in m.mapped for b in range(g * G, (g + 1) * G)} - set(in_use)
            assert m.available() == m.P - len(in_use)
