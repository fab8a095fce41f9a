"""GPU checks of the elastic KV pool (MAG_FLAG_ELASTIC_POOL; "Magnitude" 2.2 layer 1 and 3.2, hot and
cold pools): groups of blocks mapped on demand and given back, lowest block first, the hot size set by
the load profile.

Every block a session holds (mag_debug_kv_locate) and the mapped / free / hot counts are compared
exactly with the oracle's ElasticPoolModel driven by the same calls; decode steps on the sessions are
compared with the model oracle before and after groups are released and mapped again (mapped memory is
zeroed, so a reused group reads as a fresh one).

* Tiny layer, FP16: three sessions across two groups; closing one gives its group back; a new session
  maps it again.
* Two 8B-shaped layers (FP16: 32-block groups; INT4: 512-block groups): sessions spread over several
  groups in every layer's range, release and regrow, decode against the oracle.
* The hot size follows the profile's P90 (window 4, every step recorded): a long session raises it,
  short ones bring it back to one group.
* A pool that can not hold an append says KV_FULL and changes nothing.
"""
import numpy as np
import pytest
import torch

import oracle
import quantized_decode_step_gb300 as mag
import synth
from oracle import adapt
from synth import driver
from synth.workloads import KV_FP16, KV_INT4, LLAMA8B, TINY, Workload, shrink
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


class _Elastic:
    """A context with an elastic pool, the pool model and the oracle's stores, driven together."""

    def __init__(self, shape, dt, pool_blocks, max_sessions, max_context, seed):
        self.shape, self.dt, self.seed = shape, dt, seed
        wl = Workload("elastic", shape, dt, max_sessions, (0,))
        cfg = mag.make_config(shape, kv_dtype=dt, pool_blocks=pool_blocks, max_sessions=max_sessions,
                              max_batch=max_sessions, max_context=max_context, flags=mag.FLAG_ELASTIC_POOL)
        self.ctx = mag.Context(cfg, torch.cuda.current_stream().cuda_stream)
        driver.load_weights(self.ctx, shape, seed, random_gain=True)
        self.w = oracle_weights(shape, seed, True)
        self.ocfg = model_cfg(shape, dt)
        st = self.ctx.memory_stats()
        self.G = st["pool_group_blocks"]
        self.model = adapt.ElasticPoolModel(pool_blocks, self.G)
        assert st["pool_blocks_total"] == self.model.P
        self.c, self.s = oracle.rope_table(max_context + 2, shape.head_dim, shape.rope_base)
        self.sess = {}  # sid -> dict(kv, blocks, index)
        self.n_step = 0
        del wl

    def open(self, index, n_tok):
        sid = self.ctx.session_open()
        kv = oracle.KV(self.ocfg, n_tok + 64)
        blocks = []
        for t0 in range(0, n_tok, 4096):  # the driver appends in chunks of 4096 tokens
            n = min(4096, n_tok - t0)
            blocks += self.model.alloc(-(-(t0 + n) // 16) - len(blocks))
        driver.append_prior(self.ctx, sid, self.shape, self.seed, index, n_tok)
        if n_tok:
            kv.append(*prior_kv(self.shape, self.seed, index, n_tok))
        self.sess[sid] = dict(kv=kv, blocks=blocks)
        return sid

    def close(self, sid):
        self.ctx.session_close(sid)
        self.model.release(self.sess.pop(sid)["blocks"])

    def decode(self, sids):
        for sid in sids:
            n = self.ctx.session_length(sid)
            if n % 16 == 0:
                self.sess[sid]["blocks"] += self.model.alloc(1)
        x = synth.hidden_f16(self.seed, len(sids), self.shape.hidden, tag=f"e{self.n_step}")
        self.n_step += 1
        width = self.shape.vocab or self.shape.hidden
        out = torch.empty((len(sids), width), dtype=torch.float16, device="cuda")
        self.ctx.decode_step(sids, torch.from_numpy(x).cuda(), out)
        self.ctx.sync()
        ref = oracle.forward(self.ocfg, self.w, [self.sess[s]["kv"] for s in sids], [1] * len(sids), x, self.c, self.s)
        _compare(out.cpu().numpy(), ref, f"elastic decode {self.n_step}")

    def settle(self):
        """Let releases whose stream work is done finish (closing an empty session runs the trim)."""
        self.ctx.sync()
        self.ctx.session_close(self.ctx.session_open())

    def check(self):
        st = self.ctx.memory_stats()
        m = self.model
        assert st["pool_blocks_mapped"] == len(m.mapped) * self.G, (st, sorted(m.mapped))
        assert st["pool_blocks_free"] == m.available()
        assert st["pool_blocks_hot"] == m.hot * self.G
        assert st["kv_pool_mapped_bytes"] == len(m.mapped) * self.G * self.shape.n_layers * st["kv_block_bytes"]
        for sid, e in self.sess.items():
            n = self.ctx.session_length(sid)
            for t in range(0, n, 16):
                assert self.ctx.debug_kv_locate(sid, 0, t)[4] == e["blocks"][t // 16], (sid, t)


def test_tiny_groups_map_release_and_map_again():
    e = _Elastic(TINY, KV_FP16, 600, 4, 5200, 81)
    G = e.G
    assert G * TINY.n_layers * e.ctx.memory_stats()["kv_block_bytes"] % (1 << 21) == 0  # whole 2 MiB pages
    a = e.open(0, 3000)
    c = e.open(1, 5)
    b = e.open(2, 2000)
    e.check()
    assert len(e.model.mapped) >= 2
    e.decode([a, c, b])
    e.check()
    e.close(b)  # its group has no other user: given back once the stream has passed it
    e.settle()
    e.check()
    d = e.open(3, 2000)  # maps it again
    e.check()
    e.decode([a, c, d])
    e.decode([d])
    e.check()


@pytest.mark.slow
@pytest.mark.parametrize("dt,lens", [(KV_FP16, (1500, 700, 600)), (KV_INT4, (9000, 300, 200))])
def test_8b_two_layers_across_groups(dt, lens):
    shape = shrink(LLAMA8B, n_layers=2)
    e = _Elastic(shape, dt, -(-sum(lens) // 16) + 64, 3, max(lens) + 64, 83 + dt)
    a = e.open(0, lens[0])
    b = e.open(1, lens[1])
    e.check()
    assert len(e.model.mapped) >= 2
    e.decode([a, b])
    e.close(a)
    e.settle()
    e.check()
    c = e.open(2, lens[2])
    e.check()
    e.decode([b, c])
    e.check()


def test_tiny_hot_pool_follows_profile():
    e = _Elastic(TINY, KV_FP16, 1200, 2, 5100, 85)
    e.ctx.set_adaptive(True, adaptive_window_size=4, adaptive_sample_rate=1)
    win = adapt.LoadWindow(4, 1)
    long_ = e.open(0, 5000)
    for sids in ([long_],) * 4:
        e.decode(sids)
        win.observe(e.ctx.session_length(long_))
        if win.full():
            e.model.set_hot(adapt.hot_pool_blocks(win.quantile(0.9), len(e.sess), "1.2"))
    assert e.ctx.profile()["hot_blocks"] == adapt.hot_pool_blocks(win.quantile(0.9), 1, "1.2")
    e.check()
    assert e.model.hot >= 2  # 5000 tokens x 1.2 need two groups of 256 blocks
    e.close(long_)
    e.settle()
    e.check()  # the hot groups stay mapped with no session
    short = e.open(1, 10)
    for _ in range(4):
        e.decode([short])
        win.observe(e.ctx.session_length(short))
        e.model.set_hot(adapt.hot_pool_blocks(win.quantile(0.9), len(e.sess), "1.2"))
    e.settle()
    e.check()
    assert e.model.hot == 1 and len(e.model.mapped) == 1


def test_tiny_elastic_kv_full_changes_nothing():
    e = _Elastic(TINY, KV_FP16, 10, 2, 5000, 87)  # one group
    a = e.open(0, e.G * 16)  # the whole pool
    e.check()
    before = e.ctx.memory_stats()
    sid = e.ctx.session_open()
    k = torch.zeros((TINY.n_layers, 1, TINY.n_kv_heads, TINY.head_dim), dtype=torch.float16, device="cuda")
    with pytest.raises(mag.MagError) as err:
        e.ctx.kv_append(sid, 1, k, k)
    assert err.value.status == mag.ERR_KV_FULL
    assert e.ctx.session_length(sid) == 0 and e.ctx.memory_stats() == {**before, "sessions_open": 2}
    e.ctx.session_close(sid)
    assert e.ctx.session_length(a) == e.G * 16
