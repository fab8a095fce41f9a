"""Host logic of the step-timeline reader (quantized_decode_step_gb300/timeline.py) on synthetic records:
launches of the same GEMV shape in two layers, their blocks entering in any order and overlapping the
launch before them, attention launches tagged by layer; no GPU."""
import numpy as np

from quantized_decode_step_gb300 import timeline as tl

GEMV_QKV = (1 << 60) | (384 << 32) | (64 << 8) | 1
GEMV_O = (1 << 60) | (256 << 32) | (64 << 8) | 1


def attn(layer):
    return (2 << 60) | layer


def recs_of(spec):
    """spec: (tag, blocks, t0, per-event offsets): records of every block, block b shifted by b ns."""
    out = []
    for tag, blocks, t0, offs in spec:
        for b in blocks:
            for ev, dt in enumerate(offs):
                out.append((tag, b, ev, t0 + dt + b))
    rng = np.random.default_rng(0)
    a = np.array(out, dtype=np.int64)
    return a[rng.permutation(len(a))]


def test_kind_of():
    assert tl.kind_of(GEMV_QKV) == (tl.GEMV, 384, 64, 1)
    assert tl.kind_of(attn(7)) == (tl.ATTN, 7, 0, 0)


def test_launches_and_phases():
    blocks = list(range(4))
    spec = [(GEMV_QKV, blocks, 1000, (0, 100, 400)),
            (attn(0), [0, 1], 1450, (0, 300, 900, 1500)),  # enters before the QKV launch's last stamps
            (GEMV_O, blocks, 3000, (0, 50, 300)),
            (GEMV_QKV, blocks, 5000, (0, 100, 400)),      # the next layer: same tag, same blocks
            (attn(1), [0, 1], 5450, (0, 300, 900, 1500))]
    Ls = tl.launches(recs_of(spec))
    assert [L["kind"][0] for L in Ls] == [tl.GEMV, tl.ATTN, tl.GEMV, tl.GEMV, tl.ATTN]
    assert [L["tag"] for L in Ls] == [s[0] for s in spec]
    for L, (tag, blks, t0, offs) in zip(Ls, spec):
        assert L["blocks"] == set(blks)
        for ev, dt in enumerate(offs):
            assert L["ev"][ev] == sorted(t0 + dt + b for b in blks)
    rows = tl.phases(Ls)
    assert rows[0]["entry_first"] == 0.0 and rows[0]["entry_last"] == 0.003
    assert abs(rows[0]["ready_med"] - 0.402) < 1e-9  # the median block's staging (event 2)
    assert abs(rows[1]["ready_med"] - (1450 + 300 + 1 - 1000) / 1000) < 1e-9  # attention: after its wait
    assert abs(rows[1]["end_last"] - (1450 + 1500 + 1 - 1000) / 1000) < 1e-9
    assert abs(rows[3]["entry_first"] - 4.0) < 1e-9
