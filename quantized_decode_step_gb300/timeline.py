"""Reading a step timeline (``Context.timeline``): group the records into launches and give each launch's
phase times. A record is four uint64: tag, block (x | y << 20 | z << 40), event, global-timer ns.

GEMV tags are (1 << 60) | n_mtiles << 32 | n_chunks << 8 | batch, attention tags (2 << 60) | layer. The
launches of one step follow one another on one stream, so a launch is the run of records with one tag
between the first entry of a block already seen and the next such entry.
"""
from __future__ import annotations

import numpy as np

GEMV, ATTN = 1, 2


def kind_of(tag: int) -> tuple[int, int, int, int]:
    """(class, n_mtiles or layer, n_chunks, batch) of a record tag."""
    cls = tag >> 60
    if cls == GEMV:
        return GEMV, (tag >> 32) & 0xFFFFFFF, (tag >> 8) & 0xFFFFFF, tag & 0xFF
    return cls, tag & 0xFFFFFFFF, 0, 0


def launches(recs: np.ndarray) -> list[dict]:
    """The step's launches in order: dicts with 'tag', 'kind', 'blocks' (blocks seen) and 'ev' (event ->
    sorted list of ns)."""
    recs = recs[np.argsort(recs[:, 3], kind="stable")]
    out, cur = [], {}
    for tag, blk, ev, t in recs.tolist():
        L = cur.get(tag)
        if ev == 0 and (L is None or blk in L["blocks"]):
            L = {"tag": tag, "kind": kind_of(tag), "blocks": set(), "ev": {}}
            cur[tag] = L
            out.append(L)
        if L is None:
            continue
        if ev == 0:
            L["blocks"].add(blk)
        L["ev"].setdefault(ev, []).append(t)
    for L in out:
        for v in L["ev"].values():
            v.sort()
    out.sort(key=lambda L: L["ev"][0][0])
    return out


def phases(Ls: list[dict]) -> list[dict]:
    """Per launch, in us from the step's first stamp: first and last block entry, the median block's wait
    release (GEMV: the median block's staging done; attention: after its wait) and, where the next launch
    exists, the gap from this launch's last stamp to the next launch's first entry."""
    t0 = Ls[0]["ev"][0][0]

    def us(x):
        return (x - t0) / 1000.0

    rows = []
    for i, L in enumerate(Ls):
        e = L["ev"]
        cls = L["kind"][0]
        ready = e.get(2 if cls == GEMV else 1, e[0])
        row = {"kind": L["kind"], "blocks": len(L["blocks"]), "entry_first": us(e[0][0]), "entry_last": us(e[0][-1]),
               "ready_med": us(ready[len(ready) // 2]), "ready_last": us(ready[-1])}
        if cls == ATTN and 3 in e:
            row["keys_med"] = us(e[2][len(e[2]) // 2])
            row["end_last"] = us(e[3][-1])
        rows.append(row)
    return rows
