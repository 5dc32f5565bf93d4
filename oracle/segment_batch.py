"""Segment-batch form of the replay, derived from the op log by formula.

Test infrastructure only.  Restates the single-prefill restoration of
"Cache Engineering for Agents", paper review page section 4.2 (Appendix
A.1.1, Figure 10): queries are cut wherever a drop or repos acts; each
segment attends causally over its own tokens plus the still-active KV of
earlier segments; a dropped entry stays visible to the segments before its
drop and is hidden from the later ones; with repos each segment reads keys at
the positions of the version current during it.

Nothing here walks the active cache: every table is a closed-form function of
the op log, so agreement with ``core.replay`` is a real cross-check.
"""
from __future__ import annotations

import bisect
import math

import numpy as np

from .core import NEVER, rope, validate, widen


def segment_tables(msg_start, drop_after, drop_target, repos_after):
    """Per-token integer tables of the segment-batch rule.

    seg[t]       number of op-carrying boundaries b < msg(t)
    drop_seg[u]  1 + index of the op boundary where msg(u) is first dropped
                 (NEVER if it never is): the first segment u is hidden from
    seg_ver[s]   number of repos boundaries among the first s op boundaries
    pos[v][u]    position of u while version v is current (-1 where u is not
                 alive during version v): version 0 numbers tokens from 0; the
                 repos that opens version v at boundary b numbers the tokens
                 alive at b 0..r-1 in logical order, and later tokens continue
                 from r in order of appending.
    """
    validate(msg_start, drop_after, drop_target, repos_after)
    ms = np.asarray(msg_start, dtype=np.int64)
    n_msgs = len(ms) - 1
    T = int(ms[-1])
    op_b = sorted(set(int(a) for a in drop_after) | set(int(a) for a in repos_after))
    rep_b = sorted(set(int(a) for a in repos_after))
    msg_of = np.searchsorted(ms, np.arange(T), side="right") - 1 if T else np.zeros(0, np.int64)
    seg_of_msg = np.array([bisect.bisect_left(op_b, m) for m in range(n_msgs)], dtype=np.int64)
    first_drop = {}
    for a, t in zip(drop_after, drop_target):
        a, t = int(a), int(t)
        first_drop[t] = min(a, first_drop.get(t, a))
    seg = seg_of_msg[msg_of] if T else np.zeros(0, np.int64)
    drop_seg_msg = np.full(n_msgs, NEVER, dtype=np.int64)
    for j, b in first_drop.items():
        drop_seg_msg[j] = bisect.bisect_right(op_b, b)
    drop_seg = drop_seg_msg[msg_of] if T else np.zeros(0, np.int64)
    n_seg = len(op_b) + 1
    seg_ver = np.array([sum(1 for b in op_b[:s] if b in set(rep_b)) for s in range(n_seg)],
                       dtype=np.int64)
    n_ver = len(rep_b) + 1
    pos = np.full((n_ver, T), -1, dtype=np.int64)
    # version 0: appended positions 0..; valid until the first repos
    end0 = ms[rep_b[0] + 1] if rep_b else T
    pos[0, :end0] = np.arange(end0)
    for v in range(1, n_ver):
        b = rep_b[v - 1]
        last = ms[rep_b[v] + 1] if v < len(rep_b) else T
        alive = np.array([(msg_of[u] <= b) and not (msg_of[u] in first_drop
                                                    and first_drop[msg_of[u]] <= b)
                          for u in range(int(ms[b + 1]))], dtype=bool)
        r = int(alive.sum())
        pos[v, :int(ms[b + 1])][alive] = np.arange(r)
        pos[v, int(ms[b + 1]):last] = r + np.arange(last - int(ms[b + 1]))
    return dict(seg=seg, drop_seg=drop_seg, seg_ver=seg_ver, pos=pos, n_seg=n_seg, n_ver=n_ver,
                op_boundaries=op_b, repos_boundaries=rep_b)


def segment_batch_attention(msg_start, drop_after, drop_target, repos_after, q, k, v,
                            dtype: str, base: float):
    """All rows at once with the visibility mask
    visible(t, u) <=> u <= t and seg(t) < drop_seg(u), query and keys at the
    positions of version seg_ver[seg(t)].  Dense; small T only."""
    tab = segment_tables(msg_start, drop_after, drop_target, repos_after)
    T, Hq, D = q.shape
    Hkv = k.shape[1]
    grp = Hq // Hkv
    Q, K, V = widen(q, dtype), widen(k, dtype), widen(v, dtype)
    seg, dseg = tab["seg"], tab["drop_seg"]
    tver = tab["seg_ver"][seg]
    mask = (np.arange(T)[None, :] <= np.arange(T)[:, None]) & (seg[:, None] < dseg[None, :])
    out = np.zeros((T, Hq, D))
    for ver in range(tab["n_ver"]):
        rows = np.nonzero(tver == ver)[0]
        if len(rows) == 0:
            continue
        p = tab["pos"][ver]
        qr = rope(Q[rows], p[rows][:, None], base)
        kr = rope(K, np.maximum(p, 0)[:, None], base)
        m = mask[rows]
        for g in range(Hkv):
            for hh in range(grp):
                h = g * grp + hh
                s = qr[:, h] @ kr[:, g].T / math.sqrt(D)
                s = np.where(m, s, -np.inf)
                s -= s.max(axis=1, keepdims=True)
                w = np.exp(s)
                w /= w.sum(axis=1, keepdims=True)
                out[rows, h] = w @ V[:, g]
    return out, tab
