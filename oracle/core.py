"""Sequential replay of the cache-operation log, in float64.

Test infrastructure only (see the package docstring).

Definitions restated from "Cache Engineering for Agents" (arXiv 2610.28577),
paper review page, section 3.3 "three cache operations", section 3.4, and the
operate-after request grammar of Figure 6 / section 4:

* append: the token's KV joins the active cache C <- [C; C_{t+1}] at the next
  position, and the token attends over C including itself;
* drop(P): C <- C \\ {C_i : i in P}; survivors keep values, positions and
  logical tokens, and the next position does not move;
* repos: survivors are renumbered 0..r-1 in logical order, a key moving from
  p to q is rotated by R(q - p) and its value is unchanged; the next append
  position becomes r.
* "drop {i: [j]}" acts after message i ends; "reposition [i]" likewise; at one
  boundary every drop happens before the repos (Figure 6; system README
  example {"drop_message": {"4": [2]}, "reposition": [4]}).

Readings where the pages are silent (each also listed in the design notes):
RoPE pairs coordinate i with i + D/2 and turns it by p * base^(-2i/D);
scores are scaled by 1/sqrt(D); a boundary that lists at least one op starts
a new segment; dropping an already-dropped message is a no-op; a drop target
must not be later than its boundary.
"""
from __future__ import annotations

import math

import numpy as np

NEVER = np.iinfo(np.int32).max  # drop segment of a token that is never dropped


class OpLogError(ValueError):
    """The op log is not a valid operate-after log for these messages."""


def widen(x: np.ndarray, dtype: str) -> np.ndarray:
    """float32 values or bfloat16 bit patterns -> float64 (exact); "f64" passes through."""
    if dtype == "f64":
        return np.asarray(x, dtype=np.float64)
    if dtype == "f32":
        return np.asarray(x, dtype=np.float32).astype(np.float64)
    if dtype == "bf16":
        b = np.asarray(x, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
        return b.view(np.float32).astype(np.float64)
    raise ValueError(dtype)


def rope(x: np.ndarray, pos, base: float) -> np.ndarray:
    """R(pos) x for rotary position embedding, last axis of size D.

    Coordinates i and i + D/2 form a pair turned by the angle
    pos * base^(-2i/D), i < D/2.  ``pos`` broadcasts against x[..., 0]."""
    x = np.asarray(x, dtype=np.float64)
    D = x.shape[-1]
    h = D // 2
    theta = base ** (-2.0 * np.arange(h, dtype=np.float64) / D)
    ang = np.asarray(pos, dtype=np.float64)[..., None] * theta
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :h], x[..., h:]
    return np.concatenate([x1 * c - x2 * s, x1 * s + x2 * c], axis=-1)


def validate(msg_start, drop_after, drop_target, repos_after) -> None:
    """Reject logs the operate-after grammar cannot express."""
    ms = np.asarray(msg_start)
    if ms.ndim != 1 or len(ms) < 1 or ms[0] != 0 or np.any(np.diff(ms) < 0):
        raise OpLogError("message starts must begin at 0 and not decrease")
    n = len(ms) - 1
    da, dt, ra = (np.asarray(a, dtype=np.int64) for a in (drop_after, drop_target, repos_after))
    if len(da) != len(dt):
        raise OpLogError("drop boundary / target arrays differ in length")
    if np.any((da < 0) | (da >= n)):
        raise OpLogError("drop boundary out of range")
    if np.any((dt < 0) | (dt > da)):
        raise OpLogError("drop target must be an already appended message")
    if np.any((ra < 0) | (ra >= n)):
        raise OpLogError("repos boundary out of range")


class ReplayResult:
    """Integer record of a replay.

    tok_pos[t]  position token t was appended at
    tok_seg[t]  number of op-carrying boundaries before t's message
    tok_ver[t]  number of repos before t's message
    drop_seg[u] segment index from which u is no longer visible (NEVER if kept)
    active_u / active_p  active cache at the stop point (logical order)
    next_pos    next append position at the stop point
    """

    def __init__(self, T):
        self.tok_pos = np.full(T, -1, dtype=np.int64)
        self.tok_seg = np.full(T, -1, dtype=np.int64)
        self.tok_ver = np.full(T, -1, dtype=np.int64)
        self.drop_seg = np.full(T, NEVER, dtype=np.int64)
        self.active_u = None
        self.active_p = None
        self.next_pos = 0
        self.n_seg = 0
        self.n_ver = 0


def replay(msg_start, drop_after, drop_target, repos_after, on_token=None, upto=None,
           pos_offset: int = 0) -> ReplayResult:
    """Run the op sequence from an empty cache, one token at a time.

    ``on_token(t, p, act_u, act_p)`` is called right after token t is appended
    at position p, with the active cache (lists, logical order, t included).
    ``upto``: stop after the drops of boundary ``upto`` (before its repos).
    ``pos_offset`` adds a constant to every position (a RoPE invariance check)."""
    validate(msg_start, drop_after, drop_target, repos_after)
    ms = [int(x) for x in msg_start]
    n_msgs = len(ms) - 1
    T = ms[-1]
    drops_at: dict[int, list[int]] = {}
    for a, t in zip(drop_after, drop_target):
        drops_at.setdefault(int(a), []).append(int(t))
    repos_at = {int(a) for a in repos_after}

    res = ReplayResult(T)
    act_u: list[int] = []
    act_p: list[int] = []
    next_pos = pos_offset
    seg = 0
    ver = 0
    for m in range(n_msgs):
        for t in range(ms[m], ms[m + 1]):
            p = next_pos
            next_pos += 1
            act_u.append(t)
            act_p.append(p)
            res.tok_pos[t], res.tok_seg[t], res.tok_ver[t] = p, seg, ver
            if on_token is not None:
                on_token(t, p, act_u, act_p)
        targets = drops_at.get(m, [])
        if targets:
            gone = set()
            for j in targets:
                gone.update(range(ms[j], ms[j + 1]))
            keep_u, keep_p = [], []
            for u, p in zip(act_u, act_p):
                if u in gone:
                    res.drop_seg[u] = seg + 1
                else:
                    keep_u.append(u)
                    keep_p.append(p)
            act_u, act_p = keep_u, keep_p
        if upto is not None and m == upto:
            break
        if m in repos_at:
            act_p = [pos_offset + i for i in range(len(act_u))]
            next_pos = pos_offset + len(act_u)
            ver += 1
        if targets or m in repos_at:
            seg += 1
    res.active_u = np.array(act_u, dtype=np.int64)
    res.active_p = np.array(act_p, dtype=np.int64)
    res.next_pos = next_pos
    res.n_seg = seg + 1
    res.n_ver = ver + 1
    return res


def _attend_row(q_row, p_t, keys_u, keys_p, K, V, dtype, base):
    """Attention of one raw query row [Hq, D] at position p_t over raw keys
    K[keys_u] rotated at keys_p, values V[keys_u]; softmax with the row max
    subtracted, scale 1/sqrt(D).  GQA: query head h reads KV head h // (Hq/Hkv)."""
    Hq, D = q_row.shape
    Hkv = K.shape[1]
    grp = Hq // Hkv
    qr = rope(widen(q_row, dtype), p_t, base)
    kr = rope(widen(K[keys_u], dtype), np.asarray(keys_p)[:, None], base)
    vv = widen(V[keys_u], dtype)
    out = np.empty((Hq, D), dtype=np.float64)
    for g in range(Hkv):
        s = qr[g * grp:(g + 1) * grp] @ kr[:, g].T / math.sqrt(D)
        s -= s.max(axis=1, keepdims=True)
        w = np.exp(s)
        w /= w.sum(axis=1, keepdims=True)
        out[g * grp:(g + 1) * grp] = w @ vv[:, g]
    return out


def replay_attention(msg_start, drop_after, drop_target, repos_after, q, k, v, dtype: str,
                     base: float, rows=None, pos_offset: int = 0):
    """Single-layer attention outputs for ``rows`` (all rows if None), float64.

    Row t attends, with its query rotated at its append position, over the
    active cache at its append time, each key rotated at its current position.
    Returns (out [len(rows), Hq, D], ReplayResult)."""
    T = int(msg_start[-1])
    rows = np.arange(T) if rows is None else np.asarray(rows, dtype=np.int64)
    where = {int(t): i for i, t in enumerate(rows)}
    Hq, D = q.shape[1], q.shape[2]
    out = np.full((len(rows), Hq, D), np.nan)

    def on_token(t, p, act_u, act_p):
        i = where.get(t)
        if i is not None:
            out[i] = _attend_row(q[t], p, np.array(act_u), np.array(act_p), k, v, dtype, base)

    res = replay(msg_start, drop_after, drop_target, repos_after, on_token, pos_offset=pos_offset)
    return out, res


def visible_counts(msg_start, drop_after, drop_target, repos_after) -> np.ndarray:
    """Number of keys each token attends over (size of the active cache at its
    append time, itself included)."""
    T = int(msg_start[-1])
    cnt = np.zeros(T, dtype=np.int64)

    def on_token(t, p, act_u, act_p):
        cnt[t] = len(act_u)

    replay(msg_start, drop_after, drop_target, repos_after, on_token)
    return cnt


def compact(msg_start, drop_after, drop_target, repos_after, upto: int = -1):
    """Active cache after the drops of boundary ``upto`` (-1: the last message).

    Returns (logical indices ascending, their positions).  Positions are those
    in effect before any repos listed at ``upto``; a repos there would move the
    j-th survivor to position j."""
    n_msgs = len(msg_start) - 1
    if upto < 0:
        upto = n_msgs - 1
    if not 0 <= upto < n_msgs:
        raise OpLogError("boundary out of range")
    res = replay(msg_start, drop_after, drop_target, repos_after, upto=upto)
    return res.active_u, res.active_p


def repos_rotate(k_in, v_in, src_idx, pos_from, pos_to, dtype: str, base: float):
    """Move keys K[src_idx[j]] from position pos_from[j] to pos_to[j] by the
    rotation R(pos_to - pos_from); values are copied unchanged (section 3.3)."""
    src = np.asarray(src_idx, dtype=np.int64)
    delta = np.asarray(pos_to, dtype=np.float64) - np.asarray(pos_from, dtype=np.float64)
    k_out = rope(widen(k_in[src], dtype), delta[:, None], base)
    v_out = widen(v_in[src], dtype)
    return k_out, v_out


def decode_attention(q, q_pos, k_pool, v_pool, kv_indptr, kv_indices, dtype: str, base: float):
    """One query per request over its active cache in a page-size-1 pool.

    q [B, Hq, D] raw, rotated at q_pos[b]; pool keys are stored already rotated;
    request b reads slots kv_indices[kv_indptr[b]:kv_indptr[b+1]]."""
    B, Hq, D = q.shape
    Hkv = k_pool.shape[1]
    grp = Hq // Hkv
    out = np.empty((B, Hq, D), dtype=np.float64)
    for b in range(B):
        sl = np.asarray(kv_indices[kv_indptr[b]:kv_indptr[b + 1]], dtype=np.int64)
        qr = rope(widen(q[b], dtype), q_pos[b], base)
        kk = widen(k_pool[sl], dtype)
        vv = widen(v_pool[sl], dtype)
        for g in range(Hkv):
            s = qr[g * grp:(g + 1) * grp] @ kk[:, g].T / math.sqrt(D)
            s -= s.max(axis=1, keepdims=True)
            w = np.exp(s)
            w /= w.sum(axis=1, keepdims=True)
            out[b, g * grp:(g + 1) * grp] = w @ vv[:, g]
    return out
