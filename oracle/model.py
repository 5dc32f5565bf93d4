"""Multi-layer decoder replayed message by message, float64.

Test infrastructure only.  A pre-norm decoder (RMSNorm -> Q/K/V projection ->
RoPE attention over the layer's active cache -> output projection ->
residual -> RMSNorm -> SwiGLU FFN -> residual; final RMSNorm) run over one
request whose cache is shaped by an op log, as in "Cache Engineering for
Agents" (paper review page sections 3.3-3.4, Figure 5): every layer keeps its
own K/V entries, and all layers share one active set and one position table.

Tokens are appended in order.  Tokens of one message see the cache as it was
when the message began plus the message's earlier tokens, so a message is
computed as one causal block; the ops between messages are applied exactly as
``core.replay`` applies them.  Keys are kept raw and rotated at their current
position whenever they are read (R(q-p) R(p) k = R(q) k in exact arithmetic).
"""
from __future__ import annotations

import math

import numpy as np

from .core import replay, rope, widen

_ROWS = 512  # query rows per block inside a long message (rows are independent)


def rmsnorm(x: np.ndarray, eps: float) -> np.ndarray:
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)


def _silu(x):
    return x / (1.0 + np.exp(-x))


def model_replay(weights, x, msg_start, drop_after, drop_target, repos_after, Hq, Hkv, D, base,
                 eps, dtype: str = "bf16", capture_layers: bool = False):
    """Final normed hidden states [T, d] (and, with ``capture_layers``, each
    layer's attention output [T, Hq*D] before the output projection)."""
    ms = [int(a) for a in msg_start]
    T = ms[-1]
    n_msgs = len(ms) - 1
    L = len(weights)
    W = [{k: widen(v, dtype) for k, v in w.items()} for w in weights]
    X = widen(x, dtype)
    grp = Hq // Hkv

    # integer schedule: the positions each message's tokens get and the
    # active cache (logical order + current positions) before each message
    before = {}
    tok_pos = np.zeros(T, dtype=np.int64)

    def on_token(t, p, act_u, act_p):
        tok_pos[t] = p
        m = int(np.searchsorted(ms, t, side="right") - 1)
        if t == ms[m]:
            before[m] = (np.array(act_u[:-1], dtype=np.int64), np.array(act_p[:-1], dtype=np.int64))

    replay(msg_start, drop_after, drop_target, repos_after, on_token)

    Kc = [np.zeros((T, Hkv, D)) for _ in range(L)]
    Vc = [np.zeros((T, Hkv, D)) for _ in range(L)]
    out = np.zeros((T, X.shape[1]))
    attn_out = [np.zeros((T, Hq * D)) for _ in range(L)] if capture_layers else None
    for m in range(n_msgs):
        t0, t1 = ms[m], ms[m + 1]
        if t1 == t0:
            continue
        pu, pp = before[m]
        n = t1 - t0
        h = X[t0:t1].copy()
        for l in range(L):
            w = W[l]
            a = rmsnorm(h, eps)
            qn = (a @ w["wq"]).reshape(n, Hq, D)
            Kc[l][t0:t1] = (a @ w["wk"]).reshape(n, Hkv, D)
            Vc[l][t0:t1] = (a @ w["wv"]).reshape(n, Hkv, D)
            keys_u = np.concatenate([pu, np.arange(t0, t1)])
            keys_p = np.concatenate([pp, tok_pos[t0:t1]])
            qr = rope(qn, tok_pos[t0:t1][:, None], base)
            kr = rope(Kc[l][keys_u], keys_p[:, None], base)
            vv = Vc[l][keys_u]
            npre = len(pu)
            o = np.zeros((n, Hq, D))
            for r0 in range(0, n, _ROWS):
                r1 = min(n, r0 + _ROWS)
                # row i sees all earlier-active keys and message tokens 0..i
                own = np.arange(n)[None, :] <= np.arange(r0, r1)[:, None]
                vis = np.concatenate([np.ones((r1 - r0, npre), dtype=bool), own], axis=1)
                for g in range(Hkv):
                    s = np.einsum("rhd,kd->hrk", qr[r0:r1, g * grp:(g + 1) * grp], kr[:, g])
                    s = s / math.sqrt(D)
                    s = np.where(vis[None], s, -np.inf)
                    s -= s.max(axis=2, keepdims=True)
                    e = np.exp(s)
                    e /= e.sum(axis=2, keepdims=True)
                    o[r0:r1, g * grp:(g + 1) * grp] = np.einsum("hrk,kd->rhd", e, vv[:, g])
            o = o.reshape(n, Hq * D)
            if capture_layers:
                attn_out[l][t0:t1] = o
            h = h + o @ w["wo"]
            f = rmsnorm(h, eps)
            h = h + (_silu(f @ w["wg"]) * (f @ w["wu"])) @ w["wd"]
        out[t0:t1] = rmsnorm(h, eps)
    return (out, attn_out) if capture_layers else out
