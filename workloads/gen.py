"""Seeded generators for the five AKV workloads and for random parity cases.

Shapes and distributions follow the workloads the pages describe for
"Cache Engineering for Agents" (arXiv 2610.28577):

* agent trajectories of assistant reasoning + tool responses, with the
  tool-response rolling drop that keeps the last 12 tool responses
  (section 3.2 and section 5.1 of the paper review page);
* a repos whenever the next position reaches the summarisation threshold
  (96k, section 5.1);
* decode over a token-granular (page size 1) pool after drops (system
  README: drop/repos support page size 1 only);
* a small decoder whose requests share a prefix and diverge in their cache
  operations like the three trajectories of Figure 5.

Every array is drawn from ``numpy.random.default_rng`` seeded through
``SeedSequence(seed).spawn``; float inputs are standard normals in float32,
rounded to bfloat16 (round to nearest even) where the workload is bf16.
bf16 tensors are returned as their uint16 bit patterns so that both
consumers read exactly the same bytes.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

_CHUNK = 1 << 24


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns, round to nearest even (finite inputs)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    fb = x.reshape(-1).view(np.uint32)
    ob = out.reshape(-1)
    for s in range(0, fb.size, _CHUNK):
        b = fb[s:s + _CHUNK]
        r = b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))
        ob[s:s + _CHUNK] = (r >> np.uint32(16)).astype(np.uint16)
    return out


def _normals(rng: np.random.Generator, shape, dtype: str, scale: float = 1.0) -> np.ndarray:
    """N(0, scale^2) samples as float32, or as bf16 bits when dtype == 'bf16'.

    Drawn chunk by chunk from one generator, so the stream does not depend on
    the chunking."""
    n = int(np.prod(shape))
    if dtype == "f32":
        out = rng.standard_normal(n, dtype=np.float32)
        if scale != 1.0:
            out *= np.float32(scale)
        return out.reshape(shape)
    out = np.empty(n, dtype=np.uint16)
    for s in range(0, n, _CHUNK):
        m = min(_CHUNK, n - s)
        f = rng.standard_normal(m, dtype=np.float32)
        if scale != 1.0:
            f *= np.float32(scale)
        out[s:s + m] = bf16_bits(f)
    return out.reshape(shape)


def _streams(seed: int, n: int):
    return [np.random.default_rng(s) for s in np.random.SeedSequence(seed).spawn(n)]


@dataclass
class Trajectory:
    """One request: messages (token CSR), an operate-after op log and raw Q/K/V.

    ``drop_after[i], drop_target[i]``: after message ``drop_after[i]`` ends,
    drop message ``drop_target[i]``.  ``repos_after[j]``: after that message
    ends (and after that boundary's drops), re-position.  Indices are 0-based
    message indices.  Messages from ``n_prefill_msgs`` on are decode appends
    (one token each)."""
    name: str
    Hq: int
    Hkv: int
    D: int
    rope_base: float
    dtype: str
    msg_start: np.ndarray
    roles: list
    drop_after: np.ndarray
    drop_target: np.ndarray
    repos_after: np.ndarray
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    n_prefill_msgs: int = -1
    meta: dict = field(default_factory=dict)

    @property
    def T(self) -> int:
        return int(self.msg_start[-1])

    @property
    def n_msgs(self) -> int:
        return len(self.msg_start) - 1

    @property
    def T_prefill(self) -> int:
        n = self.n_msgs if self.n_prefill_msgs < 0 else self.n_prefill_msgs
        return int(self.msg_start[n])

    def ops(self):
        return (self.msg_start, self.drop_after, self.drop_target, self.repos_after)


def _ops_arrays(drops, repos):
    da = np.array([a for a, _ in drops], dtype=np.int32)
    dt = np.array([t for _, t in drops], dtype=np.int32)
    ra = np.array(sorted(repos), dtype=np.int32)
    return da, dt, ra


def tiny_config(seed: int = 1) -> Trajectory:
    """The worked request of Figure 6 with lengths 16/24/32, then 8 decodes.

    user(16), assistant(24), tool(32); drop {1: [0], 2: [1]}; reposition [2];
    then eight single-token decode appends.  fp32, 2 heads, head_dim 64."""
    lens = [16, 24, 32] + [1] * 8
    roles = ["user", "assistant", "tool"] + ["decode"] * 8
    msg_start = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T = int(msg_start[-1])
    rq, rk, rv = _streams(seed, 3)
    da, dt, ra = _ops_arrays([(1, 0), (2, 1)], [2])
    return Trajectory("tiny_fp32", 2, 2, 64, 10000.0, "f32", msg_start, roles, da, dt, ra,
                      _normals(rq, (T, 2, 64), "f32"), _normals(rk, (T, 2, 64), "f32"),
                      _normals(rv, (T, 2, 64), "f32"), n_prefill_msgs=3)


def agent_trajectory(seed: int, rounds: int | None = None, total_tokens: int | None = None,
                     keep_tools: int = 12, repos_threshold: int | None = None,
                     truncate_at_boundary: int | None = None,
                     asst_len=(100, 300), tool_len=(300, 1500)):
    """Message lengths and op log of an assistant/tool agent trajectory.

    Rolling drop: after the k-th tool response ends, if k > keep_tools, the
    tool response k - keep_tools is dropped at that same boundary.  Reasoning
    is never dropped.  With ``repos_threshold`` a repos is issued at the first
    boundary where the next position is >= threshold (after that boundary's
    drops); positions then restart at the number of surviving tokens.
    ``total_tokens`` truncates the last message so T is exact;
    ``truncate_at_boundary`` stops at the first boundary with >= that many tokens.
    Returns (msg_start, roles, drops, repos)."""
    rl = _streams(seed, 1)[0]
    lens, roles = [], []
    total = 0
    r = 0
    while True:
        if rounds is not None and r >= rounds:
            break
        for role, (lo, hi) in (("assistant", asst_len), ("tool", tool_len)):
            n = int(rl.integers(lo, hi + 1))
            if total_tokens is not None and total + n >= total_tokens:
                n = total_tokens - total
            lens.append(n)
            roles.append(role)
            total += n
            if total_tokens is not None and total >= total_tokens:
                break
            if truncate_at_boundary is not None and total >= truncate_at_boundary:
                break
        if total_tokens is not None and total >= total_tokens:
            break
        if truncate_at_boundary is not None and total >= truncate_at_boundary:
            break
        r += 1
    # policy: rolling tool drop and threshold repos (harness side of the API)
    drops, repos = [], []
    tools_seen = []
    next_pos = 0
    alive = [True] * len(lens)
    for m, (n, role) in enumerate(zip(lens, roles)):
        next_pos += n
        if role == "tool":
            tools_seen.append(m)
            if len(tools_seen) > keep_tools:
                tgt = tools_seen[len(tools_seen) - keep_tools - 1]
                drops.append((m, tgt))
                alive[tgt] = False
        if repos_threshold is not None and next_pos >= repos_threshold:
            repos.append(m)
            next_pos = sum(l for l, a in zip(lens[:m + 1], alive[:m + 1]) if a)
    msg_start = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    return msg_start, roles, drops, repos


def _trajectory(name, seed, msg_start, roles, drops, repos, Hq, Hkv, D, dtype, base=10000.0,
                q_scale=1.0):
    T = int(msg_start[-1])
    _, rq, rk, rv = _streams(seed, 4)
    da, dt, ra = _ops_arrays(drops, repos)
    return Trajectory(name, Hq, Hkv, D, base, dtype, msg_start, roles, da, dt, ra,
                      _normals(rq, (T, Hq, D), dtype, q_scale), _normals(rk, (T, Hkv, D), dtype),
                      _normals(rv, (T, Hkv, D), dtype))


def rolling_drop_config(seed: int = 2, rounds: int = 100, truncate_at_boundary: int | None = None,
                        Hq: int = 64, Hkv: int = 8, D: int = 64, q_scale: float = 1.0) -> Trajectory:
    """GQA 64/8 layer, 100 rounds (assistant U{100..300}, tool U{300..1500}),
    keep-12 rolling tool drop, no repos, bf16."""
    ms, roles, drops, repos = agent_trajectory(seed, rounds=rounds,
                                               truncate_at_boundary=truncate_at_boundary)
    tag = "" if truncate_at_boundary is None else f"_trunc{truncate_at_boundary}"
    return _trajectory(f"rolling_drop_{rounds}r{tag}", seed, ms, roles, drops, repos, Hq, Hkv, D,
                       "bf16", q_scale=q_scale)


def repos_config(seed: int = 3, total_tokens: int = 131072, repos_threshold: int = 98304,
                 Hq: int = 64, Hkv: int = 8, D: int = 64, q_scale: float = 1.0) -> Trajectory:
    """128k-token trajectory, rolling drop, repos at next position >= 96k, bf16."""
    ms, roles, drops, repos = agent_trajectory(seed, total_tokens=total_tokens,
                                               repos_threshold=repos_threshold)
    return _trajectory(f"repos_{total_tokens}", seed, ms, roles, drops, repos, Hq, Hkv, D, "bf16",
                       q_scale=q_scale)


def random_request(seed: int, n_msgs: int, max_len: int, Hq: int = 4, Hkv: int = 2, D: int = 64,
                   dtype: str = "bf16", p_drop: float = 0.3, p_repos: float = 0.2,
                   min_len: int = 0, q_scale: float = 1.0, name: str = "random") -> Trajectory:
    """A random valid request: message lengths U{min_len..max_len}, and at each
    boundary i each earlier-or-current message dropped with prob p_drop (at
    most once; re-dropping is legal but pointless) and a repos with prob p_repos."""
    rng = _streams(seed, 1)[0]
    lens = rng.integers(min_len, max_len + 1, size=n_msgs)
    msg_start = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    drops, repos = [], []
    dropped = set()
    for i in range(n_msgs):
        for j in range(i + 1):
            if j not in dropped and rng.random() < p_drop:
                drops.append((i, j))
                dropped.add(j)
        if rng.random() < p_repos:
            repos.append(i)
    t = _trajectory(name, seed + 1000, msg_start, ["msg"] * n_msgs, drops, repos, Hq, Hkv, D,
                    dtype, q_scale=q_scale)
    return t


def shared_prefix_batch(seed: int, n_req: int, prefix: int, n_msgs: int, max_len: int,
                        Hq: int = 4, Hkv: int = 2, D: int = 64, dtype: str = "bf16",
                        p_drop: float = 0.3, p_repos: float = 0.2) -> list:
    """Requests that start with the same ``prefix``-token message (identical
    Q/K/V rows), then diverge: their own message lengths U{1..max_len}, drops
    of later messages only (each at a random boundary at or after its end),
    repos at random boundaries."""
    out = []
    pre = None
    for b in range(n_req):
        rng = _streams(seed * 7919 + b, 1)[0]
        lens = [prefix] + [int(x) for x in rng.integers(1, max_len + 1, size=n_msgs - 1)]
        msg_start = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        drops, repos = [], []
        for m in range(1, n_msgs):
            if rng.random() < p_drop:
                drops.append((int(rng.integers(m, n_msgs)), m))
        for m in range(n_msgs):
            if rng.random() < p_repos:
                repos.append(m)
        t = _trajectory(f"shared_{b}", seed * 100 + b, msg_start, ["msg"] * n_msgs, drops, repos,
                        Hq, Hkv, D, dtype)
        if pre is None:
            pre = (t.q[:prefix].copy(), t.k[:prefix].copy(), t.v[:prefix].copy())
        else:
            t.q[:prefix], t.k[:prefix], t.v[:prefix] = pre
        out.append(t)
    return out


@dataclass
class DecodeWorkload:
    """B requests decoding over a page-size-1 pool.

    ``active_slots[b]``: pool slots of request b's active (surviving) tokens in
    logical order; ``L[b]``: its logical length (positions 0..L-1 were used;
    dropped tokens keep their positions).  Pool keys are treated as already
    rotated.  At decode step i request b appends token L[b]+i into
    ``append_slots[i, b]`` with raw ``k_new[i, b]`` / ``v_new[i, b]`` and
    queries with raw ``q[i, b]`` at position L[b]+i."""
    Hq: int
    Hkv: int
    D: int
    rope_base: float
    dtype: str
    L: np.ndarray
    active_slots: list
    append_slots: np.ndarray
    k_pool: np.ndarray
    v_pool: np.ndarray
    q: np.ndarray
    k_new: np.ndarray
    v_new: np.ndarray

    @property
    def B(self):
        return len(self.L)

    @property
    def steps(self):
        return self.q.shape[0]

    @property
    def S(self):
        return self.k_pool.shape[0]

    def indices_at(self, step: int):
        """CSR (indptr, indices) of the cache each request reads at ``step``:
        its active slots followed by the slots appended at steps 0..step."""
        parts, indptr = [], [0]
        for b in range(self.B):
            parts.append(self.active_slots[b])
            parts.append(self.append_slots[:step + 1, b])
            indptr.append(indptr[-1] + len(self.active_slots[b]) + step + 1)
        return (np.array(indptr, dtype=np.int32),
                np.concatenate(parts).astype(np.int32))


def decode_workload(seed: int = 4, B: int = 14, active=(20000, 90000), drop_frac=(0.30, 0.60),
                    steps: int = 256, Hq: int = 64, Hkv: int = 8, D: int = 64, spare: float = 0.10,
                    dtype: str = "bf16") -> DecodeWorkload:
    """Active length a_b ~ U{lo..hi}, dropped fraction f_b ~ U[lo, hi), logical
    length L_b = round(a_b / (1 - f_b)); the surviving logical tokens are a
    uniformly random subset of size a_b.  Pool slots are a random permutation."""
    r_len, r_perm, r_pool_k, r_pool_v, r_q, r_kn, r_vn, r_sub = _streams(seed, 8)
    a = r_len.integers(active[0], active[1] + 1, size=B)
    f = r_len.uniform(drop_frac[0], drop_frac[1], size=B)
    L = np.rint(a / (1.0 - f)).astype(np.int64)
    n_used = int(a.sum()) + B * steps
    S = int(np.ceil(n_used * (1.0 + spare)))
    perm = r_perm.permutation(S).astype(np.int32)
    active_slots, off = [], 0
    for b in range(B):
        active_slots.append(perm[off:off + int(a[b])].copy())
        off += int(a[b])
    append_slots = perm[off:off + B * steps].reshape(steps, B).copy()
    # which logical tokens survive is not needed by the kernels (keys are
    # pre-rotated); it is drawn for the record.
    _ = [np.sort(r_sub.choice(int(L[b]), size=int(a[b]), replace=False)) for b in range(B)]
    return DecodeWorkload(Hq, Hkv, D, 10000.0, dtype, L.astype(np.int32), active_slots,
                          append_slots, _normals(r_pool_k, (S, Hkv, D), dtype),
                          _normals(r_pool_v, (S, Hkv, D), dtype),
                          _normals(r_q, (steps, B, Hq, D), dtype),
                          _normals(r_kn, (steps, B, Hkv, D), dtype),
                          _normals(r_vn, (steps, B, Hkv, D), dtype))


@dataclass
class ModelWorkload:
    """A random-init decoder and a batch of requests sharing one token stream.

    Every request has the same message layout and the same input embeddings
    ``x`` (a shared prefix message followed by assistant/tool messages);
    requests differ only in their op logs.  Weights are stored [in, out]."""
    n_layers: int
    d_model: int
    Hq: int
    Hkv: int
    D: int
    d_ff: int
    rope_base: float
    eps: float
    msg_start: np.ndarray
    x: np.ndarray
    weights: list
    ops: list  # per request: (drop_after, drop_target, repos_after)

    @property
    def T(self):
        return int(self.msg_start[-1])

    @property
    def n_req(self):
        return len(self.ops)


def model_workload(seed: int = 5, n_req: int = 32, prefix: int = 8192, following: int = 24576,
                   n_layers: int = 4, d_model: int = 1024, Hq: int = 16, Hkv: int = 4, D: int = 64,
                   d_ff: int = 4096, asst_len=(100, 300), tool_len=(300, 1500)) -> ModelWorkload:
    """Requests share a ``prefix``-token user message and the same ``following``
    tokens split into assistant/tool messages; request b drops a random subset
    of tool messages, each at a random boundary at or after its end, and issues
    (b mod 3) repos at random boundaries.  x ~ N(0,1), weights ~ N(0, 0.02^2),
    bf16; RMSNorm weights are 1 and eps 1e-6."""
    r_len, r_x, r_w, r_ops = _streams(seed, 4)
    lens, roles = [prefix], ["user"]
    total = 0
    while total < following:
        for role, (lo, hi) in (("assistant", asst_len), ("tool", tool_len)):
            n = min(int(r_len.integers(lo, hi + 1)), following - total)
            lens.append(n)
            roles.append(role)
            total += n
            if total >= following:
                break
    msg_start = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    n_msgs = len(lens)
    T = int(msg_start[-1])
    x = _normals(r_x, (T, d_model), "bf16")
    weights = []
    for _ in range(n_layers):
        w = {}
        for name, shp in (("wq", (d_model, Hq * D)), ("wk", (d_model, Hkv * D)),
                          ("wv", (d_model, Hkv * D)), ("wo", (Hq * D, d_model)),
                          ("wg", (d_model, d_ff)), ("wu", (d_model, d_ff)),
                          ("wd", (d_ff, d_model))):
            w[name] = _normals(r_w, shp, "bf16", 0.02)
        weights.append(w)
    tool_msgs = [m for m, r in enumerate(roles) if r == "tool"]
    ops = []
    for b in range(n_req):
        rb = _streams(seed * 1000 + b, 1)[0]
        drops = []
        for m in tool_msgs:
            if rb.random() < 0.5:
                drops.append((int(rb.integers(m, n_msgs)), m))
        n_rep = b % 3
        repos = sorted(int(x_) for x_ in rb.choice(n_msgs, size=min(n_rep, n_msgs), replace=False))
        da, dt, ra = _ops_arrays(drops, repos)
        ops.append((da, dt, ra))
    return ModelWorkload(n_layers, d_model, Hq, Hkv, D, d_ff, 10000.0, 1e-6, msg_start, x,
                         weights, ops)
