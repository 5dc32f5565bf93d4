"""Helpers shared by the GPU parity tests: move seeded inputs to the device,
run the C-ABI calls, and compare with the oracle."""
import numpy as np

import kv_cache_drop_gb300 as akv
import oracle

BF16_MAX_ABS = 2e-2        # bf16 inputs, fp32 accumulation
BF16_REL_RMS = 2.0 ** -7   # error RMS / reference RMS
F32_MAX_ABS = 1e-4
# Queries scaled by 8 (score std ~8, a far from flat softmax) keep the same
# bars: the stated tolerance is for bf16 inputs with fp32 accumulation,
# whatever the score scale.


def run_prefill(reqs, device="cuda"):
    """Segment-batch prefill of a batch of requests; returns (out [T,Hq,D]
    float32 numpy, plan, workspace)."""
    import torch
    r0 = reqs[0]
    shp = akv.shape(r0.Hq, r0.Hkv, 64, r0.dtype, r0.rope_base)
    cu = np.concatenate([[0], np.cumsum([r.T_prefill for r in reqs])]).astype(np.int32)
    ops = []
    for r in reqs:
        n = r.n_msgs if r.n_prefill_msgs < 0 else r.n_prefill_msgs
        keep_d = r.drop_after < n
        ops.append((r.msg_start[:n + 1], r.drop_after[keep_d], r.drop_target[keep_d],
                    r.repos_after[r.repos_after < n]))
    plan = akv.Plan(shp, cu, ops)
    q = akv.to_device(np.concatenate([r.q[:r.T_prefill] for r in reqs]), r0.dtype, device)
    k = akv.to_device(np.concatenate([r.k[:r.T_prefill] for r in reqs]), r0.dtype, device)
    v = akv.to_device(np.concatenate([r.v[:r.T_prefill] for r in reqs]), r0.dtype, device)
    out = torch.zeros_like(q)
    ws = plan.workspace(device)
    akv.akv_segment_attention_run(plan, q, k, v, out, ws)
    torch.cuda.synchronize()
    assert akv.akv_workspace_status(ws) == 0, "a kernel barrier wait timed out"
    return out.float().cpu().numpy(), plan, ws


def prefill_ops(r):
    """The request's op log restricted to its prefill messages."""
    n = r.n_msgs if r.n_prefill_msgs < 0 else r.n_prefill_msgs
    keep_d = r.drop_after < n
    return (r.msg_start[:n + 1], r.drop_after[keep_d], r.drop_target[keep_d],
            r.repos_after[r.repos_after < n])


def oracle_rows(r, rows=None):
    """fp64 oracle rows of a request's prefill; more than 32 rows are spread
    over worker processes (one per host core)."""
    ops = prefill_ops(r)
    T = r.T_prefill
    if rows is not None and len(rows) > 32:
        from oracle.parallel import replay_attention_rows
        return replay_attention_rows(ops, r.q[:T], r.k[:T], r.v[:T], r.dtype, r.rope_base, rows)
    out, _ = oracle.replay_attention(*ops, r.q[:T], r.k[:T], r.v[:T], r.dtype, r.rope_base,
                                     rows=rows)
    return out


def err(got, ref):
    d = np.abs(got.astype(np.float64) - ref)
    rms_ref = float(np.sqrt(np.mean(ref * ref))) or 1.0
    return float(d.max()), float(np.sqrt(np.mean(d * d)) / rms_ref)


def assert_close(got, ref, dtype, max_abs=None):
    mx, rel = err(got, ref)
    print(f"[parity] {dtype} max_abs={mx:.3e} rel_rms={rel:.3e}")
    if dtype == "bf16":
        assert mx <= (max_abs or BF16_MAX_ABS) and rel <= BF16_REL_RMS, (mx, rel)
    else:
        assert mx <= F32_MAX_ABS, (mx, rel)
    return mx, rel


def sample_rows(r, n_random=24, seed=0):
    """Rows at message and tile edges plus random ones."""
    T = r.T_prefill
    rng = np.random.default_rng(seed)
    edges = {0, 1, T - 1, T - 2}
    for m in range(1, len(r.msg_start) - 1):
        s = int(r.msg_start[m])
        if 0 < s < T:
            edges.update({s - 1, s})
    edges = sorted(e for e in edges if 0 <= e < T)
    pick = list(rng.choice(edges, size=min(len(edges), n_random), replace=False))
    pick += list(rng.integers(0, T, size=n_random))
    for t0 in (127, 128, 129):
        if t0 < T:
            pick.append(t0)
    return np.unique(np.array(pick, dtype=np.int64))


TILE_Q = 128  # query rows per tile of the attention kernel's plan


def stratified_rows(r, n_total=256, seed=0):
    """At least ``n_total`` rows of a long request, chosen so that no part of
    the plan goes unsampled:

    * every segment (the rows between two op-carrying boundaries): its first
      and last row and one random row;
    * both sides of every op boundary (rows b-2, b-1, b, b+1);
    * the 128-row query tiles that straddle a drop boundary (tiles are
      counted from the first row of each key version, i.e. after each repos):
      the tile's first and last row and a random row.  Rows before the
      boundary still see the dropped message's keys and rows after it do
      not, so these tiles read the dropped keys through partially visible
      key windows;
    * random rows to reach ``n_total``."""
    ops = prefill_ops(r)
    T = r.T_prefill
    rep = oracle.replay(*ops)
    rng = np.random.default_rng(seed)
    pick = set()
    seg = rep.tok_seg
    for s_ in range(int(seg.max()) + 1):
        idx = np.flatnonzero(seg == s_)
        if len(idx):
            pick.update({int(idx[0]), int(idx[-1]), int(rng.choice(idx))})
    ms = ops[0]
    op_bounds = sorted({int(a) for a in ops[1]} | {int(a) for a in ops[3]})
    drop_bounds = sorted({int(a) for a in ops[1]})
    for a in op_bounds:
        b = int(ms[a + 1])
        pick.update(t for t in (b - 2, b - 1, b, b + 1) if 0 <= t < T)
    # first row of each key version
    vstart = [0] + [int(ms[a + 1]) for a in sorted({int(a) for a in ops[3]})]
    for a in drop_bounds:
        b = int(ms[a + 1])
        if not 0 < b < T:
            continue
        v0 = max(x for x in vstart if x <= b)
        t0 = v0 + (b - v0) // TILE_Q * TILE_Q
        if t0 == b:
            continue  # the boundary falls on a tile edge
        vend = min([x for x in vstart if x > b] + [T])
        t1 = min(t0 + TILE_Q, vend)
        pick.update({t0, t1 - 1, int(rng.integers(t0, t1))})
    need = n_total - len(pick)
    if need > 0:
        rest = np.setdiff1d(np.arange(T), np.fromiter(pick, dtype=np.int64))
        pick.update(int(x) for x in rng.choice(rest, size=min(need, len(rest)), replace=False))
    return np.array(sorted(pick), dtype=np.int64)
