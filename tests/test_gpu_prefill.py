"""Segment-batch restoration prefill on the GPU against the fp64 oracle."""
import numpy as np
import pytest

import kv_cache_drop_gb300 as akv
import workloads
from _util import assert_close, oracle_rows, run_prefill, sample_rows, stratified_rows

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("seed", range(6))
def test_prefill_bf16_random_logs(seed):
    r = workloads.random_request(10 + seed, n_msgs=8, max_len=260, Hq=8, Hkv=2, dtype="bf16",
                                 p_drop=0.3, p_repos=0.25)
    got, _, _ = run_prefill([r])
    assert_close(got, oracle_rows(r), "bf16")


@pytest.mark.parametrize("seed", range(3))
def test_prefill_bf16_peaky_scores(seed):
    """Queries scaled by 8: score std ~8, so the softmax is far from flat."""
    r = workloads.random_request(20 + seed, n_msgs=7, max_len=300, Hq=8, Hkv=2, dtype="bf16",
                                 p_drop=0.3, p_repos=0.3, q_scale=8.0)
    got, _, _ = run_prefill([r])
    assert_close(got, oracle_rows(r), "bf16")


def test_prefill_bf16_gqa_64_8_ragged_batch():
    reqs = [workloads.random_request(30 + i, n_msgs=4 + i, max_len=200, Hq=64, Hkv=8,
                                     dtype="bf16", p_drop=0.3, p_repos=0.3, min_len=1)
            for i in range(3)]
    got, plan, _ = run_prefill(reqs)
    off = 0
    for r in reqs:
        assert_close(got[off:off + r.T], oracle_rows(r), "bf16")
        off += r.T


@pytest.mark.parametrize("T", [1, 127, 128, 129, 256, 300])
def test_prefill_tile_edges(T):
    ms = np.array([0, T // 3, T // 3, T], dtype=np.int32)  # includes an empty message
    r = workloads.random_request(40, n_msgs=3, max_len=1, Hq=4, Hkv=2, dtype="bf16")
    rr = workloads.gen._trajectory("edge", 41, ms, ["m"] * 3, [(1, 0)], [1], 4, 2, 64, "bf16")
    got, _, _ = run_prefill([rr])
    assert_close(got, oracle_rows(rr), "bf16")


@pytest.mark.parametrize("seed", range(4))
def test_prefill_f32_random_logs(seed):
    r = workloads.random_request(50 + seed, n_msgs=7, max_len=60, Hq=4, Hkv=2, dtype="f32",
                                 p_drop=0.3, p_repos=0.3)
    got, _, _ = run_prefill([r])
    assert_close(got, oracle_rows(r), "f32")


def test_visible_counts_bit_exact():
    import torch
    import kv_cache_drop_gb300 as akv
    import oracle
    reqs = [workloads.random_request(60 + i, n_msgs=9, max_len=400, Hq=8, Hkv=2, dtype="bf16",
                                     p_drop=0.35, p_repos=0.25) for i in range(4)]
    _, plan, ws = run_prefill(reqs)
    counts = torch.zeros(plan.info["T"], dtype=torch.int32, device="cuda")
    akv.akv_segment_visible_counts(plan, counts, ws)
    got = counts.cpu().numpy()
    ref = np.concatenate([oracle.visible_counts(*r.ops()) for r in reqs])
    np.testing.assert_array_equal(got, ref)
    assert int(got.sum()) == plan.info["visible_pairs"]


def test_prefill_rolling_drop_medium():
    """25 rounds of the agent trajectory at the GQA 64/8 shape, sampled rows."""
    r = workloads.rolling_drop_config(rounds=25)
    got, _, _ = run_prefill([r])
    rows = sample_rows(r, 16)
    assert_close(got[rows], oracle_rows(r, rows), "bf16")


def test_prefill_rolling_drop_full_size():
    """The full 100-round trajectory (bench configuration): 256 or more rows
    covering every segment, both sides of every drop boundary and the query
    tiles that straddle one."""
    r = workloads.rolling_drop_config()
    got, plan, _ = run_prefill([r])
    assert np.isfinite(got).all()
    rows = stratified_rows(r, 256, seed=1)
    assert len(rows) >= 256
    assert_close(got[rows], oracle_rows(r, rows), "bf16")


def test_prefill_rolling_drop_48k_truncation():
    """The same trajectory cut at the first message boundary at or after
    49,152 tokens (the "~48k" reading of the workload), stratified rows, with
    a peaky query variant on the same rows."""
    r = workloads.rolling_drop_config(truncate_at_boundary=49152)
    assert 49152 <= r.T < 49152 + 3000
    got, _, _ = run_prefill([r])
    rows = stratified_rows(r, 160, seed=3)
    assert_close(got[rows], oracle_rows(r, rows), "bf16")
    del got
    rp = workloads.rolling_drop_config(truncate_at_boundary=49152, q_scale=8.0)
    got_p, _, _ = run_prefill([rp])
    assert_close(got_p[rows], oracle_rows(rp, rows), "bf16")


def _repos_rows(r, seed):
    """Stratified rows plus rows around the repos boundary and deep into
    key version 1 (the second rotated key copy)."""
    rows = stratified_rows(r, 256, seed=seed)
    b = int(r.msg_start[r.repos_after[0] + 1])  # first row of version 1
    extra = [b - 3, b - 1, b, b + 1, b + 127, b + 128, b + 200, b + 1000, r.T - 1]
    return np.unique(np.concatenate([rows, [t for t in extra if 0 <= t < r.T]]))


@pytest.mark.parametrize("q_scale", [1.0, 8.0])
def test_prefill_repos_full_size(q_scale):
    """128k tokens with a repos at 96k: both key versions, stratified rows
    plus rows on both sides of the repos boundary; also with queries scaled
    by 8 (peaky scores), where the version-1 rows read the second rotated
    key copy."""
    r = workloads.repos_config(q_scale=q_scale)
    assert len(r.repos_after) >= 1
    got, plan, _ = run_prefill([r])
    assert plan.info["max_versions"] == 1 + len(r.repos_after)
    assert np.isfinite(got).all()
    rows = _repos_rows(r, seed=2)
    assert len(rows) >= 256
    b = int(r.msg_start[r.repos_after[0] + 1])
    assert (rows >= b).sum() >= 32 and (rows < b).sum() >= 32
    assert_close(got[rows], oracle_rows(r, rows), "bf16")


def _run_plan(plan, reqs, rows_of, dtype="bf16"):
    """Run a plan over the given per-request row ranges of the requests'
    Q/K/V; returns out [T, Hq, D] float32."""
    torch = _torch_mod()
    q = akv.to_device(np.concatenate([r.q[a:b] for r, (a, b) in zip(reqs, rows_of)]), dtype)
    k = akv.to_device(np.concatenate([r.k[a:b] for r, (a, b) in zip(reqs, rows_of)]), dtype)
    v = akv.to_device(np.concatenate([r.v[a:b] for r, (a, b) in zip(reqs, rows_of)]), dtype)
    out = torch.zeros_like(q)
    ws = plan.workspace()
    akv.akv_segment_attention_run(plan, q, k, v, out, ws)
    torch.cuda.synchronize()
    assert akv.akv_workspace_status(ws) == 0
    return out.float().cpu().numpy()


def _torch_mod():
    import torch
    return torch


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_shared_prefix_equals_unshared(dtype):
    """Requests sharing a 256-token first message, computed once: the sharers'
    remaining rows equal, bit for bit, the same rows of an unshared batch
    (same windows, same order), and match the oracle."""
    P = 256
    rs = workloads.shared_prefix_batch(4, 3, P, 7, 400, dtype=dtype)
    shp = akv.shape(4, 2, 64, dtype)
    ops = [r.ops() for r in rs]
    cu_u = np.concatenate([[0], np.cumsum([r.T for r in rs])])
    out_u = _run_plan(akv.Plan(shp, cu_u, ops), rs, [(0, r.T) for r in rs], dtype)
    lens = [rs[0].T] + [r.T - P for r in rs[1:]]
    cu_s = np.concatenate([[0], np.cumsum(lens)])
    plan_s = akv.Plan(shp, cu_s, ops, share=[(-1, 0)] + [(0, P)] * (len(rs) - 1))
    out_s = _run_plan(plan_s, rs, [(0, rs[0].T)] + [(P, r.T) for r in rs[1:]], dtype)
    for b in range(len(rs)):
        su = slice(cu_u[b] + (P if b else 0), cu_u[b + 1])
        ss = slice(cu_s[b], cu_s[b + 1])
        assert np.array_equal(out_s[ss], out_u[su]), b
    for b in (1, 2):
        ref = oracle_rows(rs[b])
        assert_close(out_s[cu_s[b]:cu_s[b + 1]], ref[P:], dtype)


def test_calls_do_not_wait_for_the_stream():
    """Host planning and the upload of its tables do not wait for earlier
    work on the stream: with about a second of GPU work queued ahead, the
    calls return at once, and their results are right once it has run."""
    import time

    import torch
    import oracle
    r = workloads.random_request(61, n_msgs=6, max_len=200, Hq=8, Hkv=2, dtype="bf16",
                                 p_drop=0.3, p_repos=0.3, min_len=20)
    shp = akv.shape(8, 2, 64, "bf16")
    ops, cu = [r.ops()], [0, r.T]
    q, k, v = (akv.to_device(x, "bf16") for x in (r.q, r.k, r.v))
    out = torch.zeros_like(q)
    ws = torch.empty(akv.akv_segment_attention_workspace(shp, cu, ops), dtype=torch.uint8,
                     device="cuda")
    idx = torch.full((r.T,), -1, dtype=torch.int32, device="cuda")
    pos = torch.full((r.T,), -1, dtype=torch.int32, device="cuda")
    cws = torch.empty(max(1, akv.akv_compact_workspace(r.ops(), r.T)), dtype=torch.uint8,
                      device="cuda")
    akv.akv_segment_attention(shp, cu, None, ops, q, k, v, out, ws)  # first use: set-up
    akv.akv_compact(r.ops(), r.T, -1, idx, pos, cws)
    torch.cuda.synchronize()
    out.zero_()
    idx.fill_(-1)
    torch.cuda._sleep(2_000_000_000)  # about a second of spinning on the stream
    t0 = time.perf_counter()
    akv.akv_segment_attention(shp, cu, None, ops, q, k, v, out, ws)
    n = akv.akv_compact(r.ops(), r.T, -1, idx, pos, cws)
    host_s = time.perf_counter() - t0
    torch.cuda.synchronize()
    assert host_s < 0.25, f"the calls waited {host_s:.3f} s for the stream"
    assert akv.akv_workspace_status(ws) == 0
    ref, _ = oracle.replay_attention(*r.ops(), r.q, r.k, r.v, "bf16", r.rope_base)
    assert_close(out.float().cpu().numpy(), ref, "bf16")
    ou, op = oracle.compact(*r.ops(), upto=-1)
    np.testing.assert_array_equal(idx[:n].cpu().numpy(), ou)
    np.testing.assert_array_equal(pos[:n].cpu().numpy(), op)


@pytest.mark.parametrize("which", ["q", "k"])
def test_prefill_reports_fp16_range(which):
    """A query (rotated in the attention kernel's load path) or a key (rotated
    by the pre-pass) beyond the fp16 range of the tensor-core operands sets
    status bit 2; the same request without it reports 0."""
    import copy
    torch = _torch_mod()
    r = workloads.random_request(90, n_msgs=3, max_len=100, Hq=8, Hkv=2, dtype="bf16",
                                 min_len=20)
    shp = akv.shape(8, 2, 64, "bf16")
    for big in (False, True):
        rr = copy.deepcopy(r)
        if big:
            arr = getattr(rr, which)
            arr[r.T // 2, 1, 3] = workloads.bf16_bits(np.array([1.0e5], np.float32))[0]
        plan = akv.Plan(shp, [0, rr.T], [rr.ops()])
        q, k, v = (akv.to_device(x, "bf16") for x in (rr.q, rr.k, rr.v))
        out = torch.zeros_like(q)
        ws = plan.workspace()
        akv.akv_segment_attention_run(plan, q, k, v, out, ws)
        torch.cuda.synchronize()
        assert akv.akv_workspace_status(ws) == (2 if big else 0), (which, big)
