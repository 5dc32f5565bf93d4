"""Host-side checks of libakv (no GPU): exported symbols, the planner's
integer tables against the oracle, validation and injected faults."""
import os
import re
import subprocess
import sys

import numpy as np
import pytest

import oracle
import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def akv():
    import kv_cache_drop_gb300 as m
    from kv_cache_drop_gb300 import _build
    if not os.path.exists(m.LIB_PATH):
        _build.build()
    m.lib()
    return m


def test_every_declared_symbol_is_exported(akv):
    with open(os.path.join(ROOT, "include", "akv.h")) as f:
        src = f.read()
    declared = set(re.findall(r"\b(akv_[a-z0-9_]+)\s*\(", src))
    assert declared, "no declarations found"
    lib = akv.lib()
    for name in sorted(declared):
        assert hasattr(lib, name), name
    assert set(akv.EXPORTED) <= declared


def _plan_vs_oracle(akv, reqs):
    shp = akv.shape(reqs[0].Hq, reqs[0].Hkv, 64, reqs[0].dtype)
    cu = np.concatenate([[0], np.cumsum([r.T for r in reqs])])
    plan = akv.Plan(shp, cu, [r.ops() for r in reqs])
    tab = plan.tables()
    vis = 0
    for b, r in enumerate(reqs):
        res = oracle.replay(*r.ops())
        sl = slice(cu[b], cu[b + 1])
        np.testing.assert_array_equal(tab["tok_pos"][sl], res.tok_pos)
        np.testing.assert_array_equal(tab["tok_seg"][sl], res.tok_seg)
        np.testing.assert_array_equal(tab["tok_ver"][sl], res.tok_ver)
        np.testing.assert_array_equal(tab["drop_seg"][sl], np.minimum(res.drop_seg, 2**31 - 1))
        vis += int(oracle.visible_counts(*r.ops()).sum())
    assert plan.info["visible_pairs"] == vis
    assert plan.info["T"] == cu[-1]
    return plan


@pytest.mark.parametrize("seed", range(12))
def test_plan_tables_match_oracle(akv, seed):
    r = workloads.random_request(300 + seed, n_msgs=9, max_len=40, p_drop=0.3, p_repos=0.25)
    _plan_vs_oracle(akv, [r])


def test_plan_batch_of_ragged_requests(akv):
    reqs = [workloads.random_request(400 + i, n_msgs=3 + i, max_len=70, p_drop=0.3, p_repos=0.3)
            for i in range(5)]
    reqs.append(workloads.random_request(499, n_msgs=1, max_len=0))  # empty request
    _plan_vs_oracle(akv, reqs)


def test_plan_rolling_drop_trajectory(akv):
    ms, roles, drops, repos = workloads.agent_trajectory(2, rounds=30)
    r = workloads.Trajectory("t", 64, 8, 64, 10000.0, "bf16", ms, roles,
                             np.array([a for a, _ in drops], np.int32),
                             np.array([t for _, t in drops], np.int32), np.array(repos, np.int32),
                             None, None, None)
    plan = _plan_vs_oracle(akv, [r])
    # the permuted key order leaves few partially visible windows
    assert plan.info["n_full_windows"] > 0.5 * plan.info["n_windows"]


def test_plan_repos_trajectory(akv):
    ms, roles, drops, repos = workloads.agent_trajectory(3, total_tokens=40000,
                                                         repos_threshold=30000)
    assert len(repos) >= 1
    r = workloads.Trajectory("t", 64, 8, 64, 10000.0, "bf16", ms, roles,
                             np.array([a for a, _ in drops], np.int32),
                             np.array([t for _, t in drops], np.int32), np.array(repos, np.int32),
                             None, None, None)
    plan = _plan_vs_oracle(akv, [r])
    assert plan.info["max_versions"] == 1 + len(repos)


@pytest.mark.parametrize("da,dt,ra", [([1], [2], []), ([5], [0], []), ([0], [-1], []),
                                      ([], [], [3])])
def test_plan_rejects_invalid_logs(akv, da, dt, ra):
    ms = np.array([0, 2, 4, 6], dtype=np.int32)
    with pytest.raises(akv.AkvError) as e:
        akv.Plan(akv.shape(4, 2, 64, "bf16"), [0, 6], [(ms, da, dt, ra)])
    assert e.value.status == 1


def test_plan_rejects_row_count_mismatch_and_bad_shape(akv):
    ms = np.array([0, 2, 4], dtype=np.int32)
    with pytest.raises(akv.AkvError) as e:
        akv.Plan(akv.shape(4, 2, 64, "bf16"), [0, 5], [(ms, [], [], [])])
    assert e.value.status == 1
    with pytest.raises(akv.AkvError) as e:
        akv.Plan(akv.shape(4, 2, 128, "bf16"), [0, 4], [(ms, [], [], [])])
    assert e.value.status == 4
    with pytest.raises(akv.AkvError) as e:
        akv.Plan(akv.shape(6, 4, 64, "bf16"), [0, 4], [(ms, [], [], [])])
    assert e.value.status == 1
    with pytest.raises(akv.AkvError) as e:
        akv.Plan(akv.shape(4, 2, 64, "bf16"), [0, 4], [(ms, [], [], [])], logical_idx=[0, 1, 3, 2])
    assert e.value.status == 1


def test_injected_fault_reaches_python(akv):
    code = ("import sys; sys.path.insert(0, %r); import kv_cache_drop_gb300 as a, numpy as np\n"
            "try:\n"
            "    a.Plan(a.shape(4, 2, 64, 'bf16'), [0, 2], [(np.array([0, 2]), [], [], [])])\n"
            "except a.AkvError as e:\n"
            "    print('status', e.status)\n") % ROOT
    env = dict(os.environ, AKV_FAULT="cuda")
    out = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                         timeout=120)
    assert "status 2" in out.stdout, out.stderr


def test_workspace_queries_are_host_only(akv):
    r = workloads.random_request(5, n_msgs=5, max_len=300, p_drop=0.3, p_repos=0.3)
    shp = akv.shape(8, 2, 64, "bf16")
    ws = akv.akv_segment_attention_workspace(shp, [0, r.T], [r.ops()])
    plan = akv.Plan(shp, [0, r.T], [r.ops()])
    assert ws == plan.info["workspace_bytes"] > 0
    assert akv.akv_decode_workspace(shp, 14, 90000) > 0
    assert akv.akv_compact_workspace(r.ops(), r.T) > 0


@pytest.mark.parametrize("Hq,Hkv,B,max_kv", [(64, 8, 14, 90000), (16, 4, 3, 1), (8, 2, 1, 0),
                                            (128, 8, 65535, 2048), (64, 8, 2, 2_048_000)])
def test_decode_workspace_sizes(akv, Hq, Hkv, B, max_kv):
    """The decode workspaces as the header states them, on the host alone:
    split-KV partials ((m, l) pairs, then the rows' outputs: 66 floats per
    (request, query head, split)) over 1,024-key splits, or 512-key splits
    with rotation on read, each part rounded up to 256 bytes, then B x Hkv
    int32 merge counters (bf16); fp32 rotation on read has no counters."""
    r256 = lambda n: (n + 255) // 256 * 256

    def partials(chunk):
        ns = 1 if max_kv <= 0 else -(-max_kv // chunk)
        return r256(B * Hq * ns * 2 * 4) + r256(B * Hq * ns * 64 * 4)

    counters = r256(B * Hkv * 4)
    for dt in ("bf16", "f32"):
        shp = akv.shape(Hq, Hkv, 64, dt)
        assert akv.akv_decode_workspace(shp, B, max_kv) == partials(1024) + counters
    assert akv.akv_decode_rope_workspace(akv.shape(Hq, Hkv, 64, "bf16"), B, max_kv) == \
        partials(512) + counters
    assert akv.akv_decode_rope_workspace(akv.shape(Hq, Hkv, 64, "f32"), B, max_kv) == \
        partials(512)


INVALID, UNSUPPORTED = 1, 4


def _shared_batch(seed=3, n_req=3, prefix=256):
    rs = workloads.shared_prefix_batch(seed, n_req, prefix, 6, 300)
    return rs, [r.ops() for r in rs]


def test_shared_prefix_plan_tables_match_unshared(akv):
    """A sharer's stored rows carry exactly the tables its rows have in an
    unshared plan, and the visible-pair count drops by the prefix rows'."""
    rs, ops = _shared_batch()
    P = 256
    shp = akv.shape(4, 2, 64, "bf16")
    cu_u = np.concatenate([[0], np.cumsum([r.T for r in rs])])
    plan_u = akv.Plan(shp, cu_u, ops)
    lens = [rs[0].T] + [r.T - P for r in rs[1:]]
    cu_s = np.concatenate([[0], np.cumsum(lens)])
    share = [(-1, 0)] + [(0, P)] * (len(rs) - 1)
    plan_s = akv.Plan(shp, cu_s, ops, share=share)
    tu, ts = plan_u.tables(), plan_s.tables()
    for b in range(len(rs)):
        rows_u = np.arange(cu_u[b] + (P if b else 0), cu_u[b + 1])
        rows_s = np.arange(cu_s[b], cu_s[b + 1])
        for name in tu:
            np.testing.assert_array_equal(ts[name][rows_s], tu[name][rows_u], err_msg=name)
    # the skipped rows: prefix rows of the sharers, each sees its own prefix
    skipped = (len(rs) - 1) * P * (P + 1) // 2
    assert plan_s.info["visible_pairs"] == plan_u.info["visible_pairs"] - skipped
    assert plan_s.info["T"] == cu_s[-1]


def test_shared_prefix_plan_rejects_bad_sharing(akv):
    rs, ops = _shared_batch()
    shp = akv.shape(4, 2, 64, "bf16")
    P = 256

    def cu_for(lens):
        return np.concatenate([[0], np.cumsum(lens)])

    ok = [rs[0].T, rs[1].T - P, rs[2].T - P]
    cases = [
        ([(-1, 0), (0, 200), (-1, 0)], [rs[0].T, rs[1].T - 200, rs[2].T], UNSUPPORTED),
        ([(-1, 0), (2, P), (-1, 0)], ok[:2] + [rs[2].T], INVALID),  # later owner
        ([(-1, 0), (0, P), (1, P)], ok, INVALID),                     # owner shares
        ([(-1, 0), (0, P), (-1, 0)], [rs[0].T, rs[1].T, rs[2].T], INVALID),  # rows
        ([(-1, 0), (0, 384), (-1, 0)], [rs[0].T, rs[1].T - 384, rs[2].T], INVALID),
    ]
    for share, lens, code in cases:
        with pytest.raises(akv.AkvError) as e:
            akv.Plan(shp, cu_for(lens), ops, share=share)
        assert e.value.status == code, (share, e.value)
    # a drop of a prefix message
    bad = list(ops)
    ms, da, dt, ra = bad[1]
    bad[1] = (ms, np.append(da, 2).astype(np.int32), np.append(dt, 0).astype(np.int32), ra)
    with pytest.raises(akv.AkvError) as e:
        akv.Plan(shp, cu_for(ok), bad, share=[(-1, 0), (0, P), (0, P)])
    assert e.value.status == INVALID


def test_plan_rejects_key_rows_beyond_32_bit_coordinates(akv):
    """The attention kernel addresses rotated-key rows (version, KV head,
    slot) with one 32-bit TMA coordinate: 2 versions x 8 heads x 140M rows
    is refused before anything is allocated."""
    shp = akv.shape(8, 8, 64, "bf16")
    T = 140_000_000
    ms = np.array([0, T // 2, T], dtype=np.int32)
    ops = [(ms, np.zeros(0, np.int32), np.zeros(0, np.int32), np.array([0], np.int32))]
    with pytest.raises(akv.AkvError, match="UNSUPPORTED"):
        akv.Plan(shp, [0, T], ops)

