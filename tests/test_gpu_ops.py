"""Compaction, repos rotation, append and decode on the GPU against the oracle,
and the tiny fp32 workload end to end (prefill -> compact -> repos -> decode)."""
import numpy as np
import pytest

import kv_cache_drop_gb300 as akv
import oracle
import workloads
from _util import assert_close, oracle_rows, run_prefill

pytestmark = pytest.mark.gpu


def _torch():
    import torch
    return torch


def _compact(ops, T, upto):
    torch = _torch()
    idx = torch.full((max(T, 1),), -1, dtype=torch.int32, device="cuda")
    pos = torch.full((max(T, 1),), -1, dtype=torch.int32, device="cuda")
    ws = torch.empty(max(1, akv.akv_compact_workspace(ops, T)), dtype=torch.uint8, device="cuda")
    n = akv.akv_compact(ops, T, upto, idx, pos, ws)
    torch.cuda.synchronize()
    return idx[:n].cpu().numpy(), pos[:n].cpu().numpy()


@pytest.mark.parametrize("seed", range(8))
def test_compact_every_boundary_bit_exact(seed):
    r = workloads.random_request(70 + seed, n_msgs=10, max_len=3000 if seed < 2 else 40,
                                 p_drop=0.3, p_repos=0.3)
    for upto in list(range(r.n_msgs)) + [-1]:
        gi, gp = _compact(r.ops(), r.T, upto)
        ou, op = oracle.compact(*r.ops(), upto=upto)
        np.testing.assert_array_equal(gi, ou)
        np.testing.assert_array_equal(gp, op)


@pytest.mark.parametrize("runs", [255, 256, 257])
def test_compact_run_table_limit(runs):
    """Kept runs at the limit of what the compaction kernel's parameters
    carry (256) and one past it (the uploaded-table path): every other one
    of 2 * runs messages dropped, so each survivor run is one message."""
    n = 2 * runs
    lens = np.random.default_rng(runs).integers(1, 7, size=n)
    ms = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    drops = [(n - 1, j) for j in range(1, n, 2)]
    r = workloads.gen._trajectory("runs", 3, ms, ["m"] * n, drops, [], 4, 2, 64, "bf16")
    gi, gp = _compact(r.ops(), r.T, n - 1)
    ou, op = oracle.compact(*r.ops(), upto=n - 1)
    assert len(ou) == int(lens[0::2].sum())
    np.testing.assert_array_equal(gi, ou)
    np.testing.assert_array_equal(gp, op)


def test_compact_everything_dropped():
    """A boundary after which no token survives: zero entries, nothing
    written; the boundary before it still compacts."""
    ms = np.array([0, 5, 9, 16], dtype=np.int32)
    drops = [(2, 0), (2, 1), (2, 2)]
    r = workloads.gen._trajectory("gone", 4, ms, ["m"] * 3, drops, [], 4, 2, 64, "bf16")
    gi, gp = _compact(r.ops(), r.T, 2)
    assert len(gi) == 0 and len(gp) == 0
    gi, gp = _compact(r.ops(), r.T, 1)
    ou, op = oracle.compact(*r.ops(), upto=1)
    np.testing.assert_array_equal(gi, ou)
    np.testing.assert_array_equal(gp, op)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_repos_rotate(dtype):
    torch = _torch()
    rng = np.random.default_rng(5)
    S, r, Hkv = 5000, 3000, 8
    k = workloads.gen._normals(rng, (S, Hkv, 64), dtype)
    v = workloads.gen._normals(rng, (S, Hkv, 64), dtype)
    src = np.sort(rng.choice(S, size=r, replace=False)).astype(np.int32)
    pf = rng.integers(0, 131072, size=r).astype(np.int32)
    pt = np.arange(r, dtype=np.int32)
    shp = akv.shape(16, Hkv, 64, dtype)
    ko = torch.zeros((r, Hkv, 64), dtype=torch.bfloat16 if dtype == "bf16" else torch.float32,
                     device="cuda")
    vo = torch.zeros_like(ko)
    for pos_to in (akv.i32_device(pt), None):
        akv.akv_repos_rotate(shp, r, akv.i32_device(src), akv.i32_device(pf), pos_to,
                             akv.to_device(k, dtype), akv.to_device(v, dtype), ko, vo)
        torch.cuda.synchronize()
        rk, rv = oracle.repos_rotate(k, v, src, pf, pt, dtype, 10000.0)
        tol = 2 ** -8 * 4 if dtype == "bf16" else 1e-5
        assert np.max(np.abs(ko.float().cpu().numpy() - rk)) <= tol
        assert np.array_equal(vo.float().cpu().numpy(), rv)  # values copied bit for bit


def test_repos_compact_full_size():
    """128k trajectory: compact the survivors at the repos boundary and rotate
    every one of them to its new position 0..r-1."""
    torch = _torch()
    r = workloads.repos_config()
    b = int(r.repos_after[0])
    idx, pos = _compact(r.ops(), r.T, b)
    ou, op = oracle.compact(*r.ops(), upto=b)
    np.testing.assert_array_equal(idx, ou)
    np.testing.assert_array_equal(pos, op)
    n = len(idx)
    shp = akv.shape(64, 8, 64, "bf16")
    ko = torch.empty((n, 8, 64), dtype=torch.bfloat16, device="cuda")
    vo = torch.empty_like(ko)
    akv.akv_repos_rotate(shp, n, akv.i32_device(idx), akv.i32_device(pos), None,
                         akv.to_device(r.k, "bf16"), akv.to_device(r.v, "bf16"), ko, vo)
    torch.cuda.synchronize()
    rk, rv = oracle.repos_rotate(r.k, r.v, ou, op, np.arange(n), "bf16", 10000.0)
    assert np.max(np.abs(ko.float().cpu().numpy() - rk)) <= 2 ** -8 * 4
    assert np.array_equal(vo.float().cpu().numpy(), rv)


def _repos_boundary(r, upto, dtype, shp):
    torch = _torch()
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    ko = torch.full((max(r.T, 1), shp.Hkv, 64), 7.0, dtype=tdt, device="cuda")
    vo = torch.full_like(ko, 7.0)
    ws = torch.empty(max(1, akv.akv_repos_boundary_workspace(r.ops(), r.T)), dtype=torch.uint8,
                     device="cuda")
    n = akv.akv_repos_boundary(shp, r.ops(), r.T, upto, akv.to_device(r.k, dtype),
                               akv.to_device(r.v, dtype), ko, vo, ws)
    torch.cuda.synchronize()
    tail = ko[n:].float().cpu().numpy()
    assert np.all(tail == 7.0) and np.all(vo[n:].float().cpu().numpy() == 7.0)  # rows >= n untouched
    return ko[:n].float().cpu().numpy(), vo[:n].float().cpu().numpy()


@pytest.mark.parametrize("seed", range(4))
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_repos_boundary_every_boundary(seed, dtype):
    """One-pass repos at every boundary of random logs with several repos:
    same survivors, positions and rotation as compaction then repos."""
    r = workloads.random_request(90 + seed, n_msgs=12, max_len=2000 if seed < 2 else 60,
                                 p_drop=0.3, p_repos=0.4, dtype=dtype)
    shp = akv.shape(r.Hq, r.Hkv, 64, dtype)
    tol = 2 ** -8 * 4 if dtype == "bf16" else 1e-5
    for upto in list(range(r.n_msgs)) + [-1]:
        gk, gv = _repos_boundary(r, upto, dtype, shp)
        ou, op = oracle.compact(*r.ops(), upto=upto)
        rk, rv = oracle.repos_rotate(r.k, r.v, ou, op, np.arange(len(ou)), dtype, 10000.0)
        assert gk.shape == rk.shape
        if len(ou):
            assert np.max(np.abs(gk - rk)) <= tol
            assert np.array_equal(gv, rv)


@pytest.mark.parametrize("n", [600, 700])
def test_repos_boundary_many_runs(n):
    """n short messages, every other one dropped at the last boundary: n/2
    separate kept runs, more than the repos kernel's parameters carry, so the
    run tables are uploaded (600: as a copy kernel's parameters, 700: through
    pinned host memory); compaction's tables take the same two paths."""
    lens = np.random.default_rng(5).integers(1, 5, size=n)
    ms = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    drops = [(n - 1, j) for j in range(1, n, 2)]
    r = workloads.gen._trajectory("runs", 97, ms, ["m"] * n, drops, [], 4, 2, 64, "bf16")
    gk, gv = _repos_boundary(r, n - 1, "bf16", akv.shape(4, 2, 64, "bf16"))
    ou, op = oracle.compact(*r.ops(), upto=n - 1)
    rk, rv = oracle.repos_rotate(r.k, r.v, ou, op, np.arange(len(ou)), "bf16", 10000.0)
    assert gk.shape == rk.shape and len(ou) > 0
    assert np.max(np.abs(gk - rk)) <= 2 ** -8 * 4
    assert np.array_equal(gv, rv)
    gi, gp = _compact(r.ops(), r.T, n - 1)
    np.testing.assert_array_equal(gi, ou)
    np.testing.assert_array_equal(gp, op)


def test_repos_boundary_full_size():
    """128k trajectory, one-pass repos at its repos boundary."""
    r = workloads.repos_config()
    b = int(r.repos_after[0])
    gk, gv = _repos_boundary(r, b, "bf16", akv.shape(64, 8, 64, "bf16"))
    ou, op = oracle.compact(*r.ops(), upto=b)
    rk, rv = oracle.repos_rotate(r.k, r.v, ou, op, np.arange(len(ou)), "bf16", 10000.0)
    assert np.max(np.abs(gk - rk)) <= 2 ** -8 * 4
    assert np.array_equal(gv, rv)


def _decode_oracle(dw, step, q_step):
    """Oracle decode at `step`: active pool keys as stored, appended keys
    rotated by the oracle itself at their positions."""
    out = []
    for b in range(dw.B):
        ka = oracle.widen(dw.k_pool[dw.active_slots[b]], dw.dtype)
        va = oracle.widen(dw.v_pool[dw.active_slots[b]], dw.dtype)
        pos = dw.L[b] + np.arange(step + 1)
        kn = oracle.rope(oracle.widen(dw.k_new[:step + 1, b], dw.dtype), pos[:, None],
                         dw.rope_base)
        vn = oracle.widen(dw.v_new[:step + 1, b], dw.dtype)
        K = np.concatenate([ka, kn])
        V = np.concatenate([va, vn])
        o = oracle.decode_attention(q_step[b:b + 1], np.array([dw.L[b] + step]), K, V,
                                    np.array([0, len(K)]), np.arange(len(K)), "f64", dw.rope_base)
        out.append(o[0])
    return np.stack(out)


def _run_decode(dw, check_steps):
    torch = _torch()
    shp = akv.shape(dw.Hq, dw.Hkv, 64, dw.dtype)
    kp = akv.to_device(dw.k_pool, dw.dtype)
    vp = akv.to_device(dw.v_pool, dw.dtype)
    max_kv = max(len(a) for a in dw.active_slots) + dw.steps
    ws = torch.empty(max(1, akv.akv_decode_workspace(shp, dw.B, max_kv)), dtype=torch.uint8,
                     device="cuda")
    results = {}
    for step in range(dw.steps):
        pos = akv.i32_device(dw.L + step)
        akv.akv_append_kv(shp, dw.B, akv.to_device(dw.k_new[step], dw.dtype),
                          akv.to_device(dw.v_new[step], dw.dtype), pos,
                          akv.i32_device(dw.append_slots[step]), kp, vp)
        indptr, idx = dw.indices_at(step)
        q = akv.to_device(dw.q[step], dw.dtype)
        out = torch.empty_like(q)
        akv.akv_decode_attention(shp, dw.B, q, pos, kp, vp, akv.i32_device(indptr),
                                 akv.i32_device(idx), max_kv, out, ws)
        if step in check_steps:
            torch.cuda.synchronize()
            results[step] = out.float().cpu().numpy()
    return results


def _run_decode_fused(dw, check_steps):
    """The same steps through akv_decode_attention_append (append fused)."""
    torch = _torch()
    shp = akv.shape(dw.Hq, dw.Hkv, 64, dw.dtype)
    kp = akv.to_device(dw.k_pool, dw.dtype)
    vp = akv.to_device(dw.v_pool, dw.dtype)
    max_kv = max(len(a) for a in dw.active_slots) + dw.steps
    ws = torch.empty(akv.akv_decode_workspace(shp, dw.B, max_kv), dtype=torch.uint8,
                     device="cuda")
    results = {}
    for step in range(dw.steps):
        indptr, idx = dw.indices_at(step)
        q = akv.to_device(dw.q[step], dw.dtype)
        out = torch.empty_like(q)
        akv.akv_decode_attention_append(
            shp, dw.B, q, akv.i32_device(dw.L + step), akv.to_device(dw.k_new[step], dw.dtype),
            akv.to_device(dw.v_new[step], dw.dtype), akv.i32_device(dw.append_slots[step]), kp,
            vp, akv.i32_device(indptr), akv.i32_device(idx), max_kv, out, ws)
        if step in check_steps:
            torch.cuda.synchronize()
            results[step] = out.float().cpu().numpy()
    torch.cuda.synchronize()
    return results, kp, vp


# (8, 1): the per-head kernel; (8, 2), (64, 8): the all-heads kernel
@pytest.mark.parametrize("dtype,Hq,Hkv", [("bf16", 8, 1), ("bf16", 8, 2), ("f32", 8, 2),
                                          ("bf16", 64, 8)])
def test_decode_fused_append_equals_separate_calls(dtype, Hq, Hkv):
    """Append fused into the decode launch: outputs and the pool bit-identical
    to akv_append_kv followed by akv_decode_attention, and close to fp64."""
    torch = _torch()
    dw = workloads.decode_workload(seed=14, B=3, active=(100, 5000), steps=3, Hq=Hq, Hkv=Hkv,
                                   dtype=dtype)
    sep = _run_decode(dw, {0, 1, 2})
    fused, kp, vp = _run_decode_fused(dw, {0, 1, 2})
    for step in (0, 1, 2):
        assert np.array_equal(fused[step], sep[step]), step
        assert_close(fused[step], _decode_oracle(dw, step, oracle.widen(dw.q[step], dtype)), dtype)
    # the appended rows equal akv_append_kv's, bit for bit
    shp = akv.shape(dw.Hq, dw.Hkv, 64, dtype)
    kp2 = akv.to_device(dw.k_pool, dtype)
    vp2 = akv.to_device(dw.v_pool, dtype)
    for step in range(dw.steps):
        akv.akv_append_kv(shp, dw.B, akv.to_device(dw.k_new[step], dtype),
                          akv.to_device(dw.v_new[step], dtype), akv.i32_device(dw.L + step),
                          akv.i32_device(dw.append_slots[step]), kp2, vp2)
    torch.cuda.synchronize()
    assert torch.equal(kp, kp2) and torch.equal(vp, vp2)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_decode_small(dtype):
    dw = workloads.decode_workload(seed=8, B=3, active=(100, 5000), steps=3, Hq=8, Hkv=2,
                                   dtype=dtype)
    res = _run_decode(dw, {0, 1, 2})
    for step, got in res.items():
        qf = oracle.widen(dw.q[step], dtype)
        assert_close(got, _decode_oracle(dw, step, qf), dtype)


def test_decode_peaky_and_empty_request():
    torch = _torch()
    dw = workloads.decode_workload(seed=9, B=2, active=(3000, 6000), steps=1, Hq=16, Hkv=2)
    dw.q[0] = workloads.bf16_bits(oracle.widen(dw.q[0], "bf16").astype(np.float32) * 8)
    res = _run_decode(dw, {0})
    assert_close(res[0], _decode_oracle(dw, 0, oracle.widen(dw.q[0], "bf16")), "bf16")
    # a request with no keys gets zeros
    shp = akv.shape(16, 2, 64, "bf16")
    q = akv.to_device(dw.q[0], "bf16")
    out = torch.full_like(q, 7.0)
    ws = torch.empty(akv.akv_decode_workspace(shp, 2, 10), dtype=torch.uint8, device="cuda")
    akv.akv_decode_attention(shp, 2, q, akv.i32_device([5, 5]), akv.to_device(dw.k_pool, "bf16"),
                             akv.to_device(dw.v_pool, "bf16"), akv.i32_device([0, 0, 0]),
                             akv.i32_device([0]), 10, out, ws)
    torch.cuda.synchronize()
    assert float(out.abs().max()) == 0.0


def test_decode_many_splits():
    """One request of 1.5M keys on a single KV head with 16 query heads: few
    CTAs, so the key chunk shrinks and the request is cut into ~730 splits,
    whose merge weights need more shared memory than the tile buffers."""
    dw = workloads.decode_workload(seed=15, B=1, active=(1_500_000, 1_500_000), steps=1,
                                   Hq=16, Hkv=1)
    res = _run_decode(dw, {0})
    assert_close(res[0], _decode_oracle(dw, 0, oracle.widen(dw.q[0], "bf16")), "bf16")


def test_decode_index_check():
    """The debug check of decode index data (reads only the index arrays):
    clean on a real workload; flags a slot outside the pool, a negative slot,
    a non-monotone index pointer, a request longer than max_kv, and an index
    pointer running past the entries given."""
    torch = _torch()
    dw = workloads.decode_workload(seed=16, B=3, active=(100, 2000), steps=1, Hq=8, Hkv=2)
    indptr, idx = dw.indices_at(0)
    S = int(dw.k_pool.shape[0])
    max_kv = int(np.max(np.diff(indptr)))

    def check(ip, ix, s_rows, mk):
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        akv.akv_decode_check_indices(len(ip) - 1, akv.i32_device(ip), akv.i32_device(ix), s_rows,
                                     mk, st)
        torch.cuda.synchronize()
        return int(st.item())

    assert check(indptr, idx, S, max_kv) == 0
    bad = np.array(idx, copy=True)
    bad[len(bad) // 2] = S  # one past the pool
    assert check(indptr, bad, S, max_kv) == 2
    bad = np.array(idx, copy=True)
    bad[0] = -1
    assert check(indptr, bad, S, max_kv) == 2
    ip = np.array(indptr, copy=True)
    ip[1], ip[2] = ip[2], ip[1]  # request 0 longer, request 1 negative
    assert check(ip, idx, S, max_kv) & 1
    assert check(indptr, idx, S, max_kv - 1) == 1  # a request longer than max_kv
    assert check(indptr, np.array(idx[:-5]), S, max_kv) == 1  # indptr[B] past the entries


def test_decode_full_size_steps():
    """14 requests, 20k-90k active keys each, 256 decode steps with appends;
    steps 0, 1 and 255 checked in full."""
    dw = workloads.decode_workload()
    res = _run_decode(dw, {0, 1, dw.steps - 1})
    for step, got in res.items():
        assert_close(got, _decode_oracle(dw, step, oracle.widen(dw.q[step], "bf16")), "bf16")


def _rope_positions(dw, seed=11):
    """Positions of the active entries when the pool holds raw keys: request
    b's survivors sit at a sorted random subset of 0..L_b-1."""
    rng = np.random.default_rng(seed)
    return [np.sort(rng.choice(int(dw.L[b]), size=len(dw.active_slots[b]), replace=False))
            .astype(np.int32) for b in range(dw.B)]


def _decode_rope_oracle(dw, step, pos_act, q_step, renumber=False):
    """fp64 decode at `step` over raw keys rotated at their positions; with
    `renumber` every entry of request b is at its list index (a repos) and the
    query follows them."""
    out = []
    for b in range(dw.B):
        ka = oracle.widen(dw.k_pool[dw.active_slots[b]], dw.dtype)
        kn = oracle.widen(dw.k_new[:step + 1, b], dw.dtype)
        K = np.concatenate([ka, kn])
        V = np.concatenate([oracle.widen(dw.v_pool[dw.active_slots[b]], dw.dtype),
                            oracle.widen(dw.v_new[:step + 1, b], dw.dtype)])
        if renumber:
            pos = np.arange(len(K))
        else:
            pos = np.concatenate([pos_act[b], dw.L[b] + np.arange(step + 1)])
        Kr = oracle.rope(K, pos[:, None], dw.rope_base)
        o = oracle.decode_attention(q_step[b:b + 1], np.array([pos[-1]]), Kr, V,
                                    np.array([0, len(K)]), np.arange(len(K)), "f64", dw.rope_base)
        out.append(o[0])
    return np.stack(out)


def _run_decode_rope(dw, check_steps, pos_act, renumber_from=None):
    """Rotate-on-read decode with the append fused; from step `renumber_from`
    on, every request's entries are renumbered 0..n-1 (a repos done by
    rewriting positions only)."""
    torch = _torch()
    shp = akv.shape(dw.Hq, dw.Hkv, 64, dw.dtype)
    kp = akv.to_device(dw.k_pool, dw.dtype)
    vp = akv.to_device(dw.v_pool, dw.dtype)
    max_kv = max(len(a) for a in dw.active_slots) + dw.steps
    ws = torch.empty(max(1, akv.akv_decode_rope_workspace(shp, dw.B, max_kv)), dtype=torch.uint8,
                     device="cuda")
    results = {}
    for step in range(dw.steps):
        indptr, idx = dw.indices_at(step)
        ren = renumber_from is not None and step >= renumber_from
        kvpos, qpos = [], []
        for b in range(dw.B):
            n = int(indptr[b + 1] - indptr[b])
            p = (np.arange(n) if ren else
                 np.concatenate([pos_act[b], dw.L[b] + np.arange(step + 1)]))
            kvpos.append(p)
            qpos.append(p[-1])
        q = akv.to_device(dw.q[step], dw.dtype)
        out = torch.empty_like(q)
        akv.akv_decode_attention_rope(
            shp, dw.B, q, akv.i32_device(np.array(qpos)), akv.to_device(dw.k_new[step], dw.dtype),
            akv.to_device(dw.v_new[step], dw.dtype), akv.i32_device(dw.append_slots[step]), kp, vp,
            akv.i32_device(indptr), akv.i32_device(idx), akv.i32_device(np.concatenate(kvpos)),
            max_kv, out, ws)
        if step in check_steps:
            torch.cuda.synchronize()
            results[step] = out.float().cpu().numpy()
    torch.cuda.synchronize()
    return results, kp, vp


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_decode_rope_small(dtype):
    """Raw-key pool, positions per entry, append fused: three steps against
    fp64, and the appended raw rows land in the pool."""
    dw = workloads.decode_workload(seed=8, B=3, active=(100, 5000), steps=3, Hq=8, Hkv=2,
                                   dtype=dtype)
    pos = _rope_positions(dw)
    res, kp, vp = _run_decode_rope(dw, {0, 1, 2}, pos)
    for step, got in res.items():
        assert_close(got, _decode_rope_oracle(dw, step, pos, oracle.widen(dw.q[step], dtype)),
                     dtype)
    torch = _torch()
    sl = torch.from_numpy(dw.append_slots.reshape(-1).astype(np.int64)).cuda()
    for pool, new in ((kp, dw.k_new), (vp, dw.v_new)):
        got = pool[sl]
        got = got.view(torch.int16).cpu().numpy().view(np.uint16) if dtype == "bf16" else \
            got.cpu().numpy()
        assert np.array_equal(got, new.reshape(-1, dw.Hkv, 64))  # raw rows, bit for bit


def test_decode_rope_sparse_and_large_positions():
    """Keys whose angles the kernel cannot take from its tile's first
    position (gaps of 64 positions or more within a 16-key tile), and
    positions past 2^18 (the double-precision angle path): request 0 at a
    sparse random subset of 0..2e6, request 1 in runs of 10 positions 100
    apart, request 2 dense, starting at 300,000."""
    dw = workloads.decode_workload(seed=21, B=3, active=(300, 3000), steps=2, Hq=8, Hkv=2)
    rng = np.random.default_rng(22)
    n = [len(a) for a in dw.active_slots]
    runs = (100 * np.arange((n[1] + 9) // 10)[:, None] + np.arange(10)[None, :]).reshape(-1)
    pos = [np.sort(rng.choice(2_000_000, size=n[0], replace=False)).astype(np.int32),
           runs[:n[1]].astype(np.int32),
           (300_000 + np.arange(n[2])).astype(np.int32)]
    res, _, _ = _run_decode_rope(dw, {0, 1}, pos)
    for step, got in res.items():
        assert_close(got, _decode_rope_oracle(dw, step, pos, oracle.widen(dw.q[step], "bf16")),
                     "bf16")


def test_decode_rope_repos_by_positions():
    """A repos mid-decode done by rewriting positions only (entries renumbered
    0..n-1, keys untouched): matches fp64 with the keys rotated at the new
    positions, before and after."""
    dw = workloads.decode_workload(seed=12, B=4, active=(500, 6000), steps=4, Hq=16, Hkv=4)
    dw.q[3] = workloads.bf16_bits(oracle.widen(dw.q[3], "bf16").astype(np.float32) * 8)  # peaky
    pos = _rope_positions(dw, seed=13)
    res, _, _ = _run_decode_rope(dw, {1, 2, 3}, pos, renumber_from=2)
    assert_close(res[1], _decode_rope_oracle(dw, 1, pos, oracle.widen(dw.q[1], "bf16")), "bf16")
    for step in (2, 3):
        ref = _decode_rope_oracle(dw, step, pos, oracle.widen(dw.q[step], "bf16"), renumber=True)
        assert_close(res[step], ref, "bf16")


def test_decode_rope_many_splits():
    """One request of a million raw keys behind a single KV head with 16
    query heads: about a thousand key chunks, so the merge of the splits
    runs in several passes of a few query heads each; the positions pass
    2^18 (the double-precision angle path)."""
    dw = workloads.decode_workload(seed=31, B=1, active=(1_000_000, 1_000_000), steps=1, Hq=16,
                                   Hkv=1)
    pos = _rope_positions(dw, seed=32)
    res, _, _ = _run_decode_rope(dw, {0}, pos)
    assert_close(res[0], _decode_rope_oracle(dw, 0, pos, oracle.widen(dw.q[0], "bf16")), "bf16")


@pytest.mark.parametrize("Hq,Hkv", [(32, 16), (24, 3)])
def test_decode_rope_other_kv_head_counts(Hq, Hkv):
    """16 KV heads (the all-heads kernel with 16 warps, half of them filling
    the angle table) and 3 (the per-head kernel)."""
    dw = workloads.decode_workload(seed=33, B=3, active=(200, 4000), steps=2, Hq=Hq, Hkv=Hkv)
    pos = _rope_positions(dw, seed=34)
    res, _, _ = _run_decode_rope(dw, {0, 1}, pos)
    for step, got in res.items():
        assert_close(got, _decode_rope_oracle(dw, step, pos, oracle.widen(dw.q[step], "bf16")),
                     "bf16")


@pytest.mark.parametrize("rope", [True, False])
@pytest.mark.parametrize("Hq,Hkv", [(64, 8), (128, 8), (16, 4), (16, 2), (32, 16)])
def test_decode_edges_all_heads_kernel(Hq, Hkv, rope):
    """2, 4, 8 or 16 KV heads (one CTA per key chunk takes all KV heads -- with
    rotation on read, for 4, 8 and 16 -- and the chunk partials are merged by
    a dependent launch; the other case runs the per-head kernel), with
    rotation on read or over a pre-rotated pool: requests with no entry, one entry, 15/16/17
    entries (tile edges), many short requests, two long ones cut into many
    chunks, positions past 2^18 and a negative one, peaky scores for every
    fourth request; no fused append; two calls in a row on one workspace."""
    torch = _torch()
    rng = np.random.default_rng(41)
    lens = [0, 1, 15, 16, 17, 0, 5000, 3, 2, 1, 0, 33, 64, 9000, 0, 7] + \
        [int(x) for x in rng.integers(0, 40, size=60)]
    B, S = len(lens), 20000
    shp = akv.shape(Hq, Hkv, 64, "bf16")
    kpool = workloads.bf16_bits(rng.standard_normal((S, Hkv, 64)).astype(np.float32))
    vpool = workloads.bf16_bits(rng.standard_normal((S, Hkv, 64)).astype(np.float32))
    qf = rng.standard_normal((B, Hq, 64)).astype(np.float32)
    qf[1::4] *= 8  # peaky scores (std ~ 8) for every fourth request
    q = workloads.bf16_bits(qf)
    indptr = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    idx = rng.integers(0, S, size=int(indptr[-1])).astype(np.int32)
    pos, qpos = [], []
    for b, n in enumerate(lens):
        base = [0, 300_000, 3_000_000][b % 3]
        p = base + np.sort(rng.choice(4 * n + 8, size=n, replace=False))
        if b == 6:
            p[0] = -5
        pos.append(p.astype(np.int32))
        qpos.append(int(p[-1]) + 1 if n else base)
    kvpos = np.concatenate(pos).astype(np.int32)
    max_kv = max(lens)
    out = torch.full((B, Hq, 64), 7.0, dtype=torch.bfloat16, device="cuda")
    wsb = (akv.akv_decode_rope_workspace if rope else akv.akv_decode_workspace)(shp, B, max_kv)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    kp, vp = akv.to_device(kpool, "bf16"), akv.to_device(vpool, "bf16")
    ref = np.zeros((B, Hq, 64))
    for b, n in enumerate(lens):
        if n == 0:
            continue
        sl = idx[indptr[b]:indptr[b + 1]]
        kk = oracle.widen(kpool[sl], "bf16")
        if rope:  # the pool holds raw keys, rotated at their entries' positions
            kk = oracle.rope(kk, pos[b][:, None], 10000.0)
        ref[b] = oracle.decode_attention(oracle.widen(q[b:b + 1], "bf16"),
                                         np.array([qpos[b]]), kk,
                                         oracle.widen(vpool[sl], "bf16"),
                                         np.array([0, n]), np.arange(n), "f64", 10000.0)[0]
    for _ in range(2):  # the workspace is reused as it stands
        args = (shp, B, akv.to_device(q, "bf16"), akv.i32_device(qpos))
        if rope:
            akv.akv_decode_attention_rope(*args, None, None, None, kp, vp, akv.i32_device(indptr),
                                          akv.i32_device(idx), akv.i32_device(kvpos), max_kv,
                                          out, ws)
        else:
            akv.akv_decode_attention(*args, kp, vp, akv.i32_device(indptr), akv.i32_device(idx),
                                     max_kv, out, ws)
        torch.cuda.synchronize()
        got = out.float().cpu().numpy()
        assert_close(got, ref, "bf16")
        assert not np.any(got[np.array(lens) == 0])  # no entries: zeros


@pytest.mark.parametrize("rope", [False, True])
def test_decode_steps_in_a_cuda_graph(rope):
    """A serving step (decode with the append fused, GQA 64/8: the all-heads
    kernel and its dependent merge launch) captured once in a CUDA graph and
    replayed for three steps, each step's inputs copied into the captured
    buffers first: outputs and pools equal the same steps called eagerly,
    bit for bit."""
    torch = _torch()
    dw = workloads.decode_workload(seed=51, B=4, active=(2000, 9000), steps=3, Hq=64, Hkv=8)
    shp = akv.shape(dw.Hq, dw.Hkv, 64, "bf16")
    max_kv = max(len(a) for a in dw.active_slots) + dw.steps
    pos_act = _rope_positions(dw, seed=52)
    wsb = (akv.akv_decode_rope_workspace if rope else akv.akv_decode_workspace)(shp, dw.B, max_kv)

    def inputs(step):
        indptr, idx = dw.indices_at(step)
        kvpos = np.concatenate([np.concatenate([pos_act[b], dw.L[b] + np.arange(step + 1)])
                                for b in range(dw.B)]).astype(np.int32)
        qpos = dw.L + step
        return dict(q=akv.to_device(dw.q[step], "bf16"), pos=akv.i32_device(qpos),
                    kn=akv.to_device(dw.k_new[step], "bf16"),
                    vn=akv.to_device(dw.v_new[step], "bf16"),
                    slots=akv.i32_device(dw.append_slots[step]), indptr=akv.i32_device(indptr),
                    idx=akv.i32_device(idx), kvpos=akv.i32_device(kvpos))

    def step_call(t, kp, vp, out, ws):
        if rope:
            akv.akv_decode_attention_rope(shp, dw.B, t["q"], t["pos"], t["kn"], t["vn"],
                                          t["slots"], kp, vp, t["indptr"], t["idx"], t["kvpos"],
                                          max_kv, out, ws)
        else:
            akv.akv_decode_attention_append(shp, dw.B, t["q"], t["pos"], t["kn"], t["vn"],
                                            t["slots"], kp, vp, t["indptr"], t["idx"], max_kv,
                                            out, ws)

    # eager
    kp_e, vp_e = akv.to_device(dw.k_pool, "bf16"), akv.to_device(dw.v_pool, "bf16")
    ws_e = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    eager = []
    for step in range(dw.steps):
        out = torch.empty((dw.B, dw.Hq, 64), dtype=torch.bfloat16, device="cuda")
        step_call(inputs(step), kp_e, vp_e, out, ws_e)
        eager.append(out)
    # captured: buffers sized for the last step (the index lists grow by one
    # entry per request and step; the grid depends only on max_kv)
    kp_g, vp_g = akv.to_device(dw.k_pool, "bf16"), akv.to_device(dw.v_pool, "bf16")
    ws_g = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    last = inputs(dw.steps - 1)
    buf = {k: torch.zeros_like(v) for k, v in last.items()}
    out_g = torch.empty((dw.B, dw.Hq, 64), dtype=torch.bfloat16, device="cuda")

    def load(step):
        for k, v in inputs(step).items():
            buf[k][:v.numel()].copy_(v)

    load(0)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm-up outside the capture
        step_call(buf, kp_g, vp_g, out_g, ws_g)
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step_call(buf, kp_g, vp_g, out_g, ws_g)
    for step in range(dw.steps):
        load(step)
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out_g, eager[step]), f"step {step}"
    assert torch.equal(kp_g, kp_e) and torch.equal(vp_g, vp_e)


def test_decode_rope_full_size():
    """14 requests, 20k-90k keys, GQA 64/8 (one CTA reads whole pool rows):
    256 steps with the append fused; steps 0 and 255 checked in full."""
    dw = workloads.decode_workload()
    pos = _rope_positions(dw)
    res, _, _ = _run_decode_rope(dw, {0, dw.steps - 1}, pos)
    for step, got in res.items():
        assert_close(got, _decode_rope_oracle(dw, step, pos, oracle.widen(dw.q[step], "bf16")),
                     "bf16")


def test_tiny_fp32_end_to_end():
    """User 16 / assistant 24 / tool 32 with drop {1:[0], 2:[1]}, reposition
    [2], then 8 decode appends: attention outputs, the active-index list and
    the post-repos keys."""
    torch = _torch()
    r = workloads.tiny_config()
    shp = akv.shape(2, 2, 64, "f32")
    Tp = r.T_prefill
    got, plan, _ = run_prefill([r])
    ref_all, _ = oracle.replay_attention(*r.ops(), r.q, r.k, r.v, "f32", r.rope_base)
    assert_close(got, ref_all[:Tp], "f32")
    # keys of the prefill go to a pool at their append positions
    kp = torch.zeros((256, 2, 64), dtype=torch.float32, device="cuda")
    vp = torch.zeros_like(kp)
    tpos = plan.tables()["tok_pos"]
    akv.akv_append_kv(shp, Tp, akv.to_device(r.k[:Tp], "f32"), akv.to_device(r.v[:Tp], "f32"),
                      akv.i32_device(tpos), akv.i32_device(np.arange(Tp)), kp, vp)
    # compact at the boundary after message 2 and re-position the survivors
    ops3 = (r.msg_start[:4], r.drop_after, r.drop_target, r.repos_after)
    idx, pos = _compact(ops3, Tp, 2)
    np.testing.assert_array_equal(idx, np.arange(40, 72))
    np.testing.assert_array_equal(pos, np.arange(40, 72))
    n = len(idx)
    base = 100  # the compacted cache lives at pool slots 100..
    akv.akv_repos_rotate(shp, n, akv.i32_device(idx), akv.i32_device(pos), None, kp, vp,
                         kp[base:base + n], vp[base:base + n])
    torch.cuda.synchronize()
    ref_k = oracle.rope(oracle.widen(r.k[idx], "f32"), np.arange(n)[:, None], r.rope_base)
    assert np.max(np.abs(kp[base:base + n].cpu().numpy() - ref_k)) <= 1e-4
    # eight decode steps over the compacted cache
    ws = torch.empty(akv.akv_decode_workspace(shp, 1, 64), dtype=torch.uint8, device="cuda")
    for i in range(8):
        t = Tp + i
        p = n + i
        akv.akv_append_kv(shp, 1, akv.to_device(r.k[t:t + 1], "f32"),
                          akv.to_device(r.v[t:t + 1], "f32"), akv.i32_device([p]),
                          akv.i32_device([base + p]), kp, vp)
        out = torch.empty((1, 2, 64), dtype=torch.float32, device="cuda")
        akv.akv_decode_attention(shp, 1, akv.to_device(r.q[t:t + 1], "f32"), akv.i32_device([p]),
                                 kp, vp, akv.i32_device([0, p + 1]),
                                 akv.i32_device(base + np.arange(p + 1)), 64, out, ws)
        torch.cuda.synchronize()
        assert_close(out.cpu().numpy(), ref_all[t:t + 1], "f32")
    res = oracle.replay(*r.ops())
    np.testing.assert_array_equal(res.active_u, np.arange(40, 80))


def test_errors_are_reported_before_launch():
    torch = _torch()
    r = workloads.random_request(3, n_msgs=3, max_len=50, Hq=8, Hkv=2)
    plan = akv.Plan(akv.shape(8, 2, 64, "bf16"), [0, r.T], [r.ops()])
    q = akv.to_device(r.q, "bf16")
    k = akv.to_device(r.k, "bf16")
    v = akv.to_device(r.v, "bf16")
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(akv.AkvError) as e:
        akv.akv_segment_attention_run(plan, q, k, v, torch.empty_like(q), small)
    assert e.value.status == 3
    with pytest.raises(akv.AkvError) as e:
        akv.Plan(akv.shape(6, 2, 64, "bf16"), [0, r.T], [r.ops()]).__class__  # valid plan
        p2 = akv.Plan(akv.shape(6, 2, 64, "bf16"), [0, r.T], [r.ops()])
        akv.akv_segment_attention_run(p2, q, k, v, torch.empty_like(q), p2.workspace())
    assert e.value.status == 4  # odd query heads per KV head in bf16


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_append_rotation_across_position_ranges(dtype):
    """Positions on both sides of the fp32 angle-reduction range (|pos| <= 2^18)
    and far beyond it rotate like the fp64 oracle."""
    torch = _torch()
    pos = np.array([0, 1, 4095, 131071, 262143, 262144, 262145, 300000, 1 << 20, (1 << 24) + 3,
                    (1 << 30) + 7, 2**31 - 1], dtype=np.int64)
    n = len(pos)
    rng = np.random.default_rng(12)
    k = workloads.gen._normals(rng, (n, 4, 64), dtype)
    v = workloads.gen._normals(rng, (n, 4, 64), dtype)
    shp = akv.shape(8, 4, 64, dtype)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    kp = torch.zeros((n, 4, 64), dtype=tdt, device="cuda")
    vp = torch.zeros_like(kp)
    akv.akv_append_kv(shp, n, akv.to_device(k, dtype), akv.to_device(v, dtype),
                      akv.i32_device(pos), akv.i32_device(np.arange(n)[::-1].copy()), kp, vp)
    torch.cuda.synchronize()
    ref = oracle.rope(oracle.widen(k, dtype), pos[:, None], 10000.0)[::-1]
    tol = 2 ** -8 * 4 if dtype == "bf16" else 2e-5
    assert np.max(np.abs(kp.float().cpu().numpy() - ref)) <= tol
    assert np.array_equal(vp.float().cpu().numpy(), oracle.widen(v, dtype)[::-1])
