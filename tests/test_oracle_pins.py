"""Pins for the fp64 oracle: checks against what the pages and mathematics fix.

Each test ties the oracle to something other than itself: torch's
scaled_dot_product_attention (a library routine), a dense visibility mask
written from set semantics, closed forms of the RoPE rotation, the worked
requests printed on the pages, and brute force over every op log on 8 tokens.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rope_complex(x, pos, base):
    """Rotary embedding as a complex multiplication: the pair (x_i, x_{i+D/2})
    is the complex number x_i + j x_{i+D/2}, multiplied by exp(j pos theta_i)."""
    D = x.shape[-1]
    h = D // 2
    z = x[..., :h] + 1j * x[..., h:]
    theta = np.power(float(base), -np.arange(0, D, 2, dtype=np.float64) / D)
    z = z * np.exp(1j * np.asarray(pos, dtype=np.float64)[..., None] * theta)
    return np.concatenate([z.real, z.imag], axis=-1)


def sdpa_fp64(qr, kr, v, mask):
    """torch SDPA in fp64 on CPU; qr [T,Hq,D], kr/v [S,Hkv,D], mask [T,S] bool."""
    Hq, Hkv = qr.shape[1], kr.shape[1]
    grp = Hq // Hkv
    q = torch.from_numpy(qr).permute(1, 0, 2)
    k = torch.from_numpy(kr).permute(1, 0, 2).repeat_interleave(grp, 0)
    vv = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(grp, 0)
    o = torch.nn.functional.scaled_dot_product_attention(q, k, vv, attn_mask=torch.from_numpy(mask))
    return o.permute(1, 0, 2).numpy()


def dense_visibility(msg_start, drop_after, drop_target):
    """visible[t, u] from sets: u <= t and u's message was not a drop target
    at any boundary before t's message."""
    ms = np.asarray(msg_start)
    T = int(ms[-1])
    msg_of = np.searchsorted(ms, np.arange(T), side="right") - 1
    vis = np.zeros((T, T), dtype=bool)
    for t in range(T):
        gone = {int(j) for a, j in zip(drop_after, drop_target) if a < msg_of[t]}
        for u in range(t + 1):
            vis[t, u] = msg_of[u] not in gone
    return vis


def small_request(seed, n_msgs=5, max_len=7, dtype="bf16", p_drop=0.3, p_repos=0.2, Hq=4, Hkv=2):
    return workloads.random_request(seed, n_msgs, max_len, Hq=Hq, Hkv=Hkv, D=64, dtype=dtype,
                                    p_drop=p_drop, p_repos=p_repos)


# -- closed forms ---------------------------------------------------------

def test_rope_matches_complex_form():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((5, 3, 64))
    pos = rng.integers(0, 200000, size=(5, 3))
    np.testing.assert_allclose(oracle.rope(x, pos, 10000.0), rope_complex(x, pos, 10000.0),
                               rtol=0, atol=1e-9)


def test_rotation_composition():
    """R(q - p) applied to a key already rotated at p equals R(q) k (section 3.3)."""
    rng = np.random.default_rng(1)
    k = rng.standard_normal((40, 2, 64))
    p = rng.integers(0, 100000, size=40)
    q = rng.integers(0, 100000, size=40)
    kp = oracle.rope(k, p[:, None], 10000.0)
    moved = oracle.rope(kp, (q - p)[:, None], 10000.0)
    np.testing.assert_allclose(moved, rope_complex(k, q[:, None], 10000.0), rtol=0, atol=1e-9)
    # the same through the repos entry point, values untouched
    k32 = kp.astype(np.float32)
    v32 = rng.standard_normal((40, 2, 64)).astype(np.float32)
    ko, vo = oracle.repos_rotate(k32, v32, np.arange(40), p, q, "f32", 10000.0)
    np.testing.assert_allclose(ko, rope_complex(k32.astype(np.float64), (q - p)[:, None], 10000.0),
                               rtol=0, atol=1e-9)
    assert np.array_equal(vo, v32.astype(np.float64))


def test_rotation_preserves_norm_and_dot_relativity():
    rng = np.random.default_rng(2)
    a, b = rng.standard_normal((2, 64))
    for p, q in [(0, 5), (1000, 1005), (77777, 77782)]:
        da = oracle.rope(a, p, 10000.0) @ oracle.rope(b, q, 10000.0)
        assert abs(da - oracle.rope(a, 0, 10000.0) @ oracle.rope(b, q - p, 10000.0)) < 1e-9
    assert abs(np.linalg.norm(oracle.rope(a, 12345, 10000.0)) - np.linalg.norm(a)) < 1e-12


# -- attention definitions ------------------------------------------------

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_empty_log_is_causal_attention(dtype):
    """No ops: every token sees all earlier tokens at positions 0..T-1."""
    r = workloads.random_request(11, 4, 20, Hq=8, Hkv=2, dtype=dtype, p_drop=0, p_repos=0,
                                 min_len=3)
    out, res = oracle.replay_attention(*r.ops(), r.q, r.k, r.v, dtype, r.rope_base)
    T = r.T
    pos = np.arange(T)
    qr = rope_complex(oracle.widen(r.q, dtype), pos[:, None], r.rope_base)
    kr = rope_complex(oracle.widen(r.k, dtype), pos[:, None], r.rope_base)
    ref = sdpa_fp64(qr, kr, oracle.widen(r.v, dtype), np.tril(np.ones((T, T), dtype=bool)))
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
    assert np.array_equal(res.tok_pos, pos)


@pytest.mark.parametrize("seed", range(6))
def test_drop_only_logs_match_dense_mask(seed):
    r = small_request(100 + seed, n_msgs=6, max_len=9, p_repos=0.0, p_drop=0.35)
    out, _ = oracle.replay_attention(*r.ops(), r.q, r.k, r.v, "bf16", r.rope_base)
    vis = dense_visibility(r.msg_start, r.drop_after, r.drop_target)
    pos = np.arange(r.T)
    qr = rope_complex(oracle.widen(r.q, "bf16"), pos[:, None], r.rope_base)
    kr = rope_complex(oracle.widen(r.k, "bf16"), pos[:, None], r.rope_base)
    ref = sdpa_fp64(qr, kr, oracle.widen(r.v, "bf16"), vis)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
    np.testing.assert_array_equal(oracle.visible_counts(*r.ops()), vis.sum(1))


def test_rope_relativity_under_position_shift():
    r = small_request(7, n_msgs=6, max_len=8, p_drop=0.3, p_repos=0.4)
    a, _ = oracle.replay_attention(*r.ops(), r.q, r.k, r.v, "bf16", r.rope_base)
    b, _ = oracle.replay_attention(*r.ops(), r.q, r.k, r.v, "bf16", r.rope_base, pos_offset=4321)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-10)


def test_repos_without_prior_drop_is_identity():
    r = small_request(8, n_msgs=5, max_len=8, p_drop=0.0, p_repos=0.0)
    with_repos = (r.msg_start, r.drop_after, r.drop_target, np.array([1, 3], dtype=np.int32))
    a, ra = oracle.replay_attention(*r.ops(), r.q, r.k, r.v, "bf16", r.rope_base)
    b, rb = oracle.replay_attention(*with_repos, r.q, r.k, r.v, "bf16", r.rope_base)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-13)
    assert np.array_equal(ra.tok_pos, rb.tok_pos)


def test_repos_changes_positions_after_drop():
    """Drop alone keeps the next position; repos resets it to the survivor count."""
    ms = np.array([0, 4, 7, 9], dtype=np.int32)
    drop_only = oracle.replay(ms, [1], [0], [])
    assert drop_only.next_pos == 9 and list(drop_only.active_p) == list(range(4, 9))
    with_repos = oracle.replay(ms, [1], [0], [1])
    assert list(with_repos.active_p) == [0, 1, 2, 3, 4]
    assert list(with_repos.tok_pos) == [0, 1, 2, 3, 4, 5, 6, 3, 4]
    assert with_repos.next_pos == 5


@pytest.mark.parametrize("seed", range(8))
def test_segment_batch_equals_sequential_replay(seed):
    """One-prefill restoration reproduces the multi-pass replay (section 4.2)."""
    r = small_request(200 + seed, n_msgs=7, max_len=9, p_drop=0.3, p_repos=0.3)
    a, res = oracle.replay_attention(*r.ops(), r.q, r.k, r.v, "bf16", r.rope_base)
    b, tab = oracle.segment_batch_attention(*r.ops(), r.q, r.k, r.v, "bf16", r.rope_base)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)
    np.testing.assert_array_equal(res.tok_seg, tab["seg"])
    np.testing.assert_array_equal(res.drop_seg, tab["drop_seg"])
    np.testing.assert_array_equal(res.tok_ver, tab["seg_ver"][tab["seg"]])
    np.testing.assert_array_equal(res.tok_pos, tab["pos"][res.tok_ver, np.arange(r.T)])


def test_decode_equals_last_prefill_row():
    r = small_request(9, n_msgs=6, max_len=9, p_drop=0.3, p_repos=0.3)
    T = r.T
    snap = {}

    def grab(t, p, au, ap):
        if t == T - 1:
            snap["u"], snap["p"], snap["pt"] = np.array(au), np.array(ap), p

    oracle.replay(*r.ops(), on_token=grab)
    out, _ = oracle.replay_attention(*r.ops(), r.q, r.k, r.v, "bf16", r.rope_base, rows=[T - 1])
    pool = oracle.rope(oracle.widen(r.k[snap["u"]], "bf16"), snap["p"][:, None], r.rope_base)
    n = len(snap["u"])
    q32 = oracle.widen(r.q[T - 1:T], "bf16").astype(np.float32)
    dec = oracle.decode_attention(q32, np.array([snap["pt"]]), pool.astype(np.float32),
                                  oracle.widen(r.v[snap["u"]], "bf16").astype(np.float32),
                                  np.array([0, n]), np.arange(n), "f32", r.rope_base)
    # pool keys were stored as f32, so compare at f32 rounding
    np.testing.assert_allclose(dec[0], out[0], rtol=0, atol=1e-5)


# -- the pages' worked requests -------------------------------------------

def test_figure6_worked_request():
    with open(os.path.join(GOLDEN, "fig6_worked_request.json")) as f:
        g = json.load(f)
    ms = np.array(g["msg_start"], dtype=np.int32)
    da = [int(a) for a, ts in g["drop"].items() for _ in ts]
    dt = [int(t) for _, ts in g["drop"].items() for t in ts]
    ra = g["reposition"]
    for b, exp in g["after_boundary"].items():
        u, p = oracle.compact(ms, da, dt, ra, upto=int(b))
        assert list(u) == exp["active"], b
        assert list(p) == exp["positions_before_repos"], b
    res = oracle.replay(ms, da, dt, ra)
    assert res.next_pos == g["next_position_at_end"]
    assert list(res.active_p) == g["final_positions"]
    # the tiny workload is this request plus eight decode appends
    tiny = workloads.tiny_config()
    res = oracle.replay(*tiny.ops())
    assert list(res.active_u) == g["with_8_decodes"]["active"]
    assert list(res.active_p) == g["with_8_decodes"]["positions"]


def test_readme_example_drop_then_repos():
    with open(os.path.join(GOLDEN, "readme_drop_message_example.json")) as f:
        g = json.load(f)
    ms = np.array(g["msg_start"], dtype=np.int32)
    da = [int(a) for a, ts in g["drop_message"].items() for _ in ts]
    dt = [int(t) for _, ts in g["drop_message"].items() for t in ts]
    res = oracle.replay(ms, da, dt, g["reposition"])
    assert list(res.active_u) == g["active"]
    assert list(res.active_p) == g["positions"]
    assert res.next_pos == g["next_position"]


@pytest.mark.parametrize("bad", [
    dict(da=[1], dt=[2], ra=[]),      # target later than its boundary
    dict(da=[5], dt=[0], ra=[]),      # boundary out of range
    dict(da=[0], dt=[-1], ra=[]),     # negative target
    dict(da=[], dt=[], ra=[3]),       # repos boundary out of range
])
def test_invalid_logs_rejected(bad):
    ms = np.array([0, 2, 4, 6], dtype=np.int32)
    with pytest.raises(oracle.OpLogError):
        oracle.replay(ms, bad["da"], bad["dt"], bad["ra"])


def test_redrop_and_double_repos_are_noops():
    ms = np.array([0, 3, 5, 8], dtype=np.int32)
    a = oracle.replay(ms, [1], [0], [2])
    b = oracle.replay(ms, [1, 2, 2], [0, 0, 1], [2, 2])
    c = oracle.replay(ms, [1, 2], [0, 1], [2])
    assert list(b.active_u) == list(c.active_u) and list(b.active_p) == list(c.active_p)
    assert list(a.active_u) != list(c.active_u)


# -- brute force over every op log on 8 tokens ---------------------------

def _compositions(n, kmax):
    for k in range(1, kmax + 1):
        for cuts in itertools.combinations(range(1, n), k - 1):
            b = (0,) + cuts + (n,)
            yield [b[i + 1] - b[i] for i in range(k)]


def _all_logs(n_msgs):
    """Every log: each message dropped at one boundary >= itself or never, and
    a repos on/off at each boundary."""
    choices = [list(range(j, n_msgs)) + [None] for j in range(n_msgs)]
    for drop_at in itertools.product(*choices):
        for rep in itertools.product([0, 1], repeat=n_msgs):
            da = [a for a in drop_at if a is not None]
            dt = [j for j, a in enumerate(drop_at) if a is not None]
            ra = [i for i in range(n_msgs) if rep[i]]
            yield da, dt, ra


def test_brute_force_integer_tables_8_tokens():
    """Every log on every split of 8 tokens into <= 4 messages: replay and the
    segment-batch formula agree on segments, drop segments and positions, and
    the visible-key counts match the dense set-semantics mask."""
    n_logs = 0
    for lens in _compositions(8, 4):
        ms = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        for da, dt, ra in _all_logs(len(lens)):
            res = oracle.replay(ms, da, dt, ra)
            tab = oracle.segment_tables(ms, da, dt, ra)
            assert np.array_equal(res.tok_seg, tab["seg"])
            assert np.array_equal(res.drop_seg, tab["drop_seg"])
            assert np.array_equal(res.tok_pos, tab["pos"][res.tok_ver, np.arange(8)])
            vis = dense_visibility(ms, da, dt)
            cnt = (np.arange(8)[None, :] <= np.arange(8)[:, None]) & \
                (tab["seg"][:, None] < tab["drop_seg"][None, :])
            assert np.array_equal(cnt, vis)
            n_logs += 1
    assert n_logs == 35 * 1920 + 21 * 192 + 7 * 24 + 4


def test_brute_force_attention_8_tokens():
    """Attention values for every log of one split per message count."""
    rng = np.random.default_rng(3)
    q = rng.standard_normal((8, 2, 64)).astype(np.float32) * 3
    k = rng.standard_normal((8, 1, 64)).astype(np.float32)
    v = rng.standard_normal((8, 1, 64)).astype(np.float32)
    for lens in ([8], [3, 5], [2, 3, 3], [2, 2, 2, 2]):
        ms = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        for da, dt, ra in _all_logs(len(lens)):
            a, _ = oracle.replay_attention(ms, da, dt, ra, q, k, v, "f32", 10000.0)
            b, _ = oracle.segment_batch_attention(ms, da, dt, ra, q, k, v, "f32", 10000.0)
            assert np.max(np.abs(a - b)) < 1e-12


# -- Figure 5: same surviving tokens, different histories -----------------

def _fig5_model(n_layers, seed=5):
    mw = workloads.model_workload(seed=seed, n_req=1, prefix=6, following=0, n_layers=n_layers,
                                  d_model=64, Hq=4, Hkv=2, D=16, d_ff=128)
    return mw


def test_figure5_three_histories_are_distinct():
    """Trajectories keeping B and C: (1) A,B,C then drop A; (2) A,B, drop A, then
    C; (3) B,C.  With two layers C's state differs in all three, and B's state
    is the same in (1) and (2) (conditioned on A) but not in (3).  One layer
    cannot separate (2) from (3): RoPE is relative and raw K/V are inputs."""
    rng = np.random.default_rng(55)
    nA, nB, nC, d = 5, 4, 6, 64
    xa, xb, xc = (workloads.bf16_bits(rng.standard_normal((n, d)).astype(np.float32))
                  for n in (nA, nB, nC))
    mw = _fig5_model(2)
    W = mw.weights
    args = dict(Hq=4, Hkv=2, D=16, base=10000.0, eps=1e-6)
    x3 = np.concatenate([xa, xb, xc])
    ms3 = np.array([0, nA, nA + nB, nA + nB + nC], dtype=np.int32)
    o1 = oracle.model_replay(W, x3, ms3, [2], [0], [], **args)
    o2 = oracle.model_replay(W, x3, ms3, [1], [0], [], **args)
    o3 = oracle.model_replay(W, np.concatenate([xb, xc]), np.array([0, nB, nB + nC], np.int32),
                             [], [], [], **args)
    c1, c2, c3 = o1[nA + nB:], o2[nA + nB:], o3[nB:]
    b1, b2, b3 = o1[nA:nA + nB], o2[nA:nA + nB], o3[:nB]
    tol = 1e-9
    for x, y in ((c1, c2), (c1, c3), (c2, c3)):
        assert np.max(np.abs(x - y)) > 100 * tol
    assert np.max(np.abs(b1 - b2)) < tol
    assert np.max(np.abs(b1 - b3)) > 100 * tol
    # single layer: (2) and (3) coincide for C
    W1 = W[:1]
    p2 = oracle.model_replay(W1, x3, ms3, [1], [0], [], **args)[nA + nB:]
    p3 = oracle.model_replay(W1, np.concatenate([xb, xc]), np.array([0, nB, nB + nC], np.int32),
                             [], [], [], **args)[nB:]
    assert np.max(np.abs(p2 - p3)) < 1e-9


def _plain_forward(W, x, Hq, Hkv, D, base, eps):
    """Whole-sequence causal decoder forward, no cache ops, positions 0..T-1,
    attention through torch SDPA."""
    h = oracle.widen(x, "bf16")
    T = h.shape[0]
    pos = np.arange(T)
    causal = np.tril(np.ones((T, T), dtype=bool))
    for w in W:
        w = {k: oracle.widen(v, "bf16") for k, v in w.items()}
        a = h / np.sqrt((h * h).mean(-1, keepdims=True) + eps)
        qn = (a @ w["wq"]).reshape(T, Hq, D)
        kn = (a @ w["wk"]).reshape(T, Hkv, D)
        vn = (a @ w["wv"]).reshape(T, Hkv, D)
        o = sdpa_fp64(rope_complex(qn, pos[:, None], base), rope_complex(kn, pos[:, None], base),
                      vn, causal)
        h = h + o.reshape(T, Hq * D) @ w["wo"]
        f = h / np.sqrt((h * h).mean(-1, keepdims=True) + eps)
        g = f @ w["wg"]
        h = h + ((g / (1 + np.exp(-g))) * (f @ w["wu"])) @ w["wd"]
    return h / np.sqrt((h * h).mean(-1, keepdims=True) + eps)


def test_model_replay_without_ops_is_plain_forward():
    mw = workloads.model_workload(seed=9, n_req=1, prefix=40, following=700, n_layers=2,
                                  d_model=64, Hq=4, Hkv=2, D=16, d_ff=96,
                                  asst_len=(10, 30), tool_len=(30, 90))
    ref = _plain_forward(mw.weights, mw.x, 4, 2, 16, 10000.0, 1e-6)
    out = oracle.model_replay(mw.weights, mw.x, mw.msg_start, [], [], [], 4, 2, 16, 10000.0, 1e-6)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-10)


def test_model_replay_one_layer_matches_single_layer_replay():
    """The attention inside the model equals the single-layer replay fed the
    layer's own projections (checks the model's cache handling with ops)."""
    mw = workloads.model_workload(seed=10, n_req=3, prefix=12, following=120, n_layers=1,
                                  d_model=64, Hq=4, Hkv=2, D=16, d_ff=96,
                                  asst_len=(5, 15), tool_len=(10, 30))
    da, dt, ra = mw.ops[2]
    _, att = oracle.model_replay(mw.weights, mw.x, mw.msg_start, da, dt, ra, 4, 2, 16, 10000.0,
                                 1e-6, capture_layers=True)
    w = {k: oracle.widen(v, "bf16") for k, v in mw.weights[0].items()}
    h = oracle.widen(mw.x, "bf16")
    a = oracle.rmsnorm(h, 1e-6)
    T = mw.T
    q = (a @ w["wq"]).reshape(T, 4, 16).astype(np.float32)
    k = (a @ w["wk"]).reshape(T, 2, 16).astype(np.float32)
    v = (a @ w["wv"]).reshape(T, 2, 16).astype(np.float32)
    ref, _ = oracle.replay_attention(mw.msg_start, da, dt, ra, q, k, v, "f32", 10000.0)
    np.testing.assert_allclose(att[0].reshape(T, 4, 16), ref, rtol=0, atol=1e-5)
