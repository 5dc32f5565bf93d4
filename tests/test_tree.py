"""Cache-history tree and drop-aware eviction (host library code, no GPU):
Figure 5's three histories, then random histories and operation sequences
against the reference model in oracle/tree.py (integers, bit-exact)."""
import numpy as np
import pytest

from oracle.tree import TreeModel


@pytest.fixture(scope="module")
def akv():
    import os
    import kv_cache_drop_gb300 as m
    from kv_cache_drop_gb300 import _build
    if not os.path.exists(m.LIB_PATH):
        _build.build()
    m.lib()
    return m


def _hist(msgs, drops=(), repos=()):
    """msgs: list of token-id lists; drops: (after, target); repos: boundaries."""
    ms = np.concatenate([[0], np.cumsum([len(m) for m in msgs])]).astype(np.int32)
    tok = np.concatenate([np.asarray(m, dtype=np.int32) for m in msgs]) if msgs else \
        np.zeros(0, np.int32)
    da = np.array([a for a, _ in drops], np.int32)
    dt = np.array([t for _, t in drops], np.int32)
    ra = np.array(sorted(repos), np.int32)
    return (ms, da, dt, ra), tok


A, B, C = [1, 2, 3], [4, 5], [6, 7, 8, 9]


def test_figure5_histories_branch(akv):
    """Figure 5: (1) A, B, C then drop A; (2) A, B, drop A, then C; (3) B, C.
    (1) and (2) share A and B; C differs in all three; B of (3) is a
    separate branch."""
    h1 = _hist([A, B, C], drops=[(2, 0)])
    h2 = _hist([A, B, C], drops=[(1, 0)])
    h3 = _hist([B, C])
    t = akv.Tree()
    t.insert(*h1, 1)
    # (2) after (1): A and B are there, the drop of A after B is not
    m = t.match(*h2)
    assert m["matched_msgs"] == 2 and m["kind"] == "prefill_suffix"
    assert m["reuse_tokens"] == len(B) and m["prefill_tokens"] == len(C)  # A is gone for C
    t.insert(*h2, 2)
    m3 = t.match(*h3)
    assert m3["matched_msgs"] == 0 and m3["prefill_tokens"] == len(B) + len(C)
    t.insert(*h3, 3)
    # root, A, B, C(1), drop-A after C(1), drop-A after B(2), C(2), B(3), C(3)
    assert t.stats()["nodes"] == 9
    for h in (h1, h2, h3):
        r = t.match(*h)
        assert r["kind"] == "reuse" and r["prefill_tokens"] == 0


def test_repos_copies_and_rotation(akv):
    """A repos opens a new position version.  A cached history that now
    ends with a repos needs its survivors at new positions: converted by
    rotation.  Once that history ran, the re-rotated copies exist and are
    reused as is; evicted, the state must be restored.  A message whose
    positions a repos does not change is reused as is."""
    X, Y, Z = [1] * 5, [2] * 7, [3] * 4
    t = akv.Tree()
    t.insert(*_hist([X, Y], drops=[(1, 0)]), 1)              # X dropped after Y, no repos
    with_repos = _hist([X, Y], drops=[(1, 0)], repos=[1])    # same, then a repos: Y -> 0..6
    m = t.match(*with_repos)
    assert m["kind"] == "rotate" and m["rotate_tokens"] == len(Y) and m["reuse_tokens"] == 0
    t.insert(*with_repos, 2)
    m = t.match(*with_repos)
    assert m["kind"] == "reuse" and m["reuse_tokens"] == len(Y)
    # a repos that moves nothing (nothing dropped before Z): Z reused as is
    keep = _hist([Z, Y], repos=[1])
    t.insert(*_hist([Z, Y]), 3)
    m = t.match(*keep)
    assert m["kind"] == "reuse" and m["reuse_tokens"] == len(Z) + len(Y)
    for r in (1, 2, 3):
        t.finish(r)
    assert t.evict(10 ** 9) == len(X) + 3 * len(Y) + len(Z)  # X, Y, Y's copy, Z, Y after Z
    assert t.stats()["resident_tokens"] == 0
    assert t.match(*with_repos)["kind"] == "restore"


def test_errors(akv):
    t = akv.Tree()
    h = _hist([A, B])
    t.insert(*h, 5)
    with pytest.raises(akv.AkvError):
        t.insert(*h, 5)  # already running
    with pytest.raises(akv.AkvError):
        t.finish(6)  # not running
    bad = _hist([A, B], drops=[(0, 1)])  # target later than its boundary
    with pytest.raises(akv.AkvError):
        t.match(*bad)


def _random_history(rng, alphabet=3, max_msgs=7):
    n = int(rng.integers(1, max_msgs + 1))
    msgs = [list(rng.integers(0, alphabet, size=int(rng.integers(1, 4)))) for _ in range(n)]
    drops, repos = [], []
    for m in range(n):
        for j in range(m + 1):
            if rng.random() < 0.15:
                drops.append((m, j))
        if rng.random() < 0.2:
            repos.append(m)
    return _hist(msgs, drops, repos)


@pytest.mark.parametrize("seed", range(6))
def test_random_operations_match_reference(akv, seed):
    """Random inserts / matches / finishes / evictions over histories drawn
    from a small token alphabet (so prefixes are shared and diverge on
    tokens and on operations): every result equals the reference model."""
    rng = np.random.default_rng(seed)
    pool = [_random_history(rng) for _ in range(12)]
    # extend some histories with more messages of an existing one (shared prefixes)
    for _ in range(8):
        base = pool[int(rng.integers(len(pool)))]
        ms, da, dt, ra = base[0]
        n = len(ms) - 1
        cut = int(rng.integers(1, n + 1))
        msgs = [list(base[1][ms[m]:ms[m + 1]]) for m in range(cut)]
        msgs += [list(rng.integers(0, 3, size=int(rng.integers(1, 4))))
                 for _ in range(int(rng.integers(0, 3)))]
        keep = [(int(a), int(b)) for a, b in zip(da, dt)
                if a < cut - 1 or (a == cut - 1 and rng.random() < 0.5)]
        rep = [int(r) for r in ra if r < cut - 1]
        pool.append(_hist(msgs, keep, rep))
    t, ref = akv.Tree(), TreeModel()
    running = []
    rid = 0
    for step in range(300):
        op = rng.random()
        h = pool[int(rng.integers(len(pool)))]
        if op < 0.4:
            assert t.match(*h) == ref.match(*h), step
        elif op < 0.7:
            rid += 1
            t.insert(*h, rid)
            ref.insert(*h, rid)
            running.append(rid)
        elif op < 0.85 and running:
            r = running.pop(int(rng.integers(len(running))))
            t.finish(r)
            ref.finish(r)
        else:
            want = int(rng.integers(1, 20))
            assert t.evict(want) == ref.evict(want), step
        assert t.stats() == ref.stats(), step
