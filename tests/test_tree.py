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


@pytest.fixture(params=["library", "model"])
def tree(request, akv):
    """The library's tree, or the model in oracle/tree.py: the hand-derived
    cases below hold for both."""
    return akv.Tree() if request.param == "library" else TreeModel()


def test_figure5_histories_branch(tree):
    """Figure 5: (1) A, B, C then drop A; (2) A, B, drop A, then C; (3) B, C.
    (1) and (2) share A and B; C differs in all three; B of (3) is a
    separate branch."""
    h1 = _hist([A, B, C], drops=[(2, 0)])
    h2 = _hist([A, B, C], drops=[(1, 0)])
    h3 = _hist([B, C])
    t = tree
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


def test_repos_copies_and_rotation(tree):
    """A repos opens a new position version.  A cached history that now
    ends with a repos needs its survivors at new positions: converted by
    rotation.  Once that history ran, the re-rotated copies exist and are
    reused as is; evicted, the state must be restored.  A message whose
    positions a repos does not change is reused as is."""
    X, Y, Z = [1] * 5, [2] * 7, [3] * 4
    t = tree
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


# --- drop-aware eviction, pinned to the rules of the paper review page,
# section 4.2 ("drop-aware eviction") and Appendix A.1.2:
#   (1) physical KV is freed only when no running computation or restore
#       still uses it -- and KV a running request no longer uses (it dropped
#       it) is reclaimable before that request ends;
#   (2) dropped KV is evicted before the KV of finished requests (the latter
#       is likely to be reused by the next round);
#   (3) tree nodes stay as empty placeholders, so what lies below them stays
#       reachable;
#   (4) each position version is evicted on its own.
# The expected values below are worked out by hand from these rules; each
# case runs against the library's tree and against the model in
# oracle/tree.py.

P_, Q_, R_, S_ = [11] * 6, [12] * 5, [13] * 4, [14] * 3


def test_evict_dropped_before_finished(tree):
    """A finished request's KV was used longer ago than a dropped message, so
    an order by age alone would take it first; rule (2) takes the dropped
    message first."""
    done = _hist([R_, S_])                        # request 1: nothing dropped
    tree.insert(*done, 1)
    tree.finish(1)
    dropped = _hist([P_, Q_], drops=[(1, 0)])     # request 2: P dropped after Q
    tree.insert(*dropped, 2)
    tree.finish(2)
    assert tree.evict(len(P_)) == len(P_)
    # P is gone (a history that needs it must restore); R, S and Q are kept
    assert tree.match(*_hist([P_]))["kind"] == "restore"
    assert tree.match(*done)["kind"] == "reuse"
    assert tree.match(*dropped)["kind"] == "reuse"
    # next: the finished request's units, oldest insert first (R, S), then Q
    assert tree.evict(len(R_)) == len(R_)
    assert tree.match(*done)["kind"] == "restore"
    assert tree.match(*dropped)["kind"] == "reuse"


def test_evict_never_frees_what_a_running_request_uses(tree):
    """Rule (1): everything a running request reads at the end of its
    history stays resident, however much is asked for; what it dropped is
    freed while it still runs."""
    h = _hist([P_, Q_, R_], drops=[(1, 0)])       # P dropped after Q; Q, R active
    tree.insert(*h, 7)
    assert tree.evict(10 ** 9) == len(P_)         # only the dropped P
    st = tree.stats()
    assert st["resident_tokens"] == len(Q_) + len(R_) == st["pinned_tokens"]
    assert tree.match(*h)["kind"] == "reuse"
    assert tree.evict(10 ** 9) == 0
    tree.finish(7)                                # no longer in use: all of it goes
    assert tree.evict(10 ** 9) == len(Q_) + len(R_)
    assert tree.stats()["resident_tokens"] == 0


def test_restore_in_progress_holds_its_kv(tree):
    """A request restoring an evicted state holds it while the restore runs
    (it is inserted, so it pins what it reads): eviction during the restore
    frees none of it."""
    h = _hist([P_, Q_])
    tree.insert(*h, 1)
    tree.finish(1)
    assert tree.evict(10 ** 9) == len(P_) + len(Q_)
    assert tree.match(*h)["kind"] == "restore"
    tree.insert(*h, 2)                            # the restore runs
    assert tree.evict(10 ** 9) == 0
    assert tree.match(*h)["kind"] == "reuse"


def test_evicted_nodes_stay_as_placeholders(tree):
    """Rule (3): with the KV of the first messages evicted, their nodes still
    lead to the later messages: a longer history still matches all of its
    messages and needs only the evicted part restored."""
    h = _hist([P_, Q_, R_])
    tree.insert(*_hist([P_]), 1)
    tree.finish(1)
    tree.insert(*h, 2)                            # P held again, then Q, R
    tree.finish(2)
    nodes = tree.stats()["nodes"]
    assert tree.evict(len(P_)) == len(P_)         # same insert: P is the oldest
    assert tree.stats()["nodes"] == nodes
    m = tree.match(*h)
    assert m["matched_msgs"] == 3 and m["kind"] == "restore"
    assert m["restore_tokens"] == len(P_) and m["reuse_tokens"] == len(Q_) + len(R_)


def test_position_versions_evicted_separately(tree):
    """Rule (4): Q at its first positions and Q re-numbered by a repos are two
    copies.  A running request reads only the re-numbered one, so the other
    can be evicted, after which a history needing the first positions must
    restore while the running one still reuses."""
    v0 = _hist([P_, Q_])                               # Q at positions 6..10
    v1 = _hist([P_, Q_], drops=[(1, 0)], repos=[1])    # P dropped, Q moved to 0..4
    tree.insert(*v0, 1)
    tree.finish(1)
    tree.insert(*v1, 2)                                # runs on Q's new copy
    assert tree.evict(len(P_)) == len(P_)              # the dropped P first
    assert tree.evict(len(Q_)) == len(Q_)              # Q's first-position copy
    assert tree.match(*v1)["kind"] == "reuse"
    m = tree.match(*v0)
    assert m["kind"] == "restore" and m["restore_tokens"] == len(P_) + len(Q_)
    assert tree.evict(10 ** 9) == 0                    # the new copy is in use
    tree.finish(2)
    assert tree.evict(10 ** 9) == len(Q_)


# --- pool trees: the tree hands out the slots of a page-size-1 KV pool


def test_pool_cache_lists_match_replay(akv):
    """For random histories, the active cache a pool tree lists for a running
    request is the oracle replay's active cache: the same logical tokens at
    the same positions, in logical order; every slot is distinct and in the
    pool, and a fresh insert's writes cover every token of its history
    (each message once, plus one copy per survivor at each repos)."""
    import oracle
    rng = np.random.default_rng(5)
    for i in range(40):
        ops, tok = _random_history(rng)
        ms = ops[0]
        t = akv.Tree(pool_slots=4096)
        t.insert(ops, tok, 1)
        c = t.request_cache(1)
        rep = oracle.replay(*ops)
        np.testing.assert_array_equal(c["logical"], rep.active_u)
        np.testing.assert_array_equal(c["pos"], rep.active_p)
        assert len(set(c["slots"].tolist())) == len(c["slots"])
        assert ((c["slots"] >= 0) & (c["slots"] < 4096)).all()
        w = t.request_writes(1)
        n_copies = 0
        for a in sorted({int(x) for x in ops[3]}):
            n_copies += len(oracle.compact(*ops, upto=a)[0])
        assert len(w["slots"]) == int(ms[-1]) + n_copies
        assert len(set(w["slots"].tolist())) == len(w["slots"])
        # the listed cache slots are among the written ones, holding the same
        # token at the same position
        wmap = {int(s): (int(u), int(p)) for s, u, p in zip(w["slots"], w["logical"], w["pos"])}
        for s, u, p in zip(c["slots"], c["logical"], c["pos"]):
            assert wmap[int(s)] == (int(u), int(p))


def test_pool_insert_takes_the_dropped_slots_first(akv):
    """A full pool: the next insert evicts, in the drop-aware order, just the
    dropped message, and its tokens land in exactly the slots it freed."""
    done = _hist([R_, S_])
    dropped = _hist([P_, Q_], drops=[(1, 0)])
    S = len(R_) + len(S_) + len(P_) + len(Q_)
    t = akv.Tree(pool_slots=S)
    t.insert(*done, 1)
    t.finish(1)
    t.insert(*dropped, 2)
    w = t.request_writes(2)
    p_slots = sorted(int(s) for s, u in zip(w["slots"], w["logical"]) if u < len(P_))
    t.finish(2)
    assert t.pool_info() == {"pool_slots": S, "free_slots": 0}
    X = [15] * len(P_)
    t.insert(*_hist([X]), 3)
    assert sorted(t.request_writes(3)["slots"].tolist()) == p_slots
    assert t.match(*done)["kind"] == "reuse" and t.match(*dropped)["kind"] == "reuse"
    assert t.match(*_hist([P_]))["kind"] == "restore"


def test_pool_full_of_pinned_units_refuses(akv):
    """Every slot read by a running request: an insert that needs more
    fails, frees nothing and leaves that request not running; a reserve
    beyond the free slots fails the same way."""
    h = _hist([P_, Q_])
    t = akv.Tree(pool_slots=len(P_) + len(Q_) + 2)
    t.insert(*h, 1)
    with pytest.raises(akv.AkvError) as e:
        t.insert(*_hist([R_]), 2)
    assert e.value.status == 3
    assert t.pool_info()["free_slots"] == 2 and t.stats()["running"] == 1
    with pytest.raises(akv.AkvError):
        t.finish(2)
    tail = t.reserve(1, 2)
    assert sorted(tail.tolist()) == [len(P_) + len(Q_), len(P_) + len(Q_) + 1]
    with pytest.raises(akv.AkvError):
        t.reserve(1, 1)
    t.finish(1)  # the tail comes back; the units stay resident until evicted
    assert t.pool_info()["free_slots"] == 2
    assert t.evict(10 ** 9) == len(P_) + len(Q_)
    assert t.pool_info()["free_slots"] == len(P_) + len(Q_) + 2


@pytest.mark.parametrize("seed", range(4))
def test_pool_random_operations_keep_slots_consistent(akv, seed):
    """Random inserts, finishes, evictions and reserves on a small pool:
    resident tokens + held tails + free slots always add up to the pool; a
    slot listed by several running requests holds the same token at the
    same position for each; tails never overlap a listed slot; an insert
    that cannot get slots fails without changing the pool."""
    rng = np.random.default_rng(100 + seed)
    hist = [_random_history(rng, max_msgs=6) for _ in range(16)]
    S = 48
    t = akv.Tree(pool_slots=S)
    running, tails, rid = {}, {}, 0
    for step in range(300):
        op = rng.random()
        if op < 0.45:
            rid += 1
            before = t.pool_info()["free_slots"]
            try:
                t.insert(*hist[int(rng.integers(len(hist)))], rid)
                running[rid] = True
                tails[rid] = []
            except akv.AkvError as e:
                assert e.status == 3
                assert t.pool_info()["free_slots"] >= before  # evictions only
        elif op < 0.7 and running:
            r = list(running)[int(rng.integers(len(running)))]
            t.finish(r)
            del running[r], tails[r]
        elif op < 0.85 and running:
            r = list(running)[int(rng.integers(len(running)))]
            try:
                tails[r] += t.reserve(r, int(rng.integers(1, 4))).tolist()
            except akv.AkvError as e:
                assert e.status == 3
        else:
            t.evict(int(rng.integers(1, 20)))
        info, st = t.pool_info(), t.stats()
        held = sum(len(v) for v in tails.values())
        assert st["resident_tokens"] + held + info["free_slots"] == S, step
        owner = {}
        for r in running:
            c = t.request_cache(r)
            for s, u, p in zip(c["slots"].tolist(), c["logical"].tolist(), c["pos"].tolist()):
                assert 0 <= s < S
                assert owner.setdefault(s, (u, p)) == (u, p), step
        all_tails = [s for v in tails.values() for s in v]
        assert len(set(all_tails)) == len(all_tails)
        assert not set(all_tails) & set(owner), step
