"""Reference model of the cache-history tree and drop-aware eviction
(test infrastructure only; nothing of the library path imports it).

Follows the paper review page, section 4.2 ("AKV serving": a radix tree whose
paths carry the cache-operation history next to the tokens, drop nodes,
repos branches, eviction that frees KV only when no running request uses it,
dropped entries first, nodes kept as placeholders, each position version
separately) and section 3.4 / Figure 5 (the KV of a message depends on the
whole history before it).

No tree here: a storage unit is named by the history prefix it depends on,
written out as a tuple -- ("own", prefix through message m) for a message's
KV as computed, ("ver", prefix through the operations of a repos boundary r,
prefix through message j) for message j's re-rotated copy at that repos --
and every question is answered by looking such names up in flat
dictionaries.  The readings it shares with the library (which copy counts as
"at the right positions", eviction order) are the ones written in the
header comment of the library's tree API.

Pins: hand-worked cases from the page's rules, independent of both this
model and the library -- Figure 5's three histories, rotate / reuse / restore
after a repos, and the four eviction rules (dropped before finished, nothing
a running request or restore reads is freed, placeholders keep the path,
position versions evicted separately) -- run against this model as well as
against the library.
"""
from __future__ import annotations

from dataclasses import dataclass, field


def _ops_at(ms, drop_after, drop_target, repos_after):
    n = len(ms) - 1
    drops = [set() for _ in range(n)]
    for a, t in zip(drop_after, drop_target):
        drops[int(a)].add(int(t))
    repos = [False] * n
    for a in repos_after:
        repos[int(a)] = True
    return [(tuple(sorted(drops[m])), repos[m]) for m in range(n)]


def _events(ops, tokens):
    """(message token tuples, per-boundary op tuples or None)."""
    ms = [int(x) for x in ops[0]]
    n = len(ms) - 1
    toks = [tuple(int(t) for t in tokens[ms[m]:ms[m + 1]]) for m in range(n)]
    opl = _ops_at(*ops)
    return toks, [o if (o[0] or o[1]) else None for o in opl]


def _msg_key(toks, opl, m):
    key = []
    for i in range(m + 1):
        key.append(("m", toks[i]))
        if i < m and opl[i] is not None:
            key.append(("o", opl[i]))
    return tuple(key)


def _ops_key(toks, opl, r):
    return _msg_key(toks, opl, r) + (("o", opl[r]),)


def _replay(ms, opl_raw):
    """alive_before[m], alive_end, ver_of[m], first_pos[v][j] by a plain walk
    over the history (positions restart at 0 after each repos)."""
    n = len(ms) - 1
    alive = [False] * n
    alive_before, ver_of = [], []
    first_pos = [[None] * n]
    nxt, v = 0, 0
    for m in range(n):
        alive_before.append(list(alive))
        ver_of.append(v)
        first_pos[v][m] = nxt
        nxt += ms[m + 1] - ms[m]
        alive[m] = True
        drops, repos = opl_raw[m]
        for j in drops:
            alive[j] = False
        if repos:
            v += 1
            first_pos.append([None] * n)
            p = 0
            for j in range(m + 1):
                if alive[j]:
                    first_pos[v][j] = p
                    p += ms[j + 1] - ms[j]
            nxt = p
    return alive_before, list(alive), ver_of, first_pos


@dataclass
class _Unit:
    tokens: int
    seq: int
    resident: bool = True
    dropped: bool = False
    pins: int = 0
    last_use: int = 0


@dataclass
class TreeModel:
    units: dict = field(default_factory=dict)
    op_nodes: set = field(default_factory=set)
    running: dict = field(default_factory=dict)
    tick: int = 0
    created: int = 0

    def _unit(self, name, tokens):
        u = self.units.get(name)
        if u is None:
            self.created += 1
            u = self.units[name] = _Unit(tokens, self.created)
        return u

    def match(self, ops, tokens) -> dict:
        ms = [int(x) for x in ops[0]]
        n = len(ms) - 1
        toks, opl = _events(ops, tokens)
        opl_raw = _ops_at(*ops)
        k = 0
        while k < n and ("own", _msg_key(toks, opl, k)) in self.units:
            k += 1
        alive_before, alive_end, ver_of, first_pos = _replay(ms, opl_raw)
        full = k == n
        need = alive_end if full else alive_before[k]
        vfin = len(first_pos) - 1
        res = dict(kind=None, matched_msgs=k, reuse_tokens=0, rotate_tokens=0,
                   restore_tokens=0, prefill_tokens=sum(ms[m + 1] - ms[m] for m in range(k, n)))
        for j in range(k):
            if not need[j]:
                continue
            ln = ms[j + 1] - ms[j]
            copies = [(ver_of[j], self.units[("own", _msg_key(toks, opl, j))])]
            for r in range(j, k):
                if opl[r] is not None and opl[r][1]:
                    name = ("ver", _ops_key(toks, opl, r), _msg_key(toks, opl, j))
                    if name in self.units:
                        copies.append((ver_of[r] + 1, self.units[name]))
            res_any = any(u.resident for _, u in copies)
            same = any(u.resident and first_pos[v][j] == first_pos[vfin][j] for v, u in copies)
            if not res_any:
                res["restore_tokens"] += ln
            elif full and not same:
                res["rotate_tokens"] += ln
            else:
                res["reuse_tokens"] += ln
        if res["restore_tokens"]:
            res["kind"] = "restore"
        elif not full:
            res["kind"] = "prefill_suffix"
        elif res["rotate_tokens"]:
            res["kind"] = "rotate"
        else:
            res["kind"] = "reuse"
        return res

    def insert(self, ops, tokens, rid):
        assert rid not in self.running
        ms = [int(x) for x in ops[0]]
        n = len(ms) - 1
        toks, opl = _events(ops, tokens)
        opl_raw = _ops_at(*ops)
        self.tick += 1
        own = []
        for m in range(n):  # message units first, in order, then repos copies
            u = self._unit(("own", _msg_key(toks, opl, m)), ms[m + 1] - ms[m])
            own.append(u)
            if opl[m] is not None:
                self.op_nodes.add(_ops_key(toks, opl, m))
        alive = [False] * n
        copies = {}  # j -> list of its repos copies in history order
        for m in range(n):
            own[m].resident = True
            own[m].last_use = self.tick
            alive[m] = True
            for j in opl_raw[m][0]:
                alive[j] = False
            if opl_raw[m][1]:
                for j in range(m + 1):
                    if alive[j]:
                        c = self._unit(("ver", _ops_key(toks, opl, m), _msg_key(toks, opl, j)),
                                       ms[j + 1] - ms[j])
                        c.resident = True
                        c.last_use = self.tick
                        copies.setdefault(j, []).append(c)
        pins = []
        for j in range(n):
            act = alive[j]
            own[j].dropped = not act
            for c in copies.get(j, []):
                c.dropped = not act
            if act:
                newest = copies[j][-1] if j in copies else own[j]
                newest.pins += 1
                pins.append(newest)
        self.running[rid] = pins

    def finish(self, rid):
        for u in self.running.pop(rid):
            u.pins -= 1

    def evict(self, tokens) -> int:
        cand = [u for u in self.units.values() if u.resident and u.pins == 0]
        cand.sort(key=lambda u: (not u.dropped, u.last_use, u.seq))
        freed = 0
        for u in cand:
            if freed >= tokens:
                break
            u.resident = False
            freed += u.tokens
        return freed

    def stats(self) -> dict:
        msg_nodes = sum(1 for name in self.units if name[0] == "own")
        return dict(nodes=1 + msg_nodes + len(self.op_nodes), running=len(self.running),
                    resident_tokens=sum(u.tokens for u in self.units.values() if u.resident),
                    pinned_tokens=sum(u.tokens for u in self.units.values() if u.pins))
