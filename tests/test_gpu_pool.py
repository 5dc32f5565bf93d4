"""Drop-aware eviction over a page-size-1 KV pool on the GPU: a pool tree hands
out the slots, the caller fills them with akv_append_kv, a later request's
insert evicts dropped messages and reuses their slots, and decode over the
slots the tree lists matches the fp64 oracle."""
import numpy as np
import pytest

import kv_cache_drop_gb300 as akv
import oracle
import workloads
from _util import assert_close

pytestmark = pytest.mark.gpu


def _history(r, n_msgs, drops=(), repos=()):
    ms = r.msg_start[:n_msgs + 1].astype(np.int32)
    da = np.array([a for a, _ in drops], np.int32)
    dt = np.array([t for _, t in drops], np.int32)
    ra = np.array(sorted(repos), np.int32)
    return (ms, da, dt, ra)


def _fill(tree, rid, r, shp, kp, vp):
    """Write the slots request rid's insert allocated: K rotated at the
    listed position and V of the listed token."""
    w = tree.request_writes(rid)
    n = len(w["slots"])
    if n:
        akv.akv_append_kv(shp, n, akv.to_device(r.k[w["logical"]], "bf16"),
                          akv.to_device(r.v[w["logical"]], "bf16"), akv.i32_device(w["pos"]),
                          akv.i32_device(w["slots"]), kp, vp)
    return w


def test_pool_tree_evict_reuse_decode():
    import torch
    Hq, Hkv = 8, 2
    shp = akv.shape(Hq, Hkv, 64, "bf16")
    conv1 = workloads.random_request(71, n_msgs=10, max_len=120, Hq=Hq, Hkv=Hkv, dtype="bf16",
                                     p_drop=0.0, p_repos=0.0, min_len=20)
    conv2 = workloads.random_request(72, n_msgs=6, max_len=120, Hq=Hq, Hkv=Hkv, dtype="bf16",
                                     p_drop=0.0, p_repos=0.0, min_len=20)
    tok1 = np.arange(conv1.T, dtype=np.int32)
    tok2 = np.arange(conv2.T, dtype=np.int32) + 1_000_000  # never equal to conv1's
    hA = _history(conv1, 6)
    hB = _history(conv1, 8, drops=[(5, 1), (6, 3)], repos=[6])
    hC = _history(conv2, 5, drops=[(2, 0)])
    ms1, ms2 = conv1.msg_start, conv2.msg_start
    # size the pool so that C fits only once B's two dropped messages are evicted
    probe = akv.Tree(pool_slots=1 << 20)
    probe.insert(hA, tok1[:ms1[6]], 1)
    probe.insert(hB, tok1[:ms1[8]], 2)
    probe.finish(1)
    used_ab = (1 << 20) - probe.pool_info()["free_slots"]
    probe.insert(hC, tok2[:ms2[5]], 3)
    need_c = len(probe.request_writes(3)["slots"])
    dropped = int(ms1[2] - ms1[1] + ms1[4] - ms1[3])
    S = used_ab + need_c - dropped + 3
    assert 0 < S - used_ab < need_c

    tree = akv.Tree(pool_slots=S)
    kp = torch.zeros((S, Hkv, 64), dtype=torch.bfloat16, device="cuda")
    vp = torch.zeros_like(kp)
    tree.insert(hA, tok1[:ms1[6]], 1)
    wA = _fill(tree, 1, conv1, shp, kp, vp)
    assert tree.match(hA, tok1[:ms1[6]])["kind"] == "reuse"
    tree.insert(hB, tok1[:ms1[8]], 2)           # reuses A's messages 0..5
    _fill(tree, 2, conv1, shp, kp, vp)
    tree.finish(1)
    # the slots of messages 1 and 3 (written for A, dropped by B)
    drop_slots = {s for s, u in zip(wA["slots"].tolist(), wA["logical"].tolist())
                  if ms1[1] <= u < ms1[2] or ms1[3] <= u < ms1[4]}
    assert len(drop_slots) == dropped
    tree.insert(hC, tok2[:ms2[5]], 3)           # must evict the dropped messages
    wC = _fill(tree, 3, conv2, shp, kp, vp)
    assert drop_slots <= set(wC["slots"].tolist()), "the freed slots were not reused"
    assert tree.match(hA, tok1[:ms1[6]])["kind"] == "restore"   # A needs message 1 again
    assert tree.match(hB, tok1[:ms1[8]])["kind"] == "reuse"     # B runs on, untouched
    torch.cuda.synchronize()

    # decode one new token per running request (B, C) over the listed slots
    reqs = [(2, conv1, hB, tok1, 8), (3, conv2, hC, tok2, 5)]
    indptr, indices, qpos, new_slot, qs, ks, vs, refs = [0], [], [], [], [], [], [], []
    for rid, conv, h, _, nm in reqs:
        c = tree.request_cache(rid)
        rep = oracle.replay(*h)
        np.testing.assert_array_equal(c["logical"], rep.active_u)   # bit-exact
        np.testing.assert_array_equal(c["pos"], rep.active_p)
        vrows = vp[torch.from_numpy(c["slots"].astype(np.int64)).cuda()]
        np.testing.assert_array_equal(vrows.view(torch.int16).cpu().numpy().view(np.uint16),
                                      conv.v[c["logical"]])
        s_new = tree.reserve(rid, 1)
        t_new = int(conv.msg_start[nm])                  # next token of the conversation
        indices += c["slots"].tolist() + s_new.tolist()
        indptr.append(len(indices))
        qpos.append(rep.next_pos)
        new_slot.append(int(s_new[0]))
        qs.append(conv.q[t_new])
        ks.append(conv.k[t_new])
        vs.append(conv.v[t_new])
        # the oracle: the same history plus the decode token as one more message
        ms_ext = np.concatenate([h[0], [h[0][-1] + 1]]).astype(np.int32)
        rows = np.concatenate([np.arange(h[0][-1]), [t_new]])
        ref, _ = oracle.replay_attention(ms_ext, h[1], h[2], h[3], conv.q[rows], conv.k[rows],
                                         conv.v[rows], "bf16", conv.rope_base,
                                         rows=[int(h[0][-1])])
        refs.append(ref[0])
    B = len(reqs)
    max_kv = int(np.max(np.diff(indptr)))
    out = torch.empty((B, Hq, 64), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(akv.akv_decode_workspace(shp, B, max_kv), dtype=torch.uint8,
                     device="cuda")
    akv.akv_decode_attention_append(shp, B, akv.to_device(np.stack(qs), "bf16"),
                                    akv.i32_device(qpos), akv.to_device(np.stack(ks), "bf16"),
                                    akv.to_device(np.stack(vs), "bf16"),
                                    akv.i32_device(new_slot), kp, vp, akv.i32_device(indptr),
                                    akv.i32_device(indices), max_kv, out, ws)
    torch.cuda.synchronize()
    assert_close(out.float().cpu().numpy(), np.stack(refs), "bf16")
    for rid, *_ in reqs:
        tree.finish(rid)
    assert tree.pool_info()["free_slots"] == S - tree.stats()["resident_tokens"]
