"""Decoder layers of the single-prefill restoration: GEMM, RMSNorm, SwiGLU and
the multi-layer forward with segmented attention, against fp64 references."""
import numpy as np
import pytest

import kv_cache_drop_gb300 as akv
import oracle
import workloads
from _util import assert_close

pytestmark = pytest.mark.gpu

# Decoder outputs are final-RMSNorm states (unit RMS).  Every GEMM input is
# rounded to bf16 (relative 2^-9) across four layers while the oracle runs
# fp64 end to end: gate the relative RMS error at 2e-2 and the worst element
# at 0.25 (about 8 sigma of that error at unit scale).
MODEL_REL_RMS = 2e-2
MODEL_MAX_ABS = 0.25


def _torch():
    import torch
    return torch


def _bf16(a, dev="cuda"):
    return akv.to_device(np.ascontiguousarray(a), "bf16", dev)


@pytest.mark.parametrize("M,N,K", [(300, 352, 200), (128, 256, 64), (1000, 1024, 1024),
                                   (77, 4096, 1024),
                                   # one M tile, N of 32 (both W halves mostly or
                                   # wholly past N), K below one block
                                   (64, 32, 16), (384, 96, 72),
                                   # 65 x 9 = 585 tiles, 297 pairs of vertically
                                   # adjacent tiles: about four per two-CTA cluster of
                                   # the persistent kernel (both accumulators, each
                                   # reused after its epilogue), an odd tile count (the
                                   # last pair's second tile lies past M), ragged last
                                   # tile row and column, a partial last K block
                                   (8200, 2208, 328)])
def test_gemm_modes(M, N, K):
    torch = _torch()
    rng = np.random.default_rng(M + N + K)
    x = workloads.gen._normals(rng, (M, K), "bf16")
    w = workloads.gen._normals(rng, (N, K), "bf16", 0.05)
    ref = oracle.widen(x, "bf16") @ oracle.widen(w, "bf16").T
    scale = float(np.sqrt(np.mean(ref * ref)))
    yb = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    akv.akv_gemm_bf16(M, N, K, _bf16(x), _bf16(w), yb, 0)
    yf = torch.empty((M, N), dtype=torch.float32, device="cuda")
    akv.akv_gemm_bf16(M, N, K, _bf16(x), _bf16(w), yf, 1)
    acc = torch.full((M, N), 0.5, dtype=torch.float32, device="cuda")
    akv.akv_gemm_bf16(M, N, K, _bf16(x), _bf16(w), acc, 2)
    torch.cuda.synchronize()
    # fp32 accumulation over K products: relative error well under 1e-5 of scale
    assert np.max(np.abs(yf.cpu().numpy() - ref)) <= 1e-4 * scale * np.sqrt(K / 64)
    assert np.max(np.abs(acc.cpu().numpy() - 0.5 - ref)) <= 1e-4 * scale * np.sqrt(K / 64) + 1e-6
    # bf16 store: one rounding, relative 2^-9
    assert np.max(np.abs(yb.float().cpu().numpy() - ref) / (np.abs(ref) + 1e-3 * scale)) <= 2 ** -8


def test_rmsnorm_and_swiglu():
    torch = _torch()
    rng = np.random.default_rng(4)
    x = rng.standard_normal((37, 1024)).astype(np.float32) * 3
    y = torch.empty((37, 1024), dtype=torch.float32, device="cuda")
    akv.akv_rmsnorm(37, 1024, 1e-6, torch.from_numpy(x).cuda(), y)
    ref = oracle.rmsnorm(x.astype(np.float64), 1e-6)
    g = workloads.gen._normals(rng, (5000,), "bf16")
    u = workloads.gen._normals(rng, (5000,), "bf16")
    out = torch.empty(5000, dtype=torch.bfloat16, device="cuda")
    akv.akv_swiglu(5000, _bf16(g), _bf16(u), out)
    torch.cuda.synchronize()
    assert np.max(np.abs(y.cpu().numpy() - ref)) <= 1e-5
    gg, uu = oracle.widen(g, "bf16"), oracle.widen(u, "bf16")
    sref = gg / (1 + np.exp(-gg)) * uu
    assert np.max(np.abs(out.float().cpu().numpy() - sref) / (np.abs(sref) + 1e-3)) <= 2 ** -7
    # a ragged tail (4,999 = 624 groups of 8 + 7) and pointers one element off
    # 16-byte alignment (the element-wise path): the same values bit for bit
    gd, ud = _bf16(g), _bf16(u)
    for off, n in ((0, 4999), (1, 4998)):
        o2 = torch.zeros(5000, dtype=torch.bfloat16, device="cuda")
        akv.akv_swiglu(n, gd[off:off + n], ud[off:off + n], o2[off:off + n])
        torch.cuda.synchronize()
        assert torch.equal(o2[off:off + n], out[off:off + n]), (off, n)


def _gpu_weights(mw):
    return [{k: _bf16(np.ascontiguousarray(v.T)) for k, v in w.items()} for w in mw.weights]


def run_decoder(mw, reqs=None):
    """Forward of requests `reqs` (default all) of a model workload; returns
    fp32 numpy [n_req * T, d]."""
    torch = _torch()
    reqs = list(range(mw.n_req)) if reqs is None else reqs
    T = mw.T
    shp = akv.shape(mw.Hq, mw.Hkv, mw.D, "bf16", mw.rope_base)
    ops = [(mw.msg_start, *mw.ops[b]) for b in reqs]
    cu = np.arange(len(reqs) + 1, dtype=np.int64) * T
    plan = akv.Plan(shp, cu, ops)
    x = _bf16(np.concatenate([mw.x] * len(reqs)))
    out = torch.empty((len(reqs) * T, mw.d_model), dtype=torch.float32, device="cuda")
    ws = torch.empty(akv.akv_decoder_workspace(plan, mw.d_model, mw.d_ff), dtype=torch.uint8,
                     device="cuda")
    weights = _gpu_weights(mw)  # must outlive the asynchronous kernels
    akv.akv_decoder_forward(plan, weights, mw.d_model, mw.d_ff, mw.eps, x, out, ws)
    torch.cuda.synchronize()
    del weights
    assert akv.akv_workspace_status(ws) == 0, "a kernel barrier wait timed out"
    return out.cpu().numpy()


def run_decoder_shared(mw, prefix):
    """Forward with the first request owning the shared prefix and the others
    holding only their rows after it; returns fp32 numpy [stored rows, d]."""
    torch = _torch()
    T, n = mw.T, mw.n_req
    shp = akv.shape(mw.Hq, mw.Hkv, mw.D, "bf16", mw.rope_base)
    ops = [(mw.msg_start, *mw.ops[b]) for b in range(n)]
    lens = [T] + [T - prefix] * (n - 1)
    cu = np.concatenate([[0], np.cumsum(lens)])
    plan = akv.Plan(shp, cu, ops, share=[(-1, 0)] + [(0, prefix)] * (n - 1))
    x = _bf16(np.concatenate([mw.x] + [mw.x[prefix:]] * (n - 1)))
    out = torch.empty((int(cu[-1]), mw.d_model), dtype=torch.float32, device="cuda")
    ws = torch.empty(akv.akv_decoder_workspace(plan, mw.d_model, mw.d_ff), dtype=torch.uint8,
                     device="cuda")
    weights = _gpu_weights(mw)
    akv.akv_decoder_forward(plan, weights, mw.d_model, mw.d_ff, mw.eps, x, out, ws)
    torch.cuda.synchronize()
    del weights
    assert akv.akv_workspace_status(ws) == 0, "a kernel barrier wait timed out"
    return out.cpu().numpy(), cu


def _check_shared_equals_unshared(mw, prefix, full):
    got, cu = run_decoder_shared(mw, prefix)
    T = mw.T
    assert np.array_equal(got[:T], full[:T])
    for b in range(1, mw.n_req):
        assert np.array_equal(got[cu[b]:cu[b + 1]], full[b * T + prefix:(b + 1) * T]), b


def test_decoder_shared_prefix_small():
    """The 128-token shared prefix computed once: every stored row equals the
    unshared forward bit for bit (the prefix keys are the same windows in the
    same order)."""
    mw = workloads.model_workload(seed=5, n_req=3, prefix=128, following=640,
                                  asst_len=(20, 60), tool_len=(60, 150))
    _check_shared_equals_unshared(mw, 128, run_decoder(mw))


def _rel(got, ref):
    d = got - ref
    return float(np.sqrt(np.mean(d * d)) / np.sqrt(np.mean(ref * ref))), float(np.abs(d).max())


def test_decoder_ffn_two_gemms():
    """d_ff = 1056, not a multiple of 128: gate and up run as two GEMMs and a
    separate SwiGLU instead of one GEMM with a SwiGLU epilogue."""
    mw = workloads.model_workload(seed=6, n_req=1, prefix=128, following=384, n_layers=2,
                                  d_ff=1056, asst_len=(20, 60), tool_len=(60, 150))
    got = run_decoder(mw)
    ref = oracle.model_replay(mw.weights, mw.x, mw.msg_start, *mw.ops[0], mw.Hq, mw.Hkv, mw.D,
                              mw.rope_base, mw.eps)
    rel, mx = _rel(got, ref)
    print(f"[parity] decoder d_ff=1056: rel_rms={rel:.3e} max_abs={mx:.3e}")
    assert rel <= MODEL_REL_RMS and mx <= MODEL_MAX_ABS


def test_decoder_small_vs_oracle():
    """Three requests, 4 layers at the full layer shape (d 1024, 16/4 heads,
    SwiGLU 4096), shared 128-token prefix + 640 diverging tokens."""
    mw = workloads.model_workload(seed=5, n_req=3, prefix=128, following=640,
                                  asst_len=(20, 60), tool_len=(60, 150))
    got = run_decoder(mw)
    T = mw.T
    for b in range(mw.n_req):
        ref = oracle.model_replay(mw.weights, mw.x, mw.msg_start, *mw.ops[b], mw.Hq, mw.Hkv,
                                  mw.D, mw.rope_base, mw.eps)
        rel, mx = _rel(got[b * T:(b + 1) * T], ref)
        print(f"[parity] decoder request {b}: rel_rms={rel:.3e} max_abs={mx:.3e}")
        assert rel <= MODEL_REL_RMS and mx <= MODEL_MAX_ABS


def test_decoder_full_size_properties():
    """32 requests x (8192 shared + 24576 diverging) tokens: every request's
    shared-prefix rows are bit-identical, a request alone equals the same
    request inside the batch bit for bit, the batch with the prefix computed
    once (akv_plan_create_shared) equals it bit for bit, and the first 1024
    prefix rows match the oracle."""
    mw = workloads.model_workload()
    T, P = mw.T, 8192
    got = run_decoder(mw)
    assert np.isfinite(got).all()
    pref = got[:P]
    for b in range(1, mw.n_req):
        assert np.array_equal(got[b * T:b * T + P], pref), b
    alone = run_decoder(mw, reqs=[5])
    assert np.array_equal(alone, got[5 * T:6 * T])
    _check_shared_equals_unshared(mw, P, got)  # the prefix computed once
    n = 1024
    ref = oracle.model_replay(mw.weights, mw.x[:n], np.array([0, n], np.int32), [], [], [],
                              mw.Hq, mw.Hkv, mw.D, mw.rope_base, mw.eps)
    rel, mx = _rel(pref[:n], ref)
    print(f"[parity] decoder prefix rows: rel_rms={rel:.3e} max_abs={mx:.3e}")
    assert rel <= MODEL_REL_RMS and mx <= MODEL_MAX_ABS


def _op_rows(mw, b, n_total=64, seed=0):
    """Rows of request b next to each of its op boundaries (the last row
    before it, the first two after it), then random rows up to n_total."""
    _, da, _, ra = (mw.msg_start, *mw.ops[b])
    T = mw.T
    pick = set()
    for a in sorted({int(x) for x in da} | {int(x) for x in ra}):
        s = int(mw.msg_start[a + 1])
        pick.update(t for t in (s - 1, s, s + 1) if 0 <= t < T)
    rng = np.random.default_rng(seed + b)
    while len(pick) < n_total:
        pick.add(int(rng.integers(0, T)))
    return np.array(sorted(pick), dtype=np.int64)


def test_decoder_full_size_teacher_forced_layers():
    """Full-size decoder workload (8,192 shared + 24,576 diverging tokens),
    requests 1, 2 and 5 (one, two and two repos): every layer's segmented
    attention on op-bearing rows against the oracle fed the GPU's own layer
    input.

    Layer l's input: akv_decoder_forward run with the first l layers returns
    the final RMSNorm of the residual stream after those layers, which (the
    RMSNorm weights are 1) is layer l's normalised input.  Rounded to bf16,
    it goes through layer l's Q/K/V projections (akv_gemm_bf16, the
    forward's GEMM kernel) and then the segment attention over the batch's
    plan; the oracle replays the request's op log over the same Q/K/V bytes.
    Rows right after each drop and repos boundary are always among the
    compared ones."""
    from oracle.parallel import replay_attention_rows
    torch = _torch()
    full = workloads.model_workload()
    reqs = [1, 2, 5]
    assert [len(full.ops[b][2]) for b in reqs] == [1, 2, 2]
    T, d = full.T, full.d_model
    shp = akv.shape(full.Hq, full.Hkv, full.D, "bf16", full.rope_base)
    ops = [(full.msg_start, *full.ops[b]) for b in reqs]
    plan = akv.Plan(shp, np.arange(len(reqs) + 1) * T, ops)
    x = _bf16(np.concatenate([full.x] * len(reqs)))
    weights = _gpu_weights(full)
    n = len(reqs) * T
    dq, dkv = full.Hq * full.D, full.Hkv * full.D
    ws = torch.empty(akv.akv_decoder_workspace(plan, d, full.d_ff), dtype=torch.uint8,
                     device="cuda")
    aws = plan.workspace()
    h = torch.empty((n, d), dtype=torch.float32, device="cuda")
    worst = 0.0
    for l in range(full.n_layers):
        akv.akv_decoder_forward(plan, weights[:l], d, full.d_ff, full.eps, x, h, ws)
        a = h.to(torch.bfloat16)
        q = torch.empty((n, dq), dtype=torch.bfloat16, device="cuda")
        k = torch.empty((n, dkv), dtype=torch.bfloat16, device="cuda")
        v = torch.empty((n, dkv), dtype=torch.bfloat16, device="cuda")
        akv.akv_gemm_bf16(n, dq, d, a, weights[l]["wq"], q, 0)
        akv.akv_gemm_bf16(n, dkv, d, a, weights[l]["wk"], k, 0)
        akv.akv_gemm_bf16(n, dkv, d, a, weights[l]["wv"], v, 0)
        o = torch.empty_like(q)
        akv.akv_segment_attention_run(plan, q, k, v, o, aws)
        torch.cuda.synchronize()
        assert akv.akv_workspace_status(aws) == 0, "a kernel barrier wait timed out"
        qs, ks, vs, os_ = (t.view(torch.int16).cpu().numpy().view(np.uint16)
                           for t in (q, k, v, o))
        for i, b in enumerate(reqs):
            sl = slice(i * T, (i + 1) * T)
            rows = _op_rows(full, b, seed=10 * l)
            ref = replay_attention_rows(
                ops[i], qs[sl].reshape(T, full.Hq, full.D), ks[sl].reshape(T, full.Hkv, full.D),
                vs[sl].reshape(T, full.Hkv, full.D), "bf16", full.rope_base, rows)
            got = oracle.widen(os_[sl].reshape(T, full.Hq, full.D)[rows], "bf16")
            print(f"[parity] layer {l} request {b}: {len(rows)} rows")
            mx, _ = assert_close(got, ref, "bf16")
            worst = max(worst, mx)
    del weights
    print(f"[parity] teacher-forced layers: worst max_abs {worst:.3e}")
