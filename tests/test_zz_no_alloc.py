"""akv_decode_attention_static: decode for callers that cannot allocate.

Some callers cannot call cudaMalloc (a plug-in inside a framework that owns
the device memory pool, a request path that must not allocate), so they cannot
hand akv_decode_attention a workspace.  The static variant keeps its split-KV
partials in a fixed device array of the library instead.  These tests call it
through the C ABI and compare it with the workspace entry point, twice in a
row (the array is reused and keeps the previous call's contents).  The file
is named so that pytest collects it last.
"""
import numpy as np
import pytest

import kv_cache_drop_gb300 as akv
import workloads
from _util import assert_close

pytestmark = pytest.mark.gpu


def _inputs(dtype, seed):
    dw = workloads.decode_workload(seed=seed, B=3, active=(1500, 7000), steps=2, Hq=16, Hkv=2,
                                   dtype=dtype)
    return dw


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_static_decode_matches_workspace_decode(dtype):
    import torch
    dw = _inputs(dtype, 21)
    shp = akv.shape(dw.Hq, dw.Hkv, 64, dtype)
    kp = akv.to_device(dw.k_pool, dtype)
    vp = akv.to_device(dw.v_pool, dtype)
    max_kv = max(len(a) for a in dw.active_slots) + dw.steps
    ws = torch.empty(akv.akv_decode_workspace(shp, dw.B, max_kv), dtype=torch.uint8,
                     device="cuda")
    for step in range(dw.steps):  # two calls in a row on the shared array
        indptr, idx = dw.indices_at(step)
        pos = akv.i32_device(dw.L + step)
        akv.akv_append_kv(shp, dw.B, akv.to_device(dw.k_new[step], dtype),
                          akv.to_device(dw.v_new[step], dtype), pos,
                          akv.i32_device(dw.append_slots[step]), kp, vp)
        q = akv.to_device(dw.q[step], dtype)
        ip, ix = akv.i32_device(indptr), akv.i32_device(idx)
        ref = torch.empty_like(q)
        got = torch.full_like(q, float("nan"))
        akv.akv_decode_attention(shp, dw.B, q, pos, kp, vp, ip, ix, max_kv, ref, ws)
        akv.akv_decode_attention_static(shp, dw.B, q, pos, kp, vp, ip, ix, max_kv, got)
        torch.cuda.synchronize()
        g, r = got.float().cpu().numpy(), ref.float().cpu().numpy()
        assert np.isfinite(g).all()
        assert_close(g, r.astype(np.float64), dtype)


def test_static_decode_rejects_oversized_requests():
    import torch
    shp = akv.shape(64, 8, 64, "bf16")
    cap = akv.akv_decode_static_scratch_bytes()
    assert cap == 16 << 20
    q = torch.zeros((64, 64, 64), dtype=torch.bfloat16, device="cuda")
    dummy = torch.zeros(16, dtype=torch.int32, device="cuda")
    with pytest.raises(akv.AkvError) as e:
        # 64 requests x 64 heads x 100 splits of partials do not fit 16 MiB
        akv.akv_decode_attention_static(shp, 64, q, dummy, q, q, dummy, dummy, 200000, q)
    assert e.value.status == 4
    assert "static scratch" in str(e.value)
