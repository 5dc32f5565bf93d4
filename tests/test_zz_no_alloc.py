"""akv_decode_attention_static: decode for callers that cannot allocate.

Some callers cannot call cudaMalloc (a plug-in inside a framework that owns
the device memory pool, a request path that must not allocate), so they cannot
hand akv_decode_attention a workspace.  The static variant keeps its split-KV
partials in a fixed device array of the library instead.  These tests call it
through the C ABI and compare it with the workspace entry point, twice in a
row (the array is reused and keeps the previous call's contents): the two run
the same kernel on the same inputs, so the outputs must be equal bit for bit;
the fp64 oracle checks the values.  They also check that the calls leave the
device's free memory unchanged and that the array's address is looked up
again after a device reset.  The file is named so that pytest collects it
last.
"""
import os
import subprocess
import sys
import textwrap

import numpy as np
import pytest

import kv_cache_drop_gb300 as akv
import oracle
import workloads
from _util import assert_close

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _inputs(dtype, seed, Hq=16, Hkv=2):
    dw = workloads.decode_workload(seed=seed, B=3, active=(1500, 7000), steps=2, Hq=Hq, Hkv=Hkv,
                                   dtype=dtype)
    return dw


# (16, 1): the per-head kernel, merge in the launch; (64, 8), (16, 4), (16, 2):
# the all-heads kernel and its dependent merge launch
@pytest.mark.parametrize("dtype,Hq,Hkv", [("bf16", 16, 1), ("bf16", 16, 2), ("bf16", 64, 8),
                                          ("bf16", 16, 4), ("f32", 16, 2)])
def test_static_decode_matches_workspace_decode(dtype, Hq, Hkv):
    import torch
    dw = _inputs(dtype, 21, Hq, Hkv)
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
        assert torch.equal(got, ref), f"step {step}: static and workspace decode differ"
        # the values against fp64: the pool as it stands after the append
        # (keys stored rotated), the query rotated at its position
        store = np.uint16 if dtype == "bf16" else np.float32
        kpool = kp.view(torch.int16 if dtype == "bf16" else torch.float32).cpu().numpy()
        vpool = vp.view(torch.int16 if dtype == "bf16" else torch.float32).cpu().numpy()
        want = oracle.decode_attention(dw.q[step], dw.L + step, kpool.view(store),
                                       vpool.view(store), indptr, idx, dtype, 10000.0)
        assert_close(got.float().cpu().numpy(), want, dtype)


@pytest.mark.parametrize("Hq,Hkv", [(16, 1), (64, 8)])
def test_static_decode_allocates_nothing(Hq, Hkv):
    """After a first call (which may load the module holding the array), more
    calls leave the device's free memory exactly where it was; a call with
    B = 0 is accepted (set-up only)."""
    import torch
    dtype = "bf16"
    dw = _inputs(dtype, 23, Hq, Hkv)
    shp = akv.shape(dw.Hq, dw.Hkv, 64, dtype)
    kp = akv.to_device(dw.k_pool, dtype)
    vp = akv.to_device(dw.v_pool, dtype)
    max_kv = max(len(a) for a in dw.active_slots)
    indptr, idx = dw.indices_at(0)
    q = akv.to_device(dw.q[0], dtype)
    pos = akv.i32_device(dw.L)
    ip, ix = akv.i32_device(indptr), akv.i32_device(idx)
    out = torch.empty_like(q)
    akv.akv_decode_attention_static(shp, 0, q, pos, kp, vp, ip, ix, max_kv, out)
    akv.akv_decode_attention_static(shp, dw.B, q, pos, kp, vp, ip, ix, max_kv, out)
    torch.cuda.synchronize()
    first = out.clone()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(5):
        akv.akv_decode_attention_static(shp, dw.B, q, pos, kp, vp, ip, ix, max_kv, out)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, f"free device memory moved by {free0 - free1} bytes"
    assert torch.equal(out, first)


# Runs in a child process without torch: raw cudaMalloc'd buffers (the test
# may allocate; only the entry point may not), a static call and a workspace
# call, then cudaDeviceReset, which unloads the library's modules and frees
# the array, and the same two calls again on new buffers.
_RESET_CHILD = textwrap.dedent("""
    import ctypes, sys
    import numpy as np
    sys.path.insert(0, ROOT)
    import kv_cache_drop_gb300 as akv
    import workloads
    L = akv.lib()
    rt = ctypes.CDLL("libcudart.so.13")
    rt.cudaMalloc.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.c_size_t]
    rt.cudaMemcpy.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int]
    rt.cudaFree.argtypes = [ctypes.c_void_p]

    def ok(e, what):
        if e != 0:
            raise SystemExit(f"{what}: CUDA error {e}")

    dw = workloads.decode_workload(seed=25, B=3, active=(1500, 7000), steps=1, Hq=16, Hkv=2)
    indptr, idx = dw.indices_at(0)
    max_kv = int(max(np.diff(indptr)))
    host = dict(q=dw.q[0], pos=np.asarray(dw.L, np.int32), kp=dw.k_pool, vp=dw.v_pool,
                ip=np.asarray(indptr, np.int32), ix=np.asarray(idx, np.int32))
    shp = akv.Shape(16, 2, 64, akv.AKV_BF16, 10000.0)

    def run(static):
        dev = {}
        for name, a in host.items():
            a = np.ascontiguousarray(a)
            p = ctypes.c_void_p()
            ok(rt.cudaMalloc(ctypes.byref(p), a.nbytes), "cudaMalloc")
            ok(rt.cudaMemcpy(p, a.ctypes.data, a.nbytes, 1), "copy in")
            dev[name] = p
        nout = host["q"].nbytes
        out = ctypes.c_void_p()
        ok(rt.cudaMalloc(ctypes.byref(out), nout), "cudaMalloc")
        args = (ctypes.byref(shp), 3, dev["q"], dev["pos"], dev["kp"], dev["vp"], dev["ip"],
                dev["ix"], max_kv, out)
        ws = ctypes.c_void_p()
        if static:
            st = L.akv_decode_attention_static(*args, None)
        else:
            n = L.akv_decode_workspace(ctypes.byref(shp), 3, max_kv)
            ok(rt.cudaMalloc(ctypes.byref(ws), n), "cudaMalloc")
            st = L.akv_decode_attention(*args, ws, n, None)
        if st != 0:
            raise SystemExit(f"decode status {st}: {L.akv_last_error().decode()}")
        ok(rt.cudaDeviceSynchronize(), "synchronize")
        res = np.empty(nout, np.uint8)
        ok(rt.cudaMemcpy(res.ctypes.data, out, nout, 2), "copy out")
        for p in list(dev.values()) + [out] + ([ws] if ws.value else []):
            ok(rt.cudaFree(p), "cudaFree")
        return res

    before = [run(True), run(False)]
    ok(rt.cudaDeviceReset(), "cudaDeviceReset")
    after = [run(True), run(False)]
    for i, r in enumerate(before[1:] + after):
        if not np.array_equal(r, before[0]):
            raise SystemExit(f"result {i + 1} differs from the first static call")
    print("STATIC_RESET_OK")
""").replace("ROOT", repr(ROOT))


def test_static_decode_after_device_reset():
    """A device reset between calls: the static call looks the array up again
    and still equals the workspace call bit for bit."""
    env = dict(os.environ)
    r = subprocess.run([sys.executable, "-c", _RESET_CHILD], capture_output=True, text=True,
                       timeout=300, env=env, cwd=ROOT)
    print(r.stdout[-2000:], r.stderr[-2000:])
    assert r.returncode == 0 and "STATIC_RESET_OK" in r.stdout


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
