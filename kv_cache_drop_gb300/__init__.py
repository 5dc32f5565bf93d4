"""Python binding of libakv, the GB300 (sm_103a) AKV hot path.

Argument marshalling only: every function below forwards to the C entry point
of the same name in ``libakv.so`` (declared in ``include/akv.h``), passing
device pointers of torch tensors, host arrays of the op logs and the current
CUDA stream.  There is no fallback: if the library is missing or a call
fails, an exception is raised.

Op logs are passed per request as ``(msg_start, drop_after, drop_target,
repos_after)`` integer arrays in the operate-after form of the pages'
request grammar (drop the KV of message ``drop_target[i]`` after message
``drop_after[i]`` ends; re-position after ``repos_after[j]``; drops before
the repos at one boundary).
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libakv.so")

AKV_F32, AKV_BF16 = 0, 1
_STATUS = {0: "AKV_OK", 1: "AKV_ERR_INVALID", 2: "AKV_ERR_CUDA", 3: "AKV_ERR_WORKSPACE",
           4: "AKV_ERR_UNSUPPORTED", 5: "AKV_ERR_DEVICE"}

_i32p = ctypes.POINTER(ctypes.c_int32)


class AkvError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{_STATUS.get(status, status)}: {msg}")
        self.status = status


class Shape(ctypes.Structure):
    _fields_ = [("Hq", ctypes.c_int32), ("Hkv", ctypes.c_int32), ("D", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("rope_base", ctypes.c_float)]


class OpLog(ctypes.Structure):
    _fields_ = [("n_msgs", ctypes.c_int32), ("msg_start", _i32p),
                ("n_drops", ctypes.c_int32), ("drop_after", _i32p), ("drop_target", _i32p),
                ("n_repos", ctypes.c_int32), ("repos_after", _i32p)]


class PlanInfo(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("n_qtiles", ctypes.c_int64),
                ("n_windows", ctypes.c_int64), ("n_full_windows", ctypes.c_int64),
                ("visible_pairs", ctypes.c_int64), ("n_segments", ctypes.c_int64),
                ("max_versions", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("workspace_bytes", ctypes.c_size_t)]

    def as_dict(self):
        return {k: getattr(self, k) for k, _ in self._fields_ if k != "reserved"}


class LayerWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("wq", "wk", "wv", "wo", "wg", "wu", "wd")]


class TreeMatch(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("matched_msgs", ctypes.c_int32),
                ("reuse_tokens", ctypes.c_int64), ("rotate_tokens", ctypes.c_int64),
                ("restore_tokens", ctypes.c_int64), ("prefill_tokens", ctypes.c_int64)]

    def as_dict(self):
        return {k: getattr(self, k) for k, _ in self._fields_}


class TreeStats(ctypes.Structure):
    _fields_ = [("nodes", ctypes.c_int64), ("running", ctypes.c_int64),
                ("resident_tokens", ctypes.c_int64), ("pinned_tokens", ctypes.c_int64)]

    def as_dict(self):
        return {k: getattr(self, k) for k, _ in self._fields_}


TREE_KINDS = {0: "reuse", 1: "rotate", 2: "prefill_suffix", 3: "restore"}

_lib = None

_SIGS = {
    "akv_last_error": (ctypes.c_char_p, []),
    "akv_version": (ctypes.c_char_p, []),
    "akv_plan_create": (ctypes.c_int, [ctypes.POINTER(Shape), ctypes.c_int32, _i32p, _i32p,
                                       ctypes.POINTER(OpLog), ctypes.POINTER(ctypes.c_void_p)]),
    "akv_plan_create_shared": (ctypes.c_int, [ctypes.POINTER(Shape), ctypes.c_int32, _i32p,
                                              ctypes.POINTER(OpLog), _i32p, _i32p,
                                              ctypes.POINTER(ctypes.c_void_p)]),
    "akv_plan_destroy": (None, [ctypes.c_void_p]),
    "akv_tree_create": (ctypes.c_int, [ctypes.POINTER(ctypes.c_void_p)]),
    "akv_tree_destroy": (None, [ctypes.c_void_p]),
    "akv_tree_match": (ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(OpLog), _i32p,
                                      ctypes.POINTER(TreeMatch)]),
    "akv_tree_insert": (ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(OpLog), _i32p,
                                       ctypes.c_int64]),
    "akv_tree_finish": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int64]),
    "akv_tree_evict": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int64,
                                      ctypes.POINTER(ctypes.c_int64)]),
    "akv_tree_stats": (ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(TreeStats)]),
    "akv_tree_create_pool": (ctypes.c_int, [ctypes.c_int64, ctypes.POINTER(ctypes.c_void_p)]),
    "akv_tree_request_writes": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int64, _i32p, _i32p,
                                               _i32p, ctypes.c_int64,
                                               ctypes.POINTER(ctypes.c_int64)]),
    "akv_tree_request_cache": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int64, _i32p, _i32p,
                                              _i32p, ctypes.c_int64,
                                              ctypes.POINTER(ctypes.c_int64)]),
    "akv_tree_reserve": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                                        _i32p]),
    "akv_tree_pool_info": (ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(ctypes.c_int64),
                                          ctypes.POINTER(ctypes.c_int64)]),
    "akv_plan_get_info": (ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(PlanInfo)]),
    "akv_plan_tables": (ctypes.c_int, [ctypes.c_void_p, _i32p, _i32p, _i32p, _i32p]),
    "akv_segment_attention_run": (ctypes.c_int, [ctypes.c_void_p] + [ctypes.c_void_p] * 5 +
                                  [ctypes.c_size_t, ctypes.c_void_p]),
    "akv_segment_prepare": (ctypes.c_int, [ctypes.c_void_p] * 5 + [ctypes.c_size_t,
                                                                   ctypes.c_void_p]),
    "akv_segment_attend": (ctypes.c_int, [ctypes.c_void_p] * 4 + [ctypes.c_size_t,
                                                                  ctypes.c_void_p]),
    "akv_segment_attention_workspace": (ctypes.c_size_t, [ctypes.POINTER(Shape), ctypes.c_int32,
                                                          _i32p, ctypes.POINTER(OpLog)]),
    "akv_segment_attention": (ctypes.c_int, [ctypes.POINTER(Shape), ctypes.c_int32, _i32p, _i32p,
                                             ctypes.POINTER(OpLog)] + [ctypes.c_void_p] * 5 +
                              [ctypes.c_size_t, ctypes.c_void_p]),
    "akv_segment_visible_counts": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p,
                                                  ctypes.c_void_p, ctypes.c_size_t,
                                                  ctypes.c_void_p]),
    "akv_workspace_status": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p,
                                            ctypes.POINTER(ctypes.c_uint32)]),
    "akv_compact_workspace": (ctypes.c_size_t, [ctypes.POINTER(OpLog), ctypes.c_int32]),
    "akv_compact": (ctypes.c_int, [ctypes.POINTER(OpLog), ctypes.c_int32, ctypes.c_int32,
                                   ctypes.c_void_p, ctypes.c_void_p, _i32p, ctypes.c_void_p,
                                   ctypes.c_size_t, ctypes.c_void_p]),
    "akv_repos_rotate": (ctypes.c_int, [ctypes.POINTER(Shape), ctypes.c_int32] +
                         [ctypes.c_void_p] * 7 + [ctypes.c_void_p]),
    "akv_repos_boundary_workspace": (ctypes.c_size_t, [ctypes.POINTER(OpLog), ctypes.c_int32]),
    "akv_repos_boundary": (ctypes.c_int, [ctypes.POINTER(Shape), ctypes.POINTER(OpLog),
                                          ctypes.c_int32, ctypes.c_int32] +
                           [ctypes.c_void_p] * 4 + [_i32p, ctypes.c_void_p, ctypes.c_size_t,
                                                    ctypes.c_void_p]),
    "akv_decode_attention_append": (ctypes.c_int, [ctypes.POINTER(Shape), ctypes.c_int32] +
                                    [ctypes.c_void_p] * 9 + [ctypes.c_int32, ctypes.c_void_p,
                                                             ctypes.c_void_p, ctypes.c_size_t,
                                                             ctypes.c_void_p]),
    "akv_decode_rope_workspace": (ctypes.c_size_t, [ctypes.POINTER(Shape), ctypes.c_int32,
                                                    ctypes.c_int32]),
    "akv_decode_attention_rope": (ctypes.c_int, [ctypes.POINTER(Shape), ctypes.c_int32] +
                                  [ctypes.c_void_p] * 10 + [ctypes.c_int32, ctypes.c_void_p,
                                                            ctypes.c_void_p, ctypes.c_size_t,
                                                            ctypes.c_void_p]),
    "akv_decode_workspace": (ctypes.c_size_t, [ctypes.POINTER(Shape), ctypes.c_int32,
                                               ctypes.c_int32]),
    "akv_decode_attention": (ctypes.c_int, [ctypes.POINTER(Shape), ctypes.c_int32] +
                             [ctypes.c_void_p] * 6 + [ctypes.c_int32, ctypes.c_void_p,
                                                      ctypes.c_void_p, ctypes.c_size_t,
                                                      ctypes.c_void_p]),
    "akv_decode_attention_static": (ctypes.c_int, [ctypes.POINTER(Shape), ctypes.c_int32] +
                                    [ctypes.c_void_p] * 6 + [ctypes.c_int32, ctypes.c_void_p,
                                                             ctypes.c_void_p]),
    "akv_decode_static_scratch_bytes": (ctypes.c_size_t, []),
    "akv_decode_check_indices": (ctypes.c_int, [ctypes.c_int32] + [ctypes.c_void_p] * 2 +
                                 [ctypes.c_int32] * 3 + [ctypes.c_void_p, ctypes.c_void_p]),
    "akv_gemm_bf16": (ctypes.c_int, [ctypes.c_int32] * 3 + [ctypes.c_void_p] * 3 +
                      [ctypes.c_int32, ctypes.c_void_p]),
    "akv_rmsnorm": (ctypes.c_int, [ctypes.c_int32, ctypes.c_int32, ctypes.c_float, ctypes.c_int32,
                                   ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                                   ctypes.c_void_p, ctypes.c_void_p]),
    "akv_swiglu": (ctypes.c_int, [ctypes.c_int64] + [ctypes.c_void_p] * 4),
    "akv_decoder_workspace": (ctypes.c_size_t, [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32]),
    "akv_decoder_forward": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32,
                                           ctypes.POINTER(LayerWeights), ctypes.c_int32,
                                           ctypes.c_int32, ctypes.c_float] +
                            [ctypes.c_void_p] * 3 + [ctypes.c_size_t, ctypes.c_void_p]),
    "akv_append_kv": (ctypes.c_int, [ctypes.POINTER(Shape), ctypes.c_int32] +
                      [ctypes.c_void_p] * 6 + [ctypes.c_void_p]),
}

EXPORTED = sorted(_SIGS)


def lib():
    """Load libakv.so (built by ``__graft_entry__.build()``); raise if absent."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libakv.so is not built ({LIB_PATH}); run __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _check(status: int):
    if status != 0:
        raise AkvError(status, lib().akv_last_error().decode())


def _dtype_code(dtype) -> int:
    import torch
    if dtype in ("f32", torch.float32, AKV_F32):
        return AKV_F32
    if dtype in ("bf16", torch.bfloat16, AKV_BF16):
        return AKV_BF16
    raise ValueError(f"unsupported dtype {dtype}")


def shape(Hq: int, Hkv: int, D: int = 64, dtype="bf16", rope_base: float = 10000.0) -> Shape:
    return Shape(Hq, Hkv, D, _dtype_code(dtype), rope_base)


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


class _Ops:
    """Keeps the numpy arrays of a batch of op logs alive for a C call."""

    def __init__(self, ops):
        self.keep = []
        self.arr = (OpLog * max(1, len(ops)))()
        for i, (ms, da, dt, ra) in enumerate(ops):
            ms, da, dt, ra = _i32(ms), _i32(da), _i32(dt), _i32(ra)
            self.keep += [ms, da, dt, ra]
            self.arr[i] = OpLog(len(ms) - 1, ms.ctypes.data_as(_i32p), len(da),
                                da.ctypes.data_as(_i32p), dt.ctypes.data_as(_i32p), len(ra),
                                ra.ctypes.data_as(_i32p))

    def ptr(self, i: int = 0):
        return ctypes.pointer(self.arr[i])

    @property
    def base(self):
        return ctypes.cast(self.arr, ctypes.POINTER(OpLog))


def _dev(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensor must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


class Tree:
    """Cache-history tree with drop-aware eviction (akv_tree_*).  A history
    is (ops, token_ids): an op log tuple as for Plan and the messages' token
    ids (int32, msg_start[-1] of them)."""

    def __init__(self, pool_slots: int = 0):
        """pool_slots > 0: the tree also manages the token slots of a
        page-size-1 KV pool of that many slots (akv_tree_create_pool)."""
        self._lib = lib()
        h = ctypes.c_void_p()
        if pool_slots:
            _check(self._lib.akv_tree_create_pool(pool_slots, ctypes.byref(h)))
        else:
            _check(self._lib.akv_tree_create(ctypes.byref(h)))
        self.handle = h

    def __del__(self):
        if getattr(self, "handle", None):
            self._lib.akv_tree_destroy(self.handle)
            self.handle = None

    @staticmethod
    def _args(ops, token_ids):
        o = _Ops([ops])
        tok = _i32(token_ids)
        return o, tok

    def match(self, ops, token_ids) -> dict:
        o, tok = self._args(ops, token_ids)
        r = TreeMatch()
        _check(self._lib.akv_tree_match(self.handle, o.ptr(), tok.ctypes.data_as(_i32p),
                                        ctypes.byref(r)))
        d = r.as_dict()
        d["kind"] = TREE_KINDS[d["kind"]]
        return d

    def insert(self, ops, token_ids, request_id: int):
        o, tok = self._args(ops, token_ids)
        _check(self._lib.akv_tree_insert(self.handle, o.ptr(), tok.ctypes.data_as(_i32p),
                                         request_id))

    def finish(self, request_id: int):
        _check(self._lib.akv_tree_finish(self.handle, request_id))

    def evict(self, tokens: int) -> int:
        f = ctypes.c_int64(0)
        _check(self._lib.akv_tree_evict(self.handle, tokens, ctypes.byref(f)))
        return f.value

    def stats(self) -> dict:
        st = TreeStats()
        _check(self._lib.akv_tree_stats(self.handle, ctypes.byref(st)))
        return st.as_dict()

    def _list(self, fn, request_id: int):
        n = ctypes.c_int64(0)
        _check(fn(self.handle, request_id, None, None, None, 0, ctypes.byref(n)))
        out = [np.empty(n.value, dtype=np.int32) for _ in range(3)]
        _check(fn(self.handle, request_id, *[o.ctypes.data_as(_i32p) for o in out], n.value,
                  ctypes.byref(n)))
        return dict(slots=out[0], logical=out[1], pos=out[2])

    def request_writes(self, request_id: int) -> dict:
        """Slots the request's insert allocated: dict of int32 arrays slots,
        logical, pos (fill slot with K rotated at pos and V of token logical)."""
        return self._list(self._lib.akv_tree_request_writes, request_id)

    def request_cache(self, request_id: int) -> dict:
        """The request's active cache in logical order: slots, logical, pos."""
        return self._list(self._lib.akv_tree_request_cache, request_id)

    def reserve(self, request_id: int, n: int) -> np.ndarray:
        out = np.empty(n, dtype=np.int32)
        _check(self._lib.akv_tree_reserve(self.handle, request_id, n,
                                          out.ctypes.data_as(_i32p)))
        return out

    def pool_info(self) -> dict:
        a, b = ctypes.c_int64(0), ctypes.c_int64(0)
        _check(self._lib.akv_tree_pool_info(self.handle, ctypes.byref(a), ctypes.byref(b)))
        return dict(pool_slots=a.value, free_slots=b.value)


class Plan:
    """Host plan of a segment-batch restoration prefill (akv_plan_create)."""

    def __init__(self, shp: Shape, cu_seqlens, ops, logical_idx=None, share=None):
        """share: None, or per request (from, length) -- request b's first
        `length` logical rows are request `from`'s and are not in the batch
        (akv_plan_create_shared); (-1, 0) for a request that shares nothing."""
        self._lib = lib()
        self.shape = shp
        self._ops = _Ops(ops)
        cu = _i32(cu_seqlens)
        li = None if logical_idx is None else _i32(logical_idx)
        h = ctypes.c_void_p()
        if share is None:
            _check(self._lib.akv_plan_create(ctypes.byref(shp), len(ops),
                                             cu.ctypes.data_as(_i32p),
                                             None if li is None else li.ctypes.data_as(_i32p),
                                             self._ops.base, ctypes.byref(h)))
        else:
            sf = _i32([f for f, _ in share])
            sl = _i32([n for _, n in share])
            _check(self._lib.akv_plan_create_shared(ctypes.byref(shp), len(ops),
                                                    cu.ctypes.data_as(_i32p), self._ops.base,
                                                    sf.ctypes.data_as(_i32p),
                                                    sl.ctypes.data_as(_i32p), ctypes.byref(h)))
        self.handle = h
        info = PlanInfo()
        _check(self._lib.akv_plan_get_info(h, ctypes.byref(info)))
        self.info = info.as_dict()

    def tables(self):
        T = self.info["T"]
        out = [np.empty(T, dtype=np.int32) for _ in range(4)]
        _check(self._lib.akv_plan_tables(self.handle, *[o.ctypes.data_as(_i32p) for o in out]))
        return dict(tok_pos=out[0], tok_seg=out[1], tok_ver=out[2], drop_seg=out[3])

    def workspace(self, device="cuda"):
        import torch
        return torch.empty(max(1, self.info["workspace_bytes"]), dtype=torch.uint8, device=device)

    def __del__(self):
        h = getattr(self, "handle", None)
        if h is not None and h.value:
            self._lib.akv_plan_destroy(h)
            self.handle = None


def akv_plan_create(shp: Shape, cu_seqlens, ops, logical_idx=None) -> Plan:
    return Plan(shp, cu_seqlens, ops, logical_idx)


def akv_segment_attention_run(plan: Plan, q, k, v, out, workspace, stream=None):
    _check(lib().akv_segment_attention_run(plan.handle, _dev(q), _dev(k), _dev(v), _dev(out),
                                           _dev(workspace), workspace.numel(), _stream(stream)))


def akv_segment_prepare(plan: Plan, q, k, v, workspace, stream=None):
    _check(lib().akv_segment_prepare(plan.handle, _dev(q), _dev(k), _dev(v), _dev(workspace),
                                     workspace.numel(), _stream(stream)))


def akv_segment_attend(plan: Plan, q, out, workspace, stream=None):
    _check(lib().akv_segment_attend(plan.handle, _dev(q), _dev(out), _dev(workspace),
                                    workspace.numel(),
                                    _stream(stream)))


def akv_segment_attention_workspace(shp: Shape, cu_seqlens, ops) -> int:
    o = _Ops(ops)
    cu = _i32(cu_seqlens)
    return lib().akv_segment_attention_workspace(ctypes.byref(shp), len(ops),
                                                 cu.ctypes.data_as(_i32p), o.base)


def akv_segment_attention(shp: Shape, cu_seqlens, logical_idx, ops, q, k, v, out, workspace,
                          stream=None):
    o = _Ops(ops)
    cu = _i32(cu_seqlens)
    li = None if logical_idx is None else _i32(logical_idx)
    _check(lib().akv_segment_attention(ctypes.byref(shp), len(ops), cu.ctypes.data_as(_i32p),
                                       None if li is None else li.ctypes.data_as(_i32p), o.base,
                                       _dev(q), _dev(k), _dev(v), _dev(out), _dev(workspace),
                                       workspace.numel(), _stream(stream)))


def akv_segment_visible_counts(plan: Plan, counts, workspace, stream=None):
    _check(lib().akv_segment_visible_counts(plan.handle, _dev(counts), _dev(workspace),
                                            workspace.numel(), _stream(stream)))


def akv_workspace_status(workspace, stream=None) -> int:
    code = ctypes.c_uint32(0)
    st = lib().akv_workspace_status(_dev(workspace), _stream(stream), ctypes.byref(code))
    if st not in (0, 5):
        _check(st)
    return code.value


def akv_compact_workspace(ops, T: int) -> int:
    o = _Ops([ops])
    return lib().akv_compact_workspace(o.ptr(), T)


def akv_compact(ops, T: int, upto: int, active_idx, active_pos, workspace, stream=None) -> int:
    o = _Ops([ops])
    n = ctypes.c_int32(0)
    _check(lib().akv_compact(o.ptr(), T, upto, _dev(active_idx), _dev(active_pos),
                             ctypes.byref(n), _dev(workspace),
                             0 if workspace is None else workspace.numel(), _stream(stream)))
    return n.value


def akv_repos_rotate(shp: Shape, r: int, src_idx, pos_from, pos_to, k_in, v_in, k_out, v_out,
                     stream=None):
    _check(lib().akv_repos_rotate(ctypes.byref(shp), r, _dev(src_idx), _dev(pos_from),
                                  _dev(pos_to), _dev(k_in), _dev(v_in), _dev(k_out), _dev(v_out),
                                  _stream(stream)))


def akv_repos_boundary_workspace(ops, T: int) -> int:
    o = _Ops([ops])
    return lib().akv_repos_boundary_workspace(o.ptr(), T)


def akv_repos_boundary(shp: Shape, ops, T: int, upto: int, k_in, v_in, k_out, v_out, workspace,
                       stream=None) -> int:
    """Survivors of boundary `upto` gathered, keys re-rotated to 0..n-1; returns n."""
    o = _Ops([ops])
    n = ctypes.c_int32(0)
    _check(lib().akv_repos_boundary(ctypes.byref(shp), o.ptr(), T, upto, _dev(k_in), _dev(v_in),
                                    _dev(k_out), _dev(v_out), ctypes.byref(n), _dev(workspace),
                                    0 if workspace is None else workspace.numel(),
                                    _stream(stream)))
    return n.value


def akv_decode_workspace(shp: Shape, B: int, max_kv: int) -> int:
    return lib().akv_decode_workspace(ctypes.byref(shp), B, max_kv)


def akv_decode_attention(shp: Shape, B: int, q, q_pos, k_pool, v_pool, kv_indptr, kv_indices,
                         max_kv: int, out, workspace, stream=None):
    _check(lib().akv_decode_attention(ctypes.byref(shp), B, _dev(q), _dev(q_pos), _dev(k_pool),
                                      _dev(v_pool), _dev(kv_indptr), _dev(kv_indices), max_kv,
                                      _dev(out), _dev(workspace),
                                      0 if workspace is None else workspace.numel(),
                                      _stream(stream)))


def akv_decode_attention_append(shp: Shape, B: int, q, q_pos, k_new, v_new, new_slot, k_pool,
                                v_pool, kv_indptr, kv_indices, max_kv: int, out, workspace,
                                stream=None):
    """Append the step's token (key rotated at q_pos) and decode, one launch."""
    _check(lib().akv_decode_attention_append(ctypes.byref(shp), B, _dev(q), _dev(q_pos),
                                             _dev(k_new), _dev(v_new), _dev(new_slot),
                                             _dev(k_pool), _dev(v_pool), _dev(kv_indptr),
                                             _dev(kv_indices), max_kv, _dev(out),
                                             _dev(workspace),
                                             0 if workspace is None else workspace.numel(),
                                             _stream(stream)))


def akv_decode_rope_workspace(shp: Shape, B: int, max_kv: int) -> int:
    return lib().akv_decode_rope_workspace(ctypes.byref(shp), B, max_kv)


def akv_decode_attention_rope(shp: Shape, B: int, q, q_pos, k_new, v_new, new_slot, k_pool,
                              v_pool, kv_indptr, kv_indices, kv_pos, max_kv: int, out, workspace,
                              stream=None):
    """Decode over a pool of keys stored before RoPE, each entry rotated at
    kv_pos as it is read; k_new/v_new/new_slot (or all None) append the step's
    token first."""
    _check(lib().akv_decode_attention_rope(ctypes.byref(shp), B, _dev(q), _dev(q_pos),
                                           _dev(k_new), _dev(v_new), _dev(new_slot),
                                           _dev(k_pool), _dev(v_pool), _dev(kv_indptr),
                                           _dev(kv_indices), _dev(kv_pos), max_kv, _dev(out),
                                           _dev(workspace),
                                           0 if workspace is None else workspace.numel(),
                                           _stream(stream)))


def akv_decode_attention_static(shp: Shape, B: int, q, q_pos, k_pool, v_pool, kv_indptr,
                                kv_indices, max_kv: int, out, stream=None):
    """Decode with the split-KV partials in the library's static device array
    (no workspace; see include/akv.h for the size limit and sharing rules)."""
    _check(lib().akv_decode_attention_static(ctypes.byref(shp), B, _dev(q), _dev(q_pos),
                                             _dev(k_pool), _dev(v_pool), _dev(kv_indptr),
                                             _dev(kv_indices), max_kv, _dev(out),
                                             _stream(stream)))


def akv_decode_check_indices(B: int, kv_indptr, kv_indices, S: int, max_kv: int, status,
                             stream=None):
    """Device check of decode index data (see include/akv.h); ORs violation
    bits into ``status`` (a zeroed CUDA uint32/int32 tensor of one element)."""
    _check(lib().akv_decode_check_indices(B, _dev(kv_indptr), _dev(kv_indices),
                                          kv_indices.numel(), S, max_kv, _dev(status),
                                          _stream(stream)))


def akv_decode_static_scratch_bytes() -> int:
    return lib().akv_decode_static_scratch_bytes()


def akv_append_kv(shp: Shape, n: int, k_new, v_new, pos, slot, k_pool, v_pool, stream=None):
    _check(lib().akv_append_kv(ctypes.byref(shp), n, _dev(k_new), _dev(v_new), _dev(pos),
                               _dev(slot), _dev(k_pool), _dev(v_pool), _stream(stream)))


def to_device(arr: np.ndarray, dtype: str, device="cuda"):
    """numpy float32 array or bf16 bit patterns (uint16) -> torch tensor on device."""
    import torch
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).to(device).view(
            torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(arr, dtype=np.float32)).to(device)


def i32_device(a, device="cuda"):
    import torch
    return torch.from_numpy(_i32(a)).to(device)


def akv_gemm_bf16(M: int, N: int, K: int, x, w, y, out_mode: int = 0, stream=None):
    _check(lib().akv_gemm_bf16(M, N, K, _dev(x), _dev(w), _dev(y), out_mode, _stream(stream)))


def akv_rmsnorm(rows: int, d: int, eps: float, x, y, weight=None, stream=None):
    import torch
    code = {torch.float32: AKV_F32, torch.bfloat16: AKV_BF16}
    _check(lib().akv_rmsnorm(rows, d, eps, code[x.dtype], _dev(x), _dev(weight), code[y.dtype],
                             _dev(y), _stream(stream)))


def akv_swiglu(n: int, g, u, out, stream=None):
    _check(lib().akv_swiglu(n, _dev(g), _dev(u), _dev(out), _stream(stream)))


def akv_decoder_workspace(plan: Plan, d_model: int, d_ff: int) -> int:
    return lib().akv_decoder_workspace(plan.handle, d_model, d_ff)


def akv_decoder_forward(plan: Plan, layers, d_model: int, d_ff: int, eps: float, x, out,
                        workspace, stream=None):
    """layers: list of dicts of device bf16 tensors wq..wd, each [out, in]."""
    arr = (LayerWeights * max(1, len(layers)))()
    for i, w in enumerate(layers):
        arr[i] = LayerWeights(*[w[n].data_ptr() for n in ("wq", "wk", "wv", "wo", "wg", "wu",
                                                          "wd")])
    _check(lib().akv_decoder_forward(plan.handle, len(layers), arr, d_model, d_ff, eps, _dev(x),
                                     _dev(out), _dev(workspace), workspace.numel(),
                                     _stream(stream)))
