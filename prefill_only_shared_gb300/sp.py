"""ctypes binding of libsp (include/sp.h): argument marshalling only.

Every function here has the name of the C entry point it wraps and does no
arithmetic of the method: it checks dtypes / devices / contiguity, passes raw
pointers and the current CUDA stream, and raises ``SpError`` on a non-OK
status.  Device memory comes from torch and is owned by the caller.

There is no fallback: if ``libsp.so`` has not been built, importing the
library fails with an error that says how to build it.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

from . import build as _build

SP_OK = 0
SP_ALL_ROUNDS = -1
SP_QTYPE_NOUL, SP_QTYPE_CHOICE, SP_QTYPE_SCORE = 0, 1, 2
STATUS_NAMES = {0: "SP_OK", 1: "SP_ERR_ARG", 2: "SP_ERR_LIMIT", 3: "SP_ERR_POOL_FULL",
                4: "SP_ERR_CUDA", 5: "SP_ERR_DEVICE_TIMEOUT", 6: "SP_ERR_DEVICE_BOUNDS",
                7: "SP_ERR_WORKSPACE"}


class SpError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)} ({sp_status_str(status)})")


class sp_shape(ctypes.Structure):
    _fields_ = [("n_q_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("hidden", ctypes.c_int32), ("vocab", ctypes.c_int32)]


class sp_plan_stats(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in (
        "n_requests", "n_branches", "n_segments", "n_shared_segments", "n_rounds",
        "logical_tokens", "computed_tokens", "reused_tokens", "node_tokens", "pages_used",
        "desc_bytes", "attn_workspace_bytes", "cache_hit_tokens")]

    def as_dict(self):
        return {n: int(getattr(self, n)) for n, _ in self._fields_}


_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I32P = ctypes.POINTER(ctypes.c_int32)
_I64P = ctypes.POINTER(ctypes.c_int64)
_SZ = ctypes.c_size_t


class sp_input_set(ctypes.Structure):
    """One device input set of sp_run_pass_host (device buffers, pinned
    descriptor staging, the set's two CUDA events)."""
    _fields_ = [("q", _P), ("k", _P), ("v", _P), ("h", _P), ("label_off", _P),
                ("label_ids", _P), ("q_rows", ctypes.c_int64), ("h_rows", ctypes.c_int64),
                ("labels_cap", ctypes.c_int64), ("desc_host", _P), ("desc_host_bytes", _SZ),
                ("done_event", _P), ("copied_event", _P)]

# Every symbol declared in include/sp.h, with its ctypes signature.
SIGNATURES = {
    "sp_plan_build": (_I32, [ctypes.POINTER(sp_shape), _I32, _I32P, _I64P, _I32P, _I32, _I32,
                             ctypes.POINTER(_P)]),
    "sp_plan_free": (None, [_P]),
    "sp_cache_create": (_I32, [_I32, ctypes.POINTER(_P)]),
    "sp_cache_free": (None, [_P]),
    "sp_cache_get_stats": (_I32, [_P, _I64P]),
    "sp_plan_build_cached": (_I32, [ctypes.POINTER(sp_shape), _P, _I32, _I32P, _I64P, _I32P, _I32,
                                    ctypes.POINTER(_P)]),
    "sp_cache_commit": (_I32, [_P, _P]),
    "sp_batcher_create": (_I32, [ctypes.POINTER(sp_shape), ctypes.c_int64, _I32, ctypes.POINTER(_P)]),
    "sp_batcher_free": (None, [_P]),
    "sp_batcher_submit": (_I32, [_P, _I32, _I64P, _I32P, _I64P, _I64P]),
    "sp_batcher_pending": (_I32, [_P, _I32P, _I64P]),
    "sp_batcher_next": (_I32, [_P, _I32, _I32, ctypes.POINTER(_P), _I32P, ctypes.POINTER(_I64P),
                               ctypes.POINTER(_I32P), ctypes.POINTER(_I64P)]),
    "sp_plan_get_stats": (_I32, [_P, ctypes.POINTER(sp_plan_stats)]),
    "sp_plan_rounds": (_I32, [_P, _I32P, ctypes.POINTER(_I32P), ctypes.POINTER(_I32P)]),
    "sp_plan_segments": (_I32, [_P, _I32P] + [ctypes.POINTER(_I32P)] * 2 + [ctypes.POINTER(_I64P)]
                         + [ctypes.POINTER(_I32P)] * 4),
    "sp_plan_segment_sources": (_I32, [_P, ctypes.POINTER(_I32P), ctypes.POINTER(_I32P)]),
    "sp_plan_branches": (_I32, [_P, ctypes.POINTER(_I32P), ctypes.POINTER(_I64P),
                                ctypes.POINTER(_I32P), ctypes.POINTER(_I32P)]),
    "sp_plan_descriptor": (_I32, [_P, ctypes.POINTER(_P), ctypes.POINTER(_SZ)]),
    "sp_plan_call_info": (_I32, [_P, _I32, _I32, _I64P]),
    "sp_plan_upload": (_I32, [_P, _P, _SZ, _P]),
    "sp_prefix_attn": (_I32, [_P, _P, _I32, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "sp_branch_attn": (_I32, [_P, _P, _I32, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "sp_tree_attn": (_I32, [_P, _P, _I32, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "sp_label_workspace_bytes": (_SZ, [_I32, _I32, _I32]),
    "sp_label_logprobs": (_I32, [_P, _P, _I32, _I32, _I32, _P, _P, _I32, _P, _P, _P, _SZ, _P]),
    "sp_label_logprobs_noalloc": (_I32, [_P, _P, _I32, _I32, _I32, _P, _P, _I32, _P, _P, _P]),
    "sp_label_softmax": (_I32, [_P, _P, _I32, _P, _P, _P]),
    "sp_label_decide": (_I32, [_P, _P, _P, _I32, _P, _P, _P, _P, _P]),
    "sp_candidate_decide": (_I32, [_P, _P, _I32, _P, _P, _I32, _P, _P, _P, _P, _P]),
    "sp_wait_flag": (_I32, [_P, ctypes.c_uint32, ctypes.c_int64, _P]),
    "sp_check_labels": (_I32, [_I32P, _I32P, _I32, _I32]),
    "sp_option_softmax": (_I32, [_P, _I32, _P, _I32, _P, _I32, _P, _P, _P, _P, _P]),
    "sp_run_pass": (_I32, [ctypes.POINTER(sp_shape), _I32, _I32P, _I64P, _I32P, ctypes.c_int64,
                           _P, _P, _P, _P, _I32, _P, _P, _P, _SZ, _P, _SZ, _P, _P, _P, _P, _I32,
                           _P, _P, _P, _SZ, _P, _P, _P, ctypes.POINTER(sp_plan_stats)]),
    "sp_run_pass_host": (_I32, [ctypes.POINTER(sp_shape), _I32, _I32P, _I64P, _I32P,
                                ctypes.c_int64, _P, _P, _P, _P, _P, _P, _I32,
                                ctypes.POINTER(sp_input_set), _P, _I32, _P, _P, _P, _SZ, _P, _SZ,
                                _P, _P, _P, _P, _SZ, _P, _P, _P, _P, _P, _P,
                                ctypes.POINTER(sp_plan_stats)]),
    "sp_check_options": (_I32, [_I32P, _I32, _I32, _I32P, _I32]),
    "sp_check_device_error": (_I32, [_P]),
    "sp_status_str": (ctypes.c_char_p, [_I32]),
    "sp_last_launch_count": (_I32, []),
}

_LIB = None


def lib() -> ctypes.CDLL:
    """The loaded libsp.so; raises if it has not been built."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(_build.LIB):
            raise RuntimeError(
                "libsp.so is not built (CUDA path required, no fallback): run "
                "`python -c 'import __graft_entry__ as g; g.build()'` or "
                "prefill_only_shared_gb300.build.build()")
        L = ctypes.CDLL(_build.LIB)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _LIB = L
    return _LIB


def sp_status_str(status: int) -> str:
    try:
        return lib().sp_status_str(int(status)).decode()
    except Exception:  # library missing: still produce a message
        return STATUS_NAMES.get(status, str(status))


def _check(status: int, where: str):
    if status != SP_OK:
        raise SpError(status, where)


def _stream(stream):
    """A cudaStream_t from None (torch's current stream), a torch stream or a
    raw handle (int)."""
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _dev(t: torch.Tensor, dtype, name: str):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _np(a, dtype):
    return np.ascontiguousarray(np.asarray(a), dtype=dtype)


class Plan:
    """Owns an sp_plan*; host-only.  A plan built with a prefix cache keeps the
    cache alive (the plan must be freed first)."""

    def __init__(self, ptr: ctypes.c_void_p, shape: sp_shape, cache=None):
        self._ptr = ptr
        self.shape = shape
        self._stats = None
        self.cache = cache

    @property
    def ptr(self):
        return self._ptr

    def free(self):
        if self._ptr:
            lib().sp_plan_free(self._ptr)
            self._ptr = None

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass

    def stats(self) -> dict:
        """Token and launch accounting (a plan is immutable: read once)."""
        if self._stats is None:
            st = sp_plan_stats()
            _check(lib().sp_plan_get_stats(self._ptr, ctypes.byref(st)), "sp_plan_get_stats")
            self._stats = st.as_dict()
        return dict(self._stats)

    def rounds(self) -> list:
        n = _I32()
        off = _I32P()
        br = _I32P()
        _check(lib().sp_plan_rounds(self._ptr, ctypes.byref(n), ctypes.byref(off), ctypes.byref(br)),
               "sp_plan_rounds")
        offs = np.ctypeslib.as_array(off, shape=(n.value + 1,)).copy()
        brs = np.ctypeslib.as_array(br, shape=(int(offs[-1]),)).copy() if offs[-1] else np.zeros(0, np.int32)
        return [brs[offs[r]:offs[r + 1]].tolist() for r in range(n.value)]

    def segments(self) -> dict:
        n = _I32()
        ptrs = [_I32P(), _I32P(), _I64P(), _I32P(), _I32P(), _I32P(), _I32P()]
        _check(lib().sp_plan_segments(self._ptr, ctypes.byref(n), *[ctypes.byref(p) for p in ptrs]),
               "sp_plan_segments")
        names = ["req", "parent", "node_start", "len", "round", "shared", "first_page"]
        return {k: np.ctypeslib.as_array(p, shape=(n.value,)).copy() if n.value else np.zeros(0)
                for k, p in zip(names, ptrs)}

    def descriptor(self) -> bytes:
        """Host copy of the device descriptor image."""
        data = ctypes.c_void_p()
        n = ctypes.c_size_t()
        _check(lib().sp_plan_descriptor(self._ptr, ctypes.byref(data), ctypes.byref(n)),
               "sp_plan_descriptor")
        return ctypes.string_at(data, n.value)

    def call_info(self, rnd: int, kind: int) -> dict:
        info = (ctypes.c_int64 * 7)()
        _check(lib().sp_plan_call_info(self._ptr, int(rnd), int(kind), info), "sp_plan_call_info")
        keys = ["append_off", "n_append", "tile_off", "n_tiles", "merge_off", "n_merges", "n_parts"]
        return {k: int(x) for k, x in zip(keys, info)}

    def segment_sources(self) -> dict:
        """Per segment: a branch through it and its first token's position in
        that branch."""
        n = self.stats()["n_segments"]
        ptrs = [_I32P(), _I32P()]
        _check(lib().sp_plan_segment_sources(self._ptr, *[ctypes.byref(p) for p in ptrs]),
               "sp_plan_segment_sources")
        return {k: np.ctypeslib.as_array(p, shape=(n,)).copy() if n else np.zeros(0, np.int32)
                for k, p in zip(("branch", "pos"), ptrs)}

    def row_sources(self):
        """(branch, position) of every node-token row, int64 arrays."""
        seg, src = self.segments(), self.segment_sources()
        lens = seg["len"].astype(np.int64)
        rows_b = np.repeat(src["branch"].astype(np.int64), lens)
        start = np.repeat(seg["node_start"].astype(np.int64), lens)
        pos0 = np.repeat(src["pos"].astype(np.int64), lens)
        r = np.arange(int(lens.sum()), dtype=np.int64)  # segments are in row order
        return rows_b, pos0 + (r - start)

    def branches(self) -> dict:
        nb = self.stats()["n_branches"]
        ptrs = [_I32P(), _I64P(), _I32P(), _I32P()]
        _check(lib().sp_plan_branches(self._ptr, *[ctypes.byref(p) for p in ptrs]), "sp_plan_branches")
        names = ["last_seg", "last_row", "round", "recompute"]
        return {k: np.ctypeslib.as_array(p, shape=(nb,)).copy() for k, p in zip(names, ptrs)}


class Cache:
    """Owns an sp_cache*: the radix cache of shared segments over a KV pool of
    n_pages pages, kept across calls.  Host-only; one thread at a time."""

    STAT_NAMES = ("segments", "tokens", "pages_used", "pages_free", "evictions")

    def __init__(self, n_pages: int):
        self._ptr = None
        out = ctypes.c_void_p()
        _check(lib().sp_cache_create(int(n_pages), ctypes.byref(out)), "sp_cache_create")
        self._ptr = out
        self.n_pages = int(n_pages)

    @property
    def ptr(self):
        return self._ptr

    def stats(self) -> dict:
        out = (ctypes.c_int64 * 5)()
        _check(lib().sp_cache_get_stats(self._ptr, out), "sp_cache_get_stats")
        return {k: int(x) for k, x in zip(self.STAT_NAMES, out)}

    def __del__(self):
        try:
            if self._ptr:
                lib().sp_cache_free(self._ptr)
                self._ptr = None
        except Exception:
            pass


class Batcher:
    """Owns an sp_batcher*: the first-in first-out request queue of continuous
    batching and its admission rule (max_batch_tokens node tokens and
    max_batch_requests requests per batch).  Host-only; one thread at a time."""

    def __init__(self, shape: sp_shape, max_batch_tokens: int, max_batch_requests: int):
        self._ptr = None
        self.shape = shape
        out = ctypes.c_void_p()
        _check(lib().sp_batcher_create(ctypes.byref(shape), int(max_batch_tokens),
                                       int(max_batch_requests), ctypes.byref(out)),
               "sp_batcher_create")
        self._ptr = out

    def submit(self, tok_offsets, tokens):
        """Enqueue a request (its branches as a CSR of token ids); returns
        (request id, node tokens)."""
        off = _np(tok_offsets, np.int64)
        tok = _np(tokens, np.int32)
        rid, nt = ctypes.c_int64(), ctypes.c_int64()
        _check(lib().sp_batcher_submit(self._ptr, len(off) - 1, off.ctypes.data_as(_I64P),
                                       tok.ctypes.data_as(_I32P), ctypes.byref(rid),
                                       ctypes.byref(nt)), "sp_batcher_submit")
        return int(rid.value), int(nt.value)

    def pending(self):
        n, t = ctypes.c_int32(), ctypes.c_int64()
        _check(lib().sp_batcher_pending(self._ptr, ctypes.byref(n), ctypes.byref(t)),
               "sp_batcher_pending")
        return int(n.value), int(t.value)

    def next(self, max_pages: int = (1 << 31) - 1, n_sms: int = 0):
        """The next batch: (plan, request ids, branch offsets, row offsets) as
        a Plan and numpy copies, or None when the queue is empty."""
        plan = ctypes.c_void_p()
        n = ctypes.c_int32()
        ids, boff, roff = _I64P(), _I32P(), _I64P()
        _check(lib().sp_batcher_next(self._ptr, int(max_pages), int(n_sms), ctypes.byref(plan),
                                     ctypes.byref(n), ctypes.byref(ids), ctypes.byref(boff),
                                     ctypes.byref(roff)), "sp_batcher_next")
        k = int(n.value)
        if k == 0:
            return None
        return (Plan(plan, self.shape), np.ctypeslib.as_array(ids, (k,)).copy(),
                np.ctypeslib.as_array(boff, (k + 1,)).copy(),
                np.ctypeslib.as_array(roff, (k + 1,)).copy())

    def __del__(self):
        try:
            if self._ptr:
                lib().sp_batcher_free(self._ptr)
                self._ptr = None
        except Exception:
            pass


def make_shape(n_q_heads, n_kv_heads, head_dim, page_size, hidden, vocab) -> sp_shape:
    return sp_shape(n_q_heads, n_kv_heads, head_dim, page_size, hidden, vocab)


def sp_plan_build(shape: sp_shape, req_of_branch, tok_offsets, tokens, max_pages: int,
                  n_sms: int = 0) -> Plan:
    req = _np(req_of_branch, np.int32)
    off = _np(tok_offsets, np.int64)
    tok = _np(tokens, np.int32)
    if len(off) != len(req) + 1:
        raise ValueError("tok_offsets must have n_branches + 1 entries")
    out = ctypes.c_void_p()
    st = lib().sp_plan_build(ctypes.byref(shape), len(req), req.ctypes.data_as(_I32P),
                             off.ctypes.data_as(_I64P), tok.ctypes.data_as(_I32P), int(max_pages),
                             int(n_sms), ctypes.byref(out))
    _check(st, "sp_plan_build")
    return Plan(out, shape)


def sp_plan_build_cached(shape: sp_shape, cache: Cache, req_of_branch, tok_offsets, tokens,
                         n_sms: int = 0) -> Plan:
    req = _np(req_of_branch, np.int32)
    off = _np(tok_offsets, np.int64)
    tok = _np(tokens, np.int32)
    if len(off) != len(req) + 1:
        raise ValueError("tok_offsets must have n_branches + 1 entries")
    out = ctypes.c_void_p()
    st = lib().sp_plan_build_cached(ctypes.byref(shape), cache.ptr, len(req),
                                    req.ctypes.data_as(_I32P), off.ctypes.data_as(_I64P),
                                    tok.ctypes.data_as(_I32P), int(n_sms), ctypes.byref(out))
    _check(st, "sp_plan_build_cached")
    return Plan(out, shape, cache)


def sp_cache_commit(cache: Cache, plan: Plan):
    _check(lib().sp_cache_commit(cache.ptr, plan.ptr), "sp_cache_commit")


def sp_plan_upload(plan: Plan, dev_desc: torch.Tensor, stream=None):
    _check(lib().sp_plan_upload(plan.ptr, _dev(dev_desc, torch.uint8, "dev_desc"),
                                dev_desc.numel(), _stream(stream)), "sp_plan_upload")


def _attn(fn, name, plan, dev_desc, rnd, q, k, v, kv_pool, out, lse, workspace, stream):
    ws_ptr = _dev(workspace, torch.uint8, "workspace") if workspace is not None and workspace.numel() else None
    ws_n = workspace.numel() if workspace is not None else 0
    st = fn(plan.ptr, _dev(dev_desc, torch.uint8, "dev_desc"), int(rnd),
            _dev(q, torch.bfloat16, "q"), _dev(k, torch.bfloat16, "k"), _dev(v, torch.bfloat16, "v"),
            _dev(kv_pool, torch.bfloat16, "kv_pool"), _dev(out, torch.bfloat16, "out"),
            _dev(lse, torch.float32, "lse"), ws_ptr, ws_n, _stream(stream))
    _check(st, name)


def sp_prefix_attn(plan, dev_desc, rnd, q, k, v, kv_pool, out, lse, workspace, stream=None):
    _attn(lib().sp_prefix_attn, "sp_prefix_attn", plan, dev_desc, rnd, q, k, v, kv_pool, out, lse,
          workspace, stream)


def sp_branch_attn(plan, dev_desc, rnd, q, k, v, kv_pool, out, lse, workspace, stream=None):
    _attn(lib().sp_branch_attn, "sp_branch_attn", plan, dev_desc, rnd, q, k, v, kv_pool, out, lse,
          workspace, stream)


def sp_tree_attn(plan, dev_desc, rnd, q, k, v, kv_pool, out, lse, workspace, stream=None):
    _attn(lib().sp_tree_attn, "sp_tree_attn", plan, dev_desc, rnd, q, k, v, kv_pool, out, lse,
          workspace, stream)


def sp_label_workspace_bytes(n_branches: int, vocab: int, n_sms: int = 0) -> int:
    return int(lib().sp_label_workspace_bytes(int(n_branches), int(vocab), int(n_sms)))


def sp_check_labels(label_off, label_ids, vocab: int):
    off = _np(label_off, np.int32)
    ids = _np(label_ids, np.int32)
    _check(lib().sp_check_labels(off.ctypes.data_as(_I32P), ids.ctypes.data_as(_I32P),
                                 len(off) - 1, int(vocab)), "sp_check_labels")


def sp_label_logprobs(h, W, label_off, label_ids, n_labels: int, logprobs, lse, workspace,
                      stream=None):
    N, H = h.shape
    V = W.shape[0]
    if W.shape[1] != H:
        raise ValueError("W must be [V, H] with the hidden size of h")
    st = lib().sp_label_logprobs(
        _dev(h, torch.bfloat16, "h"), _dev(W, torch.bfloat16, "W"), N, H, V,
        _dev(label_off, torch.int32, "label_off"), _dev(label_ids, torch.int32, "label_ids"),
        int(n_labels), _dev(logprobs, torch.float32, "logprobs"), _dev(lse, torch.float32, "lse"),
        _dev(workspace, torch.uint8, "workspace"), workspace.numel(), _stream(stream))
    _check(st, "sp_label_logprobs")


def sp_label_logprobs_noalloc(h, W, label_off, label_ids, n_labels: int, logprobs, lse,
                              stream=None):
    """sp_label_logprobs without a workspace: for callers that cannot allocate
    device memory (the scratch is a static array inside libsp; N <= 1024)."""
    N, H = h.shape
    V = W.shape[0]
    if W.shape[1] != H:
        raise ValueError("W must be [V, H] with the hidden size of h")
    st = lib().sp_label_logprobs_noalloc(
        _dev(h, torch.bfloat16, "h"), _dev(W, torch.bfloat16, "W"), N, H, V,
        _dev(label_off, torch.int32, "label_off"), _dev(label_ids, torch.int32, "label_ids"),
        int(n_labels), _dev(logprobs, torch.float32, "logprobs"), _dev(lse, torch.float32, "lse"),
        _stream(stream))
    _check(st, "sp_label_logprobs_noalloc")


def sp_label_softmax(logprobs, label_off, probs, argmax, stream=None):
    N = label_off.numel() - 1
    st = lib().sp_label_softmax(
        _dev(logprobs, torch.float32, "logprobs"), _dev(label_off, torch.int32, "label_off"), N,
        _dev(probs, torch.float32, "probs"), _dev(argmax, torch.int32, "argmax"), _stream(stream))
    _check(st, "sp_label_softmax")


def sp_label_decide(logprobs, label_off, qtype, probs, argmax, value, confidence, stream=None):
    N = label_off.numel() - 1
    if qtype.numel() != N:
        raise ValueError("qtype must have one entry per branch")
    st = lib().sp_label_decide(
        _dev(logprobs, torch.float32, "logprobs"), _dev(label_off, torch.int32, "label_off"),
        _dev(qtype, torch.int32, "qtype"), N, _dev(probs, torch.float32, "probs"),
        _dev(argmax, torch.int32, "argmax"), _dev(value, torch.float32, "value"),
        _dev(confidence, torch.float32, "confidence"), _stream(stream))
    _check(st, "sp_label_decide")


def sp_option_softmax(row_logprobs, opt_off, q_off, scores, probs, argmax, prior=None,
                      stream=None):
    n_rows = row_logprobs.numel()
    n_opts = opt_off.numel() - 1
    Q = q_off.numel() - 1
    if prior is not None and prior.numel() != n_opts:
        raise ValueError("prior must have one entry per option")
    st = lib().sp_option_softmax(
        _dev(row_logprobs, torch.float32, "row_logprobs"), n_rows,
        _dev(opt_off, torch.int32, "opt_off"), n_opts, _dev(q_off, torch.int32, "q_off"), Q,
        _dev(prior, torch.float32, "prior") if prior is not None else None,
        _dev(scores, torch.float32, "scores"), _dev(probs, torch.float32, "probs"),
        _dev(argmax, torch.int32, "argmax"), _stream(stream))
    _check(st, "sp_option_softmax")


def sp_run_pass(shape: sp_shape, req_of_branch, tok_offsets, tokens, q, k, v, kv_pool, out,
                lse, desc, attn_ws, h, W, label_off, label_ids, logprobs, lse_vocab, lm_ws, probs,
                argmax, stream=None):
    """One whole pass (plan, upload, tree attention, readout, softmax) in one
    call.  Returns (status, plan stats dict): SP_ERR_WORKSPACE and
    SP_ERR_POOL_FULL come back with the stats (nothing launched) so the
    caller can grow its buffers and call again; other errors raise."""
    req = _np(req_of_branch, np.int32)
    off = _np(tok_offsets, np.int64)
    tok = _np(tokens, np.int32)
    st = sp_plan_stats()
    status = lib().sp_run_pass(
        ctypes.byref(shape), len(req), req.ctypes.data_as(_I32P), off.ctypes.data_as(_I64P),
        tok.ctypes.data_as(_I32P), int(q.shape[0]), _dev(q, torch.bfloat16, "q"),
        _dev(k, torch.bfloat16, "k"), _dev(v, torch.bfloat16, "v"),
        _dev(kv_pool, torch.bfloat16, "kv_pool"), int(kv_pool.shape[0]),
        _dev(out, torch.bfloat16, "out"), _dev(lse, torch.float32, "lse"),
        _dev(desc, torch.uint8, "desc"), desc.numel(),
        _dev(attn_ws, torch.uint8, "attn_ws") if attn_ws.numel() else None, attn_ws.numel(),
        _dev(h, torch.bfloat16, "h"), _dev(W, torch.bfloat16, "W"),
        _dev(label_off, torch.int32, "label_off"), _dev(label_ids, torch.int32, "label_ids"),
        label_ids.numel(), _dev(logprobs, torch.float32, "logprobs"),
        _dev(lse_vocab, torch.float32, "lse_vocab"), _dev(lm_ws, torch.uint8, "lm_ws"),
        lm_ws.numel(), _dev(probs, torch.float32, "probs"), _dev(argmax, torch.int32, "argmax"),
        _stream(stream), ctypes.byref(st))
    if status not in (SP_OK, 3, 7):  # SP_ERR_POOL_FULL, SP_ERR_WORKSPACE: the caller grows
        _check(status, "sp_run_pass")
    return status, st.as_dict()


def _host(t: torch.Tensor, dtype, name: str):
    if not isinstance(t, torch.Tensor) or t.device.type != "cpu":
        raise ValueError(f"{name} must be a host tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def sp_run_pass_host(shape: sp_shape, req_of_branch, tok_offsets, tokens, q_host, k_host, v_host,
                     h_host, label_off_host, label_ids_host, in_set: sp_input_set, kv_pool, out,
                     lse, desc, attn_ws, W, logprobs, lse_vocab, lm_ws, probs, argmax, probs_host,
                     argmax_host, stream, copy_stream):
    """sp_run_pass with host inputs and outputs (pinned for asynchronous
    copies), copied through the device input set `in_set`.  Returns (status,
    plan stats dict) as sp_run_pass: SP_ERR_WORKSPACE and SP_ERR_POOL_FULL come
    back with the stats (nothing enqueued); other errors raise."""
    req = _np(req_of_branch, np.int32)
    off = _np(tok_offsets, np.int64)
    tok = _np(tokens, np.int32)
    st = sp_plan_stats()
    status = lib().sp_run_pass_host(
        ctypes.byref(shape), len(req), req.ctypes.data_as(_I32P), off.ctypes.data_as(_I64P),
        tok.ctypes.data_as(_I32P), int(q_host.shape[0]),
        _host(q_host, torch.bfloat16, "q_host"), _host(k_host, torch.bfloat16, "k_host"),
        _host(v_host, torch.bfloat16, "v_host"), _host(h_host, torch.bfloat16, "h_host"),
        _host(label_off_host, torch.int32, "label_off_host"),
        _host(label_ids_host, torch.int32, "label_ids_host"), label_ids_host.numel(),
        ctypes.byref(in_set), _dev(kv_pool, torch.bfloat16, "kv_pool"), int(kv_pool.shape[0]),
        _dev(out, torch.bfloat16, "out"), _dev(lse, torch.float32, "lse"),
        _dev(desc, torch.uint8, "desc"), desc.numel(),
        _dev(attn_ws, torch.uint8, "attn_ws") if attn_ws.numel() else None, attn_ws.numel(),
        _dev(W, torch.bfloat16, "W"), _dev(logprobs, torch.float32, "logprobs"),
        _dev(lse_vocab, torch.float32, "lse_vocab"), _dev(lm_ws, torch.uint8, "lm_ws"),
        lm_ws.numel(), _dev(probs, torch.float32, "probs"), _dev(argmax, torch.int32, "argmax"),
        _host(probs_host, torch.float32, "probs_host"),
        _host(argmax_host, torch.int32, "argmax_host"), _stream(stream), _stream(copy_stream),
        ctypes.byref(st))
    if status not in (SP_OK, 3, 7):  # SP_ERR_POOL_FULL, SP_ERR_WORKSPACE: the caller grows
        _check(status, "sp_run_pass_host")
    return status, st.as_dict()


def sp_check_options(opt_off, n_rows: int, q_off):
    oo = _np(opt_off, np.int32)
    qo = _np(q_off, np.int32)
    _check(lib().sp_check_options(oo.ctypes.data_as(_I32P), len(oo) - 1, int(n_rows),
                                  qo.ctypes.data_as(_I32P), len(qo) - 1), "sp_check_options")


def sp_candidate_decide(probs, label_off, cand_off, qtype, dist, argmax, value, confidence,
                        stream=None):
    n_branches = label_off.numel() - 1
    Q = cand_off.numel() - 1
    if qtype.numel() != Q:
        raise ValueError("qtype must have one entry per question")
    st = lib().sp_candidate_decide(
        _dev(probs, torch.float32, "probs"), _dev(label_off, torch.int32, "label_off"), n_branches,
        _dev(cand_off, torch.int32, "cand_off"), _dev(qtype, torch.int32, "qtype"), Q,
        _dev(dist, torch.float32, "dist"), _dev(argmax, torch.int32, "argmax"),
        _dev(value, torch.float32, "value"), _dev(confidence, torch.float32, "confidence"),
        _stream(stream))
    _check(st, "sp_candidate_decide")


def sp_wait_flag(flag, expect: int, limit_ns: int, stream=None):
    """Bounded device wait until flag[0] == expect (flag: CUDA int32 tensor)."""
    _check(lib().sp_wait_flag(_dev(flag, torch.int32, "flag"), int(expect) & 0xffffffff,
                              int(limit_ns), _stream(stream)), "sp_wait_flag")


def sp_check_device_error(stream=None):
    _check(lib().sp_check_device_error(_stream(stream)), "sp_check_device_error")


def sp_last_launch_count() -> int:
    return int(lib().sp_last_launch_count())
