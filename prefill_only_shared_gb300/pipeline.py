"""One pass of the shared-prefix classifier path through libsp.

``SharedPrefixClassifier.run`` is the call a user makes: it plans the branches
(host trie, rounds, pages), uploads the plan, runs every round's prefix and
branch attention, reads the label log-probabilities out of the LM head and
renormalises them.  It only orchestrates libsp entry points and owns the
device buffers (grow-only, so a steady stream of calls allocates nothing new
after the first); every step of the computation runs in libsp's kernels.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

from . import sp


def _torch_stream(stream, device):
    """A torch stream object for `stream` (None: torch's current stream on
    `device`; a raw cudaStream_t handle is wrapped)."""
    if stream is None:
        return torch.cuda.current_stream(device)
    if isinstance(stream, torch.cuda.Stream):
        return stream
    return torch.cuda.ExternalStream(int(stream), device=device)


@dataclass
class PassOutputs:
    out: torch.Tensor  # bf16 [node_tokens, Hq, d] (device)
    lse: torch.Tensor  # fp32 [node_tokens, Hq]
    logprobs: torch.Tensor  # fp32 [n_labels]
    lse_vocab: torch.Tensor  # fp32 [N]
    probs: torch.Tensor  # fp32 [n_labels]
    argmax: torch.Tensor  # int32 [N]
    plan: "sp.Plan | None"  # None from run_pass (the plan lives inside the native call)
    value: torch.Tensor | None = None  # fp32 [N], with question types
    confidence: torch.Tensor | None = None  # fp32 [N], with question types


class SharedPrefixClassifier:
    def __init__(self, n_q_heads, n_kv_heads, head_dim, hidden, vocab, max_pages=None,
                 device="cuda:0", page_size=16, prefix_cache_pages=None):
        """``max_pages``: fixed KV pool capacity (plans that need more fail
        with SP_ERR_POOL_FULL); None grows the pool to what each plan needs.

        ``prefix_cache_pages``: keep the shared segments that calls compute in
        a radix cache over a fixed pool of that many pages (it replaces
        ``max_pages``), so later calls compute only their uncached remainders
        (repeated state, hot requests).  A plan is then committed to the cache
        when its attention is enqueued; all calls must use one stream, since
        pages freed by one plan are written by the next."""
        self.shape = sp.make_shape(n_q_heads, n_kv_heads, head_dim, page_size, hidden, vocab)
        self.device = torch.device(device)
        self.cache = None
        if prefix_cache_pages is not None:
            self.cache = sp.Cache(int(prefix_cache_pages))
            max_pages = int(prefix_cache_pages)
        self.fixed_pool = max_pages is not None
        self.n_sms = torch.cuda.get_device_properties(self.device).multi_processor_count
        # SMs the planner sizes attention calls for (splits of small calls,
        # pairing of leaf tails); the device's count unless set
        self.plan_sms = None
        self._bufs = {}
        self._views = {}
        self._lm_ws_key = None
        self._lm_ws_bytes = 0
        self.kv_pool = None
        self._ensure_pool(int(max_pages) if max_pages is not None else 0)

    def _ensure_pool(self, pages):
        if self.kv_pool is not None and self.kv_pool.shape[0] >= pages:
            return
        s = self.shape
        if self.kv_pool is not None:
            # passes enqueued on other streams may still read the old pool:
            # let them finish before its memory can be handed out again
            torch.cuda.synchronize(self.device)
        self.kv_pool = torch.empty((max(pages, 1), 2, s.n_kv_heads, s.page_size, s.head_dim),
                                   dtype=torch.bfloat16, device=self.device)

    @property
    def max_pages(self):
        return self.kv_pool.shape[0] if self.fixed_pool else (1 << 31) - 1

    def _buf(self, name, numel, dtype):
        """A view of `numel` elements of the grow-only buffer `name` (views are
        reused while the buffer stays)."""
        key = (name, int(numel), dtype)
        view = self._views.get(key)
        if view is not None:
            return view
        b = self._bufs.get(name)
        if b is None or b.numel() < numel or b.dtype != dtype:
            if b is not None:  # as for the pool: the old buffer's readers finish first
                torch.cuda.synchronize(self.device)
            b = torch.empty(max(int(numel), 1), dtype=dtype, device=self.device)
            self._bufs[name] = b
            self._views = {k: v for k, v in self._views.items() if k[0] != name}
        view = b[:max(int(numel), 1)] if numel else b[:0]
        self._views[key] = view
        return view

    def _stream(self, stream):
        """Raw cudaStream_t of `stream` (None: torch's current stream)."""
        if stream is None:
            return torch.cuda.current_stream(self.device).cuda_stream
        if isinstance(stream, torch.cuda.Stream):
            return stream.cuda_stream
        return int(stream)

    def plan(self, req_of_branch, tok_offsets, tokens) -> "sp.Plan":
        """The plan of one call.  With a prefix cache it covers only the
        uncached remainders: q / k / v rows exist for those alone."""
        if self.cache is not None:
            return sp.sp_plan_build_cached(self.shape, self.cache, req_of_branch, tok_offsets,
                                           tokens, self.plan_sms or self.n_sms)
        plan = sp.sp_plan_build(self.shape, req_of_branch, tok_offsets, tokens, self.max_pages,
                                self.plan_sms or self.n_sms)
        self._ensure_pool(plan.stats()["pages_used"])
        return plan

    def attention(self, plan, q, k, v, stream=None, schedule="rounds", out=None, lse=None):
        """schedule "rounds": one prefix and one branch call per staged round,
        in round order; "all": one prefix call and one branch call covering
        every round; "tree": one call for the whole trie.  Same results,
        fewer launches.  out / lse: the caller's output tensors ([node
        tokens, Hq, d] bf16, [node tokens, Hq] fp32), else the classifier's
        own buffers."""
        stream = self._stream(stream)
        st = plan.stats()
        T = st["node_tokens"]
        Hq, d = self.shape.n_q_heads, self.shape.head_dim
        desc = self._desc_view(st["desc_bytes"])
        sp.sp_plan_upload(plan, desc, stream)
        ws = self._buf("attn_ws", st["attn_workspace_bytes"], torch.uint8)
        if out is None:
            out = self._buf("out", T * Hq * d, torch.bfloat16).view(T, Hq, d)
        if lse is None:
            lse = self._buf("lse", T * Hq, torch.float32).view(T, Hq)
        launches = 0
        if schedule == "tree":
            sp.sp_tree_attn(plan, desc, sp.SP_ALL_ROUNDS, q, k, v, self.kv_pool, out, lse, ws,
                            stream)
            launches += sp.sp_last_launch_count()
        else:
            if schedule not in ("rounds", "all"):
                raise ValueError(f"unknown schedule {schedule!r}")
            rounds = range(st["n_rounds"]) if schedule == "rounds" else [sp.SP_ALL_ROUNDS]
            for r in rounds:
                sp.sp_prefix_attn(plan, desc, r, q, k, v, self.kv_pool, out, lse, ws, stream)
                launches += sp.sp_last_launch_count()
                sp.sp_branch_attn(plan, desc, r, q, k, v, self.kv_pool, out, lse, ws, stream)
                launches += sp.sp_last_launch_count()
        self.last_attention_launches = launches
        if plan.cache is not None:  # later plans on this stream may read its segments
            sp.sp_cache_commit(plan.cache, plan)
        return out, lse

    def _desc_view(self, nbytes):
        """A 256-byte-aligned device view of `nbytes` for the plan descriptor."""
        key = ("desc", -int(nbytes), "aligned")  # dropped with the "desc" buffer
        view = self._views.get(key)
        if view is None:
            raw = self._buf("desc", nbytes + 256, torch.uint8)
            off = (-raw.data_ptr()) % 256
            view = raw[off:off + nbytes]
            self._views[key] = view
        return view

    def logprobs(self, h, W, label_off, label_ids, n_labels, stream=None):
        stream = self._stream(stream)
        N = h.shape[0]
        wkey = (N, W.shape[0])
        if self._lm_ws_key != wkey:
            self._lm_ws_bytes = sp.sp_label_workspace_bytes(N, W.shape[0], self.n_sms)
            self._lm_ws_key = wkey
        ws = self._buf("lm_ws", self._lm_ws_bytes, torch.uint8)
        logprobs = self._buf("logprobs", n_labels, torch.float32)
        lse = self._buf("lse_vocab", N, torch.float32)
        sp.sp_label_logprobs(h, W, label_off, label_ids, n_labels, logprobs, lse, ws, stream)
        self.last_logprob_launches = sp.sp_last_launch_count()
        return logprobs, lse

    def softmax(self, logprobs, label_off, stream=None):
        stream = self._stream(stream)
        N = label_off.numel() - 1
        probs = self._buf("probs", logprobs.numel(), torch.float32)
        argmax = self._buf("argmax", N, torch.int32)
        sp.sp_label_softmax(logprobs, label_off, probs, argmax, stream)
        self.last_softmax_launches = sp.sp_last_launch_count()
        return probs, argmax

    def decide(self, logprobs, label_off, qtype, stream=None):
        """One question per branch, its options the branch's labels: label
        softmax fused with the question type's value and the confidence.
        Returns (probs, argmax, value, confidence)."""
        stream = self._stream(stream)
        N = label_off.numel() - 1
        probs = self._buf("probs", logprobs.numel(), torch.float32)
        argmax = self._buf("argmax", N, torch.int32)
        value = self._buf("value", N, torch.float32)
        conf = self._buf("confidence", N, torch.float32)
        sp.sp_label_decide(logprobs, label_off, qtype, probs, argmax, value, conf, stream)
        self.last_softmax_launches = sp.sp_last_launch_count()
        return probs, argmax, value, conf

    def candidates(self, probs, label_off, cand_off, qtype, stream=None):
        """Questions assembled from yes/no candidate branches (consecutive
        branches per question).  Returns (dist, argmax, value, confidence)."""
        stream = self._stream(stream)
        Q = cand_off.numel() - 1
        dist = self._buf("dist", label_off.numel() - 1, torch.float32)  # >= cand_off[-1]
        argmax = self._buf("q_argmax", Q, torch.int32)
        value = self._buf("q_value", Q, torch.float32)
        conf = self._buf("q_confidence", Q, torch.float32)
        sp.sp_candidate_decide(probs, label_off, cand_off, qtype, dist, argmax, value, conf, stream)
        self.last_candidate_launches = sp.sp_last_launch_count()
        return dist, argmax, value, conf

    def options(self, h_rows, W, opt_off, opt_tokens, q_off, prior=None, stream=None):
        """Multi-token options: the readout with one label per row (each
        option token at the position before it), then the option scores and
        their (optionally prior-calibrated) softmax per question.  Returns
        (row_logprobs, scores, probs, argmax)."""
        stream = self._stream(stream)
        n_rows = h_rows.shape[0]
        row_off = self._buf("row_off", n_rows + 1, torch.int32)
        if not getattr(self, "_row_off_n", None) == n_rows:
            row_off.copy_(torch.arange(n_rows + 1, dtype=torch.int32))  # host index, copied
            self._row_off_n = n_rows
        lp, _ = self.logprobs(h_rows, W, row_off, opt_tokens, n_rows, stream)
        n_opts = opt_off.numel() - 1
        scores = self._buf("opt_scores", n_opts, torch.float32)
        probs = self._buf("opt_probs", n_opts, torch.float32)
        argmax = self._buf("opt_argmax", q_off.numel() - 1, torch.int32)
        sp.sp_option_softmax(lp, opt_off, q_off, scores, probs, argmax, prior, stream)
        self.last_option_launches = self.last_logprob_launches + sp.sp_last_launch_count()
        return lp, scores, probs, argmax

    def readout(self, h, W, label_off, label_ids, n_labels, stream=None, qtype=None):
        """LM-head label log-probabilities, then the label softmax; with
        ``qtype`` (device int32 [N]) the softmax is the fused decision and the
        value / confidence are returned too (else None)."""
        stream = self._stream(stream)
        logprobs, lse = self.logprobs(h, W, label_off, label_ids, n_labels, stream)
        value = conf = None
        if qtype is None:
            probs, argmax = self.softmax(logprobs, label_off, stream)
        else:
            probs, argmax, value, conf = self.decide(logprobs, label_off, qtype, stream)
        self.last_readout_launches = self.last_logprob_launches + self.last_softmax_launches
        return logprobs, lse, probs, argmax, value, conf

    def run(self, req_of_branch, tok_offsets, tokens, q, k, v, h, W, label_off, label_ids,
            stream=None, schedule="rounds", qtype=None) -> PassOutputs:
        """q/k/v in node-token order of the plan (see sp_plan_segments)."""
        stream = self._stream(stream)
        plan = self.plan(req_of_branch, tok_offsets, tokens)
        out, lse = self.attention(plan, q, k, v, stream, schedule)
        n_labels = int(label_ids.numel())
        logprobs, lse_v, probs, argmax, value, conf = self.readout(
            h, W, label_off, label_ids, n_labels, stream, qtype)
        return PassOutputs(out, lse, logprobs, lse_v, probs, argmax, plan, value, conf)

    def _pass_outputs(self, T, N, nl, W):
        """Output and readout buffers of a whole pass: T node rows, N branches,
        nl labels."""
        s = self.shape
        out = self._buf("out", T * s.n_q_heads * s.head_dim, torch.bfloat16).view(
            T, s.n_q_heads, s.head_dim)
        lse = self._buf("lse", T * s.n_q_heads, torch.float32).view(T, s.n_q_heads)
        logprobs = self._buf("logprobs", nl, torch.float32)
        lse_v = self._buf("lse_vocab", N, torch.float32)
        probs = self._buf("probs", nl, torch.float32)
        argmax = self._buf("argmax", N, torch.int32)
        wkey = (N, W.shape[0])
        if self._lm_ws_key != wkey:
            self._lm_ws_bytes = sp.sp_label_workspace_bytes(N, W.shape[0], self.n_sms)
            self._lm_ws_key = wkey
        lm_ws = self._buf("lm_ws", self._lm_ws_bytes, torch.uint8)
        if not hasattr(self, "_pass_need"):
            self._pass_need = {"desc_bytes": 4096, "attn_workspace_bytes": 0}
        return out, lse, logprobs, lse_v, probs, argmax, lm_ws

    def _grow_pass_needs(self, status, st, where):
        """After SP_ERR_WORKSPACE / SP_ERR_POOL_FULL from a whole-pass call:
        grow the descriptor, workspace and pool sizes to what it reported."""
        need = self._pass_need
        need["desc_bytes"] = max(need["desc_bytes"], st["desc_bytes"])
        need["attn_workspace_bytes"] = max(need["attn_workspace_bytes"], st["attn_workspace_bytes"])
        if status == 3:  # SP_ERR_POOL_FULL
            if self.fixed_pool:
                raise sp.SpError(status, where)
            self._ensure_pool(st["pages_used"])

    def run_pass(self, req_of_branch, tok_offsets, tokens, q, k, v, h, W, label_off, label_ids,
                 stream=None) -> PassOutputs:
        """The whole pass in one native call (sp_run_pass: plan, upload, one
        tree attention call, readout, softmax), so the host work is the C++
        planner's.  Buffers grow when the call reports SP_ERR_WORKSPACE or
        SP_ERR_POOL_FULL (nothing is launched then) and the call is repeated.
        Not with a prefix cache (its plans come from sp_plan_build_cached)."""
        if self.cache is not None:
            raise ValueError("run_pass plans without the prefix cache")
        stream = self._stream(stream)
        out, lse, logprobs, lse_v, probs, argmax, lm_ws = self._pass_outputs(
            int(q.shape[0]), int(h.shape[0]), int(label_ids.numel()), W)
        for _ in range(3):
            need = self._pass_need
            desc = self._desc_view(need["desc_bytes"])
            ws = self._buf("attn_ws", need["attn_workspace_bytes"], torch.uint8)
            status, st = sp.sp_run_pass(self.shape, req_of_branch, tok_offsets, tokens, q, k, v,
                                        self.kv_pool, out, lse, desc, ws, h, W, label_off,
                                        label_ids, logprobs, lse_v, lm_ws, probs, argmax, stream)
            if status == sp.SP_OK:
                break
            self._grow_pass_needs(status, st, "sp_run_pass")
        else:
            raise sp.SpError(status, "sp_run_pass")
        self.last_pass_launches = sp.sp_last_launch_count()
        return PassOutputs(out, lse, logprobs, lse_v, probs, argmax, None)

    def run_from_host(self, req_of_branch, tok_offsets, tokens, q, k, v, h, W, label_off,
                      label_ids, probs_out, argmax_out, stream=None, schedule="rounds",
                      qtype=None) -> PassOutputs:
        """``run`` with the inputs in host memory: q, k, v, h, label_off and
        label_ids (pinned, for asynchronous copies) are copied in on a side
        stream into the next of two device input sets, so this call's copies
        overlap the previous call's kernels; the pass runs on `stream` once
        its copies are done, and its probabilities and argmax are copied out
        into probs_out / argmax_out (pinned host tensors).  Asynchronous:
        synchronise `stream` before reading the outputs.  W stays on the
        device (model state).  The tree schedule without question types or a
        prefix cache is one native call (sp_run_pass_host: copies, pass and
        read-back); the other forms copy through torch and call ``run``."""
        st = _torch_stream(stream, self.device)
        cs = self.copy_stream
        i = self._in_next
        self._in_next ^= 1
        srcs = {"q": q, "k": k, "v": v, "h": h, "label_off": label_off, "label_ids": label_ids}
        self._grow_input_set(i, srcs)
        if schedule == "tree" and qtype is None and self.cache is None:
            return self._run_pass_host(i, req_of_branch, tok_offsets, tokens, srcs, W, probs_out,
                                       argmax_out, st, cs)
        dev_in = self._in_sets[i]
        cs.wait_event(self._in_done[i])  # the pass that read this set is done
        views = {}
        with torch.cuda.stream(cs):
            for name, src in srcs.items():
                view = dev_in[name][:src.numel()].view(src.shape)
                view.copy_(src, non_blocking=True)
                views[name] = view
            self._in_copied[i].record(cs)
        st.wait_event(self._in_copied[i])
        res = self.run(req_of_branch, tok_offsets, tokens, views["q"], views["k"], views["v"],
                       views["h"], W, views["label_off"], views["label_ids"], st.cuda_stream,
                       schedule, qtype)
        with torch.cuda.stream(st):
            probs_out.copy_(res.probs, non_blocking=True)
            argmax_out.copy_(res.argmax, non_blocking=True)
            self._in_done[i].record(st)
        return res

    def _grow_input_set(self, i, srcs):
        """Grow device input set i to hold `srcs`; a buffer is replaced only
        after the last pass that read the set has finished."""
        dev_in = self._in_sets[i]
        for name, src in srcs.items():
            d = dev_in.get(name)
            if d is None or d.numel() < src.numel() or d.dtype != src.dtype:
                self._in_done[i].synchronize()
                dev_in[name] = torch.empty(max(src.numel(), 1), dtype=src.dtype,
                                           device=self.device)
                self._in_struct[i] = None

    def _input_struct(self, i, desc_bytes):
        """The sp_input_set of device input set i, with at least desc_bytes of
        pinned descriptor staging."""
        c = self._in_struct[i]
        if c is not None and c.desc_host_bytes >= desc_bytes:
            return c
        dh = self._in_desc_host[i]
        if dh is None or dh.numel() < desc_bytes:
            self._in_done[i].synchronize()  # its last upload has run
            dh = torch.empty(int(desc_bytes), dtype=torch.uint8).pin_memory()
            self._in_desc_host[i] = dh
        d, s = self._in_sets[i], self.shape
        rows = min(d["q"].numel() // (s.n_q_heads * s.head_dim),
                   d["k"].numel() // (s.n_kv_heads * s.head_dim),
                   d["v"].numel() // (s.n_kv_heads * s.head_dim))
        c = sp.sp_input_set(
            q=d["q"].data_ptr(), k=d["k"].data_ptr(), v=d["v"].data_ptr(), h=d["h"].data_ptr(),
            label_off=d["label_off"].data_ptr(), label_ids=d["label_ids"].data_ptr(),
            q_rows=rows, h_rows=min(d["h"].numel() // s.hidden, d["label_off"].numel() - 1),
            labels_cap=d["label_ids"].numel(), desc_host=dh.data_ptr(),
            desc_host_bytes=dh.numel(), done_event=self._in_done[i].cuda_event,
            copied_event=self._in_copied[i].cuda_event)
        self._in_struct[i] = c
        return c

    def _run_pass_host(self, i, req_of_branch, tok_offsets, tokens, srcs, W, probs_out,
                       argmax_out, st, cs) -> PassOutputs:
        s = self.shape
        q, k, v, h = srcs["q"], srcs["k"], srcs["v"], srcs["h"]
        T, N = int(q.shape[0]), int(h.shape[0])
        if (q.numel() != T * s.n_q_heads * s.head_dim or k.numel() != T * s.n_kv_heads * s.head_dim
                or v.numel() != k.numel() or h.numel() != N * s.hidden
                or srcs["label_off"].numel() != N + 1 or probs_out.numel() < srcs["label_ids"].numel()
                or argmax_out.numel() < N):
            raise ValueError("host inputs / outputs do not match the model shape")
        out, lse, logprobs, lse_v, probs, argmax, lm_ws = self._pass_outputs(
            T, N, int(srcs["label_ids"].numel()), W)
        for _ in range(3):
            need = self._pass_need
            desc = self._desc_view(need["desc_bytes"])
            ws = self._buf("attn_ws", need["attn_workspace_bytes"], torch.uint8)
            iset = self._input_struct(i, need["desc_bytes"])
            status, stt = sp.sp_run_pass_host(
                s, req_of_branch, tok_offsets, tokens, q, k, v, h, srcs["label_off"],
                srcs["label_ids"], iset, self.kv_pool, out, lse, desc, ws, W, logprobs, lse_v,
                lm_ws, probs, argmax, probs_out, argmax_out, st.cuda_stream, cs.cuda_stream)
            if status == sp.SP_OK:
                break
            self._grow_pass_needs(status, stt, "sp_run_pass_host")
        else:
            raise sp.SpError(status, "sp_run_pass_host")
        self.last_pass_launches = sp.sp_last_launch_count()
        return PassOutputs(out, lse, logprobs, lse_v, probs, argmax, None)

    @property
    def copy_stream(self) -> torch.cuda.Stream:
        """The side stream run_from_host copies inputs on (created on first use)."""
        if getattr(self, "_copy_stream", None) is None:
            cs = torch.cuda.Stream(self.device)
            self._in_sets = [{}, {}]
            self._in_struct = [None, None]
            self._in_desc_host = [None, None]
            self._in_next = 0
            # per set: done (its last pass has finished) and copied (its
            # inputs are in); recorded once here so that each has a CUDA event
            self._in_done = [torch.cuda.Event(), torch.cuda.Event()]
            self._in_copied = [torch.cuda.Event(), torch.cuda.Event()]
            for e in self._in_done + self._in_copied:
                e.record(cs)
            self._copy_stream = cs
        return self._copy_stream

    @property
    def last_launches(self) -> int:
        return (getattr(self, "last_attention_launches", 0) + getattr(self, "last_logprob_launches", 0)
                + getattr(self, "last_softmax_launches", 0))


@dataclass
class _Req:
    row0: int
    n_rows: int
    br0: int
    n_br: int
    lab0: int
    label_off: np.ndarray  # the request's own label CSR offsets (from 0)


class ContinuousBatcher:
    """Continuous batching of independent requests over one classifier.

    Requests are queued first-in first-out by a native batcher (include/sp.h,
    sp_batcher_*): each batch takes requests from the head of the queue while
    its node tokens stay within ``max_batch_tokens`` and its size within
    ``max_batch_requests``, and gets one plan, one attention call and one
    readout for all its requests.  Requests never share K/V, so a request's
    results do not depend on its batch; what batching saves is the LM head,
    streamed once per batch instead of once per request, and attention grids
    that fill the GPU.

    ``submit`` stores a request's inputs right after the previous request's in
    device arenas sized at construction (its q / k / v rows in the node-token
    order of its own plan, its final hidden states, its label ids), so a batch
    of consecutive requests reads one contiguous slice of each: nothing is
    gathered.  ``run`` forms and enqueues the batches on one stream; planning a
    batch on the host overlaps the GPU's work on the previous one.  Results
    stay in the arenas until ``reset``.
    """

    def __init__(self, clf: SharedPrefixClassifier, W, max_batch_tokens: int,
                 max_batch_requests: int = 64, capacity_rows: int = 1 << 15,
                 capacity_branches: int = 4096, capacity_labels: int = 1 << 16,
                 schedule: str = "tree"):
        if clf.cache is not None:
            raise ValueError("continuous batching plans without a prefix cache: use a classifier "
                             "built without prefix_cache_pages")
        s = clf.shape
        dev = clf.device
        self.clf, self.W, self.schedule = clf, W, schedule
        self._live_plans = []
        self.batcher = sp.Batcher(s, max_batch_tokens, max_batch_requests)
        self.q = torch.empty(capacity_rows, s.n_q_heads, s.head_dim, dtype=torch.bfloat16, device=dev)
        self.k = torch.empty(capacity_rows, s.n_kv_heads, s.head_dim, dtype=torch.bfloat16, device=dev)
        self.v = torch.empty_like(self.k)
        self.out = torch.empty_like(self.q)
        self.lse = torch.empty(capacity_rows, s.n_q_heads, dtype=torch.float32, device=dev)
        self.h = torch.empty(capacity_branches, s.hidden, dtype=torch.bfloat16, device=dev)
        self.label_ids = torch.empty(capacity_labels, dtype=torch.int32, device=dev)
        self.logprobs = torch.empty(capacity_labels, dtype=torch.float32, device=dev)
        self.probs = torch.empty(capacity_labels, dtype=torch.float32, device=dev)
        self.lse_vocab = torch.empty(capacity_branches, dtype=torch.float32, device=dev)
        self.argmax = torch.empty(capacity_branches, dtype=torch.int32, device=dev)
        # batch label offsets: a small ring of pinned host slots and device
        # copies, a slot reused only once its last copy has completed
        self._ring = [(torch.empty(capacity_branches + 1, dtype=torch.int32).pin_memory(),
                       torch.empty(capacity_branches + 1, dtype=torch.int32, device=dev),
                       torch.cuda.Event()) for _ in range(4)]
        self._ring_used = [False] * 4
        self._n_batches = 0
        self.reset()

    def reset(self):
        """Forget every request and result (call with nothing in flight)."""
        self._reqs = {}
        self._rows = self._brs = self._labs = 0
        self.batch_sizes = []

    def submit(self, tok_offsets, tokens, q, k, v, h, label_off, label_ids, stream=None):
        """Queue one request: its branches as a CSR of token ids (host), its
        q / k / v rows in the node-token order of its own plan, its final
        hidden states [branches, H] and its label CSR (host offsets, ids).
        The tensors may live on the host (pinned for an asynchronous copy) or
        on the device.  Returns the request id."""
        rid, nt = self.batcher.submit(tok_offsets, tokens)
        off = np.asarray(label_off, dtype=np.int64)
        nb, nl = len(off) - 1, int(off[-1])
        if q.shape[0] != nt or k.shape[0] != nt or v.shape[0] != nt or h.shape[0] != nb:
            raise ValueError("q/k/v need one row per node token, h one row per branch")
        if (self._rows + nt > self.q.shape[0] or self._brs + nb > self.h.shape[0]
                or self._labs + nl > self.label_ids.shape[0]):
            raise ValueError("ContinuousBatcher arenas are full: reset() or raise the capacities")
        st = _torch_stream(stream, self.clf.device)
        with torch.cuda.stream(st):
            r0, b0, l0 = self._rows, self._brs, self._labs
            self.q[r0:r0 + nt].copy_(q, non_blocking=True)
            self.k[r0:r0 + nt].copy_(k, non_blocking=True)
            self.v[r0:r0 + nt].copy_(v, non_blocking=True)
            self.h[b0:b0 + nb].copy_(h, non_blocking=True)
            self.label_ids[l0:l0 + nl].copy_(torch.as_tensor(np.asarray(label_ids, np.int32)),
                                             non_blocking=True)
        self._reqs[rid] = _Req(r0, nt, b0, nb, l0, off)
        self._rows, self._brs, self._labs = r0 + nt, b0 + nb, l0 + nl
        return rid

    def run(self, stream=None) -> int:
        """Form and enqueue every batch of the queue on `stream`; returns the
        number of batches.  Asynchronous: synchronise before reading results."""
        st = _torch_stream(stream, self.clf.device)
        raw = st.cuda_stream
        clf = self.clf
        V = self.W.shape[0]
        n = 0
        while True:
            # planning here overlaps the GPU's work on the previous batch
            nxt = self.batcher.next(clf.max_pages, clf.n_sms)
            if nxt is None:
                break
            plan, ids, boff, roff = nxt
            first = self._reqs[int(ids[0])]
            for i, rid in enumerate(ids):  # consecutive requests, consecutive rows
                r = self._reqs[int(rid)]
                if r.row0 != first.row0 + roff[i] or r.br0 != first.br0 + boff[i]:
                    raise RuntimeError("batch requests are not stored consecutively")
            if not clf.fixed_pool:
                clf._ensure_pool(plan.stats()["pages_used"])
            rows = slice(first.row0, first.row0 + int(roff[-1]))
            nb = int(boff[-1])
            brs = slice(first.br0, first.br0 + nb)
            clf.attention(plan, self.q[rows], self.k[rows], self.v[rows], raw, self.schedule,
                          self.out[rows], self.lse[rows])
            # the batch's label CSR, offsets from 0
            offs = [0]
            for rid in ids:
                o = self._reqs[int(rid)].label_off
                offs.extend((offs[-1] + o[1:]).tolist())
            nl = offs[-1]
            slot = self._n_batches % len(self._ring)
            host, dev_off, ev = self._ring[slot]
            if self._ring_used[slot]:
                ev.synchronize()  # the slot's previous copy has been read
            host[:nb + 1].numpy()[:] = np.asarray(offs, dtype=np.int32)
            with torch.cuda.stream(st):
                dev_off[:nb + 1].copy_(host[:nb + 1], non_blocking=True)
                ev.record(st)
            self._ring_used[slot] = True
            labs = slice(first.lab0, first.lab0 + nl)
            ws = clf._buf("lm_ws", sp.sp_label_workspace_bytes(nb, V, clf.n_sms), torch.uint8)
            sp.sp_label_logprobs(self.h[brs], self.W, dev_off[:nb + 1], self.label_ids[labs], nl,
                                 self.logprobs[labs], self.lse_vocab[brs], ws, raw)
            sp.sp_label_softmax(self.logprobs[labs], dev_off[:nb + 1], self.probs[labs],
                                self.argmax[brs], raw)
            self.batch_sizes.append(len(ids))
            self._n_batches += 1
            n += 1
            # the plan's descriptor is copied on the stream from the plan's host
            # memory: keep the plan until the batch's work has passed that copy
            done = torch.cuda.Event()
            done.record(st)
            self._live_plans = [(p, e) for p, e in self._live_plans if not e.query()]
            self._live_plans.append((plan, done))
        return n

    def result(self, rid: int) -> dict:
        """A request's outputs as views of the device arenas: attention out /
        lse (its node rows, in its own plan's node-token order), label
        log-probabilities, vocabulary lse, probabilities and argmax."""
        r = self._reqs[rid]
        nl = int(r.label_off[-1])
        rows = slice(r.row0, r.row0 + r.n_rows)
        labs = slice(r.lab0, r.lab0 + nl)
        brs = slice(r.br0, r.br0 + r.n_br)
        return {"out": self.out[rows], "lse": self.lse[rows], "logprobs": self.logprobs[labs],
                "lse_vocab": self.lse_vocab[brs], "probs": self.probs[labs],
                "argmax": self.argmax[brs]}
