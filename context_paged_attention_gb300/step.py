"""One attention step over a striped pool, orchestrated through the C ABI.

A decode step (one new token a row) is: ``cp_kv_write`` of the new K/V, then
``cp_paged_attn_partial`` over each row's full length, then ``lse_merge`` of
the P partner partials.  A non-decode step attends the pool for the context
only and its new tokens apart: ``cp_kv_write``, ``cp_paged_attn_partial``
(kv_len = context), ``own_token_attn``, then ``lse_merge`` of P + 1 partials
(mstar PR #1124 "Context / Sequence Parallel 1/5", description; vLLM "[Core]
Add explicit layer parallel plans", _forward_with_dcp).

This module only allocates device buffers and sequences the library calls;
all arithmetic runs in libcpattn.
"""

from __future__ import annotations

import numpy as np
import torch

from . import binding as B


def _to_torch(a: np.ndarray, device) -> torch.Tensor:
    """Host array -> device tensor; uint16 arrays are bfloat16 bit patterns."""
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def desc_for(w) -> B.PoolDesc:
    fp8 = getattr(w, "kv_dtype", "same") == "fp8"
    return B.PoolDesc(P=w.P, page_size=w.page_size, num_pages=w.num_pages, num_kv_heads=w.num_kv_heads,
                      head_dim=w.head_dim, head_dim_v=w.head_dim_v,
                      dtype=B.DTYPE_BF16 if w.dtype == "bf16" else B.DTYPE_FP32,
                      interleave=w.interleave, kv_dtype=B.DTYPE_FP8_E4M3 if fp8 else 0,
                      k_descale=w.k_descale if fp8 else 0.0, v_descale=w.v_descale if fp8 else 0.0)


def pack_tensors(tensors, device, align=256):
    """One uint8 buffer on ``device`` holding copies of ``tensors`` at
    ``align``-byte offsets, and views of it with each tensor's dtype and shape
    (in order).  Empty tensors get empty views."""
    offs, end = [], 0
    for t in tensors:
        end = (end + align - 1) // align * align
        offs.append(end)
        end += t.numel() * t.element_size()
    buf = torch.empty((max(end, align),), dtype=torch.uint8, device=device)
    views = []
    for t, o in zip(tensors, offs):
        v = buf[o: o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
        v.copy_(t)
        views.append(v)
    return buf, views


class StripedAttention:
    """Device state of one workload: the striped pool, the step's inputs and outputs.

    ``w`` is a ``workloads.Workload``.  The pool is filled with NaN (so any read
    of an unwritten slot would surface) and then with every row's context
    through ``cp_kv_write``; ``run_step`` then performs the step.
    """

    def __init__(self, w, device="cuda", fill_history=True, out_dtype=None):
        self.w = w
        self.device = torch.device(device)
        self.desc = desc_for(w)
        dt = self.desc.torch_dtype()
        pdt = self.desc.pool_torch_dtype()
        nan = B.FP8_NAN_CODE if self.desc.fp8 else float("nan")
        self.pool_k = torch.full(self.desc.pool_shape(False), nan, dtype=pdt, device=self.device)
        self.pool_v = None if w.mla else torch.full(self.desc.pool_shape(True), nan, dtype=pdt, device=self.device)
        self.dev_status = torch.zeros(1, dtype=torch.int32, device=self.device)
        # step inputs
        self.q = _to_torch(w.q, self.device)
        self.k_new = _to_torch(w.k_new, self.device)
        self.v_new = None if w.v_new is None else _to_torch(w.v_new, self.device)
        self.positions = _to_torch(w.positions, self.device)
        self.qo_indptr = _to_torch(w.qo_indptr, self.device)
        self.kv_len = _to_torch(w.kv_len, self.device)
        self.page_indptr = _to_torch(w.kv_page_indptr, self.device)
        self.page_indices = _to_torch(w.kv_page_indices, self.device)
        self.max_kv_len = int(max(1, w.kv_len.max(initial=0)))
        self.max_q_len = int(w.new_len.max(initial=0))
        # outputs
        T, Hq, Dv, P = w.num_tokens, w.num_q_heads, w.head_dim_v, w.P
        nparts = P if w.decode else P + 1
        self.o_parts = torch.empty((nparts, T, Hq, Dv), dtype=torch.float32, device=self.device)
        self.lse_parts = torch.empty((nparts, T, Hq), dtype=torch.float32, device=self.device)
        odt = out_dtype if out_dtype is not None else dt
        self.out = torch.empty((T, Hq, Dv), dtype=odt, device=self.device)
        self.lse = torch.empty((T, Hq), dtype=torch.float32, device=self.device)
        ws = B.workspace_bytes(self.desc, Hq, T, self.max_kv_len)
        self.workspace = torch.empty((max(ws, 256),), dtype=torch.uint8, device=self.device)
        self._fused_ws = None
        self.graph = None
        # dispatch order of the rows: longest first (the host knows the lengths)
        order = np.argsort(-w.kv_len.astype(np.int64), kind="stable").astype(np.int32)
        self.row_order = _to_torch(order, self.device)
        # the step's inputs and outputs as views into one buffer each, so that
        # a caller feeding the step from host memory makes one copy in and one
        # copy out a step (``packed_inputs`` / ``packed_outputs``)
        self.packed_inputs = self._pack(self.INPUTS)
        self.packed_outputs = self._pack(("out", "lse"))
        if fill_history:
            self.fill_history()

    # per-step inputs, in the order they are packed
    INPUTS = ("q", "k_new", "v_new", "positions", "qo_indptr", "kv_len", "page_indptr", "page_indices", "row_order")

    def _pack(self, names):
        """Move the named tensors into one device buffer and rebind them to
        views of it; returns the buffer."""
        items = [(n, getattr(self, n)) for n in names if getattr(self, n) is not None]
        buf, views = pack_tensors([t for _, t in items], self.device)
        for (n, _), v in zip(items, views):
            setattr(self, n, v)
        return buf

    def fill_history(self):
        """Write every real row's context (positions 0 .. ctx-1) through cp_kv_write."""
        from .workloads import history_tokens

        qo, pos, k, v = history_tokens(self.w)
        if len(pos) == 0:
            return
        B.cp_kv_write(self.desc, self.pool_k, self.pool_v, _to_torch(k, self.device),
                      None if v is None else _to_torch(v, self.device), _to_torch(pos, self.device),
                      _to_torch(qo, self.device), self.page_indptr, self.page_indices, dev_status=self.dev_status)

    # -- the step's calls
    def write_new(self, stream=None):
        B.cp_kv_write(self.desc, self.pool_k, self.pool_v, self.k_new, self.v_new, self.positions, self.qo_indptr,
                      self.page_indptr, self.page_indices, dev_status=self.dev_status, stream=stream)

    def partial(self, stream=None):
        P = self.w.P
        # one token a row (a decode step): the call takes no token -> row map
        one_per_row = self.w.decode and self.w.num_tokens == self.w.num_rows
        B.cp_paged_attn_partial_ex(self.desc, self.pool_k, self.pool_v, self.q, self.kv_len, self.max_kv_len,
                                   self.page_indptr, self.page_indices, self.w.scale, self.o_parts[:P],
                                   self.lse_parts[:P], self.workspace,
                                   qo_indptr=None if one_per_row else self.qo_indptr,
                                   num_rows=self.w.num_rows, row_order=self.row_order if one_per_row else None,
                                   dev_status=self.dev_status, stream=stream)

    def own(self, stream=None):
        P = self.w.P
        B.own_token_attn(self.q, self.k_new, self.v_new, self.qo_indptr, self.w.num_real_rows, self.max_q_len,
                         self.w.scale, self.o_parts[P], self.lse_parts[P], stream=stream)

    def merge(self, stream=None):
        B.lse_merge(self.o_parts, self.lse_parts, self.out, self.lse, stream=stream)

    def run_step(self, stream=None):
        self.write_new(stream)
        self.partial(stream)
        if not self.w.decode:
            self.own(stream)
        self.merge(stream)
        return self.out, self.lse

    # -- fused path: partials of every partner merged inside the partial launch
    def fused(self, stream=None, out=None, lse=None):
        """All partners' partials and their merge in one launch; a non-decode
        step folds in the own-token partial (computed first by ``own``).
        ``out``/``lse`` default to this object's output buffers."""
        if self._fused_ws is None:
            n = B.fused_workspace_bytes(self.desc, self.w.num_q_heads, self.w.num_tokens, self.max_kv_len)
            self._fused_ws = torch.empty((max(n, 256),), dtype=torch.uint8, device=self.device)
        P = self.w.P
        one_per_row = self.w.decode and self.w.num_tokens == self.w.num_rows
        extra_o = None if self.w.decode else self.o_parts[P]
        extra_lse = None if self.w.decode else self.lse_parts[P]
        B.cp_paged_attn_fused(self.desc, self.pool_k, self.pool_v, self.q, self.kv_len, self.max_kv_len,
                              self.page_indptr, self.page_indices, self.w.scale,
                              self.out if out is None else out, self._fused_ws,
                              lse_out=self.lse if lse is None else lse, extra_o=extra_o, extra_lse=extra_lse,
                              qo_indptr=None if one_per_row else self.qo_indptr, num_rows=self.w.num_rows,
                              row_order=self.row_order if one_per_row else None,
                              dev_status=self.dev_status, stream=stream)

    def run_step_fused(self, stream=None, out=None, lse=None):
        self.write_new(stream)
        if not self.w.decode:
            self.own(stream)
        self.fused(stream, out, lse)
        return (self.out if out is None else out), (self.lse if lse is None else lse)

    # -- TP-mode head layout (vLLM _forward_with_dcp): every partner attends the
    # gathered query heads of all P ranks; its LSE comes head-major ([H, B]);
    # rank r then combines the partners' partials of its own head slice and
    # merges the result with its own-token partial.
    def run_step_tp(self, stream=None, out=None, lse=None):
        w = self.w
        P, T, Hq, Dv = w.P, w.num_tokens, w.num_q_heads, w.head_dim_v
        if Hq % P != 0:
            raise ValueError("TP mode needs the query heads to split evenly over the P ranks")
        Hl = Hq // P
        out = self.out if out is None else out
        lse = self.lse if lse is None else lse
        if getattr(self, "_lse_hm", None) is None:
            self._lse_hm = torch.empty((P, Hq, T), dtype=torch.float32, device=self.device)
            self._cor = torch.empty((P, T, Hl, Dv), dtype=torch.float32, device=self.device)
            self._lse_cor = torch.empty((P, Hl, T), dtype=torch.float32, device=self.device)
        one_per_row = w.decode and w.num_tokens == w.num_rows
        self.write_new(stream)
        B.cp_paged_attn_partial_ex(self.desc, self.pool_k, self.pool_v, self.q, self.kv_len, self.max_kv_len,
                                   self.page_indptr, self.page_indices, w.scale, self.o_parts[:P], self._lse_hm,
                                   self.workspace, lse_layout=B.LSE_HEAD_MAJOR,
                                   qo_indptr=None if one_per_row else self.qo_indptr, num_rows=w.num_rows,
                                   dev_status=self.dev_status, stream=stream)
        if not w.decode:
            self.own(stream)
        for r in range(P):
            # dcp_combine for rank r: the P partners' rows of heads [r*Hl, (r+1)*Hl)
            views = [B.view(self.o_parts, self._lse_hm, Hq * Dv, Dv, 1, T,
                            o_offset=(p * T * Hq + r * Hl) * Dv, lse_offset=(p * Hq + r * Hl) * T)
                     for p in range(P)]
            if w.decode:  # no own-token partial: the combine is the rank's output
                B.lse_merge_views(views, T, Hl, Dv, out, Hq * Dv, Dv, lse, Hq, 1, out_offset=r * Hl * Dv,
                                  lse_out_offset=r * Hl, stream=stream)
                continue
            B.lse_merge_views(views, T, Hl, Dv, self._cor, Hl * Dv, Dv, self._lse_cor, 1, T,
                              out_offset=r * T * Hl * Dv, lse_out_offset=r * Hl * T, stream=stream)
            # merge_attn_states(context, own query partial) for the rank's heads
            final = [B.view(self._cor, self._lse_cor, Hl * Dv, Dv, 1, T, o_offset=r * T * Hl * Dv,
                            lse_offset=r * Hl * T),
                     B.view(self.o_parts, self.lse_parts, Hq * Dv, Dv, Hq, 1, o_offset=(P * T * Hq + r * Hl) * Dv,
                            lse_offset=P * T * Hq + r * Hl)]
            B.lse_merge_views(final, T, Hl, Dv, out, Hq * Dv, Dv, lse, Hq, 1, out_offset=r * Hl * Dv,
                              lse_out_offset=r * Hl, stream=stream)
        return out, lse

    def capture(self, fused=True):
        """Record the step (fused, or partial + merge) into a CUDA graph over
        this object's buffers (a captured bucket: later steps refill the same
        inputs and replay)."""
        run = self.run_step_fused if fused else self.run_step
        side = torch.cuda.Stream(device=self.device)
        side.wait_stream(torch.cuda.current_stream(self.device))
        with torch.cuda.stream(side):
            run(side)  # first call outside capture: workspace and kernel attributes
        torch.cuda.current_stream(self.device).wait_stream(side)
        torch.cuda.synchronize(self.device)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            run(torch.cuda.current_stream(self.device))
        return self.graph

    def replay(self):
        self.graph.replay()
        return self.out, self.lse

    def status(self) -> int:
        return int(self.dev_status.item())
