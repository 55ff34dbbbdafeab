"""Rotation of Q and K, and attention with rotary Q and K, on tensors that
live in pinned host memory.

The tensors are split along the batch dimension into chunks.  Chunk i is
copied host->device on one stream, processed by the CUDA library on a second
and copied device->host on a third, so the copies in both directions and the
kernels of neighbouring chunks overlap.  Device staging buffers (`slots`
chunks per tensor, three by default: measured faster than two, no better
with four) are allocated once per shape and reused, the pieces of successive
calls taking them in turn.  Only argument
marshalling and stream ordering happen here; the work is one library call
per chunk.
"""
from __future__ import annotations

import torch

from . import _DTYPE_CODE, _LAYOUT_CODE, _shape4, rope_apply_qk_out, rope_attention_fwd


def _on_streams(t: torch.Tensor, streams) -> torch.Tensor:
    """Mark a staging tensor as used on the pipeline's streams, so that the
    caching allocator does not reuse its memory, once it is dropped, before
    the work queued there by then has finished."""
    for s in streams:
        t.record_stream(s)
    return t


def _head_groups(B: int, heads: tuple, chunks: int) -> int:
    """Groups per batch entry when a call is cut into more pieces than batch
    entries: the largest power of two with B * groups <= chunks that divides
    every head count (1: batch pieces only)."""
    groups = 1
    while B * groups * 2 <= chunks and all(h % (groups * 2) == 0 for h in heads if h):
        groups *= 2
    return groups


class HostRotator:
    """Rotation of pinned host Q and K into pinned host outputs.  A piece is a
    run of whole batch entries or, with more pieces than batch entries and
    the [B,H,S,D] layout (each entry's heads contiguous), one entry's heads
    split into equal groups of Q heads and of K heads.  Every head is rotated
    on its own, so every split gives the same bits."""

    def __init__(self, device=None, chunks: int = 4, slots: int = 3):
        self.device = torch.device("cuda") if device is None else torch.device(device)
        self.chunks = chunks
        self.nslots = max(2, int(slots))
        self.s_in = torch.cuda.Stream(self.device)
        self.s_run = torch.cuda.Stream(self.device)
        self.s_out = torch.cuda.Stream(self.device)
        self._key = None
        self._slots = None
        self._free = [None] * self.nslots  # event: staging slot's device->host copy done
        self._next = 0                     # slot of the next piece (pieces of calls in turn)

    def _staging(self, q, k, dims_q, dims_k):
        key = (tuple(q.shape), None if k is None else tuple(k.shape), q.dtype, dims_q, dims_k)
        if key != self._key:
            def dev(dims):
                return _on_streams(torch.empty(dims, dtype=q.dtype, device=self.device),
                                   (self.s_in, self.s_run, self.s_out))
            # the old slots may still be in use by copies and calls queued on
            # the three streams: recorded on them at creation, their memory is
            # not handed out again before that work is done
            self._slots = [(dev(dims_q), None if k is None else dev(dims_k))
                           for _ in range(self.nslots)]
            self._key = key
            self._free = [None] * self.nslots
        return self._slots

    def apply_qk(self, q: torch.Tensor, k: torch.Tensor | None, cos: torch.Tensor,
                 sin: torch.Tensor, q_out: torch.Tensor, k_out: torch.Tensor | None,
                 pos_idx: torch.Tensor | None = None, rotary_dim: int | None = None,
                 layout: str = "split_half", seq_before_head: bool = False,
                 backward: bool = False, after: torch.cuda.Event | None = None):
        """Rotate pinned host tensors q, k into pinned host tensors q_out, k_out.

        cos, sin and pos_idx ([S] int32) are device tensors.  Work is ordered
        after the event `after` (if given).  Returns the event recorded when
        the last device->host copy is done.
        """
        B, Hq, S, D = _shape4(q, seq_before_head)
        Hk = 0 if k is None else _shape4(k, seq_before_head)[1]
        for t in (q, k, q_out, k_out):
            if t is not None and (t.is_cuda or not t.is_pinned() or not t.is_contiguous()):
                raise ValueError("host tensors must be contiguous pinned CPU memory")
        rd = 2 * cos.shape[1] if rotary_dim is None else rotary_dim
        groups = 1 if seq_before_head else _head_groups(B, (Hq, Hk), self.chunks)
        if groups == 1:
            n = max(1, min(self.chunks, B))
            per = (B + n - 1) // n
            pieces = [(b0, min(B, b0 + per), 0, 1) for b0 in range(0, B, per)]
        else:
            per = 1
            pieces = [(b, b + 1, g, groups) for b in range(B) for g in range(groups)]
        hq_c, hk_c = Hq // groups, Hk // groups
        slots = self._staging(q, k, (per,) + tuple(q.shape[1:]) if groups == 1 else (1, hq_c, S, D),
                              None if k is None else
                              ((per,) + tuple(k.shape[1:]) if groups == 1 else (1, hk_c, S, D)))
        for s in (self.s_in, self.s_run, self.s_out):
            if after is not None:
                s.wait_event(after)
        done = None
        for b0, b1, g, ng in pieces:
            slot = self._next
            self._next = (self._next + 1) % self.nslots
            dq, dk = slots[slot]
            dq, dk = dq[: b1 - b0], None if dk is None else dk[: b1 - b0]
            if ng == 1:                    # whole batch entries
                src_q, src_k = q[b0:b1], None if k is None else k[b0:b1]
                dst_q, dst_k = q_out[b0:b1], None if k is None else k_out[b0:b1]
            else:                          # heads of one entry ([B,H,S,D]: contiguous)
                src_q, dst_q = q[b0, g * hq_c:(g + 1) * hq_c], q_out[b0, g * hq_c:(g + 1) * hq_c]
                src_k = None if k is None else k[b0, g * hk_c:(g + 1) * hk_c]
                dst_k = None if k is None else k_out[b0, g * hk_c:(g + 1) * hk_c]
                dq = dq[0]
                dk = None if dk is None else dk[0]
            if self._free[slot] is not None:
                self.s_in.wait_event(self._free[slot])
            with torch.cuda.stream(self.s_in):
                dq.copy_(src_q, non_blocking=True)
                if k is not None:
                    dk.copy_(src_k, non_blocking=True)
                ready = torch.cuda.Event()
                ready.record(self.s_in)
            self.s_run.wait_event(ready)
            rope_apply_qk_out(dq, dk, dq, dk, cos, sin, pos_idx, 0, b1 - b0, Hq // ng, Hk // ng,
                              S, D, rd, _LAYOUT_CODE[layout], int(seq_before_head), int(backward),
                              _DTYPE_CODE[q.dtype], cos.shape[0], self.s_run)
            rotated = torch.cuda.Event()
            rotated.record(self.s_run)
            self.s_out.wait_event(rotated)
            with torch.cuda.stream(self.s_out):
                dst_q.copy_(dq, non_blocking=True)
                if k is not None:
                    dst_k.copy_(dk, non_blocking=True)
                done = torch.cuda.Event()
                done.record(self.s_out)
            self._free[slot] = done
        return done


class HostAttention:
    """softmax(scale * rot(q) rot(k)^T + mask) v for pinned host q, k, v into
    a pinned host o, through rope_attention_fwd with a key workspace, one call
    per piece.  A piece is a run of whole batch entries, or, with more pieces
    than batch entries, one batch entry's key/value heads split into equal
    groups (with their query heads).  Each output row depends only on its own
    query row and its key/value head, so every split gives the same bits.  Each
    piece's copies of q, k, v in, the call, and the copy of o out run on three
    streams, so neighbouring pieces overlap; more pieces leave less of the
    first copy in and the last copy out exposed."""

    def __init__(self, device=None, chunks: int = 4, slots: int = 3):
        self.device = torch.device("cuda") if device is None else torch.device(device)
        self.chunks = chunks
        self.nslots = max(2, int(slots))
        self.s_in = torch.cuda.Stream(self.device)
        self.s_run = torch.cuda.Stream(self.device)
        self.s_out = torch.cuda.Stream(self.device)
        self._key = None
        self._slots = None
        self._ws = None
        self._free = [None] * self.nslots
        self._next = 0

    def _pieces(self, B: int, Hk: int):
        """(b0, b1, kv0, kv1) ranges covering [0, B) x [0, Hk)."""
        if self.chunks <= B:
            n = max(1, self.chunks)
            per = (B + n - 1) // n
            return [(b0, min(B, b0 + per), 0, Hk) for b0 in range(0, B, per)]
        groups = _head_groups(B, (Hk,), self.chunks)
        kv = Hk // groups
        return [(b, b + 1, g * kv, (g + 1) * kv) for b in range(B) for g in range(groups)]

    def _staging(self, q, k, nb, nkv, grp):
        key = (tuple(q.shape), tuple(k.shape), q.dtype, nb, nkv)
        if key != self._key:
            def dev(t, heads):
                return _on_streams(torch.empty((nb, heads) + tuple(t.shape[2:]), dtype=t.dtype,
                                               device=self.device),
                                   (self.s_in, self.s_run, self.s_out))
            self._slots = [(dev(q, nkv * grp), dev(k, nkv), dev(k, nkv), dev(q, nkv * grp))
                           for _ in range(self.nslots)]
            # the calls all run on s_run, one after another: one workspace serves them
            self._ws = dev(k, nkv)
            self._key = key
            self._free = [None] * self.nslots
        return self._slots, self._ws

    def forward(self, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor,
                cos: torch.Tensor, sin: torch.Tensor, pos_q: torch.Tensor | None = None,
                pos_k: torch.Tensor | None = None, rotary_dim: int | None = None,
                layout: str = "split_half", causal: bool = False, scale: float | None = None,
                after: torch.cuda.Event | None = None):
        """q [B,Hq,Sq,D], k and v [B,Hk,Sk,D], o like q: contiguous pinned CPU
        tensors.  cos, sin and pos_q [Sq], pos_k [Sk] (int32) are device
        tensors.  Work is ordered after the event `after` (if given).  Returns
        the event recorded when the last copy of o to the host is done."""
        for t in (q, k, v, o):
            if t.is_cuda or not t.is_pinned() or not t.is_contiguous():
                raise ValueError("host tensors must be contiguous pinned CPU memory")
        B, Hq, Sq, D = q.shape
        _, Hk, Sk, _ = k.shape
        if v.shape != k.shape or o.shape != q.shape:
            raise ValueError("v must have k's shape and o q's shape")
        if Hk < 1 or Hq % Hk:
            raise ValueError("Hq must be a multiple of Hk")
        grp = Hq // Hk
        rd = 2 * cos.shape[1] if rotary_dim is None else rotary_dim
        pieces = self._pieces(B, Hk)
        nb = max(p[1] - p[0] for p in pieces)
        nkv = max(p[3] - p[2] for p in pieces)
        slots, ws = self._staging(q, k, nb, nkv, grp)
        ws_bytes = ws.numel() * ws.element_size()
        for s in (self.s_in, self.s_run, self.s_out):
            if after is not None:
                s.wait_event(after)
        done = None
        for b0, b1, kv0, kv1 in pieces:
            slot = self._next
            self._next = (self._next + 1) % self.nslots
            hq0, hq1 = kv0 * grp, kv1 * grp
            # a piece is whole batch entries or one entry's heads: contiguous either way
            dq, dk, dv, do = slots[slot]
            dq, do = dq[: b1 - b0, : hq1 - hq0], do[: b1 - b0, : hq1 - hq0]
            dk, dv = dk[: b1 - b0, : kv1 - kv0], dv[: b1 - b0, : kv1 - kv0]
            if self._free[slot] is not None:
                self.s_in.wait_event(self._free[slot])
            with torch.cuda.stream(self.s_in):
                dq.copy_(q[b0:b1, hq0:hq1], non_blocking=True)
                dk.copy_(k[b0:b1, kv0:kv1], non_blocking=True)
                dv.copy_(v[b0:b1, kv0:kv1], non_blocking=True)
                ready = torch.cuda.Event()
                ready.record(self.s_in)
            self.s_run.wait_event(ready)
            rope_attention_fwd(dq, dk, dv, do, cos, sin, pos_q, pos_k, b1 - b0, hq1 - hq0,
                               kv1 - kv0, Sq, Sk, D, rd, _LAYOUT_CODE[layout], int(causal),
                               -1.0 if scale is None else scale, _DTYPE_CODE[q.dtype],
                               cos.shape[0], ws, ws_bytes, self.s_run)
            computed = torch.cuda.Event()
            computed.record(self.s_run)
            self.s_out.wait_event(computed)
            with torch.cuda.stream(self.s_out):
                o[b0:b1, hq0:hq1].copy_(do, non_blocking=True)
                done = torch.cuda.Event()
                done.record(self.s_out)
            self._free[slot] = done
        return done
