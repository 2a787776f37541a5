"""A prefill chunk from pinned host buffers to a pinned host output.

The three library calls (indexer scores, top-k, sparse MLA attention) run on
device copies of the inputs; this module only schedules the host<->device
copies around them so that they overlap the kernels:

  copy stream : indexer inputs | kv | q slice 0 | q slice 1 | ...   (host -> device)
  compute     :                 indexer | top-k | attn 0 | attn 2 | ...
  compute 2   :                                     attn 1 | attn 3 | ...
  copy stream :                                     out 0 |  out 1 | ... (device -> host)

Attention runs per slice of the chunk's queries (each slice is one
`mla_sparse_attn_prefill` call over its rows of q, idx and out), so a slice
starts as soon as its part of q has landed and its output is copied back while
the next slice computes.  By default a slice is two rounds of the attention's
persistent CTAs (2 x the SM count queries): the device->host copy of a slice
(about 0.11 ms for 304 queries) then keeps pace with the attention, and only
the last slice's copy trails the compute.  Even and odd slices alternate
between two streams, so the last round of one slice's persistent CTAs overlaps
the next slice's start.  Every step of the method still runs in the library's
kernels; nothing here computes.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import _lib


class HostPrefill:
    """Reusable device buffers, streams and events for chunks of one shape.

    Shapes (batch 1 prefill chunk): qI [1,L,32,128], kI [1,N,128] (bf16 bits as
    int16/bfloat16), w [1,L,32] f32, q_pos0 / kv_len [1] int32, q [1,L,64,576],
    kv [1,N,576] (bf16 bits), out [L,64,512] bf16.  Host tensors must be pinned
    for the copies to be asynchronous.
    """

    def __init__(self, L: int, N: int, top_k: int, device=None, slices: Optional[int] = None,
                 out_dtype=torch.float32):
        self.L, self.N, self.top_k = L, N, top_k
        self.dev = torch.device(device if device is not None else "cuda")
        if slices is None:   # two rounds of one attention CTA per SM a slice
            per_slice = 2 * torch.cuda.get_device_properties(self.dev).multi_processor_count
            slices = (L + per_slice - 1) // per_slice
        self.slices = max(1, min(slices, L))
        dev = self.dev
        self.d_qi = torch.empty((1, L, 32, 128), dtype=torch.int16, device=dev)
        self.d_ki = torch.empty((1, N, 128), dtype=torch.int16, device=dev)
        self.d_w = torch.empty((1, L, 32), dtype=torch.float32, device=dev)
        self.d_pos = torch.empty((1,), dtype=torch.int32, device=dev)
        self.d_len = torch.empty((1,), dtype=torch.int32, device=dev)
        self.d_q = torch.empty((1, L, 64, 576), dtype=torch.int16, device=dev)
        self.d_kv = torch.empty((1, N, 576), dtype=torch.int16, device=dev)
        ld = (N + 3) // 4 * 4
        self.d_S = torch.empty((1, L, ld), dtype=torch.float32, device=dev)
        self.d_idx = torch.empty((1, L, top_k), dtype=torch.int32, device=dev)
        self.d_out = torch.empty((L, 64, 512), dtype=out_dtype, device=dev)
        self.copy_in = torch.cuda.Stream(device=dev)
        self.copy_out = torch.cuda.Stream(device=dev)
        self.attn2 = torch.cuda.Stream(device=dev)   # odd slices: their launch tails overlap the even ones
        per = (L + self.slices - 1) // self.slices
        self.bounds = [(i, min(L, i + per)) for i in range(0, L, per)]

    def __call__(self, h_qi, h_ki, h_w, h_pos, h_len, h_q, h_kv, h_out, scale: float, stream=None):
        """Enqueue one chunk on `stream` (default: the current stream).  On return
        the work is queued; `h_out` holds the result once `stream` reaches this
        point (synchronise it, or record an event on it)."""
        main = stream if stream is not None else torch.cuda.current_stream(self.dev)
        cin, cout = self.copy_in, self.copy_out
        cin.wait_stream(main)       # the previous chunk's users of the device buffers are done
        cout.wait_stream(main)
        with torch.cuda.stream(cin):
            for d, h in ((self.d_qi, h_qi), (self.d_ki, h_ki), (self.d_w, h_w), (self.d_pos, h_pos),
                         (self.d_len, h_len)):
                d.copy_(_as(h, d), non_blocking=True)
            ev_idx_in = torch.cuda.Event()
            ev_idx_in.record(cin)
            self.d_kv.copy_(_as(h_kv, self.d_kv), non_blocking=True)
            ev_q = []
            for a, b in self.bounds:
                self.d_q[:, a:b].copy_(_as(h_q, self.d_q)[:, a:b], non_blocking=True)
                e = torch.cuda.Event()
                e.record(cin)
                ev_q.append(e)
        main.wait_event(ev_idx_in)
        _lib.indexer_scores(self.d_qi, self.d_ki, self.d_w, self.d_pos, self.d_len, scores=self.d_S, stream=main)
        _lib.topk(self.d_S, self.d_pos, self.d_len, self.N, self.top_k, idx=self.d_idx, stream=main)
        self.attn2.wait_stream(main)    # the selection is complete for every slice
        for k, ((a, b), e) in enumerate(zip(self.bounds, ev_q)):
            st = main if k % 2 == 0 else self.attn2
            st.wait_event(e)
            _lib.mla_sparse_attn_prefill(self.d_q[0, a:b], self.d_kv[0], self.d_idx[0, a:b], scale,
                                         out=self.d_out[a:b], stream=st)
            done = torch.cuda.Event()
            done.record(st)
            cout.wait_event(done)
            with torch.cuda.stream(cout):
                _as(h_out, self.d_out)[a:b].copy_(self.d_out[a:b], non_blocking=True)
        main.wait_stream(self.attn2)
        main.wait_stream(cout)      # the chunk ends when its last output slice is on the host
        return h_out


def _as(h: torch.Tensor, like: torch.Tensor) -> torch.Tensor:
    """View 16-bit host data with the device buffer's dtype (bf16 bits travel as int16)."""
    if h.dtype != like.dtype and h.element_size() == like.element_size():
        return h.view(like.dtype)
    return h
