"""A prefill chunk from pinned host buffers to a pinned host output.

The three library calls (indexer scores, top-k, sparse MLA attention) run on
device copies of the inputs; this module only schedules the host<->device
copies around them so that they overlap the kernels:

  copy stream : indexer inputs | kv | q slice 0 | q slice 1 | ...   (host -> device)
  compute     :                 indexer | top-k | attn 0 | attn 2 | ...
  compute 2   :                                     attn 1 | attn 3 | ...
  copy stream :                                     out 0 |  out 1 | ... (device -> host)

All four are the runner's own streams; the caller's stream only orders a chunk after the work
already on it (and, with one buffer set, waits for the chunk's end).

Attention runs per slice of the chunk's queries (each slice is one
`mla_sparse_attn_prefill` call over its rows of q, idx and out), so a slice
starts as soon as its part of q has landed and its output is copied back while
the next slice computes.  By default a slice is two rounds of the attention's
persistent CTAs (2 x the SM count queries): the device->host copy of a slice
(about 0.11 ms for 304 queries) then keeps pace with the attention, and only
the last slice's copy trails the compute.  Even and odd slices alternate
between two streams, so the last round of one slice's persistent CTAs overlaps
the next slice's start.

With `sets=2` the device buffers come in two sets used by alternate chunks, and
a chunk no longer waits for the previous chunk's output to reach the host: the
next chunk's uploads and kernels run under the previous chunk's download, which
is what bounds a chunk with a float32 output (537 MB at 4096 queries).  Every
step of the method still runs in the library's kernels; nothing here computes.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import _lib


class _DeviceSet:
    """The device buffers one chunk uses."""

    def __init__(self, L: int, N: int, top_k: int, dev, out_dtype):
        self.qi = torch.empty((1, L, 32, 128), dtype=torch.int16, device=dev)
        self.ki = torch.empty((1, N, 128), dtype=torch.int16, device=dev)
        self.w = torch.empty((1, L, 32), dtype=torch.float32, device=dev)
        self.pos = torch.empty((1,), dtype=torch.int32, device=dev)
        self.len = torch.empty((1,), dtype=torch.int32, device=dev)
        self.q = torch.empty((1, L, 64, 576), dtype=torch.int16, device=dev)
        self.kv = torch.empty((1, N, 576), dtype=torch.int16, device=dev)
        ld = (N + 3) // 4 * 4
        self.S = torch.empty((1, L, ld), dtype=torch.float32, device=dev)
        self.idx = torch.empty((1, L, top_k), dtype=torch.int32, device=dev)
        self.out = torch.empty((L, 64, 512), dtype=out_dtype, device=dev)
        self.free = None            # event: the last chunk that used this set is completely done


class HostPrefill:
    """Reusable device buffers, streams and events for chunks of one shape.

    Shapes (batch 1 prefill chunk): qI [1,L,32,128], kI [1,N,128] (bf16 bits as
    int16/bfloat16), w [1,L,32] f32, q_pos0 / kv_len [1] int32, q [1,L,64,576],
    kv [1,N,576] (bf16 bits), out [L,64,512] (float32, or bf16 with out_dtype).
    Host tensors must be pinned for the copies to be asynchronous.  With sets=2,
    consecutive chunks overlap: pass each chunk its own host output buffer and
    wait for the event a call returns before reading or reusing that buffer.
    """

    def __init__(self, L: int, N: int, top_k: int, device=None, slices: Optional[int] = None,
                 out_dtype=torch.float32, sets: int = 1):
        self.L, self.N, self.top_k = L, N, top_k
        self.dev = torch.device(device if device is not None else "cuda")
        if slices is None:   # two rounds of one attention CTA per SM a slice
            per_slice = 2 * torch.cuda.get_device_properties(self.dev).multi_processor_count
            slices = (L + per_slice - 1) // per_slice
        self.slices = max(1, min(slices, L))
        if sets < 1:
            raise ValueError("sets must be >= 1")
        self.sets = [_DeviceSet(L, N, top_k, self.dev, out_dtype) for _ in range(sets)]
        self.calls = 0
        dev = self.dev
        self.copy_in = torch.cuda.Stream(device=dev)
        self.copy_out = torch.cuda.Stream(device=dev)
        self.comp = torch.cuda.Stream(device=dev)    # indexer, top-k and the even slices
        self.attn2 = torch.cuda.Stream(device=dev)   # odd slices: their launch tails overlap the even ones
        per = (L + self.slices - 1) // self.slices
        self.bounds = [(i, min(L, i + per)) for i in range(0, L, per)]

    def __call__(self, h_qi, h_ki, h_w, h_pos, h_len, h_q, h_kv, h_out, scale: float, stream=None):
        """Enqueue one chunk after the work already on `stream` (default: the current stream) and
        return an event that completes when `h_out` holds the result.  The copies and kernels run on
        the runner's own streams; with one set `stream` also waits for that event (the chunk ends
        when its last output slice is on the host), with two it does not."""
        self._check(h_qi, h_ki, h_w, h_pos, h_len, h_q, h_kv, h_out)
        main = stream if stream is not None else torch.cuda.current_stream(self.dev)
        ds = self.sets[self.calls % len(self.sets)]
        self.calls += 1
        cin, cout, comp, comp2 = self.copy_in, self.copy_out, self.comp, self.attn2
        entry = torch.cuda.Event()
        entry.record(main)
        for st in (cin, cout, comp, comp2):
            st.wait_event(entry)        # the caller's earlier work (on these host buffers too)
            if ds.free is not None:
                st.wait_event(ds.free)  # the chunk that last used this device set is completely done
        with torch.cuda.stream(cin):
            for d, h in ((ds.qi, h_qi), (ds.ki, h_ki), (ds.w, h_w), (ds.pos, h_pos), (ds.len, h_len)):
                d.copy_(_as(h, d), non_blocking=True)
            ev_idx_in = torch.cuda.Event()
            ev_idx_in.record(cin)
            ds.kv.copy_(_as(h_kv, ds.kv), non_blocking=True)
            ev_q = []
            for a, b in self.bounds:
                ds.q[:, a:b].copy_(_as(h_q, ds.q)[:, a:b], non_blocking=True)
                e = torch.cuda.Event()
                e.record(cin)
                ev_q.append(e)
        comp.wait_event(ev_idx_in)
        _lib.indexer_scores(ds.qi, ds.ki, ds.w, ds.pos, ds.len, scores=ds.S, stream=comp)
        _lib.topk(ds.S, ds.pos, ds.len, self.N, self.top_k, idx=ds.idx, stream=comp)
        comp2.wait_stream(comp)         # the selection is complete for every slice
        for k, ((a, b), e) in enumerate(zip(self.bounds, ev_q)):
            st = comp if k % 2 == 0 else comp2
            st.wait_event(e)
            _lib.mla_sparse_attn_prefill(ds.q[0, a:b], ds.kv[0], ds.idx[0, a:b], scale,
                                         out=ds.out[a:b], stream=st)
            done = torch.cuda.Event()
            done.record(st)
            cout.wait_event(done)
            with torch.cuda.stream(cout):
                _as(h_out, ds.out)[a:b].copy_(ds.out[a:b], non_blocking=True)
        cout.wait_stream(comp2)
        cout.wait_stream(comp)
        cout.wait_stream(cin)
        finished = torch.cuda.Event()
        finished.record(cout)           # every kernel and copy of this chunk is done
        ds.free = finished
        if len(self.sets) == 1:
            main.wait_event(finished)
        return finished


    def _check(self, h_qi, h_ki, h_w, h_pos, h_len, h_q, h_kv, h_out):
        """Host buffers must match this runner's shapes (16-bit data as bf16 bits in int16 or
        bfloat16) before anything is enqueued."""
        ds = self.sets[0]
        for name, h, d in (("h_qi", h_qi, ds.qi), ("h_ki", h_ki, ds.ki), ("h_w", h_w, ds.w), ("h_pos", h_pos, ds.pos),
                           ("h_len", h_len, ds.len), ("h_q", h_q, ds.q), ("h_kv", h_kv, ds.kv), ("h_out", h_out, ds.out)):
            if tuple(h.shape) != tuple(d.shape):
                raise ValueError(f"{name}: expected shape {tuple(d.shape)}, got {tuple(h.shape)}")
            # 16-bit data may be bf16 bits in either int16 or bfloat16; 32-bit data must match kind
            if h.element_size() != d.element_size() or (d.element_size() == 4 and h.dtype != d.dtype):
                raise ValueError(f"{name}: expected {d.dtype} (or the same bits), got {h.dtype}")
            if h.is_cuda:
                raise ValueError(f"{name}: expected a host tensor (pinned for asynchronous copies)")
            if not h.is_contiguous():
                raise ValueError(f"{name}: expected a contiguous tensor")


def _as(h: torch.Tensor, like: torch.Tensor) -> torch.Tensor:
    """View 16-bit host data with the device buffer's dtype (bf16 bits travel as int16)."""
    if h.dtype != like.dtype and h.element_size() == like.element_size():
        return h.view(like.dtype)
    return h
