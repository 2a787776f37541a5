"""A batched decode step from pinned host buffers, replayed as one CUDA graph.

A decode step (one new token for each of B sequences) is a few microseconds of
work in four short kernels: the indexer over each sequence's keys, the top-k,
the split attention and the merge of its splits.  Launched one call at a time
from the host, the launches and the small host<->device copies cost more than
the work.  HostDecode captures the whole step once -- the uploads of the new
tokens' inputs from fixed pinned buffers, the library calls, and the download of
the output into a fixed pinned buffer -- and replays it with a single launch.
The sequences' caches (indexer keys and latent rows) stay on the device; the
caller appends each new token's rows to them before the step, and writes the
token's inputs into the pinned buffers `h_qi`, `h_w`, `h_q`, `h_pos`, `h_len`.
Every step of the method still runs in the library's kernels; nothing here
computes.
"""
from __future__ import annotations

import torch

from . import _lib


class HostDecode:
    """Decode steps for B sequences over device-resident caches.

    k_idx  [B, Nmax, 128] bf16 (as int16 or bfloat16) indexer keys, on the device
    kv     [B, Nmax, 576] bf16 latent cache rows, on the device
    Per step (pinned host buffers owned by this object, filled by the caller):
      h_qi [B, 1, 32, 128] int16 (bf16 bits), h_w [B, 1, 32] f32, h_q [B, 64, 576] int16,
      h_pos [B] int32 (the new token's position, kv_len - 1), h_len [B] int32 (keys in each cache)
    Result: h_out [B, 64, 512] (float32 by default, or bf16), valid once the stream reaches the
    point where __call__ returned (synchronise it, or record an event on it).
    """

    def __init__(self, k_idx: torch.Tensor, kv: torch.Tensor, top_k: int, scale: float,
                 out_dtype=torch.float32, stream=None):
        B, Nmax = kv.shape[0], kv.shape[1]
        dev = kv.device
        self.B, self.Nmax, self.top_k, self.scale = B, Nmax, top_k, float(scale)
        self.k_idx, self.kv = k_idx, kv
        pin = lambda shape, dt: torch.empty(shape, dtype=dt).pin_memory()
        self.h_qi = pin((B, 1, 32, 128), torch.int16)
        self.h_w = pin((B, 1, 32), torch.float32)
        self.h_q = pin((B, 64, 576), torch.int16)
        self.h_pos = pin((B,), torch.int32)
        self.h_len = pin((B,), torch.int32)
        self.h_out = pin((B, 64, 512), out_dtype)
        self.d_qi = torch.empty((B, 1, 32, 128), dtype=torch.int16, device=dev)
        self.d_w = torch.empty((B, 1, 32), dtype=torch.float32, device=dev)
        self.d_q = torch.empty((B, 64, 576), dtype=torch.int16, device=dev)
        self.d_pos = torch.empty((B,), dtype=torch.int32, device=dev)
        self.d_len = torch.empty((B,), dtype=torch.int32, device=dev)
        ld = (Nmax + 3) // 4 * 4
        self.d_S = torch.empty((B, 1, ld), dtype=torch.float32, device=dev)
        self.d_idx = torch.empty((B, 1, top_k), dtype=torch.int32, device=dev)
        self.d_out = torch.empty((B, 64, 512), dtype=out_dtype, device=dev)
        self.ws = torch.empty((_lib.attn_workspace_size(B, top_k),), dtype=torch.uint8, device=dev)
        self.h2d_bytes = sum(t.numel() * t.element_size() for t in (self.h_qi, self.h_w, self.h_q, self.h_pos,
                                                                    self.h_len))
        self.d2h_bytes = self.h_out.numel() * self.h_out.element_size()
        self.graph = None
        self._stream = stream

    def _step(self):
        for d, h in ((self.d_qi, self.h_qi), (self.d_w, self.h_w), (self.d_q, self.h_q), (self.d_pos, self.h_pos),
                     (self.d_len, self.h_len)):
            d.copy_(h, non_blocking=True)
        _lib.indexer_scores(self.d_qi, self.k_idx, self.d_w, self.d_pos, self.d_len, scores=self.d_S)
        _lib.topk(self.d_S, self.d_pos, self.d_len, self.Nmax, self.top_k, idx=self.d_idx)
        _lib.mla_sparse_attn_decode(self.d_q, self.kv, self.d_len, self.d_idx[:, 0], self.scale, out=self.d_out,
                                    workspace=self.ws)
        self.h_out.copy_(self.d_out, non_blocking=True)

    def __call__(self, stream=None):
        """Enqueue one step on `stream` (default: the current stream) and return h_out."""
        main = stream if stream is not None else torch.cuda.current_stream(self.kv.device)
        if self.graph is None:
            side = torch.cuda.Stream(device=self.kv.device)
            side.wait_stream(main)
            with torch.cuda.stream(side):
                self._step()                # first use: the library's per-kernel setup, outside capture
            main.wait_stream(side)
            torch.cuda.synchronize(self.kv.device)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                self._step()
            self.graph = g
        with torch.cuda.stream(main):
            self.graph.replay()
        return self.h_out
