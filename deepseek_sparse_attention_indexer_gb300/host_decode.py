"""A batched decode step from pinned host buffers, replayed as one CUDA graph.

A decode step (one new token for each of B sequences) is a few microseconds of
work in four short kernels: the indexer over each sequence's keys, the top-k,
the split attention and the merge of its splits.  Launched one call at a time
from the host, the launches and the small host<->device copies cost more than
the work.  HostDecode captures the whole step once -- the upload of the new
tokens' inputs from one fixed pinned staging buffer, the library calls, and the
download of the output into a fixed pinned buffer -- and replays it with a single
launch.
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
        # The five per-step inputs live in one pinned staging buffer (256-byte aligned sections) and
        # go up in one copy into the same layout on the device: a step's copies are latency, not
        # bandwidth (about 0.7 MB at B = 8), and each separate copy costs a few microseconds.
        parts = (("qi", (B, 1, 32, 128), torch.int16), ("w", (B, 1, 32), torch.float32),
                 ("q", (B, 64, 576), torch.int16), ("pos", (B,), torch.int32), ("len", (B,), torch.int32))
        offs, total = [], 0
        for _, shape, dt in parts:
            offs.append(total)
            n = torch.Size(shape).numel() * torch.empty((), dtype=dt).element_size()
            total += (n + 255) // 256 * 256
        self._h_stage = torch.empty((total,), dtype=torch.uint8).pin_memory()
        self._d_stage = torch.empty((total,), dtype=torch.uint8, device=dev)

        def view(buf, k):
            _, shape, dt = parts[k]
            n = torch.Size(shape).numel() * torch.empty((), dtype=dt).element_size()
            return buf[offs[k]:offs[k] + n].view(dt).view(shape)

        self.h_qi, self.h_w, self.h_q, self.h_pos, self.h_len = (view(self._h_stage, k) for k in range(5))
        self.d_qi, self.d_w, self.d_q, self.d_pos, self.d_len = (view(self._d_stage, k) for k in range(5))
        self.h_out = torch.empty((B, 64, 512), dtype=out_dtype).pin_memory()
        ld = (Nmax + 3) // 4 * 4
        self.d_S = torch.empty((B, 1, ld), dtype=torch.float32, device=dev)
        self.d_idx = torch.empty((B, 1, top_k), dtype=torch.int32, device=dev)
        self.d_out = torch.empty((B, 64, 512), dtype=out_dtype, device=dev)
        self.ws = torch.empty((_lib.attn_workspace_size(B, top_k),), dtype=torch.uint8, device=dev)
        self.h2d_bytes = total
        self.d2h_bytes = self.h_out.numel() * self.h_out.element_size()
        self.graph = None
        self._stream = stream

    def _step(self):
        self._d_stage.copy_(self._h_stage, non_blocking=True)
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
