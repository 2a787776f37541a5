"""ctypes binding of libdsa_gb300.so (the C ABI in include/dsa.h).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  Tensors are torch CUDA tensors (PyTorch provides device memory and
streams); bf16 tensors may be torch.bfloat16 or 16-bit integer views of the
same bits.  If the library is missing or the device is not sm_103, calls raise
instead of falling back to anything else.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

from . import _build

DSA_OK = 0
DSA_OUT_F32 = 0     # attention output element types (include/dsa.h)
DSA_OUT_BF16 = 1
STATUS_NAMES = {
    0: "DSA_OK", 1: "DSA_ERR_INVALID_ARG", 2: "DSA_ERR_UNSUPPORTED_SHAPE", 3: "DSA_ERR_MISALIGNED",
    4: "DSA_ERR_WORKSPACE_TOO_SMALL", 5: "DSA_ERR_CUDA", 6: "DSA_ERR_DEVICE_TIMEOUT",
    7: "DSA_ERR_DEVICE_BOUNDS", 8: "DSA_ERR_UNSUPPORTED_DEVICE", 9: "DSA_ERR_SCRATCH_TOO_SMALL",
}

# every symbol include/dsa.h declares, with (restype, argtypes)
_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t
_F = ctypes.c_float
SIGNATURES = {
    "dsa_status_string": (ctypes.c_char_p, [ctypes.c_int32]),
    "dsa_abi_version": (ctypes.c_int, []),
    "dsa_indexer_scores": (ctypes.c_int32, [_P, _P, _P, _P, _P, _I, _I, _I, _P, _I64, _P]),
    "dsa_topk_workspace_size": (_SZ, [_I, _I, _I, _I]),
    "dsa_topk": (ctypes.c_int32, [_P, _I64, _P, _P, _I, _I, _I, _I, _P, _P, _SZ, _P]),
    "mla_sparse_attn_prefill": (ctypes.c_int32, [_P, _P, _P, _I, _I, _I, _F, _P, _I, _P, _P, _SZ, _P]),
    "mla_sparse_attn_workspace_size": (_SZ, [_I, _I, _I, _I]),
    "mla_sparse_attn_decode": (ctypes.c_int32, [_P, _P, _P, _P, _I, _I, _I, _F, _P, _I, _P, _P, _SZ, _P]),
    "mla_sparse_attn_decode_noalloc": (ctypes.c_int32, [_P, _P, _P, _P, _I, _I, _I, _F, _P, _I, _P, _P]),
    "dsa_indexer_scores_paged": (ctypes.c_int32, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _I64, _P]),
    "mla_sparse_attn_decode_paged": (ctypes.c_int32, [_P, _P, _P, _P, _I, _I, _I, _P, _I, _I, _I, _F, _P, _I, _P,
                                                      _P, _SZ, _P]),
    "mla_sparse_attn_prefill_paged": (ctypes.c_int32, [_P, _P, _P, _I, _I, _P, _I, _I, _I, _F, _P, _I, _P, _P, _SZ,
                                                       _P]),
    "mla_value_up_proj": (ctypes.c_int32, [_P, _P, _I, _P, _P]),
    "dsa_indexer_source_layer": (ctypes.c_int, [_I, _I, _I]),
    "dsa_device_status": (ctypes.c_int32, [_P, ctypes.POINTER(ctypes.c_int32), _I]),
    "dsa_selftest_wait_timeout": (ctypes.c_int32, [_I, ctypes.c_uint64, _P]),
}

_lock = threading.Lock()
_lib: Optional[ctypes.CDLL] = None


class DsaError(RuntimeError):
    def __init__(self, fn: str, code: int):
        self.code = code
        super().__init__(f"{fn} failed: {STATUS_NAMES.get(code, code)} ({status_string(code)})")


def lib_path() -> str:
    return _build.LIB_PATH


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Load the library (it must have been built: see __graft_entry__.build())."""
    global _lib
    with _lock:
        if _lib is None:
            p = path or _build.LIB_PATH
            if not os.path.exists(p):
                raise RuntimeError(f"{p} is missing: build the CUDA library first "
                                   "(python -c 'import __graft_entry__ as g; g.build()')")
            lib = ctypes.CDLL(p)
            for name, (res, args) in SIGNATURES.items():
                f = getattr(lib, name)
                f.restype = res
                f.argtypes = args
            _lib = lib
    return _lib


def status_string(code: int) -> str:
    return load().dsa_status_string(code).decode()


def _check(fn: str, code: int):
    if code != DSA_OK:
        raise DsaError(fn, code)


def _stream(stream=None) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def _is16(t: torch.Tensor) -> bool:
    return t.dtype in (torch.bfloat16, torch.int16, torch.uint16)


def _out_dtype(out: torch.Tensor) -> int:
    """The C ABI's out_dtype for an attention output tensor: float32, or bf16 (or a 16-bit view of it)."""
    if out.dtype == torch.float32:
        return DSA_OUT_F32
    if _is16(out):
        return DSA_OUT_BF16
    raise ValueError(f"attention output must be float32 or bf16, got {out.dtype}")


def _new_out(rows: int, device, dtype) -> torch.Tensor:
    if dtype not in (torch.float32, torch.bfloat16):
        raise ValueError(f"attention output must be float32 or bf16, got {dtype}")
    return torch.empty((rows, 64, 512), dtype=dtype, device=device)


# ----------------------------------------------------------------------------- entry points

def indexer_scores(q_idx: torch.Tensor, k_idx: torch.Tensor, w: torch.Tensor, q_pos0: torch.Tensor,
                   kv_len: torch.Tensor, scores: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """scores [B, L, ld] f32 from q_idx [B,L,32,128], k_idx [B,Nmax,128] (bf16), w [B,L,32] f32."""
    B, L, Hi, Di = q_idx.shape
    Nmax = k_idx.shape[1]
    assert _is16(q_idx) and _is16(k_idx) and w.dtype == torch.float32
    if scores is None:
        ld = (Nmax + 3) // 4 * 4
        scores = torch.empty((B, L, ld), dtype=torch.float32, device=q_idx.device)
    ld = scores.shape[-1]
    rc = load().dsa_indexer_scores(_ptr(q_idx), _ptr(k_idx), _ptr(w), _ptr(q_pos0), _ptr(kv_len),
                                   B, L, Nmax, _ptr(scores), ld, _stream(stream))
    _check("dsa_indexer_scores", rc)
    return scores


def topk(scores: torch.Tensor, q_pos0: torch.Tensor, kv_len: torch.Tensor, Nmax: int, top_k: int,
         idx: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """idx [B, L, top_k] int32 (ascending key order, -1 padded)."""
    B, L, ld = scores.shape
    if idx is None:
        idx = torch.empty((B, L, top_k), dtype=torch.int32, device=scores.device)
    rc = load().dsa_topk(_ptr(scores), ld, _ptr(q_pos0), _ptr(kv_len), B, L, Nmax, top_k, _ptr(idx),
                         None, 0, _stream(stream))
    _check("dsa_topk", rc)
    return idx


def mla_sparse_attn_prefill(q: torch.Tensor, kv: torch.Tensor, idx: torch.Tensor, scale: float,
                            out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                            want_lse: bool = False, stream=None, out_dtype=torch.float32):
    """out [L, 64, 512] (float32 by default, or bf16: the float32 result rounded; a given `out`
    decides) and lse [L, 64] f32, for q [L,64,576], kv [N,576], idx [L,top_k]."""
    L = q.shape[0]
    N = kv.shape[0]
    top_k = idx.shape[-1]
    assert _is16(q) and _is16(kv) and idx.dtype == torch.int32
    if out is None:
        out = _new_out(L, q.device, out_dtype)
    if lse is None and want_lse:
        lse = torch.empty((L, 64), dtype=torch.float32, device=q.device)
    rc = load().mla_sparse_attn_prefill(_ptr(q), _ptr(kv), _ptr(idx), L, N, top_k, float(scale), _ptr(out),
                                        _out_dtype(out), _ptr(lse), None, 0, _stream(stream))
    _check("mla_sparse_attn_prefill", rc)
    return (out, lse) if want_lse else out


def attn_workspace_size(B: int, top_k: int, is_decode: bool = True) -> int:
    return int(load().mla_sparse_attn_workspace_size(B, 1, top_k, 1 if is_decode else 0))


def mla_sparse_attn_decode(q: torch.Tensor, kv: torch.Tensor, kv_len: torch.Tensor, idx: torch.Tensor,
                           scale: float, out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                           workspace: Optional[torch.Tensor] = None, want_lse: bool = False, stream=None,
                           out_dtype=torch.float32):
    """out [B, 64, 512] (float32 by default, or bf16) for q [B,64,576], kv [B,Nmax,576], kv_len [B],
    idx [B,top_k]."""
    B = q.shape[0]
    Nmax = kv.shape[1]
    top_k = idx.shape[-1]
    if out is None:
        out = _new_out(B, q.device, out_dtype)
    if lse is None and want_lse:
        lse = torch.empty((B, 64), dtype=torch.float32, device=q.device)
    ws_bytes = attn_workspace_size(B, top_k)
    if workspace is None:
        workspace = torch.empty((ws_bytes,), dtype=torch.uint8, device=q.device)
    rc = load().mla_sparse_attn_decode(_ptr(q), _ptr(kv), _ptr(kv_len), _ptr(idx), B, Nmax, top_k, float(scale),
                                       _ptr(out), _out_dtype(out), _ptr(lse), _ptr(workspace), workspace.numel(),
                                       _stream(stream))
    _check("mla_sparse_attn_decode", rc)
    return (out, lse) if want_lse else out


def mla_sparse_attn_decode_noalloc(q: torch.Tensor, kv: torch.Tensor, kv_len: torch.Tensor, idx: torch.Tensor,
                                   scale: float, out: Optional[torch.Tensor] = None,
                                   lse: Optional[torch.Tensor] = None, want_lse: bool = False, stream=None,
                                   out_dtype=torch.float32):
    """Decode attention without a workspace, for callers that may not allocate
    device memory: the library keeps the split partials in its own fixed device
    scratch (B <= 63).  Pass preallocated `out` (and `lse`) to allocate nothing
    here either.  Calls that overlap on the GPU share that scratch and race."""
    B = q.shape[0]
    Nmax = kv.shape[1]
    top_k = idx.shape[-1]
    if out is None:
        out = _new_out(B, q.device, out_dtype)
    if lse is None and want_lse:
        lse = torch.empty((B, 64), dtype=torch.float32, device=q.device)
    rc = load().mla_sparse_attn_decode_noalloc(_ptr(q), _ptr(kv), _ptr(kv_len), _ptr(idx), B, Nmax, top_k,
                                               float(scale), _ptr(out), _out_dtype(out), _ptr(lse), _stream(stream))
    _check("mla_sparse_attn_decode_noalloc", rc)
    return (out, lse) if want_lse else out


def indexer_scores_paged(q_idx: torch.Tensor, k_pool: torch.Tensor, w: torch.Tensor, q_pos0: torch.Tensor,
                         kv_len: torch.Tensor, block_table: torch.Tensor, page_size: int, Nmax: int,
                         scores: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """indexer_scores over a paged key cache: k_pool [num_pages * page_size, 128] bf16,
    block_table [B, bt_stride] int32 (pool page of each logical page of a sequence)."""
    B, L, Hi, Di = q_idx.shape
    assert _is16(q_idx) and _is16(k_pool) and w.dtype == torch.float32 and block_table.dtype == torch.int32
    num_pages = k_pool.shape[0] // page_size
    if scores is None:
        ld = (Nmax + 3) // 4 * 4
        scores = torch.empty((B, L, ld), dtype=torch.float32, device=q_idx.device)
    ld = scores.shape[-1]
    rc = load().dsa_indexer_scores_paged(_ptr(q_idx), _ptr(k_pool), _ptr(w), _ptr(q_pos0), _ptr(kv_len),
                                         _ptr(block_table), block_table.shape[1], page_size, num_pages,
                                         B, L, Nmax, _ptr(scores), ld, _stream(stream))
    _check("dsa_indexer_scores_paged", rc)
    return scores


def mla_sparse_attn_decode_paged(q: torch.Tensor, kv_pool: torch.Tensor, kv_len: torch.Tensor,
                                 block_table: torch.Tensor, page_size: int, idx: torch.Tensor, scale: float,
                                 Nmax: int, out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                                 workspace: Optional[torch.Tensor] = None, want_lse: bool = False, stream=None,
                                 out_dtype=torch.float32):
    """mla_sparse_attn_decode over a paged cache: kv_pool [num_pages * page_size, 576] bf16,
    block_table [B, bt_stride] int32; idx holds logical key positions."""
    B = q.shape[0]
    top_k = idx.shape[-1]
    assert _is16(q) and _is16(kv_pool) and idx.dtype == torch.int32 and block_table.dtype == torch.int32
    num_pages = kv_pool.shape[0] // page_size
    if out is None:
        out = _new_out(B, q.device, out_dtype)
    if lse is None and want_lse:
        lse = torch.empty((B, 64), dtype=torch.float32, device=q.device)
    ws_bytes = attn_workspace_size(B, top_k)
    if workspace is None:
        workspace = torch.empty((ws_bytes,), dtype=torch.uint8, device=q.device)
    rc = load().mla_sparse_attn_decode_paged(_ptr(q), _ptr(kv_pool), _ptr(kv_len), _ptr(block_table),
                                             block_table.shape[1], page_size, num_pages, _ptr(idx), B, Nmax,
                                             top_k, float(scale), _ptr(out), _out_dtype(out), _ptr(lse),
                                             _ptr(workspace),
                                             workspace.numel(), _stream(stream))
    _check("mla_sparse_attn_decode_paged", rc)
    return (out, lse) if want_lse else out


def mla_sparse_attn_prefill_paged(q: torch.Tensor, kv_pool: torch.Tensor, block_table: torch.Tensor,
                                  page_size: int, idx: torch.Tensor, scale: float, N: int,
                                  out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                                  want_lse: bool = False, stream=None, out_dtype=torch.float32):
    """mla_sparse_attn_prefill over one sequence's paged cache: kv_pool [num_pages * page_size, 576]
    bf16, block_table int32 with ceil(N / page_size) entries; idx holds logical key positions < N."""
    L = q.shape[0]
    top_k = idx.shape[-1]
    assert _is16(q) and _is16(kv_pool) and idx.dtype == torch.int32 and block_table.dtype == torch.int32
    num_pages = kv_pool.shape[0] // page_size
    if out is None:
        out = _new_out(L, q.device, out_dtype)
    if lse is None and want_lse:
        lse = torch.empty((L, 64), dtype=torch.float32, device=q.device)
    rc = load().mla_sparse_attn_prefill_paged(_ptr(q), _ptr(kv_pool), _ptr(block_table), page_size, num_pages,
                                              _ptr(idx), L, N, top_k, float(scale), _ptr(out), _out_dtype(out),
                                              _ptr(lse), None, 0, _stream(stream))
    _check("mla_sparse_attn_prefill_paged", rc)
    return (out, lse) if want_lse else out


def mla_value_up_proj(o: torch.Tensor, wv_b: torch.Tensor, v: Optional[torch.Tensor] = None,
                      stream=None) -> torch.Tensor:
    """v [R, 64, 256] bf16 = per head o[r, h, :] (512 latent dims) times wv_b[h]^T,
    for o [R, 64, 512] and wv_b [64, 256, 512] (bf16)."""
    R = o.shape[0]
    assert _is16(o) and _is16(wv_b)
    assert tuple(o.shape[1:]) == (64, 512) and tuple(wv_b.shape) == (64, 256, 512)
    if v is None:
        v = torch.empty((R, 64, 256), dtype=torch.bfloat16, device=o.device)
    rc = load().mla_value_up_proj(_ptr(o), _ptr(wv_b), R, _ptr(v), _stream(stream))
    _check("mla_value_up_proj", rc)
    return v


def indexer_source_layer(layer: int, topk_freq: int = 4, skip_offset: int = 3) -> int:
    """The layer whose top-k selection `layer` attends with (itself if it runs the
    indexer); GLM-5.x shares the indexer with index_topk_freq 4, index_skip_topk_offset 3."""
    r = load().dsa_indexer_source_layer(layer, topk_freq, skip_offset)
    if r < 0:
        raise ValueError(f"invalid layer schedule arguments ({layer}, {topk_freq}, {skip_offset})")
    return r


def selftest_wait_timeout(spin: bool = False, limit_ns: int = 1_000_000, stream=None) -> None:
    """Launch the failure-detection self-test: one thread waits, with the kernels' bounded wait
    (spin: the polling form), on an mbarrier nothing arrives on; the wait gives up after limit_ns
    and the timeout shows in device_status()."""
    rc = load().dsa_selftest_wait_timeout(1 if spin else 0, ctypes.c_uint64(int(limit_ns)), _stream(stream))
    _check("dsa_selftest_wait_timeout", rc)


def device_status(reset: bool = True, stream=None) -> int:
    code = ctypes.c_int32(0)
    rc = load().dsa_device_status(_stream(stream), ctypes.byref(code), 1 if reset else 0)
    _check("dsa_device_status", rc)
    return code.value
