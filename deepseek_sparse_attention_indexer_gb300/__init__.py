"""GB300-native (sm_103a) DSA sparse-attention hot path.

DSA indexer scores -> per-query top-k -> sparse absorbed-MLA attention, as
hand-written CUDA kernels behind the C ABI in include/dsa.h
(libdsa_gb300.so).  The Python names below are the same calls, marshalling
torch CUDA tensors into device pointers and the current stream.

    from deepseek_sparse_attention_indexer_gb300 import indexer_scores, topk, \
        mla_sparse_attn_prefill, mla_sparse_attn_decode

HostPrefill runs a prefill chunk from pinned host buffers with the copies
overlapped with the kernels (see host_prefill.py); HostDecode replays a batched
decode step -- uploads, the library calls and the download -- as one CUDA graph
(see host_decode.py).
"""

_API = ("indexer_scores", "topk", "mla_sparse_attn_prefill", "mla_sparse_attn_decode",
        "mla_sparse_attn_decode_noalloc", "indexer_scores_paged", "mla_sparse_attn_decode_paged",
        "mla_sparse_attn_prefill_paged", "mla_value_up_proj", "indexer_source_layer",
        "attn_workspace_size", "device_status", "selftest_wait_timeout", "status_string", "load", "lib_path",
        "DsaError")

__all__ = list(_API) + ["workloads", "build", "HostPrefill", "HostDecode", "sharding"]


def __getattr__(name):
    # torch is imported only when a library call is first used
    if name in _API:
        from . import _lib
        return getattr(_lib, name)
    if name == "build":
        from ._build import build
        return build
    if name == "HostPrefill":
        from .host_prefill import HostPrefill
        return HostPrefill
    if name == "HostDecode":
        from .host_decode import HostDecode
        return HostDecode
    if name in ("workloads", "sharding"):
        import importlib
        return importlib.import_module("." + name, __name__)
    raise AttributeError(name)
