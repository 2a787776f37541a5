"""C ABI checks that need no GPU: the library builds, loads, exports every
function include/dsa.h declares, and rejects bad arguments on the host with
the documented status codes before touching the device."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dsa.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    from deepseek_sparse_attention_indexer_gb300 import _build
    path = _build.build()
    from deepseek_sparse_attention_indexer_gb300 import _lib
    return _lib.load(path)


def test_header_declares_the_path():
    names = declared_functions()
    for n in ["dsa_indexer_scores", "dsa_topk", "mla_sparse_attn_prefill", "mla_sparse_attn_decode",
              "dsa_status_string", "dsa_abi_version", "dsa_device_status", "dsa_topk_workspace_size",
              "mla_sparse_attn_workspace_size", "dsa_indexer_scores_paged", "mla_sparse_attn_decode_paged",
              "mla_sparse_attn_prefill_paged", "mla_value_up_proj", "dsa_indexer_source_layer",
              "dsa_selftest_wait_timeout"]:
        assert n in names


def test_exports_every_declared_symbol(lib):
    from deepseek_sparse_attention_indexer_gb300 import _build
    out = subprocess.run(["nm", "-D", "--defined-only", _build.LIB_PATH], capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for n in declared_functions():
        assert n in exported, n
        assert getattr(lib, n) is not None
    from deepseek_sparse_attention_indexer_gb300 import _lib
    assert set(_lib.SIGNATURES) == set(declared_functions())


def test_version_and_strings(lib):
    assert lib.dsa_abi_version() == 5
    for code in range(0, 10):
        s = lib.dsa_status_string(code)
        assert s and len(s) > 1
    assert lib.dsa_status_string(12345) == b"unknown status"


def test_host_validation_rejects_bad_arguments(lib):
    P = 4096                          # any 16-byte aligned non-null address (never dereferenced)
    stream = None
    # null pointers
    assert lib.dsa_indexer_scores(None, P, P, P, P, 1, 1, 16, P, 16, stream) == 1
    # sizes
    assert lib.dsa_indexer_scores(P, P, P, P, P, 0, 1, 16, P, 16, stream) == 1
    assert lib.dsa_indexer_scores(P, P, P, P, P, 1, 1, 16, P, 8, stream) == 1     # ld < Nmax
    # alignment
    assert lib.dsa_indexer_scores(P + 2, P, P, P, P, 1, 1, 16, P, 16, stream) == 3
    assert lib.dsa_indexer_scores(P, P, P, P, P, 1, 1, 16, P, 18, stream) == 3    # ld % 4
    # top-k range
    assert lib.dsa_topk(P, 16, P, P, 1, 1, 16, 0, P, None, 0, stream) == 2
    assert lib.dsa_topk(P, 16, P, P, 1, 1, 16, 2049, P, None, 0, stream) == 2
    assert lib.dsa_topk_workspace_size(1, 4096, 65536, 2048) == 0
    # attention
    assert lib.mla_sparse_attn_prefill(P, P, P, 4, 64, 4096, 0.0625, P, 0, None, None, 0, stream) == 2
    assert lib.mla_sparse_attn_prefill(P, P, P, 4, 64, 32, -1.0, P, 0, None, None, 0, stream) == 1
    assert lib.mla_sparse_attn_prefill(P, P + 8, P, 4, 64, 32, 0.0625, P, 0, None, None, 0, stream) == 3
    assert lib.mla_sparse_attn_prefill(P, P, P, 4, 64, 32, 0.0625, P, 2, None, None, 0, stream) == 1  # out_dtype
    ws = lib.mla_sparse_attn_workspace_size(8, 1, 2048, 1)
    assert ws > 0 and lib.mla_sparse_attn_workspace_size(1, 4096, 2048, 0) == 0
    assert lib.mla_sparse_attn_decode(P, P, P, P, 8, 4096, 2048, 0.0625, P, 0, None, P, ws - 1, stream) == 4
    assert lib.mla_sparse_attn_decode(P, P, P, P, 8, 4096, 2048, 0.0625, P, 1, None, None, ws, stream) == 1
    assert lib.mla_sparse_attn_decode(P, P, P, P, 8, 4096, 2048, 0.0625, P, -1, None, P, ws, stream) == 1
    # paged caches: (block_table, bt_stride, page_size, num_pages) geometry
    idx_paged = lib.dsa_indexer_scores_paged
    assert idx_paged(P, P, P, P, P, None, 4, 64, 8, 1, 1, 256, P, 256, stream) == 1        # no table
    assert idx_paged(P, P, P, P, P, P, 4, 48, 8, 1, 1, 192, P, 192, stream) == 2           # not a power of two
    assert idx_paged(P, P, P, P, P, P, 4, 8, 8, 1, 1, 32, P, 32, stream) == 2              # below 16 rows
    assert idx_paged(P, P, P, P, P, P, 4, 64, 8, 1, 1, 257, P, 260, stream) == 1           # Nmax > 4 pages
    assert idx_paged(P, P, P, P, P, P, 4, 65536, 1 << 16, 1, 1, 256, P, 256, stream) == 2  # pool rows > 2^31-1
    assert idx_paged(P, P + 2, P, P, P, P, 4, 64, 8, 1, 1, 256, P, 256, stream) == 3       # k_pool misaligned
    dec_paged = lib.mla_sparse_attn_decode_paged
    assert dec_paged(P, P, P, P, 4, 64, 8, P, 8, 256, 2048, 0.0625, P, 0, None, P, ws - 1, stream) == 4
    assert dec_paged(P, P, P, P, 0, 64, 8, P, 8, 256, 2048, 0.0625, P, 0, None, P, ws, stream) == 1
    assert dec_paged(P, P, P, P, 4, 100, 8, P, 8, 256, 2048, 0.0625, P, 0, None, P, ws, stream) == 2
    assert dec_paged(P, P, P, P, 4, 64, 8, P, 8, 256, 0, 0.0625, P, 0, None, P, ws, stream) == 2
    pre_paged = lib.mla_sparse_attn_prefill_paged
    assert pre_paged(P, P, None, 64, 8, P, 4, 256, 32, 0.0625, P, 0, None, None, 0, stream) == 1       # no table
    assert pre_paged(P, P, P, 48, 8, P, 4, 256, 32, 0.0625, P, 0, None, None, 0, stream) == 2         # page size
    assert pre_paged(P, P, P, 64, 8, P, 4, 256, 4096, 0.0625, P, 0, None, None, 0, stream) == 2       # top_k
    assert pre_paged(P, P + 4, P, 64, 8, P, 4, 256, 32, 0.0625, P, 0, None, None, 0, stream) == 3     # kv_pool
    # value up-projection
    assert lib.mla_value_up_proj(None, P, 4, P, stream) == 1
    assert lib.mla_value_up_proj(P, P, 0, P, stream) == 1
    assert lib.mla_value_up_proj(P, P, 1 << 30, P, stream) == 2                    # R * 64 > 2^31 - 1
    assert lib.mla_value_up_proj(P, P + 8, 4, P, stream) == 3
    assert lib.mla_value_up_proj(P, P, 4, P + 2, stream) == 3
    code = ctypes.c_int32(0)
    assert lib.dsa_device_status(None, None, 0) == 1


def test_valid_call_without_gpu_reports_instead_of_crashing(lib):
    """With no usable device a valid call returns a CUDA / device error code."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    P = 4096
    rc = lib.dsa_indexer_scores(P, P, P, P, P, 1, 1, 16, P, 16, None)
    assert rc in (5, 8)


def test_package_fails_loudly_without_library(tmp_path):
    from deepseek_sparse_attention_indexer_gb300 import _lib
    saved = _lib._lib
    try:
        _lib._lib = None
        with pytest.raises(RuntimeError, match="missing"):
            _lib.load(str(tmp_path / "nope.so"))
    finally:
        _lib._lib = saved


def test_wait_timeout_selftest_validates_before_any_launch(lib):
    """The failure-detection self-test rejects a spin flag other than 0/1 and a limit outside
    (0, 1 s] on the host (DSA_ERR_INVALID_ARG = 1), before touching the device."""
    import ctypes
    f = lib.dsa_selftest_wait_timeout
    assert f(2, ctypes.c_uint64(1000000), None) == 1
    assert f(-1, ctypes.c_uint64(1000000), None) == 1
    assert f(0, ctypes.c_uint64(0), None) == 1
    assert f(1, ctypes.c_uint64(1000000001), None) == 1
