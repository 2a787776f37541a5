"""The allocation-free decode entry point, checked against the regular one.

mla_sparse_attn_decode_noalloc exists for callers that may not allocate
device memory (plugins inside an engine that owns all device memory through
its own pool, or decode loops where an allocation, which can synchronise the
device, is forbidden).  It keeps the split partials in a fixed scratch array
inside the library instead of a caller workspace.  Here it is called through
the C ABI twice in a row (the second call reuses the scratch the first one
left behind) and each result must match mla_sparse_attn_decode within the
attention tolerance of the parity tests.  This file is collected last.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from deepseek_sparse_attention_indexer_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from deepseek_sparse_attention_indexer_gb300 import _build, _lib
    _build.build()
    _lib.load()
    return _lib


def _dev(a):
    a = np.ascontiguousarray(a)
    return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).cuda()


def _close(got, ref):
    got = got.float().cpu().numpy().astype(np.float64)
    ref = ref.float().cpu().numpy().astype(np.float64)
    err = np.abs(got - ref)
    assert err.max() <= 1e-2 * np.abs(ref).max()
    assert err.sum() / np.abs(ref).sum() <= 2e-3


def _bf16_bits(t):
    return t.to(torch.bfloat16).view(torch.int16)


# B = 63 fills the whole scratch (one split per sequence); B = 32 is the first batch where the
# scratch, not the SM count, caps the splits at one per sequence.
CASES = [W.WORKLOADS["decode_b8"], W.WORKLOADS["decode_b1"],
         W.custom("decode_b63", B=63, L=1, p0=4095, N=4096, top_k=2048, seed=1063),
         W.custom("decode_b32", B=32, L=1, p0=4095, N=4096, top_k=2048, seed=1032)]


@pytest.mark.parametrize("wl", CASES, ids=lambda w: w.name)
def test_noalloc_decode_matches_workspace_decode_twice(dsa, wl):
    qi, ki, w = W.make_indexer_inputs(wl)
    q, kv = W.make_attention_inputs(wl)
    q_pos0, kv_len = W.positions(wl)
    d_pos, d_len = _dev(q_pos0), _dev(kv_len)
    S = dsa.indexer_scores(_dev(qi), _dev(ki), _dev(w), d_pos, d_len)
    idx = dsa.topk(S, d_pos, d_len, wl.N, wl.top_k)[:, 0].contiguous()
    dq, dkv = _dev(q[:, 0]), _dev(kv)
    ref, ref_lse = dsa.mla_sparse_attn_decode(dq, dkv, d_len, idx, W.SCALE, want_lse=True)
    out = torch.empty_like(ref)
    lse = torch.empty_like(ref_lse)
    for _ in range(2):
        out.zero_()
        lse.zero_()
        dsa.mla_sparse_attn_decode_noalloc(dq, dkv, d_len, idx, W.SCALE, out=out, lse=lse)
        torch.cuda.synchronize()
        _close(out, ref)
        np.testing.assert_allclose(lse.cpu().numpy(), ref_lse.cpu().numpy(), rtol=1e-5, atol=1e-5)
    # the bf16 output is the float32 result rounded to nearest even
    out16 = dsa.mla_sparse_attn_decode_noalloc(dq, dkv, d_len, idx, W.SCALE, out_dtype=torch.bfloat16)
    again = dsa.mla_sparse_attn_decode_noalloc(dq, dkv, d_len, idx, W.SCALE)
    torch.cuda.synchronize()
    assert torch.equal(out16.view(torch.int16), _bf16_bits(again))
    assert dsa.device_status() == 0


def test_noalloc_rejects_batches_beyond_the_scratch(dsa):
    P = torch.empty(16, dtype=torch.uint8, device="cuda").data_ptr()
    rc = dsa.load().mla_sparse_attn_decode_noalloc(P, P, P, P, 64, 4096, 2048, 0.0625, P, 0, None, None)
    assert rc == 9        # DSA_ERR_SCRATCH_TOO_SMALL, nothing launched
