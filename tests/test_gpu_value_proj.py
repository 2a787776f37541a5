"""GPU parity of the value up-projection (wv_b) against the float64 oracle.

v[r, h, e] = sum_d o[r, h, d] * wv[h, e, d] with bf16 inputs, float32
accumulation in the tensor cores and a bf16 output.  Tolerance derived from the
arithmetic, per element: the bf16 rounding of the output (relative 2^-9) plus
float32 accumulation error over 512 terms (well inside 2^-14 times the sum of
the absolute terms), so |gpu - ref| <= 2^-8 |ref| + 2^-14 sum_d |o_d w_d|;
plus the attention's global bound (max err <= 1e-2 max|ref|, mean relative
error <= 2e-3).  Sizes span one partial tile, several full tiles with a ragged
tail, and the 4096-query chunk (sampled rows) in the launch the benchmark
times.
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
    _lib.device_status(reset=True)
    return _lib


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


def to_f64(v_gpu):
    bits = v_gpu.view(torch.int16).cpu().numpy().view(np.uint16)
    return W.bf16_bits_to_f32(bits).astype(np.float64)


def check(gpu, ref, abs_terms, what):
    err = np.abs(gpu - ref)
    bound = 2.0 ** -8 * np.abs(ref) + 2.0 ** -14 * abs_terms
    worst = np.argmax(err - bound)
    assert (err <= bound).all(), f"{what}: err {err.flat[worst]:.3e} > bound {bound.flat[worst]:.3e}"
    assert err.max() <= 1e-2 * np.abs(ref).max(), what
    assert err.sum() / np.abs(ref).sum() <= 2e-3, what


def run(dsa, o, wv, pad_rows=0):
    R = o.shape[0]
    v = torch.full((R + pad_rows, 64, 256), -7.0, dtype=torch.bfloat16, device="cuda")
    dsa.mla_value_up_proj(dev(o), dev(wv), v=v[:R])
    torch.cuda.synchronize()
    assert dsa.device_status(reset=True) == 0
    if pad_rows:
        assert (v[R:] == -7.0).all(), "rows past R were written"
    return to_f64(v[:R])


@pytest.mark.parametrize("R", [1, 8, 128, 300, 1000])
def test_value_up_proj_full_compare(dsa, oracle_mod, R):
    o, wv = W.make_value_proj_inputs(R, seed=2000 + R)
    gpu = run(dsa, o, wv, pad_rows=3)
    th = oracle_mod.default_threads()
    ref = oracle_mod.value_up_proj(o, wv, threads=th)
    abs_terms = oracle_mod.value_up_proj(o & np.uint16(0x7FFF), wv & np.uint16(0x7FFF), threads=th)
    check(gpu, ref, abs_terms, f"R={R}")


def test_value_up_proj_chunk_sampled_rows(dsa, oracle_mod):
    """The 4096-query chunk (2048 tiles over the persistent CTAs, several tiles per CTA
    through both TMEM accumulators), checked on sampled rows the oracle computes one by one."""
    R = 4096
    o, wv = W.make_value_proj_inputs(R, seed=2096)
    gpu = run(dsa, o, wv)
    rng = np.random.default_rng(0)
    rows = sorted({0, 127, 128, 2047, 4095} | set(rng.choice(R, 11, replace=False).tolist()))
    th = oracle_mod.default_threads()
    ref = oracle_mod.value_up_proj(o, wv, rows=rows, threads=th)
    abs_terms = oracle_mod.value_up_proj(o & np.uint16(0x7FFF), wv & np.uint16(0x7FFF), rows=rows, threads=th)
    check(gpu[rows], ref, abs_terms, "R=4096 sampled")


def test_value_up_proj_selection_weights_are_exact(dsa):
    """Permutation weights make every output a copy of one input element: bit-exact."""
    R = 200
    rng = np.random.default_rng(3)
    o = W.f32_to_bf16_bits(rng.standard_normal((R, 64, 512), dtype=np.float32))
    sig = np.stack([rng.permutation(512)[:256] for _ in range(64)])
    wv = np.zeros((64, 256, 512), np.float32)
    for h in range(64):
        wv[h, np.arange(256), sig[h]] = 1.0
    gpu = run(dsa, o, W.f32_to_bf16_bits(wv))
    of = W.bf16_bits_to_f32(o).astype(np.float64)
    expect = np.stack([of[:, h, sig[h]] for h in range(64)], axis=1)
    np.testing.assert_array_equal(gpu, expect)


def test_value_up_proj_after_attention_chain(dsa, oracle_mod):
    """The chain a layer runs: attention output of the 1k workload straight into the
    up-projection on the device.  Checked against the oracle's up-projection of the oracle's
    own attention output (no GPU value feeds the oracle), within the attention bound."""
    wl = W.WORKLOADS["tiny_1k"]
    q, kv = W.make_attention_inputs(wl)
    qi, ki, w = W.make_indexer_inputs(wl)
    q_pos0, kv_len = W.positions(wl)
    S = dsa.indexer_scores(dev(qi), dev(ki), torch.from_numpy(w).cuda(), torch.from_numpy(q_pos0).cuda(),
                           torch.from_numpy(kv_len).cuda())
    idx = dsa.topk(S, torch.from_numpy(q_pos0).cuda(), torch.from_numpy(kv_len).cuda(), wl.N, wl.top_k)
    out = dsa.mla_sparse_attn_prefill(dev(q[0]), dev(kv[0]), idx[0], W.SCALE, out_dtype=torch.bfloat16)
    _, wv = W.make_value_proj_inputs(1, seed=2001)
    v = dsa.mla_value_up_proj(out, dev(wv))
    torch.cuda.synchronize()
    gpu = to_f64(v)
    th = oracle_mod.default_threads()
    S_ref = oracle_mod.indexer(qi, ki, w, q_pos0, kv_len, threads=th).astype(np.float32)
    idx_ref = oracle_mod.topk(S_ref, q_pos0, kv_len, wl.B, wl.L, wl.top_k, threads=th)
    o_ref, _ = oracle_mod.attention(q[0], kv, idx_ref, np.zeros(wl.L, np.int32), W.SCALE, threads=th)
    # the oracle's up-projection takes bf16 bits: round its attention output as the kernel does
    o_bits = W.f32_to_bf16_bits(o_ref.astype(np.float32))
    ref = oracle_mod.value_up_proj(o_bits, wv, threads=th)
    err = np.abs(gpu - ref)
    assert err.max() <= 1e-2 * np.abs(ref).max()
    # the attention's bound (2e-3) plus the projection's own bf16 rounding (2^-9 ~ 2e-3)
    assert err.sum() / np.abs(ref).sum() <= 4e-3
