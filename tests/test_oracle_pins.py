"""Pins for the float64 CPU oracle: checks against what the pages and the
mathematics fix, none of which reuses the oracle's own code.

* indexer: hand-worked example, exact integer recomputation on the grid,
  single-head / zero-weight special cases, the causal mask;
* top-k: hand-worked example, brute force over all K-subsets on tiny rows,
  numpy's lexsort as an independent library routine, permutation invariance,
  the "query before position top_k keeps every earlier key" rule;
* attention: closed form on two keys, dense causal softmax attention (scipy)
  whenever top_k covers every causal key, one-key and zero-query cases,
  invariance to the order of the selected indices;
* value up-projection: permutation weights (pure selection), prefix-sum
  weights (numpy cumsum), independence of heads and rows;
* indexer layer schedule: the pages' 8-layer example and its structure.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import scipy.special

from deepseek_sparse_attention_indexer_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf(x):
    return W.f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def _f(x):
    return float("-inf") if x == "-inf" else (-0.0 if x == "-0.0" else float(x))


# ----------------------------------------------------------------------------- indexer

def test_indexer_hand_example(oracle_mod):
    g = json.load(open(os.path.join(GOLDEN, "indexer_hand_example.json")))
    qI = _bf(g["qI"])[None, None]            # [1,1,Hi,Di]
    kI = _bf(g["kI"])[None]                  # [1,N,Di]
    w = np.asarray(g["w"], np.float32)[None, None]
    q_pos0 = np.array([g["q_pos"]], np.int32)
    kv_len = np.array([kI.shape[1]], np.int32)
    S = oracle_mod.indexer(qI, kI, w, q_pos0, kv_len)
    exp = np.array([_f(v) for v in g["expected_S"]])
    np.testing.assert_array_equal(S[0], exp)


def _int_grid(rng, shape):
    return rng.integers(-8, 9, size=shape).astype(np.int64)


@pytest.mark.parametrize("B,L,N,p0,Hi,Di", [(1, 7, 29, 22, 32, 128), (2, 5, 40, 3, 5, 16),
                                             (3, 1, 17, 16, 32, 128)])
def test_indexer_exact_integer_grid(oracle_mod, B, L, N, p0, Hi, Di):
    """On the 2^-3 / 2^-4 grid, 1024*S is an integer computed here in int64."""
    rng = np.random.default_rng(B * 1000 + L * 10 + N)
    qi_i = _int_grid(rng, (B, L, Hi, Di))
    ki_i = _int_grid(rng, (B, N, Di))
    w_i = _int_grid(rng, (B, L, Hi))
    q_pos0 = rng.integers(0, max(1, N - L + 1), size=B).astype(np.int32)
    q_pos0[0] = min(p0, N - L)
    kv_len = np.minimum(q_pos0 + L, N).astype(np.int32)
    kv_len[-1] = N                      # one batch whose cache runs past its queries
    qI = _bf(qi_i / 8.0)
    kI = _bf(ki_i / 8.0)
    w = (w_i / 16.0).astype(np.float32)
    S = oracle_mod.indexer(qI, kI, w, q_pos0, kv_len).reshape(B, L, N)
    dots = np.einsum("blhd,bnd->blhn", qi_i, ki_i)           # 64 * q.k
    s_int = np.einsum("blh,blhn->bln", w_i, np.maximum(dots, 0))  # 1024 * S
    for b in range(B):
        for i in range(L):
            last = min(int(q_pos0[b]) + i, int(kv_len[b]) - 1)
            j = np.arange(N)
            exp = np.where(j <= last, s_int[b, i] / 1024.0, -np.inf)
            np.testing.assert_array_equal(S[b, i], exp)


def test_indexer_special_cases(oracle_mod):
    rng = np.random.default_rng(5)
    B, L, N, Hi, Di = 1, 3, 11, 32, 128
    qf = rng.integers(-8, 9, (B, L, Hi, Di)) / 8.0
    kf = rng.integers(-8, 9, (B, N, Di)) / 8.0
    q_pos0 = np.array([8], np.int32)
    kv_len = np.array([N], np.int32)
    # all weights zero -> every causal score is zero
    S = oracle_mod.indexer(_bf(qf), _bf(kf), np.zeros((B, L, Hi), np.float32), q_pos0, kv_len)
    for i in range(L):
        assert np.all(S[i, : 9 + i] == 0.0)
        assert np.all(np.isneginf(S[i, 9 + i:]))
    # a single head with weight 1 -> relu of a plain matrix product
    w = np.zeros((B, L, Hi), np.float32)
    w[..., 17] = 1.0
    S = oracle_mod.indexer(_bf(qf), _bf(kf), w, q_pos0, kv_len)
    ref = np.maximum(qf[0, :, 17, :] @ kf[0].T, 0.0)
    for i in range(L):
        np.testing.assert_array_equal(S[i, : 9 + i], ref[i, : 9 + i])
    # queries only non-positive, keys only non-negative -> relu kills everything
    S = oracle_mod.indexer(_bf(-np.abs(qf)), _bf(np.abs(kf)), np.ones((B, L, Hi), np.float32),
                           q_pos0, kv_len)
    assert np.all(S[0, :9] == 0.0)


# ----------------------------------------------------------------------------- top-k

def test_topk_hand_example(oracle_mod):
    g = json.load(open(os.path.join(GOLDEN, "topk_hand_example.json")))
    S = np.array([[_f(v) for v in row] for row in g["scores"]], np.float32)
    R = S.shape[0]
    # every row is its own batch so each gets its own position
    q_pos0 = np.array(g["q_pos"], np.int32)
    kv_len = np.full(R, S.shape[1], np.int32)
    idx = oracle_mod.topk(S, q_pos0, kv_len, B=R, L=1, K=g["top_k"])
    np.testing.assert_array_equal(idx, np.array(g["expected_idx"], np.int32))


def _brute_topk(s, K):
    """Among all K-subsets with the largest score sum, the lexicographically
    smallest ascending index tuple (this is the lower-index tie rule)."""
    best, best_key = None, None
    for comb in itertools.combinations(range(len(s)), K):
        tot = sum(float(s[j]) for j in comb)
        key = (-tot, comb)
        if best_key is None or key < best_key:
            best, best_key = comb, key
    return list(best)


def test_topk_brute_force_tiny(oracle_mod):
    rng = np.random.default_rng(11)
    for trial in range(60):
        n = int(rng.integers(1, 11))
        K = int(rng.integers(1, 9))
        vals = rng.integers(-3, 4, size=n).astype(np.float32) / 2  # many ties
        S = vals[None, :]
        idx = oracle_mod.topk(S, np.array([n - 1], np.int32), np.array([n], np.int32), 1, 1, K)[0]
        if n <= K:
            exp = list(range(n)) + [-1] * (K - n)
        else:
            exp = _brute_topk(vals, K)
        assert list(idx) == exp, (vals, K, idx, exp)


def test_topk_matches_lexsort_with_ties(oracle_mod):
    rows, n, K = 24, 700, 64
    S = W.random_scores(rows, n, seed=3)
    q_pos0 = np.array([n - rows], np.int32)
    kv_len = np.array([n], np.int32)
    idx = oracle_mod.topk(S, q_pos0, kv_len, 1, rows, K)
    for r in range(rows):
        m = n - rows + r + 1
        s = S[r, :m].astype(np.float64) + 0.0      # +0.0 folds -0.0 into +0.0
        order = np.lexsort((np.arange(m), -s))     # score desc, then index asc
        exp = np.sort(order[:K])
        np.testing.assert_array_equal(idx[r], exp)


def test_topk_permutation_invariance(oracle_mod):
    """Permuting keys permutes the chosen set (a unique K-th score here)."""
    rng = np.random.default_rng(2)
    n, K = 300, 40
    s = rng.permutation(n).astype(np.float32)          # distinct scores
    perm = rng.permutation(n)
    a = oracle_mod.topk(s[None], np.array([n - 1], np.int32), np.array([n], np.int32), 1, 1, K)[0]
    b = oracle_mod.topk(s[perm][None], np.array([n - 1], np.int32), np.array([n], np.int32), 1, 1, K)[0]
    assert set(a.tolist()) == set(perm[b].tolist())


def test_topk_early_queries_take_every_key(oracle_mod):
    L, K, N = 40, 16, 40
    S = np.random.default_rng(0).standard_normal((L, N)).astype(np.float32)
    idx = oracle_mod.topk(S, np.array([0], np.int32), np.array([N], np.int32), 1, L, K)
    for i in range(L):
        if i + 1 <= K:
            assert list(idx[i]) == list(range(i + 1)) + [-1] * (K - i - 1)
        else:
            assert len(set(idx[i].tolist())) == K and idx[i].max() <= i


# ----------------------------------------------------------------------------- attention

def test_attention_two_key_closed_form(oracle_mod):
    """H=1, D=66 (Dv=2): scores [0, 1] with scale 1 -> weights 1/(1+e), e/(1+e)."""
    q = np.zeros((1, 1, 66), np.float32)
    q[0, 0, 0] = 1.0
    kv = np.zeros((1, 2, 66), np.float32)
    kv[0, 0, :2] = [0.0, 2.0]
    kv[0, 1, :2] = [1.0, -4.0]
    out, lse = oracle_mod.attention(_bf(q), _bf(kv), np.array([[0, 1]], np.int32),
                                    np.zeros(1, np.int32), 1.0)
    e = math.e
    assert out[0, 0, 0] == pytest.approx(e / (1 + e), rel=1e-15)
    assert out[0, 0, 1] == pytest.approx((2.0 - 4.0 * e) / (1 + e), rel=1e-15)
    assert lse[0, 0] == pytest.approx(math.log(1 + e), rel=1e-15)


def _dense_causal(qf, kvf, p, scale):
    """Textbook dense softmax attention of one query over keys 0..p (scipy)."""
    s = scale * (qf @ kvf[: p + 1].T)                       # [H, p+1]
    a = scipy.special.softmax(s, axis=-1)
    return a @ kvf[: p + 1, :512], scipy.special.logsumexp(s, axis=-1)


def test_attention_sparse_equals_dense_when_topk_covers(oracle_mod):
    wl = W.custom("t", B=1, L=6, p0=20, N=26, top_k=32, seed=9)
    q, kv = W.make_attention_inputs(wl)
    qf = W.bf16_bits_to_f32(q).astype(np.float64)
    kvf = W.bf16_bits_to_f32(kv).astype(np.float64)
    idx = np.full((wl.L, wl.top_k), -1, np.int32)
    for i in range(wl.L):
        idx[i, : wl.p0 + i + 1] = np.arange(wl.p0 + i + 1)
    out, lse = oracle_mod.attention(q[0], kv, idx, np.zeros(wl.L, np.int32), W.SCALE)
    for i in range(wl.L):
        o_ref, l_ref = _dense_causal(qf[0, i], kvf[0], wl.p0 + i, W.SCALE)
        np.testing.assert_allclose(out[i], o_ref, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(lse[i], l_ref, rtol=1e-12, atol=1e-12)


def test_attention_special_cases(oracle_mod):
    wl = W.custom("t", B=2, L=1, p0=0, N=50, top_k=8, seed=4)
    q, kv = W.make_attention_inputs(wl)
    kvf = W.bf16_bits_to_f32(kv).astype(np.float64)
    rb = np.array([0, 1], np.int32)
    # one selected key -> that key's latent row, lse = its scaled score
    idx = np.full((2, 8), -1, np.int32)
    idx[0, 3] = 17
    idx[1, 0] = 42
    out, lse = oracle_mod.attention(q[:, 0], kv, idx, rb, W.SCALE)
    np.testing.assert_array_equal(out[0, 5], kvf[0, 17, :512])
    np.testing.assert_array_equal(out[1, 63], kvf[1, 42, :512])
    qf = W.bf16_bits_to_f32(q).astype(np.float64)
    assert lse[0, 5] == pytest.approx(W.SCALE * float(qf[0, 0, 5] @ kvf[0, 17]), rel=1e-13)
    # zero query -> plain mean of the selected latent rows, lse = log(n)
    sel = np.array([[1, 4, 9, 30, 31, 2, 0, 49], [5, 6, 7, -1, -1, -1, -1, -1]], np.int32)
    out, lse = oracle_mod.attention(np.zeros_like(q[:, 0]), kv, sel, rb, W.SCALE)
    np.testing.assert_allclose(out[0, 0], kvf[0, sel[0], :512].mean(0), rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(out[1, 0], kvf[1, sel[1, :3], :512].mean(0), rtol=1e-13, atol=1e-14)
    assert lse[1, 0] == pytest.approx(math.log(3), rel=1e-14)
    # no key selected -> zero output, lse -inf
    out, lse = oracle_mod.attention(q[:, 0], kv, np.full((2, 8), -1, np.int32), rb, W.SCALE)
    assert np.all(out == 0.0) and np.all(np.isneginf(lse))


def test_attention_order_of_indices_irrelevant(oracle_mod):
    wl = W.custom("t", B=1, L=2, p0=100, N=200, top_k=64, seed=6)
    q, kv = W.make_attention_inputs(wl)
    rng = np.random.default_rng(1)
    idx = np.stack([np.sort(rng.choice(200, 64, replace=False)) for _ in range(2)]).astype(np.int32)
    idx[1, 50:] = -1
    perm = idx.copy()
    for r in range(2):
        perm[r] = rng.permutation(perm[r])
    a, la = oracle_mod.attention(q[0], kv, idx, np.zeros(2, np.int32), W.SCALE)
    b, lb = oracle_mod.attention(q[0], kv, perm, np.zeros(2, np.int32), W.SCALE)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(la, lb, rtol=1e-13)


# ----------------------------------------------------------------------------- generator

def test_generator_grid_and_ties():
    wl = W.WORKLOADS["tiny_1k"]
    qi, ki, w = W.make_indexer_inputs(wl)
    qf = W.bf16_bits_to_f32(qi) * 8
    assert np.all(qf == np.round(qf)) and qf.min() >= -8 and qf.max() <= 8
    assert np.all(w * 16 == np.round(w * 16))
    wl2 = W.custom("d", B=1, L=1, p0=999, N=1000, top_k=10, seed=3, dup_frac=0.05)
    _, ki2, _ = W.make_indexer_inputs(wl2)
    rows = {r.tobytes() for r in ki2[0]}
    assert len(rows) <= 1000 - 45          # about 50 keys copy another key's row
    a, b = W.make_attention_inputs(wl)
    a2, b2 = W.make_attention_inputs(wl)
    assert np.array_equal(a, a2) and np.array_equal(b, b2)


# ----------------------------------------------------------------------------- paged caches

def test_unpage_hand_example(oracle_mod):
    """Pool row r holds the value r (one column); pages of 2 rows.  Sequence 0 has 3 keys in
    pool pages 3 then 0; sequence 1 has 4 keys in pages 1 then 2; page 4 is never referenced.
    Worked by hand: keys of sequence 0 are pool rows 6, 7, 0; of sequence 1 rows 2, 3, 4, 5."""
    pool = np.arange(10, dtype=np.int64).reshape(10, 1)
    table = np.array([[3, 0], [1, 2]], np.int32)
    got = oracle_mod.unpage(pool, table, 2, [3, 4], 4)
    expect = np.array([[[6], [7], [0], [0]], [[2], [3], [4], [5]]])
    np.testing.assert_array_equal(got, expect)
    # an entry outside the pool reads as zeros; entries past kv_len are never read
    bad = np.array([[3, 9], [1, -1]], np.int32)
    got = oracle_mod.unpage(pool, bad, 2, [3, 2], 4)
    np.testing.assert_array_equal(got, np.array([[[6], [7], [0], [0]], [[2], [3], [0], [0]]]))


def test_paginate_then_unpage_is_identity(oracle_mod):
    """The seeded page scatter of the input generator and the oracle's page lookup are
    inverses on every key a sequence holds, for page sizes below, at and above a tile."""
    rng = np.random.default_rng(5)
    dense = W.f32_to_bf16_bits(rng.standard_normal((3, 300, 8), dtype=np.float32))
    kv_len = np.array([300, 17, 129])
    for ps in (16, 128, 256):
        pool, table = W.paginate(dense, kv_len, ps, extra_pages=3, seed=ps)
        assert pool.shape == ((sum(-(-n // ps) for n in kv_len) + 3) * ps, 8)
        used = table[table >= 0]
        assert len(set(used.tolist())) == len(used)          # no page shared by two places
        back = oracle_mod.unpage(pool, table, ps, kv_len, 300)
        for b, n in enumerate(kv_len):
            np.testing.assert_array_equal(back[b, :n], dense[b, :n])
            assert not back[b, n:].any()


# ----------------------------------------------------------------------------- value up-projection

def _bf16_f64(bits):
    return W.bf16_bits_to_f32(bits).astype(np.float64)


def test_value_up_proj_permutation_weights(oracle_mod):
    """wv[h, e, d] = 1 exactly when d = sigma_h(e) (a different permutation per head): the
    projection only selects, v[r, h, e] = o[r, h, sigma_h(e)].  A transposed weight, a
    wrong head or a dropped term changes the result."""
    rng = np.random.default_rng(11)
    R, H, Dv, E = 5, 3, 24, 10
    o = _bf(rng.standard_normal((R, H, Dv)))
    sig = np.stack([rng.permutation(Dv)[:E] for _ in range(H)])
    wv = np.zeros((H, E, Dv), np.float32)
    for h in range(H):
        wv[h, np.arange(E), sig[h]] = 1.0
    v = oracle_mod.value_up_proj(o, _bf(wv))
    of = _bf16_f64(o)
    expect = np.stack([of[:, h, sig[h]] for h in range(H)], axis=1)
    np.testing.assert_array_equal(v, expect)


def test_value_up_proj_prefix_sum_weights(oracle_mod):
    """wv[h, e, d] = c_h for d <= e, else 0, with c_h a power of two: v[r, h, e] is c_h times
    the prefix sum of the head's latent row up to e (numpy cumsum; exact in float64 for
    bf16 inputs of this range)."""
    rng = np.random.default_rng(12)
    R, H, Dv, E = 4, 4, 64, 64
    o = _bf(rng.standard_normal((R, H, Dv)))
    c = np.array([1.0, 0.5, 2.0, 0.25], np.float32)
    tri = np.tril(np.ones((E, Dv), np.float32))          # row e: ones at d <= e
    wv = c[:, None, None] * tri[None]
    v = oracle_mod.value_up_proj(o, _bf(wv))
    expect = np.cumsum(_bf16_f64(o), axis=2) * c.astype(np.float64)[None, :, None]
    np.testing.assert_array_equal(v, expect)


def test_value_up_proj_heads_are_independent(oracle_mod):
    """Zeroing every head's weights but one zeroes every other head's output and leaves that
    head's output as it was; the rows are independent too (a row subset gives the same rows)."""
    R, H = 6, 64
    o, wv = W.make_value_proj_inputs(R, seed=13)
    o, wv = o[:, :, :], wv[:, :32, :]                     # E = 32 keeps the pin fast
    full = oracle_mod.value_up_proj(o, wv)
    only = np.zeros_like(wv)
    only[17] = wv[17]
    v = oracle_mod.value_up_proj(o, only)
    assert not np.delete(v, 17, axis=1).any()
    np.testing.assert_array_equal(v[:, 17], full[:, 17])
    sub = oracle_mod.value_up_proj(o, wv, rows=[1, 4, 5])
    np.testing.assert_array_equal(sub, full[[1, 4, 5]])


# ----------------------------------------------------------------------------- indexer layer schedule

def test_indexer_schedule_matches_the_pages_example():
    """The first 8 GLM-5.3 layers (index_topk_freq 4, index_skip_topk_offset 3): layers
    0, 1, 2 and 6 run the indexer, 3, 4, 5 and 7 reuse a selection (worked example printed
    on the exo page; stored under tests/golden with its citation)."""
    from deepseek_sparse_attention_indexer_gb300 import _build, _lib
    _build.build()
    g = json.load(open(os.path.join(GOLDEN, "indexer_layer_schedule.json")))
    f, off = g["index_topk_freq"], g["index_skip_topk_offset"]
    for layer in g["indexer_layers"]:
        assert _lib.indexer_source_layer(layer, f, off) == layer
    for layer in g["shared_layers"]:
        assert _lib.indexer_source_layer(layer, f, off) != layer


@pytest.mark.parametrize("freq,off", [(4, 3), (1, 1), (2, 5), (3, 1)])
def test_indexer_schedule_reuses_the_nearest_indexer_layer(freq, off):
    """Every shared layer reuses the nearest earlier layer that ran the indexer, and runs of
    shared layers between two indexer layers are freq - 1 long after the offset."""
    from deepseek_sparse_attention_indexer_gb300 import _build, _lib
    _build.build()
    src = [_lib.indexer_source_layer(layer, freq, off) for layer in range(40)]
    runs = [layer for layer in range(40) if src[layer] == layer]
    assert runs[:off] == list(range(off))
    for layer in range(40):
        if src[layer] != layer:
            assert src[layer] < layer and src[src[layer]] == src[layer]
            assert not any(src[m] == m for m in range(src[layer] + 1, layer))
    after = [layer for layer in runs if layer >= off]
    assert all(b - a == freq for a, b in zip(after, after[1:]))
    assert not after or after[0] == off + freq - 1
    for bad in [(-1, freq, off), (0, 0, off), (0, freq, 0)]:
        with pytest.raises(ValueError):
            _lib.indexer_source_layer(*bad)
