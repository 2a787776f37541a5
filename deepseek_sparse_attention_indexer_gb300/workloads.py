"""Seeded synthetic inputs for the DSA indexer -> top-k -> sparse absorbed-MLA path.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic.  Both the CUDA path (through the C-ABI) and the float64
CPU oracle read the very same arrays, so the two sides see identical bits.

Shapes follow the GLM-5.x / DeepSeek sparse-attention layer traced on the pages
(SlimServe "GLM52_PIPELINE_TRACE.md", Config line and section 6 "Attention core
(absorbed MLA)"; exo PR #2539, section "Prefill"):

* indexer query  qI  [B, L, 32, 128]  bf16 (32 indexer heads, head dim 128)
* indexer key    kI  [B, N, 128]      bf16
* head weights   w   [B, L, 32]       f32
* absorbed query q   [B, L, 64, 576]  bf16 ([q_nope.wk_b 512 | q_pe 64])
* latent KV row  kv  [B, N, 576]      bf16 ([kv_cmpr 512 | k_pe 64])
* attention out  o   [R, 64, 512]     bf16 (input of the value up-projection)
* value weights  wv  [64, 256, 512]   bf16 (wv_b: one 512-wide row per value feature)

Value recipes (fixed per workload, seeded):

* q, kv: standard normal drawn in float32 with numpy's PCG64 generator and
  rounded to bf16 with round-to-nearest-even.  The 64k workload draws the rope
  slice kv[..., 512:576] with standard deviation 0.5.
* qI, kI: integers uniform on [-8, 8] times 2^-3; w: integers uniform on
  [-8, 8] times 2^-4.  Every indexer product and head sum is then an exact
  multiple of 2^-10 far inside float32's 24-bit mantissa, so float32 scores
  are exact and the top-k sets are unique under the lower-index tie rule.
* o: standard normal rounded to bf16; wv: standard normal times 2^-5 rounded
  to bf16 (so each 512-term value sum has standard deviation about 0.7).
* The 64k workload copies indexer-key rows onto 5% of the keys (distinct
  seeded targets, seeded sources), so those keys score exactly like another
  key for every query that sees both: a tie stress for the top-2048 boundary.

numpy's PCG64 stream and the integer bf16 rounding below are platform
independent, so x86 and Arm hosts produce identical bytes for a seed.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, Optional

import numpy as np

N_IDX_HEADS = 32      # indexer heads
IDX_DIM = 128         # indexer head dim
N_HEADS = 64          # attention query heads
QK_DIM = 576          # kv_lora_rank 512 + qk_rope_head_dim 64
V_DIM = 512           # kv_lora_rank
V_HEAD_DIM = 256      # v_head_dim (value width per head after the wv_b up-projection)
SCALE = 1.0 / 16.0    # 1/sqrt(qk_nope_head_dim 192 + qk_rope_head_dim 64)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    L: int
    p0: int
    N: int
    top_k: int
    seed: int
    rope_std: float = 1.0
    dup_frac: float = 0.0
    desc: str = ""
    page_size: int = 0     # > 0: the caches live in pages of this many rows (see paginate)

    @property
    def n_rows(self) -> int:
        return self.B * self.L


WORKLOADS: Dict[str, Workload] = {
    "tiny_1k": Workload(
        "tiny_1k", B=1, L=64, p0=960, N=1024, top_k=256, seed=1001,
        desc="64 queries at positions 960..1023 over 1024 keys, top_k 256"),
    "first_chunk_4k": Workload(
        "first_chunk_4k", B=1, L=4096, p0=0, N=4096, top_k=2048, seed=1002,
        desc="first 4096-query prefill chunk at positions 0..4095, top_k 2048"),
    "prefill_16k": Workload(
        "prefill_16k", B=1, L=4096, p0=12288, N=16384, top_k=2048, seed=1003,
        desc="4096 queries at positions 12288..16383 over 16384 keys, top_k 2048"),
    "decode_b8": Workload(
        "decode_b8", B=8, L=1, p0=4095, N=4096, top_k=2048, seed=1004,
        desc="8 sequences, one query each at position 4095 over 4096 keys"),
    "decode_b4": Workload(
        "decode_b4", B=4, L=1, p0=4095, N=4096, top_k=2048, seed=1014,
        desc="4 sequences, one query each at position 4095 over 4096 keys"),
    "decode_b1": Workload(
        "decode_b1", B=1, L=1, p0=4095, N=4096, top_k=2048, seed=1024,
        desc="1 sequence, one query at position 4095 over 4096 keys"),
    "decode_b8_paged": Workload(
        "decode_b8_paged", B=8, L=1, p0=4095, N=4096, top_k=2048, seed=1004, page_size=64,
        desc="decode_b8's sequences with their caches in 64-row pages of a shuffled pool"),
    "prefill_64k": Workload(
        "prefill_64k", B=1, L=4096, p0=61440, N=65536, top_k=2048, seed=1005,
        rope_std=0.5, dup_frac=0.05,
        desc="4096 queries at positions 61440..65535 over 65536 keys, rope "
             "slice std 0.5, 5% duplicated indexer keys, top_k 2048"),
}


def custom(name: str, B: int, L: int, p0: int, N: int, top_k: int, seed: int,
           rope_std: float = 1.0, dup_frac: float = 0.0) -> Workload:
    """A workload with explicit sizes (edge cases: ragged tails, tiny N, ...)."""
    return Workload(name, B, L, p0, N, top_k, seed, rope_std, dup_frac)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest, ties to even) and return the uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bits to float32 (exact)."""
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def _grid(rng: np.random.Generator, shape, step_log2: int) -> np.ndarray:
    ints = rng.integers(-8, 9, size=shape, dtype=np.int32)
    return ints.astype(np.float32) * np.float32(2.0 ** (-step_log2))


def make_indexer_inputs(wl: Workload, seed: Optional[int] = None):
    """qI [B,L,32,128] bf16 bits, kI [B,N,128] bf16 bits, w [B,L,32] f32."""
    rng = np.random.Generator(np.random.PCG64(wl.seed if seed is None else seed))
    qi = f32_to_bf16_bits(_grid(rng, (wl.B, wl.L, N_IDX_HEADS, IDX_DIM), 3))
    ki = f32_to_bf16_bits(_grid(rng, (wl.B, wl.N, IDX_DIM), 3))
    w = _grid(rng, (wl.B, wl.L, N_IDX_HEADS), 4)
    if wl.dup_frac > 0.0:
        n_dup = int(wl.dup_frac * wl.N)
        for b in range(wl.B):
            dst = rng.choice(wl.N, size=n_dup, replace=False)
            src = rng.integers(0, wl.N - 1, size=n_dup)
            src = src + (src >= dst)          # any key other than dst itself
            ki[b, dst] = ki[b, src]
    return qi, ki, w


def make_attention_inputs(wl: Workload, seed: Optional[int] = None):
    """q [B,L,64,576] bf16 bits and kv [B,N,576] bf16 bits."""
    s = (wl.seed if seed is None else seed) + 7919
    rng = np.random.Generator(np.random.PCG64(s))
    q = f32_to_bf16_bits(rng.standard_normal((wl.B, wl.L, N_HEADS, QK_DIM), dtype=np.float32))
    kv32 = rng.standard_normal((wl.B, wl.N, QK_DIM), dtype=np.float32)
    if wl.rope_std != 1.0:
        kv32[..., V_DIM:] *= np.float32(wl.rope_std)
    kv = f32_to_bf16_bits(kv32)
    return q, kv


def make_value_proj_inputs(R: int, seed: int):
    """o [R, 64, 512] bf16 bits (attention-output stand-in) and wv [64, 256, 512] bf16 bits."""
    rng = np.random.Generator(np.random.PCG64(seed))
    o = f32_to_bf16_bits(rng.standard_normal((R, N_HEADS, V_DIM), dtype=np.float32))
    wv = f32_to_bf16_bits(rng.standard_normal((N_HEADS, V_HEAD_DIM, V_DIM), dtype=np.float32)
                          * np.float32(2.0 ** -5))
    return o, wv


def positions(wl: Workload):
    """q_pos0 [B] and kv_len [B] as int32 (query i of batch b sits at q_pos0[b]+i)."""
    q_pos0 = np.full((wl.B,), wl.p0, dtype=np.int32)
    kv_len = np.full((wl.B,), wl.N, dtype=np.int32)
    return q_pos0, kv_len


def random_scores(rows: int, n: int, seed: int, ties: bool = True) -> np.ndarray:
    """A float32 score matrix for testing top-k on its own.

    Values come from a small set of magnitudes (so ties are frequent) mixed with
    continuous draws, signed zeros of both signs, and large magnitudes.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    s = rng.standard_normal((rows, n), dtype=np.float32)
    if ties:
        m = rng.random((rows, n)) < 0.5
        s[m] = np.round(s[m] * 4.0) / 4.0
        z = rng.random((rows, n)) < 0.02
        s[z] = np.where(rng.random(int(z.sum())) < 0.5, np.float32(0.0), np.float32(-0.0))
        big = rng.random((rows, n)) < 0.01
        s[big] *= np.float32(1e30)
    return s


def paginate(dense: np.ndarray, kv_len, page_size: int, extra_pages: int = 0, seed: int = 0):
    """Lay dense per-sequence cache rows [B, Nmax, D] out as a paged pool.

    Every page that holds a key j < kv_len[b] goes to a distinct, seeded-random
    page of the pool; `extra_pages` more pages (never referenced) and the tail
    rows of each sequence's last page hold seeded junk, so a wrong page lookup
    changes the result.  Table entries of pages past kv_len[b] are -1.
    Returns (pool [num_pages * page_size, D], block_table int32 [B, ceil(Nmax / page_size)]).
    """
    B, Nmax, D = dense.shape
    kv_len = np.asarray(kv_len, np.int64)
    stride = -(-Nmax // page_size)
    used = [int(-(-int(n) // page_size)) for n in kv_len]
    num_pages = sum(used) + extra_pages
    rng = np.random.default_rng(seed)
    perm = rng.permutation(num_pages)
    if dense.dtype == np.uint16:
        pool = f32_to_bf16_bits(rng.standard_normal((num_pages * page_size, D), dtype=np.float32))
    else:
        pool = rng.standard_normal((num_pages * page_size, D)).astype(dense.dtype)
    table = np.full((B, stride), -1, np.int32)
    k = 0
    for b in range(B):
        for lp in range(used[b]):
            page = int(perm[k])
            k += 1
            table[b, lp] = page
            lo = lp * page_size
            hi = min(lo + page_size, int(kv_len[b]))
            pool[page * page_size: page * page_size + hi - lo] = dense[b, lo:hi]
    return pool, table
