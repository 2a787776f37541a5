"""Replicas on disjoint query rows (the path's multi-GPU form): the row blocks cover the chunk
exactly once, and the rows computed rank by rank concatenate to the single-process result.

The CPU tests run two gloo ranks over the float64 oracle; the GPU test runs two processes on the
same device (independent kernels, no device-side waits between them) through the library and
requires the gathered result to be bit-identical to one call over the whole chunk."""
import os
import socket
import sys

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from deepseek_sparse_attention_indexer_gb300 import sharding
from deepseek_sparse_attention_indexer_gb300 import workloads as W


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.parametrize("L,world", [(4096, 2), (4096, 8), (64, 3), (5, 8), (1, 1), (0, 4), (300, 7)])
def test_shard_rows_cover_every_row_once(L, world):
    seen = np.zeros(L, np.int32)
    sizes = []
    prev_stop = 0
    for r in range(world):
        a, b = sharding.shard_rows(L, world, r)
        assert a == prev_stop and a <= b <= L
        seen[a:b] += 1
        sizes.append(b - a)
        prev_stop = b
    assert prev_stop == L and np.all(seen == 1)
    assert max(sizes) - min(sizes) <= 1


def test_shard_positions_keep_each_row_at_its_position():
    for rank in range(3):
        a, b, p = sharding.shard_prefill_positions(12288, 4096, 3, rank)
        assert p == 12288 + a
    with pytest.raises(ValueError):
        sharding.shard_rows(10, 2, 2)


def _oracle_rank(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import oracle
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        wl = W.WORKLOADS["tiny_1k"]
        qi, ki, w = W.make_indexer_inputs(wl)
        q, kv = W.make_attention_inputs(wl)
        q_pos0, kv_len = W.positions(wl)
        a, b, p = sharding.shard_prefill_positions(wl.p0, wl.L, world, rank)
        pos = np.array([p], np.int32)
        # this rank's block of the chunk as a chunk of its own (rows a..b at positions p0 + a ..)
        S = oracle.indexer(qi[:, a:b], ki, w[:, a:b], pos, kv_len)
        idx = oracle.topk(S.astype(np.float32), pos, kv_len, 1, b - a, wl.top_k)
        out, lse = oracle.attention(q[0, a:b], kv, idx, np.zeros(b - a, np.int32), W.SCALE)
        parts = [None] * world
        dist.all_gather_object(parts, (a, b, idx, out, lse))
        if rank == 0:
            results["parts"] = parts
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_oracle_rows_concatenate():
    world = 2
    results = mp.get_context("spawn").Manager().dict()   # no fork once CUDA may be initialised
    mp.spawn(_oracle_rank, args=(world, _free_port(), results), nprocs=world, join=True)
    import oracle
    wl = W.WORKLOADS["tiny_1k"]
    qi, ki, w = W.make_indexer_inputs(wl)
    q, kv = W.make_attention_inputs(wl)
    q_pos0, kv_len = W.positions(wl)
    S = oracle.indexer(qi, ki, w, q_pos0, kv_len)
    idx = oracle.topk(S.astype(np.float32), q_pos0, kv_len, 1, wl.L, wl.top_k)
    out, lse = oracle.attention(q[0], kv, idx, np.zeros(wl.L, np.int32), W.SCALE)
    parts = sorted(results["parts"], key=lambda t: t[0])
    assert parts[0][0] == 0 and parts[-1][1] == wl.L
    np.testing.assert_array_equal(np.concatenate([t[2] for t in parts]), idx)
    np.testing.assert_array_equal(np.concatenate([t[3] for t in parts]), out)
    np.testing.assert_array_equal(np.concatenate([t[4] for t in parts]), lse)


def _gpu_rank(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    from deepseek_sparse_attention_indexer_gb300 import _lib as dsa
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        torch.cuda.set_device(0)
        dsa.load()
        wl = W.custom("shard_chunk", B=1, L=300, p0=1748, N=2048, top_k=256, seed=81)
        qi, ki, w = W.make_indexer_inputs(wl)
        q, kv = W.make_attention_inputs(wl)
        q_pos0, kv_len = W.positions(wl)
        d = lambda x: torch.from_numpy(np.ascontiguousarray(x.view(np.int16) if x.dtype == np.uint16 else x)).cuda()
        a, b, p = sharding.shard_prefill_positions(wl.p0, wl.L, world, rank)
        pos = d(np.array([p], np.int32))
        S = dsa.indexer_scores(d(qi[:, a:b]), d(ki), d(w[:, a:b]), pos, d(kv_len))
        idx = dsa.topk(S, pos, d(kv_len), wl.N, wl.top_k)
        out = dsa.mla_sparse_attn_prefill(d(q[0, a:b]), d(kv[0]), idx[0], W.SCALE)
        torch.cuda.synchronize()
        assert dsa.device_status() == 0
        parts = [None] * world
        dist.all_gather_object(parts, (a, b, S[0, :, : wl.N].cpu().numpy(), idx[0].cpu().numpy(), out.cpu().numpy()))
        if rank == 0:
            results["parts"] = parts
    finally:
        dist.destroy_process_group()


@pytest.mark.gpu
def test_two_replicas_on_disjoint_rows_match_one_call():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from deepseek_sparse_attention_indexer_gb300 import _build, _lib as dsa
    _build.build()
    world = 2
    results = mp.get_context("spawn").Manager().dict()   # no fork once CUDA may be initialised
    mp.spawn(_gpu_rank, args=(world, _free_port(), results), nprocs=world, join=True)
    dsa.load()
    wl = W.custom("shard_chunk", B=1, L=300, p0=1748, N=2048, top_k=256, seed=81)
    qi, ki, w = W.make_indexer_inputs(wl)
    q, kv = W.make_attention_inputs(wl)
    q_pos0, kv_len = W.positions(wl)
    d = lambda x: torch.from_numpy(np.ascontiguousarray(x.view(np.int16) if x.dtype == np.uint16 else x)).cuda()
    S = dsa.indexer_scores(d(qi), d(ki), d(w), d(q_pos0), d(kv_len))
    idx = dsa.topk(S, d(q_pos0), d(kv_len), wl.N, wl.top_k)
    out = dsa.mla_sparse_attn_prefill(d(q[0]), d(kv[0]), idx[0], W.SCALE)
    torch.cuda.synchronize()
    parts = sorted(results["parts"], key=lambda t: t[0])
    np.testing.assert_array_equal(np.concatenate([t[2] for t in parts]), S[0, :, : wl.N].cpu().numpy())
    np.testing.assert_array_equal(np.concatenate([t[3] for t in parts]), idx[0].cpu().numpy())
    np.testing.assert_array_equal(np.concatenate([t[4] for t in parts]), out.cpu().numpy())
