"""float64 CPU oracle for the DSA indexer -> top-k -> sparse absorbed-MLA path.

TEST INFRASTRUCTURE.  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's ``cpu_baseline`` / ``--impl reference`` legs may import this
package.  The product library never calls it and shares no code with it.

The arithmetic lives in ``dsa_oracle.c`` (plain C, double precision, one row at
a time).  This module compiles it with gcc, loads it with ctypes and offers
numpy wrappers that spread rows over host threads (ctypes drops the GIL during
the call, and each row's code stays single-threaded).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dsa_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libdsa_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle (gcc -O2, IEEE semantics: no fast-math)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or \
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-fno-fast-math", "-ffp-contract=off",
                               "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I = ctypes.c_int
            lib.oracle_indexer.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, P]
            lib.oracle_topk.argtypes = [P, ctypes.c_int64, P, P, I, I, I, I, I, P]
            lib.oracle_attn.argtypes = [P, P, P, P, I, I, I, I, I, ctypes.c_double,
                                        I, I, P, P]
            lib.oracle_value_up_proj.argtypes = [P, P, I, I, I, I, I, P]
            for f in (lib.oracle_indexer, lib.oracle_topk, lib.oracle_attn, lib.oracle_value_up_proj):
                f.restype = None
            _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def _split(rows: Sequence[int], threads: int):
    """Cut the sorted row list into (begin, end, position) runs of consecutive
    rows; `position` is where row `begin` sits in the compact output."""
    runs = []
    for k, r in enumerate(rows):
        if runs and runs[-1][1] == r:
            runs[-1][1] = r + 1
        else:
            runs.append([r, r + 1, k])
    chunk = max(1, (len(rows) + 4 * threads - 1) // (4 * threads))
    out = []
    for b, e, k in runs:
        while b < e:
            n = min(chunk, e - b)
            out.append((b, b + n, k))
            b += n
            k += n
    return out


def _run(fn, ranges, threads: int):
    if threads <= 1 or len(ranges) <= 1:
        for be in ranges:
            fn(*be)
        return
    with ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(lambda be: fn(*be), ranges))


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def indexer(qI: np.ndarray, kI: np.ndarray, w: np.ndarray, q_pos0: np.ndarray,
            kv_len: np.ndarray, rows: Optional[Sequence[int]] = None,
            threads: int = 1) -> np.ndarray:
    """Scores float64: [B*L, Nmax], or [len(rows), Nmax] for the sorted `rows`."""
    lib = _load()
    B, L, Hi, Di = qI.shape
    Nmax = kI.shape[1]
    qI = np.ascontiguousarray(qI, np.uint16)
    kI = np.ascontiguousarray(kI, np.uint16)
    w = np.ascontiguousarray(w, np.float32)
    q_pos0 = np.ascontiguousarray(q_pos0, np.int32)
    kv_len = np.ascontiguousarray(kv_len, np.int32)
    rows = list(range(B * L)) if rows is None else sorted(rows)
    S = np.full((len(rows), Nmax), np.nan, dtype=np.float64)

    def fn(b, e, k):
        lib.oracle_indexer(_ptr(qI), _ptr(kI), _ptr(w), _ptr(q_pos0), _ptr(kv_len),
                           B, L, Nmax, Hi, Di, b, e, _ptr(S) + k * Nmax * 8)
    _run(fn, _split(rows, threads), threads)
    return S


def topk(S: np.ndarray, q_pos0: np.ndarray, kv_len: np.ndarray, B: int, L: int,
         K: int, rows: Optional[Sequence[int]] = None, threads: int = 1) -> np.ndarray:
    """Top-k indices int32 [B*L, K] from float32 scores [B*L, ld]; with `rows`,
    the scores and the result hold only those (sorted) rows."""
    lib = _load()
    S = np.ascontiguousarray(S, np.float32)
    q_pos0 = np.ascontiguousarray(q_pos0, np.int32)
    kv_len = np.ascontiguousarray(kv_len, np.int32)
    rows = list(range(B * L)) if rows is None else sorted(rows)
    assert S.shape[0] == len(rows)
    idx = np.full((len(rows), K), -2, dtype=np.int32)
    ld = S.shape[1]

    def fn(b, e, k):
        lib.oracle_topk(_ptr(S) + k * ld * 4, ld, _ptr(q_pos0), _ptr(kv_len), B, L, K,
                        b, e, _ptr(idx) + k * K * 4)
    _run(fn, _split(rows, threads), threads)
    return idx


def attention(q: np.ndarray, kv: np.ndarray, idx: np.ndarray, row_batch: np.ndarray,
              scale: float, rows: Optional[Sequence[int]] = None, threads: int = 1):
    """out [R, H, Dv] float64 and lse [R, H] float64 (Dv = D - 64).

    q [R, H, D] bf16 bits, kv [B, Nmax, D] bf16 bits, idx [R, K] int32.  With
    `rows`, idx, out and lse hold only those (sorted) rows.
    """
    lib = _load()
    R, H, D = q.shape
    B, Nmax, D2 = kv.shape
    assert D2 == D
    Dv = D - 64
    K = idx.shape[1]
    q = np.ascontiguousarray(q, np.uint16)
    kv = np.ascontiguousarray(kv, np.uint16)
    idx = np.ascontiguousarray(idx, np.int32)
    row_batch = np.ascontiguousarray(row_batch, np.int32)
    rows = list(range(R)) if rows is None else sorted(rows)
    assert idx.shape[0] == len(rows)
    out = np.full((len(rows), H, Dv), np.nan, dtype=np.float64)
    lse = np.full((len(rows), H), np.nan, dtype=np.float64)

    def fn(b, e, k):
        lib.oracle_attn(_ptr(q), _ptr(kv), _ptr(idx) + k * K * 4, _ptr(row_batch), Nmax, K, H, D,
                        Dv, float(scale), b, e, _ptr(out) + k * H * Dv * 8, _ptr(lse) + k * H * 8)
    _run(fn, _split(rows, threads), threads)
    return out, lse


def value_up_proj(o: np.ndarray, wv: np.ndarray, rows: Optional[Sequence[int]] = None,
                  threads: int = 1) -> np.ndarray:
    """v [R, H, E] float64 = per head o[r, h, :] . wv[h, e, :] (the wv_b up-projection).

    o [R, H, Dv] bf16 bits, wv [H, E, Dv] bf16 bits.  With `rows`, v holds only
    those (sorted) rows.
    """
    lib = _load()
    R, H, Dv = o.shape
    H2, E, Dv2 = wv.shape
    assert H2 == H and Dv2 == Dv
    o = np.ascontiguousarray(o, np.uint16)
    wv = np.ascontiguousarray(wv, np.uint16)
    rows = list(range(R)) if rows is None else sorted(rows)
    v = np.full((len(rows), H, E), np.nan, dtype=np.float64)

    def fn(b, e, k):
        lib.oracle_value_up_proj(_ptr(o), _ptr(wv), H, Dv, E, b, e, _ptr(v) + k * H * E * 8)
    _run(fn, _split(rows, threads), threads)
    return v


def unpage(pool: np.ndarray, block_table: np.ndarray, page_size: int, kv_len,
           Nmax: int) -> np.ndarray:
    """Dense [B, Nmax, D] cache of a paged one, by the page-table definition.

    Row j < kv_len[b] of sequence b is pool row
    block_table[b, j // page_size] * page_size + j % page_size.  A table entry
    outside [0, num_pages) reads as a zero row (the library's stated reading of
    a bad entry), and rows j >= kv_len[b] are zero: nothing downstream reads
    them.  Paging only moves rows; no arithmetic happens here.  The pages
    describe exo's per-sequence decode "batch caches" (exo PR #2539, section
    "Decode") without fixing a memory layout; the page table is the library's.
    """
    B = block_table.shape[0]
    D = pool.shape[1]
    num_pages = pool.shape[0] // page_size
    out = np.zeros((B, Nmax, D), dtype=pool.dtype)
    for b in range(B):
        for j in range(int(kv_len[b])):
            page = int(block_table[b, j // page_size])
            if 0 <= page < num_pages:
                out[b, j] = pool[page * page_size + j % page_size]
    return out
