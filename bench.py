#!/usr/bin/env python
"""Benchmark of the DSA sparse-attention hot path on GB300.

One step = one pass of the whole path over one 4096-query prefill chunk at
16k keys of context (4096 queries at positions 12288..16383, top_k 2048):
DSA indexer scores -> top-k selection -> sparse absorbed-MLA attention, the
three C-ABI calls of libdsa_gb300.so on inputs resident in HBM.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                    [--workload NAME] [--queries N] [--no-cpu-baseline]

--workload picks another of the seeded workloads (the 4k first chunk, the 64k
chunk, the 1k tiny chunk, or a decode batch: one new token for each of B
sequences, through the batched decode entry point, reported in us/step).

Prints one JSON line (rank 0).  Under torchrun each rank processes its own
chunk on its own GPU (independent problems, no data-path collective), so
`value` is the chunk queries of all ranks divided by the slowest rank's time
(weak scaling).  `--impl reference` times the float64 CPU oracle instead, on
the host cores, on a bounded sample of the same workload.
"""
import argparse
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from deepseek_sparse_attention_indexer_gb300 import workloads as W  # noqa: E402

METRIC = "prefill queries/s (indexer+top-k+sparse MLA) at 16k ctx; % of roofline"


def metric_name(wl):
    """The metric string of a workload's line: the headline string for the 16k chunk, the same
    wording with the workload's own context for the other prefill chunks, a time for decode."""
    if wl.L == 1:
        return f"decode us/step (indexer+top-k+sparse MLA, batch {wl.B}, {wl.N} keys)"
    if wl.name == DEFAULT_WORKLOAD:
        return METRIC
    ctx = f"{wl.N // 1024}k" if wl.N % 1024 == 0 else f"{wl.N} keys"
    return (f"prefill queries/s (indexer+top-k+sparse MLA) at {ctx} ctx "
            f"({wl.L} queries at positions {wl.p0}..{wl.p0 + wl.L - 1}); % of roofline")
UNIT = "queries/s"
DEFAULT_WORKLOAD = "prefill_16k"
PEAKS_PATH = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def algorithmic(wl):
    """Per-step algorithmic work of the path (causal pairs / selected slots only)."""
    pos = wl.p0 + np.arange(wl.L, dtype=np.int64)
    pairs = int(np.minimum(pos + 1, wl.N).sum()) * wl.B
    slots = int(np.minimum(pos + 1, wl.top_k).sum()) * wl.B
    return {
        "indexer_flop": pairs * 32 * 128 * 2,
        "topk_bytes": pairs * 4,
        "attn_flop": slots * 64 * (576 + 512) * 2,
        "gather_bytes": slots * 1152,
        "pairs": pairs,
        "slots": slots,
    }


def step_roofline(work, peak_tflops, hbm_gbs, step_ms):
    """The step's ideal time (indexer FLOP at the bf16 peak + causal score bytes at the HBM rate +
    attention FLOP at the bf16 peak) and the measured step's fraction of it."""
    ideal_ms = 1e3 * (work["indexer_flop"] / (peak_tflops * 1e12) + work["topk_bytes"] / (hbm_gbs * 1e9)
                      + work["attn_flop"] / (peak_tflops * 1e12))
    return {"ideal_ms": ideal_ms, "measured_ms": float(step_ms), "frac": ideal_ms / float(step_ms),
            "terms": "indexer FLOP / bf16 peak + causal score bytes / HBM + attention FLOP / bf16 peak"}


def max_over_ranks(x, world, device=None):
    """The slowest rank's value (the job ends when its last rank does).  One rank: x itself.  The
    collective runs on the process group's backend (NCCL on the GPU machine, gloo in the CPU tests)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    on = device if (device is not None and dist.get_backend() == "nccl") else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=on)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replicas_rate(units_per_rank, world, ms):
    """Whole-job throughput of `world` independent replicas that each process `units_per_rank`
    in at most `ms` milliseconds (weak scaling: per-rank work fixed as the job grows)."""
    return units_per_rank * world / (ms * 1e-3)


def attention_traffic(wl, decode):
    """DRAM bytes (read + write) of one attention launch at this workload, from the ncu record in
    profiles/, or None when there is none or the kernel source changed since it was taken."""
    import hashlib
    name = "mla_sparse_attn_decode" if decode else "mla_sparse_attn_prefill"
    src = os.path.join(ROOT, "deepseek_sparse_attention_indexer_gb300", "csrc", "mla_attn.cu")
    try:
        sha = hashlib.sha1(open(src, "rb").read()).hexdigest()
    except OSError:
        return None
    pdir = os.path.join(ROOT, "profiles")
    for fn in sorted(os.listdir(pdir)) if os.path.isdir(pdir) else []:
        if not (fn.startswith("attention_traffic_") and fn.endswith(".txt")):
            continue
        rec = {}
        for line in open(os.path.join(pdir, fn)):
            parts = line.split()
            if len(parts) == 2 and not line.startswith("#"):
                rec[parts[0]] = parts[1]
        if rec.get("workload") == wl.name and rec.get("kernel") == name and rec.get("source_sha1") == sha:
            return int(rec["bytes_per_launch"])
    return None


def value_proj_line(R, ms, peaks, peak_kind):
    """Roofline of one mla_value_up_proj launch over R rows (bound by HBM: o in, v out)."""
    nbytes = R * 64 * 512 * 2 + 64 * 256 * 512 * 2 + R * 64 * 256 * 2
    flop = R * 64 * 256 * 512 * 2
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    gbs = nbytes / (ms * 1e-3) / 1e9
    tf = flop / (ms * 1e-3) / 1e12
    return {"rows": R, "ms": ms, "bound": "hbm", "achieved_gbs": gbs, "frac": gbs / hbm,
            "peak_kind": f"{peak_kind} HBM copy", "bytes_per_launch": nbytes, "tflops": tf,
            "note": "wv_b up-projection of the step's attention output, timed after the step (not in the metric)"}


def load_peaks():
    try:
        with open(PEAKS_PATH) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# ----------------------------------------------------------------------------- clocks

def nvsmi_device_id(local_rank):
    """The identity nvidia-smi should sample for CUDA device `local_rank`: its UUID (or PCI bus
    id), which names the same physical GPU whatever CUDA_VISIBLE_DEVICES does to the ordinals.
    Falls back to the ordinal only when the device reports neither."""
    import torch
    props = torch.cuda.get_device_properties(local_rank)
    uuid = getattr(props, "uuid", None)
    if uuid:
        u = str(uuid)
        return u if u.startswith(("GPU-", "MIG-")) else "GPU-" + u
    bus = getattr(props, "pci_bus_id", None)
    if bus is not None:
        dom = getattr(props, "pci_domain_id", 0) or 0
        devn = getattr(props, "pci_device_id", 0) or 0
        return f"{dom:08X}:{bus:02X}:{devn:02X}.0"
    return str(local_rank)


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_id):
        self.device_id = device_id      # UUID or PCI bus id (nvsmi_device_id), not a CUDA ordinal
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.device_id), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                "device": str(self.device_id)}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) != 6:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[2:]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm), "device": str(self.device_id)}


# ----------------------------------------------------------------------------- oracle (CPU) timing

def is_decode(wl):
    """One query per sequence: the batched decode entry point serves it."""
    return wl.L == 1


def oracle_sample(wl, inputs, rows, threads):
    """Run the float64 oracle chain on the given query rows (flat b*L+i); return seconds."""
    import oracle
    qi, ki, w, q, kv, q_pos0, kv_len = inputs
    t0 = time.perf_counter()
    S = oracle.indexer(qi, ki, w, q_pos0, kv_len, rows=rows, threads=threads)
    idx = oracle.topk(S.astype(np.float32), q_pos0, kv_len, wl.B, wl.L, wl.top_k, rows=rows, threads=threads)
    qf = q.reshape(wl.B * wl.L, q.shape[2], q.shape[3])
    row_batch = (np.arange(wl.B * wl.L) // wl.L).astype(np.int32)
    oracle.attention(qf, kv, idx, row_batch, W.SCALE, rows=rows, threads=threads)
    return time.perf_counter() - t0


def sample_rows(wl, n, seed):
    rng = np.random.default_rng(seed)
    R = wl.B * wl.L
    return sorted(rng.choice(R, size=min(n, R), replace=False).tolist())


def run_reference(args, wl, rank, world):
    """--impl reference: the oracle as it stands, on this host's cores."""
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    inputs = make_inputs(wl)
    threads = oracle.default_threads()
    decode = is_decode(wl)
    rows_per_step = wl.B * wl.L if decode else threads   # decode: the whole batch's new tokens
    for s in range(args.warmup):
        oracle_sample(wl, inputs, sample_rows(wl, rows_per_step, 100 + s), threads)
    tot = 0.0
    for s in range(args.steps):
        tot += oracle_sample(wl, inputs, sample_rows(wl, rows_per_step, 1000 + s), threads)
    metric = metric_name(wl)
    if decode:
        value, unit, hib = 1e6 * tot / args.steps, "us/step", False
        what = f"all {rows_per_step} sequences of the batch per step, {args.steps} steps"
    else:
        value, unit, hib = rows_per_step * args.steps / tot, UNIT, True
        what = (f"{rows_per_step} query rows per step (indexer over all causal keys, top-k, attention over "
                f"{wl.top_k} keys), {args.steps} steps")
    line = {
        "impl": "reference", "metric": metric, "value": value, "unit": unit, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot / args.steps,
        "higher_is_better": hib, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_block(wl, world),
        "cpu_baseline": {"value": value, "unit": unit, "cores": threads, "kind": "oracle", "sample": what},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- GPU arm

def make_inputs(wl):
    qi, ki, w = W.make_indexer_inputs(wl)
    q, kv = W.make_attention_inputs(wl)
    q_pos0, kv_len = W.positions(wl)
    return qi, ki, w, q, kv, q_pos0, kv_len


def config_block(wl, world):
    return {"workload": wl.name, "desc": wl.desc, "batch": wl.B, "queries": wl.L, "kv_len": wl.N,
            "q_pos0": wl.p0, "top_k": wl.top_k, "heads": 64, "qk_dim": 576, "v_dim": 512,
            "indexer_heads": 32, "indexer_dim": 128, "global_batch": wl.B * wl.L * world,
            "parallelism": f"replicas{world}" if world > 1 else "single",
            "l2": "flushed between timed steps (write of a 512 MiB buffer); inputs larger than L2",
            **({"page_size": wl.page_size} if wl.page_size else {})}


def run_gpu(args, wl, rank, world, local_rank):
    import torch
    import torch.distributed as dist
    from deepseek_sparse_attention_indexer_gb300 import _lib as dsa

    torch.cuda.set_device(local_rank)
    dsa.load()
    inputs = make_inputs(wl)
    qi, ki, w, q, kv, q_pos0, kv_len = inputs
    dev = torch.device("cuda", local_rank)

    def d(a):
        a = np.ascontiguousarray(a)
        return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).to(dev)

    if wl.page_size:
        # paged caches: the same rows, scattered over a shuffled pool of pages
        ki, table = W.paginate(ki, kv_len, wl.page_size, extra_pages=8, seed=wl.seed + 7)
        kv, _ = W.paginate(kv, kv_len, wl.page_size, extra_pages=8, seed=wl.seed + 7)
        dtab = d(table)
    dqi, dki, dw, dpos, dlen, dq, dkv = map(d, (qi, ki, w, q_pos0, kv_len, q, kv))
    ld = (wl.N + 3) // 4 * 4
    S = torch.empty((wl.B, wl.L, ld), dtype=torch.float32, device=dev)
    idx = torch.empty((wl.B, wl.L, wl.top_k), dtype=torch.int32, device=dev)
    decode = is_decode(wl)
    # the attention output in float32 (DSA_OUT_F32): the configuration the parity tests check
    out = torch.empty((wl.B if decode else wl.L, 64, 512), dtype=torch.float32, device=dev)
    ws = torch.empty((dsa.attn_workspace_size(wl.B, wl.top_k),), dtype=torch.uint8, device=dev) if decode else None
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def indexer(a_qi, a_ki, a_w, a_pos, a_len):
        if wl.page_size:
            dsa.indexer_scores_paged(a_qi, a_ki, a_w, a_pos, a_len, dtab, wl.page_size, wl.N, scores=S)
        else:
            dsa.indexer_scores(a_qi, a_ki, a_w, a_pos, a_len, scores=S)

    def attention(a_q, a_kv, a_len):
        if wl.page_size:
            dsa.mla_sparse_attn_decode_paged(a_q[:, 0], a_kv, a_len, dtab, wl.page_size, idx[:, 0], W.SCALE,
                                             wl.N, out=out, workspace=ws)
        elif decode:   # one query per sequence: the batched decode entry point
            dsa.mla_sparse_attn_decode(a_q[:, 0], a_kv, a_len, idx[:, 0], W.SCALE, out=out, workspace=ws)
        else:
            dsa.mla_sparse_attn_prefill(a_q[0], a_kv[0], idx[0], W.SCALE, out=out)

    def step(ev=None):
        if ev:
            ev[0].record(stream)
        indexer(dqi, dki, dw, dpos, dlen)
        if ev:
            ev[1].record(stream)
        dsa.topk(S, dpos, dlen, wl.N, wl.top_k, idx=idx)
        if ev:
            ev[2].record(stream)
        attention(dq, dkv, dlen)
        if ev:
            ev[3].record(stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    if dsa.device_status() != 0:
        raise RuntimeError("device error word set during warm-up")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    sampler = ClockSampler(nvsmi_device_id(local_rank))
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    t_load = time.time() + 0.4       # untimed steps while the clock sampler starts (GPU under the same load)
    while time.time() < t_load:
        flush.zero_()
        step()
    torch.cuda.synchronize()
    for k in range(args.steps):
        flush.zero_()
        step(evs[k])
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    per = np.array([[evs[k][i].elapsed_time(evs[k][i + 1]) for i in range(3)] for k in range(args.steps)])
    step_ms = float(per.sum(axis=1).mean())
    step_stats = {"mean": step_ms, "median": float(np.median(per.sum(axis=1))), "min": float(per.sum(axis=1).min())}
    kern_ms = per.mean(axis=0)  # indexer, topk, attention
    step_ms_max = max_over_ranks(step_ms, world, dev)
    status = dsa.device_status()

    # ---- the same step replayed as one CUDA graph (launch gaps removed); for
    # decode, where the kernels are microseconds long, this is the step time a
    # serving loop that captures its decode step sees
    graph_ms = None
    try:
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            step()                          # warm the library's per-kernel setup on this stream
        stream.wait_stream(side)
        torch.cuda.synchronize()
        with torch.cuda.graph(g):
            step()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        reps = max(20, args.steps)
        g0 = torch.cuda.Event(enable_timing=True)
        g1 = torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        for _ in range(reps):
            g.replay()
        g1.record(stream)
        torch.cuda.synchronize()
        graph_ms = g0.elapsed_time(g1) / reps
        del g
    except RuntimeError as exc:            # capture unsupported here: report why, keep the line
        graph_ms = f"unavailable: {exc}"
    if dsa.device_status() != 0:
        raise RuntimeError("device error word set during the graph replays")

    # ---- end to end through the public API with host buffers (pinned), copies timed.  A decode
    # step's inputs are the new tokens (indexer query, head weights, absorbed query, positions):
    # the sequences' key caches (kI, kv) stay resident on the device between steps.
    host_in = [torch.from_numpy(np.ascontiguousarray(a.view(np.int16) if a.dtype == np.uint16 else a)).pin_memory()
               for a in (qi, ki, w, q_pos0, kv_len, q, kv)]
    host_out = torch.empty(tuple(out.shape), dtype=out.dtype).pin_memory()
    dev_in = [h.to(dev) for h in host_in]
    per_step = (0, 2, 3, 4, 5) if decode else range(7)
    h2d = sum(host_in[i].numel() * host_in[i].element_size() for i in per_step)
    d2h = host_out.numel() * host_out.element_size()

    e2e_pipelined = False
    e2e_rounds = None
    if not decode and wl.B == 1:
        # the package's host-buffer prefill: copies on side streams overlap the kernels
        from deepseek_sparse_attention_indexer_gb300.host_prefill import HostPrefill
        runner = HostPrefill(wl.L, wl.N, wl.top_k, device=dev, out_dtype=out.dtype, sets=2)
        e2e_api = (f"HostPrefill: H2D of the inputs, the three calls and D2H of the output overlapped "
                   f"({runner.slices} query slices); two chunks in flight (two device buffer sets), "
                   f"each chunk's inputs uploaded and its output downloaded, consecutive chunks timed "
                   f"back to back")
        host_out2 = torch.empty_like(host_out).pin_memory()
        e2e_pipelined = True

        def e2e_step(k=0):
            return runner(*host_in, host_out if k % 2 == 0 else host_out2, W.SCALE, stream=stream)
    elif decode and not wl.page_size:
        # the package's decode step: uploads of the new tokens' inputs, the calls and the download,
        # replayed as one CUDA graph over device-resident caches
        from deepseek_sparse_attention_indexer_gb300.host_decode import HostDecode
        runner = HostDecode(dev_in[1], dev_in[6], wl.top_k, W.SCALE, out_dtype=out.dtype)
        runner.h_qi.copy_(host_in[0].view(torch.int16))
        runner.h_w.copy_(host_in[2])
        runner.h_pos.copy_(host_in[3])
        runner.h_len.copy_(host_in[4])
        runner.h_q.copy_(host_in[5].view(torch.int16)[:, 0])
        e2e_api = ("HostDecode: H2D of the new tokens' inputs (caches resident), the calls and D2H of the "
                   "output, replayed as one CUDA graph")
        h2d, d2h = runner.h2d_bytes, runner.d2h_bytes

        def e2e_step():
            runner(stream=stream)
            return None
    else:
        e2e_api = ("H2D of the new tokens' inputs (caches resident), the calls, D2H of the output, in stream "
                   "order" if decode else "H2D of every input, the calls, D2H of the output, in stream order")

        def e2e_step():
            for i in per_step:
                dev_in[i].copy_(host_in[i], non_blocking=True)
            a_qi, a_ki, a_w, a_pos, a_len, a_q, a_kv = dev_in
            indexer(a_qi, a_ki, a_w, a_pos, a_len)
            dsa.topk(S, a_pos, a_len, wl.N, wl.top_k, idx=idx)
            attention(a_q, a_kv, a_len)
            host_out.copy_(out, non_blocking=True)
            return None

    e2e_step()
    torch.cuda.synchronize()
    e2e_ms = []
    for _ in range(max(3, min(args.steps, 10))):
        flush.zero_()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        done = e2e_step()
        if done is not None:
            stream.wait_event(done)
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms.append(e0.elapsed_time(e1))
    e2e_single = float(np.mean(e2e_ms))      # one chunk alone: its latency from host to host
    if e2e_pipelined:
        # consecutive chunks, each from its host inputs to its host output, with the next chunk's
        # uploads and kernels under the previous chunk's download; every chunk's inputs (302 MB of q
        # alone) are larger than L2 and re-uploaded, so no flush between chunks
        n_chunks = max(4, min(args.steps, 12))
        for k in range(2):
            e2e_step(k)
        torch.cuda.synchronize()
        rounds = []
        for _ in range(3):        # median of three rounds: host copies share the box's memory system
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for k in range(n_chunks):
                done = e2e_step(k)
            stream.wait_event(done)
            e1.record(stream)
            torch.cuda.synchronize()
            rounds.append(e0.elapsed_time(e1) / n_chunks)
        e2e_rounds = [round(r, 4) for r in rounds]
        e2e_mean = max_over_ranks(float(np.median(rounds)), world, dev)
    else:
        e2e_mean = max_over_ranks(e2e_single, world, dev)

    # ---- the value up-projection (wv_b) of this step's attention output: the layer's next
    # call after the path, timed on its own (not part of the metric); L2 flushed before each call.
    # It reads bf16 rows: the step's attention output rounded (the library's bf16 output option).
    out16 = torch.empty(tuple(out.shape), dtype=torch.bfloat16, device=dev)
    if wl.page_size:
        dsa.mla_sparse_attn_decode_paged(dq[:, 0], dkv, dlen, dtab, wl.page_size, idx[:, 0], W.SCALE, wl.N,
                                         out=out16, workspace=ws)
    elif decode:
        dsa.mla_sparse_attn_decode(dq[:, 0], dkv, dlen, idx[:, 0], W.SCALE, out=out16, workspace=ws)
    else:
        dsa.mla_sparse_attn_prefill(dq[0], dkv[0], idx[0], W.SCALE, out=out16)
    R_v = out.shape[0]
    _, wv_host = W.make_value_proj_inputs(1, seed=wl.seed + 31)
    dwv = d(wv_host)
    vout = torch.empty((R_v, 64, 256), dtype=torch.bfloat16, device=dev)
    for _ in range(3):
        dsa.mla_value_up_proj(out16, dwv, v=vout)
    vp_ms = []
    for _ in range(max(3, min(args.steps, 20))):
        flush.zero_()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        dsa.mla_value_up_proj(out16, dwv, v=vout)
        e1.record(stream)
        torch.cuda.synchronize()
        vp_ms.append(e0.elapsed_time(e1))
    vp_ms = float(np.mean(vp_ms))

    if rank != 0:
        return 0

    work = algorithmic(wl)
    peaks, peak_kind = load_peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    attn_tf = work["attn_flop"] / (kern_ms[2] * 1e-3) / 1e12
    idx_tf = work["indexer_flop"] / (kern_ms[0] * 1e-3) / 1e12
    topk_gbs = work["topk_bytes"] / (kern_ms[1] * 1e-3) / 1e9
    traffic = attention_traffic(wl, decode)
    attn_name = "mla_sparse_attn_decode" if decode else "mla_sparse_attn_prefill"
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    gather_gbs = work["gather_bytes"] / (kern_ms[2] * 1e-3) / 1e9
    metric = metric_name(wl)
    if decode:
        # decode: a step is one new token for each of the B sequences; time-like metric
        value, unit, hib = step_ms_max * 1e3, "us/step", False
        e2e_value = e2e_mean * 1e3
        roof = {"bound": "hbm", "kernel": attn_name, "achieved": gather_gbs, "peak": hbm, "unit": "GB/s",
                "frac": gather_gbs / hbm, "traffic": traffic, "peak_kind": f"{peak_kind} HBM copy",
                "bytes_per_launch": work["gather_bytes"]}
    else:
        value, unit, hib = replicas_rate(wl.L * wl.B, world, step_ms_max), UNIT, True
        e2e_value = replicas_rate(wl.L * wl.B, world, e2e_mean)
        roof = {"bound": "tensor", "kernel": attn_name, "achieved": attn_tf, "peak": peak, "unit": "TFLOP/s",
                "frac": attn_tf / peak, "traffic": traffic, "peak_kind": f"{peak_kind} bf16 dense burst",
                "flop_per_launch": work["attn_flop"]}
    line = {
        "metric": metric,
        "value": value,
        "unit": unit,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": max(3, args.warmup),
        "ms_per_step": step_ms_max,
        "ms_per_step_stats": step_stats,   # this rank's timed steps: mean (used for value), median, min
        "higher_is_better": hib,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "attention_output": "float32 (DSA_OUT_F32)",
        "data": "synthetic",
        "config": config_block(wl, world),
        "roofline": roof,
        # indexer + top-k per chunk (the selection stage on its own)
        "indexer_topk_ms": float(kern_ms[0] + kern_ms[1]),
        # the step against its ideal: every kernel at its own roofline, back to back
        "step_roofline": step_roofline(work, peak, hbm, step_ms_max),
        "kernels_ms": {"dsa_indexer_scores": float(kern_ms[0]), "dsa_topk": float(kern_ms[1]),
                       attn_name: float(kern_ms[2])},
        "kernel_rooflines": {
            "dsa_indexer_scores": {"bound": "tensor", "achieved_tflops": idx_tf, "frac": idx_tf / peak},
            "dsa_topk": {"bound": "hbm", "achieved_gbs": topk_gbs, "frac": topk_gbs / hbm},
            attn_name: {"bound": "tensor", "achieved_tflops": attn_tf, "frac": attn_tf / peak,
                        "gather_gbs": gather_gbs, "gather_frac_of_hbm": gather_gbs / hbm},
        },
        "e2e": {"value": e2e_value, "unit": unit,
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "api": e2e_api,
                "ms_per_step": round(e2e_mean, 4), "single_step_latency_ms": round(e2e_single, 4),
                **({"rounds_ms_per_step": e2e_rounds} if e2e_rounds else {})},
        "graph": ({"ms_per_step": graph_ms, "note": "the step replayed as one CUDA graph, inputs resident, "
                   "no L2 flush between replays"} if isinstance(graph_ms, float) else {"ms_per_step": None,
                                                                                     "note": graph_ms}),
        "value_up_proj": value_proj_line(R_v, vp_ms, peaks, peak_kind),
        "gpu_launches": (4 if decode else 3) * args.steps,
        "clocks": clocks,
        "device_status": status,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, inputs, decode)
    print(json.dumps(line), flush=True)
    return 0


CPU_BASELINE_SECONDS = 10.0   # oracle work the CPU baseline times (bounded sample of the workload)


def cpu_baseline(wl, inputs, decode, target_s=CPU_BASELINE_SECONDS):
    """The oracle as it stands on this host's cores, timed on a seeded sample of the workload sized
    from a short probe to about target_s seconds of work (prefill: query rows; decode: whole steps)."""
    import oracle
    oracle.build()
    threads = oracle.default_threads()
    if decode:
        rows = list(range(wl.B * wl.L))
        secs = oracle_sample(wl, inputs, rows, threads)
        reps = max(1, min(1000, int(target_s / max(secs, 1e-6))))
        tot = secs + sum(oracle_sample(wl, inputs, rows, threads) for _ in range(reps - 1))
        return {"value": 1e6 * tot / reps, "unit": "us/step", "cores": threads, "kind": "oracle",
                "sample": f"{reps} decode steps (all {len(rows)} sequences of the batch: indexer, top-k and "
                          f"attention for each new token), {tot:.1f} s"}
    probe = sample_rows(wl, threads, 7)
    per_row = oracle_sample(wl, inputs, probe, threads) / len(probe)
    n = max(len(probe), min(wl.B * wl.L, int(target_s / max(per_row, 1e-9))))
    rows = sample_rows(wl, n, 8)
    secs = oracle_sample(wl, inputs, rows, threads)
    return {"value": len(rows) / secs, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": (f"{len(rows)} seeded query rows of the same chunk (indexer over all their causal keys, "
                       f"top-k, attention over their {wl.top_k} keys), {secs:.1f} s")}


def resolve_workload(name, queries=0, batch=0):
    """The named workload, narrowed to its last `queries` queries (prefill) or widened to `batch`
    sequences (decode)."""
    wl = W.WORKLOADS[name]
    if queries and queries < wl.L:
        wl = W.custom(f"{wl.name}_last{queries}", B=wl.B, L=queries, p0=wl.N - queries, N=wl.N,
                      top_k=wl.top_k, seed=wl.seed, rope_std=wl.rope_std, dup_frac=wl.dup_frac)
    if batch:
        if wl.L != 1:
            raise ValueError("--batch applies to decode workloads")
        if batch < 1:
            raise ValueError("--batch must be positive")
        wl = dataclasses.replace(wl, name=f"{wl.name}_batch{batch}", B=batch,
                                 desc=f"{batch} sequences, one new query each at position {wl.p0} "
                                      f"over its own {wl.N}-key cache, top_k {wl.top_k}")
    return wl


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(W.WORKLOADS))
    ap.add_argument("--queries", type=int, default=0,
                    help="profiling aid: keep the context, time only the last N queries of the chunk")
    ap.add_argument("--batch", type=int, default=0,
                    help="decode workloads: the same step for this many sequences (batch scaling)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    try:
        wl = resolve_workload(args.workload, args.queries, args.batch)
    except ValueError as exc:
        ap.error(str(exc))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, wl, rank, world)
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        return run_gpu(args, wl, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
