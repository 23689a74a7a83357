"""Benchmark: paged GQA decode on the Llama-3-8B-shaped f16 workload.

One step = for each of the 32 layers: the KV store of the decode token's new
K/V rows into their resolved cells, then paged decode attention (split-K
decode + combine) over that layer's paged f16 K/V pools. 64 sequences,
context lengths log-uniform in [512, 16384], 32 query / 8 KV heads,
head_dim 128, block_size 16, block tables drawn from a pool of 1.1x the
blocks needed (seeded synthetic data; ~42 GB of K/V resident in HBM).

Prints one JSON line. `value` is algorithmic KV bytes per second (K and V
rows attended, block-table entries read, Q read, output written, rows
stored), device-timed with CUDA events with inputs already in HBM; `e2e` is
the same metric through the same C-ABI calls with each step's inputs copied
from pinned host memory and the outputs copied back inside the timed region.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl mtkv|reference]

`--impl reference` times the CPU oracle (the only reference this method has)
on a bounded sample of the same workload, on the host's cores.
Under torchrun with N > 1 every rank runs an independent replica (the path
has no exchange step); rank 0 prints the line with the max time over ranks.
"""
from __future__ import annotations

import os

# each CPU oracle worker runs single-threaded (the workers spread over the
# host's cores); fix the BLAS pools before numpy loads
for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse
import hashlib
import json
import math
import multiprocessing as mp
import statistics
import subprocess
import sys
import time

import numpy as np

if __name__ != "__mp_main__":
    # the oracle workers (spawned children that import this file) need numpy only
    import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_kv_cache_gqa_gb300 import workloads  # noqa: E402

METRIC = "paged GQA decode: KV HBM GB/s (fraction of GB300 peak) and attended tokens/s"
WORKLOAD = ("llama3-8b-shaped paged GQA decode, f16 KV: 32 layers, 64 seqs, ctx log-uniform "
            "[512,16384], 32/8 heads, head_dim 128, block_size 16, pool 1.1x, store+attention "
            "per layer")
SEED = 1003
N_LAYERS = 32
FALLBACK_HBM_GBS = 6800.0


def _peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def _tensor_peak():
    """Dense f16/bf16 tensor peak (same rate on this part): the measured
    burst figure for kernels timed alone."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured (bf16 burst; f16 same rate)"
    except Exception:
        return 1900.0, "fallback"


def max_over_ranks(x: float, world: int, device=None) -> float:
    """The largest value of x over all ranks (x itself when running alone)."""
    if world <= 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int) -> None:
    if world > 1:
        torch.distributed.barrier()


def whole_job_rate(bytes_per_rank: float, seconds: float, world: int) -> float:
    """Aggregate GB/s of `world` independent replicas that each moved
    bytes_per_rank in (at most) `seconds`."""
    return world * bytes_per_rank / seconds / 1e9


def _structure():
    return workloads.llama3_f16(seed=SEED, hist=False)


def decode_bytes(w, seqs=None):
    """Algorithmic bytes of one decode call (one layer): K and V rows of the
    attended positions for every KV head, the block-table entries those
    positions use, the context lengths, Q read and the output written."""
    seqs = range(w.n_seqs) if seqs is None else seqs
    hkv, d, bs = w.n_kv_heads, w.head_dim, w.block_size
    seg = d * 2  # f16 head segment
    toks = sum(int(w.context_lens[s]) for s in seqs)
    blocks = sum(-(-int(w.context_lens[s]) // bs) for s in seqs)
    n = len(list(seqs))
    return (toks * hkv * seg * 2 + blocks * 4 + n * 4 + 2 * n * w.n_heads * d * 4), toks


def store_bytes(w):
    row = w.n_kv_heads * w.head_dim
    return w.n_seqs * (2 * row * 4 + 2 * row * 2 + 8)


class Clocks:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.proc = None
        self.sel = None
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            self.sel = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
            self.sel = vis.split(",")[device_index] if vis else str(device_index)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.sel, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=10)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons, power = [], [], set(), []
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in out.strip().splitlines():
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(power) if power else None,
                "samples": len(sm), "reasons": sorted(reasons)}


def _traffic_from_profile():
    """DRAM bytes (read + write) per decode launch from the committed ncu
    counters in profiles/decode_traffic.json, if they were taken on the
    current decode kernel source (else None)."""
    data = os.path.join(ROOT, "profiles", "decode_traffic.json")
    src = os.path.join(ROOT, "paged_kv_cache_gqa_gb300", "csrc", "decode.cu")
    try:
        with open(data) as f:
            rec = json.load(f)
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        if rec.get("source_sha256_16") == sha:
            return float(rec["traffic_bytes_per_launch"])
    except (OSError, ValueError, KeyError):
        pass
    return None


class OracleSample:
    """The CPU oracle (store + decode of one layer) on the sequences `seqs`
    of the workload, on pool rows generated for those sequences (each
    sequence's rows from its own seeded generator, so a sequence's data do
    not depend on how the batch is split over workers). The sample's blocks
    are renumbered into a compact pool (same shapes and lengths; only the
    physical ids differ), so a worker holds only its own rows."""

    def __init__(self, w, seqs):
        from oracle import formats as ofmt
        self.w, self.seqs = w, list(seqs)
        hkv, d, bs = w.n_kv_heads, w.head_dim, w.block_size
        rb = ofmt.row_bytes("f16", hkv, d)
        nbs = [-(-int(w.context_lens[s]) // bs) for s in self.seqs]
        self.table = np.full_like(w.block_table, -1)
        self.cells = np.full(w.n_seqs, -1, dtype=np.int64)
        self.kp = np.empty((sum(nbs) * bs, rb), np.uint8)
        self.vp = np.empty_like(self.kp)
        nxt = 0
        for s, nb in zip(self.seqs, nbs):
            self.table[s, :nb] = np.arange(nxt, nxt + nb, dtype=self.table.dtype)
            c = int(w.context_lens[s]) - 1
            self.cells[s] = (nxt + c // bs) * bs + c % bs
            rng = np.random.default_rng((SEED + 7, s))
            rows = rng.standard_normal((2, nb * bs, hkv * d), dtype=np.float32)
            self.kp[nxt * bs:(nxt + nb) * bs] = ofmt.encode_rows("f16", rows[0], hkv, d)
            self.vp[nxt * bs:(nxt + nb) * bs] = ofmt.encode_rows("f16", rows[1], hkv, d)
            nxt += nb
        db, self.toks = decode_bytes(w, self.seqs)
        self.bytes = db + store_bytes(w) * len(self.seqs) // w.n_seqs

    def run(self) -> float:
        from oracle import attention as oatt
        w, sq = self.w, self.seqs
        t0 = time.perf_counter()
        oatt.kv_store("f16", self.kp, self.vp, w.k_new[sq], w.v_new[sq], self.cells[sq],
                      w.n_kv_heads, w.head_dim)
        oatt.paged_attn_decode("f16", w.q, self.kp, self.vp, self.table, w.context_lens, None,
                               w.n_heads, w.n_kv_heads, w.head_dim, w.block_size, w.scale,
                               seqs=sq)
        return time.perf_counter() - t0


def _oracle_worker(seqs, reps, bar):
    """One CPU core's share of the oracle layer: build its sequences' pools,
    then run store + decode once per repetition between two barriers."""
    smp = OracleSample(_structure(), seqs)
    bar.wait()                      # data ready
    for _ in range(reps):
        bar.wait()                  # start together
        smp.run()
        bar.wait()                  # all done


def _balanced_split(lengths, n):
    """Sequences dealt to n workers, longest first to the least loaded."""
    load = [0] * n
    parts = [[] for _ in range(n)]
    for s in sorted(range(len(lengths)), key=lambda i: -int(lengths[i])):
        j = min(range(n), key=lambda k: load[k])
        parts[j].append(s)
        load[j] += int(lengths[s])
    return [sorted(p) for p in parts if p]


def oracle_layer_times(reps: int, max_workers: int | None = None):
    """Wall-clock seconds of the CPU oracle's store + decode of one whole
    layer (all sequences), spread over the host's cores by sequence: one
    spawned single-threaded worker per core (each runs the oracle as it
    stands on its share). Returns (times, cores, sample)."""
    w = _structure()
    cores = len(os.sched_getaffinity(0))
    n = max(1, min(cores, w.n_seqs, max_workers or cores))
    parts = _balanced_split(w.context_lens, n)
    ctx = mp.get_context("spawn")
    bar = ctx.Barrier(len(parts) + 1)
    procs = [ctx.Process(target=_oracle_worker, args=(p, reps, bar), daemon=True) for p in parts]
    for pr in procs:
        pr.start()
    times = []
    try:
        bar.wait(timeout=600)
        for _ in range(reps):
            bar.wait(timeout=600)
            t0 = time.perf_counter()
            bar.wait(timeout=600)
            times.append(time.perf_counter() - t0)
    finally:
        for pr in procs:
            pr.join(timeout=60)
            if pr.is_alive():
                pr.terminate()
    db, toks = decode_bytes(w)
    layer_bytes = db + store_bytes(w)
    sample = (f"store+decode of all {w.n_seqs} sequences of one layer ({toks} attended "
              f"positions), float64 numpy oracle, sequences split over {len(parts)} "
              f"single-threaded worker processes")
    return times, len(parts), sample, layer_bytes, toks


def run_reference(args, rank):
    """The reference arm: the CPU oracle, as it stands, on the host cores
    (one step = store + decode of one whole layer)."""
    if rank != 0:
        return None
    times, cores, sample, layer_bytes, toks = oracle_layer_times(args.warmup + args.steps)
    times = times[args.warmup:]
    sec = statistics.median(times)
    val = layer_bytes / sec / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(val, 5), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(sec * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "kv_format": "f16",
                   "sample": "all 64 sequences of one layer per step"},
        "step_ms": {"median": round(sec * 1e3, 3), "min": round(min(times) * 1e3, 3),
                    "max": round(max(times) * 1e3, 3), "n": len(times)},
        "attended_tokens_per_s": round(toks / sec, 1),
        "cpu_baseline": {"value": round(val, 5), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(val, 5), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    return line


def run_gpu(args, rank, world, local_rank):
    n_layers = args.layers
    from paged_kv_cache_gqa_gb300 import mtkv
    import __graft_entry__
    __graft_entry__.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    w = _structure()
    hkv, d, bs, hq, B = w.n_kv_heads, w.head_dim, w.block_size, w.n_heads, w.n_seqs
    n_cells = w.n_cells
    g = torch.Generator(device=dev)
    g.manual_seed(SEED + 100 * rank)
    k_pools, v_pools, qs, k_news, v_news, outs = [], [], [], [], [], []
    for _ in range(n_layers):
        k_pools.append(torch.randn(n_cells, hkv * d, generator=g, device=dev, dtype=torch.float16))
        v_pools.append(torch.randn(n_cells, hkv * d, generator=g, device=dev, dtype=torch.float16))
        qs.append(torch.randn(B, hq, d, generator=g, device=dev, dtype=torch.float32))
        k_news.append(torch.randn(B, hkv * d, generator=g, device=dev, dtype=torch.float32))
        v_news.append(torch.randn(B, hkv * d, generator=g, device=dev, dtype=torch.float32))
        outs.append(torch.empty(B, hq, d, device=dev, dtype=torch.float32))
    table = torch.from_numpy(w.block_table).to(dev)
    ctx = torch.from_numpy(w.context_lens).to(dev)
    cells = torch.from_numpy(w.new_cells).to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    args_l = [mtkv.paged_attn_args("f16", qs[l], k_pools[l], v_pools[l], table, ctx, outs[l],
                                   n_kv_heads=hkv, block_size=bs, n_phys_blocks=w.n_phys_blocks,
                                   scale=w.scale) for l in range(n_layers)]
    ws = torch.zeros(mtkv.mt_paged_attn_workspace_bytes(args_l[0]), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(n_layers)]

    fused = args.store == "fused"

    def layer(l):
        if fused:
            mtkv.mt_paged_attn_decode_append(args_l[l], k_news[l], v_news[l], ws)
        else:
            mtkv.mt_kv_store("f16", k_pools[l], v_pools[l], hkv, d, k_news[l], v_news[l], cells,
                             status=status)
            mtkv.mt_paged_attn_decode(args_l[l], ws)

    def step(record=False):
        for l in range(n_layers):
            if fused:
                if record:
                    ev[l][0].record(stream)
                mtkv.mt_paged_attn_decode_append(args_l[l], k_news[l], v_news[l], ws)
                if record:
                    ev[l][1].record(stream)
            else:
                mtkv.mt_kv_store("f16", k_pools[l], v_pools[l], hkv, d, k_news[l], v_news[l],
                                 cells, status=status)
                if record:
                    ev[l][0].record(stream)
                mtkv.mt_paged_attn_decode(args_l[l], ws)
                if record:
                    ev[l][1].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert mtkv.mt_check_device_status(status) == 0, mtkv.mt_last_error()
    assert mtkv.mt_check_device_status(ws) == 0, mtkv.mt_last_error()

    graph = None
    if args.graph:
        # the whole L-layer step as one CUDA graph (every kernel was
        # configured by the warm-up steps; the calls neither allocate nor
        # synchronise)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        graph.replay()
        torch.cuda.synchronize()
        assert mtkv.mt_check_device_status(ws) == 0, mtkv.mt_last_error()

    clocks = Clocks(local_rank)
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    # one event between consecutive steps: the total and each step's time
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    dec_ms = []
    marks[0].record(stream)
    for i in range(args.steps):
        if graph is not None:
            graph.replay()
        else:
            step(record=True)
            # per-call decode durations of this step (read back after the run)
            dec_ms.append([e for e in ev])
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(n_layers)]
        marks[i + 1].record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    barrier(world)
    total_ms = max_over_ranks(marks[0].elapsed_time(marks[-1]), world, dev)
    per_step = [marks[i].elapsed_time(marks[i + 1]) for i in range(args.steps)]
    if graph is not None:
        # per-call durations for the roofline from a few eager steps
        for _ in range(3):
            step(record=True)
            dec_ms.append([e for e in ev])
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(n_layers)]
        torch.cuda.synchronize()
    dec_times = [a.elapsed_time(b) for st in dec_ms for (a, b) in st]

    dbytes, toks = decode_bytes(w)
    step_bytes = n_layers * (dbytes + store_bytes(w))
    ms_per_step = total_ms / args.steps
    value = whole_job_rate(step_bytes, ms_per_step * 1e-3, world)
    peak, peak_kind = _peak()
    dec_avg_ms = statistics.mean(dec_times)
    # the timed call: decode + combine, with the row store when it is fused
    call_bytes = dbytes + (store_bytes(w) if fused else 0)
    achieved = call_bytes / (dec_avg_ms * 1e-3) / 1e9

    # ---- end to end: inputs from pinned host memory, outputs back to host
    h_q = [q.cpu().pin_memory() for q in qs]
    h_k = [k.cpu().pin_memory() for k in k_news]
    h_v = [v.cpu().pin_memory() for v in v_news]
    h_table = torch.from_numpy(w.block_table).pin_memory()
    h_ctx = torch.from_numpy(w.context_lens).pin_memory()
    h_cells = torch.from_numpy(w.new_cells).pin_memory()
    h_out = [torch.empty(B, hq, d, dtype=torch.float32).pin_memory() for _ in range(n_layers)]
    h_meta = [h_table, h_ctx] + ([] if fused else [h_cells])
    h2d = sum(t.numel() * t.element_size() for t in h_q + h_k + h_v + h_meta)
    d2h = sum(t.numel() * t.element_size() for t in h_out)

    # Copies run on two copy streams next to the compute stream: every input
    # of the step is sent host -> device up front (layer l waits only for its
    # own inputs), and each layer's output goes back device -> host as soon
    # as that layer is done, overlapping the later layers. Every byte still
    # crosses the host link inside the timed region of every step.
    s_h2d, s_d2h = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(n_layers)]
    ev_done = [torch.cuda.Event() for _ in range(n_layers)]

    def e2e_step():
        main = torch.cuda.current_stream()
        s_h2d.wait_stream(main)  # the previous step is done with the buffers
        s_d2h.wait_stream(main)
        with torch.cuda.stream(s_h2d):
            table.copy_(h_table, non_blocking=True)
            ctx.copy_(h_ctx, non_blocking=True)
            if not fused:
                cells.copy_(h_cells, non_blocking=True)
            for l in range(n_layers):
                qs[l].copy_(h_q[l], non_blocking=True)
                k_news[l].copy_(h_k[l], non_blocking=True)
                v_news[l].copy_(h_v[l], non_blocking=True)
                ev_in[l].record(s_h2d)
        for l in range(n_layers):
            main.wait_event(ev_in[l])
            layer(l)
            ev_done[l].record(main)
            with torch.cuda.stream(s_d2h):
                s_d2h.wait_event(ev_done[l])
                h_out[l].copy_(outs[l], non_blocking=True)
        main.wait_stream(s_h2d)
        main.wait_stream(s_d2h)

    e2e_steps = max(3, args.steps // 4)
    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    run_e2e = e2e_step
    if args.graph:
        # the copies from and to pinned host memory are captured with the step
        g_e2e = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_e2e):
            e2e_step()
        run_e2e = g_e2e.replay
        run_e2e()
        torch.cuda.synchronize()
    barrier(world)
    e0 = time.perf_counter()
    for _ in range(e2e_steps):
        run_e2e()
    torch.cuda.synchronize()
    e2e_s = max_over_ranks((time.perf_counter() - e0) / e2e_steps, world, dev)
    assert mtkv.mt_check_device_status(status) == 0, mtkv.mt_last_error()
    assert mtkv.mt_check_device_status(ws) == 0, mtkv.mt_last_error()

    if rank != 0:
        return None
    cpu = None
    if args.cpu_seconds > 0:
        times, cores, sample, layer_bytes, ltoks = oracle_layer_times(3)
        cpu_t = statistics.median(times)
        cpu = {"value": round(layer_bytes / cpu_t / 1e9, 5), "unit": "GB/s", "cores": cores,
               "kind": "oracle", "attended_tokens_per_s": round(ltoks / cpu_t, 1),
               "sample": sample + f", median of 3 runs ({cpu_t:.2f} s wall each)"}
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "kv_format": "f16", "n_layers": n_layers,
                   "n_seqs": B, "attended_tokens_per_layer": toks,
                   "store": ("fused into the decode launch" if fused else
                             "separate mt_kv_store launch"),
                   "launch": ("one CUDA graph per 32-layer step" if args.graph else
                              "eager launches (programmatic dependent launch)"),
                   "l2": "inputs larger than L2 (1.3 GB of K/V per layer, 42 GB per step)",
                   "parallelism": f"replicas x{world}"},
        "frac_of_peak": round(value / peak, 4),
        "step_ms": _spread(per_step),
        "attended_tokens_per_s": round(world * n_layers * toks / (ms_per_step * 1e-3), 1),
        "roofline": {"bound": "hbm",
                     "kernel": ("mt_paged_attn_decode_append (decode with the row store fused, "
                                "+ combine)" if fused else
                                "mt_paged_attn_decode (split-K decode + combine)"),
                     "achieved": round(achieved, 2), "peak": peak, "peak_kind": peak_kind,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "bytes_per_launch": call_bytes, "avg_launch_ms": round(dec_avg_ms, 5),
                     "traffic": _traffic_from_profile()},
        "e2e": {"value": round(whole_job_rate(step_bytes, e2e_s, world), 2), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_s * 1e3, 4),
                "copies": "pinned host buffers; all inputs host->device on one copy stream "
                          "at the step start, each layer's output device->host on a second "
                          "copy stream once that layer is done (overlapping later layers)"},
        "gpu_launches": args.steps * n_layers * (2 if fused else 3),
        "clocks": clk,
        "cpu_baseline": cpu,
    }
    return line


# ----------------------------------------------------------------- other workloads
#
# `--workload` selects one of the other synthetic configurations to measure the
# remaining kernels on GB300; the default line is the Llama-3 f16 step above.

def _spread(ms):
    """Median, min and max of per-step times (ms) from CUDA events."""
    return {"median": round(statistics.median(ms), 4), "min": round(min(ms), 4),
            "max": round(max(ms), 4), "n": len(ms)}


def _gpu_time(fn, steps, warmup, stream, graph=False, spread=None):
    """Mean ms per call of `fn` over `steps` timed calls after `warmup`;
    `spread`, if given, receives the per-call median / min / max."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    if graph:
        # time replays of `fn` captured as one CUDA graph
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        g.replay()
        torch.cuda.synchronize()
        fn = g.replay
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    marks[0].record(stream)
    for i in range(steps):
        fn()
        marks[i + 1].record(stream)
    torch.cuda.synchronize()
    if spread is not None:
        spread.update(_spread([marks[i].elapsed_time(marks[i + 1]) for i in range(steps)]))
    return marks[0].elapsed_time(marks[-1]) / steps


def _decode_setup(mtkv, w, n_pools, dev, g, table=None):
    """n_pools K/V pool pairs filled through mt_kv_store from N(0,1) rows."""
    hkv, d, bs = w.n_kv_heads, w.head_dim, w.block_size
    rb = mtkv.mt_kv_row_bytes(w.fmt, hkv, d)
    table = torch.from_numpy(w.block_table if table is None else table).to(dev)
    ctx = torch.from_numpy(w.context_lens).to(dev)
    spans = None if w.spans is None else torch.from_numpy(w.spans).to(dev)
    cells_all = torch.arange(w.n_cells, device=dev, dtype=torch.int64)
    layers = []
    for _ in range(n_pools):
        kp = torch.empty(w.n_cells, rb, dtype=torch.uint8, device=dev)
        vp = torch.empty_like(kp)
        for c0 in range(0, w.n_cells, 1 << 16):
            cells = cells_all[c0:c0 + (1 << 16)]
            rows = torch.randn(cells.numel(), hkv * d, generator=g, device=dev)
            mtkv.mt_kv_store(w.fmt, kp, vp, hkv, d, rows, -rows, cells)
        q = torch.randn(w.n_seqs, w.n_heads, d, generator=g, device=dev)
        out = torch.empty_like(q)
        args = mtkv.paged_attn_args(w.fmt, q, kp, vp, table, ctx, out, n_kv_heads=hkv,
                                    block_size=bs, n_phys_blocks=w.n_phys_blocks, scale=w.scale,
                                    spans=spans)
        k_new = torch.randn(w.n_seqs, hkv * d, generator=g, device=dev)
        layers.append((kp, vp, args, k_new))
    ws = torch.zeros(mtkv.mt_paged_attn_workspace_bytes(layers[0][2]), dtype=torch.uint8,
                     device=dev)
    return layers, ws, rb


def _window_bytes(w, rb_seg, table=None):
    """(unique-cell bytes, per-sequence logical bytes, attended positions) of
    one decode call: K+V head segments of attended positions (distinct
    physical cells counted once for the unique figure), table entries, Q, out."""
    table = w.block_table if table is None else table
    bs = w.block_size
    uniq, toks, blocks = set(), 0, 0
    for s in range(w.n_seqs):
        lo, hi = 0, int(w.context_lens[s])
        if w.spans is not None:
            lo, hi = max(int(w.spans[s, 0]), 0), min(int(w.spans[s, 1]), hi)
        for lb in range(lo // bs, (hi - 1) // bs + 1 if hi > lo else lo // bs):
            b = int(table[s, lb])
            blocks += 1
            if b < 0:
                continue
            a, z = max(lo, lb * bs), min(hi, lb * bs + bs)
            toks += z - a
            uniq.update(b * bs + p - lb * bs for p in range(a, z))
    fixed = blocks * 4 + w.n_seqs * 4 + 2 * w.n_seqs * w.n_heads * w.head_dim * 4
    per = w.n_kv_heads * rb_seg * 2
    return len(uniq) * per + fixed, toks * per + fixed, toks


def run_extra(args, rank, world, local_rank):
    from paged_kv_cache_gqa_gb300 import mtkv
    import __graft_entry__
    __graft_entry__.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    g = torch.Generator(device=dev)
    g.manual_seed(SEED + 7)
    peak, peak_kind = _peak()
    steps, warmup = args.steps, args.warmup
    clocks = Clocks(local_rank)
    res = {}
    if args.workload == "smollm2_f32":
        w = workloads.smollm2_f32(hist=False)
        layers, ws, rb = _decode_setup(mtkv, w, w.n_layers, dev, g)
        cells = torch.from_numpy(w.new_cells).to(dev)

        def step():
            for kp, vp, a, kn in layers:
                if args.store == "fused":
                    mtkv.mt_paged_attn_decode_append(a, kn, kn, ws)
                else:
                    mtkv.mt_kv_store("f32", kp, vp, w.n_kv_heads, w.head_dim, kn, kn, cells)
                    mtkv.mt_paged_attn_decode(a, ws)

        clocks.start()
        sp = {}
        ms = _gpu_time(step, steps, warmup, stream, graph=args.graph, spread=sp)
        ub, lb_, toks = _window_bytes(w, w.head_dim * 4)
        step_bytes = w.n_layers * (ub + store_bytes(w))
        value = step_bytes / (ms * 1e-3) / 1e9
        # grow-on-demand re-layout: 30 layers x kv_dim 192 f32, K and V, 64 -> 8192
        row = 192 * 4
        caps = [64]
        while caps[-1] < 8192:
            caps.append(mtkv.mt_kv_grow_capacity(caps[-1], caps[-1] + 1, 8192))
        bufs = [(torch.empty(30 * c * row, dtype=torch.uint8, device=dev),
                 torch.empty(30 * c * row, dtype=torch.uint8, device=dev)) for c in caps]

        def grow():
            for i in range(len(caps) - 1):
                for kv in range(2):
                    mtkv.mt_kv_relayout(bufs[i][kv], bufs[i + 1][kv], 30, caps[i], caps[i + 1], row)

        g_ms = _gpu_time(grow, steps, warmup, stream, graph=args.graph)
        g_bytes = sum(2 * 2 * 30 * c * row for c in caps[:-1])
        # copy_cells: 1000 overlapping run moves on the 60 pools (30 layers x K, V)
        moves, n_cells = workloads.compaction_moves(seed=SEED)
        ordered = np.asarray(mtkv.mt_order_moves(moves), dtype=np.int64)
        pools = [torch.empty(n_cells, row, dtype=torch.uint8, device=dev) for _ in range(60)]
        c_ms = _gpu_time(lambda: mtkv.mt_copy_cells(pools, row, n_cells, ordered), steps, warmup,
                         stream)
        c_bytes = int(ordered[:, 2].sum()) * row * 60 * 2
        clk = clocks.stop()
        res = {"metric": METRIC, "value": round(value, 2), "unit": "GB/s",
               "ms_per_step": round(ms, 4), "step_ms": sp, "frac_of_peak": round(value / peak, 4),
               "attended_tokens_per_s": round(w.n_layers * toks / (ms * 1e-3), 1),
               "config": {"workload": "smollm2-135m-shaped f32 paged decode: 30 layers, 8 seqs, "
                                      "ctx U[2048,8192], 9/3 heads, head_dim 64, bs 16",
                          "store": args.store, "graph": bool(args.graph)},
               "relayout": {"what": "grow 64->8192, 30 layers x kv_dim 192 f32, K and V",
                            "ms": round(g_ms, 4), "bytes": g_bytes,
                            "GB/s": round(g_bytes / (g_ms * 1e-3) / 1e9, 1),
                            "frac": round(g_bytes / (g_ms * 1e-3) / 1e9 / peak, 4)},
               "copy_cells": {"what": "1000 ordered overlapping run moves x 60 pools, 768 B rows",
                              "ms": round(c_ms, 4), "bytes": c_bytes,
                              "GB/s": round(c_bytes / (c_ms * 1e-3) / 1e9, 1),
                              "frac": round(c_bytes / (c_ms * 1e-3) / 1e9 / peak, 4)},
               "clocks": clk}
    elif args.workload == "q8_prefix":
        w = workloads.llama3_q8_prefix(hist=False, windows=args.windows)
        layers, ws, rb = _decode_setup(mtkv, w, 32, dev, g)
        cells = torch.from_numpy(w.new_cells).to(dev)
        groups = [(0, w.n_seqs, w.extra["prefix"] // w.block_size)]
        cascade = args.prefix == "cascade"
        if cascade:
            ws = torch.zeros(mtkv.mt_paged_attn_cascade_workspace_bytes(layers[0][2], groups),
                             dtype=torch.uint8, device=dev)

        fused = args.store == "fused"

        def step():
            for kp, vp, a, kn in layers:
                if fused and cascade:
                    mtkv.mt_paged_attn_decode_cascade_append(a, groups, kn, kn, ws)
                elif fused:
                    mtkv.mt_paged_attn_decode_append(a, kn, kn, ws)
                else:
                    mtkv.mt_kv_store("q8_0", kp, vp, w.n_kv_heads, w.head_dim, kn, kn, cells)
                    if cascade:
                        mtkv.mt_paged_attn_decode_cascade(a, groups, ws)
                    else:
                        mtkv.mt_paged_attn_decode(a, ws)

        clocks.start()
        sp = {}
        ms = _gpu_time(step, steps, warmup, stream, graph=args.graph, spread=sp)
        clk = clocks.stop()
        ub, lb_, toks = _window_bytes(w, (w.head_dim // 32) * 34)
        value = 32 * (ub + store_bytes(w)) / (ms * 1e-3) / 1e9
        res = {"metric": METRIC, "value": round(value, 2), "unit": "GB/s",
               "value_kind": "unique physical cells (shared prefix counted once)",
               "logical_GB/s": round(32 * lb_ / (ms * 1e-3) / 1e9, 1),
               "ms_per_step": round(ms, 4), "step_ms": sp, "frac_of_peak": round(value / peak, 4),
               "attended_tokens_per_s": round(32 * toks / (ms * 1e-3), 1),
               "config": {"workload": "llama3-8b-shaped q8_0 paged decode: 32 layers, 32 seqs "
                                      "sharing a 4096-token prefix + U[64,1024] suffix, " +
                                      ("random windows" if args.windows else "no windows") +
                                      ", 32/8 heads, head_dim 128, bs 32",
                          "prefix": ("cascade: shared blocks read once per group "
                                     "(mt_paged_attn_decode_cascade)" if cascade else
                                     "per-sequence decode (mt_paged_attn_decode)"),
                          "store": args.store, "graph": bool(args.graph)},
               "clocks": clk}
    elif args.workload == "llama3_formats":
        # The decode call (decode + combine, no store) on the Llama-3-8B-shaped
        # batch with each KV format in turn: 64 seqs, ctx log-uniform in
        # [512, 16384], 32/8 heads, head_dim 128; 4 rotated pool pairs per
        # format, so every call reads its K/V from HBM. Shows what the
        # format's in-register dequantisation costs against the HBM roofline.
        formats = {}
        clocks.start()
        for fmt, bs in (("f16", 16), ("f32", 16), ("q8_0", 16), ("q8_0", 32)):
            w = workloads.llama3_f16(fmt=fmt, block_size=bs, hist=False)
            layers, ws, rb = _decode_setup(mtkv, w, 4, dev, g)

            def decode():
                for kp, vp, a, kn in layers:
                    mtkv.mt_paged_attn_decode(a, ws)

            ms = _gpu_time(decode, steps, warmup, stream) / len(layers)
            assert mtkv.mt_check_device_status(ws) == 0, mtkv.mt_last_error()
            seg = {"f32": w.head_dim * 4, "f16": w.head_dim * 2,
                   "q8_0": (w.head_dim // 32) * 34}[fmt]
            ub, _lb, toks = _window_bytes(w, seg)
            gbs = ub / (ms * 1e-3) / 1e9
            formats[f"{fmt}_bs{bs}"] = {"row_bytes": rb, "bytes_per_call": ub,
                                        "us_per_call": round(ms * 1e3, 2),
                                        "GB/s": round(gbs, 1), "frac": round(gbs / peak, 4),
                                        "attended_tokens_per_s": round(toks / (ms * 1e-3), 1)}
            del layers, ws
            torch.cuda.empty_cache()
        clk = clocks.stop()
        q8 = formats["q8_0_bs32"]
        res = {"metric": METRIC, "value": q8["GB/s"], "unit": "GB/s",
               "value_kind": "q8_0 pools, block_size 32 (every format in `formats`)",
               "frac_of_peak": q8["frac"], "formats": formats,
               "config": {"workload": "llama3-8b-shaped paged decode call (decode + combine) per "
                                      "KV format: 64 seqs, ctx log-uniform [512,16384], 32/8 "
                                      "heads, head_dim 128; 4 rotated pool pairs per format"},
               "clocks": clk}
    elif args.workload in ("prefill_f16", "prefill_f16_long", "prefill_smollm2"):
        # chunked prefill through the paged cache, Llama-3-8B-shaped heads, f16
        # pools, the queries' K/V rows already stored; 8 layers with their own
        # pools, so successive calls do not hit in L2. prefill_f16: 16
        # sequences at context 2048 whose last 512 positions are the queries;
        # prefill_f16_long: one sequence at context 32768 whose last 256
        # positions are the queries (one chunk of a long prompt: 64 tiles,
        # fewer than the SMs); prefill_smollm2: SmolLM2-135M heads (9/3,
        # head_dim 64), 8 sequences at context 4096 whose last 512 positions
        # are the queries
        long_ = args.workload == "prefill_f16_long"
        smol = args.workload == "prefill_smollm2"
        n_seqs_p, ctx_p, n_q = (1, 32768, 256) if long_ else (8, 4096, 512) if smol else (16, 2048, 512)
        pfmt = args.prefill_format
        heads = dict(n_heads=9, n_kv_heads=3, head_dim=64) if smol else {}
        w = workloads.llama3_f16(seed=SEED + 9, n_seqs=n_seqs_p, ctx_lo=ctx_p, ctx_hi=ctx_p,
                                 hist=False, fmt=pfmt, **heads)
        layers, _, rb = _decode_setup(mtkv, w, 8, dev, g)
        table = torch.from_numpy(w.block_table).to(dev)
        ctx_d = torch.from_numpy(w.context_lens).to(dev)
        q_start = torch.arange(0, n_q * w.n_seqs + 1, n_q, dtype=torch.int32, device=dev)
        calls = []
        for kp, vp, _a, _kn in layers:
            q = torch.randn(n_q * w.n_seqs, w.n_heads, w.head_dim, generator=g, device=dev)
            out = torch.empty_like(q)
            a = mtkv.prefill_args(pfmt, q, kp, vp, table, ctx_d, q_start, out,
                                  n_kv_heads=w.n_kv_heads, block_size=w.block_size,
                                  n_phys_blocks=w.n_phys_blocks, scale=w.scale)
            calls.append(a)
        ws = torch.zeros(mtkv.mt_paged_prefill_workspace_bytes(calls[0]), dtype=torch.uint8,
                         device=dev)

        def step():
            for a in calls:
                mtkv.mt_paged_attn_prefill(a, ws)

        clocks.start()
        sp = {}
        ms = _gpu_time(step, steps, warmup, stream, spread=sp)
        clk = clocks.stop()
        assert mtkv.mt_check_device_status(ws) == 0, mtkv.mt_last_error()
        # each query j (position ctx - n + j) reads j + ctx - n + 1 positions;
        # per (query, head, position): q.k and p.v, 2 * head_dim MACs
        ctx0 = int(w.context_lens[0])
        pairs = w.n_seqs * sum(ctx0 - n_q + j + 1 for j in range(n_q))
        flop = 4.0 * pairs * w.n_heads * w.head_dim
        kv_bytes = 2 * int(w.context_lens.sum()) * rb
        tflops = len(calls) * flop / (ms * 1e-3) / 1e12
        tpeak = _tensor_peak()
        res = {"metric": "paged prefill attention TFLOP/s (f16 operands, f32 accumulate)"
                         + ("" if pfmt == "f16" else f", {pfmt} pools"),
               "value": round(tflops, 2), "unit": "TFLOP/s", "ms_per_step": round(ms, 4),
               "step_ms": sp,
               "ms_per_call": round(ms / len(calls), 5),
               "query_tokens_per_s": round(len(calls) * n_q * w.n_seqs / (ms * 1e-3), 1),
               "roofline": {"bound": "tensor", "achieved": round(tflops, 2),
                            "peak": tpeak[0], "peak_kind": tpeak[1], "unit": "TFLOP/s",
                            "frac": round(tflops / tpeak[0], 4),
                            "note": "useful FLOPs (4 * pairs * heads * head_dim); the kernel "
                                    "also multiplies the low half of q and padding rows"},
               "kv_GB_per_s": round(len(calls) * kv_bytes / (ms * 1e-3) / 1e9, 1),
               "config": {"workload": f"{'smollm2-135m' if smol else 'llama3-8b'}-shaped {pfmt} "
                                      f"chunked prefill: {n_seqs_p} seqs x ctx {ctx_p}, last "
                                      f"{n_q} positions as queries, "
                                      f"{w.n_heads}/{w.n_kv_heads} heads, head_dim "
                                      f"{w.head_dim}, bs 16, 8 layers"},
               "clocks": clk}
    elif args.workload == "longctx_int4":
        w = workloads.longctx_f16_int4(hist=False)
        table = workloads.retarget_cold(w)
        layers, ws, rb = _decode_setup(mtkv, w, min(4, args.layers), dev, g, table=table)
        src = torch.from_numpy(w.extra["cold_src"]).to(dev)
        dst = torch.from_numpy(w.extra["cold_dst"]).to(dev)
        n_el = w.block_size * w.n_kv_heads * w.head_dim
        scales = torch.empty(len(src), dtype=torch.float32, device=dev)
        nib = torch.empty(len(src), n_el // 2, dtype=torch.uint8, device=dev)

        def quant():
            for kp, vp, a, kn in layers:
                for pool in (kp, vp):
                    mtkv.mt_kv_quant_int4("f16", pool, w.block_size, w.n_kv_heads, w.head_dim,
                                          w.n_phys_blocks, src, scales, nib)

        def dequant():
            for kp, vp, a, kn in layers:
                for pool in (kp, vp):
                    mtkv.mt_kv_dequant_int4("f16", pool, w.block_size, w.n_kv_heads, w.head_dim,
                                            w.n_phys_blocks, dst, scales, nib)

        def decode():
            for kp, vp, a, kn in layers:
                mtkv.mt_paged_attn_decode(a, ws)

        clocks.start()
        d_ms = _gpu_time(decode, steps, warmup, stream) / len(layers)
        q_ms = _gpu_time(quant, steps, warmup, stream) / (2 * len(layers))
        dq_ms = _gpu_time(dequant, steps, warmup, stream) / (2 * len(layers))
        clk = clocks.stop()
        ub, lb_, toks = _window_bytes(w, w.head_dim * 2, table=table)
        value = ub / (d_ms * 1e-3) / 1e9
        q_bytes = len(src) * (n_el * 2 + n_el // 2 + 4)
        res = {"metric": METRIC, "value": round(value, 2), "unit": "GB/s",
               "ms_per_decode": round(d_ms, 4), "frac_of_peak": round(value / peak, 4),
               "attended_tokens_per_s": round(toks / (d_ms * 1e-3), 1),
               "int4_quant": {"blocks": len(src), "ms": round(q_ms, 4),
                              "GB/s": round(q_bytes / (q_ms * 1e-3) / 1e9, 1),
                              "frac": round(q_bytes / (q_ms * 1e-3) / 1e9 / peak, 4)},
               "int4_dequant": {"blocks": len(dst), "ms": round(dq_ms, 4),
                                "GB/s": round(q_bytes / (dq_ms * 1e-3) / 1e9, 1),
                                "frac": round(q_bytes / (dq_ms * 1e-3) / 1e9 / peak, 4)},
               "config": {"workload": "long-context f16 paged decode: 16 seqs x 32768, 16/4 heads, "
                                      "head_dim 256, bs 16, 5% holes, 25% of blocks through int4 "
                                      "into fresh ids; 4 rotated pool pairs"},
               "clocks": clk}
    else:
        raise SystemExit(f"unknown workload {args.workload}")
    res.update({"n_gpus": 1, "steps": steps, "warmup": warmup, "higher_is_better": True,
                "peak": peak, "peak_kind": peak_kind, "data": "synthetic",
                "workload_name": args.workload})
    return res


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="mtkv", choices=["mtkv", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="0 skips the CPU oracle baseline (profiling runs); any other value "
                         "runs it: one whole layer over all host cores, three times")
    ap.add_argument("--workload", default="llama3_f16",
                    choices=["llama3_f16", "smollm2_f32", "q8_prefix", "longctx_int4",
                             "llama3_formats", "prefill_f16", "prefill_f16_long",
                             "prefill_smollm2"],
                    help="llama3_f16 is the benchmark line; the others measure the other kernels")
    ap.add_argument("--prefill-format", default="f16", choices=["f16", "q8_0", "f32"],
                    help="KV pool format of the prefill workloads (all on the tcgen05 "
                         "kernel: q8_0 after staging as f16 rows, f32 after staging as "
                         "high/low f16 pairs)")
    ap.add_argument("--store", default=None, choices=["fused", "separate"],
                    help="store each layer's new row inside the decode launch "
                         "(mt_paged_attn_decode_append) or with its own mt_kv_store launch; "
                         "default: fused for f32/f16 pools, separate for q8_0 (whose "
                         "quantiser would run on the copy-issuing warp)")
    ap.add_argument("--prefix", default="cascade", choices=["cascade", "plain"],
                    help="q8_prefix workload: decode the shared prefix once per group "
                         "(mt_paged_attn_decode_cascade) or per sequence")
    ap.add_argument("--windows", action=argparse.BooleanOptionalAction, default=True,
                    help="q8_prefix workload: each query's random attn_span window (the "
                         "configuration) or its whole context")
    ap.add_argument("--graph", action=argparse.BooleanOptionalAction, default=True,
                    help="replay the L-layer step as one captured CUDA graph")
    ap.add_argument("--layers", type=int, default=N_LAYERS,
                    help="layers per step; fewer than 32 only for profiling captures")
    args = ap.parse_args()
    if args.store is None:
        args.store = "separate" if args.workload == "q8_prefix" else "fused"
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group(backend)
    if args.impl == "reference":
        line = run_reference(args, rank)
    elif args.workload != "llama3_f16":
        line = run_extra(args, rank, world, local_rank)
    else:
        line = run_gpu(args, rank, world, local_rank)
    if line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
