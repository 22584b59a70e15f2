#!/usr/bin/env python3
"""Benchmark of the NVFP4 KV-cache quantizer on GB300.

Metric: NVFP4 smooth+quantize GB/s (and fraction of HBM peak) per KV chunk.
Workload (one step): one layer's chunk of the LongLive-2.0 KV write -- K and V,
each 7040 tokens (8 frames x 880) x 24 heads x 128 channels, bf16, resident in
HBM -- K smoothed and both quantized with Four-Over-Six NVFP4 scales in one
batched enqueue.  Algorithmic bytes per element: 2 read + 0.5 codes + 1/16
scale = 2.5625 B.

Timed region: K steps replayed from a CUDA graph over rotating input/output
sets whose footprint exceeds 2x L2 (reads come from HBM), bracketed by a
barrier and cudaDeviceSynchronize, measured with CUDA events on the launching
stream, max over ranks.  N > 1 runs independent replicas (weak scaling).

--impl reference times the CPU oracle (the plain C statement of the method)
on the host cores on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

T_CHUNK, HEADS, HEAD_DIM = 7040, 24, 128
QUANT_BYTES_PER_ELEM = 2.0 + 0.5 + 1.0 / 16.0      # bf16 in, nibble codes out, one E4M3 scale per 16
DEQUANT_BYTES_PER_ELEM = 0.5 + 1.0 / 16.0 + 2.0    # codes + scales in, bf16 out
W2D_BYTES_PER_ELEM = 2.0 + 0.5 + 1.0 / 256.0       # bf16 in, codes out, one scale per 16x16 tile
METRIC = "NVFP4 smooth+quantize GB/s and fraction of GB300 HBM peak per KV chunk"
FALLBACK_HBM_GBS = 6800.0

# DRAM bytes (read + write) per launch of each kernel on this step's workload, from one ncu
# capture of this script (dram__bytes_read.sum + dram__bytes_write.sum); drop an entry when its
# kernel changes.  The quantization kernel's entry is dropped: its wait loop's sleep interval
# changed after that capture (22.0 MB per launch then).
NCU_TRAFFIC = {"kv_stats": 114275200, "kv_quant": None}
# ALU-pipe warp instructions per launch of the quantization kernel on this step (same capture,
# sm__inst_executed_pipe_alu.sum); the pass is bound by instruction issue (half of it on the
# half-rate ALU pipe), not by HBM.  The later sleep-interval change touches only the wait loop.
NCU_ALU_INST = {"kv_quant": 7.526e6}
ALU_PEAK_PER_SM_CLK = 2.0  # warp instructions: one per SM sub-partition every 2 cycles


def parse():
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20000)
    p.add_argument("--warmup", type=int, default=200)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--no-rows", action="store_true", help="skip the secondary rows (dequant, weights, 30 layers)")
    p.add_argument("--rows", nargs="+", default=None, metavar="ROW",
                   help="run only these secondary rows: kv_write_30_layers kv_cache_read_dequant kv_cache_view_gather "
                        "kv_attention_decode kv_attention_prefill gemm_w4a4 weight_quant_2d activation_quant_1d k_only_smooth_quant")
    p.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline")
    p.add_argument("--e2e-steps", type=int, default=30)
    return p.parse_args()


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# ---------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.proc = None
        self.lines = []

    def __enter__(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50"]
        if self.uuid:
            cmd += ["-i", self.uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------- distributed
def dist_setup():
    import torch

    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(ws, v: float) -> float:
    if ws == 1:
        return v
    import torch
    import torch.distributed as dist

    t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------- CPU oracle
def cpu_oracle_run(tokens: int, reps: int = 1):
    """Time the oracle on K and V of the first `tokens` tokens of the chunk; returns (GB/s, seconds, elems)."""
    import numpy as np  # noqa: F401

    import oracle
    from nvfp4_block_quantization_gb300 import workloads as W

    oracle.build()
    K = W.to_bf16_bits(W.chunk_k(2000))[:tokens].copy()
    V = W.to_bf16_bits(W.chunk_v(2001))[:tokens].copy()
    t0 = time.perf_counter()
    for _ in range(reps):
        oracle.kv_smooth_quant(K, smooth=True)
        oracle.kv_smooth_quant(V, smooth=False)
    dt = time.perf_counter() - t0
    elems = 2 * K.size * reps
    return elems * QUANT_BYTES_PER_ELEM / dt / 1e9, dt, elems


def cpu_oracle_threads_run(tokens: int, threads: int):
    """The same step on `threads` host threads (the oracle's threaded driver: bit-identical results);
    returns (GB/s, seconds, elems)."""
    import oracle
    from nvfp4_block_quantization_gb300 import workloads as W

    oracle.build()
    K = W.to_bf16_bits(W.chunk_k(2000))[:tokens].copy()
    V = W.to_bf16_bits(W.chunk_v(2001))[:tokens].copy()
    t0 = time.perf_counter()
    oracle.kv_smooth_quant_threads(K, True, threads)
    oracle.kv_smooth_quant_threads(V, False, threads)
    dt = time.perf_counter() - t0
    elems = 2 * K.size
    return elems * QUANT_BYTES_PER_ELEM / dt / 1e9, dt, elems


def cpu_oracle_rows(threads: int) -> dict:
    """The oracle on configs 3-5 with the rows' byte accounting, each on a stated sample scaled up by
    bytes (so the default run stays within about half a minute of CPU time).  The KV quantizer runs
    on `threads` host threads (the threaded driver, bit-identical); dequant and the weight quantizer
    have single-threaded statements only."""
    import numpy as np

    import oracle
    from nvfp4_block_quantization_gb300 import workloads as W

    oracle.build()
    rows = {}
    # config 3: 30 layers of K (smoothed) and V with their per-layer seeds; layers 0 and 29 timed
    secs = 0.0
    for layer in (0, 29):
        sk, sv = W.layer_seeds(layer)
        K = W.to_bf16_bits(W.chunk_k(sk))
        V = W.to_bf16_bits(W.chunk_v(sv))
        t0 = time.perf_counter()
        oracle.kv_smooth_quant_threads(K, True, threads)
        oracle.kv_smooth_quant_threads(V, False, threads)
        secs += time.perf_counter() - t0
    per_layer = 2 * K.size * QUANT_BYTES_PER_ELEM
    rows["kv_write_30_layers"] = {"GB/s": 2 * per_layer / secs / 1e9, "threads": threads, "seconds_sample": secs,
                                  "sample": "layers 0 and 29 of 30 (seeds 3000 + 2l, 3001 + 2l), scaled by bytes"}
    # config 4: dequant of a 21-frame view (18,480 tokens) of K (mean re-added, per-frame groups) and V;
    # the codes are the config-2 chunk's, repeated to the view's length
    qk = oracle.kv_smooth_quant_threads(W.to_bf16_bits(W.chunk_k(2000)), True, threads)
    qv = oracle.kv_smooth_quant_threads(W.to_bf16_bits(W.chunk_v(2001)), False, threads)
    n_tok, L = 21 * 880, 880
    rep = lambda a: np.ascontiguousarray(np.concatenate([a] * 3, axis=0)[:n_tok])
    groups = n_tok // L
    gk = np.full(groups, qk["g"], np.float32)
    gv = np.full(groups, qv["g"], np.float32)
    mk = np.ascontiguousarray(np.broadcast_to(qk["mean"][None], (groups,) + qk["mean"].shape), dtype=np.float32)
    ck, sk_, cv, sv_ = rep(qk["codes"]), rep(qk["scales"]), rep(qv["codes"]), rep(qv["scales"])
    t0 = time.perf_counter()
    oracle.kv_dequant(ck, sk_, gk, mk, tokens_per_group=L)
    oracle.kv_dequant(cv, sv_, gv, None, tokens_per_group=L)
    secs = time.perf_counter() - t0
    deq_bytes = 2 * n_tok * HEADS * HEAD_DIM * QUANT_BYTES_PER_ELEM
    rows["kv_cache_read_dequant"] = {"GB/s": deq_bytes / secs / 1e9, "threads": 1, "seconds_sample": secs,
                                     "sample": "K (mean) and V of one 21-frame view"}
    # config 5: weights (one matrix of each shape timed, scaled by bytes to all six) and activations
    secs, el = 0.0, 0
    for i, (M, N) in ((0, W.WEIGHT_SHAPES[0]), (4, W.WEIGHT_SHAPES[4])):
        w = W.to_bf16_bits(W.weight(i, M, N))
        t0 = time.perf_counter()
        oracle.weight_quant_2d(w)
        secs += time.perf_counter() - t0
        el += M * N
    rows["weight_quant_2d"] = {"GB/s": el * (2 + 0.5 + 1.0 / 256) / secs / 1e9, "threads": 1, "seconds_sample": secs,
                               "sample": "matrices 0 (3072x3072) and 4 (3072x14336) of six, scaled by bytes"}
    x = W.to_bf16_bits(W.activations()).reshape(T_CHUNK, 1, 3072)
    t0 = time.perf_counter()
    oracle.kv_smooth_quant_threads(x, False, threads)
    secs = time.perf_counter() - t0
    rows["activation_quant_1d"] = {"GB/s": x.size * QUANT_BYTES_PER_ELEM / secs / 1e9, "threads": threads,
                                   "seconds_sample": secs, "sample": "the whole 7040x3072 activation"}
    return rows


def cpu_model() -> str:
    """The host CPU's name from /proc/cpuinfo (x86: model name; Arm: implementer and part), or ''."""
    try:
        info = {}
        with open("/proc/cpuinfo") as f:
            for ln in f:
                if ":" in ln:
                    k, v = ln.split(":", 1)
                    info.setdefault(k.strip(), v.strip())
        if "model name" in info:
            return info["model name"]
        return " ".join(f"{k} {info[k]}" for k in ("CPU implementer", "CPU part") if k in info)
    except OSError:
        return ""


def run_reference(args, ws, rank):
    if rank != 0:
        return
    # Each step is a bounded sample (the first n tokens of K and V) sized so the whole run stays
    # within about 90 s of single-core oracle time.
    probe_gbs, probe_s, probe_el = cpu_oracle_run(64)
    el_per_s = probe_el / probe_s
    steps_total = args.steps + args.warmup
    tokens = int(max(1, min(T_CHUNK, 90.0 * el_per_s / max(steps_total, 1) / (2 * HEADS * HEAD_DIM))))
    import oracle
    from nvfp4_block_quantization_gb300 import workloads as W

    K = W.to_bf16_bits(W.chunk_k(2000))[:tokens].copy()
    V = W.to_bf16_bits(W.chunk_v(2001))[:tokens].copy()
    for _ in range(args.warmup):
        oracle.kv_smooth_quant(K, smooth=True)
        oracle.kv_smooth_quant(V, smooth=False)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.kv_smooth_quant(K, smooth=True)
        oracle.kv_smooth_quant(V, smooth=False)
    dt = time.perf_counter() - t0
    step_bytes = 2 * K.size * QUANT_BYTES_PER_ELEM
    value = step_bytes * args.steps / dt / 1e9
    sample = f"K and V of tokens 0..{tokens - 1} of the 7040x24x128 bf16 chunk per step"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / max(args.steps, 1) * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "kv_chunk_7040x24x128_bf16_K_smooth+V", "tokens": T_CHUNK, "heads": HEADS,
                   "head_dim": HEAD_DIM, "input": "bf16", "parallelism": f"replicas{args.gpus}"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "host_cores": os.cpu_count(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------- GPU (ours)
def run_ours(args, ws, rank):
    import numpy as np
    import torch

    import nvfp4_block_quantization_gb300 as nv
    from nvfp4_block_quantization_gb300 import workloads as W
    from nvfp4_block_quantization_gb300.build import build

    build()
    nv.load_library()
    dev = torch.device("cuda", torch.cuda.current_device())
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 128 << 20))
    uuid = None
    try:
        uuid = "GPU-" + str(props.uuid)
    except Exception:
        pass

    # ---- inputs: one chunk's K and V (seeded), replicated into rotating sets
    Kb, Vb = W.chunk_kv_bf16(2000, 2001)
    K0 = torch.from_numpy(Kb.view(np.int16)).view(torch.bfloat16).to(dev)
    V0 = torch.from_numpy(Vb.view(np.int16)).view(torch.bfloat16).to(dev)
    n_el = K0.numel()
    step_bytes = 2 * n_el * QUANT_BYTES_PER_ELEM
    rot = max(4, int(np.ceil(2.0 * l2 / step_bytes)) + 1)
    sets = []
    for _ in range(rot):
        xs = [K0.clone(), V0.clone()]
        outs, status = nv.kv_smooth_quant_batched(xs, [True, False])  # allocates outputs + status
        ws_t = nv.kv_workspace(T_CHUNK, HEADS, HEAD_DIM, 2, dev)
        sets.append((xs, outs, status, ws_t))
    torch.cuda.synchronize()

    def step(i):
        xs, outs, status, ws_t = sets[i % rot]
        nv.kv_smooth_quant_batched(xs, [True, False], workspace=ws_t, outs=outs, status=status)

    # ---- capture one round (rot steps) in a CUDA graph
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for i in range(rot):
            step(i)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    # a graph of one rotation round (rot steps) plus one single-step graph per rotation set:
    # whole rounds run from the round graph and the remainder from single-step graphs, so
    # exactly W warm-up steps and K timed steps run
    g_round = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_round):
        for i in range(rot):
            step(i)
    singles = []
    for i in range(rot):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step(i)
        singles.append(g)

    def run_steps(n):
        for _ in range(n // rot):
            g_round.replay()
        for i in range(n % rot):
            singles[i].replay()

    steps = max(1, args.steps)
    warm = max(3, args.warmup)
    run_steps(warm)
    torch.cuda.synchronize()

    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(uuid) as clk:
        barrier(ws)
        torch.cuda.synchronize()
        ev0.record()
        run_steps(steps)
        ev1.record()
        torch.cuda.synchronize()
        barrier(ws)
    ms = ev0.elapsed_time(ev1)
    ms = max_over_ranks(ws, ms)
    ms_per_step = ms / steps
    value = ws * steps * step_bytes / (ms * 1e-3) / 1e9
    per_gpu_gbs = steps * step_bytes / (ms * 1e-3) / 1e9

    # status check: every set must report finite inputs
    for xs, outs, status, _ in sets:
        assert int(status.item()) == 0

    # ---- end to end through the public API with host buffers.  Every step copies its K and V
    # from pinned host memory and its codes, scales, tensor scales, mean and status back.  Two
    # buffer sets and three streams: step i's host->device copy runs while step i-1 is
    # quantized and step i-2's results go back, so the host link (about 207 GB/s each way on
    # this part, copy engine or SM loads alike) is the bound, not the sum of the three phases.
    kh = torch.empty_like(K0, device="cpu").pin_memory()
    vh = torch.empty_like(V0, device="cpu").pin_memory()
    kh.copy_(K0.cpu())
    vh.copy_(V0.cpu())
    ws_d = nv.kv_workspace(T_CHUNK, HEADS, HEAD_DIM, 2, dev)

    class _Set:
        def __init__(self):
            self.xs = [torch.empty_like(K0), torch.empty_like(V0)]
            self.outs, self.status = nv.kv_smooth_quant_batched(self.xs, [True, False], workspace=ws_d)
            self.host = [(torch.empty_like(o.codes, device="cpu").pin_memory(),
                          torch.empty_like(o.scales, device="cpu").pin_memory(),
                          torch.empty_like(o.tensor_scale, device="cpu").pin_memory()) for o in self.outs]
            self.mean_h = torch.empty_like(self.outs[0].mean, device="cpu").pin_memory()
            self.status_h = torch.empty(1, dtype=torch.int32).pin_memory()
            self.loaded, self.computed, self.drained = (torch.cuda.Event() for _ in range(3))

    e2e_sets = [_Set(), _Set()]
    outs_d = e2e_sets[0].outs
    d2h_bytes = sum(o.codes.numel() + o.scales.numel() + 4 for o in outs_d) + outs_d[0].mean.numel() * 4 + 4
    h2d_bytes = (K0.numel() + V0.numel()) * 2
    main_s, h2d_s, d2h_s = torch.cuda.current_stream(), torch.cuda.Stream(), torch.cuda.Stream()

    def e2e_step(i):
        b = e2e_sets[i % 2]
        with torch.cuda.stream(h2d_s):
            h2d_s.wait_event(b.computed)  # step i-2 has read these input buffers
            b.xs[0].copy_(kh, non_blocking=True)
            b.xs[1].copy_(vh, non_blocking=True)
            b.loaded.record(h2d_s)
        main_s.wait_event(b.loaded)
        main_s.wait_event(b.drained)  # step i-2's results have left these output buffers
        nv.kv_smooth_quant_batched(b.xs, [True, False], workspace=ws_d, outs=b.outs, status=b.status)
        b.computed.record(main_s)
        with torch.cuda.stream(d2h_s):
            d2h_s.wait_event(b.computed)
            for o, (hc, hs, hg) in zip(b.outs, b.host):
                hc.copy_(o.codes, non_blocking=True)
                hs.copy_(o.scales, non_blocking=True)
                hg.copy_(o.tensor_scale, non_blocking=True)
            b.mean_h.copy_(b.outs[0].mean, non_blocking=True)
            b.status_h.copy_(b.status, non_blocking=True)
            b.drained.record(d2h_s)

    for i in range(3):
        e2e_step(i)
    main_s.wait_stream(d2h_s)
    torch.cuda.synchronize()
    barrier(ws)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(main_s)
    for i in range(args.e2e_steps):
        e2e_step(i)
    main_s.wait_stream(h2d_s)
    main_s.wait_stream(d2h_s)
    e1.record(main_s)
    torch.cuda.synchronize()
    barrier(ws)
    e2e_ms = max_over_ranks(ws, e0.elapsed_time(e1))
    e2e_value = ws * args.e2e_steps * step_bytes / (e2e_ms * 1e-3) / 1e9
    for b in e2e_sets:
        assert int(b.status_h.item()) == 0
        assert torch.equal(b.host[0][0], b.outs[0].codes.cpu()) and torch.equal(b.host[1][1], b.outs[1].scales.cpu())

    # ---- per-kernel launch durations, live: the same step as its two enqueues with CUDA events
    # between them on the launching stream (queue kept ahead of the GPU)
    ka, kb = [], []
    n_k = min(400, max(40, steps // 50))
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
            torch.cuda.Event(enable_timing=True)) for _ in range(n_k)]
    torch.cuda.synchronize()
    for i, (ea, eb, ec) in enumerate(evs):
        xs, outs, status, ws_t = sets[i % rot]
        ea.record()
        nv.kv_stats_batched(xs, [True, False], ws_t, outs)
        eb.record()
        nv.kv_quant_batched(xs, [True, False], ws_t, outs, status)
        ec.record()
    torch.cuda.synchronize()
    for ea, eb, ec in evs[4:]:
        ka.append(ea.elapsed_time(eb))
        kb.append(eb.elapsed_time(ec))
    stats_ms, quant_ms = statistics.mean(ka), statistics.mean(kb)
    stats_bytes = 2 * n_el * 2.0       # K and V read once (the algorithmic read)
    quant_bytes = 2 * n_el * 0.5625    # codes and scales written (its re-read of K and V is not algorithmic)
    kernels = {"kv_stats": {"ms_per_launch": stats_ms, "algorithmic_bytes": stats_bytes,
                            "GB/s": stats_bytes / (stats_ms * 1e-3) / 1e9},
               "kv_quant": {"ms_per_launch": quant_ms, "algorithmic_bytes": quant_bytes,
                            "GB/s": quant_bytes / (quant_ms * 1e-3) / 1e9},
               "launches_timed": len(ka),
               "method": "the step's two passes enqueued separately with CUDA events between them; the event "
                         "stops the quantization grid from starting beside the statistics grid, so the two "
                         "durations add up to more than the step",
               "step_ms": ms_per_step,
               "overlap_ms": stats_ms + quant_ms - ms_per_step}
    dom = "kv_quant" if quant_ms >= stats_ms else "kv_stats"

    peak, peak_kind = measured_peaks()
    clocks = clk.summary()
    if dom == "kv_quant":
        sm_mhz = clocks.get("sm_mhz") or 2070.0
        alu_peak = props.multi_processor_count * ALU_PEAK_PER_SM_CLK * sm_mhz * 1e6 / 1e9
        alu_ach = NCU_ALU_INST["kv_quant"] / (quant_ms * 1e-3) / 1e9
        roofline = {"bound": "alu", "achieved": alu_ach, "peak": alu_peak, "unit": "G warp-inst/s (ALU pipe)",
                    "frac": alu_ach / alu_peak, "traffic": NCU_TRAFFIC.get(dom), "kernel": dom,
                    "peak_source": "SMs x 2 ALU warp-instructions per SM per clock x sampled SM clock",
                    "alu_inst_per_launch": NCU_ALU_INST["kv_quant"],
                    "hbm_frac": kernels[dom]["GB/s"] / peak, "step_frac": per_gpu_gbs / peak}
    else:
        roofline = {"bound": "hbm", "achieved": kernels[dom]["GB/s"], "peak": peak, "unit": "GB/s",
                    "frac": kernels[dom]["GB/s"] / peak, "traffic": NCU_TRAFFIC.get(dom),
                    "kernel": dom, "peak_source": f"{peak_kind} hbm_gbs",
                    "algorithmic_bytes_per_launch": kernels[dom]["algorithmic_bytes"],
                    "step_frac": per_gpu_gbs / peak}
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws, "steps": steps, "warmup": warm,
        "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded numpy PCG64; K offsets N(0,9)+N(0,1) with 0.5% x16 channels, V N(0,1))",
        "config": {"workload": "kv_chunk_7040x24x128_bf16_K_smooth+V", "tokens": T_CHUNK, "frames": 8,
                   "tokens_per_frame": 880, "heads": HEADS, "head_dim": HEAD_DIM, "input": "bf16",
                   "tensors_per_step": 2, "bytes_per_step": step_bytes,
                   "l2": f"rotating {rot} input/output sets ({rot * step_bytes / 1e6:.0f} MB > 2x L2 {l2 / 1e6:.0f} MB)",
                   "graph": "CUDA graph of one rotation round, single-step graphs for the remainder",
                   "parallelism": f"replicas{ws}"},
        "elements_per_s": ws * steps * 2 * n_el / (ms * 1e-3),
        "roofline": roofline,
        "kernels": kernels,
        "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d_bytes, "d2h_bytes_per_step": d2h_bytes,
                "ms_per_step": e2e_ms / args.e2e_steps},
        "gpu_launches": steps * 2,
        "clocks": clocks,
    }

    if not args.no_rows:
        line["rows"] = secondary_rows(nv, W, torch, dev, peak, args.rows)
        line["size_ceiling"] = size_ceiling_rows(torch, dev, l2)
        batched = line["rows"].get("kv_write_30_layers")
        if isinstance(batched, dict) and "frac" in batched:
            # the same quantizer over a 30-layer batch (each layer's quantization overlapping the next
            # layer's statistics): the headline's companion
            line["batched_companion"] = {"row": "kv_write_30_layers", "value": batched.get("GB/s"), "unit": "GB/s",
                                         "frac_of_hbm_peak": batched["frac"]}
    if not args.no_cpu and rank == 0:
        gbs, secs, elems = cpu_oracle_run(T_CHUNK)
        nthreads = os.cpu_count() or 1
        tgbs, tsecs, _ = cpu_oracle_threads_run(T_CHUNK, nthreads)
        line["cpu_baseline"] = {"value": gbs, "unit": "GB/s", "cores": 1, "host_cores": os.cpu_count(), "kind": "oracle",
                                "cpu_model": cpu_model(),
                                "sample": f"the whole step: K (smoothed) and V of the 7040x24x128 chunk, "
                                          f"{elems} elements, {secs:.1f} s single-threaded",
                                "all_cores": {"value": tgbs, "unit": "GB/s", "cores": nthreads, "seconds": tsecs,
                                              "kind": "oracle, threaded driver (channel, element and block ranges "
                                                      "split over the host's cores; bit-identical results)"},
                                "rows": cpu_oracle_rows(nthreads)}
    if rank == 0:
        print(json.dumps(line), flush=True)


def _time_graph(torch, fn, reps_in_graph, replays, warm=2):
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for i in range(reps_in_graph):
            fn(i)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(reps_in_graph):
            fn(i)
    for _ in range(warm):
        g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(replays):
        g.replay()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / (reps_in_graph * replays)  # ms per fn call


def size_ceiling_rows(torch, dev, l2):
    """What a plain device copy (torch's, not this library) reaches at this step's sizes.

    Same method as the step: a CUDA graph replayed over rotating buffers whose
    footprint exceeds 2x L2, so every read comes from HBM and no dirty lines are
    left for the timed kernel to write back.  Bytes are read + written.
    """
    out = {}
    for label, n in (("one_tensor_43MB", T_CHUNK * HEADS * HEAD_DIM), ("k_and_v_86MB", 2 * T_CHUNK * HEADS * HEAD_DIM)):
        nbuf = max(4, int(2 * 2.5 * l2 // (n * 2)) + 1)
        srcs = [torch.empty(n, dtype=torch.bfloat16, device=dev).fill_(1.0) for _ in range(nbuf)]
        dsts = [torch.empty_like(srcs[0]) for _ in range(nbuf)]
        ms = _time_graph(torch, lambda i: dsts[i % nbuf].copy_(srcs[i % nbuf]), nbuf, 10)
        nbytes = n * 2 * 2
        out[f"torch_copy_{label}"] = {"GB/s": nbytes / (ms * 1e-3) / 1e9, "us": ms * 1e3, "bytes": nbytes,
                                      "method": f"graph over {nbuf} rotating buffer pairs"}
        del srcs, dsts
    return out


def _chunk_k_device(torch, gen, dev):
    """One layer's K chunk on the device: per-(head, channel) offsets N(0, 3^2) plus N(0, 1) noise,
    15 whole channels (0.5%) scaled by 16, bf16 (the same law as the step's K)."""
    off = torch.randn((HEADS, HEAD_DIM), generator=gen, device=dev) * 3.0
    k = torch.randn((T_CHUNK, HEADS, HEAD_DIM), generator=gen, device=dev) + off
    ch = torch.randperm(HEADS * HEAD_DIM, generator=gen, device=dev)[:15]
    k.view(T_CHUNK, -1)[:, ch] *= 16.0
    return k.to(torch.bfloat16)


def row_kv_write_30_layers(nv, W, torch, dev, peak):
    """Full-model chunk write: K and V of all 30 layers in one batched call.  Layer l's K and V
    are drawn with the per-layer seeds 3000 + 2l and 3001 + 2l (numpy PCG64, the step's laws)."""
    import numpy as np

    L = 30
    xs, flags = [], []
    for layer in range(L):
        sk, sv = W.layer_seeds(layer)
        for bits in (W.to_bf16_bits(W.chunk_k(sk)), W.to_bf16_bits(W.chunk_v(sv))):
            xs.append(torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(dev))
        flags += [True, False]
    outs, status = nv.kv_smooth_quant_batched(xs, flags)
    wsb = nv.kv_workspace(T_CHUNK, HEADS, HEAD_DIM, 2 * L, dev)
    ms = _time_graph(torch, lambda i: nv.kv_smooth_quant_batched(xs, flags, workspace=wsb, outs=outs, status=status),
                     1, 20)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    b = 2 * L * T_CHUNK * HEADS * HEAD_DIM * QUANT_BYTES_PER_ELEM
    return {"GB/s": b / ms / 1e6, "ms": ms, "bytes": b, "frac": b / ms / 1e6 / peak,
            "inputs": "numpy PCG64, K seed 3000 + 2l, V seed 3001 + 2l"}


def row_kv_cache_read_dequant(nv, W, torch, dev, peak):
    """Cache read: 21 frames (3 global-sink frames of chunk 0 + the 18 most recent frames of
    chunks 0..2) x 880 tokens, quantized by this library from seeded chunks; four caches, K and V
    of two layers.  K's per-frame groups carry each frame's chunk tensor scale and mean (re-added
    on the way out), V's only the tensor scale."""
    gen = torch.Generator(device=dev)
    gen.manual_seed(3000)
    Tc, F = 21 * 880, 880
    frame_src = [(0, f) for f in range(3)] + [(0, 6), (0, 7)] + [(1, f) for f in range(8)] + [(2, f) for f in range(8)]
    caches = []
    for t in range(4):
        is_k = t % 2 == 0
        chunk_q = []
        for c in range(3):
            x = _chunk_k_device(torch, gen, dev) if is_k else \
                torch.randn((T_CHUNK, HEADS, HEAD_DIM), generator=gen, device=dev).to(torch.bfloat16)
            chunk_q.append(nv.kv_smooth_quant(x, is_k))
            del x
        codes = torch.cat([chunk_q[c].codes[f * F:(f + 1) * F] for c, f in frame_src])
        scales = torch.cat([chunk_q[c].scales[f * F:(f + 1) * F] for c, f in frame_src])
        gs = torch.cat([chunk_q[c].tensor_scale for c, f in frame_src])
        means = torch.stack([chunk_q[c].mean for c, f in frame_src]) if is_k else None
        out = torch.empty((Tc, HEADS, HEAD_DIM), dtype=torch.bfloat16, device=dev)
        caches.append((codes, scales, gs, means, out))
        del chunk_q
    ms = _time_graph(torch, lambda i: nv.kv_dequant(*caches[i % 4][:3], mean=caches[i % 4][3],
                                                    tokens_per_group=F, out=caches[i % 4][4]), 8, 20)
    ms_k = _time_graph(torch, lambda i: nv.kv_dequant(*caches[2 * (i % 2)][:3], mean=caches[2 * (i % 2)][3],
                                                      tokens_per_group=F, out=caches[2 * (i % 2)][4]), 8, 20)
    b = Tc * HEADS * HEAD_DIM * DEQUANT_BYTES_PER_ELEM
    return {"GB/s": b / ms / 1e6, "ms_per_tensor": ms, "ms_per_k_tensor": ms_k, "bytes": b,
            "frac": b / ms / 1e6 / peak}


def row_kv_cache_view_gather(nv, W, torch, dev, peak):
    """Cache read through the multi-shot cache manager: five 8-frame chunks written straight into
    pool slots, then the next chunk's view (3 global-sink frames + the 18 most recent frames = 21
    frames x 880 tokens) expanded by the gathered read from its slots; K (mean re-added) and V of
    two layers, four pools in rotation."""
    gen = torch.Generator(device=dev)
    gen.manual_seed(3100)
    F, Lf = 8, 880
    pools, views = [], []
    for layer in range(2):
        cache = nv.KvCache(F, Lf, 3, 3, 18)
        pk = nv.KvCachePool.allocate(cache, HEADS, HEAD_DIM, smooth=True, device=dev)
        pv = nv.KvCachePool.allocate(cache, HEADS, HEAD_DIM, smooth=False, device=dev)
        for c in range(5):
            slot = cache.append()
            k = _chunk_k_device(torch, gen, dev)
            v = torch.randn((T_CHUNK, HEADS, HEAD_DIM), generator=gen, device=dev).to(torch.bfloat16)
            st = torch.zeros(1, dtype=torch.int32, device=dev)
            nv.kv_smooth_quant_batched([k, v], [True, False],
                                       outs=[pk.slot_outputs(cache, slot, st), pv.slot_outputs(cache, slot, st)],
                                       status=st)
            del k, v
        fi, fr, fs = cache.view()
        assert len(fi) == 21
        for pool, is_k in ((pk, True), (pv, False)):
            out = torch.empty((len(fi) * Lf, HEADS, HEAD_DIM), dtype=torch.bfloat16, device=dev)
            pools.append((pool, fr, fs, is_k, out))
    torch.cuda.synchronize()

    def call(i):
        pool, fr, fs, is_k, out = pools[i % 4]
        nv.kv_gather_dequant(pool, fr, fs, Lf, with_mean=is_k, out=out)

    ms = _time_graph(torch, call, 8, 20)
    b = 21 * Lf * HEADS * HEAD_DIM * DEQUANT_BYTES_PER_ELEM
    return {"GB/s": b / ms / 1e6, "ms_per_tensor": ms, "bytes": b, "frac": b / ms / 1e6 / peak,
            "view_frames": 21, "slots_per_pool": 5}


def row_kv_attention_decode(nv, W, torch, dev, peak):
    """Attention reading the NVFP4 cache: 1 and 4 query tokens per head over the 21-frame view (3 sink
    + 18 rolling frames x 880 tokens, 24 heads x 128) of two layers' K and V pools, K and V dequantized
    in registers.  Bytes: the view's K and V codes and scales (0.5625 B per cached element each)."""
    gen = torch.Generator(device=dev)
    gen.manual_seed(3200)
    F, Lf = 8, 880
    layers = []
    for layer in range(2):
        cache = nv.KvCache(F, Lf, 3, 3, 18)
        pk = nv.KvCachePool.allocate(cache, HEADS, HEAD_DIM, smooth=True, device=dev)
        pv = nv.KvCachePool.allocate(cache, HEADS, HEAD_DIM, smooth=False, device=dev)
        for c in range(5):
            slot = cache.append()
            k = _chunk_k_device(torch, gen, dev)
            v = torch.randn((T_CHUNK, HEADS, HEAD_DIM), generator=gen, device=dev).to(torch.bfloat16)
            st = torch.zeros(1, dtype=torch.int32, device=dev)
            nv.kv_smooth_quant_batched([k, v], [True, False],
                                       outs=[pk.slot_outputs(cache, slot, st), pv.slot_outputs(cache, slot, st)],
                                       status=st)
            del k, v
        fi, fr, fs = cache.view()
        layers.append((pk, pv, fr, fs))
    n_tok = 21 * Lf
    b = 2 * n_tok * HEADS * HEAD_DIM * (0.5 + 1.0 / 16.0)
    out = {"bytes": b, "view_tokens": n_tok}
    for n_q in (1, 4):
        q = torch.randn((n_q, HEADS, HEAD_DIM), generator=gen, device=dev)
        wsp = torch.empty(nv._lib.nvfp4_kv_attention_workspace_bytes(21, Lf, HEADS, HEAD_DIM, n_q),
                          dtype=torch.uint8, device=dev)
        o = torch.empty((n_q, HEADS, HEAD_DIM), dtype=torch.float32, device=dev)

        def call(i):
            pk, pv, fr, fs = layers[i % 2]
            nv.kv_attention_decode(q, pk, pv, fr, fs, Lf, HEAD_DIM ** -0.5, workspace=wsp, out=o)

        ms = _time_graph(torch, call, 8, 20)
        out[f"n_q={n_q}"] = {"ms": ms, "GB/s": b / ms / 1e6, "frac": b / ms / 1e6 / peak}
    return out


def row_kv_attention_prefill(nv, W, torch, dev, peak):
    """Attention of a whole new chunk (7040 query tokens, 24 heads x 128, bf16) over the 21-frame view
    (3 sink + 18 rolling frames x 880 tokens) read from one layer's NVFP4 K and V pools, on the tensor
    cores (nvfp4_kv_attention_prefill).  FLOPs: 4 n_q n_keys D per head (Q K^T and P V)."""
    gen = torch.Generator(device=dev)
    gen.manual_seed(3300)
    F, Lf = 8, 880
    cache = nv.KvCache(F, Lf, 3, 3, 18)
    pk = nv.KvCachePool.allocate(cache, HEADS, HEAD_DIM, smooth=True, device=dev)
    pv = nv.KvCachePool.allocate(cache, HEADS, HEAD_DIM, smooth=False, device=dev)
    for c in range(5):
        slot = cache.append()
        k = _chunk_k_device(torch, gen, dev)
        v = torch.randn((T_CHUNK, HEADS, HEAD_DIM), generator=gen, device=dev).to(torch.bfloat16)
        st = torch.zeros(1, dtype=torch.int32, device=dev)
        nv.kv_smooth_quant_batched([k, v], [True, False],
                                   outs=[pk.slot_outputs(cache, slot, st), pv.slot_outputs(cache, slot, st)],
                                   status=st)
        del k, v
    fi, fr, fs = cache.view()
    n_keys = len(fr) * Lf
    q = (torch.randn((T_CHUNK, HEADS, HEAD_DIM), generator=gen, device=dev) * 0.5).to(torch.bfloat16)
    o = torch.empty((T_CHUNK, HEADS, HEAD_DIM), dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    # the last, partial wave of (query tile, head) units runs split along the keys, in this workspace
    ws_bytes = nv._lib.nvfp4_kv_attention_prefill_workspace_bytes(T_CHUNK, HEADS, len(fr), Lf)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)

    def call(i):
        nv.kv_attention_prefill(q, pk, pv, fr, fs, Lf, HEAD_DIM ** -0.5, out=o, status=status, workspace=ws)

    def call_whole(i):
        nv.kv_attention_prefill(q, pk, pv, fr, fs, Lf, HEAD_DIM ** -0.5, out=o, status=status, split=False)

    ms = _time_graph(torch, call, 2, 5)
    ms_whole = _time_graph(torch, call_whole, 2, 5)
    fl = 4.0 * T_CHUNK * n_keys * HEAD_DIM * HEADS
    pk_tf, src = bf16_peak_tflops()
    torch.cuda.synchronize()
    return {"ms": ms, "TFLOP/s": fl / ms / 1e9, "flops": fl, "n_q": T_CHUNK, "n_keys": n_keys,
            "peak_tflops": pk_tf, "peak_source": src, "frac": fl / ms / 1e9 / pk_tf,
            "split_units": ws_bytes // (2 * (256 * 128 + 512) * 4), "ms_without_key_split": ms_whole,
            "dev_status": int(status.item())}


FALLBACK_BF16_TFLOPS = 1900.0
FP4_OVER_BF16 = 13.5 / 2.25  # nominal dense FP4 / BF16 tensor rates of the part


FALLBACK_BF16_TFLOPS_SUSTAINED = 1700.0


def bf16_peak_tflops():
    """Dense bf16 peak for a kernel timed in a long loop: the measured cuBLAS bf16 rate sustained over
    seconds under the power cap."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops_sustained"]), "measured bf16 sustained"
    except Exception:
        return FALLBACK_BF16_TFLOPS_SUSTAINED, "fallback bf16 sustained"


def fp4_peak_tflops():
    """Dense FP4 peak: the measured cuBLAS bf16 burst rate times the nominal FP4/BF16 ratio."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]) * FP4_OVER_BF16, "measured bf16 x nominal fp4/bf16 ratio 6"
    except Exception:
        return FALLBACK_BF16_TFLOPS * FP4_OVER_BF16, "fallback bf16 x nominal fp4/bf16 ratio 6"


def row_gemm_w4a4(nv, W, torch, dev, peak):
    """W4A4 linear layer: activations 7040 x 3072 ~ N(0, 1) quantized with 1-D blocks, four 3072 x 3072
    weights ~ N(0, 0.02^2) quantized with 16x16 tiles (weights and their tensor-core scales prepared
    once), Y = X W^T in bf16.  Times the GEMM alone (four weights in rotation) and the whole linear
    step: quantize X, rearrange its scales, GEMM."""
    gen = torch.Generator(device=dev)
    gen.manual_seed(5200)
    M, N, K = T_CHUNK, 3072, 3072
    x = torch.randn((M, 1, K), generator=gen, device=dev).to(torch.bfloat16)
    xq = nv.kv_smooth_quant(x, False)
    xs = nv.mma_scales(xq.scales.view(M, K // 16), K)
    wts = []
    for i in range(4):
        w = (torch.randn((N, K), generator=gen, device=dev) * 0.02).to(torch.bfloat16)
        wq = nv.weight_quant_2d(w)
        wts.append((wq, nv.mma_scales(wq.scales, K, tile2d=True)))
        del w
    plan = nv.GemmPlan(M, N, K)
    ws = nv.gemm_workspace(dev)
    ys = [torch.empty((M, N), dtype=torch.bfloat16, device=dev) for _ in range(4)]
    xc = xq.codes.view(M, K // 2)

    def gemm(i):
        wq, wsc = wts[i % 4]
        nv.gemm_w4a4(plan, xc, xs, xq.tensor_scale, wq.codes, wsc, wq.tensor_scale, ws, out=ys[i % 4])

    ms = _time_graph(torch, gemm, 8, 20)
    aws = nv.kv_workspace(M, 1, K, 1, dev)

    def linear(i):
        nv.kv_smooth_quant(x, False, workspace=aws, out=xq)
        nv.mma_scales(xq.scales.view(M, K // 16), K, out=xs)
        gemm(i)

    ms_lin = _time_graph(torch, linear, 8, 20)
    fl = 2.0 * M * N * K
    pk, src = fp4_peak_tflops()
    out = {"TFLOP/s": fl / ms / 1e9, "ms_gemm": ms, "ms_linear_step": ms_lin, "flops": fl,
           "peak_tflops": pk, "peak_source": src, "frac": fl / ms / 1e9 / pk}

    # the wide weight shape of the workload: 14336 outputs from 3072 inputs
    N2 = 14336
    w2 = (torch.randn((N2, K), generator=gen, device=dev) * 0.02).to(torch.bfloat16)
    w2q = nv.weight_quant_2d(w2)
    w2s = nv.mma_scales(w2q.scales, K, tile2d=True)
    del w2
    plan2 = nv.GemmPlan(M, N2, K)
    y2 = torch.empty((M, N2), dtype=torch.bfloat16, device=dev)
    ms2 = _time_graph(torch, lambda i: nv.gemm_w4a4(plan2, xc, xs, xq.tensor_scale, w2q.codes, w2s,
                                                    w2q.tensor_scale, ws, out=y2), 4, 20)
    fl2 = 2.0 * M * N2 * K
    out["gemm_7040x14336x3072"] = {"TFLOP/s": fl2 / ms2 / 1e9, "ms": ms2, "frac": fl2 / ms2 / 1e9 / pk}
    torch.cuda.synchronize()
    out["kernel_error_flag"] = int(ws[:4].view(torch.int32).item())  # set by a bounded wait that gave up

    # random Hadamard transform of the activation (bf16 in, fp32 out: 6 bytes per element)
    signs = int(torch.randint(0, 1 << 16, (1,), generator=gen, device=dev).item())
    xr = torch.empty((M, K), dtype=torch.float32, device=dev)
    ms_rht = _time_graph(torch, lambda i: nv.rht16(x.view(M, K), signs, out=xr), 8, 20)
    out["rht16_activation"] = {"ms": ms_rht, "bytes": 6.0 * M * K, "GB/s": 6.0 * M * K / ms_rht / 1e6,
                               "frac": 6.0 * M * K / ms_rht / 1e6 / peak}
    # error of Y against the exact product, without and with the transform, on a weight with the
    # workload's outliers (0.1% of entries x30)
    w = torch.randn((N, K), generator=gen, device=dev) * 0.02
    idx = torch.randperm(N * K, generator=gen, device=dev)[: N * K // 1000]
    w.view(-1)[idx] *= 30.0
    w = w.to(torch.bfloat16)
    exact = x.view(M, K).double() @ w.double().T

    def rel(y):
        return float(torch.linalg.norm(y.double() - exact) / torch.linalg.norm(exact))

    xq = nv.kv_smooth_quant(x, False)
    wq = nv.weight_quant_2d(w)
    y0 = nv.gemm_w4a4(plan, xq.codes.view(M, K // 2), nv.mma_scales(xq.scales.view(M, K // 16), K),
                      xq.tensor_scale, wq.codes, nv.mma_scales(wq.scales, K, tile2d=True), wq.tensor_scale, ws)
    xrq = nv.kv_smooth_quant(nv.rht16(x.view(M, K), signs).view(M, 1, K), False)
    wrq = nv.weight_quant_2d(nv.rht16(w, signs))
    y1 = nv.gemm_w4a4(plan, xrq.codes.view(M, K // 2), nv.mma_scales(xrq.scales.view(M, K // 16), K),
                      xrq.tensor_scale, wrq.codes, nv.mma_scales(wrq.scales, K, tile2d=True), wrq.tensor_scale, ws)
    out["rel_frobenius_error_vs_exact"] = {"w4a4": rel(y0), "w4a4_with_rht16": rel(y1)}

    # the activation side fused (transform, quantize, scales in the tensor-core layout) against
    # the separate calls, each followed by the GEMM with a weight prepared once
    wr_s = nv.mma_scales(wrq.scales, K, tile2d=True)
    aq = nv.act_quant_mma(x.view(M, K))
    aws2 = torch.empty(nv._lib.nvfp4_act_quant_workspace_bytes(), dtype=torch.uint8, device=dev)
    xw = nv.kv_workspace(M, 1, K, 1, dev)
    xrq_o = nv.kv_smooth_quant(xr.view(M, 1, K), False)
    xr_s = nv.mma_scales(xrq_o.scales.view(M, K // 16), K)
    yy = torch.empty((M, N), dtype=torch.bfloat16, device=dev)

    def fused_plain(i):
        nv.act_quant_mma(x.view(M, K), None, workspace=aws2, out=aq)
        nv.gemm_w4a4(plan, aq.codes, aq.scales_mma, aq.tensor_scale, wts[i % 4][0].codes, wts[i % 4][1],
                     wts[i % 4][0].tensor_scale, ws, out=ys[i % 4])

    def composed_rht(i):
        nv.rht16(x.view(M, K), signs, out=xr)
        nv.kv_smooth_quant(xr.view(M, 1, K), False, workspace=xw, out=xrq_o)
        nv.mma_scales(xrq_o.scales.view(M, K // 16), K, out=xr_s)
        nv.gemm_w4a4(plan, xrq_o.codes.view(M, K // 2), xr_s, xrq_o.tensor_scale, wrq.codes, wr_s,
                     wrq.tensor_scale, ws, out=yy)

    def fused_rht(i):
        nv.act_quant_mma(x.view(M, K), signs, workspace=aws2, out=aq)
        nv.gemm_w4a4(plan, aq.codes, aq.scales_mma, aq.tensor_scale, wrq.codes, wr_s, wrq.tensor_scale, ws, out=yy)

    out["linear_step_ms"] = {"quantize+scales+gemm": ms_lin, "fused_quant+gemm": _time_graph(torch, fused_plain, 8, 20),
                             "rht+quantize+scales+gemm": _time_graph(torch, composed_rht, 8, 20),
                             "fused_rht_quant+gemm": _time_graph(torch, fused_rht, 8, 20)}
    return out


def row_weight_quant_2d(nv, W, torch, dev, peak):
    """Weights: 4 x 3072x3072 and 2 x 3072x14336 bf16, N(0, 0.02^2), 16x16 tiles, in one batched call
    (and, for comparison, as six single calls)."""
    gen = torch.Generator(device=dev)
    ws_ = []
    for i, (M, N) in enumerate(W.WEIGHT_SHAPES):
        gen.manual_seed(5000 + i)
        w = (torch.randn((M, N), generator=gen, device=dev) * 0.02).to(torch.bfloat16)
        ws_.append((w, nv.weight_quant_2d(w), nv.w2d_workspace(M, N, dev)))
    mats = [w for (w, _, _) in ws_]
    bouts, bstatus = nv.weight_quant_2d_batched(mats)
    bws = nv.w2d_batched_workspace(len(mats), dev)
    ms = _time_graph(torch, lambda i: nv.weight_quant_2d_batched(mats, workspace=bws, outs=bouts, status=bstatus),
                     1, 10)
    ms_single = _time_graph(torch, lambda i: [nv.weight_quant_2d(w, workspace=wk, out=o) for (w, o, wk) in ws_],
                            1, 10)
    b = sum(M * N for (M, N) in W.WEIGHT_SHAPES) * W2D_BYTES_PER_ELEM
    return {"GB/s": b / ms / 1e6, "ms_all_six": ms, "ms_six_single_calls": ms_single, "bytes": b,
            "frac": b / ms / 1e6 / peak}


def row_activation_quant_1d(nv, W, torch, dev, peak):
    """Activations 7040 x 3072 bf16 ~ N(0, 1), 1-D 16-element blocks (four rotating matrices)."""
    gen = torch.Generator(device=dev)
    gen.manual_seed(5100)
    acts = [torch.randn((T_CHUNK, 1, 3072), generator=gen, device=dev).to(torch.bfloat16) for _ in range(4)]
    aouts = [nv.kv_smooth_quant(a, False) for a in acts]
    aws = nv.kv_workspace(T_CHUNK, 1, 3072, 1, dev)
    ms = _time_graph(torch, lambda i: nv.kv_smooth_quant(acts[i % 4], False, workspace=aws, out=aouts[i % 4]), 8, 20)
    b = T_CHUNK * 3072 * QUANT_BYTES_PER_ELEM
    return {"GB/s": b / ms / 1e6, "ms": ms, "bytes": b, "frac": b / ms / 1e6 / peak}


def row_k_only_smooth_quant(nv, W, torch, dev, peak):
    """A single K tensor smoothed and quantized alone (no V to overlap with); four rotating K."""
    gen = torch.Generator(device=dev)
    gen.manual_seed(3000)
    kx = [_chunk_k_device(torch, gen, dev) for _ in range(4)]
    kouts = [nv.kv_smooth_quant(k, True) for k in kx]
    kws = nv.kv_workspace(T_CHUNK, HEADS, HEAD_DIM, 1, dev)
    ms = _time_graph(torch, lambda i: nv.kv_smooth_quant(kx[i % 4], True, workspace=kws, out=kouts[i % 4]), 8, 20)
    b = T_CHUNK * HEADS * HEAD_DIM * QUANT_BYTES_PER_ELEM
    return {"GB/s": b / ms / 1e6, "ms": ms, "bytes": b, "frac": b / ms / 1e6 / peak}


ROWS = {"kv_write_30_layers": row_kv_write_30_layers, "kv_cache_read_dequant": row_kv_cache_read_dequant,
        "kv_cache_view_gather": row_kv_cache_view_gather, "kv_attention_decode": row_kv_attention_decode,
        "kv_attention_prefill": row_kv_attention_prefill,
        "gemm_w4a4": row_gemm_w4a4,
        "weight_quant_2d": row_weight_quant_2d, "activation_quant_1d": row_activation_quant_1d,
        "k_only_smooth_quant": row_k_only_smooth_quant}


def secondary_rows(nv, W, torch, dev, peak, names=None):
    """The other hot-path rows, each on its own seeded synthetic workload (device-generated)."""
    rows = {}
    for name in (names or list(ROWS)):
        rows[name] = ROWS[name](nv, W, torch, dev, peak)
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    return rows


def main():
    args = parse()
    ws, rank, _ = dist_setup()
    if args.impl == "reference":
        run_reference(args, ws, rank)
    else:
        run_ours(args, ws, rank)
    if ws > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
