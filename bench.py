"""Benchmark of the CSA2 layer step on GB300 (prints one JSON line).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload decode|decode_fp8kv|prefill|hierarchical|
                    ragged|encoder_stack|decoder_stack|decoder_stack_prefill|decoder_replay|ced_compress]
    python bench.py --impl reference ...      # the CPU oracle on a bounded sample

A step is one pass of the layer group over one batch of synthetic input,
inputs resident in HBM: for the default decode workload (32 sequences x one
token over a 131,072-token context, Full mode) that is window pack, index
scoring of every visible entry, Top-512 and sparse attention.  L2 is flushed
before every timed step: 512 MB are written and then 512 MB of another
buffer are read, so that no input is resident and the L2 holds clean lines
(a write alone leaves ~126 MB of dirty lines whose write-back would be
charged to the first kernels of the step).  Under torchrun each rank runs an
independent replica on its own GPU (weak scaling, no collective on the data
path); rank 0 prints the line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "CSA2 sparse-attn tokens/s (decode@128K, prefill@64K); % HBM/TC roofline"
FLUSH_BYTES = 512 << 20


# ---------------------------------------------------------------------------------
# workload bytes / flops (algorithmic: what the method must move or compute)

def workload_config(wl):
    """The workload's shape keys of the JSON line's config (the same in both arms)."""
    return {"workload": wl.name, "description": wl.description, "B": wl.B, "tokens_per_step": wl.B * wl.Tq,
            "layers": "".join(wl.layers), "K": wl.K, "Hq": wl.Hq, "d": wl.d, "W": wl.W,
            "indexer": f"{wl.Hi}x{wl.Di} {wl.idx_dtype}", "kv": kv_desc(wl)}


def kv_desc(wl):
    if getattr(wl, "kv_format", "mxfp4") == "fp8":
        return f"FP8 E4M3 + fp32 scale, {wl.d + 4} B/entry, 64-entry pages"
    return f"MXFP4 {wl.d // 2 + wl.d // 16} B/entry, 64-entry pages"


def algorithmic(wl):
    """Per-step algorithmic work of the workload's hot path: unique HBM bytes and FLOPs.

    Bytes count what a step must move at least once: each sequence's visible
    indexer keys per Full layer (all query tokens of a sequence share them),
    the pooled keys per Reindex layer (the pools of one sequence's tokens overlap,
    so at most its visible keys), the selected MXFP4 (or FP8) entries (at most the
    entries that exist), the queries read, the outputs written and the index
    scores written and read back once, plus the hidden states of a prefill
    chunk.  For one query token per sequence this is the per-query sum.
    """
    d, Di, K, W, Hq = wl.d, wl.Di, wl.K, wl.W, wl.Hq
    fp8kv = getattr(wl, "kv_format", "mxfp4") == "fp8"
    entry_bytes = d + 4 if fp8kv else d // 2 + d // 16    # 516 B FP8 / 288 B MXFP4 entry (d = 512)
    idx_elt = 2 if wl.idx_dtype == "bf16" else 4
    scan = 0          # indexer keys read by Full layers (unique per sequence)
    pooled = 0        # indexer keys read by Reindex layers
    gathered = 0      # selected MXFP4 entries gathered by attention (unique bound)
    io = 0            # queries, outputs, index scores
    attn_flops = 0
    idx_flops = 0
    for b in range(wl.B):
        n_ent = wl.entries_after(b)
        nvs = [max(0, min(n_ent, (wl.t_first[b] + i + 1) // 4)) for i in range(wl.Tq)]
        for mode in wl.layers:
            if mode == "F":
                scan += max(nvs) * Di * idx_elt
            sel = 0
            pooled_seq = 0
            for i in range(wl.Tq):
                t = wl.t_first[b] + i
                nv = nvs[i]
                nk = min(K, nv)
                # a rebuilt window (SWA Bounded Replay) starts at the first replayed token
                nwin = min(W, t + 1) if wl.replay_H is None else min(W, i + 1)
                sel += nk
                if mode == "F":
                    idx_flops += 2 * nv * wl.Hi * Di
                    io += 2 * nv * 4                     # score written, read back by the Top-K
                elif mode == "X":
                    npos = min(nv, wl.pool_blocks * wl.pool_block)
                    pooled_seq += npos
                    idx_flops += 2 * npos * wl.Hi * Di
                    io += 2 * npos * 4
                attn_flops += 4 * Hq * d * (nk + nwin)
            gathered += min(sel, n_ent) * entry_bytes
            pooled += min(pooled_seq, max(nvs)) * Di * idx_elt   # a sequence's pools overlap: unique keys
            io += wl.Tq * Hq * d * (2 + 4)                # Q (bf16) in, O (fp32) out
    compress_flops = 0
    if wl.H is not None:
        compress_flops = 2 * sum(wl.new_entries(b) for b in range(wl.B)) * 4 * wl.H * (d + Di)
        io += wl.B * wl.Tq * wl.H * 2                     # hidden states (bf16)
    if wl.replay_H is not None:
        # every layer projects its replayed tokens onto window rows: hidden states in, FP8 rows out
        n_rows = wl.B * wl.Tq * len(wl.layers)
        compress_flops += 2 * n_rows * wl.replay_H * d
        io += n_rows * (wl.replay_H * 2 + d + 4)
    n_full = max(1, sum(1 for m in wl.layers if m == "F"))
    return {"scan_bytes": scan, "pooled_bytes": pooled, "gathered_bytes": gathered, "io_bytes": io,
            "step_bytes": scan + pooled + gathered + io, "attn_flops": attn_flops, "index_flops": idx_flops,
            "compress_flops": compress_flops,
            # one launch of the dominant kernels: a Full layer's scan, one layer's attention
            # (every layer of a step attends over the same key counts)
            "scan_bytes_per_launch": scan // n_full, "attn_flops_per_launch": attn_flops // len(wl.layers)}


def replica_seed(seed: int, rank: int) -> int:
    """Every rank runs an independent replica: its own seeded batch of sequences."""
    return seed + 1000 * rank


def max_over_ranks(x: float, dist, device="cpu") -> float:
    """The slowest rank's value (the job is done when the last replica is)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t)


def make_workload(name):
    from csa2_inputs import workloads as WL
    return WL.ALL[name]()


# ---------------------------------------------------------------------------------
# clocks sampled during the timed region

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits", "-lms", "50",
                 "-i", str(self.dev)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        time.sleep(0.1)
        self.lines = []
        if self.proc:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        if not self.lines:
            return None
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            try:
                sm.append(float(f[1]))
                mx = max(mx, float(f[2]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------------
# ncu traffic figure committed under profiles/ (used only while the kernel is unchanged)

def kernel_source_hash(path):
    return hashlib.sha256(open(path, "rb").read()).hexdigest()[:16]


def committed_traffic(profile_md, src_path):
    try:
        text = open(profile_md).read()
    except OSError:
        return None
    m_sha = re.search(r"source_sha256_16:\s*([0-9a-f]{16})", text)
    m_tr = re.search(r"traffic_bytes_per_launch:\s*([0-9.e+]+)", text)
    if not (m_sha and m_tr) or m_sha.group(1) != kernel_source_hash(src_path):
        return None
    return float(m_tr.group(1))


# ---------------------------------------------------------------------------------
# GPU arm

def run_gpu(args, rank, world, dist):
    import torch

    from compressed_sparse_attention_05_gb300 import build

    build.build()
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    line = measure(args, args.workload, args.steps, rank, world, dist, local)
    # the metric's second configuration (prefill@64K) rides on the default decode line
    if args.workload == "decode" and not args.no_prefill:
        sub = measure(args, "prefill", max(3, min(args.steps, 400)), rank, world, dist, local)
        if sub is not None:
            for k in ("metric", "n_gpus", "higher_is_better", "scaling", "vs_baseline", "dtype", "data"):
                sub.pop(k, None)
            line["prefill"] = sub
    if rank == 0:
        print(json.dumps(line), flush=True)


def measure(args, workload, steps, rank, world, dist, local):
    """Times `steps` steps of one workload (after args.warmup warm-up steps) and returns
    its JSON object on rank 0 (None elsewhere)."""
    import torch

    from compressed_sparse_attention_05_gb300 import abi, harness

    dev = torch.device("cuda", local)
    wl = make_workload(workload)
    wl.seed = replica_seed(wl.seed, rank)
    alg = algorithmic(wl)
    g = harness.LayerGroup(wl, f"cuda:{local}")
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream()

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    for w in range(args.warmup):
        flush(w)
        g.step()
    torch.cuda.synchronize()
    assert abi.csa2_get_status() == 0

    # ---- headline: K steps, inputs resident, L2 flushed before each
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    barrier()
    n0 = abi.csa2_launch_count()
    with ClockSampler(local) as clk:
        for k in range(steps):
            flush(k)
            ev[k][0].record(stream)
            g.step()
            ev[k][1].record(stream)
        barrier()
    launches = abi.csa2_launch_count() - n0
    step_ms = [a.elapsed_time(b) for a, b in ev]
    ms = sum(step_ms) / steps
    ms_all = max_over_ranks(ms, dist, dev)

    # ---- dominant kernel, timed alone on the same stream through its own entry point
    kern = time_dominant_kernel(args, g, wl, flush, stream)

    # ---- a replay step's own kernels: one layer's window rebuild, timed alone
    replay = time_replay(args, g, wl, flush, stream) if wl.replay_H is not None else None

    # ---- end to end through the public call with host buffers
    e2e = time_e2e(args, g, flush, stream, dist)

    status = abi.csa2_get_status()
    if rank != 0:
        return None
    tokens = wl.B * wl.Tq
    value = world * tokens / (ms_all / 1e3)
    peaks = load_peaks()
    roof = roofline(wl, alg, kern, peaks)
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": steps,
        "warmup": args.warmup, "ms_per_step": ms_all, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": dict(workload_config(wl),
                       l2="flushed before every timed step (512 MB written, then 512 MB read)",
                       parallelism=f"replicas x{world}" if world > 1 else "single GPU"),
        "roofline": roof,
        "step_roofline": step_roofline(wl, alg, ms, peaks),
        "e2e": e2e,
        "gpu_launches": launches,
        "status_word": status,
        "step_ms_p50": statistics.median(step_ms), "step_ms_min": min(step_ms),
        "clocks": clk.summary(),
    }
    if replay is not None:
        flops = 2 * wl.B * wl.Tq * wl.replay_H * wl.d
        achieved = flops / (replay / 1e3) / 1e12
        line["replay_roofline"] = {
            "bound": "tensor", "kernel": "k_compress_gemm_tma (one token per row) + k_norm_rope_fp8_window",
            "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
            "frac": achieved / peaks["bf16_tflops"], "traffic": None, "algorithmic_flops_per_launch": flops,
            "kernel_ms": replay, "peak_source": peaks["source"] + " (bf16 burst)",
            "note": "one layer's csa2_swa_replay (projection GEMM + RMSNorm/RoPE/FP8 epilogue), L2 flushed"}
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline_all(workload, args.cpu_seconds)
    return line


# ---------------------------------------------------------------------------------
# the decoder layers' KV from one hidden state (csa2_compress_layers)

CED_LAYERS = 20   # the decoder layers of the pages' 40-layer model


def ced_setup(dev):
    """The prefill chunk's hidden states and CED_LAYERS layers' stacked weights, one
    page pool per layer (the chunk's 1,024 entries after 15,360 cached ones)."""
    import torch

    from compressed_sparse_attention_05_gb300 import abi
    wl = make_workload("prefill")
    G = wl.n_new // 4
    first = wl.entries_before(0)
    pages = (first + G + 63) // 64
    hidden = wl.hidden(dev)
    W_all = wl.w_layers(CED_LAYERS, dev)
    gamma = torch.stack([wl.gamma(dev)] * CED_LAYERS)
    keep, caches = [], []
    for l in range(CED_LAYERS):
        t = {"codes": torch.zeros(pages * 64, wl.d // 2, dtype=torch.uint8, device=dev),
             "scales": torch.zeros(pages * 64, wl.d // 16, dtype=torch.uint8, device=dev),
             "idx": torch.zeros(pages * 64, wl.Di, dtype=torch.bfloat16, device=dev),
             "pt": torch.arange(pages, dtype=torch.int32, device=dev).reshape(1, pages),
             "n": torch.tensor([first + G], dtype=torch.int32, device=dev)}
        keep.append(t)
        caches.append(abi.Cache(kv_codes=t["codes"].data_ptr(), kv_scales=t["scales"].data_ptr(),
                                idx_k=t["idx"].data_ptr(), page_table=t["pt"].data_ptr(),
                                n_entries=t["n"].data_ptr(), n_pages=pages))
    dims = abi.Dims(B=1, Tq=wl.n_new, d=wl.d, r=wl.r, Hq=wl.Hq, Hi=wl.Hi, Di=wl.Di, idx_dtype=abi.CSA2_BF16,
                    K=wl.K, W=wl.W, max_pages=pages, n_pool_blocks=0, pool_block=8, swa_cap=0)
    fe = torch.tensor([first], dtype=torch.int32, device=dev)
    ws = torch.empty(abi.csa2_compress_layers_workspace_size(1, wl.n_new, wl.H, CED_LAYERS, wl.d, wl.Di),
                     dtype=torch.uint8, device=dev)

    def step():
        abi.csa2_compress_layers(hidden, W_all, wl.Di, gamma, wl.eps, wl.rope_base, fe, dims, caches, ws)

    return wl, hidden, keep, step


def run_ced(args, rank, world, dist):
    """--workload ced_compress: one step = CED_LAYERS layers' KV of the prefill chunk
    from one hidden state (one GEMM over the stacked weights, then every layer's pack in one launch)."""
    import torch

    from compressed_sparse_attention_05_gb300 import abi, build

    build.build()
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl, hidden, keep, step = ced_setup(dev)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream()
    for w in range(args.warmup):
        flush(w)
        step()
    torch.cuda.synchronize()
    assert abi.csa2_get_status() == 0
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    n0 = abi.csa2_launch_count()
    with ClockSampler(local) as clk:
        for k in range(args.steps):
            flush(k)
            ev[k][0].record(stream)
            step()
            ev[k][1].record(stream)
        torch.cuda.synchronize()
    launches = abi.csa2_launch_count() - n0
    step_ms = [a.elapsed_time(b) for a, b in ev]
    ms = max_over_ranks(sum(step_ms) / args.steps, dist, dev)
    # end to end, as a serving loop runs it: the chunk's hidden states in from pinned host
    # memory and the last layer's codes back, two buffer sets (hidden state and caches),
    # uploads and downloads on two copy streams overlapping each other and the steps
    sets = [(hidden, keep, step), ced_setup(dev)[1:]]
    h_in = hidden.cpu().pin_memory()
    h_out = [torch.empty(keep[-1]["codes"].shape, dtype=torch.uint8, pin_memory=True) for _ in range(2)]
    cs_up, cs_dn = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    def e2e_run(n_steps):
        up = [torch.cuda.Event() for _ in range(2)]
        done = [torch.cuda.Event() for _ in range(2)]
        down = [torch.cuda.Event() for _ in range(2)]
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(cs_up)
        cs_dn.wait_event(t0)
        for i in range(n_steps + 2):
            j = i % 2
            hid, kp, st = sets[j]
            if i >= 2:   # set j: step i-2 has finished; its last layer's codes go to the host
                with torch.cuda.stream(cs_dn):
                    cs_dn.wait_event(done[j])
                    h_out[j].copy_(kp[-1]["codes"], non_blocking=True)
                    down[j].record(cs_dn)
            if i < n_steps:
                with torch.cuda.stream(cs_up):
                    if i >= 2:
                        cs_up.wait_event(done[j])
                    hid.copy_(h_in, non_blocking=True)
                    up[j].record(cs_up)
                stream.wait_event(up[j])
                if i >= 2:
                    stream.wait_event(down[j])
                st()
                done[j].record(stream)
        t1.record(cs_dn)
        t1.synchronize()
        return t0.elapsed_time(t1)

    e2e_run(3)   # warm-up
    n = max(3, min(args.steps, 50))
    tot = e2e_run(n)
    e2e_ms = max_over_ranks(tot / n, dist, dev)
    status = abi.csa2_get_status()
    if rank != 0:
        return
    G = wl.n_new // 4
    flops = 2.0 * G * 4 * wl.H * CED_LAYERS * (wl.d + wl.Di)
    peaks = load_peaks()
    achieved = flops / (ms / 1e3) / 1e12
    line = {
        "metric": METRIC, "value": world * wl.n_new / (ms / 1e3), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"ced_compress_{CED_LAYERS}layers_chunk{wl.n_new}",
                   "description": f"{CED_LAYERS} layers' KV of a {wl.n_new}-token chunk (hidden {wl.H}) from one "
                                  "hidden state: one GEMM over the stacked weights, then every layer's RMSNorm/RoPE/MXFP4 "
                                  "in one launch",
                   "tokens_per_step": wl.n_new, "layers": CED_LAYERS, "d": wl.d, "Di": wl.Di,
                   "l2": "flushed before every timed step (512 MB written, then 512 MB read)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": {"bound": "tensor", "kernel": "k_compress_gemm_tma (+ k_norm_rope_pack_layers)",
                     "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": achieved / peaks["bf16_tflops"], "traffic": None, "algorithmic_flops_per_launch": flops,
                     "kernel_ms": ms, "peak_source": peaks["source"] + " (bf16 burst)"},
        "e2e": {"value": world * wl.n_new / (e2e_ms / 1e3), "unit": "tokens/s", "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": hidden.numel() * 2, "d2h_bytes_per_step": h_out[0].numel(),
                "pipeline": "two buffer sets (hidden state and caches); uploads and downloads on two copy "
                            "streams overlap each other and the steps; no L2 flush"},
        "gpu_launches": launches, "status_word": status,
        "step_ms_p50": statistics.median(step_ms), "step_ms_min": min(step_ms), "clocks": clk.summary(),
    }
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline_all("ced_compress", args.cpu_seconds)
    print(json.dumps(line), flush=True)


def ced_cpu_worker(seconds, ref_steps=0):
    """The oracle's compression of the chunk for one layer (whole layers until `seconds`
    are used, at least one), scaled to CED_LAYERS layers."""
    import torch
    torch.set_num_threads(1)
    from oracle import compress as Cm
    wl = make_workload("prefill")
    hid = wl.hidden()[0].double().numpy()
    W_all = wl.w_layers(1)
    gamma = wl.gamma().double().numpy()
    first = wl.entries_before(0)
    W, Wi = W_all[0, :wl.d].double().numpy(), W_all[0, wl.d:].double().numpy()
    times = []
    t_tot = 0.0
    while not times or t_tot < seconds:
        t0 = time.perf_counter()
        Cm.compress_pack(hid, W, gamma, wl.eps, wl.r, wl.rope_base, first, W_idx=Wi)
        times.append(time.perf_counter() - t0)
        t_tot += times[-1]
    per_layer = t_tot / len(times)
    value = wl.n_new / (per_layer * CED_LAYERS)
    out = {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
           "sample": f"{len(times)} layer(s) of the {wl.n_new}-token chunk's compression, {t_tot:.1f} s of "
                     f"single-thread float64 numpy, scaled to {CED_LAYERS} layers"}
    if ref_steps > 0:
        out["step_values"] = [wl.n_new / (t * CED_LAYERS) for t in times] * ref_steps
        out["step_values"] = out["step_values"][:ref_steps]
    print(json.dumps(out))


class L2Flush:
    """Evicts the step's inputs from L2: writes FLUSH_BYTES, then reads another
    FLUSH_BYTES, so that the L2 ends up holding clean lines of neither."""

    def __init__(self, dev):
        import torch
        self.device = dev
        self.w = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.r = torch.ones(FLUSH_BYTES // 8, dtype=torch.int64, device=dev)
        self.acc = torch.zeros((), dtype=torch.int64, device=dev)

    def __call__(self, k):
        self.w.fill_(k & 255)
        self.acc += self.r.sum()


def time_dominant_kernel(args, g, wl, flush, stream):
    """Average duration of the dominant kernel of the step, launched as in the step."""
    import torch

    from compressed_sparse_attention_05_gb300 import abi

    n = max(3, min(args.steps, 200))
    if wl.Tq == 1:     # decode-type workloads: the Full layer's indexer scan
        stride = g.max_entries
        scores = torch.empty(wl.B * wl.Tq, stride, dtype=torch.float32, device=flush.device)
        fn = lambda: abi.csa2_index_scores(g.dims(), g.cache(), g.idx_q[0], g.idx_w[0], g.q_pos, scores)  # noqa
        name = "k_index_scan_pages"
    else:              # prefill and replay: attention of the Full layer
        fn = lambda: abi.csa2_sparse_attn(g.dims(), g.cache(), g.window(0), g.Q[0], g.q_pos, g.idx[0],  # noqa
                                          g.cnt[0], 1.0 / math.sqrt(wl.d), g.O[0], g.lse[0])
        name = "k_sparse_attn_tc"
    fn()
    tot = 0.0
    for k in range(n):
        flush(k)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        b.synchronize()
        tot += a.elapsed_time(b)
    return {"name": name, "ms": tot / n, "launches_timed": n}


def time_replay(args, g, wl, flush, stream):
    """Average duration (ms) of one layer's window rebuild (csa2_swa_replay), launched as
    in the step, L2 flushed before each."""
    import torch

    n = max(3, min(args.steps, 200))
    g.replay_window(0)
    tot = 0.0
    for k in range(n):
        flush(k)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        g.replay_window(0)
        b.record(stream)
        b.synchronize()
        tot += a.elapsed_time(b)
    return tot / n


def time_e2e(args, g, flush, stream, dist):
    """The metric end to end through the public call (csa2_layer) with host buffers,
    as a serving loop runs it: two sets of device input/output buffers (a second
    layer group over an identical cache), an upload stream that copies step i+1's
    inputs from pinned host memory and a download stream that copies step i-1's
    outputs back while step i computes (the two directions run on separate copy
    engines at once).  Every step's inputs are copied in and its outputs copied out
    inside the timed region, which runs from the first upload to the last download.
    No L2 flush between steps: each step streams more than L2 (its keys and cache)."""
    import torch

    from compressed_sparse_attention_05_gb300 import harness

    g2 = harness.LayerGroup(g.wl, g.Q[0].device)
    groups = [g, g2]
    ins = [x.step_inputs() for x in groups]
    outs = [x.step_outputs() for x in groups]
    h_in = [t.detach().cpu().pin_memory() for t in ins[0]]
    h_out = [[torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs[0]] for _ in range(2)]
    bi = sum(t.numel() * t.element_size() for t in ins[0])
    bo = sum(t.numel() * t.element_size() for t in outs[0])
    cs_up = torch.cuda.Stream(device=g.Q[0].device)
    cs_dn = torch.cuda.Stream(device=g.Q[0].device)
    n = max(4, min(args.steps, 200))

    def run(n_steps):
        up = [torch.cuda.Event() for _ in range(2)]     # set j's inputs are on the device
        done = [torch.cuda.Event() for _ in range(2)]   # set j's step has finished
        down = [torch.cuda.Event() for _ in range(2)]   # set j's outputs are on the host
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(cs_up)
        cs_dn.wait_event(start)
        for i in range(n_steps + 2):
            j = i % 2
            if i >= 2:   # buffer set j: step i-2 has finished; its outputs go to the host
                with torch.cuda.stream(cs_dn):
                    cs_dn.wait_event(done[j])
                    for h, d_ in zip(h_out[j], outs[j]):
                        h.copy_(d_, non_blocking=True)
                    down[j].record(cs_dn)
            if i < n_steps:   # step i's inputs, once step i-2 no longer reads set j
                with torch.cuda.stream(cs_up):
                    if i >= 2:
                        cs_up.wait_event(done[j])
                    for d_, h in zip(ins[j], h_in):
                        d_.copy_(h, non_blocking=True)
                    up[j].record(cs_up)
                stream.wait_event(up[j])
                if i >= 2:
                    stream.wait_event(down[j])   # step i overwrites set j's outputs
                groups[j].step(stream=stream)
                done[j].record(stream)
        end.record(cs_dn)
        end.synchronize()
        return start.elapsed_time(end)

    run(4)   # warm-up
    if dist is not None:
        dist.barrier()
    ms = max_over_ranks(run(n) / n, dist, flush.device)
    world = dist.get_world_size() if dist is not None else 1
    wl = g.wl
    del g2
    return {"value": world * wl.B * wl.Tq / (ms / 1e3), "unit": "tokens/s", "ms_per_step": ms,
            "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
            "pipeline": "two buffer sets; uploads and downloads on two copy streams (separate copy engines) "
                        "overlap each other and the steps' compute; no L2 flush (each step streams more than L2)"}


def load_peaks():
    try:
        p = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained"), "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def roofline(wl, alg, kern, peaks):
    src = os.path.join(ROOT, "compressed_sparse_attention_05_gb300", "csrc")
    if kern["name"] == "k_index_scan_pages":
        bytes_ = alg["scan_bytes_per_launch"]
        achieved = bytes_ / (kern["ms"] / 1e3) / 1e9
        traffic = committed_traffic(os.path.join(ROOT, "profiles", f"index_scores_{wl.name}.md"),
                                    os.path.join(src, "indexer.cu"))
        return {"bound": "hbm", "kernel": kern["name"], "achieved": achieved, "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
                "algorithmic_bytes_per_launch": bytes_, "kernel_ms": kern["ms"],
                "peak_source": peaks["source"] + " (hbm copy)"}
    flops = alg["attn_flops_per_launch"]
    achieved = flops / (kern["ms"] / 1e3) / 1e12
    traffic = committed_traffic(os.path.join(ROOT, "profiles", f"sparse_attn_{wl.name}.md"),
                                os.path.join(src, "attention_tc.cu"))
    return {"bound": "tensor", "kernel": kern["name"], "achieved": achieved, "peak": peaks["bf16_tflops"],
            "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops"], "traffic": traffic,
            "algorithmic_flops_per_launch": flops, "kernel_ms": kern["ms"],
            "peak_source": peaks["source"] + " (bf16 burst)"}


def step_roofline(wl, alg, ms, peaks):
    t_bytes = alg["step_bytes"] / (peaks["hbm_gbs"] * 1e9)
    t_flops = (alg["attn_flops"] + alg["index_flops"] + alg["compress_flops"]) / (peaks["bf16_tflops"] * 1e12)
    bound = max(t_bytes, t_flops)
    return {"bound": "hbm" if t_bytes >= t_flops else "tensor", "algorithmic_bytes": alg["step_bytes"],
            "algorithmic_flops": alg["attn_flops"] + alg["index_flops"] + alg["compress_flops"],
            "ideal_ms": bound * 1e3, "frac": bound * 1e3 / ms}


# ---------------------------------------------------------------------------------
# the CPU oracle on a bounded sample

def _cpu_cmd(workload, seconds, ref_steps, part=0):
    return [sys.executable, os.path.join(ROOT, "bench.py"), "--cpu-worker", "--workload", workload,
            "--cpu-seconds", str(seconds), "--ref-steps", str(ref_steps), "--cpu-part", str(part)]


_CPU_ENV = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
                CUDA_VISIBLE_DEVICES="")


def cpu_baseline(workload, seconds, ref_steps=0):
    """The oracle in one single-threaded worker process."""
    r = subprocess.run(_cpu_cmd(workload, seconds, ref_steps), capture_output=True, text=True, env=_CPU_ENV,
                       timeout=max(600, 20 * seconds))
    if r.returncode != 0:
        return {"error": r.stderr[-500:]}
    return json.loads(r.stdout.strip().splitlines()[-1])


def cpu_baseline_all(workload, seconds):
    """The oracle on every host core: one single-threaded worker per core, each on its own
    query tokens, run at the same time; throughput = the workers' sum.  The single-thread
    run is reported beside it."""
    single = cpu_baseline(workload, seconds)
    n = os.cpu_count() or 1
    procs = [subprocess.Popen(_cpu_cmd(workload, seconds, 0, part=p), stdout=subprocess.PIPE,
                              stderr=subprocess.PIPE, text=True, env=_CPU_ENV) for p in range(n)]
    vals, err = [], None
    for p in procs:
        try:
            out, e = p.communicate(timeout=max(600, 30 * seconds))
        except subprocess.TimeoutExpired:
            p.kill()
            out, e = p.communicate()
        if p.returncode != 0:
            err = e[-300:]
            continue
        vals.append(json.loads(out.strip().splitlines()[-1]))
    if not vals:
        return {"error": err, "single_thread": single}
    return {"value": sum(v["value"] for v in vals), "unit": "tokens/s", "cores": len(vals), "kind": "oracle",
            "sample": f"{len(vals)} single-threaded float64 numpy workers at once (one per host core, "
                      f"os.cpu_count() = {n}), each: {vals[0]['sample']}; throughput summed",
            "single_thread": single}


def cpu_worker(workload, seconds, ref_steps=0, part=0):
    """Times the oracle's arithmetic for whole query tokens of the workload (inputs and
    cached state prepared outside the timer), single-threaded.

    ref_steps > 0 (the reference arm): `seconds` is shared out over ref_steps timed
    steps; each step runs whole layers of query tokens (in schedule order, at least
    one layer) until its slice is used, so the run stays bounded whatever the
    step count; the per-step and aggregate throughputs are reported."""
    import numpy as np
    import torch

    torch.set_num_threads(1)
    from oracle import attention as A
    from oracle import formats as F
    from oracle import indexer as I
    from oracle import layer as OL
    from oracle import replay as R

    wl = make_workload(workload)
    tau = 1.0 / math.sqrt(wl.d)
    replay = wl.replay_H is not None
    W_swa = [wl.w_swa(l).double().numpy() for l in range(len(wl.layers))] if replay else None
    # the sample: one sequence (the median-length one; worker `part` of an all-cores run
    # takes the part-th sequence around it), its query tokens prepared once
    lens = [wl.entries_before(b) for b in range(wl.B)]
    b = sorted(range(wl.B), key=lambda x: lens[x])[(wl.B // 2 + part) % wl.B]
    st = OL.SequenceState(wl, b)
    Kall = st.indexer_keys()
    prepared = []
    for i in ([0] if wl.Tq == 1 else [(j + 37 * part) % wl.Tq for j in (0, wl.Tq // 2, wl.Tq - 1)]):
        t = wl.t_first[b] + i
        nv = I.n_visible(Kall.shape[0], t)
        L = len(wl.layers)
        qs = [(wl.idx_q_row(l, b, i).double().numpy(), wl.idx_w_row(l, b, i).double().numpy()) for l in range(L)]
        Qs = [wl.q_row(l, b, i).double().numpy() for l in range(L)]
        win_pos = OL.window_of(wl, b, t)
        if replay:
            # the window's other rows were rebuilt by the tokens before this one; this
            # token rebuilds its own row inside the timed layer
            k = win_pos - wl.t_first[b]
            win_lat = [(st.replay_rows(l)["codes"][k], st.replay_rows(l)["scales"][k],
                        wl.replay_hidden_rows(l, b)[i:i + 1].double().numpy()) for l in range(L)]
        else:
            win_lat = [wl.swa_latent(l, b, torch.from_numpy(win_pos)).numpy() for l in range(L)]
        # cached state: packed rows of every entry the schedule can gather (each Full
        # layer's selection and, for the pooled indexer, every pooled position)
        cand = []
        for l in range(L):
            if wl.layers[l] != "F":
                continue
            sc = I.index_scores(qs[l][0], qs[l][1], Kall[:nv])
            cand.append(I.topk(sc, wl.K))
            if wl.hierarchical:
                cand.append(I.pool_positions(I.block_pool(sc, wl.pool_blocks, wl.pool_block), nv, wl.pool_block))
        cand = np.unique(np.concatenate(cand))
        c, s = st.packed_rows(cand)
        prepared.append((t, nv, qs, Qs, win_lat, cand, c, s))

    def one_layer(l, state, t, nv, qs, Qs, win_lat, cand, c, s):
        """Layer l of one query token; state carries the previous layer's indices and the pool."""
        mode = wl.layers[l]
        if mode == "F":
            sc = I.index_scores(qs[l][0], qs[l][1], Kall[:nv])
            idx = I.topk(sc, wl.K)
            if wl.hierarchical:
                state["pool"] = I.block_pool(sc, wl.pool_blocks, wl.pool_block)
        elif mode == "X":
            pos = I.pool_positions(state["pool"], nv, wl.pool_block)
            idx = pos[I.topk(I.index_scores(qs[l][0], qs[l][1], Kall[pos]), wl.K)]
        else:
            idx = state["prev"]
        state["prev"] = idx
        rows = np.searchsorted(cand, idx)
        assert np.array_equal(cand[rows], idx), "a gathered entry was not prepared"
        kv = F.fp8_unpack_bf16(c[rows], s[rows]) if st.kv_format == "fp8" else F.mxfp4_unpack(c[rows], s[rows])
        if replay:
            wc, ws, own_h = win_lat[l]
            own = R.window_rows(own_h, W_swa[l], st.gamma, wl.eps, wl.r, wl.rope_base, t)
            wc, ws = wc.copy(), ws.copy()
            wc[-1], ws[-1] = own["codes"][0], own["scales"][0]
        else:
            wc, ws = F.fp8_pack(win_lat[l])
        A.sparse_attention(Qs[l], kv, F.fp8_unpack_bf16(wc, ws), tau)

    L = len(wl.layers)
    unit = [0]   # (token, layer) units run so far, in schedule order
    state = {}

    def run_units(slice_s):
        """Whole layers, in order, until slice_s seconds are used (at least one)."""
        t, n = 0.0, 0
        while n == 0 or t < slice_s:
            k = unit[0]
            l = k % L
            if l == 0:
                state.clear()
            p = prepared[(k // L) % len(prepared)]
            t0 = time.perf_counter()
            one_layer(l, state, *p)
            t += time.perf_counter() - t0
            n += 1
            unit[0] += 1
        return t, n

    step_tokens = []   # (seconds, tokens) of every reference step
    if ref_steps > 0:
        slice_s = seconds / ref_steps
        for _ in range(ref_steps):
            t, n = run_units(slice_s)
            step_tokens.append((t, n / L))
        t_tot = sum(t for t, _ in step_tokens)
        tokens = sum(n for _, n in step_tokens)
    else:
        t_tot, tokens = 0.0, 0
        while t_tot < seconds:
            t, n = run_units(seconds - t_tot)
            t_tot += t
            tokens += n / L
    per_token = t_tot / max(tokens, 1e-9)
    # prefill: the step also compresses the chunk; time the oracle's compression once
    extra = ""
    t_comp = 0.0
    if wl.H is not None:
        from oracle import compress as Cm
        st = OL.SequenceState(wl, 0)
        hid = st.wl.hidden()[0].double().numpy()
        W = st.wl.w_compress().double().numpy()
        Wi = st.wl.w_index().double().numpy()
        t0 = time.perf_counter()
        Cm.compress_pack(hid, W, st.gamma, wl.eps, wl.r, wl.rope_base, st.n_before, W_idx=Wi)
        t_comp = time.perf_counter() - t0
        extra = f"; compression of the {wl.n_new}-token chunk timed once ({t_comp:.2f} s)"

    def step_value(sec_per_token):
        step_s = t_comp + sec_per_token * wl.Tq * wl.B
        return wl.B * wl.Tq / step_s

    value = step_value(per_token)
    out = {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
           "sample": f"{tokens:.2f} query tokens of {wl.name} through all {L} layer(s) (whole layers, in "
                     f"schedule order), {t_tot:.1f} s of single-thread float64 numpy, scaled to the "
                     f"{wl.B * wl.Tq}-token step{extra}",
           "seconds_per_token": per_token}
    if ref_steps > 0:
        out["step_values"] = [step_value(t / n) for t, n in step_tokens]
    print(json.dumps(out))


# ---------------------------------------------------------------------------------
# reference arm: the oracle as it stands, timed on the host cores

def run_reference(args, rank, world):
    """The oracle as the reference arm: one worker process times warmup + steps
    steps, each a slice of a fixed CPU budget (--ref-seconds in all), so the run
    is bounded whatever the step count; value = the timed steps' aggregate
    throughput (tokens over seconds)."""
    if rank != 0:
        return
    n = args.warmup + args.steps
    r = cpu_baseline(args.workload, args.ref_seconds, ref_steps=n)
    if "error" in r:
        print(json.dumps({"impl": "reference", "unavailable": "oracle run failed: " + r["error"][-200:]}))
        return
    timed = r["step_values"][args.warmup:]
    # aggregate over the timed steps: total tokens / total seconds (harmonic mean of the step rates)
    value = len(timed) / sum(1.0 / v for v in timed) if timed else r["value"]
    last = r
    wl = make_workload("prefill" if args.workload == "ced_compress" else args.workload)
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": wl.B * wl.Tq / value * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": ({"workload": f"ced_compress_{CED_LAYERS}layers_chunk{wl.n_new}",
                    "description": f"{CED_LAYERS} layers' KV of a {wl.n_new}-token chunk from one hidden state"}
                   if args.workload == "ced_compress"
                   else dict(workload_config(wl), l2="not applicable (host cores)",
                             parallelism="one single-threaded host process")),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": last["cores"], "kind": "oracle",
                         "sample": last["sample"]},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="decode",
                    choices=["decode", "decode_fp8kv", "prefill", "hierarchical", "ragged", "encoder_stack",
                             "decoder_stack",
                             "decoder_stack_prefill", "decoder_replay", "ced_compress"])
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-seconds", type=float, default=120.0,
                    help="CPU budget of the whole reference run, shared out over warmup + steps")
    ap.add_argument("--ref-steps", type=int, default=0, help=argparse.SUPPRESS)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true",
                    help="default decode run: skip the prefill@64K object")
    ap.add_argument("--cpu-part", type=int, default=0, help=argparse.SUPPRESS)
    ap.add_argument("--cpu-worker", action="store_true")
    args = ap.parse_args()
    if args.cpu_worker:
        if args.workload == "ced_compress":
            ced_cpu_worker(args.cpu_seconds, args.ref_steps)
        else:
            cpu_worker(args.workload, args.cpu_seconds, args.ref_steps, args.cpu_part)
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist_mod
        if args.impl == "reference":
            run_reference(args, rank, world)
            return
        import torch
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist_mod.init_process_group("nccl")
        dist = dist_mod
    if args.impl == "reference":
        run_reference(args, rank, world)
    elif args.workload == "ced_compress":
        run_ced(args, rank, world, dist)
    else:
        run_gpu(args, rank, world, dist)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
