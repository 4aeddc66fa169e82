"""MLA decode benchmark: one JSON line per run.

A step is one pass of the whole decode hot path over the DeepSeek-V2-shaped
workload (batch 64, 128 heads, d_h 128, d_c 512, d_h^R 64, 4096 cached tokens
per sequence, bf16 cache, one query token): mla_append_absorb (the cache append
of this step's 64 tokens and the query absorption, overlapped) -> mla_decode
(+ combine) -> mla_unabsorb.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

`value` is latent-KV throughput: bytes of latent cache the step's attention
reads (sum_b L_b * 1152 B) per second of step time, inputs resident in HBM.
L2 is flushed (a 2x-L2 buffer write) before every timed step, outside the
step's events. `e2e` is the same metric through the public API with pinned
HOST inputs copied in and the output copied back inside the timed region.
`other_workloads` adds mla_decode timings of the ragged (128 x U[1024, 32768]),
long-context (8 x 131072) and FP8 two-token (128 x 8192) workloads, the last with
the default (fused dequantising) kernel, with FP8 scores and with the cache staged
to bf16 first; `next_rows` the fused upstream append, W^O and a prompt prefill.
`--impl reference` times the fp64 CPU oracle on a bounded sample of the same
workload. With N > 1 each rank runs an independent replica (the path has no
exchange step), so `scaling` is weak.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MLA decode: latent-KV GB/s & TFLOPS vs B300 roofline; µs per decode step"
WORKLOAD_ID = 2


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0,
            "source": "fallback"}


def _workload_sizes(wl):
    bytes_per_tok = {"bf16": (wl.C + wl.R) * 2, "f32": (wl.C + wl.R) * 4,
                     "fp8": wl.C + 2 * wl.R + 4 * (wl.C // 128)}[wl.cache]
    act = 2 if wl.act == "bf16" else 4
    cache_bytes = sum(wl.seq_lens) * bytes_per_tok
    qo_bytes = wl.B * wl.n_q * wl.H * ((wl.C + wl.R) + wl.C) * act + wl.B * wl.n_q * wl.H * 4
    # QK^T over C+R plus P.V over C, per head, per query row, per visible token
    flops = sum(2 * wl.H * (2 * wl.C + wl.R) * (L - wl.n_q + 1 + j)
                for L in wl.seq_lens for j in range(wl.n_q))
    return cache_bytes, qo_bytes, flops


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"mla_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def _cpu_oracle_sample(wl, budget_s: float = 12.0, max_heads: int = 1 << 30):
    """Time the fp64 oracle (as it stands) on whole heads of sequence 0, then 1, ...
    until about budget_s of CPU work. Returns (GB/s equivalent, sample description, threads)."""
    from oracle import mla_oracle as O

    w_uk, w_uv = wl.weights()
    q_c, q_r = wl.queries()
    bytes_per_tok = (wl.C + wl.R) * 2 if wl.cache == "bf16" else wl.C + 2 * wl.R + 4 * (wl.C // 128)
    done_bytes, heads_done, seqs = 0.0, 0, 0
    t_total = 0.0
    for b in range(wl.B):
        c, r = wl.latents(b)
        L = wl.seq_lens[b]
        ce = O.cache_entries(c, r, np.arange(L), wl.cache, wl.rope_base)
        seqs += 1
        for h0 in range(0, wl.H, 8):
            heads = np.arange(h0, min(wl.H, h0 + 8))
            t0 = time.perf_counter()
            O.mla_decode_naive(ce["c"], ce["k_r"], q_c[b], q_r[b], w_uk, w_uv, wl.positions(b),
                               wl.rope_base, heads=heads)
            t_total += time.perf_counter() - t0
            heads_done += len(heads)
            # the share of this sequence's latent-cache work these heads stand for
            done_bytes += L * bytes_per_tok * len(heads) / wl.H
            if t_total >= budget_s or heads_done >= max_heads:
                break
        if t_total >= budget_s or heads_done >= max_heads:
            break
    threads = _blas_threads()
    sample = (f"fp64 oracle (explicit k^C/v^C decompression per head) on the first {seqs} "
              f"sequence(s) of L={wl.seq_lens[0]} ({heads_done} (sequence, head) pairs of "
              f"{wl.B * wl.H}); bytes credited = L * {bytes_per_tok} B * heads/{wl.H} per sequence")
    return done_bytes / t_total / 1e9, sample, threads, t_total


PROFILE = os.path.join(ROOT, "profiles", "decode_tc_v2_b64_l4096.json")
DECODE_SOURCE = os.path.join(ROOT, "mla_latent_kv_78_b300", "csrc", "decode_tc.cu")


def _ncu_traffic():
    """DRAM bytes (read + write) per decode launch from the committed ncu record (a JSON file
    beside the summary), or None when it is missing or was taken on a different decode_tc.cu
    (its recorded sha256)."""
    import hashlib

    try:
        rec = json.load(open(PROFILE))
        sha = hashlib.sha256(open(DECODE_SOURCE, "rb").read()).hexdigest()
    except (OSError, ValueError):
        return None
    if rec.get("source_sha256") != sha:
        return None
    v = rec.get("dram_bytes_per_launch")
    return int(v) if isinstance(v, (int, float)) else None


def reduce_max_over_ranks(xs, device):
    """Element-wise max of xs over all ranks (the slowest rank's times); identity when the
    process group is absent or has one rank."""
    import torch
    import torch.distributed as dist

    t = torch.tensor(list(xs), dtype=torch.float64, device=device)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t]


def whole_job_gbs(world: int, bytes_per_step: float, steps: int, total_ms: float) -> float:
    """Latent-cache GB/s of the whole job: every rank's replica moved bytes_per_step per step,
    and the job took the slowest rank's total_ms."""
    return world * bytes_per_step * steps / (total_ms * 1e-3) / 1e9


def _workload_config(wl, extra=None):
    """The `config` object of the JSON line: the workload by name and its sizes."""
    c = {"workload": wl.name, "batch": wl.B, "seq_len": wl.seq_lens[0], "n_heads": wl.H,
         "d_head": wl.D, "d_latent": wl.C, "d_rope": wl.R, "n_q": wl.n_q, "page_size": wl.P,
         "cache": wl.cache, "l2": "flushed before every timed step"}
    c.update(extra or {})
    return c


def _combine_launches(M, cfg, wl, splits) -> int:
    """1 if mla_decode runs a split-KV combine kernel for this workload, else 0."""
    if M.mla_decode_kernel(cfg, wl.B, wl.n_q) == M.MLA_KERNEL_TC:
        # the tensor-core kernel's workspace holds partials only when it splits
        base = M.mla_decode_workspace_size(cfg, wl.B, wl.n_q, wl.max_seq_len, 1)
        return int(M.mla_decode_workspace_size(cfg, wl.B, wl.n_q, wl.max_seq_len, splits) > base)
    return int(M.mla_decode_workspace_size(cfg, wl.B, wl.n_q, wl.max_seq_len, splits) > 0)


def _blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


def run_reference(args, world, rank):
    import workloads as W

    if rank != 0:
        return 0
    wl = W.config(WORKLOAD_ID)
    rates, secs = [], []
    sample = ""
    threads = 1
    for i in range(args.warmup + args.steps):
        v, sample, threads, t = _cpu_oracle_sample(wl, budget_s=args.ref_seconds_per_step)
        if i >= args.warmup:
            rates.append(v)
            secs.append(t)
    value = statistics.median(rates)
    cache_bytes, _, flops = _workload_sizes(wl)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        # a whole step of the oracle would take this long at the sampled rate (an
        # extrapolation); each timed step ran for sample_seconds_per_step
        "ms_per_step": cache_bytes / (value * 1e9) * 1e3,
        "ms_per_step_is": "extrapolated from the sampled rate",
        "sample_seconds_per_step": statistics.median(secs),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": _workload_config(wl, {"parallelism": "single", "decode_kernel": "fp64 oracle (CPU)",
                                        "num_splits": 0}),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def _other_workloads(M, W, torch, dev, flush, peaks, steps: int = 5):
    """mla_decode alone on the ragged, long-context and FP8 two-token workloads (the last
    also with its scores on FP8 tensor cores, MLA_KERNEL_TC_FP8_SCORES, and with the cache
    staged to bf16 first, MLA_KERNEL_TC_FP8_STAGED), device resident, over
    a pool filled with seeded random latents (their values do not change the work; parity on
    these workloads is checked by the full-size tests). L2 flushed before each timed call."""
    out = {}
    g = torch.Generator(device=dev)
    suffix = {M.MLA_KERNEL_AUTO: "", M.MLA_KERNEL_TC_FP8_SCORES: "-fp8-scores",
              M.MLA_KERNEL_TC_FP8_STAGED: "-fp8-staged"}
    for n, kern in ((3, M.MLA_KERNEL_AUTO), (4, M.MLA_KERNEL_AUTO), (5, M.MLA_KERNEL_AUTO),
                    (5, M.MLA_KERNEL_TC_FP8_SCORES), (5, M.MLA_KERNEL_TC_FP8_STAGED)):
        wl = W.config(n)
        g.manual_seed(7800 + n)
        cfg = M.make_config(wl.H, wl.D, wl.C, wl.R, wl.P, cache=wl.cache, act=wl.act, kernel=kern)
        eb = M.mla_cache_entry_bytes(cfg)
        if wl.cache == "fp8":
            pool = torch.randint(0, 0x76, (wl.num_pages, wl.P, eb), dtype=torch.uint8, device=dev,
                                 generator=g)
            scales = torch.full((wl.num_pages, wl.P, wl.C // 128), 2.0 ** -6, device=dev)
            pool[:, :, wl.C + 2 * wl.R:] = scales.view(torch.uint8).reshape(wl.num_pages, wl.P, -1)
            krope = torch.randn(wl.num_pages, wl.P, wl.R, device=dev, generator=g).to(torch.bfloat16)
            pool[:, :, wl.C:wl.C + 2 * wl.R] = krope.view(torch.uint8).reshape(wl.num_pages, wl.P, -1)
        else:
            pool = torch.randn(wl.num_pages, wl.P, wl.C + wl.R, device=dev, generator=g).to(
                torch.bfloat16).view(torch.uint8).reshape(wl.num_pages, wl.P, eb)
        bt = torch.from_numpy(wl.block_table()).to(dev)
        sl = torch.tensor(wl.seq_lens, dtype=torch.int32, device=dev)
        T = wl.B * wl.n_q
        q = (torch.randn(T, wl.H, wl.C + wl.R, device=dev, generator=g) * 0.15).to(torch.bfloat16)
        o = torch.empty(T, wl.H, wl.C, dtype=torch.bfloat16, device=dev)
        lse = torch.empty(T, wl.H, dtype=torch.float32, device=dev)
        st = torch.zeros(1, dtype=torch.int32, device=dev)
        wsz = M.mla_decode_workspace_size(cfg, wl.B, wl.n_q, wl.max_seq_len, 0)
        ws = torch.empty(max(wsz, 16), dtype=torch.uint8, device=dev)

        def call():
            M.mla_decode(cfg, q, pool, bt, sl, wl.n_q, wl.max_seq_len, o, lse, ws, 0,
                         wl.num_pages, st)

        for _ in range(3):
            call()
        ts = []
        for k in range(steps):
            flush.fill_(float(k))
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            call()
            b.record()
            b.synchronize()
            ts.append(a.elapsed_time(b))
        ms = statistics.median(ts)
        cache_bytes, qo_bytes, flops = _workload_sizes(wl)
        gbs = (cache_bytes + qo_bytes) / (ms * 1e-3) / 1e9
        tfl = flops / (ms * 1e-3) / 1e12
        out[wl.name + suffix[kern]] = {
            "decode_us": ms * 1e3, "gbs": gbs, "tflops": tfl,
            "hbm_frac": gbs / peaks["hbm_gbs"], "tensor_frac": tfl / peaks["bf16_tflops"],
            "kernel": {1: "simt", 2: "tcgen05", 3: "tcgen05 (FP8 scores)",
                       4: "FP8 staged to bf16 + tcgen05"}.get(M.mla_decode_kernel(cfg, wl.B, wl.n_q)),
            "status": int(st.item()),
        }
        del pool, q, o, lse, ws
        torch.cuda.empty_cache()
    return out


def _time_ms(torch, fn, flush, steps=7):
    """Median CUDA-event time of fn() captured once as a CUDA graph and replayed `steps` times,
    L2 flushed before each replay (so host-side launch work is not timed)."""
    fn()   # first call outside the capture: one-time per-process set-up
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    ev = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(2)]
    with torch.cuda.graph(graph):
        ev[0].record()
        fn()
        ev[1].record()
    ts = []
    for k in range(steps + 2):
        flush.fill_(float(k))
        graph.replay()
        torch.cuda.synchronize()
        if k >= 2:
            ts.append(ev[0].elapsed_time(ev[1]))
    return statistics.median(ts)


def _next_rows(M, W, torch, dev, flush, peaks):
    """The steps either side of the decode, at DeepSeek-V2 sizes (d = 5120), each against its
    roofline: the fused upstream append for one decode step's 64 tokens, the W^O output
    projection for those tokens, and the non-absorbed prefill of a 4096-token prompt."""
    bf = torch.bfloat16
    g = torch.Generator(device=dev)
    g.manual_seed(7890)
    H, D, C, R, P, d_model = 128, 128, 512, 64, 64, 5120
    out = {}
    # fused upstream append: h [64][5120] -> cache entries of 64 sequences
    T = 64
    cfg = M.make_config(H, D, C, R, P)
    h = torch.randn(T, d_model, device=dev, generator=g).to(bf)
    w = (torch.randn(C + R, d_model, device=dev, generator=g) * 0.02).to(bf)
    gain = torch.rand(C, device=dev, generator=g) + 0.5
    bt = torch.arange(T, dtype=torch.int32, device=dev).reshape(T, 1)
    pool = torch.zeros(T, P, M.mla_cache_entry_bytes(cfg), dtype=torch.uint8, device=dev)
    seq = torch.arange(T, dtype=torch.int32, device=dev)
    pos = torch.full((T,), 17, dtype=torch.int32, device=dev)
    ws = torch.empty(M.mla_project_append_workspace_size(cfg, d_model, T), dtype=torch.uint8, device=dev)
    ms = _time_ms(torch, lambda: M.mla_project_append(cfg, h, w, gain, 1e-6, seq, pos, bt, pool, ws), flush)
    byt = (C + R) * d_model * 2 + T * d_model * 2 + T * (C + R) * 2
    out["project_append_t64"] = {"us": ms * 1e3, "gbs": byt / (ms * 1e-3) / 1e9,
                                 "hbm_frac": byt / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                                 "algorithmic_bytes": byt, "bound": "hbm (weights)"}
    # W^O: u [64][5120] = o [64][16384] . W^O^T
    o = (torch.randn(T, H * D, device=dev, generator=g) * 0.05).to(bf)
    w_o = (torch.randn(d_model, H * D, device=dev, generator=g) * 0.006).to(bf)
    u = torch.empty(T, d_model, device=dev)
    ws2 = torch.empty(max(M.mla_output_projection_workspace_size(cfg, d_model, T), 16), dtype=torch.uint8, device=dev)
    ms = _time_ms(torch, lambda: M.mla_output_projection(cfg, o, w_o, u, ws2), flush)
    byt = d_model * H * D * 2 + T * H * D * 2 + T * d_model * 4
    out["output_projection_t64"] = {"us": ms * 1e3, "gbs": byt / (ms * 1e-3) / 1e9,
                                    "hbm_frac": byt / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                                    "algorithmic_bytes": byt, "bound": "hbm (weights)"}
    del o, w_o, u, ws2
    # prefill of one 4096-token prompt: decompression GEMMs + causal attention
    L = 4096
    c = torch.randn(L, C, device=dev, generator=g).to(bf)
    k_r = torch.randn(L, R, device=dev, generator=g).to(bf)
    q_c = torch.randn(L, H, D, device=dev, generator=g).to(bf)
    q_r = torch.randn(L, H, R, device=dev, generator=g).to(bf)
    w_uk = (torch.randn(H, D, C, device=dev, generator=g) * 0.02).to(bf)
    w_uv = (torch.randn(H, D, C, device=dev, generator=g) * 0.02).to(bf)
    op = torch.empty(L, H, D, device=dev)
    ws3 = torch.empty(M.mla_prefill_workspace_size(cfg, L), dtype=torch.uint8, device=dev)
    ms = _time_ms(torch, lambda: M.mla_prefill(cfg, c, k_r, q_c, q_r, w_uk, w_uv, op, ws3), flush, steps=5)
    flops = 2 * 2 * L * C * H * D + H * (L * (L + 1) // 2) * 2 * (D + R + D)
    out["prefill_l4096"] = {"us": ms * 1e3, "tflops": flops / (ms * 1e-3) / 1e12,
                            "tensor_frac": flops / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"],
                            "flops": flops, "bound": "tensor"}
    del c, k_r, q_c, q_r, w_uk, w_uv, op, ws3
    torch.cuda.empty_cache()
    return out


def run_ours(args, world, rank, local_rank):
    import torch

    import mla_latent_kv_78_b300 as M
    import workloads as W

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    wl = W.config(WORKLOAD_ID)
    cfg = M.make_config(wl.H, wl.D, wl.C, wl.R, wl.P, cache=wl.cache, act=wl.act,
                        kernel=args.kernel)
    act = torch.bfloat16 if wl.act == "bf16" else torch.float32
    lat = torch.bfloat16 if wl.latent_storage == "bf16" else torch.float32
    w_uk, w_uv = wl.weights()
    step = M.DecodeStep(cfg, torch.from_numpy(wl.block_table()), wl.seq_lens, wl.n_q, wl.num_pages,
                        torch.from_numpy(w_uk).to(dev).to(act), torch.from_numpy(w_uv).to(dev).to(act),
                        num_splits=args.splits, device=str(dev))
    # cache fill: every token before this step's, via the library's append
    new_c, new_r = [], []
    for b in range(wl.B):
        c, r = wl.latents(b)
        keep = wl.seq_lens[b] - wl.n_q
        step.prefill(torch.from_numpy(c[:keep]).to(dev).to(lat), torch.from_numpy(r[:keep]).to(dev).to(lat),
                     torch.full((keep,), b, dtype=torch.int32, device=dev),
                     torch.arange(keep, dtype=torch.int32, device=dev))
        new_c.append(c[keep:])
        new_r.append(r[keep:])
    q_c, q_r = wl.queries()
    T = wl.B * wl.n_q
    inputs_host = {
        "c": torch.from_numpy(np.concatenate(new_c)).to(lat).pin_memory(),
        "r": torch.from_numpy(np.concatenate(new_r)).to(lat).pin_memory(),
        "qc": torch.from_numpy(q_c.reshape(T, wl.H, wl.D)).to(act).pin_memory(),
        "qr": torch.from_numpy(q_r.reshape(T, wl.H, wl.R)).to(act).pin_memory(),
    }
    inputs_dev = {k: v.to(dev) for k, v in inputs_host.items()}
    out_host = torch.empty(step.o.shape, dtype=torch.float32).pin_memory()
    torch.cuda.synchronize()
    assert step.status() == 0, "device status flagged during cache fill"

    stream = torch.cuda.current_stream()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(2 * l2 // 4 + 1024, dtype=torch.float32, device=dev)
    launches_per_step = 4 + _combine_launches(M, cfg, wl, args.splits)

    # The decode alone is timed in a copy of the step's graph with events around mla_decode;
    # the step (value) and e2e use the graph without them, whose decode and unabsorb launches
    # keep their programmatic edges. Clocks are sampled over both timed loops.
    clocks = ClockSampler(local_rank)
    step.capture(inputs_dev["c"], inputs_dev["r"], inputs_dev["qc"], inputs_dev["qr"],
                 time_decode=True)
    for _ in range(args.warmup):
        step.replay()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.25)
    dec_ms = []
    for k in range(args.steps):
        flush.fill_(float(k))
        step.replay()
        torch.cuda.synchronize()
        dec_ms.append(step.decode_ms())
    step.capture(inputs_dev["c"], inputs_dev["r"], inputs_dev["qc"], inputs_dev["qr"], timing=True)
    for _ in range(args.warmup):
        step.replay()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.perf_counter()
    step_ms = []
    for k in range(args.steps):
        # L2 flush between timed steps (a 2 x L2 write), outside the step's events
        flush.fill_(float(k))
        step.replay()
        torch.cuda.synchronize()
        step_ms.append(step.step_ms())
    wall = time.perf_counter() - t_wall0
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clk = clocks.stop()
    assert step.status() == 0, f"device status {step.status()} after timed steps"

    # end to end through the public API: pinned host inputs copied in, the step's graph,
    # o copied back, all inside the timed region
    e2e_ms = []
    h2d = sum(t.numel() * t.element_size() for t in inputs_host.values())
    d2h = out_host.numel() * out_host.element_size()
    for k in range(args.steps + args.warmup):
        flush.fill_(float(k))
        a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for key, t in inputs_host.items():
            inputs_dev[key].copy_(t, non_blocking=True)
        step.replay()
        out_host.copy_(step.o, non_blocking=True)
        b_.record(stream)
        b_.synchronize()
        if k >= args.warmup:
            e2e_ms.append(a.elapsed_time(b_))

    cache_bytes, qo_bytes, flops = _workload_sizes(wl)
    total_ms, total_e2e = reduce_max_over_ranks([sum(step_ms), sum(e2e_ms)], dev)
    ms_per_step = total_ms / args.steps
    value = whole_job_gbs(world, cache_bytes, args.steps, total_ms)
    e2e_value = whole_job_gbs(world, cache_bytes, args.steps, total_e2e)
    peaks = _peaks()
    dec_avg_ms = sum(dec_ms) / len(dec_ms)
    dec_bytes = cache_bytes + qo_bytes
    achieved = dec_bytes / (dec_avg_ms * 1e-3) / 1e9
    kernel_used = M.mla_decode_kernel(cfg, wl.B, wl.n_q)
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": _workload_config(wl, {
            "parallelism": f"replicas{world}" if world > 1 else "single",
            "decode_kernel": {1: "simt", 2: "tcgen05"}.get(kernel_used, str(kernel_used)),
            "num_splits": args.splits}),
        "us_per_step": ms_per_step * 1e3,
        "step_tflops": flops / (ms_per_step * 1e-3) / 1e12,
        "decode": {"us": dec_avg_ms * 1e3, "gbs": achieved,
                   "tflops": flops / (dec_avg_ms * 1e-3) / 1e12,
                   "algorithmic_bytes": dec_bytes, "flops": flops},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"], "traffic": _ncu_traffic(),
                     "kernel": "mla_decode", "peak_source": peaks["source"],
                     "tensor_frac": flops / (dec_avg_ms * 1e-3) / 1e12 / peaks["bf16_tflops"]},
        "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": total_e2e / args.steps},
        "gpu_launches": launches_per_step * args.steps,
        "launch": "one CUDA graph per step (append, absorb_q, decode, unabsorb)",
        "clocks": clk,
        "wall_s_timed": wall,
    }
    if not args.no_extra:
        line["other_workloads"] = _other_workloads(M, W, torch, dev, flush, peaks)
        line["next_rows"] = _next_rows(M, W, torch, dev, flush, peaks)
    if rank == 0 and not args.no_cpu_baseline:
        v, sample, threads, t = _cpu_oracle_sample(wl, budget_s=args.cpu_seconds)
        line["cpu_baseline"] = {"value": v, "unit": "GB/s", "cores": threads, "kind": "oracle",
                                "sample": sample, "seconds": t}
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--kernel", type=int, default=0, help="0 auto, 1 SIMT, 2 tensor-core decode")
    ap.add_argument("--splits", type=int, default=0)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-seconds-per-step", type=float, default=4.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the decode timings of the ragged, 128K and FP8 workloads")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, world, rank)
    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    try:
        return run_ours(args, world, rank, local_rank)
    finally:
        if world > 1:
            import torch
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
