"""Throughput of the indexer -> top-k -> sparse MLA layer step on GB300.

One step = one pass of the whole hot path over one batch of synthetic input:
the fused indexer + exact top-k kernel, then the sparse-MLA kernel, for the
16,384-token prefill workload (64 heads, 32x128 FP8 indexer, top-2048, BF16
latent cache). Metric: query tokens per second per layer.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl smla|reference]

N > 1 is launched with torchrun: every rank runs its own replica of the
workload on its GPU (query tokens are independent given the cache), so the
aggregate is weak scaling with no data-path collective.
--impl reference times the CPU oracle on the host cores on a bounded sample of
the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import indexer_top_sparse_score_gb300 as smla  # noqa: E402
from indexer_top_sparse_score_gb300 import counting  # noqa: E402
from indexer_top_sparse_score_gb300 import workloads as wl  # noqa: E402

METRIC = "query tokens/s per layer (indexer+top-k+sparse MLA)"
UNIT = "tokens/s"
WORKLOAD = "prefill16k"
L2_FLUSH_BYTES = 256 << 20
E2E_CHUNK = 2048  # query tokens per host-buffer chunk in the middle of the e2e schedule


def e2e_chunks(T: int):
    """Chunk sizes of the e2e measurement: E2E_CHUNK tokens, tapered at both
    ends (256, 768, 1024, then 2048s, then 1024, 768, 256) when T allows, so the
    copy-in before the first kernel and the copy-out after the last are short
    (16K tokens: 9.77 ms per step against 9.97 with even 2048-token chunks, on
    one GB300)."""
    ends = [256, 768, 1024]
    mid = T - 2 * sum(ends)
    if mid <= 0 or mid % E2E_CHUNK:
        return E2E_CHUNK
    return ends + [E2E_CHUNK] * (mid // E2E_CHUNK) + ends[::-1]


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return dict(hbm=d["hbm_gbs"], bf16=d["bf16_tflops"], bf16_sust=d["bf16_tflops_sustained"],
                    src="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sust=1700.0, src="fallback")


def kernel_sources_digest():
    """SHA-256 (first 16 hex digits) of the kernel sources and the C header,
    each file hashed as its repository path then its bytes, in path order."""
    csrc = os.path.join("indexer_top_sparse_score_gb300", "csrc")
    rel = sorted([os.path.join(csrc, f) for f in os.listdir(os.path.join(ROOT, csrc))
                  if os.path.isfile(os.path.join(ROOT, csrc, f))] + [os.path.join("include", "smla.h")])
    h = hashlib.sha256()
    for r in rel:
        h.update(r.replace(os.sep, "/").encode())
        with open(os.path.join(ROOT, r), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_traffic(kernel, summary="dram_traffic_prefill16k.md"):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, or None
    when there is none or the kernel sources changed since it was captured."""
    path = os.path.join(ROOT, "profiles", summary)
    if not os.path.exists(path):
        return None
    digest = kernel_sources_digest()
    for line in open(path):
        f = line.split()
        if len(f) == 5 and f[0] == "traffic" and f[1] == kernel and f[3] == "sources":
            return int(f[2]) if f[4] == digest else None
    return None


def dist_setup(n_gpus):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
        return dist.get_rank(), ws, int(os.environ.get("LOCAL_RANK", "0"))
    return 0, 1, 0


def reduce_max(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() and dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, max_mhz_default=2070.0):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx) if mx else max_mhz_default,
                "reasons": sorted(reasons), "samples": len(sm)}


def host_sample_rows(T: int, n: int, seed: int = 2024):
    rng = np.random.default_rng(seed)
    return np.sort(rng.choice(T, size=n, replace=False))


def cpu_oracle_sample(spec, dev, n_rows):
    """Time the CPU oracle (all host cores) on n_rows random rows of the workload."""
    import oracle
    rows = host_sample_rows(spec.n_tokens, n_rows)
    cache_h = dev.cache.to("cpu")
    oracle.build()
    t0 = time.perf_counter()
    _, _, _, _, used, _ = oracle.prefill_rows(dev, rows, cache_host=cache_h)
    dt = time.perf_counter() - t0
    return dict(value=n_rows / dt, unit=UNIT, cores=int(used), kind="oracle",
                sample=f"{n_rows} random query rows of {spec.name} (full indexer over their causal keys, "
                       f"full-sort top-{spec.topk}, fp64 attention), {dt:.1f} s wall")


def run_reference(args, rank, world):
    """--impl reference: the CPU oracle, timed on the host cores, on rank 0 only."""
    if rank != 0:
        return
    spec = wl.SPECS[WORKLOAD]
    dev_name = "cuda" if torch.cuda.is_available() else "cpu"
    dev = wl.make(spec, dev_name)
    rows_per_step = 256
    for _ in range(args.warmup):
        cpu_oracle_sample(spec, dev, 4)
    vals = []
    t0 = time.perf_counter()
    for _ in range(args.steps):
        r = cpu_oracle_sample(spec, dev, rows_per_step)
        vals.append(r["value"])
    wall = time.perf_counter() - t0
    value = float(np.mean(vals))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * wall / max(1, args.steps),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": spec.name, "n_tokens": spec.n_tokens, "prefix_len": spec.prefix_len,
                   "n_heads": spec.n_heads, "topk": spec.topk, "step_sample_rows": rows_per_step},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": r["cores"], "kind": "oracle",
                         "sample": f"{rows_per_step} random query rows per step of {spec.name}"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_e2e(args, spec, dev, out, lse, stream, world):
    """Same step from pinned HOST buffers through the package's host-buffer
    prefill (smla_sparse_mla_prefill per chunk of E2E_CHUNK query tokens): every
    step copies q, q_I and w in and reads out and lse back, the copies of one
    chunk overlapping the kernels of the others."""
    T, H, k, P = spec.n_tokens, spec.n_heads, spec.topk, spec.prefix_len
    q_h = dev.q.cpu().pin_memory()
    qi_h = dev.q_idx.cpu().pin_memory()
    w_h = dev.w.cpu().pin_memory()
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    lse_h = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    hp = smla.HostPrefill(dev.cache, dev.page_table, P, T, H, spec.h_idx, spec.d_idx, spec.idx_dtype, k,
                          spec.sm_scale, chunk=e2e_chunks(T))

    def e2e_step():
        hp.run(q_h, qi_h, w_h, out_h, lse_h, stream=stream)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    barrier(world)
    e_s, e_e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n_e2e = max(3, min(args.steps, 10))
    e_s.record(stream)
    for _ in range(n_e2e):
        e2e_step()
    e_e.record(stream)
    torch.cuda.synchronize()
    assert smla.read_status(hp.ws)[0] == 0
    # the host copy of the result is the device result
    assert torch.equal(out_h.view(torch.int16), hp.out.cpu().view(torch.int16))
    ms_e2e = reduce_max(e_s.elapsed_time(e_e) / n_e2e, world)
    h2d = q_h.numel() * q_h.element_size() + qi_h.numel() * qi_h.element_size() + w_h.numel() * 4
    d2h = out_h.numel() * 2 + lse_h.numel() * 4
    return ms_e2e, h2d, d2h


def measure_decode(args, stream, flush):
    """The decode workload (64 requests x 2 MTP tokens, 8K-128K keys each, FP8
    cache in a shuffled pool): one step = smla_sparse_mla_decode (split-key
    indexer, candidate merge, sparse MLA). Reported next to the headline; its
    roofline is HBM bandwidth over the algorithmic bytes of the step."""
    spec = wl.SPECS["decode"]
    dev = wl.make(spec, "cuda")
    lens = dev.seq_lens
    max_len = int(lens.max().item())
    H, k = spec.n_heads, spec.topk
    rows = spec.n_seqs * spec.q_per_seq
    out = torch.empty((rows, H, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((rows, H), dtype=torch.float32, device="cuda")
    idx = torch.empty((rows, k), dtype=torch.int32, device="cuda")
    ws = smla.workspace(smla.decode_workspace_bytes(spec.n_seqs, max_len, spec.q_per_seq, H, spec.h_idx, k))

    def step():
        smla.sparse_mla_decode(dev.cache, dev.page_table, lens, max_len, spec.q_per_seq, dev.q, dev.q_idx, dev.w,
                               k, spec.sm_scale, out=out, lse=lse, out_idx=idx, ws=ws)

    for _ in range(max(3, args.warmup)):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    assert smla.read_status(ws)[0] == 0
    n = max(5, min(args.steps, 20))

    def timed(run):
        ev = []
        for _ in range(n):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            run()
            e1.record(stream)
            ev.append((e0, e1))
        torch.cuda.synchronize()
        return float(np.median([a.elapsed_time(b) for a, b in ev]))

    # a decode step is a few short kernels: launched one by one from Python the
    # host work between launches shows up as device idle time, so the step is
    # captured once in a CUDA graph (as a serving loop would) and replayed
    ms_eager = timed(step)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    torch.cuda.synchronize()
    ms = timed(graph.replay)
    assert smla.read_status(ws)[0] == 0
    # the same step with the latent cache (rows and scales) in page-locked host
    # memory: the attention gathers only the selected rows over the host link
    host_cache = wl.Cache(dev.cache.kv.cpu().pin_memory(), dev.cache.kv_scale.cpu().pin_memory(), dev.cache.k_idx,
                          dev.cache.k_idx_scale, spec.kv_dtype, spec.idx_dtype)
    out_h = torch.empty_like(out)

    def step_host():
        smla.sparse_mla_decode(host_cache, dev.page_table, lens, max_len, spec.q_per_seq, dev.q, dev.q_idx, dev.w,
                               k, spec.sm_scale, out=out_h, lse=lse, out_idx=idx, ws=ws)

    for _ in range(3):
        step_host()
    torch.cuda.synchronize()
    graph_h = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph_h):
        step_host()
    torch.cuda.synchronize()
    ms_host = timed(graph_h.replay)
    assert smla.read_status(ws)[0] == 0
    assert torch.equal(out_h.view(torch.int16), out.view(torch.int16))
    host_bytes = rows * k * (576 + 4)  # selected FP8 rows and their scales
    cnt = counting.decode_counts([int(x) for x in lens.tolist()], spec.q_per_seq, H, spec.h_idx, spec.d_idx, k,
                                 spec.kv_dtype, 1)
    alg = cnt["idx_bytes"] + cnt["mla_bytes"]
    pk = peaks()
    gbs = alg / (ms / 1e3) / 1e9
    return {"workload": f"decode: {spec.n_seqs} requests x {spec.q_per_seq} tokens, keys U[{spec.len_min}, "
                        f"{spec.len_max}], FP8 KV + FP8 indexer, top-{k}, shuffled pages",
            "ms_per_step": ms, "tokens_per_s": rows / (ms / 1e3), "algorithmic_bytes": alg,
            "gbs_algorithmic": gbs, "hbm_peak_gbs": pk["hbm"], "frac_of_hbm": gbs / pk["hbm"],
            "ms_per_step_eager": ms_eager, "launch": "CUDA graph of one step, replayed",
            "host_kv": {"ms_per_step": ms_host, "tokens_per_s": rows / (ms_host / 1e3),
                        "gathered_host_bytes": host_bytes, "gbs_host_gather": host_bytes / (ms_host / 1e3) / 1e9,
                        "what": "latent cache rows and scales in page-locked host memory, indexer keys in HBM"},
            "gpu_launches_per_step": 4, "l2": "256 MB buffer written between timed steps"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="smla", choices=["smla", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-rows", type=int, default=2560)
    ap.add_argument("--workload", default=WORKLOAD, choices=["prefill16k"],
                    help="benchmarked workload (the 16,384-token prefill)")
    ap.add_argument("--tokens", type=int, default=0,
                    help="profiling only: use this many query tokens instead of the workload's")
    ap.add_argument("--no-e2e", action="store_true", help="profiling only: skip the host-buffer pass")
    ap.add_argument("--no-decode", action="store_true", help="profiling only: skip the decode measurement")
    ap.add_argument("--decode-only", action="store_true",
                    help="profiling only: run and print the decode measurement alone")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    rank, world, local = dist_setup(args.gpus)
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    torch.cuda.set_device(local)
    if rank == 0:
        smla.build()
    barrier(world)
    L = smla.lib()
    if args.decode_only:
        flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
        d = measure_decode(args, torch.cuda.current_stream(), flush)
        if rank == 0:
            print(json.dumps({"decode": d}))
        return
    spec = wl.SPECS[args.workload]
    if args.tokens:
        spec = wl.scaled(spec, n_tokens=args.tokens)
    dev = wl.make(spec, "cuda")
    T, H, k = spec.n_tokens, spec.n_heads, spec.topk
    P = spec.prefix_len
    stream = torch.cuda.current_stream()
    seq_lens = torch.tensor([P + T], dtype=torch.int32, device="cuda")
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    out = torch.empty((T, H, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((T, H), dtype=torch.float32, device="cuda")
    ws_i = smla.workspace(L.smla_indexer_topk_workspace_size(1, P + T, T, spec.h_idx, k))
    ws_m = smla.workspace(L.smla_sparse_mla_fwd_workspace_size(P + T, T, H, k, smla._dtype_code(spec.kv_dtype)))
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")

    def step():
        smla.indexer_topk(dev.cache, dev.page_table, seq_lens, P + T, T, dev.q_idx, dev.w, k, out_idx=idx,
                          ws=ws_i)
        e_mid = torch.cuda.Event(enable_timing=True)
        e_mid.record(stream)
        smla.sparse_mla_fwd(dev.cache, dev.page_table, dev.q, idx, spec.sm_scale, prefix_len=P, out=out,
                            lse=lse, ws=ws_m)
        return e_mid

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    assert smla.read_status(ws_i)[0] == 0 and smla.read_status(ws_m)[0] == 0
    barrier(world)
    torch.cuda.synchronize()
    t_idx, t_mla, t_step = [], [], []
    with ClockSampler(local) as clk:
        wall0 = time.perf_counter()
        for _ in range(args.steps):
            flush.zero_()  # write > L2 between steps
            e0 = torch.cuda.Event(enable_timing=True)
            e2 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            e1 = step()
            e2.record(stream)
            t_step.append((e0, e1, e2))
        torch.cuda.synchronize()
        wall = time.perf_counter() - wall0
    barrier(world)
    for e0, e1, e2 in t_step:
        t_idx.append(e0.elapsed_time(e1))
        t_mla.append(e1.elapsed_time(e2))
    ms_step = float(np.mean([a + b for a, b in zip(t_idx, t_mla)]))
    ms_step_max = reduce_max(ms_step, world)
    ms_idx, ms_mla = float(np.mean(t_idx)), float(np.mean(t_mla))
    value = world * T / (ms_step_max / 1e3)

    # ------------------------------------------------------------------ e2e through host buffers
    if args.no_e2e:
        ms_e2e, h2d, d2h = float("nan"), 0, 0
    else:
        ms_e2e, h2d, d2h = run_e2e(args, spec, dev, out, lse, stream, world)

    decode = None if args.no_decode else measure_decode(args, stream, flush)

    # ------------------------------------------------------------------ roofline
    pk = peaks()
    cnt = counting.prefill_counts(P, T, H, spec.h_idx, spec.d_idx, k, spec.kv_dtype,
                                  1 if spec.idx_dtype == "fp8" else 2)
    mla_tflops = cnt["mla_flops"] / (ms_mla / 1e3) / 1e12
    idx_tflops = cnt["idx_flops"] / (ms_idx / 1e3) / 1e12
    fp8_peak = 2 * pk["bf16"]
    dominant_is_mla = ms_mla >= ms_idx
    roof = {"kernel": "sparse_mla (mla_kernel)" if dominant_is_mla else "indexer_topk (indexer_kernel)",
            "bound": "tensor", "unit": "TFLOP/s",
            "achieved": mla_tflops if dominant_is_mla else idx_tflops,
            "peak": pk["bf16"] if dominant_is_mla else fp8_peak,
            "peak_src": (f"{pk['src']} bf16 burst" if dominant_is_mla else
                         f"{pk['src']} bf16 burst x2 (nominal fp8/bf16 ratio)"),
            "traffic": measured_traffic("mla_kernel" if dominant_is_mla else "indexer_kernel")}
    if T != wl.SPECS[args.workload].n_tokens:
        roof["traffic"] = None  # the capture is of the full-size workload
    roof["frac"] = roof["achieved"] / roof["peak"]
    kernels = {
        "indexer_topk": {"ms": ms_idx, "share": ms_idx / (ms_idx + ms_mla), "tflops_fp8": idx_tflops,
                         "frac_of_fp8_peak": idx_tflops / fp8_peak},
        "sparse_mla": {"ms": ms_mla, "share": ms_mla / (ms_idx + ms_mla), "tflops_bf16": mla_tflops,
                       "frac_of_bf16_peak": mla_tflops / pk["bf16"],
                       "gbs_algorithmic": cnt["mla_bytes"] / (ms_mla / 1e3) / 1e9},
    }
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step_max, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": {"workload": f"{spec.name}: T={T} new tokens, prefix {P}, {H} heads, latent 576 BF16 KV, "
                               f"indexer {spec.h_idx}x{spec.d_idx} FP8, top-{k}",
                   "indexer_dtype": "fp8(e4m3) operands, fp32 accumulate",
                   "mla_dtype": "bf16 q and cache widened exactly to f16 MMA operands, f16 P, fp32 accumulate, "
                                "bf16 output",
                   "parallelism": f"replicas x{world}",
                   "l2": "256 MB buffer written between timed steps", "wall_s_timed_region": wall},
        "roofline": roof, "kernels": kernels,
        "e2e": {"value": world * T / (ms_e2e / 1e3) if ms_e2e == ms_e2e else None, "unit": UNIT,
                "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": ms_e2e,
                "path": "pinned host q/q_I/w -> H2D -> smla_sparse_mla_prefill -> D2H out/lse, pipelined in "
                        f"chunks of query tokens {e2e_chunks(T)} (HostPrefill)"},
        # per step: indexer_kernel, shadow_convert_kernel (BF16 cache only), mla_kernel
        "gpu_launches": (3 if spec.kv_dtype == "bf16" else 2) * args.steps,
        "decode": decode,
        "clocks": clk.summary(),
    }
    if rank == 0:
        if not args.no_cpu_baseline and world == 1:
            line["cpu_baseline"] = cpu_oracle_sample(spec, dev, args.cpu_rows)
        elif not args.no_cpu_baseline:
            line["cpu_baseline"] = None
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
