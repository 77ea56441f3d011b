"""Throughput of the indexer -> top-k -> sparse MLA layer step on GB300.

One step = one pass of the whole hot path over one batch of synthetic input.
The headline workload is the long prefill: 131,072 query tokens of one
sequence (64 heads, 32x128 FP8 indexer, top-2048, FP8 latent cache with a
per-token scale), processed as 8,192-token query chunks against the growing
cache, each chunk one call of the product entry smla_sparse_mla_prefill
(indexer + exact top-k, then sparse MLA). Metric: query tokens per second per
layer.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl smla|reference]

Next to the headline the line carries a per-kernel split of the same step
(indexer and attention timed in a separate pass), the 16,384-token prefill, the
million-token prefix extension and the decode batch as extra keys.

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
WORKLOAD = "prefill128k"
L2_FLUSH_BYTES = 256 << 20
# oracle rows timed for the CPU baseline (about 10-30 s of host work per workload)
CPU_ROWS = {"prefill128k": 1600, "prefill16k": 2560, "prefix1m": 64}


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


def measured_traffic(kernel, summary):
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


def stage_traffic(kernels, summary):
    """Summed DRAM bytes per launch of the kernels of one stage, or None if any
    is missing or stale."""
    parts = [measured_traffic(k, summary) for k in kernels]
    return None if any(x is None for x in parts) else sum(parts)


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
        sm, mx, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
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
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx) if mx else max_mhz_default,
                "reasons": sorted(reasons), "samples": len(sm), "power_w_max": max(power) if power else None}


def chunk_list(spec):
    """(prefix, n_tokens) of every prefill call of one step of `spec`."""
    step = spec.chunk if spec.chunk > 0 else spec.n_tokens
    return [(spec.prefix_len + a, min(spec.n_tokens, a + step) - a) for a in range(0, spec.n_tokens, step)]


class PrefillStep:
    """One step of a prefill workload on resident device inputs: every chunk is
    one smla_sparse_mla_prefill call (the product entry) on one workspace."""

    def __init__(self, spec, dev):
        self.spec, self.dev = spec, dev
        T, H = spec.n_tokens, spec.n_heads
        self.out = torch.empty((T, H, 512), dtype=torch.bfloat16, device="cuda")
        self.lse = torch.empty((T, H), dtype=torch.float32, device="cuda")
        self.chunks = chunk_list(spec)
        need = max(smla.prefill_workspace_bytes(P, n, H, spec.h_idx, spec.topk, spec.kv_dtype)
                   for P, n in self.chunks)
        # chunk c's workspace starts 256 bytes after chunk c-1's: its own status word
        self.ws = smla.workspace(need + smla.STATUS_BYTES * len(self.chunks))

    def run(self, stream=None):
        s, d = self.spec, self.dev
        for c, (P, n) in enumerate(self.chunks):
            a = P - s.prefix_len
            smla.sparse_mla_prefill(d.cache, d.page_table, P, d.q[a:a + n], d.q_idx[a:a + n], d.w[a:a + n],
                                    s.topk, s.sm_scale, out=self.out[a:a + n], lse=self.lse[a:a + n],
                                    ws=self.ws[smla.STATUS_BYTES * c:], stream=stream)

    def status(self):
        return smla.read_status_chunks(self.ws, len(self.chunks))[0]

    def launches(self):
        """Kernels one step launches: per chunk the indexer and, for rows longer
        than 16,384 keys, the selection kernel once per row block of the score
        array (the library's rule: blocks of the rows that 16 GiB holds, in
        whole waves of 8 rows per SM when several are needed), the f16 copy of
        the rows (BF16 and per-token FP8 caches) and the attention."""
        sms = torch.cuda.get_device_properties(0).multi_processor_count
        n = 0
        for P, T in self.chunks:
            n += 2 + (self.spec.kv_dtype in ("bf16", "fp8"))  # indexer, attention, the f16 copy
            if P + T > 16384:
                stride = (P + T + 31) // 32 * 32
                fit = max(min(T, 608), min(T, (16 << 30) // (stride * 4) // 4 * 4))
                block = fit
                if fit < T:
                    wave = 8 * sms
                    if fit >= wave:
                        block = fit // wave * wave
                    else:
                        nb = -(-T // fit)
                        block = min(fit, (-(-T // nb) + 3) // 4 * 4)
                blocks = -(-T // block)
                n += 2 * blocks - 1  # one indexer per block (one counted above), one selection per block
        return n


def time_steps(run, n, stream, flush):
    """CUDA-event time (ms) of each of n calls of run(), L2 flushed before each."""
    ev = []
    for _ in range(n):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        run()
        e1.record(stream)
        ev.append((e0, e1))
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


def stage_split(spec, dev, stream, flush, n_steps):
    """Per-kernel split of a prefill step: every chunk as smla_indexer_topk
    (indexer + exact top-k, the same kernels the prefill entry launches) then
    smla_sparse_mla_fwd on its index list (with the f16 shadow for BF16
    caches), events between them. Returns mean ms of the indexer and the
    attention per step."""
    H, k = spec.n_heads, spec.topk
    chunks = chunk_list(spec)
    nmax = max(n for _, n in chunks)
    idx = torch.empty((nmax, k), dtype=torch.int32, device="cuda")
    out = torch.empty((nmax, H, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((nmax, H), dtype=torch.float32, device="cuda")
    L = smla.lib()
    ws_i = smla.workspace(max(L.smla_indexer_topk_workspace_size(1, P + n, n, spec.h_idx, k) for P, n in chunks))
    ws_m = smla.workspace(max(L.smla_sparse_mla_fwd_workspace_size(P + n, n, H, k, smla._dtype_code(spec.kv_dtype))
                              for P, n in chunks))
    lens = [torch.tensor([P + n], dtype=torch.int32, device="cuda") for P, n in chunks]

    def one(evs):
        for c, (P, n) in enumerate(chunks):
            a = P - spec.prefix_len
            e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
            e[0].record(stream)
            smla.indexer_topk(dev.cache, dev.page_table, lens[c], P + n, n, dev.q_idx[a:a + n], dev.w[a:a + n], k,
                              out_idx=idx[:n], ws=ws_i, stream=stream)
            e[1].record(stream)
            smla.sparse_mla_fwd(dev.cache, dev.page_table, dev.q[a:a + n], idx[:n], spec.sm_scale, prefix_len=P,
                                out=out[:n], lse=lse[:n], ws=ws_m, stream=stream)
            e[2].record(stream)
            evs.append(e)

    one([])
    torch.cuda.synchronize()
    assert smla.read_status(ws_i)[0] == 0 and smla.read_status(ws_m)[0] == 0
    t_idx, t_mla = [], []
    for _ in range(n_steps):
        flush.zero_()
        evs = []
        one(evs)
        torch.cuda.synchronize()
        t_idx.append(sum(e[0].elapsed_time(e[1]) for e in evs))
        t_mla.append(sum(e[1].elapsed_time(e[2]) for e in evs))
        per_chunk = [(e[0].elapsed_time(e[1]), e[1].elapsed_time(e[2])) for e in evs]
    return float(np.mean(t_idx)), float(np.mean(t_mla)), per_chunk


def stage_report(spec, ms_idx, ms_mla, pk):
    """Achieved rates of the two stages against their rooflines."""
    cnt = {"pairs": 0, "idx_flops": 0, "mla_flops": 0, "mla_bytes": 0, "mla_gather_bytes": 0, "idx_bytes": 0}
    for P, n in chunk_list(spec):
        c = counting.prefill_counts(P, n, spec.n_heads, spec.h_idx, spec.d_idx, spec.topk, spec.kv_dtype,
                                    1 if spec.idx_dtype == "fp8" else 2)
        for key in cnt:
            cnt[key] += c[key]
    fp8_burst, fp8_sust = 2 * pk["bf16"], 2 * pk["bf16_sust"]
    idx_tf = cnt["idx_flops"] / (ms_idx / 1e3) / 1e12
    mla_tf = cnt["mla_flops"] / (ms_mla / 1e3) / 1e12
    return cnt, {
        "indexer_topk": {"ms": ms_idx, "share": ms_idx / (ms_idx + ms_mla), "tflops_fp8": idx_tf,
                         "frac_of_fp8_peak_sustained": idx_tf / fp8_sust, "frac_of_fp8_peak_burst": idx_tf / fp8_burst,
                         "flops": cnt["idx_flops"], "pairs": cnt["pairs"]},
        "sparse_mla": {"ms": ms_mla, "share": ms_mla / (ms_idx + ms_mla), "tflops_bf16": mla_tf,
                       "frac_of_bf16_peak_sustained": mla_tf / pk["bf16_sust"],
                       "frac_of_bf16_peak_burst": mla_tf / pk["bf16"], "flops": cnt["mla_flops"],
                       "gbs_hbm_algorithmic": cnt["mla_bytes"] / (ms_mla / 1e3) / 1e9,
                       "gbs_l2_gathers": cnt["mla_gather_bytes"] / (ms_mla / 1e3) / 1e9},
    }


def host_sample_rows(T: int, n: int, seed: int = 2024):
    rng = np.random.default_rng(seed)
    return np.sort(rng.choice(T, size=n, replace=False))


def cpu_oracle_sample(spec, dev, n_rows, cache_h=None):
    """Time the CPU oracle (all host cores) on n_rows random rows of the workload."""
    import oracle
    rows = host_sample_rows(spec.n_tokens, n_rows)
    if cache_h is None:
        cache_h = dev.cache.to("cpu")
    oracle.build()
    t0 = time.perf_counter()
    _, _, _, _, used, _ = oracle.prefill_rows(dev, rows, cache_host=cache_h)
    dt = time.perf_counter() - t0
    return dict(value=n_rows / dt, unit=UNIT, cores=int(used), kind="oracle",
                sample=f"{n_rows} random query rows of {spec.name} (full indexer over their causal keys, "
                       f"full-sort top-{spec.topk}, fp64 attention), {dt:.1f} s wall; tokens/s of the sample, "
                       "extrapolated to the workload")


def run_reference(args, rank, world):
    """--impl reference: the CPU oracle, timed on the host cores, on rank 0 only."""
    if rank != 0:
        return
    spec = wl.SPECS[WORKLOAD]
    dev_name = "cuda" if torch.cuda.is_available() else "cpu"
    dev = wl.make(spec, dev_name)
    cache_h = dev.cache.to("cpu")
    rows_per_step = 32
    for _ in range(args.warmup):
        cpu_oracle_sample(spec, dev, 2, cache_h)
    vals = []
    t0 = time.perf_counter()
    for _ in range(args.steps):
        r = cpu_oracle_sample(spec, dev, rows_per_step, cache_h)
        vals.append(r["value"])
    wall = time.perf_counter() - t0
    value = float(np.mean(vals))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * wall / max(1, args.steps),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": spec.name, "n_tokens": spec.n_tokens, "prefix_len": spec.prefix_len,
                   "chunk": spec.chunk, "n_heads": spec.n_heads, "topk": spec.topk,
                   "step_sample_rows": rows_per_step},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": r["cores"], "kind": "oracle",
                         "sample": f"{rows_per_step} random query rows per step of {spec.name}"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_e2e(args, spec, dev, ref_out, stream, world):
    """The step from pinned HOST buffers through the package's host-buffer
    prefill: every step copies q, q_I and w in and reads out and lse back, chunk
    by chunk (the workload's own 8,192-token chunks, each one
    smla_sparse_mla_prefill call), the copies of one chunk overlapping the
    kernels of the others."""
    T, H, k, P = spec.n_tokens, spec.n_heads, spec.topk, spec.prefix_len
    q_h = dev.q.cpu().pin_memory()
    qi_h = dev.q_idx.cpu().pin_memory()
    w_h = dev.w.cpu().pin_memory()
    out_h = torch.empty((T, H, 512), dtype=torch.bfloat16).pin_memory()
    lse_h = torch.empty((T, H), dtype=torch.float32).pin_memory()
    chunk = spec.chunk if spec.chunk > 0 else T
    hp = smla.HostPrefill(dev.cache, dev.page_table, P, T, H, spec.h_idx, spec.d_idx, spec.idx_dtype, k,
                          spec.sm_scale, chunk=chunk)

    def e2e_step():
        hp.run(q_h, qi_h, w_h, out_h, lse_h, stream=stream)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    barrier(world)
    n_e2e = max(3, min(args.steps, 8))
    times = []
    for _ in range(n_e2e):
        e_s, e_e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e_s.record(stream)
        e2e_step()
        e_e.record(stream)
        times.append((e_s, e_e))
    torch.cuda.synchronize()
    assert hp.read_status()[0] == 0
    # the host copy of the result is the device-resident step's result
    assert torch.equal(out_h.view(torch.int16), ref_out.cpu().view(torch.int16))
    per = [a.elapsed_time(b) for a, b in times]
    ms_e2e = reduce_max(float(np.mean(per)), world)
    h2d = q_h.numel() * q_h.element_size() + qi_h.numel() * qi_h.element_size() + w_h.numel() * 4
    d2h = out_h.numel() * 2 + lse_h.numel() * 4
    spread = {"steps": len(per), "min": float(np.min(per)), "median": float(np.median(per)), "max": float(np.max(per))}
    return ms_e2e, h2d, d2h, chunk, spread


def measure_extra_prefill(name, args, stream, flush):
    """An extra prefill workload: the step through the product entry, then the
    per-kernel split."""
    spec = wl.SPECS[name]
    dev = wl.make(spec, "cuda")
    ps = PrefillStep(spec, dev)
    for _ in range(3):
        ps.run(stream)
    torch.cuda.synchronize()
    assert ps.status() == 0
    n = max(3, min(args.steps, 10))
    ms = float(np.mean(time_steps(lambda: ps.run(stream), n, stream, flush)))
    ms_idx, ms_mla, _ = stage_split(spec, dev, stream, flush, 2)
    _, kern = stage_report(spec, ms_idx, ms_mla, peaks())
    res = {"workload": f"{spec.name}: T={spec.n_tokens} new tokens after a prefix of {spec.prefix_len}"
                       + (f" in {spec.chunk}-token chunks" if spec.chunk else "")
                       + f", {spec.n_heads} heads, {spec.kv_dtype} latent cache, indexer {spec.h_idx}x{spec.d_idx} "
                       f"{spec.idx_dtype}, top-{spec.topk}" + (", shuffled pages" if spec.shuffled else ""),
           "ms_per_step": ms, "tokens_per_s": spec.n_tokens / (ms / 1e3), "kernels": kern,
           "gpu_launches_per_step": ps.launches()}
    del ps, dev
    torch.cuda.empty_cache()
    return res


def measure_decode(args, stream, flush):
    """The decode workload (64 requests x 2 MTP tokens, 8K-128K keys each, FP8
    cache in a shuffled pool): one step = smla_sparse_mla_decode (split-key
    indexer, candidate merge, sparse MLA). Its roofline is HBM bandwidth over
    the algorithmic bytes of the step."""
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
        return float(np.median(time_steps(run, n, stream, flush)))

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
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="smla", choices=["smla", "reference"])
    ap.add_argument("--workload", default=WORKLOAD, choices=["prefill128k", "prefill16k", "prefix1m"],
                    help="benchmarked prefill workload (default: the 131,072-token prefill in 8,192-token chunks)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-rows", type=int, default=0, help="oracle rows of the CPU baseline (0: the default)")
    ap.add_argument("--tokens", type=int, default=0,
                    help="profiling only: use this many query tokens instead of the workload's")
    ap.add_argument("--prefix", type=int, default=-1,
                    help="profiling only: use this prefix length (with --tokens: one chunk of the workload at that "
                         "position)")
    ap.add_argument("--no-e2e", action="store_true", help="profiling only: skip the host-buffer pass")
    ap.add_argument("--no-extras", action="store_true",
                    help="profiling only: skip the extra workloads (16K prefill, 1M prefix, decode)")
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
    smla.lib()
    stream = torch.cuda.current_stream()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    if args.decode_only:
        d = measure_decode(args, stream, flush)
        if rank == 0:
            print(json.dumps({"decode": d}))
        return
    spec = wl.SPECS[args.workload]
    if args.tokens:
        spec = wl.scaled(spec, n_tokens=args.tokens)
    if args.prefix >= 0:
        spec = wl.scaled(spec, prefix_len=args.prefix)
    dev = wl.make(spec, "cuda")
    T, H, k, P = spec.n_tokens, spec.n_heads, spec.topk, spec.prefix_len
    ps = PrefillStep(spec, dev)
    for _ in range(args.warmup):
        flush.zero_()
        ps.run(stream)
    torch.cuda.synchronize()
    assert ps.status() == 0
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        wall0 = time.perf_counter()
        t_step = time_steps(lambda: ps.run(stream), args.steps, stream, flush)
        wall = time.perf_counter() - wall0
    barrier(world)
    assert ps.status() == 0
    ms_step = float(np.mean(t_step))
    ms_step_max = reduce_max(ms_step, world)
    value = world * T / (ms_step_max / 1e3)

    # ------------------------------------------------------------------ per-kernel split (separate pass)
    ms_idx, ms_mla, per_chunk = stage_split(spec, dev, stream, flush, 2)
    pk = peaks()
    cnt, kernels = stage_report(spec, ms_idx, ms_mla, pk)
    kernels["split_pass"] = ("the same chunks as smla_indexer_topk + smla_sparse_mla_fwd calls with events between "
                             "them, mean of 2 steps; the headline times the smla_sparse_mla_prefill calls")
    kernels["last_chunk_ms"] = {"indexer_topk": per_chunk[-1][0], "sparse_mla": per_chunk[-1][1]}

    # ------------------------------------------------------------------ e2e through host buffers
    if args.no_e2e:
        ms_e2e, h2d, d2h, e2e_chunk, e2e_spread = float("nan"), 0, 0, 0, None
    else:
        ms_e2e, h2d, d2h, e2e_chunk, e2e_spread = run_e2e(args, spec, dev, ps.out, stream, world)

    # ------------------------------------------------------------------ roofline of the dominant kernel
    dominant_is_mla = ms_mla >= ms_idx
    n_launch = len(ps.chunks)
    if dominant_is_mla:
        roof = {"kernel": "mla_kernel (sparse MLA)", "bound": "tensor", "unit": "TFLOP/s",
                "achieved": kernels["sparse_mla"]["tflops_bf16"], "peak": pk["bf16_sust"],
                "peak_src": f"{pk['src']} bf16 sustained (the kernel runs inside a long step)",
                "traffic": measured_traffic("mla_kernel", f"dram_traffic_{spec.name}.md")}
    else:
        roof = {"kernel": "indexer_kernel + its selection kernel (one smla_indexer_topk call per chunk)",
                "bound": "tensor", "unit": "TFLOP/s",
                "achieved": kernels["indexer_topk"]["tflops_fp8"], "peak": 2 * pk["bf16_sust"],
                "peak_src": f"{pk['src']} bf16 sustained x2 (the nominal fp8/bf16 ratio; the kernel runs inside "
                            "a long step)",
                "traffic": stage_traffic(("indexer_kernel", "select_sampled_kernel"), f"dram_traffic_{spec.name}.md")}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["per_launch"] = (f"achieved = the stage's algorithmic FLOPs over the step's {n_launch} calls / their summed "
                          "event time (the indexer stage times the scoring kernel and the selection kernel together)")
    if args.tokens or args.prefix >= 0:
        roof["traffic"] = None

    launches_per_step = ps.launches()
    cpu_base = None
    if rank == 0 and not args.no_cpu_baseline and world == 1:
        cpu_base = cpu_oracle_sample(spec, dev, args.cpu_rows or CPU_ROWS.get(spec.name, 256))
    extras = {}
    if not args.no_extras:
        del dev, ps
        torch.cuda.empty_cache()
        for name in ("prefill16k", "prefix1m"):
            if name != spec.name:
                extras[name] = measure_extra_prefill(name, args, stream, flush)
        extras["decode"] = measure_decode(args, stream, flush)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step_max, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "fp8" if spec.kv_dtype == "fp8" else "bf16", "data": "synthetic",
        "config": {"workload": f"{spec.name}: T={T} new tokens after a prefix of {P}"
                               + (f", in {spec.chunk}-token chunks against the growing cache" if spec.chunk else "")
                               + f", {H} heads, latent 576 {spec.kv_dtype} KV"
                               + (" with a per-token fp32 scale" if spec.kv_dtype == "fp8" else "")
                               + f", indexer {spec.h_idx}x{spec.d_idx} {spec.idx_dtype}, top-{k}",
                   "entry": "smla_sparse_mla_prefill per chunk",
                   "indexer_dtype": "e4m3 operands, fp32 accumulate, fp32 head-weighted sum",
                   "mla_dtype": "cache rows widened exactly to f16 MMA operands, f16 q and P, fp32 accumulate, "
                                "bf16 output",
                   "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2, and a 256 MB buffer written between timed steps",
                   "wall_s_timed_region": wall},
        "roofline": roof, "kernels": kernels,
        "e2e": {"value": world * T / (ms_e2e / 1e3) if ms_e2e == ms_e2e else None, "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms_e2e,
                "path": "pinned host q/q_I/w -> H2D -> smla_sparse_mla_prefill -> D2H out/lse, pipelined in "
                        f"chunks of {e2e_chunk} query tokens (HostPrefill)",
                "ms_spread": e2e_spread,
                "note": "value is the mean over the steps; the host link is shared with other jobs on the machine "
                        "and copies to host memory slow down at times, hence the spread"},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk.summary(),
    }
    line.update(extras)
    if rank == 0:
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_base
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
