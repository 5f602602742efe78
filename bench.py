"""Benchmark of the paged decode step (default) and of the chunked-prefill step on GB300.

One step = copy-on-write block copy (when the workload has pairs) + paged KV write of
the step's new tokens + paged decode attention (plan, split-K partitions, LSE merge),
all through the C ABI of libpagedkv.so on one stream.

Prints ONE JSON line.  ``value`` is KV-read GB/s of the whole step (algorithmic bytes:
every context token's K and V row of every KV head, read once) with inputs resident in
HBM; ``e2e`` is the same metric with the step's inputs copied from pinned host memory
and the output copied back inside the timed region.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config 1..5]
                    [--variant auto|fma|mma] [--impl ours|reference]
    python bench.py --path prefill [--config 1..3]

With ``--path prefill`` one step = paged KV write of every sequence's new chunk +
chunked-prefill attention (causal, tensor cores); ``value`` is attention TFLOP/s of the
whole step (algorithmic flops: 4 head_dim per visible (query row, key) pair).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_kv_cache_272_gb300 import workloads  # noqa: E402

DEFAULT_CONFIG = 2
METRIC = "paged-attn decode KV-read GB/s (% of GB300 HBM peak); seq-steps/sec/layer"
L2_BYTES = 129 * 1024 * 1024
ATTN_SOURCES = ["paged_kv_cache_272_gb300/csrc/attention.cu",
                "paged_kv_cache_272_gb300/csrc/attention_mma.cu",
                "paged_kv_cache_272_gb300/csrc/attention.cuh",
                "paged_kv_cache_272_gb300/csrc/tc_common.cuh",
                "paged_kv_cache_272_gb300/csrc/pkv_common.cuh"]
PREFILL_SOURCES = ["paged_kv_cache_272_gb300/csrc/prefill.cu",
                   "paged_kv_cache_272_gb300/csrc/tc_common.cuh",
                   "paged_kv_cache_272_gb300/csrc/pkv_common.cuh"]
PREFILL_METRIC = "chunked-prefill paged attention TFLOP/s (% of GB300 bf16 tensor peak)"


def attn_source_hash(sources=None) -> str:
    h = hashlib.sha256()
    for p in sources or ATTN_SOURCES:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


def recorded_traffic(workload: str, variant: str, sources=None):
    """DRAM bytes per attention call from the committed ncu summary, only if it was
    taken on the current attention sources."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    e = rec.get(f"{workload}/{variant}")
    if not e or e.get("source_hash") != attn_source_hash(sources):
        return None
    return e.get("dram_bytes_per_call")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
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
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def setup_dist(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device="cuda") -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(bytes_per_rank_step: int, steps: int, rank_ms: float, world: int,
                   device="cuda") -> tuple[float, float]:
    """Whole-job GB/s of `world` replicas: all ranks' bytes over the slowest rank's
    time.  Returns (GB/s, max milliseconds)."""
    ms = max_over_ranks(rank_ms, world, device)
    return world * bytes_per_rank_step * steps / (ms / 1e3) / 1e9, ms


# -------------------------------------------------------------------------------------
# CPU oracle baseline (a bounded sample of the same workload)
# -------------------------------------------------------------------------------------
FP8_K_SCALE, FP8_V_SCALE = 0.02, 0.015  # N(0,1) data stays well inside E4M3's +-448


def oracle_sample_step(w, n_seqs: int, nthreads: int, k_host, v_host):
    import oracle
    sub_bt = np.ascontiguousarray(w.block_tables[:n_seqs])
    sub_ctx = np.ascontiguousarray(w.context_lens[:n_seqs])
    q = w.q[:n_seqs].cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    t0 = time.perf_counter()
    if k_host.dtype == np.uint8:
        oracle.attention_fp8(q, k_host, v_host, sub_bt, sub_ctx, w.scale, FP8_K_SCALE,
                             FP8_V_SCALE, nthreads=nthreads)
    else:
        oracle.attention(q, k_host, v_host, sub_bt, sub_ctx, w.scale, nthreads=nthreads)
    return time.perf_counter() - t0, int(sub_ctx.astype(np.int64).sum())


def host_caches(w, fp8: bool):
    """The oracle's copy of the pre-step cache (E4M3 codes quantised by the oracle)."""
    import oracle
    k_host = w.k_cache.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    v_host = w.v_cache.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    if not fp8:
        return k_host, v_host
    NB, Hkv, bs, D = k_host.shape
    rows = lambda c: np.ascontiguousarray(c.transpose(0, 2, 1, 3).reshape(NB * bs, Hkv, D))
    kq = np.zeros((NB, Hkv, bs, D), np.uint8)
    vq = np.zeros_like(kq)
    oracle.kv_write_fp8(kq, vq, rows(k_host), rows(v_host), np.arange(NB * bs), FP8_K_SCALE,
                        FP8_V_SCALE)
    return kq, vq


def cpu_baseline(w, budget_s: float = 12.0, fp8: bool = False):
    """Time the oracle, as it stands, on all host cores over the first sequences of the
    workload, growing the sample until it takes about budget_s / 3, then once more."""
    nthreads = os.cpu_count() or 1
    k_host, v_host = host_caches(w, fp8)
    n = min(w.num_seqs, 2)
    while True:
        dt, tok = oracle_sample_step(w, n, nthreads, k_host, v_host)
        if dt > budget_s / 3 or n >= w.num_seqs:
            break
        n = min(w.num_seqs, max(n + 1, int(n * min(8.0, (budget_s / 3) / max(dt, 1e-3)))))
    reps, dt, tok = 0, 0.0, 0
    while reps == 0 or dt < budget_s / 3:  # repeat short samples for a stable time
        d, t = oracle_sample_step(w, n, nthreads, k_host, v_host)
        reps, dt, tok = reps + 1, dt + d, tok + t
    kv_bytes = tok * 2 * w.num_kv_heads * w.head_dim * (1 if fp8 else 2)
    return {"value": kv_bytes / dt / 1e9, "unit": "GB/s", "cores": nthreads, "kind": "oracle",
            "sample": f"first {n} of {w.num_seqs} sequences, all {w.num_q_heads} query heads, "
                      f"{tok // reps} context tokens, {reps} repetitions; fp64 C oracle, "
                      f"OpenMP over (sequence, head)",
            "seconds": dt, "seq_steps_per_s_per_layer": reps * n / dt}


# -------------------------------------------------------------------------------------
def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = workloads.make_config(args.config, device="cpu" if args.config == 1 else "cuda"
                              if torch.cuda.is_available() else "cpu")
    nthreads = os.cpu_count() or 1
    k_host = w.k_cache.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    v_host = w.v_cache.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    # size one step to about 2 s of oracle work
    n = min(w.num_seqs, 2)
    while True:
        dt, tok = oracle_sample_step(w, n, nthreads, k_host, v_host)
        if dt > 0.7 or n >= w.num_seqs:
            break
        n = min(w.num_seqs, max(n + 1, int(n * min(8.0, 0.7 / max(dt, 1e-3)))))
    for _ in range(args.warmup):
        oracle_sample_step(w, n, nthreads, k_host, v_host)
    tot_t, tot_tok = 0.0, 0
    for _ in range(args.steps):
        dt, tok = oracle_sample_step(w, n, nthreads, k_host, v_host)
        tot_t += dt
        tot_tok += tok
    kv = tot_tok * 2 * w.num_kv_heads * w.head_dim * 2
    value = kv / tot_t / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": tot_t / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "sample_seqs": n, "num_seqs": w.num_seqs},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": nthreads, "kind": "oracle",
                         "sample": f"first {n} of {w.num_seqs} sequences per step"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "world_size": world,
    }
    print(json.dumps(line), flush=True)


def run_ours(args):
    from paged_kv_cache_272_gb300 import ops
    world, rank, local = setup_dist(args.gpus)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    variant = {"auto": ops.PKV_ATTN_AUTO, "fma": ops.PKV_ATTN_FMA,
               "mma": ops.PKV_ATTN_MMA}[args.variant]
    ops.set_attention_variant(variant)

    w = workloads.make_config(args.config, device="cuda")
    S, Hq, Hkv, D = w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim
    fp8 = args.kv_dtype == "fp8"
    if fp8:
        # Quantise the whole pre-step cache once (untimed) with the library's own write.
        NB = w.num_blocks
        k = torch.empty(NB, Hkv, 16, D, dtype=torch.uint8, device=dev)
        v = torch.empty_like(k)
        rows = lambda c: c.permute(0, 2, 1, 3).reshape(NB * 16, Hkv, D).contiguous()
        ops.paged_kv_write_fp8(rows(w.k_cache), rows(w.v_cache),
                               torch.arange(NB * 16, dtype=torch.int64, device=dev), k, v,
                               FP8_K_SCALE, FP8_V_SCALE)
        torch.cuda.synchronize()
    else:
        k = w.k_cache.to(dev).contiguous()
        v = w.v_cache.to(dev).contiguous()
    q = w.q.to(dev).contiguous()
    k_new, v_new = w.k_new.to(dev).contiguous(), w.v_new.to(dev).contiguous()
    slots = torch.as_tensor(w.slot_mapping, dtype=torch.int64, device=dev)
    pairs = torch.as_tensor(w.cow_pairs.reshape(-1, 2), dtype=torch.int32, device=dev)
    bt = torch.as_tensor(w.block_tables, dtype=torch.int32, device=dev)
    ctx = torch.as_tensor(w.context_lens, dtype=torch.int32, device=dev)
    out = torch.empty(S, Hq, D, dtype=torch.bfloat16, device=dev)
    P = args.partition or w.partition_size
    mcl = w.max_context_len
    ws = ops.alloc_workspace(S, Hq, D, mcl, P, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    kv_bytes = workloads.kv_read_bytes(w) // (2 if fp8 else 1)
    max_parts = (mcl + P - 1) // P
    launches_per_step = (1 if pairs.numel() else 0) + 1 + 2 + (1 if max_parts > 1 else 0)
    working_set = kv_bytes + q.numel() * 2 * 2
    flush = working_set < 2 * L2_BYTES
    scratch = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev) if flush else None

    def do_copy(pr):
        (ops.paged_block_copy_fp8 if fp8 else ops.paged_block_copy)(k, v, pr, err_flag=err,
                                                                     stream=stream)

    def do_write(kn, vn, sl):
        if fp8:
            ops.paged_kv_write_fp8(kn, vn, sl, k, v, FP8_K_SCALE, FP8_V_SCALE, err_flag=err,
                                   stream=stream)
        else:
            ops.paged_kv_write(kn, vn, sl, k, v, err_flag=err, stream=stream)

    def do_attn(qq, btt, cx):
        if fp8:
            ops.paged_attention_decode_fp8(out, qq, k, v, btt, cx, w.scale, FP8_K_SCALE,
                                           FP8_V_SCALE, mcl, ws, P, err_flag=err, stream=stream)
        else:
            ops.paged_attention_decode(out, qq, k, v, btt, cx, w.scale, mcl, ws, P, err_flag=err,
                                       stream=stream)

    def step():
        if pairs.numel():
            do_copy(pairs)
        do_write(k_new, v_new, slots)
        do_attn(q, bt, ctx)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    if err.item() != 0:
        raise RuntimeError(f"device error flag {err.item()} during warm-up")

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    with ClockSampler(local) as clk:
        t_end = time.perf_counter() + 0.8          # bring clocks to their loaded state
        while time.perf_counter() < t_end:
            step()
            torch.cuda.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        for i in range(args.steps):
            if flush:
                scratch.zero_()
            e0, e1, e2 = ev[i]
            e0.record(stream)
            if pairs.numel():
                do_copy(pairs)
            do_write(k_new, v_new, slots)
            e1.record(stream)
            do_attn(q, bt, ctx)
            e2.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        t_end = time.perf_counter() + 0.4
        while time.perf_counter() < t_end:
            step()
            torch.cuda.synchronize()
    step_ms = [a.elapsed_time(c) for a, b, c in ev]
    attn_ms = [b.elapsed_time(c) for a, b, c in ev]
    value, total_ms = job_throughput(kv_bytes, args.steps, sum(step_ms), world)
    attn_avg_ms = max_over_ranks(sum(attn_ms) / len(attn_ms), world)
    ms_per_step = total_ms / args.steps

    # ---- end to end through the public API, host buffers ------------------------------
    h = {name: t.cpu().pin_memory() for name, t in
         (("q", q), ("k_new", k_new), ("v_new", v_new), ("slots", slots), ("pairs", pairs),
          ("bt", bt), ("ctx", ctx))}
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    dq, dkn, dvn = torch.empty_like(q), torch.empty_like(k_new), torch.empty_like(v_new)
    dsl, dpr = torch.empty_like(slots), torch.empty_like(pairs)
    dbt, dctx = torch.empty_like(bt), torch.empty_like(ctx)
    h2d = sum(t.numel() * t.element_size() for t in h.values())
    d2h = out.numel() * out.element_size()

    def e2e_step():
        dq.copy_(h["q"], non_blocking=True)
        dkn.copy_(h["k_new"], non_blocking=True)
        dvn.copy_(h["v_new"], non_blocking=True)
        dsl.copy_(h["slots"], non_blocking=True)
        dbt.copy_(h["bt"], non_blocking=True)
        dctx.copy_(h["ctx"], non_blocking=True)
        if dpr.numel():
            dpr.copy_(h["pairs"], non_blocking=True)
            do_copy(dpr)
        do_write(dkn, dvn, dsl)
        do_attn(dq, dbt, dctx)
        out_h.copy_(out, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    e2e_ms = 0.0
    for _ in range(args.steps):
        if flush:
            scratch.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        e2e_step()
        b.record(stream)
        b.synchronize()  # the host has the step's output
        e2e_ms += a.elapsed_time(b)
    e2e_value, e2e_ms = job_throughput(kv_bytes, args.steps, e2e_ms, world)

    torch.cuda.synchronize()
    if err.item() != 0:
        raise RuntimeError(f"device error flag {err.item()}")

    peaks, peak_kind = measured_peaks()
    peak = float(peaks["hbm_gbs"])
    achieved = kv_bytes / (attn_avg_ms / 1e3) / 1e9
    G = Hq // Hkv
    # the kernel AUTO picks: tensor-core tiles once a KV head serves 4+ query heads
    vname = {1: "fma", 2: "mma"}.get(variant, "mma" if G >= 4 else "fma")
    if fp8:
        vname = "mma-fp8"  # the E4M3 cache always runs the tensor-core kernel
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3 KV / f16 tiles" if fp8 else "bf16",
        "data": "synthetic",
        "config": {
            "workload": w.name, "kv_dtype": args.kv_dtype, "num_seqs": S, "num_q_heads": Hq, "num_kv_heads": Hkv,
            "head_dim": D, "block_size": w.block_size, "partition_size": P,
            "num_blocks": w.num_blocks, "mean_context": float(w.context_lens.mean()),
            "max_context": mcl, "kv_bytes_per_step": kv_bytes,
            "cow_pairs_per_step": int(w.cow_pairs.shape[0]),
            "new_tokens_per_step": int(w.slot_mapping.shape[0]),
            "l2": ("L2 flushed (256 MB write) before every timed step" if flush else
                   "inputs larger than L2 (KV read per step >> 129 MB)"),
            "attention_variant": args.variant, "attention_kernel": vname,
            "parallelism": "replicas" if world > 1 else "single"},
        "pct_of_hbm_peak": 100.0 * value / peak,
        "seq_steps_per_s_per_layer": world * S / (ms_per_step / 1e3),
        "attention_ms": attn_avg_ms,
        "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms / args.steps},
        "gpu_launches": launches_per_step * args.steps,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak,
                     "traffic": recorded_traffic(w.name, vname),
                     "kernel": "paged_attention_decode: plan + partition (%s) + merge kernels"
                               % vname,
                     "peak_source": f"{peak_kind} hbm_gbs"},
        "clocks": clk.summary(),
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, fp8=fp8)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# -------------------------------------------------------------------------------------
# Chunked prefill
# -------------------------------------------------------------------------------------
def prefill_oracle_sample(w, sel, nthreads, k_host, v_host):
    import oracle
    t0 = time.perf_counter()
    oracle.attention_prefill(w.q.cpu(), k_host, v_host, w.block_tables, w.context_lens,
                             w.query_start, w.scale, sel=sel, nthreads=nthreads)
    dt = time.perf_counter() - t0
    # flops of the sampled rows: 4 D per visible key
    seq = np.searchsorted(w.query_start, sel[:, 0], side="right") - 1
    L = w.query_start[seq + 1] - w.query_start[seq]
    pos = w.context_lens[seq] - L + (sel[:, 0] - w.query_start[seq])
    return dt, int((pos.astype(np.int64) + 1).sum()) * 4 * w.head_dim


def prefill_host_caches(w):
    """The oracle's copy of the cache after the step's write."""
    import oracle
    k = w.k_cache.cpu().contiguous().view(torch.int16).numpy().view(np.uint16).copy()
    v = w.v_cache.cpu().contiguous().view(torch.int16).numpy().view(np.uint16).copy()
    oracle.kv_write(k, v, w.k_new.cpu(), w.v_new.cpu(), w.slot_mapping)
    return k, v


def prefill_sample_rows(w, budget_s, nthreads, k_host, v_host, seed=0):
    """Random (token, head) rows, grown until the oracle takes about budget_s."""
    rng = np.random.default_rng(seed)
    n = 64
    while True:
        sel = np.stack([rng.integers(0, w.num_tokens, n), rng.integers(0, w.num_q_heads, n)],
                       axis=1).astype(np.int32)
        dt, fl = prefill_oracle_sample(w, sel, nthreads, k_host, v_host)
        if dt > budget_s or n >= 1 << 20:
            return sel, dt, fl
        n = int(n * min(8.0, max(1.5, budget_s / max(dt, 1e-3))))


def prefill_cpu_baseline(w, budget_s: float = 12.0):
    nthreads = os.cpu_count() or 1
    k_host, v_host = prefill_host_caches(w)
    sel, dt, fl = prefill_sample_rows(w, budget_s / 3, nthreads, k_host, v_host)
    reps, tot_t, tot_f = 0, 0.0, 0
    while reps == 0 or tot_t < budget_s / 3:
        d, f = prefill_oracle_sample(w, sel, nthreads, k_host, v_host)
        reps, tot_t, tot_f = reps + 1, tot_t + d, tot_f + f
    return {"value": tot_f / tot_t / 1e12, "unit": "TFLOP/s", "cores": nthreads,
            "kind": "oracle",
            "sample": f"{sel.shape[0]} random (token, head) rows of {w.num_tokens} x "
                      f"{w.num_q_heads}, {reps} repetitions; fp64 C oracle, OpenMP over rows",
            "seconds": tot_t}


def run_prefill_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = workloads.make_prefill_config(args.config, device="cpu")
    nthreads = os.cpu_count() or 1
    k_host, v_host = prefill_host_caches(w)
    sel, _, _ = prefill_sample_rows(w, 0.7, nthreads, k_host, v_host)
    for _ in range(args.warmup):
        prefill_oracle_sample(w, sel, nthreads, k_host, v_host)
    tot_t, tot_f = 0.0, 0
    for _ in range(args.steps):
        d, f = prefill_oracle_sample(w, sel, nthreads, k_host, v_host)
        tot_t, tot_f = tot_t + d, tot_f + f
    value = tot_f / tot_t / 1e12
    line = {
        "impl": "reference", "metric": PREFILL_METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": tot_t / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "sample_rows": int(sel.shape[0])},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": nthreads,
                         "kind": "oracle",
                         "sample": f"{sel.shape[0]} random (token, head) rows per step"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_prefill(args):
    from paged_kv_cache_272_gb300 import ops
    world, rank, local = setup_dist(args.gpus)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = workloads.make_prefill_config(args.config, device="cuda")
    T, Hq, Hkv, D = w.num_tokens, w.num_q_heads, w.num_kv_heads, w.head_dim
    k = w.k_cache.to(dev).contiguous()
    v = w.v_cache.to(dev).contiguous()
    q = w.q.to(dev).contiguous()
    k_new, v_new = w.k_new.to(dev).contiguous(), w.v_new.to(dev).contiguous()
    slots = torch.as_tensor(w.slot_mapping, dtype=torch.int64, device=dev)
    bt = torch.as_tensor(w.block_tables, dtype=torch.int32, device=dev)
    ctx = torch.as_tensor(w.context_lens, dtype=torch.int32, device=dev)
    qs = torch.as_tensor(w.query_start, dtype=torch.int32, device=dev)
    out = torch.empty(T, Hq, D, dtype=torch.bfloat16, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    flops = workloads.prefill_flops(w)
    kv_bytes = int(w.context_lens.astype(np.int64).sum()) * 2 * Hkv * D * 2
    working_set = kv_bytes + 2 * q.numel() * 2
    flush = working_set < 2 * L2_BYTES
    scratch = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev) if flush else None

    def do_write(kn, vn, sl):
        ops.paged_kv_write(kn, vn, sl, k, v, err_flag=err, stream=stream)

    def do_attn(qq, btt, cx, qss):
        ops.paged_attention_prefill(out, qq, k, v, btt, cx, qss, w.scale, w.max_query_len,
                                    err_flag=err, stream=stream)

    def step():
        do_write(k_new, v_new, slots)
        do_attn(q, bt, ctx, qs)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    if err.item() != 0:
        raise RuntimeError(f"device error flag {err.item()} during warm-up")
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    with ClockSampler(local) as clk:
        t_end = time.perf_counter() + 0.8
        while time.perf_counter() < t_end:
            step()
            torch.cuda.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        for i in range(args.steps):
            if flush:
                scratch.zero_()
            e0, e1, e2 = ev[i]
            e0.record(stream)
            do_write(k_new, v_new, slots)
            e1.record(stream)
            do_attn(q, bt, ctx, qs)
            e2.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        t_end = time.perf_counter() + 0.4
        while time.perf_counter() < t_end:
            step()
            torch.cuda.synchronize()
    step_ms = max_over_ranks(sum(a.elapsed_time(c) for a, b, c in ev), world)
    attn_ms = max_over_ranks(sum(b.elapsed_time(c) for a, b, c in ev) / args.steps, world)
    value = world * flops * args.steps / (step_ms / 1e3) / 1e12

    h = {name: t.cpu().pin_memory() for name, t in
         (("q", q), ("k_new", k_new), ("v_new", v_new), ("slots", slots), ("bt", bt),
          ("ctx", ctx), ("qs", qs))}
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    dd = {n: torch.empty_like(t, device=dev) for n, t in h.items()}
    h2d = sum(t.numel() * t.element_size() for t in h.values())
    d2h = out.numel() * out.element_size()

    def e2e_step():
        for n in h:
            dd[n].copy_(h[n], non_blocking=True)
        do_write(dd["k_new"], dd["v_new"], dd["slots"])
        do_attn(dd["q"], dd["bt"], dd["ctx"], dd["qs"])
        out_h.copy_(out, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    e2e_ms = 0.0
    for _ in range(args.steps):
        if flush:
            scratch.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        e2e_step()
        b.record(stream)
        b.synchronize()
        e2e_ms += a.elapsed_time(b)
    e2e_ms = max_over_ranks(e2e_ms, world)
    torch.cuda.synchronize()
    if err.item() != 0:
        raise RuntimeError(f"device error flag {err.item()}")

    peaks, peak_kind = measured_peaks()
    peak = float(peaks["bf16_tflops"])
    achieved = flops / (attn_ms / 1e3) / 1e12
    line = {
        "metric": PREFILL_METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {
            "workload": w.name, "num_seqs": w.num_seqs, "new_tokens_per_step": T,
            "max_query_len": w.max_query_len, "num_q_heads": Hq, "num_kv_heads": Hkv,
            "head_dim": D, "block_size": w.block_size, "num_blocks": w.num_blocks,
            "mean_context": float(w.context_lens.mean()), "max_context": w.max_context_len,
            "flops_per_step": flops, "kv_bytes_per_step": kv_bytes,
            "l2": ("L2 flushed (256 MB write) before every timed step" if flush else
                   "working set (KV + q + out) larger than twice L2"),
            "parallelism": "replicas" if world > 1 else "single"},
        "pct_of_bf16_peak": 100.0 * value / peak,
        "attention_ms": attn_ms,
        "e2e": {"value": world * flops * args.steps / (e2e_ms / 1e3) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms / args.steps},
        "gpu_launches": 2 * args.steps,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak,
                     "traffic": recorded_traffic(w.name, "prefill", PREFILL_SOURCES),
                     "kernel": "paged_attention_prefill (prefill_kernel, mma.sync bf16)",
                     "peak_source": f"{peak_kind} bf16_tflops (burst)"},
        "clocks": clk.summary(),
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = prefill_cpu_baseline(w)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--path", default="decode", choices=["decode", "prefill"],
                    help="decode step (default) or chunked-prefill step")
    ap.add_argument("--config", type=int, default=None, choices=[1, 2, 3, 4, 5],
                    help="workload number (decode 1..5, default 2; prefill 1..3, default 2)")
    ap.add_argument("--variant", default="auto", choices=["auto", "fma", "mma"])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--partition", type=int, default=0,
                    help="split-K partition size in tokens (default: the workload's, 512)")
    ap.add_argument("--kv-dtype", default="bf16", choices=["bf16", "fp8"],
                    help="KV cache element type: bf16, or fp8 (E4M3 codes with one scale each)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.config is None:
        args.config = DEFAULT_CONFIG
    if args.path == "prefill":
        if args.config not in workloads.PREFILL_CONFIG_NAMES:
            ap.error("--path prefill takes --config 1..3")
        (run_prefill_reference if args.impl == "reference" else run_prefill)(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
