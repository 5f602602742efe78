"""Benchmark of the paged decode step (default) and of the chunked-prefill step on GB300.

One step = copy-on-write block copy (when the workload has pairs) + paged KV write of
the step's new tokens + paged decode attention (plan, split-K partitions, LSE merge),
all through the C ABI of libpagedkv.so on one stream: by default one paged_decode_step
call (the copies, the write and the plan share one launch), with --step-api separate
the three calls paged_block_copy, paged_kv_write and paged_attention_decode.

Prints ONE JSON line.  ``value`` is KV-read GB/s of the whole step (algorithmic bytes:
every context token's K and V row of every KV head, read once) with inputs resident in
HBM; ``e2e`` is the same metric with the step's inputs copied from pinned host memory
and the output copied back inside the timed region.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config 1..5]
                    [--variant auto|fma|mma] [--impl ours|reference]
    python bench.py --path prefill [--config 1..4]

With ``--path prefill`` one step = paged KV write of every sequence's new chunk +
chunked-prefill attention (causal, tensor cores); ``value`` is attention TFLOP/s of the
whole step (algorithmic flops: 4 head_dim per visible (query row, key) pair).
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch
from torch.cuda import nvtx

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_kv_cache_272_gb300 import workloads  # noqa: E402

# decode: the long-context mixed batch (the largest single-GPU workload); prefill and
# serving runs: their workload 2
DEFAULT_CONFIG = {"decode": 5, "prefill": 2, "serve": 2}
METRIC = "paged-attn decode KV-read GB/s (% of GB300 HBM peak); seq-steps/sec/layer"
L2_BYTES = 129 * 1024 * 1024


class L2Flush:
    """Empties L2 of the step's data between timed steps: writes a buffer of twice the L2
    size, then reads a second one of that size, so that L2 holds only clean lines of
    unrelated data when the step starts (the write alone would leave it full of dirty
    lines whose write-back would land inside the timed step)."""

    def __init__(self, device):
        self.w = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=device)
        self.r = torch.zeros(2 * L2_BYTES // 4, dtype=torch.float32, device=device)
        self.sink = torch.empty((), dtype=torch.float32, device=device)

    def __call__(self):
        self.w.zero_()
        torch.sum(self.r, dim=0, out=self.sink)
ATTN_SOURCES = ["paged_kv_cache_272_gb300/csrc/attention.cu",
                "paged_kv_cache_272_gb300/csrc/attention_mma.cu",
                "paged_kv_cache_272_gb300/csrc/attention.cuh",
                "paged_kv_cache_272_gb300/csrc/plan.cuh",
                "paged_kv_cache_272_gb300/csrc/merge.cuh",
                "paged_kv_cache_272_gb300/csrc/decode_step.cu",
                "paged_kv_cache_272_gb300/csrc/kv_rows.cuh",
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


def per_head_fp8_scales(w):
    """Per-KV-head E4M3 scales calibrated on the pre-step cache: the largest finite |value|
    of each head divided by 448 (E4M3's largest value).  float32 tensors [Hkv] on the
    cache's device."""
    def amax(c):  # one KV head at a time (bounded temporaries on large caches)
        out = []
        for h in range(c.shape[1]):
            x = c[:, h].float().abs()
            out.append(torch.where(torch.isfinite(x), x, torch.zeros_like(x)).amax())
        return (torch.stack(out) / 448.0).clamp_min(1e-12).contiguous()
    return amax(w.k_cache), amax(w.v_cache)


def oracle_sample_step(w, n_seqs: int, nthreads: int, k_host, v_host, ks=FP8_K_SCALE,
                       vs=FP8_V_SCALE):
    import oracle
    sub_bt = np.ascontiguousarray(w.block_tables[:n_seqs])
    sub_ctx = np.ascontiguousarray(w.context_lens[:n_seqs])
    q = w.q[:n_seqs].cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    t0 = time.perf_counter()
    if k_host.dtype == np.uint8:
        oracle.attention_fp8(q, k_host, v_host, sub_bt, sub_ctx, w.scale, ks, vs,
                             nthreads=nthreads)
    else:
        oracle.attention(q, k_host, v_host, sub_bt, sub_ctx, w.scale, nthreads=nthreads)
    return time.perf_counter() - t0, int(sub_ctx.astype(np.int64).sum())


def host_caches(w, fp8: bool, ks=FP8_K_SCALE, vs=FP8_V_SCALE):
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
    oracle.kv_write_fp8(kq, vq, rows(k_host), rows(v_host), np.arange(NB * bs), ks, vs)
    return kq, vq


def cpu_baseline(w, budget_s: float = 12.0, fp8: bool = False, ks=FP8_K_SCALE,
                 vs=FP8_V_SCALE):
    """Time the oracle, as it stands, on all host cores over the first sequences of the
    workload, growing the sample until it takes about budget_s / 3, then once more.
    ks/vs: the E4M3 scales (one each, or one per KV head)."""
    nthreads = os.cpu_count() or 1
    k_host, v_host = host_caches(w, fp8, ks, vs)
    n = min(w.num_seqs, 2)
    while True:
        dt, tok = oracle_sample_step(w, n, nthreads, k_host, v_host, ks, vs)
        if dt > budget_s / 3 or n >= w.num_seqs:
            break
        n = min(w.num_seqs, max(n + 1, int(n * min(8.0, (budget_s / 3) / max(dt, 1e-3)))))
    reps, dt, tok = 0, 0.0, 0
    while reps == 0 or dt < budget_s / 3:  # repeat short samples for a stable time
        d, t = oracle_sample_step(w, n, nthreads, k_host, v_host, ks, vs)
        reps, dt, tok = reps + 1, dt + d, tok + t
    kv_bytes = tok * 2 * w.num_kv_heads * w.head_dim * (1 if fp8 else 2)
    # The same oracle on one thread, over a smaller sample (about budget_s / 4).
    n1 = 1
    while True:
        d1, t1 = oracle_sample_step(w, n1, 1, k_host, v_host, ks, vs)
        if d1 > budget_s / 8 or n1 >= n:
            break
        n1 = min(n, max(n1 + 1, int(n1 * min(8.0, (budget_s / 8) / max(d1, 1e-3)))))
    d1, t1 = oracle_sample_step(w, n1, 1, k_host, v_host, ks, vs)
    kv1 = t1 * 2 * w.num_kv_heads * w.head_dim * (1 if fp8 else 2)
    return {"value": kv_bytes / dt / 1e9, "unit": "GB/s", "cores": nthreads, "kind": "oracle",
            "sample": f"first {n} of {w.num_seqs} sequences, all {w.num_q_heads} query heads, "
                      f"{tok // reps} context tokens, {reps} repetitions; fp64 C oracle, "
                      f"OpenMP over (sequence, head)",
            "seconds": dt, "seq_steps_per_s_per_layer": reps * n / dt,
            "one_thread": {"value": kv1 / d1 / 1e9, "unit": "GB/s", "cores": 1,
                           "sample": f"first {n1} sequences, {t1} context tokens",
                           "seconds": d1, "seq_steps_per_s_per_layer": n1 / d1}}


def sample_parity(w, out, fp8: bool = False, ks=FP8_K_SCALE, vs=FP8_V_SCALE, n_pairs: int = 96,
                  nthreads: int | None = None) -> dict:
    """The bench's own output against the oracle on sampled (sequence, head) rows: one head
    per KV head of the longest sequence plus random rows.  The oracle's caches are the
    pre-step cache with the step applied (copy-on-write, then the new tokens' write) --
    applying it to a cache that already holds it changes nothing.  Tolerance per element
    1e-2 + 1e-2 |ref|, mean |err| <= 2e-3."""
    import oracle
    nthreads = nthreads or os.cpu_count() or 1
    k_host, v_host = host_caches(w, fp8, ks, vs)
    k_host, v_host = np.array(k_host), np.array(v_host)  # private, writable copies
    u16 = lambda t: t.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    if w.cow_pairs.size:
        (oracle.block_copy_fp8 if fp8 else oracle.block_copy)(k_host, v_host, w.cow_pairs)
    if w.slot_mapping.size:
        if fp8:
            oracle.kv_write_fp8(k_host, v_host, u16(w.k_new), u16(w.v_new), w.slot_mapping, ks,
                                vs)
        else:
            oracle.kv_write(k_host, v_host, u16(w.k_new), u16(w.v_new), w.slot_mapping)
    rng = np.random.default_rng(7)
    G = w.num_q_heads // w.num_kv_heads
    s_long = int(np.argmax(w.context_lens))
    pairs = [(s_long, g * G + int(rng.integers(G))) for g in range(w.num_kv_heads)]
    while len(pairs) < n_pairs:
        pairs.append((int(rng.integers(w.num_seqs)), int(rng.integers(w.num_q_heads))))
    sel = np.array(pairs, dtype=np.int32)
    q = u16(w.q)
    if fp8:
        ref = oracle.attention_fp8(q, k_host, v_host, w.block_tables, w.context_lens, w.scale,
                                   ks, vs, sel=sel, nthreads=nthreads)
    else:
        ref = oracle.attention(q, k_host, v_host, w.block_tables, w.context_lens, w.scale,
                               sel=sel, nthreads=nthreads)
    idx_s = torch.as_tensor(sel[:, 0].astype(np.int64), device=out.device)
    idx_h = torch.as_tensor(sel[:, 1].astype(np.int64), device=out.device)
    got = out[idx_s, idx_h].float().cpu().double().numpy()
    err = np.abs(got - ref)
    bad = int(np.count_nonzero(~(err <= 1e-2 + 1e-2 * np.abs(ref))))
    return {"rows": int(sel.shape[0]), "max_abs_err": float(err.max()),
            "mean_abs_err": float(err.mean()), "elements_out_of_tolerance": bad,
            "within_tolerance": bool(bad == 0 and err.mean() <= 2e-3),
            "tolerance": "|err| <= 1e-2 + 1e-2 |ref| per element, mean |err| <= 2e-3",
            "reference": "fp64 oracle on (sequence, head) rows: one head per KV head of the "
                         "longest sequence plus random rows"}


# -------------------------------------------------------------------------------------
def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = workloads.make_config(args.config, device="cpu" if args.config == 1 else "cuda"
                              if torch.cuda.is_available() else "cpu", seed=args.seed)
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

    w = workloads.make_config(args.config, device="cuda", seed=args.seed)
    S, Hq, Hkv, D = w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim
    fp8 = args.kv_dtype == "fp8"
    per_head = fp8 and args.fp8_scales == "head"
    KS, VS = FP8_K_SCALE, FP8_V_SCALE
    if per_head:
        ks_dev, vs_dev = per_head_fp8_scales(w)
        KS, VS = ks_dev.cpu().numpy(), vs_dev.cpu().numpy()
    if fp8:
        # Quantise the whole pre-step cache once (untimed) with the library's own write.
        NB = w.num_blocks
        k = torch.empty(NB, Hkv, 16, D, dtype=torch.uint8, device=dev)
        v = torch.empty_like(k)
        rows = lambda c: c.permute(0, 2, 1, 3).reshape(NB * 16, Hkv, D).contiguous()
        all_slots = torch.arange(NB * 16, dtype=torch.int64, device=dev)
        if per_head:
            ops.paged_kv_write_fp8_per_head(rows(w.k_cache), rows(w.v_cache), all_slots, k, v,
                                            ks_dev, vs_dev)
        else:
            ops.paged_kv_write_fp8(rows(w.k_cache), rows(w.v_cache), all_slots, k, v,
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
    # 0: the automatic split (each call's plan picks 512 ... 4096 tokens)
    P = 0 if args.partition is None else args.partition
    mcl = w.max_context_len
    ws = ops.alloc_workspace(S, Hq, D, mcl, P, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    kv_bytes = workloads.kv_read_bytes(w) // (2 if fp8 else 1)
    max_parts = (mcl + (P or 512) - 1) // (P or 512)  # the workspace's partitions
    if args.step_api == "fused":  # prologue (copies + write + plan), partition, merge
        launches_per_step = (1 if pairs.shape[0] > 1024 else 0) + 2 + (1 if max_parts > 1 else 0)
    else:
        launches_per_step = (1 if pairs.numel() else 0) + 1 + 2 + (1 if max_parts > 1 else 0)
    # distinct bytes a step touches: a shared prefix block counts once (it stays in L2
    # from one step to the next unless flushed)
    unique_kv = workloads.unique_kv_read_bytes(w) // (2 if fp8 else 1)
    working_set = unique_kv + q.numel() * 2 * 2
    flush = working_set < 2 * L2_BYTES
    scratch = L2Flush(dev) if flush else None

    def do_copy(pr):
        (ops.paged_block_copy_fp8 if fp8 else ops.paged_block_copy)(k, v, pr, err_flag=err,
                                                                     stream=stream)

    def do_write(kn, vn, sl):
        if per_head:
            ops.paged_kv_write_fp8_per_head(kn, vn, sl, k, v, ks_dev, vs_dev, err_flag=err,
                                            stream=stream)
        elif fp8:
            ops.paged_kv_write_fp8(kn, vn, sl, k, v, FP8_K_SCALE, FP8_V_SCALE, err_flag=err,
                                   stream=stream)
        else:
            ops.paged_kv_write(kn, vn, sl, k, v, err_flag=err, stream=stream)

    def do_attn(qq, btt, cx):
        if per_head:
            ops.paged_attention_decode_fp8_per_head(out, qq, k, v, btt, cx, w.scale, ks_dev,
                                                    vs_dev, mcl, ws, P, err_flag=err,
                                                    stream=stream)
        elif fp8:
            ops.paged_attention_decode_fp8(out, qq, k, v, btt, cx, w.scale, FP8_K_SCALE,
                                           FP8_V_SCALE, mcl, ws, P, err_flag=err, stream=stream)
        else:
            ops.paged_attention_decode(out, qq, k, v, btt, cx, w.scale, mcl, ws, P, err_flag=err,
                                       stream=stream)

    fused = args.step_api == "fused"

    def do_step(qq, btt, cx, kn, vn, sl, pr):
        """The whole step in one call of the fused entry point."""
        if fp8:
            ops.paged_decode_step_fp8(out, qq, k, v, btt, cx, w.scale,
                                      ks_dev if per_head else FP8_K_SCALE,
                                      vs_dev if per_head else FP8_V_SCALE, mcl, ws, k_new=kn,
                                      v_new=vn, slot_mapping=sl, block_pairs=pr,
                                      partition_size=P, err_flag=err, stream=stream)
        else:
            ops.paged_decode_step(out, qq, k, v, btt, cx, w.scale, mcl, ws, k_new=kn, v_new=vn,
                                  slot_mapping=sl, block_pairs=pr, partition_size=P,
                                  err_flag=err, stream=stream)

    def step():
        if fused:
            do_step(q, bt, ctx, k_new, v_new, slots, pairs)
            return
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
        nvtx.range_push("timed decode steps")
        for i in range(args.steps):
            if flush:
                scratch()
            e0, e1, e2 = ev[i]
            nvtx.range_push(f"step {i}")
            e0.record(stream)
            if fused:
                # one call: e1 = e0, the "attention" time is the whole step's
                e1.record(stream)
                nvtx.range_push("paged_decode_step")
                do_step(q, bt, ctx, k_new, v_new, slots, pairs)
                nvtx.range_pop()
            else:
                if pairs.numel():
                    do_copy(pairs)
                do_write(k_new, v_new, slots)
                e1.record(stream)
                nvtx.range_push("paged_attention_decode")
                do_attn(q, bt, ctx)
                nvtx.range_pop()
            e2.record(stream)
            nvtx.range_pop()
        nvtx.range_pop()
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
    # The step's inputs sit in one pinned host buffer, each at a 256-byte aligned offset,
    # and cross in one copy; the output comes back in one copy.
    srcs = (("q", q), ("k_new", k_new), ("v_new", v_new), ("slots", slots), ("pairs", pairs),
            ("bt", bt), ("ctx", ctx))
    offs, off = {}, 0
    for name, t in srcs:
        nb = t.numel() * t.element_size()
        offs[name] = (off, nb)
        off += (nb + 255) & ~255
    h_in = torch.empty(max(off, 256), dtype=torch.uint8).pin_memory()
    d_in = torch.empty(h_in.numel(), dtype=torch.uint8, device=dev)
    dv = {}
    for name, t in srcs:
        o, nb = offs[name]
        h_in[o:o + nb].copy_(t.contiguous().reshape(-1).view(torch.uint8).cpu())
        dv[name] = d_in[o:o + nb].view(t.dtype).view(t.shape)
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = h_in.numel()
    d2h = out.numel() * out.element_size()

    def e2e_step():
        d_in.copy_(h_in, non_blocking=True)
        if fused:
            do_step(dv["q"], dv["bt"], dv["ctx"], dv["k_new"], dv["v_new"], dv["slots"],
                    dv["pairs"])
        else:
            if dv["pairs"].numel():
                do_copy(dv["pairs"])
            do_write(dv["k_new"], dv["v_new"], dv["slots"])
            do_attn(dv["q"], dv["bt"], dv["ctx"])
        out_h.copy_(out, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    e2e_ms = 0.0
    for _ in range(args.steps):
        if flush:
            scratch()
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
            "workload": w.name, "kv_dtype": args.kv_dtype,
            **({"seed": args.seed} if args.seed is not None else {}),
            **({"fp8_scales": "one per KV head (amax / 448)" if per_head else "one per cache"}
               if fp8 else {}),
            "num_seqs": S, "num_q_heads": Hq, "num_kv_heads": Hkv,
            "head_dim": D, "block_size": w.block_size,
            "partition_size": P if P else "auto (512-4096 tokens, chosen per call on the device)",
            **({"partition_chosen": int(ws[4:8].view(torch.int32).item())} if not P else {}),
            "num_blocks": w.num_blocks, "mean_context": float(w.context_lens.mean()),
            "max_context": mcl, "kv_bytes_per_step": kv_bytes,
            "unique_kv_bytes_per_step": unique_kv,
            "cow_pairs_per_step": int(w.cow_pairs.shape[0]),
            "new_tokens_per_step": int(w.slot_mapping.shape[0]),
            "l2": ("L2 flushed (256 MB write, then 256 MB read) before every timed step"
                   if flush else
                   "inputs larger than L2 (KV read per step >> 129 MB)"),
            "attention_variant": args.variant, "attention_kernel": vname,
            "step_api": ("paged_decode_step (one call)" if fused else
                         "paged_block_copy + paged_kv_write + paged_attention_decode"),
            "parallelism": "replicas" if world > 1 else "single"},
        "pct_of_hbm_peak": 100.0 * value / peak,
        "seq_steps_per_s_per_layer": world * S / (ms_per_step / 1e3),
        "attention_ms": attn_avg_ms,
        "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms / args.steps},
        "gpu_launches": launches_per_step * args.steps,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak,
                     # captured on the default draw of each workload only
                     "traffic": (recorded_traffic(w.name, vname + ("-step" if fused else ""))
                                 if args.seed is None else None),
                     "kernel": ("paged_decode_step: prologue (copies + write + plan) + "
                                "partition (%s) + merge kernels, timed over the whole step"
                                if fused else
                                "paged_attention_decode: plan + partition (%s) + merge kernels")
                               % vname,
                     "peak_source": f"{peak_kind} hbm_gbs"},
        "clocks": clk.summary(),
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, fp8=fp8, ks=KS, vs=VS)
        try:  # the output of the last timed step against the oracle
            line["parity"] = sample_parity(w, out, fp8, KS, VS)
        except Exception as e:  # reported, never fatal to the measurement line
            line["parity"] = {"error": f"{type(e).__name__}: {e}"}
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


def prefill_sample_parity(w, out, n_rows: int = 128, nthreads: int | None = None) -> dict:
    """The bench's own prefill output against the oracle on sampled (token, head) rows: the
    last token of every chunk plus random rows (cache = the pre-step cache with the
    step's write applied; re-applying it to a cache that holds it changes nothing)."""
    import oracle
    nthreads = nthreads or os.cpu_count() or 1
    k_host, v_host = prefill_host_caches(w)
    rng = np.random.default_rng(11)
    rows = [(int(w.query_start[s + 1]) - 1, int(rng.integers(w.num_q_heads)))
            for s in range(w.num_seqs) if w.query_start[s + 1] > w.query_start[s]]
    while len(rows) < n_rows:
        rows.append((int(rng.integers(w.num_tokens)), int(rng.integers(w.num_q_heads))))
    sel = np.array(rows, dtype=np.int32)
    ref = oracle.attention_prefill(w.q.cpu(), k_host, v_host, w.block_tables, w.context_lens,
                                   w.query_start, w.scale, sel=sel, nthreads=nthreads)
    idx_t = torch.as_tensor(sel[:, 0].astype(np.int64), device=out.device)
    idx_h = torch.as_tensor(sel[:, 1].astype(np.int64), device=out.device)
    got = out[idx_t, idx_h].float().cpu().double().numpy()
    err = np.abs(got - ref)
    bad = int(np.count_nonzero(~(err <= 1e-2 + 1e-2 * np.abs(ref))))
    return {"rows": int(sel.shape[0]), "max_abs_err": float(err.max()),
            "mean_abs_err": float(err.mean()), "elements_out_of_tolerance": bad,
            "within_tolerance": bool(bad == 0 and err.mean() <= 2e-3),
            "tolerance": "|err| <= 1e-2 + 1e-2 |ref| per element, mean |err| <= 2e-3",
            "reference": "fp64 oracle on (token, head) rows: the last token of every chunk "
                         "plus random rows"}


def run_prefill_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = workloads.make_prefill_config(args.config, device="cpu", seed=args.seed)
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
    pk = {"auto": ops.PKV_PREFILL_AUTO, "mma": ops.PKV_PREFILL_MMA,
          "tc": ops.PKV_PREFILL_TC, "tc_pair": ops.PKV_PREFILL_TC_PAIR,
          "tc_2sm": ops.PKV_PREFILL_TC_2SM, "tc_sep": ops.PKV_PREFILL_TC_SEP}[args.prefill_kernel]
    ops.set_prefill_variant(pk)
    w = workloads.make_prefill_config(args.config, device="cuda", seed=args.seed)
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
    scratch = L2Flush(dev) if flush else None

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
        nvtx.range_push("timed prefill steps")
        for i in range(args.steps):
            if flush:
                scratch()
            e0, e1, e2 = ev[i]
            nvtx.range_push(f"step {i}")
            e0.record(stream)
            do_write(k_new, v_new, slots)
            e1.record(stream)
            nvtx.range_push("paged_attention_prefill")
            do_attn(q, bt, ctx, qs)
            nvtx.range_pop()
            e2.record(stream)
            nvtx.range_pop()
        nvtx.range_pop()
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
            scratch()
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
    # AUTO runs the separate-P tcgen05 kernel (head_dim 64 and 128)
    kname = {ops.PKV_PREFILL_TC_PAIR: "prefill-tc-pair", ops.PKV_PREFILL_MMA: "prefill-mma",
             ops.PKV_PREFILL_TC_2SM: "prefill-tc-2sm", ops.PKV_PREFILL_TC: "prefill-tc",
             ops.PKV_PREFILL_TC_SEP: "prefill-tc-sep"}.get(pk, "prefill-tc-sep")
    line = {
        "metric": PREFILL_METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {
            "workload": w.name, **({"seed": args.seed} if args.seed is not None else {}),
            "num_seqs": w.num_seqs, "new_tokens_per_step": T,
            "max_query_len": w.max_query_len, "num_q_heads": Hq, "num_kv_heads": Hkv,
            "head_dim": D, "block_size": w.block_size, "num_blocks": w.num_blocks,
            "mean_context": float(w.context_lens.mean()), "max_context": w.max_context_len,
            "flops_per_step": flops, "kv_bytes_per_step": kv_bytes,
            "prefill_kernel": kname,
            "l2": ("L2 flushed (256 MB write, then 256 MB read) before every timed step"
                   if flush else
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
                     "traffic": (recorded_traffic(w.name, kname, PREFILL_SOURCES)
                                 if args.seed is None else None),
                     "kernel": {"prefill-tc": "paged_attention_prefill: prefill_tc_kernel "
                                              "(tcgen05.mma, TMEM accumulators)",
                                "prefill-tc-pair": "paged_attention_prefill: "
                                                   "prefill_tc_pair_kernel (tcgen05.mma, two "
                                                   "query tiles per CTA sharing K/V tiles)",
                                "prefill-tc-sep": "paged_attention_prefill: "
                                                  "prefill_tcs_kernel (tcgen05.mma, one S "
                                                  "buffer, P and half of Q in TMEM)",
                                "prefill-tc-2sm": "paged_attention_prefill: "
                                                  "prefill_tc2sm_kernel (tcgen05.mma "
                                                  "cta_group::2, SM pairs)",
                                "prefill-mma": "paged_attention_prefill: prefill_kernel "
                                               "(mma.sync)"}[kname],
                     "peak_source": f"{peak_kind} bf16_tflops (burst)"},
        "clocks": clk.summary(),
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = prefill_cpu_baseline(w)
        try:  # the output of the last timed step against the oracle
            line["parity"] = prefill_sample_parity(w, out)
        except Exception as e:  # reported, never fatal to the measurement line
            line["parity"] = {"error": f"{type(e).__name__}: {e}"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# -------------------------------------------------------------------------------------
# Continuous-batching serving run (scheduler + prefix cache + all kernels)
# -------------------------------------------------------------------------------------
SERVE_METRIC = "continuous-batching serving throughput, output tokens/s (paged KV, Llama-3-70B attention shapes)"
SERVE_CONFIGS = {
    1: dict(name="serve-pareto-1024req-gqa8", kind="pareto", n=1024, cache=None),
    2: dict(name="serve-shared-prefix-1000req-gqa8", kind="shared-prefix", n=1000, cache=4096),
}
SERVE_SHAPE = dict(Hq=64, Hkv=8, D=128, max_num_seqs=128, budget=2048)


def serve_setup(cfg, static=False, n=None, device="cuda"):
    from paged_kv_cache_272_gb300.block_pool import BlockPool
    from paged_kv_cache_272_gb300.driver import ServingDriver
    from paged_kv_cache_272_gb300.serving import PrefixCache, Scheduler
    reqs = workloads.make_requests(cfg["kind"], seed=3000, n=cfg["n"] if n is None else n)
    sh = SERVE_SHAPE
    max_ctx = max(len(r.prompt) + r.output_len for r in reqs)
    blocks = sh["max_num_seqs"] * ((max_ctx + 15) // 16) + (cfg["cache"] or 0)
    pool = BlockPool(blocks)
    cache = PrefixCache(pool, cfg["cache"]) if cfg["cache"] else None
    sched = Scheduler(pool, sh["max_num_seqs"], sh["budget"], static=static, cache=cache)
    drv = ServingDriver(sched, blocks, sh["Hq"], sh["Hkv"], sh["D"], max_ctx, seed=7,
                        device=device)
    for r in reqs:
        drv.add_request(r.rid, r.prompt, r.output_len)
    return reqs, pool, cache, sched, drv


def serve_run(drv, stream, decode_bytes_per_token):
    """Run the stream to completion, one native call per step (pkv_engine_step: the
    scheduler step, its plan packed into pinned staging, the copy in, the fused decode
    step, the prefill and the copy out).  Every step's outputs are read back to the host (what a
    sampler would read: every decode row, the last row of every prefill chunk); the host
    keeps two steps in flight -- it plans and queues step k + 1 (staging and output
    buffers of the other slot) before it waits for step k's outputs, since the
    scheduler's decisions do not depend on the sampled values.  Returns timing and
    counts."""
    tot = dict(dev_ms=0.0, dec_ms=0.0, dec_bytes=0, steps=0, outs=0)

    def retire(item):
        pk, slot, b_prev, b, dev_pair = item
        b.synchronize()  # this step's outputs are on the host
        tot["steps"] += 1
        tot["outs"] += pk.outputs
        tot["dev_ms"] += b_prev.elapsed_time(b)
        nd = pk.num_decode
        if nd and dev_pair is not None:
            tot["dec_ms"] += dev_pair[0].elapsed_time(dev_pair[1])
            ctx = drv.f_np[slot][:nd]
            tot["dec_bytes"] += int(ctx.sum(dtype=np.int64)) * decode_bytes_per_token

    # Timing events, reused: a set is free again once its step has retired.  A step's
    # device time runs from its first copy to its last (GPU idle time between steps is
    # not counted).  The decode attention is timed on every 4th step (events cost host
    # time on every step they are recorded); the roofline uses those steps' bytes and
    # times.  The native step call records them (handles passed as a ctypes array).
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(4)]
    ev_dec = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    for e in [x for pair in ev for x in pair] + list(ev_dec):
        e.record(stream)  # creates the event, so that its handle exists
    stream.synchronize()
    handles = [(ctypes.c_void_p * 3)(ev[k][0].cuda_event,
                                      ev_dec[0].cuda_event if k == 0 else None,
                                      ev_dec[1].cuda_event if k == 0 else None)
               for k in range(4)]
    t0 = time.perf_counter()
    slot, pending, k = 0, [], 0
    while not drv.done():
        # the step that used this slot has retired
        pk, _, _ = drv.engine_step(slot, handles[k % 4])
        if pk.num_tokens == 0:  # nothing computed this step
            continue
        a, b = ev[k % 4]
        b.record(stream)
        pending.append((pk, slot, a, b, ev_dec if k % 4 == 0 else None))
        k += 1
        slot ^= 1
        if len(pending) == 2:
            retire(pending.pop(0))
    while pending:
        retire(pending.pop(0))
    wall = time.perf_counter() - t0
    return dict(wall_s=wall, device_ms=tot["dev_ms"], decode_ms=tot["dec_ms"],
                decode_bytes=tot["dec_bytes"], steps=tot["steps"], output_tokens=tot["outs"])


def serve_cpu_baseline(cfg, budget_s=12.0):
    """The oracle (plain-Python scheduler on the reference block manager and prefix
    trie, fp64 C attention) on the host cores over the first steps of the same stream."""
    import oracle
    from oracle.block_manager import BlockManager
    from oracle.prefix_trie import PrefixTrie
    from oracle.scheduler import Scheduler as RefScheduler
    from paged_kv_cache_272_gb300 import driver as drvmod
    sh = SERVE_SHAPE
    reqs = workloads.make_requests(cfg["kind"], seed=3000, n=cfg["n"])
    max_ctx = max(len(r.prompt) + r.output_len for r in reqs)
    blocks = sh["max_num_seqs"] * ((max_ctx + 15) // 16) + (cfg["cache"] or 0)
    bm = BlockManager(blocks)
    cache = PrefixTrie(bm, cfg["cache"]) if cfg["cache"] else None
    sch = RefScheduler(bm, sh["max_num_seqs"], sh["budget"], cache=cache)
    prompts = {}
    for r in reqs:
        prompts[r.rid] = r.prompt
        sch.add_request(r.rid, r.prompt.tolist(), r.output_len)
    g = torch.Generator().manual_seed(7)
    bf = lambda *s_: torch.randn(*s_, generator=g).to(torch.bfloat16)
    rows = 4096
    k_tab, v_tab, q_tab = bf(rows, sh["Hkv"], sh["D"]), bf(rows, sh["Hkv"], sh["D"]), bf(rows, sh["Hq"], sh["D"])
    u16 = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
    kh = np.zeros((blocks, sh["Hkv"], 16, sh["D"]), np.uint16)
    vh = np.zeros_like(kh)
    nthreads = os.cpu_count() or 1
    t0 = time.perf_counter()
    steps = outs = 0
    while not sch.done() and time.perf_counter() - t0 < budget_s:
        pl = sch.step()
        if not pl.seqs:
            continue
        n = len(pl.seqs)
        MB = max(len(bm.tables[r]) for r in pl.seqs)
        tables, _ = bm.export(pl.seqs, MB)
        qst = np.concatenate([[0], np.cumsum(pl.query_lens)]).astype(np.int32)
        from paged_kv_cache_272_gb300.serving import Plan
        plan = Plan(seq_ids=np.array(pl.seqs, np.int64), num_decode=pl.num_decode,
                    query_lens=np.array(pl.query_lens, np.int32),
                    context_lens=np.array(pl.context_lens, np.int32), query_start=qst,
                    slot_mapping=np.array(pl.slots, np.int64),
                    block_tables=np.array(tables, np.int32),
                    cow_pairs=np.array(pl.cow_pairs, np.int32).reshape(-1, 2),
                    finished=pl.finished, preempted=pl.preempted, running=0, waiting=0)
        x = drvmod.prepare(plan, prompts, rows, rows)
        if plan.cow_pairs.size:
            oracle.block_copy(kh, vh, plan.cow_pairs)
        idx = torch.from_numpy(x.kv_rows)
        oracle.kv_write(kh, vh, u16(k_tab[idx]), u16(v_tab[idx]), plan.slot_mapping)
        q = u16(q_tab[torch.from_numpy(x.q_rows)])
        nd = plan.num_decode
        if nd:
            oracle.attention(q[:nd], kh, vh, plan.block_tables[:nd], plan.context_lens[:nd],
                             sh["D"] ** -0.5, nthreads=nthreads)
        if n > nd:
            oracle.attention_prefill(q[nd:], kh, vh, plan.block_tables[nd:],
                                     plan.context_lens[nd:], x.prefill_query_start,
                                     sh["D"] ** -0.5, nthreads=nthreads)
        steps += 1
        outs += nd + sum(1 for i in range(nd, n)
                         if plan.context_lens[i] == len(prompts[int(plan.seq_ids[i])]))
    dt = time.perf_counter() - t0
    return {"value": outs / dt, "unit": "output tokens/s", "cores": nthreads, "kind": "oracle",
            "sample": f"first {steps} scheduler steps of the stream ({outs} output tokens); "
                      "plain-Python scheduler, fp64 C attention with OpenMP",
            "seconds": dt, "steps": steps}


def run_serve_reference(args):
    if int(os.environ.get("RANK", "0")) != 0:
        return
    cfg = SERVE_CONFIGS[args.config]
    r = serve_cpu_baseline(cfg, budget_s=max(3.0, 1.0 * (args.steps + args.warmup)))
    line = {"impl": "reference", "metric": SERVE_METRIC, "value": r["value"],
            "unit": "output tokens/s", "n_gpus": args.gpus, "steps": r["steps"],
            "warmup": 0, "ms_per_step": r["seconds"] / max(1, r["steps"]) * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": cfg["name"]},
            "cpu_baseline": {k: r[k] for k in ("value", "unit", "cores", "kind", "sample")},
            "e2e": {"value": r["value"], "unit": "output tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_serve(args):
    world, rank, local = setup_dist(args.gpus)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    cfg = SERVE_CONFIGS[args.config]
    sh = SERVE_SHAPE
    stream = torch.cuda.current_stream(dev)
    per_tok = 2 * sh["Hkv"] * sh["D"] * 2
    # warm-up: the first requests of the stream, run to completion
    for _ in range(max(1, args.warmup)):
        _, _, _, _, drv = serve_setup(cfg, n=64, device=dev)
        serve_run(drv, stream, per_tok)
    with ClockSampler(local) as clk:
        barrier(world)
        reqs, pool, cache, sched, drv = serve_setup(cfg, device=dev)
        res = serve_run(drv, stream, per_tok)
        barrier(world)
    if int(drv.err.item()) != 0:
        raise RuntimeError(f"device error flag {int(drv.err.item())}")
    st = sched.stats()
    cs = cache.stats() if cache is not None else None
    _, _, _, ssched, sdrv = serve_setup(cfg, static=True, device=dev)
    sres = serve_run(sdrv, stream, per_tok)
    dev_s = max_over_ranks(res["device_ms"], world) / 1e3
    wall = max_over_ranks(res["wall_s"], world)
    outs = res["output_tokens"]
    peaks, peak_kind = measured_peaks()
    peak = float(peaks["hbm_gbs"])
    achieved = res["decode_bytes"] / (res["decode_ms"] / 1e3) / 1e9 if res["decode_ms"] else 0.0
    line = {
        "metric": SERVE_METRIC, "value": world * outs / dev_s, "unit": "output tokens/s",
        "n_gpus": world, "steps": res["steps"], "warmup": args.warmup,
        "ms_per_step": res["device_ms"] / res["steps"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": cfg["name"], "requests": len(reqs),
                   "max_num_seqs": sh["max_num_seqs"], "max_batched_tokens": sh["budget"],
                   "num_q_heads": sh["Hq"], "num_kv_heads": sh["Hkv"], "head_dim": sh["D"],
                   "num_blocks": pool.num_blocks,
                   "prefix_cache_entries": cfg["cache"],
                   "output_tokens": outs,
                   "l2": "per-step working sets are the live KV of the batch; no flush (a "
                         "serving loop runs back to back)",
                   "parallelism": "replicas" if world > 1 else "single"},
        "e2e": {"value": world * outs / wall, "unit": "output tokens/s",
                "h2d_bytes_per_step": drv.h2d_bytes / res["steps"],
                "d2h_bytes_per_step": drv.d2h_bytes / res["steps"],
                "wall_s": wall, "note": "whole loop: host scheduler, pinned copies in and "
                                        "out, kernels; the host waits for every step's "
                                        "outputs with at most two steps in flight"},
        "gpu_launches": drv.launches,
        "value_note": "value: output tokens over the device time of the steps (copies in, "
                      "kernels, copies out); e2e: over the wall time of the whole loop",
        "utilisation": {"fill_all_steps": st["fill_sum"] / st["steps"],
                        "fill_while_queued": (st["busy_fill_sum"] / st["busy_steps"]
                                              if st["busy_steps"] else None),
                        "kv_waste": st["slots_unused"] / max(1, st["slots_held"]),
                        "preemptions": st["preemptions"]},
        "static_batching": {"e2e_output_tokens_per_s": sres["output_tokens"] / sres["wall_s"],
                            "device_output_tokens_per_s": sres["output_tokens"] / (sres["device_ms"] / 1e3),
                            "steps": sres["steps"],
                            "fill_all_steps": ssched.stats()["fill_sum"] / ssched.stats()["steps"]},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": None,
                     "kernel": "paged_attention_decode inside the serving loop (algorithmic KV "
                               "bytes of the decode entries / decode attention time)",
                     "peak_source": f"{peak_kind} hbm_gbs"},
        "clocks": clk.summary(),
    }
    if cs is not None:
        line["prefix_cache"] = {"request_hit_rate": cs["hits"] / max(1, cs["lookups"]),
                                "token_hit_rate": cs["matched_tokens"] / max(1, cs["query_tokens"]),
                                **cs}
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = serve_cpu_baseline(cfg)
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
    ap.add_argument("--path", default="decode", choices=["decode", "prefill", "serve"],
                    help="decode step (default), chunked-prefill step, or a whole "
                         "continuous-batching serving run")
    ap.add_argument("--config", type=int, default=None, choices=[1, 2, 3, 4, 5],
                    help="workload number (decode 1..5, default 5; prefill 1..4, default 2; "
                         "serve 1..2, default 2)")
    ap.add_argument("--variant", default="auto", choices=["auto", "fma", "mma"])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--partition", type=int, default=None,
                    help="split-K partition size in tokens (default: automatic, chosen per "
                         "call from the context lengths)")
    ap.add_argument("--seed", type=int, default=None,
                    help="draw the decode or prefill workload with this seed instead of its "
                         "default (1000 + config, 2000 + config); the recorded DRAM traffic "
                         "is then not reported")
    ap.add_argument("--kv-dtype", default="bf16", choices=["bf16", "fp8"],
                    help="KV cache element type: bf16, or fp8 (E4M3 codes with one scale each)")
    ap.add_argument("--fp8-scales", default="cache", choices=["cache", "head"],
                    help="with --kv-dtype fp8: one E4M3 scale per cache, or one per KV head")
    ap.add_argument("--prefill-kernel", default="auto",
                    choices=["auto", "mma", "tc", "tc_sep", "tc_pair", "tc_2sm"],
                    help="chunked-prefill kernel: tcgen05 variants (tc_sep, tc, tc_pair, "
                         "tc_2sm) or mma.sync (mma); auto = tc_sep")
    ap.add_argument("--step-api", default="fused", choices=["fused", "separate"],
                    help="decode step through paged_decode_step (one call, default) or the "
                         "three separate calls (copy, write, attention)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.config is None:
        args.config = DEFAULT_CONFIG[args.path]
    if args.path == "serve":
        if args.config not in SERVE_CONFIGS:
            ap.error("--path serve takes --config 1..2")
        (run_serve_reference if args.impl == "reference" else run_serve)(args)
    elif args.path == "prefill":
        if args.config not in workloads.PREFILL_CONFIG_NAMES:
            ap.error("--path prefill takes --config 1..4")
        (run_prefill_reference if args.impl == "reference" else run_prefill)(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
