"""Benchmark of the fused attention forward on GB300.

Default workload: B=2, H=16, N=8192, d=128, bf16, causal (the long-sequence headline case).
One step = one fa_fwd call over the whole batch. Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl gb300|reference]

* value: attention-forward TFLOP/s, FLOPs = 4*B*H*N^2*d (halved when causal), inputs resident
  in HBM, kernel time from CUDA events on the launching stream, L2 flushed (256 MiB write)
  before every timed step.
* e2e: the same metric through the user API with host buffers: pinned host -> device copies of
  Q, K, V, the kernel, and device -> host copies of O and LSE inside every timed step.
* roofline: tensor-bound; achieved = metric FLOPs per launch / mean launch time, peak = the
  measured dense bf16 matmul rate of this GPU type (burst), frac = achieved / peak.
* cpu_baseline: the fp64 oracle timed on this host's cores on a bounded sample of the same
  workload (uniformly sampled query rows), in the same unit.
* --gpus N > 1 (under torchrun): N independent replicas, one per GPU, no collective on the
  data path; value = all FLOPs / max-over-ranks time ("weak" scaling).
* --impl reference: the oracle, timed on the host cores (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from io_aware_attention_fa2_gb300.inputs import WORKLOADS, make_workload, sample_rows  # noqa

DEFAULT_WORKLOAD = "n8k_d128_causal"
FALLBACK_BF16_TFLOPS = 1900.0
L2_FLUSH_BYTES = 256 << 20
# --check auto compares every element with the oracle up to this many metric FLOPs (the plain
# fp64 oracle takes about a minute per 1e12 on 16 host cores), sampled rows above it.
FULL_CHECK_MAX_FLOPS = 1.2e12
WARM_L2_MAX_BYTES = 64 << 20   # workloads this small are also timed without the flush
# The sources each pass's dominant kernel is built from: a committed DRAM-traffic record is
# only reported while their hash is the one the record was taken on.
KERNEL_SOURCES = {
    "fwd": ["io_aware_attention_fa2_gb300/csrc/fa_fwd_kernel.cu",
            "io_aware_attention_fa2_gb300/csrc/ptx_sm103.cuh",
            "io_aware_attention_fa2_gb300/csrc/fa_internal.h"],
    "bwd": ["io_aware_attention_fa2_gb300/csrc/fa_bwd_kernel.cu",
            "io_aware_attention_fa2_gb300/csrc/ptx_sm103.cuh",
            "io_aware_attention_fa2_gb300/csrc/fa_internal.h"],
}


def allowed_pairs(w) -> int:
    """Exact number of (b, h, query, key) pairs the workload's masks allow: key j is visible
    to the query at position p (= i + Nk - Nq) when j < len_b, j <= p (causal),
    p - left <= j (left >= 0) and j <= p + right (right >= 0)."""
    nq, nk = w.N, w.n_keys
    pos = np.arange(nq, dtype=np.int64) + (nk - nq)
    total = 0
    for b in range(w.B):
        hi = np.full(nq, w.seqlens_k[b] if w.seqlens_k else nk, dtype=np.int64)
        if w.causal:
            hi = np.minimum(hi, pos + 1)
        if w.window[1] >= 0:
            hi = np.minimum(hi, pos + w.window[1] + 1)
        lo = np.maximum(0, pos - w.window[0]) if w.window[0] >= 0 else np.zeros(nq, np.int64)
        total += int(np.maximum(hi - lo, 0).sum())
    return total * w.H


def metric_name(w, bwd: bool) -> str:
    """The JSON line's metric; the same string on both arms for the same workload."""
    if bwd:
        return "attn bwd TFLOP/s (2.5x the forward's FLOPs)"
    if w.name == DEFAULT_WORKLOAD:
        return "attn fwd TFLOP/s (causal N=8K d=128 headline)"
    return "attn fwd TFLOP/s"


def metric_flops(w) -> float:
    """4*B*H*N^2*d (halved when causal) for Nq = Nk; with fewer queries than keys, 4*B*H*d per
    visible (query, key) pair (causal: query i sees i + Nk - Nq + 1 keys); with a padding or
    window mask, 4*d per allowed pair, counted exactly."""
    if w.masked:
        return 4.0 * w.d * allowed_pairs(w)
    if not w.Nk:
        f = 4.0 * w.B * w.H * w.N * w.N * w.d
        return f / 2 if w.causal else f
    nq, nk = w.N, w.Nk
    pairs = nq * (nk - nq) + nq * (nq + 1) / 2 if w.causal else nq * nk
    return 4.0 * w.B * w.H * w.d * pairs


def algorithmic_bytes(w) -> int:
    """Q, K, V read once, O written once (2 bytes each), LSE written once (4 bytes)."""
    nk = w.n_keys
    return (2 * w.N + 2 * nk) * w.B * w.H * w.d * 2 + w.B * w.H * w.N * 4


def memory_bound(w, bwd: bool = False) -> bool:
    """Decoding-style workloads (a few queries per head) are bound by reading K and V. The
    backward does 2.5 times the forward's FLOPs on about twice its bytes (Q, K, V, O, dO read;
    dQ, dK, dV written), so it is compared on that ratio."""
    if bwd:
        return 2.5 * metric_flops(w) / (2 * algorithmic_bytes(w)) < 275.0
    return metric_flops(w) / algorithmic_bytes(w) < 275.0


def kernel_source_hash(kind: str = "fwd") -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kind]:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


FALLBACK_HBM_GBS = 6800.0


def measured_peaks():
    """(bf16 TFLOP/s burst, bf16 TFLOP/s sustained, HBM GB/s, source)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return (float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", 0)),
                float(p.get("hbm_gbs", FALLBACK_HBM_GBS)), "measured")
    except (OSError, KeyError, ValueError):
        return FALLBACK_BF16_TFLOPS, 0.0, FALLBACK_HBM_GBS, "fallback"


def traffic_record(workload: str, kind: str = "fwd"):
    """DRAM bytes per launch of the pass's dominant kernel from the committed ncu summary, if
    taken on the current kernel sources."""
    path = os.path.join(ROOT, "profiles", "fa_%s_%s_dram.txt" % (kind, workload))
    try:
        rec = {}
        with open(path) as f:
            for line in f:
                if "=" in line and not line.startswith("#"):
                    key, val = line.split("=", 1)
                    rec[key.strip()] = val.strip()
        if rec.get("kernel_source_hash") != kernel_source_hash(kind):
            return None
        return int(float(rec["dram_bytes_per_launch"]))
    except (OSError, KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.out = None

    def __enter__(self):
        try:
            self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.out, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.out is None:
            return None
        self.out.flush()
        with open(self.out.name) as f:
            rows = [r.split(",") for r in f.read().strip().splitlines() if r.count(",") >= 8]
        os.unlink(self.out.name)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        smax = max(float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit())
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4)
                          if r[5 + i].strip().lower() == "active"})
        loaded = [s for s in sm if s > 0.5 * smax] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None, "sm_max_mhz": smax,
                "reasons": reasons, "samples": len(rows)}


def bench_config(w, world: int) -> dict:
    """The JSON line's ``config``: the same keys and values on both arms for one workload."""
    return {"workload": w.name, "shape": w.describe(),
            "l2": "256 MiB flush write before every timed step; per-step CUDA events around "
                  "the kernel only",
            "parallelism": "replicas x%d" % world}


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(values, world: int, device=None):
    """Each timing (ms) replaced by its maximum over the ranks of the default process group
    (the slowest rank sets the job's time); unchanged when world == 1."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def job_tflops(world: int, flops_per_rank_step: float, steps: int, max_ms: float) -> float:
    """Whole-job throughput: the FLOPs all ranks processed in `steps` steps over the slowest
    rank's time for them (each rank runs its own replica of the workload)."""
    return world * flops_per_rank_step * steps / (max_ms * 1e-3) / 1e12


class OracleSampler:
    """Times the oracle on uniformly sampled query rows of a workload (bounded CPU work)."""

    def __init__(self, w, qb, kb, vb):
        import oracle
        self.oracle = oracle
        self.lib = oracle.load()
        self.w, self.qb, self.kb, self.vb = w, qb, kb, vb
        self.total_rows = w.B * w.H * w.N
        self.rng = np.random.Generator(np.random.PCG64(w.seed + 11))
        self.rows_per_s = None
        self.fixed_s = 0.0

    def pick(self, n):
        w = self.w
        flat = self.rng.choice(self.total_rows, size=min(n, self.total_rows), replace=False)
        return np.stack([flat // (w.N * w.H), (flat // w.N) % w.H, flat % w.N], axis=1)

    def run(self, n_rows):
        """(metric FLOPs of the sampled rows, seconds, rows)."""
        w = self.w
        rows = self.pick(n_rows)
        t0 = time.perf_counter()
        self.oracle.attention_rows(self.qb, self.kb, self.vb, rows, w.causal, w.scale,
                                   dtype=w.dtype, lib=self.lib, window=w.window,
                                   seqlens_k=list(w.seqlens_k) or None)
        dt = time.perf_counter() - t0
        return metric_flops(w) * (len(rows) / self.total_rows), dt, len(rows)

    def rows_for(self, seconds, min_rows=16):
        """Rows that take about `seconds` in one call. Every call first decodes the inputs (a
        cost independent of the rows), so the rate is taken from two calls of different sizes
        and that cost is set apart."""
        if self.rows_per_s is None:
            _, dt1, n1 = self.run(64)
            _, dt2, n2 = self.run(512)
            per_row = (dt2 - dt1) / max(n2 - n1, 1)
            if per_row <= 0:
                per_row = dt2 / max(n2, 1)
            self.fixed_s = max(dt1 - n1 * per_row, 0.0)
            self.rows_per_s = 1.0 / max(per_row, 1e-9)
        budget = max(seconds - self.fixed_s, 0.0)
        return int(min(self.total_rows, max(min_rows, self.rows_per_s * budget)))

    def cores(self):
        return self.oracle.max_threads(self.lib)


def cpu_baseline(w, qb, kb, vb, target_s: float = 15.0):
    s = OracleSampler(w, qb, kb, vb)
    flops, dt, n = s.run(s.rows_for(target_s))
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": s.cores(),
            "kind": "oracle",
            "sample": "%d uniformly sampled query rows of %d (%.2f%%) in %.1f s; FLOPs pro "
                      "rata of the workload's metric FLOPs" %
                      (n, s.total_rows, 100.0 * n / s.total_rows, dt)}


def run_reference(args, w):
    """The oracle as it stands, timed on the host cores: every step is a bounded sample of the
    workload (uniform query rows), sized so that warm-up + timed steps take about
    --ref-total-seconds altogether."""
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    qb, kb, vb = make_workload(w)
    s = OracleSampler(w, qb, kb, vb)
    per_step = args.ref_total_seconds / (args.steps + args.warmup)
    n_rows = s.rows_for(per_step)
    for _ in range(args.warmup):
        s.run(n_rows)
    flops = secs = 0.0
    for _ in range(args.steps):
        f, dt, n = s.run(n_rows)
        flops += f
        secs += dt
    value = flops / secs / 1e12
    sample = ("%d uniformly sampled query rows of %d per step (%.3f%% of the workload); FLOPs "
              "pro rata of the workload's metric FLOPs" % (n, s.total_rows,
                                                           100.0 * n / s.total_rows))
    line = {
        "impl": "reference", "metric": metric_name(w, False), "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * secs / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": bench_config(w, world),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": s.cores(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# Standard attention's HBM accesses for one head, in the order "FlashAttention V2 核心原理与架构设计"
# §1.1 lists them: Q and K read, S = QK^T written, S read, P = softmax(S) written, P and V read,
# O = PV written.
STANDARD_ATTENTION_HBM_ACCESSES = ("read Q", "read K", "write S", "read S", "write P", "read P",
                                   "read V", "write O")


def score_matrix_bytes(n: int, elem_bytes: int) -> int:
    """Bytes of one N x N attention score (or probability) matrix."""
    return n * n * elem_bytes


def standard_attention_hbm_bytes(n: int, d: int, elem_bytes: int) -> int:
    """HBM bytes of the accesses above for one head: the N x d operands once each, the N x N
    matrices S and P each written and read once."""
    sizes = {"Q": n * d, "K": n * d, "V": n * d, "O": n * d, "S": n * n, "P": n * n}
    return sum(sizes[a.split()[1]] for a in STANDARD_ATTENTION_HBM_ACCESSES) * elem_bytes


def standard_scores(qh, kh, scale, fp32_scores: bool):
    """S = scale * Q K^T for [B, H, N, d] operands, materialised: in fp32 (the products
    accumulated and kept in fp32, the same precision the fused kernel's S has) or rounded to
    the 16-bit input type. Returns (S, how the fp32 scores were made or None)."""
    import torch
    if not fp32_scores:
        return torch.matmul(qh, kh.transpose(-1, -2)) * scale, None
    b, h, n, d = qh.shape
    q3, k3 = qh.reshape(b * h, n, d), kh.reshape(b * h, -1, d)
    try:
        s = torch.bmm(q3, k3.transpose(1, 2), out_dtype=torch.float32)
        how = "16-bit matmul with fp32 output"
    except (TypeError, RuntimeError):
        # 16-bit values are exact in TF32, and TF32 products accumulate in fp32
        prev = torch.backends.cuda.matmul.allow_tf32
        torch.backends.cuda.matmul.allow_tf32 = True
        try:
            s = torch.bmm(q3.float(), k3.float().transpose(1, 2))
        finally:
            torch.backends.cuda.matmul.allow_tf32 = prev
        how = "TF32 matmul of the 16-bit values (exact inputs, fp32 accumulation)"
    return s.view(b, h, n, -1).mul_(scale), how


def time_standard_attention(q, k, v, w, steps, flush, stream, fp32_scores=True):
    """The standard three-step attention (S = QK^T, P = softmax(S), O = PV, with S and P
    written to and read back from HBM), in PyTorch on the same device: the comparison the pages
    make against the fused kernel. With ``fp32_scores`` S and the softmax are fp32 and P is
    rounded to the input type for P V (the fused kernel's precision); otherwise S and P are
    both in the 16-bit input type. Times `steps` calls with the same L2 flush and per-step CUDA
    events; returns (mean ms, O in [B, N, H, d], how the scores were computed)."""
    import torch
    qh, kh, vh = (t.permute(0, 2, 1, 3).contiguous() for t in (q, k, v))   # [B, H, N, d]
    mask = None
    if w.causal:
        mask = torch.ones(w.N, w.N, dtype=torch.bool, device=q.device).triu_(1)
    how = [None]

    def step():
        s, how[0] = standard_scores(qh, kh, w.scale, fp32_scores)
        if mask is not None:
            s.masked_fill_(mask, float("-inf"))
        p = torch.softmax(s, dim=-1).to(q.dtype)
        return torch.matmul(p, vh)

    for _ in range(2):
        step()
    times = []
    out = None
    for _ in range(steps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        out = step()
        b.record(stream)
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b))
    return statistics.mean(times), out.permute(0, 2, 1, 3), how[0] or "16-bit matmul"


def check_forward(w, qb, kb, vb, o, lse, mode, with_abs_v=False):
    """Parity of a forward's O and LSE (device tensors; ``lse`` None for an output without
    one) with the fp64 oracle under the bar of ``oracle.tolerance``: every element (mode
    "full") or sampled rows of every head; ``with_abs_v`` also has the oracle compute the
    attention of |V| for the bar's rounding term (without it the bar is stricter)."""
    import torch

    import oracle
    from oracle.tolerance import magnitude_bits, stats
    lens = list(w.seqlens_k) or None
    kw = dict(dtype=w.dtype, window=w.window, seqlens_k=lens)
    a_ref = None
    if mode == "full":
        og = o.cpu().float().double().numpy()
        o_ref, l_ref = oracle.attention(qb, kb, vb, w.causal, w.scale, **kw)
        if with_abs_v:
            a_ref, _ = oracle.attention(qb, kb, magnitude_bits(vb), w.causal, w.scale, **kw)
        lg = l_ref if lse is None else lse.cpu().double().numpy()
        out = {"mode": "full", **stats(og, lg, o_ref, l_ref, w.dtype, a_ref)}
    else:
        rows = sample_rows(w.B, w.H, w.N, 8, seed=w.seed + 5)
        o_ref, l_ref = oracle.attention_rows(qb, kb, vb, rows, w.causal, w.scale, **kw)
        if with_abs_v:
            a_ref, _ = oracle.attention_rows(qb, kb, magnitude_bits(vb), rows, w.causal,
                                             w.scale, **kw)
        idx = [torch.from_numpy(rows[:, c]).to(o.device) for c in range(3)]
        og = o[idx[0], idx[2], idx[1]].double().cpu().numpy()
        lg = l_ref if lse is None else lse[idx[0], idx[1], idx[2]].double().cpu().numpy()
        out = {"mode": "sample", "rows": int(len(rows)),
               **stats(og, lg, o_ref, l_ref, w.dtype, a_ref)}
    out["abs_v_term"] = bool(with_abs_v)
    if lse is None:
        del out["max_abs_lse"]
    return out


def run_gpu(args, w):
    import torch
    import torch.distributed as dist

    from io_aware_attention_fa2_gb300 import binding
    from io_aware_attention_fa2_gb300 import build as fa_build

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0:
        fa_build.build()
    if world > 1:
        dist.barrier()   # the other ranks load what rank 0 built
    binding.load_library()

    qb, kb, vb = make_workload(w)
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float16
    host = [torch.from_numpy(x.view(np.int16)).view(tdt).pin_memory() for x in (qb, kb, vb)]
    q, k, v = (t.to(dev) for t in host)
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    # Fewer queries than keys: the split-K/V forward, its workspace allocated up front.
    num_splits = binding.splitkv_num_splits(w.B, w.H, w.N, w.n_keys) if w.Nk else 1
    workspace = None
    if w.Nk and num_splits > 1:
        workspace = torch.empty(binding.splitkv_workspace_size(w.B, w.H, w.N, w.d, num_splits),
                                dtype=torch.uint8, device=dev)

    # parity against the fp64 oracle before timing (rank 0): every element, or sampled rows
    parity = None
    lens_host = (torch.tensor(w.seqlens_k, dtype=torch.int32).pin_memory() if w.seqlens_k
                 else None)
    lens_dev = lens_host.to(dev) if w.seqlens_k else None

    def call():
        if w.Nk:
            binding.fa_fwd_splitkv(q, k, v, o, lse, w.causal, w.scale, num_splits, workspace,
                                   stream)
        else:
            binding.fa_fwd(q, k, v, o, lse, w.causal, w.scale, stream, window=w.window,
                           seqlens_k=lens_dev)

    check = args.check
    if check == "auto":
        check = "full" if metric_flops(w) <= FULL_CHECK_MAX_FLOPS else "sample"
    if rank == 0 and check != "none":
        call()
        if binding.device_error(stream) != 0:
            raise RuntimeError("kernel wait timed out")
        parity = check_forward(w, qb, kb, vb, o, lse, check)
        if not parity["ok"]:
            print(json.dumps({"error": "parity failed", "parity": parity}), flush=True)
            return 3

    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def step():
        call()

    bwd = args.pass_ == "bwd"
    if bwd:
        # O and LSE from the forward (outside the timed region), a seeded upstream gradient,
        # one workspace: each timed step is one fa_bwd call (three kernels).
        from io_aware_attention_fa2_gb300.inputs import normal, round_to_bits
        call()
        dob = round_to_bits(normal(qb.shape, w.seed + 9), w.dtype)
        host.append(torch.from_numpy(dob.view(np.int16)).view(tdt).pin_memory())
        dout = host[-1].to(dev)
        dq, dk, dv = (torch.empty_like(q) for _ in range(3))
        bwd_ws = torch.empty(binding.bwd_workspace_size(w.B, w.H, w.N, w.d), dtype=torch.uint8,
                             device=dev)

        def step():
            binding.fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, w.causal, w.scale, bwd_ws,
                           stream, w.window, lens_dev)

        if rank == 0 and check != "none":
            # parity of dQ, dK, dV on sampled positions of one head against the fp64 oracle
            import oracle
            step()
            if binding.device_error(stream) != 0:
                raise RuntimeError("kernel wait timed out")
            b0, h0 = w.B - 1, w.H // 2
            pos = np.unique(np.concatenate([
                [0, 1, 127, 128, w.N // 2, w.N - 1],
                np.random.default_rng(w.seed + 6).integers(0, w.N, 6)]))
            sq, sk, sv = oracle.attention_bwd_sampled(
                qb, kb, vb, dob, w.causal, w.scale, [(b0, h0)], pos, pos, dtype=w.dtype,
                window=w.window, seqlens_k=list(w.seqlens_k) if w.seqlens_k else None)
            from oracle.tolerance import dq_allowance_for, grad_stats
            allow = dq_allowance_for(qb, kb, vb, dob, w.causal, w.scale, w.dtype,
                                     [(b0, h0, i) for i in pos], w.window,
                                     list(w.seqlens_k) if w.seqlens_k else None)
            sel = torch.from_numpy(pos).to(dev)
            got = [t[b0, sel, h0].double().cpu().numpy() for t in (dq, dk, dv)]
            parity = {"forward": parity, "head": [int(b0), int(h0)],
                      "positions": int(len(pos))}
            bad = False
            for name, g, r in zip(("dq", "dk", "dv"), got, (sq[0], sk[0], sv[0])):
                st = grad_stats(g, r, w.dtype, name, allow if name == "dq" else None)
                parity["rel_l2_" + name] = st.get("rel_l2")
                parity["rel_max_" + name] = st.get("rel_max")
                bad |= not st["ok"]
            if bad:
                print(json.dumps({"error": "parity failed", "parity": parity}), flush=True)
                return 3

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(local) as clocks:
        # The warm-up steps run right before the timed ones, after the sampler has started: a
        # step that follows an idle GPU (the sampler's start-up) ran 2-20 % slower than the rest.
        for _ in range(args.warmup):
            flush.zero_()
            step()
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)
        t_wall = time.perf_counter()
        for i in range(args.steps):
            flush.zero_()
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
        t_wall = time.perf_counter() - t_wall
        if world > 1:
            dist.barrier()
    if binding.device_error(stream) != 0:
        raise RuntimeError("kernel wait timed out during timing")
    per_step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    kernel_ms = statistics.mean(per_step_ms)
    total_ms = sum(per_step_ms)

    # Workloads whose data fits in L2 are also timed warm (no flush between steps, so the
    # inputs stay in L2 from the previous step): a supplementary figure beside the flushed one.
    warm_ms = None
    if algorithmic_bytes(w) < WARM_L2_MAX_BYTES:
        for i in range(args.steps):
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
        if binding.device_error(stream) != 0:
            raise RuntimeError("kernel wait timed out during the warm-L2 timing")
        warm_ms = statistics.mean(s.elapsed_time(e) for s, e in zip(starts, ends))

    # end to end through the user API with host buffers (pinned), copies in the timed region
    o_host = torch.empty(q.shape, dtype=tdt, pin_memory=True)
    l_host = torch.empty((w.B, w.H, w.N), dtype=torch.float32, pin_memory=True)

    def e2e_step():
        binding.attention_forward(*host[:3], causal=w.causal, scale=w.scale, out=o_host,
                                  lse=l_host, stream=stream, device=dev, window=w.window,
                                  seqlens_k=lens_host)

    if bwd:
        o_pin = o.cpu().pin_memory()
        l_pin = lse.cpu().pin_memory()

        def e2e_step():
            binding.attention_backward(*host[:3], o_pin, host[3], l_pin, causal=w.causal,
                                       scale=w.scale, stream=stream, device=dev,
                                       window=w.window, seqlens_k=lens_host)

    for _ in range(max(1, args.warmup // 2)):
        e2e_step()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        e2e_step()
    torch.cuda.synchronize(dev)
    e2e_ms = 1e3 * (time.perf_counter() - t0) / args.steps

    flops = metric_flops(w) * (2.5 if bwd else 1.0)
    total_ms, e2e_ms = max_over_ranks([total_ms, e2e_ms], world, dev)
    ms_per_step = total_ms / args.steps
    value = job_tflops(world, flops, args.steps, total_ms)
    e2e_value = job_tflops(world, flops, 1, e2e_ms)

    if rank == 0:
        peak, peak_sus, hbm_peak, peak_src = measured_peaks()
        achieved = flops / (kernel_ms * 1e-3) / 1e12
        line = {
            "metric": metric_name(w, bwd),
            "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
            "config": bench_config(w, world),
            "pct_of_peak": 100.0 * achieved / peak,
            "peak_denominator": "%s bf16 dense %.1f TFLOP/s" % (peak_src, peak),
            "roofline": ({"bound": "tensor", "achieved": achieved, "peak": peak,
                          "unit": "TFLOP/s", "frac": achieved / peak,
                          "peak_source": "%s (burst)" % peak_src,
                          "traffic": traffic_record(w.name, "bwd" if bwd else "fwd"),
                          "algorithmic_bytes": algorithmic_bytes(w)}
                         if not memory_bound(w, bwd) else
                         {"bound": "hbm",
                          "achieved": algorithmic_bytes(w) / (kernel_ms * 1e-3) / 1e9,
                          "peak": hbm_peak, "unit": "GB/s",
                          "frac": algorithmic_bytes(w) / (kernel_ms * 1e-3) / 1e9 / hbm_peak,
                          "peak_source": "%s copy bandwidth" % peak_src,
                          "traffic": traffic_record(w.name),
                          "algorithmic_bytes": algorithmic_bytes(w)}),
            "num_splits": num_splits,
            "gpu_launches_per_step": 3 if bwd else 2 if num_splits > 1 else 1,
            "pass": "bwd" if bwd else "fwd",
            "e2e": {"value": e2e_value, "unit": "TFLOP/s",
                    "h2d_bytes_per_step": (sum(t.numel() * t.element_size() for t in host) +
                                           ((o.numel() * 2 + lse.numel() * 4) if bwd else
                                            (4 * len(w.seqlens_k)))),
                    "d2h_bytes_per_step": (3 * o.numel() * 2 if bwd else
                                           o_host.numel() * 2 + l_host.numel() * 4),
                    "ms_per_step": e2e_ms},
            "gpu_launches": args.steps * (3 if bwd else 2 if num_splits > 1 else 1),
            "kernel_ms": {"mean": kernel_ms, "min": min(per_step_ms),
                          "max": max(per_step_ms)},
            "wall_s_timed_region": t_wall,
            "clocks": clocks.summary(),
            "parity": parity,
        }
        if peak_sus and not memory_bound(w, bwd):
            line["roofline"]["frac_of_sustained"] = achieved / peak_sus
        if warm_ms is not None:
            line["warm_l2"] = {"ms_per_step": warm_ms, "value": flops / (warm_ms * 1e-3) / 1e12,
                               "unit": "TFLOP/s",
                               "what": "the same steps back to back without the L2 flush "
                                       "(inputs resident in L2); not the headline value"}
        if args.vs_standard and not w.Nk and not w.masked:
            # Standard attention twice: with fp32 scores (the fused kernel's precision; it must
            # meet the same parity bar, or no comparison is reported) and all in 16 bits (S
            # and P rounded to the input type: faster, and reported with its own parity).
            for key, fp32_scores in (("standard_attention", True),
                                     ("standard_attention_16bit", False)):
                std_ms, o_std, how = time_standard_attention(q, k, v, w, min(args.steps, 20),
                                                             flush, stream, fp32_scores)
                s_bytes = 4 if fp32_scores else 2
                std = {"ms": std_ms, "tflops": flops / (std_ms * 1e-3) / 1e12,
                       "fused_speedup": std_ms / kernel_ms, "scores": how,
                       "what": "PyTorch matmul -> softmax -> matmul, S and P materialised in "
                               "HBM, same L2 flush and CUDA-event timing",
                       "materialised_bytes": w.B * w.H * (score_matrix_bytes(w.N, s_bytes) +
                                                          score_matrix_bytes(w.N, 2)),
                       "hbm_bytes_model": w.B * w.H * standard_attention_hbm_bytes(w.N, w.d,
                                                                                   2),
                       "fused_algorithmic_bytes": algorithmic_bytes(w)}
                if check != "none":
                    std["parity"] = check_forward(w, qb, kb, vb, o_std.contiguous(), None,
                                                  check, with_abs_v=True)
                    if fp32_scores and not std["parity"]["ok"]:
                        print(json.dumps({"error": "standard attention parity failed",
                                          "parity": std["parity"]}), flush=True)
                        return 3
                del o_std
                line[key] = std
        if not args.no_cpu_baseline and world == 1 and not bwd:
            line["cpu_baseline"] = {k: v for k, v in
                                    cpu_baseline(w, qb, kb, vb, args.cpu_seconds).items()}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--check", default="auto", choices=["auto", "full", "sample", "none"],
                    help="parity against the fp64 oracle before timing: every element (full), "
                         "sampled rows of every head (sample), or none; auto = full up to "
                         "%.1e metric FLOPs" % FULL_CHECK_MAX_FLOPS)
    ap.add_argument("--no-check", action="store_true", help="same as --check none")
    ap.add_argument("--pass", dest="pass_", default="fwd", choices=["fwd", "bwd"],
                    help="time the forward (default) or the backward (dQ, dK, dV)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--vs-standard", action="store_true",
                    help="also time standard (materialised S, P) attention in PyTorch")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--ref-total-seconds", type=float, default=120.0)
    args = ap.parse_args()
    if args.no_check:
        args.check = "none"
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    w = WORKLOADS[args.workload]
    if args.pass_ == "bwd" and w.Nk:
        ap.error("the backward takes one length N (queries and keys)")
    if args.impl == "reference":
        if args.pass_ == "bwd":
            ap.error("the reference arm times the forward oracle only")
        return run_reference(args, w)
    return run_gpu(args, w)


if __name__ == "__main__":
    sys.exit(main())
