#!/usr/bin/env python
"""Benchmark of the batch-invariant LM-head log-prob library on GB300.

One step = one pass of the fused hot path over one batch: the fused forward
(vocab projection + online log-softmax + label gather + entropy, lse kept)
followed by the fused backward (recomputed logits -> dlogits -> grad_hidden,
grad_weight). Workload: T=16384 tokens, H=3584, V=152064, inv_temperature =
1/0.7 (fp32), bf16 hidden ~ N(0,1), weight ~ N(0, 0.02^2), labels uniform,
upstream grad ~ N(0,1). Inputs (weight 1.09 GB) are larger than L2, so no L2
flush is needed between steps.

Prints ONE JSON line (rank 0). Besides the contract keys it carries:
  roofline       the dominant kernel of the step against the measured peak
  kernels        per-kernel average durations measured with CUDA events
  fwd_only       forward-only tokens/s of the same workload and of
                 T=4096 H=4096 V=32000
  logits_path    the sampler formula on bf16 logits [8192, 152064] vs HBM,
                 and its division (sampler-parity) form
  sampler_parity fp32-bit mismatch counts against torch's fp32 sampler
                 formula on [4096, 152064] logits
  next_rows      the entropy-gradient step and the sum_pi_squared variants of
                 the forward and of the logits path, on the same workloads
  vocab_shards_fwd  the forward as two vocab shards plus the merge (what a
                 vocab-parallel rank pair runs), on one GPU
  cpu_baseline   the fp64 CPU oracle timed on a bounded sample on host cores
  e2e            the same step from pinned host inputs: the host-staged
                 forward (copies overlapped with the forward) and the
                 backward, log-probs/entropy copied back every step

Multi-GPU (torchrun): every rank runs its own replica of the workload on its
own GPU (weak scaling, no data-path collective); the step time is the max over
ranks and `value` sums the tokens of all ranks.

--impl reference times the fp64 CPU oracle (the reference arm)
on host cores, on a bounded row sample of the same workload per step.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "tokens/s fused LM-head logprob fwd & fwd+bwd; % bf16 tensor peak / % HBM"
WORKLOAD = "fused forward+backward T=16384 H=3584 V=152064 inv_T=1/0.7 (bf16 in, fp32 accumulate)"
T_, H_, V_ = 16384, 3584, 152064
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
GEMM_KINDS = ("fused_fwd_gemm", "dlogits_gemm", "grad_hidden_gemm", "grad_weight_gemm")


def n_fwd_chunks(V: int) -> int:
    """1024-column vocabulary chunks of the forward's partials."""
    return (V + 1023) // 1024


def inv_temperature() -> float:
    import numpy as np

    return float(np.float32(1.0 / 0.7))


# ----------------------------------------------------------------------------- helpers
def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "of measured"
    return dict(FALLBACK_PEAKS), "of fallback"


def sources_sha(paths) -> str | None:
    """sha256 prefix of the named repository files, concatenated in order."""
    h = hashlib.sha256()
    for rel in paths:
        full = os.path.join(ROOT, rel)
        if not os.path.exists(full):
            return None
        with open(full, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_for(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, or None when a
    source file that shapes the kernel's memory traffic has changed since the
    counters were taken."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    k = d.get("kernels", {}).get(kernel)
    if not k:
        return None
    files = k.get("source_files") or []
    if not files or sources_sha(files) != k.get("source_sha"):
        return None
    return k.get("dram_bytes_per_full_launch")


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""

    FIELDS = ("index,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="lmh_clocks_", suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 10:
                    continue
                if self.uuid and parts[1] != self.uuid:
                    continue
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        mhz = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        mx = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[6 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(mhz) if mhz else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max(x: float, ws: int, device) -> float:
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws: int):
    if ws > 1:
        import torch.distributed as dist

        dist.barrier()


def aggregate_tokens_per_s(tokens_per_rank: int, world: int, steps: int, max_ms: float) -> float:
    """Whole-job throughput: tokens of all ranks over the slowest rank's time."""
    return tokens_per_rank * world * steps / (max_ms / 1e3)


# ----------------------------------------------------------------------------- oracle legs
_SAMPLE_CACHE = {}


def oracle_sample(n_rows: int):
    """The first n_rows rows of the workload's seeded CPU inputs (full H and V)."""
    import workloads as W

    wl = W.QWEN
    if "full" not in _SAMPLE_CACHE or _SAMPLE_CACHE["full"][0].shape[0] < n_rows:
        inp = W.fused_inputs(wl, T=max(n_rows, 256))
        _SAMPLE_CACHE["full"] = (W.bf16_bits_to_f32(inp["hidden"]), W.bf16_bits_to_f32(inp["weight"]),
                                 inp["labels"], inp["grad"])
    h, w, lab, g = _SAMPLE_CACHE["full"]
    return h[:n_rows], w, lab[:n_rows], g[:n_rows], wl.inv_temperature


def oracle_step(sample):
    import oracle

    h, w, lab, g, s = sample
    oracle.fused_forward(h, w, lab, s)
    oracle.fused_backward(h, w, lab, g, s)


def cpu_model() -> str:
    """The host CPU as /proc/cpuinfo names it: the model name where the kernel
    gives one (x86), else the architecture with the Arm implementer and part
    numbers of the first core."""
    import platform

    fields = {}
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if ":" in line:
                    k, v = (x.strip() for x in line.split(":", 1))
                    fields.setdefault(k, v)
    except OSError:
        pass
    if fields.get("model name"):
        return fields["model name"]
    if "CPU implementer" in fields:
        return (f"{platform.machine()} (implementer {fields['CPU implementer']}, "
                f"part {fields.get('CPU part', '?')})")
    return platform.machine() or "unknown"


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def cpu_baseline(target_s: float = 15.0, rows: int = 128):
    """fp64 oracle fwd+bwd on a row sample of the workload (full H and V),
    repeated until about target_s seconds of CPU work have been timed."""
    sample = oracle_sample(rows)
    oracle_step(sample)  # warm-up (page-in, thread pools)
    n = 0
    t0 = time.perf_counter()
    while True:
        oracle_step(sample)
        n += 1
        dt = time.perf_counter() - t0
        if dt >= target_s or n >= 50:
            break
    return {"value": rows * n / dt, "unit": "tokens/s", "cores": cpu_cores(), "cpu": cpu_model(),
            "kind": "oracle",
            "sample": f"{rows} rows of the workload (full H={H_}, V={V_}), fp64 forward+backward "
                      f"incl. grad_weight over the sampled rows, repeated {n}x in {dt:.1f} s"}


def cpu_oracle_logits(target_s: float = 3.0, rows: int = 64, divide: bool = False):
    """fp64 oracle of the sampler formula (or its division form) on a row
    sample of the logits workload, repeated for about target_s seconds."""
    import oracle
    import workloads as W

    inp = W.logits_inputs(W.LOGITS, T=rows)
    x = W.bf16_bits_to_f32(inp["logits"])
    lab = inp["labels"]

    def step():
        if divide:
            oracle.logprob_from_logits_div(x, lab, 0.7)
        else:
            oracle.logprob_from_logits(x, lab, 1.0)

    step()
    n = 0
    t0 = time.perf_counter()
    while True:
        step()
        n += 1
        dt = time.perf_counter() - t0
        if dt >= target_s or n >= 100:
            break
    return {"value": rows * n / dt, "unit": "tokens/s", "cores": cpu_cores(), "cpu": cpu_model(),
            "kind": "oracle",
            "sample": f"{rows} rows of the logits workload (V={W.LOGITS.V}), fp64, "
                      f"repeated {n}x in {dt:.1f} s"}


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    probe = oracle_sample(4)
    t0 = time.perf_counter()
    oracle_step(probe)
    per_step_4 = time.perf_counter() - t0
    budget = 150.0 / max(1, args.steps + args.warmup)
    rows = int(max(1, min(64, 4 * budget / max(per_step_4, 1e-3))))
    sample = oracle_sample(rows)
    for _ in range(args.warmup):
        oracle_step(sample)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(sample)
    dt = time.perf_counter() - t0
    value = rows * args.steps / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "T": T_, "H": H_, "V": V_,
                   "inv_temperature": inv_temperature(),
                   "sample_rows_per_step": rows, "l2": "host run; not applicable"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cpu_cores(),
                         "cpu": cpu_model(), "kind": "oracle",
                         "sample": f"{rows} rows per step of the workload (full H, V), fp64 "
                                   f"forward+backward"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- GPU arm
def make_inputs(T, H, V, seed, dev):
    import torch

    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    hidden = torch.randn(T, H, generator=g, device=dev).to(torch.bfloat16)
    weight = (torch.randn(V, H, generator=g, device=dev) * 0.02).to(torch.bfloat16)
    labels = torch.randint(0, V, (T,), generator=g, device=dev, dtype=torch.int32)
    grad = torch.randn(T, generator=g, device=dev)
    return hidden, weight, labels, grad


def invariance_cases(run, T, subs, window=1024, shifts=(1, 63, 127), seeds=(11, 12, 13),
                     embed=4096, dev=None):
    """Bit-mismatch counts of a row-wise result under re-batching. run(rows)
    computes it on exactly these rows (an index tensor, in that order) and
    returns its per-row outputs; each case is compared with the whole batch's
    rows, in fp32 or bf16 bits. The cases: sub-batches ((size, starts) pairs),
    windows of `window` rows shifted by 1..127, shuffled packings of the
    whole batch, and the batch as the first T rows of a larger one (rows on
    `dev`, the current CUDA device by default)."""
    import torch

    def bits(t):
        return t.view(torch.int32) if t.dtype == torch.float32 else t.view(torch.int16)

    if dev is None:
        dev = torch.device("cuda", torch.cuda.current_device())
    full = [x.clone() for x in run(torch.arange(T, device=dev))]
    out = {"rows_compared": 0, "mismatched_values": 0, "cases": []}

    def compare(rows, part):
        n = sum(int((bits(a[:rows.numel()]) != bits(b[rows])).sum().item())
                for a, b in zip(part, full))
        out["rows_compared"] += int(rows.numel())
        out["mismatched_values"] += n
        return n

    for bs, starts in subs:
        for r0 in starts:
            rows = torch.arange(r0, r0 + bs, device=dev)
            out["cases"].append({"batch": bs, "start": r0, "mismatched": compare(rows, run(rows))})
    for shift in shifts:
        rows = torch.arange(shift, min(T, shift + window), device=dev)
        out["cases"].append({"batch": int(rows.numel()), "shift": shift,
                             "mismatched": compare(rows, run(rows))})
    for seed in seeds:
        perm = torch.randperm(T, generator=torch.Generator().manual_seed(seed)).to(dev)
        out["cases"].append({"batch": T, "shuffled": seed, "mismatched": compare(perm, run(perm))})
    if embed:
        rows = torch.arange(T, device=dev)
        bigger = torch.cat([rows, torch.arange(0, min(T, embed), device=dev)])
        out["cases"].append({"batch": int(bigger.numel()), "embedded_rows": T,
                             "mismatched": compare(rows, run(bigger))})
    return out


def invariance_counts(lmh, hidden, weight, labels, s, lp, ent, lse):
    """The fused forward's invariance cases on the main workload."""
    T = hidden.shape[0]

    def run(rows):
        return lmh.lmhead_logprob_fwd(hidden[rows].contiguous(), weight, labels[rows].contiguous(),
                                      s, want_lse=True)

    return invariance_cases(run, T, ((1, (0, 1, T - 1)), (7, (0, 4093)), (256, (0, 8000))))


def packed_invariance(run, lengths, seeds=(21, 22, 23), alone=(0, 7, 31), dev=None):
    """Bit-mismatch counts of a row-wise result on a packed batch of
    sequences: the sequences re-packed in shuffled orders, and single
    sequences run alone, each compared with the original packing's rows."""
    import torch

    def bits(t):
        return t.view(torch.int32) if t.dtype == torch.float32 else t.view(torch.int16)

    if dev is None:
        dev = torch.device("cuda", torch.cuda.current_device())
    offs = [0]
    for n in lengths:
        offs.append(offs[-1] + int(n))
    T = offs[-1]
    full = [x.clone() for x in run(torch.arange(T, device=dev))]
    out = {"rows_compared": 0, "mismatched_values": 0, "cases": []}

    def compare(rows, part):
        n = sum(int((bits(a) != bits(b[rows])).sum().item()) for a, b in zip(part, full))
        out["rows_compared"] += int(rows.numel())
        out["mismatched_values"] += n
        return n

    for seed in seeds:
        order = torch.randperm(len(lengths), generator=torch.Generator().manual_seed(seed)).tolist()
        rows = torch.cat([torch.arange(offs[i], offs[i + 1], device=dev) for i in order])
        out["cases"].append({"sequences_shuffled": seed, "mismatched": compare(rows, run(rows))})
    for i in alone:
        rows = torch.arange(offs[i], offs[i + 1], device=dev)
        out["cases"].append({"sequence_alone": i, "rows": int(rows.numel()),
                             "mismatched": compare(rows, run(rows))})
    return out


def sampler_parity(lmh, x, lab):
    """Row counts whose fp32 log-prob bits differ from torch's fp32 sampler
    formula on the GPU (log_softmax of the fp32 logits divided by the
    temperature, then gather), for the pages' 4096 x 152064 comparison: their
    two unfused branches, and this library's multiplied and divided forms."""
    import numpy as np
    import torch

    T = x.shape[0]
    idx = lab.long()[:, None]

    def sampler(t):
        temps = torch.full((T,), t, dtype=torch.float32, device=x.device)
        return torch.log_softmax(x.float() / temps[:, None], dim=-1).gather(1, idx)[:, 0]

    def count(a, b):
        return {"mismatched_rows": int((a.view(torch.int32) != b.view(torch.int32)).sum()),
                "max_abs": float((a.double() - b.double()).abs().max())}

    ref1 = sampler(1.0)
    out = {"rows": T, "vocab": x.shape[1], "reference": "torch fp32 log_softmax(logits / t).gather",
           "t=1": {
               "torch_bf16_log_softmax": count(
                   torch.log_softmax(x, dim=-1).gather(1, idx)[:, 0].float(), ref1),
               "torch_gather_minus_logsumexp": count(
                   x.float().gather(1, idx)[:, 0] - torch.logsumexp(x.float(), dim=-1), ref1),
               "logprob_from_logits": count(lmh.logprob_from_logits(x, lab, 1.0)[0], ref1),
               "logprob_from_logits_div": count(lmh.logprob_from_logits_div(x, lab, 1.0)[0],
                                                ref1)}}
    ref7 = sampler(0.7)
    out["t=0.7"] = {
        "logprob_from_logits (s = fp32(1/0.7))": count(
            lmh.logprob_from_logits(x, lab, float(np.float32(1.0 / 0.7)))[0], ref7),
        "logprob_from_logits_div": count(lmh.logprob_from_logits_div(x, lab, 0.7)[0], ref7)}
    torch.cuda.synchronize()
    return out


def kernel_ms(lmh, fn, steps, warmup, names):
    """Average per-call device time of the named library kernels (CUDA events
    recorded by the library on the launching stream), excluding host gaps."""
    import torch

    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    lmh.lmhead_timing_enable(True)
    for _ in range(steps):
        fn()
    recs = lmh.lmhead_timing_read()
    lmh.lmhead_timing_enable(False)
    return sum(ms for n, ms in recs if n in names) / steps


def kernel_breakdown(lmh, fn, steps, warmup):
    """Average device time per call of each library kernel kind (CUDA events
    recorded by the library on the launching stream)."""
    import torch

    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    lmh.lmhead_timing_enable(True)
    for _ in range(steps):
        fn()
    recs = lmh.lmhead_timing_read()
    lmh.lmhead_timing_enable(False)
    per = {}
    for name, ms in recs:
        per[name] = per.get(name, 0.0) + ms / steps
    return per


def peak_mem(workspace_bytes: int):
    """Device memory of a leg: torch's peak allocation since the last reset
    (every buffer of the leg, the library's workspace included; the library
    itself allocates nothing) and the workspace handed to the library."""
    import torch

    return {"max_memory_allocated_gb": round(torch.cuda.max_memory_allocated() / 1e9, 3),
            "library_workspace_gb": round(workspace_bytes / 1e9, 3)}


def bwd_roofline_ms(T, H, V, peaks):
    """Per-kernel lower bounds of the backward of T rows (T <= 16384): each
    GEMM at max(its 2THV flops at the burst bf16 peak, its algorithmic bytes at
    the HBM peak), the transpose at HBM speed."""
    flop_ms = 2.0 * T * H * V / (peaks["bf16_tflops"] * 1e12) * 1e3

    def hbm(b):
        return b / (peaks["hbm_gbs"] * 1e9) * 1e3

    return {
        # read W and hidden, write bf16 dl
        "dlogits_gemm": max(flop_ms, hbm(2.0 * V * H + 2.0 * T * H + 2.0 * T * V)),
        # read dl and W, write bf16 grad_hidden
        "grad_hidden_gemm": max(flop_ms, hbm(2.0 * T * V + 2.0 * V * H + 2.0 * T * H)),
        "hidden_transpose": hbm(4.0 * T * H),
        # read the two fp32 partials of grad_hidden, write it in bf16
        "grad_hidden_sum": hbm(10.0 * T * H),
        # read hidden^T and dl, write fp32 grad_weight
        "grad_weight_gemm": max(flop_ms, hbm(2.0 * T * H + 2.0 * T * V + 4.0 * V * H)),
    }


def bwd_joint_roofline_ms(T, H, V, peaks):
    """Lower bound of the whole backward of T rows when its kernels may run
    side by side: the three GEMMs' 6THV flops at the burst bf16 peak, or the
    three GEMMs' algorithmic bytes at the HBM peak, whichever is longer."""
    flop_ms = 6.0 * T * H * V / (peaks["bf16_tflops"] * 1e12) * 1e3
    nbytes = ((2.0 * V * H + 2.0 * T * H + 2.0 * T * V)      # dlogits: W, hidden in; dl out
              + (2.0 * T * V + 2.0 * V * H + 2.0 * T * H)    # grad_hidden: dl, W in; bf16 out
              + (2.0 * T * H + 2.0 * T * V + 4.0 * V * H))   # grad_weight: fp32 out
    return max(flop_ms, nbytes / (peaks["hbm_gbs"] * 1e9) * 1e3)


def timed_steps(fn, steps, warmup):
    """Mean ms per call over `steps` calls (total time / steps, as timed()),
    and each call's own ms: an event on the current stream after every call."""
    import torch

    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    evs[0].record()
    for i in range(steps):
        fn()
        evs[i + 1].record()
    torch.cuda.synchronize()
    per = [evs[i].elapsed_time(evs[i + 1]) for i in range(steps)]
    return evs[0].elapsed_time(evs[-1]) / steps, per


def timed(fn, steps, warmup):
    import torch

    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(steps):
        fn()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / steps


def run_gpu(args):
    import torch

    import invariant_lm_head_gb300 as lmh

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    lmh.build()
    lmh.library()
    peaks, peak_src = load_peaks()
    s = inv_temperature()

    T, H, V = T_, H_, V_
    hidden, weight, labels, grad = make_inputs(T, H, V, 1234 + rank, dev)
    lp = torch.empty(T, device=dev)
    ent = torch.empty(T, device=dev)
    lse = torch.empty(T, device=dev)
    gh = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    gw = torch.empty(V, H, dtype=torch.float32, device=dev)
    ws_f = torch.empty(lmh.lmhead_workspace_size(lmh.LMH_OP_FWD, T, H, V), dtype=torch.uint8,
                       device=dev)
    ws_b = torch.empty(lmh.lmhead_workspace_size(lmh.LMH_OP_BWD, T, H, V), dtype=torch.uint8,
                       device=dev)

    def fwd():
        lmh.lmhead_logprob_fwd(hidden, weight, labels, s, out_logprob=lp, out_entropy=ent,
                               out_lse=lse, workspace=ws_f)

    def bwd():
        lmh.lmhead_logprob_bwd(hidden, weight, labels, grad, s, lse=lse, grad_hidden=gh,
                               grad_weight=gw, workspace=ws_b)

    torch.cuda.reset_peak_memory_stats(dev)
    for _ in range(args.warmup):
        fwd()
        bwd()
    torch.cuda.synchronize()
    lmh.lmhead_device_status()
    main_mem = peak_mem(ws_f.numel() + ws_b.numel())

    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    clocks = ClockSampler(uuid)
    clocks.start()
    time.sleep(0.3)
    launches0 = lmh.lmhead_kernel_launches()
    lmh.lmhead_timing_enable(True)
    barrier(ws)
    torch.cuda.synchronize()
    ev_start = torch.cuda.Event(enable_timing=True)
    ev_end = torch.cuda.Event(enable_timing=True)
    ev_start.record()
    for _ in range(args.steps):
        fwd()
        bwd()
    ev_end.record()
    torch.cuda.synchronize()
    barrier(ws)
    total_ms = ev_start.elapsed_time(ev_end)
    launches = lmh.lmhead_kernel_launches() - launches0
    recs = lmh.lmhead_timing_read()
    lmh.lmhead_timing_enable(False)
    clk = clocks.stop()
    lmh.lmhead_device_status()
    max_ms = reduce_max(total_ms, ws, dev)
    ms_per_step = max_ms / args.steps
    value = aggregate_tokens_per_s(T, ws, args.steps, max_ms)

    # per-kernel durations (CUDA events on the launching stream, timed region)
    per = {}
    for name, ms in recs:
        per.setdefault(name, []).append(ms)
    kernels = {k: {"launches": len(v), "avg_ms": sum(v) / len(v), "total_ms": sum(v)}
               for k, v in per.items()}
    rows_per_chunk = 16384
    flops_per_launch = {
        "fused_fwd_gemm": 2.0 * T * H * V,
        "dlogits_gemm": 2.0 * min(T, rows_per_chunk) * H * V,
        "grad_hidden_gemm": 2.0 * min(T, rows_per_chunk) * H * V,
        "grad_weight_gemm": 2.0 * min(T, rows_per_chunk) * H * V,
    }
    bytes_per_launch = {  # HBM-bound helpers of the step
        "fwd_merge": (12.0 * n_fwd_chunks(V) + 20.0) * T,  # m, s, u; zl, label; 3 outputs
        "hidden_transpose": 4.0 * min(T, rows_per_chunk) * H,
        # the two K segments' fp32 partials of grad_hidden in, bf16 out
        "grad_hidden_sum": 10.0 * min(T, rows_per_chunk) * H,
    }
    for k, info in kernels.items():
        if k in flops_per_launch:
            info["tflops"] = flops_per_launch[k] / (info["avg_ms"] * 1e-3) / 1e12
        if k in bytes_per_launch:
            info["gbs"] = bytes_per_launch[k] / (info["avg_ms"] * 1e-3) / 1e9
    dominant = max(kernels, key=lambda k: kernels[k]["total_ms"]) if kernels else None
    peak = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"])
    roofline = None
    if dominant in flops_per_launch:
        ach = kernels[dominant]["tflops"]
        roofline = {"kernel": dominant, "bound": "tensor", "achieved": round(ach, 1),
                    "peak": peak, "unit": "TFLOP/s", "frac": round(ach / peak, 4),
                    "peak_source": f"bf16_tflops_sustained {peak_src} (kernel timed inside a "
                                   f"multi-kernel step)",
                    "traffic": traffic_for(dominant),
                    "algorithmic_flops_per_launch": flops_per_launch[dominant]}

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "T": T, "H": H, "V": V, "inv_temperature": s,
                   "parallelism": f"replicas x{ws} (rows per GPU fixed)",
                   "l2": "inputs larger than L2 (weight 1.09 GB); no flush"},
        "gpu_launches": launches, "roofline": roofline, "kernels": kernels, "clocks": clk,
        "peak_mem": main_mem,
        "model_tflops_per_gpu": 6.0 * T * H * V / (ms_per_step * 1e-3) / 1e12,
        # the whole step against the same sustained rate: 8THV flops as executed
        # (forward, recomputed logits, grad_hidden, grad_weight)
        "step_tensor": {"flops_per_step": 8.0 * T * H * V,
                        "achieved_tflops": round(8.0 * T * H * V / (ms_per_step * 1e-3) / 1e12, 1),
                        "peak": peak, "frac": round(8.0 * T * H * V / (ms_per_step * 1e-3) / 1e12
                                                    / peak, 4)},
    }

    # ------------------------------------------------------------- e2e (host buffers)
    # Timed right after the device-resident step, before any other leg, so
    # that both see the same clocks under the power cap.
    h_host = hidden.cpu().pin_memory()
    w_host = weight.cpu().pin_memory()
    l_host = labels.cpu().pin_memory()
    g_host = grad.cpu().pin_memory()
    lp_host = torch.empty(T, dtype=torch.float32).pin_memory()
    ent_host = torch.empty(T, dtype=torch.float32).pin_memory()

    def e2e_step():
        # host inputs in, host results out, through the library: the staged
        # forward overlaps the weight's host-to-device copy with the forward
        lmh.lmhead_logprob_fwd_host(h_host, w_host, l_host, s, hidden=hidden, weight=weight,
                                    labels=labels, out_logprob=lp, out_entropy=ent, out_lse=lse,
                                    out_logprob_host=lp_host, out_entropy_host=ent_host,
                                    workspace=ws_f)
        grad.copy_(g_host, non_blocking=True)
        bwd()

    # the host-to-device copy rate these inputs see (pinned memory, one stream)
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    weight.copy_(w_host, non_blocking=True)
    c0.record()
    weight.copy_(w_host, non_blocking=True)
    c1.record()
    torch.cuda.synchronize()
    h2d_gbs = w_host.numel() * 2 / (c0.elapsed_time(c1) * 1e-3) / 1e9
    barrier(ws)
    e2e_mean, e2e_per = timed_steps(e2e_step, args.steps, 2)
    e2e_ms = reduce_max(e2e_mean * args.steps, ws, dev)
    e2e_sorted = sorted(e2e_per)
    h2d = sum(t.numel() * t.element_size() for t in (h_host, w_host, l_host, g_host))
    line["e2e"] = {"value": aggregate_tokens_per_s(T, ws, args.steps, e2e_ms), "unit": "tokens/s",
                   "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": 2 * T * 4,
                   "path": "lmhead_logprob_fwd_host (pinned host inputs, copies overlapped with "
                           "the forward) + lmhead_logprob_bwd; logprob and entropy to host",
                   "h2d_copy_gbs": round(h2d_gbs, 1),
                   # this rank's steps one by one (events after every step): the host-staged
                   # copies make single steps vary more than the device-resident ones
                   "ms_per_step_min_median_max": [round(e2e_sorted[0], 3),
                                                  round(e2e_sorted[len(e2e_sorted) // 2], 3),
                                                  round(e2e_sorted[-1], 3)]}
    del h_host, w_host

    # ------------------------------------------------- batch invariance (bit mismatches)
    # Forward outputs of the full batch against the same rows run as
    # sub-batches of 1, 7 and 256 rows, shifted by 1..127 rows, in three
    # shuffled packings and inside a larger batch; counted in fp32 bits
    # (target 0). The backward's grad_hidden rows the same way, in bf16 bits
    # (grad_weight sums over the batch's rows, so it has no per-row bits).
    if not args.no_extras:
        line["invariance"] = invariance_counts(lmh, hidden, weight, labels, s, lp, ent, lse)
        lse_full = lse.clone()

        def bwd_rows(rows):
            gh_r, _ = lmh.lmhead_logprob_bwd(hidden[rows].contiguous(), weight,
                                             labels[rows].contiguous(), grad[rows].contiguous(), s,
                                             lse=lse_full[rows].contiguous())
            return (gh_r,)

        line["invariance_grad_hidden"] = invariance_cases(
            bwd_rows, T, ((1, (0, T - 1)), (7, (4093,)), (256, (8000,))))
        torch.cuda.empty_cache()

    if ws == 1 and not args.no_extras:
        # forward only, same workload
        fwd_kernels = ("fused_fwd_gemm", "fwd_merge")
        f_ms = timed(fwd, args.steps, 2)
        fk = kernel_ms(lmh, fwd, args.steps, 2, fwd_kernels)
        extras = {"fwd_only": {"T=16384 H=3584 V=152064": {
            "tokens_per_s": T / (f_ms * 1e-3), "ms_per_call": f_ms, "ms_kernels": fk,
            "tflops_kernels": 2.0 * T * H * V / (fk * 1e-3) / 1e12}}}
        # small batches of the same head: the forward then reads W (1.09 GB)
        # once per call and is bound by HBM, not by the tensor cores
        small = {}
        for Ts in (1, 64, 512):
            fs = lambda: lmh.lmhead_logprob_fwd(hidden[:Ts], weight, labels[:Ts], s,  # noqa: E731
                                                out_logprob=lp[:Ts], out_entropy=ent[:Ts],
                                                workspace=ws_f)
            ks = kernel_ms(lmh, fs, args.steps, 3, fwd_kernels)
            small[f"T={Ts}"] = {"ms_kernels": ks, "tokens_per_s": Ts / (ks * 1e-3),
                                "weight_gbs": V * H * 2 / (ks * 1e-3) / 1e9,
                                "weight_frac_of_hbm": V * H * 2 / (ks * 1e-3) / 1e9
                                / peaks["hbm_gbs"]}
        extras["fwd_only"]["small_batches H=3584 V=152064"] = small
        # the next rows on the same workload: the backward with an entropy
        # gradient, and the forward that also returns sum_pi_squared
        g_ent = torch.randn(T, generator=torch.Generator(device=dev).manual_seed(11), device=dev)

        def ent_step():
            lmh.lmhead_logprob_fwd(hidden, weight, labels, s, out_logprob=lp, out_entropy=ent,
                                   out_lse=lse, workspace=ws_f)
            lmh.lmhead_logprob_entropy_bwd(hidden, weight, labels, grad, g_ent, s, lse=lse,
                                           entropy=ent, grad_hidden=gh, grad_weight=gw,
                                           workspace=ws_b)

        step_kernels = ("fused_fwd_gemm", "fwd_merge", "dlogits_gemm", "grad_hidden_gemm",
                        "grad_hidden_sum", "hidden_transpose", "grad_weight_gemm")
        e_ms = kernel_ms(lmh, ent_step, args.steps, 2, step_kernels)
        q2 = torch.empty(T, device=dev)
        fq = lambda: lmh.lmhead_logprob_fwd_stats(hidden, weight, labels, s,  # noqa: E731
                                                  out_logprob=lp, out_entropy=ent, out_lse=lse,
                                                  out_sum_p2=q2, workspace=ws_f)
        q_ms = kernel_ms(lmh, fq, args.steps, 2, fwd_kernels)
        # vocab shards (two, cut at a 1024-column boundary) and the merge, as a
        # vocab-parallel rank pair would run them, on one GPU
        n_chunks = n_fwd_chunks(V)
        pm_ = torch.empty(n_chunks, T, device=dev)
        ps_, pu_ = torch.empty_like(pm_), torch.empty_like(pm_)
        zl_a, zl_b = torch.empty(T, device=dev), torch.empty(T, device=dev)
        cut = (n_chunks // 2) * 1024
        w_a, w_b = weight[:cut], weight[cut:]

        def sharded():
            lmh.lmhead_logprob_fwd_partials(hidden, w_a, labels, 0, s, part_m=pm_[:cut // 1024],
                                            part_s=ps_[:cut // 1024], part_u=pu_[:cut // 1024],
                                            label_logit=zl_a)
            lmh.lmhead_logprob_fwd_partials(hidden, w_b, labels, cut, s,
                                            part_m=pm_[cut // 1024:], part_s=ps_[cut // 1024:],
                                            part_u=pu_[cut // 1024:], label_logit=zl_b)
            zl_a.add_(zl_b)
            lmh.lmhead_logprob_merge(pm_, ps_, pu_, zl_a, labels, V, out_logprob=lp,
                                     out_entropy=ent, out_lse=lse)

        sh_ms = kernel_ms(lmh, sharded, args.steps, 2, fwd_kernels)
        extras["vocab_shards_fwd"] = {"shards": 2, "ms_kernels": sh_ms,
                                      "tflops": 2.0 * T * H * V / (sh_ms * 1e-3) / 1e12}
        extras["next_rows"] = {
            "entropy_grad_fwd_bwd": {"ms_kernels_per_step": e_ms, "tokens_per_s": T / (e_ms * 1e-3),
                                     "tflops_as_executed": 8.0 * T * H * V / (e_ms * 1e-3) / 1e12},
            "fwd_with_sum_p2": {"ms_kernels": q_ms, "tokens_per_s": T / (q_ms * 1e-3),
                                "tflops": 2.0 * T * H * V / (q_ms * 1e-3) / 1e12}}
        # the backward of short batches of the same head (the row counts of a
        # rollout's log-prob recompute and of training micro-batches), per kernel
        # against its roofline: each GEMM at max(2THV flops at the burst peak,
        # its algorithmic bytes at HBM speed). The call's own time (events
        # around the call on its stream) is held against the joint bound too,
        # max(all flops at the tensor peak, all bytes at HBM speed), which is
        # what kernels running side by side can approach.
        small_b = {}
        for Ts in (128, 512, 1024, 2048):
            lmh.lmhead_logprob_fwd(hidden[:Ts], weight, labels[:Ts], s, out_logprob=lp[:Ts],
                                   out_entropy=ent[:Ts], out_lse=lse[:Ts], workspace=ws_f)
            fb = lambda: lmh.lmhead_logprob_bwd(hidden[:Ts], weight, labels[:Ts],  # noqa: E731
                                                grad[:Ts], s, lse=lse[:Ts], grad_hidden=gh[:Ts],
                                                grad_weight=gw, workspace=ws_b)
            call_ms = timed(fb, args.steps, 3)
            per = kernel_breakdown(lmh, fb, args.steps, 3)
            bound = bwd_roofline_ms(Ts, H, V, peaks)
            joint = bwd_joint_roofline_ms(Ts, H, V, peaks)
            tot = sum(per.values())
            small_b[f"T={Ts}"] = {
                "ms_per_call": round(call_ms, 4), "tokens_per_s": Ts / (call_ms * 1e-3),
                "ms_kernels_summed": round(tot, 4),
                "kernels_ms": {k: round(v, 4) for k, v in per.items()},
                "roofline_ms_serial": round(sum(bound.values()), 4),
                "roofline_ms_joint": round(joint, 4),
                "frac_of_joint_roofline": round(joint / call_ms, 4),
                "kernel_frac": {k: round(bound[k] / per[k], 4) for k in bound if k in per}}
        extras["bwd_small_batches"] = {
            "workload": "backward of T rows, H=3584 V=152064, lse given",
            "peaks": f"bf16_tflops (burst) {peaks['bf16_tflops']} and hbm_gbs "
                     f"{peaks['hbm_gbs']} {peak_src}", **small_b}
        # the backward's memory lever: a smaller row chunk shrinks the dl
        # scratch (bf16 [row_chunk, V]) at some cost in time; the default
        # workspace is freed first, so each peak holds one workspace
        ws_b = None
        torch.cuda.empty_cache()
        chunks = {}
        for rc in (16384, 8192, 4096):
            wsb_c = torch.empty(lmh.lmhead_workspace_size_bwd(T, H, V, rc), dtype=torch.uint8,
                                device=dev)
            torch.cuda.reset_peak_memory_stats(dev)
            fc = lambda: lmh.lmhead_logprob_bwd_chunked(  # noqa: E731
                hidden, weight, labels, grad, s, row_chunk=rc, lse=lse, grad_hidden=gh,
                grad_weight=gw, workspace=wsb_c)
            per = kernel_breakdown(lmh, fc, max(3, args.steps // 4), 2)
            chunks[f"row_chunk={rc}"] = {"bwd_ms_kernels": round(sum(per.values()), 4),
                                         "peak_mem": peak_mem(wsb_c.numel())}
            del wsb_c
        extras["bwd_row_chunks"] = {"workload": WORKLOAD + ", backward only", **chunks}
        gh = gw = ws_b = hidden = weight = None  # free before the next legs
        torch.cuda.empty_cache()
        # forward only, Llama-like shape
        T2, H2, V2 = 4096, 4096, 32000
        torch.cuda.reset_peak_memory_stats(dev)
        h2, w2, l2, _ = make_inputs(T2, H2, V2, 99, dev)
        ws2 = torch.empty(lmh.lmhead_workspace_size(lmh.LMH_OP_FWD, T2, H2, V2), dtype=torch.uint8,
                          device=dev)
        lp2 = torch.empty(T2, device=dev)
        ent2 = torch.empty(T2, device=dev)
        fwd2 = lambda: lmh.lmhead_logprob_fwd(h2, w2, l2, 1.0, out_logprob=lp2,  # noqa: E731
                                              out_entropy=ent2, workspace=ws2)
        f2 = timed(fwd2, args.steps, 3)
        fk2 = kernel_ms(lmh, fwd2, args.steps, 3, fwd_kernels)
        extras["fwd_only"]["T=4096 H=4096 V=32000"] = {
            "tokens_per_s": T2 / (f2 * 1e-3), "ms_per_call": f2, "ms_kernels": fk2,
            "tflops_kernels": 2.0 * T2 * H2 * V2 / (fk2 * 1e-3) / 1e12,
            "frac_of_burst_peak": 2.0 * T2 * H2 * V2 / (fk2 * 1e-3) / 1e12 / peaks["bf16_tflops"],
            "peak_mem": peak_mem(ws2.numel())}
        extras["fwd_only"]["T=4096 H=4096 V=32000"]["invariance"] = invariance_cases(
            lambda rows: lmh.lmhead_logprob_fwd(h2[rows].contiguous(), w2, l2[rows].contiguous(),
                                                1.0, want_lse=True),
            T2, ((1, (0, T2 - 1)), (7, (0, 2045)), (256, (0, 3840))))
        del h2, w2
        # tiny fused forward T=64 H=256 V=4096: a latency figure, no roofline
        Tt, Ht, Vt = 64, 256, 4096
        torch.cuda.reset_peak_memory_stats(dev)
        ht_, wt_, lt_, _ = make_inputs(Tt, Ht, Vt, 1, dev)
        wst = torch.empty(lmh.lmhead_workspace_size(lmh.LMH_OP_FWD, Tt, Ht, Vt), dtype=torch.uint8,
                          device=dev)
        lpt, entt = torch.empty(Tt, device=dev), torch.empty(Tt, device=dev)
        fwdt = lambda: lmh.lmhead_logprob_fwd(ht_, wt_, lt_, 1.0, out_logprob=lpt,  # noqa: E731
                                              out_entropy=entt, workspace=wst)
        extras["tiny_fwd"] = {"workload": "fused forward T=64 H=256 V=4096",
                              "ms_per_call": timed(fwdt, 50, 5),
                              "ms_kernels": kernel_ms(lmh, fwdt, 50, 5, fwd_kernels),
                              "peak_mem": peak_mem(wst.numel())}
        # sub-batches of 1, 7 and the whole 64, windows shifted by 1..15
        extras["tiny_fwd"]["invariance"] = invariance_cases(
            lambda rows: lmh.lmhead_logprob_fwd(ht_[rows].contiguous(), wt_, lt_[rows].contiguous(),
                                                1.0, want_lse=True),
            Tt, ((1, (0, 1, 63)), (7, (0, 57)), (64, (0,))), window=48, shifts=(1, 7, 15), embed=64)
        del ht_, wt_
        # packed variable-length batch: 32 sequences of seeded lengths in
        # [128, 4096], concatenated; H=5120 V=152064; one fwd+bwd step
        import workloads as W

        Tp, Hp, Vp = int(sum(W.packed_lengths())), 5120, 152064
        torch.cuda.reset_peak_memory_stats(dev)
        hp, wp, lbp, gp = make_inputs(Tp, Hp, Vp, 5, dev)
        lpp, entp, lsep = (torch.empty(Tp, device=dev) for _ in range(3))
        ghp = torch.empty(Tp, Hp, dtype=torch.bfloat16, device=dev)
        gwp = torch.empty(Vp, Hp, device=dev)
        wsfp = torch.empty(lmh.lmhead_workspace_size(lmh.LMH_OP_FWD, Tp, Hp, Vp), dtype=torch.uint8,
                           device=dev)
        wsbp = torch.empty(lmh.lmhead_workspace_size(lmh.LMH_OP_BWD, Tp, Hp, Vp), dtype=torch.uint8,
                           device=dev)

        def packed_step():
            lmh.lmhead_logprob_fwd(hp, wp, lbp, 1.0, out_logprob=lpp, out_entropy=entp,
                                   out_lse=lsep, workspace=wsfp)
            lmh.lmhead_logprob_bwd(hp, wp, lbp, gp, 1.0, lse=lsep, grad_hidden=ghp,
                                   grad_weight=gwp, workspace=wsbp)

        p_ms = kernel_ms(lmh, packed_step, 3, 2, step_kernels)
        p_tf = 8.0 * Tp * Hp * Vp / (p_ms * 1e-3) / 1e12
        extras["packed_varlen_fwd_bwd"] = {
            "workload": f"32 sequences, lengths in [128, 4096], T={Tp} H={Hp} V={Vp}",
            "ms_kernels_per_step": p_ms, "tokens_per_s": Tp / (p_ms * 1e-3),
            "tflops_as_executed": p_tf, "frac_of_sustained": p_tf / peak,
            "peak_mem": peak_mem(wsfp.numel() + wsbp.numel())}
        del ghp, gwp, wsfp, wsbp
        torch.cuda.empty_cache()

        # the same rows re-packed: sequences in shuffled orders, and alone
        def packed_rows(rows):
            h_r, l_r = hp[rows].contiguous(), lbp[rows].contiguous()
            lp_r, ent_r, lse_r = lmh.lmhead_logprob_fwd(h_r, wp, l_r, 1.0, want_lse=True)
            gh_r, _ = lmh.lmhead_logprob_bwd(h_r, wp, l_r, gp[rows].contiguous(), 1.0, lse=lse_r)
            return lp_r, ent_r, lse_r, gh_r

        extras["packed_varlen_fwd_bwd"]["invariance"] = packed_invariance(
            packed_rows, W.packed_lengths())
        del hp, wp
        torch.cuda.empty_cache()
        # logits path: bf16 logits [8192, 152064] (2.49 GB > L2)
        T3, V3 = 8192, 152064
        torch.cuda.reset_peak_memory_stats(dev)
        g3 = torch.Generator(device=dev)
        g3.manual_seed(7)
        x = (torch.randn(T3, V3, generator=g3, device=dev) * 2.0
             + torch.randn(T3, 1, generator=g3, device=dev)).to(torch.bfloat16)
        l3 = torch.randint(0, V3, (T3,), generator=g3, device=dev, dtype=torch.int32)
        lp3 = torch.empty(T3, device=dev)
        ent3 = torch.empty(T3, device=dev)
        # The legs before this one keep the tensor cores at the power cap for
        # seconds; an idle second lets the clocks settle before a leg whose
        # issue rate matters, and this leg's own clocks are reported with it.
        torch.cuda.synchronize()
        time.sleep(1.0)
        l_clocks = ClockSampler(uuid)
        l_clocks.start()
        t_end = time.time() + 0.6  # keep the leg loaded long enough for a few clock samples
        while time.time() < t_end:
            for _ in range(50):
                lmh.logprob_from_logits(x, l3, 1.0, out_logprob=lp3, out_entropy=ent3)
            torch.cuda.synchronize()
        lmh.lmhead_timing_enable(True)
        l_ms = timed(lambda: lmh.logprob_from_logits(x, l3, 1.0, out_logprob=lp3,
                                                     out_entropy=ent3), args.steps, 3)
        krec = [ms for name, ms in lmh.lmhead_timing_read() if name == "logits_rowwise"]
        l_clk = l_clocks.stop()
        lmh.lmhead_timing_enable(False)
        k_ms = sum(krec) / len(krec)
        gbs = T3 * V3 * 2 / (k_ms * 1e-3) / 1e9
        extras["logits_path"] = {
            "workload": "sampler formula on bf16 logits T=8192 V=152064",
            "tokens_per_s": T3 / (l_ms * 1e-3), "ms": l_ms,
            "roofline": {"kernel": "logits_rowwise", "bound": "hbm", "achieved": round(gbs, 1),
                         "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(gbs / peaks["hbm_gbs"], 4),
                         "peak_source": f"hbm_gbs {peak_src}",
                         "traffic": traffic_for("logits_rowwise"),
                         "algorithmic_bytes_per_launch": T3 * V3 * 2},
            "clocks": l_clk, "peak_mem": peak_mem(0)}
        extras["logits_path"]["invariance"] = invariance_cases(
            lambda rows: lmh.logprob_from_logits(x[rows].contiguous(), l3[rows].contiguous(), 1.0,
                                                 want_lse=True),
            T3, ((1, (0, T3 - 1)), (7, (0, 4093)), (256, (0, 7936))))
        # sampler-parity (division) form on the same logits, and the mismatch
        # counts against torch's own fp32 sampler formula on the GPU
        temps = torch.full((T3,), 0.7, dtype=torch.float32, device=dev)
        lmh.lmhead_timing_enable(True)
        d_ms = timed(lambda: lmh.logprob_from_logits_div(x, l3, temps, out_logprob=lp3,
                                                         out_entropy=ent3), args.steps, 3)
        drec = [ms for name, ms in lmh.lmhead_timing_read() if name == "logits_rowwise_div"]
        lmh.lmhead_timing_enable(False)
        dk_ms = sum(drec) / len(drec)
        dgbs = T3 * V3 * 2 / (dk_ms * 1e-3) / 1e9
        q3 = torch.empty(T3, device=dev)
        sq = lambda: lmh.logprob_from_logits_stats(x, l3, 1.0, out_logprob=lp3,  # noqa: E731
                                                   out_entropy=ent3, out_sum_p2=q3)
        sq_ms = kernel_ms(lmh, sq, args.steps, 3, ("logits_rowwise",))
        extras["next_rows"]["logits_with_sum_p2"] = {
            "kernel_ms": sq_ms, "achieved_gbs": round(T3 * V3 * 2 / (sq_ms * 1e-3) / 1e9, 1),
            "frac": round(T3 * V3 * 2 / (sq_ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4)}
        extras["logits_path"]["division_form"] = {
            "tokens_per_s": T3 / (d_ms * 1e-3), "ms": d_ms, "kernel_ms": dk_ms,
            "achieved_gbs": round(dgbs, 1), "frac": round(dgbs / peaks["hbm_gbs"], 4),
            "traffic": traffic_for("logits_rowwise_div")}
        extras["sampler_parity"] = sampler_parity(lmh, x[:4096], l3[:4096])
        if rank == 0 and not args.no_cpu_baseline:
            extras["logits_path"]["cpu_oracle"] = cpu_oracle_logits()
            extras["logits_path"]["division_form"]["cpu_oracle"] = cpu_oracle_logits(divide=True)
        del x
        torch.cuda.empty_cache()
        line.update(extras)

    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


def run_case(args):
    """One kernel family on one shape, for profiling: --case fwd|bwd|logits|logits_div|logits_stats
    --shape ..."""
    import torch

    import invariant_lm_head_gb300 as lmh

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    lmh.build()
    dims = [int(x) for x in args.shape.split(",")]
    s = inv_temperature()
    if args.case in ("logits", "logits_div", "logits_stats"):
        T, V = dims
        g = torch.Generator(device=dev)
        g.manual_seed(7)
        x = (torch.randn(T, V, generator=g, device=dev) * 2.0
             + torch.randn(T, 1, generator=g, device=dev)).to(torch.bfloat16)
        lab = torch.randint(0, V, (T,), generator=g, device=dev, dtype=torch.int32)
        lp = torch.empty(T, device=dev)
        ent = torch.empty(T, device=dev)
        if args.case == "logits":
            fn = lambda: lmh.logprob_from_logits(x, lab, s, out_logprob=lp,  # noqa: E731
                                                 out_entropy=ent)
        elif args.case == "logits_stats":
            q = torch.empty(T, device=dev)
            fn = lambda: lmh.logprob_from_logits_stats(x, lab, s, out_logprob=lp,  # noqa: E731
                                                       out_entropy=ent, out_sum_p2=q)
        else:
            temps = torch.full((T,), 0.7, dtype=torch.float32, device=dev)
            fn = lambda: lmh.logprob_from_logits_div(x, lab, temps, out_logprob=lp,  # noqa: E731
                                                     out_entropy=ent)
        work = {"bytes": T * V * 2}
    else:
        T, H, V = dims
        hidden, weight, labels, grad = make_inputs(T, H, V, 1234, dev)
        lp = torch.empty(T, device=dev)
        ent = torch.empty(T, device=dev)
        lse = torch.empty(T, device=dev)
        ws_f = torch.empty(lmh.lmhead_workspace_size(lmh.LMH_OP_FWD, T, H, V), dtype=torch.uint8,
                           device=dev)
        lmh.lmhead_logprob_fwd(hidden, weight, labels, s, out_logprob=lp, out_entropy=ent,
                               out_lse=lse, workspace=ws_f)
        if args.case == "fwd":
            fn = lambda: lmh.lmhead_logprob_fwd(hidden, weight, labels, s, out_logprob=lp,  # noqa: E731
                                                out_entropy=ent, out_lse=lse, workspace=ws_f)
            work = {"flops": 2.0 * T * H * V}
        else:
            gh = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
            gw = torch.empty(V, H, device=dev)
            ws_b = torch.empty(lmh.lmhead_workspace_size(lmh.LMH_OP_BWD, T, H, V),
                               dtype=torch.uint8, device=dev)
            fn = lambda: lmh.lmhead_logprob_bwd(hidden, weight, labels, grad, s, lse=lse,  # noqa: E731
                                                grad_hidden=gh, grad_weight=gw, workspace=ws_b)
            work = {"flops": 6.0 * T * H * V}
    lmh.lmhead_timing_enable(True)
    ms = timed(fn, args.steps, args.warmup)
    recs = lmh.lmhead_timing_read()
    lmh.lmhead_timing_enable(False)
    lmh.lmhead_device_status()
    per = {}
    for name, t in recs:
        per.setdefault(name, []).append(t)
    out = {"case": args.case, "shape": dims, "ms": ms,
           "kernels_avg_ms": {k: sum(v) / len(v) for k, v in per.items()}}
    if "flops" in work:
        out["tflops"] = work["flops"] / (ms * 1e-3) / 1e12
    else:
        out["gbs"] = work["bytes"] / (ms * 1e-3) / 1e9
    print(json.dumps(out), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-extras", action="store_true", help="skip fwd-only and logits-path legs")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--case", choices=["fwd", "bwd", "logits", "logits_div", "logits_stats"],
                    default=None,
                    help="time one entry point on --shape only (profiling aid; no contract line)")
    ap.add_argument("--shape", default="4096,4096,32000", help="T,H,V (fwd/bwd) or T,V (logits)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        return run_reference(args)
    if args.case:
        return run_case(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
