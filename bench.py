"""Benchmark of the exact attention forward pass (one JSON line on stdout).

One step = one fa_fwd call over the whole workload (every step of the path:
Q-tile loads, K/V streaming, S = QK^T, masking, online softmax, rescale,
O += PV, the O / l and LSE epilogue).  Default workload: B=1, H=32, N=8192,
D=128, causal, fp16 -- the configuration the throughput target is quoted on.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]
    python bench.py --pass bwd ...      the backward pass (fa_bwd) on the same workloads

Metric: attention forward TFLOP/s with the causal-adjusted FLOP model
(4*B*H*N^2*D, halved when causal), whole job over all ranks.
  * value      device time: inputs already in HBM; per-step CUDA events on
               the launching stream; the 129 MB L2 is flushed (a 256 MiB
               write) between timed steps, outside the events.
  * e2e        the same metric through the same C entry point with host
               buffers: pinned host -> device copies of Q, K, V, the call,
               and the device -> host copy of O and LSE, all inside the
               timed region.
  * roofline   tensor-bound: achieved = FLOPs per launch / mean launch time,
               against the measured dense bf16 peak (fp16 has the same
               nominal dense rate, so the ratio is 1).
  * cpu_baseline  the FP64 CPU oracle timed on the machine's host cores: the
               plain (naive) form over every row of the workload when that
               fits about 40 s (else a bounded row sample), the blocked
               online form on a bounded set of heads, and the naive form on
               one core.
  * accuracy   the device result against that naive oracle run: max-abs, RMS
               and relative L2 error of O, max-abs error of the LSE, and the
               output type's own rounding floor max|round_t(O_ref) - O_ref|.
N > 1: one rank per GPU (torchrun; `--gpus N` without torchrun launches the N
ranks itself).  Every rank runs the full workload on its own GPU (weak
scaling, no collective on the data path); rank 0 prints the line with the
slowest rank's time.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import fa_inputs  # noqa: E402

DEFAULT_WORKLOAD = "causal_fp16_b1h32n8192d128"
# Pages' number for this exact workload and metric: PyTorch SDPA flash backend,
# RTX 3060 Laptop (SM86), 25.854 ms at N=8192 ("CUDA FlashAttention: from online
# softmax to the long-sequence IO limit", section 8, benchmark table).
PAGE_MS = {"causal_fp16_b1h32n8192d128": 25.854, "causal_fp16_b1h32n4096d128": 6.573,
           "causal_fp16_b1h32n2048d128": 1.704, "causal_fp16_b1h32n1024d128": 0.447,
           "causal_fp16_b1h32n512d128": 0.149}
L2_FLUSH_BYTES = 256 << 20


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(values, device=None):
    """Element-wise MAX of a list of floats over all ranks (identity at world 1)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(x) for x in values]
    t = torch.tensor([float(x) for x in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def job_tflops(world, flops_per_rank, ms_per_step):
    """Whole-job throughput: every rank did flops_per_rank in (at most) ms_per_step."""
    return world * flops_per_rank / (ms_per_step * 1e-3) / 1e12


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), float(d.get("hbm_gbs", 6797.6)), "measured"
    return 1900.0, 6800.0, "fallback"


def measured_sustained():
    """The dense bf16 rate of a seconds-long GEMM loop under the power cap, if
    measured (reported beside the burst figure the fractions use: each timed
    step here is one launch, timed alone)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            v = json.load(f).get("bf16_tflops_sustained")
        return float(v) if v else None
    return None


def p95(xs):
    """95th percentile (nearest rank) of the per-step times."""
    ys = sorted(xs)
    return ys[min(len(ys) - 1, max(0, -(-95 * len(ys) // 100) - 1))]


def group_median(xs, groups=7):
    """Median of the means of `groups` consecutive groups of the per-step
    times (the timing protocol of "CUDA FlashAttention: from online softmax to
    the long-sequence IO limit", section 8: groups of repetitions, median of
    the group means).  None with fewer steps than groups."""
    if len(xs) < groups:
        return None
    per = len(xs) // groups
    return statistics.median(sum(xs[g * per:(g + 1) * per]) / per for g in range(groups))


def round_to(x, dtype):
    """float64 array rounded once, to nearest even, to fp16 or bf16 (values
    returned as float64)."""
    import numpy as np

    x = np.asarray(x, dtype=np.float64)
    if dtype == "fp16":
        return x.astype(np.float16).astype(np.float64)
    m, e = np.frexp(x)                      # x = m * 2^e, 0.5 <= |m| < 1
    return np.ldexp(np.rint(m * 256.0) / 256.0, e)   # 8 significant bits


def accuracy_stats(o, lse, o_ref, lse_ref, dtype):
    """Errors of a device result (O, LSE as float arrays) against the FP64
    oracle on the same rows: max-abs, RMS and relative L2 of O, max-abs of
    the LSE, and the floor that rounding the exact O to the output type alone
    gives, max|round_t(O_ref) - O_ref|."""
    import numpy as np

    o = np.asarray(o, dtype=np.float64).reshape(o_ref.shape)
    lse = np.asarray(lse, dtype=np.float64).reshape(lse_ref.shape)
    d = o - o_ref
    return {"max_abs_o": float(np.abs(d).max()), "rms_o": float(np.sqrt(np.mean(d * d))),
            "rel_l2_o": float(np.linalg.norm(d) / max(np.linalg.norm(o_ref), 1e-300)),
            "max_abs_lse": float(np.abs(lse - lse_ref).max()),
            "quant_floor_o": float(np.abs(round_to(o_ref, dtype) - o_ref).max()),
            "elements": int(d.size)}


def kernel_source_hash(kernel="fa_fwd.cu"):
    """Short hash of a kernel's source file and the PTX wrappers it includes."""
    h = hashlib.sha256()
    for rel in ("exact_attention_22_gb300/csrc/" + kernel, "exact_attention_22_gb300/csrc/sm103_ptx.cuh"):
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(key, kernel="fa_fwd.cu"):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the kernel source as it is now (else None).  Backward entries are keyed
    "bwd:<workload>" and hashed on fa_bwd.cu."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    rec = d.get(key)
    if not rec or rec.get("kernel_source_sha") != kernel_source_hash(kernel):
        return None
    return float(rec["dram_bytes_per_launch"])


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()
        return False

    def summary(self):
        rows = []
        for line in (self.out or "").strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != 6:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), parts[2:]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, flags in rows for i, f in enumerate(flags) if f.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


_INPUT_CACHE = {}


def _oracle_inputs(w, seed):
    key = (w.name, seed)
    if key not in _INPUT_CACHE:
        q, k, v = fa_inputs.make_qkv(w, seed=seed)
        _INPUT_CACHE.clear()
        _INPUT_CACHE[key] = (fa_inputs.bits(q), fa_inputs.bits(k), fa_inputs.bits(v))
    return _INPUT_CACHE[key]


def cpu_oracle_sample(w, seconds=12.0, seed=0, nthreads=0):
    """Time the FP64 oracle on a bounded, fixed-order sample of the workload's
    rows (all host cores, or ``nthreads``).  Returns (TFLOP/s, rows, seconds,
    threads, flops)."""
    import numpy as np

    from oracle import fa_ref

    qb, kb, vb = _oracle_inputs(w, seed)
    rng = np.random.default_rng(1234)
    BH, N = w.B * w.H, w.N
    order_bh = rng.integers(0, BH, 1 << 20)
    order_row = rng.integers(0, N, 1 << 20)
    threads = nthreads if nthreads > 0 else fa_ref.max_threads()
    chunk = max(threads * 4, 64)
    done, flops, t_total = 0, 0.0, 0.0
    while (done == 0 or t_total < seconds) and done + chunk <= len(order_row):
        bh = order_bh[done:done + chunk]
        rows = order_row[done:done + chunk]
        t0 = time.perf_counter()
        fa_ref.naive_rows(qb, kb, vb, w.scale, w.causal, bh, rows, enc=fa_inputs.enc(w), nthreads=threads)
        t_total += time.perf_counter() - t0
        vis = (rows + 1) if w.causal else np.full(len(rows), N)
        flops += float(np.sum(4.0 * vis * w.D))
        done += chunk
    # The FLOP model counts a causal row's half of the full square; the rows'
    # exact visible-key count is used here, which is the same on average.
    return flops / t_total / 1e12, done, t_total, threads, flops


def cpu_oracle_blocked(w, seconds=8.0, seed=0, rate_hint=None):
    """Time the blocked (online-softmax) FP64 oracle, 128 x 128 blocks, on the
    first min(threads, B*H) heads of the workload, each cut to its first n
    positions so that the run takes about ``seconds`` (n = N when it fits).
    Returns (TFLOP/s, heads, n, seconds, threads)."""
    import numpy as np

    from oracle import fa_ref

    qb, kb, vb = _oracle_inputs(w, seed)
    threads = fa_ref.max_threads()
    BH = w.B * w.H
    heads = min(threads, BH)
    per_head = 4.0 * w.N * w.N * w.D / (2.0 if w.causal else 1.0)
    n = w.N
    if rate_hint:
        # per-thread rate of the oracle: cut the heads so the run fits
        budget = rate_hint * 1e12 / threads * seconds
        if per_head > budget:
            n = max(256, int(w.N * (budget / per_head) ** 0.5))
    sl = [np.ascontiguousarray(x.reshape(BH, w.N, w.D)[:heads, :n]).reshape(1, heads, n, w.D) for x in (qb, kb, vb)]
    t0 = time.perf_counter()
    fa_ref.blocked(*sl, w.scale, w.causal, Br=128, Bc=128, enc=fa_inputs.enc(w))
    secs = time.perf_counter() - t0
    flops = heads * 4.0 * n * n * w.D / (2.0 if w.causal else 1.0)
    return flops / secs / 1e12, heads, n, secs, threads


def cpu_baseline_and_accuracy(w, o, lse, seconds=12.0, seed=0, full_limit=40.0):
    """The cpu_baseline leg: the naive FP64 oracle on all host cores, over
    every row of the workload when the estimated time is within
    ``full_limit`` seconds (else on a bounded random row sample), the blocked
    oracle beside it, and the naive oracle on one core.  The device result
    (o, lse: the tensors of the timed run) is compared with the naive run's
    rows: that comparison is the line's ``accuracy``."""
    import numpy as np

    from oracle import fa_ref

    est_tf, _, _, threads, _ = cpu_oracle_sample(w, seconds=1.0, seed=seed)
    full = w.flops / (est_tf * 1e12) <= full_limit
    o_np = o.float().cpu().numpy()
    l_np = lse.float().cpu().numpy()
    if full:
        qb, kb, vb = _oracle_inputs(w, seed)
        t0 = time.perf_counter()
        o_ref, lse_ref = fa_ref.naive(qb, kb, vb, w.scale, w.causal, enc=fa_inputs.enc(w))
        secs = time.perf_counter() - t0
        tf, rows = w.flops / secs / 1e12, w.B * w.H * w.N
        sample = ("every one of the workload's %d query rows, naive FP64 oracle, %.1f s" % (rows, secs))
        acc = accuracy_stats(o_np, l_np, o_ref, lse_ref, w.dtype)
        acc["rows"] = "all %d" % rows
    else:
        tf, rows, secs, threads, _ = cpu_oracle_sample(w, seconds=seconds, seed=seed)
        sample = ("%d query rows drawn uniformly at random (with replacement) from the workload's %d rows, "
                  "naive FP64 oracle, %.1f s" % (rows, w.B * w.H * w.N, secs))
        rng = np.random.default_rng(4321)
        bh = rng.integers(0, w.B * w.H, 4096)
        rr = rng.integers(0, w.N, 4096)
        qb, kb, vb = _oracle_inputs(w, seed)
        o_ref, lse_ref = fa_ref.naive_rows(qb, kb, vb, w.scale, w.causal, bh, rr, enc=fa_inputs.enc(w))
        o_s = o_np.reshape(w.B * w.H, w.N, w.D)[bh, rr]
        l_s = l_np.reshape(w.B * w.H, w.N)[bh, rr]
        acc = accuracy_stats(o_s, l_s, o_ref, lse_ref, w.dtype)
        acc["rows"] = "4096 sampled of %d" % (w.B * w.H * w.N)
    acc["oracle"] = "naive FP64 (plain safe softmax per row) on the same 16-bit inputs"
    tf1, rows1, secs1, _, _ = cpu_oracle_sample(w, seconds=3.0, seed=seed, nthreads=1)
    btf, bheads, bn, bsecs, _ = cpu_oracle_blocked(w, seconds=8.0, seed=seed, rate_hint=tf)
    base = {
        "value": tf, "unit": "TFLOP/s", "cores": threads, "kind": "oracle", "sample": sample,
        "blocked": {"value": btf, "unit": "TFLOP/s", "cores": threads,
                    "sample": "blocked online-softmax FP64 oracle (128 x 128 blocks) on %d head(s), first %d of "
                              "%d positions each, %.1f s" % (bheads, bn, w.N, bsecs)},
        "one_thread": {"value": tf1, "unit": "TFLOP/s", "sample": "%d random rows of the workload, naive FP64 "
                       "oracle on one core, %.1f s" % (rows1, secs1)}}
    return base, acc


def run_reference(args, w):
    world, rank, _ = _dist()
    if rank != 0:
        return 0
    # The whole run is held to about two minutes of oracle time: each step is a
    # row sample of seconds = 120 / (steps + warmup), at least one chunk of rows.
    per_step = 120.0 / max(1, args.steps + args.warmup)
    for _ in range(args.warmup):
        cpu_oracle_sample(w, seconds=per_step)
    vals, rows, secs, threads = [], 0, 0.0, 1
    for _ in range(args.steps):
        tf, r, s, threads, _ = cpu_oracle_sample(w, seconds=per_step)
        vals.append(tf)
        rows += r
        secs += s
    value = statistics.median(vals)
    sample = ("%d query rows drawn uniformly at random (with replacement) from all %d rows of the workload, "
              "%.1f s of FP64 oracle time" % (rows, w.B * w.H * w.N, secs))
    line = {
        "impl": "reference", "metric": "attention fwd TFLOP/s (causal-adjusted)", "value": value,
        "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": secs / max(1, args.steps) * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded N(0,1) inputs, see fa_inputs.py)",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "D": w.D, "causal": w.causal,
                   "input_dtype": w.dtype},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args, w):
    import torch
    import torch.distributed as dist

    import exact_attention_22_gb300 as fa

    world, rank, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if world > 1:
            dist.barrier()

    fp8 = args.fp8
    if fp8:
        # E4M3 inputs quantized per 128-row block; V handed over transposed per head
        (q_h, k_h, v8), scales_h = fa_inputs.make_qkv_fp8(w, seed=args.seed + rank)
        v_h = v8.transpose(2, 3).contiguous()
        scales = [t.to(dev) for t in scales_h]
    else:
        q_h, k_h, v_h = fa_inputs.make_qkv(w, seed=args.seed + rank)
    q, k, v = (t.to(dev) for t in (q_h, k_h, v_h))
    o = torch.empty((w.B, w.H, w.N, w.D), dtype=torch.bfloat16, device=dev) if fp8 else torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    handle = stream.cuda_stream
    dt = fa.FA_BF16 if w.dtype == "bf16" else fa.FA_FP16

    splits = args.num_splits
    ws = ws_bytes = None
    if splits > 0:
        ws_bytes = fa.fa_splitkv_workspace_bytes(w.B, w.H, w.N, w.D, splits)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)

    def launch(qq, kk, vv, oo, ll):
        if fp8:
            st = fa.fa_fwd_fp8(qq.data_ptr(), kk.data_ptr(), vv.data_ptr(), scales[0].data_ptr(),
                               scales[1].data_ptr(), scales[2].data_ptr(), oo.data_ptr(), ll.data_ptr(), w.B, w.H,
                               w.N, w.D, w.scale, int(w.causal), handle)
        elif splits > 0:
            st = fa.fa_fwd_splitkv(qq.data_ptr(), kk.data_ptr(), vv.data_ptr(), oo.data_ptr(), ll.data_ptr(), w.B,
                                   w.H, w.N, w.D, w.scale, int(w.causal), dt, splits, ws.data_ptr(), ws_bytes,
                                   handle)
        else:
            st = fa.fa_fwd(qq.data_ptr(), kk.data_ptr(), vv.data_ptr(), oo.data_ptr(), ll.data_ptr(), w.B, w.H,
                           w.N, w.D, w.scale, int(w.causal), dt, handle)
        if st != fa.FA_OK:
            raise fa.FaError(st, "fa_fwd")

    for _ in range(args.warmup):
        flush.zero_()
        launch(q, k, v, o, lse)
    torch.cuda.synchronize()
    status = fa.fa_get_device_status(handle)
    if status != fa.FA_OK:
        raise fa.FaError(status, "warm-up")

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(local) as clocks:
        barrier()
        torch.cuda.synchronize()
        for i in range(args.steps):
            flush.zero_()
            starts[i].record(stream)
            launch(q, k, v, o, lse)
            ends[i].record(stream)
        torch.cuda.synchronize()
        barrier()
    launches = args.steps * (2 if splits > 0 else 1)   # split-K: forward + merge kernel
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total_ms = sum(step_ms)
    status = fa.fa_get_device_status(handle)
    if status != fa.FA_OK:
        raise fa.FaError(status, "timed region")

    # End to end through host buffers: H2D of Q, K, V; the call; D2H of O, LSE.
    # The 16-bit unsplit path goes through fa_fwd_host, the library's entry
    # point for host-resident tensors (copies overlapped with the kernel in
    # chunks of heads); the other modes copy, launch and copy back in order.
    qp, kp, vp = (t.pin_memory() for t in (q_h, k_h, v_h))
    op = torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
    lp = torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)
    host_api = splits == 0
    if host_api:
        hws_bytes = (fa.fa_fwd_fp8_host_workspace_bytes if fp8 else fa.fa_fwd_host_workspace_bytes)(w.B, w.H, w.N,
                                                                                                    w.D)
        hws = torch.empty(hws_bytes, dtype=torch.uint8, device=dev)
        if fp8:
            scp = [t.pin_memory() for t in scales_h]

    def e2e_step():
        if host_api and fp8:
            st = fa.fa_fwd_fp8_host(qp.data_ptr(), kp.data_ptr(), vp.data_ptr(), scp[0].data_ptr(), scp[1].data_ptr(),
                                    scp[2].data_ptr(), op.data_ptr(), lp.data_ptr(), w.B, w.H, w.N, w.D, w.scale,
                                    int(w.causal), hws.data_ptr(), hws_bytes, handle)
            if st != fa.FA_OK:
                raise fa.FaError(st, "fa_fwd_fp8_host")
            return
        if host_api:
            st = fa.fa_fwd_host(qp.data_ptr(), kp.data_ptr(), vp.data_ptr(), op.data_ptr(), lp.data_ptr(), w.B, w.H,
                                w.N, w.D, w.scale, int(w.causal), dt, hws.data_ptr(), hws_bytes, handle)
            if st != fa.FA_OK:
                raise fa.FaError(st, "fa_fwd_host")
            return
        q.copy_(qp, non_blocking=True); k.copy_(kp, non_blocking=True); v.copy_(vp, non_blocking=True)
        launch(q, k, v, o, lse)
        op.copy_(o, non_blocking=True); lp.copy_(lse, non_blocking=True)

    e2e_steps = max(3, min(args.steps, 50))
    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    if host_api:
        status = fa.fa_get_device_status(handle)
        if status != fa.FA_OK:
            raise fa.FaError(status, "end-to-end steps")
        # the host-buffer path computes what the device path computed
        if not (torch.equal(op, o.cpu()) and torch.equal(lp, lse.cpu())):
            raise RuntimeError("host-buffer entry results differ from the device entry's")
    h2d = sum(t.numel() * t.element_size() for t in (q, k, v))
    if fp8:
        h2d += sum(t.numel() * t.element_size() for t in scales_h)   # the block scales travel too
    d2h = o.numel() * o.element_size() + lse.numel() * lse.element_size()

    total_ms, e2e_ms = max_over_ranks([total_ms, e2e_ms], device=dev)
    ms_per_step = total_ms / args.steps
    value = job_tflops(world, w.flops, ms_per_step)
    e2e_value = job_tflops(world, w.flops, e2e_ms)
    peak, hbm, peak_kind = measured_peaks()
    peak_note = "%s dense bf16 (burst); fp16/bf16 nominal ratio 1" % peak_kind
    if fp8:
        peak *= 2.0   # dense FP8 runs at twice the dense bf16 rate (nominal ratio)
        peak_note = "%s dense bf16 (burst) x 2, the nominal fp8/bf16 dense ratio" % peak_kind
    achieved = w.flops / (ms_per_step * 1e-3) / 1e12
    sustained = measured_sustained()
    if sustained and fp8:
        sustained *= 2.0
    clk = clocks.summary()

    line = {
        "metric": "attention fwd TFLOP/s (causal-adjusted)", "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": (value / (w.flops / (PAGE_MS[w.name] * 1e-3) / 1e12)) if (w.name in PAGE_MS and not fp8)
        else None,
        "dtype": "e4m3 (bf16 out)" if fp8 else w.dtype,
        "data": "synthetic (seeded N(0,1) inputs%s, see fa_inputs.py)" % (", E4M3 per-128-row-block scales" if fp8 else ""),
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "D": w.D, "causal": w.causal,
                   "scale": w.scale, "parallelism": "replica per GPU" if world > 1 else "single GPU",
                   "l2": "flushed between timed steps (256 MiB write, outside the events)",
                   "ms_p50": statistics.median(step_ms), "ms_p95": p95(step_ms), "ms_min": min(step_ms),
                   "ms_median_of_7_group_means": group_median(step_ms),
                   "num_splits": splits,
                   "entry": "fa_fwd_fp8" if fp8 else ("fa_fwd_splitkv" if splits > 0 else "fa_fwd")},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": None if fp8 else recorded_traffic(w.name),
                     "peak_kind": peak_note,
                     "peak_sustained": sustained, "frac_sustained": achieved / sustained if sustained else None,
                     "effective_GBps": w.io_bytes / (ms_per_step * 1e-3) / 1e9},
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms, "api": ("fa_fwd_fp8_host" if fp8 else "fa_fwd_host") if host_api else
                "copies + fa_fwd_splitkv + copies in order"},
        "gpu_launches": launches,
        "clocks": clk,
        "kernel_source_sha": kernel_source_hash(),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not fp8:
        line["cpu_baseline"], line["accuracy"] = cpu_baseline_and_accuracy(w, o, lse, seconds=args.cpu_seconds,
                                                                           seed=args.seed)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_ours_bwd(args, w):
    """The backward pass (fa_bwd: Delta kernel, main kernel, dQ conversion) on
    the same workload: one step = one fa_bwd call; FLOPs = 2.5x the forward's
    (five N x N x D GEMMs -- S, dP, dV, dK, dQ -- against the forward's two)."""
    import torch
    import torch.distributed as dist

    import exact_attention_22_gb300 as fa

    world, rank, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if world > 1:
            dist.barrier()

    q_h, k_h, v_h = fa_inputs.make_qkv(w, seed=args.seed + rank)
    g = torch.Generator().manual_seed(args.seed + rank + 1000)
    do_h = torch.randn(q_h.shape, generator=g).to(q_h.dtype)
    q, k, v, do = (t.to(dev) for t in (q_h, k_h, v_h, do_h))
    o, lse = fa.attention(q, k, v, causal=w.causal, scale=w.scale)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    ws_bytes = fa.fa_bwd_workspace_bytes(w.B, w.H, w.N, w.D)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    handle = stream.cuda_stream
    dt = fa.FA_BF16 if w.dtype == "bf16" else fa.FA_FP16
    flops = 2.5 * w.flops

    def launch():
        st = fa.fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(), lse.data_ptr(),
                       dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), w.B, w.H, w.N, w.D, w.scale, int(w.causal), dt,
                       ws.data_ptr(), ws_bytes, handle)
        if st != fa.FA_OK:
            raise fa.FaError(st, "fa_bwd")

    for _ in range(args.warmup):
        flush.zero_()
        launch()
    torch.cuda.synchronize()
    status = fa.fa_get_device_status(handle)
    if status != fa.FA_OK:
        raise fa.FaError(status, "warm-up")
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(local) as clocks:
        barrier()
        torch.cuda.synchronize()
        for i in range(args.steps):
            flush.zero_()
            starts[i].record(stream)
            launch()
            ends[i].record(stream)
        torch.cuda.synchronize()
        barrier()
    step_ms = [s_.elapsed_time(e_) for s_, e_ in zip(starts, ends)]
    status = fa.fa_get_device_status(handle)
    if status != fa.FA_OK:
        raise fa.FaError(status, "timed region")

    # End to end through fa_bwd_host, the library's entry point for host-resident
    # tensors: H2D of Q, K, V, O, dO, LSE, the pass, D2H of dQ, dK, dV, in
    # chunks of heads with the copies overlapping the kernels.
    pins = [t.pin_memory() for t in (q_h, k_h, v_h, o.cpu(), do_h, lse.cpu())]
    devs = [q, k, v, o, do, lse]
    outs_h = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (dq, dk, dv)]
    e2e_steps = max(3, min(args.steps, 30))
    hws_bytes = fa.fa_bwd_host_workspace_bytes(w.B, w.H, w.N, w.D)
    hws = torch.empty(hws_bytes, dtype=torch.uint8, device=dev)

    def e2e_step():
        st = fa.fa_bwd_host(*(t.data_ptr() for t in pins[:6]), *(t.data_ptr() for t in outs_h), w.B, w.H, w.N, w.D,
                            w.scale, int(w.causal), dt, hws.data_ptr(), hws_bytes, handle)
        if st != fa.FA_OK:
            raise fa.FaError(st, "fa_bwd_host")

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    status = fa.fa_get_device_status(handle)
    if status != fa.FA_OK:
        raise fa.FaError(status, "end-to-end steps")
    # dK, dV as the device path gave them; dQ up to the order of its fp32 additions
    if not (torch.equal(outs_h[1], dk.cpu()) and torch.equal(outs_h[2], dv.cpu())):
        raise RuntimeError("fa_bwd_host dK / dV differ from fa_bwd")
    if (outs_h[0].float() - dq.cpu().float()).abs().max().item() > 2.0 ** -9 * max(1.0, dq.float().abs().max().item()):
        raise RuntimeError("fa_bwd_host dQ differs from fa_bwd")
    h2d = sum(t.numel() * t.element_size() for t in devs)
    d2h = sum(t.numel() * t.element_size() for t in (dq, dk, dv))

    total_ms, e2e_ms = max_over_ranks([sum(step_ms), e2e_ms], device=dev)
    ms_per_step = total_ms / args.steps
    value = job_tflops(world, flops, ms_per_step)
    peak, hbm, peak_kind = measured_peaks()
    achieved = flops / (ms_per_step * 1e-3) / 1e12
    sustained = measured_sustained()
    line = {
        "metric": "attention bwd TFLOP/s (causal-adjusted, 2.5x the forward FLOPs)", "value": value,
        "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic (seeded N(0,1) inputs and dO, see fa_inputs.py)",
        "config": {"workload": w.name, "pass": "bwd", "B": w.B, "H": w.H, "N": w.N, "D": w.D, "causal": w.causal,
                   "scale": w.scale, "parallelism": "replica per GPU" if world > 1 else "single GPU",
                   "l2": "flushed between timed steps (256 MiB write, outside the events)",
                   "ms_p50": statistics.median(step_ms), "ms_p95": p95(step_ms), "ms_min": min(step_ms),
                   "ms_median_of_7_group_means": group_median(step_ms), "entry": "fa_bwd"},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": recorded_traffic("bwd:" + w.name, "fa_bwd.cu"),
                     "traffic_kernel": "fa_bwd_kernel (main kernel of the three)",
                     "peak_kind": "%s dense bf16 (burst); fp16/bf16 nominal ratio 1" % peak_kind,
                     "peak_sustained": sustained, "frac_sustained": achieved / sustained if sustained else None},
        "e2e": {"value": job_tflops(world, flops, e2e_ms), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "api": "fa_bwd_host"},
        "gpu_launches": 3 * args.steps,
        "clocks": clocks.summary(),
        "kernel_source_sha": kernel_source_hash("fa_bwd.cu"),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        from oracle import fa_ref

        e = fa_inputs.enc(w)
        one = [fa_inputs.bits(t[:1, :1]) for t in (q_h, k_h, v_h, do_h)]
        t0 = time.time()
        fa_ref.backward(*one, w.scale, w.causal, enc=e)
        secs = time.time() - t0
        line["cpu_baseline"] = {
            "value": flops / (w.B * w.H) / secs / 1e12, "unit": "TFLOP/s", "cores": fa_ref.max_threads(),
            "kind": "oracle", "sample": "head (0, 0) of the workload: every row and key, FP64 backward oracle, "
                                        "%.1f s" % secs}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


# Decode: one new query per head against a long K/V sequence (fa_fwd_kv).
#   name: (B, H, H_kv, Nq, Nk, D, dtype)
DECODE_WORKLOADS = {
    "decode_bf16_b8h32kv8_nk32768d128": (8, 32, 8, 1, 32768, 128, "bf16"),
    "decode_bf16_b1h32kv8_nk131072d128": (1, 32, 8, 1, 131072, 128, "bf16"),
}


def run_decode(args):
    """fa_fwd_kv on a decode shape: HBM-bound, reported as the bandwidth of the
    bytes one call must move (K, V read once, Q read, O and LSE written)."""
    import torch

    import exact_attention_22_gb300 as fa

    B, H, H_kv, Nq, Nk, D, dtype = DECODE_WORKLOADS[args.decode]
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    g = torch.Generator().manual_seed(args.seed)
    td = torch.bfloat16 if dtype == "bf16" else torch.float16
    q = torch.randn(B, H, Nq, D, generator=g).to(td).to(dev)
    k = torch.randn(B, H_kv, Nk, D, generator=g).to(td).to(dev)
    v = torch.randn(B, H_kv, Nk, D, generator=g).to(td).to(dev)
    o = torch.empty_like(q)
    lse = torch.empty(B, H, Nq, dtype=torch.float32, device=dev)
    if args.num_splits_auto:
        splits = fa.fa_fwd_kv_splits_hint(B, H, H_kv, Nq, Nk, D, 1)
        if splits < 0:
            raise RuntimeError("fa_fwd_kv_splits_hint failed")
    else:
        splits = args.num_splits
    ws_bytes = fa.fa_fwd_kv_workspace_bytes(B, H, Nq, D, splits) if splits > 0 else 0
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    handle = stream.cuda_stream
    dt = fa.FA_BF16 if dtype == "bf16" else fa.FA_FP16

    def launch():
        st = fa.fa_fwd_kv(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, H_kv, Nq,
                          Nk, D, D ** -0.5, 1, dt, splits, ws.data_ptr() if splits > 0 else 0, ws_bytes, handle)
        if st != fa.FA_OK:
            raise fa.FaError(st, "fa_fwd_kv")

    for _ in range(args.warmup):
        flush.zero_()
        launch()
    torch.cuda.synchronize()
    if fa.fa_get_device_status(handle) != fa.FA_OK:
        raise RuntimeError("device status after warm-up")
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(0) as clocks:
        torch.cuda.synchronize()
        for i in range(args.steps):
            flush.zero_()
            starts[i].record(stream)
            launch()
            ends[i].record(stream)
        torch.cuda.synchronize()
    step_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    ms = sum(step_ms) / len(step_ms)
    if fa.fa_get_device_status(handle) != fa.FA_OK:
        raise RuntimeError("device status after the timed region")
    # End to end: a decode step's new queries come from the host and its outputs
    # go back; the K/V cache stays resident on the device, as it does in serving.
    q_h = q.cpu().pin_memory()
    o_h = torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
    l_h = torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)
    e2e_steps = max(3, min(args.steps, 50))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(e2e_steps):
        q.copy_(q_h, non_blocking=True)
        launch()
        o_h.copy_(o, non_blocking=True)
        l_h.copy_(lse, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    nbytes = 2 * B * H_kv * Nk * D * 2 + 2 * B * H * Nq * D * 2 + B * H * Nq * 4
    gbps = nbytes / (ms * 1e-3) / 1e9
    _, hbm, peak_kind = measured_peaks()
    line = {
        "metric": "decode bytes moved / time (GB/s)", "value": gbps, "unit": "GB/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": dtype, "data": "synthetic (seeded N(0,1))",
        "config": {"workload": args.decode, "B": B, "H": H, "H_kv": H_kv, "Nq": Nq, "Nk": Nk, "D": D,
                   "causal": True, "num_splits": splits, "entry": "fa_fwd_kv",
                   "l2": "flushed between timed steps (256 MiB write, outside the events)",
                   "ms_p50": statistics.median(step_ms), "ms_p95": p95(step_ms), "ms_min": min(step_ms),
                   "ms_median_of_7_group_means": group_median(step_ms)},
        "roofline": {"bound": "hbm", "achieved": gbps, "peak": hbm, "unit": "GB/s", "frac": gbps / hbm,
                     "traffic": None, "peak_kind": "%s copy bandwidth" % peak_kind},
        "e2e": {"value": nbytes / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s", "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": q.numel() * q.element_size(),
                "d2h_bytes_per_step": o.numel() * o.element_size() + lse.numel() * lse.element_size(),
                "api": "copy of Q, fa_fwd_kv, copy of O and LSE; the K/V cache resident on the device"},
        "gpu_launches": args.steps * (2 if splits > 0 else 1),
        "clocks": clocks.summary(),
        "kernel_source_sha": kernel_source_hash(),
    }
    print(json.dumps(line), flush=True)
    return 0


def launch_ranks(n, argv):
    """Run this script as n ranks, one per GPU, through torch.distributed.run
    on 127.0.0.1 (used when --gpus N > 1 is given without a launcher)."""
    import socket

    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", str(n),
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__)] + list(argv)
    return subprocess.call(cmd)


def run_dry(args):
    """The multi-rank plumbing alone, without a GPU: each rank joins a gloo
    group, the slowest rank's (stand-in) time is taken, and rank 0 prints one
    line."""
    import torch.distributed as dist

    world, rank, _ = _dist()
    if world > 1:
        dist.init_process_group("gloo")
    ms = max_over_ranks([1.0 + rank])[0]
    if rank == 0:
        print(json.dumps({"dry_run": True, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                          "ms_per_step": ms}), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    argv = list(sys.argv[1:] if argv is None else argv)
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(fa_inputs.WORKLOADS))
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--num-splits", default="0",
                    help="time fa_fwd_splitkv with this many K/V chunks per query block (0: fa_fwd); with "
                         "--decode, 'auto' takes fa_fwd_kv_splits_hint's count")
    ap.add_argument("--decode", choices=sorted(DECODE_WORKLOADS), default=None,
                    help="time fa_fwd_kv on a decode shape (HBM bandwidth); --num-splits selects split-K")
    ap.add_argument("--fp8", action="store_true",
                    help="time fa_fwd_fp8 on the workload's shape with E4M3 inputs (D = 128, N a multiple of 16)")
    ap.add_argument("--pass", dest="which", choices=["fwd", "bwd"], default="fwd",
                    help="time the forward pass (default, the headline) or the backward pass")
    ap.add_argument("--dry-run", action="store_true",
                    help="only the rank plumbing (launch, process group, slowest-rank time), no GPU work")
    args = ap.parse_args(argv)
    if args.gpus < 1:
        ap.error("--gpus must be >= 1")
    world = _dist()[0]
    if args.gpus != world:
        if "WORLD_SIZE" in os.environ:
            ap.error("--gpus %d does not match WORLD_SIZE=%d (one rank per GPU)" % (args.gpus, world))
        return launch_ranks(args.gpus, argv)
    if args.dry_run:
        return run_dry(args)
    args.num_splits_auto = args.num_splits == "auto"
    if args.num_splits_auto and args.decode is None:
        ap.error("--num-splits auto applies to --decode")
    args.num_splits = 0 if args.num_splits_auto else int(args.num_splits)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.decode:
        return run_decode(args)
    w = fa_inputs.WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, w)
    if args.which == "bwd":
        return run_ours_bwd(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
