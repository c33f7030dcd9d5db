"""Benchmark of the fused chunked KL distillation loss (forward + backward).

One step = kd_kl_forward + kd_kl_backward over one batch of synthetic input:
the GPT-OSS-20B-like student head at 32,768 tokens (d = 2880, V = 201,088,
K = 100 teacher entries, chunk = 2048, tau = 1). Prints ONE JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl {kdkl,reference}]

With N > 1 it is launched by torch.distributed.run, one rank per GPU; every
rank runs its own batch (weak scaling, no data-path collective) and rank 0
reports the max time over ranks. ``--impl reference`` times the fp64 CPU
oracle on bounded token samples of the same workload instead.
"""
from __future__ import annotations

import argparse
import functools
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "fused chunked KL fwd+bwd tokens/s, % of BF16 tensor peak, peak HBM GiB"
WORKLOAD = "gptoss20b_32k"
SPEC_BF16_TFLOPS = 2250.0
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# GEMM kernels and the GEMM-equivalents (2 N V d flops each) one step runs in
# each: the backward's dW and dH share one launch per block
GEMM_KERNELS = {"fwd_lse_gemm": 1, "bwd_grad_gemm": 1, "dH_gemm": 1, "dW_gemm": 1,
                "dW_dH_gemm": 2, "fwd_lse_mix_gemm": 1, "bwd_grad_mix_gemm": 1}
MIX_ALPHA, MIX_TAU_SQ = 0.5, True  # --path mix: alpha * tau^2 * KL + (1 - alpha) * CE
BAD_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown")


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK), "fallback"


def _code_only(text: str) -> str:
    """Source text without comments, blank lines or trailing spaces, so that a
    comment edit does not invalidate counters taken on the same code."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def csrc_digest() -> str:
    h = hashlib.sha256()
    cdir = os.path.join(ROOT, "lm_head_top_gb300", "csrc")
    for name in sorted(os.listdir(cdir)):
        with open(os.path.join(cdir, name), encoding="utf-8") as f:
            h.update(name.encode() + _code_only(f.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str = WORKLOAD):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, if the
    summary was taken on the current kernel sources and this workload;
    otherwise None."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    if d.get("csrc_sha256_16") != csrc_digest() or d.get("workload") != workload:
        return None
    k = d.get("kernels", {}).get(kernel)
    return None if k is None else float(k["dram_bytes_per_launch"])


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def __enter__(self):
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        self.file.flush()
        return False

    def summary(self):
        rows = []
        try:
            with open(self.file.name) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) >= 9 and parts[1].replace(".", "").isdigit():
                        rows.append(parts)
        finally:
            os.unlink(self.file.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[1]) for r in rows]
        reasons = set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for r in rows:
            for name, val in zip(names, r[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": float(rows[0][2]),
                "reasons": sorted(reasons), "samples": len(rows)}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        torch.distributed.barrier()


# --------------------------------------------------------------- oracle timing

def oracle_sample_step(x_np, w, rows, block: int = 1024):
    """fp64 oracle forward + backward on a sample of token rows (all V, all d),
    1024 rows at a time so the dense logit block stays a few GB."""
    import oracle.kl_oracle as ok
    H, W, idx, logit, mask = x_np
    for b in range(0, len(rows), block):
        r = rows[b:b + block]
        Hs, idxs, lgs, ms = H[r], idx[r], logit[r], mask[r]
        ok.forward(Hs, W, idxs, lgs, ms, w.tau)
        ok.backward(Hs, W, idxs, lgs, ms, w.tau, 1.0)


def oracle_rkl_sample_step(x_np, w, rows, block: int = 1024):
    """fp64 oracle reverse-KL forward + backward on a sample of token rows."""
    import oracle.kl_oracle as ok
    H, W, idx, logit, mask = x_np
    for b in range(0, len(rows), block):
        r = rows[b:b + block]
        ok.reverse_kl_forward(H[r], W, idx[r], logit[r], mask[r], w.tau)
        ok.reverse_kl_backward(H[r], W, idx[r], logit[r], mask[r], w.tau, 1.0)


def oracle_topk_sample_step(x_np, w, rows, K: int = 100, block: int = 512):
    """fp64 oracle top-K (dense row of logits, then the ordered K largest) on
    a sample of token rows."""
    import oracle.kl_oracle as ok
    H, W = x_np[0], x_np[1]
    for b in range(0, len(rows), block):
        ok.topk_logits(H[rows[b:b + block]], W, K)


def step_marks(n: int):
    """One timing event per step, created before the timed loop."""
    return [torch.cuda.Event(enable_timing=True) for _ in range(n)]


def step_stats(ev0, marks):
    """(median, min) ms of the individual steps between ev0 and the marks."""
    ms = [ev0.elapsed_time(marks[0])] + [a.elapsed_time(b) for a, b in zip(marks, marks[1:])]
    return round(float(np.median(ms)), 3), round(float(min(ms)), 3)


def kernel_pass(kdkl, step_fn, steps: int, stream, dev):
    """Runs `steps` more steps with the library's per-launch event timing on;
    returns [(kernel, launches, total ms)] and the pass's own elapsed ms."""
    torch.cuda.synchronize(dev)
    kdkl.kd_timing_begin()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        step_fn()
    b.record(stream)
    torch.cuda.synchronize(dev)
    rows = kdkl.kd_timing_end()
    return rows, a.elapsed_time(b)


def cpu_baseline(step_fn, x_np, w, n_tokens: int, what: str):
    """Times step_fn (an oracle sample step) on n_tokens random rows of w."""
    rng = np.random.default_rng(0)
    rows = np.sort(rng.choice(w.T, size=min(n_tokens, w.T), replace=False))
    t0 = time.perf_counter()
    step_fn(x_np, w, rows)
    t = time.perf_counter() - t0
    return {"value": round(len(rows) / t, 3), "unit": "tokens/s", "cores": blas_threads(),
            "kind": "oracle",
            "sample": "fp64 oracle %s on %d random tokens of %s (all V=%d, d=%d), %.1f s"
                      % (what, len(rows), w.name, w.V, w.d, t)}


def oracle_mix_sample_step(x_np, w, rows, labels, block: int = 1024):
    """fp64 oracle of the mixed soft + hard-label loss, forward + backward, on
    a sample of token rows."""
    import oracle.kl_oracle as ok
    H, W, idx, logit, mask = x_np
    for b in range(0, len(rows), block):
        r = rows[b:b + block]
        a = (H[r], W, idx[r], logit[r], mask[r], w.tau, MIX_ALPHA, MIX_TAU_SQ, labels[r])
        ok.forward_mixed(*a)
        ok.backward_mixed(*a, 1.0)


def oracle_arrays(x):
    import oracle.kl_oracle as ok
    return (ok.bf16_bits_to_f64(x["H"].view(torch.int16).numpy()),
            ok.bf16_bits_to_f64(x["W"].view(torch.int16).numpy()),
            x["topk_idx"].numpy().astype(np.int64), x["topk_logit"].numpy().astype(np.float64),
            x["mask"].numpy())


def blas_threads() -> int:
    """Threads the oracle's BLAS runs its products on: the library's own
    count where it can be read, else the thread variables it honours, else
    every core (the OpenBLAS default)."""
    try:
        from threadpoolctl import threadpool_info
    except ImportError:  # not installed on every host
        threadpool_info = None
    if threadpool_info is not None:
        n = [i["num_threads"] for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    try:  # the OpenBLAS numpy loaded, asked directly
        import ctypes
        with open("/proc/self/maps") as f:
            libs = {ln.split()[-1] for ln in f if "openblas" in ln.lower() and ".so" in ln}
        for lib in sorted(libs):
            h = ctypes.CDLL(lib)
            for sym in ("scipy_openblas_get_num_threads64_", "openblas_get_num_threads64_",
                        "openblas_get_num_threads"):
                fn = getattr(h, sym, None)
                if fn is not None:
                    fn.restype = ctypes.c_int
                    n = int(fn())
                    if n > 0:
                        return n
    except (OSError, ValueError):  # no /proc, or a library ctypes cannot open
        pass
    for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        v = os.environ.get(k, "")
        if v.isdigit() and int(v) > 0:
            return int(v)
    return os.cpu_count() or 1


def time_oracle(x_np, w, n_tokens: int, repeats: int = 1):
    rng = np.random.default_rng(0)
    times = []
    for _ in range(repeats):
        rows = np.sort(rng.choice(w.T, size=min(n_tokens, w.T), replace=False))
        t0 = time.perf_counter()
        oracle_sample_step(x_np, w, rows)
        times.append(time.perf_counter() - t0)
    return times


# ------------------------------------------------------------------- main arm

def apply_overrides(w, args):
    """The workload with --tokens/--K/--tau/--chunk applied, and the name it is
    reported under (the plain name when nothing is overridden)."""
    kw = {}
    if args.tokens:
        kw["T"] = args.tokens
    if args.vocab:
        kw["V"] = args.vocab
    if args.K:
        kw["K"] = args.K
    if args.tau:
        kw["tau"] = args.tau
    if args.chunk:
        kw["chunk"] = args.chunk
    if not kw:
        return w, w.name
    w2 = w.with_(**kw)
    return w2, "%s_T%d_V%d_K%d_tau%g_chunk%d" % (w.name, w2.T, w2.V, w2.K, w2.tau, w2.chunk)


def run_kdkl(args):
    from lm_head_top_gb300 import kdkl
    from lm_head_top_gb300.inputs import WORKLOADS, make_inputs

    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=dev)
    kdkl.load()
    w, wname = apply_overrides(WORKLOADS[args.workload], args)
    x = make_inputs(w, seed=args.seed + rank, topk_device=dev)
    T, d, V, K = w.T, w.d, w.V, w.K

    torch.cuda.reset_peak_memory_stats(dev)
    g = {k: v.to(dev) for k, v in x.items()}
    mix = args.path == "mix"
    ws_f = torch.empty(kdkl.kd_kl_workspace_size(T, d, V, K, w.tau, w.chunk, 2 if mix else 0),
                       dtype=torch.uint8, device=dev)
    # the backward reuses the teacher rows the forward prepared in ws_f
    ws_b = torch.empty(kdkl.kd_kl_workspace_size(T, d, V, K, w.tau, w.chunk, 4),
                       dtype=torch.uint8, device=dev)
    # --path mix: hard labels, seeded uniform over the vocabulary
    labels = torch.randint(0, V, (T,), dtype=torch.int32,
                           generator=torch.Generator().manual_seed(args.seed + rank)).to(dev)
    out = {"loss": None}
    loss = torch.empty(1, dtype=torch.float32, device=dev)
    lse = torch.empty(T, dtype=torch.float32, device=dev)
    dH = torch.empty(T, d, dtype=torch.bfloat16, device=dev)
    dW = torch.empty(V, d, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(gg):
        s = torch.cuda.current_stream(dev)  # the capture stream inside a graph capture
        if mix:
            a = (gg["H"], g["W"], gg["topk_idx"], gg["topk_logit"], gg["mask"], labels)
            kw = dict(temperature=w.tau, chunk=w.chunk, alpha=MIX_ALPHA, scale_tau_sq=MIX_TAU_SQ,
                      stream=s)
            out["loss"], lse_t, lse_1, _ = kdkl.kd_kl_forward_ex(*a, workspace=ws_f, **kw)
            kdkl.kd_kl_backward_ex(*a, lse_t, lse_1, grad_loss=1.0, dH=dH, dW=dW, workspace=ws_b,
                                   fwd_workspace=ws_f, **kw)
            return
        kdkl.kd_kl_forward(gg["H"], g["W"], gg["topk_idx"], gg["topk_logit"], gg["mask"],
                           temperature=w.tau, chunk=w.chunk, loss=loss, lse=lse, workspace=ws_f,
                           stream=s)
        kdkl.kd_kl_backward(gg["H"], g["W"], gg["topk_idx"], gg["topk_logit"], gg["mask"], lse,
                            temperature=w.tau, chunk=w.chunk, grad_loss=1.0, dH=dH, dW=dW,
                            workspace=ws_b, fwd_workspace=ws_f, stream=s)

    for _ in range(args.warmup):
        step(g)
    torch.cuda.synchronize(dev)
    st = kdkl.kd_kl_check_status(ws_f)
    st_b = kdkl.kd_kl_check_status(ws_b)
    if st or st_b:
        raise SystemExit("device status after warm-up: %s / %s" % (kdkl.kd_status_string(st),
                                                                   kdkl.kd_status_string(st_b)))

    # ---- device-resident timed region: the steps alone, bracketed by two
    # events (and one event per step for the spread); no per-kernel timing
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches0 = kdkl.kd_launch_count()
    with ClockSampler(local) as clocks:
        barrier(world)
        torch.cuda.synchronize(dev)
        marks = step_marks(args.steps)
        ev0.record(stream)
        for i in range(args.steps):
            step(g)
            marks[i].record(stream)
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
    launches = kdkl.kd_launch_count() - launches0
    elapsed_ms = max_over_ranks(ev0.elapsed_time(ev1), world, dev)
    med_ms, min_ms = step_stats(ev0, marks)  # this rank's steps
    clk = clocks.summary()
    peak_hbm = torch.cuda.max_memory_allocated(dev) / 2 ** 30

    # ---- per-kernel device times: the same steps again, every launch
    # bracketed by events on its stream (a separate pass, so the events do not
    # sit inside the headline timing)
    per_kernel, prof_ms = kernel_pass(kdkl, lambda: step(g), args.steps, stream, dev)

    # ---- the same step captured once in a CUDA graph and replayed (launch-bound
    # small shapes); reported beside the eager numbers
    graph_res = None
    if args.graph and not mix:
        per_step = launches // args.steps
        graph = torch.cuda.CUDAGraph()
        torch.cuda.synchronize(dev)
        n0 = kdkl.kd_launch_count()
        with torch.cuda.graph(graph):
            step(g)
        if kdkl.kd_launch_count() - n0 != per_step:
            raise SystemExit("graph capture recorded %d launches, expected %d"
                             % (kdkl.kd_launch_count() - n0, per_step))
        for _ in range(args.warmup):
            graph.replay()
        gs = torch.cuda.current_stream(dev)
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize(dev)
        g0.record(gs)
        for _ in range(args.steps):
            graph.replay()
        g1.record(gs)
        torch.cuda.synchronize(dev)
        barrier(world)
        gms = max_over_ranks(g0.elapsed_time(g1), world, dev)
        graph_res = {"value": round(T * world * args.steps / (gms / 1e3), 1), "unit": "tokens/s",
                     "ms_per_step": round(gms / args.steps, 4),
                     "gpu_launches": per_step * args.steps,
                     "note": "one captured step replayed; eager numbers above"}
        del graph

    # ---- end to end: pinned host inputs copied in, loss read back, every step
    e2e_ms, h2d = None, 0
    if not args.no_e2e:
        host = {k: v.pin_memory() for k, v in x.items() if k != "W"}
        loss_host = torch.empty(1, dtype=torch.float32).pin_memory()
        gin = {k: torch.empty_like(v, device=dev) for k, v in host.items()}
        h2d = sum(v.numel() * v.element_size() for v in host.values())
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize(dev)
        e0.record(stream)
        for _ in range(args.steps):
            for k in gin:
                gin[k].copy_(host[k], non_blocking=True)
            step(gin)
            loss_host.copy_(out["loss"] if mix else loss, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
        e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)

    result = None
    if rank == 0:
        pk, pk_src = peaks()
        tokens = T * world * args.steps
        # Masked tokens are compacted away before any GEMM, so the work done is
        # that of the counted tokens: 4 GEMM-equivalents of 2 N V d each.
        n_counted = int(x["mask"].sum())
        flops_step = 8.0 * n_counted * V * d
        tflops = flops_step * args.steps / (elapsed_ms / 1e3) / 1e12
        # dominant kernel by device time; algorithmic flops per launch = 2 N V d
        # per step for each of the four GEMM kinds, split over its launches
        rows = {n: (c, ms) for n, c, ms in per_kernel}
        dom = max(rows, key=lambda n: rows[n][1])
        run_name = wname  # traffic is recorded for the plain workloads only
        dom_launches, dom_ms = rows[dom]
        if dom in GEMM_KERNELS:
            per_launch_flops = (GEMM_KERNELS[dom] * 2.0 * n_counted * V * d * args.steps
                                / dom_launches)
            achieved = per_launch_flops / (dom_ms / dom_launches / 1e3) / 1e12
            peak = pk["bf16_tflops_sustained"]
            roof = {"bound": "tensor", "kernel": dom, "achieved": round(achieved, 1),
                    "peak": peak, "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                    "peak_source": "%s bf16_tflops_sustained" % pk_src,
                    "flops_per_launch": per_launch_flops,
                    "avg_launch_ms": round(dom_ms / dom_launches, 4),
                    "traffic": recorded_traffic(dom, run_name)}
        else:
            roof = {"bound": "hbm", "kernel": dom, "achieved": None, "peak": pk["hbm_gbs"],
                    "unit": "GB/s", "frac": None, "traffic": recorded_traffic(dom, run_name)}
        # CPU baseline: the fp64 oracle on a bounded token sample, this host
        cpu = None
        if world == 1 and not args.no_cpu_baseline and mix:
            lab_np = labels.cpu().numpy().astype(np.int64)
            cpu = cpu_baseline(lambda xn, ww, rows: oracle_mix_sample_step(xn, ww, rows, lab_np),
                               oracle_arrays(x), w, args.cpu_tokens,
                               "mixed-loss forward+backward")
        elif world == 1 and not args.no_cpu_baseline:
            x_np = oracle_arrays(x)
            n_cpu = args.cpu_tokens
            t = time_oracle(x_np, w, n_cpu)[0]
            cpu = {"value": round(n_cpu / t, 3), "unit": "tokens/s", "cores": blas_threads(),
                   "kind": "oracle",
                   "sample": "fp64 oracle forward+backward on %d random tokens of %s (all V=%d, "
                             "d=%d; dense logits row blocks), %.1f s" % (min(n_cpu, T), wname, V,
                                                                        d, t)}
        result = {
            "metric": METRIC if not mix else
            "mixed soft + hard-label distillation loss fwd+bwd tokens/s",
            "value": round(tokens / (elapsed_ms / 1e3), 1),
            "unit": "tokens/s",
            "value_counts": "every token of the batch, masked ones included",
            "counted_tokens_per_s": round(n_counted * world * args.steps / (elapsed_ms / 1e3), 1),
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": round(elapsed_ms / args.steps, 3),
            "ms_per_step_median": med_ms,
            "ms_per_step_min": min_ms,
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16",
            "data": "synthetic (seeded; bf16 H~N(0,1), W~N(0,1/d); teacher top-%d %s)" % (
                K, "half from the student's own top-%d" % K if w.teacher == "half_overlap"
                else "uniform distinct ids"),
            "config": {"workload": wname, "T": T, "counted_tokens": n_counted, "d": d, "V": V,
                       "K": K, "chunk": w.chunk,
                       "tau": w.tau, "seed": args.seed, "global_batch_tokens": T * world,
                       "parallelism": "dp%d (independent batches)" % world,
                       "l2": "inputs larger than L2 (W is %.2f GB); no flush" % (V * d * 2 / 1e9)},
            "tflops": round(tflops, 1),
            "pct_bf16_spec_peak": round(100 * tflops / SPEC_BF16_TFLOPS, 2),
            "pct_bf16_measured_sustained": round(100 * tflops / pk["bf16_tflops_sustained"], 2),
            "peak_hbm_gib": round(peak_hbm, 3),
            "roofline": roof,
            "cpu_baseline": cpu,
            "e2e": None if e2e_ms is None else {
                "value": round(tokens / (e2e_ms / 1e3), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": 4,
                "copies": "in: H, topk_idx, topk_logit, mask from pinned host memory; out: the "
                          "loss (4 bytes). dH and dW stay on the device, where a training "
                          "step's optimizer consumes them"},
            "gpu_launches": launches,
            "kernel_ms_per_step": {n: round(ms / args.steps, 3) for n, c, ms in per_kernel},
            "kernel_pass_ms_per_step": round(prof_ms / args.steps, 3),
            "clocks": clk,
        }
        if graph_res is not None:
            result["graph"] = graph_res
        if mix:
            result["path"] = "mix"
            result["config"].update({"workload": wname + "_mix", "alpha": MIX_ALPHA,
                                     "scale_tau_sq": MIX_TAU_SQ,
                                     "labels": "seeded uniform over the vocabulary"})
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    return result


def run_topk(args):
    """The offline top-K cache producer on the same head shapes: the teacher's
    K = 100 (or --K) largest logits per token over V = 201,088 (no logit grid
    stored)."""
    from lm_head_top_gb300 import kdkl
    from lm_head_top_gb300.inputs import WORKLOADS, make_inputs

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=dev)
    kdkl.load()
    w = WORKLOADS[args.workload].with_(teacher="uniform")
    if args.tokens:
        w = w.with_(T=args.tokens)
    x = make_inputs(w, seed=args.seed + rank)
    T, d, V, K = w.T, w.d, w.V, (args.K or 100)
    torch.cuda.reset_peak_memory_stats(dev)
    H, W = x["H"].to(dev), x["W"].to(dev)
    ws = torch.empty(kdkl.kd_lmhead_topk_workspace_size(T, d, V, K), dtype=torch.uint8, device=dev)
    idx = torch.empty(T, K, dtype=torch.int32, device=dev)
    val = torch.empty(T, K, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        kdkl.kd_lmhead_topk(H, W, K, topk_idx=idx, topk_logit=val, workspace=ws, stream=stream)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize(dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches0 = kdkl.kd_launch_count()
    with ClockSampler(local) as clocks:
        barrier(world)
        torch.cuda.synchronize(dev)
        marks = step_marks(args.steps)
        ev0.record(stream)
        for i in range(args.steps):
            step()
            marks[i].record(stream)
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
    elapsed_ms = max_over_ranks(ev0.elapsed_time(ev1), world, dev)
    med_ms, min_ms = step_stats(ev0, marks)  # this rank's steps
    launches = kdkl.kd_launch_count() - launches0
    per_kernel, _ = kernel_pass(kdkl, step, args.steps, stream, dev)

    # ---- end to end: pinned host H copied in, the cache (ids + logits) read back
    e2e = None
    if not args.no_e2e:
        H_host = x["H"].pin_memory()
        idx_host = torch.empty(T, K, dtype=torch.int32).pin_memory()
        val_host = torch.empty(T, K, dtype=torch.float32).pin_memory()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize(dev)
        e0.record(stream)
        for _ in range(args.steps):
            H.copy_(H_host, non_blocking=True)
            step()
            idx_host.copy_(idx, non_blocking=True)
            val_host.copy_(val, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
        e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
        e2e = {"value": round(T * world * args.steps / (e2e_ms / 1e3), 1), "unit": "tokens/s",
               "h2d_bytes_per_step": T * d * 2, "d2h_bytes_per_step": T * K * 8}
    if rank != 0:
        return None
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(functools.partial(oracle_topk_sample_step, K=K), oracle_arrays(x), w,
                           args.cpu_tokens // 2, "top-%d (dense logit rows, ordered selection)" % K)
    pk, pk_src = peaks()
    rows = {n: (c, ms) for n, c, ms in per_kernel}
    c, ms = rows["topk_gemm"]
    flops = 2.0 * T * V * d
    achieved = flops / (ms / c / 1e3) / 1e12  # one topk_gemm launch per step
    return {
        "metric": "offline top-K teacher cache (LM head x top-%d) tokens/s" % K, "path": "topk",
        "value": round(T * world * args.steps / (elapsed_ms / 1e3), 1), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": max(args.warmup, 3),
        "ms_per_step": round(elapsed_ms / args.steps, 3), "ms_per_step_median": med_ms,
        "ms_per_step_min": min_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "%s_topk%s" % (w.name, "" if K == 100 else "_K%d" % K), "T": T, "d": d, "V": V, "K": K,
                   "l2": "inputs larger than L2 (W is %.2f GB); no flush" % (V * d * 2 / 1e9)},
        "tflops": round(flops * args.steps / (elapsed_ms / 1e3) / 1e12, 1),
        "peak_hbm_gib": round(torch.cuda.max_memory_allocated(dev) / 2 ** 30, 3),
        "roofline": {"bound": "tensor", "kernel": "topk_gemm", "achieved": round(achieved, 1),
                     "peak": pk["bf16_tflops_sustained"], "unit": "TFLOP/s",
                     "frac": round(achieved / pk["bf16_tflops_sustained"], 4),
                     "peak_source": "%s bf16_tflops_sustained" % pk_src,
                     "traffic": recorded_traffic("topk_gemm", w.name if not args.tokens else "")},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches,
        "kernel_ms_per_step": {n: round(v / args.steps, 3) for n, cc, v in per_kernel},
        "clocks": clocks.summary(),
    }


def run_rkl(args):
    """Reverse KL over the cached ids (the loss-choice variant) on the same
    workload: kd_rkl_forward + kd_rkl_backward per step."""
    from lm_head_top_gb300 import kdkl
    from lm_head_top_gb300.inputs import WORKLOADS, make_inputs

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=dev)
    kdkl.load()
    w, wname = apply_overrides(WORKLOADS[args.workload], args)
    x = make_inputs(w, seed=args.seed + rank, topk_device=dev)
    T, d, V, K = w.T, w.d, w.V, w.K
    torch.cuda.reset_peak_memory_stats(dev)
    g = {k: v.to(dev) for k, v in x.items()}
    ws = torch.empty(kdkl.kd_rkl_workspace_size(T, d, V, K, w.tau), dtype=torch.uint8, device=dev)
    loss = torch.empty(1, dtype=torch.float32, device=dev)
    gz = torch.empty(T, K, dtype=torch.float32, device=dev)
    dH = torch.empty(T, d, dtype=torch.bfloat16, device=dev)
    dW = torch.empty(V, d, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        kdkl.kd_rkl_forward(g["H"], g["W"], g["topk_idx"], g["topk_logit"], g["mask"],
                            temperature=w.tau, loss=loss, grad_z=gz, workspace=ws, stream=stream)
        kdkl.kd_rkl_backward(g["H"], g["W"], g["topk_idx"], g["topk_logit"], g["mask"],
                             temperature=w.tau, grad_z=gz, dH=dH, dW=dW, workspace=ws,
                             stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if kdkl.kd_kl_check_status(ws):
        raise SystemExit("device status after warm-up: %s"
                         % kdkl.kd_status_string(kdkl.kd_kl_check_status(ws)))
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches0 = kdkl.kd_launch_count()
    with ClockSampler(local) as clocks:
        barrier(world)
        torch.cuda.synchronize(dev)
        marks = step_marks(args.steps)
        ev0.record(stream)
        for i in range(args.steps):
            step()
            marks[i].record(stream)
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
    elapsed_ms = max_over_ranks(ev0.elapsed_time(ev1), world, dev)
    med_ms, min_ms = step_stats(ev0, marks)  # this rank's steps
    launches = kdkl.kd_launch_count() - launches0
    per_kernel, _ = kernel_pass(kdkl, step, args.steps, stream, dev)

    # ---- end to end: pinned host H and teacher cache copied in, loss read back
    e2e = None
    if not args.no_e2e:
        host = {k: v.pin_memory() for k, v in x.items() if k != "W"}
        loss_host = torch.empty(1, dtype=torch.float32).pin_memory()
        h2d = sum(v.numel() * v.element_size() for v in host.values())
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize(dev)
        e0.record(stream)
        for _ in range(args.steps):
            for k in host:
                g[k].copy_(host[k], non_blocking=True)
            step()
            loss_host.copy_(loss, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
        e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
        e2e = {"value": round(T * world * args.steps / (e2e_ms / 1e3), 1), "unit": "tokens/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": 4}
    if rank != 0:
        return None
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(oracle_rkl_sample_step, oracle_arrays(x), w, args.cpu_tokens,
                           "reverse-KL forward+backward")
    pk, pk_src = peaks()
    # Algorithmic bytes per launch of each large kernel: every distinct W row
    # the cache names read once, H read once, the cache (ids, logits or the
    # saved gradient) read once, outputs written once.
    distinct = int(np.unique(x["topk_idx"].numpy()).size)
    pairs = T * K
    algo_bytes = {
        "rkl_z_segment": distinct * d * 2 + T * d * 2 + pairs * 12,
        "rkl_dH": distinct * d * 2 + pairs * 8 + T * d * 2,
        "rkl_dW_segment": T * d * 2 + pairs * 12 + distinct * d * 4,
    }
    rows = {n: (c, ms) for n, c, ms in per_kernel}
    dom = max(algo_bytes, key=lambda n: rows.get(n, (1, 0.0))[1])
    c, ms = rows[dom]
    algo = algo_bytes[dom]
    achieved = algo / (ms / c / 1e3) / 1e9
    # what the design streams: one row (W for rkl_dH, H for the z and dW
    # segments) of d bf16 per (token, id) pair, whatever the cache hits
    gather_gbs = pairs * d * 2 / (ms / c / 1e3) / 1e9
    return {
        "metric": "reverse KL over the cached ids fwd+bwd tokens/s", "path": "rkl",
        "value": round(T * world * args.steps / (elapsed_ms / 1e3), 1), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(elapsed_ms / args.steps, 3), "ms_per_step_median": med_ms,
        "ms_per_step_min": min_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "%s_rkl" % wname,
                   "T": T, "d": d, "V": V, "K": K, "tau": w.tau, "distinct_ids": distinct,
                   "l2": "inputs larger than L2 (W is %.2f GB); no flush" % (V * d * 2 / 1e9)},
        "peak_hbm_gib": round(torch.cuda.max_memory_allocated(dev) / 2 ** 30, 3),
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1),
                     "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": round(achieved / pk["hbm_gbs"], 4),
                     "peak_source": "%s hbm_gbs" % pk_src, "bytes_per_launch": algo,
                     "pair_gather_gbs": round(gather_gbs, 1),
                     "pair_gather_frac": round(gather_gbs / pk["hbm_gbs"], 4),
                     "traffic": recorded_traffic(dom, wname)},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches,
        "kernel_ms_per_step": {n: round(v / args.steps, 3) for n, cc, v in per_kernel},
        "clocks": clocks.summary(),
    }


def run_reference(args):
    """The fp64 CPU oracle on bounded token samples of the same workload."""
    from lm_head_top_gb300.inputs import WORKLOADS, make_inputs
    world, rank, _ = dist_env()
    if rank != 0:
        return None
    w = WORKLOADS[WORKLOAD]
    x = make_inputs(w, seed=args.seed)
    x_np = oracle_arrays(x)
    n = args.ref_tokens
    for _ in range(args.warmup):
        time_oracle(x_np, w, n)
    times = time_oracle(x_np, w, n, repeats=args.steps)
    total = sum(times)
    value = n * args.steps / total
    cpu = {"value": round(value, 3), "unit": "tokens/s", "cores": blas_threads(), "kind": "oracle",
           "sample": "fp64 oracle forward+backward on %d random tokens of %s per step "
                     "(all V=%d, d=%d)" % (n, WORKLOAD, w.V, w.d)}
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * total / args.steps, 1), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "T": w.T, "d": w.d, "V": w.V, "K": w.K, "chunk": w.chunk,
                   "tau": w.tau, "sample_tokens_per_step": n},
        "cpu_baseline": cpu,
        "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("kdkl", "reference"), default="kdkl")
    ap.add_argument("--path", choices=("kl", "mix", "topk", "rkl"), default="kl",
                    help="kl: fused KL fwd+bwd (the headline); mix: the mixed soft + "
                         "hard-label loss; topk: offline top-K cache producer; rkl: reverse KL "
                         "over the cached ids")
    ap.add_argument("--cpu-tokens", type=int, default=1024)
    ap.add_argument("--ref-tokens", type=int, default=256)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end pass")
    ap.add_argument("--workload", default=WORKLOAD,
                    help="another workload's shapes, for profiling small cases")
    ap.add_argument("--seed", type=int, default=0,
                    help="input seed (rank r of a multi-GPU run uses seed + r)")
    ap.add_argument("--tokens", type=int, default=0, help="override T (profiling cases)")
    ap.add_argument("--vocab", type=int, default=0,
                    help="override V (profiling cases: a smaller vocabulary with a larger chunk "
                         "keeps the backward's per-launch shapes)")
    ap.add_argument("--K", type=int, default=0, help="override K (config sweeps)")
    ap.add_argument("--tau", type=float, default=0.0, help="override the temperature")
    ap.add_argument("--chunk", type=int, default=0, help="override chunk")
    ap.add_argument("--graph", action="store_true",
                    help="also time the step captured in a CUDA graph and replayed")
    args = ap.parse_args()
    if args.impl == "kdkl":
        args.warmup = max(args.warmup, 3)  # timing rule: at least 3 warm-up steps
    if args.impl == "reference":
        res = run_reference(args)
    elif args.path == "topk":
        res = run_topk(args)
    elif args.path == "rkl":
        res = run_rkl(args)
    else:
        res = run_kdkl(args)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
