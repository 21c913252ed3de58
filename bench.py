"""Benchmark of the fused output-projection + cross-entropy forward+backward.

One step = one lce_forward_backward over the whole batch of the workload
(compaction, logits + online log-sum-exp, loss, recomputed logits -> G, dW, dH).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload llama8b] [--impl lce|reference]

Prints one JSON line (rank 0). `value` is valid tokens/s with inputs resident in
HBM; `e2e` is the same metric through the public call with H and targets copied
from pinned host memory and the loss read back every step (W, the weight
matrix, stays resident as in training). Under torchrun each rank runs its own
batch (independent problems, no collective): weak scaling.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused linear-CE fwd+bwd valid tokens/sec; % of dense BF16 tensor peak"
UNIT = "valid tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# DRAM bytes (read + write) per backward k_gemm launch of the llama8b shape,
# from an ncu capture of a reduced-V case with the same per-launch tile
# counts; valid only for the kernel sources it was captured from (sha256
# prefix below) and the default vocab chunk, else reported null.
NCU_TRAFFIC = {"workload": "llama8b", "kernel": "backward", "bytes_per_launch": 1198.7e6,
               "src_sha256": "11cb97543dbc797e"}


def kernel_src_sha256(texts=None) -> str:
    """Hash of the code that defines the GEMM kernels (engine and PTX
    wrappers), with // comments and blank lines removed so that comment edits
    leave it unchanged; the launch configuration is pinned separately
    (default vocab chunk, no options). `texts` replaces the files' contents."""
    import hashlib
    import re
    if texts is None:
        texts = []
        for f in ("lce_gemm.cuh", "tc_ptx.cuh"):
            with open(os.path.join(ROOT, "chunked_vocab_cross_gb300", "csrc", f), encoding="utf-8") as fh:
                texts.append(fh.read())
    h = hashlib.sha256()
    for text in texts:
        code = [re.sub(r"\s*//.*$", "", line).rstrip() for line in text.splitlines()]
        h.update("\n".join(line for line in code if line).encode())
    return h.hexdigest()[:16]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons every 50 ms, each sample with its
    timestamp; summary() keeps the samples inside the window set by mark()
    (the timed region). Start it a few untimed steps before timing so that
    nvidia-smi is already sampling when the timed region begins."""
    Q = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.window = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits", "-lms", "50",
                 "-i", str(self.index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def mark(self, t0: float, t1: float):
        """The timed region, as host wall-clock times (time.time())."""
        self.window = (t0, t1)

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    @staticmethod
    def _epoch(stamp: str):
        import datetime
        for fmt in ("%Y/%m/%d %H:%M:%S.%f", "%Y/%m/%d %H:%M:%S"):
            try:
                return datetime.datetime.strptime(stamp, fmt).timestamp()
            except ValueError:
                continue
        return None

    def summary(self):
        rows = []
        for line in (self.out or "").strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != 8:
                continue
            try:
                rows.append((self._epoch(parts[0]), float(parts[1]), float(parts[2]), parts[4:]))
            except ValueError:
                continue
        inside = rows
        if self.window is not None:
            t0, t1 = self.window
            inside = [r for r in rows if r[0] is not None and t0 <= r[0] <= t1]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no clock sample inside the timed region"],
                    "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for _, _, _, flags in inside for n, f in zip(names, flags) if f.lower() == "active"})
        return {"sm_mhz": float(np.median([r[1] for r in inside])), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": reasons, "samples": len(inside)}


def dist_setup(gpus: int):
    import torch
    rank, world = int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1))
    local = int(os.environ.get("LOCAL_RANK", 0))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device: str = "cuda") -> float:
    """Slowest rank's value (the step time every rank waits for)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int, device: str = "cuda") -> float:
    """Whole-job total (valid tokens of all ranks)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t)
    return float(t.item())


def _oracle_rows(x, rows: int):
    """H rows and targets of the first `rows` valid positions (as stored:
    bf16 bit patterns or fp32), the oracle's input for a sample."""
    valid = np.nonzero(x.targets != -100)[0][:rows]
    return np.ascontiguousarray(x.H[valid]), np.ascontiguousarray(x.targets[valid])


def cpu_oracle_time(x, rows: int, threads: int) -> float:
    """Seconds the plain C++ fp64 oracle, as it stands, takes for the
    forward + backward of the first `rows` valid rows of the batch over the
    full V and d (their loss, their dH rows and their contribution to every
    dW row), on `threads` host threads."""
    from oracle import cpp_oracle
    Hs, ts = _oracle_rows(x, rows)
    t0 = time.perf_counter()
    cpp_oracle.forward_backward(Hs, x.W, ts, -100, threads=threads, bf16=x.bf16)
    return time.perf_counter() - t0


def cpu_oracle_sample_rows(x, budget_s: float, threads: int) -> int:
    """Rows of a sample that takes about `budget_s` (from a timed 16-row run)."""
    nv = int((x.targets != -100).sum())
    r0 = min(16, nv)
    t0 = cpu_oracle_time(x, r0, threads)
    return int(max(r0, min(nv, round(budget_s / max(t0, 1e-6) * r0))))


def cpu_oracle_rate(x, budget_s: float):
    """The C++ oracle's rate in valid tokens/s on a bounded sample of the
    batch (about `budget_s` of work), with the thread count it used."""
    from oracle import cpp_oracle
    threads = cpp_oracle.default_threads()
    rows = cpu_oracle_sample_rows(x, budget_s, threads)
    el = cpu_oracle_time(x, rows, threads)
    return rows / el, el, rows, threads


def workload_desc(x, nv):
    w = x.workload
    return {"workload": f"{w.name}: N={w.N} ({w.seqs}x{w.N // w.seqs}), d={w.d}, V={w.V}, Nv={nv}, {w.dtype}, "
                        f"targets {w.targets}, padding {w.padding}, W~N(0,1/d)*{w.w_scale}, seed {w.seed}",
            "N": w.N, "d": w.d, "V": w.V, "n_valid": int(nv),
            "l2": "inputs larger than L2 (W alone %.2f GB > 129 MB L2); no flush needed" % (w.V * w.d * 2 / 1e9)}


def run_reference(args):
    """The reference arm: the plain C++ fp64 oracle on the host cores. One
    step = the oracle's forward + backward of the first R valid rows of the
    batch over the full V and d (R sized so a step takes about
    LCE_REF_STEP_S seconds, default 6); ms_per_step is the timed step."""
    rank, world = int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1))
    if rank != 0:
        return
    from oracle import cpp_oracle
    from synth_inputs import make_inputs
    x = make_inputs(args.workload)
    nv = int((x.targets != -100).sum())
    threads = cpp_oracle.default_threads()
    budget = float(os.environ.get("LCE_REF_STEP_S", "6"))
    rows = cpu_oracle_sample_rows(x, budget, threads)
    for _ in range(args.warmup):
        cpu_oracle_time(x, min(16, rows), threads)
    times = [cpu_oracle_time(x, rows, threads) for _ in range(args.steps)]
    ms_step = 1e3 * float(np.mean(times))
    value = rows / (ms_step / 1e3)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "ms_per_step_median": 1e3 * float(np.median(times)),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_desc(x, nv),
            "step": f"forward + backward of the first {rows} of the batch's {nv} valid rows over full "
                    f"V={x.workload.V} and d={x.workload.d} (a bounded sample; the whole batch would take "
                    f"about {nv / value:.0f} s at this rate)",
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "threads": threads, "kind": "oracle",
                             "sample": f"each step: the first {rows} valid rows of the batch, plain C++ fp64 "
                                       f"oracle forward + backward over full V and d on {threads} std::threads"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_cpu_table(args):
    """The C++ oracle's rate on every workload, on this host's cores: the
    small workloads (tiny, gpt1b, smallvocab) in full, the large ones
    (llama8b, vocab256k) as the full-row LSE sweep every sampled parity check
    needs plus a forward + backward of their first valid rows, with the
    per-row rates and the whole-batch time extrapolated from them. One JSON
    line per workload."""
    from oracle import cpp_oracle
    from synth_inputs import make_inputs
    threads = cpp_oracle.default_threads()
    names = args.cpu_table.split(",") if args.cpu_table != "all" else \
        ["tiny", "gpt1b", "smallvocab", "llama8b", "vocab256k"]
    for name in names:
        x = make_inputs(name)
        w = x.workload
        nv = int((x.targets != -100).sum())
        rec = {"cpu_table": name, "N": w.N, "d": w.d, "V": w.V, "n_valid": nv, "threads": threads,
               "kind": "plain C++ fp64 oracle (std::thread)"}
        if name in ("tiny", "gpt1b", "smallvocab"):
            t0 = time.perf_counter()
            cpp_oracle.forward_backward(x.H, x.W, x.targets, -100, threads=threads, bf16=x.bf16)
            el = time.perf_counter() - t0
            rec.update(what="forward + backward of the whole batch", seconds=el, valid_tokens_per_s=nv / el)
        else:
            t0 = time.perf_counter()
            cpp_oracle.forward(x.H, x.W, x.targets, -100, threads=threads, bf16=x.bf16)
            sweep = time.perf_counter() - t0
            rows = 64
            el = cpu_oracle_time(x, rows, threads)
            rec.update(what="full-row LSE sweep (every valid row, forward only) + forward + backward of the "
                            f"first {rows} valid rows",
                       lse_sweep_seconds=sweep, lse_rows_per_s=nv / sweep,
                       fwd_bwd_rows=rows, fwd_bwd_seconds=el, valid_tokens_per_s=rows / el,
                       whole_batch_seconds_extrapolated=nv * el / rows)
        print(json.dumps(rec), flush=True)


def run_embedding(args):
    """Input-embedding lookup skipping padding + its gradient accumulated into
    an fp32 dW (the tied-W training step's input side), on the workload's
    tokens (padding -> id 0). HBM-bound: the roofline is algorithmic bytes
    (valid W rows read, E written, valid dE rows read, the touched dW rows
    read and written) over the measured copy bandwidth. The step (seven
    small launches with a caller workspace) is captured in a CUDA graph and
    replayed, as a training step would run it; the eager time (one host call
    per launch) is reported beside it."""
    import torch

    import chunked_vocab_cross_gb300 as lce
    from chunked_vocab_cross_gb300.build import build
    from synth_inputs import make_inputs
    torch.cuda.set_device(0)
    build()
    x = make_inputs(args.workload)
    w = x.workload
    pad = 0
    tok = np.where(x.targets == -100, pad, x.targets)
    nv = int((tok != pad).sum())
    distinct = int(np.unique(tok[tok != pad]).size)
    W = host_tensors(x)[1].cuda()
    t = torch.from_numpy(tok).cuda()
    dE = torch.randn(w.N, w.d, device="cuda").to(W.dtype)
    dW = torch.zeros(w.V, w.d, dtype=torch.float32, device="cuda")
    E = torch.empty(w.N, w.d, dtype=W.dtype, device="cuda")
    ws = torch.empty(lce.embedding_workspace_size(w.N, w.d), dtype=torch.uint8, device="cuda")
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")   # 256 MB > L2, written between steps
    stream = torch.cuda.Stream()

    def step():
        lce.embedding_forward(W, t, pad, out=E, stream=stream)
        lce.embedding_backward(dE, t, pad, w.V, dW=dW, accumulate=True, workspace=ws, stream=stream)

    def timed(run, n):
        ms = []
        with torch.cuda.stream(stream):
            for _ in range(n):
                flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                run()
                e1.record(stream)
                torch.cuda.synchronize()
                ms.append(e0.elapsed_time(e1))
        return float(np.median(ms))

    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            step()
    torch.cuda.synchronize()
    eager = timed(step, args.steps)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for _ in range(3):
            graph.replay()
    med = timed(graph.replay, args.steps)
    status = lce.device_status()
    elt = W.element_size()
    bytes_alg = nv * w.d * elt + w.N * w.d * elt + nv * w.d * elt + distinct * w.d * 8
    peaks, src = load_peaks()
    peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    gbs = bytes_alg / (med / 1e3) / 1e9
    print(json.dumps({
        "metric": "input-embedding lookup + gradient (tied W), tokens/s", "value": w.N / (med / 1e3),
        "unit": "tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": med,
        "ms_per_step_eager": eager, "higher_is_better": True, "dtype": ("bf16" if x.bf16 else "f32") + " (fp32 dW)",
        "data": "synthetic",
        "config": {"workload": w.name, "N": w.N, "d": w.d, "V": w.V, "valid": nv, "distinct_tokens": distinct,
                   "l2": "256 MB buffer written between steps", "launch": "CUDA graph replay of the step"},
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                     "traffic": None, "peak_kind": f"hbm_gbs ({src})", "bytes_per_step": bytes_alg},
        "device_status": status}), flush=True)


def host_tensors(x):
    """(H, W) of a synthetic batch as CPU torch tensors of the workload's
    dtype: bf16 bit patterns reinterpreted, fp32 arrays as they are."""
    import torch
    if x.bf16:
        return (torch.from_numpy(x.H.view(np.int16)).view(torch.bfloat16),
                torch.from_numpy(x.W.view(np.int16)).view(torch.bfloat16))
    return torch.from_numpy(x.H), torch.from_numpy(x.W)


def eager_context(H, W, t, nv, steps):
    """Context only (not a baseline of this metric's reference arm): the same
    fwd+bwd in eager PyTorch, which materialises the N x V logits (cuBLAS bf16
    GEMMs, F.cross_entropy over fp32 logits, autograd). Time per step with
    CUDA events and the peak device memory it adds; None if it does not fit."""
    import torch
    import torch.nn.functional as F
    Hr = H.detach().clone().requires_grad_(True)
    Wr = W.detach().clone().requires_grad_(True)

    def step():
        Hr.grad = None
        Wr.grad = None
        loss = F.cross_entropy((Hr @ Wr.t()).float(), t, ignore_index=-100)
        loss.backward()
        return loss

    try:
        torch.cuda.synchronize()
        for _ in range(2):
            step()
        torch.cuda.synchronize()
        base = torch.cuda.memory_allocated()
        torch.cuda.reset_peak_memory_stats()
        n = max(3, min(steps, 10))
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record()
        for _ in range(n):
            step()
        s1.record()
        torch.cuda.synchronize()
        ms = s0.elapsed_time(s1) / n
        peak = torch.cuda.max_memory_allocated() - base
    except torch.cuda.OutOfMemoryError:
        return None
    finally:
        del Hr, Wr
        torch.cuda.empty_cache()
    return {"ms_per_step": ms, "valid_tokens_per_s": nv / (ms / 1e3), "peak_extra_bytes": int(peak),
            "what": "eager PyTorch: H @ W^T (bf16 cuBLAS), F.cross_entropy on fp32 logits, autograd; "
                    "materialises N x V logits; context, not this path"}


def cublas_context(H, W, t, nv, reps=5):
    """Context only: the three contractions of the step as plain cuBLAS bf16
    GEMMs on the valid rows (torch.matmul, materialised outputs): logits
    Hc @ W^T [Nv, V], dH = G @ W [Nv, d] and dW = G^T @ Hc [V, d] for a bf16
    G [Nv, V]. Each timed alone with CUDA events (median of `reps` after two
    warm-ups); the library runs these three plus the logits recomputation
    (four contractions of 2*Nv*d*V FLOPs). None if it does not fit."""
    import torch
    try:
        Hc = H[t != -100].contiguous()
        G = (torch.randn(Hc.shape[0], W.shape[0], device=H.device) * 1e-6).to(H.dtype)
        out = {}
        for name, fn in (("logits", lambda: Hc @ W.t()), ("dH", lambda: G @ W), ("dW", lambda: G.t() @ Hc)):
            for _ in range(2):
                fn()
            times = []
            for _ in range(reps):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                fn()
                e1.record()
                torch.cuda.synchronize()
                times.append(e0.elapsed_time(e1))
            out[name + "_ms"] = float(np.median(times))
        flops = 2.0 * Hc.shape[0] * H.shape[1] * W.shape[0]
        out["tflops_each"] = {k[:-3]: flops / (v / 1e3) / 1e12 for k, v in list(out.items())}
        # the four contractions this path executes per step (logits twice, dH,
        # dW) back to back, as long a run as the timed steps: the rate under
        # the same power cap
        def four():
            Hc @ W.t()
            Hc @ W.t()
            G @ W
            G.t() @ Hc
        for _ in range(2):
            four()
        n = 10
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(n):
            four()
        e1.record()
        torch.cuda.synchronize()
        out["four_contractions_ms"] = e0.elapsed_time(e1) / n
        out["four_contractions_tflops"] = 4 * flops / (out["four_contractions_ms"] / 1e3) / 1e12
        out["what"] = ("cuBLAS bf16 GEMMs of the same shapes with materialised outputs: each alone (median of "
                       "5, burst), and the four this path executes per step (logits twice, dH, dW) back to back "
                       "over 10 steps; context only")
        del Hc, G
        return out
    except torch.cuda.OutOfMemoryError:
        return None
    finally:
        torch.cuda.empty_cache()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="llama8b")
    ap.add_argument("--impl", default="lce", choices=["lce", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--vocab", type=int, default=0,
                    help="override V (a smaller case with the same per-launch shape, for profiling)")
    ap.add_argument("--vocab-chunk", type=int, default=0, help="backward vocab chunk (0 = library default)")
    ap.add_argument("--optim", default="none", choices=["none", "sgd", "adamw"],
                    help="fuse an optimizer step on W into the backward (no dW buffer; W is updated every step)")
    ap.add_argument("--optim-state", default="fp32", choices=["fp32", "bf16"],
                    help="dtype of the fused optimizer's state (moments / momentum buffer)")
    ap.add_argument("--dw-dtype", default="fp32", choices=["fp32", "bf16"],
                    help="dtype of the dW output (bf16: each fp32 accumulator rounded once, half the dW bytes)")
    ap.add_argument("--two-call", action="store_true",
                    help="forward (storing the per-row lse) and backward from the stored lse as two calls")
    ap.add_argument("--token-chunk", type=int, default=0,
                    help="process the rows this many positions at a time (0 = all at once)")
    ap.add_argument("--embedding", action="store_true",
                    help="time the input-embedding lookup + its gradient (tied W) instead of the loss path")
    ap.add_argument("--no-context", action="store_true",
                    help="skip the eager PyTorch context measurement (logits materialised)")
    ap.add_argument("--row-gather", action="store_true",
                    help="GEMMs read H's valid rows by TMA gather4 instead of a compacted copy")
    ap.add_argument("--cpu-table", default="",
                    help="time the C++ oracle per workload ('all' or a comma list) instead of the GPU path")
    args = ap.parse_args()
    if args.cpu_table:
        run_cpu_table(args)
        return
    if args.impl == "reference":
        run_reference(args)
        return
    if args.embedding:
        run_embedding(args)
        return

    import torch

    import chunked_vocab_cross_gb300 as lce
    from chunked_vocab_cross_gb300.build import build
    from synth_inputs import make_inputs

    rank, world, local = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0:
        build()
    barrier(world)

    # each rank draws its own batch (seed = rank): independent problems
    over = {"seed": rank}
    if args.vocab:
        over["V"] = args.vocab
    x = make_inputs(args.workload, **over)
    nv = int((x.targets != -100).sum())
    w = x.workload
    H_cpu, W_cpu = host_tensors(x)
    H_host = H_cpu.pin_memory()
    t_host = torch.from_numpy(x.targets).pin_memory()
    H = H_host.to(dev)
    W = W_cpu.to(dev)
    t = t_host.to(dev)
    loss = torch.empty((), dtype=torch.float32, device=dev)
    dH = torch.empty_like(H)
    fused = args.optim != "none"
    dw_dtype = torch.bfloat16 if args.dw_dtype == "bf16" else torch.float32
    dW = None if fused else torch.empty(W.shape, dtype=dw_dtype, device=dev)
    ws = torch.empty(lce.workspace_size(w.N, w.d, w.V, dtype=W.dtype, vocab_chunk=args.vocab_chunk,
                                        token_chunk=args.token_chunk,
                                        fused_optimizer=fused, row_gather=args.row_gather),
                     dtype=torch.uint8, device=dev)
    lse_buf = torch.empty(w.N, dtype=torch.float32, device=dev) if args.two_call else None
    state_dtype = torch.bfloat16 if args.optim_state == "bf16" else torch.float32
    opt = lce.FusedOptimizer(W, args.optim, lr=1e-5, state_dtype=state_dtype) if fused else None

    def run(Hx, tx, lx, dHx):
        kw = dict(workspace=ws, vocab_chunk=args.vocab_chunk, token_chunk=args.token_chunk,
                  row_gather=args.row_gather)
        if opt is not None:
            opt.step_count += 1
            kw["optim"] = opt.optim_args()
        if args.two_call:
            # forward storing lse, then the backward alone from it
            lce.lce_run(Hx, W, tx, -100, loss=lx, lse=lse_buf, **kw)
            lce.lce_run(Hx, W, tx, -100, dH=dHx, dW=dW, lse_in=lse_buf, **kw)
        else:
            lce.lce_run(Hx, W, tx, -100, loss=lx, dH=dHx, dW=dW, **kw)

    def step():
        run(H, t, loss, dH)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    lce.device_status()

    # ------------------------------------------------------------ timed region
    stream = torch.cuda.current_stream()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        for _ in range(3):   # untimed, while the sampler starts
            step()
        torch.cuda.synchronize()
        l0 = lce.launch_count()   # this library's launches inside the timed region
        t_wall0 = time.time()
        # an event before every step as well (steps start with an ordinary
        # launch, so the events do not split a dependent-launch chain)
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ev0.record(stream)
        for i in range(args.steps):
            if i:
                evs[i - 1].record(stream)
            step()
        ev1.record(stream)
        torch.cuda.synchronize()
        clk.mark(t_wall0, time.time())
    marks = [ev0] + evs[:args.steps - 1] + [ev1]
    step_ms = [marks[i].elapsed_time(marks[i + 1]) for i in range(args.steps)]
    barrier(world)
    launches = lce.launch_count() - l0
    ms_step = max_over_ranks(ev0.elapsed_time(ev1) / args.steps, world)
    status = lce.device_status()
    nv_all = sum_over_ranks(nv, world)
    value = nv_all / (ms_step / 1e3)

    # -------------------------------------------- per-phase events (roofline)
    lce.profile_begin()
    prof_steps = max(3, min(args.steps, 10))
    for _ in range(prof_steps):
        step()
    phases = lce.profile_end()
    torch.cuda.synchronize()

    # ------------------------------------------------ end to end (host buffers)
    # Every step copies its H and targets from pinned host memory and reads
    # its loss back. The copies run on a second stream into two alternating
    # device buffers, so the copy for step i+1 overlaps step i's compute; a
    # buffer is refilled only after the step that used it has finished.
    e2e_loss = torch.empty((), dtype=torch.float32).pin_memory()
    copy_stream = torch.cuda.Stream(device=dev)
    bufs = [(torch.empty_like(H), torch.empty_like(t)) for _ in range(2)]
    copied = [torch.cuda.Event() for _ in range(2)]
    freed = [torch.cuda.Event() for _ in range(2)]
    freed_set = [False, False]

    def issue_copy(i):
        b = i % 2
        with torch.cuda.stream(copy_stream):
            if freed_set[b]:
                copy_stream.wait_event(freed[b])
            bufs[b][0].copy_(H_host, non_blocking=True)
            bufs[b][1].copy_(t_host, non_blocking=True)
            copied[b].record(copy_stream)

    def e2e_step(i, n):
        b = i % 2
        stream.wait_event(copied[b])
        H_e, t_e = bufs[b]
        if opt is None and args.dw_dtype == "fp32" and not (args.row_gather or args.two_call or args.token_chunk):
            l, _, _ = lce.lce_forward_backward(H_e, W, t_e, -100, vocab_chunk=args.vocab_chunk, workspace=ws)
        else:
            l = torch.empty((), dtype=torch.float32, device=dev)
            run(H_e, t_e, l, torch.empty_like(H_e))
        freed[b].record(stream)
        freed_set[b] = True
        e2e_loss.copy_(l, non_blocking=True)
        if i + 2 < n:
            issue_copy(i + 2)

    def e2e_run(n):
        issue_copy(0)
        if n > 1:
            issue_copy(1)
        for i in range(n):
            e2e_step(i, n)

    e2e_run(2)
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    copy_stream.wait_event(e0)
    e2e_run(args.steps)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world)

    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    context = None if args.no_context else eager_context(H, W, t, nv, args.steps)
    cublas = None if args.no_context else cublas_context(H, W, t, nv)

    peaks, peak_src = load_peaks()
    useful_flops = 6.0 * nv * w.d * w.V
    executed_flops = 8.0 * nv * w.d * w.V
    tflops_useful = useful_flops / (ms_step / 1e3) / 1e12 * 1.0
    # dominant kernel: largest share of the profiled step time. The forward is
    # one k_gemm<LSE> launch (2*Nv*d*V FLOPs); the backward is one k_gemm<BWD>
    # launch per vocab chunk plus one (3 * 2*Nv*d*V FLOPs over all of them).
    gemm_flops = {"logits_lse": 2.0 * nv * w.d * w.V, "backward": 6.0 * nv * w.d * w.V}
    name = max(gemm_flops, key=lambda k: phases[k]["ms"])
    ph = phases[name]
    per_launch_ms = ph["ms"] / max(1, ph["launches"])
    flops_launch = gemm_flops[name] / max(1, ph["launches"] // prof_steps)
    achieved = flops_launch / (per_launch_ms / 1e3) / 1e12
    traffic = None
    if (NCU_TRAFFIC["workload"] == w.name and NCU_TRAFFIC["kernel"] == name and w.V == 128256
            and NCU_TRAFFIC["src_sha256"] == kernel_src_sha256() and not args.vocab_chunk and opt is None
            and args.dw_dtype == "fp32" and not (args.row_gather or args.two_call or args.token_chunk)):
        traffic = NCU_TRAFFIC["bytes_per_launch"]
    # The roofline is quoted against the burst bf16 peak (a 20-step timed
    # region is well under a second of work); the sustained peak, measured
    # over seconds under the power cap, is given beside it.
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    peak_sus = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    total_prof = sum(p["ms"] for p in phases.values())
    cpu = None
    if not args.no_cpu_baseline:
        rate, el, rows, threads = cpu_oracle_rate(x, args.cpu_budget)
        cpu = {"value": rate, "unit": UNIT, "cores": threads, "threads": threads, "kind": "oracle",
               "sample": f"first {rows} valid rows of the batch, plain C++ fp64 oracle forward + backward over "
                         f"full V={w.V} and d={w.d} on {threads} std::threads ({el:.1f} s), "
                         f"as valid tokens/s"}
    clocks = clk.summary()
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms_step, "ms_per_step_median": float(np.median(step_ms)),
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if x.bf16 else "f32 (bf16 hi/lo split products)",
        "data": "synthetic",
        "config": workload_desc(x, nv),
        "pct_dense_bf16_peak": {
            "useful_tflops": tflops_useful,
            "of_burst": tflops_useful / peak,
            "of_sustained": tflops_useful / peak_sus, "peaks": peak_src,
            "note": "useful FLOPs = 6*Nv*d*V; the path executes 8*Nv*d*V (logits recomputed in backward)"},
        "roofline": {"bound": "tensor", "kernel": f"k_gemm ({name})", "achieved": achieved, "peak": peak,
                     "unit": "TFLOP/s", "frac": achieved / peak, "traffic": traffic,
                     "peak_kind": f"bf16_tflops burst ({peak_src})", "frac_of_sustained": achieved / peak_sus,
                     "flops_per_launch": flops_launch, "ms_per_launch": per_launch_ms},
        "phases_ms_per_step": {k: v["ms"] / prof_steps for k, v in phases.items()},
        "phase_share": {k: (v["ms"] / total_prof if total_prof else None) for k, v in phases.items()},
        "cpu_baseline": cpu,
        "e2e": {"value": nv / (e2e_ms / 1e3) * world, "unit": UNIT,
                "h2d_bytes_per_step": int(H.numel() * H.element_size() + t.numel() * 8), "d2h_bytes_per_step": 4,
                "resident": "W (weights)", "ms_per_step": e2e_ms,
                "copies": "H2D on a second stream into two alternating buffers (overlapping the previous step)",
                "call": "lce_forward_backward(H, W, targets, ...) with a caller workspace"},
        "gpu_launches": int(launches),
        "device_status": status,
        "clocks": clocks,
        "workspace_bytes": int(ws.numel()),
        "vocab_chunk": args.vocab_chunk or "library default (6144-row chunks evened out over V)",
        "fused_optimizer": None if opt is None else f"{args.optim} on W in place (state {args.optim_state} [V,d]; no dW buffer)",
        "dW_dtype": None if opt is not None else args.dw_dtype,
        "row_gather": bool(args.row_gather),
        "two_call": bool(args.two_call),
        "token_chunk": args.token_chunk or None,
        "logits_bytes_avoided": int(w.N * w.V * 4),
        "context_torch_eager": context,
        "context_cublas_gemms": cublas,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
