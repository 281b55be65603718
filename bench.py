"""Benchmark: exact-attention forward TFLOP/s on GB300.

One step = one fa_fwd call over the whole workload (all of the hot path: tile
loads, QK^T, masking, online softmax, PV, epilogue) on inputs resident in HBM.
Workload at one GPU: B=8, H=32, Nq=Nk=8192, d=128, bf16, causal
(4*B*H*N^2*d/2 = 4.398 TFLOP per step); its 1.6 GB of inputs exceed the
129 MB L2, so no flush is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl fa|reference]
                  [--pass fwd|bwd]

``--varlen`` times fa_fwd_varlen on a packed batch of 32 sequences with
lengths drawn uniformly from 512..8192 (seeded; token-major [total, 16, 128]
bf16, causal within each sequence); FLOPs are counted exactly per sequence
(4*H*d per allowed (query, key) pair).

``--pass bwd`` times the backward instead (one step = one fa_bwd call: the
per-row D / LSE kernel, the tensor-core gradient kernel and the dq rounding),
reporting 2.5x the forward's FLOPs (five products of 2*Nq*Nk*d where the
forward has two), the usual convention for attention backward.

Under torchrun (N > 1) each rank runs its own copy of the workload on its own
GPU (weak scaling; the heads are independent, so nothing is exchanged); the
timed region is bracketed by barriers and the max over ranks is reported.
``--impl reference`` times the float64 CPU oracle on a bounded sample of the
same workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import glob
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attn fwd TFLOP/s (4·B·H·N²·d, ½ if causal) and % of GB300 dense peak"
METRIC_BWD = "attn bwd TFLOP/s (10·B·H·N²·d, ½ if causal) and % of GB300 dense peak"


# Sources a kernel's behaviour depends on: its template, instantiation,
# shared headers and the host code that encodes its tensor maps and launches.
KERNEL_SOURCES = {
    "fa_tc_fwd_kernel": ["fa_tc.cuh", "fa_tc_bf16_d128.cu", "fa_tc_bf16_d64.cu", "fa_tc_f16_d128.cu",
                         "fa_tc_f16_d64.cu", "fa_tc_f32_d64.cu", "fa_tc_f32s_d64.cu",
                         "fa_tc_f32s_d128.cu"],
    "fa_bwd": ["fa_bwd.cuh", "fa_bwd_bf16.cu", "fa_bwd_f16.cu", "fa_bwd_aux.cu"],
}
COMMON_SOURCES = ["ptx.cuh", "fa_wait.cuh", "fa_internal.h", "fa_api.cu"]


def code_only(text: str) -> str:
    """C/C++ source without its comments and with whitespace runs collapsed
    (string literals kept as they are): an edit of comments or layout leaves
    the code, and so the validity of a profile taken on it, unchanged."""
    out, i, n = [], 0, len(text)
    while i < n:
        if text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        elif text[i] == '"':
            j = i + 1
            while j < n and text[j] != '"':
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        else:
            out.append(text[i])
            i += 1
    return " ".join("".join(out).split())


def kernel_source_hash(kernel: str, read=None) -> str:
    """Hash of the code (comments and layout aside) of the sources of the
    kernel family named by the key's prefix; read(name) gives a source's
    text (default: the working tree)."""
    fam = next(f for f in KERNEL_SOURCES if kernel.startswith(f))
    if read is None:
        def read(name):
            with open(os.path.join(ROOT, "exact_attention_57_gb300", "csrc", name)) as f:
                return f.read()
    h = hashlib.sha256()
    for name in sorted(KERNEL_SOURCES[fam] + COMMON_SOURCES):
        h.update(name.encode())
        h.update(code_only(read(name)).encode())
    return h.hexdigest()[:16]


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def profiled_traffic(kernel: str, workload: str):
    """(DRAM bytes per launch, note) from the committed ncu summary, if it was
    taken on the current kernel sources; else (None, None).  The note says
    how to read the figure (e.g. a lower bound when the capture's writes
    stayed in L2)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None, None
    with open(path) as f:
        rec = json.load(f)
    ent = rec.get(kernel, {}).get(workload)
    if not ent or ent.get("source_hash") != kernel_source_hash(kernel):
        return None, None
    return ent.get("dram_bytes_per_launch"), ent.get("note")


class ClockSampler:
    """nvidia-smi clocks/throttle reasons sampled every 100 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


def max_over_ranks(x: float, device=None) -> float:
    """Max of a per-rank scalar over every rank (identity without a group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def oracle_inputs(w):
    """The workload's seeded CPU inputs as float32 numpy arrays for the oracle."""
    from exact_attention_57_gb300.workloads import workload_inputs
    return tuple(t.float().numpy() for t in workload_inputs(w))


def cpu_oracle_sample(w, budget_s: float, seed: int = 7, arrays=None):
    """Time the float64 oracle on sampled query rows of the workload.

    Returns (GFLOP/s in the metric's units, threads, description).  Rows are
    drawn uniformly over (b, h, i); the metric FLOPs of row i are
    4*d*|K(i)| (|K(i)| = i+1 keys when causal), so the rate is comparable with
    the GPU's 4*B*H*N^2*d/2.
    """
    import numpy as np

    import oracle

    qf, kf, vf = arrays if arrays is not None else oracle_inputs(w)
    causal = w.causal[0]
    rng = np.random.default_rng(seed)
    threads = os.cpu_count() or 1

    def run(n):
        rows = rng.integers(0, w.B * w.H * w.Nq, size=n)
        i = rows % w.Nq
        keys = np.minimum(i + 1, w.Nk) if causal else np.full(n, w.Nk)
        flops = float(np.sum(4.0 * w.d * keys))
        t0 = time.perf_counter()
        oracle.attn_rows(qf, kf, vf, rows, w.scale, causal, nthreads=threads)
        return flops, time.perf_counter() - t0

    n = 256
    flops, dt = run(n)
    while dt < budget_s / 8 and n < 1 << 20:
        n *= 4
        flops, dt = run(n)
    if dt < budget_s / 2:
        n = int(n * budget_s / max(dt, 1e-3))
        flops, dt = run(n)
    desc = (f"{n} query rows sampled uniformly from the workload, full key range each "
            f"({'causal' if causal else 'non-causal'}), float64, {threads} threads")
    return flops / dt / 1e9, threads, desc, dt


def run_reference(args, w):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    rates = []
    per_step = max(2.0, 120.0 / max(1, args.steps + args.warmup))
    tot_t = 0.0
    arrays = oracle_inputs(w)
    for s in range(args.warmup + args.steps):
        g, threads, desc, dt = cpu_oracle_sample(w, per_step, seed=100 + s, arrays=arrays)
        if s >= args.warmup:
            rates.append(g)
            tot_t += dt
    value = statistics.median(rates) / 1e3  # TFLOP/s
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * tot_t / max(1, args.steps), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "Nq": w.Nq, "Nk": w.Nk, "d": w.d,
                   "causal": w.causal[0], "io_dtype": "bf16"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads,
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="fa", choices=["fa", "reference"])
    ap.add_argument("--workload", default=None)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--splits", type=int, default=None,
                    help="run fa_fwd_splitkv with this many key chunks (0 = automatic)")
    ap.add_argument("--pass", dest="which", default="fwd", choices=["fwd", "bwd"])
    ap.add_argument("--no-staging", action="store_true",
                    help="fp32 workloads: time fa_fwd instead of fa_fwd_staged")
    ap.add_argument("--varlen", action="store_true",
                    help="packed variable-length batch through fa_fwd_varlen")
    ap.add_argument("--no-graph", action="store_true",
                    help="launch the timed steps one by one instead of replaying a CUDA graph")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)

    from exact_attention_57_gb300.workloads import BENCH_WORKLOAD, PROFILE_WORKLOADS, WORKLOADS
    w = {**WORKLOADS, **PROFILE_WORKLOADS}[args.workload or BENCH_WORKLOAD]
    if args.impl == "reference":
        return run_reference(args, w)

    import torch
    import torch.distributed as dist

    from exact_attention_57_gb300 import fa
    from exact_attention_57_gb300.workloads import DTYPE_NAMES

    ws, rank, local = dist_env()
    if ws > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if ws > 1 else 0)
    torch.cuda.set_device(dev)
    causal = w.causal[0]
    tdt = w.torch_dtype

    # Inputs drawn on the device (seeded per rank), resident before timing.
    g = torch.Generator(device=dev).manual_seed(w.seed + 1000 * rank)
    q = torch.randn(w.B, w.H, w.Nq, w.d, device=dev, generator=g).to(tdt)
    k = torch.randn(w.B, w.H, w.Nk, w.d, device=dev, generator=g).mul_(w.k_mult).to(tdt)
    v = torch.randn(w.B, w.H, w.Nk, w.d, device=dev, generator=g).to(tdt)
    o = torch.empty_like(q)
    lse = torch.empty(w.B, w.H, w.Nq, device=dev, dtype=torch.float32)
    # A workload whose tensors fit in L2 gets copies used in turn, together
    # at least twice the L2 size, so that each step reads its inputs from HBM
    # as a large one does (no L2 flush between steps is needed either way).
    l2_bytes = torch.cuda.get_device_properties(dev).L2_cache_size
    set_bytes = sum(t.numel() * t.element_size() for t in (q, k, v, o, lse))
    copies = [(q, k, v, o, lse)]
    if set_bytes < 2 * l2_bytes and not args.varlen and args.which == "fwd":
        n_copies = min(256, -(-2 * l2_bytes // set_bytes))
        copies += [tuple(t.clone() for t in (q, k, v, o, lse)) for _ in range(n_copies - 1)]
    l2_note = ("inputs larger than L2 (no flush)" if len(copies) == 1 and set_bytes >= l2_bytes
               else f"{len(copies)} copies of the tensors used in turn, together "
                    f"{len(copies) * set_bytes / 2 ** 20:.0f} MB >= 2x L2 (no flush)"
               if len(copies) > 1 else "tensors fit in L2: steps after the first may hit L2")
    turn = [0]  # next copy
    stream = torch.cuda.Stream(device=dev)
    sh = stream.cuda_stream
    impl = "simt" if w.dtype == 2 else "tc"

    # fp32 (TF32) workloads run through fa_fwd_staged unless told otherwise:
    # its workspace is allocated here, outside the timed region.
    stage_ws = None
    if w.dtype == 1 and not args.no_staging and args.splits is None:
        sb = fa.fa_fwd_staged_workspace(w.B, w.H, w.Nk, w.d, w.dtype)
        stage_ws = torch.empty(max(sb, 256), dtype=torch.uint8, device=dev)
    wspace = None  # split-KV workspace
    if args.splits is not None:
        wsb = fa.fa_fwd_splitkv_workspace(w.B, w.H, w.Nq, w.d, args.splits if args.splits else 64)
        wspace = torch.empty(max(wsb, 256), dtype=torch.uint8, device=dev)

    bwd = args.which == "bwd"
    varlen = None
    if args.varlen:
        # 32 sequences, lengths uniform in 512..8192, causal within each.
        import numpy as np
        rs = np.random.default_rng(57100 + rank)
        lens = rs.integers(512, 8193, size=32)
        Hv, dv_ = 16, 128
        total = int(lens.sum())
        cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device=dev)
        qv = torch.randn(total, Hv, dv_, device=dev, generator=g).to(torch.bfloat16)
        kv = torch.randn(total, Hv, dv_, device=dev, generator=g).to(torch.bfloat16)
        vv = torch.randn(total, Hv, dv_, device=dev, generator=g).to(torch.bfloat16)
        ov = torch.empty_like(qv)
        lv = torch.empty(Hv, total, device=dev, dtype=torch.float32)
        pairs = float(sum(int(L) * (int(L) + 1) // 2 for L in lens))
        varlen = dict(lens=lens, H=Hv, d=dv_, total=total, cu=cu, q=qv, k=kv, v=vv, o=ov,
                      lse=lv, flops=4.0 * Hv * dv_ * pairs, maxlen=int(lens.max()))
        args.no_e2e = True
        args.no_cpu_baseline = True
    if bwd:
        if w.dtype not in (0, 1, 3):
            raise SystemExit("--pass bwd needs a bf16, fp16 or fp32 workload")
        # forward outputs and upstream gradient, resident before timing
        fa.attention(q, k, v, scale=w.scale, causal=causal, out=o, lse=lse)
        dout = torch.randn(w.B, w.H, w.Nq, w.d, device=dev, generator=g).to(tdt)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        bws = fa.fa_bwd_workspace(w.B, w.H, w.Nq, w.d)
        bwork = torch.empty(bws, dtype=torch.uint8, device=dev)
        args.no_e2e = True
        args.no_cpu_baseline = True

    def step():
        if varlen is not None:
            vl = varlen
            st = fa.fa_fwd_varlen(vl["q"].data_ptr(), vl["k"].data_ptr(), vl["v"].data_ptr(),
                                  vl["o"].data_ptr(), vl["lse"].data_ptr(), vl["cu"].data_ptr(),
                                  vl["cu"].data_ptr(), len(vl["lens"]), vl["H"], vl["total"],
                                  vl["total"], vl["maxlen"], vl["d"], vl["d"] ** -0.5, 1,
                                  fa.FA_DTYPE_BF16, sh)
            if st != fa.FA_OK:
                raise fa.FaError(st, "fa_fwd_varlen")
            return
        if bwd:
            st = fa.fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                           dout.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), w.B,
                           w.H, w.Nq, w.Nk, w.d, w.scale, int(causal), w.dtype,
                           bwork.data_ptr(), bws, sh)
            if st != fa.FA_OK:
                raise fa.FaError(st, "fa_bwd")
            return
        qc, kc, vc, oc, lc = copies[turn[0] % len(copies)]
        turn[0] += 1
        if stage_ws is not None:
            st = fa.fa_fwd_staged(qc.data_ptr(), kc.data_ptr(), vc.data_ptr(), oc.data_ptr(),
                                  lc.data_ptr(), w.B, w.H, w.Nq, w.Nk, w.d, w.scale,
                                  int(causal), w.dtype, stage_ws.data_ptr(), stage_ws.numel(),
                                  sh)
        elif wspace is None:
            st = fa.fa_fwd(qc.data_ptr(), kc.data_ptr(), vc.data_ptr(), oc.data_ptr(),
                           lc.data_ptr(), w.B, w.H, w.Nq, w.Nk, w.d, w.scale, int(causal),
                           w.dtype, sh)
        else:
            st = fa.fa_fwd_splitkv(qc.data_ptr(), kc.data_ptr(), vc.data_ptr(), oc.data_ptr(),
                                   lc.data_ptr(), w.B, w.H, w.Nq, w.Nk, w.d, w.scale,
                                   int(causal), w.dtype, args.splits, wspace.data_ptr(),
                                   wspace.numel(), sh)
        if st != fa.FA_OK:
            raise fa.FaError(st, "fa_fwd")

    # The clock sampler starts before the warm-up, so that no idle gap (in
    # which the GPU would clock down) separates the warm-up from the timed
    # steps.
    sampler = ClockSampler(dev.index) if rank == 0 or ws > 1 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    torch.cuda.synchronize(dev)
    for _ in range(args.warmup):
        step()
    st, word = fa.fa_fwd_status(sh)
    if st != fa.FA_OK:
        raise RuntimeError(f"warm-up device status {word}")
    # The K timed steps are captured once into a CUDA graph on the stream the
    # library launches on, and the timed region replays it: every kernel of
    # the K steps runs back to back, with no host launch gap between steps
    # (which otherwise dominates workloads of a few tens of microseconds).
    # --no-graph launches the steps one by one instead.
    graph = None
    if not args.no_graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for _ in range(args.steps):
                step()
        torch.cuda.synchronize(dev)
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    with torch.cuda.stream(stream):
        ev[0].record(stream)
        if graph is not None:
            graph.replay()
            ev[-1].record(stream)
        else:
            for i in range(args.steps):
                step()
                ev[i + 1].record(stream)
    stream.synchronize()
    torch.cuda.synchronize(dev)
    if ws > 1:
        dist.barrier()
    local_ms = ev[0].elapsed_time(ev[-1])
    total_ms = max_over_ranks(local_ms, dev)
    ms_per_step = total_ms / args.steps
    # per-step times (diagnostic, not the value): the same steps launched one
    # by one, an event between consecutive steps
    if graph is not None:
        with torch.cuda.stream(stream):
            ev[0].record(stream)
            for i in range(args.steps):
                step()
                ev[i + 1].record(stream)
        stream.synchronize()
    clocks = sampler.stop() if sampler else None
    st, word = fa.fa_fwd_status(sh)
    if st != fa.FA_OK:
        raise RuntimeError(f"timed-region device status {word}")
    launch_ms = [ev[i].elapsed_time(ev[i + 1]) for i in range(args.steps)]
    flops_step = varlen["flops"] if varlen is not None else w.flops(causal) * (2.5 if bwd else 1.0)
    # the persistent grid of the timed forward (fa_fwd's own choice; the
    # other entry points run one CTA per query tile)
    plain_fwd = not bwd and varlen is None and stage_ws is None and wspace is None
    grid = None
    if plain_fwd:
        _, ctas, groups, block = fa.fa_fwd_schedule(
            w.B, w.H, w.Nq, w.Nk, w.d, causal, w.dtype,
            torch.cuda.get_device_properties(dev).multi_processor_count)
        if ctas > 0 and block > 0:
            grid = {"schedule": "blocked", "ctas": ctas, "items_per_cta": block}
        elif ctas > 0:
            grid = {"schedule": "persistent", "ctas": ctas, "planes_per_group": groups}
    value = ws * flops_step * args.steps / (total_ms / 1e3) / 1e12

    # End to end through the host-buffer entry point: H2D of q, k, v from
    # pinned memory, the forward, D2H of o and lse, every step.
    e2e = None
    if not args.no_e2e:
        qh, kh, vh = (t.cpu().pin_memory() for t in (q, k, v))
        oh = torch.empty(o.shape, dtype=o.dtype).pin_memory()
        lh = torch.empty(lse.shape, dtype=torch.float32).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in (qh, kh, vh))
        d2h = oh.numel() * oh.element_size() + lh.numel() * 4

        def e2e_step():
            r = fa.fa_fwd_host(qh.data_ptr(), kh.data_ptr(), vh.data_ptr(), oh.data_ptr(),
                               lh.data_ptr(), q.data_ptr(), k.data_ptr(), v.data_ptr(),
                               o.data_ptr(), lse.data_ptr(), w.B, w.H, w.Nq, w.Nk, w.d,
                               w.scale, int(causal), w.dtype, sh)
            if r != fa.FA_OK:
                raise fa.FaError(r, "fa_fwd_host")

        e2e_steps = max(3, min(args.steps, 10))
        for _ in range(2):
            e2e_step()
        if ws > 1:
            dist.barrier()
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            e2e_step()
        dt = max_over_ranks(time.perf_counter() - t0, dev)
        e2e = {"value": ws * flops_step * e2e_steps / dt / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": 1e3 * dt / e2e_steps}

    if rank != 0:
        if ws > 1:
            dist.barrier()
            dist.destroy_process_group()
        return

    peaks, peak_src = measured_peaks()
    # the timed region's average step on this rank (a step is one launch of
    # the forward kernel; two or three launches for staged, split-KV and
    # backward steps, where `achieved` is then a lower bound for the main kernel)
    avg_launch_ms = local_ms / args.steps
    achieved = flops_step / (avg_launch_ms / 1e3) / 1e12
    half_io = w.dtype in (0, 3)   # bf16 / fp16: the same kind::f16 tensor rate
    # SIMT kernels (the plain fp32 forward, every fp32 backward): no tensor
    # cores; the FP32 FMA rate is SMs x 128 lanes x 2 FLOP
    # per cycle at the maximum SM clock.
    simt = w.dtype == 2 or (bwd and w.dtype == 1)
    n_sms = torch.cuda.get_device_properties(dev).multi_processor_count
    fma_peak = n_sms * 128 * 2 * float(peaks.get("sm_max_mhz", 2070.0)) * 1e6 / 1e12
    peak = (float(peaks["bf16_tflops"]) if half_io else
            fma_peak if simt else float(peaks["bf16_tflops"]) / 2.0)
    kname = {0: "fa_tc_fwd_kernel<bf16>", 1: "fa_tc_fwd_kernel<tf32>",
             2: "fa_simt_fwd_kernel", 3: "fa_tc_fwd_kernel<f16>"}[w.dtype]
    if bwd:
        # The step's three launches (prep, gradient kernel, dq rounding) are
        # timed together, so `achieved` is a lower bound for the gradient
        # kernel alone; `traffic` is the gradient kernel's.
        kname = {0: "fa_bwd_kernel<bf16>", 1: "fa_bwd_simt_kernel<f32>",
                 3: "fa_bwd_kernel<f16>"}[w.dtype]
    traffic, traffic_note = profiled_traffic(kname, w.name)
    roofline = {"bound": "alu" if simt else "tensor", "achieved": achieved, "peak": peak,
                "unit": "TFLOP/s", "frac": achieved / peak, "traffic": traffic,
                "peak_source": (f"{peak_src} bf16 burst" if half_io else
                                f"FP32 FMA: {n_sms} SMs x 128 lanes x 2 x max SM clock" if simt else
                                f"{peak_src} bf16 burst / 2 (tf32 nominal ratio)"),
                "kernel": kname}
    if traffic_note:
        roofline["traffic_note"] = traffic_note

    cpu = None
    if not args.no_cpu_baseline:
        g, threads, desc, _ = cpu_oracle_sample(w, 15.0)
        cpu = {"value": g / 1e3, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
               "sample": desc}

    line = {
        "metric": METRIC_BWD if bwd else METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": DTYPE_NAMES[w.dtype] if w.dtype != 0 else "bf16",
        "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "Nq": w.Nq, "Nk": w.Nk, "d": w.d,
                   "causal": causal, "flops_per_step": flops_step,
                   "parallelism": f"replicas{ws}" if ws > 1 else "single",
                   "key_splits": args.splits, "pass": args.which,
                   "grid": grid,
                   "staged": stage_ws is not None,
                   "varlen": (None if varlen is None else
                              {"sequences": len(varlen["lens"]), "total_tokens": varlen["total"],
                               "lengths": "uniform 512..8192 (seeded)", "H": varlen["H"],
                               "d": varlen["d"], "causal": True}),
                   "l2": l2_note,
                   "launch": ("CUDA graph of the timed steps" if graph is not None
                              else "one by one")},
        "roofline": roofline,
        "pct_of_peak": 100.0 * value / ws / peak,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": args.steps * (3 if bwd or stage_ws is not None
                                      else 2 if wspace is not None else 1),
        "clocks": clocks,
        # per step, the steps launched one by one with an event between
        # consecutive steps (diagnostic; the value comes from the timed region)
        "step_ms": {"min": min(launch_ms), "median": sorted(launch_ms)[len(launch_ms) // 2],
                    "max": max(launch_ms)},
    }
    if varlen is not None:
        line["config"] = {"workload": "varlen32-l512to8192-h16-d128-bf16-causal",
                          "flops_per_step": flops_step, "parallelism": line["config"]["parallelism"],
                          "varlen": line["config"]["varlen"],
                          "l2": "inputs larger than L2 (no flush)"}
    print(json.dumps(line), flush=True)
    if ws > 1:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
