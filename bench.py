"""Benchmark of the Ulysses attention block on GB300.

One step = the whole hot path on one batch of the GPT-7B-like layer (B=1, L=32768, H=32,
d_h=128, P=8 token shards, causal): attention forward with the seq->head relayout of
Q, K, V fused into its loads and the head->seq relayout of O fused into its stores, then
the backward with dO read and dQ, dK, dV written in the token-sharded layout. Inputs are
seeded synthetic bf16 tensors resident in HBM before timing starts.

Metric: attention fwd+bwd TFLOP/s over permitted (query, key) pairs only, 4*d_h flops per
pair forward and 8*d_h backward (recompute not credited). The standalone relayout is
timed beside it in HBM GB/s (2 bytes read + 2 written per element).

  python bench.py [--gpus N --steps K --warmup W] [--impl reference] [--workload NAME]

The line's e2e figure runs the same steps through the public calls with every step's inputs
copied in from pinned host memory and its results copied out, pipelined over three streams
(copies in, kernels, copies out) and two device buffer sets.

With --impl reference the CPU oracle is timed instead, on a bounded sample of rows.
Under torchrun (N > 1) the processes are real Ulysses ranks: each owns L/N tokens on its own
GPU, the all-to-alls run through NCCL, and rank 0 prints one JSON line with the whole-job
value (strong scaling: the total work is the one layer's). --dist runs that path on one GPU.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "Ulysses attn fwd+bwd TFLOP/s & % BF16 peak; relayout HBM GB/s"

# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) of the attention kernels
# on the full-size GPT-7B-like layer, from single-pass ncu captures of that workload (the
# summaries sit under profiles/). A figure is reported only while the kernel sources still
# hash to the value recorded with it; after any change it reads as null until re-captured.
NCU_TRAFFIC = {
    "attn_bwd_kernel": {"bytes": 2687532856, "workload": "gpt7b", "sha": "1062dff41e3172b8",
                        "sources": ["ulysses_sequence_gb300/csrc/attn_bwd.cu", "ulysses_sequence_gb300/csrc/common.cuh"]},
    "attn_fwd_kernel": {"bytes": 1060603761, "workload": "gpt7b", "sha": "dc08a5dc375912d9",
                        "sources": ["ulysses_sequence_gb300/csrc/attn_fwd.cu", "ulysses_sequence_gb300/csrc/common.cuh"]},
}


def ncu_traffic(kernel: str, workload: str):
    import hashlib
    rec = NCU_TRAFFIC.get(kernel)
    if rec is None or rec["workload"] != workload:
        return None
    h = hashlib.sha256()
    for f in rec["sources"]:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return rec["bytes"] if h.hexdigest()[:16] == rec["sha"] else None


def permitted_pairs(w: workloads.Workload) -> int:
    """Permitted (query, key) pairs of one (batch, head)."""
    if w.mask == "causal":
        return w.L * (w.L + 1) // 2
    if w.mask == "none":
        return w.L * w.L
    n = -(-w.L // w.tile)
    qt = np.arange(n)[:, None]
    kt = np.arange(n)[None, :]
    act = ((kt >= qt - w.window_before) & (kt <= qt + w.window_after)) | (kt % w.global_stride == 0)
    rows = np.minimum(w.tile, w.L - np.arange(n) * w.tile)
    return int((act * rows[:, None] * rows[None, :]).sum())


def flops(w: workloads.Workload, fwd_only: bool = False):
    pairs = permitted_pairs(w) * w.B * w.H
    f_fwd = 4 * w.d * pairs
    f_bwd = 0 if (fwd_only or not w.backward) else 8 * w.d * pairs
    return f_fwd, f_bwd


def accounted_alltoall_bytes(w: workloads.Workload) -> int:
    """bf16 bytes one rank exchanges in the forward pass's two all-to-alls: Q and O with H
    heads, K and V with H_kv (each head group receives H_kv/P heads, or one copy when
    P > H_kv). For multi-head attention this is 4Nh/P."""
    kv_per_group = w.Hkv // w.P if w.Hkv % w.P == 0 else 1
    return (2 * w.H + 2 * kv_per_group * w.P) * w.B * w.L * w.d * 2 // w.P


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.dev), "--query-gpu=" + self.FIELDS,
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
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
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
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d.get("bf16_tflops", 1900.0), d.get("hbm_gbs", 6800.0), "measured"
    return 1900.0, 6800.0, "fallback"


def dist_setup(force: bool = False):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 or force:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        # keep stdout to rank 0's one JSON line (NCCL's version banner goes there otherwise)
        os.environ.setdefault("NCCL_DEBUG", "WARN")
        if world == 1:
            os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
            os.environ.setdefault("MASTER_PORT", "29511")
            os.environ.setdefault("RANK", "0")
            os.environ.setdefault("WORLD_SIZE", "1")
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        if dist.get_backend() == "nccl":
            dist.barrier(device_ids=[torch.cuda.current_device()])
        else:
            dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- CPU oracle arm

def sample_flops(w: workloads.Workload, rows, heads) -> int:
    """Algorithmic flops of the oracle sample: permitted pairs of the sampled rows."""
    import oracle
    mask = oracle.mask_for(w)
    n_pairs = 0
    for b in range(w.B):
        r = rows[rows[:, 0] == b, 1]
        if len(r):
            n_pairs += int(mask.rows(r, w.L).sum())
    n_pairs *= len(heads)
    return 4 * w.d * n_pairs + (8 * w.d * n_pairs if w.backward else 0)


def oracle_sample_step(w: workloads.Workload, t_bits, rows, heads):
    """One oracle pass (forward + backward) on a bounded sample of rows and heads."""
    import oracle
    for _ in oracle.attention_sampled(t_bits["q"], t_bits["k"], t_bits["v"], t_bits["do"], w.P, oracle.mask_for(w),
                                      rows, heads=heads):
        pass


def cpu_sample(w: workloads.Workload, n_rows: int, n_heads: int):
    rows = workloads.sample_rows(w.B, w.L, n_rows, seed=w.seed + 100)
    heads = list(range(0, w.H, max(1, w.H // n_heads)))[:n_heads]
    return rows, heads


def run_reference(args, w, world, rank):
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    t = workloads.draw_workload(w)
    bits = {n: workloads.to_bf16_bits(x) for n, x in t.items()}
    rows, heads = cpu_sample(w, args.ref_rows, args.ref_heads)
    f_step = sample_flops(w, rows, heads)
    for _ in range(args.warmup):
        oracle_sample_step(w, bits, rows, heads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_sample_step(w, bits, rows, heads)
    dt = time.perf_counter() - t0
    f = f_step * args.steps
    value = f / dt / 1e12
    sample = f"{len(rows)} sampled query rows x {len(heads)} heads of {w.name}, fwd+bwd, per step"
    cores = os.cpu_count()
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": w.name, "B": w.B, "L": w.L, "H": w.H, "d_h": w.d, "P": w.P, "mask": w.mask},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- GPU arm, N > 1

def run_distributed(args, w, world, rank, local):
    """The layer over `world` GPUs as real Ulysses ranks: each process owns L/world tokens of
    every head on its own GPU, the two all-to-alls per pass run through NCCL
    (ulysses_sequence_gb300.distributed), and each rank attends over the whole sequence for
    its H/world heads. The total work is the one layer's, so this is strong scaling."""
    import ulysses_sequence_gb300 as U
    from ulysses_sequence_gb300.distributed import UlyssesAttention
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    if w.H % world or w.Hkv % world or w.L % world:
        raise SystemExit(f"{w.name}: H={w.H}, H_kv={w.Hkv} and L={w.L} must split over {world} ranks")
    f_fwd, f_bwd = flops(w)
    total_flops = f_fwd + f_bwd
    # the same logical tensors on every rank; this rank keeps its token shard [B][L/world][H][d]
    t = workloads.draw(w.B, w.L, w.H, w.d, world, w.seed, q_scale=w.q_scale, H_kv=w.H_kv)
    host = {n: x[rank].contiguous().pin_memory() for n, x in t.items()}
    del t
    x = {n: v.to(dev) for n, v in host.items()}
    mask = U.Mask.causal() if w.mask == "causal" else (
        U.Mask.none() if w.mask == "none" else
        U.Mask.window_global(w.L, w.tile, w.window_before, w.window_after, w.global_stride, device=dev))
    ua = UlyssesAttention(mask=mask)

    def step(inp):
        o, ctx = ua.forward(inp["q"], inp["k"], inp["v"])
        if not w.backward:
            return (o,), ctx
        return (o,) + ua.backward(ctx, inp["do"]), ctx

    for _ in range(args.warmup):
        step(x)
    torch.cuda.synchronize()
    st, word = U.device_status()
    U.check(st, f"device status after warm-up ({word:#x})")
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step(x)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    elapsed_ms = max_over_ranks(e0.elapsed_time(e1), world)
    ms_per_step = elapsed_ms / args.steps
    value = total_flops * args.steps / (elapsed_ms * 1e-3) / 1e12

    # the local attention alone (this rank's head group, inputs already exchanged)
    outs, ctx = step(x)
    qh, kh, vh, oh, lse = ctx
    doh = ua.to_heads(x["do"]) if w.backward else None
    fwd_ms = cuda_events_time(lambda: ua.ops.attn_fwd(qh, kh, vh), stream, 3)
    bwd_ms = cuda_events_time(lambda: ua.ops.attn_bwd(qh, kh, vh, oh, lse, doh), stream, 3) if w.backward else 0.0
    fwd_ms, bwd_ms = max_over_ranks(fwd_ms, world), max_over_ranks(bwd_ms, world)

    # end to end: this rank's shards from pinned host memory, results back, every step
    out_host = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in outs]
    dev_in = {n: torch.empty_like(v) for n, v in x.items()}
    barrier(world)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(args.steps):
        for n in dev_in:
            dev_in[n].copy_(host[n], non_blocking=True)
        res, _ = step(dev_in)
        for h, r in zip(out_host, res):
            h.copy_(r, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world)
    st, word = U.device_status()
    U.check(st, f"device status after timed steps ({word:#x})")
    peak_tf, _, peak_src = measured_peaks()
    dom_ms, dom_flops, dom_name = (bwd_ms, f_bwd / world, "attn_bwd (local head group)") if w.backward else (
        fwd_ms, f_fwd / world, "attn_fwd (local head group)")
    achieved = dom_flops / (dom_ms * 1e-3) / 1e12
    if rank == 0:
        h2d = sum(v.numel() * v.element_size() for v in host.values())
        d2h = sum(h.numel() * h.element_size() for h in out_host)
        comm = w.B * w.L * (2 * w.H + 2 * w.Hkv) * w.d * 2 // world  # Q, K, V in and O out, bf16, per rank
        # packs and unpacks per batch row, the attention calls (the backward's prep, main and convert
        # kernels, plus the two schedule kernels for a block-sparse mask)
        kernels = (4 * w.B + 1) + ((4 * w.B + 3 + (2 if w.mask == "block_sparse" else 0)) if w.backward else 0)
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "strong",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "L": w.L, "H": w.H, "H_kv": w.Hkv, "d_h": w.d, "P": world,
                       "mask": w.mask, "passes": "fwd+bwd" if w.backward else "fwd",
                       "l2": "inputs larger than L2 (the layer's 4 tensors)",
                       "parallelism": f"ulysses sp{world}: one token shard per GPU, NCCL all-to-all"},
            "frac_of_peak": value / world / peak_tf,
            "local_fwd_ms": fwd_ms, "local_bwd_ms": bwd_ms,
            "alltoall_bytes_per_rank_per_pass": comm,
            "roofline": {"bound": "tensor", "kernel": dom_name, "achieved": achieved, "peak": peak_tf,
                         "unit": "TFLOP/s", "frac": achieved / peak_tf, "traffic": None,
                         "peak_source": f"{peak_src} bf16 dense (burst)"},
            "cpu_baseline": None,
            "e2e": {"value": total_flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                    "note": "per rank: its token shards in from pinned host memory, its results out"},
            "gpu_launches": args.steps * kernels,
            "clocks": clk,
        }
        print(json.dumps(line), flush=True)
    import torch.distributed as dist
    dist.destroy_process_group()
    return 0


# ----------------------------------------------------------------------------- GPU arm

def cuda_events_time(fn, stream, iters):
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(iters):
        fn()
    end.record(stream)
    end.synchronize()
    return start.elapsed_time(end) / iters


def e2e_pipeline(U, w, mask, host_in, sets, host_out, steps, stream):
    """Run `steps` forward(+backward) steps through the public calls, each copying its inputs in
    from pinned host memory and its results out, as a training loop that streams its inputs
    would: three streams (copies in, kernels, copies out) over two device buffer sets, so that
    one step's copies run under another step's kernels. Within a step Q, K, V go in first and
    the forward waits for them alone; dO follows under the forward; O and lse go out under the
    backward, dQ, dK and dV after it. Events order the reuse of a buffer set: its inputs are
    overwritten only once the kernels of the step two back have read them, and its outputs
    only once they were copied out.

    Step i reads host_in[i % len(host_in)] and writes host_out[i % len(host_out)]. Returns the
    elapsed ms of all steps (events on `stream`, which every stream joins at both ends) and the
    kernel stream's own mean ms per step."""
    out_fwd, out_bwd = ("o", "lse"), (("dq", "dk", "dv") if w.backward else ())
    dev = sets[0]["o"].device
    s_in, s_run, s_out = (torch.cuda.Stream(device=dev) for _ in range(3))
    # per buffer set, created once and recorded again each step (a wait takes the record made
    # before it): inputs in, forward done, kernels done (its inputs read), outputs copied out
    names = ("qkv_in", "do_in", "fwd_done", "run_done", "fwd_out", "bwd_out")
    evs = [{n: torch.cuda.Event() for n in names} for _ in range(2)]
    k_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]

    def one(i):
        k = i % 2
        b, e = sets[k], evs[k]
        hin, hout = host_in[i % len(host_in)], host_out[i % len(host_out)]
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(e["run_done"])
            for n in ("q", "k", "v"):
                b["x"][n].copy_(hin[n], non_blocking=True)
            e["qkv_in"].record(s_in)
            if w.backward:
                b["x"]["do"].copy_(hin["do"], non_blocking=True)
                e["do_in"].record(s_in)
        with torch.cuda.stream(s_run):
            s_run.wait_event(e["qkv_in"])
            if i >= 2:
                s_run.wait_event(e["fwd_out"])
            k_ev[i][0].record(s_run)
            U.attn_fwd(b["x"]["q"], b["x"]["k"], b["x"]["v"], w.P, mask, o=b["o"], lse=b["lse"], stream=s_run)
            e["fwd_done"].record(s_run)
            if w.backward:
                s_run.wait_event(e["do_in"])
                if i >= 2:
                    s_run.wait_event(e["bwd_out"])
                U.attn_bwd(b["x"]["q"], b["x"]["k"], b["x"]["v"], b["o"], b["lse"], b["x"]["do"], w.P, mask,
                           dq=b["dq"], dk=b["dk"], dv=b["dv"], workspace=b["ws"], stream=s_run)
            e["run_done"].record(s_run)
            k_ev[i][1].record(s_run)
        with torch.cuda.stream(s_out):
            s_out.wait_event(e["fwd_done"])
            for n in out_fwd:
                hout[n].copy_(b[n], non_blocking=True)
            e["fwd_out"].record(s_out)
            if out_bwd:
                s_out.wait_event(e["run_done"])
                for n in out_bwd:
                    hout[n].copy_(b[n], non_blocking=True)
                e["bwd_out"].record(s_out)

    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for st in (s_in, s_run, s_out):
        st.wait_event(start)
    for i in range(steps):
        one(i)
    for st in (s_in, s_run, s_out):
        done = torch.cuda.Event()
        done.record(st)
        stream.wait_event(done)
    end.record(stream)
    end.synchronize()
    kernel_ms = sum(a.elapsed_time(b) for a, b in k_ev) / steps
    return start.elapsed_time(end), kernel_ms


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="gpt7b", choices=list(workloads.WORKLOADS))
    ap.add_argument("--L", type=int, default=0, help="override the sequence length (smaller profiling cases)")
    ap.add_argument("--cpu-rows", type=int, default=3072)
    ap.add_argument("--cpu-heads", type=int, default=4)
    ap.add_argument("--ref-rows", type=int, default=64)
    ap.add_argument("--ref-heads", type=int, default=2)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--dist", action="store_true",
                    help="run the multi-process Ulysses path (NCCL all-to-alls) even on one GPU")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    w = workloads.WORKLOADS[args.workload]
    if args.L:
        import dataclasses
        w = dataclasses.replace(w, name=f"{w.name}@L{args.L}", L=args.L)
    world, rank, local = dist_setup(force=args.dist and args.impl != "reference")
    if args.impl == "reference":
        return run_reference(args, w, world, rank)
    if world > 1 or args.dist:
        return run_distributed(args, w, world, rank, local)

    import ulysses_sequence_gb300 as U
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    f_fwd, f_bwd = flops(w)
    total_flops = f_fwd + f_bwd

    t = workloads.draw(w.B, w.L, w.H, w.d, w.P, w.seed + 1000 * rank, q_scale=w.q_scale, H_kv=w.H_kv)
    host = {n: x.pin_memory() for n, x in t.items()}
    x = {n: v.to(dev) for n, v in host.items()}
    mask = U.Mask.causal() if w.mask == "causal" else (
        U.Mask.none() if w.mask == "none" else
        U.Mask.window_global(w.L, w.tile, w.window_before, w.window_after, w.global_stride, device=dev))
    o = torch.empty_like(x["q"])
    lse = torch.empty((w.P, w.B, w.Hp, w.L), dtype=torch.float32, device=dev)
    dq, dk, dv = (torch.empty_like(x["q"]) for _ in range(3))
    ws = U.bwd_workspace(x["q"], w.P)

    def fwd():
        U.attn_fwd(x["q"], x["k"], x["v"], w.P, mask, o=o, lse=lse)

    def bwd():
        U.attn_bwd(x["q"], x["k"], x["v"], o, lse, x["do"], w.P, mask, dq=dq, dk=dk, dv=dv, workspace=ws)

    def step():
        fwd()
        if w.backward:
            bwd()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    st, word = U.device_status()
    U.check(st, f"device status after warm-up ({word:#x})")

    # The timed steps replay the forward call and the backward call as two CUDA graphs,
    # captured once after the warm-up: the same kernels with the same arguments, without the
    # per-call host work (argument checks, tensor-map encoding, Python) between launches.
    g_fwd = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_fwd):
        fwd()
    g_bwd = None
    if w.backward:
        g_bwd = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_bwd):
            bwd()
    g_fwd.replay()
    if g_bwd is not None:
        g_bwd.replay()
    torch.cuda.synchronize()
    st, word = U.device_status()
    U.check(st, f"device status after the graph replays ({word:#x})")

    # ---- timed region: K steps, device-resident inputs
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        ev[i][0].record(stream)
        g_fwd.replay()
        ev[i][1].record(stream)
        if g_bwd is not None:
            g_bwd.replay()
        ev[i][2].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    elapsed_ms = t_start.elapsed_time(t_end)
    fwd_ms = [a.elapsed_time(b) for a, b, _ in ev]
    bwd_ms = [b.elapsed_time(c) for _, b, c in ev]
    st, word = U.device_status()
    U.check(st, f"device status after timed steps ({word:#x})")
    elapsed_ms = max_over_ranks(elapsed_ms, world)
    ms_per_step = elapsed_ms / args.steps
    value = total_flops * world * args.steps / (elapsed_ms * 1e-3) / 1e12

    # ---- end to end through the public API with host buffers (pinned), pipelined (e2e_pipeline)
    sets = [{"x": x, "o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv, "ws": ws},
            {"x": {n: torch.empty_like(v) for n, v in x.items()}, "o": torch.empty_like(o),
             "lse": torch.empty_like(lse), "dq": torch.empty_like(dq), "dk": torch.empty_like(dk),
             "dv": torch.empty_like(dv), "ws": torch.empty_like(ws)}]
    out_names = ("o", "lse") + (("dq", "dk", "dv") if w.backward else ())
    host_out = [{n: torch.empty(sets[0][n].shape, dtype=sets[0][n].dtype, pin_memory=True) for n in out_names}
                for _ in range(2)]
    e2e_pipeline(U, w, mask, [host], sets, host_out, 2, stream)  # warm-up
    barrier(world)
    n_e2e = max(2, args.steps)
    e2e_elapsed, e2e_kernel_ms = e2e_pipeline(U, w, mask, [host], sets, host_out, n_e2e, stream)
    e2e_ms = max_over_ranks(e2e_elapsed / n_e2e, world)
    st_e2e, word_e2e = U.device_status()
    U.check(st_e2e, f"device status after the end-to-end steps ({word_e2e:#x})")
    del sets[1]

    in_names = ("q", "k", "v", "do") if w.backward else ("q", "k", "v")
    h2d = sum(host[n].numel() * host[n].element_size() for n in in_names)
    d2h = sum(v.numel() * v.element_size() for v in host_out[0].values())

    # ---- standalone relayout (seq->head of one tensor), HBM bound; launched through the raw
    # C call with prepared arguments so the host side keeps ahead of the ~80 us kernel
    heads = torch.empty((w.P, w.B, w.L, w.Hp, w.d), dtype=torch.bfloat16, device=dev)
    lib = U.load()
    rl_args = (U.token_shape(x["q"], w.P), x["q"].data_ptr(), heads.data_ptr(), stream.cuda_stream)
    relayout = lambda: lib.ulysses_seq_to_head(*rl_args)  # noqa: E731
    for _ in range(3):
        relayout()
    # 20 back-to-back launches replayed as one CUDA graph, so that the timing sees the kernels
    # and not the host's launch gaps between them (each launch is about 80 us)
    g_rl = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_rl):
        cs = torch.cuda.current_stream().cuda_stream
        for _ in range(20):
            U.check(lib.ulysses_seq_to_head(rl_args[0], rl_args[1], rl_args[2], cs), "seq_to_head")
    g_rl.replay()
    torch.cuda.synchronize()
    rl_ms = cuda_events_time(g_rl.replay, stream, 5) / 20
    rl_bytes = 2 * x["q"].numel() * x["q"].element_size()
    peak_tf, peak_gbs, peak_src = measured_peaks()

    # ---- the projections on either side of the block (hidden = H d_h): QKV into the
    # token-sharded layout the attention reads, and the output projection of O
    hidden = w.H * w.d
    xs = workloads.draw_hidden(w.B, w.L, hidden, w.P, seed=w.seed + 7).to(dev)
    w_qkv = workloads.draw_weight((w.H + 2 * w.Hkv) * w.d, hidden, seed=w.seed + 8).to(dev)
    w_o = workloads.draw_weight(hidden, w.H * w.d, seed=w.seed + 9).to(dev)
    pq, pk, pv = torch.empty_like(x["q"]), torch.empty_like(x["k"]), torch.empty_like(x["v"])
    py = torch.empty_like(xs)
    qkv_call = lambda: U.qkv_proj(xs, w_qkv, w.P, w.H, w.Hkv, w.d, q=pq, k=pk, v=pv)  # noqa: E731
    out_call = lambda: U.out_proj(o, w_o, w.P, y=py)  # noqa: E731
    for _ in range(3):
        qkv_call()
        out_call()
    qkv_ms = cuda_events_time(qkv_call, stream, 10)
    out_ms = cuda_events_time(out_call, stream, 10)
    # cuBLAS on the same bf16 operands, timed beside them as the library-GEMM comparison
    x2d, o2d = xs.reshape(-1, hidden), o.reshape(-1, w.H * w.d)
    cb_qkv = lambda: torch.matmul(x2d, w_qkv.t())  # noqa: E731
    cb_out = lambda: torch.matmul(o2d, w_o.t())  # noqa: E731
    for _ in range(3):
        cb_qkv()
        cb_out()
    cb_qkv_ms = cuda_events_time(cb_qkv, stream, 10)
    cb_out_ms = cuda_events_time(cb_out, stream, 10)
    rows = w.B * w.L
    qkv_flops = 2 * rows * (w.H + 2 * w.Hkv) * w.d * hidden
    out_flops = 2 * rows * hidden * w.H * w.d
    del xs, w_qkv, w_o, pq, pk, pv, py, x2d, o2d

    # ---- the Ulysses-ring hybrid on the same tensors: P = 2H shards (beyond the head cut's
    # P <= H) as P_ring = 2 ring blocks of P_u = H shards; the same attention, so the same flops
    usp = None
    if w.mask in ("causal", "none") and (w.Hkv % w.H == 0 or w.H % w.Hkv == 0):
        P_ring, P_usp = 2, 2 * w.H
        Pu = P_usp // P_ring
        if w.L % P_usp == 0 and (w.L // P_usp) % 8 == 0 and (Pu % w.Hkv == 0 or w.Hkv % Pu == 0):
            # the token-sharded bytes of P shards are those of any other shard count: re-view them
            uq, uk, uv, udo = (x[n].reshape(P_usp, w.B, w.L // P_usp, x[n].shape[3], w.d)
                               for n in ("q", "k", "v", "do"))
            uo = torch.empty_like(uq)
            ulse = torch.empty((P_ring, Pu, w.B, w.H // Pu, w.L // P_ring), dtype=torch.float32, device=dev)
            udq, udk, udv = torch.empty_like(uq), torch.empty_like(uk), torch.empty_like(uv)
            uws = U.usp_workspace(uq, P_usp, P_ring, w.Hkv)
            ufwd = lambda: U.usp_attn_fwd(uq, uk, uv, P_usp, P_ring, mask, o=uo, lse=ulse, workspace=uws)  # noqa: E731
            ubwd = lambda: U.usp_attn_bwd(uq, uk, uv, uo, ulse, udo, P_usp, P_ring, mask, dq=udq, dk=udk,  # noqa: E731
                                          dv=udv, workspace=uws)
            for _ in range(3):
                ufwd()
                if w.backward:
                    ubwd()
            ufwd_ms = cuda_events_time(ufwd, stream, 5)
            # a forward-only workload times (and credits) the forward alone
            ubwd_ms = cuda_events_time(ubwd, stream, 5) if w.backward else None
            pairs_fwd = 3 if w.mask == "causal" else 4
            usp = {"P": P_usp, "P_ring": P_ring, "P_u": Pu, "fwd_ms": ufwd_ms, "bwd_ms": ubwd_ms,
                   "fwd_tflops": f_fwd / (ufwd_ms * 1e-3) / 1e12,
                   "bwd_tflops": f_bwd / (ubwd_ms * 1e-3) / 1e12 if w.backward else None,
                   "fwd_bwd_tflops": ((f_fwd + f_bwd) / ((ufwd_ms + ubwd_ms) * 1e-3) / 1e12
                                      if w.backward else None),
                   # fwd: one attention per block pair (the merge is in its epilogue); bwd: one
                   # backward per pair + Delta prep and dQ conversion per query block
                   "launches_per_step": pairs_fwd + ((pairs_fwd + 2 * P_ring) if w.backward else 0),
                   "note": "same tensors and mask, P > H; block-pair attention merged in fp32 in its "
                           "epilogue (fwd), block-pair backward + fp32 gradient sums (bwd); not part of the step"}
            del uo, ulse, udq, udk, udv, uws

    # ---- dominant launch group: the backward call (Delta prep + main + dQ convert)
    bwd_avg = statistics.mean(bwd_ms) if w.backward else 0.0
    fwd_avg = statistics.mean(fwd_ms)
    if w.backward and bwd_avg >= fwd_avg:
        dom_name, dom_flops, dom_ms = "attn_bwd (Delta prep + main + dQ convert)", f_bwd, bwd_avg
        dom_traffic = ncu_traffic("attn_bwd_kernel", w.name)
    else:
        dom_name, dom_flops, dom_ms = "attn_fwd", f_fwd, fwd_avg
        dom_traffic = ncu_traffic("attn_fwd_kernel", w.name)
    achieved = dom_flops / (dom_ms * 1e-3) / 1e12

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        try:
            import oracle
            oracle.build()
            bits = {n: workloads.to_bf16_bits(v) for n, v in t.items()}
            rows, heads_s = cpu_sample(w, args.cpu_rows, args.cpu_heads)
            fc = sample_flops(w, rows, heads_s)
            t0 = time.perf_counter()
            oracle_sample_step(w, bits, rows, heads_s)
            dt = time.perf_counter() - t0
            cpu = {"value": fc / dt / 1e12, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
                   "sample": f"{len(rows)} sampled query rows x {len(heads_s)} heads of {w.name}, fwd+bwd "
                             f"({fc / 1e9:.1f} GFLOP in {dt:.1f} s)",
                   # the sample's time scaled to the whole workload by algorithmic flops (the
                   # sampled rows' permitted pairs against all of them): an extrapolation, not a run
                   "full_workload_s_extrapolated": dt * total_flops / fc,
                   "extrapolation": "t_sample x flops(workload) / flops(sample); not measured"}
        except Exception as exc:  # the baseline must not hide the GPU line
            cpu = {"value": None, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
                   "sample": f"failed: {exc}"}

    # The chip's nominal dense bf16 rate: SMs x SM clock x 8192 flops per clock per SM (one
    # M=128, N=256, K=16 tcgen05 MMA, 2*128*256*16 flops, every 128 cycles: twice the previous
    # generation's 4096), at the median SM clock sampled in the timed region
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    nom_mhz = clk.get("sm_mhz") or clk.get("sm_max_mhz")
    nominal = None
    if nom_mhz:
        nom_tf = sms * nom_mhz * 1e6 * 8192 / 1e12
        nominal = {"tflops": nom_tf, "sms": sms, "sm_mhz": nom_mhz, "flops_per_clk_per_sm": 8192,
                   "frac": value / world / nom_tf, "roofline_frac": achieved / nom_tf,
                   "note": "SM count x sampled SM clock x 8192 bf16 flops/clk/SM; beside the measured peak"}

    if rank == 0:
        pairs = permitted_pairs(w)
        comm = accounted_alltoall_bytes(w)
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "L": w.L, "H": w.H, "H_kv": w.Hkv, "d_h": w.d, "P": w.P,
                       "mask": w.mask, "passes": "fwd+bwd" if w.backward else "fwd", "layout": "token-sharded (relayouts fused)",
                       "l2": "inputs larger than L2 (4 x %.0f MB bf16)" % (x["q"].numel() * 2 / 1e6),
                       "timed_steps": "CUDA-graph replays of the forward and backward calls",
                       "parallelism": "single GPU"},
            "frac_of_peak": value / world / peak_tf,
            "fwd_ms": fwd_avg, "bwd_ms": bwd_avg,
            "fwd_tflops": f_fwd / (fwd_avg * 1e-3) / 1e12,
            "bwd_tflops": (f_bwd / (bwd_avg * 1e-3) / 1e12) if w.backward else None,
            "fa_convention_tflops": (f_fwd + f_bwd * 10 / 8) * world * args.steps / (elapsed_ms * 1e-3) / 1e12,
            "permitted_pairs_per_head": pairs,
            "relayout": {"kernel": "seq_to_head (one tensor)", "gbs": rl_bytes / (rl_ms * 1e-3) / 1e9,
                         "ms": rl_ms, "bytes": rl_bytes, "frac_of_measured_hbm": rl_bytes / (rl_ms * 1e-3) / 1e9 / peak_gbs},
            "projections": {"qkv_tflops": qkv_flops / (qkv_ms * 1e-3) / 1e12, "qkv_ms": qkv_ms,
                            "out_tflops": out_flops / (out_ms * 1e-3) / 1e12, "out_ms": out_ms,
                            "cublas_qkv_tflops": qkv_flops / (cb_qkv_ms * 1e-3) / 1e12,
                            "cublas_out_tflops": out_flops / (cb_out_ms * 1e-3) / 1e12,
                            "qkv_frac": qkv_flops / (qkv_ms * 1e-3) / 1e12 / peak_tf,
                            "out_frac": out_flops / (out_ms * 1e-3) / 1e12 / peak_tf,
                            "note": "x [B*L][H*d_h] -> Q, K, V token-sharded; O -> y; not part of the step"},
            "usp": usp,
            # the backward mirrors the forward's exchanges: dO in, dQ out (H heads); dK, dV out
            # (the key/value heads), the same bytes as Q, O in and K, V
            "accounted_alltoall_bytes_per_rank": {"fwd": comm, "bwd": comm if w.backward else 0,
                                                  "leaves_rank": comm * (w.P - 1) // w.P,
                                                  "note": "4Nh/P in bf16 bytes per pass, accounted, not measured "
                                                          "over a link; leaves_rank is the forward's (P-1)/P share"},
            "roofline": {"bound": "tensor", "kernel": dom_name, "achieved": achieved, "peak": peak_tf,
                         "unit": "TFLOP/s", "frac": achieved / peak_tf, "traffic": dom_traffic,
                         "peak_source": f"{peak_src} bf16 dense (burst)"},
            "nominal_peak": nominal,
            "cpu_baseline": cpu,
            "e2e": {"value": total_flops * world / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                    "kernel_ms_per_step": e2e_kernel_ms,
                    "overlap": "copies in, kernels and copies out on three streams over two device buffer "
                               "sets: one step's copies run under another step's kernels; dO in under the "
                               "forward, O and lse out under the backward"},
            # per step: the forward; the backward call's Delta prep, main kernel and dQ convert,
            # plus the two block-sparse schedule kernels for that mask
            "gpu_launches": args.steps * (1 + ((3 + (2 if w.mask == "block_sparse" else 0)) if w.backward else 0)),
            "clocks": clk,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
