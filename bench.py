#!/usr/bin/env python3
"""Benchmark of the Inkling attention hot path on GB300.

One step = one pass of the whole path over the sliding-window prefill layer
(8192 tokens, Hq=64, Hkv=8, window 4096, rel_extent 512): inkattn_prologue then
inkattn_prefill, inputs resident in HBM.  value = algorithmic attention TFLOP/s of
the step.  The same line carries the MTP-verify decode workload (32 x 9 queries,
KV 32768, split-KV decode + combine) as KV GB/s, per-kernel rooflines, the
end-to-end number through the C ABI with pinned host buffers, the SM clocks seen
during the timed region, and the fp64 oracle timed on a bounded sample on the host
cores.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

With N > 1 (launched by torch.distributed.run) every rank runs an independent
replica of the workload on its own GPU; value = units of all ranks / max time.
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

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "rel-bias attn prefill TFLOP/s & decode KV GB/s (1 GB300, % of roofline)"
L2_FLUSH_BYTES = 256 << 20
KERNEL_SOURCES = {
    "k_prefill_tc": ["relative_bias_hybrid_gb300/csrc/prefill_tc.cu", "relative_bias_hybrid_gb300/csrc/tcgen05.cuh",
                     "relative_bias_hybrid_gb300/csrc/common.cuh"],
    "k_decode_tc": ["relative_bias_hybrid_gb300/csrc/decode_tc.cu", "relative_bias_hybrid_gb300/csrc/tcgen05.cuh",
                    "relative_bias_hybrid_gb300/csrc/common.cuh"],
    "k_prologue": ["relative_bias_hybrid_gb300/csrc/prologue.cu", "relative_bias_hybrid_gb300/csrc/common.cuh"],
}


# ---------------------------------------------------------------- algorithmic work

def visible_pairs(w) -> int:
    """Number of (query, key) pairs the method attends over (per query head)."""
    total = 0
    for n, pre in zip(w.q_lens, w.prefix_lens):
        i = np.arange(pre, pre + n, dtype=np.int64)
        vis = i + 1 if w.window == 0 else np.minimum(i + 1, w.window)
        total += int(vis.sum())
    return total


def biased_pairs(w) -> int:
    """Pairs with 0 <= i-j < rel_extent (and visible): the ones that get a bias term."""
    total = 0
    lim = w.rel_extent if w.window == 0 else min(w.rel_extent, w.window)
    for n, pre in zip(w.q_lens, w.prefix_lens):
        i = np.arange(pre, pre + n, dtype=np.int64)
        total += int(np.minimum(i + 1, lim).sum())
    return total


def attention_flops(w) -> float:
    """QK^T and PV (2 FLOP per multiply-add, 2 contractions of length d) plus the bias
    projections r.P for the biased pairs; masked or skipped work is not counted."""
    return (4.0 * w.head_dim * visible_pairs(w) * w.Hq + 2.0 * w.d_r * biased_pairs(w) * w.Hq)


def prologue_bytes(w) -> float:
    """q in/out, k and v in, normed K and V out, slot mapping, conv state read + write."""
    per_tok = 2 * (w.Hq * w.head_dim * 2) + 2 * (w.Hkv * w.head_dim * 2) * 2 + 4
    return float(per_tok * w.N_tok + w.B * 2 * 2 * 3 * w.Hkv * w.head_dim * 2)


def decode_bytes(w) -> float:
    """Every visible K and V row once per (sequence, KV head), plus q, out, r, P, table."""
    kv = 0
    for n, pre in zip(w.q_lens, w.prefix_lens):
        T = n + pre
        first = 0 if w.window == 0 else max(0, pre - w.window + 1)
        kv += (T - first) * w.Hkv * w.head_dim * 2 * 2
    q = w.N_tok * w.Hq * w.head_dim * 2
    r = w.N_tok * w.Hq * w.d_r * 2
    P = w.Hq * w.d_r * w.rel_extent * 4
    table = w.B * w.max_blocks * 4
    return float(kv + 2 * q + r + P + table)


# ---------------------------------------------------------------- helpers

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm": float(d["hbm_gbs"]), "bf16": float(d["bf16_tflops"]),
                "bf16_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "src": "of measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm": 6800.0, "bf16": 1900.0, "bf16_sustained": 1700.0, "src": "of fallback"}


def source_hash(kernel: str) -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, or None when no summary
    exists or the kernel source changed since it was taken."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}_traffic.txt")
    try:
        kv = {}
        with open(path) as f:
            for line in f:
                if ":" in line and not line.startswith("#"):
                    k, v = line.split(":", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("source_sha256") != source_hash(kernel):
            return None
        return float(kv["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.path = None
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            self.target = uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"
        except Exception:
            self.target = str(device_index)

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.target, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        try:
            with open(self.path) as f:
                for line in f:
                    parts = [x.strip() for x in line.split(",")]
                    if len(parts) < 8:
                        continue
                    try:
                        sm.append(float(parts[0]))
                        mx.append(float(parts[1]))
                    except ValueError:
                        continue
                    for name, val in zip(names, parts[4:8]):
                        if val.lower() == "active":
                            reasons.add(name)
            os.unlink(self.path)
        except OSError:
            pass
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def aggregate_over_ranks(local_ms: float, local_units: float, world: int):
    """(max time over ranks in ms, total units over ranks).  Replicas: no data exchange;
    this reduction is on two scalars for the report only."""
    if world == 1:
        return local_ms, local_units
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([local_ms], dtype=torch.float64, device=dev)
    u = torch.tensor([local_units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


# ---------------------------------------------------------------- oracle arm

def oracle_sample(w, x_cpu, q_bits, kc_bits, vc_bits, rows, n_threads):
    import oracle
    t0 = time.perf_counter()
    oracle.attention_for_inputs(x_cpu, w, q_bits, kc_bits, vc_bits, rows=rows, n_threads=n_threads)
    return time.perf_counter() - t0


def sample_flops(w, rows, cu):
    """Algorithmic FLOPs of the attention for the listed token rows (all heads)."""
    total = 0.0
    seq = np.searchsorted(cu, rows, side="right") - 1
    for t, b in zip(rows, seq):
        i = w.prefix_lens[b] + (t - cu[b])
        vis = i + 1 if w.window == 0 else min(i + 1, w.window)
        lim = w.rel_extent if w.window == 0 else min(w.rel_extent, w.window)
        total += (4.0 * w.head_dim * vis + 2.0 * w.d_r * min(i + 1, lim)) * w.Hq
    return total


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_oracle_baseline(w, x_dev, target_s=12.0, seed=0):
    """fp64 oracle on a bounded sample of the workload's query rows (all heads), timed
    on all host cores; returns the cpu_baseline object in the bench's unit."""
    import oracle  # noqa: F401  (test infrastructure; only this leg of the bench uses it)
    from relative_bias_hybrid_gb300 import inputs as gen
    x_cpu = {k: x_dev[k].cpu() for k in ("cu_seqlens_q", "seqlen_k", "r", "P", "block_table")}
    q_bits = gen.bits(x_dev["q"])
    kc, vc = gen.bits(x_dev["k_cache"]), gen.bits(x_dev["v_cache"])
    cu = x_cpu["cu_seqlens_q"].numpy()
    rng = np.random.default_rng(seed)
    cores = host_cores()
    n = 16
    rows = np.sort(rng.choice(w.N_tok, size=n, replace=False)).astype(np.int32)
    dt = oracle_sample(w, x_cpu, q_bits, kc, vc, rows, cores)
    if dt < target_s / 4:
        n = int(min(w.N_tok, max(n, n * target_s / max(dt, 1e-3))))
        rows = np.sort(rng.choice(w.N_tok, size=n, replace=False)).astype(np.int32)
        dt = oracle_sample(w, x_cpu, q_bits, kc, vc, rows, cores)
    fl = sample_flops(w, rows, cu)
    return {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"{len(rows)} of {w.N_tok} query rows (all {w.Hq} heads), {fl:.3g} FLOP in {dt:.1f} s"}


def run_reference(args, world, rank):
    """--impl reference: the fp64 CPU oracle, timed on the host cores, on the same
    workload and metric (each step a bounded sample of query rows)."""
    if rank != 0:
        return
    from relative_bias_hybrid_gb300 import inputs as gen
    import oracle
    oracle.build()
    w = gen.workload("swa")
    x = gen.make_inputs(w, seed=0, device="cpu")
    ref = oracle.prologue_for_inputs(x, w)
    cu = x["cu_seqlens_q"].numpy()
    cores = host_cores()
    rng = np.random.default_rng(1)
    rows_per_step = 96
    times, flops = [], []
    for it in range(args.warmup + args.steps):
        rows = np.sort(rng.choice(w.N_tok, size=rows_per_step, replace=False)).astype(np.int32)
        dt = oracle_sample(w, x, ref["q_out"], ref["k_cache"], ref["v_cache"], rows, cores)
        if it >= args.warmup:
            times.append(dt)
            flops.append(sample_flops(w, rows, cu))
    value = sum(flops) / sum(times) / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sum(times) / len(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": w.describe(), "sample": f"{rows_per_step} query rows x {w.Hq} heads per step"},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "sample": f"{rows_per_step} of {w.N_tok} query rows per step, all heads"},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- GPU arm

def timed_steps(step, steps, warmup, flush, stream, kernel_split=True):
    """Runs warmup + steps passes; each timed pass is bracketed by CUDA events on the
    launching stream, with an L2 flush (a 256 MiB write) between passes, outside the
    events.  Returns (per-step ms list, per-step attention-kernel ms list)."""
    for _ in range(warmup):
        step.run(stream)
    torch.cuda.synchronize()
    tot, att = [], []
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
            torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    with torch.cuda.stream(stream):
        for e0, e1, e2 in evs:
            flush.zero_()
            e0.record(stream)
            step.run_prologue(stream)
            e1.record(stream)
            step.run_attention(stream)
            e2.record(stream)
    torch.cuda.synchronize()
    for e0, e1, e2 in evs:
        tot.append(e0.elapsed_time(e2))
        att.append(e1.elapsed_time(e2))
    pro = [t - a for t, a in zip(tot, att)]
    return tot, att, pro


def e2e_steps(steps_pair, x_host, steps, warmup, stream):
    """Per step: pinned host -> device copies of the step's inputs, the two C-ABI calls and
    the device -> pinned host copy of its output, every one inside the timed events.  Two
    sets of input and output buffers alternate, so that the copies of step i + 1 (in) and
    step i - 1 (out) run on their own streams while step i computes; the calls themselves
    stay in order on one stream, since consecutive steps share the KV cache and the conv
    state."""
    names = ["q", "k", "v", "r"]
    dev = steps_pair[0].out.device
    out_host = [torch.empty(s.out.shape, dtype=s.out.dtype, pin_memory=True) for s in steps_pair]
    h2d = sum(x_host[n].numel() * x_host[n].element_size() for n in names)
    d2h = out_host[0].numel() * out_host[0].element_size()
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    def pipeline(n_steps):
        ev = lambda: torch.cuda.Event()
        in_done, comp_done, out_done = [], [], []
        for i in range(n_steps):
            st, buf = steps_pair[i % 2], i % 2
            # inputs of step i: the buffer was last read by step i - 2
            if i >= 2:
                s_in.wait_event(comp_done[i - 2])
            with torch.cuda.stream(s_in):
                for n in names:
                    st.x[n].copy_(x_host[n], non_blocking=True)
            in_done.append(ev())
            in_done[i].record(s_in)
            # the step: after its inputs, and after step i - 2's output left this buffer
            stream.wait_event(in_done[i])
            if i >= 2:
                stream.wait_event(out_done[i - 2])
            st.run(stream)
            comp_done.append(ev())
            comp_done[i].record(stream)
            # its output back to the host
            s_out.wait_event(comp_done[i])
            with torch.cuda.stream(s_out):
                out_host[buf].copy_(st.out, non_blocking=True)
            out_done.append(ev())
            out_done[i].record(s_out)
        stream.wait_event(out_done[-1])

    pipeline(warmup)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_in.wait_event(e0)
    s_out.wait_event(e0)
    pipeline(steps)
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps, h2d, d2h


def run_gpu(args, world, rank, local):
    from relative_bias_hybrid_gb300 import build as _b
    from relative_bias_hybrid_gb300 import inputs as gen
    from relative_bias_hybrid_gb300.step import AttentionStep
    _b.build()
    peaks = load_peaks()
    dev = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.Stream(device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    # ---- prefill layer (the headline workload)
    w = gen.workload("swa")
    x = gen.make_inputs(w, seed=rank, device=dev)
    step = AttentionStep(w, x, mode="prefill")
    fl = attention_flops(w)

    # ---- decode workload
    wd = gen.workload("decode")
    xd = gen.make_inputs(wd, seed=rank, device=dev)
    dstep = AttentionStep(wd, xd, mode="decode")
    dbytes = decode_bytes(wd)

    clocks = ClockSampler(dev.index)
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    tot, att, pro = timed_steps(step, args.steps, args.warmup, flush, stream)
    dtot, datt, dpro = timed_steps(dstep, args.steps, args.warmup, flush, stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    status = step.device_status() | dstep.device_status()
    if status != 0:
        raise RuntimeError(f"device status {status} during the bench")

    ms = sum(tot) / len(tot)
    ms_max, units = aggregate_over_ranks(ms, fl, world)
    value = units / (ms_max * 1e-3) / 1e12

    # ---- end to end through the C ABI with pinned host buffers
    x_host = {n: x[n].cpu().pin_memory() for n in ("q", "k", "v", "r")}
    # a second set of input/output buffers over the same cache and conv state
    x2 = dict(x)
    for n in ("q", "k", "v", "r"):
        x2[n] = torch.empty_like(x[n])
    step2 = AttentionStep(w, x2, mode="prefill")
    e2e_ms, h2d, d2h = e2e_steps((step, step2), x_host, args.steps, args.warmup, stream)
    if step.device_status() | step2.device_status():
        raise RuntimeError("device status set during the end-to-end steps")
    e2e_ms_max, e2e_units = aggregate_over_ranks(e2e_ms, fl, world)

    att_ms = sum(att) / len(att)
    pro_ms = sum(pro) / len(pro)
    dec_ms = sum(datt) / len(datt)
    prefill_tf = fl / (att_ms * 1e-3) / 1e12
    pro_gbs = prologue_bytes(w) / (pro_ms * 1e-3) / 1e9
    dec_gbs = dbytes / (dec_ms * 1e-3) / 1e9
    traffic = ncu_traffic("k_prefill_tc", "swa")
    roof = {"bound": "tensor", "kernel": "k_prefill_tc", "achieved": prefill_tf, "peak": peaks["bf16"],
            "unit": "TFLOP/s", "frac": prefill_tf / peaks["bf16"], "peak_src": peaks["src"] + " (burst bf16)",
            "traffic": traffic, "algorithmic_flop_per_launch": fl}
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.describe() + "; step = inkattn_prologue + inkattn_prefill",
                   "global_batch": w.B * world, "seq_len": w.N_tok, "parallelism": f"replicas x{world}",
                   "l2": "flushed between steps (256 MiB write, outside the timed events)"},
        "roofline": roof,
        "rooflines": {
            "k_prologue": {"bound": "hbm", "achieved": pro_gbs, "peak": peaks["hbm"], "unit": "GB/s",
                           "frac": pro_gbs / peaks["hbm"], "traffic": ncu_traffic("k_prologue", "swa"),
                           "algorithmic_bytes_per_launch": prologue_bytes(w), "ms": pro_ms},
            "k_decode_tc+k_combine": {"bound": "hbm", "achieved": dec_gbs, "peak": peaks["hbm"], "unit": "GB/s",
                                      "frac": dec_gbs / peaks["hbm"], "traffic": ncu_traffic("k_decode_tc", "decode"),
                                   "algorithmic_bytes_per_launch": dbytes, "ms": dec_ms,
                                   "num_splits": dstep.num_splits},
        },
        "decode": {"workload": wd.describe() + "; step = inkattn_prologue + inkattn_decode + inkattn_combine",
                   "value": dec_gbs, "unit": "GB/s", "kv_bytes_per_step": dbytes,
                   "ms_per_step": sum(dtot) / len(dtot), "ms_attention": dec_ms,
                   "num_splits": dstep.num_splits, "frac_of_hbm": dec_gbs / peaks["hbm"]},
        "e2e": {"value": e2e_units / (e2e_ms_max * 1e-3) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms_max},
        "gpu_launches": args.steps * (step.launches_per_run() + dstep.launches_per_run()),
        "clocks": clk,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_oracle_baseline(w, x)
    if rank == 0:
        print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["inkattn", "reference"], default="inkattn")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)     # at least 3 untimed warm-up steps, reported as used
    world, rank, local = dist_setup(args)
    try:
        if args.impl == "reference":
            run_reference(args, world, rank)
        else:
            run_gpu(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
