#!/usr/bin/env python3
"""Benchmark of the Inkling attention hot path on one GB300.

One step = one pass of the whole path over one workload, inputs resident in HBM:
inkattn_prologue then inkattn_prefill (prefill layers), or inkattn_prologue then
inkattn_decode + inkattn_combine (decode).  The headline is the full-attention prefill
layer (B=1, T=32768, Hq=64, Hkv=8, rel_extent=1024, logits scaled by ln T / ln 8192):
value = its algorithmic attention TFLOP/s per step.  The same JSON line carries the
sliding-window layer, the ragged mixed-prefill batch, the full layer over an E4M3 cache
and the MTP-verify decode (bf16 and E4M3 caches) under "workloads", each with its kernel rooflines, the end-to-end number through the C ABI
with host buffers, and the fp64 oracle timed on a bounded sample on the host cores;
plus the SM clocks sampled during the timed regions.  Beside the step, each prefill
workload also times two kernels alone: the attention-output ShortConv (k_output_conv) and
the qkvr projections with the prologue fused in (k_qkvr, from hidden states of width
8192), each with its own roofline entry.

  python bench.py [--steps K] [--warmup W] [--impl reference] [--only NAME ...]

One GPU only.  The prefill kernel multicasts K/V tiles inside a CTA pair, a form the
library confines to single-GPU runs: --gpus N > 1 (or a torch.distributed launch with
more than one rank) is refused before any GPU is touched.  The reference arm (the CPU
oracle) touches no GPU; under a multi-rank launch its rank 0 alone runs.
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
                    "relative_bias_hybrid_gb300/csrc/fp8.cuh", "relative_bias_hybrid_gb300/csrc/common.cuh"],
    "k_prologue": ["relative_bias_hybrid_gb300/csrc/prologue.cu", "relative_bias_hybrid_gb300/csrc/conv4.cuh",
                   "relative_bias_hybrid_gb300/csrc/fp8.cuh", "relative_bias_hybrid_gb300/csrc/common.cuh"],
    "k_combine": ["relative_bias_hybrid_gb300/csrc/decode.cu", "relative_bias_hybrid_gb300/csrc/common.cuh"],
    "k_output_conv": ["relative_bias_hybrid_gb300/csrc/output_conv.cu", "relative_bias_hybrid_gb300/csrc/conv4.cuh",
                      "relative_bias_hybrid_gb300/csrc/common.cuh"],
    "k_qkvr": ["relative_bias_hybrid_gb300/csrc/qkvr.cu", "relative_bias_hybrid_gb300/csrc/tcgen05.cuh",
               "relative_bias_hybrid_gb300/csrc/cta_pair.cuh",
               "relative_bias_hybrid_gb300/csrc/conv4.cuh", "relative_bias_hybrid_gb300/csrc/fp8.cuh",
               "relative_bias_hybrid_gb300/csrc/common.cuh"],
}
QKVR_D_MODEL = 8192     # hidden width of the qkvr projections' input (Hq * 128)


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


def output_conv_bytes(w, D: int) -> float:
    """y and the residual in, h and out written (bf16 rows of D), conv state read + write,
    taps and gains once."""
    return float(4 * 2 * D * w.N_tok + w.B * 2 * 3 * D * 2 + D * (4 * 4 + 4))


def qkvr_flops(w, d_model: int) -> float:
    """The projections y = x . w^T of the new tokens: 2 FLOP per multiply-add, F = Hq*d +
    2*Hkv*d + Hq*d_r outputs of length d_model each.  The 3 rows per 125-token tile that
    the kernel recomputes for the conv, and the prologue's arithmetic, are not counted."""
    F = (w.Hq + 2 * w.Hkv) * w.head_dim + w.Hq * w.d_r
    return 2.0 * w.N_tok * F * d_model


def decode_bytes(w, kv_dtype: str = "bf16") -> float:
    """Every visible K and V row once per (sequence, KV head), plus q, out, r, P, table.
    An E4M3 row is 128 one-byte codes and a 4-byte scale."""
    row = w.head_dim * 2 if kv_dtype == "bf16" else w.head_dim + 4
    kv = 0
    for n, pre in zip(w.q_lens, w.prefix_lens):
        T = n + pre
        first = 0 if w.window == 0 else max(0, pre - w.window + 1)
        kv += (T - first) * w.Hkv * row * 2
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
    """nvidia-smi sampling of SM clocks, power and throttle reasons during the timed regions
    (every 100 ms).  sm_mhz is the median over the samples taken under load (power at
    least half of the largest seen)."""
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
                 "-lms", "100", "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
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
        sm, mx, pw, reasons = [], [], [], set()
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
                        pw.append(float(parts[2]))
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
        top = max(pw)
        loaded = [c for c, w in zip(sm, pw) if w >= 0.5 * top]
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm), "samples_under_load": len(loaded),
                "sm_mhz_median_all": statistics.median(sm), "power_w_max": top}


def world_from_env():
    """(world size, rank) of a torch.distributed launch, (1, 0) otherwise."""
    return int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0"))


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ---------------------------------------------------------------- oracle (CPU) samples

def sample_flops(w, rows, cu):
    """Algorithmic FLOPs of the attention for the listed token rows (all heads)."""
    total = 0.0
    seq = np.searchsorted(cu, rows, side="right") - 1
    lim = w.rel_extent if w.window == 0 else min(w.rel_extent, w.window)
    for t, b in zip(rows, seq):
        i = w.prefix_lens[b] + (t - cu[b])
        vis = i + 1 if w.window == 0 else min(i + 1, w.window)
        total += (4.0 * w.head_dim * vis + 2.0 * w.d_r * min(i + 1, lim)) * w.Hq
    return total


class HostCopy:
    """What the oracle needs of a measured workload, copied to the host before the device
    buffers are freed: normalised queries and caches (bf16 bits), r, P, lengths, table."""

    def __init__(self, w, x, q_out, seqs=None):
        from relative_bias_hybrid_gb300 import inputs as gen
        self.w = w
        self.B_full = w.B
        self.e4m3 = x["k_cache"].dtype == torch.uint8
        if seqs is None:
            self.x = {k: x[k].cpu() for k in ("cu_seqlens_q", "seqlen_k", "r", "P", "block_table")}
            self.q = gen.bits(q_out)
            if self.e4m3:
                # codes and row scales; the oracle leg dequantises them
                self.kc = (x["k_cache"].cpu().numpy(), x["k_scale"].cpu().numpy())
                self.vc = (x["v_cache"].cpu().numpy(), x["v_scale"].cpu().numpy())
            else:
                self.kc, self.vc = gen.bits(x["k_cache"]), gen.bits(x["v_cache"])
            return
        # decode: a few whole sequences, their cache blocks gathered and renumbered
        import dataclasses
        bt = x["block_table"].cpu().numpy()
        sk = x["seqlen_k"].cpu().numpy()
        cu = x["cu_seqlens_q"].cpu().numpy()
        blocks, table = [], np.full((len(seqs), bt.shape[1]), -1, np.int32)
        for i, b in enumerate(seqs):
            n = (int(sk[b]) + w.block_size - 1) // w.block_size
            table[i, :n] = np.arange(len(blocks), len(blocks) + n)
            blocks.extend(bt[b, :n].tolist())
        idx = torch.as_tensor(np.asarray(blocks, np.int64), device=x["k_cache"].device)
        if self.e4m3:
            # codes and row scales; the oracle leg dequantises them
            self.kc = (x["k_cache"].index_select(0, idx).cpu().numpy(), x["k_scale"].index_select(0, idx).cpu().numpy())
            self.vc = (x["v_cache"].index_select(0, idx).cpu().numpy(), x["v_scale"].index_select(0, idx).cpu().numpy())
        else:
            self.kc = gen.bits(x["k_cache"].index_select(0, idx))
            self.vc = gen.bits(x["v_cache"].index_select(0, idx))
        rows = np.concatenate([np.arange(cu[b], cu[b + 1]) for b in seqs]).astype(np.int64)
        ridx = torch.as_tensor(rows, device=q_out.device)
        self.q = gen.bits(q_out.index_select(0, ridx))
        q_lens = [int(cu[b + 1] - cu[b]) for b in seqs]
        self.w = dataclasses.replace(w, name=f"{w.name}[{len(seqs)} seqs]", q_lens=q_lens,
                                     prefix_lens=[int(sk[b]) - q for b, q in zip(seqs, q_lens)])
        cus = np.zeros(len(seqs) + 1, np.int32)
        cus[1:] = np.cumsum(q_lens)
        self.x = {"cu_seqlens_q": torch.from_numpy(cus), "seqlen_k": torch.from_numpy(sk[list(seqs)].copy()),
                  "r": x["r"].index_select(0, ridx).cpu(), "P": x["P"].cpu(),
                  "block_table": torch.from_numpy(table)}


def _dequantise_host_cache(h):
    """An E4M3 host copy's cache as the kernels read it: code * scale, exact in bf16."""
    if h.e4m3:
        import oracle
        from relative_bias_hybrid_gb300 import inputs as gen
        h.kc, h.vc = (gen.bits(torch.from_numpy(oracle.dequantize_e4m3(c, sc)).to(torch.bfloat16))
                      for c, sc in (h.kc, h.vc))
        h.e4m3 = False


def _oracle_time(h, rows, n_threads):
    import oracle
    t0 = time.perf_counter()
    oracle.attention_for_inputs(h.x, h.w, h.q, h.kc, h.vc, rows=rows, n_threads=n_threads)
    return time.perf_counter() - t0


def cpu_baseline_prefill(h, target_s, seed=0):
    """fp64 oracle on a bounded sample of a prefill workload's query rows (all heads), on
    all host cores; scaled to TFLOP/s by the sample's algorithmic FLOP."""
    import oracle
    oracle.build()
    _dequantise_host_cache(h)
    w = h.w
    cu = h.x["cu_seqlens_q"].numpy()
    rng = np.random.default_rng(seed)
    cores = host_cores()
    n = 8
    rows = np.sort(rng.choice(w.N_tok, size=n, replace=False)).astype(np.int32)
    dt = _oracle_time(h, rows, cores)
    if dt < target_s / 3:
        n = int(min(w.N_tok, max(n, n * target_s / max(dt, 1e-3))))
        rows = np.sort(rng.choice(w.N_tok, size=n, replace=False)).astype(np.int32)
        dt = _oracle_time(h, rows, cores)
    fl = sample_flops(w, rows, cu)
    return {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"{len(rows)} of {w.N_tok} query rows (all {w.Hq} heads), {fl:.3g} FLOP in {dt:.1f} s"}


def cpu_baseline_decode(h, target_s):
    """fp64 oracle on the first sequences of the copied decode sample (all their rows and
    heads), as many as fit about target_s; scaled to GB/s by their algorithmic bytes."""
    import dataclasses
    import oracle
    oracle.build()
    kv = "e4m3" if h.e4m3 else "bf16"
    _dequantise_host_cache(h)
    cores = host_cores()
    cu = h.x["cu_seqlens_q"].numpy()
    n_seq = 1
    while True:
        rows = np.arange(0, cu[n_seq], dtype=np.int32)
        dt = _oracle_time(h, rows, cores)
        if dt >= target_s / 3 or n_seq == h.w.B:
            break
        n_seq = int(min(h.w.B, max(n_seq + 1, n_seq * target_s / max(dt, 1e-3))))
    sub = dataclasses.replace(h.w, q_lens=h.w.q_lens[:n_seq], prefix_lens=h.w.prefix_lens[:n_seq])
    nbytes = decode_bytes(sub, kv)
    return {"value": nbytes / dt / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{n_seq} of {h.B_full} sequences (all {cu[n_seq]} query rows, all {h.w.Hq} heads), "
                      f"{nbytes:.3g} algorithmic bytes in {dt:.1f} s"}


def run_reference(args, world, rank):
    """--impl reference: the fp64 CPU oracle, timed on the host cores, on the headline
    workload and metric (each step a bounded sample of query rows)."""
    if rank != 0:
        return
    from relative_bias_hybrid_gb300 import inputs as gen
    import oracle
    oracle.build()
    w = gen.workload("full")
    x = gen.make_inputs(w, seed=0, device="cpu")
    ref = oracle.prologue_for_inputs(x, w)
    h = HostCopy.__new__(HostCopy)
    h.w, h.q, h.kc, h.vc = w, ref["q_out"], ref["k_cache"], ref["v_cache"]
    h.x = {k: x[k] for k in ("cu_seqlens_q", "seqlen_k", "r", "P", "block_table")}
    cu = x["cu_seqlens_q"].numpy()
    cores = host_cores()
    rng = np.random.default_rng(1)
    rows_per_step = 16
    times, flops = [], []
    for it in range(args.warmup + args.steps):
        rows = np.sort(rng.choice(w.N_tok, size=rows_per_step, replace=False)).astype(np.int32)
        dt = _oracle_time(h, rows, cores)
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

def timed_steps(step, steps, warmup, flush, stream):
    """Three timed loops of warmup + steps passes, each pass bracketed by CUDA events on the
    launching stream with an L2 flush (a 256 MiB write) before it, outside the events: the
    whole step (prologue then attention, nothing recorded between them, so the attention
    kernel's launch may overlap the prologue's tail), the attention call(s) alone and the
    prologue alone.  Returns the per-pass ms lists of the three."""
    def loop(body):
        with torch.cuda.stream(stream):
            for _ in range(warmup):
                flush.zero_()
                body()
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        with torch.cuda.stream(stream):
            for e0, e1 in evs:
                flush.zero_()
                e0.record(stream)
                body()
                e1.record(stream)
        torch.cuda.synchronize()
        return [e0.elapsed_time(e1) for e0, e1 in evs]

    tot = loop(lambda: step.run(stream))
    att = loop(lambda: step.run_attention(stream))
    pro = loop(lambda: step.run_prologue(stream))
    return tot, att, pro


def e2e_steps(steps_pair, x_host, steps, warmup, stream):
    """Per step: pinned host -> device copies of the step's inputs, the C-ABI calls and
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


DECODE_ORACLE_SEQS = 16


def time_output_conv(w, args, dev, stream, flush, peaks, name):
    """The attention-output ShortConv + residual + RMSNorm over the workload's new tokens
    at hidden width Hq * 128, timed alone: warm-up calls, then args.steps calls each
    bracketed by CUDA events on the launching stream, with the L2 flush between them
    (outside the events).  Returns its roofline entry and the launches timed."""
    from relative_bias_hybrid_gb300 import inputs as gen
    from relative_bias_hybrid_gb300.step import OutputConvStep
    D = w.Hq * w.head_dim
    x = gen.make_output_conv_inputs(w, seed=0, D=D, device=dev)
    oc = OutputConvStep(w, x)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            flush.zero_()
            oc.run(stream)
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    with torch.cuda.stream(stream):
        for e0, e1 in evs:
            flush.zero_()
            e0.record(stream)
            oc.run(stream)
            e1.record(stream)
    torch.cuda.synchronize()
    if oc.device_status() != 0:
        raise RuntimeError(f"{name}: output conv device status {oc.device_status()}")
    ms = sum(e0.elapsed_time(e1) for e0, e1 in evs) / len(evs)
    nbytes = output_conv_bytes(w, D)
    gbs = nbytes / (ms * 1e-3) / 1e9
    roof = {"bound": "hbm", "kernel": "k_output_conv", "achieved": gbs, "peak": peaks["hbm"],
            "unit": "GB/s", "frac": gbs / peaks["hbm"], "traffic": ncu_traffic("k_output_conv", name),
            "algorithmic_bytes_per_launch": nbytes, "ms": ms, "hidden": D,
            "note": "timed alone, outside the step (its input stands in for the o_proj output)"}
    del x, oc
    return roof, args.steps


def time_qkvr(w, args, dev, stream, flush, peaks, name):
    """The qkvr projections of the workload's new tokens (hidden width QKVR_D_MODEL) with the
    prologue fused in, timed alone like the output conv.  Returns its roofline entry and the
    launches timed."""
    from relative_bias_hybrid_gb300 import inputs as gen
    from relative_bias_hybrid_gb300.step import QkvrStep
    x = gen.make_qkvr_inputs(w, QKVR_D_MODEL, seed=0, device=dev)
    qk = QkvrStep(w, x)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            flush.zero_()
            qk.run(stream)
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    with torch.cuda.stream(stream):
        for e0, e1 in evs:
            flush.zero_()
            e0.record(stream)
            qk.run(stream)
            e1.record(stream)
    torch.cuda.synchronize()
    if qk.device_status() != 0:
        raise RuntimeError(f"{name}: qkvr device status {qk.device_status()}")
    ms = sum(e0.elapsed_time(e1) for e0, e1 in evs) / len(evs)
    fl = qkvr_flops(w, QKVR_D_MODEL)
    tf = fl / (ms * 1e-3) / 1e12
    roof = {"bound": "tensor", "kernel": "k_qkvr", "achieved": tf, "peak": peaks["bf16"], "unit": "TFLOP/s",
            "frac": tf / peaks["bf16"], "peak_src": peaks["src"] + " (burst bf16)",
            "frac_of_sustained": tf / peaks["bf16_sustained"], "traffic": ncu_traffic("k_qkvr", name),
            "algorithmic_flop_per_launch": fl, "ms": ms, "d_model": QKVR_D_MODEL,
            "note": "timed alone, outside the step: the qkvr projections with the prologue fused in, "
                    "from synthetic hidden states"}
    del x, qk
    return roof, args.steps


def measure(name, args, peaks, dev, stream, flush):
    """Device-timed steps, then end-to-end steps, of one workload.  Returns its report
    (without cpu_baseline), the launches inside its timed regions and the host copy the
    oracle sample needs."""
    from relative_bias_hybrid_gb300 import inputs as gen
    from relative_bias_hybrid_gb300.step import AttentionStep
    kv = "e4m3" if name.endswith("_e4m3") else "bf16"
    w = gen.workload(name.replace("_e4m3", ""))
    mode = "decode" if name.startswith("decode") else "prefill"
    x = gen.make_inputs(w, seed=0, device=dev, kv_dtype=kv)
    step = AttentionStep(w, x, mode=mode)
    tot, att, pro = timed_steps(step, args.steps, args.warmup, flush, stream)
    if step.device_status() != 0:
        raise RuntimeError(f"{name}: device status {step.device_status()} during the timed steps")
    ms, att_ms, pro_ms = (sum(v) / len(v) for v in (tot, att, pro))

    # end to end through the C ABI: a second set of input/output buffers over the same
    # cache and conv state
    x_host = {n: x[n].cpu().pin_memory() for n in ("q", "k", "v", "r")}
    x2 = dict(x)
    for n in ("q", "k", "v", "r"):
        x2[n] = torch.empty_like(x[n])
    step2 = AttentionStep(w, x2, mode=mode, num_splits=step.num_splits)
    e2e_ms, h2d, d2h = e2e_steps((step, step2), x_host, args.steps, args.warmup, stream)
    if step.device_status() | step2.device_status():
        raise RuntimeError(f"{name}: device status set during the end-to-end steps")
    # timed: the step loop, the attention loop, the prologue loop, the end-to-end loop
    n_att = step.launches_per_run() - 1
    launches = args.steps * (2 * step.launches_per_run() + n_att + 1)
    oc_roof = qk_roof = None
    if kv == "bf16":            # (the output conv does not depend on the cache type)
        oc_roof, oc_launches = time_output_conv(w, args, dev, stream, flush, peaks, name)
        launches += oc_launches
    if mode == "prefill" and kv == "bf16":   # (the qkvr kernel's tiles are made for prefill)
        qk_roof, qk_launches = time_qkvr(w, args, dev, stream, flush, peaks, name)
        launches += qk_launches
    extra = {**({"k_output_conv": oc_roof} if oc_roof else {}), **({"k_qkvr": qk_roof} if qk_roof else {})}

    pro_bytes = prologue_bytes(w)
    prologue = {"bound": "hbm", "kernel": "k_prologue", "achieved": pro_bytes / (pro_ms * 1e-3) / 1e9,
                "peak": peaks["hbm"], "unit": "GB/s", "traffic": ncu_traffic("k_prologue", name),
                "algorithmic_bytes_per_launch": pro_bytes, "ms": pro_ms}
    prologue["frac"] = prologue["achieved"] / peaks["hbm"]
    if mode == "prefill":
        fl = attention_flops(w)
        tf = fl / (att_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "kernel": "k_prefill_tc" if kv == "bf16" else "k_dequant_e4m3+k_prefill_tc",
                "achieved": tf, "peak": peaks["bf16"],
                "unit": "TFLOP/s", "frac": tf / peaks["bf16"], "peak_src": peaks["src"] + " (burst bf16)",
                "frac_of_sustained": tf / peaks["bf16_sustained"], "traffic": ncu_traffic("k_prefill_tc", name),
                "algorithmic_flop_per_launch": fl, "ms": att_ms}
        rep = {"workload": w.describe() + ("; step = inkattn_prologue + inkattn_prefill" if kv == "bf16" else
                                           ", E4M3 KV cache with a power-of-two scale per row; step = "
                                           "inkattn_prologue + inkattn_prefill_e4m3 (the blocks read expanded "
                                           "to bf16, then the bf16 prefill)"),
               "value": fl / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": ms,
               "roofline": roof, "rooflines": {"k_prologue": prologue, **extra},
               "e2e": {"value": fl / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                       "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms}}
        host = HostCopy(w, x, step.q_out)
    else:
        nbytes = decode_bytes(w, kv)
        gbs = nbytes / (att_ms * 1e-3) / 1e9
        traffic = ncu_traffic("k_decode_tc", name)
        if step.num_splits > 1 and traffic is not None:
            comb = ncu_traffic("k_combine", name)
            traffic = traffic + comb if comb is not None else None
        roof = {"bound": "hbm", "kernel": "k_decode_tc" + ("+k_combine" if step.num_splits > 1 else ""),
                "achieved": gbs, "peak": peaks["hbm"], "unit": "GB/s", "frac": gbs / peaks["hbm"],
                "peak_src": peaks["src"] + " (copy bandwidth)", "traffic": traffic,
                "algorithmic_bytes_per_launch": nbytes, "ms": att_ms, "num_splits": step.num_splits}
        rep = {"workload": w.describe() + (", E4M3 KV cache with a power-of-two scale per row" if kv == "e4m3" else "")
                           + "; step = inkattn_prologue + inkattn_decode (+ inkattn_combine)",
               "value": nbytes / (ms * 1e-3) / 1e9, "unit": "GB/s", "ms_per_step": ms,
               "roofline": roof, "rooflines": {"k_prologue": prologue, **extra},
               "e2e": {"value": nbytes / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                       "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms}}
        host = HostCopy(w, x, step.q_out, seqs=list(range(DECODE_ORACLE_SEQS)))
    return rep, launches, host


WORKLOADS = ("full", "swa", "ragged", "full_e4m3", "decode", "decode_e4m3")


def run_gpu(args):
    from relative_bias_hybrid_gb300 import build as _b
    _b.build()
    torch.cuda.set_device(0)
    peaks = load_peaks()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.Stream(device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    names = [n for n in WORKLOADS if not args.only or n in args.only]

    reps, hosts, launches = {}, {}, 0
    clocks = ClockSampler(dev.index)
    torch.cuda.synchronize()
    clocks.start()
    for name in names:
        reps[name], n_launch, hosts[name] = measure(name, args, peaks, dev, stream, flush)
        launches += n_launch
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    clk = clocks.stop()
    if not args.no_cpu_baseline:
        per = args.cpu_seconds / len(names)
        for name in names:
            h = hosts.pop(name)
            reps[name]["cpu_baseline"] = (cpu_baseline_decode(h, per) if name.startswith("decode")
                                          else cpu_baseline_prefill(h, per))
    head_name = names[0]
    head = reps.pop(head_name)
    line = {
        "metric": METRIC, "value": head["value"], "unit": head["unit"], "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": head["workload"], "global_batch": 1, "parallelism": "single GPU",
                   "l2": "flushed between steps (256 MiB write, outside the timed events)"},
        "roofline": head["roofline"],
        "rooflines": head["rooflines"],
        "e2e": head["e2e"],
        "workloads": reps,
        "gpu_launches": launches,
        "clocks": clk,
    }
    if "cpu_baseline" in head:
        line["cpu_baseline"] = head["cpu_baseline"]
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["inkattn", "reference"], default="inkattn")
    ap.add_argument("--only", nargs="*", choices=list(WORKLOADS), default=None,
                    help="measure only these workloads (the first one listed in the default order heads the line)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=24.0,
                    help="host-core seconds of oracle work over all workloads' cpu_baseline samples")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)     # at least 3 untimed warm-up steps, reported as used
    world, rank = world_from_env()
    if args.impl == "reference":
        run_reference(args, max(world, args.gpus), rank)
        return 0
    if args.gpus != 1 or world != 1:
        sys.stderr.write("bench.py: one GPU only.  The prefill kernel multicasts K/V tiles inside a CTA pair, "
                         "a form the library confines to single-GPU runs; --gpus must be 1 (no multi-rank launch).\n")
        return 2
    run_gpu(args)
    return 0


if __name__ == "__main__":
    sys.exit(main())
