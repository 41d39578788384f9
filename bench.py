#!/usr/bin/env python
"""Benchmark of the Gated Delta Rule-2 hot path on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one gdr2_forward over the GDN-2 1.3B layer workload (B=4, H=16,
T=4096, d_k=d_v=128, bf16 inputs and o, fp32 state, zero S0): 16,384 tokens
per step.  The headline value is tokens/s with inputs resident in HBM (402 MB
of inputs > the 126 MB L2, so no flush is needed between steps).  The same
JSON line carries:

* roofline: the prefill's algorithmic bytes per call (473.96 MB) / the call's
  mean CUDA-event duration, against the measured HBM copy bandwidth, with the
  mean, median, first and slowest call;
* prefill_fp32_o: the same prefill writing o in fp32 (541.1 MB per call);
* decode: the in-place decode step (B=256, H=16, d=128, fp32 state of 268 MB)
  over 1024 consecutive steps, in HBM GB/s, with its own roofline;
* e2e: the same prefill through the public API from pinned host buffers, the
  host->device copies of every step's inputs and the device->host copies of o
  and S_T inside the timed region (uploads, computation and downloads
  pipelined on three streams);
* long_context: the long-context workload (B=1, H=16, T=65536) through the
  chunk-parallel scan over sequence segments, beside the sequential state pass;
* backward: gdr2_backward (all input gradients) over the same GDN-2 layer
  workload;
* cpu_baseline: the fp64 CPU oracle (as it stands) on a bounded sample of the
  same workload on the host cores;
* clocks: nvidia-smi samples taken during the timed region.

Under torchrun (N > 1) every rank runs its own independent batch (weak
scaling, no collective on the data path); timing is bracketed by barriers and
the slowest rank's time is reported.  ``--impl reference`` times the CPU
oracle instead (rank 0 only) on a bounded sample of the same workload.
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
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

# The B300's nominal HBM3e bandwidth: the roofline's spec figure, reported beside the
# fraction of the measured copy rate (the "peak" of every roofline record)
SPEC_HBM_GBS = 8000.0
METRIC = "GDR-2 fwd tokens/sec at H16 d128 T4K (1×B300); % of roofline; decode GB/s"
WORKLOAD = "gdn2_layer_T4096"
FALLBACK_HBM_GBS = 6400.0
FALLBACK_BF16_TFLOPS = 1800.0


# --------------------------------------------------------------------------
# algorithmic work per launch
# --------------------------------------------------------------------------
def prefill_bytes(B, T, H, dk, dv, esz=2, osz=4, s0=False, st=True):
    """Bytes a perfect prefill must move: the six token inputs read once (esz
    bytes each), o written once (osz bytes), S0 read (if given) and S_T
    written once (fp32)."""
    tok = B * T * H * (4 * dk + 2 * dv) * esz + B * T * H * dv * osz
    state = B * H * dk * dv * 4
    return tok + (state if s0 else 0) + (state if st else 0)


def prefill_flops(B, T, H, dk, dv, C=64):
    """Algorithmic flops of the chunked form per token-head:
    6*dk*dv (three dk x dv state products) + 3*C*dk + 2*C*dv (the C x C
    triangular intra-chunk products counted at half)."""
    return B * T * H * (6 * dk * dv + 3 * C * dk + 2 * C * dv)


def decode_bytes(B, H, dk, dv, esz=2, osz=4):
    """Per decode step: the fp32 state read and written, six token inputs
    read, o written."""
    return B * H * (2 * dk * dv * 4 + (4 * dk + 2 * dv) * esz + dv * osz)


# --------------------------------------------------------------------------
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


def kernel_source_hash(files):
    """Hash of the kernel sources a traffic record was taken on."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "gated_delta_rule_166_b300", "csrc")
    for name in sorted(files):
        try:
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode() + f.read())
        except OSError:
            return None
    return h.hexdigest()[:16]


def traffic_record(kernel_key):
    """dram bytes per launch from the committed ncu summary (profiles/traffic.json),
    if it was taken on the kernel's current sources; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(kernel_key)
    except Exception:
        return None
    current = kernel_source_hash(rec.get("sources", [])) if rec else None
    if not rec or current is None or rec.get("source_hash") != current:
        return None
    return rec.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# --------------------------------------------------------------------------
def dist_setup(args):
    """One process per GPU (torchrun env vars); NCCL on GPUs, gloo without."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        if torch.cuda.is_available():
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:
            dist.init_process_group("gloo")
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def rank_seed(base_seed, rank):
    """Weak scaling: every rank draws its own independent batch."""
    return base_seed + rank


def aggregate_tokens_per_s(tokens_per_rank, ms_max, world):
    """Whole-job throughput: the units all ranks processed / the slowest rank's time."""
    return world * tokens_per_rank / (ms_max / 1e3)


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------------------
def bench_prefill(gdr2, x, steps, warmup, world, out_dtype=torch.bfloat16):
    B, T, H, dk = x.q.shape
    dv = x.v.shape[-1]
    stream = torch.cuda.current_stream()
    o = torch.empty((B, T, H, dv), dtype=out_dtype, device="cuda")
    ST = torch.empty((B, H, dk, dv), dtype=torch.float32, device="cuda")
    for _ in range(warmup):
        gdr2.forward(*x.tensors(), x.S0, o=o, S_T=ST)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    barrier(world)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(steps):
        ev[i][0].record(stream)
        gdr2.forward(*x.tensors(), x.S0, o=o, S_T=ST)
        ev[i][1].record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    total_ms = t0.elapsed_time(t1)
    per_launch = [a.elapsed_time(b) for a, b in ev]
    if gdr2.gdr2_device_status() != 0:
        raise RuntimeError("device-side failure during the timed prefill")
    # each bf16 gdr2_forward launches two kernels: preparation, then the state pass
    return total_ms / steps, per_launch, 2 * steps


def launch_stats(per_launch):
    """Mean, median, first and slowest of the per-call CUDA-event durations (ms)."""
    return {"mean_ms": sum(per_launch) / len(per_launch), "median_ms": statistics.median(per_launch),
            "first_ms": per_launch[0], "max_ms": max(per_launch), "calls": len(per_launch)}


def bench_decode(gdr2, steps=1024, seed=5):
    """1024 in-place decode steps, launched eagerly and replayed from one CUDA
    graph (the launch-bound inner loop of serving); GB/s from the graph replay.
    Every step takes its own token (1024 sets, 6.4 GB, drawn on the device by
    the seeded generator with the decode distributions), so no step's inputs
    are in L2 from an earlier one."""
    from gated_delta_rule_166_b300.inputs import DECODE_WORKLOAD, PrefillInputs, make_decode_state, \
        make_prefill_inputs

    W = DECODE_WORKLOAD
    B, H, dk, dv = W["B"], W["H"], W["dk"], W["dv"]
    S = make_decode_state(B, H, dk, dv, seed=seed).cuda()
    allt = make_prefill_inputs(B, steps, H, dk, dv, dtype=torch.bfloat16, seed=seed * 1_000_003 + 1, device="cuda")
    per_step = [t.transpose(0, 1).contiguous() for t in allt.tensors()]   # [steps, B, H, d]
    del allt
    toks = [PrefillInputs(*(t[s] for t in per_step), None) for s in range(steps)]
    pool = steps
    o = torch.empty((B, H, dv), dtype=torch.float32, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for s in range(8):
            gdr2.decode_step(*toks[s % pool].tensors(), S, o=o)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()

    def timed(fn):
        stream = torch.cuda.current_stream()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b)

    ms_eager = timed(lambda: [gdr2.decode_step(*toks[s % pool].tensors(), S, o=o) for s in range(steps)])
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for s in range(steps):
            gdr2.decode_step(*toks[s % pool].tensors(), S, o=o)
    graph.replay()
    torch.cuda.synchronize()
    ms = timed(graph.replay)
    if gdr2.gdr2_device_status() != 0:
        raise RuntimeError("device-side failure during decode")
    nbytes = decode_bytes(B, H, dk, dv)
    per_step_s = ms / 1e3 / steps
    return {"workload": f"decode B{B} H{H} d{dk} fp32 state, {steps} in-place steps (one CUDA graph)",
            "gbs": nbytes / per_step_s / 1e9, "us_per_step": per_step_s * 1e6,
            "gbs_eager_launches": nbytes / (ms_eager / 1e3 / steps) / 1e9,
            "tokens_per_s": B * steps / (ms / 1e3), "bytes_per_step": nbytes,
            "launches": steps, "input_pool": pool}


def bench_long(gdr2, hbm_gbs, steps=10, warmup=3):
    """The long-context workload (B=1, H=16, T=65536): gdr2_forward with the
    library's segment count for the chunk-parallel scan, and the sequential state
    pass (segments=1) for comparison; CUDA events around `steps` calls each."""
    from gated_delta_rule_166_b300.inputs import WORKLOADS, make_workload

    name = "long_T65536"
    cfg = WORKLOADS[name]
    B, T, H, dk, dv = cfg["B"], cfg["T"], cfg["H"], cfg["dk"], cfg["dv"]
    x = make_workload(name).to("cuda")
    o = torch.empty((B, T, H, dv), dtype=torch.bfloat16, device="cuda")
    ST = torch.empty((B, H, dk, dv), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()

    def timed(segments):
        for _ in range(warmup):
            gdr2.forward(*x.tensors(), x.S0, o=o, S_T=ST, segments=segments)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            gdr2.forward(*x.tensors(), x.S0, o=o, S_T=ST, segments=segments)
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / steps

    ms_auto, ms_seq = timed(None), timed(1)
    if gdr2.gdr2_device_status() != 0:
        raise RuntimeError("device-side failure during the long-context prefill")
    nbytes = prefill_bytes(B, T, H, dk, dv, esz=2, osz=2, s0=x.S0 is not None, st=True)
    achieved = nbytes / (ms_auto / 1e3) / 1e9
    return {"workload": f"{name}: B={B} H={H} T={T} d_k=d_v={dk}, bf16 inputs and o, fp32 S0 and state",
            "ms_per_call": ms_auto, "tokens_per_s": B * T / (ms_auto / 1e3),
            "ms_per_call_sequential": ms_seq, "speedup_vs_sequential": ms_seq / ms_auto,
            "segments": "library choice (gdr2_forward)", "steps": steps, "warmup": warmup,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_gbs, "unit": "GB/s",
                         "frac": achieved / hbm_gbs, "algorithmic_bytes_per_launch": nbytes,
                         "traffic": traffic_record("prefill_" + name),
                         "kernel": "gdr2 prefill: prep2_kernel + chain_kernel (segments) + scan_kernel + correct_kernel"}}


def backward_bytes(B, T, H, dk, dv, esz=2):
    """Bytes a perfect backward pass must move: the six forward inputs and the
    fp32 gradient at o read once, the six fp32 input gradients and dS0 written
    once."""
    tok = B * T * H * ((4 * dk + 2 * dv) * esz + dv * 4 + (4 * dk + 2 * dv) * 4)
    return tok + B * H * dk * dv * 4


def bench_backward(gdr2, hbm_gbs, x, steps=5, warmup=3, batch=None, chunked=True):
    """The gradients over the GDN-2 layer workload (or its first `batch` sequences)
    with a seeded fp32 gradient at o (no gradient at S_T), CUDA events around
    `steps` calls: gdr2_backward_chunked (chunkwise WY form on tensor cores) or,
    with chunked=False, the exact token-sequential gdr2_backward."""
    if batch is not None and batch < x.q.shape[0]:
        from gated_delta_rule_166_b300.inputs import PrefillInputs

        x = PrefillInputs(*(t[:batch].contiguous() for t in x.tensors()),
                          None if x.S0 is None else x.S0[:batch].contiguous())
    B, T, H, dk = x.q.shape
    dv = x.v.shape[-1]
    gen = torch.Generator().manual_seed(11)
    d_o = torch.randn(B, T, H, dv, generator=gen).to("cuda")
    stream = torch.cuda.current_stream()
    fn = gdr2.backward_chunked if chunked else gdr2.backward
    for _ in range(warmup):
        fn(*x.tensors(), x.S0, d_o, None)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        fn(*x.tensors(), x.S0, d_o, None)
    b.record(stream)
    torch.cuda.synchronize()
    if gdr2.gdr2_device_status() != 0:
        raise RuntimeError("device-side failure during the backward pass")
    ms = a.elapsed_time(b) / steps
    nbytes = backward_bytes(B, T, H, dk, dv)
    achieved = nbytes / (ms / 1e3) / 1e9
    kind = "chunked" if chunked else "exact"
    kernels = ("gdr2_backward_chunked: prep2_kernel (maps and backward records) + chain_kernel (start "
               "states) + rchain_kernel + cgrad_kernel per call" if chunked else
               "gdr2_backward: bwd_kernel + bwd_reduce_kernel per call")
    return {"workload": f"{WORKLOAD} backward (B={B}): gradients of all six inputs and S0, fp32, from a "
                        f"seeded fp32 gradient at o",
            "path": kind, "ms_per_call": ms, "tokens_per_s": B * T / (ms / 1e3), "steps": steps,
            "warmup": warmup, "launches_per_call": 4 if chunked else 2,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_gbs, "unit": "GB/s",
                         "frac": achieved / hbm_gbs, "algorithmic_bytes_per_launch": nbytes,
                         "traffic": (traffic_record(("backward_chunked_" if chunked else "backward_") + WORKLOAD)
                                     if batch is None else None),   # the records cover the full workload
                         "kernel": kernels}}


def bench_train_step(gdr2, hbm_gbs, x, steps=5, warmup=3):
    """One training step of the layer (forward, then the gradients of all inputs
    from a seeded fp32 gradient at o) at the GDN-2 layer workload, CUDA events
    around `steps` steps, two ways: gdr2_forward_train + gdr2_backward_from_context
    (the per-chunk context kept, 773 MB) and gdr2_forward + gdr2_backward_chunked
    (recomputed)."""
    B, T, H, dk = x.q.shape
    dv = x.v.shape[-1]
    gen = torch.Generator().manual_seed(11)
    d_o = torch.randn(B, T, H, dv, generator=gen).to("cuda")
    o = torch.empty((B, T, H, dv), dtype=torch.bfloat16, device="cuda")
    S_T = torch.empty((B, H, dk, dv), dtype=torch.float32, device="cuda")
    ctx = torch.empty(gdr2.gdr2_train_context_bytes(B, T, H, dk, dv), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def kept():
        gdr2.forward_train(*x.tensors(), x.S0, o=o, S_T=S_T, ctx=ctx)
        gdr2.backward_from_context(ctx, *x.tensors(), x.S0, d_o, None)

    def recomputed():
        gdr2.forward(*x.tensors(), x.S0, o=o, S_T=S_T)
        gdr2.backward_chunked(*x.tensors(), x.S0, d_o, None)

    def timed(fn):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        if gdr2.gdr2_device_status() != 0:
            raise RuntimeError("device-side failure in the training-step leg")
        return a.elapsed_time(b) / steps

    ms_kept, ms_rec = timed(kept), timed(recomputed)
    return {"workload": f"{WORKLOAD} training step (B={B}): forward (bf16 o) and the gradients of all six "
                        f"inputs, fp32, from a seeded fp32 gradient at o",
            "context_kept": {"ms_per_step": ms_kept, "tokens_per_s": B * T / (ms_kept / 1e3),
                             "context_bytes": ctx.numel(),
                             "kernels": "gdr2_forward_train (prep2_kernel with backward records + chain_kernel "
                                        "keeping every start state) + gdr2_backward_from_context (rchain_kernel + "
                                        "cgrad_kernel)"},
            "recomputed": {"ms_per_step": ms_rec, "tokens_per_s": B * T / (ms_rec / 1e3),
                           "kernels": "gdr2_forward (prep2_kernel + chain_kernel) + gdr2_backward_chunked "
                                      "(prep2_kernel + chain_kernel + rchain_kernel + cgrad_kernel)"},
            "steps": steps, "warmup": warmup}


def packed_offsets(total, n, seed=12):
    """cu_seqlens of `n` ragged sequences covering `total` token rows: n - 1 seeded
    cut points, distinct and uniform over the rows (lengths not multiples of 64)."""
    rng = np.random.default_rng(seed)
    cuts = np.sort(rng.choice(np.arange(1, total), size=n - 1, replace=False))
    return torch.tensor(np.concatenate([[0], cuts, [total]]), dtype=torch.int32)


def bench_packed(gdr2, hbm_gbs, x, steps=20, warmup=3, nseq=8):
    """The GDN-2 layer workload's 16,384 token rows as `nseq` packed sequences of
    seeded ragged lengths (the serving and packed-training layout): CUDA events
    around gdr2_forward_varlen (bf16 o, per-sequence S_T) and around
    gdr2_backward_chunked_varlen (seeded fp32 gradient at o)."""
    B, T, H, dk = x.q.shape
    dv = x.v.shape[-1]
    total = B * T
    toks = [t.reshape(total, H, -1) for t in x.tensors()]
    cu = packed_offsets(total, nseq).to("cuda")
    o = torch.empty((total, H, dv), dtype=torch.bfloat16, device="cuda")
    S_T = torch.empty((nseq, H, dk, dv), dtype=torch.float32, device="cuda")
    gen = torch.Generator().manual_seed(13)
    d_o = torch.randn(total, H, dv, generator=gen).to("cuda")
    stream = torch.cuda.current_stream()

    def timed(fn, n):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(n):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        if gdr2.gdr2_device_status() != 0:
            raise RuntimeError("device-side failure in the packed-sequence leg")
        return a.elapsed_time(b) / n

    fwd_ms = timed(lambda: gdr2.forward_varlen(*toks, cu, None, o=o, S_T=S_T), steps)
    bwd_steps = max(1, min(steps, 5))
    bwd_ms = timed(lambda: gdr2.backward_chunked_varlen(*toks, cu, None, d_o, None), bwd_steps)
    fbytes = total * H * ((4 * dk + 2 * dv) * 2 + dv * 2) + nseq * H * dk * dv * 4
    bbytes = total * H * ((4 * dk + 2 * dv) * 2 + dv * 4 + (4 * dk + 2 * dv) * 4) + nseq * H * dk * dv * 4
    lengths = (cu[1:] - cu[:-1]).tolist()
    return {"workload": f"{WORKLOAD} rows as {nseq} packed sequences of lengths {lengths} (H={H}, "
                        f"d_k=d_v={dk}, bf16 inputs, S0=0)",
            "forward": {"ms_per_call": fwd_ms, "tokens_per_s": total / (fwd_ms / 1e3), "steps": steps,
                        "warmup": warmup, "algorithmic_bytes_per_launch": fbytes,
                        "roofline_frac": fbytes / (fwd_ms / 1e3) / 1e9 / hbm_gbs,
                        "kernel": "gdr2_forward_varlen: chunk_base_kernel + prep2_kernel + chain_kernel"},
            "backward_chunked": {"ms_per_call": bwd_ms, "tokens_per_s": total / (bwd_ms / 1e3),
                                 "steps": bwd_steps, "warmup": warmup, "algorithmic_bytes_per_launch": bbytes,
                                 "roofline_frac": bbytes / (bwd_ms / 1e3) / 1e9 / hbm_gbs,
                                 "kernel": "gdr2_backward_chunked_varlen: chunk_base_kernel + prep2_kernel + "
                                           "chain_kernel + rchain_kernel + cgrad_kernel"}}


def bench_sparse(gdr2, hbm_gbs, steps=10, warmup=3):
    """gdr2_sparse_write over the slot-memory workload (B4 H16 T4096, 2048 slots,
    32 selected per token, d_v 128, bf16 inputs and o): CUDA events around
    `steps` calls, the memory updated in place call after call."""
    from gated_delta_rule_166_b300.inputs import SPARSE_WORKLOAD, make_sparse_workload

    cfg = SPARSE_WORKLOAD
    B, T, H, M, K, dv = cfg["B"], cfg["T"], cfg["H"], cfg["M"], cfg["K"], cfg["dv"]
    x = make_sparse_workload().to("cuda")
    S = x.S0.clone()
    o = torch.empty((B, T, H, dv), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        gdr2.sparse_write(*x.tensors(), S, o=o)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        gdr2.sparse_write(*x.tensors(), S, o=o)
    b.record(stream)
    torch.cuda.synchronize()
    if gdr2.gdr2_device_status() != 0:
        raise RuntimeError("device-side failure during the sparse write")
    ms = a.elapsed_time(b) / steps
    # idx (int32) and q, k, b, log_decay (bf16) per selected slot; v, w in and o out
    # per value channel; the slot memory read and written once
    nbytes = B * T * H * (K * (4 + 4 * 2) + dv * 3 * 2) + 2 * B * H * M * dv * 4
    achieved = nbytes / (ms / 1e3) / 1e9
    return {"workload": f"sparse gated delta write: B={B} H={H} T={T}, M={M} slots, K={K} selected per token, "
                        f"d_v={dv}, bf16 inputs and o, fp32 slot memory",
            "ms_per_call": ms, "tokens_per_s": B * T / (ms / 1e3), "steps": steps, "warmup": warmup,
            "roofline": {"bound": "latency (token-sequential per column tile; memory tile in shared memory)",
                         "achieved": achieved, "peak": hbm_gbs, "unit": "GB/s", "frac": achieved / hbm_gbs,
                         "algorithmic_bytes_per_launch": nbytes, "traffic": None,
                         "kernel": "gdr2 sparse write: sparse_tile_kernel"}}


def bench_e2e(gdr2, x_host, steps, warmup):
    """Pinned host inputs -> device -> gdr2_forward -> o and S_T back to host, every
    step.  Steps are pipelined the way a serving loop would run them: inputs and
    outputs are double-buffered on the device, and the uploads, the computation and
    the downloads run on three streams, so step i + 1's upload overlaps step i's
    download (separate copy engines).  The timed region spans all copies of all
    steps."""
    B, T, H, dk = x_host.q.shape
    dv = x_host.v.shape[-1]
    pinned = [t.pin_memory() for t in x_host.tensors()]
    dev_in = [[torch.empty_like(t, device="cuda") for t in pinned] for _ in range(2)]
    o_h = [torch.empty((B, T, H, dv), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    S_h = [torch.empty((B, H, dk, dv), dtype=torch.float32).pin_memory() for _ in range(2)]
    o_d = [torch.empty((B, T, H, dv), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    S_d = [torch.empty((B, H, dk, dv), dtype=torch.float32, device="cuda") for _ in range(2)]
    up, comp, down = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    done_comp = [torch.cuda.Event() for _ in range(2)]   # step's inputs consumed, outputs written
    done_up = [torch.cuda.Event() for _ in range(2)]
    done_down = [torch.cuda.Event() for _ in range(2)]   # step's outputs read back
    for e in done_comp + done_down:
        e.record(torch.cuda.current_stream())
    torch.cuda.synchronize()

    def step(i):
        k = i & 1
        up.wait_event(done_comp[k])                      # step i - 2 no longer reads these inputs
        with torch.cuda.stream(up):
            for h, d in zip(pinned, dev_in[k]):
                d.copy_(h, non_blocking=True)
        done_up[k].record(up)
        comp.wait_event(done_up[k])
        comp.wait_event(done_down[k])                    # step i - 2's outputs have been read back
        gdr2.forward(*dev_in[k], None, o=o_d[k], S_T=S_d[k], stream=comp)
        done_comp[k].record(comp)
        down.wait_event(done_comp[k])
        with torch.cuda.stream(down):
            o_h[k].copy_(o_d[k], non_blocking=True)
            S_h[k].copy_(S_d[k], non_blocking=True)
        done_down[k].record(down)

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(up)
    for i in range(steps):
        step(warmup + i)
    down.wait_stream(up)
    down.wait_stream(comp)
    b.record(down)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    if gdr2.gdr2_device_status() != 0:
        raise RuntimeError("device-side failure during the end-to-end prefill")
    h2d = sum(t.numel() * t.element_size() for t in pinned)
    d2h = o_h[0].numel() * o_h[0].element_size() + S_h[0].numel() * S_h[0].element_size()
    return ms, h2d, d2h


def oracle_sample(x, pairs):
    """Run the oracle on the (batch, head) pairs in `pairs`; returns seconds,
    token-heads processed and threads used."""
    import oracle

    idx_b = sorted({p[0] for p in pairs})
    hs = sorted({p[1] for p in pairs})
    sel = [t[idx_b][:, :, hs].contiguous() for t in x.tensors()]
    S0 = None if x.S0 is None else x.S0[idx_b][:, hs].contiguous()
    threads = min(oracle.default_threads(), len(idx_b) * len(hs))
    oracle.build()
    t = time.perf_counter()
    oracle.forward(*sel, S0, nthreads=threads)
    dt = time.perf_counter() - t
    return dt, len(idx_b) * len(hs) * x.q.shape[1], threads


def cpu_baseline(x, budget_s=15.0):
    """Time the oracle on a bounded sample: whole sequences of as many heads
    as fit ~budget_s, taken from batch 0 first; also its one-thread times for one
    head of this workload and for the tiny fp32 workload."""
    B, T, H, _ = x.q.shape
    probe = [(0, 0)]
    dt1, th, _ = oracle_sample(x, probe)            # one head, one thread
    rate1 = th / max(dt1, 1e-6)                     # token-heads/s on one thread
    import oracle
    from gated_delta_rule_166_b300.inputs import make_workload

    cores = oracle.default_threads()
    n_pairs = max(1, min(B * H, int(budget_s * rate1 * cores / T)))
    pairs = [(i // H, i % H) for i in range(n_pairs)]
    if n_pairs >= H:                                 # whole batch rows
        n_rows = n_pairs // H
        pairs = [(bi, h) for bi in range(n_rows) for h in range(H)]
    dt, tokheads, threads = oracle_sample(x, pairs)
    tiny = make_workload("tiny_f32")
    t0 = time.perf_counter()
    oracle.forward(*tiny.tensors(), tiny.S0, nthreads=1)
    dt_tiny = time.perf_counter() - t0
    return {"value": (tokheads / H) / dt, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"{len(pairs)} of {B * H} (batch, head) sequences x {T} tokens "
                      f"({tokheads} token-heads, {dt:.1f} s)",
            "one_thread_s": {f"{WORKLOAD}_one_head": dt1, "tiny_f32": dt_tiny}}


# --------------------------------------------------------------------------
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-long", action="store_true", help="skip the long-context prefill leg")
    ap.add_argument("--no-backward", action="store_true", help="skip the backward-pass leg")
    ap.add_argument("--backward-batch", type=int, default=None,
                    help="profiling aid: the backward leg on the first N sequences only")
    ap.add_argument("--no-sparse", action="store_true", help="skip the sparse-write leg")
    ap.add_argument("--no-packed", action="store_true", help="skip the packed-sequence leg")
    ap.add_argument("--no-train", action="store_true", help="skip the training-step leg")
    ap.add_argument("--only", choices=["all", "prefill", "decode", "long", "backward", "sparse", "packed", "train"],
                    default="all",
                    help="profiling aid: run just one leg (decode and long print only that leg)")
    ap.add_argument("--decode-steps", type=int, default=1024)
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    from gated_delta_rule_166_b300.inputs import WORKLOADS, make_workload

    cfg = WORKLOADS[WORKLOAD]
    B, T, H, dk, dv = cfg["B"], cfg["T"], cfg["H"], cfg["dk"], cfg["dv"]
    config = {"workload": f"{WORKLOAD}: B={B} H={H} T={T} d_k=d_v={dk}, bf16 inputs and o, "
                          f"fp32 state, S0=0, chunk 64",
              "global_batch": B, "seq_len": T, "heads": H, "head_dim": dk,
              "l2": "inputs (402 MB) larger than L2 (126 MB); no flush"}

    if args.impl == "reference":
        import oracle

        rank = int(os.environ.get("RANK", "0"))
        world = int(os.environ.get("WORLD_SIZE", "1"))
        if rank != 0:
            return
        x = make_workload(WORKLOAD)
        # each step: the oracle over whole sequences of `per_step` (batch, head) pairs,
        # sized from a one-sequence probe so that the whole run stays near two minutes
        t_pair, _, _ = oracle_sample(x, [(0, 0)])
        per_step = max(1, min(B * H, int(120.0 / (args.steps + args.warmup) / max(t_pair, 1e-3)
                                         * oracle.default_threads())))
        pairs_all = [(i // H, i % H) for i in range(B * H)]
        for s in range(args.warmup):
            oracle_sample(x, [pairs_all[(s * per_step + i) % (B * H)] for i in range(per_step)])
        times, tokheads, threads = [], 0, 0
        for s in range(args.steps):
            pairs = [pairs_all[(s * per_step + i) % (B * H)] for i in range(per_step)]
            dt, th, threads = oracle_sample(x, pairs)
            times.append(dt)
            tokheads += th
        total_s = sum(times)
        ms = 1e3 * total_s / len(times)
        value = (tokheads / H) / total_s
        sample = (f"per step: {per_step} whole (batch, head) sequences x {T} tokens of {WORKLOAD}, "
                  f"fp64 oracle")
        print(json.dumps({
            "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config,
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
        }))
        return

    world, rank, local = dist_setup(args)
    import gated_delta_rule_166_b300 as gdr2

    hbm_gbs, bf16_tflops, peak_src = load_peaks()
    x_host = make_workload(WORKLOAD, seed=rank_seed(cfg["seed"], rank))
    x = x_host.to("cuda")
    torch.cuda.synchronize()

    if args.only == "decode":
        dec = bench_decode(gdr2, steps=args.decode_steps)
        if rank == 0:
            print(json.dumps({"decode": dec}))
        return
    if args.only == "backward":
        bw = bench_backward(gdr2, hbm_gbs, x, steps=min(args.steps, 5), warmup=args.warmup,
                            batch=args.backward_batch)
        bx = bench_backward(gdr2, hbm_gbs, x, steps=min(args.steps, 5), warmup=args.warmup,
                            batch=args.backward_batch, chunked=False)
        if rank == 0:
            print(json.dumps({"backward": bw, "backward_exact": bx}))
        return
    if args.only == "long":
        lc = bench_long(gdr2, hbm_gbs, steps=min(args.steps, 10), warmup=args.warmup)
        if rank == 0:
            print(json.dumps({"long_context": lc}))
        return
    if args.only == "sparse":
        sp = bench_sparse(gdr2, hbm_gbs, steps=min(args.steps, 10), warmup=args.warmup)
        if rank == 0:
            print(json.dumps({"sparse_write": sp}))
        return
    if args.only == "packed":
        pk = bench_packed(gdr2, hbm_gbs, x, steps=min(args.steps, 20), warmup=args.warmup)
        if rank == 0:
            print(json.dumps({"packed": pk}))
        return
    if args.only == "train":
        ts = bench_train_step(gdr2, hbm_gbs, x, steps=min(args.steps, 5), warmup=args.warmup)
        if rank == 0:
            print(json.dumps({"train_step": ts}))
        return

    with ClockSampler(local) as clk:
        ms, per_launch, launches = bench_prefill(gdr2, x, args.steps, args.warmup, world)
    clocks = clk.summary()
    ms_max = max_over_ranks(ms, world)
    tokens = B * T
    value = aggregate_tokens_per_s(tokens, ms_max, world)

    kern_ms = sum(per_launch) / len(per_launch)
    nbytes = prefill_bytes(B, T, H, dk, dv, esz=2, osz=2, s0=False, st=True)
    nflops = prefill_flops(B, T, H, dk, dv)
    achieved = nbytes / (kern_ms / 1e3) / 1e9
    traffic = traffic_record("prefill_" + WORKLOAD)
    roofline = {"bound": "hbm", "achieved": achieved, "peak": hbm_gbs, "unit": "GB/s",
                "frac": achieved / hbm_gbs, "traffic": traffic,
                "spec_peak": SPEC_HBM_GBS, "frac_of_spec": achieved / SPEC_HBM_GBS,
                "kernel": "gdr2 prefill: prep2_kernel + chain_kernel per call",
                "peak_source": f"{peak_src} hbm_gbs (burst copy)",
                "algorithmic_bytes_per_launch": nbytes,
                "tflops": nflops / (kern_ms / 1e3) / 1e12,
                "tensor_frac_of_bf16_peak": nflops / (kern_ms / 1e3) / 1e12 / bf16_tflops,
                "per_call": launch_stats(per_launch)}

    out = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
           "data": "synthetic (seeded; distributions of the GDN-2 layer workload)",
           "config": config, "roofline": roofline, "clocks": clocks,
           "gpu_launches": launches}

    # the same prefill with fp32 o (541.1 MB per call): a secondary figure
    ms32, pl32, _ = bench_prefill(gdr2, x, max(args.steps, 20), args.warmup, world, out_dtype=torch.float32)
    b32 = prefill_bytes(B, T, H, dk, dv, esz=2, osz=4, s0=False, st=True)
    k32 = sum(pl32) / len(pl32)
    out["prefill_fp32_o"] = {"ms_per_call": ms32, "tokens_per_s": tokens / (ms32 / 1e3),
                             "algorithmic_bytes_per_launch": b32,
                             "roofline_frac": b32 / (k32 / 1e3) / 1e9 / hbm_gbs,
                             "per_call": launch_stats(pl32)}

    if args.only == "prefill":
        args.no_e2e = args.no_decode = args.no_cpu_baseline = args.no_long = args.no_backward = True
        args.no_sparse = args.no_packed = args.no_train = True
    if not args.no_e2e:
        e2e_ms, h2d, d2h = bench_e2e(gdr2, x_host, max(3, args.steps // 4), 2)
        e2e_ms = max_over_ranks(e2e_ms, world)
        out["e2e"] = {"value": aggregate_tokens_per_s(tokens, e2e_ms, world), "unit": "tokens/s",
                      "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                      "ms_per_step": e2e_ms}
    if not args.no_decode:
        dec = bench_decode(gdr2, steps=args.decode_steps)
        dtraffic = traffic_record("decode_B256_H16_d128")
        dec["roofline"] = {"bound": "hbm", "achieved": dec["gbs"], "peak": hbm_gbs, "unit": "GB/s",
                           "frac": dec["gbs"] / hbm_gbs, "traffic": dtraffic}
        if dtraffic:
            # part of the in-place state is still in L2 from the previous step, so the
            # DRAM bytes per step are below the algorithmic ones: both rates reported
            dram_gbs = dtraffic / (dec["us_per_step"] / 1e6) / 1e9
            dec["roofline"]["dram_gbs"] = dram_gbs
            dec["roofline"]["dram_frac"] = dram_gbs / hbm_gbs
        out["decode"] = dec
        out["gpu_launches"] = launches  # timed prefill region only; decode launches in out["decode"]
    if not args.no_long:
        out["long_context"] = bench_long(gdr2, hbm_gbs)
    if not args.no_backward:
        out["backward"] = bench_backward(gdr2, hbm_gbs, x)
        out["backward_exact"] = bench_backward(gdr2, hbm_gbs, x, chunked=False)
    if not args.no_sparse:
        out["sparse_write"] = bench_sparse(gdr2, hbm_gbs)
    if not args.no_packed:
        out["packed"] = bench_packed(gdr2, hbm_gbs, x)
    if not args.no_train:
        out["train_step"] = bench_train_step(gdr2, hbm_gbs, x)
    if rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(x_host)
    if rank == 0:
        print(json.dumps(out))
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
