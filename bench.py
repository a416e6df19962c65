"""Benchmark of the Ulysses DistributedAttention forward on GB300.

One step = one pass of the whole hot path over the DiT-like workload (P=4 virtual ranks,
b=2, s=4096, h=32, d=128, bf16 N(0,1)), for both the non-causal and the causal mask:
    all-to-all #1 on Q, K, V  ->  local attention  ->  all-to-all #2 on O   (unfused)
    the fused kernel (exchanges folded into the attention tiles)             (fused)
Every kernel launch is bracketed by CUDA events on the launching stream.

value   = algorithmic attention FLOP of the step / step time (TFLOP/s), whole job.
roofline = the attention kernel against the measured bf16 tensor peak.
e2e     = the same metric with host buffers: per step the pinned-host Q/K/V go to the
          device, the forward runs through the public API, the outputs come back; the
          copies run on two copy streams with three device buffer sets, so the next steps'
          inputs and the previous steps' outputs move while a step computes.
cpu_baseline / --impl reference = the fp64 CPU oracle on a bounded sample of the workload.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
Multi-GPU (torchrun): every rank runs an independent replica (the path needs no exchange
between GPUs on this single-GPU emulation); value sums ranks over the slowest rank's time.
"""
from __future__ import annotations

import argparse
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

METRIC = "Ulysses attn fwd TFLOP/s + a2a permute GB/s, as fraction of GB300 roofline"
# The default line is the DiT-like workload; the others are the named configurations,
# measured on request (--workload).
WORKLOADS = {
    "dit": dict(P=4, b=2, s=4096, h_q=32, h_kv=32, d=128, dtype="bf16", masks=(False, True),
                name="DiT-like MHA: P=4 b=2 s=4096 h=32 d=128 bf16, non-causal + causal, unfused + fused forward"),
    "gqa": dict(P=8, b=1, s=32768, h_q=32, h_kv=8, d=128, dtype="bf16", masks=(True,),
                name="GQA causal: P=8 b=1 s=32768 h_q=32 h_kv=8 d=128 bf16, unfused + fused forward"),
    "long": dict(P=8, b=1, s=131072, h_q=64, h_kv=64, d=128, dtype="bf16", masks=(True,),
                 name="Long-sequence causal: P=8 b=1 s=131072 h=64 d=128 bf16, unfused + fused forward"),
    "usp": dict(P=8, Pu=4, Pr=2, b=1, s=262144, h_q=16, h_kv=16, d=128, dtype="bf16", masks=(True,),
                name="Ulysses x Ring causal: 256K tokens, Ulysses 4 x Ring 2 (P=8), b=1 h=16 d=128 bf16"),
    "tiny": dict(P=2, b=1, s=64, h_q=4, h_kv=4, d=16, dtype="fp32", masks=(False,),
                 name="Tiny exactness case: P=2 b=1 s=64 h=4 d=16 fp32, non-causal, unfused forward"),
}
WORKLOAD = WORKLOADS["dit"]
WORKLOAD_NAME = WORKLOAD["name"]
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def reduce_max_over_ranks(values, device="cpu"):
    """Element-wise maximum over all ranks of the job (identity when not distributed)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return list(values)
    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def job_throughput(units_per_rank, world, slowest_ms):
    """Whole-job rate: every rank processed units_per_rank; the job took the slowest rank's time."""
    return world * units_per_rank / (slowest_ms * 1e-3)


def attn_flops(b, s, hq, d, causal):
    """Algorithmic FLOP of attention: 4*b*h*d per visible (query, key) pair."""
    pairs = s * (s + 1) // 2 if causal else s * s
    return 4 * b * hq * d * pairs


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:  # noqa: BLE001
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.tmp = None

    def start(self):
        try:
            self.tmp = tempfile.NamedTemporaryFile(mode="w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=self.tmp, stderr=subprocess.DEVNULL)
        except Exception:  # noqa: BLE001
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:  # noqa: BLE001
            self.proc.kill()
        self.tmp.flush()
        rows = []
        with open(self.tmp.name) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.tmp.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k in range(4) if r[5 + k].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------------- GPU arm
def run_gpu(args, rank, world):
    import torch

    import sequence_attention_seq_gb300 as uly
    from sequence_attention_seq_gb300 import build as uly_build
    from sequence_attention_seq_gb300.inputs import seq_shards_qkv

    if rank == 0 or not os.path.exists(uly.library_path()):
        uly_build.build()
    if world > 1:
        torch.distributed.barrier()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    w = WORKLOADS[args.workload]
    P, b, s, hq, hkv, d = w["P"], w["b"], w["s"], w["h_q"], w["h_kv"], w["d"]
    S = s // P
    dt = torch.bfloat16 if w["dtype"] == "bf16" else torch.float32
    esz = 2 if dt == torch.bfloat16 else 4
    fused_ok = dt == torch.bfloat16 and S % 128 == 0 and P <= 16
    qs, ks, vs = seq_shards_qkv(P, b, s, hq, hkv, d, dt, seed=rank, device=str(dev))
    q_head = [torch.empty((b, s, hq // P, d), dtype=dt, device=dev) for _ in range(P)]
    k_head = [torch.empty((b, s, hkv // P, d), dtype=dt, device=dev) for _ in range(P)]
    v_head = [torch.empty((b, s, hkv // P, d), dtype=dt, device=dev) for _ in range(P)]
    o_head = [torch.empty((b, s, hq // P, d), dtype=dt, device=dev) for _ in range(P)]
    o_seq = [torch.empty((b, S, hq, d), dtype=dt, device=dev) for _ in range(P)]
    o_fused = [torch.empty((b, S, hq, d), dtype=dt, device=dev) for _ in range(P)]
    stream = torch.cuda.current_stream(dev)

    # (label, kind, bytes moved, flops, callable); one kernel launch each
    tensor_bytes = b * s * hq * d * esz
    kv_bytes = b * s * hkv * d * esz
    ops = []
    for causal in w["masks"]:
        fl = attn_flops(b, s, hq, d, causal)
        tag = "causal" if causal else "noncausal"
        ops += [
            (f"a2a_seq2head_q", "permute", 2 * tensor_bytes, 0, lambda: uly.ulysses_a2a_seq2head(qs, q_head)),
            (f"a2a_seq2head_k", "permute", 2 * kv_bytes, 0, lambda: uly.ulysses_a2a_seq2head(ks, k_head)),
            (f"a2a_seq2head_v", "permute", 2 * kv_bytes, 0, lambda: uly.ulysses_a2a_seq2head(vs, v_head)),
            (f"attn_{tag}", "attention", 0, fl,
             (lambda c=causal: uly.ulysses_local_attention(q_head, k_head, v_head, c, o_head))),
            (f"a2a_head2seq_o", "permute", 2 * tensor_bytes, 0, lambda: uly.ulysses_a2a_head2seq(o_head, o_seq)),
        ]
        if fused_ok:
            ops.append((f"fused_{tag}", "fused", 0, fl,
                        (lambda c=causal: uly.ulysses_dist_attn_fwd(qs, ks, vs, c, fused=True, out_seq=o_fused))))
    step_flops = sum(op[3] for op in ops)

    def step(events=None):
        for n, op in enumerate(ops):
            if events is not None:
                events[n][0].record(stream)
            op[4]()
            if events is not None:
                events[n][1].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if uly.ulysses_device_status(clear=True) != 0:
        raise RuntimeError("a kernel's bounded wait gave up during warm-up")

    ev = [[[torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)] for _ in ops]
          for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    clocks.start()
    time.sleep(0.3)  # let the sampler come up before the timed region
    t_start.record(stream)
    for k in range(args.steps):
        step(ev[k])
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    if world > 1:
        torch.distributed.barrier()
    total_ms = t_start.elapsed_time(t_end)
    if uly.ulysses_device_status(clear=True) != 0:
        raise RuntimeError("a kernel's bounded wait gave up during the timed steps")

    per_op = {}
    for n, op in enumerate(ops):
        per_op.setdefault(op[0], []).extend(ev[k][n][0].elapsed_time(ev[k][n][1]) for k in range(args.steps))

    # attention kernel (fused launches carry the whole forward in one launch)
    attn_launch_ms, attn_launch_flops = [], []
    for n, op in enumerate(ops):
        if op[1] in ("attention", "fused"):
            for k in range(args.steps):
                attn_launch_ms.append(ev[k][n][0].elapsed_time(ev[k][n][1]))
                attn_launch_flops.append(op[3])
    attn_tflops = sum(attn_launch_flops) / (sum(attn_launch_ms) * 1e-3) / 1e12
    perm_ms = [ev[k][n][0].elapsed_time(ev[k][n][1]) for n, op in enumerate(ops) if op[1] == "permute"
               for k in range(args.steps)]
    perm_bytes = [op[2] for op in ops if op[1] == "permute"] * args.steps
    perm_gbs = sum(perm_bytes) / (sum(perm_ms) * 1e-3) / 1e9

    # end to end through the public API with pinned host buffers.  Every step copies its
    # inputs host -> device and every output device -> host inside the timed region; the
    # copies run on their own streams with NBUF device buffer sets, so the next steps' inputs
    # and the previous steps' outputs move while a step computes (as a training loop
    # prefetches its next batches).  The host link carries both directions at once, and with
    # three sets it always has a copy queued (two sets left it idle between steps).
    host_q = [t.cpu().pin_memory() for t in qs]
    host_k = [t.cpu().pin_memory() for t in ks]
    host_v = [t.cpu().pin_memory() for t in vs]
    fused_modes = (False, True) if fused_ok else (False,)
    variants = [(c, f) for c in w["masks"] for f in fused_modes]
    host_o = [[torch.empty((b, S, hq, d), dtype=dt).pin_memory() for _ in range(P)] for _ in variants]
    NBUF = 3
    dev_in = [[[torch.empty_like(t) for t in src] for src in (qs, ks, vs)] for _ in range(NBUF)]
    dev_out = [[[torch.empty((b, S, hq, d), dtype=dt, device=dev) for _ in range(P)] for _ in variants]
               for _ in range(NBUF)]
    h2d = sum(t.numel() * esz for t in host_q + host_k + host_v)
    d2h = sum(t.numel() * esz for ho in host_o for t in ho)
    ws = [torch.empty(uly.ulysses_dist_attn_workspace_bytes(P, b, s, hq, hkv, d, dt, False),
                      dtype=torch.uint8, device=dev) for _ in range(NBUF)]
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(NBUF)]       # inputs of buffer i have landed
    ev_done = [torch.cuda.Event() for _ in range(NBUF)]     # compute on buffer i has finished
    ev_copied = [torch.cuda.Event() for _ in range(NBUF)]   # outputs of buffer i are on the host

    def upload(k):
        i = k % NBUF
        s_in.wait_event(ev_done[i])  # step k-NBUF has finished reading these inputs
        with torch.cuda.stream(s_in):
            for src, dst in zip(host_q + host_k + host_v, [t for grp in dev_in[i] for t in grp]):
                dst.copy_(src, non_blocking=True)
        ev_in[i].record(s_in)

    def compute_and_download(k):
        i = k % NBUF
        stream.wait_event(ev_in[i])
        stream.wait_event(ev_copied[i])  # step k-NBUF's outputs have left these buffers
        q_i, k_i, v_i = dev_in[i]
        for n, (causal, fused) in enumerate(variants):
            uly.ulysses_dist_attn_fwd(q_i, k_i, v_i, causal, fused=fused, out_seq=dev_out[i][n],
                                      workspace=None if fused else ws[i], stream=stream)
        ev_done[i].record(stream)
        s_out.wait_event(ev_done[i])
        with torch.cuda.stream(s_out):
            for n in range(len(variants)):
                for o, ho in zip(dev_out[i][n], host_o[n]):
                    ho.copy_(o, non_blocking=True)
        ev_copied[i].record(s_out)

    def run_e2e(n_steps):
        for i in range(NBUF):  # nothing is pending on any buffer
            ev_done[i].record(stream)
            ev_copied[i].record(stream)
        for k in range(min(NBUF - 1, n_steps)):
            upload(k)
        for k in range(n_steps):
            if k + NBUF - 1 < n_steps:
                upload(k + NBUF - 1)
            compute_and_download(k)
        stream.wait_stream(s_out)  # the last outputs are on the host before the clock stops

    run_e2e(max(1, args.warmup))
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    run_e2e(args.steps)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = e0.elapsed_time(e1)

    res = dict(total_ms=total_ms, e2e_ms=e2e_ms, attn_tflops=attn_tflops, perm_gbs=perm_gbs, clocks=clk,
               per_op={k: statistics.mean(v) for k, v in per_op.items()}, step_flops=step_flops,
               attn_launch_ms=statistics.mean(attn_launch_ms), h2d=h2d, d2h=d2h,
               n_launches=len(ops) * args.steps)
    return res


# -------------------------------------------------------------------- CPU oracle
def oracle_sample(budget_s=12.0, seed=0):
    """Times the fp64 oracle on a bounded sample of the workload: the exchanges at full size
    and sampled attention rows (each row exact), until the time budget is spent."""
    import random

    import torch

    import oracle
    from sequence_attention_seq_gb300.inputs import seq_shards_qkv

    w = WORKLOAD
    P, b, s, hq, hkv, d = w["P"], w["b"], w["s"], w["h_q"], w["h_kv"], w["d"]
    qs, ks, vs = seq_shards_qkv(P, b, s, hq, hkv, d, torch.bfloat16, seed=seed)
    t0 = time.perf_counter()
    q_head = oracle.seq2head(qs)
    oracle.seq2head(ks)
    oracle.seq2head(vs)
    oracle.head2seq(q_head)
    t_perm = time.perf_counter() - t0
    perm_bytes = 2 * 4 * b * s * hq * d * 2
    rng = random.Random(seed)
    flops, rows, t_attn = 0, 0, 0.0
    S = s // P
    while t_attn < budget_s:
        causal = rows % 2 == 1
        smp = [(rng.randrange(P), rng.randrange(b), rng.randrange(S), rng.randrange(hq)) for _ in range(8)]
        t1 = time.perf_counter()
        oracle.dist_attn_rows(qs, ks, vs, causal, smp)
        t_attn += time.perf_counter() - t1
        for (j, _, t, _) in smp:
            keys = (j * S + t + 1) if causal else s
            flops += 4 * d * keys
        rows += len(smp)
    return dict(tflops=flops / t_attn / 1e12, rows=rows, t_attn=t_attn, perm_gbs=perm_bytes / t_perm / 1e9,
                t_perm=t_perm)


def cpu_baseline_obj(smp):
    return {"value": smp["tflops"], "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
            "sample": (f"{smp['rows']} attention rows (exact fp64, mixed causal/non-causal) of the DiT workload in "
                       f"{smp['t_attn']:.1f} s, plus the four exchanges at full size "
                       f"({smp['perm_gbs']:.2f} GB/s); single thread of {os.cpu_count()} host cores")}


KERNEL_REGION_END = b"// ---------------------------------------------------------------- host side"


def kernel_source_digest():
    """Digest of the forward attention kernel's source: attn_tc.cu up to its host-side
    section (the kernel and its device helpers) and device_common.cuh.  The traffic figure
    belongs to one version of that code; launchers and the backward do not change it."""
    import hashlib

    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "sequence_attention_seq_gb300", "csrc")
    with open(os.path.join(csrc, "attn_tc.cu"), "rb") as f:
        text = f.read()
    if KERNEL_REGION_END not in text:
        return None
    h.update(text.split(KERNEL_REGION_END)[0])
    with open(os.path.join(csrc, "device_common.cuh"), "rb") as f:
        h.update(f.read())
    return h.hexdigest()


def measured_traffic(workload):
    """DRAM bytes per attention launch from the committed ncu capture, if it was taken on
    this exact kernel source and workload; else None."""
    path = os.path.join(ROOT, "profiles", "attn_tc_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except Exception:  # noqa: BLE001
        return None
    if rec.get("source_sha256") != kernel_source_digest() or rec.get("workload") != workload:
        return None
    return rec.get("dram_bytes_per_launch_mean")


def run_permute_sweep(args):
    """Exchange bandwidth over bf16 [P][1, s/P, 64, 128] with uniform random bits."""
    import torch

    import sequence_attention_seq_gb300 as uly
    from sequence_attention_seq_gb300 import build as uly_build
    from sequence_attention_seq_gb300.inputs import random_bits

    uly_build.build()
    peaks, _ = load_peaks()
    h, d = 64, 128
    rows = []
    for s in (8192, 32768, 131072, 262144):
        for P in (2, 4, 8, 16, 32, 64):
            xs = [random_bits((1, s // P, h, d), torch.bfloat16, seed=j, device="cuda") for j in range(P)]
            hd = [torch.empty((1, s, h // P, d), dtype=torch.bfloat16, device="cuda") for _ in range(P)]
            back = [torch.empty_like(x) for x in xs]
            nbytes = 2 * s * h * d * 2
            res = {}
            for name, fn in (("seq2head", lambda: uly.ulysses_a2a_seq2head(xs, hd)),
                             ("head2seq", lambda: uly.ulysses_a2a_head2seq(hd, back))):
                for _ in range(max(3, args.warmup)):
                    fn()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                reps = 20
                torch.cuda.synchronize()
                e0.record()
                for _ in range(reps):
                    fn()
                e1.record()
                torch.cuda.synchronize()
                res[name] = nbytes / (e0.elapsed_time(e1) / reps * 1e-3) / 1e9
            exact = all(torch.equal(a.view(torch.int16), c.view(torch.int16)) for a, c in zip(xs, back))
            row = {"s": s, "P": P, "run_bytes": h // P * d * 2, "seq2head_gbs": res["seq2head"],
                   "head2seq_gbs": res["head2seq"], "round_trip_bit_exact": exact}
            rows.append(row)
            print(json.dumps(row))
            del xs, hd, back
            torch.cuda.empty_cache()
    allv = [r[k] for r in rows for k in ("seq2head_gbs", "head2seq_gbs")]
    print(json.dumps({"metric": "a2a permute GB/s (read+write), bf16 [P][1,s/P,64,128] sweep", "unit": "GB/s",
                      "min": min(allv), "median": statistics.median(allv), "max": max(allv),
                      "peak": peaks["hbm_gbs"], "median_frac": statistics.median(allv) / peaks["hbm_gbs"],
                      "all_bit_exact": all(r["round_trip_bit_exact"] for r in rows)}))


def run_backward(args):
    """Backward of the Ulysses attention (not part of the default line): per mask, the local
    backward alone (row statistics + dK/dV + dQ kernels, head layout) and the whole
    distributed backward (exchange of Q, K, V, dO; local backward; exchange of dQ, dK, dV),
    each call bracketed by CUDA events.  FLOP/s count the algorithmic 2.5x forward FLOPs
    (the five tile products S, dP, dV, dK, dQ); the kernels execute 3.5x (S and dP twice)."""
    import torch

    import sequence_attention_seq_gb300 as uly
    from sequence_attention_seq_gb300 import build as uly_build
    from sequence_attention_seq_gb300.inputs import global_grad, seq_shards_qkv, shard_seq

    uly_build.build()
    w = WORKLOADS[args.workload]
    P, b, s, hq, hkv, d = w["P"], w["b"], w["s"], w["h_q"], w["h_kv"], w["d"]
    if w["dtype"] != "bf16":
        raise SystemExit("the backward kernels are bf16 only")
    dev = torch.device("cuda", 0)
    qs, ks, vs = seq_shards_qkv(P, b, s, hq, hkv, d, torch.bfloat16, seed=0, device="cuda")
    dos = shard_seq(global_grad(b, s, hq, d, torch.bfloat16, seed=1, device="cuda"), P)
    qh, kh, vh, doh = (uly.ulysses_a2a_seq2head(x) for x in (qs, ks, vs, dos))
    peaks, peak_src = load_peaks()
    clocks = ClockSampler(0)
    rows = {}
    clocks.start()
    time.sleep(0.3)
    for causal in w["masks"]:
        tag = "causal" if causal else "noncausal"
        o, lse = uly.ulysses_dist_attn_fwd_lse(qs, ks, vs, causal)
        oh = uly.ulysses_a2a_seq2head(o)
        grads_h = ([torch.empty_like(x) for x in qh], [torch.empty_like(x) for x in kh],
                   [torch.empty_like(x) for x in vh])
        grads_s = ([torch.empty_like(x) for x in qs], [torch.empty_like(x) for x in ks],
                   [torch.empty_like(x) for x in vs])
        ws_l = torch.empty(uly.ulysses_attn_bwd_workspace_bytes(P, b, s, hq, hkv, d, torch.bfloat16, False),
                           dtype=torch.uint8, device=dev)
        ws_d = torch.empty(uly.ulysses_attn_bwd_workspace_bytes(P, b, s, hq, hkv, d, torch.bfloat16, True),
                           dtype=torch.uint8, device=dev)
        calls = {
            "local_bwd": lambda: uly.ulysses_local_attention_bwd(qh, kh, vh, oh, doh, lse, causal, grads=grads_h,
                                                                 workspace=ws_l),
            "dist_bwd": lambda: uly.ulysses_dist_attn_bwd(qs, ks, vs, o, dos, lse, causal, grads=grads_s,
                                                          workspace=ws_d),
        }
        if P <= 16 and (s // P) % 128 == 0:  # the exchanges folded into the kernels' tile addressing
            calls["dist_bwd_fused"] = lambda: uly.ulysses_dist_attn_bwd(qs, ks, vs, o, dos, lse, causal,
                                                                        grads=grads_s, workspace=ws_l, fused=True)
        fl = 2.5 * attn_flops(b, s, hq, d, causal)
        for name, fn in calls.items():
            for _ in range(max(3, args.warmup)):
                fn()
            torch.cuda.synchronize()
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(args.steps)]
            for e0, e1 in evs:
                e0.record()
                fn()
                e1.record()
            torch.cuda.synchronize()
            ms = statistics.mean(e0.elapsed_time(e1) for e0, e1 in evs)
            rows[f"{name}_{tag}"] = {"ms": ms, "tflops": fl / (ms * 1e-3) / 1e12,
                                     "frac": fl / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"]}
        if uly.ulysses_device_status(clear=True) != 0:
            raise RuntimeError("a kernel's bounded wait gave up")
    clk = clocks.stop()
    print(json.dumps({"metric": "Ulysses attn bwd TFLOP/s (algorithmic: 2.5x forward FLOPs)", "unit": "TFLOP/s",
                      "workload": w["name"], "steps": args.steps, "peak": peaks["bf16_tflops"],
                      "peak_source": f"{peak_src} (bf16 dense, burst)", "results": rows, "clocks": clk}))


def run_overlap(args):
    """The unfused forward against the overlapped one (n_chunks head groups, exchanges on a
    side stream), per mask, each call bracketed by CUDA events on the main stream."""
    import torch

    import sequence_attention_seq_gb300 as uly
    from sequence_attention_seq_gb300 import build as uly_build
    from sequence_attention_seq_gb300.inputs import seq_shards_qkv

    uly_build.build()
    w = WORKLOADS[args.workload]
    P, b, s, hq, hkv, d = w["P"], w["b"], w["s"], w["h_q"], w["h_kv"], w["d"]
    dt = torch.bfloat16 if w["dtype"] == "bf16" else torch.float32
    qs, ks, vs = seq_shards_qkv(P, b, s, hq, hkv, d, dt, seed=0, device="cuda")
    out = [torch.empty_like(q) for q in qs]
    ws = torch.empty(max(1, uly.ulysses_dist_attn_workspace_bytes(P, b, s, hq, hkv, d, dt, False)),
                     dtype=torch.uint8, device="cuda")
    Hq, Hk = hq // P, hkv // P
    chunks = [c for c in (2, 4, 8) if Hq % c == 0 and (Hk % c == 0 or c % Hk == 0)]
    wso = {c: torch.empty(uly.ulysses_dist_attn_overlap_workspace_bytes(P, b, s, hq, hkv, d, dt, c),
                          dtype=torch.uint8, device="cuda") for c in chunks}
    rows = {}
    clocks = ClockSampler(0)
    clocks.start()
    time.sleep(0.3)
    for causal in w["masks"]:
        tag = "causal" if causal else "noncausal"
        fl = attn_flops(b, s, hq, d, causal)
        calls = {"unfused": lambda: uly.ulysses_dist_attn_fwd(qs, ks, vs, causal, fused=False, out_seq=out,
                                                              workspace=ws)}
        for c in chunks:
            calls[f"overlap_{c}"] = (lambda c=c: uly.ulysses_dist_attn_fwd_overlap(qs, ks, vs, causal, n_chunks=c,
                                                                                  out_seq=out, workspace=wso[c]))
        for name, fn in calls.items():
            for _ in range(max(3, args.warmup)):
                fn()
            torch.cuda.synchronize()
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(args.steps)]
            for e0, e1 in evs:
                e0.record()
                fn()
                e1.record()
            torch.cuda.synchronize()
            ms = statistics.mean(e0.elapsed_time(e1) for e0, e1 in evs)
            rows[f"{name}_{tag}"] = {"ms": ms, "tflops": fl / (ms * 1e-3) / 1e12}
    if uly.ulysses_device_status(clear=True) != 0:
        raise RuntimeError("a kernel's bounded wait gave up")
    clk = clocks.stop()
    print(json.dumps({"metric": "Ulysses unfused forward, plain vs exchanges overlapped by head group",
                      "unit": "TFLOP/s (algorithmic attention flops / whole forward time)", "workload": w["name"],
                      "steps": args.steps, "results": rows, "clocks": clk}))


def run_usp(args):
    """The two-level (Ulysses x Ring) forward against the plain Ulysses forward (unfused and
    fused) over the same ranks, each call bracketed by CUDA events; with --backward, the two
    paths' backward instead."""
    import torch

    import sequence_attention_seq_gb300 as uly
    from sequence_attention_seq_gb300 import build as uly_build
    from sequence_attention_seq_gb300.inputs import seq_shards_qkv

    uly_build.build()
    w = WORKLOADS["usp"]
    P, Pu, Pr, b, s, hq, hkv, d = w["P"], w["Pu"], w["Pr"], w["b"], w["s"], w["h_q"], w["h_kv"], w["d"]
    qs, ks, vs = seq_shards_qkv(P, b, s, hq, hkv, d, torch.bfloat16, seed=0, device="cuda")
    out = [torch.empty_like(q) for q in qs]
    ws_u = torch.empty(uly.ulysses_usp_workspace_bytes(Pu, Pr, b, s, hq, hkv, d, torch.bfloat16),
                       dtype=torch.uint8, device="cuda")
    ws_d = torch.empty(uly.ulysses_dist_attn_workspace_bytes(P, b, s, hq, hkv, d, torch.bfloat16, False),
                       dtype=torch.uint8, device="cuda")
    fl = attn_flops(b, s, hq, d, True)
    calls = {
        "usp_4x2": lambda: uly.ulysses_usp_attn_fwd(qs, ks, vs, True, Pu, Pr, out_seq=out, workspace=ws_u),
        "ulysses_unfused_p8": lambda: uly.ulysses_dist_attn_fwd(qs, ks, vs, True, fused=False, out_seq=out,
                                                                workspace=ws_d),
        "ulysses_fused_p8": lambda: uly.ulysses_dist_attn_fwd(qs, ks, vs, True, fused=True, out_seq=out),
    }
    flops = {name: fl for name in calls}
    if args.backward:  # training: the backward of each path (2.5x the forward's algorithmic FLOPs)
        from sequence_attention_seq_gb300.inputs import global_grad, shard_seq

        del ws_d
        dos = shard_seq(global_grad(b, s, hq, d, torch.bfloat16, seed=1, device="cuda"), P)
        o_u, lse_u = uly.ulysses_usp_attn_fwd_lse(qs, ks, vs, True, Pu, Pr)
        o_p, lse_p = uly.ulysses_dist_attn_fwd_lse(qs, ks, vs, True, fused=True)
        grads = ([torch.empty_like(x) for x in qs], [torch.empty_like(x) for x in ks],
                 [torch.empty_like(x) for x in vs])
        ws_ub = torch.empty(uly.ulysses_usp_bwd_workspace_bytes(Pu, Pr, b, s, hq, hkv, d, torch.bfloat16),
                            dtype=torch.uint8, device="cuda")
        ws_pb = torch.empty(max(1, uly.ulysses_attn_bwd_workspace_bytes(P, b, s, hq, hkv, d, torch.bfloat16, True,
                                                                        True)), dtype=torch.uint8, device="cuda")
        calls = {
            "usp_4x2_bwd": lambda: uly.ulysses_usp_attn_bwd(qs, ks, vs, o_u, dos, lse_u, True, Pu, Pr, grads=grads,
                                                            workspace=ws_ub),
            "ulysses_fused_p8_bwd": lambda: uly.ulysses_dist_attn_bwd(qs, ks, vs, o_p, dos, lse_p, True,
                                                                      grads=grads, workspace=ws_pb, fused=True),
        }
        flops = {name: 2.5 * fl for name in calls}
    rows = {}
    clocks = ClockSampler(0)
    clocks.start()
    time.sleep(0.3)
    for name, fn in calls.items():
        for _ in range(max(3, args.warmup)):
            fn()
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        for e0, e1 in evs:
            e0.record()
            fn()
            e1.record()
        torch.cuda.synchronize()
        ms = statistics.mean(e0.elapsed_time(e1) for e0, e1 in evs)
        rows[name] = {"ms": ms, "tflops": flops[name] / (ms * 1e-3) / 1e12}
    if uly.ulysses_device_status(clear=True) != 0:
        raise RuntimeError("a kernel's bounded wait gave up")
    clk = clocks.stop()
    what = "backward" if args.backward else "forward"
    print(json.dumps({"metric": f"two-level Ulysses x Ring {what} vs plain Ulysses over the same 8 ranks",
                      "unit": f"TFLOP/s (algorithmic attention flops / whole {what} time)", "workload": w["name"],
                      "steps": args.steps, "results": rows, "clocks": clk}))


# -------------------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", default="dit", choices=sorted(WORKLOADS))
    ap.add_argument("--permute-sweep", action="store_true",
                    help="measure the exchanges over the permute-only sweep instead of the forward")
    ap.add_argument("--backward", action="store_true",
                    help="measure the attention backward (local and distributed) instead of the forward")
    ap.add_argument("--usp", action="store_true",
                    help="measure the two-level Ulysses x Ring forward on its 256K-token workload")
    ap.add_argument("--overlap", action="store_true",
                    help="measure the unfused forward against the overlapped (chunked) forward")
    args = ap.parse_args()

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.overlap:
        if rank == 0:
            run_overlap(args)
        return
    if args.usp:
        if rank == 0:
            run_usp(args)
        return
    if args.backward:
        if rank == 0:
            run_backward(args)
        return
    if args.permute_sweep:
        if rank == 0:
            run_permute_sweep(args)
        return
    w = WORKLOADS[args.workload]
    esz = 2 if w["dtype"] == "bf16" else 4
    io_bytes = (2 * w["h_q"] + 2 * w["h_kv"]) * w["b"] * w["s"] * w["d"] * esz
    config = {"workload": w["name"], "P": w["P"], "b": w["b"], "s": w["s"], "h_q": w["h_q"], "h_kv": w["h_kv"],
              "d": w["d"], "l2": (f"inputs larger than L2 (Q+K+V+O = {io_bytes / 2**20:.0f} MiB > 129 MB); no flush"
                                  if io_bytes > 129e6 else "inputs smaller than L2: latency-bound exactness case")}

    if args.impl == "reference":
        if rank != 0:
            return
        steps = []
        for k in range(args.warmup + args.steps):
            smp = oracle_sample(budget_s=2.0, seed=k)
            if k >= args.warmup:
                steps.append(smp)
        v = sum(x["tflops"] for x in steps) / len(steps)
        line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "dtype": "f64",
                "data": "synthetic", "config": config,
                "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
                                 "sample": "per step: the four exchanges at full size and ~2 s of exact fp64 "
                                           "attention rows of the DiT workload, single thread"},
                "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    import torch

    if world > 1:
        torch.distributed.init_process_group("nccl")
    res = run_gpu(args, rank, world)
    total_ms, e2e_ms = reduce_max_over_ranks([res["total_ms"], res["e2e_ms"]], device="cuda")
    if rank != 0:
        torch.distributed.destroy_process_group()
        return
    peaks, peak_src = load_peaks()
    if w["dtype"] == "bf16":
        kernel, bound, peak, peak_note = "attn_tc_kernel<%d> (all attention launches of the step)" % w["d"], \
            "tensor", peaks["bf16_tflops"], f"{peak_src} (bf16 dense, burst)"
    else:  # fp32 FMA attention: plain ALU peak, 152 SMs x 128 FMA lanes x 2 flop x max SM clock
        kernel, bound = "attn_fp32_kernel (all attention launches of the step)", "alu"
        peak = 152 * 128 * 2 * peaks.get("sm_max_mhz", 2070.0) * 1e6 / 1e12
        peak_note = "derived: 152 SMs x 128 fp32 FMA/clk x 2 flop x 2070 MHz"
    traffic = measured_traffic(args.workload)
    value = job_throughput(res["step_flops"] * args.steps, world, total_ms) / 1e12
    e2e_value = job_throughput(res["step_flops"] * args.steps, world, e2e_ms) / 1e12
    cpu = None
    if not args.no_cpu_baseline and world == 1 and args.workload == "dit":
        cpu = cpu_baseline_obj(oracle_sample(budget_s=12.0))
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w["dtype"], "data": f"synthetic (seeded N(0,1) {w['dtype']})",
        "config": config,
        "roofline": {"kernel": kernel, "bound": bound,
                     "achieved": res["attn_tflops"], "peak": peak, "unit": "TFLOP/s",
                     "frac": res["attn_tflops"] / peak,
                     "frac_of_sustained": (res["attn_tflops"] / peaks["bf16_tflops_sustained"]
                                           if bound == "tensor" else None),
                     "peak_source": peak_note, "traffic": traffic},
        "permute": {"achieved": res["perm_gbs"], "peak": peaks["hbm_gbs"], "unit": "GB/s",
                    "frac": res["perm_gbs"] / peaks["hbm_gbs"], "bytes": "read+write of all ranks' data"},
        "per_launch_ms": res["per_op"],
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": res["h2d"],
                "d2h_bytes_per_step": res["d2h"]},
        "gpu_launches": res["n_launches"] * world,
        "clocks": res["clocks"],
        "cpu_baseline": cpu,
    }
    print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
