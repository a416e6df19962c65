"""Benchmark of the Ulysses DistributedAttention forward on GB300.

The default line is the Long-sequence causal workload (P=8 virtual ranks, b=1, s=131072,
h=64, d=128, bf16 N(0,1)).  One step = one pass of the whole hot path over it:
    all-to-all #1 on Q, K, V  ->  local attention  ->  all-to-all #2 on O   (unfused)
    the fused kernel (both exchanges folded into the attention tiles)         (fused)
Every kernel launch is bracketed by CUDA events on the launching stream.

value    = algorithmic attention FLOP of the step / step time (TFLOP/s), whole job.
roofline = the fused attention launch against the measured bf16 tensor peak (burst, and
           the sustained figure beside it); the unfused attention launch is reported too.
permute  = the exchanges of the step (2 GiB tensors, far beyond L2) against the measured
           HBM copy rate.
e2e      = the fused forward through the public API with host buffers: per step the
           pinned-host Q/K/V go to the device, the call runs, the output comes back; the
           copies run on two copy streams with three device buffer sets, so the next steps'
           inputs and the previous steps' outputs move while a step computes.
extra    = the DiT-like and GQA workloads, each in a timed region of its own after the
           main one (attention launches and exchanges), and their training backward
           (the fused distributed backward, per mask).
cpu_baseline / --impl reference = the fp64 CPU oracle on a bounded sample of the workload
           (exact output rows, extrapolated to a rate).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference] [--workload W]
       python bench.py --permute-sweep | --exchange-kernels | --backward | --overlap | --usp
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
WORKLOADS = {
    "long": dict(P=8, b=1, s=131072, h_q=64, h_kv=64, d=128, dtype="bf16", masks=(True,),
                 name="Long-sequence causal: P=8 b=1 s=131072 h=64 d=128 bf16, unfused + fused forward"),
    "dit": dict(P=4, b=2, s=4096, h_q=32, h_kv=32, d=128, dtype="bf16", masks=(False, True),
                name="DiT-like MHA: P=4 b=2 s=4096 h=32 d=128 bf16, non-causal + causal, unfused + fused forward"),
    "gqa": dict(P=8, b=1, s=32768, h_q=32, h_kv=8, d=128, dtype="bf16", masks=(True,),
                name="GQA causal: P=8 b=1 s=32768 h_q=32 h_kv=8 d=128 bf16, unfused + fused forward"),
    "usp": dict(P=8, Pu=4, Pr=2, b=1, s=262144, h_q=16, h_kv=16, d=128, dtype="bf16", masks=(True,),
                name="Ulysses x Ring causal: 256K tokens, Ulysses 4 x Ring 2 (P=8), b=1 h=16 d=128 bf16"),
    "tiny": dict(P=2, b=1, s=64, h_q=4, h_kv=4, d=16, dtype="fp32", masks=(False,),
                 name="Tiny exactness case: P=2 b=1 s=64 h=4 d=16 fp32, non-causal, unfused forward"),
}
DEFAULT_WORKLOAD = "long"
# timed steps when --steps is not given: a multi-second timed region for every workload
DEFAULT_STEPS = {"long": 20, "gqa": 100, "dit": 2000, "usp": 10, "tiny": 400}
# the other named workloads, measured after the main line's timed region: (workload, steps)
EXTRAS = {"long": (("dit", 1000), ("gqa", 60))}
# and the training backward (fused distributed backward) of these: (workload, calls per mask)
EXTRAS_BWD = {"long": (("dit", 300), ("gqa", 30))}
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
        pw = [num(r[3]) for r in rows if num(r[3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k in range(4) if r[5 + k].lower().startswith("active")})
        capped = sum(1 for r in rows if r[8].lower().startswith("active"))
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "sm_mhz_min": min(sm) if sm else None, "power_w_median": statistics.median(pw) if pw else None,
                "reasons": reasons, "samples": len(rows), "samples_sw_power_cap": capped}


# ------------------------------------------------------------------------- GPU arm
def forward_ops(uly, torch, w, dev, seed):
    """The launches of one step of workload w, (label, kind, bytes moved, flops, callable),
    one kernel launch each, plus the seq-layout inputs."""
    from sequence_attention_seq_gb300.inputs import seq_shards_qkv

    P, b, s, hq, hkv, d = w["P"], w["b"], w["s"], w["h_q"], w["h_kv"], w["d"]
    S = s // P
    dt = torch.bfloat16 if w["dtype"] == "bf16" else torch.float32
    esz = 2 if dt == torch.bfloat16 else 4
    fused_ok = dt == torch.bfloat16 and S % 128 == 0
    qs, ks, vs = seq_shards_qkv(P, b, s, hq, hkv, d, dt, seed=seed, device=str(dev))
    q_head = [torch.empty((b, s, hq // P, d), dtype=dt, device=dev) for _ in range(P)]
    k_head = [torch.empty((b, s, hkv // P, d), dtype=dt, device=dev) for _ in range(P)]
    v_head = [torch.empty((b, s, hkv // P, d), dtype=dt, device=dev) for _ in range(P)]
    o_head = [torch.empty((b, s, hq // P, d), dtype=dt, device=dev) for _ in range(P)]
    o_seq = [torch.empty((b, S, hq, d), dtype=dt, device=dev) for _ in range(P)]
    o_fused = [torch.empty((b, S, hq, d), dtype=dt, device=dev) for _ in range(P)]
    tensor_bytes = b * s * hq * d * esz
    kv_bytes = b * s * hkv * d * esz
    ops = []
    for causal in w["masks"]:
        fl = attn_flops(b, s, hq, d, causal)
        tag = "causal" if causal else "noncausal"
        ops += [
            ("a2a_seq2head_q", "permute", 2 * tensor_bytes, 0, lambda: uly.ulysses_a2a_seq2head(qs, q_head)),
            ("a2a_seq2head_k", "permute", 2 * kv_bytes, 0, lambda: uly.ulysses_a2a_seq2head(ks, k_head)),
            ("a2a_seq2head_v", "permute", 2 * kv_bytes, 0, lambda: uly.ulysses_a2a_seq2head(vs, v_head)),
            (f"attn_{tag}", "attention", 0, fl,
             (lambda c=causal: uly.ulysses_local_attention(q_head, k_head, v_head, c, o_head))),
            ("a2a_head2seq_o", "permute", 2 * tensor_bytes, 0, lambda: uly.ulysses_a2a_head2seq(o_head, o_seq)),
        ]
        if fused_ok:
            ops.append((f"fused_{tag}", "fused", 0, fl,
                        (lambda c=causal: uly.ulysses_dist_attn_fwd(qs, ks, vs, c, fused=True, out_seq=o_fused))))
    return ops, (qs, ks, vs), fused_ok


def time_ops(torch, uly, ops, steps, warmup, dev, stream, clocks=None, world=1):
    """W untimed steps, then exactly K timed steps bracketed by a barrier and a device
    synchronisation on both sides; every launch between CUDA events on its stream."""
    def step(events=None):
        for n, op in enumerate(ops):
            if events is not None:
                events[n][0].record(stream)
            op[4]()
            if events is not None:
                events[n][1].record(stream)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize(dev)
    if uly.ulysses_device_status(clear=True) != 0:
        raise RuntimeError("a kernel's bounded wait gave up during warm-up")
    ev = [[[torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)] for _ in ops]
          for _ in range(steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    if clocks is not None:
        clocks.start()
        time.sleep(0.3)  # let the sampler come up before the timed region
    t_start.record(stream)
    for k in range(steps):
        step(ev[k])
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    clk = clocks.stop() if clocks is not None else None
    if world > 1:
        torch.distributed.barrier()
    if uly.ulysses_device_status(clear=True) != 0:
        raise RuntimeError("a kernel's bounded wait gave up during the timed steps")
    per_op = {}
    for n, op in enumerate(ops):
        per_op.setdefault(op[0], []).extend(ev[k][n][0].elapsed_time(ev[k][n][1]) for k in range(steps))
    return t_start.elapsed_time(t_end), per_op, clk


def summarize(ops, per_op, steps, peaks):
    """Per-kind rates from the per-launch event times: attention and fused launches in
    TFLOP/s against the bf16 peak, exchanges in GB/s against the copy bandwidth."""
    out = {}
    labels = {}
    for op in ops:
        labels.setdefault(op[1], {}).setdefault(op[0], 0)
    for kind in ("attention", "fused"):
        sel = [op for op in ops if op[1] == kind]
        if not sel:
            continue
        ms = sum(sum(per_op[lab]) for lab in labels[kind]) / steps
        tf = sum(op[3] for op in sel) / (ms * 1e-3) / 1e12
        out[kind] = {"tflops": tf, "frac": tf / peaks["bf16_tflops"], "ms_per_step": ms,
                     "per_launch_ms": {lab: statistics.mean(per_op[lab]) for lab in labels[kind]}}
    if "permute" in labels:
        ms = sum(sum(per_op[lab]) for lab in labels["permute"]) / steps
        nbytes = sum(op[2] for op in ops if op[1] == "permute")
        gbs = nbytes / (ms * 1e-3) / 1e9
        out["permute"] = {"gbs": gbs, "frac": gbs / peaks["hbm_gbs"], "bytes_per_step": nbytes,
                          "ms_per_step": ms}
    return out


def run_e2e(torch, uly, w, ins, dev, stream, steps, warmup):
    """The fused forward (unfused where fused does not apply) end to end through the public
    API: every step copies its inputs host -> device from pinned memory and its output
    device -> host, inside the timed region.  The copies run on their own streams with
    NBUF device buffer sets, so the next steps' inputs and the previous steps' outputs move
    while a step computes (as a training loop prefetches its next batches); the host link
    carries both directions at once, and with three sets it always has a copy queued."""
    P, b, s, hq, hkv, d = w["P"], w["b"], w["s"], w["h_q"], w["h_kv"], w["d"]
    S = s // P
    qs, ks, vs = ins
    dt = qs[0].dtype
    esz = qs[0].element_size()
    fused = dt == torch.bfloat16 and S % 128 == 0
    causal = w["masks"][-1]
    host_in = [[t.cpu().pin_memory() for t in src] for src in (qs, ks, vs)]
    host_o = [torch.empty((b, S, hq, d), dtype=dt).pin_memory() for _ in range(P)]
    NBUF = 3
    dev_in = [[[torch.empty_like(t) for t in src] for src in (qs, ks, vs)] for _ in range(NBUF)]
    dev_out = [[torch.empty((b, S, hq, d), dtype=dt, device=dev) for _ in range(P)] for _ in range(NBUF)]
    ws = None if fused else [torch.empty(uly.ulysses_dist_attn_workspace_bytes(P, b, s, hq, hkv, d, dt, False),
                                         dtype=torch.uint8, device=dev) for _ in range(NBUF)]
    h2d = sum(t.numel() * esz for grp in host_in for t in grp)
    d2h = sum(t.numel() * esz for t in host_o)
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(NBUF)]       # inputs of buffer i have landed
    ev_done = [torch.cuda.Event() for _ in range(NBUF)]     # compute on buffer i has finished
    ev_copied = [torch.cuda.Event() for _ in range(NBUF)]   # outputs of buffer i are on the host
    flat_host = [t for grp in host_in for t in grp]

    def upload(k):
        i = k % NBUF
        s_in.wait_event(ev_done[i])  # step k-NBUF has finished reading these inputs
        with torch.cuda.stream(s_in):
            for src, dst in zip(flat_host, [t for grp in dev_in[i] for t in grp]):
                dst.copy_(src, non_blocking=True)
        ev_in[i].record(s_in)

    def compute_and_download(k):
        i = k % NBUF
        stream.wait_event(ev_in[i])
        stream.wait_event(ev_copied[i])  # step k-NBUF's outputs have left these buffers
        q_i, k_i, v_i = dev_in[i]
        uly.ulysses_dist_attn_fwd(q_i, k_i, v_i, causal, fused=fused, out_seq=dev_out[i],
                                  workspace=None if fused else ws[i], stream=stream)
        ev_done[i].record(stream)
        s_out.wait_event(ev_done[i])
        with torch.cuda.stream(s_out):
            for o, ho in zip(dev_out[i], host_o):
                ho.copy_(o, non_blocking=True)
        ev_copied[i].record(s_out)

    def run(n_steps):
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

    run(max(1, warmup))
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    clocks.start()
    time.sleep(0.3)
    e0.record(stream)
    run(steps)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    if uly.ulysses_device_status(clear=True) != 0:
        raise RuntimeError("a kernel's bounded wait gave up during the end-to-end steps")
    fl = attn_flops(b, s, hq, d, causal)
    del dev_in, dev_out, ws
    return dict(e2e_ms=e0.elapsed_time(e1), step_flops=fl, h2d=h2d, d2h=d2h, host_in=host_in, clocks=clk,
                call="ulysses_dist_attn_fwd(fused=%d, causal=%d)" % (int(fused), int(causal)))


def run_gpu(args, rank, world):
    import torch

    import sequence_attention_seq_gb300 as uly
    from sequence_attention_seq_gb300 import build as uly_build

    if rank == 0 or not os.path.exists(uly.library_path()):
        uly_build.build()
    if world > 1:
        torch.distributed.barrier()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    peaks, _ = load_peaks()
    w = WORKLOADS[args.workload]
    ops, ins, fused_ok = forward_ops(uly, torch, w, dev, seed=rank)
    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    total_ms, per_op, clk = time_ops(torch, uly, ops, args.steps, args.warmup, dev, stream, clocks, world)
    res = dict(total_ms=total_ms, clocks=clk, per_op={k: statistics.mean(v) for k, v in per_op.items()},
               per_op_median={k: statistics.median(v) for k, v in per_op.items()},
               step_flops=sum(op[3] for op in ops), n_launches=len(ops) * args.steps,
               summary=summarize(ops, per_op, args.steps, peaks), fused_ok=fused_ok)
    del ops
    e2e = run_e2e(torch, uly, w, ins, dev, stream, args.steps, args.warmup)
    res["e2e"] = e2e
    del ins
    torch.cuda.empty_cache()
    res["extra"] = {}
    if not args.no_extras:
        for name, steps in EXTRAS.get(args.workload, ()):
            wx = WORKLOADS[name]
            ops_x, ins_x, _ = forward_ops(uly, torch, wx, dev, seed=rank)
            ms_x, per_x, clk_x = time_ops(torch, uly, ops_x, steps, max(3, args.warmup), dev, stream,
                                          ClockSampler(dev.index if dev.index is not None else 0), world)
            sm = summarize(ops_x, per_x, steps, peaks)
            sm.update({"workload": wx["name"], "steps": steps, "ms_per_step": ms_x / steps,
                       "per_launch_ms": {k: statistics.mean(v) for k, v in per_x.items()}, "clocks": clk_x})
            if name == "dit":
                sm["permute"]["note"] = ("64 MiB tensors, smaller than the 129 MB L2: the output exchange reads O "
                                         "just written by attention, partly from L2")
            res["extra"][name] = sm
            del ops_x, ins_x
            torch.cuda.empty_cache()
        for name, steps in EXTRAS_BWD.get(args.workload, ()):
            res["extra"][name + "_backward"] = backward_extra(torch, uly, WORKLOADS[name], dev, steps,
                                                              max(3, args.warmup), peaks)
            torch.cuda.empty_cache()
    return res


def backward_extra(torch, uly, w, dev, steps, warmup, peaks):
    """The whole DistributedAttention backward of workload w through its fused path (both
    exchanges in the kernels' tile addressing, as in training after the fused forward), per
    mask: `steps` calls, each between CUDA events on the current stream.  FLOP/s count the
    algorithmic 2.5x forward FLOPs (the five tile products S, dP, dV, dK, dQ)."""
    from sequence_attention_seq_gb300.inputs import global_grad, seq_shards_qkv, shard_seq

    P, b, s, hq, hkv, d = w["P"], w["b"], w["s"], w["h_q"], w["h_kv"], w["d"]
    qs, ks, vs = seq_shards_qkv(P, b, s, hq, hkv, d, torch.bfloat16, seed=0, device=dev)
    dos = shard_seq(global_grad(b, s, hq, d, torch.bfloat16, seed=1, device=dev), P)
    grads = ([torch.empty_like(x) for x in qs], [torch.empty_like(x) for x in ks], [torch.empty_like(x) for x in vs])
    ws = torch.empty(max(1, uly.ulysses_attn_bwd_workspace_bytes(P, b, s, hq, hkv, d, torch.bfloat16, True, True)),
                     dtype=torch.uint8, device=dev)
    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    out = {"workload": w["name"], "call": "ulysses_dist_attn_bwd(fused=1)", "steps": steps,
           "flops": "algorithmic, 2.5x the forward's", "peak": peaks["bf16_tflops"]}
    clocks.start()
    time.sleep(0.3)
    for causal in w["masks"]:
        o, lse = uly.ulysses_dist_attn_fwd_lse(qs, ks, vs, causal, fused=True)

        def call():
            uly.ulysses_dist_attn_bwd(qs, ks, vs, o, dos, lse, causal, grads=grads, workspace=ws, fused=True)

        for _ in range(warmup):
            call()
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for e0, e1 in evs:
            e0.record()
            call()
            e1.record()
        torch.cuda.synchronize()
        ms = statistics.mean(e0.elapsed_time(e1) for e0, e1 in evs)
        tf = 2.5 * attn_flops(b, s, hq, d, causal) / (ms * 1e-3) / 1e12
        out["causal" if causal else "noncausal"] = {"ms": ms, "tflops": tf, "frac": tf / peaks["bf16_tflops"]}
    out["clocks"] = clocks.stop()
    if uly.ulysses_device_status(clear=True) != 0:
        raise RuntimeError("a kernel's bounded wait gave up")
    return out


# -------------------------------------------------------------------- CPU oracle
def oracle_sample(w, ins, budget_s=12.0, seed=0, with_exchange=True):
    """Times the fp64 oracle on a bounded sample of workload w (seq-layout CPU inputs
    `ins`): one exchange at full size (Q, seq->head) and exact attention output rows drawn
    at random, until the time budget is spent.  Returns the rates (attention: algorithmic
    FLOP of the rows computed / their time)."""
    import random

    import oracle

    qs, ks, vs = ins
    P, b, s, hq, d = w["P"], w["b"], w["s"], w["h_q"], w["d"]
    S = s // P
    t_perm, perm_bytes = None, 2 * b * s * hq * d * qs[0].element_size()
    if with_exchange:
        t0 = time.perf_counter()
        oracle.seq2head(qs)
        t_perm = time.perf_counter() - t0
    rng = random.Random(seed)
    flops, rows, t_attn, k = 0, 0, 0.0, 0
    masks = w["masks"]
    while t_attn < budget_s:
        causal = masks[k % len(masks)]
        k += 1
        smp = [(rng.randrange(P), rng.randrange(b), rng.randrange(S), rng.randrange(hq)) for _ in range(8)]
        t1 = time.perf_counter()
        oracle.dist_attn_rows(qs, ks, vs, causal, smp)
        t_attn += time.perf_counter() - t1
        for (j, _, t, _) in smp:
            keys = (j * S + t + 1) if causal else s
            flops += 4 * d * keys
        rows += len(smp)
    return dict(tflops=flops / t_attn / 1e12, rows=rows, t_attn=t_attn,
                perm_gbs=(perm_bytes / t_perm / 1e9) if t_perm else None, t_perm=t_perm)


def cpu_baseline_obj(w, smp):
    ex = (f", plus the Q exchange (seq->head) at full size ({smp['perm_gbs']:.2f} GB/s)"
          if smp["perm_gbs"] else "")
    return {"value": smp["tflops"], "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
            "sample": (f"{smp['rows']} exact fp64 attention output rows of the workload ({w['name']}), random "
                       f"(rank, batch, token, head), in {smp['t_attn']:.1f} s, rate extrapolated from them{ex}; "
                       f"single thread of {os.cpu_count()} host cores")}


KERNEL_REGION_END = b"// ---------------------------------------------------------------- host side"


def _code_only(text):
    """C/CUDA source without its comments and blank lines: edits to comments leave it alone."""
    import re

    text = re.sub(rb"/\*.*?\*/", b"", text, flags=re.S)
    text = re.sub(rb"//[^\n]*", b"", text)
    return b"\n".join(line.rstrip() for line in text.split(b"\n") if line.strip())


def kernel_source_digest():
    """Digest of the forward attention kernel's code: attn_tc.cu up to its host-side section
    (the kernel and its device helpers) and device_common.cuh, comments removed.  The
    traffic figure belongs to one version of that code; launchers, the backward and comment
    edits do not change it."""
    import hashlib

    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "sequence_attention_seq_gb300", "csrc")
    with open(os.path.join(csrc, "attn_tc.cu"), "rb") as f:
        text = f.read()
    if KERNEL_REGION_END not in text:
        return None
    h.update(_code_only(text.split(KERNEL_REGION_END)[0]))
    with open(os.path.join(csrc, "device_common.cuh"), "rb") as f:
        h.update(_code_only(f.read()))
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
    """Exchange bandwidth over bf16 [P][1, s/P, 64, 128] with uniform random bits: the
    kernels alone (20 calls replayed from a CUDA graph) and through the public call with
    its host work (20 calls back to back), each between CUDA events."""
    import torch

    import sequence_attention_seq_gb300 as uly
    from sequence_attention_seq_gb300 import build as uly_build
    from sequence_attention_seq_gb300.inputs import random_bits

    uly_build.build()
    peaks, _ = load_peaks()
    h, d = 64, 128
    rows = []
    shapes = [(s, P) for s in (8192, 32768, 131072, 262144) for P in (2, 4, 8, 16, 32, 64)]
    if args.sweep_only:
        shapes = [tuple(int(x) for x in item.split(",")) for item in args.sweep_only]
    clocks = ClockSampler(0)
    clocks.start()
    time.sleep(0.3)
    for s, P in shapes:
        xs = [random_bits((1, s // P, h, d), torch.bfloat16, seed=j, device="cuda") for j in range(P)]
        hd = [torch.empty((1, s, h // P, d), dtype=torch.bfloat16, device="cuda") for _ in range(P)]
        back = [torch.empty_like(x) for x in xs]
        nbytes = 2 * s * h * d * 2
        res = {}
        for name, fn in (("seq2head", lambda: uly.ulysses_a2a_seq2head(xs, hd)),
                         ("head2seq", lambda: uly.ulysses_a2a_head2seq(hd, back))):
            for _ in range(max(3, args.warmup)):
                fn()
            reps = 20
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            # kernels alone: the reps captured in a CUDA graph and replayed, so the host's
            # per-call argument handling (P pointers per side) is out of the timed region
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=side):
                for _ in range(reps):
                    fn()
            graph.replay()
            torch.cuda.synchronize()
            e0.record()
            graph.replay()
            e1.record()
            torch.cuda.synchronize()
            res[name] = nbytes / (e0.elapsed_time(e1) / reps * 1e-3) / 1e9
            # and through the public call, host work included
            e0.record()
            for _ in range(reps):
                fn()
            e1.record()
            torch.cuda.synchronize()
            res[name + "_eager"] = nbytes / (e0.elapsed_time(e1) / reps * 1e-3) / 1e9
            del graph
        exact = all(torch.equal(a.view(torch.int16), c.view(torch.int16)) for a, c in zip(xs, back))
        row = {"s": s, "P": P, "run_bytes": h // P * d * 2, "seq2head_gbs": res["seq2head"],
               "head2seq_gbs": res["head2seq"], "seq2head_gbs_eager": res["seq2head_eager"],
               "head2seq_gbs_eager": res["head2seq_eager"], "round_trip_bit_exact": exact}
        rows.append(row)
        print(json.dumps(row))
        del xs, hd, back
        torch.cuda.empty_cache()
    clk = clocks.stop()
    allv = [r[k] for r in rows for k in ("seq2head_gbs", "head2seq_gbs")]
    print(json.dumps({"metric": "a2a permute GB/s (read+write), bf16 [P][1,s/P,64,128] sweep", "unit": "GB/s",
                      "min": min(allv), "median": statistics.median(allv), "max": max(allv),
                      "peak": peaks["hbm_gbs"], "median_frac": statistics.median(allv) / peaks["hbm_gbs"],
                      "min_frac": min(allv) / peaks["hbm_gbs"],
                      "all_bit_exact": all(r["round_trip_bit_exact"] for r in rows), "clocks": clk}))


def run_exchange_kernels(args):
    """The per-process halves of the exchange across GPUs (ulysses_a2a_pack before the
    process-group all-to-all, ulysses_a2a_unpack after it) for one rank's bf16 shard
    [1, s/P, 64, 128] (direction 0) or [1, s, 64/P, 128] (direction 1), kernels alone: 20
    calls replayed from a CUDA graph between CUDA events.  Each call reads and writes the
    shard once.  unpack(pack(x, 0), 1) == x and unpack(pack(y, 1), 0) == y are checked."""
    import torch

    import sequence_attention_seq_gb300 as uly
    from sequence_attention_seq_gb300 import build as uly_build
    from sequence_attention_seq_gb300.inputs import random_bits

    uly_build.build()
    peaks, _ = load_peaks()
    h, d, reps = 64, 128, 20
    shapes = [(s, P) for s in (131072, 262144) for P in (2, 4, 8, 16, 32, 64)]
    if args.sweep_only:
        shapes = [tuple(int(x) for x in item.split(",")) for item in args.sweep_only]
    clocks = ClockSampler(0)
    clocks.start()
    time.sleep(0.3)
    rows = []
    for s, P in shapes:
        S = s // P
        seq = random_bits((1, S, h, d), torch.bfloat16, seed=s + P, device="cuda")
        head = random_bits((1, s, h // P, d), torch.bfloat16, seed=s + P + 1, device="cuda")
        send0 = torch.empty((P, 1, S, h // P, d), dtype=torch.bfloat16, device="cuda")
        send1 = torch.empty_like(send0)
        seq_back, head_back = torch.empty_like(seq), torch.empty_like(head)
        nbytes = 2 * seq.numel() * 2
        ops = (("pack_seq2head", lambda: uly.ulysses_a2a_pack(seq, 0, P, out=send0)),
               ("unpack_seq2head", lambda: uly.ulysses_a2a_unpack(send1, 0, out=head_back)),
               ("pack_head2seq", lambda: uly.ulysses_a2a_pack(head, 1, P, out=send1)),
               ("unpack_head2seq", lambda: uly.ulysses_a2a_unpack(send0, 1, out=seq_back)))
        row = {"s": s, "P": P, "shard_mib": seq.numel() * 2 / 2**20, "run_bytes": h // P * d * 2}
        for name, fn in ops:
            for _ in range(max(3, args.warmup)):
                fn()
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=side):
                for _ in range(reps):
                    fn()
            graph.replay()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            graph.replay()
            e1.record()
            torch.cuda.synchronize()
            row[name + "_gbs"] = nbytes / (e0.elapsed_time(e1) / reps * 1e-3) / 1e9
            del graph
        uly.ulysses_a2a_pack(seq, 0, P, out=send0)
        uly.ulysses_a2a_unpack(send0, 1, out=seq_back)
        uly.ulysses_a2a_pack(head, 1, P, out=send1)
        uly.ulysses_a2a_unpack(send1, 0, out=head_back)
        torch.cuda.synchronize()
        row["round_trips_bit_exact"] = bool(torch.equal(seq.view(torch.int16), seq_back.view(torch.int16))
                                            and torch.equal(head.view(torch.int16), head_back.view(torch.int16)))
        rows.append(row)
        print(json.dumps(row))
        del seq, head, send0, send1, seq_back, head_back
        torch.cuda.empty_cache()
    clk = clocks.stop()
    allv = [r[k + "_gbs"] for r in rows for k, _ in (("pack_seq2head", 0), ("unpack_seq2head", 0),
                                                      ("pack_head2seq", 0), ("unpack_head2seq", 0))]
    print(json.dumps({"metric": "per-process exchange kernels GB/s (read+write), one rank's bf16 shard",
                      "unit": "GB/s", "min": min(allv), "median": statistics.median(allv), "max": max(allv),
                      "peak": peaks["hbm_gbs"], "median_frac": statistics.median(allv) / peaks["hbm_gbs"],
                      "min_frac": min(allv) / peaks["hbm_gbs"],
                      "all_bit_exact": all(r["round_trips_bit_exact"] for r in rows), "clocks": clk}))


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
        if P <= 48 and (s // P) % 128 == 0:  # the exchanges folded into the kernels' tile addressing
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
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: a multi-second timed region for the chosen workload)")
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true", help="skip the extra workloads after the main line")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--permute-sweep", action="store_true",
                    help="measure the exchanges over the permute-only sweep instead of the forward")
    ap.add_argument("--exchange-kernels", action="store_true",
                    help="measure the per-process pack and unpack kernels of the exchange across GPUs")
    ap.add_argument("--sweep-only", nargs="*", metavar="S,P",
                    help="with --permute-sweep or --exchange-kernels: only these (sequence length, ranks) shapes")
    ap.add_argument("--backward", action="store_true",
                    help="measure the attention backward (local and distributed) instead of the forward")
    ap.add_argument("--usp", action="store_true",
                    help="measure the two-level Ulysses x Ring forward on its 256K-token workload")
    ap.add_argument("--overlap", action="store_true",
                    help="measure the unfused forward against the overlapped (chunked) forward")
    args = ap.parse_args()
    if args.steps is None:
        args.steps = DEFAULT_STEPS[args.workload]

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
    if args.exchange_kernels:
        if rank == 0:
            run_exchange_kernels(args)
        return
    w = WORKLOADS[args.workload]
    esz = 2 if w["dtype"] == "bf16" else 4
    io_bytes = (2 * w["h_q"] + 2 * w["h_kv"]) * w["b"] * w["s"] * w["d"] * esz
    config = {"workload": w["name"], "P": w["P"], "b": w["b"], "s": w["s"], "h_q": w["h_q"], "h_kv": w["h_kv"],
              "d": w["d"], "causal": list(w["masks"]),
              "l2": (f"inputs larger than L2 (Q+K+V+O = {io_bytes / 2**20:.0f} MiB > 129 MB); no flush"
                     if io_bytes > 129e6 else "inputs smaller than L2: latency-bound exactness case")}

    if args.impl == "reference":
        if rank != 0:
            return
        import torch

        from sequence_attention_seq_gb300.inputs import seq_shards_qkv

        dt = torch.bfloat16 if w["dtype"] == "bf16" else torch.float32
        ins = seq_shards_qkv(w["P"], w["b"], w["s"], w["h_q"], w["h_kv"], w["d"], dt, seed=0)
        steps = []
        for k in range(args.warmup + args.steps):
            smp = oracle_sample(w, ins, budget_s=2.0, seed=k, with_exchange=False)
            if k >= args.warmup:
                steps.append(smp)
        v = sum(x["tflops"] for x in steps) / len(steps)
        rows = sum(x["rows"] for x in steps)
        line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "dtype": "f64",
                "data": "synthetic (seeded N(0,1), CPU generator)", "config": config,
                "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
                                 "sample": (f"per step ~2 s of exact fp64 attention output rows of the workload "
                                            f"({rows} rows over {args.steps} steps), rate extrapolated from them; "
                                            f"single thread of {os.cpu_count()} host cores")},
                "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    import torch

    if world > 1:
        torch.distributed.init_process_group("nccl")
    res = run_gpu(args, rank, world)
    total_ms, e2e_ms = reduce_max_over_ranks([res["total_ms"], res["e2e"]["e2e_ms"]], device="cuda")
    if rank != 0:
        torch.distributed.destroy_process_group()
        return
    peaks, peak_src = load_peaks()
    summ = res["summary"]
    if w["dtype"] == "bf16":
        main_kind = "fused" if "fused" in summ else "attention"
        kernel = ("attn_tc_kernel<%d>, fused launch (both exchanges in its tile addressing)" % w["d"]
                  if main_kind == "fused" else "attn_tc_kernel<%d>, unfused launch (head layout)" % w["d"])
        bound, peak, peak_note = "tensor", peaks["bf16_tflops"], f"{peak_src} (bf16 dense, burst)"
    else:  # fp32 FMA attention: plain ALU peak, 152 SMs x 128 FMA lanes x 2 flop x max SM clock
        main_kind = "attention"
        kernel, bound = "attn_fp32_kernel (attention launches of the step)", "alu"
        peak = 152 * 128 * 2 * peaks.get("sm_max_mhz", 2070.0) * 1e6 / 1e12
        peak_note = "derived: 152 SMs x 128 fp32 FMA/clk x 2 flop x 2070 MHz"
    achieved = summ[main_kind]["tflops"]
    traffic = measured_traffic(args.workload) if main_kind == "fused" else None
    value = job_throughput(res["step_flops"] * args.steps, world, total_ms) / 1e12
    e2e = res["e2e"]
    e2e_value = job_throughput(e2e["step_flops"] * args.steps, world, e2e_ms) / 1e12
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        cpu = cpu_baseline_obj(w, oracle_sample(w, e2e["host_in"], budget_s=12.0))
    extra = {}
    for name, sm in res["extra"].items():
        if name.endswith("_backward"):
            extra[name] = sm
            continue
        ent = {"workload": sm["workload"], "steps": sm["steps"], "ms_per_step": sm["ms_per_step"],
               "per_launch_ms": sm["per_launch_ms"], "clocks": sm["clocks"]}
        for kind in ("fused", "attention", "permute"):
            if kind in sm:
                ent[kind] = sm[kind]
        extra[name] = ent
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w["dtype"], "data": f"synthetic (seeded N(0,1) {w['dtype']}, CUDA generator)",
        "config": config,
        "roofline": {"kernel": kernel, "bound": bound, "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak,
                     "frac_of_sustained": (achieved / peaks["bf16_tflops_sustained"] if bound == "tensor" else None),
                     "peak_source": peak_note, "traffic": traffic,
                     "flops_per_launch": attn_flops(w["b"], w["s"], w["h_q"], w["d"], w["masks"][-1]),
                     "launch_ms": summ[main_kind]["ms_per_step"] / max(1, len(w["masks"])),
                     "launch_ms_median": {lab: res["per_op_median"][lab] for lab in summ[main_kind]["per_launch_ms"]}},
        "attention_unfused": summ.get("attention") if main_kind == "fused" else None,
        "permute": ({"achieved": summ["permute"]["gbs"], "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": summ["permute"]["frac"], "bytes_per_step": summ["permute"]["bytes_per_step"],
                     "bytes": "read+write of all ranks' data"} if "permute" in summ else None),
        "per_launch_ms": res["per_op"],
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": e2e["h2d"],
                "d2h_bytes_per_step": e2e["d2h"], "call": e2e["call"], "ms_per_step": e2e_ms / args.steps,
                "clocks": e2e["clocks"]},
        "gpu_launches": res["n_launches"] * world,
        "clocks": res["clocks"],
        "cpu_baseline": cpu,
        "extra": extra,
    }
    print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
