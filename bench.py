"""Frame-step benchmark: aggregate frames/s and step latency of the full PersonaPlex
shape at B = 1 (250-frame forced prompt, then decode frames), against the HBM roofline.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

One JSON line on rank 0.  With torchrun (N > 1) every rank runs the same
workload on its own GPU (independent replicas: slots never interact), and the
value is all ranks' frames over the slowest rank's time.

--impl reference times the CPU oracle (the plain fp64 definition) on this
machine's host cores over a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

WORKLOAD = synth.WORKLOADS["full_b1"]
PROMPT = 250
METRIC = "aggregate frames/s (B=1 full PersonaPlex frame step)"
UNIT = "frames/s"


def algorithmic_bytes(s, lens):
    """Bytes one step must move: every streamed weight once, the embedding rows
    read, and per slot (lens = window length of each slot in the step) the
    keys/values of its window plus this frame's writes."""
    wb = 2 if s.weight_dtype == "bf16" else 4
    kvb = 2 if s.kv_dtype == "bf16" else 4
    d, F, V, C, S, L = s.d, s.ffn, s.text_vocab, s.card, s.dep_steps, s.n_layers
    dd, dF, dL = s.dep_d, s.dep_ffn, s.dep_layers
    weights = L * (4 * d * d + 3 * F * d) * wb + (V + S * dd) * d * wb
    weights += S * (dL * (4 * dd * dd + 3 * dd * dF) + C * dd) * wb
    per_slot_rows = 17 * d * wb + S * dd * wb
    kv_pos = L * 2 * d * kvb
    return weights + sum(per_slot_rows + ln * kv_pos + kv_pos for ln in lens)


def read_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def read_bf16_peak():
    """Dense bf16 tensor throughput (TFLOP/s) for a kernel timed alone: the measured burst figure."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        if "bf16_tflops" in j:
            return float(j["bf16_tflops"]), "measured bf16_tflops (burst)"
    return 1900.0, "fallback bf16 burst"


def kernel_source_digest():
    """Digest of the step kernel's device sources (its template, internal layout
    and the instantiation units), which decide its DRAM traffic."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "full_duplex_speech_frame_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name in ("mfs_kernels.cuh", "mfs_internal.h") or (name.startswith("mfs_k_") and name.endswith(".cu")):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode())
                h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload):
    """DRAM bytes per launch from the committed ncu summary of this kernel and
    workload, or None if the kernel source changed since it was taken."""
    p = os.path.join(ROOT, "profiles", f"step_kernel_{workload}.txt")
    if not os.path.exists(p):
        return None
    vals = {}
    for line in open(p):
        if ":" in line:
            k, v = line.split(":", 1)
            vals[k.strip()] = v.strip()
    if (vals.get("kernel_source_digest") or "?").split()[0] != kernel_source_digest():
        return None
    try:
        return float(vals["dram_bytes_per_launch"].split()[0])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup(n_gpus):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("gloo")
    return rank, world


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world):
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def cpu_oracle_sample(frames=6, prompt=8, warmup=0):
    """Time the CPU oracle on a bounded sample of the workload: a short forced
    prompt and `warmup` decode frames (untimed), then `frames` decode frames (timed)."""
    import oracle
    s = WORKLOAD.shape
    w = synth.make_weights(s, WORKLOAD.weight_seed)
    orc = oracle.Oracle(s, w)
    orc.prefill(0, synth.forced_frames(s, WORKLOAD.input_seed, synth.STREAM_PROMPT, prompt, 1)[:, 0])
    u = synth.user_frames(s, WORKLOAD.input_seed, warmup + frames, 1)
    for p in range(warmup):
        orc.step([0], u[p])
    u = u[warmup:]
    t0 = time.perf_counter()
    for p in range(frames):
        orc.step([0], u[p])
    dt = time.perf_counter() - t0
    cores = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    return {"value": frames / dt, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{frames} decode frames of the full shape at B=1 after a {prompt}-frame prompt "
                      f"(fp64 oracle, OpenMP over output rows); {dt:.1f} s"}


def run_reference(args, rank, world):
    if rank != 0:
        return
    # the GPU arm's workload: the same 250-frame prompt and warm-up count; the timed
    # frames are capped so that the run stays within a few minutes
    frames = max(1, min(args.steps, 30))
    cb = cpu_oracle_sample(frames=frames, prompt=PROMPT, warmup=args.warmup)
    line = {"impl": "reference", "metric": METRIC, "value": cb["value"], "unit": UNIT, "n_gpus": args.gpus,
            "steps": frames, "warmup": args.warmup, "ms_per_step": 1000.0 / cb["value"],
            "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "full_b1: full PersonaPlex shape (4096-d/32-layer temporal, 1024-d/6-layer "
                                   "16-substep depformer), bf16 weights N(0,0.02) seed 0, B=1, ring prompt 250 "
                                   "forced frames, then decode frames with user rows supplied, greedy",
                       "batch": 1, "prompt_frames": PROMPT,
                       "positions": [PROMPT + args.warmup, PROMPT + args.warmup + frames]},
            "cpu_baseline": cb,
            "e2e": {"value": cb["value"], "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_gpu(args, rank, world):
    import torch
    from full_duplex_speech_frame_gb300 import mfs

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    # a stream of our own: the library enqueues on it and the events below time it
    side = torch.cuda.Stream()
    torch.cuda.set_stream(side)
    s = WORKLOAD.shape.replace(max_slots=32)  # slot 0 runs the B = 1 workload, all 32 the batched ones
    n = WORKLOAD.batch
    need = 3 * args.warmup + 4 * args.steps
    if PROMPT + need > s.max_pos:
        raise SystemExit("too many steps for the position range")
    w = synth.make_weights(s, WORKLOAD.weight_seed)
    ctx = mfs.context_with_weights(s, w)
    del w
    prompt = synth.forced_frames(s, WORKLOAD.input_seed, synth.STREAM_PROMPT, PROMPT, n)
    mfs.mfs_prefill(ctx, list(range(n)), prompt.transpose(1, 0, 2))
    frames = synth.user_frames(s, WORKLOAD.input_seed, need, n)
    slots = list(range(n))
    d_codes = torch.from_numpy(frames).cuda()
    d_text = torch.empty(n, dtype=torch.int32, device="cuda")
    d_out = torch.empty(n, 16, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()

    # warm-up
    for p in range(args.warmup):
        mfs.mfs_step_device(ctx, slots, d_codes[p], d_text, d_out)
    mfs.mfs_sync(ctx)
    base = args.warmup

    # device-resident timed region (the value)
    lens = [[min(PROMPT + base + k + 1, s.window)] * n for k in range(args.steps)]
    mfs.mfs_set_timing(ctx, 1)
    mfs.mfs_kernel_time(ctx)
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        e0.record(stream)
        for k in range(args.steps):
            mfs.mfs_step_device(ctx, slots, d_codes[base + k], d_text, d_out)
        e1.record(stream)
        mfs.mfs_sync(ctx)
        torch.cuda.synchronize()
    barrier(world)
    ms = e0.elapsed_time(e1)
    kms, ksteps = mfs.mfs_kernel_time(ctx)
    mfs.mfs_set_timing(ctx, 0)
    launches = mfs.mfs_launches_per_step(ctx) * args.steps
    ms_max = max_over_ranks(ms, world)
    value = n * args.steps * world / (ms_max / 1000.0)

    # variant: trailing depformer substeps whose outputs are supplied are skipped
    # (user streams 9..16 here: substeps 8..15); every output is unchanged
    mfs.mfs_set_skip_settled(ctx, True)
    vb = base + args.steps
    for p in range(args.warmup):
        mfs.mfs_step_device(ctx, slots, d_codes[vb + p], d_text, d_out)
    vb += args.warmup
    mfs.mfs_sync(ctx)
    mfs.mfs_set_timing(ctx, 1)
    mfs.mfs_kernel_time(ctx)
    barrier(world)
    torch.cuda.synchronize()
    e0.record(stream)
    for k in range(args.steps):
        mfs.mfs_step_device(ctx, slots, d_codes[vb + k], d_text, d_out)
    e1.record(stream)
    mfs.mfs_sync(ctx)
    torch.cuda.synchronize()
    barrier(world)
    ms_v = max_over_ranks(e0.elapsed_time(e1), world)
    vkms, vks = mfs.mfs_kernel_time(ctx)
    mfs.mfs_set_timing(ctx, 0)
    mfs.mfs_set_skip_settled(ctx, False)

    # variant: sampling heads (text 0.7 / top-25, audio 0.8 / top-250), host-buffer calls
    sb = vb + args.steps
    mfs.mfs_set_sampling(ctx, 0, 0.7, 25, 0.8, 250)
    unif = ((synth.uniform_int(WORKLOAD.input_seed, 97, (args.warmup + args.steps) * 17, 0, 1 << 24)
             .reshape(-1, 1, 17)) + 0.5) / float(1 << 24)
    for p in range(args.warmup):
        mfs.mfs_step_sampled(ctx, slots, frames[sb + p], unif[p])
    sb += args.warmup
    mfs.mfs_set_timing(ctx, 1)
    mfs.mfs_kernel_time(ctx)
    for k in range(args.steps):
        mfs.mfs_step_sampled(ctx, slots, frames[sb + k], unif[args.warmup + k])
    skms, sks = mfs.mfs_kernel_time(ctx)
    mfs.mfs_set_timing(ctx, 0)
    mfs.mfs_set_sampling(ctx, 0, 0.0, 0, 0.0, 0)

    # end to end through the public host-buffer call
    base2 = sb + args.steps
    pinned = torch.from_numpy(frames[base2:base2 + args.steps]).pin_memory().numpy()
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for k in range(args.steps):
        text, codes = mfs.mfs_step(ctx, slots, pinned[k])
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(time.perf_counter() - t0, world)
    barrier(world)

    batched = run_batched(args, mfs, ctx, s, stream, world) if not args.no_batched else {}

    # the Mimi split RVQ encoder on 152 x 16 frames (D 256, 2048 codewords per codebook)
    Tq, Dq, Cq = 2432, 256, 2048
    zq = torch.from_numpy(synth.normal_f32(WORKLOAD.input_seed, 501, 2 * Tq * Dq).reshape(2, Tq, Dq)).cuda()
    cbq = torch.from_numpy(synth.normal_f32(WORKLOAD.input_seed, 503, 8 * Cq * Dq).reshape(8, Cq, Dq)).cuda()
    cq = torch.empty(Tq, 8, dtype=torch.int32, device="cuda")
    for _ in range(args.warmup):
        mfs.mfs_rvq_encode(zq[0], zq[1], cbq, cq)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(args.steps):
        mfs.mfs_rvq_encode(zq[0], zq[1], cbq, cq)
    e1.record(stream)
    torch.cuda.synchronize()
    rvq_ms = e0.elapsed_time(e1) / args.steps

    if rank != 0:
        return
    hbm, peak_kind = read_peaks()
    bf16_peak, bf16_kind = read_bf16_peak()
    bytes_step = sum(algorithmic_bytes(s, l) for l in lens) / args.steps
    kernel_ms = kms / max(ksteps, 1)
    achieved = bytes_step / (kernel_ms / 1000.0) / 1e9
    traffic = recorded_traffic("full_b1")
    desc_bytes = 16 + 64 * 4 * 2 + 64 * 17 * 4
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "full_b1: full PersonaPlex shape (4096-d/32-layer temporal, 1024-d/6-layer "
                               "16-substep depformer), bf16 weights N(0,0.02) seed 0, B=1, ring prompt 250 "
                               "forced frames, then decode frames with user rows supplied, greedy",
                   "batch": n, "prompt_frames": PROMPT, "positions": [PROMPT + base, PROMPT + base + args.steps],
                   "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2: every step streams 16.1 GB of weights"},
        "latency_ms_per_step": ms_max / args.steps,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": achieved / hbm, "traffic": traffic, "peak_kind": f"{peak_kind} hbm_gbs",
                     "kernel": "step_kernel (one persistent launch per step)",
                     "kernel_ms": kernel_ms, "algorithmic_bytes_per_launch": bytes_step},
        "e2e": {"value": n * args.steps * world / e2e_s, "unit": UNIT, "h2d_bytes_per_step": desc_bytes,
                "d2h_bytes_per_step": n * 4 + n * 16 * 4 + 8},
        "gpu_launches": launches,
        "clocks": clk.summary(),
        "variants": {
            "skip_settled_substeps": {
                "what": "mfs_set_skip_settled: depformer substeps 8..15 skipped because user streams 9..16 are "
                        "supplied; outputs identical, weights streamed 1.25 GB less",
                "value": n * args.steps * world / (ms_v / 1000.0), "unit": UNIT, "ms_per_step": ms_v / args.steps,
                "kernel_ms": vkms / max(vks, 1),
            },
            "rvq_encode": {
                "what": "mfs_rvq_encode, Mimi split RVQ argmin quantizer: 2432 frames, D 256, 8 codebooks of 2048; "
                        "r.c on the tensor cores (bf16 high/low parts) in CTA pairs of 32 frames, fp32 re-rank of the candidates near the best score",
                "kernel_ms": rvq_ms, "value": Tq / (rvq_ms / 1000.0), "unit": "frames/s",
                "roofline": {"bound": "tensor", "unit": "TFLOP/s",
                             "achieved": 2.0 * Tq * 8 * Cq * Dq / (rvq_ms / 1000.0) / 1e12,
                             "peak": bf16_peak, "frac": 2.0 * Tq * 8 * Cq * Dq / (rvq_ms / 1000.0) / 1e12 / bf16_peak,
                             "peak_kind": bf16_kind,
                             "flops": "2 T 8 Cb D: one product r.c per distance (the four bf16 part products and "
                                      "the re-rank are not counted)"},
            },
            **batched,
            "sampling_heads": {
                "what": "mfs_step_sampled with text temperature 0.7 / top-25 and audio 0.8 / top-250 "
                        "(uniforms supplied per step); device time of the step kernel",
                "kernel_ms": skms / max(sks, 1), "value": 1000.0 / (skms / max(sks, 1)), "unit": UNIT,
            },
        },
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_oracle_sample(frames=40)
    print(json.dumps(line), flush=True)


def run_batched(args, mfs, ctx, s, stream, world):
    """The batched workloads on slots 0..B-1 of the same context, device-resident
    (inputs in HBM, no host copies in the timed region).  Every step streams the
    16.1 GB of weights once for all slots (the tensor-core pass) plus each slot's
    key/value window, more than L2 holds, so no flush is needed.
      B = 8:  per-slot windows uniform in [0, 3000] (synthetic ring states)
      B = 16: 250-frame prompts for every slot (timed as well: the prompt path),
              then decode frames from position 250
      B = 32: every ring full (3000 keys, positions past 3000: every step wraps)
    Returns {name: line}, each with aggregate frames/s, ms per step, algorithmic
    bytes per step and the fraction of the measured HBM bandwidth."""
    import torch
    hbm, peak_kind = read_peaks()
    shared = synth.slot_state(s, WORKLOAD.input_seed, 300, 0)
    out = {}
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def time_steps(B, lens_of_step, seed):
        slots = list(range(B))
        frames = torch.from_numpy(synth.user_frames(s, seed, args.warmup + args.steps, B)).cuda()
        d_text = torch.empty(B, dtype=torch.int32, device="cuda")
        d_out = torch.empty(B, 16, dtype=torch.int32, device="cuda")
        for p in range(args.warmup):
            mfs.mfs_step_device(ctx, slots, frames[p], d_text, d_out)
        mfs.mfs_sync(ctx)
        lens = [lens_of_step(args.warmup + k) for k in range(args.steps)]
        barrier(world)
        torch.cuda.synchronize()
        e0.record(stream)
        for k in range(args.steps):
            mfs.mfs_step_device(ctx, slots, frames[args.warmup + k], d_text, d_out)
        e1.record(stream)
        mfs.mfs_sync(ctx)
        torch.cuda.synchronize()
        barrier(world)
        ms = max_over_ranks(e0.elapsed_time(e1), world) / args.steps
        byts = sum(algorithmic_bytes(s, l) for l in lens) / args.steps
        return {"value": B * world / (ms / 1000.0), "unit": UNIT, "ms_per_step": ms, "batch": B,
                "algorithmic_bytes_per_step": byts,
                "roofline": {"bound": "hbm", "achieved": byts / (ms / 1000.0) / 1e9, "peak": hbm, "unit": "GB/s",
                             "frac": byts / (ms / 1000.0) / 1e9 / hbm, "peak_kind": f"{peak_kind} hbm_gbs"},
                "launches_per_step": mfs.mfs_launches_per_step(ctx)}

    # B = 8: windows uniform in [0, 3000]
    lens8 = synth.prefill_lengths(WORKLOAD.input_seed, 8, 0, 3000)
    for i in range(8):
        shared[4:8] = np.frombuffer(np.int32(lens8[i]).tobytes(), np.uint8)
        mfs.mfs_import_slot(ctx, i, shared)
    r = time_steps(8, lambda k: [min(int(lens8[i]) + k + 1, s.window) for i in range(8)], 11)
    r["what"] = ("B=8 decode, per-slot windows uniform in [0, 3000] (synthetic ring states); temporal stack and text "
                 "head on the tensor-core pass, depformer on the CUDA-core pass (two launches per step)")
    out["batch_8"] = r

    # B = 16: 250-frame prompts (timed), then decode
    for i in range(16):
        mfs.mfs_reset_slot(ctx, i)
    prompt = torch.from_numpy(synth.forced_frames(s, WORKLOAD.input_seed, synth.STREAM_PROMPT, PROMPT, 16)
                              .transpose(1, 0, 2).copy())
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    mfs.mfs_prefill(ctx, list(range(16)), prompt.numpy())
    torch.cuda.synchronize()
    pre_s = time.perf_counter() - t0
    r = time_steps(16, lambda k: [min(PROMPT + k + 1, s.window)] * 16, 12)
    r["what"] = ("B=16 decode after 250-frame prompts; the whole step on the tensor-core pass (one launch per step)")
    r["prompt"] = {"frames": 16 * PROMPT, "seconds": pre_s, "value": 16 * PROMPT / pre_s, "unit": "prompt frames/s",
                   "what": "mfs_prefill of 16 slots x 250 frames: 125 launches of 32 rows (two frames of every "
                           "slot) on the tensor-core pass (host call, includes the token upload)"}
    out["batch_16"] = r

    # B = 32: full rings, every step wraps
    pos32 = 3000 + synth.uniform_int(WORKLOAD.input_seed, synth.STREAM_LENGTHS + 1, 32, 0, 2000)
    for i in range(32):
        shared[4:8] = np.frombuffer(np.int32(pos32[i]).tobytes(), np.uint8)
        mfs.mfs_import_slot(ctx, i, shared)
    r = time_steps(32, lambda k: [s.window] * 32, 13)
    r["what"] = ("B=32 decode, every ring full (3000 keys, every step wraps); the whole step on the tensor-core pass "
                 "(one launch per step)")
    out["batch_32"] = r
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gpu", choices=["gpu", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-batched", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    rank, world = dist_setup(args.gpus)
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_gpu(args, rank, world)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
