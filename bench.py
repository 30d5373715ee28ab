"""Throughput benchmark of the So400m/14 SigLIP image encoder on GB300.

One step = one forward pass of the whole path (patch-embedding GEMM, 27
encoder layers, final LayerNorm, MAP pooling) over one batch of synthetic
pixels, through the library's C ABI. The default workload is the 27-layer
encoder + MAP at 378 px, F16 GEMM operands, batch 128 per GPU (the largest
batch of the throughput sweep; the tensor-core target is quoted for batch >= 32);
weights are drawn by the seeded generator and resident in HBM; pixels are
uniform in [-1, 1].

  python bench.py [--gpus N] [--steps K] [--warmup W] [--batch B] [--dtype f16|e4m3] [--unfused-qkv]
                  [--fp8-attention] [--no-configs] [--no-cpu-baseline]
  python bench.py --impl reference ...   # the CPU oracle, timed on the host cores

Prints one JSON line (rank 0). On one GPU the line also carries `configs`: the
batch-1 and batch-32 F16 and the batch-2 and batch-128 E4M3 workloads, each timed
in the same run after the main one, with its own warm-up and clock record. Multi-GPU runs (torchrun, one rank per GPU)
are independent replicas on disjoint images: no collective on the data path,
only a barrier and a max-over-ranks of the elapsed time.
"""
from __future__ import annotations

import argparse
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

METRIC = "images/s for 27-layer So400m/14 @378px, 1 GB300; % of dense tensor-core peak"
T, P, D, H, F, L27, DH = 729, 588, 1152, 16, 4304, 27, 72
IMG = 378  # image side in pixels (27 x 27 patches of 14)


def flops_per_image(layers: int = L27) -> float:
    """Algorithmic FLOPs of one image (head width 72, 729 keys; padding not counted)."""
    patch = 2.0 * T * P * D
    layer = 2.0 * T * D * 3 * D + 4.0 * H * T * T * DH + 2.0 * T * D * D + 2 * 2.0 * T * D * F
    mapf = 2.0 * D * D + 2.0 * T * D * 2 * D + 4.0 * T * D + 2.0 * D * D + 2 * 2.0 * D * F
    return patch + layers * layer + mapf


# DRAM traffic of the dense-GEMM kernel per launch: dram__bytes_read.sum +
# dram__bytes_write.sum from one ncu capture of the four encoder GEMMs of a layer at
# batch 32, F16 (QKV, output projection, MLP up, MLP down; their mean), valid only for
# the kernel sources it was taken on (first 16 hex digits of sha256 of each file).
GEMM_TRAFFIC = {"batch": 32, "bytes_per_launch": 213.7e6,
                "weight_bytes_per_launch": 7.6e6,  # mean F16 weight bytes of the four
                "sources": {"vision_transformer_gb300/csrc/gemm_tc.cu": "54a41cc577e35712",
                            "vision_transformer_gb300/csrc/ptx.cuh": "0d440f4ccbdf05b8"}}


def gemm_traffic(batch: int, dtype: str):
    """Per-launch DRAM traffic of the GEMM kernel for this workload, or None once the kernel
    sources differ from the profiled ones (or for E4M3 operands, never profiled). Other batch
    sizes scale the capture by rows: activations and outputs grow with the batch, the weights
    are read once per launch."""
    import hashlib
    if dtype != "f16":
        return None
    for rel, h in GEMM_TRAFFIC["sources"].items():
        try:
            with open(os.path.join(ROOT, rel), "rb") as f:
                if hashlib.sha256(f.read()).hexdigest()[:16] != h:
                    return None
        except OSError:
            return None
    w = GEMM_TRAFFIC["weight_bytes_per_launch"]
    return w + (GEMM_TRAFFIC["bytes_per_launch"] - w) * batch / GEMM_TRAFFIC["batch"]


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self.thread is not None:
                self.thread.join(timeout=5)

    def summary(self):
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        sm, mx, reasons = [], [], set()
        for line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) != 6:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[2:]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def shard_images(global_batch: int, world: int, rank: int) -> tuple[int, int]:
    """Disjoint image range [start, start+count) of this rank (weak scaling: equal shares)."""
    per = global_batch // world
    return rank * per, per


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def oracle_sample(min_seconds: float, max_images: int = 4, seed: int = 0):
    """Times the CPU oracle as it stands on whole 27-layer images (patch embedding, 27
    layers, final LayerNorm, MAP), one at a time, until min_seconds have passed or
    max_images are done. Returns (seconds, images, threads)."""
    import oracle
    import synth
    m = oracle.OracleModel.from_synth(seed, synth.so400m(L27))
    t, n = 0.0, 0
    while n < max_images and t < min_seconds:
        pix = synth.pixels(2000 + n, 1)
        t0 = time.perf_counter()
        m.encode(pix)
        t += time.perf_counter() - t0
        n += 1
    return t, n, oracle.threads()


def run_reference(args, world, rank):
    """CPU oracle arm: each timed step is one whole image (patch embedding, 27 layers, final
    LayerNorm, MAP) through the oracle as it stands; the warm-up steps run one image through
    one layer each (they only warm the host threads and caches)."""
    if rank != 0:
        return 0
    import oracle
    import synth
    m = oracle.OracleModel.from_synth(0, synth.so400m(L27))
    warm = synth.pixels(1, 1)
    for _ in range(args.warmup):
        m.encode(warm, 1)
    times = []
    for i in range(args.steps):
        pix = synth.pixels(2000 + i, 1)
        t0 = time.perf_counter()
        m.encode(pix)
        times.append(time.perf_counter() - t0)
    per_img = statistics.mean(times)
    value = 1.0 / per_img
    cores = oracle.threads()
    sample = (f"{args.steps} whole images, one per step (patch embedding, 27 layers, final LayerNorm, MAP), FP32 "
              f"oracle with double accumulation, {sum(times):.1f} s; warm-up steps: one image through one layer each")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "images/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_img * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": config(args, world),
            "cpu_baseline": {"value": value, "unit": "images/s", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "images/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# The other configurations of the throughput sweep and the latency cases, timed in the
# same run after the main workload (single-GPU runs): (name, batch, gemm dtype).
EXTRA_CONFIGS = (("b1_f16", 1, "f16"), ("b2_e4m3", 2, "e4m3"), ("b32_f16", 32, "f16"), ("b128_e4m3", 128, "e4m3"))
CONFIG_MIN_S = 0.25  # seconds of warm-up and of timed steps at least, per configuration


def time_config(vt, torch, dev, stream, batch, dtype, steps, warmup, local):
    """Images/s and per-step latency of sv_encode for one (batch, dtype) on device-resident
    pixels, with its own warm-up, CUDA events on the launching stream and clock record."""
    gdt = vt.SV_GEMM_F16 if dtype == "f16" else vt.SV_GEMM_E4M3
    pix = torch.empty(batch, T, P, dtype=torch.float16, device=dev)
    vt.sv_make_pixels(3000, batch, pix)
    out = torch.empty(batch, 1, D, dtype=torch.float16, device=dev)
    # Warm-up of at least `warmup` steps and about 0.25 s, each step waited for, so that the
    # clocks leave the power state of the workload timed before (a one-image step takes
    # about 2 ms); then at least `steps` timed steps covering about 0.25 s as well.
    t0, n_warm, step_s = time.perf_counter(), 0, 0.0
    while n_warm < warmup or time.perf_counter() - t0 < CONFIG_MIN_S:
        t1 = time.perf_counter()
        vt.sv_encode(pix, out, batch, L27, gdt, stream)
        vt.sv_sync(stream)
        step_s = time.perf_counter() - t1
        n_warm += 1
    torch.cuda.synchronize(dev)
    steps = max(steps, int(CONFIG_MIN_S / max(step_s, 1e-4)) + 1)
    warmup = n_warm
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    with ClockSampler(local) as clk:
        ev[0].record(stream)
        for i in range(steps):
            vt.sv_encode(pix, out, batch, L27, gdt, stream)
            ev[i + 1].record(stream)
        torch.cuda.synchronize(dev)
    vt.sv_sync(stream)
    step_ms = [ev[i].elapsed_time(ev[i + 1]) for i in range(steps)]
    ms = ev[0].elapsed_time(ev[-1]) / steps
    return {"batch": batch, "gemm_dtype": dtype, "value": batch / (ms / 1e3), "unit": "images/s",
            "ms_per_step": ms, "latency_ms": {"median": statistics.median(step_ms), "min": min(step_ms),
                                              "max": max(step_ms)},
            "steps": steps, "warmup": warmup, "clocks": clk.summary()}


def config(args, world):
    qk = ", E4M3 attention scores" if getattr(args, "fp8_attention", False) else ""
    return {"workload": f"27-layer So400m/14 @378px + MAP pooling, {args.dtype.upper()} GEMM operands{qk}, "
                        f"batch {args.batch} per GPU",
            "global_batch": args.batch * world, "layers": L27, "tokens": T, "width": D,
            "gemm_dtype": args.dtype, "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            "qkv": "three GEMMs" if getattr(args, "unfused_qkv", False) else "one fused GEMM",
            "attention_scores": "E4M3 Q, K" if getattr(args, "fp8_attention", False) else "F16 Q, K",
            "l2": "no flush: every step streams 0.85 GB of F16 weights and several GB of activations, "
                  "far above the 129 MB L2"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--batch", type=int, default=128, help="images per GPU per step")
    ap.add_argument("--dtype", choices=("f16", "e4m3"), default="f16")
    ap.add_argument("--unfused-qkv", action="store_true", help="Q, K, V as three GEMMs (comparison only)")
    ap.add_argument("--fp8-attention", action="store_true", help="scores on E4M3 Q and K (FP8 attention products)")
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="skip the other configurations (configs key)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="minimum CPU time of the oracle sample")
    args = ap.parse_args()
    world, rank, local = dist_env()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" else "gloo"
        if backend == "nccl":
            import torch
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    if args.impl == "reference":
        rc = run_reference(args, world, rank)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return rc

    import torch
    import vision_transformer_gb300 as vt

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    B = args.batch
    gdt = vt.SV_GEMM_F16 if args.dtype == "f16" else vt.SV_GEMM_E4M3
    vt.sv_init_weights(0)
    start, count = shard_images(B * world, world, rank)
    pix = torch.empty(count, T, P, dtype=torch.float16, device=dev)
    vt.sv_make_pixels(1000 + rank, count, pix)  # disjoint images per rank
    out = torch.empty(count, 1, D, dtype=torch.float16, device=dev)
    stream = torch.cuda.current_stream(dev)

    flags = (vt.SV_ENCODE_UNFUSED_QKV if args.unfused_qkv else 0) | \
        (vt.SV_ENCODE_FP8_ATTENTION if args.fp8_attention else 0)

    def step():
        vt.sv_encode_ex(pix, out, count, L27, gdt, flags, stream)

    for _ in range(args.warmup):
        step()
    vt.sv_sync(stream)

    # ---- timed region: device-resident inputs, CUDA events on the launching stream
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize(dev)
    vt.sv_launch_count()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]  # one after each step
    with ClockSampler(local) as clk:
        ev[0].record(stream)
        for i in range(args.steps):
            step()
            ev[i + 1].record(stream)
        torch.cuda.synchronize(dev)
    vt.sv_sync(stream)
    launches = vt.sv_launch_count()
    elapsed_ms = max_over_ranks(ev[0].elapsed_time(ev[-1]), world)
    step_ms = [ev[i].elapsed_time(ev[i + 1]) for i in range(args.steps)]  # this rank's batch latencies
    ms_per_step = elapsed_ms / args.steps
    value = B * world / (ms_per_step / 1e3)

    # ---- per-kernel times: the same steps again, every library launch bracketed by
    # CUDA events on its stream (the brackets add small gaps, so this second timed region
    # gives the kernel durations and shares, not the step time above)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize(dev)
    vt.sv_profile_enable(True)
    for k in range(vt.KIND_OTHER + 1):
        vt.sv_profile_read(k)  # drop earlier records
    for _ in range(args.steps):
        step()
    vt.sv_sync(stream)
    vt.sv_profile_enable(False)
    prof = {vt.KIND_NAMES[k]: vt.sv_profile_read(k) for k in range(vt.KIND_OTHER + 1)}

    # ---- end to end: whole images [B, 378, 378, 3] f16 from pinned host memory, packed into
    # patch rows on the GPU (sv_pack_patches), encoded, embedding back to pinned host memory,
    # every step (the synthetic images are the synthetic pixel values laid out as images)
    host_img = pix.reshape(count, IMG, IMG, 3).cpu().pin_memory()
    img = torch.empty(host_img.shape, dtype=torch.float16, device=dev)
    host_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()

    def e2e_step():
        img.copy_(host_img, non_blocking=True)
        vt.sv_pack_patches(img, pix, count, IMG, 3, 14, stream)
        step()
        host_out.copy_(out, non_blocking=True)

    for _ in range(args.warmup):
        e2e_step()
    torch.cuda.synchronize(dev)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    e2, e3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2.record(stream)
    for _ in range(args.steps):
        e2e_step()
    e3.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e2.elapsed_time(e3), world) / args.steps
    e2e_value = B * world / (e2e_ms / 1e3)

    peaks = measured_peaks()
    g = prof["gemm_tc"]
    gemm_tflops = g["flops"] / (g["ms"] / 1e3) / 1e12 if g["ms"] > 0 else 0.0
    # E4M3 GEMMs are rated against the E4M3 peak: the measured F16/bf16 peak times the
    # nominal dense E4M3 / F16 tensor-core ratio (4.5 / 2.25 PFLOP/s)
    ratio = 2.0 if args.dtype == "e4m3" else 1.0
    scaled = " x 2 (nominal dense E4M3 / F16 ratio)" if ratio != 1.0 else ""
    peak = peaks["bf16_tflops_sustained"] * ratio
    burst = peaks["bf16_tflops"] * ratio
    step_flops = flops_per_image() * B
    whole_tflops = step_flops / (ms_per_step / 1e3) / 1e12
    kernels = {k: {"ms_per_step": v["ms"] / args.steps, "launches_per_step": v["launches"] / args.steps,
                   "share": v["ms"] / max(1e-9, sum(x["ms"] for x in prof.values()))}
               for k, v in prof.items() if v["launches"]}

    line = {"metric": METRIC, "value": value, "unit": "images/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": args.dtype, "data": "synthetic", "config": config(args, world),
            "fraction_of_peak": {"value": whole_tflops / burst, "achieved_tflops": whole_tflops,
                                 "peak_tflops": burst, "basis": "algorithmic FLOPs of the whole "
                                 f"step ({flops_per_image() / 1e9:.2f} GFLOP/image) / step time, of "
                                 f"{peaks['source']} dense bf16 burst peak{scaled}"},
            "roofline": {"kernel": "gemm_tc (all dense-GEMM launches of the step)", "bound": "tensor",
                         "achieved": gemm_tflops, "peak": peak, "unit": "TFLOP/s",
                         "frac": gemm_tflops / peak if peak else None, "traffic": gemm_traffic(B, args.dtype),
                         "traffic_unit": "bytes per launch (ncu DRAM read + write, mean of the 4 encoder GEMMs, "
                                         "captured at batch 32 and scaled by rows to this batch)",
                         "peak_kind": f"{peaks['source']} bf16 sustained{scaled}"},
            "latency_ms": {"mean": ms_per_step, "median": statistics.median(step_ms), "min": min(step_ms),
                           "max": max(step_ms), "basis": "per-step CUDA events on rank 0's launching "
                                                         "stream; mean = the timed region's max over ranks / steps"},
            "kernels": kernels,
            "e2e": {"value": e2e_value, "unit": "images/s", "h2d_bytes_per_step": host_img.numel() * 2,
                    "d2h_bytes_per_step": host_out.numel() * 2,
                    "includes": "pinned H2D of whole 378x378x3 f16 images, patch packing on the GPU, "
                                "the encoder, D2H of the embeddings"},
            "gpu_launches": launches,
            "clocks": clk.summary()}

    if rank == 0 and world == 1 and not args.no_configs:
        # the other configurations, same weights, same box, same run (one by one after the main workload)
        peaks_all = measured_peaks()
        extra = {}
        for name, b, dt in EXTRA_CONFIGS:
            if b == B and dt == args.dtype:
                continue
            r = time_config(vt, torch, dev, stream, b, dt, args.steps, args.warmup, local)
            burst_c = peaks_all["bf16_tflops"] * (2.0 if dt == "e4m3" else 1.0)
            r["fraction_of_peak"] = flops_per_image() * b / (r["ms_per_step"] / 1e3) / 1e12 / burst_c
            r["peak_kind"] = f"{peaks_all['source']} dense bf16 burst" + (" x 2 (E4M3)" if dt == "e4m3" else "")
            extra[name] = r
        line["configs"] = extra
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        t, n, cores = oracle_sample(args.cpu_seconds)
        line["cpu_baseline"] = {"value": n / t, "unit": "images/s", "cores": cores, "kind": "oracle",
                                "sample": f"{n} whole images (patch embedding, 27 layers, final LayerNorm, MAP), "
                                          f"one at a time, {t:.1f} s"}
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    vt.sv_shutdown()
    return 0


if __name__ == "__main__":
    sys.exit(main())
