"""Benchmark: U-Net denoise megapixels/s at 1080p fp16 on GB300.

Workload: full OIDN-shaped U-Net denoise of a 1920x1080 image (colour,
albedo, normal; HDR, log transfer, inputScale 1), fp16 storage with fp32
accumulation, whole image as one 1920x1088 tile.  Inputs are seeded
synthetic images (see synth/).  One step = one oidnx_filter_execute (input
pass, 16 conv kernels, output pass).  L2 is flushed (a 256 MiB write)
before every timed step; the flush is outside the per-step CUDA events.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

With N > 1 (torchrun, one rank per GPU) every rank denoises its own frame:
replicas, weak scaling, no collective on the data path.
`--impl reference` times the CPU oracle (the pages' computation restated in
numpy float64) on a bounded crop of the same workload.
"""

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "U-Net denoise megapixels/s at 1080p fp16 on 1 GB300; conv TFLOP/s vs FP16 peak"
# --precision fp32: the same workload with fp32 storage (3xTF32 products)
METRIC_FP32 = "U-Net denoise megapixels/s at 1080p fp32 (3xTF32) on 1 GB300; conv TFLOP/s vs TF32 peak / 3"
WIDTH, HEIGHT = 1920, 1080
WORKLOAD = "OIDN-shaped U-Net denoise, 1920x1080 HDR colour+albedo+normal (9 ch), fp16, single tile"
MAX_TILE, OVERLAP = 0, -1   # single tile (0 = whole image), default overlap
# --workload 4k-tiled: the 3840x2160 tiled configuration (a parity-test
# workload, timed on request; not the headline)
WORKLOADS = {
    "1080p": (1920, 1080, 0, -1, METRIC, WORKLOAD),
    "4k-tiled": (3840, 2160, 1024, 96,
                 "U-Net denoise megapixels/s at 3840x2160 (maxTileSize 1024, overlap 96) fp16 on 1 GB300",
                 "OIDN-shaped U-Net denoise, 3840x2160 HDR colour+albedo+normal (9 ch), fp16, "
                 "maxTileSize 1024, overlap 96 (15 tiles)"),
}
CPU_CROP = 768          # oracle sample: a 768x768 crop denoised as one tile
CPU_BASELINE_RUNS = 3   # cpu_baseline of our arm: three runs of that crop (~10 s)
REF_BUDGET_S = 120.0    # reference arm: the whole run's oracle time
FLUSH_BYTES = 256 << 20


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def wait_first_sample(self, timeout=10.0):
        t0 = time.time()
        while self.proc and not self.lines and time.time() - t0 < timeout:
            time.sleep(0.05)

    def summary(self):
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax = float(parts[1])
            except ValueError:
                continue
            for name, flag in zip(names, parts[4:8]):
                if flag.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": smax, "reasons": [], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


def _cpu_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return max(n)
    except Exception:
        pass
    return os.cpu_count()


def metric_name(fp32):
    """The metric of the selected workload and precision."""
    if not fp32:
        return METRIC
    return METRIC_FP32 if METRIC == WORKLOADS["1080p"][4] else METRIC.replace("fp16", "fp32 (3xTF32)")


def cpu_oracle_sample(steps=1, precision="fp16", crop=CPU_CROP):
    """Oracle denoise of a crop x crop crop of the bench inputs, `steps` times."""
    import synth
    from oracle import unet
    imgs = [im[:crop, :crop].copy() for im in synth.denoise_inputs(WIDTH, HEIGHT, 3, hdr=True)]
    weights = synth.unet_weights(9)
    times = []
    for _ in range(steps):
        t0 = time.perf_counter()
        unet.denoise(imgs, weights, hdr=True, input_scale=1.0, precision=precision)
        times.append(time.perf_counter() - t0)
    px = crop * crop
    return {"value": px / 1e6 / float(np.mean(times)), "unit": "MP/s", "cores": _cpu_threads(),
            "kind": "oracle",
            "sample": f"oracle (numpy float64) denoise of one {crop}x{crop} crop of the "
                      f"1920x1080 inputs as one tile, {precision} storage; {steps} run(s)",
            "seconds": float(np.mean(times)), "crop": crop}


def reference_crop(steps, precision, budget_s=REF_BUDGET_S):
    """Crop side (multiple of 16, 64 .. CPU_CROP) for which `steps` oracle
    runs take about budget_s on this host, from the rate of one 128 x 128 run."""
    probe = cpu_oracle_sample(1, precision, crop=128)
    px = probe["value"] * 1e6 * budget_s / max(steps, 1)
    return int(max(64, min(CPU_CROP, int(np.sqrt(px)) // 16 * 16)))


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def aggregate(ms_per_rank, px_per_rank):
    """Whole-job throughput: all ranks' pixels over the slowest rank's time."""
    slowest = max(ms_per_rank)
    return sum(px_per_rank) / 1e6 / (slowest / 1e3), slowest


def max_over_ranks(values):
    """Element-wise max of per-rank timings (identity on a single process)."""
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return list(values)
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor(list(values), dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def run_reference(args):
    world, rank, _ = _dist()
    if rank != 0:
        return
    # warm-up: the oracle has no warm-up state; the calibration run that
    # sizes each step's crop (K steps in about REF_BUDGET_S) stands in for it
    crop = reference_crop(args.steps, args.precision)
    cpu = cpu_oracle_sample(args.steps, args.precision, crop=crop)
    line = {
        "impl": "reference", "metric": metric_name(args.precision == "fp32"),
        "value": cpu["value"], "unit": "MP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": cpu["seconds"] * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "sample": f"{crop}x{crop} crop per step",
                   "l2": "n/a (CPU)"},
        "cpu_baseline": {k: cpu[k] for k in ("value", "unit", "cores", "kind", "sample")},
        "e2e": {"value": cpu["value"], "unit": "MP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args):
    import torch
    world, rank, local = _dist()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    dev = torch.cuda.current_device()

    import conv2d_implicit_gemm_gb300 as ox
    import synth

    imgs = synth.denoise_inputs(WIDTH, HEIGHT, 3, hdr=True)
    weights = synth.unet_weights(9)
    fp32 = args.precision == "fp32"
    f = ox.oidnx_filter_create(ox.write_weight_blob(weights),
                               ox.PRECISION_FP32 if fp32 else ox.PRECISION_FP16)
    d_imgs = [torch.from_numpy(im).cuda() for im in imgs]
    d_out = torch.zeros((HEIGHT, WIDTH, 4), dtype=torch.float32, device="cuda")
    for i, t in enumerate(d_imgs):
        ox.oidnx_filter_set_image(f, i, t.data_ptr(), 0)
    ox.oidnx_filter_set_image(f, ox.IMAGE_OUTPUT, d_out.data_ptr(), 0)
    ox.oidnx_filter_set_int(f, "width", WIDTH)
    ox.oidnx_filter_set_int(f, "height", HEIGHT)
    ox.oidnx_filter_set_int(f, "maxTileSize", MAX_TILE)
    ox.oidnx_filter_set_int(f, "overlap", OVERLAP)
    ox.oidnx_filter_set_int(f, "hdr", 1)
    ox.oidnx_filter_set_int(f, "transfer", ox.TRANSFER_LOG)
    ox.oidnx_filter_set_float(f, "inputScale", 1.0)
    ox.oidnx_filter_commit(f)
    tiles = ox.oidnx_filter_get_int(f, "tiles")
    stream = torch.cuda.current_stream()
    sptr = stream.cuda_stream
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")

    for _ in range(max(args.warmup, 3)):
        flush.fill_(1)
        ox.oidnx_filter_execute(f, sptr)
    ox.oidnx_filter_sync_status(f)

    layer_ms, layer_flop, layer_bytes, layer_mma = {}, {}, {}, {}
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(dev) as clocks:
        clocks.wait_first_sample()
        # Timed region: K denoise steps, L2 flushed before each, CUDA events on
        # the launching stream around each step (the flush is outside them).
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        for k in range(args.steps):
            flush.fill_(k & 0xFF)
            starts[k].record(stream)
            ox.oidnx_filter_execute(f, sptr)
            ends[k].record(stream)
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        ox.oidnx_filter_sync_status(f)
        step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
        # Profiled steps: the same execution with a CUDA event after every
        # kernel (recorded inside the graph on the launching stream).  Events
        # between kernels stop the next kernel's prologue from overlapping the
        # previous one, so these per-kernel times are slightly pessimistic.
        ox.oidnx_filter_set_int(f, "profile", 1)
        ox.oidnx_filter_execute(f, sptr)
        ox.oidnx_get_profile(f)
        prof_steps = []
        for k in range(args.steps):
            flush.fill_(k & 0xFF)
            ox.oidnx_filter_execute(f, sptr)
            prof = ox.oidnx_get_profile(f)   # waits for this step's events
            prof_steps.append(prof["totalMs"])
            launches_per_step = sum(l["launches"] for l in prof["layers"])
            for l in prof["layers"]:
                layer_ms[l["id"]] = layer_ms.get(l["id"], 0.0) + l["ms"]
                layer_flop[l["id"]] = l["flop"]
                layer_bytes[l["id"]] = l["bytes"]
                layer_mma[l["id"]] = l.get("mmaFlop", 0)
        ox.oidnx_filter_set_int(f, "profile", 0)
        torch.cuda.synchronize()
    ox.oidnx_filter_sync_status(f)
    mean_ms = float(np.mean(step_ms))

    # end to end through the host-buffer call: H2D inputs, denoise, D2H output
    pinned = [torch.from_numpy(im).pin_memory() for im in imgs]
    host_out = torch.empty((HEIGHT, WIDTH, 4), dtype=torch.float32).pin_memory()
    host_ptr = [p.data_ptr() for p in pinned]
    for _ in range(3):
        ox._check(ox._lib.oidnx_filter_execute_host(f, *host_ptr, host_out.data_ptr(), sptr))
    e2e_ms = []
    for k in range(args.steps):
        flush.fill_(k & 0xFF)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        ox._check(ox._lib.oidnx_filter_execute_host(f, *host_ptr, host_out.data_ptr(), sptr))
        e2e_ms.append((time.perf_counter() - t0) * 1e3)
    # a stream of K frames through the enqueue-only host call: every step
    # still uploads its inputs and downloads its output, but one frame's
    # copies overlap another frame's denoise (two device staging sets); the
    # wall clock runs from the first enqueue to the last output in host
    # memory (device working set per step > L2, no flush in between)
    outs = [torch.empty((HEIGHT, WIDTH, 4), dtype=torch.float32).pin_memory() for _ in range(2)]
    for k in range(3):
        ox._check(ox._lib.oidnx_filter_execute_host_async(f, *host_ptr, outs[k & 1].data_ptr(), sptr))
    ox._check(ox._lib.oidnx_filter_wait_host(f))
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for k in range(args.steps):
        ox._check(ox._lib.oidnx_filter_execute_host_async(f, *host_ptr, outs[k & 1].data_ptr(), sptr))
    ox._check(ox._lib.oidnx_filter_wait_host(f))
    stream_ms = (time.perf_counter() - t0) * 1e3 / args.steps
    ox.oidnx_filter_release(f)

    px = WIDTH * HEIGHT
    mean_ms, e2e_mean, stream_ms = max_over_ranks([mean_ms, float(np.mean(e2e_ms)), stream_ms])
    value, _ = aggregate([mean_ms] * world, [px] * world)
    e2e_value, _ = aggregate([stream_ms] * world, [px] * world)
    e2e_sync_value, _ = aggregate([e2e_mean] * world, [px] * world)

    steps = args.steps
    avg = {k: v / steps for k, v in layer_ms.items()}
    conv_ids = [k for k in avg if k not in ("input-pack", "output")]
    conv_ms = sum(avg[k] for k in conv_ids)
    conv_flop = sum(layer_flop[k] for k in conv_ids)
    peaks = _peaks()
    tensor_peak = peaks["bf16_tflops_sustained"]   # fp16 dense rate = bf16 dense rate
    if fp32:
        # tf32 dense rate = bf16 rate x nominal 1.1 / 2.25; three tf32 MMAs per product
        tensor_peak *= (1.1 / 2.25) / 3.0
    top = max(conv_ids, key=lambda k: avg[k])
    top_flop, top_bytes = layer_flop[top], layer_bytes[top]
    ridge = tensor_peak * 1e12 / (peaks["hbm_gbs"] * 1e9)
    if top_flop / max(top_bytes, 1) >= ridge:
        roof = {"kernel": top, "bound": "tensor", "achieved": top_flop / (avg[top] * 1e-3) / 1e12,
                "peak": tensor_peak, "unit": "TFLOP/s"}
    else:
        roof = {"kernel": top, "bound": "hbm", "achieved": top_bytes / (avg[top] * 1e-3) / 1e9,
                "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    if roof["bound"] == "tensor" and layer_mma.get(top):
        # achieved counts the logical conv FLOPs; the tensor cores execute
        # mmaFlop (padded tiles; 4 of 9 taps on a sub-pixel decoder's
        # upsampled channels; three tf32 products per fp32 product, against
        # a peak that is already divided by three)
        executed = layer_mma[top] / (3.0 if fp32 else 1.0) / (avg[top] * 1e-3) / 1e12
        roof["executed"] = executed
        roof["executed_frac"] = executed / tensor_peak
    roof["traffic"] = None if fp32 or (WIDTH, HEIGHT, MAX_TILE) != (1920, 1080, 0) else TRAFFIC.get(top)
    roof["traffic_unit"] = "bytes per launch (ncu dram read + write)"
    roof["peak_source"] = peaks["source"] + (
        (" sustained bf16 x tf32/bf16 nominal ratio (1.1/2.25) / 3 (three tf32 MMAs per product)"
         if fp32 else " sustained bf16 (dense fp16 = bf16 rate)")
        if roof["bound"] == "tensor" else " HBM copy")
    roof["launch_ms"] = avg[top] / tiles
    layers = {k: {"ms": round(avg[k], 5),
                  "tflops": round(layer_flop[k] / (avg[k] * 1e-3) / 1e12, 2) if layer_flop[k] else None,
                  "gbs": round(layer_bytes[k] / (avg[k] * 1e-3) / 1e9, 1)} for k in avg}

    if rank == 0:
        cpu = cpu_oracle_sample(CPU_BASELINE_RUNS, args.precision) if world == 1 else None
        line = {
            "metric": metric_name(fp32), "value": value, "unit": "MP/s", "n_gpus": world,
            "steps": steps, "warmup": max(args.warmup, 3), "ms_per_step": mean_ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32" if fp32 else "f16", "data": "synthetic",
            "config": {"workload": WORKLOAD.replace("fp16", "fp32") if fp32 else WORKLOAD,
                       "width": WIDTH, "height": HEIGHT, "tiles": tiles,
                       "precision": ("fp32 storage, 3xTF32 products, fp32 accumulate" if fp32
                                     else "fp16 storage, fp32 accumulate"), "hdr": True,
                       "transfer": "log", "l2": "flushed (256 MiB write) before every step",
                       "parallelism": f"replicas x{world}"},
            "conv_tflops": conv_flop / (conv_ms * 1e-3) / 1e12,
            "conv_frac_of_peak": conv_flop / (conv_ms * 1e-3) / 1e12 / tensor_peak,
            "roofline": roof,
            "layers": layers,
            "e2e_sync": {"value": e2e_sync_value, "unit": "MP/s", "ms_per_step": e2e_mean,
                         "mode": "one blocking host-buffer call per step (L2 flushed before each)"},
            "e2e": {"value": e2e_value, "unit": "MP/s", "h2d_bytes_per_step": 3 * px * 16,
                    "d2h_bytes_per_step": px * 16, "ms_per_step": stream_ms,
                    "mode": "frame stream through the enqueue-only host-buffer call (uploads and "
                            "downloads overlap other frames' denoise), K steps then one wait"},
            "gpu_launches": steps * launches_per_step,
            "profiled_ms_per_step": float(np.mean(prof_steps)),
            "layers_note": "per-kernel times from the profiled steps (event after every kernel)",
            "clocks": clocks.summary(),
        }
        if cpu:
            line["cpu_baseline"] = {k: cpu[k] for k in ("value", "unit", "cores", "kind", "sample")}
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) of the
# two largest layers, from one ncu capture of this workload with the current
# kernels (its summary is kept under profiles/); to be emptied whenever these
# kernels change after that capture (traffic is then reported null).
TRAFFIC = {"dec_conv1a": 134.141440e6 + 207.531776e6,
           "dec_conv1b": 267.567872e6 + 97.209600e6}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--precision", choices=["fp16", "fp32"], default="fp16",
                    help="activation storage (fp32: 3xTF32 products); the headline is fp16")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="1080p",
                    help="1080p single tile (the headline) or the 3840x2160 tiled configuration")
    args = ap.parse_args()
    global WIDTH, HEIGHT, MAX_TILE, OVERLAP, METRIC, WORKLOAD
    WIDTH, HEIGHT, MAX_TILE, OVERLAP, METRIC, WORKLOAD = WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
