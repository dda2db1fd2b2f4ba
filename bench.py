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
    """nvidia-smi clocks and throttle reasons, sampled every 20 ms from just
    before the timed region to the end of the profiled and host-buffer steps
    that follow it."""

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
                 "--format=csv,noheader,nounits", "-lms", "20"],
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


CPU_SINGLE_CROP = 256   # single-core sample of the 1080p workload


def _cpu_configs_once(precision, crop2):
    """Oracle timings of the small configurations on this process's BLAS
    threads: the 128 x 128 fp32 denoise, the single 512 x 512 64 -> 64 conv
    (fp16-rounded inputs and weights, float64 sums), and a crop2 x crop2
    crop of the 1080p workload."""
    import synth
    from oracle import layers, unet
    from oracle.numerics import round_storage
    out = {}
    imgs = synth.denoise_inputs(128, 128, 3, hdr=True)
    weights = synth.unet_weights(9)
    t0 = time.perf_counter()
    unet.denoise(imgs, weights, hdr=True, input_scale=1.0, precision="fp32")
    t = time.perf_counter() - t0
    out["config0_128x128_fp32"] = {"value": 128 * 128 / 1e6 / t, "unit": "MP/s", "seconds": t}
    x = round_storage(synth.uniform_activations(512, 512, 64, seed=11), "fp16").astype(np.float64)
    wt, b = synth.he_uniform_conv(64, 64, seed=1001, bias_scale=0.1)
    wq = round_storage(wt, "fp16").astype(np.float64)
    t0 = time.perf_counter()
    layers.conv3x3(x, wq, b.astype(np.float64), relu=True)
    t = time.perf_counter() - t0
    out["config1_single_conv_512x512_64to64"] = {
        "value": 2.0 * 9 * 64 * 64 * 512 * 512 / t / 1e9, "unit": "GFLOP/s", "seconds": t}
    c = cpu_oracle_sample(1, precision, crop=crop2)
    out["config2_1080p_crop"] = {"value": c["value"], "unit": "MP/s", "seconds": c["seconds"],
                                 "sample": f"{crop2}x{crop2} crop of the 1920x1080 inputs, one tile"}
    return out


def cpu_baseline_configs(precision):
    """The oracle on all host threads (this process) and on one core (a
    child process whose BLAS and OpenMP pools are limited to one thread)."""
    res = {"all_cores": _cpu_configs_once(precision, CPU_CROP // 2),
           "all_cores_threads": _cpu_threads()}
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    try:
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-single",
                            "--precision", precision], env=env, capture_output=True, text=True,
                           timeout=600)
        res["single_core"] = json.loads(r.stdout.strip().splitlines()[-1])
    except (subprocess.TimeoutExpired, ValueError, IndexError) as e:
        res["single_core"] = {"error": f"{type(e).__name__}"}
    res["kind"] = "oracle"
    res["note"] = "numpy float64 oracle; all_cores: BLAS threads of this process"
    return res


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


def _tensor_peak(peaks, fp32):
    """Dense tensor peak (TFLOP/s) for kernels timed inside a sub-millisecond
    step: the measured burst bf16 rate (dense fp16 = bf16 rate); for fp32
    storage the tf32 rate (bf16 x nominal 1.1 / 2.25) divided by the three
    tf32 MMAs each fp32 product takes."""
    peak = peaks["bf16_tflops"]
    return peak * (1.1 / 2.25) / 3.0 if fp32 else peak


def layer_rooflines(avg, flop, nbytes, mma, peaks, fp32):
    """Per kernel: ms, TFLOP/s, GB/s, the bound (tensor when the layer's
    arithmetic intensity, logical FLOPs over algorithmic bytes, is at or
    above the ridge, else HBM) and the fraction of that bound's peak; tensor
    layers also give the executed fraction (what the tensor cores run)."""
    tpeak = _tensor_peak(peaks, fp32)
    ridge = tpeak * 1e12 / (peaks["hbm_gbs"] * 1e9)
    out = {}
    for k, ms in avg.items():
        sec = ms * 1e-3
        e = {"ms": round(ms, 5), "tflops": None, "gbs": round(nbytes[k] / sec / 1e9, 1)}
        if flop[k]:
            e["tflops"] = round(flop[k] / sec / 1e12, 2)
        if flop[k] and flop[k] / max(nbytes[k], 1) >= ridge:
            e["bound"] = "tensor"
            e["frac"] = round(flop[k] / sec / 1e12 / tpeak, 4)
            if mma.get(k):
                e["executed_frac"] = round(mma[k] / (3.0 if fp32 else 1.0) / sec / 1e12 / tpeak, 4)
        else:
            e["bound"] = "hbm"
            e["frac"] = round(nbytes[k] / sec / 1e9 / peaks["hbm_gbs"], 4)
        out[k] = e
    return out


def _kernel_sources_sha():
    import hashlib
    h = hashlib.sha256()
    for name in TRAFFIC_SOURCES:
        with open(os.path.join(ROOT, "conv2d_implicit_gemm_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def _setup_denoise(ox, torch, width, height, sources, hdr, nan_fraction, fp32, max_tile, overlap):
    """A committed filter over device images of one denoise workload."""
    import synth
    imgs = synth.denoise_inputs(width, height, sources, hdr=hdr, nan_fraction=nan_fraction)
    weights = synth.unet_weights(3 * sources)
    f = ox.oidnx_filter_create(ox.write_weight_blob(weights),
                               ox.PRECISION_FP32 if fp32 else ox.PRECISION_FP16)
    d_imgs = [torch.from_numpy(im).cuda() for im in imgs]
    d_out = torch.zeros((height, width, 4), dtype=torch.float32, device="cuda")
    for i, t in enumerate(d_imgs):
        ox.oidnx_filter_set_image(f, i, t.data_ptr(), 0)
    ox.oidnx_filter_set_image(f, ox.IMAGE_OUTPUT, d_out.data_ptr(), 0)
    ox.oidnx_filter_set_int(f, "width", width)
    ox.oidnx_filter_set_int(f, "height", height)
    ox.oidnx_filter_set_int(f, "maxTileSize", max_tile)
    ox.oidnx_filter_set_int(f, "overlap", overlap)
    ox.oidnx_filter_set_int(f, "hdr", int(hdr))
    ox.oidnx_filter_set_int(f, "transfer", ox.TRANSFER_LOG)
    ox.oidnx_filter_set_float(f, "inputScale", 1.0)
    ox.oidnx_filter_commit(f)
    return f, imgs, (d_imgs, d_out)


def _profile_steps(ox, f, sptr, flush, steps):
    """`steps` executions with an event after every kernel: per-kernel mean
    ms, FLOPs, bytes and executed tensor FLOPs, launches per step."""
    ms, flop, nbytes, mma, totals = {}, {}, {}, {}, []
    launches = 0
    ox.oidnx_filter_set_int(f, "profile", 1)
    ox.oidnx_filter_execute(f, sptr)
    ox.oidnx_get_profile(f)
    for k in range(steps):
        flush.fill_(k & 0xFF)
        ox.oidnx_filter_execute(f, sptr)
        prof = ox.oidnx_get_profile(f)   # waits for this step's events
        totals.append(prof["totalMs"])
        launches = sum(l["launches"] for l in prof["layers"])
        for l in prof["layers"]:
            ms[l["id"]] = ms.get(l["id"], 0.0) + l["ms"] / steps
            flop[l["id"]] = l["flop"]
            nbytes[l["id"]] = l["bytes"]
            mma[l["id"]] = l.get("mmaFlop", 0)
    ox.oidnx_filter_set_int(f, "profile", 0)
    return ms, flop, nbytes, mma, float(np.mean(totals)), launches


def _timed_steps(ox, f, torch, stream, flush, steps, warmup):
    sptr = stream.cuda_stream
    for _ in range(max(warmup, 3)):
        flush.fill_(1)
        ox.oidnx_filter_execute(f, sptr)
    ox.oidnx_filter_sync_status(f)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    torch.cuda.synchronize()
    for k in range(steps):
        flush.fill_(k & 0xFF)
        starts[k].record(stream)
        ox.oidnx_filter_execute(f, sptr)
        ends[k].record(stream)
    torch.cuda.synchronize()
    ox.oidnx_filter_sync_status(f)
    return float(np.mean([s.elapsed_time(e) for s, e in zip(starts, ends)]))


def _conv_summary(avg, flop, mma, peaks, fp32):
    conv_ids = [k for k in avg if k not in ("input-pack", "output")]
    conv_ms = sum(avg[k] for k in conv_ids)
    conv_flop = sum(flop[k] for k in conv_ids)
    conv_mma = sum(mma.get(k, 0) for k in conv_ids)
    tpeak = _tensor_peak(peaks, fp32)
    t = conv_flop / (conv_ms * 1e-3) / 1e12
    ex = conv_mma / (3.0 if fp32 else 1.0) / (conv_ms * 1e-3) / 1e12
    return {"conv_tflops": t, "conv_frac_of_peak": t / tpeak,
            "conv_executed_frac_of_peak": ex / tpeak, "conv_ms": conv_ms}


def measure_denoise_config(ox, torch, stream, flush, peaks, name, width, height, sources, hdr,
                           nan_fraction, fp32, max_tile, overlap, steps=10, warmup=3):
    """MP/s and conv TFLOP/s of one more denoise configuration (a few ms of
    GPU work): timed steps, then profiled steps for the conv share."""
    f, _, keep = _setup_denoise(ox, torch, width, height, sources, hdr, nan_fraction, fp32,
                                max_tile, overlap)
    try:
        tiles = ox.oidnx_filter_get_int(f, "tiles")
        ms = _timed_steps(ox, f, torch, stream, flush, steps, warmup)
        avg, flop, nbytes, mma, prof_ms, launches = _profile_steps(ox, f, stream.cuda_stream, flush,
                                                                   max(3, steps // 2))
    finally:
        ox.oidnx_filter_release(f)
    del keep
    conv = _conv_summary(avg, flop, mma, peaks, fp32)
    return {"config": name, "value": width * height / 1e6 / (ms * 1e-3), "unit": "MP/s",
            "ms_per_step": ms, "steps": steps, "tiles": tiles,
            "conv_tflops": round(conv["conv_tflops"], 2),
            "conv_frac_of_peak": round(conv["conv_frac_of_peak"], 4),
            "conv_executed_frac_of_peak": round(conv["conv_executed_frac_of_peak"], 4),
            "peak": "burst bf16" + (" x 1.1/2.25 / 3 (3xTF32)" if fp32 else ""),
            "profiled_ms_per_step": round(prof_ms, 4), "gpu_launches_per_step": launches,
            "flop_basis": "logical conv FLOPs over the tiles' input areas (overlap recompute "
                          "included)"}


def measure_single_conv(ox, torch, stream, flush, peaks, steps=20, warmup=3):
    """The single-layer workload: 3x3 conv + bias + ReLU, 512 x 512, 64 -> 64,
    fp16 activations (U[-1, 1]), He-uniform weights, fp32 accumulate; CUDA
    events around each launch, L2 flushed before each."""
    import synth
    w = h = 512
    cin = cout = 64
    x = synth.uniform_activations(h, w, cin, seed=11).astype(np.float16)
    wt, b = synth.he_uniform_conv(cout, cin, seed=1001, bias_scale=0.1)
    # library activation layout [H][C/8][W][8]
    xi = np.ascontiguousarray(x.reshape(h, w, cin // 8, 8).transpose(0, 2, 1, 3))
    d_in = torch.from_numpy(xi.view(np.uint8).reshape(-1).copy()).cuda()
    d_out = torch.empty(h * w * cout * 2, dtype=torch.uint8, device="cuda")
    c = ox.oidnx_conv_create(wt, b, ox.PRECISION_FP16)
    sptr = stream.cuda_stream
    try:
        for _ in range(max(warmup, 3)):
            ox.oidnx_conv_execute(c, d_in.data_ptr(), d_out.data_ptr(), w, h, 1, sptr)
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        torch.cuda.synchronize()
        for k in range(steps):
            flush.fill_(k & 0xFF)
            starts[k].record(stream)
            ox.oidnx_conv_execute(c, d_in.data_ptr(), d_out.data_ptr(), w, h, 1, sptr)
            ends[k].record(stream)
        torch.cuda.synchronize()
        ms = float(np.mean([s.elapsed_time(e) for s, e in zip(starts, ends)]))
    finally:
        ox.oidnx_conv_release(c)
    flop = 2.0 * 9 * cin * cout * w * h
    nbytes = 2.0 * w * h * (cin + cout) + 9 * cin * cout * 2 + cout * 4
    tflops = flop / (ms * 1e-3) / 1e12
    gbs = nbytes / (ms * 1e-3) / 1e9
    tpeak = _tensor_peak(peaks, False)
    ridge = tpeak * 1e12 / (peaks["hbm_gbs"] * 1e9)
    return {"config": "single 3x3 conv + bias + ReLU, 512x512, 64->64, fp16, fp32 accumulate",
            "ms": ms, "steps": steps, "tflops": tflops, "frac_of_tensor_peak": tflops / tpeak,
            "gbs": gbs, "frac_of_hbm": gbs / peaks["hbm_gbs"],
            "arithmetic_intensity": flop / nbytes, "ridge": ridge,
            "bound": "tensor" if flop / nbytes >= ridge else "hbm",
            "l2": "flushed (256 MiB write) before every launch"}


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

    fp32 = args.precision == "fp32"
    f, imgs, keep = _setup_denoise(ox, torch, WIDTH, HEIGHT, 3, True, 0.0, fp32, MAX_TILE, OVERLAP)
    tiles = ox.oidnx_filter_get_int(f, "tiles")
    stream = torch.cuda.current_stream()
    sptr = stream.cuda_stream
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    peaks = _peaks()

    for _ in range(max(args.warmup, 3)):
        flush.fill_(1)
        ox.oidnx_filter_execute(f, sptr)
    ox.oidnx_filter_sync_status(f)

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
        avg, layer_flop, layer_bytes, layer_mma, prof_ms, launches_per_step = _profile_steps(
            ox, f, sptr, flush, args.steps)
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
    del keep

    px = WIDTH * HEIGHT
    mean_ms, e2e_mean, stream_ms = max_over_ranks([mean_ms, float(np.mean(e2e_ms)), stream_ms])
    value, _ = aggregate([mean_ms] * world, [px] * world)
    e2e_value, _ = aggregate([stream_ms] * world, [px] * world)
    e2e_sync_value, _ = aggregate([e2e_mean] * world, [px] * world)

    steps = args.steps
    conv = _conv_summary(avg, layer_flop, layer_mma, peaks, fp32)
    tensor_peak = _tensor_peak(peaks, fp32)
    layers = layer_rooflines(avg, layer_flop, layer_bytes, layer_mma, peaks, fp32)
    conv_ids = [k for k in avg if k not in ("input-pack", "output")]
    top = max(conv_ids, key=lambda k: avg[k])
    L = layers[top]
    if L["bound"] == "tensor":
        roof = {"kernel": top, "bound": "tensor", "achieved": layer_flop[top] / (avg[top] * 1e-3) / 1e12,
                "peak": tensor_peak, "unit": "TFLOP/s"}
    else:
        roof = {"kernel": top, "bound": "hbm", "achieved": layer_bytes[top] / (avg[top] * 1e-3) / 1e9,
                "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["frac_basis"] = ("logical conv FLOPs (2 x 9 x Cin x Cout per pixel) over the kernel's "
                          "event-timed duration" if roof["bound"] == "tensor" else
                          "algorithmic bytes (inputs read once, output written once)")
    if roof["bound"] == "tensor" and layer_mma.get(top):
        # the tensor cores execute mmaFlop: padded tiles; 4 of the 9 taps on a
        # sub-pixel decoder's upsampled channels; three tf32 products per fp32
        # product (against a peak already divided by three)
        executed = layer_mma[top] / (3.0 if fp32 else 1.0) / (avg[top] * 1e-3) / 1e12
        roof["executed"] = executed
        roof["executed_frac"] = executed / tensor_peak
    sha = _kernel_sources_sha()
    current = (not fp32 and (WIDTH, HEIGHT, MAX_TILE) == (1920, 1080, 0)
               and sha == TRAFFIC.get("sources_sha"))
    roof["traffic"] = TRAFFIC.get(top) if current else None
    roof["traffic_unit"] = "bytes per launch (ncu dram read + write)"
    roof["traffic_note"] = ("from the ncu capture of the current kernel sources" if current else
                            "null: no ncu capture of the current kernel sources for this workload")
    roof["peak_source"] = peaks["source"] + (
        (" burst bf16 x tf32/bf16 nominal ratio (1.1/2.25) / 3 (three tf32 MMAs per product)"
         if fp32 else " burst bf16 (dense fp16 = bf16 rate; the kernel runs inside a 0.5 ms step)")
        if roof["bound"] == "tensor" else " HBM copy")
    roof["launch_ms"] = avg[top] / tiles
    # the input pass against the pages' bytes: 16 B per source image read,
    # 8 B per 4-channel fp16 block (16 B fp32) written
    pack = layers.get("input-pack")
    if pack:
        tile_px = layer_bytes["input-pack"] / (16.0 * 3 + 9 * (4 if fp32 else 2))
        pages_bytes = tile_px * (16.0 * 3 + 3 * (16 if fp32 else 8))
        pack["bytes_pages"] = pages_bytes
        pack["frac_pages_bytes"] = round(pages_bytes / (avg["input-pack"] * 1e-3) / 1e9 / peaks["hbm_gbs"], 4)

    if rank == 0:
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
            "conv_tflops": conv["conv_tflops"],
            "conv_frac_of_peak": conv["conv_frac_of_peak"],
            "conv_executed_frac_of_peak": conv["conv_executed_frac_of_peak"],
            "conv_peak": "measured burst bf16" + (" x 1.1/2.25 / 3" if fp32 else ""),
            "roofline": roof,
            "layers": layers,
            "pools": "fused into the epilogues of enc_conv1..enc_conv4 (2x2 max of the ReLU "
                     "outputs before the store): no pass of their own; their HBM bytes are the "
                     "pooled outputs those layers write, inside each layer's figures",
            "e2e_sync": {"value": e2e_sync_value, "unit": "MP/s", "ms_per_step": e2e_mean,
                         "mode": "one blocking host-buffer call per step (L2 flushed before each)"},
            "e2e": {"value": e2e_value, "unit": "MP/s", "h2d_bytes_per_step": 3 * px * 16,
                    "d2h_bytes_per_step": px * 16, "ms_per_step": stream_ms,
                    "mode": "frame stream through the enqueue-only host-buffer call (uploads and "
                            "downloads overlap other frames' denoise), K steps then one wait"},
            "gpu_launches": steps * launches_per_step,
            "profiled_ms_per_step": prof_ms,
            "layers_note": "per-kernel times from the profiled steps (event after every kernel); "
                           "frac against the measured burst peaks (kernels timed inside a "
                           "sub-millisecond step)",
            "clocks": clocks.summary(),
        }
        if world == 1 and not args.no_extra and (WIDTH, HEIGHT) == (1920, 1080) and not fp32:
            line["configs"] = {
                "config0_128x128_fp32": measure_denoise_config(
                    ox, torch, stream, flush, peaks, "128x128 HDR colour+albedo+normal, fp32, one tile",
                    128, 128, 3, True, 0.0, True, 0, -1, steps=20),
                "config1_single_conv_512x512_64to64": measure_single_conv(ox, torch, stream, flush, peaks),
                "config3_3840x2160_tiled_fp16": measure_denoise_config(
                    ox, torch, stream, flush, peaks,
                    "3840x2160 HDR colour+albedo+normal, fp16, maxTileSize 1024, overlap 96",
                    3840, 2160, 3, True, 0.0, False, 1024, 96),
                "config4_3840x2160_fp32_ldr_colour": measure_denoise_config(
                    ox, torch, stream, flush, peaks,
                    "3840x2160 LDR colour only (5% NaN/Inf), fp32 (3xTF32), one tile",
                    3840, 2160, 1, False, 0.05, True, 0, -1),
            }
        if world == 1:
            cpu = cpu_oracle_sample(CPU_BASELINE_RUNS, args.precision)
            line["cpu_baseline"] = {k: cpu[k] for k in ("value", "unit", "cores", "kind", "sample")}
            if not args.no_extra:
                line["cpu_baseline_configs"] = cpu_baseline_configs(args.precision)
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) of the
# two largest kernels, from one ncu capture of this workload (the per-kernel
# table kept under profiles/), with sources_sha the hash of TRAFFIC_SOURCES
# at that capture.
TRAFFIC = {"sources_sha": "38c7d8e33e899790", "dec_conv1a": 380.959744e6,
           "dec_conv1b+dec_conv0+output": 325.794048e6}
# the kernel sources those figures were taken with: traffic is reported
# null once their hash differs from sources_sha
TRAFFIC_SOURCES = ("conv_tc.cu", "conv_tail.cu", "passes.cuh", "ptx.cuh", "internal.h")


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
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the other configurations and the per-config CPU timings")
    ap.add_argument("--cpu-single", action="store_true", help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.cpu_single:   # child of cpu_baseline_configs: one BLAS thread
        out = _cpu_configs_once(args.precision, CPU_SINGLE_CROP)
        out["threads"] = 1
        print(json.dumps(out), flush=True)
        return
    global WIDTH, HEIGHT, MAX_TILE, OVERLAP, METRIC, WORKLOAD
    WIDTH, HEIGHT, MAX_TILE, OVERLAP, METRIC, WORKLOAD = WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
