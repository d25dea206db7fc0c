"""Benchmark of the NCC hot path on GB300.

One step = the whole path on a batch of 4096x4096 uint8 images with one 16x16
uint8 template: for each image, build both int64 summed-area tables, then the
numerator and coefficients for all 4081 x 4081 valid shifts, in one ncc_match
call (the correlation kernel overlaps the table build's tail).  The batch is
the workload image and seeded circular shifts of it, sized so a step lasts
about 40 ms of device time (the clock sampler then sees the load).  The same
steps are also timed as separate ncc_sat_build + ncc_correlate calls with
events between the kernels, for the per-kernel times and rooflines, and the
table build alone is timed on the 8192x8192 image.  Prints one JSON line: the
throughput, per-kernel timings, the roofline of the dominant kernel, the CPU
oracle baseline, the end-to-end figure and clocks.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Under torchrun each rank matches its own copy of the image (independent
problems, no data-path collective): weak scaling, value = all ranks'
coefficients / the slowest rank's time.  `--impl reference` times the CPU
oracle on the host cores instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from normalized_cross_correlation_gb300 import inputs  # noqa: E402

METRIC = "NCC coefficients/s (4096², 16×16 tmpl); SAT build GB/s vs HBM peak"
UNIT = "coefficients/s"
DEFAULT_WORKLOAD = "ncc_4096_t16"
# summed-area-table builders (ncc_sat_build_variant): the fused single pass is
# the product path; the naive and two-pass builds are the ones it is compared with
SAT_VARIANTS = {"fused": 0, "naive": 1, "two_pass": 2}
SAT_BYTES_PER_PX = 17          # 1 B read + 8 B (S) + 8 B (Q) written per pixel
CORR_BYTES_PER_COEFF = 21      # S and Q corners (16 B after reuse) + 1 B image + 4 B out
L2_FLUSH_BYTES = 512 << 20     # > 129 MB L2


def load_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        d["source"] = "measured"
        return d
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "sm_max_mhz": 2070.0,
            "source": "fallback"}


# Integer dot-product pipe: dp4a instructions per SM per clock on sm_103a,
# measured by a throughput microbenchmark (eight independent dp4a chains per
# thread: 63.9 per SM per clock, the same rate as IMAD); the ALU
# roofline is this times 152 SMs times the maximum SM clock.
DP4A_PER_SM_CLK = 64
N_SMS = 152
# Transform numerator: radix-2 modular butterflies per 256 x 256 tile (two
# halves of 128 rows; forward and inverse; 256-point row transforms on 128
# rows, 128-point column transforms on 256 columns).  Its ALU roofline is
# the SM's instruction issue rate (4 schedulers x 32 lanes per clock) at 7
# instructions per butterfly (the kernel's butterfly with a twiddle factor:
# three additions and a minimum on one output, an addition and a Shoup
# multiplication -- one high and two low products -- on the other).
NTT_BUTTERFLIES_PER_TILE = 2 * 2 * (128 * 128 * 8 + 256 * 64 * 7)
NTT_LANE_INSTR_PER_SM_CLK = 128
NTT_INSTR_PER_BUTTERFLY = 7


def ntt_tiles(W: int, H: int, wT: int, hT: int) -> int:
    """Tiles of the transform numerator (257 - hT rows by (257 - wT) rounded
    down to 16 columns of shifts each)."""
    vx, vy = (257 - wT) & ~15, 257 - hT
    return -(-(W - wT + 1) // vx) * -(-(H - hT + 1) // vy)

# DRAM bytes (read + write) of one launch, from one ncu capture of the bench
# command (dram__bytes_read.sum + dram__bytes_write.sum; summaries under
# profiles/).  Keyed by (kernel, workload); an entry is removed whenever its
# kernel changes, so a stale count is never reported.
NCU_TRAFFIC_BYTES = {
    ("sat_build", "ncc_4096_t16"): 229.4e6,
    ("sat_build", "large_8192_t64"): 1106.8e6,
    ("sat_build", "sat_8192"): 1106.8e6,
    ("bank_tc", "bank_2048_64x16"): 1104.4e6,
    ("corr_toeplitz_tc", "large_8192_t64"): 1393.3e6,
    ("corr_ntt", "wide_4096_t128"): 338.2e6,
}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, dist, device) -> float:
    """The largest of every rank's x (the slowest rank sets the job's time);
    x itself when running alone."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank: int, world_size: int, slowest_ms: float) -> float:
    """Whole-job throughput under weak scaling: every rank processes the same
    number of units; the job takes as long as its slowest rank."""
    return world_size * units_per_rank / (slowest_ms * 1e-3)


class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"ncc_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self) -> dict:
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        loaded = [v for v in sm if v >= 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(smax),
                "samples": len(sm), "samples_under_load": len(loaded),
                "reasons": sorted(reasons)}


def oracle_sample_rate(w: inputs.Workload, band_rows: int, threads: int) -> tuple[float, float]:
    """Times the CPU oracle on the top band of the workload: the tables of the
    band's image rows plus every coefficient of `band_rows` output rows.
    Returns (coefficients per second, seconds)."""
    import oracle
    sub = np.ascontiguousarray(w.image[: band_rows + w.hT - 1])
    t0 = time.perf_counter()
    oracle.sat(sub)
    oracle.correlate(sub, w.templates, threads=threads)
    dt = time.perf_counter() - t0
    return w.nT * band_rows * w.Ox / dt, dt


def sample_rows(w: inputs.Workload, requested: int | None) -> int:
    """Output rows of the oracle's bounded sample: the request, else as many
    rows as fit about 2e10 multiply-adds (a few seconds on many cores)."""
    if requested:
        return max(1, min(requested, w.Oy))
    return max(1, min(w.Oy, int(2e10 // (w.nT * w.Ox * w.wT * w.hT))))


def run_reference(args, w: inputs.Workload) -> dict:
    import oracle
    threads = oracle.default_threads()
    band = sample_rows(w, args.ref_rows)
    for _ in range(args.warmup):
        oracle_sample_rate(w, band, threads)
    times = []
    for _ in range(args.steps):
        _, dt = oracle_sample_rate(w, band, threads)
        times.append(dt)
    per_step = statistics.mean(times)
    rate = w.nT * band * w.Ox / per_step
    sample = (f"tables of the top {band + w.hT - 1} image rows + all {w.nT}x{band}x{w.Ox} "
              f"coefficients of those rows, per step")
    metric = METRIC if w.name == DEFAULT_WORKLOAD else f"NCC coefficients/s ({w.name})"
    return {
        "impl": "reference", "metric": metric, "value": rate, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": per_step * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "u8", "data": "synthetic",
        "config": {"workload": w.name, "image": f"{w.W}x{w.H} u8",
                   "templates": f"{w.nT}x{w.hT}x{w.wT} u8", "sample_rows": band},
        "cpu_baseline": {"value": rate, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": rate, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def device_batch(torch, img, n: int):
    """n distinct device images of img's shape and pixel distribution: img and
    n-1 seeded circular shifts of it (see inputs.batch_shifts)."""
    H, W = img.shape
    shifts = inputs.batch_shifts(n, W, H)
    return [img] + [torch.roll(img, shifts=(int(dy), int(dx)), dims=(0, 1))
                    for dy, dx in shifts[1:]]


def batch_size(per_call_ms: float, target_ms: float, image_bytes: int, cap_bytes: float) -> int:
    """Images per step: enough that one step lasts about target_ms, bounded so
    the batch's distinct images stay within cap_bytes of device memory."""
    b = int(np.ceil(target_ms / max(per_call_ms, 1e-3)))
    return int(max(1, min(b, cap_bytes // max(image_bytes, 1), 4096)))


def timed_steps(torch, stream, flush, steps: int, body) -> list[float]:
    """Times `steps` calls of body() with CUDA events on `stream`, the L2
    flushed before each; returns milliseconds per step."""
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for k in range(steps):
        flush.zero_()                          # L2 flushed between timed steps
        ev0[k].record(stream)
        body(k)
        ev1[k].record(stream)
    torch.cuda.synchronize()
    return [ev0[k].elapsed_time(ev1[k]) for k in range(steps)]


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part")):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def run_gpu(args, w: inputs.Workload) -> dict | None:
    import torch
    from normalized_cross_correlation_gb300 import ncc

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dist = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    L = ncc.lib()
    stream = torch.cuda.current_stream()
    sh = stream.cuda_stream
    dev = torch.device("cuda", local)

    nT = w.nT
    img0 = torch.from_numpy(w.image).to(dev)
    S = torch.empty((w.H, w.W), dtype=torch.int64, device=dev)
    Q = torch.empty((w.H, w.W), dtype=torch.int64, device=dev)
    if nT:
        tmpl = torch.from_numpy(w.templates).to(dev)
        out = torch.empty((nT, w.Oy, w.Ox), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    variant = SAT_VARIANTS[args.sat_variant]
    # The whole path in one call: the table build, then the correlation,
    # which (one template) overlaps the build's tail.  Only the single-pass
    # builder lets its dependents start early; the compared builders run the
    # two calls separately.
    fused = bool(nT) and variant == 0

    def sat(im, SS=S, QQ=Q):
        if variant == 0:
            rc = L.ncc_sat_build(im.data_ptr(), im.shape[1], im.shape[0], SS.data_ptr(),
                                 QQ.data_ptr(), sh)
        else:
            rc = L.ncc_sat_build_variant(im.data_ptr(), im.shape[1], im.shape[0], SS.data_ptr(),
                                         QQ.data_ptr(), variant, sh)
        assert rc == 0, rc

    def correlate(im):
        if nT == 1:
            rc = L.ncc_correlate(im.data_ptr(), w.W, w.H, tmpl.data_ptr(), w.wT, w.hT,
                                 S.data_ptr(), Q.data_ptr(), out.data_ptr(), sh)
        else:
            rc = L.ncc_correlate_bank(im.data_ptr(), w.W, w.H, tmpl.data_ptr(), w.wT, w.hT, nT,
                                      S.data_ptr(), Q.data_ptr(), out.data_ptr(), sh)
        assert rc == 0, rc

    def match(im):
        rc = L.ncc_match(im.data_ptr(), w.W, w.H, tmpl.data_ptr(), w.wT, w.hT, nT,
                         S.data_ptr(), Q.data_ptr(), out.data_ptr(), sh)
        assert rc == 0, rc

    def one_call(im):
        if fused:
            match(im)
        else:
            sat(im)
            if nT:
                correlate(im)

    # warm-up, then a calibration of one call's time (untimed for the result)
    for _ in range(args.warmup):
        flush.zero_()
        one_call(img0)
    cal = timed_steps(torch, stream, flush, 3, lambda k: one_call(img0))
    assert ncc.ncc_sync_status() == 0
    path = ncc.ncc_debug_last_path() if nT else ncc.NCC_PATH_NONE   # the kernel that ran
    B = args.batch or batch_size(statistics.mean(cal), args.step_ms, w.W * w.H, 4e9)
    images = device_batch(torch, img0, B)
    for im in images:                           # every image once, untimed
        one_call(im)
    torch.cuda.synchronize()
    assert ncc.ncc_sync_status() == 0

    # per-kernel events of the separate-call loop: SAT start, SAT end /
    # correlation start, correlation end, for every image of every step
    ev_s = [[torch.cuda.Event(enable_timing=True) for _ in range(B)] for _ in range(args.steps)]
    ev_m = [[torch.cuda.Event(enable_timing=True) for _ in range(B)] for _ in range(args.steps)]
    ev_e = [[torch.cuda.Event(enable_timing=True) for _ in range(B)] for _ in range(args.steps)]

    def split_step(k):
        for b, im in enumerate(images):
            ev_s[k][b].record(stream)
            sat(im)
            ev_m[k][b].record(stream)
            if nT:
                correlate(im)
            ev_e[k][b].record(stream)

    def fused_step(k):
        for im in images:
            match(im)

    # the table build alone on the 8192x8192 image of the large workload,
    # where the 129 MB L2 cannot hold back any of the 1.07 GB of tables
    # (prepared here, timed inside the sampled region below)
    large = None
    if args.sat_large and variant == 0 and w.W * w.H < 8192 * 8192:
        bimg = torch.from_numpy(inputs.large_8192().image).to(dev)
        S8 = torch.empty((8192, 8192), dtype=torch.int64, device=dev)
        Q8 = torch.empty_like(S8)
        for _ in range(3):
            sat(bimg, S8, Q8)
        cal8 = timed_steps(torch, stream, flush, 3, lambda k: sat(bimg, S8, Q8))
        B8 = batch_size(statistics.mean(cal8), args.step_ms / 2, 8192 * 8192, 4e9)
        large = (device_batch(torch, bimg, B8), S8, Q8)
        del bimg
        torch.cuda.synchronize()

    def large_step(k):
        bimgs, S8, Q8 = large
        for im in bimgs:
            sat(im, S8, Q8)

    clocks = ClockSampler(local)
    with clocks:
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        # timed region 1: the steps as a user runs them (ncc_match per image)
        t_fused = timed_steps(torch, stream, flush, args.steps, fused_step) if fused else None
        # timed region 2: the same steps as separate calls, with events
        # between the kernels for the per-kernel times and rooflines
        t_split = timed_steps(torch, stream, flush, args.steps, split_step)
        # timed region 3: the table build alone at 8192x8192
        t8 = timed_steps(torch, stream, flush, args.steps, large_step) if large else None
        if dist is not None:
            dist.barrier()
    assert ncc.ncc_sync_status() == 0
    t_sat = [ev_s[k][b].elapsed_time(ev_m[k][b]) for k in range(args.steps) for b in range(B)]
    t_corr = [ev_m[k][b].elapsed_time(ev_e[k][b]) for k in range(args.steps) for b in range(B)]
    t_step = t_fused if fused else t_split
    ms_step = max_over_ranks(statistics.mean(t_step), dist, dev)
    ms_split = max_over_ranks(statistics.mean(t_split), dist, dev)
    per_image = nT * w.Ox * w.Oy if nT else w.W * w.H
    value = job_rate(B * per_image, ws, ms_step)
    del images
    sat_large = None
    if large:
        B8 = len(large[0])
        sat_large = {"image": "8192x8192 u8 (large_8192_t64) and seeded circular shifts",
                     "images_per_step": B8,
                     "ms": max_over_ranks(statistics.mean(t8) / B8, dist, dev)}
        large = None

    # end to end through the host-buffer entry point (pinned host memory)
    e2e = None
    if nT:
        himg = torch.from_numpy(w.image).pin_memory()
        htmp = torch.from_numpy(w.templates).pin_memory()
        hout = torch.empty((nT, w.Oy, w.Ox), dtype=torch.float32).pin_memory()
        e2e_steps = max(3, min(args.steps, 10))
        for _ in range(2):
            ncc.ncc_match_host(himg, htmp, hout)
        e2e_t = []
        for _ in range(e2e_steps):
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            ncc.ncc_match_host(himg, htmp, hout)      # synchronizes the stream
            e2e_t.append(time.perf_counter() - t0)
        e2e_ms = max_over_ranks(statistics.mean(e2e_t) * 1e3, dist, dev)
        e2e = {"value": job_rate(per_image, ws, e2e_ms), "unit": UNIT, "ms_per_step": e2e_ms,
               "h2d_bytes_per_step": int(w.image.nbytes + w.templates.nbytes),
               "d2h_bytes_per_step": int(per_image * 4)}
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    if rank != 0:
        return None

    peaks = load_peaks()
    hbm = float(peaks["hbm_gbs"])
    sat_ms, corr_ms = statistics.mean(t_sat), statistics.mean(t_corr)
    sat_gbs = SAT_BYTES_PER_PX * w.W * w.H / (sat_ms * 1e-3) / 1e9
    roof_sat = {"kernel": "sat_build", "workload": w.name, "bound": "hbm", "achieved": sat_gbs,
                "peak": hbm, "unit": "GB/s", "frac": sat_gbs / hbm,
                "traffic": NCU_TRAFFIC_BYTES.get(("sat_build", w.name)) if variant == 0 else None,
                "peak_source": peaks["source"]}
    rooflines = [roof_sat]
    if sat_large:
        gbs8 = SAT_BYTES_PER_PX * 8192 * 8192 / (sat_large["ms"] * 1e-3) / 1e9
        sat_large.update({"GB/s": gbs8, "frac_of_hbm": gbs8 / hbm})
        rooflines.append({"kernel": "sat_build", "workload": "large_8192_t64", "bound": "hbm",
                          "achieved": gbs8, "peak": hbm, "unit": "GB/s", "frac": gbs8 / hbm,
                          "traffic": NCU_TRAFFIC_BYTES.get(("sat_build", "large_8192_t64")),
                          "peak_source": peaks["source"]})
    corr = None
    dominant = roof_sat
    if nT:
        macs = per_image * w.wT * w.hT
        if nT == 1 and path == ncc.NCC_PATH_TOEPLITZ:
            # useful multiply-adds only (the Toeplitz form issues about Kp/wT
            # times as many) against the f16 tensor rate (= the bf16 rate)
            corr_bytes = CORR_BYTES_PER_COEFF * w.Ox * w.Oy
            tflops = 2.0 * macs / (corr_ms * 1e-3) / 1e12
            peak_tc = float(peaks.get("bf16_tflops", 1900.0))
            r2 = {"kernel": "corr_toeplitz_tc", "workload": w.name, "bound": "tensor",
                  "achieved": tflops, "peak": peak_tc, "unit": "TFLOP/s", "frac": tflops / peak_tc,
                  "traffic": NCU_TRAFFIC_BYTES.get(("corr_toeplitz_tc", w.name))}
        elif nT == 1 and path == ncc.NCC_PATH_NTT:
            # modular butterflies (the spectrum kernel's share is in corr_ms
            # too) against the instruction-issue roofline
            corr_bytes = CORR_BYTES_PER_COEFF * w.Ox * w.Oy
            bfly = ntt_tiles(w.W, w.H, w.wT, w.hT) * NTT_BUTTERFLIES_PER_TILE
            peak_b = (NTT_LANE_INSTR_PER_SM_CLK * N_SMS * float(peaks.get("sm_max_mhz", 2070.0)) * 1e6 /
                      NTT_INSTR_PER_BUTTERFLY)
            r2 = {"kernel": "corr_ntt", "workload": w.name, "bound": "alu",
                  "achieved": bfly / (corr_ms * 1e-3) / 1e12, "peak": peak_b / 1e12,
                  "unit": "Tbutterfly/s", "frac": bfly / (corr_ms * 1e-3) / peak_b,
                  "traffic": NCU_TRAFFIC_BYTES.get(("corr_ntt", w.name))}
        elif nT == 1:
            # S and Q corners (16 B after reuse) + 1 B image + 4 B out per coefficient
            corr_bytes = CORR_BYTES_PER_COEFF * w.Ox * w.Oy
            dp4a = w.Ox * w.Oy * ((w.wT + 3) // 4) * w.hT
            alu_peak = DP4A_PER_SM_CLK * N_SMS * float(peaks.get("sm_max_mhz", 2070.0)) * 1e6
            r2 = {"kernel": "corr_dp4a", "workload": w.name, "bound": "alu",
                  "achieved": dp4a / (corr_ms * 1e-3) / 1e12, "peak": alu_peak / 1e12,
                  "unit": "Tdp4a/s", "frac": dp4a / (corr_ms * 1e-3) / alu_peak,
                  "traffic": NCU_TRAFFIC_BYTES.get(("corr_dp4a", w.name))}
        else:
            # 4 B out per coefficient + S and Q (16 B) + image (1 B) per shift
            corr_bytes = 4 * per_image + 17 * w.Ox * w.Oy
            tflops = 2.0 * macs / (corr_ms * 1e-3) / 1e12
            peak_tc = float(peaks.get("bf16_tflops", 1900.0))  # f16 runs at the bf16 rate
            r2 = {"kernel": "bank_tc", "workload": w.name, "bound": "tensor", "achieved": tflops,
                  "peak": peak_tc, "unit": "TFLOP/s", "frac": tflops / peak_tc,
                  "traffic": NCU_TRAFFIC_BYTES.get(("bank_tc", w.name))}
        corr_gbs = corr_bytes / (corr_ms * 1e-3) / 1e9
        r1 = {"kernel": r2["kernel"], "workload": w.name, "bound": "hbm", "achieved": corr_gbs,
              "peak": hbm, "unit": "GB/s", "frac": corr_gbs / hbm, "traffic": r2["traffic"]}
        rooflines += [r1, r2]
        corr_roof = max(r1, r2, key=lambda r: r["frac"])
        dominant = roof_sat if sat_ms >= corr_ms else corr_roof
        corr = {"kernel": r2["kernel"], "ms": corr_ms, "GB/s": corr_gbs,
                "GMAC/s": macs / (corr_ms * 1e-3) / 1e9}

    cpu = None
    if args.cpu_baseline and nT and rank == 0:
        import oracle
        threads = oracle.default_threads()
        rows = sample_rows(w, args.ref_rows)
        rate, dt = oracle_sample_rate(w, rows, threads)
        rows1 = max(1, rows // 4)
        rate1, dt1 = oracle_sample_rate(w, rows1, 1)
        cpu = {"value": rate, "unit": UNIT, "cores": threads, "kind": "oracle",
               "model": cpu_model(),
               "sample": f"tables of the top {rows + w.hT - 1} image rows + all "
                         f"{nT}x{rows}x{w.Ox} coefficients of those rows ({dt:.1f} s)",
               "single_thread": {"value": rate1, "unit": UNIT, "cores": 1,
                                 "sample": f"the same for the top {rows1} output rows "
                                           f"({dt1:.1f} s)"}}

    metric = METRIC if w.name == DEFAULT_WORKLOAD else f"NCC coefficients/s ({w.name})"
    calls = ("ncc_sat_build + " + ("ncc_correlate" if nT == 1 else
                                   "ncc_correlate_bank" if nT else "nothing"))
    launches_per_image = ((2 if path == ncc.NCC_PATH_NTT else 1) if nT else 0) + (1 if variant == 0 else 2)
    return {
        "metric": metric, "value": value, "unit": UNIT if nT else "pixels/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u8",
        "data": "synthetic",
        "config": {"workload": w.name, "image": f"{w.W}x{w.H} u8",
                   "templates": f"{nT}x{w.hT}x{w.wT} u8" if nT else None,
                   "images_per_step": B,
                   "batch": "the workload image and seeded circular shifts of it, one call each",
                   "step": ("ncc_match per image (ncc_sat_build, then ncc_correlate" +
                            (", overlapped)" if nT == 1 else "_bank)")) if fused else
                           calls + " per image",
                   "sat_builder": args.sat_variant,
                   "l2": "flushed between timed steps (512 MB write); within a step the images "
                         "differ and each one's tables exceed L2"},
        "ms_per_image": ms_step / B,
        "split_step": {"ms": ms_split, "ms_per_image": ms_split / B, "calls": calls,
                       "note": "the per-kernel times and rooflines come from these steps"},
        "sat_build": {"ms": sat_ms, "GB/s": sat_gbs, "frac_of_hbm": sat_gbs / hbm},
        "sat_build_8192": sat_large,
        "correlate": corr,
        "correlate_path": {ncc.NCC_PATH_DP4A: "dp4a", ncc.NCC_PATH_TOEPLITZ: "toeplitz_tc",
                           ncc.NCC_PATH_NTT: "ntt", ncc.NCC_PATH_BANK: "bank_tc"}.get(path),
        "roofline": {k: dominant[k] for k in ("bound", "achieved", "peak", "unit", "frac", "traffic")},
        "rooflines": rooflines,
        "cpu_baseline": cpu,
        "e2e": e2e,
        # this library's kernels in the timed loops
        "gpu_launches": launches_per_image * B * args.steps * (2 if fused else 1) +
                        (sat_large["images_per_step"] * args.steps if sat_large else 0),
        "clocks": clocks.summary(),
    }


def run_gpu_direct(args, w: inputs.Workload) -> dict | None:
    """The direct-moment correlation (ncc_correlate_direct): one kernel per
    template and step, no summed-area tables.  A comparison line, not the
    headline: the method's denominators come from the tables."""
    import torch
    from normalized_cross_correlation_gb300 import ncc

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dist = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    L = ncc.lib()
    stream = torch.cuda.current_stream()
    sh = stream.cuda_stream
    dev = torch.device("cuda", local)
    nT = w.nT
    img0 = torch.from_numpy(w.image).to(dev)
    tmpl = torch.from_numpy(w.templates).to(dev)
    out = torch.empty((nT, w.Oy, w.Ox), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def call(im):
        rc = L.ncc_correlate_direct(im.data_ptr(), w.W, w.H, tmpl.data_ptr(), w.wT, w.hT, nT,
                                    out.data_ptr(), sh)
        assert rc == 0, rc

    for _ in range(args.warmup):
        flush.zero_()
        call(img0)
    cal = timed_steps(torch, stream, flush, 3, lambda k: call(img0))
    assert ncc.ncc_sync_status() == 0
    B = args.batch or batch_size(statistics.mean(cal), args.step_ms, w.W * w.H, 4e9)
    images = device_batch(torch, img0, B)
    for im in images:
        call(im)
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    with clocks:
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        t = timed_steps(torch, stream, flush, args.steps, lambda k: [call(im) for im in images])
        if dist is not None:
            dist.barrier()
    assert ncc.ncc_sync_status() == 0
    ms_step = max_over_ranks(statistics.mean(t), dist, dev)
    ms = ms_step / B                            # one image
    coeffs = nT * w.Ox * w.Oy
    value = job_rate(B * coeffs, ws, ms_step)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    if rank != 0:
        return None
    peaks = load_peaks()
    hbm = float(peaks["hbm_gbs"])
    dp4a = coeffs * ((w.wT + 3) // 4) * w.hT
    alu_peak = DP4A_PER_SM_CLK * N_SMS * float(peaks.get("sm_max_mhz", 2070.0)) * 1e6
    corr_bytes = 4 * coeffs + w.W * w.H * nT      # coefficients out, the image once per template
    r_alu = {"kernel": "corr_dp4a_direct", "bound": "alu", "achieved": dp4a / (ms * 1e-3) / 1e12,
             "peak": alu_peak / 1e12, "unit": "Tdp4a/s", "frac": dp4a / (ms * 1e-3) / alu_peak,
             "traffic": NCU_TRAFFIC_BYTES.get(("corr_dp4a_direct", w.name))}
    gbs = corr_bytes / (ms * 1e-3) / 1e9
    r_hbm = {"kernel": "corr_dp4a_direct", "bound": "hbm", "achieved": gbs, "peak": hbm,
             "unit": "GB/s", "frac": gbs / hbm, "traffic": r_alu["traffic"]}
    dominant = max(r_alu, r_hbm, key=lambda r: r["frac"])
    return {
        "metric": f"NCC coefficients/s ({w.name}, direct moments)", "value": value, "unit": UNIT,
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "ms_per_image": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u8",
        "data": "synthetic",
        "config": {"workload": w.name, "image": f"{w.W}x{w.H} u8",
                   "templates": f"{nT}x{w.hT}x{w.wT} u8", "images_per_step": B,
                   "batch": "the workload image and seeded circular shifts of it, one call each",
                   "step": "ncc_correlate_direct per image",
                   "moments": "direct (staged image tile, no summed-area tables)",
                   "l2": "flushed between timed steps (512 MB write)"},
        "correlate": {"kernel": "corr_dp4a_direct", "ms": ms, "GB/s": gbs,
                      "GMAC/s": coeffs * w.wT * w.hT / (ms * 1e-3) / 1e9},
        "roofline": {k: dominant[k] for k in ("bound", "achieved", "peak", "unit", "frac", "traffic")},
        "rooflines": [r_alu, r_hbm],
        "cpu_baseline": None,
        "e2e": None,
        "gpu_launches": nT * B * args.steps,
        "clocks": clocks.summary(),
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--ref-rows", type=int, default=None,
                    help="output rows of the oracle's bounded sample per step "
                         "(default: about 2e10 multiply-adds' worth)")
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--batch", type=int, default=0,
                    help="images per timed step (default: enough for about --step-ms)")
    ap.add_argument("--step-ms", type=float, default=40.0,
                    help="target device time of one timed step, which sets the batch")
    ap.add_argument("--no-sat-large", dest="sat_large", action="store_false",
                    help="skip the table-build roofline on the 8192x8192 image")
    ap.add_argument("--sat-variant", default="fused", choices=sorted(SAT_VARIANTS),
                    help="summed-area-table builder: the single pass (default) or one of the "
                         "builds it is compared with")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(inputs.NAMED),
                    help="workload to time (the default is the headline metric's)")
    ap.add_argument("--moments", default="sat", choices=["sat", "direct"],
                    help="window moments from the summed-area tables (the method, default) or "
                         "from the staged image tile (ncc_correlate_direct, a comparison line)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3) if args.impl == "gb300" else args.warmup

    w = inputs.NAMED[args.workload]()
    ws, rank, _ = dist_env()
    if args.impl == "reference":
        if rank != 0 or not w.nT:
            return
        print(json.dumps(run_reference(args, w)), flush=True)
        return
    if args.moments == "direct" and not w.nT:
        return
    res = run_gpu_direct(args, w) if args.moments == "direct" else run_gpu(args, w)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
