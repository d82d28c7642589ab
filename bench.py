"""Benchmark of the tile stitch (and, alongside, every other kernel) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one tb_stitch2d call over the 2048x2048 bf16 workload: batch 4,
3 channels, a 6x6 grid of 512 px decoded tiles (latent tile 64, overlap 0.25,
scale 8; blend 128, row_limit 384, last tiles 128 px), synthetic smooth-field
tiles already resident in HBM.  The metric is GB/s moved (algorithmic bytes:
every tile element read once plus the output written once, 274.07 MB per
step), with % of the measured HBM peak and output Mpixel/s.  Three input /
output sets rotate between steps (822 MB, far above the 129 MB L2), so no
step finds its inputs in L2.

The JSON line also carries:
  e2e         the same metric through the C ABI with host buffers: every
              step copies the tiles from pinned host memory, stitches, and
              copies the image back;
  roofline    achieved vs measured HBM bandwidth for the stitch kernel, with
              the DRAM traffic of the last ncu capture of the same kernel
              source (null if the source changed since);
  kernels     every kernel on its own workload: rotating buffer sets (no
              L2 reuse), launches replayed from a CUDA graph, CUDA events
              (us); the single-launch duration under ncu recorded in
              profiles/single_launch.txt for the current kernel source
              (us_ncu_single); and one launch at a time after an L2 flush,
              GPU-side launch included (us_single);
  cpu_baseline  the CPU oracle timed on this host: whole steps for about 10 s
              on all cores (one plane per thread) and 10 s single-threaded.

Under torchrun (N > 1) every rank runs the same step on its own GPU (weak
scaling, no collective on the data path); the time is the max over ranks.

--impl reference times the CPU oracle (the unoptimised restatement of the
method) on bounded samples of the same workload: the only other
implementation of this path available here.
"""
import argparse
import dataclasses
import ctypes
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "stitch GB/s moved and % of GB300 HBM peak; output Mpixel/s (2048² bf16 grid)"
WORKLOAD = "image_2048_bf16"
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 1024 * 1024


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------

def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def stitch_bytes(layouts, planes, esize):
    """Algorithmic bytes of one stitch: each tile element that is kept or lent
    to a neighbour's band, read once, plus the output written once."""
    reads = []
    for lay in layouts:
        r = []
        for n in range(lay.n):
            e_next = lay.blends[n + 1] if n + 1 < lay.n else 0
            r.append(min(lay.extents[n], lay.kept[n] + e_next))
        reads.append(r)
    tile_elems = 0
    if len(layouts) == 2:
        for ry in reads[0]:
            for rx in reads[1]:
                tile_elems += ry * rx
    else:
        for rt in reads[0]:
            for ry in reads[1]:
                for rx in reads[2]:
                    tile_elems += rt * ry * rx
    out_elems = 1
    for lay in layouts:
        out_elems *= lay.out_extent
    return planes * (tile_elems + out_elems) * esize, planes * tile_elems * esize, planes * out_elems * esize


def ramp_bytes(ay, ax, planes, esize):
    """Algorithmic bytes of a normalised-ramp stitch: every tile sample with
    positive weight read once, plus the output written once."""
    def positive(a):
        n = len(a.origins)
        counts = []
        for t in range(n):
            c = 0
            for q in range(a.tile_extent):
                lo = t == 0 or q - a.zero > 0
                hi = t == n - 1 or (a.tile_extent - 1 - q) - a.zero > 0
                c += 1 if (lo and hi) else 0
            counts.append(c)
        return counts
    py, px = positive(ay), positive(ax)
    return planes * (sum(y * x for y in py for x in px) + ay.out_extent * ax.out_extent) * esize


def source_digest(path):
    return hashlib.sha256(open(path, "rb").read()).hexdigest()[:16]


def profiled_traffic(kernel_key, src_path):
    """DRAM bytes per launch (read + write) recorded by the last ncu capture of
    this kernel on this workload (profiles/traffic.txt), if that capture was
    taken on the current kernel source; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.txt")
    try:
        for line in open(p):
            if line.startswith("#") or not line.strip():
                continue
            f = line.split()
            if f[0] != kernel_key:
                continue
            if f[5] != source_digest(os.path.join(ROOT, f[4])):
                return None, f[6] + " (kernel source changed since)"
            return int(f[1]), f[6]
    except OSError:
        pass
    return None, None


def profiled_single_us(kernel_key):
    """Median single-launch duration under ncu recorded in
    profiles/single_launch.txt for this kernel/workload, while the kernel
    source still matches the capture; else None."""
    p = os.path.join(ROOT, "profiles", "single_launch.txt")
    try:
        for line in open(p):
            if line.startswith("#") or not line.strip():
                continue
            f = line.split()
            if f[0] == kernel_key:
                return float(f[1]) if f[3] == source_digest(os.path.join(ROOT, f[2])) else None
    except OSError:
        pass
    return None


# A child process that reads the SM clock and the clock-event reasons
# through NVML (the driver's library, by ctypes: read-only queries) every
# half millisecond, so a timed region of a millisecond still holds samples.
# It prints "ready" once NVML answers, keeps its samples in memory and, when
# terminated, prints one line per sample: wall time, SM MHz, max SM MHz,
# reasons bitmask.
NVML_CHILD = r"""
import ctypes, signal, sys, time
uuid = sys.argv[1].encode()
nv = ctypes.CDLL("libnvidia-ml.so.1")
if nv.nvmlInit_v2() != 0:
    sys.exit(1)
h = ctypes.c_void_p()
if nv.nvmlDeviceGetHandleByUUID(uuid, ctypes.byref(h)) != 0:
    sys.exit(1)
try:
    reasons_fn = nv.nvmlDeviceGetCurrentClocksEventReasons
except AttributeError:
    reasons_fn = nv.nvmlDeviceGetCurrentClocksThrottleReasons
mx = ctypes.c_uint()
nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))
sm, rs = ctypes.c_uint(), ctypes.c_ulonglong()
stop = []
signal.signal(signal.SIGTERM, lambda *a: stop.append(1))
print("ready", flush=True)
rows = []
while not stop:
    if nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(sm)) == 0 and reasons_fn(h, ctypes.byref(rs)) == 0:
        rows.append((time.time(), sm.value, mx.value, rs.value))
    time.sleep(0.0005)
sys.stdout.write("".join("%.6f %d %d %d\n" % r for r in rows))
sys.stdout.flush()
"""


class NvmlSampler:
    """SM clock and clock-event reasons every 0.5 ms from a child process
    (NVML through ctypes); no rows if NVML cannot be used."""
    # NVML clock-event reason bits (nvml.h)
    BITS = (("hw", 0x8), ("hw_thermal", 0x40), ("sw_thermal", 0x20), ("sw_power", 0x4))

    def __init__(self, gpu_uuid):
        self.proc = None
        self.first = ""
        if gpu_uuid is None:
            return
        try:
            self.proc = subprocess.Popen([sys.executable, "-c", NVML_CHILD, gpu_uuid], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None


    def wait_ready(self, timeout=3.0):
        """Waits (at most `timeout` s) for the child's first sample."""
        if self.proc is None:
            return
        import select
        if select.select([self.proc.stdout], [], [], timeout)[0]:
            self.first = self.proc.stdout.readline()

    def stop(self):
        if self.proc is None:
            return []
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in (self.first + out).splitlines():
            f = line.split()
            if len(f) != 4:
                continue
            bits = int(f[3])
            row = dict(t=float(f[0]), sm=float(f[1]), sm_max=float(f[2]))
            for k, b in self.BITS:
                row[k] = "Active" if bits & b else "Not Active"
            rows.append(row)
        return rows


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""
    Q = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.proc = None
        self.lines = []
        try:
            args = ["nvidia-smi", "--query-gpu=" + self.Q, "--format=csv,noheader,nounits", "-lms", "100"]
            if gpu_id is not None:
                args += ["-i", str(gpu_id)]
            self.proc = subprocess.Popen(args, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return []
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                ts = time.mktime(time.strptime(f[0].split(".")[0], "%Y/%m/%d %H:%M:%S")) + \
                    (float("0." + f[0].split(".")[1]) if "." in f[0] else 0.0)
                rows.append(dict(t=ts, sm=float(f[1]), sm_max=float(f[2]), hw=f[5], hw_thermal=f[6],
                                 sw_thermal=f[7], sw_power=f[8]))
            except Exception:
                continue
        return rows

    @staticmethod
    def summarise(rows, t0, t1, margin=0.05, source="nvidia-smi every 100 ms"):
        if not rows:
            return None
        inside = [r for r in rows if t0 - margin <= r["t"] <= t1 + margin]
        window = "timed region" if margin == 0 else "timed region +- %.0f ms" % (margin * 1e3)
        if not inside:
            # the region was shorter than the sampling period: nearest samples
            mid = 0.5 * (t0 + t1)
            inside = sorted(rows, key=lambda r: abs(r["t"] - mid))[:3]
            window = "nearest samples (timed region %.3f s)" % (t1 - t0)
        reasons = set()
        for r in inside:
            for k, name in (("hw", "hw_slowdown"), ("hw_thermal", "hw_thermal_slowdown"),
                            ("sw_thermal", "sw_thermal_slowdown"), ("sw_power", "sw_power_cap")):
                if r[k].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in inside), "sm_max_mhz": max(r["sm_max"] for r in inside),
                "sm_min_mhz": min(r["sm"] for r in inside), "reasons": sorted(reasons), "samples": len(inside),
                "window": window, "source": source}


# ---------------------------------------------------------------------------
# multi-GPU aggregation (one process per GPU, weak scaling, no data collective)
# ---------------------------------------------------------------------------

def max_over_ranks(torch, dist, world, value, device):
    """The largest of every rank's `value` (the slowest rank's time)."""
    if world <= 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(bytes_per_rank_step, ms_per_step_slowest, world):
    """Aggregate GB/s: every rank moves its own step's bytes; the job takes
    as long as its slowest rank."""
    return bytes_per_rank_step * world / (ms_per_step_slowest * 1e-3) / 1e9


def link_rates(torch, dev, nbytes=256 << 20, reps=3):
    """This GPU's host link with pinned memory, measured: GB/s of host->device
    copies, of device->host copies, and of both at once (summed), each
    `reps` copies of `nbytes` on their own stream, after a warm-up."""
    h_in = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    h_out = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    d_in = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    d_out = torch.zeros(nbytes, dtype=torch.uint8, device=dev)
    s1, s2 = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def timed(h2d, d2h):
        torch.cuda.synchronize(dev)
        a, b, c = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        a.record(s1)
        s2.wait_event(a)
        for _ in range(reps):
            if h2d:
                with torch.cuda.stream(s1):
                    d_in.copy_(h_in, non_blocking=True)
            if d2h:
                with torch.cuda.stream(s2):
                    h_out.copy_(d_out, non_blocking=True)
        c.record(s2)
        s1.wait_event(c)
        b.record(s1)
        b.synchronize()
        return (h2d + d2h) * nbytes * reps / (a.elapsed_time(b) * 1e-3) / 1e9

    timed(True, True)
    rates = {"h2d_gbs": round(timed(True, False), 1), "d2h_gbs": round(timed(False, True), 1),
             "both_gbs": round(timed(True, True), 1)}
    del h_in, h_out, d_in, d_out
    return rates


def link_bound_ms(rates, h2d_bytes, d2h_bytes):
    """Least time per step the measured link allows for these copies: no
    faster than either direction alone, nor than both directions' sum."""
    return 1e3 * max(h2d_bytes / (rates["h2d_gbs"] * 1e9), d2h_bytes / (rates["d2h_gbs"] * 1e9),
                     (h2d_bytes + d2h_bytes) / (rates["both_gbs"] * 1e9))


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def run_ours(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    from patch_groupnorm_gb300 import build as lib_build
    lib_build.build()
    from patch_groupnorm_gb300 import tileblend as tb
    from patch_groupnorm_gb300 import workloads as W

    w = W.STITCH[args.workload]
    axes = [tb.Axis(a.latent_extent, a.latent_tile, a.overlap, a.scale) for a in w.axes]
    lays = [tb.tb_axis_layout(a) for a in axes]
    boxes = [list(zip(l.origins, l.extents)) for l in lays]
    out_ext = [l.out_extent for l in lays]
    tiles_cpu = W.make_stitch_tiles(w, boxes, out_ext)
    esize = 4 if w.dtype == "f32" else 2
    alg_bytes, tile_bytes, out_bytes = stitch_bytes(lays, w.B * w.C, esize)
    out_shape = (w.B, w.C, *out_ext)
    tdt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[w.dtype]

    nsets = 3
    sets = []
    for s in range(nsets):
        dev_tiles = [[t.to(dev) for t in row] for row in tiles_cpu]
        out = torch.empty(out_shape, dtype=tdt, device=dev)
        sets.append((dev_tiles, out))
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    a_y, a_x = axes[0].c(), axes[1].c()
    code = {"f32": tb.TB_F32, "f16": tb.TB_F16, "bf16": tb.TB_BF16}[w.dtype]
    calls = []
    for dev_tiles, out in sets:
        arr = (ctypes.c_void_p * (lays[0].n * lays[1].n))(*[t.data_ptr() for row in dev_tiles for t in row])
        calls.append((arr, out.data_ptr()))
    fn = tb._lib.tb_stitch2d
    H, Wd = out_ext

    def step(i):
        arr, optr = calls[i % nsets]
        st = fn(arr, code, w.B, w.C, ctypes.byref(a_y), ctypes.byref(a_x), optr, H, Wd, sh)
        if st != 0:
            raise tb.TileBlendError(st, "tb_stitch2d")

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    gpu_id = None
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        gpu_id = None
    sampler = ClockSampler(gpu_id)
    fine = NvmlSampler(gpu_id)
    time.sleep(0.3)  # the samplers' first readings
    fine.wait_ready()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    # Untimed, the GPU first spins long enough for the host to queue the K
    # calls behind the start event (about 60 us of host time per call), so a
    # short timed region measures the device, not the host's enqueue rate;
    # longer runs simply overlap the two.
    torch.cuda._sleep(int(min(args.steps * 120_000, 100_000_000)))
    t_wall0 = time.time()
    e0.record(stream)
    for i in range(args.steps):
        step(i)
    e1.record(stream)
    e1.synchronize()
    t_wall1 = time.time()
    if world > 1:
        dist.barrier()
    time.sleep(0.15)
    fine_rows = fine.stop()
    rows = sampler.stop()
    ms = max_over_ranks(torch, dist, world, e0.elapsed_time(e1), dev)
    ms_per_step = ms / args.steps
    gbs = alg_bytes / (ms_per_step * 1e-3) / 1e9
    value = whole_job_gbs(alg_bytes, ms_per_step, world)
    peak, peak_kind = measured_peaks()
    mpix = w.B * H * Wd / (ms_per_step * 1e-3) / 1e6 * world
    if any(t_wall0 <= r["t"] <= t_wall1 for r in fine_rows):
        clocks = ClockSampler.summarise(fine_rows, t_wall0, t_wall1, 0.0, "NVML every 0.5 ms (read-only queries)")
    else:
        clocks = ClockSampler.summarise(rows, t_wall0, t_wall1)

    # end to end through the C ABI with host buffers: every step copies its
    # tiles in from pinned host memory and its image back out.  The tiles sit
    # in one pinned staging buffer (each at a 256-byte aligned offset), so a
    # step's tiles come in with one copy into the same layout on the device
    # (36 copies of 4.8 MB run at 195 GB/s on this host link, one of 173 MB
    # at 211 GB/s).  Copies in, stitch and copies out run on three streams
    # over three rotating buffer sets, so step k+1's copy in overlaps step
    # k's stitch and copy out.
    e2e = None
    if not args.no_e2e:
        def packed(device, pin):
            offs, total = [], 0
            for row in tiles_cpu:
                for t in row:
                    offs.append(total)
                    total += (t.numel() * t.element_size() + 255) // 256 * 256
            flat = torch.empty(total, dtype=torch.uint8, device=device)
            if pin:
                flat = flat.pin_memory()
            views, k = [], 0
            for row in tiles_cpu:
                vr = []
                for t in row:
                    nb = t.numel() * t.element_size()
                    vr.append(flat[offs[k]:offs[k] + nb].view(t.dtype).view(t.shape))
                    k += 1
                views.append(vr)
            return flat, views

        host_flat, host_views = packed("cpu", True)
        for rh, rc in zip(host_views, tiles_cpu):
            for th, tc in zip(rh, rc):
                th.copy_(tc)
        e2e_sets = []
        for _ in range(nsets):
            dflat, dviews = packed(dev, False)
            dout = torch.empty(out_shape, dtype=tdt, device=dev)
            arr = (ctypes.c_void_p * (lays[0].n * lays[1].n))(*[t.data_ptr() for row in dviews for t in row])
            e2e_sets.append((dflat, arr, dout))
        host_out = [torch.empty(out_shape, dtype=tdt).pin_memory() for _ in range(nsets)]
        s_in, s_run, s_out = (torch.cuda.Stream(dev) for _ in range(3))
        ev_in = [torch.cuda.Event() for _ in range(nsets)]
        ev_run = [torch.cuda.Event() for _ in range(nsets)]
        ev_out = [torch.cuda.Event() for _ in range(nsets)]
        k_e2e = max(3, min(args.steps, args.e2e_steps))

        def e2e_step(i):
            q = i % nsets
            dflat, arr, out = e2e_sets[q]
            with torch.cuda.stream(s_in):
                if i >= nsets:
                    s_in.wait_event(ev_run[q])          # set q's tiles no longer read
                dflat.copy_(host_flat, non_blocking=True)
                ev_in[q].record(s_in)
            s_run.wait_event(ev_in[q])
            if i >= nsets:
                s_run.wait_event(ev_out[q])             # set q's image already copied out
            st = fn(arr, code, w.B, w.C, ctypes.byref(a_y), ctypes.byref(a_x), out.data_ptr(), H, Wd,
                    s_run.cuda_stream)
            if st != 0:
                raise tb.TileBlendError(st, "tb_stitch2d")
            ev_run[q].record(s_run)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_run[q])
                host_out[q].copy_(out, non_blocking=True)
                ev_out[q].record(s_out)

        for i in range(nsets):
            e2e_step(i)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        f0 = torch.cuda.Event(enable_timing=True)
        f1 = torch.cuda.Event(enable_timing=True)
        f0.record(s_in)
        for i in range(k_e2e):
            e2e_step(i)
        for q in range(nsets):
            s_out.wait_event(ev_out[q])
        f1.record(s_out)
        f1.synchronize()
        ems = max_over_ranks(torch, dist, world, f0.elapsed_time(f1), dev)
        rates = link_rates(torch, dev)
        bound_ms = link_bound_ms(rates, host_flat.numel(), out_bytes)
        e2e_gbs = whole_job_gbs(alg_bytes, ems / k_e2e, world)
        e2e = {"value": round(e2e_gbs, 2), "unit": "GB/s",
               "h2d_bytes_per_step": host_flat.numel(), "d2h_bytes_per_step": out_bytes, "steps": k_e2e,
               "ms_per_step": round(ems / k_e2e, 4),
               "link": dict(rates, bound_ms_per_step=round(bound_ms, 4),
                            bound_gbs=round(whole_job_gbs(alg_bytes, bound_ms, world), 1),
                            frac_of_bound=round(bound_ms / (ems / k_e2e), 4),
                            how="pinned copies of 256 MB x3 per direction, and both directions at once; the bound "
                                "is the larger of the step's copies in at the host-to-device rate, its copies out "
                                "at the device-to-host rate, and both at the two-way rate"),
               "how": "per step: the 36 tiles copied in from one pinned staging buffer (one copy), tb_stitch2d, "
                      "image copied out to pinned host memory; three streams, %d rotating buffer sets" % nsets}
        del host_flat, host_views, host_out, e2e_sets

    traffic, capture = profiled_traffic("stitch2d/" + args.workload, None)
    roofline = {"kernel": "tb::stitch_kernel<2D,bf16>", "bound": "hbm", "achieved": round(gbs, 1),
                "peak": peak, "peak_kind": "%s (%s)" % (peak_kind, "burst copy, kernel timed alone"),
                "unit": "GB/s", "frac": round(gbs / peak, 4), "traffic": traffic,
                "traffic_capture": capture, "algorithmic_bytes": alg_bytes}

    kernels = None
    if not args.no_kernels and rank == 0:
        kernels = per_kernel(torch, tb, W, dev, peak, args.kernel_reps)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = cpu_baseline(w, lays, tiles_cpu, alg_bytes)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
            "pct_of_hbm_peak": round(100 * gbs / peak, 2), "mpixel_per_s": round(mpix, 1),
            "config": {"workload": args.workload, "B": w.B, "C": w.C, "out_hw": out_ext,
                       "grid": [lays[0].n, lays[1].n], "latent_tile": 64, "overlap": 0.25, "scale": 8,
                       "algorithmic_bytes_per_step": alg_bytes,
                       "l2": "3 rotating input/output sets (%.0f MB) > 129 MB L2; no flush" % (
                           nsets * alg_bytes / 1e6),
                       "parallelism": "dp%d" % world if world > 1 else "single GPU",
                       "sharding": "every rank stitches its own batch of %d images (independent images: no "
                                   "exchange, no collective on the data path)" % w.B},
            "clocks": clocks, "e2e": e2e, "gpu_launches": args.steps, "roofline": roofline,
            "cpu_baseline": cpu, "kernels": kernels,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def per_kernel(torch, tb, W, dev, peak, reps, only=None):
    """Every kernel on its own workload, timed two ways.

    replay: enough input/output sets rotate that no launch finds its data in
    L2 (> 3x the 129 MB L2 between reuses); the launches are captured in a
    CUDA graph and replayed back to back, so host call overhead is excluded;
    per-launch time = replay time / launches (median of reps).
    single: one launch at a time, cold: before each, a 258 MB fill evicts L2
    and the GPU then spins for about 2 ms while the host queues the start
    event, a graph holding that one launch, and the end event, so the events
    bracket the launch alone (no host time); median of reps.  This is the
    figure comparable with ncu's serialised gpu__time_duration."""
    stream = torch.cuda.Stream(dev)
    res = []
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)

    def single_ms(launch_set, nsets):
        # each set's launch alone in a graph, replayed after the flush and a
        # GPU spin (the host's call and launch overheads stay outside)
        graphs = []
        for q in range(nsets):
            g1 = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g1, stream=stream):
                launch_set(q)
            graphs.append(g1)
        cur = torch.cuda.current_stream(dev)
        ts = []
        for r in range(reps + 2):
            flush.fill_(float(r))
            torch.cuda._sleep(4_000_000)     # ~2 ms at 2 GHz: the host queues what follows
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(cur)
            graphs[r % nsets].replay()
            b.record(cur)
            b.synchronize()
            if r >= 2:
                ts.append(a.elapsed_time(b))
        del graphs
        return statistics.median(ts)

    def timed(launch_set, nsets, nbytes, name, workload, per_graph=60):
        if only and workload not in only and name not in only:
            return
        with torch.cuda.stream(stream):
            for q in range(nsets):          # warm-up, outside capture
                launch_set(q)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for q in range(per_graph):
                launch_set(q % nsets)
        ts = []
        cur = torch.cuda.current_stream(dev)  # replay() launches on the current stream
        for r in range(reps + 2):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(cur)
            g.replay()
            b.record(cur)
            b.synchronize()
            if r >= 2:
                ts.append(a.elapsed_time(b) / per_graph)
        ms = statistics.median(ts)
        gbs = nbytes / (ms * 1e-3) / 1e9
        del g
        ms1 = single_ms(launch_set, nsets)
        gbs1 = nbytes / (ms1 * 1e-3) / 1e9
        ncu_us = profiled_single_us("%s/%s" % (name, workload))
        res.append({"kernel": name, "workload": workload, "us": round(ms * 1e3, 2), "GB/s": round(gbs, 1),
                    "frac_of_peak": round(gbs / peak, 4),
                    "us_ncu_single": ncu_us,
                    "frac_ncu_single": round(nbytes / (ncu_us * 1e-6) / 1e9 / peak, 4) if ncu_us else None,
                    "us_single": round(ms1 * 1e3, 2), "GB/s_single": round(gbs1, 1),
                    "frac_single": round(gbs1 / peak, 4), "bytes": nbytes, "sets": nsets})

    def nsets_for(nbytes):
        return max(2, math.ceil(3 * L2_BYTES / nbytes) + 1)

    def wanted(name, *kernels):
        return not only or name in only or any(k in only for k in kernels)

    for name, w in W.STITCH.items():
        if not wanted(name, "stitch2d", "stitch3d"):
            continue
        axes = [tb.Axis(a.latent_extent, a.latent_tile, a.overlap, a.scale) for a in w.axes]
        lays = [tb.tb_axis_layout(a) for a in axes]
        tiles = W.make_stitch_tiles(w, [list(zip(l.origins, l.extents)) for l in lays], [l.out_extent for l in lays])
        esize = 4 if w.dtype == "f32" else 2
        nbytes, _, _ = stitch_bytes(lays, w.B * w.C, esize)
        tdt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[w.dtype]
        ns = nsets_for(nbytes)
        shape = (w.B, w.C, *[l.out_extent for l in lays])
        if w.ndim == 2:
            sets = [([[t.to(dev) for t in row] for row in tiles], torch.empty(shape, dtype=tdt, device=dev))
                    for _ in range(ns)]
            timed(lambda q: tb.tb_stitch2d(sets[q][0], axes[0], axes[1], sets[q][1]), ns, nbytes, "stitch2d", name)
        else:
            sets = [([[[t.to(dev) for t in row] for row in pl] for pl in tiles], torch.empty(shape, dtype=tdt, device=dev))
                    for _ in range(ns)]
            timed(lambda q: tb.tb_stitch3d(sets[q][0], axes[0], axes[1], axes[2], sets[q][1]), ns, nbytes,
                  "stitch3d", name)
        del sets
        torch.cuda.empty_cache()
    for name in ("image_2048_bf16", "video_49x480x832_bf16"):
        # the band the first of two ranks packs for the second in a
        # row-sharded stitch: read once, written once
        if not wanted(name, "halo_pack"):
            continue
        w = W.STITCH[name]
        axes = [tb.Axis(a.latent_extent, a.latent_tile, a.overlap, a.scale) for a in w.axes]
        lays = [tb.tb_axis_layout(a) for a in axes]
        tiles = W.make_stitch_tiles(w, [list(zip(l.origins, l.extents)) for l in lays], [l.out_extent for l in lays])
        at, ay, ax = (None, axes[0], axes[1]) if w.ndim == 2 else axes
        lay = tb.tb_stitch_shard_layout(at, ay, ax, w.B, w.C, 2, 0)
        row = lay.row_end - 1
        tdt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[w.dtype]
        esize = 4 if w.dtype == "f32" else 2
        nbytes = 2 * lay.send_elems * esize
        ns = nsets_for(nbytes)
        sets = []
        for _ in range(ns):
            rt = [t.to(dev) for t in tiles[row]] if w.ndim == 2 else [[t.to(dev) for t in pl[row]] for pl in tiles]
            sets.append((rt, torch.empty(lay.send_elems, dtype=tdt, device=dev)))
        timed(lambda q: tb.tb_stitch_halo_pack(sets[q][0], at, ay, ax, row, sets[q][1]), ns, nbytes, "halo_pack",
              name)
        del sets
        torch.cuda.empty_cache()
    for name, w in W.RAMP.items():
        if not wanted(name, "stitch2d_ramp"):
            continue
        ay = tb.RampAxis.spread(w.latent_hw[0], w.latent_tile, w.n_tiles[0], w.scale)
        ax = tb.RampAxis.spread(w.latent_hw[1], w.latent_tile, w.n_tiles[1], w.scale)
        tiles = W.make_ramp_tiles(w, ay, ax)
        esize = 4 if w.dtype == "f32" else 2
        nbytes = ramp_bytes(ay, ax, w.B * w.C, esize)
        tdt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[w.dtype]
        ns = nsets_for(nbytes)
        shape = (w.B, w.C, ay.out_extent, ax.out_extent)
        sets = [([[t.to(dev) for t in row] for row in tiles], torch.empty(shape, dtype=tdt, device=dev))
                for _ in range(ns)]
        timed(lambda q: tb.tb_stitch2d_ramp(sets[q][0], ay, ax, sets[q][1]), ns, nbytes, "stitch2d_ramp", name)
        del sets
        torch.cuda.empty_cache()
    for name, w in W.GROUPNORM.items():
        if not wanted(name, "gn_stats", "gn_apply"):
            continue
        patches, gamma, beta = W.make_groupnorm_inputs(w)
        elems = sum(p.numel() for p in patches)
        es = patches[0].element_size()
        g, b = gamma.to(dev), beta.to(dev)
        ns = nsets_for(elems * es)
        sets = []
        for _ in range(ns):
            dp = [p.to(dev) for p in patches]
            sets.append((dp, [torch.empty_like(p) for p in dp], tb.new_partials(len(dp), dp[0].shape[0], w.groups, dev)))
        timed(lambda q: tb.tb_patch_gn_stats(sets[q][0], w.groups, sets[q][2]), ns, elems * es, "gn_stats", name)
        timed(lambda q: tb.tb_patch_gn_apply(sets[q][0], sets[q][1], w.groups, sets[q][2], g, b, w.eps, True), ns,
              2 * elems * es, "gn_apply", name)
        del sets
        torch.cuda.empty_cache()
    for name, w in W.PATCHIFY.items():
        if not wanted(name, "patchify", "gather_patches"):
            continue
        x = W.make_patchify_input(w)
        nbytes = 2 * x.numel() * x.element_size()     # every element read once and written once
        _, sizes = tb.tb_patchify_layout(w.shape[w.axis], w.factor, w.ranks)
        ns = nsets_for(nbytes)
        sets = []
        for _ in range(ns):
            xd = x.to(dev)
            parts = tb.tb_patchify(xd, w.axis, w.factor, w.ranks)
            sets.append((xd, parts, torch.empty_like(xd)))
        timed(lambda q: tb.tb_patchify(sets[q][0], w.axis, w.factor, w.ranks, patches=sets[q][1]), ns, nbytes,
              "patchify", name)
        timed(lambda q: tb.tb_gather_patches(sets[q][1], sizes, w.axis, out=sets[q][2]), ns, nbytes,
              "gather_patches", name)
        del sets
        torch.cuda.empty_cache()
    return res


def run_kernels_only(args):
    """Per-kernel timings of the named workloads or kernels, one JSON line."""
    import torch
    from patch_groupnorm_gb300 import build as lib_build
    if not os.environ.get("TILEBLEND_LIB"):
        lib_build.build()
    from patch_groupnorm_gb300 import tileblend as tb
    from patch_groupnorm_gb300 import workloads as W
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peak, _ = measured_peaks()
    only = set(args.kernels_only.split(","))
    res = per_kernel(torch, tb, W, dev, peak, args.kernel_reps, only=only)
    print(json.dumps({"lib": tb.LIB_PATH, "kernels": res}), flush=True)


def run_profile_target(args):
    """Launch one kernel on one workload W + K times with plain launches (no
    graph, no rotation): the command line ncu captures are taken from."""
    import torch
    from patch_groupnorm_gb300 import build as lib_build
    lib_build.build()
    from patch_groupnorm_gb300 import tileblend as tb
    from patch_groupnorm_gb300 import workloads as W
    kernel, _, name = args.profile.partition(":")
    dev = torch.device("cuda", 0)
    if kernel in ("stitch2d", "stitch3d"):
        w = W.STITCH[name]
        axes = [tb.Axis(a.latent_extent, a.latent_tile, a.overlap, a.scale) for a in w.axes]
        lays = [tb.tb_axis_layout(a) for a in axes]
        tiles = W.make_stitch_tiles(w, [list(zip(l.origins, l.extents)) for l in lays], [l.out_extent for l in lays])
        tdt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[w.dtype]
        out = torch.empty((w.B, w.C, *[l.out_extent for l in lays]), dtype=tdt, device=dev)
        if w.ndim == 2:
            dt = [[t.to(dev) for t in row] for row in tiles]
            launch = lambda: tb.tb_stitch2d(dt, axes[0], axes[1], out)
        else:
            dt = [[[t.to(dev) for t in row] for row in pl] for pl in tiles]
            launch = lambda: tb.tb_stitch3d(dt, axes[0], axes[1], axes[2], out)
    elif kernel == "stitch2d_ramp":
        w = W.RAMP[name]
        ay = tb.RampAxis.spread(w.latent_hw[0], w.latent_tile, w.n_tiles[0], w.scale)
        ax = tb.RampAxis.spread(w.latent_hw[1], w.latent_tile, w.n_tiles[1], w.scale)
        dt = [[t.to(dev) for t in row] for row in W.make_ramp_tiles(w, ay, ax)]
        tdt = dt[0][0].dtype
        out = torch.empty((w.B, w.C, ay.out_extent, ax.out_extent), dtype=tdt, device=dev)
        launch = lambda: tb.tb_stitch2d_ramp(dt, ay, ax, out)
    elif kernel == "halo_pack":
        # the band the first of two ranks sends in a row-sharded stitch
        w = W.STITCH[name]
        axes = [tb.Axis(a.latent_extent, a.latent_tile, a.overlap, a.scale) for a in w.axes]
        lays = [tb.tb_axis_layout(a) for a in axes]
        tiles = W.make_stitch_tiles(w, [list(zip(l.origins, l.extents)) for l in lays], [l.out_extent for l in lays])
        at, ay, ax = (None, axes[0], axes[1]) if w.ndim == 2 else axes
        lay = tb.tb_stitch_shard_layout(at, ay, ax, w.B, w.C, 2, 0)
        row = lay.row_end - 1
        tdt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[w.dtype]
        if w.ndim == 2:
            rt = [t.to(dev) for t in tiles[row]]
        else:
            rt = [[t.to(dev) for t in pl[row]] for pl in tiles]
        band = torch.empty(lay.send_elems, dtype=tdt, device=dev)
        launch = lambda: tb.tb_stitch_halo_pack(rt, at, ay, ax, row, band)
    elif kernel == "copy":
        # a plain copy of WORKLOAD megabytes (half read, half written) through
        # the library's copy kernel: the single-launch reference for a
        # streaming kernel of that many bytes
        nbytes = int(float(name) * 1e6) // 2 // 16 * 16
        xd = torch.empty(nbytes // 2, dtype=torch.bfloat16, device=dev).fill_(1.0)
        dst = [torch.empty_like(xd)]
        launch = lambda: tb.tb_patchify(xd, 0, 1, 1, patches=dst)
    elif kernel in ("patchify", "gather_patches"):
        w = W.PATCHIFY[name]
        xd = W.make_patchify_input(w).to(dev)
        parts = tb.tb_patchify(xd, w.axis, w.factor, w.ranks)
        back = torch.empty_like(xd)
        sizes = [p.shape[w.axis] for p in parts]
        if kernel == "patchify":
            launch = lambda: tb.tb_patchify(xd, w.axis, w.factor, w.ranks, patches=parts)
        else:
            launch = lambda: tb.tb_gather_patches(parts, sizes, w.axis, out=back)
    else:
        w = W.GROUPNORM[name]
        patches, gamma, beta = W.make_groupnorm_inputs(w)
        dp = [p.to(dev) for p in patches]
        outs = [torch.empty_like(p) for p in dp]
        part = tb.new_partials(len(dp), dp[0].shape[0], w.groups, dev)
        g, b = gamma.to(dev), beta.to(dev)
        tb.tb_patch_gn_stats(dp, w.groups, part)
        if kernel == "gn_stats":
            launch = lambda: tb.tb_patch_gn_stats(dp, w.groups, part)
        else:
            launch = lambda: tb.tb_patch_gn_apply(dp, outs, w.groups, part, g, b, w.eps, True)
    for _ in range(args.warmup + args.steps):
        launch()
    torch.cuda.synchronize()
    print(json.dumps({"profile": args.profile, "launches": args.warmup + args.steps}))


def cpu_baseline(w, lays_lib, tiles_cpu, alg_bytes):
    """The CPU oracle, as it stands, on whole steps of the workload (about
    10 s each way): on all host cores, one (batch, channel) plane per task
    (the C oracle releases the GIL), and single-threaded."""
    import concurrent.futures
    import numpy as np
    import torch
    from oracle.geometry import axis_layout
    from oracle.stitch import stitch as oracle_stitch

    lays = [axis_layout(a.latent_extent, a.latent_tile, a.overlap, a.scale) for a in w.axes]

    def raw(t):
        return t.view(torch.int16).numpy().view(np.uint16) if w.dtype != "f32" else t.numpy()

    whole = [[raw(t) for t in row] for row in tiles_cpu]
    planes = [[[np.ascontiguousarray(raw(t)[b:b + 1, c:c + 1]) for t in row] for row in tiles_cpu]
              for b in range(w.B) for c in range(w.C)]

    def timed(run):
        t0 = time.perf_counter()
        steps = 0
        while True:
            run()
            steps += 1
            dt = time.perf_counter() - t0
            if dt >= 10.0:
                return steps, dt

    cores = min(os.cpu_count() or 1, len(planes))
    with concurrent.futures.ThreadPoolExecutor(max_workers=cores) as ex:
        steps, dt = timed(lambda: list(ex.map(lambda pl: oracle_stitch(pl, lays, w.dtype), planes)))
    steps1, dt1 = timed(lambda: oracle_stitch(whole, lays, w.dtype))
    return {"value": round(steps * alg_bytes / dt / 1e9, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "seconds": round(dt, 3), "steps": steps,
            "sample": "%d full steps (%s: %d tiles, %.1f MB algorithmic each), C oracle, one (batch, channel) "
                      "plane per thread on %d host threads" % (steps, w.name, len(whole) * len(whole[0]),
                                                               alg_bytes / 1e6, cores),
            "single_thread": {"value": round(steps1 * alg_bytes / dt1 / 1e9, 4), "unit": "GB/s", "cores": 1,
                              "seconds": round(dt1, 3), "steps": steps1}}


# ---------------------------------------------------------------------------
# reference arm: the CPU oracle on bounded samples
# ---------------------------------------------------------------------------

def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import numpy as np
    import torch
    from oracle.geometry import axis_layout
    from oracle.stitch import stitch as oracle_stitch
    from patch_groupnorm_gb300 import workloads as W

    w = W.STITCH[args.workload]
    lays = [axis_layout(a.latent_extent, a.latent_tile, a.overlap, a.scale) for a in w.axes]
    boxes = [[(o * a.scale, L) for o, L in zip(l.origins, l.extents)] for l, a in zip(lays, w.axes)]
    tiles = W.make_stitch_tiles(w, boxes, [l.out_extent for l in lays])
    # one (batch, channel) plane of the workload
    plane = [[(t[:1, :1].contiguous().view(torch.int16).numpy().view(np.uint16) if w.dtype != "f32"
               else t[:1, :1].contiguous().numpy()) for t in row] for row in tiles]
    esize = 4 if w.dtype == "f32" else 2
    # Bound the whole run to about two minutes whatever --steps is: the sample
    # per step is the largest top-left sub-grid of r x q tiles of the plane
    # whose measured time fits (the recurrence of a top-left sub-grid does not
    # depend on the tiles below or to the right of it, so the sample is the
    # stitch of that part of the image).
    def head(l, m):
        kept = l.kept[:m]
        return dataclasses.replace(l, origins=l.origins[:m], extents=l.extents[:m], blends=l.blends[:m],
                                   kept=kept, offsets=l.offsets[:m], out_extent=sum(kept))

    ny, nx = lays[0].n, lays[1].n
    cands = sorted({(min(ny, a), min(nx, b)) for a in (ny, ny // 2, 3, 2, 1) for b in (nx, nx // 2, 3, 2, 1)
                    if a >= 1 and b >= 1}, key=lambda rq: -rq[0] * rq[1])
    limit = 120.0 / max(1, args.steps + args.warmup)
    for r, q in cands:
        sl = [head(lays[0], r), head(lays[1], q)]
        st = [row[:q] for row in plane[:r]]
        t0 = time.perf_counter()
        oracle_stitch(st, sl, w.dtype)
        if time.perf_counter() - t0 <= limit:
            break
    nbytes, _, _ = stitch_bytes(sl, 1, esize)
    for _ in range(args.warmup):
        oracle_stitch(st, sl, w.dtype)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_stitch(st, sl, w.dtype)
    dt = (time.perf_counter() - t0) / max(1, args.steps)
    value = nbytes / dt / 1e9
    sample = "per step the top-left %d x %d tiles of one (batch, channel) plane of %s (%.2f MB algorithmic)" % (
        r, q, w.name, nbytes / 1e6)
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
            "data": "synthetic", "config": {"workload": args.workload, "sample": sample},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--kernel-reps", type=int, default=50)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-kernels", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--kernels-only", default=None,
                    help="comma-separated workloads or kernel names: print only their per-kernel timings")
    ap.add_argument("--profile", default=None,
                    help="KERNEL:WORKLOAD (stitch2d|stitch3d|stitch2d_ramp|gn_stats|gn_apply|patchify|"
                         "gather_patches|halo_pack, or copy:MEGABYTES): plain launches for ncu")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.profile:
        run_profile_target(args)
        return
    if args.kernels_only:
        run_kernels_only(args)
        return
    if args.impl == "reference":
        if "--steps" not in sys.argv:
            args.steps = 5
        if "--warmup" not in sys.argv:
            args.warmup = 1
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
