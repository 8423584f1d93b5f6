"""Benchmark of the local W4A16 MoE forward on one GB300.

Workload (default): 384 experts, hidden 7168, intermediate 256, gated SwiGLU,
top-k 8, INT4 group-32 weights with BF16 scales, BF16 activations, seeded
synthetic inputs, renormalize=False.  One step = route preparation + gate/up
GEMM + SwiGLU + down GEMM + FP32 top-k combine over one batch of T tokens
(default T = 2048), replayed from a CUDA graph.  The L2 is flushed (a 512 MB
write) before every timed step, outside the timed events.  The token sweep
1, 8, 32, 256, 1024 is measured the same way and reported under "sweep"; the
other workloads (the 32-of-256-expert local shape, the per-channel BF16 and
FP16 shapes, the skewed ReLU^2 shape) under "workloads".

Prints ONE JSON line.  ``--impl reference`` times the CPU oracle instead (the
same workload on the host cores; whole batches, fewer steps).
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
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from workloads import gen  # noqa: E402

HEADLINE_TOKENS = 2048
SWEEP_TOKENS = (1, 8, 32, 256, 1024)
GEMM_PATHS = {"auto": 0, "tc": 1, "cc": 2}
PATH_NAMES = {1: "tensor_cores", 2: "cuda_cores"}
# Pages' number for this exact workload and metric (CuTe W4A16, one H200, T=2048,
# LMDeploy PR page, Benchmark table): context from another machine.
PAGE_LATENCY_US = {2048: 1280.327, 1024: 844.461, 256: 604.272, 32: 269.418, 8: 91.890, 1: 22.690}
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def kernel_source_hash():
    """Hash of the GEMM kernel sources; a committed traffic capture counts only
    while it matches."""
    import hashlib
    h = hashlib.sha256()
    for f in ("weight_only_int4_histogram_gb300/csrc/gemm.cuh",
              "weight_only_int4_histogram_gb300/csrc/gemv.cuh",
              "weight_only_int4_histogram_gb300/csrc/gemv_fused.cuh",
              "weight_only_int4_histogram_gb300/csrc/common.cuh"):
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_traffic(workload, tokens, kernel, path_name):
    """DRAM bytes per launch from the committed ncu summaries, or None when no
    capture matches this workload, kernel and GEMM path, or the kernel
    sources have changed since."""
    path = os.path.join(ROOT, "profiles", "roofline_traffic.json")
    try:
        with open(path) as f:
            tr = json.load(f)
    except (OSError, ValueError):
        return None
    if tr.get("kernel_source_hash") != kernel_source_hash():
        return None
    for c in tr.get("captures", []):
        if (c.get("workload"), c.get("tokens"), c.get("kernel"), c.get("gemm_path")) == \
                (workload, tokens, kernel, path_name):
            return int(c["dram_bytes"])
    return None


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), float(pk["bf16_tflops"]), "measured"
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    """SM clock and clock-event reasons sampled during the timed region.

    Polls NVML (read-only queries through ctypes) from a background thread
    every millisecond, so that even a timed region of a few milliseconds gets
    samples; falls back to `nvidia-smi -lms 200` when NVML cannot be loaded.
    Nothing here changes a GPU setting."""

    REASON_BITS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                   0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.tmp = None
        self.thread = None
        self.samples = []
        self.reasons = set()
        self.max_mhz = None
        self.nvml = None
        self.handle = None

    def _open_nvml(self):
        import ctypes
        for name in ("libnvidia-ml.so.1", "libnvidia-ml.so"):
            try:
                lib = ctypes.CDLL(name)
                break
            except OSError:
                lib = None
        if lib is None or lib.nvmlInit_v2() != 0:
            return False
        handle = ctypes.c_void_p()
        bus = None
        try:
            props = torch.cuda.get_device_properties(self.dev)
            bus = "%08x:%02x:%02x.0" % (props.pci_domain_id, props.pci_bus_id, props.pci_device_id)
        except Exception:
            pass
        ok = bus is not None and lib.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(handle)) == 0
        if not ok and lib.nvmlDeviceGetHandleByIndex_v2(self.dev, ctypes.byref(handle)) != 0:
            return False
        mx = ctypes.c_uint()
        if lib.nvmlDeviceGetMaxClockInfo(handle, 1, ctypes.byref(mx)) == 0:  # NVML_CLOCK_SM
            self.max_mhz = float(mx.value)
        self.reasons_fn = (getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None)
                           or getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons", None))
        self.nvml, self.handle = lib, handle
        return True

    def _poll(self):
        import ctypes
        mhz = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        while not self._stop:
            if self.nvml.nvmlDeviceGetClockInfo(self.handle, 1, ctypes.byref(mhz)) == 0:
                self.samples.append(float(mhz.value))
            if self.reasons_fn is not None and self.reasons_fn(self.handle, ctypes.byref(rs)) == 0:
                for bit, name in self.REASON_BITS.items():
                    if rs.value & bit:
                        self.reasons.add(name)
            time.sleep(0.001)

    def start(self):
        import threading
        try:
            if self._open_nvml():
                self._stop = False
                self.thread = threading.Thread(target=self._poll, daemon=True)
                self.thread.start()
                time.sleep(0.01)  # first samples before the timed region
                return
        except Exception:
            self.nvml = None
        try:
            self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.dev}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.tmp, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.thread is not None:
            self._stop = True
            self.thread.join(timeout=5)
            # samples taken while the GPU ran the timed steps (the last few
            # milliseconds of idle are dropped with the tail)
            sm = self.samples
            return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": self.max_mhz,
                    "reasons": sorted(self.reasons), "samples": len(sm), "source": "nvml"}
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.tmp.flush()
        self.tmp.seek(0)
        rows = [r.strip().split(",") for r in self.tmp.read().splitlines() if r.strip()]
        self.tmp.close()
        os.unlink(self.tmp.name)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx = float(r[2])
                for n, v in zip(names, r[5:9]):
                    if v.strip().lower() == "active":
                        reasons.add(n)
            except (ValueError, IndexError):
                continue
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm), "source": "nvidia-smi"}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def l2_flush_buffer(device):
    return torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=device)


def capture(moe, w, x, ids, tw, out, stream):
    with torch.cuda.stream(stream):
        for _ in range(2):
            moe(x, w, tw, ids, out=out, stream=stream)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        moe(x, w, tw, ids, out=out, stream=stream)
    torch.cuda.synchronize()
    return g


def time_graph(g, flush, stream, steps, warmup):
    for _ in range(warmup):
        flush.zero_()
        g.replay()
    torch.cuda.synchronize()
    times = []
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    with torch.cuda.stream(stream):
        for a, b in ev:
            flush.zero_()
            a.record(stream)
            g.replay()
            b.record(stream)
    torch.cuda.synchronize()
    for a, b in ev:
        times.append(a.elapsed_time(b) * 1000.0)  # us
    return times


def time_warm(g, stream, samples=3, reps=10):
    """The pages' protocol, for comparison with their figures: warm CUDA-graph
    replays (no L2 flush), each sample the mean of `reps` back-to-back
    replays, the median of `samples` samples."""
    out = []
    with torch.cuda.stream(stream):
        for _ in range(samples):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(reps):
                g.replay()
            b.record(stream)
            torch.cuda.synchronize()
            out.append(a.elapsed_time(b) * 1000.0 / reps)
    return statistics.median(out)


def time_stages(moe, w, x, ids, tw, out, flush, stream, steps):
    """Per-kernel device time of the GEMMs and combine (eager launches, events
    recorded by the library between kernels, L2 flushed before each step)."""
    from weight_only_int4_histogram_gb300 import _lib
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    for e in evs:           # torch creates the CUDA event on first record
        e.record(stream)
    torch.cuda.synchronize()
    _lib.w4a16_moe_set_stage_events(moe.plan, [e.cuda_event for e in evs])
    acc = [[], [], []]
    try:
        for _ in range(steps):
            with torch.cuda.stream(stream):
                flush.zero_()
                moe(x, w, tw, ids, out=out, stream=stream)
            torch.cuda.synchronize()
            for i in range(3):
                acc[i].append(evs[i].elapsed_time(evs[i + 1]) * 1000.0)
    finally:
        _lib.w4a16_moe_set_stage_events(moe.plan, [])
    return [statistics.mean(a) for a in acc]


def time_router(cfg, T, flush, stream, steps, hbm):
    """The router step (softmax + top-k over the workload's logits), timed on
    its own: the pages keep it outside the forward's timed region.  L2 flushed
    before every launch; algorithmic bytes = logits read + ids/weights written."""
    import weight_only_int4_histogram_gb300 as W
    logits = gen.make_logits(cfg, T, "cuda")
    for _ in range(3):
        W.route_topk(logits, cfg.top_k, stream=stream)
    times = []
    for _ in range(steps):
        with torch.cuda.stream(stream):
            flush.zero_()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        W.route_topk(logits, cfg.top_k, stream=stream)
        b.record(stream)
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b) * 1000.0)
    us = statistics.median(times)
    nbytes = T * cfg.n_global * 4 + T * cfg.top_k * 8
    gbs = nbytes / (us * 1e-6) / 1e9
    return {"us": round(us, 3), "gbs": round(gbs, 1), "frac": round(gbs / hbm, 4), "alg_bytes": nbytes,
            "what": "router softmax + top-k of the same tokens (outside the forward's timed region)"}


def time_masked(cfg, ids, w, flush, stream, steps, hbm, layout=0):
    """The masked-count entry point on the rows a dispatch of the same routes
    would deliver: counts[e] = routes to local expert e, rows padded to
    max_rows = max count rounded up to 16.  Same kernels as the forward (each
    row one route of weight 1); algorithmic bytes = touched experts' weights
    and scales + the valid rows in and out."""
    from weight_only_int4_histogram_gb300 import W4A16MoE
    loc = ids.long() - cfg.expert_offset
    valid = (ids >= 0) & (loc >= 0) & (loc < cfg.num_experts)
    counts = torch.bincount(loc[valid], minlength=cfg.num_experts).to(torch.int32)
    M = int((int(counts.max()) + 15) // 16 * 16)
    E = cfg.num_experts
    mcfg = cfg.with_(top_k=1)
    moe = W4A16MoE.from_config(mcfg, max_tokens=E * M)
    moe.set_weight_layout(layout)
    x = gen.make_activations(mcfg, E * M, "cuda").view(E, M, cfg.hidden)
    cnt = counts.cuda()
    y = torch.empty_like(x)
    for _ in range(3):
        moe.forward_masked(x, w, cnt, out=y, stream=stream)
    times = []
    for _ in range(steps):
        with torch.cuda.stream(stream):
            flush.zero_()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        moe.forward_masked(x, w, cnt, out=y, stream=stream)
        b.record(stream)
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b) * 1000.0)
    moe.check_device_error()
    us = statistics.median(times)
    b1, b2, _ = stage_bytes(cfg, ids)
    rows = int(counts.sum())
    nbytes = b1 - ids.shape[0] * cfg.hidden * 2 + b2 + 2 * rows * cfg.hidden * 2
    gbs = nbytes / (us * 1e-6) / 1e9
    moe.close()
    return {"us": round(us, 3), "gbs": round(gbs, 1), "frac": round(gbs / hbm, 4), "alg_bytes": nbytes,
            "rows": rows, "max_rows": M,
            "what": "masked-count layout entry (per-expert rows of the same routes; eager launches, L2 flushed)"}


def stage_bytes(cfg, ids):
    """Algorithmic bytes per launch of each kernel: the touched experts'
    packed weights + scales, the activations it must read, the output."""
    T = ids.shape[0]
    loc = ids.long() - cfg.expert_offset
    valid = (ids >= 0) & (loc >= 0) & (loc < cfg.num_experts)
    touched = int(torch.unique(loc[valid]).numel())
    H, I, N1 = cfg.hidden, cfg.inter, cfg.n1
    g = cfg.scale_kind == gen.SCALE_GROUP32
    b1 = touched * (H * N1 // 2 + (H * N1 // 32 * 2 if g else N1 * 2)) + T * H * 2
    b2 = touched * (I * H // 2 + (I * H // 32 * 2 if g else H * 2))
    b3 = T * H * 2 + T * cfg.top_k * 8
    return b1, b2, b3


def max_over_ranks(values, dist, device):
    """Element-wise maximum of per-rank times: the job takes as long as its
    slowest rank (replicas run the same work on every GPU)."""
    if dist is None:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def run_ncu_target(args):
    """A short, profiler-friendly run: the workload's weights and one batch,
    `--warmup` eager forwards, then one more, synchronised.  Prints one line.
    (Kernel launches per forward: route preparation (one or two), the gate/up
    GEMM, the down GEMM, the combine.)"""
    from weight_only_int4_histogram_gb300 import W4A16MoE, build
    build.build()
    torch.cuda.set_device(0)
    cfg = gen.CONFIGS[args.config]
    w_ckpt = gen.make_weights(cfg, "cuda")
    moe = W4A16MoE.from_config(cfg, max_tokens=args.tokens)
    moe.set_gemm_path(GEMM_PATHS[args.gemm_path])
    w = moe.relayout_weights(w_ckpt) if args.weights == "interleaved" else w_ckpt
    x = gen.make_activations(cfg, args.tokens, "cuda")
    ids, tw = gen.make_routes(cfg, args.tokens, "cuda")
    for _ in range(args.warmup + 1):
        moe(x, w, tw, ids)
    torch.cuda.synchronize()
    moe.check_device_error()
    info = moe.route_info(args.tokens)
    print(json.dumps({"ncu_target": cfg.name, "tokens": args.tokens, "forwards": args.warmup + 1,
                      "gemm_path": PATH_NAMES[info.gemm_path], "tile_rows": info.tile_rows,
                      "splits": [info.gemm1_splits, info.gemm2_splits]}))


# Other workloads reported beside the headline: (workload, tokens).
OTHER_WORKLOADS = (("deepseek_local_e32of256_h7168_i2048_k8", 2048),
                   ("deepseek_local_e32of256_h7168_i2048_k8", 64),
                   ("per_channel_e60_h2048_i1408_k4", 1024),
                   ("per_channel_fp16_e60_h2048_i1408_k4", 1024),
                   ("relu2_skew_e64_h2688_i1856_k6", 4096),
                   ("relu2_skew_e64_h2688_i1856_k6", 32))


def metric_name(cfg):
    return f"W4A16 MoE forward latency (us), {cfg.name}"


def roofline_of(cfg, ids, us, hbm, bf16):
    nbytes = gen.algorithmic_bytes(cfg, ids)
    flops = gen.algorithmic_flops(cfg, ids)
    t_hbm = nbytes / (hbm * 1e9) * 1e6
    t_tc = flops / (bf16 * 1e12) * 1e6
    t_roof = max(t_hbm, t_tc)
    return dict(gbs=round(nbytes / us / 1e3, 1), alg_bytes=nbytes, alg_flops=flops,
                roofline_us=round(t_roof, 3), roofline_frac=round(t_roof / us, 4),
                hbm_frac=round(t_hbm / us, 4), tensor_frac=round(t_tc / us, 4),
                bound="hbm" if t_hbm >= t_tc else "tensor")


def measure_other_workloads(dev, flush, stream, hbm, bf16, steps, weights_layout):
    """Each other workload at its listed token count: its own weights and
    plan, relaid out like the headline's, CUDA-graph replay with the L2
    flushed, median of `steps`."""
    from weight_only_int4_histogram_gb300 import W4A16MoE
    out = {}
    cache = {}
    for name, T in OTHER_WORKLOADS:
        cfg = gen.CONFIGS[name]
        if name not in cache:
            cache.clear()
            w_ckpt = gen.make_weights(cfg, dev)
            moe = W4A16MoE.from_config(cfg, max_tokens=max(cfg.tokens), device=dev)
            w = moe.relayout_weights(w_ckpt) if weights_layout == "interleaved" else w_ckpt
            cache[name] = (moe, w)
        moe, w = cache[name]
        x = gen.make_activations(cfg, T, dev)
        ids, tw = gen.make_routes(cfg, T, dev)
        o = torch.empty(T, cfg.hidden, dtype=cfg.torch_act_dtype(), device=dev)
        g = capture(moe, w, x, ids, tw, o, stream)
        times = time_graph(g, flush, stream, steps, 3)
        moe.check_device_error()
        med = statistics.median(times)
        r = dict(tokens=T, us=round(med, 3), gemm_path=PATH_NAMES[moe.route_info(T).gemm_path])
        r.update(roofline_of(cfg, ids, med, hbm, bf16))
        out[f"{name}@{T}"] = r
        del g
    cache.clear()
    torch.cuda.empty_cache()
    return out


def run_gpu(args):
    from weight_only_int4_histogram_gb300 import W4A16MoE, build
    build.build()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    cfg = gen.CONFIGS[args.config]
    hbm, bf16, peak_kind = load_peaks()

    w_ckpt = gen.make_weights(cfg, dev)
    moe = W4A16MoE.from_config(cfg, max_tokens=max(max(cfg.tokens), args.tokens, max(args.sweep_tokens)),
                               device=dev)
    moe.set_gemm_path(GEMM_PATHS[args.gemm_path])
    # setup, outside every timed region: the plan-time relayout of the packed weights
    w = moe.relayout_weights(w_ckpt) if args.weights == "interleaved" else w_ckpt
    torch.cuda.synchronize()
    flush = l2_flush_buffer(dev)
    stream = torch.cuda.Stream(device=dev)

    def measure(T, steps, warmup, sample_clocks=False):
        x = gen.make_activations(cfg, T, dev)
        ids, tw = gen.make_routes(cfg, T, dev)
        out = torch.empty(T, cfg.hidden, dtype=cfg.torch_act_dtype(), device=dev)
        g = capture(moe, w, x, ids, tw, out, stream)
        clk = ClockSampler(local_rank)
        if sample_clocks:
            clk.start()
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        times = time_graph(g, flush, stream, steps, warmup)
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        clocks = clk.stop() if sample_clocks else None
        moe.check_device_error()
        med = statistics.median(times)
        res = dict(tokens=T, us=round(med, 3), us_min=round(min(times), 3),
                   gemm_path=PATH_NAMES[moe.route_info(T).gemm_path])
        res.update(roofline_of(cfg, ids, med, hbm, bf16))
        return res, (x, ids, tw, out, g), times, clocks

    head, (x, ids, tw, out, g), times, clocks = measure(args.tokens, args.steps, args.warmup, True)
    warm = time_warm(g, stream)
    # the dominant kernel's live timing and roofline
    st = time_stages(moe, w, x, ids, tw, out, flush, stream, max(args.steps, 5))
    b = list(stage_bytes(cfg, ids))
    names = ["gate_up_gemm", "down_gemm", "combine"]
    if moe.route_info(args.tokens).fused_gemms:
        # CUDA-core path with both GEMMs in one launch: its events coincide
        names = ["expert_gemms_fused", "down_gemm_in_fused", "combine"]
        b = [b[0] + b[1], 0, b[2]]
    k = max(range(3), key=lambda i: st[i])
    achieved = b[k] / (st[k] * 1e-6) / 1e9
    roof = {"kernel": names[k], "bound": "hbm", "achieved": round(achieved, 1), "peak": hbm,
            "peak_kind": f"{peak_kind} hbm_gbs", "unit": "GB/s",
            "frac": round(achieved / hbm, 4),
            "traffic": measured_traffic(cfg.name, args.tokens, names[k], head["gemm_path"]),
            "alg_bytes_per_launch": b[k], "launch_us": round(st[k], 3),
            "stage_us": {n: round(v, 3) for n, v in zip(names, st)}}
    router = time_router(cfg, args.tokens, flush, stream, max(args.steps, 5), hbm)
    masked = time_masked(cfg, ids, w, flush, stream, max(args.steps, 5), hbm,
                         layout=1 if args.weights == "interleaved" else 0)

    sweep = []
    if not args.no_sweep:
        for T in args.sweep_tokens:
            if T == args.tokens:
                continue
            r, *_ = measure(T, max(10, args.steps // 2), args.warmup)
            sweep.append(r)
        sweep.append(head)
        sweep.sort(key=lambda r: r["tokens"])

    # end to end through the C ABI with pinned host buffers (copies in the timed region)
    xh = x.cpu().pin_memory()
    idh = ids.cpu().pin_memory()
    twh = tw.cpu().pin_memory()
    oh = torch.empty(args.tokens, cfg.hidden, dtype=cfg.torch_act_dtype(), pin_memory=True)
    for _ in range(args.warmup):
        moe.forward_host(xh, w, twh, idh, out_host=oh, stream=stream)
    e2e = []
    for _ in range(args.steps):
        flush.zero_()
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        bb = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        moe.forward_host(xh, w, twh, idh, out_host=oh, stream=stream)
        bb.record(stream)
        torch.cuda.synchronize()
        e2e.append(a.elapsed_time(bb) * 1000.0)
    e2e_med = statistics.median(e2e)
    h2d = xh.numel() * 2 + idh.numel() * 4 + twh.numel() * 4
    d2h = oh.numel() * 2

    med, e2e_med, warm = max_over_ranks([head["us"], e2e_med, warm], dist, dev)
    workloads = {}
    if not args.no_workloads:
        workloads = measure_other_workloads(dev, flush, stream, hbm, bf16, max(10, args.steps // 2), args.weights)
    line = {
        "metric": metric_name(cfg),
        "value": round(med, 3),
        "unit": "us",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(med / 1000.0, 6),
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": round(med / PAGE_LATENCY_US[args.tokens], 4) if args.tokens in PAGE_LATENCY_US and cfg is gen.KIMI else None,
        "dtype": "bf16" if cfg.act_dtype == gen.DT_BF16 else "f16",
        "data": "synthetic (seeded; weights N(0,0.02) quantised to INT4 g32, x N(0,1), softmax top-k routes)",
        "config": {"workload": cfg.name, "tokens": args.tokens, "experts": cfg.num_experts,
                   "hidden": cfg.hidden, "inter": cfg.inter, "top_k": cfg.top_k,
                   "weights": args.weights,
                   "timing": "CUDA-graph replay, median of steps, CUDA events on the launch stream",
                   "l2": "flushed before every timed step (512 MB write)",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": roof,
        "headline": head,
        "sweep": sweep,
        "e2e": {"value": round(e2e_med, 3), "unit": "us", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        # route prep, two GEMMs, combine
        "gpu_launches": 4 * args.steps,
        "warm_replay": {"us": round(warm, 3),
                        "protocol": "the pages' timing: warm CUDA-graph replays, mean of 10, median of 3 samples"},
        "router": router,
        "masked_layout": masked,
        "workloads": workloads,
        "clocks": clocks,
    }
    if not args.no_cpu_baseline and rank == 0 and world == 1:
        line["cpu_baseline"] = cpu_baseline(cfg, args.tokens, (w_ckpt.to("cpu"), x.cpu(), ids.cpu(), tw.cpu()))
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


# ---------------------------------------------------------------------------
# CPU oracle (reported baseline / reference arm)
# ---------------------------------------------------------------------------

def cpu_baseline(cfg, tokens, inputs=None):
    """The CPU oracle (plain loops, OpenMP) on the host cores: the whole batch
    once, measured, plus one token on a single thread."""
    import oracle
    oracle.build()
    if inputs is None:
        inputs = make_inputs_for_cpu(cfg, tokens)
    w, x, ids, tw = inputs
    cores = oracle.num_threads()
    t0 = time.perf_counter()
    oracle.moe_forward(cfg, x, w, tw, ids, nthreads=cores)
    dt = time.perf_counter() - t0
    t1 = time.perf_counter()
    oracle.moe_forward(cfg, x[:1], w, tw[:1], ids[:1], nthreads=1)
    dt1 = time.perf_counter() - t1
    return {"value": round(dt * 1e6, 1), "unit": "us", "cores": cores, "kind": "oracle",
            "sample": f"the whole {tokens}-token batch once ({dt:.2f} s on {cores} threads)",
            "single_thread": {"tokens": 1, "us": round(dt1 * 1e6, 1), "cores": 1}}


def make_inputs_for_cpu(cfg, tokens):
    # Generated on the GPU when there is one (seconds instead of a minute), then
    # copied to host memory; input generation is never timed.
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    w = gen.make_weights(cfg, dev).to("cpu")
    x = gen.make_activations(cfg, tokens, dev).cpu()
    ids, tw = gen.make_routes(cfg, tokens, dev)
    return w, x, ids.cpu(), tw.cpu()


def run_reference(args):
    """The CPU oracle as the reference arm: every step is the whole batch of
    the same workload (no extrapolation); steps are capped so that the run
    stays within minutes."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    cfg = gen.CONFIGS[args.config]
    import oracle
    oracle.build()
    w, x, ids, tw = make_inputs_for_cpu(cfg, args.tokens)
    steps = max(1, min(args.steps, args.ref_max_steps))
    cores = oracle.num_threads()
    for _ in range(min(args.warmup, 1)):
        oracle.moe_forward(cfg, x[:1], w, tw[:1], ids[:1], nthreads=cores)
    times = []
    for _ in range(steps):
        t0 = time.perf_counter()
        oracle.moe_forward(cfg, x, w, tw, ids, nthreads=cores)
        times.append((time.perf_counter() - t0) * 1e6)
    v = statistics.median(times)
    line = {
        "impl": "reference",
        "metric": metric_name(cfg),
        "value": round(v, 1), "unit": "us", "n_gpus": int(os.environ.get("WORLD_SIZE", "1")),
        "steps": steps, "warmup": min(args.warmup, 1), "ms_per_step": round(v / 1000.0, 3),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)",
        "config": {"workload": cfg.name, "tokens": args.tokens},
        "cpu_baseline": {"value": round(v, 1), "unit": "us", "cores": cores,
                         "kind": "oracle",
                         "sample": f"every step the whole {args.tokens}-token batch; {steps} steps "
                                   f"(requested {args.steps}, capped at {args.ref_max_steps})"},
        "e2e": {"value": round(v, 1), "unit": "us", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default=gen.KIMI.name, choices=list(gen.CONFIGS))
    ap.add_argument("--tokens", type=int, default=HEADLINE_TOKENS)
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--sweep", default=",".join(str(t) for t in SWEEP_TOKENS),
                    help="comma-separated token counts of the sweep")
    ap.add_argument("--gemm-path", default="auto", choices=list(GEMM_PATHS),
                    help="where the expert GEMMs run (auto: planner's choice per batch)")
    ap.add_argument("--weights", default="interleaved", choices=["interleaved", "checkpoint"],
                    help="packed weight layout the forward reads (interleaved: relaid out once at setup)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ncu", action="store_true",
                    help="profiler target: --warmup eager forwards + 1 of one batch, no timing")
    ap.add_argument("--ref-max-steps", type=int, default=3,
                    help="reference arm: at most this many whole-batch oracle steps")
    ap.add_argument("--no-workloads", action="store_true", help="skip the other workloads")
    args = ap.parse_args()
    args.sweep_tokens = tuple(int(t) for t in args.sweep.split(",") if t.strip())
    if args.ncu:
        run_ncu_target(args)
        return
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
