"""Benchmark of the FP8 quantized actor linear layer on GB300.

One step = one pass of the whole hot path over the 8B-shaped training
workload (X bf16 [8192, 4096], W bf16 [14336, 4096], dY bf16 [8192, 14336]):

  1. UAQ fold of W and of a norm weight (R = 1), in place
     (the channel scale alternates between s and 1/s so W stays stationary)
  2. fused 1x128 + 128x1 quantization of X
  3. fused 1x128 + 128x1 quantization of dY
  4. 128x128 quantization of W (no transposed copy: DGrad reads the FProp codes
     MN-major, as fast as the K-major copy and 58.7 MB of writes cheaper)
  5. FProp  Y  = X W^T
  6. DGrad  dX = dY W
  7. WGrad  dW = dY^T X

Every step launches only this library's kernels (7 launches; the fold of W and
of the norm weight is one).  L2 is flushed
(a 256 MB device write, outside the timed events) before every step; each
step is timed with CUDA events on the launching stream, per kernel and whole.

``value`` is the step's GEMM throughput, 3 * 2*M*N*K FLOP / step time, so the
quantizers and the fold count against it.  Per-kernel TFLOP/s and GB/s, each
against its roofline, are in ``kernels``.  ``e2e`` repeats the step through
host buffers (pinned host -> device copies of X, W, dY; device -> host copies of
Y, dX, dW inside the timed region).  ``cpu_baseline`` and ``--impl reference``
time the test oracle (plain C + NumPy fp64) on the host cores over a bounded
sample of the same workload.

Multi-GPU: the path has no exchange step, so N GPUs run N independent replicas
("weak" scaling): value = total FLOP over all ranks / max step time.
"""
from __future__ import annotations

import argparse
import json
import os
import platform
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

M_, N_, K_ = 8192, 14336, 4096
WORKLOAD = "8B-shaped training step (Llama-3.1-8B MLP up-proj): fold + quant X/dY/W + FProp/DGrad/WGrad"
METRIC = "FP8 block-scaled GEMM TFLOPS & % FP8 peak; quantizer GB/s & % of HBM BW"
UAQ_S = 1.5  # QuRL's recommended fold factor

# algorithmic bytes per element
B_DUAL = 2 + 1 + 1 + 4 / 128 + 4 / 128
B_WEIGHT_T = 2 + 1 + 1 + 4 / 16384
B_FOLD_W = 4  # read + write bf16 per weight element
B_ROWS = 2 + 1 + 4 / 128
B_WEIGHT = 2 + 1 + 4 / 16384

# Rate a probe of back-to-back tcgen05.mma.kind::f8f6f4 from shared memory sustained on
# all SMs of a GB300 (no TMA, no epilogue): reported as context beside the roofline.
FP8_MMA_PROBE_TFLOPS = 4860.0


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_burst": p["bf16_tflops"],
                "bf16_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_burst": 1900.0, "bf16_sustained": 1700.0, "source": "fallback"}


# ----------------------------------------------------------------- dist ---

def _dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        if torch.cuda.is_available():
            torch.cuda.set_device(local)  # before the group: NCCL binds each rank to its current device
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
        return dist, rank, world, local
    return None, 0, 1, local


def _barrier(dist):
    if dist is not None:
        dist.barrier()


def _max_over_ranks(dist, v: float) -> float:
    if dist is None:
        return v
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------- clocks ---

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            # nvidia-smi takes a moment to print its first sample: start the timed
            # region only once sampling is running (at most 3 s of waiting).
            t_end = time.time() + 3.0
            while not self.lines and time.time() < t_end and self.proc.poll() is None:
                time.sleep(0.01)
        except (OSError, FileNotFoundError):
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

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- step ---

class Step:
    """Device buffers and the launch sequence of one step."""

    def __init__(self, dev, host):
        from fp8_block_scaled_quantize_gb300 import rlq
        self.rlq = rlq
        M, N, K = M_, N_, K_
        self.dev = dev
        bf = torch.bfloat16
        self.x = torch.empty((M, K), dtype=bf, device=dev)
        self.w = torch.empty((N, K), dtype=bf, device=dev)
        self.dy = torch.empty((M, N), dtype=bf, device=dev)
        self.gamma = torch.ones((1, K), dtype=bf, device=dev)
        self.s_fwd = torch.full((K,), UAQ_S, dtype=torch.float32, device=dev)
        self.s_bwd = torch.full((K,), 1.0 / UAQ_S, dtype=torch.float32, device=dev)
        u8, f32 = torch.uint8, torch.float32
        self.qx = torch.empty((M, K), dtype=u8, device=dev)
        self.sx = torch.empty((K // 128, M), dtype=f32, device=dev)
        self.qxT = torch.empty((K, M), dtype=u8, device=dev)
        self.sxc = torch.empty((M // 128, K), dtype=f32, device=dev)
        self.qdy = torch.empty((M, N), dtype=u8, device=dev)
        self.sdy = torch.empty((N // 128, M), dtype=f32, device=dev)
        self.qdyT = torch.empty((N, M), dtype=u8, device=dev)
        self.sdyc = torch.empty((M // 128, N), dtype=f32, device=dev)
        self.qw = torch.empty((N, K), dtype=u8, device=dev)
        self.sw = torch.empty((N // 128, K // 128), dtype=f32, device=dev)
        self.y = torch.empty((M, N), dtype=bf, device=dev)
        self.dx = torch.empty((M, K), dtype=bf, device=dev)
        self.dw = torch.empty((N, K), dtype=bf, device=dev)
        self.x.copy_(host["x"])
        self.w.copy_(host["w"])
        self.dy.copy_(host["dy"])
        self.parity = 0
        self.launches_per_step = 7

    def run(self, stream: int, events=None):
        """Launch the step; if `events` (8 CUDA events) is given, record them
        around the kernels."""
        r = self.rlq
        M, N, K = M_, N_, K_
        s = self.s_fwd if self.parity == 0 else self.s_bwd
        self.parity ^= 1
        rec = (lambda i: events[i].record()) if events is not None else (lambda i: None)
        rec(0)
        r.rlq_uaq_fold(self.w.data_ptr(), N, K, K, s.data_ptr(), self.gamma.data_ptr(), 1, K, stream)
        rec(1)
        r.rlq_quant_act_1x128(self.x.data_ptr(), M, K, K, self.qx.data_ptr(), K, self.sx.data_ptr(), M,
                              self.qxT.data_ptr(), M, self.sxc.data_ptr(), K, stream)
        rec(2)
        r.rlq_quant_act_1x128(self.dy.data_ptr(), M, N, N, self.qdy.data_ptr(), N, self.sdy.data_ptr(), M,
                              self.qdyT.data_ptr(), M, self.sdyc.data_ptr(), N, stream)
        rec(3)
        r.rlq_quant_weight_128x128(self.w.data_ptr(), N, K, K, self.qw.data_ptr(), K, self.sw.data_ptr(), K // 128,
                                   None, 0, stream)
        rec(4)
        r.rlq_gemm_fprop(self.qx.data_ptr(), K, self.sx.data_ptr(), M, self.qw.data_ptr(), K, self.sw.data_ptr(),
                         K // 128, self.y.data_ptr(), N, M, N, K, stream)
        rec(5)
        r.rlq_gemm_dgrad(self.qdy.data_ptr(), N, self.sdy.data_ptr(), M, self.qw.data_ptr(), K, 0,
                         self.sw.data_ptr(), K // 128, self.dx.data_ptr(), K, M, N, K, stream)
        rec(6)
        r.rlq_gemm_wgrad(self.qdyT.data_ptr(), M, self.sdyc.data_ptr(), N, self.qxT.data_ptr(), M,
                         self.sxc.data_ptr(), K, self.dw.data_ptr(), K, M, N, K, stream)
        rec(7)


KERNELS = ["uaq_fold", "quant_dual_x", "quant_dual_dy", "quant_weight_128x128", "gemm_fprop", "gemm_dgrad",
           "gemm_wgrad"]


def kernel_work():
    """Algorithmic work per launch: ("bytes", B) or ("flop", F)."""
    M, N, K = M_, N_, K_
    return {
        "uaq_fold": ("bytes", B_FOLD_W * N * K + 4 * K + 4 * K),
        "quant_dual_x": ("bytes", B_DUAL * M * K),
        "quant_dual_dy": ("bytes", B_DUAL * M * N),
        "quant_weight_128x128": ("bytes", B_WEIGHT * N * K),
        "gemm_fprop": ("flop", 2.0 * M * N * K),
        "gemm_dgrad": ("flop", 2.0 * M * N * K),
        "gemm_wgrad": ("flop", 2.0 * M * N * K),
    }


def make_host_inputs():
    from fp8_block_scaled_quantize_gb300 import inputs as I
    d = I.train_step_8b()
    return {k: I.to_torch(v) for k, v in d.items()}


def run_ours(args):
    from fp8_block_scaled_quantize_gb300 import rlq

    dist, rank, world, local = _dist_setup(args.gpus)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    rlq.lib()
    peaks = _peaks()
    host = make_host_inputs()
    st = Step(dev, host)
    stream = torch.cuda.current_stream()
    sh = stream.cuda_stream
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size if hasattr(torch.cuda.get_device_properties(dev), "L2_cache_size") else 128 << 20
    flush = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)

    for _ in range(args.warmup):
        flush.zero_()
        st.run(sh)
    rlq.check(sh)
    torch.cuda.synchronize()

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(8)] for _ in range(args.steps)]
    _barrier(dist)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        for i in range(args.steps):
            flush.zero_()  # outside the timed events
            st.run(sh, evs[i])
        torch.cuda.synchronize()
    _barrier(dist)
    rlq.check(sh)

    # the same steps with only a start and an end event each: the per-kernel events
    # above sit between the kernels in the stream and keep each kernel from being
    # scheduled while the previous one drains (programmatic dependent launch)
    plain = []
    for _ in range(args.steps):
        flush.zero_()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record()
        st.run(sh)
        a1.record()
        plain.append((a0, a1))
    torch.cuda.synchronize()
    rlq.check(sh)
    plain_ms = _max_over_ranks(dist, statistics.mean(a0.elapsed_time(a1) for a0, a1 in plain))

    per_kernel = {k: [] for k in KERNELS}
    step_ms = []
    for e in evs:
        for j, k in enumerate(KERNELS):
            per_kernel[k].append(e[j].elapsed_time(e[j + 1]))
        step_ms.append(e[0].elapsed_time(e[7]))
    ms = statistics.mean(step_ms)
    ms_max = _max_over_ranks(dist, ms)
    flop_step = 3 * 2.0 * M_ * N_ * K_
    value = world * flop_step / (ms_max * 1e-3) / 1e12

    # Each kernel is timed per launch inside a ~1.4 ms step, so the burst peak is the
    # denominator: dense FP8 = 2 x the measured dense bf16 burst (nominal 4.5 / 2.25 PF).
    fp8_peak = 2.0 * peaks["bf16_burst"]
    kern = {}
    for k, (kind, amount) in kernel_work().items():
        t = statistics.mean(per_kernel[k])
        if kind == "flop":
            a = amount / (t * 1e-3) / 1e12
            kern[k] = {"ms": round(t, 4), "tflops": round(a, 1), "frac_fp8_peak": round(a / fp8_peak, 3)}
        else:
            a = amount / (t * 1e-3) / 1e9
            kern[k] = {"ms": round(t, 4), "gbs": round(a, 1), "frac_hbm": round(a / peaks["hbm_gbs"], 3)}
    dom = max(KERNELS, key=lambda k: statistics.mean(per_kernel[k]))
    dkind, damount = kernel_work()[dom]
    dt = statistics.mean(per_kernel[dom])
    traffic = _load_traffic(dom)
    if dkind == "flop":
        ach = damount / (dt * 1e-3) / 1e12
        roof = {"kernel": dom, "bound": "tensor", "achieved": round(ach, 1), "peak": round(fp8_peak, 1),
                "unit": "TFLOP/s", "frac": round(ach / fp8_peak, 3), "traffic": traffic,
                "peak_source": f"{peaks['source']}: 2 x bf16 burst {peaks['bf16_burst']} TFLOP/s",
                "context": {"frac_of_2x_bf16_sustained": round(ach / (2.0 * peaks["bf16_sustained"]), 3),
                            "frac_of_fp8_mma_probe_4860": round(ach / FP8_MMA_PROBE_TFLOPS, 3)}}
    else:
        ach = damount / (dt * 1e-3) / 1e9
        roof = {"kernel": dom, "bound": "hbm", "achieved": round(ach, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(ach / peaks["hbm_gbs"], 3), "traffic": traffic, "peak_source": peaks["source"]}

    e2e = run_e2e(st, host, args, dist, world, flop_step)
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args.cpu_rows, args.cpu_cols, {k: v.view(torch.int16).numpy().view(np.uint16)
                                                          for k, v in host.items()})

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_max, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "e4m3 x e4m3 -> f32 (bf16 in/out)", "data": "synthetic (seeded N(0,1) X, "
            "N(0,0.02) W, N(0,1e-3) dY; no weights or datasets)",
            "config": {"workload": WORKLOAD, "M": M_, "N": N_, "K": K_, "uaq_s": UAQ_S,
                       "l2": "flushed before every step (256 MB device write outside the timed events)",
                       "parallelism": f"{world} independent replica(s)"},
            "kernels": kern, "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": st.launches_per_step * args.steps,
            "step_without_kernel_events": {
                "ms_per_step": round(plain_ms, 4),
                "value": round(flop_step / (plain_ms * 1e-3) / 1e12, 1),
                "note": "the same steps timed with a start and an end event only (informational; "
                        "value and kernels come from the per-kernel-event loop)"},
            "clocks": clk.summary(),
        }
        print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()


def kernel_source_hash(path: str, fn: str) -> str | None:
    """sha256 (16 hex digits) of the source text that defines kernel `fn`: the file
    from its start to the closing brace of `fn`'s body, so the helpers above it count
    and code added after it does not."""
    import hashlib
    import re
    text = open(path, encoding="utf-8").read()
    m = re.search(r"__global__[^;{]*?\b" + re.escape(fn) + r"\s*\(", text, flags=re.S)
    if not m:
        return None
    i = text.find("{", m.end())
    depth = 0
    for j in range(i, len(text)):
        if text[j] == "{":
            depth += 1
        elif text[j] == "}":
            depth -= 1
            if depth == 0:
                return hashlib.sha256(text[:j + 1].encode()).hexdigest()[:16]
    return None


def _load_traffic(kernel: str):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, or None
    when there is none or the kernel's source changed since it was captured."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        t = json.load(f)
    v = t.get(kernel)
    if not isinstance(v, dict):
        return None
    src = os.path.join(ROOT, v.get("source", ""))
    if not os.path.exists(src) or not v.get("kernel_fn"):
        return None
    sha = kernel_source_hash(src, v["kernel_fn"])
    return v.get("dram_bytes_per_launch") if sha is not None and sha == v.get("source_sha256_16") else None


def run_e2e(st: Step, host, args, dist, world, flop_step):
    """The same step through host buffers, every step's H2D of X, W, dY from pinned
    memory and D2H of Y, dX, dW into pinned memory inside the timed region.

    Steps are pipelined the way a training loop would run them: three streams
    (copy in, compute, copy out) and two device buffer sets, so step i+1's inputs
    arrive and step i-1's results leave while step i computes.  Events order each
    set's reuse: a set's inputs are rewritten only after its previous compute, its
    outputs only after their previous copy out."""
    dev = st.dev
    sets = [st, Step(dev, host)]
    pin = {k: v.pin_memory() for k, v in host.items()}
    outs = [{"y": torch.empty(st.y.shape, dtype=torch.bfloat16).pin_memory(),
             "dx": torch.empty(st.dx.shape, dtype=torch.bfloat16).pin_memory(),
             "dw": torch.empty(st.dw.shape, dtype=torch.bfloat16).pin_memory()} for _ in range(2)]
    s_in, s_comp, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("in", "comp", "out")}
    started = [False, False]

    def one(i):
        b = i % 2
        S, o = sets[b], outs[b]
        if started[b]:
            s_in.wait_event(ev["comp"][b])    # the set's previous compute has read its inputs
            s_comp.wait_event(ev["out"][b])   # ... and its previous results have left
        with torch.cuda.stream(s_in):
            S.x.copy_(pin["x"], non_blocking=True)
            S.w.copy_(pin["w"], non_blocking=True)
            S.dy.copy_(pin["dy"], non_blocking=True)
            ev["in"][b].record(s_in)
        s_comp.wait_event(ev["in"][b])
        S.run(s_comp.cuda_stream)
        ev["comp"][b].record(s_comp)
        s_out.wait_event(ev["comp"][b])
        with torch.cuda.stream(s_out):
            o["y"].copy_(S.y, non_blocking=True)
            o["dx"].copy_(S.dx, non_blocking=True)
            o["dw"].copy_(S.dw, non_blocking=True)
            ev["out"][b].record(s_out)
        started[b] = True

    for i in range(max(2, args.warmup // 2)):
        one(i)
    torch.cuda.synchronize()
    n = max(2, args.steps // 2)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    _barrier(dist)
    e0.record(s_in)
    for i in range(n):
        one(i)
    s_in.wait_stream(s_out)
    e1.record(s_in)
    torch.cuda.synchronize()
    ms = _max_over_ranks(dist, e0.elapsed_time(e1) / n)
    h2d = sum(v.numel() * v.element_size() for v in pin.values())
    d2h = sum(v.numel() * v.element_size() for v in outs[0].values())
    del sets[1]
    return {"value": round(world * flop_step / (ms * 1e-3) / 1e12, 1), "unit": "TFLOP/s", "ms_per_step": round(ms, 3),
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n,
            "pipelining": "copy in / compute / copy out on three streams, two device buffer sets"}


# ------------------------------------------------------------------ CPU ---

def cpu_baseline(rows: int, cols: int, data=None):
    """The oracle as it stands, on a bounded sample of the same workload: the
    sub-problem of `rows` tokens and `cols` output channels.  It folds and
    128x128-quantizes W[:cols], quantizes X[:rows] and dY[:rows, :cols]
    (1x128 and 128x1), and computes Y[:rows, :cols], the dX[:rows] contribution
    of those channels, and dW[:cols] over those tokens: 6 * rows * cols * K FLOP.
    Returns throughput in the GPU line's unit (GEMM TFLOP/s over the sample,
    quantization and dequantization time included)."""
    import oracle
    from fp8_block_scaled_quantize_gb300 import inputs as I

    oracle.build()
    K = K_
    rows = max(128, rows // 128 * 128)
    cols = max(128, cols // 128 * 128)
    d = data if data is not None else I.train_step_8b()
    x = np.ascontiguousarray(d["x"][:rows])
    w = np.ascontiguousarray(d["w"][:cols])
    dy = np.ascontiguousarray(d["dy"][:rows, :cols])
    s = np.full(K, UAQ_S, np.float32)

    def quantize():
        w_f, _ = oracle.uaq_fold(w, s)
        qw, sw, _ = oracle.quant_weight_128x128(w_f)
        return (qw, sw) + oracle.quant_rows_1x128(x) + oracle.quant_rows_1x128(dy) + \
            oracle.quant_cols_128x1(x) + oracle.quant_cols_128x1(dy)

    t0 = time.perf_counter()
    qw, sw, qx, sx, qdy, sdy, qxT, sxc, qdyT, sdyc = quantize()
    t1 = time.perf_counter()
    oracle.gemm_fprop(qx, sx, qw, sw)
    oracle.gemm_dgrad(qdy, sdy, qw, sw)
    oracle.gemm_wgrad(qdyT, sdyc, qxT, sxc)
    t2 = time.perf_counter()
    cores = oracle.num_threads()
    # the quantizers and fold once more on a single core (the GEMMs' BLAS is not limited)
    oracle.set_num_threads(1)
    try:
        t3 = time.perf_counter()
        quantize()
        t4 = time.perf_counter()
    finally:
        oracle.set_num_threads(cores)
    dt = t2 - t0
    flop = 6.0 * rows * cols * K
    qbytes = (4 + 3) * cols * K + B_DUAL * (rows * K + rows * cols)  # fold + weight quant + dual X, dY
    return {"value": round(flop / dt / 1e12, 6), "unit": "TFLOP/s", "cores": cores,
            "kind": "oracle", "seconds": round(dt, 3), "cpu_model": _cpu_model(),
            "quant_fold_seconds": round(t1 - t0, 3), "quant_fold_gbs": round(qbytes / (t1 - t0) / 1e9, 3),
            "quant_fold_gbs_1core": round(qbytes / (t4 - t3) / 1e9, 3),
            "gemm_seconds": round(t2 - t1, 3),
            "sample": f"sub-problem of {rows} tokens x {cols} output channels of the [{M_},{N_},{K_}] step: fold and "
                      f"128x128 quant of W[:{cols}], 1x128 + 128x1 quant of X[:{rows}] and dY[:{rows},:{cols}], "
                      f"FProp / DGrad / WGrad restricted to it (C with OpenMP + NumPy fp64; the GEMMs "
                      f"dequantize per block inside gemm_seconds)"}


def _cpu_model() -> str:
    """The host CPU's name as /proc/cpuinfo gives it (model name, else implementer/part)."""
    try:
        txt = open("/proc/cpuinfo").read()
    except OSError:
        return platform.machine()
    fields = {}
    for line in txt.splitlines():
        if ":" in line:
            k, v = line.split(":", 1)
            fields.setdefault(k.strip(), v.strip())
    if "model name" in fields:
        return fields["model name"]
    parts = [f"{k} {fields[k]}" for k in ("CPU implementer", "CPU part") if k in fields]
    return f"{platform.machine()} ({', '.join(parts)})" if parts else platform.machine()


def run_reference(args):
    """--impl reference: the oracle timed on the host cores (rank 0 only)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from fp8_block_scaled_quantize_gb300 import inputs as I
    data = I.train_step_8b()
    steps = []
    for i in range(args.warmup + args.steps):
        r = cpu_baseline(args.ref_rows, args.ref_cols, data)
        if i >= args.warmup:
            steps.append(r)
    val = statistics.mean(r["value"] for r in steps)
    sec = statistics.mean(r["seconds"] for r in steps)
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(sec * 1e3, 1), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)", "data": "synthetic",
            "config": {"workload": WORKLOAD, "M": M_, "N": N_, "K": K_, "sample_rows": args.ref_rows,
                       "sample_cols": args.ref_cols},
            "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": steps[-1]["cores"], "kind": "oracle",
                             "sample": steps[-1]["sample"], "cpu_model": steps[-1]["cpu_model"],
                             "quant_fold_gbs": steps[-1]["quant_fold_gbs"],
                             "quant_fold_gbs_1core": steps[-1]["quant_fold_gbs_1core"]},
            "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


# ----------------------------------------------------------------- sweep ---

SWEEP_DOC = """Per-configuration report (--sweep): every kernel of each workload timed on
its own (5 warm-ups, 20 repetitions, median; L2 flushed before each repetition,
then a short device-side wait so that the host's call overhead is not timed),
against its binding roofline; the HBM-bound kernels also streamed (launched back to
back over rotating input copies larger than 3x L2, per-launch time), as they run
inside a step.  For a GEMM that is max(FLOP / FP8 peak,
algorithmic bytes / HBM bandwidth): at small M the weight read dominates and the
kernel is bound by HBM, not by the tensor cores."""


def _dev_normal(gen, shape, std, outlier_frac=0.0, factor=1.0, t_frac=0.0, dev="cuda"):
    """Seeded device-side draw with the recipes of inputs.py (for timing only)."""
    x = torch.randn(shape, generator=gen, device=dev, dtype=torch.float32)
    if std != 1.0:
        x *= std
    K = shape[1]
    if outlier_frac:
        idx = torch.randperm(K, generator=gen, device=dev)[: int(np.ceil(outlier_frac * K))]
        x[:, idx] *= factor
    if t_frac:
        idx = torch.randperm(K, generator=gen, device=dev)[: int(np.ceil(t_frac * K))]
        # Student-t(3) = N / sqrt(chi2_3 / 3)
        z = torch.randn((shape[0], idx.numel()), generator=gen, device=dev)
        c = torch.randn((shape[0], idx.numel(), 3), generator=gen, device=dev).pow(2).sum(-1) / 3
        x[:, idx] = z / c.sqrt()
    return x.to(torch.bfloat16)


def _time_ms(fn, flush, reps=20, warm=5):
    """Median device time of fn over `reps` calls, L2 flushed before each.  A short
    device-side wait after the flush lets the host finish enqueueing fn (argument
    marshalling, output allocation) before the start event runs, so the host's
    call overhead stays out of the kernel's time."""
    for _ in range(warm):
        fn()
    ts = []
    for _ in range(reps):
        flush.zero_()
        torch.cuda._sleep(1_000_000)  # about 0.5 ms of device time
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    ts.sort()
    return ts[len(ts) // 2]


def run_sweep(args):
    from fp8_block_scaled_quantize_gb300 import rlq

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    rlq.lib()
    peaks = _peaks()
    bw = peaks["hbm_gbs"]
    fp8 = 2.0 * peaks["bf16_burst"]  # kernels are timed one at a time: burst peak
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    rows = []

    def emit(cfg, kernel, ms, nbytes=None, flop=None, ms_stream=None):
        r = {"sweep": True, "config": cfg, "kernel": kernel, "ms": round(ms, 4)}
        if flop is None:
            r["gbs"] = round(nbytes / (ms * 1e-3) / 1e9, 1)
            r["frac_hbm"] = round(r["gbs"] / bw, 3)
            r["bound"] = "hbm"
            if ms_stream is not None:
                r["ms_stream"] = round(ms_stream, 4)
                r["frac_stream"] = round(nbytes / (ms_stream * 1e-3) / 1e9 / bw, 3)
        else:
            r["tflops"] = round(flop / (ms * 1e-3) / 1e12, 1)
            t_roof = max(flop / (fp8 * 1e12), nbytes / (bw * 1e9)) * 1e3
            r["bound"] = "tensor" if flop / (fp8 * 1e12) >= nbytes / (bw * 1e9) else "hbm"
            r["frac_roofline"] = round(t_roof / ms, 3)
            r["frac_fp8_peak"] = round(r["tflops"] / fp8, 3)
        rows.append(r)
        print(json.dumps(r), flush=True)

    def streamed_ms(fn, srcs):
        """Per-launch device time of fn launched back to back over rotating copies of
        its inputs (srcs: the tensors fn takes), the copies together larger than 3x
        L2, so each launch reads from HBM without a flush in between; the launches
        are enqueued behind a device-side wait, so the host's call overhead is not
        timed.  The fixed cost of one event pair and one launch ramp is spread over
        the launches, as inside a step.  None for inputs under 16 MB (the host's
        launch rate would set the time)."""
        nb = sum(t.numel() * t.element_size() for t in srcs)
        if nb < (16 << 20):
            return None  # too small to stream from HBM without the host's launch rate binding
        n = max(2, -(-(400 << 20) // nb))
        sets = [srcs] + [[t.clone() for t in srcs] for _ in range(n - 1)]
        reps = max(8, n)
        for i in range(n):
            fn(*sets[i])
        ts = []
        for _ in range(5):
            torch.cuda._sleep(4_000_000)  # about 2 ms: the host enqueues all launches behind it
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for i in range(reps):
                fn(*sets[i % n])
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) / reps)
        del sets
        ts.sort()
        return ts[len(ts) // 2]

    def _splitk_ws(kind, M, N, K):
        """Workspace for the split-K plan of this GEMM, None when it runs one pass
        (the split rows are then not reported)."""
        nb = rlq.rlq_gemm_splitk_workspace_bytes(kind, M, N, K)
        return torch.empty(nb, dtype=torch.uint8, device=dev) if nb else None

    def gemm_bytes(Mr, Nc, L):
        return Mr * L + Nc * L + 2 * Mr * Nc + 4 * (Mr + Nc) * ((L + 127) // 128)

    def nvfp4_gemm_row(cfg, x, w):
        """NVFP4 weight-only GEMM (bf16 X, FP4 weights): bytes X + codes + block
        scales + bf16 Y; bound by HBM or by the bf16 tensor rate."""
        M, K = x.shape
        N = w.shape[0]
        q4, sb4, st4 = rlq.quant_nvfp4(w)
        y4 = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        nbytes = 2 * M * K + N * K // 2 + N * K // 16 + 2 * M * N
        flop = 2.0 * M * N * K
        ws = _splitk_ws(rlq.GEMM_NVFP4_WEIGHT_ONLY, M, N, K)
        variants = [("gemm_nvfp4_weight_only", lambda: rlq.gemm_nvfp4_weight_only(x, q4, sb4, st4, out=y4))]
        if ws is not None:
            variants.append(("gemm_nvfp4_weight_only_splitk",
                             lambda: rlq.gemm_nvfp4_weight_only(x, q4, sb4, st4, out=y4, split_k=True,
                                                                workspace=ws)))
        for name, fn in variants:
            ms = _time_ms(fn, flush)
            r = {"sweep": True, "config": cfg, "kernel": name, "ms": round(ms, 4),
                 "tflops": round(flop / (ms * 1e-3) / 1e12, 1), "gbs": round(nbytes / (ms * 1e-3) / 1e9, 1)}
            t_roof = max(flop / (peaks["bf16_burst"] * 1e12), nbytes / (bw * 1e9)) * 1e3
            r["bound"] = "tensor (bf16)" if flop / (peaks["bf16_burst"] * 1e12) >= nbytes / (bw * 1e9) else "hbm"
            r["frac_roofline"] = round(t_roof / ms, 3)
            rows.append(r)
            print(json.dumps(r), flush=True)
        del q4, sb4, st4, y4, ws

    def linear(cfg, x, w, dy=None, s=None, full=False, per_channel=False, norm=False, nvfp4=False):
        """Time the quantizers, fold and GEMMs of one linear layer (with
        ``per_channel`` also the per-token / per-channel quantizers and FProp)."""
        M, K = x.shape
        N = w.shape[0]
        if s is not None:
            st = torch.from_numpy(s).to(dev)
            inv = (1.0 / st).contiguous()
            wf, xf = w.clone(), x.clone()
            par = {}

            def fold(wt, xt):
                # alternate s and 1/s per tensor so repeated folds keep it stationary
                p_ = par.get(wt.data_ptr(), 0)
                rlq.uaq_fold_(wt, st if p_ == 0 else inv, xt)
                par[wt.data_ptr()] = p_ ^ 1
            emit(cfg, "uaq_fold", _time_ms(lambda: fold(wf, xf), flush), nbytes=4 * (N * K + M * K),
                 ms_stream=streamed_ms(fold, [wf, xf]))
            if per_channel:
                # AQN on a norm scale of K channels: read 2 + 4, write 2 bytes per channel
                gam = torch.ones(K, dtype=torch.bfloat16, device=dev)
                zz = torch.randn(K, generator=torch.Generator(device=dev).manual_seed(5), device=dev)
                emit(cfg, "aqn_perturb", _time_ms(lambda: rlq.aqn_perturb_(gam, zz, 1e-3), flush), nbytes=8 * K)
        emit(cfg, "quant_rows_x", _time_ms(lambda: rlq.quant_act_1x128(x), flush), nbytes=B_ROWS * M * K,
             ms_stream=streamed_ms(lambda t: rlq.quant_act_1x128(t), [x]))
        if norm:
            # RMSNorm of a hidden state of X's shape fused with the quantizer (x here
            # stands in for the hidden state): one read of h, the codes, the scales
            # and the per-row factors
            gam = torch.ones(K, dtype=torch.bfloat16, device=dev)
            emit(cfg, "rmsnorm_quant_rows_x", _time_ms(lambda: rlq.rmsnorm_quant_act_1x128(x, gam, 1e-5), flush),
                 nbytes=B_ROWS * M * K + 4 * M,
                 ms_stream=streamed_ms(lambda t: rlq.rmsnorm_quant_act_1x128(t, gam, 1e-5), [x]))
            emit(cfg, "rmsnorm_quant_dual_x",
                 _time_ms(lambda: rlq.rmsnorm_quant_act_1x128(x, gam, 1e-5, colwise=True), flush),
                 nbytes=B_DUAL * M * K + 4 * M,
                 ms_stream=streamed_ms(lambda t: rlq.rmsnorm_quant_act_1x128(t, gam, 1e-5, colwise=True), [x]))
        if full:
            emit(cfg, "quant_dual_x", _time_ms(lambda: rlq.quant_act_1x128(x, colwise=True), flush),
                 nbytes=B_DUAL * M * K, ms_stream=streamed_ms(lambda t: rlq.quant_act_1x128(t, colwise=True), [x]))
        emit(cfg, "quant_weight" + ("_t" if full else ""),
             _time_ms(lambda: rlq.quant_weight_128x128(w, transposed=full), flush),
             nbytes=(B_WEIGHT_T if full else B_WEIGHT) * N * K,
             ms_stream=streamed_ms(lambda t: rlq.quant_weight_128x128(t, transposed=full), [w]))
        if nvfp4:
            nvfp4_gemm_row(cfg, x, w)
        qx, sx, qxT, sxc = rlq.quant_act_1x128(x, colwise=full)
        qw, sw, qwT = rlq.quant_weight_128x128(w, transposed=full)
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        emit(cfg, "gemm_fprop", _time_ms(lambda: rlq.gemm_fprop(qx, sx, qw, sw, out=y), flush),
             nbytes=gemm_bytes(M, N, K), flop=2.0 * M * N * K)
        ws = _splitk_ws(rlq.GEMM_FPROP, M, N, K)
        if ws is not None:
            emit(cfg, "gemm_fprop_splitk",
                 _time_ms(lambda: rlq.gemm_fprop(qx, sx, qw, sw, out=y, split_k=True, workspace=ws), flush),
                 nbytes=gemm_bytes(M, N, K), flop=2.0 * M * N * K)
        if per_channel:
            # read 2 + write 1 bytes per element, the row scale and its K/128 copies
            emit(cfg, "quant_per_row_x", _time_ms(lambda: rlq.quant_per_row(x), flush),
                 nbytes=3 * M * K + 4 * M * (1 + K // 128), ms_stream=streamed_ms(lambda t: rlq.quant_per_row(t), [x]))
            emit(cfg, "quant_per_row_w", _time_ms(lambda: rlq.quant_per_row(w), flush),
                 nbytes=3 * N * K + 4 * N * (1 + K // 128), ms_stream=streamed_ms(lambda t: rlq.quant_per_row(t), [w]))
            # NVFP4 weights: read 2, write 0.5 (codes) + 1/16 (block scales) bytes per element
            emit(cfg, "quant_nvfp4_w", _time_ms(lambda: rlq.quant_nvfp4(w), flush), nbytes=2.5625 * N * K,
                 ms_stream=streamed_ms(lambda t: rlq.quant_nvfp4(t), [w]))
            pqx, _, psx = rlq.quant_per_row(x)
            pqw, _, psw = rlq.quant_per_row(w)
            emit(cfg, "gemm_fprop_per_channel",
                 _time_ms(lambda: rlq.gemm_fprop_per_channel(pqx, psx, pqw, psw, out=y), flush),
                 nbytes=gemm_bytes(M, N, K), flop=2.0 * M * N * K)
            ws = _splitk_ws(rlq.GEMM_FPROP, M, N, K)
            if ws is not None:
                emit(cfg, "gemm_fprop_per_channel_splitk",
                     _time_ms(lambda: rlq.gemm_fprop_per_channel(pqx, psx, pqw, psw, out=y, split_k=True,
                                                                 workspace=ws), flush),
                     nbytes=gemm_bytes(M, N, K), flop=2.0 * M * N * K)
            del pqx, pqw, psx, psw
        if full:
            emit(cfg, "quant_dual_dy", _time_ms(lambda: rlq.quant_act_1x128(dy, colwise=True), flush),
                 nbytes=B_DUAL * M * N, ms_stream=streamed_ms(lambda t: rlq.quant_act_1x128(t, colwise=True), [dy]))
            qdy, sdy, qdyT, sdyc = rlq.quant_act_1x128(dy, colwise=True)
            dx = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
            dw = torch.empty((N, K), dtype=torch.bfloat16, device=dev)
            emit(cfg, "gemm_dgrad", _time_ms(lambda: rlq.gemm_dgrad(qdy, sdy, qwT, sw, out=dx), flush),
                 nbytes=gemm_bytes(M, K, N), flop=2.0 * M * N * K)
            emit(cfg, "gemm_dgrad_mn",
                 _time_ms(lambda: rlq.gemm_dgrad(qdy, sdy, qw, sw, transposed=False, out=dx), flush),
                 nbytes=gemm_bytes(M, K, N), flop=2.0 * M * N * K)
            ws = _splitk_ws(rlq.GEMM_DGRAD, M, N, K)
            if ws is not None:
                emit(cfg, "gemm_dgrad_splitk",
                     _time_ms(lambda: rlq.gemm_dgrad(qdy, sdy, qwT, sw, out=dx, split_k=True, workspace=ws), flush),
                     nbytes=gemm_bytes(M, K, N), flop=2.0 * M * N * K)
            emit(cfg, "gemm_wgrad", _time_ms(lambda: rlq.gemm_wgrad(qdyT, sdyc, qxT, sxc, out=dw), flush),
                 nbytes=gemm_bytes(N, K, M), flop=2.0 * M * N * K)
            if cfg.startswith("train_step_8b"):
                emit(cfg, "quant_nvfp4_w", _time_ms(lambda: rlq.quant_nvfp4(w), flush), nbytes=2.5625 * N * K,
                     ms_stream=streamed_ms(lambda t: rlq.quant_nvfp4(t), [w]))
                # fp32 accumulation (micro-batches): the operands, and the fp32 gradient
                # read and written by the epilogue (no bf16 output)
                acc = torch.zeros((N, K), dtype=torch.float32, device=dev)
                emit(cfg, "gemm_wgrad_accumulate",
                     _time_ms(lambda: rlq.gemm_wgrad_accumulate_(acc, qdyT, sdyc, qxT, sxc), flush),
                     nbytes=gemm_bytes(N, K, M) - 2 * N * K + 8 * N * K, flop=2.0 * M * N * K)
                del acc
            ws = _splitk_ws(rlq.GEMM_WGRAD, M, N, K)
            if ws is not None:
                emit(cfg, "gemm_wgrad_splitk",
                     _time_ms(lambda: rlq.gemm_wgrad(qdyT, sdyc, qxT, sxc, out=dw, split_k=True, workspace=ws),
                              flush),
                     nbytes=gemm_bytes(N, K, M), flop=2.0 * M * N * K)
        rlq.check()

    from fp8_block_scaled_quantize_gb300 import inputs as I
    gen = torch.Generator(device=dev)
    # tiny single linear, fold with s = 4
    d = I.tiny_single_linear()
    linear("tiny_single_linear M=128 N=256 K=256", I.to_torch(d["x"], dev), I.to_torch(d["w"], dev), s=d["s"])
    # decode up-projection, 8B shapes
    gen.manual_seed(1)
    linear("decode_upproj_8b M=256 N=14336 K=4096", _dev_normal(gen, (256, 4096), 1.0, 0.01, 20.0),
           _dev_normal(gen, (14336, 4096), 0.02), nvfp4=True)
    # 8B training step
    gen.manual_seed(2)
    linear("train_step_8b M=8192 N=14336 K=4096", _dev_normal(gen, (8192, 4096), 1.0),
           _dev_normal(gen, (14336, 4096), 0.02), dy=_dev_normal(gen, (8192, 14336), 1e-3), full=True, norm=True)
    # Qwen2.5-7B layer set: fold + quant + FProp
    gen.manual_seed(3)
    for which, (N, K) in (("gate_up", (18944, 3584)), ("down", (3584, 18944))):
        w = _dev_normal(gen, (N, K), 0.02)
        s = np.random.default_rng(3).uniform(1.5, 4.0, K).astype(np.float32)
        for M in I.QWEN7B_M:
            linear(f"qwen7b_{which} M={M} N={N} K={K}", _dev_normal(gen, (M, K), 1.0, t_frac=0.01), w, s=s,
                   per_channel=True, norm=(which == "gate_up"), nvfp4=True)
        del w
    # 32B sweep: all three passes per M
    gen.manual_seed(4)
    for orient, (N, K) in (("up", (27648, 5120)), ("down", (5120, 27648))):
        w = _dev_normal(gen, (N, K), 0.015)
        for M in I.SWEEP_32B_M:
            x = _dev_normal(gen, (M, K), 1.0, 0.005, 50.0)
            dy = _dev_normal(gen, (M, N), 1e-3)
            linear(f"sweep_32b_{orient} M={M} N={N} K={K}", x, w, dy=dy, full=True, norm=(orient == "up"),
                   nvfp4=(M <= 1024))
            del x, dy
            torch.cuda.empty_cache()
        del w
    if args.sweep_md:
        with open(args.sweep_md, "w") as f:
            f.write("| Config | Kernel | ms | TFLOP/s | GB/s | bound | fraction of roofline | streamed ms (fraction) |\n"
                    "|---|---|---:|---:|---:|---|---:|---:|\n")
            for r in rows:
                frac = r.get("frac_roofline", r.get("frac_hbm"))
                stream = f"{r['ms_stream']} ({r['frac_stream']})" if "ms_stream" in r else ""
                f.write(f"| {r['config']} | {r['kernel']} | {r['ms']} | {r.get('tflops', '')} | {r.get('gbs', '')} | "
                        f"{r['bound']} | {frac} | {stream} |\n")


# ------------------------------------------------------------- one kernel ---

CASE_DOC = """Run one kernel of the path on one shape --case-reps times (after 2 warm-up
calls), for profiler captures of a small case: gemm_fprop, gemm_dgrad,
gemm_dgrad_mn (untransposed weight codes), gemm_wgrad (optionally --split-k), gemm_wgrad_accumulate,
gemm_fprop_per_channel, gemm_nvfp4, quant_rows, quant_dual,
rmsnorm_quant, rmsnorm_quant_dual, quant_weight (with the transposed copy),
quant_weight_nt (without), quant_nvfp4, uaq_fold.  Prints the
median CUDA-event time; no JSON line."""


def run_case(args):
    from fp8_block_scaled_quantize_gb300 import rlq

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    rlq.lib()
    M, N, K = args.case_m, args.case_n, args.case_k
    gen = torch.Generator(device=dev)
    gen.manual_seed(7)
    x = _dev_normal(gen, (M, K), 1.0)
    w = _dev_normal(gen, (N, K), 0.02)
    name = args.case
    if name == "gemm_fprop":
        qx, sx, _, _ = rlq.quant_act_1x128(x)
        qw, sw, _ = rlq.quant_weight_128x128(w)
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        fn = lambda: rlq.gemm_fprop(qx, sx, qw, sw, out=y, split_k=args.split_k)
    elif name == "gemm_nvfp4":
        q4, sb4, st4 = rlq.quant_nvfp4(w)
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        fn = lambda: rlq.gemm_nvfp4_weight_only(x, q4, sb4, st4, out=y, split_k=args.split_k)
    elif name == "gemm_fprop_per_channel":
        qx, _, sx = rlq.quant_per_row(x)
        qw, _, sw = rlq.quant_per_row(w)
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        fn = lambda: rlq.gemm_fprop_per_channel(qx, sx, qw, sw, out=y, split_k=args.split_k)
    elif name == "gemm_wgrad_accumulate":
        dy = _dev_normal(gen, (M, N), 1e-3)
        _, _, qxT, sxc = rlq.quant_act_1x128(x, colwise=True)
        _, _, qdyT, sdyc = rlq.quant_act_1x128(dy, colwise=True)
        acc = torch.zeros((N, K), dtype=torch.float32, device=dev)
        fn = lambda: rlq.gemm_wgrad_accumulate_(acc, qdyT, sdyc, qxT, sxc)
    elif name in ("gemm_dgrad", "gemm_dgrad_mn", "gemm_wgrad"):
        dy = _dev_normal(gen, (M, N), 1e-3)
        qw, sw, qwT = rlq.quant_weight_128x128(w, transposed=True)
        qx, sx, qxT, sxc = rlq.quant_act_1x128(x, colwise=True)
        qdy, sdy, qdyT, sdyc = rlq.quant_act_1x128(dy, colwise=True)
        if name == "gemm_dgrad":
            dx = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
            fn = lambda: rlq.gemm_dgrad(qdy, sdy, qwT, sw, out=dx, split_k=args.split_k)
        elif name == "gemm_dgrad_mn":  # the FProp weight codes read MN-major, no transposed copy
            dx = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
            fn = lambda: rlq.gemm_dgrad(qdy, sdy, qw, sw, transposed=False, out=dx, split_k=args.split_k)
        else:
            dw = torch.empty((N, K), dtype=torch.bfloat16, device=dev)
            fn = lambda: rlq.gemm_wgrad(qdyT, sdyc, qxT, sxc, out=dw, split_k=args.split_k)
    elif name == "quant_rows":
        fn = lambda: rlq.quant_act_1x128(x)
    elif name in ("rmsnorm_quant", "rmsnorm_quant_dual"):
        gam = torch.ones(K, dtype=torch.bfloat16, device=dev)
        fn = lambda: rlq.rmsnorm_quant_act_1x128(x, gam, 1e-5, colwise=name.endswith("dual"))
    elif name == "quant_dual":
        fn = lambda: rlq.quant_act_1x128(x, colwise=True)
    elif name == "quant_weight":
        fn = lambda: rlq.quant_weight_128x128(w, transposed=True)
    elif name == "quant_nvfp4":
        fn = lambda: rlq.quant_nvfp4(w)
    elif name == "quant_weight_nt":  # without the transposed copy (the bench step's form)
        fn = lambda: rlq.quant_weight_128x128(w)
    elif name == "uaq_fold":
        s = torch.full((K,), 1.5, dtype=torch.float32, device=dev)
        fn = lambda: rlq.uaq_fold_(w, s, x)
    else:
        raise SystemExit(f"unknown --case {name}")
    for _ in range(2):
        fn()
    ts = []
    for _ in range(args.case_reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    # back to back: the host enqueues ahead of the GPU, so host-side overhead of the
    # helpers (output allocation, argument marshalling) drops out; inputs below the
    # L2 size stay warm between calls
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.case_reps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    b2b = e0.elapsed_time(e1) / args.case_reps
    rlq.check()
    ts.sort()
    print(f"{name} M={M} N={N} K={K} split_k={args.split_k}: median {ts[len(ts) // 2] * 1e3:.1f} us, "
          f"back-to-back {b2b * 1e3:.1f} us")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-rows", type=int, default=1024)
    ap.add_argument("--cpu-cols", type=int, default=14336)
    ap.add_argument("--ref-rows", type=int, default=256)
    ap.add_argument("--ref-cols", type=int, default=1024)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sweep", action="store_true", help=SWEEP_DOC)
    ap.add_argument("--sweep-md", default=None, help="also write the sweep as a markdown table to this path")
    ap.add_argument("--case", default=None, help=CASE_DOC)
    ap.add_argument("--case-m", type=int, default=8192)
    ap.add_argument("--case-n", type=int, default=8192)
    ap.add_argument("--case-k", type=int, default=4096)
    ap.add_argument("--case-reps", type=int, default=3)
    ap.add_argument("--split-k", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.case:
        run_case(args)
    elif args.sweep:
        run_sweep(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
