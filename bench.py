"""Benchmark of the context-parallel attention path on B300.

One step = the ring-emulation hot path on the video-DiT workload (B=1, H=16, S=44,160, D=128,
bf16): attn_fwd_chunked over P=8 KV chunks, then attn_lse_merge of the eight partials.  The
metric is attention TFLOP/s = 4*B*H*Sq*Skv*D per step / step time.  The roofline object holds
the attention kernel alone against the measured burst dense-bf16 peak (with the sustained figure
and the clock-derived nominal at the SM clock sampled during the timed region as notes) and its
DRAM traffic from a full-size ncu capture.  Extra legs: the merge (L2 flushed) and Ulysses layout
kernels in GB/s against HBM, the Ulysses, ring, e4m3 and short-chunk (image, P = 8) paths, an
end-to-end number through the same API with host buffers, and the CPU oracle timed on a bounded
sample.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]
                    [--no-cpu-baseline] [--no-e2e]
    python bench.py --profile attn|merge|layout|ulysses|fp8   # one kernel, reduced case, for ncu
    python bench.py --probe                         # tensor-core calibration probes

Prints one JSON line (rank 0).  With torchrun each rank runs an independent replica of the same
workload on its own GPU (the path needs no exchange on one box); ``value`` is the sum over ranks
divided by the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from context_math_non_b300.inputs import WORKLOADS, draw_qkv  # noqa: E402

WORKLOAD = WORKLOADS["video"]
P_CHUNKS = 8
METRIC = "attention fwd TFLOP/s (4*B*H*Sq*Skv*D per step; KV in P=8 chunks + LSE merge)"
UNIT = "TFLOP/s"
CONFIG = {
    "workload": "video-DiT long sequence: B=1 H=16 S=44160 D=128 bf16 N(0,1), non-causal, "
                "KV split into P=8 chunks (per-chunk O + LSE), then LSE merge",
    "B": 1, "H": 16, "S": 44160, "D": 128, "P": P_CHUNKS,
    "l2": "step: every input is larger than L2 (Q/K/V 181 MB each, partials 1.45 GB); the "
          "merge and layout legs are timed apart with an L2 flush / rotated buffers",
    "parallelism": "replicas",
}
ATTN_SOURCES = ["context_math_non_b300/csrc/attn_fwd_sm103.cu",
                "context_math_non_b300/csrc/ptx_sm103.cuh"]


def _dist():
    if "RANK" in os.environ and "WORLD_SIZE" in os.environ and int(os.environ["WORLD_SIZE"]) > 1:
        return int(os.environ["RANK"]), int(os.environ["WORLD_SIZE"]), int(
            os.environ.get("LOCAL_RANK", 0))
    return 0, 1, 0


def reduce_max(value: float, device) -> float:
    """Max of `value` over all ranks (the slowest rank's time); identity on one process."""
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return value
    if torch.distributed.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def aggregate_tflops(world: int, flops_per_step: float, steps: int, ms: float) -> float:
    """Whole-job throughput: every rank does flops_per_step per step (weak scaling)."""
    return world * flops_per_step * steps / (ms * 1e-3) / 1e12


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16": d["bf16_tflops"],
                "bf16_sustained": d["bf16_tflops_sustained"], "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6400.0, "bf16": 1800.0, "bf16_sustained": 1400.0, "source": "fallback"}


def _src_hash() -> str:
    """Hash of the attention kernel's code (comments and layout stripped), so the ncu traffic
    recorded for one build is only reused for code that is byte-for-byte the same."""
    h = hashlib.sha256()
    for p in ATTN_SOURCES:
        with open(os.path.join(ROOT, p)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def _traffic():
    """DRAM bytes (read + write) of one full-size attention launch, from the committed ncu
    capture of exactly that launch, if it was taken on the current kernel source (else None)."""
    try:
        with open(os.path.join(ROOT, "profiles", "attn_fwd_traffic.json")) as f:
            d = json.load(f)
        if d.get("kernel_source_sha") == _src_hash():
            return d["dram_bytes_read"] + d["dram_bytes_write"]
    except (OSError, KeyError, ValueError):
        pass
    return None


class ClockSampler:
    """Samples SM clock and throttle reasons with nvidia-smi while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.skip = 0

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            t0 = time.time()
            while not self.lines and time.time() - t0 < 3.0:   # sampler running before timing
                time.sleep(0.02)
            self.skip = len(self.lines)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=5)

    def summary(self):
        sm, mx = [], None
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines[self.skip:]:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) != 6:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, val in zip(names, parts[2:]):
                if val.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "samples": len(sm),
                "reasons": sorted(reasons)}


# ----------------------------------------------------------------------------- native arm

def run_native(args, rank, world, local_rank):
    from context_math_non_b300 import cpattn

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    w = WORKLOAD
    q, k, v = draw_qkv(w)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    B, H, S, D = w.B, w.H, w.S, w.D
    op = torch.empty((P_CHUNKS, B, H, S, D), dtype=w.dtype, device=dev)
    lp = torch.empty((P_CHUNKS, B, H, S), dtype=torch.float32, device=dev)
    o = torch.empty((B, H, S, D), dtype=w.dtype, device=dev)
    lse = torch.empty((B, H, S), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    flops = w.attention_flops()
    merge_bytes = (P_CHUNKS + 1) * B * H * S * (D * 2 + 4)

    def step():
        cpattn.attn_fwd_chunked(qd, kd, vd, P_CHUNKS, op, lp, stream=stream)
        cpattn.attn_lse_merge(op, lp, o, lse, stream=stream)

    for _ in range(args.warmup):
        step()
    st = cpattn.attn_device_status(stream)
    if st != cpattn.ATTN_OK:
        raise RuntimeError(f"device status after warm-up: {cpattn.attn_status_string(st)}")

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local_rank) as clocks:
        t_start.record(stream)
        for i in range(args.steps):
            ev[i][0].record(stream)
            cpattn.attn_fwd_chunked(qd, kd, vd, P_CHUNKS, op, lp, stream=stream)
            ev[i][1].record(stream)
            cpattn.attn_lse_merge(op, lp, o, lse, stream=stream)
            ev[i][2].record(stream)
        t_end.record(stream)
        torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    total_ms = t_start.elapsed_time(t_end)
    # the timed step's merged output for its first query rows, checked by the CPU-baseline leg
    check_rows = min(w.S, PARITY_ROWS)
    gpu_head = (o[:, :, :check_rows].cpu(), lse[:, :, :check_rows].cpu())
    attn_ms = [e[0].elapsed_time(e[1]) for e in ev]
    merge_ms = [e[1].elapsed_time(e[2]) for e in ev]
    st = cpattn.attn_device_status(stream)
    if st != cpattn.ATTN_OK:
        raise RuntimeError(f"device status after timing: {cpattn.attn_status_string(st)}")

    total_ms = reduce_max(total_ms, dev)
    ms_per_step = total_ms / args.steps
    value = aggregate_tflops(world, flops, args.steps, total_ms)

    peaks = _peaks()
    attn_avg = sum(attn_ms) / len(attn_ms)
    achieved = flops / (attn_avg * 1e-3) / 1e12
    merge_avg = sum(merge_ms) / len(merge_ms)
    roofline = {
        "kernel": "attn_fwd_kernel<128,bf16> (attn_fwd_chunked, P=8)",
        "bound": "tensor", "achieved": round(achieved, 2),
        "peak": peaks["bf16"], "unit": "TFLOP/s",
        "frac": round(achieved / peaks["bf16"], 4),
        "peak_note": f"{peaks['source']} burst dense bf16 (the timed region lasts well under a "
                     f"second); of {peaks['source']} sustained {peaks['bf16_sustained']} (taken "
                     f"over seconds at a lower clock): {achieved / peaks['bf16_sustained']:.4f}",
        "avg_launch_ms": round(attn_avg, 4),
        "traffic": _traffic(),
        "algorithmic_flops_per_launch": flops,
    }
    legs = {
        "lse_merge_in_step": {"avg_ms": round(merge_avg, 4), "bytes": merge_bytes,
                              "note": "inside the timed step, right after the chunked kernel "
                                      "wrote the partials (part of them may still be in L2)"},
    }
    legs.update(_merge_leg(cpattn, op, lp, o, lse, dev, stream, peaks, merge_bytes))
    legs.update(_layout_leg(cpattn, dev, stream, peaks))
    legs.update(_ulysses_leg(cpattn, dev, stream))
    legs.update(_ring_leg(cpattn, qd, kd, vd, o, lse, dev, stream, flops, ms_per_step))
    legs.update(_fp8_leg(cpattn, qd, kd, vd, o, lse, dev, stream, flops, peaks))
    legs.update(_image_leg(cpattn, dev, stream))
    clk = clocks.summary()
    # clock-derived nominal: SMs x 8192 dense bf16 flop per clock (one M128 N256 K16 MMA per
    # 64 clocks) at the median SM clock seen during the timed region, and at the maximum clock
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    if clk is not None:
        nominal = sms * 8192 * clk["sm_mhz"] * 1e6 / 1e12
        roofline["clock_nominal"] = {
            "peak_at_median_clock": round(nominal, 1),
            "frac": round(achieved / nominal, 4),
            "peak_at_max_clock": round(sms * 8192 * clk["sm_max_mhz"] * 1e6 / 1e12, 1)}

    e2e = None
    if not args.no_e2e:
        e2e = _e2e_leg(cpattn, q, k, v, dev, stream, args, flops, world)
    del op, lp, qd, kd, vd
    torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(q, k, v, budget_s=args.cpu_seconds, gpu_head=gpu_head)
        if not cpu["parity"]["ok"]:
            raise RuntimeError(f"the timed step's output fails the oracle check: {cpu['parity']}")

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic: seeded N(0,1) bf16 draws of the video-DiT shape",
        "config": CONFIG, "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": 2 * args.steps, "clocks": clk, "legs": legs,
    }
    return line


NOMINAL_HBM_GBS = 8000.0   # the nominal B300 HBM3e bandwidth the merge and layout are held to


def _merge_leg(cpattn, op, lp, o, lse, dev, stream, peaks, nbytes, iters=10):
    """attn_lse_merge alone on the video partials (1653 MB per call): before every timed launch a
    512 MB buffer is written, which evicts the 126 MB L2, so every partial comes from DRAM."""
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    cpattn.attn_lse_merge(op, lp, o, lse, stream=stream)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(iters)]
    for i in range(iters):
        flush.fill_(i & 0xFF)
        evs[i][0].record(stream)
        cpattn.attn_lse_merge(op, lp, o, lse, stream=stream)
        evs[i][1].record(stream)
    torch.cuda.synchronize(dev)
    ms = statistics.median(a.elapsed_time(b) for a, b in evs)
    gbs = nbytes / (ms * 1e-3) / 1e9
    del flush
    return {"lse_merge": {"median_ms": round(ms, 4), "bytes": nbytes, "GB/s": round(gbs, 1),
                          "frac_of_hbm": round(gbs / peaks["hbm_gbs"], 4),
                          "frac_of_nominal_8TBs": round(gbs / NOMINAL_HBM_GBS, 4),
                          "l2": "flushed (512 MB write) before every timed launch"}}


def _layout_leg(cpattn, dev, stream, peaks, iters=10):
    """Ulysses seq2head on the Ulysses workload shape ([8][2][2048][32][64] fp16, 134 MB):
    the buffers are rotated over 4 sets (1.07 GB) so no iteration reads from L2."""
    w = WORKLOADS["ulysses"]
    P, B, S, H, D = w.P[0], w.B, w.S, w.H, w.D
    nbytes = P * B * (S // P) * H * D * 2
    sets = [(torch.empty((P, B, S // P, H, D), dtype=torch.float16, device=dev).normal_(),
             torch.empty((P, B, H // P, S, D), dtype=torch.float16, device=dev))
            for _ in range(4)]
    for x, y in sets:
        cpattn.cp_layout_seq2head(x, y, stream=stream)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(iters)]
    for i in range(iters):
        x, y = sets[i % 4]
        evs[i][0].record(stream)
        cpattn.cp_layout_seq2head(x, y, stream=stream)
        evs[i][1].record(stream)
    torch.cuda.synchronize(dev)
    ms = statistics.median(a.elapsed_time(b) for a, b in evs)
    gbs = 2 * nbytes / (ms * 1e-3) / 1e9
    del sets
    return {"cp_layout_seq2head": {"median_ms": round(ms, 4), "bytes": 2 * nbytes,
                                   "GB/s": round(gbs, 1),
                                   "frac_of_hbm": round(gbs / peaks["hbm_gbs"], 4),
                                   "frac_of_nominal_8TBs": round(gbs / NOMINAL_HBM_GBS, 4),
                                   "l2": "4 rotated buffer sets (1.07 GB)"}}


def _e2e_leg(cpattn, q, k, v, dev, stream, args, flops, world):
    """Same step through the same API, with every step's Q/K/V copied from pinned host memory and
    its merged O and LSE copied back to pinned host memory inside the timed region.  The copies
    run on their own streams, double-buffered, so step i's compute overlaps the host-to-device
    copy of step i+1 and the device-to-host copy of step i-1 (what a serving loop would do)."""
    w = WORKLOAD
    hq, hk, hv = (t.pin_memory() for t in (q, k, v))
    din = [[torch.empty_like(t, device=dev) for t in (q, k, v)] for _ in range(2)]
    op = torch.empty((P_CHUNKS, w.B, w.H, w.S, w.D), dtype=w.dtype, device=dev)
    lp = torch.empty((P_CHUNKS, w.B, w.H, w.S), dtype=torch.float32, device=dev)
    dout = [(torch.empty((w.B, w.H, w.S, w.D), dtype=w.dtype, device=dev),
             torch.empty((w.B, w.H, w.S), dtype=torch.float32, device=dev)) for _ in range(2)]
    hout = [(torch.empty(dout[0][0].shape, dtype=w.dtype).pin_memory(),
             torch.empty(dout[0][1].shape, dtype=torch.float32).pin_memory()) for _ in range(2)]
    s_in = torch.cuda.Stream(dev)
    s_out = torch.cuda.Stream(dev)
    s_cmp = stream
    ev = lambda: torch.cuda.Event()
    in_ready = [ev(), ev()]
    in_free = [ev(), ev()]
    cmp_done = [ev(), ev()]
    out_free = [ev(), ev()]
    for e in in_free + out_free:
        e.record(s_cmp)

    def step(i):
        b = i % 2
        s_in.wait_event(in_free[b])
        with torch.cuda.stream(s_in):
            for dst, src in zip(din[b], (hq, hk, hv)):
                dst.copy_(src, non_blocking=True)
        in_ready[b].record(s_in)
        s_cmp.wait_event(in_ready[b])
        s_cmp.wait_event(out_free[b])
        dq, dk, dv = din[b]
        o, lse = dout[b]
        cpattn.attn_fwd_chunked(dq, dk, dv, P_CHUNKS, op, lp, stream=s_cmp)
        cpattn.attn_lse_merge(op, lp, o, lse, stream=s_cmp)
        in_free[b].record(s_cmp)
        cmp_done[b].record(s_cmp)
        s_out.wait_event(cmp_done[b])
        with torch.cuda.stream(s_out):
            hout[b][0].copy_(o, non_blocking=True)
            hout[b][1].copy_(lse, non_blocking=True)
        out_free[b].record(s_out)

    for i in range(max(1, args.warmup)):
        step(i)
    torch.cuda.synchronize(dev)
    # as many steps as the device-timed loop; the first step's upload and the last step's
    # download are inside the timed region and not overlapped (pipeline fill and drain)
    steps = max(2, args.steps)
    if world > 1:
        torch.distributed.barrier()
    a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(s_in)
    for i in range(steps):
        step(i)
    s_in.wait_stream(s_out)
    b_.record(s_in)
    torch.cuda.synchronize(dev)
    ms = reduce_max(a.elapsed_time(b_), dev)
    h2d = sum(t.numel() * t.element_size() for t in (q, k, v))
    d2h = hout[0][0].numel() * hout[0][0].element_size() + hout[0][1].numel() * 4
    return {"value": round(aggregate_tflops(world, flops, steps, ms), 2), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "ms_per_step": round(ms / steps, 3),
            "overlap": "double-buffered: H2D of step i+1 and D2H of step i-1 overlap step i"}


# ----------------------------------------------------------------------------- CPU oracle

def _oracle_sample(q, k, v, rows_per_head: int, heads: int):
    """Oracle chunked attention (P=8) + merge for the first rows of the first heads."""
    import oracle
    qs = q[:, :heads, :rows_per_head]
    op, lp = oracle.attention_chunked(qs, k[:, :heads], v[:, :heads], P_CHUNKS)
    return oracle.lse_merge(op, lp)


def _blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [d["num_threads"] for d in threadpool_info() if d.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:  # noqa: BLE001 - informational only
        pass
    return os.cpu_count() or 1


PARITY_ROWS = 4096   # first query rows of every head copied back for the check


def _parity(o_ref, lse_ref, gpu_head):
    """The GPU step's merged O / LSE on the sampled rows against the oracle's: max and mean
    |dO| and max |dLSE| with the bf16 attention bounds (1e-2 beyond half a bf16 spacing of the
    exact value, 1e-3, 1e-3)."""
    o_g, l_g = (t.double().numpy() for t in gpu_head)
    n = min(o_ref.shape[-2], o_g.shape[-2])
    o_r, l_r = o_ref[..., :n, :], lse_ref[..., :n]
    o_g, l_g = o_g[..., :n, :], l_g[..., :n]
    err = np.abs(o_g - o_r)
    half = np.exp2(np.floor(np.log2(np.maximum(np.abs(o_r), 2.0 ** -126))) - 8)
    out = {"rows_per_head": int(n), "max_abs": float(err.max()), "mean_abs": float(err.mean()),
           "lse_max_abs": float(np.abs(l_g - l_r).max())}
    out["ok"] = bool((err - half).max() <= 1e-2 and out["mean_abs"] <= 1e-3 and
                     out["lse_max_abs"] <= 1e-3)
    return out


def cpu_baseline(q, k, v, budget_s: float = 15.0, gpu_head=None):
    """The float64 oracle, as it stands, timed on this host on a bounded sample of the same
    workload: R query rows of every head through chunked attention (P=8) and the merge.  With
    gpu_head (the timed step's O and LSE for the first rows of every head) the same oracle
    output also checks the GPU result on those rows."""
    w = WORKLOAD
    _oracle_sample(q, k, v, 16, 1)                  # warm BLAS and the allocator
    rows = 32
    while True:                                     # calibrate on one head
        t0 = time.perf_counter()
        _oracle_sample(q, k, v, rows, 1)
        t_cal = time.perf_counter() - t0
        if t_cal >= 0.05 * budget_s or rows >= w.S:
            break
        rows = min(w.S, rows * 2)
    per_row = t_cal / rows
    rows = int(max(16, min(w.S, budget_s / per_row / w.H)))
    t0 = time.perf_counter()
    o_ref, lse_ref = _oracle_sample(q, k, v, rows, w.H)
    dt = time.perf_counter() - t0
    flops = 4.0 * w.B * w.H * rows * w.S * w.D
    return {"value": round(flops / dt / 1e12, 6), "unit": UNIT, "cores": _blas_threads(),
            "parity": None if gpu_head is None else _parity(o_ref, lse_ref, gpu_head),
            "kind": "oracle", "seconds": round(dt, 2),
            "extrapolated_full_seconds": round(dt * w.S / rows, 1),
            "sample": f"first {rows} query rows of each of the {w.H} heads (of {w.S}), full KV, "
                      f"P=8 chunks + merge, float64 numpy"}


def run_reference(args):
    """Reference arm: the CPU oracle as it stands, one bounded sample per step."""
    w = WORKLOAD
    q, k, v = draw_qkv(w)
    rows = args.ref_rows
    for _ in range(args.warmup):
        _oracle_sample(q, k, v, rows, w.H)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _oracle_sample(q, k, v, rows, w.H)
    dt = time.perf_counter() - t0
    flops = 4.0 * w.B * w.H * rows * w.S * w.D * args.steps
    value = flops / dt / 1e12
    sample = (f"each step: first {rows} query rows of each of the {w.H} heads (of {w.S}), full KV,"
              f" P=8 chunks + merge, float64 numpy")
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT,
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": CONFIG,
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": _blas_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def _ring_leg(cpattn, qd, kd, vd, o, lse, dev, stream, flops, step_ms, iters=6):
    """The same video problem through attn_fwd_ring (P = 8 ring steps, merge fused into the
    kernel: no partial outputs in HBM, no merge launch) and through the chunked step + merge,
    launched alternately so both see the same clocks and power state."""
    w = WORKLOAD
    op = torch.empty((P_CHUNKS, w.B, w.H, w.S, w.D), dtype=w.dtype, device=dev)
    lp = torch.empty((P_CHUNKS, w.B, w.H, w.S), dtype=torch.float32, device=dev)

    def ring():
        cpattn.attn_fwd_ring(qd, kd, vd, P_CHUNKS, o, lse, stream=stream)

    def chunked():
        cpattn.attn_fwd_chunked(qd, kd, vd, P_CHUNKS, op, lp, stream=stream)
        cpattn.attn_lse_merge(op, lp, o, lse, stream=stream)

    ms = _interleaved({"ring": ring, "chunked_plus_merge": chunked}, dev, stream, iters)
    st = cpattn.attn_device_status(stream)
    if st != cpattn.ATTN_OK:
        raise RuntimeError(f"device status after ring leg: {cpattn.attn_status_string(st)}")
    del op, lp
    return {"attn_fwd_ring_P8": {"median_ms": round(ms["ring"], 4),
                                 "TFLOP/s": round(flops / (ms["ring"] * 1e-3) / 1e12, 1),
                                 "chunked_plus_merge_median_ms":
                                     round(ms["chunked_plus_merge"], 4),
                                 "order": "launched alternately with the chunked step"}}


def _image_leg(cpattn, dev, stream, iters=15):
    """The image-DiT shape (B=1 H=24 S=4608 D=128 bf16) with KV in P = 8 chunks of 576 keys
    (4.5 tiles each): the chunked kernel alone, chunked + merge, and the ring path with the merge
    on chip, against plain attention (P = 1), launched alternately."""
    w = WORKLOADS["image"]
    q, k, v = (t.to(dev) for t in draw_qkv(w))
    P = 8
    op = torch.empty((P, w.B, w.H, w.S, w.D), dtype=w.dtype, device=dev)
    lp = torch.empty((P, w.B, w.H, w.S), dtype=torch.float32, device=dev)
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.S), dtype=torch.float32, device=dev)
    fns = {
        "plain_P1": lambda: cpattn.attn_fwd(q, k, v, o, lse, stream=stream),
        "chunked_P8": lambda: cpattn.attn_fwd_chunked(q, k, v, P, op, lp, stream=stream),
        "chunked_P8_plus_merge": lambda: (cpattn.attn_fwd_chunked(q, k, v, P, op, lp,
                                                                  stream=stream),
                                          cpattn.attn_lse_merge(op, lp, o, lse, stream=stream)),
        "ring_P8": lambda: cpattn.attn_fwd_ring(q, k, v, P, o, lse, stream=stream),
    }
    ms = _interleaved(fns, dev, stream, iters)
    st = cpattn.attn_device_status(stream)
    if st != cpattn.ATTN_OK:
        raise RuntimeError(f"device status after image leg: {cpattn.attn_status_string(st)}")
    flops = w.attention_flops()
    out = {n: {"median_ms": round(t, 4), "TFLOP/s": round(flops / (t * 1e-3) / 1e12, 1)}
           for n, t in ms.items()}
    out["order"] = "launched alternately; inputs 28 MB per tensor (L2-resident across launches)"
    del q, k, v, op, lp, o, lse
    return {"image_P8": out}


def _interleaved(fns, dev, stream, iters):
    """Median CUDA-event time of each callable, the callables launched in turn `iters` times
    (one warm-up round first), so slow drifts of clock and power affect all alike."""
    for fn in fns.values():
        fn()
    torch.cuda.synchronize(dev)
    times = {n: [] for n in fns}
    for _ in range(iters):
        for n, fn in fns.items():
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            torch.cuda.synchronize(dev)
            times[n].append(a.elapsed_time(b))
    return {n: statistics.median(t) for n, t in times.items()}


def _fp8_leg(cpattn, qd, kd, vd, o, lse, dev, stream, flops, peaks, iters=5):
    """The video problem in e4m3: per-tensor scales amax/448 (cp_absmax), quantisation
    (cp_quantize_e4m3; V transposed), then attn_fwd_fp8 over P = 8 ring steps.  The attention
    launch is timed alone; the quantisation of Q, K, V is reported beside it."""
    scales = [cpattn.cp_absmax(t, stream=stream).item() / 448.0 for t in (qd, kd, vd)]
    q8 = cpattn.cp_quantize_e4m3(qd, scales[0], stream=stream)
    k8 = cpattn.cp_quantize_e4m3(kd, scales[1], stream=stream)
    vt8 = cpattn.cp_quantize_e4m3(vd, scales[2], transpose=True, stream=stream)

    def quant():
        cpattn.cp_quantize_e4m3(qd, scales[0], out=q8, stream=stream)
        cpattn.cp_quantize_e4m3(kd, scales[1], out=k8, stream=stream)
        cpattn.cp_quantize_e4m3(vd, scales[2], transpose=True, out=vt8, stream=stream)

    def attn():
        cpattn.attn_fwd_fp8(q8, k8, vt8, P_CHUNKS, *scales, o=o, lse=lse, stream=stream)

    out = {}
    for name, fn in (("attention", attn), ("quantize_qkv", quant)):
        fn()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(iters)]
        for a, b in evs:
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize(dev)
        out[name] = statistics.median(a.elapsed_time(b) for a, b in evs)
    st = cpattn.attn_device_status(stream)
    if st != cpattn.ATTN_OK:
        raise RuntimeError(f"device status after fp8 leg: {cpattn.attn_status_string(st)}")
    tf = flops / (out["attention"] * 1e-3) / 1e12
    fp8_peak = 2 * peaks["bf16"]   # dense e4m3 is twice the dense bf16 rate
    del q8, k8, vt8
    return {"attn_fwd_fp8_P8": {"median_ms": round(out["attention"], 4), "TFLOP/s": round(tf, 1),
                                "frac_of_fp8_peak": round(tf / fp8_peak, 4),
                                "fp8_peak_note": f"2 x {peaks['source']} burst dense bf16 "
                                                 f"({peaks['bf16']}), the nominal e4m3/bf16 ratio",
                                "quantize_qkv_ms": round(out["quantize_qkv"], 4)}}


def _ulysses_leg(cpattn, dev, stream, iters=6):
    """Ulysses attention on [8][2][2048][32][64] fp16 (S = 16384, 32 heads): the fused kernel
    (sequence-sharded addressing, no re-layout passes) against the unfused chain of
    seq2head(Q, K, V) -> attention on [16][4][16384][64] -> head2seq(O)."""
    w = WORKLOADS["ulysses"]
    P, B, S, H, D = w.P[0], w.B, w.S, w.H, w.D
    q, k, v = (t.to(dev) for t in draw_qkv(w))
    o = torch.empty_like(q)
    lse = torch.empty((P, B, H // P, S), dtype=torch.float32, device=dev)
    qh, kh, vh, oh = (torch.empty((P * B, H // P, S, D), dtype=q.dtype, device=dev)
                      for _ in range(4))
    lh = torch.empty((P * B, H // P, S), dtype=torch.float32, device=dev)

    def fused():
        cpattn.attn_fwd_ulysses(q, k, v, o, lse, stream=stream)

    def chain():
        for x, y in ((q, qh), (k, kh), (v, vh)):
            cpattn.cp_layout_seq2head(x, y.view(P, B, H // P, S, D), stream=stream)
        cpattn.attn_fwd(qh, kh, vh, oh, lh, stream=stream)
        cpattn.cp_layout_head2seq(oh.view(P, B, H // P, S, D), o, stream=stream)

    flops = 4.0 * B * H * S * S * D
    ms = _interleaved({"fused": fused, "unfused_chain": chain}, dev, stream, iters)
    out = {n: {"median_ms": round(t, 4), "TFLOP/s": round(flops / (t * 1e-3) / 1e12, 1)}
           for n, t in ms.items()}
    out["order"] = "launched alternately"
    st = cpattn.attn_device_status(stream)
    if st != cpattn.ATTN_OK:
        raise RuntimeError(f"device status after Ulysses leg: {cpattn.attn_status_string(st)}")
    del q, k, v, o, lse, qh, kh, vh, oh, lh
    return {"ulysses_attention": out}


def run_profile_case(args):
    """One kernel only, for an ncu capture: W + K launches on a reduced case that still exceeds
    L2 -- attn: the video shape with --heads heads (default 2: Q/K/V 22.6 MB each, partials
    181 MB), P=8; merge: the same partials; layout: the Ulysses shape (134 MB each side);
    ulysses: the fused Ulysses attention on the full Ulysses shape ([8][2][2048][32][64] fp16,
    134 MB per tensor); fp8: the e4m3 attention on the video shape with --heads heads, P=8."""
    from context_math_non_b300 import cpattn
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    w = WORKLOAD
    H = args.heads or 2
    if args.profile in ("attn", "merge"):
        q, k, v = (t.to(dev) for t in draw_qkv(w, H=H))
        op, lp = cpattn.attn_fwd_chunked(q, k, v, P_CHUNKS)
        for _ in range(args.warmup + args.steps):
            if args.profile == "attn":
                cpattn.attn_fwd_chunked(q, k, v, P_CHUNKS, op, lp)
            else:
                cpattn.attn_lse_merge(op, lp)
    elif args.profile == "ulysses":
        q, k, v = (t.to(dev) for t in draw_qkv(WORKLOADS["ulysses"]))
        o, lse = cpattn.attn_fwd_ulysses(q, k, v)
        for _ in range(args.warmup + args.steps):
            cpattn.attn_fwd_ulysses(q, k, v, o, lse)
    elif args.profile == "fp8":
        q, k, v = (t.to(dev) for t in draw_qkv(w, H=H))
        scales = [cpattn.cp_absmax(t).item() / 448.0 for t in (q, k, v)]
        q8 = cpattn.cp_quantize_e4m3(q, scales[0])
        k8 = cpattn.cp_quantize_e4m3(k, scales[1])
        vt8 = cpattn.cp_quantize_e4m3(v, scales[2], transpose=True)
        o, lse = cpattn.attn_fwd_fp8(q8, k8, vt8, P_CHUNKS, *scales)
        for _ in range(args.warmup + args.steps):
            cpattn.attn_fwd_fp8(q8, k8, vt8, P_CHUNKS, *scales, o=o, lse=lse)
    else:
        wu = WORKLOADS["ulysses"]
        x = draw_qkv(wu)[0].to(dev)
        y = cpattn.cp_layout_seq2head(x)
        for _ in range(args.warmup + args.steps):
            cpattn.cp_layout_seq2head(x, y)
    torch.cuda.synchronize(dev)
    st = cpattn.attn_device_status()
    if st != cpattn.ATTN_OK:
        raise RuntimeError(cpattn.attn_status_string(st))
    print(f"profile case {args.profile} done", flush=True)


def run_mma_probe():
    """Tensor-core calibration (attn_probe_mma): achievable tcgen05 rates of the MMA forms the
    attention kernel uses, its per-step sequence with and without neighbours, and the latency
    of one GEMM -> consumer -> GEMM hand-off.  Prints one JSON line."""
    from context_math_non_b300 import cpattn
    torch.cuda.set_device(0)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def rate(n, mode, iters):
        cpattn.attn_probe_mma(n, mode, max(32, iters // 20))
        torch.cuda.synchronize()
        a.record()
        cpattn.attn_probe_mma(n, mode, iters)
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b)

    out = {"unit": "TFLOP/s", "sms": sms}
    names = {0: "SS", 1: "TS"}
    for n in (64, 128, 256):
        for mode in (0, 1):
            ms = rate(n, mode, 20000)
            out[f"M128_N{n}_{names[mode]}"] = round(sms * 20000 * 2 * 128 * n * 16 / ms / 1e9, 1)
    labels = {2: "attention_step_sequence", 3: "step_sequence_with_fence",
              5: "step_sequence_with_tmem_streaming_neighbours",
              6: "step_sequence_with_dependent_fma_neighbours",
              7: "step_sequence_with_independent_fma_neighbours"}
    for mode, label in labels.items():
        ms = rate(128, mode, 64000)
        out[label] = round(sms * 64000 * 2 * 128 * 128 * 16 / ms / 1e9, 1)
    for mode, label, D in ((8, "d64_step_sequence_one_lane", 64),
                           (9, "d64_step_sequence_converged_warp_elect", 64),
                           (10, "d128_step_sequence_converged_warp_elect", 128)):
        per_step = 2 * (8 + D // 16)
        steps = 48000 // per_step
        ms = rate(128, mode, steps * per_step)
        out[label] = round(sms * steps * 2 * 4 * 128 * 128 * D / ms / 1e9, 1)
    ms = rate(128, 4, 32000)
    out["handoff_round_trip_ns"] = round(ms * 1e6 / 4000, 1)
    # ALU rates of the softmax's instruction mix (ops per ns per SM; per clock = / GHz)
    alu = {}
    for mode, label in ((0, "ex2_approx"), (1, "cvt_bf16x2"), (2, "fma_f32x2_pairs"),
                        (3, "fma_f32"), (4, "ex2_approx_bf16x2_pairs"),
                        (5, "ex2_approx_f16x2_pairs")):
        iters = 4096
        cpattn.attn_probe_alu(mode, 256)
        torch.cuda.synchronize()
        a.record()
        cpattn.attn_probe_alu(mode, iters)
        b.record()
        torch.cuda.synchronize()
        alu[label] = round(2 * 512 * iters * 8 / (a.elapsed_time(b) * 1e6), 2)
    out["alu_ops_per_ns_per_sm"] = alu
    out["gemm_128x128x128_ns_at_peak"] = round(2 * 128 ** 3 / (2.26e15 / sms) * 1e9, 1)
    st = cpattn.attn_device_status()
    if st != cpattn.ATTN_OK:
        raise RuntimeError(cpattn.attn_status_string(st))
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--ref-rows", type=int, default=24)
    ap.add_argument("--profile", choices=["attn", "merge", "layout", "ulysses", "fp8"],
                    default=None,
                    help="run one kernel on the reduced profiling case (for ncu) and exit")
    ap.add_argument("--heads", type=int, default=None)
    ap.add_argument("--probe", action="store_true",
                    help="run the tensor-core calibration probes and exit")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, world, local_rank = _dist()
    if args.profile:
        run_profile_case(args)
        return
    if args.probe:
        run_mma_probe()
        return

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        line = run_native(args, rank, world, local_rank)
        if rank == 0:
            print(json.dumps(line), flush=True)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
