#!/usr/bin/env python3
"""Benchmark of the quantized decode path on GB300.

One step = one greedy generation of the 135M-shaped model (dim 576, 30 layers, 9/3 heads,
head_dim 64, ffn 1536, vocab 49152, Q4_0 matrices, tied Q8_0 embedding, f32 KV cache):
128 seeded prompt ids then 128 generated tokens, i.e. 256 calls of qd_decode_step
(positions 0..255, batch 1), starting from an empty cache.  ``value`` is tokens processed
per second with the prompt already resident in device memory; ``e2e`` is the same through
the C ABI with pinned host token buffers (a 4-byte host->device copy and a 4-byte
device->host copy per token inside the timed region).

L2 is flushed (a 256 MB device write) between timed steps, outside the step's events.  Within
a step, consecutive tokens re-read the same 90 MB of weights, which the 129 MB L2 may hold.

The JSON line also carries: the roofline of the dominant kernel (timed live with CUDA events
on the launching stream), the q_gemv GB/s sweep at the 7B-like and TinyLlama shapes, the
1.7B-shaped INT8 step at context 4096 (batch 1 and 16), the oracle's CPU rate on a bounded
sample, SM clocks sampled during the timed region, and the kernel-launch count.

Multi-GPU: the decode path is replicated, one independent sequence per rank, with no
collective on the data path ("weak" scaling); rank 0 prints the aggregate.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "q_gemv achieved HBM GB/s (% of peak); decode tokens/s at 135M and 1.7B shapes"
PROMPT, GEN = 128, 128
L2_FLUSH_BYTES = 256 << 20


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d.get("bf16_tflops", 1913.0)), "measured"
    return 6800.0, 1900.0, "fallback"


# ----------------------------------------------------------------------------- distributed

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, backend):
    if world > 1:
        import torch.distributed as dist

        if not dist.is_initialized():
            dist.init_process_group(backend=backend)


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def reduce_max(value: float, world: int) -> float:
    """Max of a float over ranks (host-side coordination only)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world: int, steps: int, units_per_step: int, t_max: float) -> float:
    """Units processed by all ranks over the slowest rank's timed seconds (weak scaling:
    every rank runs its own replica of the workload)."""
    return world * steps * units_per_step / t_max


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampled every 200 ms while the timed region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        # nvidia-smi numbers GPUs physically; under CUDA_VISIBLE_DEVICES the torch index can
        # name another GPU, so query by the device's UUID (read-only, as before)
        self.gpu = str(gpu_index)
        try:
            import torch

            uuid = str(torch.cuda.get_device_properties(gpu_index).uuid)
            if uuid:
                self.gpu = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            pass
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", self.gpu, f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        mhz, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                mhz.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not mhz:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(mhz)}


# ----------------------------------------------------------------------------- our arm

def build_smol135m(qd, torch, seed, path=None):
    import qdsynth

    cfg = qdsynth.SMOL_135M
    host = qdsynth.model_tensors(cfg, seed)
    srcs = [None if t is None else torch.from_numpy(np.ascontiguousarray(t)).cuda() for t in host]
    model = qd.Model(qd.make_config(cfg, PROMPT + GEN, 1), srcs)
    if path:
        model.set_step_path(qd.STEP_CLUSTER if path == "cluster" else qd.STEP_KERNEL_CHAIN)
    torch.cuda.synchronize()
    del srcs
    return cfg, model


def time_gemv_cold(qd, torch, fmt, rows, cols, batch, stream, reps=None, seed=0, overlap=False):
    """Average device time of one q_gemv launch.  The launches run back to back from a
    CUDA graph (so host launch overhead is not measured), each on a distinct weight copy so
    the weights come from HBM: the copies total >= 2x L2, and L2 is flushed before each
    replay.  overlap=True launches with QD_GEMV_OVERLAP, the decode step's launch mode (the
    next launch streams its weights while the previous one finishes).  Returns (seconds,
    launches per replay)."""
    import qdsynth

    src = qdsynth.weight_src(fmt, seed, f"bench.{fmt}.{rows}x{cols}", rows, cols)
    pb = qd.packed_bytes(fmt, rows, cols)
    pbuf = torch.empty(pb, dtype=torch.uint8, device="cuda")
    qd.repack(fmt, torch.from_numpy(src).cuda(), rows, cols, pbuf)
    n = max(8, min(400, (2 * L2_FLUSH_BYTES) // pb + 1)) if reps is None else reps
    copies = pbuf.repeat(n).view(n, pb)  # n contiguous copies; pb % 16 == 0 keeps each aligned
    x = torch.from_numpy(qdsynth.activations(seed, "bench.x", batch, cols)).cuda()
    y = torch.empty(batch, rows, device="cuda")
    ptrs = [copies[i].data_ptr() for i in range(n)]
    flags = qd.GEMV_OVERLAP if overlap else 0
    for p in ptrs[:3]:
        qd.q_gemv_ex(fmt, p, rows, cols, x, y, batch, flags, stream=stream)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for p in ptrs:
            qd.q_gemv_ex(fmt, p, rows, cols, x, y, batch, flags)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    best = None
    for _ in range(4):
        flush.fill_(1)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        t = e0.elapsed_time(e1) / 1e3 / len(ptrs)
        best = t if best is None else min(best, t)
    del g, copies, flush
    return best, len(ptrs)


_CEIL_CACHE = {}


def time_read_ceiling(qd, torch, nbytes, overlap, reps=None):
    """The plain-read ceiling for a buffer of nbytes in the same harness as time_gemv_cold
    (distinct copies, L2 flushed before each replay of back-to-back launches): the best
    over a few launch shapes of qd_read_ceiling.  Returns (seconds, config)."""
    key = (nbytes, overlap)
    if key in _CEIL_CACHE:
        return _CEIL_CACHE[key]
    nb = (nbytes + 15) // 16 * 16
    n = max(8, min(400, (2 * L2_FLUSH_BYTES) // nb + 1)) if reps is None else reps
    buf = torch.randint(0, 255, (n, nb), dtype=torch.uint8, device="cuda")
    sink = torch.zeros(1, dtype=torch.int32, device="cuda")
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    flags = qd.GEMV_OVERLAP if overlap else 0
    best = None
    for cps, thr in ((1, 512), (2, 512), (2, 256), (4, 256)):
        ptrs = [buf[i].data_ptr() for i in range(n)]
        for ptr in ptrs[:3]:
            qd.read_ceiling(ptr, nb, cps, thr, flags, sink)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for ptr in ptrs:
                qd.read_ceiling(ptr, nb, cps, thr, flags, sink)
        for _ in range(3):
            flush.fill_(1)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            g.replay()
            e1.record()
            torch.cuda.synchronize()
            t = e0.elapsed_time(e1) / 1e3 / n
            if best is None or t < best[0]:
                best = (t, f"{cps} CTA/SM x {thr} threads")
        del g
    del buf, flush
    _CEIL_CACHE[key] = best
    return best


def algorithmic_bytes(fmt, rows, cols, batch, qd):
    return qd.packed_bytes(fmt, rows, cols) + 4 * batch * (rows + cols)


def run_ours(args, world, rank, local):
    import torch

    import qdsynth
    import quantized_decode_gemv_gb300 as qd

    torch.cuda.set_device(local)
    init_dist(world, "nccl")
    if not os.path.exists(qd.LIB_PATH):
        qd.build()
    qd.load()
    stream = torch.cuda.current_stream()
    cfg, model = build_smol135m(qd, torch, seed=rank, path=args.step_path)
    T = PROMPT + GEN
    prompt = qdsynth.tokens(rank, "smol135m.prompt", PROMPT, cfg["vocab"]).astype(np.int32)
    # device-resident token slots: slot t is the input of position t; outputs of prompt
    # positions go to scratch, outputs from position 127 on feed the next slot.
    tok = torch.zeros(T + 1, dtype=torch.int32, device="cuda")
    tok[:PROMPT] = torch.from_numpy(prompt).cuda()
    scratch = torch.zeros(T, dtype=torch.int32, device="cuda")
    tok_h = torch.zeros(T + 1, dtype=torch.int32).pin_memory()
    tok_h[:PROMPT] = torch.from_numpy(prompt)
    scratch_h = torch.zeros(T, dtype=torch.int32).pin_memory()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")

    def step(dev_side: bool, mid=None):
        model.reset(stream)
        t_in, s_out = (tok, scratch) if dev_side else (tok_h, scratch_h)
        base_in, base_s = t_in.data_ptr(), s_out.data_ptr()
        for t in range(T):
            if t == PROMPT and mid is not None:
                mid.record(stream)  # prompt positions 0..127 done; generated tokens from here
            out = base_in + 4 * (t + 1) if t >= PROMPT - 1 else base_s + 4 * t
            model.decode_step(base_in + 4 * t, 1, out, None, stream)

    for _ in range(args.warmup):
        step(True)
    torch.cuda.synchronize()
    gen_dev = tok[PROMPT:T].cpu().numpy().copy()
    launches_token = model.launches_per_step()
    reset_launches = 6  # zeroing kernels of qd_model_reset

    # ---- timed region: device-resident inputs
    times = []
    with ClockSampler(local) as clk:
        barrier(world)
        torch.cuda.synchronize()
        wall0 = time.perf_counter()
        for _ in range(args.steps):
            flush.fill_(0)  # L2 flush between steps (outside the step's events)
            e0, em, e1 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
            e0.record(stream)
            step(True, em)
            e1.record(stream)
            times.append((e0, em, e1))
        torch.cuda.synchronize()
        barrier(world)
        wall = time.perf_counter() - wall0
    step_s = [a.elapsed_time(b) / 1e3 for a, _, b in times]
    prefill_s = [a.elapsed_time(m) / 1e3 for a, m, _ in times]
    decode_s = [m.elapsed_time(b) / 1e3 for _, m, b in times]
    t_total = reduce_max(sum(step_s), world)
    value = whole_job_rate(world, args.steps, T, t_total)
    assert np.array_equal(tok[PROMPT:T].cpu().numpy(), gen_dev), "generation changed between runs"

    # ---- end to end: pinned host token buffers through the C ABI
    for _ in range(2):
        step(False)
    torch.cuda.synchronize()
    e_times = []
    barrier(world)
    for _ in range(args.steps):
        flush.fill_(0)
        torch.cuda.synchronize()
        w0 = time.perf_counter()
        step(False)
        torch.cuda.synchronize()
        got = tok_h[PROMPT:T].numpy().copy()  # the step's result, read on the host
        e_times.append(time.perf_counter() - w0)
    assert np.array_equal(got, gen_dev), "host-buffer generation differs from device-buffer generation"
    e2e_total = reduce_max(sum(e_times), world)
    e2e_value = whole_job_rate(world, args.steps, T, e2e_total)

    hbm, bf16, peak_kind = peaks()
    # weight-bytes-per-token roofline: every weight byte (tied head once) + the KV rows read
    kv_per_pos = 2 * cfg["layers"] * cfg["n_kv_heads"] * cfg["head_dim"] * 4
    wbytes = model.weights.numel()

    def phase(ts, p0, p1):
        n = p1 - p0
        tput = n / statistics.median(ts)
        bytes_ = sum(wbytes + kv_per_pos * (p + 1) for p in range(p0, p1))
        roof = n / (bytes_ / (hbm * 1e9))
        return {"tokens/s": round(tput, 1), "roofline_tokens/s": round(roof, 1), "frac": round(tput / roof, 4),
                "frac_nominal_8tbs": round(tput / (n / (bytes_ / 8e12)), 4)}

    phases = {"prefill (positions 0-127)": phase(prefill_s, 0, PROMPT),
              "decode (positions 128-255)": phase(decode_s, PROMPT, T),
              "whole step": phase(step_s, 0, T)}
    out = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(1e3 * t_total / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32 activations; q4_0/q8_0 weights",
        "data": "synthetic (seeded SplitMix64 weights and prompt, 135M-shaped)",
        "config": {"workload": "135M-shaped greedy decode: 128 prompt ids + 128 generated tokens, batch 1",
                   "model": "llama-style 135M shape (dim 576, 30 layers, 9/3 heads, ffn 1536, vocab 49152)",
                   "w_fmt": "q4_0", "emb_fmt": "q8_0 (tied)", "global_batch": world, "seq_len": T,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "flushed (256 MB write) between timed steps; inputs (90 MB weights) fit in L2 within a step"},
        "e2e": {"value": round(e2e_value, 1), "unit": "tokens/s", "h2d_bytes_per_step": 4 * T,
                "d2h_bytes_per_step": 4 * T},
        "gpu_launches": int(args.steps * (T * launches_token + reset_launches)),
        "launches_per_token": launches_token,
        "wall_s_timed": round(wall, 3),
        "ms_per_token": round(1e3 * t_total / (args.steps * T), 4),
        "phases": phases,
        "bytes_per_token": {"weights": int(wbytes), "kv_per_position": kv_per_pos},
    }
    out["clocks"] = clk.summary()

    if rank == 0 and not args.quick:
        out["roofline"] = roofline_dominant(qd, torch, stream, hbm, peak_kind)
        out["q_gemv_sweep"] = gemv_sweep(qd, torch, stream, hbm, args)
        out["quantize_i8"] = bench_quantize(qd, torch, 49152, 2048, hbm)
        _, bf16, _ = peaks()
        out["prefill_gemm"] = []
        for fmt, r_, c_ in (("q4_0", 14336, 4096), ("q8_0", 14336, 4096), ("i8", 8192, 2048)):
            g = bench_gemm(qd, torch, fmt, r_, c_, 512, 10)
            g["frac_of_bf16_peak"] = round(g["useful_TFLOP/s"] / bf16, 4)
            out["prefill_gemm"].append(g)
        del model
        torch.cuda.empty_cache()
        out["decode_135m_modes"] = bench_135m_modes(qd, torch, stream)
        out["prefill_135m"] = bench_prefill_135m(qd, torch, stream)
        if not args.no_1p7b:
            out["decode_1p7b"] = bench_1p7b(qd, torch, stream, args, hbm)
            out["decode_1p7b"].update(bench_1p7b(qd, torch, stream, args, hbm, kv_f16=True))
        if world == 1:
            out["cpu_baseline"] = cpu_baseline(cfg, seconds=args.cpu_seconds)
            try:  # an auxiliary host measurement: a failure is recorded, not fatal to the line
                out["cpu_baseline_1p7b"] = cpu_baseline_1p7b()
            except Exception as e:  # noqa: BLE001
                out["cpu_baseline_1p7b"] = {"error": f"{type(e).__name__}: {e}"}
    if rank == 0:
        print(json.dumps(out))
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


def gemv_source_sha() -> str:
    """sha256 over the streaming GEMV's sources (the kernel and its integer-dot header)."""
    h = hashlib.sha256()
    for f in ("qd_gemv_stream.cu", "qd_intdot.cuh"):
        h.update(open(os.path.join(ROOT, "quantized_decode_gemv_gb300", "csrc", f), "rb").read())
    return h.hexdigest()


def profile_traffic(summary: str):
    """Per-launch DRAM bytes from a committed ncu summary under profiles/, or None when the
    GEMV kernel source changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", summary)
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    h = re.search(r"source_sha256:\s*([0-9a-f]{16,64})", text)
    cur = gemv_source_sha()
    if not m or not h or not cur.startswith(h.group(1)):
        return None
    return float(m.group(1))


DECODE_SHAPES = [(960, 576), (576, 576), (3072, 576), (576, 1536)]  # QKV, Wo, gate/up, down


def roofline_dominant(qd, torch, stream, hbm, peak_kind):
    """The step's dominant kernel is the Q4_0 streaming GEMV, k_gemv_warp (120 of the 152
    launches per token, over the four per-layer shapes).  Achieved bandwidth: algorithmic
    bytes of the four shapes over the sum of their average launch durations, each shape
    timed as back-to-back launches on cold weights in the decode step's launch mode
    (QD_GEMV_OVERLAP)."""
    tot_b, tot_t = 0, 0.0
    per = {}
    for r, c in DECODE_SHAPES:
        t, n = time_gemv_cold(qd, torch, "q4_0", r, c, 1, stream, overlap=True)
        b = algorithmic_bytes("q4_0", r, c, 1, qd)
        tot_b += b
        tot_t += t
        per[f"{r}x{c}"] = {"us": round(t * 1e6, 2), "GB/s": round(b / t / 1e9, 1)}
    achieved = tot_b / tot_t / 1e9
    traffic = profile_traffic("q_gemv_q4_0_decode_shapes.md")
    return {"kernel": "k_gemv_warp<Q4_0> (decode-step shapes 960x576, 576x576, 3072x576, 576x1536)",
            "bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
            "frac": round(achieved / hbm, 4), "peak_kind": peak_kind,
            "traffic": traffic, "algorithmic_bytes_per_launch": round(tot_b / len(DECODE_SHAPES)),
            "per_shape": per}


def bench_quantize(qd, torch, rows, cols, hbm, reps=10):
    """Load-time per-row INT8 quantisation of a BF16 matrix (qd_quantize_i8_rows): average
    device time per launch over `reps` launches, L2 flushed before each (the bf16 input of
    the default shape, 201 MB, also exceeds L2).  Algorithmic bytes: 2 read + 1 written per
    weight, 4 written per row."""
    g = torch.Generator(device="cuda").manual_seed(7)
    w = torch.randn(rows, cols, generator=g, device="cuda").to(torch.bfloat16).view(torch.int16)
    out = torch.empty(qd.src_bytes("i8", rows, cols), dtype=torch.uint8, device="cuda")
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    for _ in range(3):
        qd.quantize_i8_rows(w, rows, cols, out)
    torch.cuda.synchronize()
    ts = []
    for _ in range(reps):
        flush.fill_(1)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        qd.quantize_i8_rows(w, rows, cols, out)
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1) / 1e3)
    t = statistics.median(ts)
    by = 3 * rows * cols + 4 * rows
    del w, out, flush
    return {"shape": f"{rows}x{cols}", "us": round(t * 1e6, 2), "us_best": round(min(ts) * 1e6, 2),
            "algorithmic_bytes": by, "GB/s": round(by / t / 1e9, 1), "frac": round(by / t / 1e9 / hbm, 4)}


def gemv_sweep(qd, torch, stream, hbm, args):
    """q_gemv at the sweep shapes: 'chained' = back-to-back launches in the decode step's
    launch mode (QD_GEMV_OVERLAP), 'isolated' = plain launches (each waits for the previous
    one to finish).  Cold weights throughout."""
    res = {}
    shapes = [("q4_0", 576, 1536)]
    for fmt in ("q8_0", "q4_0"):
        for r, c in [(4096, 4096), (11008, 4096), (4096, 11008), (14336, 4096)]:
            shapes.append((fmt, r, c))
    for r, c in [(2048, 2048), (5632, 2048), (2048, 5632), (32000, 2048)]:
        shapes.append(("q4_k", r, c))
    for r, c in [(6144, 2048), (2048, 2048), (16384, 2048), (2048, 8192), (49152, 2048)]:
        shapes.append(("i8", r, c))
    batches = (1,) if args.batch1_sweep else (1, 2, 4, 8)
    for fmt, r, c in shapes:
        bs = (1, 16) if fmt == "i8" else (batches if fmt != "q4_k" and (r, c) != (576, 1536) else (1,))
        for b in bs:
            by = algorithmic_bytes(fmt, r, c, b, qd)
            row = {}
            # the isolated launch mode at batch 1 only (the batch 2-8 lines keep the run short)
            modes = (("chained", True), ("isolated", False)) if b == 1 or args.full_sweep else (("chained", True),)
            for mode, ov in modes:
                t, n = time_gemv_cold(qd, torch, fmt, r, c, b, stream, overlap=ov)
                row[mode] = {"us": round(t * 1e6, 2), "GB/s": round(by / t / 1e9, 1),
                             "frac": round(by / t / 1e9 / hbm, 3)}
                if fmt != "i8" and (r, c) != (576, 1536) and fmt != "q4_k":
                    # the same bytes read by a plain read kernel, same harness and mode
                    tc_, how = time_read_ceiling(qd, torch, qd.packed_bytes(fmt, r, c), ov)
                    row[mode]["read_ceiling_us"] = round(tc_ * 1e6, 2)
                    row[mode]["frac_of_read_ceiling"] = round(tc_ / t, 3)
            res[f"{fmt} {r}x{c} b{b}"] = row
    return res


def bench_1p7b(qd, torch, stream, args, hbm, batches=(1, 16), layers=None, kv_f16=False):
    """1.7B-shaped INT8 step at context 4096 (pos 4095): batch 1 and 16, cache entries N(0,1)
    drawn on the device with a seeded torch generator (timing only; the parity tests use the
    host generator)."""
    import qdsynth

    cfg = qdsynth.SMOL_1_7B if not layers else dict(qdsynth.SMOL_1_7B, layers=layers)
    cfg = dict(cfg, kv_f16=kv_f16)
    esz = 2 if kv_f16 else 4  # bytes per cache element
    ctx = 4096
    host = qdsynth.model_tensors(cfg, 0)
    out = {}
    for batch in batches:
        srcs = [None if t is None else torch.from_numpy(np.ascontiguousarray(t)).cuda() for t in host]
        m = qd.Model(qd.make_config(cfg, ctx, batch), srcs)
        torch.cuda.synchronize()
        del srcs
        kp, vp = m.kv_cache_ptrs()
        base = m.state.data_ptr()
        n = cfg["layers"] * batch * cfg["n_kv_heads"] * ctx * cfg["head_dim"]
        g = torch.Generator(device="cuda").manual_seed(1234)
        for ptr in (kp, vp):
            m.state[ptr - base:ptr - base + esz * n].view(torch.float16 if kv_f16 else torch.float32).normal_(
                generator=g)
        toks = torch.from_numpy(qdsynth.tokens(0, "c5.tokens", 16, cfg["vocab"])[:batch].astype(np.int32)).cuda()
        outt = torch.empty(batch, dtype=torch.int32, device="cuda")
        flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
        ts = []
        for i in range(3 + 20):
            m.set_pos([ctx - 1] * batch, stream)
            flush.fill_(0)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            m.decode_step(toks, batch, outt, None, stream)
            e1.record(stream)
            torch.cuda.synchronize()
            if i >= 3:
                ts.append(e0.elapsed_time(e1) / 1e3)
        t = statistics.median(ts)
        wbytes = m.weights.numel()
        kv = 2 * n * esz
        gbs = (wbytes + kv) / t / 1e9
        roof = batch / ((wbytes + kv) / (hbm * 1e9))
        out[f"batch{batch}" + ("_kv_f16" if kv_f16 else "")] = {"ms_per_step": round(t * 1e3, 3), "ms_per_step_best": round(min(ts) * 1e3, 3),
                                "launches_per_step": m.launches_per_step(),
                                "tokens/s": round(batch / t, 1), "bytes_per_step": int(wbytes + kv),
                                "GB/s": round(gbs, 1), "roofline_tokens/s": round(roof, 1),
                                "frac": round(gbs / hbm, 4), "frac_nominal_8tbs": round(gbs / 8000, 4)}
        m.close()
        del m, flush
        torch.cuda.empty_cache()
    return out


def bench_135m_modes(qd, torch, stream, steps=50):
    """135M-shaped decode, batch 1, in the default mode (f32 activations, f32 cache), in
    the pages' ggml-exact mode (Q8_0 activations before every product, binary16 cache) and
    on the optional cluster path (the layers as one thread-block cluster): tokens/s over
    `steps` consecutive steps from position 150 (graph replays)."""
    import qdsynth

    out = {}
    for name, extra, path in (("f32", {}, None), ("ggml_exact", {"act_q8": True, "kv_f16": True}, None),
                              ("f32_cluster_path", {}, "cluster")):
        cfg = dict(qdsynth.SMOL_135M, **extra)
        host = qdsynth.model_tensors(cfg, 0)
        srcs = [None if t is None else torch.from_numpy(np.ascontiguousarray(t)).cuda() for t in host]
        m = qd.Model(qd.make_config(cfg, 256, 1), srcs)
        del srcs
        if path == "cluster":
            if not m.cluster_available():
                out[name] = {"unavailable": "the device cannot schedule the cluster"}
                m.close()
                continue
            m.set_step_path(qd.STEP_CLUSTER)
        tok = torch.zeros(1, dtype=torch.int32, device="cuda")
        outt = torch.empty(1, dtype=torch.int32, device="cuda")
        for _ in range(3):
            m.set_pos([150], stream)
            m.decode_step(tok, 1, outt, None, stream)
        m.set_pos([150], stream)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            m.decode_step(outt, 1, outt, None, stream)
        e1.record(stream)
        torch.cuda.synchronize()
        t = e0.elapsed_time(e1) / 1e3 / steps
        out[name] = {"ms_per_token": round(t * 1e3, 4), "tokens/s": round(1 / t, 1),
                     "launches_per_token": m.launches_per_step()}
        m.close()
        del m
        torch.cuda.empty_cache()
    return out


def bench_prefill_135m(qd, torch, stream, reps=10):
    """The 135M-shaped model's 128-token prompt in one qd_prefill call (batched prefill), on
    the tensor-core GEMM (flags 0) and on the batched GEMV (QD_PREFILL_EXACT), against the
    same prompt as 128 decode steps: prompt tokens/s, CUDA events around the prefill call
    only (the cache reset before each is outside them); L2 flushed before each rep."""
    import qdsynth

    cfg = qdsynth.SMOL_135M
    host = qdsynth.model_tensors(cfg, 0)
    srcs = [None if t is None else torch.from_numpy(np.ascontiguousarray(t)).cuda() for t in host]
    m = qd.Model(qd.make_config(cfg, PROMPT + GEN, 1), srcs)
    del srcs
    prompt = torch.from_numpy(qdsynth.tokens(0, "smol135m.prompt", PROMPT, cfg["vocab"]).astype(np.int32)).cuda()
    ws = torch.empty(m.prefill_workspace(PROMPT), dtype=torch.uint8, device="cuda")
    outt = torch.empty(1, dtype=torch.int32, device="cuda")
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    res = {"tokens": PROMPT, "model": "135M-shaped, q4_0 layers, q8_0 tied head"}
    toks = {}
    for name, flags in (("gemm", 0), ("exact", qd.PREFILL_EXACT), ("decode_steps", None)):
        def once(flags=flags):
            if flags is None:
                for i in range(PROMPT):
                    m.decode_step(prompt.data_ptr() + 4 * i, 1, outt, None, stream)
            else:
                m.prefill(0, prompt, PROMPT, outt, None, flags=flags, workspace=ws, stream=stream)
        for _ in range(3):
            m.reset(stream)
            once()
        ts = []
        for _ in range(reps):
            flush.fill_(0)
            m.reset(stream)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            once()
            e1.record(stream)
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) / 1e3)
        assert m.check() == 0
        toks[name] = int(outt.item())
        t = statistics.median(ts)
        res[name] = {"ms": round(t * 1e3, 3), "prompt_tokens/s": round(PROMPT / t, 1)}
    # the token after the prompt: the exact path and the decode steps agree (same products);
    # the GEMM's binary16 weights may move a near-tie
    res["next_token"] = toks
    res["speedup_vs_decode_steps"] = {k: round(res["decode_steps"]["ms"] / res[k]["ms"], 2) for k in ("gemm", "exact")}
    m.close()
    del m
    torch.cuda.empty_cache()
    return res


def cpu_baseline(cfg, seconds=15.0, max_tokens=64):
    """The oracle, as it stands, on the host cores: the first tokens of the same run (prompt
    positions 0, 1, ...), until about `seconds` of CPU work."""
    import oracle
    import qdsynth

    host = qdsynth.model_tensors(cfg, 0)
    om = oracle.Model(dict(cfg, max_ctx=PROMPT + GEN), host)
    L, hk, hd = cfg["layers"], cfg["n_kv_heads"], cfg["head_dim"]
    ctx = PROMPT + GEN
    kc = np.zeros(L * hk * ctx * hd, np.float32)
    vc = np.zeros_like(kc)
    prompt = qdsynth.tokens(0, "smol135m.prompt", PROMPT, cfg["vocab"])
    def run(threads, budget):
        cores = oracle.set_threads(threads)
        kc[:] = 0
        vc[:] = 0
        t0 = time.perf_counter()
        n = 0
        while n < max_tokens and (time.perf_counter() - t0) < budget:
            om.decode_step(kc, vc, hk * ctx * hd, n, int(prompt[n]))
            n += 1
        return n, time.perf_counter() - t0, cores

    n1, dt1, _ = run(1, seconds / 2)
    n, dt, cores = run(os.cpu_count() or 1, seconds / 2)
    return {"value": round(n / dt, 3), "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"first {n} tokens (positions 0..{n - 1}) of the 135M 128+128 run, batch 1, "
                      f"{dt:.1f} s; oracle C code, double accumulation, OpenMP over matrix rows",
            "single_thread": {"value": round(n1 / dt1, 3), "unit": "tokens/s", "cores": 1,
                              "sample": f"first {n1} tokens, {dt1:.1f} s"}}


def cpu_baseline_1p7b():
    """The oracle on the host cores at the 1.7B shape, context 4096 (one step at position
    4095 over a 4095-entry N(0,1) cache): one step on all cores and on one core, and a
    batch-16 step as 16 sequences' steps one after another (the oracle takes one sequence
    per call; the 16 calls share one cache here, which changes no arithmetic)."""
    import oracle
    import qdsynth

    cfg = qdsynth.SMOL_1_7B
    ctx = 4096
    host = qdsynth.model_tensors(cfg, 0)
    om = oracle.Model(dict(cfg, max_ctx=ctx), host)
    L, hk, hd = cfg["layers"], cfg["n_kv_heads"], cfg["head_dim"]
    n = L * hk * ctx * hd
    kc = qdsynth.normal_f32(0, "c5.kc", n)
    vc = qdsynth.normal_f32(0, "c5.vc", n)
    toks = qdsynth.tokens(0, "c5.tokens", 16, cfg["vocab"])

    def steps(threads, count):
        cores = oracle.set_threads(threads)
        t0 = time.perf_counter()
        for i in range(count):
            om.decode_step(kc, vc, hk * ctx * hd, ctx - 1, int(toks[i]))
        return time.perf_counter() - t0, cores

    t_all, cores = steps(os.cpu_count() or 1, 1)
    t_one, _ = steps(1, 1)
    t_b16, _ = steps(os.cpu_count() or 1, 16)
    return {"kind": "oracle", "cores": cores, "unit": "ms/step",
            "batch1": round(t_all * 1e3, 1), "batch1_single_thread": round(t_one * 1e3, 1),
            "batch16": round(t_b16 * 1e3, 1), "batch16_tokens/s": round(16 / t_b16, 2),
            "sample": "one step at position 4095 per sequence (context 4096), INT8 1.7B shape; batch 16 as "
                      "16 one-sequence calls sharing one cache; oracle C code, double accumulation"}


# ----------------------------------------------------------------------------- reference arm

def run_reference(args, world, rank, local):
    """The oracle timed as the reference arm, on the same workload: each step is a bounded
    sample (the first `ref_tokens` positions of the 135M run)."""
    if rank != 0:
        return
    import oracle
    import qdsynth

    cfg = qdsynth.SMOL_135M
    host = qdsynth.model_tensors(cfg, 0)
    ctx = PROMPT + GEN
    om = oracle.Model(dict(cfg, max_ctx=ctx), host)
    L, hk, hd = cfg["layers"], cfg["n_kv_heads"], cfg["head_dim"]
    prompt = qdsynth.tokens(0, "smol135m.prompt", PROMPT, cfg["vocab"])
    nt = args.ref_tokens

    def one():
        kc = np.zeros(L * hk * ctx * hd, np.float32)
        vc = np.zeros_like(kc)
        for p in range(nt):
            om.decode_step(kc, vc, hk * ctx * hd, p, int(prompt[p]))

    for _ in range(args.warmup):
        one()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one()
    dt = time.perf_counter() - t0
    v = args.steps * nt / dt
    cores = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    sample = f"{nt} tokens per step (positions 0..{nt - 1} of the 135M 128+128 run), batch 1"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(v, 3), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * dt / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64 accumulation",
        "data": "synthetic (seeded SplitMix64 weights and prompt, 135M-shaped)",
        "config": {"workload": "135M-shaped greedy decode: 128 prompt ids + 128 generated tokens, batch 1",
                   "global_batch": 1, "seq_len": PROMPT + GEN, "parallelism": "CPU oracle"},
        "cpu_baseline": {"value": round(v, 3), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(v, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


def run_gemv_only(spec: str, reps: int, ceiling: bool = True):
    """Microbenchmark of one q_gemv shape, e.g. "q4_0:14336x4096:1" (format:rowsxcols:batch):
    `reps` cold-weight passes; prints one JSON line (not the benchmark contract line)."""
    import torch

    import quantized_decode_gemv_gb300 as qd

    fmt, shape, b = spec.split(":")
    r, c = (int(v) for v in shape.split("x"))
    b = int(b)
    if not os.path.exists(qd.LIB_PATH):
        qd.build()
    qd.load()
    stream = torch.cuda.current_stream()
    by = algorithmic_bytes(fmt, r, c, b, qd)
    hbm, _, kind = peaks()
    out = {"gemv": spec, "peak": hbm, "peak_kind": kind, "algorithmic_bytes": by}
    for mode, ov in (("chained", True), ("isolated", False)):
        ts = []
        for _ in range(reps):
            t, n = time_gemv_cold(qd, torch, fmt, r, c, b, stream, overlap=ov)
            ts.append(t)
        t = min(ts)
        out[mode] = {"us": round(t * 1e6, 3), "GB/s": round(by / t / 1e9, 1), "frac": round(by / t / 1e9 / hbm, 4),
                     "launches_per_pass": n}
        if ceiling:
            tc_, how = time_read_ceiling(qd, torch, qd.packed_bytes(fmt, r, c), ov)
            out[mode].update({"read_ceiling_us": round(tc_ * 1e6, 3), "read_ceiling_launch": how,
                              "frac_of_read_ceiling": round(tc_ / t, 4)})
    print(json.dumps(out))


def bench_gemm(qd, torch, fmt, rows, cols, t, reps=20):
    """The prefill product (qd_q_gemm) at t tokens: median and best of `reps` launches of the
    call (the x split prologue and the tensor-core kernel) with L2 flushed before each, the
    useful flops 2 t rows cols, and the two kernels' shares timed apart (CUDA events on the
    launching stream)."""
    import qdsynth

    src = qdsynth.weight_src(fmt, 0, f"gemm{rows}x{cols}", rows, cols)
    s = torch.from_numpy(np.ascontiguousarray(src.reshape(-1).view(np.uint8))).cuda()
    w = torch.empty(qd.packed_bytes(fmt, rows, cols), dtype=torch.uint8, device="cuda")
    qd.repack(fmt, s, rows, cols, w)
    del s
    x = torch.from_numpy(qdsynth.activations(0, f"gemmx{cols}", t, cols)).cuda()
    y = torch.empty(t, rows, dtype=torch.float32, device="cuda")
    ws = torch.empty(qd.q_gemm_workspace(fmt, rows, cols, t), dtype=torch.uint8, device="cuda")
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    ts = []
    for i in range(3 + reps):
        flush.fill_(0)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        qd.q_gemm(fmt, w, rows, cols, x, y, t, ws, stream=stream)
        e1.record(stream)
        torch.cuda.synchronize()
        if i >= 3:
            ts.append(e0.elapsed_time(e1) / 1e3)
    flops = 2.0 * t * rows * cols
    med, best = statistics.median(ts), min(ts)
    return {"fmt": fmt, "rows": rows, "cols": cols, "t": t, "us": round(med * 1e6, 2), "us_best": round(best * 1e6, 2),
            "useful_TFLOP/s": round(flops / med / 1e12, 1), "weight_bytes": int(w.numel()),
            "note": "cold L2 per launch; includes the x split prologue"}


def run_gemm_only(spec: str, reps: int):
    """The prefill product alone, e.g. "q4_0:14336x4096:512" (format:rowsxcols:tokens); prints
    one JSON line (not the benchmark contract line)."""
    import torch

    import quantized_decode_gemv_gb300 as qd

    fmt, shape, t = spec.split(":")
    r, c = (int(v) for v in shape.split("x"))
    if not os.path.exists(qd.LIB_PATH):
        qd.build()
    qd.load()
    _, bf16, kind = peaks()
    res = bench_gemm(qd, torch, fmt, r, c, int(t), max(reps, 5))
    res["frac_of_bf16_peak"] = round(res["useful_TFLOP/s"] / bf16, 4)
    print(json.dumps({"gemm": res, "bf16_peak_tflops": bf16, "peak_kind": kind}))


def run_q8act_only(spec: str, reps: int):
    """The ggml-exact activation path alone, e.g. "q4_0:14336x4096:1": the Q8 quantiser and
    the integer product, each timed with L2 flushed before every launch; prints one JSON
    line (not the benchmark contract line)."""
    import torch

    import qdsynth
    import quantized_decode_gemv_gb300 as qd

    fmt, shape, b = spec.split(":")
    rows, cols = (int(v) for v in shape.split("x"))
    batch = int(b)
    if not os.path.exists(qd.LIB_PATH):
        qd.build()
    qd.load()
    hbm, _, kind = peaks()
    src = qdsynth.weight_src(fmt, 0, f"q8a{rows}x{cols}", rows, cols)
    s = torch.from_numpy(np.ascontiguousarray(src.reshape(-1).view(np.uint8))).cuda()
    w = torch.empty(qd.packed_bytes(fmt, rows, cols), dtype=torch.uint8, device="cuda")
    qd.repack(fmt, s, rows, cols, w)
    x = torch.from_numpy(qdsynth.activations(0, f"q8ax{cols}", batch, cols)).cuda()
    with_sum = fmt == "q4_1"
    xq = torch.empty(qd.q8_bytes(batch, cols, with_sum), dtype=torch.uint8, device="cuda")
    y = torch.empty(batch, rows, dtype=torch.float32, device="cuda")
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    res = {}
    for name, call in (("quantize", lambda: qd.quantize_q8(x, batch, cols, xq, with_sum, stream=stream)),
                       ("product", lambda: qd.q_gemv_q8(fmt, w, rows, cols, xq, y, batch, stream=stream))):
        ts = []
        for i in range(3 + max(reps, 10)):
            flush.fill_(0)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            call()
            e1.record(stream)
            torch.cuda.synchronize()
            if i >= 3:
                ts.append(e0.elapsed_time(e1) / 1e3)
        res[name] = {"us": round(statistics.median(ts) * 1e6, 2)}
    by = qd.packed_bytes(fmt, rows, cols) + xq.numel() + 4 * batch * rows
    t = res["product"]["us"] / 1e6
    res["product"].update({"algorithmic_bytes": int(by), "GB/s": round(by / t / 1e9, 1),
                           "frac": round(by / t / 1e9 / hbm, 4)})
    print(json.dumps({"q8act": spec, **res, "peak": hbm, "peak_kind": kind}))


def run_quantize_only(spec: str, reps: int):
    """The BF16 -> INT8 quantiser alone at ROWSxCOLS; prints one JSON line (not the
    benchmark contract line)."""
    import torch

    import quantized_decode_gemv_gb300 as qd

    rows, cols = (int(v) for v in spec.split("x"))
    if not os.path.exists(qd.LIB_PATH):
        qd.build()
    qd.load()
    hbm, _, kind = peaks()
    print(json.dumps({"quantize_i8": bench_quantize(qd, torch, rows, cols, hbm, max(reps, 3)), "peak": hbm,
                      "peak_kind": kind}))


def run_1p7b_only(spec: str, layers=None, kv_f16=False):
    """The 1.7B-shaped INT8 step alone at the given batches ("1", "16" or "1,16"), optionally
    with fewer layers (a small case for profiling); prints one JSON line (not the benchmark
    contract line)."""
    import torch

    import quantized_decode_gemv_gb300 as qd

    if not os.path.exists(qd.LIB_PATH):
        qd.build()
    qd.load()
    stream = torch.cuda.current_stream()
    hbm, _, kind = peaks()
    res = bench_1p7b(qd, torch, stream, None, hbm, tuple(int(b) for b in spec.split(",")), layers, kv_f16)
    print(json.dumps({"decode_1p7b": res, "layers": layers, "peak": hbm, "peak_kind": kind}))


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--quick", action="store_true", help="main line only (no sweep, 1.7B, CPU baseline)")
    ap.add_argument("--no-1p7b", action="store_true")
    ap.add_argument("--full-sweep", action="store_true", help="q_gemv sweep: both launch modes at every batch size")
    ap.add_argument("--batch1-sweep", action="store_true", help="q_gemv sweep at batch 1 only")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--ref-tokens", type=int, default=8)
    ap.add_argument("--gemv", default=None, help="microbenchmark one shape, FMT:ROWSxCOLS:BATCH")
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--no-ceiling", action="store_true", help="with --gemv: skip the plain-read ceiling")
    ap.add_argument("--decode-1p7b", default=None, help="the 1.7B-shaped step alone, at batches e.g. 1,16")
    ap.add_argument("--layers", type=int, default=None, help="with --decode-1p7b: fewer layers (profiling)")
    ap.add_argument("--quantize", default=None, help="the BF16 -> INT8 quantiser alone at ROWSxCOLS")
    ap.add_argument("--gemm", default=None, help="the prefill product alone, FMT:ROWSxCOLS:TOKENS")
    ap.add_argument("--q8act", default=None, help="the ggml-exact activation path alone, FMT:ROWSxCOLS:BATCH")
    ap.add_argument("--modes-135m", action="store_true", help="135M decode in the default and ggml-exact modes")
    ap.add_argument("--prefill-135m", action="store_true", help="the 135M prompt through qd_prefill alone")
    ap.add_argument("--kv-f16", action="store_true", help="with --decode-1p7b: binary16 KV cache")
    ap.add_argument("--step-path", choices=["chain", "cluster"], default=None,
                    help="force the 135M decode step's path (default: the library's choice)")
    args = ap.parse_args(argv)
    if args.gemv:
        run_gemv_only(args.gemv, args.reps, ceiling=not args.no_ceiling)
        return
    if args.decode_1p7b:
        run_1p7b_only(args.decode_1p7b, args.layers, args.kv_f16)
        return
    if args.quantize:
        run_quantize_only(args.quantize, args.reps)
        return
    if args.gemm:
        run_gemm_only(args.gemm, args.reps)
        return
    if args.q8act:
        run_q8act_only(args.q8act, args.reps)
        return
    if args.prefill_135m:
        import torch

        import quantized_decode_gemv_gb300 as qd

        qd.load()
        print(json.dumps({"prefill_135m": bench_prefill_135m(qd, torch, torch.cuda.current_stream())}))
        return
    if args.modes_135m:
        import torch

        import quantized_decode_gemv_gb300 as qd

        qd.load()
        print(json.dumps({"decode_135m_modes": bench_135m_modes(qd, torch, torch.cuda.current_stream())}))
        return
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    world, rank, local = dist_env()
    if args.impl == "reference":
        run_reference(args, world, rank, local)
    else:
        run_ours(args, world, rank, local)


if __name__ == "__main__":
    main()
