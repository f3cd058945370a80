"""Benchmark of the KV-cache codec hot path: NVFP4 quant-scatter + paged restore.

Workload: the long-context prefill case -- 1,048,576 tokens x 4 KV heads x head_dim
256, bf16 N(0,1) with 0.5% of entries x50, quantised into a 1,048,576-slot paged
NVFP4 pool (block size 16, slots shuffled at block granularity), then restored in
full through the block table.  A step is one quant-scatter of K and V plus one
restore of K and V.  Inputs (4 GiB) and outputs (4 GiB) are far larger than L2,
so no flush is needed between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl {ours,reference}]

Prints one JSON line.  ``value`` is codec GB/s (algorithmic bytes read + written by
both kernels / device time), summed over ranks for N > 1 (weak scaling: each rank
runs its own copy of the workload, no collective on the data path).  The
reference arm (``--impl reference``) times the scalar CPU definition of the codec
on every host core at once (one thread per core) over a bounded sample of the same
workload.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "KV codec GB/s (NVFP4 quant-scatter + paged restore), % of GB300 HBM peak"
T_TOKENS, HEADS, HEAD_DIM, BLOCK = 1 << 20, 4, 256, 16
SEED = 5
WORKLOAD = ("long-context prefill: 1,048,576 tokens x 4 KV heads x head_dim 256 bf16 "
            "(N(0,1), 0.5% x50 outliers) -> NVFP4 quant-scatter into a 1,048,576-slot paged "
            "pool (block 16, block-shuffled slots) -> full paged restore to bf16")


# ---------------------------------------------------------------------------
# algorithmic bytes
# ---------------------------------------------------------------------------
def row_bytes(D: int) -> int:
    return D // 2 + D // 16 + 4


def scatter_bytes(T: int, H: int, D: int, tensors: int = 2) -> int:
    """bf16 read + NVFP4 written per row, plus the int64 slot id per token."""
    return tensors * T * H * (2 * D + row_bytes(D)) + 8 * T


def restore_bytes(T: int, H: int, D: int, nblocks: int, S: int = 1, tensors: int = 2) -> int:
    """NVFP4 read + bf16 written per row, plus the int32 block table and lengths."""
    return tensors * T * H * (row_bytes(D) + 2 * D) + 4 * nblocks + 4 * S


# ---------------------------------------------------------------------------
# distributed plumbing (one process per GPU, weak scaling)
# ---------------------------------------------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world: int, backend: str):
    if world > 1:
        import torch.distributed as dist

        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
        return dist
    return None


def barrier(dist, device=None):
    if dist is not None:
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def max_over_ranks(dist, value: float, device) -> float:
    if dist is None:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# clocks sampled while the timed region runs
# ---------------------------------------------------------------------------
REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]


class ClockSampler:
    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.samples = []
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        q = "timestamp,clocks.sm,clocks.max.sm,power.draw," + ",".join(
            "clocks_event_reasons." + r for r in REASONS)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.4)

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def mark(self, begin: bool):
        if begin:
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = [s for (ts, s) in self.samples if self.t0 - 0.15 <= ts <= self.t1 + 0.15]
        sm, mx, reasons = [], [], set()
        for r in rows:
            parts = [p.strip() for p in r.split(",")]
            if len(parts) < 4 + len(REASONS):
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(REASONS, parts[4:]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def gpu_id_for(device) -> str:
    try:
        uuid = str(torch.cuda.get_device_properties(device).uuid)
        return uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        return str(device.index or 0)


# ---------------------------------------------------------------------------
# roofline inputs
# ---------------------------------------------------------------------------
def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def sources_hash(paths) -> str:
    """sha256 (16 hex digits) of the concatenated kernel sources a capture measured."""
    import hashlib

    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def nearest_rank(xs, q: float) -> float:
    """The q-quantile of xs by the nearest-rank rule (the smallest value with at least
    a fraction q of the values at or below it)."""
    ys = sorted(xs)
    return ys[min(len(ys) - 1, max(0, math.ceil(q * len(ys)) - 1))]


def kernel_row(times_ms, nbytes: int, peak: float) -> dict:
    """One kernel's line: mean, P50 and P90 of its per-step event times, and the
    mean's bandwidth as GB/s and as a fraction of the peak."""
    ms = sum(times_ms) / len(times_ms)
    return {"ms": round(ms, 4), "p50_ms": round(nearest_rank(times_ms, 0.5), 4),
            "p90_ms": round(nearest_rank(times_ms, 0.9), 4), "bytes": nbytes,
            "GB/s": round(nbytes / ms / 1e6, 1), "frac": round(nbytes / ms / 1e6 / peak, 4)}


def ncu_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    kernel source changed since the capture."""
    import hashlib

    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        rec = d[kernel]
        if sources_hash(rec["sources"]) != rec["sources_sha256_16"]:
            return None
        return int(rec["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


# ---------------------------------------------------------------------------
# the workload
# ---------------------------------------------------------------------------
def make_workload(device, seed=SEED, T=T_TOKENS, H=HEADS, D=HEAD_DIM, bs=BLOCK):
    from quantized_kv_cache_nvfp4_gb300 import synth

    nblocks = T // bs
    perm = synth.block_permutation(nblocks, seed).to(device)
    t = torch.arange(T, device=device)
    slots = (perm[t // bs].long() * bs + t % bs).contiguous()
    k = synth.normal_bf16((T, H, D), seed, synth.STREAM_K, 0.005, 50.0, device=str(device))
    v = synth.normal_bf16((T, H, D), seed, synth.STREAM_V, 0.005, 50.0, device=str(device))
    table = perm.view(1, nblocks).contiguous()
    lens = torch.tensor([T], dtype=torch.int32, device=device)
    return k, v, slots, table, lens


def run_ours(args):
    import quantized_kv_cache_nvfp4_gb300 as kvq

    world, rank, local = dist_env()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    dist = init_dist(world, "nccl")
    T, H, D, bs = args.tokens, HEADS, HEAD_DIM, BLOCK
    nblocks = T // bs
    k, v, slots, table, lens = make_workload(device, seed=SEED + 1000 * rank, T=T)
    pool = kvq.Nvfp4Pool.empty(T, H, D, bs, device=device)
    ko = torch.empty((1, T, H, D), dtype=torch.bfloat16, device=device)
    vo = torch.empty_like(ko)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    stream = torch.cuda.current_stream(device)

    def step():
        kvq.kvq_quant_scatter(k, v, slots, pool, status)
        kvq.kvq_restore(pool, table, lens, T, ko, vo, status)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert int(status.item()) == 0, "device status flagged an error"

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    sampler = ClockSampler(gpu_id_for(device)) if rank == 0 else None
    if sampler:
        sampler.start()
    barrier(dist, device)
    torch.cuda.synchronize()
    if sampler:
        sampler.mark(True)
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(K):
        ev[i][0].record(stream)
        kvq.kvq_quant_scatter(k, v, slots, pool, status)
        ev[i][1].record(stream)
        kvq.kvq_restore(pool, table, lens, T, ko, vo, status)
        ev[i][2].record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    if sampler:
        sampler.mark(False)
    barrier(dist, device)
    total_ms = start.elapsed_time(end)
    scat_t = [e[0].elapsed_time(e[1]) for e in ev]
    rest_t = [e[1].elapsed_time(e[2]) for e in ev]
    scat_ms, rest_ms = sum(scat_t) / K, sum(rest_t) / K
    total_ms = max_over_ranks(dist, total_ms, device)
    clocks = sampler.stop() if sampler else None

    # information: reconstruction RMSE against the bf16 input, and the status word
    rmse = float((vo[0].float() - v.float()).pow(2).mean().sqrt().item())
    st_final = int(status.item())

    e2e = run_e2e(args, kvq, device, k, v, slots, table, lens, pool, dist, T) if not args.no_e2e else None
    rows_other = None
    if not args.no_other_rows and rank == 0:
        rows_other = other_rows(kvq, device, peak=measured_peaks()[0])
        rows_other["latency_us_one_residual_loop"] = residual_loop_latency(kvq, device)
        rows_other["decode_attention"] = attention_rows(kvq, device, peak=measured_peaks()[0])
        rows_other["decode_step_store"] = decode_step_latency(kvq, device)
        try:  # an auxiliary latency row: a failure is reported in the line, not fatal
            rows_other["one_layer_latency"] = one_layer_latency(kvq, device)
        except Exception as e:  # noqa: BLE001
            rows_other["one_layer_latency"] = {"error": f"{type(e).__name__}: {e}"}

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return
    sb, rb = scatter_bytes(T, H, D), restore_bytes(T, H, D, nblocks)
    step_bytes = sb + rb
    ms_per_step = total_ms / K
    value = world * step_bytes / (ms_per_step * 1e-3) / 1e9
    peak, peak_kind = measured_peaks()
    dom, dom_ms, dom_bytes = ("kvq_restore", rest_ms, rb) if rest_ms >= scat_ms else ("kvq_quant_scatter", scat_ms, sb)
    achieved = dom_bytes / (dom_ms * 1e-3) / 1e9
    cpu = cpu_baseline(args) if not args.no_cpu_baseline else None
    out = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded N(0,1) bf16 with 0.5% x50 outliers, generated on the GPU)",
        "config": {
            "workload": WORKLOAD if T == T_TOKENS else WORKLOAD.replace("1,048,576", f"{T:,}"), "tokens": T, "kv_heads": H, "head_dim": D, "block_size": BLOCK,
            "pool_slots": T, "parallelism": f"replicas x{world}", "l2": "inputs and outputs larger than L2 (no flush)",
            "bytes_per_step": step_bytes,
        },
        "frac_of_hbm_peak": round(value / world / peak, 4),
        "rows_per_s": round(world * 4 * T * H / (ms_per_step * 1e-3), 1),
        "kernels": {
            "kvq_quant_scatter": kernel_row(scat_t, sb, peak),
            "kvq_restore": kernel_row(rest_t, rb, peak),
        },
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1), "peak": peak,
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured" else "fallback",
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": ncu_traffic(dom)},
        "gpu_launches": 2 * K,
        "rmse_v": round(rmse, 5),
        "device_status": st_final,
        "clocks": clocks,
        "e2e": e2e,
        "other_rows": rows_other,
        "cpu_baseline": cpu,
    }
    print(json.dumps(out), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def run_e2e(args, kvq, device, k, v, slots, table, lens, pool, dist, T):
    """Same metric through the public API with host buffers.

    Every step copies the step's inputs host->device from pinned memory (K, V, slot
    ids, block table, lengths) and the restored K/V device->host.  The step is cut
    into chunks of tokens on three streams, so that the copy-in of chunk c+1, the
    scatter + restore of chunk c and the copy-out of chunk c-1 overlap (the two copy
    directions run concurrently on the host link).  Chunk c's restore reads the
    block-table slice of its own tokens, so the chunks together do exactly the work
    of one scatter and one restore of the whole workload."""
    H, D = HEADS, HEAD_DIM
    nch = max(1, args.e2e_chunks)
    while T % (nch * BLOCK) != 0:
        nch -= 1
    C = T // nch
    hk = torch.empty(k.shape, dtype=k.dtype, pin_memory=True)
    hv = torch.empty(v.shape, dtype=v.dtype, pin_memory=True)
    hs = torch.empty(slots.shape, dtype=slots.dtype, pin_memory=True)
    ht = torch.empty(table.shape, dtype=table.dtype, pin_memory=True)
    hl = torch.full((nch,), C, dtype=torch.int32).pin_memory()
    hk.copy_(k)
    hv.copy_(v)
    hs.copy_(slots)
    ht.copy_(table)
    ok = torch.empty((T, H, D), dtype=torch.bfloat16, pin_memory=True)
    ov = torch.empty((T, H, D), dtype=torch.bfloat16, pin_memory=True)  # empty_like would not pin
    dk, dv, ds, dt = (torch.empty_like(x) for x in (k, v, slots, table))
    dl = torch.empty((nch,), dtype=torch.int32, device=device)
    yk = torch.empty((T, H, D), dtype=torch.bfloat16, device=device)
    yv = torch.empty_like(yk)
    s_in, s_cmp, s_out = (torch.cuda.Stream(device) for _ in range(3))
    ev = lambda: torch.cuda.Event()
    consumed = [ev() for _ in range(nch)]  # the scatter of chunk c read its inputs
    restored = [ev() for _ in range(nch)]  # the restore of chunk c wrote its output
    shipped = [ev() for _ in range(nch)]   # the copy-out of chunk c finished
    arrived = [ev() for _ in range(nch)]   # the copy-in of chunk c finished
    bpc = C // BLOCK
    first = [True]

    def step():
        for c in range(nch):
            sl = slice(c * C, (c + 1) * C)
            with torch.cuda.stream(s_in):
                if not first[0]:
                    s_in.wait_event(consumed[c])
                dk[sl].copy_(hk[sl], non_blocking=True)
                dv[sl].copy_(hv[sl], non_blocking=True)
                ds[sl].copy_(hs[sl], non_blocking=True)
                dt[:, c * bpc:(c + 1) * bpc].copy_(ht[:, c * bpc:(c + 1) * bpc], non_blocking=True)
                dl[c:c + 1].copy_(hl[c:c + 1], non_blocking=True)
                arrived[c].record(s_in)
            with torch.cuda.stream(s_cmp):
                s_cmp.wait_event(arrived[c])
                if not first[0]:
                    s_cmp.wait_event(shipped[c])
                kvq.kvq_quant_scatter(dk[sl], dv[sl], ds[sl], pool, stream=s_cmp)
                consumed[c].record(s_cmp)
                kvq.kvq_restore(pool, dt[:, c * bpc:(c + 1) * bpc], dl[c:c + 1], C,
                                yk[sl].unsqueeze(0), yv[sl].unsqueeze(0), stream=s_cmp)
                restored[c].record(s_cmp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(restored[c])
                ok[sl].copy_(yk[sl], non_blocking=True)
                ov[sl].copy_(yv[sl], non_blocking=True)
                shipped[c].record(s_out)
        first[0] = False

    for _ in range(max(1, min(args.warmup, 2))):
        step()
    torch.cuda.synchronize(device)
    K = max(1, min(args.steps, args.e2e_steps))
    barrier(dist, device)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    cur = torch.cuda.current_stream(device)
    t0.record(cur)
    for st in (s_in, s_cmp, s_out):
        st.wait_event(t0)
    for _ in range(K):
        step()
    for e in shipped:
        cur.wait_event(e)
    t1.record(cur)
    torch.cuda.synchronize(device)
    ms = max_over_ranks(dist, t0.elapsed_time(t1) / K, device)
    # the host copy of the restored V equals what the device restored
    same = bool(torch.equal(ov[: 4096].to(device).view(torch.int16), yv[:4096].view(torch.int16)))
    world = dist.get_world_size() if dist is not None else 1
    step_bytes = scatter_bytes(T, H, D) + restore_bytes(T, H, D, T // BLOCK)
    bi = sum(x.numel() * x.element_size() for x in (hk, hv, hs, ht)) + 4 * nch
    bo = ok.numel() * ok.element_size() * 2
    return {"value": round(world * step_bytes / (ms * 1e-3) / 1e9, 1), "unit": "GB/s",
            "ms_per_step": round(ms, 3), "steps": K, "chunks": nch, "streams": 3,
            "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
            "h2d_plus_d2h_GBps": round((bi + bo) / (ms * 1e-3) / 1e9, 1), "output_matches": same}


# ---------------------------------------------------------------------------
# the other rows of the hot path: INT4 and NVFP4 logical codecs, residuals
# ---------------------------------------------------------------------------
def int4_meta_bytes(kind: int, rows: int, H: int, D: int, G: int) -> int:
    groups = (-(-rows // G)) * H * D if kind == 0 else rows * H * (-(-D // G))
    return 4 * groups


def other_rows(kvq, device, T=262144, H=8, D=128, G=64, P=None, iters=20, peak=6795.5):
    """GB/s of every other entry point on a [T, H, D] bf16 case (inputs far larger
    than L2), each timed alone with CUDA events over `iters` back-to-back calls."""
    from quantized_kv_cache_nvfp4_gb300 import synth

    P = P if P is not None else T // 4
    cur, prev = synth.layer_kv(T, H, D, seed=4, device=str(device))
    pos = synth.sorted_positions(T, P, 4).to(device)
    y = torch.empty_like(cur)
    out = {}

    def timed(name, fn, nbytes):
        for _ in range(3):
            fn()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(iters):
            fn()
        b.record()
        torch.cuda.synchronize(device)
        ms = a.elapsed_time(b) / iters
        out[name] = {"ms": round(ms, 4), "bytes": nbytes, "GB/s": round(nbytes / ms / 1e6, 1),
                     "frac": round(nbytes / ms / 1e6 / peak, 4)}

    rows_b = T * H * 2 * D  # bf16 bytes of the whole tensor
    nv = kvq.Packed.empty(kvq.FMT_NVFP4, 0, T, H, D, device=device)
    nvb = T * H * (D // 2 + D // 16 + 4)
    timed("kvq_pack nvfp4", lambda: kvq.kvq_pack(cur, nv), rows_b + nvb)
    timed("kvq_unpack nvfp4", lambda: kvq.kvq_unpack(nv, y), nvb + rows_b)
    for kind, kname in ((0, "key"), (1, "value")):
        pk = kvq.Packed.empty(kvq.FMT_INT4, kind, T, H, D, G, device=device)
        ib = T * H * (D // 2) + int4_meta_bytes(kind, T, H, D, G)
        timed(f"kvq_pack int4 {kname} G{G}", lambda: kvq.kvq_pack(cur, pk), rows_b + ib)
        timed(f"kvq_unpack int4 {kname} G{G}", lambda: kvq.kvq_unpack(pk, y), ib + rows_b)
        pay = kvq.Packed.empty(kvq.FMT_INT4, kind, P, H, D, G, device=device)
        pb = P * H * (D // 2) + int4_meta_bytes(kind, P, H, D, G)
        kept_b = P * H * 2 * D
        timed(f"kvq_encode_residual int4 {kname} 25%", lambda: kvq.kvq_encode_residual(cur, prev, pos, pay),
              2 * kept_b + 4 * P + pb)
        timed(f"kvq_decode_residual int4 {kname} 25% copy", lambda: kvq.kvq_decode_residual(pay, pos, prev, y),
              rows_b + pb + 4 * P + rows_b)
        ip = prev.clone()
        timed(f"kvq_decode_residual int4 {kname} 25% in place",
              lambda: kvq.kvq_decode_residual(pay, pos, ip, ip), kept_b + pb + 4 * P + kept_b)
    pay = kvq.Packed.empty(kvq.FMT_NVFP4, 0, P, H, D, device=device)
    pb = P * H * (D // 2 + D // 16 + 4)
    timed("kvq_encode_residual nvfp4 25%", lambda: kvq.kvq_encode_residual(cur, prev, pos, pay),
          2 * P * H * 2 * D + 4 * P + pb)
    timed("kvq_decode_residual nvfp4 25% copy", lambda: kvq.kvq_decode_residual(pay, pos, prev, y),
          rows_b + pb + 4 * P + rows_b)
    # FP8 E4M3 rows: D code bytes + one FP32 scale per (token, head)
    f8 = kvq.Packed.empty(kvq.FMT_FP8, 0, T, H, D, device=device)
    f8b = T * H * (D + 4)
    timed("kvq_pack fp8", lambda: kvq.kvq_pack(cur, f8), rows_b + f8b)
    timed("kvq_unpack fp8", lambda: kvq.kvq_unpack(f8, y), f8b + rows_b)
    nblk = -(-T // 16)
    perm = synth.block_permutation(nblk, 4).to(device)
    t = torch.arange(T, device=device)
    slots = perm[t // 16].long() * 16 + t % 16
    pool = kvq.KvPool.empty(nblk * 16, H, D, 16, device=device, fmt=kvq.FMT_FP8)
    timed("kvq_quant_scatter fp8 (K only)", lambda: kvq.kvq_quant_scatter(cur, None, slots, pool),
          rows_b + 8 * T + f8b)
    lens = torch.tensor([T], dtype=torch.int32, device=device)
    table = perm.view(1, -1).contiguous()
    timed("kvq_restore fp8 (K only)", lambda: kvq.kvq_restore(pool, table, lens, T, y, None),
          f8b + 4 * nblk + rows_b)
    pay = kvq.Packed.empty(kvq.FMT_FP8, 0, P, H, D, device=device)
    pb = P * H * (D + 4)
    timed("kvq_encode_residual fp8 25%", lambda: kvq.kvq_encode_residual(cur, prev, pos, pay),
          2 * P * H * 2 * D + 4 * P + pb)
    timed("kvq_decode_residual fp8 25% copy", lambda: kvq.kvq_decode_residual(pay, pos, prev, y),
          rows_b + pb + 4 * P + rows_b)
    # NVFP4 with one FP32 scale per tensor: pack reads the tensor twice (the amax pass,
    # then the block encode); blocks run over 16 token rows (K) or 16 channels (V)
    for kind, kname in ((0, "key"), (1, "value")):
        nt = kvq.Packed.empty(kvq.FMT_NVFP4_TENSOR, kind, T, H, D, device=device)
        ntb = T * H * (D // 2) + (-(-T // 16) * H * D if kind == 0 else T * H * (D // 16)) + 4
        timed(f"kvq_pack nvfp4_tensor {kname}", lambda: kvq.kvq_pack(cur, nt), 2 * rows_b + ntb)
        timed(f"kvq_unpack nvfp4_tensor {kname}", lambda: kvq.kvq_unpack(nt, y), ntb + rows_b)
    return {"workload": f"[{T} tokens, {H} KV heads, D{D}] bf16, INT4 G{G}, residual rows kept {P}/{T}",
            "kernels": out}


def attention_rows(kvq, device, peak=6795.5, iters=20, S=32, T=8192, H=8, Hq=32, D=128):
    """Decode attention reading the quantised pool (K and V decoded in registers) on the
    paged-restore workload's pool: S sequences x T tokens, H KV heads, Hq query heads,
    D128.  Bytes: the pool rows read (K and V) + q + out + block table.  The unfused
    path (restore to bf16, then torch SDPA) is timed beside it for context."""
    import math

    from quantized_kv_cache_nvfp4_gb300 import synth

    bs = BLOCK
    nblocks = S * T // bs
    perm = synth.block_permutation(nblocks, 3).to(device)
    table = perm.view(S, T // bs).contiguous()
    t = torch.arange(T, device=device)
    slots = (table[:, t // bs].long() * bs + t % bs).reshape(-1)
    lens = torch.full((S,), T, dtype=torch.int32, device=device)
    q = synth.normal_bf16((S, Hq, D), 3, 9, device=str(device))
    out = torch.empty_like(q)
    res = {}
    for name, fk, fv in (("nvfp4", kvq.FMT_NVFP4, None), ("fp8", kvq.FMT_FP8, None),
                         ("k8v4 (FP8 K, NVFP4 V)", kvq.FMT_FP8, kvq.FMT_NVFP4)):
        pool = kvq.KvPool.empty(nblocks * bs, H, D, bs, device=device, fmt=fk, v_fmt=fv)
        k = synth.normal_bf16((S * T, H, D), 3, synth.STREAM_K, device=str(device))
        v = synth.normal_bf16((S * T, H, D), 3, synth.STREAM_V, device=str(device))
        kvq.kvq_quant_scatter(k, v, slots, pool)
        del k, v
        ws = torch.empty(max(kvq.kvq_decode_attention_workspace(S, H, Hq, D, T), 16), dtype=torch.uint8,
                         device=device)
        fn = lambda: kvq.kvq_decode_attention(pool, table, lens, T, q, 1.0 / math.sqrt(D), out, workspace=ws)
        for _ in range(3):
            fn()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(iters):
            fn()
        b.record()
        torch.cuda.synchronize(device)
        ms = a.elapsed_time(b) / iters
        nbytes = pool.nbytes() + 2 * q.numel() * 2 + table.numel() * 4
        res[f"kvq_decode_attention {name}"] = {"ms": round(ms, 4), "bytes": nbytes,
                                               "GB/s": round(nbytes / ms / 1e6, 1),
                                               "frac": round(nbytes / ms / 1e6 / peak, 4)}
        if name == "nvfp4":  # the paged restore of the same pool, then the unfused path
            ko = torch.empty((S, T, H, D), dtype=torch.bfloat16, device=device)
            vo = torch.empty_like(ko)
            for _ in range(3):
                kvq.kvq_restore(pool, table, lens, T, ko, vo)
            a.record()
            for _ in range(iters):
                kvq.kvq_restore(pool, table, lens, T, ko, vo)
            b.record()
            torch.cuda.synchronize(device)
            ms = a.elapsed_time(b) / iters
            rb = restore_bytes(S * T, H, D, nblocks, S)
            res[f"kvq_restore nvfp4 ({S} x {T} tokens)"] = {"ms": round(ms, 4), "bytes": rb,
                                                           "GB/s": round(rb / ms / 1e6, 1),
                                                           "frac": round(rb / ms / 1e6 / peak, 4)}

            def unfused():
                kvq.kvq_restore(pool, table, lens, T, ko, vo)
                kk = ko.permute(0, 2, 1, 3).repeat_interleave(Hq // H, dim=1)
                vv = vo.permute(0, 2, 1, 3).repeat_interleave(Hq // H, dim=1)
                return torch.nn.functional.scaled_dot_product_attention(q[:, :, None], kk, vv,
                                                                        scale=1.0 / math.sqrt(D))

            for _ in range(2):
                unfused()
            a.record()
            for _ in range(5):
                unfused()
            b.record()
            torch.cuda.synchronize(device)
            res["unfused restore + torch SDPA (nvfp4)"] = {"ms": round(a.elapsed_time(b) / 5, 4)}
            del ko, vo
        del pool
    return {"workload": f"decode attention: {S} sequences x {T} tokens, {H} KV heads, {Hq} query heads, "
                        f"D{D}, block size {bs}, shuffled block table", "kernels": res}


def decode_step_latency(kvq, device, iters=200):
    """The decode-step store: 256 requests append one token each (H8, D128), K a view
    of a fused qkv tensor (row pitch 1152), V its own tensor, into a 65,536-slot pool;
    the quant-scatter captured in a CUDA graph, microseconds per replay."""
    from quantized_kv_cache_nvfp4_gb300 import synth

    qkv, _, v, slots = synth.decode_step_case(seed=2)
    qkv, v, slots = qkv.to(device), v.to(device), slots.to(device)
    k = qkv[:, :1024].unflatten(1, (8, 128))
    pool = kvq.Nvfp4Pool.empty(65536, 8, 128, BLOCK, device=device)
    stream = torch.cuda.Stream(device)
    with torch.cuda.stream(stream):
        for _ in range(3):
            kvq.kvq_quant_scatter(k, v, slots, pool, stream=stream)
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        kvq.kvq_quant_scatter(k, v, slots, pool, stream=stream)
    for _ in range(10):
        graph.replay()
    torch.cuda.synchronize(device)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(iters):
        graph.replay()
    b.record()
    torch.cuda.synchronize(device)
    replay_us = a.elapsed_time(b) / iters * 1000
    # the same call made eagerly, back to back through the Python binding and the C ABI:
    # device time per call between events, and host time per call (argument checks,
    # marshalling and the launch)
    with torch.cuda.stream(stream):
        a.record(stream)
        t0 = time.perf_counter()
        for _ in range(iters):
            kvq.kvq_quant_scatter(k, v, slots, pool, stream=stream)
        host_s = time.perf_counter() - t0
        b.record(stream)
    torch.cuda.synchronize(device)
    return {"workload": "256 tokens x 8 KV heads x D128 (K a view of qkv [256, 1152]) into a 65,536-slot pool, "
                        "one graph replay", "us_per_replay": round(replay_us, 2),
            "eager_us_per_call": round(a.elapsed_time(b) / iters * 1000, 2),
            "eager_host_us_per_call": round(host_s / iters * 1e6, 2),
            "bytes": scatter_bytes(256, 8, 128)}


def one_layer_latency(kvq, device, iters=200):
    """The one-layer parity case as a latency row: K, V [256, 8, 128] (N(0,1), 1% x20)
    quant-scattered into a 256-slot pool (16 blocks, slots 0..255), then restored
    through the identity block table; each call captured in a CUDA graph, microseconds
    per replay."""
    from quantized_kv_cache_nvfp4_gb300 import synth

    k, v, slots = synth.one_layer_case(seed=0)
    k, v, slots = k.to(device), v.to(device), slots.to(device)
    pool = kvq.Nvfp4Pool.empty(256, 8, 128, BLOCK, device=device)
    table = torch.arange(256 // BLOCK, dtype=torch.int32, device=device).view(1, 256 // BLOCK)
    lens = torch.tensor([256], dtype=torch.int32, device=device)
    ko = torch.empty((1, 256, 8, 128), dtype=torch.bfloat16, device=device)
    vo = torch.empty_like(ko)
    stream = torch.cuda.Stream(device)
    calls = (("kvq_quant_scatter", lambda: kvq.kvq_quant_scatter(k, v, slots, pool, stream=stream)),
             ("kvq_restore", lambda: kvq.kvq_restore(pool, table, lens, 256, ko, vo, stream=stream)))
    out = {"workload": "K, V [256, 8, 128] into a 256-slot pool and back, one graph replay per call"}
    for name, fn in calls:
        with torch.cuda.stream(stream):
            for _ in range(3):
                fn()
        stream.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            fn()
        for _ in range(10):
            graph.replay()
        torch.cuda.synchronize(device)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(iters):
            graph.replay()
        b.record()
        torch.cuda.synchronize(device)
        out[name + "_us"] = round(a.elapsed_time(b) / iters * 1000, 2)
    return out


def residual_loop_latency(kvq, device, iters=50):
    """Microseconds per call on one residual loop of the INT4 + residual case:
    [4096, 8, 128], 1024 kept rows (the sizes of the pages' loop study)."""
    r = other_rows(kvq, device, T=4096, H=8, D=128, G=64, P=1024, iters=iters)
    return {k: round(v["ms"] * 1000, 2) for k, v in r["kernels"].items()}


# ---------------------------------------------------------------------------
# CPU definition of the codec (the oracle) on the host cores
# ---------------------------------------------------------------------------
def oracle_sample(tokens: int, seed=SEED, H=HEADS, D=HEAD_DIM, bs=BLOCK):
    """A bounded sample of the workload: the first `tokens` tokens with their own
    block-shuffled pool of tokens/16 blocks (same shapes, same generator recipe)."""
    from quantized_kv_cache_nvfp4_gb300 import synth

    nb = tokens // bs
    perm = synth.block_permutation(nb, seed).numpy()
    t = np.arange(tokens)
    slots = (perm[t // bs].astype(np.int64) * bs + t % bs)
    k = synth.bf16_bits(synth.normal_bf16((tokens, H, D), seed, synth.STREAM_K, 0.005, 50.0))
    v = synth.bf16_bits(synth.normal_bf16((tokens, H, D), seed, synth.STREAM_V, 0.005, 50.0))
    return k, v, slots, perm.reshape(1, nb).astype(np.int32)


def oracle_step(O, k, v, slots, table, H=HEADS, D=HEAD_DIM, bs=BLOCK):
    tokens = k.shape[0]
    pool_k, pool_v = O.new_pool(tokens, H, D), O.new_pool(tokens, H, D)
    O.nvfp4_scatter(k, H * D, D, tokens, H, D, slots, pool_k)
    O.nvfp4_scatter(v, H * D, D, tokens, H, D, slots, pool_v)
    lens = np.array([tokens], np.int32)
    O.nvfp4_restore(pool_k, bs, table, lens, tokens)
    O.nvfp4_restore(pool_v, bs, table, lens, tokens)


def oracle_gbs(tokens: int, seconds: float) -> float:
    H, D = HEADS, HEAD_DIM
    b = scatter_bytes(tokens, H, D) + restore_bytes(tokens, H, D, tokens // BLOCK)
    return b / seconds / 1e9


def host_cores() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except (AttributeError, OSError):
        return max(1, os.cpu_count() or 1)


def oracle_all_cores(O, sample, threads: int) -> float:
    """Wall seconds of `threads` oracle steps run at once, one per host thread, each on
    the same read-only sample into its own pools and outputs (the C oracle keeps no
    global state and ctypes releases the interpreter lock during each call)."""
    import threading

    k, v, slots, table = sample
    go = threading.Barrier(threads + 1)

    def work():
        go.wait()
        oracle_step(O, k, v, slots, table)

    ts = [threading.Thread(target=work) for _ in range(threads)]
    for t in ts:
        t.start()
    go.wait()
    t0 = time.perf_counter()
    for t in ts:
        t.join()
    return time.perf_counter() - t0


def cpu_baseline(args):
    import oracle as O

    tokens = args.cpu_tokens
    sample = oracle_sample(tokens)
    t0 = time.perf_counter()
    oracle_step(O, *sample)
    dt = time.perf_counter() - t0
    n = host_cores()
    dt_all = oracle_all_cores(O, sample, n)
    return {"value": round(oracle_gbs(tokens, dt), 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "seconds": round(dt, 2),
            "sample": f"first {tokens} tokens of the workload (x4 heads x D256, K and V) with their own "
                      f"block-shuffled {tokens // BLOCK}-block pool: scatter + restore, single-threaded scalar C",
            "all_cores": {"value": round(n * oracle_gbs(tokens, dt_all), 4), "unit": "GB/s", "cores": n,
                          "seconds": round(dt_all, 2),
                          "sample": f"the same sample on {n} host threads at once, one oracle step each"}}


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle as O

    # calibrate: per-token cost of one scatter + restore of K and V
    k, v, slots, table = oracle_sample(256)
    t0 = time.perf_counter()
    oracle_step(O, k, v, slots, table)
    per_tok = (time.perf_counter() - t0) / 256
    budget = args.ref_seconds / max(1, args.steps + args.warmup)
    n = host_cores()
    tokens = int(max(BLOCK, min(32768, budget / per_tok)) // BLOCK * BLOCK)
    sample = oracle_sample(tokens)
    for _ in range(args.warmup):
        oracle_all_cores(O, sample, n)
    dt = sum(oracle_all_cores(O, sample, n) for _ in range(args.steps)) / args.steps
    val = n * oracle_gbs(tokens, dt)
    sample = (f"first {tokens} tokens of the workload (x4 heads x D256, K and V) with their own "
              f"block-shuffled pool, on {n} host threads at once: scatter + restore per thread, scalar C")
    out = {
        "impl": "reference", "metric": METRIC, "value": round(val, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded N(0,1) bf16 with 0.5% x50 outliers)",
        "config": {"workload": WORKLOAD, "tokens": T_TOKENS, "kv_heads": HEADS, "head_dim": HEAD_DIM,
                   "block_size": BLOCK, "sample_tokens_per_step": tokens},
        "cpu_baseline": {"value": round(val, 4), "unit": "GB/s", "cores": n, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(val, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(out), flush=True)


CASES = ("attention_nvfp4", "attention_fp8", "attention_k8v4",
         "scatter_nvfp4", "scatter_fp8", "restore_nvfp4", "restore_fp8",
         "int4_pack_key", "int4_pack_value", "int4_unpack_key", "int4_unpack_value",
         "int4_residual_key", "int4_residual_value", "int4_decode_copy_key", "int4_decode_copy_value",
         "int4_decode_inplace_key", "int4_decode_inplace_value",
         "nvfp4_pack", "nvfp4_unpack", "nvfp4_residual", "nvfp4_decode_copy", "nvfp4_decode_inplace",
         "fp8_pack", "fp8_unpack", "fp8_residual", "fp8_decode_copy", "fp8_decode_inplace",
         "nvfp4t_pack_key", "nvfp4t_pack_value", "nvfp4t_unpack_key", "nvfp4t_unpack_value")


def run_case(args):
    """One kernel's workload alone (for profiler captures): `args.warmup` untimed calls,
    then `args.steps` timed ones; prints one JSON line with the mean time per call.
    attention_*: the decode-attention pool of 32 x 8192 tokens, 8 KV / 32 query heads,
    D128; scatter_* / restore_*: K and V of the same 32 x 8192-token paged workload; the
    codec cases, <format>_<operation>[_<decode mode>][_<kind>]: a
    [131072, 8, 128] bf16 tensor (residual encode and decode: 25% of rows kept)."""
    import math

    import quantized_kv_cache_nvfp4_gb300 as kvq
    from quantized_kv_cache_nvfp4_gb300 import synth

    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    name = args.case
    if name.startswith(("scatter", "restore")):
        # the paged restore workload: 32 sequences x 8192 tokens, 8 KV heads, D128, a
        # shuffled table of 16,384 blocks; K and V
        S, T, H, D, bs = 32, 8192, 8, 128, BLOCK
        fmt = kvq.FMT_NVFP4 if name.endswith("nvfp4") else kvq.FMT_FP8
        nblocks = S * T // bs
        table = synth.block_permutation(nblocks, 3).to(device).view(S, T // bs).contiguous()
        t = torch.arange(T, device=device)
        slots = (table[:, t // bs].long() * bs + t % bs).reshape(-1)
        lens = torch.full((S,), T, dtype=torch.int32, device=device)
        pool = kvq.KvPool.empty(nblocks * bs, H, D, bs, device=device, fmt=fmt)
        k = synth.normal_bf16((S * T, H, D), 3, synth.STREAM_K, device=str(device))
        v = synth.normal_bf16((S * T, H, D), 3, synth.STREAM_V, device=str(device))
        kvq.kvq_quant_scatter(k, v, slots, pool)
        if name.startswith("scatter"):
            fn = lambda: kvq.kvq_quant_scatter(k, v, slots, pool)
        else:
            del k, v
            ko = torch.empty((S, T, H, D), dtype=torch.bfloat16, device=device)
            vo = torch.empty_like(ko)
            fn = lambda: kvq.kvq_restore(pool, table, lens, T, ko, vo)
    elif name.startswith("attention"):
        S, T, H, Hq, D, bs = 32, 8192, 8, 32, 128, BLOCK
        fk, fv = {"attention_nvfp4": (kvq.FMT_NVFP4, None), "attention_fp8": (kvq.FMT_FP8, None),
                  "attention_k8v4": (kvq.FMT_FP8, kvq.FMT_NVFP4)}[name]
        nblocks = S * T // bs
        perm = synth.block_permutation(nblocks, 3).to(device)
        table = perm.view(S, T // bs).contiguous()
        t = torch.arange(T, device=device)
        slots = (table[:, t // bs].long() * bs + t % bs).reshape(-1)
        lens = torch.full((S,), T, dtype=torch.int32, device=device)
        q = synth.normal_bf16((S, Hq, D), 3, 9, device=str(device))
        out = torch.empty_like(q)
        pool = kvq.KvPool.empty(nblocks * bs, H, D, bs, device=device, fmt=fk, v_fmt=fv)
        k = synth.normal_bf16((S * T, H, D), 3, synth.STREAM_K, device=str(device))
        v = synth.normal_bf16((S * T, H, D), 3, synth.STREAM_V, device=str(device))
        kvq.kvq_quant_scatter(k, v, slots, pool)
        del k, v
        ws = torch.empty(max(kvq.kvq_decode_attention_workspace(S, H, Hq, D, T), 16), dtype=torch.uint8,
                         device=device)
        fn = lambda: kvq.kvq_decode_attention(pool, table, lens, T, q, 1.0 / math.sqrt(D), out, workspace=ws)
    else:
        # <format>_<operation>[_<decode mode>][_<kind>] on a [131072, 8, 128] bf16 tensor
        T, H, D, G = 131072, 8, 128, 64
        cur, prev = synth.layer_kv(T, H, D, seed=4, device=str(device))
        parts = name.split("_")
        fmt = {"int4": kvq.FMT_INT4, "nvfp4": kvq.FMT_NVFP4, "fp8": kvq.FMT_FP8,
               "nvfp4t": kvq.FMT_NVFP4_TENSOR}[parts[0]]
        op = parts[1]
        kind = kvq.KIND_KEY if name.endswith("key") else kvq.KIND_VALUE
        if op in ("pack", "unpack"):
            pk = kvq.Packed.empty(fmt, kind, T, H, D, G, device=device)
            if op == "pack":
                fn = lambda: kvq.kvq_pack(cur, pk)
            else:
                kvq.kvq_pack(cur, pk)
                y = torch.empty_like(cur)
                fn = lambda: kvq.kvq_unpack(pk, y)
        else:  # residual encode, or decode into a separate output / in place; 25% of rows kept
            pos = synth.sorted_positions(T, T // 4, 4).to(device)
            pay = kvq.Packed.empty(fmt, kind, T // 4, H, D, G, device=device)
            if op == "residual":
                fn = lambda: kvq.kvq_encode_residual(cur, prev, pos, pay)
            else:
                kvq.kvq_encode_residual(cur, prev, pos, pay)
                if parts[2] == "copy":
                    out = torch.empty_like(prev)
                    fn = lambda: kvq.kvq_decode_residual(pay, pos, prev, out)
                else:
                    y = prev.clone()
                    fn = lambda: kvq.kvq_decode_residual(pay, pos, y, y)
    for _ in range(max(args.warmup, 1)):
        fn()
    torch.cuda.synchronize(device)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(max(args.steps, 1)):
        fn()
    b.record()
    torch.cuda.synchronize(device)
    print(json.dumps({"case": name, "steps": args.steps, "ms_per_call": round(a.elapsed_time(b) / max(args.steps, 1), 4)}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--e2e-chunks", type=int, default=16)
    ap.add_argument("--cpu-tokens", type=int, default=16384)
    ap.add_argument("--ref-seconds", type=float, default=150.0,
                    help="reference arm: CPU seconds the whole --steps/--warmup run may take")
    ap.add_argument("--tokens", type=int, default=T_TOKENS,
                    help="tokens of the workload (default: the 1,048,576-token case); smaller "
                         "values give the same kernels on a smaller case for profiling")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-other-rows", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--case", choices=CASES, default=None,
                    help="run one kernel's workload alone (for profiler captures) instead of the bench")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.case is not None:
        run_case(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
