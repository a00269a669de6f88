#!/usr/bin/env python3
"""Benchmark of the MLA latent-KV decode hot path on GB300.

One step = mla_absorb_q -> mla_decode (+ split merge when split) -> mla_out_proj over one batch of
the DeepSeek-V3-shaped decode workload: B=64 requests, Sq=1, H=128 heads, ctx 4096 tokens each,
576-element bf16 rows in 64-token pages behind a random-permuted block table (302 MB of KV),
q / kv N(0,1), W_UK_T / W_UV N(0, 1/512), scale 1/sqrt(192). Synthetic, seeded inputs.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

N > 1 runs under torchrun, one process per GPU, each with its own replica of the workload (the
path has no exchange step: requests are independent), barrier + max-over-ranks timing. Rank 0
prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import mla_inputs as mi  # noqa: E402

METRIC = "MLA decode tokens/s & effective KV GB/s; % of min(HBM,TC) roofline, 1 GB300"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="dsv3", choices=sorted(mi.WORKLOADS))
    ap.add_argument("--component", default="step", choices=["step", "cache_write", "prefill"],
                    help="step: absorb -> decode -> out_proj (the hot path); cache_write: the KV cache "
                         "write that precedes it, measured alone (FP8 quantise for the fp8 workload); "
                         "prefill: the compute-friendly prefill route on a DeepSeek-V3-shaped batch")
    ap.add_argument("--num-splits", type=int, default=-1,
                    help="-1: GB300 planner, 0: the pages' Triton rule, >0 forced")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="oracle CPU-baseline sample budget")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--o-dtype", default="bf16", choices=["bf16", "fp32"],
                    help="dtype of o_latent and o: the model dtype (bf16) that the attention output is kept "
                         "in, or fp32; the LSE and split-KV partials are fp32 either way")
    ap.add_argument("--flush-mb", type=int, default=256, help="L2 flush buffer written between steps")
    return ap.parse_args()


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# what each decode kernel compiles from (bf16 cache, FP8 cache)
DECODE_SOURCES = {
    "decode_sm103.cu": ("decode_sm103.cu", "decode_common.cuh", "sm103_ptx.cuh", "internal.h"),
    "decode_fp8_sm103.cu": ("decode_fp8_sm103.cu", "decode_common.cuh", "sm103_ptx.cuh", "internal.h"),
}


def decode_kernel_sha256(kernel="decode_sm103.cu"):
    """sha256 over one decode kernel's source files, in DECODE_SOURCES order."""
    h = hashlib.sha256()
    for name in DECODE_SOURCES[kernel]:
        with open(os.path.join(ROOT, "mla_latent_kv_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def measured_traffic(workload, kernel="decode_sm103.cu"):
    """DRAM bytes per decode launch from the committed ncu capture (profiles/traffic.json), or
    None when that capture was of another workload (name and o_latent dtype, e.g. "dsv3/o_bf16")
    or of a different decode kernel source."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f)[kernel]
        h = decode_kernel_sha256(kernel)
    except (OSError, KeyError, ValueError):
        return None
    w = rec.get("workloads", {}).get(workload)
    if rec.get("sha256") != h or w is None:
        return None
    return int(w["dram_bytes_read"]) + int(w["dram_bytes_write"])


def workload_inputs(name, seed_offset=0):
    w = mi.WORKLOADS[name]
    c = mi.decode_case(w["B"], w["Sq"], w["H"], w["lens"], kv=w["kv"], seed=w["seed"] + seed_offset)
    rng = np.random.default_rng(w["seed"] + 1000 + seed_offset)
    B, Sq, H = c["B"], c["Sq"], c["H"]
    c["q_nope"] = mi.normal_bf16(rng, (B * Sq, H, mi.P))
    c["q_pe"] = mi.normal_bf16(rng, (B * Sq, H, mi.R))
    c["w_uk_t"] = mi.normal_bf16(rng, (H, mi.P, mi.L), std=1 / math.sqrt(512))
    c["w_uv"] = mi.normal_bf16(rng, (H, mi.L, mi.V), std=1 / math.sqrt(512))
    return c


def algorithmic(c, o_bytes=4):
    """Bytes and flops one decode launch must move / do (the absorbed algorithm, nothing else):
    KV rows of every visible token + q + o_latent (o_bytes per element) + lse + block-table entries
    + seq_lens; flops 2 * (576 + 512) per (query row, visible token, head)."""
    B, Sq, H = c["B"], c["Sq"], c["H"]
    rb = mi.ROW_BYTES[c["kv"]]
    lens = np.asarray(c["seq_lens"], np.int64)
    n_rows = np.array([[max(0, int(s) - (Sq - 1 - t)) for t in range(Sq)] for s in lens])
    kv_bytes = int(lens.sum()) * rb  # each request's rows are read once for all its query rows
    pages = int(((lens + 63) // 64).sum())
    byts = kv_bytes + B * Sq * H * (576 * 2 + 512 * o_bytes + 4) + pages * 4 + B * 4
    flops = int(n_rows.sum()) * H * 2 * (576 + 512)
    return byts, flops, kv_bytes


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_uuid=None):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"]
        if device_uuid:
            cmd += ["-i", device_uuid]
        try:
            self.p = subprocess.Popen(cmd, stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None

    def stop(self):
        if self.p is not None:
            self.p.terminate()
            try:
                self.p.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.p.kill()
        self.f.flush()
        self.f.seek(0)
        rows = [ln.strip().split(",") for ln in self.f.read().splitlines() if ln.strip()]
        os.unlink(self.f.name)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [x.strip() for x in r]
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except (ValueError, IndexError):
                continue
            for nm, v in zip(names, r[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- oracle leg
def oracle_sample_rate(c, budget_s, min_items=8):
    """Route-A oracle on a bounded sample of (request, query row, head) items; returns
    (tokens/s, items, seconds, threads)."""
    import oracle
    B, Sq, H = c["B"], c["Sq"], c["H"]
    all_items = np.array([(b, t, h) for b in range(B) for t in range(Sq) for h in range(H)], np.int32)
    rng = np.random.default_rng(123)
    order = rng.permutation(len(all_items))
    q64 = oracle.widen_bf16(c["q"])  # widened once, outside the timed calls

    def run(n):
        sel = all_items[order[:n]]
        t0 = time.perf_counter()
        oracle.decode_absorbed(q64, c["cache"], c["kv"], c["num_blocks"], c["block_table"], c["seq_lens"], B, Sq,
                               H, c["scale"], sel=sel)
        return time.perf_counter() - t0

    n = min_items
    dt = run(n)
    while dt < budget_s / 8 and n < len(all_items):
        n = min(len(all_items), n * 4)
        dt = run(n)
    if dt < budget_s / 2 and n < len(all_items):
        n = min(len(all_items), max(n, int(n * budget_s / max(dt, 1e-6) * 0.8)))
        dt = run(n)
    items_per_s = n / dt
    threads = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    return items_per_s / H, n, dt, threads


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    c = workload_inputs(args.workload)
    import oracle
    T, H = c["B"] * c["Sq"], c["H"]
    qa = oracle.absorb_q(c["q_nope"], c["q_pe"], c["w_uk_t"], T, H)
    # per step: a bounded sample, sized so that warmup + steps finish in about two minutes
    per_step_budget = max(0.02, 120.0 / max(1, args.steps + args.warmup))
    all_items = np.array([(b, t, h) for b in range(c["B"]) for t in range(c["Sq"]) for h in range(H)], np.int32)
    rng = np.random.default_rng(7)
    t0 = time.perf_counter()
    oracle.decode_absorbed(qa.reshape(c["B"], c["Sq"], H, mi.D), c["cache"], c["kv"], c["num_blocks"],
                           c["block_table"], c["seq_lens"], c["B"], c["Sq"], H, c["scale"], sel=all_items[:4])
    per_item = (time.perf_counter() - t0) / 4
    n_items = max(1, int(per_step_budget / max(per_item, 1e-9)))
    total_items, total_t = 0, 0.0
    for k in range(args.warmup + args.steps):
        sel = all_items[rng.integers(0, len(all_items), n_items)]
        t0 = time.perf_counter()
        oracle.decode_absorbed(qa.reshape(c["B"], c["Sq"], H, mi.D), c["cache"], c["kv"], c["num_blocks"],
                               c["block_table"], c["seq_lens"], c["B"], c["Sq"], H, c["scale"], sel=sel)
        dt = time.perf_counter() - t0
        if k >= args.warmup:
            total_items += n_items
            total_t += dt
    tok_s = total_items / H / total_t
    threads = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    line = {"impl": "reference", "metric": METRIC, "value": tok_s, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_t / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": workload_name(args.workload), "B": c["B"], "Sq": c["Sq"], "H": H},
            "cpu_baseline": {"value": tok_s, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                             "sample": f"{n_items} random (request, row, head) items per step, absorbed fp64 route"},
            "e2e": {"value": tok_s, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def workload_name(name):
    w = mi.WORKLOADS[name]
    kv = "fp8" if w["kv"] == mi.KV_FP8 else "bf16"
    lens = w["lens"] if isinstance(w["lens"], str) else w["lens"][0]
    return f"{name}: MLA decode B={w['B']} Sq={w['Sq']} H={w['H']} ctx={lens} page=64 {kv} cache"


# ----------------------------------------------------------------------------- our leg
def run_ours(args):
    import torch

    import mla_latent_kv_gb300 as mla

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    mla.lib()  # fail loudly if the native library is missing

    c = workload_inputs(args.workload, seed_offset=rank)
    B, Sq, H = c["B"], c["Sq"], c["H"]
    T = B * Sq

    def bf(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

    q_nope, q_pe = bf(c["q_nope"]), bf(c["q_pe"])
    w_uk_t, w_uv = bf(c["w_uk_t"]), bf(c["w_uv"])
    cache = torch.from_numpy(c["cache"]).to(dev)
    bt = torch.from_numpy(c["block_table"]).to(dev)
    sl = torch.from_numpy(np.asarray(c["seq_lens"], np.int32)).to(dev)
    max_len = int(np.max(c["seq_lens"]))
    S = mla.resolve_num_splits(args.num_splits, B, Sq, H, max_len)
    ws_n = mla.workspace_bytes(B, Sq, H, S, c["kv"], max_len)
    ws = torch.empty(max(ws_n, 256), dtype=torch.uint8, device=dev)
    q = torch.empty((T, H, mi.D), dtype=torch.bfloat16, device=dev)
    odt = torch.bfloat16 if args.o_dtype == "bf16" else torch.float32
    o_lat = torch.empty((B, Sq, H, mi.L), dtype=odt, device=dev)
    lse = torch.empty((B, Sq, H), dtype=torch.float32, device=dev)
    o = torch.empty((T, H, mi.V), dtype=odt, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.empty(args.flush_mb * (1 << 20), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def decode_call():
        mla.decode(q.view(B, Sq, H, mi.D), cache, bt, sl, max_len, c["scale"], kv_dtype=c["kv"], num_splits=S,
                   workspace=ws, o_latent=o_lat, lse=lse, dev_status=status, stream=stream,
                   num_blocks=c["num_blocks"])

    def step():
        mla.absorb_q(q_nope, q_pe, w_uk_t, out=q, stream=stream)
        decode_call()
        mla.out_proj(o_lat.view(T, H, mi.L), w_uv, out=o, stream=stream)

    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)

    K = args.steps
    starts, ends = [ev() for _ in range(K)], [ev() for _ in range(K)]
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    sampler = ClockSampler(uuid)
    time.sleep(0.3)
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    for k in range(K):
        flush.zero_()  # evict L2 between steps (outside the timed events)
        starts[k].record(stream)
        step()
        ends[k].record(stream)
    torch.cuda.synchronize(dev)
    # Decode alone, for the roofline: a loop of its own, whatever --steps is. Each launch follows
    # an L2 flush and is bracketed by events on the launching stream; the median is reported.
    n_dec = max(50, min(K, 200))
    dec0, dec1 = [ev() for _ in range(n_dec)], [ev() for _ in range(n_dec)]
    for k in range(n_dec):
        flush.zero_()
        dec0[k].record(stream)
        decode_call()
        dec1[k].record(stream)
    torch.cuda.synchronize(dev)
    if dist:
        dist.barrier()
    clocks = sampler.stop()
    step_ms = sum(s.elapsed_time(e) for s, e in zip(starts, ends)) / K
    dec_ms = statistics.median(a.elapsed_time(b) for a, b in zip(dec0, dec1))
    assert int(status.item()) == 0, f"device status {int(status.item())}"

    # ---------------- end to end through the public API with host buffers
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).pin_memory()  # noqa
    h_qn, h_qp = pin(c["q_nope"]), pin(c["q_pe"])
    h_bt = torch.from_numpy(c["block_table"]).pin_memory()
    h_sl = torch.from_numpy(np.asarray(c["seq_lens"], np.int32)).pin_memory()
    Ke = max(10, min(K, 200))
    # Two buffer sets, as a serving loop would run: step k copies its inputs into set k % 2 on
    # one copy stream, computes on the compute stream, and copies its result out on another, so
    # step k + 1's H2D and step k's D2H overlap step k + 1's compute. Every step still moves its
    # own inputs in and its own result out; the time is the whole run's over its step count.
    sets = [dict(qn=torch.empty_like(q_nope), qp=torch.empty_like(q_pe), bt=torch.empty_like(bt),
                 sl=torch.empty_like(sl), q=torch.empty_like(q), ol=torch.empty_like(o_lat), lse=torch.empty_like(lse),
                 o=torch.empty_like(o), ws=torch.empty_like(ws),
                 h_o=torch.empty((T, H, mi.V), dtype=odt).pin_memory()) for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    sync_ev = lambda: torch.cuda.Event()  # noqa: E731

    def e2e_run(n):
        comp_done, out_done = [None] * n, [None] * n
        e0, e1 = ev(), ev()
        e0.record(s_in)
        for k in range(n):
            b = sets[k % 2]
            if k >= 2:
                s_in.wait_event(comp_done[k - 2])  # step k - 2 has read this set's inputs
            with torch.cuda.stream(s_in):
                b["qn"].copy_(h_qn, non_blocking=True)
                b["qp"].copy_(h_qp, non_blocking=True)
                b["bt"].copy_(h_bt, non_blocking=True)
                b["sl"].copy_(h_sl, non_blocking=True)
            in_ready = sync_ev()
            in_ready.record(s_in)
            stream.wait_event(in_ready)
            if k >= 2:
                stream.wait_event(out_done[k - 2])  # step k - 2's result has left this set
            mla.absorb_q(b["qn"], b["qp"], w_uk_t, out=b["q"], stream=stream)
            mla.decode(b["q"].view(B, Sq, H, mi.D), cache, b["bt"], b["sl"], max_len, c["scale"], kv_dtype=c["kv"],
                       num_splits=S, workspace=b["ws"], o_latent=b["ol"], lse=b["lse"], dev_status=status,
                       stream=stream, num_blocks=c["num_blocks"])
            mla.out_proj(b["ol"].view(T, H, mi.L), w_uv, out=b["o"], stream=stream)
            comp_done[k] = sync_ev()
            comp_done[k].record(stream)
            s_out.wait_event(comp_done[k])
            with torch.cuda.stream(s_out):
                b["h_o"].copy_(b["o"], non_blocking=True)
            out_done[k] = sync_ev()
            out_done[k].record(s_out)
        s_out.wait_event(comp_done[n - 1])
        e1.record(s_out)
        return e0, e1

    e2e_run(4)
    torch.cuda.synchronize(dev)
    e_s, e_e = e2e_run(Ke)
    torch.cuda.synchronize(dev)
    e2e_ms = e_s.elapsed_time(e_e) / Ke
    h_o = sets[0]["h_o"]
    h2d = sum(t.numel() * t.element_size() for t in (h_qn, h_qp, h_bt, h_sl))
    d2h = h_o.numel() * h_o.element_size()

    # ---------------- max over ranks
    t = torch.tensor([step_ms, dec_ms, e2e_ms], dtype=torch.float64, device=dev)
    if dist:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    step_ms, dec_ms, e2e_ms = (float(x) for x in t.tolist())
    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return

    peaks, peak_src = load_peaks()
    byts, flops, kv_bytes = algorithmic(c, o_bytes=2 if args.o_dtype == "bf16" else 4)
    traffic_key = f"{args.workload}/o_{args.o_dtype}"
    traffic_kernel = "decode_fp8_sm103.cu" if c["kv"] == mi.KV_FP8 else "decode_sm103.cu"
    dec_s = dec_ms * 1e-3
    gbs = byts / dec_s / 1e9
    tflops = flops / dec_s / 1e12
    t_hbm = byts / (peaks["hbm_gbs"] * 1e9)
    t_tc = flops / (peaks["bf16_tflops_sustained"] * 1e12)
    bound = "hbm" if t_hbm >= t_tc else "tensor"
    if bound == "hbm":
        roof = {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": gbs / peaks["hbm_gbs"], "traffic": measured_traffic(traffic_key, traffic_kernel)}
    else:
        pk = peaks["bf16_tflops_sustained"]
        roof = {"bound": "tensor", "achieved": tflops, "peak": pk, "unit": "TFLOP/s", "frac": tflops / pk,
                "traffic": measured_traffic(traffic_key, traffic_kernel)}
    roof.update({"kernel": "mla_decode", "peak_source": f"{peak_src} (MEASURED_PEAKS.json)",
                 "bytes_per_launch": byts, "flops_per_launch": flops,
                 "min_roofline_frac": max(t_hbm, t_tc) / dec_s})

    cpu = None
    if not args.no_cpu_baseline:
        tok_s_cpu, n_items, dt, threads = oracle_sample_rate(c, args.cpu_seconds)
        n_all = B * Sq * H
        what = (f"the whole workload (all {n_all} (request, row, head) items)" if n_items >= n_all else
                f"{n_items} of its {n_all} (request, row, head) items, drawn at random")
        cpu = {"value": tok_s_cpu, "unit": "tokens/s", "cores": threads, "kind": "oracle",
               "sample": f"{what}, absorbed fp64 route (decode only), {dt:.1f} s, "
                         f"scaled by H={H} items per token"}
    tokens = T * world
    launches_per_step = 3 + (1 if (S > 1 or S == -2) else 0) + (1 if S == -2 else 0)  # + merge, + plan
    line = {"metric": METRIC, "value": tokens / (step_ms * 1e-3), "unit": "tokens/s", "n_gpus": world,
            "steps": K, "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": workload_name(args.workload), "B": B, "Sq": Sq, "H": H,
                       "kv_dtype": "fp8" if c["kv"] == mi.KV_FP8 else "bf16", "num_splits": S,
                       "o_dtype": args.o_dtype,
                       "l2": f"KV {kv_bytes / 1e6:.0f} MB > L2, plus a {args.flush_mb} MB L2 flush between steps",
                       "decode_timing": f"median of {n_dec} launches of mla_decode alone, each after an L2 flush and "
                                        "bracketed by CUDA events on its stream",
                       "e2e_timing": "pinned host inputs copied in and the result copied out every step, two "
                                     "buffer sets so that copies overlap the next step's compute; run time / steps, "
                                     "no flush (KV > L2)",
                       "parallelism": f"replicas x{world}"},
            "effective_kv_gbs": kv_bytes / dec_s / 1e9, "decode_tflops": tflops, "decode_us": dec_ms * 1e3,
            "roofline": roof, "cpu_baseline": cpu,
            "e2e": {"value": tokens / (e2e_ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
            "gpu_launches": launches_per_step * K + (launches_per_step - 2) * n_dec, "clocks": clocks}
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def run_cache_write(args):
    """mla_cache_write on one prefill-sized chunk of new tokens (65536 rows) of the workload's
    cache format; HBM-bound: 1152 bytes read and row_bytes written per token."""
    import torch
    import mla_latent_kv_gb300 as mla
    mla.lib()
    dev = torch.device("cuda", 0)
    kv = mi.WORKLOADS[args.workload]["kv"]
    T = 65536
    rng = np.random.default_rng(7)
    nb = T // 64 + 16
    kv_c = torch.randn(T, 512, device=dev).bfloat16()
    k_pe = torch.randn(T, 64, device=dev).bfloat16()
    slots = torch.from_numpy(rng.permutation(nb * 64)[:T].astype(np.int64)).to(dev)
    rb = mi.ROW_BYTES[kv]
    cache = torch.zeros(nb, 64 * rb, dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.empty(args.flush_mb * (1 << 20), dtype=torch.uint8, device=dev)
    for _ in range(max(3, args.warmup)):
        mla.cache_write(kv_c, k_pe, slots, cache, kv_dtype=kv, dev_status=status)
    torch.cuda.synchronize(dev)
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    sampler = ClockSampler(None)
    for a, b in ev:
        flush.zero_()
        a.record()
        mla.cache_write(kv_c, k_pe, slots, cache, kv_dtype=kv, dev_status=status)
        b.record()
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    assert int(status.item()) == 0
    ms = sum(a.elapsed_time(b) for a, b in ev) / K
    byts = T * (1152 + rb + 8)  # rows read, rows written, slot ids
    peaks, src = load_peaks()
    gbs = byts / (ms * 1e-3) / 1e9
    line = {"metric": "KV cache write tokens/s", "value": T / (ms * 1e-3), "unit": "tokens/s", "n_gpus": 1,
            "steps": K, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "fp8" if kv == mi.KV_FP8 else "bf16", "data": "synthetic",
            "config": {"workload": f"cache_write: {T} new tokens into a {'584' if kv else '1152'}-byte-row cache",
                       "l2": f"{args.flush_mb} MB L2 flush between launches"},
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / peaks["hbm_gbs"], "traffic": None, "kernel": "mla_cache_write",
                         "bytes_per_launch": byts, "peak_source": f"{src} (MEASURED_PEAKS.json)"},
            "gpu_launches": K, "clocks": clocks}
    print(json.dumps(line), flush=True)


PREFILL = dict(ctx=4096, q=1024, B=4, H=128, chunk_rows=65536)  # the page's 64k-row budget


def prefill_flops(ctx, ql, H):
    """Algorithmic flops of the prefill route: the up-projection of every gathered and new row
    (512 -> 128 + 128 per head) and the attention over each query's visible keys (192-dim q.k,
    128-dim p.v per head)."""
    ctx, ql = np.asarray(ctx, np.int64), np.asarray(ql, np.int64)
    rows = int(ctx.sum() + ql.sum())
    pairs = int((ql * ctx + ql * (ql + 1) // 2).sum())
    up = rows * H * 2 * 512 * 256
    attn = pairs * H * 2 * (192 + 128)
    return up + attn, up, attn


def run_prefill(args):
    """mla_prefill on a DeepSeek-V3-shaped chunked-prefill batch: B requests, each with `ctx`
    cached tokens and `q` new ones, H = 128, bf16 cache (FP8 for the fp8 workload). Tensor-bound:
    roofline against the dense bf16 peak, counting the route's algorithmic flops."""
    import torch
    import mla_latent_kv_gb300 as mla
    mla.lib()
    dev = torch.device("cuda", 0)
    kv = mi.WORKLOADS[args.workload]["kv"]
    w = PREFILL
    B, H = w["B"], w["H"]
    c = mi.prefill_case([w["ctx"]] * B, [w["q"]] * B, H, kv=kv, seed=31, poison=False)
    d16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)  # noqa
    q, kv_c, k_pe = d16(c["q"]), d16(c["kv_c_new"]), d16(c["k_pe_new"])
    wk, wv = d16(c["w_uk_t"]), d16(c["w_uv"])
    cache = torch.from_numpy(c["cache"]).to(dev)
    bt = torch.from_numpy(c["block_table"]).to(dev)
    ctx_d = torch.from_numpy(c["ctx_lens"]).to(dev)
    qsl_d = torch.from_numpy(c["query_start_loc"]).to(dev)
    ctx_h = torch.from_numpy(c["ctx_lens"].copy())
    qsl_h = torch.from_numpy(c["query_start_loc"].copy())
    T = int(c["query_start_loc"][-1])
    ws = torch.empty(mla.prefill_workspace_bytes(B, T, H, w["chunk_rows"]), dtype=torch.uint8, device=dev)
    o = torch.empty((T, H, 128), dtype=torch.float32, device=dev)
    lse = torch.empty((T, H), dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.empty(args.flush_mb * (1 << 20), dtype=torch.uint8, device=dev)

    def call():
        mla.prefill(q, kv_c, k_pe, cache, bt, ctx_d, qsl_d, wk, wv, c["scale"], kv_dtype=kv,
                    chunk_rows=w["chunk_rows"], workspace=ws, o=o, lse=lse, dev_status=status,
                    num_blocks=c["num_blocks"], ctx_lens_host=ctx_h, query_start_loc_host=qsl_h)
    for _ in range(max(3, args.warmup)):
        call()
    torch.cuda.synchronize(dev)
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    sampler = ClockSampler(None)
    for a, b in ev:
        flush.zero_()
        a.record()
        call()
        b.record()
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    assert int(status.item()) == 0
    ms = sum(a.elapsed_time(b) for a, b in ev) / K
    flops, up, attn = prefill_flops(c["ctx_lens"], np.diff(c["query_start_loc"]), H)
    n_chunks = int(mla.prefill_chunk_plan(c["ctx_lens"], w["chunk_rows"])[:, 0].max()) + 1
    one_pass = int(np.sum(c["ctx_lens"])) <= w["chunk_rows"]
    # prefix sum, then per segment: gather, two up-projections, attention
    launches = 1 + 4 * (1 if one_pass else 1 + n_chunks)
    peaks, src = load_peaks()
    tf = flops / (ms * 1e-3) / 1e12
    line = {"metric": "MLA prefill new tokens/s (compute-friendly route)", "value": T / (ms * 1e-3),
            "unit": "tokens/s", "n_gpus": 1, "steps": K, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"prefill: B={B} requests x {w['q']} new tokens over {w['ctx']} cached tokens, "
                                   f"H={H}, {'FP8' if kv else 'bf16'} cache, chunk_rows={w['chunk_rows']}",
                       "l2": f"{args.flush_mb} MB L2 flush between calls", "chunks": n_chunks,
                       "passes": "one (context and new tokens together)" if one_pass else "new tokens + chunks"},
            "prefill_tflops": tf,
            "roofline": {"bound": "tensor", "achieved": tf, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": tf / peaks["bf16_tflops"], "traffic": None,
                         "kernel": "mla_prefill (gather, up-projection GEMMs, attention; whole call)",
                         "flops_per_launch": flops, "flops_up_projection": up, "flops_attention": attn,
                         "peak_source": f"{src} bf16 burst (MEASURED_PEAKS.json)"},
            "gpu_launches": launches * K, "clocks": clocks}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    elif args.component == "cache_write":
        run_cache_write(args)
    elif args.component == "prefill":
        run_prefill(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
