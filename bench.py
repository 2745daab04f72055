#!/usr/bin/env python
"""Benchmark of MLA paged-KV decode on GB300.

One step = one decode of one batch: one mla_decode_run through the C ABI (a
single kernel: TMA page staging, tcgen05 attention, in-kernel split-KV merge)
over a synthetic batch shaped like the DeepSeek-V2-Lite memory-bound workload
(batch 64, h_q 16, page 64, kv_len 4096; seeded gaussian bf16, random page
placement).  The plan is built once per batch composition, outside the
timed region, as a serving loop would reuse it across layers.

Prints ONE JSON line (rank 0).  Metric: KV GB/s (algorithmic bytes / time;
bytes = tokens x 1152 + q + out + lse + page indices).  A secondary object
reports TFLOPS on the DeepSeek-V3-shaped compute workload (batch 128,
h_q 128, kv 8192).  --impl reference times the fp64 CPU oracle instead.
Multi-GPU (torchrun): every rank decodes its own batch on its own GPU (the
path has no exchange step, so ranks are replicas); value = all ranks' bytes /
the slowest rank's time.
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

import torch  # noqa: E402

from workloads import WORKLOADS, algorithmic_bytes, algorithmic_flops, make_inputs  # noqa: E402

METRIC = "MLA decode: KV GB/s (h_q=16) & TFLOPS (h_q=128) vs GB300 roofline"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d.get("hbm_gbs", FALLBACK_HBM_GBS), d.get("bf16_tflops", FALLBACK_BF16_TFLOPS), \
            d.get("bf16_tflops_sustained"), "measured"
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, None, "fallback"


NOMINAL_HBM_GBS = 7900.0   # GB300 HBM3e, nominal


def strip_comments(src: str) -> str:
    """C/C++ source without its comments, trailing blanks and empty lines (the sources hold
    no comment marker inside a string literal)."""
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    lines = (re.sub(r"//.*", "", ln).rstrip() for ln in src.splitlines())
    return "\n".join(ln for ln in lines if ln)


def kernel_source_hash() -> str:
    """Hash of the code the attention kernels are built from, comments left out (the prologue
    kernel, a separate translation unit, is not one of them): a change of the compiled code
    changes it, an edit of a comment does not."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "mla_paged_kv_decode_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f == "prologue.cu":
            continue
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            h.update(f.encode() + strip_comments(fh.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """dram bytes per launch of the attention kernel from a committed ncu summary,
    only if it was taken on the current kernel sources."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(workload)
    if not e or e.get("kernel_sources") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 50 ms in a background process."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)

    def summary(self, t0, t1):
        rows = []
        for ts, line in self.samples:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            rows.append((ts, parts))
        inside = [r for r in rows if t0 <= r[0] <= t1]
        window = "timed region"
        if not inside and rows:  # region shorter than the sampling period: nearest samples
            inside = sorted(rows, key=lambda r: min(abs(r[0] - t0), abs(r[0] - t1)))[:2]
            window = "nearest to the timed region"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(p[1]) for _, p in inside if p[1].replace(".", "").isdigit()]
        smax = [float(p[2]) for _, p in inside if p[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for _, p in inside for n, v in zip(names, p[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(inside), "window": window}


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def max_over_ranks(x: float, world: int, device) -> float:
    """The largest of the ranks' values (the slowest rank's time); x itself on one rank."""
    if world <= 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t)


def aggregate(per_rank_seconds, per_rank_units, world):
    """Whole-job throughput: units of every rank / the slowest rank's time."""
    t = max(per_rank_seconds)
    return sum(per_rank_units) / t, t


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def time_oracle(inp, requests, threads):
    import oracle
    t0 = time.perf_counter()
    oracle.decode_subset(inp, requests, threads=threads)
    return time.perf_counter() - t0


def subset_bytes(inp, requests):
    H = inp.h_q
    per_tok = 644 if inp.ckv_scale is not None else 1152
    L = int(inp.kv_lens[requests].sum())
    n = sum(int(inp.kv_indptr[b + 1] - inp.kv_indptr[b]) for b in requests)
    return L * per_tok + len(requests) * (H * 576 * 2 + H * 512 * 4 + H * 4 + 8) + 4 * n


def cpu_baseline(inp, workload: str, sample_requests: int) -> dict:
    """The oracle on a bounded sample of the workload: on every host core, and on one core for
    an eighth of the sample."""
    cores = cpu_cores()
    sample = list(range(min(sample_requests, inp.batch)))
    time_oracle(inp, sample[:1], cores)
    sec = time_oracle(inp, sample, cores)
    one = sample[: max(1, len(sample) // 8)]
    sec1 = time_oracle(inp, one, 1)
    return {"value": subset_bytes(inp, sample) / sec / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{len(sample)} of {inp.batch} requests of {workload}, one pass, fp64",
            "single_thread": {"value": subset_bytes(inp, one) / sec1 / 1e9, "unit": "GB/s", "cores": 1,
                              "sample": f"{len(one)} of {inp.batch} requests of {workload}, one pass, fp64"}}


def run_reference(args):
    """The oracle, as it stands, on the host cores: a bounded sample of the workload per step."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    inp = make_inputs(WORKLOADS[args.workload])
    cores = cpu_cores()
    sample = list(range(min(args.sample_requests, inp.batch)))
    # the whole --steps/--warmup run stays within about two minutes: halve the sample while a
    # step would take longer than its share
    share = 120.0 / max(1, args.steps + args.warmup)
    while len(sample) > 1 and time_oracle(inp, sample, cores) > share:
        sample = sample[: len(sample) // 2]
    for _ in range(args.warmup):
        time_oracle(inp, sample, cores)
    ts = [time_oracle(inp, sample, cores) for _ in range(args.steps)]
    sec = sum(ts) / len(ts)
    gbs = subset_bytes(inp, sample) / sec / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload, "desc": WORKLOADS[args.workload].description,
                       "sample_requests": len(sample)},
            "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": f"{len(sample)} of {inp.batch} requests of {args.workload} per step"},
            "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def kv_dtype_of(inp):
    """The cache type of a workloads.Inputs: bf16, e4m3 codes (uint8) or INT8 codes (int8)."""
    import mla_paged_kv_decode_gb300 as mla
    if inp.ckv_scale is None:
        return mla.MLA_KV_F16 if inp.ckv.dtype == torch.float16 else mla.MLA_KV_BF16
    return mla.MLA_KV_INT8 if inp.ckv.dtype == torch.int8 else mla.MLA_KV_FP8_E4M3


def time_workload(inp, n, stream):
    """Seconds per decode step (one event pair around n steps after 5 warm-up steps)."""
    dec, step, keep = bench_device(inp, 0, 5, stream)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(n):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    del keep, dec
    return e0.elapsed_time(e1) / n / 1e3


def plan_balance(plan, h_q: int, kv_dtype: int) -> dict:
    """Max / mean unit cost of a plan: a unit's cost is its tiles plus the plan's segment cost per
    segment after its first (the measure whose maximum the planner minimises)."""
    import mla_paged_kv_decode_gb300 as mla
    tile = 128 if (h_q >= 64 and kv_dtype != mla.MLA_KV_INT8) else 32   # tcgen05 kernels: 128-token tiles
    segs, uptr = mla.mla_plan_get_segments(plan)
    c = mla.mla_plan_segment_cost_tiles(plan)
    cost, tiles = [], []
    for u in range(len(uptr) - 1):
        s = [x for x in segs[uptr[u]:uptr[u + 1]] if x[2] > x[1]]
        nt = sum((int(t1) - int(t0) + tile - 1) // tile for _, t0, t1, _ in s)
        tiles.append(nt)
        cost.append(nt + c * max(0, len(s) - 1))
    ratio = lambda v: (max(v) * len(v) / sum(v)) if sum(v) else None
    return {"units": len(cost), "tile": tile, "segment_cost_tiles": c, "cost_max_over_mean": ratio(cost),
            "tiles_max_over_mean": ratio(tiles), "segments": int(len(segs)),
            "partials": mla.mla_plan_num_partials(plan)}


def per_call_medians(name: str, stream, n: int = 100, **overrides) -> dict:
    """One workload: the median of n single decodes timed one by one (an event pair around each
    call on the launching stream), launched eagerly and as replays of a captured CUDA graph.
    ``overrides`` go to ``make_inputs`` (e.g. the INT8 cache for the 8-bit shape)."""
    import mla_paged_kv_decode_gb300 as mla
    inp = make_inputs(WORKLOADS[name], **overrides)
    b, f = algorithmic_bytes(inp), algorithmic_flops(inp)
    dec, step, keep = bench_device(inp, 0, 5, stream)
    out, lse, d = keep

    def timed(fn):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):   # replays go to the current stream
            for e0, e1 in evs:
                e0.record(stream)
                fn()
                e1.record(stream)
        torch.cuda.synchronize()
        return statistics.median(e0.elapsed_time(e1) for e0, e1 in evs) * 1e3

    eager = timed(step)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        step()
    with torch.cuda.stream(stream):
        for _ in range(3):
            g.replay()
    graph = timed(lambda: g.replay())
    st = dec.device_status(stream)
    kvd = kv_dtype_of(inp)
    desc = WORKLOADS[name].description
    if overrides.get("int8"):
        desc = desc.replace("e4m3 ckv", "INT8 ckv")
    res = {"desc": desc, "us_eager_median": eager, "us_graph_median": graph,
           "gbs": b / graph / 1e3, "tflops": f / graph / 1e6, "alg_bytes": b, "alg_flops": f,
           "tokens": int(inp.kv_lens.sum()), "calls": n, "status": st,
           "plan": plan_balance(dec.plan, inp.h_q, kvd)}
    del g, keep, dec, d, out, lse, inp
    torch.cuda.empty_cache()
    return res


def bench_device(inp, steps, warmup, stream):
    """Device-timed steps with resident inputs.  Returns per-step and per-kernel times (s)."""
    import mla_paged_kv_decode_gb300 as mla
    d = inp.to("cuda")
    kvd = kv_dtype_of(inp)
    dec = mla.Decoder(inp.kv_indptr, inp.kv_last_page_len, inp.h_q, inp.page_size, kv_dtype=kvd, stream=stream)
    out = torch.empty(inp.batch, inp.h_q, 512, dtype=torch.float32, device="cuda")
    lse = torch.empty(inp.batch, inp.h_q, dtype=torch.float32, device="cuda")
    args = (d.q_nope, d.q_pe, d.ckv, d.ckv_scale, d.kpe, d.kv_indices, d.kv_indptr, d.kv_last_page_len,
            inp.sm_scale, out, lse, dec.workspace)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        mla.mla_decode_run(dec.plan, *args, stream=stream)
        if ev is not None:
            ev[1].record(stream)

    with torch.cuda.stream(stream):
        for _ in range(warmup):
            step()
    torch.cuda.synchronize()
    return dec, step, (out, lse, d)


def packed_e2e(inp, d, dec, stream):
    """The end-to-end step: the inputs of one decode packed in one pinned host buffer (q_nope,
    q_pe, kv_indices, kv_indptr, kv_last_page_len, each at a 256-byte boundary) mirrored by one
    device buffer whose views the decode reads, and out + lse in one device buffer mirrored by one
    pinned host buffer.  Captured as a CUDA graph: H2D copy, mla_decode_run, D2H copy.  Returns the
    step, the bytes each way, and a check that the host copy of the result equals the device's."""
    import mla_paged_kv_decode_gb300 as mla
    align = lambda n: (n + 255) // 256 * 256
    srcs = [inp.q_nope, inp.q_pe, inp.kv_indices.to(torch.int32), inp.kv_indptr.to(torch.int32),
            inp.kv_last_page_len.to(torch.int32)]
    offs, total = [], 0
    for t in srcs:
        offs.append(total)
        total += align(t.numel() * t.element_size())
    host_in = torch.empty(total, dtype=torch.uint8).pin_memory()
    dev_in = torch.empty(total, dtype=torch.uint8, device="cuda")
    views = []
    for t, o in zip(srcs, offs):
        n = t.numel() * t.element_size()
        host_in[o:o + n].copy_(t.contiguous().view(-1).view(torch.uint8))
        views.append(dev_in[o:o + n].view(t.dtype).view(t.shape))
    q_nope, q_pe, kv_indices, kv_indptr, kv_last = views
    n_out = inp.batch * inp.h_q * 512 * 4
    n_lse = inp.batch * inp.h_q * 4
    dev_out = torch.empty(n_out + n_lse, dtype=torch.uint8, device="cuda")
    host_out = torch.empty(n_out + n_lse, dtype=torch.uint8).pin_memory()
    out = dev_out[:n_out].view(torch.float32).view(inp.batch, inp.h_q, 512)
    lse = dev_out[n_out:].view(torch.float32).view(inp.batch, inp.h_q)

    def body():
        dev_in.copy_(host_in, non_blocking=True)
        mla.mla_decode_run(dec.plan, q_nope, q_pe, d.ckv, d.ckv_scale, d.kpe, kv_indices, kv_indptr, kv_last,
                           inp.sm_scale, out, lse, dec.workspace, stream=stream)
        host_out.copy_(dev_out, non_blocking=True)

    with torch.cuda.stream(stream):   # warm-up outside the capture (tensor maps for these buffers)
        body()
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        body()

    def step():
        with torch.cuda.stream(stream):
            g.replay()
        stream.synchronize()

    def launch():
        """Replay without waiting; returns an event the host waits on for this step's result."""
        with torch.cuda.stream(stream):
            g.replay()
        ev = torch.cuda.Event()
        ev.record(stream)
        return ev

    def check():
        step()
        return bool(torch.equal(host_out[:n_out].view(torch.float32), out.cpu().view(-1).view(torch.float32)))

    return {"step": step, "launch": launch, "h2d": total, "d2h": n_out + n_lse, "check": check, "graph": g,
            "keep": (host_in, dev_in, dev_out, host_out)}


def bench_layer(batches=(1, 8, 32, 64), kv_len: int = 4096, reps: int = 30) -> dict:
    """Row f4: one MLA decode layer (DeepSeek-V2-Lite-shaped: 2048 wide, 16 heads; synthetic
    weights) as one CUDA graph -- q and kv projections (cuBLAS), the prologue (RoPE and the new
    token's cache write), the decode, the value and output projections -- at kv_len cached
    tokens per request (the new token the last), page 64, bf16 and e4m3 caches.  Each replay
    is timed by its own event pair after L2 is flushed (a 512 MB write), as a layer of a deep
    model finds its weights and cache cold; the median per batch size."""
    import mla_paged_kv_decode_gb300 as mla
    from mla_paged_kv_decode_gb300.layer import DecodeLayer, LayerWeights
    from workloads import layer_hidden, layer_weights, rope_table
    flush = torch.empty(512 * 2 ** 20, dtype=torch.uint8, device="cuda")
    w = LayerWeights(**vars(layer_weights(7))).to("cuda")
    rope = rope_table(kv_len + 1)
    res = {"shape": "hidden 2048, 16 heads, q_nope 128, q_pe 64, latent 512, v 128; page 64", "kv_len": kv_len,
           "timing": "CUDA graph replay, median of %d, L2 flushed before each" % reps, "us_per_layer": {}}
    for cache, fp8 in (("bf16", False), ("e4m3", True)):
        res["us_per_layer"][cache] = {}
        for b in batches:
            inp = make_inputs(WORKLOADS["membound"], kv_lens=[kv_len] * b, batch=b, fp8=fp8)
            d = inp.to("cuda")
            layer = DecodeLayer(w, inp.kv_indptr, inp.kv_last_page_len, inp.page_size, rope,
                                kv_dtype=mla.MLA_KV_FP8_E4M3 if fp8 else mla.MLA_KV_BF16)
            x = layer_hidden(b, 8).cuda()
            layer.capture(x, d.ckv, d.kpe, d.kv_indices, d.kv_indptr, d.kv_last_page_len, ckv_scale=d.ckv_scale)
            ts = []
            for i in range(reps + 3):
                flush.fill_(i & 0xFF)
                a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                layer.replay()
                e.record()
                torch.cuda.synchronize()
                if i >= 3:
                    ts.append(a.elapsed_time(e) * 1e3)
            assert mla.mla_decode_device_status(layer.plan, layer.workspace) == mla.MLA_OK
            res["us_per_layer"][cache][str(b)] = sorted(ts)[len(ts) // 2]
            del layer, d, inp
    return res


def profile_only(args):
    """warmup + steps decodes of one workload through the library, checked, for ncu captures."""
    import mla_paged_kv_decode_gb300 as mla
    torch.cuda.set_device(0)
    mla.load()
    w = WORKLOADS[args.workload]
    kw = {} if args.kv_len is None else {"kv_lens": [args.kv_len] * w.batch, "batch": w.batch}
    if args.cache == "int8":
        kw.update(fp8=False, int8=True)
    elif args.cache == "bf16":
        kw.update(fp8=False)
    inp = make_inputs(w, **kw)
    stream = torch.cuda.Stream()
    dec, step, keep = bench_device(inp, args.steps, args.warmup, stream)
    with torch.cuda.stream(stream):
        for _ in range(args.steps):
            step()
    torch.cuda.synchronize()
    st = mla.mla_decode_device_status(dec.plan, dec.workspace, stream)
    out = keep[0]
    assert st == 0 and bool(torch.isfinite(out).all()), f"status {st}"
    print(f"profile-only: {args.workload} ({args.cache} cache) batch {inp.batch} h_q {inp.h_q} "
          f"launches {args.warmup + args.steps} ok")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="membound", choices=sorted(WORKLOADS))
    ap.add_argument("--secondary", default="compute", help="second workload to report (TFLOPS), or 'none'")
    ap.add_argument("--sample-requests", type=int, default=16)
    ap.add_argument("--fp8", type=int, default=1, help="also time the 8-bit cache workload against bf16 (1/0)")
    ap.add_argument("--layer", type=int, default=1,
                    help="also time one decode layer as a CUDA graph at batch 1, 8, 32, 64 (1/0)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--configs", type=int, default=1,
                    help="also report every workload's per-call median, eager and CUDA-graph replay (1/0)")
    ap.add_argument("--profile-only", action="store_true",
                    help="run warmup + steps decodes of --workload on the device and exit, no timing or JSON "
                         "(the program the profiles' ncu commands capture)")
    ap.add_argument("--cache", default="workload", choices=["workload", "bf16", "int8"],
                    help="with --profile-only: the workload's own cache, or the same shape with a bf16 or INT8 cache")
    ap.add_argument("--kv-len", type=int, default=None,
                    help="with --profile-only: every request's kv_len (a smaller case of the workload)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    if args.profile_only:
        profile_only(args)
        return

    if args.impl == "reference":
        run_reference(args)
        return

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    import mla_paged_kv_decode_gb300 as mla
    mla.load()

    hbm_gbs, bf16_tf, bf16_tf_sus, peak_src = peaks()
    inp = make_inputs(WORKLOADS[args.workload])
    alg_bytes = algorithmic_bytes(inp)
    alg_flops = algorithmic_flops(inp)
    stream = torch.cuda.Stream()
    dec, step, keep = bench_device(inp, args.steps, args.warmup, stream)
    launches_per_step = mla.mla_plan_num_launches(dec.plan)

    # ---- device-timed region (inputs resident in HBM, 302 MB > 129 MB L2 per step: no flush).
    # One event pair brackets the K steps; a step is exactly one kernel launch, so the
    # kernel's average duration is the step time (per-step events would add their own gaps).
    assert launches_per_step == 1
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(args.steps):
        step()
    end.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    if world > 1:
        torch.distributed.barrier()
    sampler.stop()
    total_s = start.elapsed_time(end) / 1e3
    clocks = sampler.summary(t_wall0, t_wall1)

    total_max = max_over_ranks(total_s, world, "cuda")
    value, _ = aggregate([total_max], [alg_bytes * args.steps * world], world)
    value /= 1e9
    attn_avg = total_s / args.steps
    achieved = alg_bytes / attn_avg / 1e9

    # ---- end to end through the public API with host buffers.  The step's inputs (q_nope, q_pe
    # and the page table) live in one pinned host buffer laid out as one device buffer, and out +
    # lse in one device buffer laid out as one pinned host buffer, so a step is one H2D copy, the
    # decode and one D2H copy, all three captured in a CUDA graph (the decode call is graph-safe):
    # per step one graph launch and one host synchronisation.
    out, lse, d = keep
    e2e = packed_e2e(inp, d, dec, stream)
    e2e_steps = max(10, min(args.steps, 500))
    for _ in range(3):
        e2e["step"]()
    if world > 1:
        torch.distributed.barrier()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e["step"]()
    e2e_s = (time.perf_counter() - t0) / e2e_steps
    e2e_s = max_over_ranks(e2e_s, world, "cuda")
    e2e_seq_value = alg_bytes * world / e2e_s / 1e9
    h2d, d2h = e2e["h2d"], e2e["d2h"]
    e2e_ok = e2e["check"]()

    # Two independent batches of the workload (their own inputs and cache) alternate on two
    # streams, as a server interleaves batches: every step still copies its batch's inputs in
    # and its result out, and the host waits for a batch's previous result before launching its
    # next step; one batch's copies overlap the other's decode.
    inp_b = make_inputs(WORKLOADS[args.workload], seed=WORKLOADS[args.workload].seed + 100)
    d_b = inp_b.to("cuda")
    stream_b = torch.cuda.Stream()
    dec_b = mla.Decoder(inp_b.kv_indptr, inp_b.kv_last_page_len, inp_b.h_q, inp_b.page_size,
                        kv_dtype=kv_dtype_of(inp_b), stream=stream_b)
    e2e_b = packed_e2e(inp_b, d_b, dec_b, stream_b)
    pair, pend = (e2e, e2e_b), [None, None]

    def alternate(k):
        if pend[k % 2] is not None:
            pend[k % 2].synchronize()
        pend[k % 2] = pair[k % 2]["launch"]()

    for k in range(4):
        alternate(k)
    for ev in pend:
        ev.synchronize()
    pend = [None, None]
    if world > 1:
        torch.distributed.barrier()
    t0 = time.perf_counter()
    for k in range(e2e_steps):
        alternate(k)
    for ev in pend:
        if ev is not None:
            ev.synchronize()
    e2e_pipe_s = max_over_ranks((time.perf_counter() - t0) / e2e_steps, world, "cuda")
    e2e_value = alg_bytes * world / e2e_pipe_s / 1e9
    e2e_ok = e2e_ok and e2e_b["check"]()
    del e2e, e2e_b, dec_b, d_b, inp_b

    # ---- secondary: compute-shaped workload (TFLOPS), device-timed the same way
    secondary = None
    fp8 = None
    if (args.secondary != "none" or args.fp8) and rank == 0 and world == 1:
        del keep, dec
        torch.cuda.empty_cache()
    if args.secondary != "none" and rank == 0 and world == 1:
        inp2 = make_inputs(WORKLOADS[args.secondary])
        s2 = time_workload(inp2, max(20, min(args.steps // 10, 200)), stream)
        f2 = algorithmic_flops(inp2)
        b2 = algorithmic_bytes(inp2)
        secondary = {"workload": args.secondary, "desc": WORKLOADS[args.secondary].description,
                     "us_per_step": s2 * 1e6, "tflops": f2 / s2 / 1e12, "kv_gbs": b2 / s2 / 1e9,
                     "tensor_frac": f2 / s2 / 1e12 / bf16_tf, "hbm_frac": b2 / s2 / 1e9 / hbm_gbs,
                     "alg_flops": f2, "alg_bytes": b2, "traffic": recorded_traffic(args.secondary)}
        del inp2
        torch.cuda.empty_cache()

    # ---- 8-bit cache: e4m3 + per-token scale against the same shape with a bf16 cache
    if args.fp8 and rank == 0 and world == 1:
        n8 = max(20, min(args.steps // 20, 100))
        inp8 = make_inputs(WORKLOADS["fp8"])
        t8 = time_workload(inp8, n8, stream)
        b8 = algorithmic_bytes(inp8)
        tok = int(inp8.kv_lens.sum())
        del inp8
        torch.cuda.empty_cache()
        inp16 = make_inputs(WORKLOADS["fp8"], fp8=False)
        t16 = time_workload(inp16, n8, stream)
        b16 = algorithmic_bytes(inp16)
        del inp16
        torch.cuda.empty_cache()
        inpi = make_inputs(WORKLOADS["fp8"], fp8=False, int8=True)
        ti = time_workload(inpi, n8, stream)
        bi = algorithmic_bytes(inpi)
        del inpi
        torch.cuda.empty_cache()
        fp8 = {"workload": "fp8", "desc": WORKLOADS["fp8"].description, "us_per_step": t8 * 1e6,
               "gbs": b8 / t8 / 1e9, "hbm_frac": b8 / t8 / 1e9 / hbm_gbs, "tokens_per_s": tok / t8,
               "bf16_us_per_step": t16 * 1e6, "bf16_gbs": b16 / t16 / 1e9,
               "speedup_vs_bf16": t16 / t8, "bytes_per_token": {"fp8": 644, "int8": 644, "bf16": 1152},
               "traffic": recorded_traffic("fp8"),
               "int8": {"us_per_step": ti * 1e6, "gbs": bi / ti / 1e9, "hbm_frac": bi / ti / 1e9 / hbm_gbs,
                        "speedup_vs_bf16": t16 / ti, "traffic": recorded_traffic("int8")}}

    # ---- row f4: one decode layer as a CUDA graph
    layer = bench_layer() if (args.layer and rank == 0 and world == 1) else None

    # ---- every workload of the measurement table, one decode at a time: eager and graph replay
    configs = None
    if args.configs and rank == 0 and world == 1:
        configs = {}
        for key, name, kw in (("membound", "membound", {}), ("compute", "compute", {}),
                              ("b768_kv1024", "b768_kv1024", {}), ("b768_kv2048", "b768_kv2048", {}),
                              ("ragged", "ragged", {}), ("fp8", "fp8", {}),
                              ("int8", "fp8", {"fp8": False, "int8": True})):
            try:
                c = per_call_medians(name, stream, **kw)
                c["hbm_frac"] = c["gbs"] / hbm_gbs
                c["tensor_frac"] = c["tflops"] / bf16_tf
            except Exception as e:   # reported in the line; the step's own figures above stand
                c = {"error": f"{type(e).__name__}: {e}"[:300]}
                torch.cuda.empty_cache()
            configs[key] = c

    # ---- cpu baseline: the oracle on a bounded sample, host cores, rank 0 at N=1
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(inp, args.workload, args.sample_requests)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total_max / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": args.workload, "desc": WORKLOADS[args.workload].description,
                       "global_batch": inp.batch * world, "kv_len": int(inp.kv_lens[0]), "h_q": inp.h_q,
                       "page_size": inp.page_size, "parallelism": f"replicas x{world}",
                       "l2": "no flush: each step streams 302 MB of KV, > 129 MB L2",
                       "alg_bytes_per_step": alg_bytes, "alg_flops_per_step": alg_flops,
                       "tflops": alg_flops * args.steps * world / total_max / 1e12},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_gbs, "unit": "GB/s",
                         "frac": achieved / hbm_gbs, "traffic": recorded_traffic(args.workload),
                         "kernel": ("mla_decode_narrow_kernel" if inp.h_q <= 32 else "mla_decode_pair_kernel"),
                         "peak_source": peak_src,
                         "nominal_peak": NOMINAL_HBM_GBS, "frac_of_nominal": achieved / NOMINAL_HBM_GBS,
                         "kernel_us": attn_avg * 1e6},
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "steps": e2e_steps, "copies_checked": e2e_ok, "sequential_value": e2e_seq_value,
                    "note": "per step: one H2D copy of one batch's q + page table from pinned memory, its decode, "
                            "one D2H copy of its out + lse, as one CUDA graph replay; two independent batches of "
                            "the workload alternate on two streams and the host waits for a batch's previous "
                            "result before its next step (value); sequential_value: one batch, each step waited "
                            "for before the next; KV resident"},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clocks,
            "secondary": secondary,
            "fp8": fp8,
            "layer": layer,
            "configs": configs,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
