#!/usr/bin/env python3
"""Benchmark of the GroupQueryAttention hot path over a shared KV buffer.

Headline: batched decode (16 sequences, 32 query / 8 KV heads, head size
128, bf16, buffer of 4096 slots, past lengths uniform in [1, 4095], one new
token each).  One step = one gqa_forward call: rotary embedding of the new
query/key rows, scatter-append of the new K/V rows, split-KV attention over
each sequence's true length, split combine.  The metric is algorithmic KV
bytes per second (visible K and V rows, plus query, output and the appended
rows) over the whole step.

The other workloads (long-context decode with and without a 4096 window,
the 2048-token prefill and the chunked prefill with bias) are timed after it
and reported under "also".

--impl reference times the CPU oracle (the plain reference implementation
of the same operator) on the host cores, on a bounded sample of the same
workload.

Multi-GPU (torchrun): every rank runs its own replica of the workload; there
is no data exchange between ranks (replicas only, weak scaling).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

HEADLINE = "decode_b16"
METRIC = "GQA decode KV GB/s"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-also", action="store_true", help="skip the other workloads")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU baseline")
    ap.add_argument("--workload", default=HEADLINE,
                    help="workload to time as the headline (default: the batched decode)")
    ap.add_argument("--quick", action="store_true",
                    help="headline workload only: no burn-in, one end-to-end step, no other workloads or CPU "
                         "baseline (for profiler runs)")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# distributed plumbing (replicas only)
# ---------------------------------------------------------------------------
def dist_init(backend):
    import torch.distributed as dist
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws > 1 and not dist.is_initialized():
        dist.init_process_group(backend)
    return int(os.environ.get("RANK", "0")), ws


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, ws, device=None):
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# clocks sampled while the GPU works
# ---------------------------------------------------------------------------
class ClockSampler:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.samples = []
        self.proc = None
        self.gpu_id = gpu_id

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", self.gpu_id], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        threading.Thread(target=self._read, daemon=True).start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        rows = [r for (t, r) in self.samples if t0 <= t <= t1 and len(r) >= 9]
        in_window = bool(rows)
        if not rows:
            rows = [r for (_, r) in self.samples if len(r) >= 9]
        if not rows:
            return {"error": "no nvidia-smi samples"}
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for n, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": num(rows[0][2]),
                "reasons": sorted(reasons), "samples": len(rows), "in_window": in_window,
                "power_w_max": max((num(r[3]) or 0.0) for r in rows)}


REJECTING_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown")


def clocks_rejected(c) -> bool:
    """True when a clock record voids the timing taken under it: a hardware or
    thermal slowdown was active, or the SM clock sat well below its maximum
    with no reason at all (a clock lock left on the GPU).  A power cap is
    kept (it is normal under a dense load)."""
    if not c or "error" in c:
        return False
    if any(r in REJECTING_REASONS for r in c.get("reasons", [])):
        return True
    sm, mx = c.get("sm_mhz"), c.get("sm_max_mhz")
    return bool(sm and mx and not c.get("reasons") and sm < 0.85 * mx)


def gpu_selector(torch, dev):
    try:
        return "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        return str(dev)


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained"), "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
class Problem:
    """Device-resident inputs of one workload, with `sets` copies of the
    buffers that consecutive steps rotate through (so a step never finds the
    previous step's KV rows in L2 when one set is smaller than L2)."""

    def __init__(self, name, device, sets=1):
        import torch
        import shared_kv_cache_gb300 as gqa
        from shared_kv_cache_gb300 import workloads as W
        self.w = W.CONFIGS[name]
        inp = W.make_inputs(self.w, device=device, sentinel=False)
        self.inp = inp
        self.past = inp["seqlens_k"].cpu()
        w = self.w
        self.dims = gqa.make_dims(w.batch, w.seq_len, w.num_heads, w.kv_num_heads, w.head_size, w.max_seq_len,
                                  w.dtype, 0, inp["cos"].shape[0] if inp["cos"] is not None else 0,
                                  *(inp["attention_bias"].shape[:2] if inp["attention_bias"] is not None else (1, 1)),
                                  kv_eviction=1 if w.kv_eviction else 0)
        # packed QKV: one query tensor with each token's query, key and value heads
        self.qkv = None
        if w.packed:
            B, S, D = w.batch, w.seq_len, w.head_size
            self.qkv = torch.cat([inp["query"].view(B, S, w.num_heads, D), inp["key"].view(B, S, w.kv_num_heads, D),
                                  inp["value"].view(B, S, w.kv_num_heads, D)], dim=2).reshape(B, S, -1).contiguous()
        self.total = inp["total_sequence_length"]
        self.ws_bytes = gqa.gqa_workspace_size(self.dims, self.total, w.local_window_size)
        self.ws = torch.empty(max(self.ws_bytes, 256), dtype=torch.uint8, device=device)
        self.kbufs = [inp["k_buf"]] + [inp["k_buf"].clone() for _ in range(sets - 1)]
        self.vbufs = [inp["v_buf"]] + [inp["v_buf"].clone() for _ in range(sets - 1)]
        self.out = torch.empty_like(inp["query"])
        self.decode = w.seq_len == 1
        self.bytes = W.decode_bytes(w, self.past)
        self.flops = W.prefill_flops(w, self.past) if not self.decode else 0
        self.gqa = gqa

    def step(self, i, stream):
        d = self.inp
        r = i % len(self.kbufs)
        q, k, v = (self.qkv, None, None) if self.qkv is not None else (d["query"], d["key"], d["value"])
        st = self.gqa.gqa_forward(self.dims, q, k, v, self.kbufs[r], self.vbufs[r],
                                  self.kbufs[r], self.vbufs[r], d["seqlens_k"], self.total, d["cos"], d["sin"],
                                  d["scale"], d["local_window_size"], d["attention_bias"], self.out, self.ws,
                                  self.ws.numel(), stream)
        if st != 0:
            raise RuntimeError(self.gqa.gqa_status_string(st))

    def launches_per_step(self):
        # decode: one kernel (append, split-KV attention and the split combine),
        # plus the eviction kernel on an evicting cache; prefill: the
        # rotary/append kernel plus the attention kernel
        if self.decode:
            return 2 if self.w.kv_eviction else 1
        return 2


def time_steps(prob, steps, warmup, stream, ws_count=1, device=None):
    import torch
    for i in range(warmup):
        prob.step(i, stream)
    torch.cuda.synchronize()
    barrier(ws_count)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    t0 = time.time()
    e0.record(stream)
    for i in range(steps):
        prob.step(i, stream)
    e1.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    barrier(ws_count)
    ms = e0.elapsed_time(e1) / steps
    return max_over_ranks(ms, ws_count, device), t0, t1


def e2e_decode(prob, steps, warmup, stream):
    """End to end through the host-buffer entry (forward_host, i.e.
    gqa_forward_host): every step takes its new query/key/value rows and
    seqlens_k from pinned host memory and returns its output to pinned host
    memory; the library's copy kernels move them over the host link, chained
    to the attention kernel by programmatic dependent launch.

    Returns (ms/step, h2d bytes, d2h bytes, copy-engine ms/step).  The last is
    the same step written with torch copies (copy engine) around forward() on
    one stream, for comparison."""
    import torch
    import shared_kv_cache_gb300 as gqa
    d = prob.inp
    # the step's host inputs (query, key, value rows and seqlens_k) packed in
    # one pinned buffer
    parts = [d[n] for n in ("query", "key", "value")] + [d["seqlens_k"]]
    nbytes = [t.numel() * t.element_size() for t in parts]
    offs = [0]
    for nb in nbytes:
        offs.append(offs[-1] + (nb + 255) // 256 * 256)
    host = torch.empty(offs[-1], dtype=torch.uint8).pin_memory()
    for t, o, nb in zip(parts, offs, nbytes):
        host[o:o + nb].copy_(t.contiguous().view(torch.uint8).reshape(-1).cpu())
    hviews = [host[o:o + nb].view(t.dtype).view(t.shape) for t, o, nb in zip(parts, offs, nbytes)]
    hout = torch.empty(prob.out.shape, dtype=prob.out.dtype).pin_memory()
    dev = torch.empty_like(host, device=prob.out.device)
    dviews = [dev[o:o + nb].view(t.dtype).view(t.shape) for t, o, nb in zip(parts, offs, nbytes)]
    wsp = gqa.Workspace()
    w = prob.w

    def host_step(i):
        hq, hk, hv, hs = hviews
        r = i % len(prob.kbufs)
        gqa.forward_host(hq, hk, hv, prob.kbufs[r], prob.vbufs[r], hs, prob.total, w.num_heads, w.kv_num_heads,
                         d["cos"], d["sin"], d["scale"], d["local_window_size"], d["attention_bias"],
                         output=hout, workspace=wsp, stream=stream, kv_eviction=int(w.kv_eviction))

    def copy_engine_step(i):
        dq, dk, dv, ds = dviews
        r = i % len(prob.kbufs)
        dev.copy_(host, non_blocking=True)
        out = gqa.forward(dq, dk, dv, prob.kbufs[r], prob.vbufs[r], ds, prob.total, w.num_heads, w.kv_num_heads,
                          d["cos"], d["sin"], d["scale"], d["local_window_size"], d["attention_bias"],
                          output=prob.out, workspace=wsp, stream=stream, kv_eviction=int(w.kv_eviction))
        hout.copy_(out, non_blocking=True)

    def timed(step_fn):
        with torch.cuda.stream(stream):
            for i in range(warmup):
                step_fn(i)
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for i in range(steps):
                step_fn(i)
            e1.record(stream)
            torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps

    ms = timed(host_step)
    ms_ce = timed(copy_engine_step)
    return ms, sum(nbytes), hout.numel() * hout.element_size(), ms_ce


_ORACLE_LOOP = """
import json, sys, time
sys.path.insert(0, {root!r})
import oracle
from shared_kv_cache_gb300 import workloads as W
w = W.CONFIGS[{name!r}]
inp = W.make_inputs(w, sentinel=False)
args = (W.bits(inp["query"]), W.bits(inp["key"]), W.bits(inp["value"]), W.bits(inp["k_buf"]), W.bits(inp["v_buf"]),
        inp["seqlens_k"].numpy(), inp["total_sequence_length"], W.bits(inp["cos"]), W.bits(inp["sin"]),
        w.num_heads, w.kv_num_heads, inp["scale"], inp["local_window_size"], None, w.dtype)
sel = {batches!r}
nbytes = W.decode_bytes(w.with_(batch=len(sel)), inp["seqlens_k"][sel])
print("ready", flush=True)
sys.stdin.readline()  # start together
n, t0 = 0, time.perf_counter()
while True:
    st = oracle.gqa_forward(*args, batches=sel)[0]
    assert st == 0
    n += 1
    if time.perf_counter() - t0 >= {min_seconds!r}:
        break
dt = time.perf_counter() - t0
print(json.dumps({{"value": nbytes * n / dt / 1e9, "calls": n, "seconds": dt, "sequences": len(sel)}}))
"""


def _oracle_rates(name, shares, min_seconds):
    """Runs the CPU oracle in one fresh interpreter per share of the batch's
    sequences (spawned: no CUDA state is inherited), each on one host thread,
    all timed over the same window.  Returns each process's result."""
    env = dict(os.environ)
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[v] = "1"
    env["CUDA_VISIBLE_DEVICES"] = ""
    procs = [subprocess.Popen([sys.executable, "-c", _ORACLE_LOOP.format(root=ROOT, name=name, batches=sel,
                                                                        min_seconds=min_seconds)],
                              stdin=subprocess.PIPE, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True,
                              env=env) for sel in shares]
    try:
        for p in procs:  # wait until every process has built its inputs
            if p.stdout.readline().strip() != "ready":
                raise RuntimeError(p.communicate(timeout=60)[1].strip().splitlines()[-1:])
        for p in procs:
            p.stdin.write("go\n")
            p.stdin.flush()
        out = []
        for p in procs:
            o, e = p.communicate(timeout=600)
            if p.returncode != 0:
                raise RuntimeError(e.strip().splitlines()[-1:] if e.strip() else "failed")
            out.append(json.loads(o.strip().splitlines()[-1]))
        return out
    finally:
        for p in procs:
            if p.poll() is None:
                p.kill()


def cpu_baseline(name, min_seconds=10.0):
    """The CPU oracle on the host cores: on one thread over the whole batch,
    and on every core (one single-threaded process per core, the batch's
    sequences dealt out round-robin, all timed together; their rates add)."""
    from shared_kv_cache_gb300 import workloads as W
    B = W.CONFIGS[name].batch
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    try:
        one = _oracle_rates(name, [list(range(B))], min_seconds)[0]
        n = min(cores, B)
        many = _oracle_rates(name, [list(range(i, B, n)) for i in range(n)], min_seconds)
    except (RuntimeError, subprocess.TimeoutExpired, ValueError) as e:
        return {"error": str(e)}
    calls = sum(r["calls"] for r in many)
    return {"value": sum(r["value"] for r in many), "unit": "GB/s", "cores": n, "kind": "oracle",
            "sample": f"all {B} sequences of the batch, one single-threaded process per core ({n}), "
                      f"{calls} oracle calls in {max(r['seconds'] for r in many):.1f} s (numpy float64)",
            "single_thread": {"value": one["value"], "unit": "GB/s", "cores": 1,
                              "sample": f"all {B} sequences per call, {one['calls']} calls in "
                                        f"{one['seconds']:.1f} s on one thread"}}


# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of the dominant
# kernel per launch, from the ncu captures summarised in profiles/; a kernel
# changed since its capture has no entry (reported as null).
TRAFFIC = {
    "decode_b16": 111568384 + 3243264,     # decode_dyn_kernel, profiles/decode_dyn_kernel_decode_b16.md
    "prefill_2k": 111838464 + 31110144,    # prefill_dual_kernel, profiles/prefill_dual_kernel_prefill_2k.md
    "chunked_prefill": 65992960 + 6409728,  # prefill_head_kernel, profiles/prefill_head_kernel_chunked_prefill.md
}
# the attention kernel of each prefill workload: two query heads per CTA
# where the group size is even and there is no bias or window
PREFILL_KERNEL = {"prefill_2k": "prefill_dual_kernel", "chunked_prefill": "prefill_head_kernel"}


def metric_of(prob):
    """(metric, unit, value per second scale) of a workload: decode steps are
    HBM-bound and counted in algorithmic KV bytes, prefill steps in attention
    FLOPs."""
    if prob.decode:
        return "GQA decode KV GB/s", "GB/s", prob.bytes / 1e9
    return "GQA prefill attention TFLOP/s", "TFLOP/s", prob.flops / 1e12


def run_ours(args):
    import torch
    rank, ws = dist_init("nccl")
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    device = f"cuda:{local}"
    import shared_kv_cache_gb300 as gqa
    from shared_kv_cache_gb300 import workloads as W
    gqa.load_library()
    pk = peaks()
    stream = torch.cuda.Stream(device)

    name = args.workload
    w = W.CONFIGS[name]
    kv_bytes = 2 * w.batch * w.kv_num_heads * w.max_seq_len * w.head_size * 2
    # rotate buffer sets so that consecutive steps do not find their KV rows in L2
    sets = 4 if kv_bytes < (1 << 30) else 1
    prob = Problem(name, device, sets=sets)
    metric, unit, work = metric_of(prob)
    sampler = ClockSampler(gpu_selector(torch, local))
    sampler.start()
    # keep the GPU busy for ~1 s before timing so that the clock record reflects load
    tb = time.time()
    i = 0
    while not args.quick and time.time() - tb < 1.0:
        prob.step(i, stream)
        i += 1
        if i % 200 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    ms, t0, t1 = time_steps(prob, args.steps, max(args.warmup, 3), stream, ws, device)
    clocks = sampler.summary(tb, t1)
    # a rejected clock record on any rank: every rank times the step once more
    if max_over_ranks(float(clocks_rejected(clocks)), ws, device) > 0:
        first = clocks
        ms, t0, t1 = time_steps(prob, args.steps, max(args.warmup, 3), stream, ws, device)
        clocks = sampler.summary(t0, t1)
        clocks["remeasured_after"] = first
    rate = work / (ms * 1e-3)
    value = rate * ws

    e2e_ms, h2d, d2h, ce_ms = e2e_decode(prob, args.steps if not args.quick else 1,
                                         1 if args.quick else max(args.warmup, 3), stream)
    e2e = {"value": work * ws / (e2e_ms * 1e-3), "unit": unit,
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
           "api": "forward_host (gqa_forward_host): pinned host inputs and output, copied by the library's kernels",
           "copy_engine": {"value": work * ws / (ce_ms * 1e-3), "ms_per_step": ce_ms,
                           "api": "torch copies on the copy engine around forward() on one stream"}}

    if prob.decode:
        roofline = {"kernel": "decode_dyn_kernel (one gqa_forward call)", "bound": "hbm",
                    "achieved": rate, "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": rate / pk["hbm_gbs"],
                    "peak_source": pk["source"], "frac_of_nominal_8tbs": rate / 8000.0,
                    "bytes_per_launch": prob.bytes, "traffic": TRAFFIC.get(name),
                    "traffic_kernel": "decode_dyn_kernel"}
    else:
        kern = PREFILL_KERNEL.get(name, "prefill_head_kernel")
        roofline = {"kernel": f"rope_append_kernel + {kern} (one gqa_forward call)", "bound": "tensor",
                    "achieved": rate, "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                    "frac": rate / pk["bf16_tflops"], "peak_source": pk["source"],
                    "flops_per_launch": prob.flops, "traffic": TRAFFIC.get(name),
                    "traffic_kernel": kern}

    also = []
    if not args.no_also and not args.quick:
        for other in ("decode_b16", "long_decode", "long_decode_w4096", "prefill_2k", "chunked_prefill",
                      "decode_b16_packed", "swa_decode_b16"):
            if other == name:
                continue
            wo = W.CONFIGS[other]
            kvo = 2 * wo.batch * wo.kv_num_heads * wo.max_seq_len * wo.head_size * 2
            p2 = Problem(other, device, sets=4 if kvo < (1 << 30) else 1)
            steps = 50
            # ~0.5 s of load first, so that the clock samples cover this workload
            tb2 = time.time()
            k = 0
            while time.time() - tb2 < 0.5:
                p2.step(k, stream)
                k += 1
                if k % 50 == 0:
                    torch.cuda.synchronize()
            torch.cuda.synchronize()
            m, _, t2 = time_steps(p2, steps, 3, stream, ws, device)
            mt, un, wk = metric_of(p2)
            v = wk / (m * 1e-3)
            peak = pk["hbm_gbs"] if p2.decode else pk["bf16_tflops"]
            entry = {"workload": other, "metric": mt, "value": v, "unit": un, "ms_per_step": m,
                     "frac": v / peak, "peak": peak, "clocks": sampler.summary(tb2, t2)}
            if not p2.decode:
                entry["kv_gbs"] = p2.bytes / (m * 1e-3) / 1e9
            also.append(entry)
            del p2
            torch.cuda.empty_cache()

    sampler.stop()
    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu and not args.quick and prob.decode:
        cpu = cpu_baseline(name)

    line = {
        "metric": metric, "value": value, "unit": unit, "n_gpus": ws, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic (seeded N(0,1) Q/K/V and cache)",
        "config": {"workload": name, "batch": w.batch, "num_heads": w.num_heads,
                   "kv_num_heads": w.kv_num_heads, "head_size": w.head_size, "max_seq_len": w.max_seq_len,
                   "new_tokens": w.seq_len, "past_lengths": f"uniform [{w.past_lo}, {w.past_hi}]",
                   "local_window_size": w.local_window_size, "rotary": True,
                   "bytes_per_step": prob.bytes, "flops_per_step": prob.flops,
                   "l2": (f"{sets} rotating KV buffer sets ({sets} x {kv_bytes >> 20} MiB)" if sets > 1 else
                          f"KV buffers of {kv_bytes >> 20} MiB") + " vs 129 MB L2",
                   "parallelism": f"replicas x{ws}"},
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": prob.launches_per_step() * args.steps,
        "clocks": clocks, "also": also,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ---------------------------------------------------------------------------
# reference arm: the CPU oracle
# ---------------------------------------------------------------------------
def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    # one host thread (set before numpy loads), so the core count is exact
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[v] = "1"
    import numpy as np  # noqa: F401
    import oracle
    from shared_kv_cache_gb300 import workloads as W
    w = W.CONFIGS[HEADLINE]
    inp = W.make_inputs(w, sentinel=False)
    sel = [0, 1]   # a bounded sample: two of the sixteen sequences per step
    a = (W.bits(inp["query"]), W.bits(inp["key"]), W.bits(inp["value"]), W.bits(inp["k_buf"]),
         W.bits(inp["v_buf"]), inp["seqlens_k"].numpy(), inp["total_sequence_length"], W.bits(inp["cos"]),
         W.bits(inp["sin"]), w.num_heads, w.kv_num_heads, inp["scale"], 0, None, w.dtype)
    nbytes = W.decode_bytes(w.with_(batch=len(sel)), inp["seqlens_k"][sel])
    for _ in range(max(args.warmup, 3)):
        oracle.gqa_forward(*a, batches=sel)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.gqa_forward(*a, batches=sel)
    dt = time.perf_counter() - t0
    ms = dt * 1e3 / args.steps
    value = nbytes / (ms * 1e-3) / 1e9
    cores = 1
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": 1,
        "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded N(0,1))",
        "config": {"workload": HEADLINE, "batch": w.batch, "num_heads": w.num_heads,
                   "kv_num_heads": w.kv_num_heads, "head_size": w.head_size, "max_seq_len": w.max_seq_len},
        "cpu_baseline": {"kind": "oracle", "cores": cores, "value": value, "unit": "GB/s",
                         "sample": f"sequences {sel} of the {w.batch}-sequence batch per step, one thread"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
