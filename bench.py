"""Benchmark of the paged-KV attention hot path on GB300.

One step = one batch of one layer through the whole path: save_kv_cache
(pkv_set_kv_buffer for the step's new tokens), the metadata build, and the
ForwardMode-dispatched forward (decode, extend or verify). Inputs are seeded
synthetic tensors shaped like the pages' serving cases (no dataset, no
weights); the KV pools are resident in HBM and larger than L2 for every
named workload, so timed iterations do not run from L2.

Default workload: Llama-3-8B-shaped paged decode (batch 64, 32/8 heads,
head_dim 128, contexts uniform in [1024, 8192], page_size 16). The metric is
KV GB/s of the step (algorithmic K+V bytes read / step time); extend workloads
report TFLOP/s.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference] [--spec-mode prefill|decode] [--batch N]

With --gpus N > 1 (launched by torch.distributed.run), every rank runs its own
replica of the workload on its own GPU ("replicas only": the path has no
exchange step); value = all ranks' work / max-over-ranks time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "paged decode KV GB/s (% HBM peak); extend TFLOP/s (% bf16 peak); µs/call"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0

# DRAM traffic per launch of the dominant kernel from one ncu capture of the
# workload (dram__bytes_read.sum + dram__bytes_write.sum), valid only while the
# kernel's source file is unchanged (src_sha: first 16 hex digits of its sha256).
NCU_TRAFFIC = {
    ("decode_splitkv", "llama3_8b_decode"): {"src_sha": "8e2560c6c19b5067", "bytes_per_launch": 1386290688},
    ("decode_splitkv", "long_fp8_decode"): {"src_sha": "8e2560c6c19b5067", "bytes_per_launch": 1471689728},
    ("extend_tc", "prefix_extend"): {"src_sha": "a645927089a35229", "bytes_per_launch": 271852032},
    ("extend_tc", "prefix_extend_fp8"): {"src_sha": "a645927089a35229", "bytes_per_launch": 193205760},
    ("extend_tc", "spec_verify/decode_path"): {"src_sha": "a645927089a35229", "bytes_per_launch": 599808000},
    ("extend_tc", "spec_verify/prefill_path"): {"src_sha": "a645927089a35229", "bytes_per_launch": 599735296},
}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", 0)), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


def src_sha(name):
    with open(os.path.join(ROOT, "paged_kv_cache_15_gb300", "csrc", name), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def work_of(W):
    """Algorithmic work of one forward over workload W.

    bytes: K and V of every visible key of every (request, KV head) once, plus
    Q in, O out, LSE out, page indices. flops: 2 * (D + Dv) per (query row,
    visible key) pair (QK^T over the K width and PV over the V width, as
    multiply-adds); D = Dv = head_dim unless K and V heads differ in width."""
    esz = 1 if W.is_fp8 else 2
    L = W.seq_lens.astype(np.int64)
    kv_bytes = int(L.sum()) * W.num_kv_heads * (W.head_dim + W.dv) * esz
    T = W.total_q
    io_bytes = T * W.num_q_heads * (W.head_dim + W.dv) * 2 + T * W.num_q_heads * 4
    idx_bytes = int(((L + W.page_size - 1) // W.page_size).sum()) * 4
    N = W.qo_lens.astype(np.int64)
    P = L - N
    pairs = int((N * P + N * (N + 1) // 2).sum())  # visible (row, key) pairs per q-head
    flops = 2 * (W.head_dim + W.dv) * W.num_q_heads * pairs
    return dict(kv_bytes=kv_bytes, bytes=kv_bytes + io_bytes + idx_bytes, flops=flops, pairs=pairs)


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.idx = device_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup(n_gpus):
    if n_gpus <= 1 and "RANK" not in os.environ:
        return 0, 1, 0
    import torch.distributed as dist
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    local = int(os.environ.get("LOCAL_RANK", 0))
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    backend = "nccl" if torch.cuda.is_available() else "gloo"
    if torch.cuda.is_available():
        torch.cuda.set_device(local)
    dist.init_process_group(backend=backend, rank=rank, world_size=world)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world <= 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def metric_value(W, work, seconds):
    """(value, unit) of the workload's headline metric for one step taking `seconds`."""
    if W.mode == "extend":
        return work["flops"] / seconds / 1e12, "TFLOP/s"
    return work["kv_bytes"] / seconds / 1e9, "GB/s"


def oracle_sample(W, budget_s=15.0):
    """Time the fp64 oracle on a bounded sample of W: whole requests (every
    query head) for decode and verify, blocks of query tokens (every head) for
    extend, until about budget_s of wall time on all host cores."""
    sys.path.insert(0, ROOT)
    import oracle
    from tests._pipeline import oracle_pools
    from paged_kv_cache_15_gb300.workloads import bf16_bits
    kp, vp = oracle_pools(W)
    meta = oracle.build_metadata(W.seq_lens, W.page_table, W.page_size,
                                 qo_lens=None if W.mode == "decode" else W.qo_lens)
    qo_indptr = meta["qo_indptr"]
    qbits = bf16_bits(W.q)
    nthreads = os.cpu_count() or 1
    kv = oracle.KV_FP8_E4M3 if W.is_fp8 else oracle.KV_BF16
    esz = 1 if W.is_fp8 else 2
    block = 8 if W.mode == "extend" else 1 << 30  # tokens per oracle call
    done_kv = done_pairs = done_tok = 0
    reqs = set()
    t0 = time.perf_counter()
    for b in range(W.bs):
        q0, q1 = int(qo_indptr[b]), int(qo_indptr[b + 1])
        L, N = int(W.seq_lens[b]), int(W.qo_lens[b])
        for t_lo in range(q0, q1, min(block, max(q1 - q0, 1))):
            t_hi = min(q1, t_lo + block)
            rows = np.array([(t, h) for t in range(t_lo, t_hi) for h in range(W.num_q_heads)], dtype=np.int32)
            oracle.attention(qbits, kp, vp, meta, W.num_q_heads, W.num_kv_heads, W.page_size, W.sm_scale,
                             kv_dtype=kv, k_scale=W.k_scale, v_scale=W.v_scale, rows=rows, nthreads=nthreads)
            # token i of the request sees L - N + i + 1 keys
            done_pairs += sum(L - N + (t - q0) + 1 for t in range(t_lo, t_hi))
            done_tok += t_hi - t_lo
            reqs.add(b)
            if t_hi == q1:
                done_kv += L * W.num_kv_heads * (W.head_dim + W.dv) * esz
            if time.perf_counter() - t0 > budget_s:
                break
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    if W.mode == "extend":
        val, unit = 2 * (W.head_dim + W.dv) * W.num_q_heads * done_pairs / dt / 1e12, "TFLOP/s"
        what = f"{done_tok} of {W.total_q} query tokens in {len(reqs)} of {W.bs} requests"
    else:
        val, unit = done_kv / dt / 1e9, "GB/s"
        what = f"{len(reqs)} of {W.bs} requests"
    return {"value": val, "unit": unit, "cores": nthreads, "kind": "oracle",
            "sample": f"{what} (all query heads), {dt:.1f} s, fp64 C oracle"}, dt


def config_of(W, spec_mode, world):
    """The workload as the JSON line names it (both arms print the same keys)."""
    return {"workload": W.name, "batch": W.bs, "num_q_heads": W.num_q_heads, "num_kv_heads": W.num_kv_heads,
            "head_dim": W.head_dim, "head_dim_v": W.dv, "page_size": W.page_size, "kv_dtype": W.kv_dtype, "mode": W.mode,
            "spec_mode": spec_mode, "total_kv_tokens": int(W.seq_lens.sum()), "total_q_rows": W.total_q,
            "l2": "inputs larger than L2 (K+V pools "
                  f"{2 * W.k_pool.numel() * W.k_pool.element_size() / 1e9:.2f} GB)",
            "parallelism": f"replicas x{world}"}


def run_reference(args, W, rank, world):
    if rank != 0:
        return
    per_step = []
    cpu = None
    for i in range(args.warmup + args.steps):
        cpu, dt = oracle_sample(W, budget_s=args.ref_budget)
        if i >= args.warmup:
            per_step.append((cpu["value"], dt))
    value = statistics.median(v for v, _ in per_step)
    ms = statistics.median(dt for _, dt in per_step) * 1e3
    cpu["value"] = value
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": cpu["unit"], "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(W, args.spec_mode, world),
            "cpu_baseline": cpu,
            "e2e": {"value": value, "unit": cpu["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def graph_step_us(d, step, steps, stream):
    """Per-step time of the same step captured once in a CUDA graph and replayed
    (serving replays decode graphs); None if capture is unavailable."""
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        step()
    stream.wait_stream(side)
    with torch.cuda.graph(g):
        step()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    g0 = torch.cuda.Event(enable_timing=True)
    g1 = torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    for _ in range(steps):
        g.replay()
    g1.record(stream)
    torch.cuda.synchronize()
    del g
    return g0.elapsed_time(g1) / steps * 1e3


def roofline_of(W, work, fwd_s, spec, B):
    hbm_peak, tf_peak, _, peak_kind = peaks()
    on_extend = W.mode == "extend" or (W.mode == "verify" and spec == B.PKV_SPEC_PREFILL)
    if W.mode == "extend":
        achieved = work["flops"] / fwd_s / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": tf_peak, "unit": "TFLOP/s",
                "frac": achieved / tf_peak, "peak_kind": f"{peak_kind} bf16 dense (burst)"}
    else:
        achieved = work["bytes"] / fwd_s / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                "frac": achieved / hbm_peak, "peak_kind": f"{peak_kind} HBM copy"}
    # the verify shapes run on the tcgen05 tile kernel on both paths (over the
    # decode plan on the decode path)
    on_tc = on_extend or W.mode == "verify"
    key = "extend_tc" if on_tc else "decode_splitkv"
    name = W.name if W.mode != "verify" else f"{W.name}/{'prefill' if on_extend else 'decode'}_path"
    tr = NCU_TRAFFIC.get((key, name))
    roof["traffic"] = None
    if tr and tr["src_sha"] == src_sha("extend.cu" if on_tc else "decode.cu"):
        roof["traffic"] = tr["bytes_per_launch"]
    roof["kernel"] = key
    roof["timed"] = ("forward call (attention kernel plus the split merge kernel), CUDA events on the "
                     "launching stream around each call, over a second pass of the K steps")
    return roof


def pack_pinned(d, names, fill=True):
    """Moves the named tensors of DeviceBatch d into one device buffer (each at
    a 256-byte aligned offset, the attribute replaced by a view of the same
    shape and type) with a pinned host twin of the same layout; with fill, the
    host twin holds the current values. Returns (host, device) uint8 buffers."""
    live = [(n, getattr(d, n)) for n in names if getattr(d, n) is not None]
    offs, total = [], 0
    for _, t in live:
        offs.append(total)
        total = (total + t.numel() * t.element_size() + 255) // 256 * 256
    dev = torch.empty(total, dtype=torch.uint8, device=live[0][1].device)
    host = torch.empty(total, dtype=torch.uint8).pin_memory()
    for (n, t), o in zip(live, offs):
        nb = t.numel() * t.element_size()
        view = dev[o:o + nb].view(t.dtype).view(t.shape)
        view.copy_(t)
        setattr(d, n, view)
        if fill:
            host[o:o + nb].copy_(t.contiguous().view(-1).view(torch.uint8).cpu())
    torch.cuda.synchronize()
    return host, dev


def timed_steps(d, spec, steps, world):
    """Whole-step time and forward-call time on the launching stream.

    The K steps that give the step time carry no events between their
    kernels: an event recorded between two launches ends the overlap of the
    next kernel's launch with the previous one. The forward call is then
    timed over a second pass of K steps with events around each call.
    """
    stream = torch.cuda.current_stream()
    barrier(world)
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(steps):
        d.set_kv_buffer()
        d.build_metadata()
        d.forward(spec)
    end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    step_s = max_over_ranks(start.elapsed_time(end) / steps / 1e3, world)

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    barrier(world)
    torch.cuda.synchronize()
    for i in range(steps):
        d.set_kv_buffer()
        d.build_metadata()
        ev[i][0].record(stream)
        d.forward(spec)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    fwd_s = max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in ev) / 1e3, world)
    return step_s, fwd_s


def secondary(name, spec_name, local, steps, world, cpu_budget, page_size=16, head_dims=None, bs=None):
    """Short measurement of another workload (no e2e), with the oracle timed
    beside it on a bounded sample (rank 0 of a single-GPU run only)."""
    from paged_kv_cache_15_gb300 import binding as B
    from paged_kv_cache_15_gb300.runner import DeviceBatch
    from paged_kv_cache_15_gb300.workloads import preset
    W = preset(name, bs=bs, page_size=page_size, head_dims=head_dims)
    spec = B.PKV_SPEC_DECODE if spec_name == "decode" else B.PKV_SPEC_PREFILL
    d = DeviceBatch(W, device=f"cuda:{local}")

    def step():
        d.set_kv_buffer()
        d.build_metadata()
        d.forward(spec)

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    if d.device_error():
        raise RuntimeError(f"device error on {name}")
    step_s, fwd_s = timed_steps(d, spec, steps, world)
    work = work_of(W)
    value, unit = metric_value(W, work, step_s)
    roof = roofline_of(W, work, fwd_s, spec, B)
    out = {"metric_value": value * world, "unit": unit, "us_per_call": fwd_s * 1e6, "step_us": step_s * 1e6,
           "graph_step_us": graph_step_us(d, step, steps, torch.cuda.current_stream()),
           "roofline_frac": roof["frac"], "achieved": roof["achieved"], "achieved_unit": roof["unit"],
           "kernel": roof["kernel"], "path": spec_name if W.mode == "verify" else
           ("decode" if W.mode == "decode" else "extend"),
           "steps": steps, "page_size": W.page_size, "head_dims": [W.head_dim, W.dv], "batch": W.bs,
           "cpu_baseline": None}
    del d
    torch.cuda.empty_cache()
    if world == 1 and cpu_budget > 0:
        out["cpu_baseline"], _ = oracle_sample(W, budget_s=cpu_budget)
    return out


def run_ours(args, W, rank, world, local):
    from paged_kv_cache_15_gb300 import binding as B
    from paged_kv_cache_15_gb300.runner import DeviceBatch

    spec = B.PKV_SPEC_DECODE if args.spec_mode == "decode" else B.PKV_SPEC_PREFILL
    d = DeviceBatch(W, device=f"cuda:{local}")
    work = work_of(W)
    stream = torch.cuda.current_stream()

    def step():
        d.set_kv_buffer()
        d.build_metadata()
        d.forward(spec)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    err = d.device_error()
    if err:
        raise RuntimeError(f"device error {err}")

    # --- device-resident timed region: K steps, events on the launching stream
    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    step_s, fwd_s = timed_steps(d, spec, args.steps, world)
    clocks = sampler.stop() if sampler else None
    launches = 4 * args.steps  # set_kv, metadata, attention, split merge (exits early when nothing was split)

    graph_us = None if args.no_graph else max_over_ranks(graph_step_us(d, step, args.steps, stream), world)

    # --- end to end through the C ABI with host buffers (pinned), inputs copied every step.
    # The step's inputs (q, new K/V, slots, lengths, page table) sit in one
    # pinned host buffer and one device buffer, and the outputs (out, LSE) in
    # another pair, so a step makes one host->device and one device->host copy.
    # Two such sets alternate, as in a serving loop: a side stream copies step
    # i+1's inputs in and step i-1's outputs out while step i's kernels run;
    # events order each set's copies and kernels. The timed region holds every
    # copy of every step.
    in_names = ["q", "k_new", "v_new", "loc", "seq_lens", "qo_lens", "page_table"]
    out_names = ["out", "lse"]
    sets = []
    for _ in range(2):
        h_in, d_in = pack_pinned(d, in_names)
        h_res, d_res = pack_pinned(d, out_names, fill=False)
        sets.append({"h_in": h_in, "d_in": d_in, "h_res": h_res, "d_res": d_res,
                     "views": {n: getattr(d, n) for n in in_names + out_names}})
    h2d = sets[0]["h_in"].numel()
    d2h = sets[0]["h_res"].numel()
    e2e_steps = max(1, min(args.steps, 50))
    side = torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    in_ready = [ev(), ev()]
    done = [ev(), ev()]
    out_read = [ev(), ev()]
    for k in range(2):  # nothing pending on either set yet
        done[k].record(stream)
        out_read[k].record(stream)

    def copy_in(i):  # step i's inputs into set i % 2, once step i-2 has read that set
        k = i % 2
        with torch.cuda.stream(side):
            side.wait_event(done[k])
            sets[k]["d_in"].copy_(sets[k]["h_in"], non_blocking=True)
            in_ready[k].record(side)

    def run(i, n):  # step i of n: its kernels, with step i+1's inputs moving meanwhile
        k = i % 2
        if i + 1 < n:
            copy_in(i + 1)
        stream.wait_event(in_ready[k])
        stream.wait_event(out_read[k])  # step i-2's outputs have left this set
        for name, t in sets[k]["views"].items():
            setattr(d, name, t)
        step()
        done[k].record(stream)
        with torch.cuda.stream(side):
            side.wait_event(done[k])
            sets[k]["h_res"].copy_(sets[k]["d_res"], non_blocking=True)
            out_read[k].record(side)

    def loop(n):
        copy_in(0)
        for i in range(n):
            run(i, n)
        stream.wait_event(out_read[(n - 1) % 2])
        if n > 1:
            stream.wait_event(out_read[n % 2])

    loop(4)  # warm both sets' paths
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    loop(e2e_steps)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(e0.elapsed_time(e1) / e2e_steps / 1e3, world)
    describe = B.pkv_describe(d.ctx)
    del d
    torch.cuda.empty_cache()

    # --- the other named workloads of the metric, short runs
    others = {}
    if not args.no_secondary:
        # (workload, speculative attention mode, page size, head widths, batch)
        for name, sp, ps, hd, nb in (("tiny_decode", "prefill", 16, None, None),
                                     ("prefix_extend", "prefill", 16, None, None),
                                     ("prefix_extend_fp8", "prefill", 16, None, None),
                                     ("spec_verify", "decode", 16, None, None),
                                     ("spec_verify", "prefill", 16, None, None),
                                     ("long_fp8_decode", "prefill", 16, None, None),
                                     ("long_fp8_decode", "prefill", 16, None, 1),
                                     ("llama3_8b_decode", "prefill", 128, None, None),
                                     ("llama3_8b_decode", "prefill", 16, (192, 128), None),
                                     ("prefix_extend", "prefill", 16, (192, 128), None)):
            if (name == W.name and sp == args.spec_mode and ps == W.page_size and hd is None and nb is None
                    and W.dv == W.head_dim and args.batch is None):
                continue
            key = name if name != "spec_verify" else f"spec_verify/{sp}_path"
            if ps != 16:
                key += f"/page_size_{ps}"
            if hd is not None:
                key += f"/head_dims_{hd[0]}_{hd[1]}"
            if nb is not None:
                key += f"/batch_{nb}"
            others[key] = secondary(name, sp, local, args.secondary_steps, world,
                                    0.0 if args.no_cpu_baseline else args.secondary_cpu_budget, page_size=ps,
                                    head_dims=hd, bs=nb)

    if rank != 0:
        return
    value, unit = metric_value(W, work, step_s)
    value *= world  # every rank ran one replica
    e2e_value = metric_value(W, work, e2e_s)[0] * world
    roof = roofline_of(W, work, fwd_s, spec, B)
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cpu, _ = oracle_sample(W, budget_s=args.ref_budget)
    line = {"metric": METRIC, "value": value, "unit": unit, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": step_s * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "fp8_e4m3 kv / bf16 q" if W.is_fp8 else "bf16",
            "data": "synthetic",
            "config": config_of(W, args.spec_mode, world),
            "us_per_call": fwd_s * 1e6,
            "step_us": step_s * 1e6,
            "graph_step_us": graph_us,
            "work": work,
            "roofline": roof,
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": unit, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "steps": e2e_steps, "api": "pkv_set_kv_buffer + pkv_build_metadata + pkv_forward",
                    "copies": "per step, one pinned H2D copy of the packed inputs (q, new K/V, slots, lengths, "
                              "page table) and one D2H copy of the packed out + LSE, on a side stream, double "
                              "buffered: step i+1's inputs and step i-1's outputs move while step i computes"},
            "gpu_launches": launches,
            "clocks": clocks,
            "workloads": others,
            "describe": describe}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="llama3_8b_decode")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--spec-mode", default="prefill", choices=["prefill", "decode"])
    ap.add_argument("--page-size", type=int, default=16, choices=[16, 128])
    ap.add_argument("--kv-dtype", default=None, choices=["bf16", "fp8_e4m3"],
                    help="pool element type (default: the workload's own)")
    ap.add_argument("--head-dims", type=int, nargs=2, default=None, metavar=("DK", "DV"),
                    help="widths of the Q/K and V heads (default: the workload's own)")
    ap.add_argument("--batch", type=int, default=None, help="requests in the batch (default: the workload's own)")
    ap.add_argument("--ref-budget", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--no-secondary", action="store_true", help="skip the short runs of the other workloads")
    ap.add_argument("--secondary-steps", type=int, default=30)
    ap.add_argument("--secondary-cpu-budget", type=float, default=6.0,
                    help="seconds of oracle time beside each of the other workloads")
    args = ap.parse_args()
    rank, world, local = dist_setup(args.gpus)
    from paged_kv_cache_15_gb300.workloads import preset
    W = preset(args.workload, bs=args.batch, page_size=args.page_size, kv_dtype=args.kv_dtype,
               head_dims=tuple(args.head_dims) if args.head_dims else None)
    if args.impl == "reference":
        run_reference(args, W, rank, world)
    else:
        if not torch.cuda.is_available():
            raise SystemExit("bench.py needs a CUDA device")
        from paged_kv_cache_15_gb300 import build
        build.build()
        run_ours(args, W, rank, world, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
