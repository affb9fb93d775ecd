"""Benchmark: one paged decode step (KV append + paged attention) per step.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload llama7b] [--impl native|reference]

A step is one pass of the hot path over one batch: the slot-mapped append of
every sequence's new token (copy-on-write copies first when there are any),
then paged decode attention over all context tokens (split-K partitions and
their merge when a context spans several partitions).  The step is repeated on
the same batch (each step rewrites the same slots), so every step does the
same work.  Inputs are synthetic N(0,1), resident in HBM when the timed region
starts, and larger than L2 (the K/V read per step is ~1.2 GB for llama7b).

Prints one JSON line.  `value` is algorithmic bytes per step (K/V read through
the tables, table entries, queries, outputs, the appended K/V) / device step
time, in GB/s; `seq_steps_per_s` = sequences x steps / time.
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
sys.path.insert(0, ROOT)

METRIC = "paged decode-attention achieved HBM GB/s (% of GB300 peak); seq-steps/sec"
FALLBACK_HBM_GBS = 6800.0


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


ELEM = {"f16": 2, "bf16": 2, "e4m3": 1}


def bits(t: torch.Tensor) -> np.ndarray:
    """Raw element bits of a tensor (uint16 or uint8 numpy array) for the oracle."""
    t = t.detach().contiguous().cpu()
    if t.dtype in (torch.uint8, torch.float8_e4m3fn):
        return t.view(torch.uint8).numpy()
    return t.view(torch.int16).numpy().view(np.uint16)


def algorithmic_bytes(wl, lens: np.ndarray):
    """Bytes the method must move for one step (decode part, append part)."""
    e = ELEM[wl.cache_dtype]
    ea = ELEM[wl.act_dtype]
    L = lens.astype(np.int64)
    B = len(L)
    kv = int(L.sum()) * 2 * wl.num_kv_heads * wl.head_dim * e
    tables = int(np.sum(-(-L // wl.block_size))) * 4 + B * 4
    qo = 2 * B * wl.num_q_heads * wl.head_dim * ea
    decode = kv + tables + qo
    append = B * wl.num_kv_heads * wl.head_dim * 2 * (ea + e) + B * 8
    return decode, append


class ClockSampler:
    """nvidia-smi SM clock / throttle-reason samples every 200 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.rows = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200",
                 "-i", str(gpu_index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                self.rows.append((time.time(), parts))

    def mark(self):
        return time.time()

    def stop(self, t0, t1):
        if not self.proc:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=2)
        except Exception:
            self.proc.kill()
        return self.summary(t0, t1)

    def summary(self, t0, t1):
        """Median SM clock, max clock and active throttle reasons of the samples in [t0, t1]."""
        if not self.proc:
            return None
        rows = [r for t, r in list(self.rows) if t0 - 0.25 <= t <= t1 + 0.25] or [r for _, r in list(self.rows)]
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
        return dist, dist.get_rank(), ws, int(os.environ.get("LOCAL_RANK", "0"))
    return None, 0, 1, 0


# every source the partition kernel (with its fused append) is compiled from
TRAFFIC_SOURCES = ("decode_bf16_bf16.cu", "decode_inst.cuh", "decode.cuh", "pkv_device.cuh", "kernels.h")


def traffic_sources_sha256() -> str:
    """sha256 over the partition kernel's sources, in TRAFFIC_SOURCES order."""
    import hashlib
    h = hashlib.sha256()
    for name in TRAFFIC_SOURCES:
        with open(os.path.join(ROOT, "paged_kv_cache_102_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def _traffic(workload: str):
    """dram bytes per decode launch from a committed ncu summary, if it still matches the kernel sources."""
    path = os.path.join(ROOT, "profiles", "decode_traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
        if t.get("sources_sha256") != traffic_sources_sha256() or t.get("workload") != workload:
            return None
        return float(t["dram_bytes_per_launch"])
    except Exception:
        return None


def reduce_over_ranks(dist, dev, seconds: float, work: dict):
    """Replicas share no data: the job's time is the slowest rank's and its
    work the sum of every rank's (ranks draw different batches).  Returns
    (max seconds, {key: summed work}); identity without a process group."""
    if dist is None:
        return seconds, {k: float(v) for k, v in work.items()}
    keys = sorted(work)
    t = torch.tensor([float(seconds)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    w = torch.tensor([float(work[k]) for k in keys], dtype=torch.float64, device=dev)
    dist.all_reduce(w, op=dist.ReduceOp.SUM)
    return float(t.item()), dict(zip(keys, w.tolist()))


def setup(pkv, W, workload: str, seed: int, dev, batch: int = 0):
    import dataclasses
    wl = W.WORKLOADS[workload]
    if batch:
        # a smaller batch of the same workload (profiling captures that must stay small)
        wl = dataclasses.replace(wl, batch=batch, name=f"{wl.name}[batch={batch}]")
    d = W.draw(wl, seed)
    wl = d.workload
    vals = W.make_values(d, device=dev)
    B = len(d.context_lens)
    ids = np.arange(B)
    bm = pkv.BlockManager(d.num_blocks, wl.block_size, free_list=d.free_list)
    cow_pairs = 0
    if wl.samples_per_prompt > 1:
        # parallel sampling: each prompt's blocks are shared by its samples (ref count n);
        # every sample then appends its divergent tokens one step at a time, which
        # copies the shared partial block on the first divergent write of all but the
        # last holder (untimed set-up; the timed step is the next token of every sample)
        n = wl.samples_per_prompt
        for pi, plen in enumerate(d.prompt_lens):
            bm.add_sequence(pi * n, int(plen))
            for j in range(1, n):
                bm.fork(pi * n, pi * n + j)
        g = torch.Generator(device=dev)
        g.manual_seed(seed + 1000)
        act = W.DTYPES[wl.act_dtype]
        for step in range(int(d.divergent.max())):
            active = np.nonzero(d.divergent > step)[0]
            slots, pairs = bm.append_slots(active)
            if len(pairs):
                cow_pairs += len(pairs)
                pkv.paged_block_copy(vals["k_cache"], vals["v_cache"], torch.from_numpy(pairs).to(dev))
            kn = torch.randn(len(active), wl.num_kv_heads, wl.head_dim, generator=g, device=dev).to(act)
            vn = torch.randn(len(active), wl.num_kv_heads, wl.head_dim, generator=g, device=dev).to(act)
            pkv.paged_kv_append(kn, vn, torch.from_numpy(slots).to(dev), vals["k_cache"], vals["v_cache"])
    else:
        for i, c in enumerate(d.context_lens):
            bm.add_sequence(i, int(c))
    slots, pairs = bm.append_slots(ids)
    cow_pairs += len(pairs)
    if len(pairs):
        # copies needed before this step's own append (run once; the timed step rewrites the same slots)
        pkv.paged_block_copy(vals["k_cache"], vals["v_cache"], torch.from_numpy(pairs).to(dev))
    tables, lens = bm.tables(ids)
    unique_blocks = len({int(b) for i in ids for b in tables[i, : -(-int(lens[i]) // wl.block_size)]})
    st = dict(d=d, wl=wl, vals=vals, bm=bm, ids=ids, slots_h=slots, tables_h=tables, lens_h=lens,
              slots=torch.from_numpy(slots).to(dev), pairs=torch.zeros((0, 2), dtype=torch.int32, device=dev),
              tables=torch.from_numpy(tables).to(dev), lens=torch.from_numpy(lens).to(dev),
              cow_pairs=cow_pairs, unique_blocks=unique_blocks)
    st["out"] = torch.empty_like(vals["q"])
    return st


def run_native(args):
    import paged_kv_cache_102_gb300 as pkv
    from paged_kv_cache_102_gb300 import workloads as W

    dist, rank, world, local = _dist()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pkv.load()
    pkv.set_kernel_path(args.kernel_path)
    st = setup(pkv, W, args.workload, args.seed + rank, dev, args.batch)
    wl, vals = st["wl"], st["vals"]
    B = len(st["ids"])
    ps = args.partition_size
    need = pkv.workspace_size(B, wl.num_q_heads, wl.num_kv_heads, wl.head_dim, st["tables_h"].shape[1],
                              wl.block_size, ps)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    max_parts = math.ceil(st["tables_h"].shape[1] * wl.block_size /
                          pkv.resolve_partition_size(B, wl.num_q_heads, wl.num_kv_heads, wl.head_dim,
                                                     st["tables_h"].shape[1], wl.block_size, ps))
    ks, vs = vals.get("k_scale"), vals.get("v_scale")
    stream = torch.cuda.current_stream(dev)
    npairs = st["pairs"].shape[0]
    # the fused step through the public plan API: validated and marshalled once
    # for the step's fixed buffers, one C call per step
    plan = pkv.DecodePlan(vals["q"], vals["k_cache"], vals["v_cache"], st["tables"], st["lens"], wl.scale,
                          out=st["out"], k_scale=ks, v_scale=vs, partition_size=ps, workspace=ws, stream=stream,
                          k_new=vals["k_new"], v_new=vals["v_new"], slot_mapping=st["slots"]) if args.fused else None

    def step(ev_mid=None):
        if npairs:
            pkv.paged_block_copy(vals["k_cache"], vals["v_cache"], st["pairs"])
        if args.fused:
            if ev_mid is not None:
                ev_mid.record(stream)
            plan.run()
            return
        pkv.paged_kv_append(vals["k_new"], vals["v_new"], st["slots"], vals["k_cache"], vals["v_cache"], ks, vs)
        if ev_mid is not None:
            ev_mid.record(stream)
        pkv.paged_attention_decode(vals["q"], vals["k_cache"], vals["v_cache"], st["tables"], st["lens"], wl.scale,
                                   out=st["out"], k_scale=ks, v_scale=vs, partition_size=ps, workspace=ws)

    launches_per_step = (1 if npairs else 0) + (0 if args.fused else 1) + 1 + (1 if max_parts > 1 else 0)
    dec_bytes, app_bytes = algorithmic_bytes(wl, st["lens_h"])
    step_bytes = dec_bytes + app_bytes

    sampler = None if args.ncu else ClockSampler(
        dev.index if not os.environ.get("CUDA_VISIBLE_DEVICES") else
        int(os.environ["CUDA_VISIBLE_DEVICES"].split(",")[local]))
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    # keep the GPU busy long enough for the clock sampler to see it under load
    t_soak = time.time()
    while sampler is not None and time.time() - t_soak < 0.6:
        for _ in range(20):
            step()
        torch.cuda.synchronize(dev)
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    t0 = time.time()
    ev_start = torch.cuda.Event(enable_timing=True)
    ev_end = torch.cuda.Event(enable_timing=True)
    mids = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ev_start.record(stream)
    for i in range(args.steps):
        step(mids[i])
        ends[i].record(stream)
    ev_end.record(stream)
    torch.cuda.synchronize(dev)
    if dist:
        dist.barrier()
    t1 = time.time()
    ms_total = ev_start.elapsed_time(ev_end)
    dec_ms = [mids[i].elapsed_time(ends[i]) for i in range(args.steps)]
    clocks = sampler.stop(t_soak, t1) if sampler else None
    ms_total, job = reduce_over_ranks(dist, dev, ms_total, {"bytes": step_bytes, "seqs": B})

    ms_step = ms_total / args.steps
    value = job["bytes"] / (ms_step * 1e-3) / 1e9
    peak, peak_src = _peaks()
    dec_avg_ms = statistics.mean(dec_ms)
    kernel_bytes = dec_bytes + (app_bytes if args.fused else 0)  # the fused launch also does the append
    achieved = kernel_bytes / (dec_avg_ms * 1e-3) / 1e9
    traffic = _traffic(args.workload)

    # end to end through the public API: pinned host inputs -> device, step, output -> host
    e2e = None
    if not (args.no_e2e or args.ncu):
        # Every step's inputs (q, new K/V, slots, block tables, lengths) travel in
        # one packed pinned buffer and one host->device copy; the output comes
        # back with one device->host copy.  The pinned inputs are double
        # buffered so the host block manager fills step n+1's tables while the
        # GPU runs step n (a serving loop's overlap); each step still copies its
        # own inputs in and its output out inside the timed region.
        parts = [("q", vals["q"]), ("k_new", vals["k_new"]), ("v_new", vals["v_new"]), ("slots", st["slots"]),
                 ("tables", st["tables"]), ("lens", st["lens"])]
        offs, off = {}, 0
        for name, t in parts:
            offs[name] = off
            off += (t.numel() * t.element_size() + 255) // 256 * 256
        h_in = [torch.empty(off, dtype=torch.uint8).pin_memory() for _ in range(2)]
        d_in = torch.empty(off, dtype=torch.uint8, device=dev)

        def view(buf, name):
            t = dict(parts)[name]
            nbytes = t.numel() * t.element_size()
            return buf[offs[name]: offs[name] + nbytes].view(t.dtype).view(t.shape)

        for hb in h_in:
            for name in ("q", "k_new", "v_new", "slots"):
                view(hb, name).copy_(dict(parts)[name].cpu())
        dv_ = {name: view(d_in, name) for name, _ in parts}
        out_h = torch.empty(st["out"].shape, dtype=st["out"].dtype).pin_memory()
        h2d = off
        d2h = out_h.numel() * out_h.element_size()
        stream_e2e = torch.cuda.current_stream(dev)
        state = {"n": 0}

        def prep(hb):
            tab, lens = st["bm"].tables(st["ids"], st["tables_h"].shape[1])  # host block manager (C++)
            view(hb, "tables").numpy()[...] = tab
            view(hb, "lens").numpy()[...] = lens

        prep(h_in[0])

        # the fused step as a serving loop issues it: validated and marshalled
        # once for its fixed buffers, then one C call per step
        plan = pkv.DecodePlan(dv_["q"], vals["k_cache"], vals["v_cache"], dv_["tables"], dv_["lens"], wl.scale,
                              out=st["out"], k_scale=ks, v_scale=vs, partition_size=ps, workspace=ws,
                              stream=stream_e2e, k_new=dv_["k_new"], v_new=dv_["v_new"], slot_mapping=dv_["slots"])

        def e2e_step():
            hb = h_in[state["n"] % 2]
            state["n"] += 1
            d_in.copy_(hb, non_blocking=True)
            if args.fused:
                plan.run()
            else:
                pkv.paged_kv_append(dv_["k_new"], dv_["v_new"], dv_["slots"], vals["k_cache"], vals["v_cache"], ks,
                                    vs)
                pkv.paged_attention_decode(dv_["q"], vals["k_cache"], vals["v_cache"], dv_["tables"], dv_["lens"],
                                           wl.scale, out=st["out"], k_scale=ks, v_scale=vs, partition_size=ps,
                                           workspace=ws)
            out_h.copy_(st["out"], non_blocking=True)
            prep(h_in[state["n"] % 2])  # the next step's tables, while the GPU runs this one
            stream_e2e.synchronize()

        for _ in range(max(3, args.warmup)):
            e2e_step()
        if dist:
            dist.barrier()
        te0 = time.perf_counter()
        for _ in range(args.steps):
            e2e_step()
        te = (time.perf_counter() - te0) / args.steps
        te, _ = reduce_over_ranks(dist, dev, te, {})
        e2e = {"value": round(job["bytes"] / te / 1e9, 2), "unit": "GB/s",
               "ms_per_step": round(te * 1e3, 4), "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "seq_steps_per_s": round(job["seqs"] / te, 1),
               "call": "DecodePlan.run (fused append + decode)" if args.fused else
                       "paged_kv_append + paged_attention_decode"}
        if not torch.equal(out_h, st["out"].cpu()):
            raise RuntimeError("e2e output differs from the device-resident step")

    if pkv.device_error(reset=True, device=dev):
        raise RuntimeError("a kernel flagged a device-side error during the benchmark")

    cpu = None
    if rank == 0 and world == 1 and not (args.no_cpu_baseline or args.ncu):
        cpu = cpu_baseline(st, budget_s=args.cpu_budget)


    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": wl.cache_dtype, "data": "synthetic N(0,1), seeded",
        "config": {"workload": wl.name, "description": wl.description, "num_seqs": B,
                   "num_q_heads": wl.num_q_heads, "num_kv_heads": wl.num_kv_heads, "head_dim": wl.head_dim,
                   "block_size": wl.block_size, "act_dtype": wl.act_dtype, "cache_dtype": wl.cache_dtype,
                   "mean_context": float(st["lens_h"].mean()), "total_context_tokens": int(st["lens_h"].sum()),
                   "pool_blocks": st["d"].num_blocks,
                   "unique_kv_bytes_read": st["unique_blocks"] * wl.num_kv_heads * wl.block_size * wl.head_dim
                                           * 2 * ELEM[wl.cache_dtype],
                   "cow_block_copies_in_setup": st["cow_pairs"],
                   "partition_size": pkv.resolve_partition_size(B, wl.num_q_heads, wl.num_kv_heads, wl.head_dim,
                                                                st["tables_h"].shape[1], wl.block_size, ps),
                   "l2": "inputs larger than L2 (K/V read per step %.2f GB vs 129 MB L2)" % (dec_bytes / 1e9),
                   "parallelism": f"replicas x{world} (sequences sharded, no collective)",
                   "kernel_path": args.kernel_path, "fused_append": bool(args.fused)},
        "pct_of_peak": round(100 * value / (peak * world), 2),  # per GPU
        "seq_steps_per_s": round(job["seqs"] / (ms_step * 1e-3), 1),
        "bytes_per_step": {"decode": dec_bytes, "append": app_bytes},
        "roofline": {"bound": "hbm",
                     "kernel": ("paged_attention_decode_append" if args.fused else "paged_attention_decode")
                               + " (partition + merge kernels)",
                     "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)",
                     "traffic": traffic, "avg_launch_us": round(dec_avg_ms * 1e3, 3),
                     "algorithmic_bytes_per_launch": kernel_bytes},
        "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
        "cpu_baseline": cpu,
    }
    # the other target configurations, device-timed on the same box in the same run
    if world == 1 and not (args.ncu or args.no_workloads) and args.workload == "llama7b" and not args.batch:
        del plan
        st.clear()
        vals = None
        torch.cuda.empty_cache()
        line["workloads"] = {}
        for name in OTHER_WORKLOADS:
            line["workloads"][name] = time_workload(pkv, W, name, dev, args, peak)
            torch.cuda.empty_cache()
    print(json.dumps(line), flush=True)


# the grouped-query, E4M3 and long-context configurations reported beside the headline line
OTHER_WORKLOADS = ("gqa_bs16", "gqa_bs32", "long_gqa", "fp8_13b", "gqa_fp8", "gqa_g2", "gqa_d64")


def time_workload(pkv, W, name, dev, args, peak):
    """One workload's fused decode step (append + decode through DecodePlan,
    library-chosen kernel and partition size), warmed up, then `steps` steps
    each bracketed by CUDA events on the launching stream; the clock sampler
    runs over the soak and the timed region."""
    st = setup(pkv, W, name, args.seed, dev)
    wl, vals = st["wl"], st["vals"]
    B = len(st["ids"])
    need = pkv.workspace_size(B, wl.num_q_heads, wl.num_kv_heads, wl.head_dim, st["tables_h"].shape[1],
                              wl.block_size, -1)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    plan = pkv.DecodePlan(vals["q"], vals["k_cache"], vals["v_cache"], st["tables"], st["lens"], wl.scale,
                          out=st["out"], k_scale=vals.get("k_scale"), v_scale=vals.get("v_scale"), partition_size=-1,
                          workspace=ws, stream=stream, k_new=vals["k_new"], v_new=vals["v_new"],
                          slot_mapping=st["slots"])
    dec_bytes, app_bytes = algorithmic_bytes(wl, st["lens_h"])
    sampler = ClockSampler(dev.index if not os.environ.get("CUDA_VISIBLE_DEVICES") else
                           int(os.environ["CUDA_VISIBLE_DEVICES"].split(",")[0]))
    for _ in range(args.warmup):
        plan.run()
    torch.cuda.synchronize(dev)
    t_soak = time.time()
    while time.time() - t_soak < 0.6:
        for _ in range(20):
            plan.run()
        torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    e0.record(stream)
    for i in range(args.steps):
        starts[i].record(stream)
        plan.run()
        ends[i].record(stream)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    t1 = time.time()
    clocks = sampler.stop(t_soak, t1)
    if pkv.device_error(reset=True, device=dev):
        raise RuntimeError(f"a kernel flagged a device-side error in workload {name}")
    call_us = statistics.mean(starts[i].elapsed_time(ends[i]) for i in range(args.steps)) * 1e3
    step_ms = e0.elapsed_time(e1) / args.steps
    call_gbs = (dec_bytes + app_bytes) / (call_us * 1e-6) / 1e9
    step_gbs = (dec_bytes + app_bytes) / (step_ms * 1e-3) / 1e9
    P = pkv.resolve_partition_size(B, wl.num_q_heads, wl.num_kv_heads, wl.head_dim, st["tables_h"].shape[1],
                                   wl.block_size, -1)
    # the library's automatic choice: tensor cores for >= 4 query heads per kv head at head_dim 128, or
    # at head_dim 64 with a 16-bit cache and an even kv-head count (two kv heads per item), with
    # partitions of at most 512 tokens (batches above 2048 sequences in several launches)
    dims = wl.head_dim == 128 or (wl.head_dim == 64 and wl.cache_dtype != "e4m3" and wl.num_kv_heads % 2 == 0)
    grouped = wl.num_q_heads // wl.num_kv_heads >= 4 and dims and P <= 512
    path = "tensor-core" if grouped else "CUDA-core"
    res = {"description": wl.description, "kernel": path, "partition_size": P,
           "decode_call_gbs": round(call_gbs, 1), "frac": round(call_gbs / peak, 4),
           "avg_call_us": round(call_us, 2), "step_gbs": round(step_gbs, 1), "step_frac": round(step_gbs / peak, 4),
           "algorithmic_bytes_per_step": dec_bytes + app_bytes,
           "seq_steps_per_s": round(B / (step_ms * 1e-3), 1), "clocks": clocks}
    del plan, ws, st
    return res


def cpu_baseline(st, budget_s=20.0, max_seqs=None):
    """The float64 oracle on a bounded sample of the same batch (host cores)."""
    import oracle

    wl, vals = st["wl"], st["vals"]
    lens = st["lens_h"]
    order = np.argsort(lens)[::-1] if max_seqs else np.arange(len(lens))
    # time one sequence first to size the sample to the budget
    idx = [int(order[0])]
    code = {"f16": oracle.F16, "bf16": oracle.BF16, "e4m3": oracle.E4M3}
    kc, vc = bits(vals["k_cache"]), bits(vals["v_cache"])
    ks = float(vals["k_scale"].item()) if "k_scale" in vals else 1.0
    vs = float(vals["v_scale"].item()) if "v_scale" in vals else 1.0
    q = bits(vals["q"])

    def run(sel):
        sel = np.asarray(sel)
        t = time.perf_counter()
        oracle.paged_decode(np.ascontiguousarray(q[sel]), code[wl.act_dtype], kc, vc, code[wl.cache_dtype],
                            st["tables_h"][sel], lens[sel], wl.scale, k_scale=ks, v_scale=vs)
        return time.perf_counter() - t

    t1 = run(idx)
    n = int(min(len(lens), max(1, budget_s / max(t1, 1e-6) * 0.8)))
    sel = np.arange(len(lens))[:n]
    # repeat the sample until about budget_s seconds of CPU work have been timed
    t, reps = 0.0, 0
    while reps == 0 or t < budget_s * 0.8:
        t += run(sel)
        reps += 1
    t /= reps
    e = ELEM[wl.cache_dtype]
    kv = int(lens[sel].astype(np.int64).sum()) * 2 * wl.num_kv_heads * wl.head_dim * e
    dec, _ = algorithmic_bytes(wl, lens[sel])
    return {"value": round(dec / t / 1e9, 4), "unit": "GB/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"float64 oracle decode of {n} of {len(lens)} sequences of the {wl.name} batch "
                      f"({kv / 1e9:.3f} GB of K/V), {reps} repetitions, {t:.3f} s each",
            "seconds": round(t, 3)}


def run_reference(args):
    """The reference arm: the float64 CPU oracle, timed on the host cores, same metric."""
    dist, rank, world, local = _dist()
    if rank != 0:
        return
    import oracle
    from paged_kv_cache_102_gb300 import workloads as W
    from oracle.block_manager_ref import RefBlockManager

    oracle.build()
    d = W.draw(args.workload, args.seed)
    wl = d.workload
    vals = W.make_values(d, device="cpu")
    B = len(d.context_lens)
    ref = RefBlockManager(d.num_blocks, wl.block_size, free_list=d.free_list)
    for i, c in enumerate(d.context_lens):
        ref.add_sequence(i, int(c))
    slots = np.array([ref.append_slot(i)[0] for i in range(B)], np.int64)
    maxb = max(len(t) for t in ref.tables.values())
    tables = np.zeros((B, maxb), np.int32)
    for i in range(B):
        tables[i, : len(ref.tables[i])] = ref.tables[i]
    lens = (d.context_lens + 1).astype(np.int32)
    code = {"f16": oracle.F16, "bf16": oracle.BF16, "e4m3": oracle.E4M3}
    kc, vc = bits(vals["k_cache"]).copy(), bits(vals["v_cache"]).copy()
    ks = float(vals["k_scale"].item()) if "k_scale" in vals else 1.0
    vs = float(vals["v_scale"].item()) if "v_scale" in vals else 1.0
    q = bits(vals["q"])
    # size each step's sample so that warmup + steps take about budget seconds
    t = time.perf_counter()
    oracle.paged_decode(q[:1].copy(), code[wl.act_dtype], kc, vc, code[wl.cache_dtype], tables[:1], lens[:1],
                        wl.scale, k_scale=ks, v_scale=vs)
    t1 = max(time.perf_counter() - t, 1e-6) * float(lens.mean()) / float(lens[0])
    per_step = args.cpu_budget / max(1, args.steps + args.warmup)
    n = int(min(B, max(1, per_step / t1)))
    sel = np.arange(n)

    def step():
        oracle.append(bits(vals["k_new"][sel]), bits(vals["v_new"][sel]), code[wl.act_dtype], slots[sel], kc, vc,
                      code[wl.cache_dtype], k_scale=ks, v_scale=vs)
        oracle.paged_decode(np.ascontiguousarray(q[sel]), code[wl.act_dtype], kc, vc, code[wl.cache_dtype],
                            tables[sel], lens[sel], wl.scale, k_scale=ks, v_scale=vs)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    dec, app = algorithmic_bytes(wl, lens[sel])
    value = (dec + app) / dt / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic N(0,1), seeded",
        "config": {"workload": wl.name, "description": wl.description, "sample_seqs": n, "num_seqs": B},
        "seq_steps_per_s": round(n / dt, 3),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": f"{n} of {B} sequences of the {wl.name} batch per step (append + decode)"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_swap(args):
    """Swap bandwidth between the pools and pinned host memory, by block size:
    one gather/scatter launch for all blocks vs one cudaMemcpyAsync per block."""
    import paged_kv_cache_102_gb300 as pkv
    dev = torch.device("cuda", 0)
    pkv.load()
    Hkv, D = 32, 128
    total = 1 << 30  # bytes of K+V moved per direction
    # the ceiling on this machine: one contiguous 1 GiB cudaMemcpyAsync per direction
    dbuf = torch.empty(total, dtype=torch.uint8, device=dev).fill_(1)
    hbuf = torch.empty(total, dtype=torch.uint8).pin_memory()
    ceiling = {}
    for name, (dst, src) in (("out", (hbuf, dbuf)), ("in", (dbuf, hbuf))):
        for _ in range(2):
            dst.copy_(src, non_blocking=True)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(args.steps):
            dst.copy_(src, non_blocking=True)
        e1.record()
        torch.cuda.synchronize()
        ceiling[name] = total * args.steps / (e0.elapsed_time(e1) * 1e-3) / 1e9
    del dbuf, hbuf
    print(json.dumps({"measure": "ceiling: one contiguous 1 GiB pinned cudaMemcpyAsync per direction",
                      "memcpy_out_gbs": round(ceiling["out"], 1), "memcpy_in_gbs": round(ceiling["in"], 1)}),
          flush=True)
    for bs in (1, 4, 16, 32, 64):
        block_bytes = Hkv * bs * D * 2
        n = total // (2 * block_bytes)
        NB = 2 * n
        kc = torch.empty(NB, Hkv, bs, D, dtype=torch.bfloat16, device=dev).normal_()
        vc = torch.empty_like(kc).normal_()
        ids = torch.randperm(NB, device=dev)[:n].to(torch.int32)
        staging = torch.empty(n, 2, block_bytes, dtype=torch.uint8).pin_memory()
        res = {}
        for name, direction in (("out", pkv.SWAP_OUT), ("in", pkv.SWAP_IN)):
            for _ in range(2):
                pkv.paged_block_swap(kc, vc, ids, staging, direction)
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(args.steps):
                pkv.paged_block_swap(kc, vc, ids, staging, direction)
            e1.record()
            torch.cuda.synchronize()
            res[f"kernel_{name}_gbs"] = round(total * args.steps / (e0.elapsed_time(e1) * 1e-3) / 1e9, 1)
        # per-block copies (what a loop of cudaMemcpyAsync calls would do), swap-out direction
        ids_h = ids.cpu().numpy()
        kflat, vflat = kc.view(NB, -1).view(torch.uint8), vc.view(NB, -1).view(torch.uint8)
        m = min(n, 4096)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record()
        for j in range(m):
            staging[j, 0].copy_(kflat[int(ids_h[j])], non_blocking=True)
            staging[j, 1].copy_(vflat[int(ids_h[j])], non_blocking=True)
        e1.record()
        torch.cuda.synchronize()
        res["per_block_memcpy_out_gbs"] = round(2 * block_bytes * m / (e0.elapsed_time(e1) * 1e-3) / 1e9, 1)
        res["kernel_out_frac_of_memcpy"] = round(res["kernel_out_gbs"] / ceiling["out"], 3)
        res["kernel_in_frac_of_memcpy"] = round(res["kernel_in_gbs"] / ceiling["in"], 3)
        print(json.dumps({"measure": "block swap, pools <-> pinned host memory", "block_size_tokens": bs,
                          "block_bytes_per_cache": block_bytes, "blocks": int(n), "bytes_per_direction": total,
                          **res}), flush=True)
        del kc, vc, staging


def run_quest(args):
    """QUEST step (append, metadata update, top-K selection, sparse decode) vs full decode."""
    import paged_kv_cache_102_gb300 as pkv
    from paged_kv_cache_102_gb300 import workloads as W
    dev = torch.device("cuda", 0)
    pkv.load()
    st = setup(pkv, W, args.workload, args.seed, dev, args.batch)
    wl, vals = st["wl"], st["vals"]
    bs = wl.block_size
    budget = max(1, args.quest // bs)
    kc, vc = vals["k_cache"], vals["v_cache"]
    ks, vs = vals.get("k_scale"), vals.get("v_scale")  # E4M3 caches
    kmeta = pkv.quest_block_minmax(kc, st["tables"], st["lens"], meta_dtype=W.DTYPES[wl.act_dtype])
    B = len(st["ids"])
    sel = torch.empty(B, wl.num_kv_heads, budget, dtype=torch.int32, device=dev)
    slen = torch.empty(B, wl.num_kv_heads, dtype=torch.int32, device=dev)
    out = torch.empty_like(vals["q"])

    def quest_step():
        pkv.paged_kv_append(vals["k_new"], vals["v_new"], st["slots"], kc, vc, ks, vs)
        pkv.quest_append_minmax(vals["k_new"], st["slots"], kmeta, bs, k_scale=ks)
        pkv.quest_select(vals["q"], kmeta, st["tables"], st["lens"], bs, budget, sel, slen)
        pkv.paged_attention_decode_sparse(vals["q"], kc, vc, sel, slen, wl.scale, out=out, k_scale=ks, v_scale=vs)

    def full_step():
        pkv.paged_attention_decode_append(vals["q"], vals["k_new"], vals["v_new"], st["slots"], kc, vc, st["tables"],
                                          st["lens"], wl.scale, out=out, k_scale=ks, v_scale=vs)

    def graph_us(fn):
        # one CUDA graph per phase: the four small launches of a QUEST step are
        # host-bound when issued one by one through the binding
        side = torch.cuda.Stream(dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            for _ in range(args.warmup):
                fn()
        torch.cuda.current_stream(dev).wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        for _ in range(args.warmup):
            g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(args.steps):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
        return round(e0.elapsed_time(e1) * 1e3 / args.steps, 2)

    res = {}
    phases = {"append": lambda: pkv.paged_kv_append(vals["k_new"], vals["v_new"], st["slots"], kc, vc, ks, vs),
              "metadata": lambda: pkv.quest_append_minmax(vals["k_new"], st["slots"], kmeta, bs, k_scale=ks),
              "select": lambda: pkv.quest_select(vals["q"], kmeta, st["tables"], st["lens"], bs, budget, sel, slen),
              "sparse_decode": lambda: pkv.paged_attention_decode_sparse(vals["q"], kc, vc, sel, slen, wl.scale,
                                                                         out=out, k_scale=ks, v_scale=vs)}
    for name, fn in phases.items():
        res[f"{name}_us"] = graph_us(fn)
    for name, fn in (("full", full_step), ("quest", quest_step)):
        res[f"{name}_us_per_step"] = graph_us(fn)
    res["timing"] = "CUDA graph replays, CUDA events; metadata (< L2) may stay L2-resident between isolated phase replays"
    e = ELEM[wl.cache_dtype]
    sel_tokens = int(slen.sum().item())
    full_tokens = int(st["lens_h"].sum()) * wl.num_kv_heads
    meta_bytes = sum(-(-int(L) // bs) for L in st["lens_h"]) * wl.num_kv_heads * 2 * wl.head_dim * e
    print(json.dumps({"measure": "QUEST top-K blocks vs full decode", "workload": wl.name,
                      "budget_tokens": budget * bs, "selected_kv_tokens": sel_tokens, "full_kv_tokens": full_tokens,
                      "kv_bytes_full": full_tokens * 2 * wl.head_dim * e,
                      "kv_bytes_selected": sel_tokens * 2 * wl.head_dim * e, "metadata_bytes": meta_bytes,
                      **res, "speedup": round(res["full_us_per_step"] / res["quest_us_per_step"], 2)}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="llama7b")
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--partition-size", type=int, default=-1)
    ap.add_argument("--batch", type=int, default=0, help="override the workload's batch (profiling only)")
    ap.add_argument("--swap", action="store_true", help="measure block swap bandwidth instead")
    ap.add_argument("--quest", type=int, default=0, help="measure QUEST with this token budget instead")
    ap.add_argument("--fused", type=int, default=1, help="1: append fused into the decode launch (default), 0: two launches")
    ap.add_argument("--kernel-path", type=int, default=0,
                    help="decode kernel: 0 library choice, 1 CUDA-core, 2/3 tensor-core (1 or 2 CTAs per SM)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the other target configurations reported in the line's `workloads` object")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--ncu", action="store_true",
                    help="profiling run: only warmup + timed steps (no clock soak, e2e or CPU baseline)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.swap:
        run_swap(args)
    elif args.quest:
        run_quest(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_native(args)


if __name__ == "__main__":
    main()
