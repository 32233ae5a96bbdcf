#!/usr/bin/env python3
"""Bench: gathered multi-LoRA shrink+expand on GB300, one JSON line on rank 0.

Headline workload (one "step"): the LoRA delta of a whole Llama-2-7B decode step at batch 32,
Distinct adapters (row i -> adapter i), r = 16, bf16: all seven projections (q, k, v, o
4096->4096; gate, up 4096->11008; down 11008->4096) of all 32 layers, rows grouped into SGMV
segments once and reused by every op. The step is issued as 128 grouped fused calls (q/k/v,
o, gate/up, down per layer) through the C ABI and replayed as a CUDA graph.

  value     rows/s with every input resident in HBM (2.8 GB of algorithmic traffic per step,
            far above the 129 MB L2, so no flush is needed between steps)
  e2e       the same metric with the step's inputs (x, base y) copied from pinned host memory
            and the result y copied back inside the timed region, each step issued by one call
            into the library (e2e.graph: the same with the step replayed as a CUDA graph)
  roofline  algorithmic bytes of the step's launches / their time, against the measured HBM copy
            bandwidth (MEASURED_PEAKS.json)
  cpu_baseline / --impl reference: the fp64 oracle on the host cores, on a bounded sample of the
            same step (some of its layers), scaled to the whole step
  configs   roofline fraction of each of the five workloads (small ones timed per call with an
            L2 flush in between)

Multi-GPU: the op has no exchange step; N ranks run N independent replicas (weak scaling), with
a barrier and the max over ranks around the timed region.
"""
from __future__ import annotations

import argparse
import hashlib
import json
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

import workloads as W  # noqa: E402
from workloads import costmodel as C  # noqa: E402

METRIC = "LoRA shrink+expand rows/s and % of HBM/tensor roofline, 7B decode bs32"
UNIT = "rows/s"
WORKLOAD = ("Llama-2-7B decode step, bs32, r16, bf16, Distinct (32 adapters): SGMV delta of q,k,v,o,gate,up,down "
            "x 32 layers (224 ops)")
FALLBACK_HBM = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


# ---------------------------------------------------------------------------------------------
# helpers


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM, "fallback"


def tensor_fraction(flops: float, secs: float) -> dict:
    """Tensor-pipe roofline of a contraction timed in isolation: algorithmic flops / time against
    the measured dense bf16 peak (cuBLAS, burst; fp16 has the same nominal rate)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        peak, src = float(json.load(open(p))["bf16_tflops"]), "measured bf16_tflops (cuBLAS, burst)"
    else:
        peak, src = FALLBACK_BF16_TFLOPS, "fallback"
    achieved = flops / secs / 1e12
    return {"achieved_tflops": round(achieved, 1), "peak_tflops": peak, "frac": round(achieved / peak, 4),
            "peak_source": src}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    return ws, int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0"))


def max_over_ranks(x: float, device=None) -> float:
    """The largest `x` over all ranks (the job is as slow as its slowest replica); x itself when
    there is no process group."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rows_per_s(world_size: int, rows_per_step: int, steps: int, slowest_secs: float) -> float:
    """Whole-job throughput of `world_size` replicas: every rank processed rows_per_step rows per
    step, the job took as long as its slowest rank."""
    return world_size * rows_per_step * steps / slowest_secs


class ClockSampler:
    """nvidia-smi clocks/throttle reasons sampled every 200 ms; keep the samples taken between
    start() and stop()."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.lines, self.proc, self.t0, self.t1 = [], None, None, None
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "200", "-i", str(gpu_index)], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.th = threading.Thread(target=self._read, daemon=True)
        self.th.start()
        deadline = time.time() + 5
        while not self.lines and time.time() < deadline:
            time.sleep(0.05)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def start(self):
        self.t0 = time.time()

    def stop(self):
        self.t1 = time.time()
        time.sleep(0.25)
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        rows = [l.split(", ") for t, l in self.lines if self.t0 - 0.2 <= t <= self.t1 + 0.2]
        rows = [r for r in rows if len(r) >= 9]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.strip().lower() == "active"})
        pw = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "power_w_max": max(pw) if pw else None}


def kernel_source_hash():
    """Hash of the decode kernel's sources: a committed ncu traffic figure counts only for them."""
    h = hashlib.sha256()
    for f in ("decode_impl.cuh", "decode_fused.cu", "decode_launch.cu", "common.cuh", "launch.h"):
        h.update(open(os.path.join(ROOT, "adapter_gemv_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, workload_key: str):
    """Per-launch DRAM bytes from a committed ncu summary, if it was taken on the current kernel source."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    e = d.get(workload_key)
    if not e or e.get("kernel") != kernel or e.get("source_hash") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


# ---------------------------------------------------------------------------------------------
# the headline step


def io_set(w, dev):
    """The step's activations (every distinct x) and base outputs (every y) re-homed into two flat
    device buffers, with ops that point at them: one host-to-device copy of each buffer brings a
    whole step's inputs in, one device-to-host copy of the y buffer takes its result out."""
    xs = []
    for op in w.ops:
        if all(op.x.data_ptr() != x.data_ptr() for x in xs):
            xs.append(op.x)
    xbuf = torch.empty(sum(x.numel() for x in xs), dtype=w.dtype, device=dev)
    ybuf = torch.empty(sum(op.y.numel() for op in w.ops), dtype=w.dtype, device=dev)
    xview, o = {}, 0
    for x in xs:
        v = xbuf[o:o + x.numel()].view(x.shape)
        v.copy_(x)
        xview[x.data_ptr()] = v
        o += x.numel()
    ops, o = [], 0
    for op in w.ops:
        v = ybuf[o:o + op.y.numel()].view(op.y.shape)
        v.copy_(op.y)
        ops.append(W.Op(op.name, op.pool, op.layer, xview[op.x.data_ptr()], v))
        o += op.y.numel()
    return ops, xbuf, ybuf


def build_step(dev, dist="distinct"):
    import adapter_gemv_gb300 as m
    from adapter_gemv_gb300.plan import StepPlan
    w = W.sgmv_decode_7b(device=dev, dist=dist)
    w.ops, xbuf, ybuf = io_set(w, dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    plan = StepPlan(w.ops, w.batch, status)
    return w, plan, ybuf, xbuf, status, m


def e2e_pipeline(plans, graphs, xbufs, ybufs, steps, dev, use_graphs):
    """End-to-end time of `steps` decode steps with host buffers: step k's activations and base
    outputs are copied in from pinned host memory and its result copied back, every step. Three
    device buffer sets rotate, so step k+1's input copy and step k-1's output copy run on their
    own streams while step k computes (the copies are inside the timed region; they only overlap
    with compute). Step k is issued through the library's public API: one lora_sgmv_sequence call
    (use_graphs False) or a replay of a CUDA graph captured from it (use_graphs True).
    Returns (seconds, h2d bytes per step, d2h bytes per step)."""
    n = len(plans)
    comp, cin, cout = (torch.cuda.Stream(device=dev) for _ in range(3))
    host_x = torch.empty(xbufs[0].shape, dtype=xbufs[0].dtype, pin_memory=True)
    host_y = torch.empty(ybufs[0].shape, dtype=ybufs[0].dtype, pin_memory=True)
    host_x.copy_(xbufs[0])
    host_y.copy_(ybufs[0])
    host_out = [torch.empty(host_y.shape, dtype=host_y.dtype, pin_memory=True) for _ in range(n)]
    ev_in = [torch.cuda.Event() for _ in range(n)]
    ev_comp = [torch.cuda.Event() for _ in range(n)]
    ev_out = [torch.cuda.Event() for _ in range(n)]
    torch.cuda.synchronize()

    def copy_in(k):
        b = k % n
        cin.wait_event(ev_out[b])  # the buffer's previous result has been copied out
        with torch.cuda.stream(cin):
            xbufs[b].copy_(host_x, non_blocking=True)
            ybufs[b].copy_(host_y, non_blocking=True)
        ev_in[b].record(cin)

    def run(steps_, start=None, end=None):
        if start is not None:
            start.record(cin)
        copy_in(0)
        for k in range(steps_):
            b = k % n
            if k + 1 < steps_:
                copy_in(k + 1)
            comp.wait_event(ev_in[b])
            if use_graphs:
                with torch.cuda.stream(comp):
                    graphs[b].replay()
            else:
                plans[b](comp)
            ev_comp[b].record(comp)
            cout.wait_event(ev_comp[b])
            with torch.cuda.stream(cout):
                host_out[b].copy_(ybufs[b], non_blocking=True)
            ev_out[b].record(cout)
        if end is not None:
            end.record(cout)

    run(2 * n)  # warm-up
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    run(steps, start, end)
    end.synchronize()
    torch.cuda.synchronize()
    h2d = xbufs[0].numel() * xbufs[0].element_size() + ybufs[0].numel() * ybufs[0].element_size()
    d2h = ybufs[0].numel() * ybufs[0].element_size()
    return start.elapsed_time(end) / 1e3, h2d, d2h


def step_bytes(w):
    slots = w.batch.row_slot.cpu().numpy()
    rs = {id(p): p.rank.cpu().numpy() for p in w.pools}
    total = 0
    for op in w.ops:
        r = rs[id(op.pool)]
        row_ranks = [int(r[s]) for s in slots if s >= 0]
        distinct = [int(r[s]) for s in np.unique(slots[slots >= 0])]
        total += C.op_bytes(d_in=op.pool.d_in, d_out=op.pool.d_out, row_ranks=row_ranks, distinct_ranks=distinct,
                            v_roundtrip=False)
    return total


def time_graph(graph, stream, steps, sampler=None):
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
    with torch.cuda.stream(stream):  # replay() launches on the current stream
        start.record(stream)
        for _ in range(steps):
            graph.replay()
        end.record(stream)
    end.synchronize()
    if sampler:
        sampler.stop()
    return start.elapsed_time(end) / 1e3  # seconds


def capture(fn, stream):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        fn(stream)  # warm: sets kernel attributes outside capture
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=stream):
            fn(stream)
    torch.cuda.synchronize()
    return g


# ---------------------------------------------------------------------------------------------
# CPU oracle on a bounded sample of the step


def _oracle_layer_inputs(w, layer):
    import oracle
    bits = lambda t: t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)
    out = []
    for op in w.ops:
        if op.layer != layer:
            continue
        p = op.pool
        opool = oracle.Pool(dtype=oracle.DTYPE_BF16, num_slots=p.num_slots, num_layers=1, r_max=p.r_max,
                            d_in=p.d_in, d_out=p.d_out, rank=p.rank.cpu().numpy(), scale=p.scale.cpu().numpy(),
                            a_t=bits(p.a_t[:, layer:layer + 1]), b=bits(p.b[:, layer:layer + 1]))
        out.append((opool, bits(op.x), bits(op.y)))
    return out


def oracle_sample(w, budget_s: float):
    import oracle
    off = w.batch.seg_offsets.cpu().numpy()
    ss = w.batch.seg_slot.cpu().numpy()
    spent, layers = 0.0, 0
    for layer in range(32):
        inputs = _oracle_layer_inputs(w, layer)
        t0 = time.perf_counter()
        for opool, x, y in inputs:
            oracle.sgmv(opool, 0, x, y, off, ss)
        spent += time.perf_counter() - t0
        layers += 1
        if spent >= budget_s:
            break
    per_step = spent / layers * 32
    return per_step, layers


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_sample_all_cores(w, budget_s: float, threads: int = 0):
    """The same oracle on every host core: one thread per layer, in batches of as many layers as
    there are threads (ctypes releases the GIL around each C call, so the threads run at once).
    Only the batches' compute is timed; each batch's inputs are copied to host memory before it.
    Returns (seconds per whole step, layers sampled, threads used)."""
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    off = w.batch.seg_offsets.cpu().numpy()
    ss = w.batch.seg_slot.cpu().numpy()
    n_layers = 1 + max(op.layer for op in w.ops)
    threads = threads or host_cores()
    lib = oracle.default()  # built before the threads start

    def run_layer(inputs):
        for opool, x, y in inputs:
            lib.sgmv(opool, 0, x, y, off, ss)

    spent, layers, used = 0.0, 0, 0
    with ThreadPoolExecutor(threads) as ex:
        for base in range(0, n_layers, threads):
            batch = [_oracle_layer_inputs(w, layer) for layer in range(base, min(n_layers, base + threads))]
            t0 = time.perf_counter()
            list(ex.map(run_layer, batch))
            spent += time.perf_counter() - t0
            layers += len(batch)
            used = max(used, len(batch))
            if spent >= budget_s:
                break
    return spent / layers * n_layers, layers, used


# ---------------------------------------------------------------------------------------------
# per-workload roofline fractions


def flush_l2(buf):
    buf.add_(1)


def time_calls(fn, stream, iters, flush):
    """Device time of one call with a cold L2: replay a graph of `iters` x [flush, call] and one of
    `iters` x [flush], both without host gaps, and take the difference per call."""
    def body_both(s):
        for _ in range(iters):
            flush_l2(flush)
            fn(s)

    def body_flush(s):
        for _ in range(iters):
            flush_l2(flush)

    g_both, g_flush = capture(body_both, stream), capture(body_flush, stream)
    best = []
    for _ in range(3):
        tb = time_graph(g_both, stream, 1)
        tf = time_graph(g_flush, stream, 1)
        best.append((tb - tf) / iters)
    return max(min(best), 1e-9)


def config_fractions(dev, stream, peak, iters=30):
    import adapter_gemv_gb300 as m
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)  # 256 MB > 129 MB L2
    res = {}

    def op_bytes_of(op, batch, v_roundtrip=False):
        slots = batch.row_slot.cpu().numpy()
        r = op.pool.rank.cpu().numpy()
        return C.op_bytes(d_in=op.pool.d_in, d_out=op.pool.d_out, row_ranks=[int(r[s]) for s in slots if s >= 0],
                          distinct_ranks=[int(r[s]) for s in np.unique(slots[slots >= 0])], v_roundtrip=v_roundtrip)

    def op_flops_of(op, batch):
        slots = batch.row_slot.cpu().numpy()
        r = op.pool.rank.cpu().numpy()
        return C.op_flops(d_in=op.pool.d_in, d_out=op.pool.d_out, row_ranks=[int(r[s]) for s in slots if s >= 0])

    def single(name, w, form):
        op = w.ops[0]
        h = m.make_pool(op.pool)
        v = torch.empty((w.batch.M, op.pool.r_max), dtype=torch.float32, device=dev)
        b = w.batch
        if form == "sgmv":
            fused = lambda s: m.lora_sgmv(op.y, op.x, h, b.seg_offsets, b.seg_slot, op.layer, v, stream=s)
            two = lambda s: (m.lora_sgmv_shrink(v, op.x, h, b.seg_offsets, b.seg_slot, op.layer, stream=s),
                             m.lora_sgmv_expand(op.y, v, h, b.seg_offsets, b.seg_slot, op.layer, stream=s))
        else:
            fused = lambda s: m.lora_bgmv(op.y, op.x, h, b.row_slot, op.layer, v, stream=s)
            two = lambda s: (m.lora_bgmv_shrink(v, op.x, h, b.row_slot, op.layer, stream=s),
                             m.lora_bgmv_expand(op.y, v, h, b.row_slot, op.layer, stream=s))
        out = {}
        for label, fn, vr in (("fused", fused, False), ("two_launch", two, True)):
            t = time_calls(fn, stream, iters, flush)
            by = op_bytes_of(op, b, vr)
            out[label] = {"us": round(t * 1e6, 2), "bytes": by, "gbs": round(by / t / 1e9, 1),
                          "frac": round(by / t / 1e9 / peak, 4)}
        res[name] = out

    single("1_tiny_sgmv_fp16", W.tiny_sgmv(device=dev), "sgmv")
    single("2_bgmv_q_proj_distinct", W.bgmv_decode_q(device=dev), "bgmv")
    for dist in ("distinct", "uniform", "skewed", "identical"):
        w, plan, *_ = build_step(dev, dist)
        g = capture(plan, stream)
        t = time_graph(g, stream, 20) / 20
        by = step_bytes(w)
        res[f"3_decode_7b_{dist}"] = {"us_per_step": round(t * 1e6, 1), "bytes": by, "gbs": round(by / t / 1e9, 1),
                                      "frac": round(by / t / 1e9 / peak, 4), "launches": plan.launches}
        del w, plan, g
        torch.cuda.empty_cache()
    def seven_ops(name, w):
        """The 7 projections of a prefill-sized batch, one fused call each (L2 flushed per call)."""
        tot_t, tot_b, tot_f = 0.0, 0, 0
        for op in w.ops:
            h = m.make_pool(op.pool)
            v = torch.empty((w.batch.M, op.pool.r_max), dtype=torch.float32, device=dev)
            fn = lambda s, op=op, h=h, v=v: m.lora_sgmv(op.y, op.x, h, w.batch.seg_offsets, w.batch.seg_slot, 0, v,
                                                         stream=s)
            tot_t += time_calls(fn, stream, 5, flush)
            tot_b += op_bytes_of(op, w.batch)
            tot_f += op_flops_of(op, w.batch)
        res[name] = {"us_7_ops": round(tot_t * 1e6, 1), "bytes": tot_b, "gbs": round(tot_b / tot_t / 1e9, 1),
                     "frac": round(tot_b / tot_t / 1e9 / peak, 4), "rows": w.batch.M, "segments": int(w.batch.seg_slot.numel()),
                     "flops": tot_f, "tensor": tensor_fraction(tot_f, tot_t)}

    seven_ops("4_prefill_13b", W.sgmv_prefill_13b(device=dev))
    torch.cuda.empty_cache()
    seven_ops("6_mixed_prefill_decode_13b", W.mixed_prefill_decode_13b(device=dev))
    torch.cuda.empty_cache()
    single("5_paged_hetero_70b", W.paged_decode_70b(device=dev), "bgmv")
    # the same pool with 2048 rows: the adapters the rows use (about 1.1 GB) exceed L2, so reading
    # each once per call needs the rows grouped by adapter (device-side grouping, lora_bgmv's default
    # from 128 rows) -- timed with and without it
    w = W.paged_decode_70b(device=dev, M=2048)
    op = w.ops[0]
    h = m.make_pool(op.pool)
    v = torch.empty((w.batch.M, op.pool.r_max), dtype=torch.float32, device=dev)
    by = op_bytes_of(op, w.batch)
    out = {}
    for label, fl in (("grouped", m.LAUNCH_GROUP_ROWS), ("ungrouped", m.LAUNCH_NO_GROUPING)):
        t = time_calls(lambda s, fl=fl: m.lora_bgmv_ex(op.y, op.x, h, w.batch.row_slot, 0, v, fl, stream=s), stream,
                       10, flush)
        out[label] = {"us": round(t * 1e6, 1), "bytes": by, "gbs": round(by / t / 1e9, 1),
                      "frac": round(by / t / 1e9 / peak, 4)}
    res["5b_paged_70b_2048_rows"] = out
    del w, op, h, v
    torch.cuda.empty_cache()
    return res


# ---------------------------------------------------------------------------------------------


def run_ours(args):
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(device=dev)
    hbm, peak_kind = peaks()

    w, plan, ybuf, xbuf, status, m = build_step(dev, "distinct")
    rows = w.batch.M
    bytes_step = step_bytes(w)
    g = capture(plan, stream)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            g.replay()
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {status.item()} during warm-up")

    def barrier():
        if ws > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    sampler = ClockSampler(dev.index if dev.index is not None else 0) if rank == 0 else None
    barrier()
    secs = time_graph(g, stream, args.steps, sampler)
    barrier()
    secs = max_over_ranks(secs, dev)
    ms = secs / args.steps * 1e3
    value = job_rows_per_s(ws, rows, args.steps, secs)

    # e2e: pinned host inputs -> device, the step, result back to the host, every step; three
    # buffer sets so the copies of the neighbouring steps overlap this step's compute
    from adapter_gemv_gb300.plan import StepPlan
    plans, graphs, xbufs, ybufs = [plan], [g], [xbuf], [ybuf]
    for _ in range(2):
        ops_k, xb_k, yb_k = io_set(w, dev)
        p_k = StepPlan(ops_k, w.batch, status)
        plans.append(p_k)
        graphs.append(capture(p_k, stream))
        xbufs.append(xb_k)
        ybufs.append(yb_k)
    e2e_steps = max(3, min(args.steps, 200))
    e2e_secs, h2d, d2h = e2e_pipeline(plans, graphs, xbufs, ybufs, e2e_steps, dev, use_graphs=False)
    e2e_secs = max_over_ranks(e2e_secs, dev)
    e2e_g_secs, _, _ = e2e_pipeline(plans, graphs, xbufs, ybufs, e2e_steps, dev, use_graphs=True)
    e2e_g_secs = max_over_ranks(e2e_g_secs, dev)
    del plans, graphs, xbufs, ybufs
    if rank != 0:
        if ws > 1:
            torch.distributed.destroy_process_group()
        return

    achieved = bytes_step / (secs / args.steps) / 1e9
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "global_batch": rows * ws, "rows_per_step_per_gpu": rows, "rank": 16,
                   "ops_per_step": len(w.ops), "launch": f"CUDA graph of {plan.launches} grouped fused calls",
                   "l2": "inputs larger than L2 (2.8 GB of adapter weights and activations per step)",
                   "parallelism": f"replicas x{ws}"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(achieved / hbm, 4), "peak_source": f"{peak_kind} hbm_gbs (copy)",
                     "kernel": "decode_kernel<bf16, FUSED> (every launch of the step)",
                     "algorithmic_bytes_per_launch": bytes_step // plan.launches,
                     "traffic": ncu_traffic("decode_kernel_fused", "decode7b_distinct")},
        "e2e": {"value": round(job_rows_per_s(ws, rows, e2e_steps, e2e_secs), 1), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_secs / e2e_steps * 1e3, 4),
                "api": f"one lora_sgmv_sequence call per step (its {plan.launches} grouped calls issued by the "
                       "library, no CUDA graph); x and base y copied in from pinned host memory and y copied "
                       "out every step, the copies of the next and previous steps overlapping this step's compute",
                "graph": {"value": round(job_rows_per_s(ws, rows, e2e_steps, e2e_g_secs), 1),
                          "ms_per_step": round(e2e_g_secs / e2e_steps * 1e3, 4),
                          "api": "the same, each step a replay of a CUDA graph captured from that call"}},
        "gpu_launches": plan.launches * args.steps,
        "clocks": sampler.summary() if sampler else None,
    }
    if ws == 1 and not args.no_cpu_baseline:
        per_step, layers = oracle_sample(w, args.cpu_seconds)
        line["cpu_baseline"] = {"value": round(rows / per_step, 3), "unit": UNIT, "cores": 1, "kind": "oracle",
                                "sample": f"fp64 oracle on {layers} of 32 layers (all 7 ops each) of the same step, "
                                          f"single thread, scaled x{32 / layers:.2f} to the step"}
        per_step_mc, layers_mc, used = oracle_sample_all_cores(w, args.cpu_seconds)
        line["cpu_baseline"]["all_cores"] = {
            "value": round(rows / per_step_mc, 3), "unit": UNIT, "cores": used,
            "sample": f"the same oracle, one thread per layer ({used} at once) on {layers_mc} of 32 layers, "
                      f"scaled x{32 / layers_mc:.2f} to the step"}
    del g, plan, w
    torch.cuda.empty_cache()
    if not args.no_configs:
        line["configs"] = config_fractions(dev, stream, hbm)
    print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


def run_reference(args):
    """The oracle as the reference arm: all host cores, same metric and workload. Each step is a
    bounded sample -- some rows of one layer's 7 projections, split over one thread per core
    (ctypes releases the GIL around each C call) -- scaled to the whole step (32 rows x 224
    ops), sized so that the whole --steps/--warmup run takes about REFERENCE_BUDGET_S seconds."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    from concurrent.futures import ThreadPoolExecutor
    w = W.sgmv_decode_7b(device="cpu", dist="distinct", num_layers=1)  # one layer: the step's per-layer work
    import oracle
    lib = oracle.default()
    off, ss = w.batch.seg_offsets.numpy(), w.batch.seg_slot.numpy()
    inputs = _oracle_layer_inputs(w, 0)
    M = w.batch.M
    threads = host_cores()

    def rows_part(rows):
        for opool, x, y in inputs:
            lib.sgmv(opool, 0, x, y, off, ss, rows=rows)

    with ThreadPoolExecutor(threads) as ex:
        def one(rows):  # the rows dealt round-robin over the threads; wall time
            parts = [rows[i::threads] for i in range(threads) if rows[i::threads]]
            t0 = time.perf_counter()
            list(ex.map(rows_part, parts))
            return time.perf_counter() - t0, len(parts)

        per_row, _ = one([0])  # calibration: one row of the 7 ops on one thread
        budget = REFERENCE_BUDGET_S / max(1, args.steps + args.warmup)
        n = int(min(M, max(1, threads * (budget // max(per_row, 1e-9)))))
        for k in range(args.warmup):
            one([(k * n + i) % M for i in range(n)])
        per_step, used = [], 0
        for k in range(args.steps):
            t, u = one([(k * n + i) % M for i in range(n)])
            per_step.append(t * (M / n) * 32)  # scale to all rows and all 32 layers
            used = max(used, u)
    step_s = sum(per_step) / len(per_step)
    value = M / step_s
    sample = (f"each step: the fp64 oracle on {n} of {M} rows of one layer's 7 projections, {used} threads "
              f"(one per host core, rows split between them), scaled x{M / n * 32:.0f}")
    line = {"metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(step_s * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": WORKLOAD},
            "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": used, "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


REFERENCE_BUDGET_S = 120.0


NCU_TARGETS = ("decode7b", "decode7b-2layers", "decode7b-identical-2layers", "q_proj", "prefill13b-q", "paged70b", "paged70b-ungrouped")


def run_ncu_target(name: str, reps: int):
    """Run one workload `reps` times with no timing, as a target for ncu (nothing is printed but
    'ok'). decode7b-2layers is the decode step with 2 layers: the same launches per layer, a
    smaller footprint for multi-pass captures; decode7b-identical-2layers the same with every row
    on one adapter; paged70b-ungrouped the paged 70B batch with no row grouping."""
    import adapter_gemv_gb300 as m
    from adapter_gemv_gb300.plan import StepPlan
    dev = torch.device("cuda", 0)
    if name.startswith("decode7b"):
        w = W.sgmv_decode_7b(device=dev, num_layers=2 if name.endswith("2layers") else 32,
                             dist="identical" if "identical" in name else "distinct")
        plan = StepPlan(w.ops, w.batch)
        for _ in range(reps):
            plan()
    elif name == "q_proj":
        w = W.bgmv_decode_q(device=dev)
        op = w.ops[0]
        h = m.make_pool(op.pool)
        v = torch.empty((w.batch.M, op.pool.r_max), dtype=torch.float32, device=dev)
        for _ in range(reps):
            m.lora_bgmv(op.y, op.x, h, w.batch.row_slot, 0, v)
    elif name == "prefill13b-q":
        w = W.sgmv_prefill_13b(device=dev, projections=W.LLAMA2_13B[:1])
        op = w.ops[0]
        h = m.make_pool(op.pool)
        v = torch.empty((w.batch.M, op.pool.r_max), dtype=torch.float32, device=dev)
        for _ in range(reps):
            m.lora_sgmv(op.y, op.x, h, w.batch.seg_offsets, w.batch.seg_slot, 0, v)
    elif name.startswith("paged70b"):
        w = W.paged_decode_70b(device=dev)
        op = w.ops[0]
        h = m.make_pool(op.pool)
        v = torch.empty((w.batch.M, op.pool.r_max), dtype=torch.float32, device=dev)
        fl = m.LAUNCH_NO_GROUPING if name.endswith("ungrouped") else 0
        for _ in range(reps):
            m.lora_bgmv_ex(op.y, op.x, h, w.batch.row_slot, 0, v, fl)
    torch.cuda.synchronize()
    print("ok", name)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true")
    ap.add_argument("--ncu-target", choices=NCU_TARGETS, help="run one workload untimed, as an ncu target")
    ap.add_argument("--reps", type=int, default=2)
    args = ap.parse_args()
    if args.ncu_target:
        run_ncu_target(args.ncu_target, args.reps)
        return
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
