#!/usr/bin/env python3
"""Benchmark of the sliding-window GQA path on one GB300 (or N replicas).

One bench step is one whole single-stream job, every row of the hot path:
prefill of an 8192-token prompt into the prompt-sized cache for 26 sliding
layers (causal plan), compaction into the W + 64 = 1088-row buffer, then 512
decode steps (positions 8192..8703) -- per step one runtime mask shared by the
26 layers and 26 single-token decodes, replayed from one captured CUDA graph --
with the roll every 64 decode tokens (7 rolls).  B=1, Hq=4, Hkv=2, D=256,
W=1024, bf16 storage, fp32 accumulation, seeded synthetic N(0,1) data.

Headline: decode microseconds per layer (lower is better) = decode-phase
device time / (512 steps x 26 layers).  The same line carries prefill
TFLOP/s, the roofline of the dominant kernel, an end-to-end variant through
pinned host buffers, the CPU oracle baseline, and secondary workloads
(batched decode GB/s, chunked VLM prefill and packed-document prefill TFLOP/s,
and the packed-document training step: forward + backward TFLOP/s).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun every rank runs its own replica (the path shards by
independent sequences with no exchange); rank 0 prints one JSON line.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "SWA decode µs/layer & HBM GB/s; prefill TFLOP/s; % of GB300 roofline"
WORKLOAD = "single-stream decode: B=1 Hq=4 Hkv=2 D=256 W=1024, prompt 8192, 26 layers, 512 steps (7 rolls)"
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# Runtime-mask SWA warm median at this decode shape (B=1, Hq=4, Hkv=2, D=256, W=1024, 1088
# rows) on IBM Spyre: the only published figure for this metric and workload (other hardware).
SPYRE_RUNTIME_MASK_US = 562.0
# The dominant kernel of the bench step and the committed summary of its ncu capture; the summary
# records the DRAM bytes of one launch and the SHA-256 of the kernel source it was taken on, and the
# bench reports that traffic only while the source is unchanged (else null).
DOMINANT_KERNEL = "decode_small_kernel<256, 2>"
DOMINANT_SOURCE = os.path.join("sliding_window_gqa_swa_gb300", "csrc", "decode_small_sm103.cu")
DOMINANT_PROFILE = os.path.join("profiles", "decode_small_kernel_single_stream.md")


# ----------------------------------------------------------------------------- helpers
def dist_env():
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(values, device=None):
    """Element-wise maximum of a list of floats over all ranks (identity when
    torch.distributed is not initialised or has one rank)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, "measured"
    except Exception:
        return dict(PEAKS_FALLBACK), "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"swa_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "200", "-i", str(self.gpu)], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        try:
            for line in open(self.path):
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        except Exception:
            pass
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        busy = [x for x in sm if x > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(busy), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


def profiled_traffic():
    """(DRAM bytes per launch, source) of the dominant kernel from its committed ncu summary, or
    (None, reason) when there is none or the kernel source changed since the capture."""
    import hashlib
    try:
        src = open(os.path.join(ROOT, DOMINANT_SOURCE), "rb").read()
        text = open(os.path.join(ROOT, DOMINANT_PROFILE)).read()
    except OSError:
        return None, "no ncu summary of the current kernel"
    fields = {}
    for line in text.splitlines():
        line = line.strip().strip("`")
        if ":" in line:
            k, v = line.split(":", 1)
            fields[k.strip()] = v.strip()
    try:
        nbytes = int(fields["traffic_bytes_per_launch"])
        sha = fields["kernel_source_sha256"]
    except (KeyError, ValueError):
        return None, "ncu summary without a traffic line"
    if hashlib.sha256(src).hexdigest() != sha:
        return None, "kernel changed since the ncu capture"
    return nbytes, DOMINANT_PROFILE


def host_threads():
    """Host cores and the BLAS thread count NumPy's matrix products use (best effort)."""
    info = {"cores": os.cpu_count()}
    try:
        import threadpoolctl
        pools = threadpoolctl.threadpool_info()
        blas = [p_["num_threads"] for p_ in pools if p_.get("user_api") == "blas"]
        if blas:
            info["blas_threads"] = int(max(blas))
            return info
    except Exception:
        pass
    try:  # the OpenBLAS that NumPy loaded, asked directly
        import ctypes
        libs = set()
        with open("/proc/self/maps") as f:
            for line in f:
                path = line.split()[-1] if line.split() else ""
                if "openblas" in os.path.basename(path).lower():
                    libs.add(path)
        for path in libs:
            lib = ctypes.CDLL(path)
            for name in ("scipy_openblas_get_num_threads64_", "openblas_get_num_threads64_",
                         "openblas_get_num_threads", "scipy_openblas_get_num_threads"):
                fn = getattr(lib, name, None)
                if fn is not None:
                    info["blas_threads"] = int(fn())
                    return info
    except Exception:
        pass
    env = os.environ.get("OPENBLAS_NUM_THREADS") or os.environ.get("OMP_NUM_THREADS")
    info["blas_threads"] = int(env) if env else None
    return info


def admitted_pairs(seq_len: int, window: int, pad: int, img) -> int:
    """Admitted pairs per head of one padded sequence with image blocks: a
    query q >= pad sees keys [max(pad, q - W + 1), q], extended to the end of
    its image block when q is an image token (window AND (causal OR same image))."""
    q = np.arange(seq_len)
    lo = np.maximum(pad, q - window + 1)
    img = np.asarray(img)
    run_end = np.arange(seq_len)
    for i in range(seq_len - 2, -1, -1):
        if img[i] >= 0 and img[i + 1] == img[i]:
            run_end[i] = run_end[i + 1]
    hi = np.where(img >= 0, np.maximum(q, run_end), q)
    return int(np.where(q >= pad, hi - lo + 1, 0).sum())


def causal_pairs(seq_len: int, window: int) -> int:
    """Admitted (query, key) pairs per head of one unpadded causal sliding prompt."""
    w = min(window, seq_len)
    return w * (w + 1) // 2 + (seq_len - w) * window


def ev():
    return torch.cuda.Event(enable_timing=True)


# ----------------------------------------------------------------------------- the job
class SingleStreamJob:
    """The whole single-stream job on one GPU (one bench step)."""

    def __init__(self, swa, case, dev, e2e=False, ring=False, l2_flush=None):
        self.swa, self.dev, self.e2e = swa, dev, e2e
        # optional scratch buffer larger than L2, overwritten before every decode step's graph
        self.l2_flush = l2_flush
        c = case
        self.L, self.S, self.W, self.D = c.layers, c.prompt_len, c.window, c.head_dim
        self.B, self.Hq, self.Hkv, self.T = c.batch, c.q_heads, c.kv_heads, c.steps
        self.scale = self.D ** -0.5
        place = (lambda t: t.pin_memory()) if e2e else (lambda t: t.to(dev))
        self.pq, self.pk, self.pv = place(c.prompt_q), place(c.prompt_k), place(c.prompt_v)
        # each decode step's q, k_new and v_new for all layers, packed in one row so the step
        # stages its inputs with one copy
        T = c.steps
        self.nq, self.nk = c.dec_q[0].numel(), c.dec_k[0].numel()
        self.dec = place(torch.cat([c.dec_q.reshape(T, -1), c.dec_k.reshape(T, -1), c.dec_v.reshape(T, -1)], 1))
        if e2e:
            self.d_pq = torch.empty(c.prompt_q.shape, dtype=torch.bfloat16, device=dev)
            self.d_pk = torch.empty(c.prompt_k.shape, dtype=torch.bfloat16, device=dev)
            self.d_pv = torch.empty(c.prompt_v.shape, dtype=torch.bfloat16, device=dev)
            self.outs = torch.empty((self.T, self.L, self.B, self.Hq, self.D), dtype=torch.bfloat16).pin_memory()
        else:
            self.d_pq, self.d_pk, self.d_pv = self.pq, self.pk, self.pv
            self.outs = torch.empty((self.T, self.L, self.B, self.Hq, self.D), dtype=torch.bfloat16, device=dev)
        self.prefill_out = torch.empty((self.B, self.S, self.Hq, self.D), dtype=torch.bfloat16, device=dev)
        self.pre = swa.Cache(swa.CACHE_PREFILL, self.L, self.B, self.Hkv, self.D, self.W, self.S)
        # the anchored W + 64 buffer with a roll every 64 steps, or the modular ring of W rows
        self.cmp = swa.Cache(swa.CACHE_RING if ring else swa.CACHE_COMPACT, self.L, self.B, self.Hkv, self.D,
                             self.W, self.S)
        self.meta = swa.Meta(self.B, self.S, 0, self.S, self.W)
        self.mask = torch.empty(self.B, self.cmp.rows, dtype=torch.uint8, device=dev)
        self.ws = swa.decode_workspace(self.cmp, self.Hq)
        # staging buffers the captured step graph reads (views of one buffer) and writes: two
        # sets (one graph each, steps alternate), so a copy stream stages the next step's inputs
        # and stores the previous step's outputs while a step runs; one set, copied in line,
        # when L2 is flushed before every step (that variant times each step's graph alone)
        self.nbuf = 1 if l2_flush is not None else 2
        self.stage = [torch.empty(self.nq + 2 * self.nk, dtype=torch.bfloat16, device=dev) for _ in range(self.nbuf)]
        self.ob = [torch.empty((self.L, self.B, self.Hq, self.D), dtype=torch.bfloat16, device=dev)
                   for _ in range(self.nbuf)]
        self.graphs = [None] * self.nbuf
        self.copy_stream = torch.cuda.Stream(dev) if self.nbuf == 2 else None
        self.rolls = 0 if ring else (self.T - 1) // 64
        # kernels of ours per job: 2 cache bindings, (K/V write + attention) per layer, compaction,
        # (mask + one decode per layer) per step, rolls
        self.launches = 2 + 2 * self.L + 1 + self.T * (1 + self.L) + self.rolls
        self.h2d_bytes = (c.prompt_q.numel() + c.prompt_k.numel() + c.prompt_v.numel()
                          + self.dec.numel()) * 2 if e2e else 0
        self.d2h_bytes = self.outs.numel() * 2 if e2e else 0

    def _views(self, i):
        st = self.stage[i]
        return (st[:self.nq].view(self.L, self.B, self.Hq, self.D),
                st[self.nq:self.nq + self.nk].view(self.L, self.B, self.Hkv, self.D),
                st[self.nq + self.nk:].view(self.L, self.B, self.Hkv, self.D))

    def _capture(self, i):
        swa = self.swa
        qb, kb, vb = self._views(i)
        s = torch.cuda.Stream(self.dev)
        s.wait_stream(torch.cuda.current_stream(self.dev))
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            swa.build_decode_mask(self.cmp, self.mask, stream=s)
            for layer in range(self.L):
                # the step's inputs of every layer are staged before the mask kernel, so from
                # layer 1 on the kernel launched just before (the previous layer's decode) writes
                # none of them: SWA_DECODE_INPUTS_READY
                swa.decode(self.cmp, layer, qb[layer], kb[layer], vb[layer], self.mask,
                           self.scale, self.ob[i][layer], self.ws, stream=s, inputs_ready=layer > 0)
        torch.cuda.current_stream(self.dev).wait_stream(s)
        return g

    def _replay(self, i):
        if self.graphs[i] is None:
            self.graphs[i] = self._capture(i)
            # the capture advanced the host mirror once; this replay advances the device
            self.graphs[i].replay()
        else:
            self.graphs[i].replay()
            self.cmp.advance(1)

    def make_events(self):
        return {"start": ev(), "inputs": ev(), "prefill": ev(), "decode_start": ev(), "end": ev(),
                "step_s": [ev() for _ in range(self.T)], "step_e": [ev() for _ in range(self.T)]}

    def run(self, e):
        swa = self.swa
        e["start"].record()
        if self.e2e:
            self.d_pq.copy_(self.pq, non_blocking=True)
            self.d_pk.copy_(self.pk, non_blocking=True)
            self.d_pv.copy_(self.pv, non_blocking=True)
        e["inputs"].record()
        self.pre.bind()
        self.cmp.bind()
        for layer in range(self.L):
            swa.prefill(self.pre, layer, swa.MODE_CAUSAL, self.d_pq[layer], self.d_pk[layer], self.d_pv[layer],
                        self.meta, self.scale, self.prefill_out)
        e["prefill"].record()
        swa.compact(self.pre, self.cmp)
        e["decode_start"].record()
        if self.nbuf == 2:
            self._decode_steps_overlapped(e)
        else:
            for t in range(self.T):
                if self.cmp.needs_roll():
                    swa.roll(self.cmp)
                self.stage[0].copy_(self.dec[t], non_blocking=True)
                if self.l2_flush is not None:
                    self.l2_flush.fill_(t & 127)
                e["step_s"][t].record()
                self._replay(0)
                e["step_e"][t].record()
                self.outs[t].copy_(self.ob[0], non_blocking=True)
        e["end"].record()

    def _decode_steps_overlapped(self, e):
        """The decode steps: step t uses staging set t % 2.  On the copy stream the copy of step
        t + 1's inputs into its set (after step t - 1, the set's last reader) and the copy of step
        t's outputs out of its set run while the compute stream replays the next graph; end to
        end these are the host uploads and downloads."""
        swa, cs = self.swa, self.copy_stream
        main = torch.cuda.current_stream(self.dev)
        up = [torch.cuda.Event() for _ in range(2)]    # inputs of the set landed
        done = [torch.cuda.Event() for _ in range(2)]  # the set's graph finished
        down = [torch.cuda.Event() for _ in range(2)]  # the set's outputs left
        cs.wait_stream(main)
        with torch.cuda.stream(cs):
            self.stage[0].copy_(self.dec[0], non_blocking=True)
            up[0].record(cs)
        for t in range(self.T):
            i = t % 2
            if t + 1 < self.T:
                with torch.cuda.stream(cs):
                    if t >= 1:
                        cs.wait_event(done[1 - i])
                    self.stage[1 - i].copy_(self.dec[t + 1], non_blocking=True)
                    up[1 - i].record(cs)
            if self.cmp.needs_roll():
                swa.roll(self.cmp)
            main.wait_event(up[i])
            if t >= 2:
                main.wait_event(down[i])
            e["step_s"][t].record()
            self._replay(i)
            e["step_e"][t].record()
            done[i].record(main)
            with torch.cuda.stream(cs):
                cs.wait_event(done[i])
                self.outs[t].copy_(self.ob[i], non_blocking=True)
                down[i].record(cs)
        main.wait_stream(cs)


# ----------------------------------------------------------------------------- our arm
def run_ours(args):
    ws, rank, local = dist_env()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    from sliding_window_gqa_swa_gb300 import build
    build.build()
    from sliding_window_gqa_swa_gb300 import swa, synth
    peaks, peaks_src = load_peaks()

    case = synth.workload2(layers=args.layers, steps=args.decode_steps)
    job = SingleStreamJob(swa, case, dev)
    L, T = job.L, job.T

    def barrier():
        if ws > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        job.run(job.make_events())
    barrier()
    evs = [job.make_events() for _ in range(args.steps)]
    with ClockSampler(local) as clocks:
        barrier()
        t0, t1 = ev(), ev()
        t0.record()
        for k in range(args.steps):
            job.run(evs[k])
        t1.record()
        barrier()
    decode_ms = sum(e["decode_start"].elapsed_time(e["end"]) for e in evs)
    prefill_ms = sum(e["inputs"].elapsed_time(e["prefill"]) for e in evs)
    graph_ms = sum(sum(e["step_s"][t].elapsed_time(e["step_e"][t]) for t in range(T)) for e in evs)
    # the slowest replica sets every reported time
    total_ms, decode_ms, prefill_ms, graph_ms = max_over_ranks(
        [t0.elapsed_time(t1), decode_ms, prefill_ms, graph_ms], dev)
    us_per_layer = decode_ms * 1e3 / (args.steps * T * L)
    launch_us = graph_ms * 1e3 / (args.steps * T * L)  # the shared mask's share is included
    # algorithmic bytes of one decode launch: the W admitted K and V rows of both kv heads,
    # plus q, k_new, v_new, out and the mask row
    dec_bytes = (job.W * job.B * job.Hkv * job.D * 2 * 2
                 + job.B * (2 * job.Hq + 2 * job.Hkv) * job.D * 2 + job.B * job.cmp.rows)
    achieved_gbs = dec_bytes / (launch_us * 1e-6) / 1e9
    traffic, traffic_src = profiled_traffic()
    pre_flops = 4.0 * job.D * job.Hq * causal_pairs(job.S, job.W) * job.B * L
    pre_tflops = pre_flops / (prefill_ms / args.steps * 1e-3) / 1e12
    launches = job.launches * args.steps
    warm_step_med = statistics.median(
        e["step_s"][t].elapsed_time(e["step_e"][t]) for e in evs for t in range(T))
    del job
    torch.cuda.empty_cache()

    e2e = None
    if not args.no_e2e:
        ejob = SingleStreamJob(swa, case, dev, e2e=True)
        for _ in range(max(1, min(args.warmup, 2))):
            ejob.run(ejob.make_events())
        torch.cuda.synchronize()
        eev = [ejob.make_events() for _ in range(args.steps)]
        for k in range(args.steps):
            ejob.run(eev[k])
        torch.cuda.synchronize()
        e_dec = sum(e["decode_start"].elapsed_time(e["end"]) for e in eev)
        e2e = {"value": round(e_dec * 1e3 / (args.steps * T * L), 4), "unit": "us/layer",
               "h2d_bytes_per_step": int(ejob.h2d_bytes), "d2h_bytes_per_step": int(ejob.d2h_bytes),
               "job_ms": round(sum(e["start"].elapsed_time(e["end"]) for e in eev) / args.steps, 3),
               "note": "per decode step: H2D of that step's q/k/v for 26 layers from pinned memory and D2H of "
                       "its outputs, inside the decode phase, on a copy stream overlapping the neighbouring "
                       "steps' graphs; the prompt upload is inside job_ms"}
        del ejob
        torch.cuda.empty_cache()

    secondary = {} if args.no_secondary else run_secondary(swa, synth, dev, peaks, args.training_docs)
    if not args.no_secondary:
        # the same job through the modular ring cache (W rows, no roll)
        rjob = SingleStreamJob(swa, case, dev, ring=True)
        for _ in range(max(1, min(args.warmup, 2))):
            rjob.run(rjob.make_events())
        torch.cuda.synchronize()
        rev = [rjob.make_events() for _ in range(args.steps)]
        for k in range(args.steps):
            rjob.run(rev[k])
        torch.cuda.synchronize()
        r_dec = sum(e["decode_start"].elapsed_time(e["end"]) for e in rev)
        r_graph = sum(sum(e["step_s"][t].elapsed_time(e["step_e"][t]) for t in range(T)) for e in rev)
        secondary["single_stream_ring"] = {
            "workload": "the single-stream job with a modular ring cache of W rows (position p in row p % W, "
                        "no roll) instead of the anchored W + 64 buffer",
            "us_per_layer": round(r_dec * 1e3 / (args.steps * T * L), 4),
            "decode_launch_us": round(r_graph * 1e3 / (args.steps * T * L), 4),
            "anchored_us_per_layer": round(us_per_layer, 4)}
        del rjob
        torch.cuda.empty_cache()
        # the same job with L2 flushed before every step: a 2 x L2 scratch write evicts the
        # compact cache, q/k/v and the state, so each step's graph starts from HBM
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        flush = torch.empty(2 * l2, dtype=torch.uint8, device=dev)
        cjob = SingleStreamJob(swa, case, dev, l2_flush=flush)
        for _ in range(max(1, min(args.warmup, 2))):
            cjob.run(cjob.make_events())
        torch.cuda.synchronize()
        cev = [cjob.make_events() for _ in range(args.steps)]
        for k in range(args.steps):
            cjob.run(cev[k])
        torch.cuda.synchronize()
        cold_med = statistics.median(
            e["step_s"][t].elapsed_time(e["step_e"][t]) for e in cev for t in range(T))
        secondary["single_stream_l2_cold"] = {
            "workload": "the single-stream job with L2 flushed (a write of 2 x L2 bytes) before every decode step",
            "us_per_layer": round(cold_med * 1e3 / L, 4),
            "warm_us_per_layer": round(warm_step_med * 1e3 / L, 4),
            "timing": "median over all steps of the step graph (shared mask + one decode per layer) / layers; "
                      "the flush runs before the step's start event",
            "flush_bytes": int(2 * l2)}
        del cjob, flush
        torch.cuda.empty_cache()
    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(case, args.cpu_seconds)
    if rank != 0:
        return
    line = {
        "metric": METRIC,
        "value": round(us_per_layer, 4),
        "unit": "us/layer",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(total_ms / args.steps, 3),
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": round(us_per_layer / SPYRE_RUNTIME_MASK_US, 5),
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16, workload seed 1002)",
        "config": {"workload": WORKLOAD, "layers": L, "decode_steps": T, "prompt_len": case.prompt_len,
                   "l2": "inputs larger than L2: each step streams 1.3 GB of prompt Q/K/V and prefill cache; the "
                         "58 MB compact cache stays L2-resident within a step, as in serving",
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
                   "decode_chaining": "one step graph: the shared mask, then the 26 layers' decodes chained by "
                                      "programmatic launch; the step's inputs of all layers are staged before "
                                      "the mask, so layers 1-25 use SWA_DECODE_INPUTS_READY",
                   "staging": "two staging sets, steps alternate: a copy stream stages step t+1's inputs and "
                              "stores step t-1's outputs while step t's graph runs (inside the timed region)"},
        "decode_us_per_layer": round(us_per_layer, 4),
        "decode_launch_us": round(launch_us, 4),
        "prefill_ms_per_job": round(prefill_ms / args.steps, 3),
        "prefill_tflops": round(pre_tflops, 2),
        "roofline": {"bound": "hbm", "kernel": DOMINANT_KERNEL, "achieved": round(achieved_gbs, 1),
                     "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": round(achieved_gbs / peaks["hbm_gbs"], 4),
                     "traffic": traffic, "traffic_source": traffic_src, "peak_source": peaks_src,
                     "per_launch_bytes": int(dec_bytes),
                     "note": "launch duration = per-step graph time (shared mask + 26 decodes) / 26; the working "
                             "set is L2-resident within a step, so the kernel is latency-bound"},
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clocks.summary(),
        "cpu_baseline": cpu,
        "secondary": secondary,
        "context": {"spyre_runtime_mask_swa_us": SPYRE_RUNTIME_MASK_US},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- secondary workloads
def oracle_rate(fn, seconds: float, max_calls: int = 100000):
    """Seconds per call of ``fn`` (the fp64 oracle on one sample unit), timed over about ``seconds``."""
    t0 = time.perf_counter()
    n = 0
    while n < max_calls and (n == 0 or time.perf_counter() - t0 < seconds):
        fn(n)
        n += 1
    return (time.perf_counter() - t0) / n, n


def run_secondary(swa, synth, dev, peaks, training_docs=4, oracle_seconds=4.0):
    out = {}
    for name, fn in (("batched_decode", bench_batched_decode), ("chunked_vlm_prefill", bench_vlm_prefill),
                     ("packed_prefill_d512", bench_packed),
                     ("packed_training_d512", lambda *a: bench_training(*a, docs=training_docs))):
        try:
            out[name] = fn(swa, synth, dev, peaks)
        except Exception as e:  # reported in the line, never hidden
            out[name] = {"error": repr(e)}
        torch.cuda.empty_cache()
    if oracle_seconds > 0:
        for name, fn in (("batched_decode", oracle_batched_decode), ("chunked_vlm_prefill", oracle_vlm_prefill),
                         ("packed_prefill_d512", oracle_packed)):
            if name in out and "error" not in out[name]:
                try:
                    out[name]["cpu_baseline"] = fn(synth, oracle_seconds)
                except Exception as e:
                    out[name]["cpu_baseline"] = {"error": repr(e)}
    return out


def oracle_batched_decode(synth, seconds):
    """The fp64 oracle on (sequence, step) queries of the batched decode workload, scaled to one step of
    all 64 sequences (every query head of a sequence per call)."""
    from oracle import reference
    c = synth.workload3(steps=256)
    B, W, D, S = c.batch, c.window, c.head_dim, c.prompt_len

    def one(n):
        b, t = n % B, (n // B) % c.steps
        reference.decode_full(c.prompt_k[0][b:b + 1], c.prompt_v[0][b:b + 1], c.dec_q[:, 0, b:b + 1],
                              c.dec_k[:, 0, b:b + 1], c.dec_v[:, 0, b:b + 1], S, W, D ** -0.5,
                              c.valid_start[b:b + 1].numpy(), steps=[t])
    sec, n = oracle_rate(one, seconds)
    th = host_threads()
    return {"value": round(sec * B * 1e6, 1), "unit": "us/step", "cores": th["cores"],
            "blas_threads": th.get("blas_threads"), "kind": "oracle",
            "sample": f"{n} (sequence, step) decode queries (16 query heads each), scaled by 64 sequences"}


def oracle_vlm_prefill(synth, seconds):
    """The fp64 oracle on query rows of the chunked VLM prefill (sequence 1, with the image blocks),
    scaled to all B x S rows."""
    from oracle import reference
    c = synth.workload4()
    B, S, W, D = c.batch, c.seq_len, c.window, c.head_dim
    rows = list(range(1024, S, 97))

    def one(n):
        r = rows[n % len(rows)]
        reference.prefill_rows(c.q, c.k, c.v, W, D ** -0.5, 1, [r], c.valid_start.numpy(), c.img_id.numpy())
    sec, n = oracle_rate(one, seconds)
    th = host_threads()
    pairs = sum(admitted_pairs(S, W, int(c.valid_start[b]), c.img_id[b].numpy()) for b in range(B))
    total_s = sec * B * S
    return {"value": round(total_s * 1e3, 1), "unit": "ms", "tflops": round(4.0 * D * c.q_heads * pairs / total_s / 1e12, 6),
            "cores": th["cores"], "blas_threads": th.get("blas_threads"), "kind": "oracle",
            "sample": f"{n} query rows (8 heads each) of sequence 1, scaled to {B} x {S} rows"}


def oracle_packed(synth, seconds):
    """The fp64 oracle on query rows of the packed documents (D = 512), scaled to all 16384 rows."""
    from oracle import reference
    c = synth.workload5()
    T, W, D = int(c.cu_seqlens[-1]), c.window, c.head_dim
    cu = c.cu_seqlens.numpy()
    rows = list(range(37, T, 211))

    def one(n):
        r = rows[n % len(rows)]
        reference.varlen_rows(c.q, c.k, c.v, cu, W, D ** -0.5, [r])
    sec, n = oracle_rate(one, seconds)
    th = host_threads()
    total_s = sec * T
    pairs = 4 * causal_pairs(4096, W)
    return {"value": round(total_s * 1e3, 1), "unit": "ms", "tflops": round(4.0 * D * c.q_heads * pairs / total_s / 1e12, 6),
            "cores": th["cores"], "blas_threads": th.get("blas_threads"), "kind": "oracle",
            "sample": f"{n} query rows (16 heads each), scaled to {T} rows"}


def bench_batched_decode(swa, synth, dev, peaks, steps=256, reps=3):
    """Batched decode phase: per step one captured graph (runtime mask + decode),
    replayed back to back; rolls every 64 steps; best of ``reps`` phases."""
    c = synth.workload3(steps=steps)
    S, W, D, B, Hq, Hkv = c.prompt_len, c.window, c.head_dim, c.batch, c.q_heads, c.kv_heads
    cache = swa.Cache(swa.CACHE_COMPACT, 1, B, Hkv, D, W, S, c.valid_start.to(dev))
    k0 = c.prompt_k[0].transpose(1, 2).contiguous().to(dev)
    v0 = c.prompt_v[0].transpose(1, 2).contiguous().to(dev)
    mask = torch.empty(B, cache.rows, dtype=torch.uint8, device=dev)
    wsp = swa.decode_workspace(cache, Hq)
    dq, dk, dv = c.dec_q[:, 0].to(dev), c.dec_k[:, 0].to(dev), c.dec_v[:, 0].to(dev)
    qb = torch.empty(B, Hq, D, dtype=torch.bfloat16, device=dev)
    kb = torch.empty(B, Hkv, D, dtype=torch.bfloat16, device=dev)
    vb = torch.empty_like(kb)
    o = torch.empty(B, Hq, D, dtype=torch.bfloat16, device=dev)
    lens = S - c.valid_start.numpy()
    g_mask = g_dec = None
    best_phase = best_dec = None
    for rep in range(reps + 1):
        cache.bind()                      # zero-fill and initial state
        cache.k[0, :, :, :W].copy_(k0)    # rows [0, W) hold positions [S - W, S)
        cache.v[0, :, :, :W].copy_(v0)
        p0, p1 = ev(), ev()
        evs = []
        p0.record()
        for t in range(steps):
            if cache.needs_roll():
                swa.roll(cache)
            qb.copy_(dq[t], non_blocking=True)
            kb.copy_(dk[t], non_blocking=True)
            vb.copy_(dv[t], non_blocking=True)
            if g_mask is None:
                s_ = torch.cuda.Stream(dev)
                s_.wait_stream(torch.cuda.current_stream(dev))
                g_mask, g_dec = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
                with torch.cuda.graph(g_mask, stream=s_):
                    swa.build_decode_mask(cache, mask, stream=s_)
                with torch.cuda.graph(g_dec, stream=s_):
                    swa.decode(cache, 0, qb, kb, vb, mask, D ** -0.5, o, wsp, stream=s_)
                torch.cuda.current_stream(dev).wait_stream(s_)
                g_mask.replay()  # the capture advanced the host mirror once
            else:
                g_mask.replay()
                cache.advance(1)
            e0, e1 = ev(), ev()
            e0.record()
            g_dec.replay()
            e1.record()
            evs.append((e0, e1))
        p1.record()
        torch.cuda.synchronize()
        if rep > 0:  # the first phase warms up (and captures)
            ph = p0.elapsed_time(p1)
            dec = sum(a.elapsed_time(b) for a, b in evs)
            best_phase = ph if best_phase is None else min(best_phase, ph)
            best_dec = dec if best_dec is None else min(best_dec, dec)
    cache.check()
    dec_bytes = sum(int(np.minimum(lens + t + 1, W).sum()) * Hkv * D * 2 * 2 + B * (2 * Hq + 2 * Hkv) * D * 2
                    + B * cache.rows for t in range(steps))
    rolls = (steps - 1) // 64
    roll_bytes = rolls * 2 * 2 * B * Hkv * W * D * 2          # K and V, read + write
    mask_bytes = steps * B * cache.rows
    dec_gbs = dec_bytes / (best_dec * 1e-3) / 1e9
    phase_gbs = (dec_bytes + roll_bytes + mask_bytes) / (best_phase * 1e-3) / 1e9
    return {"workload": "batched decode B=64 Hq=16 Hkv=8 D=256 W=1024, lengths U{16..8192}, 256 steps",
            "us_per_step": round(best_dec * 1e3 / steps, 2), "hbm_gbs": round(dec_gbs, 1),
            "hbm_frac": round(dec_gbs / peaks["hbm_gbs"], 4), "mb_per_step_mean": round(dec_bytes / steps / 1e6, 1),
            "phase_us_per_step": round(best_phase * 1e3 / steps, 2), "phase_gbs": round(phase_gbs, 1),
            "timing": f"decode kernel: events around each step's decode graph replay, summed over 256 steps; "
                      f"phase: the whole 256-step loop (mask, input copies, 3 rolls); best of {reps}",
            "l2": "per-step K/V (~500 MB) larger than L2"}


def bench_vlm_prefill(swa, synth, dev, peaks):
    c = synth.workload4()
    B, S, Hq, Hkv, D, W, C = c.batch, c.seq_len, c.q_heads, c.kv_heads, c.head_dim, c.window, c.chunk
    vs, img = c.valid_start.to(dev), c.img_id.to(dev)
    q, k, v = c.q.to(dev), c.k.to(dev), c.v.to(dev)
    cache = swa.Cache(swa.CACHE_PREFILL, 1, B, Hkv, D, W, S, vs)
    o = torch.empty(B, C, Hq, D, dtype=torch.bfloat16, device=dev)
    chunks = []
    for c0 in range(0, S, C):
        meta = swa.Meta(B, S, c0, C, W, valid_start=vs, img_id=img)
        chunks.append((meta, q[:, c0:c0 + C].contiguous(), k[:, c0:c0 + C].contiguous(),
                       v[:, c0:c0 + C].contiguous()))

    def run():
        e0, e1 = ev(), ev()
        e0.record()
        for meta, qc, kc, vc in chunks:
            swa.build_prefill_plan(meta, cache)
            swa.prefill(cache, 0, swa.MODE_GENERIC, qc, kc, vc, meta, D ** -0.5, o)
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)

    run()
    ms = min(run() for _ in range(3))
    pairs = sum(admitted_pairs(S, W, int(c.valid_start[b]), c.img_id[b].numpy()) for b in range(B))
    tf = 4.0 * D * Hq * pairs / (ms * 1e-3) / 1e12
    executed = sum(executed_tile_pairs(meta.plan, B, C) for meta, *_ in chunks)
    return {"workload": "chunked prefill B=4 S=8192 (4 x 2048) Hq=8 Hkv=4 D=256 W=1024, image blocks",
            "ms": round(ms, 3), "tflops": round(tf, 2), "tensor_frac": round(tf / peaks["bf16_tflops"], 4),
            "pairs_per_head": pairs, "executed_pairs_per_head": executed,
            "useful_frac": round(pairs / executed, 4) if executed else None,
            "tiles": "128 query rows x 128 keys per executed tile (head size 256 kernel); a tile's key range "
                     "is the plan's per-query-tile range",
            "includes": "plan build + K/V write + attention, 4 chunks"}


def executed_tile_pairs(plan, batch, chunk_len, bm=128, bn=128):
    """(query, key) pairs the head-size-256 prefill computes for one chunk and head: for every
    128-row query tile, the 128-key tiles spanning the plan's key range [klo, khi).  The plan
    buffer is header (256 B) | row_lo [B, C] | row_hi [B, C] | tile_klo [B, T] | tile_khi [B, T],
    int32, each part 256-byte aligned (T = ceil(C / 128))."""
    def a256(x):
        return (x + 255) & ~255
    nqt = (chunk_len + bm - 1) // bm
    raw = plan.cpu().numpy()
    rows = a256(batch * chunk_len * 4)
    off_tlo = 256 + 2 * rows
    off_thi = off_tlo + a256(batch * nqt * 4)
    klo = raw[off_tlo:off_tlo + batch * nqt * 4].view(np.int32).astype(np.int64)
    khi = raw[off_thi:off_thi + batch * nqt * 4].view(np.int32).astype(np.int64)
    n = np.where(khi > klo, (khi - 1) // bn - klo // bn + 1, 0)
    return int(n.sum()) * bm * bn


def bench_packed(swa, synth, dev, peaks):
    c = synth.workload5()
    T = int(c.cu_seqlens[-1])
    Hq, D, W = c.q_heads, c.head_dim, c.window
    meta = swa.Meta(1, T, 0, T, W, cu_seqlens=c.cu_seqlens.to(dev))
    q, k, v = c.q.to(dev), c.k.to(dev), c.v.to(dev)
    o = torch.empty(T, Hq, D, dtype=torch.bfloat16, device=dev)

    def run():
        e0, e1 = ev(), ev()
        e0.record()
        swa.build_prefill_plan(meta)
        swa.prefill(None, 0, swa.MODE_GENERIC, q, k, v, meta, D ** -0.5, o)
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)

    run()
    ms = min(run() for _ in range(3))
    pairs = 4 * causal_pairs(4096, W)
    tf = 4.0 * D * Hq * pairs / (ms * 1e-3) / 1e12
    return {"workload": "packed documents 4 x 4096, Hq=16 Hkv=8 D=512 W=4096 (document-causal)",
            "ms": round(ms, 3), "tflops": round(tf, 2), "tensor_frac": round(tf / peaks["bf16_tflops"], 4)}


# Forward + backward of one packed 16K-token batch (4 x 4096) at head size 512, 16/8
# heads, as the Fast-LLM page times it on H100 (sdpa-nested, bf16, fwd+bwd wall)
FASTLLM_H100_FWD_BWD_MS = 88.0


def bench_training(swa, synth, dev, peaks, docs=4):
    """Training step of the packed workload: plan + forward (out, lse) + backward
    (dq, dk, dv for an N(0,1) upstream gradient); best of 3 after one warm-up.
    ``docs`` < 4 packs fewer 4096-token documents (a smaller case for profiling)."""
    c = synth.workload5() if docs == 4 else synth.varlen_case(
        synth.SEED_BASE + 5, doc_lens=[4096] * docs, q_heads=16, kv_heads=8, head_dim=512, window=4096)
    T = int(c.cu_seqlens[-1])
    Hq, D, W = c.q_heads, c.head_dim, c.window
    meta = swa.Meta(1, T, 0, T, W, cu_seqlens=c.cu_seqlens.to(dev))
    q, k, v = c.q.to(dev), c.k.to(dev), c.v.to(dev)
    g = synth.upstream_grad(synth.SEED_BASE + 5, c.q.shape).to(dev)
    o = torch.empty(T, Hq, D, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(T, Hq, dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    swa.build_prefill_plan(meta)
    ws = swa.backward_workspace(Hq, meta, device=dev)

    def run():
        e0, e1, e2 = ev(), ev(), ev()
        e0.record()
        swa.build_prefill_plan(meta, out=meta.plan)
        swa.prefill(None, 0, swa.MODE_GENERIC, q, k, v, meta, D ** -0.5, o, lse)
        e1.record()
        swa.prefill_backward(q, k, v, o, g, lse, meta, D ** -0.5, dq, dk, dv, ws)
        e2.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1), e1.elapsed_time(e2)

    run()
    fwd_ms, bwd_ms = min((run() for _ in range(3)), key=lambda t: t[0] + t[1])
    pairs = docs * causal_pairs(4096, W)
    fwd_flop, bwd_flop = 4.0 * D * Hq * pairs, 10.0 * D * Hq * pairs
    tf = (fwd_flop + bwd_flop) / ((fwd_ms + bwd_ms) * 1e-3) / 1e12
    bwd_tf = bwd_flop / (bwd_ms * 1e-3) / 1e12
    return {"workload": f"training step of packed documents {docs} x 4096, Hq=16 Hkv=8 D=512 W=4096: forward + "
                        "backward",
            "fwd_ms": round(fwd_ms, 3), "bwd_ms": round(bwd_ms, 3), "fwd_bwd_ms": round(fwd_ms + bwd_ms, 3),
            "tflops": round(tf, 2), "bwd_tflops": round(bwd_tf, 2), "tensor_frac": round(tf / peaks["bf16_tflops"], 4),
            "flop": "forward 4 D Hq pairs, backward 10 D Hq pairs (QK^T, dO V^T, dV, dK, dQ)",
            "workspace_gb": round(ws.numel() / 1e9, 2),
            "context_h100_sdpa_nested_fwd_bwd_ms": FASTLLM_H100_FWD_BWD_MS}


# ----------------------------------------------------------------------------- CPU oracle
def _oracle_decode_queries(case, n_queries, first=0):
    """Run the fp64 oracle on ``n_queries`` (step, layer) decode queries."""
    from oracle import reference
    W = case.window
    for i in range(first, first + n_queries):
        layer = i % case.layers
        t = (i // case.layers) % case.steps
        # the last W prompt rows are all the window ever admits (same oracle result)
        reference.decode_full(case.prompt_k[layer, :, -W:], case.prompt_v[layer, :, -W:], case.dec_q[:, layer],
                              case.dec_k[:, layer], case.dec_v[:, layer], case.prompt_len, W,
                              case.head_dim ** -0.5, None, steps=[t])


def cpu_baseline(case, seconds: float):
    """The fp64 oracle, as it stands, on a bounded sample of the decode workload."""
    t0 = time.perf_counter()
    n = 0
    while time.perf_counter() - t0 < seconds and n < case.steps * case.layers:
        _oracle_decode_queries(case, 26, n)
        n += 26
    el = time.perf_counter() - t0
    th = host_threads()
    return {"value": round(el * 1e6 / n, 1), "unit": "us/layer", "cores": th["cores"],
            "blas_threads": th.get("blas_threads"), "kind": "oracle",
            "sample": f"{n} (step, layer) decode queries of the single-stream workload, fp64 NumPy"}


def run_reference(args):
    ws, rank, local = dist_env()
    if rank != 0:
        return
    from sliding_window_gqa_swa_gb300 import synth
    case = synth.workload2(layers=args.layers, steps=args.decode_steps, with_prompt_q=False)
    per = max(1, args.ref_queries)
    for k in range(args.warmup):
        _oracle_decode_queries(case, per, k * per)
    t0 = time.perf_counter()
    for k in range(args.steps):
        _oracle_decode_queries(case, per, (args.warmup + k) * per)
    tot = time.perf_counter() - t0
    us = tot * 1e6 / (per * args.steps)
    cores = host_threads()["cores"]
    line = {"impl": "reference", "metric": METRIC, "value": round(us, 1), "unit": "us/layer", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(tot * 1e3 / args.steps, 3),
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,1) bf16, workload seed 1002)",
            "config": {"workload": WORKLOAD, "layers": case.layers, "decode_steps": case.steps},
            "cpu_baseline": {"value": round(us, 1), "unit": "us/layer", "cores": cores, "kind": "oracle",
                             "sample": f"{per} (step, layer) decode queries per bench step"},
            "e2e": {"value": round(us, 1), "unit": "us/layer", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--layers", type=int, default=26)
    ap.add_argument("--decode-steps", type=int, default=512)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--ref-queries", type=int, default=104)
    ap.add_argument("--training-docs", type=int, default=4, choices=[1, 2, 3, 4],
                    help="4096-token documents in the training-step secondary line (4 = the full workload)")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
