#!/usr/bin/env python3
"""Benchmark of one paged-KV decode step on GB300.

A step is the whole hot path over one batch: paged_kv_append of the step's
new K/V (32 tokens) followed by paged_attention (split over a persistent grid,
merged in-kernel) on the continuous-batch decode workload: 32 sequences,
32 query / 8 KV heads, head_dim 128, block size 16, context lengths uniform in
[256, 2048], bf16 K/V ~ N(0, 1), block tables from a shuffled 5,000-block pool.

Prints ONE JSON line (rank 0).  `value` is KV GB/s of the whole step
(algorithmic KV bytes / device time of append + attention), inputs resident in
HBM.  By default the timed steps rotate over enough copies of the workload
that no step finds its K/V in L2, and K steps are timed back to back as one
CUDA-event interval behind a queued spin kernel, so the interval holds the
GPU's time and not the host's launch overhead; `--l2 flush` writes a buffer of
twice the L2 size before every step instead (timed per step, the flush
excluded), which also evicts the kernels' code.  The attention kernel's
roofline uses its own device time per launch, taken the same way over K
launches.  `--impl reference` times the CPU oracle on the host cores instead
(a deliberately slow reference).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
For N > 1 launch with torchrun (one rank per GPU); every rank runs its own
replica of the workload (weak scaling, no collective on the data path).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged-attn decode KV GB/s (% of HBM peak) and seq-steps/s at B=32, d=128"
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=2, help="named workload (default: the decode config)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="CPU baseline sample budget")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--graph", action="store_true",
                    help="replay CUDA graphs of the steps instead of launching them through the binding")
    ap.add_argument("--l2", choices=["flush", "rotate"], default="rotate",
                    help="keep timed inputs out of L2: flush it before every step (a write of 2x its size), "
                         "or rotate over enough copies of the workload that the data read by a step is not in L2")
    ap.add_argument("--cascade", action="store_true",
                    help="attend through the shared-prefix cascade (workloads whose sequences share prefix blocks)")
    ap.add_argument("--prefill", nargs="?", const="prefill_b4_q2048_d128", default=None,
                    help="time the paged chunked-prefill step (append of the window + pkv_paged_prefill) on a "
                         "named prefill workload instead: prefill_b4_q2048_d128 (default) or "
                         "chunked_prefill_b8_q512_d128")
    ap.add_argument("--soak-seconds", type=float, default=1.5,
                    help="untimed steps run right before the timed region while clocks are sampled")
    return ap.parse_args()


PREFILL_METRIC = "causal prefill attention TFLOP/s (% of bf16 tensor peak)"
FALLBACK_BF16_TFLOPS = 1900.0


def tensor_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback"


def hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def attn_algorithmic_bytes(w) -> int:
    """Bytes the attention must move once: KV (+ FP8 scales) counting each
    distinct physical block once (blocks shared by several sequences' tables
    are one read), q, out, the block-table entries it reads and the two length
    arrays."""
    nblk = int(((w.context_lens.astype(np.int64) + 15) // 16).sum())
    return w.unique_kv_bytes() + 2 * w.q.nbytes + 4 * nblk + 8 * w.num_seqs


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_decode_14_gb300", "csrc")
    for n in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, n), "rb") as f:
            h.update(n.encode() + f.read())
    return h.hexdigest()[:16]


def load_traffic(workload: str):
    """DRAM bytes per attention launch from a committed ncu capture, if it was
    taken on the current kernel sources (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
        e = d.get(workload)
        if e and e.get("source_hash") == kernel_source_hash():
            return float(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 100 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"clocks_bench_{os.getpid()}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None:
            return None
        sms, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        try:
            for ln in open(self.path):
                parts = [x.strip() for x in ln.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sms.append(float(parts[1]))
                    mx = float(parts[2])
                except ValueError:
                    continue
                for nm, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(nm)
        except Exception:
            return None
        if not sms:
            return None
        return {"sm_mhz": float(np.median(sms)), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sms)}


class OracleStepper:
    """The CPU oracle, as it stands, on the host cores.  One sample step =
    the oracle's append of the step's new tokens plus its attention for a
    slice of the batch's sequences (`seqs_per_step` of them, rotating), so a
    step stays bounded; the KV bytes of the slice give the throughput."""

    def __init__(self, w, seqs_per_step: int):
        import oracle
        self.oracle = oracle
        self.w = w
        self.kc, self.vc = oracle.build_cache(w, with_step=False)
        self.kd = oracle.KV_FP8 if w.kv_dtype == "fp8" else oracle.KV_BF16
        self.threads = os.cpu_count() or 1
        self.spp = max(1, min(seqs_per_step, w.num_seqs))
        self.qoff = np.concatenate([[0], np.cumsum(w.q_lens)]).astype(np.int64)
        self.i = 0

    def step(self):
        """Returns (KV bytes processed, seconds)."""
        w, o = self.w, self.oracle
        b0 = (self.i * self.spp) % w.num_seqs
        bs = [(b0 + j) % w.num_seqs for j in range(self.spp)]
        self.i += 1
        rows = np.concatenate([np.arange(self.qoff[b], self.qoff[b + 1]) for b in bs])
        L = w.context_lens[bs]
        t0 = time.perf_counter()
        o.paged_kv_append(self.kd, self.kc, self.vc, w.k_scales, w.v_scales, w.num_blocks, w.num_kv_heads,
                          w.head_dim, w.k_new[rows], w.v_new[rows], w.slots[rows])
        o.paged_attention(self.kd, self.kc, self.vc, w.k_scales, w.v_scales, w.num_blocks, w.num_kv_heads,
                          w.head_dim, w.q[rows], w.num_q_heads, w.block_tables[bs], L, w.q_lens[bs], w.scale,
                          self.threads)
        el = time.perf_counter() - t0
        kvb = int(L.astype(np.int64).sum()) * w.num_kv_heads * w.head_dim * 2 * w.elem_bytes
        return kvb, el


def cpu_baseline(w, seconds: float, seqs_per_step: int = 8):
    """Oracle throughput over ~`seconds` of sample steps:
    (GB/s, threads, steps, s, sequences per step)."""
    st = OracleStepper(w, seqs_per_step)
    tot_b, tot_t, n = 0, 0.0, 0
    while tot_t < seconds:
        b, t = st.step()
        tot_b += b
        tot_t += t
        n += 1
    return tot_b / tot_t / 1e9, st.threads, n, tot_t, st.spp


class PrefillOracleSample:
    """The CPU oracle on a bounded slice of a prefill workload: for one
    sequence at a time (rotating), its last `rows` queries against the whole
    resident context (the most expensive rows).  FLOPs as causal_flops counts
    them for those rows."""

    def __init__(self, w, rows: int = 64):
        import oracle
        self.oracle, self.w = oracle, w
        self.kc, self.vc = oracle.build_cache(w)
        self.qoff = np.concatenate([[0], np.cumsum(w.q_lens)]).astype(np.int64)
        # (the oracle spreads (sequence, kv-head) units over its threads: one sequence has Hkv of them)
        self.threads = min(os.cpu_count() or 1, w.num_kv_heads)
        self.rows, self.i = rows, 0

    def step(self):
        w, o = self.w, self.oracle
        b = self.i % w.num_seqs
        self.i += 1
        L, Q = int(w.context_lens[b]), int(w.q_lens[b])
        n = min(self.rows, Q)
        rows = np.arange(self.qoff[b + 1] - n, self.qoff[b + 1])
        t0 = time.perf_counter()
        o.paged_attention(o.KV_BF16, self.kc, self.vc, None, None, w.num_blocks, w.num_kv_heads, w.head_dim,
                          w.q[rows], w.num_q_heads, w.block_tables[b:b + 1], np.array([L], np.int32),
                          np.array([n], np.int32), w.scale, self.threads)
        el = time.perf_counter() - t0
        keys = n * (L - n) + n * (n + 1) // 2
        return 4 * w.head_dim * w.num_q_heads * keys, el


def run_prefill(args):
    """--prefill: one step = the append of every sequence's query window
    (the prompt chunk's K/V) + pkv_paged_prefill over the batch."""
    from paged_kv_decode_14_gb300 import workloads as wl
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.prefill not in wl.PREFILL_WORKLOADS:
        raise SystemExit(f"unknown prefill workload {args.prefill}: {sorted(wl.PREFILL_WORKLOADS)}")
    w = wl.PREFILL_WORKLOADS[args.prefill]()
    flops = wl.causal_flops(w)
    if args.impl == "reference":
        if rank != 0:
            return 0
        st = PrefillOracleSample(w)
        for _ in range(args.warmup):
            st.step()
        tf, tt = 0, 0.0
        for _ in range(args.steps):
            f_, t_ = st.step()
            tf += f_
            tt += t_
        val = tf / tt / 1e12
        line = {"impl": "reference", "metric": PREFILL_METRIC, "value": val, "unit": "TFLOP/s",
                "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": 1e3 * flops / (val * 1e12), "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": workload_config(w),
                "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": st.threads, "kind": "oracle",
                                 "sample": f"each step: the last {st.rows} queries of one sequence (rotating) "
                                           f"against its whole context; ms_per_step scaled to the batch"},
                "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return 0

    import torch
    import torch.distributed as dist
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from paged_kv_decode_14_gb300 import _native as nat
    from paged_kv_decode_14_gb300.runner import DeviceWorkload
    nat.lib()
    stream = torch.cuda.current_stream(dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    kvb = w.unique_kv_bytes()
    n_copies = min(16, max(2, -(-3 * l2 // max(1, kvb))))
    dws = []
    for _ in range(n_copies):
        d = DeviceWorkload(w, device=dev)
        d.prefill()
        dws.append(d)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    def timed(fn, n):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        queue_ahead(torch)
        e0.record(stream)
        for i in range(n):
            fn(i)
        e1.record(stream)
        barrier()
        return e0.elapsed_time(e1) * 1e3 / n

    def run_step(i):
        d = dws[i % n_copies]
        d.append_step()
        d.attend_prefill()

    def run_attn(i):
        dws[i % n_copies].attend_prefill()

    for i in range(max(args.warmup, 1)):
        run_step(i)
    barrier()
    clocks = ClockSampler(local) if not args.no_clocks else None
    if clocks:
        clocks.__enter__()
        t_end = time.perf_counter() + args.soak_seconds
        while time.perf_counter() < t_end:
            for i in range(8):
                run_step(i)
            torch.cuda.synchronize(dev)
    barrier()
    step_us = timed(run_step, args.steps)
    if clocks:
        clocks.__exit__()
    tot_ms = max_over_ranks(step_us * args.steps / 1e3, world, dev)
    value = world * flops * args.steps / (tot_ms / 1e3) / 1e12
    attn_us = timed(run_attn, args.steps)

    pins = [d.pinned_io() for d in dws]
    host_out = torch.empty(dws[0].out.shape, dtype=dws[0].out.dtype).pin_memory()

    def compute_step(i):
        d = dws[i % n_copies]
        d.append_step()
        d.attend_prefill()

    e2e_pipelined(torch, stream, dws, pins, host_out, compute_step, max(args.warmup, 2), barrier)
    e2e_us = e2e_pipelined(torch, stream, dws, pins, host_out, compute_step, args.steps, barrier)
    e2e_tot = max_over_ranks(e2e_us * args.steps / 1e3, world, dev)
    peak, kind = tensor_peak()
    achieved = flops / (attn_us * 1e-6) / 1e12
    line = {"metric": PREFILL_METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": tot_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16 q.k, fp16 p.v", "data": "synthetic",
            "config": {**workload_config(w),
                       "l2": f"inputs rotated over {n_copies} copies ({n_copies * kvb / 1e6:.0f} MB of KV); "
                             f"within a launch every query block of a sequence re-reads its K/V from L2",
                       "launch": "eager, through the binding",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "flops_per_step": flops, "attention_us": attn_us, "append_us": step_us - attn_us,
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                         "frac": achieved / peak, "traffic": load_traffic(w.name),
                         "peak_kind": f"{kind} (cuBLAS bf16 GEMM burst; fp16 runs at the same rate)",
                         "kernel": "paged chunked prefill (tcgen05, two 128-row tiles per CTA)",
                         "algorithmic_flops_per_launch": flops, "avg_launch_us": attn_us,
                         "timing": "back-to-back launches over rotating copies, one event interval, host ahead"},
            "e2e": {"value": world * flops * args.steps / (e2e_tot / 1e3) / 1e12, "unit": "TFLOP/s",
                    "copies": "one upload and one read-back per step on a second stream, pipelined with the kernels",
                    "h2d_bytes_per_step": int(dws[0].io.numel()),
                    "d2h_bytes_per_step": int(dws[0].out.numel() * dws[0].out.element_size()),
                    "ms_per_step": e2e_tot / args.steps},
            "gpu_launches": 2 * args.steps}
    if clocks:
        line["clocks"] = clocks.summary()
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        st = PrefillOracleSample(w)
        tf, tt, n = 0, 0.0, 0
        while tt < args.cpu_seconds:
            f_, t_ = st.step()
            tf += f_
            tt += t_
            n += 1
        line["cpu_baseline"] = {"value": tf / tt / 1e12, "unit": "TFLOP/s", "cores": st.threads, "kind": "oracle",
                                "sample": f"{n} oracle steps in {tt:.1f} s, each the last {st.rows} queries of "
                                          f"one sequence (rotating) against its whole context"}
    errs = [e for d in dws for e in d.errors()]
    if any(errs):
        line["device_errors"] = errs
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    from paged_kv_decode_14_gb300 import workloads as wl
    w = wl.WORKLOADS[args.config]()
    spp = 2
    st = OracleStepper(w, spp)
    for _ in range(args.warmup):
        st.step()
    tot_b, tot_t = 0, 0.0
    for _ in range(args.steps):
        b, t = st.step()
        tot_b += b
        tot_t += t
    val = tot_b / tot_t / 1e9
    # ms for a full batch step at this rate
    ms = 1e3 * w.kv_bytes() / (val * 1e9)
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w),
            "seq_steps_per_s": w.num_seqs / (ms / 1e3),
            "cpu_baseline": {"value": val, "unit": "GB/s", "cores": st.threads, "kind": "oracle",
                             "sample": f"each step: oracle append + attention for {spp} of the {w.num_seqs} "
                                       f"sequences (rotating); ms_per_step scaled to the whole batch"},
            "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def max_over_ranks(value: float, world: int, device=None) -> float:
    """The largest per-rank value (the slowest rank's time) across the job."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput_gbs(bytes_per_step: int, steps: int, max_ms: float, world: int) -> float:
    """Whole-job throughput: every rank moves bytes_per_step per step (weak
    scaling, one replica per GPU), timed by the slowest rank."""
    return world * bytes_per_step * steps / (max_ms / 1e3) / 1e9


def queue_ahead(torch, ms: float = 25.0):
    """Queue a spin kernel of ~`ms` on the current stream before a timed
    region: the host enqueues the timed launches while it runs, so the events
    measure the GPU's time, not the Python launch overhead of the binding (a
    serving loop launches from native code or a CUDA graph)."""
    torch.cuda._sleep(int(ms * 1e-3 * 2.0e9))


def e2e_pipelined(torch, stream, dws, pins, host_out, compute, n, barrier):
    """End-to-end time per step (us) of n steps through the public API, host
    buffers in and out: every step uploads its inputs from pinned host memory
    (one copy) and reads its output back to pinned host memory.  The copies
    run on a second stream, ordered by events, so that step i + 1's upload and
    step i's read-back overlap the steps' kernels, as a serving loop would
    pipeline them; the timed interval ends when the last read-back is done.
    The device copies `dws` rotate, so a copy's buffers are reused only after
    its previous step's kernels have read them and its result has left."""
    cs = torch.cuda.Stream(device=stream.device)
    nb = len(dws)
    ready = [torch.cuda.Event() for _ in range(n)]
    done = [torch.cuda.Event() for _ in range(n)]
    back = [torch.cuda.Event() for _ in range(n)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def upload(i):
        if i >= nb:
            cs.wait_event(done[i - nb])            # the copy's inputs were read by step i - nb
        with torch.cuda.stream(cs):
            dws[i % nb].io.copy_(pins[i % nb], non_blocking=True)
        ready[i].record(cs)

    queue_ahead(torch)
    e0.record(stream)
    cs.wait_event(e0)
    upload(0)
    for i in range(n):
        if i + 1 < n:
            upload(i + 1)
        stream.wait_event(ready[i])
        if i >= nb:
            stream.wait_event(back[i - nb])        # the copy's output of step i - nb has been read back
        compute(i)
        done[i].record(stream)
        cs.wait_event(done[i])
        with torch.cuda.stream(cs):
            host_out.copy_(dws[i % nb].out, non_blocking=True)
        back[i].record(cs)
    stream.wait_event(back[n - 1])
    e1.record(stream)
    barrier()
    return e0.elapsed_time(e1) * 1e3 / n


def run_ours(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    from paged_kv_decode_14_gb300 import _native as nat
    from paged_kv_decode_14_gb300 import workloads as wl
    from paged_kv_decode_14_gb300.runner import DeviceWorkload

    nat.lib()
    w = wl.WORKLOADS[args.config]()
    stream = torch.cuda.current_stream(dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    kvb = w.unique_kv_bytes()            # algorithmic KV bytes of a step (shared blocks once)
    if args.l2 == "rotate":
        # independent copies (own cache, q, tables) until 3x the L2 size is
        # covered, at most 16 (a small workload stays L2-resident: said below)
        n_copies = min(16, max(2, -(-3 * l2 // max(1, kvb))))
        flush = None
    else:
        n_copies = 1
        flush = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)
    dws = []
    for _ in range(n_copies):
        d = DeviceWorkload(w, device=dev)
        d.prefill()
        dws.append(d)
    dw = dws[0]
    if flush is not None:
        l2_note = f"flushed before every timed step ({flush.numel() >> 20} MiB write)"
    elif n_copies * kvb > l2:
        l2_note = (f"inputs rotated over {n_copies} copies ({n_copies * kvb / 1e6:.0f} MB of KV > "
                   f"{l2 / 1e6:.0f} MB L2), no flush")
    else:
        l2_note = (f"inputs rotated over {n_copies} copies ({n_copies * kvb / 1e6:.1f} MB of KV, L2-resident: "
                   f"{l2 / 1e6:.0f} MB L2)")

    # --graph: each copy's step (append + attention) and, for the per-kernel
    # split, its append and its attention alone are captured as CUDA graphs
    # and replayed.  By default steps launch through the binding.
    use_graph = args.graph
    g_step, g_app, g_att = [], [], []
    if args.cascade and not w.info.get("shared_prefix"):
        raise SystemExit("--cascade needs a workload whose sequences share prefix blocks")
    if use_graph:
        for d in dws:
            d.step()                      # first launches (attributes, lazy loads) outside capture
            if args.cascade:
                d.attend_cascade()
        torch.cuda.synchronize(dev)
        cs = torch.cuda.Stream(dev)
        for d in dws:
            att = d.attend_cascade if args.cascade else d.attend
            stp = (lambda d=d, att=att: (d.append_step(), att()))
            for lst, fn in ((g_step, stp), (g_app, d.append_step), (g_att, att)):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=cs):
                    fn()
                lst.append(g)
        torch.cuda.synchronize(dev)

    def attend(d):
        return d.attend_cascade() if args.cascade else d.attend()

    def run_step(i):
        if use_graph:
            g_step[i % n_copies].replay()
        else:
            d = dws[i % n_copies]
            d.append_step()
            attend(d)

    def run_attn(i):
        if use_graph:
            g_att[i % n_copies].replay()
        else:
            attend(dws[i % n_copies])

    def run_app(i):
        if use_graph:
            g_app[i % n_copies].replay()
        else:
            dws[i % n_copies].append_step()

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    def timed(fn, n):
        """Device time of n calls fn(0..n-1), us per call: back to back in one
        event interval (rotate mode), or each after an L2 flush that the events
        exclude (flush mode)."""
        if flush is None:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            queue_ahead(torch)
            e0.record(stream)
            for i in range(n):
                fn(i)
            e1.record(stream)
            barrier()
            return e0.elapsed_time(e1) * 1e3 / n
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for i, (a, b) in enumerate(evs):
            flush.zero_()
            a.record(stream)
            fn(i)
            b.record(stream)
        barrier()
        return 1e3 * float(np.sum([a.elapsed_time(b) for a, b in evs])) / n

    # ---------------- device-resident timing of the whole step
    for i in range(args.warmup):
        run_step(i)
    barrier()
    clocks = ClockSampler(local) if not args.no_clocks else None
    if clocks:
        clocks.__enter__()
        # keep the GPU under the same load while the sampler starts up, right
        # before the timed region (the timed region alone is a few ms)
        t_end = time.perf_counter() + args.soak_seconds
        while time.perf_counter() < t_end:
            for i in range(20):
                run_step(i)
            torch.cuda.synchronize(dev)
    barrier()
    wall0 = time.perf_counter()
    step_us = timed(run_step, args.steps)
    wall = time.perf_counter() - wall0
    if clocks:
        clocks.__exit__()
    tot_ms = max_over_ranks(step_us * args.steps / 1e3, world, dev)
    ms = tot_ms / args.steps
    value = job_throughput_gbs(kvb, args.steps, tot_ms, world)

    # ---------------- per-kernel split (the roofline of the attention kernel)
    attn_us = timed(run_attn, args.steps)
    app_us = timed(run_app, args.steps)

    # ---------------- end to end through the public API, host buffers
    # every step uploads its inputs (one pinned buffer, one copy), runs the
    # step and reads its output back to pinned host memory
    pins = [d.pinned_io() for d in dws]
    host_out = torch.empty(dw.out.shape, dtype=dw.out.dtype).pin_memory()

    def compute_step(i):
        d = dws[i % n_copies]
        d.append_step()
        attend(d)

    e2e_pipelined(torch, stream, dws, pins, host_out, compute_step, max(args.warmup, 2), barrier)
    e2e_us = e2e_pipelined(torch, stream, dws, pins, host_out, compute_step, args.steps, barrier)
    e2e_tot = max_over_ranks(e2e_us * args.steps / 1e3, world, dev)
    e2e_val = job_throughput_gbs(kvb, args.steps, e2e_tot, world)
    hin, hout = int(dw.io.numel()), int(dw.out.numel() * dw.out.element_size())

    # ---------------- roofline of the dominant kernel (attention)
    peak, peak_kind = hbm_peak()
    abytes = attn_algorithmic_bytes(w)
    achieved = abytes / (attn_us * 1e-6) / 1e9
    roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
            "traffic": load_traffic(w.name), "peak_kind": f"{peak_kind} (copy bandwidth)",
            "kernel": "paged attention (persistent split-KV, in-kernel merge)",
            "algorithmic_bytes_per_launch": abytes, "avg_launch_us": attn_us,
            "timing": ("back-to-back launches over rotating copies, one event interval, host ahead"
                       if flush is None else "per launch, L2 flushed before each (flush excluded)")}

    line = {"metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16" if w.kv_dtype == "bf16" else "e4m3", "data": "synthetic",
            "config": {**workload_config(w), "l2": l2_note,
                       **({"attention": "shared-prefix cascade (prefix pass + suffix pass)"} if args.cascade else {}),
                       "launch": "CUDA graph replay per step" if use_graph else "eager, through the binding",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "pct_of_hbm_peak": 100.0 * value / peak,
            "seq_steps_per_s": world * w.num_seqs * args.steps / (tot_ms / 1e3),
            "attention_us": attn_us, "append_us": app_us,
            "roofline": roof,
            "e2e": {"value": e2e_val, "unit": "GB/s", "h2d_bytes_per_step": hin, "d2h_bytes_per_step": hout,
                    "copies": "one upload and one read-back per step on a second stream, pipelined with the kernels",
                    "ms_per_step": e2e_tot / args.steps},
            "gpu_launches": 2 * args.steps,
            "wall_s_timed_region": wall}
    if kvb != w.kv_bytes():
        line["kv_bytes_logical_per_step"] = w.kv_bytes()
        line["value_logical_kv"] = job_throughput_gbs(w.kv_bytes(), args.steps, tot_ms, world)
    if clocks:
        line["clocks"] = clocks.summary()
        if line["clocks"] is not None:
            line["clocks"]["window"] = f"{args.soak_seconds:.1f} s of identical untimed steps + the timed region"

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        gbs, threads, n, el, spp = cpu_baseline(w, args.cpu_seconds)
        line["cpu_baseline"] = {"value": gbs, "unit": "GB/s", "cores": threads, "kind": "oracle",
                                "sample": f"{n} oracle steps in {el:.1f} s, each the append of the step's new "
                                          f"tokens and the attention of {spp} of the {w.num_seqs} sequences "
                                          f"(rotating); GB/s from the KV bytes of those sequences"}
    errs = [e for d in dws for e in d.errors()]
    if any(errs):
        line["device_errors"] = errs
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def lens_summary(w):
    L = np.asarray(w.context_lens)
    return f"min {int(L.min())}, median {int(np.median(L))}, max {int(L.max())}, mean {float(L.mean()):.0f}"


def workload_config(w) -> dict:
    """The workload keys of the JSON line's config (the same in both arms)."""
    return {"workload": w.name, "num_seqs": w.num_seqs, "num_q_heads": w.num_q_heads,
            "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim, "block_size": 16,
            "kv_dtype": w.kv_dtype, "context_lens": lens_summary(w), "q_len_max": int(w.q_lens.max()),
            "pool_blocks": w.num_blocks, "kv_bytes_per_step": w.kv_bytes()}


def main():
    args = parse()
    if args.prefill:
        return run_prefill(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
