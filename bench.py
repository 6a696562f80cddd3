#!/usr/bin/env python
"""Benchmark of block-sparse attention forward (plan + forward per step).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl {gb300,reference}]

One step = the whole hot path over one synthetic problem: bsa_plan (three
kernels) then bsa_forward (one persistent kernel), inputs already resident in
HBM.  Metric: effective TFLOP/s over active tiles = (selected logical blocks x
4*bq*bk*d) / step time.  Default workload: the video-DiT configuration
(B=1, H=24, N=16384, d=128, 128x128 blocks, 3D-local + 5% random mask).

Multi-GPU (torchrun, one rank per GPU): every rank runs an independent replica
of the workload (the path needs no exchange); value = work of all ranks / the
slowest rank's time ("scaling": "weak").

--impl reference times the fp64 CPU oracle (the only reference implementation
this method has) on the host cores, a bounded sample of the same workload per
step.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)


def _cores() -> int:
    return len(os.sched_getaffinity(0))


# The CPU oracle uses NumPy's BLAS: one thread per usable core.
os.environ.setdefault("OPENBLAS_NUM_THREADS", str(_cores()))

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "effective TFLOP/s over active tiles & % of GB300 BF16 tensor peak"

# DRAM bytes (read + write) per launch of the forward kernel, from one
# `ncu --set full` capture of that workload (summaries under profiles/), and the
# hash of the kernel sources it was taken on: a changed kernel reports null.
NCU_TRAFFIC = {
    "video_dit": (302.436096e6 + 82.249472e6, "933485cdae9b26a4"),
}
KERNEL_SOURCES = ("block_sparse_attention_plan_gb300/csrc/bsa_forward.cu",
                  "block_sparse_attention_plan_gb300/csrc/bsa_fwd_common.cuh",
                  "block_sparse_attention_plan_gb300/csrc/bsa_device.cuh")


def _kernel_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def _traffic(workload: str):
    t = NCU_TRAFFIC.get(workload)
    if t is None or t[1] != _kernel_hash():
        return None
    return t[0]
UNIT = "TFLOP/s"
L2_BYTES = 129e6


def _hbm_gbs() -> float:
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"])
    except Exception:
        return 6800.0  # fallback figure


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    except Exception:
        return 1900.0, 1700.0, "fallback"


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clock/throttle samples (wall-clock stamped) for one GPU."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id: str, period_ms: int = 20):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(period_ms), "-i", gpu_id],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm, smax = float(parts[1]), float(parts[2])
            except ValueError:
                continue
            reasons = [n for n, v in zip(self.NAMES, parts[5:9]) if v.lower() == "active"]
            self.samples.append((time.time(), sm, smax, reasons))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        win = [s for s in self.samples if t0 <= s[0] <= t1]
        src = "timed_region"
        if not win and self.samples:
            # region shorter than the sampling period: nearest samples around it
            win = sorted(self.samples, key=lambda s: abs(s[0] - 0.5 * (t0 + t1)))[:3]
            src = "nearest_to_timed_region"
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        reasons = sorted({r for s in win for r in s[3]})
        return {"sm_mhz": statistics.median(s[1] for s in win), "sm_max_mhz": max(s[2] for s in win),
                "reasons": reasons, "samples": len(win), "window": src}


# ---------------------------------------------------------------- CPU oracle timing
def oracle_sample_rate(w, budget_s: float, seed: int = 0, start: int = 0):
    """Time the fp64 oracle on (b, h, q-block) samples taken in a seeded
    permutation order until ``budget_s`` seconds pass.  Returns
    (TFLOP/s over active tiles, seconds, samples done, next start)."""
    from oracle import attention as OA
    B, H, NQB = w.mask.shape[:3]
    cnt = (w.mask != 0).sum(-1).numpy()
    perm = np.random.default_rng(seed).permutation(B * H * NQB)
    flop_blk = 4.0 * w.bq * w.bk * w.d
    t0 = time.perf_counter()
    flop = 0.0
    done = 0
    i = start
    while time.perf_counter() - t0 < budget_s and done < perm.size:
        chunk = []
        for _ in range(8):
            f = int(perm[i % perm.size])
            i += 1
            b, rem = divmod(f, H * NQB)
            h, qb = divmod(rem, NQB)
            chunk.append((b, h, qb))
        OA.sampled_qblocks(w.q, w.k, w.v, w.mask, w.bq, w.bk, chunk)
        flop += sum(flop_blk * cnt[b, h, qb] for b, h, qb in chunk)
        done += len(chunk)
    dt = time.perf_counter() - t0
    return flop / dt / 1e12, dt, done, i


def max_over_ranks(values, device=None):
    """Element-wise maximum of ``values`` over the ranks of the default
    process group (identity without one): the job's time is its slowest
    rank's."""
    import torch
    import torch.distributed as td
    if not (td.is_available() and td.is_initialized()) or td.get_world_size() == 1:
        return [float(x) for x in values]
    t = torch.tensor([float(x) for x in values], dtype=torch.float64, device=device)
    td.all_reduce(t, op=td.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def whole_job_tflops(flop_per_rank: float, ms: float, world: int) -> float:
    """Replicas (weak scaling): every rank runs the same workload, so the
    job does world x the FLOP of one rank in the slowest rank's time."""
    return flop_per_rank * world / (ms * 1e-3) / 1e12


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def run_reference(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return 0
    from block_sparse_attention_plan_gb300 import workloads as W
    w = W.make_workload(args.config)
    per_step = max(0.5, min(10.0, 150.0 / max(1, args.steps + args.warmup)))
    start = 0
    for _ in range(args.warmup):
        _, _, _, start = oracle_sample_rate(w, per_step, start=start)
    rates, secs, n = [], 0.0, 0
    for _ in range(args.steps):
        r, dt, done, start = oracle_sample_rate(w, per_step, start=start)
        rates.append(r)
        secs += dt
        n += done
    value = float(np.mean(rates))
    B, H, NQB = w.mask.shape[:3]
    sample = (f"{n} (b,h,q-block) rows of {B * H * NQB} in a seeded permutation, "
              f"{per_step:.1f} s per step, fp64 NumPy oracle")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / max(1, args.steps),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": _config(w, gpu=False),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": _cores(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def _input_bytes(w) -> int:
    return (w.q.numel() + w.k.numel() + w.v.numel()) * 2 if w.q is not None else 0


def _needs_flush(w) -> bool:
    return _input_bytes(w) <= L2_BYTES


def _config(w, gpu: bool = True):
    c = {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "Nq": w.Nq, "Nk": w.Nk,
         "d": w.d, "bq": w.bq, "bk": w.bk, "active_blocks": w.active_blocks,
         "density": round(w.density, 4), "active_flop_per_step": w.active_flop}
    if gpu:
        inputs = _input_bytes(w)
        c["l2"] = (f"inputs {inputs / 1e6:.0f} MB > L2 {L2_BYTES / 1e6:.0f} MB, no flush"
                   if not _needs_flush(w) else
                   f"inputs {inputs / 1e6:.0f} MB fit in L2: a 256 MB buffer is written between "
                   "steps, outside the per-step events")
    return c


class _Case:
    """One workload resident on the device, with the buffers and the step of
    the hot path (plan, then forward) for it."""

    def __init__(self, bsa, W, w, dev, stream, remap=False, page_size=0, causal=False,
                 affine=False, flags=None):
        self.bsa, self.w, self.dev, self.stream = bsa, w, dev, stream
        self.mask_d = w.mask.to(dev)
        q, k, v = w.q.to(dev), w.k.to(dev), w.v.to(dev)
        self.fwd_extra = {"causal": bool(causal)}
        if page_size:
            # paged K/V: the sequence's pages scattered over the pools in a
            # seeded random order, read through the block table (bsa_forward_ex)
            ps = page_size
            B_, Hkv_, Nk_, d_ = k.shape
            if Nk_ % ps:
                raise SystemExit(f"--page-size {ps} does not divide Nk = {Nk_}")
            npg = Nk_ // ps
            perm = torch.randperm(B_ * npg, generator=torch.Generator().manual_seed(5)).to(dev)

            def to_pool(t):
                pages = t.view(B_, Hkv_, npg, ps, d_).permute(0, 2, 1, 3, 4).reshape(B_ * npg, Hkv_, ps, d_)
                pool = torch.empty(pages.shape, dtype=pages.dtype, device=dev)
                pool[perm] = pages
                return pool
            k, v = to_pool(k), to_pool(v)
            self.fwd_extra["block_table"] = perm.view(B_, npg).to(torch.int32).contiguous()
        self.q, self.k, self.v = q, k, v
        self.o = torch.empty_like(q)
        self.lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
        self.plan_flags = (bsa.PLAN_REMAP if remap else 0) if flags is None else int(flags)
        L = bsa.plan_layout(*w.mask.shape, w.bq, w.bk, w.gqa_group, self.plan_flags)
        self.wsbuf = torch.empty(int(L.workspace_bytes), dtype=torch.uint8, device=dev)
        self.tile_rows = L.qu * L.rq
        self.remap_active = bool((self.plan_flags & bsa.PLAN_REMAP) and L.rq > 1 and w.gqa_group == 1
                                 and L.NQT <= 8192)
        self.affine = None
        if affine:
            # sliding, strided and dilated heads as affine row segments, the
            # BigBird-style heads as mask rows (bsa_plan_create_affine)
            if w.name != "regular":
                raise SystemExit("--affine describes the regular workload's patterns")
            segs, _ = W.regular_segments(w.Hq, w.mask.shape[3])
            self.affine = (bsa._lib.affine_segments(segs, dev), self.mask_d)
        self.side = torch.cuda.Stream(device=dev)
        self.fork = torch.cuda.Event()
        self.flush = (torch.empty(256 << 20, dtype=torch.uint8, device=dev)
                      if _needs_flush(w) else None)
        self.p = None

    # per step: 3 plan kernels (+1 when regrouping is active) + key norms,
    # row bounds, bounded pass, exact pass
    @property
    def launches_per_step(self) -> int:
        return 7 + int(self.remap_active)

    def step(self, ev=None):
        """A step: the plan kernels on the launching stream and, beside them on
        a side stream, the key-norm pass (it reads only K and V); then the
        row-bound, bounded and exact passes once both are done
        (bsa_forward_stage).  Events: step start, plan + key norms done,
        bounded pass start, bounded pass end, step end, plan kernels done,
        key-norm pass start and end (on the side stream)."""
        bsa, w, stream = self.bsa, self.w, self.stream
        if ev is not None:
            ev[0].record(stream)
        self.fork.record(stream)
        if self.affine is not None:
            p = bsa.plan_affine(self.affine[0], w.B, w.mask.shape[2], w.mask.shape[3], w.bq, w.bk,
                                w.gqa_group, mask=self.affine[1], workspace=self.wsbuf,
                                flags=self.plan_flags)
        else:
            p = bsa.plan(self.mask_d, w.bq, w.bk, w.gqa_group, workspace=self.wsbuf,
                         flags=self.plan_flags)
        if ev is not None:
            ev[5].record(stream)  # the plan kernels are done
        self.side.wait_event(self.fork)  # starts with the plan kernels, not after them
        args = (p, self.q, self.k, self.v)
        kw = dict(out=self.o, lse=self.lse, **self.fwd_extra)
        if ev is not None:
            ev[6].record(self.side)
        bsa.forward(*args, stages=bsa.STAGE_KNORM, stream=self.side, **kw)
        if ev is not None:
            ev[7].record(self.side)
        stream.wait_stream(self.side)
        if ev is not None:
            ev[1].record(stream)
        bsa.forward(*args, stages=bsa.STAGE_ROWBOUND, **kw)
        if ev is not None:
            ev[2].record(stream)
        bsa.forward(*args, stages=bsa.STAGE_BOUNDED, **kw)
        if ev is not None:
            ev[3].record(stream)
        bsa.forward(*args, stages=bsa.STAGE_EXACT, **kw)
        if ev is not None:
            ev[4].record(stream)
        self.p = p
        return p

    def check(self, when):
        st, det = self.bsa.sync_status(self.p)
        if st != 0:
            raise RuntimeError(f"{self.w.name}: device status {st} detail {det:#x} {when}")

    def warm(self, n):
        for _ in range(n):
            self.step()
        torch.cuda.synchronize()
        self.check("during warm-up")

    def timed(self, steps, barrier=lambda: None):
        """Time `steps` steps; returns (per-step events, wall t0, wall t1)."""
        fev = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(8)) for _ in range(steps)]
        barrier()
        torch.cuda.synchronize()
        t0 = time.time()
        for i in range(steps):
            if self.flush is not None:
                self.flush.fill_(i & 0xff)
            self.step(fev[i])
        torch.cuda.synchronize()
        t1 = time.time()
        barrier()
        self.check("in the timed region")
        return fev, t0, t1

    def plan_stats(self):
        """Plan totals: algorithmic plan bytes, computed FLOP (every slot
        computes 128 query rows x 128 keys) and computed / selected."""
        w = self.w
        tot = self.p.arrays()["totals"]
        S_, U_ = int(tot[0]), int(tot[2])
        Lp = self.p.layout
        plan_bytes = (w.mask.numel() + 4 * (Lp.rows + 1) + 4 * S_ * Lp.rk + 4 * S_ + 4 * Lp.rows
                      + 4 * (Lp.urows + 1) + 4 * U_)
        computed = 4.0 * self.tile_rows * 128 * w.d * S_
        return plan_bytes, computed, computed / w.active_flop

    def free(self):
        for n in ("q", "k", "v", "o", "lse", "wsbuf", "mask_d", "flush", "p", "affine"):
            setattr(self, n, None)


def _times(fev):
    """Mean over the timed steps: step, forward (after the preparation),
    preparation (plan and key norms side by side), bounded pass, plan kernels
    alone, key-norm pass alone (ms)."""
    ms = float(np.mean([e[0].elapsed_time(e[4]) for e in fev]))
    fwd_ms = float(np.mean([e[1].elapsed_time(e[4]) for e in fev]))
    prep_ms = float(np.mean([e[0].elapsed_time(e[1]) for e in fev]))
    bounded_ms = float(np.mean([e[2].elapsed_time(e[3]) for e in fev]))
    plan_ms = float(np.mean([e[0].elapsed_time(e[5]) for e in fev]))
    knorm_ms = float(np.mean([e[6].elapsed_time(e[7]) for e in fev]))
    return ms, fwd_ms, prep_ms, bounded_ms, plan_ms, knorm_ms


# GB300 nominal dense bf16 tensor throughput per GPU (datasheet figure without
# 2:4 sparsity), reported beside the measured peak.
NOMINAL_BF16_TFLOPS = 2250.0
PER_CONFIG = ("long_video_dit", "chunked_prefill", "regular", "tiny")


def per_config_entry(bsa, W, name, dev, stream, clocks, peak, target_s=0.5):
    """Measure one more workload in this process: the same step, timed over
    enough steps for about `target_s` seconds (20 .. 2000 steps)."""
    w = W.make_workload(name)
    remap = w.bq < 128 and w.gqa_group == 1
    c = _Case(bsa, W, w, dev, stream, remap=remap)
    c.warm(3)
    t0 = time.perf_counter()
    for _ in range(3):
        c.step()
    torch.cuda.synchronize()
    est = (time.perf_counter() - t0) / 3
    steps = int(min(2000, max(20, math.ceil(target_s / max(est, 1e-6)))))
    fev, w0, w1 = c.timed(steps)
    ms, fwd_ms, prep_ms, bounded_ms, plan_ms, knorm_ms = _times(fev)
    _, computed, ratio = c.plan_stats()
    flop = w.active_flop
    kern = flop / (bounded_ms * 1e-3) / 1e12
    e = {"workload": name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "Nq": w.Nq, "Nk": w.Nk, "d": w.d,
         "bq": w.bq, "bk": w.bk, "density": round(w.density, 4), "active_flop": flop,
         "computed_over_selected": ratio, "plan_flags": "BSA_PLAN_REMAP" if c.remap_active else 0,
         "steps": steps, "step_ms": ms, "value": flop / (ms * 1e-3) / 1e12,
         "kernel": "bsa_fwd_kernel<%d, bounded>" % w.d, "kernel_ms": bounded_ms,
         "roofline": {"achieved": kern, "peak": peak, "frac": kern / peak,
                      "frac_of_nominal": kern / NOMINAL_BF16_TFLOPS},
         "forward_ms": fwd_ms, "plan_ms": plan_ms, "knorm_ms": knorm_ms, "prep_ms": prep_ms,
         "clocks": clocks.summary(w0, w1)}
    c.free()
    del c, w
    torch.cuda.empty_cache()
    return e


def _e2e(bsa, w, args, ws, dev, barrier):
    """End to end through the public API: host (pinned) buffers, the copies
    in the timed region (bsa.attention -> bsa_attention_host)."""
    mask_h = w.mask.pin_memory()
    q_h, k_h, v_h = w.q.pin_memory(), w.k.pin_memory(), w.v.pin_memory()
    n_e2e = max(2, min(args.steps, args.e2e_steps))
    o_pin = torch.empty(w.q.shape, dtype=w.q.dtype, pin_memory=True)
    l_pin = torch.empty(w.q.shape[:3], dtype=torch.float32, pin_memory=True)
    bsa.attention(mask_h, q_h, k_h, v_h, w.bq, w.bk, out=o_pin, lse_out=l_pin)
    barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(n_e2e):
        oh, lh = bsa.attention(mask_h, q_h, k_h, v_h, w.bq, w.bk, out=o_pin, lse_out=l_pin)
    torch.cuda.synchronize()
    e2e_ms = (time.perf_counter() - t0) * 1e3 / n_e2e
    (e2e_ms,) = max_over_ranks([e2e_ms], dev)
    h2d = mask_h.numel() + (q_h.numel() + k_h.numel() + v_h.numel()) * 2
    d2h = oh.numel() * 2 + lh.numel() * 4
    del mask_h, q_h, k_h, v_h, o_pin, l_pin, oh, lh
    bsa._lib._host_buffers.clear()
    torch.cuda.empty_cache()
    return {"value": whole_job_tflops(w.active_flop, e2e_ms, ws), "unit": UNIT,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "ms_per_step": e2e_ms}


def run_gb300(args):
    ws, rank, local = _dist()
    import block_sparse_attention_plan_gb300 as bsa
    from block_sparse_attention_plan_gb300 import workloads as W

    w = W.make_workload(args.config)
    peak, peak_sus, peak_src = _peaks()
    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        # before any CUDA work: the oracle on the host cores, bounded sample
        r, dt, n, _ = oracle_sample_rate(w, args.cpu_seconds)
        B, H, NQB = w.mask.shape[:3]
        from oracle import plan as OP
        t0 = time.perf_counter()
        OP.build_plan(w.mask.numpy(), w.bq, w.bk, w.gqa_group)
        plan_s = time.perf_counter() - t0
        cpu = {"value": r, "unit": UNIT, "cores": _cores(), "kind": "oracle",
               "sample": f"{n} of {B * H * NQB} (b,h,q-block) rows of the same workload, seeded "
                         f"permutation, {dt:.1f} s, fp64 NumPy oracle",
               "plan_oracle_s": plan_s, "plan_oracle_cores": 1}

    dist = ws > 1
    if dist:
        import torch.distributed as td
        td.init_process_group("nccl", device_id=torch.device(f"cuda:{local}"))
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()

    c = _Case(bsa, W, w, dev, stream, remap=args.remap, page_size=args.page_size,
              causal=args.causal, affine=args.affine, flags=args.plan_flags)
    flop = w.active_flop

    def barrier():
        if dist:
            torch.distributed.barrier()

    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        uuid = str(local)
    clocks = ClockSampler(uuid)

    c.warm(args.warmup)
    fev, t_wall0, t_wall1 = c.timed(args.steps, barrier)
    plan_bytes, computed, ratio = c.plan_stats()
    # key-norm pass: K and V read once, a float per unit and tensor written
    Lk = c.p.layout
    knorm_bytes = 2 * w.k.numel() * 2 + 2 * 4 * Lk.B * Lk.Hkv * Lk.NKU
    # a step = plan start -> forward end, timed with events on the launching stream
    ms, fwd_ms, prep_ms, bounded_ms, plan_ms, knorm_ms = _times(fev)
    ms, fwd_ms, bounded_ms = max_over_ranks([ms, fwd_ms, bounded_ms], dev)
    clk = clocks.summary(t_wall0, t_wall1)
    launches = c.launches_per_step * args.steps
    c.free()
    e2e = None
    if not args.no_e2e:
        e2e = _e2e(bsa, w, args, ws, dev, barrier)

    per_config = None
    if rank == 0 and ws == 1 and not args.no_per_config:
        per_config = [per_config_entry(bsa, W, name, dev, stream, clocks, peak)
                      for name in PER_CONFIG if name != w.name]
    clocks.stop()

    value = whole_job_tflops(flop, ms, ws)
    achieved = flop / (bounded_ms * 1e-3) / 1e12      # the dominant kernel's launch
    achieved_fwd = flop / (fwd_ms * 1e-3) / 1e12      # the whole bsa_forward
    cfg = _config(w)
    cfg["computed_over_selected"] = ratio
    if args.page_size:
        cfg["kv_pages"] = (f"page_size {args.page_size}, pages shuffled across the pool, read "
                           "through a block table (e2e stays on contiguous host buffers)")
    if args.remap:
        cfg["plan_flags"] = "BSA_PLAN_REMAP: per-plane q-unit grouping stride chosen by slot count"
    if args.affine:
        cfg["plan_input"] = ("affine row segments for the sliding, strided and dilated heads; the "
                             "BigBird-style heads' rows read from the mask")
    if args.causal:
        cfg["causal"] = ("intra-block causal element mask; FLOP counted over whole selected "
                         "blocks, as the tensor cores execute them")
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": cfg,
        "pct_of_peak": 100.0 * value / ws / peak,
        "pct_of_nominal_peak": 100.0 * value / ws / NOMINAL_BF16_TFLOPS,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak,
                     "traffic": (args.traffic if args.traffic is not None else
                                 None if (args.page_size or args.causal) else _traffic(w.name)),
                     # achieved: over the bounded pass's launch (CUDA events
                     # around it, mean over the timed steps); forward_*: from
                     # the end of the plan and key-norm pass (which run side
                     # by side) to the end of the step: row-bound, bounded
                     # and exact passes.
                     "kernel": "bsa_fwd_kernel<%d, bounded>" % w.d, "kernel_ms": bounded_ms,
                     "forward_ms": fwd_ms, "forward_achieved": achieved_fwd,
                     "forward_frac": achieved_fwd / peak, "peak_source": f"{peak_src} bf16 burst",
                     "frac_of_sustained": achieved / peak_sus,
                     "frac_of_nominal": achieved / NOMINAL_BF16_TFLOPS,
                     "nominal_peak": NOMINAL_BF16_TFLOPS},
        "e2e": e2e,
        "plan_ms": plan_ms,
        "plan": {"ms": plan_ms, "bytes": int(plan_bytes),
                 "gbs": plan_bytes / (plan_ms * 1e-3) / 1e9,
                 "frac_of_hbm": plan_bytes / (plan_ms * 1e-3) / 1e9 / _hbm_gbs(),
                 "knorm_ms": knorm_ms, "knorm_bytes": int(knorm_bytes),
                 "knorm_gbs": knorm_bytes / (knorm_ms * 1e-3) / 1e9,
                 "knorm_frac_of_hbm": knorm_bytes / (knorm_ms * 1e-3) / 1e9 / _hbm_gbs(),
                 "prep_ms": prep_ms,
                 "note": "ms: step start until the plan kernels are done (their own time, beside "
                         "the key-norm pass on a second stream); knorm_ms: the key-norm pass, "
                         "which reads K and V once; prep_ms: step start until both are done. The "
                         "plan kernels are latency-bound at these sizes"},
        "gpu_launches": launches,
        "clocks": clk,
    }
    if cpu is not None:
        line["cpu_baseline"] = cpu
    if per_config is not None:
        line["per_config"] = per_config
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        torch.distributed.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--config", default="video_dit")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--page-size", type=int, default=0,
                    help="read K/V through a block table of pages of this many keys (0: contiguous)")
    ap.add_argument("--remap", action="store_true",
                    help="plan with BSA_PLAN_REMAP (per-plane q-unit grouping stride)")
    ap.add_argument("--affine", action="store_true",
                    help="regular workload: plan from affine row segments (+ residual mask bytes)")
    ap.add_argument("--causal", action="store_true",
                    help="intra-block causal masking (queries are the last Nq positions)")
    ap.add_argument("--plan-flags", type=int, default=None,
                    help="plan flags (BSA_PLAN_*) for the timed step; overrides --remap")
    ap.add_argument("--no-e2e", action="store_true",
                    help="skip the end-to-end leg (sweeps of the device path only)")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the per_config record of the other workloads")
    ap.add_argument("--traffic", type=float, default=None,
                    help="DRAM bytes per forward launch from an ncu capture of this kernel")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_gb300(args)


if __name__ == "__main__":
    sys.exit(main())
