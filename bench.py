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
    "video_dit": (302.4256e6 + 79.938048e6, "75d86ea2a5bd10e4"),
}
KERNEL_SOURCES = ("block_sparse_attention_plan_gb300/csrc/bsa_forward.cu",
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

    mask_d = w.mask.to(dev)
    q, k, v = w.q.to(dev), w.k.to(dev), w.v.to(dev)
    fwd_extra = {"causal": bool(args.causal)}
    if args.page_size:
        # paged K/V: the sequence's pages scattered over the pools in a seeded
        # random order, read through the block table (bsa_forward_ex)
        ps = args.page_size
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
        fwd_extra["block_table"] = perm.view(B_, npg).to(torch.int32).contiguous()
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    L = bsa.plan_layout(*w.mask.shape, w.bq, w.bk, w.gqa_group)
    wsbuf = torch.empty(int(L.workspace_bytes), dtype=torch.uint8, device=dev)
    flop = w.active_flop

    plan_flags = bsa.PLAN_REMAP if args.remap else 0
    remap_active = bool(args.remap and w.bq < 128 and w.gqa_group == 1 and w.Nq // 128 <= 8192)
    affine = None
    if args.affine:
        # sliding, strided and dilated heads as affine row segments, the
        # BigBird-style heads as mask rows (bsa_plan_create_affine)
        if w.name != "regular":
            raise SystemExit("--affine describes the regular workload's patterns")
        segs, _ = W.regular_segments(w.Hq, w.mask.shape[3])
        affine = (bsa._lib.affine_segments(segs, dev), mask_d)  # only BigBird heads' rows are read

    # A step: the plan kernels on the launching stream and, beside them on a
    # side stream, the key-norm pass (it reads only K); then the row-bound,
    # bounded and exact passes once both are done (bsa_forward_stage).
    # Events of a timed step: step start, plan + key norms done, bounded pass
    # start, bounded pass end, step end.
    side = torch.cuda.Stream(device=dev)
    fork = torch.cuda.Event()

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        fork.record(stream)
        if affine is not None:
            p = bsa.plan_affine(affine[0], w.B, w.mask.shape[2], w.mask.shape[3], w.bq, w.bk,
                                w.gqa_group, mask=affine[1], workspace=wsbuf, flags=plan_flags)
        else:
            p = bsa.plan(mask_d, w.bq, w.bk, w.gqa_group, workspace=wsbuf, flags=plan_flags)
        side.wait_event(fork)  # starts with the plan kernels, not after them
        bsa.forward(p, q, k, v, out=o, lse=lse, stages=bsa.STAGE_KNORM, stream=side, **fwd_extra)
        stream.wait_stream(side)
        if ev is not None:
            ev[1].record(stream)
        bsa.forward(p, q, k, v, out=o, lse=lse, stages=bsa.STAGE_ROWBOUND, **fwd_extra)
        if ev is not None:
            ev[2].record(stream)
        bsa.forward(p, q, k, v, out=o, lse=lse, stages=bsa.STAGE_BOUNDED, **fwd_extra)
        if ev is not None:
            ev[3].record(stream)
        bsa.forward(p, q, k, v, out=o, lse=lse, stages=bsa.STAGE_EXACT, **fwd_extra)
        if ev is not None:
            ev[4].record(stream)
        return p

    def barrier():
        if dist:
            torch.distributed.barrier()

    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        uuid = str(local)
    clocks = ClockSampler(uuid)

    p = None
    for _ in range(args.warmup):
        p = step()
    torch.cuda.synchronize()
    if p is not None:
        st, det = bsa.sync_status(p)
        if st != 0:
            raise RuntimeError(f"device status {st} detail {det:#x} during warm-up")

    fev = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(5)) for _ in range(args.steps)]
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if _needs_flush(w) else None
    barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    for i in range(args.steps):
        if flush is not None:
            flush.fill_(i & 0xff)
        p = step(fev[i])
    torch.cuda.synchronize()
    t_wall1 = time.time()
    barrier()
    st, det = bsa.sync_status(p)
    if st != 0:
        raise RuntimeError(f"device status {st} detail {det:#x} in the timed region")
    # plan bytes (algorithmic): the mask read once (none for affine heads'
    # rows, counted anyway), the plan arrays written once
    tot = p.arrays()["totals"]
    S_, U_ = int(tot[0]), int(tot[2])
    R_ = p.layout.rows
    plan_bytes = (w.mask.numel() + 4 * (R_ + 1) + 4 * S_ * p.layout.rk + 4 * S_ + 4 * R_
                  + 4 * (p.layout.urows + 1) + 4 * U_)
    # a step = plan start -> forward end, timed with events on the launching stream
    ms = float(np.mean([e[0].elapsed_time(e[4]) for e in fev]))
    fwd_ms = float(np.mean([e[1].elapsed_time(e[4]) for e in fev]))
    plan_ms = float(np.mean([e[0].elapsed_time(e[1]) for e in fev]))
    bounded_ms = float(np.mean([e[2].elapsed_time(e[3]) for e in fev]))
    ms, fwd_ms, bounded_ms = max_over_ranks([ms, fwd_ms, bounded_ms], dev)
    clk = clocks.summary(t_wall0, t_wall1)

    # end to end through the public API, host (pinned) buffers, copies timed
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
    clocks.stop()
    h2d = mask_h.numel() + (q_h.numel() + k_h.numel() + v_h.numel()) * 2
    d2h = oh.numel() * 2 + lh.numel() * 4

    value = whole_job_tflops(flop, ms, ws)
    achieved = flop / (bounded_ms * 1e-3) / 1e12      # the dominant kernel's launch
    achieved_fwd = flop / (fwd_ms * 1e-3) / 1e12      # the whole bsa_forward
    cfg = _config(w)
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
                     "frac_of_sustained": achieved / peak_sus},
        "e2e": {"value": whole_job_tflops(flop, e2e_ms, ws), "unit": UNIT,
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "ms_per_step": e2e_ms},
        "plan_ms": plan_ms,
        "plan": {"ms": plan_ms, "bytes": int(plan_bytes),
                 "gbs": plan_bytes / (plan_ms * 1e-3) / 1e9,
                 "frac_of_hbm": plan_bytes / (plan_ms * 1e-3) / 1e9 / _hbm_gbs(),
                 "note": "ms: step start until the plan kernels and the key-norm pass, run side by "
                         "side, are both done; the plan kernels are latency-bound at these sizes"},
        # per step: 3 plan kernels (+1 when regrouping is active) + key norms,
        # row bounds, bounded pass, exact pass
        "gpu_launches": (7 + int(remap_active)) * args.steps,
        "clocks": clk,
    }
    if cpu is not None:
        line["cpu_baseline"] = cpu
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
