#!/usr/bin/env python
"""Benchmark of the batched pentadiagonal solves on GB300.

Default workload: the shared-matrix solve, N = 1024, batch = 65536, fp64,
bands [1, -4, 7, -4, 1] (sigma = 1, non-cyclic), factored once; one step = one
solve of the whole batch (read f, write x: 2 x 512 MB).  Other workloads
(--workload small | cyclic | persys | ch) time the other rows of the hot path.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints ONE JSON line (rank 0).  `value` is whole-job throughput with inputs
resident in HBM; `e2e` is the same metric through the public Python API with
pinned host buffers, both copies inside the timed region; `roofline` is the
dominant kernel's algorithmic bandwidth against the measured HBM peak;
`cpu_baseline` times the CPU oracle on a bounded sample.  With --gpus > 1 (under
torchrun) every rank solves its own batch (weak scaling, no collective on the
data path); the timed region is bracketed by barriers and the max over ranks is
taken.
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "pentadiagonal system-solves/s (N=1024, fp64) and HBM GB/s vs GB300 peak"
FALLBACK_HBM_GBS = 6800.0

WORKLOADS = {
    "shared": dict(N=1024, batch=65536, kind="shared", sigma=1.0, cyclic=False, dtype="f64",
                   desc="shared-matrix pentadiagonal solve, N=1024, batch=65536, fp64, "
                        "bands [1,-4,7,-4,1] (sigma=1), non-cyclic, factor once"),
    "small": dict(N=128, batch=1024, kind="shared", sigma=1.0, cyclic=False, dtype="f64",
                  desc="shared-matrix pentadiagonal solve, N=128, batch=1024, fp64, sigma=1"),
    "long": dict(N=1 << 20, batch=16, kind="shared", sigma=1.0, cyclic=False, dtype="f64",
                 desc="shared-matrix pentadiagonal solve of few long systems, N=1048576, batch=16, "
                      "fp64, sigma=1 (partitioned solve across CTAs)"),
    "cyclic": dict(N=512, batch=4096, kind="hyper", sigma=0.5, cyclic=True, dtype="f64",
                   desc="periodic hyperdiffusion step, cyclic I+0.5*D4, N=512, batch=4096, fp64"),
    "tri": dict(N=256, batch=262144, kind="tri", dtype="f32",
                desc="per-system tridiagonal factor+solve (Thomas), N=256, batch=262144, fp32, "
                     "diagonally dominant"),
    "tri64": dict(N=256, batch=262144, kind="tri", dtype="f64",
                  desc="per-system tridiagonal factor+solve (Thomas), N=256, batch=262144, fp64, "
                       "diagonally dominant"),
    "tri_bi16": dict(N=256, batch=262144, kind="tri", dtype="f32", bs=16,
                     desc="per-system tridiagonal factor+solve, block-interleaved layout (blocks of 16 "
                          "systems), N=256, batch=262144, fp32, diagonally dominant"),
    "persys64": dict(N=256, batch=262144, kind="persys", dtype="f64",
                     desc="per-system factor+solve, N=256, batch=262144, fp64, diagonally dominant"),
    "persys_bi16": dict(N=256, batch=262144, kind="persys", dtype="f32", bs=16,
                        desc="per-system factor+solve, block-interleaved layout (blocks of 16 systems), "
                             "N=256, batch=262144, fp32, diagonally dominant"),
    "persys": dict(N=256, batch=262144, kind="persys", dtype="f32",
                   desc="per-system factor+solve, N=256, batch=262144, fp32, diagonally dominant"),
    "cn": dict(N=512, batch=4096, kind="cn", sigma=0.25, cyclic=True, dtype="f64",
               desc="periodic Crank-Nicolson hyperdiffusion step, (I+0.25*D4)C'=(I-0.25*D4)C, "
                    "N=512, batch=4096, fp64"),
    "cyclic100": dict(N=512, batch=4096, kind="hyper", sigma=0.5, cyclic=True, dtype="f64", nsub=100,
                      desc="periodic hyperdiffusion, 100 steps per call (persistent multi-step kernel), "
                           "cyclic I+0.5*D4, N=512, batch=4096, fp64"),
    "cn100": dict(N=512, batch=4096, kind="cn", sigma=0.25, cyclic=True, dtype="f64", nsub=100,
                  desc="periodic Crank-Nicolson hyperdiffusion, 100 steps per call (persistent "
                       "multi-step kernel), sigma_x=0.25, N=512, batch=4096, fp64"),
    "ch100": dict(N=1024, batch=16384, kind="ch", cyclic=True, dtype="f64", nsub=100,
                  desc="semi-implicit Cahn-Hilliard, 100 steps per call (persistent multi-step "
                       "kernel), N=1024, batch=16384, fp64, gamma=1e-4, dt=0.1dx^2"),
    "ch": dict(N=1024, batch=16384, kind="ch", cyclic=True, dtype="f64",
               desc="semi-implicit Cahn-Hilliard step (fused RHS + cyclic solve), N=1024, "
                    "batch=16384, fp64, gamma=1e-4, dt=0.1dx^2"),
    "ch2000": dict(N=1024, batch=16384, kind="ch", cyclic=True, dtype="f64", nsub=2000,
                   desc="semi-implicit Cahn-Hilliard, 2000 steps per call (the whole run of the "
                        "workload in one persistent multi-step launch), N=1024, batch=16384, fp64, "
                        "gamma=1e-4, dt=0.1dx^2, C0 ~ U[-0.1, 0.1]"),
}


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# ----------------------------------------------------------------------------
# distributed plumbing (one process per GPU, NCCL only for barrier / max)
# ----------------------------------------------------------------------------
class Dist:
    def __init__(self, ngpus: int):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch
            import torch.distributed as dist
            backend = "nccl" if torch.cuda.is_available() else "gloo"
            if backend == "nccl":
                torch.cuda.set_device(self.local)
            dist.init_process_group(backend)
            self.pg = dist

    def barrier(self):
        if self.pg is not None:
            self.pg.barrier()

    def max(self, v: float) -> float:
        if self.pg is None:
            return v
        import torch
        dev = "cuda" if torch.cuda.is_available() else "cpu"
        t = torch.tensor([v], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg is not None:
            self.pg.destroy_process_group()


def shard(batch: int, world: int, rank: int, weak: bool = True):
    """Systems of this rank.  Weak scaling: every rank gets the full per-GPU batch."""
    if weak:
        return batch
    base, rem = divmod(batch, world)
    return base + (1 if rank < rem else 0)


# ----------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.05)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()
        return False

    def summary(self):
        rows = []
        for line in (self.out or "").strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                rows.append(dict(sm=float(parts[0]), max=float(parts[1]), power=float(parts[2]),
                                 hw=parts[4], hwt=parts[5], swt=parts[6], swp=parts[7]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        reasons = set()
        for r in rows:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("swp", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        loaded = [r["sm"] for r in rows if r["power"] > 0] or [r["sm"] for r in rows]
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(r["max"] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows),
                "power_w_max": max(r["power"] for r in rows)}


# ----------------------------------------------------------------------------
# peaks and ncu traffic
# ----------------------------------------------------------------------------
def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            return float(json.load(fh)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def source_digest(kernel_file: str) -> str:
    """Digest of a kernel's source file and the local headers it includes (the
    plan/launcher declarations in pent_internal.cuh are left out: they do not change
    the kernel's code)."""
    csrc = os.path.join(ROOT, "implicit_pde_stepping_gb300", "csrc")
    h = hashlib.sha256()
    path = os.path.join(csrc, kernel_file)
    if not os.path.exists(path):
        return ""
    text = open(path, "rb").read()
    h.update(text)
    for line in text.decode(errors="replace").splitlines():
        line = line.strip()
        if line.startswith('#include "') and "pent_internal.cuh" not in line:
            inc = os.path.join(csrc, line.split('"')[1])
            if os.path.exists(inc):
                with open(inc, "rb") as fh:
                    h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_record(kernel: str, kernel_file: str, workload: str):
    """The committed ncu summary of `kernel` on `workload` (profiles/ncu_traffic.json):
    DRAM bytes and, where captured, warp instructions and issue activity of one launch
    on `units` systems.  None if missing or if the kernel changed since the capture."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as fh:
            table = json.load(fh)
    except (OSError, ValueError):
        return None
    rec = table.get(f"{kernel}@{workload}")
    if not rec or rec.get("source_digest") != source_digest(kernel_file):
        return None
    return rec


def ncu_traffic(kernel: str, kernel_file: str, workload: str, units: int):
    """DRAM bytes per launch from the committed ncu summary, scaled to `units` systems when
    the capture was taken on a smaller case; None if the kernel changed since the capture."""
    rec = ncu_record(kernel, kernel_file, workload)
    if rec is None or "dram_bytes_per_launch" not in rec:
        return None
    return float(rec["dram_bytes_per_launch"]) * units / float(rec["units"])


# ----------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------
def run_ours(args, W: dict, dist: Dist):
    import numpy as np
    import torch

    from implicit_pde_stepping_gb300 import inputs, pent

    dev_index = dist.local if dist.world > 1 else 0
    torch.cuda.set_device(dev_index)
    stream = torch.cuda.Stream()
    N = W["N"]
    batch = shard(args.batch or W["batch"], dist.world, dist.rank, weak=True)
    kind = W["kind"]
    seed = dist.rank
    fdt = torch.float64 if W["dtype"] == "f64" else torch.float32
    elem = 8 if W["dtype"] == "f64" else 4

    # ---- inputs (host generator -> HBM), plan
    plan = None
    k2 = None
    if kind in ("shared", "hyper", "cn"):
        plan = pent.pent_factor(inputs.hyper_bands(N, W["sigma"]), batch, cyclic=W["cyclic"])
        bufs = [torch.from_numpy(inputs.rhs_uniform(N, batch, seed=seed + r) if kind == "shared"
                                 else inputs.fourier_initial(N, batch, seed=seed + r)).to("cuda")
                for r in range(2)]
    elif kind == "ch":
        sigma, k2 = inputs.ch_params(N)
        plan = pent.pent_factor(inputs.hyper_bands(N, sigma), batch, cyclic=True)
        bufs = [torch.from_numpy(inputs.ch_initial(N, batch, seed=seed + r)).to("cuda")
                for r in range(2)]
    elif kind in ("tri", "persys"):
        bs = W.get("bs", 0)

        def lay(x):   # interleaved [N][batch] -> the workload's layout
            if not bs:
                return np.ascontiguousarray(x)
            return np.ascontiguousarray(x.reshape(N, batch // bs, bs).transpose(1, 0, 2))
        gen = inputs.tri_bands if kind == "tri" else inputs.persys_bands
        npdt = np.float64 if W["dtype"] == "f64" else np.float32
        bands = [torch.from_numpy(lay(v)).to("cuda") for v in gen(N, batch, seed=seed, dtype=npdt)]
        bufs = [torch.from_numpy(lay(inputs.rhs_uniform(N, batch, seed=seed + r).astype(npdt)))
                .to("cuda") for r in range(2)]
        # scratch only where the kernel that runs uses it: the fp32 partitioned kernels
        # (N <= 512) keep everything on chip and take none
        code = pent.F64 if W["dtype"] == "f64" else pent.F32
        split_runs = (W["dtype"] == "f32" and N <= 512 and args.variant in ("auto", "split"))
        wb = (pent.tri_factor_solve_work_bytes if kind == "tri" else pent.pent_factor_solve_work_bytes)
        need = 0 if split_runs else wb(N, batch, code)
        work = torch.empty(need, dtype=torch.uint8, device="cuda") if need else None
    if plan is not None and args.variant != "auto":
        plan.set_variant(args.variant)
    variant = plan.variant(batch) if plan is not None else pent.VARIANT_THREAD
    tri_variant = args.variant if args.variant in ("thread", "split", "thread_df") else "auto"
    if kind in ("tri", "persys"):
        # per-system workloads: fp32 takes the partitioned kernel, fp64 the double-float
        # one-thread kernel, unless another variant is asked for
        if tri_variant != "auto":
            variant = pent.VARIANTS[tri_variant]
        else:
            variant = pent.VARIANT_THREAD_DF if W["dtype"] == "f64" else pent.VARIANT_SPLIT
    # inputs smaller than twice the L2: write a buffer larger than L2 between timed
    # steps, outside the per-step events, and time the steps by those events
    l2_bytes = getattr(torch.cuda.get_device_properties(dev_index), "L2_cache_size", 0) or (129 << 20)
    buf_bytes = bufs[0].numel() * bufs[0].element_size()
    # per-system matrices: solving in place again and again applies A^-1 over and over,
    # and for random diagonally dominant matrices that can grow some systems without
    # bound (into the native fp64 fallback); so every step starts again from the
    # right-hand side it was given, copied back outside the per-step events and
    # followed by the L2 flush
    refresh = kind in ("tri", "persys")
    pristine = [b.clone() for b in bufs] if refresh else None
    flush = buf_bytes < 2 * l2_bytes or refresh
    scratch = torch.empty(2 * l2_bytes // 4, dtype=torch.int32, device="cuda") if flush else None
    torch.cuda.synchronize()

    nsub = W.get("nsub", 1)     # time steps per call (one launch for all of them)

    def call(pl, st, X, wk, bnds):
        """One call of the workload's public entry point on stream st."""
        if kind == "shared":
            pent.pent_solve(pl, X, stream=st)
        elif kind == "hyper":
            pent.hyperdiffusion_step(pl, X, nsub, stream=st)
        elif kind == "ch":
            pent.ch_step(pl, X, k2, nsub, stream=st)
        elif kind == "cn":
            pent.cn_step(pl, X, nsub, stream=st)
        elif kind == "tri":
            pent.tri_factor_solve(*bnds, X, variant=tri_variant, work=wk, stream=st,
                                  block_size=W.get("bs", 0))
        else:
            pent.pent_factor_solve(*bnds, X, work=wk, stream=st, variant=tri_variant,
                                   block_size=W.get("bs", 0))

    def step(k, X=None):
        call(plan, stream, bufs[k % 2] if X is None else X, work if kind in ("tri", "persys") else None,
             bands if kind in ("tri", "persys") else None)

    # ---- device-resident timing
    with torch.cuda.stream(stream):
        for k in range(args.warmup):
            if refresh:
                bufs[k % 2].copy_(pristine[k % 2])
            step(k)
    stream.synchronize()
    torch.cuda.synchronize()
    dist.barrier()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    l0 = pent.launch_count()
    with ClockSampler(dev_index) as clocks:
        with torch.cuda.stream(stream):
            t_start.record(stream)
            for k in range(args.steps):
                if refresh:
                    bufs[k % 2].copy_(pristine[k % 2])
                if flush:
                    scratch.fill_(k)
                ev[k][0].record(stream)
                step(k)
                ev[k][1].record(stream)
            t_end.record(stream)
        stream.synchronize()
        torch.cuda.synchronize()
    launches = pent.launch_count() - l0
    dist.barrier()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    ms_local = sum(step_ms) if flush else t_start.elapsed_time(t_end)
    ms = dist.max(ms_local)
    kernel_ms = statistics.mean(step_ms)
    total_units = batch * nsub * args.steps * dist.world
    value = total_units / (ms / 1e3)

    # ---- end to end through the public API: pinned host in, host out, every step.
    # Two slots (each its own plan, stream, pinned host buffers and device buffers)
    # take the steps in turn, as a streaming application double-buffers: a step's
    # copy-in overlaps the previous step's copy-out.  Every step still copies its
    # own inputs in and its result out inside the timed region.
    e2e = None
    if not args.no_e2e:
        def new_plan():
            if kind in ("shared", "hyper", "cn"):
                q = pent.pent_factor(inputs.hyper_bands(N, W["sigma"]), batch, cyclic=W["cyclic"])
            elif kind == "ch":
                q = pent.pent_factor(inputs.hyper_bands(N, inputs.ch_params(N)[0]), batch, cyclic=True)
            else:
                return None
            if args.variant != "auto":
                q.set_variant(args.variant)
            return q

        # every input of a step comes from pinned host memory: the right-hand side, and for
        # per-system matrices also the five bands (the shared matrix lives in the plan)
        host_bands = [b.cpu().pin_memory() for b in bands] if kind in ("persys", "tri") else []
        slots = []
        for si in range(2):
            sl = {"stream": stream if si == 0 else torch.cuda.Stream(),
                  "plan": plan if si == 0 else new_plan(),
                  "host_in": bufs[si].cpu().pin_memory()}
            sl["host_out"] = torch.empty_like(sl["host_in"]).pin_memory()
            if kind != "shared":
                sl["Xd"] = torch.empty_like(bufs[0])
            sl["dev_bands"] = [torch.empty_like(b) for b in bands] if kind in ("persys", "tri") else None
            sl["work"] = (torch.empty_like(work) if (kind in ("persys", "tri") and work is not None)
                          else None)
            slots.append(sl)

        def e2e_step(sl):
            st = sl["stream"]
            with torch.cuda.stream(st):
                if kind == "shared":
                    # the library's host-buffer call: copy in, solve, copy out, overlapped
                    pent.pent_solve_host(sl["plan"], sl["host_in"], sl["host_out"],
                                         chunks=args.e2e_chunks, stream=st)
                    return
                for hb, db in zip(host_bands, sl["dev_bands"] or []):
                    db.copy_(hb, non_blocking=True)
                sl["Xd"].copy_(sl["host_in"], non_blocking=True)
                call(sl["plan"], st, sl["Xd"], sl["work"], sl["dev_bands"])
                sl["host_out"].copy_(sl["Xd"], non_blocking=True)

        ke = max(1, min(args.steps, args.e2e_steps))
        for _ in range(2):
            for sl in slots:
                e2e_step(sl)
        torch.cuda.synchronize()
        dist.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0, s1 = slots[0]["stream"], slots[1]["stream"]
        e0.record(s0)
        s1.wait_event(e0)
        for i in range(ke):
            e2e_step(slots[i % 2])
        last = torch.cuda.Event()
        last.record(s1)
        s0.wait_event(last)
        e1.record(s0)
        torch.cuda.synchronize()
        dist.barrier()
        ems = dist.max(e0.elapsed_time(e1))
        host_in = slots[0]["host_in"]
        nbytes_out = host_in.numel() * host_in.element_size()
        nbytes = nbytes_out + sum(b.numel() * b.element_size() for b in host_bands)
        e2e = {"value": batch * nsub * ke * dist.world / (ems / 1e3), "unit": "system-solves/s"
               if kind in ("shared", "persys", "tri") else "system-steps/s",
               "h2d_bytes_per_step": nbytes, "d2h_bytes_per_step": nbytes_out, "steps": ke,
               "ms_per_step": ems / ke,
               "api": ("pent_solve_host (pinned host in/out, chunks=%s)" % (args.e2e_chunks or "auto")
                       if kind == "shared" else "pinned host copies + the device-buffer call"),
               "pipelining": "two slots (plan, stream, pinned buffers each) take the steps in turn"}
        for sl in slots[1:]:
            if sl["plan"] is not None:
                sl["plan"].close()

    # ---- roofline of the dominant kernel (one kernel per step on every path)
    per_unit = {"shared": 2 * N * elem, "hyper": 2 * N * elem, "ch": 2 * N * elem,
                "cn": 2 * N * elem, "persys": 7 * N * elem, "tri": 5 * N * elem}[kind]
    alg_bytes = per_unit * batch
    achieved = alg_bytes / (kernel_ms / 1e3) / 1e9
    peak, peak_kind = hbm_peak()
    # the kernel one launch of the step runs (the fused CH / CN steps use the
    # partitioned kernel for every double-float variant)
    twisted = "k_twisted_async"
    split = ("k_split_df", "pent_split_df.cu")
    kernel_names = {
        ("shared", pent.VARIANT_THREAD): ("k_shared_thread", "pent_shared.cu"),
        ("hyper", pent.VARIANT_THREAD): ("k_shared_thread", "pent_shared.cu"),
        ("ch", pent.VARIANT_THREAD): ("k_ch_thread_f64", "pent_ch.cu"),
        ("cn", pent.VARIANT_THREAD): ("k_cn_thread_f64", "pent_ch.cu"),
        ("persys", pent.VARIANT_THREAD): ("k_persys_thread", "pent_persys.cu"),
        ("persys", pent.VARIANT_SPLIT): ("k_persys_split", "pent_persys_split.cu"),
        ("persys", pent.VARIANT_THREAD_DF): ("k_persys_thread_df", "pent_persys.cu"),
        ("tri", pent.VARIANT_THREAD): ("k_tri_thread", "pent_tri.cu"),
        ("tri", pent.VARIANT_SPLIT): ("k_tri_split", "pent_tri.cu"),
        ("tri", pent.VARIANT_THREAD_DF): ("k_tri_thread_df", "pent_tri.cu"),
        ("shared", pent.VARIANT_THREAD_DF): (twisted, "pent_twisted_df.cu"),
        ("hyper", pent.VARIANT_THREAD_DF): (twisted, "pent_twisted_df.cu"),
        ("ch", pent.VARIANT_THREAD_DF): split, ("ch", pent.VARIANT_SPLIT): split,
        ("cn", pent.VARIANT_THREAD_DF): split, ("cn", pent.VARIANT_SPLIT): split,
        ("shared", pent.VARIANT_SPLIT): split, ("hyper", pent.VARIANT_SPLIT): split,
    }
    kname, kfile = kernel_names.get((kind, variant), ("?", "?"))
    # non-cyclic partitioned solves of 256 to 2048 rows run the fixed-grid kernel
    if kind == "shared" and variant == pent.VARIANT_SPLIT and not W["cyclic"] and 256 <= N <= 2048:
        kname, kfile = "k_fg", "pent_fg.cu"
    if nsub > 1 and variant in (pent.VARIANT_SPLIT, pent.VARIANT_THREAD_DF):
        kname, kfile = "k_steps_df", "pent_steps_df.cu"
    # systems longer than one CTA holds (64 chunks of 32 rows; 32 when periodic)
    # run the partitioned solve as several kernels; the step is their sum
    if kind == "shared" and variant == pent.VARIANT_SPLIT and \
            (N - (2 if W["cyclic"] else 0)) > (1024 if W["cyclic"] else 2048):
        kname, kfile = "k_big", "pent_split_big.cu"
    traffic = ncu_traffic(kname, kfile, args.workload, batch)
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": traffic,
                "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind ==
                "measured" else "fallback 6.8 TB/s",
                "kernel": kname, "kernel_ms": round(kernel_ms, 4),
                "algorithmic_bytes_per_launch": alg_bytes,
                "bytes_per_unit": per_unit, "units_per_launch": batch}
    # instruction counts of the same capture, where recorded: instructions per point
    # (per point and step for the multi-step kernel)
    wl_rec = args.workload if nsub == 1 else ("cyclic100" if kind == "hyper" else
                                              "cn100" if kind == "cn" else "ch100")
    rec = ncu_record(kname, kfile, wl_rec)
    if rec is not None and "warp_inst_per_launch" in rec:
        rec_steps = float(rec.get("steps_per_launch", 1))
        roofline["inst_per_point"] = round(32.0 * float(rec["warp_inst_per_launch"]) /
                                           (float(rec["units"]) * N * rec_steps), 1)
        roofline["issue_active_pct_ncu"] = rec.get("issue_active_pct")
    if nsub > 1:
        # Many steps per launch: memory is touched once per launch and the kernel is
        # bound by instruction issue (double-float arithmetic on the FP32 pipe).  The
        # roof is the GPU's issue rate, one warp instruction per cycle per SM
        # sub-partition at the SM clock sampled during the run; the achieved rate is the
        # kernel's warp instructions (ncu, scaled per point and step from the committed
        # capture) over its CUDA-event time.  Both come from measurements.
        sms = torch.cuda.get_device_properties(dev_index).multi_processor_count
        clk = clocks.summary().get("sm_mhz") or 0.0
        peak_issue = sms * 4 * clk * 1e6
        achieved = None
        if rec is not None and "warp_inst_per_launch" in rec:
            per_ps = float(rec["warp_inst_per_launch"]) / (float(rec["units"]) * float(rec.get("steps_per_launch", 1)))
            achieved = per_ps * batch * nsub / (kernel_ms / 1e3)
        roofline = {"bound": "issue",
                    "achieved": None if achieved is None else round(achieved / 1e9, 2),
                    "peak": round(peak_issue / 1e9, 2) if peak_issue else None,
                    "unit": "G warp-instructions/s",
                    "frac": None if (achieved is None or not peak_issue) else round(achieved / peak_issue, 4),
                    "traffic": traffic,
                    "peak_source": f"{sms} SMs x 4 sub-partitions x 1 warp instruction per cycle x "
                                   f"the median SM clock sampled during the run ({clk} MHz)",
                    "kernel": kname, "kernel_ms": round(kernel_ms, 4),
                    "inst_per_point_step": None if rec is None or "warp_inst_per_launch" not in rec else
                    round(32.0 * float(rec["warp_inst_per_launch"]) /
                          (float(rec["units"]) * N * float(rec.get("steps_per_launch", 1))), 1),
                    "issue_active_pct_ncu": None if rec is None else rec.get("issue_active_pct"),
                    "instruction_source": f"ncu smsp__inst_executed.sum of {kname} on {wl_rec} "
                                          "(profiles/ncu_traffic.json)",
                    "steps_per_launch": nsub, "units_per_launch": batch * nsub,
                    "hbm_bytes_per_launch": alg_bytes}

    unit = "system-solves/s" if kind in ("shared", "persys", "tri") else "system-steps/s"
    res = {
        "metric": METRIC if args.workload == "shared" else f"{W['desc']} throughput",
        "value": value, "unit": unit, "n_gpus": dist.world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": W["dtype"],
        "data": "synthetic (seeded SplitMix64 counter-based generator)",
        "config": {"workload": W["desc"], "N": N, "batch_per_gpu": batch,
                   "global_batch": batch * dist.world, "time_steps_per_call": nsub,
                   "parallelism": f"replicas x{dist.world} "
                   "(batch split, no collective)", "variant": variant,
                   "l2": (("right-hand side restored from a pristine copy, then " if refresh else "") +
                          f"L2 flushed between timed steps ({2 * l2_bytes >> 20} MB write outside the "
                          "per-step events); time = sum of per-step events") if flush else
                         f"inputs larger than L2 (two {buf_bytes >> 20} MB buffers alternated)",
                   "solves_per_second_whole_job": value},
        "clocks": clocks.summary(), "gpu_launches": int(launches) * dist.world,
        "e2e": e2e, "roofline": roofline,
    }
    return res


def oracle_sample(W: dict):
    """The bounded sample of a workload that the CPU oracle is timed on (the same for
    the cpu_baseline of our arm and for the reference arm): S systems, one call of
    the oracle per step (one solve, or one time step for the stepping workloads)."""
    import numpy as np

    import oracle
    from implicit_pde_stepping_gb300 import inputs
    N, kind = W["N"], W["kind"]
    S = {"shared": 1024, "hyper": 256, "cn": 256, "ch": 64, "persys": 2048, "tri": 8192}[kind]
    S = max(1, min(S, (S * 1024) // N))   # long systems: about the same rows per step
    if kind == "shared":
        bands = inputs.hyper_bands(N, W["sigma"])
        F = inputs.rhs_uniform(N, S, seed=0)
        fn = lambda: oracle.batch_shared(bands, F, cyclic=W["cyclic"])  # noqa: E731
    elif kind == "hyper":
        F = inputs.fourier_initial(N, S)
        fn = lambda: oracle.batch_hyperdiffusion(F, W["sigma"], 1)  # noqa: E731
    elif kind == "ch":
        sigma, k2 = inputs.ch_params(N)
        F = inputs.ch_initial(N, S)
        fn = lambda: oracle.batch_ch(F, sigma, k2, 1)  # noqa: E731
    elif kind == "cn":
        F = inputs.fourier_initial(N, S)
        fn = lambda: oracle.batch_cn(F, W["sigma"], 1)  # noqa: E731
    elif kind == "tri":
        npdt = np.float64 if W["dtype"] == "f64" else np.float32
        a, b, c = inputs.tri_bands(N, S, dtype=npdt)
        F = inputs.rhs_uniform(N, S).astype(npdt)
        fn = lambda: oracle.batch_tri(a, b, c, F)  # noqa: E731
    else:
        npdt = np.float64 if W["dtype"] == "f64" else np.float32
        a, b, c, d, e = inputs.persys_bands(N, S, dtype=npdt)
        F = inputs.rhs_uniform(N, S).astype(npdt)
        fn = lambda: oracle.batch_persys(a, b, c, d, e, F)  # noqa: E731
    unit = "system-solves/s" if kind in ("shared", "persys", "tri") else "system-steps/s"
    return S, fn, unit


def time_oracle(W: dict, seconds: float):
    """Oracle rate (systems per second) on this process's OpenMP threads."""
    import oracle
    S, fn, unit = oracle_sample(W)
    fn()
    reps, t0 = 0, time.perf_counter()
    while True:
        fn()
        reps += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    return {"value": S * reps / el, "unit": unit, "cores": oracle.num_threads(), "systems": S,
            "reps": reps, "seconds": round(el, 2)}


def run_cpu_baseline(W: dict, seconds: float, workload: str):
    """The oracle as it stands, on this host's cores (OpenMP over systems, the pages'
    parallel baseline) and on one core (their serial baseline), same sample."""
    omp = time_oracle(W, seconds)
    single = None
    try:
        # one thread: a child interpreter with OMP_NUM_THREADS=1 (the oracle reads it
        # when its OpenMP runtime starts)
        env = dict(os.environ, OMP_NUM_THREADS="1")
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-child", workload,
                            "--cpu-seconds", str(max(2.0, seconds / 2))],
                           capture_output=True, text=True, env=env, timeout=600)
        if r.returncode == 0:
            single = json.loads(r.stdout.strip().splitlines()[-1])
    except (OSError, ValueError, subprocess.SubprocessError, IndexError):
        single = None
    sample = f"{omp['systems']} systems of the workload (N={W['N']}) per call"
    return {"value": omp["value"], "unit": omp["unit"], "cores": omp["cores"], "kind": "oracle",
            "sample": sample + f" x {omp['reps']} calls, {omp['seconds']} s",
            "single_thread": None if single is None else
            {"value": single["value"], "unit": single["unit"], "cores": single["cores"],
             "sample": sample + f" x {single['reps']} calls, {single['seconds']} s"}}


def run_reference(args, W: dict, dist: Dist):
    """Reference arm: the CPU oracle as it stands, timed on this host's cores on the
    same sample as our arm's cpu_baseline."""
    import oracle
    S, fn, unit = oracle_sample(W)
    for _ in range(args.warmup):
        fn()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        fn()
    el = time.perf_counter() - t0
    value = S * args.steps / el
    sample = f"{S} systems of the workload (N={W['N']}) per step"
    return {
        "impl": "reference", "metric": METRIC if args.workload == "shared" else
        f"{W['desc']} throughput", "value": value, "unit": unit, "n_gpus": dist.world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": W["dtype"],
        "data": "synthetic (seeded SplitMix64 counter-based generator)",
        "config": {"workload": W["desc"], "N": W["N"], "sample_systems_per_step": S},
        "cpu_baseline": {"value": value, "unit": unit, "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="shared")
    from implicit_pde_stepping_gb300.pent import VARIANTS
    ap.add_argument("--variant", default="auto", choices=sorted(VARIANTS))
    ap.add_argument("--batch", type=int, default=0, help="override the per-GPU batch")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-chunks", type=int, default=0,
                    help="blocks of systems the host-buffer solve pipelines (shared workloads; 0: "
                         "the library's choice)")
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--cpu-child", choices=sorted(WORKLOADS), default=None,
                    help=argparse.SUPPRESS)   # internal: time the oracle in this process and exit
    args = ap.parse_args(argv)
    if args.cpu_child:
        print(json.dumps(time_oracle(WORKLOADS[args.cpu_child], args.cpu_seconds)), flush=True)
        return 0
    if args.warmup < 3:
        log("warning: fewer than 3 warm-up steps")
    W = WORKLOADS[args.workload]
    dist = Dist(args.gpus)
    try:
        if args.impl == "reference":
            if dist.rank == 0:
                print(json.dumps(run_reference(args, W, dist)), flush=True)
            return 0
        from implicit_pde_stepping_gb300 import build as b
        if dist.rank == 0:
            b.build()
        dist.barrier()
        res = run_ours(args, W, dist)
        if dist.rank == 0:
            if dist.world == 1 and not args.no_cpu_baseline:
                res["cpu_baseline"] = run_cpu_baseline(W, args.cpu_seconds, args.workload)
            else:
                res["cpu_baseline"] = None
            print(json.dumps(res), flush=True)
        return 0
    finally:
        dist.close()


if __name__ == "__main__":
    sys.exit(main())
