#!/usr/bin/env python
"""Benchmark of the sharded RS+AdamW+AG step (FSDP / ZeRO-3 per-step pass) on GB300.

One step = the whole hot path over one synthetic batch of gradients, by
default as one fsdp_sharded_step launch over every fully_shard group:
  - the reduce-scatter: N virtual ranks' bf16 gradients summed in fp32 in
    rank order and divided by N;
  - AdamW on every rank's shard of the fp32 master/moments, bf16 shards
    written;
  - the all-gather + unpack: the new values written into full per-parameter
    bf16 tensors (n_out replicas, default 1).
--step-kind two_calls runs the same step as fsdp_reduce_scatter_adamw then
fsdp_all_gather_unpack (two launches, bit-identical results).
Default workload: the 1.2B Llama-shaped model (24 layers, hidden 2048, FFN
5632, vocab 32000, untied embeddings) with N = 8 virtual ranks, FSDP2
per-parameter dim-0 layout, 24 block groups + 1 root group, 1,364,297,728
parameters.  Every buffer is resident in HBM; the 60 GB a step moves are far
larger than L2, so no flush is needed between steps.

Prints ONE JSON line (rank 0).  `--impl reference` times the CPU oracle
instead, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "sharded RS+AdamW+AG step: params/s and HBM GB/s vs GB300 peak (1 GPU)"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--workload", default="llama_1b2",
                    choices=["llama_1b2", "llama_block_4096", "probe", "tiny_mlp"],
                    help="step mode: the timed model; rows mode: the model of the llama rows "
                         "(llama_1b2, or probe for a few-GB profiling case)")
    ap.add_argument("--n-out", type=int, default=1, help="all-gather replicas (1 or N)")
    ap.add_argument("--e2e-steps", type=int, default=8,
                    help="timed end-to-end steps (each moves 24.6 GB over the host link; "
                         "single steps vary by up to 20 %% on a shared host)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--mode", choices=["step", "rows"], default="step",
                    help="step: the one-line headline; rows: one JSON line per hot-path row")
    ap.add_argument("--rows", default="all",
                    help="rows mode: comma list of llama,block4096,tiny,awkward,awkward_large,"
                         "awkward_n16,world_sizes,ddp (default all; awkward_large: only the large "
                         "awkward sets; awkward_n16: the 1-D awkward set at N = 16 and 800 "
                         "per-parameter-layout params in one group; world_sizes: the 1.2B model "
                         "at N = 2, 4, 16 and 32)")
    ap.add_argument("--step-kind", default="fused", choices=["two_calls", "fused", "copy_in"],
                    help="timed step: the one-pass fsdp_sharded_step from packed gradients "
                         "(default), RS+AdamW then all-gather as two calls, or the one pass "
                         "reading N per-parameter gradient sets (fused copy-in)")
    ap.add_argument("--ddp-large", type=int, default=600,
                    help="rows mode: number of 4M-element DDP tensors (600 = the full list)")
    ap.add_argument("--awkward-scale", type=float, default=1.0,
                    help="rows mode: scale of the large awkward sets (1.0: 218M and 134M params; "
                         "0.25 keeps a profiling capture to a few GB)")
    return ap.parse_args()


def make_workload(name: str) -> W.ParamSet:
    if name == "llama_1b2":
        return W.llama_1b2()
    if name == "llama_block_4096":
        return W.llama_block_4096()
    if name == "probe":  # one block + small root: a few GB, larger than L2 (profiling case)
        return W.llama_1b2(layers=1, vocab=4096)
    return W.tiny_mlp()


def step_bytes(N: int, total: int, unpadded: int, n_out: int) -> dict:
    """Algorithmic bytes: RS+AdamW reads N grads (2 B) + master/m/v (12 B), writes
    master/m/v (12 B) + the bf16 shard (2 B) for every packed element; the
    all-gather reads each parameter element's shard (2 B) and writes n_out copies."""
    rs = (2 * N + 26) * total
    ag = (2 + 2 * n_out) * unpadded
    return {"rs_adamw": rs, "all_gather": ag, "step": rs + ag}


def workload_config(ps: W.ParamSet, info, n_out: int) -> dict:
    return {"workload": f"{ps.description}; N={ps.world_size} virtual ranks",
            "params": int(info["unpadded_numel"]), "packed_numel": int(info["total_numel"]),
            "world_size": ps.world_size, "groups": len(ps.groups), "tensors": ps.num_params,
            "layout": W.LAYOUT_NAMES[ps.layout], "n_out": n_out,
            "storage": "bf16 grads/params, fp32 master/exp_avg/exp_avg_sq",
            "adamw": {k: v for k, v in W.adamw_hparams().items() if k != "step"},
            "l2": "no flush: the bytes every step moves (>= 60 GB at the default workload) exceed L2"}


def ncu_traffic(kernel: str, units: int):
    """DRAM bytes per launch of `kernel` from the committed ncu capture
    (per-element read + write bytes x units), or None if none was taken."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)[kernel]
        return (d["dram_read_bytes_per_element"] + d["dram_write_bytes_per_element"]) * units
    except Exception:
        return None


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, local_rank: int, enabled: bool = True):
        self.proc = None
        self.path = None
        if not enabled:
            return
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        dev = str(local_rank)
        if vis:
            parts = [p.strip() for p in vis.split(",") if p.strip()]
            if local_rank < len(parts):
                dev = parts[local_rank]
        self.path = f"/tmp/ss_clocks_{os.getpid()}.csv"
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", dev], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        try:
            with open(self.path) as f:
                for line in f:
                    cols = [c.strip() for c in line.split(",")]
                    if len(cols) < 9:
                        continue
                    try:
                        sm.append(float(cols[1]))
                        smax.append(float(cols[2]))
                        power.append(float(cols[3]))
                    except ValueError:
                        continue
                    for nm, val in zip(names, cols[5:9]):
                        if val.lower() == "active":
                            reasons.add(nm)
            os.unlink(self.path)
        except Exception:
            return None
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}


# ---------------------------------------------------------------------------
# distributed plumbing (replicas: no data-path collective)
# ---------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_init(world: int, local: int):
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        return dist
    torch.cuda.set_device(local)
    return None


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(dist, x: float) -> float:
    """Largest value over ranks (the slowest replica's time)."""
    if dist is None:
        return x
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def host_stall(steps_ms) -> bool:
    """True if one timed step took over 5x the median step and more than 1 ms
    above it: the signature of a host thread that stalled between launches
    while the GPU ran dry, not of the GPU work."""
    if not steps_ms:
        return False
    med = statistics.median(steps_ms)
    worst = max(steps_ms)
    return worst > 5 * med and worst - med > 1.0


def job_value(units_per_rank: int, steps: int, world: int, ms_max: float) -> float:
    """Whole-job throughput: the units every replica processed over the slowest
    replica's time (replicas each run the full workload: weak scaling)."""
    return units_per_rank * steps * world / (ms_max / 1e3)


# ---------------------------------------------------------------------------
# native arm
# ---------------------------------------------------------------------------

class Step:
    """Device buffers and the two C-ABI calls of one step."""

    def __init__(self, ss, ps: W.ParamSet, n_out: int):
        self.ss = ss
        self.ps = ps
        self.N = ps.world_size
        self.n_out = n_out
        d0, inner = ps.dim0_inner()
        eb = 2 if ps.dtype == torch.bfloat16 else 4
        self.plan = ss.fsdp_plan_create(ps.layout, self.N, eb, d0, inner, group_num_params=ps.groups)
        self.info = self.plan.info().as_dict()
        total = self.info["total_numel"]
        dev = "cuda"
        # parameters -> shards, fp32 state
        params = W.make_params(ps, device=dev)
        self.shards = torch.empty(total, dtype=ps.dtype, device=dev)
        ss.fsdp_pack(self.plan, params, self.shards)
        del params
        self.master = torch.empty(total, dtype=torch.float32, device=dev)
        self.m = torch.empty_like(self.master)
        self.v = torch.empty_like(self.master)
        ss.fsdp_init_master(self.plan, self.shards, self.master, self.m, self.v)
        # every rank's gradient, generated per parameter then packed (pads zero)
        self.grads = []
        for r, rank in enumerate(self._rank_grad_iter(dev)):
            buf = torch.empty(total, dtype=ps.dtype, device=dev)
            ss.fsdp_pack(self.plan, rank, buf)
            self.grads.append(buf)
            del rank
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        # outputs: n_out replicas, each one flat buffer with 16-byte aligned params
        numels = ps.numels()
        offs, pos = [], 0
        for n in numels:
            offs.append(pos)
            pos += (n + 7) // 8 * 8
        self.out_numel = pos
        self.out_flat = [torch.empty(pos, dtype=ps.dtype, device=dev) for _ in range(n_out)]
        self.outs = [o[off:off + n] for o in self.out_flat for off, n in zip(offs, numels)]
        self.out_offs = offs
        # pointer arrays marshalled once; the timed calls pass them straight through
        self._grads_arr = ss.ptr_array(self.grads)
        self._outs_arr = ss.ptr_array(self.outs)
        self.t = 0

    def _rank_grad_iter(self, dev):
        ps = self.ps
        g = torch.Generator(device=dev)
        g.manual_seed(ps.seed * 7919 + 17)
        for _ in range(self.N):
            yield [(torch.randn(n, generator=g, device=dev) * ps.grad_std).to(ps.dtype)
                   for n in ps.numels()]

    def next_hp(self):
        """AdamW hyper-parameters of the next optimizer step."""
        self.t += 1
        return self.ss.adamw_params(step=self.t, **{k: v for k, v in W.adamw_hparams().items()
                                                     if k != "step"})

    def rs_adamw(self, stream=None, group=-1, hp=None):
        """One fused reduce-scatter + AdamW call (every group, or one group with
        the step's shared hyper-parameters)."""
        if hp is None:
            hp = self.next_hp()
        self.ss.fsdp_reduce_scatter_adamw(self.plan, self._grads_arr, self.master, self.m, self.v,
                                          self.shards, hp, None, group, stream)

    def fused_step(self, stream=None, param_grads=None, group=-1, hp=None):
        """fsdp_sharded_step: RS+AdamW with the all-gather written in the same pass
        (every group, or one group with the step's shared hyper-parameters)."""
        if hp is None:
            hp = self.next_hp()
        if param_grads is None:
            self.ss.fsdp_sharded_step(self.plan, self.master, self.m, self.v, self.shards, hp,
                                      rank_grads=self._grads_arr, params_out=self._outs_arr,
                                      n_out=self.n_out, group=group, stream=stream)
        else:
            self.ss.fsdp_sharded_step(self.plan, self.master, self.m, self.v, self.shards, hp,
                                      rank_param_grads=param_grads, params_out=self._outs_arr,
                                      n_out=self.n_out, group=group, stream=stream)

    def all_gather(self, stream=None, group=-1):
        self.ss.fsdp_all_gather_unpack(self.plan, self.shards, self._outs_arr, self.n_out, group,
                                       stream)


def run_native(args, world, rank, local, dist):
    import __graft_entry__
    __graft_entry__.build()
    import sharded_state_gb300 as ss
    ps = make_workload(args.workload)
    st = Step(ss, ps, args.n_out)
    P = st.info["unpadded_numel"]
    total = st.info["total_numel"]
    N = st.N
    by = step_bytes(N, total, P, args.n_out)
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream

    fused = args.step_kind in ("fused", "copy_in")
    # the fused copy-in reads N per-parameter gradient sets instead of the
    # packed rank buffers
    param_grads = None
    if args.step_kind == "copy_in":
        param_grads = ss.ptr_array([g for rank in st._rank_grad_iter("cuda") for g in rank])
    for _ in range(max(args.warmup, 0)):
        if fused:
            st.fused_step(sp, param_grads=param_grads)
        else:
            st.rs_adamw(sp)
            st.all_gather(sp)
    torch.cuda.synchronize()

    K = args.steps

    def timed_region():
        """Exactly K steps between a barrier + synchronize on both sides."""
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        barrier(dist)
        torch.cuda.synchronize()
        clocks = ClockSampler(local, enabled=not args.no_clocks)
        time.sleep(0.3 if clocks.proc else 0)  # let the sampler start
        launches0 = ss.ss_launch_count()
        e0.record(stream)
        for k in range(K):
            ev[k][0].record(stream)
            if fused:
                st.fused_step(sp, param_grads=param_grads)
            else:
                st.rs_adamw(sp)
            ev[k][1].record(stream)
            if not fused:
                st.all_gather(sp)
            ev[k][2].record(stream)
        e1.record(stream)
        torch.cuda.synchronize()
        launches = ss.ss_launch_count() - launches0
        clk = clocks.stop()
        barrier(dist)
        return (e0.elapsed_time(e1), [ev[k][0].elapsed_time(ev[k][1]) for k in range(K)],
                [ev[k][1].elapsed_time(ev[k][2]) for k in range(K)], launches, clk)

    # A host thread that stalls between two launches lets the GPU drain, and
    # the stall lands inside one step's events.  If any rank saw a step over 5x
    # the median (and > 1 ms above it), every rank times the K steps again, at
    # most twice; the line reports how many times.
    retimed = 0
    while True:
        ms, rs_ms, ag_ms, launches, clk = timed_region()
        stalled = host_stall([a + b for a, b in zip(rs_ms, ag_ms)])
        if retimed >= 2 or max_over_ranks(dist, 1.0 if stalled else 0.0) == 0.0:
            break
        retimed += 1
    ms_max = max_over_ranks(dist, ms)
    value = job_value(P, K, world, ms_max)
    if fused:  # one kernel: 2N + 26 bytes per packed element + 2 * n_out per parameter
        by = {"rs_adamw": (2 * N + 26) * total + 2 * args.n_out * P, "all_gather": 0,
              "step": (2 * N + 26) * total + 2 * args.n_out * P}
    hbm = by["step"] * K / (ms / 1e3) / 1e9

    peak, peak_kind = measured_peak()
    rs_avg = sum(rs_ms) / K
    rs_gbs = by["rs_adamw"] / (rs_avg / 1e3) / 1e9
    ag_avg = sum(ag_ms) / K
    ag_gbs = by["all_gather"] / (ag_avg / 1e3) / 1e9 if by["all_gather"] else 0.0

    out = {"metric": METRIC, "value": value, "unit": "params/s", "n_gpus": world, "steps": K,
           "warmup": args.warmup, "ms_per_step": ms_max / K, "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
           "impl": "native", "config": dict(workload_config(ps, st.info, args.n_out),
                                            step_kind=args.step_kind),
           "hbm_gbs": hbm, "bytes_per_step": by["step"],
           "frac_of_measured_peak": hbm / peak, "frac_of_nominal_8tbs": hbm / NOMINAL_HBM_GBS,
           "kernels": ({"one_pass_step": {"ms": rs_avg, "ms_min": min(rs_ms), "gbs": rs_gbs,
                                          "bytes": by["rs_adamw"]}} if fused else
                       {"rs_adamw": {"ms": rs_avg, "ms_min": min(rs_ms), "gbs": rs_gbs,
                                     "bytes": by["rs_adamw"]},
                        "all_gather_unpack": {"ms": ag_avg, "ms_min": min(ag_ms), "gbs": ag_gbs,
                                              "bytes": by["all_gather"]}}),
           "roofline": {"bound": "hbm",
                        "kernel": ("fused_step_flat_rounds_kernel (one-pass RS+AdamW+AG, "
                                   "fused copy-in)" if param_grads is not None else
                                   "fused_step_flat_kernel (one-pass RS+AdamW+AG)" if fused
                                   else "rs_adamw_bf16_kernel"),
                        "achieved": rs_gbs, "peak": peak,
                        "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"
                        if peak_kind == "measured" else "fallback 6.8 TB/s",
                        "unit": "GB/s", "frac": rs_gbs / peak,
                        "traffic": None if N != 8 or (fused and args.n_out != 1) else
                        ncu_traffic("fused_step_flat_rounds_kernel<8>" if param_grads is not None
                                    else "fused_step_flat_kernel<8>" if fused
                                    else "rs_adamw_bf16_kernel<8,1,0,1,0>", total),
                        "traffic_source": "ncu capture per element x elements per launch "
                                          "(profiles/ncu_traffic.json)",
                        "per_unit_bytes": 2 * N + 26 + (2 * args.n_out if fused else 0),
                        "units_per_launch": total,
                        # how many times the K steps were timed again after a
                        # host stall (0: this is the first timing)
                        "retimed": retimed},
           "gpu_launches": launches, "clocks": clk, "retimed": retimed}
    if retimed:
        out["retime_reason"] = ("a step in an earlier timing took over 5x the median step: a host "
                                "stall between launches; the K steps were timed again")

    # e2e: the same step through the C ABI with host buffers
    if not args.no_e2e:
        out["e2e"] = run_e2e(st, args, stream, dist)
    # CPU oracle baseline (rank 0, N=1)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(st, ps, args)
    if rank == 0:
        print(json.dumps(out), flush=True)


def run_e2e(st: Step, args, stream, dist) -> dict:
    """The same step end to end through the C ABI with host buffers.  Per step:
    every rank's gradient buffer comes in from pinned host memory, the two
    calls run, and the gathered parameters go back to pinned host memory.  The
    work is pipelined group by group on three streams, as FSDP overlaps
    communication with compute: group g's reduce-scatter + AdamW + all-gather
    starts once its gradients have arrived, while group g+1's are still in
    flight, and group g's parameters leave while later groups compute."""
    import sharded_state_gb300 as ss
    total = st.info["total_numel"]
    N = st.N
    need = N * total * 2 + st.n_out * st.out_numel * 2
    try:
        phys = os.sysconf("SC_PHYS_PAGES") * os.sysconf("SC_PAGE_SIZE")
    except Exception:
        phys = 0
    # every rank on this node pins its own copy: keep all of them under half the RAM
    local_ranks = int(os.environ.get("LOCAL_WORLD_SIZE", "1"))
    if phys and need * local_ranks * 2 > phys:
        return {"value": None, "unit": "params/s",
                "skipped": f"needs {need / 1e9:.1f} GB pinned host per rank x {local_ranks} ranks"}
    host_g, host_out, err = [], [], None
    try:
        for r in range(N):
            h = torch.empty(total, dtype=st.ps.dtype, pin_memory=True)
            h.copy_(st.grads[r])
            host_g.append(h)
        host_out = [torch.empty(st.out_numel, dtype=st.ps.dtype, pin_memory=True)
                    for _ in range(st.n_out)]
    except RuntimeError as e:  # pinned allocation refused
        err = str(e).splitlines()[0][:120] if str(e) else "RuntimeError"
    # every rank leaves together if any rank could not pin its buffers, so no
    # rank is left waiting at the timed region's barrier
    if max_over_ranks(dist, 1.0 if err else 0.0) > 0.0:
        del host_g, host_out
        return {"value": None, "unit": "params/s",
                "skipped": f"pinned host allocation failed on a rank: {err or 'another rank'}"}
    G = len(st.ps.groups)
    groups = [ss.fsdp_plan_group(st.plan, g) for g in range(G)]
    numels = st.ps.numels()
    out_rng = []
    for grp in groups:
        a, b = grp["first_param"], grp["first_param"] + grp["num_params"]
        lo = st.out_offs[a] if b > a else 0
        hi = st.out_offs[b - 1] + (numels[b - 1] + 7) // 8 * 8 if b > a else 0
        out_rng.append((lo, hi))
    h2d = torch.cuda.Stream()
    d2h = torch.cuda.Stream()
    sp = stream.cuda_stream
    torch.cuda.synchronize()
    K = max(args.e2e_steps, 1)
    P = st.info["unpadded_numel"]

    order = list(range(G))  # registration order (root-first and largest-in-the-middle measured slower)

    def one_step():
        hp = st.next_hp()
        ev_in = [torch.cuda.Event() for _ in range(G)]
        ev_done = [torch.cuda.Event() for _ in range(G)]
        h2d.wait_stream(stream)
        with torch.cuda.stream(h2d):
            for g in order:
                grp = groups[g]
                lo, hi = grp["base"], grp["base"] + N * grp["shard_numel"]
                for r in range(N):
                    st.grads[r][lo:hi].copy_(host_g[r][lo:hi], non_blocking=True)
                ev_in[g].record(h2d)
        for g in order:
            stream.wait_event(ev_in[g])
            if args.step_kind != "two_calls":  # the copy-in kind, too, from packed buffers here
                st.fused_step(sp, group=g, hp=hp)
            else:
                st.rs_adamw(sp, group=g, hp=hp)
                st.all_gather(sp, group=g)
            ev_done[g].record(stream)
            d2h.wait_event(ev_done[g])
            lo, hi = out_rng[g]
            with torch.cuda.stream(d2h):
                for j in range(st.n_out):
                    host_out[j][lo:hi].copy_(st.out_flat[j][lo:hi], non_blocking=True)
        stream.wait_stream(d2h)

    for _ in range(2):  # untimed passes: the first host-to-device pass runs up to 25 % slow
        one_step()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    barrier(dist)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(K):
        one_step()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(dist, e0.elapsed_time(e1))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    res = {"value": job_value(P, K, world, ms), "unit": "params/s", "steps": K,
           "ms_per_step": ms / K, "h2d_bytes_per_step": N * total * 2,
           "d2h_bytes_per_step": st.n_out * st.out_numel * 2,
           "pipeline": f"{G} groups on 3 streams (H2D / compute / D2H)"}
    del host_g, host_out
    return res


# ---------------------------------------------------------------------------
# CPU oracle: baseline leg and reference arm
# ---------------------------------------------------------------------------

def _host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def _host_free_bytes() -> int:
    try:
        return os.sysconf("SC_AVPHYS_PAGES") * os.sysconf("SC_PAGE_SIZE")
    except (ValueError, OSError, AttributeError):
        return 0


def _oracle_group0_from_step(st: Step) -> dict:
    """Group 0 of a step's device buffers, copied to the host, in the form
    _oracle_step takes (the rows' per-row oracle timings)."""
    import sharded_state_gb300 as ss
    grp = ss.fsdp_plan_group(st.plan, 0)
    base, span = grp["base"], st.N * grp["shard_numel"]
    a, b = grp["first_param"], grp["first_param"] + grp["num_params"]
    sl = slice(base, base + span)
    to_u16 = lambda t: t[sl].cpu().view(torch.int16).numpy().view(np.uint16).copy()
    g0 = {"grads": [to_u16(g) for g in st.grads], "master": st.master[sl].cpu().numpy().copy(),
          "m": st.m[sl].cpu().numpy().copy(), "v": st.v[sl].cpu().numpy().copy(),
          "shard_numel": grp["shard_numel"], "params": a, "params_end": b, "span": span}
    return {"groups": [g0], "whole": False, "params": int(sum(st.ps.numels()[a:b]))}


def _oracle_config(ps: W.ParamSet) -> dict:
    """The whole workload on the host for the oracle: every group with its own
    fp32 master (the widened bf16 parameters), exp_avg and exp_avg_sq, so one
    oracle step touches every parameter of the model once.  Inputs are drawn
    once per distinct group shape and shared by the groups of that shape (the
    24 blocks of the Llama-shaped model share one draw): the oracle's work and
    bytes per step are the whole model's, only the random values repeat.  If
    the state would take more than half the host's free memory, only the
    first group is kept, and `whole` says so."""
    import oracle
    d0, inner = ps.dim0_inner()
    N = ps.world_size
    spans, first = [], 0
    for cnt in ps.groups:
        lay = oracle.layout(ps.layout, N, 2, d0[first:first + cnt], inner[first:first + cnt])
        spans.append((first, first + cnt, lay["shard_numel"], lay["total_numel"]))
        first += cnt
    state_bytes = 14 * sum(sp[3] for sp in spans)
    whole = state_bytes <= _host_free_bytes() // 2
    if not whole:
        spans = spans[:1]
    gen = torch.Generator().manual_seed(ps.seed)
    drawn, groups = {}, []
    for a, b, shard, span in spans:
        key = (tuple(d0[a:b]), tuple(inner[a:b]))
        if key not in drawn:
            params = (torch.randn(span, generator=gen) * ps.param_std).to(ps.dtype)
            grads = [(torch.randn(span, generator=gen) * ps.grad_std).to(ps.dtype)
                     .view(torch.int16).numpy().view(np.uint16) for _ in range(N)]
            drawn[key] = (params.float().numpy(), grads)
        master0, grads = drawn[key]
        groups.append({"params": a, "params_end": b, "shard_numel": shard, "span": span,
                       "grads": grads, "master": master0.copy(), "m": np.zeros(span, np.float32),
                       "v": np.zeros(span, np.float32)})
    P = sum(int(sum(ps.numels()[g["params"]:g["params_end"]])) for g in groups)
    return {"groups": groups, "whole": whole, "params": P}


def _oracle_step(ps: W.ParamSet, cfg: dict, t: int, groups=None) -> int:
    """One oracle step over the kept groups: reduce-scatter + AdamW of every
    rank's shard, then the all-gather + unpack.  Returns the parameters it
    updated."""
    import oracle
    hp = W.adamw_hparams(t)
    d0, inner = ps.dim0_inner()
    done = 0
    for g in (cfg["groups"] if groups is None else groups):
        a, b = g["params"], g["params_end"]
        shards, _ = oracle.reduce_scatter_adamw(
            ps.world_size, g["shard_numel"], g["grads"], g["master"], g["m"], g["v"],
            **{k: hp[k] for k in ("lr", "beta1", "beta2", "eps", "weight_decay", "step")})
        oracle.all_gather_unpack(ps.layout, ps.world_size, 2, d0[a:b], inner[a:b], shards)
        done += int(sum(ps.numels()[a:b]))
    return done


def _oracle_sample_text(ps: W.ParamSet, cfg: dict) -> str:
    if cfg["whole"]:
        ng = len(cfg["groups"])
        return (f"the whole workload per step: {'all %d groups' % ng if ng > 1 else 'its one group'}, "
                f"{cfg['params']:,} params, each group with its own optimizer state; "
                f"inputs drawn on the host once per group shape")
    return (f"group 0 only ({cfg['params']:,} params) per step: the whole workload's state "
            f"would take more than half the host's free memory")


def cpu_baseline(st: Step, ps: W.ParamSet, args) -> dict:
    """The oracle as written on the host's cores: whole-workload steps for
    args.cpu_seconds (at least one), then the definitional single-thread run
    on group 0 of the same inputs for half that time."""
    import oracle
    cores = _host_cores()
    oracle.set_threads(cores)
    used = cores if oracle.has_openmp() else 1
    cfg = _oracle_config(ps)
    _oracle_step(ps, cfg, 999)  # untimed: touches the freshly allocated host memory once
    t0 = time.perf_counter()
    reps, params = 0, 0
    while True:
        params += _oracle_step(ps, cfg, 1000 + reps)
        reps += 1
        if time.perf_counter() - t0 >= args.cpu_seconds:
            break
    dt = time.perf_counter() - t0
    # the definitional oracle on one thread, on group 0 (half the budget)
    oracle.set_threads(1)
    g0 = cfg["groups"][:1]
    t1 = time.perf_counter()
    reps1, params1 = 0, 0
    while True:
        params1 += _oracle_step(ps, cfg, 5000 + reps1, groups=g0)
        reps1 += 1
        if time.perf_counter() - t1 >= args.cpu_seconds / 2:
            break
    dt1 = time.perf_counter() - t1
    oracle.set_threads(cores)
    single = params1 / dt1
    return {"value": params / dt, "unit": "params/s", "cores": used, "kind": "oracle",
            "sample": f"{_oracle_sample_text(ps, cfg)}; {reps} oracle RS+AdamW+AG steps in "
                      f"{dt:.1f} s on {used} threads. One thread (the definitional oracle): "
                      f"{single:.4g} params/s on group 0 ({params1 // reps1:,} params), "
                      f"{reps1} steps in {dt1:.1f} s",
            "single_thread": {"value": single, "unit": "params/s", "cores": 1,
                              "sample": f"group 0, {reps1} steps, {dt1:.1f} s"}}


# Most seconds the reference arm's warm-up and timed steps together take.
REFERENCE_BUDGET_S = 240.0


def run_reference(args, world, rank):
    if rank != 0:
        return
    import oracle
    ps = make_workload(args.workload)
    cores = _host_cores()
    oracle.set_threads(cores)
    used = cores if oracle.has_openmp() else 1
    cfg = _oracle_config(ps)
    groups = cfg["groups"]
    note = ""
    for w in range(max(args.warmup, 0)):
        t1 = time.perf_counter()
        _oracle_step(ps, cfg, w + 1, groups)
        if w == 0:
            # keep the whole run within REFERENCE_BUDGET_S: a step over fewer
            # groups if the whole workload would take longer
            step_s = time.perf_counter() - t1
            budget = REFERENCE_BUDGET_S / max(args.steps + args.warmup - 1, 1)
            if step_s > budget and len(groups) > 1:
                keep = max(1, int(len(groups) * budget / step_s))
                groups = groups[:keep]
                kept = sum(int(sum(ps.numels()[g["params"]:g["params_end"]])) for g in groups)
                note = (f"the first {keep} of {len(cfg['groups'])} groups per step ({kept:,} params), "
                        f"each with its own optimizer state: the whole workload's "
                        f"{args.warmup + args.steps} steps would take about "
                        f"{step_s * (args.warmup + args.steps):.0f} s")
    t0 = time.perf_counter()
    params = 0
    for k in range(args.steps):
        params += _oracle_step(ps, cfg, args.warmup + k + 1, groups)
    dt = time.perf_counter() - t0
    info = {"unpadded_numel": ps.total_unpadded(), "total_numel": _packed_numel(ps)}
    value = params / dt
    sample = f"{note or _oracle_sample_text(ps, cfg)}; {args.steps} timed oracle RS+AdamW+AG steps"
    out = {"metric": METRIC, "value": value, "unit": "params/s", "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": dt / max(args.steps, 1) * 1e3, "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
           "impl": "reference",
           "config": dict(workload_config(ps, info, args.n_out), step_kind=args.step_kind),
           "cpu_baseline": {"value": value, "unit": "params/s", "cores": used, "kind": "oracle",
                            "sample": sample},
           "e2e": {"value": value, "unit": "params/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def _packed_numel(ps: W.ParamSet) -> int:
    """Elements of one packed buffer of the workload's plan (the oracle's layout)."""
    import oracle
    d0, inner = ps.dim0_inner()
    total, first = 0, 0
    for cnt in ps.groups:
        total += oracle.layout(ps.layout, ps.world_size, 2, d0[first:first + cnt],
                               inner[first:first + cnt])["total_numel"]
        first += cnt
    return total


# ---------------------------------------------------------------------------
# per-row measurements (--mode rows): every hot-path row on its own workload
# ---------------------------------------------------------------------------

# per-iteration times of the latest _time_stream call (its row reports their median)
_LAST_TIMES: list = []


def _time_stream(fn, K: int, warmup: int = 3):
    """Mean / min CUDA-event time (ms) of fn() on the current stream."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    ts = []
    for _ in range(K):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        ts.append((a, b))
    torch.cuda.synchronize()
    ms = [a.elapsed_time(b) for a, b in ts]
    _LAST_TIMES[:] = ms
    return sum(ms) / len(ms), min(ms)


def _time_back_to_back(fn, steps: int = 2000, reps: int = 5, warmup: int = 50):
    """Per-call time (ms) of fn() issued `steps` times back to back between two
    CUDA events on the current stream, as the median and min over `reps`
    batches: the rate a loop of launch-bound steps runs at (host issue and GPU
    work overlap; an event per call would add its own host time to every
    call)."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    per = []
    for _ in range(reps):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        per.append(a.elapsed_time(b) / steps)
    _LAST_TIMES[:] = per
    return statistics.median(per), min(per)


def _time_cpu(fn, seconds: float):
    t0 = time.perf_counter()
    reps = 0
    while True:
        fn()
        reps += 1
        if time.perf_counter() - t0 >= seconds:
            break
    return (time.perf_counter() - t0) / reps, reps


def _oracle_pair(fn, seconds: float, units: int, unit: str, sample: str) -> dict:
    """A row's oracle baseline: fn (the oracle on `units` units of the row's
    work) timed on all the host's threads, then on one thread for half as
    long; the all-thread figure is the row's cpu_baseline value."""
    import oracle
    cores = _host_cores()
    used = cores if oracle.has_openmp() else 1
    oracle.set_threads(cores)
    t_all, reps = _time_cpu(fn, seconds)
    oracle.set_threads(1)
    try:
        t_one, reps1 = _time_cpu(fn, seconds / 2)
    finally:
        oracle.set_threads(cores)
    return {"value": units / t_all, "unit": unit, "cores": used, "kind": "oracle",
            "sample": f"{sample}, {reps} reps; one thread: {units / t_one:.4g} {unit}",
            "single_thread": {"value": units / t_one, "unit": unit, "cores": 1, "reps": reps1}}


def _row(name, unit_count, unit, ms, ms_min, nbytes, peak, cpu=None, extra=None):
    """One row: value and roofline from the median of the timed calls (a host
    stall between two launches lands in one call's events and would move the
    mean); the mean (`ms`) and the minimum beside it."""
    med = statistics.median(_LAST_TIMES) if _LAST_TIMES else ms
    gbs = nbytes / (med / 1e3) / 1e9
    d = {"row": name, "value": unit_count / (med / 1e3), "unit": unit, "ms": ms, "ms_min": ms_min,
         "ms_median": med,
         "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s",
                      "frac": gbs / peak, "algorithmic_bytes": nbytes, "from": "median"}}
    if cpu is not None:
        d["cpu_baseline"] = cpu
    if extra:
        d.update(extra)
    print(json.dumps(d), flush=True)


def run_rows(args):
    import __graft_entry__
    __graft_entry__.build()
    import oracle
    import sharded_state_gb300 as ss
    torch.cuda.set_device(0)
    peak, _ = measured_peak()
    cores = _host_cores()
    oracle.set_threads(cores)
    used = cores if oracle.has_openmp() else 1
    K = max(args.steps, 5)
    bits = lambda t: t.reshape(-1).cpu().view(torch.int16).numpy().view(np.uint16).copy()
    want = set(args.rows.split(",")) if args.rows != "all" else {"llama", "block4096", "tiny",
                                                                 "awkward", "awkward_n16",
                                                                 "world_sizes", "ddp"}
    if "llama" in want:
        _rows_llama(args, ss, oracle, peak, used, K, bits)
    if "block4096" in want:
        _rows_block4096(ss, peak, K, args.cpu_seconds)
    if want & {"tiny", "awkward", "awkward_large"}:
        _rows_small(ss, peak, want, args.awkward_scale, args.cpu_seconds)
    if "awkward_n16" in want:
        _rows_awkward_wide(ss, peak, args.awkward_scale)
    if "world_sizes" in want:
        _rows_world_sizes(ss, peak)
    if "ddp" in want:
        _rows_ddp(args, ss, oracle, peak, used, K, bits)


def _rows_llama(args, ss, oracle, peak, used, K, bits):
    # -- a1/a2/a3/a4 on the 1.2B model (or a smaller Llama for profiling) ---
    ps = make_workload(args.workload) if args.workload != "llama_1b2" else W.llama_1b2()
    tag = "1.2B" if args.workload == "llama_1b2" else args.workload
    d0_, inner_ = ps.dim0_inner()
    t0 = time.perf_counter()
    for _ in range(5):
        plan_ = ss.fsdp_plan_create(ps.layout, ps.world_size, 2, d0_, inner_,
                                    group_num_params=ps.groups)
        plan_.destroy()
    t_plan = (time.perf_counter() - t0) / 5
    t_cpu, reps = _time_cpu(lambda: [oracle.layout(ps.layout, ps.world_size, 2, d0_[a:a + g],
                                                   inner_[a:a + g])
                                     for a, g in zip(np.cumsum([0] + ps.groups[:-1]), ps.groups)],
                            1.0)
    print(json.dumps({"row": "a1 plan: layout, segment and tile tables + device upload "
                             f"({tag} model, {ps.num_params} params, {len(ps.groups)} groups, "
                             f"N={ps.world_size})",
                      "value": 1.0 / t_plan, "unit": "plans/s", "ms": t_plan * 1e3,
                      "host_only": "runs once per model; not on the per-step path",
                      "cpu_baseline": {"value": 1.0 / t_cpu, "unit": "layouts/s", "cores": 1,
                                       "kind": "oracle", "sample": f"the {len(ps.groups)} group layouts, {reps} reps"}}),
          flush=True)
    st = Step(ss, ps, 1)
    P, total, N = st.info["unpadded_numel"], st.info["total_numel"], st.N
    d0, inner = ps.dim0_inner()
    grad_params = next(st._rank_grad_iter("cuda"))
    packed = torch.empty(total, dtype=torch.bfloat16, device="cuda")
    ms, mn = _time_stream(lambda: ss.fsdp_pack(st.plan, grad_params, packed), K)
    # oracle: pack of block group 0 of one rank
    g0 = ps.groups[0]
    sample = [bits(t) for t in grad_params[:g0]]
    p0 = sum(ps.numels()[:g0])
    cpu = _oracle_pair(lambda: oracle.pack(ps.layout, N, 2, d0[:g0], inner[:g0], sample),
                       args.cpu_seconds / 4, p0, "params/s",
                       f"block group 0 ({p0:,} params) of one rank, oracle packs")
    _row(f"a2 pack (one rank's gradients, {tag} model, N=8)", P, "params/s", ms, mn, 4 * P, peak,
         cpu)
    del grad_params

    del packed
    rs_ms, rs_mn = _time_stream(lambda: st.rs_adamw(), K)
    smp = _oracle_group0_from_step(st)
    cpu = _oracle_pair(lambda: _oracle_step(ps, smp, 10_000), args.cpu_seconds / 2, p0,
                       "params/s", "block group 0, oracle RS+AdamW+AG steps")
    _row(f"a3 reduce-scatter + AdamW ({tag} model, N=8)", P, "params/s", rs_ms, rs_mn,
         (2 * N + 26) * total, peak, cpu)
    ag_ms, ag_mn = _time_stream(lambda: st.all_gather(), K)
    g0p = ps.groups[0]
    shards0 = bits(st.shards[:N * ss.fsdp_plan_group(st.plan, 0)["shard_numel"]])
    cpu = _oracle_pair(lambda: oracle.all_gather_unpack(ps.layout, N, 2, d0[:g0p], inner[:g0p],
                                                        shards0),
                       args.cpu_seconds / 4, p0, "params/s", "block group 0, oracle unpacks")
    _row(f"a4 all-gather + unpack, n_out=1 ({tag} model, N=8)", P, "params/s", ag_ms, ag_mn, 4 * P,
         peak, cpu)
    ms, mn = _time_stream(lambda: st.fused_step(), K)
    _row(f"one-pass step: packed grads -> RS+AdamW -> shards + unpacked params ({tag}, N=8)", P,
         "params/s", ms, mn, (2 * N + 28) * P, peak)
    rank_sets = list(st._rank_grad_iter("cuda"))  # N distinct per-parameter gradient sets
    flat_pg = ss.ptr_array([g for rank in rank_sets for g in rank])
    ms, mn = _time_stream(lambda: st.fused_step(param_grads=flat_pg), K)
    _row("one-pass step with fused copy-in: N per-parameter grad sets -> RS+AdamW -> shards + "
         f"unpacked params ({tag}, N=8)", P, "params/s", ms, mn, (2 * N + 28) * P, peak)
    # its unfused counterpart: pack each rank's set (the copy-in), then the two calls
    set_arrs = [ss.ptr_array(rank) for rank in rank_sets]

    def pack_then_step():
        for r in range(N):
            ss.fsdp_pack(st.plan, set_arrs[r], st.grads[r])
        st.rs_adamw()
        st.all_gather()
    ms, mn = _time_stream(pack_then_step, max(K // 4, 5))
    _row("F1 counterpart: N packs of the per-parameter grad sets, then RS+AdamW and all-gather "
         f"({tag}, N=8)", P, "params/s", ms, mn, 4 * N * P + (2 * N + 26) * total + 4 * P, peak)
    del rank_sets, flat_pg, set_arrs
    # F2: FULL_SHARD gathers the parameters twice per iteration (forward and
    # backward), SHARD_GRAD_OP once ("FSDP1 vs FSDP2", strategy table)
    def full_shard():
        st.all_gather()
        st.all_gather()
        st.rs_adamw()

    def shard_grad_op():
        st.all_gather()
        st.rs_adamw()
    for name, fn, nag in (("FULL_SHARD", full_shard, 2), ("SHARD_GRAD_OP", shard_grad_op, 1)):
        ms, mn = _time_stream(fn, K)
        _row(f"strategy {name}: {nag} all-gather(s) + RS+AdamW per iteration ({tag}, N=8)", P,
             "params/s", ms, mn, (2 * N + 26) * total + nag * 4 * P, peak,
             extra={"all_gathers": nag})
    # F3: gradient accumulation over 4 micro-batches (same gradients each time)
    accum = torch.empty(total, device="cuda")
    kmic = 4

    def accumulate_step():
        st.t += 1
        hp = ss.adamw_params(step=st.t)
        for j in range(kmic):
            last = j == kmic - 1
            ss.fsdp_reduce_scatter_accumulate(st.plan, st._grads_arr, accum, j, kmic, st.master,
                                              st.m, st.v, st.shards, hp if last else None)
    ms, mn = _time_stream(accumulate_step, max(K // 4, 5))
    acc_bytes = (2 * N + 4) + 2 * (2 * N + 8) + (2 * N + 30)

    g0 = smp["groups"][0]  # block group 0, copied from the device above

    def oracle_accumulate():
        acc = None
        for _ in range(kmic):
            acc = oracle.accumulate(N, g0["shard_numel"], g0["grads"], acc)
        g = oracle.accumulated_grad(acc, kmic)
        oracle.adamw(g, g0["master"], g0["m"], g0["v"], lr=1e-3, beta1=0.9, beta2=0.999,
                     eps=1e-8, weight_decay=0.01, step=20_000)
    cpu = _oracle_pair(oracle_accumulate, args.cpu_seconds / 4, p0, "params/s",
                       f"block group 0, oracle optimizer steps of {kmic} micro-batches")
    _row(f"gradient accumulation: {kmic} micro-batches per optimizer step ({tag}, N=8)", P,
         "params/s", ms, mn, acc_bytes * total, peak, cpu,
         extra={"micro_batches": kmic, "ms_per_micro_batch": ms / kmic})
    del accum
    # F4: AdamW without fp32 master weights (bf16 shard updated in place)
    def no_master():
        st.t += 1
        ss.fsdp_reduce_scatter_adamw(st.plan, st._grads_arr, None, st.m, st.v, st.shards,
                                     ss.adamw_params(step=st.t))
    ms, mn = _time_stream(no_master, K)
    _row(f"RS + AdamW without fp32 master (2 B params + 8 B moments, {tag}, N=8)", P, "params/s",
         ms, mn, (2 * N + 20) * total, peak)
    st8 = st
    outs8 = [torch.empty(s, dtype=torch.bfloat16, device="cuda") for _ in range(N)
             for s in ps.shapes]
    ms, mn = _time_stream(lambda: ss.fsdp_all_gather_unpack(st8.plan, st8.shards, outs8, N), K)
    _row("a4 all-gather + unpack, n_out=N=8 (every rank's copy)", P, "params/s", ms, mn,
         (2 + 2 * N) * P, peak)
    # F4: the ZeRO-1/2 step ("Scaling data parallel" 9.1-9.2): reduce-scatter
    # the full per-rank gradients, AdamW on each rank's own 1/N, then all-gather
    # the updated bf16 parameters to every rank (n_out = N), the all-reduce
    # split into RS + AG with the AG moved onto the parameters
    outs8_arr = ss.ptr_array(outs8)

    def zero12_two_calls():
        st8.rs_adamw()
        ss.fsdp_all_gather_unpack(st8.plan, st8.shards, outs8_arr, N)

    def zero12_one_pass():
        ss.fsdp_sharded_step(st8.plan, st8.master, st8.m, st8.v, st8.shards, st8.next_hp(),
                             rank_grads=st8._grads_arr, params_out=outs8_arr, n_out=N)
    ms, mn = _time_stream(zero12_two_calls, K)
    _row(f"ZeRO-1/2 step: RS+AdamW, then all-gather to all N=8 ranks (two calls, {tag})", P,
         "params/s", ms, mn, (2 * N + 26) * total + (2 + 2 * N) * P, peak, extra={"n_out": N})
    ms, mn = _time_stream(zero12_one_pass, K)
    _row("ZeRO-1/2 step: RS+AdamW writing all N=8 ranks' parameters in the same pass "
         f"(fsdp_sharded_step, {tag})", P, "params/s", ms, mn,
         (2 * N + 26) * total + 2 * N * P, peak, extra={"n_out": N})
    # the same with the fused copy-in: N + N pointers per parameter exceed one
    # kernel-parameter table, so the call runs in windows of parameters
    rank_sets = list(st8._rank_grad_iter("cuda"))
    flat_pg = ss.ptr_array([g for rank in rank_sets for g in rank])

    def zero12_copy_in():
        ss.fsdp_sharded_step(st8.plan, st8.master, st8.m, st8.v, st8.shards, st8.next_hp(),
                             rank_param_grads=flat_pg, params_out=outs8_arr, n_out=N)
    ms, mn = _time_stream(zero12_copy_in, K)
    _row("ZeRO-1/2 step with the fused copy-in: N per-parameter grad sets -> RS+AdamW -> all N=8 "
         f"ranks' parameters in one pass, in parameter windows (fsdp_sharded_step, {tag})", P,
         "params/s", ms, mn, (2 * N + 26) * total + 2 * N * P, peak,
         extra={"n_out": N, "windows": -(-ps.num_params // (2048 // (2 * N)))})
    del outs8, outs8_arr, st, st8, rank_sets, flat_pg
    torch.cuda.empty_cache()


def _rows_block4096(ss, peak, K, cpu_seconds):
    # -- config 2: one 4096 block ---------------------------------------------
    ps2 = W.llama_block_4096()
    st2 = Step(ss, ps2, 1)
    P2, total2 = st2.info["unpadded_numel"], st2.info["total_numel"]

    def step2():
        st2.rs_adamw()
        st2.all_gather()
    ms, mn = _time_stream(step2, K)
    by = step_bytes(8, total2, P2, 1)
    _row("step on one Llama block, hidden 4096 (202M params, N=8): two calls", P2, "params/s", ms,
         mn, by["step"], peak)
    ms, mn = _time_stream(lambda: st2.fused_step(), K)
    cfg2 = _oracle_config(ps2)
    cpu = _oracle_pair(lambda: _oracle_step(ps2, cfg2, 10_000), cpu_seconds, cfg2["params"],
                       "params/s", _oracle_sample_text(ps2, cfg2) + "; oracle RS+AdamW+AG steps")
    del cfg2
    _row("step on one Llama block, hidden 4096 (202M params, N=8): one pass", P2, "params/s", ms,
         mn, (2 * 8 + 26) * total2 + 2 * P2, peak, cpu)
    del st2
    torch.cuda.empty_cache()


def _rows_small(ss, peak, want, awkward_scale=1.0, cpu_seconds=4.0):
    # -- config 1: tiny MLP, launch-bound -------------------------------------
    # Each row is the per-step time of 2000 steps issued back to back between
    # two CUDA events (median of 5 such batches): the rate a training loop of
    # tiny steps runs at.
    if "tiny" in want:
        ps1 = W.tiny_mlp()
        st1 = Step(ss, ps1, 1)
        P1, T1 = st1.info["unpadded_numel"], st1.info["total_numel"]
        one_pass_bytes = (2 * 2 + 26) * T1 + 2 * P1
        timing = "2000 steps back to back between two CUDA events, median of 5 batches"

        def step1():
            st1.rs_adamw()
            st1.all_gather()
        ms, mn = _time_back_to_back(step1)
        by = step_bytes(2, T1, P1, 1)
        _row("step on the tiny MLP (16,640 params, N=2): latency, two calls", P1, "params/s", ms,
             mn, by["step"], peak, extra={"us_per_step": ms * 1e3, "timing": timing})
        ms, mn = _time_back_to_back(lambda: st1.fused_step())
        _row("step on the tiny MLP (16,640 params, N=2): latency, one fsdp_sharded_step call",
             P1, "params/s", ms, mn, one_pass_bytes, peak,
             extra={"us_per_step": ms * 1e3, "timing": timing})
        # the same call with its arguments marshalled once (ss.ShardedStep)
        call = ss.ShardedStep(st1.plan, st1.master, st1.m, st1.v, st1.shards, st1.next_hp(),
                              rank_grads=st1._grads_arr, params_out=st1._outs_arr, n_out=1,
                              stream=torch.cuda.current_stream())
        step_no = [st1.t]

        def prepared():
            step_no[0] += 1
            call(step_no[0])
        ms, mn = _time_back_to_back(prepared)
        cfg1 = _oracle_config(ps1)
        cpu = _oracle_pair(lambda: _oracle_step(ps1, cfg1, 10_000), cpu_seconds, cfg1["params"],
                           "params/s", _oracle_sample_text(ps1, cfg1) + "; oracle RS+AdamW+AG steps")
        _row("step on the tiny MLP (16,640 params, N=2): latency, one prepared fsdp_sharded_step "
             "call (ss.ShardedStep)", P1, "params/s", ms, mn, one_pass_bytes, peak, cpu,
             extra={"us_per_step": ms * 1e3, "timing": timing})
        del call
        # the same C-ABI calls captured once in a CUDA graph and replayed (the
        # AdamW step count is frozen in the captured arguments, which does not
        # change the work done): two calls, then the one-pass kernel
        s_ = torch.cuda.Stream()
        s_.wait_stream(torch.cuda.current_stream())
        graphs = []
        for fn in (step1, lambda: st1.fused_step()):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(s_):
                fn()
                torch.cuda.synchronize()
                with torch.cuda.graph(g, stream=s_):
                    fn()
            graphs.append(g)
        torch.cuda.current_stream().wait_stream(s_)
        ms, mn = _time_back_to_back(lambda: graphs[0].replay())
        _row("step on the tiny MLP (16,640 params, N=2): two calls replayed from a CUDA graph",
             P1, "params/s", ms, mn, by["step"], peak,
             extra={"us_per_step": ms * 1e3, "timing": timing})
        ms, mn = _time_back_to_back(lambda: graphs[1].replay())
        _row("step on the tiny MLP (16,640 params, N=2): one-pass kernel replayed from a graph",
             P1, "params/s", ms, mn, one_pass_bytes, peak,
             extra={"us_per_step": ms * 1e3, "timing": timing})
        del graphs

    # -- config 3: awkward sizes, N=7 ------------------------------------------
    for kind in ((W.FLAT_ORIG_FALSE, W.FLAT_ORIG_TRUE) if "awkward" in want else ()):
        ps3 = W.awkward_1d(7, kind, torch.bfloat16)
        st3 = Step(ss, ps3, 1)

        def step3():
            st3.rs_adamw()
            st3.all_gather()
        ms, mn = _time_stream(step3, 100, warmup=10)
        by = step_bytes(7, st3.info["total_numel"], st3.info["unpadded_numel"], 1)
        cfg3 = _oracle_config(ps3)
        cpu = _oracle_pair(lambda: _oracle_step(ps3, cfg3, 10_000), cpu_seconds, cfg3["params"],
                           "params/s", _oracle_sample_text(ps3, cfg3) + "; oracle RS+AdamW+AG steps")
        _row(f"step on 200 awkward params ({W.LAYOUT_NAMES[kind]}, N=7)",
             st3.info["unpadded_numel"], "params/s", ms, mn, by["step"], peak, cpu,
             extra={"us_per_step": ms * 1e3})
        # the one pass as a prepared call (ss.ShardedStep), 2000 steps back to back
        call3 = ss.ShardedStep(st3.plan, st3.master, st3.m, st3.v, st3.shards, st3.next_hp(),
                               rank_grads=st3._grads_arr, params_out=st3._outs_arr, n_out=1,
                               stream=torch.cuda.current_stream())
        step3_no = [st3.t]

        def prepared3():
            step3_no[0] += 1
            call3(step3_no[0])
        ms, mn = _time_back_to_back(prepared3)
        P3, T3 = st3.info["unpadded_numel"], st3.info["total_numel"]
        _row(f"step on 200 awkward params ({W.LAYOUT_NAMES[kind]}, N=7): one prepared "
             "fsdp_sharded_step call (ss.ShardedStep)", P3, "params/s", ms, mn,
             (2 * 7 + 26) * T3 + 2 * P3, peak,
             extra={"us_per_step": ms * 1e3,
                    "timing": "2000 steps back to back between two CUDA events, median of 5 batches"})
        del call3

    # -- the same awkward shapes scaled up until they are bandwidth-bound:
    # odd-sized parameters at odd flat offsets (runs not congruent mod 16 bytes)
    large = "awkward" in want or "awkward_large" in want
    for kind in ((W.FLAT_ORIG_FALSE, W.PER_PARAM_DIM0) if large else ()):
        if kind == W.PER_PARAM_DIM0:
            ps4 = W.awkward_2d(7, count=200, max_rows=int(400_000 * awkward_scale))
        else:
            ps4 = W.awkward_1d(7, kind, torch.bfloat16, count=200,
                               max_len=int(2_000_000 * awkward_scale))
        st4 = Step(ss, ps4, 1)
        P4, tot4 = st4.info["unpadded_numel"], st4.info["total_numel"]
        g4 = next(st4._rank_grad_iter("cuda"))
        buf4 = torch.empty(tot4, dtype=torch.bfloat16, device="cuda")
        name = W.LAYOUT_NAMES[kind]
        ms, mn = _time_stream(lambda: ss.fsdp_pack(st4.plan, g4, buf4), 20)
        _row(f"large awkward ({name}, {P4:,} params, N=7): pack", P4, "params/s", ms, mn,
             2 * P4 + 2 * tot4, peak)
        ms, mn = _time_stream(lambda: st4.rs_adamw(), 20)
        _row(f"large awkward ({name}, N=7): RS + AdamW", P4, "params/s", ms, mn,
             (2 * 7 + 26) * tot4, peak)
        ms, mn = _time_stream(lambda: st4.all_gather(), 20)
        _row(f"large awkward ({name}, N=7): all-gather + unpack", P4, "params/s", ms, mn, 4 * P4,
             peak)
        # context for the two rows above: torch's own device copy of the same
        # bytes (P4 bf16 elements read and written), the operation the measured
        # peak is taken with, at this size
        src = torch.empty(P4, dtype=torch.bfloat16, device="cuda")
        dst = torch.empty_like(src)
        ms, mn = _time_stream(lambda: dst.copy_(src), 20)
        _row(f"large awkward ({name}, N=7): torch copy_ of the same bytes (context)", P4,
             "params/s", ms, mn, 4 * P4, peak)
        del src, dst
        # every rank's copy (n_out = N = 7 replicas, separately allocated)
        outs7 = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(7)
                 for n in ps4.numels()]
        outs7_arr = ss.ptr_array(outs7)
        ms, mn = _time_stream(
            lambda: ss.fsdp_all_gather_unpack(st4.plan, st4.shards, outs7_arr, 7), 10)
        _row(f"large awkward ({name}, N=7): all-gather + unpack, n_out=N=7", P4, "params/s", ms,
             mn, (2 + 2 * 7) * P4, peak)
        del outs7, outs7_arr
        ms, mn = _time_stream(lambda: st4.fused_step(), 20)
        _row(f"large awkward ({name}, N=7): one-pass step", P4, "params/s", ms, mn,
             (2 * 7 + 26) * tot4 + 2 * P4, peak)
        # fused copy-in: the 7 per-parameter gradient sets read in place, at
        # their misaligned offsets inside each parameter
        del g4
        rank_sets = list(st4._rank_grad_iter("cuda"))
        flat_pg = ss.ptr_array([g for rank in rank_sets for g in rank])
        ms, mn = _time_stream(lambda: st4.fused_step(param_grads=flat_pg), 20)
        _row(f"large awkward ({name}, N=7): one-pass step with fused copy-in", P4, "params/s",
             ms, mn, (2 * 7 + 2) * P4 + 26 * tot4, peak)
        del rank_sets, flat_pg, st4, buf4
        torch.cuda.empty_cache()
    # the same 1-D awkward set in fp32 (a FlatParameter of fp32 parameters)
    if large:
        ps5 = W.awkward_1d(7, W.FLAT_ORIG_FALSE, torch.float32, count=200,
                           max_len=int(2_000_000 * awkward_scale))
        st5 = Step(ss, ps5, 1)
        P5, tot5 = st5.info["unpadded_numel"], st5.info["total_numel"]
        ms, mn = _time_stream(lambda: st5.rs_adamw(), 20)
        _row(f"large awkward fp32 (flat_orig_false, {P5:,} params, N=7): RS + AdamW", P5,
             "params/s", ms, mn, (4 * 7 + 28) * tot5, peak)
        ms, mn = _time_stream(lambda: st5.all_gather(), 20)
        _row(f"large awkward fp32 (flat_orig_false, N=7): all-gather + unpack", P5, "params/s",
             ms, mn, 8 * P5, peak)
        del st5
        torch.cuda.empty_cache()



def _rows_awkward_wide(ss, peak, awkward_scale=1.0):
    # -- the 1-D awkward set at N = 16: misaligned runs with ranks beyond the
    # first 8, which the kernels' general instances read in further batches
    N = 16
    ps = W.awkward_1d(N, W.FLAT_ORIG_FALSE, torch.bfloat16, count=200,
                      max_len=int(2_000_000 * awkward_scale))
    st = Step(ss, ps, 1)
    P, tot = st.info["unpadded_numel"], st.info["total_numel"]
    ms, mn = _time_stream(lambda: st.fused_step(), 20)
    _row(f"large awkward (flat_orig_false, {P:,} params, N={N}): one-pass step", P, "params/s",
         ms, mn, (2 * N + 26) * tot + 2 * P, peak)
    rank_sets = list(st._rank_grad_iter("cuda"))
    flat_pg = ss.ptr_array([g for rank in rank_sets for g in rank])
    ms, mn = _time_stream(lambda: st.fused_step(param_grads=flat_pg), 20)
    _row(f"large awkward (flat_orig_false, N={N}): one-pass step with fused copy-in", P,
         "params/s", ms, mn, (2 * N + 2) * P + 26 * tot, peak)
    del rank_sets, flat_pg, st
    torch.cuda.empty_cache()
    # -- 800 PER_PARAM_DIM0 parameters in one group at N = 7: with per-parameter
    # gradients the pointers (8 per parameter) overflow one table, so the call
    # runs in parameter windows, each window's data in 7 runs (one per shard)
    ps = W.awkward_2d(7, count=800, max_rows=int(100_000 * awkward_scale))
    st = Step(ss, ps, 1)
    P, tot = st.info["unpadded_numel"], st.info["total_numel"]
    ms, mn = _time_stream(lambda: st.fused_step(), 20)
    _row(f"large awkward (per_param_dim0, 800 params in one group, {P:,} params, N=7): one-pass step",
         P, "params/s", ms, mn, (2 * 7 + 26) * tot + 2 * P, peak)
    rank_sets = list(st._rank_grad_iter("cuda"))
    flat_pg = ss.ptr_array([g for rank in rank_sets for g in rank])
    ms, mn = _time_stream(lambda: st.fused_step(param_grads=flat_pg), 20)
    _row("large awkward (per_param_dim0, 800 params in one group, N=7): one-pass step with fused "
         "copy-in (4 parameter windows x 7 runs)", P, "params/s", ms, mn, (2 * 7 + 2) * P + 26 * tot,
         peak)
    del rank_sets, flat_pg, st
    torch.cuda.empty_cache()


def _rows_world_sizes(ss, peak):
    # -- the 1.2B model at other world sizes: N = 2 and 4 (unrolled
    # instances), 16 (its own instance) and 32 (the general instance)
    for N in (2, 4, 16, 32):
        ps = W.llama_1b2(world_size=N)
        st = Step(ss, ps, 1)
        P, tot = st.info["unpadded_numel"], st.info["total_numel"]
        ms, mn = _time_stream(lambda: st.rs_adamw(), 20)
        _row(f"1.2B model, N={N}: RS + AdamW", P, "params/s", ms, mn, (2 * N + 26) * tot, peak,
             extra={"world_size": N})
        ms, mn = _time_stream(lambda: st.fused_step(), 20)
        _row(f"1.2B model, N={N}: one-pass step", P, "params/s", ms, mn, (2 * N + 26) * tot + 2 * P,
             peak, extra={"world_size": N})
        del st
        torch.cuda.empty_cache()


def _rows_ddp(args, ss, oracle, peak, used, K, bits):
    # -- a5: DDP bucketed average, cap sweep (config 4) -----------------------
    ds = W.ddp_grads(n_large=args.ddp_large)
    grads = W.make_ddp_grads(ds, device="cuda")
    outs = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for n in ds.numels]
    Pd = sum(ds.numels)
    small = [[bits(grads[r][t]) for t in range(40)] for r in range(ds.world_size)]
    psmall = sum(ds.numels[:40])
    cpu = _oracle_pair(lambda: oracle.ddp_average(small), args.cpu_seconds / 4, psmall,
                       "elements/s", f"first 40 tensors ({psmall:,} elements, N=8), oracle averages")
    import ctypes
    T = len(ds.numels)
    flat_arr = ss.ptr_array([g for rank in grads for g in rank])
    outs_arr = ss.ptr_array(outs)
    numels_arr = (ctypes.c_int64 * T)(*ds.numels)
    nb_out = ctypes.c_int()
    sp = torch.cuda.current_stream().cuda_stream

    def ddp_call(cap):
        st_ = ss.lib().ddp_bucket_pack_average(ds.world_size, T, numels_arr, flat_arr, cap,
                                               outs_arr, ctypes.byref(nb_out), sp)
        if st_ != 0:
            raise RuntimeError(f"ddp_bucket_pack_average: {ss.ss_strerror(st_)}")
    for cap in W.DDP_BUCKET_CAPS:
        nb = ss.ddp_bucket_assign(ds.numels, 2, cap)[1]
        ms, mn = _time_stream(lambda: ddp_call(cap), max(K // 10, 5))
        _row(f"a5 DDP bucketed average, cap {cap} B ({len(ds.numels)} grads, "
             f"{2 * Pd / 1e9:.2f} GB/rank, N=8)", Pd,
             "elements/s", ms, mn, (2 * ds.world_size + 2) * Pd, peak, cpu,
             extra={"bucket_cap_bytes": cap, "buckets": nb})
        cpu = None
    # the allocation-free entry point on the same list at the 25 MiB cap: its
    # table goes to the library's fixed device array instead of a
    # stream-ordered allocation
    cap = 25 << 20

    def ddp_noalloc():
        st_ = ss.lib().ddp_bucket_pack_average_noalloc(ds.world_size, T, numels_arr, flat_arr, cap,
                                                       outs_arr, ctypes.byref(nb_out), sp)
        if st_ != 0:
            raise RuntimeError(f"ddp_bucket_pack_average_noalloc: {ss.ss_strerror(st_)}")
    for name, fn in (("ddp_bucket_pack_average", lambda: ddp_call(cap)),
                     ("ddp_bucket_pack_average_noalloc", ddp_noalloc)):
        ms, mn = _time_stream(fn, max(K // 10, 5))
        _row(f"a5 DDP bucketed average through {name}, cap {cap} B ({len(ds.numels)} grads, N=8)",
             Pd, "elements/s", ms, mn, (2 * ds.world_size + 2) * Pd, peak,
             extra={"bucket_cap_bytes": cap, "entry_point": name})


def main():
    args = parse_args()
    world, rank, local = dist_env()
    if args.impl == "reference":
        run_reference(args, world, rank)
        return
    if args.mode == "rows":
        run_rows(args)
        return
    dist = dist_init(world, local)
    try:
        run_native(args, world, rank, local, dist)
    finally:
        if dist is not None:
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
