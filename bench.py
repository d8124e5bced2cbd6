#!/usr/bin/env python
"""Throughput of the fused IQL + HER train step on one GB300 (one JSON line).

A step is one pass of the whole path over one batch: HER index sampling and
relabel, V forward + expectile loss + policy + V backward, the primary
gradient reduction with the per-source norms and budget coefficients, and
Adam.  Inputs are synthetic (seeded, see synth/), resident in HBM before the
timed region; per step a fresh Q [B, A] is read.  With --gpus N under
torchrun every rank runs an independent replica (the step has no exchange).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

METRIC = "IQL+HER train steps/s and samples/s at B=16384; % tensor/HBM roofline"
UNIT = "samples/s"
SMS = 152
FP32_LANES_PER_SM = 128
PROFILE_NOTE = "profiles/ (ncu launch list and per-kernel summaries)"
# The sources each dominant kernel is compiled from: their hash keys the ncu
# traffic figure below, so a changed kernel reports null until captured again.
KERNEL_SOURCES = {
    "vnet_tc (tcgen05)": ("vnet_tc.cu", "common.cuh", "tc_image.cuh", "umma.cuh"),
    "vnet_wide fwd + wgrad (tcgen05, TMA)": ("vnet_wide.cu", "common.cuh", "tc_image.cuh", "umma.cuh"),
}
# dram__bytes_read.sum + dram__bytes_write.sum of one launch of the dominant
# kernel from the ncu capture summarised under profiles/, with the hash of
# the kernel sources the capture ran (source_hash)
NCU_TRAFFIC = {
    # profiles/vnet_tc_prod_fp32_B16384_H128.md (ncu --set full, one launch)
    ("vnet_tc (tcgen05)", "prod_fp32_B16384_S50_H128_A5"): ("5f87a55b6e9d31be", 6908928),
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default=synth.PROD.name, choices=[w.name for w in synth.ALL])
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="bounded oracle sample (CPU baseline)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--repeats", type=int, default=5, help="timed regions of --steps steps; the median is reported")
    ap.add_argument("--no-workloads", action="store_true", help="skip the per-workload table of the other configs")
    ap.add_argument("--no-forward", action="store_true", help="skip the IQL-target (V forward) measurement")
    ap.add_argument("--vnet-path", default=None, choices=("tc_fused", "tc_layered", "cuda_cores"),
                    help="V forward/backward implementation (default: the library's choice for the shape)")
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "sm_max_mhz": 2070.0}, \
        "fallback"


def algorithmic(w):
    """Algorithmic work of one step, per phase: bytes moved and flops."""
    b, s, a, p, n, g = w.batch, w.state_dim, w.num_actions, w.n_params, w.n_nets, w.goal_dim
    nh = w.her_count
    relabel = b * (2 * s * 4 + 12) * 2 + b * 8 + nh * 4 * g + (nh * 4 if w.strategy != "random" else 0)
    vnet_bytes = b * s * 4 + b * 4 + b * a * 4 + n * (p * 4 + b * 4 * (2 + a) + p * 4)
    flops = n * 2 * b * (2 * s * w.hidden + 3 * w.hidden ** 2 + 3 * w.hidden)
    optim_bytes = n * 4 * p * (6 + 2 + 2 * w.n_aux)
    return dict(relabel_bytes=relabel, vnet_bytes=vnet_bytes, vnet_flops=flops, optim_bytes=optim_bytes,
                total_bytes=relabel + vnet_bytes + optim_bytes)


class Clocks:
    """nvidia-smi samples (every 200 ms) while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        # nvidia-smi's start-up queries the driver for a while and slows
        # kernel launches meanwhile: begin timing once it has printed a sample
        t0 = time.time()
        while time.time() - t0 < 5.0 and self.proc.poll() is None:
            if os.path.getsize(self.path) > 0:
                break
            time.sleep(0.05)
        time.sleep(0.05)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        self.proc.wait()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": float(rows[0][2]) if rows[0][2].replace(".", "").isdigit() else None,
                "reasons": reasons, "samples": len(rows)}


def _oracle_steps(w, n_steps, seconds, batch=None):
    """Time up to n_steps oracle steps (stopping after `seconds`) of workload w, or of a row sample of
    its batch; returns (steps, seconds)."""
    from oracle import step as ostep
    ws = w if batch is None or batch >= w.batch else synth.scaled(w, batch=batch)
    rep = synth.make_replay(w)
    cfg = ostep.config_from_workload(ws)
    nets = [ostep.NetState.fresh(synth.make_params(w, k), w.taus[k]) for k in range(w.n_nets)]
    k = 0
    t0 = time.perf_counter()
    while k < n_steps:
        q = synth.make_q(ws, k)
        aux = [synth.make_aux(w, k, n) for n in range(w.n_nets)] if w.n_aux else None
        ostep.train_step(cfg, rep, k, q, nets, aux)
        k += 1
        if time.perf_counter() - t0 >= seconds:
            break
    return k, time.perf_counter() - t0


_SINGLE_CORE = """
import json, sys
sys.path.insert(0, {root!r})
import synth, bench
w = synth.BY_NAME[{name!r}]
bench._oracle_steps(w, 1, 1e9)                      # warm-up (imports, first-touch)
k, el = bench._oracle_steps(w, {steps}, {seconds})
print(json.dumps([k, el]))
"""


def cpu_baseline(w, seconds):
    """The oracle as it stands, on this host, on a bounded sample of the workload: whole steps with numpy's
    default BLAS threading for `seconds` of CPU work, and (a separate process, one BLAS thread) the first
    few steps on one core."""
    k, el = _oracle_steps(w, 10 ** 6, seconds)
    out = {"value": k * w.batch / el, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
           "sample": f"{k} full steps (B={w.batch}) of {w.name} in {el:.1f} s, numpy fp64 with its default "
                     f"BLAS threading; index sampling in single-threaded Python"}
    env = dict(os.environ)
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        env[var] = "1"
    try:
        r = subprocess.run([sys.executable, "-c", _SINGLE_CORE.format(root=ROOT, name=w.name, steps=5,
                                                                      seconds=seconds)],
                           capture_output=True, text=True, env=env, timeout=300)
        k1, el1 = json.loads(r.stdout.strip().splitlines()[-1])
        out["single_core"] = {"value": k1 * w.batch / el1, "unit": UNIT, "cores": 1,
                              "sample": f"{k1} full steps after one warm-up step, one BLAS thread"}
    except (subprocess.SubprocessError, ValueError, IndexError, OSError):
        out["single_core"] = None
    return out


def run_reference(args, w):
    """--impl reference: the CPU oracle (the slow definition) timed on this host, whole steps of the
    workload (a row sample of each step's batch only if whole steps would not finish in a few minutes)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from oracle import step as ostep
    # one step's cost decides the sample: whole batches when K + W of them fit in about two minutes
    k1, t1 = _oracle_steps(w, 1, 1e9)
    rows = w.batch
    if (args.steps + args.warmup) * t1 > 120.0:
        rows = max(256, int(w.batch * 120.0 / ((args.steps + args.warmup) * t1)) // 256 * 256)
    ws = synth.scaled(w, batch=rows) if rows < w.batch else w
    rep = synth.make_replay(w)
    cfg = ostep.config_from_workload(ws)
    nets = [ostep.NetState.fresh(synth.make_params(w, k), w.taus[k]) for k in range(w.n_nets)]

    def one(k):
        q = synth.make_q(ws, k)
        aux = [synth.make_aux(w, k, n) for n in range(w.n_nets)] if w.n_aux else None
        ostep.train_step(cfg, rep, k, q, nets, aux)

    for k in range(args.warmup):
        one(k)
    t0 = time.perf_counter()
    for k in range(args.steps):
        one(args.warmup + k)
    el = time.perf_counter() - t0
    value = args.steps * rows / el
    sample = (f"each step: {'the whole' if rows == w.batch else f'{rows} rows of the'} {w.name} batch "
              f"(B={w.batch}; full-size replay buffer and V network), numpy fp64 oracle")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "batch": rows, "hidden": w.hidden, "state_dim": w.state_dim},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


def max_over_ranks(x, device):
    """Largest value of the float x over the ranks of the process group (x itself with one process)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world, steps, rows_per_rank, ms_max):
    """Rows per second of the whole job: every rank processed steps x rows_per_rank rows, and the job took
    the slowest rank's time."""
    return world * steps * rows_per_rank / (ms_max / 1e3)


def source_hash(files):
    """First 16 hex digits of the sha256 of the given package sources (a kernel and the headers it includes)."""
    import hashlib
    hsh = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "offline_rl_step_gb300", "csrc", f), "rb") as fh:
            hsh.update(fh.read())
    return hsh.hexdigest()[:16]


class Run:
    """One workload set up on the GPU: replay buffer, context, networks, a pre-marshalled step, and every
    step's Q (device and pinned host) and auxiliary sources resident before any timing."""

    def __init__(self, w, rank, steps, warmup, vnet_path=None):
        import torch

        import offline_rl_step_gb300 as ofrl
        self.torch, self.ofrl, self.w = torch, ofrl, w
        dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
        rep = synth.make_replay(w)
        self.replay = ofrl.Replay(dev(rep["states"]), dev(rep["next_states"]), dev(rep["actions"]),
                                  dev(rep["rewards"]), dev(rep["dones"]), w.state_dim, w.goal_dim,
                                  dev(rep["episode_ends"]))
        self.replay_bytes = sum(t.numel() * t.element_size() for t in (self.replay.states, self.replay.next_states))
        del rep
        self.her = ofrl.HerConfig(w.batch, w.her_count, w.strategy, w.goal_threshold, w.seed + rank)
        self.ctx = ofrl.Context(w.state_dim, w.hidden, w.num_actions, w.prec, max_batch=w.batch, max_nets=w.n_nets)
        if vnet_path is not None:
            self.ctx.select_vnet_path(vnet_path)
        self.nets = [ofrl.VNet.from_params(torch.from_numpy(synth.make_params(w, k)), w.taus[k])
                     for k in range(w.n_nets)]
        self.opt = ofrl.Opt(lr=w.lr, beta1=w.beta1, beta2=w.beta2, eps=w.eps, weight_decay=w.weight_decay,
                            max_grad_norm=w.max_grad_norm, beta=w.beta, budget=w.budget)
        self.batch = ofrl.Batch.empty(w.batch, w.state_stride)
        n, b, a = w.n_nets, w.batch, w.num_actions
        self.v_out = torch.empty(n, b, device="cuda")
        self.pi_out = torch.empty(n, b, a, device="cuda")
        self.am_out = torch.empty(n, b, dtype=torch.int32, device="cuda")
        self.loss_out = torch.empty(n, device="cuda")
        self.norms_out = torch.empty(n, 5, device="cuda")
        self.total = warmup + steps
        self.warmup, self.steps = warmup, steps
        self.q_host = np.stack([synth.make_q(w, k) for k in range(self.total)])
        self.q_dev = dev(self.q_host)
        self.aux_dev = None
        if w.n_aux:
            self.aux_dev = [[dev(x) for x in synth.make_aux(w, k, 0)] for k in range(self.total)]
        self.plan = ofrl.StepPlan(self.ctx, self.replay, self.her, self.batch, self.nets, self.opt, n_aux=w.n_aux,
                                  v_out=self.v_out, pi_out=self.pi_out, argmax_out=self.am_out,
                                  loss_out=self.loss_out, norms_out=self.norms_out)
        self.qh = self.loss_h = self.norms_h = self.hplan = None

    def auxk(self, k):
        return [self.aux_dev[k]] if self.aux_dev is not None else None

    def warm(self):
        for k in range(self.warmup):
            self.plan.run(k, self.q_dev[k], self.auxk(k))
        self.torch.cuda.synchronize()

    def host_io(self):
        """The end-to-end form: Q read in place from pinned host memory, loss and norms written in place to
        pinned host memory (the public train_step call with host buffers)."""
        torch = self.torch
        if self.hplan is None:
            self.qh = torch.from_numpy(self.q_host).pin_memory()
            self.loss_h = torch.empty(self.w.n_nets, pin_memory=True)
            self.norms_h = torch.empty(self.w.n_nets, 5, pin_memory=True)
            self.plan.sync_t()
            self.hplan = self.ofrl.StepPlan(self.ctx, self.replay, self.her, self.batch, self.nets, self.opt,
                                            n_aux=self.w.n_aux, v_out=self.v_out, pi_out=self.pi_out,
                                            argmax_out=self.am_out, loss_out=self.loss_h, norms_out=self.norms_h)
            for k in range(self.warmup):
                self.hplan.run(k, self.qh[k], self.auxk(k))
            torch.cuda.synchronize()
            self.hplan.sync_t()
            self.plan.reload_t()

    def region(self, e2e=False, world=1):
        """One timed region of `steps` steps (CUDA events on the launching stream, a barrier and a
        synchronize on both sides); returns the milliseconds, max over ranks."""
        torch = self.torch
        import torch.distributed as dist
        if e2e:
            self.host_io()
            self.hplan.reload_t()
            plan, q = self.hplan, self.qh
        else:
            plan, q = self.plan, self.q_dev
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for k in range(self.warmup, self.total):
            plan.run(k, q[k], self.auxk(k))
        e1.record()
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        plan.sync_t()
        if e2e:
            self.plan.reload_t()
        return max_over_ranks(e0.elapsed_time(e1), "cuda")

    def phases(self):
        """Per-phase device milliseconds per step (one event pair per phase on the step's stream)."""
        self.ofrl.profile_begin(self.ctx, self.steps)
        for k in range(self.warmup, self.total):
            self.plan.run(k, self.q_dev[k], self.auxk(k))
        phase_ms, nprof = self.ofrl.profile_end(self.ctx)
        self.plan.sync_t()
        return {p: v / max(nprof, 1) for p, v in phase_ms.items()}

    def close(self):
        self.ctx.close()


def roofline(w, phase_avg, path, region_s, pk, pk_kind):
    """The dominant kernel against its roof, and every phase against its own."""
    alg = algorithmic(w)
    dominant = max(phase_avg, key=phase_avg.get)
    dur_s = phase_avg[dominant] / 1e3
    sm_mhz = pk.get("sm_max_mhz", 2070.0)
    # a kernel inside a timed region under a second long runs at the burst
    # rate; the sustained figure is for kernels inside seconds-long loops
    burst = region_s < 1.0
    tpk = pk["bf16_tflops"] if burst or "bf16_tflops_sustained" not in pk else pk["bf16_tflops_sustained"]
    tpk_name = "bf16_tflops" if burst or "bf16_tflops_sustained" not in pk else "bf16_tflops_sustained"
    if dominant == "vnet" and path in ("tc_fused", "tc_layered"):
        # tensor-core kernels: bf16 MMAs (three-term split, six products per
        # K-step, for fp32 workloads); algorithmic flops over the bf16 peak
        ach = alg["vnet_flops"] / dur_s / 1e12
        # MMA work as executed: 128-row tiles, S padded to 64, five GEMMs;
        # one product per K-step (bf16), or through the fp32 split six for
        # the forward z1, z2 and three for the backward GEMMs (fused: dh1,
        # dW2, dW1; layered: dW2, dW1, its dh1 six)
        tiles = -(-w.batch // 128)
        hp = max(w.hidden, 128)   # hidden 64 runs zero-padded to 128 units on the fused kernel
        fwd = hp * 64 + hp ** 2              # z1, z2 per row
        dh1 = hp ** 2
        wgr = hp * 64 + hp ** 2              # dW1, dW2 per row
        if w.prec == "bf16":
            per_row = fwd + dh1 + wgr
        elif path == "tc_fused":
            per_row = 6 * fwd + 3 * (dh1 + wgr)
        else:
            per_row = 6 * (fwd + dh1) + 3 * wgr
        mma = w.n_nets * tiles * 128 * 2 * per_row
        kname = "vnet_tc (tcgen05)" if path == "tc_fused" else "vnet_wide fwd + wgrad (tcgen05, TMA)"
        entry = NCU_TRAFFIC.get((kname, w.name))
        traffic = None
        if entry is not None and entry[0] == source_hash(KERNEL_SOURCES[kname]):
            traffic = entry[1]
        roof = {"kernel": kname, "bound": "tensor", "achieved": ach, "peak": tpk,
                "unit": "TFLOP/s", "frac": ach / tpk, "traffic": traffic,
                "peak_source": f"{tpk_name} ({pk_kind}; timed region {region_s * 1e3:.1f} ms)",
                "kernel_source_sha16": source_hash(KERNEL_SOURCES[kname]),
                "mma_tflops_executed": mma / dur_s / 1e12, "mma_frac_executed": mma / dur_s / 1e12 / tpk}
    elif dominant == "vnet":
        fp32_peak = SMS * FP32_LANES_PER_SM * 2 * sm_mhz * 1e6 / 1e12
        ach = alg["vnet_flops"] / dur_s / 1e12
        roof = {"kernel": "vnet_fwd_bwd", "bound": "alu", "achieved": ach, "peak": fp32_peak, "unit": "TFLOP/s",
                "frac": ach / fp32_peak, "traffic": None,
                "peak_source": f"fp32 FMA: {SMS} SMs x {FP32_LANES_PER_SM} lanes x 2 x {sm_mhz:.0f} MHz"}
    else:
        key = {"relabel": "relabel_bytes", "reduce": "optim_bytes", "adam": "optim_bytes"}[dominant]
        ach = alg[key] / dur_s / 1e9
        roof = {"kernel": dominant, "bound": "hbm", "achieved": ach, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": ach / pk["hbm_gbs"], "traffic": None, "peak_source": f"hbm_gbs ({pk_kind})"}
    roof["phase_ms"] = {p: round(v, 5) for p, v in phase_avg.items()}
    roof["relabel_hbm_frac"] = alg["relabel_bytes"] / (phase_avg["relabel"] / 1e3) / 1e9 / pk["hbm_gbs"]
    # every phase against its own roof, algorithmic work over the phase's
    # event-timed duration: relabel and the optimizer (reduce, norms, Adam)
    # against measured HBM, the V forward / backward against the bf16 peak
    # (the fp32 workloads reach it through the split)
    t_rl = phase_avg["relabel"] / 1e3
    t_v = phase_avg["vnet"] / 1e3
    t_opt = (phase_avg["reduce"] + phase_avg.get("adam", 0.0)) / 1e3
    roof["phases"] = {
        "relabel": {"bound": "hbm", "bytes": alg["relabel_bytes"], "achieved_gbs": alg["relabel_bytes"] / t_rl / 1e9,
                    "frac": alg["relabel_bytes"] / t_rl / 1e9 / pk["hbm_gbs"]},
        "vnet": {"bound": "tensor", "flops": alg["vnet_flops"], "achieved_tflops": alg["vnet_flops"] / t_v / 1e12,
                 "frac": alg["vnet_flops"] / t_v / 1e12 / tpk},
        "reduce_norms_adam": {"bound": "hbm", "bytes": alg["optim_bytes"],
                              "achieved_gbs": alg["optim_bytes"] / t_opt / 1e9,
                              "frac": alg["optim_bytes"] / t_opt / 1e9 / pk["hbm_gbs"],
                              "note": "parameter buffers (<= 2.2 MB) are L2-resident"},
    }
    return roof


def run_ours(args, w):
    import torch
    import torch.distributed as dist

    import offline_rl_step_gb300 as ofrl  # noqa: F401

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    pk, pk_kind = peaks()

    run = Run(w, rank, args.steps, args.warmup, args.vnet_path)
    run.warm()

    # ---- timed regions: R regions of K steps each (device Q), each followed
    # by one region of the end-to-end form (host Q in, loss / norms out in
    # place), interleaved so both see the same box state; medians reported ----
    clocks = Clocks(local)
    clocks.start()
    dev_ms, e2e_ms = [], []
    for _ in range(args.repeats):
        dev_ms.append(run.region(world=world))
        if not args.no_e2e:
            e2e_ms.append(run.region(e2e=True, world=world))
    clk = clocks.stop()
    ms = statistics.median(dev_ms)
    ms_per_step = ms / args.steps
    value = whole_job_rate(world, args.steps, w.batch, ms)

    phase_avg = run.phases()
    path = run.ctx.vnet_path(w.n_nets)
    roof = roofline(w, phase_avg, path, ms / 1e3, pk, pk_kind)

    e2e = None
    if not args.no_e2e:
        e2e = {"value": whole_job_rate(world, args.steps, w.batch, statistics.median(e2e_ms)), "unit": UNIT,
               "h2d_bytes_per_step": int(w.batch * w.num_actions * 4),
               "d2h_bytes_per_step": int(w.n_nets * 4 + w.n_nets * 5 * 4),
               "ms_per_step_regions": [round(x / args.steps, 5) for x in e2e_ms],
               "path": "train_step with Q read in place from pinned host memory and loss / norms written in place "
                       "to pinned host memory (NVLink-C2C); median of the regions interleaved with the device ones"}
        e2e.update(other_e2e_forms(run, world))
    fwd = None if args.no_forward else forward_bench(run, args.steps, args.repeats, pk, pk_kind, world)
    status = run.ctx.poll_status()
    launches = run.plan.kernels() * args.steps
    replay_bytes = run.replay_bytes
    run.close()
    del run
    torch.cuda.empty_cache()

    workloads = None
    if rank == 0 and world == 1 and not args.no_workloads:
        workloads = {}
        for ow in synth.ALL:
            r2 = Run(ow, rank, args.steps, args.warmup)
            r2.warm()
            regions = [r2.region() for _ in range(args.repeats)]
            m = statistics.median(regions)
            ph = r2.phases()
            rf = roofline(ow, ph, r2.ctx.vnet_path(ow.n_nets), m / 1e3, pk, pk_kind)
            workloads[ow.name] = {
                "value": ow.batch * args.steps / (m / 1e3), "unit": UNIT, "ms_per_step": m / args.steps,
                "ms_per_step_regions": [round(x / args.steps, 5) for x in regions],
                "vnet_path": r2.ctx.vnet_path(ow.n_nets), "dominant_kernel": rf["kernel"],
                "dominant_frac": rf["frac"], "vnet_frac": rf["phases"]["vnet"]["frac"],
                "vnet_mma_frac_executed": rf.get("mma_frac_executed"),
                "relabel_hbm_frac": rf["relabel_hbm_frac"],
                "reduce_norms_adam_hbm_frac": rf["phases"]["reduce_norms_adam"]["frac"],
                "phase_ms": rf["phase_ms"]}
            r2.close()
            del r2
            torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, args.cpu_seconds)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "steps_per_s": 1e3 / ms_per_step * world,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if w.prec == "bf16" else "f32", "data": "synthetic",
            "repeats": {"n": args.repeats, "statistic": "median",
                        "ms_per_step_regions": [round(x / args.steps, 5) for x in dev_ms],
                        "spread": (max(dev_ms) - min(dev_ms)) / ms},
            "config": {"workload": w.name, "batch": w.batch, "state_dim": w.state_dim, "hidden": w.hidden,
                       "num_actions": w.num_actions, "n_nets": w.n_nets, "her": f"{w.strategy} {w.her_ratio}",
                       "capacity": w.capacity, "parallelism": f"replicas{world}",
                       "launch": "direct kernel launches chained by programmatic dependent launch",
                       "vnet_path": path,
                       "l2": f"inputs larger than L2: replay buffer {replay_bytes / 2**20:.0f} MiB read at "
                             f"random rows every step"},
            "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "workloads": workloads, "iql_target": fwd,
            "gpu_launches": launches, "clocks": clk, "status": status,
        }
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


def forward_bench(run, steps, repeats, pk, pk_kind, world):
    """The IQL bootstrap target r + gamma (1 - done) V(s') of the relabelled batch (ofrl_iql_target: V
    forward on the next states, tensor cores where the step's V kernel is the fused one): median of
    `repeats` regions of `steps` calls through the API, and of the same calls replayed from a CUDA graph
    (the device's time); rows/s, and the forward's flops against the bf16 peak."""
    torch, ofrl, w = run.torch, run.ofrl, run.w
    b = w.batch
    tgt = torch.empty(b, device="cuda")
    vn = torch.empty(b, device="cuda")
    prm = run.nets[0].params
    call = lambda: ofrl.iql_target(run.ctx, prm, run.batch.next_states, run.batch.rewards, run.batch.dones, 0.99,
                                   tgt, v_next_out=vn)
    for _ in range(3):
        call()
    torch.cuda.synchronize()
    regions = []
    for _ in range(repeats):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            call()
        e1.record()
        torch.cuda.synchronize()
        regions.append(max_over_ranks(e0.elapsed_time(e1), "cuda"))
    ms = statistics.median(regions) / steps
    # the same calls captured once in a CUDA graph and replayed: the device's
    # time per call, free of the host's per-call argument checks and launches
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(steps):
            call()
    graph.replay()
    torch.cuda.synchronize()
    gregions = []
    for _ in range(repeats):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        graph.replay()
        e1.record()
        torch.cuda.synchronize()
        gregions.append(max_over_ranks(e0.elapsed_time(e1), "cuda"))
    del graph
    gms = statistics.median(gregions) / steps
    flops = 2 * b * (w.state_dim * w.hidden + w.hidden ** 2 + w.hidden)
    tpk = pk["bf16_tflops"]
    return {"rows_per_s": whole_job_rate(world, 1, b, ms), "us_per_call": ms * 1e3, "batch": b,
            "device_rows_per_s": whole_job_rate(world, 1, b, gms), "device_us_per_call": gms * 1e3,
            "vnet_path": run.ctx.vnet_path(1),
            "tflops": flops / (gms / 1e3) / 1e12, "frac_of_bf16_burst_peak": flops / (gms / 1e3) / 1e12 / tpk,
            "peak_source": f"bf16_tflops ({pk_kind})",
            "note": "one call = weight pack + forward kernel; us_per_call: median of regions of back-to-back "
                    "calls through the API (bound by the host's per-call cost when it exceeds the device's); "
                    "device_us_per_call and tflops: the same calls replayed from a CUDA graph"}


def other_e2e_forms(run, world):
    """Other end-to-end forms, one region each: (a) the step graph captured with the pinned host Q and
    loss / norms buffers themselves; (b) the step graph with a Q copy-in node and loss / norms copy-out
    nodes; (c) direct calls with a torch copy of Q in and two copies out."""
    torch, ofrl = run.torch, run.ofrl
    run.host_io()
    qh, loss_h, norms_h, auxk = run.qh, run.loss_h, run.norms_h, run.auxk
    b = run.w.batch
    out = {}

    def timed(fn):
        e2, e3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e2.record()
        for k in range(run.warmup, run.total):
            fn(k)
        e3.record()
        torch.cuda.synchronize()
        return max_over_ranks(e2.elapsed_time(e3), "cuda")

    kw = dict(v_out=run.v_out, pi_out=run.pi_out, argmax_out=run.am_out)
    sgh = ofrl.StepGraph(run.ctx, run.replay, run.her, run.batch, run.nets, run.opt, qh[0], aux=auxk(0),
                         loss_out=loss_h, norms_out=norms_h, **kw)
    for k in range(run.warmup):
        sgh.launch(k, qh[k], auxk(k))
    torch.cuda.synchronize()
    gms = timed(lambda k: sgh.launch(k, qh[k], auxk(k)))
    sgh.sync_t()
    sgh.close()
    q_stage = torch.empty_like(run.q_dev[0])
    sg = ofrl.StepGraph(run.ctx, run.replay, run.her, run.batch, run.nets, run.opt, q_stage, aux=auxk(0),
                        loss_out=run.loss_out, norms_out=run.norms_out, q_host=qh[0], loss_host=loss_h,
                        norms_host=norms_h, **kw)
    for k in range(run.warmup):
        sg.launch_io(k, qh[k], auxk(k), loss_h, norms_h)
    torch.cuda.synchronize()
    ems = timed(lambda k: sg.launch_io(k, qh[k], auxk(k), loss_h, norms_h))
    sg.sync_t()
    sg.close()
    run.plan.reload_t()

    def copy_step(k):
        q_stage.copy_(qh[k], non_blocking=True)
        run.plan.run(k, q_stage, auxk(k))
        loss_h.copy_(run.loss_out, non_blocking=True)
        norms_h.copy_(run.norms_out, non_blocking=True)
    dms = timed(copy_step)
    run.plan.sync_t()
    rate = lambda m: whole_job_rate(world, run.steps, b, m)
    out["graph_value"] = rate(gms)
    out["graph_path"] = ("StepGraph captured with the pinned host Q and loss / norms buffers: one graph launch per "
                         "step, Q staged by the relabel, loss / norms written in place")
    out["graph_copy_value"] = rate(ems)
    out["graph_copy_path"] = ("StepGraph.launch_io: one graph launch per step (Q copy-in node, step, loss / norms "
                              "copy-out nodes)")
    out["copy_value"] = rate(dms)
    out["copy_path"] = "torch copy of Q in, train_step (three kernel launches), two copies out"
    return out


def main():
    args = parse()
    w = synth.BY_NAME[args.workload]
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
