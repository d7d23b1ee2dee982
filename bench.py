"""Benchmark: one step = the whole memory-bound hot path on one GPU.

A step runs, on synthetic data already resident in HBM:
  * the fused AdamW update over the Llama-7B parameter table (291 tensors,
    6,738,415,616 params; bf16 grads, fp32 master/m/v, bf16 working copy);
  * the softmax backward of an attention block at B=8, H=12, S=1024
    (98,304 x 1,024, causal), once in fp32 and once in bf16;
  * the LayerNorm backward at B=8, S=2048, D=4096 (bf16 I/O, fp32 dgamma/dbeta).
Every input is larger than the 129 MB L2, so nothing stays cached between
launches.  `value` is the algorithmic HBM bytes of a step (30 B/param for
AdamW, 12 or 6 B/element for softmax, 6 B/element + stats for LayerNorm)
divided by the device time of the step, summed over ranks for N > 1 (each rank
runs an independent replica: weak scaling).

Timing: CUDA events bracket the timed steps and, inside each step, the AdamW
launch (its mean duration is the roofline's `achieved`).  No event sits between
the backward kernels, which run back to back as in a training step; their total
per step is `backward_in_step`, and each one's own duration comes from a loop of
back-to-back calls of it after the timed region (`kernels`).

Usage:  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
With --impl reference the CPU oracle is timed on the host's cores instead (rank 0
only), one proportional sample of the workload per step.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = ("AdamW step Gparams/s + GB/s as % of GB300 HBM peak; softmax/LN bwd GB/s")
HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
LOSS_SCALE = 65536.0

# Workloads.  "full": the sizes of the headline configurations.  "small": the same
# kernels on the GPT-2-small table and half the attention rows (~3 GB resident),
# used for profiler captures.
SM_ROWS, SM_COLS = 8 * 12 * 1024, 1024
LN_ROWS, LN_D = 8 * 2048, 4096
WORKLOADS = {
    "full": dict(table="llama7b", grad_std=1e-4, sm_rows=SM_ROWS, ln_rows=LN_ROWS),
    "small": dict(table="gpt2", grad_std=1e-3, sm_rows=SM_ROWS // 2, ln_rows=LN_ROWS),
}
FALLBACK_HBM_GBS = 6800.0
WORKLOAD_TEXT = {
    "full": ("Llama-7B-shaped fused AdamW (291 tensors, 6,738,415,616 params, bf16 grads x65536, "
             "fp32 master/m/v, bf16 copy) + softmax bwd 98,304x1,024 causal fp32 and bf16 + "
             "LayerNorm bwd 16,384x4,096 bf16"),
    "small": ("GPT-2-small-shaped fused AdamW (148 tensors, 124,439,808 params) + softmax bwd "
              "49,152x1,024 causal fp32 and bf16 + LayerNorm bwd 16,384x4,096 bf16 "
              "(profiling size)"),
}


def adamw_bytes(n_params: int) -> int:
    # read grad 2 + theta 4 + m 4 + v 4; write theta 4 + m 4 + v 4 + copy 2 + grad 2
    return 30 * n_params


def softmax_bytes(rows: int, cols: int, esize: int) -> int:
    return 3 * esize * rows * cols              # read P, dY; write dX


def layernorm_bytes(rows: int, D: int, esize: int) -> int:
    # read x, dY; write dX; + mean/inv_std per row; + gamma, dgamma, dbeta per column
    return 3 * esize * rows * D + 8 * rows + 12 * D


def causal_softmax_bytes(rows: int, cols: int, period: int, offset: int, esize: int) -> int:
    """Reads of the 16-byte vectors holding an open column of P and dY, plus all of dX."""
    import numpy as np
    per_vec = 16 // esize
    r = np.arange(rows, dtype=np.int64)
    valid = np.minimum(cols, r % period + 1 + offset)
    vecs = (valid + per_vec - 1) // per_vec
    return int(2 * 16 * vecs.sum() + esize * rows * cols)


def rmsnorm_bytes(rows: int, D: int, esize: int) -> int:
    # read x, dY; write dX; + inv_rms per row; + gamma, dgamma per column
    return 3 * esize * rows * D + 4 * rows + 8 * D


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# ----------------------------------------------------------------------------- ranks
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_over_ranks(values, op="max"):
    """Max (or sum) of a list of floats over all ranks; identity without a process group."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return list(values)
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor(list(values), dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
    return t.cpu().tolist()


def job_gbs(world: int, bytes_per_step: int, steps: int, max_ms: float) -> float:
    """Whole-job throughput: every rank's bytes over the slowest rank's time."""
    return world * bytes_per_step * steps / (max_ms / 1e3) / 1e9


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampled every 200 ms while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200", "-f", self.path],
                stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows),
                "power_w_max": max((float(r[3]) for r in rows
                                    if r[3].replace(".", "").isdigit()), default=None)}


# ----------------------------------------------------------------------------- our arm
class HotPath:
    """Device buffers and the C-ABI calls of one step."""

    def __init__(self, device, workload="full"):
        import torch
        import ln_backward_gb300 as tb
        from ln_backward_gb300 import synth
        self.tb, self.torch = tb, torch
        self.dev = device
        w = WORKLOADS[workload]
        shapes = synth.llama7b_shapes() if w["table"] == "llama7b" else synth.gpt2_small_shapes()
        sm_rows, ln_rows = w["sm_rows"], w["ln_rows"]
        self.st = synth.make_adamw_state(shapes, seed=0, device=device,
                                         grad_std=w["grad_std"], loss_scale=LOSS_SCALE)
        k = len(self.st.sizes)
        self.plan = tb.tb_adamw_plan_create(*[[self.st.tensor(a, i) for i in range(k)]
                                              for a in ("theta", "m", "v", "grad", "copy")])
        self.P32, self.dY32 = synth.softmax_inputs(sm_rows, SM_COLS, torch.float32, seed=1,
                                                   device=device, causal_period=1024)
        self.P16, self.dY16 = synth.softmax_inputs(sm_rows, SM_COLS, torch.bfloat16, seed=2,
                                                   device=device, causal_period=1024)
        self.dX32 = torch.empty_like(self.P32)
        self.dX16 = torch.empty_like(self.P16)
        (self.x, self.ldY, self.mean, self.rstd,
         self.gamma) = synth.layernorm_inputs(ln_rows, LN_D, torch.bfloat16, seed=3, device=device,
                                              eps=1e-5, dy_std=1e-2)
        self.ldX = torch.empty_like(self.x)
        self.dg = torch.empty(LN_D, device=device)
        self.db = torch.empty(LN_D, device=device)
        ws = tb.tb_layernorm_bwd_workspace_size(ln_rows, LN_D, torch.bfloat16)
        self.ws = torch.empty(ws, dtype=torch.uint8, device=device)
        self.t = 0
        self.n_params = self.st.n_params
        self.bytes = {
            "adamw": adamw_bytes(self.n_params),
            "softmax_f32": softmax_bytes(sm_rows, SM_COLS, 4),
            "softmax_bf16": softmax_bytes(sm_rows, SM_COLS, 2),
            "layernorm_bf16": layernorm_bytes(ln_rows, LN_D, 2),
        }
        self.launches_per_step = 1 + 1 + 1 + 2
        self.sm_rows, self.ln_rows = sm_rows, ln_rows
        # Inputs of the rows beyond the timed step (measured separately).
        (self.rx, self.rdY, self.rinv, self.rgamma) = synth.rmsnorm_inputs(
            ln_rows, LN_D, torch.bfloat16, seed=4, device=device, dy_std=1e-2)
        self.rdX = torch.empty_like(self.rx)
        self.rdg = torch.empty(LN_D, device=device)
        self.rws = torch.empty(tb.tb_rmsnorm_bwd_workspace_size(ln_rows, LN_D, torch.bfloat16),
                               dtype=torch.uint8, device=device)
        # the pages' unfused tail: fp32 gradients, a plan without working copies
        self.g32 = torch.zeros(self.st.grad.numel(), dtype=torch.float32, device=device)
        self.plan32 = tb.tb_adamw_plan_create(
            [self.st.tensor("theta", i) for i in range(k)], [self.st.tensor("m", i) for i in range(k)],
            [self.st.tensor("v", i) for i in range(k)],
            [self.g32.narrow(0, self.st.offsets[i], self.st.sizes[i]) for i in range(k)],
            [None] * k)
        self.clip = torch.zeros(3, device=device)
        self.nws = torch.empty(tb.tb_adamw_grad_norm_workspace_size(self.plan), dtype=torch.uint8,
                               device=device)
        self._bwd = list(self.backward().values())

    def extras(self):
        """name -> (callable, algorithmic bytes) for the kernels outside the step."""
        tb = self.tb
        return {
            "softmax_causal_f32": (lambda: tb.tb_softmax_bwd_causal(self.dY32, self.P32, self.dX32,
                                                                    period=1024),
                                   causal_softmax_bytes(self.sm_rows, SM_COLS, 1024, 0, 4)),
            "softmax_causal_bf16": (lambda: tb.tb_softmax_bwd_causal(self.dY16, self.P16, self.dX16,
                                                                     period=1024),
                                    causal_softmax_bytes(self.sm_rows, SM_COLS, 1024, 0, 2)),
            "rmsnorm_bf16": (lambda: tb.tb_rmsnorm_bwd(self.rdY, self.rx, self.rinv, self.rgamma,
                                                       self.rdX, self.rdg, self.rws),
                             rmsnorm_bytes(self.ln_rows, LN_D, 2)),
            "adamw_grad_norm": (lambda: tb.tb_adamw_grad_norm(self.plan, 1.0 / LOSS_SCALE, 1.0,
                                                              self.clip, self.nws),
                                2 * self.n_params),
            "adamw_step_clipped": (lambda: tb.tb_adamw_step_clipped(
                self.plan, self.t + 1, inv_loss_scale=1.0 / LOSS_SCALE, clip=self.clip, **HP),
                adamw_bytes(self.n_params)),
            # cast 16-bit grad -> fp32 (6 B) + AdamW on fp32 grads (32 B) + cast copy (6 B)
            "unfused_adamw_pipeline": (self._unfused, 44 * self.n_params),
        }

    def _unfused(self):
        """The pages' unfused optimizer tail, for comparison with the fused step."""
        tb = self.tb
        tb.tb_cast_to_f32(self.st.grad, self.g32, scale=1.0 / LOSS_SCALE)
        tb.tb_adamw_step(self.plan32, self.t + 1, inv_loss_scale=1.0, **HP)
        tb.tb_cast_from_f32(self.st.theta, self.st.copy)

    def backward(self):
        """name -> callable of the backward kernels of the step, in step order."""
        tb = self.tb
        return {
            "softmax_f32": lambda: tb.tb_softmax_bwd(self.dY32, self.P32, self.dX32),
            "softmax_bf16": lambda: tb.tb_softmax_bwd(self.dY16, self.P16, self.dX16),
            "layernorm_bf16": lambda: tb.tb_layernorm_bwd(self.ldY, self.x, self.mean, self.rstd,
                                                          self.gamma, self.ldX, self.dg, self.db,
                                                          self.ws),
        }

    def step(self, events=None):
        """One step.  `events` (two CUDA events, or None) bracket the AdamW launch only:
        an event recorded between two kernels makes the second wait for the first to
        complete and flush before it is even placed, so the backward kernels run back
        to back, as in a training step, and each overlaps its set-up with the drain of
        the one before it (programmatic dependent launch)."""
        tb = self.tb
        self.t += 1
        if events is not None:
            events[0].record()
        tb.tb_adamw_step(self.plan, self.t, inv_loss_scale=1.0 / LOSS_SCALE, **HP)
        if events is not None:
            events[1].record()
        for fn in self._bwd:
            fn()


def run_ours(args):
    import torch
    import torch.distributed as dist
    world, rank, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    hp_path = HotPath(dev, args.workload)
    names = ["adamw", "softmax_f32", "softmax_bf16", "layernorm_bf16"]
    K, W = args.steps, args.warmup

    for _ in range(W):
        hp_path.step()
    torch.cuda.synchronize()
    if hp_path.tb.tb_device_error(reset=True) != 0:
        raise RuntimeError("a kernel's bounded wait gave up during warm-up")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    wall0 = time.perf_counter()
    start.record()
    for k in range(K):
        hp_path.step(evs[k])
    end.record()
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    barrier()
    clk = clocks.stop()
    total_ms = start.elapsed_time(end)
    adamw_ms = statistics.fmean(evs[k][0].elapsed_time(evs[k][1]) for k in range(K))
    # the backward kernels of step k run from AdamW's end to the start of step k+1
    bwd_ms = statistics.fmean(evs[k][1].elapsed_time(evs[k + 1][0] if k + 1 < K else end)
                              for k in range(K))
    total_ms, adamw_ms, bwd_ms = reduce_over_ranks([total_ms, adamw_ms, bwd_ms], "max")
    # each backward kernel on its own: a loop of back-to-back calls after the timed region
    iso = {n: time_loop(fn, reps=max(K, 20)) for n, fn in hp_path.backward().items()}
    mean_ms = dict(adamw=adamw_ms, **iso)

    step_bytes = sum(hp_path.bytes.values())
    value = job_gbs(world, step_bytes, K, total_ms)
    peak, peak_kind = measured_peak()
    kernels = {}
    for n in names:
        gbs = hp_path.bytes[n] / (mean_ms[n] / 1e3) / 1e9
        kernels[n] = {"ms": round(mean_ms[n], 4), "GB_s": round(gbs, 1),
                      "frac_of_peak": round(gbs / peak, 4), "bytes": hp_path.bytes[n],
                      "timing": "in step" if n == "adamw" else "back-to-back calls"}
    kernels["adamw"]["gparams_s"] = round(hp_path.n_params / (mean_ms["adamw"] / 1e3) / 1e9, 2)
    bwd_bytes = step_bytes - hp_path.bytes["adamw"]
    backward_in_step = {"ms": round(bwd_ms, 4),
                        "GB_s": round(bwd_bytes / (bwd_ms / 1e3) / 1e9, 1),
                        "frac_of_peak": round(bwd_bytes / (bwd_ms / 1e3) / 1e9 / peak, 4),
                        "bytes": bwd_bytes,
                        "sum_of_back_to_back_ms": round(sum(iso.values()), 4)}
    ad_gbs = kernels["adamw"]["GB_s"]

    extras = (None if args.no_extras
              else time_extras(hp_path, reps=max(K, 10), peak=measured_peak()[0]))
    e2e = run_e2e(hp_path, K) if not args.no_e2e else None
    if e2e is not None:
        e2e_ms = reduce_over_ranks([e2e.pop("ms")], "max")[0]
        e2e["value"] = round(job_gbs(world, step_bytes, K, e2e_ms), 1)
        # a pipelined step can be no shorter than its copies in both directions at
        # once, nor than its kernels: the floor, and how close the loop came to it
        floor_ms = max(e2e["link"]["both_ms"], total_ms / K)
        e2e["step_ms"] = round(e2e_ms / K, 2)
        e2e["floor_ms"] = round(floor_ms, 2)
        e2e["frac_of_floor"] = round(floor_ms / (e2e_ms / K), 3)

    cpu = None
    if world == 1 and rank == 0 and not args.no_cpu_baseline and args.workload == "full":
        cpu = cpu_baseline(seconds_budget=args.cpu_seconds)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "GB/s",
            "n_gpus": world, "steps": K, "warmup": W,
            "ms_per_step": round(total_ms / K, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": config_block(args.workload, world, step_bytes),
            "wall_s_timed_region": round(wall, 3),
            "kernels": kernels,
            "backward_in_step": backward_in_step,
            "extras": extras,
            "roofline": {"bound": "hbm", "achieved": ad_gbs, "peak": peak, "unit": "GB/s",
                         "frac": round(ad_gbs / peak, 4),
                         "traffic": ADAMW_TRAFFIC_PER_LAUNCH if args.workload == "full" else None,
                         "kernel": "adamw_multi_tensor_kernel", "peak_source": peak_kind},
            "clocks": clk,
            "gpu_launches": hp_path.launches_per_step * K,
            "e2e": e2e,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


# Per-launch DRAM bytes (read + write) of the AdamW kernel at the 7B workload, or None
# while no capture of the current kernel exists.  Must go back to None whenever the
# kernel changes until it is captured again.  From one ncu capture of the kernel on
# the GPT-2-small table (124,439,808 params): 1,742,311,168 B read, 1,930,455,552 B
# written.  Reads scale with the parameter count (14.0012 B/param); writes are
# 16 B/param less a fixed 60,581,376 B still dirty in L2 when the kernel ends.  At
# 6,738,415,616 params: 94.346 + 107.754 GB.
ADAMW_TRAFFIC_PER_LAUNCH = 202.100218406e9


def config_block(workload, world, step_bytes):
    """The `config` object of both arms: the workload only, no measured values."""
    return {"workload": WORKLOAD_TEXT[workload],
            "bytes_per_step": step_bytes,
            "l2": "no flush: every launch streams far more than the 129 MB L2",
            "parallelism": f"replicas x{world}"}


def time_loop(fn, reps, name=None):
    """Mean ms per call of `fn` in a loop of `reps` back-to-back calls (CUDA events
    on the current stream, after 3 untimed calls), max over ranks."""
    import torch
    if name:
        torch.cuda.nvtx.range_push(name)     # lets a profiler pick this kernel's launches
    for _ in range(3):
        fn()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    s.record()
    for _ in range(reps):
        fn()
    e.record()
    torch.cuda.synchronize()
    if name:
        torch.cuda.nvtx.range_pop()
    return reduce_over_ranks([s.elapsed_time(e) / reps], "max")[0]


def time_extras(hp_path, reps, peak):
    """Per-kernel CUDA-event timing of the kernels that are not part of the step."""
    out = {}
    for name, (fn, nbytes) in hp_path.extras().items():
        ms = time_loop(fn, reps, name)
        gbs = nbytes / (ms / 1e3) / 1e9
        out[name] = {"ms": round(ms, 4), "GB_s": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4),
                     "bytes": nbytes}
    return out


E2E_BUFFER_SETS = 2


def run_e2e(hp_path, K):
    """Same step through the public API, starting from pinned host buffers: every step
    copies its gradients and activations host->device, runs the kernels and copies the
    working copy and every backward output device->host.  Steps are pipelined the way a
    training loop would overlap them: the inputs of step k+1 go up on one stream while
    step k computes on a second and the results of step k-1 come down on a third, with
    E2E_BUFFER_SETS device buffers for every copied tensor (as many AdamW plans over the
    same theta/m/v).  (Three sets, which let uploads start a step earlier, measured
    slower than two on the same box: e2e 1,744 and 1,370 against 1,884 and 1,628 GB/s.)
    The timed region spans all K steps, copies included."""
    import torch
    tb, st = hp_path.tb, hp_path.st
    k_t = len(st.sizes)
    pin = dict(pin_memory=True)
    nb = E2E_BUFFER_SETS
    # device side: buffer set 0 is the step's own tensors, the others copies of them
    grads = [st.grad] + [torch.empty_like(st.grad) for _ in range(nb - 1)]
    copies = [st.copy] + [torch.empty_like(st.copy) for _ in range(nb - 1)]
    ins0 = [hp_path.P32, hp_path.dY32, hp_path.P16, hp_path.dY16, hp_path.x, hp_path.ldY,
            hp_path.mean, hp_path.rstd]
    outs0 = [hp_path.dX32, hp_path.dX16, hp_path.ldX, hp_path.dg, hp_path.db]
    ins = [ins0] + [[torch.empty_like(t) for t in ins0] for _ in range(nb - 1)]
    outs = [outs0] + [[torch.empty_like(t) for t in outs0] for _ in range(nb - 1)]
    plans = [hp_path.plan] + [tb.tb_adamw_plan_create(
        *[[st.tensor(a, i) for i in range(k_t)] for a in ("theta", "m", "v")],
        [grads[b].narrow(0, st.offsets[i], st.sizes[i]) for i in range(k_t)],
        [copies[b].narrow(0, st.offsets[i], st.sizes[i]) for i in range(k_t)])
        for b in range(1, nb)]
    ws = [hp_path.ws] + [torch.empty_like(hp_path.ws) for _ in range(nb - 1)]
    # host side
    h_grad = torch.empty_like(st.grad, device="cpu", **pin)
    h_grad.copy_(st.grad)
    h_ins = [torch.empty_like(t, device="cpu", **pin) for t in ins0]
    for h, t in zip(h_ins, ins0):
        h.copy_(t)
    h_copy = torch.empty_like(st.copy, device="cpu", **pin)
    h_outs = [torch.empty_like(t, device="cpu", **pin) for t in outs0]
    h2d = h_grad.numel() * h_grad.element_size() + sum(h.numel() * h.element_size() for h in h_ins)
    d2h = h_copy.numel() * h_copy.element_size() + sum(h.numel() * h.element_size() for h in h_outs)

    s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()

    def run(n_steps, t0):
        in_done, cmp_done, out_done = {}, {}, {}

        def upload(k):
            b = k % nb
            with torch.cuda.stream(s_in):
                if k - nb in cmp_done:       # step k-nb has finished reading set b
                    s_in.wait_event(cmp_done[k - nb])
                grads[b].copy_(h_grad, non_blocking=True)
                for d, h in zip(ins[b], h_ins):
                    d.copy_(h, non_blocking=True)
                in_done[k] = ev()
                in_done[k].record(s_in)

        upload(0)
        for k in range(n_steps):
            b = k % nb
            if k + 1 < n_steps:
                upload(k + 1)
            with torch.cuda.stream(s_cmp):
                s_cmp.wait_event(in_done[k])
                if k - nb in out_done:       # the results of step k-nb (set b) are down
                    s_cmp.wait_event(out_done[k - nb])
                tb.tb_adamw_step(plans[b], t0 + k, inv_loss_scale=1.0 / LOSS_SCALE, **HP)
                tb.tb_softmax_bwd(ins[b][1], ins[b][0], outs[b][0])
                tb.tb_softmax_bwd(ins[b][3], ins[b][2], outs[b][1])
                tb.tb_layernorm_bwd(ins[b][5], ins[b][4], ins[b][6], ins[b][7], hp_path.gamma,
                                    outs[b][2], outs[b][3], outs[b][4], ws[b])
                cmp_done[k] = ev()
                cmp_done[k].record(s_cmp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(cmp_done[k])
                h_copy.copy_(copies[b], non_blocking=True)
                for h, d in zip(h_outs, outs[b]):
                    h.copy_(d, non_blocking=True)
                out_done[k] = ev()
                out_done[k].record(s_out)
        return out_done[n_steps - 1]

    cur = torch.cuda.current_stream()
    torch.cuda.synchronize()
    run(nb, hp_path.t + 1)                   # warm-up: every buffer set, all streams
    hp_path.t += nb
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    s.record(cur)
    for q in (s_in, s_cmp, s_out):
        q.wait_event(s)
    last = run(K, hp_path.t + 1)
    hp_path.t += K
    cur.wait_stream(s_in)
    cur.wait_stream(s_cmp)
    cur.wait_event(last)
    e.record(cur)
    torch.cuda.synchronize()
    barrier()
    for pl in plans[1:]:
        pl.close()

    # The host link on its own, with the same buffers: one step's uploads, its
    # downloads, and both at once (best of three each, after the timed region).
    def link_ms(up, down):
        best = float("inf")
        for _ in range(3):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            a.record(cur)
            for q in (s_in, s_out):
                q.wait_event(a)
            if up:
                with torch.cuda.stream(s_in):
                    grads[0].copy_(h_grad, non_blocking=True)
                    for d, h in zip(ins[0], h_ins):
                        d.copy_(h, non_blocking=True)
            if down:
                with torch.cuda.stream(s_out):
                    h_copy.copy_(copies[0], non_blocking=True)
                    for h, d in zip(h_outs, outs[0]):
                        h.copy_(d, non_blocking=True)
            cur.wait_stream(s_in)
            cur.wait_stream(s_out)
            b.record(cur)
            torch.cuda.synchronize()
            best = min(best, a.elapsed_time(b))
        return best

    up_ms, down_ms, both_ms = link_ms(True, False), link_ms(False, True), link_ms(True, True)
    return {"ms": s.elapsed_time(e), "unit": "GB/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h,
            "link": {"h2d_ms": round(up_ms, 2), "d2h_ms": round(down_ms, 2),
                     "both_ms": round(both_ms, 2),
                     "h2d_GB_s": round(h2d / up_ms / 1e6, 1),
                     "d2h_GB_s": round(d2h / down_ms / 1e6, 1),
                     "both_GB_s": round((h2d + d2h) / both_ms / 1e6, 1)},
            "note": "algorithmic HBM bytes per step / step time of a pipelined loop whose every "
                    "step copies its gradients and activations up from pinned host memory and "
                    "its bf16 working copy and backward outputs back down (three streams, "
                    f"{nb} device buffer sets)"}


# ----------------------------------------------------------------------------- CPU oracle
LLAMA7B_PARAMS = 6_738_415_616
FULL_STEP_BYTES = (adamw_bytes(LLAMA7B_PARAMS) + softmax_bytes(SM_ROWS, SM_COLS, 4)
                   + softmax_bytes(SM_ROWS, SM_COLS, 2) + layernorm_bytes(LN_ROWS, LN_D, 2))
# The CPU oracle runs on a proportional sample of the full step: 1/64 of the AdamW
# parameters, of the softmax rows (fp32 and bf16 instances) and of the LayerNorm rows.
# Every term of the step's byte count divides by 64, so a sample step stands for
# exactly FULL_STEP_BYTES / 64 algorithmic bytes.
SAMPLE_DIV = 64
SAMPLE_BYTES = FULL_STEP_BYTES // SAMPLE_DIV
assert SAMPLE_BYTES * SAMPLE_DIV == FULL_STEP_BYTES


def host_cpu():
    """Core count and CPU model of this host (lscpu where available)."""
    info = {"cpu_count": os.cpu_count()}
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            k, _, v = line.partition(":")
            k, v = k.strip(), v.strip()
            if k in ("Model name", "Socket(s)", "Architecture", "Thread(s) per core"):
                info[k.lower().replace("(s)", "s").replace(" ", "_")] = v
    except Exception:
        pass
    return info


class OracleSample:
    """Inputs of one sample step of the CPU oracle, cut into `threads` disjoint slices
    (contiguous parameter ranges and row blocks).  A sample step calls the float64 C
    oracle on every slice, one Python thread per slice (ctypes releases the GIL, so
    the slices run on separate cores), and stands for SAMPLE_BYTES of the workload."""

    def __init__(self, threads):
        import numpy as np
        import oracle
        oracle.build()
        self.oracle = oracle
        self.threads = threads
        rng = np.random.default_rng(0)
        n = LLAMA7B_PARAMS // SAMPLE_DIV
        self.th = rng.standard_normal(n) * 0.02
        self.m = np.zeros(n)
        self.v = np.zeros(n)
        self.g = oracle.encode16(rng.standard_normal(n) * 1e-4 * LOSS_SCALE, "bf16")
        sm_rows = 2 * SM_ROWS // SAMPLE_DIV          # the fp32 and the bf16 instance
        self.P = rng.random((sm_rows, SM_COLS))
        self.P /= self.P.sum(axis=1, keepdims=True)
        self.sdY = rng.standard_normal((sm_rows, SM_COLS))
        ln_rows = LN_ROWS // SAMPLE_DIV
        self.x = rng.standard_normal((ln_rows, LN_D))
        self.ldY = rng.standard_normal((ln_rows, LN_D)) * 1e-2
        self.mu = self.x.mean(axis=1)
        self.rs = 1.0 / np.sqrt(self.x.var(axis=1) + 1e-5)
        self.gam = 1.0 + 0.1 * rng.standard_normal(LN_D)
        cut = lambda total: [total * i // threads for i in range(threads + 1)]
        self.pa, self.ps, self.pl = cut(n), cut(sm_rows), cut(ln_rows)
        self.t = 0
        self._pool = None
        if threads > 1:
            import concurrent.futures as cf
            self._pool = cf.ThreadPoolExecutor(max_workers=threads)

    def _slice(self, i, t):
        o = self.oracle
        a0, a1 = self.pa[i], self.pa[i + 1]
        o.adamw_step_f64(self.th[a0:a1], self.m[a0:a1], self.v[a0:a1], self.g[a0:a1], "bf16",
                         1.0 / LOSS_SCALE, t, **HP)
        s0, s1 = self.ps[i], self.ps[i + 1]
        if s1 > s0:
            o.softmax_bwd_f64(self.sdY[s0:s1], self.P[s0:s1])
        l0, l1 = self.pl[i], self.pl[i + 1]
        if l1 > l0:
            o.layernorm_bwd_f64(self.ldY[l0:l1], self.x[l0:l1], self.mu[l0:l1], self.rs[l0:l1],
                                self.gam)

    def step(self):
        """One sample step; returns its wall time in seconds."""
        self.t += 1
        t0 = time.perf_counter()
        if self._pool is None:
            self._slice(0, self.t)
        else:
            list(self._pool.map(lambda i: self._slice(i, self.t), range(self.threads)))
        return time.perf_counter() - t0

    def close(self):
        if self._pool is not None:
            self._pool.shutdown()


def cpu_baseline(seconds_budget=15.0):
    """The oracle on this host's cores: sample steps on every core, then one on a
    single core.  GB/s = SAMPLE_BYTES per sample step over its wall time."""
    host = host_cpu()
    threads = max(1, host["cpu_count"] or 1)
    smp = OracleSample(threads)
    smp.step()                                   # untimed: first touch of every page
    times = []
    t_end = time.perf_counter() + 0.6 * seconds_budget
    while len(times) < 3 or (time.perf_counter() < t_end and len(times) < 20):
        times.append(smp.step())
    smp.close()
    ms = statistics.fmean(times) * 1e3
    one = OracleSample(1)
    one_ms = one.step() * 1e3
    gbs = SAMPLE_BYTES / (ms / 1e3) / 1e9
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": (f"float64 C oracle on 1/{SAMPLE_DIV} of the step ({LLAMA7B_PARAMS // SAMPLE_DIV:,} "
                       f"AdamW params, {2 * SM_ROWS // SAMPLE_DIV} softmax rows of {SM_COLS}, "
                       f"{LN_ROWS // SAMPLE_DIV} LayerNorm rows of {LN_D}) cut into {threads} "
                       f"disjoint slices, one thread each; {len(times)} sample steps of "
                       f"{ms:.0f} ms"),
            "ms_per_sample_step": round(ms, 1),
            "full_step_s_extrapolated": round(ms * SAMPLE_DIV / 1e3, 1),
            "single_thread": {"value": round(SAMPLE_BYTES / (one_ms / 1e3) / 1e9, 4), "cores": 1,
                              "ms_per_sample_step": round(one_ms, 1)},
            "host": host}


def run_reference(args):
    """The reference arm: the CPU oracle (float64 C, plain loops) on this host's cores,
    one sample step (1/SAMPLE_DIV of the workload) per step."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    host = host_cpu()
    threads = max(1, host["cpu_count"] or 1)
    smp = OracleSample(threads)
    for _ in range(args.warmup):
        smp.step()
    t0 = time.perf_counter()
    times = [smp.step() for _ in range(args.steps)]
    wall = time.perf_counter() - t0
    smp.close()
    ms = statistics.fmean(times) * 1e3
    gbs = SAMPLE_BYTES / (ms / 1e3) / 1e9
    line = {
        "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "impl": "reference",
        "config": config_block("full", world, FULL_STEP_BYTES),
        "sample_bytes_per_step": SAMPLE_BYTES,
        "wall_s_timed_region": round(wall, 3),
        "full_step_s_extrapolated": round(ms * SAMPLE_DIV / 1e3, 1),
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": (f"each step: float64 C oracle on 1/{SAMPLE_DIV} of the full step "
                                    f"({LLAMA7B_PARAMS // SAMPLE_DIV:,} AdamW params, "
                                    f"{2 * SM_ROWS // SAMPLE_DIV} softmax rows, "
                                    f"{LN_ROWS // SAMPLE_DIV} LayerNorm rows) in {threads} "
                                    f"disjoint slices, one thread each"),
                         "host": host},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def run_layernorm_sweep(args):
    """LayerNorm (and RMSNorm) backward at D = 4096 over a range of row counts, and a
    least-squares fit time = bytes / BW + F that separates the streaming rate from the
    fixed cost of a call.  One JSON line per dtype; not part of the benchmark contract."""
    import numpy as np
    import torch
    import ln_backward_gb300 as tb
    from ln_backward_gb300 import synth
    dev = torch.device("cuda")
    D = LN_D

    def best_ms(fn, reps=30):
        for _ in range(5):
            fn()
        torch.cuda.synchronize()
        best = float("inf")
        for _ in range(3):
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record()
            for _ in range(reps):
                fn()
            e.record()
            torch.cuda.synchronize()
            best = min(best, s.elapsed_time(e) / reps)
        return best

    for op in ("layernorm", "rmsnorm"):
        for dt in (torch.bfloat16, torch.float32):
            es = torch.empty((), dtype=dt).element_size()
            pts = []
            for rows in (2048, 4096, 8192, 16384, 32768, 65536, 131072):
                dg = torch.empty(D, device=dev)
                if op == "layernorm":
                    x, dy, mu, rs, g = synth.layernorm_inputs(rows, D, dt, 3, dev, dy_std=1e-2)
                    dX, db = torch.empty_like(x), torch.empty(D, device=dev)
                    ws = torch.empty(tb.tb_layernorm_bwd_workspace_size(rows, D, dt),
                                     dtype=torch.uint8, device=dev)
                    fn = lambda: tb.tb_layernorm_bwd(dy, x, mu, rs, g, dX, dg, db, ws)
                    nbytes = layernorm_bytes(rows, D, es)
                else:
                    x, dy, inv, g = synth.rmsnorm_inputs(rows, D, dt, 4, dev, dy_std=1e-2)
                    dX = torch.empty_like(x)
                    ws = torch.empty(tb.tb_rmsnorm_bwd_workspace_size(rows, D, dt),
                                     dtype=torch.uint8, device=dev)
                    fn = lambda: tb.tb_rmsnorm_bwd(dy, x, inv, g, dX, dg, ws)
                    nbytes = rmsnorm_bytes(rows, D, es)
                ms = best_ms(fn)
                pts.append((rows, nbytes, ms))
                del x, dy, dX, ws
                torch.cuda.empty_cache()
            A = np.array([[b, 1.0] for _, b, _ in pts])
            (inv_bw, fixed), *_ = np.linalg.lstsq(A, np.array([ms * 1e-3 for _, _, ms in pts]),
                                                  rcond=None)
            print(json.dumps({
                "sweep": f"{op}_bwd", "dtype": str(dt).replace("torch.", ""), "D": D,
                "points": [{"rows": r, "us": round(ms * 1e3, 1), "GB_s": round(b / ms / 1e6, 1)}
                           for r, b, ms in pts],
                "fit_streaming_GB_s": round(1.0 / inv_bw / 1e9, 1),
                "fit_fixed_us": round(fixed * 1e6, 2)}))
    if tb.tb_device_error(reset=True) != 0:
        raise RuntimeError("a kernel's bounded wait gave up during the sweep")


HIDDEN_SWEEP_SHAPES = ("bf16:256,bf16:512,bf16:768,bf16:1024,bf16:1536,bf16:2048,bf16:4096,"
                       "bf16:5120,bf16:6144,bf16:8192,bf16:10240,bf16:12288,bf16:16384,"
                       "bf16:20480,bf16:32768,f32:768,f32:1024,f32:4096,f32:5120,f32:8192,"
                       "f32:12288,f32:16384")


def sweep_best_ms(fn, reps):
    """Best of three CUDA-event timings of `reps` back-to-back calls, after three warm-up
    calls, in ms per call (the hidden-size and causal sweeps)."""
    import torch
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    best = float("inf")
    for _ in range(3):
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        for _ in range(reps):
            fn()
        e.record()
        torch.cuda.synchronize()
        best = min(best, s.elapsed_time(e) / reps)
    return best


def run_hidden_sweep(args):
    """LayerNorm and RMSNorm backward over hidden sizes D, each with as many rows as
    make one input tensor args.sweep_mb MB: the short-row ring, the 512-thread ring
    and the cluster-split path in turn.  One JSON line per op, dtype and D; not part
    of the benchmark contract.  With --sweep-reps 0 each shape is called once,
    untimed (for profiler captures)."""
    import torch
    import ln_backward_gb300 as tb
    from ln_backward_gb300 import synth
    dev = torch.device("cuda")
    peak, peak_kind = measured_peak()
    dtypes = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}

    for item in (args.sweep_shapes or HIDDEN_SWEEP_SHAPES).split(","):
        name, d = item.split(":")
        dt, D = dtypes[name], int(d)
        es = torch.empty((), dtype=dt).element_size()
        rows = max(1, (args.sweep_mb << 20) // (D * es))
        x, dy, mu, rs, g = synth.layernorm_inputs(rows, D, dt, 3, dev, eps=1e-5, dy_std=1e-2)
        dX = torch.empty_like(x)
        dg, db = torch.empty(D, device=dev), torch.empty(D, device=dev)
        ws = torch.empty(tb.tb_layernorm_bwd_workspace_size(rows, D, dt), dtype=torch.uint8,
                         device=dev)
        wr = torch.empty(tb.tb_rmsnorm_bwd_workspace_size(rows, D, dt), dtype=torch.uint8,
                         device=dev)
        ops = (("layernorm_bwd", lambda: tb.tb_layernorm_bwd(dy, x, mu, rs, g, dX, dg, db, ws),
                layernorm_bytes(rows, D, es)),
               ("rmsnorm_bwd", lambda: tb.tb_rmsnorm_bwd(dy, x, rs, g, dX, dg, wr),
                rmsnorm_bytes(rows, D, es)))
        for op, fn, nbytes in ops:
            if args.sweep_reps == 0:
                fn()
                torch.cuda.synchronize()
                continue
            ms = sweep_best_ms(fn, args.sweep_reps)
            gbs = nbytes / ms / 1e6
            print(json.dumps({"sweep": "hidden", "op": op, "dtype": name, "D": D, "rows": rows,
                              "us": round(ms * 1e3, 1), "GB_s": round(gbs, 1),
                              "frac": round(gbs / peak, 3), "peak": f"{peak:.1f} ({peak_kind})"}))
        del x, dy, dX, ws, wr
        torch.cuda.empty_cache()
    if tb.tb_device_error(reset=True) != 0:
        raise RuntimeError("a kernel's bounded wait gave up during the sweep")


CAUSAL_SWEEP_SHAPES = ("bf16:256,bf16:512,bf16:768,bf16:1024,bf16:2048,bf16:3072,bf16:4096,"
                       "bf16:8192,bf16:12288,bf16:16384,f16:1024,f16:4096,f32:512,f32:1024,"
                       "f32:2048,f32:4096,f32:8192")


def run_causal_sweep(args):
    """Causal softmax backward over sequence lengths S: rows of S columns in whole S x S
    causal blocks (period S; as many blocks as make one input tensor args.sweep_mb MB, at
    least one), with the dense call on the same tensors beside it.  One JSON line per
    dtype and S; not part of the benchmark contract.  With --sweep-reps 0 each shape is
    called once, untimed (for profiler captures)."""
    import torch
    import ln_backward_gb300 as tb
    from ln_backward_gb300 import synth
    dev = torch.device("cuda")
    peak, peak_kind = measured_peak()
    dtypes = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}
    for item in (args.sweep_shapes or CAUSAL_SWEEP_SHAPES).split(","):
        name, s = item.split(":")
        dt, S = dtypes[name], int(s)
        es = torch.empty((), dtype=dt).element_size()
        rows = S * max(1, (args.sweep_mb << 20) // (S * S * es))
        P, dY = synth.softmax_inputs(rows, S, dt, seed=S, device=dev, causal_period=S)
        dX = torch.empty_like(P)
        causal = lambda: tb.tb_softmax_bwd_causal(dY, P, dX, period=S)
        dense = lambda: tb.tb_softmax_bwd(dY, P, dX)
        if args.sweep_reps == 0:
            causal()
            dense()
            torch.cuda.synchronize()
        else:
            cb = causal_softmax_bytes(rows, S, S, 0, es)
            db = softmax_bytes(rows, S, es)
            cms = sweep_best_ms(causal, args.sweep_reps)
            dms = sweep_best_ms(dense, args.sweep_reps)
            print(json.dumps({"sweep": "causal_softmax", "dtype": name, "S": S, "rows": rows,
                              "us": round(cms * 1e3, 1), "GB_s": round(cb / cms / 1e6, 1),
                              "frac": round(cb / cms / 1e6 / peak, 3),
                              "dense_us": round(dms * 1e3, 1),
                              "dense_frac": round(db / dms / 1e6 / peak, 3),
                              "peak": f"{peak:.1f} ({peak_kind})"}))
        del P, dY, dX
        torch.cuda.empty_cache()
    if tb.tb_device_error(reset=True) != 0:
        raise RuntimeError("a kernel's bounded wait gave up during the sweep")


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip timing the kernels outside the step (for profiler launch lists)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="full")
    ap.add_argument("--sweep-layernorm", action="store_true",
                    help="time the LayerNorm/RMSNorm backward over row counts and fit "
                         "bytes/BW + fixed cost (one JSON line per op and dtype)")
    ap.add_argument("--sweep-hidden", action="store_true",
                    help="time the LayerNorm/RMSNorm backward over hidden sizes (one JSON "
                         "line per op, dtype and D)")
    ap.add_argument("--sweep-causal", action="store_true",
                    help="time the causal softmax backward over sequence lengths S (whole "
                         "S x S causal blocks; one JSON line per dtype and S)")
    ap.add_argument("--sweep-shapes", default=None,
                    help="dtype:D (or dtype:S) list for --sweep-hidden and --sweep-causal "
                         "(dtype bf16, f16 or f32)")
    ap.add_argument("--sweep-mb", type=int, default=256,
                    help="MB per input tensor for --sweep-hidden and --sweep-causal")
    ap.add_argument("--sweep-reps", type=int, default=20,
                    help="timed calls per repetition for the sweeps (0: one untimed call)")
    args = ap.parse_args(argv)
    if args.warmup < 1:
        ap.error("--warmup must be >= 1 (timed numbers use the default of 3)")
    if args.sweep_hidden:
        run_hidden_sweep(args)
    elif args.sweep_causal:
        run_causal_sweep(args)
    elif args.sweep_layernorm:
        run_layernorm_sweep(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
