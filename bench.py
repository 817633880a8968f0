"""Benchmark of the ZeRO per-rank mixed-precision AdamW step on GB300.

One step = the whole hot path over one rank's shard: pass 1 (unscale,
overflow, global squared norm), the decision kernel and pass 2 (clip, AdamW,
cast), all through the C ABI (zero_step on one GPU; zero_grad_norm_overflow,
the cross-rank sum and zero_adam_step on several).  Default workload: the
whole GPT-2 1.5B model state on one GPU (Nd = 1, 1,557,611,264 params
padded: 24.9 GB of fp16 gradient and parameters and fp32 master, momentum
and variance), fp16 gradients at loss scale 1, global-norm clipping at 1.0.
--workload gpt2_1p5b_nd16 runs one rank's shard of the same model in 16
ZeRO shards (97,350,784 params, x65536 loss scale).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

N > 1 (under torchrun): rank r updates shard r of the workload's layout and the
ranks sum their 16-byte (sum g^2, found_inf) partials with one all-reduce
between the passes: the one exchange of the step (weak scaling).
--impl reference times the oracle (plain scalar C, host cores) on a bounded
sample of the same workload.  Prints one JSON line (rank 0).
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
sys.path.insert(0, ROOT)

METRIC = "Adam-step params/sec & achieved HBM GB/s vs GB300 roofline (28 B/param), 1 GPU"
UNIT = "params/s"
# the default step: the largest single-GPU configuration, the whole GPT-2 1.5B
# state unpartitioned (24.9 GB of fp16 param/grad + fp32 master/m/v)
WORKLOAD = "gpt2_1p5b_full"
# the Nd = 16 layout of the same model: the shard the stage-2, stage-3 and
# 1-bit workloads use
SHARDED = "gpt2_1p5b_nd16"
TITLES = {
    "gpt2_1p5b_nd16": "GPT-2 1.5B state (48 layers, hidden 1600, vocab 50257) in 16 "
                      "ZeRO shards, one shard per GPU",
    "gpt2_1p5b_full": "GPT-2 1.5B state unpartitioned (Nd = 1) on one GPU, clip 1.0",
    "tiny": "2-layer hidden-256 transformer state (14 tensors), Nd = 1",
    "stack_100b_nd400": "100B GPT layer stack (125 x hidden 8192) in 400 ZeRO shards, "
                        "one shard; 4 bf16 micro-batch gradients accumulated, clip 1.0",
    "frag_10k": "10,000 separately allocated tensors (log-normal sizes, median 4096, "
                "max 2^24), unflattened multi-tensor path",
}


def step_config(title, w, S, l2, world=1):
    """The `config` of a step line: the workload and its shard, the same for
    both arms."""
    return {
        "workload": title,
        "shard_params": S, "grad_dtype": w["gdtype"], "param_dtype": w["pdtype"],
        "state_dtype": "f32", "loss_scale": w["loss_scale"], "clip": w["max_norm"],
        "micro_batches": w["micro_batches"], "l2": l2,
        "parallelism": f"zero-dp{world}" if world > 1 else "zero-shard",
    }


L2_BYTES = 129e6
# nominal HBM3e bandwidth of a GB300 (the fraction "of nominal")
NOMINAL_HBM_GBS = 7900.0
# the gradient tail pass 1 loads with evict-last priority for pass 2 (the
# library's choice for flat shards: 96 MiB)
KEEP_L2_BYTES = 96 << 20


def nvtx(call, *args):
    """torch.cuda.nvtx.range_push / range_pop, for a profiler's timeline; a
    torch built without NVTX raises RuntimeError, and the bench runs on."""
    import torch
    try:
        getattr(torch.cuda.nvtx, call)(*args)
    except RuntimeError:
        pass


def kernel_source_hash() -> str:
    """sha256 (first 16 hex) of the files that define passes 1 and 2: the
    kernel file and the headers it includes."""
    csrc = os.path.join(ROOT, "zero_partitioned_mixed_layout_gb300", "csrc")
    h = hashlib.sha256()
    for f in ("zero_pml.cu", "common.cuh", "zero_pml_internal.h"):
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def committed_traffic(workload: str = WORKLOAD):
    """DRAM bytes per pass-2 launch on `workload` from the committed ncu
    record (profiles/adam_pass2_<workload>_traffic.json), if it was taken on
    the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", f"adam_pass2_{workload}_traffic.json")
    try:
        d = json.load(open(path))
    except (OSError, ValueError):
        return None
    if d.get("kernel_source_sha256_16") != kernel_source_hash():
        return None
    return d.get("dram_bytes_per_launch")


def measured_peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.rows = []
        if self.proc is None:
            return False
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        for line in out.splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                self.rows.append(parts)
        return False

    def summary(self):
        if not getattr(self, "rows", None):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(self.rows)}


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


# ------------------------------------------------------------------ oracle arm

def _oracle_inputs(w, n_sample: int, seed: int):
    """A sample of the workload's inputs for the oracle: the master, zero
    moments, the stored gradient of step 0 (the workload's type and loss
    scale), the hyper-parameters (its clip threshold) and a fresh scaler."""
    import numpy as np

    import oracle
    import zero_synth as zs
    p = zs.host_master(n_sample, seed)
    m = np.zeros(n_sample, np.float32)
    v = np.zeros(n_sample, np.float32)
    plp = np.zeros(n_sample, np.uint16)
    g = zs.host_grad(n_sample, seed, 0, w["loss_scale"], w["gdtype"])
    hp = oracle.HParams(**zs.HPARAMS, max_norm=w["max_norm"])
    return p, m, v, plp, g, hp, oracle.Scaler(loss_scale=w["loss_scale"])


def oracle_workload(name: str) -> str:
    """The workload whose inputs the oracle legs draw: the timed one when it
    is a single-buffer flat step (one gradient array, the oracle's own full
    step), else the bench line's default."""
    import zero_synth as zs
    w = zs.WORKLOADS.get(name)
    return name if w is not None and w.get("micro_batches", 1) == 1 and name != "frag_10k" else WORKLOAD


def oracle_run(n_sample: int, steps: int, warmup: int, keep: bool = False, name: str = WORKLOAD):
    """The oracle as it stands (single-threaded scalar C) on the first
    n_sample elements of the workload's shard: `warmup` untimed and `steps`
    timed full steps (norm, decision, update).  Returns (params/s, seconds,
    the final (master, m, v, p_lp) arrays if `keep`, else None)."""
    import numpy as np

    import oracle
    import zero_synth as zs
    w = zs.WORKLOADS[name]
    oracle.build()
    p, m, v, plp, g, hp, sc = _oracle_inputs(w, n_sample, 0)
    gt, pt = w["gdtype"], w["pdtype"]
    for _ in range(warmup):
        oracle.adam_step([g], gt, [p], [m], [v], [plp], pt, hp, sc)
    t0 = time.perf_counter()
    for _ in range(steps):
        oracle.adam_step([g], gt, [p], [m], [v], [plp], pt, hp, sc)
    dt = time.perf_counter() - t0
    return n_sample * steps / dt, dt, ((p, m, v, plp) if keep else None)


def parity_vs_oracle(dev, n_sample: int, steps: int, final, name: str = WORKLOAD) -> dict:
    """The library on the oracle run's inputs (the same seeded arrays and
    hyper-parameters, the same number of steps), outside the timed region:
    its final state against the oracle's, element by element.  ulp distances
    of the fp32 arrays are counted on the ordered integer images of the
    values."""
    import numpy as np
    import torch

    import zero_partitioned_mixed_layout_gb300 as zp
    import zero_synth as zs
    w = zs.WORKLOADS[name]
    p = torch.from_numpy(zs.host_master(n_sample, 0)).to(dev)
    hg = zs.host_grad(n_sample, 0, 0, w["loss_scale"], w["gdtype"])
    g = torch.from_numpy(hg.view(np.int16)).view(torch.bfloat16).to(dev) if w["gdtype"] == "bf16" \
        else torch.from_numpy(hg).to(dev)
    m, v = torch.zeros_like(p), torch.zeros_like(p)
    plp = torch.zeros(n_sample, dtype={"f16": torch.float16, "bf16": torch.bfloat16}[w["pdtype"]], device=dev)
    state, ws = zp.new_state(w["loss_scale"], dev), zp.new_workspace(1, n_sample, dev)
    hp = zp.HParams(**zs.HPARAMS, max_norm=w["max_norm"])
    for _ in range(steps):
        zp.zero_step(g, p, m, v, plp, hp, state, ws)
    torch.cuda.synchronize(dev)

    def ordered(a):
        i = a.view(np.int32).astype(np.int64)
        return np.where(i < 0, -(i & 0x7FFFFFFF), i)

    out = {"elements": n_sample, "steps": steps}
    hist = {"0": 0, "1": 0, "2-4": 0, ">4": 0}
    for name, got, want in (("master", p, final[0]), ("m", m, final[1]), ("v", v, final[2])):
        a = got.cpu().numpy()
        d = np.abs(ordered(a) - ordered(want))
        out[f"{name}_bitwise_equal"] = bool(a.tobytes() == want.tobytes())
        err = np.abs(a.astype(np.float64) - want.astype(np.float64))
        out[f"{name}_max_abs_err"] = float(err.max())
        out[f"{name}_max_rel_err"] = float((err / np.maximum(np.abs(want.astype(np.float64)), 1e-300)).max())
        hist["0"] += int((d == 0).sum())
        hist["1"] += int((d == 1).sum())
        hist["2-4"] += int(((d >= 2) & (d <= 4)).sum())
        hist[">4"] += int((d > 4).sum())
    out["fp32_ulp_histogram"] = hist
    out["p_lp_bitwise_equal"] = bool(plp.cpu().view(torch.int16).numpy().view(np.uint16).tobytes()
                                     == final[3].tobytes())
    return out


def _oracle_worker(k, n_sample, steps, warmup, barrier, out, name=WORKLOAD):
    """One process of the all-core oracle timing: its own slice of inputs
    (seeded by its index), then steps in lockstep start with the others."""
    import numpy as np

    import oracle
    import zero_synth as zs
    w = zs.WORKLOADS[name]
    oracle.build()
    p, m, v, plp, g, hp, sc = _oracle_inputs(w, n_sample, k)
    gt, pt = w["gdtype"], w["pdtype"]
    for _ in range(warmup):
        oracle.adam_step([g], gt, [p], [m], [v], [plp], pt, hp, sc)
    barrier.wait()
    t0 = time.time()
    for _ in range(steps):
        oracle.adam_step([g], gt, [p], [m], [v], [plp], pt, hp, sc)
    out.put((k, t0, time.time()))


def oracle_run_all_cores(n_sample: int, steps: int, warmup: int, name: str = WORKLOAD):
    """The same single-threaded oracle on every host core at once: one
    process per core (started with spawn), each on its own n_sample
    elements; params/s = all processes' elements x steps / the wall time
    from the first start to the last finish.  Returns (params/s, seconds,
    processes)."""
    import multiprocessing as mp
    try:
        procs = len(os.sched_getaffinity(0))
    except AttributeError:
        procs = os.cpu_count() or 1
    ctx = mp.get_context("spawn")
    barrier, out = ctx.Barrier(procs), ctx.Queue()
    ps = [ctx.Process(target=_oracle_worker, args=(k, n_sample, steps, warmup, barrier, out, name))
          for k in range(procs)]
    for q in ps:
        q.start()
    res = [out.get(timeout=600) for _ in ps]
    for q in ps:
        q.join(timeout=60)
    wall = max(r[2] for r in res) - min(r[1] for r in res)
    return procs * n_sample * steps / wall, wall, procs


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    import zero_synth as zs
    name = oracle_workload(args.workload)
    w = zs.WORKLOADS[name]
    S = oracle.partition_layout(w["numel"](), w["nd"], w["align"]).shard_numel
    n_sample = min(1 << 24, S)
    one, one_dt, _ = oracle_run(n_sample, args.steps, args.warmup, name=name)
    value, dt, procs = oracle_run_all_cores(n_sample, args.steps, args.warmup, name=name)
    sample = (f"{procs} processes (one per host core), each on its own {n_sample} params of the "
              f"{name} rank-0 shard's inputs, {args.steps} timed steps after {args.warmup} "
              f"warm-up; full step (norm, decision, update) per step")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": dict(step_config(TITLES[name], w, S, "host cores: each process steps its own sample of the "
                                   "shard (the oracle does not use the GPU)", args.gpus),
                       sample_params=n_sample),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": procs, "kind": "oracle",
                         "sample": sample,
                         "single_core": {"value": one, "unit": UNIT, "cores": 1,
                                         "seconds": one_dt}},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ our arm

class Workload:
    """Device buffers and the step of one benchmark workload on one rank."""

    def __init__(self, name, log2n, rank, dev, prepared=False):
        import torch

        import zero_partitioned_mixed_layout_gb300 as zp
        import zero_synth as zs
        self.zp, self.name, self.dev = zp, name, dev
        if name == "flat":
            w = dict(zs.WORKLOADS["tiny"], nd=1, rank=0)
            numel = [1 << log2n]
            self.title = f"flat shard of 2^{log2n} params, fp16 grads x1024"
        else:
            w = zs.WORKLOADS[name]
            numel = w["numel"]()
            self.title = TITLES[name]
        self.w = w
        self.listmode = name == "frag_10k"
        shard = rank % w["nd"]
        seed = 1000 + shard
        self.scale = w["loss_scale"]
        gdt = {"f16": torch.float16, "bf16": torch.bfloat16}[w["gdtype"]]
        pdt = {"f16": torch.float16, "bf16": torch.bfloat16}[w["pdtype"]]
        self.micro = w["micro_batches"]
        if self.listmode:
            sizes = numel
            self.S = sum(sizes)
            flat_p = torch.empty(self.S, dtype=torch.float32, device=dev)
            zs.device_master_into(flat_p, seed)
            flat_g = torch.empty(self.S, dtype=gdt, device=dev)
            zs.device_grad_into(flat_g, seed, 0, self.scale)
            offs = [0]
            for n in sizes:
                offs.append(offs[-1] + n)
            # every tensor its own allocation, as an unflattened model's are
            p = [flat_p[offs[i]:offs[i + 1]].clone() for i in range(len(sizes))]
            g = [flat_g[offs[i]:offs[i + 1]].clone() for i in range(len(sizes))]
            del flat_p, flat_g
            self.p = zp.TensorList(p, "master")
            self.g = zp.TensorList(g, "grads")
            self.m = zp.TensorList([torch.zeros(n, device=dev) for n in sizes], "m")
            self.v = zp.TensorList([torch.zeros(n, device=dev) for n in sizes], "v")
            self.lp = zp.TensorList([torch.empty(n, dtype=pdt, device=dev) for n in sizes], "p_lp")
            self.ws = zp.new_workspace(len(sizes), self.S, dev)
            # prepared: the tables copied once, each step copies nothing
            self.plan = (zp.zero_list_prepare(self.g, self.p, self.m, self.v, self.lp, self.ws)
                         if prepared else None)
        else:
            lay = zp.zero_partition_layout(numel, w["nd"], w["align"])
            S = self.S = lay.shard_numel
            self.p = torch.empty(S, dtype=torch.float32, device=dev)
            zs.device_master_into(self.p, seed)
            self.m = torch.zeros(S, dtype=torch.float32, device=dev)
            self.v = torch.zeros(S, dtype=torch.float32, device=dev)
            self.lp = torch.empty(S, dtype=pdt, device=dev)
            if self.micro > 1:
                self.bufs = [torch.empty(S, dtype=gdt, device=dev) for _ in range(self.micro)]
                for j, b in enumerate(self.bufs):
                    zs.device_grad_into(b, seed, 0, self.scale, micro=j)
                self.g = torch.empty(S, dtype=torch.float32, device=dev)
            else:
                self.g = torch.empty(S, dtype=gdt, device=dev)
                zs.device_grad_into(self.g, seed, 0, self.scale)
            self.ws = zp.new_workspace(1, S, dev)
        self.state = zp.new_state(self.scale, dev)
        self.hp = zp.HParams(**zs.HPARAMS, max_norm=w["max_norm"])
        g_bytes = 4 if self.micro > 1 else 2
        p_bytes = 2
        # algorithmic bytes per param of pass 2 and of the whole step
        self.bytes_adam = g_bytes + 12 + 12 + p_bytes
        # micro-batches: the accumulation carries pass 1 (the fp32 sums are
        # not read back), so pass 1 adds no bytes of its own
        self.bytes_step = self.bytes_adam + (self.micro * 2 + 4 if self.micro > 1 else g_bytes)
        self.l2_resident = self.bytes_step * self.S < 2 * L2_BYTES

    def launches_per_step(self, exchange=None) -> int:
        """Library kernels one timed step launches: zero_step on a flat shard
        or a list is pass 1 (with the decision in its last block) and pass
        2; a step with a cross-rank exchange also launches the decision
        kernel; micro-batches: the accumulation with pass 1, the decision
        and pass 2."""
        if self.micro > 1:
            return 3
        return 2 if exchange is None else 3

    def step(self, stream, exchange=None, ev=None, g=None, lp=None):
        """One step; `g` and `lp` replace the gradient input and the
        low-precision parameter output (flat shards)."""
        zp = self.zp
        g = self.g if g is None else g
        lp = self.lp if lp is None else lp
        if self.micro > 1:
            # the accumulation with pass 1 fused, then the decision and pass 2
            zp.zero_accumulate_grads_norm(g, self.bufs, self.state, self.ws, overwrite=True, stream=stream)
            if exchange is not None:
                exchange(self.state)
            if ev is not None:
                ev[0].record(stream)
            zp.zero_adam_step(g, self.p, self.m, self.v, self.lp, self.hp, self.state, self.ws, stream=stream)
            if ev is not None:
                ev[1].record(stream)
            return
        if exchange is None and ev is None:
            # one rank: the whole step in one call
            if getattr(self, "plan", None) is not None:
                zp.zero_step_prepared(self.plan, self.hp, self.state, self.ws, stream=stream)
            else:
                zp.zero_step(g, self.p, self.m, self.v, lp, self.hp, self.state, self.ws,
                             stream=stream)
            return
        zp.zero_grad_norm_overflow(g, self.state, self.ws, stream=stream)
        if exchange is not None:
            exchange(self.state)
        if ev is not None:
            ev[0].record(stream)
        zp.zero_adam_step(g, self.p, self.m, self.v, lp, self.hp, self.state, self.ws,
                          stream=stream)
        if ev is not None:
            ev[1].record(stream)


def run_ours(args):
    import torch
    import torch.distributed as dist

    import zero_partitioned_mixed_layout_gb300 as zp
    from zero_partitioned_mixed_layout_gb300.dist import exchange_partials

    rank, world, local = dist_env()
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", torch.cuda.current_device())
    if world > 1 and args.workload == WORKLOAD:
        # several GPUs: each rank one ZeRO shard of the same model (rank r
        # shard r of 16), the per-GPU work fixed as N grows
        args.workload = SHARDED
    wl = Workload(args.workload, args.log2n, rank, dev, prepared=args.prepared)
    S = wl.S
    stream = torch.cuda.current_stream(dev)
    exchange = exchange_partials if world > 1 else None
    # a buffer larger than L2, rewritten between timed steps of workloads
    # whose working set would otherwise stay in L2
    flush = torch.empty(int(2 * L2_BYTES), dtype=torch.uint8, device=dev) if wl.l2_resident else None

    def step(ev=None):
        wl.step(stream, exchange, ev)

    def barrier():
        torch.cuda.synchronize(dev)
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    nvtx("range_push", f"warm-up ({wl.name})")
    for _ in range(args.warmup):
        step()
    nvtx("range_pop")
    barrier()
    st = zp.parse_state(wl.state)
    assert st["last_skipped"] == 0 and st["step"] == args.warmup, st

    def pairs():
        return [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(args.steps)]

    events = pairs()          # decision + pass 2, in the instrumented run
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # per-step times of the whole step: in the timed run itself when L2 is
    # flushed before each step, else in a run of their own
    step_events = pairs()
    with ClockSampler(dev.index if world == 1 else local) as clk:
        # the sampler polls every 200 ms: keep the GPU in the same step for a
        # second right before the timed region so that the clock record
        # describes the state the timed steps run in
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < args.clock_preroll:
            for _ in range(20):
                step()
            torch.cuda.synchronize(dev)
        barrier()
        # the timed steps: nothing else in the stream between kernels, so
        # each kernel launches while the previous one drains (the NVTX range
        # only marks them on a profiler's timeline)
        nvtx("range_push", f"timed steps ({wl.name})")
        t_start.record(stream)
        for k in range(args.steps):
            if flush is not None:
                flush.fill_(k & 255)
                step_events[k][0].record(stream)
            step()
            if flush is not None:
                step_events[k][1].record(stream)
        t_end.record(stream)
        nvtx("range_pop")
        barrier()
        # the same number of steps again with events around zero_adam_step,
        # for the dominant kernel's own duration (the events break the launch
        # overlap, so these steps are not the ones the step time comes from)
        for k in range(args.steps):
            if flush is not None:
                flush.fill_(k & 255)
            step(events[k])
        barrier()
        if flush is None:
            # and once more with events around each whole step (between
            # steps, where no launch overlaps anyway)
            for k in range(args.steps):
                step_events[k][0].record(stream)
                step()
                step_events[k][1].record(stream)
            barrier()
    step_times = [a.elapsed_time(b) for a, b in step_events]
    adam_times = [a.elapsed_time(b) for a, b in events]
    if flush is not None:  # the step alone, L2 flushed before each one
        ms = sum(step_times)
    else:
        ms = t_start.elapsed_time(t_end)
    adam_ms = statistics.mean(adam_times)
    st = zp.parse_state(wl.state)
    assert st["last_skipped"] == 0 and st["step"] >= args.warmup + args.steps, st
    if world > 1:
        t = torch.tensor([ms, adam_ms], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms, adam_ms = t.tolist()
    ms_per_step = ms / args.steps
    value = world * S / (ms_per_step * 1e-3)

    # end to end through the public API between pinned host memory and the
    # GPU: every step copies its gradient in (H2D), runs, and copies its
    # product out (D2H) -- the updated low-precision parameters, which the
    # next forward pass (or the parameter all-gather of ZeRO stages 1 and 2)
    # consumes -- plus its 64-byte state into a pinned slot of its own.  The
    # gradient and the parameter output are double-buffered on the device,
    # the two copies run on streams of their own and events order them, so
    # that step k computes while the next steps' gradients come in and the
    # previous steps' parameters go out: the host link carries both
    # directions at once and the host never waits inside the loop.  Every step's state is read and
    # checked on the host after the loop (the copies are inside the timed
    # region).
    e2e = None
    if not wl.listmode and wl.micro == 1:
        hg = torch.empty(S, dtype=wl.g.dtype, pin_memory=True)
        hg.copy_(wl.g)
        NB = 2  # three measured the same: the host link is the limit
        gbuf = [wl.g] + [torch.empty_like(wl.g) for _ in range(NB - 1)]
        lpbuf = [wl.lp] + [torch.empty_like(wl.lp) for _ in range(NB - 1)]
        hlp = [torch.empty(S, dtype=wl.lp.dtype, pin_memory=True) for _ in range(NB)]
        h2d_stream, d2h_stream = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        h2d_done = [torch.cuda.Event() for _ in range(NB)]
        step_done = [torch.cuda.Event() for _ in range(NB)]
        d2h_done = [torch.cuda.Event() for _ in range(NB)]
        for b in range(NB):
            step_done[b].record(stream)
            d2h_done[b].record(d2h_stream)

        def e2e_steps(count):
            hs = torch.empty((count, zp.STATE_BYTES), dtype=torch.uint8, pin_memory=True)
            for k in range(count):
                b = k % NB
                # the gradient in, once the step that last read buffer b is done
                h2d_stream.wait_event(step_done[b])
                with torch.cuda.stream(h2d_stream):
                    gbuf[b].copy_(hg, non_blocking=True)
                h2d_done[b].record(h2d_stream)
                # the step, once its gradient is in and the parameters that
                # output buffer b held NB steps ago are out
                stream.wait_event(h2d_done[b])
                stream.wait_event(d2h_done[b])
                wl.step(stream, exchange, g=gbuf[b], lp=lpbuf[b])
                step_done[b].record(stream)
                hs[k].copy_(wl.state, non_blocking=True)
                # the parameters out
                d2h_stream.wait_event(step_done[b])
                with torch.cuda.stream(d2h_stream):
                    hlp[b].copy_(lpbuf[b], non_blocking=True)
                d2h_done[b].record(d2h_stream)
            return hs

        def check(hs):
            for k in range(hs.shape[0]):
                assert zp.parse_state(bytes(hs[k].numpy().tobytes()))["last_skipped"] == 0

        hs = e2e_steps(3)
        barrier()
        check(hs)
        t0 = time.perf_counter()
        hs = e2e_steps(args.steps)
        barrier()
        e2e_s = (time.perf_counter() - t0) / args.steps
        check(hs)
        # the copied-out parameters are the step's product: the last step's
        # equal the device's copy (checked on its first and last 2^20)
        last = (args.steps - 1) % NB
        for sl in (slice(0, 1 << 20), slice(max(0, S - (1 << 20)), S)):
            assert torch.equal(hlp[last][sl], lpbuf[last][sl].cpu())
        if world > 1:
            t = torch.tensor([e2e_s], dtype=torch.float64, device=dev)
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
            e2e_s = t.item()
        h2d = hg.numel() * hg.element_size()
        d2h = hlp[0].numel() * hlp[0].element_size() + zp.STATE_BYTES
        e2e = {"value": world * S / e2e_s, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": e2e_s * 1e3, "host_link_gbs": (h2d + d2h) / e2e_s / 1e9,
               "note": "every step: the gradient copied in from pinned host memory, the step, the "
                       "updated low-precision parameters and the 64-byte state copied out to pinned host "
                       "memory; copies in and out on streams of their own ordered by events, "
                       "overlapping the neighbouring steps (double-buffered on the device); every "
                       "step's state checked on the host after the timed loop"}

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    peaks = measured_peaks()
    peak = peaks["hbm_gbs"] if peaks else 6800.0
    achieved = wl.bytes_adam * S / (adam_ms * 1e-3) / 1e9
    whole = wl.bytes_step * S / (ms_per_step * 1e-3) / 1e9
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        # about 10-20 s of CPU work in all: 10 full steps of 2^24 params on
        # one core, then on every core at once
        oname = oracle_workload(args.workload)
        n_sample, c_steps = 1 << 24, 10
        if oname == args.workload:
            n_sample = min(n_sample, S)
        cv, cdt, final = oracle_run(n_sample, c_steps, 1, keep=True, name=oname)
        av, adt, procs = oracle_run_all_cores(n_sample, c_steps, 1, name=oname)
        cpu = {"value": av, "unit": UNIT, "cores": procs, "kind": "oracle",
               "sample": f"{procs} processes (one per host core), each {c_steps} full steps on its own "
                         f"{n_sample} params drawn as the workload's ({TITLES[oname]}), "
                         f"{adt:.1f} s wall ({procs * adt:.0f} s of CPU); the oracle as it stands "
                         f"(single-threaded scalar C)",
               "single_core": {"value": cv, "unit": UNIT, "cores": 1, "seconds": cdt,
                               "sample": f"first {n_sample} params of the shard, {c_steps} full steps"},
               # the library on the single-core run's inputs, against its result
               "parity": parity_vs_oracle(dev, n_sample, c_steps + 1, final, oname)}
    default = args.workload == WORKLOAD
    traffic = committed_traffic(args.workload) if not args.prepared else None
    # the part of pass 2's gradient reads that pass 1 leaves in L2 (its
    # evict-last tail): pass-2 fractions above 1 of a copy peak come from it
    l2_tail = min(KEEP_L2_BYTES, wl.S * wl.g.element_size()) if not wl.listmode and wl.micro == 1 else 0

    def stats(xs):
        return {"median": statistics.median(xs), "min": min(xs), "max": max(xs), "n": len(xs)}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": step_config(
            wl.title + ("; the list step prepared once (zero_step_prepared)" if getattr(wl, "plan", None) else ""),
            wl.w, S,
            "L2 flushed (256 MB written) before each timed step; time is the sum of the steps alone"
            if flush is not None else
            f"inputs larger than L2 ({wl.bytes_step * S / 1e9:.2f} GB per step vs {L2_BYTES / 1e6:.0f} MB), "
            "no flush", world),
        "hbm_gbs_adam": achieved,
        "hbm_gbs_step": whole,
        "bytes_per_param": {"adam_pass": wl.bytes_adam, "whole_step": wl.bytes_step},
        "passes_ms": {"adam_step": adam_ms, "adam_step_per_step": stats(adam_times),
                      "whole_step": ms_per_step, "whole_step_per_step": stats(step_times),
                      "note": "whole_step: the timed steps' total over their count; adam_step (decision "
                              "+ pass 2): the mean over a second run of as many steps with events around "
                              "it; *_per_step: median, min and max of the per-step event times"
                              + ("" if flush is not None else " (the whole step's from a third run with "
                                 "events between the steps)")},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "kernel": f"zero_adam_step (decision + pass 2: k_adam_flat), {wl.bytes_adam} B/param",
                     "peak_source": "MEASURED_PEAKS.json hbm_gbs (of measured)" if peaks
                     else "fallback 6.8 TB/s (of fallback)",
                     "peak_record": {k: peaks.get(k) for k in ("hbm_gbs", "how", "when", "gpu_name", "torch")}
                     if peaks else None,
                     "frac_of_nominal": achieved / NOMINAL_HBM_GBS,
                     "nominal_gbs": NOMINAL_HBM_GBS,
                     "l2_assisted_bytes": l2_tail,
                     "l2_assisted_share": l2_tail / (wl.bytes_adam * S),
                     "note": "the peak is a copy benchmark (one read and one write stream); a fraction "
                             "above 1 is this kernel streaming faster than that copy, plus the share of "
                             "its gradient reads that pass 1 left in L2 (l2_assisted_share); the "
                             "whole-step figure counts every byte of every kernel of the step",
                     "whole_step": {"bytes_per_param": wl.bytes_step, "achieved": whole,
                                    "frac": whole / peak, "frac_of_nominal": whole / NOMINAL_HBM_GBS,
                                    "note": "every kernel of the step over ms_per_step: no L2 carry-over "
                                            "counted"}},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": wl.launches_per_step(exchange) * args.steps,
        "clocks": dict(clk.summary(), window=f"{args.clock_preroll:.1f} s of the same step "
                       "just before the timed region, and the timed region"),
    }
    if not default:
        line["config"]["bench_workload"] = args.workload
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_stage2(args):
    """ZeRO stage 2 on one GPU for the GPT-2 1.5B Nd=16 rank-0 shard: the 16
    ranks' fp16 gradient slices of the shard reduced to their mean with pass
    1 fused (zero_reduce_grads, 32 + 2 B/param), then the decision and pass 2
    (zero_adam_step, 28 B/param)."""
    import torch

    import zero_partitioned_mixed_layout_gb300 as zp
    import zero_synth as zs
    dev = torch.device("cuda", torch.cuda.current_device())
    w = zs.WORKLOADS[SHARDED]
    S = zp.zero_partition_layout(w["numel"](), w["nd"], w["align"]).shard_numel
    nd = w["nd"]
    scale = w["loss_scale"]
    reps = []
    for r in range(nd):
        t = torch.empty(S, dtype=torch.float16, device=dev)
        zs.device_grad_into(t, 2000 + r, 0, scale)
        reps.append(t)
    dg = torch.empty(S, dtype=torch.float16, device=dev)
    dp = torch.empty(S, dtype=torch.float32, device=dev)
    zs.device_master_into(dp, 2000)
    dm, dv = torch.zeros(S, device=dev), torch.zeros(S, device=dev)
    dlp = torch.empty(S, dtype=torch.float16, device=dev)
    st, ws = zp.new_state(scale, dev), zp.new_workspace(1, S, dev)
    hp = zp.HParams(**zs.HPARAMS)
    stream = torch.cuda.current_stream(dev)

    def step(ev=None):
        if ev:
            ev[0].record(stream)
        zp.zero_reduce_grads(reps, dg, st, ws, stream=stream)
        if ev:
            ev[1].record(stream)
        zp.zero_adam_step(dg, dp, dm, dv, dlp, hp, st, ws, stream=stream)
        if ev:
            ev[2].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clk:
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
        for k in range(args.steps):
            step(evs[k])
        torch.cuda.synchronize(dev)
    dt = e0.elapsed_time(e1) / args.steps * 1e-3
    red_ms = statistics.mean(a.elapsed_time(b) for a, b, _ in evs)
    adam_ms = statistics.mean(b.elapsed_time(c) for _, b, c in evs)
    assert zp.parse_state(st)["last_skipped"] == 0
    peaks = measured_peaks()
    peak = peaks["hbm_gbs"] if peaks else 6800.0
    red_bytes = 2 * nd + 2
    achieved = red_bytes * S / (red_ms * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": S / dt, "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": "ZeRO stage 2 on one GPU, GPT-2 1.5B Nd=16 rank-0 shard: mean of "
                               "the 16 ranks' fp16 gradient slices with pass 1 fused, then the "
                               "decision and AdamW", "shard_params": S, "replicas": nd,
                   "l2": "inputs larger than L2, no flush"},
        "bytes_per_param": {"reduce": red_bytes, "adam_pass": 28, "whole_step": red_bytes + 28},
        "passes_ms": {"reduce": red_ms, "adam_step": adam_ms, "whole_step": dt * 1e3},
        "hbm_gbs_step": (red_bytes + 28) * S / dt / 1e9,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": None,
                     "kernel": f"zero_reduce_grads (reduction + pass 1), {red_bytes} B/param",
                     "peak_source": "MEASURED_PEAKS.json hbm_gbs (of measured)" if peaks
                     else "fallback 6.8 TB/s (of fallback)"},
        "adam_pass_gbs": 28 * S / (adam_ms * 1e-3) / 1e9,
        "gpu_launches": 3 * args.steps,  # reduction + pass 1, decision, pass 2
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)


def run_gather(args):
    """ZeRO stage 3 on one GPU, the GPT-2 1.5B parameters in 16 fp16 shards
    (S = 97,350,784): the parameter gather back into the 580 tensors
    (zero_gather_params, one call, 2 + 2 B/param), the same gather layer by
    layer into one reused layer buffer (the stage-3 schedule of
    zero_gather_plan: 50 calls), and the inverse scatter (tensors -> shards)."""
    import torch

    import zero_partitioned_mixed_layout_gb300 as zp
    import zero_synth as zs
    dev = torch.device("cuda", torch.cuda.current_device())
    numel = zs.WORKLOADS[SHARDED]["numel"]()
    nd, align = 16, 128
    lay = zp.zero_partition_layout(numel, nd, align)
    S, total = lay.shard_numel, sum(numel)
    offs = [int(o) for o in lay.tensor_offset]
    gen = torch.Generator(device=dev)
    gen.manual_seed(zs.stream_seed(0, "misc"))
    shards = [torch.randint(-32768, 32767, (S,), dtype=torch.int16, device=dev, generator=gen)
              .view(torch.float16) for _ in range(nd)]
    tens = zp.TensorList([torch.empty(n, dtype=torch.float16, device=dev) for n in numel])
    lf = zs.gpt2_layer_first()
    plan = zp.zero_gather_plan(numel, lf, nd, align)
    layer_buf = torch.empty(plan.max_layer_numel, dtype=torch.float16, device=dev)
    layers = [(layer_buf[:int(plan.layer_flat[L + 1] - plan.layer_flat[L])], int(plan.layer_flat[L]))
              for L in range(len(lf) - 1)]
    ws = torch.empty(zp.zero_gather_workspace_bytes(len(numel), nd), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def full():
        zp.zero_gather_params(shards, tens, offs, ws, stream=stream)

    def per_layer():
        for view, o in layers:
            zp.zero_gather_params(shards, [view], [o], ws, stream=stream)

    def scatter():
        zp.zero_scatter_params(tens, offs, shards, ws, stream=stream)

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / args.steps * 1e-3

    with ClockSampler(dev.index) as clk:
        dt = timed(full)
        dt_layers = timed(per_layer)
        dt_scatter = timed(scatter)
    peaks = measured_peaks()
    peak = peaks["hbm_gbs"] if peaks else 6800.0
    achieved = 4 * total / dt / 1e9
    line = {
        "metric": "stage-3 parameter gather params/sec & achieved HBM GB/s (4 B/param), 1 GPU",
        "value": total / dt, "unit": "params/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": {"workload": "ZeRO stage 3 on one GPU: the GPT-2 1.5B parameters (580 tensors, "
                               "1,557,611,200 fp16 elements) gathered from their 16 flat shards",
                   "shards": nd, "shard_params": S, "tensors": len(numel),
                   "l2": "inputs larger than L2 (3.1 GB), no flush"},
        "per_layer": {"calls": len(layers), "ms_per_pass": dt_layers * 1e3,
                      "params_per_s": total / dt_layers,
                      "gbs": 4 * total / dt_layers / 1e9,
                      "max_layer_params": int(plan.max_layer_numel)},
        "scatter": {"ms_per_pass": dt_scatter * 1e3, "params_per_s": total / dt_scatter,
                    "gbs": 4 * total / dt_scatter / 1e9},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": None,
                     "kernel": "zero_gather_params (one launch over 580 tensors), 4 B/param",
                     "peak_source": "MEASURED_PEAKS.json hbm_gbs (of measured)" if peaks
                     else "fallback 6.8 TB/s (of fallback)"},
        "gpu_launches": args.steps,
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)


def run_onebit(args):
    """1-bit Adam's compression stage on rank 0 of 16 for GPT-2 1.5B: every
    worker holds the whole model (n = 16 x 97,350,784 padded elements); a
    step is pass 1 on the local fp16 gradient, the worker compression (local
    momentum + error feedback -> signs and a scale), the server compression
    of chunk 0 from the 16 workers' signs (the other 15 are received
    messages), and the update from the 16 servers' signs with the frozen
    variance.  The synchronised momentum stays in its compressed form
    between steps (the previous servers' signs and scales): the worker reads
    it from there and the update writes no dense copy.  The worker and
    server errors are held in deferred form (each compression's input and
    scale), so each compression is one pass."""
    import torch

    import zero_partitioned_mixed_layout_gb300 as zp
    import zero_synth as zs
    dev = torch.device("cuda", torch.cuda.current_device())
    numel_list = zs.WORKLOADS[SHARDED]["numel"]()
    nd = 16
    S = zp.zero_partition_layout(numel_list, nd, 128).shard_numel
    numel, n = sum(numel_list), nd * S
    g = torch.empty(n, dtype=torch.float16, device=dev)
    zs.device_grad_into(g, 40, 0, 65536.0)
    v = zs.device_normal(n, 1e-3, 41, "misc", 2).square_()
    p = zs.device_normal(n, 0.02, 41, "master")
    plp = p.half()
    x_w = torch.zeros(n, device=dev)
    x_s = torch.zeros(S, device=dev)
    gen = torch.Generator(device=dev)
    gen.manual_seed(zs.stream_seed(0, "misc", 42))
    bits = torch.zeros(n // 32, dtype=torch.int32, device=dev)
    others = [torch.randint(-2 ** 31, 2 ** 31 - 1, (S // 32,), dtype=torch.int32, device=dev, generator=gen)
              for _ in range(nd - 1)]
    wscale = torch.rand(nd, device=dev, generator=gen) * 1e-3 + 1e-4
    sbits = torch.randint(-2 ** 31, 2 ** 31 - 1, (n // 32,), dtype=torch.int32, device=dev, generator=gen)
    sscale = torch.rand(nd, device=dev, generator=gen) * 1e-3 + 1e-4
    state = torch.frombuffer(bytearray(zp.zero_state_init(65536.0)), dtype=torch.uint8).to(dev)
    state[24:32] = torch.tensor([1000], dtype=torch.int64).view(torch.uint8).to(dev)  # warm-up done
    ws = zp.new_workspace(1, n, dev)
    hp = zp.HParams(**zs.HPARAMS)
    stream = torch.cuda.current_stream(dev)
    wlist = [bits[:S // 32]] + others

    def step(ev=None):
        if ev:
            ev[0].record(stream)
        zp.zero_grad_norm_overflow(g, state, ws, stream=stream)
        # the momentum: last step's server signs and scales (chunk 0 from this
        # rank's server, the rest received), read before this step's server
        # overwrites chunk 0
        zp.zero_onebit_worker(g, (sbits, sscale), x_w, bits, wscale[0:1], hp, 1000, state, ws, stream=stream)
        if ev:
            ev[1].record(stream)
        zp.zero_onebit_server(wlist, wscale, x_s, sbits[:S // 32], sscale[0:1], ws, stream=stream)
        if ev:
            ev[2].record(stream)
        zp.zero_onebit_update(sbits, sscale, S, numel, p, None, v, plp, ws, stream=stream)
        if ev:
            ev[3].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clk:
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
        for k in range(args.steps):
            step(evs[k])
        torch.cuda.synchronize(dev)
    st = zp.parse_state(state)
    assert st["last_skipped"] == 0 and st["step"] == 1000 + 2 * args.steps + args.warmup
    dt = e0.elapsed_time(e1) / args.steps * 1e-3
    ms = [statistics.mean(ev[k].elapsed_time(ev[k + 1]) for ev in evs) for k in range(3)]
    # bytes per element of the padded buffer (the momentum read as signs: 1/8)
    b_worker = 2 + (2 + 1 / 8 + 8 + 1 / 8)         # pass 1; worker: g, m, x in and out, signs
    b_server = (nd / 8 + 8 + 1 / 8) / nd             # per element of the whole buffer
    b_update = 1 / 8 + 8 + 4 + 2                     # signs, v and p; p and p_lp
    b_step = b_worker + b_server + b_update
    peaks = measured_peaks()
    peak = peaks["hbm_gbs"] if peaks else 6800.0
    achieved = b_step * n / dt / 1e9
    line = {
        "metric": "1-bit Adam compression-stage step params/sec & achieved HBM GB/s, 1 GPU",
        "value": n / dt, "unit": "params/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": "1-bit Adam, GPT-2 1.5B (1,557,611,200 params padded to 16 x 97,350,784), "
                               "rank 0 of 16, fp16 gradient and parameters, fp32 state; the other ranks' "
                               "signs and scales are synthetic messages", "elements": n,
                   "l2": "inputs larger than L2, no flush"},
        "bytes_per_param": {"pass1_and_worker": b_worker, "server": b_server, "update": b_update,
                            "whole_step": b_step},
        "passes_ms": {"pass1_and_worker": ms[0], "server": ms[1], "update": ms[2], "whole_step": dt * 1e3},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": None, "kernel": f"whole compression-stage step, {b_step:.2f} B/param",
                     "peak_source": "MEASURED_PEAKS.json hbm_gbs (of measured)" if peaks
                     else "fallback 6.8 TB/s (of fallback)"},
        # pass 1, the decision, the worker, the server and the update
        "gpu_launches": 5 * args.steps,
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)


def run_graph(args):
    """Small shards, back to back and L2-resident (no flush: the state of
    these shards fits in L2 and stays there): the step issued as calls
    through the Python binding, against the same step captured once into a
    CUDA graph and replayed.  Below a few million params the GPU work of a
    step is a few microseconds and the host's cost per call (argument
    marshalling and checks, two launches) sets the pace; a replay launches
    both kernels with one call.  The tiny configuration (1,836,288 params)
    is the line's value; flat 2^16 and 2^20 shards are reported beside it."""
    import torch

    dev = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.current_stream(dev)

    def measure(wl):
        for _ in range(args.warmup):
            wl.step(stream)
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0 = time.perf_counter()
        e0.record(stream)
        for _ in range(args.steps):
            wl.step(stream)
        e1.record(stream)
        host_eager = (time.perf_counter() - t0) / args.steps
        torch.cuda.synchronize(dev)
        eager = e0.elapsed_time(e1) / args.steps
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            wl.step(torch.cuda.current_stream(dev))
        for _ in range(args.warmup):
            graph.replay()
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        e0.record(stream)
        for _ in range(args.steps):
            graph.replay()
        e1.record(stream)
        host_graph = (time.perf_counter() - t0) / args.steps
        torch.cuda.synchronize(dev)
        replay = e0.elapsed_time(e1) / args.steps
        st = wl.zp.parse_state(wl.state)
        assert st["last_skipped"] == 0 and st["step"] == 2 * (args.warmup + args.steps), st
        return {"params": wl.S, "eager_ms": eager, "graph_ms": replay,
                "eager_params_per_s": wl.S / (eager * 1e-3), "graph_params_per_s": wl.S / (replay * 1e-3),
                "host_us_per_call": host_eager * 1e6, "host_us_per_replay": host_graph * 1e6}

    with ClockSampler(dev.index) as clk:
        tiny = measure(Workload("tiny", 0, 0, dev))
        flat = {f"2^{k}": measure(Workload("flat", k, 0, dev)) for k in (16, 20)}
    peaks = measured_peaks()
    line = {
        "metric": "Adam-step params/sec, small L2-resident shard, CUDA-graph replay (eager calls beside it), 1 GPU",
        "value": tiny["graph_params_per_s"], "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": tiny["graph_ms"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": "2-layer hidden-256 transformer state (14 tensors, 1,836,288 params), Nd = 1, "
                               "fp16 grads x 1024; zero_step captured once and replayed",
                   "l2": "L2-resident: no flush, the 55 MB step stays in the 126 MB L2 (labelled, not a "
                         "roofline figure)"},
        "tiny": tiny, "flat": flat,
        "roofline": {"bound": "latency", "achieved": None, "peak": peaks["hbm_gbs"] if peaks else 6800.0,
                     "unit": "GB/s", "frac": None, "traffic": None,
                     "kernel": "two launches per step; the step is bound by launch and host latency"},
        "gpu_launches": 3 * 2 * 2 * args.steps,  # 3 shards x (calls + replays) x 2 kernels a step
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)


def run_onebit_server(args):
    """1-bit Adam's server call alone: chunk 0 of the GPT-2 1.5B layout in
    16 shards (S = 97,350,784 elements), the 16 workers' signs and scales as
    received messages; per call one pass: the workers' mean from the
    tabulated rank-order sums, plus the server error (formed from the
    previous input and scale), its signs and its squared norm.  About 0.6 GB
    on the device: the size for a full ncu capture of the server kernel."""
    import torch

    import zero_partitioned_mixed_layout_gb300 as zp
    import zero_synth as zs
    dev = torch.device("cuda", torch.cuda.current_device())
    nd = 16
    S = zp.zero_partition_layout(zs.WORKLOADS[SHARDED]["numel"](), nd, 128).shard_numel
    gen = torch.Generator(device=dev)
    gen.manual_seed(zs.stream_seed(0, "misc", 43))
    wbits = [torch.randint(-2 ** 31, 2 ** 31 - 1, (S // 32,), dtype=torch.int32, device=dev, generator=gen)
             for _ in range(nd)]
    wscale = torch.rand(nd, device=dev, generator=gen) * 1e-3 + 1e-4
    x_s = zs.device_normal(S, 1e-4, 44, "misc", 5)
    sbits = torch.zeros(S // 32, dtype=torch.int32, device=dev)
    sscale = torch.zeros(1, device=dev)
    state = torch.frombuffer(bytearray(zp.zero_state_init(65536.0)), dtype=torch.uint8).to(dev)
    state[24:32] = torch.tensor([1000], dtype=torch.int64).view(torch.uint8).to(dev)  # warm-up done
    ws = zp.new_workspace(nd, nd * S, dev)
    stream = torch.cuda.current_stream(dev)
    # the step's decision (no overflow) in the workspace, from a worker call
    # on 32 elements
    z = torch.zeros(32, device=dev)
    zp.zero_onebit_worker(torch.zeros(32, dtype=torch.float16, device=dev), z, z.clone(),
                          torch.zeros(1, dtype=torch.int32, device=dev), torch.zeros(1, device=dev),
                          zp.HParams(**zs.HPARAMS), 1000, state, ws, stream=stream)

    def step():
        zp.zero_onebit_server(wbits, wscale, x_s, sbits, sscale, ws, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clk:
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < args.clock_preroll:
            for _ in range(20):
                step()
            torch.cuda.synchronize(dev)
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
    dt = e0.elapsed_time(e1) / args.steps * 1e-3
    # per chunk element: the workers' signs, the previous input read, the
    # new one and its signs written
    b_elem = nd / 8 + 8 + 1 / 8
    peaks = measured_peaks()
    peak = peaks["hbm_gbs"] if peaks else 6800.0
    achieved = b_elem * S / dt / 1e9
    line = {
        "metric": "1-bit Adam server call chunk elements/sec & achieved HBM GB/s, 1 GPU",
        "value": S / dt, "unit": "elements/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": "1-bit Adam server, chunk 0 of GPT-2 1.5B in 16 shards (97,350,784 elements), "
                               "16 workers' random signs and scales", "elements": S, "workers": nd,
                   "l2": "inputs larger than L2 (0.6 GB per call), no flush"},
        "bytes_per_element": b_elem,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": None, "kernel": f"server call (one pass), {b_elem:.3f} B/element",
                     "peak_source": "MEASURED_PEAKS.json hbm_gbs (of measured)" if peaks
                     else "fallback 6.8 TB/s (of fallback)"},
        "gpu_launches": args.steps,
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)


def run_offload(args):
    """ZeRO-Offload on the GPT-2 1.5B Nd=16 shard: the fp32 master, momentum
    and variance (12 B/param) live in pinned host memory, the gradient and
    the fp16 parameters in HBM.  Main measurement: zero_step with the GPU
    streaming the host-resident state over NVLink-C2C (12 B/param each way).
    Also measured: the update on the host cores (zero_offload_decide /
    zero_offload_apply), with the gradient sent over the link in chunks and
    the fp16 parameters sent back."""
    import numpy as np
    import torch

    import zero_partitioned_mixed_layout_gb300 as zp
    import zero_synth as zs
    dev = torch.device("cuda", torch.cuda.current_device())
    w = zs.WORKLOADS[SHARDED]
    S = zp.zero_partition_layout(w["numel"](), w["nd"], w["align"]).shard_numel
    threads = zp.default_host_threads()
    scale = w["loss_scale"]
    dg = torch.empty(S, dtype=torch.float16, device=dev)
    zs.device_grad_into(dg, 1000, 0, scale)
    d_lp = torch.empty(S, dtype=torch.float16, device=dev)
    hp = zp.HParams(**zs.HPARAMS)
    stream = torch.cuda.current_stream(dev)

    # -- the GPU streams the host-resident state over the link
    p = torch.from_numpy(zs.host_master(S, 1000)).pin_memory()
    m, v = torch.zeros(S).pin_memory(), torch.zeros(S).pin_memory()
    d_state = zp.new_state(scale, dev)
    ws = zp.new_workspace(1, S, dev)
    for _ in range(args.warmup):
        zp.zero_step(dg, p, m, v, d_lp, hp, d_state, ws, stream=stream)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clk:
        e0.record(stream)
        for _ in range(args.steps):
            zp.zero_step(dg, p, m, v, d_lp, hp, d_state, ws, stream=stream)
        e1.record(stream)
        torch.cuda.synchronize(dev)
    dt_gpu = e0.elapsed_time(e1) / args.steps * 1e-3
    assert zp.parse_state(d_state)["last_skipped"] == 0
    # the link's two directions at once: copy-engine H2D and D2H of 1 GiB
    hb = torch.empty(1 << 30, dtype=torch.uint8, pin_memory=True)
    db = torch.empty(1 << 30, dtype=torch.uint8, device=dev)
    hb2 = torch.empty(1 << 30, dtype=torch.uint8, pin_memory=True)
    db2 = torch.empty(1 << 30, dtype=torch.uint8, device=dev)
    s2 = torch.cuda.Stream(dev)
    best = float("inf")
    for _ in range(3):
        torch.cuda.synchronize(dev)
        c0 = time.perf_counter()
        db.copy_(hb, non_blocking=True)
        with torch.cuda.stream(s2):
            hb2.copy_(db2, non_blocking=True)
        torch.cuda.synchronize(dev)
        best = min(best, time.perf_counter() - c0)
    link_peak = 2 * (1 << 30) / best / 1e9
    del hb, db, hb2, db2

    # -- the update on the host cores
    hp_, hm_, hv_ = p.clone(), torch.zeros(S), torch.zeros(S)
    h_g = torch.empty(S, dtype=torch.float16, pin_memory=True)
    h_lp = torch.empty(S, dtype=torch.float16, pin_memory=True)
    h_state = torch.empty(zp.STATE_BYTES, dtype=torch.uint8, pin_memory=True)
    d_state2 = zp.new_state(scale, dev)
    up = torch.cuda.Stream(dev)
    chunks = 16
    edges = [S * c // chunks // 2048 * 2048 for c in range(chunks)] + [S]
    got = [torch.cuda.Event() for _ in range(chunks)]
    state_ev, sent = torch.cuda.Event(), torch.cuda.Event()

    def host_step():
        zp.zero_grad_norm_overflow(dg, d_state2, ws, stream=stream)
        h_state.copy_(d_state2, non_blocking=True)
        state_ev.record(stream)
        for c in range(chunks):
            h_g[edges[c]:edges[c + 1]].copy_(dg[edges[c]:edges[c + 1]], non_blocking=True)
            got[c].record(stream)
        state_ev.synchronize()
        sc = zp.zero_offload_decide(h_state, hp)
        for c in range(chunks):
            lo, hi = edges[c], edges[c + 1]
            got[c].synchronize()
            zp.zero_offload_apply(h_g[lo:hi], hp_[lo:hi], hm_[lo:hi], hv_[lo:hi], h_lp[lo:hi], sc,
                                  n_threads=threads)
            with torch.cuda.stream(up):
                d_lp[lo:hi].copy_(h_lp[lo:hi], non_blocking=True)
        with torch.cuda.stream(up):
            d_state2.copy_(h_state, non_blocking=True)
        sent.record(up)
        stream.wait_event(sent)
        sent.synchronize()

    for _ in range(min(args.warmup, 3)):
        host_step()
    host_steps = max(3, min(args.steps, 10))
    t0 = time.perf_counter()
    for _ in range(host_steps):
        host_step()
    dt_host = (time.perf_counter() - t0) / host_steps
    a = np.ones(1 << 28, np.float32)
    b = np.empty_like(a)
    zp.zero_offload_copy(b, a, threads)
    cbest = float("inf")
    for _ in range(3):
        c0 = time.perf_counter()
        zp.zero_offload_copy(b, a, threads)
        cbest = min(cbest, time.perf_counter() - c0)
    host_peak = 2 * a.nbytes / cbest / 1e9

    achieved = 24 * S / dt_gpu / 1e9
    line = {
        "metric": METRIC, "value": S / dt_gpu, "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": dt_gpu * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": "ZeRO-Offload on the GPT-2 1.5B Nd=16 rank-0 shard: fp32 master, "
                               "momentum, variance in pinned host memory, streamed by the GPU over "
                               "NVLink-C2C (zero_step); gradient and fp16 params in HBM",
                   "shard_params": S, "c2c_bytes_per_param": {"to_gpu": 12, "to_host": 12}},
        "roofline": {"bound": "host-link", "achieved": achieved, "peak": link_peak, "unit": "GB/s",
                     "frac": achieved / link_peak, "traffic": None,
                     "kernel": "zero_step with host-resident state, 24 B/param over NVLink-C2C",
                     "peak_source": "copy-engine H2D + D2H of 1 GiB at once, measured in this run"},
        "host_compute_mode": {
            "value": S / dt_host, "unit": UNIT, "ms_per_step": dt_host * 1e3, "host_threads": threads,
            "host_gbs_28B": 28 * S / dt_host / 1e9, "host_copy_peak_gbs": host_peak,
            "note": "update on the host cores (zero_offload_apply); gradient to the host and fp16 "
                    "params back over the link in 16 chunks each step"},
        "gpu_launches": 2 * args.steps,  # zero_step on a flat shard: pass 1 (+ decision), pass 2
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", default=WORKLOAD,
                    choices=["gpt2_1p5b_nd16", "tiny", "gpt2_1p5b_full", "stack_100b_nd400",
                             "frag_10k", "flat", "offload", "stage2", "gather", "onebit", "onebit_server",
                             "graph"],
                    help="default: the whole GPT-2 1.5B state (Nd = 1), the largest configuration "
                         "that fits one GPU; under torchrun each rank takes one shard of the same "
                         "model in 16 ZeRO shards instead")
    ap.add_argument("--log2n", type=int, default=26, help="size of the flat workload (2^k)")
    ap.add_argument("--prepared", action="store_true",
                    help="frag_10k: the list step prepared once (zero_list_prepare / zero_step_prepared)")
    ap.add_argument("--clock-preroll", type=float, default=1.0,
                    help="seconds of untimed steps, sampled for clocks, before the timed ones")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    elif args.workload in ("offload", "stage2", "gather", "onebit", "onebit_server", "graph"):
        from zero_partitioned_mixed_layout_gb300 import _build
        _build.build()
        {"offload": run_offload, "stage2": run_stage2, "gather": run_gather,
         "onebit": run_onebit, "onebit_server": run_onebit_server, "graph": run_graph}[args.workload](args)
    else:
        import zero_partitioned_mixed_layout_gb300 as zp
        from zero_partitioned_mixed_layout_gb300 import _build
        _build.build()
        zp.lib()
        run_ours(args)


if __name__ == "__main__":
    main()
