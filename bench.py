"""Benchmark of the sketching hot path on GB300.

One step = the whole path over one batch of synthetic input for a stack of
linear layers: draw every layer's projection (unless it is fixed), then for
each microbatch project every layer's input (XP = X P) and accumulate every
layer's sketch (C += D^T XP), then rebuild-and-update every layer's BF16
weights (normalized SGD, or LoGRA's SGD for the LoGRA worked example).

Default workload: the Qwen3-8B-shaped stack (36 blocks x q,k,v,o,gate,up,down =
252 linears, 6.95e9 weights), rank 64, 32768 tokens per step in 4096-token
microbatches, refreshed Gaussian-QR projections, normalized SGD with tau=1e-3.
Other workloads: ``--workload`` (a name in ``synth.WORKLOADS``), ``--rank``,
``--tokens`` (tokens per step) and ``--projection``.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl {gb300,reference}]

Prints one JSON line (rank 0).  ``value`` is whole-job tokens/s with inputs
resident in HBM; ``e2e`` repeats the step with every input copied from pinned
host memory inside the timed region.  ``--impl reference`` times the CPU oracle
(the plain C statement of the method) on a bounded sample of the same workload.
"""
import argparse
import dataclasses
import json
import math
import multiprocessing
import os
import platform
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "sketch-accumulate tokens/s and update weights/s on 1 GB300, % of HBM roofline"
L2_BYTES = 129 * 1024 * 1024
MAX_GROUP_RANK = 256  # rank of one grouped projection call (m r)


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--workload", default="qwen3-8b-stack")
    ap.add_argument("--rank", type=int, default=None, help="default: the workload's first rank")
    ap.add_argument("--tokens", type=int, default=None,
                    help="tokens per step (default: the workload's); microbatch = min(tokens, workload's)")
    ap.add_argument("--projection", choices=["qr-refreshed", "rademacher-fixed"], default=None,
                    help="default: the workload's (Gaussian-QR refreshed where it names both)")
    ap.add_argument("--e2e-steps", type=int, default=None,
                    help="steps in the end-to-end (host buffers) measurement; default = --steps")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-procs", type=int, default=None,
                    help="processes of the all-cores CPU baseline (default: every host core)")
    ap.add_argument("--no-shared-x", action="store_true",
                    help="give q/k/v and gate/up inputs of their own instead of one shared X each")
    ap.add_argument("--layers", type=int, default=None,
                    help="keep only the first N layers of the workload (a smaller case for profiling)")
    return ap.parse_args(argv)


@dataclasses.dataclass
class Run:
    """One benchmark configuration: a workload with its rank, token count and
    projection kind resolved."""
    name: str
    layers: list
    r: int
    tokens_per_step: int
    microbatch: int
    projection: str   # "qr-refreshed" or "rademacher-fixed"
    update: str       # "normsgd" or "sgd"
    step_size: float
    heavy_tail: bool

    @property
    def microbatches(self):
        return max(1, self.tokens_per_step // self.microbatch)

    @property
    def weights(self):
        return sum(d * k for _, d, k in self.layers)

    @property
    def refreshed(self):
        return self.projection == "qr-refreshed"


def resolve(args):
    from rank_gradient_sketching_philox_gb300 import synth
    wl = synth.WORKLOADS[args.workload]
    layers = wl.layers[:args.layers] if args.layers else wl.layers
    r = args.rank if args.rank is not None else wl.ranks[0]
    tokens = args.tokens if args.tokens is not None else wl.tokens_per_step
    mb = min(tokens, wl.microbatch)
    if tokens % mb:
        raise SystemExit("--tokens must be a multiple of the microbatch (%d)" % mb)
    proj = args.projection or ("qr-refreshed" if wl.projection in ("both", "qr-refreshed") else wl.projection)
    name = wl.name + ("[:%d]" % args.layers if args.layers else "")
    return Run(name, layers, r, tokens, mb, proj, wl.update, wl.step_size, wl.heavy_tail)


# DRAM bytes (read + write) per algorithmic byte of each phase's main kernel, from
# one ncu capture (dram__bytes_read.sum + dram__bytes_write.sum) of ten Qwen3-8B
# blocks (70 linears, one 4096-token microbatch, every layer's inputs its own:
# launches as large as the full stack's, so the same kernels run): the persistent
# accumulation 3329.1 MB against 3423.6 MB (XP and part of C still in L2 from the
# projection), the three persistent projection launches 2176.9 MB against
# 2144.3 MB.  Traffic grows with the units processed, so a full launch's traffic
# is this ratio times its algorithmic bytes.
TRAFFIC_PER_ALGORITHMIC_BYTE = {"accumulate": 3329.14 / 3423.60, "project_inputs": 2176.94 / 2144.34}


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            m = json.load(f)
        return float(m["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def input_note(groups):
    return ("q/k/v and gate/up read one X each, projected together (grouped splits)"
            if any(len(g) > 1 for g in groups) else "every layer reads its own X")


def workload_groups(wl, r, no_shared_x):
    """Layers that read one X (q/k/v, gate/up), or one group per layer.  A
    group is split into singletons when its members' XP would not start on a
    16-byte boundary (r not a multiple of 8) or its rank m r exceeds one
    projection call's."""
    from rank_gradient_sketching_philox_gb300 import synth
    if no_shared_x or r % 8 != 0:
        return [[li] for li in range(len(wl.layers))]
    out = []
    for g in synth.input_groups(wl.layers):
        if len(g) * r <= MAX_GROUP_RANK:
            out.append(g)
        else:
            out.extend([li] for li in g)
    return out


def input_sets(bytes_per_set):
    """Input sets that alternate over consecutive microbatches so that a
    buffer's reuse distance is at least four times L2 (at least two sets)."""
    return max(2, 1 + math.ceil(4 * L2_BYTES / max(1, bytes_per_set)))


def workload_config(run, n, groups=None, nsets=None):
    upd = ("normsgd tau=%g, ||W||^2 carried between steps" % run.step_size if run.update == "normsgd"
           else "sgd alpha*eta=%g" % run.step_size)
    cfg = {
        "workload": run.name,
        "layers": len(run.layers),
        "weights": run.weights,
        "rank": run.r,
        "tokens_per_step_per_gpu": run.tokens_per_step,
        "microbatch_tokens": run.microbatch,
        "projection": ("gaussian-qr refreshed every step" if run.refreshed
                       else "rademacher fixed (drawn once, step 0)"),
        "update": upd,
        "heavy_tailed_d": run.heavy_tail,
        "parallelism": "dp%d" % n,
    }
    if nsets is not None:
        cfg["l2"] = ("every layer its own D and every input group its own X, %d sets alternating over "
                     "microbatches (reuse distance >= 4x L2); W, C, P per layer; L2 flushed before "
                     "each phase timing" % nsets)
    if groups is not None:
        cfg["inputs"] = input_note(groups)
    return cfg


# --------------------------------------------------------------------------
# CPU baseline: the oracle on a bounded sample of the workload
# --------------------------------------------------------------------------

def _first_block(layers):
    seen, block = set(), []
    for name, d, k in layers:
        tag = name.split(".")[-1]
        if tag in seen:
            break
        seen.add(tag)
        block.append((name, d, k))
    return block


def oracle_sample(run, tokens_sample=16, rows_sample=4):
    """Time the CPU oracle on one block of the stack and scale to one step.

    Sample: the first transformer block's linears (or every layer of a
    workload without blocks); the projection of each (drawn every step when
    refreshed, else not timed: a fixed projection is drawn once);
    projection + accumulation of ``tokens_sample`` tokens; the update's norms
    (normalized SGD: ||W|| and the Gram-route ||H||) and the update of
    ``rows_sample`` rows of each.  Per-layer, per-token and per-row costs are
    measured, then multiplied by the step's counts (blocks, tokens, rows)."""
    import numpy as np
    import torch

    import oracle as orc
    from rank_gradient_sketching_philox_gb300 import synth

    def u16(t):
        return t.contiguous().view(torch.int16).numpy().view(np.uint16)

    orc.lib()
    block = _first_block(run.layers)
    nblocks = len(run.layers) / len(block)
    T, r = tokens_sample, run.r
    t_sample = t_tok = t_norm = t_rows = 0.0
    for li, (_, d, k) in enumerate(block):
        t0 = time.perf_counter()
        P = (orc.sample_qr(0, li, 0, k, r) if run.refreshed else orc.sample_rademacher(0, li, 0, k, r))
        t1 = time.perf_counter()
        X = u16(synth.normal_bf16((T, k), 1.0, 5 + li))
        D = u16(synth.normal_bf16((T, d), 1e-3, 9 + li))
        t2 = time.perf_counter()
        XP = orc.project_inputs(X, P)
        C = orc.accumulate(D, XP, np.zeros((d, r), np.float32), overwrite=True)
        t3 = time.perf_counter()
        W = u16(synth.normal_bf16((rows_sample, k), synth.W_STD, 1000 + li)) if run.update == "sgd" \
            else u16(synth.layer_weight(d, k, li))
        t4 = time.perf_counter()
        if run.update == "normsgd":
            s, _ = orc.normsgd_scale(orc.norm_w(W), orc.norm_h_gram(C, P), run.step_size)
        else:
            s = run.step_size
        t5 = time.perf_counter()
        orc.update_rows(W[:rows_sample], np.arange(rows_sample, dtype=np.int32), C, P, s, 0, li, 0)
        t6 = time.perf_counter()
        if run.refreshed:
            t_sample += t1 - t0
        t_tok += t3 - t2
        t_norm += t5 - t4
        t_rows += (t6 - t5) * (d / rows_sample)
    per_step = nblocks * (t_sample + t_tok * (run.tokens_per_step / T) + t_norm + t_rows)
    return {
        "step_seconds": per_step,
        "tokens_per_s": run.tokens_per_step / per_step,
        "sample": ("oracle on %s (%d linears, r=%d): %sprojection+accumulation of %d tokens, %s"
                   "update of %d rows each; scaled to %g x %d tokens x all rows" %
                   ("block 0 of the stack" if nblocks > 1 else "every layer", len(block), r,
                    "QR projection of each, " if run.refreshed else "", T,
                    "||W|| and Gram ||H||, " if run.update == "normsgd" else "", rows_sample,
                    nblocks, run.tokens_per_step)),
    }


def _oracle_worker(run, tokens_sample, rows_sample, barrier, out):
    import oracle as orc
    orc.lib()
    barrier.wait()  # every process starts its timed sample at once
    out.put(oracle_sample(run, tokens_sample, rows_sample)["step_seconds"])


def host_cpu():
    model = platform.processor() or platform.machine()
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key = line.split(":")[0].strip().lower()
                if key in ("model name", "cpu part", "hardware"):
                    model = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                model = line.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    return model


def cpu_baseline(run, procs=None, tokens_sample=16, rows_sample=4):
    """The oracle timed on one host core, and on every core at once: one
    process per core, all released by one barrier, each timing the same
    sample (the units are independent, so the all-cores rate is the sum of
    the processes' rates measured while all of them ran).  Processes are
    spawned, never forked from a process that has used the GPU."""
    procs = procs or os.cpu_count() or 1
    single = oracle_sample(run, tokens_sample, rows_sample)
    ctx = multiprocessing.get_context("spawn")
    barrier, out = ctx.Barrier(procs), ctx.Queue()
    workers = [ctx.Process(target=_oracle_worker, args=(run, tokens_sample, rows_sample, barrier, out))
               for _ in range(procs)]
    t0 = time.perf_counter()
    for w in workers:
        w.start()
    step_seconds = [out.get() for _ in workers]
    for w in workers:
        w.join()
    wall = time.perf_counter() - t0
    return {
        "value": sum(run.tokens_per_step / s for s in step_seconds),
        "unit": "tokens/s",
        "cores": procs,
        "kind": "oracle",
        "sample": single["sample"] + "; all cores: %d spawned processes timed the sample at once "
                                     "(%.1f s wall)" % (procs, wall),
        "single_core_value": single["tokens_per_s"],
        "host_cpu": host_cpu(),
        "nproc": os.cpu_count(),
    }


def run_reference(args):
    """The reference arm: the CPU oracle as it stands, on the host cores."""
    if int(os.environ.get("RANK", "0")) != 0:
        return
    run = resolve(args)
    times, rates, res = [], [], None
    for _ in range(args.warmup):
        oracle_sample(run, tokens_sample=8, rows_sample=2)
    for _ in range(args.steps):
        t0 = time.perf_counter()
        res = oracle_sample(run, tokens_sample=8, rows_sample=2)
        times.append(time.perf_counter() - t0)
        rates.append(res["tokens_per_s"])
    value = statistics.median(rates)
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": "tokens/s",
        "n_gpus": args.gpus,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": run.tokens_per_step / value * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": workload_config(run, args.gpus,
                                  groups=workload_groups(run, run.r, args.no_shared_x)),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": res["sample"], "wall_seconds_per_sample": statistics.median(times),
                         "host_cpu": host_cpu(), "nproc": os.cpu_count()},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------
# GPU arm
# --------------------------------------------------------------------------

class ClockSampler:
    """nvidia-smi clock and throttle-reason samples during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            parts = [p.strip() for p in l.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
        return
    import torch
    import torch.distributed as dist

    import __graft_entry__ as entry
    import rank_gradient_sketching_philox_gb300 as rgs
    from rank_gradient_sketching_philox_gb300 import binding, dataparallel, synth

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    entry.build()

    run = resolve(args)
    r, T, nmb, layers = run.r, run.microbatch, run.microbatches, run.layers
    L = len(layers)
    kind = rgs.PROJ_GAUSSIAN_QR if run.refreshed else rgs.PROJ_RADEMACHER
    normsgd = run.update == "normsgd"
    seed = 0
    stream = torch.cuda.current_stream(dev)

    # ---- resident state -------------------------------------------------
    W = [synth.normal_bf16((d, k), synth.W_STD, synth.seed_w(li), device=dev)
         for li, (_, d, k) in enumerate(layers)]
    # every layer's sketch in one buffer: one all-reduce per step across replicas
    C_flat, C = dataparallel.flat_sketches([(d, r) for _, d, _ in layers], dev)
    P = [torch.empty(k, r, dtype=torch.float32, device=dev) for _, _, k in layers]
    # layers that read one X (q/k/v, gate/up) are projected together: one call
    # with the split of their concatenated P reads X once; each layer's XP is a
    # column block of its group's result
    groups = workload_groups(run, r, args.no_shared_x)
    XPg = [torch.empty(T, max(8, (len(g) * r + 7) // 8 * 8), dtype=torch.bfloat16, device=dev)[:, :len(g) * r]
           for g in groups]
    XP = [None] * L
    for gi, g in enumerate(groups):
        for q, li in enumerate(g):
            XP[li] = XPg[gi][:, q * r:(q + 1) * r]
    sizes = sorted({len(g) for g in groups})
    by_size = {m: [gi for gi, g in enumerate(groups) if len(g) == m] for m in sizes}
    wn2 = torch.zeros(L, dtype=torch.float64, device=dev)
    status = torch.zeros(L, dtype=torch.int32, device=dev)
    # Inputs: every input group its own X and every layer its own D, as in a
    # real step, in `nsets` sets that alternate over consecutive microbatches
    # so that no buffer is read again before at least 4x L2 of other inputs.
    gk = [layers[g[0]][2] for g in groups]
    x_bytes, d_bytes = 2 * T * sum(gk), 2 * T * sum(d for _, d, _ in layers)
    nsets = input_sets(min(x_bytes, d_bytes))
    xsets = [[synth.normal_bf16((T, k), synth.X_STD, 7_000_000 + 1000 * s + gi, device=dev)
              for gi, k in enumerate(gk)] for s in range(nsets)]
    dsets = [[synth.layer_d(T, d, li, s, device=dev, heavy_tail=run.heavy_tail)
              for li, (_, d, _) in enumerate(layers)] for s in range(nsets)]
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
    torch.cuda.synchronize()

    layer_ids = list(range(L))
    # workspaces of the batched calls, allocated once
    ws_sample = torch.empty(rgs.workspace_bytes_batched(
        binding.OP_SAMPLE_PROJECTION, k=[k for _, _, k in layers], r=r) if kind == rgs.PROJ_GAUSSIAN_QR
        else 1, dtype=torch.uint8, device=dev)
    ws_project = {m: torch.empty(max(1, rgs.workspace_bytes_batched(
        binding.OP_PROJECT_INPUTS, T=[T] * len(by_size[m]), k=[gk[gi] for gi in by_size[m]],
        r=m * r)), dtype=torch.uint8, device=dev) for m in sizes}
    op_update = binding.OP_UPDATE_NORMSGD if normsgd else binding.OP_UPDATE_SGD
    ws_update = torch.empty(max(1, rgs.workspace_bytes_batched(
        op_update, d=[d for _, d, _ in layers], k=[k for _, _, k in layers], r=r)),
        dtype=torch.uint8, device=dev)
    wn2_views = [wn2[li:li + 1] for li in range(L)]
    status_views = [status[li:li + 1] for li in range(L)]

    # the BF16 split of each group's concatenated P, made once per refresh and
    # read by every microbatch's projection
    P_split = [torch.empty(rgs.projection_split_elems(gk[gi], len(g) * r), dtype=torch.int16, device=dev)
               for gi, g in enumerate(groups)]

    def sample_phase(s):
        rgs.sample_projection_batched(kind, seed, s, P, layer_ids, ws=ws_sample)
        rgs.split_projection_grouped([[P[li] for li in g] for g in groups], splits=P_split)

    # The projection's independent launches (one per input-group size) go to
    # side streams that fork from and join back to the main stream, so that one
    # persistent launch's last CTAs overlap the next launch's first instead of
    # leaving SMs idle.
    side = [torch.cuda.Stream(dev) for _ in range(3)]

    def fork_join(fns):
        ev = torch.cuda.Event()
        ev.record(stream)
        done = []
        for fn, ss in zip(fns, side):
            ss.wait_event(ev)
            fn(ss)
            e = torch.cuda.Event()
            e.record(ss)
            done.append(e)
        for e in done:
            stream.wait_event(e)

    def project_phase(Xs):
        def launch(size):
            gis = by_size[size]
            return lambda ss: rgs.project_inputs_grouped_batched(
                [Xs[gi] for gi in gis], [P_split[gi] for gi in gis], size * r, [XPg[gi] for gi in gis],
                ws=ws_project[size], stream=ss)
        fork_join([launch(size) for size in sizes])

    def accumulate_phase(m, Ds):
        rgs.accumulate_batched(Ds, XP, C, overwrite=(m == 0))

    def update_phase(s, carried):
        if normsgd:
            rgs.apply_update_normsgd_batched(W, C, P, run.step_size, seed, layer_ids, s,
                                             wnorm2_in=wn2_views if carried else None,
                                             wnorm2_out=wn2_views, dev_status=status_views, ws=ws_update)
        else:
            rgs.apply_update_sgd_batched(W, C, P, run.step_size, seed, layer_ids, s,
                                         dev_status=status_views, ws=ws_update)

    def allreduce_sketch():
        # data parallel: each rank sketches its own microbatches; the sketches add
        dataparallel.allreduce_sketches(C_flat)

    mb_count = [0]  # microbatches so far: picks the input set

    def next_set():
        s_ = mb_count[0] % nsets
        mb_count[0] += 1
        return s_

    def step(s, carried=True):
        if run.refreshed:
            sample_phase(s)
        for m in range(nmb):
            si = next_set()
            project_phase(xsets[si])
            accumulate_phase(m, dsets[si])
        allreduce_sketch()
        update_phase(s, carried)

    if not run.refreshed:  # a fixed projection is drawn once
        sample_phase(0)

    # ---- warm-up ---------------------------------------------------------
    for s in range(args.warmup):
        step(s, carried=(s > 0))
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()

    # ---- timed region: K steps, inputs resident in HBM --------------------
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    with ClockSampler(local) as clocks:
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        launches0 = rgs.kernel_launches()
        ev[0].record(stream)
        for s in range(args.warmup, args.warmup + args.steps):
            step(s)
        ev[1].record(stream)
        launches = rgs.kernel_launches() - launches0
        torch.cuda.synchronize()
    elapsed = ev[0].elapsed_time(ev[1]) / 1e3
    if world > 1:
        t = torch.tensor([elapsed], device=dev, dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        elapsed = float(t.item())
        dist.barrier()
    ms_per_step = elapsed / args.steps * 1e3
    value = run.tokens_per_step * args.steps * world / elapsed

    # ---- per-phase timings (each phase alone, same buffers, L2 flushed) ---
    phase_launches = {}

    def timed(fn, name):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        flush.zero_()  # nothing of the previous phase stays in L2
        torch.cuda.synchronize()
        l0 = rgs.kernel_launches()
        # the GPU first spins ~10 ms, so that the host's launch work for the phase
        # is queued before the start event and the phase is timed on the device
        torch.cuda._sleep(20_000_000)
        a.record(stream)
        fn()
        b.record(stream)
        phase_launches[name] = rgs.kernel_launches() - l0
        torch.cuda.synchronize()
        return a.elapsed_time(b) / 1e3

    s_next = args.warmup + args.steps
    t_sample = timed(lambda: sample_phase(s_next if run.refreshed else 0), "sample")
    sets = [next_set() for _ in range(nmb)]
    t_project = timed(lambda: [project_phase(xsets[si]) for si in sets], "project")
    t_accum = timed(lambda: [accumulate_phase(m, dsets[si]) for m, si in enumerate(sets)], "accumulate")
    rgs.read_exact_count()
    t_update = timed(lambda: update_phase(s_next, True), "update")
    exact_weights = rgs.read_exact_count()
    nst = int((status != 0).sum().item())

    # algorithmic bytes: the minimum each call must move
    acc_bytes = sum(nmb * (2 * T * d + 2 * T * r + 8 * d * r) for _, d, _ in layers)
    proj_bytes = sum(nmb * (2 * T * gk[gi] + (2 * T + 4 * gk[gi]) * len(g) * r) for gi, g in enumerate(groups))
    if normsgd:
        upd_bytes = sum(4 * d * k + 8 * d * r + 8 * k * r for _, d, k in layers)
        upd_model = "4 B/weight (W read+write, ||W||^2 carried) + 8dr + 8kr"
    else:
        upd_bytes = sum(4 * d * k + 4 * d * r + 4 * k * r for _, d, k in layers)
        upd_model = "4 B/weight (W read+write) + 4dr + 4kr"
    peak, peak_kind = measured_peaks()

    def gbs(bytes_, secs):
        return bytes_ / secs / 1e9

    # launches of each phase, counted by the library; the dominant kernel of a
    # phase is its skinny GEMM (projection, accumulation) or the persistent
    # rebuild+update kernel (one per 56 layers)
    n_sample = phase_launches["sample"]
    n_proj = phase_launches["project"]
    n_acc = phase_launches["accumulate"]
    n_upd = -(-L // 56)
    upd_name = "update_normsgd" if normsgd else "update_sgd"
    components = {
        "sample_projection": {"ms_per_step": t_sample * 1e3 if run.refreshed else 0.0,
                              "launches": n_sample if run.refreshed else 0,
                              "note": "refreshed every step" if run.refreshed
                              else "fixed: drawn once, outside the step (%.3f ms)" % (t_sample * 1e3)},
        "project_inputs": {"ms_per_step": t_project * 1e3, "tokens_per_s": run.tokens_per_step / t_project,
                           "gbs": gbs(proj_bytes, t_project),
                           "hbm_frac": gbs(proj_bytes, t_project) / peak, "launches": n_proj},
        "accumulate": {"ms_per_step": t_accum * 1e3, "tokens_per_s": run.tokens_per_step / t_accum,
                       "gbs": gbs(acc_bytes, t_accum), "hbm_frac": gbs(acc_bytes, t_accum) / peak,
                       "launches": n_acc},
        upd_name: {"ms_per_step": t_update * 1e3, "weights_per_s": run.weights / t_update,
                   "gbs": gbs(upd_bytes, t_update), "hbm_frac": gbs(upd_bytes, t_update) / peak,
                   "launches": phase_launches["update"], "bytes_model": upd_model,
                   "exact_path_weights": exact_weights},
        "nonzero_device_status": nst,
    }
    name, secs, bytes_, nl = max(("accumulate", t_accum, acc_bytes, n_acc),
                                 ("project_inputs", t_project, proj_bytes, n_proj),
                                 ("update", t_update, upd_bytes, n_upd), key=lambda x: x[1])
    ratio = TRAFFIC_PER_ALGORITHMIC_BYTE.get(name)
    roofline = {
        "kernel": upd_name if name == "update" else name,
        "bound": "hbm",
        "achieved": gbs(bytes_, secs),
        "peak": peak,
        "unit": "GB/s",
        "frac": gbs(bytes_, secs) / peak,
        "peak_source": ("measured (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                        else "fallback 6.8 TB/s"),
        "bytes_per_launch": bytes_ / nl,
        "avg_launch_ms": secs / nl * 1e3,
        "traffic": ratio * bytes_ / nl if ratio is not None else None,
        "traffic_source": ("ncu dram__bytes_read.sum + dram__bytes_write.sum of the kernel on ten "
                           "Qwen3-8B blocks (70 linears, inputs of their own), scaled to a full launch by "
                           "algorithmic bytes" if ratio is not None else None),
    }

    # ---- end to end: inputs copied from pinned host memory every step -----
    e2e_steps = args.e2e_steps if args.e2e_steps is not None else args.steps
    e2e = None
    if e2e_steps > 0:
        # Every microbatch's X (per input group) and D (per layer) come from
        # pinned host memory (two host buffers per shape).  The copies run on
        # their own streams into two device sets used alternately, so the
        # copies of microbatch m+1 overlap the kernels of microbatch m.
        hx, hd = {}, {}
        for gi, k in enumerate(gk):
            if k not in hx:
                hx[k] = [xsets[i][gi].cpu().pin_memory() for i in range(2)]
        for li, (_, d, _) in enumerate(layers):
            if d not in hd:
                hd[d] = [dsets[i][li].cpu().pin_memory() for i in range(2)]
        h2d = nmb * (x_bytes + d_bytes)
        d2h = status.numel() * 4 + wn2.numel() * 8
        # several copy streams, so that more than one copy engine moves data
        copy_streams = [torch.cuda.Stream(dev) for _ in range(4)]
        copied = [[torch.cuda.Event() for _ in copy_streams] for _ in range(2)]
        consumed = [torch.cuda.Event() for _ in range(2)]
        for b in range(2):
            consumed[b].record(stream)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for s in range(s_next + 1, s_next + 1 + e2e_steps):
            if run.refreshed:
                sample_phase(s)
            for m in range(nmb):
                b = m % 2
                jobs = ([(xsets[b][gi], hx[k][(gi + m) % 2]) for gi, k in enumerate(gk)] +
                        [(dsets[b][li], hd[d][(li + m) % 2]) for li, (_, d, _) in enumerate(layers)])
                for ci, cs in enumerate(copy_streams):
                    cs.wait_event(consumed[b])  # the kernels that read set b are done
                    with torch.cuda.stream(cs):
                        for dst, src in jobs[ci::len(copy_streams)]:
                            dst.copy_(src, non_blocking=True)
                    copied[b][ci].record(cs)
                for ev in copied[b]:
                    stream.wait_event(ev)
                project_phase(xsets[b])
                accumulate_phase(m, dsets[b])
                consumed[b].record(stream)
            allreduce_sketch()
            update_phase(s, True)
            _ = status.cpu(), wn2.cpu()  # the step's result read back to the host
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_elapsed = e0.elapsed_time(e1) / 1e3
        if world > 1:
            t = torch.tensor([e2e_elapsed], device=dev, dtype=torch.float64)
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
            e2e_elapsed = float(t.item())
        e2e = {"value": run.tokens_per_step * e2e_steps * world / e2e_elapsed, "unit": "tokens/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
               "h2d_gbs": h2d * e2e_steps / e2e_elapsed / 1e9,
               "copies": "four copy streams, two device sets alternating: microbatch m+1's copies "
                         "overlap microbatch m's kernels"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(run, procs=args.cpu_procs)

    if rank == 0:
        line = {
            "metric": METRIC,
            "value": value,
            "unit": "tokens/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": ms_per_step,
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16+fp32",
            "data": "synthetic",
            "config": workload_config(run, world, groups=groups, nsets=nsets),
            "components": components,
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": launches,
            "clocks": clocks.summary(),
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
