"""Benchmark of the sketching hot path on GB300.

One step = the whole path over one batch of synthetic input for a stack of
linear layers: draw every layer's projection, then for each microbatch project
every layer's input (XP = X P) and accumulate every layer's sketch
(C += D^T XP), then rebuild-and-update every layer's BF16 weights.

Default workload: the Qwen3-8B-shaped stack (36 blocks x q,k,v,o,gate,up,down =
252 linears, 6.95e9 weights), rank 64, 32768 tokens per step in 4096-token
microbatches, refreshed Gaussian-QR projections, normalized SGD with tau=1e-3.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl {gb300,reference}]

Prints one JSON line (rank 0).  ``value`` is whole-job tokens/s with inputs
resident in HBM; ``e2e`` repeats the step with every input copied from pinned
host memory inside the timed region.  ``--impl reference`` times the CPU oracle
(the plain C statement of the method) on a bounded sample of the same workload.
"""
import argparse
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "sketch-accumulate tokens/s and update weights/s on 1 GB300, % of HBM roofline"
NBUF = 3  # input buffers per distinct shape; consecutive uses of one buffer are > 4x L2 apart


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--workload", default="qwen3-8b-stack")
    ap.add_argument("--rank", type=int, default=64)
    ap.add_argument("--e2e-steps", type=int, default=None,
                    help="steps in the end-to-end (host buffers) measurement; default = --steps")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-shared-x", action="store_true",
                    help="give q/k/v and gate/up inputs of their own instead of one shared X each")
    ap.add_argument("--layers", type=int, default=None,
                    help="keep only the first N layers of the workload (a smaller case for profiling)")
    return ap.parse_args()


# DRAM bytes (read + write) per algorithmic byte of each phase's main kernel, from
# one ncu capture of one Qwen3-8B block (profiles/qwen3_8b_one_block_kernels.md);
# traffic grows with the units processed, so a full launch's traffic is this
# ratio times its algorithmic bytes.
TRAFFIC_PER_ALGORITHMIC_BYTE = {"project_inputs": 214.3 / 214.4, "accumulate": 268.8 / 342.4,
                                "update_normsgd": 786.3 / 791.4}


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
    """Layers that read one X (q/k/v, gate/up), or one group per layer."""
    from rank_gradient_sketching_philox_gb300 import synth
    if no_shared_x or r % 8 != 0:
        return [[li] for li in range(len(wl.layers))]
    return synth.input_groups(wl.layers)


def workload_config(wl, r, n, shared_x=None):
    cfg = {
        "workload": wl.name,
        "layers": len(wl.layers),
        "weights": wl.weights,
        "rank": r,
        "tokens_per_step_per_gpu": wl.tokens_per_step,
        "microbatch_tokens": wl.microbatch,
        "projection": "gaussian-qr refreshed every step" if "qr" in wl.projection else wl.projection,
        "update": "%s step_size=%g, ||W||^2 carried between steps" % (wl.update, wl.step_size),
        "parallelism": "dp%d" % n,
        "l2": "inputs rotate through %d buffers per shape (reuse distance > 4x L2); W, C, P per layer"
              % NBUF,
    }
    if shared_x is not None:
        cfg["inputs"] = shared_x
    return cfg


# --------------------------------------------------------------------------
# CPU baseline: the oracle on a bounded sample of the workload
# --------------------------------------------------------------------------

def oracle_sample(wl, r, tokens_sample=16, rows_sample=4):
    """Time the CPU oracle on one block of the stack and scale to one step.

    Sample: the first transformer block's linears; the QR (or Rademacher)
    projection of each; projection + accumulation of ``tokens_sample`` tokens;
    ||W|| and the Gram-route ||H||; the update of ``rows_sample`` rows of each.
    Per-layer, per-token and per-row costs are measured, then multiplied by the
    step's counts (blocks, tokens, rows)."""
    import numpy as np
    import torch

    import oracle as orc
    from rank_gradient_sketching_philox_gb300 import synth

    def u16(t):
        return t.contiguous().view(torch.int16).numpy().view(np.uint16)

    orc.lib()
    seen, block = set(), []
    for name, d, k in wl.layers:
        tag = name.split(".")[-1]
        if tag in seen:
            break
        seen.add(tag)
        block.append((name, d, k))
    nblocks = len(wl.layers) // len(block)
    T = tokens_sample
    t_sample = t_tok = t_norm = t_rows = 0.0
    for li, (_, d, k) in enumerate(block):
        t0 = time.perf_counter()
        P = (orc.sample_qr(0, li, 0, k, r) if "qr" in wl.projection
             else orc.sample_rademacher(0, li, 0, k, r))
        t1 = time.perf_counter()
        X = u16(synth.normal_bf16((T, k), 1.0, 5 + li))
        D = u16(synth.normal_bf16((T, d), 1e-3, 9 + li))
        t2 = time.perf_counter()
        XP = orc.project_inputs(X, P)
        C = orc.accumulate(D, XP, np.zeros((d, r), np.float32), overwrite=True)
        t3 = time.perf_counter()
        W = u16(synth.layer_weight(d, k, li))
        t4 = time.perf_counter()
        s, _ = orc.normsgd_scale(orc.norm_w(W), orc.norm_h_gram(C, P), wl.step_size)
        t5 = time.perf_counter()
        orc.update_rows(W[:rows_sample], np.arange(rows_sample, dtype=np.int32), C, P, s, 0, li, 0)
        t6 = time.perf_counter()
        t_sample += t1 - t0
        t_tok += t3 - t2
        t_norm += t5 - t4
        t_rows += (t6 - t5) * (d / rows_sample)
    per_step = nblocks * (t_sample + t_tok * (wl.tokens_per_step / T) + t_norm + t_rows)
    return {
        "step_seconds": per_step,
        "tokens_per_s": wl.tokens_per_step / per_step,
        "sample": ("oracle on block 0 of the stack (%d linears, r=%d): projection of each, "
                   "projection+accumulation of %d tokens, ||W|| and Gram ||H||, update of %d rows "
                   "each; scaled to %d blocks x %d tokens x all rows" %
                   (len(block), r, T, rows_sample, nblocks, wl.tokens_per_step)),
    }


def run_reference(args):
    """The reference arm: the CPU oracle as it stands, on the host cores."""
    if int(os.environ.get("RANK", "0")) != 0:
        return
    from rank_gradient_sketching_philox_gb300 import synth
    wl = synth.WORKLOADS[args.workload]
    times, rates, res = [], [], None
    for _ in range(args.warmup):
        oracle_sample(wl, args.rank, tokens_sample=8, rows_sample=2)
    for _ in range(args.steps):
        t0 = time.perf_counter()
        res = oracle_sample(wl, args.rank, tokens_sample=8, rows_sample=2)
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
        "ms_per_step": wl.tokens_per_step / value * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": workload_config(wl, args.rank, args.gpus,
                                  shared_x=input_note(workload_groups(wl, args.rank, args.no_shared_x))),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": res["sample"], "wall_seconds_per_sample": statistics.median(times)},
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

    wl = synth.WORKLOADS[args.workload]
    if args.layers:
        wl = dataclasses.replace(wl, name="%s[:%d]" % (wl.name, args.layers), layers=wl.layers[:args.layers])
    r = args.rank
    T = wl.microbatch
    nmb = wl.microbatches
    layers = wl.layers
    L = len(layers)
    kind = rgs.PROJ_GAUSSIAN_QR if "qr" in wl.projection else rgs.PROJ_RADEMACHER
    seed = 0
    tau = wl.step_size
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
    groups = workload_groups(wl, r, args.no_shared_x)
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
    xpool, dpool = {}, {}
    for li, (_, d, k) in enumerate(layers):
        if k not in xpool:
            xpool[k] = [synth.normal_bf16((T, k), synth.X_STD, 7000 + 10 * k + b, device=dev)
                        for b in range(NBUF)]
        if d not in dpool:
            dpool[d] = [synth.layer_d(T, d, 9000 + d, b, device=dev, heavy_tail=wl.heavy_tail)
                        for b in range(NBUF)]
    torch.cuda.synchronize()

    def xbuf(li, m):
        return xpool[layers[li][2]][(li + m) % NBUF]

    def dbuf(li, m):
        return dpool[layers[li][1]][(li + 2 * m + 1) % NBUF]

    layer_ids = list(range(L))
    # workspaces of the batched calls, allocated once
    ws_sample = torch.empty(rgs.workspace_bytes_batched(
        binding.OP_SAMPLE_PROJECTION, k=[k for _, _, k in layers], r=r) if kind == rgs.PROJ_GAUSSIAN_QR
        else 1, dtype=torch.uint8, device=dev)
    ws_project = {m: torch.empty(max(1, rgs.workspace_bytes_batched(
        binding.OP_PROJECT_INPUTS, T=[T] * len(by_size[m]), k=[layers[groups[gi][0]][2] for gi in by_size[m]],
        r=m * r)), dtype=torch.uint8, device=dev) for m in sizes}
    ws_update = torch.empty(rgs.workspace_bytes_batched(
        binding.OP_UPDATE_NORMSGD, d=[d for _, d, _ in layers], k=[k for _, _, k in layers], r=r),
        dtype=torch.uint8, device=dev)
    wn2_views = [wn2[li:li + 1] for li in range(L)]
    status_views = [status[li:li + 1] for li in range(L)]

    # the BF16 split of each group's concatenated P, made once per refresh and
    # read by every microbatch's projection
    P_split = [torch.empty(rgs.projection_split_elems(layers[g[0]][2], len(g) * r), dtype=torch.int16, device=dev)
               for g in groups]

    def sample_phase(s):
        rgs.sample_projection_batched(kind, seed, s, P, layer_ids, ws=ws_sample)
        rgs.split_projection_grouped([[P[li] for li in g] for g in groups], splits=P_split)

    def project_phase(m, Xs=None):
        # Xs: one input per group (default: the group's first layer's buffer)
        for size in sizes:
            gis = by_size[size]
            rgs.project_inputs_grouped_batched(
                [Xs[gi] if Xs is not None else xbuf(groups[gi][0], m) for gi in gis],
                [P_split[gi] for gi in gis], size * r, [XPg[gi] for gi in gis], ws=ws_project[size])

    def accumulate_phase(m, Ds=None):
        rgs.accumulate_batched(Ds if Ds is not None else [dbuf(li, m) for li in range(L)], XP, C,
                               overwrite=(m == 0))

    def update_phase(s, carried):
        rgs.apply_update_normsgd_batched(W, C, P, tau, seed, layer_ids, s,
                                         wnorm2_in=wn2_views if carried else None,
                                         wnorm2_out=wn2_views, dev_status=status_views, ws=ws_update)

    def allreduce_sketch():
        # data parallel: each rank sketches its own microbatches; the sketches add
        dataparallel.allreduce_sketches(C_flat)

    def step(s, carried=True):
        sample_phase(s)
        for m in range(nmb):
            project_phase(m)
            accumulate_phase(m)
        allreduce_sketch()
        update_phase(s, carried)

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
    value = wl.tokens_per_step * args.steps * world / elapsed

    # ---- per-phase timings (each phase alone, same buffers) ---------------
    phase_launches = {}

    def timed(fn, name):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
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
    t_sample = timed(lambda: sample_phase(s_next), "sample")
    t_project = timed(lambda: [project_phase(m) for m in range(nmb)], "project")
    t_accum = timed(lambda: [accumulate_phase(m) for m in range(nmb)], "accumulate")
    t_update = timed(lambda: update_phase(s_next, True), "update")
    nst = int((status != 0).sum().item())

    # algorithmic bytes: the minimum each call must move
    acc_bytes = sum(nmb * (2 * T * d + 2 * T * r + 8 * d * r) for _, d, _ in layers)
    proj_bytes = sum(nmb * (2 * T * layers[g[0]][2] + (2 * T + 4 * layers[g[0]][2]) * len(g) * r)
                     for g in groups)
    upd_bytes = sum(4 * d * k + 8 * d * r + 8 * k * r for _, d, k in layers)
    peak, peak_kind = measured_peaks()

    def gbs(bytes_, secs):
        return bytes_ / secs / 1e9

    # launches of each phase, counted by the library; the dominant kernel of a
    # phase is its skinny GEMM (projection, accumulation) or the persistent
    # rebuild+update kernel (one per 56 layers)
    ceil = lambda a, b: -(-a // b)
    n_sample = phase_launches["sample"]
    n_proj = phase_launches["project"]        # skinny GEMM launches (P split once per step)
    n_acc = phase_launches["accumulate"]
    n_upd = ceil(L, 56)  # layers per rebuild+update launch
    n_upd_aux = phase_launches["update"] - n_upd
    components = {
        "sample_projection": {"ms_per_step": t_sample * 1e3, "launches": n_sample},
        "project_inputs": {"ms_per_step": t_project * 1e3, "tokens_per_s": wl.tokens_per_step / t_project,
                           "gbs": gbs(proj_bytes, t_project),
                           "hbm_frac": gbs(proj_bytes, t_project) / peak, "launches": n_proj},
        "accumulate": {"ms_per_step": t_accum * 1e3, "tokens_per_s": wl.tokens_per_step / t_accum,
                       "gbs": gbs(acc_bytes, t_accum), "hbm_frac": gbs(acc_bytes, t_accum) / peak,
                       "launches": n_acc},
        "update_normsgd": {"ms_per_step": t_update * 1e3, "weights_per_s": wl.weights / t_update,
                           "gbs": gbs(upd_bytes, t_update), "hbm_frac": gbs(upd_bytes, t_update) / peak,
                           "launches": n_upd + n_upd_aux,
                           "bytes_model": "4 B/weight (W read+write, ||W||^2 carried) + 8dr + 8kr"},
        "nonzero_device_status": nst,
    }
    name, secs, bytes_, nl = max(("accumulate", t_accum, acc_bytes, n_acc),
                                 ("project_inputs", t_project, proj_bytes, n_proj),
                                 ("update_normsgd", t_update, upd_bytes, n_upd), key=lambda x: x[1])
    roofline = {
        "kernel": name,
        "bound": "hbm",
        "achieved": gbs(bytes_, secs),
        "peak": peak,
        "unit": "GB/s",
        "frac": gbs(bytes_, secs) / peak,
        "peak_source": ("measured (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                        else "fallback 6.8 TB/s"),
        "bytes_per_launch": bytes_ / nl,
        "avg_launch_ms": secs / nl * 1e3,
        "traffic": (TRAFFIC_PER_ALGORITHMIC_BYTE[name] * bytes_ / nl
                    if name in TRAFFIC_PER_ALGORITHMIC_BYTE else None),
        "traffic_source": "ncu dram__bytes_read.sum + dram__bytes_write.sum on one Qwen3-8B block, scaled "
                          "to a full launch by algorithmic bytes (profiles/qwen3_8b_one_block_kernels.md)",
    }

    # ---- end to end: inputs copied from pinned host memory every step -----
    e2e_steps = args.e2e_steps if args.e2e_steps is not None else args.steps
    e2e = None
    if e2e_steps > 0:
        # every layer's X and D of a microbatch come from pinned host memory
        hx = {k: [b.cpu().pin_memory() for b in v] for k, v in xpool.items()}
        hd = {d: [b.cpu().pin_memory() for b in v] for d, v in dpool.items()}
        stage_x = [torch.empty(T, layers[g[0]][2], dtype=torch.bfloat16, device=dev) for g in groups]
        stage_d = [torch.empty(T, d, dtype=torch.bfloat16, device=dev) for _, d, _ in layers]
        h2d = nmb * (sum(x.numel() * 2 for x in stage_x) + sum(d_.numel() * 2 for d_ in stage_d))
        d2h = status.numel() * 4 + wn2.numel() * 8
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for s in range(s_next + 1, s_next + 1 + e2e_steps):
            sample_phase(s)
            for m in range(nmb):
                for gi, g in enumerate(groups):
                    stage_x[gi].copy_(hx[layers[g[0]][2]][(g[0] + m) % NBUF], non_blocking=True)
                project_phase(m, stage_x)
                for li, (_, d, k) in enumerate(layers):
                    stage_d[li].copy_(hd[d][(li + 2 * m + 1) % NBUF], non_blocking=True)
                accumulate_phase(m, stage_d)
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
        e2e = {"value": wl.tokens_per_step * e2e_steps * world / e2e_elapsed, "unit": "tokens/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        res = oracle_sample(wl, r)
        cpu = {"value": res["tokens_per_s"], "unit": "tokens/s", "cores": 1, "kind": "oracle",
               "sample": res["sample"]}

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
            "config": workload_config(wl, r, world, shared_x=input_note(groups)),
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
