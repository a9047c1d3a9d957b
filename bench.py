"""MuonH optimizer-step benchmark (one JSON line on stdout).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

A step is one full MuonH step (momentum, Newton-Schulz, hyperball projection)
over every matrix of the workload, through the library's C ABI.  Default
workload: the 2B-class set (28 Qwen3-style decoder layers, 196 matrices,
1.409 G parameters).  value = steps/s over all ranks (each rank steps its own
replica: weak scaling, no collective on the data path).

Reported beside it:
  roofline      the Newton-Schulz GEMM kernel (the dominant one): symmetric-
                aware algorithmic TFLOP/s from CUDA events recorded by the
                library around each launch, against the measured sustained
                bf16 peak
  cpu_baseline  the float64 oracle on this host, on one matrix of each shape
                (three steps), scaled to steps/s of the full set by the
                sample's share of the Newton-Schulz flops
  e2e           steps/s with gradients copied in from pinned host memory and
                the status word read back every step (the next step's copy
                overlaps the current step on a side stream)
  clocks        nvidia-smi samples taken during the timed region
--impl reference times the oracle alone (the reference arm).
"""

from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MuonH steps/s on a 2B param set (1 B300); NS GEMM % of bf16 tensor peak"
METRIC_MUON = "Muon steps/s on a 2B param set (1 B300); NS GEMM % of bf16 tensor peak"
METRIC_ADAMW = "AdamW steps/s on the 2B model's non-matrix group (1 B300); % of HBM bandwidth"
MUON_WD = 0.1
ADAMW_BETAS, ADAMW_EPS, ADAMW_WD = (0.9, 0.95), 1e-8, 0.1
PROFILE_DIR = os.path.join(ROOT, "profiles")


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16": d["bf16_tflops"], "bf16_sustained": d["bf16_tflops_sustained"],
                "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16": 1800.0, "bf16_sustained": 1400.0, "source": "fallback"}


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def launch_plan(gpus: int, env) -> str:
    """How a run with --gpus N starts: "run" (this process is one of the N
    ranks, or N = 1), "relaunch" (N > 1 and no launcher: start N ranks with
    torch.distributed.run) or an error text (a launcher started a different
    number of ranks than --gpus asks for)."""
    if gpus < 1:
        return f"--gpus must be >= 1, got {gpus}"
    if "WORLD_SIZE" in env:
        world = int(env["WORLD_SIZE"])
        if world != gpus:
            return f"--gpus {gpus} but the launcher started WORLD_SIZE={world} ranks"
        return "run"
    return "run" if gpus == 1 else "relaunch"


def _relaunch(gpus: int):
    """Re-runs this command as `gpus` ranks on 127.0.0.1 (one per GPU)."""
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={gpus}",
           "--master-addr=127.0.0.1", f"--master-port={port}", os.path.abspath(__file__), *sys.argv[1:]]
    os.execv(sys.executable, cmd)


class ClockSampler:
    """nvidia-smi clock/throttle samples in the background (every 200 ms)."""

    FIELDS = "clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown," \
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown," \
             "clocks_event_reasons.sw_power_cap"

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        mhz, maxes, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                mhz.append(float(parts[0]))
                maxes.append(float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not mhz:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        mhz.sort()
        return {"sm_mhz": mhz[len(mhz) // 2], "sm_max_mhz": max(maxes), "reasons": sorted(reasons),
                "samples": len(mhz)}


def _ns_traffic_from_profiles():
    """Per-launch DRAM bytes of the NS GEMM kernel from the committed ncu summary, if current."""
    p = os.path.join(PROFILE_DIR, "ns_gemm_traffic.json")
    if not os.path.exists(p):
        return None
    try:
        with open(p) as f:
            d = json.load(f)
        return d
    except (OSError, ValueError):
        return None


L2_BYTES = 126 * 2 ** 20


def _l2_note(work, optimizer):
    """Whether a step's inputs exceed L2 (the timed steps do not flush it)."""
    per_el = 28 if optimizer == "adamw" else 22   # bytes of state a step reads and writes per element
    b = per_el * work.n_params
    if b > 2 * L2_BYTES:
        return f"inputs larger than L2 ({b / 1e9:.2f} GB of optimizer state touched per step)"
    return (f"inputs fit in L2 ({b / 1e6:.2f} MB of optimizer state per step), not flushed between steps: "
            "a latency figure")


def _oracle_cores():
    try:
        from threadpoolctl import threadpool_info
        return max((i.get("num_threads", 1) for i in threadpool_info()), default=os.cpu_count())
    except Exception:  # threadpoolctl missing: report the host's logical cores
        return os.cpu_count()


def _ns_flops(shapes):
    return sum(3 * min(r, c) ** 2 * max(r, c) + min(r, c) ** 3 for r, c in shapes)


def oracle_sample_indices(work):
    """A bounded sample of the workload for the oracle: the first matrix of
    every distinct shape (4 of the 2B set's 196 matrices), capped at 64."""
    seen, idx = set(), []
    for i, sh in enumerate(work.shapes):
        if sh not in seen:
            seen.add(sh)
            idx.append(i)
    return idx[:64]


def oracle_sample_adamw(work, repeats=1, warmup=0):
    """The AdamW oracle on a bounded sample of the AdamW group: the first
    16384 rows of the embedding and every norm vector; scaled to steps/s of
    the whole group by the sample's share of the elements (the method is
    elementwise)."""
    import numpy as np
    from oracle import muonh as om
    rows = 16384
    ps = [work.weight(0, "cpu")[:rows].numpy()] + [w.numpy() for w in work.weights("cpu", range(1, len(work.shapes)))]
    gs = [work.grad(0, 0, "cpu")[:rows].numpy()] + [g.numpy() for g in work.grads(0, "cpu", range(1, len(work.shapes)))]
    ms = [np.zeros_like(p) for p in ps]
    vs = [np.zeros_like(p) for p in ps]
    for t in range(warmup):
        om.adamw_step(ps, gs, ms, vs, t + 1, work.lr, *ADAMW_BETAS, ADAMW_EPS, ADAMW_WD)
    t0 = time.perf_counter()
    for t in range(repeats):
        om.adamw_step(ps, gs, ms, vs, t + 1, work.lr, *ADAMW_BETAS, ADAMW_EPS, ADAMW_WD)
    dt = (time.perf_counter() - t0) / max(repeats, 1)
    frac = sum(p.size for p in ps) / work.n_params
    sample = (f"oracle (NumPy float64) AdamW on {sum(p.size for p in ps)} of {work.n_params} elements (first "
              f"{rows} embedding rows and all norm vectors), {repeats} timed step(s) of {dt:.2f} s each; scaled by "
              f"the element share ({frac:.4f})")
    return frac / dt, _oracle_cores(), sample


def oracle_sample(work, repeats=1, warmup=0, optimizer="muonh"):
    """Time the float64 oracle (MuonH, or plain Muon) on the sample; returns
    steps/s of the whole workload (sample time scaled by the sample's share
    of the step's Newton-Schulz flops), threads used and a description."""
    import numpy as np
    from oracle import muonh as om
    idx = oracle_sample_indices(work)
    ws = [w.numpy() for w in work.weights("cpu", idx)]
    gs = [g.numpy() for g in work.grads(0, "cpu", idx)]
    ms = [np.zeros_like(w) for w in ws]
    r0 = om.capture_norms(ws)

    def one():
        if optimizer == "muon":
            om.muon_step(ws, gs, ms, work.lr, work.beta, MUON_WD, work.ns_steps, work.coeffs, work.eps)
        else:
            om.muonh_step(ws, gs, ms, r0, work.lr, work.beta, work.ns_steps, work.coeffs, work.eps)
    for _ in range(warmup):
        one()
    t0 = time.perf_counter()
    for _ in range(repeats):
        one()
    dt = (time.perf_counter() - t0) / max(repeats, 1)
    frac = _ns_flops([work.shapes[i] for i in idx]) / _ns_flops(work.shapes)
    sample = (f"oracle (NumPy float64) on {len(idx)} of {len(work.shapes)} matrices (one of each shape), "
              f"{repeats} timed step(s) of {dt:.2f} s each; scaled by their share ({frac:.4f}) of the "
              f"step's Newton-Schulz flops")
    return frac / dt, _oracle_cores(), sample


def run_reference(args, work, world, rank):
    """The reference arm: the oracle, as it stands, on this host's cores;
    W untimed and K timed steps, each on the bounded sample."""
    if rank != 0:
        return
    if args.optimizer == "adamw":
        v, cores, sample = oracle_sample_adamw(work, repeats=args.steps, warmup=args.warmup)
    else:
        v, cores, sample = oracle_sample(work, repeats=args.steps, warmup=args.warmup, optimizer=args.optimizer)
    line = {
        "impl": "reference", "metric": {"muon": METRIC_MUON, "adamw": METRIC_ADAMW}.get(args.optimizer, METRIC),
        "value": v, "unit": "steps/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 / v, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": work.name, "matrices": len(work.shapes), "params": work.n_params},
        "cpu_baseline": {"value": v, "unit": "steps/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": v, "unit": "steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="qwen3_2b_28layers")
    ap.add_argument("--layers", type=int, default=None,
                    help="first N decoder layers of the 2B set (a smaller case for profiling)")
    ap.add_argument("--impl", default="cuda", choices=["cuda", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--gemm", default="pair", choices=["pair", "pair_one_step", "1sm"],
                    help="Newton-Schulz GEMM kernel: CTA pair per 256x256 tile (two K steps per pipeline "
                         "stage where the shape allows; pair_one_step: always one), or one SM per 128x256 tile")
    ap.add_argument("--one-stream", action="store_true",
                    help="every Newton-Schulz launch on the caller's stream (no side streams for independent "
                         "buckets)")
    ap.add_argument("--optimizer", default="muonh", choices=["muonh", "muon", "adamw"],
                    help="muon: plain Muon (decoupled weight decay 0.1, no hyperball), the baseline MuonH is "
                         "compared with; adamw: AdamW on the non-matrix group (workload qwen3_2b_adamw_group)")
    args = ap.parse_args()

    import muonh_workloads as wl
    if args.layers is not None:
        if args.workload != "qwen3_2b_28layers":
            raise SystemExit("--layers applies to the qwen3_2b_28layers workload only")
        work = wl.qwen3_2b(layers=args.layers)
    elif args.optimizer == "adamw" and args.workload == "qwen3_2b_28layers":
        work = wl.adamw_group()
    else:
        work = wl.ALL[args.workload]()
    world, rank, local = _dist()

    if args.impl == "reference":
        run_reference(args, work, world, rank)
        return

    plan = launch_plan(args.gpus, os.environ)
    if plan == "relaunch":
        _relaunch(args.gpus)
    elif plan != "run":
        raise SystemExit(plan)

    import torch
    import torch.distributed as dist

    # the oracle's BLAS pool is started before any CUDA work
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = (oracle_sample_adamw(work, repeats=3) if args.optimizer == "adamw"
               else oracle_sample(work, repeats=3, optimizer=args.optimizer))

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    import hyperball_constrained_muon_muonh_b300 as mh

    ws = work.weights(dev)
    grads = [work.grads(t, dev) for t in range(2)]   # two gradient sets, alternated
    gemm_flags = {"pair": 0, "pair_one_step": mh.FLAG_GEMM_ONE_STEP,
                  "1sm": mh.FLAG_GEMM_1SM}[args.gemm] | (mh.FLAG_ONE_STREAM if args.one_stream else 0)
    if args.optimizer == "adamw":
        ws = [w.reshape(-1) for w in ws]
        grads = [[g.reshape(-1) for g in gs] for gs in grads]
        opt = mh.AdamW(ws, lr=work.lr, betas=ADAMW_BETAS, eps=ADAMW_EPS, weight_decay=ADAMW_WD, bf16_copies=True)
    elif args.optimizer == "muon":
        opt = mh.Muon(ws, lr=work.lr, beta=work.beta, weight_decay=MUON_WD, ns_steps=work.ns_steps,
                      ns_coeffs=work.coeffs, eps=work.eps, bf16_copies=True, flags=gemm_flags)
    else:
        opt = mh.MuonH(ws, lr=work.lr, beta=work.beta, ns_steps=work.ns_steps, ns_coeffs=work.coeffs,
                       eps=work.eps, bf16_copies=True, flags=gemm_flags)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()

    for t in range(args.warmup):
        opt.step(grads[t % 2])
    torch.cuda.synchronize()
    st = mh.get_status()
    if st:
        raise SystemExit(f"device status {st:#x} after warm-up")

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    # The headline: K steps with no tracing (the library's per-launch events
    # off), between a barrier and a synchronise on each side.
    n_launch0 = mh.lib.muonh_launch_count()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ else local) as clk:
        barrier()
        ev0.record(stream)
        for t in range(args.steps):
            opt.step(grads[t % 2])
        ev1.record(stream)
        barrier()
    gpu_launches = mh.lib.muonh_launch_count() - n_launch0
    ms_total = ev0.elapsed_time(ev1)
    if world > 1:
        t_ = torch.tensor([ms_total], device=dev)
        dist.all_reduce(t_, op=dist.ReduceOp.MAX)
        ms_total = t_.item()
    ms_step = ms_total / args.steps
    value = world * args.steps / (ms_total / 1000.0)

    # The per-kernel breakdown and the roofline: more steps of the same
    # schedule with the library's CUDA events around every launch (on the
    # stream it is launched on), outside the headline's timed region.
    prof_steps = min(args.steps, 10)
    mh.lib.muonh_profile_enable(1)
    pe0, pe1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    pe0.record(stream)
    for t in range(prof_steps):
        opt.step(grads[t % 2])
    pe1.record(stream)
    torch.cuda.synchronize()
    prof = mh.profile_read()
    mh.lib.muonh_profile_enable(0)
    prof_ms_step = pe0.elapsed_time(pe1) / prof_steps

    # The HBM kernels' roofline comes from a few more steps with every launch
    # on the caller's stream: on the side streams a bucket's momentum or
    # hyperball launch can wait for SMs that other buckets' GEMMs hold, and
    # its event interval counts that wait.
    prof_hbm, hbm_steps = prof, prof_steps
    if args.optimizer != "adamw" and not args.one_stream:
        hbm_steps = 3
        flags1 = gemm_flags | mh.FLAG_ONE_STREAM
        if args.optimizer == "muon":
            opt1 = mh.Muon(ws, lr=work.lr, beta=work.beta, weight_decay=MUON_WD, ns_steps=work.ns_steps,
                           ns_coeffs=work.coeffs, eps=work.eps, bf16_copies=True, flags=flags1)
        else:
            opt1 = mh.MuonH(ws, lr=work.lr, beta=work.beta, ns_steps=work.ns_steps, ns_coeffs=work.coeffs,
                            eps=work.eps, bf16_copies=True, flags=flags1)
        for t in range(2):
            opt1.step(grads[t % 2])
        torch.cuda.synchronize()
        mh.lib.muonh_profile_enable(1)
        for t in range(hbm_steps):
            opt1.step(grads[t % 2])
        torch.cuda.synchronize()
        prof_hbm = mh.profile_read()
        mh.lib.muonh_profile_enable(0)
        del opt1
        torch.cuda.empty_cache()

    # ---- multi-GPU only: the sharded step (each rank steps the matrices it
    # owns, then every updated weight is broadcast from its owner, NCCL inside
    # the timed region): strong scaling of one step of the set ----
    sharded = None
    if world > 1 and args.optimizer == "muonh":
        try:
            ws_s = work.weights(dev)
            sopt = mh.ShardedMuonH(ws_s, lr=work.lr, beta=work.beta, ns_steps=work.ns_steps,
                                   ns_coeffs=work.coeffs, eps=work.eps, bf16_copies=True, flags=gemm_flags)
            for t in range(args.warmup):
                sopt.step(grads[t % 2])
            s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            barrier()
            s0.record(stream)
            for t in range(args.steps):
                sopt.step(grads[t % 2])
            s1.record(stream)
            barrier()
            t_ = torch.tensor([s0.elapsed_time(s1)], device=dev)
            dist.all_reduce(t_, op=dist.ReduceOp.MAX)
            sms = t_.item() / args.steps
            sharded = {"value": 1000.0 / sms, "unit": "steps/s", "ms_per_step": sms, "scaling": "strong",
                       "what": "one step of the whole set split across the ranks by Newton-Schulz cost "
                               "(muonh_partition), then one NCCL broadcast per rank of its updated fp32 weights",
                       "matrices_on_rank0": len(sopt.mine)}
            del sopt, ws_s
            torch.cuda.empty_cache()
        except Exception as exc:  # reported, not fatal: the replica line above stands
            sharded = {"error": f"{type(exc).__name__}: {exc}"[:300]}

    # ---- end to end: host gradients in, status word out, every step ----
    # Each step's gradients come from pinned host memory.  The copy for step
    # t+1 runs on a side stream while step t computes (two device gradient
    # sets, events order the reuse); every copy is inside the timed region,
    # and each step ends with a blocking 4-byte read of the status word.
    e2e = None
    if not args.no_e2e:
        host = [g.to("cpu").pin_memory() for g in grads[0]]
        h2d = sum(h.numel() * h.element_size() for h in host)
        copy_stream = torch.cuda.Stream()
        compute = torch.cuda.current_stream()
        copied = [torch.cuda.Event(), torch.cuda.Event()]
        consumed = [torch.cuda.Event(), torch.cuda.Event()]

        def copy_in(k):
            with torch.cuda.stream(copy_stream):
                copy_stream.wait_event(consumed[k])
                for d, h in zip(grads[k], host):
                    d.copy_(h, non_blocking=True)
                copied[k].record(copy_stream)

        def run(n_steps):
            for k in range(2):
                consumed[k].record(compute)
            copy_in(0)
            for t in range(n_steps):
                k = t % 2
                if t + 1 < n_steps:
                    copy_in(1 - k)
                compute.wait_event(copied[k])
                opt.step(grads[k])
                consumed[k].record(compute)
                mh.get_status()           # synchronises the compute stream; 4-byte device->host read

        run(2)
        e_steps = max(20, args.steps)
        barrier()
        t0 = time.perf_counter()
        run(e_steps)
        torch.cuda.synchronize()
        dt = time.perf_counter() - t0
        if world > 1:
            t_ = torch.tensor([dt], device=dev)
            dist.all_reduce(t_, op=dist.ReduceOp.MAX)
            dt = t_.item()
        e2e = {"value": world * e_steps / dt, "unit": "steps/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": 4, "copy": "next step's gradients copied on a side stream during the step"}

        # The same loop with bf16 gradients (MUONH_FLAG_GRAD_BF16): half the
        # host->device bytes.  A second optimizer on the same weights; reported
        # beside the fp32-gradient line, which stays the headline.
        if args.optimizer != "adamw":
            host_f32 = host
            host = [h.to(torch.bfloat16).pin_memory() for h in host_f32]
            del host_f32
            grads = [[g.to(torch.bfloat16) for g in gs] for gs in grads]
            flags16 = gemm_flags | mh.FLAG_GRAD_BF16
            if args.optimizer == "muon":
                opt = mh.Muon(ws, lr=work.lr, beta=work.beta, weight_decay=MUON_WD, ns_steps=work.ns_steps,
                              ns_coeffs=work.coeffs, eps=work.eps, bf16_copies=True, flags=flags16)
            else:
                opt = mh.MuonH(ws, lr=work.lr, beta=work.beta, ns_steps=work.ns_steps, ns_coeffs=work.coeffs,
                               eps=work.eps, bf16_copies=True, flags=flags16)
            h2d16 = sum(h.numel() * h.element_size() for h in host)
            run(2)
            barrier()
            t0 = time.perf_counter()
            run(e_steps)
            torch.cuda.synchronize()
            dt = time.perf_counter() - t0
            if world > 1:
                t_ = torch.tensor([dt], device=dev)
                dist.all_reduce(t_, op=dist.ReduceOp.MAX)
                dt = t_.item()
            e2e["grad_bf16"] = {"value": world * e_steps / dt, "unit": "steps/s", "h2d_bytes_per_step": h2d16,
                                "d2h_bytes_per_step": 4, "flags": "MUONH_FLAG_GRAD_BF16"}

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    peaks = _peaks()
    ns_kinds = ("ns_gram", "ns_poly", "ns_apply", "ns_apply_in", "ns_apply_out", "ns_apply_in_out", "ns_apply_outw",
                "ns_apply_in_outw")
    ns_ms = sum(prof[k]["ms"] for k in ns_kinds if k in prof)
    ns_sum_ms = ns_ms
    ns_flops = sum(prof[k]["flops"] for k in ns_kinds if k in prof)
    ns_launches = sum(prof[k]["launches"] for k in ns_kinds if k in prof)
    if "ns_busy" in prof and ns_launches == prof["ns_busy"]["launches"]:
        # launches on the side streams overlap: time = union of their intervals
        ns_ms = prof["ns_busy"]["ms"]
    achieved = ns_flops / (ns_ms / 1000.0) / 1e12 if ns_ms > 0 else 0.0
    tr = _ns_traffic_from_profiles()
    if args.optimizer == "adamw":
        a = prof.get("adamw", {"ms": 0.0, "bytes": 0.0, "launches": 0})
        gbs = a["bytes"] / (a["ms"] / 1000.0) / 1e9 if a["ms"] > 0 else 0.0
        roofline = {
            "bound": "hbm", "kernel": "adamw_kernel", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": gbs / peaks["hbm_gbs"], "peak_kind": f"HBM copy bandwidth, {peaks['source']}",
            "traffic": None, "launches": a["launches"], "bytes_per_launch": a["bytes"] / max(a["launches"], 1),
            "ms_per_launch": a["ms"] / max(a["launches"], 1),
        }
    elif ns_launches == 0 and "small_step" in prof:
        # every matrix of the workload took the on-chip small-matrix step
        sm = prof["small_step"]
        tfl = sm["flops"] / (sm["ms"] / 1000.0) / 1e12 if sm["ms"] > 0 else 0.0
        gbs = sm["bytes"] / (sm["ms"] / 1000.0) / 1e9 if sm["ms"] > 0 else 0.0
        roofline = {
            "bound": "tensor", "kernel": "small_step_kernel (whole step on chip, one CTA pair per matrix)",
            "achieved": tfl, "peak": peaks["bf16_sustained"], "unit": "TFLOP/s",
            "frac": tfl / peaks["bf16_sustained"], "peak_kind": f"bf16 dense sustained, {peaks['source']}",
            "frac_of_burst": tfl / peaks["bf16"],
            "hbm": {"achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"],
                    "bytes_per_step": sm["bytes"] / prof_steps},
            "traffic": None, "launches": sm["launches"], "flops_per_launch": sm["flops"] / max(sm["launches"], 1),
            "ms_per_launch": sm["ms"] / max(sm["launches"], 1),
            "timing": f"per-launch CUDA events over {prof_steps} profiled steps after the headline loop",
            "note": "latency-bound: 15 serial 256x256x256 GEMMs and their epilogues per matrix",
        }
    else:
        roofline = {
            "bound": "tensor", "kernel": "ns_gemm_kernel (Gram, polynomial, apply launches)",
            "achieved": achieved, "peak": peaks["bf16_sustained"], "unit": "TFLOP/s",
            "frac": achieved / peaks["bf16_sustained"],
            "peak_kind": f"bf16 dense sustained, {peaks['source']}",
            "frac_of_burst": achieved / peaks["bf16"],
            "traffic": tr["bytes_per_launch"] if tr and tr.get("current") and tr.get("workload") == work.name
                       else None,
            "launches": ns_launches, "flops_per_launch": ns_flops / max(ns_launches, 1),
            "ms_per_launch": ns_ms / max(ns_launches, 1),
            "ns_ms_per_step": ns_ms / prof_steps,
            "ns_kind_busy_sum_per_step": ns_sum_ms / prof_steps,
            "timing": f"per-launch CUDA events on each launch's stream over {prof_steps} profiled steps after the "
                      "headline loop; time = union of the launch intervals (per kind in 'kernels', over all "
                      "Newton-Schulz kinds here)",
            "ns_share_of_step": ns_ms / prof_steps / max(prof_ms_step, 1e-9),
            "profiled_ms_per_step": prof_ms_step,
        }
    hbm = {}
    for k in ("momentum", "hyperball_norm", "hyperball_apply", "hyperball_scale", "muon_finish"):
        if k in prof_hbm and prof_hbm[k]["ms"] > 0:
            gbs = prof_hbm[k]["bytes"] / (prof_hbm[k]["ms"] / 1000.0) / 1e9
            hbm[k] = {"GB/s": gbs, "frac": gbs / peaks["hbm_gbs"], "ms_per_step": prof_hbm[k]["ms"] / hbm_steps}
    if hbm and prof_hbm is not prof:
        hbm["timing"] = f"{hbm_steps} extra steps with every launch on one stream (MUONH_FLAG_ONE_STREAM)"
    line = {
        "metric": {"muon": METRIC_MUON, "adamw": METRIC_ADAMW}.get(args.optimizer, METRIC), "value": value,
        "unit": "steps/s",
        "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": work.name, "matrices": len(work.shapes), "params": work.n_params,
                   "ns_steps": work.ns_steps, "ns_coeffs": list(work.coeffs), "beta": work.beta, "lr": work.lr,
                   "eps": work.eps, "state": "fp32 W/M/G + bf16 W copy; NS bf16 operands, iterate as bf16 hi + bf16 lo (fp32 in the first and last iterations)",
                   "l2": _l2_note(work, args.optimizer),
                   "parallelism": f"replica x{world}",
                   "ns_streams": "caller's stream only" if args.one_stream else
                                 "independent buckets on up to 4 streams (caller's + 3 side streams)",
                   "ns_gemm": {"pair": "2-SM pair 256x256 tiles, two K steps (32 KB TMA boxes) per stage",
                               "pair_one_step": "2-SM pair 256x256 tiles, one K step (16 KB TMA boxes) per stage",
                               "1sm": "1-SM 128x256 tiles"}[args.gemm],
                   "optimizer": {"muon": "muon (weight decay 0.1)",
                                 "adamw": f"adamw (betas {ADAMW_BETAS}, eps {ADAMW_EPS}, weight decay {ADAMW_WD})"
                                 }.get(args.optimizer, "muonh")},
        "ns_tflops": achieved,
        "roofline": roofline,
        "hbm_kernels": hbm,
        "gpu_launches": gpu_launches,
        "clocks": clk.summary(),
        "e2e": e2e,
        **({"sharded": sharded} if sharded is not None else {}),
        "kernels": {k: {"launches": v["launches"], "ms_per_step": v["ms"] / prof_steps,
                        **({"tflops": v["flops"] / (v["ms"] / 1000.0) / 1e12} if v["flops"] and v["ms"] > 0 else {}),
                        **({"GB/s": v["bytes"] / (v["ms"] / 1000.0) / 1e9} if not v["flops"] and v["bytes"] and
                           v["ms"] > 0 else {})}
                    for k, v in prof.items()},
        "kernels_timing": f"per kind, the union of its launches' event intervals over {prof_steps} profiled steps "
                          "(not the headline loop, which runs without per-launch events); with side streams an "
                          "interval includes time a launch waits for SMs held by other buckets' launches",
    }
    if cpu is not None:
        v, cores, sample = cpu
        line["cpu_baseline"] = {"value": v, "unit": "steps/s", "cores": cores, "kind": "oracle", "sample": sample}
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
