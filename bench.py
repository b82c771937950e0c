"""Benchmark of the fused-group hot path on GB300.

One step = one execution of the diamond workload's plan (X, Z [8192, 4096]
float32, bias [4096]; P = X + bias, relu(P) + exp(0.01 P) + P*Z, transposed
to [4096, 8192]): the post-dominator pass fuses all seven operators into one
group, so a step is one kernel launch.  The headline is that group's HBM
throughput counted in algorithmic bytes (each leaf read once, the output
written once) per second, whole job over all ranks.

Printed as one JSON line (rank 0), kept under 3 KB.  Beside the headline the
line carries: the roofline of the dominant kernel, the end-to-end number
through the C ABI with host buffers, the CPU oracle's throughput on a bounded
sample, and `rows`: every other hot-path row measured in the same process,
three significant digits each (us = microseconds per run: the median of
back-to-back runs, or for a flushed single launch the mean of the middle
half of 20 samples; x = speed-up over one kernel per operator, frac =
fraction of the measured HBM copy peak, frac_bf16 = of the measured bf16
peak): the diamond fused and unfused, the
RNNLM chain (1 and 2 groups; as is and scaled to [65536, 1024]), row sums,
the diamond with P returned under the three explicit-fusion plans, the tuple
concatenation, the MLP pattern group, pack and unpack, the AllReduce buckets,
the training-step simulator, the sufficient-factor update at K = 512 and
4096, the random DAG, and the oracle's own times.

Inputs (256 MiB) and the output (128 MiB) together exceed the 129 MB L2, so
the timed loop needs no L2 flush; the smaller rows flush L2 between reps.

Multi-GPU: the fused groups run as replicas -- every rank runs the same plan
on its own data (data-parallel replicas, weak scaling; the headline needs no
collective).  The one exchange step of the path, the AllReduce of the packed
gradient buckets, is the `exchange` row: NCCL over the ranks' bucket byte
ranges, each started as soon as its bucket's count says it is complete.
`--impl reference` times the CPU oracle on a bounded sample instead.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

R, C = 8192, 4096
METRIC = "fused-group HBM GB/s (diamond group, algorithmic bytes)"
WORKLOAD = {"workload": "diamond DAG X,Z[8192,4096] fp32 + bias[4096] -> transpose [4096,8192]",
            "group": "1 fused group of 7 operators", "l2": "inputs+output 384 MiB > L2 (129 MB), no flush"}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return d["hbm_gbs"], d.get("bf16_tflops"), d.get("bf16_tflops_sustained"), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


# ---------------------------------------------------------------------------
class Clocks:
    """nvidia-smi sampled every 20 ms while the timed region runs (the timed
    region starts once the first sample has arrived)."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index, self.rows, self.proc = index, [], None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            t0 = time.time()
            while not self.rows and time.time() - t0 < 5.0 and self.proc.poll() is None:
                time.sleep(0.005)
            self.rows.clear()           # keep the samples taken during the timed region
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([x.strip() for x in line.split(",")])

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.03)
            self.proc.terminate()
            self.proc.wait()

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["not sampled"]}
        sm = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in self.rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.rows)}


# ---------------------------------------------------------------------------
def setup_dist(args):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "native" else "gloo"
        dist.init_process_group(backend)
        return dist, rank, ws, local
    return None, rank, ws, local


def cudart():
    """The CUDA runtime, for pitched copies (cudaMemcpy2DAsync)."""
    import glob
    cands = ["libcudart.so", "/usr/local/cuda/lib64/libcudart.so", "/usr/local/cuda/targets/*/lib/libcudart.so*"]
    for c in cands:
        for path in (glob.glob(c) if "*" in c else [c]):
            try:
                lib = ctypes.CDLL(path)
            except OSError:
                continue
            lib.cudaMemcpy2DAsync.restype = ctypes.c_int
            lib.cudaMemcpy2DAsync.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_size_t,
                                              ctypes.c_size_t, ctypes.c_size_t, ctypes.c_int, ctypes.c_void_p]
            lib.cudaSetDevice.argtypes = [ctypes.c_int]
            return lib
    raise RuntimeError("libcudart not found")


def cpu_sample(rows=1024, reps=3):
    """The oracle, as it stands, on a slab of the diamond workload: `rows` rows
    of X and Z (the same columns), op by op in float64 rounded to float32."""
    import workloads as W
    from oracle import execute as OE
    spec = W.diamond(rows, C)
    ins = W.make_inputs(spec, 0)
    alg = (2 * rows * C + C + rows * C) * 4
    times = []
    for _ in range(reps):
        t0 = time.perf_counter()
        OE.run_unfused(spec, ins)
        times.append(time.perf_counter() - t0)
    t = min(times)
    return {"value": alg / t / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"diamond X,Z[{rows},{C}] slab, best of {reps} ({t:.2f} s)"}


def oracle_samples():
    """The oracle, as it stands, beside the other configurations' GPU rows:
    each on a bounded sample, its wall time and the sample's algorithmic
    throughput (numpy ufuncs run on one core; the float64 matmul of the SF
    update on every BLAS thread)."""
    import workloads as W
    from oracle import execute as OE
    from oracle import pack as OP

    def best(f, reps=2):
        ts = []
        for _ in range(reps):
            t0 = time.perf_counter()
            f()
            ts.append(time.perf_counter() - t0)
        return min(ts)

    out = {}
    sp = W.rnnlm_chain()
    ins = W.make_inputs(sp, 0)
    out["rnnlm_ms"] = best(lambda: OE.run_unfused(sp, ins), 3) * 1e3          # the whole chain, 1 core
    # SF update on rows 0..255 of W (1/16 of the output; BLAS on every core),
    # scaled to the full output
    sp = W.sf_update(512, 256, 4096)
    ins = W.make_inputs(sp, 0)
    out["sf_k512_ms_est"] = best(lambda: OE.run_unfused(sp, ins)) * 16e3
    out["sf_cores"] = os.cpu_count()
    sizes = W.tensor_fusion_sizes(0)
    xs = W.tensor_fusion_inputs(sizes)
    out["pack_GBps"] = int(sizes.sum()) * 6 / best(lambda: OP.pack(xs, 0.125)) / 1e9    # all 161 tensors
    # the 200-operator graph on [512,256] values (1/256 of the elements), scaled
    sp = W.random_dag(0, R=512, C=256, nominal_R=8192, nominal_C=4096)
    ins = W.make_inputs(sp, 0)
    out["dag200_ms_est"] = best(lambda: OE.run_unfused(sp, ins), 1) * 256e3
    return out


def run_reference(args):
    dist, rank, ws, _ = setup_dist(args)
    if rank != 0:
        return
    # each step a slab of the workload (256 rows, fewer when many steps are
    # asked for) so that the whole run stays within a minute and a half of CPU
    # time; the oracle takes about 1.1 ms per 4096-wide row
    rows = max(8, min(256, int(90.0 / (args.steps + args.warmup) / 1.1e-3) // 8 * 8))
    for _ in range(args.warmup):
        cpu_sample(rows, 1)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        s = cpu_sample(rows, 1)
    t = time.perf_counter() - t0
    alg = (3 * rows * C + C) * 4
    v = alg * args.steps / t / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": t / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": dict(WORKLOAD, sample=f"CPU oracle on a [{rows},{C}] slab per step"),
            "cpu_baseline": {"value": v, "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": f"diamond slab X,Z[{rows},{C}] per step"},
            "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--no-rows", action="store_true", help="skip the secondary rows")
    ap.add_argument("--workload", default="diamond",
                    choices=["diamond", "sf_update", "sf_update_k4096", "pack", "unpack", "rowsum", "rnnlm"],
                    help="diamond is the headline; the others time one kernel of another row "
                         "(used for profiling), with the same JSON fields")
    ap.add_argument("--flags", type=lambda x: int(x, 0), default=0,
                    help="plan tuning flags (fg_build_opts.flags) for --workload runs")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    if args.workload != "diamond":
        return run_single(args)

    import torch
    import workloads as W
    from group_execution_gb300 import graph_from_spec, _lib

    dist, rank, ws, local = setup_dist(args)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    hbm, bf16, bf16s, peak_kind = peaks()

    spec = W.diamond(R, C)
    plan = graph_from_spec(spec).build()
    assert plan.n_groups == 1
    info = plan.groups[0]
    ins = W.make_inputs(spec, seed=rank)
    dv = {k: torch.from_numpy(v).to(dev) for k, v in ins.items()}
    out = torch.empty((C, R), device=dev)
    tensors = {v: dv[v] for v in info.leaves} | {info.out: out}
    ptrs = plan._ptrs(tensors)
    sh = ctypes.c_void_p(stream.cuda_stream)

    def step():
        st = plan.launch_group_ptrs(0, ptrs, sh)
        if st:
            _lib.check(st)

    def barrier():
        if dist:
            dist.barrier()

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with Clocks(local) as clk:
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    barrier()
    if dist:
        t = torch.tensor([ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    plan.sync()
    ms_step = ms / args.steps
    value = ws * info.alg_bytes * args.steps / (ms * 1e-3) / 1e9
    achieved = info.alg_bytes / (ms_step * 1e-3) / 1e9

    # end to end through the C ABI: pinned host inputs in, the result back in
    # host memory, per step.  Pipelined over row slabs of X and Z: each slab
    # is a diamond group of its own whose transposed output is a column slab
    # of the result (written back with a pitched copy); host-to-device copies,
    # kernels and device-to-host copies run on three streams, so both copy
    # directions and the kernels overlap.
    hin = {v: dv[v].cpu().pin_memory() for v in info.leaves}
    hout = torch.empty((C, R), pin_memory=True)
    e2e_steps = max(3, min(args.steps, 8))
    RC, NSLOT = 1024, 3
    cplan = graph_from_spec(W.diamond(RC, C)).build()
    cinfo = cplan.groups[0]
    XV, BV, ZV = 0, 1, 2                      # value ids of X, bias, Z in a diamond graph
    slots = [{XV: torch.empty((RC, C), device=dev), ZV: torch.empty((RC, C), device=dev),
              BV: torch.empty((C,), device=dev), cinfo.out: torch.empty((C, RC), device=dev)} for _ in range(NSLOT)]
    cptrs = [cplan._ptrs({v: sl[v] for v in cinfo.leaves + [cinfo.out]}) for sl in slots]
    s_in, s_run, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev_run = [torch.cuda.Event() for _ in range(NSLOT)]
    ev_in = [torch.cuda.Event() for _ in range(NSLOT)]
    ev_out = [torch.cuda.Event() for _ in range(NSLOT)]
    rt = cudart()
    rt.cudaSetDevice(local)

    def e2e_step():
        for k in range(R // RC):
            sl, r0 = k % NSLOT, k * RC
            with torch.cuda.stream(s_in):
                if k >= NSLOT:
                    s_in.wait_event(ev_run[sl])          # the slot's inputs have been read
                slots[sl][XV].copy_(hin[XV][r0:r0 + RC], non_blocking=True)
                slots[sl][ZV].copy_(hin[ZV][r0:r0 + RC], non_blocking=True)
                slots[sl][BV].copy_(hin[BV], non_blocking=True)
                ev_in[sl].record(s_in)
            s_run.wait_event(ev_in[sl])
            if k >= NSLOT:
                s_run.wait_event(ev_out[sl])             # the slot's output has been copied out
            st = cplan.launch_group_ptrs(0, cptrs[sl], ctypes.c_void_p(s_run.cuda_stream))
            if st:
                _lib.check(st)
            ev_run[sl].record(s_run)
            s_out.wait_event(ev_run[sl])
            err = rt.cudaMemcpy2DAsync(ctypes.c_void_p(hout.data_ptr() + r0 * 4), ctypes.c_size_t(R * 4),
                                       ctypes.c_void_p(slots[sl][cinfo.out].data_ptr()), ctypes.c_size_t(RC * 4),
                                       ctypes.c_size_t(RC * 4), ctypes.c_size_t(C), 2,
                                       ctypes.c_void_p(s_out.cuda_stream))
            if err:
                raise RuntimeError(f"cudaMemcpy2DAsync failed ({err})")
            ev_out[sl].record(s_out)

    def bracket(fn):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for s_ in (s_in, s_run, s_out):
            s_.wait_stream(stream)
        fn()
        for s_ in (s_in, s_run, s_out):
            stream.wait_stream(s_)
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b)

    bracket(e2e_step)
    assert torch.equal(hout, out.cpu()), "end-to-end result differs from the device result"
    barrier()
    ms_e2e = bracket(lambda: [e2e_step() for _ in range(e2e_steps)]) / e2e_steps
    h2d = sum(hin[v].numel() * 4 for v in info.leaves) + (R // RC - 1) * hin[BV].numel() * 4
    e2e = {"value": ws * info.alg_bytes / (ms_e2e * 1e-3) / 1e9, "unit": "GB/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": hout.numel() * 4, "ms_per_step": ms_e2e,
           "pipeline": f"{R // RC} row slabs of {RC}, {NSLOT} buffer slots, 3 streams"}

    line = {"metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": dict(WORKLOAD, parallelism=f"replicas x{ws}"),
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                         "frac": achieved / hbm, "traffic": traffic_for("fg_jit_ew_group", "diamond"),
                         "kernel": "fg_jit_ew_group", "peak_source": peak_kind,
                         "alg_bytes_per_launch": info.alg_bytes},
            "e2e": e2e, "gpu_launches": args.steps, "clocks": clk.summary()}
    if not args.no_rows:
        xrow = exchange_row(torch, dist, ws, rank, hbm)   # every rank takes part
    if rank == 0 and not args.no_rows:
        line["rows"] = secondary_rows(torch, W, graph_from_spec, plan, spec, dv, out, hbm, bf16, bf16s)
        line["rows"]["exchange"] = _round(xrow)
        line["cpu_baseline"] = cpu_sample()
        line["rows"]["oracle"] = _round(oracle_samples())
    if rank == 0:
        for k in [k for k in ("roofline", "e2e", "cpu_baseline") if k in line]:
            line[k] = {a: (float(f"{b:.5g}") if isinstance(b, float) else b) for a, b in line[k].items()}
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def exchange_row(torch, dist, ws, rank, hbm):
    """The data-parallel gradient exchange around tensor fusion (DisCo,
    Background and Introduction; ring AllReduce in DisCo, Simulator), on every
    rank: the 161 gradients packed into AllReduce buckets (8 MiB threshold) in
    one launch, scaled by 1/N; a second stream waits for each bucket's ready
    word and all-reduces the bucket's byte range over NCCL (bf16 sum of the
    scaled gradients = their mean); every gradient unpacked after the last
    bucket.  One rank has nothing to exchange: the same pipeline without the
    collective.  Time per step: max over ranks of 20 steps after 3."""
    import workloads as W
    from group_execution_gb300 import TensorFusion, plan_threshold
    sizes = W.tensor_fusion_sizes(0)
    xs = [torch.from_numpy(x).cuda() for x in W.tensor_fusion_inputs(sizes, rank)]
    tf = TensorFusion(xs)
    bounds = plan_threshold(list(sizes), 8 << 20)
    tf.set_buckets(bounds)
    buf = torch.empty((tf.total_bytes,), dtype=torch.uint8, device="cuda")
    views = [buf[a:b].view(torch.bfloat16) for a, b in tf.bucket_ranges(bounds)]
    main, comm = torch.cuda.current_stream(), torch.cuda.Stream()

    def step():
        tf.pack_buckets(1.0 / ws, buf, stream=main)
        for k, v in enumerate(views):
            tf.bucket_wait(k, stream=comm)
            if ws > 1:
                with torch.cuda.stream(comm):
                    dist.all_reduce(v)
        main.wait_stream(comm)
        tf.unpack(1.0, buf, stream=main)

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(main)
    for _ in range(20):
        step()
    b.record(main)
    torch.cuda.synchronize()
    us = a.elapsed_time(b) / 20 * 1e3
    if dist:
        t = torch.tensor([us], device="cuda")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        us = float(t.item())
    nbytes = sum(b - a for a, b in tf.bucket_ranges(bounds))
    row = {"n": ws, "buckets": len(views), "us": us, "bf16_MB": nbytes / 1e6}
    if ws > 1:
        row["busbw_GBps"] = 2 * (ws - 1) / ws * nbytes / (us * 1e-6) / 1e9
    else:
        row["allreduce"] = "none (1 rank)"
    del xs, buf
    return row


def run_single(args):
    """One other hot-path row on one GPU: warm-up, then K timed launches."""
    import torch
    import workloads as W
    from group_execution_gb300 import graph_from_spec, TensorFusion
    torch.cuda.set_device(0)
    hbm, bf16, _, peak_kind = peaks()
    flops = 0
    if args.workload in ("pack", "unpack"):
        sizes = W.tensor_fusion_sizes(0)
        xs = [torch.from_numpy(x).cuda() for x in W.tensor_fusion_inputs(sizes)]
        tf = TensorFusion(xs)
        buf = torch.empty((tf.total_bytes,), dtype=torch.uint8, device="cuda")
        tf.pack(0.125, buf)
        fn = (lambda: tf.pack(0.125, buf)) if args.workload == "pack" else (lambda: tf.unpack(1.0, buf))
        alg, kernel, wl = int(sizes.sum()) * 6, "tf_" + args.workload + "_kernel", "161 gradient tensors, 25.6M elements"
    else:
        if args.workload == "rowsum":
            spec = W.GraphSpec("rowsum")
            x = spec.input((R, C))
            spec.mark_output(spec.op("rowsum", (x,)))
        elif args.workload == "rnnlm":
            spec = W.rnnlm_chain()
        else:
            spec = W.sf_update(4096 if args.workload == "sf_update_k4096" else 512, 4096, 4096)
        plan = graph_from_spec(spec).build(allow_reduce_epilogue=args.workload == "rnnlm", flags=args.flags)
        env = {}
        for k, v in W.make_inputs(spec).items():
            t = torch.from_numpy(v).cuda()
            env[k] = t.to(torch.bfloat16) if spec.values[k].dtype == "bf16" else t
        for gi in plan.groups:
            env[gi.out] = torch.empty(spec.values[gi.out].shape, device="cuda")

        sh = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        launches = [(gid, plan._ptrs({v: env[v] for v in gi.leaves + [gi.out]})) for gid, gi in enumerate(plan.groups)]

        def fn():
            for gid, ptrs in launches:
                st = plan.launch_group_ptrs(gid, ptrs, sh)
                if st:
                    raise RuntimeError(f"launch failed ({st})")
        alg = sum(gi.alg_bytes for gi in plan.groups)
        flops = sum(gi.alg_flops for gi in plan.groups)
        kernel = {"elementwise": "fg_jit_ew_group", "reduce": "fg_jit_reduce_group",
                  "gemm": "fg_jit_gemm_group"}[plan.groups[-1].kind]
        if plan.direct_info(len(plan.groups) - 1)["direct"]:
            kernel = "fg_jit_small_group"   # the direct kernel (leaves read straight from global memory)
        wl = spec.name
    for _ in range(max(3, args.warmup)):
        fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with Clocks(0) as clk:
        a.record()
        for _ in range(args.steps):
            fn()
        b.record()
        torch.cuda.synchronize()
    ms = a.elapsed_time(b) / args.steps
    gbps = alg / (ms * 1e-3) / 1e9
    line = {"metric": f"{args.workload} HBM GB/s (algorithmic bytes)", "value": gbps, "unit": "GB/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": wl}, "gpu_launches": args.steps,
            "roofline": {"bound": "hbm", "achieved": gbps, "peak": hbm, "unit": "GB/s", "frac": gbps / hbm,
                         "traffic": traffic_for(kernel, {"sf_update": "sfk512", "sf_update_k4096": "sfk4096"}.get(
                             args.workload, args.workload)), "kernel": kernel, "peak_source": peak_kind},
            "clocks": clk.summary()}
    if flops:
        line["TFLOPs"] = flops / (ms * 1e-3) / 1e12
        line["frac_of_bf16_peak"] = line["TFLOPs"] / bf16
    print(json.dumps(line), flush=True)


# The sources that define each kernel: its device code, its generated program
# and its launch configuration.  A committed capture counts only while these
# hash to the value recorded with it.
_GROUP = ("fg_abi.h", "fg_device.cuh", "group_kernels.cuh", "jit.cpp", "host_compile.cpp", "api.cpp")
KERNEL_SOURCES = {
    "fg_jit_ew_group": _GROUP, "fg_jit_reduce_group": _GROUP, "fg_jit_small_group": _GROUP,
    "fg_jit_gemm_group": ("fg_abi.h", "fg_device.cuh", "gemm_kernel.cuh", "jit.cpp", "host_compile.cpp", "api.cpp"),
    "tf_pack_kernel": ("fg_abi.h", "fg_device.cuh", "k_pack.cu", "launch.h", "api.cpp"),
    "tf_unpack_kernel": ("fg_abi.h", "fg_device.cuh", "k_pack.cu", "launch.h", "api.cpp"),
}


def traffic_for(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the kernel's current sources."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        d = json.load(open(p))[workload]
    except Exception:
        return None
    if d.get("kernel") != kernel or d.get("sources") != sources_hash(kernel):
        return None
    return d.get("dram_bytes_per_launch")


def sources_hash(kernel):
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "group_execution_gb300", "csrc")
    for f in KERNEL_SOURCES[kernel]:
        h.update(f.encode())
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


# ---------------------------------------------------------------------------
def secondary_rows(torch, W, graph_from_spec, plan, spec, dv, out, hbm, bf16, bf16s):
    """Other hot-path rows, measured outside the headline's timed region."""
    from group_execution_gb300 import _lib
    rows = {}
    l2 = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    l2r = torch.zeros(256 << 20, dtype=torch.uint8, device="cuda")

    def timed(fn, reps=10, flush=True, inner=None):
        """Typical and min ms of `inner` back-to-back calls (L2 flushed first
        when asked: written, then evicted clean), over `reps` repetitions.
        Without a flush the calls run ten at a time by default: a single call
        after a synchronize would also count the host's launch work, during
        which the device is idle (after a flush, the flush kernel covers it);
        the typical value is the median.  A flushed single call is timed 20
        times and the typical value is the mean of the middle half: event
        times move in steps of about 1 us on this GPU, and the median of such
        samples lands on one step or the next from run to run."""
        if inner is None:
            inner = 1 if flush else 10
        if flush and inner == 1:
            reps = max(reps, 20)
        fn()
        torch.cuda.synchronize()
        ts = []
        for _ in range(reps):
            if flush:
                # write a buffer twice L2's size, then read another: L2 ends
                # cold and clean, so the timed launch neither hits its own
                # data nor writes back the flush's dirty lines
                l2.fill_(1)
                l2r.max()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            for _ in range(inner):
                fn()
            b.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b) / inner)
        if flush and inner == 1:
            mid = sorted(ts)[len(ts) // 4: len(ts) - len(ts) // 4]
            return sum(mid) / len(mid), min(ts)
        return statistics.median(ts), min(ts)

    def graphed(fn, n=1):
        """n runs of fn's launches captured once into a CUDA graph and
        replayed: device time without per-launch host work."""
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            fn()
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(n):
                fn()
        return g.replay

    def run_plan(p, sp, env, fused=True):
        """Every group (or every operator) of the plan in order, with the
        pointer arrays marshalled once: the host's per-launch work stays
        below the kernels' time."""
        if fused:
            launches = [(p.lib.fg_launch_group, gid, p._ptrs({v: env[v] for v in gi.leaves + gi.outs}))
                        for gid, gi in enumerate(p.groups)]
        else:
            launches, node = [], 0
            for v in sp.values:
                if not v.is_input:
                    launches.append((p.lib.fg_launch_unfused, node,
                                     p._ptrs({a: env[a] for a in v.args} | {v.vid: env[v.vid]})))
                    node += 1

        def f():
            # the stream current at the call (a CUDA-graph capture's, too)
            sh = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
            for fn, k, ptrs in launches:
                st = fn(p.h, k, ptrs, sh)
                if st:
                    _lib.check(st)
        return f

    # diamond, unfused: seven kernels, intermediates in HBM
    env = dict(dv)
    for v in spec.ops:
        env[v.vid] = torch.empty(v.shape, device="cuda")
    env[spec.outputs[0]] = out
    med_f, _ = timed(run_plan(plan, spec, env, True), flush=False)
    med_u, _ = timed(run_plan(plan, spec, env, False), flush=False)
    rows["diamond"] = {"us": med_f * 1e3, "unf_us": med_u * 1e3, "x": med_u / med_f,
                       "frac": plan.groups[0].alg_bytes / (med_f * 1e-3) / 1e9 / hbm}

    # RNNLM chain, both partitions (launch-bound by construction): one run
    # after an L2 flush (us), and 20 runs back to back replayed from a CUDA
    # graph, per run (graph_us: no host work between launches)
    for epi in (False, True):
        sp = W.rnnlm_chain()
        p = graph_from_spec(sp).build(allow_reduce_epilogue=epi)
        e = {k: torch.from_numpy(v).cuda() for k, v in W.make_inputs(sp).items()}
        for gi in p.groups:
            e[gi.out] = torch.empty(sp.values[gi.out].shape, device="cuda")
        for v in sp.ops:
            e.setdefault(v.vid, torch.empty(v.shape, device="cuda"))
        med, mn = timed(run_plan(p, sp, e, True))
        medu, _ = timed(run_plan(p, sp, e, False))
        gmed, _ = timed(graphed(run_plan(p, sp, e, True), 20), flush=False, inner=1)
        gmedu, _ = timed(graphed(run_plan(p, sp, e, False), 20), flush=False, inner=1)
        gmed, gmedu = gmed / 20, gmedu / 20
        rows["rnnlm_" + ("1g" if epi else "2g")] = {
            "us": med * 1e3, "unf_us": medu * 1e3, "graph_us": gmed * 1e3, "graph_unf_us": gmedu * 1e3}

    # the same chain scaled to X, Y [65536, 1024] (512 MiB): bandwidth-bound,
    # so its roofline fraction means something; inputs exceed L2, no flush
    for epi in (False, True):
        sp = W.rnnlm_chain(65536, 1024)
        p = graph_from_spec(sp).build(allow_reduce_epilogue=epi)
        gen = torch.Generator(device="cuda").manual_seed(0)
        e = {v.vid: torch.empty(v.shape, device="cuda").uniform_(-1.0, 1.0, generator=gen)
             for v in sp.values if v.is_input}
        for v in sp.ops:
            e[v.vid] = torch.empty(v.shape, device="cuda")
        med, mn = timed(run_plan(p, sp, e, True), flush=False)
        medu, _ = timed(run_plan(p, sp, e, False), flush=False)
        alg = sum(gi.alg_bytes for gi in p.groups)
        rows["rnnlm65536_" + ("1g" if epi else "2g")] = {
            "us": med * 1e3, "x": medu / med, "frac": alg / (med * 1e-3) / 1e9 / hbm}
        del e

    # row sums over [8192, 4096] and [4096, 8192] (134 MB each, above L2)
    for shp in ((8192, 4096), (4096, 8192)):
        sp = W.GraphSpec("rowsum")
        x = sp.input(shp)
        sp.mark_output(sp.op("rowsum", (x,)))
        p = graph_from_spec(sp).build()
        gen = torch.Generator(device="cuda").manual_seed(3)
        e = {x: torch.empty(shp, device="cuda").uniform_(-1, 1, generator=gen),
             sp.outputs[0]: torch.empty((shp[0],), device="cuda")}
        med, _ = timed(run_plan(p, sp, e, True), flush=False)
        rows[f"rowsum{shp[0]}x{shp[1]}"] = {"us": med * 1e3,
                                            "frac": p.groups[0].alg_bytes / (med * 1e-3) / 1e9 / hbm}
        del e

    # explicit fusion moves on the diamond when P = X + bias is also a result
    # the caller keeps: FuseOps ends a group at P (2 groups, P written and
    # read back); non-duplicate fusion of relu with P gives one group with P
    # as an extra output; duplicate fusion copies P into each of its readers'
    # group (P recomputed there; the two groups no longer depend on each other)
    sp = W.diamond(R, C)
    sp.mark_output(sp.ops[0].vid)
    gsp = graph_from_spec(sp)
    e = dict(dv)
    for v in sp.ops:
        e[v.vid] = torch.empty(v.shape, device="cuda")
    plans = {"fuseops": gsp.build()}
    pn = gsp.partition(from_fuseops=True)
    pn.fuse(1, 0, False)
    plans["nondup"] = pn.build()
    pd = gsp.partition(from_fuseops=True)
    for reader in (1, 2, 4):
        pd.fuse(reader, 0, True)
    plans["dup"] = pd.build()
    row = {}
    for k, pl in plans.items():
        med, _ = timed(run_plan(pl, sp, e, True), flush=False)
        alg = sum(gi.alg_bytes for gi in pl.groups)
        row[k + "_us"] = med * 1e3
        row[k + "_frac"] = alg / (med * 1e-3) / 1e9 / hbm
    rows["diamond_P"] = row
    del e

    # two branches joined by a tuple and a concatenation (FuseOps phases 1 and
    # 2): relu(X1), exp(X2) [4096, 4096] each -> concat [8192, 4096] -> scale,
    # one group, against one kernel per operator
    tsp = W.GraphSpec("inception")
    t1 = tsp.op("relu", (tsp.input((4096, 4096)),))
    t2 = tsp.op("exp", (tsp.input((4096, 4096)),))
    tsp.mark_output(tsp.op("scale", (tsp.op("concat", (tsp.op("tuple", (t1, t2)),)),), (0.5,)))
    tplan = graph_from_spec(tsp).build()
    gen = torch.Generator(device="cuda").manual_seed(2)
    te = {v.vid: torch.empty(v.shape, device="cuda").uniform_(-1, 1, generator=gen) for v in tsp.values if v.is_input}
    for v in tsp.ops:
        te[v.vid] = torch.empty(v.shape, device="cuda")
    med, _ = timed(run_plan(tplan, tsp, te, True), flush=False)
    medu, _ = timed(run_plan(tplan, tsp, te, False), flush=False)
    alg = sum(gi.alg_bytes for gi in tplan.groups)
    rows["tuple"] = {"us": med * 1e3, "x": medu / med, "frac": alg / (med * 1e-3) / 1e9 / hbm}
    del te

    # an MLP layer grouped by pattern (FuseOpsByPattern with the page's matmul +
    # bias pattern extended by relu): Y = relu(X W + b), X [4096, 4096],
    # W [4096, 4096] bf16, one GEMM-epilogue group; L2 flushed between runs
    msp = W.GraphSpec("mlp")
    mx = msp.input((4096, 4096), "bf16")
    mw = msp.input((4096, 4096), "bf16")
    mb = msp.input((4096,))
    my = msp.op("relu", (msp.op("badd_col", (msp.op("matmul_bf16", (mx, mw), (0, 0)), mb)),))
    msp.mark_output(my)
    mpart = graph_from_spec(msp).partition(patterns=[("matmul_bias_relu", ["matmul_bf16", "badd_col", "relu"], True)])
    mplan = mpart.build()
    gen = torch.Generator(device="cuda").manual_seed(1)
    me = {mx: torch.empty((4096, 4096), device="cuda").normal_(generator=gen).to(torch.bfloat16),
          mw: torch.empty((4096, 4096), device="cuda").normal_(generator=gen).to(torch.bfloat16),
          mb: torch.empty((4096,), device="cuda").uniform_(-1, 1, generator=gen),
          my: torch.empty((4096, 4096), device="cuda")}
    mgi = mplan.groups[0]
    med, _ = timed(lambda: mplan.launch_group(0, {v: me[v] for v in mgi.leaves + mgi.outs}))
    tf_ = mgi.alg_flops / (med * 1e-3) / 1e12
    rows["mlp"] = {"us": med * 1e3, "TFLOPs": tf_, "frac": tf_ / bf16}
    del me

    # tensor-fusion pack / unpack
    from group_execution_gb300 import TensorFusion
    sizes = W.tensor_fusion_sizes(0)
    xs = [torch.from_numpy(x).cuda() for x in W.tensor_fusion_inputs(sizes)]
    tf = TensorFusion(xs)
    buf = torch.empty((tf.total_bytes,), dtype=torch.uint8, device="cuda")
    nbytes = int(sizes.sum()) * 6
    # 153.6 MB per call exceeds L2: back-to-back calls, no flush
    mp, _ = timed(lambda: tf.pack(0.125, buf), flush=False, inner=10)
    mu, _ = timed(lambda: tf.unpack(1.0, buf), flush=False, inner=10)
    rows["pack"] = {"us": mp * 1e3, "frac": nbytes / (mp * 1e-3) / 1e9 / hbm}
    rows["unpack"] = {"us": mu * 1e3, "frac": nbytes / (mu * 1e-3) / 1e9 / hbm}

    # the same gradients cut into AllReduce buckets by an 8 MiB fusion
    # threshold: packed one launch per bucket (replayed from a CUDA graph),
    # and every bucket in one launch with per-bucket chunk counts; ready_us:
    # when a second stream waiting on each bucket's word passes it, from the
    # launch's start (an L2 flush runs first on the launching stream, so that
    # every wait is enqueued before the pack starts)
    from group_execution_gb300 import plan_threshold
    bounds = plan_threshold(list(sizes), 8 << 20)
    nb = len(bounds) - 1

    def each_bucket(fn, s):
        return lambda: [fn(bounds[k], bounds[k + 1] - bounds[k], s, buf) for k in range(nb)]

    gp, _ = timed(graphed(each_bucket(tf.pack_range, 0.125)), flush=False, inner=10)
    gu, _ = timed(graphed(each_bucket(tf.unpack_range, 1.0)), flush=False, inner=10)
    tf.set_buckets(bounds)
    ob, _ = timed(lambda: tf.pack_buckets(0.125, buf), flush=False, inner=10)
    s2 = torch.cuda.Stream()
    ready = [[] for _ in range(nb)]
    for _ in range(10):
        torch.cuda.synchronize()
        l2.fill_(1)
        l2r.max()
        st = torch.cuda.Event(enable_timing=True)
        st.record()
        tf.pack_buckets(0.125, buf)
        evs = []
        for k in range(nb):
            tf.bucket_wait(k, s2)
            ev = torch.cuda.Event(enable_timing=True)
            ev.record(s2)
            evs.append(ev)
        torch.cuda.synchronize()
        for k in range(nb):
            ready[k].append(st.elapsed_time(evs[k]) * 1e3)
    # the same launch with one more CTA consuming the bucket counts on the
    # device: how long before the last packing CTA finished each bucket was
    # seen ready (median of 10)
    tms = torch.zeros(nb + 1, dtype=torch.int64, device="cuda")
    lead = [[] for _ in range(nb)]
    for _ in range(10):
        tf.pack_buckets_observed(0.125, buf, tms)
        tf.sync()
        t = tms.cpu().numpy()
        for k in range(nb):
            lead[k].append((int(t[nb]) - int(t[k])) / 1e3)
    rows["buckets8MiB"] = {"n": nb, "graph_pack_us": gp * 1e3, "graph_unpack_us": gu * 1e3,
                           "one_launch_us": ob * 1e3, "one_launch_frac": nbytes / (ob * 1e-3) / 1e9 / hbm,
                           "ready_us": [round(statistics.median(r), 1) for r in ready],
                           "dev_lead_us": [round(statistics.median(r), 1) for r in lead]}

    # training-step simulator fed by measured group times: a backward pass of
    # 161 gradient computations (g_i = 0.5 * relu(x_i) over the gradient set's
    # sizes, one group each, run in production order), every group timed on
    # this GPU (device time per launch: 20 launches replayed from a CUDA
    # graph), then the step simulated with AllReduce buckets of the bf16
    # gradients for several fusion thresholds on an 8-GPU ring
    # T = 2(N-1)x/(B N) + D with B = 900 GB/s per link direction and
    # D = 20 us per AllReduce (assumed: the pages give none)
    from group_execution_gb300 import simulate
    bsp = W.GraphSpec("backward")
    grads = []
    for n_i in sizes:
        x_i = bsp.input((int(n_i),))
        grads.append(bsp.op("scale", (bsp.op("relu", (x_i,)),), (0.5,)))
        bsp.mark_output(grads[-1])
    bplan = graph_from_spec(bsp).build()
    be = {}
    for v in bsp.values:
        be[v.vid] = torch.empty(v.shape, device="cuda").uniform_(-1, 1) if v.is_input else torch.empty(v.shape, device="cuda")
    op_time = []
    for gid, gi in enumerate(bplan.groups):
        ptrs = {v: be[v] for v in gi.leaves + gi.outs}
        rep = graphed(lambda gid=gid, ptrs=ptrs: [bplan.launch_group(gid, ptrs) for _ in range(20)])
        med, _ = timed(rep, reps=3, flush=False)
        op_time.append(med * 1e-3 / 20)
    edges = [(k, k + 1) for k in range(len(op_time) - 1)]
    gbytes = [int(n_i) * 2 for n_i in sizes]
    c_ring = 2.0 * 7 / (900e9 * 8)
    sim = {}
    for thr in (0, 1 << 20, 4 << 20, 16 << 20, 1 << 40):
        bb = plan_threshold(list(sizes), thr)
        buckets = [list(range(bb[k], bb[k + 1])) for k in range(len(bb) - 1)]
        tot, *_ = simulate(op_time, edges, list(range(len(sizes))), gbytes, buckets, c_ring, 20e-6)
        sim["one" if thr >= 1 << 40 else "per_tensor" if thr == 0 else str(thr >> 20) + "MiB"] = tot * 1e6
    rows["sim161"] = {"compute_us": sum(op_time) * 1e6, "step_us": sim}
    del be

    # sufficient-factor gradient + update: one tcgen05 GEMM-epilogue group,
    # L2 flushed before each launch
    for B, label in ((512, "sf_k512"), (4096, "sf_k4096")):
        sp = W.sf_update(B, 4096, 4096)
        p = graph_from_spec(sp).build()
        e = {}
        for k, v in W.make_inputs(sp).items():
            t = torch.from_numpy(v).cuda()
            e[k] = t.to(torch.bfloat16) if sp.values[k].dtype == "bf16" else t
        for v in sp.ops:
            e[v.vid] = torch.empty(v.shape, device="cuda")
        gi = p.groups[0]
        med, mn = timed(run_plan(p, sp, e, True))
        medu, _ = timed(run_plan(p, sp, e, False))
        tflops = gi.alg_flops / (med * 1e-3) / 1e12
        gbps = gi.alg_bytes / (med * 1e-3) / 1e9
        rows[label] = {"us": med * 1e3, "x": medu / med, "TFLOPs": tflops, "frac_bf16": tflops / bf16,
                       "frac_hbm": gbps / hbm}
        del e
    torch.cuda.empty_cache()

    # random DAG (seed 0), every group in order vs one kernel per operator
    sp = W.random_dag(0)
    p = graph_from_spec(sp).build()
    e = {k: torch.from_numpy(v).cuda() for k, v in W.make_inputs(sp).items()}
    for v in sp.ops:
        e[v.vid] = torch.empty(v.shape, device="cuda")
    medf, _ = timed(run_plan(p, sp, e, True), reps=3, flush=False)
    medu, _ = timed(run_plan(p, sp, e, False), reps=3, flush=False)
    alg = sum(gi.alg_bytes for gi in p.groups)
    rows["dag200"] = {"groups": p.n_groups, "ms": medf, "unf_ms": medu, "x": medu / medf,
                      "frac": alg / (medf * 1e-3) / 1e9 / hbm}
    del e
    torch.cuda.empty_cache()
    return {k: _round(v) for k, v in rows.items()}


def _round(v):
    """Three significant digits: the line stays short."""
    if isinstance(v, dict):
        return {k: _round(x) for k, x in v.items()}
    if isinstance(v, list):
        return [_round(x) for x in v]
    if isinstance(v, float):
        return float(f"{v:.3g}")
    return v


if __name__ == "__main__":
    main()
