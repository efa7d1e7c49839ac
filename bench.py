#!/usr/bin/env python
"""Benchmark of exact blockwise ring attention on GB300: causal fwd+bwd TFLOP/s.

One step = the whole path on one batch of synthetic input: ra_fwd (forward kernel)
then the backward's three stages (preprocess, main kernel, dQ finalize).  FLOPs count
causal-useful work only: per unmasked (query, key) pair 4*D forward and 10*D backward
(five products, the recompute included).

  python bench.py [--gpus N] [--steps K] [--warmup W]
                  [--workload 1m|262k|32k|8k|32k-gqa|32k-d64|32k-bpt]
                  [--layout striped|contiguous|zigzag] [--impl ours|reference]

The default workload is the largest one: 1,048,576 tokens, 8 heads of 128, P = 32 virtual
shards, block 256, causal, striped.

N > 1 runs under torchrun: every rank runs an independent replica on its own GPU (the
path has no exchange between GPUs); the rate is all ranks' FLOPs over the slowest
rank's time.  ``--impl reference`` times the fp64 CPU oracle on a bounded sample of the
same workload (rank 0 only).  Rank 0 prints one JSON line.
"""

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

METRIC = "causal attention fwd+bwd TFLOP/s and % of GB300 dense BF16 peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: 4 for the 1M-token workload, else 10)")
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="1m",
                    choices=["8k", "32k", "262k", "1m", "32k-gqa", "32k-d64", "32k-bpt"])
    ap.add_argument("--layout", default=None, choices=["striped", "contiguous", "zigzag"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-merge", action="store_true")
    ap.add_argument("--train", action="store_true",
                    help="layer workload only: forward + backward of the layer per step")
    ap.add_argument("--heads", type=int, default=None,
                    help="run the workload with this many heads (a smaller case of the same "
                         "kernels, e.g. for a profiler capture)")
    a = ap.parse_args()
    a.warmup = max(3, a.warmup)
    if a.steps is None:
        a.steps = 4 if a.workload == "1m" else 10
    return a


def workload(name, layout, heads=None):
    from exact_blockwise_ring_gb300.synthetic import WORKLOADS, SEEDS
    w = dict(WORKLOADS[name])
    w["name"] = name
    w["seed"] = SEEDS[name]
    w["layout"] = layout or w["layouts"][0]
    if heads is not None and heads != w["heads"]:
        # fewer (or more) heads of the same shape: grouped-query workloads keep their
        # group size
        g = w["heads"] // w.get("kv_heads", w["heads"])
        if heads % g:
            raise SystemExit("--heads must be a multiple of the group size %d" % g)
        w["heads"] = heads
        if "kv_heads" in w:
            w["kv_heads"] = heads // g
        w["name"] = "%s-h%d" % (name, heads)
    return w


def workload_key(w):
    """The shape a traffic capture belongs to (heads excluded: heads are independent
    problems run one after another, so DRAM traffic scales with their number)."""
    return "L%d-g%d-D%d-P%d-b%d-%s%s" % (
        w["seq_len"], w["heads"] // w.get("kv_heads", w["heads"]), w["head_dim"], w["P"],
        w["block"], w["layout"], "" if w["causal"] else "-noncausal")


def pairs_of(L, causal):
    return L * (L + 1) // 2 if causal else L * L


def flops_of(w, batch_heads=None):
    bh = batch_heads if batch_heads is not None else w["batch"] * w["heads"]
    pr = bh * pairs_of(w["seq_len"], w["causal"])
    D = w["head_dim"]
    return 4 * D * pr, 10 * D * pr


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def config_of(w):
    L, H, D = w["seq_len"], w["heads"], w["head_dim"]
    tensor_mib = w["batch"] * L * H * D * 2 / 2 ** 20
    what = "one blockwise transformer layer forward" if "d_ff" in w else "causal fwd+bwd"
    return {"workload": "%s %s, %s layout" % (w["name"], what, w["layout"]),
            "batch": w["batch"], "heads": H, "kv_heads": w.get("kv_heads", H),
            "head_dim": D, "seq_len": L, "P": w["P"],
            "block": w["block"], "layout": w["layout"], "causal": w["causal"],
            "l2": "inputs larger than L2 (%.0f MiB per bf16 tensor, L2 129 MB)" % tensor_mib,
            "flops_per_step": sum(flops_of(w))}


# ---------------------------------------------------------------- clocks -----------
class ClockSampler:
    """nvidia-smi sampling every 200 ms while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid):
        self.proc = None
        self.uuid = uuid

    def start(self):
        try:
            cmd = ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                   "-lms", "200"]
            if self.uuid:
                cmd += ["-i", self.uuid]
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in out.splitlines():
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for nm, val in zip(names, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- distributed ------
def dist_init(args):
    import torch
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws <= 1:
        return 0, 1, 0
    import torch.distributed as dist
    rank = int(os.environ["RANK"])
    local = int(os.environ.get("LOCAL_RANK", rank))
    torch.cuda.set_device(local)
    dist.init_process_group("nccl")
    return rank, ws, local


def dist_max(x, world):
    """Max of x over the ranks (the slowest rank's time sets the job's time)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(world, flops_per_rank_step, steps, max_ms):
    """Whole-job TFLOP/s: the useful FLOPs every rank did over the slowest rank's time
    (every rank runs the same workload on its own GPU: weak scaling)."""
    return world * flops_per_rank_step * steps / (max_ms * 1e-3) / 1e12


def dist_barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------- CPU oracle -------
def oracle_sample(w, tokens, reps=1):
    """fp64 oracle fwd+bwd on one head of `tokens` tokens of the workload's input
    distribution.  Returns (seconds per rep, useful TFLOP per rep, cores)."""
    import numpy as np
    import oracle
    from exact_blockwise_ring_gb300.synthetic import make_inputs, to_f64
    q, k, v, do = to_f64(*make_inputs(1, tokens, 1, w["head_dim"], seed=w["seed"]))
    cores = len(os.sched_getaffinity(0))
    t = 0.0
    for _ in range(reps):
        t0 = time.perf_counter()
        oracle.attention_fwd(q, k, v, w["causal"])
        oracle.attention_bwd(q, k, v, do, w["causal"])
        t += time.perf_counter() - t0
    pr = pairs_of(tokens, w["causal"])
    return t / reps, 14 * w["head_dim"] * pr / 1e12, cores


CPU_SAMPLE_TOKENS = 32768       # one full head of the 32k workload: ~10-15 s on 16 Grace cores
REF_STEP_TOKENS = 8192          # one head per reference step


def cpu_baseline(w):
    t, tf, cores = oracle_sample(w, CPU_SAMPLE_TOKENS)
    return {"value": tf / t, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": "fp64 oracle fwd+bwd, 1 head x %d tokens (causal) of the workload's "
                      "input distribution, %.1f s; useful-FLOP convention of the GPU line"
                      % (CPU_SAMPLE_TOKENS, t),
            "one_thread": oracle_one_thread()}


def oracle_one_thread():
    """The oracle with its BLAS on one thread (a child process with the thread-count
    variables set before NumPy loads), on one head of the tiny and the 8k workloads."""
    code = ("import json, sys, bench; w = bench.workload(sys.argv[1], None); "
            "t, tf, c = bench.oracle_sample(w, w['seq_len']); print(json.dumps([t, tf]))")
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS",
              "BLIS_NUM_THREADS"):
        env[k] = "1"
    res = {}
    for name in ("tiny", "8k"):
        try:
            r = subprocess.run([sys.executable, "-c", code, name], cwd=ROOT, env=env,
                               capture_output=True, text=True, timeout=300)
            t, tf = json.loads(r.stdout.strip().splitlines()[-1])
            res[name] = {"tflops": tf / t, "seconds": round(t, 3)}
        except Exception as e:          # a report field: never fails the bench
            res[name] = {"error": str(e)[:120]}
    return res


def source_hash(*names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "exact_blockwise_ring_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_for(kernel, src_files, w):
    """DRAM bytes per launch of `kernel` on workload `w`, from the committed ncu summary
    (profiles/ncu_traffic.txt): a capture of the same shape (workload_key) with the same
    kernel source, taken with H_c heads, scaled by H / H_c (heads are independent and run
    one after another).  Returns (bytes, note) or (None, reason)."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(p):
        return None, "no capture"
    key, heads, h = workload_key(w), w["batch"] * w["heads"], source_hash(*src_files)
    stale = False
    with open(p) as f:
        for ln in f:
            fl = ln.split()
            if len(fl) < 7 or ln.startswith("#") or fl[0] != kernel or fl[5] != key:
                continue
            if fl[4] != h:
                stale = True
                continue
            cap_heads = int(fl[6])
            scaled = int(fl[1]) * heads // cap_heads
            if cap_heads == heads:
                return scaled, "captured on this workload"
            return scaled, "scaled x%g from a capture with %d of the %d heads" % (
                heads / cap_heads, cap_heads, heads)
    return None, ("kernel source changed since the capture" if stale
                  else "no capture of this workload")


def hbm_line(nbytes, ms, peak_gbs):
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"bytes": int(nbytes), "ms": round(ms, 4), "achieved_gbs": round(gbs, 1),
            "frac": round(gbs / peak_gbs, 4)}


def time_merge(era, B, L, H, D, dev, stream, peak_gbs, n_parts=4, reps=5):
    """ra_merge on n_parts fp32 partials [n, B, L, H, D] (inputs larger than L2), CUDA
    events on the launching stream; algorithmic bytes = partials and their lse read once,
    bf16 output and lse written once."""
    import torch
    g = torch.Generator(device=dev)
    g.manual_seed(4242)
    o_parts = torch.randn((n_parts, B, L, H, D), generator=g, device=dev, dtype=torch.float32)
    lse_parts = torch.randn((n_parts, B, H, L), generator=g, device=dev, dtype=torch.float32)
    for _ in range(2):
        era.ra_merge(o_parts, lse_parts, stream=stream)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        era.ra_merge(o_parts, lse_parts, stream=stream)
    e1.record(stream)
    torch.cuda.synchronize()
    rows = B * L * H
    nbytes = n_parts * rows * (4 * D + 4) + rows * (2 * D + 4)
    line = hbm_line(nbytes, e0.elapsed_time(e1) / reps, peak_gbs)
    line["n_parts"] = n_parts
    return line


# ---------------------------------------------------------------- our arm ----------
def run_ours(args, w, rank, world, local):
    import torch
    import exact_blockwise_ring_gb300 as era
    from exact_blockwise_ring_gb300.synthetic import make_inputs

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    B, L, H, D, P, blk = (w["batch"], w["seq_len"], w["heads"], w["head_dim"], w["P"],
                          w["block"])
    layout, causal = w["layout"], w["causal"]
    q, k, v, do = make_inputs(B, L, H, D, w["seed"] + 7919 * rank, device=dev,
                              kv_heads=w.get("kv_heads"))
    out = torch.empty_like(q)
    lse = torch.empty((B, H, L), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = era.Workspace(dev)
    stream = torch.cuda.current_stream(dev)

    def step(evs=None):
        if evs is not None:
            evs[0].record(stream)
        era.ra_fwd(q, k, v, P, blk, layout, causal, out=out, lse=lse, workspace=ws)
        era.ra_bwd_stages(q, k, v, out, lse, do, dq, dk, dv, P, blk, layout, causal,
                          workspace=ws,
                          between=(lambda i: evs[i + 1].record(stream)) if evs else None)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    ws.check()
    dist_barrier(world)

    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(K)]
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        uuid = None
    clocks = ClockSampler(uuid)
    clocks.start()
    time.sleep(0.3)
    torch.cuda.synchronize()
    dist_barrier(world)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for s in range(K):
        step(evs[s])
    t1.record(stream)
    torch.cuda.synchronize()
    dist_barrier(world)
    clk = clocks.stop()
    ws.check()
    total_ms = t0.elapsed_time(t1)
    total_ms_max = dist_max(total_ms, world)
    stage = [[e[i].elapsed_time(e[i + 1]) for e in evs] for i in range(4)]
    fwd_ms, pre_ms, main_ms, fin_ms = (statistics.mean(x) for x in stage)

    f_fwd, f_bwd = flops_of(w)
    step_flops = f_fwd + f_bwd
    ms_per_step = total_ms_max / K
    value = job_rate(world, step_flops, K, total_ms_max)
    pk, pk_kind = peaks()
    peak_tf = pk.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    peak_sus = pk.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])

    # dominant kernel and its roofline (tensor-bound contraction)
    hdrs = ("ra_internal.h", "ra_ptx.cuh", "ra_rows.cuh", "ra_exp2.cuh")   # shared headers
    if main_ms >= fwd_ms:
        dom, dom_ms, dom_flops, files = "ra_bwd_kernel", main_ms, f_bwd, ("ra_bwd.cu",) + hdrs
    else:
        dom, dom_ms, dom_flops, files = "ra_fwd_kernel", fwd_ms, f_fwd, ("ra_fwd.cu",) + hdrs
    achieved = dom_flops / (dom_ms * 1e-3) / 1e12
    # the burst peak for a step shorter than a second, the sustained one (a seconds-long
    # loop under the power cap) for longer steps
    if ms_per_step < 1000.0:
        peak_use, peak_name = peak_tf, "bf16_tflops (burst: timed step under 1 s)"
    else:
        peak_use, peak_name = peak_sus, "bf16_tflops_sustained (timed step of 1 s or more)"
    traffic, traffic_note = traffic_for(dom, files, w)
    roofline = {"bound": "tensor", "kernel": dom, "achieved": round(achieved, 1),
                "peak": peak_use, "unit": "TFLOP/s", "frac": round(achieved / peak_use, 4),
                "peak_kind": "%s of %s" % (peak_name, pk_kind),
                "frac_of_burst": round(achieved / peak_tf, 4),
                "frac_of_sustained": round(achieved / peak_sus, 4),
                "flops_per_launch": dom_flops, "ms_per_launch": round(dom_ms, 3),
                "traffic": traffic, "traffic_note": traffic_note}

    # end to end through the public API with host buffers: every step copies its inputs
    # from pinned host memory, makes the two calls, and copies every result back.  Steps
    # alternate between two sets of device buffers, so that step s+1's inputs go up (and
    # step s-1's results come down) on copy streams while step s computes.
    e2e = None
    if not args.no_e2e:
        # host side: one pinned allocation holding the inputs and one set of results (every
        # step's results land there in turn).  Separate pinned buffers per tensor and per
        # set stalled the copies for tens of ms now and then on a virtualised host.
        ins, outs = [q, k, v, do], [out, lse, dq, dk, dv]
        blob = torch.empty(sum(t.numel() * t.element_size() for t in ins + outs),
                           dtype=torch.uint8, pin_memory=True)
        views, off = [], 0
        for t in ins + outs:
            nb = t.numel() * t.element_size()
            views.append(blob[off:off + nb].view(t.dtype).view(t.shape))
            off += nb
        hin, hout_shared = views[:4], views[4:]
        for h_, t in zip(hin, ins):
            h_.copy_(t.cpu())
        h2d = sum(t.numel() * t.element_size() for t in hin)
        sets = []
        for bset in range(2):
            din = ins if bset == 0 else [torch.empty_like(t) for t in ins]
            dout = outs if bset == 0 else [torch.empty_like(t) for t in outs]
            ev = {n: torch.cuda.Event() for n in ("up", "done", "down")}
            sets.append((din, dout, hout_shared, ev))
        d2h = sum(t.numel() * t.element_size() for t in sets[0][2])
        s_up, s_down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

        def e2e_step(sidx):
            din, dout, hout, ev = sets[sidx % 2]
            with torch.cuda.stream(s_up):
                if sidx >= 2:
                    s_up.wait_event(ev["done"])          # inputs of step s-2 consumed
                for d_, h_ in zip(din, hin):
                    d_.copy_(h_, non_blocking=True)
                ev["up"].record(s_up)
            stream.wait_event(ev["up"])
            if sidx >= 2:
                stream.wait_event(ev["down"])            # results of step s-2 copied out
            qq, kk, vv, dd = din
            oo, ll, gq, gk, gv = dout
            # one workspace: the calls run in order on the compute stream
            era.ra_fwd(qq, kk, vv, P, blk, layout, causal, out=oo, lse=ll, workspace=ws)
            era.ra_bwd_stages(qq, kk, vv, oo, ll, dd, gq, gk, gv, P, blk, layout, causal,
                              workspace=ws)
            ev["done"].record(stream)
            with torch.cuda.stream(s_down):
                s_down.wait_event(ev["done"])
                for h_, d_ in zip(hout, dout):
                    h_.copy_(d_, non_blocking=True)
                ev["down"].record(s_down)

        for sidx in range(2):
            e2e_step(sidx)
        torch.cuda.synchronize()
        # three timed windows of Ke steps each (Ke = K, or fewer when K steps take over
        # 10 s, but two at least when K allows, so that a window holds a step whose copies
        # run under its neighbour's compute; about 15 s of steps at most); the line reports
        # the median window and lists all three (on a virtualised host a single host-memory
        # copy can stall for ~100 ms, which one window cannot absorb)
        Ke = K if ms_per_step * K <= 10000.0 else max(min(K, 2), int(15000.0 // ms_per_step))
        windows = []
        for _ in range(3):
            dist_barrier(world)
            a0 = torch.cuda.Event(enable_timing=True)
            a1 = torch.cuda.Event(enable_timing=True)
            a0.record(s_up)
            for sidx in range(Ke):
                e2e_step(sidx)
            s_down.wait_stream(stream)
            a1.record(s_down)
            torch.cuda.synchronize()
            windows.append(dist_max(a0.elapsed_time(a1), world))
        ws.check()
        e_ms = sorted(windows)[1]
        # this machine's host link, after the timed region: one step's copies each way
        # alone, same pinned buffers and streams (explains an e2e gap to the device rate)
        link = {}
        din0, dout0, hout0, _ = sets[0]
        for name, s_, pairs_, nb in (("h2d_gbs", s_up, list(zip(din0, hin)), h2d),
                                     ("d2h_gbs", s_down, list(zip(hout0, dout0)), d2h)):
            c0 = torch.cuda.Event(enable_timing=True)
            c1 = torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            with torch.cuda.stream(s_):
                c0.record(s_)
                for dst, src in pairs_:
                    dst.copy_(src, non_blocking=True)
                c1.record(s_)
            torch.cuda.synchronize()
            link[name] = round(nb / (c0.elapsed_time(c1) * 1e-3) / 1e9, 1)
        e2e = {"value": round(job_rate(world, step_flops, Ke, e_ms), 2),
               "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": round(e_ms / Ke, 3), "steps_per_window": Ke,
               "windows": [round(job_rate(world, step_flops, Ke, x), 2) for x in windows],
               "host_link": link,
               "copies": "each step's H2D and D2H overlap the neighbouring steps' compute "
                         "(two buffer sets, two copy streams); value = the median of three "
                         "timed windows of steps_per_window steps (all three in windows)"}

    # the bandwidth-bound kernels against the measured HBM copy rate: the backward's
    # preprocess and finalize (timed inside the steps above) and the partial merge (timed
    # here, after the steps, on 4 fp32 partials of the workload's shape)
    hbm = pk.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    rows = B * L * H
    pre_bytes = rows * (2 * D + out.element_size() * D + 4 + 8 + 4 * D)
    fin_bytes = rows * D * (4 + 2)
    hbm_kernels = {
        "peak_gbs": hbm, "peak_kind": "hbm_gbs of %s" % pk_kind,
        "bwd_pre_kernel": hbm_line(pre_bytes, pre_ms, hbm),
        "dq_convert_kernel": hbm_line(fin_bytes, fin_ms, hbm),
    }
    if not args.no_merge:
        hbm_kernels["merge_kernel"] = time_merge(era, B, L, H, D, dev, stream, hbm)

    # the secondary ceiling: one exp per unmasked pair in the forward and one in the
    # backward, against the measured MUFU rate (32 exp2 per clock per SM on this part)
    # at the median SM clock seen
    pairs = B * H * pairs_of(L, causal)
    mhz = (clk or {}).get("sm_mhz") or 2070.0
    ceil = 32.0 * 152 * mhz * 1e6
    mufu = {"exp_per_s_fwd": round(pairs / (fwd_ms * 1e-3), 0),
            "exp_per_s_bwd": round(pairs / (main_ms * 1e-3), 0),
            "ceiling_exp_per_s": round(ceil, 0),
            "frac_fwd": round(pairs / (fwd_ms * 1e-3) / ceil, 4),
            "frac_bwd": round(pairs / (main_ms * 1e-3) / ceil, 4),
            "ceiling_kind": "32 exp2/clk/SM (microbenchmark on this part) x 152 SMs x median SM clock"}

    # per-shard causal work: the host model for every layout (equal to the device counters,
    # which the tests check bit for bit) and the device counters of this layout, from one
    # forward outside the timed region
    balance = {}
    for lay in ("contiguous", "striped", "zigzag"):
        try:
            m = era.ra_shard_work_model(L, P, blk, lay, causal)
        except Exception:            # e.g. zigzag needs L divisible by 2 * P * block
            continue
        balance[lay] = {u: round(max(m[u]) / (sum(m[u]) / P), 5) for u in ("tiles", "pairs", "visits")}
    _, _, sw = era.ra_fwd(q, k, v, P, blk, layout, causal, shard_work=True, workspace=ws)
    swc = sw.cpu().double()
    balance["device_" + layout] = {u: round(float(swc[n].max() / swc[n].mean()), 5)
                                   for n, u in enumerate(("tiles", "pairs", "visits"))}
    balance["unit"] = "max / mean over the P shards"

    # the step's time scaled to the maximum SM clock (time x median clock / max clock):
    # compares layouts or runs whose clocks differed (the power cap), assuming the
    # tensor-bound kernels scale with the SM clock
    clock_norm = None
    if clk and clk.get("sm_mhz") and clk.get("sm_max_mhz"):
        f = clk["sm_mhz"] / clk["sm_max_mhz"]
        clock_norm = {"ms_per_step": round(ms_per_step * f, 3),
                      "fwd_ms": round(fwd_ms * f, 3), "bwd_main_ms": round(main_ms * f, 3),
                      "value": round(value / f, 2),
                      "rule": "time x median SM MHz / max SM MHz over the timed region"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = cpu_baseline(w)
    if rank == 0:
        line = {"metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
                "steps": K, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 3),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "bf16", "data": "synthetic",
                "pct_of_bf16_peak": round(100.0 * value / world / peak_tf, 2),
                "pct_of_bf16_peak_sustained": round(100.0 * value / world / peak_sus, 2),
                "config": config_of(w),
                "stage_ms": {"fwd": round(fwd_ms, 3), "bwd_preprocess": round(pre_ms, 3),
                             "bwd_main": round(main_ms, 3), "bwd_finalize": round(fin_ms, 3)},
                "roofline": roofline, "hbm_kernels": hbm_kernels, "shard_balance": balance,
                "cpu_baseline": cpu,
                "e2e": e2e,
                "tflops_12d": round(value * 12.0 / 14.0, 2),
                "mufu": mufu, "gpu_launches": 4 * K, "clocks": clk,
                "at_max_clock": clock_norm}
        print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- BPT layer --------
BPT_METRIC = "blockwise transformer layer forward TFLOP/s (projections, causal ring attention, FFN)"
BPT_TRAIN_METRIC = "blockwise transformer layer forward + backward TFLOP/s (useful FLOPs)"


def bpt_flops(w, train=False):
    """Useful FLOPs of one layer forward: Q, K, V, O projections 4 * 2 L d^2, feed-forward
    2 * 2 L d d_ff, causal attention 4 D per unmasked pair per head.  With the backward:
    twice the dense forward again (input and weight gradients) and 10 D per pair for the
    attention (its recompute included); the dense recompute of the BPT backward is not
    counted."""
    rows = w["batch"] * w["seq_len"]
    d = w["heads"] * w["head_dim"]
    pairs = w["batch"] * w["heads"] * pairs_of(w["seq_len"], w["causal"])
    dense = 8 * rows * d * d + 4 * rows * d * w["d_ff"]
    if train:
        return 3 * dense + 14 * w["head_dim"] * pairs
    return dense + 4 * w["head_dim"] * pairs


def bpt_oracle_sample(w, tokens=1024, d=1024, d_ff=4096, train=False):
    """fp64 oracle layer forward (and backward) on a bounded sample: 1 x `tokens` x d,
    d_ff, d / 128 heads."""
    import numpy as np
    import oracle
    from exact_blockwise_ring_gb300.synthetic import make_bpt_weights, to_f64
    rng = np.random.default_rng(w["seed"])
    x = rng.standard_normal((1, tokens, d))
    wt = {k: to_f64(v)[0] for k, v in make_bpt_weights(d, d_ff, w["seed"]).items()}
    t0 = time.perf_counter()
    oracle.bpt_layer_fwd(x, wt, d // 128, w["causal"])
    if train:
        oracle.bpt_layer_bwd(x, wt, d // 128, w["causal"], rng.standard_normal(x.shape))
    t = time.perf_counter() - t0
    sw = dict(w, batch=1, seq_len=tokens, heads=d // 128, head_dim=128, d_ff=d_ff)
    return t, bpt_flops(sw, train) / 1e12, len(os.sched_getaffinity(0))


def run_bpt(args, w, rank, world, local):
    import torch
    import exact_blockwise_ring_gb300 as era
    from exact_blockwise_ring_gb300.synthetic import make_bpt_weights, make_inputs

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    B, L, H, D, P, blk = (w["batch"], w["seq_len"], w["heads"], w["head_dim"], w["P"],
                          w["block"])
    d, d_ff, br = H * D, w["d_ff"], w["block_rows"]
    x = make_inputs(B, L, 1, d, w["seed"] + 7919 * rank, device=dev, with_dout=False)[0]
    x = x.view(B, L, d)
    wt = make_bpt_weights(d, d_ff, w["seed"] + 1, device=dev)
    out = torch.empty((B, L, d), dtype=torch.bfloat16, device=dev)
    ws = era.Workspace(dev)
    stream = torch.cuda.current_stream(dev)
    train = args.train
    dout = make_inputs(B, L, 1, d, w["seed"] + 2, device=dev, with_dout=False)[0].view(B, L, d)

    def step():
        era.ra_bpt_fwd(x, wt, H, P, blk, w["layout"], w["causal"], block_rows=br, workspace=ws,
                       out=out, train=train)
        if train:
            era.ra_bpt_bwd(x, wt, dout, H, P, blk, w["layout"], w["causal"], block_rows=br,
                           workspace=ws)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    ws.check()
    dist_barrier(world)
    K = args.steps
    clocks = ClockSampler(None)
    clocks.start()
    time.sleep(0.3)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(K):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    dist_barrier(world)
    clk = clocks.stop()
    ws.check()
    total_ms = dist_max(t0.elapsed_time(t1), world)
    flops = bpt_flops(w, train)
    value = job_rate(world, flops, K, total_ms)

    # dominant kernel: the feed-forward GEMM of one block (rows br, d -> d_ff, GELU), timed
    # alone with CUDA events on the launching stream
    pk, pk_kind = peaks()
    peak_tf = pk.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    h1 = torch.randn((br, d), device=dev).to(torch.bfloat16)
    f = torch.empty((br, d_ff), dtype=torch.bfloat16, device=dev)
    for _ in range(3):
        era.ra_linear(h1, wt["w1"], wt["b1"], "bias_gelu", workspace=ws, out=f)
    g0 = torch.cuda.Event(enable_timing=True)
    g1 = torch.cuda.Event(enable_timing=True)
    reps = 10
    g0.record(stream)
    for _ in range(reps):
        era.ra_linear(h1, wt["w1"], wt["b1"], "bias_gelu", workspace=ws, out=f)
    g1.record(stream)
    torch.cuda.synchronize()
    ws.check()
    g_ms = g0.elapsed_time(g1) / reps
    g_tf = 2.0 * br * d * d_ff / (g_ms * 1e-3) / 1e12
    roofline = {"bound": "tensor", "kernel": "gemm_kernel (FFN W1 + bias + GELU)",
                "achieved": round(g_tf, 1), "peak": peak_tf, "unit": "TFLOP/s",
                "frac": round(g_tf / peak_tf, 4), "peak_kind": "bf16_tflops (burst) of %s" % pk_kind,
                "traffic": None, "shape": [br, d_ff, d]}

    e2e = None
    if not args.no_e2e:
        hx = x.cpu().pin_memory()
        ho = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)

        def e2e_step():
            x.copy_(hx, non_blocking=True)
            step()
            ho.copy_(out, non_blocking=True)

        e2e_step()
        torch.cuda.synchronize()
        a0 = torch.cuda.Event(enable_timing=True)
        a1 = torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for _ in range(K):
            e2e_step()
        a1.record(stream)
        torch.cuda.synchronize()
        e_ms = dist_max(a0.elapsed_time(a1), world)
        e2e = {"value": round(job_rate(world, flops, K, e_ms), 2), "unit": "TFLOP/s",
               "h2d_bytes_per_step": hx.numel() * 2, "d2h_bytes_per_step": ho.numel() * 2,
               "ms_per_step": round(e_ms / K, 3)}
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        t, tf, cores = bpt_oracle_sample(w, train=train)
        cpu = {"value": tf / t, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
               "sample": "fp64 oracle layer %s, 1 x 1024 tokens, d 1024, d_ff 4096, 8 heads, "
                         "causal, %.1f s; useful-FLOP convention of the GPU line"
                         % ("forward + backward" if train else "forward", t)}
    n_blocks = -(-(B * L) // br)
    # per step: 3 projection GEMMs, the attention (1 kernel, + merge when split), and per
    # block 3 GEMMs and 2 LayerNorms; the backward: per block 9 GEMMs (3 recomputing the
    # forward), 1 LayerNorm, 2 LayerNorm backward, 3 column sums; then the attention's 3
    # kernels, 6 GEMMs and 3 column sums for the projections, and the dx conversion
    launches = 3 + 1 + 5 * n_blocks + ((15 * n_blocks + 13) if train else 0)
    if rank == 0:
        line = {"metric": BPT_TRAIN_METRIC if train else BPT_METRIC, "value": round(value, 2),
                "unit": "TFLOP/s",
                "n_gpus": world, "steps": K, "warmup": args.warmup,
                "ms_per_step": round(total_ms / K, 3), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "pct_of_bf16_peak": round(100.0 * value / world / peak_tf, 2),
                "config": {"workload": "%s: one blockwise transformer layer %s, %s layout"
                           % (w["name"], "forward + backward" if train else "forward",
                              w["layout"]), "batch": B, "seq_len": L, "d_model": d,
                           "heads": H, "d_ff": d_ff, "P": P, "block": blk, "block_rows": br,
                           "causal": w["causal"], "flops_per_step": flops,
                           "l2": "inputs larger than L2 (x %.0f MiB, weights %.0f MiB)"
                           % (x.numel() * 2 / 2 ** 20,
                              sum(t.numel() * t.element_size() for t in wt.values()) / 2 ** 20)},
                "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": launches * K, "clocks": clk}
        print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- reference arm ----
def run_reference(args, w, rank, world):
    if rank != 0:
        return
    bpt = "d_ff" in w
    t_steps = []
    for s in range(args.warmup + args.steps):
        t, tf, cores = bpt_oracle_sample(w) if bpt else oracle_sample(w, REF_STEP_TOKENS)
        if s >= args.warmup:
            t_steps.append(t)
    total = sum(t_steps)
    value = tf * len(t_steps) / total
    if bpt:
        sample = ("fp64 oracle layer forward per step: 1 x 1024 tokens, d 1024, d_ff 4096, "
                  "8 heads, causal; useful-FLOP convention of the GPU line")
    else:
        sample = ("fp64 oracle fwd+bwd per step: 1 head x %d tokens (causal) of the workload's "
                  "input distribution; useful-FLOP convention of the GPU line" % REF_STEP_TOKENS)
    line = {"impl": "reference", "metric": BPT_METRIC if bpt else METRIC, "value": round(value, 5),
            "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * total / len(t_steps), 1), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(w),
            "cpu_baseline": {"value": round(value, 5), "unit": "TFLOP/s", "cores": cores,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 5), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)

def main():
    args = parse_args()
    w = workload(args.workload, args.layout, args.heads)
    if args.impl == "reference":
        # the oracle runs on rank 0's host cores; other ranks exit without work
        run_reference(args, w, int(os.environ.get("RANK", "0")),
                      int(os.environ.get("WORLD_SIZE", "1")))
        return
    rank, world, local = dist_init(args)
    try:
        if "d_ff" in w:
            run_bpt(args, w, rank, world, local)
        else:
            run_ours(args, w, rank, world, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
