"""Decode-step weight-stream benchmark.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

One step = one whole decode step (bws_decode_step_stream) of the 27B-shape
dense stack: 64 NVFP4 layers (17.82 GB) plus the FP8 248320x5120 output layer,
19.097 GB of weights read per step, for 1 token (the headline) and, as a
second line of the same JSON object, for 8 tokens (speculative verify). The
MoE stack (Ling-shape, MXFP4, N=1 and N=4) is measured too unless --no-moe.

The metric is the decode-step weight bandwidth: algorithmic weight bytes per
step / step time, in GB/s (1 GB = 1e9 B). Inputs are synthetic (seeded
N(0, 0.02) weights quantized on the GPU, N(0, 1) BF16 activations). The
weights of one step (19 GB) are far larger than L2, so no flush is needed
between steps.

Under torchrun (--gpus N > 1) each rank runs an independent replica of the
step on its own GPU (the path has no exchange step); value is the sum of all
ranks' bytes over the slowest rank's time.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode-step weight GB/s"
UNIT = "GB/s"


# ---- multi-process plumbing (testable on CPU) -------------------------------

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def aggregate(bytes_per_rank, seconds_per_rank):
    """Whole-job throughput: all ranks' bytes over the slowest rank's time."""
    t = max(seconds_per_rank)
    return sum(bytes_per_rank) / t if t > 0 else 0.0, t


def all_gather_floats(vals, world):
    import torch
    import torch.distributed as dist
    if world == 1:
        return [list(vals)]
    t = torch.tensor(vals, dtype=torch.float64)
    if dist.get_backend() == "nccl":
        t = t.cuda()
    out = [torch.zeros_like(t) for _ in range(world)]
    dist.all_gather(out, t)
    return [o.cpu().tolist() for o in out]


# ---- clocks -----------------------------------------------------------------

CLOCK_QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
               "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
               "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    """Samples nvidia-smi every 100 ms while running (in a background process)."""

    def __init__(self, gpu_index=0):
        self.gpu_index = gpu_index
        self.lines = []
        self.proc = None
        self.thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_index}", f"--query-gpu={CLOCK_QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=5)

    def summary(self):
        return parse_clock_lines(self.lines)


def parse_clock_lines(lines):
    sm, mx, reasons = [], [], set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for ln in lines:
        f = [x.strip() for x in ln.split(",")]
        if len(f) < 9:
            continue
        try:
            sm.append(float(f[1]))
            mx.append(float(f[2]))
        except ValueError:
            continue
        for n, v in zip(names, f[5:9]):
            if v.lower().startswith("active"):
                reasons.add(n)
    if not sm:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
    return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons), "samples": len(sm)}


# ---- CPU baseline (the oracle) ------------------------------------------------

_ONE_THREAD = {k: "1" for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}


def _oracle_worker(path, barrier, out):
    """One host core (numpy with one BLAS thread): loads a matrix, waits for
    the others, then times the oracle's NVFP4 product on it (N = 1)."""
    os.environ.update(_ONE_THREAD)
    import numpy as np
    from oracle import products as P
    d = np.load(path)
    codes, scales, ts = d["c"], d["s"], np.float32(d["t"])
    x = np.random.default_rng(0).standard_normal((1, codes.shape[1] * 2)).astype(np.float32)
    barrier.wait(timeout=300)
    t0 = time.perf_counter()
    P.nvfp4_gemv(codes, scales, ts, x)
    t1 = time.perf_counter()
    out.put((codes.nbytes + scales.nbytes, t0, t1))


def cpu_oracle_rate(sample, procs):
    """The oracle's NVFP4 product timed on `procs` host cores at once: one
    spawned process per core, one BLAS thread each, every process running the
    product over the same sample matrix (codes, scales, s_t). Returns
    algorithmic bytes per second of wall time (first start to last end)."""
    import multiprocessing as mp
    import tempfile
    import numpy as np
    codes, scales, ts = sample
    ctx = mp.get_context("spawn")
    with tempfile.TemporaryDirectory() as tmp:
        path = os.path.join(tmp, "m.npz")
        np.savez(path, c=codes, s=scales, t=np.float32(ts))
        barrier, out = ctx.Barrier(procs), ctx.Queue()
        ps = [ctx.Process(target=_oracle_worker, args=(path, barrier, out)) for _ in range(procs)]
        for p in ps:
            p.start()
        try:
            res = [out.get(timeout=600) for _ in ps]
        finally:
            for p in ps:
                p.join(timeout=30)
                if p.is_alive():
                    p.kill()
    nbytes = sum(r[0] for r in res)
    wall = max(r[2] for r in res) - min(r[1] for r in res)
    return nbytes / wall / 1e9


def cpu_baseline(sample):
    """The oracle on the host cores: all cores at once (the reported value)
    and one core, with the core counts."""
    cores = os.cpu_count() or 1
    all_cores = cpu_oracle_rate(sample, cores)
    one = cpu_oracle_rate(sample, 1)
    rows = sample[0].shape[0]
    cols = sample[0].shape[1] * 2
    desc = (f"oracle NVFP4 GEMV (FP64 products, numpy, one BLAS thread per process) over one of the step's "
            f"matrices ({rows}x{cols}, N=1), once per core")
    return {"value": round(all_cores, 4), "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc,
            "one_core": {"value": round(one, 4), "unit": UNIT, "cores": 1}}


def host_copy(stack, rows=8192):
    """Host copy (codes, scales, s_t) of the first `rows` rows of the stack's
    first MLP gate matrix: a bounded sample of the step's weights."""
    for L in stack.layers_py:
        m = L.get("gate")
        if m is not None and m.fmt == 1:
            return m.codes[:rows].cpu().numpy(), m.scales[:rows].cpu().numpy(), float(m.scale32.item())
    raise RuntimeError("no NVFP4 gate matrix in the stack")


# ---- the GPU arm ------------------------------------------------------------------

def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def time_steps(fn, steps, warmup, stream):
    import torch
    for _ in range(warmup):
        fn()
    stream.synchronize()
    s = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    s.record(stream)
    for _ in range(steps):
        fn()
    e.record(stream)
    e.synchronize()
    return s.elapsed_time(e) / 1e3 / steps


# DRAM read + write bytes per algorithmic byte of the NVFP4 product kernel,
# by token count, from ncu's dram__bytes_read.sum + dram__bytes_write.sum
# over two launches of each of the step's five product shapes (46336x5120,
# 14336x5120, 34816x5120, 5120x17408, 5120x6144), weighted by the step's
# launches per shape. Taken on the current kernel; to be dropped when the
# kernel changes.
TRAFFIC_PER_BYTE = {1: 1.0339, 8: 1.0366}
TRAFFIC_BASIS = ("ncu dram__bytes_read.sum + dram__bytes_write.sum of the product kernel on the step's five shapes "
                 "(two launches each), weighted by launches per shape: {r} x algorithmic bytes at {n} token(s)")


def product_groups(stack):
    """The step's NVFP4 products by type, one entry per launch of the step:
    (name, [matrix lists]). The step runs a layer's mixer-input matrices
    (query, key and value of a full-attention layer) as one product and its
    gate and up matrices as one SwiGLU product; each list is one such launch."""
    g = {"mixer-in": [], "mixer-out": [], "gate/up": [], "down": []}
    for L in stack.layers_py:
        if L.get("mixer_in"):
            g["mixer-in"].append(list(L["mixer_in"]))
        if "mixer_out" in L:
            g["mixer-out"].append([L["mixer_out"]])
        if "gate" in L:
            g["gate/up"].append([L["gate"], L["up"]])
        if "down" in L:
            g["down"].append([L["down"]])
    return [(k, [ms for ms in v if all(m.fmt == 1 for m in ms)]) for k, v in g.items()]


def launch_matrix(ms):
    """One launch's matrices as one NVFP4 matrix: rows concatenated (codes
    and block scales), so that a single standalone product streams the same
    bytes in the same launch as the step's product over those matrices."""
    import torch
    from bit_weight_streaming_gb300.stack import QMatrix
    if len(ms) == 1:
        return ms[0]
    return QMatrix(ms[0].fmt, torch.cat([m.codes for m in ms]), torch.cat([m.scales for m in ms]), ms[0].scale32)


def time_dominant_kernel(stack, stream, reps=3):
    """The NVFP4 product kernel as it runs inside the step: each type of the
    step's products (mixer inputs, mixer outputs, gate and up, down) is
    captured as one CUDA graph of back-to-back launches, one per product of
    that type in the step (bws_nvfp4_gemv_prepared, chained with
    programmatic dependent launch as in the step; every launch reads cold
    weights, the whole set being far larger than L2), on activations
    prepared once per input width. CUDA events on the launching stream
    around `reps` replays. Returns {type: (launches, bytes, seconds per
    replay)}."""
    import torch
    import bit_weight_streaming_gb300 as bws
    dev = stack.device
    out = {}
    for name, launches in product_groups(stack):
        if not launches:
            continue
        mats = [launch_matrix(ms) for ms in launches]
        d_in = mats[0].d_in
        assert all(m.d_in == d_in for m in mats)
        ws = bws.Workspace(dev)
        ys = {m.d_out: torch.empty((stack.N, m.d_out), dtype=torch.bfloat16, device=dev) for m in mats}
        x = torch.randn((stack.N, d_in), device=dev).to(torch.bfloat16)
        with torch.cuda.stream(stream):
            bws.nvfp4_prepare(x, max(m.d_out for m in mats), ws)
            for m in mats[:4]:   # warm-up outside the graph (tensor-map encoder, attributes)
                bws.nvfp4_gemv_prepared(m.codes, m.scales, m.scale32, stack.N, d_in, ws, y=ys[m.d_out])
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for m in mats:
                bws.nvfp4_gemv_prepared(m.codes, m.scales, m.scale32, stack.N, d_in, ws, y=ys[m.d_out])
        with torch.cuda.stream(stream):
            g.replay()
            stream.synchronize()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(reps):
                g.replay()
            b.record(stream)
            b.synchronize()
        out[name] = (len(mats), sum(m.nbytes() for m in mats), a.elapsed_time(b) / 1e3 / reps)
        del g, mats
    return out


def roofline_entry(dk, peak, peak_kind, ms_per_step, tokens=1):
    launches = sum(v[0] for v in dk.values())
    nbytes = sum(v[1] for v in dk.values())
    secs = sum(v[2] for v in dk.values())
    achieved = nbytes / secs / 1e9
    per_launch = nbytes / launches
    return {
        "bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
        "frac": round(achieved / peak, 4),
        "traffic": round(TRAFFIC_PER_BYTE[tokens] * per_launch) if tokens in TRAFFIC_PER_BYTE else None,
        "traffic_basis": TRAFFIC_BASIS.format(r=TRAFFIC_PER_BYTE[tokens], n=tokens) if tokens in TRAFFIC_PER_BYTE else None,
        "kernel": "NVFP4 weight-stream product kernel (gemv_tma_kernel): one launch per product of the step "
                  "(a layer's q, k, v as one; its gate and up as one), launched back to back in CUDA graphs by "
                  "type, activations prepared beforehand",
        "launches_timed": launches, "bytes_per_launch": round(per_launch), "peak_kind": peak_kind,
        "by_type": {k: {"launches": v[0], "us_per_launch": round(v[2] / v[0] * 1e6, 2),
                        "GBs": round(v[1] / v[2] / 1e9, 1), "frac": round(v[1] / v[2] / 1e9 / peak, 4)}
                    for k, v in dk.items()},
        "product_ms_per_step": round(secs * 1e3, 4),
        "product_ms_within_step": bool(secs * 1e3 <= ms_per_step),
    }


def run_gpu(args):
    import torch
    import torch.distributed as dist
    world, rank, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import __graft_entry__ as g
    if rank == 0:
        g.build()
    if world > 1:
        dist.barrier()
    import bit_weight_streaming_gb300 as bws
    from bit_weight_streaming_gb300 import workloads as W
    import synth

    stream = torch.cuda.Stream(dev)
    t_build = time.time()
    with torch.cuda.stream(stream):
        stack1 = W.dense_27b(1, seed=args.seed, device=dev)
    stream.synchronize()
    t_build = time.time() - t_build
    nbytes = stack1.weight_bytes()
    x1 = synth.activation_bf16(1, stack1.hidden, seed=args.seed, device=dev)
    logits1 = torch.empty((1, stack1.head.d_out), dtype=torch.float32, device=dev)

    def step1():
        stack1.step(x1, logits1)

    with torch.cuda.stream(stream):
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        with ClockSampler(local) as clocks:
            t_step = time_steps(step1, args.steps, args.warmup, stream)
        torch.cuda.synchronize()
    clk = clocks.summary()
    per_rank = all_gather_floats([nbytes, t_step], world)
    value, t_max = aggregate([r[0] for r in per_rank], [r[1] for r in per_rank])
    value /= 1e9

    # end to end through the public API, host buffers: H2D x0, the greedy
    # step (the next token chosen inside the output layer), D2H the token ids
    x_host = x1.cpu().pin_memory()
    x_dev = torch.empty_like(x1)
    tok_dev = torch.empty(1, dtype=torch.int32, device=dev)
    tok_host = torch.empty(1, dtype=torch.int32).pin_memory()

    def step_e2e():
        x_dev.copy_(x_host, non_blocking=True)
        stack1.step_greedy(x_dev, tokens=tok_dev)
        tok_host.copy_(tok_dev, non_blocking=True)

    # the same with the whole logits row brought back instead
    out_host = torch.empty_like(logits1, device="cpu").pin_memory()

    def step_e2e_logits():
        x_dev.copy_(x_host, non_blocking=True)
        stack1.step(x_dev, logits1)
        out_host.copy_(logits1, non_blocking=True)

    with torch.cuda.stream(stream):
        t_e2e = time_steps(step_e2e, args.steps, args.warmup, stream)
        t_e2e_lg = time_steps(step_e2e_logits, args.steps, args.warmup, stream)
    per_rank_e2e = all_gather_floats([nbytes, t_e2e], world)
    e2e_val, _ = aggregate([r[0] for r in per_rank_e2e], [r[1] for r in per_rank_e2e])

    # the speculative-verify shape (8 tokens) on the same weights
    with torch.cuda.stream(stream):
        stack8 = bws.stack.DecodeStack(stack1.hidden, stack1.layers_py, stack1.head, 8, device=dev)
        x8 = synth.activation_bf16(8, stack1.hidden, seed=args.seed, device=dev)
        logits8 = torch.empty((8, stack1.head.d_out), dtype=torch.float32, device=dev)
        t_step8 = time_steps(lambda: stack8.step(x8, logits8), args.steps, args.warmup, stream)

    # dominant kernel: the NVFP4 product, by product type, as in the step
    peak, peak_kind = peaks()
    with torch.cuda.stream(stream):
        dk1 = time_dominant_kernel(stack1, stream)
        dk8 = time_dominant_kernel(stack8, stream)
    del stack8

    # output layers with the greedy choice fused (the full head and the
    # reduced-vocabulary draft head of 100,032 rows), no logits stored
    heads = {}
    with torch.cuda.stream(stream):
        for V, hm in ((stack1.head.d_out, stack1.head),
                      (100032, W.make_matrix(3, (100032, stack1.hidden), args.seed, 100003, device=dev))):
            hws = bws.Workspace(dev)
            t = time_steps(lambda: bws.fp8_lmhead_argmax(hm.codes, hm.scale32, x1, ws=hws), args.steps, args.warmup,
                           stream)
            heads[str(V)] = {"us_per_call": round(t * 1e6, 1), "GBs": round(hm.nbytes() / t / 1e9, 1),
                             "frac_of_hbm_peak": round(hm.nbytes() / t / 1e9 / peak, 4),
                             "weight_bytes": hm.nbytes(), "note": "activation prep + product with fused argmax, N=1"}

    mixed = run_mixed(args, dev, stream, peak)
    w4a8 = run_w4a8(args, dev, stream, peak)

    moe = moe_routed = None
    if not args.no_moe:
        moe = run_moe(args, dev, stream)
        moe_routed = run_moe(args, dev, stream, router=True)

    cpu = cpu_baseline(host_copy(stack1)) if rank == 0 else None

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(t_max * 1e3, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "nvfp4/fp8 weights, bf16 activations, fp32 accumulate",
            "data": "synthetic: seeded N(0,0.02) weights quantized on the GPU, N(0,1) bf16 activations",
            "config": {"workload": "27B-shape dense decode step: 64 NVFP4 layers (48 linear-attention, 16 full-attention, "
                                   "MLP 17408x5120) + FP8 248320x5120 output layer, N=1 token",
                       "weight_bytes_per_step": nbytes, "tokens": 1, "l2": "not flushed: 19.1 GB per step >> 129 MB L2",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                       "graph": "one CUDA graph per step, kernels chained with programmatic dependent launch",
                       "build_s": round(t_build, 1)},
            "us_per_step": round(t_max * 1e6, 1),
            "tokens_per_s": round(world * 1 / t_max, 2),
            "frac_of_hbm_peak": round(value / world / peak, 4),
            "n8": {"value": round(nbytes / t_step8 / 1e9, 2), "unit": UNIT, "us_per_step": round(t_step8 * 1e6, 1),
                   "tokens_per_s": round(8 / t_step8, 1), "frac_of_hbm_peak": round(nbytes / t_step8 / 1e9 / peak, 4)},
            "moe": moe,
            "moe_routed": moe_routed,
            "mixed": mixed,
            "w4a8": w4a8,
            "heads_argmax": heads,
            "e2e": {"value": round(e2e_val / 1e9, 2), "unit": UNIT, "h2d_bytes_per_step": x_host.numel() * 2,
                    "d2h_bytes_per_step": tok_host.numel() * 4,
                    "path": "H2D x0, bws_decode_step_greedy (next token chosen in the output layer), D2H the token id",
                    "with_logits": {"value": round(nbytes / t_e2e_lg / 1e9, 2), "unit": UNIT,
                                    "d2h_bytes_per_step": out_host.numel() * 4}},
            "gpu_launches": stack1.kernel_count * args.steps,
            "roofline": roofline_entry(dk1, peak, peak_kind, t_max * 1e3),
            "roofline_n8": roofline_entry(dk8, peak, peak_kind, t_step8 * 1e3, tokens=8),
            "clocks": clk,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def run_mixed(args, dev, stream, peak, tokens=(1, 8)):
    """The pages' mixed checkpoint: FP8 mixer projections in every layer,
    NVFP4 MLPs in layers 0-55, FP8 MLPs in 56-63, FP8 output layer."""
    import torch
    from bit_weight_streaming_gb300 import workloads as W
    import bit_weight_streaming_gb300 as bws
    import synth
    with torch.cuda.stream(stream):
        base = W.dense_27b_mixed(1, seed=args.seed, device=dev)
    stream.synchronize()
    nbytes = base.weight_bytes()
    out = {"workload": "27B-shape mixed checkpoint: FP8 attention and linear-attention projections (14336x5120, "
                       "5120x8192), NVFP4 MLPs in layers 0-55, FP8 MLPs in 56-63, FP8 248320x5120 output layer",
           "weight_bytes_per_step": nbytes}
    for N in tokens:
        S = base if N == 1 else bws.stack.DecodeStack(base.hidden, base.layers_py, base.head, N, device=dev)
        x = synth.activation_bf16(N, base.hidden, seed=args.seed, device=dev)
        lg = torch.empty((N, base.head.d_out), dtype=torch.float32, device=dev)
        with torch.cuda.stream(stream):
            t = time_steps(lambda: S.step(x, lg), args.steps, args.warmup, stream)
        out[f"n{N}"] = {"value": round(nbytes / t / 1e9, 2), "unit": UNIT, "us_per_step": round(t * 1e6, 1),
                        "frac_of_hbm_peak": round(nbytes / t / 1e9 / peak, 4)}
        del S
    del base
    torch.cuda.empty_cache()
    return out


def run_w4a8(args, dev, stream, peak, shapes=((46336, 5120), (17408, 5120)), tokens=(1, 8), copies=4):
    """W4A8 products (MXFP4 weights, MXFP8 activations, tensor cores) on two
    of the 27B-shape step's matrix shapes held in MXFP4: each call quantizes
    the activations, then streams the weights; a CUDA graph of back-to-back
    calls over four weight copies (each read cold), CUDA events around it."""
    import torch
    import bit_weight_streaming_gb300 as bws
    from bit_weight_streaming_gb300 import workloads as W
    import synth
    out = {}
    for d_out, d_in in shapes:
        with torch.cuda.stream(stream):
            mats = [W.make_matrix(2, (d_out, d_in), args.seed, 500 + i, device=dev) for i in range(copies)]
        stream.synchronize()
        nbytes = mats[0].nbytes()
        for N in tokens:
            x = synth.activation_bf16(N, d_in, seed=args.seed, device=dev)
            y = torch.empty((N, d_out), dtype=torch.bfloat16, device=dev)
            ws = bws.Workspace(dev)
            with torch.cuda.stream(stream):
                for m in mats:
                    bws.mxfp4_w4a8_gemv(m.codes, m.scales, x, y=y, ws=ws)
                stream.synchronize()
                g = torch.cuda.CUDAGraph()
                reps = 5
                with torch.cuda.graph(g, stream=stream):
                    for _ in range(reps):
                        for m in mats:
                            bws.mxfp4_w4a8_gemv(m.codes, m.scales, x, y=y, ws=ws)
                g.replay()
                stream.synchronize()
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record(stream)
                for _ in range(3):
                    g.replay()
                b.record(stream)
                b.synchronize()
            t = a.elapsed_time(b) / 1e3 / (3 * reps * copies)
            out[f"{d_out}x{d_in}_n{N}"] = {"us_per_call": round(t * 1e6, 2), "GBs": round(nbytes / t / 1e9, 1),
                                          "frac_of_hbm_peak": round(nbytes / t / 1e9 / peak, 4),
                                          "weight_bytes": nbytes}
            del g
        del mats
        torch.cuda.empty_cache()
    out["note"] = ("bws_mxfp4_w4a8_gemv: activation quantizer + tcgen05 product per call; weight bytes = MXFP4 codes "
                   "+ E8M0 scales")
    return out


def run_moe(args, dev, stream, tokens=(1, 4), router=False):
    """The Ling-shape MoE step at each N of tokens: with seeded expert ids
    (router=False), or routed by a BF16 512x2560 router per MoE layer inside
    the step (router=True: the distinct experts are those the step chose,
    the routers' bytes count)."""
    import torch
    from bit_weight_streaming_gb300 import workloads as W
    import synth
    out = {}
    for N in tokens:
        t0 = time.time()
        with torch.cuda.stream(stream):
            st = W.moe_ling(N, seed=args.seed, device=dev, router=router)
        stream.synchronize()
        tb = time.time() - t0
        x = synth.activation_bf16(N, st.hidden, seed=args.seed, device=dev)
        lg = torch.empty((N, st.head.d_out), dtype=torch.float32, device=dev)

        def step():   # 1.6 GB (N=1) to 4.5 GB (N=4) of weights per step: no L2 flush needed
            st.step(x, lg)

        with torch.cuda.stream(stream):
            t = time_steps(step, args.steps, args.warmup, stream)
        distinct = W.distinct_per_moe_layer(st)   # routed: the ids the timed steps chose
        nbytes = st.weight_bytes(distinct)
        out[f"n{N}"] = {"value": round(nbytes / t / 1e9, 2), "unit": UNIT, "us_per_step": round(t * 1e6, 1),
                        "weight_bytes_per_step": nbytes, "distinct_experts_mean": round(sum(distinct) / len(distinct), 2),
                        "build_s": round(tb, 1)}
        del st
        torch.cuda.empty_cache()
    out["workload"] = ("Ling-shape MoE decode step: 2 dense MXFP4 MLP layers (6912) + 40 MoE layers (512 experts, "
                       "inter 768, top-8 + 1 shared, MXFP4) + FP8 157184x2560 output layer"
                       + ("; each MoE layer routed in the step by a BF16 512x2560 router (top-8 of its logits, "
                          "softmax weights)" if router else "; seeded expert ids and combine weights"))
    return out


# ---- the reference arm: the oracle on the host cores -------------------------------

def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import numpy as np
    import synth
    from oracle import quant as Q
    # A bounded sample of the same workload: MLP matrices of the 27B-shape
    # stack (gate/up 17408x5120, down 5120x17408), quantized by the oracle.
    mats = []
    shapes = [(17408, 5120)]
    for i, s in enumerate(shapes):
        W = synth.weight_fp32(s, seed=args.seed, index=i).numpy()
        mats.append(Q.nvfp4_quantize(W))
    from oracle import products as P
    rng = np.random.default_rng(args.seed)

    def one_step():
        """The oracle's product over the sample, in this process (numpy uses
        what threads its BLAS starts); returns (seconds, CPU seconds)."""
        t0, c0 = time.perf_counter(), sum(os.times()[:2])
        for codes, scales, ts in mats:
            P.nvfp4_gemv(codes, scales, ts, rng.standard_normal((1, codes.shape[1] * 2)).astype(np.float32))
        return time.perf_counter() - t0, sum(os.times()[:2]) - c0

    for _ in range(args.warmup):
        one_step()
    rates, cpu_s, wall_s = [], 0.0, 0.0
    nbytes = sum(c.nbytes + s.nbytes for c, s, _ in mats)
    for _ in range(args.steps):
        w, c = one_step()
        rates.append(nbytes / w / 1e9)
        wall_s += w
        cpu_s += c
    cores = max(1, round(cpu_s / wall_s))
    desc = (f"oracle NVFP4 GEMV (FP64 products, numpy) over the 17408x5120 gate projection, N=1, in one "
            f"process ({cores} threads busy on average)")
    value = statistics.median(rates)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(nbytes / (value * 1e9) * 1e3, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic: seeded N(0,0.02) weights, N(0,1) bf16 activations",
        "config": {"workload": "27B-shape dense decode step, bounded sample: the MLP gate projection "
                               f"(17408x5120 NVFP4, {nbytes/1e9:.4f} GB) per step, N=1 token", "sample_bytes_per_step": nbytes},
        "cpu_baseline": {"kind": "oracle", "cores": cores, "sample": desc, "value": round(value, 4)},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_product_only(args):
    """Times repeated calls of one NVFP4 product (a small, single-kernel
    workload for profiler captures): --product ROWSxCOLS --tokens N."""
    import torch
    import __graft_entry__ as g
    g.build()
    import bit_weight_streaming_gb300 as bws
    from bit_weight_streaming_gb300 import workloads as W
    import synth
    rows, cols = (int(v) for v in args.product.lower().split("x"))
    dev = torch.device("cuda", 0)
    mats = [W.make_matrix(1, (rows, cols), args.seed, i, device=dev) for i in range(args.copies)]
    x = synth.activation_bf16(args.tokens, cols, seed=args.seed, device=dev)
    y = torch.empty((args.tokens, rows), dtype=torch.bfloat16, device=dev)
    ws = bws.Workspace(dev)
    k = [0]

    def call():
        m = mats[k[0] % len(mats)]
        k[0] += 1
        bws.nvfp4_gemv(m.codes, m.scales, m.scale32, x, y=y, ws=ws)

    stream = torch.cuda.current_stream(dev)
    t = time_steps(call, args.steps, args.warmup, stream)
    nb = mats[0].nbytes()
    print(json.dumps({"product": f"{rows}x{cols}", "tokens": args.tokens, "copies": args.copies,
                      "us_per_call": round(t * 1e6, 2), "GB/s": round(nb / t / 1e9, 1)}), flush=True)


def run_w4a8_only(args):
    """Times repeated W4A8 calls on one MXFP4 matrix shape (a small,
    two-kernel workload for profiler captures): --w4a8 ROWSxCOLS --tokens N."""
    import torch
    import __graft_entry__ as g
    g.build()
    import bit_weight_streaming_gb300 as bws
    from bit_weight_streaming_gb300 import workloads as W
    import synth
    rows, cols = (int(v) for v in args.w4a8.lower().split("x"))
    dev = torch.device("cuda", 0)
    mats = [W.make_matrix(2, (rows, cols), args.seed, 500 + i, device=dev) for i in range(args.copies)]
    x = synth.activation_bf16(args.tokens, cols, seed=args.seed, device=dev)
    y = torch.empty((args.tokens, rows), dtype=torch.bfloat16, device=dev)
    ws = bws.Workspace(dev)
    k = [0]

    def call():
        m = mats[k[0] % len(mats)]
        k[0] += 1
        bws.mxfp4_w4a8_gemv(m.codes, m.scales, x, y=y, ws=ws)

    stream = torch.cuda.current_stream(dev)
    t = time_steps(call, args.steps, args.warmup, stream)
    nb = mats[0].nbytes()
    print(json.dumps({"w4a8": f"{rows}x{cols}", "tokens": args.tokens, "copies": args.copies,
                      "us_per_call": round(t * 1e6, 2), "GB/s": round(nb / t / 1e9, 1)}), flush=True)


def run_moe_layer_only(args):
    """Times repeated calls of one Ling-shape MoE layer (512 MXFP4 experts,
    hidden 2560, inter 768, top-8 + shared; 1.6 GB on the device) through
    bws_mxfp4_moe_gemv at --tokens N: a small workload for profiler captures
    of the expert kernels."""
    import torch
    import __graft_entry__ as g
    g.build()
    import bit_weight_streaming_gb300 as bws
    from bit_weight_streaming_gb300 import workloads as W
    import synth
    dev = torch.device("cuda", 0)
    N, topk = args.tokens, 8
    w = W.moe_weights(512, 2560, 768, args.seed, 2, True, device=dev)
    ids = synth.expert_ids(N, topk, 512, seed=args.seed, layer=2).to(dev)
    rw = synth.route_weights(N, topk, seed=args.seed, layer=2).to(dev)
    x = synth.activation_bf16(N, 2560, seed=args.seed, device=dev)
    y = torch.empty((N, 2560), dtype=torch.bfloat16, device=dev)
    ws = bws.Workspace(dev)
    stream = torch.cuda.current_stream(dev)
    t = time_steps(lambda: bws.mxfp4_moe_gemv(w, ids, rw, x, y=y, ws=ws), args.steps, args.warmup, stream)
    print(json.dumps({"moe_layer": "512 experts, 2560 x 768, top-8 + shared", "tokens": N,
                      "us_per_call": round(t * 1e6, 2)}), flush=True)


def run_dense_only(args):
    """The 27B-shape dense step alone at --tokens N (a workload for profiler
    launch lists): one JSON line with its timing."""
    import torch
    import __graft_entry__ as g
    g.build()
    from bit_weight_streaming_gb300 import workloads as W
    import synth
    dev = torch.device("cuda", 0)
    stream = torch.cuda.Stream(dev)
    with torch.cuda.stream(stream):
        st = W.dense_27b(args.tokens, seed=args.seed, device=dev)
    stream.synchronize()
    x = synth.activation_bf16(args.tokens, st.hidden, seed=args.seed, device=dev)
    lg = torch.empty((args.tokens, st.head.d_out), dtype=torch.float32, device=dev)
    with torch.cuda.stream(stream):
        t = time_steps(lambda: st.step(x, lg), args.steps, args.warmup, stream)
    nbytes = st.weight_bytes()
    print(json.dumps({"dense_only": {f"n{args.tokens}": {"value": round(nbytes / t / 1e9, 2), "unit": UNIT,
                                                         "us_per_step": round(t * 1e6, 1)}}}), flush=True)


def run_moe_only(args):
    """The MoE step alone at --tokens N (a short workload for profiler launch
    lists): one JSON line with its timing."""
    import torch
    import __graft_entry__ as g
    g.build()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.Stream(dev)
    out = run_moe(args, dev, stream, tokens=(args.tokens,), router=args.router)
    print(json.dumps({"moe_only": out}), flush=True)


# ---- opt-in timestamp trace of one step (profiling aid) ---------------------
#
# With --trace dense|moe the library is rebuilt with -DBWS_TRACE: every CTA of
# the product, MoE expert and prep kernels records global-timer readings
# (kernel start, its waits returning, first stage, loop done, end; for preps:
# wait, loads done, statistics, stores, end). One step is recorded after
# warm-up and summarised per product boundary. Timing runs never use this
# build (the build script rebuilds when the flags change).

TRACE_DTYPE = [("kind", "<u8"), ("cta", "<u8"), ("t", "<u8", (6,))]


def trace_read(lib):
    import ctypes as C
    import numpy as np
    cap = 1 << 17
    buf = np.zeros(cap, dtype=np.dtype(TRACE_DTYPE))
    out = []
    for fn in ("bws_trace_read_tma", "bws_trace_read_prep", "bws_trace_read_moe"):
        f = getattr(lib, fn)
        f.restype = C.c_int
        n = f(C.c_void_p(buf.ctypes.data), cap)
        if n < 0:
            raise RuntimeError(f"{fn} failed")
        out.append(buf[:n].copy())
    return np.concatenate(out)


def trace_launches(rec):
    """The step's launches in start order: (kind, record indices), a new
    launch wherever the kernel kind changes (consecutive launches of the
    step's chain always differ in kind)."""
    import numpy as np
    t0 = rec["t"][:, 0]
    order = np.argsort(t0, kind="stable")
    segs, cur, ck = [], [], None
    for i in order:
        k = int(rec["kind"][i])
        if ck is not None and k != ck:
            segs.append((ck, np.array(cur)))
            cur = []
        cur.append(i)
        ck = k
    if cur:
        segs.append((ck, np.array(cur)))
    return segs


def trace_summary_dense(rec):
    """Per product kind (kind 1000 + 100 fmt + 10 epilogue + deposit), the
    average microseconds of each piece of a product and the boundary after it."""
    import numpy as np
    t = rec["t"].astype(np.int64)
    segs = trace_launches(rec)
    P = [s for s in segs if s[0] // 1000 == 1]
    Q = [s for s in segs if s[0] // 1000 in (2, 3)]
    med = lambda a: float(np.median(a))
    names = ["wait->first stage", "stream (median CTA)", "CTA spread", "last CTA -> prep wait", "prep loads",
             "prep statistics barrier", "prep bands and stores", "prep end -> next wait", "next wait -> first stage"]
    agg = {}
    for k in range(min(len(P) - 1, len(Q) - 1)):
        (pk, p), (_, q), (_, pn) = P[k], Q[k + 1], P[k + 1]
        v = [med(t[p, 3]) - med(t[p, 2]), med(t[p, 4]) - med(t[p, 3]), t[p, 4].max() - med(t[p, 4]),
             t[q, 1].min() - t[p, 5].max(), t[q, 2].max() - t[q, 1].min(), t[q, 3].max() - t[q, 2].max(),
             t[q, 4].max() - t[q, 3].max(), med(t[pn, 2]) - t[q, 5].max(), med(t[pn, 3]) - med(t[pn, 2])]
        agg.setdefault(pk, []).append(v)
    out = {}
    for pk, v in agg.items():
        a = np.mean(np.array(v), axis=0) / 1e3
        out[str(pk)] = {"launches": len(v), **{n: round(float(x), 2) for n, x in zip(names, a)}}
    span = (t[:, 5].max() - t[:, 0].min()) / 1e3
    return {"span_us": round(float(span), 1), "by_product_kind_us": out}


def trace_summary_moe(rec):
    """Per MoE layer (prep 3100 + CL, gate/up 403x, h prep 3001, down 401x),
    the average microseconds of each kernel's pieces and the hops between."""
    import numpy as np
    t = rec["t"].astype(np.int64)
    segs = trace_launches(rec)
    med = lambda a: float(np.median(a))
    names = ["prev end -> prep wait", "MoE prep", "-> gate/up wait", "gate/up wait -> first stage",
             "gate/up stream (median CTA)", "gate/up CTA spread", "-> h prep wait", "h prep",
             "-> down wait", "down wait -> first stage", "down stream (median CTA)", "down CTA spread",
             "-> next prep wait", "layer"]
    rows = []
    for i in range(1, len(segs) - 4):
        ks = [segs[i + j][0] for j in range(5)]
        if not (ks[0] // 100 == 31 and ks[1] // 10 == 403 and ks[2] == 3001 and ks[3] // 10 == 401
                and ks[4] // 100 == 31):
            continue
        pv, p, g, h, d, p2 = (segs[i + j][1] for j in range(-1, 5))
        rows.append([t[p, 1].min() - t[pv, 5].max(), t[p, 5].max() - t[p, 1].min(),
                     med(t[g, 2]) - t[p, 5].max(), med(t[g, 3]) - med(t[g, 2]), med(t[g, 4]) - med(t[g, 3]),
                     t[g, 4].max() - med(t[g, 4]), t[h, 1].min() - t[g, 5].max(), t[h, 5].max() - t[h, 1].min(),
                     med(t[d, 2]) - t[h, 5].max(), med(t[d, 3]) - med(t[d, 2]), med(t[d, 4]) - med(t[d, 3]),
                     t[d, 4].max() - med(t[d, 4]), t[p2, 1].min() - t[d, 5].max(), t[p2, 0].min() - t[p, 0].min()])
    a = np.mean(np.array(rows), axis=0) / 1e3 if rows else []
    span = (t[:, 5].max() - t[:, 0].min()) / 1e3
    return {"span_us": round(float(span), 1), "moe_layers": len(rows),
            "per_layer_us": {n: round(float(x), 2) for n, x in zip(names, a)}}


def run_trace(args):
    """One step of the dense (--trace dense) or MoE (--trace moe) stack at
    --tokens N, recorded with the opt-in timestamp trace."""
    os.environ["BWS_NVCC_FLAGS"] = (os.environ.get("BWS_NVCC_FLAGS", "") + " -DBWS_TRACE").strip()
    import torch
    import __graft_entry__ as g
    g.build()
    from bit_weight_streaming_gb300._lib import lib
    from bit_weight_streaming_gb300 import workloads as W
    import synth
    L = lib()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.Stream(dev)
    N = args.tokens
    with torch.cuda.stream(stream):
        st = W.dense_27b(N, seed=args.seed, device=dev) if args.trace == "dense" else \
            W.moe_ling(N, seed=args.seed, device=dev)
    stream.synchronize()
    x = synth.activation_bf16(N, st.hidden, seed=args.seed, device=dev)
    lg = torch.empty((N, st.head.d_out), dtype=torch.float32, device=dev)
    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 3)):
            st.step(x, lg)
        stream.synchronize()
        trace_read(L)            # drop the warm-up steps' records
        st.step(x, lg)
        stream.synchronize()
    rec = trace_read(L)
    summ = trace_summary_dense(rec) if args.trace == "dense" else trace_summary_moe(rec)
    print(json.dumps({"trace": args.trace, "tokens": N, "records": int(len(rec)), **summ}), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-moe", action="store_true")
    ap.add_argument("--product", default=None, help="ROWSxCOLS: time one NVFP4 product only (profiling)")
    ap.add_argument("--moe-only", action="store_true", help="time the MoE step alone at --tokens N (profiling)")
    ap.add_argument("--dense-only", action="store_true", help="time the dense step alone at --tokens N (profiling)")
    ap.add_argument("--w4a8", default=None, help="ROWSxCOLS: time one W4A8 product only (profiling)")
    ap.add_argument("--moe-layer", action="store_true",
                    help="time one Ling-shape MoE layer call at --tokens N (profiling)")
    ap.add_argument("--tokens", type=int, default=1)
    ap.add_argument("--trace", choices=["dense", "moe"], default=None,
                    help="record one step of the dense or MoE stack with the opt-in timestamp trace (profiling)")
    ap.add_argument("--router", action="store_true", help="--moe-only: MoE layers routed inside the step")
    ap.add_argument("--copies", type=int, default=4, help="--product: distinct weight copies to rotate")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.trace:
        run_trace(args)
    elif args.product:
        run_product_only(args)
    elif args.w4a8:
        run_w4a8_only(args)
    elif args.moe_layer:
        run_moe_layer_only(args)
    elif args.moe_only:
        run_moe_only(args)
    elif args.dense_only:
        run_dense_only(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
