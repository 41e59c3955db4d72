"""Benchmark of the MoE expert layer (one GB300 per process).

A step is one moe_forward over one batch of the large skewed workload (T=16384 tokens,
d=7168, E=256 experts, top-8, d_ff=2048, router logits with a Zipf(1.2) bias): routing,
dispatch, grouped GEMM1 + SwiGLU, grouped GEMM2 and the fp32 combine, all in libmoe.so.
Inputs are synthetic (moe_synth) and resident in HBM; the 22.5 GB of expert weights are far
larger than the 129 MB L2, so no L2 flush is needed between steps.

Prints one JSON line (rank 0).  With --gpus N > 1 (under torchrun) every rank runs an
independent replica on its own GPU (the layer does not shard); value = all tokens / the
slowest rank's time.  The line also carries the forward + backward time of the fwd_bwd
workload (T=8192, d=4096, E=128, top-8, d_ff=1536) unless --no-backward, and the time of the
overlapped-wave forward variant.  --impl reference times the fp64 CPU oracle instead, on a
bounded sample of the same workload.
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import moe_synth  # noqa: E402

METRIC = "MoE layer tokens/s; grouped-GEMM bf16 TFLOP/s and dispatch GB/s as % of peak"
UNIT = "tokens/s"
WORKLOAD = "large_skewed"


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return dict(hbm=p["hbm_gbs"], bf16=p["bf16_tflops"],
                    bf16_sustained=p.get("bf16_tflops_sustained", p["bf16_tflops"]),
                    source="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sustained=1700.0, source="fallback")


def _workload_config(w):
    return {"workload": "%s: T=%d d=%d E=%d top-%d d_ff=%d %s, logits N(0,1) - %.1f ln(e+1)"
                        % (w.name, w.T, w.d, w.E, w.k, w.dff,
                           "SwiGLU" if w.gated else "squared ReLU (no gate projection)",
                           w.zipf_s),
            "T": w.T, "d": w.d, "E": w.E, "k": w.k, "d_ff": w.dff,
            "l2": "inputs larger than L2 (%.1f GB of expert weights read every step)"
                  % (w.E * (3 if w.gated else 2) * w.d * w.dff * 2 / 1e9),
            "activation": "SwiGLU" if w.gated else "squared ReLU",
            "parallelism": "replicas (one independent layer per GPU)"}


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        try:
            with open(self.path) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) < 9:
                        continue
                    try:
                        sm.append(float(parts[1]))
                        mx.append(float(parts[2]))
                    except ValueError:
                        continue
                    for n, v in zip(names, parts[5:9]):
                        if v.lower() == "active":
                            reasons.add(n)
            os.unlink(self.path)
        except OSError:
            pass
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        load = [s for s in sm if s > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(load), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def _algorithmic(w, P):
    d, dff, T, E, k = w.d, w.dff, w.T, w.E, w.k
    n1 = 2 if w.gated else 1  # projections in GEMM1: gate + up (SwiGLU) or up alone
    return dict(
        gemm_flops=(2 * n1 + 2) * d * dff * P,  # 6 d dff per pair (4 d dff without the gate)
        gemm1_flops=2 * n1 * d * dff * P,       # gate + up projections (or up alone)
        gemm2_flops=2 * d * dff * P,            # down projection
        # logits read; topk, gate, pos, perm written; x read; x_perm written
        dispatch_bytes=T * E * 4 + T * k * 16 + T * d * 2 + P * d * 2,
        # the routing part alone (when GEMM1 copies the rows): logits read, topk, gate, pos,
        # perm written
        dispatch_route_bytes=T * E * 4 + T * k * 16,
        # combine: bf16 expert-output rows read (the pages' BF16 gather), gate + pos read,
        # out written (bf16)
        combine_bytes=P * d * 2 + T * k * 8 + T * d * 2,
    )


def max_over_ranks(value, device):
    """The largest `value` over all ranks (the slowest rank's time); `value` itself with one
    process."""
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return value
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def _row_pairs(T, k, d, dff):
    # the library's rule for CTA pairs in the row-grouped GEMMs (MOE_GEMM_PAIR: "0" never,
    # "1" whenever T > 128, else T > 128 and T k d d_ff >= 2^37)
    mode = os.environ.get("MOE_GEMM_PAIR", "")
    if mode == "0" or T <= 128:
        return False
    return mode == "1" or T * k * d * dff >= 2 ** 37


def _swap_size(T, k, d, dff):
    # the library's size rule for the swapped-operand GEMMs: T <= 128, wherever row tiles
    # would pair, and (unless MOE_GEMM_PAIR is set) from T k d d_ff >= 2^36
    if T <= 128 or _row_pairs(T, k, d, dff):
        return True
    return os.environ.get("MOE_GEMM_PAIR", "") not in ("0", "1") and T * k * d * dff >= 2 ** 36


def _forward_swap(T, k, d, dff):
    # the library's rule for the swapped forward GEMMs (MOE_FWD_SWAP: "0" never, "1" always,
    # else the size rule); never with MOE_GEMM_PAIR "0"
    mode = os.environ.get("MOE_FWD_SWAP", "")
    if mode == "0" or os.environ.get("MOE_GEMM_PAIR", "") == "0":
        return False
    return mode == "1" or _swap_size(T, k, d, dff)


def _gemm_row_copy(T, k, d, dff):
    # the library's rule for the swapped GEMM1 copying the permuted rows itself
    # (MOE_FWD_ROW_COPY "0" leaves them to the dispatch's scatter): T > 128, swapped GEMMs as
    # two launches
    if os.environ.get("MOE_FWD_ROW_COPY", "") == "0":
        return False
    return T > 128 and _forward_swap(T, k, d, dff) and not _forward_fused(T, k, d, dff)


def _forward_fused(T, k, d, dff):
    # both swapped GEMMs in one launch: the library's rule (MOE_FWD_FUSED "1" always, "0"
    # never, else T <= 64)
    mode = os.environ.get("MOE_FWD_FUSED", "")
    return _forward_swap(T, k, d, dff) and mode != "0" and (mode == "1" or T <= 64)


def fwd_launches(T, k, d, dff, save=False):
    # dispatch: routing, column scan, offsets/tile tables, scatter, padding rows; or, for
    # T <= 128, the library's single dispatch launch (plus the zeroing of the padding rows
    # when saving for the backward).  GEMM1 and GEMM2: one swapped launch each, or one
    # together for T <= 64; with row-tile CTA pairs each is a pair launch plus a single-CTA
    # launch for the other tiles.  Then the combine.
    if 0 < T <= 128:
        dispatch = 2 if save else 1
    else:
        dispatch = 5
    if _forward_swap(T, k, d, dff):
        gemms = 1 if _forward_fused(T, k, d, dff) else 2
    else:
        gemms = 4 if _row_pairs(T, k, d, dff) else 2
    return dispatch + gemms + 1


def _backward_swap(T, k, d, dff):
    # the library's rule for the backward's swapped dX GEMM (MOE_BWD_SWAP: "0" never, "1"
    # always, else the forward's size rule); never with MOE_GEMM_PAIR "0"
    mode = os.environ.get("MOE_BWD_SWAP", "")
    if mode == "0" or os.environ.get("MOE_GEMM_PAIR", "") == "0":
        return False
    return mode == "1" or _swap_size(T, k, d, dff)


def _backward_swap_dh(T, k, d, dff):
    # the library's rule for the backward's swapped dH GEMM (MOE_BWD_DH_SWAP: "0" never, "1"
    # always, else as the swapped dX); never with MOE_GEMM_PAIR "0"
    mode = os.environ.get("MOE_BWD_DH_SWAP", "")
    if mode == "0" or os.environ.get("MOE_GEMM_PAIR", "") == "0":
        return False
    return mode == "1" or _backward_swap(T, k, d, dff)


def bwd_launches(T, k, d, dff):
    # gate grads (rows + per token), dO padding, dH and dX (each: pair tiles + single-CTA
    # tiles, or one swapped launch), dX combine, dW2, dW1/dW3
    pairs = _row_pairs(T, k, d, dff)
    dh = 1 if _backward_swap_dh(T, k, d, dff) or not pairs else 2
    dx = 1 if _backward_swap(T, k, d, dff) or not pairs else 2
    return 6 + dh + dx


def bench_fwd_bwd(moe, dev, steps, warmup, shape=None):
    """Forward (saving for backward) + backward of the fwd_bwd workload (T=8192, d=4096,
    E=128, top-8, d_ff=1536; or `shape` = (T, d, E, k, d_ff)), device-resident, with the
    backward's stage times."""
    w = moe_synth.by_name("fwd_bwd")
    if shape:
        w = moe_synth.custom(*shape, seed=w.seed, name="fwd_bwd_custom")
    g = moe_synth.generate(w, device=dev, with_dy=True)
    T, d, E, k, dff = w.T, w.d, w.E, w.k, w.dff
    ws = torch.empty(moe.moe_workspace_bytes(T, d, E, k, dff, True), dtype=torch.uint8,
                     device=dev)
    out = torch.empty(T, d, dtype=torch.bfloat16, device=dev)
    res = dict(dx=torch.empty(T, d, dtype=torch.bfloat16, device=dev),
               dW1=torch.empty(E, d, dff, dtype=torch.float32, device=dev),
               dW3=torch.empty(E, d, dff, dtype=torch.float32, device=dev),
               dW2=torch.empty(E, dff, d, dtype=torch.float32, device=dev),
               dgate=torch.empty(T, k, dtype=torch.float32, device=dev),
               dlogits=torch.empty(T, E, dtype=torch.float32, device=dev))
    stream = torch.cuda.current_stream(dev)
    nb = moe.MOE_BWD_NUM_EVENTS
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nb)] for _ in range(steps)]

    def step(ev=None):
        moe.moe_forward(g["x"], g["logits"], g["W1"], g.get("W3"), g["W2"], k, out, ws,
                        flags=moe.MOE_FWD_SAVE_FOR_BACKWARD, stream=stream)
        moe.moe_backward(g["dy"], g["x"], g["logits"], g["W1"], g.get("W3"), g["W2"], k,
                         res["dx"], res["dW1"], res["dW3"], res["dW2"], res["dgate"],
                         res["dlogits"], ws, stage_events=ev, stream=stream)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(steps):
        step()
    stop.record(stream)
    torch.cuda.synchronize()
    ms = start.elapsed_time(stop) / steps
    # the backward's stage times, from a second pass that records the stage events (kept out
    # of the timed pass: recording them costs time of its own at small sizes)
    for i in range(steps):
        step(evs[i])
    torch.cuda.synchronize()
    st = moe.moe_get_error(ws)
    if st != 0:
        raise RuntimeError("device error in forward + backward: " + moe.moe_status_string(st))
    names = ["gate_grads", "dh_swiglu_bwd", "dx_gemm", "dx_combine", "dw2", "dw13"]
    stages = {n: sum(e[j].elapsed_time(e[j + 1]) for e in evs) / steps
              for j, n in enumerate(names)}
    bwd_ms = sum(stages.values())
    P = T * k
    # backward GEMM flops per token-expert pair: dH = dO W2^T (2 d dff), dX from dA and dB
    # (4 d dff), dW1 and dW3 (4 d dff), dW2 (2 d dff): 12 d dff in total
    bwd_flops = 12 * d * dff * P
    return {"workload": "fwd_bwd: T=%d d=%d E=%d top-%d d_ff=%d" % (T, d, E, k, dff),
            "ms_per_step": ms, "tokens_per_s": T / (ms * 1e-3),
            "backward_ms": bwd_ms, "backward_stages_ms": stages,
            "backward_tflops": bwd_flops / (bwd_ms * 1e-3) / 1e12,
            "launches_per_step": fwd_launches(T, k, d, dff, save=True) + bwd_launches(T, k, d, dff)}


def run_cpu_baseline(w, inp_np, budget_s=15.0):
    import oracle
    cores = oracle.num_threads()
    tok_all = np.random.default_rng(0).permutation(w.T)
    n = 8
    t0 = time.perf_counter()
    oracle.forward_tokens(inp_np, w.k, tokens=tok_all[:n])
    dt = time.perf_counter() - t0
    n2 = int(max(n, min(w.T, n * budget_s / max(dt, 1e-3))))
    t0 = time.perf_counter()
    oracle.forward_tokens(inp_np, w.k, tokens=tok_all[:n2])
    dt2 = time.perf_counter() - t0
    return {"value": n2 / dt2, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": "%d random tokens of the %s workload, fp64, %.1f s" % (n2, w.name, dt2)}


def bench_reference(args, w):
    world, rank, _ = _dist()
    if rank != 0:
        return 0
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    g = moe_synth.generate(w, device=dev)
    inp = moe_synth.to_numpy(g)
    del g
    import oracle
    cores = oracle.num_threads()
    rng = np.random.default_rng(0)
    per_step = 16
    for _ in range(args.warmup):
        oracle.forward_tokens(inp, w.k, tokens=rng.choice(w.T, per_step, replace=False))
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.forward_tokens(inp, w.k, tokens=rng.choice(w.T, per_step, replace=False))
    dt = time.perf_counter() - t0
    value = per_step * args.steps / dt
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * dt / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": _workload_config(w),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": "%d random tokens per step of the %s workload"
                                       % (per_step, w.name)},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def bench_native(args, w):
    import combine_fp32_router_gb300 as moe

    world, rank, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    g = moe_synth.generate(w, device=dev)
    T, d, E, k, dff = w.T, w.d, w.E, w.k, w.dff
    ws = torch.empty(moe.moe_workspace_bytes(T, d, E, k, dff, False), dtype=torch.uint8,
                     device=dev)
    out = torch.empty(T, d, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)
    nev = moe.MOE_FWD_NUM_EVENTS
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nev)] for _ in range(args.steps)]

    def step(ev=None):
        moe.moe_forward(g["x"], g["logits"], g["W1"], g.get("W3"), g["W2"], k, out, ws,
                        stage_events=ev, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    st = moe.moe_get_error(ws)
    if st != 0:
        raise RuntimeError("device error during warm-up: " + moe.moe_status_string(st))

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        barrier()
        start.record(stream)
        for i in range(args.steps):
            step()
        stop.record(stream)
        barrier()
    ms = max_over_ranks(start.elapsed_time(stop), dev)
    # stage times from a second pass that records the library's stage events (kept out of the
    # timed pass: recording them costs time of its own at small sizes)
    for i in range(args.steps):
        step(evs[i])
    barrier()
    st = moe.moe_get_error(ws)
    if st != 0:
        raise RuntimeError("device error: " + moe.moe_status_string(st))

    stage_ms = [0.0] * (nev - 1)
    for e in evs:
        for j in range(nev - 1):
            stage_ms[j] += e[j].elapsed_time(e[j + 1])
    stage_ms = [s / args.steps for s in stage_ms]
    P = T * k
    alg = _algorithmic(w, P)
    peaks = _peaks()
    ms_step = ms / args.steps
    value = world * T * args.steps / (ms / 1e3)

    # end to end through the public API with host buffers: each step copies its x and logits
    # from page-locked host memory into a workspace, runs the layer and copies the output back
    # (moe_forward_host_pipelined).  The layers run one after another on one compute stream;
    # two workspaces, each with its own copy stream, take alternate steps, so one step's copies
    # overlap its neighbours' layers.  Every step still moves its own inputs and output.
    ws_io = [torch.empty(moe.moe_workspace_bytes(T, d, E, k, dff, False, host_io=True),
                         dtype=torch.uint8, device=dev) for _ in range(2)]
    compute = torch.cuda.Stream(dev)
    copy_streams = [torch.cuda.Stream(dev) for _ in range(2)]
    copy_events = [[torch.cuda.Event(), torch.cuda.Event()] for _ in range(2)]
    hx = [g["x"].cpu().pin_memory() for _ in range(2)]
    hl = [g["logits"].cpu().pin_memory() for _ in range(2)]
    ho = [torch.empty(T, d, dtype=torch.bfloat16).pin_memory() for _ in range(2)]

    def e2e_step(i):
        j = i % 2
        moe.moe_forward_host_pipelined(hx[j], hl[j], g["W1"], g.get("W3"), g["W2"], k, ho[j],
                                       ws_io[j], copy_stream=copy_streams[j],
                                       events=copy_events[j], stream=compute)

    for i in range(max(2, args.warmup)):
        e2e_step(i)
    barrier()
    used = [compute] + copy_streams
    ends = [torch.cuda.Event() for _ in used]
    start.record(stream)
    for s_ in used:
        s_.wait_event(start)
    for i in range(args.steps):
        e2e_step(i)
    for s_, e_ in zip(used, ends):
        e_.record(s_)
        stream.wait_event(e_)
    stop.record(stream)
    barrier()
    ms_e2e = max_over_ranks(start.elapsed_time(stop), dev)
    for wsi in ws_io:
        st = moe.moe_get_error(wsi)
        if st != 0:
            raise RuntimeError("device error (host-buffer forward): " + moe.moe_status_string(st))
    e2e_out = ho[(args.steps - 1) % 2]
    if not torch.equal(e2e_out.view(torch.int16), out.cpu().view(torch.int16)):
        raise RuntimeError("host-buffer forward differs from the device forward")
    del ws_io

    # the same step replayed from a captured CUDA graph (the launch-overhead path)
    graph = moe.moe_forward_graph_create(g["x"], g["logits"], g["W1"], g.get("W3"), g["W2"], k, out,
                                         ws)
    for _ in range(2):
        graph.launch(stream)
    barrier()
    n_graph = max(1, min(args.steps, 20))
    start.record(stream)
    for _ in range(n_graph):
        graph.launch(stream)
    stop.record(stream)
    barrier()
    graph_ms = start.elapsed_time(stop) / n_graph
    graph.close()
    st = moe.moe_get_error(ws)
    if st != 0:
        raise RuntimeError("device error (graph replay): " + moe.moe_status_string(st))

    # the same step with the FP8 dispatch payload (E4M3 rows and W1 / W3, quantized outside
    # the timed region), with its stage times
    fp8 = None
    if "W3" in g:
        W1q, s1 = moe.moe_quantize_weights_fp8(g["W1"])
        W3q, s3 = moe.moe_quantize_weights_fp8(g["W3"])
        n_fp8 = max(1, min(args.steps, 20))
        evf = [[torch.cuda.Event(enable_timing=True) for _ in range(nev)] for _ in range(n_fp8)]
        for _ in range(2):
            moe.moe_forward_fp8(g["x"], g["logits"], W1q, W3q, s1, s3, g["W2"], k, out, ws,
                                stream=stream)
        barrier()
        start.record(stream)
        for i in range(n_fp8):
            moe.moe_forward_fp8(g["x"], g["logits"], W1q, W3q, s1, s3, g["W2"], k, out, ws,
                                stream=stream)
        stop.record(stream)
        barrier()
        for i in range(n_fp8):      # stage times, from a pass of their own
            moe.moe_forward_fp8(g["x"], g["logits"], W1q, W3q, s1, s3, g["W2"], k, out, ws,
                                stage_events=evf[i], stream=stream)
        barrier()
        st = moe.moe_get_error(ws)
        if st != 0:
            raise RuntimeError("device error (fp8 forward): " + moe.moe_status_string(st))
        f_ms = start.elapsed_time(stop) / n_fp8
        f_st = [sum(e[j].elapsed_time(e[j + 1]) for e in evf) / n_fp8 for j in range(nev - 1)]
        fp8 = {"ms_per_step": f_ms, "tokens_per_s": world * T / (f_ms * 1e-3),
               "stages_ms": dict(zip(["dispatch", "gemm1_swiglu_fp8", "gemm2", "combine"], f_st)),
               "gemm1_tflops": 4 * d * dff * T * k / (f_st[1] * 1e-3) / 1e12}
        del W1q, W3q, s1, s3

    # the overlapped-wave variant (GEMM1 gathers rows from x, GEMM2 fuses the combine),
    # timed for comparison; bitwise the same output
    wave_flags = moe.MOE_FWD_GATHER_ROWS | moe.MOE_FWD_FUSED_COMBINE
    for _ in range(2):
        moe.moe_forward(g["x"], g["logits"], g["W1"], g.get("W3"), g["W2"], k, out, ws,
                        flags=wave_flags, stream=stream)
    barrier()
    n_wave = max(1, min(args.steps, 10))
    start.record(stream)
    for _ in range(n_wave):
        moe.moe_forward(g["x"], g["logits"], g["W1"], g.get("W3"), g["W2"], k, out, ws,
                        flags=wave_flags, stream=stream)
    stop.record(stream)
    barrier()
    waved_ms = start.elapsed_time(stop) / n_wave
    st = moe.moe_get_error(ws)
    if st != 0:
        raise RuntimeError("device error (waved forward): " + moe.moe_status_string(st))

    e2e = {"value": world * T * args.steps / (ms_e2e / 1e3), "unit": UNIT,
           "h2d_bytes_per_step": T * d * 2 + T * E * 4, "d2h_bytes_per_step": T * d * 2,
           "api": "moe_forward_host_pipelined: page-locked host buffers; layers on one "
                  "compute stream, two workspaces with a copy stream each taking alternate "
                  "steps"}

    names = ["dispatch", "gemm1_swiglu", "gemm2", "combine"]
    stages = dict(zip(names, stage_ms))
    # per-expert roofline of the grouped GEMMs under this workload's load: every active expert
    # streams its 3 weight matrices once and does 6 d d_ff FLOP per routed row
    counts = torch.bincount(torch.topk(g["logits"], k, dim=1).indices.flatten(),
                            minlength=E).double().cpu().numpy()
    active = counts > 0
    w_bytes = (3 if w.gated else 2) * 2 * d * dff  # per active expert
    fpr = (6 if w.gated else 4) * d * dff  # FLOP per routed row
    t_e = np.maximum(fpr * counts[active] / (peaks["bf16"] * 1e12), w_bytes / (peaks["hbm"] * 1e9))
    gemm_ms = stages["gemm1_swiglu"] + stages["gemm2"]
    roof = {"per_expert_sum_ms": float(t_e.sum() * 1e3),
            "overlapped_ms": float(max(fpr * counts.sum() / (peaks["bf16"] * 1e12),
                                       active.sum() * w_bytes / (peaks["hbm"] * 1e9)) * 1e3),
            "active_experts": int(active.sum()),
            "weights_gb": float(active.sum() * w_bytes / 1e9),
            "weights_gbs": float(active.sum() * w_bytes / (gemm_ms * 1e-3) / 1e9)}
    roof["gemm_frac_of_per_expert_sum"] = roof["per_expert_sum_ms"] / gemm_ms
    roof["gemm_frac_of_overlapped"] = roof["overlapped_ms"] / gemm_ms
    fused = _forward_fused(T, k, d, dff)
    # the dominant kernel: GEMM1 + SwiGLU, or both GEMMs when they run as one launch (its
    # stage then spans both and the GEMM2 stage is empty)
    g1_flops = alg["gemm_flops"] if fused else alg["gemm1_flops"]
    g1_tflops = g1_flops / (stages["gemm1_swiglu"] * 1e-3) / 1e12
    g_tflops = alg["gemm_flops"] / ((stages["gemm1_swiglu"] + stages["gemm2"]) * 1e-3) / 1e12
    # with GEMM1 copying the rows, the dispatch stage moves only the routing bytes
    row_copy = _gemm_row_copy(T, k, d, dff)
    disp_bytes = alg["dispatch_route_bytes"] if row_copy else alg["dispatch_bytes"]
    disp_gbs = disp_bytes / (stages["dispatch"] * 1e-3) / 1e9
    comb_gbs = alg["combine_bytes"] / (stages["combine"] * 1e-3) / 1e9
    # GEMM1 runs for milliseconds inside a sub-second timed loop: the burst peak applies
    peak = peaks["bf16"]
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": _workload_config(w),
        "e2e": e2e,
        "roofline": {"kernel": ("grouped GEMM1 + SwiGLU + GEMM2, one tcgen05 launch" if fused
                                else "grouped GEMM1 + SwiGLU (tcgen05)"), "bound": "tensor",
                     "achieved": g1_tflops, "peak": peak, "unit": "TFLOP/s",
                     "frac": g1_tflops / peak,
                     "peak_source": "%s bf16 burst (MEASURED_PEAKS.json)" % peaks["source"],
                     "frac_of_sustained": g1_tflops / peaks["bf16_sustained"],
                     # DRAM bytes of one full-size launch are not captured (over the
                     # capture-size rule) and do not scale with the units; skewed
                     # T=8192 d=4096 E=64 captures read 1.28-1.45x their algorithmic bytes
                     "traffic": None},
        "stages_ms": stages,
        "gemm_tflops": g_tflops,
        "gemm_frac_of_bf16_burst": g_tflops / peaks["bf16"],
        "gemm_roofline_under_load": roof,
        "dispatch_gbs": disp_gbs, "dispatch_frac_of_hbm": disp_gbs / peaks["hbm"],
        "dispatch_rows_copied_by": "gemm1" if row_copy else "scatter",
        "combine_gbs": comb_gbs, "combine_frac_of_hbm": comb_gbs / peaks["hbm"],
        "waved_forward_ms_per_step": waved_ms,
        "graph_forward_ms_per_step": graph_ms,
        "fp8_forward": fp8,
        "clocks": clocks.summary(),
        "gpu_launches": fwd_launches(T, k, d, dff) * args.steps,
    }
    if not args.no_backward:
        del ws
        torch.cuda.empty_cache()
        bshape = tuple(int(v) for v in args.bwd_shape.split(",")) if args.bwd_shape else None
        line["fwd_bwd"] = bench_fwd_bwd(moe, dev, max(1, min(args.steps, 10)), args.warmup,
                                        bshape)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        del out
        torch.cuda.empty_cache()
        line["cpu_baseline"] = run_cpu_baseline(w, moe_synth.to_numpy(g))
    if world > 1:
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def probe_dram():
    """Per-SM DRAM read rate against the number of streaming SMs (moe_probe_dram_read): one
    JSON line per (path, SMs)."""
    import combine_fp32_router_gb300 as moe
    buf = torch.empty(6 << 30, dtype=torch.uint8, device="cuda")
    buf.fill_(1)
    out = torch.zeros(1024, dtype=torch.int32, device="cuda")
    per_cta = (buf.numel() // 152) // 16384 * 16384
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for ctas in (4, 8, 16, 38, 76, 152):
        for mode, name in ((0, "loads, 32 KB in flight"), (1, "bulk copies, 6 x 16 KB"),
                           (2, "bulk copies, 12 x 16 KB"),
                           (3, "64x64 boxes, rows 4 KB apart, 6 x 16 KB"),
                           (4, "64x64 boxes, contiguous rows, 6 x 16 KB")):
            moe.moe_probe_dram_read(buf, ctas, mode, out)
            a.record()
            moe.moe_probe_dram_read(buf, ctas, mode, out)
            b.record()
            torch.cuda.synchronize()
            ms = a.elapsed_time(b)
            if mode < 3:
                nbytes = per_cta
            else:  # 256 bytes of each of the CTA's rows (the probe's split of the matrix)
                cols = 2048 if mode == 3 else 128
                nblk = cols // 128
                rows = buf.numel() // (cols * 2)
                nbytes = rows // ((152 + nblk - 1) // nblk) // 64 * 64 * 256
            print(json.dumps({"path": name, "sms": ctas, "total_gbs": ctas * nbytes / ms / 1e6,
                              "per_sm_gbs": nbytes / ms / 1e6,
                              "timed_out": int(out[:ctas].sum().item())}), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--shape", default=None,
                    help="T,d,E,k,d_ff of a custom workload (profiling captures of one kernel)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--tokens", type=int, default=None,
                    help="override the workload's token count T (e.g. the small-batch sweep)")
    ap.add_argument("--bwd-shape", default=None,
                    help="T,d,E,k,d_ff of the forward + backward timing (profiling captures)")
    ap.add_argument("--no-backward", action="store_true",
                    help="skip the forward + backward timing of the fwd_bwd workload")
    ap.add_argument("--probe-dram", action="store_true",
                    help="print the per-SM DRAM read rate by load path and SM count, then exit")
    args = ap.parse_args()
    if args.probe_dram:
        return probe_dram()
    if args.warmup < 3:
        args.warmup = 3
    if args.shape:
        T, d, E, k, dff = (int(v) for v in args.shape.split(","))
        w = moe_synth.custom(T, d, E, k, dff, seed=1003, zipf_s=1.2, name="custom")
    else:
        w = moe_synth.by_name(args.workload)
    if args.tokens is not None:
        import dataclasses
        w = dataclasses.replace(w, T=args.tokens)
    if args.impl == "reference":
        return bench_reference(args, w)
    return bench_native(args, w)


if __name__ == "__main__":
    sys.exit(main())
