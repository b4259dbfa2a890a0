"""Benchmark of the NVFP4 W4A4 + RAC MoE hot path on GB300.

One step = one rollout MoE layer forward of the prefill workload (16384 tokens,
hidden 4096, 128 experts top-8 with Zipf(1.1) routing, intermediate 1536,
SwiGLU, RAC k = 128 on both projections): route -> amax -> quantize x with its
residual, dispatched to routed rows -> clear padding -> W4A4+RAC gate_up GEMM
with fused SwiGLU and amax -> quantize h -> W4A4+RAC down GEMM -> combine.
The metric is the GEMM work of the step (FP4 + RAC BF16 FLOPs) per second.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  With --impl reference the CPU oracle is
timed on a bounded sample of the same workload on this host's cores.
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
sys.path.insert(0, ROOT)

METRIC = "W4A4+RAC MoE GEMM TFLOPS (% FP4 peak); quantize GB/s (% HBM)"
WORKLOAD = 5
NOMINAL_FP4_OVER_BF16 = 13.5 / 2.25  # dense tensor-core ratio, nominal


# DRAM bytes (read + write) of one gate_up GEMM launch at this workload's launch shape, from
# one ncu capture of the gemm13_moe profile case, valid only for the kernel
# sources it was taken on (common.cuh, gemm_common.cuh, gemm_single.cu): reported as null
# once they change.
GATE_UP_TRAFFIC = {"bytes": 1362283776 + 414498816,
                   "sources_sha256": "c34e61804bcabb1c549cd4e6cc5b1632d45941c6c6710f1d08c5055407934a1b"}


def gate_up_traffic():
    import hashlib

    h = hashlib.sha256()
    for f in ("common.cuh", "gemm_common.cuh", "gemm_single.cu"):
        with open(os.path.join(ROOT, "nvfp4_precision_moe_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return GATE_UP_TRAFFIC["bytes"] if h.hexdigest() == GATE_UP_TRAFFIC["sources_sha256"] else None


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=d["hbm_gbs"], bf16=d["bf16_tflops"], bf16_sus=d.get("bf16_tflops_sustained"),
                    src="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q, "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 7:
                continue
            try:
                sm.append(float(f[0]))
                mx = float(f[1])
            except ValueError:
                continue
            for n, v in zip(names, f[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "samples": len(sm),
                "reasons": sorted(reasons)}


def setup_distributed(n, backend="nccl"):
    rank, world = int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group(backend)
    return rank, world, local


def job_time(ms, world, device=None):
    """The job's timed-region length: the slowest rank's, every rank returning it
    (replicas run the same step independently; the reduction and the barriers are
    the only collectives)."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.barrier()
    return float(t.item())


def job_value(units_per_rank, world, ms_job):
    """Whole-job throughput: the units all ranks processed over the job's time."""
    return world * units_per_rank / (ms_job * 1e-3)


def build_workload(dev, cfg=WORKLOAD):
    """A rollout MoE workload on `dev`: seeded activations, logits and expert
    weights, RAC channel sets calibrated on an independent batch (x: the
    calibration batch; h: the calibration batch's own h), and the layer with
    its weights prepared."""
    import torch

    import nvfp4_precision_moe_gb300 as nv
    import synth

    c = synth.CONFIGS[cfg]
    E, H, I, T, topk, k = c["E"], c["H"], c["I"], c["T"], c["topk"], c["k"]
    x = synth.activations(cfg).to(dev)
    logits = synth.router_logits(cfg).to(dev)
    w13 = torch.empty((E, 2 * I, H), dtype=torch.bfloat16, device=dev)
    wd = torch.empty((E, H, I), dtype=torch.bfloat16, device=dev)
    for e in range(E):
        w13[e].copy_(synth.expert_weight(cfg, e, "w13"))
        wd[e].copy_(synth.expert_weight(cfg, e, "down"))
    # channel calibration (offline, Eq. 23-24) on an independent calibration batch
    xc = synth.activations(cfg, batch=1).to(dev)
    amax = torch.zeros(1, dtype=torch.float32, device=dev)
    nv.nvfp4_amax(xc, amax)
    S13 = torch.empty(k, dtype=torch.int32, device=dev)
    nv.nvfp4_rac_select_channels(xc, amax, k, S13, torch.empty(H, dtype=torch.float64, device=dev))
    # the down projection's channels: calibrate on the calibration batch's h
    g = torch.Generator().manual_seed(5)
    Sd0 = torch.sort(torch.randperm(I, generator=g)[:k]).values.to(torch.int32).to(dev)
    cal = nv.RolloutMoE(w13, wd, S13, Sd0, topk, T)
    cal.forward(xc, synth.router_logits(cfg).roll(1, 0).to(dev))
    hmax = torch.zeros(1, dtype=torch.float32, device=dev)
    nv.nvfp4_amax(cal.h, hmax)
    Sd = torch.empty(k, dtype=torch.int32, device=dev)
    nv.nvfp4_rac_select_channels(cal.h, hmax, k, Sd, torch.empty(I, dtype=torch.float64, device=dev))
    del cal, xc
    layer = nv.RolloutMoE(w13, wd, S13, Sd, topk, T)  # weight prep (A7), once per weight update
    torch.cuda.synchronize()
    return c, layer, x, logits, (w13, wd)


def run_ours(args):
    import torch

    rank, world, local = setup_distributed(args.gpus)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    import nvfp4_precision_moe_gb300 as nv
    import synth

    nv.load(build=True)
    c, layer, x, logits, w_bf16 = build_workload(dev)
    T, H, E, I, k = c["T"], c["H"], c["E"], c["I"], c["k"]
    f4, fb = synth.flops_moe(WORKLOAD)
    f4_13 = 2 * T * c["topk"] * 2 * I * H
    fb_13 = 2 * T * c["topk"] * 2 * I * k
    stream = torch.cuda.current_stream()

    # per-stage events of one step (all launches are on `stream`)
    nstage = 9

    def step(ev=None):
        layer.forward(x, logits, mark=(lambda i: ev[i].record(stream)) if ev is not None else None)

    launches_per_step = layer.LAUNCHES
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert int(layer.dev_status.item()) == 0, nv.STATUS.get(int(layer.dev_status.item()))

    # the timed step: the layer forward replayed as one CUDA graph (the same launches as
    # an eager forward, issued at once), on inputs resident in HBM
    graph, g_out = layer.capture(x, logits)
    for _ in range(args.warmup):
        graph.replay()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ else local)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.15)
    t0.record(stream)
    for i in range(args.steps):
        graph.replay()
    t1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = t0.elapsed_time(t1)
    ms = job_time(ms, world, dev)
    ms_step = ms / args.steps
    assert int(layer.dev_status.item()) == 0
    g_res = g_out.clone()
    assert torch.equal(g_res, layer.forward(x, logits))

    # the stage breakdown: eager forwards with CUDA events between the stages
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nstage)] for _ in range(args.steps)]
    torch.cuda.synchronize()
    for i in range(args.steps):
        step(evs[i])
    torch.cuda.synchronize()
    eager_ms = job_time(evs[0][0].elapsed_time(evs[-1][nstage - 1]), world, dev) / args.steps
    names = ["route", "amax_x_wait", "quantize_x", "clear_padding_wait", "gemm_gate_up", "quantize_h", "gemm_down",
             "combine"]
    stage = {n: statistics.median([evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(args.steps)])
             for j, n in enumerate(names)}
    gemm13_ms = statistics.mean([evs[i][4].elapsed_time(evs[i][5]) for i in range(args.steps)])

    # ---- end to end through host buffers: each step's inputs H2D from pinned
    # memory and its FP32 result D2H, all inside the timed region.  Copies run
    # on two copy streams and are double-buffered against the compute stream:
    # step i+1's inputs upload and step i's result downloads while step i+1 /
    # step i compute, as a serving loop would overlap them.
    xh = x.cpu().pin_memory()
    lh = logits.cpu().pin_memory()
    oh = [torch.empty((T, H), dtype=torch.float32).pin_memory() for _ in range(2)]
    xd = [torch.empty_like(x) for _ in range(2)]
    ld = [torch.empty_like(logits) for _ in range(2)]
    od = [torch.empty((T, H), dtype=torch.float32, device=dev) for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    for i in range(2):
        xd[i].copy_(x)
        ld[i].copy_(logits)
    graphs = [layer.capture(xd[i], ld[i], out=od[i])[0] for i in range(2)]  # one per buffer slot

    def e2e_run(n):
        h2d = [torch.cuda.Event() for _ in range(2)]
        comp = [None, None]
        d2h = [None, None]
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(s_in)
        with torch.cuda.stream(s_in):
            xd[0].copy_(xh, non_blocking=True)
            ld[0].copy_(lh, non_blocking=True)
            h2d[0].record(s_in)
        for i in range(n):
            slot, nxt = i % 2, (i + 1) % 2
            if i + 1 < n:  # upload step i+1's inputs once step i-1 is done with that slot
                if comp[nxt] is not None:
                    s_in.wait_event(comp[nxt])
                with torch.cuda.stream(s_in):
                    xd[nxt].copy_(xh, non_blocking=True)
                    ld[nxt].copy_(lh, non_blocking=True)
                    h2d[nxt] = torch.cuda.Event()
                    h2d[nxt].record(s_in)
            stream.wait_event(h2d[slot])
            if d2h[slot] is not None:  # step i-2's result has left this output buffer
                stream.wait_event(d2h[slot])
            graphs[slot].replay()
            comp[slot] = torch.cuda.Event()
            comp[slot].record(stream)
            s_out.wait_event(comp[slot])
            with torch.cuda.stream(s_out):
                oh[slot].copy_(od[slot], non_blocking=True)
                d2h[slot] = torch.cuda.Event()
                d2h[slot].record(s_out)
        stream.wait_stream(s_out)
        end.record(stream)
        return start, end

    e2e_run(max(2, args.warmup // 2))
    torch.cuda.synchronize()
    e0, e1 = e2e_run(args.steps)
    torch.cuda.synchronize()
    e2e_ms = job_time(e0.elapsed_time(e1), world, dev) / args.steps
    assert int(layer.dev_status.item()) == 0
    assert torch.equal(oh[(args.steps - 1) % 2], layer.forward(x, logits).cpu())
    # the host link's own copy rates on this machine (each copy alone, three times): the e2e step
    # hides its copies only while the FP32 output's download is shorter than the step
    link = {}
    for name, dst, src in (("d2h", oh[0], od[0]), ("h2d", xd[0], xh)):
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        for _ in range(3):
            dst.copy_(src, non_blocking=True)
        c1.record(stream)
        torch.cuda.synchronize()
        link[name + "_gbs"] = round(3 * src.numel() * src.element_size() / (c0.elapsed_time(c1) * 1e6), 1)
    # both directions at once, as the e2e step runs them (a step's output down, the next inputs up)
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    c0.record(stream)
    s_in.wait_stream(stream)
    s_out.wait_stream(stream)
    for _ in range(3):
        with torch.cuda.stream(s_out):
            oh[0].copy_(od[0], non_blocking=True)
        with torch.cuda.stream(s_in):
            xd[0].copy_(xh, non_blocking=True)
            ld[0].copy_(lh, non_blocking=True)
    stream.wait_stream(s_in)
    stream.wait_stream(s_out)
    c1.record(stream)
    torch.cuda.synchronize()
    link["both_ms"] = round(c0.elapsed_time(c1) / 3, 4)  # one step's 142.6 MB up and 268.4 MB down together

    pk = peaks()
    fp4_peak = pk["bf16"] * NOMINAL_FP4_OVER_BF16
    value = job_value(f4 + fb, world, ms_step) / 1e12
    gemm13_tflops = f4_13 / (gemm13_ms * 1e-3) / 1e12
    R = T * c["topk"]
    q_bytes = 2 * T * H + R * (H // 2 + H // 16 + 2 * k)  # read x, write routed codes/scales/residual
    q_gbs = q_bytes / (stage["quantize_x"] * 1e-3) / 1e9
    rows_h = int(layer.route.offsets[-1].item())  # the routed rows up to the last segment's end
    qh_bytes = rows_h * (2 * I + I // 2 + I // 16 + 2 * k)  # read h's routed rows, write codes/scales/residual
    qh_gbs = qh_bytes / (stage["quantize_h"] * 1e-3) / 1e9
    out = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e2m1 (fp32 accum) + bf16 RAC", "data": "synthetic",
        "config": {"workload": "moe_prefill T=16384 H=4096 E=128 top8 zipf1.1 I=1536 k=128",
                   "T": T, "H": H, "E": E, "topk": c["topk"], "I": I, "k": k, "parallelism": "replicas",
                   "l2": "no flush: every step streams ~3 GB, far more than the 129 MB L2",
                   "launch": "each step is one CUDA-graph replay of the layer forward (RolloutMoE.capture)"},
        "fp4_peak_frac_step": round(world * f4 / (ms_step * 1e-3) / 1e12 / fp4_peak, 4),
        "quantize_x": {"gbs": round(q_gbs, 1), "hbm_frac": round(q_gbs / pk["hbm"], 4), "bytes": q_bytes},
        "quantize_h": {"gbs": round(qh_gbs, 1), "hbm_frac": round(qh_gbs / pk["hbm"], 4), "bytes": qh_bytes},
        "stages_ms": {n: round(v, 4) for n, v in stage.items()},
        "stages_what": "eager forwards with CUDA events between the stages: each stage's share of the critical "
                       "path on the layer's stream; the amax of x runs on a side "
                       "stream beside the routing and the padding-row clear beside the quantization of x (the "
                       "*_wait stages are what is left of them)",
        "roofline": {"kernel": "single_gemm_kernel<fp4> (gate_up, SwiGLU)", "bound": "tensor",
                     "achieved": round(gemm13_tflops, 1), "peak": round(fp4_peak, 1), "unit": "TFLOP/s",
                     "frac": round(gemm13_tflops / fp4_peak, 4), "traffic": gate_up_traffic(),
                     "peak_src": "%s bf16 burst x nominal fp4/bf16 ratio 6" % pk["src"]},
        "e2e": {"value": round(world * (f4 + fb) / (e2e_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": int(x.numel() * 2 + logits.numel() * 4),
                "d2h_bytes_per_step": int(T * H * 4),
                "overlap": "double-buffered: step i+1 H2D and step i D2H on copy streams beside step i's compute",
                "link": link},
        "eager": {"ms_per_step": round(eager_ms, 4), "value": round(job_value(f4 + fb, world, eager_ms) / 1e12, 2),
                  "unit": "TFLOP/s", "what": "the same step launched eagerly with CUDA events between its stages "
                                            "(where stages_ms comes from); the timed step replays it as one CUDA graph"},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
    }
    if rank == 0:
        out["decode"] = decode_measure(dev, max(3, min(args.steps, 20)), pk)
        out["quantize_dense"] = quantize_dense_measure(dev, pk)
        out["qat"] = qat_measure(dev, max(3, min(args.steps, 10)))
        out["mismatch"] = mismatch_measure(layer, x, logits, *w_bf16)
        out["cpu_baseline"] = cpu_baseline(seconds=args.cpu_seconds)
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def graph_step_ms(layer, x, logits, steps, stream):
    """The layer step as a CUDA-graph replay (RolloutMoE.capture: the same
    launches, issued at once, no per-stage events): ms per step over `steps`
    replays after three, the replayed output checked against an eager forward."""
    import torch

    graph, out = layer.capture(x, logits)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    for _ in range(steps):
        graph.replay()
    g1.record(stream)
    torch.cuda.synchronize()
    assert int(layer.dev_status.item()) == 0
    got = out.clone()
    assert torch.equal(got, layer.forward(x, logits))
    return g0.elapsed_time(g1) / steps


def decode_measure(dev, steps, pk):
    """The rollout decode workload (2048 tokens top-8 over 64 experts, hidden
    2048, intermediate 768, k = 64; QUADS §4.4.2 Fig. 9a measures rollout
    decode): layer step time and per-stage CUDA events, inputs resident.  The
    two GEMMs are bound by the bytes they move (the weights of all 64 experts
    for about 256 routed rows each), so they are reported as GB/s of those
    algorithmic bytes against the measured HBM bandwidth: weight codes and
    scales, the selected weight columns, the routed A operands (codes, scales,
    residual) and the outputs (h, y), each once."""
    import torch

    import synth

    c, layer, x, logits, _ = build_workload(dev, 3)
    T, H, E, I, k, topk = c["T"], c["H"], c["E"], c["I"], c["k"], c["topk"]
    stream = torch.cuda.current_stream()
    for _ in range(3):
        layer.forward(x, logits)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(9)] for _ in range(steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(steps):
        layer.forward(x, logits, mark=lambda j, i=i: evs[i][j].record(stream))
    t1.record(stream)
    torch.cuda.synchronize()
    assert int(layer.dev_status.item()) == 0
    ms = t0.elapsed_time(t1) / steps
    names = ["route", "amax_x_wait", "quantize_x", "clear_padding_wait", "gemm_gate_up", "quantize_h", "gemm_down",
             "combine"]
    stage = {n: statistics.median([evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(steps)])
             for j, n in enumerate(names)}
    rows = int(layer.route.offsets[-1].item())  # routed rows incl. segment padding
    w_bytes = E * (2 * I * (H // 2 + H // 16 + 2 * k) + H * (I // 2 + I // 16 + 2 * k))
    a_bytes = rows * (H // 2 + H // 16 + 2 * k) + rows * (I // 2 + I // 16 + 2 * k)
    o_bytes = rows * I * 2 + rows * H * 2
    g_bytes = w_bytes + a_bytes + o_bytes
    g_ms = stage["gemm_gate_up"] + stage["gemm_down"]
    f4, fb = synth.flops_moe(3)
    graph_ms = graph_step_ms(layer, x, logits, steps, stream)
    return {"workload": "moe_decode T=2048 H=2048 E=64 top8 I=768 k=64", "ms_per_step": round(ms, 4),
            "tflops": round((f4 + fb) / (ms * 1e-3) / 1e12, 1),
            "graph_ms_per_step": round(graph_ms, 4), "graph_tflops": round((f4 + fb) / (graph_ms * 1e-3) / 1e12, 1),
            "stages_ms": {n: round(v, 4) for n, v in stage.items()},
            "gemm_bytes": g_bytes, "gemm_gbs": round(g_bytes / (g_ms * 1e-3) / 1e9, 1),
            "gemm_hbm_frac": round(g_bytes / (g_ms * 1e-3) / 1e9 / pk["hbm"], 4),
            "what": "both W4A4+RAC GEMMs: weights (codes, scales, selected columns) + routed A operands + "
                    "outputs, once each, over the two GEMMs' CUDA-event time"}


def quantize_dense_measure(dev, pk, reps=20):
    """nvfp4_quantize alone on the dense decode workload's X (256 x 4096
    Student-t with outliers, k = 128 RAC channels: a latency-class launch,
    reported in microseconds) and W (4096 x 4096, no residual: GB/s of read
    2NK + written NK/2 + NK/16 bytes against the measured HBM bandwidth).
    Both fit in L2, so a 512 MB buffer is overwritten between timed launches
    and each launch is timed on its own."""
    import torch

    import nvfp4_precision_moe_gb300 as nv
    import synth

    x = synth.activations(2).to(dev)
    w = synth.dense_weight(2).to(dev)
    M, K = x.shape
    N = w.shape[0]
    xc = synth.activations(2, batch=1).to(dev)
    amax = torch.zeros(1, dtype=torch.float32, device=dev)
    nv.nvfp4_amax(xc, amax)
    S = torch.empty(128, dtype=torch.int32, device=dev)
    nv.nvfp4_rac_select_channels(xc, amax, 128, S, torch.empty(K, dtype=torch.float64, device=dev))
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    res = {}
    for name, t, SS in (("x", x, S), ("w", w, None)):
        rows, cols = t.shape
        am = torch.zeros(1, dtype=torch.float32, device=dev)
        codes = torch.empty((rows, cols // 2), dtype=torch.uint8, device=dev)
        scales = torch.empty(nv.scale_bytes(rows, cols), dtype=torch.uint8, device=dev)
        resid = torch.empty((rows, 128), dtype=torch.bfloat16, device=dev) if SS is not None else None
        nv.nvfp4_amax(t, am)
        ts = {"quantize": [], "amax+quantize": []}
        for r in range(reps + 3):
            for key in ts:
                flush.fill_(r & 255)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                if key == "amax+quantize":
                    nv.nvfp4_amax(t, am)
                nv.nvfp4_quantize(t, am, codes, scales, resid=resid, S=SS)
                e1.record()
                torch.cuda.synchronize()
                if r >= 3:
                    ts[key].append(e0.elapsed_time(e1))
        qb = 2 * rows * cols + rows * cols // 2 + rows * cols // 16 + (2 * rows * 128 if SS is not None else 0)
        med = {kk: statistics.median(v) for kk, v in ts.items()}
        res[name] = {"shape": [rows, cols], "k": 128 if SS is not None else 0,
                     "us": round(med["quantize"] * 1e3, 2), "us_with_amax": round(med["amax+quantize"] * 1e3, 2),
                     "bytes": qb, "gbs": round(qb / (med["quantize"] * 1e-3) / 1e9, 1),
                     "hbm_frac": round(qb / (med["quantize"] * 1e-3) / 1e9 / pk["hbm"], 4)}
    res["l2"] = "a 512 MB buffer is overwritten between timed launches (cold L2)"
    return res


def build_qat_workload(dev):
    """The QAT workload's inputs: 128 experts of random BF16 weights N(0, 0.02)
    drawn on the device (seeded), the workload's seeded activations and logits."""
    import torch

    import synth

    c = synth.CONFIGS[4]
    E, H, I = c["E"], c["H"], c["I"]
    g = torch.Generator(device=dev)
    g.manual_seed(44)
    w13 = torch.empty((E, 2 * I, H), dtype=torch.bfloat16, device=dev)
    wd = torch.empty((E, H, I), dtype=torch.bfloat16, device=dev)
    for e in range(E):
        w13[e].copy_(torch.randn((2 * I, H), device=dev, generator=g) * 0.02)
        wd[e].copy_(torch.randn((H, I), device=dev, generator=g) * 0.02)
    return c, w13, wd, synth.activations(4).to(dev), synth.router_logits(4).to(dev)


def qat_measure(dev, steps):
    """The trainer side at the QAT workload (128 experts, W13 3072x4096 and down
    4096x1536 fake-quantized every step, 4096 tokens top-8 through the BF16
    grouped GEMMs): per-stage CUDA events over `steps` forwards.  Weights are
    random BF16 drawn on the device (values do not change the work)."""
    import torch

    import nvfp4_precision_moe_gb300 as nv

    c, w13, wd, x, logits = build_qat_workload(dev)
    E, H, I, T, topk = c["E"], c["H"], c["I"], c["T"], c["topk"]
    layer = nv.QatMoE(w13, wd, topk, T)
    stream = torch.cuda.current_stream()
    for _ in range(3):
        layer.forward(x, logits)
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(7)] for _ in range(steps)]
    for i in range(steps):
        layer.forward(x, logits, mark=lambda j, i=i: ev[i][j].record(stream))
    torch.cuda.synchronize()
    assert int(layer.dev_status.item()) == 0
    st = lambda a, b: statistics.median([ev[i][a].elapsed_time(ev[i][b]) for i in range(steps)])
    fq_ms, g13_ms, gd_ms, fwd_ms = st(0, 1), st(3, 4), st(4, 5), st(0, 6)
    del layer
    # the training step's backward (QUADS §3.2 Eq. 13): forward with saved pre-activations, then backward
    tl = nv.QatMoE(w13, wd, topk, T, train=True)
    g2 = torch.Generator(device=dev)
    g2.manual_seed(45)
    dout = torch.randn((T, H), device=dev, generator=g2)
    for _ in range(2):
        tl.forward(x, logits)
        tl.backward(dout)
    torch.cuda.synchronize()
    bev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    sev = [[torch.cuda.Event(enable_timing=True) for _ in range(7)] for _ in range(steps)]
    for i in range(steps):
        bev[i][0].record(stream)
        tl.forward(x, logits)
        bev[i][1].record(stream)
        tl.backward(dout, mark=lambda k, i=i: sev[i][k].record(stream))
        bev[i][2].record(stream)
    torch.cuda.synchronize()
    assert int(tl.dev_status.item()) == 0
    tfwd = statistics.median([bev[i][0].elapsed_time(bev[i][1]) for i in range(steps)])
    tbwd = statistics.median([bev[i][1].elapsed_time(bev[i][2]) for i in range(steps)])
    bnames = ["combine_backward", "dgrad_down_swiglu_bwd", "wgrad_down", "dgrad_gate_up", "wgrad_gate_up", "dx_combine"]
    bstages = {n: round(statistics.median(sev[i][k].elapsed_time(sev[i][k + 1]) for i in range(steps)), 4)
               for k, n in enumerate(bnames)}
    # the same step with every BF16 GEMM on each pipeline (the choice is process-wide)
    by_pipe = {}
    for pname, which in (("single", nv.NVFP4_PIPELINE_SINGLE), ("pair", nv.NVFP4_PIPELINE_PAIR)):
        prev = nv.nvfp4_gemm_pipeline(which)
        try:
            pev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
            tl.forward(x, logits)
            tl.backward(dout)
            for i in range(steps):
                pev[i][0].record(stream)
                tl.forward(x, logits)
                pev[i][1].record(stream)
                tl.backward(dout)
                pev[i][2].record(stream)
            torch.cuda.synchronize()
        finally:
            nv.nvfp4_gemm_pipeline(prev)
        by_pipe[pname] = {"forward_ms": round(statistics.median(pev[i][0].elapsed_time(pev[i][1]) for i in range(steps)), 4),
                          "backward_ms": round(statistics.median(pev[i][1].elapsed_time(pev[i][2]) for i in range(steps)), 4)}
    # the wgrad launches alone: dW_down then dW_13, on the buffers the backward left
    r = tl.route
    wev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    wev[0].record(stream)
    for _ in range(5):
        nv.nvfp4_bf16_grouped_gemm_wgrad_rows(tl.dy, tl.h, r.offsets, E, tl.dwd, dev_status=tl.dev_status)
    wev[1].record(stream)
    for _ in range(5):
        nv.nvfp4_bf16_grouped_gemm_wgrad_rows(tl.dgu, tl.xr, r.offsets, E, tl.dw13, dev_status=tl.dev_status)
    wev[2].record(stream)
    torch.cuda.synchronize()
    wd_ms, w13_ms = wev[0].elapsed_time(wev[1]) / 5, wev[1].elapsed_time(wev[2]) / 5
    del tl
    n_w = E * (2 * I * H + H * I)
    fq_bytes = 4 * n_w  # read and write every BF16 weight once
    # the weight gradients write FP32 [E, 2I, H] and [E, H, I] and read the routed rows once
    used = int(r.offsets[-1].item())
    wg_bytes = 4 * n_w + 2 * used * (H + I + 2 * I + H)
    R = T * topk
    fl13, fld = 2 * R * 2 * I * H, 2 * R * H * I
    pk = peaks()
    return {"workload": "qat E=128 W13 3072x4096 down 4096x1536 fake-quantized per step, T=4096 top8",
            "fake_quant": {"ms": round(fq_ms, 4), "gbs": round(fq_bytes / (fq_ms * 1e-3) / 1e9, 1),
                           "hbm_frac": round(fq_bytes / (fq_ms * 1e-3) / 1e9 / pk["hbm"], 4), "bytes": fq_bytes},
            "bf16_gemm": {"gate_up_ms": round(g13_ms, 4), "down_ms": round(gd_ms, 4),
                          "tflops": round((fl13 + fld) / ((g13_ms + gd_ms) * 1e-3) / 1e12, 1),
                          "bf16_frac": round((fl13 + fld) / ((g13_ms + gd_ms) * 1e-3) / 1e12 / pk["bf16"], 4)},
            "forward_ms": round(fwd_ms, 4),
            "train_step": {"forward_ms": round(tfwd, 4), "backward_ms": round(tbwd, 4), "backward_stages_ms": bstages,
                           "by_pipeline": by_pipe,
                           "wgrad_down_ms": round(wd_ms, 4), "wgrad_gate_up_ms": round(w13_ms, 4),
                           "wgrad_tflops": round((fld + fl13) / ((wd_ms + w13_ms) * 1e-3) / 1e12, 1),
                           "wgrad_bf16_frac": round((fld + fl13) / ((wd_ms + w13_ms) * 1e-3) / 1e12 / pk["bf16"], 4),
                           "wgrad_gbs": round(wg_bytes / ((wd_ms + w13_ms) * 1e-3) / 1e9, 1),
                           "wgrad_hbm_frac": round(wg_bytes / ((wd_ms + w13_ms) * 1e-3) / 1e9 / pk["hbm"], 4),
                           "wgrad_bytes": wg_bytes,
                           "what": "QatMoE(train=True): forward keeping the gate/up pre-activations, then the "
                                   "straight-through backward (dX, dW_13, dW_down, the combine weights' gradient); "
                                   "the weight gradients are bound by their FP32 writes (wgrad_hbm_frac)"}}


def mismatch_measure(layer, x, logits, w13, wd):
    """Layer-wise forward mismatch of QUADS §3.1 Eq. 11 (Fig. 4b) on the
    benchmark's own batch and weights, ||Y_rollout - Y_trainer|| / ||Y_trainer||
    (norms by nvfp4_mismatch_norm in binary64), for the W4A4 rollout against
    the BF16 trainer (no QAT), against the W4A16 QAT trainer, the W4A4 + RAC
    rollout (`layer`) against the QAT trainer, and the W4A4 rollout against
    the symmetric W4A4 QAT trainer (§4.3.1 Fig. 7).  `eta` repeats them with
    the rollout's input drifted by ~2^-10 relative (Eq. 8), next to the
    drift's own effect on the BF16 layer."""
    import torch

    import nvfp4_precision_moe_gb300 as nv
    import synth

    T = x.shape[0]
    xe = synth.engine_drift(x.cpu(), 2.0 ** -10, 1).to(x.device)
    outs = {"w4a4_rac": layer.forward(x, logits).clone(), "w4a4_rac@eta": layer.forward(xe, logits).clone()}
    step_ms = {}
    for name, mk, drift in [("w4a4", lambda: nv.RolloutMoE(w13, wd, None, None, layer.topk, T), True),
                            ("w16a16", lambda: nv.QatMoE(w13, wd, layer.topk, T, fake=False), True),
                            ("w4a16", lambda: nv.QatMoE(w13, wd, layer.topk, T, fake=True), False),
                            ("w4a4_sym", lambda: nv.QatMoE(w13, wd, layer.topk, T, sym=True), False),
                            ("w4a4_rac_fp4", lambda: nv.RolloutMoE(w13, wd, layer.S13, layer.Sd, layer.topk, T,
                                                                   resid_fp4=True), False),
                            ("w4a4_rac_online", lambda: nv.RolloutMoE(w13, wd, layer.S13, layer.Sd, layer.topk, T,
                                                                      online=True), False)]:
        lay = mk()
        outs[name] = lay.forward(x, logits).clone()
        if name in ("w4a4_rac_fp4", "w4a4_rac_online"):  # the variant's step time, inputs resident
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
            for _ in range(3):
                lay.forward(x, logits)
            ev[0].record()
            for _ in range(10):
                lay.forward(x, logits)
            ev[1].record()
            torch.cuda.synchronize()
            step_ms[name] = round(ev[0].elapsed_time(ev[1]) / 10, 4)
            if name == "w4a4_rac_online":  # its stages: the selection passes sit in amax_x and quantize_h
                sev = [[torch.cuda.Event(enable_timing=True) for _ in range(9)] for _ in range(5)]
                for i in range(5):
                    lay.forward(x, logits, mark=lambda k, i=i: sev[i][k].record())
                torch.cuda.synchronize()
                names = ["route", "amax_x+select_x_wait", "quantize_x", "clear_padding_wait", "gemm_gate_up",
                         "select_h+quantize_h", "gemm_down", "combine"]
                step_ms["online_stages"] = {n: round(statistics.median(sev[i][k].elapsed_time(sev[i][k + 1])
                                                                      for i in range(5)), 4)
                                            for k, n in enumerate(names)}
        if drift:
            outs[name + "@eta"] = lay.forward(xe, logits).clone()
        torch.cuda.synchronize()
        assert int(lay.dev_status.item()) == 0
        del lay
    acc = torch.zeros(2, dtype=torch.float64, device=x.device)

    def rel(a, b):
        d, n = nv.nvfp4_mismatch_norm(outs[a], outs[b], acc)
        return round(d / n, 6)

    res = {"no_qat": rel("w4a4", "w16a16"), "qat": rel("w4a4", "w4a16"), "qat_rac": rel("w4a4_rac", "w4a16"),
           "qat_rac_fp4": rel("w4a4_rac_fp4", "w4a16"), "qat_rac_online": rel("w4a4_rac_online", "w4a16"),
           "variant_ms_per_step": {"rac_fp4_residual": step_ms["w4a4_rac_fp4"],
                                   "rac_online_selection": step_ms["w4a4_rac_online"],
                                   "rac_online_selection_stages": step_ms["online_stages"]},
           "sym_qat": rel("w4a4", "w4a4_sym"),
           "eta": {"rel": 2.0 ** -10, "bf16": rel("w16a16@eta", "w16a16"), "no_qat": rel("w4a4@eta", "w16a16"),
                   "qat": rel("w4a4@eta", "w4a16"), "qat_rac": rel("w4a4_rac@eta", "w4a16"),
                   "sym_qat": rel("w4a4@eta", "w4a4_sym")}}
    res["what"] = ("||Y_infer - Y_train|| / ||Y_train||: W4A4 vs BF16, W4A4 vs W4A16 QAT, W4A4+RAC vs W4A16 "
                   "QAT (BF16 residual; FP4 residual of the literal Eq. 21; channels chosen online per forward, Eq. 23-24), "
                   "W4A4 vs symmetric W4A4 QAT; eta: "
                   "the rollout's input drifted (bf16: the drift alone)")
    return res


def _oracle_worker(rows, barrier, in_q, out_q):
    """One host core of the CPU baseline: prepares one expert's weights with the
    plain C oracle (not timed), then for every request runs batches of `rows`
    routed rows of that expert through both W4A4+RAC projections for the
    requested seconds (one batch when 0), starting with the other workers."""
    import numpy as np

    import oracle
    import synth

    c = synth.CONFIGS[WORKLOAD]
    H, I, k = c["H"], c["I"], c["k"]
    x = synth.u16(synth.activations(WORKLOAD, rows=rows))
    S13 = np.arange(0, H, H // k, dtype=np.int32)
    Sd = np.arange(0, I, I // k, dtype=np.int32)
    cw, sw, _, gw = oracle.quantize(synth.u16(synth.expert_weight(WORKLOAD, 0, "w13")))
    cd, sd, _, gd = oracle.quantize(synth.u16(synth.expert_weight(WORKLOAD, 0, "down")))
    wq13, wqd = oracle.dequantize_exact(cw, sw, gw), oracle.dequantize_exact(cd, sd, gd)
    while True:
        seconds = in_q.get()
        if seconds is None:
            return
        barrier.wait()
        t_start = time.perf_counter()
        batches = 0
        while batches == 0 or time.perf_counter() - t_start < seconds:
            ca, sa, ra, ga = oracle.quantize(x, S=S13)
            y = oracle.rac_gemm(oracle.dequantize_exact(ca, sa, ga), wq13, ra, S13, ga)
            h = oracle.bf16_round(oracle.swiglu(y, I).astype(np.float32))
            ch, sh, rh, gh = oracle.quantize(h, S=Sd)
            oracle.rac_gemm(oracle.dequantize_exact(ch, sh, gh), wqd, rh, Sd, gh)
            batches += 1
        dt = time.perf_counter() - t_start
        out_q.put((batches * (2 * rows * (2 * I) * (H + k) + 2 * rows * H * (I + k)), dt, batches))


class OraclePool:
    """The CPU baseline's processes: one per host core (the oracle is single-
    threaded), spawned -- never forked from a process that holds a CUDA
    context -- and kept for several runs."""

    def __init__(self, rows, workers=None):
        import multiprocessing as mp

        from oracle.build import build_oracle

        build_oracle()
        self.rows = rows
        self.cores = os.cpu_count() or 1
        self.workers = workers or self.cores
        ctx = mp.get_context("spawn")
        self.barrier = ctx.Barrier(self.workers)
        self.out_q = ctx.Queue()
        self.in_q = [ctx.Queue() for _ in range(self.workers)]
        self.procs = [ctx.Process(target=_oracle_worker, args=(rows, self.barrier, q, self.out_q), daemon=True)
                      for q in self.in_q]
        for p in self.procs:
            p.start()

    def run(self, seconds):
        """TFLOP/s of GEMM work summed over the processes, all running at once."""
        for q in self.in_q:
            q.put(seconds)
        res = [self.out_q.get() for _ in self.procs]
        rate = sum(fl / dt for fl, dt, _ in res)
        batches = sum(b for _, _, b in res)
        dt = max(dt for _, dt, _ in res)
        return {"value": round(rate / 1e12, 6), "unit": "TFLOP/s", "cores": self.workers,
                "host_cores": self.cores, "kind": "oracle",
                "sample": "%d processes x batches of %d routed rows of one expert (%d batches in all, %.2f s): "
                          "quantize x, W4A4+RAC gate_up, SwiGLU, quantize h, W4A4+RAC down; plain C oracle, "
                          "one thread per process" % (self.workers, self.rows, batches, dt)}

    def close(self):
        for q in self.in_q:
            q.put(None)
        for p in self.procs:
            p.join()


def cpu_baseline(seconds=10.0, rows=64):
    """The oracle as it stands, timed on every host core at once on a bounded
    sample of the workload (see OraclePool)."""
    t_start = time.perf_counter()
    pool = OraclePool(rows)
    try:
        out = pool.run(seconds)
    finally:
        pool.close()
    out["seconds"] = round(time.perf_counter() - t_start, 2)
    return out


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    vals = []
    pool = OraclePool(32)
    try:
        for _ in range(args.warmup):
            pool.run(0)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            vals.append(pool.run(0))
        wall = time.perf_counter() - t0
    finally:
        pool.close()
    v = statistics.median(x["value"] for x in vals)
    out = {"impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s", "n_gpus": args.gpus,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(wall / args.steps * 1e3, 2),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)",
           "data": "synthetic",
           "config": {"workload": "moe_prefill T=16384 H=4096 E=128 top8 zipf1.1 I=1536 k=128",
                      "sample": "32 routed rows of one expert per process per step (the CPU oracle, one "
                                "process per host core)"},
           "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": vals[0]["cores"],
                            "host_cores": vals[0]["host_cores"], "kind": "oracle", "sample": vals[0]["sample"]},
           "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def run_profile_case(args):
    """A single kernel on a reduced case sized for ncu (inputs above L2, a few
    hundred MB in all): `gemm13` (gate_up W4A4+RAC GEMM with SwiGLU, 32
    experts x 512 rows, N=3072, K=4096, k=128), `gemm_down` (N=4096, K=1536),
    `gemm13_moe` / `gemm_down_moe` (the same GEMMs at the prefill layer's own
    launch shape: 128 experts, segments of the Zipf routing, about 2 GB),
    `quantize_x` (16384 x 4096 scatter-quantize, top-8), `quantize_h`
    (147456 x 1536, k=128), `combine` (16384 tokens x 8 x 4096), `bf16_gemm`
    (QAT gate_up, BF16, same shape as gemm13), `wgrad` (the training step's dW_13 at the QAT
    shapes for 16 experts x 256 rows, FP32 output, transposed operands), `wgrad_rows` (the same
    from the routed rows as stored), `dgrad` (the input gradient with W13_hat as stored),
    `fake_quant` / `fake_quant_down` (the QAT workload's W13 / down weights), `train_step` (the
    QAT workload's training step: the forward keeping the pre-activations, then the backward; a
    dozen launches, for a launch list).  Runs the case `--steps` times."""
    import torch

    import nvfp4_precision_moe_gb300 as nv

    nv.load(build=True)
    nv.nvfp4_gemm_pipeline({"auto": 0, "single": 1, "pair": 2}[args.pipeline])
    dev = torch.device("cuda", 0)
    g = torch.Generator(device=dev)
    g.manual_seed(7)
    E, per = 32, 512
    rows = E * per
    offsets = torch.arange(0, rows + 1, per, dtype=torch.int32, device=dev)
    case = args.profile_case
    if case in ("gemm13_moe", "gemm_down_moe"):
        # the prefill layer's own launch shape: 128 experts, the Zipf routing's padded segments
        import synth

        c = synth.CONFIGS[WORKLOAD]
        T, E, topk = c["T"], c["E"], c["topk"]
        rows = nv.rows_capacity(T, topk, E)
        logits = synth.router_logits(WORKLOAD).to(dev)
        ids = torch.empty((T, topk), dtype=torch.int32, device=dev)
        rw = torch.empty((T, topk), dtype=torch.float32, device=dev)
        counts = torch.empty(E, dtype=torch.int32, device=dev)
        offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
        dst = torch.empty((T, topk), dtype=torch.int32, device=dev)
        nv.nvfp4_route_topk(logits, topk, ids, rw, counts, offsets, dst)
        case = case.replace("_moe", "")
    if case in ("gemm13", "gemm_down"):
        N, K = (3072, 4096) if case == "gemm13" else (4096, 1536)
        k = 128
        a = torch.randint(0, 256, (rows, K // 2), dtype=torch.uint8, device=dev, generator=g)
        a_s = torch.randint(0x28, 0x40, (nv.scale_bytes(rows, K),), dtype=torch.uint8, device=dev, generator=g)
        r = (torch.randn((rows, k), device=dev, generator=g) * 0.1).to(torch.bfloat16)
        w = torch.randint(0, 256, (E, N, K // 2), dtype=torch.uint8, device=dev, generator=g)
        w_s = torch.randint(0x28, 0x40, (E * nv.scale_bytes(N, K),), dtype=torch.uint8, device=dev,
                            generator=g)
        sel = torch.randn((E, N, k), device=dev, generator=g).to(torch.bfloat16)
        gs_a = torch.full((1,), 0.01, device=dev)
        gs_w = torch.full((E,), 0.001, device=dev)
        swi = case == "gemm13"
        y = torch.empty((rows, N // 2 if swi else N), dtype=torch.bfloat16, device=dev)
        amax = torch.zeros(1, device=dev)
        fn = lambda: nv.nvfp4_w4a4_rac_grouped_gemm(
            a, a_s, r, gs_a, w, w_s, gs_w, sel, k, offsets, E, N, K, y,
            epilogue=nv.NVFP4_EPI_SWIGLU if swi else nv.NVFP4_EPI_NONE, out_dtype=nv.NVFP4_OUT_BF16,
            amax_out=amax if swi else None)
        flops = 2 * int(offsets[-1].item()) * N * K
    elif case == "bf16_gemm":
        N, K = 3072, 4096
        x = torch.randn((rows, K), device=dev, generator=g).to(torch.bfloat16)
        w = (torch.randn((E, N, K), device=dev, generator=g) * 0.02).to(torch.bfloat16)
        y = torch.empty((rows, N // 2), dtype=torch.bfloat16, device=dev)
        fn = lambda: nv.nvfp4_bf16_grouped_gemm(x, w, offsets, E, N, K, y, out_dtype=nv.NVFP4_OUT_BF16,
                                                epilogue=nv.NVFP4_EPI_SWIGLU)
        flops = 2 * rows * N * K
    elif case == "wgrad":
        # the training step's weight gradient dW_13 at the QAT shapes, 16 experts x 256 routed rows:
        # a_t = d(gate|up)^T [3072, R], b_t = x_routed^T [4096, R], FP32 output [16, 3072, 4096]
        E, per, M, N = 16, 256, 3072, 4096
        R = E * per
        offsets = torch.arange(0, R + 1, per, dtype=torch.int32, device=dev)
        a_t = torch.randn((M, R), device=dev, generator=g).to(torch.bfloat16)
        b_t = torch.randn((N, R), device=dev, generator=g).to(torch.bfloat16)
        dw = torch.empty((E, M, N), dtype=torch.float32, device=dev)
        fn = lambda: nv.nvfp4_bf16_grouped_gemm_wgrad(a_t, b_t, offsets, E, dw)
        flops = 2 * R * M * N
    elif case in ("wgrad_rows", "dgrad"):
        # the same dW_13 from the routed rows as stored (a = d(gate|up) [R, 3072], b = x_routed
        # [R, 4096]); or the input gradient dx = d(gate|up) . W13_hat with W13_hat [16, 3072, 4096] as stored
        E, per, M, N = 16, 256, 3072, 4096
        R = E * per
        offsets = torch.arange(0, R + 1, per, dtype=torch.int32, device=dev)
        a = torch.randn((R, M), device=dev, generator=g).to(torch.bfloat16)
        if case == "wgrad_rows":
            b = torch.randn((R, N), device=dev, generator=g).to(torch.bfloat16)
            dw = torch.empty((E, M, N), dtype=torch.float32, device=dev)
            fn = lambda: nv.nvfp4_bf16_grouped_gemm_wgrad_rows(a, b, offsets, E, dw)
        else:
            w = (torch.randn((E, M, N), device=dev, generator=g) * 0.02).to(torch.bfloat16)
            y = torch.empty((R, N), dtype=torch.bfloat16, device=dev)
            fn = lambda: nv.nvfp4_bf16_grouped_gemm_dgrad(a, w, offsets, E, N, M, y, out_dtype=nv.NVFP4_OUT_BF16)
        flops = 2 * R * M * N
    elif case in ("fake_quant", "fake_quant_down"):
        # the QAT workload's W13 fake-quant: 128 experts x 3072 x 4096 BF16 (3.2 GB read, 3.2 GB
        # written), or its down projection's: 128 x 4096 x 1536
        E = int(os.environ.get("NVFP4_PROFILE_E", "128"))
        N, K = (3072, 4096) if case == "fake_quant" else (4096, 1536)
        w = (torch.randn((E, N, K), device=dev, generator=g) * 0.02).to(torch.bfloat16)
        w_hat = torch.empty_like(w)
        ws = torch.zeros(2 * E + 1, dtype=torch.float32, device=dev)
        gsw = torch.empty(E, dtype=torch.float32, device=dev)
        fn = lambda: nv.nvfp4_fake_quant(w, w_hat, ws, gs_out=gsw)
        flops = 0
    elif case == "quantize_x_syn":
        # a synthetic stand-in for ncu: 16384 x 4096 dispatched to 8 routed rows each (a random
        # permutation of the rows), k = 128 channels clustered in the first 512-element segment
        T, H, topk, k = 16384, 4096, 8, 128
        x = torch.randn((T, H), device=dev, generator=g).to(torch.bfloat16)
        cap = T * topk
        dst = torch.randperm(cap, device=dev, generator=g).to(torch.int32).view(T, topk)
        codes = torch.empty((cap, H // 2), dtype=torch.uint8, device=dev)
        scales = torch.empty(nv.scale_bytes(cap, H), dtype=torch.uint8, device=dev)
        resid = torch.empty((cap, k), dtype=torch.bfloat16, device=dev)
        S = torch.arange(k, dtype=torch.int32, device=dev)
        amax = torch.zeros(1, device=dev)
        nv.nvfp4_amax(x, amax)
        fn = lambda: nv.nvfp4_quantize(x, amax, codes, scales, resid=resid, S=S, dst_row=dst, fanout=topk,
                                       rows_out=cap)
        flops = 0
    elif case == "quantize_h_syn":
        # a synthetic stand-in for ncu (few launches before it): 147456 x 1536, the k = 128
        # selected channels clustered in the first 512-element segment
        rows, I, k = 147456, 1536, 128
        x = (torch.randn((rows, I), device=dev, generator=g) * 0.1).to(torch.bfloat16)
        codes = torch.empty((rows, I // 2), dtype=torch.uint8, device=dev)
        scales = torch.empty(nv.scale_bytes(rows, I), dtype=torch.uint8, device=dev)
        resid = torch.empty((rows, k), dtype=torch.bfloat16, device=dev)
        S = torch.arange(k, dtype=torch.int32, device=dev)
        amax = torch.zeros(1, device=dev)
        nv.nvfp4_amax(x, amax)
        fn = lambda: nv.nvfp4_quantize(x, amax, codes, scales, resid=resid, S=S)
        flops = 0
    elif case in ("quantize_x", "quantize_h"):
        # the layer's own launches: the prefill workload's x dispatched to its routed rows with the
        # calibrated S13, or the forward's h with the calibrated S_down
        c, layer, x, logits, _ = build_workload(dev)
        layer.forward(x, logits)
        torch.cuda.synchronize()
        r, xa, ha = layer.route, layer.xa, layer.ha
        if case == "quantize_x":
            fn = lambda: nv.nvfp4_quantize(x, xa.amax, xa.codes, xa.scales, resid=xa.resid, S=layer.S13,
                                           gs_out=xa.gs, dst_row=r.dst_row, fanout=layer.topk,
                                           rows_out=layer.rows_cap)
        else:
            fn = lambda: nv.nvfp4_quantize(layer.h, ha.amax, ha.codes, ha.scales, resid=ha.resid, S=layer.Sd,
                                           gs_out=ha.gs)
        flops = 0
    elif case in ("gather_w13", "gather_down"):
        # the online mode's re-gather of the selected weight columns, k = 128, from packed weights of the
        # prefill shapes: W13 128 x 3072 x 4096 or down 128 x 4096 x 1536
        E, N, K, k = (128, 3072, 4096, 128) if case == "gather_w13" else (128, 4096, 1536, 128)
        codes = torch.randint(0, 256, (E, N, K // 2), dtype=torch.uint8, device=dev, generator=g)
        scales = torch.randint(0x28, 0x40, (E * nv.scale_bytes(N, K),), dtype=torch.uint8, device=dev, generator=g)
        S = torch.sort(torch.randperm(K, device=dev, generator=g)[:k])[0].to(torch.int32)
        wsel = torch.empty((E, N, k), dtype=torch.bfloat16, device=dev)
        fn = lambda: nv.nvfp4_gather_selected_weights(codes, scales, E, N, K, S, wsel)
        flops = 0
    elif case == "online_step":
        # the prefill layer forward with the channel sets chosen online (QUADS §3.3 Eq. 23-24)
        c, layer, x, logits, w = build_workload(dev)
        lay = nv.RolloutMoE(w[0], w[1], layer.S13, layer.Sd, layer.topk, c["T"], online=True)
        del layer
        fn = lambda: lay.forward(x, logits)
        flops = 0
    elif case == "train_step":
        c, w13, wd, x, logits = build_qat_workload(dev)
        tl = nv.QatMoE(w13, wd, c["topk"], c["T"], train=True)
        dout = torch.randn((c["T"], c["H"]), device=dev, generator=g)

        def fn():
            tl.forward(x, logits)
            tl.backward(dout)

        flops = 0
        # launches from here on form the profiler range (ncu --profile-from-start off)
        torch.cuda.synchronize()
        torch.cuda.profiler.start()
    elif case == "combine":
        T, topk, H = 16384, 8, 4096
        rows = T * topk
        y = (torch.randn((rows, H), device=dev, generator=g)).to(torch.bfloat16)
        dst = torch.randperm(rows, device=dev, generator=g).to(torch.int32).view(T, topk)
        w = torch.rand((T, topk), device=dev, generator=g)
        out = torch.empty((T, H), dtype=torch.float32, device=dev)
        fn = lambda: nv.nvfp4_moe_combine(y, dst, w, topk, out)
        flops = 0
    else:
        raise SystemExit("unknown --profile-case " + case)
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(args.steps):
        fn()
    t1.record()
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / args.steps
    if case == "train_step":
        torch.cuda.profiler.stop()
    print(json.dumps({"profile_case": case, "ms": round(ms, 4),
                      "tflops": round(flops / ms / 1e9, 1) if flops else None}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--profile-case", default=None,
                    help="run one kernel on a reduced case for ncu: gemm13, gemm_down, quantize_x, bf16_gemm")
    ap.add_argument("--pipeline", default="auto", choices=["auto", "single", "pair"],
                    help="GEMM pipeline of the profile cases")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.profile_case:
        run_profile_case(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
