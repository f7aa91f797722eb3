#!/usr/bin/env python3
"""Benchmark of the B300 routed-MoE block (libds4g) — one JSON line.

Default workload (config 1): full-depth decode of DeepSeek-V4-Flash MoE
layers — 43 stacked layers, each with 256 routed experts (IQ2_XXS gate/up,
Q2_K down, 78 GB packed in HBM) plus a bf16 shared expert and an fp32 router;
one step = 64 consecutive tokens, each a fresh N(0,1) hidden vector, passed
through rmsnorm -> route -> MoE forward for all 43 layers.  The step is
captured once as a CUDA graph and replayed.  Metric: tokens/s (whole job).

--impl reference times the CPU oracle (plain C, fp64) on a bounded sample of
the same workload on this host's cores.
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

import numpy as np  # noqa: E402

import synth  # noqa: E402

H, F, E, K = 4096, 2048, 256, 6
NLAYER = 43
SEED = 0
CFG = 1
# algorithmic bytes of one token through one layer: 6 selected experts'
# packed gate/up/down + bf16 shared expert + fp32 router (+ activations)
ROUTED_BYTES = 6 * (2 * 2162688 + 2752512)          # 42,467,328
SHARED_BYTES = 3 * F * H * 2                        # 50,331,648
ROUTER_BYTES = E * H * 4                            # 4,194,304
ROUTED_BYTES_Q4 = 6 * 3 * 4718592                   # Q4_K gate/up/down: 84,934,656
Q4_LAYERS = 6                                       # q2-q4 model: the last 6 layers at Q4_K
ACT_BYTES = 2 * H * 4 + E * 4                       # x in, out, bias
LAYER_BYTES = ROUTED_BYTES + SHARED_BYTES + ROUTER_BYTES + ACT_BYTES
LAYER_BYTES_Q4 = ROUTED_BYTES_Q4 + SHARED_BYTES + ROUTER_BYTES + ACT_BYTES
# gate/up launch (dominant kernel): routed gate+up + shared gate+up + x
GATEUP_BYTES = 6 * 2 * 2162688 + 2 * F * H * 2 + H * 4
METRIC = "routed-MoE tokens/s (decode, prefill) and achieved HBM GB/s vs B300 peak"
# decode arithmetic: exact quant codes on fp16 tensor cores against the activation as an fp16 hi + lo
# pair, fp32 scales and accumulation; the shared expert's bf16 weights against a bf16 hi + lo pair
DECODE_DTYPE = "fp16x2-split activations x exact codes -> f32 (shared expert bf16x2-split)"
WORKLOAD = ("config1 full-depth decode: 43 MoE layers x 256 experts (IQ2_XXS gate/up, Q2_K down, "
            "bf16 shared, fp32 router), 1 token at a time, 64 tokens per step")
WORKLOAD_Q2Q4 = ("q2-q4 full-depth decode: 43 MoE layers x 256 experts, layers 0-36 IQ2_XXS gate/up + Q2_K "
                 "down, layers 37-42 Q4_K gate/up/down, bf16 shared, fp32 router, 1 token at a time, "
                 "64 tokens per step")
WORKLOAD_Q4 = ("q4 full-depth decode: 43 MoE layers x 256 experts, Q4_K gate/up/down, bf16 shared, fp32 "
               "router, 1 token at a time, 64 tokens per step")


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6400.0, "fallback"


def traffic_record(kernel):
    """Per-launch DRAM traffic of `kernel` from the committed ncu summary, if
    it was taken on the current source of that kernel (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(kernel)
    if not d:
        return None
    src = os.path.join(ROOT, d["source"])
    h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16] if os.path.exists(src) else None
    return d["bytes_per_launch"] if h == d["source_sha"] else None


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        # the fused decode kernel keeps one CTA on every SM and its CTAs wait
        # on each other: another process's kernels on this GPU would stall it
        # (bounded) and void the timing, so they are recorded and reported
        self.others = []
        try:
            q = subprocess.run(["nvidia-smi", "-i", str(self.index), "--query-compute-apps=pid",
                                "--format=csv,noheader"], capture_output=True, text=True, timeout=30)
            self.others = sorted({int(v) for v in q.stdout.split() if v.isdigit() and int(v) != os.getpid()})
        except (OSError, subprocess.SubprocessError):
            pass
        if self.others:
            print(f"bench: other compute processes on GPU {self.index}: {self.others}", file=sys.stderr)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.samples = []
        if self.proc is None:
            return False
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        for line in out.strip().splitlines():
            parts = [s.strip() for s in line.split(",")]
            if len(parts) >= 7:
                self.samples.append(parts)
        return False

    def summary(self):
        if not getattr(self, "samples", None):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"],
                    "other_gpu_processes": getattr(self, "others", [])}
        sm = [float(s[0]) for s in self.samples if s[0].replace(".", "").isdigit()]
        mx = [float(s[1]) for s in self.samples if s[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in self.samples for i in range(4) if s[3 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.samples), "other_gpu_processes": self.others}


# ------------------------------------------------------------------ our arm
def build_model(dev, nlayer, cfg=CFG, q4_layers=0, zipf=False):
    """nlayer layers of 256 experts generated on the device; the last
    q4_layers of them with Q4_K gate/up/down, the others IQ2_XXS/Q2_K; the
    router bias ~N(0, 0.1^2), or Zipf(1.1)-ranked with zipf=True."""
    import torch
    import bit_quantized_moe_bias_b300 as B
    grid = torch.from_numpy(np.ascontiguousarray(synth.iq2_grid(SEED)).view(np.int64).reshape(256)).to(dev)
    tmp = torch.empty(B.ds4g_packed_size(2, F, H), dtype=torch.uint8, device=dev)
    layers = []
    for l in range(nlayer):
        gut, dt = (2, 2) if l >= nlayer - q4_layers else (0, 1)
        mats = {}
        for kind, qt, rows, cols in ((synth.KIND_GATE, gut, F, H), (synth.KIND_UP, gut, F, H),
                                     (synth.KIND_DOWN, dt, H, F)):
            t = torch.empty(E, B.ds4g_packed_size(qt, rows, cols), dtype=torch.uint8, device=dev)
            for e in range(E):
                synth.gguf_matrix_device(qt, rows, cols, SEED, synth.stream_id(cfg, l, kind, e), tmp.data_ptr(),
                                         torch.cuda.current_stream().cuda_stream)
                B.ds4g_quantize_pack_device(qt, rows, cols, tmp, t[e])
            mats[kind] = t
        shg, shu, shd = synth.shared(SEED, cfg, l)
        sh = [torch.from_numpy(a.view(np.int16)).to(dev) for a in (shg, shu, shd)]
        L = B.MoELayer(mats[synth.KIND_GATE], mats[synth.KIND_UP], mats[synth.KIND_DOWN], *sh,
                       grid if gut == 0 else None, gut, dt)
        R = torch.from_numpy(synth.router(SEED, cfg, l)).to(dev)
        b = torch.from_numpy((synth.bias_zipf if zipf else synth.bias_normal)(SEED, cfg, l)).to(dev)
        layers.append((L, R, b))
    torch.cuda.synchronize()
    return layers


def max_over_ranks(times, world, dev):
    """Element-wise maximum of per-rank timings: the slowest replica sets the
    step time of the whole job (replicas only; no data-path collective)."""
    if world <= 1:
        return list(times)
    import torch
    import torch.distributed as dist
    t = torch.tensor(times, device=dev, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def graph_kernels(graph):
    """Kernel nodes of a captured CUDA graph (captured with keep_graph=True),
    or None if the graph cannot be inspected."""
    try:
        from cuda.bindings import runtime as rt
        g = rt.cudaGraph_t(init_value=graph.raw_cuda_graph())
        err, _, n = rt.cudaGraphGetNodes(g, 0)
        if err != rt.cudaError_t.cudaSuccess:
            return None
        err, nodes, n = rt.cudaGraphGetNodes(g, n)
        if err != rt.cudaError_t.cudaSuccess:
            return None
        kern = 0
        for nd in nodes[:n]:
            err, ty = rt.cudaGraphNodeGetType(nd)
            if err == rt.cudaError_t.cudaSuccess and ty == rt.cudaGraphNodeType.cudaGraphNodeTypeKernel:
                kern += 1
        return kern
    except Exception:   # noqa: BLE001 - an inspection failure only loses the count
        return None


def run_ours(args, rank, world, local_rank):
    import torch
    import bit_quantized_moe_bias_b300 as B
    torch.cuda.set_device(local_rank)
    dev = f"cuda:{local_rank}"
    ntok = args.tokens
    nl = args.layers
    q4 = {"q2-q4": min(Q4_LAYERS, nl), "q4": nl}.get(args.model, 0)
    if q4 and args.decode_path != "fused":
        raise SystemExit("--model q2-q4 / q4 run through the decode stack (--decode-path fused)")
    t_setup = time.time()
    layers = build_model(dev, nl, q4_layers=q4)
    setup_s = time.time() - t_setup
    # per-step inputs: fresh N(0,1) hidden vectors, one per token
    x_host = torch.from_numpy(synth.hidden(SEED + rank, CFG, ntok, layer=999, normalise=False)).pin_memory()
    y_host = torch.empty(ntok, H, dtype=torch.float32).pin_memory()
    x_dev = x_host.to(dev)
    xn = torch.empty(1, H, device=dev)
    act = [torch.empty(1, H, device=dev) for _ in range(2)]
    out_all = torch.empty(ntok, H, device=dev)
    ids = torch.empty(1, K, dtype=torch.int32, device=dev)
    w = torch.empty(1, K, dtype=torch.float32, device=dev)
    rws = B.workspace(B.ds4g_route_workspace(1), dev)
    fws = B.workspace(B.ds4g_forward_workspace(1), dev)
    lws = B.workspace(B.ds4g_decode_stack_workspace() if q4 else B.ds4g_layer_decode_workspace(), dev)
    fused = args.decode_path in ("fused", "layer")
    stacked = args.decode_path == "fused"
    # fused: one launch per layer (IQ2_XXS/Q2_K or Q4_K); split: four
    launches_per_step = ntok * nl * (1 if fused else 4)
    stack = B.DecodeStack([(L.struct, R, b) for L, R, b in layers])
    ids_all = torch.empty(nl, K, dtype=torch.int32, device=dev)
    w_all = torch.empty(nl, K, dtype=torch.float32, device=dev)
    hbuf = torch.empty(2, H, device=dev)

    def step(timing=None):
        for i in range(ntok):
            cur = x_dev[i:i + 1]
            if stacked:
                # one call per token: 43 layer launches, each after the first a
                # programmatic dependent of the one before
                B.ds4g_moe_decode_stack(cur, stack, ids_all, w_all, hbuf, out_all[i], lws)
                continue
            for l, (L, R, b) in enumerate(layers):
                dst = out_all[i:i + 1] if l == nl - 1 else act[l & 1]
                if fused:
                    # one launch: rmsnorm + router + top-6 + routed and shared experts
                    if timing is not None and i < timing[2]:
                        timing[0][l + nl * i].record()
                    B.ds4g_moe_layer_decode(cur, R, b, L.struct, ids, w, dst, lws)
                    if timing is not None and i < timing[2]:
                        timing[1][l + nl * i].record()
                    cur = dst
                    continue
                B.ds4g_rmsnorm(cur, xn)
                B.ds4g_moe_route(xn, R, b, ids, w, rws)
                if args.decode_path == "q8":
                    # int8 activations for the routed gate/up (timed: the whole forward)
                    if timing is not None and i < timing[2]:
                        timing[0][l + nl * i].record()
                    B.ds4g_moe_forward_q8(xn, L.struct, ids, w, dst, fws)
                    if timing is not None and i < timing[2]:
                        timing[1][l + nl * i].record()
                elif timing is not None and i < timing[2]:
                    timing[0][l + nl * i].record()
                    B.ds4g_moe_gate_up(xn, L.struct, ids, w, dst, fws)
                    timing[1][l + nl * i].record()
                    B.ds4g_moe_down(xn, L.struct, ids, w, dst, fws)
                else:
                    B.ds4g_moe_forward(xn, L.struct, ids, w, dst, fws)
                cur = dst

    # eager warm-up (sets kernel attributes, checks status), then capture
    step()
    torch.cuda.synchronize()
    st = B.ds4g_last_error(rws) or B.ds4g_last_error(fws) or B.ds4g_last_error(lws)
    if st:
        raise RuntimeError(f"device status {st} during warm-up")
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    # ---- timed region (device value): K graph replays, inputs resident
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    with ClockSampler(local_rank) as clk:
        ev0.record()
        for _ in range(args.steps):
            graph.replay()
        ev1.record()
        torch.cuda.synchronize()
    barrier()
    dev_s = ev0.elapsed_time(ev1) / 1e3
    # ---- end to end: host inputs copied in, result read back, every step
    barrier()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        x_dev.copy_(x_host, non_blocking=True)
        graph.replay()
        y_host.copy_(out_all, non_blocking=True)
        torch.cuda.synchronize()
    e2e_s = time.perf_counter() - t0
    barrier()
    # ---- roofline of the dominant kernel (gate/up), CUDA events on its stream
    if fused:
        # one kernel per layer: its average duration over the timed graph
        # replays (CUDA events on the replay stream) is the step time divided
        # by the launches; eager per-launch events would include host gaps
        gu_us = dev_s / args.steps / (ntok * nl) * 1e6
    else:
        ntime = min(ntok, 8)
        evs = ([torch.cuda.Event(enable_timing=True) for _ in range(nl * ntime)],
               [torch.cuda.Event(enable_timing=True) for _ in range(nl * ntime)], ntime)
        step(timing=evs)
        torch.cuda.synchronize()
        gu_us = statistics.mean(a.elapsed_time(b) * 1e3 for a, b in zip(evs[0], evs[1]))
    st = B.ds4g_last_error(rws) or B.ds4g_last_error(fws) or B.ds4g_last_error(lws)
    if st:
        raise RuntimeError(f"device status {st} after the timed region")

    dev_s, e2e_s = max_over_ranks([dev_s, e2e_s], world, dev)
    if rank != 0:
        return None
    tokens = ntok * args.steps * world
    value = tokens / dev_s
    hbm, kind = peaks()
    kbytes = LAYER_BYTES if fused else GATEUP_BYTES
    kname = "decode_t1_kernel (whole layer)" if fused else "gateup_decode_kernel"
    if args.decode_path == "q8":
        kbytes = ROUTED_BYTES + SHARED_BYTES + ACT_BYTES
        kname = "ds4g_moe_forward_q8 (gate/up with int8 activations + down; per-slot kernels)"
    token_bytes = (nl - q4) * LAYER_BYTES + q4 * LAYER_BYTES_Q4
    workload = WORKLOAD
    if q4:
        # Q4_K layers in the stack: one fused launch per layer of either type;
        # the figure is the whole step's, layer bytes averaged over the layers
        kbytes = token_bytes // nl
        kname = "decode_t1_kernel (whole stack: %d IQ2_XXS/Q2_K + %d Q4_K layers)" % (nl - q4, q4)
        workload = WORKLOAD_Q4 if q4 == nl else WORKLOAD_Q2Q4
    achieved = kbytes / (gu_us * 1e-6) / 1e9
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(dev_s / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": DECODE_DTYPE, "data": "synthetic",
        "config": {"workload": workload, "layers": nl, "q4_layers": q4, "tokens_per_step": ntok, "global_batch": 1,
                   "seq_len": 1, "parallelism": "replicas" if world > 1 else "single",
                   "l2": f"no flush: each token streams {token_bytes / 1e9:.2f} GB of weights >> 126 MB L2",
                   "weight_gb_per_token": round(token_bytes / 1e9, 4),
                   "achieved_hbm_gbs_block": round(value / world * token_bytes / 1e9, 1),
                   "decode_path": args.decode_path, "setup_s": round(setup_s, 1)},
        "e2e": {"value": round(tokens / e2e_s, 3), "unit": "tokens/s",
                "h2d_bytes_per_step": int(x_host.numel() * 4), "d2h_bytes_per_step": int(y_host.numel() * 4)},
        "roofline": {"bound": "hbm", "kernel": kname, "achieved": round(achieved, 1),
                     "peak": hbm, "peak_kind": kind, "unit": "GB/s", "frac": round(achieved / hbm, 4),
                     "bytes_per_launch": kbytes, "launch_us": round(gu_us, 3),
                     "traffic": None if q4 or args.decode_path == "q8" else traffic_record(
                         "decode_t1_kernel" if fused else "gateup_decode_kernel")},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk.summary(),
    }
    if not args.no_cpu_baseline and not q4:
        line["cpu_baseline"] = cpu_baseline("decode", args.cpu_size or NLAYER, 1)
    return line



# ------------------------------------------------ single-layer workload
S1_CFG, S1_COPIES = 0, 8
S1_WORKLOAD = ("config0 single layer: 1 token through 1 MoE layer x 256 experts (IQ2_XXS gate/up, Q2_K down, "
               "bf16 shared, fp32 router), route + forward in one ds4g_moe_layer_decode call; a step = {ntok} calls, "
               "each on the next of {copies} independent layer copies")


def run_single_layer(args, rank, world, local_rank):
    """One token through one layer per call (rmsnorm + router + top-6 +
    routed and shared experts: ds4g_moe_layer_decode, one launch), a fresh
    N(0,1) token per call, the calls rotating over independent layer copies
    so that every call reads its layer's weights from HBM (the copies
    together are far larger than L2).  The launches are independent (no
    programmatic overlap): each call's time is the single-layer latency."""
    import torch
    import bit_quantized_moe_bias_b300 as B
    torch.cuda.set_device(local_rank)
    dev = f"cuda:{local_rank}"
    ntok, nc = args.tokens, S1_COPIES
    t_setup = time.time()
    layers = build_model(dev, nc, cfg=S1_CFG)
    setup_s = time.time() - t_setup
    x_host = torch.from_numpy(synth.hidden(SEED + rank, S1_CFG, ntok, layer=999, normalise=False)).pin_memory()
    y_host = torch.empty(ntok, H, dtype=torch.float32).pin_memory()
    x_dev = x_host.to(dev)
    out_all = torch.empty(ntok, H, device=dev)
    # one ids / w pair reused by every call (16-byte aligned, as the ABI requires)
    ids = torch.empty(1, K, dtype=torch.int32, device=dev)
    w = torch.empty(1, K, dtype=torch.float32, device=dev)
    lws = B.workspace(B.ds4g_layer_decode_workspace(), dev)

    def step():
        for i in range(ntok):
            L, R, b = layers[i % nc]
            B.ds4g_moe_layer_decode(x_dev[i:i + 1], R, b, L.struct, ids, w, out_all[i:i + 1], lws)

    step()
    torch.cuda.synchronize()
    st = B.ds4g_last_error(lws)
    if st:
        raise RuntimeError(f"device status {st} during warm-up")
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    with ClockSampler(local_rank) as clk:
        ev0.record()
        for _ in range(args.steps):
            graph.replay()
        ev1.record()
        torch.cuda.synchronize()
    barrier()
    dev_s = ev0.elapsed_time(ev1) / 1e3
    barrier()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        x_dev.copy_(x_host, non_blocking=True)
        graph.replay()
        y_host.copy_(out_all, non_blocking=True)
        torch.cuda.synchronize()
    e2e_s = time.perf_counter() - t0
    barrier()
    st = B.ds4g_last_error(lws)
    if st:
        raise RuntimeError(f"device status {st} after the timed region")
    dev_s, e2e_s = max_over_ranks([dev_s, e2e_s], world, dev)
    if rank != 0:
        return None
    tokens = ntok * args.steps * world
    value = tokens / dev_s
    call_us = dev_s / (ntok * args.steps) * 1e6
    hbm, kind = peaks()
    achieved = LAYER_BYTES / (call_us * 1e-6) / 1e9
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(dev_s / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": DECODE_DTYPE, "data": "synthetic",
        "config": {"workload": S1_WORKLOAD.format(ntok=ntok, copies=nc), "layers": 1, "layer_copies": nc,
                   "tokens_per_step": ntok, "global_batch": 1, "seq_len": 1,
                   "parallelism": "replicas" if world > 1 else "single",
                   "l2": f"no flush: {nc} layer copies of 1.86 GB used in turn (>> 126 MB L2)",
                   "us_per_call": round(call_us, 3),
                   "packed_routed_gbs": round(ROUTED_BYTES / (call_us * 1e-6) / 1e9, 1),
                   "setup_s": round(setup_s, 1)},
        "e2e": {"value": round(tokens / e2e_s, 3), "unit": "tokens/s",
                "h2d_bytes_per_step": int(x_host.numel() * 4), "d2h_bytes_per_step": int(y_host.numel() * 4)},
        "roofline": {"bound": "hbm", "kernel": "decode_t1_kernel (whole layer, independent launches)",
                     "achieved": round(achieved, 1), "peak": hbm, "peak_kind": kind, "unit": "GB/s",
                     "frac": round(achieved / hbm, 4), "bytes_per_launch": LAYER_BYTES,
                     "launch_us": round(call_us, 3), "traffic": traffic_record("decode_t1_kernel")},
        "gpu_launches": ntok * args.steps,
        "clocks": clk.summary(),
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline("single-layer", args.cpu_size, 4)
    return line

# ------------------------------------------------------ streamed workload
ST_WORKLOAD = ("expert streaming decode: {nl} MoE layers x 256 experts (IQ2_XXS gate/up, Q2_K down) with the routed "
               "experts in pinned host memory and an HBM cache of {slots} expert slots (LRU), bf16 shared and fp32 "
               "router resident, 1 token at a time, {ntok} tokens per step")


def run_stream(args, rank, world, local_rank):
    """Decode with the routed experts streamed from host memory: per token
    and layer, rmsnorm + route + ds4g_moe_forward_streamed (ids read back,
    missing experts copied into the cache, forward kernels)."""
    import torch
    import bit_quantized_moe_bias_b300 as B
    torch.cuda.set_device(local_rank)
    dev = f"cuda:{local_rank}"
    nl, ntok, slots = args.stream_layers, args.tokens, args.cache_slots
    t_setup = time.time()
    built = build_model(dev, nl)
    per_expert = 2 * B.ds4g_packed_size(0, F, H) + B.ds4g_packed_size(1, H, F)
    layers = []
    for L, R, b in built:
        host = [torch.empty(t.shape, dtype=torch.uint8, pin_memory=True) for t in L.tensors[:3]]
        for hb, t in zip(host, L.tensors[:3]):
            hb.copy_(t)
        src = B.HostExperts(*[{e: hb[e] for e in range(E)} for hb in host])
        if args.stream_source == "file":
            # the layer's experts in an expert file; the host copies are dropped
            path = os.path.join(args.stream_dir, "ds4g_layer%d.ds4gexp" % len(layers))
            B.ds4g_expert_file_write(path, src)
            src, host = B.ExpertFile(path), None
        layers.append((src, host, L.tensors[3:7], R, b))
    del built, L, t
    torch.cuda.synchronize()
    torch.cuda.empty_cache()        # the routed experts now live only in host memory
    setup_s = time.time() - t_setup
    cache = B.ExpertCache(slots, max_tokens=1, device=dev)
    x_host = torch.from_numpy(synth.hidden(SEED + rank, CFG, ntok, layer=999, normalise=False)).pin_memory()
    y_host = torch.empty(ntok, H, dtype=torch.float32).pin_memory()
    x_dev = x_host.to(dev)
    xn = torch.empty(1, H, device=dev)
    act = [torch.empty(1, H, device=dev) for _ in range(2)]
    out_all = torch.empty(ntok, H, device=dev)
    ids = torch.empty(1, K, dtype=torch.int32, device=dev)
    w = torch.empty(1, K, dtype=torch.float32, device=dev)
    rws = B.workspace(B.ds4g_route_workspace(1), dev)
    fws = B.workspace(B.ds4g_forward_workspace(1), dev)

    def step():
        for i in range(ntok):
            cur = x_dev[i:i + 1]
            for l, (src, _, (sg, su, sd, grid), R, b) in enumerate(layers):
                dst = out_all[i:i + 1] if l == nl - 1 else act[l & 1]
                B.ds4g_rmsnorm(cur, xn)
                B.ds4g_moe_route(xn, R, b, ids, w, rws)
                if args.stream_source == "file":
                    B.ds4g_moe_forward_streamed_file(xn, l, src, sg, su, sd, grid, ids, w, dst, cache, fws)
                else:
                    B.ds4g_moe_forward_streamed(xn, l, src, sg, su, sd, grid, ids, w, dst, cache, fws)
                cur = dst

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    st = B.ds4g_last_error(rws) or B.ds4g_last_error(fws)
    if st:
        raise RuntimeError(f"device status {st} during warm-up")

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    h0 = cache.stats()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    with ClockSampler(local_rank) as clk:
        ev0.record()
        for _ in range(args.steps):
            step()
        ev1.record()
        torch.cuda.synchronize()
    barrier()
    dev_s = ev0.elapsed_time(ev1) / 1e3
    h1 = cache.stats()
    barrier()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        x_dev.copy_(x_host, non_blocking=True)
        step()
        y_host.copy_(out_all, non_blocking=True)
        torch.cuda.synchronize()
    e2e_s = time.perf_counter() - t0
    barrier()
    # pinned host -> device copy bandwidth of this machine (the ceiling of the misses)
    big = torch.empty(1 << 30, dtype=torch.uint8, pin_memory=True)
    dbig = torch.empty(1 << 30, dtype=torch.uint8, device=dev)
    bw = []
    for _ in range(3):
        a, c = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        dbig.copy_(big, non_blocking=True)
        c.record()
        torch.cuda.synchronize()
        bw.append((1 << 30) / (a.elapsed_time(c) / 1e3) / 1e9)
    h2d_peak = max(bw)
    st = B.ds4g_last_error(rws) or B.ds4g_last_error(fws)
    if st:
        raise RuntimeError(f"device status {st} after the timed region")
    dev_s, e2e_s = max_over_ranks([dev_s, e2e_s], world, dev)
    if rank != 0:
        return None
    hits, misses, nbytes = (h1[0] - h0[0], h1[1] - h0[1], h1[2] - h0[2])
    tokens = ntok * args.steps * world
    achieved = nbytes / dev_s * world / 1e9
    line = {
        "metric": METRIC, "value": round(tokens / dev_s, 3), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dev_s / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": DECODE_DTYPE, "data": "synthetic",
        "config": {"workload": ST_WORKLOAD.format(nl=nl, slots=slots, ntok=ntok).replace(
                       "in pinned host memory", "in pinned host memory" if args.stream_source == "host"
                       else "in expert files (read with pread on a miss)"), "layers": nl,
                   "tokens_per_step": ntok, "cache_slots": slots,
                   "cache_gb": round(slots * per_expert / 1e9, 3), "host_expert_gb": round(nl * E * per_expert / 1e9, 2),
                   "global_batch": 1, "seq_len": 1, "parallelism": "replicas" if world > 1 else "single",
                   "l2": "no flush: every miss copies 7.1 MB from host memory; resident weights 55 MB per layer",
                   "hit_rate": round(hits / max(hits + misses, 1), 4), "misses_per_token_layer":
                       round(misses / (ntok * args.steps * nl), 3), "setup_s": round(setup_s, 1)},
        "e2e": {"value": round(tokens / e2e_s, 3), "unit": "tokens/s",
                "h2d_bytes_per_step": int(x_host.numel() * 4), "d2h_bytes_per_step": int(y_host.numel() * 4)},
        "roofline": {"bound": "h2d", "kernel": ("expert copies host -> HBM (cudaMemcpyAsync from pinned memory)"
                                                if args.stream_source == "host" else
                                                "expert reads (pread, 2 pinned staging buffers) + copies -> HBM"),
                     "achieved": round(achieved, 2), "peak": round(h2d_peak, 2),
                     "peak_kind": "measured in this run: 1 GiB pinned host -> device copy", "unit": "GB/s",
                     "frac": round(achieved / h2d_peak, 4), "bytes_copied": int(nbytes), "traffic": None},
        "gpu_launches": ntok * nl * 4 * args.steps,
        "clocks": clk.summary(),
    }
    cache.close()
    return line


# --------------------------------------------------------- prefill workload
PF_T = 2048
PF_CFG = 3
# algorithmic FLOPs of the gate/up phase (routed 6T slots + shared T tokens)
PF_GATEUP_FLOP = 2 * (6 * PF_T + PF_T) * 2 * F * H
PF_FLOP = 2 * (6 * PF_T + PF_T) * 3 * F * H + 2 * PF_T * E * H   # + router
PF_WORKLOAD = ("config3 chunked prefill: 1 MoE layer x 256 experts (IQ2_XXS gate/up, Q2_K down, bf16 shared, "
               "fp32 router), T=2048 tokens per chunk, route + forward per step")


def run_prefill(args, rank, world, local_rank):
    import torch
    import bit_quantized_moe_bias_b300 as B
    torch.cuda.set_device(local_rank)
    dev = f"cuda:{local_rank}"
    T = PF_T
    (L, R, b), = build_model(dev, 1, PF_CFG)
    x_host = torch.from_numpy(synth.hidden(SEED + rank, PF_CFG, T)).pin_memory()
    y_host = torch.empty(T, H, dtype=torch.float32).pin_memory()
    x = x_host.to(dev)
    ids = torch.empty(T, K, dtype=torch.int32, device=dev)
    w = torch.empty(T, K, dtype=torch.float32, device=dev)
    out = torch.empty(T, H, device=dev)
    rws = B.workspace(B.ds4g_route_workspace(T), dev)
    fws = B.workspace(B.ds4g_forward_workspace(T), dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)   # > 126 MB L2

    def step(ev=None):
        B.ds4g_moe_route(x, R, b, ids, w, rws)
        if ev is not None:
            ev[0].record()
        B.ds4g_moe_gate_up(x, L.struct, ids, w, out, fws)
        if ev is not None:
            ev[1].record()
        B.ds4g_moe_down(x, L.struct, ids, w, out, fws)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    st = B.ds4g_last_error(rws) or B.ds4g_last_error(fws)
    if st:
        raise RuntimeError(f"device status {st} during warm-up")

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    mk = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    evs = [(mk(), mk(), mk(), mk()) for _ in range(args.steps)]
    barrier()
    with ClockSampler(local_rank) as clk:
        for e0, g0, g1, e1 in evs:
            flush.zero_()
            e0.record()
            step((g0, g1))
            e1.record()
        torch.cuda.synchronize()
    barrier()
    dev_s = sum(e0.elapsed_time(e1) for e0, _, _, e1 in evs) / 1e3
    gu_us = statistics.mean(g0.elapsed_time(g1) for _, g0, g1, _ in evs) * 1e3
    # end to end through the same calls: host hidden in, host output back
    barrier()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        x.copy_(x_host, non_blocking=True)
        step()
        y_host.copy_(out, non_blocking=True)
        torch.cuda.synchronize()
    e2e_s = time.perf_counter() - t0
    barrier()
    st = B.ds4g_last_error(rws) or B.ds4g_last_error(fws)
    if st:
        raise RuntimeError(f"device status {st} after the timed region")
    dev_s, e2e_s = max_over_ranks([dev_s, e2e_s], world, dev)
    if rank != 0:
        return None
    tokens = T * args.steps * world
    meas = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))) if os.path.exists(
        os.path.join(ROOT, "MEASURED_PEAKS.json")) else {}
    peak, kind = (float(meas["bf16_tflops"]), "measured burst") if "bf16_tflops" in meas else (1800.0, "fallback")
    achieved = PF_GATEUP_FLOP / (gu_us * 1e-6) / 1e12
    line = {
        "metric": METRIC, "value": round(tokens / dev_s, 1), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dev_s / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16/bf16 x f16/bf16 -> f32",
        "data": "synthetic",
        "config": {"workload": PF_WORKLOAD, "tokens_per_step": T, "layers": 1,
                   "parallelism": "replicas" if world > 1 else "single",
                   "l2": "flushed (512 MB write) before every timed step",
                   "achieved_tflops_block": round(PF_FLOP / (dev_s / args.steps) / 1e12, 1)},
        "e2e": {"value": round(tokens / e2e_s, 1), "unit": "tokens/s", "h2d_bytes_per_step": int(x_host.numel() * 4),
                "d2h_bytes_per_step": int(y_host.numel() * 4)},
        "roofline": {"bound": "tensor", "kernel": "prefill_gemm_kernel (gate/up phase, incl. bucket + permute)",
                     "achieved": round(achieved, 1), "peak": peak, "peak_kind": kind, "unit": "TFLOP/s",
                     "frac": round(achieved / peak, 4), "flop_per_launch": PF_GATEUP_FLOP,
                     "launch_us": round(gu_us, 2), "traffic": traffic_record("prefill_gemm_kernel")},
        "gpu_launches": 7 * args.steps,   # route, bucket, permute, gemm, h cast, gemm, combine
        "clocks": clk.summary(),
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline("prefill", args.cpu_size, 1)
    return line


# --------------------------------------------------- batched decode workload
B2_T, B2_CFG, B2_COPIES = 32, 2, 8
B2_WORKLOAD = ("config2 batched decode: T=32 independent tokens through 1 MoE layer x 256 experts (IQ2_XXS gate/up, "
               "Q2_K down, bf16 shared, fp32 router), router bias Zipf(1.1)-ranked; a step = route + forward of the "
               "batch on each of 8 independent layer copies in turn")
EXPERT_BYTES_Q2 = 2 * 2162688 + 2752512             # 7,077,888


def _barrier(world):
    import torch
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()


def run_batched(args, rank, world, local_rank):
    """Config 2: T = 32 tokens per layer call with Zipf-skewed routing, so
    the six selections of the 32 tokens overlap heavily.  Eight independent
    layer copies (1.86 GB each) are used in turn, so every call finds its
    weights cold in L2.  Algorithmic bytes per call: the distinct selected
    experts' packed bytes + shared expert + router + activations."""
    import torch
    import bit_quantized_moe_bias_b300 as B
    torch.cuda.set_device(local_rank)
    dev = f"cuda:{local_rank}"
    T, nc = B2_T, args.batched_copies
    t_setup = time.time()
    layers = build_model(dev, nc, B2_CFG, zipf=True)
    setup_s = time.time() - t_setup
    x_host = torch.from_numpy(synth.hidden(SEED + rank, B2_CFG, T)).pin_memory()
    y_host = torch.empty(nc, T, H, dtype=torch.float32).pin_memory()
    x = x_host.to(dev)
    ids = torch.empty(nc, T, K, dtype=torch.int32, device=dev)
    w = torch.empty(nc, T, K, dtype=torch.float32, device=dev)
    out = torch.empty(nc, T, H, device=dev)
    rws = B.workspace(B.ds4g_route_workspace(T), dev)
    fws = B.workspace(B.ds4g_forward_workspace(T), dev)

    def step(ev=None):
        for c, (L, R, b) in enumerate(layers):
            B.ds4g_moe_route(x, R, b, ids[c], w[c], rws)
            if ev is not None:
                ev[c][0].record()
            B.ds4g_moe_forward(x, L.struct, ids[c], w[c], out[c], fws)
            if ev is not None:
                ev[c][1].record()

    step()
    torch.cuda.synchronize()
    st = B.ds4g_last_error(rws) or B.ds4g_last_error(fws)
    if st:
        raise RuntimeError(f"device status {st} during warm-up")
    ids_h = ids.cpu().numpy()
    distinct = [len(set(ids_h[c].reshape(-1).tolist())) for c in range(nc)]
    step_bytes = sum(u * EXPERT_BYTES_Q2 + SHARED_BYTES + ROUTER_BYTES + E * 4 + 2 * T * H * 4 for u in distinct)
    graph = torch.cuda.CUDAGraph(keep_graph=True)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            step()
    torch.cuda.current_stream().wait_stream(s)
    nkern = graph_kernels(graph)
    graph.instantiate()
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    _barrier(world)
    with ClockSampler(local_rank) as clk:
        ev0.record()
        for _ in range(args.steps):
            graph.replay()
        ev1.record()
        torch.cuda.synchronize()
    _barrier(world)
    dev_s = ev0.elapsed_time(ev1) / 1e3
    _barrier(world)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        x.copy_(x_host, non_blocking=True)
        graph.replay()
        y_host.copy_(out, non_blocking=True)
        torch.cuda.synchronize()
    e2e_s = time.perf_counter() - t0
    _barrier(world)
    # the forward alone (eager, CUDA events on the launching stream), per copy
    mk = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    fw_us = []
    for _ in range(3):
        evs = [(mk(), mk()) for _ in range(nc)]
        step(evs)
        torch.cuda.synchronize()
        fw_us.append([a.elapsed_time(b) * 1e3 for a, b in evs])
    fw_us = [statistics.median(v[c] for v in fw_us) for c in range(nc)]
    st = B.ds4g_last_error(rws) or B.ds4g_last_error(fws)
    if st:
        raise RuntimeError(f"device status {st} after the timed region")
    dev_s, e2e_s = max_over_ranks([dev_s, e2e_s], world, dev)
    if rank != 0:
        return None
    tokens = T * nc * args.steps * world
    hbm, kind = peaks()
    fw_bytes = [u * EXPERT_BYTES_Q2 + SHARED_BYTES + 2 * T * H * 4 + 2 * T * K * 4 for u in distinct]
    achieved = sum(fw_bytes) / (sum(fw_us) * 1e-6) / 1e9
    line = {
        "metric": METRIC, "value": round(tokens / dev_s, 1), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dev_s / args.steps * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp16x2-split activations x exact codes -> f32", "data": "synthetic",
        "config": {"workload": B2_WORKLOAD if nc == B2_COPIES else B2_WORKLOAD.replace("8 independent", f"{nc} independent"),
                   "tokens_per_call": T, "layer_copies": nc, "global_batch": T,
                   "seq_len": 1, "parallelism": "replicas" if world > 1 else "single",
                   "l2": "no flush: 8 layer copies of 1.86 GB used in turn (>> 126 MB L2)",
                   "distinct_experts_per_call": distinct,
                   "achieved_hbm_gbs_block": round(step_bytes * args.steps / dev_s / 1e9, 1),
                   "setup_s": round(setup_s, 1)},
        "e2e": {"value": round(tokens / e2e_s, 1), "unit": "tokens/s", "h2d_bytes_per_step": int(x_host.numel() * 4),
                "d2h_bytes_per_step": int(y_host.numel() * 4)},
        "roofline": {"bound": "hbm", "kernel": "ds4g_moe_forward at T=32 (all its launches)",
                     "achieved": round(achieved, 1), "peak": hbm, "peak_kind": kind, "unit": "GB/s",
                     "frac": round(achieved / hbm, 4), "bytes_per_launch": int(sum(fw_bytes) / nc),
                     "launch_us": round(sum(fw_us) / nc, 2), "traffic": None},
        "gpu_launches": (nkern * args.steps) if nkern is not None else None,
        "clocks": clk.summary(),
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline("batched", args.cpu_size, 8)
    return line


# ------------------------------------------------- q2-q4 prefill workload
Q4P_T, Q4P_CFG, Q4P_LAYERS = 4096, 4, 8
Q4P_WORKLOAD = ("config4 mixed-precision prefill: T=4096 tokens through 8 MoE layers x 256 experts (layers 0-1 "
                "IQ2_XXS gate/up + Q2_K down, layers 2-7 Q4_K gate/up/down), bf16 shared, fp32 router, Zipf(1.1) "
                "router bias, rmsnorm between layers; a step = the whole 8-layer chain")


def run_q2q4_prefill(args, rank, world, local_rank):
    import torch
    import bit_quantized_moe_bias_b300 as B
    torch.cuda.set_device(local_rank)
    dev = f"cuda:{local_rank}"
    T, nl = Q4P_T, Q4P_LAYERS
    t_setup = time.time()
    layers = build_model(dev, nl, Q4P_CFG, q4_layers=Q4_LAYERS, zipf=True)
    setup_s = time.time() - t_setup
    x_host = torch.from_numpy(synth.hidden(SEED + rank, Q4P_CFG, T)).pin_memory()
    y_host = torch.empty(T, H, dtype=torch.float32).pin_memory()
    x = x_host.to(dev)
    hb = [torch.empty(T, H, device=dev) for _ in range(2)]
    out = torch.empty(T, H, device=dev)
    ids = torch.empty(T, K, dtype=torch.int32, device=dev)
    w = torch.empty(T, K, dtype=torch.float32, device=dev)
    rws = B.workspace(B.ds4g_route_workspace(T), dev)
    fws = B.workspace(B.ds4g_forward_workspace(T), dev)

    def step(ev=None):
        h = x
        for l, (L, R, b) in enumerate(layers):
            B.ds4g_moe_route(h, R, b, ids, w, rws)
            if ev is not None:
                ev[l][0].record()
            dst = out if l == nl - 1 else hb[0]
            B.ds4g_moe_gate_up(h, L.struct, ids, w, dst, fws)
            if ev is not None:
                ev[l][1].record()
            B.ds4g_moe_down(h, L.struct, ids, w, dst, fws)
            if l < nl - 1:
                B.ds4g_rmsnorm(dst, hb[1])
                h = hb[1]

    for _ in range(max(args.warmup, 1)):
        step()
    torch.cuda.synchronize()
    st = B.ds4g_last_error(rws) or B.ds4g_last_error(fws)
    if st:
        raise RuntimeError(f"device status {st} during warm-up")
    mk = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    evs = [[(mk(), mk()) for _ in range(nl)] for _ in range(args.steps)]
    e0, e1 = mk(), mk()
    _barrier(world)
    with ClockSampler(local_rank) as clk:
        e0.record()
        for i in range(args.steps):
            step(evs[i])
        e1.record()
        torch.cuda.synchronize()
    _barrier(world)
    dev_s = e0.elapsed_time(e1) / 1e3
    gu_us = statistics.mean(sum(a.elapsed_time(b) for a, b in ev) for ev in evs) * 1e3
    _barrier(world)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        x.copy_(x_host, non_blocking=True)
        step()
        y_host.copy_(out, non_blocking=True)
        torch.cuda.synchronize()
    e2e_s = time.perf_counter() - t0
    _barrier(world)
    st = B.ds4g_last_error(rws) or B.ds4g_last_error(fws)
    if st:
        raise RuntimeError(f"device status {st} after the timed region")
    dev_s, e2e_s = max_over_ranks([dev_s, e2e_s], world, dev)
    if rank != 0:
        return None
    tokens = T * args.steps * world
    meas = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))) if os.path.exists(
        os.path.join(ROOT, "MEASURED_PEAKS.json")) else {}
    peak, kind = (float(meas["bf16_tflops"]), "measured burst") if "bf16_tflops" in meas else (1800.0, "fallback")
    gu_flop = nl * 2 * (K * T + T) * 2 * F * H
    layer_flop = 2 * (K * T + T) * 3 * F * H + 2 * T * E * H
    achieved = gu_flop / (gu_us * 1e-6) / 1e12
    line = {
        "metric": METRIC, "value": round(tokens / dev_s, 1), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dev_s / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16/bf16 x f16/bf16 -> f32", "data": "synthetic",
        "config": {"workload": Q4P_WORKLOAD, "tokens_per_step": T, "layers": nl, "q4_layers": Q4_LAYERS,
                   "parallelism": "replicas" if world > 1 else "single",
                   "l2": "no flush: 25.8 GB of layer weights per step (>> 126 MB L2)",
                   "achieved_tflops_block": round(nl * layer_flop / (dev_s / args.steps) / 1e12, 1),
                   "setup_s": round(setup_s, 1)},
        "e2e": {"value": round(tokens / e2e_s, 1), "unit": "tokens/s", "h2d_bytes_per_step": int(x_host.numel() * 4),
                "d2h_bytes_per_step": int(y_host.numel() * 4)},
        "roofline": {"bound": "tensor", "kernel": "prefill_gemm_kernel (gate/up phase, incl. bucket + permute), "
                                                  "8 layers", "achieved": round(achieved, 1), "peak": peak,
                     "peak_kind": kind, "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                     "flop_per_launch": gu_flop // nl, "launch_us": round(gu_us / nl, 2), "traffic": None},
        "gpu_launches": (nl * 7 + (nl - 1)) * args.steps,   # per layer as in the prefill line; rmsnorm between
        "clocks": clk.summary(),
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline("q2q4-prefill", args.cpu_size, 2)
    return line


WORKLOADS = {"decode": WORKLOAD, "prefill": PF_WORKLOAD, "batched": B2_WORKLOAD, "q2q4-prefill": Q4P_WORKLOAD,
             "decode-stream": WORKLOAD, "single-layer": S1_WORKLOAD.format(ntok=64, copies=S1_COPIES)}


# ------------------------------------------------------------- CPU oracle
# The oracle (plain C, fp64 accumulation, OpenMP over output rows) timed on a
# bounded sample of each workload.  Generating the synthetic weights is not
# timed.  The GPU arm runs these samples in a fresh interpreter (the same
# code path as --impl reference): in the GPU arm's own process the oracle's
# OpenMP threads competed with torch's thread pool and ran about 4x slower.
_CACHE = {}


def _cached(key, fn):
    if key not in _CACHE:
        _CACHE[key] = fn()
    return _CACHE[key]


def _experts(cfg, layer, ids, gut=0, dt=1):
    gate, up, down = [None] * E, [None] * E, [None] * E
    for e in sorted(set(int(v) for v in np.asarray(ids).reshape(-1))):
        gate[e], up[e], down[e] = _cached(("X", cfg, layer, e, gut),
                                          lambda: synth.expert(SEED, cfg, layer, e, gut, dt))
    return gate, up, down


def oracle_sample(nlayers, nthreads=0):
    """Decode (full-depth workload): 1 token through the first `nlayers`
    layers of the chain.  Returns (seconds of oracle compute, tokens)."""
    import oracle
    x = synth.hidden(SEED, CFG, 1, layer=999, normalise=False)
    grid = synth.iq2_grid(SEED)
    t = 0.0
    for l in range(nlayers):
        R, b, sh = _cached(("L", CFG, l), lambda: (synth.router(SEED, CFG, l), synth.bias_normal(SEED, CFG, l),
                                                   synth.shared(SEED, CFG, l)))
        t0 = time.perf_counter()
        xn = oracle.rmsnorm(x)
        ids, w, _, _ = oracle.route(xn, R, b)
        t += time.perf_counter() - t0
        gate, up, down = _experts(CFG, l, ids)
        t0 = time.perf_counter()
        x = oracle.moe_forward(xn, ids, w, gate, up, down, *sh, grid, nthreads=nthreads)
        t += time.perf_counter() - t0
    return t, 1


def oracle_sample_layer(cfg, ntok, zipf, nthreads=0):
    """One layer (prefill or batched decode): route + forward of the first
    `ntok` tokens of the workload's batch.  Returns (seconds, tokens)."""
    import oracle
    x = synth.hidden(SEED, cfg, ntok)
    R, b, sh = _cached(("L", cfg, 0), lambda: (synth.router(SEED, cfg, 0), (synth.bias_zipf if zipf else
                                               synth.bias_normal)(SEED, cfg, 0), synth.shared(SEED, cfg, 0)))
    grid = synth.iq2_grid(SEED)
    t0 = time.perf_counter()
    ids, w, _, _ = oracle.route(x, R, b)
    t = time.perf_counter() - t0
    gate, up, down = _experts(cfg, 0, ids)
    t0 = time.perf_counter()
    oracle.moe_forward(x, ids, w, gate, up, down, *sh, grid, nthreads=nthreads)
    return t + time.perf_counter() - t0, ntok


def oracle_sample_q2q4(ntok, nthreads=0):
    """q2-q4 prefill chain: the first `ntok` tokens through all 8 layers
    (route, forward, rmsnorm between layers).  Tokens are independent of one
    another through the whole chain.  Returns (seconds, tokens)."""
    import oracle
    h = synth.hidden(SEED, Q4P_CFG, ntok)
    grid = synth.iq2_grid(SEED)
    t = 0.0
    for l in range(Q4P_LAYERS):
        q4 = l >= Q4P_LAYERS - Q4_LAYERS
        gut, dt = (2, 2) if q4 else (0, 1)
        R, b, sh = _cached(("L", Q4P_CFG, l), lambda: (synth.router(SEED, Q4P_CFG, l),
                                                        synth.bias_zipf(SEED, Q4P_CFG, l),
                                                        synth.shared(SEED, Q4P_CFG, l)))
        t0 = time.perf_counter()
        ids, w, _, _ = oracle.route(h, R, b)
        t += time.perf_counter() - t0
        gate, up, down = _experts(Q4P_CFG, l, ids, gut, dt)
        t0 = time.perf_counter()
        out = oracle.moe_forward(h, ids, w, gate, up, down, *sh, grid, gut, dt, nthreads=nthreads)
        h = oracle.rmsnorm(out) if l + 1 < Q4P_LAYERS else out
        t += time.perf_counter() - t0
    return t, ntok


def cpu_model():
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or "unknown"


# per workload: (sample function of (size, nthreads), total tokens of one
# GPU step's workload unit, description of a sample of `size`)
def _sampler(workload, size):
    if workload == "prefill":
        return (lambda n: oracle_sample_layer(PF_CFG, size, False, n),
                f"first {size} of the {PF_T} tokens of the chunk (oracle route + forward)")
    if workload == "batched":
        return (lambda n: oracle_sample_layer(B2_CFG, size, True, n),
                f"first {size} of the {B2_T} tokens of the batch (oracle route + forward)")
    if workload == "single-layer":
        return (lambda n: oracle_sample_layer(S1_CFG, size, False, n),
                f"{size} tokens through one layer (oracle route + forward of a batch of {size} tokens)")
    if workload == "q2q4-prefill":
        return (lambda n: oracle_sample_q2q4(size, n),
                f"first {size} of the {Q4P_T} tokens through all {Q4P_LAYERS} layers (oracle route + forward, "
                "rmsnorm between layers); tokens are independent through the chain")
    nl = size
    return (lambda n: (lambda r: (r[0] * NLAYER / nl, r[1]))(oracle_sample(nl, n)),
            f"1 token through the first {nl} of {NLAYER} layers (oracle rmsnorm + route + forward), "
            f"extrapolated linearly to {NLAYER} layers")


def default_cpu_size(workload):
    return {"prefill": 8, "batched": 32, "q2q4-prefill": 4, "single-layer": 16}.get(workload, NLAYER)


def run_reference(args):
    """The oracle on this host's cores, on a bounded sample of the workload
    per step; value = sample tokens / oracle seconds (higher is better)."""
    size = args.cpu_size or default_cpu_size(args.workload)
    fn, desc = _sampler(args.workload, size)
    for _ in range(args.warmup):
        fn(args.cpu_threads)
    tokens, secs = 0, 0.0
    for _ in range(args.steps):
        t, n = fn(args.cpu_threads)
        secs += t
        tokens += n
    value = tokens / secs
    cores = args.cpu_threads or os.cpu_count()
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 5), "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(secs / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOADS[args.workload]},
        "cpu_baseline": {"value": round(value, 5), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "cpu_model": cpu_model(), "sample": f"per step: {desc}; fp64, OpenMP over output rows"},
        "e2e": {"value": round(value, 5), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def cpu_baseline(workload, size=None, size_1thread=None):
    """The oracle timed in a fresh interpreter (bench.py --impl reference):
    all cores on `size`, and one thread on `size_1thread`."""
    def sub(sz, threads):
        cmd = [sys.executable, os.path.abspath(__file__), "--impl", "reference", "--workload", workload,
               "--steps", "1", "--warmup", "0", "--cpu-threads", str(threads)]
        if sz:
            cmd += ["--cpu-size", str(sz)]
        env = {k: v for k, v in os.environ.items() if k not in ("OMP_NUM_THREADS", "RANK", "WORLD_SIZE",
                                                               "LOCAL_RANK")}
        out = subprocess.run(cmd, capture_output=True, text=True, env=env, timeout=900, check=True).stdout
        return json.loads(out.strip().splitlines()[-1])["cpu_baseline"]
    full = sub(size, 0)
    if size_1thread is not None:
        one = sub(size_1thread, 1)
        full["value_1thread"] = one["value"]
        full["sample_1thread"] = one["sample"]
    full["process"] = "fresh interpreter (bench.py --impl reference), no torch loaded"
    return full


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--tokens", type=int, default=64)
    ap.add_argument("--layers", type=int, default=NLAYER,
                    help="stacked layers (43 = the full-depth workload; fewer only for profiling)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-size", type=int, default=0,
                    help="oracle sample per step: layers (decode) or tokens (other workloads); 0 = default")
    ap.add_argument("--cpu-threads", type=int, default=0, help="oracle OpenMP threads (0 = all cores)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", choices=list(WORKLOADS), default="decode",
                    help="decode = 43-layer full-depth decode (headline); prefill = T=2048 chunk, one layer; "
                         "batched = T=32 tokens, one layer, Zipf routing; q2q4-prefill = T=4096 through 8 "
                         "layers (2 q2, 6 q4), Zipf routing; decode-stream = routed experts streamed from host "
                         "memory through an HBM cache; single-layer = 1 token through 1 layer per call, 8 layer "
                         "copies in turn")
    ap.add_argument("--stream-layers", type=int, default=4, help="decode-stream: layers (host memory 1.8 GB each)")
    ap.add_argument("--cache-slots", type=int, default=256, help="decode-stream: HBM cache slots (7.1 MB each)")
    ap.add_argument("--stream-source", choices=["host", "file"], default="host",
                    help="decode-stream: routed experts in pinned host memory, or in expert files read on a miss")
    ap.add_argument("--stream-dir", default="/tmp", help="decode-stream --stream-source file: directory of the files")
    ap.add_argument("--batched-copies", type=int, default=B2_COPIES,
                    help="batched: layer copies used in turn (8 keeps every call cold in L2; fewer only for profiling)")
    ap.add_argument("--model", choices=["q2", "q2-q4", "q4"], default="q2",
                    help="decode model: q2 = every layer IQ2_XXS/Q2_K (headline); q2-q4 = last 6 layers Q4_K; "
                         "q4 = every layer Q4_K")
    ap.add_argument("--decode-path", choices=["fused", "layer", "split", "q8"], default="fused",
                    help="fused = one stack call per token (one launch per layer, programmatic dependent "
                         "launches); layer = one call per layer; split = rmsnorm, route, gate/up, down launches")
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    run = {"prefill": run_prefill, "decode-stream": run_stream, "batched": run_batched,
           "q2q4-prefill": run_q2q4_prefill, "single-layer": run_single_layer}.get(args.workload, run_ours)
    line = run(args, rank, world, local_rank)
    if line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
