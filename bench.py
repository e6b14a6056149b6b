"""Benchmark of the routed MoE layer forward pass on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step is one pass of the whole layer (router + top-k, residency bind with
its fill copies, dispatch, expert FFN, combine) over one batch of the
workload: one decode token for the default 'decode' workload (hidden 4096,
256 experts, top-6, intermediate 2048, 37% of experts resident, LRU, Zipf(1.1)
routing), the whole 8192-token block for 'prefill', four stacked layers for
'long_prefill'.  Inputs are synthetic (seeded; see moe_inputs) and resident
in HBM before the timed region; each step is one moe_layer_forward call per
layer, timed with CUDA events on its stream, and L2 is flushed (256 MB write)
between steps outside the events.  Prints one JSON line on rank 0: the decode
workload's figures at the top level and, as sub-records of the same line,
the 'prefill' and 'long_prefill' workloads and the decode step with MXFP4
experts 'decode_mxfp4' (at least 20 timed steps each; --extra selects them).  --impl reference times the CPU fp64 oracle instead.
"""
import argparse
import json
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from moe_inputs import CONFIGS, gen  # noqa: E402

METRIC = "MoE-layer tokens/s (decode, prefill) and % of GB300 HBM / bf16 tensor peak"
UNIT = "tokens/s"
CLOCK_QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
               "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
               "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ------------------------------------------------------------------ clocks
class ClockSampler:
    def __init__(self, gpu_index):
        self.proc = None
        self.path = None
        self.gpu_index = gpu_index

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={CLOCK_QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------ algorithmic work
def expert_ffn_flops(cfg):
    return 2.0 * cfg.T * cfg.k * 3 * cfg.H * cfg.I


def router_flops(cfg):
    return 2.0 * cfg.T * cfg.H * cfg.E


# DRAM bytes (read + write) per launch of the dominant kernel, from the ncu
# captures summarised under profiles/ (a workload without an entry, or whose
# kernels changed since their capture, reports null).
#  decode: decode_layer_kernel captured on decode_profile (same six 50.3 MB
#    experts per step, one cache fill) plus the 224 extra 16 KB router rows
#    of the 256-expert layer.
#  prefill: the two gemm_kernel launches captured on prefill_profile (64
#    experts x ~192 rows) scaled by the units processed (4x the experts, 4x
#    the rows): traffic there is each weight byte once plus the activations,
#    both proportional.
FFN_TRAFFIC = {"decode": 302663424 + 30414336 + 224 * 16384,
               "prefill": 4 * (2255529216 + 48149760 + 1126688000 + 89227008)}
# DRAM bytes per launch of the FP4 kernels, from the captures summarised in
# profiles/fp4_gemm_kernel_prefill_profile.md and profiles/decode_fp4_kernel_decode_profile.md
FP4_TRAFFIC = {
    # gate/up + down GEMMs of prefill_profile (64 experts, 2048 tokens), x4 for the 8192-token block over 256 experts
    "prefill_mxfp4": 4 * (913240832 + 31427072 + 473911296 + 142872064),
    # one decode_profile step with a fill: six experts' codes and scales, 0.5 MB of router rows, one fill written
    "decode_mxfp4": 80890880 + 13875456,
}
FP4_TRAFFIC_NOTE = {
    "prefill_mxfp4": "ncu capture of the two fp4_gemm_kernel launches on prefill_profile, x4 (units processed)",
    "decode_mxfp4": "ncu capture of decode_fp4_kernel on a decode_profile step with one fill (32 experts: 0.5 MB of "
                    "router rows instead of 4.19 MB)",
}
MX_TRAFFIC = 81629184   # mx_ring_kernel on the MXFP4 decode call: 1.8826 TB/s x 43.36 us (ncu)
TRAFFIC_NOTE = {"decode": ("ncu capture of decode_layer_kernel on decode_profile (1 fill) + 224 router rows; "
                           "the rest of the fill's 50 MB is still in L2 when the kernel ends"),
                "prefill": ("ncu capture of the layer call's two gemm_kernel launches on prefill_profile (bf16 expert "
                            "rows), x4 (units processed); the timed public call writes fp32 rows: +T*k*H*2 B")}


FFN_MODES = {"auto": lambda m: m.MOE_FFN_AUTO, "gemv": lambda m: m.MOE_FFN_GEMV, "gemm": lambda m: m.MOE_FFN_GEMM}


# ------------------------------------------------------------------ our arm
# sub-records of the default line.  The host-pool records read pinned host memory over the CPU-GPU link,
# whose rate varied with the process's history (measured: 78-205 GB/s for the same 51.5 GB streamed stack);
# the arrangement that measured the link rate steadily: the host-pool decode in a child process of its own,
# the streamed stack last
EXTRA_DEFAULT = ("prefill,long_prefill,decode_host_pool,decode_mxfp4,decode_nvfp4,prefill_mxfp4,prefill_nvfp4,"
                 "long_prefill_streamed")


L2_BYTES = 129 << 20   # the GB300's L2


def inputs_exceed_l2(cfg):
    """Whether every step reads more than twice the L2 in expert weights alone
    (at least k distinct experts per token, every layer), so that steps can
    run back to back with no flush between them: a step cannot find the
    previous step's weights in L2."""
    return cfg.n_layers * cfg.k * cfg.expert_bytes > 2 * L2_BYTES


def run_workload(cfg, args, world, dev, stream, peaks, moe, torch):
    """Measure one workload: ``args.warmup`` untimed steps, then ``args.steps``
    timed steps.  A step is one moe_layer_forward call per layer of the
    workload, launched directly on ``stream`` (the decode layer is one kernel,
    so a graph would only add its replay).  Timing: where every step reads
    more than twice the L2 in expert weights (decode, prefill, long prefill),
    the timed steps run back to back between one pair of CUDA events, as a
    serving loop issues them; otherwise CUDA events bracket each step and L2
    is flushed (256 MB write) between steps, outside the events.  Decode-like
    workloads also get the isolated-step figures: the same trace again from
    the initial state, each step between its own events after a flush.
    Returns the measurement record (tokens/s, step times, the dominant
    kernel's roofline, clocks, end to end, launch counts)."""
    from moe_inputs.device import DeviceCache, DeviceLayer, to_dev_bf16

    decode_like = cfg.steps > 1
    back_to_back = inputs_exceed_l2(cfg)
    n_steps = args.warmup + args.steps
    dc = DeviceCache(cfg, dev)
    layers = [DeviceLayer(cfg, l, dev) for l in range(cfg.n_layers)]
    # back to back, consecutive steps read their router weights from copies (equal values) that together
    # exceed twice the L2, as the layers of a model would: no step finds its router rows in L2 (the expert
    # weights stream evict-first, so a few router copies would stay resident)
    router_sets = [[dl.struct for dl in layers]]
    router_copies = []
    if back_to_back:
        per_set = cfg.n_layers * cfg.E * cfg.H * 4
        for _ in range(-(-2 * L2_BYTES // per_set)):
            row = []
            for dl in layers:
                w = dl.w_router.clone()
                router_copies.append(w)
                row.append(moe.moe_layer(w.data_ptr(), dl.struct.bias, dl.layer, cfg.E, cfg.k, cfg.H, cfg.I))
            router_sets.append(row)
    # per-step inputs (decode: a stream of tokens; prefill: one block per layer, reused every step)
    if decode_like:
        xs = [to_dev_bf16(gen.x_bits(cfg, 0, s), dev) for s in range(n_steps)]
    else:
        xs = [to_dev_bf16(gen.x_bits(cfg, l, 0), dev) for l in range(cfg.n_layers)]
    T, H = cfg.T, cfg.H
    mode = FFN_MODES[args.ffn_mode](moe)
    ws_bytes = moe.moe_layer_workspace_size(layers[0].struct, dc.struct, T, mode)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stats = torch.zeros((n_steps, 8), dtype=torch.int32, device=dev)   # each step's residency counts
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def step_body(i):
        # decode: step i's token row; prefill: every layer's resident block
        lay = router_sets[i % len(router_sets)]
        for l in range(cfg.n_layers):
            moe.moe_layer_forward(lay[l], dc.struct, xs[i] if decode_like else xs[l], T, out, cfg.phi_q16,
                                  cfg.min_fill, cfg.fill_policy, 1000 + l, mode, None, ws, ws_bytes, status,
                                  stats[i], stream)

    # one call sets kernel attributes and occupancy caches; then the trace starts from the initial state
    with torch.cuda.stream(stream):
        step_body(0)
    torch.cuda.synchronize()
    dc.reset()
    torch.cuda.synchronize()

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    def isolated_steps():
        """Each step of the trace between its own events, L2 flushed before it."""
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_steps)]
        with torch.cuda.stream(stream):
            for i in range(n_steps):
                flush.zero_()
                ev[i][0].record(stream)
                step_body(i)
                ev[i][1].record(stream)
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in ev[args.warmup:]]

    if back_to_back:
        with torch.cuda.stream(stream):
            for s in range(args.warmup):
                step_body(s)
    else:
        with torch.cuda.stream(stream):
            for s in range(args.warmup):
                step_body(s)
                flush.zero_()
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(dev.index)
    clocks.start()
    n0 = moe.moe_kernel_launch_count()
    t0 = time.perf_counter()
    if back_to_back:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for i in range(args.steps):
                step_body(args.warmup + i)
            e1.record(stream)
        torch.cuda.synchronize()
        total_ms = e0.elapsed_time(e1)
        step_ms = None
    else:
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
        with torch.cuda.stream(stream):
            for i in range(args.steps):
                ev[i][0].record(stream)
                step_body(args.warmup + i)
                ev[i][1].record(stream)
                flush.zero_()
        torch.cuda.synchronize()
        step_ms = [a.elapsed_time(b) for a, b in ev]
        total_ms = sum(step_ms)
    barrier()
    bracket_s = time.perf_counter() - t0
    launches = moe.moe_kernel_launch_count() - n0
    clk = clocks.stop()
    total_s = total_ms / 1e3
    dev_status = int(status.cpu().numpy().view(np.uint32)[0])
    step_stats = stats[args.warmup:].cpu().numpy()
    total_s, value = aggregate_replicas(total_s, args.steps, T, world, dev)
    kernels_per_step = launches / args.steps
    isolated = None
    if decode_like:
        dc.reset()
        torch.cuda.synchronize()
        iso_ms = isolated_steps()
        isolated = {"ms_per_step": round(float(np.mean(iso_ms)), 5),
                    "step_ms_p10_p50_p90": [round(float(np.percentile(iso_ms, q)), 5) for q in (10, 50, 90)],
                    "tokens_per_s": round(len(iso_ms) * T / (sum(iso_ms) / 1e3), 3),
                    "note": "the same trace from the initial state, each step between its own CUDA events "
                            "after a 256 MB L2-flush write: the latency of one call, launch included"}

    # ---- dominant kernel: decode-sized calls run the whole layer as one kernel (the timed
    # step itself); otherwise the expert-FFN call, timed alone
    if kernels_per_step == cfg.n_layers:
        roof = decode_step_roofline(cfg, total_ms, args.steps, step_stats, peaks, back_to_back)
    else:
        roof = measure_ffn_roofline(cfg, dc, layers, xs, decode_like, stream, peaks, args, moe, torch)
    e2e = measure_e2e(cfg, dc, layers, decode_like, stream, args, moe, torch, ws, ws_bytes, status, stats[0])
    rec = {"value": round(value, 3), "unit": UNIT, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(total_s * 1e3 / args.steps, 5),
           "timing": ("back to back: one CUDA-event pair around the timed steps (every step reads more than "
                      "twice the L2 in expert weights; consecutive steps read the router weights from %d "
                      "copies in turn, %.0f MB in all)" % (len(router_sets), len(router_sets) * cfg.n_layers * cfg.E
                                                            * cfg.H * 4 / 1e6)) if back_to_back else
                     "CUDA events around each step, L2 flushed between steps",
           "bracket_ms_per_step": round(bracket_s * 1e3 / args.steps, 5),
           "config": workload_config(cfg, world, back_to_back), "device_status": dev_status, "roofline": roof,
           "clocks": clk, "e2e": e2e, "gpu_launches": int(launches), "gpu_launches_per_step": kernels_per_step}
    if step_ms is not None:
        rec["step_ms_p10_p50_p90"] = [round(float(np.percentile(step_ms, q)), 5) for q in (10, 50, 90)]
    if isolated is not None:
        rec["isolated_step"] = isolated
    if not decode_like:
        # the whole step against the bf16 tensor peak (expert FFN + router FLOPs of every layer)
        fl = cfg.n_layers * (expert_ffn_flops(cfg) + router_flops(cfg))
        tf = fl * args.steps / total_s / 1e12
        rec["step_roofline"] = {"bound": "tensor", "achieved": round(tf, 2), "peak": peaks["bf16_tflops"],
                                "unit": "TFLOP/s", "frac": round(tf / peaks["bf16_tflops"], 4),
                                "flops_per_step": fl, "peak_source": peaks["source"] + " (burst cuBLAS bf16)",
                                "note": "whole step (every launch of every layer) over the CUDA-event step time"}
    return rec


def run_ours(args, rank, world):
    import torch
    import edge_moe_serving_gb300 as moe

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    peaks = load_peaks()
    stream = torch.cuda.Stream(device=dev)
    rec = run_workload(CONFIGS[args.workload], args, world, dev, stream, peaks, moe, torch)
    result = {"metric": METRIC, "value": rec["value"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
              "warmup": args.warmup, "ms_per_step": rec["ms_per_step"], "higher_is_better": True,
              "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
              "config": rec["config"], "impl": "ours"}
    result.update({k: v for k, v in rec.items() if k not in result})
    extras = [] if args.extra in ("", "none") else [w for w in args.extra.split(",") if w != args.workload]
    for name in extras:
        torch.cuda.empty_cache()
        sub = argparse.Namespace(**vars(args))
        sub.steps = max(args.steps, 20)
        if name == "decode_host_pool":
            result[name] = run_host_record_child(name, sub)
            continue
        if name == "long_prefill_streamed":
            # in this process: its 51.5 GB pool plus the generated expert arrays leave a child process short of
            # host memory beside this one (measured: the link at 77% instead of 98%)
            result[name] = run_streamed_prefill(sub, dev, stream, moe, torch)
            continue
        if name in ("prefill_mxfp4", "prefill_nvfp4"):
            result[name] = run_fp4_prefill(sub, dev, stream, moe, torch, name.split("_")[1])
            continue
        if name in ("decode_mxfp4", "decode_nvfp4"):
            result[name] = run_fp4_decode(sub, dev, stream, moe, torch, name.split("_")[1])
            if name == "decode_mxfp4" and sub.fp4_decode_workload == "decode":
                # the expert FFN call alone (every expert resident), with its own roofline
                sub.no_cpu_baseline = True
                torch.cuda.empty_cache()
                rec = run_mx(sub)
                result[name]["ffn_call"] = {k: rec[k] for k in ("value", "ms_per_step", "roofline", "clocks")}
                result[name]["ffn_call"]["note"] = ("router + top-k, dispatch, moe_expert_ffn_mxfp4 and the combine "
                                                    "as four public calls in one graph, every expert resident; "
                                                    "roofline: the FFN call alone")
            continue
        else:
            result[name] = run_workload(CONFIGS[name], sub, world, dev, stream, peaks, moe, torch)
    return result


def aggregate_replicas(local_s, steps, tokens_per_step, world, device="cpu"):
    """Whole-job throughput of N independent replicas (no data-path exchange):
    every rank processes `steps` steps of `tokens_per_step` tokens; the job time
    is the slowest rank's (max over ranks).  Returns (job seconds, tokens/s)."""
    job_s = local_s
    if world > 1:
        import torch
        import torch.distributed as dist
        t = torch.tensor([local_s], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        job_s = float(t.item())
    return job_s, world * steps * tokens_per_step / job_s


def workload_config(cfg, world, back_to_back=False):
    l2 = ("inputs larger than L2: at least %.0f MB of expert weights per step (L2 129 MB), steps back to back, "
          "no flush" % (cfg.n_layers * cfg.k * cfg.expert_bytes / 1e6)) if back_to_back else \
        "flushed between steps (256 MB write)"
    return {"workload": cfg.name, "tokens_per_layer_call": cfg.T, "hidden": cfg.H, "experts": cfg.E,
            "top_k": cfg.k, "intermediate": cfg.I, "layers_per_step": cfg.n_layers,
            "cache_slots": cfg.cache_slots if cfg.cache_slots is not None else cfg.n_layers * cfg.E,
            "phi_q16": cfg.phi_q16, "fill_policy": "random" if cfg.fill_policy else "lowest_id",
            "routing_bias": cfg.bias, "l2": l2,
            "parallelism": f"replicas x{world}", "launch": "moe_layer_forward per layer, direct launches"}


def decode_step_roofline(cfg, total_ms, steps, stats, peaks, back_to_back):
    """Decode-sized steps are one kernel (router, residency decision, fused
    gate/up + down weight streaming with cache fills, combine).  Algorithmic
    bytes per step, as the method counts them: every distinct routed expert's
    weights once, the router weights, the token row in and the output row out;
    each cache fill writes one more expert (the fill's read is the stream's
    own), reported beside them and included in the credited bytes.  Duration:
    the timed steps' CUDA-event time over the number of steps (the kernel and
    its 4 + T*k word counter reset)."""
    T, E, H = cfg.T, cfg.E, cfg.H
    n_unique, n_fill = stats[:, 0].astype(np.float64), stats[:, 4].astype(np.float64)
    method = n_unique * cfg.expert_bytes + E * H * 4 + 2 * T * H * 2
    fills = n_fill * cfg.expert_bytes
    t = total_ms / 1e3
    achieved = float(np.sum(method + fills)) / t / 1e9
    no_fill = float(np.sum(method)) / t / 1e9
    peak = peaks["hbm_gbs"]
    return {"kernel": "decode_layer_kernel (whole layer in one cooperative launch)", "bound": "hbm",
            "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
            "traffic": FFN_TRAFFIC.get(cfg.name), "traffic_note": TRAFFIC_NOTE.get(cfg.name),
            "peak_source": peaks["source"] + " (burst copy bandwidth)",
            "algorithmic_bytes_per_step": int(np.mean(method + fills)),
            "fill_bytes_per_step": int(np.mean(fills)), "fills_per_step": round(float(np.mean(n_fill)), 3),
            "frac_without_fill_bytes": round(no_fill / peak, 4),
            "step_us": round(t / steps * 1e6, 3),
            "timing": ("one CUDA-event pair around the timed steps, back to back" if back_to_back else
                       "CUDA events around each timed step") + " (the kernel is the whole step)"}


def ffn_bytes(cfg, active):
    """Algorithmic HBM bytes of one expert-FFN call, as the method counts them:
    each active expert's weights once, the layer's token rows in and its
    output rows out (bf16).  The intermediates are implementation traffic,
    reported by ffn_impl_bytes and not credited."""
    return active * cfg.expert_bytes + cfg.T * cfg.H * 2 + cfg.T * cfg.H * 2


def ffn_impl_bytes(cfg):
    """Intermediate bytes of the timed public FFN call (not credited): the
    gathered token rows written and read (GEMM path), h written and read,
    and the fp32 expert rows written (the call's output) and read back by
    the combine."""
    R = cfg.T * cfg.k
    gather = 2 * R * cfg.H * 2 if cfg.T > 2 else 0
    return gather + 2 * R * cfg.I * 2 + 2 * R * cfg.H * 4


def measure_ffn_roofline(cfg, dc, layers, xs, decode_like, stream, peaks, args, moe, torch):
    """Time moe_expert_ffn_grouped alone for the step inputs of the timed run:
    the call is captured once into a CUDA graph (as it runs inside the layer
    graph), and each replay is bracketed by CUDA events on its stream after an
    L2 flush; router + dispatch for that step run eagerly before the flush.
    Algorithmic work per call: the weights of the active experts plus the
    activations (HBM-bound decode) or the FFN FLOPs (prefill)."""
    dev = xs[0].device
    T, k, E = cfg.T, cfg.k, cfg.E
    R = T * k
    n = min(args.steps, 16)
    ids = torch.empty(R, dtype=torch.int32, device=dev)
    w = torch.empty(R, dtype=torch.float32, device=dev)
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    perm = torch.empty(R, dtype=torch.int32, device=dev)
    inv = torch.empty(R, dtype=torch.int32, device=dev)
    y = torch.empty((R, cfg.H), dtype=torch.float32, device=dev)
    xp = torch.empty((R, cfg.H), dtype=torch.bfloat16, device=dev) if T > 8 else None
    x_cur = torch.empty((T, cfg.H), dtype=torch.bfloat16, device=dev)
    layer_cur = torch.zeros(1, dtype=torch.int32)      # host value read at capture time only
    mode = FFN_MODES[args.ffn_mode](moe)
    wsb = max(moe.moe_route_topk_workspace_size(T, cfg.H, E), moe.moe_dispatch_workspace_size(T, k, E),
              moe.moe_expert_ffn_workspace_size(T, k, E, cfg.H, cfg.I, mode))
    wsx = torch.empty(max(wsb, 256), dtype=torch.uint8, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def prep(i):
        l = 0 if decode_like else i % cfg.n_layers
        x_cur.copy_(xs[args.warmup + i] if decode_like else xs[l])
        moe.moe_route_topk(x_cur, T, cfg.H, layers[l].w_router, layers[l].bias, E, k, ids, w, None, wsx, wsb, st,
                           stream)
        moe.moe_dispatch(ids, T, k, E, counts, offsets, perm, inv, x_cur if xp is not None else None, cfg.H, xp,
                         wsx, wsb, st, stream)
        return l

    def ffn(l):
        moe.moe_expert_ffn_grouped(dc.struct, l, counts, offsets, perm, x_cur, xp, T, k, None, mode, y, wsx, wsb,
                                   st, stream)

    # prefill layers of one workload share a slot layout per layer; one graph per layer index
    graphs = {}
    with torch.cuda.stream(stream):
        for i in range(min(n, cfg.n_layers) if not decode_like else 1):
            l = prep(i)
            ffn(l)                                   # eager once: kernel attributes before capture
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                ffn(l)
            graphs[l] = g
    torch.cuda.synchronize()
    times, byts, flops, t_mixed = [], [], [], []
    with torch.cuda.stream(stream):
        for i in range(n):
            l = prep(i)
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            graphs[l].replay()
            b.record(stream)
            torch.cuda.synchronize()
            times.append(a.elapsed_time(b) / 1e3)
            cnt = counts.cpu().numpy().astype(np.float64)
            active = int((cnt > 0).sum())
            byts.append(ffn_bytes(cfg, active))
            flops.append(expert_ffn_flops(cfg))
            # per-expert roofline: each group takes the longer of its bytes at the HBM peak and its
            # FLOPs at the tensor peak (weights once + its rows' activations; 2*3*H*I FLOP per row)
            g_bytes = (cnt > 0) * cfg.expert_bytes + cnt * (cfg.H * 2 + cfg.H * 2) / cfg.k
            g_flops = cnt * 2.0 * 3 * cfg.H * cfg.I
            t_mixed.append(float(np.sum(np.maximum(g_bytes / (peaks["hbm_gbs"] * 1e9),
                                                   g_flops / (peaks["bf16_tflops"] * 1e12)))))
    t = float(np.mean(times))
    traffic = FFN_TRAFFIC.get(cfg.name)
    # both rooflines; the one whose time at peak is longer binds
    hbm = float(np.mean(byts)) / t / 1e9
    tc = float(np.mean(flops)) / t / 1e12
    t_hbm = float(np.mean(byts)) / (peaks["hbm_gbs"] * 1e9)
    t_tc = float(np.mean(flops)) / (peaks["bf16_tflops"] * 1e12)
    hbm_part = {"bound": "hbm", "achieved": round(hbm, 2), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(hbm / peaks["hbm_gbs"], 4), "peak_source": peaks["source"] + " (burst copy bandwidth)",
                "algorithmic_bytes_per_call": int(np.mean(byts)),
                "implementation_bytes_per_call": int(ffn_impl_bytes(cfg)),
                "bytes_note": "weights of the active experts once + token rows in + output rows out; "
                              "implementation bytes (gathered rows, h, fp32 expert rows) reported, not credited"}
    tc_part = {"bound": "tensor", "achieved": round(tc, 2), "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
               "frac": round(tc / peaks["bf16_tflops"], 4), "peak_source": peaks["source"] + " (burst cuBLAS bf16)",
               "flops_per_call": float(np.mean(flops))}
    main, other = (hbm_part, tc_part) if t_hbm >= t_tc else (tc_part, hbm_part)
    kernel = ("moe_expert_ffn_grouped (fused gate/up + down GEMV, one launch)" if decode_like and cfg.T <= 8
              else "moe_expert_ffn_grouped (tcgen05 gate/up + down GEMM, GEMV for groups of <= 2 rows)")
    out = {"kernel": kernel, **main, "traffic": traffic, "traffic_note": TRAFFIC_NOTE.get(cfg.name),
           "call_us": round(t * 1e6, 3),
           "mixed_roofline": {"min_us": round(float(np.mean(t_mixed)) * 1e6, 3),
                              "frac": round(float(np.mean(t_mixed)) / t, 4),
                              "note": "sum over experts of max(bytes / HBM peak, FLOP / bf16 peak), "
                                      "bytes = weights once + the group's share of token rows in and out"},
           "timing": "graph replay of the FFN call, L2 flushed before each",
           "other_roofline": other}
    return out


def measure_e2e(cfg, dc, layers, decode_like, stream, args, moe, torch, ws, ws_bytes, status, stats):
    """The public call with host buffers: pinned H2D of each layer's input
    block (decode: the step's token), moe_layer_forward, D2H of the output,
    and the host waits for the step's outputs; wall clock."""
    dev = ws.device
    T, H = cfg.T, cfg.H
    n = args.steps
    pin = lambda bits: torch.from_numpy(np.require(bits, requirements=["C", "W"]).view(np.int16)) \
        .view(torch.bfloat16).pin_memory()
    if decode_like:
        host_x = [[pin(gen.x_bits(cfg, 0, s))] for s in range(n)]
    else:
        blocks = [pin(gen.x_bits(cfg, l, 0)) for l in range(cfg.n_layers)]
        host_x = [blocks] * n
    host_out = torch.empty((T, H), dtype=torch.bfloat16).pin_memory()
    x_dev = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    dc.reset()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for i in range(n):
            for l in range(cfg.n_layers):
                x_dev.copy_(host_x[i][l], non_blocking=True)
                moe.moe_layer_forward(layers[l].struct, dc.struct, x_dev, T, out, cfg.phi_q16, cfg.min_fill,
                                      cfg.fill_policy, 1000 + l, FFN_MODES[args.ffn_mode](moe), None, ws, ws_bytes,
                                      status, stats, stream)
                host_out.copy_(out, non_blocking=True)
            stream.synchronize()
    el = time.perf_counter() - t0
    return {"value": round(n * T / el, 3), "unit": UNIT,
            "h2d_bytes_per_step": T * H * 2 * cfg.n_layers, "d2h_bytes_per_step": T * H * 2 * cfg.n_layers,
            "note": "moe_layer_forward per layer; host waits for each step's output"}


# ------------------------------------------------------------------ host-resident source pool
def c2c_rates(moe, torch, nbytes):
    """B_P (copy engine) and B_H (SMs in place) of pinned host memory, GB/s."""
    host = torch.empty(nbytes // 4, dtype=torch.int32).pin_memory()
    dev = torch.empty(nbytes // 4, dtype=torch.int32, device="cuda")
    prof = moe.moe_bench_bandwidth(host, dev, nbytes, 5, torch.cuda.Stream(), torch.cuda.Stream())
    return prof.b_p_gbs, prof.b_h_gbs


def run_host_pool_decode(args, dev, stream, moe, torch):
    """The decode workload with its staging pool (every expert) in pinned host
    memory read over NVLink-C2C: fills are copied into HBM cache slots and
    in-place experts evaluated from host memory, with plain loads.  One
    moe_layer_forward per step, events around it, L2 flushed between steps.
    The bytes that cross the link per step (each fill's expert and each
    in-place expert, once) over the step time, against the measured rate of
    SM reads of pinned host memory."""
    from moe_inputs.device import DeviceCache, DeviceLayer, to_dev_bf16
    cfg = CONFIGS["decode"]
    n_steps = args.warmup + args.steps
    dc = DeviceCache(cfg, dev, staging_host=True)
    dl = DeviceLayer(cfg, 0, dev)
    xs = [to_dev_bf16(gen.x_bits(cfg, 0, s), dev) for s in range(n_steps)]
    mode = FFN_MODES[args.ffn_mode](moe)
    nb = moe.moe_layer_workspace_size(dl.struct, dc.struct, cfg.T, mode)
    ws = torch.empty(nb, dtype=torch.uint8, device=dev)
    out = torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stats = torch.zeros(8, dtype=torch.int32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    call = lambda i: moe.moe_layer_forward(dl.struct, dc.struct, xs[i], cfg.T, out, cfg.phi_q16, cfg.min_fill,
                                           cfg.fill_policy, 1000, mode, None, ws, nb, status, stats, stream)
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            call(i)
            flush.zero_()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    st_host = torch.zeros((args.steps, 8), dtype=torch.int32).pin_memory()
    clocks = ClockSampler(dev.index)
    clocks.start()
    n0 = moe.moe_kernel_launch_count()
    with torch.cuda.stream(stream):
        for i in range(args.steps):
            ev[i][0].record(stream)
            call(args.warmup + i)
            ev[i][1].record(stream)
            st_host[i].copy_(stats, non_blocking=True)
            flush.zero_()
    torch.cuda.synchronize()
    launches = moe.moe_kernel_launch_count() - n0
    clk = clocks.stop()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    t = sum(step_ms) / 1e3
    sh = st_host.numpy()
    fields = moe.BIND_STATS_FIELDS
    n_fill = sh[:, fields.index("n_fill")].astype(np.float64)
    n_staged = sh[:, fields.index("n_staged")].astype(np.float64)
    link_bytes = float(np.sum((n_fill + n_staged) * cfg.expert_bytes))
    b_p, b_h = c2c_rates(moe, torch, cfg.expert_bytes)
    achieved = link_bytes / t / 1e9
    return {"value": round(args.steps * cfg.T / t, 3), "unit": UNIT, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(t * 1e3 / args.steps, 5),
            "step_ms_p10_p50_p90": [round(float(np.percentile(step_ms, q)), 5) for q in (10, 50, 90)],
            "config": dict(workload_config(cfg, 1), workload="decode_host_pool",
                           staging_pool="pinned host memory, read over NVLink-C2C with plain loads"),
            "device_status": int(status.cpu().numpy().view(np.uint32)[0]),
            "roofline": {"kernel": "whole step (fills and in-place experts cross the CPU-GPU link)", "bound": "c2c",
                         "achieved": round(achieved, 2), "peak": round(b_h, 2), "unit": "GB/s",
                         "frac": round(achieved / b_h, 4) if b_h > 0 else None,
                         "peak_source": "measured in this run: SMs reading pinned host memory in place "
                                        f"(B_H; the copy engine's B_P = {b_p:.1f} GB/s)",
                         "link_bytes_per_step": int(link_bytes / args.steps),
                         "fills_per_step": round(float(np.mean(n_fill)), 3),
                         "in_place_per_step": round(float(np.mean(n_staged)), 3)},
            "clocks": clk, "gpu_launches": int(launches), "gpu_launches_per_step": launches / args.steps}


def run_streamed_prefill(args, dev, stream, moe, torch):
    """The long-prefill stack (4 layers x 16384 tokens) with every expert in
    a pinned host pool: moe_prefill_double_buffered copies each layer's
    experts into one of two HBM layer buffers with the copy engine, the next
    layer's while this one computes (overlap), or layer by layer on demand.
    Both timed; the copy rate (the layers' expert bytes over the stack time)
    against the measured copy-engine rate B_P."""
    from moe_inputs.device import DeviceCache, DeviceLayer, to_dev_bf16
    cfg = CONFIGS["long_prefill"]
    L, E, T, H = cfg.n_layers, cfg.E, cfg.T, cfg.H
    src = DeviceCache(cfg, dev, staging_host=True)
    bufs = [[torch.empty((E,) + gen.bank_shape(cfg, b), dtype=torch.bfloat16, device=dev) for b in range(3)]
            for _ in range(2)]
    source = moe.moe_pool(*[t.data_ptr() for t in src.staging], L * E, 1)
    layer_buf = [moe.moe_pool(*[t.data_ptr() for t in bb], E) for bb in bufs]
    state = moe.moe_cache()
    table = torch.from_numpy(np.tile(np.arange(E, dtype=np.int32), L)).to(dev)
    owner = torch.arange(E, dtype=torch.int32, device=dev)
    stamp = torch.zeros(E, dtype=torch.int32, device=dev)
    clock = torch.zeros(1, dtype=torch.int32, device=dev)
    state.slot_table, state.owner, state.stamp, state.clock = (table.data_ptr(), owner.data_ptr(), stamp.data_ptr(),
                                                               clock.data_ptr())
    state.n_layers, state.E, state.H, state.I = L, E, H, cfg.I
    layers = [DeviceLayer(cfg, l, dev) for l in range(L)]
    xs = [to_dev_bf16(gen.x_bits(cfg, l, 0), dev) for l in range(L)]
    outs = [torch.empty((T, H), dtype=torch.bfloat16, device=dev) for _ in range(L)]
    mode = FFN_MODES[args.ffn_mode](moe)
    nb = moe.moe_layer_workspace_size(layers[0].struct, src.struct, T, mode)
    ws = torch.empty(nb, dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    copy_stream = torch.cuda.Stream(device=dev)
    steps = max(3, min(args.steps, 8))
    res = {}
    clocks = ClockSampler(dev.index)
    clocks.start()
    for overlap in (1, 0):
        def step():
            moe.moe_prefill_double_buffered([dl.struct for dl in layers], source, layer_buf, state, xs, T, outs, mode,
                                            overlap, ws, nb, status, stream, copy_stream)
        with torch.cuda.stream(stream):
            for _ in range(2):
                step()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        with torch.cuda.stream(stream):
            for i in range(steps):
                ev[i][0].record(stream)
                step()
                ev[i][1].record(stream)
        torch.cuda.synchronize()
        res[overlap] = float(np.mean([a.elapsed_time(b) for a, b in ev]))
    clk = clocks.stop()
    copied = float(L * E * cfg.expert_bytes)
    b_p, b_h = c2c_rates(moe, torch, cfg.expert_bytes)
    achieved = copied / (res[1] / 1e3) / 1e9
    return {"value": round(T / (res[1] / 1e3), 3), "unit": UNIT, "steps": steps, "warmup": 2,
            "ms_per_step": round(res[1], 4), "ms_per_step_on_demand": round(res[0], 4),
            "overlap_gain": round(res[0] / res[1], 4),
            "config": dict(workload_config(cfg, 1), workload="long_prefill_streamed",
                           source_pool="every expert of the 4 layers in pinned host memory",
                           layer_buffers="2 x 256 experts in HBM"),
            "device_status": int(status.cpu().numpy().view(np.uint32)[0]),
            "roofline": {"kernel": "copy engine, host pool -> HBM layer buffers (overlapped with the layers)",
                         "bound": "c2c", "achieved": round(achieved, 2), "peak": round(b_p, 2), "unit": "GB/s",
                         "frac": round(achieved / b_p, 4) if b_p > 0 else None,
                         "peak_source": "measured in this run: copy engine, pinned host -> HBM (B_P)",
                         "copied_bytes_per_step": int(copied)},
            "clocks": clk}


# ------------------------------------------------------------------ oracle arm
def oracle_step(cfg, step, state, O, n_tokens=None):
    """One step of the workload through the CPU fp64 oracle: router, top-k,
    residency bind, dispatch, per-expert SwiGLU, combine.  ``n_tokens``
    limits the step to the first tokens of the workload's block."""
    for layer in range(cfg.n_layers):
        s = step if cfg.steps > 1 else 0
        xb = gen.x_bits(cfg, layer, s)
        if n_tokens is not None:
            xb = xb[:n_tokens]
        x = gen.bf16_bits_to_f64(xb)
        res = O.layer_forward(x, gen.w_router(cfg, layer), gen.bias(cfg, layer, s), cfg.k,
                              lambda e: gen.expert_f64(cfg, layer, e), E=cfg.E)
        state, _ = O.bind(state, layer, res["ids"], cfg.E, cfg.phi_q16, cfg.min_fill, cfg.fill_policy, 1000 + layer)
    return state


def run_oracle_bounded(cfg, budget_s, max_steps=None):
    """Time the oracle on a bounded sample of the workload (whole steps)."""
    from oracle import moe_oracle as O
    n_tokens = None
    note = "whole steps"
    if cfg.T > 64:
        # a prefill block takes many minutes in fp64: time its first 16 tokens (same layer shape)
        n_tokens = 16
        note = f"the first 16 tokens of the {cfg.T}-token block, {cfg.n_layers} layer(s) each"
    state = gen.initial_cache(cfg)
    t0 = time.perf_counter()
    steps = 0
    while True:
        state = oracle_step(cfg, steps, state, O, n_tokens)
        steps += 1
        el = time.perf_counter() - t0
        if el >= budget_s or (max_steps and steps >= max_steps):
            break
    tokens = steps * (n_tokens or cfg.T)
    return {"value": round(tokens / el, 5), "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{steps} step(s) of '{cfg.name}' ({note}) in {el:.1f} s, fp64 numpy, " +
                      ("BLAS on one thread" if os.environ.get("OPENBLAS_NUM_THREADS") == "1" else "BLAS on all cores")}


SINGLE_THREAD_WORKLOADS = ("tiny", "decode", "batched_decode")
ONE_THREAD_ENV = {"OPENBLAS_NUM_THREADS": "1", "OMP_NUM_THREADS": "1", "MKL_NUM_THREADS": "1"}


def run_oracle_single_thread(budget_s):
    """The oracle on one host thread (BLAS pinned to one thread in a child
    process) on the three small workloads: {workload: cpu_baseline record}."""
    out = {}
    for name in SINGLE_THREAD_WORKLOADS:
        env = dict(os.environ, **ONE_THREAD_ENV)
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-only", "--workload", name,
                            "--cpu-baseline-s", str(budget_s)], capture_output=True, text=True, env=env,
                           cwd=ROOT, timeout=budget_s * 10 + 120)
        try:
            rec = json.loads(r.stdout.strip().splitlines()[-1])
            rec["cores"] = 1
            out[name] = rec
        except (ValueError, IndexError):
            out[name] = {"error": (r.stderr or "no output").strip().splitlines()[-1:]}
    return out


def run_host_record_child(name, args):
    """The host-pool decode record measured in a child process of its own: its
    12.9 GB source pool of pinned host memory is then the process's first
    large host allocation, as at a server's start.  Allocated after tens of GB
    of host arrays had come and gone in the same process, the pool was read
    over the CPU-GPU link ~30% slower (measured), which says nothing about the
    kernels."""
    cmd = [sys.executable, os.path.abspath(__file__), "--host-record", name, "--steps", str(args.steps),
           "--warmup", str(args.warmup), "--ffn-mode", args.ffn_mode]
    r = subprocess.run(cmd, capture_output=True, text=True, cwd=ROOT, timeout=1800)
    try:
        rec = json.loads(r.stdout.strip().splitlines()[-1])
    except (ValueError, IndexError):
        return {"error": (r.stderr or "no output").strip().splitlines()[-3:]}
    rec["process"] = "a child process of its own (the pool is its first large host allocation)"
    return rec


def run_host_record(args):
    """Child side of run_host_record_child: the one record, printed as JSON."""
    import torch
    import edge_moe_serving_gb300 as moe
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(device=dev)
    return run_host_pool_decode(args, dev, stream, moe, torch)


def run_reference(args, rank, world):
    cfg = CONFIGS[args.workload]
    if rank != 0:
        return None
    per_step_budget = max(0.5, args.reference_budget_s / max(1, args.steps + args.warmup))
    run_oracle_bounded(cfg, 0.0, max_steps=max(1, min(args.warmup, 1)))
    cb = run_oracle_bounded(cfg, per_step_budget * args.steps, max_steps=args.steps)
    return {"metric": METRIC, "value": cb["value"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": None, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(cfg, world, inputs_exceed_l2(cfg)), "impl": "reference", "cpu_baseline": cb,
            "e2e": {"value": cb["value"], "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def run_bw_profile(args):
    """moe_bench_bandwidth on one expert of the workload's shape (3*H*I bf16
    bytes) in pinned host memory: B_P = copy engine into HBM, B_H = the SMs
    reading it in place over NVLink-C2C, both alone and contended, and the
    derived phi (the phi_q16 argument of the split)."""
    import torch
    import edge_moe_serving_gb300 as moe
    cfg = CONFIGS[args.workload]
    nbytes = 3 * cfg.H * cfg.I * 2
    host = torch.empty(nbytes // 4, dtype=torch.int32).pin_memory()
    host.random_(-2 ** 31, 2 ** 31 - 1)
    dev = torch.empty(nbytes // 4, dtype=torch.int32, device="cuda")
    iters = max(args.steps, 3)
    prof = moe.moe_bench_bandwidth(host, dev, nbytes, iters, torch.cuda.Stream(), torch.cuda.Stream())
    out = {f: getattr(prof, f) for f, _ in moe.moe_bw_profile._fields_ if f != "read_checksum"}
    out = {k: (round(v, 4) if isinstance(v, float) else v) for k, v in out.items()}
    return {"metric": "bandwidth profile of the q* split", "workload": cfg.name, "bytes_per_copy": nbytes,
            "iters": iters, "unit": "GB/s", **out,
            "note": "B_P: cudaMemcpyAsync pinned host -> HBM; B_H: SMs reading the pinned host buffer in place"}


# ------------------------------------------------------------------ MXFP4 experts
MX_SEED = 77


def mx_expert_bytes(H, I):
    """Bytes of one MXFP4 expert: three banks of H*I codes (half a byte each)
    plus one scale byte per 32 inputs."""
    return 3 * (H * I // 2 + H * I // 32)


def run_fp4_prefill(args, dev, stream, moe, torch, fmt_name="mxfp4"):
    """The 8192-token prefill layer (or --fp4-workload) over FP4 experts: moe_layer_forward_fp4
    (router + top-k, residency bind, dispatch, the FP4 expert FFN on the
    tensor-core GEMM, combine) with all experts resident, phi = 0.  Steps
    back to back between one pair of CUDA events (prefill: each reads 3.6 GB
    of expert codes and scales, over twice the L2).  The FFN call alone (gather +
    gate/up + down GEMMs) is then timed after route and dispatch, with an L2
    flush before it."""
    from moe_inputs.device import DeviceLayer, Fp4Cache, to_dev_bf16
    peaks = load_peaks()
    cfg = CONFIGS[args.fp4_workload]
    fmt = moe.MOE_FP4_MXFP4 if fmt_name == "mxfp4" else moe.MOE_FP4_NVFP4
    T, H, E, k, I = cfg.T, cfg.H, cfg.E, cfg.k, cfg.I
    fc = Fp4Cache(cfg, fmt, MX_SEED, dev)
    dl = DeviceLayer(cfg, 0, dev)
    x = to_dev_bf16(gen.x_bits(cfg, 0, 0), dev)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    nb = moe.moe_layer_fp4_workspace_size(dl.struct, fc.struct, T)
    ws = torch.empty(nb, dtype=torch.uint8, device=dev)

    def step():
        moe.moe_layer_forward_fp4(dl.struct, fc.struct, x, T, out, 0, 1, 0, 0, ws, nb, status, None, stream)

    with torch.cuda.stream(stream):
        step()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    torch.cuda.synchronize()
    clocks = ClockSampler(dev.index)
    clocks.start()
    n0 = moe.moe_kernel_launch_count()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    launches = moe.moe_kernel_launch_count() - n0
    step_s = e0.elapsed_time(e1) / 1e3 / args.steps

    # the FFN call alone, after route and dispatch, L2 flushed before it
    R = T * k
    i32 = lambda n: torch.empty(max(n, 1), dtype=torch.int32, device=dev)
    ids, counts, offsets, perm, inv = i32(R), i32(E), i32(E + 1), i32(R), i32(R)
    w = torch.empty(R, dtype=torch.float32, device=dev)
    y = torch.empty((R, H), dtype=torch.float32, device=dev)
    nr, nd = moe.moe_route_topk_workspace_size(T, H, E), moe.moe_dispatch_workspace_size(T, k, E)
    nf = (moe.moe_expert_ffn_mxfp4_workspace_size if fmt == moe.MOE_FP4_MXFP4 else
          moe.moe_expert_ffn_nvfp4_workspace_size)(T, k, H, I)
    ws_r, ws_d, ws_f = (torch.empty(max(n, 256), dtype=torch.uint8, device=dev) for n in (nr, nd, nf))
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    c, b = fc.struct.cache, fc.struct.staging   # both pools: experts the slot table binds to the staging pool included
    if fmt == moe.MOE_FP4_MXFP4:
        pool = moe.moe_pool_mxfp4(c.gate_q, c.gate_s, c.up_q, c.up_s, c.down_q, c.down_s, c.n_slots, 0)
        staging = moe.moe_pool_mxfp4(b.gate_q, b.gate_s, b.up_q, b.up_s, b.down_q, b.down_s, b.n_slots, 0)
        ffn_call = moe.moe_expert_ffn_mxfp4
    else:
        pool, staging = c, b
        ffn_call = moe.moe_expert_ffn_nvfp4
    with torch.cuda.stream(stream):
        moe.moe_route_topk(x, T, H, dl.w_router, dl.bias, E, k, ids, w, None, ws_r, nr, status, stream)
        moe.moe_dispatch(ids, T, k, E, counts, offsets, perm, inv, None, H, None, ws_d, nd, status, stream)
    fev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    with torch.cuda.stream(stream):
        for i in range(args.warmup + args.steps):
            flush.zero_()
            if i >= args.warmup:
                fev[i - args.warmup][0].record(stream)
            ffn_call(pool, staging, fc.table, cfg.n_layers, 0, E, H, I, counts, offsets, perm, x, T, k, y, ws_f, nf,
                     status, stream)
            if i >= args.warmup:
                fev[i - args.warmup][1].record(stream)
    torch.cuda.synchronize()
    ffn_s = sum(a.elapsed_time(b) for a, b in fev) / 1e3 / args.steps
    dev_status = int(status.cpu().numpy().view(np.uint32)[0])
    fl = expert_ffn_flops(cfg)
    tf = fl / ffn_s / 1e12
    sb = 32 if fmt == moe.MOE_FP4_MXFP4 else 16
    byts = 3 * E * (H * I // 2 + H * I // sb) + 2 * T * H * 2   # every expert's codes and scales, x in, out
    step_fl = fl + router_flops(cfg)
    return {"value": round(T / step_s, 3), "unit": UNIT, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(step_s * 1e3, 5),
            "dtype": f"{fmt_name} weights expanded to bf16 in shared memory, bf16 activations, fp32 accumulation",
            "config": {"workload": f"{cfg.name}_{fmt_name}", "tokens_per_layer_call": T, "hidden": H, "experts": E,
                       "top_k": k, "intermediate": I, "residency": f"all {E} experts resident, phi = 0",
                       "l2": "inputs larger than L2 (%.1f GB of codes and scales per step), steps back to back"
                             % (byts / 1e9),
                       "launch": "moe_layer_forward_fp4, direct launches"},
            "device_status": dev_status,
            "roofline": {"kernel": "fp4_gemm_kernel (gate/up + down) with the token-row gather: the FFN call",
                         "bound": "tensor", "achieved": round(tf, 2), "peak": peaks["bf16_tflops"],
                         "unit": "TFLOP/s", "frac": round(tf / peaks["bf16_tflops"], 4),
                         "peak_source": peaks["source"] + " (burst cuBLAS bf16; the MMAs are bf16)",
                         "flops_per_call": fl, "call_us": round(ffn_s * 1e6, 3),
                         "traffic": FP4_TRAFFIC.get(f"prefill_{fmt_name}") if cfg.name == "prefill" else None,
                         "traffic_note": FP4_TRAFFIC_NOTE.get(f"prefill_{fmt_name}"),
                         "other_roofline": {"bound": "hbm", "achieved": round(byts / ffn_s / 1e9, 2),
                                            "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                            "frac": round(byts / ffn_s / 1e9 / peaks["hbm_gbs"], 4),
                                            "algorithmic_bytes_per_call": byts},
                         "timing": "CUDA events around the FFN call, L2 flushed before each"},
            "step_roofline": {"bound": "tensor", "achieved": round(step_fl / step_s / 1e12, 2),
                              "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                              "frac": round(step_fl / step_s / 1e12 / peaks["bf16_tflops"], 4),
                              "flops_per_step": step_fl},
            "clocks": clk, "gpu_launches": int(launches), "gpu_launches_per_step": launches / args.steps}


def oracle_mx_step(cfg, step, O):
    x = gen.bf16_bits_to_f64(gen.x_bits(cfg, 0, step))
    ids, w = O.select_topk(O.router_logits(x, gen.w_router(cfg), gen.bias(cfg)), cfg.k)
    out = np.zeros((x.shape[0], cfg.H))
    for t in range(x.shape[0]):
        for j, e in enumerate(ids[t]):
            W = O.mx_expert_weights(*gen.mx_expert(MX_SEED, 0, int(e), cfg.H, cfg.I))
            out[t] += w[t, j] * O.swiglu_expert(x[t][None, :], *W)[0]
    return out


def run_fp4_decode(args, dev, stream, moe, torch, fmt_name="mxfp4"):
    """The decode workload (one token per step, 256 experts, top-6, a 95-slot
    LRU cache pool, every miss filled) with FP4 expert banks: one
    moe_layer_forward_fp4 call per step, which runs the whole layer as one
    cooperative kernel.  A step reads about 80 MB of expert codes and scales
    (under twice the L2), so each step is timed between its own CUDA events
    after a 256 MB L2-flush write.  Roofline: the method's bytes of the step
    (distinct routed experts' codes and scales, one more expert written per
    fill, the router weights, the token row in and the output row out) over
    the step time."""
    from moe_inputs.device import DeviceLayer, Fp4Cache, to_dev_bf16
    peaks = load_peaks()
    cfg = CONFIGS[args.fp4_decode_workload]
    fmt = moe.MOE_FP4_MXFP4 if fmt_name == "mxfp4" else moe.MOE_FP4_NVFP4
    T, H, E, k, I = cfg.T, cfg.H, cfg.E, cfg.k, cfg.I
    n_steps = args.warmup + args.steps
    fc = Fp4Cache(cfg, fmt, MX_SEED, dev)
    dl = DeviceLayer(cfg, 0, dev)
    xs = [to_dev_bf16(gen.x_bits(cfg, 0, s), dev) for s in range(n_steps)]
    out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stats = torch.zeros((n_steps, 8), dtype=torch.int32, device=dev)
    nb = moe.moe_layer_fp4_workspace_size(dl.struct, fc.struct, T)
    ws = torch.empty(nb, dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def step(i, st=None):
        moe.moe_layer_forward_fp4(dl.struct, fc.struct, xs[i], T, out, cfg.phi_q16, cfg.min_fill, cfg.fill_policy,
                                  1000, ws, nb, status, stats[i] if st is None else st, stream)

    with torch.cuda.stream(stream):
        step(0)
    torch.cuda.synchronize()
    fc.reset()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            step(i)
            flush.zero_()
    torch.cuda.synchronize()
    clocks = ClockSampler(dev.index)
    clocks.start()
    n0 = moe.moe_kernel_launch_count()
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for i in range(args.steps):
            ev[i][0].record(stream)
            step(args.warmup + i)
            ev[i][1].record(stream)
            flush.zero_()
    torch.cuda.synchronize()
    bracket_s = time.perf_counter() - t0
    clk = clocks.stop()
    launches = moe.moe_kernel_launch_count() - n0
    step_ms = [a.elapsed_time(b) for a, b in ev]
    dev_status = int(status.cpu().numpy().view(np.uint32)[0])
    st = stats[args.warmup:].cpu().numpy().astype(np.float64)
    sb = 32 if fmt == moe.MOE_FP4_MXFP4 else 16
    xb = 3 * (H * I // 2 + H * I // sb) + (12 if fmt == moe.MOE_FP4_NVFP4 else 0)   # one FP4 expert's bytes
    method = st[:, 0] * xb + E * H * 4 + 2 * T * H * 2
    fills = st[:, 4] * xb
    total_s = sum(step_ms) / 1e3
    achieved = float(np.sum(method + fills)) / total_s / 1e9

    # end to end: the public call with the token row from pinned host memory, the output read back
    x_host = [x.cpu().pin_memory() for x in xs[:args.steps]]
    out_host = torch.empty((T, H), dtype=torch.bfloat16).pin_memory()
    x_in = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    fc.reset()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for i in range(args.steps):
            x_in.copy_(x_host[i], non_blocking=True)
            moe.moe_layer_forward_fp4(dl.struct, fc.struct, x_in, T, out, cfg.phi_q16, cfg.min_fill,
                                      cfg.fill_policy, 1000, ws, nb, status, stats[0], stream)
            out_host.copy_(out, non_blocking=True)
            stream.synchronize()
    e2e_s = time.perf_counter() - t0
    return {"value": round(args.steps * T / total_s, 3), "unit": UNIT, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(total_s * 1e3 / args.steps, 5),
            "step_ms_p10_p50_p90": [round(float(np.percentile(step_ms, q)), 5) for q in (10, 50, 90)],
            "bracket_ms_per_step": round(bracket_s * 1e3 / args.steps, 5),
            "dtype": f"{fmt_name} weights, bf16 activations",
            "config": {"workload": f"{cfg.name}_{fmt_name}", "tokens_per_layer_call": T, "hidden": H, "experts": E,
                       "top_k": k, "intermediate": I, "cache_slots": cfg.cache_slots, "phi_q16": cfg.phi_q16,
                       "fill_policy": "lowest_id", "routing_bias": cfg.bias,
                       "l2": "flushed between steps (256 MB write)",
                       "launch": "moe_layer_forward_fp4 per step (the whole layer in one cooperative kernel)"},
            "device_status": dev_status,
            "roofline": {"kernel": "decode_fp4_kernel (the whole step)", "bound": "hbm",
                         "achieved": round(achieved, 2), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(achieved / peaks["hbm_gbs"], 4),
                         "traffic": FP4_TRAFFIC.get(f"decode_{fmt_name}") if cfg.name == "decode" else None,
                         "traffic_note": FP4_TRAFFIC_NOTE.get(f"decode_{fmt_name}"),
                         "peak_source": peaks["source"] + " (burst copy bandwidth)",
                         "algorithmic_bytes_per_step": int(np.mean(method + fills)),
                         "fill_bytes_per_step": int(np.mean(fills)), "fills_per_step": round(float(np.mean(st[:, 4])), 3),
                         "timing": "CUDA events around each step (the kernel and its barrier-word reset)"},
            "clocks": clk,
            "e2e": {"value": round(args.steps * T / e2e_s, 3), "unit": UNIT, "h2d_bytes_per_step": T * H * 2,
                    "d2h_bytes_per_step": T * H * 2,
                    "note": "moe_layer_forward_fp4 per step; host waits for each step's output"},
            "gpu_launches": int(launches), "gpu_launches_per_step": launches / args.steps}


def run_mx(args):
    """Decode step with MXFP4 experts: router + top-k, dispatch, the MXFP4
    expert FFN and the combine, each a C-ABI call, captured in one graph.
    All 256 experts are resident (identity slot table), so there is no bind."""
    import torch
    import edge_moe_serving_gb300 as moe
    from moe_inputs.device import MxPool, to_dev, to_dev_bf16

    cfg = CONFIGS["decode"]
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    peaks = load_peaks()
    T, H, E, k, I = 1, cfg.H, cfg.E, cfg.k, cfg.I
    n_steps = args.warmup + args.steps
    stream = torch.cuda.Stream(device=dev)
    pool = MxPool(E, H, I, {}, dev)
    for e in range(E):
        pool.set(e, gen.mx_expert(MX_SEED, 0, e, H, I))
    table = torch.arange(E, dtype=torch.int32, device=dev)
    wr = to_dev(gen.w_router(cfg), dev)
    bias = to_dev(gen.bias(cfg), dev)
    xs = [to_dev_bf16(gen.x_bits(cfg, 0, s), dev) for s in range(n_steps)]
    i32 = lambda n: torch.empty(max(n, 1), dtype=torch.int32, device=dev)
    ids, counts, offsets, perm, inv = i32(T * k), i32(E), i32(E + 1), i32(T * k), i32(T * k)
    w = torch.empty(T * k, dtype=torch.float32, device=dev)
    y = torch.empty((T * k, H), dtype=torch.float32, device=dev)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    x_in = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    nr, nd, nm = (moe.moe_route_topk_workspace_size(T, H, E), moe.moe_dispatch_workspace_size(T, k, E),
                  moe.moe_expert_ffn_mxfp4_workspace_size(T, k, H, I))
    ws_r, ws_d, ws_m = (torch.empty(max(n, 256), dtype=torch.uint8, device=dev) for n in (nr, nd, nm))
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def front(s):
        moe.moe_route_topk(x_in, T, H, wr, bias, E, k, ids, w, None, ws_r, nr, status, s)
        moe.moe_dispatch(ids, T, k, E, counts, offsets, perm, inv, None, H, None, ws_d, nd, status, s)

    def ffn(s):
        moe.moe_expert_ffn_mxfp4(pool.struct, None, table, 1, 0, E, H, I, counts, offsets, perm, x_in, T, k, y,
                                 ws_m, nm, status, s)

    def step(s):
        front(s)
        ffn(s)
        moe.moe_combine(y, w, T, k, H, out, None, status, s)

    with torch.cuda.stream(stream):
        x_in.copy_(xs[0])
        step(stream)   # eager: kernel attributes and grid caches before capture
    torch.cuda.synchronize()
    graphs = {}
    n0 = moe.moe_kernel_launch_count()
    for name, body in (("step", step), ("front", front), ("ffn", ffn)):
        graphs[name] = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graphs[name], stream=stream):
            body(stream)
        if name == "step":
            kernels_per_step = moe.moe_kernel_launch_count() - n0
    torch.cuda.synchronize()

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    with torch.cuda.stream(stream):
        for s in range(args.warmup):
            x_in.copy_(xs[s])
            graphs["step"].replay()
            flush.zero_()
    torch.cuda.synchronize()
    clocks = ClockSampler(dev.index)
    clocks.start()
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for i in range(args.steps):
            x_in.copy_(xs[args.warmup + i])
            ev[i][0].record(stream)
            graphs["step"].replay()
            ev[i][1].record(stream)
            flush.zero_()
    torch.cuda.synchronize()
    bracket_s = time.perf_counter() - t0
    clk = clocks.stop()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    # the expert FFN alone (its two kernels), weights cold: route + dispatch, flush, then the FFN
    fev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    with torch.cuda.stream(stream):
        for i in range(args.steps):
            x_in.copy_(xs[args.warmup + i])
            graphs["front"].replay()
            flush.zero_()
            fev[i][0].record(stream)
            graphs["ffn"].replay()
            fev[i][1].record(stream)
    torch.cuda.synchronize()
    ffn_ms = [a.elapsed_time(b) for a, b in fev]
    dev_status = int(status.cpu().numpy().view(np.uint32)[0])

    # end to end: eager public calls, x from pinned host memory, output read back every step
    x_host = [gen_x.cpu().pin_memory() for gen_x in xs[:args.steps]]
    out_host = torch.empty((T, H), dtype=torch.bfloat16).pin_memory()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for i in range(args.steps):
            x_in.copy_(x_host[i], non_blocking=True)
            step(stream)
            out_host.copy_(out, non_blocking=True)
            stream.synchronize()
    e2e_s = time.perf_counter() - t0

    step_s = sum(step_ms) / 1e3
    ffn_avg_s = sum(ffn_ms) / 1e3 / args.steps
    alg = T * k * mx_expert_bytes(H, I)   # six distinct experts per step (one token)
    achieved = alg / ffn_avg_s / 1e9
    res = {
        "metric": METRIC, "value": round(args.steps * T / step_s, 3), "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_s * 1e3 / args.steps, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "mxfp4 weights, bf16 activations",
        "data": "synthetic",
        "config": {"workload": "decode_mxfp4", "tokens_per_layer_call": T, "hidden": H, "experts": E, "top_k": k,
                   "intermediate": I, "expert_format": "MXFP4 (FP4 E2M1 codes, E8M0 scale per 32 inputs)",
                   "residency": "all experts resident (no bind step)", "routing_bias": "zipf",
                   "l2": "flushed between steps (256 MB write)", "parallelism": "replicas x1",
                   "graph": "one CUDA graph replay per step"},
        "impl": "ours",
        "step_ms_p10_p50_p90": [round(float(np.percentile(step_ms, q)), 5) for q in (10, 50, 90)],
        "bracket_ms_per_step": round(bracket_s * 1e3 / args.steps, 5),
        "device_status": dev_status,
        "roofline": {"kernel": "mx_ring_kernel (the expert FFN call: gate/up and down in one weight-streaming launch)",
                     "bound": "hbm",
                     "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(achieved / peaks["hbm_gbs"], 3), "traffic": MX_TRAFFIC,
                     "traffic_note": "ncu capture of mx_ring_kernel on this call (dram bytes per second x duration)",
                     "peak_source": f"{peaks['source']} (burst copy bandwidth)",
                     "algorithmic_bytes_per_call": alg, "ffn_us": round(ffn_avg_s * 1e6, 3),
                     "timing": "CUDA events around the FFN graph (counter reset + one kernel), L2 flushed before "
                               "each call"},
        "clocks": clk,
        "e2e": {"value": round(args.steps * T / e2e_s, 3), "unit": UNIT, "h2d_bytes_per_step": T * H * 2,
                "d2h_bytes_per_step": T * H * 2,
                "note": "four public calls per step, not graph-captured; host waits for each step's output"},
        "gpu_launches": kernels_per_step * args.steps,
        "gpu_launches_per_step": kernels_per_step,
    }
    if not args.no_cpu_baseline:
        from oracle import moe_oracle as O
        t0, n = time.perf_counter(), 0
        while n < 2 or (time.perf_counter() - t0 < args.cpu_baseline_s and n < args.steps):
            oracle_mx_step(cfg, n, O)
            n += 1
        el = time.perf_counter() - t0
        res["cpu_baseline"] = {"value": round(n * T / el, 5), "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                               "sample": f"{n} decode step(s) with MXFP4 experts in {el:.1f} s, fp64 numpy"}
    return res


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=32)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="decode", choices=sorted(CONFIGS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-baseline-s", type=float, default=15.0)
    ap.add_argument("--reference-budget-s", type=float, default=120.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ffn-mode", default="auto", choices=sorted(FFN_MODES),
                    help="expert-FFN kernel choice passed to moe_layer_forward (default: auto)")
    ap.add_argument("--mxfp4", action="store_true",
                    help="decode step with MXFP4 expert banks (route, dispatch, MXFP4 FFN, combine) instead")
    ap.add_argument("--bw-profile", action="store_true",
                    help="print the bandwidth profile of the q* split (B_P, B_H, contended pair, phi) instead")
    ap.add_argument("--extra", default=None,
                    help="comma-separated workloads measured as sub-records of the line "
                         f"(default for the decode workload: {EXTRA_DEFAULT}; 'none' for none)")
    ap.add_argument("--oracle-only", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--host-record", default=None, choices=["decode_host_pool"], help=argparse.SUPPRESS)
    ap.add_argument("--fp4-decode-workload", default="decode", choices=sorted(CONFIGS),
                    help="the layer shape of the decode_mxfp4 / decode_nvfp4 records (decode_profile: a small case "
                         "for profiling)")
    ap.add_argument("--fp4-workload", default="prefill", choices=sorted(CONFIGS),
                    help="the layer shape of the prefill_mxfp4 / prefill_nvfp4 records (prefill_profile: a small "
                         "case for profiling)")
    args = ap.parse_args()
    if args.extra is None:
        # the sub-records are one GPU's measurements: at N > 1 every rank would run them at once (the
        # streamed stack alone pins 51.5 GB of host memory per rank), so the scaled runs carry the main record
        single = int(os.environ.get("WORLD_SIZE", "1")) == 1
        args.extra = EXTRA_DEFAULT if args.workload == "decode" and single else "none"
    if args.oracle_only:
        # child process of run_oracle_single_thread: the oracle alone, as its environment sets the threads
        print(json.dumps(run_oracle_bounded(CONFIGS[args.workload], args.cpu_baseline_s)))
        return
    if args.warmup < 3:
        args.warmup = 3
    if args.host_record:
        # child process of run_host_record_child
        print(json.dumps(run_host_record(args)))
        return
    if args.bw_profile:
        print(json.dumps(run_bw_profile(args)))
        return
    if args.mxfp4:
        # one GPU's measurement: under torchrun, rank 0 alone runs and prints it
        if int(os.environ.get("RANK", "0")) == 0:
            print(json.dumps(run_mx(args)))
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        res = run_reference(args, rank, world)
        if res is not None:
            print(json.dumps(res))
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        dist.init_process_group("nccl")
    res = run_ours(args, rank, world)
    if rank == 0:
        if not args.no_cpu_baseline:
            res["cpu_baseline"] = run_oracle_bounded(CONFIGS[args.workload], args.cpu_baseline_s)
            res["cpu_baseline"]["single_thread"] = run_oracle_single_thread(min(args.cpu_baseline_s, 5.0))
        print(json.dumps(res))
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
