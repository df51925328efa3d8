#!/usr/bin/env python3
"""Benchmark of compressed-KV-cache attention on GB300.

One step = the whole hot path over one synthetic prompt of the workload:
prefill compression of every layer (scoring, pooling, top-k, gather +
quantize + pack, window init), then every decode step over all layers (append
with group flushes, split-K decode attention). Inputs are resident in HBM before
the timed region; L2 is flushed (a read of 256 MiB, outside the measured kernel
intervals) before every decode step, as the rest of a model would between two
tokens; the prefill inputs (4.3 GB for the default workload) exceed L2.

Prints one JSON line (rank 0). `--impl reference` times the CPU oracle instead.
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

METRIC = "compressed-KV decode tokens/s, cache GB/s vs HBM peak; compress ms/layer"
UNIT = "tokens/s"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", type=int, default=5,
                    help="the headline workload (default 5: long context, 2-bit)")
    ap.add_argument("--legs", default="3,4",
                    help="comma-separated workloads measured after the headline one "
                         "(decode GB/s and compression ms/layer each); empty for none")
    ap.add_argument("--decode-steps", type=int, default=None)
    ap.add_argument("--layers", type=int, default=None,
                    help="use only the first N layers (small cases for profiler captures)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-sinks", action="store_true",
                    help="skip the compression pass with the sink + recent selection")
    ap.add_argument("--no-exact16", action="store_true",
                    help="skip the decode launches over a 16-bit (unquantized) cache")
    ap.add_argument("--no-acumul", action="store_true",
                    help="skip the compression pass scored by the full-prompt cumulated attention")
    return ap.parse_args()


def rank_info():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def max_over_ranks(values, world, device=None):
    """Element-wise maximum of `values` (floats) over the ranks of the process group
    (the slowest rank decides a step's time); identity when world == 1."""
    if world <= 1:
        return [float(v) for v in values]
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def job_throughput(tokens_per_rank, world, dec_ms_max):
    """Whole-job decode tokens/s: every rank decodes its own replica of the workload
    (weak scaling), in the slowest rank's time."""
    return tokens_per_rank * world / (dec_ms_max / 1e3)


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


def workload_desc(spec, S):
    sched = (f"pyramid avg {spec.avg_budget} depth {spec.pyramid_depth}"
             if spec.schedule == "pyramid" else
             (f"uniform {spec.avg_budget}" if spec.schedule == "uniform" else "no eviction"))
    return (f"{spec.name}: {spec.n_layers} layers, {spec.n_q_heads}/{spec.n_kv_heads} heads, "
            f"d{spec.head_dim}, batch {spec.batch}, prompt {spec.prompt_len}, {sched}, "
            f"obs {spec.obs_window}, pool {spec.pool_kernel}, {spec.bits}-bit g{spec.group_size}, "
            f"bf16 window {spec.window_len}, {S} decode steps")


# ---------------------------------------------------------------- clocks
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, enabled=True):
        self.proc = None
        self.path = f"/tmp/kvc_clocks_{os.getpid()}.csv"
        if enabled:
            try:
                self.f = open(self.path, "w")
                self.proc = subprocess.Popen(
                    ["nvidia-smi", "-i", str(index), f"--query-gpu={self.QUERY}",
                     "--format=csv,noheader,nounits", "-lms", "50"],
                    stdout=self.f, stderr=subprocess.DEVNULL)
            except Exception:
                self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx = float(parts[2])
                except ValueError:
                    continue
                for nm, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(nm)
        if not sm:
            return None
        loaded = [s for s in sm if mx and s > 0.5 * mx] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- oracle (CPU)
def oracle_sample(spec, n_layers_sample=2, n_steps=8):
    """Time the CPU oracle on a bounded sample of the workload.

    Returns (compress seconds per layer, decode seconds per token per layer, text).
    """
    import synth
    from oracle import OracleCache
    budgets = _budgets_host(spec)
    t_comp, t_dec, layers = 0.0, 0.0, list(range(n_layers_sample))
    for layer in layers:
        x = synth.layer_inputs(spec, layer, device="cpu")
        k = x["k"].float().double().numpy()
        v = x["v"].float().double().numpy()
        q = x["q_obs"].float().double().numpy() if "q_obs" in x else None
        oc = OracleCache(spec.batch, spec.n_q_heads, spec.n_kv_heads, spec.head_dim, spec.bits,
                         spec.group_size, spec.window_len)
        ns = spec.prompt_len - spec.obs_window
        t0 = time.perf_counter()
        oc.prefill(k, v, spec.obs_window, budget=budgets[layer] if budgets[layer] < ns else None,
                   q_obs=q, pool_kernel=spec.pool_kernel)
        t_comp += time.perf_counter() - t0
        for t in range(n_steps):
            dx = synth.decode_inputs(spec, layer, t, device="cpu")
            args = [dx[n].float().double().numpy() for n in ("q", "k_new", "v_new")]
            t0 = time.perf_counter()
            oc.step(*args)
            t_dec += time.perf_counter() - t0
    text = (f"oracle on layers 0..{n_layers_sample - 1} (full prompt, all heads) + "
            f"{n_steps} decode steps each; extrapolated linearly to {spec.n_layers} layers")
    return t_comp / len(layers), t_dec / (len(layers) * n_steps), text


def _budgets_host(spec):
    from oracle import plan_budgets
    ns = spec.prompt_len - spec.obs_window
    if spec.schedule == "none":
        return [ns] * spec.n_layers
    return plan_budgets(spec.n_layers, spec.schedule, spec.avg_budget, spec.pyramid_depth,
                        spec.group_size, max_budget=ns)


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def cpu_model():
    """The host CPU as /proc/cpuinfo names it: its model name, else (Arm) the
    implementer and part codes; with the machine architecture."""
    import platform
    fields = {}
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                k, _, v = line.partition(":")
                k, v = k.strip().lower(), v.strip()
                if k in ("model name", "cpu implementer", "cpu part") and k not in fields:
                    fields[k] = v
    except Exception:
        pass
    if "model name" in fields:
        name = fields["model name"]
    elif "cpu part" in fields:
        name = f"implementer {fields.get('cpu implementer', '?')} part {fields['cpu part']}"
    else:
        name = "unknown"
    return f"{name} ({platform.machine()})"


def run_reference(args):
    rank, world, _ = rank_info()
    if rank != 0:
        return
    import synth
    spec = synth.workload(args.workload)
    S = args.decode_steps or spec.steps
    vals, comp, per_tok = [], [], []
    text = ""
    for i in range(args.warmup + args.steps):
        c, d, text = oracle_sample(spec, n_layers_sample=1, n_steps=4)
        if i >= args.warmup:
            per_token = d * spec.n_layers
            vals.append(spec.batch / per_token)
            comp.append(c * 1e3)
            per_tok.append(per_token)
    value = statistics.mean(vals)
    step_s = statistics.mean(comp) / 1e3 * spec.n_layers + statistics.mean(per_tok) * S
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": step_s * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64 (quantizer f32)", "data": "synthetic",
        "config": {"workload": workload_desc(spec, S)},
        "compress_ms_per_layer": statistics.mean(comp),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
                         "sample": text, "cpu": cpu_model()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- GPU arm
def kernel_hash(name):
    p = os.path.join(ROOT, "kv_cache_compression_snapkv_gb300", "csrc", name)
    with open(p, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def profiled_traffic(kernel_file):
    """DRAM bytes per launch of the dominant kernel, from the committed ncu summary
    `profiles/<kernel file stem>_traffic.txt` ("key: value" lines), if the kernel
    source is unchanged since the capture (else None)."""
    stem = os.path.splitext(kernel_file)[0]
    try:
        vals = {}
        with open(os.path.join(ROOT, "profiles", f"{stem}_traffic.txt")) as f:
            for line in f:
                if ":" in line and not line.lstrip().startswith("#"):
                    k, v = line.split(":", 1)
                    vals[k.strip()] = v.strip()
        if vals.get("source_sha256_16") != kernel_hash(kernel_file):
            return None
        return {"dram_bytes_per_launch": float(vals["dram_bytes_per_launch"])}
    except Exception:
        return None


def run_gpu(args):
    import torch
    import torch.distributed as dist
    rank, world, local = rank_info()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    import synth
    import kv_cache_compression_snapkv_gb300 as K

    spec = synth.workload(args.workload)
    S = args.decode_steps or spec.steps
    full_dims = K.dims_from_spec(spec, max_new_tokens=S)
    budgets = K.kvc_plan_budgets(full_dims, spec.schedule, spec.avg_budget, spec.pyramid_depth)
    if args.layers:     # the first N layers of the full model (with their budgets)
        import dataclasses
        spec = dataclasses.replace(spec, n_layers=min(args.layers, spec.n_layers))
        budgets = budgets[:spec.n_layers]
    L, B, Hq, Hk, D = spec.n_layers, spec.batch, spec.n_q_heads, spec.n_kv_heads, spec.head_dim
    dims = K.dims_from_spec(spec, max_new_tokens=S)
    dev = torch.device("cuda", local)

    # ---- inputs resident in HBM
    prompt = [synth.layer_inputs(spec, l, device=dev) for l in range(L)]
    qs, kns, vns = [], [], []
    for t in range(S):
        dx = synth.decode_inputs_layers(spec, t, range(L), device=dev)
        qs.append(dx["q"]); kns.append(dx["k_new"]); vns.append(dx["v_new"])
    out = torch.empty(L, B, Hq, D, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    cache = K.kvc_cache_create(dims, budgets)
    stream = torch.cuda.current_stream()
    ev = lambda: torch.cuda.Event(enable_timing=True)
    c0, c1 = ev(), ev()
    dev_ev = [(ev(), ev(), ev()) for _ in range(S)]
    block_bytes = 8 * D * (spec.bits + 1)

    dec_bytes = []   # algorithmic bytes of each decode-attention launch
    HOLD_CYCLES = 60_000_000 * max(1, S // 256)   # ~30 ms at 2 GHz per 256 decode steps

    def one_step(record_bytes=False):
        K.kvc_cache_reset(cache)
        # hold the device (outside every timed interval) while the host enqueues the
        # step: a decode call costs the host about as long as a flush + decode costs
        # the device, and a late enqueue would leave the device idle inside a timed
        # launch interval
        torch.cuda._sleep(HOLD_CYCLES)
        c0.record(stream)
        for l in range(L):
            x = prompt[l]
            K.kvc_prefill_compress(dims, budgets, l, x.get("q_obs"), x["k"], x["v"], cache=cache)
        c1.record(stream)
        for t in range(S):
            flush.max()          # evicts L2 with clean lines (a write would leave
                                 # dirty lines to be written back inside the timed kernel)
            e0, e1, e2 = dev_ev[t]
            e0.record(stream)
            e1.record(stream)
            K.kvc_decode_step(cache, 0, L, qs[t], kns[t], vns[t], out)
            e2.record(stream)
            if record_bytes:
                dec_bytes.append(decode_bytes(K, cache, spec))

    def collect():
        torch.cuda.synchronize()
        comp = c0.elapsed_time(c1)
        app = [dev_ev[t][0].elapsed_time(dev_ev[t][1]) for t in range(S)]
        att = [dev_ev[t][1].elapsed_time(dev_ev[t][2]) for t in range(S)]
        return comp, app, att

    one_step(record_bytes=True)
    collect()
    for _ in range(max(0, args.warmup - 1)):
        one_step()
        collect()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local, enabled=not args.no_clocks)
    n0 = K.kvc_launch_count()
    t_wall0 = time.perf_counter()
    comps, apps, atts = [], [], []
    for _ in range(args.steps):
        one_step()
        comp, app, att = collect()
        comps.append(comp); apps.append(app); atts.append(att)
    torch.cuda.synchronize()
    wall = (time.perf_counter() - t_wall0) / args.steps
    launches = K.kvc_launch_count() - n0
    clk = clocks.stop()
    if world > 1:
        dist.barrier()

    # the attention-sink + recent-token selection (4 sinks, no scoring): the same
    # layers compressed with it, outside the timed steps
    sink_ms = None
    if not args.no_sinks:
        cs0, cs1 = ev(), ev()
        sms = []
        for i in range(4):
            K.kvc_cache_reset(cache)
            cs0.record(stream)
            for l in range(L):
                x = prompt[l]
                K.kvc_prefill_sinks(cache, l, 4, x["k"], x["v"])
            cs1.record(stream)
            torch.cuda.synchronize()
            if i > 0:
                sms.append(cs0.elapsed_time(cs1))
        sink_ms = statistics.mean(sms) / L

    # the variance score of the last scored layer (the statistic behind Var-prop /
    # Var-inv budgets): one launch reading the layer's scores twice
    variance = None
    if any(b_ < spec.prompt_len - spec.obs_window for b_ in budgets):
        K.kvc_cache_reset(cache)
        for l in range(L):
            x = prompt[l]
            K.kvc_prefill_compress(dims, budgets, l, x.get("q_obs"), x["k"], x["v"],
                                   cache=cache)
        var = torch.empty(B, Hk, device=dev)
        v0, v1 = ev(), ev()
        for _ in range(3):
            K.kvc_score_variance(cache, var)
        # the device waits while the host enqueues the timed launches (a call costs the
        # host longer than the launch costs the device)
        torch.cuda._sleep(20_000_000)
        v0.record(stream)
        for _ in range(20):
            K.kvc_score_variance(cache, var)
        v1.record(stream)
        torch.cuda.synchronize()
        v_us = v0.elapsed_time(v1) * 1e3 / 20
        v_bytes = B * Hk * (spec.prompt_len - spec.obs_window) * 4 * 2
        variance = {"us_per_launch": v_us, "bytes": v_bytes,
                    "gbs": v_bytes / (v_us * 1e-6) / 1e9,
                    "note": "per-(sequence, kv head) variance of the last scored layer's "
                            "scores (two passes over them; they sit in L2)"}

    # selection by the full-prompt cumulated attention (every prompt query, un-normalised
    # column sums): the first two layers compressed with it, outside the timed steps
    acumul = attention = None
    if not args.no_acumul:
        LA = min(2, L)
        qfull = [synth.prompt_queries(spec, l, device=dev) for l in range(LA)]
        ca0, ca1 = ev(), ev()
        ams = []
        for i in range(4):
            K.kvc_cache_reset(cache)
            ca0.record(stream)
            for l in range(LA):
                x = prompt[l]
                K.kvc_prefill_acumul(cache, l, qfull[l], x["k"], x["v"])
            ca1.record(stream)
            torch.cuda.synchronize()
            if i > 0:
                ams.append(ca0.elapsed_time(ca1))
        a_ms = statistics.mean(ams) / LA
        # the method's flops: q.k over every causal (query, key) pair of every query head
        a_flops = 2 * D * B * Hq * spec.prompt_len * (spec.prompt_len + 1) // 2
        acumul = {"ms_per_layer": a_ms, "flops": a_flops, "layers": LA,
                  "tflops": a_flops / (a_ms / 1e3) / 1e12,
                  "note": "selection by MiniKV's full-prompt cumulated attention (key blocks of "
                          "128, running row maxima); two MMAs per tile (S and S^T) on the "
                          "tensor cores"}
        # the selective flash-attention: the same selection plus the prefill attention
        # output X_O of every query (one pass, three products per key tile)
        xo = torch.empty(B, Hq, spec.prompt_len, D, dtype=torch.bfloat16, device=dev)
        axs = []
        for i in range(4):
            K.kvc_cache_reset(cache)
            ca0.record(stream)
            for l in range(LA):
                x = prompt[l]
                K.kvc_prefill_attention(cache, l, qfull[l], x["k"], x["v"], xo)
            ca1.record(stream)
            torch.cuda.synchronize()
            if i > 0:
                axs.append(ca0.elapsed_time(ca1))
        x_ms = statistics.mean(axs) / LA
        # dense causal attention: q.k and p.v over every causal (query, key) pair
        x_flops = 4 * D * B * Hq * spec.prompt_len * (spec.prompt_len + 1) // 2
        attention = {"ms_per_layer": x_ms, "flops": x_flops, "layers": LA,
                     "tflops": x_flops / (x_ms / 1e3) / 1e12,
                     "note": "MiniKV's selective flash-attention: X_O (bf16) of every prompt "
                             "query plus the cumulated-attention selection and packing; flops "
                             "are those of dense causal attention (q.k and p.v); the kernel also "
                             "forms S^T for the fp32 column sums"}
        del qfull, xo

    # 16-bit storage (every kept token exact in the bf16 window), same selection and
    # budgets: decode launches over the exact cache, outside the timed steps
    exact16 = None
    if not args.no_exact16:
        import dataclasses
        S16 = min(32, S)
        R16 = (max(min(b_, spec.prompt_len - spec.obs_window) for b_ in budgets)
               + spec.obs_window + S16 + 31) // 32 * 32
        spec16 = dataclasses.replace(spec, bits=16, window_len=R16)
        dims16 = K.dims_from_spec(spec16, max_new_tokens=S16)
        cache16 = K.kvc_cache_create(dims16, budgets)
        for l in range(L):
            x = prompt[l]
            K.kvc_prefill_compress(dims16, budgets, l, x.get("q_obs"), x["k"], x["v"],
                                   cache=cache16)
        e16 = [(ev(), ev()) for _ in range(S16)]
        bytes16 = []
        for t in range(S16):
            tot = 0
            for l in range(L):
                info = K.kvc_layer_info_get(cache16, l)
                tot += B * Hk * (info["window_tokens"] + 1) * D * 2 * 2
            bytes16.append(tot + L * B * Hq * D * (2 + 4) + L * B * Hk * D * 2 * 2)
            flush.max()
            e16[t][0].record(stream)
            K.kvc_decode_step(cache16, 0, L, qs[t], kns[t], vns[t], out)
            e16[t][1].record(stream)
        torch.cuda.synchronize()
        us16 = statistics.mean(a.elapsed_time(b) for a, b in e16[3:]) * 1e3
        b16 = statistics.mean(bytes16[3:])
        exact16 = {"us_per_launch": us16, "bytes_per_launch": b16,
                   "gbs": b16 / (us16 * 1e-6) / 1e9, "window_len": R16,
                   "note": "bits=16: the kept tokens stay exact in the bf16 window"}
        cache16.close()

    comp_ms = statistics.mean(comps)
    dec_ms = statistics.mean([sum(a) + sum(b) for a, b in zip(apps, atts)])
    att_ms_all = [x for a in atts for x in a]
    att_ms = statistics.mean(att_ms_all)
    step_ms = comp_ms + dec_ms
    step_ms, dec_ms, comp_ms, att_ms = max_over_ranks([step_ms, dec_ms, comp_ms, att_ms], world,
                                                      device=dev)

    hbm, tc, peak_kind = peaks()
    tokens = B * S * world
    value = job_throughput(B * S, world, dec_ms)
    # decode attention: algorithmic bytes per launch / mean launch duration
    mean_bytes = statistics.mean(dec_bytes)
    dec_gbs = mean_bytes / (att_ms / 1e3) / 1e9
    # compression: algorithmic bytes and flops per layer
    ns = spec.prompt_len - spec.obs_window
    comp_bytes, comp_flops, comp_exps, t_roof, comp_bound = compress_roofline(spec, budgets,
                                                                              hbm, tc)
    comp_frac = t_roof / (comp_ms / 1e3)
    # sink + recent selection: kept rows read, packed groups and window rows written
    sink_bytes = 0
    for l in range(L):
        kept = min(budgets[l], ns)
        sink_bytes += (B * Hk * kept * D * 2 * 2 + B * Hk * (kept // 32) * block_bytes
                       + B * Hk * (kept % 32 + spec.obs_window) * D * 2 * 2 * 2)

    traffic = profiled_traffic("decode.cu")
    roofline = {"kernel": "decode_kernel (fused append + split-K decode attention, all layers "
                          "per launch)",
                "bound": "hbm", "achieved": dec_gbs, "peak": hbm, "unit": "GB/s",
                "frac": dec_gbs / hbm, "peak_source": peak_kind + " (burst copy)",
                "bytes_per_launch": mean_bytes,
                "traffic": traffic["dram_bytes_per_launch"] if traffic else None}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "int2 codes + bf16 window (fp16/bf16 mma, fp32 accumulate)",
        "data": "synthetic",
        "config": {"workload": workload_desc(spec, S),
                   "l2": "flushed (256 MiB read) before every decode step; prefill inputs exceed L2",
                   "decode_launch": (f"one fused launch per token (append + group flush + "
                                     f"split-K attention) for all {L} layers"),
                   "parallelism": f"replicas x{world}"},
        "decode_tokens_per_s": value,
        "cache_gbs": dec_gbs, "cache_frac_of_hbm": dec_gbs / hbm,
        "decode_attn_us_per_launch": att_ms * 1e3,
        "compress_ms_per_layer": comp_ms / L,
        "decode_16bit": None if exact16 is None else dict(
            exact16, frac=exact16["gbs"] / hbm),
        "score_variance": variance,
        "compress_acumul": None if acumul is None else dict(
            acumul, frac=acumul["tflops"] / tc),
        "prefill_attention": None if attention is None else dict(
            attention, frac=attention["tflops"] / tc),
        "compress_sinks": None if sink_ms is None else {
            "ms_per_layer": sink_ms, "bytes": sink_bytes,
            "frac": sink_bytes / (hbm * 1e9) / (sink_ms * L / 1e3),
            "note": "4 attention sinks + the most recent tokens within each layer's budget"},
        "compress_roofline": {"bytes": comp_bytes, "flops": comp_flops, "exps": comp_exps,
                              "bound": comp_bound, "t_roof_ms": t_roof * 1e3,
                              "frac": comp_frac},
        "wall_ms_per_step": wall * 1e3,
        "roofline": roofline,
        "gpu_launches": launches,
        "gpu_launches_per_step": launches / args.steps,
    }
    if clk:
        line["clocks"] = clk

    if not args.no_e2e:
        line["e2e"] = e2e_measure(K, spec, dims, budgets, cache, prompt, qs, kns, vns, S, dev)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # ~10 s of oracle work on the box's 16 host cores (2.7 s per long-context layer)
        c, d, text = oracle_sample(spec, n_layers_sample=4)
        per_token = d * L
        line["cpu_baseline"] = {"value": B / per_token, "unit": UNIT, "cores": cpu_cores(),
                                "kind": "oracle", "sample": text, "cpu": cpu_model(),
                                "compress_ms_per_layer": c * 1e3}
    cache.close()
    legs = [int(w) for w in args.legs.split(",") if w.strip()] if args.legs else []
    legs = [w for w in legs if w != args.workload]
    if legs and world == 1 and not args.layers:
        del prompt, qs, kns, vns, cache
        torch.cuda.empty_cache()
        line["legs"] = {str(w): run_leg(K, w, hbm, tc, dev, flush) for w in legs}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def decode_bytes(K, cache, spec):
    """Algorithmic bytes one decode launch over all layers reads and writes in the
    cache's current state (packed groups, window tokens incl. the new one, q, o,
    the new key/value)."""
    B, Hk, Hq, D, L = spec.batch, spec.n_kv_heads, spec.n_q_heads, spec.head_dim, spec.n_layers
    tot = 0
    for l in range(L):
        info = K.kvc_layer_info_get(cache, l)
        blk = 8 * D * (info["bits"] + 1) if info["bits"] != 16 else 0
        tot += B * Hk * (info["packed_tokens"] // 32 * blk + info["window_tokens"] * D * 4)
    return tot + L * B * Hq * D * (2 + 4) + L * B * Hk * D * 2 * 2


MUFU_PER_CLK_SM = 16   # exp2 results per clock per SM (special-function units, sm_100 family)


def mufu_peak():
    """exp2 results per second: the SFU rate per SM x SMs x the maximum SM clock."""
    import torch
    n_sm = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            mhz = float(json.load(f)["sm_max_mhz"])
    except Exception:
        mhz = 2070.0
    return MUFU_PER_CLK_SM * n_sm * mhz * 1e6


def compress_roofline(spec, budgets, hbm, tc):
    """Algorithmic bytes, flops and exponentials of compressing every layer, and the
    roofline time: the slowest of the three at its peak (HBM copy, bf16 tensor, SFU
    exp2). The scoring evaluates one exp2 per (observation row, key) in each of its two
    passes (row normalisers over all n keys, then the column sums over the n - alpha
    scored ones); the normalisers must be complete before any column sum."""
    B, Hk, Hq, D, L = spec.batch, spec.n_kv_heads, spec.n_q_heads, spec.head_dim, spec.n_layers
    block_bytes = 8 * D * (spec.bits + 1)
    ns = spec.prompt_len - spec.obs_window
    comp_bytes = comp_flops = comp_exps = 0
    for l in range(L):
        kept = min(budgets[l], ns)
        scored = kept < ns
        comp_bytes += (B * Hk * spec.prompt_len * D * 2 * (1 if scored else 2)
                       + (B * Hk * kept * D * 2 * 2 if scored else 0)
                       + B * Hk * (kept // 32) * block_bytes
                       + (B * Hq * spec.obs_window * D * 2 if scored else 0))
        comp_flops += 2 * B * Hq * spec.obs_window * spec.prompt_len * D if scored else 0
        comp_exps += B * Hq * spec.obs_window * (spec.prompt_len + ns) if scored else 0
    terms = {"hbm": comp_bytes / (hbm * 1e9), "tensor": comp_flops / (tc * 1e12)}
    if comp_exps:
        terms["sfu"] = comp_exps / mufu_peak()
    bound = max(terms, key=terms.get)
    return comp_bytes, comp_flops, comp_exps, terms[bound], bound


def run_leg(K, wid, hbm, tc, dev, flush):
    """One more workload, measured like the headline one: compression of every layer
    (CUDA events around each layer's call; the layer's inputs are generated just
    before, outside the timed interval, so that the largest workload need not hold
    its whole prompt), then every decode step (one launch over all layers, L2
    flushed before each, CUDA events around the launch)."""
    import torch
    import synth
    spec = synth.workload(wid)
    S = spec.steps
    L, B, Hq, D = spec.n_layers, spec.batch, spec.n_q_heads, spec.head_dim
    dims = K.dims_from_spec(spec, max_new_tokens=S)
    budgets = K.kvc_plan_budgets(dims, spec.schedule, spec.avg_budget, spec.pyramid_depth)
    stream = torch.cuda.current_stream()
    ev = lambda: torch.cuda.Event(enable_timing=True)
    cache = K.kvc_cache_create(dims, budgets)
    comp = []
    for rep_i in range(2):      # the first pass warms up
        K.kvc_cache_reset(cache)
        tot = 0.0
        for l in range(L):
            x = synth.layer_inputs(spec, l, device=dev)
            torch.cuda.synchronize()
            a, b = ev(), ev()
            a.record(stream)
            K.kvc_prefill_compress(dims, budgets, l, x.get("q_obs"), x["k"], x["v"], cache=cache)
            b.record(stream)
            torch.cuda.synchronize()
            tot += a.elapsed_time(b)
            del x
        comp.append(tot)
    comp_ms = comp[-1]
    out = torch.empty(L, B, Hq, D, device=dev)
    att, nbytes = [], []
    for t in range(S):
        dx = synth.decode_inputs_layers(spec, t, range(L), device=dev)
        nbytes.append(decode_bytes(K, cache, spec))
        flush.max()
        a, b = ev(), ev()
        a.record(stream)
        K.kvc_decode_step(cache, 0, L, dx["q"], dx["k_new"], dx["v_new"], out)
        b.record(stream)
        torch.cuda.synchronize()
        att.append(a.elapsed_time(b))
        del dx
    K.kvc_check_device(cache)
    cache.close()
    warm = 3 if S > 6 else 0    # the first launches pay one-time set-up
    att_ms = statistics.mean(att[warm:])
    mean_bytes = statistics.mean(nbytes[warm:])
    gbs = mean_bytes / (att_ms / 1e3) / 1e9
    cb, cf, ce, t_roof, cbound = compress_roofline(spec, budgets, hbm, tc)
    return {"workload": workload_desc(spec, S),
            "decode_tokens_per_s": B * S / (sum(att) / 1e3),
            "decode_attn_us_per_launch": att_ms * 1e3,
            "bytes_per_launch": mean_bytes, "cache_gbs": gbs, "cache_frac_of_hbm": gbs / hbm,
            "compress_ms_per_layer": comp_ms / L,
            "compress_roofline": {"bytes": cb, "flops": cf, "exps": ce, "bound": cbound,
                                  "t_roof_ms": t_roof * 1e3,
                                  "frac": t_roof / (comp_ms / 1e3)},
            "note": "decode: one launch per token over all layers (append + split-K attention), "
                    "L2 flushed before each; compression: each layer's call timed alone, its "
                    "inputs generated outside the timed interval"}


def e2e_measure(K, spec, dims, budgets, cache, prompt, qs, kns, vns, S, dev, steps=4,
                warmup=3):
    """Same metric through the C ABI with host buffers: every step copies the
    prompt (pinned host -> device) before compressing it, waits for the prefill,
    then copies each decode step's inputs in and its output back."""
    import torch
    L = spec.n_layers
    # the whole prompt (every layer's q_obs, k, v) as views of one pinned buffer:
    # measured ~6 % faster to copy in than the same bytes as separate pinned tensors
    names = ("q_obs", "k", "v")
    sizes = [[x[k].numel() * x[k].element_size() for k in names if k in x] for x in prompt]
    pool = torch.empty(sum(map(sum, sizes)), dtype=torch.uint8, pin_memory=True)
    hp, off = [], 0
    for x in prompt:
        d = {}
        for k in names:
            if k not in x:
                continue
            nb = x[k].numel() * x[k].element_size()
            d[k] = pool[off:off + nb].view(x[k].dtype).view(x[k].shape)
            d[k].copy_(x[k])
            off += nb
        hp.append(d)
    # each decode step's q, k_new and v_new side by side in one pinned row (one
    # host -> device copy per step), landing in one device buffer they are views of
    nq, nk, nv = qs[0].numel(), kns[0].numel(), vns[0].numel()
    assert qs[0].dtype == kns[0].dtype == vns[0].dtype
    hin = torch.empty(S, nq + nk + nv, dtype=qs[0].dtype, pin_memory=True)
    hin.copy_(torch.cat([torch.stack(x).reshape(S, -1) for x in (qs, kns, vns)], dim=1))
    hout = torch.empty(S, *qs[0].shape, dtype=torch.float32).pin_memory()
    dp = {k: torch.empty_like(v, device=dev) for k, v in hp[0].items()}
    din = torch.empty(nq + nk + nv, dtype=qs[0].dtype, device=dev)
    dq = din[:nq].view(qs[0].shape)
    dk = din[nq:nq + nk].view(kns[0].shape)
    dv = din[nq + nk:].view(vns[0].shape)
    dout = torch.empty(qs[0].shape, dtype=torch.float32, device=dev)
    h2d = sum(v.numel() * v.element_size() for x in hp for v in x.values()) + \
        hin.numel() * hin.element_size()
    d2h = hout.numel() * 4

    def step(parts=None):
        K.kvc_cache_reset(cache)
        ta = time.perf_counter()
        for l in range(L):
            for k in dp:
                dp[k].copy_(hp[l][k], non_blocking=True)
            K.kvc_prefill_compress(dims, budgets, l, dp.get("q_obs"), dp["k"], dp["v"],
                                   cache=cache)
        # the prefill is waited for before the first decode step, as a server does
        # before it emits its first token
        torch.cuda.synchronize()
        if parts is not None:
            parts["prompt_copy_and_compress_ms"] = (time.perf_counter() - ta) * 1e3
        tb = time.perf_counter()
        for t in range(S):
            din.copy_(hin[t], non_blocking=True)
            K.kvc_decode_step(cache, 0, L, dq, dk, dv, dout)
            hout[t].copy_(dout, non_blocking=True)
        torch.cuda.synchronize()
        if parts is not None:
            parts["decode_steps_ms"] = (time.perf_counter() - tb) * 1e3

    for _ in range(warmup):     # as before the device-timed steps; the first pass
        step()                  # over the pinned prompt is the slowest
    step_ms = []
    t0 = time.perf_counter()
    for _ in range(steps):
        ts = time.perf_counter()
        step()
        step_ms.append((time.perf_counter() - ts) * 1e3)
    dt = (time.perf_counter() - t0) / steps
    parts = {}
    step(parts)     # one more step, each phase's wall time recorded
    return {"value": spec.batch * S / dt, "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": dt * 1e3, "step_ms": step_ms,
            "parts": parts,
            "note": "includes the prompt's host->device copy and prefill compression (waited "
                    "for before decoding), one host->device copy of each decode step's "
                    "q|k_new|v_new and the device->host copy of its output"}


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
