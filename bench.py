#!/usr/bin/env python
"""Benchmark of the Higgs-Audio-style hot path on GB300.

One step = one pass of the whole path over one batch of synthetic input: batched BF16 prefill of
32 ragged prompts (lengths uniform in 16..256, seed 2) through the 36-layer full-width backbone
(hidden 2560, 32/8 heads, FFN 9728) into a 2048-slot cache, then one delayed-codebook frame (audio
head [8 x 1026, 2560], argmax + delay state, embedding sum) on the 32 last hiddens, then one
single-token decode pass of the 36 layers fed those embeddings.  `value` = prompt tokens per
second over the whole job; random-init weights and synthetic token ids.

Extra sections on the same line: single-layer prefill latency at P = 6 / 13, chained delayed-
codebook decode frames/s at batch 1 / 32 / 64 (L2-warm and HBM-cold), and the long-prompt
workload (8 prompts of 1024..2048 tokens, then 64 frames with a decode pass each).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
Multi-GPU (torchrun, one rank per GPU): every rank runs its own replica of the batch (weak
scaling, no data-path collective); rank 0 prints the line.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "prefill tokens/s + codebook-decode frames/s @1 GB300; % of TC/HBM roofline"
WORKLOAD = "36-layer full-width backbone, 32 ragged prompts U{16..256}, 2048-slot cache, + 1 codebook frame + 1 decode pass"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-extra", action="store_true", help="skip the secondary sections")
    ap.add_argument("--kernel-case", default=None, choices=["gate_up", "qkv", "down", "audio_head", "attention"],
                    help="run only a few launches of one kernel at a profiling size, then exit")
    ap.add_argument("--kernel-m", type=int, default=None, help="rows (tokens / batch) of the kernel case")
    ap.add_argument("--deadline", type=float, default=300.0,
                    help="seconds after start by which the JSON line is printed even if a secondary "
                         "section has not finished (it is then listed under extra.truncated)")
    return ap.parse_args()


def kernel_case(name, m=None):
    """A few launches of one kernel on inputs larger than L2 (for an ncu capture of that kernel)."""
    import torch

    import qwen3_prefill_delayed_gb300 as hra
    import workloads as W
    dev = torch.device("cuda", 0)
    g = torch.Generator(device=dev).manual_seed(7)
    d = W.full_dims(1)
    rnd = lambda *sh, std=1.0: (torch.randn(*sh, generator=g, device=dev) * std).to(torch.bfloat16)
    if name == "attention":
        # prefill of the 32 ragged prompts through 2 full-width layers: layer 0 runs the prefill
        # attention kernel over all rows (layer 1 takes the last-rows tail)
        wl = W.ragged_batch(dev, n_layers=2)
        d2, p = wl["dims"], wl["prompts"]
        bb = hra.Backbone(d2, wl["weights"])
        cache = hra.new_kv_cache(d2, 32, wl["n_slots"], dev)
        tok = p.tokens.to(dev)
        for _ in range(3):
            bb.prefill(tok, p.lengths, cache)
    elif name == "audio_head":
        wl = W.make_audio(d, g, dev)
        head = hra.AudioHead(d, wl["head_w"], wl["code_emb"])
        bsz = m or 64
        hid = rnd(bsz, d.hidden)
        state = torch.zeros(bsz, 4, dtype=torch.int32, device=dev)
        for _ in range(5):
            head.step(hid, state)
    else:
        M = m or 8192
        K, N, epi = {"gate_up": (d.hidden, d.ffn, hra.EPI_SWIGLU), "qkv": (d.hidden, d.qkv_rows, hra.EPI_STORE),
                     "down": (d.ffn, d.hidden, hra.EPI_RESIDUAL)}[name]
        a = rnd(M, K)
        w = rnd(2 * N if epi == hra.EPI_SWIGLU else N, K, std=0.02)
        out = torch.zeros(M, N, dtype=torch.bfloat16, device=dev)
        for _ in range(5):
            hra.hra_linear(a, w, epi, out=out)
    torch.cuda.synchronize()
    print(f"kernel case {name} done")


_T0 = time.perf_counter()
_EMIT = {"lock": None, "done": False}


def arm_deadline(line, extra, seconds):
    """Print `line` (with the secondary sections measured so far) and end the process if the main
    thread has not printed by `seconds` after start: a section stuck in a blocking call cannot
    keep the measured numbers from being reported."""
    import threading
    _EMIT["lock"] = threading.Lock()

    def watch():
        time.sleep(max(0.0, seconds - (time.perf_counter() - _T0)))
        with _EMIT["lock"]:
            if _EMIT["done"]:
                return
            _EMIT["done"] = True
            out = dict(line)
            out["extra"] = dict(extra)
            out["extra"]["truncated"] = f"secondary sections still running at {seconds:.0f} s were skipped"
            print(json.dumps(out), flush=True)
            log("deadline: line printed, exiting")
        os._exit(0)

    threading.Thread(target=watch, daemon=True).start()


def emit(line):
    lock = _EMIT["lock"]
    if lock is None:
        print(json.dumps(line), flush=True)
        return
    with lock:
        if _EMIT["done"]:
            return
        _EMIT["done"] = True
        print(json.dumps(line), flush=True)


def log(msg):
    """Progress on stderr (stdout carries only the JSON line)."""
    print(f"[bench {time.perf_counter() - _T0:7.1f} s] {msg}", file=sys.stderr, flush=True)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------ clocks during the timed region

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.out, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        power = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        busy = [s for s, p in zip(sm, power) if p > 200.0] or sm
        return {"sm_mhz": statistics.median(busy) if busy else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "power_w_max": max(power) if power else None}


# ------------------------------------------------------------------ helpers

def events_time(fn, n, torch):
    s = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for _ in range(n):
        fn()
    e1.record(s)
    e1.synchronize()
    return e0.elapsed_time(e1)


def max_over_ranks(x, world, device=None):
    """The largest value of `x` over all ranks (every rank gets it); `x` itself when world == 1.
    The whole-job time of a step is the slowest rank's."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world, units_per_rank, seconds_per_step):
    """Weak scaling: every rank processes `units_per_rank` per step, so the job's rate is
    world * units / (the slowest rank's time per step)."""
    return world * units_per_rank / seconds_per_step


def traffic_for(kernel, source_files):
    """DRAM bytes per launch recorded from an ncu capture, if the kernel source is unchanged."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f).get(kernel)
    if not d:
        return None
    h = hashlib.sha256()
    for sf in source_files:
        with open(os.path.join(ROOT, sf), "rb") as f:
            h.update(f.read())
    if d.get("source_sha256") != h.hexdigest():
        return None
    return d.get("bytes_per_launch")


def oracle_sample(d_full, weights_cpu_getter, prompts, n_layers_sample, seq_ids):
    """Time the CPU oracle on the first n layers for the chosen sequences; returns (s, tokens)."""
    import oracle
    import workloads as W
    d = W.Dims(**{**d_full.__dict__, "n_layers": n_layers_sample})
    w = weights_cpu_getter(n_layers_sample)
    hw = oracle.host_weights_from(d, w)
    lens = [prompts.lengths[b] for b in seq_ids]
    tok = prompts.tokens[seq_ids].numpy()
    t0 = time.perf_counter()
    oracle.prefill(d, hw, tok, lens, max(lens))
    return time.perf_counter() - t0, sum(lens)


# ------------------------------------------------------------------ reference arm: the CPU oracle

def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    import workloads as W
    oracle.build()
    d = W.full_dims(36)
    prompts = W.make_prompts(2, 32, 16, 256, d.vocab)
    g = W._gen(2, "cpu")
    one = W.make_backbone(W.Dims(**{**d.__dict__, "n_layers": 1}), 2, "cpu", gen=g)
    order = sorted(range(32), key=lambda b: prompts.lengths[b])
    seq = [order[len(order) // 2]]          # the median-length prompt
    getter = lambda n: one
    times, toks = [], 0
    for i in range(args.warmup + args.steps):
        t, toks = oracle_sample(d, getter, prompts, 1, seq)
        if i >= args.warmup:
            times.append(t)
    per_step = sum(times) / len(times)
    # one layer of one prompt; a full step is 36 layers of 32 prompts: scale to tokens/s of the model
    value = toks / (per_step * 36)
    cores = oracle.max_threads()
    sample = f"oracle prefill of 1 prompt ({toks} tokens) through 1 of 36 layers per step; tokens/s scaled by 1/36"
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": per_step * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": WORKLOAD, "global_batch": 32, "seq_len": "16..256", "parallelism": "replicas"},
            "impl": "reference",
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ our arm

def main():
    args = parse()
    if args.kernel_case:
        return kernel_case(args.kernel_case, args.kernel_m)
    if args.impl == "reference":
        return run_reference(args)
    import torch
    import torch.distributed as dist

    import qwen3_prefill_delayed_gb300 as hra
    import workloads as W

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    hra.lib()
    peaks, peaks_kind = load_peaks()

    # ---------------- main workload
    log("main workload")
    wl = W.ragged_batch(dev)
    d, p, w = wl["dims"], wl["prompts"], wl["weights"]
    B = len(p.lengths)
    tokens_per_step = p.total
    bb = hra.Backbone(d, w)
    head = hra.AudioHead(d, wl["audio"]["head_w"], wl["audio"]["code_emb"])
    cache = hra.new_kv_cache(d, B, wl["n_slots"], dev)
    tok_dev = p.tokens.to(dev)
    last = torch.empty(B, d.hidden, dtype=torch.bfloat16, device=dev)
    hid2 = torch.empty_like(last)
    state = torch.zeros(B, 4, dtype=torch.int32, device=dev)
    state[:, 1] = -1
    codes = torch.empty(B, d.n_codebooks, dtype=torch.int32, device=dev)
    nxt = torch.empty_like(last)
    done = torch.empty(B, dtype=torch.int32, device=dev)
    pos = list(p.lengths)
    ws = torch.empty(max(bb.prefill_workspace_size(B, p.total, p.max_len),
                         bb.decode_workspace_size(B, wl["n_slots"])), dtype=torch.uint8, device=dev)
    hws = torch.empty(head.workspace_size(B), dtype=torch.uint8, device=dev)

    def step():
        bb.prefill(tok_dev, p.lengths, cache, out=last, workspace=ws)
        head.step(last, state, codes=codes, next_emb=nxt, done=done, workspace=hws)
        bb.decode(nxt, pos, cache, out=hid2, workspace=ws)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert hra.hra_device_error(ws) == 0

    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    n0 = hra.hra_launch_counter()
    hra.hra_probe_select("gate_up")
    ms = events_time(step, args.steps, torch)
    hra.hra_probe_select("none")
    launches = hra.hra_launch_counter() - n0
    clk = clocks.stop()
    torch.cuda.synchronize()
    probe_ms, probe_n, probe_flops = hra.hra_probe_collect()
    ms = max_over_ranks(ms, world, dev)
    if world > 1:
        dist.barrier()
    ms_step = ms / args.steps
    value = whole_job_rate(world, tokens_per_step, ms_step / 1e3)

    # roofline of the dominant kernel: the gate/up + SwiGLU projection of the full prefill layers.
    # The timed region is sub-second and the box holds its full clock through it, so the peak is the
    # measured burst bf16 rate; the sustained-peak and clock-normalised fractions are given beside it.
    gu_ms = probe_ms / max(probe_n, 1)
    gu_flops = probe_flops / max(probe_n, 1)
    achieved = gu_flops / (gu_ms / 1e3) / 1e12
    peak = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    sustained = peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])
    sm_max = peaks.get("sm_max_mhz") or (clk or {}).get("sm_max_mhz")
    sm_run = (clk or {}).get("sm_mhz")
    roofline = {"bound": "tensor", "kernel": "gemm_bf16_tc_kernel<256,SwiGLU,bf16,pair> (gate/up on 2-CTA clusters, full layers)",
                "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                "peak_kind": f"{peaks_kind} bf16 burst",
                "frac_of_sustained": achieved / sustained,
                "frac_at_max_clock": (achieved * sm_max / sm_run / peak) if sm_max and sm_run else None,
                "traffic": traffic_for("gate_up", ["qwen3_prefill_delayed_gb300/csrc/gemm_tc.cu",
                                                      "qwen3_prefill_delayed_gb300/csrc/common.cuh"]),
                "launch_ms": gu_ms, "flops_per_launch": gu_flops, "launches_timed": probe_n}

    # ---------------- end to end through the public API with host buffers
    log("end to end")
    tok_host = p.tokens.clone().pin_memory()
    hid_host = torch.empty(B, d.hidden, dtype=torch.bfloat16).pin_memory()
    codes_host = torch.empty(B, d.n_codebooks, dtype=torch.int32).pin_memory()

    def e2e_step():
        tok_dev.copy_(tok_host, non_blocking=True)
        step()
        hid_host.copy_(hid2, non_blocking=True)
        codes_host.copy_(codes, non_blocking=True)
        torch.cuda.current_stream().synchronize()

    for _ in range(2):
        e2e_step()
    if world > 1:
        dist.barrier()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        e2e_step()
    e2e_s = max_over_ranks((time.perf_counter() - t0) / args.steps, world, dev)
    e2e = {"value": whole_job_rate(world, tokens_per_step, e2e_s), "unit": "tokens/s",
           "h2d_bytes_per_step": tok_host.numel() * 4,
           "d2h_bytes_per_step": hid_host.numel() * 2 + codes_host.numel() * 4}

    extra = {}
    cpu_baseline = None
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded random-init weights and token ids)",
            "config": {"workload": WORKLOAD, "global_batch": B * world, "seq_len": "16..256",
                       "tokens_per_step": tokens_per_step, "parallelism": f"replicas x{world}",
                       "l2": "inputs larger than L2 (8.05 GB of weights streamed per step)"},
            "roofline": roofline, "cpu_baseline": {"error": "not reached before the deadline"}, "e2e": e2e,
            "gpu_launches": int(launches), "clocks": clk, "extra": extra}
    if rank == 0:
        arm_deadline(line, extra, args.deadline)
    if rank == 0 and world == 1:
        try:
            import oracle
            oracle.build()
            order = sorted(range(B), key=lambda b: p.lengths[b])
            seq = [order[len(order) // 2]]

            def getter(n):
                return {"embed": w["embed"].cpu(), "final_norm": w["final_norm"].cpu(),
                        "layers": [{k: v.cpu() for k, v in w["layers"][i].items()} for i in range(n)]}
            oracle.set_threads(oracle.max_threads())
            log("cpu baseline")
            t_s, toks = oracle_sample(d, getter, p, d.n_layers, seq)
            cpu_baseline = {"value": toks / t_s, "unit": "tokens/s", "cores": oracle.max_threads(),
                            "kind": "oracle",
                            "sample": f"oracle prefill of the median prompt ({toks} tokens) through all "
                                      f"{d.n_layers} layers ({t_s:.1f} s), OpenMP over all host cores"}
        except Exception as ex:   # the baseline is reported, never required
            cpu_baseline = {"error": repr(ex)}
    line["cpu_baseline"] = cpu_baseline
    del cache
    torch.cuda.empty_cache()

    # the secondary sections (other configurations, the CPU oracle's timings) run at N = 1 only: the
    # multi-GPU lines report the replicated main workload, and N ranks would share the host's cores
    if not args.no_extra and world == 1:
        run_extra(hra, W, torch, dev, peaks, peaks_kind, w_backbone=w, out=extra)

    log("done")
    if rank == 0:
        emit(line)
    if world > 1:
        dist.destroy_process_group()


def run_extra(hra, W, torch, dev, peaks, peaks_kind, w_backbone, out):
    """Fill `out` section by section (a deadline print reports the sections done so far)."""
    hbm = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    # ---- single full-width layer, batch 1, P = 6 and 13 (HBM-bound: 201.85 MB of weights)
    log("single full-width layer")
    try:
        wl = W.single_layer(13, dev)
        d = wl["dims"]
        bb = hra.Backbone(d, wl["weights"])
        wbytes = sum(t.numel() * 2 for k, t in wl["weights"]["layers"][0].items())
        res = {}
        for P in (6, 13):
            pr = W.make_prompts(1, 1, P, P, d.vocab, fixed_len=P)
            tok = pr.tokens.to(dev)
            cache = hra.new_kv_cache(d, 1, 2048, dev)
            f = lambda: bb.prefill(tok, pr.lengths, cache, full_last_layer=True)
            for _ in range(5):
                f()
            ms = events_time(f, 50, torch) / 50
            res[f"P{P}"] = {"ms_per_layer": ms, "x36_projection_ms": ms * 36,
                            "hbm_gbs": wbytes / (ms / 1e3) / 1e9,
                            "hbm_frac": wbytes / (ms / 1e3) / 1e9 / hbm}
        out["single_layer_prefill"] = res
        del bb, wl
    except Exception as ex:
        out["single_layer_prefill"] = {"error": repr(ex)}
    # ---- chained codebook decode, 200 steps in one CUDA graph
    log("codebook decode")
    try:
        out["codebook_decode"] = bench_codebook(hra, W, torch, dev, hbm, peaks_kind)
    except Exception as ex:
        out["codebook_decode"] = {"error": repr(ex)}
    # ---- the ragged batch prefilled in two chunks (the second reads the first from the cache)
    log("chunked prefill")
    try:
        out["chunked_prefill"] = bench_chunked(hra, W, torch, dev, w_backbone)
    except Exception as ex:
        out["chunked_prefill"] = {"error": repr(ex)}
    torch.cuda.empty_cache()
    # ---- the static-FP8 variant of the prefill projections on the same ragged batch
    log("fp8 prefill")
    try:
        out["fp8_prefill"] = bench_fp8(hra, W, torch, dev, w_backbone, peaks)
    except Exception as ex:
        out["fp8_prefill"] = {"error": repr(ex)}
    torch.cuda.empty_cache()
    # ---- the NVFP4 band of the prefill projections on the same ragged batch
    log("nvfp4 prefill")
    try:
        out["nvfp4_prefill"] = bench_nvfp4(hra, W, torch, dev, w_backbone, peaks)
    except Exception as ex:
        out["nvfp4_prefill"] = {"error": repr(ex)}
    torch.cuda.empty_cache()
    # ---- long prompts + 64 AR frames
    log("long prompts")
    try:
        out["long_prompts"] = bench_long(hra, W, torch, dev, w_backbone)
    except Exception as ex:
        out["long_prompts"] = {"error": repr(ex)}
    torch.cuda.empty_cache()
    # ---- the CPU oracle on each configuration's workload (single thread and all host cores)
    log("oracle timing")
    try:
        out["oracle_timing"] = bench_oracle_configs(W)
    except Exception as ex:
        out["oracle_timing"] = {"error": repr(ex)}
    return out


def bench_oracle_configs(W):
    """The oracle as it stands, timed on the host cores for each configuration's workload: the tiny
    model's whole run and one full-width layer at P = 6 / 13 single-threaded; the codebook step at
    batch 1 single-threaded and at 1 / 32 / 64 on all cores; the long-prompt workload as one prompt
    of 1024 tokens through one layer on all cores (a stated subset, scaled per layer)."""
    import numpy as np

    import oracle
    oracle.build()
    ncore = oracle.max_threads()
    res = {"cores_all": ncore}

    def timed(fn, threads):
        oracle.set_threads(threads)
        t0 = time.perf_counter()
        r = fn()
        return time.perf_counter() - t0, r

    # tiny model: P = 13 prefill, then 6 frames of codebook step + decode pass (2 layers, K = 4)
    wl = W.tiny_reference("cpu")
    d, pr = wl["dims"], wl["prompts"]
    hw = oracle.host_weights_from(d, wl["weights"])
    head_u, tab_u = W.to_u16(wl["audio"]["head_w"]), W.to_u16(wl["audio"]["code_emb"])

    def tiny_run():
        kv, h = oracle.prefill(d, hw, pr.tokens.numpy(), pr.lengths, wl["n_slots"])
        st = np.array([[0, -1, 0, 0]], np.int32)
        for t in range(wl["frames"]):
            _, nxt, _, _ = oracle.codebook_step(d, h, head_u, tab_u, st, wl["eoc_bias"][t].numpy())
            h = oracle.decode(d, hw, nxt, [pr.lengths[0] + t], kv, wl["n_slots"])
    t1, _ = timed(tiny_run, 1)
    res["tiny_prefill13_plus_6_frames"] = {"threads": 1, "seconds": t1}
    # one full-width layer, batch 1, P = 6 and 13
    sl = W.single_layer(13, "cpu")
    ds = sl["dims"]
    hws = oracle.host_weights_from(ds, sl["weights"])
    for P in (6, 13):
        pp = W.make_prompts(1, 1, P, P, ds.vocab, fixed_len=P)
        for thr in (1, ncore):
            t, _ = timed(lambda: oracle.prefill(ds, hws, pp.tokens.numpy(), pp.lengths, 2048), thr)
            res[f"single_layer_P{P}_threads{thr}"] = {"ms_per_layer": t * 1e3}
    del hws, sl
    # codebook step: head [8 x 1026, 2560], 8 tables
    dc = W.full_dims(0)
    au = W.make_audio(dc, W._gen(3, "cpu"), "cpu")
    hu, tu = W.to_u16(au["head_w"]), W.to_u16(au["code_emb"])
    for B, thr in ((1, 1), (1, ncore), (32, ncore), (64, ncore)):
        ch = W.make_decode_chain(dc, 3, B, 1)
        st = ch.state0.numpy().copy()
        t, _ = timed(lambda: oracle.codebook_step(dc, W.to_u16(ch.hidden[0]), hu, tu, st, ch.eoc_bias[0].numpy()), thr)
        res[f"codebook_B{B}_threads{thr}"] = {"seconds_per_step": t, "frames_per_s": B / t}
    # long prompts: one 1024-token prompt through one full-width layer, all cores
    dl = W.full_dims(1)
    wlay = W.make_backbone(dl, 4, "cpu")
    hwl = oracle.host_weights_from(dl, wlay)
    pl = W.make_prompts(4, 1, 1024, 1024, dl.vocab, fixed_len=1024)
    t, _ = timed(lambda: oracle.prefill(dl, hwl, pl.tokens.numpy(), pl.lengths, 1024), ncore)
    res["long_prompt_1024_one_layer_threads_all"] = {"seconds": t, "tokens_per_s_36_layers": 1024 / (t * 36)}
    oracle.set_threads(ncore)
    return res


def bench_codebook(hra, W, torch, dev, hbm, peaks_kind):
    res = {}
    d = W.full_dims(0)
    g = W._gen(3, dev)
    copies = [W.make_audio(d, g, dev) for _ in range(4)]     # 4 x 84 MB > L2 for the cold figure
    K, Vc, H = d.n_codebooks, d.codebook_size, d.hidden
    head_bytes = K * Vc * H * 2
    steps = 200
    for B in (1, 32, 64):
        chain = W.make_decode_chain(d, 3, B, steps, device=dev)
        state = chain.state0.clone()
        codes = torch.empty(steps, B, K, dtype=torch.int32, device=dev)
        nxt = torch.empty(steps, B, H, dtype=torch.bfloat16, device=dev)
        done = torch.empty(steps, B, dtype=torch.int32, device=dev)
        heads = [hra.AudioHead(d, c["head_w"], c["code_emb"]) for c in copies]
        ws = torch.empty(heads[0].workspace_size(B), dtype=torch.uint8, device=dev)
        stream = torch.cuda.Stream()
        result = {}
        seeds = torch.arange(1, B + 1, dtype=torch.int64, device=dev) * 0x9E3779B97F4A7C1
        # greedy with the head warm in L2 and cold (4 copies), then sampled (temperature 1, top-k 50,
        # top-p 0.95: the pages' serving setting) cold
        for mode, rot, sampling in (("l2_warm", 1, None), ("hbm_cold", 4, None),
                                    ("sampled_hbm_cold", 4, (1.0, 50, 0.95))):
            sk = {} if sampling is None else {"sampling": sampling, "seeds": seeds}
            with torch.cuda.stream(stream):
                heads[0].step(chain.hidden[0], state.clone(), eoc_bias=chain.eoc_bias[0], workspace=ws, **sk)
            torch.cuda.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=stream):
                for s in range(steps):
                    heads[s % rot].step(chain.hidden[s], state, eoc_bias=chain.eoc_bias[s], codes=codes[s],
                                        next_emb=nxt[s], done=done[s], workspace=ws, **sk)
            for _ in range(3):
                state.copy_(chain.state0)
                graph.replay()
            torch.cuda.synchronize()
            reps = 10
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            tot = 0.0
            for _ in range(reps):
                state.copy_(chain.state0)
                e0.record()
                graph.replay()
                e1.record()
                e1.synchronize()
                tot += e0.elapsed_time(e1)
            ms_step = tot / reps / steps
            # algorithmic bytes per step: head weights + per row (hidden, K gathered rows, next, codes/state)
            bytes_step = head_bytes + B * (H * 2 + K * H * 2 + H * 2 + K * 4 + 16 + 4)
            result[mode] = {"frames_per_s": B / (ms_step / 1e3), "us_per_step": ms_step * 1e3,
                            "gbs": bytes_step / (ms_step / 1e3) / 1e9,
                            "hbm_frac": bytes_step / (ms_step / 1e3) / 1e9 / hbm}
            del graph
        res[f"B{B}"] = result
    res["note"] = (f"200 chained steps in one CUDA graph; hbm_cold rotates 4 weight copies (336 MB > L2); "
                   f"sampled: temperature 1, top-k 50, top-p 0.95, per-row seeds; "
                   f"hbm_frac is of the {peaks_kind} copy bandwidth")
    return res


def bench_chunked(hra, W, torch, dev, w_backbone):
    """The 32 ragged prompts as two chunks per sequence: the first ceil(len/2) tokens from position
    0, then the rest after them (hra_prefill_chunk), against the whole prompts in one call."""
    d = W.full_dims(36)
    p = W.make_prompts(2, 32, 16, 256, d.vocab)       # the ragged batch's prompts
    bb = hra.Backbone(d, w_backbone)
    B = len(p.lengths)
    lens = list(p.lengths)
    first = [(n + 1) // 2 for n in lens]
    rest = [n - f for n, f in zip(lens, first)]
    tok = p.tokens.to(dev)
    tok1 = p.tokens[:, :max(first)].contiguous().to(dev)
    tok2 = torch.zeros(B, max(rest), dtype=torch.int32)
    for b in range(B):
        tok2[b, :rest[b]] = p.tokens[b, first[b]:lens[b]]
    tok2 = tok2.to(dev)
    cache = hra.new_kv_cache(d, B, 2048, dev)
    out = torch.empty(B, d.hidden, dtype=torch.bfloat16, device=dev)
    ws = torch.empty(max(bb.prefill_workspace_size(B, sum(lens), max(lens)),
                         bb.prefill_chunk_workspace_size(B, sum(rest), max(rest), max(lens))),
                     dtype=torch.uint8, device=dev)
    whole = lambda: bb.prefill(tok, lens, cache, out=out, workspace=ws)
    c1 = lambda: bb.prefill(tok1, first, cache, out=out, workspace=ws)
    c2 = lambda: bb.prefill(tok2, rest, cache, out=out, workspace=ws, start_pos=first)
    for f in (whole, c1, c2):
        for _ in range(2):
            f()
    torch.cuda.synchronize()
    ms_whole = events_time(whole, 5, torch) / 5
    ms_c1 = events_time(c1, 5, torch) / 5
    c1()
    ms_c2 = events_time(c2, 5, torch) / 5
    del cache
    return {"whole_tokens_per_s": sum(lens) / (ms_whole / 1e3), "whole_ms": ms_whole,
            "chunk1_ms": ms_c1, "chunk2_ms": ms_c2, "chunk2_tokens": sum(rest),
            "chunk2_tokens_per_s": sum(rest) / (ms_c2 / 1e3),
            "two_chunks_tokens_per_s": sum(lens) / ((ms_c1 + ms_c2) / 1e3)}


def bench_fp8(hra, W, torch, dev, w_backbone, peaks):
    """FP8 (E4M3) projections with static activation scales calibrated on a fixed calibration batch
    (4 prompts of 64 tokens, their own seed), then the ragged batch's prefill; the gate/up GEMM is
    reported against the FP8 peak = the measured bf16 burst peak x 2 (the nominal dense FP8 / BF16
    tensor-rate ratio of the part)."""
    d = W.full_dims(36)
    p = W.make_prompts(2, 32, 16, 256, d.vocab)
    bb = hra.Backbone(d, w_backbone)
    f8 = hra.Fp8Backbone(bb)
    cal = W.make_prompts(99, 4, 64, 64, d.vocab, fixed_len=64)
    cache = hra.new_kv_cache(d, 32, 2048, dev)
    f8.calibrate(cal.tokens.to(dev), cal.lengths, cache)
    tok = p.tokens.to(dev)
    out = torch.empty(32, d.hidden, dtype=torch.bfloat16, device=dev)
    ws = torch.empty(f8.prefill_workspace_size(32, p.total, p.max_len), dtype=torch.uint8, device=dev)
    run = lambda: f8.prefill(tok, p.lengths, cache, out=out, workspace=ws)
    run16 = lambda: bb.prefill(tok, p.lengths, cache, out=out)
    for f in (run, run16):
        for _ in range(2):
            f()
    torch.cuda.synchronize()
    ms = events_time(run, 5, torch) / 5
    ms16 = events_time(run16, 5, torch) / 5
    hra.hra_probe_select("gate_up")
    run()
    hra.hra_probe_select("none")
    gu_ms, gu_n, gu_flops = hra.hra_probe_collect()
    peak8 = 2.0 * peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    tf = gu_flops / (gu_ms / 1e3) / 1e12 if gu_ms > 0 else None
    del cache, f8
    return {"prefill_tokens_per_s": p.total / (ms / 1e3), "prefill_ms": ms, "bf16_prefill_ms": ms16,
            "gate_up_tflops": tf, "gate_up_frac_of_fp8_peak": tf / peak8 if tf else None,
            "fp8_peak_tflops": peak8, "calibration": "4 prompts x 64 tokens, seed 99"}


def bench_nvfp4(hra, W, torch, dev, w_backbone, peaks):
    """The NVFP4 band (QKV in static FP8; output, gate/up and down in NVFP4 with per-call block
    scales), calibrated on the FP8 variant's calibration batch, then the ragged batch's prefill.
    The gate/up NVFP4 GEMM runs its MMAs on the exact f16 expansion of the NVFP4 values, so it is
    reported against the measured bf16 burst peak (the rate of those MMAs) and against the nominal
    dense FP4 rate (6 x that peak, the part's FP4 / BF16 ratio)."""
    d = W.full_dims(36)
    p = W.make_prompts(2, 32, 16, 256, d.vocab)
    bb = hra.Backbone(d, w_backbone)
    nv = hra.Nvfp4Backbone(bb)
    cal = W.make_prompts(99, 4, 64, 64, d.vocab, fixed_len=64)
    cache = hra.new_kv_cache(d, 32, 2048, dev)
    nv.calibrate(cal.tokens.to(dev), cal.lengths, cache)
    tok = p.tokens.to(dev)
    out = torch.empty(32, d.hidden, dtype=torch.bfloat16, device=dev)
    ws = torch.empty(nv.prefill_workspace_size(32, p.total, p.max_len), dtype=torch.uint8, device=dev)
    run = lambda: nv.prefill(tok, p.lengths, cache, out=out, workspace=ws)
    for _ in range(2):
        run()
    torch.cuda.synchronize()
    ms = events_time(run, 5, torch) / 5
    hra.hra_probe_select("gate_up")
    run()
    hra.hra_probe_select("none")
    gu_ms, gu_n, gu_flops = hra.hra_probe_collect()
    bf = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    tf = gu_flops / (gu_ms / 1e3) / 1e12 if gu_ms > 0 else None
    wbytes = sum(nv.keep[l]["codes"][q].numel() + nv.keep[l]["scales"][q].numel()
                 for l in range(d.n_layers) for q in (1, 2, 3))
    del cache, nv
    return {"prefill_tokens_per_s": p.total / (ms / 1e3), "prefill_ms": ms, "gate_up_tflops": tf,
            "gate_up_frac_of_bf16_burst": tf / bf if tf else None,
            "gate_up_frac_of_fp4_nominal": tf / (6.0 * bf) if tf else None,
            "nvfp4_weight_bytes": wbytes, "calibration": "4 prompts x 64 tokens, seed 99"}


def bench_long(hra, W, torch, dev, w_backbone):
    wl = W.long_prompts(dev)
    d, p = wl["dims"], wl["prompts"]
    bb = hra.Backbone(d, wl["weights"])
    head = hra.AudioHead(d, wl["audio"]["head_w"], wl["audio"]["code_emb"])
    B = len(p.lengths)
    cache = hra.new_kv_cache(d, B, wl["n_slots"], dev)
    tok = p.tokens.to(dev)
    last = torch.empty(B, d.hidden, dtype=torch.bfloat16, device=dev)
    state = torch.zeros(B, 4, dtype=torch.int32, device=dev)
    frames = wl["frames"]

    def prefill():
        bb.prefill(tok, p.lengths, cache, out=last)

    def ar():
        state.zero_()
        state[:, 1] = -1
        hid = last
        for f in range(frames):
            _, nxt, _ = head.step(hid, state)
            hid = bb.decode(nxt, [n + f for n in p.lengths], cache)

    prefill()
    ar()
    torch.cuda.synchronize()
    hra.hra_probe_select("attention")
    ms_pf = events_time(prefill, 3, torch) / 3
    hra.hra_probe_select("none")
    att_ms, att_n, att_flops = hra.hra_probe_collect()
    ms_ar = events_time(ar, 2, torch) / 2
    # the same loop on device-resident state: all 64 frames captured once in a CUDA graph
    prefill()
    loop = hra.ARLoop(bb, head, cache, last.clone(), p.lengths, max(p.lengths) + frames)
    hid0 = loop.hidden.clone()
    loop.capture(frames)

    def ar_graph():
        loop.state.zero_()
        loop.state[:, 1] = -1
        loop.pos.copy_(torch.tensor(p.lengths, dtype=torch.int32))
        loop.hidden.copy_(hid0)
        loop.replay()

    ar_graph()
    torch.cuda.synchronize()
    ms_graph = events_time(ar_graph, 3, torch) / 3
    return {"prefill_tokens_per_s": p.total / (ms_pf / 1e3), "prefill_ms": ms_pf, "tokens": p.total,
            "ar_ms_per_frame": ms_ar / frames, "ar_graph_ms_per_frame": ms_graph / frames, "frames": frames,
            "attention_tflops": att_flops / (att_ms / 1e3) / 1e12 if att_ms > 0 else None,
            "attention_ms_per_step": att_ms / 3}


if __name__ == "__main__":
    main()
