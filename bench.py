"""Benchmark: batch-1 greedy decode tok/s on one GB300 and the fraction of the
HBM roofline it reaches.

Workload (default): the Llama-3.2-1B-shaped decoder (16 layers, hidden 2048,
32/8 heads, head_dim 64, FFN 8192, vocab 128256, tied embeddings, llama3 RoPE)
with seed-generated BF16 weights N(0, 0.02), a KV cache pre-filled with 1,023
positions of N(0, 1), one seeded input token, 64 greedy tokens. One "step" is
one decode call of those 64 tokens (one cooperative launch of the persistent
kernel); each call rewrites positions 1023..1086, so repeats are identical and
are checked bit for bit.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME]
                  [--scheduler counters|waves|flags|all] [--impl ours|reference] [--tokens T]
                  [--weights bf16|int8] [--kv bf16|int8]
                  [--mode decode|prefill|verify] [--prompt N] [--k K]

--weights int8: weight-only INT8 GEMVs; --kv int8: the INT8 KV cache with
smoothed keys (built from the BF16 prefill outside the timed region); each
changes the algorithmic bytes the roofline fraction is taken on. --mode
prefill / verify time the multi-token pass (tensor roofline on the weight
FLOPs) and the greedy verify step.

With N > 1 (launched by torchrun) every rank runs an independent replica: a
batch-1 decode has no exchange step to shard (replicas only). `--impl
reference` times the CPU oracle on the host cores on a bounded sample of the
same workload. Prints one JSON line on stdout.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "batch-1 decode tok/s on 1 GB300; % of HBM roofline (weight+KV bytes/token)"
UNIT = "tok/s"
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "megakernel_traffic.json")


SCHEDULERS = {"counters": 1, "waves": 0, "flags": 2}   # tiles_plan_opts.scheduler values


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(values, device="cpu"):
    """Element-wise maximum of a list of timings over all ranks (the list
    unchanged when no process group is up). Every rank gets the same list."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def whole_job_rate(units_per_rank, seconds, device="cpu"):
    """(units all ranks processed / the slowest rank's seconds, that time):
    the replicas' aggregate throughput over the wall time of the whole job."""
    import torch.distributed as dist
    ws = dist.get_world_size() if dist.is_available() and dist.is_initialized() else 1
    (slowest,) = max_over_ranks([seconds], device)
    return units_per_rank * ws / slowest, slowest


def workload_config(cfg, int8=False, kv8=False):
    return {"workload": f"{cfg.name}: {cfg.n_layers} layers, hidden {cfg.hidden}, "
                        f"{cfg.n_q_heads}/{cfg.n_kv_heads} heads x {cfg.head_dim}, ffn {cfg.ffn}, "
                        f"vocab {cfg.vocab}, {cfg.start_pos} cached positions, "
                        f"{cfg.n_new} greedy tokens per step",
            "weights": WEIGHT_DESC[int8], "kv_cache": KV_DESC[kv8],
            "tokens_per_step": cfg.n_new, "cached_positions": cfg.start_pos,
            "bytes_per_token": int(round(cfg.algorithmic_bytes_per_token(int8, kv8))),
            "l2": "inputs larger than L2 (every token streams all weights, >0.5 GB)"}


WEIGHT_DESC = {False: "bf16",
               True: "int8 codes with one fp32 scale per output row (GEMV matrices and LM head)"}
DTYPE = {False: "bf16", True: "int8 weights x bf16 activations, fp32 accumulate"}
KV_DESC = {False: "bf16",
           True: "int8 codes with one fp32 scale per cached row, keys minus a per-channel mean"}


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except (OSError, ValueError):
        return None


# sources the decode kernel's launch depends on (the multi-token pass in
# forward.cu is a separate set of kernels and does not change its traffic)
DECODE_SOURCES = ("kernels_bf16.cu", "kernels_bf16_mma.cu", "kernels_int8.cu", "kernels_int8_mma.cu",
                  "kernels_bf16_kv8.cu", "kernels_int8_kv8.cu", "megakernel.cu", "megakernel.cuh",
                  "planner.cpp", "runtime.cu", "tiles_internal.h")


def kernel_source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "tile_scheduled_persistent_gb300", "csrc")
    for name in DECODE_SOURCES:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(config_name, n_tokens):
    """DRAM bytes per launch of `n_tokens` tokens, from the per-token figure of a
    committed ncu capture (dram__bytes_read.sum + dram__bytes_write.sum of one
    launch over its token count), if it was taken on the current kernel
    source; else None."""
    try:
        with open(TRAFFIC_FILE) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    e = d.get(config_name)
    if not e or e.get("source_hash") != kernel_source_hash():
        return None
    per_token = e.get("dram_bytes_per_token")
    return None if per_token is None else per_token * n_tokens


class ClockSampler:
    """nvidia-smi samples (every 200 ms) while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
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
        return False

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------- CPU oracle arm
def oracle_sample(cfg, w, k, v, prompt, n_tokens, qweights=None, n_threads=0, kv_int8=False):
    """Time the oracle on n_tokens decode steps of the workload (all host cores,
    or n_threads); with qweights, its weight-only INT8 form; with kv_int8, its
    INT8 KV cache (built from the prefill inside the call)."""
    import oracle
    kk, vv = k.copy(), v.copy()
    t0 = time.perf_counter()
    oracle.decode(cfg, w, kk, vv, prompt, cfg.start_pos, n_tokens, want_logits=False,
                  qweights=qweights, n_threads=n_threads, kv_int8=kv_int8)
    return time.perf_counter() - t0


def oracle_qweights(w, int8):
    """The oracle's INT8 weights (quantized once, outside any timed region), or None."""
    if not int8:
        return None
    import oracle
    return oracle.quantize_model(w)


def run_reference(args):
    import synthetic as S
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    cfg = S.CONFIGS[args.config]
    log(f"[reference] generating {cfg.name} inputs ...")
    w = S.model_weights(cfg)
    k, v = S.kv_prefill(cfg)
    prompt = S.prompt(cfg)
    int8 = args.weights == "int8"
    kv8 = args.kv == "int8"
    qw = oracle_qweights(w, int8)
    n_tok = args.ref_tokens
    for _ in range(args.warmup):
        oracle_sample(cfg, w, k, v, prompt, n_tok, qw, kv_int8=kv8)
    times = [oracle_sample(cfg, w, k, v, prompt, n_tok, qw, kv_int8=kv8) for _ in range(args.steps)]
    tot = sum(times)
    value = n_tok * args.steps / tot
    cores = os.cpu_count()
    sample = (f"{n_tok} decode tokens of the workload from position {cfg.start_pos} per step "
              f"(of {cfg.n_new}), OpenMP over output rows and heads")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * tot / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": DTYPE[int8],
            "data": "synthetic", "config": workload_config(cfg, int8, kv8),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------- GPU arm
def run_ours(args):
    import numpy as np
    import torch

    import synthetic as S
    import tile_scheduled_persistent_gb300 as tsp

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    dev = torch.cuda.current_device()
    tsp.build()
    cfg = S.CONFIGS[args.config]
    if args.tokens:
        from dataclasses import replace
        cfg = replace(cfg, n_new=args.tokens)
    log(f"[rank {rank}] generating {cfg.name} inputs ...")
    t0 = time.time()
    w = S.model_weights(cfg)
    k_np, v_np = S.kv_prefill(cfg)
    prompt_np = S.prompt(cfg)
    log(f"[rank {rank}] generated in {time.time() - t0:.1f}s; uploading")
    dw = tsp.upload_weights(w)
    kc = tsp.to_device_bf16(k_np)
    vc = tsp.to_device_bf16(v_np)
    dprompt = torch.from_numpy(prompt_np).cuda()
    stream = torch.cuda.current_stream()

    # HBM copy peak measured in this run (read + write bytes, best of 10)
    n_copy = 1 << 30
    a = torch.empty(n_copy, dtype=torch.int16, device="cuda")
    b = torch.empty_like(a)
    a.fill_(1)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    best = 1e30
    for _ in range(12):
        e0.record()
        tsp.copy_bw(b, a)
        e1.record()
        e1.synchronize()
        best = min(best, e0.elapsed_time(e1) / 1e3)
    copy_gbs = 2 * a.numel() * 2 / best / 1e9
    del a, b
    torch.cuda.empty_cache()
    try:
        barrier_ns = tsp.barrier_cost(0, 2000)
    except tsp.TilesError:
        barrier_ns = None

    int8 = args.weights == "int8"
    kv8 = args.kv == "int8"
    bytes_per_token = cfg.algorithmic_bytes_per_token(int8, kv8)
    if kv8:
        # the INT8 cache of the prefill (outside the timed region); decode steps
        # overwrite positions from start_pos on, like the BF16 cache's
        cache8 = tsp.KV8Cache(tsp.ModelDesc.from_config(cfg)).from_bf16(kc, vc, cfg.start_pos)
        kc, vc = cache8.k, cache8.v
    results = {}
    scheds = list(SCHEDULERS) if args.scheduler == "all" else [args.scheduler]
    for sname in scheds:
        plan = tsp.Plan(tsp.ModelDesc.from_config(cfg), dw,
                        tsp.make_opts(scheduler=SCHEDULERS[sname],
                                      weight_format=tsp.WEIGHTS_INT8 if int8 else tsp.WEIGHTS_BF16,
                                      kv_format=tsp.KV_INT8 if kv8 else tsp.KV_BF16))
        info = plan.info()
        toks = torch.zeros(cfg.n_new, dtype=torch.int32, device="cuda")
        ref_toks = None
        for _ in range(args.warmup):
            plan.decode(kc, vc, dprompt, cfg.start_pos, cfg.n_new, toks)
        plan.check()
        ref_toks = toks.clone()
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        all_toks = torch.zeros((args.steps, cfg.n_new), dtype=torch.int32, device="cuda")
        if ws > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        with ClockSampler(dev) as clk:
            g0 = torch.cuda.Event(enable_timing=True)
            g1 = torch.cuda.Event(enable_timing=True)
            g0.record(stream)
            for i in range(args.steps):
                starts[i].record(stream)
                plan.decode(kc, vc, dprompt, cfg.start_pos, cfg.n_new, all_toks[i])
                ends[i].record(stream)
            g1.record(stream)
            torch.cuda.synchronize()
        if ws > 1:
            torch.distributed.barrier()
        plan.check()
        total_s = g0.elapsed_time(g1) / 1e3
        per_launch = [s.elapsed_time(e) / 1e3 for s, e in zip(starts, ends)]
        bitwise = bool((all_toks == ref_toks[None, :]).all().item())
        results[sname] = dict(total_s=total_s, per_launch=per_launch, clocks=clk.summary(),
                              bitwise=bitwise, info=info, plan=plan,
                              tokens=ref_toks.cpu().numpy())
        log(f"[rank {rank}] {sname}: {args.steps * cfg.n_new / total_s:.1f} tok/s, "
            f"launch {statistics.mean(per_launch) * 1e6:.0f} us, bitwise {bitwise}")
    # keep the faster scheduler on evidence: its slowest rank decides
    names = list(results)
    slowest = dict(zip(names, max_over_ranks([results[s]["total_s"] for s in names], "cuda")))
    chosen = min(names, key=lambda s: slowest[s])
    r = results[chosen]
    value, total_s = whole_job_rate(args.steps * cfg.n_new, r["total_s"], "cuda")
    launch_s = statistics.mean(r["per_launch"])
    achieved_gbs = bytes_per_token * cfg.n_new / launch_s / 1e9
    peaks = measured_peaks()
    if peaks and peaks.get("hbm_gbs"):
        peak, peak_src = float(peaks["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs)"
    else:
        peak, peak_src = 6800.0, "fallback 6.8 TB/s"
    traffic = recorded_traffic(cfg.name + ("_int8" if int8 else "") + ("_kv8" if kv8 else ""), cfg.n_new)

    # end to end through the host-buffer entry point (copies inside the timed region)
    plan = r["plan"]
    pin_prompt = torch.from_numpy(prompt_np.copy()).pin_memory().numpy()
    host_toks = torch.zeros(cfg.n_new, dtype=torch.int32).pin_memory().numpy()
    plan.decode_host(kc, vc, pin_prompt, cfg.start_pos, cfg.n_new, host_toks)
    if ws > 1:
        torch.distributed.barrier()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        plan.decode_host(kc, vc, pin_prompt, cfg.start_pos, cfg.n_new, host_toks)
    e2e_value, _ = whole_job_rate(args.steps * cfg.n_new, time.perf_counter() - t0, "cuda")
    e2e_same = bool(np.array_equal(host_toks, r["tokens"]))

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        n_tok = args.ref_tokens
        qw = oracle_qweights(w, int8)
        secs = oracle_sample(cfg, w, k_np, v_np, prompt_np, n_tok, qw, kv_int8=kv8)
        cpu = {"value": n_tok / secs, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
               "sample": f"first {n_tok} of the {cfg.n_new} decode tokens from position "
                         f"{cfg.start_pos}, OpenMP over output rows and heads on all host cores"
                         + (", the oracle's weight-only INT8 path" if int8 else "")
                         + (", the oracle's INT8 KV cache (built from the prefill inside the timed call)"
                            if kv8 else "")}
        try:  # the same oracle on one thread, one token (information only)
            secs1 = oracle_sample(cfg, w, k_np, v_np, prompt_np, 1, qw, n_threads=1, kv_int8=kv8)
            cpu["single_thread"] = {"value": 1 / secs1, "unit": UNIT, "cores": 1,
                                    "sample": f"first decode token from position {cfg.start_pos}"}
        except Exception as e:  # never let the information line cost the measurement
            cpu["single_thread"] = {"error": str(e)[:200]}

    if rank == 0:
        conf = workload_config(cfg, int8, kv8)
        conf.update({"scheduler": chosen, "ctas": r["info"]["n_ctas"],
                     "ring": f"{r['info']['ring_slots']} x {r['info']['slot_bytes']} B",
                     "kv_splits": r["info"]["kv_splits"], "parallelism": f"replicas x{ws}"})
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
                "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": 1000 * total_s / args.steps, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": DTYPE[int8], "data": "synthetic",
                "config": conf,
                "roofline": {"bound": "hbm", "achieved": achieved_gbs, "peak": peak,
                             "unit": "GB/s", "frac": achieved_gbs / peak,
                             "traffic": traffic, "peak_source": peak_src,
                             "kernel": "tiles_megakernel",
                             "copy_kernel_gbs_this_run": copy_gbs,
                             "frac_of_copy_this_run": achieved_gbs / copy_gbs},
                "cpu_baseline": cpu,
                "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": 4 * prompt_np.size,
                        "d2h_bytes_per_step": 4 * cfg.n_new, "same_tokens": e2e_same},
                "gpu_launches": args.steps,
                "clocks": r["clocks"],
                "bitwise_repeat": r["bitwise"],
                "us_per_token": 1e6 * launch_s / cfg.n_new,
                "launch_us": {"mean": 1e6 * launch_s,
                              "median": 1e6 * statistics.median(r["per_launch"]),
                              "min": 1e6 * min(r["per_launch"])},
                "grid_barrier_ns": barrier_ns,
                "schedulers": {s: {"tok_s": args.steps * cfg.n_new * ws / slowest[s],
                                   "bitwise_repeat": results[s]["bitwise"]} for s in results}}
        print(json.dumps(line), flush=True)
    for s in results:
        results[s]["plan"].close()
    if ws > 1:
        torch.distributed.destroy_process_group()
    return 0


# ---------------------------------------------------------------------- multi-token arms
def run_multi(args):
    """--mode prefill: a prompt of --prompt seeded tokens from an empty cache
    through tiles_forward (passes of up to 256 tokens); tok/s and the tensor
    throughput of the weight FLOPs (2 x parameters x tokens) against the
    measured BF16 peak. --mode verify: one tiles_verify step of --k drafts at
    the workload's cached positions, the drafts being the decode kernel's own
    greedy tokens; emitted tokens per second (accepted drafts + 1 per step)."""
    import numpy as np
    import torch

    import synthetic as S
    import tile_scheduled_persistent_gb300 as tsp
    from dataclasses import replace

    torch.cuda.set_device(0)
    tsp.build()
    cfg = S.CONFIGS[args.config]
    w = S.model_weights(cfg)
    plan = tsp.Plan(tsp.ModelDesc.from_config(cfg), tsp.upload_weights(w))
    stream = torch.cuda.current_stream()

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
        with ClockSampler(0) as clk:
            for a, b in ev:
                a.record(stream)
                fn()
                b.record(stream)
            torch.cuda.synchronize()
        plan.check()
        ts = [a.elapsed_time(b) / 1e3 for a, b in ev]
        return statistics.mean(ts), statistics.median(ts), clk.summary()

    peaks = measured_peaks() or {}
    # kernels of one pass: embedding + norm; per layer Q/K/V GEMM, q/k post,
    # attention, combine, O GEMM, residual norm, gate/up GEMM, SwiGLU, down
    # GEMM, residual norm; LM-head GEMM and argmax
    launches_per_pass = 3 + 10 * cfg.n_layers
    line = {"n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic"}
    if args.mode == "prefill":
        n = args.prompt
        pc = replace(cfg, start_pos=0, max_pos=max(cfg.max_pos, n + 1))
        shape = (pc.n_layers, pc.n_kv_heads, pc.max_pos, pc.head_dim)
        kz = torch.zeros(shape, dtype=torch.bfloat16, device="cuda")
        vz = torch.zeros_like(kz)
        toks = torch.from_numpy(S.tokens(S.SEED_TOKENS, 3, n, cfg.vocab)).cuda()
        am = torch.zeros(n, dtype=torch.int32, device="cuda")
        mean_s, med_s, clk = timed(lambda: plan.forward(kz, vz, toks, 0, am))
        flops = 2.0 * (cfg.weight_bytes() / 2) * n
        peak = float(peaks.get("bf16_tflops", 1900.0))
        line.update({"metric": f"prefill tok/s, {n}-token prompt", "value": n / mean_s, "unit": "tok/s",
                     "ms_per_step": 1e3 * mean_s,
                     "config": {"workload": f"{cfg.name}: prompt of {n} seeded tokens from an empty cache, "
                                            f"passes of up to {tsp.MAX_FORWARD_TOKENS} tokens"},
                     "roofline": {"bound": "tensor", "achieved": flops / mean_s / 1e12, "peak": peak,
                                  "unit": "TFLOP/s", "frac": flops / mean_s / 1e12 / peak, "traffic": None,
                                  "note": "weight FLOPs 2 x parameters x tokens; attention not counted"},
                     "clocks": clk,
                     "gpu_launches": launches_per_pass * ((n + tsp.MAX_FORWARD_TOKENS - 1) // tsp.MAX_FORWARD_TOKENS)})
    else:
        k, v = S.kv_prefill(cfg)
        kc, vc = tsp.to_device_bf16(k), tsp.to_device_bf16(v)
        pr = torch.from_numpy(S.prompt(cfg)).cuda()
        g = torch.zeros(args.k, dtype=torch.int32, device="cuda")
        plan.decode(kc, vc, pr, cfg.start_pos, args.k, g)
        plan.check()
        inp = torch.cat([pr, g]).to(torch.int32)
        out = torch.zeros(args.k + 1, dtype=torch.int32, device="cuda")
        nacc = torch.zeros(1, dtype=torch.int32, device="cuda")
        mean_s, med_s, clk = timed(lambda: plan.verify(kc, vc, inp, cfg.start_pos, out, nacc))
        acc = int(nacc.item())
        line.update({"metric": f"verify-step emitted tok/s, k={args.k} drafts", "value": (acc + 1) / mean_s,
                     "unit": "tok/s", "ms_per_step": 1e3 * mean_s,
                     "config": {"workload": f"{cfg.name}: {cfg.start_pos} cached positions, {args.k} drafts "
                                            f"(the decode kernel's greedy tokens), {acc} accepted"},
                     "accepted": acc, "clocks": clk, "gpu_launches": launches_per_pass + 1})
    print(json.dumps(line), flush=True)
    plan.close()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--config", default="llama1b")
    ap.add_argument("--scheduler", default="all", choices=["counters", "waves", "flags", "all"])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--ref-tokens", type=int, default=2,
                    help="oracle decode tokens per timed step (CPU arms)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--weights", default="bf16", choices=["bf16", "int8"],
                    help="weight format of the plan (int8: weight-only, per-row scales)")
    ap.add_argument("--kv", default="bf16", choices=["bf16", "int8"],
                    help="KV cache format (int8: codes with per-row scales, smoothed keys)")
    ap.add_argument("--tokens", type=int, default=0,
                    help="decode tokens per step (default: the workload's 64); a smaller "
                         "launch of the same kernel, for profiler captures")
    ap.add_argument("--mode", default="decode", choices=["decode", "prefill", "verify"],
                    help="decode (the headline metric), or the multi-token arms")
    ap.add_argument("--prompt", type=int, default=512, help="prefill: prompt tokens")
    ap.add_argument("--k", type=int, default=16, help="verify: draft tokens")
    args = ap.parse_args()
    if args.mode != "decode":
        args.warmup = max(args.warmup, 3)
        return run_multi(args)
    if args.warmup < 3 and args.impl == "ours":
        log("warm-up raised to 3 steps")
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
