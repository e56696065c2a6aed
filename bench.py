#!/usr/bin/env python
"""Decode-step benchmark: tokens/s and achieved HBM GB/s per step on one GB300.

Default workload: the Llama-7B-shaped dense decoder in bf16 (E4096, H32,
Hkv32, L32, F11008, V32000), KV cache pre-filled to position 2048 with
generated N(0,1) bf16 entries, greedy decode of 128 tokens at batch 1.  A
step is one token through the whole decode path (embedding, 32 layers, LM head,
argmax), replayed from its CUDA graph.  Every 128 steps the position rewinds
to 2048 (a new 128-token decode of the same workload).  The weights (13.2 GB)
and KV cache are far larger than L2, so nothing stays cached between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Prints one JSON line (rank 0).  --impl reference times the CPU oracle (the
only reference this project has) on the same workload: whole decode steps on
the host cores, as many as --steps asks or as fit in 150 s.
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

METRIC = "decode tokens/s and achieved HBM GB/s per step vs ~8 TB/s peak, 1 GB300"
NOMINAL_HBM_GBS = 8000.0
KERNEL_SOURCES = ["transformer_decode_step_gb300/csrc/pnb_gemv.cu",
                  "transformer_decode_step_gb300/csrc/pnb_gemv_dev.cuh",
                  "transformer_decode_step_gb300/csrc/pnb_device.cuh",
                  "transformer_decode_step_gb300/csrc/pnb_kernels.cuh"]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=512)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llama7b_bf16")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layers", type=int, default=0,
                    help="use only the first N layers (small cases for ncu captures)")
    ap.add_argument("--batch", type=int, default=0,
                    help="slots of a batched workload (default: the workload's own)")
    ap.add_argument("--sample", action="store_true",
                    help="each step also draws the next token on the GPU (pnb_sample: "
                         "temperature 0.8, top-k 40, top-p 0.95, repetition penalty 1.1 "
                         "over 64 recent tokens) instead of taking the greedy one")
    ap.add_argument("--deterministic", action="store_true",
                    help="batched workloads: bitwise reproducible steps "
                         "(pnb_model_set_deterministic_batch: residual K parts in fixed point)")
    ap.add_argument("--kernel-trace", action="store_true",
                    help="single-sequence workloads: after the timed steps, one traced step "
                         "(per-CTA globaltimer stamps) gives each kernel's in-graph time, from the "
                         "previous launch's last CTA to its own, against its bytes at the measured "
                         "HBM peak (key kernel_trace of the JSON line)")
    ap.add_argument("--prefill", type=int, default=0,
                    help="instead of decode steps, time pnb_prefill of this many prompt tokens "
                         "from position 0 (one step = one prefill)")
    return ap.parse_args()


# ------------------------------------------------------------------ accounting

def step_bytes(shape, pos: int) -> int:
    """Algorithmic HBM bytes of one decode step at position pos: weights read
    (one embedding row, all projections of the chosen experts, router, norms,
    LM head), KV entries attended (window-limited) and the new KV entry."""
    es = shape.elem_bytes
    weights = int(shape.params_read_per_token() * shape.weight_bytes_per_param) + \
        (2 * shape.n_layer + 1) * shape.n_embd * 4
    n_att = pos + 1 if shape.sliding_window <= 0 else min(pos + 1, shape.sliding_window)
    per_pos = shape.n_layer * 2 * shape.n_kv_head * shape.head_dim * es
    return weights + n_att * per_pos + per_pos


def gateup_bytes(shape) -> int:
    """Algorithmic bytes of one gate/up launch: the chosen experts' [2F][E]
    weights, the residual and norm vectors read, the SwiGLU output written."""
    k = shape.expert_used if shape.expert_count > 0 else 1
    return k * shape.matrix_bytes(2 * shape.n_ff, shape.n_embd) + 2 * shape.n_embd * 4 + \
        k * shape.n_ff * 4


def kernel_hash() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """dram bytes per gate/up launch from the committed ncu summary, if it was
    taken on the current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", f"gateup_{workload}_ncu.txt")
    if not os.path.exists(path):
        return None
    vals = {}
    with open(path) as f:
        for line in f:
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                vals[k.strip()] = v.strip()
    if vals.get("kernel_sources_sha256_16") != kernel_hash():
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.samples = []
        self.proc = None
        self.t0 = self.t1 = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(gpu_index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError as e:
            self.error = str(e)

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.monotonic(), line.strip()))

    def start(self):
        self.t0 = time.monotonic()

    def stop(self):
        self.t1 = time.monotonic()

    def summary(self):
        if self.proc is None:
            return {"error": getattr(self, "error", "nvidia-smi unavailable")}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for t, line in self.samples:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            rows.append((t, parts))
        inside = [p for t, p in rows if self.t0 is not None and self.t0 <= t <= self.t1]
        use = inside or [p for _, p in rows]

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(p[1]) for p in use if num(p[1]) is not None]
        mx = [num(p[2]) for p in use if num(p[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in use for i in range(4) if p[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(inside), "power_w_max": max((num(p[3]) or 0) for p in use) if use else None}


# ------------------------------------------------------------------ distributed

def dist_setup(n_gpus: int):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world != n_gpus and world > 1:
        raise SystemExit(f"--gpus {n_gpus} but WORLD_SIZE={world}")
    return rank, world, local


def max_over_ranks(ms: float, dist=None, device: str = "cuda") -> float:
    """The slowest replica's time, on every rank (the job's time is the max)."""
    if dist is None:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ CPU oracle

def oracle_steps(w, seconds_budget: float, max_steps: int, warmup: int = 0, start_pos=None,
                 slot: int = 0):
    """Time whole greedy decode steps of the oracle (embedding, every layer, final
    norm, LM head and argmax), each step feeding the previous step's argmax from
    the workload's start token and pre-filled cache, rewinding to the start
    position when the cache is full (as the GPU arm does).  Stops after
    max_steps or once seconds_budget has passed (at least one step).
    Returns (tokens/s, steps timed, seconds, OpenMP threads used)."""
    import oracle
    import synth.workloads as wl

    P = w.prefill if start_pos is None else start_pos
    m = oracle.Model(w.shape, seed=w.seed)
    st = m.new_state()
    lo, hi = wl.kv_prefill_range(w.shape, P)
    st.prefill_synth(w.seed, slot, lo, hi)
    tok0 = wl.prompt_tokens(w, slot)[0]
    tok = tok0

    def step():
        nonlocal tok
        if st.pos >= w.shape.n_ctx:
            st.pos = P
            tok = tok0
        _, tok = st.forward(tok, want_logits=False)

    for _ in range(warmup):
        step()
    t0 = time.perf_counter()
    n = 0
    while n < max(1, max_steps):
        step()
        n += 1
        if time.perf_counter() - t0 > seconds_budget:
            break
    dt = time.perf_counter() - t0
    return n / dt, n, dt, oracle.max_threads()


def host_cpus() -> int:
    return os.cpu_count() or 0


# ------------------------------------------------------------------ main arms

def workload_config(w, extra=None, batch=None):
    s = w.shape
    batch = batch or w.batch or 1
    cfg = {"workload": f"{w.name}: E{s.n_embd} H{s.n_head} Hkv{s.n_kv_head} L{s.n_layer} "
                       f"F{s.n_ff} V{s.n_vocab} theta{s.rope_theta:g}"
                       + (f" window{s.sliding_window}" if s.sliding_window else "")
                       + (f" experts{s.expert_count}top{s.expert_used}" if s.expert_count else "")
                       + f", KV pre-filled to {w.prefill}, greedy decode of {w.steps} tokens, batch {batch}",
           "batch": batch, "weights_dtype": {0: "f32", 1: "bf16", 2: "q8_0", 3: "q4_0"}[s.dtype],
           "l2": "inputs larger than L2 (weights + KV per step >> 129 MB)"
                 if s.params_read_per_token() * s.weight_bytes_per_param > 129e6 else
                 "weights fit in L2 and stay resident between steps, as in a real decode loop "
                 "(no flush; this workload is latency-bound)"}
    if extra:
        cfg.update(extra)
    return cfg


SAMPLED = ("sampled on the GPU: temperature 0.8, top-k 40, top-p 0.95, penalty 1.1 over 64 "
           "tokens")


def is_batched(args, w) -> bool:
    return w.batch > 1 or args.batch > 1


def batched_starts(w, B: int):
    import synth.workloads as wl
    return wl.slot_positions(w.with_(batch=max(B, w.batch)))[:B]


def prefill_len(args, w) -> int:
    return min(args.prefill, w.shape.n_ctx)


def arm_config(args, w, world: int) -> dict:
    """The workload description both arms print (so the two lines name the same
    configuration)."""
    par = {"parallelism": f"replicas x{world}"}
    if args.prefill:
        T = prefill_len(args, w)
        return workload_config(w, {"prefill_tokens": T, "chunks_of_64": -(-T // 64), **par})
    if is_batched(args, w):
        B = args.batch or w.batch
        starts = batched_starts(w, B)
        extra = {**par, "slot_positions": f"U[{min(starts)}, {max(starts)}] + step"}
        if args.deterministic:
            extra["residual_k_parts"] = "64-bit fixed point (bitwise reproducible steps)"
        return workload_config(w, extra, batch=B)
    P = w.prefill
    return workload_config(w, {**par, "positions": f"{P}..{w.shape.n_ctx - 1}",
                               "next_token": SAMPLED if args.sample else "greedy (argmax)"})


def run_reference(args, w):
    """The reference arm: the CPU oracle, as it stands, on the host cores, timing
    whole decode steps of the same workload (rank 0 only under torchrun).  A
    batched workload's step is one slot's token (the oracle runs slots one at a
    time); a prefill's step is one prompt token fed from position 0."""
    rank, world, local = dist_setup(args.gpus)
    if rank != 0:
        return 0
    import synth.workloads as wl
    batched = is_batched(args, w) and not args.prefill
    if args.prefill:
        w_ref = w.with_(prefill=0, slot_pos_range=None)
        start = 0
    else:
        w_ref = w
        start = batched_starts(w, args.batch or w.batch)[0] if batched else None
    warm = min(max(args.warmup, 0), 3)
    tps, n, dt, threads = oracle_steps(w_ref, 150.0, max_steps=args.steps, warmup=warm,
                                       start_pos=start)
    what = ("tokens of slot 0 from its seeded start position (the oracle runs slots one at a time)"
            if batched else "tokens fed one per forward from position 0 (a prompt token's cost)" if args.prefill
            else "greedy decode steps from the pre-filled cache")
    line = {"impl": "reference", "metric": "prefill_tokens_per_s" if args.prefill else METRIC,
            "value": tps, "unit": "tokens/s", "n_gpus": args.gpus, "steps": n,
            "steps_requested": args.steps, "warmup": warm, "ms_per_step": 1000.0 * dt / n,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded generated weights and KV cache)",
            "config": arm_config(args, w, args.gpus),
            "step_is": "one whole token through the oracle: embedding, every layer, final norm, "
                        "LM head and argmax",
            "cpu_baseline": {"value": tps, "unit": "tokens/s", "cores": threads,
                             "host_cpus": host_cpus(), "kind": "oracle",
                             "sample": f"{n} whole {what}, {dt:.1f} s on {threads} OpenMP "
                                       f"threads (weights regenerated from the seed inside "
                                       f"each step)"},
            "e2e": {"value": tps, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args, w):
    import torch

    import transformer_decode_step_gb300 as pnb

    rank, world, local = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    s = w.shape
    P = w.prefill
    budget = s.n_ctx - P                       # decode steps one pass can take
    sm = pnb.SynthModel(s, w.seed)
    st = sm.new_state(start_pos=P, slot=rank)
    import synth
    import synth.workloads as wl
    tok0 = wl.prompt_tokens(w, rank)[0]
    am = torch.empty(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()
    sampling = pnb.sampling_params(0.8, 1.1, 40, 0.95, 1234 + rank) if args.sample else None
    lg = torch.empty(s.n_vocab, dtype=torch.float32, device="cuda") if args.sample else None
    # the penalty window: 64 seeded token ids
    recent = torch.tensor(synth.uniform_int(synth.key(w.seed, synth.TOKENS, 1, rank), 0, 64, 0,
                                            s.n_vocab), dtype=torch.int32,
                          device="cuda") if args.sample else None

    def one_pass_step(i):
        if i % budget == 0:
            st.set_pos(P)
            st.forward(tok0, argmax=am, logits=lg)
        else:
            st.forward(pnb.PNB_TOKEN_PREV, argmax=am, logits=lg)
        if sampling is not None:
            st.sample(lg, sampling, recent=recent, token=am)

    # warm-up (captures the graph)
    for i in range(max(3, args.warmup)):
        one_pass_step(i)
    torch.cuda.synchronize()
    if st.device_error():
        raise SystemExit("device error during warm-up")

    clocks = ClockSampler(local)
    time.sleep(0.3)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks.start()
    e0.record(stream)
    for i in range(args.steps):
        one_pass_step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    clocks.stop()
    if dist:
        dist.barrier()
    ms = max_over_ranks(e0.elapsed_time(e1), dist)
    err = st.device_error()
    clk = clocks.summary()
    passes = (args.steps + budget - 1) // budget
    launches = args.steps * (sm.step_kernel_count() + (1 if args.sample else 0)) + 2 * passes
    ms_step = ms / args.steps
    tokens_per_s = world * args.steps / (ms / 1000.0)
    mean_bytes = sum(step_bytes(s, P + (i % budget)) for i in range(args.steps)) / args.steps
    step_gbs = mean_bytes / (ms_step / 1000.0) / 1e9

    # dominant kernel (SwiGLU gate/up: the largest weight stream of the step) timed alone
    L = s.n_layer
    for l in range(3):
        st.run_kernel(pnb.PNB_KERNEL_GATE_UP, l % L)
    reps = 3 * L
    k0, k1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    k0.record(stream)
    for i in range(reps):
        st.run_kernel(pnb.PNB_KERNEL_GATE_UP, i % L)
    k1.record(stream)
    torch.cuda.synchronize()
    k_ms = k0.elapsed_time(k1) / reps
    kb = gateup_bytes(s)
    peaks, peak_kind = measured_peaks()
    k_gbs = kb / (k_ms / 1000.0) / 1e9
    traffic = recorded_traffic(w.name)

    # end to end through the C ABI: the host feeds each token by value and reads
    # the greedy token back (pinned host memory) before the next step
    pinned = torch.empty(1, dtype=torch.int32, pin_memory=True)
    e2e_steps = min(args.steps, budget)
    st.set_pos(P)
    torch.cuda.synchronize()
    tok = tok0
    t0 = time.perf_counter()
    for i in range(e2e_steps):
        st.forward(tok, argmax=am, logits=lg)
        if sampling is not None:
            st.sample(lg, sampling, recent=recent, token=am)
        pinned.copy_(am, non_blocking=True)
        stream.synchronize()
        tok = int(pinned[0])
    e2e_s = time.perf_counter() - t0
    e2e_tps = world * e2e_steps / e2e_s   # every rank runs the same loop
    # (after the e2e loop: turning the trace on and off re-captures the step's graph)
    ktrace = kernel_trace(st, s, P, tok0, peaks["hbm_gbs"]) if args.kernel_trace else None

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tps, n, dt, threads = oracle_steps(w, 15.0, max_steps=16)
        cpu = {"value": tps, "unit": "tokens/s", "cores": threads, "host_cpus": host_cpus(),
               "kind": "oracle",
               "sample": f"{n} whole greedy decode steps of the workload from position {P} "
                         f"(embedding, {L} layers, LM head), {dt:.1f} s on {threads} OpenMP "
                         f"threads"}

    if rank == 0:
        line = {"metric": METRIC, "value": tokens_per_s, "unit": "tokens/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": {0: "f32", 1: "bf16", 2: "q8_0", 3: "q4_0"}[s.dtype], "data": "synthetic (seeded generated weights and KV cache)",
                "config": arm_config(args, w, world),
                "hbm_gbs_step": step_gbs, "hbm_frac_of_8tbs": step_gbs / NOMINAL_HBM_GBS,
                "hbm_frac_of_measured": step_gbs / peaks["hbm_gbs"],
                "bytes_per_step": mean_bytes,
                "roofline": {"bound": "hbm", "kernel": "k_gateup (RMSNorm + gate/up GEMV + SwiGLU)",
                             "achieved": k_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                             "frac": k_gbs / peaks["hbm_gbs"], "traffic": traffic,
                             "bytes_per_launch": kb, "launch_us": k_ms * 1000.0,
                             "peak_source": f"{peak_kind} hbm_gbs (MEASURED_PEAKS.json)",
                             "timing": "CUDA events over 96 launches of the kernel alone, "
                                       "rotating over the 32 layers' weights"},
                "clocks": clk, "gpu_launches": launches, "device_error": err,
                "e2e": {"value": e2e_tps, "unit": "tokens/s", "h2d_bytes_per_step": 4,
                        "d2h_bytes_per_step": 4, "steps": e2e_steps,
                        "how": "pnb_forward with the token passed by value from the host, "
                               "argmax copied to pinned host memory and synchronised every step"},
                "cpu_baseline": cpu}
        if ktrace is not None:
            line["kernel_trace"] = ktrace
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


KERNEL_KINDS = ["qkv", "attention", "o-proj", "router", "gate/up", "down"]


def kernel_trace(st, s, P, tok0, peak_gbs):
    """In-graph time of each kernel of one decode step at position P + 3 (the
    library's per-CTA timestamps, launch order 6 * layer + kind, then the LM
    head): from the previous launch's last CTA end to this launch's last CTA
    end, averaged over the layers, beside the kernel's algorithmic bytes at the
    measured HBM peak."""
    import numpy as np
    import torch

    import transformer_decode_step_gb300 as pnb
    L = s.n_layer
    buf = torch.zeros((7 * L + 2) * 256 * 8, dtype=torch.int64, device="cuda")
    am = torch.empty(1, dtype=torch.int32, device="cuda")
    st.set_pos(P)
    st.forward(tok0, argmax=am)
    st.set_trace(buf)
    for _ in range(3):
        st.forward(pnb.PNB_TOKEN_PREV, argmax=am)
    torch.cuda.synchronize()
    st.set_trace(None)
    pos = P + 3
    t = buf.cpu().numpy().reshape(7 * L + 2, 256, 8)[:6 * L + 1].astype(np.float64)
    k = s.expert_used if s.expert_count > 0 else 1
    n_att = pos + 1 if s.sliding_window <= 0 else min(pos + 1, s.sliding_window)
    mb = s.matrix_bytes
    Hd = s.n_head * s.head_dim
    bytes_of = {"qkv": mb((s.n_head + 2 * s.n_kv_head) * s.head_dim, s.n_embd),
                "attention": n_att * 2 * s.n_kv_head * s.head_dim * s.elem_bytes,
                "o-proj": mb(s.n_embd, Hd), "router": mb(max(1, s.expert_count), s.n_embd),
                "gate/up": k * mb(2 * s.n_ff, s.n_embd), "down": k * mb(s.n_embd, s.n_ff),
                "lm head": mb(s.n_vocab, s.n_embd)}
    per = {}
    prev_end = None
    for ph in range(6 * L + 1):
        rows = t[ph][t[ph][:, 0] > 0]
        if rows.shape[0] == 0:
            continue
        end = rows[:, 5].max()
        kind = "lm head" if ph == 6 * L else KERNEL_KINDS[ph % 6]
        if prev_end is not None:
            per.setdefault(kind, []).append((end - prev_end) / 1000.0)
        prev_end = end
    out = {"unit": "us", "position": pos, "peak_gbs": peak_gbs, "kernels": {}}
    for kind, us in per.items():
        bound = bytes_of[kind] / (peak_gbs * 1e9) * 1e6
        m = float(np.mean(us))
        out["kernels"][kind] = {"launches": len(us), "us": m, "bound_us": bound,
                                "bound_frac": bound / m, "bytes": bytes_of[kind]}
    out["step_us_traced"] = float(sum(np.sum(v) for v in per.values()))
    return out


def batch_step_bytes(shape, positions) -> int:
    """Algorithmic HBM bytes of one batched step: the weights once (for MoE,
    every expert: the batched step streams each expert once for all slots), each
    slot's attended KV entries and its new entry."""
    es = shape.elem_bytes
    params = shape.params_read_per_token()
    if shape.expert_count > 0:
        params += (shape.expert_count - shape.expert_used) * 3 * shape.n_ff * shape.n_embd * \
            shape.n_layer
    weights = int(params * shape.weight_bytes_per_param) + (2 * shape.n_layer + 1) * shape.n_embd * 4
    per_pos = shape.n_layer * 2 * shape.n_kv_head * shape.head_dim * es
    kv = 0
    for p in positions:
        n_att = p + 1 if shape.sliding_window <= 0 else min(p + 1, shape.sliding_window)
        kv += (n_att + 1) * per_pos
    return weights + kv


def run_batched(args, w):
    """The batched-slot workload: B sequences at their own positions, one token
    each per step, through pnb_forward_batch."""
    import torch

    import synth.workloads as wl
    import transformer_decode_step_gb300 as pnb

    rank, world, local = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    s = w.shape
    B = args.batch or w.batch
    starts = batched_starts(w, B)
    budget = s.n_ctx - max(starts)
    sm = pnb.SynthModel(s, w.seed)
    sm.model.set_deterministic_batch(args.deterministic)
    # replica r serves its own slots (seeded by slot id r * B + b)
    states = [sm.new_state(p, slot=rank * B + b) for b, p in enumerate(starts)]
    tok0 = torch.tensor([wl.prompt_tokens(w, rank * B + b)[0] for b in range(B)],
                        dtype=torch.int32, device="cuda")
    am = torch.empty(B, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()

    def one_pass_step(i):
        if i % budget == 0:
            for b, st in enumerate(states):
                st.set_pos(starts[b])
            sm.model.forward_batch(states, tokens=tok0, argmax=am)
        else:
            sm.model.forward_batch(states, argmax=am)

    for i in range(max(3, args.warmup)):
        one_pass_step(i)
    torch.cuda.synchronize()
    if any(st.device_error() for st in states):
        raise SystemExit("device error during warm-up")
    clocks = ClockSampler(local)
    time.sleep(0.3)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks.start()
    e0.record(stream)
    for i in range(args.steps):
        one_pass_step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    clocks.stop()
    if dist:
        dist.barrier()
    ms = max_over_ranks(e0.elapsed_time(e1), dist)
    err = max(st.device_error() for st in states)
    clk = clocks.summary()
    passes = (args.steps + budget - 1) // budget
    ms_step = ms / args.steps
    tokens_per_s = world * B * args.steps / (ms / 1000.0)
    mean_bytes = sum(batch_step_bytes(s, [p + (i % budget) for p in starts])
                     for i in range(args.steps)) / args.steps
    step_gbs = mean_bytes / (ms_step / 1000.0) / 1e9
    peaks, peak_kind = measured_peaks()

    # end to end: every step the B tokens go host -> device from pinned memory
    # and the B greedy tokens come back
    pinned_in = torch.tensor([wl.prompt_tokens(w, rank * B + b)[0] for b in range(B)],
                             dtype=torch.int32).pin_memory()
    pinned_out = torch.empty(B, dtype=torch.int32, pin_memory=True)
    tk = torch.empty(B, dtype=torch.int32, device="cuda")
    e2e_steps = min(args.steps, budget)
    for b, st in enumerate(states):
        st.set_pos(starts[b])
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(e2e_steps):
        tk.copy_(pinned_in, non_blocking=True)
        sm.model.forward_batch(states, tokens=tk, argmax=am)
        pinned_out.copy_(am, non_blocking=True)
        stream.synchronize()
        pinned_in.copy_(pinned_out)
    e2e_s = time.perf_counter() - t0
    e2e_tps = world * B * e2e_steps / e2e_s

    cpu = None
    L = s.n_layer
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tps, n, dt, threads = oracle_steps(w, 15.0, max_steps=16, start_pos=starts[0])
        cpu = {"value": tps, "unit": "tokens/s", "cores": threads, "host_cpus": host_cpus(),
               "kind": "oracle",
               "sample": f"{n} whole greedy decode steps of slot 0 from position {starts[0]} "
                         f"(the oracle runs slots one at a time), {dt:.1f} s on {threads} "
                         f"OpenMP threads"}
    if rank == 0:
        line = {"metric": METRIC, "value": tokens_per_s, "unit": "tokens/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "bf16", "data": "synthetic (seeded generated weights and KV cache)",
                "config": arm_config(args, w, world),
                "hbm_gbs_step": step_gbs, "hbm_frac_of_8tbs": step_gbs / NOMINAL_HBM_GBS,
                "hbm_frac_of_measured": step_gbs / peaks["hbm_gbs"], "bytes_per_step": mean_bytes,
                "roofline": {"bound": "hbm", "kernel": "whole batched step (weights once + every slot's KV)",
                             "achieved": step_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                             "frac": step_gbs / peaks["hbm_gbs"], "traffic": None,
                             "peak_source": f"{peak_kind} hbm_gbs (MEASURED_PEAKS.json)",
                             "timing": "CUDA events over the timed steps"},
                "clocks": clk, "gpu_launches": args.steps * sm.step_kernel_count(B) + passes * B,
                "device_error": err,
                "e2e": {"value": e2e_tps, "unit": "tokens/s", "h2d_bytes_per_step": 4 * B,
                        "d2h_bytes_per_step": 4 * B, "steps": e2e_steps,
                        "how": "pnb_forward_batch with the B tokens copied from pinned host memory "
                               "and the B greedy tokens copied back and synchronised every step"},
                "cpu_baseline": cpu}
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


def run_prefill(args, w):
    """Prompt tokens per second of pnb_prefill: a seeded prompt of --prefill
    tokens fed to a state from position 0, --steps times (the position is set
    back to 0 before each; the prefill rewrites every cache position it reads)."""
    import torch

    import synth.workloads as wl
    import transformer_decode_step_gb300 as pnb

    rank, world, local = dist_setup(args.gpus)
    if world > 1 and rank != 0:
        return 0
    torch.cuda.set_device(local)
    s = w.shape
    T = prefill_len(args, w)
    sm = pnb.SynthModel(s, w.seed)
    st = sm.new_state()
    rng = __import__("numpy").random.default_rng(w.seed)
    prompt = torch.tensor(rng.integers(0, s.n_vocab, size=T), dtype=torch.int32, device="cuda")
    am = torch.empty(T, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()
    for _ in range(max(3, args.warmup)):
        st.set_pos(0)
        st.prefill(prompt, argmax=am)
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    ms = 0.0
    for _ in range(args.steps):
        st.set_pos(0)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        st.prefill(prompt, argmax=am)
        e1.record(stream)
        torch.cuda.synchronize()
        ms += e0.elapsed_time(e1)
    clocks.stop()
    err = st.device_error()
    # end to end: the prompt from pinned host memory, the last greedy token back
    pinned = prompt.cpu().pin_memory()
    out = torch.empty(1, dtype=torch.int32, pin_memory=True)
    tk = torch.empty_like(prompt)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        st.set_pos(0)
        tk.copy_(pinned, non_blocking=True)
        st.prefill(tk, argmax=am)
        out.copy_(am[-1:], non_blocking=True)
        stream.synchronize()
    e2e = T * args.steps / (time.perf_counter() - t0)
    tps = T * args.steps / (ms / 1000.0)
    line = {"metric": "prefill_tokens_per_s", "value": tps, "unit": "tokens/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded generated weights, seeded prompt)",
            "config": arm_config(args, w, 1),
            "weight_bytes_per_chunk": int(s.params_read_per_token() * s.weight_bytes_per_param),
            "clocks": clocks.summary(), "device_error": err,
            "e2e": {"value": e2e, "unit": "tokens/s", "h2d_bytes_per_step": 4 * T,
                    "d2h_bytes_per_step": 4, "how": "prompt copied from pinned host memory, "
                    "the last greedy token read back, per prefill"}}
    print(json.dumps(line), flush=True)
    return 0


def main():
    args = parse()
    import dataclasses

    import synth.workloads as wl
    w = wl.BY_NAME[args.workload]
    if args.layers:
        w = w.with_(shape=dataclasses.replace(w.shape, n_layer=args.layers),
                    name=f"{w.name}_L{args.layers}")
    import __graft_entry__
    __graft_entry__.build(import_package=args.impl == "ours")
    if args.impl == "reference":
        return run_reference(args, w)
    if args.prefill:
        return run_prefill(args, w)
    if w.batch > 1 or args.batch > 1:
        return run_batched(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
