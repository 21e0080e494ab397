#!/usr/bin/env python
"""Benchmark of the GB300 MoE layer forward: tokens/s and fraction of the binding roofline.

One step = one whole forward of the layer (route -> permute -> L1+SwiGLU -> L2 -> reduce) on
one batch of synthetic, seeded inputs already resident in HBM.  Default workload: the pages'
decode shape (T=8, H=7168, I=2048, E=256, K=6, MXFP4 weights), which is weight-bandwidth bound.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Prints one JSON line (rank 0).  Under torchrun each rank runs an independent replica (the
layer is replicated per GPU, no collective on the data path); value = tokens of all ranks /
max over ranks of the step time.
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

# The CPU baseline (the float64 oracle) runs its experts on ORACLE_THREADS worker threads with
# single-threaded BLAS, so the thread count it reports is the one that ran.  Set before numpy loads.
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import numpy as np  # noqa: E402

import synth  # noqa: E402

FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


SPIN_CYCLES = 1_000_000      # ~0.5 ms at 2 GHz, outside the timed events


def launches_per_forward(w, naive=False, single=False):
    """Kernel launches of one forward call, mirroring the library's dispatch."""
    if single:
        return 1                                  # moe_forward_single_launch: the whole layer
    tk = w.T * w.K
    route = 1 if w.T <= 16 else 3                 # fused small-batch route, else gate split + gate GEMM + top-K
    reduce = 0 if w.T <= 32 else 1                # small batches reduce inside the L2 epilogue
    if w.fmt in I8_FMTS:
        # route, per-token act quant, permute indices (one kernel up to 1024 pairs, else count + place),
        # then the row gather to fp16, L1, the per-row h requant and L2
        return route + 1 + (1 if tk <= 1024 else 2) + 4 + reduce
    # permute: the row copy inside the small kernel up to 128 pairs, else a copy kernel after the
    # small kernel (up to 1024 pairs) or after count + place
    permute = 1 if tk <= 128 else (2 if tk <= 1024 else 3)
    if naive:
        permute = 0                               # the routing launch writes the tiny-batch layout
    elif w.fmt == "nvfp4":
        permute = 1 if tk <= 1024 else 2          # NVFP4 reads the token-order rows: no row or scale copy
    if w.fmt == "mxfp4":
        ffn = 1                                   # L1 and L2 in one launch
    else:
        ffn = 4                                   # bf16 activation rows + GEMM, for L1 and for L2
    return route + permute + ffn + reduce


HEADLINE = "decode"
I8_FMTS = ("int8", "int8b")
# timed steps per workload in the per-config part of the default run (at most --steps)
PER_CONFIG_STEPS = {"tiny": 300, "decode": 300, "batched": 200, "prefill": 60, "skewed": 20}


def oracle_threads():
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except Exception:
        return max(1, os.cpu_count() or 1)


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=1000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--workload", default=None, choices=sorted(synth.WORKLOADS),
                   help="measure this workload only; by default the headline (decode) line also carries "
                        "per_config entries for the other workloads")
    p.add_argument("--no-per-config", action="store_true", help="headline workload only")
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--cpu-seconds", type=float, default=12.0,
                   help="budget of the oracle CPU baseline per workload (0 skips it, e.g. under a profiler)")
    p.add_argument("--ref-seconds", type=float, default=150.0,
                   help="time budget of the reference (oracle) arm's timed steps")
    p.add_argument("--experts", type=int, default=None,
                   help="override E (smaller cases of the same kernels for profiler captures)")
    p.add_argument("--tokens", type=int, default=None,
                   help="override T (smaller cases of the same kernels for profiler captures)")
    p.add_argument("--weights-in-l1", action="store_true",
                   help="apply the routing weights in the L1 epilogue and sum without weights "
                        "(moe_forward_l1_weighted) instead of weighting in the reduce")
    p.add_argument("--weights", default="workload", choices=["workload", "int8", "int8b"],
                   help="the workload's FP4 weight format, or the INT8 variant (int8 weights with per-channel "
                        "scales, int8 activations with per-token scales: moe_forward_i8; int8b: [256, 256] weight blocks, "
                        "per-256-group activation scales) on the same shapes")
    p.add_argument("--l1-input", default="auto", choices=["auto", "token", "permuted"],
                   help="stage-by-stage timing: the L1 GEMM reads the token-order activation through "
                        "sorted_token_ids or the permute's row copy x_perm; auto: as moe_forward does "
                        "(token order with NVFP4 weights, the copy with MXFP4)")
    p.add_argument("--layout", default="contiguous", choices=["contiguous", "batched", "naive", "single"],
                   help="permuted-row layout: expert-contiguous segments padded to align (moe_forward) or "
                        "BatchedExperts slots of max_tokens = max(16, the smallest power of two >= T) (moe_forward_batched) or "
                        "the tiny-batch layout, one 16-row block per (token, expert) pair, no sort (moe_forward_naive); "
                        "single: moe_forward's layout with the whole layer in one launch (moe_forward_single_launch, "
                        "up to 16 tokens, MXFP4)")
    return p.parse_args()


def world():
    return int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0"))


def max_over_ranks(x, device=None):
    """The largest value of x over the ranks of the default process group (x itself without one):
    the whole job takes as long as its slowest replica."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world_size, tokens_per_rank, ms):
    """Whole-job throughput: every rank processes its own tokens_per_rank in the slowest rank's ms."""
    return world_size * tokens_per_rank / (ms / 1e3)


def workload_config(w):
    acts = {"int8": "INT8 activations (fp32 scale per token)",
            "int8b": "INT8 activations (fp32 scale per token and 256-column group)"}.get(
        w.fmt, "FP8 E4M3 activations (UE8M0/128)")
    wts = {"int8": "INT8 weights (fp32 scale per channel)",
           "int8b": "INT8 weights (fp32 scale per [256, 256] block)"}.get(w.fmt, f"{w.fmt.upper()} weights")
    return {"workload": f"{w.name}: T={w.T} H={w.H} I={w.I} E={w.E} K={w.K} align={w.align} "
                        f"{w.score_fn} {wts}, {acts}",
            "T": w.T, "H": w.H, "I": w.I, "E": w.E, "K": w.K, "align": w.align, "weights": w.fmt}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


def traffic_record(kernel_file, workload):
    """DRAM bytes per launch from a committed ncu summary, if taken on the current kernel source."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            recs = json.load(f)
        with open(kernel_file, "rb") as f:
            sha = hashlib.sha256(f.read()).hexdigest()[:16]
        r = recs.get(workload)
        if r and r.get("source_sha") == sha:
            return r["bytes_per_launch"]
    except Exception:
        pass
    return None


# ------------------------------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None
        # the raw samples go to a scratch file (MOE_BENCH_CLOCKS_DIR, else the system temp
        # directory); the JSON line carries their summary
        base = os.environ.get("MOE_BENCH_CLOCKS_DIR") or tempfile.gettempdir()
        self.path = os.path.join(base, f"moe_bench_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 8:
                    continue
                try:
                    sm.append(float(parts[0]))
                    smax.append(float(parts[1]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[4:8]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------------------------------ CPU oracle

def oracle_forward(w, workers=1):
    """The oracle's whole-layer function for the workload's weight format, as f(inp, prov, tokens)."""
    if w.fmt in I8_FMTS:
        from oracle import int8 as QI
        return lambda inp, prov, tokens: QI.forward_i8(inp, prov, w.K, w.align, w.score_fn, w.renormalize,
                                                       tokens=tokens, block=w.fmt == "int8b")
    from oracle import moe as O
    return lambda inp, prov, tokens: O.forward(inp, prov, w.fmt, w.K, w.align, w.score_fn, w.renormalize,
                                               tokens=tokens, workers=workers)


ORACLE_BATCH = 8     # tokens per oracle call of the CPU baseline (the decode batch)


def oracle_tokens_per_s(w, inp, stack, budget_s):
    """Times the float64 oracle on batches of whole tokens of the workload until the budget is spent.
    Its experts run on oracle_threads() worker threads (BLAS single-threaded)."""
    n_thr = 1 if w.fmt in I8_FMTS else oracle_threads()
    fwd = oracle_forward(w, n_thr)
    prov = (lambda e: {k: (v[e] if v is not None else None) for k, v in stack.items()})
    done, t0 = 0, time.perf_counter()
    while done < w.T:
        toks = list(range(done, min(w.T, done + ORACLE_BATCH)))
        fwd(inp, prov, toks)
        done += len(toks)
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    sample = (f"{done} token(s) of the {w.name} workload in batches of up to {ORACLE_BATCH} (routing of all {w.T} "
              f"tokens each time), {dt:.1f} s, numpy float64, experts on {n_thr} thread(s), BLAS single-threaded")
    return {"value": done / dt, "unit": "tokens/s", "cores": n_thr, "kind": "oracle", "sample": sample}


def run_reference(args, w):
    """The oracle as the reference arm: each step is one token of the workload on the host cores."""
    W, rank, _ = world()
    if rank != 0:
        return
    inp = synth.layer_inputs(w)
    stack = synth.all_expert_weights(w)
    cores = 1 if w.fmt in I8_FMTS else oracle_threads()
    fwd = oracle_forward(w, cores)
    prov = (lambda e: {k: (v[e] if v is not None else None) for k, v in stack.items()})
    nb = min(ORACLE_BATCH, w.T)
    # warm-up (at most one step: each oracle step is seconds long), then as many timed steps as fit
    # the time budget, at most --steps; the line reports the number actually run
    t0 = time.perf_counter()
    for i in range(min(args.warmup, 1)):
        fwd(inp, prov, [(i * nb + j) % w.T for j in range(nb)])
    est = max(time.perf_counter() - t0, 1e-3)
    steps = max(1, min(args.steps, int(args.ref_seconds / est)))
    times = []
    for i in range(steps):
        t0 = time.perf_counter()
        fwd(inp, prov, [(i * nb + j) % w.T for j in range(nb)])
        times.append(time.perf_counter() - t0)
    ms = 1e3 * statistics.mean(times)
    value = nb * 1e3 / ms
    sample = (f"{nb} token(s) of the {w.name} workload per step (routing of all {w.T} tokens + those tokens' "
              f"experts), experts on {cores} thread(s), BLAS single-threaded")
    line = {"impl": "reference", "metric": "MoE-layer tokens/s", "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": steps, "warmup": min(args.warmup, 1), "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
            "config": workload_config(w),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------------------------ GPU arm

def algorithmic_bytes(w, n_touched):
    """Bytes the method must move per launch of each stage (padding and untouched experts excluded)."""
    TK = w.T * w.K
    if w.fmt in I8_FMTS:
        # int8 codes + fp32 channel scales; activations int8 + one fp32 scale per row
        # (int8b: one fp32 scale per [256, 256] weight block and per 256-column group of a row)
        if w.fmt == "int8":
            w13 = n_touched * (2 * w.I * w.H + 2 * w.I * 4)
            w2 = n_touched * (w.H * w.I + w.H * 4)
            sx, sh = 4, 4
        else:
            w13 = n_touched * (2 * w.I * w.H + (2 * w.I // 256) * (w.H // 256) * 4)
            w2 = n_touched * (w.H * w.I + (w.H // 256) * (w.I // 256) * 4)
            sx, sh = w.H // 256 * 4, w.I // 256 * 4
        l1 = w13 + TK * (w.H + sx) + TK * (w.I + sh)
        l2 = w2 + TK * (w.I + sh) + TK * w.H * 2
        return {"l1": l1, "l2": l2, "ffn": w13 + w2 + TK * (w.H + sx) + TK * w.H * 2,
                "layer": w13 + w2 + 4 * w.E * w.H + 2 * w.T * w.H * 2}
    if w.fmt == "mxfp4":
        w13 = n_touched * (2 * w.I * w.H // 2 + 2 * w.I * w.H // 32)
        w2 = n_touched * (w.H * w.I // 2 + w.H * w.I // 32)
    else:
        w13 = n_touched * (2 * w.I * w.H // 2 + 2 * w.I * w.H // 16 + 4)
        w2 = n_touched * (w.H * w.I // 2 + w.H * w.I // 16 + 4)
    l1 = w13 + TK * (w.H + w.H // 128) + TK * (w.I + w.I // 128)
    l2 = w2 + TK * (w.I + w.I // 128) + TK * w.H * 2
    return {"l1": l1, "l2": l2, "ffn": w13 + w2 + TK * (w.H + w.H // 128) + TK * w.H * 2,
            "layer": w13 + w2 + 4 * w.E * w.H + 2 * w.T * w.H * 2}


def kernel_name(stage, fmt):
    if fmt in I8_FMTS:
        return {"ffn": "INT8 L1 (row gather, GEMM, h requant) then L2 (h to fp16, GEMM)",
                "l1": "INT8 L1 (row gather, GEMM, h requant)", "l2": "INT8 L2 (h to fp16, GEMM)"}[stage]
    if stage == "ffn":
        return "L1+L2 grouped GEMM (one launch)" if fmt == "mxfp4" else "L1 then L2 grouped GEMM"
    return f"{stage} grouped GEMM"


def measure(args, w, steps, warmup, cpu_seconds, dev):
    """One workload: device-timed forward steps, per-stage durations, end-to-end steps, CPU baseline.
    Returns the pieces of a JSON line (rank 0 gets the CPU baseline)."""
    import torch
    import moe_expert_ffn_sqrt_gb300 as M

    W, rank, _ = world()
    inp = synth.layer_inputs(w)
    stack = synth.all_expert_weights(w)

    def d(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    i8 = w.fmt in I8_FMTS
    if i8:      # int8 codes; the channel or block scales travel as the weight's tscale
        w13 = M.Weight(d(stack["w13_q"]), None, d(stack["w13_sf"]), w.fmt, pair=2)
        w2 = M.Weight(d(stack["w2_q"]), None, d(stack["w2_sf"]), w.fmt, pair=1)
    else:
        w13 = M.Weight(d(stack["w13_q"]), d(stack["w13_sf"]), None if stack["w13_ts"] is None else d(stack["w13_ts"]),
                       w.fmt, pair=2)
        w2 = M.Weight(d(stack["w2_q"]), d(stack["w2_sf"]), None if stack["w2_ts"] is None else d(stack["w2_ts"]), w.fmt,
                      pair=1)
    T = w.T
    hidden_host = torch.from_numpy(inp["hidden"].view(np.int16)).view(torch.bfloat16).pin_memory()
    hidden = hidden_host.to(dev)
    w_gate = d(inp["w_gate"])
    gate_bias = None if inp["gate_bias"] is None else d(inp["gate_bias"])
    e_bias = None if inp["e_score_bias"] is None else d(inp["e_score_bias"])
    batched = args.layout == "batched"
    naive = args.layout == "naive"
    single = args.layout == "single"
    # BatchedExperts slot: the smallest power of two >= T, at least 16 (one expert per GEMM row block)
    S = max(16, 1 << max(0, (T - 1).bit_length()))
    if batched:
        ws = M.new_workspace_batched(T, w.H, w.I, w.E, w.K, S, device=dev)
    elif i8:
        ws = M.new_workspace_i8(T, w.H, w.I, w.E, w.K, w.align, device=dev)
    else:
        ws = M.new_workspace(T, w.H, w.I, w.E, w.K, M.NAIVE_ROWS if naive else w.align, device=dev)
    out = torch.empty(T, w.H, dtype=torch.bfloat16, device=dev)
    out_host = torch.empty(T, w.H, dtype=torch.bfloat16).pin_memory()
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)     # > L2 (126 MB)

    def step():
        if i8:
            M.forward_i8(hidden, w_gate, gate_bias, e_bias, w.I, w.K, w.align, w.score_fn, w.renormalize, w13, w2, out,
                         ws)
        elif naive:
            M.forward_naive(hidden, w_gate, gate_bias, e_bias, w.I, w.K, w.score_fn, w.renormalize, w13, w2, out, ws)
        elif batched:
            M.forward_batched(hidden, w_gate, gate_bias, e_bias, w.I, w.K, S, w.score_fn, w.renormalize, w13, w2, out,
                              ws)
        else:
            M.forward(hidden, w_gate, gate_bias, e_bias, w.I, w.K, w.align, w.score_fn, w.renormalize, w13, w2, out,
                      ws, weights_in_l1=args.weights_in_l1, single_launch=single)

    def barrier():
        if W > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    for _ in range(warmup):
        step()
    st = M.get_error(ws)
    if st != M.OK:
        raise RuntimeError(f"device status after warm-up: {M.status_str(st)}")

    # ---- timed region: one forward per step, L2 flushed between steps (outside the events)
    K = steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    clocks = ClockSampler(dev.index)
    clocks.start()
    time.sleep(0.3)
    barrier()
    for i in range(K):
        flush.fill_(i & 0xFF)
        # a GPU-side spin (outside the events) keeps the host ahead, so that a slow or contended host
        # cannot stretch the device time between the events; the end-to-end loop below has none
        torch.cuda._sleep(2 * SPIN_CYCLES)
        ev[i][0].record()
        step()
        ev[i][1].record()
    barrier()
    clk = clocks.stop()
    times = [a.elapsed_time(b) for a, b in ev]
    ms = max_over_ranks(statistics.mean(times), dev)
    st = M.get_error(ws)
    if st != M.OK:
        raise RuntimeError(f"device status after timed steps: {M.status_str(st)}")
    value = job_tokens_per_s(W, T, ms)

    # ---- per-kernel durations: the same path called stage by stage with events in between
    align = M.batched_align(T, w.K, w.E, S) if batched else (M.NAIVE_ROWS if naive else w.align)
    U = w.E * S if batched else M.msum_upper(T, w.K, w.E, align)
    ids = torch.empty(T, w.K, dtype=torch.int32, device=dev)
    tw = torch.empty(T, w.K, dtype=torch.float32, device=dev)
    xq = torch.empty(T, w.H, dtype=torch.uint8, device=dev)
    xsf = torch.empty(T, w.H // 128, dtype=torch.uint8, device=dev)
    srt = torch.empty(U, dtype=torch.int32, device=dev)
    eids = torch.empty(U, dtype=torch.int32, device=dev)
    inv = torch.empty(T, w.K, dtype=torch.int32, device=dev)
    msum = torch.empty(1, dtype=torch.int32, device=dev)
    cnt = torch.empty(w.E, dtype=torch.int32, device=dev)
    xp = torch.empty(U, w.H, dtype=torch.uint8, device=dev)
    xpsf = torch.empty(M.act_sf_tiled_bytes(U, w.H // 128, align), dtype=torch.uint8, device=dev)
    hq = torch.empty(U, w.I, dtype=torch.uint8, device=dev)
    hsf = torch.empty(M.act_sf_tiled_bytes(U, w.I // 128, align), dtype=torch.uint8, device=dev)
    y = torch.empty(U, w.H, dtype=torch.bfloat16, device=dev)
    if i8:
        xq8 = torch.empty(T, w.H, dtype=torch.int8, device=dev)
        blk = w.fmt == "int8b"      # one scale per 256-column group instead of one per row
        xs8 = torch.empty((T, w.H // 256) if blk else (T,), dtype=torch.float32, device=dev)
        hq8 = torch.empty(U, w.I, dtype=torch.int8, device=dev)
        hs8 = torch.empty((U, w.I // 256) if blk else (U,), dtype=torch.float32, device=dev)
    # MXFP4: the expert FFN is one launch (moe_grouped_ffn), timed as one stage; NVFP4: L1 and L2 apart
    # (BatchedExperts: the whole FFN through moe_grouped_ffn_batched, whose row-map kernel from the
    # per-expert counts is counted in the stage; moe_forward_batched takes the row map from the permute)
    # (tiny-batch layout: routing and layout are one stage, moe_route_naive)
    # (INT8: the routing stage includes the per-token quantisation, L1 the row gather and the h requant,
    # L2 the conversion of h to fp16 rows)
    fused = w.fmt == "mxfp4" or batched
    token_order = (args.l1_input == "token" or (args.l1_input == "auto" and w.fmt == "nvfp4")) and not (
        batched or naive or i8)
    stages = ["route", "permute", "ffn", "reduce"] if fused else ["route", "permute", "l1", "l2", "reduce"]
    if naive:
        stages.remove("permute")
    sev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(stages) + 1)] for _ in range(K)]
    barrier()
    for i in range(K):
        flush.fill_(i & 0xFF)
        # a GPU-side spin keeps the host ahead: every stage is enqueued before the GPU reaches it, so
        # the events around a stage measure its kernels, not the host's launch latency
        torch.cuda._sleep(4 * SPIN_CYCLES)
        e = sev[i]
        j = 0
        e[j].record()
        if naive:
            M.route_naive(hidden, w_gate, gate_bias, e_bias, w.K, w.score_fn, w.renormalize, ids, tw, srt, eids, inv,
                          msum, xp, xpsf, ws)
        elif i8:
            M.route(hidden, w_gate, gate_bias, e_bias, w.K, w.score_fn, w.renormalize, ids, tw, ws)
            M.act_quant_i8(hidden, xq8, xs8)
        else:
            M.route(hidden, w_gate, gate_bias, e_bias, w.K, w.score_fn, w.renormalize, ids, tw, ws, x_q=xq, x_sf=xsf)
        j += 1
        e[j].record()
        if naive:
            pass
        elif i8:
            M.permute(ids, w.E, w.align, srt, eids, inv, msum, ws, expert_counts=cnt)
        elif batched:
            M.permute_batched(ids, w.E, S, srt, eids, inv, msum, ws, expert_num_tokens=cnt, x_q=xq, x_sf=xsf,
                              x_perm=xp, x_perm_sf=xpsf)
        elif token_order:
            M.permute(ids, w.E, w.align, srt, eids, inv, msum, ws, expert_counts=cnt)
        else:
            M.permute(ids, w.E, w.align, srt, eids, inv, msum, ws, expert_counts=cnt, x_q=xq, x_sf=xsf, x_perm=xp,
                      x_perm_sf=xpsf)
        if not naive:
            j += 1
            e[j].record()
        if i8:
            M.grouped_gemm_l1_swiglu_i8(xq8, xs8, srt, eids, msum, T, w.K, w.H, w.I, w.E, align, w13, hq8, hs8, ws)
            j += 1
            e[j].record()
            M.grouped_gemm_l2_i8(hq8, hs8, eids, msum, T, w.K, w.H, w.I, w.E, align, w2, y, ws)
        elif batched:
            M.grouped_ffn_batched(xp, xpsf, cnt, T, w.K, w.H, w.I, w.E, S, w13, w2, hq, hsf, y, ws)
        elif fused and token_order:
            M.grouped_ffn(xq, xsf, eids, msum, T, w.K, w.H, w.I, w.E, align, w13, w2, hq, hsf, y, ws,
                          sorted_token_ids=srt)
        elif fused:
            M.grouped_ffn(xp, xpsf, eids, msum, T, w.K, w.H, w.I, w.E, align, w13, w2, hq, hsf, y, ws)
        else:
            if token_order:
                M.grouped_gemm_l1_swiglu(xq, xsf, eids, msum, T, w.K, w.H, w.I, w.E, align, w13, hq, hsf, ws,
                                         sorted_token_ids=srt)
            else:
                M.grouped_gemm_l1_swiglu(xp, xpsf, eids, msum, T, w.K, w.H, w.I, w.E, align, w13, hq, hsf, ws)
            j += 1
            e[j].record()
            M.grouped_gemm_l2(hq, hsf, eids, msum, T, w.K, w.H, w.I, w.E, align, w2, y, ws)
        j += 1
        e[j].record()
        M.unpermute_reduce(y, inv, tw, out)
        j += 1
        e[j].record()
    barrier()
    stage_ms = {s: statistics.mean(sev[i][j].elapsed_time(sev[i][j + 1]) for i in range(K)) for j, s in enumerate(stages)}
    if naive:     # no per-expert counts in this layout: count the distinct experts of the routing
        n_touched = int(torch.unique(ids).numel())
    else:
        n_touched = int((cnt.cpu() > 0).sum().item())
    ab = algorithmic_bytes(w, n_touched)
    hbm, bf16, peak_src = peaks()
    top = "ffn" if fused else max(("l1", "l2"), key=lambda s: stage_ms[s])
    top_key = f"{w.name}:{top}" + (":batched" if batched else "")
    kernel_file = os.path.join(ROOT, "moe_expert_ffn_sqrt_gb300", "csrc",
                               {"mxfp4": "gemm.cu", "nvfp4": "gemm_nv.cu", "int8": "gemm_i8.cu", "int8b": "gemm_i8.cu"}[w.fmt])
    tk = w.T * w.K
    flops = {"l1": 2.0 * tk * 2 * w.I * w.H, "l2": 2.0 * tk * w.I * w.H}
    flops["ffn"] = flops["l1"] + flops["l2"]
    # The binding roofline is the one whose minimum time is longer: the kernel's algorithmic bytes at
    # the measured HBM copy bandwidth, or its useful FLOPs at the tensor peak.  MXFP4 runs FP8 x FP4
    # block-scaled MMAs (FP8 rate: the measured bf16 peak x the nominal 4.5/2.25 ratio); NVFP4 runs
    # bf16 MMAs and INT8 fp16 MMAs (the measured bf16 peak; fp16 runs at the bf16 rate).
    peak_t = bf16 * (2.0 if w.fmt == "mxfp4" else 1.0)
    sec = stage_ms[top] / 1e3
    hbm_frac = ab[top] / sec / 1e9 / hbm
    tensor_frac = flops[top] / sec / 1e12 / peak_t
    common = {"traffic": traffic_record(kernel_file, top_key), "kernel": kernel_name(top, w.fmt),
              "algorithmic_bytes": ab[top], "algorithmic_flops": flops[top], "stage_ms": stage_ms,
              "experts_touched": n_touched, "hbm_frac": hbm_frac, "tensor_frac": tensor_frac,
              "layer_hbm_frac": ab["layer"] / (ms / 1e3) / 1e9 / hbm}
    if ab[top] / hbm / 1e9 >= flops[top] / peak_t / 1e12:
        roofline = {"bound": "hbm", "achieved": ab[top] / sec / 1e9, "peak": hbm, "unit": "GB/s", "frac": hbm_frac,
                    "peak_source": f"{peak_src} HBM copy bandwidth", **common}
    else:
        roofline = {"bound": "tensor", "achieved": flops[top] / sec / 1e12, "peak": peak_t, "unit": "TFLOP/s",
                    "frac": tensor_frac,
                    "peak_source": f"{peak_src} bf16 GEMM" + (" x 2 (FP8 / bf16 nominal ratio)" if w.fmt == "mxfp4" else ""),
                    **common}

    # ---- end to end through the public API with host buffers: H2D input, forward, D2H output
    e2e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    # host cost of issuing one end-to-end step, measured while a GPU-side spin holds the device (so
    # the launch queue never fills and the host never waits): steps outside the timed region
    barrier()
    n_probe = 16
    torch.cuda._sleep(100 * SPIN_CYCLES)
    h0 = time.perf_counter()
    for i in range(n_probe):
        hidden.copy_(hidden_host, non_blocking=True)
        step()
        out_host.copy_(out, non_blocking=True)
    host_us = (time.perf_counter() - h0) * 1e6 / n_probe
    barrier()
    for i in range(K):
        flush.fill_(i & 0xFF)
        e2e_ev[i][0].record()
        hidden.copy_(hidden_host, non_blocking=True)
        step()
        out_host.copy_(out, non_blocking=True)
        e2e_ev[i][1].record()
    barrier()
    e2e_ms = max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in e2e_ev), dev)
    e2e = {"value": job_tokens_per_s(W, T, e2e_ms), "unit": "tokens/s", "h2d_bytes_per_step": T * w.H * 2,
           "d2h_bytes_per_step": T * w.H * 2, "host_issue_us_per_step": host_us}

    cpu = None
    if rank == 0 and W == 1 and cpu_seconds > 0:
        cpu = oracle_tokens_per_s(w, inp, stack, cpu_seconds)
    cfg = workload_config(w)
    cfg["l2"] = "512 MiB buffer written between steps (outside the timed events); touched weights > L2"
    cfg["parallelism"] = f"replicas x{W}"
    cfg["layout"] = (f"BatchedExperts, max_tokens={S}" if batched else
                     "tiny-batch, one 16-row block per (token, expert) pair" if naive else
                     "expert-contiguous, padded to align; the whole layer in one cooperative launch (stage_ms "
                     "from the separate stage calls)" if single else
                     "expert-contiguous, padded to align")
    cfg["routing_weights"] = ("applied in the L1 epilogue, unweighted reduce (stage_ms from the reduce-weighted "
                              "stage calls)" if args.weights_in_l1 else "applied in the reduce")
    cfg["l1_input"] = ("token-order rows read through sorted_token_ids" if w.fmt == "nvfp4" and not batched else
                       "permuted row copy")
    cfg["stage_l1_input"] = "token-order" if token_order else "permuted copy"
    res = dict(value=value, ms=ms, steps=K, warmup=warmup, roofline=roofline, e2e=e2e, cpu=cpu, cfg=cfg,
               clocks=clk, launches=launches_per_forward(w, naive, single) * K,
               dtype={"mxfp4": "fp8xfp4 (fp32 accumulate)",
                      "nvfp4": "bf16 (exact fp8/nvfp4 values, fp32 accumulate)",
                      "int8": "int8xint8 as fp16 (exact codes, fp32 accumulate)",
                      "int8b": "int8xint8 as fp16 (exact codes, fp32 accumulate per 256-deep block)"}[w.fmt])
    del w13, w2, ws, flush, xp, hq, y, hidden, out
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res


def run_ours(args, w, others):
    import torch
    import moe_expert_ffn_sqrt_gb300 as M

    W, rank, local = world()
    if W > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    M.lib()
    head = measure(args, w, args.steps, args.warmup, args.cpu_seconds, dev)
    per_config = {}
    for wo in others:
        r = measure(args, wo, min(args.steps, PER_CONFIG_STEPS.get(wo.name.split("-")[0], 50)),
                    max(3, min(args.warmup, 5)), args.cpu_seconds, dev)
        rf = r["roofline"]
        per_config[wo.name] = {
            "config": r["cfg"]["workload"], "value": r["value"], "unit": "tokens/s", "ms_per_step": r["ms"],
            "steps": r["steps"], "warmup": r["warmup"], "dtype": r["dtype"],
            "roofline": {k: rf[k] for k in ("bound", "achieved", "peak", "unit", "frac", "traffic", "kernel",
                                            "algorithmic_bytes", "algorithmic_flops", "hbm_frac", "tensor_frac",
                                            "layer_hbm_frac", "experts_touched", "peak_source")},
            "stage_ms": rf["stage_ms"], "e2e": r["e2e"], "cpu_baseline": r["cpu"], "gpu_launches": r["launches"],
            "clocks": r["clocks"]}
    line = None
    if rank == 0:
        line = {"metric": "MoE-layer tokens/s", "value": head["value"], "unit": "tokens/s", "n_gpus": W,
                "steps": head["steps"], "warmup": head["warmup"], "ms_per_step": head["ms"], "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": head["dtype"], "data": "synthetic (seeded)",
                "config": head["cfg"], "roofline": head["roofline"], "cpu_baseline": head["cpu"], "e2e": head["e2e"],
                "gpu_launches": head["launches"], "clocks": head["clocks"]}
        if per_config:
            line["per_config"] = per_config
        print(json.dumps(line), flush=True)
    if W > 1:
        torch.distributed.destroy_process_group()
    return line


def main():
    args = parse_args()
    if args.weights_in_l1 and args.layout != "contiguous":
        raise SystemExit("--weights-in-l1 applies to the expert-contiguous layout")
    if args.weights in I8_FMTS and (args.weights_in_l1 or args.layout != "contiguous"):
        raise SystemExit("--weights int8/int8b runs the expert-contiguous layout with the weights applied in the reduce")
    import dataclasses

    def variant(w):
        if args.weights in I8_FMTS:
            w = dataclasses.replace(w, fmt=args.weights, name=f"{w.name}-{args.weights}")
        if args.experts or args.tokens:
            E = args.experts or w.E
            T = args.tokens or w.T
            w = dataclasses.replace(w, E=E, T=T, name=f"{w.name}-T{T}-E{E}")
        return w

    w = variant(synth.WORKLOADS[args.workload or HEADLINE])
    # the default run (no --workload, no variant switch) also measures every other workload
    plain = (args.workload is None and not args.no_per_config and args.weights == "workload" and
             args.layout == "contiguous" and not args.weights_in_l1 and not args.experts and not args.tokens)
    others = [synth.WORKLOADS[n] for n in ("tiny", "batched", "prefill", "skewed")] if plain else []
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w, others)


if __name__ == "__main__":
    main()
