"""Decode throughput of the integer-only decoder on GB300.

Workload (one "step" = one greedy decode step through every row of the hot
path: embedding, 28 layers of NormQuant / QKV GEMM + QK-norm/RoPE/KV write /
attention / o_proj / NormQuant / gate-up + SwiGLU / down, final norm, lm_head,
tie-low argmax): the Qwen3-0.6B-shaped integer model, batch 1, 64-token seeded
prompt, greedy decode (the pages' demo workload, with seeded synthetic weights
and prompt ids). Weights (596 MB) exceed the 129 MB L2, so every step streams
them from HBM; no L2 flush is needed.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl detint|reference]
Prints one JSON line (rank 0). --impl reference times the CPU oracle (the
reference arm of this method: the plain integer C program) on the same
workload on the host cores.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode tok/s at B=1/8 (Qwen3-0.6B shape), bit-exact; int8 GEMM TOPS, HBM GB/s"
SHAPE = "qwen3-0.6b"
PROMPT_LEN = 64
SEED = 0


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.p = None

    def __enter__(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                       "--format=csv,noheader,nounits", "-lms", "100"],
                                      stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.p = None
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.p:
            self.p.terminate()
            try:
                self.out, _ = self.p.communicate(timeout=5)
            except Exception:
                self.p.kill()

    def summary(self):
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 7:
                continue
            try:
                sm.append(float(f[0]))
                mx = max(mx, float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx or None,
                "reasons": sorted(reasons), "samples": len(sm)}


def max_over_ranks(ms, dist, device):
    """The slowest rank's time: replicas run independently, so the job's
    throughput is every rank's units over this time (no data exchange)."""
    import torch
    if dist is None:
        return ms
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def run_reference(args):
    """The CPU oracle on the same workload: one greedy decode step per unit."""
    ws, rank, _ = _dist()
    if rank != 0:
        return
    import oracle
    import synth
    path = synth.ensure_artifact(SHAPE, SEED)
    m = oracle.Model(path)
    prompt = synth.prompt_ids(SEED, 0, PROMPT_LEN, m.vocab)
    s = m.new_seq(PROMPT_LEN + args.warmup + args.steps + 2)
    tok, _ = s.feed(prompt)
    for _ in range(args.warmup):
        tok, _ = s.feed([tok])
    t0 = time.perf_counter()
    for _ in range(args.steps):
        tok, _ = s.feed([tok])
    dt = time.perf_counter() - t0
    v = args.steps / dt
    cores = oracle.max_threads()
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tok/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int8/int32",
            "data": "synthetic",
            "config": {"workload": "qwen3-0.6b-shape integer decode, B=1, 64-token seeded prompt",
                       "global_batch": 1, "seq_len": PROMPT_LEN, "parallelism": "replicas"},
            "cpu_baseline": {"value": v, "unit": "tok/s", "cores": cores, "kind": "oracle",
                             "sample": f"{args.steps} decode steps after a {PROMPT_LEN}-token "
                                       f"prefill and {args.warmup} warm-up steps"},
            "e2e": {"value": v, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def cpu_baseline(seconds: float = 12.0):
    """Bounded sample of the oracle on the bench workload (B=1 decode)."""
    import oracle
    import synth
    path = synth.ensure_artifact(SHAPE, SEED)
    m = oracle.Model(path)
    prompt = synth.prompt_ids(SEED, 0, PROMPT_LEN, m.vocab)
    s = m.new_seq(PROMPT_LEN + 4096)
    tok, _ = s.feed(prompt)
    n = 0
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < seconds:
        tok, _ = s.feed([tok])
        n += 1
    dt = time.perf_counter() - t0
    cores = oracle.max_threads()
    # the same workload on one core: a fresh sequence, ~seconds/3 of steps
    oracle.set_threads(1)
    try:
        s1 = m.new_seq(PROMPT_LEN + 4096)
        tok1, _ = s1.feed(prompt)
        n1 = 0
        t1 = time.perf_counter()
        while time.perf_counter() - t1 < seconds / 3:
            tok1, _ = s1.feed([tok1])
            n1 += 1
        dt1 = time.perf_counter() - t1
    finally:
        oracle.set_threads(cores)
    return {"value": n / dt, "unit": "tok/s", "cores": cores, "kind": "oracle",
            "sample": f"{n} B=1 decode steps after the {PROMPT_LEN}-token prefill "
                      f"(~{seconds:.0f} s of CPU work)",
            "single_core": {"value": n1 / dt1, "unit": "tok/s", "cores": 1,
                            "sample": f"{n1} B=1 decode steps after the {PROMPT_LEN}-token prefill "
                                      f"(~{seconds / 3:.0f} s)"}}


# DRAM bytes (read + write) of one lm_head GEMV launch at M=1, from an ncu
# capture of dram__bytes_read.sum + dram__bytes_write.sum on the current kernel
LMHEAD_DRAM_BYTES = 158621952


def int8_peak(pkg, dev, iters=4096, reps=5):
    """Integer-pipe peak of this GPU in TOPS, measured now: the library's loop
    of independent mma.sync m16n8k32 s8 operations (kind 0) and of dp4a
    (kind 1) on register operands, 4 CTAs of 256 threads per SM, best of
    `reps` CUDA-event timings. The tcgen05 tensor cores have no integer kind
    on sm_103a, so this is the rate an int8 GEMM can reach here."""
    import torch
    nsm = torch.cuda.get_device_properties(dev).multi_processor_count
    blocks = 4 * nsm
    sink = torch.empty(blocks * 256 * 8, dtype=torch.int32, device=dev)
    out = {}
    for kind, name in ((0, "mma_s8"), (1, "dp4a")):
        best = None
        for r in range(reps + 1):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            ops = pkg.detint_int8_peak_loop(kind, blocks, iters, sink)
            e1.record()
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1)
            if r and (best is None or ms < best):
                best = ms
        out[name] = ops / (best / 1e3) / 1e12
    return out


def run_gemm_w16(args):
    """Exact int8 x int16 GEMM (two int8 weight limbs) over the Llama-3.2-1B
    projection shapes; TOPS counts 2 M N K for the int16 product."""
    import torch
    from deterministic_integer_only_gb300 import build
    build.build()
    import deterministic_integer_only_gb300 as pkg
    res = []
    s = torch.cuda.Stream()
    for M in (64, 512, 4096):
        for N, K in ((2048, 2048), (3072, 2048), (16384, 2048), (2048, 8192)):
            a = torch.randint(-128, 128, (M, K), dtype=torch.int8, device="cuda")
            w = torch.randint(-32768, 32768, (N, K), dtype=torch.int16, device="cuda")
            hi, lo = pkg.detint_split_w16(w)
            c = torch.empty((M, N), dtype=torch.int64, device="cuda")
            ms = _graph_time(lambda: pkg.detint_gemm_w16(a, hi, lo, c, stream=s), s, 20)
            res.append({"M": M, "N": N, "K": K, "us": ms * 1e3, "tops": 2.0 * M * N * K / (ms / 1e3) / 1e12})
            del a, w, hi, lo, c
    print(json.dumps({"metric": "exact int8 x int16 GEMM sweep (two int8 weight limbs, Llama-3.2-1B shapes)",
                      "unit": "TOPS", "mma_s8_peak_tops": int8_peak(pkg, torch.device("cuda"))["mma_s8"],
                      "sweep": res}), flush=True)


def run_sample(args):
    """detint_sample on seeded 151936-wide logits rows (±8 in logit units):
    microseconds per call for 1, 8 and 32 rows, full distribution and
    top-k 50 / top-p 0.92."""
    import torch
    from deterministic_integer_only_gb300 import build
    build.build()
    import deterministic_integer_only_gb300 as pkg
    rng = np.random.default_rng(SEED)
    res = []
    for rows in (1, 8, 32):
        x = torch.tensor(rng.integers(-(8 << 16), 8 << 16, (rows, 151936)).astype(np.int32), device="cuda")
        for prm in ({}, {"top_k": 50, "top_p": 60000}):
            for _ in range(max(3, args.warmup)):
                pkg.detint_sample(x, prm)
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            n = max(20, args.steps)
            e0.record()
            for _ in range(n):
                pkg.detint_sample(x, prm)
            e1.record()
            torch.cuda.synchronize()
            res.append({"rows": rows, "params": prm, "us": e0.elapsed_time(e1) / n * 1e3})
    print(json.dumps({"metric": "integer sampling latency (151936-wide rows)", "unit": "us",
                      "results": res}), flush=True)


def run_llama_b32(args):
    """Llama-3.2-1B-shaped decode at batch 32 with 1024-token seeded contexts:
    32 x 1024 prefilled, then K timed decode steps (CUDA-graph replays)."""
    import torch
    import synth
    from deterministic_integer_only_gb300 import build
    build.build()
    import deterministic_integer_only_gb300 as pkg
    B, C = 32, 1024
    K, W = args.steps, args.warmup
    path = synth.ensure_artifact("llama-1b", SEED)
    model = pkg.Model(path, max_batch=B, max_ctx=((C + W + K + 64) // 64) * 64)
    dev = torch.device("cuda")
    prompts = [synth.prompt_ids(9, i, C, model.vocab) for i in range(B)]
    flat = torch.tensor(np.concatenate(prompts), dtype=torch.int32, device=dev)
    cu = np.arange(B + 1) * C
    tok = torch.empty(B, dtype=torch.int32, device=dev)
    s = model.stream
    ids = list(range(B))
    with torch.cuda.stream(s):
        model.prefill(ids, flat, cu, None, tok)
        for _ in range(W):
            model.decode_step(ids, tok, None, tok)
    s.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        e0.record(s)
        for _ in range(K):
            model.decode_step(ids, tok, None, tok)
        e1.record(s)
    s.synchronize()
    ms = e0.elapsed_time(e1) / K
    L, H, nq, nkv, d, F, V = (model.n_layers, model.hidden, model.n_q, model.n_kv, model.head_dim,
                              model.ffn, model.vocab)
    wbytes = L * ((nq + 2 * nkv) * d * H + H * nq * d + 2 * F * H + H * F) + V * H
    kv = L * nkv * d * 2 * (C + W + K / 2) * B
    peak, peak_kind = _peaks()
    step_bytes = wbytes + kv + 4 * B * V
    line = {"metric": "decode tok/s (Llama-3.2-1B shape, B=32, 1024-token contexts)",
            "value": B / (ms / 1e3), "unit": "tok/s", "ms_per_step": ms, "steps": K, "warmup": W,
            "step_roofline": {"bytes": step_bytes, "achieved_gbs": step_bytes / (ms / 1e3) / 1e9,
                              "frac": step_bytes / (ms / 1e3) / 1e9 / peak, "peak_kind": peak_kind},
            "dtype": "int8/int32", "data": "synthetic"}
    print(json.dumps(line), flush=True)
    model.close()


def prefill_rate(pkg, B, L, steps, warmup, peak_tops):
    """Prefill of B sequences x L seeded tokens (Qwen3-0.6B shape) in one
    detint_prefill call: median ms, tok/s, GEMM TOPS and its fraction of the
    measured int8 peak (the GEMMs' 2MNK; the attention's causal QK^T and two
    E.V limbs are counted separately)."""
    import torch
    import synth
    path = synth.ensure_artifact(SHAPE, SEED)
    model = pkg.Model(path, max_batch=B, max_ctx=L)
    dev = torch.device("cuda")
    prompts = [synth.prompt_ids(SEED, 200 + i, L, model.vocab) for i in range(B)]
    flat = torch.tensor(np.concatenate(prompts), dtype=torch.int32, device=dev)
    cu = np.arange(B + 1) * L
    tok = torch.empty(B, dtype=torch.int32, device=dev)
    s = model.stream
    times = []
    for it in range(warmup + steps):
        for sid in range(B):
            model.reset_seq(sid)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            e0.record(s)
            model.prefill(list(range(B)), flat, cu, None, tok)
            e1.record(s)
        s.synchronize()
        if it >= warmup:
            times.append(e0.elapsed_time(e1))
    ms = float(np.median(times))
    H, F, nq, nkv, d, Lyr = model.hidden, model.ffn, model.n_q, model.n_kv, model.head_dim, model.n_layers
    gemm_ops = 2.0 * B * L * Lyr * ((nq + 2 * nkv) * d * H + H * nq * d + 2 * F * H + H * F)
    attn_ops = 2.0 * B * Lyr * nq * d * (L * (L + 1) / 2) * 3    # QK^T + two E.V limbs, causal
    model.close()
    return {"metric": f"prefill tok/s (Qwen3-0.6B shape, {B} x {L})", "value": B * L / (ms / 1e3),
            "unit": "tok/s", "ms": ms, "steps": steps, "warmup": warmup,
            "gemm_ops_T": gemm_ops / 1e12, "attn_ops_T": attn_ops / 1e12,
            "ops_tops_overall": (gemm_ops + attn_ops) / (ms / 1e3) / 1e12,
            "int8_peak_tops": peak_tops,
            "overall_frac": (gemm_ops + attn_ops) / (ms / 1e3) / 1e12 / peak_tops,
            "note": "overall: GEMM plus attention integer operations over the whole prefill time"}


def run_prefill(args):
    """Prefill throughput: 4 sequences x 4096 seeded tokens on the Qwen3-0.6B
    shape in one detint_prefill call (last-position logits per sequence)."""
    import torch
    from deterministic_integer_only_gb300 import build
    build.build()
    import deterministic_integer_only_gb300 as pkg
    pk = int8_peak(pkg, torch.device("cuda"))["mma_s8"]
    line = prefill_rate(pkg, args.prefill_seqs, args.prefill_len, args.steps, args.warmup, pk)
    line.update({"dtype": "int8/int32", "data": "synthetic"})
    print(json.dumps(line), flush=True)


def _graph_time(fn, stream, n):
    """Milliseconds per call of fn (a CUDA launch on `stream`), timed as one
    CUDA-graph replay of n captured calls so host overhead cannot leak in."""
    import torch
    with torch.cuda.stream(stream):
        for _ in range(3):
            fn()
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(n):
            fn()
    with torch.cuda.stream(stream):
        g.replay()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        g.replay()
        e1.record(stream)
    stream.synchronize()
    return e0.elapsed_time(e1) / n


def run_lmhead(args):
    """One exact GEMM shape launched repeatedly (default: the dominant decode
    kernel, the streaming GEMV at the lm_head shape 151936 x 1024 with
    M = --batch), for profiler captures."""
    import torch
    from deterministic_integer_only_gb300 import build
    build.build()
    import deterministic_integer_only_gb300 as pkg
    dev = torch.device("cuda")
    M, N, K = (args.batch, 151936, 1024) if not args.shape else [int(v) for v in args.shape.split(",")]
    W = torch.randint(-127, 128, (N, K), dtype=torch.int8, device=dev)
    X = torch.randint(-127, 128, (M, K), dtype=torch.int8, device=dev)
    C = torch.empty((M, N), dtype=torch.int32, device=dev)
    for _ in range(args.warmup + args.steps):
        pkg.detint_gemm_i8(X, W, C)
    torch.cuda.synchronize()
    print(json.dumps({"workload": "lmhead", "launches": args.warmup + args.steps}), flush=True)


def run_int8_peak(args):
    """The integer-pipe peak loops (mma.sync m16n8k32 s8 and dp4a) and, as a
    library reference, torch._int_mm (cuBLASLt) on 8192^3."""
    import torch
    from deterministic_integer_only_gb300 import build
    build.build()
    import deterministic_integer_only_gb300 as pkg
    dev = torch.device("cuda")
    pk = int8_peak(pkg, dev)
    lib_tops = None
    try:
        a = torch.randint(-127, 128, (8192, 8192), dtype=torch.int8, device=dev)
        b = torch.randint(-127, 128, (8192, 8192), dtype=torch.int8, device=dev)
        for _ in range(2):
            torch._int_mm(a, b)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(5):
            torch._int_mm(a, b)
        e1.record()
        torch.cuda.synchronize()
        lib_tops = 2 * 8192 ** 3 * 5 / (e0.elapsed_time(e1) / 1e3) / 1e12
    except (RuntimeError, AttributeError) as e:
        lib_tops = f"unavailable: {type(e).__name__}"
    print(json.dumps({"metric": "int8 integer-pipe peak", "unit": "TOPS", "mma_s8": pk["mma_s8"],
                      "dp4a": pk["dp4a"], "torch_int_mm_8192": lib_tops,
                      "loop": "4 CTAs x 256 threads per SM, 8 independent operations per warp "
                              "(mma) or thread (dp4a) per round, 4096 rounds, best of 5"}), flush=True)


def run_oracle_configs(args):
    """The CPU oracle timed on the other configured workloads, on bounded
    samples (one core and all cores): config 3 (batch 8: row 0 and two
    co-prompt rows, each row independent by construction), config 4 (the
    2048-token prompt fed token by token; a split prefill is the same work
    for the oracle) and config 5 (two of the 32 Llama-shaped sequences at
    1024-token contexts)."""
    import oracle
    import synth
    cores = oracle.max_threads()
    res = []

    def timed(shape, prompt, steps, label, threads, budget):
        oracle.set_threads(threads)
        m = oracle.Model(synth.ensure_artifact(shape, SEED))
        s = m.new_seq(len(prompt) + steps + 1)
        t0 = time.perf_counter()
        tok, _ = s.feed(prompt)
        fed = len(prompt)
        n = 0
        while n < steps and time.perf_counter() - t0 < budget:
            tok, _ = s.feed([tok])
            n += 1
        dt = time.perf_counter() - t0
        res.append({"sample": label, "threads": threads, "prompt_tokens": fed, "decode_steps": n,
                    "seconds": dt, "tok_per_s": (fed + n) / dt})

    q = synth.prompt_ids(SEED, 0, PROMPT_LEN, 151936)
    lens = synth.coprompt_lengths(SEED, 7)
    p4 = synth.prompt_ids(SEED, 7, 2048, 151936)
    for threads, budget, cut in ((cores, 8.0, 512), (1, 2.0, 64)):
        # the long prompts cut to `cut` tokens (256 on all cores for the
        # Llama-shaped contexts) so the run stays within a few minutes
        def c(p, cap=None):
            k = cut if cap is None or threads == 1 else cap
            return p[:k]
        timed(SHAPE, q, 64, f"config 3 row 0 ({len(c(q))}-token prompt)", threads, budget)
        for i in (0, 3):
            pi = c(synth.prompt_ids(SEED, 100 + i, int(lens[i]), 151936))
            timed(SHAPE, pi, 64, f"config 3 row {i + 1} ({len(pi)} tokens of its co-prompt)", threads, budget)
        timed(SHAPE, c(p4), 8, f"config 4 ({len(c(p4))} tokens of the 2048-token prompt, token by token)",
              threads, budget)
        for b in (0, 17):
            pb = c(synth.prompt_ids(9, b, 1024, 128256), 256)
            timed("llama-1b", pb, 8, f"config 5 sequence {b} ({len(pb)}-token context)", threads, budget)
    oracle.set_threads(cores)
    print(json.dumps({"metric": "CPU oracle on configs 3-5 (bounded samples)", "unit": "tok/s",
                      "cores": cores, "samples": res}), flush=True)


def run_all_kernels(args):
    """Every kernel of the library at least once, on small shapes (for
    per-kernel counter captures such as the floating-point instruction
    classes): tiny-model prefill on the tensor-core attention and on the
    per-token one, decode through the fused step (staged and global K/V
    reads), the row kernels, the one-launch step and a batch of 12 (tiled
    GEMMs with split K), the exact mode (limb split, limb GEMM, 128-bit
    epilogue), integer sampling, the allocation-free argmax, the raw int8
    GEMMs and the peak loops."""
    import torch
    import synth
    from deterministic_integer_only_gb300 import build
    build.build()
    import deterministic_integer_only_gb300 as pkg
    dev = torch.device("cuda")
    launched = []
    for wide in (False, True):
        path = synth.ensure_artifact("tiny", SEED, wide=wide)
        for mode in ("fused", "rows", "one-launch", "tc-off", "global-attn"):
            if wide and mode != "fused":
                continue
            m = pkg.Model(path, max_batch=12, max_ctx=128)
            if mode == "rows":
                m.set_fused_decode(False)
            if mode == "one-launch":
                m.set_persistent(True)
            if mode == "tc-off":
                m.set_tc_prefill(False)
            if mode == "global-attn":
                m.set_staged_decode(False)
            prompts = [synth.prompt_ids(SEED, i, 12 + 5 * i, m.vocab) for i in range(2)]
            m.generate(prompts, 3, keep_logits=False)
            launched.append(f"{'wide ' if wide else ''}{mode}")
            m.close()
    m = pkg.Model(synth.ensure_artifact("tiny", SEED), max_batch=12, max_ctx=128)
    m.generate([synth.prompt_ids(SEED, 20 + i, 9 + i, m.vocab) for i in range(12)], 3, keep_logits=False)
    launched.append("batch 12")
    m.close()
    lg = torch.randint(-(1 << 20), 1 << 20, (2, 4096), dtype=torch.int32, device=dev)
    pkg.detint_sample(lg, {"seed": 1, "inv_temp": 65536, "top_k": 50, "top_p": 60000})
    pkg.detint_argmax_noalloc(lg, torch.empty(2, dtype=torch.int32, device=dev))
    for M in (4, 96):
        A = torch.randint(-127, 128, (M, 256), dtype=torch.int8, device=dev)
        W = torch.randint(-127, 128, (512, 256), dtype=torch.int8, device=dev)
        pkg.detint_gemm_i8(A, W, torch.empty((M, 512), dtype=torch.int32, device=dev))
    # a long weight stream (the lm_head-like variant with two CTAs per SM)
    A = torch.randint(-127, 128, (1, 1024), dtype=torch.int8, device=dev)
    W = torch.randint(-127, 128, (32768, 1024), dtype=torch.int8, device=dev)
    pkg.detint_gemm_i8(A, W, torch.empty((1, 32768), dtype=torch.int32, device=dev))
    W16 = torch.randint(-32767, 32768, (512, 256), dtype=torch.int16, device=dev)
    hi, lo = pkg.detint_split_w16(W16)
    pkg.detint_gemm_w16(torch.randint(-127, 128, (64, 256), dtype=torch.int8, device=dev), hi, lo)
    sink = torch.empty(256 * 8, dtype=torch.int32, device=dev)
    for kind in (0, 1):
        pkg.detint_int8_peak_loop(kind, 1, 16, sink)
    torch.cuda.synchronize()
    print(json.dumps({"workload": "kernels", "model_runs": launched}), flush=True)


def run_gemm_sweep(args):
    """Exact int8 GEMM (detint_gemm_i8) over M x (N, K) of the Llama-3.2-1B
    projections: TOPS = 2MNK/t and bytes = MK + NK + 4MN per launch."""
    import torch
    from deterministic_integer_only_gb300 import build
    build.build()
    import deterministic_integer_only_gb300 as pkg
    peak_gbs, _ = _peaks()
    dev = torch.device("cuda")
    pk = int8_peak(pkg, dev)["mma_s8"]
    s = torch.cuda.Stream()
    rows = []
    for (N, K) in [(2048, 2048), (512, 2048), (3072, 2048), (16384, 2048), (2048, 8192), (128256, 2048)]:
        W = torch.randint(-127, 128, (N, K), dtype=torch.int8, device=dev)
        for M in [1, 8, 64, 512, 4096]:
            A = torch.randint(-127, 128, (M, K), dtype=torch.int8, device=dev)
            C = torch.empty((M, N), dtype=torch.int32, device=dev)
            n = max(3, min(50, int(2e9 / max(1, M * N * K))))
            t = _graph_time(lambda: pkg.detint_gemm_i8(A, W, C, stream=s), s, n) / 1e3
            ops = 2.0 * M * N * K
            byt = M * K + N * K + 4 * M * N
            rows.append({"M": M, "N": N, "K": K, "us": t * 1e6, "tops": ops / t / 1e12,
                         "int8_frac": ops / t / 1e12 / pk,
                         "gbs": byt / t / 1e9, "hbm_frac": byt / t / 1e9 / peak_gbs})
            del A, C
        del W
    print(json.dumps({"metric": "int8 GEMM sweep (Llama-3.2-1B shapes)", "unit": "TOPS",
                      "mma_s8_peak_tops": pk, "hbm_peak_gbs": peak_gbs,
                      "sweep": rows}), flush=True)


def _decode_rate(pkg, path, B, K, W, dev, dist, ws, one_launch=False):
    """(tok/s over all ranks, ms per step) of K graph-replayed decode steps
    of B sequences, inputs resident on the device."""
    import torch
    import synth
    max_ctx = PROMPT_LEN + W + 2 * K + 280
    model = pkg.Model(path, max_batch=B, max_ctx=((max_ctx + 63) // 64) * 64)
    if one_launch:
        model.set_persistent(True)
    V = model.vocab
    prompts = [synth.prompt_ids(SEED, 0, PROMPT_LEN, V)]
    prompts += [synth.prompt_ids(SEED, 100 + i, int(n), V)
                for i, n in enumerate(synth.coprompt_lengths(SEED, B - 1))]
    s = model.stream
    seq_ids = list(range(B))
    cu = np.zeros(B + 1, np.int64)
    cu[1:] = np.cumsum([len(p) for p in prompts])
    flat = torch.tensor(np.concatenate(prompts), dtype=torch.int32, device=dev)
    tok = torch.empty(B, dtype=torch.int32, device=dev)
    with torch.cuda.stream(s):
        model.prefill(seq_ids, flat, cu, None, tok)
        for _ in range(W):
            model.decode_step(seq_ids, tok, None, tok)
    s.synchronize()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        e0.record(s)
        for _ in range(K):
            model.decode_step(seq_ids, tok, None, tok)
        e1.record(s)
    s.synchronize()
    ms = e0.elapsed_time(e1)
    if dist:
        ms = max_over_ranks(ms, dist, dev)
    model.close()
    return B * K * ws / (ms / 1e3), ms / K


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="detint", choices=["detint", "reference"])
    ap.add_argument("--batch", type=int, default=1)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only-steps", action="store_true",
                    help="run the prefill, warm-up and timed decode steps only, print their time "
                         "(for launch-list captures of the decode step)")
    ap.add_argument("--one-launch", action="store_true",
                    help="decode through the one-launch step (cooperative, tagged rows)")
    ap.add_argument("--no-companion", dest="companion", action="store_false",
                    help="skip the B=8 companion measurement of the decode line")
    ap.add_argument("--shape", default=None, help="M,N,K for --workload lmhead (default 1,151936,1024 "
                    "with M = --batch)")
    ap.add_argument("--prefill-seqs", type=int, default=4, help="prefill workload: sequences")
    ap.add_argument("--prefill-len", type=int, default=4096, help="prefill workload: tokens each")
    ap.add_argument("--workload", default="decode",
                    choices=["decode", "prefill", "gemm", "lmhead", "llama-b32", "sample", "gemm-w16",
                             "int8-peak", "oracle-configs", "kernels"],
                    help="decode (the headline line), prefill (4 x 4096 prompt throughput) or "
                         "gemm (exact int8 GEMM sweep over the Llama-3.2-1B projection shapes)")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    if args.workload == "prefill":
        return run_prefill(args)
    if args.workload == "llama-b32":
        return run_llama_b32(args)
    if args.workload == "sample":
        return run_sample(args)
    if args.workload == "gemm-w16":
        return run_gemm_w16(args)
    if args.workload == "gemm":
        return run_gemm_sweep(args)
    if args.workload == "lmhead":
        return run_lmhead(args)
    if args.workload == "int8-peak":
        return run_int8_peak(args)
    if args.workload == "oracle-configs":
        return run_oracle_configs(args)
    if args.workload == "kernels":
        return run_all_kernels(args)

    import torch
    import synth
    from deterministic_integer_only_gb300 import build
    build.build()
    import deterministic_integer_only_gb300 as pkg

    ws, rank, local = _dist()
    torch.cuda.set_device(local)
    dist = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")

    B = args.batch
    K, W = args.steps, args.warmup
    path = synth.ensure_artifact(SHAPE, SEED)
    co_lens = [int(n) for n in synth.coprompt_lengths(SEED, B - 1)]
    max_ctx = max([PROMPT_LEN] + co_lens) + W + 2 * K + 16
    model = pkg.Model(path, max_batch=B, max_ctx=((max_ctx + 63) // 64) * 64)
    V, H = model.vocab, model.hidden
    dev = torch.device("cuda", local)
    prompts = [synth.prompt_ids(SEED, 0, PROMPT_LEN, V)]
    prompts += [synth.prompt_ids(SEED, 100 + i, n, V) for i, n in enumerate(co_lens)]
    s = model.stream
    seq_ids = list(range(B))

    def start():
        cu = np.zeros(B + 1, np.int64)
        cu[1:] = np.cumsum([len(p) for p in prompts])
        flat = torch.tensor(np.concatenate(prompts), dtype=torch.int32, device=dev)
        tok = torch.empty(B, dtype=torch.int32, device=dev)
        with torch.cuda.stream(s):
            model.prefill(seq_ids, flat, cu, None, tok)
            for _ in range(W):
                model.decode_step(seq_ids, tok, None, tok)
        s.synchronize()
        return tok

    if args.one_launch:
        model.set_persistent(True)
    # ---- device-resident timed region: K decode steps, one graph each
    tok = start()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        with torch.cuda.stream(s):
            e0.record(s)
            for _ in range(K):
                model.decode_step(seq_ids, tok, None, tok)
            e1.record(s)
        s.synchronize()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    if dist:
        ms = max_over_ranks(ms, dist, dev)
        dist.barrier()
    value = B * K * ws / (ms / 1e3)
    if args.only_steps:
        if rank == 0:
            print(json.dumps({"workload": f"decode steps, B={B}", "steps": K, "warmup": W,
                              "ms_per_step": ms / K, "tok_s": value}), flush=True)
        model.close()
        return

    # ---- end to end through the public API with host buffers
    for sid in seq_ids:
        model.reset_seq(sid)
    tok = start()
    host_in = torch.empty(B, dtype=torch.int32, pin_memory=True)
    host_out = torch.empty(B, dtype=torch.int32, pin_memory=True)
    host_in.copy_(tok.cpu())
    nxt = torch.empty(B, dtype=torch.int32, device=dev)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    with torch.cuda.stream(s):
        for _ in range(K):
            tok.copy_(host_in, non_blocking=True)
            model.decode_step(seq_ids, tok, None, nxt)
            host_out.copy_(nxt, non_blocking=True)
            s.synchronize()
            host_in.copy_(host_out)
    e2e_s = time.perf_counter() - t0
    e2e = {"value": B * K * ws / e2e_s, "unit": "tok/s", "h2d_bytes_per_step": 4 * B,
           "d2h_bytes_per_step": 4 * B}

    # ---- dominant kernel: the weight-streaming GEMV at the lm_head shape
    peak, peak_kind = _peaks()
    wmat = torch.randint(-127, 128, (V, H), dtype=torch.int8, device=dev)
    xmat = torch.randint(-127, 128, (B, H), dtype=torch.int8, device=dev)
    cmat = torch.empty((B, V), dtype=torch.int32, device=dev)
    # cold-L2 time per launch: each launch follows a 256 MB write that evicts
    # the 129 MB L2 (graph of flush+launch minus graph of flush alone), as it
    # is inside a decode step where 440 MB of other weights pass in between
    flush = torch.empty(256 << 20, dtype=torch.int8, device=dev)

    def _flush():
        flush.fill_(1)

    def _both():
        _flush()
        pkg.detint_gemm_i8(xmat, wmat, cmat, stream=s)

    kms = _graph_time(_both, s, 20) - _graph_time(_flush, s, 20)
    kms_warm = _graph_time(lambda: pkg.detint_gemm_i8(xmat, wmat, cmat, stream=s), s, 50)
    del flush
    kbytes = V * H + B * H + 4 * B * V
    achieved = kbytes / (kms / 1e3) / 1e9
    roofline = {"bound": "hbm", "kernel": "k_sgemv (decode streaming GEMV), lm_head shape 151936x1024, M=%d" % B,
                "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "peak_kind": peak_kind, "traffic": LMHEAD_DRAM_BYTES if B == 1 else None,
                "traffic_source": "dram__bytes_read.sum + dram__bytes_write.sum of one launch "
                                  "from an ncu capture of this kernel at M=1 (LMHEAD_DRAM_BYTES)",
                "bytes_per_launch": kbytes,
                "us_per_launch": kms * 1e3, "us_per_launch_l2_warm": kms_warm * 1e3,
                "timing": "CUDA events around graph replays; L2 evicted before every launch"}
    # whole-step roofline: algorithmic bytes of one decode step
    L, nq, nkv, d, F = model.n_layers, model.n_q, model.n_kv, model.head_dim, model.ffn
    wbytes = L * ((nq + 2 * nkv) * d * H + H * nq * d + 2 * F * H + H * F) + V * H
    ctx_mean = PROMPT_LEN + W + K / 2
    kv = L * nkv * d * 2 * ctx_mean * B
    step_bytes = wbytes + kv + 4 * B * V
    step = {"bytes": step_bytes, "achieved_gbs": step_bytes / (ms / K / 1e3) / 1e9,
            "frac": step_bytes / (ms / K / 1e3) / 1e9 / peak}

    model.close()
    # companion number for the metric's second batch size: the same workload
    # with 8 sequences (row 0 = the prompt above, 7 seeded co-prompts)
    other = None
    if args.companion and B != 8:
        other = _decode_rate(pkg, path, 8, K, W, dev, dist, ws, args.one_launch)
    # companions for the metric's other parts: the measured int8 pipe peak and
    # the prefill of 4 x 4096 tokens against it
    pk = int8_peak(pkg, dev)
    pre = prefill_rate(pkg, 4, 4096, 3, 1, pk["mma_s8"]) if args.companion else None

    if rank == 0:
        cb = None
        if not args.no_cpu_baseline and ws == 1:
            cb = cpu_baseline()
        # kernels per fused decode step: embedding, 5 per layer (QKV, attention,
        # o_proj, gate/up, down; plus 4 row-quantisation kernels per layer from
        # 3 sequences on), lm_head (+ its row kernel), final argmax
        sep = B >= 3
        gpu_launches = K * (1 + L * (9 if sep else 5) + (2 if sep else 1) + 1)
        line = {"metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": ws, "steps": K,
                "warmup": W, "ms_per_step": ms / K, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "int8/int32", "data": "synthetic",
                "config": {"workload": f"qwen3-0.6b-shape integer decode, B={B}, "
                                       f"{PROMPT_LEN}-token seeded prompt, CUDA-graph step",
                           "global_batch": B * ws, "seq_len": PROMPT_LEN, "parallelism": "replicas",
                           "l2": "weights 596 MB > 129 MB L2 every step (no flush needed)"},
                "e2e": e2e, "gpu_launches": gpu_launches, "roofline": roofline,
                "step_roofline": step, "clocks": clk.summary(), "cpu_baseline": cb}
        if other is not None:
            line["batch8"] = {"value": other[0], "unit": "tok/s", "ms_per_step": other[1],
                              "config": "same workload, B=8 (7 seeded co-prompts of 16-256 tokens)"}
        line["int8_peak_tops"] = pk
        if pre is not None:
            line["prefill"] = pre
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
