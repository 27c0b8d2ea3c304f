#!/usr/bin/env python3
"""Benchmark of the gated delta rule hot path on one GB300 (or N replicas).

One step = one chunked forward over the long-context training batch
(B=4, T=32768, Hqk=16, Hv=32, K=V=128, bf16 I/O, fp32 state, chunk 64, q/k L2
norm, mixer-style gates) followed by one decode step over 256 requests (26 of
them padding) on a 512-slot fp32 state cache -- every kernel of the path.

Prints one JSON line.  ``value`` is chunked-forward tokens/s (B*T per step over
the chunked-forward time); the decode half is reported under ``decode``.  Beside
the step, and outside its timed region: the Gated Delta Product (``product``) and
the chunked backward of the same batch (``backward``), the decode step replayed from
a CUDA graph and both halves timed after an L2 flush (under ``decode``), and the
other chunk workloads (``other_configs``).
``--impl reference`` times the fp64 CPU oracle instead (the reference arm).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gdn|reference]

Defaults: 10 warm-up steps, then 50 timed steps; the per-step medians are reported beside the
means (``chunk_ms_median``, ``decode.ms_median``).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

CHUNK_WL = "long_context_bf16"
DECODE_WL = "decode_bf16"
# Algorithmic work per token of the chunked forward (triangles counted once,
# K K^T / Q K^T per query/key head, the O(C^2) solve and elementwise work left
# out): Hqk * 2 C K + Hv * (C K + 2 C V + 6 K V).
C_, K_, V_, HQK_, HV_ = 64, 128, 128, 16, 32
FLOP_PER_TOKEN = HQK_ * 2 * C_ * K_ + HV_ * (C_ * K_ + 2 * C_ * V_ + 6 * K_ * V_)
# Minimum HBM bytes per token of a fully fused pass: q, k, v, o in bf16, g fp32, beta bf16.
BYTES_PER_TOKEN = HQK_ * K_ * 2 * 2 + HV_ * V_ * 2 * 2 + HV_ * 4 + HV_ * 2
STATE_BYTES = K_ * V_ * 4
# Algorithmic work per token of the backward on top of the forward recompute (per value
# head: K dS, Q^T dO', K^T dX', dO S0^T, dX S0^T, U' dS^T (6 K V), T^T dU', P^T dO and the
# two [C][C] products over V (2 C V), the four triangular [C][C] x K products (2 C K); per
# query/key head: Q K^T and K K^T (C K)), in multiply-adds, times 2 for FLOPs.
BWD_FLOP_PER_TOKEN = FLOP_PER_TOKEN + 2 * (HV_ * (6 * K_ * V_ + 2 * C_ * V_ + 2 * C_ * K_) +
                                           HQK_ * C_ * K_)
METRIC = "chunked GDN fwd tokens/s + % tensor peak; decode tokens/s + state HBM GB/s"
WORKLOAD = ("long-context chunked fwd B=4 T=32768 Hqk=16 Hv=32 K=V=128 chunk 64 + decode 256 "
            "requests (26 padding) on 512 slots")


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d["hbm_gbs"], d["bf16_tflops"], "measured"
    return 6800.0, 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled during the timed region."""
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
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
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

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def _code_text(path):
    """A CUDA source with its comments and whitespace removed."""
    txt = open(path).read()
    txt = re.sub(r"/\*.*?\*/", " ", txt, flags=re.S)
    txt = re.sub(r"//[^\n]*", " ", txt)
    return " ".join(txt.split())


def _local_sources(path, seen=None):
    """path and, recursively, every file it includes with #include "..." from its own folder."""
    seen = set() if seen is None else seen
    path = os.path.abspath(path)
    if path in seen or not os.path.exists(path):
        return seen
    seen.add(path)
    for inc in re.findall(r'^\s*#\s*include\s+"([^"]+)"', open(path).read(), flags=re.M):
        _local_sources(os.path.join(os.path.dirname(path), inc), seen)
    return seen


def kernel_code_hash(path):
    """sha256 (16 hex digits) of a CUDA source and the local headers it includes (sorted by
    name), comments and whitespace removed: a comment-only edit keeps the hash, any change to
    the code of the kernel or of a header it includes changes it."""
    h = hashlib.sha256()
    for f in sorted(_local_sources(path), key=os.path.basename):
        h.update(_code_text(f).encode() + b"\0")
    return h.hexdigest()[:16]


def traffic_record():
    """DRAM bytes per launch of the fused chunk kernel from the committed ncu
    summary, if it was taken on the current kernel code (else None)."""
    p = os.path.join(ROOT, "profiles", "chunk_tc_traffic.json")
    src = os.path.join(ROOT, "chunked_gated_delta_gdn_gb300", "csrc", "gdn_chunk_tc.cu")
    if not os.path.exists(p):
        return None
    rec = json.load(open(p))
    if rec.get("kernel_code_sha256_16") != kernel_code_hash(src):
        return None
    return rec.get("dram_bytes_per_full_launch")


def cpu_oracle_sample(inp, tokens, nthreads=0):
    """Run the fp64 oracle on the first `tokens` tokens of sequence 0 (all heads).
    Returns (seconds, threads used)."""
    import oracle
    sl = slice(0, tokens)
    args = [x[0:1, sl] for x in (inp.q, inp.k, inp.v, inp.g, inp.beta)]
    t = time.perf_counter()
    oracle.recurrent(*args, use_qk_l2norm_in_kernel=True, nthreads=nthreads)
    dt = time.perf_counter() - t
    return dt, (nthreads or oracle.max_threads())


def _median_time(fn, reps=3):
    ts = []
    for _ in range(reps):
        t = time.perf_counter()
        fn()
        ts.append(time.perf_counter() - t)
    return statistics.median(ts)


def measure_cpu_baselines(long_inp, dec_inp, sample_tokens=1024, reps=3):
    """The fp64 oracle, as it stands, on every workload at 1 thread and on all host cores
    (median of `reps` runs each), on a bounded sample: the first `sample_tokens` tokens of the
    packed token axis of the 8192-token, varlen and long-context workloads (their sequences cut
    at the sample end), the tiny fp32 case and the decode step whole.  Tokens/s for the chunk
    workloads, real requests/s for decode.  long_inp / dec_inp: the benchmark's own inputs."""
    import oracle
    from chunked_gated_delta_gdn_gb300 import synthetic
    cores = oracle.max_threads()
    out = {"kind": "oracle", "cores": cores, "reps": reps, "statistic": "median"}
    work = [("tiny_fp32", synthetic.workload("tiny_fp32")),
            ("single_seq_bf16", synthetic.workload("single_seq_bf16")),
            ("varlen_prefill_bf16", synthetic.workload("varlen_prefill_bf16")),
            ("long_context_bf16", long_inp)]
    for name, inp in work:
        B, T = inp.q.shape[:2]
        whole = name == "tiny_fp32"
        n_tok = T if whole else min(sample_tokens, T)
        pick = (lambda x: x) if whole else (lambda x: x[0:1, 0:n_tok])
        args = [pick(x) for x in (inp.q, inp.k, inp.v, inp.g, inp.beta)]
        kw = dict(scale=inp.scale, use_qk_l2norm_in_kernel=inp.use_qk_l2norm)
        if inp.cu_seqlens is not None:
            cu = [int(x) for x in inp.cu_seqlens.tolist() if x < n_tok] + [n_tok]
            kw["cu_seqlens"] = np.array(cu)
            if inp.initial_state is not None and inp.state_indices is not None:
                slots = inp.state_indices[:len(cu) - 1].long()
                kw["initial_state"] = inp.initial_state[slots].double().numpy()
        elif inp.initial_state is not None:
            kw["initial_state"] = (inp.initial_state if whole else inp.initial_state[0:1]).double().numpy()
        tokens = n_tok * (B if whole else 1)
        res = {"sample": ("whole workload, %d tokens" if whole else "first %d tokens") % tokens +
                         ", all %d value heads" % inp.v.shape[2]}
        for label, nt in (("tokens_per_s_1thread", 1), ("tokens_per_s_all_cores", 0)):
            res[label] = tokens / _median_time(lambda: oracle.recurrent(*args, nthreads=nt, **kw), reps)
        out[name] = res
    n_real = int((dec_inp.batch_indices >= 0).sum())
    res = {"sample": "the whole step: %d requests (%d real), 512-slot cache" % (dec_inp.q.shape[0], n_real)}
    base = dec_inp.ssm_state.double().numpy()
    for label, nt in (("requests_per_s_1thread", 1), ("requests_per_s_all_cores", 0)):
        ts = []
        for _ in range(reps):
            cache = base.copy()   # the oracle updates the cache in place; copied outside the timing
            t = time.perf_counter()
            oracle.decode(dec_inp.q, dec_inp.k, dec_inp.v, dec_inp.g, dec_inp.beta, cache,
                          dec_inp.batch_indices, nthreads=nt)
            ts.append(time.perf_counter() - t)
        res[label] = n_real / statistics.median(ts)
    out["decode_bf16"] = res
    return out


def measure_product(dev, seed, steps=10, warmup=3):
    """The Gated Delta Product next to the headline: chunked forward on one 8192-token
    sequence with n_h = 2 writes per token and a decode step of 256 requests (26 padding) on
    a 512-slot cache, same head shapes.  CUDA events on the current stream, after warm-up."""
    from chunked_gated_delta_gdn_gb300 import (chunk_gated_delta_product,
                                               gated_delta_product_decode, synthetic)
    n_h, T = 2, 8192
    cin = synthetic.product_inputs(n_h=n_h, B=1, T=T, Hqk=HQK_, Hv=HV_, K=K_, V=V_,
                                   dtype=torch.bfloat16, init="randn", seed=seed)
    d = {k: getattr(cin, k).to(dev) for k in ("q", "k", "v", "g", "beta", "state")}
    o = torch.empty(1, T, HV_, V_, dtype=torch.bfloat16, device=dev)
    fin = torch.empty_like(d["state"])
    ws = torch.empty(_product_ws(T, n_h), dtype=torch.uint8, device=dev)
    din = synthetic.product_decode_inputs(n_h=n_h, n=256, Hqk=HQK_, Hv=HV_, K=K_, V=V_,
                                          dtype=torch.bfloat16, num_slots=512, pad_frac=0.1,
                                          seed=seed + 1)
    dd = {k: getattr(din, k).to(dev) for k in ("q", "k", "v", "g", "beta", "state", "slots")}
    od = torch.empty(256, HV_, V_, dtype=torch.bfloat16, device=dev)
    n_real = int((din.slots >= 0).sum())

    def chunk():
        chunk_gated_delta_product(d["q"], d["k"], d["v"], d["g"], d["beta"],
                                  initial_state=d["state"], output_final_state=True,
                                  use_qk_l2norm_in_kernel=True, out=o, final_state=fin,
                                  workspace=ws)

    def decode():
        gated_delta_product_decode(dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], dd["state"],
                                   dd["slots"], out=od)

    res = {}
    for name, fn in (("chunk", chunk), ("decode", decode)):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        res[name] = e0.elapsed_time(e1) / steps / 1000.0
    return {"workload": "Gated Delta Product, n_h=2 writes per token, Hqk=16 Hv=32 K=V=128 bf16",
            "chunk": {"tokens": T, "ms": res["chunk"] * 1e3, "tokens_per_s": T / res["chunk"],
                      "writes_per_s": T * n_h / res["chunk"]},
            "decode": {"requests": 256, "padding": 256 - n_real, "ms": res["decode"] * 1e3,
                       "requests_per_s": n_real / res["decode"],
                       "state_gbs": n_real * HV_ * STATE_BYTES * 2 / res["decode"] / 1e9}}


def measure_backward(dev, cin, d, seed, steps=5, warmup=3):
    """The chunked backward (gdn_chunk_bwd: dq, dk, dv, dg, dbeta, d_initial_state) on the
    headline batch with seeded upstream gradients d_o ~ N(0, 1) (bf16) and d_final ~ N(0, 1).
    CUDA events on the current stream, after warm-up; the whole call (five launches: chunk
    table, record-mode forward, reverse, grad, clearing of tokens outside every sequence)."""
    from chunked_gated_delta_gdn_gb300 import _lib, chunk_gated_delta_rule_bwd, synthetic
    B, T = cin.q.shape[:2]
    d_o, dfin = synthetic.output_grads(cin, seed=seed)
    d_o, dfin = d_o.to(dev), dfin.to(dev)
    init = torch.zeros(B, HV_, K_, V_, dtype=torch.float32, device=dev)
    need = int(_lib.load().gdn_chunk_bwd_workspace_size(B, T, HQK_, HV_, K_, V_, B,
                                                        _lib.GDN_BF16, _lib.GDN_BF16))
    ws = torch.empty(need, dtype=torch.uint8, device=dev)

    def bwd():
        return chunk_gated_delta_rule_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d_o, dfin,
                                          initial_state=init, use_qk_l2norm_in_kernel=True,
                                          workspace=ws)

    for _ in range(warmup):
        bwd()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        bwd()
    e1.record()
    torch.cuda.synchronize()
    sec = e0.elapsed_time(e1) / steps / 1000.0
    tokens = B * T
    tf = BWD_FLOP_PER_TOKEN * tokens / sec / 1e12
    _, bf16_peak, peak_src = load_peaks()
    # bf16 with K = V = 128 runs every product on the tensor cores: the bound is the bf16
    # tensor peak; the fp32 path would be bound by the CUDA cores' fp32 FMA rate
    return {"workload": "backward of the headline batch (B=%d T=%d Hqk=16 Hv=32 K=V=128 bf16 "
                        "I/O, fp32 accumulation), d_o and d_final_state given" % (B, T),
            "ms": sec * 1e3, "tokens_per_s": tokens / sec, "launches": 5, "steps": steps,
            "workspace_bytes": need,
            "roofline": {"bound": "tensor", "achieved": tf, "peak": bf16_peak, "unit": "TFLOP/s",
                         "frac": tf / bf16_peak, "flop_per_token": BWD_FLOP_PER_TOKEN,
                         "peak_source": peak_src,
                         "scope": "whole backward call (all five launches)"}}


def _median(xs):
    return statistics.median(xs) if xs else None


def measure_extras(dev, chunk, decode, reps=10):
    """The decode step replayed from a CUDA graph, and the chunked forward and the decode step
    timed one call at a time after an L2 flush (a 512 MiB write), median over the calls."""
    res = {}
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        for _ in range(3):
            decode()
    torch.cuda.current_stream(dev).wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        decode()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n = 50
    e0.record()
    for _ in range(n):
        graph.replay()
    e1.record()
    torch.cuda.synchronize()
    res["decode_graph_ms"] = e0.elapsed_time(e1) / n
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    for name, fn, k in (("chunk_ms_l2flush", chunk, reps), ("decode_ms_l2flush", decode, 2 * reps)):
        evs = []
        for _ in range(k):
            flush.fill_(1)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            evs.append((a, b))
        torch.cuda.synchronize()
        res[name] = _median([a.elapsed_time(b) for a, b in evs])
    return res


def measure_configs(dev, bf16_peak, steps=20, warmup=3):
    """Chunked-forward throughput on the other chunk workloads: the tiny fp32 case (B=1
    T=256 Hqk=Hv=2 K=V=64), one 8192-token bf16 sequence, and 32 packed varlen sequences
    (100-4096 tokens) reading and writing a 64-slot state cache."""
    from chunked_gated_delta_gdn_gb300 import chunk_fwd_path, chunk_gated_delta_rule, synthetic
    out = {}
    for name in ("tiny_fp32", "single_seq_bf16", "varlen_prefill_bf16"):
        inp = synthetic.workload(name)
        d = {k: (None if getattr(inp, k) is None else getattr(inp, k).to(dev))
             for k in ("q", "k", "v", "g", "beta", "initial_state", "cu_seqlens", "state_indices")}
        B, T, Hqk, K = inp.q.shape
        Hv, V = inp.v.shape[2:]
        o = torch.empty_like(d["v"])
        fin = None if inp.state_indices is not None else torch.empty_like(d["initial_state"])

        def run():
            chunk_gated_delta_rule(d["q"], d["k"], d["v"], d["g"], d["beta"],
                                   initial_state=d["initial_state"], output_final_state=True,
                                   use_qk_l2norm_in_kernel=True, cu_seqlens=d["cu_seqlens"],
                                   state_indices=d["state_indices"], out=o, final_state=fin)

        for _ in range(warmup):
            run()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            run()
        e1.record()
        torch.cuda.synchronize()
        sec = e0.elapsed_time(e1) / steps / 1000.0
        tokens = B * T
        fpt = Hqk * 2 * C_ * K + Hv * (C_ * K + 2 * C_ * V + 6 * K * V)
        path = chunk_fwd_path(K, V, inp.q.dtype)
        out[name] = {"tokens": tokens, "ms": sec * 1e3, "tokens_per_s": tokens / sec,
                     "tflops": fpt * tokens / sec / 1e12, "flop_per_token": fpt,
                     "tensor_frac": (fpt * tokens / sec / 1e12 / bf16_peak) if path == 1 else None,
                     "path": "tcgen05 fused" if path == 1 else "fp32 CUDA-core"}
    return out


def _product_ws(T, n_h):
    from chunked_gated_delta_gdn_gb300 import _lib
    return int(_lib.load().gdn_product_chunk_fwd_workspace_size(1, T, n_h, HQK_, HV_, K_, V_, 1,
                                                                _lib.GDN_BF16, _lib.GDN_BF16))


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x, world, device):
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def run_reference(args, world, rank):
    """The reference arm: the fp64 CPU oracle on the host cores, as it stands."""
    if rank != 0:
        return 0
    from chunked_gated_delta_gdn_gb300 import synthetic
    tokens = 1024
    inp = synthetic.chunk_inputs(B=1, T=tokens, Hqk=16, Hv=32, K=128, V=128, dtype=torch.bfloat16,
                                 init="none", gates="mixer", seed=1005)
    for _ in range(args.warmup):
        cpu_oracle_sample(inp, tokens)
    times, cores = [], 1
    for _ in range(args.steps):
        dt, cores = cpu_oracle_sample(inp, tokens)
        times.append(dt)
    tot = sum(times)
    val = tokens * len(times) / tot
    line = {
        "impl": "reference", "metric": METRIC, "value": val,
        "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000 * tot / len(times), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "global_batch": 4, "seq_len": 32768,
                   "reference_sample": "%d tokens x 32 value heads per step (chunked-forward "
                                       "half only; bf16 inputs read as f64)" % tokens},
        "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": "first %d tokens of sequence 0, all 32 heads, per step" % tokens},
        "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["gdn", "reference"], default="gdn")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--batch", type=int, default=None,
                    help="override B of the chunked workload (profiling runs on a smaller case)")
    ap.add_argument("--seq-len", type=int, default=None,
                    help="override T of the chunked workload (profiling runs on a smaller case)")
    ap.add_argument("--no-product", action="store_true",
                    help="skip the Gated Delta Product measurement reported beside the headline")
    ap.add_argument("--only", choices=["chunk", "decode", "backward"], default=None,
                    help="time one half of the step, or only the backward (profiling); the "
                         "JSON line keeps its keys, the parts not timed are null")
    ap.add_argument("--no-backward", action="store_true",
                    help="skip the chunked-backward measurement reported beside the headline")
    ap.add_argument("--backward-steps", type=int, default=5)
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the CUDA-graph decode, the L2-flushed timings and the other chunk "
                         "workloads reported beside the headline")
    args = ap.parse_args()
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    if args.impl == "reference":
        return run_reference(args, world, rank)
    if args.warmup < 3:
        args.warmup = 3

    from chunked_gated_delta_gdn_gb300 import (chunk_gated_delta_rule, chunk_fwd_path,
                                               chunk_workspace_size, gated_delta_decode, synthetic)
    from chunked_gated_delta_gdn_gb300 import _lib
    _lib.load()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    hbm_peak, bf16_peak, peak_src = load_peaks()

    # Inputs: each rank its own independent batch (weak scaling, no collective).
    over = {} if args.batch is None else {"B": args.batch}
    if args.seq_len is not None:
        over["T"] = args.seq_len
    cin = synthetic.workload(CHUNK_WL, seed=1005 + 1000 * rank, **over)
    din = synthetic.workload(DECODE_WL, seed=1004 + 1000 * rank)
    B, T = cin.q.shape[:2]
    tokens = B * T
    host = {k: getattr(cin, k).pin_memory() for k in ("q", "k", "v", "g", "beta")}
    d = {k: v.to(dev) for k, v in host.items()}
    dd = {k: getattr(din, k).to(dev) for k in ("q", "k", "v", "g", "beta", "ssm_state",
                                               "batch_indices")}
    o = torch.empty_like(d["v"])
    fin = torch.empty(B, HV_, K_, V_, dtype=torch.float32, device=dev)
    od = torch.empty_like(dd["v"])
    n_real = int((din.batch_indices >= 0).sum())
    stream = torch.cuda.current_stream(dev)
    path = chunk_fwd_path(K_, V_, torch.bfloat16)
    launches_per_step = (1 if path == 1 else 4) + 1

    def chunk():
        if args.only in ("decode", "backward"):
            return
        chunk_gated_delta_rule(d["q"], d["k"], d["v"], d["g"], d["beta"], output_final_state=True,
                               use_qk_l2norm_in_kernel=True, out=o, final_state=fin)

    def decode():
        if args.only in ("chunk", "backward"):
            return
        gated_delta_decode(dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], dd["ssm_state"],
                           dd["batch_indices"], out=od)

    for _ in range(args.warmup):
        chunk()
        decode()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        for e0, e1, e2 in ev:
            e0.record(stream)
            chunk()
            e1.record(stream)
            decode()
            e2.record(stream)
        t_end.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    total_ms = t_start.elapsed_time(t_end)
    chunk_ms = [a.elapsed_time(b) for a, b, _ in ev]
    dec_ms = [b.elapsed_time(c) for _, b, c in ev]
    total_ms = max_over_ranks(total_ms, world, dev)
    chunk_sum = max_over_ranks(sum(chunk_ms), world, dev)
    dec_sum = max_over_ranks(sum(dec_ms), world, dev)
    K = args.steps
    chunk_avg_s = max(chunk_sum, 1e-6) / K / 1000.0
    dec_avg_s = max(dec_sum, 1e-6) / K / 1000.0
    value = world * tokens / chunk_avg_s

    # end to end through the public API: pinned host inputs in, o and the final state out.
    # Sequential: copy in, compute, copy out, one step after another on one stream.  Pipelined:
    # the copy-in of step s + 1 and the copy-out of step s - 1 run on their own streams while
    # step s computes (double-buffered device tensors); every byte still crosses the link.
    o_host = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for _ in range(2)]
    f_host = [torch.empty(fin.shape, dtype=fin.dtype, pin_memory=True) for _ in range(2)]
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = o_host[0].numel() * o_host[0].element_size() + f_host[0].numel() * f_host[0].element_size()
    e2e_val = e2e_seq = link = dec_e2e = None
    if args.only is None:
        e2e_steps = max(2, min(K, 50))   # the timed steps, as for the device timing: the pipeline's fill and drain a small share
        # one untimed step first: the caching allocator's first blocks of these sizes (GBs) are
        # device allocations, which would otherwise land in the first timed step
        g = {k: v.to(dev, non_blocking=True) for k, v in host.items()}
        oo, ff = chunk_gated_delta_rule(g["q"], g["k"], g["v"], g["g"], g["beta"],
                                        output_final_state=True, use_qk_l2norm_in_kernel=True)
        o_host[0].copy_(oo, non_blocking=True)
        f_host[0].copy_(ff, non_blocking=True)
        del g, oo, ff
        # device buffers and the call's workspace allocated once, outside the timed region
        Bq, Tq, Hqk_, Kq = d["q"].shape
        ws_e2e = torch.empty(max(1, chunk_workspace_size(Bq, Tq, Hqk_, d["v"].shape[2], Kq, d["v"].shape[3], Bq,
                                                         d["q"].dtype, d["beta"].dtype)),
                             dtype=torch.uint8, device=dev)
        g = {k: torch.empty_like(d[k]) for k in host}
        oo, ff = torch.empty_like(o), torch.empty_like(fin)
        torch.cuda.synchronize()
        barrier(world)
        ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        phase = []   # per step: after the copy-in, after the call, after the copy-out
        ea.record(stream)
        for _ in range(e2e_steps):
            p0 = torch.cuda.Event(enable_timing=True)
            p0.record(stream)
            for k in host:
                g[k].copy_(host[k], non_blocking=True)
            p1 = torch.cuda.Event(enable_timing=True)
            p1.record(stream)
            chunk_gated_delta_rule(g["q"], g["k"], g["v"], g["g"], g["beta"], output_final_state=True,
                                   use_qk_l2norm_in_kernel=True, out=oo, final_state=ff, workspace=ws_e2e)
            p2 = torch.cuda.Event(enable_timing=True)
            p2.record(stream)
            o_host[0].copy_(oo, non_blocking=True)
            f_host[0].copy_(ff, non_blocking=True)
            p3 = torch.cuda.Event(enable_timing=True)
            p3.record(stream)
            phase.append((p0, p1, p2, p3))
        eb.record(stream)
        torch.cuda.synchronize()
        e2e_seq = world * tokens / (max_over_ranks(ea.elapsed_time(eb), world, dev) / e2e_steps / 1000.0)
        h2d_all = [a.elapsed_time(b) for a, b, _, _ in phase]
        call_all = [b.elapsed_time(c) for _, b, c, _ in phase]
        d2h_all = [c.elapsed_time(e) for _, _, c, e in phase]
        h2d_ms, call_ms, d2h_ms = _median(h2d_all), _median(call_all), _median(d2h_all)
        link = {"h2d_gbs": h2d / (h2d_ms / 1e3) / 1e9, "d2h_gbs": d2h / (d2h_ms / 1e3) / 1e9,
                "h2d_ms": h2d_ms, "d2h_ms": d2h_ms, "call_ms": call_ms,
                "h2d_ms_max": max(h2d_all), "d2h_ms_max": max(d2h_all), "call_ms_max": max(call_all),
                "h2d_slowest_step": h2d_all.index(max(h2d_all)), "d2h_slowest_step": d2h_all.index(max(d2h_all)),
                "how": "pinned host <-> device copies of one step, median (and slowest) over the "
                       "sequential end-to-end steps (CUDA events around the copies); call_ms: the "
                       "call between them. The host link and host memory are shared with other "
                       "jobs on the machine, so single slow steps show up in the maxima"}
        del g, oo, ff
        # pipelined over three streams
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        bin_ = [{k: torch.empty_like(d[k]) for k in host} for _ in range(2)]
        bout = [(torch.empty_like(o), torch.empty_like(fin)) for _ in range(2)]
        in_free, out_free = [None, None], [None, None]
        torch.cuda.synchronize()
        barrier(world)
        ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ea.record(stream)
        s_in.wait_event(ea)
        s_out.wait_event(ea)
        for st in range(e2e_steps):
            b = st % 2
            if in_free[b] is not None:
                s_in.wait_event(in_free[b])      # step st - 2 has finished reading these inputs
            with torch.cuda.stream(s_in):
                for k in host:
                    bin_[b][k].copy_(host[k], non_blocking=True)
            ev_in = torch.cuda.Event()
            ev_in.record(s_in)
            stream.wait_event(ev_in)
            if out_free[b] is not None:
                stream.wait_event(out_free[b])   # the copy-out of step st - 2 is done
            x = bin_[b]
            chunk_gated_delta_rule(x["q"], x["k"], x["v"], x["g"], x["beta"],
                                   output_final_state=True, use_qk_l2norm_in_kernel=True,
                                   out=bout[b][0], final_state=bout[b][1], workspace=ws_e2e)
            in_free[b] = torch.cuda.Event()
            in_free[b].record(stream)
            s_out.wait_event(in_free[b])
            with torch.cuda.stream(s_out):
                o_host[b].copy_(bout[b][0], non_blocking=True)
                f_host[b].copy_(bout[b][1], non_blocking=True)
            out_free[b] = torch.cuda.Event()
            out_free[b].record(s_out)
        stream.wait_stream(s_in)
        stream.wait_stream(s_out)
        eb.record(stream)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(ea.elapsed_time(eb), world, dev) / e2e_steps
        e2e_val = world * tokens / (e2e_ms / 1000.0)
        del bin_, bout
        # decode end to end: the step's inputs (q, k, v, g, beta, batch_indices) from pinned
        # host memory, the step on the resident state cache, o back into pinned host memory.
        # Pipelined like the chunked case: the copy-in of step s + 1 and the copy-out of step
        # s - 1 run on their own streams while step s updates the cache (the steps themselves
        # stay in order on the compute stream).
        dhost = {k: getattr(din, k).pin_memory() for k in ("q", "k", "v", "g", "beta", "batch_indices")}
        od_host = [torch.empty(od.shape, dtype=od.dtype, pin_memory=True) for _ in range(2)]
        dbin = [{k: torch.empty_like(v, device=dev) for k, v in dhost.items()} for _ in range(2)]
        dbout = [torch.empty_like(od) for _ in range(2)]
        d_in_free, d_out_free = [None, None], [None, None]

        def dec_e2e_step(st):
            b = st % 2
            if d_in_free[b] is not None:
                s_in.wait_event(d_in_free[b])     # step st - 2 has read these inputs
            with torch.cuda.stream(s_in):
                for k in dhost:
                    dbin[b][k].copy_(dhost[k], non_blocking=True)
            ev_in = torch.cuda.Event()
            ev_in.record(s_in)
            stream.wait_event(ev_in)
            if d_out_free[b] is not None:
                stream.wait_event(d_out_free[b])   # the copy-out of step st - 2 is done
            x = dbin[b]
            gated_delta_decode(x["q"], x["k"], x["v"], x["g"], x["beta"], dd["ssm_state"],
                               x["batch_indices"], out=dbout[b])
            d_in_free[b] = torch.cuda.Event()
            d_in_free[b].record(stream)
            s_out.wait_event(d_in_free[b])
            with torch.cuda.stream(s_out):
                od_host[b].copy_(dbout[b], non_blocking=True)
            d_out_free[b] = torch.cuda.Event()
            d_out_free[b].record(s_out)

        for st in range(3):
            dec_e2e_step(st)
        dsteps = max(5, min(K, 50))
        torch.cuda.synchronize()
        barrier(world)
        ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ea.record(stream)
        s_in.wait_event(ea)
        s_out.wait_event(ea)
        for st in range(dsteps):
            dec_e2e_step(st)
        stream.wait_stream(s_in)
        stream.wait_stream(s_out)
        eb.record(stream)
        torch.cuda.synchronize()
        dms = max_over_ranks(ea.elapsed_time(eb), world, dev) / dsteps
        dec_e2e = {"value": world * n_real / (dms / 1e3), "unit": "requests/s",
                   "h2d_bytes_per_step": sum(v.numel() * v.element_size() for v in dhost.values()),
                   "d2h_bytes_per_step": od_host[0].numel() * od_host[0].element_size(), "ms": dms,
                   "pipelined": True,
                   "how": "inputs copied in from pinned host memory and o copied out every step "
                          "(the copies of neighbouring steps overlapped with the step), the state "
                          "cache resident on the device; %d steps" % dsteps}

    flops = FLOP_PER_TOKEN * tokens
    alg_bytes = BYTES_PER_TOKEN * tokens + B * HV_ * STATE_BYTES   # + the final state written
    achieved_gbs = alg_bytes / chunk_avg_s / 1e9
    achieved_tf = flops / chunk_avg_s / 1e12
    traffic = traffic_record()
    dec_bytes = n_real * HV_ * STATE_BYTES * 2
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": total_ms / K, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "global_batch": world * B, "seq_len": T, "parallelism": "dp%d" % world,
                   "l2": "inputs larger than L2 (1.6 GB chunk inputs, 1 GiB state cache); no flush",
                   "chunk_path": "tcgen05 fused" if path == 1 else "fp32 CUDA-core"},
        "roofline": {"bound": "hbm", "achieved": achieved_gbs, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved_gbs / hbm_peak, "traffic": traffic,
                     "peak_source": peak_src, "kernel": "chunk_tc_kernel" if path == 1 else
                     "chunk kernels"},
        "tensor": {"achieved": achieved_tf, "peak": bf16_peak, "unit": "TFLOP/s",
                   "frac": achieved_tf / bf16_peak, "flop_per_token": FLOP_PER_TOKEN,
                   "peak_source": peak_src},
        "chunk_ms": chunk_avg_s * 1000.0,
        "chunk_ms_median": max_over_ranks(_median(chunk_ms), world, dev),
        "decode": {"ms": dec_avg_s * 1000.0, "ms_median": max_over_ranks(_median(dec_ms), world, dev),
                   "requests_per_s": world * n_real / dec_avg_s,
                   "tokens_per_s_incl_padding": world * din.q.shape[0] / dec_avg_s,
                   "state_gbs": dec_bytes / dec_avg_s / 1e9,
                   "hbm_frac": dec_bytes / dec_avg_s / 1e9 / hbm_peak},
        "e2e": {"value": e2e_val, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "pipelined": True, "value_sequential": e2e_seq,
                "link": link, "decode": dec_e2e},
        "gpu_launches": launches_per_step * K,
        "clocks": clk.summary(),
    }
    if args.only is None and not args.no_product:
        line["product"] = measure_product(dev, 1006 + 1000 * rank)
    if args.only is None and not args.no_extras:
        line["decode"].update(measure_extras(dev, chunk, decode))
        gsec = line["decode"]["decode_graph_ms"] / 1000.0
        line["decode"]["state_gbs_graph"] = dec_bytes / gsec / 1e9
        line["decode"]["hbm_frac_graph"] = dec_bytes / gsec / 1e9 / hbm_peak
        line["other_configs"] = measure_configs(dev, bf16_peak)
    if args.only in (None, "backward") and not args.no_backward:
        line["backward"] = measure_backward(dev, cin, d, 1007 + 1000 * rank,
                                            steps=args.backward_steps)
    if args.only == "chunk":      # profiling runs: the half that was not timed is not reported
        line["decode"] = None
    elif args.only in ("decode", "backward"):
        line.update(value=None, chunk_ms=None, roofline=None, tensor=None)
        if args.only == "backward":
            line["decode"] = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        sample = 8192
        times, cores = [], 1
        for _ in range(3):
            dt, cores = cpu_oracle_sample(cin, sample)
            times.append(dt)
        line["cpu_baseline"] = {"value": sample / statistics.median(times), "unit": "tokens/s",
                                "cores": cores, "kind": "oracle",
                                "sample": "first %d tokens of sequence 0 of the same batch, all "
                                          "32 value heads (fp64 recurrence), median of 3" % sample,
                                "per_config": measure_cpu_baselines(cin, din)}
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
