"""Timing of the chunked forward on the fp32 CUDA-core path (the shapes the tensor-core kernel
does not take: head dims other than 128, fp32 I/O).

    python -m chunked_gated_delta_gdn_gb300.microbench.cuda_core_chunk [--reps 20]

Runs three shapes through the public call and prints one JSON line each with the mean time of
``--reps`` calls (CUDA events on the current stream, after three warm-up calls):

- the tiny fp32 case of the parity tests (1 x 256 tokens, 2 heads, K = V = 64);
- 4 x 8192 tokens, 16 query/key and 32 value heads, K = V = 64, bf16 I/O;
- 1 x 8192 tokens, 16 / 32 heads, K = V = 128, fp32 I/O.
"""
from __future__ import annotations

import argparse
import json

import torch

from .. import chunk_fwd_path, chunk_gated_delta_rule, synthetic


def cases():
    return [
        ("tiny_fp32", synthetic.workload("tiny_fp32")),
        ("k64_bf16_4x8192", synthetic.chunk_inputs(B=4, T=8192, Hqk=16, Hv=32, K=64, V=64,
                                                   dtype=torch.bfloat16, init="randn", seed=5)),
        ("k128_fp32_1x8192", synthetic.chunk_inputs(B=1, T=8192, Hqk=16, Hv=32, K=128, V=128,
                                                    dtype=torch.float32, init="randn", seed=6)),
    ]


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--reps", type=int, default=20)
    args = ap.parse_args()
    dev = torch.device("cuda", 0)
    for name, inp in cases():
        d = {k: (None if getattr(inp, k) is None else getattr(inp, k).to(dev))
             for k in ("q", "k", "v", "g", "beta", "initial_state")}

        def run():
            return chunk_gated_delta_rule(d["q"], d["k"], d["v"], d["g"], d["beta"],
                                          initial_state=d["initial_state"], output_final_state=True,
                                          use_qk_l2norm_in_kernel=True)

        for _ in range(3):
            run()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(args.reps):
            run()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / args.reps
        B, T = inp.q.shape[:2]
        print(json.dumps({"case": name, "path": "tcgen05 fused" if chunk_fwd_path(
            inp.q.shape[3], inp.v.shape[3], inp.q.dtype) == 1 else "fp32 CUDA-core",
            "ms": ms, "tokens_per_s": B * T / ms * 1e3}))


if __name__ == "__main__":
    main()
