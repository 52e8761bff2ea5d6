"""Run one kernel of the library on one workload a few times (for profilers).

    python -m resident_kv_cache_gb300.profile_case prefill [--batch 2] [--iters 3]
    python -m resident_kv_cache_gb300.profile_case decode  [--batch 32] [--iters 3]
    python -m resident_kv_cache_gb300.profile_case scatter [--batch 4] [--iters 3]

prefill: causal GQA prefill (S=2048, H=32, Hk=8, D=128) of `batch` sequences;
decode:  batched decode step (H=32, Hk=8, D=128, cache length 4096, lengths U{1..4096})
         of `batch` sequences; scatter: the causal GQA cache fill of `batch` sequences.
Inputs are the seeded synthetic ones; prints the mean time per launch (CUDA events).
"""
from __future__ import annotations

import argparse
import dataclasses

import torch

from . import binding, build, inputs


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("kernel", choices=["prefill", "decode", "scatter"])
    ap.add_argument("--batch", type=int, default=None)
    ap.add_argument("--iters", type=int, default=3)
    ap.add_argument("--warmup", type=int, default=2)
    a = ap.parse_args()
    build.build()
    binding.load()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    if a.kernel in ("prefill", "scatter"):
        s = dataclasses.replace(inputs.CAUSAL_GQA, B=a.batch or inputs.CAUSAL_GQA.B)
        q, k, v = (torch.from_numpy(x).to(dev) for x in inputs.prefill_inputs(s))
        if a.kernel == "prefill":
            o = torch.empty_like(q)
            run = lambda: binding.attn_prefill(q, k, v, o, s.B, s.S, s.H, s.Hk, s.D, True)
            work, unit = s.flops / 1e12, "TFLOP/s"
        else:
            L = inputs.CAUSAL_GQA_CACHE_LEN
            kc = torch.zeros((s.B, s.Hk, L, s.D), device=dev)
            vc = torch.zeros_like(kc)
            sp = torch.zeros(s.B, dtype=torch.int32, device=dev)
            run = lambda: binding.kv_cache_scatter(k, v, kc, vc, s.B, s.S, s.Hk, s.D, L, sp)
            work, unit = 4.0 * s.B * s.S * s.Hk * s.D * 4 / 1e9, "GB/s"
    else:
        d = dataclasses.replace(inputs.BATCHED_DECODE, M=a.batch or inputs.BATCHED_DECODE.M)
        x = inputs.batched_decode_inputs(d)
        kc, vc, qd = (torch.from_numpy(x[n]).to(dev) for n in ("k_cache", "v_cache", "q"))
        ln = torch.from_numpy(x["lens"]).to(dev)
        od = torch.empty_like(qd)
        nws = binding.attn_decode_workspace_bytes(d.M, d.H, d.Hk, d.D, d.Lmax)
        ws = torch.zeros(nws, dtype=torch.uint8, device=dev)
        run = lambda: binding.attn_decode_batched(qd, kc, vc, od, d.M, d.H, d.Hk, d.D, d.Lmax, ln, 0.0, ws, nws)
        work, unit = (2.0 * d.Hk * d.D * 4 * float(x["lens"].sum()) + 2.0 * d.M * d.H * d.D * 4) / 1e9, "GB/s"
    for _ in range(a.warmup):
        run()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(a.iters):
        run()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / a.iters
    print(f"{a.kernel}: {ms:.4f} ms per launch, {work / (ms * 1e-3):.1f} {unit}")


if __name__ == "__main__":
    main()
