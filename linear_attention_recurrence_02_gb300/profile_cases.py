"""Run one workload of the library a fixed number of times, for profiler captures.

    python -m linear_attention_recurrence_02_gb300.profile_cases CASE [--B 64] [--T 4096] [--H 96]
        [--gate channel|head|none] [--dtype bf16|f32] [--warmup 3] [--reps 2]

Every call goes through the C ABI exactly as a user's does. Inputs are drawn
on the device by a seeded torch generator with the workloads' distributions
(q, k, v, x ~ N(0,1) in bf16, g = -softplus(N(0,1)), beta = sigmoid(N(0,1)),
state ~ N(0, 0.02^2); --dtype f32 keeps the prefill's q, k, v in fp32); nothing is checked, the point is a known launch
sequence: `warmup` calls, then `reps` calls, one launch of the named kernel
each (the prefill adds no other launch for one sequence). Cases:

  decode          fused short conv + decode step (kda_shortconv_decode_step)
  decode_epi      the same with the gated RMSNorm output epilogue
  decode_unfused  the decode step alone (kda_decode_step)
  shortconv_step  the short conv decode step alone (kda_shortconv_step)
  prefill         chunked prefill of one T-token sequence (C = 64)
  shortconv_prefill  the short conv over one T-token prompt with rings in and out
  epilogue        the gated RMSNorm output epilogue over T x H rows (sigmoid gate)
"""
from __future__ import annotations

import argparse

import torch
import torch.nn.functional as F

from linear_attention_recurrence_02_gb300 import kda


def main(argv=None) -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("case", choices=["decode", "decode_epi", "decode_unfused", "shortconv_step", "prefill",
                                     "shortconv_prefill", "epilogue"])
    ap.add_argument("--B", type=int, default=64)
    ap.add_argument("--T", type=int, default=4096)
    ap.add_argument("--H", type=int, default=96)
    ap.add_argument("--D", type=int, default=128)
    ap.add_argument("--gate", default="channel", choices=["channel", "head", "none"])
    ap.add_argument("--dtype", default="bf16", choices=["bf16", "f32"])
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--reps", type=int, default=2)
    a = ap.parse_args(argv)
    dev = torch.device("cuda", 0)
    gen = torch.Generator(device=dev).manual_seed(1234)
    bf = torch.bfloat16
    B, T, H, D = a.B, a.T, a.H, a.D

    def rnd(*shape, scale=1.0):
        return torch.randn(shape, generator=gen, device=dev) * scale

    def gate_of(shape):
        g = -F.softplus(rnd(*shape))
        if a.gate == "head":
            return g[..., 0].contiguous()
        return None if a.gate == "none" else g

    if a.case in ("decode", "decode_epi", "decode_unfused", "shortconv_step"):
        x, ring, w = rnd(B, 3, H, D).to(bf), rnd(B, 3, H, 3, D).to(bf), rnd(3, H, D, 4, scale=0.5)
        g, beta = gate_of((B, H, D)), torch.sigmoid(rnd(B, H))
        state = rnd(B, H, D, D, scale=0.02)
        out = torch.empty((B, H, D), dtype=bf, device=dev)
        og, nw = rnd(B, H, D).to(bf), torch.rand((D,), generator=gen, device=dev) + 0.5
        y = torch.empty((3, B, H, D), dtype=bf, device=dev)
        qkv = rnd(3, B, H, D).to(bf)

        def call():
            if a.case == "decode":
                kda.kda_shortconv_decode_step_gated(x, ring, w, g, beta, state, out, gate=a.gate)
            elif a.case == "decode_epi":
                kda.kda_shortconv_decode_step_epi(x, ring, w, g, beta, state, og, nw, out, gate=a.gate)
            elif a.case == "decode_unfused":
                kda.kda_decode_step_gated(qkv[0], qkv[1], qkv[2], g, beta, state, out, gate=a.gate)
            else:
                kda.kda_shortconv_step(x, ring, w, y)
    elif a.case == "shortconv_prefill":
        x, w = rnd(T, 3, H, D).to(bf), rnd(3, H, D, 4, scale=0.5)
        rin, rout = rnd(1, 3, H, 3, D).to(bf), torch.empty((1, 3, H, 3, D), dtype=bf, device=dev)
        y = torch.empty((3, T, H, D), dtype=bf, device=dev)

        def call():
            kda.kda_shortconv_prefill(x, w, y, ring_in=rin, ring_out=rout)
    elif a.case == "epilogue":
        o, og = rnd(T, H, D).to(bf), rnd(T, H, D, scale=2.0).to(bf)
        nw, y = torch.rand((D,), generator=gen, device=dev) + 0.5, torch.empty((T, H, D), dtype=bf, device=dev)

        def call():
            kda.kda_gated_rmsnorm(o, og, nw, y)
    else:
        dt = bf if a.dtype == "bf16" else torch.float32
        q, k, v = rnd(T, H, D).to(dt), rnd(T, H, D).to(dt), rnd(T, H, D).to(dt)
        g, beta = gate_of((T, H, D)), torch.sigmoid(rnd(T, H))
        out = torch.empty_like(q)
        sf = torch.empty((1, H, D, D), device=dev)

        def call():
            kda.kda_chunk_prefill_gated(q, k, v, g, beta, out, gate=a.gate, final_state=sf, chunk_size=64)

    for _ in range(a.warmup + a.reps):
        call()
    torch.cuda.synchronize(dev)
    kda.kda_sync_status()
    print(f"{a.case}: {a.warmup} + {a.reps} calls done")
    return 0


if __name__ == "__main__":
    raise SystemExit(main())
