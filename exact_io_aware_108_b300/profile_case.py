"""Run forward + backward of one attention problem a few times (for profilers).

    python -m exact_io_aware_108_b300.profile_case --B 2 --H 16 --N 4096 --d 128 \
        --dtype bf16 --causal --iters 2

Inputs are seeded N(0,1) (Q and K times --qk-mult); the forward writes O's
residual and the backward uses it, as in the benchmark (--plain: O and LSE
only, the inference forward).
"""
from __future__ import annotations

import argparse
import math

import torch

import exact_io_aware_108_b300 as fa


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--B", type=int, default=2)
    ap.add_argument("--H", type=int, default=16)
    ap.add_argument("--N", type=int, default=4096)
    ap.add_argument("--d", type=int, default=128)
    ap.add_argument("--dtype", choices=["f16", "bf16"], default="bf16")
    ap.add_argument("--causal", action="store_true")
    ap.add_argument("--qk-mult", type=float, default=2.0)
    ap.add_argument("--iters", type=int, default=2)
    ap.add_argument("--fwd-only", action="store_true")
    ap.add_argument("--plain", action="store_true", help="forward without O's residual")
    a = ap.parse_args()
    dt = torch.bfloat16 if a.dtype == "bf16" else torch.float16
    g = torch.Generator(device="cuda").manual_seed(0)
    shape = (a.B, a.H, a.N, a.d)
    q = (torch.randn(shape, device="cuda", generator=g) * a.qk_mult).to(dt)
    k = (torch.randn(shape, device="cuda", generator=g) * a.qk_mult).to(dt)
    v = torch.randn(shape, device="cuda", generator=g).to(dt)
    do = torch.randn(shape, device="cuda", generator=g).to(dt)
    scale = 1.0 / math.sqrt(a.d)
    ws = torch.empty(fa.fa_bwd_workspace_size(*shape), dtype=torch.uint8, device="cuda")
    for _ in range(a.iters):
        if a.plain:
            o, lse = fa.attention_forward(q, k, v, scale, a.causal)
            o_res = None
        else:
            o, lse, o_res = fa.attention_forward(q, k, v, scale, a.causal, return_residual=True)
        if not a.fwd_only:
            fa.attention_backward(q, k, v, o, lse, do, scale, a.causal, o_res=o_res, workspace=ws)
    torch.cuda.synchronize()
    assert fa.fa_get_device_error() == 0, "device error"
    print("ok", shape, a.dtype, "causal" if a.causal else "dense")


if __name__ == "__main__":
    main()
