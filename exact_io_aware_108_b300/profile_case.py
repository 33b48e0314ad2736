"""Run forward + backward of one attention problem a few times (for profilers).

    python -m exact_io_aware_108_b300.profile_case --B 2 --H 16 --N 4096 --d 128 \
        --dtype bf16 --causal --iters 2

Inputs are seeded N(0,1) (Q and K times --qk-mult); the forward writes O's
residual and the backward uses it, as in the benchmark (--plain: O and LSE
only, the inference forward).

    python -m exact_io_aware_108_b300.profile_case --decode --B 8 --H 32 --Hkv 8 \
        --ctx 4096 8192 --page-size 16 --splits 0 --iters 2

runs the paged decode instead (one new token per sequence, --nq for more);
--fp8 runs the 8-bit forward on e4m3 inputs of the given shape (d = 128);
--block-sparse P the block-sparse forward and backward (mask as in the
benchmark's block-sparse workload: tiles kept with probability P, seed 7,
diagonal kept).
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
    ap.add_argument("--decode", action="store_true", help="paged decode")
    ap.add_argument("--Hkv", type=int, default=8)
    ap.add_argument("--nq", type=int, default=1)
    ap.add_argument("--ctx", type=int, nargs=2, default=[4096, 8192])
    ap.add_argument("--page-size", type=int, default=16)
    ap.add_argument("--splits", type=int, default=0)
    ap.add_argument("--fp8", action="store_true", help="8-bit forward")
    ap.add_argument("--block-sparse", type=float, default=None, metavar="P",
                    help="block-sparse: 128x128 tiles kept with probability P (seed 7) plus the diagonal")
    a = ap.parse_args()
    if a.decode:
        return decode(a)
    if a.fp8:
        return fp8(a)
    dt = torch.bfloat16 if a.dtype == "bf16" else torch.float16
    g = torch.Generator(device="cuda").manual_seed(0)
    shape = (a.B, a.H, a.N, a.d)
    q = (torch.randn(shape, device="cuda", generator=g) * a.qk_mult).to(dt)
    k = (torch.randn(shape, device="cuda", generator=g) * a.qk_mult).to(dt)
    v = torch.randn(shape, device="cuda", generator=g).to(dt)
    do = torch.randn(shape, device="cuda", generator=g).to(dt)
    scale = 1.0 / math.sqrt(a.d)
    ws = torch.empty(fa.fa_bwd_workspace_size(*shape), dtype=torch.uint8, device="cuda")
    bm = None
    if a.block_sparse is not None:
        from exact_io_aware_108_b300 import inputs
        bm = inputs.make_block_mask(a.N, a.block_sparse, seed=7).cuda()
    causal = a.causal and bm is None
    for _ in range(a.iters):
        if a.plain:
            o, lse = fa.attention_forward(q, k, v, scale, causal, block_mask=bm)
            o_res = None
        else:
            o, lse, o_res = fa.attention_forward(q, k, v, scale, causal, block_mask=bm,
                                                 return_residual=True)
        if not a.fwd_only:
            fa.attention_backward(q, k, v, o, lse, do, scale, causal, block_mask=bm, o_res=o_res,
                                  workspace=ws)
    torch.cuda.synchronize()
    assert fa.fa_get_device_error() == 0, "device error"
    print("ok", shape, a.dtype, "causal" if a.causal else "dense")


def fp8(a):
    from exact_io_aware_108_b300 import inputs
    t = inputs.make_qkv_fp8(a.B, a.H, a.N, a.d, seed=0)
    q, k, v = (t[n].cuda() for n in ("q", "k", "v"))
    for _ in range(a.iters):
        fa.attention_forward_fp8(q, k, v, t["q_descale"], t["k_descale"], t["v_descale"], causal=a.causal)
    torch.cuda.synchronize()
    assert fa.fa_get_device_error() == 0, "device error"
    print("ok fp8", a.B, a.H, a.N, a.d, "causal" if a.causal else "dense")


def decode(a):
    from exact_io_aware_108_b300 import inputs
    t = inputs.make_paged_decode(a.B, a.H, a.Hkv, a.nq, a.d, a.dtype, a.page_size, tuple(a.ctx), seed=0)
    t = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in t.items()}
    for _ in range(a.iters):
        fa.attention_decode_paged(t["q"], t["k_cache"], t["v_cache"], t["block_table"], t["seq_len"],
                                  num_splits=a.splits)
    torch.cuda.synchronize()
    assert fa.fa_get_device_error() == 0, "device error"
    print("ok decode", a.B, a.H, a.Hkv, a.nq, a.d, a.page_size, a.ctx)


if __name__ == "__main__":
    main()
