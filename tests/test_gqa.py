"""Grouped-query (and multi-query) attention: the CUDA path vs the fp64
oracle. Query head h reads key/value head h / (H / Hkv); that is ordinary
attention on K and V with each key/value head repeated for its group, and
the gradients of K and V are the group sums of the repeated heads'
gradients, so the oracle runs on the repeated tensors."""
import math

import numpy as np
import pytest
import torch

from exact_io_aware_108_b300 import inputs
from oracle import ref
from tests.sampled import check_bwd_every_head
from tests.tolerance import TOL_GRAD, TOL_LSE, TOL_O, check, half_ulp

pytestmark = pytest.mark.gpu

CASES = [
    # B, H, Hkv, N, d, dtype, causal
    (2, 4, 2, 300, 64, "bf16", True),
    (1, 4, 1, 257, 128, "f16", False),   # multi-query
    (2, 6, 3, 384, 128, "bf16", True),
    (1, 8, 2, 200, 64, "f16", False),
]


def _repeat(x, group):
    return x.repeat_interleave(group, dim=1)


def _run(t, scale, causal, kv_len=None):
    import exact_io_aware_108_b300 as fa
    q, k, v, do = (t[n].cuda() for n in ("q", "k", "v", "dout"))
    kl = None if kv_len is None else kv_len.to(torch.int32).cuda()
    o, lse, o_res = fa.attention_forward(q, k, v, scale, causal=causal, kv_len=kl,
                                         return_residual=True)
    dq, dk, dv = fa.attention_backward(q, k, v, o, lse, do, scale, causal=causal, kv_len=kl,
                                       o_res=o_res)
    torch.cuda.synchronize()
    assert fa.fa_get_device_error() == 0
    assert dk.shape == t["k"].shape and dv.shape == t["v"].shape
    return o.cpu(), lse.cpu(), dq.cpu(), dk.cpu(), dv.cpu()


def _compare(t, H, Hkv, scale, causal, kv_len=None):
    g = H // Hkv
    o, lse, dq, dk, dv = _run(t, scale, causal, kv_len)
    kr, vr = _repeat(t["k"], g), _repeat(t["v"], g)
    o_ref, lse_ref = ref.attn_fwd(t["q"], kr, vr, scale, causal, kv_len)
    grads = ref.attn_bwd(t["q"], kr, vr, t["dout"], scale, causal, kv_len, rows_per_task=64)
    B, _, N, d = t["q"].shape
    dk_ref = np.asarray(grads[1]).reshape(B, Hkv, g, N, d).sum(axis=2)
    dv_ref = np.asarray(grads[2]).reshape(B, Hkv, g, N, d).sum(axis=2)
    dt = t["q"].dtype
    check("O", o, o_ref, TOL_O, dt)
    check("LSE", lse, lse_ref, TOL_LSE, torch.float32)
    check("dQ", dq, grads[0], TOL_GRAD, dt)
    check("dK", dk, dk_ref, TOL_GRAD, dt)
    check("dV", dv, dv_ref, TOL_GRAD, dt)


@pytest.mark.parametrize("B,H,Hkv,N,d,dt,causal", CASES)
def test_gqa_matches_oracle(B, H, Hkv, N, d, dt, causal):
    t = inputs.make_qkv(B, H, N, d, dt, seed=N + H + Hkv, hkv=Hkv)
    _compare(t, H, Hkv, 1.0 / math.sqrt(d), causal)


def test_gqa_with_key_padding():
    t = inputs.make_qkv(3, 4, 320, 128, "bf16", seed=31, hkv=2, kv_len_range=(100, 320))
    _compare(t, 4, 2, 1.0 / math.sqrt(128), False, t["kv_len"])


def test_gqa_sharp_matches_oracle():
    """Sharp softmax (Q, K x2, logit std 4) with grouped heads and key padding:
    the group sums of dK and dV collect the rounding of four heads."""
    t = inputs.make_qkv(2, 8, 640, 128, "bf16", seed=35, qk_mult=2.0, hkv=2,
                        kv_len_range=(300, 640))
    _compare(t, 8, 2, 1.0 / math.sqrt(128), True, t["kv_len"])


def test_gqa_sharp_equals_plain_path_on_repeated_kv():
    """Sharp softmax (Q, K x2) with key padding: the grouped path computes
    exactly what the plain path computes on K and V repeated per group: O
    and LSE bitwise, dQ up to the order of its fp32 reductions, dK and dV
    equal to the group sums of the plain path's per-head gradients up to
    their 16-bit rounding."""
    import exact_io_aware_108_b300 as fa
    t = inputs.make_qkv(3, 4, 320, 128, "bf16", seed=31, qk_mult=2.0, hkv=2,
                        kv_len_range=(100, 320))
    q, k, v, do = (t[n].cuda() for n in ("q", "k", "v", "dout"))
    kl = t["kv_len"].to(torch.int32).cuda()
    scale = 1.0 / math.sqrt(128)
    o, lse, res = fa.attention_forward(q, k, v, scale, kv_len=kl, return_residual=True)
    dq, dk, dv = fa.attention_backward(q, k, v, o, lse, do, scale, kv_len=kl, o_res=res)
    kr, vr = _repeat(k, 2).contiguous(), _repeat(v, 2).contiguous()
    o2, lse2, res2 = fa.attention_forward(q, kr, vr, scale, kv_len=kl, return_residual=True)
    dq2, dk2, dv2 = fa.attention_backward(q, kr, vr, o2, lse2, do, scale, kv_len=kl, o_res=res2)
    torch.cuda.synchronize()
    assert fa.fa_get_device_error() == 0
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    # dQ sums key tiles with fp32 atomics in no fixed order: the fp32 sums
    # agree to ~1e-6 relative, and their 16-bit roundings to within one ulp
    dq_a, dq_b = dq.cpu().double().numpy(), dq2.cpu().double().numpy()
    one_ulp = 2 * half_ulp(np.maximum(np.abs(dq_a), np.abs(dq_b)), torch.bfloat16)
    assert np.all(np.abs(dq_a - dq_b) <= one_ulp + 1e-4)
    for name, g, p in (("dK", dk, dk2), ("dV", dv, dv2)):
        per_head = p.cpu().double().numpy().reshape(3, 2, 2, 320, 128)
        p_sum = per_head.sum(axis=2)
        got = g.cpu().double().numpy()
        # the grouped result is rounded once, the plain path's two heads once each
        bound = half_ulp(got, torch.bfloat16) + half_ulp(per_head, torch.bfloat16).sum(axis=2)
        assert np.all(np.abs(got - p_sum) <= bound * (1 + 1e-9)), name


def test_gqa_with_hkv_equal_h_is_the_plain_path():
    """Hkv == H through the grouped entry points gives the plain results bitwise."""
    import exact_io_aware_108_b300 as fa
    t = inputs.make_qkv(2, 2, 384, 128, "bf16", seed=33, qk_mult=2.0)
    q, k, v, do = (t[n].cuda() for n in ("q", "k", "v", "dout"))
    scale = 1.0 / math.sqrt(128)
    o1, l1 = torch.empty_like(q), torch.empty(q.shape[:-1], device="cuda")
    o2, l2 = torch.empty_like(q), torch.empty(q.shape[:-1], device="cuda")
    fa.fa_fwd_ex(q, k, v, o1, l1, scale, True)
    fa.fa_fwd_gqa(q, k, v, o2, l2, scale, True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    ws = torch.empty(fa.fa_bwd_workspace_size(2, 2, 384, 128), dtype=torch.uint8, device="cuda")
    g1 = [torch.empty_like(q) for _ in range(3)]
    g2 = [torch.empty_like(q) for _ in range(3)]
    fa.fa_bwd(q, k, v, o1, l1, do, *g1, scale, True, workspace=ws)
    fa.fa_bwd_gqa(q, k, v, o1, l1, do, *g2, scale, True, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(g1[1], g2[1]) and torch.equal(g1[2], g2[2])
    # dQ: fp32 atomics in no fixed order; the 16-bit results agree to one ulp
    a_, b_ = g2[0].cpu().double().numpy(), g1[0].cpu().double().numpy()
    assert np.all(np.abs(a_ - b_) <= 2 * half_ulp(np.maximum(np.abs(a_), np.abs(b_)), q.dtype) + 1e-4)


def test_gqa_full_size_whole_heads():
    """The benchmark-sized grouped workload (sharp softmax: Q and K x 2):
    every dK and dV element of two key/value heads (the sums over their four
    query heads) and every O, LSE and dQ element of one of those query heads,
    against the oracle."""
    w = inputs.WORKLOADS["gqa_b4_h32_hkv8_n4096_d128_bf16_causal"]
    t = inputs.make_workload(w, with_dout=True)
    o, lse, dq, dk, dv = _run(t, w.scale, w.causal)
    g = w.H // w.hkv
    dt = t["q"].dtype
    for b, hkv in ((w.B - 1, 1), (0, w.hkv - 1)):
        hs = slice(hkv * g, (hkv + 1) * g)
        kr = _repeat(t["k"][b:b + 1, hkv:hkv + 1], g)
        vr = _repeat(t["v"][b:b + 1, hkv:hkv + 1], g)
        grads = ref.attn_bwd(t["q"][b:b + 1, hs], kr, vr, t["dout"][b:b + 1, hs], w.scale, w.causal,
                             rows_per_task=256)
        h0 = hkv * g  # first query head of the group: O, LSE and dQ checked there
        o_ref, lse_ref = ref.attn_fwd(t["q"][b:b + 1, h0:h0 + 1], kr[:, :1], vr[:, :1], w.scale,
                                      w.causal)
        check(f"O[{b},{h0}]", o[b, h0], o_ref[0, 0], TOL_O, dt)
        check(f"LSE[{b},{h0}]", lse[b, h0], lse_ref[0, 0], TOL_LSE, torch.float32)
        check(f"dQ[{b},{h0}]", dq[b, h0], grads[0][0, 0], TOL_GRAD, dt)
        check(f"dK[{b},{hkv}]", dk[b, hkv], np.asarray(grads[1])[0].sum(axis=0), TOL_GRAD, dt)
        check(f"dV[{b},{hkv}]", dv[b, hkv], np.asarray(grads[2])[0].sum(axis=0), TOL_GRAD, dt)


def test_gqa_full_size_every_head_sampled():
    """The same workload: dQ at sampled rows of every query head, dK and dV
    (group sums) at sampled rows of every key/value head, against the oracle."""
    w = inputs.WORKLOADS["gqa_b4_h32_hkv8_n4096_d128_bf16_causal"]
    t = inputs.make_workload(w, with_dout=True)
    _, _, dq, dk, dv = _run(t, w.scale, w.causal)
    worst = check_bwd_every_head(t, w, dq, dk, dv, seed=1)
    print("\ngqa sharp: max |d grad| over sampled rows of every head: "
          + ", ".join(f"{k} {v:.4g}" for k, v in worst.items()))
