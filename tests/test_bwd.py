"""Backward parity: the CUDA path (through the C ABI) vs the fp64 oracle."""
import math

import numpy as np
import pytest
import torch

from exact_io_aware_108_b300 import inputs
from oracle import ref
from tests.sampled import check_bwd_every_head
from tests.tolerance import TOL_GRAD, check

pytestmark = pytest.mark.gpu


def run_bwd(t, scale, causal=False, kv_len=None, block_mask=None, residual=True):
    import exact_io_aware_108_b300 as fa
    q, k, v, do = (t[n].cuda() for n in ("q", "k", "v", "dout"))
    kl = None if kv_len is None else kv_len.to(torch.int32).cuda()
    bm = None if block_mask is None else block_mask.to(torch.uint8).cuda()
    o, lse, o_res = fa.attention_forward(q, k, v, scale, causal=causal, kv_len=kl, block_mask=bm,
                                         return_residual=True)
    dq, dk, dv = fa.attention_backward(q, k, v, o, lse, do, scale, causal=causal, kv_len=kl,
                                       block_mask=bm, o_res=o_res if residual else None)
    torch.cuda.synchronize()
    assert fa.fa_get_device_error() == 0
    return dq.cpu(), dk.cpu(), dv.cpu()


def compare_full(t, scale, causal=False, kv_len=None, block_mask=None):
    dq, dk, dv = run_bwd(t, scale, causal, kv_len, block_mask)
    g = ref.attn_bwd(t["q"], t["k"], t["v"], t["dout"], scale, causal, kv_len, block_mask,
                     rows_per_task=64)
    dt = t["q"].dtype
    check("dQ", dq, g[0], TOL_GRAD, dt)
    check("dK", dk, g[1], TOL_GRAD, dt)
    check("dV", dv, g[2], TOL_GRAD, dt)
    return dq, dk, dv


SHAPES = [
    (1, 2, 256, 64, "f16", False),
    (1, 1, 1, 64, "f16", False),
    (2, 1, 100, 64, "bf16", True),
    (1, 2, 129, 128, "bf16", False),
    (2, 2, 300, 128, "f16", True),
    (1, 3, 513, 64, "bf16", True),
    (1, 1, 640, 128, "bf16", False),
    (3, 1, 257, 64, "f16", False),
]


@pytest.mark.parametrize("B,H,N,d,dt,causal", SHAPES)
def test_bwd_matches_oracle(B, H, N, d, dt, causal):
    t = inputs.make_qkv(B, H, N, d, dt, seed=N + d + 1)
    compare_full(t, 1.0 / math.sqrt(d), causal)


@pytest.mark.parametrize("d,dt", [(64, "f16"), (128, "bf16")])
def test_bwd_sharp_softmax(d, dt):
    t = inputs.make_qkv(2, 2, 384, d, dt, seed=4, qk_mult=2.0)
    compare_full(t, 1.0 / math.sqrt(d), causal=True)


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_kv_len_edges(causal):
    N, d = 300, 64
    t = inputs.make_qkv(8, 1, N, d, "f16", seed=12)
    kv_len = torch.tensor([1, 127, 128, 129, 300, 0, 1000, 255], dtype=torch.int32)
    dq, dk, dv = compare_full(t, 0.125, causal, kv_len=kv_len)
    assert torch.all(dq[5] == 0) and torch.all(dk[5] == 0) and torch.all(dv[5] == 0)
    assert torch.all(dk[1, :, 127:] == 0) and torch.all(dv[1, :, 127:] == 0)


def test_bwd_blocksparse_matches_oracle():
    N, d = 640, 64
    t = inputs.make_qkv(2, 2, N, d, "f16", seed=15)
    bm = inputs.make_block_mask(N, 0.4, seed=7)
    bm[3, :] = 0
    bm[:, 1] = 0  # key tile 1 is seen by nobody: dK = dV = 0 there
    bm[1, 1] = 0
    dq, dk, dv = compare_full(t, 0.125, block_mask=bm)
    assert torch.all(dk[:, :, 128:256] == 0) and torch.all(dv[:, :, 128:256] == 0)
    assert torch.all(dq[:, :, 384:512] == 0)


def test_bwd_blocksparse_all_ones_equals_dense():
    N, d = 512, 128
    t = inputs.make_qkv(1, 2, N, d, "bf16", seed=16)
    ones = torch.ones((4, 4), dtype=torch.uint8)
    a = run_bwd(t, 0.09, block_mask=ones)
    b = run_bwd(t, 0.09)
    # dK and dV are accumulated in a fixed order: bitwise equal
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
    # dQ sums key tiles with fp32 atomics (order may differ): within tolerance
    g = ref.attn_bwd(t["q"], t["k"], t["v"], t["dout"], 0.09, rows_per_task=64)
    check("dQ sparse", a[0], g[0], TOL_GRAD, t["q"].dtype)
    check("dQ dense", b[0], g[0], TOL_GRAD, t["q"].dtype)


def test_bwd_without_residual_fp16():
    """Without O's residual D comes from the 16-bit O alone; with fp16 outputs
    that is still inside the gradient tolerance."""
    t = inputs.make_qkv(2, 2, 384, 128, "f16", seed=18)
    dq, dk, dv = run_bwd(t, 0.0884, True, residual=False)
    g = ref.attn_bwd(t["q"], t["k"], t["v"], t["dout"], 0.0884, True, rows_per_task=64)
    for name, x, r in (("dQ", dq, g[0]), ("dK", dk, g[1]), ("dV", dv, g[2])):
        check(name, x, r, TOL_GRAD, t["q"].dtype)


def test_bwd_dk_dv_deterministic():
    t = inputs.make_qkv(2, 2, 384, 64, "bf16", seed=17)
    a = run_bwd(t, 0.125, True)
    b = run_bwd(t, 0.125, True)
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])


@pytest.mark.parametrize("B,H,Hkv,N,d,dt,causal,sparse", [
    (4, 8, 8, 1100, 128, "bf16", True, False),   # 288 key tiles, ragged tail
    (2, 16, 4, 1536, 64, "f16", False, False),   # grouped heads: 96 items of 4 query heads each
    (1, 8, 8, 2560, 64, "bf16", False, True),    # block-sparse, 30 % of the tiles kept
])
def test_bwd_persistent_items_repeatable(B, H, Hkv, N, d, dt, causal, sparse):
    """The main kernel runs one CTA per SM that takes work items (key tile,
    key/value head) from a counter; with many more items than SMs, repeated
    calls must give bitwise the same dK and dV (each key tile is summed in
    one CTA in a fixed order, whichever CTA takes it), and dQ within the
    rounding of its unordered fp32 reductions."""
    import exact_io_aware_108_b300 as fa
    t = inputs.make_qkv(B, H, N, d, dt, seed=23, hkv=Hkv)
    q, k, v, do = (t[n].cuda() for n in ("q", "k", "v", "dout"))
    bm = inputs.make_block_mask(N, 0.3, seed=5).to(torch.uint8).cuda() if sparse else None
    scale = 1.0 / math.sqrt(d)
    o, lse, o_res = fa.attention_forward(q, k, v, scale, causal=causal, block_mask=bm, return_residual=True)
    first = None
    for _ in range(8):
        dq, dk, dv = fa.attention_backward(q, k, v, o, lse, do, scale, causal=causal, block_mask=bm,
                                           o_res=o_res)
        torch.cuda.synchronize()
        assert fa.fa_get_device_error() == 0
        if first is None:
            first = (dq.clone(), dk.clone(), dv.clone())
            assert torch.isfinite(dq).all() and torch.isfinite(dk).all() and torch.isfinite(dv).all()
            continue
        assert torch.equal(dk, first[1]) and torch.equal(dv, first[2])
        assert (dq.float() - first[0].float()).abs().max().item() <= 2.0 ** -6 * first[0].float().abs().max().item()


# ----------------------------------------------------- full-size workloads

FULL_SIZE = [
    "bert_b16_h16_n512_d64_f16_kvlen",
    "gpt2_b8_h12_n1024_d64_bf16_causal",
    "long_b8_h16_n4096_d128_bf16_causal",
    "long_b4_h16_n8192_d128_bf16_causal",
    "long_b2_h16_n16384_d128_bf16_causal",
    "blocksparse_b2_h8_n16384_d64_f16",
]


@pytest.mark.parametrize("name", FULL_SIZE)
def test_bwd_full_size_whole_heads(name):
    """Full-size workload, same launches as the benchmark; every dQ, dK, dV
    element of two whole heads is checked against the oracle."""
    w = inputs.WORKLOADS[name]
    t = inputs.make_workload(w, with_dout=True)
    dq, dk, dv = run_bwd(t, w.scale, w.causal, t.get("kv_len"), t.get("block_mask"))
    for x in (dq, dk, dv):
        assert torch.isfinite(x).all()
    dt = t["q"].dtype
    for b, h in ((w.B - 1, w.H // 2), (0, w.H - 1)):
        kl = None if "kv_len" not in t else t["kv_len"][b:b + 1]
        g = ref.attn_bwd(t["q"][b:b + 1, h:h + 1], t["k"][b:b + 1, h:h + 1],
                         t["v"][b:b + 1, h:h + 1], t["dout"][b:b + 1, h:h + 1], w.scale,
                         w.causal, kl, t.get("block_mask"), rows_per_task=256)
        check(f"dQ[{b},{h}]", dq[b, h], g[0][0, 0], TOL_GRAD, dt)
        check(f"dK[{b},{h}]", dk[b, h], g[1][0, 0], TOL_GRAD, dt)
        check(f"dV[{b},{h}]", dv[b, h], g[2][0, 0], TOL_GRAD, dt)


@pytest.mark.parametrize("name", FULL_SIZE)
def test_bwd_full_size_every_head_sampled(name):
    """Full-size workload, same launches as the benchmark; dQ at sampled
    query rows and dK, dV at sampled key rows of EVERY head (tile edges and
    seeded random rows) against the oracle."""
    w = inputs.WORKLOADS[name]
    t = inputs.make_workload(w, with_dout=True)
    dq, dk, dv = run_bwd(t, w.scale, w.causal, t.get("kv_len"), t.get("block_mask"))
    worst = check_bwd_every_head(t, w, dq, dk, dv)
    print(f"\n{name}: max |d grad| over sampled rows of every head: "
          + ", ".join(f"{k} {v:.4g}" for k, v in worst.items()))


@pytest.mark.parametrize("dt,causal", [("bf16", True), ("f16", False)])
def test_bwd_three_phases_equal_fa_bwd(dt, causal):
    """fa_bwd_prepare, fa_bwd_main and fa_bwd_finish called one by one give
    what fa_bwd gives: dK and dV bitwise, dQ (fp32 atomics in no fixed
    order) to one 16-bit ulp."""
    import exact_io_aware_108_b300 as fa
    from tests.tolerance import half_ulp
    t = inputs.make_qkv(2, 3, 600, 128, dt, seed=44, qk_mult=2.0)
    q, k, v, do = (t[n].cuda() for n in ("q", "k", "v", "dout"))
    scale = 1.0 / math.sqrt(128)
    o, lse, res = fa.attention_forward(q, k, v, scale, causal=causal, return_residual=True)
    ws = torch.empty(fa.fa_bwd_workspace_size(2, 3, 600, 128), dtype=torch.uint8, device="cuda")
    g1 = [torch.empty_like(q) for _ in range(3)]
    fa.fa_bwd(q, k, v, o, lse, do, *g1, scale, causal, None, res, ws)
    g2 = [torch.full_like(q, float("nan")) for _ in range(3)]
    fa.fa_bwd_prepare(q, v, o, res, lse, do, ws)
    fa.fa_bwd_main(q, k, v, do, g2[1], g2[2], scale, causal, workspace=ws)
    fa.fa_bwd_finish(g2[0], ws)
    torch.cuda.synchronize()
    assert fa.fa_get_device_error() == 0
    assert torch.equal(g1[1], g2[1]) and torch.equal(g1[2], g2[2])
    a_, b_ = g1[0].cpu().double().numpy(), g2[0].cpu().double().numpy()
    assert np.all(np.abs(a_ - b_) <= 2 * half_ulp(np.maximum(np.abs(a_), np.abs(b_)), q.dtype) + 1e-4)
