"""Forward parity: the CUDA path (through the C ABI) vs the fp64 oracle."""
import math

import numpy as np
import pytest
import torch

from exact_io_aware_108_b300 import inputs
from oracle import ref
from tests.tolerance import TOL_LSE, TOL_O, check, check_residual

pytestmark = pytest.mark.gpu


def _dev(t):
    return t.cuda()


def run_fwd(q, k, v, scale, causal=False, kv_len=None, block_mask=None):
    import exact_io_aware_108_b300 as fa
    qd, kd, vd = _dev(q), _dev(k), _dev(v)
    kl = None if kv_len is None else kv_len.to(torch.int32).cuda()
    bm = None if block_mask is None else block_mask.to(torch.uint8).cuda()
    o, lse = fa.attention_forward(qd, kd, vd, scale, causal=causal, kv_len=kl, block_mask=bm)
    torch.cuda.synchronize()
    assert fa.fa_get_device_error() == 0
    return o.cpu(), lse.cpu()


def compare_full(q, k, v, scale, causal=False, kv_len=None, block_mask=None):
    o, lse = run_fwd(q, k, v, scale, causal, kv_len, block_mask)
    o_ref, lse_ref = ref.attn_fwd(q, k, v, scale, causal, kv_len, block_mask)
    check("O", o, o_ref, TOL_O, q.dtype)
    check("LSE", lse, lse_ref, TOL_LSE, torch.float32)
    return o, lse


SHAPES = [
    # B, H, N, d, dtype, causal
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
def test_fwd_matches_oracle(B, H, N, d, dt, causal):
    t = inputs.make_qkv(B, H, N, d, dt, seed=N + d, with_dout=False)
    compare_full(t["q"], t["k"], t["v"], 1.0 / math.sqrt(d), causal)


@pytest.mark.parametrize("d,dt", [(64, "bf16"), (128, "f16")])
def test_fwd_sharp_softmax(d, dt):
    """Logit std ~4 (Q, K times 2): the running max moves often."""
    t = inputs.make_qkv(2, 2, 384, d, dt, seed=3, qk_mult=2.0, with_dout=False)
    compare_full(t["q"], t["k"], t["v"], 1.0 / math.sqrt(d), causal=True)


def test_fwd_config_small_workload():
    """B=1, H=2, N=256, d=64, fp16, seed 0, non-causal: every output."""
    w = inputs.WORKLOADS["fwd_b1_h2_n256_d64_f16"]
    t = inputs.make_workload(w)
    compare_full(t["q"], t["k"], t["v"], w.scale)


@pytest.mark.parametrize("causal", [False, True])
def test_fwd_kv_len_edges(causal):
    N, d = 300, 64
    t = inputs.make_qkv(8, 2, N, d, "f16", seed=11, with_dout=False)
    kv_len = torch.tensor([1, 127, 128, 129, 300, 0, 1000, 255], dtype=torch.int32)
    o, lse = compare_full(t["q"], t["k"], t["v"], 0.125, causal, kv_len=kv_len)
    # kv_len 0: every key masked -> O = 0, LSE = -inf
    assert torch.all(o[5] == 0) and torch.all(torch.isneginf(lse[5]))


def test_fwd_blocksparse_matches_oracle():
    N, d = 640, 64
    t = inputs.make_qkv(2, 2, N, d, "f16", seed=5, with_dout=False)
    bm = inputs.make_block_mask(N, 0.4, seed=7)
    bm[3, :] = 0  # one query tile keeps nothing: O = 0, LSE = -inf
    o, lse = compare_full(t["q"], t["k"], t["v"], 0.125, block_mask=bm)
    assert torch.all(o[:, :, 384:512] == 0) and torch.all(torch.isneginf(lse[:, :, 384:512]))


def test_fwd_blocksparse_all_ones_is_dense_bitwise():
    N, d = 512, 128
    t = inputs.make_qkv(1, 2, N, d, "bf16", seed=6, with_dout=False)
    ones = torch.ones((4, 4), dtype=torch.uint8)
    o1, l1 = run_fwd(t["q"], t["k"], t["v"], 0.09, block_mask=ones)
    o2, l2 = run_fwd(t["q"], t["k"], t["v"], 0.09)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_fwd_blocksparse_skipped_tiles_are_not_read():
    """Changing K/V inside a masked key tile leaves the rows that skip it
    bit-for-bit unchanged."""
    N, d = 512, 64
    t = inputs.make_qkv(1, 1, N, d, "f16", seed=8, with_dout=False)
    bm = torch.ones((4, 4), dtype=torch.uint8)
    bm[0, 2] = 0
    bm[3, 2] = 0
    o1, l1 = run_fwd(t["q"], t["k"], t["v"], 0.125, block_mask=bm)
    k2, v2 = t["k"].clone(), t["v"].clone()
    k2[:, :, 256:384] = 7.0
    v2[:, :, 256:384] = -3.0
    o2, l2 = run_fwd(t["q"], k2, v2, 0.125, block_mask=bm)
    for rows in (slice(0, 128), slice(384, 512)):
        assert torch.equal(o1[:, :, rows], o2[:, :, rows])
        assert torch.equal(l1[:, :, rows], l2[:, :, rows])
    assert not torch.equal(o1[:, :, 128:256], o2[:, :, 128:256])


def test_fwd_deterministic():
    t = inputs.make_qkv(2, 2, 384, 128, "bf16", seed=9, with_dout=False)
    a = run_fwd(t["q"], t["k"], t["v"], 0.1, True)
    b = run_fwd(t["q"], t["k"], t["v"], 0.1, True)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_fwd_on_side_stream():
    import exact_io_aware_108_b300 as fa
    t = inputs.make_qkv(1, 2, 256, 64, "f16", seed=10, with_dout=False)
    s = torch.cuda.Stream()
    q, k, v = (x.cuda() for x in (t["q"], t["k"], t["v"]))
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        o, lse = fa.attention_forward(q, k, v, 0.125, stream=s)
    s.synchronize()
    o_ref, lse_ref = ref.attn_fwd(t["q"], t["k"], t["v"], 0.125)
    check("O", o.cpu(), o_ref, TOL_O, q.dtype)
    check("LSE", lse.cpu(), lse_ref, TOL_LSE, torch.float32)


# ----------------------------------------------------- full-size workloads

def _sample_rows(N, rng, n=48):
    edges = [0, 1, 127, 128, 129, N // 2, N - 129, N - 128, N - 1]
    rows = set(r for r in edges if 0 <= r < N)
    rows.update(rng.integers(0, N, size=n - len(rows)).tolist())
    return sorted(rows)


@pytest.mark.parametrize("name", [
    "bert_b16_h16_n512_d64_f16_kvlen",
    "gpt2_b8_h12_n1024_d64_bf16_causal",
    "long_b8_h16_n4096_d128_bf16_causal",
    "long_b4_h16_n8192_d128_bf16_causal",
    "long_b2_h16_n16384_d128_bf16_causal",
    "blocksparse_b2_h8_n16384_d64_f16",
])
def test_fwd_full_size_sampled(name):
    """Full-size workload, same launch as the benchmark; sampled rows of a few
    heads are checked against the oracle one by one, and one whole head."""
    w = inputs.WORKLOADS[name]
    t = inputs.make_workload(w, with_dout=False)
    o, lse = run_fwd(t["q"], t["k"], t["v"], w.scale, w.causal, t.get("kv_len"),
                     t.get("block_mask"))
    assert torch.isfinite(o).all()
    rng = np.random.default_rng(0)
    heads = [(0, 0), (w.B - 1, w.H - 1), (w.B // 2, w.H // 3)]
    for b, h in heads:
        rows = _sample_rows(w.N, rng)
        klb = None if "kv_len" not in t else int(t["kv_len"][b])
        o_ref, lse_ref = ref.attn_fwd_rows(t["q"][b, h], t["k"][b, h], t["v"][b, h], w.scale, rows,
                                           w.causal, klb, t.get("block_mask"))
        check(f"O[{b},{h}]", o[b, h, rows], o_ref, TOL_O, t["q"].dtype)
        check(f"LSE[{b},{h}]", lse[b, h, rows], lse_ref, TOL_LSE, torch.float32)
    b, h = w.B - 1, w.H - 1
    kl = None if "kv_len" not in t else t["kv_len"][b:b + 1]
    o_ref, lse_ref = ref.attn_fwd(t["q"][b:b + 1, h:h + 1], t["k"][b:b + 1, h:h + 1],
                                  t["v"][b:b + 1, h:h + 1], w.scale, w.causal, kl,
                                  t.get("block_mask"))
    check(f"O[{b},{h}] whole head", o[b, h], o_ref[0, 0], TOL_O, t["q"].dtype)
    check(f"LSE[{b},{h}] whole head", lse[b, h], lse_ref[0, 0], TOL_LSE, torch.float32)


@pytest.mark.parametrize("B,H,N,d,dt,causal", [
    (1, 1, 3000, 128, "bf16", True),    # 24 query tiles, 12 pairs: a grid of fewer CTAs than SMs
    (1, 2, 4500, 64, "f16", False),     # 36 query tiles with a ragged tail
])
def test_fwd_few_heads_long_sequence(B, H, N, d, dt, causal):
    """Few heads of a long sequence run the one-tile-per-CTA forward (the
    two-tile grid would leave SMs idle): every element against the oracle,
    with and without O's residual."""
    import exact_io_aware_108_b300 as fa
    t = inputs.make_qkv(B, H, N, d, dt, seed=N + H, with_dout=False)
    q, k, v = (t[n].cuda() for n in ("q", "k", "v"))
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.attention_forward(q, k, v, scale, causal=causal)
    o2, lse2, o_res = fa.attention_forward(q, k, v, scale, causal=causal, return_residual=True)
    torch.cuda.synchronize()
    assert fa.fa_get_device_error() == 0
    o_ref, lse_ref = ref.attn_fwd(t["q"], t["k"], t["v"], scale, causal)
    check("O", o.cpu(), o_ref, TOL_O, q.dtype)
    check("LSE", lse.cpu(), lse_ref, TOL_LSE, torch.float32)
    check("O (residual path)", o2.cpu(), o_ref, TOL_O, q.dtype)
    o_abs, _ = ref.attn_fwd(t["q"], t["k"], t["v"].abs(), scale, causal)
    check_residual("O + o_res", o2.cpu(), o_res.cpu(), o_ref, o_abs, q.dtype)


@pytest.mark.parametrize("d,dt", [(128, "bf16"), (64, "f16")])
def test_fwd_residual_path_is_accurate(d, dt):
    """With o_res requested, O itself still passes the output tolerance and
    O + o_res is the fp32 result of the P V product: within u |O|_abs of the
    exact O (u the unit roundoff of the 16-bit probabilities), the accuracy
    the backward's D = rowsum(dO * (O + o_res)) relies on. Sharp softmax."""
    import exact_io_aware_108_b300 as fa
    t = inputs.make_qkv(2, 2, 512, d, dt, seed=21, qk_mult=2.0, with_dout=False)
    q, k, v = (t[n].cuda() for n in ("q", "k", "v"))
    scale = 1.0 / math.sqrt(d)
    o, lse, o_res = fa.attention_forward(q, k, v, scale, causal=True, return_residual=True)
    o_plain, lse_plain = fa.attention_forward(q, k, v, scale, causal=True)
    torch.cuda.synchronize()
    assert fa.fa_get_device_error() == 0
    o_ref, lse_ref = ref.attn_fwd(t["q"], t["k"], t["v"], scale, True)
    o_abs, _ = ref.attn_fwd(t["q"], t["k"], t["v"].abs(), scale, True)
    check("O", o.cpu(), o_ref, TOL_O, q.dtype)
    check("LSE", lse.cpu(), lse_ref, TOL_LSE, torch.float32)
    check_residual("O + o_res", o.cpu(), o_res.cpu(), o_ref, o_abs, q.dtype)
    # the residual is an extra output of the same computation
    assert torch.equal(o.cpu(), o_plain.cpu()) and torch.equal(lse.cpu(), lse_plain.cpu())
