"""Split-KV forward: the CUDA path vs the fp64 oracle.

The key tiles of each query tile are shared by S CTAs; each writes its
share's normalised O and LSE, and a merge kernel combines the shares with
the softmax merge identity. The oracle computes plain attention over all
keys: the merge is exact up to fp32 rounding, so the results must meet the
same tolerances as the unsplit forward. Cases cover uneven shares, shares
with no key tile at all (S above the row's tile count, the first rows of a
causal grid), key padding down to zero keys, grouped-query heads and both
head dims."""
import math

import numpy as np
import pytest
import torch

from exact_io_aware_108_b300 import inputs
from oracle import ref
from tests.tolerance import TOL_LSE, TOL_O, check, check_residual

pytestmark = pytest.mark.gpu

CASES = [
    # B, H, Hkv, N, d, dtype, causal, num_splits
    (1, 2, 2, 1000, 128, "bf16", False, 3),   # 8 key tiles in shares of 2 and 3, ragged tail
    (2, 2, 1, 640, 64, "f16", True, 2),       # causal: query tile 0 leaves share 0 empty
    (1, 3, 3, 300, 128, "bf16", True, 7),     # 3 key tiles, 7 shares: most shares empty
    (1, 4, 2, 1536, 64, "bf16", False, 5),    # grouped-query heads
    (1, 1, 1, 2048, 128, "f16", False, 0),    # the library's choice of S
]


def _splitkv(q, k, v, scale, causal, num_splits, kv_len=None, residual=False):
    import exact_io_aware_108_b300 as fa
    out = fa.attention_forward(q, k, v, scale, causal=causal, kv_len=kv_len, return_residual=residual,
                               num_splits=num_splits)
    torch.cuda.synchronize()
    assert fa.fa_get_device_error() == 0
    return out


def _oracle(t, H, Hkv, scale, causal, kv_len=None):
    g = H // Hkv
    kr = t["k"].repeat_interleave(g, dim=1)
    vr = t["v"].repeat_interleave(g, dim=1)
    return ref.attn_fwd(t["q"], kr, vr, scale, causal, kv_len)


@pytest.mark.parametrize("B,H,Hkv,N,d,dt,causal,S", CASES)
def test_splitkv_matches_oracle(B, H, Hkv, N, d, dt, causal, S):
    import exact_io_aware_108_b300 as fa
    t = inputs.make_qkv(B, H, N, d, dt, seed=N + S, hkv=Hkv, with_dout=False)
    q, k, v = (t[n].cuda() for n in ("q", "k", "v"))
    scale = 1.0 / math.sqrt(d)
    assert fa.fa_fwd_splitkv_num_splits(B, H, N, d, causal, S) >= 1
    o, lse = _splitkv(q, k, v, scale, causal, S)
    o_ref, lse_ref = _oracle(t, H, Hkv, scale, causal)
    check("O", o.cpu(), o_ref, TOL_O, q.dtype)
    check("LSE", lse.cpu(), lse_ref, TOL_LSE, torch.float32)


@pytest.mark.parametrize("d,dt", [(128, "bf16"), (64, "bf16")])
def test_splitkv_key_padding_down_to_no_keys(d, dt):
    """kv_len 0 (every share empty: O = 0, LSE = -inf), 1, a tile boundary
    and a ragged length; sharp softmax. d = 64 runs the shares two CTAs per
    SM, d = 128 one."""
    t = inputs.make_qkv(4, 2, 700, d, dt, seed=5, qk_mult=2.0, with_dout=False)
    kv_len = torch.tensor([0, 1, 256, 613], dtype=torch.int32)
    q, k, v = (t[n].cuda() for n in ("q", "k", "v"))
    scale = 1.0 / math.sqrt(d)
    o, lse = _splitkv(q, k, v, scale, False, 4, kv_len=kv_len.cuda())
    o_ref, lse_ref = ref.attn_fwd(t["q"], t["k"], t["v"], scale, False, kv_len)
    check("O", o.cpu(), o_ref, TOL_O, q.dtype)
    check("LSE", lse.cpu(), lse_ref, TOL_LSE, torch.float32)
    assert torch.all(o[0] == 0) and torch.all(torch.isneginf(lse[0]))


@pytest.mark.parametrize("d,dt", [(128, "bf16"), (64, "f16")])
def test_splitkv_residual_path_is_accurate(d, dt):
    """With o_res requested the merge rounds the fp32 result once and writes
    its rounding residual: O + o_res is within u |O|_abs of the exact O (u
    the unit roundoff of the 16-bit probabilities), as on the unsplit path."""
    t = inputs.make_qkv(2, 2, 512, d, dt, seed=21, qk_mult=2.0, with_dout=False)
    q, k, v = (t[n].cuda() for n in ("q", "k", "v"))
    scale = 1.0 / math.sqrt(d)
    o, lse, o_res = _splitkv(q, k, v, scale, True, 3, residual=True)
    o_ref, lse_ref = ref.attn_fwd(t["q"], t["k"], t["v"], scale, True)
    check("O", o.cpu(), o_ref, TOL_O, q.dtype)
    check("LSE", lse.cpu(), lse_ref, TOL_LSE, torch.float32)
    o_abs, _ = ref.attn_fwd(t["q"], t["k"], t["v"].abs(), scale, True)
    check_residual("O + o_res", o.cpu(), o_res.cpu(), o_ref, o_abs, q.dtype)


def test_splitkv_one_share_is_the_unsplit_forward():
    """num_splits = 1 takes the unsplit forward itself: bitwise equal."""
    import exact_io_aware_108_b300 as fa
    t = inputs.make_qkv(2, 4, 384, 128, "bf16", seed=3, hkv=2, with_dout=False)
    q, k, v = (t[n].cuda() for n in ("q", "k", "v"))
    scale = 1.0 / math.sqrt(128)
    assert fa.fa_fwd_splitkv_workspace_size(2, 4, 384, 128, True, 1) == 0
    o1, lse1 = _splitkv(q, k, v, scale, True, 1)
    o2, lse2 = fa.attention_forward(q, k, v, scale, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(lse1, lse2)


def test_splitkv_results_do_not_depend_on_launch_order():
    """Two runs with the same S are bitwise equal (no atomics in the merge)."""
    t = inputs.make_qkv(1, 2, 900, 64, "bf16", seed=8, with_dout=False)
    q, k, v = (t[n].cuda() for n in ("q", "k", "v"))
    a = _splitkv(q, k, v, 0.125, False, 4)
    b = _splitkv(q, k, v, 0.125, False, 4)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_splitkv_full_size_whole_head():
    """The benchmark-sized split workload in the benchmark's launch (the
    library's choice of S): every O and LSE element of the head."""
    import exact_io_aware_108_b300 as fa
    w = inputs.WORKLOADS["splitkv_b1_h1_n8192_d128_bf16"]
    assert fa.fa_fwd_splitkv_num_splits(w.B, w.H, w.N, w.d, w.causal, w.num_splits) > 1
    t = inputs.make_workload(w, with_dout=False)
    q, k, v = (t[n].cuda() for n in ("q", "k", "v"))
    o, lse = _splitkv(q, k, v, w.scale, w.causal, w.num_splits)
    o_ref, lse_ref = ref.attn_fwd(t["q"], t["k"], t["v"], w.scale, w.causal)
    check("O", o.cpu(), o_ref, TOL_O, q.dtype)
    check("LSE", lse.cpu(), lse_ref, TOL_LSE, torch.float32)
