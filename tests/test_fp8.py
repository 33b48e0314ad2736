"""8-bit forward: the CUDA path vs the fp64 oracle on the dequantised inputs.

The oracle computes exact attention on the real values q_descale * q etc.
(exact in fp64), so input quantisation is not part of the comparison. What
remains is the kernel's own rounding. Scores are products of e4m3 values
accumulated in fp32, so the LSE keeps the 1e-3 bar of the 16-bit forward.
Each probability is rounded to e4m3 (after scaling by 2^8) before the P V
product, which moves every element of O. Two bounds on that error follow from
the e4m3 format (3 fraction bits; spacing 2^-9 below the smallest normal,
2^-6):

* per element, the rounding of p' = 2^8 p moves it by at most
  max(2^-4 p', 2^-10), so |dO_ic| <= sum_j max(2^-4 p_j, 2^-18) |v_jc|
  <= 2^-4 O^abs_ic + 2^-18 sum_j |v_jc| over kept keys, where O^abs is
  attention with |V| (the oracle run on |v|); plus half a bf16 ulp of the
  output;
* rounding to nearest leaves an error with variance at most spacing^2 / 12,
  so sigma_ic^2 <= (2^-6 sum_j p_j^2 v_jc^2 + 2^-34 sum_j v_jc^2) / 12. The
  sum of p_j^2 v_jc^2 is attention at twice the scale with V^2, times
  e^(LSE(2 scale) - 2 LSE) (softmax at 2s is p^2 / sum p^2), again from the
  oracle. The rms error over a head must stay within twice the rms of sigma
  (plus the output rounding): errors of a wrong layout of P, a dropped tile
  or a wrong factor are far larger.

A uniform softmax is exact in e4m3 (q = 0: p' = 2^8 for every kept key), so
there O equals the mean of the kept V rows to fp32 accuracy; those cases pin
masks, tile walk and the dequantisation factors tightly.
"""
import math

import numpy as np
import pytest
import torch

from exact_io_aware_108_b300 import inputs
from oracle import ref
from tests.tolerance import TOL_LSE, check, half_ulp

pytestmark = pytest.mark.gpu


def _run(t, scale, causal, kv_len=None):
    import exact_io_aware_108_b300 as fa
    q, k, v = (t[n].cuda() for n in ("q", "k", "v"))
    kl = None if kv_len is None else kv_len.to(torch.int32).cuda()
    o, lse = fa.attention_forward_fp8(q, k, v, t["q_descale"], t["k_descale"], t["v_descale"], scale,
                                      causal=causal, kv_len=kl)
    torch.cuda.synchronize()
    assert fa.fa_get_device_error() == 0
    assert o.dtype == torch.bfloat16
    return o.cpu(), lse.cpu()


def _real(t, group):
    q = inputs.dequant(t["q"], t["q_descale"])
    k = inputs.dequant(t["k"], t["k_descale"]).repeat_interleave(group, dim=1)
    v = inputs.dequant(t["v"], t["v_descale"]).repeat_interleave(group, dim=1)
    return q, k, v


def _kept_sum(x, causal, kv_len):
    """sum over the kept keys j of x[..., j, :] for every query row i."""
    B, H, N, d = x.shape
    xs = x.numpy()
    out = np.empty_like(xs)
    for b in range(B):
        kl = N if kv_len is None else max(0, min(N, int(kv_len[b])))
        xm = xs[b].copy()
        xm[:, kl:, :] = 0.0
        out[b] = np.cumsum(xm, axis=1) if causal else np.broadcast_to(xm.sum(axis=1, keepdims=True), xm.shape)
    return out


def _check_fp8(o, lse, t, H, Hkv, scale, causal, kv_len=None):
    q, k, v = _real(t, H // Hkv)
    o_ref, lse_ref = ref.attn_fwd(q, k, v, scale, causal, kv_len)
    check("LSE", lse, lse_ref, TOL_LSE, torch.float32)
    o_ref = np.asarray(o_ref)
    og = o.double().numpy()
    fin = np.isfinite(np.asarray(lse_ref))[..., None] & np.ones_like(og, dtype=bool)
    assert np.all(og[~fin] == 0.0)
    err = np.abs(og - o_ref)
    # worst-case bound
    o_abs, _ = ref.attn_fwd(q, k, v.abs(), scale, causal, kv_len)
    bound = (2.0 ** -4 * np.asarray(o_abs) + 2.0 ** -18 * _kept_sum(v.abs(), causal, kv_len)
             + half_ulp(np.maximum(np.abs(og), np.abs(o_ref)), torch.bfloat16) + 1e-5)
    over = err > bound
    assert not np.any(over), (f"{int(over.sum())} elements beyond the rounding bound; worst "
                              f"err {err[over].max():.3e} vs bound {bound[over].min():.3e}")
    # statistical bound
    o2, lse2 = ref.attn_fwd(q, k, v * v, 2.0 * scale, causal, kv_len)
    with np.errstate(invalid="ignore", over="ignore"):
        w = np.exp(np.asarray(lse2) - 2.0 * np.asarray(lse_ref))
    w = np.where(np.isfinite(w), w, 0.0)[..., None]
    sp2v2 = np.asarray(o2) * w
    var = (2.0 ** -6 * sp2v2 + 2.0 ** -34 * _kept_sum(v * v, causal, kv_len)) / 12.0
    var_out = (2.0 * half_ulp(np.abs(o_ref), torch.bfloat16)) ** 2 / 12.0
    rms_err = math.sqrt(float(np.mean(err[fin] ** 2)))
    rms_sigma = math.sqrt(float(np.mean((var + var_out)[fin])))
    assert rms_err <= 2.0 * rms_sigma + 1e-6, f"rms error {rms_err:.3e} vs model {rms_sigma:.3e}"
    return rms_err, rms_sigma


CASES = [
    # B, H, Hkv, N, causal
    (1, 2, 2, 1000, False),
    (2, 2, 1, 700, True),
    (1, 4, 2, 384, True),
    (2, 1, 1, 129, False),
]


@pytest.mark.parametrize("B,H,Hkv,N,causal", CASES)
def test_fp8_matches_oracle_within_rounding_model(B, H, Hkv, N, causal):
    t = inputs.make_qkv_fp8(B, H, N, 128, seed=N + H, hkv=Hkv)
    o, lse = _run(t, 1.0 / math.sqrt(128), causal)
    _check_fp8(o, lse, t, H, Hkv, 1.0 / math.sqrt(128), causal)


def test_fp8_key_padding():
    t = inputs.make_qkv_fp8(4, 2, 520, 128, seed=9)
    kv_len = torch.tensor([0, 1, 128, 333], dtype=torch.int32)
    o, lse = _run(t, 0.1, False, kv_len)
    _check_fp8(o, lse, t, 2, 2, 0.1, False, kv_len)


@pytest.mark.parametrize("causal,kv", [(False, None), (True, None), (False, [77, 400]), (True, [300, 5])])
def test_fp8_uniform_softmax_is_exact(causal, kv):
    """q = 0: every kept key has p' = 2^8 exactly, so O is the mean of the
    kept V rows (times v_descale) up to fp32 sums and the bf16 output."""
    t = inputs.make_qkv_fp8(2, 4, 400, 128, seed=4, hkv=2)
    t["q"] = torch.zeros_like(t["q"])
    kv_len = None if kv is None else torch.tensor(kv, dtype=torch.int32)
    o, lse = _run(t, 0.125, causal, kv_len)
    q, k, v = _real(t, 2)
    o_ref, lse_ref = ref.attn_fwd(q, k, v, 0.125, causal, kv_len)
    check("O", o, o_ref, 1e-4, torch.bfloat16)
    check("LSE", lse, lse_ref, 1e-5, torch.float32)


def test_fp8_descale_factors_apply():
    """The scores use q_descale * k_descale and O uses v_descale: doubling
    q_descale while halving k_descale changes nothing, doubling v_descale
    doubles O exactly (powers of two) and leaves LSE alone."""
    t = inputs.make_qkv_fp8(1, 2, 256, 128, seed=12)
    t2 = dict(t, q_descale=2 * t["q_descale"], k_descale=t["k_descale"] / 2, v_descale=2 * t["v_descale"])
    o1, l1 = _run(t, 0.09, True)
    o2, l2 = _run(t2, 0.09, True)
    assert torch.equal(l1, l2)
    assert torch.equal(o2, 2 * o1)


def test_fp8_full_size_whole_head():
    """The benchmark's 8-bit workload in the benchmark's launch: every O and
    LSE element of one head against the oracle and the rounding model."""
    w = inputs.WORKLOADS["fp8_b4_h16_n8192_d128_e4m3_causal"]
    t = inputs.make_workload(w)
    o, lse = _run(t, w.scale, w.causal)
    b, h = w.B - 1, w.H - 1
    one = {"q": t["q"][b:b + 1, h:h + 1], "k": t["k"][b:b + 1, h:h + 1], "v": t["v"][b:b + 1, h:h + 1],
           "q_descale": t["q_descale"], "k_descale": t["k_descale"], "v_descale": t["v_descale"]}
    _check_fp8(o[b:b + 1, h:h + 1], lse[b:b + 1, h:h + 1], one, 1, 1, w.scale, w.causal)
