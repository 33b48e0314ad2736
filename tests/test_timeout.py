"""The failure path of the kernels' pipeline waits, exercised without any
fault: with the load-issuing threads switched off (fa_debug_starve_pipelines)
and a short wait limit, every CTA's first wait can only run out. The kernels
must then stop on their own, fa_get_device_error must report FA_ERR_TIMEOUT
and clear the flag, and the next normal calls must give correct results on
the same CUDA context."""
import math

import pytest
import torch

from exact_io_aware_108_b300 import inputs
from oracle import ref
from tests.tolerance import TOL_GRAD, TOL_LSE, TOL_O, check

pytestmark = pytest.mark.gpu

FA_ERR_TIMEOUT = 4


def _starved(fn):
    import exact_io_aware_108_b300 as fa
    assert fa.fa_get_device_error() == 0
    assert fa.fa_set_wait_limit_ns(2_000_000) == 0  # 2 ms
    assert fa.fa_debug_starve_pipelines(True) == 0
    try:
        out = fn()
        status = fa.fa_get_device_error()
        message = fa.fa_last_error_message()
    finally:
        assert fa.fa_debug_starve_pipelines(False) == 0
        assert fa.fa_set_wait_limit_ns(0) == 0
    assert status == FA_ERR_TIMEOUT, fa.fa_status_str(status)
    assert "timed out" in message
    assert fa.fa_get_device_error() == 0  # the flag was cleared
    return out


@pytest.mark.parametrize("B,H,N,d,causal", [
    (1, 8, 256, 64, False),     # one query tile per CTA (short sequences)
    (2, 16, 4096, 128, True),   # two query tiles per CTA
])
def test_forward_wait_runs_out_then_recovers(B, H, N, d, causal):
    import exact_io_aware_108_b300 as fa
    t = inputs.make_qkv(B, H, N, d, "bf16", seed=41, with_dout=False)
    q, k, v = (x.cuda() for x in (t["q"], t["k"], t["v"]))
    scale = 1.0 / math.sqrt(d)
    o, lse = _starved(lambda: fa.attention_forward(q, k, v, scale, causal=causal))
    # a stopped CTA writes zeros and -inf instead of leaving garbage
    assert torch.all(o == 0) and torch.all(torch.isneginf(lse))
    o, lse = fa.attention_forward(q, k, v, scale, causal=causal)
    assert fa.fa_get_device_error() == 0
    rows = list(range(0, N, max(1, N // 64))) + [N - 1]
    for h in (0, H - 1):
        b = B - 1
        o_ref, lse_ref = ref.attn_fwd_rows(t["q"][b, h], t["k"][b, h], t["v"][b, h], scale, rows, causal)
        check("O", o[b, h, rows].cpu(), o_ref, TOL_O, q.dtype)
        check("LSE", lse[b, h, rows].cpu(), lse_ref, TOL_LSE, torch.float32)


@pytest.mark.parametrize("B,H,N,d", [
    (1, 2, 384, 128),    # fewer key tiles than SMs: one work item per CTA
    (2, 8, 2048, 128),   # more key tiles than SMs: CTAs keep taking items after the stop
])
def test_backward_wait_runs_out_then_recovers(B, H, N, d):
    import exact_io_aware_108_b300 as fa
    t = inputs.make_qkv(B, H, N, d, "bf16", seed=42, qk_mult=2.0)
    q, k, v, do = (x.cuda() for x in (t["q"], t["k"], t["v"], t["dout"]))
    scale = 1.0 / math.sqrt(d)
    o, lse, res = fa.attention_forward(q, k, v, scale, causal=True, return_residual=True)
    assert fa.fa_get_device_error() == 0
    dq, dk, dv = _starved(lambda: fa.attention_backward(q, k, v, o, lse, do, scale, causal=True,
                                                        o_res=res))
    assert torch.all(dk == 0) and torch.all(dv == 0)
    dq, dk, dv = fa.attention_backward(q, k, v, o, lse, do, scale, causal=True, o_res=res)
    assert fa.fa_get_device_error() == 0
    if N > 512:  # the recovery is checked against the oracle on the small case
        assert torch.isfinite(dk).all() and torch.isfinite(dv).all() and bool((dk != 0).any())
        return
    g = ref.attn_bwd(t["q"], t["k"], t["v"], t["dout"], scale, True, rows_per_task=64)
    check("dQ", dq.cpu(), g[0], TOL_GRAD, q.dtype)
    check("dK", dk.cpu(), g[1], TOL_GRAD, q.dtype)
    check("dV", dv.cpu(), g[2], TOL_GRAD, q.dtype)


def test_decode_wait_runs_out_then_recovers():
    import exact_io_aware_108_b300 as fa
    w = inputs.Workload("decode_timeout", 2, 8, 512, 128, "bf16", kv_len_range=(200, 512), hkv=2,
                        nq=1, page_size=16, backward=False, num_splits=1)
    t = {k: (x.cuda() if torch.is_tensor(x) else x) for k, x in inputs.make_workload(w).items()}
    run = lambda: fa.attention_decode_paged(t["q"], t["k_cache"], t["v_cache"], t["block_table"],
                                            t["seq_len"], w.scale, num_splits=1)
    _starved(run)
    o, lse = run()
    assert fa.fa_get_device_error() == 0
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
