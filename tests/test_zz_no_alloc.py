"""fa_bwd_noalloc: the backward for callers that may not allocate device
memory (for example code running inside another engine's execute callback,
where device memory belongs to that engine). It takes its workspace from a
fixed scratch array inside the library; these tests check it gives the same
gradients as fa_bwd with a caller-owned workspace, twice in a row (the second
call finds the first call's leftovers in the shared scratch).

This file is collected last on purpose."""
import ctypes
import math

import pytest
import torch

from exact_io_aware_108_b300 import inputs
from tests.tolerance import TOL_GRAD, check


def test_noalloc_rejects_sizes_beyond_its_scratch():
    import exact_io_aware_108_b300 as fa
    lib = fa.load_library()
    limit = fa.fa_bwd_noalloc_max_workspace()
    assert limit == 32 << 20
    # B*H*N rows of d = 128 needing more than the scratch: rejected before any launch
    B, H, N, d = 1, 64, 2048, 128
    assert fa.fa_bwd_workspace_size(B, H, N, d) > limit
    fake = 1 << 20
    st = lib.fa_bwd_noalloc(*([fake] * 9), B, H, N, d, ctypes.c_float(0.1), 0, 0, None, None,
                            None, None)
    assert st == 1
    assert "scratch" in fa.fa_last_error_message()


@pytest.mark.gpu
@pytest.mark.parametrize("causal,sparse", [(True, False), (False, True)])
def test_noalloc_matches_fa_bwd_twice(causal, sparse):
    import exact_io_aware_108_b300 as fa
    B, H, N, d = 2, 4, 640, 128
    t = inputs.make_qkv(B, H, N, d, "bf16", seed=31)
    q, k, v, do = (t[n].cuda() for n in ("q", "k", "v", "dout"))
    scale = 1.0 / math.sqrt(d)
    bm = inputs.make_block_mask(N, 0.5, seed=3).cuda() if sparse else None
    o, lse, o_res = fa.attention_forward(q, k, v, scale, causal=causal, block_mask=bm,
                                         return_residual=True)
    want = fa.attention_backward(q, k, v, o, lse, do, scale, causal=causal, block_mask=bm,
                                 o_res=o_res)
    for _ in range(2):
        dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
        fa.fa_bwd_noalloc(q, k, v, o, lse, do, dq, dk, dv, scale, causal, None, bm, o_res)
        torch.cuda.synchronize()
        assert fa.fa_get_device_error() == 0
        # dK and dV are deterministic; dQ sums key tiles with fp32 atomics
        assert torch.equal(dk, want[1]) and torch.equal(dv, want[2])
        check("dQ noalloc vs fa_bwd", dq.cpu(), want[0].double().cpu().numpy(), TOL_GRAD, q.dtype)
