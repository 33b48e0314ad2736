"""Paged-KV decode: the CUDA path vs the fp64 oracle (oracle.ref.paged_decode).

Sequences of different lengths read their keys and values through a
shuffled block table from a shared page pool; the Nq newest tokens of each
sequence attend to the cached prefix and causally to each other. Cases
cover every page size, both head dims and dtypes, grouped and multi-query
heads, more than 128 query rows per key/value head, contexts shorter than
Nq (queries without keys), split and unsplit key walks, and non-finite
garbage in the cache slots no sequence owns."""
import math

import numpy as np
import pytest
import torch

from exact_io_aware_108_b300 import inputs
from oracle import ref
from tests.tolerance import TOL_LSE, TOL_O, check

pytestmark = pytest.mark.gpu


def _decode(t, scale, num_splits=0, k_cache=None, v_cache=None):
    import exact_io_aware_108_b300 as fa
    q = t["q"].cuda()
    kc = (t["k_cache"] if k_cache is None else k_cache).cuda()
    vc = (t["v_cache"] if v_cache is None else v_cache).cuda()
    o, lse = fa.attention_decode_paged(q, kc, vc, t["block_table"].cuda(), t["seq_len"].cuda(), scale,
                                       num_splits=num_splits)
    torch.cuda.synchronize()
    assert fa.fa_get_device_error() == 0
    return o.cpu(), lse.cpu()


def _oracle(t, scale):
    return ref.paged_decode(t["q"], t["k_cache"], t["v_cache"], t["block_table"], t["seq_len"], scale,
                            t["page_size"])


CASES = [
    # B, H, Hkv, Nq, d, dtype, page_size, ctx_range, num_splits
    (3, 8, 2, 1, 128, "bf16", 16, (1, 700), 0),
    (2, 4, 4, 3, 64, "f16", 32, (100, 400), 2),
    (4, 16, 2, 5, 128, "bf16", 64, (200, 1000), 3),
    (2, 32, 1, 4, 128, "bf16", 128, (300, 600), 1),   # 128 query rows per key/value head
    (1, 40, 1, 4, 64, "f16", 16, (500, 900), 0),      # 160 rows: two query tiles
    (2, 8, 2, 2, 64, "bf16", 16, (900, 1100), 1),     # one CTA walks 8-9 tiles: the ring wraps twice
]


@pytest.mark.parametrize("B,H,Hkv,Nq,d,dt,ps,ctx,S", CASES)
def test_decode_matches_oracle(B, H, Hkv, Nq, d, dt, ps, ctx, S):
    t = inputs.make_paged_decode(B, H, Hkv, Nq, d, dt, ps, ctx, seed=B * 100 + H + ps, spare_pages=3)
    scale = 1.0 / math.sqrt(d)
    o, lse = _decode(t, scale, S)
    o_ref, lse_ref = _oracle(t, scale)
    check("O", o, o_ref, TOL_O, t["q"].dtype)
    check("LSE", lse, lse_ref, TOL_LSE, torch.float32)


def test_decode_short_contexts():
    """seq_len 0 (no keys), 1 and 2 with Nq = 3 (the first queries see
    nothing), a page boundary and a tile boundary."""
    t = inputs.make_paged_decode(6, 4, 2, 3, 128, "bf16", 16, (1, 300), seed=3)
    t["seq_len"] = torch.tensor([0, 1, 2, 16, 128, 300], dtype=torch.int32)
    for S in (1, 3):
        o, lse = _decode(t, 0.1, S)
        o_ref, lse_ref = _oracle(t, 0.1)
        check("O", o, o_ref, TOL_O, t["q"].dtype)
        check("LSE", lse, lse_ref, TOL_LSE, torch.float32)
        assert torch.all(o[0] == 0) and torch.all(torch.isneginf(lse[0]))


def test_decode_ignores_garbage_in_unowned_slots():
    """NaN in every cache slot past each sequence's length and in the spare
    pages leaves the result bitwise unchanged."""
    t = inputs.make_paged_decode(4, 8, 2, 2, 128, "bf16", 16, (50, 500), seed=5, spare_pages=4)
    kc, vc = t["k_cache"].clone(), t["v_cache"].clone()
    owned = torch.zeros(kc.shape[0], kc.shape[2], dtype=torch.bool)
    ps = t["page_size"]
    for b in range(4):
        L = int(t["seq_len"][b])
        for j in range(L):
            owned[int(t["block_table"][b, j // ps]), j % ps] = True
    unowned = ~owned[:, None, :, None]  # [page, 1, slot, 1] over [page, Hkv, slot, d]
    kc.masked_fill_(unowned, float("nan"))
    vc.masked_fill_(unowned, float("nan"))
    for S in (1, 4):
        clean = _decode(t, 0.09, S)
        dirty = _decode(t, 0.09, S, kc, vc)
        assert torch.isfinite(dirty[0]).all()
        assert torch.equal(clean[0], dirty[0]) and torch.equal(clean[1], dirty[1])


def test_decode_full_size_sampled():
    """The benchmark's decode workload in the benchmark's launch (the
    library's S): every query of four sequences (shortest, longest and two
    others) against the oracle, and all outputs finite."""
    w = inputs.WORKLOADS["decode_b32_h32_hkv8_nq1_ctx4k8k_d128_bf16_page16"]
    t = inputs.make_workload(w)
    o, lse = _decode(t, w.scale, w.num_splits)
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    sl = t["seq_len"]
    picks = sorted({int(torch.argmin(sl)), int(torch.argmax(sl)), 0, w.B // 2})
    sub = {"q": t["q"][picks], "k_cache": t["k_cache"], "v_cache": t["v_cache"],
           "block_table": t["block_table"][picks], "seq_len": sl[picks], "page_size": t["page_size"]}
    o_ref, lse_ref = _oracle(sub, w.scale)
    check("O", o[picks], o_ref, TOL_O, t["q"].dtype)
    check("LSE", lse[picks], lse_ref, TOL_LSE, torch.float32)
