"""Sampled backward checks over every head of a full-size workload.

For each head the oracle's sampled backward (``oracle.ref.attn_bwd_sampled``)
computes dQ at a set of query rows and dK, dV at a set of key rows exactly in
fp64; the rows always include the edges of the first, a middle and the last
128-row tile, plus seeded random rows.
"""
import numpy as np
import torch

from oracle import ref
from tests.tolerance import TOL_GRAD, check


def sample_rows(N, rng, n_random=8):
    edges = {0, 1, 127, 128, 129, N // 2 - 1, N // 2, N - 129, N - 128, N - 2, N - 1}
    rows = {r for r in edges if 0 <= r < N}
    rows.update(int(x) for x in rng.integers(0, N, size=n_random))
    return np.array(sorted(rows), dtype=np.int64)


def check_bwd_every_head(t, w, dq, dk, dv, seed=0, report=None):
    """dq [B,H,N,d], dk, dv [B,Hkv,N,d] (CPU tensors) of workload w against
    the oracle at sampled rows of every head. With grouped-query heads the
    dK, dV rows of a key/value head are the sums over its query heads."""
    rng = np.random.default_rng(seed)
    dt = t["q"].dtype
    hkv = w.hkv or w.H
    g = w.H // hkv
    kl = t.get("kv_len")
    worst = {"dQ": 0.0, "dK": 0.0, "dV": 0.0}
    for b in range(w.B):
        klb = None if kl is None else int(kl[b])
        for kh in range(hkv):
            qrows = sample_rows(w.N, rng)
            krows = sample_rows(w.N, rng)
            dk_sum = 0.0
            dv_sum = 0.0
            for h in range(kh * g, (kh + 1) * g):
                gq, gk, gv, _, _ = ref.attn_bwd_sampled(
                    t["q"][b, h], t["k"][b, kh], t["v"][b, kh], t["dout"][b, h], w.scale, qrows,
                    krows, w.causal, klb, t.get("block_mask"))
                a, _ = check(f"dQ[{b},{h}] rows", dq[b, h, qrows], gq, TOL_GRAD, dt)
                worst["dQ"] = max(worst["dQ"], a)
                dk_sum = dk_sum + gk
                dv_sum = dv_sum + gv
            a, _ = check(f"dK[{b},{kh}] rows", dk[b, kh, krows], dk_sum, TOL_GRAD, dt)
            worst["dK"] = max(worst["dK"], a)
            a, _ = check(f"dV[{b},{kh}] rows", dv[b, kh, krows], dv_sum, TOL_GRAD, dt)
            worst["dV"] = max(worst["dV"], a)
    if report is not None:
        report.update(worst)
    return worst
