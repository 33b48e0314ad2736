"""Pins of the fp64 oracle to facts fixed by the pages and by mathematics.

Each ``pin_*`` function takes a loaded oracle library (the real one, or a
deliberately broken copy in the mutation test) and raises AssertionError if
the oracle disagrees with the fact it checks. None of them re-types the
oracle's formula: each checks a closed form, an invariant, a special case,
finite differences, or an independent implementation (torch's own fp64
attention and autograd; the corrected block algorithm in tiled_numpy.py).
"""
import math

import numpy as np

from oracle import ref
from tests.tiled_numpy import tiled_attention_head

TIGHT = 1e-11


def _rng(seed):
    return np.random.default_rng(seed)


def _close(a, b, tol=TIGHT, what=""):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    fin = np.isfinite(b)
    assert np.array_equal(np.isfinite(a), fin), f"{what}: finiteness differs"
    assert np.array_equal(a[~fin], b[~fin]), f"{what}: infinities differ"
    err = np.max(np.abs(a[fin] - b[fin]), initial=0.0)
    assert err <= tol, f"{what}: max abs err {err:.3e} > {tol:.1e}"


def _mask_modes(N, blk):
    """(causal, kv_len list or None, block_mask or None) cases for B=2."""
    nb = (N + blk - 1) // blk
    bm = np.ones((nb, nb), dtype=np.uint8)
    bm[0, nb - 1] = 0
    if nb > 2:
        bm[nb - 1, 1] = 0
        bm[1, 0] = 0
    return [
        (False, None, None),
        (True, None, None),
        (False, [N - 3, 2], None),
        (False, None, bm),
        (True, [N, N - 1], bm),
    ]


# ---------------------------------------------------------------- forward pins

def pin_rows_sum_to_one(lib):
    """softmax rows sum to 1: with V = 1 every row with a kept key gets O = 1."""
    rng = _rng(1)
    B, H, N, d, blk = 2, 2, 11, 3, 4
    q = rng.standard_normal((B, H, N, d))
    k = rng.standard_normal((B, H, N, d))
    v = np.ones((B, H, N, d))
    for causal, kl, bm in _mask_modes(N, blk):
        o, lse = ref.attn_fwd(q, k, v, 0.7, causal, kl, bm, blk, lib=lib)
        live = np.isfinite(lse)
        assert live.all(), "every row here has a kept key"
        _close(o, np.ones_like(o), what=f"V=1 causal={causal}")


def pin_q_zero_mean_of_values(lib):
    """Q = 0: all kept scores are 0, so O_i is the mean of the kept V rows and
    LSE_i = ln(number of kept keys)."""
    rng = _rng(2)
    B, H, N, d, blk = 2, 1, 9, 4, 3
    q = np.zeros((B, H, N, d))
    k = rng.standard_normal((B, H, N, d))
    v = rng.standard_normal((B, H, N, d))
    for causal, kl, bm in _mask_modes(N, blk):
        o, lse = ref.attn_fwd(q, k, v, 1.3, causal, kl, bm, blk, lib=lib)
        for b in range(B):
            for i in range(N):
                keep = [j for j in range(N)
                        if (not causal or j <= i)
                        and (kl is None or j < kl[b])
                        and (bm is None or bm[i // blk, j // blk])]
                exp_o = v[b, 0, keep].mean(axis=0)
                _close(o[b, 0, i], exp_o, what="mean of kept V")
                _close(lse[b, 0, i], math.log(len(keep)), what="ln(n kept)")


def pin_dominant_key(lib):
    """One key whose score exceeds all others by > 60: O_i equals its V row
    (the others' weight is below e^-60)."""
    rng = _rng(3)
    N, d = 16, 8
    q = np.zeros((1, 1, N, d))
    q[..., 0] = 10.0
    k = 0.01 * rng.standard_normal((1, 1, N, d))
    jstar = 11
    k[0, 0, jstar, 0] = 10.0
    v = rng.standard_normal((1, 1, N, d))
    o, lse = ref.attn_fwd(q, k, v, 1.0, lib=lib)
    for i in range(N):
        _close(o[0, 0, i], v[0, 0, jstar], tol=1e-20 + 1e-12, what="dominant key")
    # s* = 10 * 10 = 100; every other score is below 1, so LSE = 100 to 1e-40
    _close(lse[0, 0], np.full(N, 100.0), tol=1e-12, what="dominant key LSE")


def pin_key_permutation_invariance(lib):
    """Non-causal, unmasked attention is invariant under a joint permutation
    of the K and V rows; the backward permutes dK and dV the same way."""
    rng = _rng(4)
    B, H, N, d = 1, 2, 10, 5
    q, k, v, do = (rng.standard_normal((B, H, N, d)) for _ in range(4))
    perm = rng.permutation(N)
    o1, l1 = ref.attn_fwd(q, k, v, 0.4, lib=lib)
    o2, l2 = ref.attn_fwd(q, k[:, :, perm], v[:, :, perm], 0.4, lib=lib)
    _close(o1, o2, what="O under permutation")
    _close(l1, l2, what="LSE under permutation")
    g1 = ref.attn_bwd(q, k, v, do, 0.4, lib=lib)
    g2 = ref.attn_bwd(q, k[:, :, perm], v[:, :, perm], do, 0.4, lib=lib)
    _close(g1[0], g2[0], what="dQ under permutation")
    _close(g1[1][:, :, perm], g2[1], what="dK under permutation")
    _close(g1[2][:, :, perm], g2[2], what="dV under permutation")


def pin_causal_first_row(lib):
    """Causal: query 0 sees only key 0, so O_0 = V_0 and LSE_0 = scale q0.k0."""
    rng = _rng(5)
    B, H, N, d = 2, 3, 7, 6
    q, k, v = (rng.standard_normal((B, H, N, d)) for _ in range(3))
    o, lse = ref.attn_fwd(q, k, v, 0.25, causal=True, lib=lib)
    _close(o[:, :, 0], v[:, :, 0], what="causal O_0")
    _close(lse[:, :, 0], 0.25 * np.einsum("bhd,bhd->bh", q[:, :, 0], k[:, :, 0]),
           what="causal LSE_0")


def pin_single_key(lib):
    """N = 1: O = V and LSE = scale q.k."""
    rng = _rng(6)
    q, k, v = (rng.standard_normal((3, 2, 1, 5)) for _ in range(3))
    o, lse = ref.attn_fwd(q, k, v, 0.9, lib=lib)
    _close(o, v, what="N=1 O")
    _close(lse[..., 0], 0.9 * np.einsum("bhd,bhd->bh", q[:, :, 0], k[:, :, 0]), what="N=1 LSE")


def pin_two_key_closed_form(lib):
    """One query, two keys with scores s1, s2: p2 = 1 / (1 + e^(s1 - s2)),
    O = (1 - p2) v1 + p2 v2, LSE = s1 + ln(1 + e^(s2 - s1))."""
    q = np.array([[[[1.0, 2.0], [0.0, 0.0]]]])
    k = np.array([[[[0.5, -1.0], [2.0, 0.25]]]])
    v = np.array([[[[3.0, -1.0], [-2.0, 5.0]]]])
    scale = 0.75
    s1 = scale * (1.0 * 0.5 + 2.0 * -1.0)
    s2 = scale * (1.0 * 2.0 + 2.0 * 0.25)
    p2 = 1.0 / (1.0 + math.exp(s1 - s2))
    o, lse = ref.attn_fwd(q, k, v, scale, lib=lib)
    _close(o[0, 0, 0], (1 - p2) * v[0, 0, 0] + p2 * v[0, 0, 1], what="two-key O")
    _close(lse[0, 0, 0], s1 + math.log1p(math.exp(s2 - s1)), what="two-key LSE")
    # query 1 is zero: both scores 0, O = mean, LSE = ln 2
    _close(o[0, 0, 1], 0.5 * (v[0, 0, 0] + v[0, 0, 1]), what="two-key zero query")
    _close(lse[0, 0, 1], math.log(2.0), what="two-key zero query LSE")


def pin_merge_identity(lib):
    """Softmax over x U y from the two halves ("The Math Behind Flash
    Attention", softmax merger): with m = max(m_x, m_y) and row sums l_x, l_y
    rescaled by e^(m_x - m), e^(m_y - m), the merged LSE is
    logaddexp(LSE_x, LSE_y) and O = e^(LSE_x - LSE) O_x + e^(LSE_y - LSE) O_y.
    The halves are selected with 2x2 block masks."""
    rng = _rng(7)
    B, H, N, d = 2, 2, 12, 4
    blk = N // 2
    q, k, v = (rng.standard_normal((B, H, N, d)) for _ in range(3))
    q *= 2.0
    left = np.array([[1, 0], [1, 0]], dtype=np.uint8)
    right = np.array([[0, 1], [0, 1]], dtype=np.uint8)
    o_x, l_x = ref.attn_fwd(q, k, v, 0.6, block_mask=left, blk=blk, lib=lib)
    o_y, l_y = ref.attn_fwd(q, k, v, 0.6, block_mask=right, blk=blk, lib=lib)
    o, lse = ref.attn_fwd(q, k, v, 0.6, lib=lib)
    l_m = np.logaddexp(l_x, l_y)
    _close(lse, l_m, what="merged LSE")
    o_m = np.exp(l_x - l_m)[..., None] * o_x + np.exp(l_y - l_m)[..., None] * o_y
    _close(o, o_m, what="merged O")


def pin_tiled_algorithm(lib):
    """The corrected block algorithm (tiled_numpy.py) agrees with the oracle
    for every mask kind, ragged block edges included."""
    rng = _rng(8)
    B, H, N, d, blk = 2, 1, 13, 3, 4
    q, k, v = (rng.standard_normal((B, H, N, d)) for _ in range(3))
    for causal, kl, bm in _mask_modes(N, blk):
        o, lse = ref.attn_fwd(q, k, v, 0.8, causal, kl, bm, blk, lib=lib)
        for b in range(B):
            ot, lt = tiled_attention_head(q[b, 0], k[b, 0], v[b, 0], 0.8, block=5,
                                          causal=causal,
                                          kv_len_b=None if kl is None else kl[b],
                                          block_mask=bm, blk=blk)
            _close(o[b, 0], ot, what=f"tiled O causal={causal}")
            _close(lse[b, 0], lt, what=f"tiled LSE causal={causal}")


def pin_torch_reference(lib):
    """torch's own fp64 scaled_dot_product_attention and autograd agree with
    the oracle's forward and backward (every row keeps at least one key)."""
    import torch
    rng = _rng(9)
    B, H, N, d, blk = 2, 2, 10, 4, 4
    q, k, v, do = (rng.standard_normal((B, H, N, d)) for _ in range(4))
    for causal, kl, bm in _mask_modes(N, blk):
        keep = np.ones((B, 1, N, N), dtype=bool)
        ii = np.arange(N)[:, None]
        jj = np.arange(N)[None, :]
        for b in range(B):
            kb = np.ones((N, N), dtype=bool)
            if causal:
                kb &= jj <= ii
            if kl is not None:
                kb &= jj < kl[b]
            if bm is not None:
                kb &= bm[ii // blk, jj // blk] != 0
            keep[b, 0] = kb
        tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
        out = torch.nn.functional.scaled_dot_product_attention(
            tq, tk, tv, attn_mask=torch.tensor(keep), scale=0.55)
        out.backward(torch.tensor(do))
        o, _ = ref.attn_fwd(q, k, v, 0.55, causal, kl, bm, blk, lib=lib)
        dq, dk, dv, _ = ref.attn_bwd(q, k, v, do, 0.55, causal, kl, bm, blk, lib=lib)
        _close(o, out.detach().numpy(), tol=1e-12, what="torch O")
        _close(dq, tq.grad.numpy(), tol=1e-12, what="torch dQ")
        _close(dk, tk.grad.numpy(), tol=1e-12, what="torch dK")
        _close(dv, tv.grad.numpy(), tol=1e-12, what="torch dV")


# --------------------------------------------------------------- backward pins

def _loss(lib, q, k, v, do, scale, causal, kl, bm, blk):
    o, _ = ref.attn_fwd(q, k, v, scale, causal, kl, bm, blk, lib=lib)
    return float(np.sum(o * do))


def pin_finite_differences(lib):
    """Central finite differences of L = sum(O * dO) (fp64, eps 1e-6) match
    dQ, dK, dV to 1e-6 relative to the largest gradient entry."""
    rng = _rng(10)
    B, H, N, d, blk = 2, 1, 6, 3, 2
    q, k, v, do = (rng.standard_normal((B, H, N, d)) for _ in range(4))
    eps = 1e-6
    for causal, kl, bm in _mask_modes(N, blk):
        dq, dk, dv, _ = ref.attn_bwd(q, k, v, do, 0.9, causal, kl, bm, blk, lib=lib)
        for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
            num = np.zeros_like(x)
            for idx in np.ndindex(x.shape):
                xp = x.copy()
                xp[idx] += eps
                xm = x.copy()
                xm[idx] -= eps
                args = {"q": q, "k": k, "v": v}
                args[name] = xp
                lp = _loss(lib, args["q"], args["k"], args["v"], do, 0.9, causal, kl, bm, blk)
                args[name] = xm
                lm = _loss(lib, args["q"], args["k"], args["v"], do, 0.9, causal, kl, bm, blk)
                num[idx] = (lp - lm) / (2 * eps)
            scale = max(1.0, np.max(np.abs(g)))
            err = np.max(np.abs(num - g)) / scale
            assert err < 1e-6, f"finite differences d{name} causal={causal}: {err:.2e}"


def pin_gradient_invariants(lib):
    """sum_j dV_j = sum_i dO_i over rows with a kept key (rows of P sum to 1);
    sum_j dK_j = 0 (adding one vector to every key shifts each row's scores
    by a constant, which softmax ignores); D_i = sum_c dO_ic O_ic."""
    rng = _rng(11)
    B, H, N, d, blk = 2, 2, 9, 4, 3
    q, k, v, do = (rng.standard_normal((B, H, N, d)) for _ in range(4))
    for causal, kl, bm in _mask_modes(N, blk):
        o, lse = ref.attn_fwd(q, k, v, 0.5, causal, kl, bm, blk, lib=lib)
        dq, dk, dv, delta = ref.attn_bwd(q, k, v, do, 0.5, causal, kl, bm, blk, lib=lib)
        live = np.isfinite(lse)[..., None]
        _close(dv.sum(axis=2), (do * live).sum(axis=2), what="sum dV")
        _close(dk.sum(axis=2), np.zeros((B, H, d)), what="sum dK")
        _close(delta, np.sum(do * o, axis=-1), what="D = rowsum(dO*O)")


def pin_sampled_agree_with_full(lib):
    """Row/column-sampled forward and backward equal the full computation."""
    rng = _rng(12)
    B, H, N, d, blk = 2, 1, 12, 4, 4
    q, k, v, do = (rng.standard_normal((B, H, N, d)) for _ in range(4))
    for causal, kl, bm in _mask_modes(N, blk):
        o, lse = ref.attn_fwd(q, k, v, 0.7, causal, kl, bm, blk, lib=lib)
        dq, dk, dv, delta = ref.attn_bwd(q, k, v, do, 0.7, causal, kl, bm, blk, lib=lib)
        rows = [0, 5, 11, 3]
        for b in range(B):
            klb = None if kl is None else kl[b]
            orr, lr = ref.attn_fwd_rows(q[b, 0], k[b, 0], v[b, 0], 0.7, rows, causal, klb, bm,
                                        blk, lib=lib)
            _close(orr, o[b, 0, rows], what="fwd rows O")
            _close(lr, lse[b, 0, rows], what="fwd rows LSE")
            sq, sk, sv, sl, sd = ref.attn_bwd_sampled(q[b, 0], k[b, 0], v[b, 0], do[b, 0], 0.7,
                                                      rows, rows[::-1], causal, klb, bm, blk,
                                                      lib=lib)
            _close(sq, dq[b, 0, rows], what="sampled dQ")
            _close(sk, dk[b, 0, rows[::-1]], what="sampled dK")
            _close(sv, dv[b, 0, rows[::-1]], what="sampled dV")
            _close(sl, lse[b, 0], what="sampled LSE")
            _close(sd, delta[b, 0], what="sampled D")


def pin_empty_rows(lib):
    """A query block whose mask row keeps nothing: O = 0, LSE = -inf and it
    contributes no gradient."""
    rng = _rng(13)
    B, H, N, d, blk = 1, 1, 8, 2, 4
    q, k, v, do = (rng.standard_normal((B, H, N, d)) for _ in range(4))
    bm = np.array([[1, 1], [0, 0]], dtype=np.uint8)
    o, lse = ref.attn_fwd(q, k, v, 1.0, block_mask=bm, blk=blk, lib=lib)
    assert np.all(o[0, 0, 4:] == 0.0) and np.all(np.isneginf(lse[0, 0, 4:]))
    assert np.all(np.isfinite(lse[0, 0, :4]))
    dq, dk, dv, _ = ref.attn_bwd(q, k, v, do, 1.0, block_mask=bm, blk=blk, lib=lib)
    assert np.all(dq[0, 0, 4:] == 0.0)
    # the dead rows' dO must not reach dV
    do2 = do.copy()
    do2[0, 0, 4:] += 5.0
    _, dk2, dv2, _ = ref.attn_bwd(q, k, v, do2, 1.0, block_mask=bm, blk=blk, lib=lib)
    _close(dv2, dv, what="dead rows reach dV")
    _close(dk2, dk, what="dead rows reach dK")


ALL_PINS = [
    pin_rows_sum_to_one,
    pin_q_zero_mean_of_values,
    pin_dominant_key,
    pin_key_permutation_invariance,
    pin_causal_first_row,
    pin_single_key,
    pin_two_key_closed_form,
    pin_merge_identity,
    pin_tiled_algorithm,
    pin_torch_reference,
    pin_finite_differences,
    pin_gradient_invariants,
    pin_sampled_agree_with_full,
    pin_empty_rows,
]
