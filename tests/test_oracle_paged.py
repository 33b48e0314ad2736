"""Pins of the oracle's paged decode (CPU; oracle.ref.paged_decode).

The paged decode is a gather (each sequence's pages in logical order, cut
at seq_len) followed by the already pinned forward definition on the last
Nq positions with the causal mask. These pins check the gather and the
query placement against what the definition fixes independently:
  * one cached key: O is that slot's value row, LSE is the scaled score;
  * q = 0: O is the mean of the visible value rows, found here key by key
    through the block table (brute force), LSE = ln(count);
  * an identity page table over a contiguous cache, with every position a
    query, is the causal forward of the dense oracle;
  * permuting the pool's pages together with the table changes nothing.
A planted slip in the oracle's gather or placement must fail one of them.
"""
import inspect
import math
import re
import textwrap

import numpy as np
import pytest

from oracle import ref


def _case(rng, B, H, Hkv, Nq, d, ps, pages_per_seq, num_pages, seq_len):
    q = rng.standard_normal((B, H, Nq, d))
    kc = rng.standard_normal((num_pages, Hkv, ps, d))
    vc = rng.standard_normal((num_pages, Hkv, ps, d))
    perm = rng.permutation(num_pages)[: B * pages_per_seq].reshape(B, pages_per_seq)
    return q, kc, vc, perm.astype(np.int32), np.asarray(seq_len, dtype=np.int32)


def pin_single_key(fn):
    rng = np.random.default_rng(1)
    q, kc, vc, bt, sl = _case(rng, 2, 4, 2, 1, 8, 4, 3, 7, [1, 1])
    o, lse = fn(q, kc, vc, bt, sl, 0.7, 4)
    for b in range(2):
        for h in range(4):
            kvh = h // 2
            p = bt[b, 0]
            assert np.allclose(o[b, h, 0], vc[p, kvh, 0], atol=1e-12)
            assert abs(lse[b, h, 0] - 0.7 * float(q[b, h, 0] @ kc[p, kvh, 0])) < 1e-12


def pin_q_zero_brute_force(fn):
    rng = np.random.default_rng(2)
    ps, Nq = 4, 3
    q, kc, vc, bt, sl = _case(rng, 4, 4, 2, Nq, 8, ps, 4, 20, [10, 2, 16, 0])
    q[:] = 0.0
    o, lse = fn(q, kc, vc, bt, sl, 0.5, ps)
    for b in range(4):
        for h in range(4):
            kvh = h // 2
            for i in range(Nq):
                last = int(sl[b]) - Nq + i  # visible keys 0 .. last
                if last < 0:
                    assert np.all(o[b, h, i] == 0) and lse[b, h, i] == -np.inf
                    continue
                rows = [vc[bt[b, j // ps], kvh, j % ps] for j in range(last + 1)]
                assert np.allclose(o[b, h, i], np.mean(rows, axis=0), atol=1e-12)
                assert abs(lse[b, h, i] - math.log(last + 1)) < 1e-12


def pin_identity_table_is_dense_causal(fn):
    rng = np.random.default_rng(3)
    B, H, Hkv, L, d, ps = 2, 4, 2, 12, 8, 4
    q = rng.standard_normal((B, H, L, d))
    k = rng.standard_normal((B, Hkv, L, d))
    v = rng.standard_normal((B, Hkv, L, d))
    npp = L // ps
    kc = k.reshape(B, Hkv, npp, ps, d).transpose(0, 2, 1, 3, 4).reshape(B * npp, Hkv, ps, d)
    vc = v.reshape(B, Hkv, npp, ps, d).transpose(0, 2, 1, 3, 4).reshape(B * npp, Hkv, ps, d)
    bt = np.arange(B * npp, dtype=np.int32).reshape(B, npp)
    o, lse = fn(q, kc, vc, bt, np.full(B, L, dtype=np.int32), 0.4, ps)
    o_ref, lse_ref = ref.attn_fwd(q, np.repeat(k, H // Hkv, axis=1), np.repeat(v, H // Hkv, axis=1), 0.4, True)
    assert np.allclose(o, o_ref, atol=1e-12) and np.allclose(lse, lse_ref, atol=1e-12)


def pin_page_permutation_invariance(fn):
    rng = np.random.default_rng(4)
    q, kc, vc, bt, sl = _case(rng, 3, 2, 1, 2, 8, 4, 5, 16, [17, 5, 20])
    o1, l1 = fn(q, kc, vc, bt, sl, 0.3, 4)
    perm = rng.permutation(kc.shape[0])       # pool page p moves to slot perm[p]
    kc2, vc2 = np.empty_like(kc), np.empty_like(vc)
    kc2[perm], vc2[perm] = kc, vc
    o2, l2 = fn(q, kc2, vc2, perm[bt].astype(np.int32), sl, 0.3, 4)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


PINS = [pin_single_key, pin_q_zero_brute_force, pin_identity_table_is_dense_causal,
        pin_page_permutation_invariance]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_paged_pin(pin):
    pin(ref.paged_decode)


MUTANTS = {
    "pages_in_reverse_order": (r"pages = bt\[b, :\(L \+ page_size - 1\) // page_size\]",
                               "pages = bt[b, :(L + page_size - 1) // page_size][::-1]"),
    "query_one_position_early": (r"pos = \[L - Nq \+ i ", "pos = [L - Nq + i - 1 "),
    "first_kv_head_for_all": (r"kc\[p, kvh\]", "kc[p, 0]"),
    "context_one_key_short": (r"L = int\(min\(max\(int\(sl\[b\]\), 0\), cap\)\)",
                              "L = int(min(max(int(sl[b]) - 1, 0), cap))"),
    "new_tokens_not_causal": (r"causal=True", "causal=False"),
    "ignores_block_table": (r"for p in pages\]", "for p in range(len(pages))]"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_paged_mistake_is_caught(name):
    pattern, repl = MUTANTS[name]
    src = textwrap.dedent(inspect.getsource(ref.paged_decode))
    mutated, n = re.subn(pattern, repl, src)
    assert n >= 1, f"mutation {name} did not apply"
    ns = dict(vars(ref))
    exec(compile(mutated, "<mutant>", "exec"), ns)
    failed = []
    for pin in PINS:
        try:
            pin(ns["paged_decode"])
        except (AssertionError, IndexError, ValueError):
            failed.append(pin.__name__)
    assert failed, f"no pin caught mutant {name}"
