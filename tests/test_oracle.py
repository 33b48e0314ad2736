"""The fp64 oracle against its pins (CPU only), and a mutation check that
each plausible slip in the oracle is caught by at least one pin."""
import os
import re
import shutil
import tempfile

import numpy as np
import pytest

from oracle import ref
from tests import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin, oracle_lib):
    pin(oracle_lib)


def test_thread_count_does_not_change_results(oracle_lib):
    rng = np.random.default_rng(20)
    B, H, N, d = 2, 3, 37, 8
    q, k, v, do = (rng.standard_normal((B, H, N, d)) for _ in range(4))
    o1, l1 = ref.attn_fwd(q, k, v, 0.3, causal=True, nthreads=1, lib=oracle_lib)
    o8, l8 = ref.attn_fwd(q, k, v, 0.3, causal=True, nthreads=8, lib=oracle_lib)
    assert np.array_equal(o1, o8) and np.array_equal(l1, l8)
    g1 = ref.attn_bwd(q, k, v, do, 0.3, causal=True, rows_per_task=5, nthreads=1, lib=oracle_lib)
    g8 = ref.attn_bwd(q, k, v, do, 0.3, causal=True, rows_per_task=5, nthreads=8, lib=oracle_lib)
    for a, b in zip(g1, g8):
        assert np.array_equal(a, b)


def test_printed_block_update_is_not_the_definition(oracle_lib):
    """Reading of the page's block loop: the output update as printed (divide
    by the new row sum without first multiplying the old, normalised output
    by the old row sum) is not softmax attention once a row spans two key
    blocks; the corrected update is (pin_tiled_algorithm)."""
    from tests.tiled_numpy import tiled_attention_head
    rng = np.random.default_rng(21)
    q, k, v = (rng.standard_normal((1, 1, 8, 3)) for _ in range(3))
    o, _ = ref.attn_fwd(q, k, v, 1.0, lib=oracle_lib)
    printed, _ = tiled_attention_head(q[0, 0], k[0, 0], v[0, 0], 1.0, block=4, printed_update=True)
    assert np.max(np.abs(printed - o[0, 0])) > 1e-3


def test_bad_sizes_rejected(oracle_lib):
    q = np.zeros((1, 1, 4, 2))
    with pytest.raises(ValueError):
        ref.attn_fwd_rows(q[0, 0], q[0, 0], q[0, 0], 1.0, [4], lib=oracle_lib)
    with pytest.raises(ValueError):
        ref.attn_bwd_sampled(q[0, 0], q[0, 0], q[0, 0], q[0, 0], 1.0, [0], [-1], lib=oracle_lib)


# Plausible slips, each a (pattern, replacement) edit of attention_ref.c.
MUTANTS = {
    "dropped_scale": (r"s_row\[j\] = p->scale \* acc;", "s_row[j] = acc;"),
    "causal_off_by_one": (r"if \(p->causal && j > i\)", "if (p->causal && j >= i)"),
    "kv_len_off_by_one": (r"j >= p->kv_len\[b\]", "j > p->kv_len[b]"),
    "block_mask_transposed": (r"\[\(size_t\)\(i / p->blk\) \* nb \+ \(j / p->blk\)\]",
                              "[(size_t)(j / p->blk) * nb + (i / p->blk)]"),
    "lse_log2": (r"const double lse = m \+ log\(l\);", "const double lse = m + log2(l);"),
    "lse_missing_max": (r"const double lse = m \+ log\(l\);", "const double lse = log(l);"),
    "ds_sign": (r"const double ds = p_row\[j\] \* \(dp_row\[j\] - D\);",
                "const double ds = p_row[j] * (dp_row[j] + D);"),
    "dq_uses_q": (r"dqi\[c\] \+= p->scale \* ds \* kj\[c\];", "dqi[c] += p->scale * ds * qi[c];"),
    "dk_no_scale": (r"pkj\[c\] \+= p->scale \* ds \* qi\[c\];", "pkj[c] += ds * qi[c];"),
    "dv_uses_dp": (r"pvj\[c\] \+= p_row\[j\] \* doi\[c\];", "pvj[c] += dp_row[j] * doi[c];"),
    "o_uses_k": (r"oi\[c\] \+= p_row\[j\] \* vj\[c\];", "oi[c] += p_row[j] * kh[(size_t)j * d + c];"),
    "delta_dropped": (r"D \+= p_row\[j\] \* acc;", "D += 0.0 * acc;"),
    "sampled_dv_no_p": (r"dvj\[c\] \+= P \* doi\[c\];", "dvj[c] += doi[c];"),
    "rows_dq_sign": (r"const double ds = P \* \(dp - job->D\[i\]\);",
                     "const double ds = P * (dp + job->D[i]);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name):
    pattern, repl = MUTANTS[name]
    src = open(os.path.join(os.path.dirname(ref.__file__), "attention_ref.c")).read()
    mutated, n = re.subn(pattern, repl, src)
    assert n >= 1, f"mutation {name} did not apply"
    tmp = tempfile.mkdtemp(prefix="oracle_mutant_")
    try:
        c = os.path.join(tmp, "m.c")
        so = os.path.join(tmp, "m.so")
        open(c, "w").write(mutated)
        ref.build(force=True, src=c, out=so)
        lib = ref.load(so)
        failed = []
        for pin in oracle_pins.ALL_PINS:
            try:
                pin(lib)
            except AssertionError:
                failed.append(pin.__name__)
        assert failed, f"no pin caught mutant {name}"
    finally:
        shutil.rmtree(tmp, ignore_errors=True)
