"""Second, independent fp64 implementation for pinning the oracle.

This is the block algorithm of "Flash Attention: revolutionizing transformer
efficiency" (section "Implementation Details": outer loop over query blocks,
inner loop over key/value blocks, running row max M and row sum L), written
in numpy, with the output update corrected: the printed update divides by the
new row sum but never multiplies the previous, already-normalised output by
the previous row sum. Here the running output stays normalised:

    O <- (L_old * exp(M_old - M_new) * O + exp(S - M_new) @ V) / L_new

It shares nothing with the C oracle; tests compare the two.
"""
import numpy as np


def _mask(N, i0, i1, j0, j1, causal, kv_len_b, block_mask, blk):
    ii = np.arange(i0, i1)[:, None]
    jj = np.arange(j0, j1)[None, :]
    keep = np.ones((i1 - i0, j1 - j0), dtype=bool)
    if causal:
        keep &= jj <= ii
    if kv_len_b is not None:
        keep &= jj < kv_len_b
    if block_mask is not None:
        keep &= block_mask[ii // blk, jj // blk] != 0
    return keep


def tiled_attention_head(q, k, v, scale, block=4, causal=False, kv_len_b=None,
                         block_mask=None, blk=128, printed_update=False):
    """One head: q, k, v [N, d] float64 -> (O [N, d], LSE [N]).

    printed_update=True reproduces the update as printed (for the test that
    shows it is not the definition)."""
    N, d = q.shape
    O = np.zeros((N, d))
    LSE = np.full(N, -np.inf)
    for i0 in range(0, N, block):
        i1 = min(i0 + block, N)
        Ob = np.zeros((i1 - i0, d))
        L = np.zeros((i1 - i0, 1))
        M = np.full((i1 - i0, 1), -np.inf)
        for j0 in range(0, N, block):
            j1 = min(j0 + block, N)
            S = (q[i0:i1] @ k[j0:j1].T) * scale
            keep = _mask(N, i0, i1, j0, j1, causal, kv_len_b, block_mask, blk)
            S = np.where(keep, S, -np.inf)
            M_new = np.maximum(M, S.max(axis=1, keepdims=True))
            live = np.isfinite(M_new)[:, 0]
            Mn = np.where(np.isfinite(M_new), M_new, 0.0)
            exp_S = np.where(keep, np.exp(np.where(keep, S, 0.0) - Mn), 0.0)
            exp_M_diff = np.where(np.isfinite(M), np.exp(np.where(np.isfinite(M), M, 0.0) - Mn),
                                  0.0)
            L_new = exp_M_diff * L + exp_S.sum(axis=1, keepdims=True)
            if printed_update:
                num = exp_M_diff * Ob + exp_S @ v[j0:j1]
            else:
                num = L * exp_M_diff * Ob + exp_S @ v[j0:j1]
            safe = np.where(L_new > 0, L_new, 1.0)
            Ob = np.where(live[:, None], num / safe, Ob)
            L = np.where(live[:, None], L_new, L)
            M = np.where(live[:, None], M_new, M)
        O[i0:i1] = Ob
        LSE[i0:i1] = np.where(L[:, 0] > 0, M[:, 0] + np.log(np.where(L[:, 0] > 0, L[:, 0], 1.0)),
                              -np.inf)
    return O, LSE
