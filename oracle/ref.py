"""ctypes loader for the fp64 attention oracle (test infrastructure only).

Each function converts its inputs to contiguous float64 arrays (exact for
fp16/bf16 values), calls the C oracle in ``attention_ref.c`` and returns
float64 numpy arrays. See that file for the definition it computes and the
passages it follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attention_ref.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_i32p = ctypes.POINTER(ctypes.c_int32)
_i64p = ctypes.POINTER(ctypes.c_int64)
_u8p = ctypes.POINTER(ctypes.c_uint8)


def library_path() -> str:
    return _LIB


def build(force: bool = False, src: str | None = None, out: str | None = None,
          extra_flags: tuple[str, ...] = ()) -> str:
    """Compile the oracle with gcc (plain -O2, IEEE semantics, no fast-math)."""
    src = src or _SRC
    out = out or _LIB
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    tmp = out + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-D_DEFAULT_SOURCE", "-shared", "-fPIC",
           "-pthread", *extra_flags, "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _bind(lib):
    lib.oracle_attn_fwd.restype = ctypes.c_int
    lib.oracle_attn_fwd.argtypes = [
        _dp, _dp, _dp, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        ctypes.c_double, ctypes.c_int, _i32p, _u8p, ctypes.c_int, _dp, _dp,
        ctypes.c_int]
    lib.oracle_attn_fwd_rows.restype = ctypes.c_int
    lib.oracle_attn_fwd_rows.argtypes = [
        _dp, _dp, _dp, ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_int,
        ctypes.c_int, _u8p, ctypes.c_int, ctypes.c_int, _i64p, _dp, _dp,
        ctypes.c_int]
    lib.oracle_attn_bwd.restype = ctypes.c_int
    lib.oracle_attn_bwd.argtypes = [
        _dp, _dp, _dp, _dp, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        ctypes.c_double, ctypes.c_int, _i32p, _u8p, ctypes.c_int, _dp, _dp, _dp,
        _dp, ctypes.c_int, ctypes.c_int]
    lib.oracle_attn_bwd_sampled.restype = ctypes.c_int
    lib.oracle_attn_bwd_sampled.argtypes = [
        _dp, _dp, _dp, _dp, ctypes.c_int, ctypes.c_int, ctypes.c_double,
        ctypes.c_int, ctypes.c_int, _u8p, ctypes.c_int,
        ctypes.c_int, _i64p, _dp, ctypes.c_int, _i64p, _dp, _dp, _dp, _dp,
        ctypes.c_int]
    return lib


def load(path: str | None = None):
    """Load (building first if needed) the oracle library; cached for _LIB."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            build()
            _lib = _bind(ctypes.CDLL(_LIB))
    return _lib


def _f64(x) -> np.ndarray:
    if hasattr(x, "detach"):  # torch tensor: exact widening on the CPU
        import torch
        x = x.detach().to("cpu", torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray, t):
    return a.ctypes.data_as(t)


def _nthreads(n):
    return int(n) if n else (os.cpu_count() or 1)


def _masks(B, N, kv_len, block_mask, blk):
    kl = None
    if kv_len is not None:
        kl = np.ascontiguousarray(np.asarray(
            kv_len.cpu().numpy() if hasattr(kv_len, "cpu") else kv_len, dtype=np.int32))
        assert kl.shape == (B,)
    bm = None
    if block_mask is not None:
        bm = block_mask.cpu().numpy() if hasattr(block_mask, "cpu") else block_mask
        bm = np.ascontiguousarray((np.asarray(bm) != 0).astype(np.uint8))
        nb = (N + blk - 1) // blk
        assert bm.shape == (nb, nb), (bm.shape, nb)
    return kl, bm


def attn_fwd(q, k, v, scale, causal=False, kv_len=None, block_mask=None,
             blk=128, nthreads=None, lib=None):
    """Full forward. q, k, v: [B, H, N, d]. Returns (o [B,H,N,d], lse [B,H,N])."""
    lib = lib or load()
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, N, d = q.shape
    assert k.shape == q.shape and v.shape == q.shape
    kl, bm = _masks(B, N, kv_len, block_mask, blk)
    o = np.zeros((B, H, N, d))
    lse = np.zeros((B, H, N))
    rc = lib.oracle_attn_fwd(
        _ptr(q, _dp), _ptr(k, _dp), _ptr(v, _dp), B, H, N, d, float(scale),
        int(bool(causal)), None if kl is None else _ptr(kl, _i32p),
        None if bm is None else _ptr(bm, _u8p), blk, _ptr(o, _dp), _ptr(lse, _dp),
        _nthreads(nthreads))
    if rc != 0:
        raise ValueError("oracle_attn_fwd failed: %d" % rc)
    return o, lse


def attn_fwd_rows(q, k, v, scale, rows, causal=False, kv_len_b=None,
                  block_mask=None, blk=128, nthreads=None, lib=None):
    """Forward of selected query rows of one head. q, k, v: [N, d]."""
    lib = lib or load()
    q, k, v = _f64(q), _f64(k), _f64(v)
    N, d = q.shape
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    _, bm = _masks(1, N, None, block_mask, blk)
    o = np.zeros((len(rows), d))
    lse = np.zeros(len(rows))
    rc = lib.oracle_attn_fwd_rows(
        _ptr(q, _dp), _ptr(k, _dp), _ptr(v, _dp), N, d, float(scale),
        int(bool(causal)), -1 if kv_len_b is None else int(kv_len_b),
        None if bm is None else _ptr(bm, _u8p), blk, len(rows), _ptr(rows, _i64p),
        _ptr(o, _dp), _ptr(lse, _dp), _nthreads(nthreads))
    if rc != 0:
        raise ValueError("oracle_attn_fwd_rows failed: %d" % rc)
    return o, lse


def attn_bwd(q, k, v, dout, scale, causal=False, kv_len=None, block_mask=None,
             blk=128, rows_per_task=0, nthreads=None, lib=None):
    """Full backward. Returns (dq, dk, dv [B,H,N,d], delta [B,H,N])."""
    lib = lib or load()
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    B, H, N, d = q.shape
    kl, bm = _masks(B, N, kv_len, block_mask, blk)
    dq = np.zeros((B, H, N, d))
    dk = np.zeros((B, H, N, d))
    dv = np.zeros((B, H, N, d))
    delta = np.zeros((B, H, N))
    rc = lib.oracle_attn_bwd(
        _ptr(q, _dp), _ptr(k, _dp), _ptr(v, _dp), _ptr(dout, _dp), B, H, N, d,
        float(scale), int(bool(causal)), None if kl is None else _ptr(kl, _i32p),
        None if bm is None else _ptr(bm, _u8p), blk, _ptr(dq, _dp), _ptr(dk, _dp),
        _ptr(dv, _dp), _ptr(delta, _dp), int(rows_per_task), _nthreads(nthreads))
    if rc != 0:
        raise ValueError("oracle_attn_bwd failed: %d" % rc)
    return dq, dk, dv, delta


def attn_bwd_sampled(q, k, v, dout, scale, qrows, kcols, causal=False,
                     kv_len_b=None, block_mask=None, blk=128, nthreads=None, lib=None):
    """Backward of one head at sampled query rows (dq) and key rows (dk, dv).

    q, k, v, dout: [N, d]. Returns (dq_rows, dk_rows, dv_rows, lse [N], delta [N]).
    """
    lib = lib or load()
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    N, d = q.shape
    qrows = np.ascontiguousarray(np.asarray(qrows, dtype=np.int64))
    kcols = np.ascontiguousarray(np.asarray(kcols, dtype=np.int64))
    _, bm = _masks(1, N, None, block_mask, blk)
    dq = np.zeros((len(qrows), d))
    dk = np.zeros((len(kcols), d))
    dv = np.zeros((len(kcols), d))
    lse = np.zeros(N)
    delta = np.zeros(N)
    rc = lib.oracle_attn_bwd_sampled(
        _ptr(q, _dp), _ptr(k, _dp), _ptr(v, _dp), _ptr(dout, _dp), N, d,
        float(scale), int(bool(causal)), -1 if kv_len_b is None else int(kv_len_b),
        None if bm is None else _ptr(bm, _u8p), blk,
        len(qrows), _ptr(qrows, _i64p), _ptr(dq, _dp),
        len(kcols), _ptr(kcols, _i64p), _ptr(dk, _dp), _ptr(dv, _dp),
        _ptr(lse, _dp), _ptr(delta, _dp), _nthreads(nthreads))
    if rc != 0:
        raise ValueError("oracle_attn_bwd_sampled failed: %d" % rc)
    return dq, dk, dv, lse, delta


def paged_decode(q, k_cache, v_cache, block_table, seq_len, scale, page_size, lib=None):
    """Decode attention over a paged key/value cache (test infrastructure).

    Page "Enhancing Transformer Models: Innovations in Attention Mechanisms
    and Performance Optimization", section "From FlashAttention to
    PagedAttention": the cache lives in pages. Read here as: sequence b's
    logical page i is pool page block_table[b, i]; its first seq_len[b] keys,
    taken page by page in logical order, are its context. The Nq new query
    tokens are the last Nq positions of that context, so query i sits at
    position L - Nq + i and, with the causal mask of the forward definition,
    sees keys 0 .. L - Nq + i. Query head h reads key/value head h / (H/Hkv).

    q [B,H,Nq,d]; k_cache, v_cache [num_pages, Hkv, page_size, d];
    block_table [B, pages_per_seq]; seq_len [B]. Returns o [B,H,Nq,d] and
    lse [B,H,Nq] (float64; a query with no visible key: 0 and -inf).
    """
    q = _f64(q)
    kc, vc = k_cache, v_cache  # widened page by page below (the pool may be large)
    bt = np.asarray(block_table.cpu().numpy() if hasattr(block_table, "cpu") else block_table)
    sl = np.asarray(seq_len.cpu().numpy() if hasattr(seq_len, "cpu") else seq_len)
    B, H, Nq, d = q.shape
    Hkv = kc.shape[1]
    cap = bt.shape[1] * page_size
    o = np.zeros((B, H, Nq, d))
    lse = np.full((B, H, Nq), -np.inf)
    for b in range(B):
        L = int(min(max(int(sl[b]), 0), cap))
        if L == 0:
            continue
        pages = bt[b, :(L + page_size - 1) // page_size]
        for kvh in range(Hkv):
            keys = np.concatenate([_f64(kc[p, kvh]) for p in pages], axis=0)[:L]
            vals = np.concatenate([_f64(vc[p, kvh]) for p in pages], axis=0)[:L]
            for h in range(kvh * (H // Hkv), (kvh + 1) * (H // Hkv)):
                pos = [L - Nq + i for i in range(Nq)]
                live = [i for i in range(Nq) if pos[i] >= 0]
                if not live:
                    continue
                qf = np.zeros((L, d))
                for i in live:
                    qf[pos[i]] = q[b, h, i]
                ob, lb = attn_fwd_rows(qf, keys, vals, scale, [pos[i] for i in live], causal=True, lib=lib)
                for n, i in enumerate(live):
                    o[b, h, i] = ob[n]
                    lse[b, h, i] = lb[n]
    return o, lse
