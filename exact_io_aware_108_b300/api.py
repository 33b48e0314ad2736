"""Convenience wrappers: allocate outputs with torch, then call the C ABI."""
from __future__ import annotations

import math

import torch

from . import _binding as B


def attention_forward(q, k, v, scale=None, causal=False, kv_len=None, block_mask=None,
                      return_residual=False, num_splits=None, stream=None):
    """O [B,H,N,d] and LSE [B,H,N] fp32 of exact attention (device tensors).

    k and v may have fewer heads than q (grouped-query attention: [B,Hkv,N,d]
    with H a multiple of Hkv). With return_residual=True also returns O's
    rounding residual (same dtype), which attention_backward uses for a more
    accurate D = rowsum(dO * O). num_splits (not with block_mask) selects the
    split-KV forward: the key tiles of each query tile shared by that many
    CTAs (0: the library's choice)."""
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[-1])
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device)
    o_res = torch.empty_like(q) if return_residual else None
    if num_splits is not None:
        if block_mask is not None:
            raise ValueError("num_splits does not combine with block_mask")
        Bsz, H, N, d = q.shape
        ws_bytes = B.fa_fwd_splitkv_workspace_size(Bsz, H, N, d, causal, num_splits)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device) if ws_bytes else None
        B.fa_fwd_splitkv(q, k, v, o, lse, scale, causal, kv_len, o_res=o_res, num_splits=num_splits,
                         workspace=ws, stream=stream)
    elif block_mask is not None:
        B.fa_fwd_blocksparse(q, k, v, o, lse, scale, block_mask, o_res=o_res, stream=stream)
    elif k.shape[1] != q.shape[1]:
        B.fa_fwd_gqa(q, k, v, o, lse, scale, causal, kv_len, o_res=o_res, stream=stream)
    elif kv_len is not None or o_res is not None:
        B.fa_fwd_ex(q, k, v, o, lse, scale, causal, kv_len, o_res=o_res, stream=stream)
    else:
        B.fa_fwd(q, k, v, o, lse, scale, causal, stream=stream)
    return (o, lse, o_res) if return_residual else (o, lse)


def attention_forward_fp8(q, k, v, q_descale, k_descale, v_descale, scale=None, causal=False,
                          kv_len=None, stream=None):
    """O [B,H,N,d] bf16 and LSE [B,H,N] fp32 of exact attention on 8-bit
    inputs: q [B,H,N,128], k, v [B,Hkv,N,128] torch.float8_e4m3fn device
    tensors whose real values are descale x stored (per-tensor factors)."""
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[-1])
    Bsz, H, N, d = q.shape
    o = torch.empty(q.shape, dtype=torch.bfloat16, device=q.device)
    lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device)
    ws = torch.empty(max(1, B.fa_fwd_fp8_workspace_size(Bsz, k.shape[1], N, d)), dtype=torch.uint8,
                     device=q.device)
    B.fa_fwd_fp8(q, k, v, o, lse, scale, q_descale, k_descale, v_descale, causal, kv_len,
                 workspace=ws, stream=stream)
    return o, lse


def attention_decode_paged(q, k_cache, v_cache, block_table, seq_len, scale=None, num_splits=0,
                           stream=None):
    """O [B,H,Nq,d] and LSE [B,H,Nq] of the Nq newest tokens of B sequences
    against their paged key/value cache (k_cache, v_cache [num_pages, Hkv,
    page_size, d]; block_table int32 [B, pages_per_seq]; seq_len int32 [B]).
    num_splits: key tiles of a sequence shared by that many CTAs (0: the
    library's choice)."""
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[-1])
    Bsz, H, Nq, d = q.shape
    num_pages, Hkv, page_size, _ = k_cache.shape
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device)
    ws_bytes = B.fa_decode_paged_workspace_size(Bsz, H, Hkv, Nq, d, page_size, block_table.shape[1],
                                                num_splits)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device) if ws_bytes else None
    B.fa_decode_paged(q, k_cache, v_cache, block_table, seq_len, o, lse, scale, num_splits=num_splits,
                      workspace=ws, stream=stream)
    return o, lse


def attention_backward(q, k, v, o, lse, dout, scale=None, causal=False, kv_len=None,
                       block_mask=None, o_res=None, workspace=None, stream=None):
    """dQ, dK, dV of exact attention (device tensors); dK and dV have k's shape
    (grouped-query attention: summed over each group of query heads)."""
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[-1])
    Bsz, H, N, d = q.shape
    ws_bytes = B.fa_bwd_workspace_size(Bsz, H, N, d)
    if workspace is None or workspace.numel() * workspace.element_size() < ws_bytes:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    dq = torch.empty_like(q)
    dk = torch.empty_like(k)
    dv = torch.empty_like(v)
    if block_mask is not None:
        B.fa_bwd_blocksparse(q, k, v, o, lse, dout, dq, dk, dv, scale, block_mask, o_res=o_res,
                             workspace=workspace, stream=stream)
    elif k.shape[1] != q.shape[1]:
        B.fa_bwd_gqa(q, k, v, o, lse, dout, dq, dk, dv, scale, causal, kv_len, o_res=o_res,
                     workspace=workspace, stream=stream)
    else:
        B.fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, scale, causal, kv_len, o_res=o_res,
                 workspace=workspace, stream=stream)
    return dq, dk, dv
