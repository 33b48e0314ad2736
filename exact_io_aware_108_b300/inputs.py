"""Seeded synthetic inputs for the attention workloads (no attention math).

This module is the only code shared by the CUDA path's tests/bench and the
oracle's callers: it draws random tensors and masks and nothing else.

Recipe (the pages name BERT-large seq 512, GPT-2 seq 1K, Long-Range-Arena
1K-4K, Path-X 16K; these seeded tensors stand in for those workloads):
  * ``torch.Generator('cpu').manual_seed(seed)``; q, k, v, dO drawn in that
    order with ``torch.randn(shape, dtype=float32)`` then cast (round to
    nearest even) to fp16 / bf16;
  * optional multiplier on q and k after the cast (2 for the long-context
    sweep; exact, a power of two);
  * key-padding lengths ``torch.randint(lo, hi + 1, (B,))`` from the same
    generator, drawn after dO;
  * block mask ``torch.rand(nb, nb) < p`` from its own generator
    (``manual_seed(mask_seed)``), diagonal forced to keep;
  * paged decode: q, then the key and value page pools, drawn as above;
    context lengths randint(lo, hi + 1); the block table a random
    permutation of the pool's pages (torch.randperm);
  * 8-bit inputs: q, k, v drawn as above in fp32, each divided by its own
    power-of-two factor 2^ceil(log2(max|x| / 448)) and cast to
    ``torch.float8_e4m3fn`` (round to nearest even; no value reaches the
    448 limit); the factor is returned as the tensor's dequantisation
    factor, and ``dequant`` gives the exact real values (fp64).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

BLOCK = 128


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    dtype: str            # "f16" | "bf16" | "e4m3" (8-bit q, k, v; bf16 O)
    causal: bool = False
    kv_len_range: tuple | None = None   # (lo, hi) inclusive
    block_sparse_p: float | None = None
    mask_seed: int = 7
    qk_mult: float = 1.0
    seed: int = 0
    backward: bool = True
    hkv: int | None = None            # key/value heads (grouped-query attention), None = H
    num_splits: int | None = None     # split-KV forward (0 = the library's choice), None = off
    nq: int | None = None             # paged decode: new tokens per sequence (N = longest context)
    page_size: int = 0                # paged decode: keys per cache page
    notes: str = field(default="", compare=False)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def torch_dtype(self):
        if self.dtype == "e4m3":
            return torch.float8_e4m3fn
        return torch.float16 if self.dtype == "f16" else torch.bfloat16


# The five workloads of the method's evaluation, as synthetic stand-ins.
WORKLOADS = {
    "fwd_b1_h2_n256_d64_f16": Workload("fwd_b1_h2_n256_d64_f16", 1, 2, 256, 64, "f16",
                                       backward=False),
    "bert_b16_h16_n512_d64_f16_kvlen": Workload(
        "bert_b16_h16_n512_d64_f16_kvlen", 16, 16, 512, 64, "f16", kv_len_range=(256, 512)),
    "gpt2_b8_h12_n1024_d64_bf16_causal": Workload(
        "gpt2_b8_h12_n1024_d64_bf16_causal", 8, 12, 1024, 64, "bf16", causal=True),
    "long_b8_h16_n4096_d128_bf16_causal": Workload(
        "long_b8_h16_n4096_d128_bf16_causal", 8, 16, 4096, 128, "bf16", causal=True, qk_mult=2.0),
    "long_b4_h16_n8192_d128_bf16_causal": Workload(
        "long_b4_h16_n8192_d128_bf16_causal", 4, 16, 8192, 128, "bf16", causal=True, qk_mult=2.0),
    "long_b2_h16_n16384_d128_bf16_causal": Workload(
        "long_b2_h16_n16384_d128_bf16_causal", 2, 16, 16384, 128, "bf16", causal=True,
        qk_mult=2.0),
    "blocksparse_b2_h8_n16384_d64_f16": Workload(
        "blocksparse_b2_h8_n16384_d64_f16", 2, 8, 16384, 64, "f16", block_sparse_p=0.2),
    # grouped-query attention (32 query heads sharing 8 key/value heads)
    "gqa_b4_h32_hkv8_n4096_d128_bf16_causal": Workload(
        "gqa_b4_h32_hkv8_n4096_d128_bf16_causal", 4, 32, 4096, 128, "bf16", causal=True, hkv=8,
        qk_mult=2.0),
    # the N = 8192 long-context point with 8-bit q, k, v
    "fp8_b4_h16_n8192_d128_e4m3_causal": Workload(
        "fp8_b4_h16_n8192_d128_e4m3_causal", 4, 16, 8192, 128, "e4m3", causal=True, backward=False),
    # serving-shaped decode: 32 sequences of 4K-8K cached tokens in 16-token
    # pages, 32 query heads on 8 key/value heads, one new token each
    "decode_b32_h32_hkv8_nq1_ctx4k8k_d128_bf16_page16": Workload(
        "decode_b32_h32_hkv8_nq1_ctx4k8k_d128_bf16_page16", 32, 32, 8192, 128, "bf16",
        kv_len_range=(4096, 8192), hkv=8, nq=1, page_size=16, backward=False, num_splits=0),
    # one long head: 64 query tiles cannot fill 148 SMs without splitting the keys
    "splitkv_b1_h1_n8192_d128_bf16": Workload(
        "splitkv_b1_h1_n8192_d128_bf16", 1, 1, 8192, 128, "bf16", qk_mult=2.0, backward=False,
        num_splits=0),
}


def make_qkv(B, H, N, d, dtype, seed=0, qk_mult=1.0, with_dout=True,
             kv_len_range=None, hkv=None):
    """Draw q, k, v (and dO, kv_len) on the CPU. Returns a dict of tensors.
    hkv: number of key/value heads (k, v are [B, hkv, N, d]); None = H."""
    tdt = torch.float16 if dtype in ("f16", torch.float16) else torch.bfloat16
    g = torch.Generator(device="cpu").manual_seed(seed)
    shape = (B, H, N, d)
    kv_shape = (B, H if hkv is None else hkv, N, d)
    q = torch.randn(shape, generator=g, dtype=torch.float32).to(tdt)
    k = torch.randn(kv_shape, generator=g, dtype=torch.float32).to(tdt)
    v = torch.randn(kv_shape, generator=g, dtype=torch.float32).to(tdt)
    out = {"q": q, "k": k, "v": v}
    if with_dout or kv_len_range is not None:
        out["dout"] = torch.randn(shape, generator=g, dtype=torch.float32).to(tdt)
    if kv_len_range is not None:
        lo, hi = kv_len_range
        out["kv_len"] = torch.randint(lo, hi + 1, (B,), generator=g, dtype=torch.int64).to(
            torch.int32)
    if qk_mult != 1.0:
        out["q"] = out["q"] * qk_mult
        out["k"] = out["k"] * qk_mult
    return out


def make_block_mask(N, p, seed=7, block=BLOCK):
    """uint8 [nb, nb] keep-mask: Bernoulli(p) off the diagonal, diagonal kept."""
    nb = (N + block - 1) // block
    g = torch.Generator(device="cpu").manual_seed(seed)
    m = torch.rand((nb, nb), generator=g) < p
    m.fill_diagonal_(True)
    return m.to(torch.uint8)


def _to_e4m3(x):
    amax = float(x.abs().max())
    e = math.ceil(math.log2(amax / 448.0)) if amax > 0 else 0
    descale = 2.0 ** e
    q8 = (x / descale).to(torch.float8_e4m3fn)
    return q8, descale


def make_qkv_fp8(B, H, N, d, seed=0, hkv=None, kv_len_range=None):
    """8-bit q, k, v (float8_e4m3fn) and their dequantisation factors
    q_descale, k_descale, v_descale (powers of two)."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    kv_shape = (B, H if hkv is None else hkv, N, d)
    out = {}
    for name, shape in (("q", (B, H, N, d)), ("k", kv_shape), ("v", kv_shape)):
        out[name], out[name + "_descale"] = _to_e4m3(torch.randn(shape, generator=g, dtype=torch.float32))
    if kv_len_range is not None:
        lo, hi = kv_len_range
        out["kv_len"] = torch.randint(lo, hi + 1, (B,), generator=g, dtype=torch.int64).to(torch.int32)
    return out


def make_paged_decode(B, H, Hkv, Nq, d, dtype, page_size, ctx_range, seed=0, spare_pages=0):
    """Decode inputs over a paged cache: q [B,H,Nq,d]; k_cache, v_cache
    [num_pages, Hkv, page_size, d] drawn N(0,1) and cast like make_qkv;
    seq_len int32 [B] = randint(lo, hi + 1); block_table int32 [B,
    pages_per_seq] (pages_per_seq = ceil(hi / page_size)) holding a random
    permutation of the pool, whose size is B * pages_per_seq + spare_pages
    (pages no sequence uses)."""
    tdt = torch.float16 if dtype in ("f16", torch.float16) else torch.bfloat16
    g = torch.Generator(device="cpu").manual_seed(seed)
    lo, hi = ctx_range
    pages_per_seq = -(-hi // page_size)
    num_pages = B * pages_per_seq + spare_pages
    q = torch.randn((B, H, Nq, d), generator=g, dtype=torch.float32).to(tdt)
    k = torch.randn((num_pages, Hkv, page_size, d), generator=g, dtype=torch.float32).to(tdt)
    v = torch.randn((num_pages, Hkv, page_size, d), generator=g, dtype=torch.float32).to(tdt)
    seq_len = torch.randint(lo, hi + 1, (B,), generator=g, dtype=torch.int64).to(torch.int32)
    perm = torch.randperm(num_pages, generator=g)[: B * pages_per_seq]
    block_table = perm.reshape(B, pages_per_seq).to(torch.int32)
    return {"q": q, "k_cache": k, "v_cache": v, "seq_len": seq_len, "block_table": block_table,
            "page_size": page_size}


def dequant(x8, descale):
    """Real values of an e4m3 tensor (exact in fp64)."""
    return x8.to(torch.float64) * descale


def make_workload(w: Workload, with_dout=None):
    """All inputs of a named workload (CPU tensors)."""
    if with_dout is None:
        with_dout = w.backward
    if w.nq is not None:
        return make_paged_decode(w.B, w.H, w.hkv or w.H, w.nq, w.d, w.dtype, w.page_size, w.kv_len_range,
                                 seed=w.seed)
    if w.dtype == "e4m3":
        return make_qkv_fp8(w.B, w.H, w.N, w.d, seed=w.seed, hkv=w.hkv, kv_len_range=w.kv_len_range)
    t = make_qkv(w.B, w.H, w.N, w.d, w.dtype, seed=w.seed, qk_mult=w.qk_mult,
                 with_dout=with_dout, kv_len_range=w.kv_len_range, hkv=w.hkv)
    if w.block_sparse_p is not None:
        t["block_mask"] = make_block_mask(w.N, w.block_sparse_p, seed=w.mask_seed)
    return t


def head_slice(t, b, h):
    """[N, d] view of one head of a [B, H, N, d] tensor."""
    return t[b, h]
