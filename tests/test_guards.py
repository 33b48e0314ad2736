"""Guard bands around every output and workspace (memory-safety checks that
need no sanitizer).

Each output and workspace is a view into a larger device buffer whose bytes
before and after the view hold a known pattern; the output bytes themselves
start as NaN. After the call, every guard byte must be unchanged (nothing
wrote past either end), and every output element must have been written
(no NaN left where the result is finite). Ragged sequence lengths (1, 129,
300, 4500) leave partial tiles at the end of every head, where an off-by-one
in a tile's row count or a TMA box would land in the next head or past the
buffer.
"""
import math

import pytest
import torch

from exact_io_aware_108_b300 import inputs

pytestmark = pytest.mark.gpu

GUARD = 4096          # bytes before and after each view (keeps 256-byte alignment)
PATTERN = 0xA5


class Guarded:
    """A view of `nbytes` (then shaped as dtype/shape) inside a guarded buffer."""

    def __init__(self, shape, dtype, nbytes=None, fill=0xFF):
        elem = torch.empty((), dtype=dtype).element_size()
        n = int(math.prod(shape)) * elem if nbytes is None else nbytes
        self.n = n
        self.buf = torch.full((GUARD + n + GUARD,), PATTERN, dtype=torch.uint8, device="cuda")
        self.buf[GUARD:GUARD + n].fill_(fill)
        raw = self.buf[GUARD:GUARD + n]
        self.view = raw.view(dtype).view(shape) if nbytes is None else raw

    def check(self, name):
        head = self.buf[:GUARD]
        tail = self.buf[GUARD + self.n:]
        assert torch.all(head == PATTERN), f"{name}: bytes before the buffer were written"
        assert torch.all(tail == PATTERN), f"{name}: bytes after the buffer were written"


def _qkv(B, H, N, d, dt, seed, hkv=None):
    t = inputs.make_qkv(B, H, N, d, dt, seed=seed, hkv=hkv)
    return {n: x.cuda() for n, x in t.items()}


SHAPES = [(1, 64), (129, 128), (300, 64), (4500, 128)]


@pytest.mark.parametrize("N,d", SHAPES)
@pytest.mark.parametrize("causal", [False, True])
def test_forward_and_backward_stay_inside_their_buffers(N, d, causal):
    import exact_io_aware_108_b300 as fa
    B, H = 2, 3
    t = _qkv(B, H, N, d, "bf16", seed=N + d)
    q, k, v, do = t["q"], t["k"], t["v"], t["dout"]
    scale = 1.0 / math.sqrt(d)
    o = Guarded(q.shape, q.dtype)
    res = Guarded(q.shape, q.dtype)
    lse = Guarded(q.shape[:-1], torch.float32)
    fa.fa_fwd_ex(q, k, v, o.view, lse.view, scale, causal, None, o_res=res.view)
    torch.cuda.synchronize()
    assert fa.fa_get_device_error() == 0
    for name, g in (("o", o), ("o_res", res), ("lse", lse)):
        g.check(name)
    assert torch.isfinite(o.view).all() and torch.isfinite(res.view).all()
    assert torch.isfinite(lse.view).all()
    wsb = fa.fa_bwd_workspace_size(B, H, N, d)
    ws = Guarded(None, torch.uint8, nbytes=wsb, fill=0x7F)
    grads = [Guarded(x.shape, x.dtype) for x in (q, k, v)]
    fa.fa_bwd(q, k, v, o.view, lse.view, do, *(g.view for g in grads), scale, causal, None,
              res.view, ws.view, wsb)
    torch.cuda.synchronize()
    assert fa.fa_get_device_error() == 0
    ws.check("workspace")
    for name, g in zip(("dq", "dk", "dv"), grads):
        g.check(name)
        assert torch.isfinite(g.view).all(), name


@pytest.mark.parametrize("N,d", SHAPES)
def test_blocksparse_stays_inside_its_buffers(N, d):
    import exact_io_aware_108_b300 as fa
    Np = (N + 127) // 128 * 128  # the block-sparse calls take whole tiles
    B, H = 1, 2
    t = _qkv(B, H, Np, d, "f16", seed=Np + 1)
    q, k, v, do = t["q"], t["k"], t["v"], t["dout"]
    bm = inputs.make_block_mask(Np, 0.5, seed=5).cuda()
    o = Guarded(q.shape, q.dtype)
    lse = Guarded(q.shape[:-1], torch.float32)
    fa.fa_fwd_blocksparse(q, k, v, o.view, lse.view, 0.1, bm)
    wsb = fa.fa_bwd_workspace_size(B, H, Np, d)
    ws = Guarded(None, torch.uint8, nbytes=wsb, fill=0x7F)
    grads = [Guarded(x.shape, x.dtype) for x in (q, k, v)]
    fa.fa_bwd_blocksparse(q, k, v, o.view, lse.view, do, *(g.view for g in grads), 0.1, bm, None,
                          ws.view, wsb)
    torch.cuda.synchronize()
    assert fa.fa_get_device_error() == 0
    for name, g in (("o", o), ("lse", lse), ("workspace", ws), ("dq", grads[0]), ("dk", grads[1]),
                    ("dv", grads[2])):
        g.check(name)


@pytest.mark.parametrize("N,d", SHAPES)
def test_splitkv_stays_inside_its_buffers(N, d):
    import exact_io_aware_108_b300 as fa
    B, H, Hkv = 1, 4, 2
    t = _qkv(B, H, N, d, "bf16", seed=N + 3, hkv=Hkv)
    q, k, v = t["q"], t["k"], t["v"]
    S = 3
    o = Guarded(q.shape, q.dtype)
    res = Guarded(q.shape, q.dtype)
    lse = Guarded(q.shape[:-1], torch.float32)
    wsb = fa.fa_fwd_splitkv_workspace_size(B, H, N, d, True, S)
    ws = Guarded(None, torch.uint8, nbytes=max(wsb, 256), fill=0x7F)
    fa.fa_fwd_splitkv(q, k, v, o.view, lse.view, 0.1, True, None, o_res=res.view, num_splits=S,
                      workspace=ws.view, workspace_bytes=wsb)
    torch.cuda.synchronize()
    assert fa.fa_get_device_error() == 0
    for name, g in (("o", o), ("o_res", res), ("lse", lse), ("workspace", ws)):
        g.check(name)
    assert torch.isfinite(o.view).all()


@pytest.mark.parametrize("N", [1, 129, 300, 4500])
def test_fp8_stays_inside_its_buffers(N):
    import exact_io_aware_108_b300 as fa
    w = inputs.Workload("fp8_guard", 1, 2, N, 128, "e4m3", causal=True, backward=False)
    t = {n: (x.cuda() if torch.is_tensor(x) else x) for n, x in inputs.make_workload(w).items()}
    o = Guarded(t["q"].shape, torch.bfloat16)
    lse = Guarded(t["q"].shape[:-1], torch.float32)
    wsb = fa.fa_fwd_fp8_workspace_size(1, 2, N, 128)
    ws = Guarded(None, torch.uint8, nbytes=wsb, fill=0x7F)
    fa.fa_fwd_fp8(t["q"], t["k"], t["v"], o.view, lse.view, w.scale, t["q_descale"], t["k_descale"],
                  t["v_descale"], True, None, workspace=ws.view, workspace_bytes=wsb)
    torch.cuda.synchronize()
    assert fa.fa_get_device_error() == 0
    for name, g in (("o", o), ("lse", lse), ("workspace", ws)):
        g.check(name)
    assert torch.isfinite(o.view).all()


@pytest.mark.parametrize("d,page_size", [(64, 16), (128, 64)])
def test_decode_stays_inside_its_buffers(d, page_size):
    import exact_io_aware_108_b300 as fa
    w = inputs.Workload("decode_guard", 3, 8, 700, d, "bf16", kv_len_range=(1, 700), hkv=2, nq=3,
                        page_size=page_size, backward=False, num_splits=2)
    t = {n: (x.cuda() if torch.is_tensor(x) else x) for n, x in inputs.make_workload(w).items()}
    o = Guarded(t["q"].shape, t["q"].dtype)
    lse = Guarded(t["q"].shape[:-1], torch.float32)
    pps = t["block_table"].shape[1]
    wsb = fa.fa_decode_paged_workspace_size(3, 8, 2, 3, d, page_size, pps, 2)
    ws = Guarded(None, torch.uint8, nbytes=max(wsb, 256), fill=0x7F)
    fa.fa_decode_paged(t["q"], t["k_cache"], t["v_cache"], t["block_table"], t["seq_len"], o.view,
                       lse.view, w.scale, num_splits=2, workspace=ws.view, workspace_bytes=wsb)
    torch.cuda.synchronize()
    assert fa.fa_get_device_error() == 0
    for name, g in (("o", o), ("lse", lse), ("workspace", ws)):
        g.check(name)
