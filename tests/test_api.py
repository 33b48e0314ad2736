"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every function include/fa.h declares, and rejects bad arguments before any
launch."""
import ctypes
import os
import re

import pytest

import exact_io_aware_108_b300 as fa
from exact_io_aware_108_b300 import _binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "fa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z_0-9]+)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    lib = fa.load_library()
    declared = _declared()
    assert declared, "no declarations parsed"
    missing = [n for n in declared if not hasattr(lib, n)]
    assert not missing, missing
    assert sorted(_binding.EXPORTS) == declared


def test_status_strings_and_version():
    assert fa.fa_status_str(0) == "FA_OK"
    assert fa.fa_status_str(4) == "FA_ERR_TIMEOUT"
    assert fa.fa_status_str(5) == "FA_ERR_RANGE"
    assert re.match(r"^\d+\.\d+\.\d+$", fa.fa_version())


def test_workspace_size():
    def up(x):
        return (x + 255) // 256 * 256
    rows = 2 * 3 * 384  # query rows padded to whole 128-row tiles
    elems = 2 * 3 * 300 * 64  # fp16 copies of Q and of the scaled dO (bf16 inputs)
    assert fa.fa_bwd_workspace_size(2, 3, 300, 64) == (2 * up(rows * 4) + up(rows * 64 * 4) + 256
                                                      + 2 * up(elems * 2))
    assert fa.fa_bwd_workspace_size(1, 1, 1, 96) == 0
    assert fa.fa_bwd_workspace_size(0, 1, 1, 64) == 0


FAKE = 1 << 20  # an aligned non-null address that is never dereferenced


def _fwd(lib, q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, B=1, H=1, N=128, d=64, scale=0.125,
         causal=0, dt=0):
    return lib.fa_fwd(q, k, v, o, lse, B, H, N, d, ctypes.c_float(scale), causal, dt, None)


@pytest.mark.parametrize("kw,status", [
    ({"q": None}, 1), ({"o": None}, 1), ({"lse": None}, 1),
    ({"k": FAKE + 8}, 1),
    ({"B": 0}, 1), ({"N": 0}, 1), ({"H": -1}, 1), ({"d": 0}, 1),
    ({"d": 96}, 2), ({"d": 256}, 2),
    ({"scale": 0.0}, 1), ({"scale": float("nan")}, 1), ({"scale": -1.0}, 1),
    ({"dt": 7}, 1),
    ({"B": 70000, "H": 70000, "N": 1 << 20}, 1),
])
def test_fwd_rejects_bad_arguments(kw, status):
    lib = fa.load_library()
    assert _fwd(lib, **kw) == status
    assert fa.fa_last_error_message() != ""


def test_bwd_rejects_bad_arguments():
    lib = fa.load_library()
    c = ctypes.c_float(0.125)
    args = [FAKE] * 9
    # workspace too small
    st = lib.fa_bwd(*args, 1, 1, 128, 64, c, 0, 0, None, None, FAKE, 16, None)
    assert st == 1
    # null dq
    a2 = list(args)
    a2[6] = None
    st = lib.fa_bwd(*a2, 1, 1, 128, 64, c, 0, 0, None, None, FAKE, 1 << 30, None)
    assert st == 1
    # misaligned residual
    st = lib.fa_bwd(*args, 1, 1, 128, 64, c, 0, 0, None, FAKE + 2, FAKE, 1 << 30, None)
    assert st == 1
    # block-sparse without a mask
    st = lib.fa_bwd_blocksparse(*args, 1, 1, 128, 64, c, 0, None, None, FAKE, 1 << 30, None)
    assert st == 1


def test_bwd_rejects_key_padding_with_a_block_mask():
    """No forward computes block-sparse attention with key padding, so the
    backward entry points that take both refuse the combination."""
    lib = fa.load_library()
    c = ctypes.c_float(0.125)
    st = lib.fa_bwd_main(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 256, 64, c, 0, 0, FAKE, FAKE,
                         FAKE, 1 << 30, None)
    assert st == 1 and "kv_len" in fa.fa_last_error_message()
    st = lib.fa_bwd_noalloc(*([FAKE] * 9), 1, 1, 256, 64, c, 0, 0, FAKE, FAKE, None, None)
    assert st == 1 and "kv_len" in fa.fa_last_error_message()
    # either one alone passes the argument checks of fa_bwd_main up to the
    # workspace test (too small here, so nothing is launched)
    st = lib.fa_bwd_main(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 256, 64, c, 0, 0, FAKE, None,
                         FAKE, 16, None)
    assert st == 1 and "workspace" in fa.fa_last_error_message()


def test_gqa_rejects_bad_head_counts():
    lib = fa.load_library()
    c = ctypes.c_float(0.125)
    for Hkv in (3, 0, 5):  # must divide H = 4 and lie in [1, H]
        st = lib.fa_fwd_gqa(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 4, Hkv, 128, 64, c, 0, 0, None, None,
                            None)
        assert st == 1
        st = lib.fa_bwd_gqa(*([FAKE] * 9), 1, 4, Hkv, 128, 64, c, 0, 0, None, None, FAKE, 1 << 30,
                            None)
        assert st == 1


def test_splitkv_sizes_and_argument_checks():
    lib = fa.load_library()
    c = ctypes.c_float(0.125)
    R = 1 * 2 * 8 * 128  # query rows padded to whole tiles (N = 1000)
    assert fa.fa_fwd_splitkv_workspace_size(1, 2, 1000, 128, False, 3) == 3 * R * 129 * 4
    assert fa.fa_fwd_splitkv_workspace_size(1, 2, 1000, 128, False, 1) == 0
    assert fa.fa_fwd_splitkv_num_splits(1, 2, 1000, 128, False, 5) == 5
    assert fa.fa_fwd_splitkv_num_splits(1, 2, 1000, 96, False, 5) == 0
    assert fa.fa_fwd_splitkv_num_splits(1, 2, 1000, 128, False, 257) == 0
    # the library's choice: >= 2 shares when one head cannot fill the SMs,
    # none for a grid of thousands of CTAs, never more than the key tiles
    for causal in (False, True):
        s = fa.fa_fwd_splitkv_num_splits(1, 1, 8192, 128, causal, 0)
        assert 2 <= s <= 64
        assert fa.fa_fwd_splitkv_num_splits(16, 16, 4096, 128, causal, 0) == 1
    assert fa.fa_fwd_splitkv_num_splits(1, 1, 200, 64, False, 0) <= 2

    def call(num_splits, ws, ws_bytes, Hkv=2):
        return lib.fa_fwd_splitkv(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 2, Hkv, 1000, 128, c, 0, 1, None,
                                  None, num_splits, ws, ws_bytes, None)
    need = 4 * R * 129 * 4
    assert call(4, None, need) == 1             # workspace missing
    assert call(4, FAKE + 16, need) == 1        # not 256-byte aligned
    assert call(4, FAKE, need - 4) == 1         # too small
    assert call(300, FAKE, 1 << 40) == 1        # more than 256 shares
    assert call(4, FAKE, need, Hkv=3) == 1      # Hkv must divide H
    assert call(4, FAKE, need, Hkv=0) == 1


def test_fp8_sizes_and_argument_checks():
    lib = fa.load_library()
    assert fa.fa_fwd_fp8_workspace_size(2, 3, 300, 128) == 2 * 3 * 128 * 384
    assert fa.fa_fwd_fp8_workspace_size(2, 3, 300, 64) == 0
    f = ctypes.c_float

    def call(d=128, H=2, Hkv=2, qd=1.0, kd=1.0, vd=1.0, ws=FAKE, ws_bytes=1 << 30, q=FAKE):
        return lib.fa_fwd_fp8(q, FAKE, FAKE, FAKE, FAKE, 1, H, Hkv, 256, d, f(0.1), 0, f(qd), f(kd), f(vd),
                              None, ws, ws_bytes, None)
    assert call(d=64) == 2                       # only d = 128 is built
    assert call(qd=0.0) == 1 and call(kd=-1.0) == 1 and call(vd=float("inf")) == 1
    assert call(ws=None) == 1                    # workspace missing
    assert call(ws=FAKE + 64) == 1               # not 256-byte aligned
    assert call(ws_bytes=2 * 128 * 256 - 1) == 1 # too small
    assert call(Hkv=3) == 1 and call(Hkv=0) == 1
    assert call(q=FAKE + 8) == 1                 # q not 16-byte aligned


def test_decode_sizes_and_argument_checks():
    lib = fa.load_library()
    # R = 4 query rows per (b, kv head) -> one 128-row tile; 3 shares
    assert fa.fa_decode_paged_workspace_size(2, 8, 2, 1, 128, 16, 64, 3) == 3 * 2 * 2 * 128 * 129 * 4
    assert fa.fa_decode_paged_workspace_size(2, 8, 2, 1, 128, 16, 64, 1) == 0
    assert fa.fa_decode_paged_num_splits(2, 8, 2, 1, 128, 16, 64, 5) == 5
    assert fa.fa_decode_paged_num_splits(2, 8, 2, 1, 128, 24, 64, 5) == 0   # page size not built
    assert 2 <= fa.fa_decode_paged_num_splits(1, 8, 8, 1, 128, 16, 512, 0) <= 64
    f = ctypes.c_float

    def call(H=8, Hkv=2, Nq=1, d=128, ps=16, num_pages=64, pps=8, bt=FAKE, sl=FAKE, S=1, ws=None, wsb=0):
        return lib.fa_decode_paged(FAKE, FAKE, FAKE, bt, sl, FAKE, FAKE, 2, H, Hkv, Nq, d, ps, num_pages, pps,
                                   f(0.1), 1, S, ws, wsb, None)
    assert call(ps=8) == 2 and call(ps=256) == 2 and call(d=96) == 2
    assert call(Hkv=3) == 1 and call(Nq=0) == 1 and call(num_pages=0) == 1 and call(pps=0) == 1
    assert call(bt=None) == 1 and call(sl=FAKE + 2) == 1
    assert call(S=4) == 1                        # shares need a workspace
    assert call(S=4, ws=FAKE + 16, wsb=1 << 30) == 1


def test_blocksparse_rejects_missing_mask():
    lib = fa.load_library()
    st = lib.fa_fwd_blocksparse(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 256, 64, ctypes.c_float(0.1), 0,
                                None, None, None)
    assert st == 1


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(_binding, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(_binding, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        _binding.load_library()
