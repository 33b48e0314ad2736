"""ctypes binding of libfa.so: the C ABI of include/fa.h, same names.

Argument marshalling only: tensors become device pointers and sizes, the
stream becomes a cudaStream_t handle. Every step of the computation runs in
the library's CUDA kernels; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libfa.so")

FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED, FA_ERR_CUDA, FA_ERR_TIMEOUT = range(5)
FA_F16, FA_BF16 = 0, 1

# every symbol include/fa.h declares
EXPORTS = (
    "fa_fwd", "fa_fwd_ex", "fa_fwd_blocksparse", "fa_fwd_gqa", "fa_fwd_splitkv", "fa_fwd_splitkv_num_splits",
    "fa_fwd_splitkv_workspace_size", "fa_fwd_fp8", "fa_fwd_fp8_workspace_size", "fa_bwd_workspace_size",
    "fa_decode_paged", "fa_decode_paged_num_splits", "fa_decode_paged_workspace_size", "fa_bwd",
    "fa_bwd_gqa", "fa_bwd_blocksparse", "fa_bwd_prepare", "fa_bwd_main", "fa_bwd_finish", "fa_bwd_noalloc",
    "fa_bwd_noalloc_max_workspace",
    "fa_get_device_error", "fa_set_wait_limit_ns", "fa_debug_starve_pipelines", "fa_status_str",
    "fa_last_error_message", "fa_version",
)

_lock = threading.Lock()
_lib = None

_vp = ctypes.c_void_p
_i = ctypes.c_int
_f = ctypes.c_float
_sz = ctypes.c_size_t


class FAError(RuntimeError):
    def __init__(self, status: int, func: str, detail: str):
        self.status = status
        super().__init__(f"{func} failed: {_STATUS_NAMES.get(status, status)}: {detail}")


_STATUS_NAMES = {0: "FA_OK", 1: "FA_ERR_INVALID_ARG", 2: "FA_ERR_UNSUPPORTED",
                 3: "FA_ERR_CUDA", 4: "FA_ERR_TIMEOUT"}


def library_path() -> str:
    return LIB_PATH


def load_library():
    """Load libfa.so (raises if it was not built: no fallback exists)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with `python -m exact_io_aware_108_b300.build`")
        lib = ctypes.CDLL(LIB_PATH)
        fwd = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _i]
        lib.fa_fwd.argtypes = fwd + [_vp]
        lib.fa_fwd_ex.argtypes = fwd + [_vp, _vp, _vp]
        lib.fa_fwd_blocksparse.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _vp, _vp,
                                           _vp]
        lib.fa_fwd_gqa.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i, _i, _vp, _vp,
                                   _vp]
        lib.fa_fwd_splitkv.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i, _i, _vp, _vp,
                                       _i, _vp, _sz, _vp]
        lib.fa_fwd_splitkv_num_splits.argtypes = [_i, _i, _i, _i, _i, _i]
        lib.fa_fwd_splitkv_num_splits.restype = _i
        lib.fa_fwd_splitkv_workspace_size.argtypes = [_i, _i, _i, _i, _i, _i]
        lib.fa_fwd_splitkv_workspace_size.restype = _sz
        lib.fa_fwd_fp8.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i, _f, _f, _f, _vp, _vp,
                                   _sz, _vp]
        lib.fa_fwd_fp8_workspace_size.argtypes = [_i, _i, _i, _i]
        lib.fa_fwd_fp8_workspace_size.restype = _sz
        lib.fa_decode_paged.argtypes = [_vp] * 7 + [_i] * 8 + [_f, _i, _i, _vp, _sz, _vp]
        lib.fa_decode_paged_num_splits.argtypes = [_i] * 8
        lib.fa_decode_paged_num_splits.restype = _i
        lib.fa_decode_paged_workspace_size.argtypes = [_i] * 8
        lib.fa_decode_paged_workspace_size.restype = _sz
        lib.fa_bwd_workspace_size.argtypes = [_i, _i, _i, _i]
        lib.fa_bwd_workspace_size.restype = _sz
        bwd = [_vp] * 9 + [_i, _i, _i, _i, _f]
        lib.fa_bwd.argtypes = bwd + [_i, _i, _vp, _vp, _vp, _sz, _vp]
        lib.fa_bwd_blocksparse.argtypes = bwd + [_i, _vp, _vp, _vp, _sz, _vp]
        lib.fa_bwd_gqa.argtypes = [_vp] * 9 + [_i, _i, _i, _i, _i, _f, _i, _i, _vp, _vp, _vp, _sz, _vp]
        lib.fa_bwd_prepare.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp, _sz, _vp]
        lib.fa_bwd_main.argtypes = [_vp] * 6 + [_i, _i, _i, _i, _f, _i, _i, _vp, _vp, _vp, _sz, _vp]
        lib.fa_bwd_finish.argtypes = [_vp, _i, _i, _i, _i, _i, _vp, _sz, _vp]
        lib.fa_bwd_noalloc.argtypes = [_vp] * 9 + [_i, _i, _i, _i, _f, _i, _i, _vp, _vp, _vp, _vp]
        lib.fa_bwd_noalloc.restype = _i
        lib.fa_bwd_noalloc_max_workspace.argtypes = []
        lib.fa_bwd_noalloc_max_workspace.restype = _sz
        lib.fa_get_device_error.argtypes = [_vp]
        lib.fa_set_wait_limit_ns.argtypes = [ctypes.c_ulonglong]
        lib.fa_debug_starve_pipelines.argtypes = [_i]
        lib.fa_status_str.argtypes = [_i]
        lib.fa_status_str.restype = ctypes.c_char_p
        lib.fa_last_error_message.argtypes = []
        lib.fa_last_error_message.restype = ctypes.c_char_p
        lib.fa_version.argtypes = []
        lib.fa_version.restype = ctypes.c_char_p
        for name in ("fa_fwd", "fa_fwd_ex", "fa_fwd_blocksparse", "fa_fwd_gqa", "fa_fwd_splitkv", "fa_fwd_fp8",
                     "fa_decode_paged", "fa_bwd",
                     "fa_bwd_gqa",
                     "fa_bwd_blocksparse",
                     "fa_bwd_prepare", "fa_bwd_main", "fa_bwd_finish", "fa_get_device_error",
                     "fa_set_wait_limit_ns", "fa_debug_starve_pipelines"):
            getattr(lib, name).restype = _i
        _lib = lib
        return lib


def exported_symbols():
    """Names of include/fa.h that the loaded library resolves."""
    lib = load_library()
    return [n for n in EXPORTS if hasattr(lib, n)]


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float16:
        return FA_F16
    if t.dtype == torch.bfloat16:
        return FA_BF16
    raise TypeError(f"q must be float16 or bfloat16, got {t.dtype}")


def _check(status: int, func: str):
    if status != FA_OK:
        raise FAError(status, func, load_library().fa_last_error_message().decode())


def _dims(q):
    if q.dim() != 4:
        raise ValueError("q must be [B, H, N, d]")
    return tuple(int(x) for x in q.shape)


def fa_fwd(q, k, v, o, lse, scale, causal=False, stream=None):
    B, H, N, d = _dims(q)
    _check(load_library().fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d,
                                 float(scale), int(bool(causal)), _dtype_code(q), _stream(stream)),
           "fa_fwd")


def fa_fwd_ex(q, k, v, o, lse, scale, causal=False, kv_len=None, o_res=None, stream=None):
    B, H, N, d = _dims(q)
    _check(load_library().fa_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d,
                                    float(scale), int(bool(causal)), _dtype_code(q), _ptr(kv_len),
                                    _ptr(o_res), _stream(stream)),
           "fa_fwd_ex")


def fa_fwd_blocksparse(q, k, v, o, lse, scale, block_mask, o_res=None, stream=None):
    B, H, N, d = _dims(q)
    _check(load_library().fa_fwd_blocksparse(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H,
                                             N, d, float(scale), _dtype_code(q), _ptr(block_mask),
                                             _ptr(o_res), _stream(stream)),
           "fa_fwd_blocksparse")


def fa_fwd_gqa(q, k, v, o, lse, scale, causal=False, kv_len=None, o_res=None, stream=None):
    """q, o [B, H, N, d]; k, v [B, Hkv, N, d] (H a multiple of Hkv)."""
    B, H, N, d = _dims(q)
    Hkv = int(k.shape[1])
    _check(load_library().fa_fwd_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Hkv, N, d,
                                     float(scale), int(bool(causal)), _dtype_code(q), _ptr(kv_len),
                                     _ptr(o_res), _stream(stream)),
           "fa_fwd_gqa")


def fa_fwd_splitkv_num_splits(B, H, N, d, causal=False, num_splits=0) -> int:
    return int(load_library().fa_fwd_splitkv_num_splits(int(B), int(H), int(N), int(d), int(bool(causal)),
                                                         int(num_splits)))


def fa_fwd_splitkv_workspace_size(B, H, N, d, causal=False, num_splits=0) -> int:
    return int(load_library().fa_fwd_splitkv_workspace_size(int(B), int(H), int(N), int(d),
                                                            int(bool(causal)), int(num_splits)))


def fa_fwd_splitkv(q, k, v, o, lse, scale, causal=False, kv_len=None, o_res=None, num_splits=0,
                   workspace=None, workspace_bytes=None, stream=None):
    """q, o [B, H, N, d]; k, v [B, Hkv, N, d]; num_splits <= 0 lets the library choose."""
    B, H, N, d = _dims(q)
    Hkv = int(k.shape[1])
    _check(load_library().fa_fwd_splitkv(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Hkv, N, d,
                                         float(scale), int(bool(causal)), _dtype_code(q), _ptr(kv_len),
                                         _ptr(o_res), int(num_splits), _ptr(workspace),
                                         _ws_bytes(workspace, workspace_bytes), _stream(stream)),
           "fa_fwd_splitkv")


def fa_fwd_fp8_workspace_size(B, Hkv, N, d) -> int:
    return int(load_library().fa_fwd_fp8_workspace_size(int(B), int(Hkv), int(N), int(d)))


def fa_fwd_fp8(q, k, v, o, lse, scale, q_descale, k_descale, v_descale, causal=False, kv_len=None,
               workspace=None, workspace_bytes=None, stream=None):
    """q [B, H, N, d], k, v [B, Hkv, N, d] as float8_e4m3fn (real values = descale x stored);
    o [B, H, N, d] bf16; lse [B, H, N] fp32."""
    B, H, N, d = _dims(q)
    Hkv = int(k.shape[1])
    _check(load_library().fa_fwd_fp8(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Hkv, N, d,
                                     float(scale), int(bool(causal)), float(q_descale), float(k_descale),
                                     float(v_descale), _ptr(kv_len), _ptr(workspace),
                                     _ws_bytes(workspace, workspace_bytes), _stream(stream)),
           "fa_fwd_fp8")


def fa_decode_paged_num_splits(B, H, Hkv, Nq, d, page_size, pages_per_seq, num_splits=0) -> int:
    return int(load_library().fa_decode_paged_num_splits(int(B), int(H), int(Hkv), int(Nq), int(d),
                                                         int(page_size), int(pages_per_seq), int(num_splits)))


def fa_decode_paged_workspace_size(B, H, Hkv, Nq, d, page_size, pages_per_seq, num_splits=0) -> int:
    return int(load_library().fa_decode_paged_workspace_size(int(B), int(H), int(Hkv), int(Nq), int(d),
                                                             int(page_size), int(pages_per_seq),
                                                             int(num_splits)))


def fa_decode_paged(q, k_cache, v_cache, block_table, seq_len, o, lse, scale, num_splits=0, workspace=None,
                    workspace_bytes=None, stream=None):
    """q, o [B, H, Nq, d]; k_cache, v_cache [num_pages, Hkv, page_size, d]; block_table int32
    [B, pages_per_seq]; seq_len int32 [B]; lse [B, H, Nq] fp32."""
    B, H, Nq, d = _dims(q)
    num_pages, Hkv, page_size = (int(x) for x in k_cache.shape[:3])
    pages_per_seq = int(block_table.shape[1])
    _check(load_library().fa_decode_paged(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
                                          _ptr(seq_len), _ptr(o), _ptr(lse), B, H, Hkv, Nq, d, page_size,
                                          num_pages, pages_per_seq, float(scale), _dtype_code(q),
                                          int(num_splits), _ptr(workspace),
                                          _ws_bytes(workspace, workspace_bytes), _stream(stream)),
           "fa_decode_paged")


def fa_bwd_workspace_size(B, H, N, d) -> int:
    return int(load_library().fa_bwd_workspace_size(int(B), int(H), int(N), int(d)))


def fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, scale, causal=False, kv_len=None, o_res=None,
           workspace=None, workspace_bytes=None, stream=None):
    B, H, N, d = _dims(q)
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(load_library().fa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout),
                                 _ptr(dq), _ptr(dk), _ptr(dv), B, H, N, d, float(scale),
                                 int(bool(causal)), _dtype_code(q), _ptr(kv_len), _ptr(o_res),
                                 _ptr(workspace), int(workspace_bytes), _stream(stream)),
           "fa_bwd")


def fa_bwd_gqa(q, k, v, o, lse, dout, dq, dk, dv, scale, causal=False, kv_len=None, o_res=None,
               workspace=None, workspace_bytes=None, stream=None):
    """dq [B, H, N, d]; dk, dv [B, Hkv, N, d], summed over each group of query heads."""
    B, H, N, d = _dims(q)
    Hkv = int(k.shape[1])
    _check(load_library().fa_bwd_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout),
                                     _ptr(dq), _ptr(dk), _ptr(dv), B, H, Hkv, N, d, float(scale),
                                     int(bool(causal)), _dtype_code(q), _ptr(kv_len), _ptr(o_res),
                                     _ptr(workspace), _ws_bytes(workspace, workspace_bytes),
                                     _stream(stream)),
           "fa_bwd_gqa")


def fa_bwd_blocksparse(q, k, v, o, lse, dout, dq, dk, dv, scale, block_mask, o_res=None,
                       workspace=None, workspace_bytes=None, stream=None):
    B, H, N, d = _dims(q)
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(load_library().fa_bwd_blocksparse(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                             _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv), B, H, N, d,
                                             float(scale), _dtype_code(q), _ptr(block_mask),
                                             _ptr(o_res), _ptr(workspace), int(workspace_bytes),
                                             _stream(stream)),
           "fa_bwd_blocksparse")


def _ws_bytes(workspace, workspace_bytes):
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    return int(workspace_bytes)


def fa_bwd_prepare(q, v, o, o_res, lse, dout, workspace, workspace_bytes=None, stream=None):
    B, H, N, d = _dims(o)
    _check(load_library().fa_bwd_prepare(_ptr(q), _ptr(v), _ptr(o), _ptr(o_res), _ptr(lse), _ptr(dout), B, H, N,
                                         d, _dtype_code(o), _ptr(workspace),
                                         _ws_bytes(workspace, workspace_bytes), _stream(stream)),
           "fa_bwd_prepare")


def fa_bwd_main(q, k, v, dout, dk, dv, scale, causal=False, kv_len=None, block_mask=None,
                workspace=None, workspace_bytes=None, stream=None):
    B, H, N, d = _dims(q)
    _check(load_library().fa_bwd_main(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(dk), _ptr(dv),
                                      B, H, N, d, float(scale), int(bool(causal)), _dtype_code(q),
                                      _ptr(kv_len), _ptr(block_mask), _ptr(workspace),
                                      _ws_bytes(workspace, workspace_bytes), _stream(stream)),
           "fa_bwd_main")


def fa_bwd_finish(dq, workspace, workspace_bytes=None, stream=None):
    B, H, N, d = _dims(dq)
    _check(load_library().fa_bwd_finish(_ptr(dq), B, H, N, d, _dtype_code(dq), _ptr(workspace),
                                        _ws_bytes(workspace, workspace_bytes), _stream(stream)),
           "fa_bwd_finish")


def fa_bwd_noalloc(q, k, v, o, lse, dout, dq, dk, dv, scale, causal=False, kv_len=None,
                   block_mask=None, o_res=None, stream=None):
    """fa_bwd without a workspace argument: the library's fixed scratch is used
    (for callers that may not allocate device memory)."""
    B, H, N, d = _dims(q)
    _check(load_library().fa_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                         _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv), B, H, N, d,
                                         float(scale), int(bool(causal)), _dtype_code(q),
                                         _ptr(kv_len), _ptr(block_mask), _ptr(o_res),
                                         _stream(stream)),
           "fa_bwd_noalloc")


def fa_bwd_noalloc_max_workspace() -> int:
    return int(load_library().fa_bwd_noalloc_max_workspace())


def fa_get_device_error(stream=None) -> int:
    """Synchronise the stream and return the device error status (0 = FA_OK)."""
    return int(load_library().fa_get_device_error(_stream(stream)))


def fa_set_wait_limit_ns(ns: int) -> int:
    """Time limit of the kernels' pipeline waits (0 = the 2 s default)."""
    return int(load_library().fa_set_wait_limit_ns(int(ns)))


def fa_debug_starve_pipelines(enable: bool) -> int:
    """Test switch: the kernels' load-issuing threads issue nothing."""
    return int(load_library().fa_debug_starve_pipelines(1 if enable else 0))


def fa_status_str(status: int) -> str:
    return load_library().fa_status_str(int(status)).decode()


def fa_last_error_message() -> str:
    return load_library().fa_last_error_message().decode()


def fa_version() -> str:
    return load_library().fa_version().decode()
