"""GB300 (sm_103a) fused attention: Python binding of the C ABI in include/gbattn.h.

Only argument marshalling happens here; every step of the computation runs in
the library's CUDA kernels.  torch is used for device memory and streams.  If
the library is missing or cannot be loaded, or an operation reports an error,
an exception is raised -- there is no fallback implementation.

    o, lse = attn_fwd(q, k, v, causal=True)                  # [B,H,T,D] bf16 CUDA tensors
    o, lse = paged_attn_decode(q, k_pool, v_pool, block_table, seq_lens, max_seq_len)
"""

from __future__ import annotations

import ctypes
import math
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgbattn.so")

ATTN_OK = 0
ATTN_ERR_INVALID_ARG = 1
ATTN_ERR_UNSUPPORTED = 2
ATTN_ERR_CUDA = 3
ATTN_ERR_DEVICE = 4

EXPORTS = (
    "attn_status_string",
    "attn_fwd",
    "paged_attn_decode_workspace_size",
    "paged_attn_decode",
    "paged_attn_decode_noalloc",
    "paged_attn_prefill",
    "paged_kv_append",
    "paged_kv_gather",
    "attn_test_set_failure",
    "attn_device_status",
    "attn_version",
)

_lock = threading.Lock()
_lib = None


class GbAttnError(RuntimeError):
    def __init__(self, op: str, status: int, detail: str = ""):
        self.status = status
        name = status_string(status) if _lib is not None else str(status)
        super().__init__(f"{op} failed: {name}{(' (' + detail + ')') if detail else ''}")


def lib(build_if_missing: bool = True):
    """The loaded ctypes handle of libgbattn.so (built in-tree on first use)."""
    global _lib
    with _lock:
        if _lib is None:
            if build_if_missing:
                from . import build as _build
                _build.build()
            if not os.path.exists(LIB_PATH):
                raise ImportError(f"libgbattn.so not found at {LIB_PATH}; run build.py")
            h = ctypes.CDLL(LIB_PATH)
            _bind(h)
            _lib = h
    return _lib


def _bind(h):
    P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    h.attn_status_string.argtypes = [I]
    h.attn_status_string.restype = ctypes.c_char_p
    h.attn_fwd.argtypes = [P, P, P, P, P, I, I, I, I, I, I, F, P]
    h.attn_fwd.restype = I
    h.paged_attn_decode_workspace_size.argtypes = [I, I, I, I]
    h.paged_attn_decode_workspace_size.restype = Z
    h.paged_attn_decode.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, I, F, P, P, P, Z, P]
    h.paged_attn_decode.restype = I
    h.paged_attn_decode_noalloc.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, I, F, P, P, P]
    h.paged_attn_decode_noalloc.restype = I
    h.paged_attn_prefill.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, I, I, I, F, P, P, P]
    h.paged_attn_prefill.restype = I
    h.paged_kv_append.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, I, P]
    h.paged_kv_append.restype = I
    h.paged_kv_gather.argtypes = [P, P, P, I, I, I, I, I, I, I, P, P]
    h.paged_kv_gather.restype = I
    h.attn_test_set_failure.argtypes = [ctypes.c_ulonglong, I]
    h.attn_test_set_failure.restype = I
    h.attn_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint)]
    h.attn_device_status.restype = I
    h.attn_version.argtypes = []
    h.attn_version.restype = I


def status_string(status: int) -> str:
    return lib().attn_status_string(int(status)).decode()


def _stream_handle(stream, device):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _check_tensor(name, t, dtype, shape, device):
    """Metadata checks only (no device access): type, dtype, exact shape, layout, device."""
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.device != device:
        raise ValueError(f"{name} must be on {device}, got {t.device}")


def _check_bf16(name, t, ndim, device):
    import torch
    if isinstance(t, torch.Tensor) and t.dim() != ndim:
        raise ValueError(f"{name} must be a {ndim}-d tensor")
    _check_tensor(name, t, torch.bfloat16, None, device)


def _require_cuda(device):
    if device.type != "cuda":
        raise ValueError(f"tensors must be CUDA tensors, got {device}")


def attn_fwd(q, k, v, causal: bool = True, scale: float | None = None, out=None, lse=None,
             return_lse: bool = True, stream=None):
    """Fused attention forward through the C ABI.

    q [B,Hq,T,D], k/v [B,Hkv,T,D] bf16 CUDA tensors -> (o [B,Hq,T,D] bf16,
    lse [B,Hq,T] fp32 or None).  ``scale`` defaults to 1/sqrt(D).  ``out`` and
    ``lse``, when given, must be contiguous tensors of exactly those shapes and
    dtypes on q's device.
    """
    import torch
    device = q.device if isinstance(q, torch.Tensor) else None
    _check_bf16("q", q, 4, device)
    _check_bf16("k", k, 4, device)
    _check_bf16("v", v, 4, device)
    B, Hq, T, D = q.shape
    if k.shape[0] != B or k.shape[2] != T or k.shape[3] != D or v.shape != k.shape:
        raise ValueError("k/v must be [B, Hkv, T, D] matching q")
    Hkv = k.shape[1]
    if out is not None:
        _check_tensor("out", out, torch.bfloat16, (B, Hq, T, D), device)
    if lse is not None:
        _check_tensor("lse", lse, torch.float32, (B, Hq, T), device)
    _require_cuda(device)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    with torch.cuda.device(device):
        if out is None:
            out = torch.empty_like(q)
        if return_lse and lse is None:
            lse = torch.empty((B, Hq, T), dtype=torch.float32, device=device)
        st = lib().attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                            lse.data_ptr() if lse is not None else None, B, Hq, Hkv, T, D,
                            int(bool(causal)), float(scale), _stream_handle(stream, device))
    if st != ATTN_OK:
        raise GbAttnError("attn_fwd", st)
    return out, lse


def paged_attn_decode_workspace_size(num_seqs: int, Hq: int, D: int, max_seq_len: int) -> int:
    return int(lib().paged_attn_decode_workspace_size(num_seqs, Hq, D, max_seq_len))


def paged_attn_decode(q, k_pool, v_pool, block_table, seq_lens, max_seq_len: int,
                      scale: float | None = None, out=None, lse=None, workspace=None,
                      return_lse: bool = True, stream=None):
    """Single-token decode against a paged KV cache through the C ABI.

    q [S,Hq,D] bf16, k_pool/v_pool [NB,Hkv,16,D] bf16, block_table [S,max_blocks]
    int32, seq_lens [S] int32 (all CUDA) -> (o [S,Hq,D] bf16, lse [S,Hq] fp32).
    ``workspace`` (uint8 CUDA tensor) is allocated here when not given.
    """
    import torch
    device = q.device if isinstance(q, torch.Tensor) else None
    _check_bf16("q", q, 3, device)
    _check_bf16("k_pool", k_pool, 4, device)
    _check_bf16("v_pool", v_pool, 4, device)
    for name, t in (("block_table", block_table), ("seq_lens", seq_lens)):
        _check_tensor(name, t, torch.int32, None, device)
    S, Hq, D = q.shape
    NB, Hkv, bs, D2 = k_pool.shape
    if D2 != D or v_pool.shape != k_pool.shape or block_table.dim() != 2 or \
            block_table.shape[0] != S or tuple(seq_lens.shape) != (S,):
        raise ValueError("inconsistent paged-decode shapes")
    if out is not None:
        _check_tensor("out", out, torch.bfloat16, (S, Hq, D), device)
    if lse is not None:
        _check_tensor("lse", lse, torch.float32, (S, Hq), device)
    if workspace is not None:
        _check_tensor("workspace", workspace, torch.uint8, None, device)
    _require_cuda(device)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    need = paged_attn_decode_workspace_size(S, Hq, D, max_seq_len)
    with torch.cuda.device(device):
        if workspace is None:
            workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=device)
        if out is None:
            out = torch.empty_like(q)
        if return_lse and lse is None:
            lse = torch.empty((S, Hq), dtype=torch.float32, device=device)
        st = lib().paged_attn_decode(q.data_ptr(), k_pool.data_ptr(), v_pool.data_ptr(),
                                     block_table.data_ptr(), seq_lens.data_ptr(), bs, S, Hq, Hkv,
                                     D, block_table.shape[1], NB, int(max_seq_len), float(scale),
                                     out.data_ptr(),
                                     lse.data_ptr() if lse is not None else None,
                                     workspace.data_ptr(), workspace.numel(),
                                     _stream_handle(stream, device))
    if st != ATTN_OK:
        raise GbAttnError("paged_attn_decode", st)
    return out, lse


def paged_attn_prefill(q, k_pool, v_pool, block_table, kv_lens, max_kv_len: int,
                       causal: bool = True, scale: float | None = None, out=None, lse=None,
                       return_lse: bool = True, stream=None):
    """Chunked prefill against a paged KV cache through the C ABI.

    q [B,Hq,Tq,D] bf16 (the Tq newest tokens of each item), k_pool/v_pool
    [NB,Hkv,16,D] bf16, block_table [B,max_blocks] int32, kv_lens [B] int32 (all
    CUDA) -> (o [B,Hq,Tq,D] bf16, lse [B,Hq,Tq] fp32).  Query i of item b sits at
    logical position kv_lens[b] - Tq + i.
    """
    import torch
    device = q.device if isinstance(q, torch.Tensor) else None
    _check_bf16("q", q, 4, device)
    _check_bf16("k_pool", k_pool, 4, device)
    _check_bf16("v_pool", v_pool, 4, device)
    for name, t in (("block_table", block_table), ("kv_lens", kv_lens)):
        _check_tensor(name, t, torch.int32, None, device)
    B, Hq, Tq, D = q.shape
    NB, Hkv, bs, D2 = k_pool.shape
    if D2 != D or v_pool.shape != k_pool.shape or block_table.dim() != 2 or \
            block_table.shape[0] != B or tuple(kv_lens.shape) != (B,):
        raise ValueError("inconsistent paged-prefill shapes")
    if out is not None:
        _check_tensor("out", out, torch.bfloat16, (B, Hq, Tq, D), device)
    if lse is not None:
        _check_tensor("lse", lse, torch.float32, (B, Hq, Tq), device)
    _require_cuda(device)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    with torch.cuda.device(device):
        if out is None:
            out = torch.empty_like(q)
        if return_lse and lse is None:
            lse = torch.empty((B, Hq, Tq), dtype=torch.float32, device=device)
        st = lib().paged_attn_prefill(q.data_ptr(), k_pool.data_ptr(), v_pool.data_ptr(),
                                      block_table.data_ptr(), kv_lens.data_ptr(), bs, B, Hq, Hkv,
                                      Tq, D, block_table.shape[1], NB, int(max_kv_len),
                                      int(bool(causal)), float(scale), out.data_ptr(),
                                      lse.data_ptr() if lse is not None else None,
                                      _stream_handle(stream, device))
    if st != ATTN_OK:
        raise GbAttnError("paged_attn_prefill", st)
    return out, lse


def paged_kv_append(k_new, v_new, k_pool, v_pool, block_table, seq_lens, new_seq_lens=None,
                    stream=None):
    """Writes the Tn new tokens of each request into the paged pools (in place).

    k_new/v_new [S,Hkv,Tn,D] bf16, k_pool/v_pool [NB,Hkv,16,D] bf16, block_table
    [S,max_blocks] int32, seq_lens [S] int32 (lengths before the append);
    new_seq_lens [S] int32, if given, receives seq_lens + Tn.
    """
    import torch
    device = k_new.device if isinstance(k_new, torch.Tensor) else None
    _check_bf16("k_new", k_new, 4, device)
    _check_bf16("v_new", v_new, 4, device)
    _check_bf16("k_pool", k_pool, 4, device)
    _check_bf16("v_pool", v_pool, 4, device)
    for name, t in (("block_table", block_table), ("seq_lens", seq_lens)):
        _check_tensor(name, t, torch.int32, None, device)
    S, Hkv, Tn, D = k_new.shape
    NB, Hkv2, bs, D2 = k_pool.shape
    if v_new.shape != k_new.shape or v_pool.shape != k_pool.shape or Hkv2 != Hkv or D2 != D or \
            block_table.dim() != 2 or block_table.shape[0] != S or tuple(seq_lens.shape) != (S,):
        raise ValueError("inconsistent append shapes")
    if new_seq_lens is not None:
        _check_tensor("new_seq_lens", new_seq_lens, torch.int32, (S,), device)
    _require_cuda(device)
    with torch.cuda.device(device):
        st = lib().paged_kv_append(k_new.data_ptr(), v_new.data_ptr(), k_pool.data_ptr(),
                                   v_pool.data_ptr(), block_table.data_ptr(), seq_lens.data_ptr(),
                                   new_seq_lens.data_ptr() if new_seq_lens is not None else None,
                                   bs, S, Hkv, Tn, D, block_table.shape[1], NB,
                                   _stream_handle(stream, device))
    if st != ATTN_OK:
        raise GbAttnError("paged_kv_append", st)
    return new_seq_lens


def paged_kv_gather(pool, block_table, seq_lens, max_seq_len: int, out=None, stream=None):
    """Each request's cached rows in logical order: out [S,Hkv,max_seq_len,D] bf16
    (rows past a request's length are left as they were)."""
    import torch
    device = pool.device if isinstance(pool, torch.Tensor) else None
    _check_bf16("pool", pool, 4, device)
    for name, t in (("block_table", block_table), ("seq_lens", seq_lens)):
        _check_tensor(name, t, torch.int32, None, device)
    NB, Hkv, bs, D = pool.shape
    S = seq_lens.shape[0]
    if block_table.dim() != 2 or block_table.shape[0] != S:
        raise ValueError("inconsistent gather shapes")
    if out is not None:
        _check_tensor("out", out, torch.bfloat16, (S, Hkv, max_seq_len, D), device)
    _require_cuda(device)
    with torch.cuda.device(device):
        if out is None:
            out = torch.zeros((S, Hkv, max_seq_len, D), dtype=torch.bfloat16, device=device)
        st = lib().paged_kv_gather(pool.data_ptr(), block_table.data_ptr(), seq_lens.data_ptr(),
                                   bs, S, Hkv, D, block_table.shape[1], NB, int(max_seq_len),
                                   out.data_ptr(), _stream_handle(stream, device))
    if st != ATTN_OK:
        raise GbAttnError("paged_kv_gather", st)
    return out


def test_set_failure(wait_limit_ns: int = 0, withhold_copy: bool = False) -> None:
    """Test hook: in-kernel wait limit (0 = default 2 s) and whether the next kernels'
    copy warps withhold their first copy so that a wait runs out."""
    st = lib().attn_test_set_failure(int(wait_limit_ns), int(bool(withhold_copy)))
    if st != ATTN_OK:
        raise GbAttnError("attn_test_set_failure", st)


def attn_device_status():
    """(status, flags): synchronises the current device, reads and clears its flag word."""
    flags = ctypes.c_uint(0)
    st = lib().attn_device_status(ctypes.byref(flags))
    return st, flags.value


def version() -> str:
    v = lib().attn_version()
    return f"{v // 10000}.{(v // 100) % 100}.{v % 100}"
