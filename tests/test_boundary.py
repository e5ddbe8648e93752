"""The C-ABI boundary on the CPU: the library builds, loads, exports every symbol
include/gbattn.h declares, and rejects bad arguments before touching a device."""

import ctypes
import math
import os
import re

import pytest

import attention_flashattention_fwd_03_gb300 as gb

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gbattn.h")

A16 = 0x100000  # a 16-byte-aligned address that is never dereferenced by validation


def declared_functions():
    with open(HEADER) as fh:
        text = fh.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    pat = r"^\s*(?:const\s+)?(?:unsigned\s+)?(?:long\s+)*\w+(?:\s+|\s*\*\s*)(\w+)\s*\("
    return sorted(set(re.findall(pat, text, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    return gb.lib()


def test_header_declares_the_boundary():
    names = declared_functions()
    assert names == sorted(gb.EXPORTS), names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_status_strings(lib):
    assert gb.status_string(gb.ATTN_OK) == "ATTN_OK"
    assert gb.status_string(gb.ATTN_ERR_INVALID_ARG) == "ATTN_ERR_INVALID_ARG"
    assert gb.status_string(gb.ATTN_ERR_UNSUPPORTED) == "ATTN_ERR_UNSUPPORTED"
    assert gb.status_string(gb.ATTN_ERR_CUDA) == "ATTN_ERR_CUDA"
    assert gb.status_string(gb.ATTN_ERR_DEVICE) == "ATTN_ERR_DEVICE"
    assert gb.status_string(99) == "ATTN_ERR_UNKNOWN"
    assert gb.version() == "0.1.0"


def fwd(lib, q=A16, k=A16, v=A16, o=A16, lse=None, B=1, Hq=2, Hkv=2, T=128, D=64, causal=1,
        scale=0.125):
    return lib.attn_fwd(q, k, v, o, lse, B, Hq, Hkv, T, D, causal, scale, None)


@pytest.mark.parametrize("kw,code", [
    (dict(D=96), gb.ATTN_ERR_UNSUPPORTED),
    (dict(D=256), gb.ATTN_ERR_UNSUPPORTED),
    (dict(Hq=3, Hkv=2), gb.ATTN_ERR_INVALID_ARG),
    (dict(Hkv=0), gb.ATTN_ERR_INVALID_ARG),
    (dict(B=-1), gb.ATTN_ERR_INVALID_ARG),
    (dict(T=-5), gb.ATTN_ERR_INVALID_ARG),
    (dict(causal=2), gb.ATTN_ERR_INVALID_ARG),
    (dict(scale=float("nan")), gb.ATTN_ERR_INVALID_ARG),
    (dict(scale=float("inf")), gb.ATTN_ERR_INVALID_ARG),
    (dict(scale=0.0), gb.ATTN_ERR_INVALID_ARG),
    (dict(scale=-0.1), gb.ATTN_ERR_INVALID_ARG),
    (dict(q=None), gb.ATTN_ERR_INVALID_ARG),
    (dict(o=None), gb.ATTN_ERR_INVALID_ARG),
    (dict(k=A16 + 2), gb.ATTN_ERR_INVALID_ARG),
    (dict(o=A16 + 8), gb.ATTN_ERR_INVALID_ARG),
    (dict(lse=A16 + 2), gb.ATTN_ERR_INVALID_ARG),
    (dict(B=0), gb.ATTN_OK),
    (dict(T=0), gb.ATTN_OK),
    (dict(B=0, q=None, k=None, v=None, o=None), gb.ATTN_OK),
    (dict(B=1 << 20, Hq=1 << 12, Hkv=1 << 12), gb.ATTN_ERR_UNSUPPORTED),
])
def test_attn_fwd_validation(lib, kw, code):
    assert fwd(lib, **kw) == code


def dec(lib, q=A16, k=A16, v=A16, bt=A16, sl=A16, bs=16, S=4, Hq=12, Hkv=2, D=128, mb=512,
        nb=1000, msl=8192, scale=0.088, o=A16, lse=None, ws=A16, wsb=None):
    if wsb is None:
        wsb = lib.paged_attn_decode_workspace_size(S, Hq, D, msl)
    return lib.paged_attn_decode(q, k, v, bt, sl, bs, S, Hq, Hkv, D, mb, nb, msl, scale, o, lse,
                                 ws, wsb, None)


@pytest.mark.parametrize("kw,code", [
    (dict(bs=8), gb.ATTN_ERR_UNSUPPORTED),
    (dict(bs=32), gb.ATTN_ERR_UNSUPPORTED),
    (dict(D=80), gb.ATTN_ERR_UNSUPPORTED),
    (dict(Hq=34, Hkv=2), gb.ATTN_ERR_UNSUPPORTED),  # group 17 > 16
    (dict(Hq=12, Hkv=5), gb.ATTN_ERR_INVALID_ARG),
    (dict(wsb=16), gb.ATTN_ERR_INVALID_ARG),
    (dict(ws=None), gb.ATTN_ERR_INVALID_ARG),
    (dict(ws=A16 + 16), gb.ATTN_ERR_INVALID_ARG),  # workspace wants 256-byte alignment
    (dict(bt=None), gb.ATTN_ERR_INVALID_ARG),
    (dict(sl=A16 + 2), gb.ATTN_ERR_INVALID_ARG),
    (dict(k=A16 + 4), gb.ATTN_ERR_INVALID_ARG),
    (dict(nb=0), gb.ATTN_ERR_INVALID_ARG),
    (dict(mb=0), gb.ATTN_ERR_INVALID_ARG),
    (dict(msl=-1), gb.ATTN_ERR_INVALID_ARG),
    (dict(scale=float("nan")), gb.ATTN_ERR_INVALID_ARG),
    (dict(S=0), gb.ATTN_OK),
    (dict(nb=1 << 27), gb.ATTN_ERR_UNSUPPORTED),  # pool rows beyond int32 TMA coordinates
])
def test_paged_decode_validation(lib, kw, code):
    assert dec(lib, **kw) == code


def test_workspace_size_formula(lib):
    # Per (request, query head): at most ceil(max_seq_len / 256) + 1 pieces (ranges
    # of at least 16 blocks of 16 tokens), each D fp32 outputs and one fp32 LSE;
    # then one int64 per (request, query head) for the segment starts and two
    # int64 for the plan; every part 256-byte aligned.
    up = lambda x: (x + 255) // 256 * 256
    for S, Hq, D, msl in [(64, 12, 128, 8192), (1, 1, 64, 1), (3, 8, 128, 513), (5, 4, 64, 0)]:
        pieces = math.ceil(math.ceil(msl / 16) / 16) + 1
        n = S * Hq * pieces
        expect = up(n * D * 4) + up(n * 4) + up(S * Hq * 8) + up(16)
        assert lib.paged_attn_decode_workspace_size(S, Hq, D, msl) == expect
    assert lib.paged_attn_decode_workspace_size(-1, 1, 64, 1) == 0


def test_valid_call_without_a_device_is_an_error_not_a_fallback(lib):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a device is present; this checks the no-device path")
    assert fwd(lib) == gb.ATTN_ERR_CUDA
    assert dec(lib) == gb.ATTN_ERR_CUDA


# --------------------------------------------------------------------------- #
# the Python binding's checks (metadata only: they run before any device work)
# --------------------------------------------------------------------------- #
def _bf16(*shape):
    torch = pytest.importorskip("torch")
    return torch.zeros(shape, dtype=torch.bfloat16)


def _f32(*shape):
    torch = pytest.importorskip("torch")
    return torch.zeros(shape, dtype=torch.float32)


@pytest.mark.parametrize("bad", ["out_shape", "out_dtype", "lse_shape", "lse_dtype",
                                 "lse_strided", "cpu_tensors", "k_mismatch"])
def test_binding_rejects_bad_attn_fwd_tensors(bad):
    q, k, v = _bf16(1, 2, 8, 64), _bf16(1, 1, 8, 64), _bf16(1, 1, 8, 64)
    kw = {}
    if bad == "out_shape":
        kw["out"] = _bf16(1, 2, 8, 32)
    elif bad == "out_dtype":
        kw["out"] = _f32(1, 2, 8, 64)
    elif bad == "lse_shape":
        kw["lse"] = _f32(1, 2, 9)
    elif bad == "lse_dtype":
        kw["lse"] = _bf16(1, 2, 8)
    elif bad == "lse_strided":
        kw["lse"] = _f32(1, 2, 16)[:, :, ::2]
    elif bad == "k_mismatch":
        k = _bf16(1, 1, 7, 64)
    with pytest.raises(ValueError):
        gb.attn_fwd(q, k, v, **kw)


@pytest.mark.parametrize("bad", ["out_shape", "out_dtype", "lse_shape", "lse_dtype",
                                 "table_dtype", "ws_dtype", "cpu_tensors"])
def test_binding_rejects_bad_decode_tensors(bad):
    torch = pytest.importorskip("torch")
    q, kp, vp = _bf16(2, 4, 64), _bf16(10, 2, 16, 64), _bf16(10, 2, 16, 64)
    bt = torch.zeros((2, 4), dtype=torch.int32)
    sl = torch.ones(2, dtype=torch.int32)
    kw = {}
    if bad == "out_shape":
        kw["out"] = _bf16(2, 4, 32)
    elif bad == "out_dtype":
        kw["out"] = _f32(2, 4, 64)
    elif bad == "lse_shape":
        kw["lse"] = _f32(2, 5)
    elif bad == "lse_dtype":
        kw["lse"] = _bf16(2, 4)
    elif bad == "table_dtype":
        bt = bt.to(torch.int64)
    elif bad == "ws_dtype":
        kw["workspace"] = _f32(64)
    with pytest.raises(ValueError):
        gb.paged_attn_decode(q, kp, vp, bt, sl, 64, **kw)
