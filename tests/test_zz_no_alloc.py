"""paged_attn_decode_noalloc: paged decode whose scratch lives in the library.

Callers that cannot allocate device memory where they decode (allocator hooks,
hosts that own every device allocation, loops that must not enter the allocator)
use this entry point instead of passing a workspace.  Here it is called through
the raw C ABI with plain device pointers and compared with the ordinary entry
point, which gets a workspace allocated by torch, on two calls in a row: the
second call has different sizes, so it runs over scratch that the first call
left behind.  The file sorts last so that a run stopping at the first failure
has already run every other test.
"""

from __future__ import annotations

import numpy as np
import pytest

import synth
from gpu_util import LSE_MAX_ABS, O_MAX_ABS, O_MEAN_ABS, from_dev, to_dev, to_dev_i32

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

SCRATCH_BYTES = 16 * 1024 * 1024


@pytest.fixture(scope="module")
def gb():
    import attention_flashattention_fwd_03_gb300 as gb
    gb.lib()
    return gb


def _device_inputs(p: synth.PagedInputs):
    return (to_dev(p.q), to_dev(p.k_pool), to_dev(p.v_pool), to_dev_i32(p.block_table),
            to_dev_i32(p.seq_lens))


def _call(gb, fn_name, dev, p, scale, workspace=None):
    q, kp, vp, bt, sl = dev
    S, Hq, D = q.shape
    NB, Hkv, bs, _ = kp.shape
    o = torch.full_like(q, float("nan"))
    lse = torch.full((S, Hq), float("nan"), dtype=torch.float32, device=q.device)
    stream = torch.cuda.current_stream().cuda_stream
    lib = gb.lib()
    args = [q.data_ptr(), kp.data_ptr(), vp.data_ptr(), bt.data_ptr(), sl.data_ptr(), bs, S, Hq,
            Hkv, D, bt.shape[1], NB, p.max_seq_len, float(scale), o.data_ptr(), lse.data_ptr()]
    if fn_name == "paged_attn_decode":
        args += [workspace.data_ptr(), workspace.numel()]
    st = getattr(lib, fn_name)(*args, stream)
    assert st == gb.ATTN_OK, gb.status_string(st)
    torch.cuda.synchronize()
    return o, lse


def _reference_call(gb, dev, p, scale):
    q = dev[0]
    S, Hq, D = q.shape
    need = int(gb.lib().paged_attn_decode_workspace_size(S, Hq, D, p.max_seq_len))
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    return _call(gb, "paged_attn_decode", dev, p, scale, ws)


def _compare(o_new, l_new, o_ref, l_ref, what):
    a, b = from_dev(o_new), from_dev(o_ref)
    assert np.all(np.isfinite(a)), f"{what}: non-finite O"
    err = np.abs(a - b)
    assert err.max() <= O_MAX_ABS and err.mean() <= O_MEAN_ABS, (what, err.max(), err.mean())
    lerr = np.abs(from_dev(l_new) - from_dev(l_ref))
    assert lerr.max() <= LSE_MAX_ABS, (what, lerr.max())


def test_noalloc_decode_matches_the_workspace_entry_point_twice(gb):
    cfg = synth.CONFIGS["paged_decode"]
    first = synth.paged_inputs(cfg)  # 64 requests, lengths 512..8192
    second_cfg = synth.DecodeConfig("noalloc2", 9, 16, 2, 64, 1, 3000, 16, 51000)
    second = synth.paged_inputs(second_cfg, seq_lens=[1, 3000, 17, 512, 513, 0, 2047, 16, 999],
                                max_seq_len=3000)
    for p, c in ((first, cfg), (second, second_cfg)):
        dev = _device_inputs(p)
        o_ref, l_ref = _reference_call(gb, dev, p, c.softmax_scale)
        o_new, l_new = _call(gb, "paged_attn_decode_noalloc", dev, p, c.softmax_scale)
        # request 5 of the second call is empty: O = 0 and LSE = -inf on both sides
        live = [r for r in range(len(p.seq_lens)) if p.seq_lens[r] > 0]
        _compare(o_new[live], l_new[live], o_ref[live], l_ref[live], c.name)
        dead = [r for r in range(len(p.seq_lens)) if p.seq_lens[r] == 0]
        if dead:
            assert torch.all(o_new[dead] == 0) and torch.all(torch.isneginf(l_new[dead]))
    st, flags = gb.attn_device_status()
    assert st == gb.ATTN_OK and flags == 0, (st, flags)


def test_noalloc_decode_rejects_sizes_beyond_its_scratch(gb):
    lib = gb.lib()
    # 4096 requests x 32 heads x 8192 tokens need far more than the fixed scratch
    need = int(lib.paged_attn_decode_workspace_size(4096, 32, 128, 8192))
    assert need > SCRATCH_BYTES
    a16 = 0x100000  # never dereferenced: the size check comes first
    st = lib.paged_attn_decode_noalloc(a16, a16, a16, a16, a16, 16, 4096, 32, 8, 128, 512, 1000,
                                       8192, 0.088, a16, None, None)
    assert st == gb.ATTN_ERR_UNSUPPORTED
