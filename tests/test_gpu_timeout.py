"""The kernels' bounded waits.  For one small call the copy warps withhold their
first copy (a barrier that nothing completes) and the wait limit is cut to a
millisecond: the waiting role gives up, the kernel lets its copies and MMAs in
flight finish, frees its tensor memory and returns; the host sees the timeout
flag, and the next call with the default settings is correct again.  Nothing
here faults, traps or hangs the GPU: every wait in these kernels has a limit."""

from __future__ import annotations

import numpy as np
import pytest

import oracle
import synth
from gpu_util import check_close, from_dev, to_dev, to_dev_i32

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def gb():
    import attention_flashattention_fwd_03_gb300 as gb
    gb.lib()
    return gb


def _with_short_limit(gb, fn):
    torch.cuda.synchronize()
    gb.test_set_failure(wait_limit_ns=1_000_000, withhold_copy=True)
    try:
        fn()
        torch.cuda.synchronize()
    finally:
        gb.test_set_failure(0, False)
    return gb.attn_device_status()


def test_prefill_wait_timeout_is_reported_and_recoverable(gb):
    cfg = synth.PrefillConfig("to", 1, 8, 2, 1000, 128, True, 1.0, 23000)
    q, k, v = synth.prefill_inputs(cfg)
    qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
    st, flags = _with_short_limit(
        gb, lambda: gb.attn_fwd(qd, kd, vd, causal=True, scale=cfg.softmax_scale))
    assert st == gb.ATTN_ERR_DEVICE and flags & 1, (st, flags)
    assert gb.attn_device_status() == (gb.ATTN_OK, 0)  # read-and-clear
    o, lse = gb.attn_fwd(qd, kd, vd, causal=True, scale=cfg.softmax_scale)
    torch.cuda.synchronize()
    assert gb.attn_device_status() == (gb.ATTN_OK, 0)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, True, cfg.softmax_scale)
    check_close(from_dev(o), from_dev(lse), o_ref, lse_ref, "after timeout")


def test_decode_wait_timeout_is_reported_and_recoverable(gb):
    cfg = synth.DecodeConfig("to", 8, 12, 2, 128, 300, 3000, 16, 23100)
    p = synth.paged_inputs(cfg)
    args = (to_dev(p.q), to_dev(p.k_pool), to_dev(p.v_pool), to_dev_i32(p.block_table),
            to_dev_i32(p.seq_lens), p.max_seq_len)
    st, flags = _with_short_limit(
        gb, lambda: gb.paged_attn_decode(*args, scale=cfg.softmax_scale))
    assert st == gb.ATTN_ERR_DEVICE and flags & 1, (st, flags)
    o, lse = gb.paged_attn_decode(*args, scale=cfg.softmax_scale)
    torch.cuda.synchronize()
    assert gb.attn_device_status() == (gb.ATTN_OK, 0)
    o_ref, lse_ref = oracle.paged_decode(p.q, p.k_pool, p.v_pool, p.block_table, p.seq_lens,
                                         cfg.softmax_scale)
    check_close(from_dev(o), from_dev(lse), o_ref, lse_ref, "after timeout")


def test_paged_prefill_wait_timeout_is_reported_and_recoverable(gb):
    cfg = synth.DecodeConfig("to", 2, 8, 2, 128, 1, 2000, 16, 23200)
    p = synth.paged_inputs(cfg, seq_lens=[900, 2000], max_seq_len=2000)
    q = synth.normal_bf16(23201, (2, 8, 300, 128))
    args = (to_dev(q), to_dev(p.k_pool), to_dev(p.v_pool), to_dev_i32(p.block_table),
            to_dev_i32(p.seq_lens), p.max_seq_len)
    st, flags = _with_short_limit(gb, lambda: gb.paged_attn_prefill(*args, causal=True))
    assert st == gb.ATTN_ERR_DEVICE and flags & 1, (st, flags)
    o, lse = gb.paged_attn_prefill(*args, causal=True)
    torch.cuda.synchronize()
    assert gb.attn_device_status() == (gb.ATTN_OK, 0)
    o_ref, lse_ref = oracle.paged_prefill(q, p.k_pool, p.v_pool, p.block_table, p.seq_lens, True,
                                          cfg.softmax_scale)
    check_close(from_dev(o), from_dev(lse), o_ref, lse_ref, "after timeout")
