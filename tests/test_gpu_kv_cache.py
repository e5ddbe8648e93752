"""The paged KV cache on the GPU: appending new tokens (a byte-exact scatter through
the block table) and gathering a request's history with the attention kernels'
own translation and TMA copies (byte-exact against the oracle's gather)."""

from __future__ import annotations

import numpy as np
import pytest

import oracle
import synth
from gpu_util import bits_of, check_close, from_dev, to_dev, to_dev_i32

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def gb():
    import attention_flashattention_fwd_03_gb300 as gb
    gb.lib()
    return gb


def _cache_with_room(seed, lens_before, Tn, Hq=12, Hkv=2, D=128):
    """Pools whose block tables already cover lens_before + Tn tokens."""
    cfg = synth.DecodeConfig("append", len(lens_before), Hq, Hkv, D, 1, 9000, 16, seed)
    after = [L + Tn for L in lens_before]
    p = synth.paged_inputs(cfg, seq_lens=after, max_seq_len=max(after))
    return cfg, p


def _host_scatter(pool, table, lens_before, new):
    """pool[table[r][(L+t)//16], h, (L+t)%16] = new[r, h, t] (numpy, on a copy)."""
    out = pool.copy()
    S, Hkv, Tn, _ = new.shape
    for r in range(S):
        for t in range(Tn):
            pos = int(lens_before[r]) + t
            out[table[r, pos // 16], :, pos % 16] = new[r, :, t]
    return out


@pytest.mark.parametrize("Tn,D", [(1, 128), (1, 64), (5, 128), (37, 64)])
def test_append_is_a_byte_exact_scatter(gb, Tn, D):
    lens = [0, 1, 15, 16, 17, 31, 32, 511, 512, 4095, 8000]  # several open a new block
    cfg, p = _cache_with_room(24000 + Tn + D, lens, Tn, D=D)
    k_new = synth.normal_bf16(24001, (len(lens), cfg.Hkv, Tn, D))
    v_new = synth.normal_bf16(24002, (len(lens), cfg.Hkv, Tn, D))
    kp, vp = to_dev(p.k_pool), to_dev(p.v_pool)
    before = to_dev_i32(np.array(lens, np.int32))
    after = torch.full_like(before, -7)
    gb.paged_kv_append(to_dev(k_new), to_dev(v_new), kp, vp, to_dev_i32(p.block_table), before,
                       after)
    torch.cuda.synchronize()
    assert gb.attn_device_status() == (gb.ATTN_OK, 0)
    assert np.array_equal(after.cpu().numpy(), np.array(lens) + Tn)
    assert np.array_equal(bits_of(kp), _host_scatter(p.k_pool, p.block_table, lens, k_new))
    assert np.array_equal(bits_of(vp), _host_scatter(p.v_pool, p.block_table, lens, v_new))


def test_append_then_decode_matches_oracle(gb):
    lens = [511, 512, 1000, 4096, 16, 0]
    cfg, p = _cache_with_room(24100, lens, 1)
    k_new = synth.normal_bf16(24101, (len(lens), cfg.Hkv, 1, cfg.D))
    v_new = synth.normal_bf16(24102, (len(lens), cfg.Hkv, 1, cfg.D))
    kp, vp, bt = to_dev(p.k_pool), to_dev(p.v_pool), to_dev_i32(p.block_table)
    before = to_dev_i32(np.array(lens, np.int32))
    after = torch.empty_like(before)
    gb.paged_kv_append(to_dev(k_new), to_dev(v_new), kp, vp, bt, before, after)
    o, lse = gb.paged_attn_decode(to_dev(p.q), kp, vp, bt, after, p.max_seq_len,
                                  scale=cfg.softmax_scale)
    torch.cuda.synchronize()
    assert gb.attn_device_status() == (gb.ATTN_OK, 0)
    k_ref = _host_scatter(p.k_pool, p.block_table, lens, k_new)
    v_ref = _host_scatter(p.v_pool, p.block_table, lens, v_new)
    o_ref, lse_ref = oracle.paged_decode(p.q, k_ref, v_ref, p.block_table,
                                         np.array(lens, np.int32) + 1, cfg.softmax_scale)
    check_close(from_dev(o), from_dev(lse), o_ref, lse_ref, "append + decode")
    # the appended token is the query's own key: the last cached row is k_new
    last = bits_of(kp)[p.block_table[0, 511 // 16], :, 511 % 16]
    assert np.array_equal(last, k_new[0, :, 0])


def test_append_bad_requests_are_flagged_and_skipped(gb):
    lens = [10, 20, 30]
    cfg, p = _cache_with_room(24200, lens, 1, D=64)
    table = p.block_table.copy()
    table[1, 20 // 16] = p.num_pool_blocks + 3  # block outside the pool
    bad_lens = np.array([10, 20, table.shape[1] * 16], np.int32)  # request 2 has no room
    kp, vp = to_dev(p.k_pool), to_dev(p.v_pool)
    after = torch.empty(3, dtype=torch.int32, device="cuda")
    k_new = synth.normal_bf16(24201, (3, cfg.Hkv, 1, 64))
    gb.paged_kv_append(to_dev(k_new), to_dev(k_new), kp, vp, to_dev_i32(table),
                       to_dev_i32(bad_lens), after)
    torch.cuda.synchronize()
    st, flags = gb.attn_device_status()
    assert flags == 2 | 4, (st, flags)
    assert after.cpu().tolist() == [11, 21, int(bad_lens[2])]
    exp = _host_scatter(p.k_pool, p.block_table, [10], k_new[:1])  # only request 0 written
    assert np.array_equal(bits_of(kp), exp)


def test_gather_equals_the_oracle_gather_byte_for_byte(gb):
    """The full paged decode workload: every request, both KV heads, K and V."""
    cfg = synth.CONFIGS["paged_decode"]
    p = synth.paged_inputs(cfg)
    bt, sl = to_dev_i32(p.block_table), to_dev_i32(p.seq_lens)
    for pool in (p.k_pool, p.v_pool):
        out = gb.paged_kv_gather(to_dev(pool), bt, sl, p.max_seq_len)
        torch.cuda.synchronize()
        assert gb.attn_device_status() == (gb.ATTN_OK, 0)
        got = bits_of(out)
        for r in range(cfg.num_seqs):
            L = int(p.seq_lens[r])
            for h in range(cfg.Hkv):
                exp = oracle.paged_gather(pool, p.block_table, p.seq_lens, r, h)
                assert np.array_equal(got[r, h, :L], exp), (r, h)


def test_gather_edge_lengths(gb):
    lens = [0, 1, 15, 16, 17, 511, 512, 513, 1025]
    cfg = synth.DecodeConfig("g", len(lens), 4, 3, 64, 1, 1100, 16, 24300)
    p = synth.paged_inputs(cfg, seq_lens=lens, max_seq_len=1100)
    out = gb.paged_kv_gather(to_dev(p.k_pool), to_dev_i32(p.block_table),
                             to_dev_i32(p.seq_lens), p.max_seq_len)
    torch.cuda.synchronize()
    got = bits_of(out)
    for r, L in enumerate(lens):
        for h in range(cfg.Hkv):
            assert np.array_equal(got[r, h, :L], oracle.paged_gather(p.k_pool, p.block_table,
                                                                     p.seq_lens, r, h))
