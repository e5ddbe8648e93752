"""paged_attn_prefill (C ABI, sm_103a tcgen05 kernel reading K/V through the block
table) against the fp64 oracle: a chunk of Tq new tokens per batch item attends to
that item's paged cache, the chunk being the newest tokens (bottom-right causal)."""

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


def run(gb, q, p: synth.PagedInputs, causal, scale, expect_flags=0):
    o, lse = gb.paged_attn_prefill(to_dev(q), to_dev(p.k_pool), to_dev(p.v_pool),
                                   to_dev_i32(p.block_table), to_dev_i32(p.seq_lens),
                                   p.max_seq_len, causal=causal, scale=scale)
    torch.cuda.synchronize()
    st, flags = gb.attn_device_status()
    assert flags == expect_flags, (st, flags)
    return o, lse


def check_against_oracle(o, lse, q, p, causal, scale, what):
    o_ref, lse_ref = oracle.paged_prefill(q, p.k_pool, p.v_pool, p.block_table, p.seq_lens,
                                          causal, scale)
    og, lg = from_dev(o), from_dev(lse)
    empty = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lg), empty), what
    assert np.all(og[empty] == 0), what
    live = ~empty
    check_close(og[live], lg[live], o_ref[live], lse_ref[live], what)


CASES = [
    # Hq, Hkv, D, Tq, kv_lens
    (8, 2, 128, 1, [1, 17, 4096, 8192]),
    (8, 2, 128, 127, [127, 300, 2049, 8192]),
    (8, 2, 128, 512, [512, 700, 5000, 8192]),
    (12, 2, 128, 300, [300, 301, 1024, 3000]),
    (4, 4, 64, 257, [257, 640, 1000, 4096]),
    (16, 2, 64, 512, [600, 8192]),
]


@pytest.mark.parametrize("Hq,Hkv,D,Tq,kv_lens", CASES)
@pytest.mark.parametrize("causal", [True, False])
def test_paged_prefill_matches_oracle(gb, Hq, Hkv, D, Tq, kv_lens, causal):
    cfg = synth.DecodeConfig("pp", len(kv_lens), Hq, Hkv, D, 1, max(kv_lens), 16,
                             21000 + Tq + D + Hq)
    p = synth.paged_inputs(cfg, seq_lens=kv_lens, max_seq_len=max(kv_lens))
    q = synth.normal_bf16(cfg.seed + 9, (len(kv_lens), Hq, Tq, D))
    o, lse = run(gb, q, p, causal, cfg.softmax_scale)
    check_against_oracle(o, lse, q, p, causal, cfg.softmax_scale, f"{Hq},{Hkv},{D},{Tq},{causal}")


def test_paged_prefill_chunked_workload_full_size(gb):
    """The chunked-prefill workload at its full size, every element against the
    oracle: 16 sequences x 512 new tokens, cache lengths U[1024, 8192] with the
    chunk included, GQA 32/8, D = 128, causal, 16-token blocks in a permuted pool."""
    cfg = synth.DecodeConfig("chunked_prefill", 16, 32, 8, 128, 1024, 8192, 16, 6000)
    p = synth.paged_inputs(cfg)
    q = synth.normal_bf16(cfg.seed + 9, (cfg.num_seqs, cfg.Hq, 512, cfg.D))
    o, lse = run(gb, q, p, True, cfg.softmax_scale)
    o_ref, lse_ref = oracle.paged_prefill(q, p.k_pool, p.v_pool, p.block_table, p.seq_lens,
                                          True, cfg.softmax_scale)
    og, lg = from_dev(o), from_dev(lse)
    err = np.abs(og - o_ref)
    print(f"PARITY chunked_prefill rows={og.shape[0] * og.shape[1] * og.shape[2]} "
          f"o_max_abs={err.max():.3e} o_mean_abs={err.mean():.3e} "
          f"lse_max_abs={np.abs(lg - lse_ref).max():.3e}")
    check_close(og, lg, o_ref, lse_ref, "chunked prefill, full size")


def test_paged_prefill_short_cache_rows_see_nothing(gb):
    """kv_lens < Tq with a causal mask: the earliest queries see no key."""
    cfg = synth.DecodeConfig("short", 3, 4, 2, 128, 1, 300, 16, 21500)
    p = synth.paged_inputs(cfg, seq_lens=[5, 130, 0], max_seq_len=300)
    q = synth.normal_bf16(21501, (3, 4, 200, 128))
    o, lse = run(gb, q, p, True, cfg.softmax_scale)
    check_against_oracle(o, lse, q, p, True, cfg.softmax_scale, "short cache")


def test_paged_prefill_full_sequence_equals_contiguous_bit_exact(gb):
    """Tq = kv_len through the table gives the same bits as attn_fwd on contiguous K/V."""
    L, Hq, Hkv, D = 1000, 8, 2, 128
    cfg = synth.DecodeConfig("full", 2, Hq, Hkv, D, L, L, 16, 21600)
    p = synth.paged_inputs(cfg, seq_lens=[L, L], max_seq_len=L)
    q = synth.normal_bf16(21601, (2, Hq, L, D))
    t = np.arange(L)
    kc = np.stack([np.stack([p.k_pool[p.block_table[b, t // 16], h, t % 16] for h in range(Hkv)])
                   for b in range(2)])
    vc = np.stack([np.stack([p.v_pool[p.block_table[b, t // 16], h, t % 16] for h in range(Hkv)])
                   for b in range(2)])
    for causal in (True, False):
        o1, l1 = run(gb, q, p, causal, cfg.softmax_scale)
        o2, l2 = gb.attn_fwd(to_dev(q), to_dev(kc), to_dev(vc), causal=causal,
                             scale=cfg.softmax_scale)
        torch.cuda.synchronize()
        assert np.array_equal(bits_of(o1), bits_of(o2)) and torch.equal(l1, l2), causal


def test_paged_prefill_placement_invariance_bit_exact(gb):
    cfg = synth.DecodeConfig("place", 3, 8, 2, 128, 1, 3000, 16, 21700)
    p = synth.paged_inputs(cfg, seq_lens=[700, 3000, 129], max_seq_len=3000)
    p2 = synth.identity_paged(p, cfg.Hkv, cfg.D)
    q = synth.normal_bf16(21701, (3, 8, 129, 128))
    o1, l1 = run(gb, q, p, True, cfg.softmax_scale)
    o2, l2 = run(gb, q, p2, True, cfg.softmax_scale)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_paged_prefill_bad_length_is_flagged_not_fatal(gb):
    cfg = synth.DecodeConfig("bad", 3, 4, 2, 128, 1, 400, 16, 21800)
    p = synth.paged_inputs(cfg, seq_lens=[200, 300, 400], max_seq_len=400, poison=False)
    q = synth.normal_bf16(21801, (3, 4, 100, 128))
    p.seq_lens[1] = 401  # beyond max_kv_len
    o, lse = run(gb, q, p, True, cfg.softmax_scale, expect_flags=2)
    og, lg = from_dev(o), from_dev(lse)
    assert np.all(np.isnan(og[1])) and np.all(np.isnan(lg[1]))
    p.seq_lens[1] = 300
    o_ref, lse_ref = oracle.paged_prefill(q, p.k_pool, p.v_pool, p.block_table, p.seq_lens, True,
                                          cfg.softmax_scale)
    for b in (0, 2):
        check_close(og[b], lg[b], o_ref[b], lse_ref[b], f"good item {b}")
