"""paged_attn_decode (C ABI, sm_103a kernels) against the fp64 oracle."""

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


def run(gb, p: synth.PagedInputs, scale, max_seq_len=None, expect_flags=0):
    msl = p.max_seq_len if max_seq_len is None else max_seq_len
    o, lse = gb.paged_attn_decode(to_dev(p.q), to_dev(p.k_pool), to_dev(p.v_pool),
                                  to_dev_i32(p.block_table), to_dev_i32(p.seq_lens), msl,
                                  scale=scale)
    torch.cuda.synchronize()
    st, flags = gb.attn_device_status()
    assert flags == expect_flags, (st, flags)
    return o, lse


@pytest.fixture(scope="module")
def cfg5():
    cfg = synth.CONFIGS["paged_decode"]
    return cfg, synth.paged_inputs(cfg)


def test_decode_full_size_matches_oracle(gb, cfg5):
    cfg, p = cfg5
    o, lse = run(gb, p, cfg.softmax_scale)
    o_ref, lse_ref = oracle.paged_decode(p.q, p.k_pool, p.v_pool, p.block_table, p.seq_lens,
                                         cfg.softmax_scale)
    of, lf = from_dev(o), from_dev(lse)
    mx, mean = check_close(of, lf, o_ref, lse_ref, "paged_decode")
    print(f"PARITY paged_decode rows={of.size // cfg.D} o_max_abs={mx:.3e} o_mean_abs={mean:.3e} "
          f"lse_max_abs={float(np.abs(lf - lse_ref).max()):.3e}")


def test_decode_placement_invariance_bit_exact(gb, cfg5):
    """Random-permutation table vs an identity-like table over the same logical KV."""
    cfg, p = cfg5
    p2 = synth.identity_paged(p, cfg.Hkv, cfg.D)
    o1, l1 = run(gb, p, cfg.softmax_scale)
    o2, l2 = run(gb, p2, cfg.softmax_scale)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_decode_deterministic(gb, cfg5):
    cfg, p = cfg5
    o1, l1 = run(gb, p, cfg.softmax_scale)
    o2, l2 = run(gb, p, cfg.softmax_scale)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


EDGE_LENS = [1, 2, 15, 16, 17, 31, 255, 511, 512, 513, 1024, 1500, 2048, 2049]


@pytest.mark.parametrize("Hq,Hkv,D", [(12, 2, 128), (8, 8, 128), (16, 1, 64), (4, 2, 64),
                                      (32, 2, 128), (6, 6, 64), (20, 2, 128), (9, 1, 64)])
def test_decode_edge_lengths_and_groups(gb, Hq, Hkv, D):
    cfg = synth.DecodeConfig("edge", len(EDGE_LENS), Hq, Hkv, D, 1, 2049, 16,
                             13000 + Hq * 10 + D)
    p = synth.paged_inputs(cfg, seq_lens=EDGE_LENS, max_seq_len=2100)
    o, lse = run(gb, p, cfg.softmax_scale)
    o_ref, lse_ref = oracle.paged_decode(p.q, p.k_pool, p.v_pool, p.block_table, p.seq_lens,
                                         cfg.softmax_scale)
    check_close(from_dev(o), from_dev(lse), o_ref, lse_ref, f"edge {Hq},{Hkv},{D}")


def test_decode_long_requests_cut_into_many_pieces(gb):
    """A batch of few, long requests: the work is cut into ranges of 16 blocks, so
    the 16384-token request spans 65 pieces per head (two merge batches of 32) and
    the others 36 and 1."""
    lens = [16384, 9000, 1]
    cfg = synth.DecodeConfig("pieces", len(lens), 12, 2, 128, 1, 16384, 16, 13050)
    p = synth.paged_inputs(cfg, seq_lens=lens, max_seq_len=16384)
    o, lse = run(gb, p, cfg.softmax_scale)
    o_ref, lse_ref = oracle.paged_decode(p.q, p.k_pool, p.v_pool, p.block_table, p.seq_lens,
                                         cfg.softmax_scale)
    check_close(from_dev(o), from_dev(lse), o_ref, lse_ref, "many pieces")


def test_decode_many_short_requests(gb):
    """300 requests of 0..40 tokens: each warp's range crosses many one- to
    three-block segments and skips the empty requests between them."""
    rng = np.random.default_rng(13070)
    lens = rng.choice([0, 1, 2, 15, 16, 17, 31, 33, 40], size=300).astype(np.int32)
    cfg = synth.DecodeConfig("short", len(lens), 8, 2, 64, 0, 40, 16, 13070)
    p = synth.paged_inputs(cfg, seq_lens=lens, max_seq_len=48)
    o, lse = run(gb, p, cfg.softmax_scale)
    o_ref, lse_ref = oracle.paged_decode(p.q, p.k_pool, p.v_pool, p.block_table, p.seq_lens,
                                         cfg.softmax_scale)
    live = p.seq_lens > 0
    check_close(from_dev(o)[live], from_dev(lse)[live], o_ref[live], lse_ref[live], "short")
    assert np.all(from_dev(o)[~live] == 0) and np.all(np.isneginf(from_dev(lse)[~live]))


def test_decode_single_token_returns_v0_bit_exact(gb):
    cfg = synth.DecodeConfig("one", 3, 12, 2, 128, 1, 1, 16, 13100)
    p = synth.paged_inputs(cfg, seq_lens=[1, 1, 1], max_seq_len=16)
    o, _ = run(gb, p, cfg.softmax_scale)
    ob = bits_of(o)
    for r in range(3):
        phys = p.block_table[r, 0]
        for h in range(12):
            assert np.array_equal(ob[r, h], p.v_pool[phys, h // 6, 0])


def test_decode_empty_request(gb):
    cfg = synth.DecodeConfig("empty", 3, 8, 2, 128, 0, 40, 16, 13200)
    p = synth.paged_inputs(cfg, seq_lens=[0, 37, 0], max_seq_len=64)
    o, lse = run(gb, p, cfg.softmax_scale)
    of, lf = from_dev(o), from_dev(lse)
    assert np.all(of[0] == 0) and np.all(of[2] == 0)
    assert np.all(np.isneginf(lf[0])) and np.all(np.isneginf(lf[2]))
    o_ref, lse_ref = oracle.paged_decode(p.q, p.k_pool, p.v_pool, p.block_table, p.seq_lens,
                                         cfg.softmax_scale)
    check_close(of[1], lf[1], o_ref[1], lse_ref[1], "empty neighbours")


def test_decode_equals_last_causal_row(gb):
    """Decode over a request equals row L-1 of causal attn_fwd over the same K/V."""
    L, Hq, Hkv, D = 777, 8, 2, 128
    cfg = synth.DecodeConfig("last", 1, Hq, Hkv, D, L, L, 16, 13300)
    p = synth.paged_inputs(cfg, seq_lens=[L], max_seq_len=L)
    o_dec, l_dec = run(gb, p, cfg.softmax_scale)
    t = np.arange(L)
    phys = p.block_table[0, t // 16]
    kc = np.stack([p.k_pool[phys, h, t % 16] for h in range(Hkv)])[None]
    vc = np.stack([p.v_pool[phys, h, t % 16] for h in range(Hkv)])[None]
    qc = synth.normal_bf16(13301, (1, Hq, L, D))
    qc[0, :, L - 1] = p.q[0]
    o_full, l_full = gb.attn_fwd(to_dev(qc), to_dev(kc), to_dev(vc), causal=True,
                                 scale=cfg.softmax_scale)
    torch.cuda.synchronize()
    assert np.abs(from_dev(o_dec)[0] - from_dev(o_full)[0, :, L - 1]).max() <= 2e-2
    assert np.abs(from_dev(l_dec)[0] - from_dev(l_full)[0, :, L - 1]).max() <= 1e-3


def test_decode_bad_request_data_is_flagged_not_fatal(gb):
    cfg = synth.DecodeConfig("bad", 4, 12, 2, 128, 1, 100, 16, 13400)
    p = synth.paged_inputs(cfg, seq_lens=[40, 50, 60, 70], max_seq_len=100, poison=False)
    # request 1: a block id outside the pool; request 2: a length beyond max_seq_len
    p.block_table[1, 1] = p.num_pool_blocks + 5
    p.seq_lens[2] = 101
    o, lse = run(gb, p, cfg.softmax_scale, max_seq_len=100, expect_flags=2 | 4)
    of, lf = from_dev(o), from_dev(lse)
    assert np.all(np.isnan(of[1])) and np.all(np.isnan(lf[1]))
    assert np.all(np.isnan(of[2])) and np.all(np.isnan(lf[2]))
    p.block_table[1, 1] = 0
    p.seq_lens[2] = 60
    o_ref, lse_ref = oracle.paged_decode(p.q, p.k_pool, p.v_pool, p.block_table, p.seq_lens,
                                         cfg.softmax_scale)
    for r in (0, 3):
        check_close(of[r], lf[r], o_ref[r], lse_ref[r], f"good request {r}")
