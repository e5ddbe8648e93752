"""Pins for the fp64 oracle: checks against things other than the oracle itself.

Each ``pin_*`` takes a loaded oracle library handle and raises AssertionError
when the oracle disagrees with what the mathematics fixes.  They are collected
into ``PINS`` so the same suite can be run against deliberately broken copies of
the oracle (tests/test_oracle_mutants.py): every planted mistake has to trip at
least one pin.

The attention being pinned is softmax attention as the pages describe it (the
naive matmul, scale, causal mask, softmax, matmul sequence of the Hugging Face
profiling guide on aiexpert.news, which FlashAttention reproduces blockwise per
the-ai.news section "Atencao do tipo FlashAttention e atencao paginada"), plus
paged decode through a block table of 16-token blocks (same section).
"""

from __future__ import annotations

import json
import math
import os

import numpy as np

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def f32(bits):
    return synth.bf16_bits_to_float(bits).astype(np.float64)


def bits(x):
    return synth.float_to_bf16_bits(np.asarray(x, dtype=np.float32))


def small_int_bf16(seed, shape, lo=-3, hi=3):
    """bf16 bits of small integers: sums and shifts of them stay exact."""
    vals = synth.uniform_ints(seed, int(np.prod(shape)), lo, hi).astype(np.float32)
    return bits(vals).reshape(shape)


# --------------------------------------------------------------------------- #
# 1. brute force in 40-digit arithmetic, textbook form exp(s_j) / sum_k exp(s_k)
# --------------------------------------------------------------------------- #

def _mp_attention(qf, kf, vf, causal, scale, group):
    import mpmath as mp
    mp.mp.dps = 40
    B, Hq, T, D = qf.shape
    o = np.zeros(qf.shape)
    lse = np.zeros((B, Hq, T))
    sc = mp.mpf(scale)
    for b in range(B):
        for h in range(Hq):
            kv = h // group
            for i in range(T):
                keys = range(0, i + 1) if causal else range(T)
                e = []
                for j in keys:
                    s = sc * mp.fsum(mp.mpf(float(qf[b, h, i, d])) * mp.mpf(float(kf[b, kv, j, d]))
                                     for d in range(D))
                    e.append(mp.exp(s))
                tot = mp.fsum(e)
                for d in range(D):
                    o[b, h, i, d] = float(mp.fsum(e[n] * mp.mpf(float(vf[b, kv, j, d]))
                                                  for n, j in enumerate(keys)) / tot)
                lse[b, h, i] = float(mp.log(tot))
    return o, lse


def pin_bruteforce_highprecision(lib):
    cases = [(1, 1, 1, 1, 1), (1, 2, 2, 3, 2), (2, 4, 2, 5, 3), (1, 3, 1, 6, 4), (1, 2, 1, 8, 4)]
    for n, (B, Hq, Hkv, T, D) in enumerate(cases):
        for causal in (False, True):
            seed = 7100 + 10 * n + causal
            q = synth.normal_bf16(seed, (B, Hq, T, D))
            k = synth.normal_bf16(seed + 1, (B, Hkv, T, D), 2.0)
            v = synth.normal_bf16(seed + 2, (B, Hkv, T, D))
            scale = 0.7
            o, lse = oracle.attn_fwd(q, k, v, causal, scale, lib=lib)
            eo, el = _mp_attention(f32(q), f32(k), f32(v), causal, scale, Hq // Hkv)
            assert np.abs(o - eo).max() <= 1e-13, ("O", B, Hq, Hkv, T, D, causal)
            assert np.abs(lse - el).max() <= 1e-13, ("LSE", B, Hq, Hkv, T, D, causal)


def _mp_rect(qf, kf, vf, causal, scale, group):
    """40-digit brute force for Tq query rows against Tk keys.  The Tq queries are
    the newest tokens of a Tk-token sequence, so query i sits at position
    Tk - Tq + i and, when causal, sees keys 0 .. Tk - Tq + i; a query that sees
    no key gives O = 0 and LSE = -inf."""
    import mpmath as mp
    mp.mp.dps = 40
    B, Hq, Tq, D = qf.shape
    Tk = kf.shape[2]
    o = np.zeros(qf.shape)
    lse = np.zeros((B, Hq, Tq))
    sc = mp.mpf(scale)
    for b in range(B):
        for h in range(Hq):
            kv = h // group
            for i in range(Tq):
                pos = Tk - Tq + i
                keys = [j for j in range(Tk) if (not causal or j <= pos)]
                if not keys:
                    lse[b, h, i] = -np.inf
                    continue
                e = [mp.exp(sc * mp.fsum(mp.mpf(float(qf[b, h, i, d])) * mp.mpf(float(kf[b, kv, j, d]))
                                         for d in range(D))) for j in keys]
                tot = mp.fsum(e)
                for d in range(D):
                    o[b, h, i, d] = float(mp.fsum(e[n] * mp.mpf(float(vf[b, kv, j, d]))
                                                  for n, j in enumerate(keys)) / tot)
                lse[b, h, i] = float(mp.log(tot))
    return o, lse


def pin_bottom_right_bruteforce(lib):
    """Tq != Tk: the queries are the last Tq tokens (chunked prefill / decode)."""
    cases = [(1, 2, 1, 2, 5, 3), (1, 2, 2, 1, 4, 2), (2, 4, 2, 3, 7, 2), (1, 2, 1, 5, 3, 2),
             (1, 1, 1, 4, 4, 3)]
    for n, (B, Hq, Hkv, Tq, Tk, D) in enumerate(cases):
        for causal in (True, False):
            seed = 7600 + 10 * n + causal
            q = synth.normal_bf16(seed, (B, Hq, Tq, D))
            k = synth.normal_bf16(seed + 1, (B, Hkv, Tk, D), 2.0)
            v = synth.normal_bf16(seed + 2, (B, Hkv, Tk, D))
            o, lse = oracle.attn_fwd(q, k, v, causal, 0.6, lib=lib)
            eo, el = _mp_rect(f32(q), f32(k), f32(v), causal, 0.6, Hq // Hkv)
            assert np.abs(o - eo).max() <= 1e-13, ("O", Tq, Tk, causal)
            fin = np.isfinite(el)
            assert np.array_equal(np.isneginf(lse), ~fin), ("empty rows", Tq, Tk, causal)
            assert np.abs(lse[fin] - el[fin]).max() <= 1e-13, ("LSE", Tq, Tk, causal)


def pin_chunk_is_tail_of_full(lib):
    """Causal attention of the last Tq queries against all Tk keys equals the last Tq
    rows of causal attention of the whole Tk-token sequence, bit for bit."""
    B, Hq, Hkv, Tk, D = 1, 4, 2, 70, 16
    qfull = synth.normal_bf16(7700, (B, Hq, Tk, D))
    k = synth.normal_bf16(7701, (B, Hkv, Tk, D))
    v = synth.normal_bf16(7702, (B, Hkv, Tk, D))
    of, lf = oracle.attn_fwd(qfull, k, v, True, 0.3, lib=lib)
    for Tq in (1, 2, 17, 69, 70):
        o, lse = oracle.attn_fwd(np.ascontiguousarray(qfull[:, :, Tk - Tq:]), k, v, True, 0.3,
                                 lib=lib)
        assert np.array_equal(o, of[:, :, Tk - Tq:]) and np.array_equal(lse, lf[:, :, Tk - Tq:]), Tq


# --------------------------------------------------------------------------- #
# 2. library special case: torch SDPA (fp64, CPU) and scipy logsumexp
# --------------------------------------------------------------------------- #

def pin_library_sdpa(lib):
    import torch
    from scipy.special import logsumexp
    cases = [
        (synth.CONFIGS["tiny_causal"], None),
        (synth.PrefillConfig("gqa_cut", 2, 8, 2, 67, 64, True, 1.0, 7200), None),
        (synth.PrefillConfig("noncausal_cut", 1, 4, 4, 45, 128, False, 0.5, 7300, 0.09), None),
    ]
    for cfg, _ in cases:
        q, k, v = synth.prefill_inputs(cfg)
        scale = cfg.softmax_scale
        o, lse = oracle.attn_fwd(q, k, v, cfg.causal, scale, lib=lib)
        g = cfg.Hq // cfg.Hkv
        qt = torch.from_numpy(f32(q))
        kt = torch.from_numpy(f32(k)).repeat_interleave(g, dim=1)
        vt = torch.from_numpy(f32(v)).repeat_interleave(g, dim=1)
        ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=cfg.causal,
                                                               scale=scale)
        assert np.abs(o - ref.numpy()).max() <= 1e-12, cfg.name
        s = torch.matmul(qt, kt.transpose(-1, -2)).numpy() * scale
        if cfg.causal:
            T = cfg.T
            s = np.where(np.tril(np.ones((T, T), dtype=bool)), s, -np.inf)
        assert np.abs(lse - logsumexp(s, axis=-1)).max() <= 1e-12, cfg.name


# --------------------------------------------------------------------------- #
# 3. invariants and closed forms
# --------------------------------------------------------------------------- #

def pin_rows_sum_to_one(lib):
    for causal in (True, False):
        cfg = synth.PrefillConfig("rows", 1, 4, 2, 50, 32, causal, 1.0, 7400)
        q, k, v = synth.prefill_inputs(cfg)
        rows = np.arange(cfg.B * cfg.Hq * cfg.T)
        _, _, p = oracle.attn_rows(q, k, v, causal, cfg.softmax_scale, rows, want_probs=True,
                                   lib=lib)
        assert np.all(p >= 0)
        assert np.abs(p.sum(axis=1) - 1.0).max() <= 1e-12
        if causal:
            i = rows % cfg.T
            future = np.arange(cfg.T)[None, :] > i[:, None]
            assert np.all(p[future] == 0.0)
            assert np.all(p[~future] > 0.0)


def pin_constant_v(lib):
    for causal in (True, False):
        B, Hq, Hkv, T, D = 2, 4, 2, 37, 16
        q = synth.normal_bf16(7500, (B, Hq, T, D))
        k = synth.normal_bf16(7501, (B, Hkv, T, D))
        c = np.linspace(-2.0, 2.0, D).astype(np.float32)
        v = np.broadcast_to(bits(c), (B, Hkv, T, D)).copy()
        o, _ = oracle.attn_fwd(q, k, v, causal, 0.3, lib=lib)
        assert np.abs(o - f32(bits(c))[None, None, None, :]).max() <= 1e-12


def pin_first_causal_row(lib):
    B, Hq, Hkv, T, D = 1, 4, 2, 24, 64
    q = synth.normal_bf16(7600, (B, Hq, T, D))
    k = synth.normal_bf16(7601, (B, Hkv, T, D))
    v = synth.normal_bf16(7602, (B, Hkv, T, D))
    scale = 0.125
    o, lse = oracle.attn_fwd(q, k, v, True, scale, lib=lib)
    qf, kf, vf = f32(q), f32(k), f32(v)
    for h in range(Hq):
        kv = h // (Hq // Hkv)
        assert np.array_equal(o[0, h, 0], vf[0, kv, 0])
        # products of bf16 pairs are exact in fp64 and these sums stay exact
        s00 = scale * math.fsum(qf[0, h, 0] * kf[0, kv, 0])
        assert abs(lse[0, h, 0] - s00) <= 1e-13


def pin_zero_query(lib):
    for causal in (True, False):
        B, Hq, Hkv, T, D = 1, 2, 1, 31, 8
        q = np.zeros((B, Hq, T, D), dtype=np.uint16)
        k = synth.normal_bf16(7700, (B, Hkv, T, D))
        v = synth.normal_bf16(7701, (B, Hkv, T, D))
        o, lse = oracle.attn_fwd(q, k, v, causal, 0.5, lib=lib)
        vf = f32(v)[0, 0]
        for i in range(T):
            n = i + 1 if causal else T
            assert np.abs(o[0, :, i] - vf[:n].mean(axis=0)).max() <= 1e-13
            assert np.abs(lse[0, :, i] - math.log(n)).max() <= 1e-13


def pin_key_shift(lib):
    """k_j -> k_j + w for all j: O unchanged, LSE_i shifts by scale * q_i . w."""
    B, Hq, Hkv, T, D = 1, 2, 2, 19, 8
    q = small_int_bf16(7800, (B, Hq, T, D))
    k = small_int_bf16(7801, (B, Hkv, T, D))
    v = synth.normal_bf16(7802, (B, Hkv, T, D))
    w = np.arange(D, dtype=np.float32) - 3.0
    k2 = bits(f32(k) + w)
    assert np.array_equal(f32(k2), f32(k) + w)
    scale = 0.25
    for causal in (True, False):
        o1, l1 = oracle.attn_fwd(q, k, v, causal, scale, lib=lib)
        o2, l2 = oracle.attn_fwd(q, k2, v, causal, scale, lib=lib)
        assert np.abs(o1 - o2).max() <= 1e-12
        shift = scale * (f32(q) @ w.astype(np.float64))
        assert np.abs((l2 - l1) - shift).max() <= 1e-12


def pin_key_permutation(lib):
    """Non-causal attention does not depend on the order of the (k, v) pairs."""
    B, Hq, Hkv, T, D = 1, 2, 1, 29, 16
    q = synth.normal_bf16(7900, (B, Hq, T, D))
    k = synth.normal_bf16(7901, (B, Hkv, T, D))
    v = synth.normal_bf16(7902, (B, Hkv, T, D))
    perm = synth.permutation(7903, T)
    o1, l1 = oracle.attn_fwd(q, k, v, False, 0.3, lib=lib)
    o2, l2 = oracle.attn_fwd(q, k[:, :, perm], v[:, :, perm], False, 0.3, lib=lib)
    assert np.abs(o1 - o2).max() <= 1e-12 and np.abs(l1 - l2).max() <= 1e-12


def pin_gqa_is_repeated_mha(lib):
    B, Hq, Hkv, T, D = 2, 6, 2, 23, 16
    q = synth.normal_bf16(8000, (B, Hq, T, D))
    k = synth.normal_bf16(8001, (B, Hkv, T, D))
    v = synth.normal_bf16(8002, (B, Hkv, T, D))
    g = Hq // Hkv
    for causal in (True, False):
        o1, l1 = oracle.attn_fwd(q, k, v, causal, 0.2, lib=lib)
        o2, l2 = oracle.attn_fwd(q, np.repeat(k, g, axis=1), np.repeat(v, g, axis=1), causal, 0.2,
                                 lib=lib)
        assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def pin_scale_moves_into_q(lib):
    """Scale 2s with q equals scale s with 2q (doubling a bf16 value is exact)."""
    B, Hq, Hkv, T, D = 1, 2, 2, 17, 32
    q = synth.normal_bf16(8100, (B, Hq, T, D))
    k = synth.normal_bf16(8101, (B, Hkv, T, D))
    v = synth.normal_bf16(8102, (B, Hkv, T, D))
    q2 = bits(f32(q) * 2.0)
    for causal in (True, False):
        o1, l1 = oracle.attn_fwd(q, k, v, causal, 0.4, lib=lib)
        o2, l2 = oracle.attn_fwd(q2, k, v, causal, 0.2, lib=lib)
        assert np.abs(o1 - o2).max() <= 1e-13 and np.abs(l1 - l2).max() <= 1e-13


def pin_large_scores(lib):
    """Scores of magnitude ~1e3: no overflow, LSE between max and max + ln n."""
    B, Hq, Hkv, T, D = 1, 2, 1, 40, 16
    q = synth.normal_bf16(8200, (B, Hq, T, D), 30.0)
    k = synth.normal_bf16(8201, (B, Hkv, T, D), 30.0)
    v = synth.normal_bf16(8202, (B, Hkv, T, D))
    o, lse = oracle.attn_fwd(q, k, v, True, 1.0 / 4.0, lib=lib)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
    s = np.einsum("hid,jd->hij", f32(q)[0], f32(k)[0, 0]) * 0.25
    for i in range(T):
        m = s[:, i, :i + 1].max(axis=1)
        assert np.all(lse[0, :, i] >= m - 1e-9) and np.all(lse[0, :, i] <= m + math.log(i + 1) + 1e-9)
    # and O is a convex combination of the visible values
    vf = f32(v)[0, 0]
    for i in range(T):
        lo, hi = vf[:i + 1].min(axis=0), vf[:i + 1].max(axis=0)
        assert np.all(o[0, :, i] >= lo - 1e-12) and np.all(o[0, :, i] <= hi + 1e-12)


def pin_increasing_scores(lib):
    """Scores grow with j (k_j = j*u, q along u), the row max moves at every key."""
    T, D = 64, 8
    u = np.zeros(D, dtype=np.float32)
    u[0] = 1.0
    k = bits((np.arange(T, dtype=np.float32)[:, None] * u[None, :]) / 8.0).reshape(1, 1, T, D)
    q = bits(np.tile(u, (T, 1))).reshape(1, 1, T, D)
    v = synth.normal_bf16(8300, (1, 1, T, D))
    scale = 1.0
    o, lse = oracle.attn_fwd(q, k, v, True, scale, lib=lib)
    # closed form: s_j = j/8; LSE_i = ln sum_{j<=i} e^{j/8}; O_i = sum_j e^{j/8} v_j / sum e^{j/8}
    vf = f32(v)[0, 0]
    for i in range(T):
        w = np.exp(np.arange(i + 1) / 8.0)
        assert abs(lse[0, 0, i] - math.log(w.sum())) <= 1e-12
        assert np.abs(o[0, 0, i] - (w[:, None] * vf[:i + 1]).sum(0) / w.sum()).max() <= 1e-12


# --------------------------------------------------------------------------- #
# 4. paged decode
# --------------------------------------------------------------------------- #

def _small_paged(seed, num_seqs=5, Hq=6, Hkv=2, D=16, lens=(1, 15, 16, 17, 70)):
    cfg = synth.DecodeConfig("small", num_seqs, Hq, Hkv, D, 1, 80, 16, seed)
    return cfg, synth.paged_inputs(cfg, seq_lens=list(lens)[:num_seqs], max_seq_len=96)


def pin_paged_gather_is_table_lookup(lib):
    """The oracle's gather equals numpy indexing pool[table[t // bs], h, t % bs]."""
    cfg, p = _small_paged(8400)
    for r in range(len(p.seq_lens)):
        L = int(p.seq_lens[r])
        t = np.arange(L)
        phys = p.block_table[r, t // p.block_size]
        for h in range(cfg.Hkv):
            exp = p.k_pool[phys, h, t % p.block_size]
            got = oracle.paged_gather(p.k_pool, p.block_table, p.seq_lens, r, h, lib=lib)
            assert np.array_equal(exp, got)


def pin_paged_equals_contiguous(lib):
    """Decode through the table equals the last causal row over the gathered K/V."""
    cfg, p = _small_paged(8500)
    o, lse = oracle.paged_decode(p.q, p.k_pool, p.v_pool, p.block_table, p.seq_lens,
                                 cfg.softmax_scale, lib=lib)
    for r in range(len(p.seq_lens)):
        L = int(p.seq_lens[r])
        t = np.arange(L)
        phys = p.block_table[r, t // p.block_size]
        kc = np.stack([p.k_pool[phys, h, t % p.block_size] for h in range(cfg.Hkv)])[None]
        vc = np.stack([p.v_pool[phys, h, t % p.block_size] for h in range(cfg.Hkv)])[None]
        qf = np.zeros((1, cfg.Hq, L, cfg.D), dtype=np.uint16)
        qf[0, :, L - 1] = p.q[r]
        rows = np.array([h * L + (L - 1) for h in range(cfg.Hq)])
        oc, lc = oracle.attn_rows(qf, kc, vc, True, cfg.softmax_scale, rows, lib=lib)
        assert np.array_equal(oc, o[r]) and np.array_equal(lc, lse[r]), r


def pin_paged_placement_invariance(lib):
    """Moving the blocks (another table, same logical KV) leaves decode unchanged."""
    cfg, p = _small_paged(8600)
    p2 = synth.identity_paged(p, cfg.Hkv, cfg.D)
    o1, l1 = oracle.paged_decode(p.q, p.k_pool, p.v_pool, p.block_table, p.seq_lens,
                                 cfg.softmax_scale, lib=lib)
    o2, l2 = oracle.paged_decode(p2.q, p2.k_pool, p2.v_pool, p2.block_table, p2.seq_lens,
                                 cfg.softmax_scale, lib=lib)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def pin_paged_empty_request(lib):
    cfg, p = _small_paged(8700, num_seqs=3, lens=(0, 5, 0))
    o, lse = oracle.paged_decode(p.q, p.k_pool, p.v_pool, p.block_table, p.seq_lens,
                                 cfg.softmax_scale, lib=lib)
    assert np.all(o[0] == 0) and np.all(o[2] == 0)
    assert np.all(np.isneginf(lse[0])) and np.all(np.isneginf(lse[2]))
    assert np.all(np.isfinite(o[1])) and np.all(np.isfinite(lse[1]))


def pin_paged_prefill_is_gather_then_attention(lib):
    """Chunked prefill through the table equals attention over the gathered K/V with
    the chunk as the newest tokens; with one query it is paged decode, bit for bit."""
    cfg, p = _small_paged(8650, lens=(1, 15, 16, 17, 70))
    B, Tq = len(p.seq_lens), 1
    q1 = p.q[:, :, None, :].copy()
    o, lse = oracle.paged_prefill(q1, p.k_pool, p.v_pool, p.block_table, p.seq_lens, True,
                                  cfg.softmax_scale, lib=lib)
    od, ld = oracle.paged_decode(p.q, p.k_pool, p.v_pool, p.block_table, p.seq_lens,
                                 cfg.softmax_scale, lib=lib)
    assert np.array_equal(o[:, :, 0], od) and np.array_equal(lse[:, :, 0], ld)
    Tq = 5
    q = synth.normal_bf16(8651, (B, cfg.Hq, Tq, cfg.D))
    for causal in (True, False):
        o, lse = oracle.paged_prefill(q, p.k_pool, p.v_pool, p.block_table, p.seq_lens, causal,
                                      cfg.softmax_scale, lib=lib)
        for b in range(B):
            L = int(p.seq_lens[b])
            t = np.arange(L)
            phys = p.block_table[b, t // p.block_size]
            kc = np.stack([p.k_pool[phys, h, t % p.block_size] for h in range(cfg.Hkv)])[None]
            vc = np.stack([p.v_pool[phys, h, t % p.block_size] for h in range(cfg.Hkv)])[None]
            oc, lc = oracle.attn_fwd(q[b:b + 1], kc, vc, causal, cfg.softmax_scale, lib=lib)
            assert np.array_equal(oc[0], o[b]) and np.array_equal(lc[0], lse[b]), (b, causal)
        if causal:  # request 0 has one key: only its last query sees it
            assert np.all(o[0, :, :Tq - 1] == 0) and np.all(np.isneginf(lse[0, :, :Tq - 1]))


def pin_split_merge(lib):
    """Merging per-chunk (O_s, LSE_s) with weights e^{LSE_s - LSE} gives the unsplit result."""
    B, Hq, Hkv, T, D = 1, 2, 1, 1300, 16
    q = synth.normal_bf16(8800, (B, Hq, 1, D))
    k = synth.normal_bf16(8801, (B, Hkv, T, D))
    v = synth.normal_bf16(8802, (B, Hkv, T, D))
    o, lse = oracle.attn_fwd(q, k, v, False, 0.25, lib=lib)
    parts = [oracle.attn_fwd(q, k[:, :, c:c + 512], v[:, :, c:c + 512], False, 0.25, lib=lib)
             for c in range(0, T, 512)]
    ls = np.stack([pl for _, pl in parts])
    M = ls.max(axis=0)
    tot = np.log(np.exp(ls - M).sum(axis=0)) + M
    om = sum(np.exp(pl - tot)[..., None] * po for po, pl in parts)
    assert np.abs(tot - lse).max() <= 1e-12 and np.abs(om - o).max() <= 1e-12


# --------------------------------------------------------------------------- #
# 5. hand-derived golden fixtures
# --------------------------------------------------------------------------- #

def _ev(x):
    return np.vectorize(lambda s: float(eval(s, {"math": math})), otypes=[float])(np.array(x))


def pin_golden_attention(lib):
    for name in ("two_keys.json", "gqa_mapping.json"):
        with open(os.path.join(GOLDEN, name)) as fh:
            g = json.load(fh)
        q, k, v = bits(g["q"]), bits(g["k"]), bits(g["v"])
        scale = float(eval(g["scale"], {"math": math}))
        for mode, exp in g["expected"].items():
            o, lse = oracle.attn_fwd(q, k, v, mode == "causal", scale, lib=lib)
            assert np.abs(o - _ev(exp["o"])).max() <= 1e-14, (name, mode)
            assert np.abs(lse - _ev(exp["lse"])).max() <= 1e-14, (name, mode)


def pin_golden_paged(lib):
    with open(os.path.join(GOLDEN, "paged_translation.json")) as fh:
        g = json.load(fh)
    NB, Hkv, bs, D = g["num_pool_blocks"], g["Hkv"], g["block_size"], g["D"]
    code = (32 * np.arange(NB)[:, None, None] + 16 * np.arange(Hkv)[None, :, None]
            + np.arange(bs)[None, None, :]).astype(np.float32)
    pool = bits(np.stack([code, -code], axis=-1))
    table = np.full((1, 4), -1, dtype=np.int32)
    table[0, :2] = g["block_table"][0]
    sl = np.array(g["seq_lens"], dtype=np.int32)
    for h in range(Hkv):
        got = f32(oracle.paged_gather(pool, table, sl, 0, h, lib=lib))
        assert np.array_equal(got[:, 0], np.array(g["expected_gather_dim0"][str(h)], float))
        assert np.array_equal(got[:, 1], -got[:, 0])
    q = np.zeros((1, g["Hq"], D), dtype=np.uint16)
    o, lse = oracle.paged_decode(q, pool, pool, table, sl, 0.5, lib=lib)
    assert np.abs(o[0] - _ev(g["expected_decode_q0"]["o"])).max() <= 1e-12
    assert np.abs(lse - _ev(g["expected_decode_q0"]["lse"])).max() <= 1e-14


PINS = [
    pin_bruteforce_highprecision,
    pin_bottom_right_bruteforce,
    pin_chunk_is_tail_of_full,
    pin_paged_prefill_is_gather_then_attention,
    pin_library_sdpa,
    pin_rows_sum_to_one,
    pin_constant_v,
    pin_first_causal_row,
    pin_zero_query,
    pin_key_shift,
    pin_key_permutation,
    pin_gqa_is_repeated_mha,
    pin_scale_moves_into_q,
    pin_large_scores,
    pin_increasing_scores,
    pin_paged_gather_is_table_lookup,
    pin_paged_equals_contiguous,
    pin_paged_placement_invariance,
    pin_paged_empty_request,
    pin_split_merge,
    pin_golden_attention,
    pin_golden_paged,
]
