"""attn_fwd (C ABI, sm_103a kernel) against the fp64 oracle on the same seeded inputs."""

from __future__ import annotations

import numpy as np
import pytest

import oracle
import synth
from gpu_util import check_close, from_dev, bits_of, to_dev

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def gb():
    import attention_flashattention_fwd_03_gb300 as gb
    gb.lib()
    return gb


def run(gb, q, k, v, causal, scale):
    qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
    o, lse = gb.attn_fwd(qd, kd, vd, causal=causal, scale=scale)
    torch.cuda.synchronize()
    st, flags = gb.attn_device_status()
    assert st == 0 and flags == 0, (st, flags)
    return o, lse


SMALL = [
    # B, Hq, Hkv, T, D, causal
    (1, 2, 2, 128, 64, True),     # the tiny causal workload
    (1, 2, 2, 128, 128, True),
    (1, 1, 1, 1, 64, True),
    (1, 1, 1, 1, 128, False),
    (2, 2, 1, 127, 128, True),
    (1, 4, 2, 129, 64, True),
    (1, 3, 3, 200, 128, False),
    (2, 6, 2, 257, 128, True),
    (1, 8, 1, 383, 64, False),
    (1, 4, 4, 1000, 128, True),
    (1, 2, 2, 1000, 64, False),
    (2, 8, 2, 640, 128, False),
]


@pytest.mark.parametrize("B,Hq,Hkv,T,D,causal", SMALL)
def test_attn_fwd_matches_oracle_small(gb, B, Hq, Hkv, T, D, causal):
    seed = 11000 + 7 * T + D + Hq
    q = synth.normal_bf16(seed, (B, Hq, T, D))
    k = synth.normal_bf16(seed + 1, (B, Hkv, T, D))
    v = synth.normal_bf16(seed + 2, (B, Hkv, T, D))
    scale = 1.0 / np.sqrt(D)
    o, lse = run(gb, q, k, v, causal, scale)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, causal, scale)
    check_close(from_dev(o), from_dev(lse), o_ref, lse_ref, f"{B},{Hq},{Hkv},{T},{D},{causal}")


@pytest.mark.parametrize("name", ["prefill_mha_causal", "prefill_gqa_long_causal", "noncausal_d64"])
def test_attn_fwd_full_size_every_row(gb, name):
    """The full-size workloads against the oracle on every output element.

    The error bounds hold over the whole of O and LSE (max and mean over all
    rows of all heads), not over a sample.
    """
    cfg = synth.CONFIGS[name]
    q, k, v = synth.prefill_inputs(cfg)
    o, lse = run(gb, q, k, v, cfg.causal, cfg.softmax_scale)
    og, lg = from_dev(o), from_dev(lse)
    del o, lse
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, cfg.causal, cfg.softmax_scale)
    mx, mean = check_close(og, lg, o_ref, lse_ref, name)
    lmx = float(np.abs(lg - lse_ref).max())
    print(f"PARITY {name} rows={og.size // cfg.D} o_max_abs={mx:.3e} o_mean_abs={mean:.3e} "
          f"lse_max_abs={lmx:.3e}")


def test_first_causal_row_is_v0_bit_exact(gb):
    B, Hq, Hkv, T, D = 2, 8, 2, 300, 128
    q = synth.normal_bf16(12001, (B, Hq, T, D))
    k = synth.normal_bf16(12002, (B, Hkv, T, D))
    v = synth.normal_bf16(12003, (B, Hkv, T, D))
    o, lse = run(gb, q, k, v, True, 0.0883883)
    ob = bits_of(o)
    g = Hq // Hkv
    for b in range(B):
        for h in range(Hq):
            assert np.array_equal(ob[b, h, 0], v[b, h // g, 0]), (b, h)
    qf, kf = synth.bf16_bits_to_float(q).astype(np.float64), synth.bf16_bits_to_float(k).astype(np.float64)
    s00 = 0.0883883 * np.einsum("bhd,bhd->bh", qf[:, :, 0], np.repeat(kf[:, :, 0], g, axis=1))
    assert np.abs(from_dev(lse)[:, :, 0] - s00).max() <= 1e-3


def test_constant_v_returns_the_constant(gb):
    B, Hq, Hkv, T, D = 1, 4, 4, 333, 64
    q = synth.normal_bf16(12101, (B, Hq, T, D))
    k = synth.normal_bf16(12102, (B, Hkv, T, D))
    c = synth.float_to_bf16_bits(np.linspace(-3, 3, D).astype(np.float32))
    v = np.broadcast_to(c, (B, Hkv, T, D)).copy()
    for causal in (True, False):
        o, _ = run(gb, q, k, v, causal, 0.125)
        err = np.abs(from_dev(o) - synth.bf16_bits_to_float(c)[None, None, None, :])
        assert err.max() <= 2e-2


def test_gqa_equals_repeated_mha_bit_exact(gb):
    B, Hq, Hkv, T, D = 1, 8, 2, 517, 128
    q = synth.normal_bf16(12201, (B, Hq, T, D))
    k = synth.normal_bf16(12202, (B, Hkv, T, D))
    v = synth.normal_bf16(12203, (B, Hkv, T, D))
    for causal in (True, False):
        o1, l1 = run(gb, q, k, v, causal, 0.09)
        o2, l2 = run(gb, q, np.repeat(k, 4, axis=1), np.repeat(v, 4, axis=1), causal, 0.09)
        assert np.array_equal(bits_of(o1), bits_of(o2))
        assert torch.equal(l1, l2)


def test_deterministic_run_to_run(gb):
    cfg = synth.PrefillConfig("det", 2, 16, 4, 1100, 128, True, 1.0, 12300)
    q, k, v = synth.prefill_inputs(cfg)
    o1, l1 = run(gb, q, k, v, True, cfg.softmax_scale)
    o2, l2 = run(gb, q, k, v, True, cfg.softmax_scale)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_large_scores_and_moving_max(gb):
    """Scores of magnitude ~1e2..1e3 and a row max that grows at every KV tile."""
    B, Hq, Hkv, T, D = 1, 2, 2, 700, 64
    q = synth.normal_bf16(12401, (B, Hq, T, D), 6.0)
    k = synth.normal_bf16(12402, (B, Hkv, T, D), 6.0)
    # make key j's projection on q grow with j so m moves every tile
    kf = synth.bf16_bits_to_float(k).copy()
    kf[..., 0] = np.linspace(-20, 20, T)[None, None, :]
    qf = synth.bf16_bits_to_float(q).copy()
    qf[..., 0] = 4.0
    q, k = synth.float_to_bf16_bits(qf), synth.float_to_bf16_bits(kf)
    v = synth.normal_bf16(12403, (B, Hkv, T, D))
    for causal in (True, False):
        o, lse = run(gb, q, k, v, causal, 0.125)
        o_ref, lse_ref = oracle.attn_fwd(q, k, v, causal, 0.125)
        check_close(from_dev(o), from_dev(lse), o_ref, lse_ref, f"large causal={causal}")


def test_no_lse_and_explicit_outputs(gb):
    B, Hq, Hkv, T, D = 1, 2, 1, 130, 128
    q = synth.normal_bf16(12501, (B, Hq, T, D))
    k = synth.normal_bf16(12502, (B, Hkv, T, D))
    v = synth.normal_bf16(12503, (B, Hkv, T, D))
    qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
    out = torch.full_like(qd, float("nan"))
    o, lse = gb.attn_fwd(qd, kd, vd, causal=True, scale=0.1, out=out, return_lse=False)
    torch.cuda.synchronize()
    assert lse is None and o.data_ptr() == out.data_ptr()
    o_ref, _ = oracle.attn_fwd(q, k, v, True, 0.1)
    check_close(from_dev(o), None, o_ref, None, "no-lse")


def test_runs_on_a_side_stream(gb):
    B, Hq, Hkv, T, D = 1, 4, 2, 256, 64
    q = synth.normal_bf16(12601, (B, Hq, T, D))
    k = synth.normal_bf16(12602, (B, Hkv, T, D))
    v = synth.normal_bf16(12603, (B, Hkv, T, D))
    qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        o, lse = gb.attn_fwd(qd, kd, vd, causal=False, scale=0.125)
    s.synchronize()
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, False, 0.125)
    check_close(from_dev(o), from_dev(lse), o_ref, lse_ref, "side stream")
