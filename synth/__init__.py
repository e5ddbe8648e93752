"""Seeded synthetic inputs shared by the oracle tests, the GPU tests and the bench.

This module draws numbers and lays out buffers; it holds none of the attention
arithmetic.  Everything is a pure function of (seed, shape), so the CUDA path and
the fp64 oracle always see identical bytes.

Recipe (the same on every machine, numpy only):

* ``splitmix64`` as a counter-based generator: draw ``i`` of a stream seeded with
  ``s`` is ``mix64(s + (i + 1) * 0x9E3779B97F4A7C15)`` (Steele, Lea & Flood,
  "Fast splittable pseudorandom number generators", OOPSLA 2014).
* Uniforms ``u = (x >> 11) * 2**-53`` in [0, 1).
* Normals by Box-Muller on consecutive uniform pairs:
  ``r = sqrt(-2 ln(1 - u0))``, ``z0 = r cos(2 pi u1)``, ``z1 = r sin(2 pi u1)``.
* Values are scaled in float64, cast to float32, then rounded to bfloat16 with
  round-to-nearest-even; tensors are returned as ``uint16`` arrays of bf16 bit
  patterns so both sides start from the exact same numbers.

The workloads are the ones the pages' method is run on: causal and non-causal
prefill attention in the ``[B, H, T, D]`` layout of
``torch.nn.functional.scaled_dot_product_attention``, and single-token decode
against a paged KV cache of 16-token blocks whose block tables are a random
permutation of free pool slots.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

BF16_NAN = np.uint16(0x7FC0)


def splitmix64(seed: int, n: int, offset: int = 0) -> np.ndarray:
    """Draws ``offset .. offset+n-1`` of the splitmix64 stream seeded by ``seed``."""
    z = np.arange(offset + 1, offset + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        np.multiply(z, _GOLDEN, out=z)
        np.add(z, np.uint64(seed & 0xFFFFFFFFFFFFFFFF), out=z)
        np.bitwise_xor(z, z >> np.uint64(30), out=z)
        np.multiply(z, _M1, out=z)
        np.bitwise_xor(z, z >> np.uint64(27), out=z)
        np.multiply(z, _M2, out=z)
        np.bitwise_xor(z, z >> np.uint64(31), out=z)
    return z


def uniforms(seed: int, n: int, offset: int = 0) -> np.ndarray:
    """``n`` float64 uniforms in [0, 1) with 53 random bits each."""
    return (splitmix64(seed, n, offset) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


_CHUNK = 1 << 21


def normals(seed: int, n: int) -> np.ndarray:
    """``n`` float64 N(0, 1) draws (Box-Muller on pairs of uniforms)."""
    m = (n + 1) // 2
    out = np.empty(2 * m, dtype=np.float64)
    for c0 in range(0, m, _CHUNK):
        c1 = min(m, c0 + _CHUNK)
        u = uniforms(seed, 2 * (c1 - c0), 2 * c0)
        u0, u1 = u[0::2], u[1::2]
        r = np.sqrt(-2.0 * np.log1p(-u0))
        ang = (2.0 * math.pi) * u1
        out[2 * c0:2 * c1:2] = r * np.cos(ang)
        out[2 * c0 + 1:2 * c1:2] = r * np.sin(ang)
    return out[:n]


def float_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, round-to-nearest-even (NaN kept quiet)."""
    f = np.ascontiguousarray(x, dtype=np.float32)
    b = f.view(np.uint32)
    rounding = ((b >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    with np.errstate(over="ignore"):
        out = ((b + rounding) >> np.uint32(16)).astype(np.uint16)
    nan = np.isnan(f)
    if nan.any():
        out[nan] = BF16_NAN
    return out


def bf16_bits_to_float(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float32 (exact)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32)


def normal_bf16(seed: int, shape, mult: float = 1.0) -> np.ndarray:
    """Seeded iid N(0,1)*mult tensor as bf16 bits of the given shape."""
    n = int(np.prod(shape))
    vals = normals(seed, n) * mult
    return float_to_bf16_bits(vals.astype(np.float32)).reshape(shape)


def uniform_ints(seed: int, n: int, lo: int, hi: int) -> np.ndarray:
    """``n`` integers uniform on [lo, hi] inclusive (modulo reduction of 64-bit draws)."""
    span = np.uint64(hi - lo + 1)
    return (splitmix64(seed, n) % span).astype(np.int64) + lo


def permutation(seed: int, n: int) -> np.ndarray:
    """Fisher-Yates shuffle of ``range(n)`` driven by splitmix64 draws."""
    perm = np.arange(n, dtype=np.int64)
    draws = splitmix64(seed, max(n - 1, 0))
    for step, i in enumerate(range(n - 1, 0, -1)):
        j = int(draws[step] % np.uint64(i + 1))
        perm[i], perm[j] = perm[j], perm[i]
    return perm


# --------------------------------------------------------------------------- #
# Workload definitions
# --------------------------------------------------------------------------- #

@dataclass(frozen=True)
class PrefillConfig:
    name: str
    B: int
    Hq: int
    Hkv: int
    T: int
    D: int
    causal: bool
    mult: float = 1.0
    seed: int = 0
    scale: float | None = None  # None -> 1/sqrt(D)

    @property
    def softmax_scale(self) -> float:
        return self.scale if self.scale is not None else 1.0 / math.sqrt(self.D)

    def flops(self) -> float:
        """FlashAttention convention: 4*B*Hq*T*T*D, halved when causal."""
        f = 4.0 * self.B * self.Hq * self.T * self.T * self.D
        return f / 2 if self.causal else f

    def flops_exact(self) -> float:
        """Multiply-adds actually required: causal visits T(T+1)/2 (i, j) pairs."""
        pairs = self.T * (self.T + 1) / 2 if self.causal else self.T * self.T
        return 4.0 * self.B * self.Hq * pairs * self.D

    def io_bytes(self) -> int:
        """Q, K, V read once and O (bf16) + LSE (fp32) written once."""
        q = self.B * self.Hq * self.T * self.D * 2
        kv = 2 * self.B * self.Hkv * self.T * self.D * 2
        o = q
        lse = self.B * self.Hq * self.T * 4
        return q + kv + o + lse


@dataclass(frozen=True)
class DecodeConfig:
    name: str
    num_seqs: int
    Hq: int
    Hkv: int
    D: int
    len_lo: int
    len_hi: int
    block_size: int = 16
    seed: int = 0
    scale: float | None = None
    mult: float = 1.0
    spare_frac: int = 8  # pool = used blocks + ceil(used / spare_frac)

    @property
    def softmax_scale(self) -> float:
        return self.scale if self.scale is not None else 1.0 / math.sqrt(self.D)


CONFIGS = {
    "tiny_causal": PrefillConfig("tiny_causal", 1, 2, 2, 128, 64, True, 1.0, 1000),
    "prefill_mha_causal": PrefillConfig("prefill_mha_causal", 4, 16, 16, 2048, 128, True, 1.0, 2000),
    "prefill_gqa_long_causal": PrefillConfig("prefill_gqa_long_causal", 1, 32, 8, 16384, 128, True, 1.0, 3000),
    "noncausal_d64": PrefillConfig("noncausal_d64", 8, 16, 16, 4096, 64, False, 0.5, 4000),
    "paged_decode": DecodeConfig("paged_decode", 64, 12, 2, 128, 512, 8192, 16, 5000),
}


def prefill_inputs(cfg: PrefillConfig, T: int | None = None, seed: int | None = None):
    """q [B,Hq,T,D], k/v [B,Hkv,T,D] as bf16 bits (seeds s, s+1, s+2)."""
    T = cfg.T if T is None else T
    s = cfg.seed if seed is None else seed
    q = normal_bf16(s, (cfg.B, cfg.Hq, T, cfg.D), cfg.mult)
    k = normal_bf16(s + 1, (cfg.B, cfg.Hkv, T, cfg.D), cfg.mult)
    v = normal_bf16(s + 2, (cfg.B, cfg.Hkv, T, cfg.D), cfg.mult)
    return q, k, v


@dataclass
class PagedInputs:
    q: np.ndarray            # [num_seqs, Hq, D] bf16 bits
    k_pool: np.ndarray       # [num_pool_blocks, Hkv, block_size, D] bf16 bits
    v_pool: np.ndarray       # same
    block_table: np.ndarray  # [num_seqs, max_blocks_per_seq] int32, padding -1
    seq_lens: np.ndarray     # [num_seqs] int32
    block_size: int
    max_seq_len: int
    meta: dict = field(default_factory=dict)

    @property
    def num_pool_blocks(self) -> int:
        return int(self.k_pool.shape[0])

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_table.shape[1])

    def kv_bytes(self, Hkv: int, D: int) -> int:
        """Bytes of K and V the decode must read: sum_r L_r * Hkv * D * 2 B * 2."""
        return int(self.seq_lens.astype(np.int64).sum()) * Hkv * D * 2 * 2


def paged_inputs(cfg: DecodeConfig, seq_lens=None, seed: int | None = None,
                 max_seq_len: int | None = None, poison: bool = True) -> PagedInputs:
    """Paged-KV decode inputs.

    Seeds: q = s, K pool = s+1, V pool = s+2, seq_lens = s+3, pool permutation = s+4.
    Request r owns ceil(L_r/bs) blocks taken in order from one seeded permutation of
    all pool indices; the pool has ``ceil(N/spare_frac)`` spare blocks beyond the
    N that are used.  Unused blocks and the slots past L_r in each request's last
    block hold NaN (``poison``), and block-table padding is -1.
    """
    s = cfg.seed if seed is None else seed
    bs = cfg.block_size
    if seq_lens is None:
        seq_lens = uniform_ints(s + 3, cfg.num_seqs, cfg.len_lo, cfg.len_hi)
    seq_lens = np.asarray(seq_lens, dtype=np.int64)
    num_seqs = len(seq_lens)
    if max_seq_len is None:
        max_seq_len = max(int(seq_lens.max()) if num_seqs else 0, cfg.len_hi)
    max_blocks = max(1, -(-max_seq_len // bs))
    nblk = [-(-int(L) // bs) for L in seq_lens]
    used = int(sum(nblk))
    pool_n = max(1, used + -(-used // cfg.spare_frac))
    perm = permutation(s + 4, pool_n)
    table = np.full((num_seqs, max_blocks), -1, dtype=np.int32)
    pos = 0
    for r, nb in enumerate(nblk):
        table[r, :nb] = perm[pos:pos + nb]
        pos += nb
    q = normal_bf16(s, (num_seqs, cfg.Hq, cfg.D), cfg.mult)
    k_pool = normal_bf16(s + 1, (pool_n, cfg.Hkv, bs, cfg.D), cfg.mult)
    v_pool = normal_bf16(s + 2, (pool_n, cfg.Hkv, bs, cfg.D), cfg.mult)
    if poison:
        live = np.zeros((pool_n, bs), dtype=bool)
        for r, nb in enumerate(nblk):
            L = int(seq_lens[r])
            for lb in range(nb):
                n_valid = min(bs, L - lb * bs)
                live[table[r, lb], :n_valid] = True
        bi, si = np.nonzero(~live)
        k_pool[bi, :, si, :] = BF16_NAN
        v_pool[bi, :, si, :] = BF16_NAN
    return PagedInputs(q, k_pool, v_pool, table, seq_lens.astype(np.int32), bs,
                       int(max_seq_len), {"used_blocks": used, "pool_blocks": pool_n})


def identity_paged(p: PagedInputs, Hkv: int, D: int) -> PagedInputs:
    """The same logical KV laid out with an identity-like block table.

    Request r's logical block lb moves to physical block ``base_r + lb``; the
    content of each logical (token, head, dim) is unchanged.  Used to check that
    results depend only on logical positions.
    """
    bs = p.block_size
    num_seqs = len(p.seq_lens)
    nblk = [-(-int(L) // bs) for L in p.seq_lens]
    total = max(1, sum(nblk))
    k_new = np.full((total, Hkv, bs, D), BF16_NAN, dtype=np.uint16)
    v_new = np.full((total, Hkv, bs, D), BF16_NAN, dtype=np.uint16)
    table = np.full_like(p.block_table, -1)
    base = 0
    for r in range(num_seqs):
        for lb in range(nblk[r]):
            phys = p.block_table[r, lb]
            k_new[base + lb] = p.k_pool[phys]
            v_new[base + lb] = p.v_pool[phys]
            table[r, lb] = base + lb
        base += nblk[r]
    return PagedInputs(p.q.copy(), k_new, v_new, table, p.seq_lens.copy(), bs,
                       p.max_seq_len, dict(p.meta))
