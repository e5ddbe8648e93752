// attn_fwd.cu -- fused softmax attention forward for sm_103a.
//
// The method (the-ai.news, "Kernels de atencao rapida e fusao de operadores",
// section "Atencao do tipo FlashAttention e atencao paginada"): queries, keys
// and values are processed block by block; for each block a part of the scores
// is computed, the softmax statistics are updated, and the matching output is
// accumulated in on-chip memory, so the Tq x Tk score matrix never reaches HBM.
// The same section describes the paged KV cache (fixed 16-token blocks, every
// logical position translated through a block table); with PAGED the key/value
// tiles are gathered block by block through that table, which is what chunked
// prefill against a paged cache needs.
//
// GB300 realisation.  One CTA per SM, persistent over work units; a unit is two
// 128-row query tiles of one (batch, head) that share every K/V tile:
//   warp 0        producer: TMA loads of the unit's two Q tiles, then K_j, V_j
//                 into one ring of 128-key slots (128-byte swizzle); in paged
//                 mode lanes 0-7 read the tile's block-table entries (the next
//                 tile's while this one is copied) and each copies its block's
//                 16 rows
//   warp 1        MMA warp (the converged warp runs the issue code; elect.sync
//                 picks the lane that issues): S_i = Q_i K_j^T into TMEM (fp32),
//                 then O_i += P_i V_j with P_i read from TMEM (tcgen05 A operand
//                 in tensor memory), in the order P_0 V_j, S_0(j+1), P_1 V_j,
//                 S_1(j+1); completion is signalled through tcgen05.commit on
//                 mbarriers
//   warps 4-7     softmax of query tile 0, warps 8-11 softmax of tile 1: one
//                 query row per thread (TMEM lane = row).  Each reads S_i from
//                 TMEM, masks, keeps the row max m and sum l, writes
//                 P = 2^(c s - c m) as bf16 back into the S_i columns (c =
//                 scale * log2 e folds the softmax scale into exp2), and at the
//                 end writes O / l (bf16) and LSE = scale m + ln l.
// The two tiles ping-pong: while the softmax warps of one tile work, the tensor
// core computes the other tile's S and P V.  The running max is only moved
// (and O rescaled in TMEM) when a row's max grows by more than 2^8 in exp2
// units, so the rescale is rare; P stays below 2^8, harmless in bf16 and fp32.
// S_i(j+1) completes after P_i(j) V_j (the MMAs of one thread execute in issue
// order), so when the softmax warps see S_i(j+1), O_i is final for tile j and
// the rescale of O_i never waits for the tensor core.
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

// With GBATTN_EXP2_POLY_PAIRS = n > 0, one key pair in every n of an unmasked
// tile has its probabilities computed on the FMA pipe (exp2_fma2) instead of
// the special-function unit.  Measured on GB300 the kernel is limited by issue
// slots and latency rather than by the special-function unit, and every setting
// tried (n = 2, 3, 4) was slower than 0, so it is off by default.
#ifndef GBATTN_EXP2_POLY_PAIRS
#define GBATTN_EXP2_POLY_PAIRS 0
#endif

namespace gbattn {

namespace {

constexpr int BM = 128;          // query rows per tile (= TMEM lanes)
constexpr int BN = 128;          // keys per K/V tile
constexpr int kBS = 16;          // tokens per paged KV block
constexpr int kThreads = 384;    // warpgroup 0: producer, MMA, 2 idle warps; 1, 2: softmax
constexpr float kRescaleLog2 = 8.f;  // move the running max only if it grows by > 2^8
// Registers per thread: the block launches with 168 (384 threads, one block per
// SM); warpgroup 0 gives some up so the softmax warpgroups, which hold a whole
// 128-key score row each, get more: 104 + 200 + 200 = 3 x 168.
constexpr int kRegsLaunch = 168, kRegsWg0 = 104, kRegsSoftmax = 200;
static_assert(kRegsWg0 + 2 * kRegsSoftmax <= 3 * kRegsLaunch, "register split exceeds the launch");

template <int D>
struct Cfg {
  static constexpr int KB = D / 64;                   // 64-column (128-byte) boxes per row
  static constexpr int BOX_BYTES = 128 * 128;         // 128 rows x 128 bytes
  static constexpr int TILE_BYTES = BM * D * 2;       // one Q, K or V tile
  static constexpr int NSLOT = (D == 64) ? 8 : 5;     // K/V ring slots
  static constexpr int OFF_Q = 0;                     // the unit's two Q tiles
  static constexpr int OFF_RING = 2 * TILE_BYTES;
  static constexpr int OFF_BAR = OFF_RING + NSLOT * TILE_BYTES;
  static constexpr int NBAR = 2 + 2 * NSLOT + 6 + 1;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;  // + slack for 1024-byte alignment
  static constexpr uint32_t TMEM_COLS = 512;
  // TMEM columns: S_0 [0,128), S_1 [128,256), O_0 and O_1 from 256 (D each).
  // P_i (bf16 pairs, 64 columns) overwrites the upper half of S_i.
  __device__ static constexpr uint32_t s_col(int i) { return 128u * i; }
  __device__ static constexpr uint32_t p_col(int i) { return 128u * i + 64u; }
  __device__ static constexpr uint32_t o_col(int i) { return 256u + static_cast<uint32_t>(D) * i; }
};
static_assert(Cfg<128>::SMEM_BYTES <= 232448, "shared memory budget");
static_assert(Cfg<64>::SMEM_BYTES <= 232448, "shared memory budget");

template <int D>
struct Bars {
  uint32_t base;
  __device__ uint32_t q_full() const { return base; }
  __device__ uint32_t q_empty() const { return base + 8; }
  __device__ uint32_t slot_full(int s) const { return base + 8 * (2 + s); }
  __device__ uint32_t slot_empty(int s) const { return base + 8 * (2 + Cfg<D>::NSLOT + s); }
  __device__ uint32_t s_full(int i) const { return base + 8 * (2 + 2 * Cfg<D>::NSLOT + i); }
  __device__ uint32_t s_free(int i) const { return base + 8 * (4 + 2 * Cfg<D>::NSLOT + i); }
  __device__ uint32_t p_full(int i) const { return base + 8 * (6 + 2 * Cfg<D>::NSLOT + i); }
  __device__ uint32_t teardown() const { return base + 8 * (8 + 2 * Cfg<D>::NSLOT); }
};

// One work unit: query rows [256 qp, 256 qp + 256) of one (batch, head).
struct Unit {
  int b, bh, kvh, bkv, qp;
  int L;     // keys of this batch item
  int n[2];  // K/V tiles query tile i visits (0: tile past Tq, or no visible key)
  int nkv;   // tiles loaded for the unit = max(n[0], n[1])
  bool bad;  // paged: the batch item's key count is outside its bounds
};

// Keys visible to query row qpos: [0, kv_end).  Causal masks align the last
// query with the last key (query i sits at logical position L - Tq + i).
__device__ __forceinline__ int kv_end_of(int qpos, int L, const FwdParams& p) {
  if (!p.causal) return L;
  const int e = qpos + 1 + (L - p.Tq);
  return e < 0 ? 0 : (e > L ? L : e);
}

// Unit u: query-pair index decreasing (the longest causal rows first); within
// one pair index, heads of a batch item are adjacent so heads that share K/V run
// at the same time.
__device__ __forceinline__ Unit unit_at(int u, const FwdParams& p, bool paged) {
  const int BH = p.B * p.Hq;
  const int qi = u / BH;
  Unit U;
  U.bh = u - qi * BH;
  U.qp = p.n_qpairs - 1 - qi;
  U.b = U.bh / p.Hq;
  const int h = U.bh - U.b * p.Hq;
  U.kvh = h / p.group;
  U.bkv = U.b * p.Hkv + U.kvh;
  U.bad = false;
  U.L = p.Tk;
  if (paged) {
    U.L = p.kv_lens[U.b];
    if (U.L < 0 || U.L > p.max_kv_len || U.L > p.max_blocks * kBS) {
      U.bad = true;
      U.L = 0;
    }
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int r0 = 256 * U.qp + 128 * i;
    if (r0 >= p.Tq) {
      U.n[i] = 0;
    } else {
      const int r1 = min(r0 + 127, p.Tq - 1);
      U.n[i] = (kv_end_of(r1, U.L, p) + BN - 1) / BN;
    }
  }
  U.nkv = max(U.n[0], U.n[1]);
  return U;
}

// Snake order over rounds of gridDim.x units: each CTA alternates between the
// heavier and the lighter end of a round, which evens out causal work.
__device__ __forceinline__ int unit_of_round(int r) {
  return r * static_cast<int>(gridDim.x) +
         ((r & 1) ? static_cast<int>(gridDim.x - 1 - blockIdx.x) : static_cast<int>(blockIdx.x));
}

__device__ __forceinline__ void reg_fence32(uint32_t (&r)[32]) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                 "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                 "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                 "+r"(r[30]), "+r"(r[31]));
}

// Keeps the compiler from using TMEM-load results before tcgen05.wait::ld.
__device__ __forceinline__ void reg_fence16(uint32_t (&r)[16]) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]));
}

// ---------------------------------------------------------------------------
// producer warp: TMA loads
// ---------------------------------------------------------------------------
template <int D, bool PAGED>
__device__ void producer_warp(const CUtensorMap* tmQ, const CUtensorMap* tmK,
                              const CUtensorMap* tmV, const FwdParams& p, uint32_t sbase,
                              const Bars<D>& bar, volatile int* abort) {
  using C = Cfg<D>;
  const int lane = threadIdx.x & 31;
  const uint32_t sQ = sbase + C::OFF_Q, sR = sbase + C::OFF_RING;
  const unsigned long long lim = p.wait_limit_ns;
  int rc = 0, uc = 0;
  bool ok = true, last_q_issued = false;
  for (int r = 0; ok && r * static_cast<int>(gridDim.x) < p.num_units; ++r) {
    const int u = unit_of_round(r);
    if (u >= p.num_units) continue;
    const Unit U = unit_at(u, p, PAGED);
    if (PAGED && U.bad && lane == 0) raise_flag(p.flags, DEVFLAG_BAD_SEQLEN);
    if (!mbar_wait_warp(bar.q_empty(), (uc & 1) ^ 1, abort, p.flags, lim)) { ok = false; break; }
    last_q_issued = !(p.withhold_copy && uc == 0);  // test hook: withhold the first Q
    if (lane == 0 && last_q_issued) {
      mbar_arrive_expect_tx(bar.q_full(), 2 * C::TILE_BYTES);
#pragma unroll
      for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int kb = 0; kb < C::KB; ++kb)
          tma_load_3d(sQ + i * C::TILE_BYTES + kb * C::BOX_BYTES, tmQ, bar.q_full(), kb * 64,
                      256 * U.qp + 128 * i, U.bh);
    }
    ++uc;
    const int nblk_total = (U.L + kBS - 1) / kBS;
    // paged: lane l < 8 reads the table entry of block l of a K/V tile; the next
    // tile's entries are requested before this tile's copies are issued, so the
    // table read is off the copy warp's path
    auto table_entry = [&](int jj) -> int {
      const int nb = min(BN / kBS, nblk_total - jj * (BN / kBS));
      return lane < nb ? p.block_table[static_cast<size_t>(U.b) * p.max_blocks + jj * (BN / kBS) + lane]
                       : 0;
    };
    int next_phys = (PAGED && U.nkv > 0) ? table_entry(0) : 0;
    for (int j = 0; j < U.nkv && ok; ++j) {
      int row_of_lane = 0, nblk = 0;
      if (PAGED) {
        nblk = min(BN / kBS, nblk_total - j * (BN / kBS));
        int phys = next_phys;
        if (j + 1 < U.nkv) next_phys = table_entry(j + 1);
        if (lane < nblk) {
          if (phys < 0 || phys >= p.num_pool_blocks) {
            raise_flag(p.flags, DEVFLAG_BAD_BLOCK);
            phys = 0;
          }
          row_of_lane = (phys * p.Hkv + U.kvh) * kBS;
        }
      }
#pragma unroll
      for (int kv = 0; kv < 2; ++kv) {
        const CUtensorMap* map = kv == 0 ? tmK : tmV;
        const int s = rc % C::NSLOT;
        if (!mbar_wait_warp(bar.slot_empty(s), ((rc / C::NSLOT) & 1) ^ 1, abort, p.flags, lim)) {
          ok = false;
          break;
        }
        const uint32_t dst = sR + s * C::TILE_BYTES;
        if (!PAGED) {
          if (lane == 0) {
            mbar_arrive_expect_tx(bar.slot_full(s), C::TILE_BYTES);
#pragma unroll
            for (int kb = 0; kb < C::KB; ++kb)
              tma_load_3d(dst + kb * C::BOX_BYTES, map, bar.slot_full(s), kb * 64, j * BN, U.bkv);
          }
        } else {
          // lane 0 posts the byte count first; then lanes 0..nblk-1 copy their
          // block's 16 rows, one box per 64-column half
          if (lane == 0) mbar_arrive_expect_tx(bar.slot_full(s), nblk * kBS * D * 2);
          __syncwarp();
          if (lane < nblk) {
#pragma unroll
            for (int kb = 0; kb < C::KB; ++kb)
              tma_load_2d(dst + kb * C::BOX_BYTES + lane * kBS * 128, map, bar.slot_full(s),
                          kb * 64, row_of_lane);
          }
          __syncwarp();
        }
        ++rc;
      }
    }
  }
  if (!ok && lane == 0) {
    // Let the copies still in flight land before the CTA's shared memory goes away.
    const unsigned long long quiet = 500000000ull;
    for (int n = (rc > C::NSLOT ? rc - C::NSLOT : 0); n < rc; ++n)
      mbar_wait_quiet(bar.slot_full(n % C::NSLOT), (n / C::NSLOT) & 1, quiet);
    if (uc > 0 && last_q_issued) mbar_wait_quiet(bar.q_full(), (uc - 1) & 1, quiet);
  }
}

// ---------------------------------------------------------------------------
// MMA warp: the whole warp runs this code, waits together and issues every
// tcgen05.mma and commit from the one lane elect.sync picks (in paged mode it
// also clears key rows past the sequence end in the last V tile).  Shared-memory
// descriptors are built once; an MMA only adds constant offsets to them.
// ---------------------------------------------------------------------------
template <int D, bool PAGED>
struct MmaWarp {
  using C = Cfg<D>;
  static constexpr uint32_t kIdescQK = idesc_bf16_f32(BM, BN, 0, 0);
  static constexpr uint32_t kIdescPV = idesc_bf16_f32(BM, D, 0, 1);  // A (P) in TMEM, V MN-major
  static constexpr uint64_t kTileStep = C::TILE_BYTES >> 4;  // descriptor address units

  const FwdParams& p;
  const Bars<D>& bar;
  volatile int* abort;
  uint32_t sR, tmem;
  uint64_t dq, dk, dv;   // descriptors of Q tile 0 and of ring slot 0 read as K and as V
  int lane;
  int base = 0;          // ring index of the unit's K_0
  int n_pv[2] = {0, 0};  // P V products issued per query tile, all units
  int s_left = 0;        // S products of the unit not yet issued
  int zeroed_j = -1;     // paged: the unit's last V tile has had its dead rows cleared

  __device__ MmaWarp(const FwdParams& p_, const Bars<D>& b_, volatile int* a_, uint32_t sbase,
                     uint32_t tmem_)
      : p(p_), bar(b_), abort(a_), sR(sbase + C::OFF_RING), tmem(tmem_),
        dq(smem_desc_sw128(sbase + C::OFF_Q, 16, 1024)),
        dk(smem_desc_sw128(sbase + C::OFF_RING, 16, 1024)),
        dv(smem_desc_sw128(sbase + C::OFF_RING, C::BOX_BYTES, 1024)),
        lane(threadIdx.x & 31) {}

  __device__ bool wait(uint32_t b, uint32_t parity) {
    return mbar_wait_warp(b, parity, abort, p.flags, p.wait_limit_ns);
  }
  __device__ int slot(int idx) const { return (base + idx) % C::NSLOT; }
  __device__ uint32_t par(int idx) const { return ((base + idx) / C::NSLOT) & 1; }

  // S_I = Q_I K_j^T.  It overwrites the TMEM columns that P_I of the previous
  // tile occupies; the P V product reading them was issued earlier by this same
  // thread, and one thread's tcgen05.mma operations execute in issue order, so
  // that product has read P_I before this one writes there.
  // Tile 1 uses the ring entries tile 0 has already waited for, whenever tile 0
  // visits the same K/V tile (j < n0); then the phase is known to be complete.
  template <int I>
  __device__ bool issue_s(int j, bool ring_seen) {
    const int ks = slot(2 * j);
    if (!ring_seen && !wait(bar.slot_full(ks), par(2 * j))) return false;
    tc_fence_after();
    const uint64_t a = dq + I * kTileStep, b = dk + static_cast<uint64_t>(ks) * kTileStep;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const uint32_t off = ((kk >> 2) * C::BOX_BYTES + (kk & 3) * 32) >> 4;
      mma_ss_warp(tmem + C::s_col(I), a + off, b + off, kIdescQK, kk > 0 ? 1u : 0u);
    }
    mma_commit_warp(bar.s_full(I));
    if (s_left == 1) mma_commit_warp(bar.q_empty());  // the unit's last read of Q
    --s_left;
    return true;
  }

  // O_I += P_I V_j (P_I from TMEM)
  template <int I>
  __device__ bool issue_pv(int j, int nkv, int L, bool ring_seen) {
    const int vs = slot(2 * j + 1);
    if (!ring_seen && !wait(bar.slot_full(vs), par(2 * j + 1))) return false;
    if (PAGED && j == nkv - 1 && zeroed_j != j) {
      zeroed_j = j;
      // Key rows past the sequence end hold stale or arbitrary data (even NaN);
      // their probabilities are 0, but 0 * NaN would reach O.  Clear those rows.
      const int row0 = max(0, L - j * BN);
      uint8_t* gv = reinterpret_cast<uint8_t*>(__cvta_shared_to_generic(sR + vs * C::TILE_BYTES));
      for (int e = row0 * 8 + lane; e < BN * 8; e += 32) {  // 8 x 16 bytes per 128-byte row
#pragma unroll
        for (int kb = 0; kb < C::KB; ++kb)
          *reinterpret_cast<uint4*>(gv + kb * C::BOX_BYTES + e * 16) = make_uint4(0, 0, 0, 0);
      }
      fence_proxy_async_smem();
      __syncwarp();
    }
    if (!wait(bar.p_full(I), n_pv[I] & 1)) return false;
    tc_fence_after();
    const uint64_t b = dv + static_cast<uint64_t>(vs) * kTileStep;
#pragma unroll
    for (int kk = 0; kk < BN / 16; ++kk)
      mma_ts_warp(tmem + C::o_col(I), tmem + C::p_col(I) + 8 * kk, b + ((kk * 16 * 128) >> 4),
                  kIdescPV, (j > 0 || kk > 0) ? 1u : 0u);
    mma_commit_warp(bar.s_free(I));
    ++n_pv[I];
    return true;
  }

  __device__ void run() {
    int uc = 0;
    for (int r = 0; r * static_cast<int>(gridDim.x) < p.num_units; ++r) {
      const int u = unit_of_round(r);
      if (u >= p.num_units) continue;
      const Unit U = unit_at(u, p, PAGED);
      if (!wait(bar.q_full(), uc & 1)) return;
      ++uc;
      const int n0 = U.n[0], n1 = U.n[1], nkv = U.nkv;
      s_left = n0 + n1;
      zeroed_j = -1;
      if (s_left == 0) mma_commit_warp(bar.q_empty());
      if (n0 > 0 && !issue_s<0>(0, false)) return;
      if (n1 > 0 && !issue_s<1>(0, n0 > 0)) return;
      if (nkv > 0) mma_commit_warp(bar.slot_empty(slot(0)));
      for (int j = 0; j < nkv; ++j) {
        if (j < n0 && !issue_pv<0>(j, nkv, U.L, false)) return;
        if (j + 1 < n0 && !issue_s<0>(j + 1, false)) return;
        if (j < n1 && !issue_pv<1>(j, nkv, U.L, j < n0)) return;
        mma_commit_warp(bar.slot_empty(slot(2 * j + 1)));
        if (j + 1 < n1 && !issue_s<1>(j + 1, j + 1 < n0)) return;
        if (j + 1 < nkv) mma_commit_warp(bar.slot_empty(slot(2 * j + 2)));
      }
      base += 2 * nkv;
    }
  }
};

// Probabilities of one row: p = 2^(c s - c m) for the 128 keys of the tile,
// summed in fp32 and written to TMEM (at p_addr) as bf16 pairs over the upper
// half of S.  Keys are handled in pairs with the packed fp32x2 instructions.
// With POLY (tiles without masked keys) one pair in GBATTN_EXP2_POLY_PAIRS uses
// the FMA-pipe exp2; masked keys (s = -inf) always go through ex2, which gives
// exactly 0 for them.
template <bool POLY>
__device__ __forceinline__ void write_p(const float (&s)[128], float sl2, float ms,
                                        uint32_t p_addr, float2 (&sum)[2]) {
  const float2 k2 = make_float2(sl2, sl2), m2 = make_float2(-ms, -ms);
  constexpr int kEvery = GBATTN_EXP2_POLY_PAIRS > 0 ? GBATTN_EXP2_POLY_PAIRS : 1;
#pragma unroll
  for (int ch = 0; ch < 8; ++ch) {  // 16 keys -> 8 packed columns per chunk
    uint32_t pk[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int c0 = 16 * ch + 2 * e;
      const float2 x = __ffma2_rn(make_float2(s[c0], s[c0 + 1]), k2, m2);
      float2 pr;
      if (POLY && GBATTN_EXP2_POLY_PAIRS > 0 && (c0 / 2) % kEvery == kEvery - 1)
        pr = exp2_fma2(x);
      else
        pr = make_float2(ex2(x.x), ex2(x.y));
      sum[e & 1] = __fadd2_rn(sum[e & 1], pr);
      pk[e] = pack_bf16x2(pr.x, pr.y);
    }
    tmem_st8(p_addr + 8 * ch, pk);
  }
}

// ---------------------------------------------------------------------------
// softmax warpgroup of query tile I (128 threads, one query row each); both
// warpgroups run this one copy of the code, which keeps the instruction cache
// footprint of the two warpgroups shared
// ---------------------------------------------------------------------------
template <int D, bool PAGED>
__device__ void softmax_wg(const FwdParams& p, uint32_t tmem, const Bars<D>& bar,
                           volatile int* abort, const int I) {
  using C = Cfg<D>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sp = warp & 3;  // TMEM sub-partition this warp may access
  const int r = sp * 32 + lane;
  const uint32_t lane_base = tmem + (static_cast<uint32_t>(sp * 32) << 16);
  const float sl2 = p.scale_log2;
  const unsigned long long lim = p.wait_limit_ns;
  int sc = 0;  // S tiles consumed (= P tiles produced), all units

  for (int rr = 0; rr * static_cast<int>(gridDim.x) < p.num_units; ++rr) {
    const int u = unit_of_round(rr);
    if (u >= p.num_units) continue;
    const Unit U = unit_at(u, p, PAGED);
    const int n = I ? U.n[1] : U.n[0];
    const int qpos = 256 * U.qp + 128 * I + r;
    const bool row_valid = qpos < p.Tq;
    const int kv_end = row_valid ? kv_end_of(qpos, U.L, p) : U.L;
    float m = -INFINITY, l = 0.f;

    for (int j = 0; j < n; ++j) {
      if (!mbar_wait_warp(bar.s_full(I), sc & 1, abort, p.flags, lim)) return;
      tc_fence_after();
      float s[128];
      {
        uint32_t u32[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(lane_base + C::s_col(I) + 32 * c, u32[c]);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 4; ++c) reg_fence32(u32[c]);
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e) s[32 * c + e] = __uint_as_float(u32[c][e]);
      }
      const int kv_lim = kv_end - j * BN;  // keys of this tile visible to the row
      const bool masked = __any_sync(0xffffffffu, kv_lim < BN);
      if (masked) {
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c >= kv_lim) s[c] = -INFINITY;
      }
      float mx0 = fmax3(s[0], s[1], s[2]), mx1 = fmax3(s[3], s[4], s[5]);
      float mx2 = fmax3(s[6], s[7], s[8]), mx3 = fmax3(s[9], s[10], s[11]);
#pragma unroll
      for (int c = 12; c < 124; c += 8) {
        mx0 = fmax3(mx0, s[c], s[c + 1]);
        mx1 = fmax3(mx1, s[c + 2], s[c + 3]);
        mx2 = fmax3(mx2, s[c + 4], s[c + 5]);
        mx3 = fmax3(mx3, s[c + 6], s[c + 7]);
      }
      mx0 = fmax3(mx0, s[124], s[125]);
      mx1 = fmax3(mx1, s[126], s[127]);
      const float m_tile = fmax3(fmaxf(mx0, mx1), mx2, mx3);
      // Move the running max only when it grows by more than 2^kRescaleLog2.
      const bool grow = (m_tile - m) * sl2 > kRescaleLog2;
      float alpha = 1.f;
      if (grow) {
        alpha = ex2((m - m_tile) * sl2);  // 0 for the first visible tile (m = -inf)
        m = m_tile;
        l *= alpha;
      }
      if (j > 0 && __any_sync(0xffffffffu, grow)) {
        // O_i already holds P_0..P_{j-1} V (S_i(j) was issued after that product
        // completed): rescale it in TMEM.
#pragma unroll 1
        for (int c = 0; c < D / 16; ++c) {
          uint32_t o[16];
          tmem_ld16(lane_base + C::o_col(I) + 16 * c, o);
          tmem_wait_ld();
          reg_fence16(o);
#pragma unroll
          for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st16(lane_base + C::o_col(I) + 16 * c, o);
        }
        tmem_wait_st();
      }
      const float ms = (m == -INFINITY) ? 0.f : m * sl2;
      float2 sum[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
      if (masked) {
        write_p<false>(s, sl2, ms, lane_base + C::p_col(I), sum);
      } else {
        write_p<true>(s, sl2, ms, lane_base + C::p_col(I), sum);
      }
      l += (sum[0].x + sum[1].x) + (sum[0].y + sum[1].y);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar.p_full(I));
      ++sc;
    }

    // epilogue: wait for the last P V, then O / l -> bf16 and LSE
    uint16_t* orow = static_cast<uint16_t*>(p.o) + (static_cast<size_t>(U.bh) * p.Tq + qpos) * D;
    const float nan = __int_as_float(0x7fc00000);
    const bool empty = !(l > 0.f);  // no visible key (or none processed)
    const float inv_l = empty ? 0.f : 1.f / l;
    if (n > 0) {
      if (!mbar_wait_warp(bar.s_free(I), (sc - 1) & 1, abort, p.flags, lim)) return;
      tc_fence_after();
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(lane_base + C::o_col(I) + 32 * c, o);
        tmem_wait_ld();
        reg_fence32(o);
        if (row_valid) {
          uint4* dst = reinterpret_cast<uint4*>(orow + 32 * c);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            float f[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) f[e] = __uint_as_float(o[8 * v + e]) * inv_l;
            if (U.bad) {
#pragma unroll
              for (int e = 0; e < 8; ++e) f[e] = nan;
            }
            dst[v] = make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]),
                                pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
          }
        }
      }
    } else if (row_valid) {
      const uint32_t w = U.bad ? pack_bf16x2(nan, nan) : 0u;
      uint4* dst = reinterpret_cast<uint4*>(orow);
#pragma unroll
      for (int v = 0; v < D / 8; ++v) dst[v] = make_uint4(w, w, w, w);
    }
    if (p.lse != nullptr && row_valid)
      p.lse[static_cast<size_t>(U.bh) * p.Tq + qpos] =
          U.bad ? nan : (empty ? -INFINITY : m * p.scale + logf(l));
  }
}

template <int D, bool PAGED>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  using C = Cfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw);
  const Bars<D> bar{sbase + C::OFF_BAR};
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(bar.q_full(), 1);
    mbar_init(bar.q_empty(), 1);
    for (int s = 0; s < C::NSLOT; ++s) {
      mbar_init(bar.slot_full(s), 1);
      mbar_init(bar.slot_empty(s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar.s_full(i), 1);
      mbar_init(bar.s_free(i), 1);
      mbar_init(bar.p_full(i), 128);
    }
    mbar_init(bar.teardown(), 1);
    *abort = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 4) {
    regs_decrease<kRegsWg0>();
    if (warp == 0) {
      producer_warp<D, PAGED>(&tmQ, &tmK, &tmV, p, sbase, bar, abort);
    } else if (warp == 1) {
      MmaWarp<D, PAGED> mma(p, bar, abort, sbase, tmem);
      mma.run();
      // Every MMA this warp issued has finished once the teardown barrier flips.
      mma_commit_warp(bar.teardown());
      if (lane == 0) mbar_wait_quiet(bar.teardown(), 0, 1000000000ull);
      __syncwarp();
    }
  } else {
    regs_increase<kRegsSoftmax>();
    softmax_wg<D, PAGED>(p, tmem, bar, abort, warp < 8 ? 0 : 1);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int D, bool PAGED>
cudaError_t set_smem() {
  return cudaFuncSetAttribute(attn_fwd_kernel<D, PAGED>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<D>::SMEM_BYTES);
}

template <int D, bool PAGED>
void launch(int grid, const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
            const FwdParams& p, cudaStream_t stream) {
  attn_fwd_kernel<D, PAGED><<<grid, kThreads, Cfg<D>::SMEM_BYTES, stream>>>(tmQ, tmK, tmV, p);
}

}  // namespace

cudaError_t prepare_attn_fwd() {
  cudaError_t e;
  if ((e = set_smem<64, false>()) != cudaSuccess) return e;
  if ((e = set_smem<128, false>()) != cudaSuccess) return e;
  if ((e = set_smem<64, true>()) != cudaSuccess) return e;
  return set_smem<128, true>();
}

cudaError_t launch_attn_fwd(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                            const FwdParams& p, int num_sms, cudaStream_t stream) {
  const int grid = p.num_units < num_sms ? p.num_units : num_sms;
  if (grid <= 0) return cudaSuccess;
  const bool paged = p.block_table != nullptr;
  if (p.D == 64) {
    if (paged) launch<64, true>(grid, tmQ, tmK, tmV, p, stream);
    else launch<64, false>(grid, tmQ, tmK, tmV, p, stream);
  } else {
    if (paged) launch<128, true>(grid, tmQ, tmK, tmV, p, stream);
    else launch<128, false>(grid, tmQ, tmK, tmV, p, stream);
  }
  return cudaGetLastError();
}

}  // namespace gbattn
