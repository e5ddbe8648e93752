// attn_fwd.cu -- fused softmax attention forward for sm_103a.
//
// The method (the-ai.news, "Kernels de atencao rapida e fusao de operadores",
// section "Atencao do tipo FlashAttention e atencao paginada"): queries, keys
// and values are processed block by block; for each block a part of the scores
// is computed, the softmax statistics are updated, and the matching output is
// accumulated in on-chip memory, so the T x T score matrix never reaches HBM.
//
// GB300 realisation (one CTA per SM, persistent over 128-row query tiles):
//   warp 0      TMA producer: Q tile once per work tile, then K_j / V_j tiles
//               into a multi-stage ring (128-byte swizzled, 128 keys per tile)
//   warp 1      MMA issuer (one thread): S_j = Q K_j^T into TMEM (fp32), then
//               O += P_j V_j into TMEM (fp32); completion goes to mbarriers
//               through tcgen05.commit
//   warps 2-5   softmax: one query row per thread (TMEM lane = row); reads S_j
//               from TMEM, masks (causal diagonal, ragged tail), keeps the
//               running row max m and sum l, writes P_j = 2^(c*s - c*m) as bf16
//               into a swizzled shared tile, rescales the O row in TMEM when m
//               grew (c = scale * log2 e folds the softmax scale into exp2),
//               and finally writes O / l (bf16) and LSE = scale*m + ln l.
// Double-buffered S (TMEM) and P (shared) let the tensor core compute S_{j+1}
// while the softmax warps work on S_j.  Causal work tiles only visit KV tiles
// 0..q_tile and are scheduled heaviest first.
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace gbattn {

namespace {

constexpr int BM = 128;  // query rows per tile (= TMEM lanes)
constexpr int BN = 128;  // keys per KV tile
constexpr int kThreads = 192;

template <int D>
struct Cfg {
  static constexpr int KB = D / 64;                   // 64-column (128-byte) boxes per row
  static constexpr int BOX_BYTES = 128 * 128;         // 128 rows x 128 bytes
  static constexpr int TILE_BYTES = BM * D * 2;       // Q, K or V tile
  static constexpr int P_BYTES = BM * BN * 2;         // bf16 probabilities
  static constexpr int NS = (D == 64) ? 3 : 2;        // K and V ring depth
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + TILE_BYTES;
  static constexpr int OFF_V = OFF_K + NS * TILE_BYTES;
  static constexpr int OFF_P = OFF_V + NS * TILE_BYTES;
  static constexpr int OFF_BAR = OFF_P + 2 * P_BYTES;
  static constexpr int NBAR = 12 + 4 * NS;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;  // + slack for 1024-byte alignment
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t O_COL = 256;
};

struct Bars {
  uint32_t base;
  int ns;
  __device__ uint32_t q_full() const { return base; }
  __device__ uint32_t q_empty() const { return base + 8; }
  __device__ uint32_t k_full(int s) const { return base + 8 * (2 + s); }
  __device__ uint32_t k_empty(int s) const { return base + 8 * (2 + ns + s); }
  __device__ uint32_t v_full(int s) const { return base + 8 * (2 + 2 * ns + s); }
  __device__ uint32_t v_empty(int s) const { return base + 8 * (2 + 3 * ns + s); }
  __device__ uint32_t s_full(int b) const { return base + 8 * (2 + 4 * ns + b); }
  __device__ uint32_t s_empty(int b) const { return base + 8 * (4 + 4 * ns + b); }
  __device__ uint32_t p_full(int b) const { return base + 8 * (6 + 4 * ns + b); }
  __device__ uint32_t p_empty(int b) const { return base + 8 * (8 + 4 * ns + b); }
  __device__ uint32_t o_done() const { return base + 8 * (10 + 4 * ns); }
  __device__ uint32_t teardown() const { return base + 8 * (11 + 4 * ns); }
};

struct Tile {
  int bh;    // b * Hq + h
  int bkv;   // b * Hkv + h / group
  int qt;    // query tile index
  int nkv;   // KV tiles to visit
};

// Work tile t -> coordinates.  Causal tiles are enumerated by decreasing query
// tile (the longest rows first); within one query tile, heads of the same batch
// are adjacent so grouped heads that share K/V run at the same time.
__device__ __forceinline__ Tile tile_at(int t, const FwdParams& p) {
  const int BH = p.B * p.Hq;
  const int qi = t / BH;
  Tile tl;
  tl.bh = t - qi * BH;
  tl.qt = p.causal ? (p.n_qtiles - 1 - qi) : qi;
  const int b = tl.bh / p.Hq;
  const int h = tl.bh - b * p.Hq;
  tl.bkv = b * p.Hkv + h / p.group;
  tl.nkv = p.causal ? (tl.qt + 1) : p.n_kvtiles;
  return tl;
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

// ---------------------------------------------------------------------------
// producer: TMA loads
// ---------------------------------------------------------------------------
template <int D>
__device__ void producer(const CUtensorMap* tmQ, const CUtensorMap* tmK, const CUtensorMap* tmV,
                         const FwdParams& p, uint32_t sbase, const Bars& bar,
                         volatile int* abort) {
  using C = Cfg<D>;
  constexpr int NS = C::NS;
  const uint32_t sQ = sbase + C::OFF_Q, sK = sbase + C::OFF_K, sV = sbase + C::OFF_V;
  int kc = 0, vc = 0, tcount = 0;
  bool ok = true;
  for (int t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x, ++tcount) {
    const Tile tl = tile_at(t, p);
    if (!mbar_wait(bar.q_empty(), (tcount & 1) ^ 1, abort, p.flags)) { ok = false; break; }
    mbar_arrive_expect_tx(bar.q_full(), C::TILE_BYTES);
#pragma unroll
    for (int kb = 0; kb < C::KB; ++kb)
      tma_load_3d(sQ + kb * C::BOX_BYTES, tmQ, bar.q_full(), kb * 64, tl.qt * BM, tl.bh);
    for (int j = 0; j < tl.nkv; ++j) {
      int s = kc % NS;
      if (!mbar_wait(bar.k_empty(s), ((kc / NS) & 1) ^ 1, abort, p.flags)) { ok = false; break; }
      mbar_arrive_expect_tx(bar.k_full(s), C::TILE_BYTES);
#pragma unroll
      for (int kb = 0; kb < C::KB; ++kb)
        tma_load_3d(sK + s * C::TILE_BYTES + kb * C::BOX_BYTES, tmK, bar.k_full(s), kb * 64,
                    j * BN, tl.bkv);
      ++kc;
      s = vc % NS;
      if (!mbar_wait(bar.v_empty(s), ((vc / NS) & 1) ^ 1, abort, p.flags)) { ok = false; break; }
      mbar_arrive_expect_tx(bar.v_full(s), C::TILE_BYTES);
#pragma unroll
      for (int kb = 0; kb < C::KB; ++kb)
        tma_load_3d(sV + s * C::TILE_BYTES + kb * C::BOX_BYTES, tmV, bar.v_full(s), kb * 64,
                    j * BN, tl.bkv);
      ++vc;
    }
  }
  if (!ok) {
    // Let copies already in flight land before the CTA's shared memory goes away.
    const unsigned long long lim = 500000000ull;
    for (int n = (kc > NS ? kc - NS : 0); n < kc; ++n)
      mbar_wait_quiet(bar.k_full(n % NS), (n / NS) & 1, lim);
    for (int n = (vc > NS ? vc - NS : 0); n < vc; ++n)
      mbar_wait_quiet(bar.v_full(n % NS), (n / NS) & 1, lim);
    if (tcount > 0) mbar_wait_quiet(bar.q_full(), (tcount - 1) & 1, lim);
  }
}

// ---------------------------------------------------------------------------
// MMA issuer (single thread)
// ---------------------------------------------------------------------------
template <int D>
__device__ bool issue_pv(const FwdParams& p, int jj, uint32_t sbase, uint32_t tmem, const Bars& bar, int& vc, int& pc,
                         volatile int* abort) {
  using C = Cfg<D>;
  constexpr int NS = C::NS;
  constexpr uint32_t idesc_pv = idesc_bf16_f32(BM, D, 0, 1);  // B (= V) is MN-major
  const uint32_t sV = sbase + C::OFF_V, sP = sbase + C::OFF_P;
  const int vs = vc % NS;
  if (!mbar_wait(bar.v_full(vs), (vc / NS) & 1, abort, p.flags)) return false;
  const int pb = pc & 1;
  if (!mbar_wait(bar.p_full(pb), (pc >> 1) & 1, abort, p.flags)) return false;
  tc_fence_after();
#pragma unroll
  for (int kk = 0; kk < BN / 16; ++kk) {
    // P: K-major over keys, 16 keys = 32 bytes per step inside a 64-key box.
    const uint32_t a_addr = sP + pb * C::P_BYTES + (kk >> 2) * C::BOX_BYTES + (kk & 3) * 32;
    // V: MN-major; 16 keys = 16 rows of 128 bytes; next 64 head dims one box further.
    const uint32_t b_addr = sV + vs * C::TILE_BYTES + kk * 16 * 128;
    mma_ss(tmem + C::O_COL, smem_desc_sw128(a_addr, 16, 1024),
           smem_desc_sw128(b_addr, C::BOX_BYTES, 1024), idesc_pv, (jj > 0 || kk > 0) ? 1u : 0u);
  }
  mma_commit(bar.v_empty(vs));
  mma_commit(bar.p_empty(pb));
  mma_commit(bar.o_done());
  ++vc;
  ++pc;
  return true;
}

template <int D>
__device__ void mma_issuer(const FwdParams& p, uint32_t sbase, uint32_t tmem, const Bars& bar,
                           volatile int* abort) {
  using C = Cfg<D>;
  constexpr int NS = C::NS;
  constexpr uint32_t idesc_qk = idesc_bf16_f32(BM, BN, 0, 0);
  const uint32_t sQ = sbase + C::OFF_Q, sK = sbase + C::OFF_K;
  int kc = 0, vc = 0, sc = 0, pc = 0, tcount = 0;
  for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x, ++tcount) {
    const Tile tl = tile_at(t, p);
    if (!mbar_wait(bar.q_full(), tcount & 1, abort, p.flags)) goto done;
    for (int j = 0; j < tl.nkv; ++j) {
      const int ks = kc % NS;
      if (!mbar_wait(bar.k_full(ks), (kc / NS) & 1, abort, p.flags)) goto done;
      const int sb = sc & 1;
      if (!mbar_wait(bar.s_empty(sb), ((sc >> 1) & 1) ^ 1, abort, p.flags)) goto done;
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (kk >> 2) * C::BOX_BYTES + (kk & 3) * 32;
        mma_ss(tmem + sb * BN, smem_desc_sw128(sQ + off, 16, 1024),
               smem_desc_sw128(sK + ks * C::TILE_BYTES + off, 16, 1024), idesc_qk,
               kk > 0 ? 1u : 0u);
      }
      mma_commit(bar.s_full(sb));
      mma_commit(bar.k_empty(ks));
      if (j == tl.nkv - 1) mma_commit(bar.q_empty());
      ++kc;
      ++sc;
      if (j > 0 && !issue_pv<D>(p, j - 1, sbase, tmem, bar, vc, pc, abort)) goto done;
    }
    if (!issue_pv<D>(p, tl.nkv - 1, sbase, tmem, bar, vc, pc, abort)) goto done;
  }
done:
  // Every MMA issued by this thread has finished once this barrier flips.
  mma_commit(bar.teardown());
  mbar_wait_quiet(bar.teardown(), 0, 1000000000ull);
}

// ---------------------------------------------------------------------------
// softmax / correction / epilogue warps (128 threads, one query row each)
// ---------------------------------------------------------------------------
template <int D>
__device__ void softmax_warps(const FwdParams& p, uint32_t sbase, uint32_t tmem, const Bars& bar,
                              volatile int* abort) {
  using C = Cfg<D>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sp = warp & 3;  // TMEM sub-partition this warp may access
  const int r = sp * 32 + lane;
  const uint32_t lane_base = tmem + (static_cast<uint32_t>(sp * 32) << 16);
  const uint32_t sP = sbase + C::OFF_P;
  const float sl2 = p.scale_log2;
  int sc = 0, pc = 0, oc = 0;

  for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x) {
    const Tile tl = tile_at(t, p);
    const int qpos = tl.qt * BM + r;
    // keys visible to this row: [0, kv_end)
    const int kv_end = p.causal ? min(qpos + 1, p.T) : p.T;
    float m = -INFINITY, l = 0.f;

    for (int j = 0; j < tl.nkv; ++j) {
      const int sb = sc & 1;
      if (!mbar_wait(bar.s_full(sb), (sc >> 1) & 1, abort, p.flags)) return;
      tc_fence_after();
      uint32_t u[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(lane_base + sb * BN + 32 * c, u[c]);
      tmem_wait_ld();
#pragma unroll
      for (int c = 0; c < 4; ++c) reg_fence32(u[c]);
      tc_fence_before();
      mbar_arrive(bar.s_empty(sb));  // S_j is in registers; the buffer may be overwritten

      float s[128];
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int i = 0; i < 32; ++i) s[32 * c + i] = __uint_as_float(u[c][i]);

      if (j == tl.nkv - 1) {  // only the last visited tile can hold masked keys
        const int lim = kv_end - j * BN;
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c >= lim) s[c] = -INFINITY;
      }
      float mx0 = s[0], mx1 = s[1], mx2 = s[2], mx3 = s[3];
#pragma unroll
      for (int c = 4; c < 128; c += 4) {
        mx0 = fmaxf(mx0, s[c]);
        mx1 = fmaxf(mx1, s[c + 1]);
        mx2 = fmaxf(mx2, s[c + 2]);
        mx3 = fmaxf(mx3, s[c + 3]);
      }
      const float m_new = fmaxf(m, fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)));
      const float ms = (m_new == -INFINITY) ? 0.f : m_new * sl2;
      const float alpha = ex2(m * sl2 - ms);  // 0 on the first tile (m = -inf)

      const int pb = pc & 1;
      if (!mbar_wait(bar.p_empty(pb), ((pc >> 1) & 1) ^ 1, abort, p.flags)) return;
      float sum0 = 0.f, sum1 = 0.f;
      const uint32_t prow = sP + pb * C::P_BYTES + r * 128;
#pragma unroll
      for (int ch = 0; ch < 16; ++ch) {  // 16 chunks of 8 keys
        float e[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) e[i] = ex2(fmaf(s[ch * 8 + i], sl2, -ms));
        sum0 += (e[0] + e[1]) + (e[2] + e[3]);
        sum1 += (e[4] + e[5]) + (e[6] + e[7]);
        const uint32_t addr =
            prow + (ch >> 3) * C::BOX_BYTES + ((static_cast<uint32_t>((ch & 7) ^ (r & 7))) << 4);
        st_shared_v4(addr, pack_bf16x2(e[0], e[1]), pack_bf16x2(e[2], e[3]),
                     pack_bf16x2(e[4], e[5]), pack_bf16x2(e[6], e[7]));
      }
      fence_proxy_async_smem();  // P (generic-proxy writes) -> visible to the tensor core

      if (j > 0) {
        // O holds P_0..P_{j-1} V once PV_{j-1} is done; rescale it by alpha.
        if (!mbar_wait(bar.o_done(), oc & 1, abort, p.flags)) return;
        ++oc;
        tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(lane_base + C::O_COL + 32 * c, o);
            tmem_wait_ld();
            reg_fence32(o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st32(lane_base + C::O_COL + 32 * c, o);
          }
          tmem_wait_st();
        }
      }
      tc_fence_before();
      mbar_arrive(bar.p_full(pb));
      l = l * alpha + (sum0 + sum1);
      m = m_new;
      ++sc;
      ++pc;
    }

    // epilogue: wait for the last PV, then O / l -> bf16, LSE
    if (!mbar_wait(bar.o_done(), oc & 1, abort, p.flags)) return;
    ++oc;
    tc_fence_after();
    const float inv_l = 1.f / l;
    uint4* orow = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.o) +
                                           (static_cast<size_t>(tl.bh) * p.T + qpos) * D);
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      uint32_t o[32];
      tmem_ld32(lane_base + C::O_COL + 32 * c, o);
      tmem_wait_ld();
      reg_fence32(o);
      if (qpos < p.T) {
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          uint4 w;
          w.x = pack_bf16x2(__uint_as_float(o[8 * v + 0]) * inv_l, __uint_as_float(o[8 * v + 1]) * inv_l);
          w.y = pack_bf16x2(__uint_as_float(o[8 * v + 2]) * inv_l, __uint_as_float(o[8 * v + 3]) * inv_l);
          w.z = pack_bf16x2(__uint_as_float(o[8 * v + 4]) * inv_l, __uint_as_float(o[8 * v + 5]) * inv_l);
          w.w = pack_bf16x2(__uint_as_float(o[8 * v + 6]) * inv_l, __uint_as_float(o[8 * v + 7]) * inv_l);
          orow[c * 4 + v] = w;
        }
      }
    }
    if (p.lse != nullptr && qpos < p.T)
      p.lse[static_cast<size_t>(tl.bh) * p.T + qpos] = m * p.scale + logf(l);
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  using C = Cfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw);
  Bars bar{sbase + C::OFF_BAR, C::NS};
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(bar.q_full(), 1);
    mbar_init(bar.q_empty(), 1);
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(bar.k_full(s), 1);
      mbar_init(bar.k_empty(s), 1);
      mbar_init(bar.v_full(s), 1);
      mbar_init(bar.v_empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar.s_full(b), 1);
      mbar_init(bar.s_empty(b), 128);
      mbar_init(bar.p_full(b), 128);
      mbar_init(bar.p_empty(b), 1);
    }
    mbar_init(bar.o_done(), 1);
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

  if (warp == 0) {
    if (lane == 0) producer<D>(&tmQ, &tmK, &tmV, p, sbase, bar, abort);
  } else if (warp == 1) {
    if (lane == 0) mma_issuer<D>(p, sbase, tmem, bar, abort);
  } else {
    softmax_warps<D>(p, sbase, tmem, bar, abort);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

}  // namespace

cudaError_t prepare_attn_fwd(int D) {
  if (D == 64)
    return cudaFuncSetAttribute(attn_fwd_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                Cfg<64>::SMEM_BYTES);
  return cudaFuncSetAttribute(attn_fwd_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              Cfg<128>::SMEM_BYTES);
}

cudaError_t launch_attn_fwd(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                            const FwdParams& p, int num_sms, cudaStream_t stream) {
  const int grid = p.num_tiles < num_sms ? p.num_tiles : num_sms;
  if (grid <= 0) return cudaSuccess;
  if (p.D == 64) {
    attn_fwd_kernel<64><<<grid, kThreads, Cfg<64>::SMEM_BYTES, stream>>>(tmQ, tmK, tmV, p);
  } else {
    attn_fwd_kernel<128><<<grid, kThreads, Cfg<128>::SMEM_BYTES, stream>>>(tmQ, tmK, tmV, p);
  }
  return cudaGetLastError();
}

}  // namespace gbattn
