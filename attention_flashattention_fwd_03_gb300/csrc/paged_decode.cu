// paged_decode.cu -- single-token attention against a paged KV cache, sm_103a.
//
// The method (the-ai.news, "Kernels de atencao rapida e fusao de operadores",
// section "Atencao do tipo FlashAttention e atencao paginada"): the KV cache is
// stored in fixed-size blocks (16 tokens in the page's vLLM example) and a block
// table maps each request's logical positions to physical blocks; the attention
// kernel translates every position through that table.
//
// GB300 realisation (HBM-bound: every K/V byte is read exactly once):
//   split kernel   one CTA per (request, KV head, 512-token chunk), three
//                  resident per SM, chunks ordered chunk-index first so that the
//                  CTAs of chunks past a request's end come last.  A producer
//                  warp reads the chunk's (at most 32) block-table entries once,
//                  then TMA-gathers each (physical block, KV head) slice -- 16
//                  contiguous rows of D bf16 -- for K and V into an 8-stage,
//                  128-byte-swizzled shared ring.  Four consumer warps take
//                  every fourth block: the GQA group's queries (rows of a
//                  16 x D tile) meet the block's keys with warp-level bf16 MMAs,
//                  the online softmax runs on the score fragments in registers
//                  (exp2 with the scale folded in), and P.V accumulates in fp32
//                  fragments.  The four warps' states are merged through shared
//                  memory and the chunk's normalised O_s and LSE_s go to the
//                  workspace.
//   merge kernel   one warp per (request, query head): LSE = M + ln sum_s
//                  e^{LSE_s - M}, O = sum_s e^{LSE_s - LSE} O_s, in split order.
//                  It is launched as a programmatic dependent of the split
//                  kernel, so its launch overlaps the split kernel's tail.
// The reduction order depends only on logical positions (fixed chunk length,
// fixed block-to-warp assignment), so any placement of the blocks in the pool
// gives bit-identical results.
#include <cuda_runtime.h>

#include "internal.h"
#include "paged.cuh"
#include "ptx.cuh"

namespace gbattn {

namespace {

constexpr int kBS = kPagedBlock;  // tokens per KV block
constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
#ifndef GBATTN_DEC_STAGES
#define GBATTN_DEC_STAGES 8
#endif
#ifndef GBATTN_DEC_CTAS_PER_SM
#define GBATTN_DEC_CTAS_PER_SM 3
#endif
constexpr int kStages = GBATTN_DEC_STAGES;          // 8 KiB K+V stages per CTA
constexpr int kCtasPerSm = GBATTN_DEC_CTAS_PER_SM;  // 3 x 66 KB of shared memory, <= 136 registers
// Block i goes to stage i % kStages and to consumer warp i % kConsumerWarps.  A
// stage must always come back to the same warp: that warp then sees every phase
// of the stage's barrier in order.  If two warps shared a stage across phases, a
// warp could wait on a phase two behind (copies may land out of order), pass the
// parity test early, read a stage that is still being written and break the
// barrier's arrival and transaction counts.
static_assert(kStages % kConsumerWarps == 0, "every stage must belong to one consumer warp");
constexpr int kBlocksPerChunk = kDecodeChunk / kBS;  // 32

template <int D>
struct DecCfg {
  static constexpr int KB = D / 64;
  static constexpr int BOX_BYTES = kBS * 128;          // 16 rows x 128 bytes
  static constexpr int BLK_BYTES = kBS * D * 2;        // one (block, head) slice of K or V
  static constexpr int STAGE_BYTES = 2 * BLK_BYTES;    // K then V
  static constexpr int OFF_BAR = kStages * STAGE_BYTES;
  static constexpr int OFF_TABLE = OFF_BAR + 2 * kStages * 8;
  static constexpr int OFF_MISC = OFF_TABLE + kBlocksPerChunk * 4;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
  // after the main loop the stage area holds the cross-warp merge scratch
  static constexpr int RED_ACC_BYTES = kConsumerWarps * 16 * D * 4;
  static_assert(RED_ACC_BYTES + kConsumerWarps * 16 * 8 <= kStages * STAGE_BYTES, "scratch");
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}

// D = A * B + D, m16n8k16, bf16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Address of the 16-byte chunk holding (row, dims col..col+7) of a 16-row slice
// stored as 64-column boxes with the 128-byte swizzle TMA applies.
__device__ __forceinline__ uint32_t swz(uint32_t base, int row, int col) {
  const int box = col >> 6;
  const int chunk = (col & 63) >> 3;
  return base + box * (kBS * 128) + row * 128 + ((chunk ^ (row & 7)) << 4);
}

template <int D>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
    paged_decode_split_kernel(const __grid_constant__ CUtensorMap tmK,
                              const __grid_constant__ CUtensorMap tmV, const DecodeParams p) {
  using C = DecCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw);
  const uint32_t bar_full = sbase + C::OFF_BAR;
  const uint32_t bar_empty = bar_full + 8 * kStages;
  int32_t* table = reinterpret_cast<int32_t*>(smem + C::OFF_TABLE);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + C::OFF_MISC);
  volatile int* bad = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  // the merge kernel may be scheduled now; it waits for this grid's results
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_rk = p.S * p.Hkv;
  const int split = blockIdx.x / n_rk;  // chunk index first: empty chunks come last
  const int rk = blockIdx.x - split * n_rk;
  const int kvh = rk % p.Hkv;
  const int r = rk / p.Hkv;
  const int L = p.seq_lens[r];
  if (L < 0 || L > p.max_seq_len || L > p.max_blocks * kBS) return;  // merge kernel reports it
  const int c0 = split * kDecodeChunk;
  if (c0 >= L) return;  // this request has fewer splits
  const int n_tok = min(kDecodeChunk, L - c0);
  const int nblk = (n_tok + kBS - 1) / kBS;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    *abort = 0;
    *bad = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ---------------- producer warp ----------------
    for (int b = lane; b < nblk; b += 32) {
      int row = paged_block_row(p.block_table, p.max_blocks, r, c0 / kBS + b, kvh, p.Hkv,
                                p.num_pool_blocks);
      if (row < 0) {
        raise_flag(p.flags, DEVFLAG_BAD_BLOCK);
        *bad = 1;
        row = kvh * kBS;  // read block 0 instead; the chunk is reported as NaN
      }
      table[b] = row;
    }
    __syncwarp();
    if (lane == 0) {
      int issued = 0;
      for (int i = 0; i < nblk; ++i) {
        const int s = i % kStages;
        if (!mbar_wait(bar_empty + 8 * s, ((i / kStages) & 1) ^ 1, abort, p.flags,
                       p.wait_limit_ns))
          break;
        const uint32_t dst = sbase + s * C::STAGE_BYTES;
        const int row = table[i];
        if (p.withhold_copy && i == 0) {  // test hook: the first block never arrives
          ++issued;
          continue;
        }
        mbar_arrive_expect_tx(bar_full + 8 * s, C::STAGE_BYTES);
#pragma unroll
        for (int kb = 0; kb < C::KB; ++kb) {
          tma_load_2d(dst + kb * C::BOX_BYTES, &tmK, bar_full + 8 * s, kb * 64, row);
          tma_load_2d(dst + C::BLK_BYTES + kb * C::BOX_BYTES, &tmV, bar_full + 8 * s, kb * 64, row);
        }
        ++issued;
      }
      if (issued < nblk) {  // aborted: let copies in flight land
        for (int i = (issued > kStages ? issued - kStages : 0); i < issued; ++i)
          if (!(p.withhold_copy && i == 0))
            mbar_wait_quiet(bar_full + 8 * (i % kStages), (i / kStages) & 1, 500000000ull);
      }
    }
    __syncthreads();  // pairs with the consumers' merge barrier below
    return;
  }

  // ---------------- consumer warps ----------------
  const int g = lane >> 2, t4 = lane & 3;
  const int group = p.group;
  const float sl2 = p.scale_log2;

  // Q fragments (A operand, rows = the group's query heads, zero past the group)
  uint32_t qa[D / 16][4];
  {
    const uint16_t* qbase =
        static_cast<const uint16_t*>(p.q) + (static_cast<size_t>(r) * p.Hq + kvh * group) * D;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {      // row g, row g + 8
        const int row = g + 8 * h;
#pragma unroll
        for (int c = 0; c < 2; ++c) {    // cols 2t4.., 2t4+8..
          const int col = kk * 16 + 2 * t4 + 8 * c;
          uint32_t v = 0;
          if (row < group) v = *reinterpret_cast<const uint32_t*>(qbase + row * D + col);
          qa[kk][h + 2 * c] = v;
        }
      }
    }
  }

  float m_lo = -INFINITY, m_hi = -INFINITY, l_lo = 0.f, l_hi = 0.f;
  float acc[D / 8][4];
#pragma unroll
  for (int n = 0; n < D / 8; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;

  for (int i = warp; i < nblk; i += kConsumerWarps) {
    const int s = i % kStages;
    if (!mbar_wait_warp(bar_full + 8 * s, (i / kStages) & 1, abort, p.flags, p.wait_limit_ns))
      break;
    const uint32_t kbase = sbase + s * C::STAGE_BYTES;
    const uint32_t vbase = kbase + C::BLK_BYTES;
    const int n_valid = min(kBS, n_tok - i * kBS);
    if (n_valid < kBS) {
      // Slots past the sequence end may hold anything (even NaN); 0 * NaN would
      // leak into O, so clear those V rows.
      for (int e = lane; e < (kBS - n_valid) * (D / 8); e += 32) {
        const int row = n_valid + e / (D / 8);
        const int col = (e % (D / 8)) * 8;
        st_shared_v4(swz(vbase, row, col), 0u, 0u, 0u, 0u);
      }
      __syncwarp();
    }

    // S = Q K^T for 16 tokens (two n-tiles of 8)
    float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    {
      const int mat = lane >> 3, rr = lane & 7;
      const int tok = (mat >> 1) * 8 + rr;
      const int dof = (mat & 1) * 8;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        uint32_t b00, b01, b10, b11;
        ldsm_x4(swz(kbase, tok, kk * 16 + dof), b00, b01, b10, b11);
        mma_bf16_16816(sc[0], qa[kk], b00, b01);
        mma_bf16_16816(sc[1], qa[kk], b10, b11);
      }
    }
    // mask tokens past the end (select, so NaN keys in dead slots cannot leak)
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const int tok = nt * 8 + 2 * t4;
      if (tok >= n_valid) { sc[nt][0] = -INFINITY; sc[nt][2] = -INFINITY; }
      if (tok + 1 >= n_valid) { sc[nt][1] = -INFINITY; sc[nt][3] = -INFINITY; }
    }
    float bm_lo = fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1]));
    float bm_hi = fmaxf(fmaxf(sc[0][2], sc[0][3]), fmaxf(sc[1][2], sc[1][3]));
    bm_lo = fmaxf(bm_lo, __shfl_xor_sync(0xffffffffu, bm_lo, 1));
    bm_lo = fmaxf(bm_lo, __shfl_xor_sync(0xffffffffu, bm_lo, 2));
    bm_hi = fmaxf(bm_hi, __shfl_xor_sync(0xffffffffu, bm_hi, 1));
    bm_hi = fmaxf(bm_hi, __shfl_xor_sync(0xffffffffu, bm_hi, 2));
    const float mn_lo = fmaxf(m_lo, bm_lo), mn_hi = fmaxf(m_hi, bm_hi);
    // every block has at least one valid token, so mn_* is finite
    const float ms_lo = mn_lo * sl2, ms_hi = mn_hi * sl2;
    const float al_lo = ex2(m_lo * sl2 - ms_lo), al_hi = ex2(m_hi * sl2 - ms_hi);
    float pr[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      pr[nt][0] = ex2(fmaf(sc[nt][0], sl2, -ms_lo));
      pr[nt][1] = ex2(fmaf(sc[nt][1], sl2, -ms_lo));
      pr[nt][2] = ex2(fmaf(sc[nt][2], sl2, -ms_hi));
      pr[nt][3] = ex2(fmaf(sc[nt][3], sl2, -ms_hi));
    }
    l_lo = l_lo * al_lo + ((pr[0][0] + pr[0][1]) + (pr[1][0] + pr[1][1]));
    l_hi = l_hi * al_hi + ((pr[0][2] + pr[0][3]) + (pr[1][2] + pr[1][3]));
    m_lo = mn_lo;
    m_hi = mn_hi;
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
      acc[n][0] *= al_lo;
      acc[n][1] *= al_lo;
      acc[n][2] *= al_hi;
      acc[n][3] *= al_hi;
    }
    // P as the A operand (k = the 16 tokens)
    uint32_t pa[4];
    pa[0] = pack_bf16x2(pr[0][0], pr[0][1]);
    pa[1] = pack_bf16x2(pr[0][2], pr[0][3]);
    pa[2] = pack_bf16x2(pr[1][0], pr[1][1]);
    pa[3] = pack_bf16x2(pr[1][2], pr[1][3]);
    {
      const int mat = lane >> 3, rr = lane & 7;
      const int tok = (mat & 1) * 8 + rr;
      const int dof = (mat >> 1) * 8;
#pragma unroll
      for (int j = 0; j < D / 16; ++j) {
        uint32_t b00, b01, b10, b11;
        ldsm_x4_t(swz(vbase, tok, j * 16 + dof), b00, b01, b10, b11);
        mma_bf16_16816(acc[2 * j], pa, b00, b01);
        mma_bf16_16816(acc[2 * j + 1], pa, b10, b11);
      }
    }
    __syncwarp();
    if (n_valid < kBS) fence_proxy_async_smem();  // our generic writes before TMA reuses the stage
    if (lane == 0) mbar_arrive(bar_empty + 8 * s);
  }

  // quad-reduce the row sums (each lane summed its own columns)
  l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 1);
  l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 2);
  l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 1);
  l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 2);

  __syncthreads();  // all warps (producer included) are done with the ring

  // cross-warp merge through the (now idle) stage area
  float* red_acc = reinterpret_cast<float*>(smem);                      // [warp][16][D]
  float* red_ml = reinterpret_cast<float*>(smem + C::RED_ACC_BYTES);    // [warp][16][2]
#pragma unroll
  for (int n = 0; n < D / 8; ++n) {
    const int col = n * 8 + 2 * t4;
    red_acc[(warp * 16 + g) * D + col] = acc[n][0];
    red_acc[(warp * 16 + g) * D + col + 1] = acc[n][1];
    red_acc[(warp * 16 + g + 8) * D + col] = acc[n][2];
    red_acc[(warp * 16 + g + 8) * D + col + 1] = acc[n][3];
  }
  if (t4 == 0) {
    red_ml[(warp * 16 + g) * 2] = m_lo;
    red_ml[(warp * 16 + g) * 2 + 1] = l_lo;
    red_ml[(warp * 16 + g + 8) * 2] = m_hi;
    red_ml[(warp * 16 + g + 8) * 2 + 1] = l_hi;
  }
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");

  const bool is_bad = *bad != 0 || *abort != 0;
  for (int idx = threadIdx.x; idx < group * D; idx += kConsumerWarps * 32) {
    const int row = idx / D, d = idx - row * D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, red_ml[(w * 16 + row) * 2]);
    float lsum = 0.f, o = 0.f;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) {
      const float mw = red_ml[(w * 16 + row) * 2];
      const float f = (mw == -INFINITY) ? 0.f : ex2((mw - M) * sl2);
      lsum += red_ml[(w * 16 + row) * 2 + 1] * f;
      o += red_acc[(w * 16 + row) * D + d] * f;
    }
    const size_t hq = static_cast<size_t>(r) * p.Hq + kvh * group + row;
    float out = o / lsum;
    float lse = M * p.scale + logf(lsum);
    if (is_bad) out = lse = __int_as_float(0x7fc00000);
    p.part_o[(hq * p.max_splits + split) * D + d] = out;
    if (d == 0) p.part_lse[hq * p.max_splits + split] = lse;
  }
}

// One warp per (request, query head).
template <int D>
__global__ void __launch_bounds__(128)
    paged_decode_merge_kernel(const DecodeParams p) {
  // launched as a programmatic dependent: the split kernel's results are complete
  // and visible once this returns
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int warp_global = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp_global >= p.S * p.Hq) return;
  const int r = warp_global / p.Hq;
  const size_t hq = warp_global;
  const int L = p.seq_lens[r];
  constexpr int PER = D / 32;  // dims per lane
  uint16_t* orow = static_cast<uint16_t*>(p.o) + hq * D + lane * PER;
  float res[PER];
  float lse_out;
  if (L < 0 || L > p.max_seq_len || L > p.max_blocks * kBS) {
    if (lane == 0) raise_flag(p.flags, DEVFLAG_BAD_SEQLEN);
#pragma unroll
    for (int i = 0; i < PER; ++i) res[i] = __int_as_float(0x7fc00000);
    lse_out = __int_as_float(0x7fc00000);
  } else if (L == 0) {
#pragma unroll
    for (int i = 0; i < PER; ++i) res[i] = 0.f;
    lse_out = -INFINITY;
  } else {
    // The LSE of split `lane` and the partial outputs of the first 16 splits are
    // loaded together, so the merge costs one memory round trip after the
    // length; longer sequences (> 16 splits) read the rest in a second pass.
    constexpr int kHeld = 16;
    const int ns = (L + kDecodeChunk - 1) / kDecodeChunk;
    const float* pl = p.part_lse + hq * p.max_splits;
    const float* po = p.part_o + hq * p.max_splits * D + lane * PER;
    const float lse_lane = (lane < ns) ? pl[lane] : -INFINITY;
    float part[kHeld][PER];
#pragma unroll
    for (int s = 0; s < kHeld; ++s)
#pragma unroll
      for (int q = 0; q < PER; ++q) part[s][q] = (s < ns) ? po[static_cast<size_t>(s) * D + q] : 0.f;
    float M = lse_lane;
    bool nan = (lse_lane != lse_lane);
    for (int s0 = 32; s0 < ns; s0 += 32) {
      const float v = (s0 + lane < ns) ? pl[s0 + lane] : -INFINITY;
      nan |= (v != v);
      M = fmaxf(M, v);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    nan = __any_sync(0xffffffffu, nan);
    // weights and sums in split order
    float tot = 0.f;
#pragma unroll
    for (int i = 0; i < PER; ++i) res[i] = 0.f;
    const float w_first = (lane < ns) ? __expf(lse_lane - M) : 0.f;
#pragma unroll
    for (int s = 0; s < kHeld; ++s) {
      const float w = __shfl_sync(0xffffffffu, w_first, s);  // 0 past ns
      tot += w;
#pragma unroll
      for (int i = 0; i < PER; ++i) res[i] += w * part[s][i];
    }
    for (int s0 = 0; s0 < ns; s0 += 32) {
      const float w_lane =
          (s0 + lane < ns) ? (s0 == 0 ? w_first : __expf(pl[s0 + lane] - M)) : 0.f;
      for (int s = max(kHeld - s0, 0); s < min(32, ns - s0); ++s) {
        const float w = __shfl_sync(0xffffffffu, w_lane, s);
        tot += w;
        const float* src = po + static_cast<size_t>(s0 + s) * D;
#pragma unroll
        for (int i = 0; i < PER; ++i) res[i] += w * src[i];
      }
    }
    const float inv = 1.f / tot;
#pragma unroll
    for (int i = 0; i < PER; ++i) res[i] *= inv;
    lse_out = M + logf(tot);
    if (nan) {
#pragma unroll
      for (int i = 0; i < PER; ++i) res[i] = __int_as_float(0x7fc00000);
      lse_out = __int_as_float(0x7fc00000);
    }
  }
#pragma unroll
  for (int i = 0; i < PER; i += 2) {
    *reinterpret_cast<uint32_t*>(orow + i) = pack_bf16x2(res[i], res[i + 1]);
  }
  if (p.lse != nullptr && lane == 0) p.lse[hq] = lse_out;
}

}  // namespace

size_t decode_workspace_bytes(int S, int Hq, int D, int max_seq_len) {
  const size_t splits = static_cast<size_t>((max_seq_len + kDecodeChunk - 1) / kDecodeChunk);
  const size_t n = static_cast<size_t>(S) * Hq * (splits > 0 ? splits : 1);
  size_t bytes = n * D * sizeof(float);
  bytes = (bytes + 255) & ~static_cast<size_t>(255);
  bytes += n * sizeof(float);
  return (bytes + 255) & ~static_cast<size_t>(255);
}

cudaError_t prepare_paged_decode() {
  cudaError_t e = cudaFuncSetAttribute(paged_decode_split_kernel<64>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       DecCfg<64>::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(paged_decode_split_kernel<128>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, DecCfg<128>::SMEM_BYTES);
}

namespace {

template <int D>
cudaError_t launch_pair(const CUtensorMap& tmK, const CUtensorMap& tmV, const DecodeParams& p,
                        cudaStream_t stream) {
  const int grid = p.S * p.Hkv * p.max_splits;
  paged_decode_split_kernel<D><<<grid, kThreads, DecCfg<D>::SMEM_BYTES, stream>>>(tmK, tmV, p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((p.S * p.Hq + 3) / 4);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, paged_decode_merge_kernel<D>, p);
}

}  // namespace

cudaError_t launch_paged_decode(const CUtensorMap& tmK, const CUtensorMap& tmV,
                                const DecodeParams& p, int num_sms, cudaStream_t stream) {
  (void)num_sms;
  if (p.S <= 0) return cudaSuccess;
  return p.D == 64 ? launch_pair<64>(tmK, tmV, p, stream) : launch_pair<128>(tmK, tmV, p, stream);
}

}  // namespace gbattn
