// paged_decode.cu -- single-token attention against a paged KV cache, sm_103a.
//
// The method (the-ai.news, "Kernels de atencao rapida e fusao de operadores",
// section "Atencao do tipo FlashAttention e atencao paginada"): the KV cache is
// stored in fixed-size blocks (16 tokens in the page's vLLM example) and a block
// table maps each request's logical positions to physical blocks; the attention
// kernel translates every position through that table.
//
// GB300 realisation (HBM-bound: every K/V byte is read exactly once):
//   split kernel   persistent, two CTAs per SM, four consumer warps each.  All
//                  (request, KV head, 16-token block) triples form one sequence,
//                  request-major; it is cut into W equal contiguous ranges, one
//                  per consumer warp (W = min(4 x grid, blocks / 16)), so every
//                  warp streams the same number of blocks and no CTA waits on a
//                  tail.  A range may cross from one (request, KV head) segment
//                  into the next; a warp ends a "piece" there and writes that
//                  piece's normalised O and LSE.  A producer warp walks the four
//                  ranges, translates each block through the block table (one
//                  batch of 32 table reads in flight while the previous batch is
//                  issued) and TMA-gathers the (physical block, KV head) slice --
//                  16 contiguous rows of D bf16 -- of K and V into an 8-stage,
//                  128-byte-swizzled shared ring.  A consumer warp meets the
//                  GQA group's queries (rows of a 16 x D tile) with the block's
//                  keys through warp-level bf16 MMAs, runs the online softmax on
//                  the score fragments in registers (exp2 with the scale folded
//                  in) and accumulates P.V in fp32 fragments.
//   merge kernel   one warp per (request, query head): LSE = M + ln sum_j
//                  e^{LSE_j - M}, O = sum_j e^{LSE_j - LSE} O_j over the pieces
//                  of the request's segment, in piece order, 32 pieces per
//                  memory round trip.  It is launched as
//                  a programmatic dependent of the split kernel, so its launch
//                  overlaps the split kernel's end.
// The ranges depend only on the sequence lengths of the batch, never on where the
// blocks sit in the pool, so any placement gives bit-identical results.
#include <cuda_runtime.h>

#include "internal.h"
#include "paged.cuh"
#include "ptx.cuh"

namespace gbattn {

namespace {

constexpr int kBS = kPagedBlock;  // tokens per KV block
constexpr int kMinBlocks = kDecodeMinRange / kBS;  // shortest warp range, in blocks
constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
// Ring depth and CTAs per SM, by query tiles (NQT = 1: groups of up to 8 query
// heads, 2: up to 16).  Measured on the 64-request workload (group 6), the split
// kernel ran fastest with about 96-128 KiB of copies in flight per SM: 4 stages x
// 3 CTAs 63.5 us, 8 x 2 65.5 us, 8 x 3 71.6 us (192 KiB in flight shared the
// memory system less evenly between SMs), 16 x 1 106 us (too few consumer warps).
// Two query tiles need more registers than three CTAs per SM leave, so they run
// 8 stages x 2 CTAs.
template <int NQT>
struct DecShape {
  static constexpr int kStages = NQT == 1 ? 4 : 8;  // 8 KiB (D = 128) K+V stages per CTA
  static constexpr int kCtasPerSm = NQT == 1 ? 3 : 2;
  // Block i goes to stage i % kStages and to consumer warp i % kConsumerWarps.  A
  // stage must always come back to the same warp: that warp then sees every phase
  // of the stage's barrier in order.  If two warps shared a stage across phases, a
  // warp could wait on a phase two behind (copies may land out of order), pass the
  // parity test early, read a stage that is still being written and break the
  // barrier's arrival and transaction counts.
  static_assert(kStages % kConsumerWarps == 0, "every stage must belong to one consumer warp");
};
static_assert(kConsumerWarps == 4, "the producer batches 8 rounds of 4 ranges per 32 lanes");

// Start of one consumer warp's range, found by the producer warp's plan.
struct RangeStart {
  long long first;  // global index of block 0 of the (request, KV head) segment
  int r, h, b;      // request, KV head, block of that head where the range starts
  int nb;           // blocks per KV head of request r
  int n;            // blocks in the range (0: no range)
  int pad;
};

template <int D, int kStages>
struct DecCfg {
  static constexpr int KB = D / 64;
  static constexpr int BOX_BYTES = kBS * 128;          // 16 rows x 128 bytes
  static constexpr int BLK_BYTES = kBS * D * 2;        // one (block, head) slice of K or V
  static constexpr int STAGE_BYTES = 2 * BLK_BYTES;    // K then V
  static constexpr int OFF_BAR = kStages * STAGE_BYTES;
  static constexpr int OFF_STAGE_BAD = OFF_BAR + 2 * kStages * 8;   // int per stage
  static constexpr int OFF_ROWS = OFF_STAGE_BAD + kStages * 4;      // producer batch: 32 rows
  static constexpr int OFF_RBAD = OFF_ROWS + 32 * 4;                // and 32 bad-block marks
  static constexpr int OFF_START = OFF_RBAD + 32 * 4;               // RangeStart per warp
  static constexpr int OFF_PLAN = OFF_START + kConsumerWarps * 32;  // NB (8 bytes), W
  static constexpr int OFF_MISC = OFF_PLAN + 16;                    // abort word
  // per consumer warp: P as [query][token] bf16, 16 x 16, the B operand of O^T += V^T P^T
  static constexpr int OFF_PS = (OFF_MISC + 16 + 127) & ~127;
  static constexpr int PS_WARP_BYTES = 16 * 16 * 2;
  static constexpr int SMEM_BYTES = OFF_PS + kConsumerWarps * PS_WARP_BYTES + 1024;
};
static_assert(sizeof(RangeStart) == 32, "RangeStart layout");

// Blocks per KV head of a request of L tokens; 0 for a length outside its bounds
// (the merge kernel reports that request).
__device__ __forceinline__ int blocks_of(const DecodeParams& p, int L) {
  return (L < 0 || L > p.max_seq_len || L > p.max_blocks * kBS) ? 0 : (L + kBS - 1) / kBS;
}

// The warp range holding block b of the global order: ranges are
// [floor(k NB / W), floor((k + 1) NB / W)), so this is the largest k whose range
// starts at or before b.
__device__ __forceinline__ int range_of(long long b, long long NB, int W) {
  return static_cast<int>(((b + 1) * W - 1) / NB);
}

// A position in the global (request, KV head, block) order.
struct Cursor {
  long long first;  // global index of block 0 of segment (r, h)
  int r, h, b, nb;
};

// Moves c forward by k blocks.  The caller guarantees the target lies inside the
// order; should the lengths say otherwise, r stops at S and the caller's checks
// see it.
__device__ __forceinline__ void advance(Cursor& c, int k, const DecodeParams& p) {
  c.b += k;
  while (c.b >= c.nb && c.r < p.S) {
    c.b -= c.nb;
    c.first += c.nb;
    if (++c.h == p.Hkv) {
      c.h = 0;
      c.nb = 0;
      while (c.nb == 0 && ++c.r < p.S) c.nb = blocks_of(p, p.seq_lens[c.r]);
    }
  }
}

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

// Q^T fragments of request r, KV head h: the B operand (k = 16 dims, n = 8
// queries) of S^T = K Q^T for every 16-dim step, per 8-query tile; queries past
// the group are zero.
template <int D, int NQT>
__device__ __forceinline__ void load_q(const DecodeParams& p, int r, int h, int g, int t4,
                                       uint32_t (&qb)[D / 16][NQT][2]) {
  const uint16_t* qbase =
      static_cast<const uint16_t*>(p.q) + (static_cast<size_t>(r) * p.Hq + h * p.group) * D;
#pragma unroll
  for (int nt = 0; nt < NQT; ++nt) {
    const int row = 8 * nt + g;  // query
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
      for (int c = 0; c < 2; ++c) {  // dims 2t4.., 2t4+8..
        uint32_t v = 0;
        if (row < p.group)
          v = *reinterpret_cast<const uint32_t*>(qbase + row * D + kk * 16 + 2 * t4 + 8 * c);
        qb[kk][nt][c] = v;
      }
    }
  }
}

__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];"
               : "=r"(r0), "=r"(r1)
               : "r"(addr)
               : "memory");
}

__device__ __forceinline__ void st_shared_u16(uint32_t addr, uint16_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

template <int D, int NQT>
__global__ void __launch_bounds__(kThreads, DecShape<NQT>::kCtasPerSm)
    paged_decode_split_kernel(const __grid_constant__ CUtensorMap tmK,
                              const __grid_constant__ CUtensorMap tmV, const DecodeParams p) {
  constexpr int kStages = DecShape<NQT>::kStages;
  using C = DecCfg<D, kStages>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw);
  const uint32_t bar_full = sbase + C::OFF_BAR;
  const uint32_t bar_empty = bar_full + 8 * kStages;
  volatile int* stage_bad = reinterpret_cast<volatile int*>(smem + C::OFF_STAGE_BAD);
  volatile int* rows = reinterpret_cast<volatile int*>(smem + C::OFF_ROWS);
  volatile int* rbad = reinterpret_cast<volatile int*>(smem + C::OFF_RBAD);
  RangeStart* start = reinterpret_cast<RangeStart*>(smem + C::OFF_START);
  long long* plan_nb = reinterpret_cast<long long*>(smem + C::OFF_PLAN);
  int* plan_w = reinterpret_cast<int*>(smem + C::OFF_PLAN + 8);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + C::OFF_MISC);

  // the merge kernel may be scheduled now; it waits for this grid's results
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    *abort = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  // Launched as a programmatic dependent of whatever precedes it on the stream
  // (the KV append of a decode step triggers early): everything up to here
  // overlaps that kernel; its writes are complete and visible past this point.
  asm volatile("griddepcontrol.wait;" ::: "memory");

  if (warp == kConsumerWarps) {
    // ---------------- plan: total blocks, range count, this CTA's four ranges ----------------
    long long nbr = 0;
    for (int r0 = 0; r0 < p.S; r0 += 32)
      if (r0 + lane < p.S) nbr += blocks_of(p, p.seq_lens[r0 + lane]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) nbr += __shfl_xor_sync(0xffffffffu, nbr, o);
    const long long NB = nbr * p.Hkv;
    const long long w_cap = static_cast<long long>(gridDim.x) * kConsumerWarps;
    const int W = NB == 0 ? 0 : static_cast<int>(max(1ll, min(w_cap, NB / kMinBlocks)));
    // lane w < 4: the range of consumer warp w
    const long long k = static_cast<long long>(blockIdx.x) * kConsumerWarps + (lane & 3);
    const long long lo = k < W ? k * NB / W : NB;
    const long long hi = k < W ? (k + 1) * NB / W : NB;
    if (lane < kConsumerWarps) {
      start[lane].n = static_cast<int>(hi - lo);
      start[lane].first = 0;
      start[lane].r = start[lane].h = start[lane].b = 0;
      start[lane].nb = 1;
    }
    // locate each range's first block: scan the requests 32 at a time
    long long before = 0;  // blocks of requests r0 - 1 and earlier
    unsigned pending = __ballot_sync(0xffffffffu, lane < kConsumerWarps && hi > lo) & 0xFu;
    for (int r0 = 0; r0 < p.S && pending; r0 += 32) {
      const int r = r0 + lane;
      const int nbl = r < p.S ? blocks_of(p, p.seq_lens[r]) : 0;
      long long incl = static_cast<long long>(nbl) * p.Hkv;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const long long v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      incl += before;
      const long long excl = incl - static_cast<long long>(nbl) * p.Hkv;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) {
        if (!(pending >> w & 1u)) continue;
        const long long lo_w = __shfl_sync(0xffffffffu, lo, w);
        const unsigned hit = __ballot_sync(0xffffffffu, nbl > 0 && excl <= lo_w && lo_w < incl);
        if (hit == 0u) continue;
        pending &= ~(1u << w);
        if (lane == __ffs(hit) - 1) {
          const long long off = lo_w - excl;
          start[w].r = r;
          start[w].nb = nbl;
          start[w].h = static_cast<int>(off / nbl);
          start[w].b = static_cast<int>(off % nbl);
          start[w].first = excl + (off / nbl) * nbl;
        }
      }
      before = __shfl_sync(0xffffffffu, incl, 31);
    }
    // a range whose first block was not found (lengths changed under the kernel) does nothing
    if (lane < kConsumerWarps && (pending >> lane & 1u)) start[lane].n = 0;
    if (lane == 0) {
      *plan_nb = NB;
      *plan_w = W;
      if (blockIdx.x == 0) {
        p.plan[0] = NB;
        p.plan[1] = W;
      }
    }
  }
  __syncthreads();
  int n_max = 0;
#pragma unroll
  for (int w = 0; w < kConsumerWarps; ++w) n_max = max(n_max, start[w].n);
  if (n_max == 0) return;  // every thread of the CTA leaves here together

  if (warp == kConsumerWarps) {
    // ---------------- producer warp ----------------
    // Lane l translates, per batch of 8 rounds, round l / 4 of range l % 4; lane 0
    // then issues the batch's copies in order i = 4 t + w (stage i % kStages).
    const int w = lane & 3, tt = lane >> 2;
    const int n_w = start[w].n;
    Cursor c{start[w].first, start[w].r, start[w].h, start[w].b, start[w].nb};
    if (tt < n_w) advance(c, tt, p);
    auto table_entry = [&](const Cursor& cc) -> int {
      return cc.r < p.S ? p.block_table[static_cast<size_t>(cc.r) * p.max_blocks + cc.b] : -1;
    };
    int phys = tt < n_w ? table_entry(c) : 0;
    int issued_end = 0;  // one past the last copy index issued
    // every K/V byte is read once: let those lines go first, ahead of the
    // partial results, queries and table entries that are read again
    const uint64_t stream_policy = l2_policy_evict_first();
    bool stop = false;
    for (int t0 = 0; t0 < n_max && !stop; t0 += 8) {
      if (t0 + tt < n_w) {
        const bool bad = phys < 0 || phys >= p.num_pool_blocks;
        if (bad) raise_flag(p.flags, DEVFLAG_BAD_BLOCK);
        // a bad entry reads block 0 instead; the piece is reported as NaN
        rows[lane] = ((bad ? 0 : phys) * p.Hkv + c.h) * kBS;
        rbad[lane] = bad ? 1 : 0;
      }
      // the next batch's table entry is read while this batch is issued
      if (t0 + 8 + tt < n_w) {
        advance(c, 8, p);
        phys = table_entry(c);
      }
      __syncwarp();
      if (lane == 0) {
        for (int l = 0; l < 32; ++l) {
          const int t = t0 + (l >> 2), ww = l & 3;
          if (t >= start[ww].n) continue;
          const int i = kConsumerWarps * t + ww;
          const int s = i % kStages;
          if (!mbar_wait(bar_empty + 8 * s, ((i / kStages) & 1) ^ 1, abort, p.flags,
                         p.wait_limit_ns)) {
            stop = true;
            break;
          }
          stage_bad[s] = rbad[l];
          issued_end = i + 1;
          if (p.withhold_copy && i == 0) continue;  // test hook: the first block never arrives
          const uint32_t dst = sbase + s * C::STAGE_BYTES;
          mbar_arrive_expect_tx(bar_full + 8 * s, C::STAGE_BYTES);
#pragma unroll
          for (int kb = 0; kb < C::KB; ++kb) {
            tma_load_2d_hint(dst + kb * C::BOX_BYTES, &tmK, bar_full + 8 * s, kb * 64, rows[l],
                             stream_policy);
            tma_load_2d_hint(dst + C::BLK_BYTES + kb * C::BOX_BYTES, &tmV, bar_full + 8 * s,
                             kb * 64, rows[l], stream_policy);
          }
        }
      }
      stop = __shfl_sync(0xffffffffu, stop ? 1 : 0, 0) != 0;
    }
    __syncthreads();  // pairs with the consumers' final barrier
    if (lane == 0 && *abort) {
      // Copies still in flight land before the CTA's shared memory goes away.
      for (int i = max(0, issued_end - kStages); i < issued_end; ++i) {
        if (i / kConsumerWarps >= start[i % kConsumerWarps].n) continue;  // never issued
        if (p.withhold_copy && i == 0) continue;
        mbar_wait_quiet(bar_full + 8 * (i % kStages), (i / kStages) & 1, 500000000ull);
      }
    }
    return;
  }

  // ---------------- consumer warps ----------------
  // Transposed products: S^T = K Q^T (m = the block's 16 tokens, n = 8 queries)
  // and O^T += V^T P^T (m = 16 dims, n = 8 queries), so the GQA group (<= 8 or
  // <= 16 queries) fills the n side of m16n8k16 and each block takes
  // D / 16 * NQT MMAs per product.  Each lane holds tokens g, g + 8 and queries
  // 2 t4, 2 t4 + 1 of every 8-query tile.
  const int g = lane >> 2, t4 = lane & 3;
  const int group = p.group;
  const float sl2 = p.scale_log2;
  const int n_w = start[warp].n;
  const int k_w = blockIdx.x * kConsumerWarps + warp;
  const uint32_t ps = sbase + C::OFF_PS + warp * C::PS_WARP_BYTES;  // P as [query][token]
  Cursor c{start[warp].first, start[warp].r, start[warp].h, start[warp].b, start[warp].nb};

  uint32_t qb[D / 16][NQT][2];
  float m_q[NQT][2], l_q[NQT][2];   // running max (raw score) and partial sum per query
  float acc[D / 16][NQT][4];        // O^T: dims 16 j + g (+ 8), queries 8 nt + 2 t4 (+ 1)
  int L = 0;
  bool pbad = false;   // the piece read a block the table could not translate
  int piece_b0 = 0;    // block of the segment where the piece starts
  auto reset = [&]() {
#pragma unroll
    for (int nt = 0; nt < NQT; ++nt) {
      m_q[nt][0] = m_q[nt][1] = -INFINITY;
      l_q[nt][0] = l_q[nt][1] = 0.f;
#pragma unroll
      for (int j = 0; j < D / 16; ++j) acc[j][nt][0] = acc[j][nt][1] = acc[j][nt][2] = acc[j][nt][3] = 0.f;
    }
  };
  reset();
  if (n_w > 0) {
    L = p.seq_lens[c.r];
    load_q<D, NQT>(p, c.r, c.h, g, t4, qb);
    piece_b0 = c.b;
  }

  for (int t = 0; t < n_w; ++t) {
    const int i = kConsumerWarps * t + warp;
    const int s = i % kStages;
    if (!mbar_wait_warp(bar_full + 8 * s, (i / kStages) & 1, abort, p.flags, p.wait_limit_ns))
      break;
    const uint32_t kbase = sbase + s * C::STAGE_BYTES;
    const uint32_t vbase = kbase + C::BLK_BYTES;
    const int n_valid = min(kBS, L - c.b * kBS);
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

    // S^T = K Q^T: A = K (16 tokens x 16 dims per step), B = Q^T
    float sc[NQT][4];
#pragma unroll
    for (int nt = 0; nt < NQT; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
    {
      const int mat = lane >> 3, rr = lane & 7;
      const int tok = (mat & 1) * 8 + rr;
      const int dof = (mat >> 1) * 8;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        uint32_t a[4];
        ldsm_x4(swz(kbase, tok, kk * 16 + dof), a[0], a[1], a[2], a[3]);
#pragma unroll
        for (int nt = 0; nt < NQT; ++nt) mma_bf16_16816(sc[nt], a, qb[kk][nt][0], qb[kk][nt][1]);
      }
    }
    // mask tokens past the end (select, so NaN keys in dead slots cannot leak)
    if (g >= n_valid) {
#pragma unroll
      for (int nt = 0; nt < NQT; ++nt) sc[nt][0] = sc[nt][1] = -INFINITY;
    }
    if (g + 8 >= n_valid) {
#pragma unroll
      for (int nt = 0; nt < NQT; ++nt) sc[nt][2] = sc[nt][3] = -INFINITY;
    }
    __syncwarp();  // the previous block's P reads are done before P is rewritten
#pragma unroll
    for (int nt = 0; nt < NQT; ++nt) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        // max over the block's 16 tokens: lanes with the same t4 hold them
        float bm = fmaxf(sc[nt][e], sc[nt][2 + e]);
        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 4));
        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 8));
        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 16));
        const float mn = fmaxf(m_q[nt][e], bm);  // finite: every block has a valid token
        const float ms = mn * sl2;
        const float al = ex2(m_q[nt][e] * sl2 - ms);
        const float p0 = ex2(fmaf(sc[nt][e], sl2, -ms));
        const float p1 = ex2(fmaf(sc[nt][2 + e], sl2, -ms));
        l_q[nt][e] = l_q[nt][e] * al + (p0 + p1);
        m_q[nt][e] = mn;
#pragma unroll
        for (int j = 0; j < D / 16; ++j) {
          acc[j][nt][e] *= al;
          acc[j][nt][2 + e] *= al;
        }
        // P[query][token] as bf16
        const uint32_t prow = ps + (8 * nt + 2 * t4 + e) * 32;
        const uint32_t pp = pack_bf16x2(p0, p1);
        st_shared_u16(prow + g * 2, static_cast<uint16_t>(pp & 0xFFFFu));
        st_shared_u16(prow + (g + 8) * 2, static_cast<uint16_t>(pp >> 16));
      }
    }
    __syncwarp();
    // O^T += V^T P^T: A = V^T (16 dims x 16 tokens per tile), B = P^T from shared memory
    uint32_t pb[NQT][2];
#pragma unroll
    for (int nt = 0; nt < NQT; ++nt) {
      // matrix 0: queries 8nt..8nt+7, tokens 0..7; matrix 1: the same queries, tokens 8..15
      const int l8 = lane & 15;
      ldsm_x2(ps + (8 * nt + (l8 & 7)) * 32 + (l8 >> 3) * 16, pb[nt][0], pb[nt][1]);
    }
    {
      const int mat = lane >> 3, rr = lane & 7;
      const int tok = (mat >> 1) * 8 + rr;
      const int dof = (mat & 1) * 8;
#pragma unroll
      for (int j = 0; j < D / 16; ++j) {
        uint32_t a[4];
        ldsm_x4_t(swz(vbase, tok, j * 16 + dof), a[0], a[1], a[2], a[3]);
#pragma unroll
        for (int nt = 0; nt < NQT; ++nt) mma_bf16_16816(acc[j][nt], a, pb[nt][0], pb[nt][1]);
      }
    }
    pbad |= stage_bad[s] != 0;
    __syncwarp();
    if (n_valid < kBS) fence_proxy_async_smem();  // our generic writes before TMA reuses the stage
    if (lane == 0) mbar_arrive(bar_empty + 8 * s);

    ++c.b;
    if (c.b < c.nb && t + 1 < n_w) continue;
    // ---- the piece ends: write its normalised O and LSE ----
    {
      const long long NB = *plan_nb;
      const int W = *plan_w;
      const int j = k_w - range_of(c.first, NB, W);  // piece index within the segment
      const float nan = __int_as_float(0x7fc00000);
      const size_t hq0 = static_cast<size_t>(c.r) * p.Hq + c.h * group;
      if (j >= 0 && j < p.max_pieces) {
#pragma unroll
        for (int nt = 0; nt < NQT; ++nt) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            float lsum = l_q[nt][e];
            lsum += __shfl_xor_sync(0xffffffffu, lsum, 4);
            lsum += __shfl_xor_sync(0xffffffffu, lsum, 8);
            lsum += __shfl_xor_sync(0xffffffffu, lsum, 16);
            const int q = 8 * nt + 2 * t4 + e;
            if (q >= group) continue;
            const float inv = 1.f / lsum;
            const size_t base = (hq0 + q) * p.max_pieces + j;
            float* dst = p.part_o + base * D;
#pragma unroll
            for (int jj = 0; jj < D / 16; ++jj) {
              dst[16 * jj + g] = pbad ? nan : acc[jj][nt][e] * inv;
              dst[16 * jj + g + 8] = pbad ? nan : acc[jj][nt][2 + e] * inv;
            }
            if (g == 0) p.part_lse[base] = pbad ? nan : m_q[nt][e] * p.scale + logf(lsum);
          }
        }
        if (piece_b0 == 0 && lane == 0) p.seg_first[static_cast<size_t>(c.r) * p.Hkv + c.h] = c.first;
      }
    }
    if (t + 1 == n_w) break;
    // the range continues in the next segment
    advance(c, 0, p);
    if (c.r >= p.S) break;  // lengths changed under the kernel: nothing valid to read
    L = p.seq_lens[c.r];
    load_q<D, NQT>(p, c.r, c.h, g, t4, qb);
    piece_b0 = 0;
    pbad = false;
    reset();
  }
  __syncthreads();  // pairs with the producer's: no copy outlives the CTA
}

// One warp per (request, query head).  Pieces are taken 32 at a time: lane s
// holds the LSE of piece b0 + s and every lane the partial outputs of all 32
// (its D / 32 dims), loaded together.
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
  constexpr int PER = D / 32;  // dims per lane
  static_assert(PER == 2 || PER == 4, "D is 64 or 128");
  constexpr int kBatch = 32;   // pieces per batch: one per lane
  const float* pl = p.part_lse + hq * p.max_pieces;
  const float* po = p.part_o + hq * p.max_pieces * D + lane * PER;
  float part[kBatch][PER];
  // Loads the partial outputs of pieces b0 .. b0 + 31 below n (entries past n are
  // zero, never read: they may hold stale NaN).
  auto load_batch = [&](int b0, int n) {
#pragma unroll
    for (int s = 0; s < kBatch; ++s) {
      if (b0 + s < n) {
        const float* src = po + static_cast<size_t>(b0 + s) * D;
        if constexpr (PER == 4) {
          const float4 v = *reinterpret_cast<const float4*>(src);
          part[s][0] = v.x;
          part[s][1] = v.y;
          part[s][2] = v.z;
          part[s][3] = v.w;
        } else {
          const float2 v = *reinterpret_cast<const float2*>(src);
          part[s][0] = v.x;
          part[s][1] = v.y;
        }
      } else {
#pragma unroll
        for (int i = 0; i < PER; ++i) part[s][i] = 0.f;
      }
    }
  };
  // First round trip: the length, the plan, the segment start and the LSEs of the
  // first 32 pieces (one word per lane, in bounds whatever the piece count turns
  // out to be).  Second: the partial outputs of exactly the pieces that exist,
  // 32 per round trip (reading the unused slots too would double the bytes).
  const int L = p.seq_lens[r];
  const long long NB = p.plan[0];
  const int W = static_cast<int>(p.plan[1]);
  const long long first =
      p.seg_first[static_cast<size_t>(r) * p.Hkv + (warp_global % p.Hq) / p.group];
  const int n_first = min(kBatch, p.max_pieces);
  const float lse_first = lane < n_first ? pl[lane] : 0.f;

  uint16_t* orow = static_cast<uint16_t*>(p.o) + hq * D + lane * PER;
  const float qnan = __int_as_float(0x7fc00000);
  float res[PER];
  float lse_out;
  const int nb = (L + kBS - 1) / kBS;
  const bool valid_len = L >= 0 && L <= p.max_seq_len && L <= p.max_blocks * kBS;
  // (the plan always covers a valid nonempty request; the guard keeps every read
  // in bounds should the lengths have changed between the two kernels)
  const bool planned = valid_len && L > 0 && NB > 0 && W > 0 && first >= 0 && first + nb <= NB;
  const int ns = planned ? range_of(first + nb - 1, NB, W) - range_of(first, NB, W) + 1 : 0;
  if (!valid_len || (L > 0 && (ns < 1 || ns > p.max_pieces))) {
    if (lane == 0) raise_flag(p.flags, DEVFLAG_BAD_SEQLEN);
#pragma unroll
    for (int i = 0; i < PER; ++i) res[i] = qnan;
    lse_out = qnan;
  } else if (L == 0) {
#pragma unroll
    for (int i = 0; i < PER; ++i) res[i] = 0.f;
    lse_out = -INFINITY;
  } else {
    // M = max_j LSE_j, and whether any piece is NaN (a block the table could not
    // translate)
    float M = lane < ns ? lse_first : -INFINITY;
    bool nan = (M != M);
    for (int b0 = kBatch; b0 < ns; b0 += kBatch) {
      const float v = (b0 + lane < ns) ? pl[b0 + lane] : -INFINITY;
      nan |= (v != v);
      M = fmaxf(M, v);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    nan = __any_sync(0xffffffffu, nan);
    // weights and sums in piece order
    float tot = 0.f;
#pragma unroll
    for (int i = 0; i < PER; ++i) res[i] = 0.f;
    for (int b0 = 0; b0 < ns; b0 += kBatch) {
      load_batch(b0, ns);
      const float lse_lane = b0 == 0 ? lse_first : (b0 + lane < ns ? pl[b0 + lane] : 0.f);
      const float w_lane = (b0 + lane < ns) ? __expf(lse_lane - M) : 0.f;
#pragma unroll
      for (int s = 0; s < kBatch; ++s) {
        const float w = __shfl_sync(0xffffffffu, w_lane, s);
        if (b0 + s < ns) {
          tot += w;
#pragma unroll
          for (int i = 0; i < PER; ++i) res[i] += w * part[s][i];
        }
      }
    }
    const float inv = 1.f / tot;
#pragma unroll
    for (int i = 0; i < PER; ++i) res[i] *= inv;
    lse_out = M + logf(tot);
    if (nan) {
#pragma unroll
      for (int i = 0; i < PER; ++i) res[i] = qnan;
      lse_out = qnan;
    }
  }
#pragma unroll
  for (int i = 0; i < PER; i += 2) {
    *reinterpret_cast<uint32_t*>(orow + i) = pack_bf16x2(res[i], res[i + 1]);
  }
  if (p.lse != nullptr && lane == 0) p.lse[hq] = lse_out;
}

}  // namespace

int decode_max_pieces(int max_seq_len) {
  const int blocks = (max_seq_len + kBS - 1) / kBS;
  return (blocks + kMinBlocks - 1) / kMinBlocks + 1;
}

DecodeWorkspace decode_workspace_layout(int S, int Hq, int D, int max_seq_len) {
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  DecodeWorkspace w;
  const size_t n = static_cast<size_t>(S) * Hq * decode_max_pieces(max_seq_len);
  w.off_part_lse = up(n * D * sizeof(float));
  w.off_seg_first = w.off_part_lse + up(n * sizeof(float));
  w.off_plan = w.off_seg_first + up(static_cast<size_t>(S) * Hq * sizeof(long long));
  w.bytes = w.off_plan + up(2 * sizeof(long long));
  return w;
}

size_t decode_workspace_bytes(int S, int Hq, int D, int max_seq_len) {
  return decode_workspace_layout(S, Hq, D, max_seq_len).bytes;
}

template <int D, int NQT>
constexpr int split_smem_bytes() {
  return DecCfg<D, DecShape<NQT>::kStages>::SMEM_BYTES;
}

cudaError_t prepare_paged_decode() {
  cudaError_t e = cudaSuccess;
  auto set = [&](const void* fn, int bytes) {
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  };
  set(reinterpret_cast<const void*>(paged_decode_split_kernel<64, 1>), split_smem_bytes<64, 1>());
  set(reinterpret_cast<const void*>(paged_decode_split_kernel<64, 2>), split_smem_bytes<64, 2>());
  set(reinterpret_cast<const void*>(paged_decode_split_kernel<128, 1>), split_smem_bytes<128, 1>());
  set(reinterpret_cast<const void*>(paged_decode_split_kernel<128, 2>), split_smem_bytes<128, 2>());
  return e;
}

namespace {

template <int D>
cudaError_t launch_pair(const CUtensorMap& tmK, const CUtensorMap& tmV, const DecodeParams& p,
                        int num_sms, cudaStream_t stream) {
  // persistent: kCtasPerSm CTAs per SM, fewer when even 16-block ranges would not fill them
  const long long most_blocks =
      static_cast<long long>(p.S) * p.Hkv * ((p.max_seq_len + kBS - 1) / kBS);
  const long long want = (most_blocks / kMinBlocks + kConsumerWarps - 1) / kConsumerWarps;
  auto grid_for = [&](int ctas_per_sm) {
    return static_cast<int>(max(1ll, min(static_cast<long long>(num_sms) * ctas_per_sm, want)));
  };
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t split = {};
  split.blockDim = dim3(kThreads);
  split.stream = stream;
  split.attrs = attr;
  split.numAttrs = 1;
  cudaError_t e;
  if (p.group <= 8) {
    split.gridDim = dim3(grid_for(DecShape<1>::kCtasPerSm));
    split.dynamicSmemBytes = split_smem_bytes<D, 1>();
    e = cudaLaunchKernelEx(&split, paged_decode_split_kernel<D, 1>, tmK, tmV, p);
  } else {
    split.gridDim = dim3(grid_for(DecShape<2>::kCtasPerSm));
    split.dynamicSmemBytes = split_smem_bytes<D, 2>();
    e = cudaLaunchKernelEx(&split, paged_decode_split_kernel<D, 2>, tmK, tmV, p);
  }
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((p.S * p.Hq + 3) / 4);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, paged_decode_merge_kernel<D>, p);
}

}  // namespace

cudaError_t launch_paged_decode(const CUtensorMap& tmK, const CUtensorMap& tmV,
                                const DecodeParams& p, int num_sms, cudaStream_t stream) {
  if (p.S <= 0) return cudaSuccess;
  return p.D == 64 ? launch_pair<64>(tmK, tmV, p, num_sms, stream)
                   : launch_pair<128>(tmK, tmV, p, num_sms, stream);
}

}  // namespace gbattn
