// kv_cache.cu -- writing new tokens into, and reading a request's history out of,
// the paged KV cache, on sm_103a.
//
// The method (the-ai.news, "Kernels de atencao rapida e fusao de operadores",
// section "Atencao do tipo FlashAttention e atencao paginada"): the KV cache grows
// token by token and is stored in fixed-size blocks; a block table maps each
// logical block of a request to a physical block.
//   append   the Tn new tokens of each request go to logical positions
//            L .. L + Tn - 1 (L = its current length): one warp per (request,
//            KV head, token) copies the token's K and V rows (D bf16 each) to
//            the translated pool row with 16-byte stores.  Pure data movement:
//            the pools change bit for bit as a host-side scatter would.
//   gather   one CTA per (request, KV head, 512-token chunk) translates the
//            chunk's blocks with the same routine the attention kernels use and
//            copies each (block, head) slice with the same TMA box (16 rows, 128-
//            byte swizzle) into shared memory, then writes the rows out in
//            logical order.  It exposes the attention kernels' gather path, so
//            its indexing can be checked byte for byte.
#include <cuda_runtime.h>

#include "internal.h"
#include "paged.cuh"
#include "ptx.cuh"

namespace gbattn {

namespace {

template <int D>
__global__ void __launch_bounds__(256)
    paged_kv_append_kernel(const AppendParams p) {
  // a decode launched next as a programmatic dependent may start its set-up now;
  // it waits for this grid's writes before it reads anything
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const long long w = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const long long total = static_cast<long long>(p.S) * p.Hkv * p.Tn;
  if (w >= total) return;
  const int t = static_cast<int>(w % p.Tn);
  const long long rh = w / p.Tn;
  const int h = static_cast<int>(rh % p.Hkv);
  const int r = static_cast<int>(rh / p.Hkv);
  const int L = p.seq_lens[r];
  const bool first = (t == 0 && h == 0 && lane == 0);
  if (L < 0 || L > p.max_blocks * kPagedBlock - p.Tn) {
    if (first) {
      raise_flag(p.flags, DEVFLAG_BAD_SEQLEN);
      if (p.new_seq_lens) p.new_seq_lens[r] = L;
    }
    return;
  }
  if (first && p.new_seq_lens) p.new_seq_lens[r] = L + p.Tn;
  const int pos = L + t;
  const int row0 = paged_block_row(p.block_table, p.max_blocks, r, pos / kPagedBlock, h, p.Hkv,
                                   p.num_pool_blocks);
  if (row0 < 0) {
    if (lane == 0) raise_flag(p.flags, DEVFLAG_BAD_BLOCK);
    return;
  }
  constexpr int CH = D / 8;  // 16-byte chunks per row
  const size_t dst = (static_cast<size_t>(row0) + pos % kPagedBlock) * D;
  const size_t src = (static_cast<size_t>(rh) * p.Tn + t) * D;
  if (lane < CH) {
    const uint4 v = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.k_new) + src)[lane];
    reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.k_pool) + dst)[lane] = v;
  } else if (lane < 2 * CH) {
    const uint4 v =
        reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.v_new) + src)[lane - CH];
    reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.v_pool) + dst)[lane - CH] = v;
  }
}

constexpr int kGatherChunk = 512;                          // tokens per CTA
constexpr int kGatherBlocks = kGatherChunk / kPagedBlock;  // 32
constexpr int kGatherThreads = 256;

template <int D>
struct GatherCfg {
  static constexpr int KB = D / 64;
  static constexpr int BOX_BYTES = kPagedBlock * 128;  // 16 rows x 128 bytes
  static constexpr int BLK_BYTES = kPagedBlock * D * 2;
  static constexpr int OFF_BAR = kGatherBlocks * BLK_BYTES;
  static constexpr int OFF_ROWS = OFF_BAR + 16;
  static constexpr int SMEM_BYTES = OFF_ROWS + kGatherBlocks * 4 + 1024;
};

template <int D>
__global__ void __launch_bounds__(kGatherThreads)
    paged_kv_gather_kernel(const __grid_constant__ CUtensorMap tmPool, const GatherParams p) {
  using C = GatherCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw);
  const uint32_t bar = sbase + C::OFF_BAR;
  int* rows = reinterpret_cast<int*>(smem + C::OFF_ROWS);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + C::OFF_BAR + 8);

  const int n_chunks = (p.max_seq_len + kGatherChunk - 1) / kGatherChunk;
  const int c = blockIdx.x % n_chunks;
  const int rh = blockIdx.x / n_chunks;
  const int h = rh % p.Hkv, r = rh / p.Hkv;
  const int L = p.seq_lens[r];
  if (L < 0 || L > p.max_seq_len || L > p.max_blocks * kPagedBlock) {
    if (threadIdx.x == 0 && c == 0 && h == 0) raise_flag(p.flags, DEVFLAG_BAD_SEQLEN);
    return;
  }
  const int t0 = c * kGatherChunk;
  if (t0 >= L) return;
  const int n_tok = min(kGatherChunk, L - t0);
  const int nblk = (n_tok + kPagedBlock - 1) / kPagedBlock;

  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    *abort = 0;
    fence_barrier_init();
  }
  if (threadIdx.x < nblk) {
    const int row = paged_block_row(p.block_table, p.max_blocks, r, t0 / kPagedBlock + threadIdx.x,
                                    h, p.Hkv, p.num_pool_blocks);
    if (row < 0) raise_flag(p.flags, DEVFLAG_BAD_BLOCK);
    rows[threadIdx.x] = row;
  }
  __syncthreads();
  if (threadIdx.x == 0 && !p.withhold_copy) {
    int valid = 0;
    for (int b = 0; b < nblk; ++b) valid += rows[b] >= 0;
    mbar_arrive_expect_tx(bar, valid * C::BLK_BYTES);
    for (int b = 0; b < nblk; ++b) {
      if (rows[b] < 0) continue;
#pragma unroll
      for (int kb = 0; kb < C::KB; ++kb)
        tma_load_2d(sbase + b * C::BLK_BYTES + kb * C::BOX_BYTES, &tmPool, bar, kb * 64, rows[b]);
    }
  }
  const bool landed = mbar_wait(bar, 0, abort, p.flags, p.wait_limit_ns);
  // copy out: one 16-byte chunk per thread and step, rows in logical order
  constexpr int CH = D / 8;
  uint4* out = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) +
                                        (static_cast<size_t>(rh) * p.max_seq_len + t0) * D);
  const uint4 nan4 = make_uint4(0x7fc07fc0u, 0x7fc07fc0u, 0x7fc07fc0u, 0x7fc07fc0u);
  for (int e = threadIdx.x; e < n_tok * CH; e += kGatherThreads) {
    const int tok = e / CH, ch = e % CH;
    const int b = tok / kPagedBlock, s = tok % kPagedBlock;
    uint4 v = nan4;
    if (landed && rows[b] >= 0) {
      const int box = ch >> 3, cc = ch & 7;
      v = *reinterpret_cast<const uint4*>(smem + b * C::BLK_BYTES + box * C::BOX_BYTES + s * 128 +
                                          ((cc ^ (s & 7)) << 4));
    }
    out[static_cast<size_t>(tok) * CH + ch] = v;
  }
  if (!landed && threadIdx.x == 0 && !p.withhold_copy)
    mbar_wait_quiet(bar, 0, 500000000ull);  // copies in flight
}

}  // namespace

cudaError_t prepare_kv_cache() {
  cudaError_t e = cudaFuncSetAttribute(paged_kv_gather_kernel<64>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       GatherCfg<64>::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(paged_kv_gather_kernel<128>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              GatherCfg<128>::SMEM_BYTES);
}

cudaError_t launch_kv_append(const AppendParams& p, cudaStream_t stream) {
  const long long warps = static_cast<long long>(p.S) * p.Hkv * p.Tn;
  if (warps <= 0) return cudaSuccess;
  const long long blocks = (warps * 32 + 255) / 256;
  if (p.D == 64)
    paged_kv_append_kernel<64><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(p);
  else
    paged_kv_append_kernel<128><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_kv_gather(const CUtensorMap& tmPool, const GatherParams& p,
                             cudaStream_t stream) {
  const int n_chunks = (p.max_seq_len + kGatherChunk - 1) / kGatherChunk;
  const long long grid = static_cast<long long>(p.S) * p.Hkv * n_chunks;
  if (grid <= 0) return cudaSuccess;
  if (p.D == 64)
    paged_kv_gather_kernel<64><<<static_cast<unsigned>(grid), kGatherThreads,
                                 GatherCfg<64>::SMEM_BYTES, stream>>>(tmPool, p);
  else
    paged_kv_gather_kernel<128><<<static_cast<unsigned>(grid), kGatherThreads,
                                  GatherCfg<128>::SMEM_BYTES, stream>>>(tmPool, p);
  return cudaGetLastError();
}

}  // namespace gbattn
