// paged.cuh -- translation of a logical cache position through the block table,
// shared by every kernel that reads or writes the paged KV cache (decode, paged
// prefill, append, gather), so they agree on the mapping bit for bit.
//
// The method (the-ai.news, "Kernels de atencao rapida e fusao de operadores",
// section "Atencao do tipo FlashAttention e atencao paginada"): the KV cache is
// cut into fixed-size blocks, a block table maps each logical block of a request
// to a physical block, and every logical position is translated through it.
// Layout here: pools are [num_pool_blocks, Hkv, 16, D], so the 16 rows of one
// (physical block, KV head) are contiguous; viewed as a 2-D tensor of D-wide rows,
// token t of request r, KV head h is row
//     (block_table[r][t / 16] * Hkv + h) * 16 + t % 16.
#pragma once

#include <cstdint>

namespace gbattn {

constexpr int kPagedBlock = 16;  // tokens per KV block

// First pool row of logical block lb of request r, KV head kvh, or -1 when the
// table entry lies outside [0, num_pool_blocks).  The caller guarantees
// lb < max_blocks.
__device__ __forceinline__ int paged_block_row(const int32_t* block_table, int max_blocks, int r,
                                               int lb, int kvh, int Hkv, int num_pool_blocks) {
  const int phys = block_table[static_cast<size_t>(r) * max_blocks + lb];
  if (phys < 0 || phys >= num_pool_blocks) return -1;
  return (phys * Hkv + kvh) * kPagedBlock;
}

}  // namespace gbattn
