// internal.h -- launch interface between the C ABI (api.cu) and the kernels.
// Not installed; the public interface is include/gbattn.h.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace gbattn {

struct FwdParams {
  void* o;            // [B, Hq, T, D] bf16
  float* lse;         // [B, Hq, T] fp32 or nullptr
  int B, Hq, Hkv, T, D;
  int group;          // Hq / Hkv
  int causal;
  int n_qtiles;       // ceil(T / 128)
  int n_kvtiles;      // ceil(T / 128)
  int num_tiles;      // B * Hq * n_qtiles
  float scale;        // softmax scale applied to q.k
  float scale_log2;   // scale * log2(e)
  unsigned* flags;    // device flag word (DEVFLAG_*)
};

// Prefill / full attention.  tm* are 3-D tiled maps over [B*H, T, D] bf16 with
// 128-byte swizzle and a 64 x 128 x 1 box.
cudaError_t launch_attn_fwd(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                            const FwdParams& p, int num_sms, cudaStream_t stream);
cudaError_t prepare_attn_fwd(int D);  // per-device one-time attributes

struct DecodeParams {
  const void* q;               // [S, Hq, D] bf16
  const int32_t* block_table;  // [S, max_blocks]
  const int32_t* seq_lens;     // [S]
  void* o;                     // [S, Hq, D] bf16
  float* lse;                  // [S, Hq] or nullptr
  float* part_o;               // [S, Hq, max_splits, D] fp32 (workspace)
  float* part_lse;             // [S, Hq, max_splits] fp32 (workspace)
  int S, Hq, Hkv, D, group;
  int block_size;
  int max_blocks;
  int num_pool_blocks;
  int max_seq_len;
  int max_splits;
  float scale;
  float scale_log2;
  unsigned* flags;             // device flag word (DEVFLAG_*)
};

constexpr int kDecodeChunk = 512;  // logical tokens per split (fixed: results depend only on logical positions)

// Paged decode.  tmK/tmV are 2-D tiled maps over the pools viewed as
// [num_pool_blocks * Hkv * block_size, D] bf16 with a 64 x 16 box, 128-byte swizzle.
cudaError_t launch_paged_decode(const CUtensorMap& tmK, const CUtensorMap& tmV,
                                const DecodeParams& p, cudaStream_t stream);
cudaError_t prepare_paged_decode();

size_t decode_workspace_bytes(int S, int Hq, int D, int max_seq_len);


}  // namespace gbattn
