// internal.h -- launch interface between the C ABI (api.cu) and the kernels.
// Not installed; the public interface is include/gbattn.h.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace gbattn {

struct FwdParams {
  void* o;            // [B, Hq, Tq, D] bf16
  float* lse;         // [B, Hq, Tq] fp32 or nullptr
  int B, Hq, Hkv, Tq, Tk, D;
  int group;          // Hq / Hkv
  int causal;         // 1: query i sees keys j <= i + (L_b - Tq) (bottom-right alignment)
  int n_qpairs;       // ceil(Tq / 256): work units of two 128-row query tiles
  int num_units;      // B * Hq * n_qpairs
  float scale;        // softmax scale applied to q.k
  float scale_log2;   // scale * log2(e)
  unsigned* flags;    // device flag word (DEVFLAG_*)
  unsigned long long wait_limit_ns;  // limit of every pipeline wait
  int withhold_copy;  // test hook: the producer skips its first copy (a wait then runs out)
  // Paged K/V (prefill against a block-table cache).  With block_table == nullptr
  // K and V are contiguous [B, Hkv, Tk, D] and every batch item has Tk keys.
  const int32_t* block_table;  // [B, max_blocks]
  const int32_t* kv_lens;      // [B]: keys of each batch item (its own queries' included)
  int max_blocks;
  int num_pool_blocks;
  int max_kv_len;
};

// Prefill / full attention.  Contiguous: tmK/tmV are 3-D tiled maps over
// [B*Hkv, Tk, D] bf16 with a 64 x 128 x 1 box; paged: 2-D maps over the pools
// viewed as [num_pool_blocks * Hkv * 16, D] with a 64 x 16 box.  tmQ is a 3-D map
// over [B*Hq, Tq, D] with a 64 x 128 x 1 box.  All use the 128-byte swizzle.
cudaError_t launch_attn_fwd(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                            const FwdParams& p, int num_sms, cudaStream_t stream);
cudaError_t prepare_attn_fwd();  // per-device one-time attributes

struct DecodeParams {
  const void* q;               // [S, Hq, D] bf16
  const int32_t* block_table;  // [S, max_blocks]
  const int32_t* seq_lens;     // [S]
  void* o;                     // [S, Hq, D] bf16
  float* lse;                  // [S, Hq] or nullptr
  float* part_o;               // [S, Hq, max_pieces, D] fp32 (workspace)
  float* part_lse;             // [S, Hq, max_pieces] fp32 (workspace)
  long long* seg_first;        // [S, Hkv] first global block of each segment (workspace)
  long long* plan;             // [2]: total blocks NB, warp ranges W (workspace)
  int S, Hq, Hkv, D, group;
  int block_size;
  int max_blocks;
  int num_pool_blocks;
  int max_seq_len;
  int max_pieces;              // bound on the pieces of one (request, KV head) segment
  float scale;
  float scale_log2;
  unsigned* flags;             // device flag word (DEVFLAG_*)
  unsigned long long wait_limit_ns;  // limit of every pipeline wait
  int withhold_copy;           // test hook: the producer skips its first copy
};

// Shortest range of (request, KV head, block) triples one decode warp streams, in
// tokens.  It bounds the pieces a request's segment is cut into, and so the
// workspace: ceil(max_seq_len / 256) + 1 pieces per (request, query head).
constexpr int kDecodeMinRange = 256;

struct DecodeWorkspace {
  size_t off_part_lse, off_seg_first, off_plan, bytes;  // byte offsets (part_o at 0), size
};
DecodeWorkspace decode_workspace_layout(int S, int Hq, int D, int max_seq_len);
int decode_max_pieces(int max_seq_len);

// Paged decode.  tmK/tmV are 2-D tiled maps over the pools viewed as
// [num_pool_blocks * Hkv * block_size, D] bf16 with a 64 x 16 box, 128-byte swizzle.
cudaError_t launch_paged_decode(const CUtensorMap& tmK, const CUtensorMap& tmV,
                                const DecodeParams& p, int num_sms, cudaStream_t stream);
cudaError_t prepare_paged_decode();

size_t decode_workspace_bytes(int S, int Hq, int D, int max_seq_len);

struct AppendParams {
  const void* k_new;           // [S, Hkv, Tn, D] bf16
  const void* v_new;           // [S, Hkv, Tn, D] bf16
  void* k_pool;                // [num_pool_blocks, Hkv, 16, D] bf16 (written)
  void* v_pool;
  const int32_t* block_table;  // [S, max_blocks]
  const int32_t* seq_lens;     // [S]: lengths before the append
  int32_t* new_seq_lens;       // [S]: seq_lens + Tn (nullable, never aliases seq_lens)
  int S, Hkv, Tn, D;
  int max_blocks;
  int num_pool_blocks;
  unsigned* flags;
};

struct GatherParams {
  const int32_t* block_table;  // [S, max_blocks]
  const int32_t* seq_lens;     // [S]
  void* out;                   // [S, Hkv, max_seq_len, D] bf16
  int S, Hkv, D;
  int max_blocks;
  int num_pool_blocks;
  int max_seq_len;
  unsigned* flags;
  unsigned long long wait_limit_ns;
  int withhold_copy;           // test hook: the copies are not issued
};

// KV-cache append and gather.  The gather's tmPool is the decode kernels' 2-D map
// over a pool viewed as [num_pool_blocks * Hkv * 16, D] with a 64 x 16 box.
cudaError_t launch_kv_append(const AppendParams& p, cudaStream_t stream);
cudaError_t launch_kv_gather(const CUtensorMap& tmPool, const GatherParams& p,
                             cudaStream_t stream);
cudaError_t prepare_kv_cache();


}  // namespace gbattn
