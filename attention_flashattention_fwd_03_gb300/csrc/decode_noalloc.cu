// decode_noalloc.cu -- paged decode for callers that cannot allocate device memory.
//
// paged_attn_decode needs a scratch workspace (the split-KV partial outputs and
// their log-sum-exps) that the caller allocates.  Some callers cannot: code that
// runs where cudaMalloc is not allowed or not available to it (inside a custom
// allocator's own callbacks, a plugin host that owns all device memory, a
// real-time loop that must not touch the allocator).  For them this file keeps
// the scratch in one file-scope device array of fixed size, reserved when the
// library's module is loaded on a device and held until the process exits.
//
// Host code cannot use the array's name as a device address (on the host it is
// only a stand-in symbol), so the address is looked up once per device with
// cudaGetSymbolAddress, with that device current, and handed to the kernels.
#include <cuda_runtime.h>

#include <mutex>

#include "gbattn.h"
#include "internal.h"

#define GBATTN_API extern "C" __attribute__((visibility("default")))

namespace gbattn {
namespace {

constexpr size_t kStaticScratchBytes = GBATTN_DECODE_NOALLOC_SCRATCH_BYTES;
static_assert(kStaticScratchBytes % 256 == 0, "scratch size must keep 256-byte alignment");

static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {};
int g_scratch_status[kMaxDevices] = {};  // 0 = not looked up yet

// Device address of the scratch array on the current device (looked up once).
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_status[dev] == 0) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess || p == nullptr) {
      g_scratch_status[dev] = ATTN_ERR_CUDA;
    } else {
      g_scratch_addr[dev] = p;
      g_scratch_status[dev] = -1;  // looked up, valid
    }
  }
  if (g_scratch_status[dev] != -1) return g_scratch_status[dev];
  *out = g_scratch_addr[dev];
  return ATTN_OK;
}

}  // namespace
}  // namespace gbattn

GBATTN_API int paged_attn_decode_noalloc(const void* q, const void* k_pool, const void* v_pool,
                                         const int32_t* block_table, const int32_t* seq_lens,
                                         int block_size, int num_seqs, int Hq, int Hkv, int D,
                                         int max_blocks_per_seq, int num_pool_blocks,
                                         int max_seq_len, float scale, void* o, float* lse,
                                         void* stream) {
  // Sizes are checked before anything touches a device; the ordinary entry point
  // repeats every other check.
  if (num_seqs < 0 || Hq <= 0 || D <= 0 || max_seq_len < 0) return ATTN_ERR_INVALID_ARG;
  if (num_seqs == 0) return ATTN_OK;
  const size_t need = gbattn::decode_workspace_bytes(num_seqs, Hq, D, max_seq_len);
  if (need > gbattn::kStaticScratchBytes) return ATTN_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  const int st = gbattn::scratch_address(&scratch);
  if (st != ATTN_OK) return st;
  return paged_attn_decode(q, k_pool, v_pool, block_table, seq_lens, block_size, num_seqs, Hq, Hkv,
                           D, max_blocks_per_seq, num_pool_blocks, max_seq_len, scale, o, lse,
                           scratch, gbattn::kStaticScratchBytes, stream);
}
