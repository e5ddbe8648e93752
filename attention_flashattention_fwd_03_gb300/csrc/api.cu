// api.cu -- the C ABI declared in include/gbattn.h: argument validation,
// per-device one-time set-up, TMA tensor-map encoding and kernel launches.
// No allocation, no host synchronisation (except attn_device_status), no
// fallback: anything the kernels do not support is reported as an error.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "gbattn.h"
#include "internal.h"

#define GBATTN_API extern "C" __attribute__((visibility("default")))

namespace gbattn {

// The library's device flag word (one per device that loads the library).
__device__ unsigned int g_flags_word;

namespace {

constexpr int kMaxDevices = 64;

struct DeviceState {
  bool initialized = false;
  int status = ATTN_OK;
  int num_sms = 0;
  unsigned* flags = nullptr;
};

std::mutex g_mutex;
DeviceState g_dev[kMaxDevices];

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
int g_encode_status = ATTN_OK;

void init_encode() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q{};
  cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                   cudaEnableDefault, &q);
  if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr) {
    g_encode_status = ATTN_ERR_CUDA;
    return;
  }
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}

// One-time per-device checks and kernel attributes; returns a status.
int device_state(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState& st = g_dev[dev];
  if (!st.initialized) {
    st.initialized = true;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&st.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      st.status = ATTN_ERR_CUDA;
    } else if (major != 10 || minor != 3) {
      st.status = ATTN_ERR_UNSUPPORTED;  // kernels are built for sm_103a only
    } else if (prepare_attn_fwd(64) != cudaSuccess || prepare_attn_fwd(128) != cudaSuccess ||
               prepare_paged_decode() != cudaSuccess ||
               cudaGetSymbolAddress(reinterpret_cast<void**>(&st.flags), g_flags_word) !=
                   cudaSuccess) {
      st.status = ATTN_ERR_CUDA;
    } else {
      st.status = ATTN_OK;
    }
  }
  *out = &st;
  return st.status;
}

int encoder(PFN_cuTensorMapEncodeTiled_v12000* fn) {
  std::call_once(g_encode_once, init_encode);
  *fn = g_encode;
  return g_encode_status;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Tiled map over a bf16 tensor of `rank` dims (innermost first), 128-byte swizzle.
int encode_bf16(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap* map, const void* base,
                int rank, const uint64_t* dims, const uint64_t* strides_bytes,
                const uint32_t* box) {
  cuuint64_t gdim[3];
  cuuint64_t gstride[2];
  cuuint32_t bdim[3];
  cuuint32_t estride[3] = {1, 1, 1};
  for (int i = 0; i < rank; ++i) {
    gdim[i] = dims[i];
    bdim[i] = box[i];
  }
  for (int i = 0; i + 1 < rank; ++i) gstride[i] = strides_bytes[i];
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, static_cast<cuuint32_t>(rank),
                   const_cast<void*>(base), gdim, gstride, bdim, estride,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_CUDA;
}

constexpr uint64_t kMaxDim = 1ull << 31;  // keeps every TMA coordinate inside int32

}  // namespace
}  // namespace gbattn

using namespace gbattn;

GBATTN_API const char* attn_status_string(int status) {
  switch (status) {
    case ATTN_OK: return "ATTN_OK";
    case ATTN_ERR_INVALID_ARG: return "ATTN_ERR_INVALID_ARG";
    case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED";
    case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA";
    case ATTN_ERR_DEVICE: return "ATTN_ERR_DEVICE";
    default: return "ATTN_ERR_UNKNOWN";
  }
}

GBATTN_API int attn_version(void) { return 100; }

GBATTN_API int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                        int Hq, int Hkv, int T, int D, int causal, float scale, void* stream) {
  // ---- validation (no device access) ----
  if (B < 0 || T < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
  if (B == 0 || T == 0) return ATTN_OK;
  if (!q || !k || !v || !o) return ATTN_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
      (lse && !aligned(lse, 4)))
    return ATTN_ERR_INVALID_ARG;
  const uint64_t bhq = static_cast<uint64_t>(B) * Hq, bhkv = static_cast<uint64_t>(B) * Hkv;
  const uint64_t n_qtiles = (static_cast<uint64_t>(T) + 127) / 128;
  if (bhq >= kMaxDim || static_cast<uint64_t>(T) >= kMaxDim || bhq * n_qtiles >= kMaxDim ||
      bhq * T >= (1ull << 40))
    return ATTN_ERR_UNSUPPORTED;

  DeviceState* ds = nullptr;
  int st = device_state(&ds);
  if (st != ATTN_OK) return st;
  PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
  if ((st = encoder(&enc)) != ATTN_OK) return st;

  CUtensorMap tmQ, tmK, tmV;
  const uint64_t row_bytes = static_cast<uint64_t>(D) * 2;
  const uint64_t strides[2] = {row_bytes, row_bytes * T};
  const uint32_t box[3] = {64, 128, 1};
  const uint64_t dq[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(T), bhq};
  const uint64_t dkv[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(T), bhkv};
  if ((st = encode_bf16(enc, &tmQ, q, 3, dq, strides, box)) != ATTN_OK) return st;
  if ((st = encode_bf16(enc, &tmK, k, 3, dkv, strides, box)) != ATTN_OK) return st;
  if ((st = encode_bf16(enc, &tmV, v, 3, dkv, strides, box)) != ATTN_OK) return st;

  FwdParams p;
  p.o = o;
  p.lse = lse;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.T = T;
  p.D = D;
  p.group = Hq / Hkv;
  p.causal = causal;
  p.n_qtiles = static_cast<int>(n_qtiles);
  p.n_kvtiles = static_cast<int>(n_qtiles);
  p.num_tiles = static_cast<int>(bhq * n_qtiles);
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.flags = ds->flags;
  if (launch_attn_fwd(tmQ, tmK, tmV, p, ds->num_sms, static_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return ATTN_ERR_CUDA;
  return ATTN_OK;
}

GBATTN_API size_t paged_attn_decode_workspace_size(int num_seqs, int Hq, int D, int max_seq_len) {
  if (num_seqs < 0 || Hq <= 0 || D <= 0 || max_seq_len < 0) return 0;
  return decode_workspace_bytes(num_seqs, Hq, D, max_seq_len);
}

GBATTN_API int paged_attn_decode(const void* q, const void* k_pool, const void* v_pool,
                                 const int32_t* block_table, const int32_t* seq_lens,
                                 int block_size, int num_seqs, int Hq, int Hkv, int D,
                                 int max_blocks_per_seq, int num_pool_blocks, int max_seq_len,
                                 float scale, void* o, float* lse, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  if (num_seqs < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || max_blocks_per_seq <= 0 ||
      num_pool_blocks <= 0 || max_seq_len < 0)
    return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_INVALID_ARG;
  if (block_size != 16 || (D != 64 && D != 128) || Hq / Hkv > 16) return ATTN_ERR_UNSUPPORTED;
  if (num_seqs == 0) return ATTN_OK;
  if (!q || !k_pool || !v_pool || !block_table || !seq_lens || !o || !workspace)
    return ATTN_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(o, 16) ||
      !aligned(block_table, 4) || !aligned(seq_lens, 4) || (lse && !aligned(lse, 4)) ||
      !aligned(workspace, 256))
    return ATTN_ERR_INVALID_ARG;
  const size_t need = decode_workspace_bytes(num_seqs, Hq, D, max_seq_len);
  if (workspace_bytes < need) return ATTN_ERR_INVALID_ARG;
  const uint64_t rows = static_cast<uint64_t>(num_pool_blocks) * Hkv * block_size;
  const int max_splits = (max_seq_len + kDecodeChunk - 1) / kDecodeChunk;
  if (rows >= kMaxDim ||
      static_cast<uint64_t>(num_seqs) * Hkv * (max_splits > 0 ? max_splits : 1) >= kMaxDim ||
      static_cast<uint64_t>(num_seqs) * max_blocks_per_seq >= (1ull << 40))
    return ATTN_ERR_UNSUPPORTED;

  DeviceState* ds = nullptr;
  int st = device_state(&ds);
  if (st != ATTN_OK) return st;
  PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
  if ((st = encoder(&enc)) != ATTN_OK) return st;

  CUtensorMap tmK, tmV;
  const uint64_t dims[2] = {static_cast<uint64_t>(D), rows};
  const uint64_t strides[1] = {static_cast<uint64_t>(D) * 2};
  const uint32_t box[2] = {64, 16};
  if ((st = encode_bf16(enc, &tmK, k_pool, 2, dims, strides, box)) != ATTN_OK) return st;
  if ((st = encode_bf16(enc, &tmV, v_pool, 2, dims, strides, box)) != ATTN_OK) return st;

  DecodeParams p;
  p.q = q;
  p.block_table = block_table;
  p.seq_lens = seq_lens;
  p.o = o;
  p.lse = lse;
  const size_t splits = static_cast<size_t>(max_splits > 0 ? max_splits : 1);
  const size_t n = static_cast<size_t>(num_seqs) * Hq * splits;
  p.part_o = static_cast<float*>(workspace);
  p.part_lse = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                        ((n * D * sizeof(float) + 255) & ~static_cast<size_t>(255)));
  p.S = num_seqs;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.D = D;
  p.group = Hq / Hkv;
  p.block_size = block_size;
  p.max_blocks = max_blocks_per_seq;
  p.num_pool_blocks = num_pool_blocks;
  p.max_seq_len = max_seq_len;
  p.max_splits = static_cast<int>(splits);
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.flags = ds->flags;
  if (launch_paged_decode(tmK, tmV, p, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return ATTN_ERR_CUDA;
  return ATTN_OK;
}

GBATTN_API int attn_device_status(unsigned int* flags) {
  if (cudaDeviceSynchronize() != cudaSuccess) return ATTN_ERR_CUDA;
  DeviceState* ds = nullptr;
  int st = device_state(&ds);
  if (st != ATTN_OK) return st;
  unsigned v = 0;
  if (cudaMemcpy(&v, ds->flags, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess)
    return ATTN_ERR_CUDA;
  if (v != 0) {
    const unsigned zero = 0;
    if (cudaMemcpy(ds->flags, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
      return ATTN_ERR_CUDA;
  }
  if (flags) *flags = v;
  return v ? ATTN_ERR_DEVICE : ATTN_OK;
}
