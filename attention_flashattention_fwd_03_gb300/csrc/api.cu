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
#include <atomic>
#include <mutex>

#include "gbattn.h"
#include "internal.h"
#include "ptx.cuh"

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
    } else if (prepare_attn_fwd() != cudaSuccess || prepare_paged_decode() != cudaSuccess ||
               prepare_kv_cache() != cudaSuccess ||
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

// Limit of every pipeline wait inside the kernels (ns); see attn_test_set_failure.
std::atomic<unsigned long long> g_wait_limit_ns{kWaitLimitNs};
std::atomic<int> g_withhold_copy{0};  // see attn_test_set_failure

FwdParams fwd_params(void* o, float* lse, int B, int Hq, int Hkv, int Tq, int Tk, int D,
                     int causal, float scale, unsigned* flags) {
  FwdParams p{};
  p.o = o;
  p.lse = lse;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.Tq = Tq;
  p.Tk = Tk;
  p.D = D;
  p.group = Hq / Hkv;
  p.causal = causal;
  p.n_qpairs = (Tq + 255) / 256;
  p.num_units = B * Hq * p.n_qpairs;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.flags = flags;
  p.wait_limit_ns = g_wait_limit_ns.load(std::memory_order_relaxed);
  p.withhold_copy = g_withhold_copy.load(std::memory_order_relaxed);
  p.block_table = nullptr;
  p.kv_lens = nullptr;
  return p;
}

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
  const uint64_t n_qpairs = (static_cast<uint64_t>(T) + 255) / 256;
  if (bhq >= kMaxDim || static_cast<uint64_t>(T) >= kMaxDim || bhq * n_qpairs >= kMaxDim ||
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

  FwdParams p = fwd_params(o, lse, B, Hq, Hkv, T, T, D, causal, scale, ds->flags);
  if (launch_attn_fwd(tmQ, tmK, tmV, p, ds->num_sms, static_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return ATTN_ERR_CUDA;
  return ATTN_OK;
}

GBATTN_API int paged_attn_prefill(const void* q, const void* k_pool, const void* v_pool,
                                  const int32_t* block_table, const int32_t* kv_lens,
                                  int block_size, int B, int Hq, int Hkv, int Tq, int D,
                                  int max_blocks_per_seq, int num_pool_blocks, int max_kv_len,
                                  int causal, float scale, void* o, float* lse, void* stream) {
  if (B < 0 || Tq < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || max_blocks_per_seq <= 0 ||
      num_pool_blocks <= 0 || max_kv_len < 0)
    return ATTN_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_INVALID_ARG;
  if (block_size != 16 || (D != 64 && D != 128)) return ATTN_ERR_UNSUPPORTED;
  if (B == 0 || Tq == 0) return ATTN_OK;
  if (!q || !k_pool || !v_pool || !block_table || !kv_lens || !o) return ATTN_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(o, 16) ||
      !aligned(block_table, 4) || !aligned(kv_lens, 4) || (lse && !aligned(lse, 4)))
    return ATTN_ERR_INVALID_ARG;
  const uint64_t bhq = static_cast<uint64_t>(B) * Hq;
  const uint64_t n_qpairs = (static_cast<uint64_t>(Tq) + 255) / 256;
  const uint64_t rows = static_cast<uint64_t>(num_pool_blocks) * Hkv * block_size;
  if (bhq >= kMaxDim || bhq * n_qpairs >= kMaxDim || bhq * Tq >= (1ull << 40) ||
      rows >= kMaxDim || static_cast<uint64_t>(B) * max_blocks_per_seq >= (1ull << 40))
    return ATTN_ERR_UNSUPPORTED;

  DeviceState* ds = nullptr;
  int st = device_state(&ds);
  if (st != ATTN_OK) return st;
  PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
  if ((st = encoder(&enc)) != ATTN_OK) return st;

  CUtensorMap tmQ, tmK, tmV;
  const uint64_t row_bytes = static_cast<uint64_t>(D) * 2;
  const uint64_t q_strides[2] = {row_bytes, row_bytes * Tq};
  const uint32_t q_box[3] = {64, 128, 1};
  const uint64_t dq[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(Tq), bhq};
  const uint64_t dpool[2] = {static_cast<uint64_t>(D), rows};
  const uint64_t pool_strides[1] = {row_bytes};
  const uint32_t pool_box[2] = {64, 16};
  if ((st = encode_bf16(enc, &tmQ, q, 3, dq, q_strides, q_box)) != ATTN_OK) return st;
  if ((st = encode_bf16(enc, &tmK, k_pool, 2, dpool, pool_strides, pool_box)) != ATTN_OK) return st;
  if ((st = encode_bf16(enc, &tmV, v_pool, 2, dpool, pool_strides, pool_box)) != ATTN_OK) return st;

  FwdParams p = fwd_params(o, lse, B, Hq, Hkv, Tq, max_kv_len, D, causal, scale, ds->flags);
  p.block_table = block_table;
  p.kv_lens = kv_lens;
  p.max_blocks = max_blocks_per_seq;
  p.num_pool_blocks = num_pool_blocks;
  p.max_kv_len = max_kv_len;
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
  if (rows >= kMaxDim || static_cast<uint64_t>(num_seqs) * Hq >= kMaxDim ||
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
  const DecodeWorkspace wl = decode_workspace_layout(num_seqs, Hq, D, max_seq_len);
  char* ws = static_cast<char*>(workspace);
  p.part_o = reinterpret_cast<float*>(ws);
  p.part_lse = reinterpret_cast<float*>(ws + wl.off_part_lse);
  p.seg_first = reinterpret_cast<long long*>(ws + wl.off_seg_first);
  p.plan = reinterpret_cast<long long*>(ws + wl.off_plan);
  p.S = num_seqs;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.D = D;
  p.group = Hq / Hkv;
  p.block_size = block_size;
  p.max_blocks = max_blocks_per_seq;
  p.num_pool_blocks = num_pool_blocks;
  p.max_seq_len = max_seq_len;
  p.max_pieces = decode_max_pieces(max_seq_len);
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.flags = ds->flags;
  p.wait_limit_ns = g_wait_limit_ns.load(std::memory_order_relaxed);
  p.withhold_copy = g_withhold_copy.load(std::memory_order_relaxed);
  if (launch_paged_decode(tmK, tmV, p, ds->num_sms, static_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return ATTN_ERR_CUDA;
  return ATTN_OK;
}

GBATTN_API int paged_kv_append(const void* k_new, const void* v_new, void* k_pool, void* v_pool,
                               const int32_t* block_table, const int32_t* seq_lens,
                               int32_t* new_seq_lens, int block_size, int num_seqs, int Hkv,
                               int Tn, int D, int max_blocks_per_seq, int num_pool_blocks,
                               void* stream) {
  if (num_seqs < 0 || Hkv <= 0 || Tn < 0 || max_blocks_per_seq <= 0 || num_pool_blocks <= 0)
    return ATTN_ERR_INVALID_ARG;
  if (block_size != 16 || (D != 64 && D != 128)) return ATTN_ERR_UNSUPPORTED;
  if (num_seqs == 0 || Tn == 0) return ATTN_OK;
  if (!k_new || !v_new || !k_pool || !v_pool || !block_table || !seq_lens)
    return ATTN_ERR_INVALID_ARG;
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) ||
      !aligned(block_table, 4) || !aligned(seq_lens, 4) ||
      (new_seq_lens && !aligned(new_seq_lens, 4)))
    return ATTN_ERR_INVALID_ARG;
  if (new_seq_lens) {  // the output lengths must not overlap the input lengths
    const uintptr_t a = reinterpret_cast<uintptr_t>(seq_lens);
    const uintptr_t b = reinterpret_cast<uintptr_t>(new_seq_lens);
    const uintptr_t n = static_cast<uintptr_t>(num_seqs) * sizeof(int32_t);
    if (a < b + n && b < a + n) return ATTN_ERR_INVALID_ARG;
  }
  const uint64_t rows = static_cast<uint64_t>(num_pool_blocks) * Hkv * block_size;
  if (rows >= kMaxDim || static_cast<uint64_t>(num_seqs) * Hkv * Tn * 32 >= (1ull << 40) ||
      static_cast<uint64_t>(max_blocks_per_seq) * block_size >= kMaxDim)
    return ATTN_ERR_UNSUPPORTED;
  DeviceState* ds = nullptr;
  const int st = device_state(&ds);
  if (st != ATTN_OK) return st;
  AppendParams p{};
  p.k_new = k_new;
  p.v_new = v_new;
  p.k_pool = k_pool;
  p.v_pool = v_pool;
  p.block_table = block_table;
  p.seq_lens = seq_lens;
  p.new_seq_lens = new_seq_lens;
  p.S = num_seqs;
  p.Hkv = Hkv;
  p.Tn = Tn;
  p.D = D;
  p.max_blocks = max_blocks_per_seq;
  p.num_pool_blocks = num_pool_blocks;
  p.flags = ds->flags;
  return launch_kv_append(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? ATTN_OK
                                                                                : ATTN_ERR_CUDA;
}

GBATTN_API int paged_kv_gather(const void* pool, const int32_t* block_table,
                               const int32_t* seq_lens, int block_size, int num_seqs, int Hkv,
                               int D, int max_blocks_per_seq, int num_pool_blocks, int max_seq_len,
                               void* out, void* stream) {
  if (num_seqs < 0 || Hkv <= 0 || max_blocks_per_seq <= 0 || num_pool_blocks <= 0 ||
      max_seq_len < 0)
    return ATTN_ERR_INVALID_ARG;
  if (block_size != 16 || (D != 64 && D != 128)) return ATTN_ERR_UNSUPPORTED;
  if (num_seqs == 0 || max_seq_len == 0) return ATTN_OK;
  if (!pool || !block_table || !seq_lens || !out) return ATTN_ERR_INVALID_ARG;
  if (!aligned(pool, 16) || !aligned(out, 16) || !aligned(block_table, 4) ||
      !aligned(seq_lens, 4))
    return ATTN_ERR_INVALID_ARG;
  const uint64_t rows = static_cast<uint64_t>(num_pool_blocks) * Hkv * block_size;
  const uint64_t chunks = (static_cast<uint64_t>(max_seq_len) + 511) / 512;
  if (rows >= kMaxDim || static_cast<uint64_t>(num_seqs) * Hkv * chunks >= kMaxDim ||
      static_cast<uint64_t>(num_seqs) * max_blocks_per_seq >= (1ull << 40))
    return ATTN_ERR_UNSUPPORTED;
  DeviceState* ds = nullptr;
  int st = device_state(&ds);
  if (st != ATTN_OK) return st;
  PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
  if ((st = encoder(&enc)) != ATTN_OK) return st;
  CUtensorMap tm;
  const uint64_t dims[2] = {static_cast<uint64_t>(D), rows};
  const uint64_t strides[1] = {static_cast<uint64_t>(D) * 2};
  const uint32_t box[2] = {64, 16};
  if ((st = encode_bf16(enc, &tm, pool, 2, dims, strides, box)) != ATTN_OK) return st;
  GatherParams p{};
  p.block_table = block_table;
  p.seq_lens = seq_lens;
  p.out = out;
  p.S = num_seqs;
  p.Hkv = Hkv;
  p.D = D;
  p.max_blocks = max_blocks_per_seq;
  p.num_pool_blocks = num_pool_blocks;
  p.max_seq_len = max_seq_len;
  p.flags = ds->flags;
  p.wait_limit_ns = g_wait_limit_ns.load(std::memory_order_relaxed);
  p.withhold_copy = g_withhold_copy.load(std::memory_order_relaxed);
  return launch_kv_gather(tm, p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? ATTN_OK
                                                                                    : ATTN_ERR_CUDA;
}

GBATTN_API int attn_test_set_failure(unsigned long long wait_limit_ns, int withhold_copy) {
  if (withhold_copy != 0 && withhold_copy != 1) return ATTN_ERR_INVALID_ARG;
  g_wait_limit_ns.store(wait_limit_ns == 0 ? kWaitLimitNs : wait_limit_ns);
  g_withhold_copy.store(withhold_copy);
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
