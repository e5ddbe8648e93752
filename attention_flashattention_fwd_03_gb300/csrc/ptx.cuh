// ptx.cuh -- thin inline-PTX wrappers for the sm_103a building blocks the
// kernels use: mbarriers, TMA tensor copies, tcgen05 MMA / TMEM, and a few
// scalar conversions.  Written from the public PTX ISA description of each
// instruction; every wait that can block has an iteration/time limit so a
// broken pipeline reports an error instead of hanging the GPU.
#pragma once

#include <cstdint>
#include <cuda.h>

namespace gbattn {

// --------------------------------------------------------------------------
// error reporting shared by all kernels (a device word read by the host API)
// --------------------------------------------------------------------------
enum : unsigned {
  DEVFLAG_TIMEOUT = 1u << 0,      // a bounded wait gave up
  DEVFLAG_BAD_SEQLEN = 1u << 1,   // decode: seq_len < 0 or beyond the table / max_seq_len
  DEVFLAG_BAD_BLOCK = 1u << 2,    // decode: block id outside the pool
};

// The flag word lives in the library's one device-global (api.cu); kernels get
// its address as a parameter so no relocatable device code is needed.
__device__ __forceinline__ void raise_flag(unsigned* flags, unsigned f) { atomicOr(flags, f); }

// Default wall-clock limit of any single wait (ns).  Kernels here run for
// milliseconds; a wait this long means a broken pipeline, not a slow one.  The
// limit actually used is a kernel parameter, so a test can shorten it.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// --------------------------------------------------------------------------
// mbarrier
// --------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking test of a phase.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// try_wait that suspends the thread for at most hint_ns while the phase is
// incomplete (it resumes as soon as the phase completes).
__device__ __forceinline__ bool mbar_try_wait_hint(uint32_t bar, uint32_t parity,
                                                   uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.b32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Optional sleep between two failed polls of a wait (ns), which leaves issue
// slots to the warps that share the waiting warp's scheduler.  Measured on the
// prefill kernel, 32, 64 and 128 ns made no difference beyond noise, so it is 0.
#ifndef GBATTN_POLL_SLEEP_NS
#define GBATTN_POLL_SLEEP_NS 0
#endif

// Suspension per poll: the wait limit, but at most 1 ms, so a limit is noticed
// within about a millisecond of running out.
__device__ __forceinline__ uint32_t poll_hint(unsigned long long limit_ns) {
  return limit_ns < 1000000ull ? static_cast<uint32_t>(limit_ns) : 1000000u;
}

// Waits (one thread) until the phase with the given parity has completed.  Gives
// up (and returns false) after limit_ns or as soon as *abort is set by another
// role of the same CTA; on a timeout it raises DEVFLAG_TIMEOUT and sets *abort.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort,
                                          unsigned* flags,
                                          unsigned long long limit_ns = kWaitLimitNs) {
  const uint32_t hint = poll_hint(limit_ns);
  if (mbar_try_wait_hint(bar, parity, hint)) return true;
  const unsigned long long t0 = globaltimer();
  for (;;) {
    if (GBATTN_POLL_SLEEP_NS > 0) __nanosleep(GBATTN_POLL_SLEEP_NS);
    if (mbar_try_wait_hint(bar, parity, hint)) return true;
    if (*abort) return false;
    if (globaltimer() - t0 > limit_ns) {
      raise_flag(flags, DEVFLAG_TIMEOUT);
      *abort = 1;
      return false;
    }
  }
}

// The same wait for a whole warp; the result (and the abort / timeout decision)
// is the same in every lane, so the warp stays converged for the .sync.aligned
// instructions that follow.  First lane 0 alone tests the phase without blocking:
// most waits find it complete, and 32 lanes polling one mbarrier made even those
// cost about 200 cycles.  (A lone lane blocking in try_wait with a suspend hint
// while the rest of the warp waited at a shuffle was measured 5x slower overall:
// the blocking poll stays warp-wide.)  The __syncwarp that follows (a barrier with memory ordering) orders
// the other lanes' reads of the copied data after lane 0's observation, and lanes
// that go on to tcgen05 work order it with tcgen05.fence::after_thread_sync.
// Otherwise every lane polls until the phase completes.
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity, volatile int* abort,
                                               unsigned* flags, unsigned long long limit_ns) {
  const uint32_t hint = poll_hint(limit_ns);
  // common case: the phase has completed; one lane tests it without blocking
  uint32_t ok = 0;
  if ((threadIdx.x & 31) == 0) ok = mbar_test_wait(bar, parity) ? 1u : 0u;
  if (__shfl_sync(0xffffffffu, ok, 0)) {
    __syncwarp();
    return true;
  }
  // waiting: every lane polls (each lane then has observed the phase itself)
  const unsigned long long t0 = globaltimer();
  for (;;) {
    if (GBATTN_POLL_SLEEP_NS > 0) __nanosleep(GBATTN_POLL_SLEEP_NS);
    if (__all_sync(0xffffffffu, mbar_try_wait_hint(bar, parity, hint))) return true;
    int give_up = 0;
    if ((threadIdx.x & 31) == 0) {
      if (*abort) {
        give_up = 1;
      } else if (globaltimer() - t0 > limit_ns) {
        raise_flag(flags, DEVFLAG_TIMEOUT);
        *abort = 1;
        give_up = 1;
      }
    }
    if (__shfl_sync(0xffffffffu, give_up, 0)) return false;
  }
}

// Bounded wait used during teardown after an abort: never raises, just gives up.
__device__ __forceinline__ void mbar_wait_quiet(uint32_t bar, uint32_t parity,
                                                unsigned long long limit_ns) {
  const unsigned long long t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > limit_ns) return;
  }
}

// --------------------------------------------------------------------------
// TMA (tensor copies, global -> shared), completion counted on an mbarrier
// --------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}

// An L2 policy that marks lines as first to evict (for data read exactly once).
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// tma_load_2d with an L2 cache policy for the fetched lines.
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                                 int c0, int c1, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "l"(policy)
      : "memory");
}

// --------------------------------------------------------------------------
// tcgen05: TMEM allocation, MMA, commit, TMEM <-> register moves
// --------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// tcgen05.mma, kind::f16 (bf16 in, fp32 accumulate), issued from a whole converged
// warp: every lane holds the same (warp-uniform) operands and elect.sync picks the
// one lane that issues.  Issuing from a converged warp keeps the operands in
// uniform registers, which makes back-to-back MMAs issue at the tensor pipe's
// rate; one lane issuing alone from a divergent branch cost up to 1.7x the pipe
// time per MMA in measurements.
// D[tmem] (+)= A[smem desc] * B[smem desc]^T
__device__ __forceinline__ void mma_ss_warp(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem desc]^T
__device__ __forceinline__ void mma_ts_warp(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// tcgen05.commit from the lane elect.sync picks in a converged warp (the lane
// that issued the MMAs above, as elect.sync picks the same lane every time): the
// mbarrier receives one arrival once every tcgen05 operation that lane issued so
// far has completed.
__device__ __forceinline__ void mma_commit_warp(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
          bar)
      : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread i of the warp gets lane
// (taddr.lane + i), columns taddr.col .. +31.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

// 32 lanes x 8 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
      : "memory");
}

// 32 lanes x 16 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

// 32 lanes x 16 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}

// --------------------------------------------------------------------------
// UMMA descriptors
// --------------------------------------------------------------------------
// Shared-memory matrix descriptor (tcgen05 form): start address >> 4 in bits
// 0-13, leading byte offset >> 4 in 16-29, stride byte offset >> 4 in 32-45,
// the fixed value 1 in bits 46-47, base offset 0, swizzle mode in 61-63
// (2 = 128-byte swizzle).  Tiles are 1024-byte aligned so the base offset is 0.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr, uint32_t lbo_bytes,
                                                    uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((addr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;
  d |= 2ull << 61;
  return d;
}

// Instruction descriptor for kind::f16 with bf16 A/B and fp32 D:
// D format bits 4-5 (1 = f32), A format 7-9 (1 = bf16), B format 10-12,
// A major bit 15 / B major bit 16 (0 = K-major, 1 = MN-major), N >> 3 in
// bits 17-22, M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, int a_mn_major,
                                                      int b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(a_mn_major) << 15) |
         (static_cast<uint32_t>(b_mn_major) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// --------------------------------------------------------------------------
// scalar helpers
// --------------------------------------------------------------------------
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Packs two floats into bf16x2 with round-to-nearest-even: lo -> bits 0-15.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Register reallocation between warpgroups (every thread of the warpgroup runs
// the same instruction).  The block is launched with a fixed total; the counts
// used with these must add up to at most that total.
template <int N>
__device__ __forceinline__ void regs_increase() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void regs_decrease() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// Largest of three floats (the three-input max of sm_100 and later).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// 2^x for a pair of values, evaluated on the FMA pipe instead of the
// special-function unit, for x <= 127 (softmax exponents here are <= 8); inputs
// below -126 are clamped there.  Cody-Waite style range reduction (W. J. Cody
// and W. Waite, "Software Manual for the Elementary Functions", 1980): x = n + f
// with n = round(x) and f in [-1/2, 1/2]; adding 1.5 * 2^23 rounds x to an
// integer in the low mantissa bits, which also yields n << 23 as an integer.
// 2^f is a degree-3 polynomial whose coefficients come from a minimax fit on
// [-1/2, 1/2] (Lawson's iteratively reweighted least squares, evaluated in
// fp32): max relative error 7.5e-5, far below the 2^-9 relative rounding of the
// bf16 probabilities it produces.  The arithmetic uses the packed fp32x2 forms.
__device__ __forceinline__ float2 exp2_fma2(float2 x) {
  const float2 kRound = make_float2(12582912.0f, 12582912.0f);  // 1.5 * 2^23
  const float2 kMinus = make_float2(-12582912.0f, -12582912.0f);
  const float2 xc = make_float2(fmaxf(x.x, -126.0f), fmaxf(x.y, -126.0f));
  const float2 t = __fadd2_rn(xc, kRound);
  const float2 n = __fadd2_rn(t, kMinus);
  const float2 f = __ffma2_rn(n, make_float2(-1.f, -1.f), xc);
  float2 p = __ffma2_rn(make_float2(0.05517149344086647f, 0.05517149344086647f), f,
                        make_float2(0.24261093139648438f, 0.24261093139648438f));
  p = __ffma2_rn(p, f, make_float2(0.6932609677314758f, 0.6932609677314758f));
  p = __ffma2_rn(p, f, make_float2(0.9999280571937561f, 0.9999280571937561f));
  return make_float2(__uint_as_float(__float_as_uint(p.x) + (__float_as_uint(t.x) << 23)),
                     __uint_as_float(__float_as_uint(p.y) + (__float_as_uint(t.y) << 23)));
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

}  // namespace gbattn
