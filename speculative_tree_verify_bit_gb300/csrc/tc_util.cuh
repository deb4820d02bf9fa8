// tc_util.cuh -- sm_103a building blocks shared by the two verify kernels
// (verify_tc.cu: the exact path and the int4 cache; verify_i8.cu: the int8
// path's per-group integer dots): mbarrier waits with a bound, bulk async
// copies, tcgen05 MMA issue and tensor-memory loads/stores, shared-memory
// matrix descriptors and the 128-byte swizzle.  Everything sits in an
// anonymous namespace, so each translation unit has its own copy.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace stv {
namespace {

constexpr uint32_t kSpinLimit = 1u << 13;   // test_wait polls before a polling wait starts suspending
constexpr uint32_t kWaitLimit = 1u << 16;   // try_wait calls before a wait gives up (about 1.3 s)
constexpr uint32_t kSuspendHintNs = 20000;  // per try_wait
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ uint32_t su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }

// ---- mbarriers ----
__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t n) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(n) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(b)) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(b)), "r"(bytes) : "memory");
}
// try_wait suspends the thread (up to the hint, in ns) until the phase
// completes, so a waiting warp does not take issue slots from working ones.
__device__ __forceinline__ bool mbar_try(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(su32(b)), "r"(parity), "r"(kSuspendHintNs)
      : "memory");
  return ok != 0;
}
// Non-blocking check of a phase (one shared-memory round trip).
__device__ __forceinline__ uint32_t probe(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile("{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
               : "=r"(ok) : "r"(su32(b)), "r"(parity) : "memory");
  return ok;
}

// Bounded waits by one thread.  False on timeout (which sets the CTA's
// abort flag) or when the CTA aborted.
//  - suspending: try_wait only;
//  - polling: test_wait first, so a phase that completes within about half a
//    millisecond is seen one shared-memory round trip after it does (a
//    suspended warp can wake up much later), then try_wait.  A poll issues a
//    handful of instructions per round trip.  Kept out of line: one copy
//    serves every call site, which keeps the warp-specialised loops small in
//    the instruction cache.
__device__ __forceinline__ bool wait_suspend(uint64_t* b, uint32_t parity, volatile int* abort_flag) {
  for (uint32_t it = 0; it < kWaitLimit; ++it) {
    if (mbar_try(b, parity)) return true;
    if ((it & 63) == 63 && *abort_flag) return false;
  }
  *abort_flag = 1;
  return false;
}
__device__ __noinline__ bool wait_poll(uint64_t* b, uint32_t parity, volatile int* abort_flag) {
  for (uint32_t it = 0; it < kSpinLimit; ++it) {
    if (probe(b, parity)) return true;
    if ((it & 255) == 255 && *abort_flag) return false;
  }
  return wait_suspend(b, parity, abort_flag);
}
template <bool kPoll>
__device__ __forceinline__ bool wait1(uint64_t* b, uint32_t parity, volatile int* abort_flag) {
  if constexpr (kPoll) return wait_poll(b, parity, abort_flag);
  else return wait_suspend(b, parity, abort_flag);
}
// Bounded wait by a whole warp; the result is warp-uniform.
template <bool kPoll>
__device__ __forceinline__ bool waitw(uint64_t* b, uint32_t parity, volatile int* abort_flag) {
  bool ok = wait1<kPoll>(b, parity, abort_flag);
  return __all_sync(0xffffffffu, ok);
}
// A warp that needs several barriers checks them all at once with `probe`
// (the round trips overlap) and then settles each one: `settle` blocks only
// if some lane saw that phase incomplete.  A phase seen complete stays so
// until the warp's own next arrival, so an early check remains valid.
template <bool kPoll>
__device__ __forceinline__ bool settle(uint64_t* b, uint32_t parity, uint32_t probed, volatile int* abort_flag) {
  if (__all_sync(0xffffffffu, probed)) return true;
  return waitw<kPoll>(b, parity, abort_flag);
}

// Bounded wait, by one thread, until a device-memory counter that other CTAs
// of the same launch increment reaches `target`.  The load is an acquire, so
// what those CTAs wrote before their increments is visible afterwards; the
// proxy fence then orders it before this thread's later bulk copies.  The
// CTAs waited for must be resident (a cooperative launch).  False on timeout
// (at most about 1.5 s: each poll is a trip to L2 and a 128 ns sleep; sets
// the CTA's abort flag) or when the CTA aborted.  The short sleep keeps the
// waiter within a fraction of a microsecond of the last increment.
constexpr uint32_t kCountWaitLimit = 1u << 21;
__device__ __forceinline__ bool wait_count(const uint32_t* c, uint32_t target, volatile int* abort_flag) {
  for (uint32_t it = 0; it < kCountWaitLimit; ++it) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(c) : "memory");
    if (v >= target) {
      asm volatile("fence.proxy.async.global;" ::: "memory");
      return true;
    }
    if ((it & 63) == 63 && *abort_flag) return false;
    __nanosleep(128);
  }
  *abort_flag = 1;
  return false;
}

// ---- copies and proxies ----
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   su32(dst)),
               "l"(src), "r"(bytes), "r"(su32(bar))
               : "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, __half2 a, __half2 b, __half2 c, __half2 d) {
  st_shared_v4(addr, h2u(a), h2u(b), h2u(c), h2u(d));
}
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// ---- tcgen05 ----
__device__ __forceinline__ void tc_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// Issued by one elected lane of a converged warp: the warp runs the MMA loop
// in uniform control flow, so descriptors stay in uniform registers.
__device__ __forceinline__ void tc_commit(uint64_t* b) {
  asm volatile(
      "{\n .reg .pred e;\n elect.sync _|e, 0xffffffff;\n"
      " @e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}\n" ::"r"(su32(b))
      : "memory");
}
// D (TMEM) = A (TMEM) x B (shared-memory descriptor) (+ D when acc != 0).
__device__ __forceinline__ void mma_tmemA(uint32_t d, uint32_t a, uint64_t bdesc, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p, e;\n setp.ne.u32 p, %4, 0;\n elect.sync _|e, 0xffffffff;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d),
      "r"(a), "l"(bdesc), "r"(idesc), "r"(acc)
      : "memory");
}
// Instruction descriptor of kind::f16: f16 A and B (K-major), f32 D.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N) {
  return (1u << 4)                     // D: f32
         | ((uint32_t)(N >> 3) << 17)  // N
         | ((uint32_t)(M >> 4) << 24);  // M
}

#define STV_R8(i) "=r"(r[i]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), "=r"(r[i + 4]), "=r"(r[i + 5]), "=r"(r[i + 6]), "=r"(r[i + 7])
#define STV_W8(i) "r"(r[i]), "r"(r[i + 1]), "r"(r[i + 2]), "r"(r[i + 3]), "r"(r[i + 4]), "r"(r[i + 5]), "r"(r[i + 6]), "r"(r[i + 7])

// 32 (16) consecutive 32-bit columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%"
      "19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : STV_R8(0), STV_R8(8), STV_R8(16), STV_R8(24)
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      STV_W8(0), STV_W8(8), STV_W8(16), STV_W8(24)
      : "memory");
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : STV_R8(0), STV_R8(8)
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      STV_W8(0), STV_W8(8)
      : "memory");
}
// Wait for this thread's TMEM loads; the n registers of r are ordered after
// the wait.
template <int n = 32>
__device__ __forceinline__ void tmem_wait_ld(uint32_t* r) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < n; ++i) asm volatile("" : "+r"(r[i]));
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor: 128-byte swizzle, K-major, 8-row groups
// 1024 bytes apart (stride byte offset), sm_100-family version field.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// 128-byte-swizzled K-major tile: rows of 128 bytes in 8-row groups of 1024
// bytes; 16-byte chunk c of row `row` sits at chunk c ^ (row % 8).  A row's
// base with its XOR term folded in makes each chunk address one XOR.
__device__ __forceinline__ uint32_t sw128_row(int row) {
  return (uint32_t)((row >> 3) * 1024 + (row & 7) * 128 + ((row & 7) << 4));
}
__device__ __forceinline__ uint32_t sw128_chunk(uint32_t row_base, int c) { return row_base ^ (uint32_t)(c << 4); }

// 2^x with the SFU's approximate exponential (inputs here are <= 8; results
// below the normal range flush to zero, which a softmax weight can afford).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Zero the pairs of `out` whose keys (32 * blk + 2m, + 1) are at or past
// `live` (stale bytes past the key range could decode to anything).
__device__ __forceinline__ void zero_dead_keys(__half2 (&out)[16], int blk, int live) {
  if (live >= 64) return;
#pragma unroll
  for (int m = 0; m < 16; ++m) {
    const int k0 = blk * 32 + 2 * m;
    if (k0 >= live) out[m] = __floats2half2_rn(0.f, 0.f);
    else if (k0 + 1 >= live) out[m] = __halves2half2(__low2half(out[m]), __float2half_rn(0.f));
  }
}

}  // namespace
}  // namespace stv
