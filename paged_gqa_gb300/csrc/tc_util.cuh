// tc_util.cuh -- inline-PTX wrappers for sm_103a: mbarriers, TMA, tcgen05 (MMA, TMEM).
//
// Every wait is bounded: after kWaitLimitNs of failed polls (global timer) it records
// kErrTimeout in the device error word, raises the CTA's abort flag and returns false, so
// no kernel can hang the GPU on a lost arrival.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_fp16.h>
#include "common.cuh"

namespace pgqa {
namespace tc {

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier --
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.b32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait for the phase with the given parity to complete. Gives up at once (false)
// when the CTA's abort flag is raised, or after limit_ns (then it records kErrTimeout and
// raises the abort flag itself).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          uint32_t* err, uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0u) {
      if (*abort_flag) return false;
      if (global_timer_ns() - t0 > limit_ns) break;
    }
  }
  atomicOr(err, kErrTimeout);
  *abort_flag = 1;
  return false;
}

// mbar_wait by one lane of a converged warp while the other lanes wait at __syncwarp (which
// orders their later accesses after lane 0's acquire): one poller per warp instead of 32, so
// warps that wait do not flood the shared-memory pipe that other warps' copies, shuffles and
// barrier arrivals use. Every lane gets the result.
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                               uint32_t* err, int lane) {
  int ok = 1;
  if (lane == 0) ok = mbar_wait(bar, parity, abort_flag, err);
  __syncwarp();
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// One arrival on `bar` for the whole warp, after every lane's earlier accesses (ordered by
// __syncwarp before lane 0's release). The barrier then counts warps, not threads.
__device__ __forceinline__ void mbar_arrive_warp(uint32_t bar, int lane) {
  __syncwarp();
  if (lane == 0) mbar_arrive(bar);
}

// Wait for this thread's own asynchronous work (TMA copies, MMAs) signalled on `bar` before
// the CTA releases its shared memory or TMEM. Unlike mbar_wait it does not give up when the
// abort flag is raised (that work is in flight either way and completes by itself); it
// is still bounded by kWaitLimitNs, after which it records kErrTimeout.
__device__ __forceinline__ bool mbar_drain(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                           uint32_t* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0u && global_timer_ns() - t0 > kWaitLimitNs) break;
  }
  atomicOr(err, kErrTimeout);
  *abort_flag = 1;
  return false;
}

// ---------------------------------------------------------------- fences --
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// ---------------------------------------------------------------- TMA --
__device__ __forceinline__ void tma_prefetch_desc(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}
// 4-D tiled load into shared memory, completion signalled on `bar` (bytes).
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const void* tmap, int c0, int c1, int c2, int c3,
                                            uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar), "l"(policy)
      : "memory");
}
// Bulk (non-tensor) copy shared -> global, tracked by this thread's bulk async-groups.
__device__ __forceinline__ void bulk_store(void* gdst, uint32_t ssrc, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst), "r"(ssrc), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Bulk (non-tensor) copy global -> shared, completion counted on `bar` (bytes).
__device__ __forceinline__ void bulk_load(uint32_t sdst, const void* gsrc, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(sdst),
               "l"(gsrc), "r"(bytes), "r"(bar)
               : "memory");
}
// The shared-memory sources of every committed bulk store have been read.
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Every committed bulk store has been written to global memory.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<uint64_t>(p)));
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ---------------------------------------------------------------- tcgen05 --
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Shared-memory matrix descriptor (sm_100 family layout).
//   start address, leading and stride byte offsets (>> 4), version 1, swizzle mode.
enum Swizzle : uint32_t { kSwNone = 0, kSw128 = 2, kSw64 = 4, kSw32 = 6 };
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo, Swizzle sw) {
  uint64_t d = 0;
  d |= (uint64_t)((addr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)sw << 61;
  return d;
}

// Instruction descriptor: fp32 accumulate; A/B e4m3 (kind::f8f6f4); major-ness; N, M.
__host__ __device__ constexpr uint32_t idesc_e4m3(int M, int N, bool a_mn_major, bool b_mn_major) {
  return (1u << 4)                                  // D format f32
         | (0u << 7) | (0u << 10)                   // A, B = e4m3
         | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16)
         | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_e4m3(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// As mma_e4m3 with the A operand in TMEM (M lanes, 4 e4m3 K-elements per 32-bit column).
__device__ __forceinline__ void mma_e4m3_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Instruction descriptor of kind::f16 with bf16 A and B (format code 1), fp32 accumulate.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn_major, bool b_mn_major) {
  return (1u << 4)                                  // D format f32
         | (1u << 7) | (1u << 10)                   // A, B = bf16
         | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16)
         | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
// D (+)= A B with A and B in shared memory, 16-bit inputs (K = 16 per instruction).
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// As mma_f16 with the A operand in TMEM (M lanes, 2 16-bit K-elements per 32-bit column).
__device__ __forceinline__ void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on `bar` once all previously issued tcgen05 async ops of this thread complete.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 32 lanes x 32 bit, 16 consecutive columns -> 16 registers per thread.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15]))
      : "memory");
}

__device__ __forceinline__ void tmem_st16u(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
      "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}

// ---------------------------------------------------------------- math --
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// The largest / smallest of three (max.f32 / min.f32 with three inputs, sm_100 and later):
// one instruction where two-input ones take two dependent steps. Same NaN rule as fmaxf.
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
__device__ __forceinline__ float min3f(float a, float b, float c) {
  float r;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
// Maximum (kMax) or minimum of N values: four independent chains of N / 4 values each, of
// three-input steps, then their combination. 34 instructions, 10 deep, for N = 64, against
// 63 dependent ones for a plain running maximum; the result is the same value.
template <bool kMax, int N>
__device__ __forceinline__ float extreme_of(const float (&t)[N]) {
  static_assert(N % 8 == 0, "four chains of an even number of values");
  constexpr int kQ = N / 4;
  auto f3 = [](float a, float b, float c) { return kMax ? max3f(a, b, c) : min3f(a, b, c); };
  auto f2 = [](float a, float b) { return kMax ? fmaxf(a, b) : fminf(a, b); };
  float a[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) a[k] = t[k * kQ];
#pragma unroll
  for (int i = 1; i + 1 < kQ; i += 2)
#pragma unroll
    for (int k = 0; k < 4; ++k) a[k] = f3(a[k], t[k * kQ + i], t[k * kQ + i + 1]);
#pragma unroll
  for (int k = 0; k < 4; ++k) a[k] = f2(a[k], t[k * kQ + kQ - 1]);
  return f3(f2(a[0], a[1]), a[2], a[3]);
}
__device__ __forceinline__ float warp_max(float v) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}
// Two floats -> two e4m3 codes, round to nearest even, saturating; `lo` in the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
// x0..x3 (exponents, <= 8) -> p = 2^x in f16, then p = hi + lo with hi, lo in e4m3:
// hi/lo get one byte per key (x0 in the low byte), s01/s23 the f16 values of p.
__device__ __forceinline__ void p_split4_f16(float x0, float x1, float x2, float x3, uint32_t& hi, uint32_t& lo,
                                             __half2& s01, __half2& s23) {
  uint32_t a, b, ha, hb, ba, bb, ra, rb;
  uint16_t ea, eb, la, lb;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(a) : "f"(x1), "f"(x0));
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(b) : "f"(x3), "f"(x2));
  asm("ex2.approx.f16x2 %0, %1;" : "=r"(ha) : "r"(a));
  asm("ex2.approx.f16x2 %0, %1;" : "=r"(hb) : "r"(b));
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(ea) : "r"(ha));
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(eb) : "r"(hb));
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(ba) : "h"(ea));
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(bb) : "h"(eb));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(ra) : "r"(ha), "r"(ba));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(rb) : "r"(hb), "r"(bb));
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(la) : "r"(ra));
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(lb) : "r"(rb));
  hi = (uint32_t)ea | ((uint32_t)eb << 16);
  lo = (uint32_t)la | ((uint32_t)lb << 16);
  s01 = *reinterpret_cast<__half2*>(&ha);
  s23 = *reinterpret_cast<__half2*>(&hb);
}

// The per-tensor e4m3 scale of a bf16 Q from the amax kernel's per-CTA maxima: descale =
// amax / 448 and its reciprocal, each rounded to nearest in fp32; an amax of zero (or not
// finite) takes descale = inv = 1. All lanes of the warp get the same pair {descale, inv}.
__device__ __forceinline__ float2 q_cast_scales(const float* parts, int n, int lane) {
  float a = 0.f;
  for (int i = lane; i < n; i += 32) a = fmaxf(a, parts[i]);
  a = warp_max(a);
  if (!(a > 0.f) || !isfinite(a)) return make_float2(1.f, 1.f);
  const float d = __fdiv_rn(a, 448.f);
  return make_float2(d, __frcp_rn(d));
}
// 16 bf16 values (two uint4, element 0 first) times inv -> 16 e4m3 codes (uint4).
__device__ __forceinline__ uint4 bf16x16_to_e4m3(uint4 a, uint4 b, float inv) {
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  uint32_t c[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t u = w[2 * i], v = w[2 * i + 1];
    c[i] = e4m3x2(__fmul_rn(__uint_as_float(u << 16), inv), __fmul_rn(__uint_as_float(u & 0xffff0000u), inv)) |
           (e4m3x2(__fmul_rn(__uint_as_float(v << 16), inv), __fmul_rn(__uint_as_float(v & 0xffff0000u), inv))
            << 16);
  }
  return make_uint4(c[0], c[1], c[2], c[3]);
}

// Two e4m3 codes (low byte first) -> two exact floats.
__device__ __forceinline__ float2 e4m3x2_to_f2(uint32_t v) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((uint16_t)v));
  __half2 h = *reinterpret_cast<__half2*>(&h2);
  return __half22float2(h);
}

// y -> (hi, lo) e4m3 bytes of 4 values packed in two words (y = hi + lo exactly when y has at
// most 8 significant bits and |y| >= 2^-2; the caller scales y into [128, 256) first).
__device__ __forceinline__ void split4(float a, float b, float c, float d, uint32_t& hi, uint32_t& lo) {
  const uint32_t h01 = e4m3x2(a, b), h23 = e4m3x2(c, d);
  const float2 f01 = e4m3x2_to_f2(h01), f23 = e4m3x2_to_f2(h23);
  const uint32_t l01 = e4m3x2(a - f01.x, b - f01.y), l23 = e4m3x2(c - f23.x, d - f23.y);
  hi = h01 | (h23 << 16);
  lo = l01 | (l23 << 16);
}

}  // namespace tc
}  // namespace pgqa
