// sparse_tc.cu -- tcgen05 (TMEM) kernel for sparse paged GQA attention: each (token, kv head)
// attends a listed subset of its sequence's keys, shared by the kv head's query heads
// ("Tune sparse GQA prefill profile on gfx942 and gfx950": ~2k selected tokens per row,
// head_dim 256, FP8 K/V, TP1-TP8 head layouts).
//
// A unit is (token t, kv head, up to 16 of its q heads): 16 query rows (padded) with one key
// list. One unit's rows are too few for a tensor-core tile, so four units share one:
//
//   * a tile holds 32 listed keys of each of 4 units (128 keys, the MMA's M, swap-AB) and the
//     4 x 16 query rows (N = 64; bf16 Q split once per quad into e4m3 hi + lo, stacked as
//     one N = 128 operand, as in the verify kernel), so S = K [Q_hi; Q_lo]^T is 8
//     kind::f8f6f4 MMAs per tile and O^T += V^T [P_hi; P_lo]^T another 8;
//   * only the diagonal blocks mean anything: unit u's keys against unit u's rows. The
//     softmax reads only those scores, and P^T is block-diagonal: the P buffers are zeroed
//     once and only diagonal entries are ever written, so each unit's O^T columns collect
//     only its own keys;
//   * the listed K/V rows are gathered by 16-byte cp.async copies (the list scatters them,
//     so no TMA box fits; gather4 would move 512 B per instruction) into the same
//     128B-swizzled stages the TMA fills in the verify kernel; a listed position goes
//     through the block table like a dense key; unused entries (padding, past the causal
//     limit, a bad page) get a zero V row and a cleared validity bit;
//   * softmax: warp w reads TMEM lane quarter u = w % 4, i.e. unit u's 32 keys of the tile,
//     and 4 of that unit's 16 rows, so a row's maximum over the tile's keys is a warp-level
//     reduction. The lazy rescale (reference moved only when a score exceeds it by 2^4) is
//     voted by the four warps that share a row subgroup, because a row's O^T columns span
//     all four lane quarters (d);
//   * persistent CTAs walk a contiguous range of quads (4 consecutive units); every unit
//     has the same number of tiles (the list length), so there is no split and no merge.
//
// Warp roles (768 threads): warp 0 = S issuer (+ TMEM owner), warp 1 = P.V issuer, warps
// 4-19 = softmax and epilogue, warps 20-21 = K gatherers, warps 22, 23, 2, 3 = V gatherers
// (V stages are held until P.V completes, so V gets more warps and stages).
// Shared memory: Q hi/lo 32 KB, 2 K + 3 V stages of 32 KB, two block-diagonal P buffers of
// 16 KB (227 KB in all).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdio>

#include "common.cuh"
#include "device_util.cuh"
#include "plan.cuh"
#include "tc_kernels.cuh"
#include "tc_util.cuh"

namespace pgqa {

namespace {

using namespace tc;

constexpr int kUnitRows = 16;                  // query rows of a unit
constexpr int kQuad = 4;                       // units per tile
constexpr int kRows = kQuad * kUnitRows;       // 64: the MMA N of one Q / P part
constexpr int kUnitKeys = kTileKeys / kQuad;   // 32 keys of each unit per tile
constexpr int kThreads = 768;
// Every warp keeps the launch's 80 registers a thread (no warpgroup register split).
constexpr int kSoftWarps = 16;
constexpr int kSoftThreads = kSoftWarps * 32;
constexpr int kSoftWarp0 = 4;
constexpr int kQChunks = kRows * 16 / kSoftThreads;  // Q chunks of 16 elements per softmax thread
static_assert(kQChunks * kSoftThreads == kRows * 16, "Q chunks");
constexpr int kKStages = 2, kVStages = 3, kPBufs = 2;
constexpr float kTau = 4.f, kSigma = 4.f, kMInit = -1.0e30f;

constexpr uint32_t kQHalf = 2 * kRows * 128;   // [Q_hi 64 rows | Q_lo 64 rows] x 128 B
constexpr uint32_t kKVHalf = kTileKeys * 128;
constexpr uint32_t kKVTile = 2 * kKVHalf;
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kOffQ + 2 * kQHalf;
constexpr uint32_t kOffV = kOffK + kKStages * kKVTile;
constexpr uint32_t kOffP = kOffV + kVStages * kKVTile;  // [128 keys][P_hi 64 B | P_lo 64 B]
constexpr uint32_t kPBuf = kTileKeys * 128;
constexpr uint32_t kOffMisc = kOffP + kPBufs * kPBuf;

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;    // 2 S buffers [S_hi | S_lo] of 128 columns
constexpr uint32_t kColO = 256;  // O^T d-half h: [O_hi | O_lo] at 256 + 128 h
constexpr uint32_t kIdescS = idesc_e4m3(128, 2 * kRows, false, false);  // K (K-major) x [Q_hi; Q_lo]
constexpr uint32_t kIdescO = idesc_e4m3(128, 2 * kRows, true, true);    // V^T (MN) x [P_hi; P_lo]^T (MN)

struct UnitInfo {
  int t, head0, rows, ok;
};

struct Misc {
  alignas(16) float alpha[kRows];
  alignas(16) float lsum[kRows];
  alignas(16) long long out_off[2][kRows];  // [quad parity][row]; -1: not a real row
  alignas(16) UnitInfo unit[2][kQuad];
  alignas(16) float amax[kSoftWarps];
  alignas(16) uint32_t vval[kVStages][kQuad];  // validity bits of the V stage's keys, per unit
  alignas(8) uint64_t k_full[kKStages], k_empty[kKStages], v_full[kVStages], v_empty[kVStages];
  uint64_t s_full[2], s_free[2];
  uint64_t p_full[kPBufs], pv_done[kPBufs], q_full, q_free, o_ready, o_free, drain[2];
  uint64_t never;  // no thread ever arrives (the failure-path test waits on it)
  float qscale[2];
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(offsetof(Misc, alpha) % 16 == 0 && offsetof(Misc, k_full) % 8 == 0, "Misc alignment");
constexpr size_t kSmemBytes = kOffMisc + sizeof(Misc) + 1024;
static_assert(kSmemBytes <= 232448, "fits the 227 KB of dynamic shared memory a CTA may use");

// A unit's token, kv head, first q head and rows, its sequence and causal limit. Called by a
// whole converged warp (the sequence search is warp-cooperative); every lane gets the result.
struct Unit {
  int t, kvh, head0, rows, s, lim, ok;
};
__device__ __forceinline__ Unit unit_info(const SparseArgs& a, long long u, int lane) {
  Unit r;
  const long long units = (long long)a.T * a.Hkv * a.HG;
  if (u >= units) {
    r.t = r.kvh = r.head0 = r.rows = r.s = 0;
    r.lim = -1;
    r.ok = 0;
    return r;
  }
  const int hg = (int)(u % a.HG);
  r.kvh = (int)((u / a.HG) % a.Hkv);
  r.t = (int)(u / ((long long)a.HG * a.Hkv));
  r.head0 = r.kvh * a.G + hg * kUnitRows;
  r.rows = min(kUnitRows, a.G - hg * kUnitRows);
  r.s = seq_of_token(a.qsl, a.num_seqs, r.t, lane);
  const int q0 = __ldg(a.qsl + r.s), q1 = __ldg(a.qsl + r.s + 1), L = __ldg(a.seq_lens + r.s);
  const int qn = q1 - q0;
  r.ok = r.t >= q0 && r.t < q1 && qn <= L;
  r.lim = L - qn + (r.t - q0);
  return r;
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait0() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void st_shared_zero16(uint32_t dst) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(dst), "r"(0) : "memory");
}

// 32 lanes x 32 bit, 4 consecutive columns -> 4 registers.
__device__ __forceinline__ void tmem_ld4(uint32_t taddr, float (&v)[4]) {
  uint32_t r[4];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 4; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_st4(uint32_t taddr, const float (&v)[4]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};" ::"r"(taddr),
               "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
               "r"(__float_as_uint(v[3]))
               : "memory");
}

__device__ __forceinline__ float2 bf2(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// 64-bit shuffle of a row offset (-1: unused key).
__device__ __forceinline__ long long shfl_off(long long v, int src) {
  const int lo = __shfl_sync(0xffffffffu, (int)(v & 0xffffffff), src);
  const int hi = __shfl_sync(0xffffffffu, (int)(v >> 32), src);
  return ((long long)hi << 32) | (unsigned)lo;
}

}  // namespace

__global__ void __launch_bounds__(kThreads, 1) sparse_tc_kernel(SparseArgs a, int stall_test_ns) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Misc& ms = *reinterpret_cast<Misc*>(smem + kOffMisc);
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_flag = &ms.abort_flag;
  auto bar = [&](const uint64_t& b) { return smem_u32(&b); };

  const long long units = (long long)a.T * a.Hkv * a.HG;
  const long long quads = (units + kQuad - 1) / kQuad;
  const long long quad_begin = (long long)blockIdx.x * quads / gridDim.x;
  const long long quad_end = (long long)(blockIdx.x + 1) * quads / gridDim.x;
  const int NT = (a.K + kUnitKeys - 1) / kUnitKeys;  // tiles per quad (>= 1 on this path)
  if (quad_begin >= quad_end) return;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(bar(ms.k_full[s]), 2);  // the K team's warps
      mbar_init(bar(ms.k_empty[s]), 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(bar(ms.v_full[s]), 4);  // the V team's warps
      mbar_init(bar(ms.v_empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(ms.s_full[b]), 1);
      mbar_init(bar(ms.s_free[b]), kSoftWarps);
    }
    for (int b = 0; b < kPBufs; ++b) {
      mbar_init(bar(ms.p_full[b]), kSoftWarps);
      mbar_init(bar(ms.pv_done[b]), 1);
    }
    mbar_init(bar(ms.q_full), kSoftWarps);
    mbar_init(bar(ms.q_free), 1);
    mbar_init(bar(ms.o_ready), 1);
    mbar_init(bar(ms.o_free), kSoftWarps);
    mbar_init(bar(ms.drain[0]), 1);
    mbar_init(bar(ms.drain[1]), 1);
    mbar_init(bar(ms.never), 1);
    ms.abort_flag = 0;
    fence_mbar_init();
  }
  // P buffers: zero once; the softmax only ever writes the diagonal blocks
  for (uint32_t o = threadIdx.x * 16; o < kPBufs * kPBuf; o += kThreads * 16) st_shared_zero16(sbase + kOffP + o);
  fence_proxy_async_smem();
  if (warp == 0) {
    tmem_alloc(smem_u32(&ms.tmem_base), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ms.tmem_base;

  const int wg = warp >> 2;
  if (wg >= 1 && wg <= 4) {
    // ------------------------------------------------------------ softmax + epilogue
    const int sw = warp - kSoftWarp0;         // 0..15
    const int gi = sw * 32 + lane;            // 0..511
    const int u = warp & 3;                   // unit of the quad = TMEM lane quarter
    const int j4 = sw >> 2;                   // row subgroup: rows 16u + 4 j4 .. + 3
    const int row0 = kUnitRows * u + 4 * j4;  // first row (column of S / P^T) this warp owns
    const int group_bar = 3 + j4;             // the four warps (one per unit) of subgroup j4
    const int key = kUnitKeys * u + lane;     // tile-local key = TMEM lane of S
    const uint32_t lane_addr = (uint32_t)(u * 32) << 16;
    bool stalled = false;
    if (stall_test_ns) {
      int ok = 1;
      if (lane == 0) ok = mbar_wait(bar(ms.never), 0, abort_flag, a.err, (uint64_t)stall_test_ns);
      stalled = __shfl_sync(0xffffffffu, ok, 0) == 0;
    }
    if (!stalled) {
    float m[4], mo[4], l[4];

    auto q_prep = [&](long long qi, int ii) {
      const int pi = ii & 1;
      if (ii >= 1) mbar_wait_warp(bar(ms.q_free), (ii - 1) & 1, abort_flag, a.err, lane);
      if (sw < kQuad) {  // one warp per unit of the quad
        const Unit U = unit_info(a, qi * kQuad + sw, lane);
        if (lane == 0) {
          ms.unit[pi][sw] = UnitInfo{U.t, U.head0, U.rows, U.ok};
          if (U.rows > 0 && !U.ok) atomicOr(a.err, kErrBounds);
        }
      }
      named_barrier(1, kSoftThreads);
      if (gi < kRows) {
        const UnitInfo& U = ms.unit[pi][gi / kUnitRows];
        const int r = gi % kUnitRows;
        ms.out_off[pi][gi] = r < U.rows ? (long long)U.t * a.o_st + (long long)(U.head0 + r) * a.o_sh : -1;
      }
      // 64 rows x 16 chunks of 16 elements; thread gi takes chunks gi + kSoftThreads k
      uint4 v[kQChunks][2];
      float amax = 0.f;
#pragma unroll
      for (int k = 0; k < kQChunks; ++k) {
        const int c = gi + k * kSoftThreads, rr = c >> 4, ch = c & 15;
        const UnitInfo& U = ms.unit[pi][rr / kUnitRows];
        const int r = rr % kUnitRows;
        if (r < U.rows) {
          const uint4* s = reinterpret_cast<const uint4*>(a.q + (long long)U.t * a.q_st +
                                                          (long long)(U.head0 + r) * a.q_sh + ch * 16);
          v[k][0] = __ldg(s);
          v[k][1] = __ldg(s + 1);
        } else {
          v[k][0] = v[k][1] = make_uint4(0, 0, 0, 0);
        }
        const uint32_t w[8] = {v[k][0].x, v[k][0].y, v[k][0].z, v[k][0].w, v[k][1].x, v[k][1].y, v[k][1].z, v[k][1].w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float2 f = bf2(w[i]);
          amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
        }
      }
      amax = warp_max(amax);
      if (lane == 0) ms.amax[sw] = amax;
      named_barrier(1, kSoftThreads);
      amax = 0.f;
#pragma unroll
      for (int w = 0; w < kSoftWarps; ++w) amax = fmaxf(amax, ms.amax[w]);
      // 2^sig * amax in [128, 256): exponent arithmetic on the bits
      int sig = 0;
      if (amax > 0.f && isfinite(amax)) sig = 7 - (int)((__float_as_uint(amax) >> 23) & 0xff) + 127;
      sig = max(-100, min(100, sig));
      const float scale = ldexpf(1.f, sig);
#pragma unroll
      for (int k = 0; k < kQChunks; ++k) {
        const int c = gi + k * kSoftThreads, rr = c >> 4, ch = c & 15;
        const uint32_t w[8] = {v[k][0].x, v[k][0].y, v[k][0].z, v[k][0].w, v[k][1].x, v[k][1].y, v[k][1].z, v[k][1].w};
        uint32_t hw[4], lw[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 f0 = bf2(w[2 * i]), f1 = bf2(w[2 * i + 1]);
          split4(f0.x * scale, f0.y * scale, f1.x * scale, f1.y * scale, hw[i], lw[i]);
        }
        // part 0 = hi rows 0..63, part 1 = lo rows 64..127 of the stacked operand
        const int h = ch >> 3, cc = ch & 7;
        const int rhi = rr, rlo = kRows + rr;
        *reinterpret_cast<uint4*>(smem + kOffQ + h * kQHalf + rhi * 128 + ((cc ^ (rhi & 7)) << 4)) =
            make_uint4(hw[0], hw[1], hw[2], hw[3]);
        *reinterpret_cast<uint4*>(smem + kOffQ + h * kQHalf + rlo * 128 + ((cc ^ (rlo & 7)) << 4)) =
            make_uint4(lw[0], lw[1], lw[2], lw[3]);
      }
      if (gi == 0) ms.qscale[pi] = ldexpf(1.f, -sig);
      fence_proxy_async_smem();
      mbar_arrive_warp(bar(ms.q_full), lane);
    };

    int ii = 0;
    uint32_t g = 0;
    q_prep(quad_begin, 0);
    for (long long qi = quad_begin; qi < quad_end; ++qi, ++ii) {
      const int pi = ii & 1;
      named_barrier(1, kSoftThreads);  // q_prep's shared writes (unit info, qscale) are visible
      const float c = a.score_scale_log2 * ms.qscale[pi];
      // this warp's rows: real rows start at an unknown reference, padding rows at 0 (finite,
      // so their discarded scores never vote)
      const int urows = ms.unit[pi][u].rows;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        m[i] = 4 * j4 + i < urows ? kMInit : 0.f;
        mo[i] = kSigma - m[i];
        l[i] = 0.f;
      }
      // A failed wait (timeout or abort) does not leave the loops: every later wait then
      // fails fast, so all softmax warps still pass the same barriers and finish.
      for (int j = 0; j < NT; ++j, ++g) {
        const int b = g & 1;
        const uint32_t vst = g % kVStages;
        float sh[4], sl[4], s[4], x[4];
        mbar_wait_warp(bar(ms.s_full[b]), (g >> 1) & 1, abort_flag, a.err, lane);
        mbar_wait_warp(bar(ms.v_full[vst]), (g / kVStages) & 1, abort_flag, a.err, lane);  // the keys' validity bits
        tc_fence_after();
        tmem_ld4(tmem + lane_addr + kColS + b * 128 + row0, sh);
        tmem_ld4(tmem + lane_addr + kColS + b * 128 + kRows + row0, sl);
        tmem_wait_ld();
        const bool valid = (ms.vval[vst][u] >> lane) & 1u;
        bool need = false;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          s[i] = sh[i] + sl[i];
          x[i] = valid ? fmaf(s[i], c, mo[i]) : -INFINITY;
          need |= x[i] > kTau + kSigma;
        }
        // the subgroup's four warps vote (a row's O^T columns span all four lane quarters)
        const bool rescale = barrier_or(group_bar, 128, need);
        if (rescale) {
          // exact tile maximum of s c per row: the row's keys are this warp's 32 lanes
          float alpha[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float tm = warp_max(valid ? s[i] * c : -INFINITY);
            const float mn = fmaxf(m[i], tm);
            alpha[i] = ex2(m[i] - mn);
            m[i] = mn;
            mo[i] = kSigma - mn;
            l[i] *= alpha[i];
            x[i] = valid ? fmaf(s[i], c, mo[i]) : -INFINITY;
          }
          if (lane < 4) ms.alpha[row0 + lane] = lane == 0 ? alpha[0] : lane == 1 ? alpha[1] : lane == 2 ? alpha[2] : alpha[3];
          named_barrier(group_bar, 128);
        }
        tc_fence_before();
        mbar_arrive_warp(bar(ms.s_free[b]), lane);
        // P = 2^x in f16, split into e4m3 hi + lo (this key, 4 rows); row sums in fp32
        uint32_t ph, pl;
        __half2 s01, s23;
        p_split4_f16(x[0], x[1], x[2], x[3], ph, pl, s01, s23);
        {
          const float2 f01 = __half22float2(s01), f23 = __half22float2(s23);
          l[0] += f01.x;
          l[1] += f01.y;
          l[2] += f23.x;
          l[3] += f23.y;
        }
        // P buffer g & 1 is free once P.V(g-2) has completed; O^T may be rescaled once
        // P.V(g-1) has.
        if (g >= 2) mbar_wait_warp(bar(ms.pv_done[g & 1]), ((g >> 1) - 1) & 1, abort_flag, a.err, lane);
        if (rescale && j > 0) mbar_wait_warp(bar(ms.pv_done[(g - 1) & 1]), ((g - 1) >> 1) & 1, abort_flag, a.err, lane);
        tc_fence_after();
        if (rescale && j > 0) {
          // O^T columns of the subgroup's 16 rows (4 of each unit), both d-halves and parts
#pragma unroll 1
          for (int hp = 0; hp < 4; ++hp) {
#pragma unroll 1
            for (int v = 0; v < kQuad; ++v) {
              float o[4];
              const int r0 = kUnitRows * v + 4 * j4;
              const uint32_t ad = tmem + lane_addr + kColO + (hp >> 1) * 128 + (hp & 1) * kRows + r0;
              tmem_ld4(ad, o);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 4; ++i) o[i] *= ms.alpha[r0 + i];
              tmem_st4(ad, o);
            }
          }
          tmem_wait_st();
        }
        // P^T row of this key: bytes (rows) row0 .. row0 + 3 of P_hi (chunk u) and of P_lo
        // (chunk 4 + u), 128-byte swizzle
        {
          uint8_t* prow = smem + kOffP + (g & 1) * kPBuf + key * 128;
          *reinterpret_cast<uint32_t*>(prow + ((u ^ (key & 7)) << 4) + 4 * j4) = ph;
          *reinterpret_cast<uint32_t*>(prow + (((4 + u) ^ (key & 7)) << 4) + 4 * j4) = pl;
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive_warp(bar(ms.p_full[g & 1]), lane);
      }
      // Q of the next quad while this quad's last P.V runs
      if (qi + 1 < quad_end) q_prep(qi + 1, ii + 1);

      // ---------------------------------------------------------- epilogue
      mbar_wait_warp(bar(ms.o_ready), ii & 1, abort_flag, a.err, lane);
      tc_fence_after();
      // row sums over this warp's 32 keys, then 1 / l per row
#pragma unroll
      for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) l[i] += __shfl_xor_sync(0xffffffffu, l[i], o);
      }
      if (lane < 4) ms.lsum[row0 + lane] = lane == 0 ? l[0] : lane == 1 ? l[1] : lane == 2 ? l[2] : l[3];
      named_barrier(1, kSoftThreads);
      // thread (lane quarter u, lane) writes d = 32 u + lane of both halves for the
      // subgroup's 16 rows
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
#pragma unroll 1
        for (int v = 0; v < kQuad; ++v) {
          float oh[4], ol[4];
          const int r0 = kUnitRows * v + 4 * j4;
          tmem_ld4(tmem + lane_addr + kColO + h * 128 + r0, oh);
          tmem_ld4(tmem + lane_addr + kColO + h * 128 + kRows + r0, ol);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const long long off = ms.out_off[pi][r0 + i];
            if (off >= 0) {
              const float lr = ms.lsum[r0 + i];
              const float inv = lr > 0.f ? __fdividef(a.out_scale, lr) : 0.f;
              reinterpret_cast<__nv_bfloat16*>(a.out)[off + h * 128 + 32 * u + lane] =
                  __float2bfloat16_rn((oh[i] + ol[i]) * inv);
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive_warp(bar(ms.o_free), lane);
    }
    }  // !stalled
  } else {
    const int kt = warp == 20 ? 0 : warp == 21 ? 1 : -1;                               // K team member
    const int vt = warp == 22 ? 0 : warp == 23 ? 1 : warp == 2 ? 2 : warp == 3 ? 3 : -1;  // V team member
    if (kt >= 0 || vt >= 0) {
      // ------------------------------------------------------------ gatherers (K, V)
      // Two teams walk every tile in order: the K team (2 warps, two units each) and the V
      // team (4 warps, one unit each). Per tile, lane l looks up entry j * 32 + l of the
      // warp's units (the list, then the block table); each group of 16 keys is copied with
      // lane pair (2k, 2k + 1) owning key k: one shuffle for the row offset, then 8 cp.async
      // of 16 bytes per lane, a warp instruction moving 32 contiguous bytes of each of 16
      // rows. A tile is published once the warp has issued the next one (two tiles in
      // flight per warp): wait for all but the newest copy group, make the copies visible to
      // the tensor core (proxy fence), arrive once on the stage's full barrier. The next
      // tile's lookups are in flight while the copies run.
      const bool is_k = kt >= 0;
      const int nu = is_k ? 2 : 1;              // units this warp copies per tile
      const int u0 = is_k ? 2 * kt : vt;        // its first unit
      const int nst = is_k ? kKStages : kVStages;
      const uint8_t* base = is_k ? a.k : a.v;
      const uint32_t region = sbase + (is_k ? kOffK : kOffV);
      uint64_t* full = is_k ? ms.k_full : ms.v_full;
      uint64_t* empty = is_k ? ms.k_empty : ms.v_empty;
      const int pmask = a.P - 1;
      const long long total = (quad_end - quad_begin) * NT;  // tiles of this CTA
      Unit U[2];
      long long uq = -1;  // quad whose units U holds
      auto load_units = [&](long long qi) {
        if (qi == uq) return;
        U[0] = unit_info(a, qi * kQuad + u0, lane);
        if (is_k) U[1] = unit_info(a, qi * kQuad + u0 + 1, lane);
        uq = qi;
      };
      // list entries of tile g (lane l: entry j * 32 + l of each unit), -1 past the list
      auto entries = [&](long long g, int (&e)[2]) {
        load_units(quad_begin + g / NT);
        const int i = (int)(g % NT) * kUnitKeys + lane;
#pragma unroll
        for (int v = 0; v < 2; ++v)
          e[v] = (v < nu && U[v].ok && i < a.K)
                     ? __ldg(a.idx + (long long)U[v].t * a.idx_st + (long long)U[v].kvh * a.idx_sh + i)
                     : -1;
      };
      auto pages = [&](const int (&e)[2], int (&pg)[2]) {
#pragma unroll
        for (int v = 0; v < 2; ++v)
          pg[v] = (e[v] >= 0 && e[v] <= U[v].lim && (e[v] >> a.p_shift) < a.W)
                      ? __ldg(a.bt + (long long)U[v].s * a.bt_stride + (e[v] >> a.p_shift))
                      : -1;
      };
      // byte offset of each entry's row for its unit's kv head, or -1 (unused: padding, past
      // the causal limit; a listed position past W * P or a bad page also sets the error word)
      auto offsets = [&](const int (&e)[2], const int (&pg)[2], long long (&o)[2]) {
#pragma unroll
        for (int v = 0; v < 2; ++v) {
          o[v] = -1;
          if (e[v] < 0 || e[v] > U[v].lim) continue;
          if ((e[v] >> a.p_shift) >= a.W) {
            if (is_k) atomicOr(a.err, kErrBounds);
            continue;
          }
          if (pg[v] < 0 || pg[v] >= a.NB) {
            if (is_k) atomicOr(a.err, kErrPage);
            continue;
          }
          o[v] = (long long)pg[v] * a.kv_sb + (long long)(e[v] & pmask) * a.kv_sp + (long long)U[v].kvh * a.kv_sh;
        }
      };
      long long o[2] = {-1, -1};
      if (total > 0) {
        int e[2], pg[2];
        entries(0, e);
        pages(e, pg);
        offsets(e, pg, o);
      }
      const int half_lane = lane >> 1, par = lane & 1;
      int pending = -1;  // stage whose copies are issued but not yet published
      for (long long g = 0; g < total; ++g) {
        // the lookups of the next tile: entries now, pages after the copies are issued
        int e[2], pg[2];
        const bool more = g + 1 < total;
        const long long next_q = more ? quad_begin + (g + 1) / NT : -1;
        if (more && next_q == uq) entries(g + 1, e);  // (a new quad's units are loaded after the copies)
        const uint32_t st = (uint32_t)(g % nst);
        int ok = 1;
        if (lane == 0) ok = mbar_wait(bar(empty[st]), (uint32_t)((g / nst) & 1) ^ 1u, abort_flag, a.err);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        const uint32_t stage = region + st * kKVTile;
#pragma unroll
        for (int v = 0; v < 2; ++v) {
          if (v >= nu) break;
#pragma unroll
          for (int h = 0; h < 2; ++h) {                       // two groups of 16 keys per unit
            const int key = kUnitKeys * (u0 + v) + 16 * h + half_lane;  // tile-local key of this lane pair
            const long long off = shfl_off(o[v], 16 * h + half_lane);
            const uint32_t row = stage + key * 128;
            const int sw = key & 7;
            if (off >= 0) {
              const uint8_t* gsrc = base + off + par * 16;
#pragma unroll
              for (int m = 0; m < 8; ++m)  // chunk c = 2m + par: half c >> 3, 16-byte slot c & 7
                cp_async16(row + (m >> 2) * kKVHalf + ((((2 * m + par) & 7) ^ sw) << 4), gsrc + m * 32);
            } else if (!is_k) {
#pragma unroll
              for (int m = 0; m < 8; ++m)  // an unused key's V row: zeros (0 x stale data could be NaN)
                st_shared_zero16(row + (m >> 2) * kKVHalf + ((((2 * m + par) & 7) ^ sw) << 4));
            }
          }
        }
        cp_async_commit();
        if (!is_k) {
          const uint32_t bits = __ballot_sync(0xffffffffu, o[0] >= 0);
          if (lane == 0) ms.vval[st][vt] = bits;
        }
        if (pending >= 0) {
          cp_async_wait1();  // the previous tile's copies have landed
          fence_proxy_async_smem();
          mbar_arrive_warp(bar(full[pending]), lane);
        }
        pending = (int)st;
        if (more) {
          if (next_q != uq) entries(g + 1, e);
          pages(e, pg);
          offsets(e, pg, o);
        }
      }
      // Every issued copy has landed before the last tile is published and before the CTA
      // may exit (also after an abort).
      cp_async_wait0();
      if (pending >= 0) {
        fence_proxy_async_smem();
        mbar_arrive_warp(bar(full[pending]), lane);
      }
      __syncwarp();
    } else if (warp == 0 || warp == 1) {
      // ------------------------------------------------------------ MMA issuers
      if (lane == 0) {
        const bool is_s = warp == 0;
        uint32_t g = 0;
        int ii = 0;
        bool ok = true;
        for (long long qi = quad_begin; qi < quad_end && ok; ++qi, ++ii) {
          for (int j = 0; j < NT && ok; ++j, ++g) {
            if (is_s) {
              if (j == 0 && !(ok = mbar_wait(bar(ms.q_full), ii & 1, abort_flag, a.err))) break;
              const uint32_t st = g % kKStages, b = g & 1;
              if (!(ok = mbar_wait(bar(ms.k_full[st]), (g / kKStages) & 1, abort_flag, a.err))) break;
              if (g >= 2 && !(ok = mbar_wait(bar(ms.s_free[b]), ((g >> 1) - 1) & 1, abort_flag, a.err))) break;
              tc_fence_after();
              const uint64_t a0 = smem_desc(sbase + kOffK + st * kKVTile, 16, 1024, kSw128);
              const uint64_t b0 = smem_desc(sbase + kOffQ, 16, 1024, kSw128);
#pragma unroll
              for (int kb = 0; kb < 8; ++kb) {
                const uint32_t off = (kb >> 2) * kKVHalf + (kb & 3) * 32, qoff = (kb >> 2) * kQHalf + (kb & 3) * 32;
                mma_e4m3(tmem + kColS + b * 128, a0 + (off >> 4), b0 + (qoff >> 4), kIdescS, kb ? 1u : 0u);
              }
              mma_commit(bar(ms.s_full[b]));
              mma_commit(bar(ms.k_empty[st]));
              if (j == NT - 1) mma_commit(bar(ms.q_free));
            } else {
              // the first P.V of a quad overwrites O^T: the previous epilogue must be done
              if (j == 0 && ii >= 1 && !(ok = mbar_wait(bar(ms.o_free), (ii - 1) & 1, abort_flag, a.err))) break;
              if (!(ok = mbar_wait(bar(ms.p_full[g & 1]), (g >> 1) & 1, abort_flag, a.err))) break;
              const uint32_t st = g % kVStages;
              if (!(ok = mbar_wait(bar(ms.v_full[st]), (g / kVStages) & 1, abort_flag, a.err))) break;
              tc_fence_after();
              const uint64_t a0 = smem_desc(sbase + kOffV + st * kKVTile, 1024, 1024, kSw128);
              const uint64_t b0 = smem_desc(sbase + kOffP + (g & 1) * kPBuf, 1024, 1024, kSw128);
#pragma unroll
              for (int h = 0; h < 2; ++h) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                  const uint32_t off = h * kKVHalf + kk * 4096, poff = kk * 4096;
                  mma_e4m3(tmem + kColO + h * 128, a0 + (off >> 4), b0 + (poff >> 4), kIdescO,
                           (j == 0 && kk == 0) ? 0u : 1u);
                }
              }
              mma_commit(bar(ms.v_empty[st]));
              mma_commit(bar(ms.pv_done[g & 1]));
              if (j == NT - 1) mma_commit(bar(ms.o_ready));
            }
          }
        }
        // Every MMA this thread issued has completed before the CTA may release TMEM.
        uint64_t& drain = is_s ? ms.drain[0] : ms.drain[1];
        mma_commit(bar(drain));
        mbar_drain(bar(drain), 0, abort_flag, a.err);
      }
      __syncwarp();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Units per tile-sharing group and the list length below which the warp-level kernel is
// used instead (a tile holds 32 keys of each unit).
int sparse_tc_min_keys() { return 2 * kUnitKeys; }

int launch_sparse_tc(const SparseArgs& a, int sms, uint32_t stall_test_ns, cudaStream_t stream) {
  const long long units = (long long)a.T * a.Hkv * a.HG;
  if (units == 0 || a.K < sparse_tc_min_keys()) return 0;
  const long long quads = (units + kQuad - 1) / kQuad;
  const int grid = (int)(quads < sms ? quads : sms);
  static int attr_done[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  cudaError_t e;
  if (dev >= 0 && dev < 64 && !attr_done[dev]) {
    e = cudaFuncSetAttribute(sparse_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) {
      char buf[160];
      snprintf(buf, sizeof buf, "cudaFuncSetAttribute(sparse): %s", cudaGetErrorString(e));
      set_tc_error(buf);
      return -1;
    }
    attr_done[dev] = 1;
  }
  sparse_tc_kernel<<<grid, kThreads, kSmemBytes, stream>>>(a, (int)stall_test_ns);
  e = cudaGetLastError();
  if (e != cudaSuccess) {
    char buf[160];
    snprintf(buf, sizeof buf, "sparse kernel launch: %s", cudaGetErrorString(e));
    set_tc_error(buf);
    return -1;
  }
  return 1;
}

}  // namespace pgqa
