// device_util.cuh -- small device helpers shared by the attention kernels.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include "common.cuh"

namespace pgqa {

// Row r of a (sequence, kv head) is query token r / G and head kvh*G + r % G.
struct RowMap {
  int t, h;
};
__device__ __forceinline__ RowMap map_row(int r, int G, int kvh) {
  RowMap m;
  m.t = r / G;
  m.h = kvh * G + (r - m.t * G);
  return m;
}

// Two e4m3 codes (low byte = first) -> two floats, exact (the f16 conversion of an
// e4m3 value is exact, as is f16 -> f32).
__device__ __forceinline__ float2 e4m3x2_to_float2(uint16_t v) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(v));
  __half2 h = *reinterpret_cast<__half2*>(&h2);
  return __half22float2(h);
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float((uint32_t)b << 16);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ void named_barrier(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Named barrier that also returns whether `pred` holds for any participating thread.
__device__ __forceinline__ bool barrier_or(int id, int nthreads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n barrier.red.or.pred q, %2, %3, p;\n selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ float2 unpack_f16x2(uint32_t v) {
  return __half22float2(*reinterpret_cast<const __half2*>(&v));
}

// Partial result slot of (block, split): f16 rows of O / l in cache-code units.
__device__ __forceinline__ uint16_t* slot_o(const ClassPlan& cp, int slot) {
  return cp.part_o + (size_t)slot * cp.slot_rows * kHeadDim;
}
__device__ __forceinline__ float* slot_lse(const ClassPlan& cp, int slot) {
  return cp.part_lse + (size_t)slot * cp.slot_rows;
}

// The sequence of token t: the last s in [0, n) with qsl[s] <= t (0 if none), found by a
// 32-way search: each step the warp probes 32 points of the remaining interval at once, so
// a batch of n sequences takes about log32(n) dependent loads. Every lane gets the answer;
// the warp must be converged. A query_start_loc that is not monotone still yields an index
// in [0, n); the caller's range check on the token then flags it.
__device__ __forceinline__ int seq_of_token(const int32_t* qsl, int n, int t, int lane) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int span = hi - lo;
    const int p = lo + (int)(((long long)(lane + 1) * span + 31) / 32);  // in (lo, hi]; lane 31: hi
    const unsigned m = __ballot_sync(0xffffffffu, __ldg(qsl + p) <= t);
    if (m == 0) {
      hi = __shfl_sync(0xffffffffu, p, 0) - 1;
    } else {
      const int k = 31 - __clz((int)m);  // the last probe at or below t
      lo = __shfl_sync(0xffffffffu, p, k);
      if (k < 31) hi = min(hi, __shfl_sync(0xffffffffu, p, k + 1) - 1);
    }
  }
  return lo;
}

constexpr int kMergeMaxSplits = 16;  // pieces whose weights fit the shared scratch

// This call's 48-bit tag for the split counters: the workspace's epoch word (advanced by
// the plan kernel once per call, after every kernel of the call that reads it has read it)
// mixed with the host's nonzero per-call value. A constant fill of the workspace never
// carries it (the mix of a nonzero value with an odd constant is nonzero below bit 48), and
// leftover bytes of other data carry it with probability 2^-48 per counter.
__device__ __forceinline__ unsigned long long split_tag(const Problem& p, const ClassPlan& cp) {
  return (__ldcg(cp.epoch) ^ ((unsigned long long)p.call_tag * 0x9E3779B97F4A7C15ull)) & kSplitTagMask;
}

// Acquire-release fence at GPU scope: around a relaxed atomic, it makes the atomic a release
// of this thread's earlier writes (for the pieces that arrive at a split counter) and an
// acquire of the other pieces' partials (for the last one). A plain message-passing pattern,
// so no sequentially consistent fence is needed.
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

// One piece of a split block has stored its partial; true for the block's last piece. The
// counter word holds (tag << 16) | arrivals (nsplit < 2^16); a word with another tag counts
// as no arrivals. The CAS loop retries only while other pieces of the block arrive.
// split_peek reads the word for split_arrive_from, so that its round trip can overlap the
// wait for the piece's partial; split_arrive reads it itself.
__device__ __forceinline__ unsigned long long split_peek(const unsigned long long* counter) {
  return *reinterpret_cast<const volatile unsigned long long*>(counter);
}
__device__ __forceinline__ bool split_arrive_from(unsigned long long* counter, unsigned long long old, int nsplit,
                                                  unsigned long long tag) {
  for (;;) {
    const unsigned arrived = (old >> 16) == tag ? (unsigned)(old & 0xffffu) : 0u;
    const unsigned long long want = (tag << 16) | (arrived + 1u);
    const unsigned long long seen = atomicCAS(counter, old, want);
    if (seen == old) return arrived + 1u == (unsigned)nsplit;
    old = seen;
  }
}
__device__ __forceinline__ bool split_arrive(unsigned long long* counter, int nsplit, unsigned long long tag) {
  return split_arrive_from(counter, split_peek(counter), nsplit, tag);
}

// Called by `nthreads` threads (ids tid = 0..nthreads-1) that share barrier `bar_id`,
// after each has written its share of this piece's partial result (normalised O in f16
// code units and log2-sum-exp per row) and executed __threadfence(). The last piece of a
// block to arrive merges all pieces of the block:
//     M = max_i lse_i,  w_i = 2^(lse_i - M) / sum_j 2^(lse_j - M),
//     out = v_descale * sum_i w_i o_i
// ("Optimize Qwen3.5 MTP unified attention on gfx950": split-KV segments reduced by
// a second pass). s_w is shared scratch of kMergeMaxSplits * kSlotRows floats.
// Returns after the merge (if any) is complete.
__device__ inline void merge_split_block(const Problem& p, const Pointers& ptr, const ClassPlan& cp,
                                         const RowBlock& rb, int tid, int nthreads, int bar_id, float* s_w);

__device__ inline void finish_split_block(const Problem& p, const Pointers& ptr, const ClassPlan& cp,
                                          int block_index, const RowBlock& rb, int tid, int nthreads,
                                          int bar_id, int* s_flag, float* s_w) {
  named_barrier(bar_id, nthreads);
  if (tid == 0) {
    __threadfence();
    *s_flag = split_arrive(cp.counters + block_index, rb.nsplit, split_tag(p, cp));
    __threadfence();
  }
  named_barrier(bar_id, nthreads);
  if (*s_flag) merge_split_block(p, ptr, cp, rb, tid, nthreads, bar_id, s_w);
}

// The merge of finish_split_block, for a caller that has arrived itself (its arriving thread
// fenced after the atomic and the callers passed a barrier since) and is the block's last.
__device__ inline void merge_split_block(const Problem& p, const Pointers& ptr, const ClassPlan& cp,
                                         const RowBlock& rb, int tid, int nthreads, int bar_id, float* s_w) {
  __threadfence();
  const int seq_q0 = ptr.qsl[rb.seq];
  const int ns = rb.nsplit;
  if (ns <= kMergeMaxSplits) {
    // per-row weights once, then every (row, 4 columns) chunk with independent loads
    for (int r = tid; r < rb.nrows; r += nthreads) {
      float lse[kMergeMaxSplits];
      float M = -INFINITY;
#pragma unroll
      for (int i = 0; i < kMergeMaxSplits; ++i) {
        lse[i] = i < ns ? __ldcg(slot_lse(cp, rb.slot_base + i) + r) : -INFINITY;
        M = fmaxf(M, lse[i]);
      }
      float sum = 0.f;
#pragma unroll
      for (int i = 0; i < kMergeMaxSplits; ++i) {
        const float w = (lse[i] == -INFINITY) ? 0.f : exp2f(lse[i] - M);
        lse[i] = w;
        sum += w;
      }
      const float inv = sum > 0.f ? p.out_scale / sum : 0.f;
#pragma unroll
      for (int i = 0; i < kMergeMaxSplits; ++i)  // static indices keep lse[] in registers
        if (i < ns) s_w[i * kSlotRows + r] = lse[i] * inv;
    }
    named_barrier(bar_id, nthreads);
#pragma unroll 4
    for (int idx = tid; idx < rb.nrows * (kHeadDim / 4); idx += nthreads) {
      const int r = idx / (kHeadDim / 4);
      const int d = (idx % (kHeadDim / 4)) * 4;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int i = 0; i < ns; ++i) {
        const float w = s_w[i * kSlotRows + r];
        const uint2 h = __ldcg(reinterpret_cast<const uint2*>(slot_o(cp, rb.slot_base + i) +
                                                              (size_t)r * kHeadDim + d));
        const float2 o01 = unpack_f16x2(h.x), o23 = unpack_f16x2(h.y);
        acc.x += w * o01.x;
        acc.y += w * o01.y;
        acc.z += w * o23.x;
        acc.w += w * o23.y;
      }
      const RowMap m = map_row(rb.row0 + r, p.G, rb.kvh);
      uint2* dst = reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(ptr.out) +
                                            (size_t)(seq_q0 + m.t) * p.o_st + (size_t)m.h * p.o_sh + d);
      *dst = make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
    }
    named_barrier(bar_id, nthreads);  // s_w may be reused right after
    return;
  }
  for (int idx = tid; idx < rb.nrows * (kHeadDim / 2); idx += nthreads) {
    const int r = idx / (kHeadDim / 2);
    const int d = (idx % (kHeadDim / 2)) * 2;
    float M = -INFINITY;
    for (int i = 0; i < ns; ++i) M = fmaxf(M, __ldcg(slot_lse(cp, rb.slot_base + i) + r));
    float wsum = 0.f, a0 = 0.f, a1 = 0.f;
    for (int i = 0; i < ns; ++i) {
      const float lse = __ldcg(slot_lse(cp, rb.slot_base + i) + r);
      const float w = (lse == -INFINITY) ? 0.f : exp2f(lse - M);
      const float2 o = unpack_f16x2(__ldcg(reinterpret_cast<const unsigned int*>(slot_o(cp, rb.slot_base + i) +
                                                                                 (size_t)r * kHeadDim + d)));
      wsum += w;
      a0 += w * o.x;
      a1 += w * o.y;
    }
    const float inv = wsum > 0.f ? p.out_scale / wsum : 0.f;
    const RowMap m = map_row(rb.row0 + r, p.G, rb.kvh);
    uint32_t* dst = reinterpret_cast<uint32_t*>(static_cast<__nv_bfloat16*>(ptr.out) +
                                                (size_t)(seq_q0 + m.t) * p.o_st +
                                                (size_t)m.h * p.o_sh + d);
    *dst = pack_bf16x2(a0 * inv, a1 * inv);
  }
}

}  // namespace pgqa
