// sparse.cu -- sparse paged GQA attention: each (token, kv head) attends a listed subset of
// its sequence's keys, shared by the kv head's query heads ("Tune sparse GQA prefill profile
// on gfx942 and gfx950": a selected list of ~2k tokens per row, head_dim 256, FP8 K/V).
//
// The tile of one unit (token t, kv head h, up to 16 of its query heads) has M = 16 rows,
// too few for a tcgen05 tile: the products run on warp-level mma.sync m16n8k16 (f16 in,
// fp32 accumulate). e4m3 K/V convert to f16 exactly; bf16 Q is converted to f16 once,
// after each warp scales its half of the unit's Q (its 128 dims) by a power of two 2^sig
// that puts that half's largest |q| in [2^14, 2^15): every bf16 value within 2^-24 of that
// maximum is then exact in f16 (bf16 values beyond f16's range, or below its normal range,
// included), and the warp multiplies its partial scores by 2^-sig (exact) before the pair
// adds them.
//
// Work split: a pair of warps per unit; warp w owns head dims [128w, 128w + 128). Per step
// of 16 listed keys each warp computes the partial S of all 16 keys over its d-half (two
// n8 tiles, 8 k-steps, Q of its half held in registers as f16 A fragments) and the pair
// adds the two partials through shared memory (a + b = b + a, so both warps hold the same
// bits and take the same softmax decisions without further exchange); each warp then
// turns S into P (an A fragment over the 16 keys) and accumulates O for its d-half
// (16 n8 tiles, one k-step). The reduction axis is permuted so that the four lanes of a
// key read 64 contiguous bytes of its K row per load (thread tig owns the 16-byte chunks
// tig and 4 + tig of the half), and the output dims of P.V are permuted so that each
// thread reads one contiguous 16-byte run of each V row it needs and ends with 32
// contiguous output dims per row. No K/V tile passes through shared memory: rows are
// loaded straight into registers (they are scattered by the index list).
//
// Online softmax in the exp2 domain with a lazy rescale (the reference moves only when a
// score exceeds it by 2^kTau), as in the dense kernels.
#include <cuda_runtime.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "common.cuh"
#include "device_util.cuh"
#include "plan.cuh"

namespace pgqa {

namespace {

constexpr int kPairs = 2;                 // units per CTA
constexpr int kSpThreads = kPairs * 64;
constexpr float kTauSp = 8.f;             // p <= 2^8 between rescales (f16 holds it exactly)

struct alignas(16) PairSmem {
  float xs[2][2][32][8];  // [step parity][warp][lane]: the warp's partial S fragment (2 n8 tiles)
};
// xs is read and written as float4: every pair's copy must start on 16 bytes
static_assert(sizeof(PairSmem) % 16 == 0, "PairSmem array elements stay 16-byte aligned");

__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two e4m3 codes (low byte first) -> f16x2 (exact).
__device__ __forceinline__ uint32_t e4m3x2_f16x2(uint32_t v16) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"((uint16_t)v16));
  return r;
}

// Byte sel of a (low) and byte sel of b (high) -> f16x2.
__device__ __forceinline__ uint32_t byte_pair_f16x2(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel | ((sel + 4) << 4)));
  return e4m3x2_f16x2(r);
}

// Two bf16 values times 2^sig (`scale`) -> f16x2.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w, float scale) {
  const __half2 h = __floats2half2_rn(__uint_as_float(w << 16) * scale, __uint_as_float(w & 0xffff0000u) * scale);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ float bf16x2_absmax(uint32_t w) {
  return fmaxf(fabsf(__uint_as_float(w << 16)), fabsf(__uint_as_float(w & 0xffff0000u)));
}

__device__ __forceinline__ uint32_t word_of(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

__device__ __forceinline__ void pair_sync(int pair) {
  asm volatile("bar.sync %0, 64;" ::"r"(1 + pair) : "memory");
}

// 64-bit shuffle of a row offset (-1: masked key).
__device__ __forceinline__ long long shfl_off(long long v, int src) {
  const int lo = __shfl_sync(0xffffffffu, (int)(v & 0xffffffff), src);
  const int hi = __shfl_sync(0xffffffffu, (int)(v >> 32), src);
  return ((long long)hi << 32) | (unsigned)lo;
}

}  // namespace

__global__ void __launch_bounds__(kSpThreads, 3) sparse_attn_kernel(SparseArgs a) {
  __shared__ PairSmem smem[kPairs];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int pair = warp >> 1, w = warp & 1;
  const int g = lane >> 2, tig = lane & 3;
  PairSmem& ps = smem[pair];

  const long long units = (long long)a.T * a.Hkv * a.HG;
  const long long u = (long long)blockIdx.x * kPairs + pair;
  if (u >= units) return;  // both warps of the pair
  const int hg = (int)(u % a.HG);
  const int kvh = (int)((u / a.HG) % a.Hkv);
  const int t = (int)(u / ((long long)a.HG * a.Hkv));
  const int head0 = kvh * a.G + hg * 16;
  const int rows = min(16, a.G - hg * 16);

  const int s = seq_of_token(a.qsl, a.num_seqs, t, lane);
  const int q0 = __ldg(a.qsl + s), q1 = __ldg(a.qsl + s + 1), L = __ldg(a.seq_lens + s);
  const int qn = q1 - q0;
  const bool unit_ok = t >= q0 && t < q1 && qn <= L;
  const int lim = L - qn + (t - q0);  // the row's causal limit
  if (!unit_ok && lane == 0 && w == 0) atomicOr(a.err, kErrBounds);

  // ---- this warp's half of Q (d in [128w, 128w + 128)) as f16 A fragments, in registers.
  // k-step kk (0..7) uses d = 128w + 16 (4 (kk >> 2) + tig) + 4 (kk & 3) .. +3, i.e. of the
  // 16-d chunks tig and 4 + tig of the half, elements 4 (kk & 3) .. +3.
  uint32_t qf[8][4];  // {row g pair 0, row g+8 pair 0, row g pair 1, row g+8 pair 1}
  uint4 raw[2][4];    // [half]: chunk tig (raw[.][0..1]) and chunk 4 + tig (raw[.][2..3]), bf16
  float qmax = 0.f;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int r = g + 8 * half;
    if (unit_ok && r < rows) {
      const uint16_t* row = a.q + (long long)t * a.q_st + (long long)(head0 + r) * a.q_sh + 128 * w;
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const uint4* src = reinterpret_cast<const uint4*>(row + 16 * (4 * i + tig));
        raw[half][2 * i] = __ldg(src);
        raw[half][2 * i + 1] = __ldg(src + 1);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) raw[half][i] = make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int k = 0; k < 4; ++k) qmax = fmaxf(qmax, bf16x2_absmax(word_of(raw[half][i], k)));
  }
  // max |q| over this warp's d-half of the unit's rows, then 2^sig with 2^sig * max in
  // [2^14, 2^15)
  qmax = fmaxf(qmax, __shfl_xor_sync(0xffffffffu, qmax, 1));
  qmax = fmaxf(qmax, __shfl_xor_sync(0xffffffffu, qmax, 2));
  qmax = fmaxf(qmax, __shfl_xor_sync(0xffffffffu, qmax, 4));
  qmax = fmaxf(qmax, __shfl_xor_sync(0xffffffffu, qmax, 8));
  qmax = fmaxf(qmax, __shfl_xor_sync(0xffffffffu, qmax, 16));
  int sig = 0;
  if (qmax > 0.f && qmax <= 3.0e38f) sig = 14 - ((int)((__float_as_uint(qmax) >> 23) & 0xff) - 127);
  sig = max(-120, min(120, sig));
  const float qscale = ldexpf(1.f, sig);
#pragma unroll
  for (int half = 0; half < 2; ++half) {
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const int e0 = 4 * (kk & 3);
      const uint4& c = raw[half][2 * (kk >> 2) + (e0 >> 3)];
      qf[kk][half] = bf16x2_to_f16x2(word_of(c, (e0 & 7) >> 1), qscale);
      qf[kk][2 + half] = bf16x2_to_f16x2(word_of(c, ((e0 & 7) >> 1) + 1), qscale);
    }
  }

  float o[16][4];
#pragma unroll
  for (int m = 0; m < 16; ++m) o[m][0] = o[m][1] = o[m][2] = o[m][3] = 0.f;
  float m_ref[2] = {-INFINITY, -INFINITY};  // rows g, g+8 (the same in both warps)
  float l_row[2] = {0.f, 0.f};             // this thread's keys' share of the row sums
  const float c = a.score_scale_log2;
  const float unscale = ldexpf(1.f, -sig);  // this warp's partial scores back to the unscaled q

  const int32_t* list = a.idx + (long long)t * a.idx_st + (long long)kvh * a.idx_sh;
  const int K = unit_ok ? a.K : 0;
  const uint8_t* kbase = a.k + 128 * w + 16 * tig;  // chunks tig and 4 + tig of my d-half
  const uint8_t* vbase = a.v + 128 * w + 16 * g;

  // Chunks of 32 listed entries (lane l holds entry c0 + l). The lookups that turn an entry
  // into a row offset are two dependent loads (position, then page), so they run ahead of
  // the chunk being computed: positions two chunks ahead, pages one chunk ahead.
  auto load_pos = [&](int c0) -> int {
    const int j = c0 + lane;
    return j < K ? __ldg(list + j) : -1;
  };
  auto usable = [&](int pos) -> bool { return pos >= 0 && pos <= lim && (pos >> a.p_shift) < a.W; };
  auto load_page = [&](int pos) -> int {
    return usable(pos) ? __ldg(a.bt + (long long)s * a.bt_stride + (pos >> a.p_shift)) : -1;
  };
  // byte offset of the entry's K/V row for this kv head, or -1 (not used: padding, past the
  // causal limit, or a bad page / block-table width, which also set the error word)
  auto row_offset = [&](int pos, int page) -> long long {
    if (pos < 0 || pos > lim) return -1;
    if ((pos >> a.p_shift) >= a.W) {  // L > W * P: the row has no such page
      atomicOr(a.err, kErrBounds);
      return -1;
    }
    if (page < 0 || page >= a.NB) {
      atomicOr(a.err, kErrPage);
      return -1;
    }
    return (long long)page * a.kv_sb + (long long)(pos & (a.P - 1)) * a.kv_sp + (long long)kvh * a.kv_sh;
  };
  int pos_c = load_pos(0), pos_n1 = load_pos(32);
  int page_c = load_page(pos_c);

  int par = 0;  // exchange buffer of the step
#pragma unroll 1
  for (int c0 = 0; c0 < K; c0 += 32) {
    const long long off_cur = row_offset(pos_c, page_c);
    const unsigned vm = __ballot_sync(0xffffffffu, off_cur >= 0);
    const int page_n1 = load_page(pos_n1);  // arrive while this chunk computes
    const int pos_n2 = load_pos(c0 + 64);
#pragma unroll 1
    for (int st = 0; st < 2; ++st) {
      if (((vm >> (16 * st)) & 0xffffu) == 0) continue;  // the same for both warps of the pair
      // K: my d-half of keys g (tile 0) and 8 + g (tile 1); V: my d-half rows of keys 2tig,
      // 2tig + 1, 8 + 2tig, 9 + 2tig (16 bytes at d = 128w + 16g)
      uint4 kr[2][2], vr[4];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const long long koff = shfl_off(off_cur, 16 * st + 8 * j + g);
#pragma unroll
        for (int i = 0; i < 2; ++i)
          kr[j][i] = koff >= 0 ? __ldg(reinterpret_cast<const uint4*>(kbase + koff + 64 * i)) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const long long voff = shfl_off(off_cur, 16 * st + 2 * tig + (i & 1) + 8 * (i >> 1));
        vr[i] = voff >= 0 ? __ldg(reinterpret_cast<const uint4*>(vbase + voff)) : make_uint4(0, 0, 0, 0);
      }
      // partial S over my d-half: rows g, g+8 x keys 2tig, 2tig+1 (tile 0) and 8+2tig, 9+2tig (tile 1)
      float sp[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const uint32_t kw = word_of(kr[j][kk >> 2], kk & 3);
          mma_f16(sp[j], qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3], e4m3x2_f16x2(kw & 0xffffu),
                  e4m3x2_f16x2(kw >> 16));
        }
      }
      // the pair's halves add up to the full S (a + b = b + a: both warps get the same bits),
      // each half first scaled back by its warp's exact power of two
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int i = 0; i < 4; ++i) sp[j][i] *= unscale;
      float4* mine = reinterpret_cast<float4*>(&ps.xs[par][w][lane][0]);
      mine[0] = make_float4(sp[0][0], sp[0][1], sp[0][2], sp[0][3]);
      mine[1] = make_float4(sp[1][0], sp[1][1], sp[1][2], sp[1][3]);
      pair_sync(pair);
      const float4* other = reinterpret_cast<const float4*>(&ps.xs[par][w ^ 1][lane][0]);
      const float4 o0 = other[0], o1 = other[1];
      par ^= 1;
      const float sfull[8] = {sp[0][0] + o0.x, sp[0][1] + o0.y, sp[0][2] + o0.z, sp[0][3] + o0.w,
                              sp[1][0] + o1.x, sp[1][1] + o1.y, sp[1][2] + o1.z, sp[1][3] + o1.w};
      // x[j][i]: tile j, {row g key a, row g key a+1, row g+8 key a, row g+8 key a+1}
      float x[8];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int kb = 16 * st + 8 * j + 2 * tig;
        const bool v0 = (vm >> kb) & 1u, v1 = (vm >> (kb + 1)) & 1u;
        x[4 * j + 0] = v0 ? sfull[4 * j + 0] * c : -INFINITY;
        x[4 * j + 1] = v1 ? sfull[4 * j + 1] * c : -INFINITY;
        x[4 * j + 2] = v0 ? sfull[4 * j + 2] * c : -INFINITY;
        x[4 * j + 3] = v1 ? sfull[4 * j + 3] * c : -INFINITY;
      }
      float mx[2] = {fmaxf(fmaxf(x[0], x[1]), fmaxf(x[4], x[5])), fmaxf(fmaxf(x[2], x[3]), fmaxf(x[6], x[7]))};
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
        // lazy rescale per row
        if (mx[r] > m_ref[r] + kTauSp || (m_ref[r] == -INFINITY && mx[r] > -INFINITY)) {
          const float alpha = exp2f(m_ref[r] - mx[r]);  // 0 when the reference was -inf
          l_row[r] *= alpha;
#pragma unroll
          for (int m = 0; m < 16; ++m) {
            o[m][2 * r] *= alpha;
            o[m][2 * r + 1] *= alpha;
          }
          m_ref[r] = mx[r];
        }
      }
      float p[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) p[i] = x[i] == -INFINITY ? 0.f : exp2f(x[i] - m_ref[(i >> 1) & 1]);
      l_row[0] += p[0] + p[1] + p[4] + p[5];
      l_row[1] += p[2] + p[3] + p[6] + p[7];
      // P as the A fragment over the step's 16 keys: tile 0 -> k 2tig.., tile 1 -> k 8+2tig..
      const __half2 a0 = __floats2half2_rn(p[0], p[1]), a1 = __floats2half2_rn(p[2], p[3]);
      const __half2 a2 = __floats2half2_rn(p[4], p[5]), a3 = __floats2half2_rn(p[6], p[7]);
      const uint32_t pa0 = *reinterpret_cast<const uint32_t*>(&a0), pa1 = *reinterpret_cast<const uint32_t*>(&a1);
      const uint32_t pa2 = *reinterpret_cast<const uint32_t*>(&a2), pa3 = *reinterpret_cast<const uint32_t*>(&a3);
#pragma unroll
      for (int m = 0; m < 16; ++m) {
        const int wi = m >> 2;
        const uint32_t sel = (uint32_t)(m & 3);
        const uint32_t b0 = byte_pair_f16x2(word_of(vr[0], wi), word_of(vr[1], wi), sel);
        const uint32_t b1 = byte_pair_f16x2(word_of(vr[2], wi), word_of(vr[3], wi), sel);
        mma_f16(o[m], pa0, pa1, pa2, pa3, b0, b1);
      }
    }
    pos_c = pos_n1;
    page_c = page_n1;
    pos_n1 = pos_n2;
  }

  // ---- epilogue: row sums (the same in both warps), normalise, bf16 rows of my d-half
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    l_row[r] += __shfl_xor_sync(0xffffffffu, l_row[r], 1);
    l_row[r] += __shfl_xor_sync(0xffffffffu, l_row[r], 2);
  }
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int row = g + 8 * r;
    if (row >= rows) continue;
    const float inv = l_row[r] > 0.f ? a.out_scale / l_row[r] : 0.f;
    uint4* dst = reinterpret_cast<uint4*>(a.out + (long long)t * a.o_st + (long long)(head0 + row) * a.o_sh +
                                          128 * w + 32 * tig);
    // dims 0..15 of my run are o[m][2r] (m = 0..15), dims 16..31 are o[m][2r + 1]
#pragma unroll
    for (int hseg = 0; hseg < 2; ++hseg) {
      uint32_t pk[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        pk[i] = pack_bf16x2(o[2 * i][2 * r + hseg] * inv, o[2 * i + 1][2 * r + hseg] * inv);
      dst[2 * hseg] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      dst[2 * hseg + 1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
    }
  }
}

cudaError_t launch_sparse(const SparseArgs& a, cudaStream_t stream) {
  const long long units = (long long)a.T * a.Hkv * a.HG;
  if (units == 0) return cudaSuccess;
  const long long grid = (units + kPairs - 1) / kPairs;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  sparse_attn_kernel<<<(unsigned)grid, kSpThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace pgqa
