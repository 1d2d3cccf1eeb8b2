// cache_write.cu -- the paged KV-cache write: new tokens' K and V, quantised to e4m3 with the
// per-tensor descale, scattered into their pages through the block table.
//
// It is the step before the attention path ("Optimize Qwen3.5 MTP unified attention on
// gfx950" and "asm FP8 FMHA for prefix-hit prefill" read an FP8 cache that this fills):
// sequence s's q_len new tokens take positions L - q_len .. L - 1 (seq_lens counts them),
// position pos lands in page block_table[s][pos / P] at slot pos % P, and each of the 256
// values of a (token, kv head) row is stored as the e4m3 code of value * inv, where inv =
// 1 / descale rounded to float32 on the host and the product is taken in float32 (then
// clamped to +-448, round to nearest even); the attention multiplies the descale back.
//
// HBM-bound: a (token, kv head) row per warp step, 8 values per lane (16-byte bf16 loads,
// 8-byte e4m3 stores). Bytes per row: 2 x 512 read + 2 x 256 written.
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "device_util.cuh"
#include "plan.cuh"
#include "tc_util.cuh"

namespace pgqa {

namespace {

constexpr int kWarps = 8;
constexpr int kCtasPerSm = 6;  // CTAs of 256 threads per SM (39 registers a thread)

// 8 bf16 values (one uint4) times scale -> 8 e4m3 codes (uint2), element 0 in the low byte.
__device__ __forceinline__ uint2 quant8(uint4 x, float scale) {
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
  uint32_t c[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    c[i] = tc::e4m3x2(__uint_as_float(w[i] << 16) * scale, __uint_as_float(w[i] & 0xffff0000u) * scale);
  return make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
}

}  // namespace

// Each warp takes a contiguous, balanced range of (token, kv head) rows, tokens major, so
// it finds its first row's sequence by one binary search and then walks forward. The next
// row's 1 KB of bf16 is loaded before the current row is converted and stored, so two rows
// are in flight per warp while the page lookup of the current token resolves.
__global__ void __launch_bounds__(kWarps * 32, kCtasPerSm) cache_write_kernel(CacheWriteArgs a) {
  const int lane = threadIdx.x & 31, d = lane * 8;
  const long long rows = (long long)a.T * a.Hkv;
  const long long nwarps = (long long)gridDim.x * kWarps;
  const long long w = (long long)blockIdx.x * kWarps + (threadIdx.x >> 5);
  const long long r_begin = w * rows / nwarps, r_end = (w + 1) * rows / nwarps;
  if (r_begin >= r_end || a.num_seqs <= 0) return;
  int t = (int)(r_begin / a.Hkv), h = (int)(r_begin - (long long)t * a.Hkv);
  auto load = [&](int tt, int hh, uint4& kx, uint4& vx) {
    kx = __ldcs(reinterpret_cast<const uint4*>(a.kn + (long long)tt * a.kn_st + (long long)hh * a.kn_sh + d));
    vx = __ldcs(reinterpret_cast<const uint4*>(a.vn + (long long)tt * a.vn_st + (long long)hh * a.vn_sh + d));
  };
  uint4 kx, vx;
  load(t, h, kx, vx);  // in flight while the sequence and page are looked up
  int s = seq_of_token(a.qsl, a.num_seqs, t, lane);
  int q0 = __ldg(a.qsl + s), q1 = __ldg(a.qsl + s + 1), L = __ldg(a.seq_lens + s);
  int page_t = -1, page = -1, slot = 0;  // page and slot of token page_t (page < 0: skip)
  for (long long r = r_begin; r < r_end; ++r) {
    // the next row, loaded before this one is finished
    int tn = t, hn = h + 1;
    if (hn == a.Hkv) {
      hn = 0;
      ++tn;
    }
    uint4 kn = make_uint4(0, 0, 0, 0), vn = kn;
    if (r + 1 < r_end) load(tn, hn, kn, vn);
    if (t != page_t) {
      page_t = t;
      while (t >= q1 && s < a.num_seqs - 1) {
        ++s;
        q0 = q1;
        q1 = __ldg(a.qsl + s + 1);
        L = __ldg(a.seq_lens + s);
      }
      const int qn = q1 - q0, pos = L - qn + (t - q0);
      page = -1;
      if (t < q0 || t >= q1 || qn > L || pos < 0 || (pos >> a.p_shift) >= a.W) {
        if (lane == 0) atomicOr(a.err, kErrBounds);
      } else {
        const int pg = __ldg(a.bt + (long long)s * a.bt_stride + (pos >> a.p_shift));
        if (pg < 0 || pg >= a.NB) {
          if (lane == 0) atomicOr(a.err, kErrPage);
        } else {
          page = pg;
          slot = pos & (a.P - 1);
        }
      }
    }
    if (page >= 0) {
      __stcs(reinterpret_cast<uint2*>(a.kc + page * a.kc_sb + slot * a.kc_sp + h * a.kc_sh + d), quant8(kx, a.k_scale));
      __stcs(reinterpret_cast<uint2*>(a.vc + page * a.vc_sb + slot * a.vc_sp + h * a.vc_sh + d), quant8(vx, a.v_scale));
    }
    t = tn;
    h = hn;
    kx = kn;
    vx = vn;
  }
}

cudaError_t launch_cache_write(const CacheWriteArgs& a, int sms, cudaStream_t stream) {
  const long long rows = (long long)a.T * a.Hkv;
  if (rows == 0) return cudaSuccess;
  // one wave; at least two rows per warp
  const long long want = (rows + 2 * kWarps - 1) / (2 * kWarps);
  const int grid = (int)(want < (long long)sms * kCtasPerSm ? want : (long long)sms * kCtasPerSm);
  cache_write_kernel<<<grid, kWarps * 32, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace pgqa
