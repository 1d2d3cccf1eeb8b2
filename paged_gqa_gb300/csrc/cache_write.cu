// cache_write.cu -- the paged KV-cache write: new tokens' K and V, quantised to e4m3 with the
// per-tensor descale, scattered into their pages through the block table.
//
// It is the step before the attention path ("Optimize Qwen3.5 MTP unified attention on
// gfx950" and "asm FP8 FMHA for prefix-hit prefill" read an FP8 cache that this fills):
// sequence s's q_len new tokens take positions L - q_len .. L - 1 (seq_lens counts them),
// position pos lands in page block_table[s][pos / P] at slot pos % P, and each of the 256
// values of a (token, kv head) row is stored as the e4m3 code of value / descale (clamped
// to +-448, round to nearest even), which the attention multiplies back.
//
// HBM-bound: one warp per (token, kv head) row, 8 values per lane (16-byte bf16 loads,
// 8-byte e4m3 stores), grid-stride over rows. Bytes per row: 2 x 512 read + 2 x 256 written.
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "plan.cuh"
#include "tc_util.cuh"

namespace pgqa {

namespace {

constexpr int kWarps = 8;

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

__global__ void __launch_bounds__(kWarps * 32) cache_write_kernel(CacheWriteArgs a) {
  const int lane = threadIdx.x & 31;
  const long long rows = (long long)a.T * a.Hkv;
  for (long long r = (long long)blockIdx.x * kWarps + (threadIdx.x >> 5); r < rows;
       r += (long long)gridDim.x * kWarps) {
    const int t = (int)(r / a.Hkv), h = (int)(r % a.Hkv);
    // the sequence of token t: the last s with query_start_loc[s] <= t
    int lo = 0, hi = a.num_seqs - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (__ldg(a.qsl + mid) <= t) lo = mid; else hi = mid - 1;
    }
    const int q0 = __ldg(a.qsl + lo), qn = __ldg(a.qsl + lo + 1) - q0, L = __ldg(a.seq_lens + lo);
    const int pos = L - qn + (t - q0);
    if (a.num_seqs == 0 || t < q0 || t >= q0 + qn || qn > L || pos < 0 || pos / a.P >= a.W) {
      if (lane == 0) atomicOr(a.err, kErrBounds);
      continue;
    }
    const int page = __ldg(a.bt + (long long)lo * a.bt_stride + pos / a.P);
    if (page < 0 || page >= a.NB) {
      if (lane == 0) atomicOr(a.err, kErrPage);
      continue;
    }
    const int slot = pos % a.P, d = lane * 8;
    const uint4 kx = *reinterpret_cast<const uint4*>(a.kn + (long long)t * a.kn_st + (long long)h * a.kn_sh + d);
    const uint4 vx = *reinterpret_cast<const uint4*>(a.vn + (long long)t * a.vn_st + (long long)h * a.vn_sh + d);
    *reinterpret_cast<uint2*>(a.kc + page * a.kc_sb + slot * a.kc_sp + h * a.kc_sh + d) = quant8(kx, a.k_scale);
    *reinterpret_cast<uint2*>(a.vc + page * a.vc_sb + slot * a.vc_sp + h * a.vc_sh + d) = quant8(vx, a.v_scale);
  }
}

cudaError_t launch_cache_write(const CacheWriteArgs& a, int sms, cudaStream_t stream) {
  const long long rows = (long long)a.T * a.Hkv;
  if (rows == 0) return cudaSuccess;
  const long long want = (rows + kWarps - 1) / kWarps;
  const int grid = (int)(want < (long long)sms * 16 ? want : (long long)sms * 16);
  cache_write_kernel<<<grid, kWarps * 32, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace pgqa
