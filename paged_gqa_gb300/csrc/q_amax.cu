// q_amax.cu -- the first half of a per-tensor FP8 quantisation of a bf16 Q inside the call:
// max |q| over the whole tensor, left as one partial maximum per CTA.
//
// "asm FP8 FMHA for prefix-hit prefill" runs its FP8 attention on a Q cast to e4m3 with one
// per-tensor scale (its summary counts the casts inside the attention time). Here the
// attention kernels do the cast while they stage Q (kQCast): each CTA reduces these
// partial maxima to amax and takes descale = amax / 448 (tc_util.cuh, q_cast_scales), so
// no zeroing launch and no atomics are needed and every CTA derives the same scale.
//
// HBM-bound: one warp per (token, head) row of 512 bytes, one 16-byte load per lane,
// four rows in flight per warp, grid-stride over rows. NaNs do not enter the maximum.
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "plan.cuh"
#include "tc_util.cuh"

namespace pgqa {

namespace {

constexpr int kWarps = 16;
constexpr int kUnroll = 4;

__device__ __forceinline__ float amax8(uint4 x) {
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
  float m = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i)
    m = fmaxf(m, fmaxf(fabsf(__uint_as_float(w[i] << 16)), fabsf(__uint_as_float(w[i] & 0xffff0000u))));
  return m;
}

}  // namespace

__global__ void __launch_bounds__(kWarps * 32) q_amax_kernel(const uint16_t* __restrict__ q, long long q_st,
                                                             long long q_sh, int T, int Hq, float* parts) {
  __shared__ float red[kWarps];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const long long rows = (long long)T * Hq;
  const long long stride = (long long)gridDim.x * kWarps;
  float m = 0.f;
  for (long long r0 = (long long)blockIdx.x * kWarps + warp; r0 < rows; r0 += stride * kUnroll) {
    uint4 x[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const long long r = r0 + u * stride;
      x[u] = make_uint4(0, 0, 0, 0);
      if (r < rows) {
        const long long t = r / Hq, h = r % Hq;
        x[u] = __ldg(reinterpret_cast<const uint4*>(q + t * q_st + h * q_sh) + lane);
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) m = fmaxf(m, amax8(x[u]));
  }
  m = tc::warp_max(m);
  if (lane == 0) red[warp] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float a = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) a = fmaxf(a, red[w]);
    parts[blockIdx.x] = a;
  }
}

int q_amax_parts(int sms) { return 2 * sms; }

cudaError_t launch_q_amax(const Problem& p, const Pointers& ptr, float* parts, cudaStream_t stream) {
  q_amax_kernel<<<p.q_amax_parts, kWarps * 32, 0, stream>>>(static_cast<const uint16_t*>(ptr.q), p.q_st, p.q_sh,
                                                            p.T, p.Hq, parts);
  return cudaGetLastError();
}

}  // namespace pgqa
