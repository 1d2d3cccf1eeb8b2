// portable.cu -- warp-level MMA (mma.sync m16n8k8 tf32) paged GQA attention.
//
// Handles every dtype mix (bf16 or e4m3 Q; bf16 or e4m3 K/V) and every block shape;
// it is the path for bf16 caches and the reference path the tcgen05 kernels are
// checked against. Each operand is widened to fp32 exactly (bf16 and e4m3 values have
// at most 8 significant bits, so they are exact in tf32); P is rounded to tf32
// (11 significant bits) before P.V; accumulation is fp32.
//
// One persistent CTA of 8 warps walks its range of work items. A warp owns 16 query
// rows of the block; K and V tiles of 32 keys are gathered page by page from the
// block table into shared memory ("Optimize Qwen3.5 MTP unified attention on gfx950":
// the kv tile is loaded once and reused by all q_len x G rows of the kv head).
// Online softmax per row with quad shuffles; split pieces write partial results that
// the last piece merges.
#include "common.cuh"
#include "device_util.cuh"
#include "plan.cuh"
#include "tc_kernels.cuh"

namespace pgqa {

namespace {

constexpr int kPWarps = 8;
constexpr int kPThreads = kPWarps * 32;
constexpr int kPKeys = 32;
constexpr int kPitch = kHeadDim + 4;  // floats; keeps fragment loads conflict-free
constexpr size_t kPSmemBytes = (size_t)(kPrefillRows + 2 * kPKeys) * kPitch * sizeof(float) +
                               (size_t)kMergeMaxSplits * kSlotRows * sizeof(float);

__device__ __forceinline__ uint32_t to_tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}

__device__ __forceinline__ void mma_tf32(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Widen 32 consecutive elements (bf16 or e4m3) at src to fp32 at dst (16-byte aligned).
__device__ __forceinline__ void load32(float* dst, const void* src, bool fp8, float fill_zero) {
  if (fill_zero != 0.f) {
#pragma unroll
    for (int i = 0; i < 32; i += 4) *reinterpret_cast<float4*>(dst + i) = make_float4(0.f, 0.f, 0.f, 0.f);
    return;
  }
  if (fp8) {
    const uint4* s = reinterpret_cast<const uint4*>(src);
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      uint4 w = s[c];
      uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float2 lo = e4m3x2_to_float2((uint16_t)(ws[j] & 0xffff));
        float2 hi = e4m3x2_to_float2((uint16_t)(ws[j] >> 16));
        *reinterpret_cast<float4*>(dst + c * 16 + j * 4) = make_float4(lo.x, lo.y, hi.x, hi.y);
      }
    }
  } else {
    const uint4* s = reinterpret_cast<const uint4*>(src);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint4 w = s[c];
      uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int j = 0; j < 4; j += 2) {
        *reinterpret_cast<float4*>(dst + c * 8 + j * 2) =
            make_float4(bf16_bits_to_float(ws[j] & 0xffff), bf16_bits_to_float(ws[j] >> 16),
                        bf16_bits_to_float(ws[j + 1] & 0xffff), bf16_bits_to_float(ws[j + 1] >> 16));
      }
    }
  }
}

}  // namespace

__global__ void __launch_bounds__(kPThreads, 1)
portable_attn_kernel(Problem p, Pointers ptr, ClassPlan cp) {
  extern __shared__ __align__(16) float smem[];
  float* Qs = smem;                          // [128][kPitch]
  float* Ks = Qs + kPrefillRows * kPitch;    // [32][kPitch]
  float* Vs = Ks + kPKeys * kPitch;          // [32][kPitch]
  __shared__ int s_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, tq = lane & 3;
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the plan kernel has completed
  const int item_begin = cp.cta_item_begin[blockIdx.x];
  const int item_end = cp.cta_item_begin[blockIdx.x + 1];
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const size_t esz_q = p.q_is_fp8 ? 1 : 2, esz_kv = p.kv_is_fp8 ? 1 : 2;

  for (int it = item_begin; it < item_end; ++it) {
    const WorkItem item = cp.items[it];
    const RowBlock rb = cp.blocks[item.block];
    const int seq_q0 = ptr.qsl[rb.seq];
    const int qn = ptr.qsl[rb.seq + 1] - seq_q0;
    const int L = ptr.seq_lens[rb.seq];
    const int key_lo = item.tile_begin * kTileKeys;
    const int key_hi = min(item.tile_end * kTileKeys, rb.kv_end);

    // ---- Q rows -> smem (fp32); rows past nrows are zero
    for (int idx = tid; idx < kPrefillRows * 8; idx += kPThreads) {
      const int r = idx >> 3, seg = idx & 7;
      const bool valid = r < rb.nrows;
      const void* src = nullptr;
      if (valid) {
        const RowMap m = map_row(rb.row0 + r, p.G, rb.kvh);
        src = static_cast<const char*>(ptr.q) +
              ((size_t)(seq_q0 + m.t) * p.q_st + (size_t)m.h * p.q_sh + seg * 32) * esz_q;
      }
      load32(Qs + r * kPitch + seg * 32, src, p.q_is_fp8, valid ? 0.f : 1.f);
    }

    // per-thread rows and their causal limits
    const int lr0 = warp * 16 + g, lr1 = lr0 + 8;
    const int lim0 = lr0 < rb.nrows ? L - qn + (rb.row0 + lr0) / p.G : -1;
    const int lim1 = lr1 < rb.nrows ? L - qn + (rb.row0 + lr1) / p.G : -1;
    const bool warp_active = warp * 16 < rb.nrows;

    float o[32][4];
#pragma unroll
    for (int i = 0; i < 32; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

    for (int k0 = key_lo; k0 < key_hi; k0 += kPKeys) {
      __syncthreads();  // previous tile fully consumed (and Q written on the first pass)
      // ---- gather K/V rows of this tile: thread -> (key = tid % 32, segment = tid / 32)
      {
        const int key = tid & 31, seg = tid >> 5;
        const int j = k0 + key;
        bool valid = j < key_hi;
        size_t koff = 0, voff = 0;
        if (valid) {
          const int blk = ptr.block_table[(size_t)rb.seq * p.bt_stride + j / p.P];
          if (blk < 0 || blk >= p.NB) {
            atomicOr(ptr.err, kErrPage);
            valid = false;
          } else {
            const int r = j % p.P;
            koff = ((size_t)blk * p.k_sb + (size_t)r * p.k_sp + (size_t)rb.kvh * p.k_sh + seg * 32) * esz_kv;
            voff = ((size_t)blk * p.v_sb + (size_t)r * p.v_sp + (size_t)rb.kvh * p.v_sh + seg * 32) * esz_kv;
          }
        }
        load32(Ks + key * kPitch + seg * 32, static_cast<const char*>(ptr.k) + koff, p.kv_is_fp8,
               valid ? 0.f : 1.f);
        load32(Vs + key * kPitch + seg * 32, static_cast<const char*>(ptr.v) + voff, p.kv_is_fp8,
               valid ? 0.f : 1.f);
      }
      __syncthreads();
      if (!warp_active) continue;

      // ---- S = Q K^T for this warp's 16 rows x 32 keys
      float s[4][4];
#pragma unroll
      for (int n = 0; n < 4; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
      const float* qa = Qs + (warp * 16 + g) * kPitch + tq;
#pragma unroll 4
      for (int kk = 0; kk < kHeadDim / 8; ++kk) {
        const uint32_t a0 = __float_as_uint(qa[kk * 8]);
        const uint32_t a1 = __float_as_uint(qa[8 * kPitch + kk * 8]);
        const uint32_t a2 = __float_as_uint(qa[kk * 8 + 4]);
        const uint32_t a3 = __float_as_uint(qa[8 * kPitch + kk * 8 + 4]);
#pragma unroll
        for (int n = 0; n < 4; ++n) {
          const float* kb = Ks + (n * 8 + g) * kPitch + kk * 8 + tq;
          mma_tf32(s[n], a0, a1, a2, a3, __float_as_uint(kb[0]), __float_as_uint(kb[4]));
        }
      }

      // ---- scale, mask, online softmax (rows g and g+8 of the warp)
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int n = 0; n < 4; ++n) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int key = k0 + n * 8 + 2 * tq + (e & 1);
          const int lim = min(key_hi - 1, (e < 2) ? lim0 : lim1);
          const float v = key <= lim ? s[n][e] * p.score_scale_log2 : -INFINITY;
          s[n][e] = v;
          if (e < 2) mx0 = fmaxf(mx0, v); else mx1 = fmaxf(mx1, v);
        }
      }
#pragma unroll
      for (int o_ = 1; o_ <= 2; o_ <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o_));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o_));
      }
      const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
      const float ref0 = mn0 == -INFINITY ? 0.f : mn0, ref1 = mn1 == -INFINITY ? 0.f : mn1;
      const float al0 = exp2f(m0 - ref0), al1 = exp2f(m1 - ref1);
      m0 = mn0;
      m1 = mn1;
      float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
      for (int n = 0; n < 4; ++n) {
        s[n][0] = exp2f(s[n][0] - ref0);
        s[n][1] = exp2f(s[n][1] - ref0);
        s[n][2] = exp2f(s[n][2] - ref1);
        s[n][3] = exp2f(s[n][3] - ref1);
        ps0 += s[n][0] + s[n][1];
        ps1 += s[n][2] + s[n][3];
      }
      l0 = l0 * al0 + ps0;
      l1 = l1 * al1 + ps1;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        o[i][0] *= al0;
        o[i][1] *= al0;
        o[i][2] *= al1;
        o[i][3] *= al1;
      }

      // ---- O += P V. The k index of the A fragment is permuted so that the S
      // accumulator layout (keys 2t, 2t+1) serves directly as the A fragment
      // (k = t -> key 2t, k = t+4 -> key 2t+1); V rows are read in the same order.
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        const uint32_t a0 = to_tf32(s[ks][0]), a1 = to_tf32(s[ks][2]);
        const uint32_t a2 = to_tf32(s[ks][1]), a3 = to_tf32(s[ks][3]);
        const float* vb0 = Vs + (ks * 8 + 2 * tq) * kPitch + g;
        const float* vb1 = vb0 + kPitch;
#pragma unroll
        for (int nd = 0; nd < 32; ++nd)
          mma_tf32(o[nd], a0, a1, a2, a3, __float_as_uint(vb0[nd * 8]), __float_as_uint(vb1[nd * 8]));
      }
    }

    // ---- finish: full row sums, normalise, write output or partial
#pragma unroll
    for (int o_ = 1; o_ <= 2; o_ <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, o_);
      l1 += __shfl_xor_sync(0xffffffffu, l1, o_);
    }
    const float inv0 = l0 > 0.f ? p.out_scale / l0 : 0.f;
    const float inv1 = l1 > 0.f ? p.out_scale / l1 : 0.f;
    const float lse0 = l0 > 0.f ? m0 + log2f(l0) : -INFINITY;
    const float lse1 = l1 > 0.f ? m1 + log2f(l1) : -INFINITY;
    if (rb.nsplit == 1) {
      if (warp_active) {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const int lr = half ? lr1 : lr0;
          if (lr >= rb.nrows) continue;
          const RowMap m = map_row(rb.row0 + lr, p.G, rb.kvh);
          __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(ptr.out) + (size_t)(seq_q0 + m.t) * p.o_st +
                               (size_t)m.h * p.o_sh + 2 * tq;
          const float inv = half ? inv1 : inv0;
#pragma unroll
          for (int nd = 0; nd < 32; ++nd)
            *reinterpret_cast<uint32_t*>(dst + nd * 8) =
                pack_bf16x2(o[nd][2 * half] * inv, o[nd][2 * half + 1] * inv);
        }
      }
      __syncthreads();  // smem reuse by the next item
    } else {
      const int slot = rb.slot_base + item.split;
      if (warp_active) {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const int lr = half ? lr1 : lr0;
          if (lr >= rb.nrows) continue;
          uint16_t* dst = slot_o(cp, slot) + (size_t)lr * kHeadDim + 2 * tq;
          // the partial leaves in code units: v_descale is applied by the merge
          const float l = half ? l1 : l0;
          const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
          for (int nd = 0; nd < 32; ++nd)
            *reinterpret_cast<uint32_t*>(dst + nd * 8) = pack_f16x2(o[nd][2 * half] * inv, o[nd][2 * half + 1] * inv);
          if (tq == 0) slot_lse(cp, slot)[lr] = half ? lse1 : lse0;
        }
      }
      __threadfence();
      finish_split_block(p, ptr, cp, item.block, rb, tid, kPThreads, 1, &s_flag, Vs + kPKeys * kPitch);
      __syncthreads();
    }
  }
}

cudaError_t launch_portable(const Problem& p, const Pointers& ptr, const ClassPlan& cp, int block_rows,
                            cudaStream_t stream) {
  (void)block_rows;
  static bool attr_set = false;  // per process; the attribute is per function, not per device
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(portable_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kPSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaError_t e = launch_pdl(false, portable_attn_kernel, cp.num_ctas, kPThreads, kPSmemBytes, stream, p, ptr, cp);
  return e == cudaSuccess ? cudaGetLastError() : e;
}

}  // namespace pgqa
