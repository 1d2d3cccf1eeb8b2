// plan.cuh -- launch entry points of the kernels, called by the host API.
#pragma once
#include "common.cuh"

namespace pgqa {

// plan_verify false: the verify class plans itself (Problem::fused_verify) and this kernel
// follows its kernel; dependent: launched as that kernel's programmatic dependent.
cudaError_t launch_plan(const Problem& p, const Pointers& ptr, const ClassPlan& verify,
                        const ClassPlan& prefill, bool plan_verify, bool dependent, cudaStream_t stream);

// Arguments of the paged KV-cache write (cache_write.cu); strides in elements.
struct CacheWriteArgs {
  const uint16_t* kn;
  const uint16_t* vn;
  long long kn_st, kn_sh, vn_st, vn_sh;  // elements
  uint8_t* kc;
  uint8_t* vc;
  long long kc_sb, kc_sp, kc_sh, vc_sb, vc_sp, vc_sh;  // bytes (elements of 1 byte)
  const int32_t* bt;
  long long bt_stride;
  const int32_t* seq_lens;
  const int32_t* qsl;
  int num_seqs, T, Hkv, P, W, NB;
  int p_shift;             // log2(P)
  float k_scale, v_scale;  // 1 / descale
  uint32_t* err;
};
// Paged KV-cache write (cache_write.cu): new tokens' K and V -> e4m3 codes in their pages.
cudaError_t launch_cache_write(const CacheWriteArgs& a, int sms, cudaStream_t stream);

// Arguments of sparse paged GQA attention (sparse.cu).
struct SparseArgs {
  const uint16_t* q;                   // [T, Hq, 256] bf16
  long long q_st, q_sh;                // elements
  const uint8_t* k;                    // [NB, P, Hkv, 256] e4m3
  const uint8_t* v;
  long long kv_sb, kv_sp, kv_sh;       // bytes, the same for K and V
  const int32_t* bt;
  long long bt_stride;
  const int32_t* seq_lens;
  const int32_t* qsl;
  const int32_t* idx;                  // [T, Hkv, K] positions
  long long idx_st, idx_sh;            // elements
  int K;
  uint16_t* out;                       // [T, Hq, 256] bf16
  long long o_st, o_sh;                // elements
  int num_seqs, T, Hq, Hkv, G, HG, P, p_shift, W, NB;  // HG = ceil(G / 16) head groups per kv head
  float score_scale_log2;              // softmax_scale * k_descale * log2(e)
  float out_scale;                     // v_descale
  uint32_t* err;
};
cudaError_t launch_sparse(const SparseArgs& a, cudaStream_t stream);
// tcgen05 kernel of sparse attention (sparse_tc.cu): 1 if launched, 0 if the call is outside
// what it handles (lists shorter than sparse_tc_min_keys()), -1 on a launch error (message
// from tc_last_error()).
int launch_sparse_tc(const SparseArgs& a, int sms, uint32_t stall_test_ns, cudaStream_t stream);
int sparse_tc_min_keys();

// Per-CTA maxima of |q| over a bf16 Q (q_amax.cu), q_amax_parts(sms) of them, for the
// per-tensor cast of Q in the tcgen05 kernels.
int q_amax_parts(int sms);
cudaError_t launch_q_amax(const Problem& p, const Pointers& ptr, float* parts, cudaStream_t stream);

// Warp-level MMA (mma.sync, tf32) kernel for one class's items; any dtype mix.
cudaError_t launch_portable(const Problem& p, const Pointers& ptr, const ClassPlan& cp,
                            int block_rows, cudaStream_t stream);

}  // namespace pgqa
