// tc_kernels.cuh -- launchers of the tcgen05 (5th-generation tensor core) kernels.
//
// Each returns 1 if it launched, 0 if the problem is outside what the kernel handles
// (the caller then uses the warp-MMA kernel), or -1 on a launch error (message from
// tc_last_error()).
#pragma once
#include <cuda.h>
#include <cstdlib>

#include "../../include/paged_gqa.h"
#include "common.cuh"

namespace pgqa {

// dependent: launch as a programmatic dependent of the kernel before it on the stream (the
// plan kernel; off unless pdl_enabled()).
int launch_verify_tc(const Problem& p, const Pointers& ptr, const ClassPlan& cp, const pg_tensor* k,
                     const pg_tensor* v, int sms, cudaStream_t stream, bool dependent);
// dependent: launch as a programmatic dependent of the kernel before it on the stream (the
// verify-class kernel), so its CTAs are already resident when that kernel ends.
int launch_prefill_tc(const Problem& p, const Pointers& ptr, const ClassPlan& cp, const pg_tensor* k,
                      const pg_tensor* v, int sms, cudaStream_t stream, bool dependent);
// bf16 q and bf16 caches, either class of row blocks (bf16_tc.cu). self_planned: the
// verify-class launch of a call with Problem::fused_verify (its CTAs plan the class).
int launch_bf16_tc(const Problem& p, const Pointers& ptr, const ClassPlan& cp, const pg_tensor* k,
                   const pg_tensor* v, cudaStream_t stream, bool dependent, bool self_planned);
const char* tc_last_error();
void set_tc_error(const char* msg);
// TMA map over an e4m3 or bf16 cache [NB, P, Hkv, 256] (128 bytes of d of one page per box).
bool make_cache_tmap(CUtensorMap* m, const pg_tensor* t, int P);

// Programmatic dependent launch of the first attention kernel (after the plan kernel) is off
// unless the environment sets PAGED_GQA_PDL=1 (a tuning knob for launch-overhead
// measurements; results are identical either way). Measured on the MTP verify batch it
// added ~12 us per call: the CTA that lands on the plan kernel's SM starts late and every
// CTA has the same amount of work. The second attention kernel is always a dependent of
// the first (its CTAs wait in griddepcontrol.wait until the first kernel has completed).
inline bool pdl_enabled() {
  static const bool on = [] {
    const char* e = getenv("PAGED_GQA_PDL");
    return e && e[0] == '1';
  }();
  return on;
}

// Launch with programmatic stream serialization: the kernel may start (and run its
// prologue up to griddepcontrol.wait) while the previous kernel on the stream finishes.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(bool dependent, void (*kernel)(KArgs...), int grid, int block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = dependent ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

}  // namespace pgqa
