// plan.cuh -- launch entry points of the kernels, called by the host API.
#pragma once
#include "common.cuh"

namespace pgqa {

cudaError_t launch_plan(const Problem& p, const Pointers& ptr, const ClassPlan& verify,
                        const ClassPlan& prefill, cudaStream_t stream);

// Warp-level MMA (mma.sync, tf32) kernel for one class's items; any dtype mix.
cudaError_t launch_portable(const Problem& p, const Pointers& ptr, const ClassPlan& cp,
                            int block_rows, cudaStream_t stream);

}  // namespace pgqa
