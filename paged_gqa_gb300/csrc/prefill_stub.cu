// prefill_stub.cu -- placeholder until the tcgen05 prefill kernel exists: prefill blocks
// use the warp-MMA kernel.
#include "tc_kernels.cuh"
namespace pgqa {
int launch_prefill_tc(const Problem&, const Pointers&, const ClassPlan&, const pg_tensor*, const pg_tensor*, int,
                      cudaStream_t) {
  return 0;
}
}  // namespace pgqa
