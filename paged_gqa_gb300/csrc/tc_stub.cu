#include "tc_kernels.cuh"
namespace pgqa {
int launch_verify_tc(const Problem&, const Pointers&, const ClassPlan&, const pg_tensor*, const pg_tensor*, int, cudaStream_t) { return 0; }
int launch_prefill_tc(const Problem&, const Pointers&, const ClassPlan&, const pg_tensor*, const pg_tensor*, int, cudaStream_t) { return 0; }
const char* tc_last_error() { return ""; }
}
