// tc_kernels.cuh -- launchers of the tcgen05 (5th-generation tensor core) kernels.
//
// Each returns 1 if it launched, 0 if the problem is outside what the kernel handles
// (the caller then uses the warp-MMA kernel), or -1 on a launch error (message from
// tc_last_error()).
#pragma once
#include "../../include/paged_gqa.h"
#include "common.cuh"

namespace pgqa {

int launch_verify_tc(const Problem& p, const Pointers& ptr, const ClassPlan& cp, const pg_tensor* k,
                     const pg_tensor* v, int sms, cudaStream_t stream);
int launch_prefill_tc(const Problem& p, const Pointers& ptr, const ClassPlan& cp, const pg_tensor* k,
                      const pg_tensor* v, int sms, cudaStream_t stream);
const char* tc_last_error();

}  // namespace pgqa
