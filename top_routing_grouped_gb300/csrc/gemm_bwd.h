// gemm_bwd.h -- launchers of the backward's grouped GEMMs on CTA pairs.
#pragma once
#include <cuda_runtime.h>

#include "moe_internal.h"

namespace moe {

// kind kBwdDH or kBwdDX (gemm_tc.h) on 2-SM CTA pairs over the forward's pair tile table;
// same operands and results as launch_gemm_bwd for those kinds.
cudaError_t launch_gemm_bwd_pair(int kind, const Shape& s, const Ws& ws, const Weights& w, int num_sms,
                                 int64_t timeout_ns, bool pdl, cudaStream_t st);

}  // namespace moe
