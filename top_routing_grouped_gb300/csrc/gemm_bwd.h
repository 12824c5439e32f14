// gemm_bwd.h -- launchers of the backward's grouped GEMMs on CTA pairs.
#pragma once
#include <cuda_runtime.h>

#include "moe_internal.h"

namespace moe {

// kind kBwdDH or kBwdDX (gemm_tc.h) on 2-SM CTA pairs over the forward's pair tile table;
// same operands and results as launch_gemm_bwd for those kinds.
cudaError_t launch_gemm_bwd_pair(int kind, const Shape& s, const Ws& ws, const Weights& w, int num_sms,
                                 int64_t timeout_ns, bool pdl, cudaStream_t st);

// kind kBwdDW13 (dw_a = dW1, dw_b = dW3) or kBwdDW2 (dw_a = dW2) on 2-SM CTA pairs; same
// results as launch_gemm_bwd for those kinds.
cudaError_t launch_gemm_dw_pair(int kind, const Shape& s, const Ws& ws, float* dw_a, float* dw_b, int num_sms,
                                int64_t timeout_ns, bool pdl, cudaStream_t st);

// Router-weight gradient partials ws.dwr_part [dwr_chunks, E, d] on the tensor cores, from
// ws.dl_hi / ws.dl_lo and x.
cudaError_t launch_dwr_tc(const Shape& s, const Ws& ws, const void* x, int64_t timeout_ns, bool pdl, cudaStream_t st);

// dx [T, d] fp32 = dlogit . W_r (tensor cores, from ws.dl_hi / ws.dl_lo) + the sum of the
// token's k rows of ws.dxslot.
cudaError_t launch_dx_tc(const Shape& s, const Ws& ws, const void* w_router, float* dx, int64_t timeout_ns, bool pdl,
                         cudaStream_t st);

}  // namespace moe
