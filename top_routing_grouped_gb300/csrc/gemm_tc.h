// gemm_tc.h -- tensor-core (tcgen05 / TMEM / TMA) kernels for sm_103a.
#pragma once
#include "moe_internal.h"

namespace moe {

// bf16 layers on MOE_PATH_AUTO run the tcgen05 kernels.
constexpr bool kTensorCorePathBuilt = true;

#include <cuda.h>

// Tensor map of a row-major bf16 [rows, cols] matrix, boxes of [box_rows, 64] elements with
// 128-byte swizzling (the K-major operand layout of the tcgen05 kernels).
cudaError_t make_tmap_bf16(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows);

// 2-SM version (CTA pairs, tcgen05.mma.cta_group::2): same arguments and results.
constexpr int kPairAccBufs = 2;  // TMEM accumulators per pair CTA (x 256 columns): double-buffered
cudaError_t launch_gemm_tc_pair(int mode, const Shape& s, const Ws& ws, const Weights& w, int num_sms,
                                int64_t timeout_ns, bool test_stall, bool pdl, cudaStream_t st);

// Backward grouped GEMMs (gemm_bwd.cu).
enum : int { kBwdDH = 0, kBwdDX = 1, kBwdDW13 = 2, kBwdDW2 = 3 };
cudaError_t launch_gemm_bwd(int kind, const Shape& s, const Ws& ws, const Weights& w, float* dw_a, float* dw_b,
                            int num_sms, int64_t timeout_ns, bool pdl, cudaStream_t st);

cudaError_t launch_route_tc(const Shape& s, const Ws& ws, const Weights& w, int num_sms, int64_t timeout_ns,
                            cudaStream_t st);
// mode 1: H = SiLU(Xp W1^T) * (Xp W3^T); mode 2: Yp = gate * (H W2^T) (expert order)
cudaError_t launch_gemm_tc(int mode, const Shape& s, const Ws& ws, const Weights& w, int num_sms,
                           int64_t timeout_ns, bool test_stall, bool pdl, cudaStream_t st);

}  // namespace moe
