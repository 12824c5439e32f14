// route.cu -- router: logits, softmax, top-k, gates, per-block histogram, local dispatch
// ranks and softmax partial sums for the balancing scalar; the last CTA to finish also runs
// the scan (route_scan.cuh).
//
// After "Distributed Training Part 4 ... MoE + Expert Parallelism" (jesamkim ai-tech-blog):
// §3 Structure (router = linear layer + softmax over experts; only the TopK experts are
// used, weighted by the router's probability), §3 Load-Balancing Loss (needs the mean
// router probability P_e and the routed fraction f_e per expert), §4 Dispatch (tokens go
// to their experts; here: a stable counting sort, whose per-block part is done here).
#include <cuda_bf16.h>
#include <float.h>

#include "device_common.cuh"
#include "route_common.cuh"
#include "route_scan.cuh"

namespace moe {

// SIMT router: one CTA per block of kRouteBlock tokens, one thread per token.  The
// logits are accumulated in shared memory in chunks of 32 columns of d (fp32 FMA).
constexpr int kRouteChunk = 32;

__global__ void __launch_bounds__(kRouteBlock) route_simt_kernel(Shape s, Ws ws, Weights w) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int ldz = s.E + 1;
  float* z_s = reinterpret_cast<float*>(smem_raw);                  // [128][E+1]
  float* x_s = z_s + kRouteBlock * ldz;                              // [128][33]
  float* w_s = x_s + kRouteBlock * (kRouteChunk + 1);                // [E][33]
  uint32_t* mask_s = reinterpret_cast<uint32_t*>(w_s + s.E * (kRouteChunk + 1));  // [E][4], then [2][128]

  const int r = threadIdx.x;
  const int blk = blockIdx.x;
  pdl_launch_dependents();
  const int64_t t0 = (int64_t)blk * kRouteBlock;
  for (int e = 0; e < s.E; ++e) z_s[r * ldz + e] = 0.f;

  for (int c0 = 0; c0 < s.d; c0 += kRouteChunk) {
    for (int i = r; i < kRouteBlock * kRouteChunk; i += kRouteBlock) {
      const int row = i / kRouteChunk, col = i % kRouteChunk;
      const int64_t t = t0 + row;
      float v = 0.f;
      if (t < s.T && c0 + col < s.d) v = load_act(w.x, s.act_bf16, t * s.d + c0 + col);
      x_s[row * (kRouteChunk + 1) + col] = v;
    }
    for (int i = r; i < s.E * kRouteChunk; i += kRouteBlock) {
      const int e = i / kRouteChunk, col = i % kRouteChunk;
      float v = 0.f;
      if (c0 + col < s.d) v = load_act(w.wr, s.act_bf16, (int64_t)e * s.d + c0 + col);
      w_s[e * (kRouteChunk + 1) + col] = v;
    }
    __syncthreads();
    const float* xr = x_s + r * (kRouteChunk + 1);
    for (int e = 0; e < s.E; ++e) {
      const float* wr = w_s + e * (kRouteChunk + 1);
      float acc = 0.f;
#pragma unroll
      for (int c = 0; c < kRouteChunk; ++c) acc = fmaf(xr[c], wr[c], acc);
      z_s[r * ldz + e] += acc;
    }
    __syncthreads();
  }
  for (int e = 0; e < s.E; ++e) {
    float v = z_s[r * ldz + e];
    if (s.has_bias) v += w.bias[e];
    z_s[r * ldz + e] = v / s.tau;
  }
  route_finish(s, ws, blk, r, z_s, ldz, mask_s, /*bar_id=*/1);
  __syncthreads();  // the block's shared tables are no longer needed: the scan may reuse them
  route_scan_if_last(s, ws, kRouteBlock, s.nblk, smem_raw);
}

size_t route_simt_smem(const Shape& s) {
  const size_t body = sizeof(float) * ((size_t)kRouteBlock * (s.E + 1) + (size_t)kRouteBlock * (kRouteChunk + 1) +
                                       (size_t)s.E * (kRouteChunk + 1)) +
                      sizeof(uint32_t) * (4 * (size_t)s.E + 2 * kRouteBlock);
  const size_t scan = route_scan_smem(s, kRouteBlock);
  return body > scan ? body : scan;
}

cudaError_t launch_route_simt(const Shape& s, const Ws& ws, const Weights& w, cudaStream_t st) {
  const size_t smem = route_simt_smem(s);
  cudaError_t err = cudaFuncSetAttribute(route_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  route_simt_kernel<<<s.nblk, kRouteBlock, smem, st>>>(s, ws, w);
  return cudaGetLastError();
}

}  // namespace moe
