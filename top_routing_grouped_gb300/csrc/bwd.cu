// bwd.cu -- the non-GEMM kernels of the backward pass.
//
// For L = sum_t dy[t] . y[t] + alpha * aux ("Distributed Training Part 4 ... MoE + Expert
// Parallelism", jesamkim ai-tech-blog, §3: the balancing loss is added to the training loss
// and acts mainly on the router):
//   gather_dy    dYp[p] = dy[t_p] and dOp[p] = gate_p * dy[t_p]   (the dispatch of dy)
//   router_bwd   dg_j = sum of the per-tile partials of dy . o  (fixed order);
//                dp_e = sum_j [idx_j = e] dg_j (renormalised gates: (dg_j - sum g dg) / S)
//                       + alpha E f_e / T;  dz = p (dp - p . dp);  dlogit = dz / tau
//   dx           dx[t] = sum_j dXslot[t k + j] + sum_e dlogit[t, e] W_r[e] (tensor cores,
//                bwd_tc.cu)
//   dwr          dW_r[e] = sum_t dlogit[t, e] x[t] (tensor cores, bwd_tc.cu, over token
//                chunks) and dbias[e] = sum_t dlogit[t, e] (per router block, here); the
//                partials are added in a fixed order
#include <cuda_bf16.h>

#include "device_common.cuh"

namespace moe {

constexpr int kGatherWarps = 8;

__device__ __forceinline__ void load8(const void* base, int out_bf16, int64_t i8, float* f) {
  if (out_bf16) {
    uint4 raw = reinterpret_cast<const uint4*>(base)[i8];
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float2 v = __bfloat1622float2(h[q]);
      f[2 * q] = v.x;
      f[2 * q + 1] = v.y;
    }
  } else {
    const float4* p = reinterpret_cast<const float4*>(base) + 2 * i8;
    const float4 a = p[0], b = p[1];
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
    f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
  }
}

__device__ __forceinline__ uint4 pack8(const float* f, float scale) {
  uint4 o;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
  for (int q = 0; q < 4; ++q) h[q] = __floats2bfloat162_rn(scale * f[2 * q], scale * f[2 * q + 1]);
  return o;
}

// One warp per token: read dy[t] once, write its k dispatched rows (plain and gate-scaled; a
// gate-scaled row in its expert's last, partial 64-row block also to dop_tail).  Then the
// warps zero the rows of dop_tail and dab_tail past each expert's end.
__global__ void __launch_bounds__(kGatherWarps * 32) gather_dy_kernel(Shape s, Ws ws, const void* dy) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = (int64_t)blockIdx.x * kGatherWarps + (threadIdx.x >> 5);
  const int64_t nwarps = (int64_t)gridDim.x * kGatherWarps;
  const int v8 = s.d / 8;
  pdl_wait();
  pdl_launch_dependents();
  for (int64_t t = warp; t < s.T; t += nwarps) {
    int64_t my_p = -1, my_tr = -1;  // row in dyp / dop, row in dop_tail (or -1)
    float my_g = 0.f;
    if (lane < s.k) {
      my_p = ws.slot_pos[t * s.k + lane];
      const int e = ws.topk_idx[t * s.k + lane];
      if (my_p < 0 || my_p >= s.N || e < 0 || e >= s.E) {
        record_error(ws, MOE_ERR_INTERNAL, 0x900u);
        my_p = -1;
      } else {
        my_g = ws.gate_perm[my_p];
        my_tr = tail_row(e, my_p, ws.offsets[e], ws.counts[e]);
      }
    }
    for (int v = lane; v < v8; v += 32) {
      float f[8];
      load8(dy, s.out_bf16, t * v8 + v, f);
      for (int j = 0; j < s.k; ++j) {
        const int64_t p = __shfl_sync(0xffffffffu, my_p, j);
        const int64_t tr = __shfl_sync(0xffffffffu, my_tr, j);
        const float g = __shfl_sync(0xffffffffu, my_g, j);
        if (p < 0) continue;
        reinterpret_cast<uint4*>(ws.dyp)[p * v8 + v] = pack8(f, 1.f);
        const uint4 o = pack8(f, g);
        reinterpret_cast<uint4*>(ws.dop)[p * v8 + v] = o;
        if (tr >= 0) reinterpret_cast<uint4*>(ws.dop_tail)[tr * v8 + v] = o;
      }
    }
  }
  // rows r of expert e's tail block at or past its count there are zero
  const int f8 = (2 * s.F) / 8;
  const uint4 z = make_uint4(0u, 0u, 0u, 0u);
  for (int64_t u = warp; u < (int64_t)s.E * 64; u += nwarps) {
    const int e = (int)(u / 64), r = (int)(u % 64);
    const int rem = ws.counts[e] % 64;
    if (rem == 0 || r < rem) continue;  // no tail block, or a routed row
    for (int v = lane; v < v8; v += 32) reinterpret_cast<uint4*>(ws.dop_tail)[u * v8 + v] = z;
    for (int v = lane; v < f8; v += 32) reinterpret_cast<uint4*>(ws.dab_tail)[u * f8 + v] = z;
  }
}

// dlogit[t, :] for a block of 128 tokens, one thread per token.  The block's softmax rows are
// staged in shared memory with coalesced loads (rows padded to E + 1 floats, so the threads'
// row walks hit 32 different banks), each thread turns its row into dlogit in place, and the
// block writes dlogit (fp32) and its two bf16 terms with coalesced stores.
//   dp[e] = c_e + delta_e,  c_e = alpha E f_e / T (balancing loss),  delta_e = the gradient of
//   the loss through gate j when e = idx[t, j] (renormalised gates: (dg_j - sum_i g_i dg_i) / S);
//   dlogit[e] = p[e] (dp[e] - sum_e' p[e'] dp[e']) / tau  (softmax backward, temperature tau).
template <int KS>  // top-k capacity of the per-thread arrays (k <= KS)
__global__ void __launch_bounds__(128) router_bwd_kernel(Shape s, Ws ws, float alpha, int n_tiles_dh) {
  extern __shared__ float smem_f[];
  const int E = s.E, k = s.k, ldp = E + 1;
  float* c_s = smem_f;        // [E] balancing-loss term of each expert
  float* p_s = smem_f + E;    // [128][E + 1] softmax rows, then dlogit rows
  const int r = threadIdx.x;
  const int64_t t0 = (int64_t)blockIdx.x * 128;
  const int rows = (int)(s.T - t0 < 128 ? s.T - t0 : 128);
  pdl_wait();
  pdl_launch_dependents();
  for (int e = r; e < E; e += 128) c_s[e] = alpha * (float)E * ((float)ws.counts[e] / ((float)s.T * (float)k)) / (float)s.T;
  const float* pg = ws.probs + t0 * E;
  for (int i = r; i < rows * E; i += 128) p_s[(i / E) * ldp + i % E] = pg[i];
  __syncthreads();
  if (r < rows) {
    const int64_t t = t0 + r;
    float* pr = p_s + r * ldp;
    int idx[KS];
    float dg[KS], pe[KS];
    float gdg = 0.f, S = 0.f;
#pragma unroll
    for (int j = 0; j < KS; ++j) {
      dg[j] = 0.f;
      idx[j] = -1;
      pe[j] = 0.f;
      if (j >= k) continue;
      const int64_t p = ws.slot_pos[t * k + j];
      if (p >= 0 && p < s.N)
        for (int n = 0; n < n_tiles_dh; ++n) dg[j] += ws.dgp[p * n_tiles_dh + n];  // tiles in order
      const int e = ws.topk_idx[t * k + j];
      if (e < 0 || e >= E) continue;
      idx[j] = e;
      pe[j] = pr[e];
      gdg += ws.topk_gate[t * k + j] * dg[j];
      S += pe[j];
    }
    // delta of each chosen expert, and sum_e p[e] dp[e] in expert order
#pragma unroll
    for (int j = 0; j < KS; ++j)
      if (j < k) dg[j] = s.renorm ? (dg[j] - gdg) / S : dg[j];
    float pdp = 0.f;
    for (int e = 0; e < E; ++e) {
      float dp = c_s[e];
#pragma unroll
      for (int j = 0; j < KS; ++j)
        if (j < k && idx[j] == e) dp += dg[j];
      pdp += pr[e] * dp;
    }
    for (int e = 0; e < E; ++e) pr[e] = pr[e] * (c_s[e] - pdp) / s.tau;
#pragma unroll
    for (int j = 0; j < KS; ++j) {  // the chosen experts add their delta (once per expert)
      if (j >= k || idx[j] < 0) continue;
      float dp = c_s[idx[j]];
      bool first = true;
#pragma unroll
      for (int i = 0; i < KS; ++i) {
        if (i >= k || idx[i] != idx[j]) continue;
        if (i < j) first = false;
        dp += dg[i];
      }
      if (first) pr[idx[j]] = pe[j] * (dp - pdp) / s.tau;
    }
  }
  __syncthreads();
  // dlogit in fp32, and as two bf16 terms (columns past E zero) for the tensor-core products
  float* dl = ws.dlogit + t0 * E;
  for (int i = r; i < rows * E; i += 128) dl[i] = p_s[(i / E) * ldp + i % E];
  const int ec = dlogit_cols(s);  // a multiple of 64
  __nv_bfloat162* hi = reinterpret_cast<__nv_bfloat162*>(reinterpret_cast<__nv_bfloat16*>(ws.dl_hi) + t0 * ec);
  __nv_bfloat162* lo = reinterpret_cast<__nv_bfloat162*>(reinterpret_cast<__nv_bfloat16*>(ws.dl_lo) + t0 * ec);
  for (int i = r; i < rows * (ec / 2); i += 128) {
    const int row = i / (ec / 2), e = 2 * (i % (ec / 2));
    const float v0 = e < E ? p_s[row * ldp + e] : 0.f;
    const float v1 = e + 1 < E ? p_s[row * ldp + e + 1] : 0.f;
    const __nv_bfloat162 h = __floats2bfloat162_rn(v0, v1);
    const float2 hf = __bfloat1622float2(h);
    hi[i] = h;
    lo[i] = __floats2bfloat162_rn(v0 - hf.x, v1 - hf.y);
  }
}

// The router-bias gradient of each router block: part_b[blk, e] = sum over the block's
// tokens of dlogit[t, e], in token order.
// Sum of n values strided by `stride`, in index order; the loads of each group of 8 are issued
// together so that their latencies overlap (the additions keep the sequential order).
__device__ __forceinline__ float ordered_sum(const float* p, int64_t stride, int n) {
  float v = 0.f;
  int i = 0;
  for (; i + 8 <= n; i += 8) {
    float x[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) x[u] = p[(int64_t)(i + u) * stride];
#pragma unroll
    for (int u = 0; u < 8; ++u) v += x[u];
  }
  for (; i < n; ++i) v += p[(int64_t)i * stride];
  return v;
}

__global__ void __launch_bounds__(128) dbias_block_kernel(Shape s, Ws ws) {
  pdl_wait();
  pdl_launch_dependents();
  const int64_t t0 = (int64_t)blockIdx.x * 128;
  const int rows = (int)(s.T - t0 < 128 ? s.T - t0 : 128);
  for (int e = threadIdx.x; e < s.E; e += 128)
    ws.dwr_part_b[(int64_t)blockIdx.x * s.E + e] = ordered_sum(ws.dlogit + t0 * s.E + e, s.E, rows);
}

// dW_r = sum of the token-chunk partials in chunk order; dbias = sum of the router-block
// partials in block order
__global__ void __launch_bounds__(256) dwr_reduce_kernel(Shape s, const float* part, const float* part_b, int chunks,
                                                         float* dwr, float* dbias) {
  pdl_wait();
  pdl_launch_dependents();
  const int64_t n = (int64_t)s.E * s.d;
  for (int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x; i < n; i += (int64_t)gridDim.x * 256)
    dwr[i] = ordered_sum(part + i, n, chunks);
  if (dbias && blockIdx.x == 0)
    for (int e = threadIdx.x; e < s.E; e += 256) dbias[e] = ordered_sum(part_b + e, s.E, s.nblk);
}

cudaError_t launch_gather_dy(const Shape& s, const Ws& ws, const void* dy, int num_sms, bool pdl, cudaStream_t st) {
  int64_t blocks = (s.T + kGatherWarps - 1) / kGatherWarps;
  if (blocks > (int64_t)num_sms * 8) blocks = (int64_t)num_sms * 8;
  return launch_kernel(gather_dy_kernel, dim3((unsigned)blocks), dim3(kGatherWarps * 32), 0, st, pdl, 1, s, ws, dy);
}

cudaError_t launch_router_bwd(const Shape& s, const Ws& ws, float alpha, int n_tiles_dh, bool pdl, cudaStream_t st) {
  const size_t smem = sizeof(float) * ((size_t)s.E + 128 * (size_t)(s.E + 1));
  auto kern = s.k <= 2 ? router_bwd_kernel<2> : s.k <= 4 ? router_bwd_kernel<4>
                                             : s.k <= 8 ? router_bwd_kernel<8> : router_bwd_kernel<kMaxTopK>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_kernel(kern, dim3((unsigned)s.nblk), dim3(128), smem, st, pdl, 1, s, ws, alpha, n_tiles_dh);
}

cudaError_t launch_dwr_reduce(const Shape& s, const Ws& ws, float* dwr, float* dbias, int num_sms, bool pdl,
                              cudaStream_t st) {
  cudaError_t e = cudaSuccess;
  if (dbias) e = launch_kernel(dbias_block_kernel, dim3((unsigned)s.nblk), dim3(128), 0, st, pdl, 1, s, ws);
  if (e != cudaSuccess) return e;
  return launch_kernel(dwr_reduce_kernel, dim3((unsigned)num_sms * 2), dim3(256), 0, st, pdl, 1, s,
                       (const float*)ws.dwr_part, (const float*)ws.dwr_part_b, dwr_chunks(s), dwr, dbias);
}

}  // namespace moe
