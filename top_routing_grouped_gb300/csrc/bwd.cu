// bwd.cu -- the non-GEMM kernels of the backward pass.
//
// For L = sum_t dy[t] . y[t] + alpha * aux ("Distributed Training Part 4 ... MoE + Expert
// Parallelism", jesamkim ai-tech-blog, §3: the balancing loss is added to the training loss
// and acts mainly on the router):
//   gather_dy    dYp[p] = dy[t_p] and dOp[p] = gate_p * dy[t_p]   (the dispatch of dy)
//   router_bwd   dg_j = sum of the per-tile partials of dy . o  (fixed order);
//                dp_e = sum_j [idx_j = e] dg_j (renormalised gates: (dg_j - sum g dg) / S)
//                       + alpha E f_e / T;  dz = p (dp - p . dp);  dlogit = dz / tau
//   dx           dx[t] = sum_j dXslot[t k + j] + sum_e dlogit[t, e] W_r[e]
//   dwr          dW_r[e] = sum_t dlogit[t, e] x[t],  dbias[e] = sum_t dlogit[t, e]
//                (split over token chunks; the chunks are added in a fixed order)
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

// One warp per token: read dy[t] once, write its k dispatched rows (plain and gate-scaled).
__global__ void __launch_bounds__(kGatherWarps * 32) gather_dy_kernel(Shape s, Ws ws, const void* dy) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = (int64_t)blockIdx.x * kGatherWarps + (threadIdx.x >> 5);
  const int64_t nwarps = (int64_t)gridDim.x * kGatherWarps;
  const int v8 = s.d / 8;
  pdl_wait();
  pdl_launch_dependents();
  for (int64_t t = warp; t < s.T; t += nwarps) {
    int64_t my_p = -1;
    float my_g = 0.f;
    if (lane < s.k) {
      my_p = ws.slot_pos[t * s.k + lane];
      if (my_p < 0 || my_p >= s.N) {
        record_error(ws, MOE_ERR_INTERNAL, 0x900u);
        my_p = -1;
      } else {
        my_g = ws.gate_perm[my_p];
      }
    }
    for (int v = lane; v < v8; v += 32) {
      float f[8];
      load8(dy, s.out_bf16, t * v8 + v, f);
      for (int j = 0; j < s.k; ++j) {
        const int64_t p = __shfl_sync(0xffffffffu, my_p, j);
        const float g = __shfl_sync(0xffffffffu, my_g, j);
        if (p < 0) continue;
        reinterpret_cast<uint4*>(ws.dyp)[p * v8 + v] = pack8(f, 1.f);
        reinterpret_cast<uint4*>(ws.dop)[p * v8 + v] = pack8(f, g);
      }
    }
  }
}

// One thread per token: dlogit[t, :] (fp32).
__global__ void __launch_bounds__(128) router_bwd_kernel(Shape s, Ws ws, float alpha, int n_tiles_dh) {
  extern __shared__ float dp_s[];  // [128][E+1]
  const int r = threadIdx.x;
  const int64_t t = (int64_t)blockIdx.x * 128 + r;
  const int E = s.E, k = s.k;
  pdl_wait();
  pdl_launch_dependents();
  if (t >= s.T) return;
  float* dp = dp_s + r * (E + 1);
  // balancing-loss term: d(alpha * aux)/dp[t,e] = alpha * E * f_e / T
  for (int e = 0; e < E; ++e) dp[e] = alpha * (float)E * ((float)ws.counts[e] / ((float)s.T * (float)k)) / (float)s.T;
  const float* pt = ws.probs + t * E;
  float dg[kMaxTopK];
  float gdg = 0.f, S = 0.f;
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) {
    dg[j] = 0.f;
    if (j >= k) continue;
    const int64_t p = ws.slot_pos[t * k + j];
    if (p >= 0 && p < s.N)
      for (int n = 0; n < n_tiles_dh; ++n) dg[j] += ws.dgp[p * n_tiles_dh + n];  // tiles in order
    const int e = ws.topk_idx[t * k + j];
    if (e < 0 || e >= E) continue;
    gdg += ws.topk_gate[t * k + j] * dg[j];
    S += pt[e];
  }
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) {
    if (j >= k) continue;
    const int e = ws.topk_idx[t * k + j];
    if (e < 0 || e >= E) continue;
    dp[e] += s.renorm ? (dg[j] - gdg) / S : dg[j];  // renormalised gates: g_j = p_j / S
  }
  float pdp = 0.f;
  for (int e = 0; e < E; ++e) pdp += pt[e] * dp[e];
  for (int e = 0; e < E; ++e) ws.dlogit[t * E + e] = pt[e] * (dp[e] - pdp) / s.tau;
}

// dx[t, c] = sum_j dXslot[t k + j, c] + sum_e dlogit[t, e] W_r[e, c].  Tiles of 64 tokens x
// 128 columns, 256 threads each holding 4 tokens x 8 columns in registers; dlogit and W_r
// staged in shared memory over E in chunks of 32.
constexpr int kDxT = 64, kDxC = 128, kDxE = 32;
__global__ void __launch_bounds__(256) dx_kernel(Shape s, Ws ws, const void* w_router, float* dx) {
  __shared__ float zl[kDxE][kDxT + 4];  // transposed: zl[e][t]
  __shared__ float wr[kDxE][kDxC + 4];
  const int tid = threadIdx.x;
  const int tg = tid / 16, cg = tid % 16;  // tokens tg*4.., columns cg*8..
  const int64_t t0 = (int64_t)blockIdx.y * kDxT;
  const int c0 = blockIdx.x * kDxC;
  pdl_wait();
  pdl_launch_dependents();
  float acc[4][8];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
  for (int e0 = 0; e0 < s.E; e0 += kDxE) {
    for (int i = tid; i < kDxT * kDxE; i += 256) {
      const int tt = i / kDxE, ee = i % kDxE;
      const int64_t t = t0 + tt;
      zl[ee][tt] = (t < s.T && e0 + ee < s.E) ? ws.dlogit[t * s.E + e0 + ee] : 0.f;
    }
    for (int i = tid; i < kDxE * kDxC; i += 256) {
      const int ee = i / kDxC, cc = i % kDxC;
      wr[ee][cc] = (e0 + ee < s.E && c0 + cc < s.d) ? load_act(w_router, 1, (int64_t)(e0 + ee) * s.d + c0 + cc) : 0.f;
    }
    __syncthreads();
#pragma unroll 4
    for (int ee = 0; ee < kDxE; ++ee) {
      const float4 za = *reinterpret_cast<const float4*>(&zl[ee][tg * 4]);
      const float4 w0 = *reinterpret_cast<const float4*>(&wr[ee][cg * 8]);
      const float4 w1 = *reinterpret_cast<const float4*>(&wr[ee][cg * 8 + 4]);
      const float zv[4] = {za.x, za.y, za.z, za.w};
      const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(zv[i], wv[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t t = t0 + tg * 4 + i;
    if (t >= s.T) continue;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int c = c0 + cg * 8 + j;
      if (c >= s.d) continue;
      float v = acc[i][j];
      for (int q = 0; q < s.k; ++q)
        v += __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(ws.dxslot)[(t * s.k + q) * s.d + c]);
      dx[t * s.d + c] = v;
    }
  }
}

// Partial router-weight gradients over chunks of kDwrTok tokens: part[chunk][e][c] and
// part_b[chunk][e] for a tile of 64 experts x 128 columns (each thread 4 experts x 8
// columns); a second kernel adds the chunks in order.
constexpr int kDwrTok = 512, kDwrE = 64, kDwrC = 128, kDwrK = 32;
__global__ void __launch_bounds__(256) dwr_partial_kernel(Shape s, Ws ws, const void* x, float* part, float* part_b) {
  __shared__ float zl[kDwrK][kDwrE + 4];
  __shared__ float xs[kDwrK][kDwrC + 4];
  const int tid = threadIdx.x;
  const int eg = tid / 16, cg = tid % 16;
  const int c0 = blockIdx.x * kDwrC;
  const int e0 = blockIdx.y * kDwrE;
  const int chunk = blockIdx.z;
  const int64_t tbeg = (int64_t)chunk * kDwrTok;
  pdl_wait();
  pdl_launch_dependents();
  float acc[4][8], bacc[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    bacc[i] = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
  }
  for (int64_t tb = tbeg; tb < tbeg + kDwrTok && tb < s.T; tb += kDwrK) {
    for (int i = tid; i < kDwrK * kDwrE; i += 256) {
      const int tt = i / kDwrE, ee = i % kDwrE;
      const int64_t t = tb + tt;
      zl[tt][ee] = (t < s.T && e0 + ee < s.E) ? ws.dlogit[t * s.E + e0 + ee] : 0.f;
    }
    for (int i = tid; i < kDwrK * kDwrC; i += 256) {
      const int tt = i / kDwrC, cc = i % kDwrC;
      const int64_t t = tb + tt;
      xs[tt][cc] = (t < s.T && c0 + cc < s.d) ? load_act(x, s.act_bf16, t * s.d + c0 + cc) : 0.f;
    }
    __syncthreads();
#pragma unroll 4
    for (int tt = 0; tt < kDwrK; ++tt) {
      const float4 za = *reinterpret_cast<const float4*>(&zl[tt][eg * 4]);
      const float4 x0 = *reinterpret_cast<const float4*>(&xs[tt][cg * 8]);
      const float4 x1 = *reinterpret_cast<const float4*>(&xs[tt][cg * 8 + 4]);
      const float zv[4] = {za.x, za.y, za.z, za.w};
      const float xv[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        bacc[i] += zv[i];
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(zv[i], xv[j], acc[i][j]);
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int e = e0 + eg * 4 + i;
    if (e >= s.E) continue;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int c = c0 + cg * 8 + j;
      if (c < s.d) part[((int64_t)chunk * s.E + e) * s.d + c] = acc[i][j];
    }
    if (blockIdx.x == 0 && cg == 0) part_b[(int64_t)chunk * s.E + e] = bacc[i];
  }
}

__global__ void __launch_bounds__(256) dwr_reduce_kernel(Shape s, const float* part, const float* part_b, int chunks,
                                                         float* dwr, float* dbias) {
  pdl_wait();
  pdl_launch_dependents();
  const int64_t n = (int64_t)s.E * s.d;
  for (int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x; i < n; i += (int64_t)gridDim.x * 256) {
    float v = 0.f;
    for (int ch = 0; ch < chunks; ++ch) v += part[(int64_t)ch * n + i];
    dwr[i] = v;
  }
  if (dbias && blockIdx.x == 0)
    for (int e = threadIdx.x; e < s.E; e += 256) {
      float v = 0.f;
      for (int ch = 0; ch < chunks; ++ch) v += part_b[(int64_t)ch * s.E + e];
      dbias[e] = v;
    }
}

int dwr_chunks(const Shape& s) { return (int)((s.T + kDwrTok - 1) / kDwrTok); }

cudaError_t launch_gather_dy(const Shape& s, const Ws& ws, const void* dy, int num_sms, bool pdl, cudaStream_t st) {
  int64_t blocks = (s.T + kGatherWarps - 1) / kGatherWarps;
  if (blocks > (int64_t)num_sms * 8) blocks = (int64_t)num_sms * 8;
  return launch_kernel(gather_dy_kernel, dim3((unsigned)blocks), dim3(kGatherWarps * 32), 0, st, pdl, 1, s, ws, dy);
}

cudaError_t launch_router_bwd(const Shape& s, const Ws& ws, float alpha, int n_tiles_dh, bool pdl, cudaStream_t st) {
  const size_t smem = sizeof(float) * 128 * (size_t)(s.E + 1);
  cudaError_t e = cudaFuncSetAttribute(router_bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_kernel(router_bwd_kernel, dim3((unsigned)s.nblk), dim3(128), smem, st, pdl, 1, s, ws, alpha, n_tiles_dh);
}

cudaError_t launch_dx(const Shape& s, const Ws& ws, const void* w_router, float* dx, bool pdl, cudaStream_t st) {
  const dim3 g((unsigned)((s.d + kDxC - 1) / kDxC), (unsigned)((s.T + kDxT - 1) / kDxT));
  return launch_kernel(dx_kernel, g, dim3(256), 0, st, pdl, 1, s, ws, w_router, dx);
}

cudaError_t launch_dwr(const Shape& s, const Ws& ws, const void* x, float* part, float* part_b, float* dwr, float* dbias,
                       int num_sms, bool pdl, cudaStream_t st) {
  const int chunks = dwr_chunks(s);
  const dim3 g((unsigned)((s.d + kDwrC - 1) / kDwrC), (unsigned)((s.E + kDwrE - 1) / kDwrE), (unsigned)chunks);
  cudaError_t e = launch_kernel(dwr_partial_kernel, g, dim3(256), 0, st, pdl, 1, s, ws, x, part, part_b);
  if (e != cudaSuccess) return e;
  return launch_kernel(dwr_reduce_kernel, dim3((unsigned)num_sms * 2), dim3(256), 0, st, true, 1, s,
                       (const float*)part, (const float*)part_b, chunks, dwr, dbias);
}

}  // namespace moe
