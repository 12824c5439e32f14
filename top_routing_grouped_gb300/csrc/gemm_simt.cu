// gemm_simt.cu -- grouped expert GEMMs on the SIMT pipes (fp32 FMA): the true-fp32 path
// for fp32 layers, and a cross-check of the tensor-core path for bf16 layers.
//
// After "Distributed Training Part 4 ... MoE + Expert Parallelism" (jesamkim ai-tech-blog):
// §3 Structure (each expert is an independent FFN, SwiGLU form here: E_e(v) =
// W2_e (SiLU(W1_e v) * (W3_e v))), §3 output formula (the expert output is weighted by the
// router's gate) and §4 Combine (outputs go back to their token; here: to the token's
// slot t*k+j, summed per token by the combine kernel).
//
//   GEMM1 (kMode = 1): H[p, f]         = SiLU(Xp[p] . W1_e[f]) * (Xp[p] . W3_e[f])
//   GEMM2 (kMode = 2): Yp[p, c] = gate(p) * (H[p] . W2_e[c])   (row p in expert order)
// for every row p of expert e, over the tile table built by the scan kernel.
#include <cuda_bf16.h>

#include <type_traits>

#include "device_common.cuh"

namespace moe {

constexpr int kSimtBN = 64;
constexpr int kSimtBK = 16;
constexpr int kSimtThreads = 256;

template <int kMode, bool kBf16>
__global__ void __launch_bounds__(kSimtThreads) gemm_simt_kernel(Shape s, Ws ws, Weights w) {
  using Act = typename std::conditional<kBf16, __nv_bfloat16, float>::type;
  __shared__ __align__(16) float a_s[kSimtBK][kTileM + 4];
  __shared__ __align__(16) float b_s[kSimtBK][kSimtBN + 4];
  __shared__ __align__(16) float b3_s[kSimtBK][kSimtBN + 4];  // W3 tile (GEMM1 only)

  const int K = kMode == 1 ? s.d : s.F;       // reduction length
  const int ncols = kMode == 1 ? s.F : s.d;   // output columns
  const int n_tiles = (ncols + kSimtBN - 1) / kSimtBN;
  const Act* A = reinterpret_cast<const Act*>(kMode == 1 ? ws.xp : ws.h);
  const Act* B = reinterpret_cast<const Act*>(kMode == 1 ? w.w1 : w.w2);
  const Act* B3 = reinterpret_cast<const Act*>(w.w3);
  pdl_wait();  // tile table, permuted rows (or H) of the previous kernels
  pdl_launch_dependents();
  const int total = (int)ws.hdr[kHdrNumMTiles] * n_tiles;

  const int tid = threadIdx.x;
  const int tx = tid % 16, ty = tid / 16;  // 4 columns x 8 rows per thread

  for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
    const TileInfo ti = decode_tile(ws, n_tiles, tile);
    const int n0 = ti.n_idx * kSimtBN;
    const int64_t wrow0 = (int64_t)ti.e * ncols;  // first weight row of this expert
    float acc[8][4], acc3[8][4];  // acc3: W3 products (GEMM1 only; unused otherwise)
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][j] = acc3[i][j] = 0.f;

    for (int k0 = 0; k0 < K; k0 += kSimtBK) {
#pragma unroll
      for (int u = 0; u < kTileM * kSimtBK / kSimtThreads; ++u) {
        const int i = tid + u * kSimtThreads;
        const int row = i / kSimtBK, kk = i % kSimtBK;
        float v = 0.f;
        if (row < ti.rows && k0 + kk < K) v = (float)A[(int64_t)(ti.row0 + row) * K + k0 + kk];
        a_s[kk][row] = v;
      }
#pragma unroll
      for (int u = 0; u < kSimtBN * kSimtBK / kSimtThreads; ++u) {
        const int i = tid + u * kSimtThreads;
        const int n = i / kSimtBK, kk = i % kSimtBK;
        float v = 0.f, v3 = 0.f;
        if (n0 + n < ncols && k0 + kk < K) {
          const int64_t off = (wrow0 + n0 + n) * K + k0 + kk;
          v = (float)B[off];
          if constexpr (kMode == 1) v3 = (float)B3[off];
        }
        b_s[kk][n] = v;
        b3_s[kk][n] = v3;
      }
      __syncthreads();
#pragma unroll
      for (int kk = 0; kk < kSimtBK; ++kk) {
        float a[8], b[4], b3[4];
#pragma unroll
        for (int i = 0; i < 8; ++i) a[i] = a_s[kk][ty * 8 + i];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          b[j] = b_s[kk][tx * 4 + j];
          b3[j] = b3_s[kk][tx * 4 + j];
        }
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
            if constexpr (kMode == 1) acc3[i][j] = fmaf(a[i], b3[j], acc3[i][j]);
          }
      }
      __syncthreads();
    }

#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int row = ty * 8 + i;
      if (row >= ti.rows) continue;
      const int64_t p = ti.row0 + row;
      if constexpr (kMode == 1) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int c = n0 + tx * 4 + j;
          if (c >= ncols) continue;
          const float a = acc[i][j];
          const float hv = a / (1.0f + expf(-a)) * acc3[i][j];
          store_act(ws.h, kBf16, p * s.F + c, hv);
        }
      } else {
        const float g = ws.gate_perm[p];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int c = n0 + tx * 4 + j;
          if (c < ncols) store_act(ws.yp, kBf16, p * s.d + c, g * acc[i][j]);
        }
      }
    }
  }
}

template <int kMode>
static cudaError_t launch_simt(const Shape& s, const Ws& ws, const Weights& w, int num_sms, bool pdl, cudaStream_t st) {
  const dim3 g(num_sms * 4), b(kSimtThreads);
  return s.act_bf16 ? launch_kernel(gemm_simt_kernel<kMode, true>, g, b, 0, st, pdl, 1, s, ws, w)
                    : launch_kernel(gemm_simt_kernel<kMode, false>, g, b, 0, st, pdl, 1, s, ws, w);
}

cudaError_t launch_gemm1_simt(const Shape& s, const Ws& ws, const Weights& w, int num_sms, bool pdl, cudaStream_t st) {
  return launch_simt<1>(s, ws, w, num_sms, pdl, st);
}
cudaError_t launch_gemm2_simt(const Shape& s, const Ws& ws, const Weights& w, int num_sms, bool pdl, cudaStream_t st) {
  return launch_simt<2>(s, ws, w, num_sms, pdl, st);
}

}  // namespace moe
