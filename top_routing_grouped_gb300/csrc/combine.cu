// combine.cu -- y[t] = sum_{j<k} Yp[slot_pos[t*k + j]], in j order, fp32 accumulation.
//
// After "Distributed Training Part 4 ... MoE + Expert Parallelism" (jesamkim ai-tech-blog),
// §3 output formula y = sum_{i in TopK} G(x)_i E_i(x) (the gate factor is already applied
// by the down-projection epilogue) and §4 Combine (expert outputs return to their token:
// Yp holds them in expert order, slot_pos[t*k + j] is the row of token t's j-th choice).
// A fixed summation order keeps y bit-reproducible (no float atomics).  A slot_pos entry
// outside the routed rows (a corrupt permutation) is clamped into them for the read and
// reported (MOE_ERR_INTERNAL, site 0x600 / 0x601) once per thread after its loop, so that
// the check adds no branch to the gather itself.
#include <cuda_bf16.h>

#include "device_common.cuh"

namespace moe {

constexpr int kCombThreads = 256;

// bf16 slots -> bf16 or fp32 y; 8 columns (one 16-byte load per slot) per thread-step.
template <bool kOutBf16>
__global__ void __launch_bounds__(kCombThreads) combine_bf16_kernel(Shape s, Ws ws, Weights w) {
  const int vec_per_row = s.d / 8;
  const int64_t total = s.T * (int64_t)vec_per_row;
  const int4* ys = reinterpret_cast<const int4*>(ws.yp);
  bool bad = false;
  pdl_wait();  // the down-projection's rows
  pdl_launch_dependents();
  for (int64_t i = (int64_t)blockIdx.x * kCombThreads + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * kCombThreads) {
    const int64_t t = i / vec_per_row;
    const int v = (int)(i % vec_per_row);
    float acc[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) acc[q] = 0.f;
    for (int j = 0; j < s.k; ++j) {
      // clamped into the routed rows, so that not even a corrupt permutation reads outside Yp
      const uint32_t sp = (uint32_t)__ldg(&ws.slot_pos[t * s.k + j]);
      bad |= sp >= (uint32_t)s.N;
      const int64_t row = min(sp, (uint32_t)(s.N - 1));
      int4 raw = __ldcs(ys + row * vec_per_row + v);
      const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 f = __bfloat1622float2(h2[q]);
        acc[2 * q] += f.x;
        acc[2 * q + 1] += f.y;
      }
    }
    if constexpr (kOutBf16) {
      int4 out;
      __nv_bfloat162* o2 = reinterpret_cast<__nv_bfloat162*>(&out);
#pragma unroll
      for (int q = 0; q < 4; ++q) o2[q] = __floats2bfloat162_rn(acc[2 * q], acc[2 * q + 1]);
      reinterpret_cast<int4*>(w.y)[t * vec_per_row + v] = out;
    } else {
      float4* yo = reinterpret_cast<float4*>(w.y) + (t * vec_per_row + v) * 2;
      yo[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
      yo[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    }
  }
  if (bad) record_error(ws, MOE_ERR_INTERNAL, 0x600u);
}

// fp32 slots -> fp32 or bf16 y; 4 columns per thread-step.
template <bool kOutBf16>
__global__ void __launch_bounds__(kCombThreads) combine_f32_kernel(Shape s, Ws ws, Weights w) {
  const int vec_per_row = s.d / 4;
  const int64_t total = s.T * (int64_t)vec_per_row;
  const float4* ys = reinterpret_cast<const float4*>(ws.yp);
  bool bad = false;
  pdl_wait();
  pdl_launch_dependents();
  for (int64_t i = (int64_t)blockIdx.x * kCombThreads + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * kCombThreads) {
    const int64_t t = i / vec_per_row;
    const int v = (int)(i % vec_per_row);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < s.k; ++j) {
      const uint32_t sp = (uint32_t)__ldg(&ws.slot_pos[t * s.k + j]);
      bad |= sp >= (uint32_t)s.N;
      const int64_t row = min(sp, (uint32_t)(s.N - 1));  // clamped
      const float4 f = ys[row * vec_per_row + v];
      acc.x += f.x;
      acc.y += f.y;
      acc.z += f.z;
      acc.w += f.w;
    }
    if constexpr (kOutBf16) {
      __nv_bfloat162* yo = reinterpret_cast<__nv_bfloat162*>(w.y) + (t * vec_per_row + v) * 2;
      yo[0] = __floats2bfloat162_rn(acc.x, acc.y);
      yo[1] = __floats2bfloat162_rn(acc.z, acc.w);
    } else {
      reinterpret_cast<float4*>(w.y)[t * vec_per_row + v] = acc;
    }
  }
  if (bad) record_error(ws, MOE_ERR_INTERNAL, 0x601u);
}

cudaError_t launch_combine(const Shape& s, const Ws& ws, const Weights& w, int num_sms, bool pdl, cudaStream_t st) {
  const int64_t per = s.act_bf16 ? 8 : 4;
  int64_t blocks = (s.T * (s.d / per) + kCombThreads - 1) / kCombThreads;
  // enough blocks that every vector has its own thread on the movers' sizes (the grid-stride
  // loop's iterations are not overlapped, so fewer, longer-lived threads are slower)
  const int64_t cap = (int64_t)num_sms * 64;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  const dim3 g((unsigned)blocks), b(kCombThreads);
  if (s.act_bf16)
    return s.out_bf16 ? launch_kernel(combine_bf16_kernel<true>, g, b, 0, st, pdl, 1, s, ws, w)
                      : launch_kernel(combine_bf16_kernel<false>, g, b, 0, st, pdl, 1, s, ws, w);
  return s.out_bf16 ? launch_kernel(combine_f32_kernel<true>, g, b, 0, st, pdl, 1, s, ws, w)
                    : launch_kernel(combine_f32_kernel<false>, g, b, 0, st, pdl, 1, s, ws, w);
}

}  // namespace moe
