// route_noalloc.cu -- routing for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at all: code running where an allocation would be
// unsafe or forbidden (inside a region whose memory budget is fixed in advance, in a
// runtime that owns every device allocation itself, or on a path that must not risk an
// allocation failure part-way through a step).  For them, moe_route_noalloc() runs the
// router, the top-k selection, the per-expert counts and the balancing scalar with all of
// its scratch memory in one statically sized device array defined in this file, so neither
// the caller nor the library allocates anything.  The caller passes only inputs and outputs.
//
// The scratch array is file-scope `static __device__`: every GPU that loads the library
// holds its kNoAllocScratchBytes until the process exits.  All calls share it and it keeps
// whatever the last call left there, so calls whose work overlaps on the GPU (two streams,
// or two host threads) race on it and must be serialised by the caller.
#include <cuda_runtime.h>
#include <stdio.h>

#include <mutex>

#include "device_common.cuh"
#include "route_common.cuh"

namespace moe {
namespace {

constexpr size_t kNoAllocScratchBytes = (size_t)MOE_NOALLOC_SCRATCH_BYTES;
constexpr int kChunk = 32;     // columns of d per shared-memory step of the logit loop
constexpr int kMaxDevices = 64;

// Scratch layout: [0, 256) the status header (the 64 words a workspace header has: the
// status word, the failure site, ...); [256, 512) the completion ticket; then the per-slot
// local ranks [T*k] int32, the per-block counts [nblk*E] int32 and softmax sums
// [nblk*E] fp32, each region starting on a 256-byte boundary.
static __device__ __align__(256) unsigned char g_route_scratch[kNoAllocScratchBytes];
constexpr size_t kTicketAt = 256, kRanksAt = 512;
static_assert(kTicketAt >= 64 * sizeof(uint32_t), "the status header holds 64 words");

size_t up256(size_t v) { return (v + 255) / 256 * 256; }

size_t scratch_needed(const Shape& s) {
  return kRanksAt + up256((size_t)s.N * 4) + 2 * up256((size_t)s.nblk * s.E * 4);
}

// Device address of g_route_scratch on each device, looked up once per device with that
// device current (the host-side name of the array is not a device address).
void* scratch_address(int device, cudaError_t* err) {
  static std::mutex mu;
  static void* addr[kMaxDevices] = {};
  std::lock_guard<std::mutex> lock(mu);
  if (device < 0 || device >= kMaxDevices) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  if (!addr[device]) {
    void* p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_route_scratch);
    if (*err != cudaSuccess) return nullptr;
    addr[device] = p;
  }
  *err = cudaSuccess;
  return addr[device];
}

// The router of moe_forward (fp32 FMA logits, then the shared softmax / top-k / per-block
// counting in route_finish) followed by a last-block reduction: the block that finishes
// last sums the per-block counts and softmax sums in block order and writes the expert
// counts and aux = E * sum_e f_e P_e, with the same summation order as the scan kernel.
// The last block also copies the status word (0, or the first error any block recorded:
// MOE_ERR_INTERNAL for a NaN logit) to *status_out.
__global__ void __launch_bounds__(kRouteBlock) route_noalloc_kernel(Shape s, Ws ws, Weights w, uint32_t* ticket,
                                                                    int32_t* counts_out, float* aux_out,
                                                                    uint32_t* status_out) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int ldz = s.E + 1;
  float* z_s = reinterpret_cast<float*>(smem_raw);                       // [128][E+1]
  float* x_s = z_s + kRouteBlock * ldz;                                   // [128][33]
  float* w_s = x_s + kRouteBlock * (kChunk + 1);                          // [E][33]
  uint32_t* mask_s = reinterpret_cast<uint32_t*>(w_s + s.E * (kChunk + 1));  // [E][4], then [2][128]
  __shared__ float red[kMaxExperts];
  __shared__ int last;

  const int r = threadIdx.x;
  const int blk = blockIdx.x;
  const int64_t t0 = (int64_t)blk * kRouteBlock;
  for (int e = 0; e < s.E; ++e) z_s[r * ldz + e] = 0.f;
  for (int c0 = 0; c0 < s.d; c0 += kChunk) {
    for (int i = r; i < kRouteBlock * kChunk; i += kRouteBlock) {
      const int row = i / kChunk, col = i % kChunk;
      const int64_t t = t0 + row;
      x_s[row * (kChunk + 1) + col] = (t < s.T && c0 + col < s.d) ? load_act(w.x, s.act_bf16, t * s.d + c0 + col) : 0.f;
    }
    for (int i = r; i < s.E * kChunk; i += kRouteBlock) {
      const int e = i / kChunk, col = i % kChunk;
      w_s[e * (kChunk + 1) + col] = (c0 + col < s.d) ? load_act(w.wr, s.act_bf16, (int64_t)e * s.d + c0 + col) : 0.f;
    }
    __syncthreads();
    const float* xr = x_s + r * (kChunk + 1);
    for (int e = 0; e < s.E; ++e) {
      const float* wr = w_s + e * (kChunk + 1);
      float acc = 0.f;
#pragma unroll
      for (int c = 0; c < kChunk; ++c) acc = fmaf(xr[c], wr[c], acc);
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

  // last block: totals over blocks in block order
  __threadfence();
  __syncthreads();
  if (r == 0) last = atomicAdd(ticket, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!last) return;
  __threadfence();
  for (int e = r; e < kMaxExperts; e += kRouteBlock) {
    float v = 0.f;
    if (e < s.E) {
      int cnt = 0;
      float psum = 0.f;
      for (int b = 0; b < s.nblk; ++b) {
        cnt += __ldcg(&ws.blk_cnt[(int64_t)b * s.E + e]);
        psum += __ldcg(&ws.blk_psum[(int64_t)b * s.E + e]);
      }
      counts_out[e] = cnt;
      v = ((float)cnt / ((float)s.T * (float)s.k)) * (psum / (float)s.T);
    }
    red[e] = v;
  }
  __syncthreads();
  for (int half = kMaxExperts / 2; half > 0; half >>= 1) {
    for (int e = r; e < half; e += kRouteBlock) red[e] += red[e + half];
    __syncthreads();
  }
  if (r == 0) {
    *aux_out = (float)s.E * red[0];
    *status_out = __ldcg(&ws.hdr[kHdrStatus]);
  }
}

thread_local char g_msg[256];

}  // namespace
}  // namespace moe

extern "C" moe_status moe_route_noalloc(moe_plan_t plan, const void* x, const void* w_router, const float* router_bias,
                                        int32_t* topk_idx, float* topk_gate, int32_t* expert_counts, float* aux,
                                        uint32_t* device_status, void* stream) {
  using namespace moe;
  // every argument check comes before the first CUDA call
  if (!plan || !x || !w_router || !topk_idx || !topk_gate || !expert_counts || !aux || !device_status) {
    snprintf(g_msg, sizeof g_msg, "moe_route_noalloc: null argument");
    return set_last_error(MOE_ERR_INVALID_ARG, g_msg);
  }
  const void* ptrs[] = {x, w_router, topk_idx, topk_gate, expert_counts, aux, device_status};
  for (const void* p : ptrs)
    if (reinterpret_cast<uintptr_t>(p) % 16 != 0) {
      snprintf(g_msg, sizeof g_msg, "moe_route_noalloc: every device pointer must be 16-byte aligned");
      return set_last_error(MOE_ERR_INVALID_ARG, g_msg);
    }
  if (!plan_is_layer(plan)) {
    snprintf(g_msg, sizeof g_msg, "moe_route_noalloc: needs a plan made by moe_plan");
    return set_last_error(MOE_ERR_INVALID_ARG, g_msg);
  }
  Shape s = *plan_shape(plan);
  if (s.has_bias && (!router_bias || reinterpret_cast<uintptr_t>(router_bias) % 16 != 0)) {
    snprintf(g_msg, sizeof g_msg, "moe_route_noalloc: the plan has a router bias: router_bias must be a 16-byte aligned pointer");
    return set_last_error(MOE_ERR_INVALID_ARG, g_msg);
  }
  const size_t need = scratch_needed(s);
  if (need > kNoAllocScratchBytes) {
    snprintf(g_msg, sizeof g_msg,
             "moe_route_noalloc: this shape needs %zu bytes of routing scratch but the static buffer holds %zu "
             "(MOE_NOALLOC_SCRATCH_BYTES); use moe_forward with a caller-owned workspace",
             need, kNoAllocScratchBytes);
    return set_last_error(MOE_ERR_UNSUPPORTED, g_msg);
  }
  // Only routing runs here: whatever else a plan's flags ask the forward to keep (logits,
  // the softmax a training plan keeps for its backward) has no place in the scratch and is
  // switched off, so that no store is gated on a region this call does not have.
  s.keep_logits = 0;
  s.training = 0;

  int dev = 0;
  unsigned char* base = nullptr;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) base = static_cast<unsigned char*>(scratch_address(dev, &e));
  if (e != cudaSuccess || !base) {
    snprintf(g_msg, sizeof g_msg, "moe_route_noalloc: looking up the scratch buffer: %s", cudaGetErrorString(e));
    return set_last_error(MOE_ERR_CUDA, g_msg);
  }
  Ws ws{};
  ws.hdr = reinterpret_cast<uint32_t*>(base);
  ws.local_rank = reinterpret_cast<int32_t*>(base + kRanksAt);
  ws.blk_cnt = reinterpret_cast<int32_t*>(base + kRanksAt + up256((size_t)s.N * 4));
  ws.blk_psum = reinterpret_cast<float*>(base + kRanksAt + up256((size_t)s.N * 4) + up256((size_t)s.nblk * s.E * 4));
  ws.topk_idx = topk_idx;
  ws.topk_gate = topk_gate;
  Weights w{x, w_router, s.has_bias ? router_bias : nullptr, nullptr, nullptr, nullptr, nullptr};

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the status header and the ticket must start at zero on every call
  if ((e = cudaMemsetAsync(base, 0, kRanksAt, st)) != cudaSuccess) {
    snprintf(g_msg, sizeof g_msg, "moe_route_noalloc: clearing the scratch header: %s", cudaGetErrorString(e));
    return set_last_error(MOE_ERR_CUDA, g_msg);
  }
  const size_t smem = sizeof(float) * ((size_t)kRouteBlock * (s.E + 1) + (size_t)kRouteBlock * (kChunk + 1) +
                                       (size_t)s.E * (kChunk + 1)) +
                      sizeof(uint32_t) * (4 * (size_t)s.E + 2 * kRouteBlock);
  if ((e = cudaFuncSetAttribute(route_noalloc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) ==
      cudaSuccess) {
    route_noalloc_kernel<<<s.nblk, kRouteBlock, smem, st>>>(s, ws, w, reinterpret_cast<uint32_t*>(base + kTicketAt),
                                                            expert_counts, aux, device_status);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) {
    snprintf(g_msg, sizeof g_msg, "moe_route_noalloc: launch: %s", cudaGetErrorString(e));
    return set_last_error(MOE_ERR_CUDA, g_msg);
  }
  return MOE_OK;
}
