// permute.cu -- dispatch on one GPU: every routed slot (t, j) gets its row
// p = blk_base[block(t), e] + local_rank(t, j) in expert-contiguous order, and x[t] is
// copied to Xp[p] for each of its k slots.
//
// After "Distributed Training Part 4 ... MoE + Expert Parallelism" (jesamkim ai-tech-blog),
// §4 Dispatch: the all-to-all that sends each token to the device of its expert; with all
// experts on one device it becomes this permutation inside HBM.
//
// One warp per token: the row is read once with 16-byte vector loads (issued first), the k
// destinations are computed by lanes 0..k-1 and broadcast, and the row is written k times
// (x is read once).
#include "device_common.cuh"

namespace moe {

constexpr int kPermWarps = 8;
constexpr int kPermVec = 8;  // 16-byte vectors per lane in flight (a 4 KB row per warp)

__global__ void __launch_bounds__(kPermWarps * 32) permute_kernel(Shape s, Ws ws, Weights w) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = (int64_t)blockIdx.x * kPermWarps + (threadIdx.x >> 5);
  const int64_t nwarps = (int64_t)gridDim.x * kPermWarps;
  const int esz = s.act_bf16 ? 2 : 4;
  const int vecs = s.d * esz / 16;  // 16-byte vectors per row (d * esz is a multiple of 16)
  const int k = s.k;
  pdl_wait();  // bases of the scan, ranks and choices of the router
  pdl_launch_dependents();

  for (int64_t t = warp; t < s.T; t += nwarps) {
    // the row's first 32 x 8 vectors are requested before the routing lookups, so that the
    // two latencies overlap
    const int4* src = reinterpret_cast<const int4*>(reinterpret_cast<const char*>(w.x) + t * (int64_t)s.d * esz);
    int4 buf[kPermVec];
#pragma unroll
    for (int u = 0; u < kPermVec; ++u) {
      const int v = u * 32 + lane;
      if (v < vecs) buf[u] = __ldcs(src + v);
    }
    int64_t my_p = -1;
    if (lane < k) {
      const int64_t slot = t * k + lane;
      const int e = ws.topk_idx[slot];
      int64_t p = -1;
      if (e >= 0 && e < s.E) p = (int64_t)ws.blk_base[(t / kRouteBlock) * s.E + e] + ws.local_rank[slot];
      if (p < 0 || p >= s.N) {
        record_error(ws, MOE_ERR_INTERNAL, 0x300u);
        p = -1;
      } else {
        ws.perm_src[p] = (int32_t)t;
        ws.perm_slot[p] = (int32_t)slot;
        ws.gate_perm[p] = ws.topk_gate[slot];
      }
      ws.slot_pos[slot] = (int32_t)p;
      my_p = p;
    }
    int64_t dst[kMaxTopK];
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) dst[j] = __shfl_sync(0xffffffffu, my_p, j);

    int4* xp = reinterpret_cast<int4*>(ws.xp);
    for (int v0 = 0;;) {
#pragma unroll
      for (int j = 0; j < kMaxTopK; ++j) {
        if (j < k && dst[j] >= 0) {
#pragma unroll
          for (int u = 0; u < kPermVec; ++u) {
            const int v = v0 + u * 32 + lane;
            if (v < vecs) xp[dst[j] * vecs + v] = buf[u];
          }
        }
      }
      v0 += 32 * kPermVec;
      if (v0 >= vecs) break;
#pragma unroll
      for (int u = 0; u < kPermVec; ++u) {
        const int v = v0 + u * 32 + lane;
        if (v < vecs) buf[u] = __ldcs(src + v);
      }
    }
  }
}

cudaError_t launch_permute(const Shape& s, const Ws& ws, const Weights& w, int num_sms, bool pdl, cudaStream_t st) {
  int64_t blocks = (s.T + kPermWarps - 1) / kPermWarps;
  const int64_t cap = (int64_t)num_sms * 8;
  if (blocks > cap) blocks = cap;
  return launch_kernel(permute_kernel, dim3((unsigned)blocks), dim3(kPermWarps * 32), 0, st, pdl, 1, s, ws, w);
}

}  // namespace moe
