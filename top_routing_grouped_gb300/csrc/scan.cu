// scan.cu -- per-expert histogram totals, exclusive scan, per-(block, expert) dispatch
// bases, the grouped-GEMM tile table and the balancing scalar.
//
// After "Distributed Training Part 4 ... MoE + Expert Parallelism" (jesamkim ai-tech-blog):
// §4 Dispatch (every routed row needs a destination; on one GPU the destination is its
// position in an expert-contiguous order, offsets[e] + rank) and §3 Load-Balancing Loss
// (aux = E * sum_e f_e P_e with f_e = count_e / (T k), P_e = mean over tokens of p[t,e]).
#include "device_common.cuh"

namespace moe {

constexpr int kScanThreads = kMaxExperts;  // one thread per expert

// Exclusive scan of one int per thread over the block; returns the thread's prefix and
// writes the total to *total.  Hillis-Steele in shared memory (log2(256) = 8 steps).
__device__ int block_exclusive_scan(int v, int* buf, int* total) {
  const int i = threadIdx.x;
  buf[i] = v;
  __syncthreads();
  for (int off = 1; off < kScanThreads; off <<= 1) {
    const int add = i >= off ? buf[i - off] : 0;
    __syncthreads();
    buf[i] += add;
    __syncthreads();
  }
  const int incl = buf[i];
  *total = buf[kScanThreads - 1];
  __syncthreads();
  return incl - v;
}

__global__ void __launch_bounds__(kScanThreads) scan_kernel(Shape s, Ws ws) {
  __shared__ int buf[kScanThreads];
  __shared__ float red[kScanThreads];
  const int e = threadIdx.x;
  const int E = s.E;
  const bool on = e < E;
  pdl_wait();  // per-block counts and sums of the router
  pdl_launch_dependents();

  int cnt = 0;
  float psum = 0.f;
  if (on) {
    for (int b = 0; b < s.nblk; ++b) {
      cnt += ws.blk_cnt[(int64_t)b * E + e];
      psum += ws.blk_psum[(int64_t)b * E + e];
    }
  }
  int n_routed;
  const int off = block_exclusive_scan(cnt, buf, &n_routed);
  const int mt = (cnt + kTileM - 1) / kTileM;
  const int ng = (mt + kGroupM - 1) / kGroupM;
  // m-tile pairs (for CTA pairs that share a weight tile): ceil(gm / 2) per group; every
  // group but an expert's last holds kGroupM (even) m-tiles
  const int last_gm = mt - (ng - 1) * kGroupM;
  const int np = ng > 0 ? (ng - 1) * (kGroupM / 2) + (last_gm + 1) / 2 : 0;
  int n_mtiles, n_groups, n_pairs;
  const int mstart = block_exclusive_scan(mt, buf, &n_mtiles);
  const int gstart = block_exclusive_scan(ng, buf, &n_groups);
  const int pstart = block_exclusive_scan(np, buf, &n_pairs);

  if (n_routed != s.N || n_groups > s.max_groups) {
    if (e == 0) record_error(ws, MOE_ERR_INTERNAL, 0x200u);
    if (e == 0) {
      ws.hdr[kHdrNumGroups] = 0;
      ws.hdr[kHdrNumMTiles] = 0;
      ws.hdr[kHdrNumPairs] = 0;
    }
    return;
  }
  if (on) {
    ws.counts[e] = cnt;
    ws.offsets[e] = off;
    int run = off;
    for (int b = 0; b < s.nblk; ++b) {
      ws.blk_base[(int64_t)b * E + e] = run;
      run += ws.blk_cnt[(int64_t)b * E + e];
    }
    for (int g = 0; g < ng; ++g) {
      ws.grp_expert[gstart + g] = e;
      ws.grp_mtile0[gstart + g] = g * kGroupM;
      ws.grp_mpre[gstart + g] = mstart + g * kGroupM;
      ws.grp_ppre[gstart + g] = pstart + g * (kGroupM / 2);
    }
  }
  if (e == 0) {
    ws.offsets[E] = n_routed;
    ws.grp_mpre[n_groups] = n_mtiles;
    ws.grp_ppre[n_groups] = n_pairs;
    ws.hdr[kHdrNumGroups] = (uint32_t)n_groups;
    ws.hdr[kHdrNumMTiles] = (uint32_t)n_mtiles;
    ws.hdr[kHdrNumPairs] = (uint32_t)n_pairs;
  }

  // aux = E * sum_e f_e * P_e, reduced over a fixed tree (deterministic)
  const float f = on ? (float)cnt / ((float)s.T * (float)s.k) : 0.f;
  const float P = on ? psum / (float)s.T : 0.f;
  red[e] = f * P;
  __syncthreads();
  for (int half = kScanThreads / 2; half > 0; half >>= 1) {
    if (e < half) red[e] += red[e + half];
    __syncthreads();
  }
  if (e == 0) *ws.aux = (float)E * red[0];
}

cudaError_t launch_scan(const Shape& s, const Ws& ws, bool pdl, cudaStream_t st) {
  return launch_kernel(scan_kernel, dim3(1), dim3(kScanThreads), 0, st, pdl, 1, s, ws);
}

}  // namespace moe
