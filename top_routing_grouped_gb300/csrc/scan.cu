// scan.cu -- per-expert histogram totals, exclusive scan, per-(block, expert) dispatch
// bases, the grouped-GEMM tile table and the balancing scalar.
//
// After "Distributed Training Part 4 ... MoE + Expert Parallelism" (jesamkim ai-tech-blog):
// §4 Dispatch (every routed row needs a destination; on one GPU the destination is its
// position in an expert-contiguous order, offsets[e] + rank) and §3 Load-Balancing Loss
// (aux = E * sum_e f_e P_e with f_e = count_e / (T k), P_e = mean over tokens of p[t,e]).
#include "device_common.cuh"

namespace moe {

constexpr int kScanThreads = kMaxExperts;   // one thread per expert for the scans over experts
constexpr int kScanBlock = 1024;            // at most: the loops over router blocks

// Exclusive scan of one int per thread (threads 0..kScanThreads-1) over the experts; returns
// the thread's prefix and writes the total to *total.  Hillis-Steele in shared memory
// (log2(256) = 8 steps); every thread of the CTA calls it (the barriers need all of them).
__device__ int block_exclusive_scan(int v, int* buf, int* total) {
  const int i = threadIdx.x;
  if (i < kScanThreads) buf[i] = v;
  __syncthreads();
  for (int off = 1; off < kScanThreads; off <<= 1) {
    const int add = (i < kScanThreads && i >= off) ? buf[i - off] : 0;
    __syncthreads();
    if (i < kScanThreads) buf[i] += add;
    __syncthreads();
  }
  const int incl = i < kScanThreads ? buf[i] : 0;
  *total = buf[kScanThreads - 1];
  __syncthreads();
  return incl - v;
}

// The router blocks are cut into chunks, one per thread of an expert's team (tpe threads per
// expert, tpe = blockDim / E rounded down to a power of two): per-chunk counts and sums of p, then
// per-expert totals and chunk prefixes (in chunk order), then the per-(block, expert) bases.
__global__ void __launch_bounds__(kScanBlock) scan_kernel(Shape s, Ws ws) {
  __shared__ int buf[kScanThreads];
  __shared__ float red[kScanThreads];
  __shared__ int ccnt[kScanBlock];    // [chunk][expert slot] counts, then their exclusive prefix
  __shared__ float cps[kScanBlock];   // [chunk][expert slot] sums of p
  __shared__ int tot_cnt[kScanThreads];
  __shared__ float tot_ps[kScanThreads];
  const int E = s.E;
  int ep = 1;  // expert slots: E rounded up to a power of two
  while (ep < E) ep <<= 1;
  const int tpe = (int)blockDim.x / ep;  // threads (block chunks) per expert
  const int te = threadIdx.x % ep, tc = threadIdx.x / ep;
  const int per = (s.nblk + tpe - 1) / tpe;
  const int b0 = tc * per, b1 = b0 + per < s.nblk ? b0 + per : s.nblk;
  pdl_wait();  // per-block counts and sums of the router
  pdl_launch_dependents();

  {
    int c = 0;
    float p = 0.f;
    if (te < E)
      for (int b = b0; b < b1; ++b) {
        c += ws.blk_cnt[(int64_t)b * E + te];
        p += ws.blk_psum[(int64_t)b * E + te];
      }
    ccnt[threadIdx.x] = c;
    cps[threadIdx.x] = p;
  }
  __syncthreads();
  if (threadIdx.x < E) {  // totals and chunk prefixes of expert e, in chunk order
    const int e = threadIdx.x;
    int run = 0;
    float ps = 0.f;
    for (int c = 0; c < tpe; ++c) {
      const int v = ccnt[c * ep + e];
      ccnt[c * ep + e] = run;
      run += v;
      ps += cps[c * ep + e];
    }
    tot_cnt[e] = run;
    tot_ps[e] = ps;
  }
  __syncthreads();

  const int e = threadIdx.x;
  const bool on = e < E;
  const int cnt = on ? tot_cnt[e] : 0;
  const float psum = on ? tot_ps[e] : 0.f;
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
    if (e == 0) {
      record_error(ws, MOE_ERR_INTERNAL, 0x200u);
      ws.hdr[kHdrNumGroups] = 0;
      ws.hdr[kHdrNumMTiles] = 0;
      ws.hdr[kHdrNumPairs] = 0;
    }
    return;
  }
  if (on) {
    ws.counts[e] = cnt;
    ws.offsets[e] = off;
    for (int g = 0; g < ng; ++g) {
      const int gm = g + 1 < ng ? kGroupM : last_gm;  // m-tiles of this group
      const int gp = (gm + 1) / 2;                      // and pairs
      const int m0 = mstart + g * kGroupM, p0 = pstart + g * (kGroupM / 2);
      const int row0 = off + g * kGroupM * kTileM;
      for (int i = 0; i < gm; ++i) ws.mt_desc[m0 + i] = make_int4(e | (gm << 20), m0, row0, off + cnt);
      for (int i = 0; i < gp; ++i) ws.pr_desc[p0 + i] = make_int4(e | (gp << 20), p0, row0, off + cnt);
    }
    buf[e] = off;  // the experts' offsets, for the per-block bases below
  }
  if (e == 0) {
    ws.offsets[E] = n_routed;
    ws.hdr[kHdrNumGroups] = (uint32_t)n_groups;
    ws.hdr[kHdrNumMTiles] = (uint32_t)n_mtiles;
    ws.hdr[kHdrNumPairs] = (uint32_t)n_pairs;
  }
  __syncthreads();
  // per-(block, expert) bases: every chunk of every expert from its prefix
  if (te < E) {
    int run = buf[te] + ccnt[threadIdx.x];
    for (int b = b0; b < b1; ++b) {
      ws.blk_base[(int64_t)b * E + te] = run;
      run += ws.blk_cnt[(int64_t)b * E + te];
    }
  }

  // aux = E * sum_e f_e * P_e, reduced over a fixed tree (deterministic)
  const float f = on ? (float)cnt / ((float)s.T * (float)s.k) : 0.f;
  const float P = on ? psum / (float)s.T : 0.f;
  if (e < kScanThreads) red[e] = f * P;
  __syncthreads();
  for (int half = kScanThreads / 2; half > 0; half >>= 1) {
    if (e < half) red[e] += red[e + half];
    __syncthreads();
  }
  if (e == 0) *ws.aux = (float)E * red[0];
}

cudaError_t launch_scan(const Shape& s, const Ws& ws, bool pdl, cudaStream_t st) {
  // enough threads for one router block per chunk, 256 .. 1024 (a power of two)
  int ep = 1;
  while (ep < s.E) ep <<= 1;
  int threads = kScanThreads;
  while (threads < kScanBlock && threads < ep * s.nblk) threads <<= 1;
  return launch_kernel(scan_kernel, dim3(1), dim3(threads), 0, st, pdl, 1, s, ws);
}

}  // namespace moe
