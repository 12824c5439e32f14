// ep_scan.cu -- the tile table of the expert stage of expert parallelism, and the balancing
// scalar from totals summed over ranks.
//
// After "Distributed Training Part 4 ... MoE + Expert Parallelism" (jesamkim ai-tech-blog),
// §4 Expert Parallelism: the experts are spread over the GPUs; Dispatch sends every routed
// row to the rank that holds its expert, the experts run there, and Combine sends the outputs
// back.  A rank's dispatch order is already expert-contiguous, so what one rank sends to
// another is a run of rows grouped by expert; the rows a rank receives from W sources are
// therefore W * E_l contiguous segments in source-major order: segment s holds the rows that
// source s / E_l sent to local expert s % E_l.  The expert GEMMs run on them in place, one
// scheduling group per segment piece, with the segment's local expert as the weight index --
// rows of one expert that came from different sources never share a tile, and nothing is
// copied into expert order first.
#include "device_common.cuh"

namespace moe {

constexpr int kSegThreads = kMaxExperts;  // one thread per segment (W * E_l <= 256)

// One CTA: segment counts (device input) -> counts, offsets, tile descriptors, header totals.
// A negative count or a total beyond the plan's row capacity is reported (MOE_ERR_INTERNAL,
// site 0x700) and leaves an empty tile table, so that no GEMM reads outside the buffers.
__global__ void __launch_bounds__(kSegThreads) seg_scan_kernel(Shape s, Ws ws, const int32_t* seg_counts, int n_seg,
                                                               int n_local) {
  __shared__ int wtot[4][kSegThreads / 32];  // warp totals of count, m-tiles, groups, pairs
  const int i = threadIdx.x, lane = i & 31, w = i >> 5;
  int cnt = i < n_seg ? seg_counts[i] : 0;
  const bool neg = cnt < 0;
  if (neg) cnt = 0;
  const int mt = (cnt + kTileM - 1) / kTileM;
  const int ng = (mt + kGroupM - 1) / kGroupM;
  const int last_gm = mt - (ng - 1) * kGroupM;
  const int np = ng > 0 ? (ng - 1) * (kGroupM / 2) + (last_gm + 1) / 2 : 0;
  const int own[4] = {cnt, mt, ng, np};
  int incl[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    int v = own[q];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += n;
    }
    incl[q] = v;
    if (lane == 31) wtot[q][w] = v;
  }
  const bool any_neg = __syncthreads_or(neg);
  int base[4], total[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    base[q] = 0;
    total[q] = 0;
    for (int ww = 0; ww < kSegThreads / 32; ++ww) {
      if (ww < w) base[q] += wtot[q][ww];
      total[q] += wtot[q][ww];
    }
  }
  const int n_rows = total[0], n_mtiles = total[1], n_groups = total[2], n_pairs = total[3];
  if (any_neg || n_rows > s.N || n_groups > s.max_groups) {
    if (i == 0) {
      record_error(ws, MOE_ERR_INTERNAL, 0x700u);
      ws.hdr[kHdrNumGroups] = 0;
      ws.hdr[kHdrNumMTiles] = 0;
      ws.hdr[kHdrNumPairs] = 0;
    }
    return;
  }
  if (i < n_seg) {
    const int off = base[0] + incl[0] - cnt;
    const int mstart = base[1] + incl[1] - mt, pstart = base[3] + incl[3] - np;
    const int we = i % n_local;  // the segment's local expert: the weight index of its tiles
    ws.counts[i] = cnt;
    ws.offsets[i] = off;
    for (int g = 0; g < ng; ++g) {
      const int gm = g + 1 < ng ? kGroupM : last_gm;
      const int gp = (gm + 1) / 2;
      const int m0 = mstart + g * kGroupM, p0 = pstart + g * (kGroupM / 2);
      const int row0 = off + g * kGroupM * kTileM;
      for (int j = 0; j < gm; ++j) ws.mt_desc[m0 + j] = make_int4(we | (gm << 20), m0, row0, off + cnt);
      for (int j = 0; j < gp; ++j) ws.pr_desc[p0 + j] = make_int4(we | (gp << 20), p0, row0, off + cnt);
    }
  }
  if (i == 0) {
    ws.offsets[n_seg] = n_rows;
    ws.hdr[kHdrNumGroups] = (uint32_t)n_groups;
    ws.hdr[kHdrNumMTiles] = (uint32_t)n_mtiles;
    ws.hdr[kHdrNumPairs] = (uint32_t)n_pairs;
  }
}

cudaError_t launch_seg_scan(const Shape& s, const Ws& ws, const int32_t* seg_counts, int n_seg, int n_local,
                            cudaStream_t st) {
  return launch_kernel(seg_scan_kernel, dim3(1), dim3(kSegThreads), 0, st, false, 1, s, ws, seg_counts, n_seg, n_local);
}

// aux = E * sum_e (count_e / (T k)) * (psum_e / T) from per-expert totals (counts and sums of
// the softmax over every token of every rank), reduced over the same fixed tree as the
// router's scan.
__global__ void __launch_bounds__(kMaxExperts) aux_totals_kernel(int E, int k, int64_t T, const int32_t* counts,
                                                                 const float* psum, float* aux_out) {
  __shared__ float red[kMaxExperts];
  const int e = threadIdx.x;
  red[e] = e < E ? ((float)counts[e] / ((float)T * (float)k)) * (psum[e] / (float)T) : 0.f;
  __syncthreads();
  for (int half = kMaxExperts / 2; half > 0; half >>= 1) {
    if (e < half) red[e] += red[e + half];
    __syncthreads();
  }
  if (e == 0) *aux_out = (float)E * red[0];
}

cudaError_t launch_aux_totals(int E, int k, int64_t T, const int32_t* counts, const float* psum, float* aux_out,
                              cudaStream_t st) {
  aux_totals_kernel<<<1, kMaxExperts, 0, st>>>(E, k, T, counts, psum, aux_out);
  return cudaGetLastError();
}

}  // namespace moe
