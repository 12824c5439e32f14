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
#include "tile_tables.cuh"

namespace moe {

constexpr int kSegThreads = kMaxExperts;  // one thread per segment (W * E_l <= 256)

// One CTA: segment counts (device input) -> counts, offsets, tile tables, header totals.  A
// negative count or a total beyond the plan's row capacity is reported (MOE_ERR_INTERNAL, site
// 0x740) and leaves empty tile tables, so that no GEMM reads outside the buffers.
__global__ void __launch_bounds__(kSegThreads) seg_scan_kernel(Shape s, Ws ws, const int32_t* seg_counts, int n_seg,
                                                               int n_local) {
  __shared__ int cnt_s[kMaxExperts], offs_s[kMaxExperts];
  __shared__ int scratch[kTileScratchInts];
  const int i = threadIdx.x;
  int cnt = i < n_seg ? seg_counts[i] : 0;
  const bool neg = cnt < 0;
  cnt_s[i] = neg ? 0 : cnt;
  if (__syncthreads_or(neg)) {
    if (i == 0) {
      record_error(ws, MOE_ERR_INTERNAL, 0x740u);
      ws.hdr[kHdrNumGroups] = 0;
      ws.hdr[kHdrNumMTiles] = 0;
      ws.hdr[kHdrNumPairs] = 0;
    }
    return;
  }
  build_tile_tables(s, ws, n_seg, n_local, cnt_s, offs_s, scratch, kSegThreads, /*exact=*/false, 0x740u);
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
