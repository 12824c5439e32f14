// route_common.cuh -- the part of the router shared by its SIMT and tensor-core forms:
// everything after the logits are known.
#pragma once
#include <float.h>

#include "device_common.cuh"

namespace moe {

__device__ __forceinline__ void named_barrier(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Called by exactly kRouteBlock threads (r = 0..127, one per token row of the block) once
// z_s[r * ldz + e] holds the finished logit z = (x.W_r[e] + b_e)/tau of token blk*128 + r.
//   1. per token: p = softmax(z) (fp32, expf), top-k by descending z with ties to the
//      lower expert (a fixed insertion network over kMaxTopK slots, strict '>'),
//      gates p[idx] (divided by their sum over the k chosen in the renormalised variant);
//      writes topk_idx / topk_gate (and the logits when kept);
//   2. per block: for every expert, a bitmask of the block's tokens that chose it; the
//      slot's rank among the block's slots of the same expert is the popcount of the
//      tokens before it (stable in token order, deterministic);
//   3. per block and expert: the count and the sum of p over the block's tokens, summed
//      in row order.
// mask_s needs 4 * E words.  z_s rows are overwritten with p.
__device__ __forceinline__ void route_finish(const Shape& s, const Ws& ws, int blk, int r, float* z_s,
                                             int ldz, uint32_t* mask_s, int bar_id) {
  const int E = s.E, k = s.k;
  const int64_t t = (int64_t)blk * kRouteBlock + r;
  const bool valid = t < s.T;
  for (int i = r; i < 4 * E; i += kRouteBlock) mask_s[i] = 0u;
  named_barrier(bar_id, kRouteBlock);

  float* zr = z_s + r * ldz;
  int bi[kMaxTopK];
  if (valid) {
    float bv[kMaxTopK];
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
      bv[j] = -INFINITY;
      bi[j] = -1;
    }
    float m = -INFINITY;
    for (int e = 0; e < E; ++e) {
      const float v = zr[e];
      if (s.keep_logits) ws.logits[t * E + e] = v;
      m = fmaxf(m, v);
      // insertion into the descending slots; strict '>' keeps the lower index on ties
#pragma unroll
      for (int j = kMaxTopK - 1; j > 0; --j) {
        if (v > bv[j - 1]) {
          bv[j] = bv[j - 1];
          bi[j] = bi[j - 1];
        } else if (v > bv[j]) {
          bv[j] = v;
          bi[j] = e;
        }
      }
      if (v > bv[0]) {
        bv[0] = v;
        bi[0] = e;
      }
    }
    // Only non-finite logits leave a chosen slot empty: flag it and fill the slot with the
    // lowest unused expert so every later index stays in range and distinct.
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
      if (j < k && bi[j] < 0) {
        record_error(ws, MOE_ERR_INTERNAL, 0x100u);
        for (int e = 0; e < E; ++e) {
          bool used = false;
#pragma unroll
          for (int q = 0; q < kMaxTopK; ++q) used |= (q < j && bi[q] == e);
          if (!used) {
            bi[j] = e;
            break;
          }
        }
      }
    }
    float sum = 0.f;
    for (int e = 0; e < E; ++e) {
      const float q = expf(zr[e] - m);
      zr[e] = q;
      sum += q;
    }
    for (int e = 0; e < E; ++e) {
      zr[e] = zr[e] / sum;
      if (s.training) ws.probs[t * E + e] = zr[e];
    }
    float chosen = 1.f;  // sum of the chosen entries, in slot order (renormalised variant)
    if (s.renorm) {
      chosen = 0.f;
#pragma unroll
      for (int j = 0; j < kMaxTopK; ++j)
        if (j < k) chosen += zr[bi[j]];
    }
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
      if (j < k) {
        const int e = bi[j];
        ws.topk_idx[t * k + j] = e;
        ws.topk_gate[t * k + j] = s.renorm ? zr[e] / chosen : zr[e];
        atomicOr(&mask_s[e * 4 + (r >> 5)], 1u << (r & 31));
      }
    }
  } else {
    for (int e = 0; e < E; ++e) zr[e] = 0.f;
  }
  named_barrier(bar_id, kRouteBlock);

  if (valid) {
    const uint32_t below = (1u << (r & 31)) - 1u;
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
      if (j < k) {
        const uint32_t* mk = mask_s + bi[j] * 4;
        int rank = __popc(mk[r >> 5] & below);
        for (int wd = 0; wd < (r >> 5); ++wd) rank += __popc(mk[wd]);
        ws.local_rank[t * k + j] = rank;
      }
    }
  }
  for (int e = r; e < E; e += kRouteBlock) {
    const uint32_t* mk = mask_s + e * 4;
    ws.blk_cnt[(int64_t)blk * E + e] = __popc(mk[0]) + __popc(mk[1]) + __popc(mk[2]) + __popc(mk[3]);
    float ps = 0.f;
    for (int rr = 0; rr < kRouteBlock; ++rr) ps += z_s[rr * ldz + e];
    ws.blk_psum[(int64_t)blk * E + e] = ps;
  }
}

}  // namespace moe
