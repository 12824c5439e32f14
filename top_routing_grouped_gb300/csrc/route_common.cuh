// route_common.cuh -- the part of the router shared by its SIMT and tensor-core forms:
// everything after the logits are known.
#pragma once
#include <float.h>

#include "device_common.cuh"

namespace moe {

__device__ __forceinline__ void named_barrier(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Called by exactly kRouteBlock threads (r = 0..127, one per token row of the block; the
// four warps r>>5 = 0..3) once z_s[r * ldz + e] holds the finished logit
// z = (x.W_r[e] + b_e)/tau of token blk*128 + r (ldz odd, so that both a row and a column
// walk are free of bank conflicts).
//   1. per token, top-k by descending z with ties to the lower expert: a pass over the E
//      logits keeps the k largest VALUES in descending registers (each new value moves
//      into place by a max/min network, no index traffic); a second pass marks, 32 experts
//      at a time, those at or above the k-th value, and each marked expert, in ascending
//      order, takes the first free slot at its value's rank (equal to the k-th value only
//      while such slots remain) -- the same choice as taking the best remaining expert k
//      times with the lower index on ties, in two passes;
//      the second pass also sums q_e = exp(z_e - max) (the softmax denominator); the gates
//      are q/sum at the chosen experts (divided by their sum over the k in the
//      renormalised variant);  writes topk_idx / topk_gate (and the logits when kept);
//   2. per block: for every expert, a bitmask of the block's tokens that chose it; the
//      slot's rank among the block's slots of the same expert is the popcount of the
//      tokens before it (stable in token order, deterministic);
//   3. per block and expert: the count, and the sum over the block's tokens of
//      p = exp(z - max) * (1/sum) (each warp owns every fourth group of four experts; a
//      lane adds rows lane, +32, +64, +96 in that order, then a fixed butterfly over the
//      lanes -- the same order on every run).
// mask_s needs 4 * E + 2 * kRouteBlock words.  z_s is only read.
// A NaN logit is reported (MOE_ERR_INTERNAL) and ranked as -inf.
template <int KS>
__device__ __forceinline__ void route_finish_k(const Shape& s, const Ws& ws, int blk, int r, float* z_s, int ldz,
                                               uint32_t* mask_s, int bar_id) {
  const int E = s.E, k = s.k;
  const int64_t t = (int64_t)blk * kRouteBlock + r;
  const bool valid = t < s.T;
  for (int i = r; i < 4 * E; i += kRouteBlock) mask_s[i] = 0u;
  named_barrier(bar_id, kRouteBlock);  // every mask word is clear before any bit is set
  // z_s is read through shared-window addresses (see ld_shared_f32)
  const uint32_t zr = static_cast<uint32_t>(__cvta_generic_to_shared(z_s + r * ldz));
  float m = 0.f, sum = 1.f;
  int bi[KS];
  if (valid) {
    // pass 1: the KS largest values, descending (bv[0] is the row maximum); fmaxf(z, -inf)
    // ranks a NaN as -inf
    float bv[KS];
#pragma unroll
    for (int j = 0; j < KS; ++j) bv[j] = -INFINITY;
    bool nan_seen = false;
    for (int e0 = 0; e0 < E; e0 += 8) {
      // eight loads in flight, then eight insertions (past E: -inf, which changes nothing)
      float z8[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) z8[u] = e0 + u < E ? ld_shared_f32(zr + 4u * (uint32_t)(e0 + u)) : -INFINITY;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (s.keep_logits && e0 + u < E) ws.logits[t * E + e0 + u] = z8[u];
        nan_seen |= (z8[u] != z8[u]);
        const float v = fmaxf(z8[u], -INFINITY);
#pragma unroll
        for (int j = KS - 1; j > 0; --j) bv[j] = fmaxf(bv[j], fminf(v, bv[j - 1]));
        bv[0] = fmaxf(bv[0], v);
      }
    }
    if (nan_seen) record_error(ws, MOE_ERR_INTERNAL, 0x100u);
    m = bv[0];
    // the k-th value: the least of the first k (taken as a min rather than bv[k-1] so that
    // bv stays in registers)
    float thr = INFINITY;
#pragma unroll
    for (int j = 0; j < KS; ++j)
      if (j < k) thr = fminf(thr, bv[j]);
    int eq_left = k;  // slots still open for logits equal to the k-th value
#pragma unroll
    for (int j = 0; j < KS; ++j) eq_left -= (j < k && bv[j] > thr) ? 1 : 0;
    // pass 2, 32 experts at a time: the softmax denominator, and a bitmask of the experts
    // at or above the k-th value; then those, in ascending order, take their slots
#pragma unroll
    for (int j = 0; j < KS; ++j) bi[j] = -1;
    uint32_t filled = 0u;
    sum = 0.f;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int n = E - e0 < 32 ? E - e0 : 32;
      uint32_t take = 0u;
      int i = 0;
      for (; i + 4 <= n; i += 4) {  // four loads in flight, then four exponentials
        float v4[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) v4[u] = fmaxf(ld_shared_f32(zr + 4u * (uint32_t)(e0 + i + u)), -INFINITY);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          sum += expf(v4[u] - m);
          take |= (v4[u] >= thr ? 1u : 0u) << (i + u);
        }
      }
      for (; i < n; ++i) {
        const float v = fmaxf(ld_shared_f32(zr + 4u * (uint32_t)(e0 + i)), -INFINITY);
        sum += expf(v - m);
        take |= (v >= thr ? 1u : 0u) << i;
      }
      while (take) {
        const int e = e0 + __ffs(take) - 1;
        take &= take - 1u;
        const float v = fmaxf(ld_shared_f32(zr + 4u * (uint32_t)e), -INFINITY);
        if (v == thr) {
          if (eq_left == 0) continue;
          --eq_left;
        }
        int pos0 = 0;
#pragma unroll
        for (int j = 0; j < KS; ++j) pos0 += (j < k && bv[j] > v) ? 1 : 0;
        const int pos = __ffs(~filled & (0xffffffffu << pos0)) - 1;
        if (pos >= 0 && pos < k) {
          filled |= 1u << pos;
#pragma unroll
          for (int j = 0; j < KS; ++j)
            if (j == pos) bi[j] = e;
        }
      }
    }
    // every slot is filled by construction; should one not be, report it and give it the
    // lowest unused expert so that every later index stays in range and distinct
    if (filled != (1u << k) - 1u) {
      record_error(ws, MOE_ERR_INTERNAL, 0x101u);
#pragma unroll
      for (int j = 0; j < KS; ++j) {
        if (j < k && bi[j] < 0) {
          for (int e = 0; e < E; ++e) {
            bool used = false;
#pragma unroll
            for (int q = 0; q < KS; ++q) used |= (q < k && bi[q] == e);
            if (!used) {
              bi[j] = e;
              break;
            }
          }
        }
      }
    }
    float gate[KS];
    float chosen = 0.f;  // sum of the chosen gates, in slot order (renormalised variant)
#pragma unroll
    for (int j = 0; j < KS; ++j) {
      gate[j] = j < k ? expf(fmaxf(ld_shared_f32(zr + 4u * (uint32_t)bi[j]), -INFINITY) - m) / sum : 0.f;
      chosen += gate[j];
    }
#pragma unroll
    for (int j = 0; j < KS; ++j) {
      if (j < k) {
        const int e = bi[j];
        ws.topk_idx[t * k + j] = e;
        ws.topk_gate[t * k + j] = s.renorm ? gate[j] / chosen : gate[j];
        atomicOr(&mask_s[e * 4 + (r >> 5)], 1u << (r & 31));
      }
    }
  }
  // the row maximum and 1/sum of every row, for the column pass below
  float* m_s = reinterpret_cast<float*>(mask_s + 4 * E);
  float* inv_s = m_s + kRouteBlock;
  m_s[r] = m;
  inv_s[r] = 1.f / sum;
  named_barrier(bar_id, kRouteBlock);

  if (valid) {
    const uint32_t below = (1u << (r & 31)) - 1u;
#pragma unroll
    for (int j = 0; j < KS; ++j) {
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
  }
  // per-expert sums of p = exp(z - max) / sum over the block's rows (rows past T add 0)
  const int w = r >> 5, lane = r & 31;
  const int64_t t_base = (int64_t)blk * kRouteBlock;
  float mrow[4], inv[4];
  bool vrow[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    mrow[j] = m_s[lane + 32 * j];
    inv[j] = inv_s[lane + 32 * j];
    vrow[j] = t_base + lane + 32 * j < s.T;
  }
  const uint32_t zc = static_cast<uint32_t>(__cvta_generic_to_shared(z_s + lane * ldz));
  // warp w takes the groups of four experts g = w, w + 4, ...: sixteen loads in flight,
  // then four interleaved butterflies
  for (int e0 = 4 * w; e0 < E; e0 += 16) {
    float zz[4][4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int u = 0; u < 4; ++u)
        zz[j][u] = e0 + u < E ? ld_shared_f32(zc + 4u * (uint32_t)(32 * j * ldz + e0 + u)) : 0.f;
    float ps[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int row = lane + 32 * j;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float p = vrow[j] ? expf(fmaxf(zz[j][u], -INFINITY) - mrow[j]) * inv[j] : 0.f;
        if (s.training && vrow[j] && e0 + u < E) ws.probs[(t_base + row) * E + e0 + u] = p;
        ps[u] += p;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
#pragma unroll
      for (int u = 0; u < 4; ++u) ps[u] += __shfl_xor_sync(0xffffffffu, ps[u], off);
    if (lane == 0)
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (e0 + u < E) ws.blk_psum[(int64_t)blk * E + e0 + u] = ps[u];
  }
}

// mask_s needs 4 * E + 2 * kRouteBlock words (the bitmasks, then two floats per row).
__device__ __forceinline__ void route_finish(const Shape& s, const Ws& ws, int blk, int r, float* z_s, int ldz,
                                             uint32_t* mask_s, int bar_id) {
  if (s.k <= 2) route_finish_k<2>(s, ws, blk, r, z_s, ldz, mask_s, bar_id);
  else if (s.k <= 4) route_finish_k<4>(s, ws, blk, r, z_s, ldz, mask_s, bar_id);
  else if (s.k <= 8) route_finish_k<8>(s, ws, blk, r, z_s, ldz, mask_s, bar_id);
  else route_finish_k<kMaxTopK>(s, ws, blk, r, z_s, ldz, mask_s, bar_id);
}

}  // namespace moe
