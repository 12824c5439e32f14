// route_tc.cu -- the router on the tensor cores: logits of 128 tokens x E experts per CTA
// with tcgen05.mma (x tile [128 x 64] and W_r tile [E_pad x 64] per stage, TMA-fed, fp32
// accumulators in TMEM), then the shared softmax / top-k / per-block counting epilogue.
//
// After "Distributed Training Part 4 ... MoE + Expert Parallelism" (jesamkim ai-tech-blog),
// §3 Structure: the router is a linear layer followed by a softmax over the experts.  The
// layer streams x once (2 bytes per element against 2E flops), so it is bound by HBM, not by
// the MMA; the tensor cores only keep the E dot products per token off the SIMT pipes.
//
// Warp roles (64 + 128 Q threads, Q = 2 or 4): warp 0 TMA producer, warp 1 TMEM allocator +
// MMA issuer, warps 2..2+4Q-1 epilogue, Q per TMEM lane quarter (warp w reads lanes
// 32*(w%4)..: rows of its 32 tokens), one for each of Q contiguous ranges of the experts; each
// token is finished by Q threads (Q = 4 when E > 64, where the per-token top-k and softmax
// work would otherwise leave the epilogue latency-bound on too few warps).
// Waits are bounded as in the expert GEMMs; if one runs out the block still finishes its
// epilogue on zero logits (valid routing, status MOE_ERR_TIMEOUT) so no barrier is left open.
// The CTA that finishes its token block last also runs the scan (route_scan.cuh).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "gemm_tc.h"
#include "route_common.cuh"
#include "route_scan.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace {

constexpr int kBK = 64;
constexpr int kMaxStages = 8;
// threads of the kernel with Q epilogue threads per token
__host__ __device__ constexpr int route_threads(int q) { return 64 + q * kRouteBlock; }
constexpr int kXBytes = kRouteBlock * kBK * 2;  // 16 KB
constexpr int kMaxAcc = 4;                       // TMEM accumulators the K loop may use

// z = (x.W_r + b) / tau from the summed dot product (a temperature of 1 divides exactly,
// so it is skipped)
__device__ __forceinline__ float finish_logit(float dot, float b, float tau) {
  const float z = dot + b;
  return tau == 1.f ? z : z / tau;
}

struct RouteCtl {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t tfull;
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int vote[16];
};

struct RouteGeom {
  int q;            // epilogue threads per token (2 or 4)
  int split;        // CTAs (one cluster) sharing one token block, each on 1/split of d
  int kb_per;       // 64-column K blocks per CTA
  int recv_bytes;   // leader's buffer for the other CTAs' partial logits
  int e_pad;        // MMA N: E rounded up to a multiple of 16 (>= 16)
  int n_acc;        // TMEM accumulators the K loop is spread over (summed in fp32 at the end)
  int stages;
  int stage_bytes;  // x tile + W_r tile
  int body_bytes;   // max(stages * stage_bytes, logits + masks)
  int keep_q;       // exp(z - max) of every logit kept in shared memory for the softmax sums
                    // (when it fits; otherwise the sums recompute it)
  uint32_t tmem_cols;
  size_t smem;      // dynamic shared memory
};

// The Q threads of a token exchange their top-k values (kMaxTopK floats each), their parts
// of the softmax denominator, their marked-expert bitmasks (8 words each) and their counts of
// experts equal to the k-th value; the chosen experts of each token's slots follow
// (kMaxTopK words per token).
__host__ __device__ constexpr int xchg_bytes(int q) {
  return q * kRouteBlock * (kMaxTopK + 1 + 8 + 1) * 4 + kRouteBlock * kMaxTopK * 4;
}

// Columns of range h of Q: whole 16-column chunks, [16 (h nch / Q), 16 ((h+1) nch / Q)).
__host__ __device__ inline int range_col(int e_pad, int h, int q) { return 16 * ((h * (e_pad / 16)) / q); }

RouteGeom route_geom(const Shape& s, int num_sms) {
  RouteGeom g;
  g.q = s.E > 64 ? 4 : 2;
  g.e_pad = ((s.E + 15) / 16) * 16;
  if (g.e_pad < 16) g.e_pad = 16;
  const int kblocks = s.d / kBK;
  // Few token blocks (small T) leave most SMs idle while each CTA streams its x rows with a
  // few stages in flight: split d over a cluster of up to 4 CTAs; the leader adds the
  // others' partial logits (in rank order) from its shared memory.
  g.split = 1;
  while (g.split < 4 && s.nblk * g.split * 2 <= num_sms && g.split * 2 <= kblocks &&
         (2 * g.split - 1) * kRouteBlock * (s.E + 1) * 4 <= 64 * 1024)
    g.split *= 2;
  g.kb_per = (kblocks + g.split - 1) / g.split;
  g.recv_bytes = (g.split - 1) * kRouteBlock * (s.E + 1) * 4;
  g.stage_bytes = kXBytes + g.e_pad * kBK * 2;
  // The ring sets the bytes in flight per SM, which bounds the rate x streams in at.  When
  // there are more CTAs than SMs, up to ~96 KB so that two CTAs share an SM; when every CTA has
  // an SM to itself, up to ~192 KB.
  const bool alone = s.nblk * g.split <= num_sms;
  g.stages = ((alone ? 192 : 96) * 1024) / g.stage_bytes;
  if (g.stages > kMaxStages) g.stages = kMaxStages;
  if (g.stages > g.kb_per) g.stages = g.kb_per;
  // and no more than the shared memory left beside the control block, the cluster's receive
  // buffer and the bias (227 KB per CTA)
  const int fixed = 1024 + (int)sizeof(RouteCtl) + 16 + g.recv_bytes + g.e_pad * 4 + 1024;  // + static, slack
  while (g.stages > 2 && g.stages * g.stage_bytes + fixed > 227 * 1024) --g.stages;
  if (g.stages < 2) g.stages = 2;
  // logits, masks and per-row floats, the exchange, then (if it fits) exp(z - max) per logit
  // for the softmax sums
  const int zs0 = kRouteBlock * (s.E + 1) * 4 + (4 * s.E + 2 * kRouteBlock) * 4 + xchg_bytes(g.q);
  const int zs1 = zs0 + kRouteBlock * (s.E + 1) * 4;
  const int ring = g.stages * g.stage_bytes;
  g.keep_q = ((ring > zs1 ? ring : zs1) + 1023) / 1024 * 1024 + fixed <= 227 * 1024 ? 1 : 0;
  const int zs = g.keep_q ? zs1 : zs0;
  g.body_bytes = ring > zs ? ring : zs;
  // the scan of the last CTA reuses the body
  const int scan = (int)route_scan_smem(s, route_threads(g.q));
  if (g.body_bytes < scan) g.body_bytes = scan;
  g.body_bytes = (g.body_bytes + 1023) / 1024 * 1024;
  // The tensor core's fp32 accumulation chain over K = d loses more than a SIMT sum; K-block
  // kb goes to accumulator kb % n_acc and the epilogue adds the n_acc partial sums in fp32
  // (round to nearest), which keeps the logits within a few 1e-7 relative.
  g.n_acc = 512 / g.e_pad;
  if (g.n_acc > kMaxAcc) g.n_acc = kMaxAcc;
  uint32_t c = 32;
  while (c < (uint32_t)(g.e_pad * g.n_acc)) c <<= 1;
  g.tmem_cols = c;
  // more than half of TMEM: make the CTA big enough in shared memory that two never share an
  // SM (the second would only wait in tcgen05.alloc)
  if (g.tmem_cols > 256 && g.body_bytes < 120 * 1024) g.body_bytes = 120 * 1024;
  g.smem = 1024 + (size_t)g.body_bytes + sizeof(RouteCtl) + 16 + (size_t)g.recv_bytes + (size_t)g.e_pad * 4;
  return g;
}

__device__ __forceinline__ void tmem_ld_16cols(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr)
      : "memory");
}

// Called by the Q*128 epilogue threads once z_s[r * ldz + e] holds the finished logits of the
// block's token r (ldz odd): thread (r, h) owns the experts [e_lo, e_hi) of range h < Q.  Same
// results as route_finish (route_common.cuh), with the per-token work split over Q threads:
//   1. each thread keeps the KS largest values of its range (max/min network); the Q threads
//      of a token swap lists through shared memory and each merges the others' into its own,
//      so all hold the KS largest of the row (the same multiset, in the same descending order);
//   2. each thread sums q = exp(z - max) over its range (keeping q for step 3), marks its
//      experts at or above the k-th value and counts those equal to it; every thread of the
//      token then adds the Q sums (range order).  When the k largest values are distinct and
//      only one expert holds the k-th (the common case), slot j holds the expert whose value is
//      the j-th largest, so each thread places its own marked experts (slot = number of larger
//      values) and writes their gates, indices and bitmask bits; otherwise the range-0 thread
//      assigns every slot over all ranges' marks in ascending expert order (ties: lower index
//      first) -- the rule itself, of which the common case is a shortcut;
//   3. ranks from the bitmasks (the token's slots split over its Q threads); per-block counts;
//      per-expert sums of p = q / sum over the block's rows by the 4Q warps (a lane adds rows
//      lane, +32, +64, +96 in that order, then a fixed butterfly).
template <int KS, int Q>
__device__ __forceinline__ void route_finishq_k(const Shape& s, const Ws& ws, int blk, int r, int h, int e_lo,
                                                int e_hi, float* z_s, int ldz, uint32_t* mask_s, int bar_id,
                                                bool keep_q) {
  constexpr int NT = Q * kRouteBlock;
  const int E = s.E, k = s.k;
  const int tid = h * kRouteBlock + r;
  const int64_t t = (int64_t)blk * kRouteBlock + r;
  const bool valid = t < s.T;
  float* m_s = reinterpret_cast<float*>(mask_s + 4 * E);
  float* inv_s = m_s + kRouteBlock;
  float* xbv = inv_s + kRouteBlock;                                         // [Q][128][kMaxTopK]
  float* xsum = xbv + Q * kRouteBlock * kMaxTopK;                           // [Q][128]
  uint32_t* xtake = reinterpret_cast<uint32_t*>(xsum + Q * kRouteBlock);   // [Q][128][8]
  for (int i = tid; i < 4 * E; i += NT) mask_s[i] = 0u;
  const uint32_t zr = static_cast<uint32_t>(__cvta_generic_to_shared(z_s + r * ldz));

  // pass 1: the KS largest values of this range (fmaxf(z, -inf) ranks a NaN as -inf)
  float bv[KS];
#pragma unroll
  for (int j = 0; j < KS; ++j) bv[j] = -INFINITY;
  bool nan_seen = false;
  if (valid) {
    for (int e0 = e_lo; e0 < e_hi; e0 += 8) {
      float z8[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) z8[u] = e0 + u < e_hi ? ld_shared_f32(zr + 4u * (uint32_t)(e0 + u)) : -INFINITY;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (s.keep_logits && e0 + u < e_hi) ws.logits[t * E + e0 + u] = z8[u];
        nan_seen |= (z8[u] != z8[u]);
        const float v = fmaxf(z8[u], -INFINITY);
#pragma unroll
        for (int j = KS - 1; j > 0; --j) bv[j] = fmaxf(bv[j], fminf(v, bv[j - 1]));
        bv[0] = fmaxf(bv[0], v);
      }
    }
  }
#pragma unroll
  for (int j = 0; j < KS; ++j) xbv[tid * kMaxTopK + j] = bv[j];
  named_barrier(bar_id, NT);
  // merge the other ranges' lists into this one
#pragma unroll
  for (int o = 1; o < Q; ++o) {
    const int hh = (h + o) % Q;
#pragma unroll
    for (int i = 0; i < KS; ++i) {
      const float v = xbv[(hh * kRouteBlock + r) * kMaxTopK + i];
#pragma unroll
      for (int j = KS - 1; j > 0; --j) bv[j] = fmaxf(bv[j], fminf(v, bv[j - 1]));
      bv[0] = fmaxf(bv[0], v);
    }
  }
  if (nan_seen) record_error(ws, MOE_ERR_INTERNAL, 0x100u);
  const float m = bv[0];
  float thr = INFINITY;  // the k-th value: the least of the first k
#pragma unroll
  for (int j = 0; j < KS; ++j)
    if (j < k) thr = fminf(thr, bv[j]);
  int eq_left = k;  // slots open for logits equal to the k-th value
#pragma unroll
  for (int j = 0; j < KS; ++j) eq_left -= (j < k && bv[j] > thr) ? 1 : 0;

  // pass 2: this range's part of the softmax denominator (q = exp(z - max) kept in qs), its
  // marked experts and its count of experts equal to the k-th value
  int* xcnt = reinterpret_cast<int*>(xtake + Q * kRouteBlock * 8);  // [Q][128]
  int* slotv = xcnt + Q * kRouteBlock;                               // [128][kMaxTopK]
  float* qs = reinterpret_cast<float*>(slotv + kRouteBlock * kMaxTopK);  // [128][ldz]
  const uint32_t qr = static_cast<uint32_t>(__cvta_generic_to_shared(qs + r * ldz));
  uint32_t* my_take = xtake + tid * 8;
#pragma unroll
  for (int w = 0; w < 8; ++w) my_take[w] = 0u;
  float sum_h = 0.f;
  int n_thr = 0;
  if (valid) {
    uint32_t cur = 0u;
    int cw = e_lo >> 5;
    for (int e0 = e_lo; e0 < e_hi; e0 += 4) {
      float v4[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        v4[u] = e0 + u < e_hi ? fmaxf(ld_shared_f32(zr + 4u * (uint32_t)(e0 + u)), -INFINITY) : -INFINITY;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int e = e0 + u;
        if (e >= e_hi) break;
        if ((e >> 5) != cw) {
          my_take[cw] = cur;
          cur = 0u;
          cw = e >> 5;
        }
        const float q = expf(v4[u] - m);
        if (keep_q) st_shared_f32(qr + 4u * (uint32_t)e, q);
        sum_h += q;
        cur |= (v4[u] >= thr ? 1u : 0u) << (e & 31);
        n_thr += v4[u] == thr ? 1 : 0;
      }
    }
    if (e_hi > e_lo) my_take[cw] = cur;
  }
  xsum[tid] = sum_h;
  xcnt[tid] = n_thr;
  named_barrier(bar_id, NT);

  float sum = 1.f;
  bool fast = false;
  if (valid) {
    sum = 0.f;
    int thr_experts = 0;
#pragma unroll
    for (int hh = 0; hh < Q; ++hh) {
      sum += xsum[hh * kRouteBlock + r];
      thr_experts += xcnt[hh * kRouteBlock + r];
    }
    bool distinct = true;
#pragma unroll
    for (int j = 0; j + 1 < KS; ++j)
      if (j + 1 < k) distinct = distinct && bv[j] > bv[j + 1];
    fast = distinct && thr_experts == 1;
  }
  if (fast) {
    // slot j holds value bv[j]; the renormalised variant divides by the chosen gates' sum in
    // slot order
    float chosen = 0.f;
#pragma unroll
    for (int j = 0; j < KS; ++j) chosen += j < k ? expf(bv[j] - m) / sum : 0.f;
    for (int w = e_lo >> 5; w <= (e_hi - 1) >> 5 && e_hi > e_lo; ++w) {
      uint32_t take = my_take[w];
      while (take) {
        const int e = w * 32 + __ffs(take) - 1;
        take &= take - 1u;
        const float v = fmaxf(ld_shared_f32(zr + 4u * (uint32_t)e), -INFINITY);
        int pos = 0;
#pragma unroll
        for (int j = 0; j < KS; ++j) pos += (j < k && bv[j] > v) ? 1 : 0;
        const float gate = expf(v - m) / sum;
        slotv[r * kMaxTopK + pos] = e;
        ws.topk_idx[t * k + pos] = e;
        ws.topk_gate[t * k + pos] = s.renorm ? gate / chosen : gate;
        atomicOr(&mask_s[e * 4 + (r >> 5)], 1u << (r & 31));
      }
    }
  }
  if (h == 0) {
    if (valid && !fast) {
      int bi[KS];
#pragma unroll
      for (int j = 0; j < KS; ++j) bi[j] = -1;
      uint32_t filled = 0u;
      for (int w = 0; w < (E + 31) / 32; ++w) {
        uint32_t take = 0u;
#pragma unroll
        for (int hh = 0; hh < Q; ++hh) take |= xtake[(hh * kRouteBlock + r) * 8 + w];
        while (take) {
          const int e = w * 32 + __ffs(take) - 1;
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
          slotv[r * kMaxTopK + j] = e;
          ws.topk_idx[t * k + j] = e;
          ws.topk_gate[t * k + j] = s.renorm ? gate[j] / chosen : gate[j];
          atomicOr(&mask_s[e * 4 + (r >> 5)], 1u << (r & 31));
        }
      }
    }
    m_s[r] = valid ? m : 0.f;
    inv_s[r] = 1.f / sum;
  }
  named_barrier(bar_id, NT);

  // ranks of the token's slots, split over its Q threads
  if (valid) {
    const uint32_t below = (1u << (r & 31)) - 1u;
    for (int j = h; j < k; j += Q) {
      const uint32_t* mk = mask_s + slotv[r * kMaxTopK + j] * 4;
      int rank = __popc(mk[r >> 5] & below);
      for (int wd = 0; wd < (r >> 5); ++wd) rank += __popc(mk[wd]);
      ws.local_rank[t * k + j] = rank;
    }
  }
  for (int e = tid; e < E; e += NT) {
    const uint32_t* mk = mask_s + e * 4;
    ws.blk_cnt[(int64_t)blk * E + e] = __popc(mk[0]) + __popc(mk[1]) + __popc(mk[2]) + __popc(mk[3]);
  }
  // per-expert sums of p = q / sum over the block's rows (rows past T add 0)
  const int w8 = tid >> 5, lane = tid & 31;
  const int64_t t_base = (int64_t)blk * kRouteBlock;
  float mrow[4], inv[4];
  bool vrow[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    mrow[j] = m_s[lane + 32 * j];
    inv[j] = inv_s[lane + 32 * j];
    vrow[j] = t_base + lane + 32 * j < s.T;
  }
  // q from pass 2, or recomputed from the logits when it was not kept (the same value)
  const uint32_t qc = static_cast<uint32_t>(__cvta_generic_to_shared((keep_q ? qs : z_s) + lane * ldz));
  for (int e0 = 4 * w8; e0 < E; e0 += 4 * (NT / 32)) {
    float qq[4][4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        qq[j][u] = (vrow[j] && e0 + u < E) ? ld_shared_f32(qc + 4u * (uint32_t)(32 * j * ldz + e0 + u)) : 0.f;
        if (!keep_q && vrow[j] && e0 + u < E) qq[j][u] = expf(fmaxf(qq[j][u], -INFINITY) - mrow[j]);
      }
    float ps[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int row = lane + 32 * j;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float p = vrow[j] ? qq[j][u] * inv[j] : 0.f;
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

template <int Q>
__device__ __forceinline__ void route_finishq(const Shape& s, const Ws& ws, int blk, int r, int h, int e_lo, int e_hi,
                                              float* z_s, int ldz, uint32_t* mask_s, int bar_id, bool keep_q) {
  if (s.k <= 2) route_finishq_k<2, Q>(s, ws, blk, r, h, e_lo, e_hi, z_s, ldz, mask_s, bar_id, keep_q);
  else if (s.k <= 4) route_finishq_k<4, Q>(s, ws, blk, r, h, e_lo, e_hi, z_s, ldz, mask_s, bar_id, keep_q);
  else if (s.k <= 8) route_finishq_k<8, Q>(s, ws, blk, r, h, e_lo, e_hi, z_s, ldz, mask_s, bar_id, keep_q);
  else route_finishq_k<kMaxTopK, Q>(s, ws, blk, r, h, e_lo, e_hi, z_s, ldz, mask_s, bar_id, keep_q);
}

template <int Q>
__global__ void __launch_bounds__(route_threads(Q), Q == 2 ? 2 : 1)
    route_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW, Shape s, Ws ws,
                    Weights w, RouteGeom g, int64_t timeout_ns) {
  constexpr int NE = Q * kRouteBlock;  // epilogue threads
  extern __shared__ uint8_t smem_raw[];
  uint8_t* body = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  RouteCtl* ctl = reinterpret_cast<RouteCtl*>(body + g.body_bytes);
  // the other CTAs' partial logits [split-1][128][E+1], then the router bias [e_pad]
  // (zero past E; 16-byte aligned, as 128 * 4 divides the first part)
  float* recv = reinterpret_cast<float*>((reinterpret_cast<uintptr_t>(ctl + 1) + 15) & ~uintptr_t(15));
  float* bias_s = recv + (g.split - 1) * kRouteBlock * (s.E + 1);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = g.split > 1 ? ptx::cluster_ctarank() : 0u;
  const int blk = g.split > 1 ? (int)ptx::cluster_id_x() : (int)blockIdx.x;  // token block
  const int kb0 = (int)rank * g.kb_per;                                          // this CTA's K range
  const int kblocks = max(0, min(s.d / kBK, kb0 + g.kb_per) - kb0);  // may be 0 for the last rank
  pdl_launch_dependents();  // the scan may be scheduled; it waits for this grid to finish

  if (threadIdx.x == 0) {
    for (int i = 0; i < g.stages; ++i) {
      ptx::mbar_init(ptx::smem_u32(&ctl->full[i]), 1);
      ptx::mbar_init(ptx::smem_u32(&ctl->empty[i]), 1);
    }
    ptx::mbar_init(ptx::smem_u32(&ctl->tfull), 1);
    ptx::mbar_init(ptx::smem_u32(&ctl->drain), 1);
    ctl->abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(&ctl->tmem_base), g.tmem_cols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  volatile int* abort_flag = &ctl->abort;
  uint32_t issued = 0, issued_phase = 0;

  if (warp == 0) {
    if (lane == 0) {
      ptx::tma_prefetch_desc(&tmX);
      ptx::tma_prefetch_desc(&tmW);
      int stage = 0;
      uint32_t phase = 0;
      for (int kb = 0; kb < kblocks; ++kb) {
        if (!ptx::mbar_wait(ptx::smem_u32(&ctl->empty[stage]), phase ^ 1u, timeout_ns, abort_flag)) {
          *abort_flag = 1;
          record_error(ws, MOE_ERR_TIMEOUT, 0x600u);
          break;
        }
        const uint32_t bar = ptx::smem_u32(&ctl->full[stage]);
        const uint32_t sa = ptx::smem_u32(body + (size_t)stage * g.stage_bytes);
        ptx::mbar_arrive_expect_tx(bar, (uint32_t)g.stage_bytes);
        ptx::tma_load_2d(sa, &tmX, (kb0 + kb) * kBK, blk * kRouteBlock, bar);
        ptx::tma_load_2d(sa + kXBytes, &tmW, (kb0 + kb) * kBK, 0, bar);
        issued |= 1u << stage;
        issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
        if (++stage == g.stages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = ptx::idesc_bf16_f32(kRouteBlock, g.e_pad);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int kb = 0; kb < kblocks; ++kb) {
        if (!ptx::mbar_wait(ptx::smem_u32(&ctl->full[stage]), phase, timeout_ns, abort_flag)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t sa = ptx::smem_u32(body + (size_t)stage * g.stage_bytes);
        const uint32_t sb = sa + kXBytes;
        const uint32_t d_tmem = tmem + (uint32_t)((kb % g.n_acc) * g.e_pad);
#pragma unroll
        for (int ks = 0; ks < kBK / 16; ++ks)
          ptx::mma_bf16(d_tmem, ptx::desc_kmajor_sw128(sa + ks * 32), ptx::desc_kmajor_sw128(sb + ks * 32), idesc,
                        (kb >= g.n_acc || ks != 0) ? 1u : 0u);
        ptx::mma_commit(ptx::smem_u32(&ctl->empty[stage]));
        if (++stage == g.stages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (ok) {
        ptx::mma_commit(ptx::smem_u32(&ctl->tfull));
      } else {
        *abort_flag = 1;
        record_error(ws, MOE_ERR_TIMEOUT, 0x610u);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ epilogue, part 1:
    // this CTA's partial logits (sum of its accumulators) into z_s (leader; finished with
    // bias and temperature when the CTA is alone) or into the leader's receive buffer; the
    // two warps of a lane quarter take the two halves of the expert columns
    const int ew = warp - 2;
    const int q = warp & 3;
    const int h = ew >> 2;        // expert range of this warp, 0..Q-1
    const int r = q * 32 + lane;  // token row of this block
    const int c_lo = range_col(g.e_pad, h, Q), c_hi = range_col(g.e_pad, h + 1, Q);  // its 16-column chunks
    for (int e = ew * 32 + lane; e < g.e_pad; e += NE) bias_s[e] = (s.has_bias && e < s.E) ? w.bias[e] : 0.f;
    bool ok = ptx::mbar_wait(ptx::smem_u32(&ctl->tfull), 0u, timeout_ns, abort_flag);
    ok = __all_sync(0xffffffffu, ok);
    if (lane == 0) ctl->vote[ew] = ok ? 1 : 0;
    named_barrier(2, NE);
    bool all_ok = true;
#pragma unroll
    for (int i = 0; i < 4 * Q; ++i) all_ok = all_ok && ctl->vote[i];
    float* z_s = reinterpret_cast<float*>(body);
    const int ldz = s.E + 1;
    const bool finish_here = g.split == 1;
    const uint32_t recv_remote =
        rank > 0 ? ptx::mapa(ptx::smem_u32(recv + ((int)rank - 1) * kRouteBlock * ldz + r * ldz), 0) : 0u;
    if (all_ok) {
      ptx::tc_fence_after();
      const uint32_t t_row = tmem + ((uint32_t)(q * 32) << 16);
      const uint32_t z_row = ptx::smem_u32(z_s + r * ldz);
      const uint32_t b_base = ptx::smem_u32(bias_s);
      const int used = kblocks < g.n_acc ? kblocks : g.n_acc;  // accumulators that were written
      for (int c = c_lo; c < c_hi; c += 16) {
        // every accumulator's 16 columns in flight at once, and the bias beside them
        uint32_t v[kMaxAcc][16];
#pragma unroll
        for (int a = 0; a < kMaxAcc; ++a)
          if (a < used) tmem_ld_16cols(t_row + (uint32_t)(a * g.e_pad + c), v[a]);
        float b[16];
#pragma unroll
        for (int i = 0; i < 16; i += 4) ld_shared_v4(b_base + 4u * (uint32_t)(c + i), b[i], b[i + 1], b[i + 2], b[i + 3]);
        ptx::tmem_ld_wait();
        float z[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          z[i] = used > 0 ? __uint_as_float(v[0][i]) : 0.f;
#pragma unroll
          for (int a = 1; a < kMaxAcc; ++a)
            if (a < used) z[i] += __uint_as_float(v[a][i]);
          if (finish_here) z[i] = finish_logit(z[i], b[i], s.tau);
        }
        const int n = s.E - c < 16 ? s.E - c : 16;
        if (rank == 0) {
#pragma unroll
          for (int i = 0; i < 16; ++i)
            if (i < n) st_shared_f32(z_row + 4u * (uint32_t)(c + i), z[i]);
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i)
            if (i < n) ptx::st_cluster_u32(recv_remote + 4u * (uint32_t)(c + i), __float_as_uint(z[i]));
        }
      }
    } else {
      if (lane == 0 && ew == 0) record_error(ws, MOE_ERR_TIMEOUT, 0x620u);
      for (int e = c_lo; e < c_hi && e < s.E; ++e) {
        if (rank == 0) z_s[r * ldz + e] = finish_here ? finish_logit(0.f, bias_s[e], s.tau) : 0.f;
        else ptx::st_cluster_u32(recv_remote + 4u * (uint32_t)e, 0u);
      }
    }
  }

  __syncthreads();
  if (g.split > 1) ptx::cluster_sync();  // the partials of every CTA are in the leader's buffer
  if (rank == 0 && warp >= 2) {
    // ------------------------------------------------------------------ epilogue, part 2
    // (leader): add the other CTAs' partials in rank order, bias, temperature; then the
    // softmax / top-k / counting, two threads per token
    const int ew = warp - 2;
    const int q = warp & 3;
    const int h = ew >> 2;
    const int r = q * 32 + lane;
    const int e_lo = min(range_col(g.e_pad, h, Q), s.E);
    const int e_hi = min(range_col(g.e_pad, h + 1, Q), s.E);
    float* z_s = reinterpret_cast<float*>(body);
    uint32_t* mask_s = reinterpret_cast<uint32_t*>(z_s + kRouteBlock * (s.E + 1));
    const int ldz = s.E + 1;
    if (g.split > 1) {
      const uint32_t z_row = ptx::smem_u32(z_s + r * ldz);
      const uint32_t r_row = ptx::smem_u32(recv + r * ldz);
      const uint32_t b_base = ptx::smem_u32(bias_s);
      for (int c = e_lo; c < e_hi; c += 16) {
        const int n = e_hi - c < 16 ? e_hi - c : 16;
        float z[16], b[16];
#pragma unroll
        for (int i = 0; i < 16; i += 4) ld_shared_v4(b_base + 4u * (uint32_t)(c + i), b[i], b[i + 1], b[i + 2], b[i + 3]);
#pragma unroll
        for (int i = 0; i < 16; ++i) z[i] = i < n ? ld_shared_f32(z_row + 4u * (uint32_t)(c + i)) : 0.f;
        for (int rr = 1; rr < g.split; ++rr) {
          const uint32_t part = r_row + (uint32_t)((rr - 1) * kRouteBlock * ldz * 4);
#pragma unroll
          for (int i = 0; i < 16; ++i)
            if (i < n) z[i] += ld_shared_f32(part + 4u * (uint32_t)(c + i));
        }
#pragma unroll
        for (int i = 0; i < 16; ++i)
          if (i < n) st_shared_f32(z_row + 4u * (uint32_t)(c + i), finish_logit(z[i], b[i], s.tau));
      }
      named_barrier(1, NE);  // the other ranges' finished logits are in z_s too
    }
    route_finishq<Q>(s, ws, blk, r, h, e_lo, e_hi, z_s, ldz, mask_s, /*bar_id=*/1, g.keep_q != 0);
  }

  __syncthreads();
  if (*abort_flag) {
    if (warp == 0 && lane == 0)
      for (int st = 0; st < g.stages; ++st)
        if (issued & (1u << st))
          ptx::mbar_wait(ptx::smem_u32(&ctl->full[st]), (issued_phase >> st) & 1u, timeout_ns, nullptr);
    if (warp == 1 && lane == 0) {
      ptx::mma_commit(ptx::smem_u32(&ctl->drain));
      ptx::mbar_wait(ptx::smem_u32(&ctl->drain), 0u, timeout_ns, nullptr);
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, g.tmem_cols);
  }
  // the token blocks' leaders count themselves in; the last one runs the scan in its body
  if (rank == 0) route_scan_if_last(s, ws, route_threads(Q), s.nblk, body);
}

}  // namespace

cudaError_t launch_route_tc(const Shape& s, const Ws& ws, const Weights& w, int num_sms, int64_t timeout_ns,
                            cudaStream_t st) {
  const RouteGeom g = route_geom(s, num_sms);
  CUtensorMap mx, mw;
  cudaError_t e;
  if ((e = make_tmap_bf16(&mx, w.x, (uint64_t)s.T, (uint64_t)s.d, kRouteBlock)) != cudaSuccess) return e;
  if ((e = make_tmap_bf16(&mw, w.wr, (uint64_t)s.E, (uint64_t)s.d, (uint32_t)g.e_pad)) != cudaSuccess) return e;
  auto kernel = g.q == 4 ? route_tc_kernel<4> : route_tc_kernel<2>;
  if ((e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)g.smem)) != cudaSuccess)
    return e;
  return launch_kernel(kernel, dim3((unsigned)(s.nblk * g.split)), dim3((unsigned)route_threads(g.q)), g.smem, st, false,
                       g.split, mx, mw, s, ws, w, g, timeout_ns);
}

}  // namespace moe
