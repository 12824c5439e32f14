// moe_internal.h -- definitions shared by the host side (api.cu) and the kernels.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

constexpr int kRouteBlock = 128;   // tokens per router CTA (= rows of one router MMA tile)
constexpr int kTileM = 128;        // rows per expert-GEMM m-tile
constexpr int kGroupM = 16;        // m-tiles per scheduling group (weight-tile reuse in L2)
constexpr int kMaxTopK = 16;
constexpr int kMaxExperts = 256;

// Status word slots in the workspace header.
// kHdrTicket counts the router CTAs that have finished (the last one runs the scan); the
// words up to kHdrClearWords are cleared before every forward.
enum : int { kHdrStatus = 0, kHdrWhere = 1, kHdrNumGroups = 2, kHdrNumMTiles = 3, kHdrNumPairs = 4, kHdrTicket = 5,
             kHdrClearWords = 8 };

// Layer shape as the kernels see it.
struct Shape {
  int64_t T;
  int64_t N;      // T * k routed rows
  int d, E, k, F;
  int nblk;       // router blocks of kRouteBlock tokens
  float tau;
  int has_bias;
  int keep_logits;
  int renorm;     // gates renormalised over the k chosen
  int training;   // the forward keeps what the backward needs (pre-activations, softmax)
  int act_bf16;   // x and weights are bf16 (else fp32)
  int out_bf16;   // y is bf16 (else fp32)
  int max_groups; // bound on the scheduling groups (sizes the tile descriptors)
};

// Device pointers into one workspace.
struct Ws {
  uint32_t* hdr;        // [64] status word, failure site, scheduler totals
  float* aux;           // scalar
  int32_t* blk_cnt;     // [nblk, E] rows per (router block, expert)
  float* blk_psum;      // [nblk, E] sum over the block's tokens of p[t,e]
  int32_t* local_rank;  // [N] rank of slot (t,j) among its block's slots with the same expert
  int32_t* topk_idx;    // [N]
  float* topk_gate;     // [N]
  int32_t* counts;      // [E]
  int32_t* offsets;     // [E+1]
  float* ptot;          // [E] sum over the tokens of p[t,e] (the router's scan; null where unused)
  int32_t* blk_base;    // [nblk, E] first row of (block, expert) in dispatch order
  // Tile descriptors: entry q describes the scheduling group that owns m-tile q (mt_desc) or
  // m-tile pair q (pr_desc), so that a tile id decodes with one load:
  //   x = expert | (m-tiles, resp. pairs, of the group) << 20, y = the group's first m-tile
  //   (pair) index, z = the group's first row, w = one past the expert's last row.
  int4* mt_desc;        // [max_groups * kGroupM]
  int4* pr_desc;        // [max_groups * kGroupM / 2]
  int32_t* perm_src;    // [N]
  int32_t* perm_slot;   // [N]
  float* gate_perm;     // [N]
  int32_t* slot_pos;    // [N]
  float* logits;        // [T, E] or null
  void* xp;             // [N, d]
  void* h;              // [N, F]
  void* yp;             // [N, d] gate * expert output of routed row p (expert order)
  // training (forward keeps, backward uses)
  void* a1;             // [N, F] bf16: W1_e . x of each routed row
  void* a3;             // [N, F] bf16: W3_e . x
  float* probs;         // [T, E] router softmax
  void* dyp;            // [N, d] bf16: dy of each routed row
  void* dop;            // [N, d] bf16: gate * dy
  void* dab;            // [N, 2F] bf16: [dA | dB], gradients of the two pre-activations
  // Each expert's last, partial 64-row block of dab and dop again, zero past the expert's
  // end (block e holds rows 64e..64e+63): the weight-gradient GEMMs, whose K runs over the
  // expert's rows, read that block from here instead of running on into the next expert.
  void* dab_tail;       // [E * 64, 2F] bf16
  void* dop_tail;       // [E * 64, d] bf16
  float* dgp;           // [N, 2 ceil(F/256)] partial dy . o per 128-column half tile
  void* dxslot;         // [N, d] bf16: expert-input gradient of each routed slot (token order)
  float* dlogit;        // [T, E]
  void* dl_hi;          // [T, dlogit_cols] bf16: dlogit rounded (zero columns past E)
  void* dl_lo;          // [T, dlogit_cols] bf16: dlogit - dl_hi, rounded
  float* dwr_part;      // [dwr_chunks, E, d] router-weight gradient partials (token chunks)
  float* dwr_part_b;    // [nblk, E] router-bias gradient partials (router blocks)
};

// Fixed layout of one workspace: byte offsets of each region.
struct WsLayout {
  size_t hdr, aux, blk_cnt, blk_psum, local_rank, topk_idx, topk_gate, counts, offsets, ptot, blk_base,
      mt_desc, pr_desc, perm_src, perm_slot, gate_perm, slot_pos, logits, xp, h,
      yp, a1, a3, probs, dyp, dop, dab, dab_tail, dop_tail, dgp, dxslot, dlogit, dl_hi, dl_lo, dwr_part, dwr_part_b, total;
};

// Columns of the bf16 dlogit terms: E rounded up to 64 (a whole 128-byte TMA box).
__host__ __device__ inline int dlogit_cols(const Shape& s) { return (s.E + 63) / 64 * 64; }
// Row of dab_tail / dop_tail that repeats routed row p of expert e (rows off .. off+cnt-1),
// or -1 when p is not in the expert's last, partial 64-row block.
__host__ __device__ inline int64_t tail_row(int e, int64_t p, int off, int cnt) {
  const int whole = cnt / 64 * 64;
  const int64_t i = p - off;
  return (cnt % 64 != 0 && i >= whole) ? (int64_t)e * 64 + (i - whole) : -1;
}
constexpr int kDwrMaxChunks = 32;  // token chunks of the router-weight gradient

WsLayout ws_layout(const Shape& s);
Ws ws_bind(const Shape& s, void* base);

struct Weights {
  const void* x;
  const void* wr;
  const float* bias;
  const void* w1;
  const void* w3;
  const void* w2;
  void* y;
};

// Launch `kernel` on `st`; `pdl` chains it to the previous kernel of the stream with
// programmatic dependent launch (the kernel calls pdl_wait() before reading that kernel's
// output); `cluster_x` > 1 launches clusters of that many CTAs.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, bool pdl,
                          int cluster_x, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  int n = 0;
  if (pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cluster_x > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = (unsigned)cluster_x;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = n ? attr : nullptr;
  cfg.numAttrs = (unsigned)n;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Kernel launchers (each returns the launch's cudaError_t).  `pdl`: see launch_kernel.
cudaError_t launch_route_simt(const Shape& s, const Ws& ws, const Weights& w, cudaStream_t st);
cudaError_t launch_permute(const Shape& s, const Ws& ws, const Weights& w, int num_sms, bool pdl, cudaStream_t st);
cudaError_t launch_gemm1_simt(const Shape& s, const Ws& ws, const Weights& w, int num_sms, bool pdl, cudaStream_t st);
cudaError_t launch_gemm2_simt(const Shape& s, const Ws& ws, const Weights& w, int num_sms, bool pdl, cudaStream_t st);
cudaError_t launch_combine(const Shape& s, const Ws& ws, const Weights& w, int num_sms, bool pdl, cudaStream_t st);
// expert stage of expert parallelism: the tile table over received segments; the balancing
// scalar from per-expert totals
cudaError_t launch_seg_scan(const Shape& s, const Ws& ws, const int32_t* seg_counts, int n_seg, int n_local,
                            cudaStream_t st);
cudaError_t launch_aux_totals(int E, int k, int64_t T, const int32_t* counts, const float* psum, float* aux_out,
                              cudaStream_t st);

cudaError_t launch_gather_dy(const Shape& s, const Ws& ws, const void* dy, int num_sms, bool pdl, cudaStream_t st);
cudaError_t launch_router_bwd(const Shape& s, const Ws& ws, float alpha, int n_tiles_dh, bool pdl, cudaStream_t st);
// the chunk partials of the router-weight gradient (and the block partials of the bias
// gradient) added in order
cudaError_t launch_dwr_reduce(const Shape& s, const Ws& ws, float* dwr, float* dbias, int num_sms, bool pdl,
                              cudaStream_t st);
int dwr_chunks(const Shape& s);
int dwr_chunk_tokens(const Shape& s);

// Plan internals for entry points defined outside api.cu.  plan_is_layer: a plan made by
// moe_plan (not an expert-stage plan).
const Shape* plan_shape(moe_plan_t plan);
bool plan_is_layer(moe_plan_t plan);
moe_status set_last_error(moe_status st, const char* msg);

}  // namespace moe
