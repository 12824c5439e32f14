// api.cu -- the C ABI (include/moe.h): plan validation, workspace layout, and the launch
// sequence of the forward.
#include <cuda_runtime.h>
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <new>
#include <string>

#include "moe_internal.h"
#include "gemm_bwd.h"
#include "gemm_tc.h"

struct moe_plan_s {
  moe_config cfg;
  moe::Shape shape;
  moe::WsLayout layout;
  bool tc;          // tensor-core router and expert GEMMs (bf16 layers, not MOE_PATH_SIMT)
  bool pair;        // expert GEMMs on CTA pairs (MOE_PATH_AUTO)
  int device = -1;  // device the cached attributes belong to
  int num_sms = 0;
  int64_t timeout_ns;
  // expert-stage plans (moe_expert_plan): rows from n_src sources, n_src * E_l segments
  bool expert_stage = false;
  int n_src = 0;
  int n_seg = 0;
};

namespace {

thread_local std::string g_last_error;

moe_status fail(moe_status st, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
moe_status fail(moe_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

moe_status cuda_fail(cudaError_t e, const char* what) {
  return fail(MOE_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// "route" covers the router, top-k, per-block counts and (in its last CTA) the scan: offsets,
// dispatch bases, tile descriptors and the balancing scalar.
constexpr const char* kStageNames[] = {"route", "permute", "gemm1_swiglu", "gemm2_gate", "combine"};
constexpr int kNumStages = 5;

// Attributes of the current device, cached on the plan.
moe_status bind_device(moe_plan_t plan) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev == plan->device) return MOE_OK;
  int sms = 0, major = 0, minor = 0;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return cuda_fail(e, "cudaDeviceGetAttribute(SM count)");
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (plan->tc && !(major == 10 && minor == 3))
    return fail(MOE_ERR_UNSUPPORTED, "tensor-core path needs an sm_103 device, found sm_%d%d", major, minor);
  plan->device = dev;
  plan->num_sms = sms;
  return MOE_OK;
}

}  // namespace

namespace moe {

WsLayout ws_layout(const Shape& s) {
  WsLayout L{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = round_up(off + bytes, 256);
    return at;
  };
  const size_t esz = s.act_bf16 ? 2 : 4;
  const size_t N = (size_t)s.N, E = (size_t)s.E, nb = (size_t)s.nblk;
  L.hdr = take(64 * sizeof(uint32_t));
  L.aux = take(sizeof(float));
  L.blk_cnt = take(nb * E * 4);
  L.blk_psum = take(nb * E * 4);
  L.local_rank = take(N * 4);
  L.topk_idx = take(N * 4);
  L.topk_gate = take(N * 4);
  L.counts = take(E * 4);
  L.offsets = take((E + 1) * 4);
  L.ptot = take(E * 4);
  L.blk_base = take(nb * E * 4);
  L.mt_desc = take((size_t)s.max_groups * moe::kGroupM * 16);
  L.pr_desc = take((size_t)s.max_groups * (moe::kGroupM / 2) * 16);
  L.perm_src = take(N * 4);
  L.perm_slot = take(N * 4);
  L.gate_perm = take(N * 4);
  L.slot_pos = take(N * 4);
  L.logits = s.keep_logits ? take((size_t)s.T * E * 4) : 0;
  L.xp = take(N * (size_t)s.d * esz);
  L.h = take(N * (size_t)s.F * esz);
  L.yp = take(N * (size_t)s.d * esz);
  if (s.training) {
    const size_t nt = 2 * (((size_t)s.F + 255) / 256), chunks = (size_t)dwr_chunks(s);
    L.a1 = take(N * (size_t)s.F * 2);
    L.a3 = take(N * (size_t)s.F * 2);
    L.probs = take((size_t)s.T * E * 4);
    L.dyp = take(N * (size_t)s.d * 2);
    L.dop = take(N * (size_t)s.d * 2);
    L.dab = take(N * 2 * (size_t)s.F * 2);
    L.dab_tail = take(E * 64 * 2 * (size_t)s.F * 2);
    L.dop_tail = take(E * 64 * (size_t)s.d * 2);
    L.dgp = take(N * nt * 4);
    L.dxslot = take(N * (size_t)s.d * 2);
    L.dlogit = take((size_t)s.T * E * 4);
    L.dl_hi = take((size_t)s.T * moe::dlogit_cols(s) * 2);
    L.dl_lo = take((size_t)s.T * moe::dlogit_cols(s) * 2);
    L.dwr_part = take(chunks * E * (size_t)s.d * 4);
    L.dwr_part_b = take(nb * E * 4);
  }
  L.total = off;
  return L;
}

Ws ws_bind(const Shape& s, void* base) {
  const WsLayout L = ws_layout(s);
  char* b = static_cast<char*>(base);
  Ws w{};
  w.hdr = reinterpret_cast<uint32_t*>(b + L.hdr);
  w.aux = reinterpret_cast<float*>(b + L.aux);
  w.blk_cnt = reinterpret_cast<int32_t*>(b + L.blk_cnt);
  w.blk_psum = reinterpret_cast<float*>(b + L.blk_psum);
  w.local_rank = reinterpret_cast<int32_t*>(b + L.local_rank);
  w.topk_idx = reinterpret_cast<int32_t*>(b + L.topk_idx);
  w.topk_gate = reinterpret_cast<float*>(b + L.topk_gate);
  w.counts = reinterpret_cast<int32_t*>(b + L.counts);
  w.offsets = reinterpret_cast<int32_t*>(b + L.offsets);
  w.ptot = reinterpret_cast<float*>(b + L.ptot);
  w.blk_base = reinterpret_cast<int32_t*>(b + L.blk_base);
  w.mt_desc = reinterpret_cast<int4*>(b + L.mt_desc);
  w.pr_desc = reinterpret_cast<int4*>(b + L.pr_desc);
  w.perm_src = reinterpret_cast<int32_t*>(b + L.perm_src);
  w.perm_slot = reinterpret_cast<int32_t*>(b + L.perm_slot);
  w.gate_perm = reinterpret_cast<float*>(b + L.gate_perm);
  w.slot_pos = reinterpret_cast<int32_t*>(b + L.slot_pos);
  w.logits = s.keep_logits ? reinterpret_cast<float*>(b + L.logits) : nullptr;
  w.xp = b + L.xp;
  w.h = b + L.h;
  w.yp = b + L.yp;
  if (s.training) {
    w.a1 = b + L.a1;
    w.a3 = b + L.a3;
    w.probs = reinterpret_cast<float*>(b + L.probs);
    w.dyp = b + L.dyp;
    w.dop = b + L.dop;
    w.dab = b + L.dab;
    w.dab_tail = b + L.dab_tail;
    w.dop_tail = b + L.dop_tail;
    w.dgp = reinterpret_cast<float*>(b + L.dgp);
    w.dxslot = b + L.dxslot;
    w.dlogit = reinterpret_cast<float*>(b + L.dlogit);
    w.dl_hi = b + L.dl_hi;
    w.dl_lo = b + L.dl_lo;
    w.dwr_part = reinterpret_cast<float*>(b + L.dwr_part);
    w.dwr_part_b = reinterpret_cast<float*>(b + L.dwr_part_b);
  }
  return w;
}

const Shape* plan_shape(moe_plan_t plan) { return &plan->shape; }
bool plan_is_layer(moe_plan_t plan) { return plan && !plan->expert_stage; }

// Workspace of an expert-stage plan: status header, per-segment counts and offsets, the tile
// descriptors and the SwiGLU hidden rows H [N, F]; the received rows, their gates and the
// output rows are the caller's buffers.
WsLayout expert_layout(const Shape& s, int n_seg) {
  WsLayout L{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = round_up(off + bytes, 256);
    return at;
  };
  L.hdr = take(64 * sizeof(uint32_t));
  L.counts = take((size_t)n_seg * 4);
  L.offsets = take(((size_t)n_seg + 1) * 4);
  L.mt_desc = take((size_t)s.max_groups * moe::kGroupM * 16);
  L.pr_desc = take((size_t)s.max_groups * (moe::kGroupM / 2) * 16);
  L.h = take((size_t)s.N * (size_t)s.F * (s.act_bf16 ? 2 : 4));
  L.total = off;
  return L;
}

moe_status set_last_error(moe_status st, const char* msg) {
  g_last_error = msg;
  return st;
}

}  // namespace moe

extern "C" {

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
    case MOE_ERR_INTERNAL: return "MOE_ERR_INTERNAL";
  }
  return "MOE_ERR_UNKNOWN";
}

const char* moe_last_error(void) { return g_last_error.c_str(); }

moe_status moe_plan(const moe_config* cfg, moe_plan_t* plan, size_t* workspace_bytes) {
  if (!cfg || !plan || !workspace_bytes) return fail(MOE_ERR_INVALID_ARG, "null argument");
  *plan = nullptr;
  const moe_config& c = *cfg;
  if (c.T < 1 || c.d_model < 1 || c.d_expert < 1) return fail(MOE_ERR_INVALID_ARG, "T, d_model, d_expert must be >= 1");
  if (c.n_experts < 1 || c.n_experts > moe::kMaxExperts)
    return fail(MOE_ERR_INVALID_ARG, "n_experts must be in [1, %d]", moe::kMaxExperts);
  if (c.top_k < 1 || c.top_k > c.n_experts || c.top_k > moe::kMaxTopK)
    return fail(MOE_ERR_INVALID_ARG, "top_k must be in [1, min(n_experts, %d)]", moe::kMaxTopK);
  if (c.act_dtype != MOE_F32 && c.act_dtype != MOE_BF16) return fail(MOE_ERR_INVALID_ARG, "bad act_dtype");
  if (c.out_dtype != MOE_F32 && c.out_dtype != MOE_BF16) return fail(MOE_ERR_INVALID_ARG, "bad out_dtype");
  if (!(c.router_temperature > 0.f) || !isfinite(c.router_temperature))
    return fail(MOE_ERR_INVALID_ARG, "router_temperature must be finite and > 0");
  if (c.has_router_bias != 0 && c.has_router_bias != 1) return fail(MOE_ERR_INVALID_ARG, "has_router_bias must be 0 or 1");
  if (c.path != MOE_PATH_AUTO && c.path != MOE_PATH_SIMT && c.path != MOE_PATH_TC_1SM)
    return fail(MOE_ERR_INVALID_ARG, "bad path");
  if (c.flags & ~(MOE_FLAG_KEEP_LOGITS | MOE_FLAG_TEST_STALL | MOE_FLAG_RENORM_GATES | MOE_FLAG_TRAINING))
    return fail(MOE_ERR_INVALID_ARG, "unknown flags");
  const int64_t N = c.T * (int64_t)c.top_k;
  if (N > (int64_t)INT32_MAX / 2 || N * (int64_t)(c.d_model > c.d_expert ? c.d_model : c.d_expert) > ((int64_t)1 << 40))
    return fail(MOE_ERR_UNSUPPORTED, "T * top_k (or the routed activations) too large");
  const bool bf16 = c.act_dtype == MOE_BF16;
  if (c.path == MOE_PATH_TC_1SM && !bf16) return fail(MOE_ERR_INVALID_ARG, "MOE_PATH_TC_1SM needs bf16 inputs");
  const bool tc = bf16 && c.path != MOE_PATH_SIMT && moe::kTensorCorePathBuilt;
  if (!bf16 && c.d_model % 4 != 0) return fail(MOE_ERR_UNSUPPORTED, "fp32 layers need d_model %% 4 == 0");
  if (bf16 && c.d_model % 8 != 0) return fail(MOE_ERR_UNSUPPORTED, "bf16 layers need d_model %% 8 == 0");
  if (tc && (c.d_model % 64 != 0 || c.d_expert % 64 != 0))
    return fail(MOE_ERR_UNSUPPORTED, "the tensor-core path needs d_model and d_expert multiples of 64 (use MOE_PATH_SIMT)");
  if ((c.flags & MOE_FLAG_TEST_STALL) && !tc)
    return fail(MOE_ERR_INVALID_ARG, "MOE_FLAG_TEST_STALL applies to the tensor-core path only");
  if ((c.flags & MOE_FLAG_TRAINING) && (!tc || c.out_dtype != MOE_BF16))
    return fail(MOE_ERR_UNSUPPORTED, "MOE_FLAG_TRAINING needs the tensor-core path (bf16 inputs) and bf16 output");

  moe_plan_s* p = new (std::nothrow) moe_plan_s();
  if (!p) return fail(MOE_ERR_INTERNAL, "out of host memory");
  p->cfg = c;
  moe::Shape& s = p->shape;
  s.T = c.T;
  s.N = N;
  s.d = c.d_model;
  s.E = c.n_experts;
  s.k = c.top_k;
  s.F = c.d_expert;
  s.nblk = (int)((c.T + moe::kRouteBlock - 1) / moe::kRouteBlock);
  s.tau = c.router_temperature;
  s.has_bias = c.has_router_bias;
  s.keep_logits = (c.flags & MOE_FLAG_KEEP_LOGITS) ? 1 : 0;
  s.renorm = (c.flags & MOE_FLAG_RENORM_GATES) ? 1 : 0;
  s.training = (c.flags & MOE_FLAG_TRAINING) ? 1 : 0;
  s.act_bf16 = bf16 ? 1 : 0;
  s.out_bf16 = c.out_dtype == MOE_BF16 ? 1 : 0;
  // groups of up to kGroupM m-tiles per expert: sum_e ceil(mt_e / G) <= MT / G + E and
  // MT = sum_e ceil(count_e / 128) <= N / 128 + E
  s.max_groups = (int)(N / ((int64_t)moe::kTileM * moe::kGroupM) + 2 * (int64_t)c.n_experts + 2);
  p->layout = moe::ws_layout(s);
  p->tc = tc;
  p->pair = tc && c.path == MOE_PATH_AUTO;
  p->timeout_ns = c.wait_timeout_ns > 0 ? c.wait_timeout_ns : 2000000000LL;
  *plan = p;
  *workspace_bytes = p->layout.total;
  g_last_error.clear();
  return MOE_OK;
}

void moe_plan_destroy(moe_plan_t plan) { delete plan; }

int32_t moe_stage_count(moe_plan_t plan) { return plan && !plan->expert_stage ? kNumStages : 0; }

const char* moe_stage_name(moe_plan_t plan, int32_t stage) {
  if (!plan || plan->expert_stage || stage < 0 || stage >= kNumStages) return nullptr;
  return kStageNames[stage];
}

static moe_status check_forward_args(moe_plan_t plan, const void* x, const void* w_router, const float* bias,
                                     const void* w1, const void* w3, const void* w2, void* y, void* workspace,
                                     size_t workspace_bytes) {
  if (!plan) return fail(MOE_ERR_INVALID_ARG, "null plan");
  if (plan->expert_stage) return fail(MOE_ERR_INVALID_ARG, "an expert-stage plan runs only moe_expert_forward");
  const void* ptrs[] = {x, w_router, w1, w3, w2, y};
  const char* names[] = {"x", "w_router", "w1", "w3", "w2", "y"};
  for (int i = 0; i < 6; ++i) {
    if (!ptrs[i]) return fail(MOE_ERR_INVALID_ARG, "%s is null", names[i]);
    if (!aligned(ptrs[i], 16)) return fail(MOE_ERR_INVALID_ARG, "%s is not 16-byte aligned", names[i]);
  }
  if (plan->shape.has_bias && (!bias || !aligned(bias, 16)))
    return fail(MOE_ERR_INVALID_ARG, "router_bias must be a 16-byte aligned pointer (plan has a bias)");
  if (!workspace || !aligned(workspace, 256)) return fail(MOE_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  if (workspace_bytes < plan->layout.total)
    return fail(MOE_ERR_INVALID_ARG, "workspace too small: %zu < %zu", workspace_bytes, plan->layout.total);
  return MOE_OK;
}

static moe_status run_stage(moe_plan_t plan, int32_t stage, const moe::Weights& w, void* workspace, cudaStream_t st) {
  const moe::Shape& s = plan->shape;
  const moe::Ws ws = moe::ws_bind(s, workspace);
  // every stage after the router is chained to its predecessor (programmatic dependent launch)
  const bool pdl = stage > 0;
  cudaError_t e = cudaSuccess;
  switch (stage) {
    case 0:
      // the status word and the router's completion ticket start at zero
      e = cudaMemsetAsync(ws.hdr, 0, moe::kHdrClearWords * sizeof(uint32_t), st);
      if (e != cudaSuccess) return cuda_fail(e, "clearing the status word");
      e = plan->tc ? moe::launch_route_tc(s, ws, w, plan->num_sms, plan->timeout_ns, st)
                   : moe::launch_route_simt(s, ws, w, st);
      break;
    case 1: e = moe::launch_permute(s, ws, w, plan->num_sms, pdl, st); break;
    case 2:
    case 3: {
      const int mode = stage == 2 ? 1 : 2;
      const bool stall = mode == 1 && (plan->cfg.flags & MOE_FLAG_TEST_STALL) != 0;
      if (plan->pair)
        e = moe::launch_gemm_tc_pair(mode, s, ws, w, plan->num_sms, plan->timeout_ns, stall, pdl, st);
      else if (plan->tc)
        e = moe::launch_gemm_tc(mode, s, ws, w, plan->num_sms, plan->timeout_ns, stall, pdl, st);
      else
        e = mode == 1 ? moe::launch_gemm1_simt(s, ws, w, plan->num_sms, pdl, st)
                      : moe::launch_gemm2_simt(s, ws, w, plan->num_sms, pdl, st);
      break;
    }
    case 4: e = moe::launch_combine(s, ws, w, plan->num_sms, pdl, st); break;
    default: return fail(MOE_ERR_INVALID_ARG, "stage %d out of range", stage);
  }
  if (e != cudaSuccess) {
    char what[64];
    snprintf(what, sizeof what, "launching stage %s", kStageNames[stage]);
    return cuda_fail(e, what);
  }
  return MOE_OK;
}

moe_status moe_forward_stage(moe_plan_t plan, int32_t stage, const void* x, const void* w_router,
                             const float* router_bias, const void* w1, const void* w3, const void* w2, void* y,
                             void* workspace, size_t workspace_bytes, void* stream) {
  moe_status st = check_forward_args(plan, x, w_router, router_bias, w1, w3, w2, y, workspace, workspace_bytes);
  if (st != MOE_OK) return st;
  if ((st = bind_device(plan)) != MOE_OK) return st;
  const moe::Weights w{x, w_router, plan->shape.has_bias ? router_bias : nullptr, w1, w3, w2, y};
  return run_stage(plan, stage, w, workspace, static_cast<cudaStream_t>(stream));
}

moe_status moe_forward(moe_plan_t plan, const void* x, const void* w_router, const float* router_bias,
                       const void* w1, const void* w3, const void* w2, void* y, void* workspace,
                       size_t workspace_bytes, void* stream) {
  moe_status st = check_forward_args(plan, x, w_router, router_bias, w1, w3, w2, y, workspace, workspace_bytes);
  if (st != MOE_OK) return st;
  if ((st = bind_device(plan)) != MOE_OK) return st;
  const moe::Weights w{x, w_router, plan->shape.has_bias ? router_bias : nullptr, w1, w3, w2, y};
  for (int i = 0; i < kNumStages; ++i)
    if ((st = run_stage(plan, i, w, workspace, static_cast<cudaStream_t>(stream))) != MOE_OK) return st;
  return MOE_OK;
}

moe_status moe_forward_host(moe_plan_t plan, const void* x_host, void* x_dev, const void* w_router,
                            const float* router_bias, const void* w1, const void* w3, const void* w2, void* y_dev,
                            void* y_host, void* workspace, size_t workspace_bytes, void* stream) {
  if (!plan || !x_host || !y_host) return fail(MOE_ERR_INVALID_ARG, "null argument");
  moe_status st = check_forward_args(plan, x_dev, w_router, router_bias, w1, w3, w2, y_dev, workspace, workspace_bytes);
  if (st != MOE_OK) return st;
  const moe::Shape& s = plan->shape;
  const size_t xbytes = (size_t)s.T * s.d * (s.act_bf16 ? 2 : 4);
  const size_t ybytes = (size_t)s.T * s.d * (s.out_bf16 ? 2 : 4);
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(x_dev, x_host, xbytes, cudaMemcpyHostToDevice, cs);
  if (e != cudaSuccess) return cuda_fail(e, "copying x to the device");
  if ((st = moe_forward(plan, x_dev, w_router, router_bias, w1, w3, w2, y_dev, workspace, workspace_bytes, stream)) != MOE_OK)
    return st;
  e = cudaMemcpyAsync(y_host, y_dev, ybytes, cudaMemcpyDeviceToHost, cs);
  if (e != cudaSuccess) return cuda_fail(e, "copying y to the host");
  return MOE_OK;
}

static constexpr const char* kBwdStageNames[] = {"gather_dy", "bwd_dh_swiglu", "bwd_dx_gemm", "bwd_dw13", "bwd_dw2",
                                                  "router_bwd", "bwd_dx_combine", "bwd_dw_router"};
static constexpr int kNumBwdStages = 8;

int32_t moe_backward_stage_count(moe_plan_t plan) { return plan ? kNumBwdStages : 0; }

const char* moe_backward_stage_name(moe_plan_t plan, int32_t stage) {
  if (!plan || stage < 0 || stage >= kNumBwdStages) return nullptr;
  return kBwdStageNames[stage];
}

moe_status moe_backward_stage(moe_plan_t plan, int32_t stage, const void* x, const void* w_router,
                              const float* router_bias, const void* w1, const void* w3, const void* w2, const void* dy,
                              float aux_weight, float* dx, float* dw_router, float* dbias, float* dw1, float* dw3,
                              float* dw2, void* workspace, size_t workspace_bytes, void* stream) {
  moe_status st =
      check_forward_args(plan, x, w_router, router_bias, w1, w3, w2, const_cast<void*>(dy), workspace, workspace_bytes);
  if (st != MOE_OK) return st;
  if (!plan->shape.training) return fail(MOE_ERR_INVALID_ARG, "moe_backward needs a plan made with MOE_FLAG_TRAINING");
  const void* outs[] = {dx, dw_router, dw1, dw3, dw2};
  for (const void* o : outs)
    if (!o || !aligned(o, 16)) return fail(MOE_ERR_INVALID_ARG, "gradient outputs must be 16-byte aligned device pointers");
  if (plan->shape.has_bias && dbias && !aligned(dbias, 16)) return fail(MOE_ERR_INVALID_ARG, "dbias must be 16-byte aligned");
  if (stage < 0 || stage >= kNumBwdStages) return fail(MOE_ERR_INVALID_ARG, "backward stage %d out of range", stage);
  if ((st = bind_device(plan)) != MOE_OK) return st;
  const moe::Shape& s = plan->shape;
  const moe::Ws ws = moe::ws_bind(s, workspace);
  const moe::Weights w{x, w_router, plan->shape.has_bias ? router_bias : nullptr, w1, w3, w2, nullptr};
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const bool pdl = stage > 0;  // chained to the previous backward kernel
  cudaError_t e = cudaSuccess;
  switch (stage) {
    case 0: e = moe::launch_gather_dy(s, ws, dy, plan->num_sms, false, cs); break;
    case 1:
    case 2: {
      const int kind = stage == 1 ? moe::kBwdDH : moe::kBwdDX;
      e = plan->pair ? moe::launch_gemm_bwd_pair(kind, s, ws, w, plan->num_sms, plan->timeout_ns, pdl, cs)
                     : moe::launch_gemm_bwd(kind, s, ws, w, nullptr, nullptr, plan->num_sms, plan->timeout_ns, pdl, cs);
      break;
    }
    case 3:
    case 4: {
      const int kind = stage == 3 ? moe::kBwdDW13 : moe::kBwdDW2;
      float* a = stage == 3 ? dw1 : dw2;
      float* b = stage == 3 ? dw3 : nullptr;
      e = plan->pair ? moe::launch_gemm_dw_pair(kind, s, ws, a, b, plan->num_sms, plan->timeout_ns, pdl, cs)
                     : moe::launch_gemm_bwd(kind, s, ws, w, a, b, plan->num_sms, plan->timeout_ns, pdl, cs);
      break;
    }
    case 5: e = moe::launch_router_bwd(s, ws, aux_weight, 2 * ((s.F + 255) / 256), pdl, cs); break;
    case 6: e = moe::launch_dx_tc(s, ws, w_router, dx, plan->timeout_ns, pdl, cs); break;
    case 7:
      e = moe::launch_dwr_tc(s, ws, x, plan->timeout_ns, pdl, cs);
      if (e == cudaSuccess)
        e = moe::launch_dwr_reduce(s, ws, dw_router, plan->shape.has_bias ? dbias : nullptr, plan->num_sms, true, cs);
      break;
  }
  if (e != cudaSuccess) {
    char what[64];
    snprintf(what, sizeof what, "launching backward stage %s", kBwdStageNames[stage]);
    return cuda_fail(e, what);
  }
  return MOE_OK;
}

moe_status moe_backward(moe_plan_t plan, const void* x, const void* w_router, const float* router_bias,
                        const void* w1, const void* w3, const void* w2, const void* dy, float aux_weight, float* dx,
                        float* dw_router, float* dbias, float* dw1, float* dw3, float* dw2, void* workspace,
                        size_t workspace_bytes, void* stream) {
  for (int i = 0; i < kNumBwdStages; ++i) {
    moe_status st = moe_backward_stage(plan, i, x, w_router, router_bias, w1, w3, w2, dy, aux_weight, dx, dw_router,
                                       dbias, dw1, dw3, dw2, workspace, workspace_bytes, stream);
    if (st != MOE_OK) return st;
  }
  return MOE_OK;
}

moe_status moe_aux_loss(moe_plan_t plan, const void* workspace, float* aux_out, void* stream) {
  if (!plan || !workspace || !aux_out) return fail(MOE_ERR_INVALID_ARG, "null argument");
  if (plan->expert_stage) return fail(MOE_ERR_INVALID_ARG, "an expert-stage plan has no balancing scalar");
  if (!aligned(workspace, 256)) return fail(MOE_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  const char* src = static_cast<const char*>(workspace) + plan->layout.aux;
  cudaError_t e = cudaMemcpyAsync(aux_out, src, sizeof(float), cudaMemcpyDeviceToDevice, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "copying aux");
  return MOE_OK;
}

moe_status moe_workspace_views(moe_plan_t plan, void* workspace, moe_views* v) {
  if (!plan || !workspace || !v) return fail(MOE_ERR_INVALID_ARG, "null argument");
  if (plan->expert_stage) return fail(MOE_ERR_INVALID_ARG, "an expert-stage plan's workspace has no views");
  const moe::Ws w = moe::ws_bind(plan->shape, workspace);
  v->status = w.hdr + moe::kHdrStatus;
  v->aux = w.aux;
  v->topk_idx = w.topk_idx;
  v->topk_gate = w.topk_gate;
  v->expert_counts = w.counts;
  v->expert_offsets = w.offsets;
  v->perm_src = w.perm_src;
  v->perm_slot = w.perm_slot;
  v->gate_perm = w.gate_perm;
  v->slot_pos = w.slot_pos;
  v->logits = w.logits;
  v->xp = w.xp;
  v->h = w.h;
  v->yp = w.yp;
  v->expert_psum = w.ptot;
  return MOE_OK;
}

moe_status moe_expert_plan(const moe_expert_config* cfg, moe_plan_t* plan, size_t* workspace_bytes) {
  if (!cfg || !plan || !workspace_bytes) return fail(MOE_ERR_INVALID_ARG, "null argument");
  *plan = nullptr;
  const moe_expert_config& c = *cfg;
  if (c.max_rows < 1 || c.d_model < 1 || c.d_expert < 1 || c.n_local_experts < 1 || c.n_sources < 1)
    return fail(MOE_ERR_INVALID_ARG, "max_rows, d_model, d_expert, n_local_experts, n_sources must be >= 1");
  if ((int64_t)c.n_local_experts * c.n_sources > moe::kMaxExperts)
    return fail(MOE_ERR_INVALID_ARG, "n_sources * n_local_experts must be <= %d", moe::kMaxExperts);
  if (c.act_dtype != MOE_F32 && c.act_dtype != MOE_BF16) return fail(MOE_ERR_INVALID_ARG, "bad act_dtype");
  if (c.path != MOE_PATH_AUTO && c.path != MOE_PATH_SIMT && c.path != MOE_PATH_TC_1SM)
    return fail(MOE_ERR_INVALID_ARG, "bad path");
  if (c.max_rows > (int64_t)INT32_MAX / 2 ||
      c.max_rows * (int64_t)(c.d_model > c.d_expert ? c.d_model : c.d_expert) > ((int64_t)1 << 40))
    return fail(MOE_ERR_UNSUPPORTED, "max_rows (or the rows' activations) too large");
  const bool bf16 = c.act_dtype == MOE_BF16;
  if (c.path == MOE_PATH_TC_1SM && !bf16) return fail(MOE_ERR_INVALID_ARG, "MOE_PATH_TC_1SM needs bf16 inputs");
  const bool tc = bf16 && c.path != MOE_PATH_SIMT && moe::kTensorCorePathBuilt;
  if (!bf16 && c.d_model % 4 != 0) return fail(MOE_ERR_UNSUPPORTED, "fp32 layers need d_model %% 4 == 0");
  if (bf16 && c.d_model % 8 != 0) return fail(MOE_ERR_UNSUPPORTED, "bf16 layers need d_model %% 8 == 0");
  if (tc && (c.d_model % 64 != 0 || c.d_expert % 64 != 0))
    return fail(MOE_ERR_UNSUPPORTED, "the tensor-core path needs d_model and d_expert multiples of 64 (use MOE_PATH_SIMT)");
  moe_plan_s* p = new (std::nothrow) moe_plan_s();
  if (!p) return fail(MOE_ERR_INTERNAL, "out of host memory");
  p->cfg = moe_config{};
  p->cfg.path = c.path;
  moe::Shape& s = p->shape;
  s.T = c.max_rows;
  s.N = c.max_rows;
  s.d = c.d_model;
  s.E = c.n_local_experts;  // weight experts: the GEMMs' weight tensors hold E_l experts
  s.k = 1;
  s.F = c.d_expert;
  s.nblk = 0;
  s.tau = 1.f;
  s.act_bf16 = bf16 ? 1 : 0;
  s.out_bf16 = s.act_bf16;
  p->n_src = c.n_sources;
  p->n_seg = c.n_sources * c.n_local_experts;
  // groups of up to kGroupM m-tiles per segment (as moe_plan bounds them per expert)
  s.max_groups = (int)(c.max_rows / ((int64_t)moe::kTileM * moe::kGroupM) + 2 * (int64_t)p->n_seg + 2);
  p->layout = moe::expert_layout(s, p->n_seg);
  p->tc = tc;
  p->pair = tc && c.path == MOE_PATH_AUTO;
  p->timeout_ns = c.wait_timeout_ns > 0 ? c.wait_timeout_ns : 2000000000LL;
  p->expert_stage = true;
  *plan = p;
  *workspace_bytes = p->layout.total;
  g_last_error.clear();
  return MOE_OK;
}

moe_status moe_expert_forward(moe_plan_t plan, const int32_t* seg_counts, const void* x_rows, const float* gates,
                              const void* w1, const void* w3, const void* w2, void* y_rows, void* workspace,
                              size_t workspace_bytes, void* stream) {
  if (!plan) return fail(MOE_ERR_INVALID_ARG, "null plan");
  if (!plan->expert_stage) return fail(MOE_ERR_INVALID_ARG, "moe_expert_forward needs a plan made by moe_expert_plan");
  const void* ptrs[] = {seg_counts, x_rows, gates, w1, w3, w2, y_rows};
  const char* names[] = {"seg_counts", "x_rows", "gates", "w1", "w3", "w2", "y_rows"};
  for (int i = 0; i < 7; ++i) {
    if (!ptrs[i]) return fail(MOE_ERR_INVALID_ARG, "%s is null", names[i]);
    if (!aligned(ptrs[i], 16)) return fail(MOE_ERR_INVALID_ARG, "%s is not 16-byte aligned", names[i]);
  }
  if (!workspace || !aligned(workspace, 256)) return fail(MOE_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  if (workspace_bytes < plan->layout.total)
    return fail(MOE_ERR_INVALID_ARG, "workspace too small: %zu < %zu", workspace_bytes, plan->layout.total);
  moe_status st = bind_device(plan);
  if (st != MOE_OK) return st;
  const moe::Shape& s = plan->shape;
  const moe::WsLayout& L = plan->layout;
  char* b = static_cast<char*>(workspace);
  moe::Ws ws{};
  ws.hdr = reinterpret_cast<uint32_t*>(b + L.hdr);
  ws.counts = reinterpret_cast<int32_t*>(b + L.counts);
  ws.offsets = reinterpret_cast<int32_t*>(b + L.offsets);
  ws.mt_desc = reinterpret_cast<int4*>(b + L.mt_desc);
  ws.pr_desc = reinterpret_cast<int4*>(b + L.pr_desc);
  ws.h = b + L.h;
  ws.xp = const_cast<void*>(x_rows);
  ws.yp = y_rows;
  ws.gate_perm = const_cast<float*>(gates);
  const moe::Weights w{nullptr, nullptr, nullptr, w1, w3, w2, nullptr};
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(ws.hdr, 0, moe::kHdrClearWords * sizeof(uint32_t), cs);
  if (e != cudaSuccess) return cuda_fail(e, "clearing the status word");
  if ((e = moe::launch_seg_scan(s, ws, seg_counts, plan->n_seg, s.E, cs)) != cudaSuccess)
    return cuda_fail(e, "launching the segment scan");
  for (int mode = 1; mode <= 2; ++mode) {
    if (plan->pair)
      e = moe::launch_gemm_tc_pair(mode, s, ws, w, plan->num_sms, plan->timeout_ns, false, true, cs);
    else if (plan->tc)
      e = moe::launch_gemm_tc(mode, s, ws, w, plan->num_sms, plan->timeout_ns, false, true, cs);
    else
      e = mode == 1 ? moe::launch_gemm1_simt(s, ws, w, plan->num_sms, true, cs)
                    : moe::launch_gemm2_simt(s, ws, w, plan->num_sms, true, cs);
    if (e != cudaSuccess) return cuda_fail(e, mode == 1 ? "launching the SwiGLU GEMM" : "launching the down-projection");
  }
  return MOE_OK;
}

moe_status moe_aux_from_totals(int32_t n_experts, int32_t top_k, int64_t n_tokens, const int32_t* counts,
                               const float* psum, float* aux_out, void* stream) {
  if (n_experts < 1 || n_experts > moe::kMaxExperts || top_k < 1 || top_k > n_experts || n_tokens < 1)
    return fail(MOE_ERR_INVALID_ARG, "need 1 <= n_experts <= %d, 1 <= top_k <= n_experts, n_tokens >= 1",
                moe::kMaxExperts);
  if (!counts || !psum || !aux_out) return fail(MOE_ERR_INVALID_ARG, "null argument");
  if (!aligned(counts, 16) || !aligned(psum, 16) || !aligned(aux_out, 4))
    return fail(MOE_ERR_INVALID_ARG, "counts and psum must be 16-byte aligned");
  cudaError_t e = moe::launch_aux_totals(n_experts, top_k, n_tokens, counts, psum, aux_out,
                                         static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "launching the balancing scalar");
  return MOE_OK;
}

moe_status moe_get_device_status(moe_plan_t plan, const void* workspace, void* stream) {
  if (!plan || !workspace) return fail(MOE_ERR_INVALID_ARG, "null argument");
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "synchronising the stream");
  uint32_t hdr[2] = {0, 0};
  e = cudaMemcpy(hdr, static_cast<const char*>(workspace) + plan->layout.hdr, sizeof hdr, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "reading the status word");
  if (hdr[0] == 0) return MOE_OK;
  if (hdr[0] == MOE_ERR_TIMEOUT || hdr[0] == MOE_ERR_INTERNAL)
    return fail((moe_status)hdr[0], "device reported %s at site 0x%x", moe_status_string((moe_status)hdr[0]), hdr[1]);
  return fail(MOE_ERR_INTERNAL, "device status word holds unknown value %u", hdr[0]);
}

}  // extern "C"
