// bwd_tc.cu -- the router's two backward products on the tensor cores: the router-weight
// gradient and the input gradient (with the experts' slot gradients added).
//
// dW_r[e, c] = sum_t dlogit[t, e] x[t, c]   (backward of the router linear layer z = x W_r^T,
// "Distributed Training Part 4 ... MoE + Expert Parallelism", jesamkim ai-tech-blog, §3:
// the router is a linear layer followed by a softmax).
//
// D[M = experts (128 per tile), N = 128 columns of d] += A . B over K = tokens, with both
// operands MN-major straight from their row-major tensors: A = dlogit [T, E64] (E rounded
// up to 64, zero columns past E), B = x [T, d].  dlogit is fp32; it is carried as
// two bf16 terms hi = bf16(v), lo = bf16(v - hi) and both are multiplied into the same fp32
// accumulator, so the product keeps about 16 bits of dlogit (x is bf16 already).  Each CTA
// owns one (expert tile, column tile, token chunk) and writes its fp32 partial; a second
// kernel adds the chunks in their order (deterministic).
//
// Warp roles (192 threads): warp 0 TMA producer, warp 1 TMEM allocator + MMA issuer,
// warps 2..5 epilogue (TMEM lanes 32 (w % 4) ..).  Waits are bounded; a wait that runs out
// records MOE_ERR_TIMEOUT and the CTA finishes without its result.
#include <cuda.h>
#include <cuda_bf16.h>

#include "bwd_common.cuh"
#include "gemm_bwd.h"
#include "gemm_tc.h"
#include "tc_ptx.cuh"

namespace moe {
namespace {

using namespace bwd;

constexpr int kBK = 64;        // tokens per K block
constexpr int kTM = 128;       // experts per tile
constexpr int kTN = 128;       // columns per tile
constexpr int kStages = 2;
constexpr int kABytes = 2 * kBoxBytes;               // 128 experts, one term
constexpr int kBBytes = 2 * kBoxBytes;               // 128 columns
constexpr int kStageBytes = 2 * kABytes + kBBytes;   // hi, lo, x: 48 KB
constexpr int kThreads = 192;

struct Ctl {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t tfull;
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};
constexpr size_t kSmemBytes = 1024 + (size_t)kStages * kStageBytes + sizeof(Ctl);


__global__ void __launch_bounds__(kThreads) dwr_tc_kernel(const __grid_constant__ CUtensorMap tmHi,
                                                         const __grid_constant__ CUtensorMap tmLo,
                                                         const __grid_constant__ CUtensorMap tmX, Shape s, Ws ws,
                                                         int chunk_tokens, int64_t timeout_ns) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* stages = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Ctl* ctl = reinterpret_cast<Ctl*>(stages + kStages * kStageBytes);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * kTN;
  const int m0 = blockIdx.y * kTM;
  const int chunk = blockIdx.z;
  const int64_t t0 = (int64_t)chunk * chunk_tokens;
  int64_t t1 = t0 + chunk_tokens;
  if (t1 > s.T) t1 = s.T;
  const int kblocks = t1 > t0 ? (int)((t1 - t0 + kBK - 1) / kBK) : 0;  // rows past T read as zero

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      ptx::mbar_init(ptx::smem_u32(&ctl->full[i]), 1);
      ptx::mbar_init(ptx::smem_u32(&ctl->empty[i]), 1);
    }
    ptx::mbar_init(ptx::smem_u32(&ctl->tfull), 1);
    ptx::mbar_init(ptx::smem_u32(&ctl->drain), 1);
    ctl->abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(&ctl->tmem_base), kTN);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  volatile int* abort_flag = &ctl->abort;
  pdl_wait();  // dlogit comes from the router backward
  pdl_launch_dependents();
  uint32_t issued = 0, issued_phase = 0;

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      for (int kb = 0; kb < kblocks; ++kb) {
        if (!ptx::mbar_wait(ptx::smem_u32(&ctl->empty[stage]), phase ^ 1u, timeout_ns, abort_flag)) {
          *abort_flag = 1;
          record_error(ws, MOE_ERR_TIMEOUT, 0xA00u);
          break;
        }
        const uint32_t bar = ptx::smem_u32(&ctl->full[stage]);
        const uint32_t sa = ptx::smem_u32(stages + (size_t)stage * kStageBytes);
        const int trow = (int)(t0 + (int64_t)kb * kBK);
        ptx::mbar_arrive_expect_tx(bar, kStageBytes);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          ptx::tma_load_2d(sa + j * kBoxBytes, &tmHi, m0 + 64 * j, trow, bar);
          ptx::tma_load_2d(sa + kABytes + j * kBoxBytes, &tmLo, m0 + 64 * j, trow, bar);
          ptx::tma_load_2d(sa + 2 * kABytes + j * kBoxBytes, &tmX, n0 + 64 * j, trow, bar);
        }
        issued |= 1u << stage;
        issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = ptx::idesc_bf16_f32(kTM, kTN) | (1u << 15) | (1u << 16);  // A, B MN-major
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int kb = 0; kb < kblocks; ++kb) {
        if (!ptx::mbar_wait(ptx::smem_u32(&ctl->full[stage]), phase, timeout_ns, abort_flag)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t sa = ptx::smem_u32(stages + (size_t)stage * kStageBytes);
#pragma unroll
        for (int ks = 0; ks < kBK / 16; ++ks) {
          const uint64_t bdesc = desc_mnmajor_sw128(sa + 2 * kABytes + ks * 2048);
          ptx::mma_bf16(tmem, desc_mnmajor_sw128(sa + ks * 2048), bdesc, idesc, (kb | ks) != 0 ? 1u : 0u);
          ptx::mma_bf16(tmem, desc_mnmajor_sw128(sa + kABytes + ks * 2048), bdesc, idesc, 1u);
        }
        ptx::mma_commit(ptx::smem_u32(&ctl->empty[stage]));
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (ok) {
        ptx::mma_commit(ptx::smem_u32(&ctl->tfull));
      } else {
        *abort_flag = 1;
        record_error(ws, MOE_ERR_TIMEOUT, 0xA10u);
      }
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- epilogue
    const int q = warp & 3;
    const int e = m0 + q * 32 + lane;
    bool ok = kblocks == 0 || ptx::mbar_wait(ptx::smem_u32(&ctl->tfull), 0u, timeout_ns, abort_flag);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) {
      if (lane == 0) record_error(ws, MOE_ERR_TIMEOUT, 0xA20u);
    } else {
      ptx::tc_fence_after();
      float* out = ws.dwr_part + ((int64_t)chunk * s.E + e) * s.d + n0;
#pragma unroll 1
      for (int c = 0; c < kTN; c += 32) {
        if (n0 + c >= s.d) break;  // uniform
        uint32_t v[32];
        if (kblocks > 0) {
          ptx::tmem_ld_32cols(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)c, v);
          ptx::tmem_ld_wait();
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = 0u;
        }
        if (e < s.E) {
          float4* o4 = reinterpret_cast<float4*>(out + c);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            o4[i] = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]), __uint_as_float(v[4 * i + 2]),
                                __uint_as_float(v[4 * i + 3]));
        }
      }
    }
  }

  __syncthreads();
  if (*abort_flag) {
    if (warp == 0 && lane == 0)
      for (int st = 0; st < kStages; ++st)
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
    ptx::tmem_dealloc(tmem, kTN);
  }
}

// ------------------------------------------------------------------------------------------
// dx[t, c] = sum_e dlogit[t, e] W_r[e, c] + sum_{j<k} dXslot[t k + j, c]
// (the router's input gradient plus the experts' input gradients of the token's k slots).
// D[M = 128 tokens, N = 128 columns] += A . B over K = experts, A = dlogit [T, E64] K-major
// (the hi and lo bf16 terms), B = W_r [E, d] MN-major (rows past E read as zero).  The
// epilogue turns each warp's 32 x 32 blocks around in shared memory and then adds the k slot
// rows and writes dx with four lanes per row segment (coalesced).
constexpr int kDxTM = 128, kDxTN = 128;
constexpr int kDxABytes = kDxTM * kBK * 2;                   // 16 KB per term
constexpr int kDxStageBytes = 2 * kDxABytes + 2 * kBoxBytes;  // hi, lo, W_r: 48 KB
constexpr int kDxXposeBytes = 32 * 32 * 4;
// Eight epilogue warps (two per TMEM lane quarter, 64 columns each) and one stage (the expert
// dimension is only 1..4 K blocks) so that two CTAs share an SM: the epilogue's slot-row
// loads are what the kernel waits on, and more warps keep more of them in flight.
constexpr int kDxThreads = 320;
constexpr int kDxEpiWarps = 8;
constexpr size_t kDxSmemBytes = 1024 + (size_t)kDxStageBytes + kDxEpiWarps * (size_t)kDxXposeBytes + sizeof(Ctl);



__global__ void __launch_bounds__(kDxThreads) dx_tc_kernel(const __grid_constant__ CUtensorMap tmHi,
                                                        const __grid_constant__ CUtensorMap tmLo,
                                                        const __grid_constant__ CUtensorMap tmW, Shape s, Ws ws,
                                                        float* dx, int64_t timeout_ns) {
  constexpr int nst = 1;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* stages = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* xpose = stages + nst * kDxStageBytes;
  Ctl* ctl = reinterpret_cast<Ctl*>(xpose + kDxEpiWarps * kDxXposeBytes);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * kDxTN;
  const int64_t t0 = (int64_t)blockIdx.y * kDxTM;
  const int kblocks = dlogit_cols(s) / kBK;

  if (threadIdx.x == 0) {
    for (int i = 0; i < nst; ++i) {
      ptx::mbar_init(ptx::smem_u32(&ctl->full[i]), 1);
      ptx::mbar_init(ptx::smem_u32(&ctl->empty[i]), 1);
    }
    ptx::mbar_init(ptx::smem_u32(&ctl->tfull), 1);
    ptx::mbar_init(ptx::smem_u32(&ctl->drain), 1);
    ctl->abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(&ctl->tmem_base), kDxTN);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  volatile int* abort_flag = &ctl->abort;
  pdl_wait();  // dlogit comes from the router backward, the slot gradients from the dX GEMM
  pdl_launch_dependents();
  uint32_t issued = 0, issued_phase = 0;

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      for (int kb = 0; kb < kblocks; ++kb) {
        if (!ptx::mbar_wait(ptx::smem_u32(&ctl->empty[stage]), phase ^ 1u, timeout_ns, abort_flag)) {
          *abort_flag = 1;
          record_error(ws, MOE_ERR_TIMEOUT, 0xA40u);
          break;
        }
        const uint32_t bar = ptx::smem_u32(&ctl->full[stage]);
        const uint32_t sa = ptx::smem_u32(stages + (size_t)stage * kDxStageBytes);
        ptx::mbar_arrive_expect_tx(bar, kDxStageBytes);
        ptx::tma_load_2d(sa, &tmHi, kb * kBK, (int)t0, bar);
        ptx::tma_load_2d(sa + kDxABytes, &tmLo, kb * kBK, (int)t0, bar);
#pragma unroll
        for (int j = 0; j < 2; ++j) ptx::tma_load_2d(sa + 2 * kDxABytes + j * kBoxBytes, &tmW, n0 + 64 * j, kb * kBK, bar);
        issued |= 1u << stage;
        issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
        if (++stage == nst) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = ptx::idesc_bf16_f32(kDxTM, kDxTN) | (1u << 16);  // B MN-major
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int kb = 0; kb < kblocks; ++kb) {
        if (!ptx::mbar_wait(ptx::smem_u32(&ctl->full[stage]), phase, timeout_ns, abort_flag)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t sa = ptx::smem_u32(stages + (size_t)stage * kDxStageBytes);
#pragma unroll
        for (int ks = 0; ks < kBK / 16; ++ks) {
          const uint64_t bdesc = desc_mnmajor_sw128(sa + 2 * kDxABytes + ks * 2048);
          ptx::mma_bf16(tmem, ptx::desc_kmajor_sw128(sa + ks * 32), bdesc, idesc, (kb | ks) != 0 ? 1u : 0u);
          ptx::mma_bf16(tmem, ptx::desc_kmajor_sw128(sa + kDxABytes + ks * 32), bdesc, idesc, 1u);
        }
        ptx::mma_commit(ptx::smem_u32(&ctl->empty[stage]));
        if (++stage == nst) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (ok) {
        ptx::mma_commit(ptx::smem_u32(&ctl->tfull));
      } else {
        *abort_flag = 1;
        record_error(ws, MOE_ERR_TIMEOUT, 0xA50u);
      }
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- epilogue
    const int q = warp & 3;
    bool ok = ptx::mbar_wait(ptx::smem_u32(&ctl->tfull), 0u, timeout_ns, abort_flag);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) {
      if (lane == 0) record_error(ws, MOE_ERR_TIMEOUT, 0xA60u);
    } else {
      ptx::tc_fence_after();
      const uint32_t xb = ptx::smem_u32(xpose + (warp - 2) * kDxXposeBytes);
      const int cg = (lane & 3) * 8;  // column group of this lane in a 32-column chunk
      const int c_beg = ((warp - 2) >> 2) * (kDxTN / 2);
#pragma unroll 1
      for (int c = c_beg; c < c_beg + kDxTN / 2; c += 32) {
        if (n0 + c >= s.d) break;  // uniform; d is a multiple of 64
        uint32_t v[32];
        ptx::tmem_ld_32cols(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)c, v);
        ptx::tmem_ld_wait();
        stage_row32(xb, lane, v);
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int br = 8 * i + (lane >> 2);  // row of the block
          const int64_t t = t0 + q * 32 + br;
          float a[8];
          ld_block_v4(xb + (uint32_t)br * 128u + (uint32_t)(((cg >> 2) ^ (br & 7)) * 16), a[0], a[1], a[2], a[3]);
          ld_block_v4(xb + (uint32_t)br * 128u + (uint32_t)((((cg >> 2) + 1) ^ (br & 7)) * 16), a[4], a[5], a[6], a[7]);
          if (t < s.T) {
            const int64_t col = n0 + c + cg;
            for (int j = 0; j < s.k; ++j) {
              const uint4 raw = *reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(ws.dxslot) +
                                                                (t * s.k + j) * s.d + col);
              const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const float2 f = __bfloat1622float2(h2[u]);
                a[2 * u] += f.x;
                a[2 * u + 1] += f.y;
              }
            }
            float4* o = reinterpret_cast<float4*>(dx + t * s.d + col);
            o[0] = make_float4(a[0], a[1], a[2], a[3]);
            o[1] = make_float4(a[4], a[5], a[6], a[7]);
          }
        }
        __syncwarp();  // the block is read before the next chunk overwrites it
      }
    }
  }

  __syncthreads();
  if (*abort_flag) {
    if (warp == 0 && lane == 0)
      for (int st = 0; st < nst; ++st)
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
    ptx::tmem_dealloc(tmem, kDxTN);
  }
}

}  // namespace

int dwr_chunk_tokens(const Shape& s) {
  int64_t c = (s.T + kDwrMaxChunks - 1) / kDwrMaxChunks;
  c = (c + kBK - 1) / kBK * kBK;
  return (int)(c < kBK ? kBK : c);
}

int dwr_chunks(const Shape& s) {
  const int64_t c = dwr_chunk_tokens(s);
  return (int)((s.T + c - 1) / c);
}

cudaError_t launch_dwr_tc(const Shape& s, const Ws& ws, const void* x, int64_t timeout_ns, bool pdl, cudaStream_t st) {
  CUtensorMap mh, ml, mx;
  cudaError_t e;
  const uint64_t e8 = (uint64_t)dlogit_cols(s);
  if ((e = make_tmap_bf16(&mh, ws.dl_hi, (uint64_t)s.T, e8, 64)) != cudaSuccess) return e;
  if ((e = make_tmap_bf16(&ml, ws.dl_lo, (uint64_t)s.T, e8, 64)) != cudaSuccess) return e;
  if ((e = make_tmap_bf16(&mx, x, (uint64_t)s.T, (uint64_t)s.d, 64)) != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(dwr_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes)) !=
      cudaSuccess)
    return e;
  const dim3 g((unsigned)((s.d + kTN - 1) / kTN), (unsigned)((s.E + kTM - 1) / kTM), (unsigned)dwr_chunks(s));
  return launch_kernel(dwr_tc_kernel, g, dim3(kThreads), kSmemBytes, st, pdl, 1, mh, ml, mx, s, ws,
                       dwr_chunk_tokens(s), timeout_ns);
}

cudaError_t launch_dx_tc(const Shape& s, const Ws& ws, const void* w_router, float* dx, int64_t timeout_ns, bool pdl,
                         cudaStream_t st) {
  CUtensorMap mh, ml, mw;
  cudaError_t e;
  const uint64_t ec = (uint64_t)dlogit_cols(s);
  if ((e = make_tmap_bf16(&mh, ws.dl_hi, (uint64_t)s.T, ec, kDxTM)) != cudaSuccess) return e;
  if ((e = make_tmap_bf16(&ml, ws.dl_lo, (uint64_t)s.T, ec, kDxTM)) != cudaSuccess) return e;
  if ((e = make_tmap_bf16(&mw, w_router, (uint64_t)s.E, (uint64_t)s.d, 64)) != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(dx_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kDxSmemBytes)) !=
      cudaSuccess)
    return e;
  const dim3 g((unsigned)((s.d + kDxTN - 1) / kDxTN), (unsigned)((s.T + kDxTM - 1) / kDxTM));
  return launch_kernel(dx_tc_kernel, g, dim3(kDxThreads), kDxSmemBytes, st, pdl, 1, mh, ml, mw, s, ws, dx, timeout_ns);
}

}  // namespace moe
