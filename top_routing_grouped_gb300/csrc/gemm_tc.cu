// gemm_tc.cu -- persistent grouped expert GEMMs on the 5th-generation tensor cores (sm_103a):
// TMA tiled loads into a shared-memory ring, one thread issuing tcgen05.mma into TMEM
// accumulators, and four epilogue warps reading TMEM back with tcgen05.ld.
//
// After "Distributed Training Part 4 ... MoE + Expert Parallelism" (jesamkim ai-tech-blog):
// §3 Structure (each expert an independent FFN; SwiGLU form E_e(v) = W2_e (SiLU(W1_e v) *
// (W3_e v))), §3 output formula (expert output weighted by the gate), §4 Combine (outputs
// return to their token slot).  The grouped GEMM is the compute item named by
// "Compute-Optimal Is Not Cluster-Optimal" (operator-level performance model).
//
//   mode 1:  H[p, n]          = SiLU(Xp[p] . W1_e[n]) * (Xp[p] . W3_e[n])   (MMA N = 128 + 128)
//   mode 2:  Yp[p, n] = gate(p) * (H[p] . W2_e[n]), row p in expert order          (MMA N = 256)
//
// Work: the tile table of the scan kernel (m-tiles of 128 rows of one expert, grouped so
// that CTAs running together share weight tiles in L2) times the n-tiles.  Every CTA
// loops over tiles blockIdx.x, blockIdx.x + gridDim.x, ... (one CTA per SM).
//
// Warp roles (256 threads):
//   warp 0      TMA producer: A tile [128 x 64] + B tile [256 x 64] per stage
//   warp 1      MMA issuer: 4 x tcgen05.mma (M128 N256 K16) per stage, commit frees the stage
//   warp 2      TMEM allocator (2 accumulators x 256 fp32 columns = 512 columns)
//   warps 4..7  epilogue: warp w reads TMEM lanes 32*(w%4).. (its 32 rows of the tile)
// TMEM is double-buffered so the epilogue of tile i overlaps the main loop of tile i+1.
// Every mbarrier wait is bounded; a wait that runs out records MOE_ERR_TIMEOUT, raises the
// CTA's abort flag, and all roles leave their loops, drain in-flight copies and MMAs, and
// free TMEM before the CTA exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "gemm_tc.h"
#include "tmap.h"
#include "tc_ptx.cuh"

namespace moe {
namespace {

constexpr int kBK = 64;                       // K elements per stage: one 128-byte swizzle row
constexpr int kStages = 4;
constexpr int kMmaM = 128;
constexpr int kMmaN = 256;
constexpr int kMmaK = 16;
constexpr int kABytes = kMmaM * kBK * 2;      // 16 KB
constexpr int kBBytes = kMmaN * kBK * 2;      // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kAccCols = kMmaN;               // fp32 accumulator columns per buffer
constexpr int kTmemCols = 2 * kAccCols;
constexpr int kThreads = 256;
constexpr int kEpiWarp0 = 4;
constexpr int kEpiThreads = 128;

struct Ctl {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

constexpr size_t kSmemBytes = 1024 /* alignment slack */ + (size_t)kStages * kStageBytes + sizeof(Ctl);

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float silu(float a) { return silu_fast(a); }

template <int kMode>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmB3, Shape s, Ws ws, int64_t timeout_ns, int stall) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* stages = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Ctl* ctl = reinterpret_cast<Ctl*>(stages + kStages * kStageBytes);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const int ncols = kMode == 1 ? s.F : s.d;           // output columns
  const int K = kMode == 1 ? s.d : s.F;               // reduction length (multiple of 64)
  const int bn = kMode == 1 ? kMmaN / 2 : kMmaN;      // output columns per tile
  const int n_tiles = (ncols + bn - 1) / bn;
  const int kblocks = K / kBK;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      ptx::mbar_init(ptx::smem_u32(&ctl->full[i]), 1);
      ptx::mbar_init(ptx::smem_u32(&ctl->empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(ptx::smem_u32(&ctl->tfull[i]), 1);
      ptx::mbar_init(ptx::smem_u32(&ctl->tempty[i]), kEpiThreads);
    }
    ptx::mbar_init(ptx::smem_u32(&ctl->drain), 1);
    ctl->abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::tma_prefetch_desc(&tmA);
    ptx::tma_prefetch_desc(&tmB);
    if (kMode == 1) ptx::tma_prefetch_desc(&tmB3);
  }
  if (warp == 2) {
    ptx::tmem_alloc(ptx::smem_u32(&ctl->tmem_base), kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  volatile int* abort_flag = &ctl->abort;
  pdl_wait();  // the tile table and the A operand come from the previous kernels
  pdl_launch_dependents();
  const int total = (int)ws.hdr[kHdrNumMTiles] * n_tiles;

  // fills issued by the producer whose landing nobody may have waited for (abort path)
  uint32_t issued = 0, issued_phase = 0;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ TMA producer
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true, first = true;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        const TileInfo ti = decode_tile(ws, n_tiles, tile);
        const int brow = kMode == 1 ? ti.e * s.F + ti.n_idx * bn : ti.e * s.d + ti.n_idx * bn;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!ptx::mbar_wait(ptx::smem_u32(&ctl->empty[stage]), phase ^ 1u, timeout_ns, abort_flag)) {
            ok = false;
            break;
          }
          if (!(stall && first)) {  // the stall hook withholds exactly one fill
            const uint32_t bar = ptx::smem_u32(&ctl->full[stage]);
            const uint32_t sa = ptx::smem_u32(stages + (size_t)stage * kStageBytes);
            ptx::mbar_arrive_expect_tx(bar, kStageBytes);
            ptx::tma_load_2d(sa, &tmA, kb * kBK, ti.row0, bar);
            if (kMode == 1) {
              ptx::tma_load_2d(sa + kABytes, &tmB, kb * kBK, brow, bar);
              ptx::tma_load_2d(sa + kABytes + kBBytes / 2, &tmB3, kb * kBK, brow, bar);
            } else {
              ptx::tma_load_2d(sa + kABytes, &tmB, kb * kBK, brow, bar);
            }
            issued |= 1u << stage;
            issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
          }
          first = false;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        *abort_flag = 1;
        record_error(ws, MOE_ERR_TIMEOUT, 0x500u + kMode);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      constexpr uint32_t idesc = ptx::idesc_bf16_f32(kMmaM, kMmaN);
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        if (!ptx::mbar_wait(ptx::smem_u32(&ctl->tempty[acc]), acc_phase ^ 1u, timeout_ns, abort_flag)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem + (uint32_t)(acc * kAccCols);
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!ptx::mbar_wait(ptx::smem_u32(&ctl->full[stage]), phase, timeout_ns, abort_flag)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t sa = ptx::smem_u32(stages + (size_t)stage * kStageBytes);
          const uint32_t sb = sa + kABytes;
#pragma unroll
          for (int ks = 0; ks < kBK / kMmaK; ++ks) {
            ptx::mma_bf16(d_tmem, ptx::desc_kmajor_sw128(sa + ks * kMmaK * 2), ptx::desc_kmajor_sw128(sb + ks * kMmaK * 2),
                          idesc, (kb | ks) != 0 ? 1u : 0u);
          }
          ptx::mma_commit(ptx::smem_u32(&ctl->empty[stage]));  // frees the stage once these MMAs finish
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        ptx::mma_commit(ptx::smem_u32(&ctl->tfull[acc]));  // accumulator ready for the epilogue
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      if (!ok) {
        *abort_flag = 1;
        record_error(ws, MOE_ERR_TIMEOUT, 0x510u + kMode);
      }
    }
    __syncwarp();
  } else if (warp >= kEpiWarp0) {
    // -------------------------------------------------------------- epilogue
    const int q = warp & 3;              // TMEM lane quarter this warp may read
    const int r = q * 32 + lane;         // row of the tile
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      const TileInfo ti = decode_tile(ws, n_tiles, tile);
      ok = ptx::mbar_wait(ptx::smem_u32(&ctl->tfull[acc]), acc_phase, timeout_ns, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      ptx::tc_fence_after();
      const uint32_t t_row = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * kAccCols);
      const bool valid = r < ti.rows;
      const int64_t p = (int64_t)ti.row0 + r;
      const int n0 = ti.n_idx * bn;
      if (kMode == 1) {
        __nv_bfloat16* hrow = reinterpret_cast<__nv_bfloat16*>(ws.h) + p * s.F + n0;
#pragma unroll 1
        for (int c = 0; c < kMmaN / 2; c += 32) {
          uint32_t a[32], g[32];
          ptx::tmem_ld_32cols(t_row + c, a);
          ptx::tmem_ld_32cols(t_row + kMmaN / 2 + c, g);
          ptx::tmem_ld_wait();
          if (valid && n0 + c < s.F) {
            uint4* dst = reinterpret_cast<uint4*>(hrow + c);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              uint4 o;
              uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const int i = v * 8 + u * 2;
                const float h0 = silu(__uint_as_float(a[i])) * __uint_as_float(g[i]);
                const float h1 = silu(__uint_as_float(a[i + 1])) * __uint_as_float(g[i + 1]);
                ow[u] = pack_bf16x2(h0, h1);
              }
              dst[v] = o;
            }
            if (s.training) {  // keep W1.x and W3.x of the row for the backward
              uint4* da1 = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(ws.a1) + p * s.F + n0 + c);
              uint4* da3 = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(ws.a3) + p * s.F + n0 + c);
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                uint4 o1, o3;
                uint32_t* w1p = reinterpret_cast<uint32_t*>(&o1);
                uint32_t* w3p = reinterpret_cast<uint32_t*>(&o3);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                  const int i = v * 8 + u * 2;
                  w1p[u] = pack_bf16x2(__uint_as_float(a[i]), __uint_as_float(a[i + 1]));
                  w3p[u] = pack_bf16x2(__uint_as_float(g[i]), __uint_as_float(g[i + 1]));
                }
                da1[v] = o1;
                da3[v] = o3;
              }
            }
          }
        }
      } else {
        const float gate = valid ? ws.gate_perm[p] : 0.f;
        __nv_bfloat16* yrow = reinterpret_cast<__nv_bfloat16*>(ws.yp) + p * s.d + n0;
#pragma unroll 1
        for (int c = 0; c < kMmaN; c += 32) {
          uint32_t a[32];
          ptx::tmem_ld_32cols(t_row + c, a);
          ptx::tmem_ld_wait();
          if (valid && n0 + c < s.d) {
            uint4* dst = reinterpret_cast<uint4*>(yrow + c);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              uint4 o;
              uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const int i = v * 8 + u * 2;
                ow[u] = pack_bf16x2(gate * __uint_as_float(a[i]), gate * __uint_as_float(a[i + 1]));
              }
              dst[v] = o;
            }
          }
        }
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(ptx::smem_u32(&ctl->tempty[acc]));
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (!ok && lane == 0) {
      *abort_flag = 1;
      record_error(ws, MOE_ERR_TIMEOUT, 0x530u + kMode);
    }
  }

  // ---------------------------------------------------------------- teardown
  __syncthreads();
  if (*abort_flag) {
    if (warp == 0 && lane == 0) {
      // let every fill this CTA issued land before its shared memory goes away
      for (int st = 0; st < kStages; ++st)
        if (issued & (1u << st))
          ptx::mbar_wait(ptx::smem_u32(&ctl->full[st]), (issued_phase >> st) & 1u, timeout_ns, nullptr);
    }
    if (warp == 1 && lane == 0) {
      // wait for every MMA this thread issued before TMEM is released
      ptx::mma_commit(ptx::smem_u32(&ctl->drain));
      ptx::mbar_wait(ptx::smem_u32(&ctl->drain), 0u, timeout_ns, nullptr);
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D bf16 row-major [rows, cols] tensor, boxes of [box_rows, 64] with 128-byte swizzle.
cudaError_t make_tmap_bf16(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kBK, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_tmap_f32_rows128(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 4};
  const cuuint32_t box[2] = {32, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t launch_gemm_tc(int mode, const Shape& s, const Ws& ws, const Weights& w, int num_sms,
                           int64_t timeout_ns, bool test_stall, bool pdl, cudaStream_t st) {
  CUtensorMap mA, mB, mB3;
  cudaError_t e;
  if (mode == 1) {
    if ((e = make_tmap_bf16(&mA, ws.xp, (uint64_t)s.N, (uint64_t)s.d, kMmaM)) != cudaSuccess) return e;
    if ((e = make_tmap_bf16(&mB, w.w1, (uint64_t)s.E * s.F, (uint64_t)s.d, kMmaN / 2)) != cudaSuccess) return e;
    if ((e = make_tmap_bf16(&mB3, w.w3, (uint64_t)s.E * s.F, (uint64_t)s.d, kMmaN / 2)) != cudaSuccess) return e;
    if ((e = cudaFuncSetAttribute(gemm_tc_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes)) !=
        cudaSuccess)
      return e;
    return launch_kernel(gemm_tc_kernel<1>, dim3(num_sms), dim3(kThreads), kSmemBytes, st, pdl, 1, mA, mB, mB3, s, ws,
                         timeout_ns, test_stall ? 1 : 0);
  } else {
    if ((e = make_tmap_bf16(&mA, ws.h, (uint64_t)s.N, (uint64_t)s.F, kMmaM)) != cudaSuccess) return e;
    if ((e = make_tmap_bf16(&mB, w.w2, (uint64_t)s.E * s.d, (uint64_t)s.F, kMmaN)) != cudaSuccess) return e;
    if ((e = cudaFuncSetAttribute(gemm_tc_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes)) !=
        cudaSuccess)
      return e;
    return launch_kernel(gemm_tc_kernel<2>, dim3(num_sms), dim3(kThreads), kSmemBytes, st, pdl, 1, mA, mB, mB, s, ws,
                         timeout_ns, test_stall ? 1 : 0);
  }
}

}  // namespace moe
