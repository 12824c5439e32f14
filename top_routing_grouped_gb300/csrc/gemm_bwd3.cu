// gemm_bwd3.cu -- the backward's weight-gradient GEMMs (grouped over K, the expert's routed
// rows) on CTA pairs (2-SM tcgen05.mma, cta_group::2).
//
// Backward of "Distributed Training Part 4 ... MoE + Expert Parallelism" (jesamkim
// ai-tech-blog) §3 (SwiGLU experts, gate-weighted sum), for expert e over its rows p:
//   kDW13 [dW1_e; dW3_e][m, c] = sum_p [da|db][p, m] Xp[p, c]
//   kDW2  dW2_e[c, f]          = sum_p g_p dy[t_p, c] h[p, f]
// Both operands are MN-major (64 x 64 TMA boxes side by side).  A cluster of two CTAs
// computes a 256 (weight rows) x 256 (columns) tile: each CTA loads its own 128 weight rows of
// A and 128 of the 256 B columns for the same K rows.
//
// The K range is the expert's rows, so its last 64-row block runs past the expert's end.  For
// that block A comes from dab_tail / dop_tail, which repeat the expert's rows of that block and
// are zero past its end; B (Xp, h) runs on into the next expert's rows (or TMA's zero fill past
// the last row), which the zeros cancel.  Every block is an ordinary pair load: no block is
// masked in shared memory and the two CTAs need no extra handshake.
//
// The fp32 gradient leaves through 32 x 32 swizzled shared-memory blocks and TMA stores.
// Waits are bounded (MOE_ERR_TIMEOUT, no trap); an abort raises the flag in both CTAs; the
// pair meets at cluster barriers before TMEM is released.
#include <cuda.h>
#include <cuda_bf16.h>

#include "bwd_common.cuh"
#include "gemm_bwd.h"
#include "gemm_tc.h"
#include "tc_ptx.cuh"
#include "tmap.h"

namespace moe {
namespace {

using namespace bwd;

constexpr int kBK = 64;
constexpr int kStages = 6;
constexpr int kMmaM = 256;  // both CTAs
constexpr int kMmaN = 256;
constexpr int kABytes = 2 * kBoxBytes;  // this CTA's 128 weight rows
constexpr int kBBytes = 2 * kBoxBytes;  // this CTA's 128 of the 256 columns
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kAccCols = kMmaN;
constexpr int kThreads = 384;
constexpr int kEpiWarp0 = 4;
constexpr int kEpiWarps = 8;  // two per TMEM lane quarter, one per 128-column half
constexpr int kOutBlockBytes = 32 * 128;

struct Ctl3 {
  uint64_t full[kStages];    // leader's: the stage's bytes (both CTAs')
  uint64_t empty[kStages];   // each CTA: stage free again (leader's multicast commit)
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  uint32_t peer_tmem_base;
  int abort;
};

constexpr size_t kSmemBytes =
    1024 + (size_t)kStages * kStageBytes + (size_t)kEpiWarps * kOutBlockBytes + sizeof(Ctl3);

struct KTile {
  int e, n_idx, row0, rows;  // row0/rows: this CTA's weight rows (rows <= 0: none)
  int k_row0, kblocks;
  int a_tail;  // row of the expert's last, partial block in dab_tail / dop_tail, or -1
};

template <int kKind>
__device__ __forceinline__ KTile decode_k(const Shape& s, const Ws& ws, int tile, int m_pairs, int n_tiles, int M,
                                          int rank) {
  KTile t;
  const int per_e = m_pairs * n_tiles;
  t.e = tile / per_e;
  const int local = tile % per_e;
  t.n_idx = local / m_pairs;
  t.row0 = (local % m_pairs) * kMmaM + rank * (kMmaM / 2);
  t.rows = M - t.row0 < kMmaM / 2 ? M - t.row0 : kMmaM / 2;
  const int cnt = __ldg(&ws.counts[t.e]);
  t.k_row0 = __ldg(&ws.offsets[t.e]);
  t.kblocks = (cnt + kBK - 1) / kBK;
  t.a_tail = cnt % kBK != 0 ? t.e * kBK : -1;
  return t;
}

__device__ __forceinline__ void raise_abort(Ctl3* ctl, uint32_t rank) {
  ctl->abort = 1;
  ptx::st_cluster_u32(ptx::mapa(ptx::smem_u32(&ctl->abort), rank ^ 1u), 1u);
}

template <int kKind>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_dw_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmAT,
                        const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmO1, const __grid_constant__ CUtensorMap tmO2, Shape s,
                        Ws ws, int64_t timeout_ns) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* stages = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* out_blocks = stages + kStages * kStageBytes;  // 1024-byte aligned
  Ctl3* ctl = reinterpret_cast<Ctl3*>(out_blocks + kEpiWarps * kOutBlockBytes);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();
  const bool leader = rank == 0;
  const int cid = (int)ptx::cluster_id_x();
  const int ncl = (int)ptx::cluster_count_x();

  const int M = kKind == kBwdDW13 ? 2 * s.F : s.d;
  const int N = kKind == kBwdDW13 ? s.d : s.F;
  const int m_pairs = (M + kMmaM - 1) / kMmaM;
  const int n_tiles = (N + kMmaN - 1) / kMmaN;
  const int total = s.E * m_pairs * n_tiles;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      ptx::mbar_init(ptx::smem_u32(&ctl->full[i]), 1);
      ptx::mbar_init(ptx::smem_u32(&ctl->empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(ptx::smem_u32(&ctl->tfull[i]), 1);
      ptx::mbar_init(ptx::smem_u32(&ctl->tempty[i]), 2 * kEpiWarps);
    }
    ptx::mbar_init(ptx::smem_u32(&ctl->drain), 1);
    ctl->abort = 0;
    ctl->peer_tmem_base = 0xFFFFFFFFu;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::tma_prefetch_desc(&tmA);
    ptx::tma_prefetch_desc(&tmAT);
    ptx::tma_prefetch_desc(&tmB);
  }
  ptx::cluster_sync();  // both CTAs' barriers exist before any cross-CTA arrive or load
  if (warp == 2) {
    ptx::tmem_alloc_pair(ptx::smem_u32(&ctl->tmem_base), 2 * kAccCols);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  if (threadIdx.x == 0) ptx::st_cluster_u32(ptx::mapa(ptx::smem_u32(&ctl->peer_tmem_base), rank ^ 1u), tmem);
  ptx::cluster_sync();
  pdl_wait();  // counts, offsets and the operands come from the previous kernels
  pdl_launch_dependents();
  int my_total = total;
  if (ctl->peer_tmem_base != tmem) {  // a pair's accumulators must sit at the same TMEM address
    if (threadIdx.x == 0) record_error(ws, MOE_ERR_INTERNAL, 0xB00u + kKind);
    my_total = 0;
  }
  volatile int* abort_flag = &ctl->abort;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------- TMA producer (both CTAs)
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int tile = cid; tile < my_total && ok; tile += ncl) {
        const KTile kt = decode_k<kKind>(s, ws, tile, m_pairs, n_tiles, M, (int)rank);
        const int nb = kt.n_idx * kMmaN + (int)rank * (kMmaN / 2);
        for (int kb = 0; kb < kt.kblocks; ++kb) {
          if (!ptx::mbar_wait(ptx::smem_u32(&ctl->empty[stage]), phase ^ 1u, timeout_ns, abort_flag)) {
            ok = false;
            break;
          }
          const int krow = kt.k_row0 + kb * kBK;  // B: Xp / h rows
          const bool tail = kb == kt.kblocks - 1 && kt.a_tail >= 0;
          const CUtensorMap* am = tail ? &tmAT : &tmA;  // A: the expert's tail block from its copy
          const int karow = tail ? kt.a_tail : krow;
          const uint32_t sa = ptx::smem_u32(stages + (size_t)stage * kStageBytes);
          const uint32_t full_local = ptx::smem_u32(&ctl->full[stage]);
          if (leader) ptx::mbar_arrive_expect_tx(full_local, 2 * kStageBytes);
          const uint32_t bar = ptx::mapa(full_local, 0);
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            ptx::tma_load_2d_pair(sa + j * kBoxBytes, am, kt.row0 + 64 * j, karow, bar);
            ptx::tma_load_2d_pair(sa + kABytes + j * kBoxBytes, &tmB, nb + 64 * j, krow, bar);
          }
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        record_error(ws, MOE_ERR_TIMEOUT, 0xB40u + kKind);
        raise_abort(ctl, rank);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // -------------------------------------------------------------- MMA issuer (leader)
    const uint32_t idesc = ptx::idesc_bf16_f32(kMmaM, kMmaN) | (1u << 15) | (1u << 16);  // A, B MN-major
    int stage = 0, acc = 0;
    uint32_t phase = 0, acc_phase = 0;
    bool ok = true;
    for (int tile = cid; leader && tile < my_total && ok; tile += ncl) {
      const KTile kt = decode_k<kKind>(s, ws, tile, m_pairs, n_tiles, M, (int)rank);
      ok = ptx::mbar_wait(ptx::smem_u32(&ctl->tempty[acc]), acc_phase ^ 1u, timeout_ns, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      ptx::tc_fence_after();
      const uint32_t d_tmem = tmem + (uint32_t)(acc * kAccCols);
      for (int kb = 0; kb < kt.kblocks; ++kb) {
        ok = ptx::mbar_wait(ptx::smem_u32(&ctl->full[stage]), phase, timeout_ns, abort_flag);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        ptx::tc_fence_after();
        if (lane == 0) {
          const uint32_t sa = ptx::smem_u32(stages + (size_t)stage * kStageBytes);
#pragma unroll
          for (int ks = 0; ks < kBK / 16; ++ks)
            ptx::mma_bf16_pair(d_tmem, desc_mnmajor_sw128(sa + ks * 2048), desc_mnmajor_sw128(sa + kABytes + ks * 2048),
                               idesc, (kb | ks) != 0 ? 1u : 0u);
          ptx::mma_commit_pair_multicast(ptx::smem_u32(&ctl->empty[stage]), 0x3);
        }
        __syncwarp();
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      if (lane == 0) ptx::mma_commit_pair_multicast(ptx::smem_u32(&ctl->tfull[acc]), 0x3);
      __syncwarp();
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (!ok && lane == 0) {
      record_error(ws, MOE_ERR_TIMEOUT, 0xB50u + kKind);
      raise_abort(ctl, rank);
    }
  } else if (warp >= kEpiWarp0) {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int q = warp & 3;
    const int half = (warp - kEpiWarp0) >> 2;  // columns [128 half, 128 half + 128)
    const int c_beg = half * (kMmaN / 2);
    const uint32_t ob = ptx::smem_u32(out_blocks + (warp - kEpiWarp0) * kOutBlockBytes);
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int tile = cid; tile < my_total; tile += ncl) {
      const KTile kt = decode_k<kKind>(s, ws, tile, m_pairs, n_tiles, M, (int)rank);
      ok = ptx::mbar_wait(ptx::smem_u32(&ctl->tfull[acc]), acc_phase, timeout_ns, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      ptx::tc_fence_after();
      const uint32_t t_row = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * kAccCols);
      const int n0 = kt.n_idx * kMmaN;
      // this warp's 32 weight rows (a whole block is valid or not: M is a multiple of 64)
      const int mblk = kt.row0 + q * 32;
      const bool blk_valid = q * 32 < kt.rows;
      const CUtensorMap* om = &tmO1;
      int orow;
      if (kKind == kBwdDW13) {
        if (mblk >= s.F) om = &tmO2;
        orow = kt.e * s.F + (mblk >= s.F ? mblk - s.F : mblk);
      } else {
        orow = kt.e * s.d + mblk;
      }
#pragma unroll 1
      for (int c = c_beg; c < c_beg + kMmaN / 2; c += 32) {
        if (n0 + c >= N) break;  // uniform
        uint32_t v[32];
        if (kt.kblocks > 0) {
          ptx::tmem_ld_32cols(t_row + c, v);
          ptx::tmem_ld_wait();
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = 0u;  // an expert without rows: zero gradient
        }
        if (blk_valid) {
          if (lane == 0) bulk_wait_read_all();  // the previous store has read the block
          __syncwarp();
          stage_row32(ob, lane, v);
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(om, n0 + c, orow, ob);
            bulk_commit();
          }
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_cluster(ptx::mapa(ptx::smem_u32(&ctl->tempty[acc]), 0));
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (!ok && lane == 0) {
      record_error(ws, MOE_ERR_TIMEOUT, 0xB70u + kKind);
      raise_abort(ctl, rank);
    }
    if (lane == 0) bulk_wait_all();  // this warp's stores are complete
  }

  // ---------------------------------------------------------------- teardown
  __syncthreads();
  if (leader && warp == 1 && lane == 0) {
    // every pair MMA of this pair has finished writing both CTAs' TMEM
    ptx::mma_commit_pair(ptx::smem_u32(&ctl->drain));
    ptx::mbar_wait(ptx::smem_u32(&ctl->drain), 0u, timeout_ns, nullptr);
  }
  __syncthreads();
  ptx::cluster_sync();  // neither CTA issues loads or MMAs any more
  if (*abort_flag && threadIdx.x == 0) {
    // copies already in flight land within microseconds; give them 200 us before the
    // shared memory they target goes away
    const uint64_t t0 = global_ns();
    while (global_ns() - t0 < 200000ull) {
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();
  if (warp == 2) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem, 2 * kAccCols);
  }
}

template <int kKind>
cudaError_t launch_dw_pair(const CUtensorMap& a, const CUtensorMap& at, const CUtensorMap& b, const CUtensorMap& o1,
                           const CUtensorMap& o2,
                           const Shape& s, const Ws& ws, int num_sms, int64_t timeout_ns, bool pdl, cudaStream_t st) {
  auto kern = gemm_dw_pair_kernel<kKind>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  int grid = num_sms & ~1;
  {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) == cudaSuccess && clusters > 0 && 2 * clusters < grid)
      grid = 2 * clusters;
  }
  return launch_kernel(kern, dim3((unsigned)grid), dim3(kThreads), kSmemBytes, st, pdl, 2, a, at, b, o1, o2, s, ws,
                       timeout_ns);
}

}  // namespace

cudaError_t launch_gemm_dw_pair(int kind, const Shape& s, const Ws& ws, float* dw_a, float* dw_b, int num_sms,
                                int64_t timeout_ns, bool pdl, cudaStream_t st) {
  CUtensorMap ma, mat, mb, mo1, mo2;
  cudaError_t e;
  const uint64_t N = (uint64_t)s.N, d = (uint64_t)s.d, F = (uint64_t)s.F, E = (uint64_t)s.E;
  if (kind == kBwdDW13) {
    if ((e = make_tmap_bf16(&ma, ws.dab, N, 2 * F, 64)) != cudaSuccess) return e;
    if ((e = make_tmap_bf16(&mat, ws.dab_tail, E * 64, 2 * F, 64)) != cudaSuccess) return e;
    if ((e = make_tmap_bf16(&mb, ws.xp, N, d, 64)) != cudaSuccess) return e;
    if ((e = make_tmap_f32_rows128(&mo1, dw_a, E * F, d, 32)) != cudaSuccess) return e;
    if ((e = make_tmap_f32_rows128(&mo2, dw_b, E * F, d, 32)) != cudaSuccess) return e;
    return launch_dw_pair<kBwdDW13>(ma, mat, mb, mo1, mo2, s, ws, num_sms, timeout_ns, pdl, st);
  }
  if (kind == kBwdDW2) {
    if ((e = make_tmap_bf16(&ma, ws.dop, N, d, 64)) != cudaSuccess) return e;
    if ((e = make_tmap_bf16(&mat, ws.dop_tail, E * 64, d, 64)) != cudaSuccess) return e;
    if ((e = make_tmap_bf16(&mb, ws.h, N, F, 64)) != cudaSuccess) return e;
    if ((e = make_tmap_f32_rows128(&mo1, dw_a, E * d, F, 32)) != cudaSuccess) return e;
    return launch_dw_pair<kBwdDW2>(ma, mat, mb, mo1, mo1, s, ws, num_sms, timeout_ns, pdl, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace moe
