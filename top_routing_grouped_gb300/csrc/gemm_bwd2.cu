// gemm_bwd2.cu -- the backward's two row-grouped GEMMs on CTA pairs (2-SM tcgen05.mma,
// cta_group::2), as the forward's pair kernels do for the forward GEMMs.
//
// Backward of "Distributed Training Part 4 ... MoE + Expert Parallelism" (jesamkim
// ai-tech-blog) §3 (SwiGLU experts, gate-weighted sum), for each routed row p of expert e:
//   kDH  dH'[p, f] = sum_c dy[t, c] W2_e[c, f]        (A = dYp K-major, B = W2 MN-major)
//        epilogue: dg partial = sum_f h[p,f] dH'[p,f];  da = g dH' b silu'(a),  db = g dH' silu(a),
//        with h = silu(a) b recomputed from the kept a, b (not read back)
//   kDX  dXslot[slot(p), c] = sum_f da[p,f] W1_e[f,c] + db[p,f] W3_e[f,c]
//                                                   (A = [da|db] K-major, B = W1|W3 MN-major)
// A cluster of two CTAs computes a 256 x 256 tile: each CTA loads its own 128 rows of A and
// 128 of the 256 B columns (two MN-major 64-column boxes), so an SM pulls 32 KB per 64-deep
// K step instead of the one-SM kernel's 48 KB.  The leader issues the MMAs and its commits
// free the stage in both CTAs and hand each CTA its 128 accumulator rows.  The dH epilogue
// turns each 32 x 32 block of dH' around in shared memory so that its loads of h, a, b and
// its stores of [da | db] move whole 64-byte row segments per four lanes; the dX epilogue
// is the one-SM kernel's (gemm_bwd.cu).  A [da | db] row in its expert's last, partial 64-row
// block is also written to dab_tail, which the weight-gradient GEMMs read for that block.
//
// Waits are bounded (MOE_ERR_TIMEOUT, no trap); an abort raises the flag in both CTAs; the
// pair meets at cluster barriers before TMEM is released.
#include <cuda.h>
#include <cuda_bf16.h>

#include "gemm_bwd.h"
#include "bwd_common.cuh"
#include "gemm_tc.h"
#include "tc_ptx.cuh"

namespace moe {
namespace {

using namespace bwd;

constexpr int kBK = 64;
constexpr int kStages = 6;
constexpr int kRowsPerCta = 128;
constexpr int kMmaM = 256;  // both CTAs
constexpr int kMmaN = 256;
constexpr int kABytes = kRowsPerCta * kBK * 2;  // 16 KB
constexpr int kBHalfBytes = 2 * kBoxBytes;      // 128 of the 256 columns
constexpr int kStageBytes = kABytes + kBHalfBytes;
constexpr int kAccCols = kMmaN;
constexpr int kThreads = 384;
constexpr int kEpiWarp0 = 4;
constexpr int kEpiWarps = 8;  // two per TMEM lane quarter, one per 128-column half

struct Ctl2 {
  uint64_t full[kStages];   // leader's: both CTAs' bytes of a stage
  uint64_t empty[kStages];  // each CTA: stage free again (leader's multicast commit)
  uint64_t tfull[2];        // each CTA: accumulator ready (leader's multicast commit)
  uint64_t tempty[2];       // leader's: both CTAs' epilogue warps done with the accumulator
  uint64_t drain;
  uint32_t tmem_base;
  uint32_t peer_tmem_base;
  int abort;
};

// dH epilogue: each epilogue warp turns its 32 rows x 32 columns of dH' around through a
// 4 KB shared block (row-per-lane out of TMEM, then 4 lanes per row for coalesced global
// traffic)
constexpr int kXposeBytes = 32 * 32 * 4;
constexpr size_t kSmemBytes = 1024 + (size_t)kStages * kStageBytes + (size_t)kEpiWarps * kXposeBytes + sizeof(Ctl2);




// The dH epilogue in the coalesced layout: lane l works on row 8 i + l / 4 (i = 0..3) of
// the warp's 32 and on the 8 columns 8 (l % 4) .. of the 32-column chunk; these are the
// rows' h, a = W1.x and b = W3.x there (one 16-byte vector each).
struct DhIn {
  uint4 a[4], b[4];  // W1.x and W3.x of the row (h = SiLU(a) b is recomputed from them)
};



__device__ __forceinline__ void raise_abort(Ctl2* ctl, uint32_t rank) {
  ctl->abort = 1;
  ptx::st_cluster_u32(ptx::mapa(ptx::smem_u32(&ctl->abort), rank ^ 1u), 1u);
}

template <int kKind>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_bwd_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                         const __grid_constant__ CUtensorMap tmB2, Shape s, Ws ws, int64_t timeout_ns) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* stages = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* xpose = stages + kStages * kStageBytes;  // 1024-byte aligned
  Ctl2* ctl = reinterpret_cast<Ctl2*>(xpose + kEpiWarps * kXposeBytes);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();
  const bool leader = rank == 0;
  const int cid = (int)ptx::cluster_id_x();
  const int ncl = (int)ptx::cluster_count_x();

  const int N = kKind == kBwdDH ? s.F : s.d;
  const int K = kKind == kBwdDH ? s.d : 2 * s.F;
  const int n_tiles = (N + kMmaN - 1) / kMmaN;
  const int kblocks = K / kBK;

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
    ptx::tma_prefetch_desc(&tmB);
    if (kKind == kBwdDX) ptx::tma_prefetch_desc(&tmB2);
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
  pdl_wait();  // the tile table and the A operand come from the previous kernels
  pdl_launch_dependents();
  int total = (int)ws.hdr[kHdrNumPairs] * n_tiles;
  if (ctl->peer_tmem_base != tmem) {  // a pair's accumulators must sit at the same TMEM address
    if (threadIdx.x == 0) record_error(ws, MOE_ERR_INTERNAL, 0x900u + kKind);
    total = 0;
  }
  volatile int* abort_flag = &ctl->abort;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------- TMA producer (both CTAs)
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int tile = cid; tile < total && ok; tile += ncl) {
        const TileInfo ti = decode_pair_tile(ws, n_tiles, tile, (int)rank);
        const int nb = ti.n_idx * kMmaN + (int)rank * (kMmaN / 2);  // this CTA's B columns
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!ptx::mbar_wait(ptx::smem_u32(&ctl->empty[stage]), phase ^ 1u, timeout_ns, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t full_local = ptx::smem_u32(&ctl->full[stage]);
          if (leader) ptx::mbar_arrive_expect_tx(full_local, 2 * kStageBytes);
          const uint32_t bar = ptx::mapa(full_local, 0);
          const uint32_t sa = ptx::smem_u32(stages + (size_t)stage * kStageBytes);
          ptx::tma_load_2d_pair(sa, &tmA, kb * kBK, ti.row0, bar);  // [128 rows, 64 K]
          const CUtensorMap* bm = &tmB;
          int brow;
          if (kKind == kBwdDH) {
            brow = ti.e * s.d + kb * kBK;
          } else {
            const int fk = s.F / kBK;
            if (kb >= fk) bm = &tmB2;
            brow = ti.e * s.F + (kb % fk) * kBK;
          }
#pragma unroll
          for (int j = 0; j < 2; ++j) ptx::tma_load_2d_pair(sa + kABytes + j * kBoxBytes, bm, nb + 64 * j, brow, bar);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        record_error(ws, MOE_ERR_TIMEOUT, 0x940u + kKind);
        raise_abort(ctl, rank);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ---------------------------------------------------------- MMA issuer (leader only)
      constexpr uint32_t idesc = ptx::idesc_bf16_f32(kMmaM, kMmaN) | (1u << 16);  // B MN-major
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int tile = cid; tile < total && ok; tile += ncl) {
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
          for (int ks = 0; ks < kBK / 16; ++ks)
            ptx::mma_bf16_pair(d_tmem, ptx::desc_kmajor_sw128(sa + ks * 32), desc_mnmajor_sw128(sb + ks * 2048),
                               idesc, (kb | ks) != 0 ? 1u : 0u);
          ptx::mma_commit_pair_multicast(ptx::smem_u32(&ctl->empty[stage]), 0x3);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        ptx::mma_commit_pair_multicast(ptx::smem_u32(&ctl->tfull[acc]), 0x3);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if (!ok) {
        record_error(ws, MOE_ERR_TIMEOUT, 0x950u + kKind);
        raise_abort(ctl, rank);
      }
    }
    __syncwarp();
  } else if (warp >= kEpiWarp0) {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int q = warp & 3;                          // TMEM lane quarter
    const int half = (warp - kEpiWarp0) >> 2;        // columns [128 half, 128 half + 128)
    const int c_beg = half * (kMmaN / 2);
    const int r = q * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int tile = cid; tile < total; tile += ncl) {
      const TileInfo ti = decode_pair_tile(ws, n_tiles, tile, (int)rank);
      const bool valid = r < ti.rows;
      const int n0 = ti.n_idx * kMmaN;
      const int64_t p = (int64_t)ti.row0 + r;
      // dH, coalesced layout: this lane's rows of the warp's 32 and their validity
      const int lrow0 = q * 32 + (lane >> 2);  // + 8 i
      const int cg = (lane & 3) * 8;           // column group within a 32-column chunk
      bool rv[4];
      int64_t prow[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        rv[i] = lrow0 + 8 * i < ti.rows;
        prow[i] = (int64_t)ti.row0 + lrow0 + 8 * i;
      }
      DhIn in;
      // the h / a / b vectors of row group i of chunk c (columns n0 + c + cg ..)
      auto fetch_row = [&](int i, int c) {
        const int64_t off = prow[i] * s.F + n0 + c + cg;
        in.a[i] = *reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(ws.a1) + off);
        in.b[i] = *reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(ws.a3) + off);
      };
      auto fetch = [&](int c) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if (rv[i]) fetch_row(i, c);
      };
      // the first chunk's operands are requested before the accumulator is ready
      if (kKind == kBwdDH && n0 + c_beg < s.F) fetch(c_beg);
      ok = ptx::mbar_wait(ptx::smem_u32(&ctl->tfull[acc]), acc_phase, timeout_ns, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      ptx::tc_fence_after();
      const uint32_t t_row = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * kAccCols);
      if (kKind == kBwdDH) {
        const int F = s.F;
        const uint32_t xb = ptx::smem_u32(xpose + (warp - kEpiWarp0) * kXposeBytes);
        int64_t trow[4];  // rows of dab_tail (or -1)
        {
          const int off_e = __ldg(&ws.offsets[ti.e]), cnt_e = __ldg(&ws.counts[ti.e]);
#pragma unroll
          for (int i = 0; i < 4; ++i) trow[i] = rv[i] ? tail_row(ti.e, prow[i], off_e, cnt_e) : -1;
        }
        float g[4], dgacc[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          g[i] = rv[i] ? ws.gate_perm[prow[i]] : 0.f;
          dgacc[i] = 0.f;
        }
#pragma unroll 1
        for (int c = c_beg; c < c_beg + kMmaN / 2; c += 32) {
          if (n0 + c >= F) break;  // uniform across the warp
          uint32_t v[32];
          ptx::tmem_ld_32cols(t_row + c, v);
          ptx::tmem_ld_wait();
          // row `lane` of the block: its 16-byte chunk j at j ^ (lane % 8)
          stage_row32(xb, lane, v);
          __syncwarp();
          // each row group's operands are replaced by the next chunk's as soon as they are used
          const bool has_next = n0 + c + 32 < F && c + 32 < c_beg + kMmaN / 2;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int br = 8 * i + (lane >> 2);  // row within the block
            float dh[8];
            ld_block_v4(xb + (uint32_t)br * 128u + (uint32_t)(((cg >> 2) ^ (br & 7)) * 16), dh[0], dh[1], dh[2], dh[3]);
            ld_block_v4(xb + (uint32_t)br * 128u + (uint32_t)((((cg >> 2) + 1) ^ (br & 7)) * 16), dh[4], dh[5], dh[6],
                         dh[7]);
            if (rv[i]) {
              float av[8], bv[8];
              unpack8(in.a[i], av);
              unpack8(in.b[i], bv);
              if (has_next) fetch_row(i, c + 32);
              uint4 oa, ob;
              uint32_t* wa = reinterpret_cast<uint32_t*>(&oa);
              uint32_t* wb = reinterpret_cast<uint32_t*>(&ob);
#pragma unroll
              for (int e2 = 0; e2 < 8; e2 += 2) {
                float da[2], db[2];
#pragma unroll
                for (int z = 0; z < 2; ++z) {
                  const float d = dh[e2 + z];
                  const float a = av[e2 + z];
                  const float sg = sigmoid_fast(a);
                  dgacc[i] += a * sg * bv[e2 + z] * d;  // h = SiLU(a) b, recomputed
                  da[z] = g[i] * d * bv[e2 + z] * sg * (1.0f + a * (1.0f - sg));
                  db[z] = g[i] * d * a * sg;
                }
                wa[e2 / 2] = pack2(da[0], da[1]);
                wb[e2 / 2] = pack2(db[0], db[1]);
              }
              __nv_bfloat16* dr = reinterpret_cast<__nv_bfloat16*>(ws.dab) + prow[i] * 2 * F + n0 + c + cg;
              *reinterpret_cast<uint4*>(dr) = oa;
              *reinterpret_cast<uint4*>(dr + F) = ob;
              if (trow[i] >= 0) {
                __nv_bfloat16* tr = reinterpret_cast<__nv_bfloat16*>(ws.dab_tail) + trow[i] * 2 * F + n0 + c + cg;
                *reinterpret_cast<uint4*>(tr) = oa;
                *reinterpret_cast<uint4*>(tr + F) = ob;
              }
            }
          }
          __syncwarp();  // the block is read before the next chunk overwrites it
        }
        // each row's partial sum of h . dH' over this warp's columns: the 4 lanes of the row
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float t = dgacc[i];
          t += __shfl_xor_sync(0xffffffffu, t, 1);
          t += __shfl_xor_sync(0xffffffffu, t, 2);
          if (rv[i] && (lane & 3) == 0) ws.dgp[prow[i] * (int64_t)(2 * n_tiles) + 2 * ti.n_idx + half] = t;
        }
      } else {
        int64_t slot = valid ? ws.perm_slot[p] : -1;
        if (slot >= s.N) slot = -1;
        __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(ws.dxslot) + slot * s.d + n0;
#pragma unroll 1
        for (int c = c_beg; c < c_beg + kMmaN / 2; c += 32) {
          if (n0 + c >= s.d) break;
          uint32_t v[32];
          ptx::tmem_ld_32cols(t_row + c, v);
          ptx::tmem_ld_wait();
          if (slot >= 0) {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              uint4 o;
              uint32_t* w = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
              for (int i = 0; i < 4; ++i)
                w[i] = pack2(__uint_as_float(v[8 * u + 2 * i]), __uint_as_float(v[8 * u + 2 * i + 1]));
              *reinterpret_cast<uint4*>(out + c + 8 * u) = o;
            }
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
      record_error(ws, MOE_ERR_TIMEOUT, 0x970u + kKind);
      raise_abort(ctl, rank);
    }
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
cudaError_t launch_pair(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& b2, const Shape& s, const Ws& ws,
                        int num_sms, int64_t timeout_ns, bool pdl, cudaStream_t st) {
  auto kern = gemm_bwd_pair_kernel<kKind>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  // as many pairs as can be resident at once (persistent loop over pair tiles)
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
  return launch_kernel(kern, dim3((unsigned)grid), dim3(kThreads), kSmemBytes, st, pdl, 2, a, b, b2, s, ws, timeout_ns);
}

}  // namespace

cudaError_t launch_gemm_bwd_pair(int kind, const Shape& s, const Ws& ws, const Weights& w, int num_sms,
                                 int64_t timeout_ns, bool pdl, cudaStream_t st) {
  CUtensorMap ma, mb, mb2;
  cudaError_t e;
  const uint64_t N = (uint64_t)s.N, d = (uint64_t)s.d, F = (uint64_t)s.F, E = (uint64_t)s.E;
  if (kind == kBwdDH) {
    if ((e = make_tmap_bf16(&ma, ws.dyp, N, d, kRowsPerCta)) != cudaSuccess) return e;
    if ((e = make_tmap_bf16(&mb, w.w2, E * d, F, 64)) != cudaSuccess) return e;
    return launch_pair<kBwdDH>(ma, mb, mb, s, ws, num_sms, timeout_ns, pdl, st);
  }
  if (kind == kBwdDX) {
    if ((e = make_tmap_bf16(&ma, ws.dab, N, 2 * F, kRowsPerCta)) != cudaSuccess) return e;
    if ((e = make_tmap_bf16(&mb, w.w1, E * F, d, 64)) != cudaSuccess) return e;
    if ((e = make_tmap_bf16(&mb2, w.w3, E * F, d, 64)) != cudaSuccess) return e;
    return launch_pair<kBwdDX>(ma, mb, mb2, s, ws, num_sms, timeout_ns, pdl, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace moe
