// gemm_tc2.cu -- the grouped expert GEMMs on CTA pairs (2-SM tcgen05.mma, cta_group::2).
//
// Same operation as gemm_tc.cu (after "Distributed Training Part 4 ... MoE + Expert
// Parallelism", jesamkim ai-tech-blog, §3 Structure / output formula, §4 Combine):
//   mode 1:  H[p, n]           = SiLU(Xp[p] . W1_e[n]) * (Xp[p] . W3_e[n])
//   mode 2:  Yp[p, n]          = gate(p) * (H[p] . W2_e[n])   (row p in expert order, like Xp
//                                and H; the combine gathers token t's rows through slot_pos)
//
// A cluster of two CTAs on two SMs computes a 256 x 256 tile with one MMA stream issued by
// the first CTA (the leader): each CTA loads only its own 128 rows of A and its half of the
// 256 B rows (mode 1: the leader the W1 tile, the peer the W3 tile; mode 2: one half each),
// so an SM pulls 32 KB per 64-deep K step instead of 48 KB and the ring holds 6 stages.
// Both CTAs' loads signal the leader's "full" barrier; the leader's commits free the stage in
// both CTAs (multicast arrive) and hand each CTA its 128 accumulator rows in its own TMEM.
// The epilogue runs per CTA; its warps release the accumulator to the leader with a
// cluster-scope arrive.  Both outputs (H, Yp) are in the expert-contiguous row order of the A
// operand, so each warp's 32 rows x 64 columns form one tile of the output: the warp stages it
// in shared memory (128-byte swizzle, double-buffered) and one lane hands it to the TMA engine
// as a tiled store.  Only a warp block that crosses the end of the expert's rows stores its
// valid rows directly (a tiled store would overwrite the next expert's first rows).  In
// training mode W1.x and W3.x are also kept, stored directly.
//
// Waits are bounded (MOE_ERR_TIMEOUT, no trap); an abort raises the flag in both CTAs; the
// pair meets at cluster barriers before TMEM is released.
#include <cuda.h>
#include <cuda_bf16.h>

#include "gemm_tc.h"
#include "tc_ptx.cuh"

namespace moe {
namespace {

constexpr int kBK = 64;
constexpr int kStages = 6;
constexpr int kRowsPerCta = 128;
constexpr int kMmaM = 256;  // both CTAs
constexpr int kMmaN = 256;
constexpr int kMmaK = 16;
constexpr int kABytes = kRowsPerCta * kBK * 2;    // 16 KB
constexpr int kBHalfBytes = (kMmaN / 2) * kBK * 2;  // 16 KB
constexpr int kStageBytes = kABytes + kBHalfBytes;
constexpr int kAccCols = kMmaN;
constexpr int kThreads = 256;
constexpr int kEpiWarp0 = 4;
constexpr int kEpiWarps = 4;

struct Ctl2 {
  uint64_t full[kStages];   // leader's: both CTAs' bytes of a stage
  uint64_t empty[kStages];  // each CTA: stage free again (leader's multicast commit)
  uint64_t tfull[2];        // each CTA: accumulator ready (leader's multicast commit)
  uint64_t tempty[2];       // leader's: both CTAs' epilogue warps done with the accumulator
  uint64_t drain;
  uint32_t tmem_base;
  uint32_t peer_tmem_base;  // the peer's allocation, written by the peer
  int abort;
};

// the epilogue's store staging: per warp two blocks of 32 rows x 64 bf16 columns (128-byte
// rows, 16-byte chunk j of row r at j ^ (r % 8): the TMA 128-byte swizzle), 1024-byte aligned
constexpr int kStgBlockBytes = 32 * 128;
constexpr int kStgBytes = kEpiWarps * 2 * kStgBlockBytes;

constexpr size_t kSmemBytes = 1024 + (size_t)kStages * kStageBytes + kStgBytes + sizeof(Ctl2);
static_assert(kSmemBytes <= 232448, "shared memory per CTA");

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float silu(float a) { return silu_fast(a); }

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// 2-D tiled TMA store of a staged block (x = column, y = row), as a bulk group of its own
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, int32_t x, int32_t y, uint32_t src) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];\n\t"
      "cp.async.bulk.commit_group;" ::"l"(reinterpret_cast<uint64_t>(map)),
      "r"(x), "r"(y), "r"(src)
      : "memory");
}
// the same with an L2 eviction-priority hint
__device__ __forceinline__ void tma_store_2d_hint(const CUtensorMap* map, int32_t x, int32_t y, uint32_t src,
                                                  uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group.L2::cache_hint [%0, {%1, %2}], [%3], %4;\n\t"
      "cp.async.bulk.commit_group;" ::"l"(reinterpret_cast<uint64_t>(map)),
      "r"(x), "r"(y), "r"(src), "l"(policy)
      : "memory");
}
// at most one of this thread's bulk groups still reading its shared-memory source
__device__ __forceinline__ void bulk_wait_read_le1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
// all of this thread's bulk groups complete (their global writes performed)
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Store 64 bf16 columns of this warp's 32 rows (pk: this lane's row).  When all 32 rows
// belong to the tile's expert (vw >= 32) the warp stages them in its next staging block and
// lane 0 issues one tiled store of the block at (x, y); otherwise each lane whose row is valid
// (lane < vw) writes its 128 bytes to dst directly, so that no row of the next expert is
// touched.  vw is the same for the whole warp.
__device__ __forceinline__ void store_rows64(const uint32_t (&pk)[32], int vw, int lane, uint32_t stg,
                                             int& stg_buf, const CUtensorMap* map, int x, int y, void* dst,
                                             uint64_t policy = 0) {
  if (vw >= 32) {
    const uint32_t blk = stg + (uint32_t)(stg_buf * kStgBlockBytes);
    if (lane == 0) bulk_wait_read_le1();  // the store issued from this block two blocks ago has read it
    __syncwarp();
#pragma unroll
    for (int j = 0; j < 8; ++j)
      st_shared_v4(blk + (uint32_t)(lane * 128 + ((j ^ (lane & 7)) * 16)), pk[4 * j], pk[4 * j + 1], pk[4 * j + 2],
                   pk[4 * j + 3]);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // visible to the TMA engine
    __syncwarp();
    if (lane == 0) {
      if (policy != 0)
        tma_store_2d_hint(map, x, y, blk, policy);
      else
        tma_store_2d(map, x, y, blk);
    }
    stg_buf ^= 1;
  } else if (lane < vw) {
    uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int v = 0; v < 8; ++v) d[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
  }
}

// L2 eviction priority of the SwiGLU GEMM's operand loads and H stores (0: the default,
// 1: evict_last, 2: evict_first).  A scheduling group's A rows are read once per n-tile, so
// they are kept (evict_last); H is not read again by this kernel (evict_first); each weight
// n-tile is read by the group's pairs one after another and keeps the default priority (as
// evict_first the weights were read from DRAM about three times over).
constexpr int kHintA = 1;
constexpr int kHintB = 0;
constexpr int kHintY = 2;

__device__ __forceinline__ uint64_t l2_policy(int hint) {
  uint64_t p = 0;
  if (hint == 1) asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  if (hint == 2) asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// tma_load_2d_pair with an L2 eviction-priority hint
__device__ __forceinline__ void tma_load_2d_pair_hint(uint32_t dst, const CUtensorMap* map, int32_t c0, int32_t c1,
                                                      uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes.cta_group::2.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void raise_abort(Ctl2* ctl, uint32_t rank) {
  ctl->abort = 1;
  ptx::st_cluster_u32(ptx::mapa(ptx::smem_u32(&ctl->abort), rank ^ 1u), 1u);
}

template <int kMode, int kAccBufs>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc2_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmB3, const __grid_constant__ CUtensorMap tmY, Shape s,
                    Ws ws, int64_t timeout_ns, int stall) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* stages = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stg_base = stages + kStages * kStageBytes;  // the epilogue's store staging
  Ctl2* ctl = reinterpret_cast<Ctl2*>(stg_base + kStgBytes);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();
  const bool leader = rank == 0;
  const int cid = (int)ptx::cluster_id_x();
  const int ncl = (int)ptx::cluster_count_x();

  const int ncols = kMode == 1 ? s.F : s.d;
  const int K = kMode == 1 ? s.d : s.F;
  const int bn = kMode == 1 ? kMmaN / 2 : kMmaN;  // output columns per tile
  const int n_tiles = (ncols + bn - 1) / bn;
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
    if (kMode == 1) ptx::tma_prefetch_desc(&tmB3);
    ptx::tma_prefetch_desc(&tmY);
  }
  ptx::cluster_sync();  // both CTAs' barriers exist before any cross-CTA arrive or load
  if (warp == 2) {
    ptx::tmem_alloc_pair(ptx::smem_u32(&ctl->tmem_base), kAccBufs * kAccCols);
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
    if (threadIdx.x == 0) record_error(ws, MOE_ERR_INTERNAL, 0x700u + kMode);
    total = 0;
  }
  volatile int* abort_flag = &ctl->abort;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------- TMA producer (both CTAs)
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true, first = true;
      const CUtensorMap* bmap = (kMode == 1 && rank == 1) ? &tmB3 : &tmB;
      const uint64_t pol_a = l2_policy(kMode == 1 ? kHintA : 0), pol_b = l2_policy(kMode == 1 ? kHintB : 0);
      for (int tile = cid; tile < total && ok; tile += ncl) {
        const TileInfo ti = decode_pair_tile(ws, n_tiles, tile, (int)rank);
        const int brow = kMode == 1 ? ti.e * s.F + ti.n_idx * bn : ti.e * s.d + ti.n_idx * bn + (int)rank * (kMmaN / 2);
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!ptx::mbar_wait(ptx::smem_u32(&ctl->empty[stage]), phase ^ 1u, timeout_ns, abort_flag)) {
            ok = false;
            break;
          }
          if (!(stall && first && leader)) {  // the stall hook withholds one stage of the leader
            const uint32_t full_local = ptx::smem_u32(&ctl->full[stage]);
            if (leader) ptx::mbar_arrive_expect_tx(full_local, 2 * kStageBytes);
            const uint32_t bar = ptx::mapa(full_local, 0);
            const uint32_t sa = ptx::smem_u32(stages + (size_t)stage * kStageBytes);
            if (kMode == 1 && kHintA != 0)
              tma_load_2d_pair_hint(sa, &tmA, kb * kBK, ti.row0, bar, pol_a);
            else
              ptx::tma_load_2d_pair(sa, &tmA, kb * kBK, ti.row0, bar);
            if (kMode == 1 && kHintB != 0)
              tma_load_2d_pair_hint(sa + kABytes, bmap, kb * kBK, brow, bar, pol_b);
            else
              ptx::tma_load_2d_pair(sa + kABytes, bmap, kb * kBK, brow, bar);
          }
          first = false;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        record_error(ws, MOE_ERR_TIMEOUT, 0x540u + kMode);
        raise_abort(ctl, rank);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ---------------------------------------------------------- MMA issuer (leader only)
      constexpr uint32_t idesc = ptx::idesc_bf16_f32(kMmaM, kMmaN);
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
          for (int ks = 0; ks < kBK / kMmaK; ++ks)
            ptx::mma_bf16_pair(d_tmem, ptx::desc_kmajor_sw128(sa + ks * kMmaK * 2),
                               ptx::desc_kmajor_sw128(sb + ks * kMmaK * 2), idesc, (kb | ks) != 0 ? 1u : 0u);
          ptx::mma_commit_pair_multicast(ptx::smem_u32(&ctl->empty[stage]), 0x3);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        ptx::mma_commit_pair_multicast(ptx::smem_u32(&ctl->tfull[acc]), 0x3);
        if (++acc == kAccBufs) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if (!ok) {
        record_error(ws, MOE_ERR_TIMEOUT, 0x550u + kMode);
        raise_abort(ctl, rank);
      }
    }
    __syncwarp();
  } else if (warp >= kEpiWarp0) {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int q = warp & 3;
    const int r = q * 32 + lane;
    const uint32_t stg = ptx::smem_u32(stg_base) + (uint32_t)(q * 2 * kStgBlockBytes);
    int stg_buf = 0;  // the staging block of this warp's next tiled store
    const uint64_t pol_y = l2_policy(kMode == 1 ? kHintY : 0);
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int tile = cid; tile < total; tile += ncl) {
      const TileInfo ti = decode_pair_tile(ws, n_tiles, tile, (int)rank);
      ok = ptx::mbar_wait(ptx::smem_u32(&ctl->tfull[acc]), acc_phase, timeout_ns, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      ptx::tc_fence_after();
      const uint32_t t_row = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * kAccCols);
      const bool valid = r < ti.rows;
      const int64_t p = (int64_t)ti.row0 + r;
      const int n0 = ti.n_idx * bn;
      // rows of this warp's 32-row block that belong to the tile's expert: all 32 -> one tiled
      // store per 64 columns; fewer -> each valid lane stores its own row piece
      const int vw = ti.rows - q * 32;
      if (kMode == 1) {
        __nv_bfloat16* hrow = reinterpret_cast<__nv_bfloat16*>(ws.h) + p * s.F + n0;
#pragma unroll 1
        for (int c = 0; c < kMmaN / 2; c += 64) {
          if (vw <= 0 || n0 + c >= s.F) break;  // warp-uniform
          uint32_t pk[32];  // the row's 64 H values
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            uint32_t a[32], g[32];
            ptx::tmem_ld_32cols(t_row + c + 32 * hh, a);
            ptx::tmem_ld_32cols(t_row + kMmaN / 2 + c + 32 * hh, g);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i)
              pk[16 * hh + i] = pack_bf16x2(silu(__uint_as_float(a[2 * i])) * __uint_as_float(g[2 * i]),
                                            silu(__uint_as_float(a[2 * i + 1])) * __uint_as_float(g[2 * i + 1]));
            if (s.training && valid) {  // keep W1.x and W3.x of the row for the backward
              const int64_t o = p * s.F + n0 + c + 32 * hh;
              uint4* da1 = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(ws.a1) + o);
              uint4* da3 = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(ws.a3) + o);
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                uint32_t w1[4], w3[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                  const int i = v * 8 + u * 2;
                  w1[u] = pack_bf16x2(__uint_as_float(a[i]), __uint_as_float(a[i + 1]));
                  w3[u] = pack_bf16x2(__uint_as_float(g[i]), __uint_as_float(g[i + 1]));
                }
                da1[v] = make_uint4(w1[0], w1[1], w1[2], w1[3]);
                da3[v] = make_uint4(w3[0], w3[1], w3[2], w3[3]);
              }
            }
          }
          store_rows64(pk, vw, lane, stg, stg_buf, &tmY, n0 + c, ti.row0 + q * 32, hrow + c, pol_y);
        }
      } else {
        const float gate = valid ? ws.gate_perm[p] : 0.f;
        __nv_bfloat16* yrow = reinterpret_cast<__nv_bfloat16*>(ws.yp) + p * s.d + n0;
#pragma unroll 1
        for (int c = 0; c < kMmaN; c += 64) {
          if (vw <= 0 || n0 + c >= s.d) break;  // warp-uniform
          uint32_t a[32], b[32];
          ptx::tmem_ld_32cols(t_row + c, a);
          ptx::tmem_ld_32cols(t_row + c + 32, b);
          ptx::tmem_ld_wait();
          uint32_t pk[32];  // the row's 64 output values
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            pk[i] = pack_bf16x2(gate * __uint_as_float(a[2 * i]), gate * __uint_as_float(a[2 * i + 1]));
            pk[16 + i] = pack_bf16x2(gate * __uint_as_float(b[2 * i]), gate * __uint_as_float(b[2 * i + 1]));
          }
          store_rows64(pk, vw, lane, stg, stg_buf, &tmY, n0 + c, ti.row0 + q * 32, yrow + c);
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_cluster(ptx::mapa(ptx::smem_u32(&ctl->tempty[acc]), 0));
      if (++acc == kAccBufs) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    bulk_wait_all();  // the tiled stores this lane issued have been written
    if (!ok && lane == 0) {
      record_error(ws, MOE_ERR_TIMEOUT, 0x570u + kMode);
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
    ptx::tmem_dealloc_pair(tmem, kAccBufs * kAccCols);
  }
}

template <int kMode, int kAccBufs>
cudaError_t launch_pair(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& b3, const CUtensorMap& y,
                        const Shape& s, const Ws& ws,
                        int num_sms, int64_t timeout_ns, bool stall, bool pdl, cudaStream_t st) {
  auto kern = gemm_tc2_kernel<kMode, kAccBufs>;
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
  return launch_kernel(kern, dim3((unsigned)grid), dim3(kThreads), kSmemBytes, st, pdl, 2, a, b, b3, y, s, ws, timeout_ns,
                       stall ? 1 : 0);
}

}  // namespace

cudaError_t launch_gemm_tc_pair(int mode, const Shape& s, const Ws& ws, const Weights& w, int num_sms,
                                int64_t timeout_ns, bool test_stall, bool pdl, cudaStream_t st) {
  CUtensorMap mA, mB, mB3, mY;
  cudaError_t e;
  if (mode == 1) {
    if ((e = make_tmap_bf16(&mA, ws.xp, (uint64_t)s.N, (uint64_t)s.d, kRowsPerCta)) != cudaSuccess) return e;
    if ((e = make_tmap_bf16(&mB, w.w1, (uint64_t)s.E * s.F, (uint64_t)s.d, kMmaN / 2)) != cudaSuccess) return e;
    if ((e = make_tmap_bf16(&mB3, w.w3, (uint64_t)s.E * s.F, (uint64_t)s.d, kMmaN / 2)) != cudaSuccess) return e;
    if ((e = make_tmap_bf16(&mY, ws.h, (uint64_t)s.N, (uint64_t)s.F, 32)) != cudaSuccess) return e;
    return launch_pair<1, kPairAccBufs>(mA, mB, mB3, mY, s, ws, num_sms, timeout_ns, test_stall, pdl, st);
  }
  if ((e = make_tmap_bf16(&mA, ws.h, (uint64_t)s.N, (uint64_t)s.F, kRowsPerCta)) != cudaSuccess) return e;
  if ((e = make_tmap_bf16(&mB, w.w2, (uint64_t)s.E * s.d, (uint64_t)s.F, kMmaN / 2)) != cudaSuccess) return e;
  if ((e = make_tmap_bf16(&mY, ws.yp, (uint64_t)s.N, (uint64_t)s.d, 32)) != cudaSuccess) return e;
  return launch_pair<2, kPairAccBufs>(mA, mB, mB, mY, s, ws, num_sms, timeout_ns, false, pdl, st);
}

}  // namespace moe
