// gemm_bwd.cu -- the grouped GEMMs of the backward pass on the tensor cores (tcgen05, one CTA
// per 128 x 256 tile, TMA-fed, accumulators in TMEM).
//
// Backward of "Distributed Training Part 4 ... MoE + Expert Parallelism" (jesamkim
// ai-tech-blog) §3 (SwiGLU experts, gate-weighted sum) and §4 (combine / dispatch reversed):
// for each routed row p of expert e (token t = perm_src[p], gate g = gate_perm[p]):
//   kDH   dH'[p, f] = sum_c dy[t, c] W2_e[c, f]               (A = dYp  K-major, B = W2 MN-major)
//         epilogue:  dg partial = sum_f h[p,f] dH'[p,f];  da = g dH' b silu'(a),  db = g dH' silu(a),
//         with h = silu(a) b recomputed from the kept a, b (not read back)
//   kDX   dXslot[slot(p), c] = sum_f da[p,f] W1_e[f,c] + db[p,f] W3_e[f,c]
//                                                          (A = [da|db] K-major, B = W1|W3 MN-major)
//   kDW13 [dW1_e; dW3_e][m, c] = sum_{p in e} [da|db][p, m] Xp[p, c]   (both operands MN-major)
//   kDW2  dW2_e[c, f]          = sum_{p in e} g dy[t, c] h[p, f]       (both operands MN-major)
// kDH and kDX are grouped over M (the expert's rows, the forward's tile table); kDW13 and
// kDW2 over K (the expert's rows are the reduction).  An expert's last, partial 64-row K
// block of A comes from dab_tail / dop_tail (the same rows, zero past the expert's end), so
// no block is masked; B (Xp, h) runs on into the next expert's rows, which the zeros cancel.
//
// MN-major operand tiles: TMA boxes of 64 (MN, contiguous) x 64 (K rows) with 128-byte
// swizzling, side by side 8 KB apart; the descriptor's leading offset is that 8 KB step
// between 64-wide MN blocks, the stride offset 1 KB between 8-row K groups, and one K=16
// MMA step is 2 KB.
#include <cuda.h>
#include <cuda_bf16.h>

#include "gemm_tc.h"
#include "bwd_common.cuh"
#include "tc_ptx.cuh"
#include "tmap.h"

namespace moe {
namespace {

using namespace bwd;

constexpr int kBK = 64;
constexpr int kStages = 4;
constexpr int kTM = 128;  // tile rows (M)
constexpr int kTN = 256;  // tile columns (N)
constexpr int kABytes = kTM * kBK * 2;
constexpr int kBBytes = kTN * kBK * 2;
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kThreads = 384;
constexpr int kEpiWarp0 = 4;
constexpr int kEpiThreads = 256;  // 8 warps: two per TMEM lane quarter, one per 128-column half

struct Ctl {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};
// weight-gradient epilogue: each epilogue warp stages a 32 x 32 fp32 block (128-byte rows,
// swizzled) and hands it to the TMA to store
constexpr int kOutBlockBytes = 32 * 128;
constexpr int kEpiWarps = kEpiThreads / 32;
constexpr size_t kSmemBytes =
    1024 + (size_t)kStages * kStageBytes + (size_t)kEpiWarps * kOutBlockBytes + sizeof(Ctl);


__host__ __device__ constexpr bool a_mn(int kind) { return kind == kBwdDW13 || kind == kBwdDW2; }
__host__ __device__ constexpr bool k_grouped(int kind) { return kind == kBwdDW13 || kind == kBwdDW2; }




__device__ __forceinline__ void tmem_ld_16cols(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr)
      : "memory");
}

// The dH epilogue's operands of one 16-column chunk of a row: h, and the two
// pre-activations a = W1.x, b = W3.x (two 16-byte vectors each).
struct DhChunk {
  uint4 a[2], b[2];  // W1.x and W3.x of the row (h = SiLU(a) b is recomputed from them)
};

__device__ __forceinline__ void dh_fetch(DhChunk& d, const __nv_bfloat16* arow, const __nv_bfloat16* brow, int c) {
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    d.a[i] = reinterpret_cast<const uint4*>(arow + c)[i];
    d.b[i] = reinterpret_cast<const uint4*>(brow + c)[i];
  }
}

// Work item of one tile.
struct BTile {
  int e;
  int row0, rows;   // M-grouped: routed rows; K-grouped: output rows m0.. (rows = valid)
  int n_idx;
  int k_row0;       // K-grouped: first routed row of the expert (the K range)
  int kblocks;
  int a_tail;       // K-grouped: row of the expert's tail block in dab_tail / dop_tail, or -1
};

struct BwdArgs {
  Shape s;
  Ws ws;
  float* dw_a;      // kDW13: dW1 [E,F,d]; kDW2: dW2 [E,d,F]
  float* dw_b;      // kDW13: dW3
};

template <int kKind>
__device__ __forceinline__ void kind_dims(const Shape& s, int& M, int& N, int& K) {
  if (kKind == kBwdDH) { M = 0; N = s.F; K = s.d; }
  if (kKind == kBwdDX) { M = 0; N = s.d; K = 2 * s.F; }
  if (kKind == kBwdDW13) { M = 2 * s.F; N = s.d; K = 0; }
  if (kKind == kBwdDW2) { M = s.d; N = s.F; K = 0; }
}

template <int kKind>
__device__ __forceinline__ BTile decode(const BwdArgs& a, int tile, int n_tiles, int m_tiles) {
  BTile b{};
  if (!k_grouped(kKind)) {
    const TileInfo ti = decode_tile(a.ws, n_tiles, tile);
    int M, N, K;
    kind_dims<kKind>(a.s, M, N, K);
    b.e = ti.e;
    b.row0 = ti.row0;
    b.rows = ti.rows;
    b.n_idx = ti.n_idx;
    b.kblocks = K / kBK;
    b.k_row0 = 0;
    b.a_tail = -1;
  } else {
    int M, N, K;
    kind_dims<kKind>(a.s, M, N, K);
    const int per_e = m_tiles * n_tiles;
    b.e = tile / per_e;
    const int local = tile % per_e;
    b.n_idx = local / m_tiles;
    const int m_idx = local % m_tiles;
    b.row0 = m_idx * kTM;
    b.rows = M - b.row0 < kTM ? M - b.row0 : kTM;
    const int cnt = __ldg(&a.ws.counts[b.e]);
    b.k_row0 = __ldg(&a.ws.offsets[b.e]);
    b.kblocks = (cnt + kBK - 1) / kBK;
    b.a_tail = cnt % kBK != 0 ? b.e * kBK : -1;
  }
  return b;
}

template <int kKind>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_bwd_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmB2, const __grid_constant__ CUtensorMap tmO1,
                    const __grid_constant__ CUtensorMap tmO2, BwdArgs args, int64_t timeout_ns) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* stages = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* out_blocks = stages + kStages * kStageBytes;  // 1024-byte aligned
  Ctl* ctl = reinterpret_cast<Ctl*>(out_blocks + kEpiWarps * kOutBlockBytes);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const Shape& s = args.s;
  const Ws& ws = args.ws;
  int M, N, K;
  kind_dims<kKind>(s, M, N, K);
  const int n_tiles = (N + kTN - 1) / kTN;
  const int m_tiles = (M + kTM - 1) / kTM;

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
  if (warp == 2) {
    ptx::tmem_alloc(ptx::smem_u32(&ctl->tmem_base), 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  volatile int* abort_flag = &ctl->abort;
  pdl_wait();
  pdl_launch_dependents();
  const int total = k_grouped(kKind) ? s.E * m_tiles * n_tiles : (int)ws.hdr[kHdrNumMTiles] * n_tiles;
  uint32_t issued = 0, issued_phase = 0;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ TMA producer
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        const BTile bt = decode<kKind>(args, tile, n_tiles, m_tiles);
        const int n0 = bt.n_idx * kTN;
        for (int kb = 0; kb < bt.kblocks; ++kb) {
          if (!ptx::mbar_wait(ptx::smem_u32(&ctl->empty[stage]), phase ^ 1u, timeout_ns, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t bar = ptx::smem_u32(&ctl->full[stage]);
          const uint32_t sa = ptx::smem_u32(stages + (size_t)stage * kStageBytes);
          const uint32_t sb = sa + kABytes;
          ptx::mbar_arrive_expect_tx(bar, kStageBytes);
          if (!a_mn(kKind)) {
            ptx::tma_load_2d(sa, &tmA, kb * kBK, bt.row0, bar);  // [rows, K]: one 128-row box
          } else {
            // the expert's last, partial block from the zero-padded tail copy (tmB2 slot)
            const bool tail = kb == bt.kblocks - 1 && bt.a_tail >= 0;
            const CUtensorMap* am = tail ? &tmB2 : &tmA;
            const int krow = tail ? bt.a_tail : bt.k_row0 + kb * kBK;
            ptx::tma_load_2d(sa, am, bt.row0, krow, bar);
            ptx::tma_load_2d(sa + kBoxBytes, am, bt.row0 + 64, krow, bar);
          }
          // B: four MN-major boxes of 64 columns
          const CUtensorMap* bm = &tmB;
          int brow;
          if (kKind == kBwdDH) {
            brow = bt.e * s.d + kb * kBK;
          } else if (kKind == kBwdDX) {
            const int fk = s.F / kBK;
            if (kb >= fk) bm = &tmB2;
            brow = bt.e * s.F + (kb % fk) * kBK;
          } else {
            brow = bt.k_row0 + kb * kBK;
          }
#pragma unroll
          for (int j = 0; j < 4; ++j) ptx::tma_load_2d(sb + j * kBoxBytes, bm, n0 + 64 * j, brow, bar);
          issued |= 1u << stage;
          issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        *abort_flag = 1;
        record_error(ws, MOE_ERR_TIMEOUT, 0x800u + kKind);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // -------------------------------------------------------------- MMA issuer
    const uint32_t idesc = ptx::idesc_bf16_f32(kTM, kTN) | (a_mn(kKind) ? (1u << 15) : 0u) | (1u << 16);
    int stage = 0, acc = 0;
    uint32_t phase = 0, acc_phase = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
      const BTile bt = decode<kKind>(args, tile, n_tiles, m_tiles);
      ok = ptx::mbar_wait(ptx::smem_u32(&ctl->tempty[acc]), acc_phase ^ 1u, timeout_ns, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      ptx::tc_fence_after();
      const uint32_t d_tmem = tmem + (uint32_t)(acc * kTN);
      for (int kb = 0; kb < bt.kblocks; ++kb) {
        ok = ptx::mbar_wait(ptx::smem_u32(&ctl->full[stage]), phase, timeout_ns, abort_flag);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        uint8_t* st_base = stages + (size_t)stage * kStageBytes;
        ptx::tc_fence_after();
        if (lane == 0) {
          const uint32_t sa = ptx::smem_u32(st_base);
          const uint32_t sb = sa + kABytes;
#pragma unroll
          for (int ks = 0; ks < kBK / 16; ++ks) {
            const uint64_t adesc =
                a_mn(kKind) ? desc_mnmajor_sw128(sa + ks * 2048) : ptx::desc_kmajor_sw128(sa + ks * 32);
            ptx::mma_bf16(d_tmem, adesc, desc_mnmajor_sw128(sb + ks * 2048), idesc, (kb | ks) != 0 ? 1u : 0u);
          }
          ptx::mma_commit(ptx::smem_u32(&ctl->empty[stage]));
        }
        __syncwarp();
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      if (lane == 0) ptx::mma_commit(ptx::smem_u32(&ctl->tfull[acc]));
      __syncwarp();
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (!ok && lane == 0) {
      *abort_flag = 1;
      record_error(ws, MOE_ERR_TIMEOUT, 0x810u + kKind);
    }
  } else if (warp >= kEpiWarp0) {
    // -------------------------------------------------------------- epilogue
    const int q = warp & 3;                          // TMEM lane quarter
    const int half = (warp - kEpiWarp0) >> 2;        // columns [128 half, 128 half + 128)
    const int c_beg = half * (kTN / 2), c_end = c_beg + kTN / 2;
    const int r = q * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      const BTile bt = decode<kKind>(args, tile, n_tiles, m_tiles);
      const bool valid = r < bt.rows;
      const int n0 = bt.n_idx * kTN;
      // dH: the row's h / a / b are requested a chunk ahead of their use, the first chunk
      // before the accumulator is ready, so that their latency hides behind the MMA
      const int64_t p_dh = (int64_t)bt.row0 + r;
      const __nv_bfloat16* arow = reinterpret_cast<const __nv_bfloat16*>(ws.a1) + p_dh * s.F + n0;
      const __nv_bfloat16* brow = reinterpret_cast<const __nv_bfloat16*>(ws.a3) + p_dh * s.F + n0;
      DhChunk pre[2];
      if (kKind == kBwdDH && valid && n0 + c_beg < s.F) dh_fetch(pre[0], arow, brow, c_beg);
      ok = ptx::mbar_wait(ptx::smem_u32(&ctl->tfull[acc]), acc_phase, timeout_ns, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      ptx::tc_fence_after();
      const uint32_t t_row = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * kTN);
      if (kKind == kBwdDH) {
        const int64_t p = p_dh;
        const int F = s.F;
        const float g = valid ? ws.gate_perm[p] : 0.f;
        __nv_bfloat16* darow = reinterpret_cast<__nv_bfloat16*>(ws.dab) + p * 2 * F + n0;
        const int64_t trow = valid ? tail_row(bt.e, p, __ldg(&ws.offsets[bt.e]), __ldg(&ws.counts[bt.e])) : -1;
        __nv_bfloat16* dtrow = reinterpret_cast<__nv_bfloat16*>(ws.dab_tail) + (trow >= 0 ? trow : 0) * 2 * F + n0;
        float dg = 0.f;
#pragma unroll
        for (int i = 0; i < (kTN / 2) / 16; ++i) {
          const int c = c_beg + 16 * i;
          if (i + 1 < (kTN / 2) / 16 && valid && n0 + c + 16 < F) dh_fetch(pre[(i + 1) & 1], arow, brow, c + 16);
          if (n0 + c < F) {  // uniform across the warp
            uint32_t v[16];
            tmem_ld_16cols(t_row + c, v);
            ptx::tmem_ld_wait();
            if (valid) {
              const DhChunk& d = pre[i & 1];
#pragma unroll
              for (int u = 0; u < 2; ++u) {
                float av[8], bv[8];
                unpack8(d.a[u], av);
                unpack8(d.b[u], bv);
                uint4 oa, ob;
                uint32_t* wa = reinterpret_cast<uint32_t*>(&oa);
                uint32_t* wb = reinterpret_cast<uint32_t*>(&ob);
#pragma unroll
                for (int e2 = 0; e2 < 8; e2 += 2) {
                  float da[2], db[2];
#pragma unroll
                  for (int z = 0; z < 2; ++z) {
                    const float dh = __uint_as_float(v[8 * u + e2 + z]);
                    const float a = av[e2 + z];
                    const float sg = sigmoid_fast(a);
                    dg += a * sg * bv[e2 + z] * dh;  // h = SiLU(a) b, recomputed
                    da[z] = g * dh * bv[e2 + z] * sg * (1.0f + a * (1.0f - sg));
                    db[z] = g * dh * a * sg;
                  }
                  wa[e2 / 2] = pack2(da[0], da[1]);
                  wb[e2 / 2] = pack2(db[0], db[1]);
                }
                *reinterpret_cast<uint4*>(darow + c + 8 * u) = oa;
                *reinterpret_cast<uint4*>(darow + F + c + 8 * u) = ob;
                if (trow >= 0) {
                  *reinterpret_cast<uint4*>(dtrow + c + 8 * u) = oa;
                  *reinterpret_cast<uint4*>(dtrow + F + c + 8 * u) = ob;
                }
              }
            }
          }
        }
        if (valid) ws.dgp[p * (int64_t)(2 * n_tiles) + 2 * bt.n_idx + half] = dg;
      } else if (kKind == kBwdDX) {
        const int64_t p = (int64_t)bt.row0 + r;
        int64_t slot = valid ? ws.perm_slot[p] : -1;
        if (slot >= s.N) slot = -1;
        __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(ws.dxslot) + slot * s.d + n0;
#pragma unroll 1
        for (int c = c_beg; c < c_end; c += 32) {
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
      } else {
        // weight gradients, fp32 row-major; an expert without rows gets zeros.  This warp's
        // 32 rows x 32 columns at a time go through its staging block to a TMA store (full
        // 128-byte lines, asynchronous), row `lane` written by lane `lane`, its 16-byte
        // chunk j at j ^ (lane % 8) (the 128-byte swizzle)
        const int mblk = bt.row0 + q * 32;  // first output row of this warp's block
        const bool blk_valid = mblk < M;    // M is a multiple of 64: whole blocks only
        const CUtensorMap* om = &tmO1;
        int orow;
        if (kKind == kBwdDW13) {
          if (mblk >= s.F) om = &tmO2;
          orow = bt.e * s.F + (mblk >= s.F ? mblk - s.F : mblk);
        } else {
          orow = bt.e * s.d + mblk;
        }
        const uint32_t ob = ptx::smem_u32(out_blocks + (warp - kEpiWarp0) * kOutBlockBytes);
#pragma unroll 1
        for (int c = c_beg; c < c_end; c += 32) {
          if (n0 + c >= N) break;
          uint32_t v[32];
          if (bt.kblocks > 0) {
            ptx::tmem_ld_32cols(t_row + c, v);
            ptx::tmem_ld_wait();
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = 0u;
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
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(ptx::smem_u32(&ctl->tempty[acc]));
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (!ok && lane == 0) {
      *abort_flag = 1;
      record_error(ws, MOE_ERR_TIMEOUT, 0x820u + kKind);
    }
    if (k_grouped(kKind) && lane == 0) bulk_wait_all();  // this warp's stores are complete
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
  if (warp == 2) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

template <int kKind>
cudaError_t launch_kind(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& b2, const CUtensorMap& o1,
                        const CUtensorMap& o2, const BwdArgs& args, int num_sms, int64_t timeout_ns, bool pdl,
                        cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(gemm_bwd_kernel<kKind>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  return launch_kernel(gemm_bwd_kernel<kKind>, dim3(num_sms), dim3(kThreads), kSmemBytes, st, pdl, 1, a, b, b2, o1, o2,
                       args, timeout_ns);
}

}  // namespace

cudaError_t launch_gemm_bwd(int kind, const Shape& s, const Ws& ws, const Weights& w, float* dw_a, float* dw_b,
                            int num_sms, int64_t timeout_ns, bool pdl, cudaStream_t st) {
  BwdArgs args{s, ws, dw_a, dw_b};
  CUtensorMap ma, mb, mb2, mo1, mo2;
  cudaError_t e;
  const uint64_t N = (uint64_t)s.N, d = (uint64_t)s.d, F = (uint64_t)s.F, E = (uint64_t)s.E;
  switch (kind) {
    case kBwdDH:
      if ((e = make_tmap_bf16(&ma, ws.dyp, N, d, 128)) != cudaSuccess) return e;
      if ((e = make_tmap_bf16(&mb, w.w2, E * d, F, 64)) != cudaSuccess) return e;
      return launch_kind<kBwdDH>(ma, mb, mb, mb, mb, args, num_sms, timeout_ns, pdl, st);
    case kBwdDX:
      if ((e = make_tmap_bf16(&ma, ws.dab, N, 2 * F, 128)) != cudaSuccess) return e;
      if ((e = make_tmap_bf16(&mb, w.w1, E * F, d, 64)) != cudaSuccess) return e;
      if ((e = make_tmap_bf16(&mb2, w.w3, E * F, d, 64)) != cudaSuccess) return e;
      return launch_kind<kBwdDX>(ma, mb, mb2, mb, mb, args, num_sms, timeout_ns, pdl, st);
    case kBwdDW13:
      if ((e = make_tmap_bf16(&ma, ws.dab, N, 2 * F, 64)) != cudaSuccess) return e;
      if ((e = make_tmap_bf16(&mb, ws.xp, N, d, 64)) != cudaSuccess) return e;
      if ((e = make_tmap_bf16(&mb2, ws.dab_tail, E * 64, 2 * F, 64)) != cudaSuccess) return e;
      if ((e = make_tmap_f32_rows128(&mo1, dw_a, E * F, d, 32)) != cudaSuccess) return e;
      if ((e = make_tmap_f32_rows128(&mo2, dw_b, E * F, d, 32)) != cudaSuccess) return e;
      return launch_kind<kBwdDW13>(ma, mb, mb2, mo1, mo2, args, num_sms, timeout_ns, pdl, st);
    case kBwdDW2:
      if ((e = make_tmap_bf16(&ma, ws.dop, N, d, 64)) != cudaSuccess) return e;
      if ((e = make_tmap_bf16(&mb, ws.h, N, F, 64)) != cudaSuccess) return e;
      if ((e = make_tmap_bf16(&mb2, ws.dop_tail, E * 64, d, 64)) != cudaSuccess) return e;
      if ((e = make_tmap_f32_rows128(&mo1, dw_a, E * d, F, 32)) != cudaSuccess) return e;
      return launch_kind<kBwdDW2>(ma, mb, mb2, mo1, mo1, args, num_sms, timeout_ns, pdl, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace moe
