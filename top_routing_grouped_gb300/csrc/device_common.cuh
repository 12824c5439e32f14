// device_common.cuh -- small device helpers shared by the kernels.
#pragma once
#include <cuda_bf16.h>
#include <stdint.h>

#include "moe_internal.h"

namespace moe {

__device__ __forceinline__ float load_act(const void* base, int bf16, int64_t i) {
  if (bf16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(base)[i]);
  return reinterpret_cast<const float*>(base)[i];
}

__device__ __forceinline__ void store_act(void* base, int bf16, int64_t i, float v) {
  if (bf16)
    reinterpret_cast<__nv_bfloat16*>(base)[i] = __float2bfloat16_rn(v);
  else
    reinterpret_cast<float*>(base)[i] = v;
}

// Logistic sigmoid through the identity sigmoid(a) = (1 + tanh(a/2)) / 2 with the hardware
// tanh approximation (relative error about 2^-11): one transcendental and no divide, well
// below the bf16 rounding the GEMM epilogues apply to their results.
__device__ __forceinline__ float sigmoid_fast(float a) {
  float t;
  asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(0.5f * a));
  return fmaf(0.5f, t, 0.5f);
}

// SiLU(a) = a * sigmoid(a) = h + h tanh(h), h = a/2.
__device__ __forceinline__ float silu_fast(float a) {
  const float h = 0.5f * a;
  float t;
  asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(h));
  return fmaf(h, t, h);
}

// shared-memory loads and stores by shared-window address: the compiler cannot tell a
// generic pointer into shared memory from a global one, and orders such accesses
// conservatively; these keep the epilogues' traffic on the shared path, issued in the
// order written
__device__ __forceinline__ float ld_shared_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ void ld_shared_v4(uint32_t addr, float& a, float& b, float& c, float& d) {
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(a), "=f"(b), "=f"(c), "=f"(d) : "r"(addr));
}

__device__ __forceinline__ void st_shared_f32(uint32_t addr, float v) {
  asm volatile("st.shared.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// First error wins; `where` records which kernel/site saw it.
__device__ __forceinline__ void record_error(const Ws& ws, uint32_t code, uint32_t where) {
  if (atomicCAS(&ws.hdr[kHdrStatus], 0u, code) == 0u) ws.hdr[kHdrWhere] = where;
}

// Programmatic dependent launch: the kernels of one forward are chained so that a kernel's
// launch and prologue overlap its predecessor.  pdl_wait() blocks until every grid this one
// depends on has completed and its memory is visible (a no-op when launched without the
// attribute); it must precede any read of a predecessor's output.  pdl_launch_dependents()
// lets the next kernel in the stream be scheduled early.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// One m x n output tile of a grouped GEMM.
struct TileInfo {
  int e;      // expert
  int row0;   // first row in dispatch order
  int rows;   // valid rows (1..kTileM)
  int n_idx;  // n-tile index
};

// Decode linear tile id -> tile.  Scheduling groups hold up to kGroupM consecutive
// m-tiles of one expert; inside a group the m-tile index runs fastest, so CTAs that run
// at the same time share the same weight n-tile (read once from HBM, then from L2).
// Group g owns tiles [n_tiles * mpre[g], n_tiles * mpre[g+1]).
// The group is found from the descriptor of entry tile / n_tiles (one load).
__device__ __forceinline__ TileInfo decode_tile(const Ws& ws, int n_tiles, int tile) {
  const int4 g = __ldg(&ws.mt_desc[tile / n_tiles]);
  const int gm = g.x >> 20;
  const int local = tile - n_tiles * g.y;
  TileInfo ti;
  ti.e = g.x & 0xFFFFF;
  ti.n_idx = local / gm;
  ti.row0 = g.z + (local % gm) * kTileM;
  const int rem = g.w - ti.row0;
  ti.rows = rem < kTileM ? rem : kTileM;
  return ti;
}

// Decode linear pair-tile id -> the m-tile of CTA `rank` (0/1) of a CTA pair.  A pair tile
// is two consecutive m-tiles of one scheduling group (the second may not exist: rows <= 0)
// times one n-tile; group g owns pair tiles [n_tiles * ppre[g], n_tiles * ppre[g+1]) and
// inside a group the pair index runs fastest.
__device__ __forceinline__ TileInfo decode_pair_tile(const Ws& ws, int n_tiles, int tile, int rank) {
  const int4 g = __ldg(&ws.pr_desc[tile / n_tiles]);
  const int gp = g.x >> 20;
  const int local = tile - n_tiles * g.y;
  TileInfo ti;
  ti.e = g.x & 0xFFFFF;
  ti.n_idx = local / gp;
  ti.row0 = g.z + (2 * (local % gp) + rank) * kTileM;
  const int rem = g.w - ti.row0;
  ti.rows = rem < kTileM ? rem : kTileM;  // <= 0: no such m-tile (odd group), nothing stored
  return ti;
}

}  // namespace moe
