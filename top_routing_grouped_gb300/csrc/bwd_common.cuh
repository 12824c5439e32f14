// bwd_common.cuh -- small device helpers shared by the backward's tensor-core kernels:
// MN-major shared-memory descriptors, bf16 packing, shared-window vector accesses and TMA
// stores of staged blocks.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace moe {
namespace bwd {

constexpr int kBoxBytes = 64 * 64 * 2;  // one 64 (MN) x 64 (K) bf16 box, 128-byte rows

// MN-major operand of 64-wide MN blocks stored kBoxBytes apart (TMA boxes side by side),
// 128-byte swizzled: leading offset = the next 64-wide MN block, stride = the next 8 K rows.
// One K=16 MMA step is 16 rows = 2 KB further.
__device__ __forceinline__ uint64_t desc_mnmajor_sw128(uint32_t addr) {
  uint64_t d = 0;
  d |= (uint64_t)((addr & 0x3FFFFu) >> 4);
  d |= (uint64_t)(kBoxBytes >> 4) << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

__device__ __forceinline__ uint32_t pack2(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ void unpack8(uint4 raw, float* f) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 v = __bfloat1622float2(h[i]);
    f[2 * i] = v.x;
    f[2 * i + 1] = v.y;
  }
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// a load that the compiler keeps after the warp barrier that publishes the block
__device__ __forceinline__ void ld_block_v4(uint32_t addr, float& a, float& b, float& c, float& d) {
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(a), "=f"(b), "=f"(c), "=f"(d) : "r"(addr) : "memory");
}

// Row `lane` of a 32-row block of 128-byte rows (32 fp32), 16-byte chunk j stored at
// j ^ (lane % 8): the 128-byte swizzle, so that the lanes' stores and a TMA store of the
// block agree and no two lanes of a phase share a bank.
__device__ __forceinline__ void stage_row32(uint32_t block, int lane, const uint32_t (&v)[32]) {
#pragma unroll
  for (int j = 0; j < 8; ++j)
    st_shared_v4(block + (uint32_t)lane * 128u + (uint32_t)((j ^ (lane & 7)) * 16), v[4 * j], v[4 * j + 1],
                 v[4 * j + 2], v[4 * j + 3]);
}

// 2-D tiled TMA store of a staged shared-memory block (bulk group of this thread).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, int32_t c0, int32_t c1, uint32_t src) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(src)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

}  // namespace bwd
}  // namespace moe
