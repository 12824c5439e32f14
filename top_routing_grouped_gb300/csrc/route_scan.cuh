// route_scan.cuh -- the end of the router: the CTA that finishes last turns every router
// block's counts and softmax sums into the per-expert counts, their exclusive scan (the
// dispatch offsets), the per-(block, expert) dispatch bases, the expert GEMMs' tile
// descriptors and the balancing scalar.
//
// After "Distributed Training Part 4 ... MoE + Expert Parallelism" (jesamkim ai-tech-blog):
// §4 Dispatch (every routed row needs a destination; on one GPU the destination is its
// position in an expert-contiguous order, offsets[e] + rank) and §3 Load-Balancing Loss
// (aux = E * sum_e f_e P_e with f_e = count_e / (T k), P_e = mean over tokens of p[t,e]).
//
// The last CTA is found with a completion ticket in the status header (cleared before every
// forward): each router CTA, once its block outputs are written, fences them and takes a
// ticket; the CTA that draws the last one runs the scan.  Nothing waits on another CTA.
//
// The scan's two passes over the [nblk, E] block table are spread over all the CTA's threads:
// thread (chunk c, expert group g) walks the blocks of its chunk for four experts at a time
// (16-byte loads when E is a multiple of 4), so the latency is a few round trips, not one per
// block.  Sums run in block order inside a chunk and over chunks in chunk order, so every
// result is the same on every run.
#pragma once
#include "device_common.cuh"
#include "tile_tables.cuh"

namespace moe {

struct ScanSplit {
  int vw;      // experts per thread step (4: int4 / float4 loads, else 1)
  int groups;  // E / vw expert groups
  int chunks;  // block chunks
  int per;     // router blocks per chunk
};

__host__ __device__ inline ScanSplit scan_split(const Shape& s, int nt) {
  ScanSplit p;
  p.vw = (s.E % 4 == 0) ? 4 : 1;
  p.groups = s.E / p.vw;
  p.chunks = nt / p.groups;
  if (p.chunks < 1) p.chunks = 1;
  if (p.chunks > s.nblk) p.chunks = s.nblk;
  p.per = (s.nblk + p.chunks - 1) / p.chunks;
  return p;
}

// Shared-memory bytes the scan needs when run by nt threads: per-(chunk, expert) counts and
// sums of p, per-expert counts, offsets, sums of p and aux terms, and the tile tables' scratch.
__host__ __device__ inline size_t route_scan_smem(const Shape& s, int nt) {
  const ScanSplit p = scan_split(s, nt);
  return (size_t)p.chunks * s.E * 8 + 4 * kMaxExperts * 4 + (size_t)kTileScratchInts * 4 + 16;
}

// Called by every thread (nt of them) of every router CTA that wrote a token block's outputs,
// after they are written; n_blocks is the number of such CTAs.  Returns whether this CTA ran
// the scan.  `scratch` is route_scan_smem(s, nt) bytes of shared memory, 16-byte aligned, free
// for the scan's use.
static __device__ __noinline__ bool route_scan_if_last(const Shape& s, const Ws& ws, int nt, int n_blocks, void* scratch) {
  __shared__ int is_last;
  const int tid = threadIdx.x;
  __threadfence();  // this block's counts, sums and ranks before its ticket
  __syncthreads();
  if (tid == 0) is_last = atomicAdd(&ws.hdr[kHdrTicket], 1u) == (uint32_t)(n_blocks - 1);
  __syncthreads();
  if (!is_last) return false;
  __threadfence();  // every other block's outputs are visible (their tickets came first)

  const int E = s.E;
  const ScanSplit sp = scan_split(s, nt);
  int* ccnt = static_cast<int*>(scratch);                             // [chunks][E]
  float* cps = reinterpret_cast<float*>(ccnt + sp.chunks * E);       // [chunks][E]
  int* rawc = reinterpret_cast<int*>(cps + sp.chunks * E);           // [256] counts per expert
  int* offs = rawc + kMaxExperts;                                    // [256] offsets per expert
  float* tps = reinterpret_cast<float*>(offs + kMaxExperts);         // [256] sums of p per expert
  float* red = tps + kMaxExperts;                                    // [256] aux terms
  int* tile_scratch = reinterpret_cast<int*>(red + kMaxExperts);     // kTileScratchInts

  // pass A: per-(chunk, expert) sums of the counts and of p, blocks in order (eight blocks'
  // loads in flight at a time)
  for (int i = tid; i < sp.groups * sp.chunks; i += nt) {
    const int g = i % sp.groups, c = i / sp.groups;
    const int b0 = c * sp.per, b1 = min(b0 + sp.per, s.nblk);
    if (sp.vw == 4) {
      int4 cs = make_int4(0, 0, 0, 0);
      float4 ps = make_float4(0.f, 0.f, 0.f, 0.f);
      const int4* cb = reinterpret_cast<const int4*>(ws.blk_cnt) + g;
      const float4* pb = reinterpret_cast<const float4*>(ws.blk_psum) + g;
      const int rs = E / 4;  // int4 per table row
      for (int b = b0; b < b1; b += 8) {
        int4 cv[8];
        float4 pv[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          cv[u] = b + u < b1 ? __ldcg(cb + (int64_t)(b + u) * rs) : make_int4(0, 0, 0, 0);
          pv[u] = b + u < b1 ? __ldcg(pb + (int64_t)(b + u) * rs) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          if (b + u >= b1) break;
          cs.x += cv[u].x; cs.y += cv[u].y; cs.z += cv[u].z; cs.w += cv[u].w;
          ps.x += pv[u].x; ps.y += pv[u].y; ps.z += pv[u].z; ps.w += pv[u].w;
        }
      }
      int* cc = ccnt + c * E + 4 * g;
      float* cp = cps + c * E + 4 * g;
      cc[0] = cs.x; cc[1] = cs.y; cc[2] = cs.z; cc[3] = cs.w;
      cp[0] = ps.x; cp[1] = ps.y; cp[2] = ps.z; cp[3] = ps.w;
    } else {
      int cs = 0;
      float ps = 0.f;
      for (int b = b0; b < b1; b += 8) {
        int cv[8];
        float pv[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          cv[u] = b + u < b1 ? __ldcg(ws.blk_cnt + (int64_t)(b + u) * E + g) : 0;
          pv[u] = b + u < b1 ? __ldcg(ws.blk_psum + (int64_t)(b + u) * E + g) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          if (b + u >= b1) break;
          cs += cv[u];
          ps += pv[u];
        }
      }
      ccnt[c * E + g] = cs;
      cps[c * E + g] = ps;
    }
  }
  __syncthreads();
  // per expert: totals, and chunk prefixes in chunk order
  for (int e = tid; e < kMaxExperts; e += nt) {
    int cnt = 0;
    float ps = 0.f;
    if (e < E)
      for (int c = 0; c < sp.chunks; ++c) {
        const int v = ccnt[c * E + e];
        ccnt[c * E + e] = cnt;
        cnt += v;
        ps += cps[c * E + e];
      }
    rawc[e] = cnt;
    tps[e] = ps;
  }
  __syncthreads();
  // counts, offsets, tile tables, header totals; every routed row must be counted once
  if (build_tile_tables(s, ws, E, E, rawc, offs, tile_scratch, nt, /*exact=*/true, 0x200u) < 0) return true;
  for (int e = tid; e < kMaxExperts; e += nt) {
    float term = 0.f;
    if (e < E) {
      if (ws.ptot) ws.ptot[e] = tps[e];
      // aux term f_e * P_e
      term = ((float)rawc[e] / ((float)s.T * (float)s.k)) * (tps[e] / (float)s.T);
    }
    red[e] = term;
  }
  __syncthreads();
  // aux = E * sum_e f_e P_e over a fixed tree
  for (int half = kMaxExperts / 2; half > 0; half >>= 1) {
    for (int e = tid; e < half; e += nt) red[e] += red[e + half];
    __syncthreads();
  }
  if (tid == 0) *ws.aux = (float)E * red[0];
  // pass B: per-(block, expert) bases = offset + chunk prefix + the chunk's earlier blocks;
  // the counts of eight blocks are requested before any is used (one round trip per eight)
  for (int i = tid; i < sp.groups * sp.chunks; i += nt) {
    const int g = i % sp.groups, c = i / sp.groups;
    const int b0 = c * sp.per, b1 = min(b0 + sp.per, s.nblk);
    if (sp.vw == 4) {
      int run[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int e = 4 * g + q;
        run[q] = offs[e] + ccnt[c * E + e];
      }
      const int rs = E / 4;
      const int4* cb = reinterpret_cast<const int4*>(ws.blk_cnt) + g;
      int4* bb = reinterpret_cast<int4*>(ws.blk_base) + g;
      for (int b = b0; b < b1; b += 8) {
        int4 cv[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) cv[u] = b + u < b1 ? __ldcg(cb + (int64_t)(b + u) * rs) : make_int4(0, 0, 0, 0);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          if (b + u < b1) bb[(int64_t)(b + u) * rs] = make_int4(run[0], run[1], run[2], run[3]);
          run[0] += cv[u].x; run[1] += cv[u].y; run[2] += cv[u].z; run[3] += cv[u].w;
        }
      }
    } else {
      int run = offs[g] + ccnt[c * E + g];
      for (int b = b0; b < b1; b += 8) {
        int cv[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) cv[u] = b + u < b1 ? __ldcg(ws.blk_cnt + (int64_t)(b + u) * E + g) : 0;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          if (b + u < b1) ws.blk_base[(int64_t)(b + u) * E + g] = run;
          run += cv[u];
        }
      }
    }
  }
  return true;
}

}  // namespace moe
