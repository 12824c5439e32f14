// tile_tables.cuh -- the expert GEMMs' tile tables, built from the rows each owner holds.
//
// An owner is an expert (the layer's forward) or a received segment (the expert stage of
// expert parallelism); owner i holds rows off[i] .. off[i] + cnt[i] - 1 of the A operand and
// multiplies them by the weights of expert i % n_weights.  Its rows are cut into 128-row
// m-tiles, grouped kGroupM at a time (the m-tiles of a group share each weight tile in L2):
//   mt_desc   one entry per m-tile (the one-CTA kernels);
//   pr_desc   one entry per CTA pair of consecutive m-tiles of a group, the last pair of a group
//             with an odd count half empty (the pair kernels).
// Entry layout (int4): x = weight expert | (m-tiles, resp. pairs, of the group) << 20,
// y = the group's first m-tile (pair) index, z = the group's first row, w = one past the
// owner's last row.
#pragma once
#include "device_common.cuh"

namespace moe {

// Shared-memory ints build_tile_tables needs as scratch.
constexpr int kTileScratchInts = 4 * kMaxExperts + 4 * 8 + 8;

__device__ __forceinline__ void owner_tiles(int cnt, int& mt, int& ng, int& last_gm, int& np) {
  mt = (cnt + kTileM - 1) / kTileM;
  ng = (mt + kGroupM - 1) / kGroupM;
  last_gm = mt - (ng - 1) * kGroupM;
  // every group but an owner's last holds kGroupM (even) m-tiles
  np = ng > 0 ? (ng - 1) * (kGroupM / 2) + (last_gm + 1) / 2 : 0;
}

// Largest i in [0, n) with st[i] <= idx (st non-decreasing, st[0] = 0 <= idx).
__device__ __forceinline__ int owner_of(const int* st, int n, int idx) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (st[mid] <= idx) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// Called by all nt threads (nt >= 32, a multiple of 32) of one CTA, with cnt_s[i] (shared,
// i < n <= kMaxExperts; zero or anything past n) holding every owner's row count.  Writes
// ws.counts[0..n), ws.offsets[0..n], the two descriptor tables and the header totals, and
// leaves each owner's first row in offs_s[i] (shared).  The rows must total exactly s.N when
// `exact`, else at most s.N; otherwise, or if the groups would overflow the tables, it records
// MOE_ERR_INTERNAL at `site`, empties the tables and returns -1.  Returns the rows' total.
static __device__ __noinline__ int build_tile_tables(const Shape& s, const Ws& ws, int n, int n_weights, const int* cnt_s,
                                              int* offs_s, int* scratch, int nt, bool exact, uint32_t site) {
  const int tid = threadIdx.x, lane = tid & 31, nw = nt >> 5;
  int* col = scratch;                 // [4][256]: counts, m-tiles, groups, pairs
  int* wtot = col + 4 * kMaxExperts;  // [4][8] warp totals, then their exclusive prefixes
  int* tot = wtot + 4 * 8;            // [4] totals
  for (int i = tid; i < kMaxExperts; i += nt) {
    const int cnt = i < n ? cnt_s[i] : 0;
    int mt, ng, last_gm, np;
    owner_tiles(cnt, mt, ng, last_gm, np);
    col[i] = cnt;
    col[kMaxExperts + i] = mt;
    col[2 * kMaxExperts + i] = ng;
    col[3 * kMaxExperts + i] = np;
  }
  __syncthreads();
  // inclusive scans of the four columns: a warp scan per 32 slots, then the warp totals in order
  for (int w = tid >> 5; w < kMaxExperts / 32; w += nw) {
    const int i = w * 32 + lane;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      int v = col[q * kMaxExperts + i];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int x = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += x;
      }
      col[q * kMaxExperts + i] = v;
      if (lane == 31) wtot[q * 8 + w] = v;
    }
  }
  __syncthreads();
  if (tid < 4) {
    int run = 0;
    for (int w = 0; w < 8; ++w) {
      const int v = wtot[tid * 8 + w];
      wtot[tid * 8 + w] = run;
      run += v;
    }
    tot[tid] = run;
  }
  __syncthreads();
  const int n_rows = tot[0], n_mtiles = tot[1], n_groups = tot[2], n_pairs = tot[3];
  if ((exact ? n_rows != s.N : n_rows > s.N) || n_groups > s.max_groups) {
    if (tid == 0) {
      record_error(ws, MOE_ERR_INTERNAL, site);
      ws.hdr[kHdrNumGroups] = 0;
      ws.hdr[kHdrNumMTiles] = 0;
      ws.hdr[kHdrNumPairs] = 0;
    }
    return -1;
  }
  // exclusive starts in place (inclusive minus the owner's own), counts and offsets out
  for (int i = tid; i < kMaxExperts; i += nt) {
    const int w = i >> 5;
    const int cnt = i < n ? cnt_s[i] : 0;
    int mt, ng, last_gm, np;
    owner_tiles(cnt, mt, ng, last_gm, np);
    const int own[4] = {cnt, mt, ng, np};
#pragma unroll
    for (int q = 0; q < 4; ++q) col[q * kMaxExperts + i] += wtot[q * 8 + w] - own[q];
    if (i < n) {
      offs_s[i] = col[i];
      ws.counts[i] = cnt;
      ws.offsets[i] = col[i];
    }
  }
  __syncthreads();
  const int* mst = col + kMaxExperts;      // first m-tile of each owner
  const int* pst = col + 3 * kMaxExperts;  // first pair
  // one thread per entry of the two tables; the owner of an entry is the last one whose first
  // entry is at or below it (owners without entries share their successor's start)
  for (int q = tid; q < n_mtiles + n_pairs; q += nt) {
    const bool pair = q >= n_mtiles;
    const int idx = pair ? q - n_mtiles : q;
    const int* st = pair ? pst : mst;
    const int i = owner_of(st, n, idx);
    const int cnt = (i + 1 < n ? offs_s[i + 1] : n_rows) - offs_s[i];
    int mt, ng, last_gm, np;
    owner_tiles(cnt, mt, ng, last_gm, np);
    const int off = offs_s[i], local = idx - st[i], we = i % n_weights;
    const int per = pair ? kGroupM / 2 : kGroupM;  // entries of a whole group
    const int g = local / per;
    const int gm = g + 1 < ng ? kGroupM : last_gm;
    const int row0 = off + g * kGroupM * kTileM;
    if (!pair) ws.mt_desc[idx] = make_int4(we | (gm << 20), mst[i] + g * kGroupM, row0, off + cnt);
    else ws.pr_desc[idx] = make_int4(we | (((gm + 1) / 2) << 20), pst[i] + g * per, row0, off + cnt);
  }
  if (tid == 0) {
    ws.offsets[n] = n_rows;
    ws.hdr[kHdrNumGroups] = (uint32_t)n_groups;
    ws.hdr[kHdrNumMTiles] = (uint32_t)n_mtiles;
    ws.hdr[kHdrNumPairs] = (uint32_t)n_pairs;
  }
  __syncthreads();
  return n_rows;
}

}  // namespace moe
