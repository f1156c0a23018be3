// Work-split metadata shared by the decode-shaped forward kernels: one split
// per lane, read with a single chain of dependent loads per 32 splits.
#pragma once

#include <cstdint>

#include "internal.h"
#include "sa_common.cuh"

namespace sa {
namespace dec {

constexpr int kMaxPages = 8;       // pages per block
constexpr int kMaxQi = 8;          // query ids of a split's first edges kept per split

// Split metadata, one split per lane.
struct SplitMeta {
  int h, nrows, edge0, bstart, bend, lk;
  int64_t q0, qo;
  uint32_t pmask;             // page p present (0 <= id < num_pages) and overlapping the live range
  int pid[kMaxPages];
  int qi[kMaxQi];             // queries of the first kMaxQi edges
};

__device__ __forceinline__ void load_meta(const ForwardArgs& a, int64_t sp, int64_t n_splits,
                                          int staged_edges, SplitMeta& m) {
  m.h = 0; m.nrows = 0; m.edge0 = 0; m.bstart = 0; m.bend = 0; m.lk = 0;
  m.q0 = 0; m.qo = 0; m.pmask = 0;
#pragma unroll
  for (int p = 0; p < kMaxPages; ++p) m.pid[p] = -1;
#pragma unroll
  for (int e = 0; e < kMaxQi; ++e) m.qi[e] = 0;
  if (sp >= n_splits) return;
  const int4 w = reinterpret_cast<const int4*>(a.splits)[sp];
  const bool sane = w.x >= 0 && w.x < a.hkv && w.y >= 0 && w.y < a.nbs && w.w >= w.z && w.z >= 0;
  const int raw = sane ? a.sel_slots[static_cast<int64_t>(w.x) * a.nbs + w.y] : -1;
  if (raw < 0 || raw >= a.nbs) {
    report(a.totals + 3, SA_ERR_SHAPE);
    return;
  }
  m.h = w.x;
  m.edge0 = w.z;
  m.nrows = (w.w - w.z) * a.qhead;
  const int b = raw / a.msb;
  const int blk = raw - b * a.msb;
  m.lk = a.used ? max(a.used[b], 0) : a.msb * a.block_size;
  m.bstart = blk * a.block_size;
  m.bend = min(m.bstart + a.block_size, m.lk);
  m.q0 = a.cu[b];
  m.qo = a.cu[b + 1] - m.q0;
  const int32_t* bt = a.block_tables + static_cast<int64_t>(b) * a.max_pages +
                      static_cast<int64_t>(blk) * a.pages_per_block;
#pragma unroll
  for (int p = 0; p < kMaxPages; ++p) {
    if (p < a.pages_per_block && m.bstart + p * a.page_size < m.bend) {
      const int id = bt[p];
      if (id >= a.num_pages) report(a.totals + 3, SA_ERR_SHAPE);
      if (id >= 0 && id < a.num_pages) {
        m.pid[p] = id;
        m.pmask |= 1u << p;
      }
    }
  }
  (void)staged_edges;
  const int ne = min(w.w - w.z, kMaxQi);
#pragma unroll
  for (int e = 0; e < kMaxQi; ++e)
    if (e < ne) m.qi[e] = a.edges[2 * (static_cast<int64_t>(w.z) + e)];
}

// Broadcast the metadata of lane `src` to the whole warp.
__device__ __forceinline__ SplitMeta bcast_meta(const SplitMeta& m, int src) {
  SplitMeta r;
  r.h = __shfl_sync(0xffffffffu, m.h, src);
  r.nrows = __shfl_sync(0xffffffffu, m.nrows, src);
  r.edge0 = __shfl_sync(0xffffffffu, m.edge0, src);
  r.bstart = __shfl_sync(0xffffffffu, m.bstart, src);
  r.bend = __shfl_sync(0xffffffffu, m.bend, src);
  r.lk = __shfl_sync(0xffffffffu, m.lk, src);
  r.q0 = __shfl_sync(0xffffffffu, m.q0, src);
  r.qo = __shfl_sync(0xffffffffu, m.qo, src);
  r.pmask = __shfl_sync(0xffffffffu, m.pmask, src);
#pragma unroll
  for (int p = 0; p < kMaxPages; ++p) r.pid[p] = __shfl_sync(0xffffffffu, m.pid[p], src);
#pragma unroll
  for (int e = 0; e < kMaxQi; ++e) r.qi[e] = __shfl_sync(0xffffffffu, m.qi[e], src);
  return r;
}

// Scalars of the metadata of lane `src` (the page ids and query ids stay in
// the per-warp shared table written by stash_meta_arrays).
__device__ __forceinline__ SplitMeta bcast_scalars(const SplitMeta& m, int src) {
  SplitMeta r;
  r.h = __shfl_sync(0xffffffffu, m.h, src);
  r.nrows = __shfl_sync(0xffffffffu, m.nrows, src);
  r.edge0 = __shfl_sync(0xffffffffu, m.edge0, src);
  r.bstart = __shfl_sync(0xffffffffu, m.bstart, src);
  r.bend = __shfl_sync(0xffffffffu, m.bend, src);
  r.lk = __shfl_sync(0xffffffffu, m.lk, src);
  r.q0 = __shfl_sync(0xffffffffu, m.q0, src);
  r.qo = __shfl_sync(0xffffffffu, m.qo, src);
  r.pmask = __shfl_sync(0xffffffffu, m.pmask, src);
  return r;
}

// Page ids and query ids of this lane's split into row `lane` of the tables.
__device__ __forceinline__ void stash_meta_arrays(const SplitMeta& m, int lane, int* pid_tab,
                                                  int* qi_tab) {
#pragma unroll
  for (int p = 0; p < kMaxPages; ++p) pid_tab[lane * kMaxPages + p] = m.pid[p];
#pragma unroll
  for (int e = 0; e < kMaxQi; ++e) qi_tab[lane * kMaxQi + e] = m.qi[e];
}

}  // namespace dec
}  // namespace sa
