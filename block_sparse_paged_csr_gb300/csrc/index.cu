// Step 1 of KV-outer sparse attention: the CSR index (KvOuterIndex, types.rs
// of alice-llm's sparse_attention) and the forward's work list (WorkSplit).
//
// Structure.  The entries (query i, kv head h, rank r) of one (h, sequence b)
// segment can only land in raw slots b*msb .. b*msb+msb-1 of head h, and
// segments in (h, b) order own consecutive slot ranges.  A segment's entries
// in (query, rank) order are cut into chunks of at most kChunkEntries; CTAs
// walk chunks with a grid stride.  One cooperative kernel, two phases:
//   phase 1  each chunk histograms its entries into msb shared-memory bins;
//            a one-chunk segment writes its totals (edges, non-empty bins,
//            work splits) directly; a segment of several chunks stores each
//            chunk's histogram, and the chunk that arrives last (atomic
//            counter after a fence) sums them and writes the totals.
//   -- one grid barrier (bounded spin; the launch is cooperative, so every
//      CTA is resident); the last CTA to arrive scans the segment totals
//      into exclusive prefixes before it releases the others --
//   phase 2  each chunk reads its segment's global prefix and its head's
//            base, rebuilds its bins, scans them, and (first chunk of the
//            segment) writes sel_slots / sel_offsets / the splits of the
//            segment; then it scatters its own edges: entries walk in
//            (query, rank) order 256 at a time, equal keys inside a warp are
//            ranked with
//            __match_any_sync and warps take their running bin counts in warp
//            order, on top of the counts of the segment's earlier chunks, so
//            each bucket is in ascending (query, rank) order and the result
//            is deterministic.  All CTAs then write the plateau of
//            sel_offsets and the -1 padding of sel_slots.
#include <algorithm>
#include <cstdint>

#include "internal.h"
#include "sa_common.cuh"

namespace sa {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_u32(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ int64_t splits_of(int64_t count, int split_edges) {
  if (count <= 0) return 0;
  if (split_edges <= 0) return 1;
  return (count + split_edges - 1) / split_edges;
}

// Grid-wide barrier for a cooperative launch.  The last CTA to arrive first
// runs `last` (with all of its threads), then resets the counter and bumps the
// generation; the others spin (bounded) on the generation.
__device__ __forceinline__ uint32_t atom_add_acq_rel_u32(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// Grid-wide barrier for a cooperative launch.  `gen0` is the generation read
// (by thread 0) at the start of the kernel: no CTA can pass this barrier
// before every CTA has arrived, so it cannot have moved since.  Arrival is an
// acquire-release add (the CTA's earlier writes, fenced by each thread, go
// first; the last arrival sees everyone's);
// the last CTA to arrive first runs `last` (with all of its threads), then
// resets the counter and publishes the next generation with a release store;
// the others poll the generation (acquire, bounded).
template <typename F>
__device__ bool grid_barrier(uint32_t* count, uint32_t* gen, uint32_t gen0, uint32_t nblocks,
                             uint32_t limit, bool stall, F last) {
  __shared__ int s_ok, s_last;
  __syncthreads();
  if (threadIdx.x == 0) {
    s_ok = 1;
    s_last = atom_add_acq_rel_u32(count, 1u) == nblocks - 1;
    if (stall) s_last = 0;   // test hook: nobody releases the barrier
  }
  __syncthreads();
  if (s_last) {
    __threadfence();
    last();
    __syncthreads();
    if (threadIdx.x == 0) {
      *reinterpret_cast<volatile uint32_t*>(count) = 0u;
      st_release_u32(gen, gen0 + 1);
    }
  } else if (threadIdx.x == 0) {
    uint32_t it = 0;
    while (ld_acquire_u32(gen) == gen0) {
      if (++it > limit) {
        s_ok = 0;
        break;
      }
      __nanosleep(32);
    }
  }
  __syncthreads();
  return s_ok != 0;
}

// Arrival-only grid barrier (the counter cleared before the launch): every
// CTA adds one (acquire-release, after its writes) and waits (bounded) until
// all have.  Nothing is computed at the barrier: the readers derive what
// they need from the published totals themselves.
__device__ bool grid_arrive_wait(uint32_t* count, uint32_t nblocks, uint32_t limit, bool stall) {
  __shared__ int s_ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    s_ok = 1;
    if (!stall) atom_add_acq_rel_u32(count, 1u);   // test hook: nobody arrives
    uint32_t it = 0;
    while (ld_acquire_u32(count) < nblocks) {
      if (++it > limit) {
        s_ok = 0;
        break;
      }
      __nanosleep(32);
    }
  }
  __syncthreads();
  return s_ok != 0;
}

// Block-wide sum of three 64-bit values; every thread gets the totals.
__device__ __forceinline__ void block_sum3(int64_t v[3], int64_t (*scratch)[kWarps]) {
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
#pragma unroll
  for (int q = 0; q < 3; ++q)
#pragma unroll
    for (int off = 16; off; off >>= 1) v[q] += __shfl_xor_sync(0xffffffffu, v[q], off);
  __syncthreads();
  if (lane == 0)
#pragma unroll
    for (int q = 0; q < 3; ++q) scratch[q][warp] = v[q];
  __syncthreads();
#pragma unroll
  for (int q = 0; q < 3; ++q) {
    int64_t t = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) t += scratch[q][w];
    v[q] = t;
  }
}

// Exclusive block scan of three values (per-thread contributions in thread
// order); also returns the block totals.
__device__ __forceinline__ void block_scan3(int64_t v[3], int64_t excl[3], int64_t tot[3],
                                            int64_t (*warp_tot)[kWarps]) {
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  int64_t inc[3] = {v[0], v[1], v[2]};
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
#pragma unroll
    for (int q = 0; q < 3; ++q) {
      const int64_t n = __shfl_up_sync(0xffffffffu, inc[q], off);
      if (lane >= off) inc[q] += n;
    }
  }
  __syncthreads();
  if (lane == 31)
#pragma unroll
    for (int q = 0; q < 3; ++q) warp_tot[q][warp] = inc[q];
  __syncthreads();
#pragma unroll
  for (int q = 0; q < 3; ++q) {
    int64_t before = 0, all = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const int64_t x = warp_tot[q][w];
      if (w < warp) before += x;
      all += x;
    }
    excl[q] = before + inc[q] - v[q];
    tot[q] = all;
  }
}

struct Shared {
  int64_t scratch[3][kWarps];
  int32_t nch_head;      // chunks per head
  int32_t nmulti_head;   // histogram slots per head
  int last;
  uint32_t gen0;         // barrier generation at the start
  int64_t my_pre[kWarps][3];  // warp-per-segment mode: the warps' segment prefixes
};

// Which (head, sequence, chunk) a chunk id names.
__device__ __forceinline__ void locate(int64_t c, const int32_t* chunk_base, int batch,
                                       int nch_head, int& h, int& b, int& k) {
  h = static_cast<int>(c / nch_head);
  const int r = static_cast<int>(c - static_cast<int64_t>(h) * nch_head);
  int lo = 0, hi = batch;   // largest b with chunk_base[b] <= r and a chunk
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (chunk_base[mid] <= r) lo = mid; else hi = mid;
  }
  b = lo;
  k = r - chunk_base[lo];
}

// ---- warp-per-segment mode (every segment holds at most 64 entries) --------
// Entry t of segment (h, b) (query cu[b] + t / topk, rank t % topk) sits in
// lane t & 31 of round t >> 5.  With 64 entries at most, every statistic of
// the counting sort comes from warp shuffles over the entries: for entry t
// with block x (kept entries only),
//   same   kept entries with block x,
//   before kept entries with block x and a smaller t (0: t opens its bucket),
//   less   kept entries with a smaller block,
//   ul     buckets (distinct blocks) below x, sl their work splits.
// All of it is local to the segment, so a warp computes it before the grid
// barrier and keeps it in registers for the scatter after it.
struct SmallSeg {
  int64_t q0;        // first query of the sequence
  int n;             // entries of the segment
  bool bad;          // an out-of-range block id was seen
  int blk[2];        // block of the entry, -1 when dropped
  int same[2], before[2], less[2], ul[2], sl[2];
};

__device__ __forceinline__ void small_segment(const IndexArgs& a, int h, int b, int lane,
                                              SmallSeg& g) {
  g.q0 = a.cu[b];
  g.n = static_cast<int>((a.cu[b + 1] - g.q0) * a.topk);
  const int n = g.n;
  const int64_t lk = a.used ? (a.used[b] > 0 ? a.used[b] : 0)
                            : static_cast<int64_t>(a.msb) * a.block_size;
  g.bad = false;
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int t = 32 * k + lane;
    g.blk[k] = -1;
    if (t < n) {
      const int64_t i = g.q0 + t / a.topk;
      const int r = t % a.topk;
      const int x = a.selected[(i * a.hkv + h) * a.topk + r];
      if (x < -1 || x >= a.msb) g.bad = true;
      if (x >= 0 && x < a.msb && static_cast<int64_t>(x) * a.block_size < lk) g.blk[k] = x;
    }
    g.same[k] = g.before[k] = g.less[k] = g.ul[k] = 0;
    g.sl[k] = 0;
  }
  // Both rounds' entry j at once (j < 32): independent shuffles, unrolled so
  // that their latencies overlap.
  const int nj = n < 32 ? n : 32;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    if (j >= nj) break;
    const int x0 = __shfl_sync(0xffffffffu, g.blk[0], j);
    const int x1 = __shfl_sync(0xffffffffu, g.blk[1], j);
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int t = 32 * k + lane;
      const int x = g.blk[k];
      // entry j (round 0) and entry 32 + j (round 1)
      const int e0 = (x0 >= 0 && x >= 0) ? (x0 == x ? 1 : 0) : 0;
      const int e1 = (x1 >= 0 && x >= 0) ? (x1 == x ? 1 : 0) : 0;
      g.same[k] += e0 + e1;
      g.before[k] += (j < t ? e0 : 0) + (32 + j < t ? e1 : 0);
      g.less[k] += (x0 >= 0 && x >= 0 && x0 < x ? 1 : 0) +
                   (x1 >= 0 && x >= 0 && x1 < x ? 1 : 0);
    }
  }
  // Buckets below each entry's block: the opening entries (before == 0) of
  // smaller blocks, and their splits.  When no block repeats (one query per
  // sequence, as in decode), every kept entry opens its bucket of one edge:
  // both are `less`.
  const bool repeats = (g.blk[0] >= 0 && g.same[0] > 1) || (g.blk[1] >= 0 && g.same[1] > 1);
  if (!__any_sync(0xffffffffu, repeats)) {
    const int one = static_cast<int>(splits_of(1, a.split_edges));
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      g.ul[k] = g.less[k];
      g.sl[k] = g.less[k] * one;
    }
    return;
  }
#pragma unroll 4
  for (int j = 0; j < nj; ++j) {
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      const int xj = __shfl_sync(0xffffffffu, g.blk[kk], j);
      const int bj = __shfl_sync(0xffffffffu, g.before[kk], j);
      const int sj = __shfl_sync(0xffffffffu, g.same[kk], j);
      const bool open = xj >= 0 && bj == 0;
#pragma unroll
      for (int k = 0; k < 2; ++k)
        if (open && g.blk[k] >= 0 && xj < g.blk[k]) {
          ++g.ul[k];
          g.sl[k] += static_cast<int>(splits_of(sj, a.split_edges));
        }
    }
  }
}

// Fill p[0, n) with v over all threads of the grid (16-byte stores on the
// aligned middle).
__device__ __forceinline__ void fill_i32(int32_t* p, int64_t n, int32_t v, int64_t tid,
                                         int64_t nthreads) {
  if (n <= 0) return;
  const int64_t mis = static_cast<int64_t>((reinterpret_cast<uintptr_t>(p) >> 2) & 3);
  const int64_t head = mis ? (4 - mis < n ? 4 - mis : n) : 0;
  if (tid < head) p[tid] = v;
  int4* q = reinterpret_cast<int4*>(p + head);
  const int64_t nv = (n - head) >> 2;
  const int4 w = make_int4(v, v, v, v);
  for (int64_t i = tid; i < nv; i += nthreads) q[i] = w;
  const int64_t tail = head + 4 * nv;
  if (tid < n - tail) p[tail + tid] = v;
}

template <bool kSmall>
__global__ void __launch_bounds__(kThreads, 4)
index_kernel(IndexArgs a, WorkspaceLayout lay, int64_t n_chunks) {
  extern __shared__ int64_t dyn64[];
  const int msb = a.msb;
  const int batch = a.batch;
  int64_t* head_tot = dyn64;                                          // [hkv][2]
  int32_t* bins = reinterpret_cast<int32_t*>(dyn64 + 2 * a.hkv);      // [msb]
  int32_t* before = bins + msb;                                       // [msb]
  int32_t* start = before + msb;                                      // [msb]
  int32_t* chunk_base = start + msb;                                  // [batch+1]
  int32_t* multi_base = chunk_base + batch + 1;                       // [batch+1]
  __shared__ Shared s;

  char* ws = static_cast<char*>(a.idx.workspace);
  uint32_t* bar_count = reinterpret_cast<uint32_t*>(ws + lay.barrier);
  uint32_t* bar_gen = bar_count + 1;
  uint32_t* seg_done = reinterpret_cast<uint32_t*>(ws + lay.seg_done);
  int32_t* seg_tot = reinterpret_cast<int32_t*>(ws + lay.seg_tot);   // [nseg][3]
  int64_t* seg_pre = reinterpret_cast<int64_t*>(ws + lay.seg_pre);   // [nseg+1][3] exclusive
  int32_t* hist = reinterpret_cast<int32_t*>(ws + lay.hist);         // [slots][msb]
  int64_t* status = a.idx.totals + 3;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int topk = a.topk;
  const int32_t* sel = a.selected;
  const int64_t cap = a.tq * a.hkv * static_cast<int64_t>(topk);
  const int nseg = a.hkv * batch;

  // ---- chunk table (every CTA builds its own copy) -------------------------
  // chunk_base[b]: chunks of the sequences before b; multi_base[b]: the same
  // over sequences of several chunks.  One block scan per kThreads sequences
  // (the cu reads of a tile are issued together, not one after another).
  if (!kSmall) {
    int64_t carry_c = 0, carry_m = 0;
    for (int base = 0; base < batch; base += kThreads) {
      const int b = base + tid;
      int64_t v[3] = {0, 0, 0};
      if (b < batch) {
        const int64_t n = (a.cu[b + 1] - a.cu[b]) * topk;
        const int64_t nc = (n + kChunkEntries - 1) / kChunkEntries;
        v[0] = nc;
        v[1] = nc > 1 ? nc : 0;
      }
      int64_t excl[3], tot[3];
      block_scan3(v, excl, tot, s.scratch);
      if (b < batch) {
        chunk_base[b] = static_cast<int32_t>(carry_c + excl[0]);
        multi_base[b] = static_cast<int32_t>(carry_m + excl[1]);
      }
      carry_c += tot[0];
      carry_m += tot[1];
    }
    if (tid == 0) {
      chunk_base[batch] = static_cast<int32_t>(carry_c);
      multi_base[batch] = static_cast<int32_t>(carry_m);
      s.nch_head = static_cast<int32_t>(carry_c);
      s.nmulti_head = static_cast<int32_t>(carry_m);
    }
  }
  if (tid == 0) s.gen0 = ld_acquire_u32(bar_gen);
  if (blockIdx.x == 0 && tid == 0 && !a.external_clear) {
    *status = 0;
    __threadfence();
  }
  __syncthreads();
  // A fused decode kernel launched behind this one reads none of its outputs
  // (only the memset workspace counters and the status word cleared above):
  // let it start now.
  griddep_launch_dependents();
  const int nch_head = s.nch_head;
  const int nmulti = s.nmulti_head;

  // ---- phase 1: per-chunk histograms and segment totals ---------------------
  const int64_t gtid = static_cast<int64_t>(blockIdx.x) * kThreads + tid;
  const int64_t gthreads = static_cast<int64_t>(gridDim.x) * kThreads;
  // Warp-per-segment mode: one segment per warp at most (the launch has
  // enough warps), spread over the CTAs first, then over their warps.
  const int my_seg = warp * gridDim.x + blockIdx.x;
  SmallSeg g;
  if (kSmall && my_seg < nseg) {
    const int h = my_seg / batch, b = my_seg - (my_seg / batch) * batch;
    small_segment(a, h, b, lane, g);
    int64_t v[3] = {0, 0, 0};
#pragma unroll
    for (int k = 0; k < 2; ++k)
      if (g.blk[k] >= 0) {
        v[0] += 1;
        if (g.before[k] == 0) {
          v[1] += 1;
          v[2] += splits_of(g.same[k], a.split_edges);
        }
      }
#pragma unroll
    for (int q = 0; q < 3; ++q)
#pragma unroll
      for (int off = 16; off; off >>= 1) v[q] += __shfl_xor_sync(0xffffffffu, v[q], off);
    if (lane == 0) {
      seg_tot[3 * my_seg + 0] = static_cast<int32_t>(v[0]);
      seg_tot[3 * my_seg + 1] = static_cast<int32_t>(v[1]);
      seg_tot[3 * my_seg + 2] = static_cast<int32_t>(v[2]);
    }
  }
  for (int64_t c = kSmall ? n_chunks : blockIdx.x; c < n_chunks; c += gridDim.x) {
    int h, b, k;
    locate(c, chunk_base, batch, nch_head, h, b, k);
    const int nc = chunk_base[b + 1] - chunk_base[b];
    const int64_t q0 = a.cu[b];
    const int64_t n_seg = (a.cu[b + 1] - q0) * topk;
    const int64_t e0 = static_cast<int64_t>(k) * kChunkEntries;
    const int64_t e1 = min(n_seg, e0 + kChunkEntries);
    const int64_t lk = a.used ? (a.used[b] > 0 ? a.used[b] : 0)
                              : static_cast<int64_t>(msb) * a.block_size;
    for (int t = tid; t < msb; t += kThreads) bins[t] = 0;
    __syncthreads();
    for (int64_t e = e0 + tid; e < e1; e += kThreads) {
      const int64_t i = q0 + e / topk;
      const int r = static_cast<int>(e % topk);
      const int blk = sel[(i * a.hkv + h) * topk + r];
      if (blk >= 0 && blk < msb && static_cast<int64_t>(blk) * a.block_size < lk)
        atomicAdd(&bins[blk], 1);
    }
    __syncthreads();
    const int seg = h * batch + b;
    bool totals_here = nc == 1;
    if (nc > 1) {
      int32_t* mine = hist + (static_cast<int64_t>(h) * nmulti + multi_base[b] + k) * msb;
      for (int t = tid; t < msb; t += kThreads) mine[t] = bins[t];
      __threadfence();
      __syncthreads();
      if (tid == 0) s.last = atomicAdd(seg_done + seg, 1u) == static_cast<uint32_t>(nc - 1);
      __syncthreads();
      totals_here = s.last != 0;
      if (totals_here) {
        __threadfence();
        const int32_t* first = hist + (static_cast<int64_t>(h) * nmulti + multi_base[b]) * msb;
        for (int t = tid; t < msb; t += kThreads) {
          int32_t sum = 0;
          for (int kk = 0; kk < nc; ++kk)
            sum += *reinterpret_cast<const volatile int32_t*>(first + static_cast<int64_t>(kk) * msb + t);
          bins[t] = sum;
        }
        __syncthreads();
      }
    }
    if (totals_here) {
      int64_t v[3] = {0, 0, 0};
      for (int t = tid; t < msb; t += kThreads) {
        const int cnt = bins[t];
        v[0] += cnt;
        v[1] += cnt > 0;
        v[2] += splits_of(cnt, a.split_edges);
      }
      block_sum3(v, s.scratch);
      if (tid == 0) {
        seg_tot[3 * seg + 0] = static_cast<int32_t>(v[0]);
        seg_tot[3 * seg + 1] = static_cast<int32_t>(v[1]);
        seg_tot[3 * seg + 2] = static_cast<int32_t>(v[2]);
      }
    }
    __syncthreads();
  }
  // Segments without entries have no chunk: their totals are zero.
  for (int64_t sg = kSmall ? nseg : gtid; sg < nseg; sg += gthreads) {
    const int b = static_cast<int>(sg % batch);
    if (chunk_base[b + 1] == chunk_base[b]) {
      seg_tot[3 * sg + 0] = 0;
      seg_tot[3 * sg + 1] = 0;
      seg_tot[3 * sg + 2] = 0;
    }
  }

  __threadfence();
  // The last CTA to finish phase 1 turns the segment totals into exclusive
  // prefixes (edges, non-empty bins, splits) for everyone.
  // Each thread takes a run of consecutive segments: all their totals are
  // loaded at once (held in registers for up to kKeep segments a thread), one
  // block scan, then the run's prefixes.
  auto scan_segments = [&]() {
    constexpr int kKeep = 4;
    const int per = (nseg + kThreads - 1) / kThreads;
    const int lo = min(tid * per, nseg);
    const int hi = min(lo + per, nseg);
    const volatile int32_t* tot_v = seg_tot;
    int32_t keep[kKeep][3];
    int64_t v[3] = {0, 0, 0};
    if (per <= kKeep) {
#pragma unroll
      for (int u = 0; u < kKeep; ++u)
#pragma unroll
        for (int j = 0; j < 3; ++j) keep[u][j] = lo + u < hi ? tot_v[3 * (lo + u) + j] : 0;
#pragma unroll
      for (int u = 0; u < kKeep; ++u)
#pragma unroll
        for (int j = 0; j < 3; ++j) v[j] += keep[u][j];
    } else {
      for (int q = lo; q < hi; ++q)
#pragma unroll
        for (int j = 0; j < 3; ++j) v[j] += tot_v[3 * q + j];
    }
    int64_t excl[3], tot[3];
    block_scan3(v, excl, tot, s.scratch);
    if (per <= kKeep) {
#pragma unroll
      for (int u = 0; u < kKeep; ++u)
        if (lo + u < hi)
#pragma unroll
          for (int j = 0; j < 3; ++j) {
            seg_pre[3 * (lo + u) + j] = excl[j];
            excl[j] += keep[u][j];
          }
    } else {
      for (int q = lo; q < hi; ++q)
#pragma unroll
        for (int j = 0; j < 3; ++j) {
          seg_pre[3 * q + j] = excl[j];
          excl[j] += tot_v[3 * q + j];
        }
    }
    if (tid == 0)
#pragma unroll
      for (int j = 0; j < 3; ++j) seg_pre[3 * nseg + j] = tot[j];
    __threadfence();
  };
  const uint32_t limit = a.spin_limit ? a.spin_limit : kSpinLimit;
  // head_start[h][j]: exclusive prefix of (edges, non-empty bins, splits) at
  // head h's first segment, [hkv] the grand totals (warp-per-segment mode)
  int64_t* head_start = head_tot + 2 * a.hkv;
  if constexpr (kSmall) {
    if (!grid_arrive_wait(bar_count, gridDim.x, limit, a.stall != 0)) {
      if (tid == 0) report(status, SA_ERR_DEVICE_TIMEOUT);
      return;
    }
    // Every CTA scans the segment totals itself (each thread loads its run
    // of segments at once, one block scan) and keeps the prefixes it needs:
    // its warps' segments and the heads' first segments.
    constexpr int kKeep = 4;
    const int per = (nseg + kThreads - 1) / kThreads;
    const int lo = min(tid * per, nseg);
    const int hi = min(lo + per, nseg);
    const volatile int32_t* tot_v = seg_tot;
    int32_t keep[kKeep][3];
    int64_t v[3] = {0, 0, 0};
    if (per <= kKeep) {
#pragma unroll
      for (int u = 0; u < kKeep; ++u)
#pragma unroll
        for (int j = 0; j < 3; ++j) keep[u][j] = lo + u < hi ? tot_v[3 * (lo + u) + j] : 0;
#pragma unroll
      for (int u = 0; u < kKeep; ++u)
#pragma unroll
        for (int j = 0; j < 3; ++j) v[j] += keep[u][j];
    } else {
      for (int q = lo; q < hi; ++q)
#pragma unroll
        for (int j = 0; j < 3; ++j) v[j] += tot_v[3 * q + j];
    }
    int64_t excl[3], tot[3];
    block_scan3(v, excl, tot, s.scratch);
    auto place = [&](int q) {
      if (q % static_cast<int>(gridDim.x) == static_cast<int>(blockIdx.x) &&
          q / static_cast<int>(gridDim.x) < kWarps)
#pragma unroll
        for (int j = 0; j < 3; ++j) s.my_pre[q / gridDim.x][j] = excl[j];
      if (q % batch == 0)
#pragma unroll
        for (int j = 0; j < 3; ++j) head_start[3 * (q / batch) + j] = excl[j];
    };
    if (per <= kKeep) {
#pragma unroll
      for (int u = 0; u < kKeep; ++u)
        if (lo + u < hi) {
          place(lo + u);
#pragma unroll
          for (int j = 0; j < 3; ++j) excl[j] += keep[u][j];
        }
    } else {
      for (int q = lo; q < hi; ++q) {
        place(q);
#pragma unroll
        for (int j = 0; j < 3; ++j) excl[j] += tot_v[3 * q + j];
      }
    }
    if (tid == 0)
#pragma unroll
      for (int j = 0; j < 3; ++j) head_start[3 * a.hkv + j] = tot[j];
    __syncthreads();
    for (int h = tid; h < a.hkv; h += kThreads) {
      head_tot[2 * h + 0] = head_start[3 * (h + 1) + 0] - head_start[3 * h + 0];
      head_tot[2 * h + 1] = head_start[3 * (h + 1) + 1] - head_start[3 * h + 1];
    }
  } else {
    if (!grid_barrier(bar_count, bar_gen, s.gen0, gridDim.x, limit, a.stall != 0,
                      scan_segments)) {
      if (tid == 0) report(status, SA_ERR_DEVICE_TIMEOUT);
      return;
    }
    // Per-head totals of edges and non-empty bins.
    for (int h = tid; h < a.hkv; h += kThreads) {
      const volatile int64_t* lo = seg_pre + 3 * static_cast<int64_t>(h) * batch;
      const volatile int64_t* hi = seg_pre + 3 * static_cast<int64_t>(h + 1) * batch;
      head_tot[2 * h + 0] = hi[0] - lo[0];
      head_tot[2 * h + 1] = hi[1] - lo[1];
    }
  }
  __syncthreads();

  // ---- phase 2: prefixes, slot writes, stable scatter ----------------------
  if (kSmall && my_seg < nseg) {
    // one warp per segment, from the registers of phase 1: entry t goes to
    // edge pre + less + before (blocks ascending, (query, rank) ascending
    // inside a block); the entry that opens a bucket writes its compact slot
    // and its work splits, placed by the buckets of smaller blocks
    const int h = my_seg / batch, b = my_seg - (my_seg / batch) * batch;
    if (__any_sync(0xffffffffu, g.bad) && lane == 0) report(status, SA_ERR_SELECTED_RANGE);
    const int64_t pre0 = s.my_pre[warp][0];
    const int64_t pre1 = s.my_pre[warp][1];
    const int64_t pre2 = s.my_pre[warp][2];
    const int64_t head_edges = head_start[3 * h + 0];
    const int64_t head_units = head_start[3 * h + 1];
    const int64_t nbs = a.nbs;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int t = 32 * k + lane;
      if (t >= g.n) continue;
      const int64_t i = g.q0 + t / topk;
      const int r = t % topk;
      const int64_t inv_at = (static_cast<int64_t>(h) * a.tq + i) * topk + r;
      if (g.blk[k] < 0) {
        a.idx.inv[inv_at] = -1;
        continue;
      }
      const int64_t first = pre0 + g.less[k];             // absolute edge of the bucket
      const int64_t pos = first + g.before[k];
      if (pos >= 0 && pos < cap) {
        reinterpret_cast<int2*>(a.idx.edges)[pos] = make_int2(static_cast<int32_t>(i), r);
        a.idx.inv[inv_at] = static_cast<int32_t>(pos - head_edges);
      }
      if (g.before[k] != 0) continue;
      const int64_t j = pre1 - head_units + g.ul[k];
      if (j >= 0 && j < nbs) {
        a.idx.sel_slots[h * nbs + j] = static_cast<int32_t>(static_cast<int64_t>(b) * msb + g.blk[k]);
        a.idx.sel_offsets[h * (nbs + 1) + j] = static_cast<int32_t>(first - head_edges);
      }
      const int cnt = g.same[k];
      const int step = a.split_edges > 0 ? a.split_edges : cnt;
      const int64_t nsp = splits_of(cnt, a.split_edges);
      for (int64_t u = 0; u < nsp; ++u) {
        const int64_t gs = pre2 + g.sl[k] + u;
        if (gs < cap) {
          const int64_t lo_e = first + u * step;
          int4 w;
          w.x = h;
          w.y = static_cast<int32_t>(j);
          w.z = static_cast<int32_t>(lo_e);
          w.w = static_cast<int32_t>(min(lo_e + step, first + cnt));
          reinterpret_cast<int4*>(a.idx.splits)[gs] = w;
        }
      }
    }
  }
  for (int64_t c = kSmall ? n_chunks : blockIdx.x; c < n_chunks; c += gridDim.x) {
    int h, b, k;
    locate(c, chunk_base, batch, nch_head, h, b, k);
    const int nc = chunk_base[b + 1] - chunk_base[b];
    const int seg = h * batch + b;
    const int64_t q0 = a.cu[b];
    const int64_t n_seg = (a.cu[b + 1] - q0) * topk;
    const int64_t e0 = static_cast<int64_t>(k) * kChunkEntries;
    const int64_t e1 = min(n_seg, e0 + kChunkEntries);
    const int64_t lk = a.used ? (a.used[b] > 0 ? a.used[b] : 0)
                              : static_cast<int64_t>(msb) * a.block_size;
    // Global exclusive prefix of this segment, and its head's base.
    int64_t pre[3];
#pragma unroll
    for (int j = 0; j < 3; ++j) pre[j] = *reinterpret_cast<volatile int64_t*>(seg_pre + 3 * seg + j);
    const int64_t head_edges =
        *reinterpret_cast<volatile int64_t*>(seg_pre + 3 * static_cast<int64_t>(h) * batch + 0);
    const int64_t head_units =
        *reinterpret_cast<volatile int64_t*>(seg_pre + 3 * static_cast<int64_t>(h) * batch + 1);
    // This chunk's bins (validating ids) and the counts of earlier chunks.
    for (int t = tid; t < msb; t += kThreads) {
      bins[t] = 0;
      before[t] = 0;
    }
    __syncthreads();
    for (int64_t e = e0 + tid; e < e1; e += kThreads) {
      const int64_t i = q0 + e / topk;
      const int r = static_cast<int>(e % topk);
      const int blk = sel[(i * a.hkv + h) * topk + r];
      if (blk < -1 || blk >= msb) {
        report(status, SA_ERR_SELECTED_RANGE);
        continue;
      }
      if (blk >= 0 && static_cast<int64_t>(blk) * a.block_size < lk) atomicAdd(&bins[blk], 1);
    }
    __syncthreads();
    if (nc > 1) {
      // Segment totals per bin (into `start` for the scan) and the counts of
      // the segment's earlier chunks (into `before`).
      const int32_t* first = hist + (static_cast<int64_t>(h) * nmulti + multi_base[b]) * msb;
      for (int t = tid; t < msb; t += kThreads) {
        int32_t sum = 0, bef = 0;
        for (int kk = 0; kk < nc; ++kk) {
          const int32_t x = first[static_cast<int64_t>(kk) * msb + t];
          sum += x;
          if (kk < k) bef += x;
        }
        start[t] = sum;
        before[t] = bef;
      }
    } else {
      for (int t = tid; t < msb; t += kThreads) start[t] = bins[t];
    }
    __syncthreads();
    // Scan of the segment's bins; slot outputs from the segment's first chunk.
    const int per = (msb + kThreads - 1) / kThreads;
    const int lo = min(tid * per, msb);
    const int hi = min(lo + per, msb);
    int64_t v[3] = {0, 0, 0};
    for (int t = lo; t < hi; ++t) {
      const int cnt = start[t];
      v[0] += cnt;
      v[1] += cnt > 0;
      v[2] += splits_of(cnt, a.split_edges);
    }
    int64_t excl[3], tot[3];
    block_scan3(v, excl, tot, s.scratch);
    {
      int64_t ge = pre[0] + excl[0];
      int64_t gu = pre[1] + excl[1];
      int64_t gs = pre[2] + excl[2];
      const int64_t nbs = a.nbs;
      for (int t = lo; t < hi; ++t) {
        const int cnt = start[t];
        if (k == 0 && cnt > 0) {
          const int64_t j = gu - head_units;
          if (j >= 0 && j < nbs) {
            a.idx.sel_slots[h * nbs + j] = static_cast<int32_t>(static_cast<int64_t>(b) * msb + t);
            a.idx.sel_offsets[h * (nbs + 1) + j] = static_cast<int32_t>(ge - head_edges);
          }
          const int step = a.split_edges > 0 ? a.split_edges : cnt;
          const int64_t nsp = splits_of(cnt, a.split_edges);
          for (int64_t u = 0; u < nsp; ++u) {
            const int64_t g = gs + u;
            if (g < cap) {
              const int64_t lo_e = ge + u * step;
              int4 w;
              w.x = h;
              w.y = static_cast<int32_t>(j);
              w.z = static_cast<int32_t>(lo_e);
              w.w = static_cast<int32_t>(min(lo_e + step, ge + cnt));
              reinterpret_cast<int4*>(a.idx.splits)[g] = w;
            }
          }
        }
        gs += splits_of(cnt, a.split_edges);
        gu += cnt > 0;
        before[t] = static_cast<int32_t>(ge) + before[t];   // first edge of this chunk's entries
        ge += cnt;
      }
    }
    __syncthreads();
    for (int t = tid; t < msb; t += kThreads) bins[t] = 0;
    __syncthreads();
    for (int64_t base = e0; base < e1; base += kThreads) {
      const int64_t e = base + tid;
      int key = -1;
      int64_t i = 0;
      int r = 0;
      if (e < e1) {
        i = q0 + e / topk;
        r = static_cast<int>(e % topk);
        const int blk = sel[(i * a.hkv + h) * topk + r];
        if (blk >= 0 && blk < msb && static_cast<int64_t>(blk) * a.block_size < lk) key = blk;
      }
      const unsigned peers = __match_any_sync(0xffffffffu, key);
      const int leader = __ffs(peers) - 1;
      const int wrank = __popc(peers & ((1u << lane) - 1u));
      int gbase = 0;
      // Warps take their running bin counts in warp order; warps past the
      // chunk's last entry have nothing to take.
      const int64_t left = e1 - base;
      const int active = left >= kThreads ? kWarps : static_cast<int>((left + 31) >> 5);
      for (int w = 0; w < active; ++w) {
        if (warp == w && key >= 0 && lane == leader) {
          gbase = bins[key];
          bins[key] = gbase + __popc(peers);
        }
        __syncthreads();
      }
      gbase = __shfl_sync(0xffffffffu, gbase, leader);
      if (e < e1) {
        const int64_t inv_at = (static_cast<int64_t>(h) * a.tq + i) * topk + r;
        if (key >= 0) {
          const int64_t pos = static_cast<int64_t>(before[key]) + gbase + wrank;
          if (pos >= 0 && pos < cap) {
            reinterpret_cast<int2*>(a.idx.edges)[pos] = make_int2(static_cast<int32_t>(i), r);
            a.idx.inv[inv_at] = static_cast<int32_t>(pos - head_edges);
          }
        } else {
          a.idx.inv[inv_at] = -1;
        }
      }
    }
    __syncthreads();
  }

  // ---- head-level outputs and the plateau -----------------------------------
  if (blockIdx.x == 0) {
    for (int h = tid; h <= a.hkv; h += kThreads) {
      a.idx.edge_head_base[h] =
          kSmall ? head_start[3 * h]
                 : *reinterpret_cast<volatile int64_t*>(seg_pre + 3 * static_cast<int64_t>(h) * batch);
      if (h < a.hkv) a.idx.num_sel[h] = static_cast<int32_t>(head_tot[2 * h + 1]);
    }
    if (tid == 0) {
      // totals: E, work splits, non-empty units (the prefixes hold edges,
      // units, splits)
      const volatile int64_t* all = seg_pre + 3 * static_cast<int64_t>(nseg);
      a.idx.totals[0] = kSmall ? head_start[3 * a.hkv + 0] : all[0];
      a.idx.totals[1] = kSmall ? head_start[3 * a.hkv + 2] : all[2];
      a.idx.totals[2] = kSmall ? head_start[3 * a.hkv + 1] : all[1];
    }
  }
  // Past each head's kept slots: sel_offsets (through index nbs) holds E_h,
  // sel_slots -1.
  for (int h = 0; h < a.hkv; ++h) {
    const int64_t kept = head_tot[2 * h + 1];
    fill_i32(a.idx.sel_offsets + static_cast<int64_t>(h) * (a.nbs + 1) + kept, a.nbs + 1 - kept,
             static_cast<int32_t>(head_tot[2 * h + 0]), gtid, gthreads);
    fill_i32(a.idx.sel_slots + static_cast<int64_t>(h) * a.nbs + kept, a.nbs - kept, -1, gtid,
             gthreads);
  }
}

size_t index_smem_bytes(int msb, int batch, int hkv) {
  return 16 * static_cast<size_t>(hkv) +
         4 * (3 * static_cast<size_t>(msb > 0 ? msb : 1) + 2 * (static_cast<size_t>(batch) + 1));
}

}  // namespace

int64_t index_chunks_per_head(const int64_t* cu_host, int32_t batch, int32_t topk,
                              int64_t* multi_slots) {
  int64_t c = 0, m = 0;
  for (int32_t b = 0; b < batch; ++b) {
    const int64_t n = (cu_host[b + 1] - cu_host[b]) * topk;
    const int64_t nc = (n + kChunkEntries - 1) / kChunkEntries;
    c += nc;
    if (nc > 1) m += nc;
  }
  if (multi_slots) *multi_slots = m;
  return c;
}

int64_t index_hist_slot_bound(int64_t tq, int32_t topk) {
  // Per head: a segment with more than one chunk has n > kChunkEntries entries
  // and ceil(n / kChunkEntries) < 2 n / kChunkEntries chunks.
  return 2 * (tq * topk) / kChunkEntries + 1;
}

WorkspaceLayout workspace_layout(int32_t hkv, int32_t batch, int64_t tq,
                                 int64_t hist_slots_per_head, int32_t msb) {
  WorkspaceLayout L{};
  const size_t nseg = static_cast<size_t>(hkv) * batch;
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  L.barrier = 0;
  L.unit_ctr = 64;
  L.seg_done = 256;
  L.item_cnt = up(L.seg_done + 4 * nseg);
  L.seg_tot = up(L.item_cnt + 4 * static_cast<size_t>(hkv) * static_cast<size_t>(tq));
  L.zero_bytes = L.seg_tot;                       // barrier and counters
  L.seg_pre = up(L.seg_tot + 12 * nseg);
  L.hist = up(L.seg_pre + 24 * (nseg + 1));
  L.total = up(L.hist + 4 * static_cast<size_t>(hkv) * static_cast<size_t>(hist_slots_per_head) *
                            static_cast<size_t>(msb > 0 ? msb : 1));
  return L;
}

LptRegion lpt_region(int64_t tq, int32_t hkv, int32_t topk, int32_t batch, int32_t msb,
                     int64_t nbs) {
  const size_t build = workspace_layout(hkv, batch, tq, index_hist_slot_bound(tq, topk), msb).total;
  const int64_t entries = tq * hkv * static_cast<int64_t>(topk);
  const int64_t slots = static_cast<int64_t>(hkv) * nbs;
  const int64_t units = entries < slots ? entries : slots;
  LptRegion r;
  r.units = units > 0 ? units : 1;
  r.offset = (build + 255) & ~static_cast<size_t>(255);
  r.counts = (4 * static_cast<size_t>(r.units) + 255) & ~static_cast<size_t>(255);
  const size_t chunks = (static_cast<size_t>(r.units) + 1023) / 1024;
  r.bytes = r.counts + ((64 * chunks + 255) & ~static_cast<size_t>(255));
  return r;
}

namespace {
// The workspace counters and the status word cleared in one launch (for a
// build that runs beside a fused decode kernel: both start from them).
__global__ void __launch_bounds__(256) clear_kernel(uint4* ws, int64_t n16, int64_t* status) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x;
  if (i < n16) ws[i] = make_uint4(0u, 0u, 0u, 0u);
  if (i == 0) *status = 0;
}
}  // namespace

cudaError_t launch_clear_for_build(void* workspace, size_t bytes, int64_t* status,
                                   cudaStream_t stream) {
  const int64_t n16 = static_cast<int64_t>(bytes / 16);
  const int64_t grid = (n16 + 255) / 256;
  clear_kernel<<<static_cast<unsigned>(grid > 0 ? grid : 1), 256, 0, stream>>>(
      static_cast<uint4*>(workspace), n16, status);
  return cudaGetLastError();
}

cudaError_t launch_build_index(const IndexArgs& a, int64_t chunks_per_head,
                               int64_t hist_slots_per_head, cudaStream_t stream) {
  const WorkspaceLayout lay =
      workspace_layout(a.hkv, a.batch, a.tq, hist_slots_per_head, a.msb);
  cudaError_t err = cudaSuccess;
  if (!a.external_clear) {
    err = cudaMemsetAsync(a.idx.workspace, 0, lay.zero_bytes, stream);
    if (err != cudaSuccess) return err;
  }
  IndexArgs args = a;
  const int sms = device_sm_count();
  // warp-per-segment mode: a warp for every segment in one launch, one CTA
  // per SM at most (a smaller barrier); its shared memory is the per-head
  // totals only
  const int64_t seg_ctas = (static_cast<int64_t>(a.hkv) * a.batch + kWarps - 1) / kWarps;
  int per_sm = 0;
  size_t smem = 16 * static_cast<size_t>(a.hkv) + 24 * (static_cast<size_t>(a.hkv) + 1);
  if (args.small) {
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, index_kernel<true>, kThreads, smem);
    if (err != cudaSuccess) return err;
    if (seg_ctas > static_cast<int64_t>(per_sm) * sms) args.small = 0;
  }
  const void* fn = reinterpret_cast<const void*>(index_kernel<true>);
  int64_t grid = 0;
  int64_t nch = 0;
  if (args.small) {
    grid = std::max<int64_t>(seg_ctas, std::min<int64_t>(seg_ctas * kWarps, sms));
  } else {
    fn = reinterpret_cast<const void*>(index_kernel<false>);
    smem = index_smem_bytes(a.msb, a.batch, a.hkv);
    if (smem > 227 * 1024) return cudaErrorNotSupported;
    if (smem > 48 * 1024) {
      err = cudaFuncSetAttribute(index_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem));
      if (err != cudaSuccess) return err;
    }
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, index_kernel<false>, kThreads, smem);
    if (err != cudaSuccess) return err;
    if (per_sm < 1) return cudaErrorNotSupported;
    nch = chunks_per_head * a.hkv;
    const int64_t plateau_ctas =
        (static_cast<int64_t>(a.hkv) * (a.nbs + 1) + 4 * kThreads - 1) / (4 * kThreads);
    grid = std::min<int64_t>(static_cast<int64_t>(per_sm) * sms,
                             std::max<int64_t>(std::max<int64_t>(nch, plateau_ctas), 1));
  }
  int site = kStallNone;
  debug_stall_setting(&site, &args.spin_limit);
  args.stall = site == kStallIndexBarrier;
  WorkspaceLayout layout = lay;
  void* params[] = {&args, &layout, &nch};
  return cudaLaunchCooperativeKernel(fn, dim3(static_cast<unsigned>(grid)), dim3(kThreads), params,
                                     smem, stream);
}

}  // namespace sa
