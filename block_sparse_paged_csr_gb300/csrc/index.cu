// Step 1 of KV-outer sparse attention: the CSR index (KvOuterIndex, types.rs
// of alice-llm's sparse_attention) and the forward's work list (WorkSplit).
//
// Structure.  Entries (query i, kv head h, rank r) that belong to one
// (h, sequence b) segment can only land in the raw slots b*msb .. b*msb+msb-1
// of head h, and segments in (h, b) order own consecutive slot ranges.  So one
// CTA per segment:
//   1. histograms its entries into msb shared-memory bins (validating ids);
//   2. scans the bins, publishes its totals and reads the totals of all
//      earlier segments with a decoupled look-back (segments are handed out
//      by an atomic ticket, so every segment it waits on is already running;
//      every wait is bounded);
//   3. writes sel_slots / sel_offsets / the split list for its non-empty bins;
//   4. scatters its edges: entries walk in (query, rank) order, 512 at a time;
//      a warp's equal keys are ranked with __match_any_sync, warps take their
//      running bin counts in warp order, so the order inside every bucket is
//      (query, rank) ascending and the result is deterministic.
// A second small kernel writes the plateau (sel_offsets past num_sel[h]) and
// the -1 padding of sel_slots, which need each head's final totals.
#include <algorithm>
#include <cstdint>

#include "internal.h"
#include "sa_common.cuh"

namespace sa {

namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr uint64_t kFlagAgg = 1ull << 62;
constexpr uint64_t kFlagIncl = 2ull << 62;
constexpr uint64_t kFlagMask = 3ull << 62;
constexpr uint64_t kLow31 = (1ull << 31) - 1;
constexpr uint64_t kLow62 = (1ull << 62) - 1;

__device__ __forceinline__ uint64_t ld_acquire(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release(uint64_t* p, uint64_t v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Segment status: word A = flag | edges, word B = flag | units << 31 | splits.
// B is stored before A, each with release order; a reader accepts a pair only
// when both carry the same flag.
__device__ __forceinline__ void publish(uint64_t* a, uint64_t* b, uint64_t flag, int64_t edges,
                                        int64_t units, int64_t splits) {
  st_release(b, flag | (static_cast<uint64_t>(units) << 31) | static_cast<uint64_t>(splits));
  st_release(a, flag | static_cast<uint64_t>(edges));
}

__device__ __forceinline__ int64_t splits_of(int64_t count, int split_edges) {
  if (count <= 0) return 0;
  if (split_edges <= 0) return 1;
  return (count + split_edges - 1) / split_edges;
}

// Exclusive block scan of three values; also returns the block totals.
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
  if (lane == 31) {
#pragma unroll
    for (int q = 0; q < 3; ++q) warp_tot[q][warp] = inc[q];
  }
  __syncthreads();
  if (warp == 0) {
#pragma unroll
    for (int q = 0; q < 3; ++q) {
      int64_t x = lane < kWarps ? warp_tot[q][lane] : 0;
      int64_t y = x;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int64_t n = __shfl_up_sync(0xffffffffu, y, off);
        if (lane >= off) y += n;
      }
      if (lane < kWarps) warp_tot[q][lane] = y - x;   // exclusive over warps
      const int64_t all = __shfl_sync(0xffffffffu, y, 31);
      if (lane == 0) tot[q] = all;
    }
  }
  __syncthreads();
#pragma unroll
  for (int q = 0; q < 3; ++q) excl[q] = warp_tot[q][warp] + inc[q] - v[q];
}

struct SegShared {
  int64_t warp_tot[3][kWarps];
  int64_t tot[3];
  int64_t prefix[3];      // global exclusive prefix: edges, units, splits
  int64_t head_edges;     // global edge index of the head's first edge
  int64_t head_units;     // global unit index of the head's first unit
  int seg;
};

__global__ void __launch_bounds__(kThreads)
index_segments_kernel(IndexArgs a, WorkspaceLayout lay, int nseg) {
  extern __shared__ int32_t dyn[];
  int32_t* bins = dyn;                // [msb] counts, later running counters
  int32_t* start = dyn + a.msb;       // [msb] global edge index of each bin's first edge
  __shared__ SegShared s;

  char* ws = static_cast<char*>(a.idx.workspace);
  uint32_t* ticket = reinterpret_cast<uint32_t*>(ws + lay.ticket);
  uint64_t* seg_a = reinterpret_cast<uint64_t*>(ws + lay.seg_a);
  uint64_t* seg_b = reinterpret_cast<uint64_t*>(ws + lay.seg_b);
  int32_t* head_units = reinterpret_cast<int32_t*>(ws + lay.head_units);
  int64_t* status = a.idx.totals + 3;

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  if (tid == 0) s.seg = static_cast<int>(atomicAdd(ticket, 1u));
  __syncthreads();
  const int seg = s.seg;
  if (seg >= nseg) return;  // cannot happen: the grid has exactly nseg CTAs
  const int h = seg / a.batch;
  const int b = seg % a.batch;
  const int msb = a.msb;
  const int topk = a.topk;
  const int64_t q0 = a.cu[b];
  const int64_t qo = a.cu[b + 1] - q0;
  const int64_t lk = a.used ? (a.used[b] > 0 ? a.used[b] : 0)
                            : static_cast<int64_t>(msb) * a.block_size;
  const int64_t n_seg = qo > 0 ? qo * topk : 0;
  const int32_t* sel = a.selected;

  // ---- 1. histogram -------------------------------------------------------
  for (int k = tid; k < msb; k += kThreads) bins[k] = 0;
  __syncthreads();
  for (int64_t e = tid; e < n_seg; e += kThreads) {
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

  // ---- 2. local scan + look-back -------------------------------------------
  const int per = (msb + kThreads - 1) / kThreads;
  const int lo = min(tid * per, msb);
  const int hi = min(lo + per, msb);
  int64_t v[3] = {0, 0, 0};
  for (int k = lo; k < hi; ++k) {
    const int c = bins[k];
    v[0] += c;
    v[1] += c > 0;
    v[2] += splits_of(c, a.split_edges);
  }
  int64_t excl[3];
  block_scan3(v, excl, s.tot, s.warp_tot);

  if (warp == 0) {
    // Decoupled look-back, 32 predecessors per step: lane j reads segment
    // (window end - j); the nearest one with an inclusive prefix ends the walk.
    if (lane == 0) publish(seg_a + seg, seg_b + seg, kFlagAgg, s.tot[0], s.tot[1], s.tot[2]);
    __syncwarp();
    int64_t pe = 0, pu = 0, ps = 0;
    bool ok = true;
    for (int hi_k = seg - 1; hi_k >= 0; hi_k -= 32) {
      const int k = hi_k - lane;
      uint64_t wa = 0, wb = 0;
      bool mine_ok = true;
      if (k >= 0) {
        uint32_t it = 0;
        for (;;) {
          wa = ld_acquire(seg_a + k);
          if (wa & kFlagMask) {
            wb = ld_acquire(seg_b + k);
            if ((wb & kFlagMask) == (wa & kFlagMask)) break;
          }
          if (++it > kSpinLimit) {
            mine_ok = false;
            break;
          }
          __nanosleep(32);
        }
      }
      if (!__all_sync(0xffffffffu, mine_ok)) {
        ok = false;
        break;
      }
      const unsigned incl =
          __ballot_sync(0xffffffffu, k >= 0 && (wa & kFlagMask) == kFlagIncl);
      const int stop = incl ? __ffs(incl) - 1 : 31;
      int64_t ce = 0, cu_ = 0, cs = 0;
      if (k >= 0 && lane <= stop) {
        ce = static_cast<int64_t>(wa & kLow62);
        cu_ = static_cast<int64_t>((wb >> 31) & kLow31);
        cs = static_cast<int64_t>(wb & kLow31);
      }
#pragma unroll
      for (int off = 16; off; off >>= 1) {
        ce += __shfl_xor_sync(0xffffffffu, ce, off);
        cu_ += __shfl_xor_sync(0xffffffffu, cu_, off);
        cs += __shfl_xor_sync(0xffffffffu, cs, off);
      }
      pe += ce;
      pu += cu_;
      ps += cs;
      if (incl) break;
    }
    if (lane == 0) {
      if (!ok) report(status, SA_ERR_DEVICE_TIMEOUT);
      s.prefix[0] = pe;
      s.prefix[1] = pu;
      s.prefix[2] = ps;
      if (b == 0) {
        // This segment opens head h: publish the head's bases before the
        // inclusive flag so that later segments of the head can read them.
        a.idx.edge_head_base[h] = pe;
        head_units[h] = static_cast<int32_t>(pu);
        s.head_edges = pe;
        s.head_units = pu;
      }
      publish(seg_a + seg, seg_b + seg, kFlagIncl, pe + s.tot[0], pu + s.tot[1], ps + s.tot[2]);
      if (b != 0) {
        const int first = seg - b;
        uint32_t it = 0;
        while ((ld_acquire(seg_a + first) & kFlagMask) != kFlagIncl) {
          if (++it > kSpinLimit) {
            report(status, SA_ERR_DEVICE_TIMEOUT);
            break;
          }
          __nanosleep(32);
        }
        s.head_edges = *reinterpret_cast<volatile int64_t*>(a.idx.edge_head_base + h);
        s.head_units = *reinterpret_cast<volatile int32_t*>(head_units + h);
      }
      if (b == a.batch - 1) a.idx.num_sel[h] = static_cast<int32_t>(pu + s.tot[1] - s.head_units);
      if (seg == nseg - 1) {
        a.idx.edge_head_base[a.hkv] = pe + s.tot[0];
        a.idx.totals[0] = pe + s.tot[0];
        a.idx.totals[1] = ps + s.tot[2];
        a.idx.totals[2] = pu + s.tot[1];
      }
    }
  }
  __syncthreads();

  // ---- 3. compact slots and work splits ------------------------------------
  const int64_t cap = static_cast<int64_t>(a.tq) * a.hkv * topk;  // edges / splits capacity
  {
    int64_t ge = s.prefix[0] + excl[0];
    int64_t gu = s.prefix[1] + excl[1];
    int64_t gs = s.prefix[2] + excl[2];
    const int64_t nbs = a.nbs;
    for (int k = lo; k < hi; ++k) {
      const int c = bins[k];
      start[k] = static_cast<int32_t>(ge);
      if (c > 0) {
        const int64_t j = gu - s.head_units;
        if (j >= 0 && j < nbs) {
          a.idx.sel_slots[h * nbs + j] = static_cast<int32_t>(static_cast<int64_t>(b) * msb + k);
          a.idx.sel_offsets[h * (nbs + 1) + j] = static_cast<int32_t>(ge - s.head_edges);
        }
        const int step = a.split_edges > 0 ? a.split_edges : c;
        const int64_t nsp = splits_of(c, a.split_edges);
        for (int64_t t = 0; t < nsp; ++t) {
          const int64_t g = gs + t;
          if (g < cap) {
            const int64_t e_lo = ge + t * step;
            const int64_t e_hi = min(e_lo + step, ge + c);
            int4 w;
            w.x = h;
            w.y = static_cast<int32_t>(j);
            w.z = static_cast<int32_t>(e_lo);
            w.w = static_cast<int32_t>(e_hi);
            reinterpret_cast<int4*>(a.idx.splits)[g] = w;
          }
        }
        gs += nsp;
        gu += 1;
      }
      ge += c;
    }
  }
  __syncthreads();
  for (int k = tid; k < msb; k += kThreads) bins[k] = 0;
  __syncthreads();

  // ---- 4. stable scatter of edges and inv ----------------------------------
  const int64_t head_edges = s.head_edges;
  for (int64_t base = 0; base < n_seg; base += kThreads) {
    const int64_t e = base + tid;
    int key = -1;
    int64_t i = 0;
    int r = 0;
    if (e < n_seg) {
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
    const int64_t left = n_seg - base;
    const int active_warps = left >= kThreads ? kWarps : static_cast<int>((left + 31) >> 5);
    for (int w = 0; w < active_warps; ++w) {
      if (warp == w && key >= 0 && lane == leader) {
        gbase = bins[key];
        bins[key] = gbase + __popc(peers);
      }
      __syncthreads();
    }
    gbase = __shfl_sync(0xffffffffu, gbase, leader);
    if (e < n_seg) {
      const int64_t inv_at = (static_cast<int64_t>(h) * a.tq + i) * topk + r;
      if (key >= 0) {
        const int64_t pos = static_cast<int64_t>(start[key]) + gbase + wrank;
        if (pos >= 0 && pos < cap) {
          reinterpret_cast<int2*>(a.idx.edges)[pos] = make_int2(static_cast<int32_t>(i), r);
          a.idx.inv[inv_at] = static_cast<int32_t>(pos - head_edges);
        }
      } else {
        a.idx.inv[inv_at] = -1;
      }
    }
  }
}

// sel_offsets[h, p] = head total and sel_slots[h, p] = -1 for p >= num_sel[h].
__global__ void index_plateau_kernel(int32_t* __restrict__ sel_slots,
                                     int32_t* __restrict__ sel_offsets,
                                     const int32_t* __restrict__ num_sel,
                                     const int64_t* __restrict__ edge_head_base, int64_t nbs) {
  const int h = blockIdx.y;
  const int64_t ns_raw = num_sel[h] > 0 ? num_sel[h] : 0;
  const int64_t ns = ns_raw < nbs + 1 ? ns_raw : nbs + 1;
  const int32_t total = static_cast<int32_t>(edge_head_base[h + 1] - edge_head_base[h]);
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t p = ns + static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; p <= nbs;
       p += stride) {
    sel_offsets[h * (nbs + 1) + p] = total;
    if (p < nbs) sel_slots[h * nbs + p] = -1;
  }
}

}  // namespace

WorkspaceLayout workspace_layout(int32_t hkv, int32_t batch) {
  WorkspaceLayout L{};
  const size_t nseg = static_cast<size_t>(hkv) * batch;
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  L.ticket = 0;
  L.seg_a = 256;
  L.seg_b = up(L.seg_a + 8 * nseg);
  L.head_units = up(L.seg_b + 8 * nseg);
  L.zero_bytes = L.head_units;
  L.total = up(L.head_units + 4 * static_cast<size_t>(hkv));
  return L;
}

cudaError_t launch_build_index(const IndexArgs& a, cudaStream_t stream) {
  const WorkspaceLayout lay = workspace_layout(a.hkv, a.batch);
  cudaError_t err = cudaMemsetAsync(a.idx.workspace, 0, lay.zero_bytes, stream);
  if (err != cudaSuccess) return err;
  err = cudaMemsetAsync(a.idx.totals, 0, 4 * sizeof(int64_t), stream);
  if (err != cudaSuccess) return err;
  const size_t smem = 2 * sizeof(int32_t) * static_cast<size_t>(a.msb > 0 ? a.msb : 1);
  if (smem > 48 * 1024) {
    err = cudaFuncSetAttribute(index_segments_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(smem));
    if (err != cudaSuccess) return err;
  }
  const int nseg = a.hkv * a.batch;
  index_segments_kernel<<<nseg, kThreads, smem, stream>>>(a, lay, nseg);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  const int64_t per_head = a.nbs + 1;
  int gx = static_cast<int>(std::min<int64_t>((per_head + 255) / 256,
                                              std::max(1, device_sm_count() * 4 / a.hkv + 1)));
  if (gx < 1) gx = 1;
  index_plateau_kernel<<<dim3(gx, a.hkv), 256, 0, stream>>>(
      a.idx.sel_slots, a.idx.sel_offsets, a.idx.num_sel, a.idx.edge_head_base, a.nbs);
  return cudaGetLastError();
}

}  // namespace sa
