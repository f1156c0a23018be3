// Step 2 of KV-outer sparse attention for decode-shaped work (few rows per
// work split, head_dim 128): per-edge partials as in process_work_unit
// (forward.rs of alice-llm's sparse_attention), pipelined per warp.
//
// Every warp is an independent pipeline over its own work splits (a static
// stride over the split list).  It streams each split's block in chunks of
// 16 keys: the chunk's rows of K and V (parts of one or more pages, each a
// contiguous run) are fetched with 1-D bulk copies into a ring of NST stages
// in the warp's own shared memory, completion on the stage's mbarrier; the
// Q rows of the split arrive with its first chunk.  While the warp computes
// one chunk the next NST-1 are in flight.
//
// Per chunk:
//   scores  lane = (key, half of head_dim): a 64-dim partial dot for every
//           row, the two halves added with one shuffle; shared reads rotate
//           their 16-byte column by key so the warp hits all banks;
//   softmax online over the chunks, in the log2 domain (row max by a 4-step
//           butterfly over the 16 key lanes);
//   PV      lane = 4 output dims, p broadcast from its key lane.
// The metadata of 32 splits (split entry, raw slot, block table entries,
// first query ids) is read one split per lane, so its dependent loads cost
// one round trip chain per 32 splits.
#include <cstdint>

#include "dec_common.cuh"
#include "internal.h"
#include "sa_common.cuh"

namespace sa {

namespace {

using dec::kMaxPages;
using dec::kMaxQi;
using dec::SplitMeta;
using dec::load_meta;
using dec::bcast_meta;

constexpr int kD = 128;
constexpr int kKC = 16;            // keys per chunk
constexpr int kQBufs = 3;          // Q buffers per warp (row groups in flight)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__host__ __device__ inline size_t up128(size_t x) { return (x + 127) & ~static_cast<size_t>(127); }

struct WarpPlan {
  size_t chunk_bytes;   // K or V of one chunk
  size_t stage_bytes;   // K + V
  size_t q_bytes;       // one Q buffer
  size_t warp_bytes;    // all of one warp's shared memory (128-aligned)
};

__host__ __device__ inline WarpPlan warp_plan(int rows, int kv_bf16, int nst) {
  WarpPlan p{};
  p.chunk_bytes = static_cast<size_t>(kKC) * kD * (kv_bf16 ? 2 : 4);
  p.stage_bytes = 2 * p.chunk_bytes;
  p.q_bytes = static_cast<size_t>(rows) * kD * 4;
  p.warp_bytes = up128(nst * p.stage_bytes + kQBufs * p.q_bytes + 8 * nst);
  return p;
}

template <bool kBf16>
__device__ __forceinline__ float4 ld_row4(const unsigned char* tile, int key, int dim) {
  if constexpr (kBf16) {
    return bf16x4_to_f32(*reinterpret_cast<const uint2*>(tile + (key * kD + dim) * 2));
  } else {
    return *reinterpret_cast<const float4*>(tile + (key * kD + dim) * 4);
  }
}

__device__ __forceinline__ float dot4(const float4 a, const float4 b) {
  return fmaf(a.x, b.x, fmaf(a.y, b.y, fmaf(a.z, b.z, a.w * b.w)));
}

template <int R, bool kBf16, int NST, int WARPS>
__global__ void __launch_bounds__(WARPS * 32, 1)
forward_dec_kernel(ForwardArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  const WarpPlan plan = warp_plan(R, kBf16 ? 1 : 0, NST);
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  unsigned char* base = smem + warp * plan.warp_bytes;
  unsigned char* stages = base;
  float* qbuf = reinterpret_cast<float*>(base + NST * plan.stage_bytes);     // [kQBufs][R][128]
  uint64_t* bars =
      reinterpret_cast<uint64_t*>(base + NST * plan.stage_bytes + kQBufs * plan.q_bytes);

  const int qhead = a.qhead;
  const int ps = a.page_size;
  const int cps = a.block_size / kKC;                  // chunks per block
  const int staged_edges = R / qhead;
  const size_t elt = kBf16 ? 2 : 4;
  const size_t row_bytes = kD * elt;
  int64_t* status = a.totals + 3;
  const int64_t n_splits = min(a.totals[1], a.max_splits);
  const int64_t tw = static_cast<int64_t>(gridDim.x) * WARPS;
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * WARPS + warp;
  const float qscale = a.scale * kLog2e;

  if (lane == 0) {
    for (int s = 0; s < NST; ++s) mbar_init(bars + s, 1);
    fence_mbar_init();
  }
  // Rows that are never copied are multiplied by p = 0: keep them finite.
  for (size_t off = 16u * lane; off < NST * plan.stage_bytes; off += 16u * 32)
    *reinterpret_cast<float4*>(stages + off) = make_float4(0.f, 0.f, 0.f, 0.f);
  fence_proxy_async_smem();
  __syncwarp();

  uint32_t chunks_issued = 0;   // stream position of the issue cursor
  uint32_t chunks_done = 0;     // stream position of the compute cursor
  uint32_t groups_issued = 0;   // row groups whose Q the issue cursor has fetched
  uint32_t groups_done = 0;     // row groups the compute cursor has finished
  bool ok = true;

  for (int64_t batch0 = 0; ok; batch0 += 32) {
    if (gw + batch0 * tw >= n_splits) break;
    SplitMeta mine;
    load_meta(a, gw + (batch0 + lane) * tw, n_splits, staged_edges, mine);
    const int64_t left = (n_splits - gw - batch0 * tw + tw - 1) / tw;
    const int nb = static_cast<int>(left < 32 ? left : 32);

    // Issue cursor over (split j of the batch, row group g, chunk c).
    int is_j = 0, is_g = 0, is_c = 0;
    SplitMeta im = bcast_meta(mine, 0);
    auto issue_one = [&]() {
      // Fill stage (chunks_issued % NST) with chunk is_c of row group is_g of
      // split is_j; the Q rows of the group come with its first chunk.
      const int stage = chunks_issued % NST;
      unsigned char* st = stages + stage * plan.stage_bytes;
      const int k0 = is_c * kKC;                      // first key of the chunk in the block
      uint32_t tx = 0;
      // Page pieces of this chunk: lane p < pieces handles piece p.
      const int pieces = ps >= kKC ? 1 : kKC / ps;
      int my_page = -1, my_row0 = 0, my_rows = 0, my_dst = 0;
      if (lane < pieces) {
        const int key = k0 + lane * min(ps, kKC);      // first key of this piece
        const int p = key / ps;
        my_rows = min(ps, kKC);
        my_row0 = key - p * ps;
        my_dst = lane * my_rows;
        const bool live = p < kMaxPages && ((im.pmask >> p) & 1u) && im.bstart + key < im.bend;
        if (live) {
          int id = im.pid[0];
#pragma unroll
          for (int q = 1; q < kMaxPages; ++q)
            if (q == p) id = im.pid[q];
          my_page = id;
        }
      }
      const uint32_t piece_bytes = static_cast<uint32_t>(my_rows * row_bytes);
      const uint32_t kv_tx = my_page >= 0 ? 2u * piece_bytes : 0u;
      tx = kv_tx;
      // Q rows of the group.
      const int rows_g = min(R, im.nrows - is_g * R);
      const int ne = (rows_g + qhead - 1) / qhead;
      int my_qi = -1;
      if (is_c == 0 && lane >= 8 && lane < 8 + ne) {
        const int e = is_g * staged_edges + (lane - 8);
        if (e < kMaxQi) {
          int v = im.qi[0];
#pragma unroll
          for (int q = 1; q < kMaxQi; ++q)
            if (q == e) v = im.qi[q];
          my_qi = v;
        } else {
          my_qi = a.edges[2 * (static_cast<int64_t>(im.edge0) + e)];
        }
        tx += static_cast<uint32_t>(qhead * kD * 4);
      }
#pragma unroll
      for (int off = 16; off; off >>= 1) tx += __shfl_xor_sync(0xffffffffu, tx, off);
      if (lane == 0) mbar_arrive_expect_tx(bars + stage, tx);
      __syncwarp();
      if (my_page >= 0) {
        const size_t src = ((static_cast<size_t>(my_page) * a.hkv + im.h) * ps + my_row0) * row_bytes;
        bulk_g2s(st + my_dst * row_bytes, static_cast<const unsigned char*>(a.k_pages) + src,
                 piece_bytes, bars + stage);
        bulk_g2s(st + plan.chunk_bytes + my_dst * row_bytes,
                 static_cast<const unsigned char*>(a.v_pages) + src, piece_bytes, bars + stage);
      }
      if (my_qi >= 0) {
        const int e_local = lane - 8;
        float* dst = qbuf + static_cast<size_t>(groups_issued % kQBufs) * R * kD +
                     static_cast<size_t>(e_local) * qhead * kD;
        const float* src = a.q + (static_cast<int64_t>(my_qi) * a.hq +
                                  static_cast<int64_t>(im.h) * qhead) * kD;
        bulk_g2s(dst, src, static_cast<uint32_t>(qhead * kD * 4), bars + stage);
      }
      ++chunks_issued;
      // Advance the cursor.
      if (++is_c == cps) {
        is_c = 0;
        ++groups_issued;
        if (++is_g * R >= max(im.nrows, 1)) {
          is_g = 0;
          ++is_j;
          if (is_j < nb) im = bcast_meta(mine, is_j);
        }
      }
    };

    // Prologue: fill the ring.
    while (is_j < nb && chunks_issued - chunks_done < static_cast<uint32_t>(NST)) issue_one();

    for (int j = 0; j < nb && ok; ++j) {
      const SplitMeta m = bcast_meta(mine, j);
      const int ngroups = max((m.nrows + R - 1) / R, 1);
      for (int g = 0; g < ngroups && ok; ++g) {
        const int rows_g = min(R, m.nrows - g * R);
        const float* qg = qbuf + static_cast<size_t>(groups_done % kQBufs) * R * kD;
        // Causal limit of each row of the group.
        int lim[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
          lim[r] = -1;
          if (r < rows_g) {
            const int e = g * staged_edges + r / qhead;
            int64_t qidx;
            if (e < kMaxQi) {
              int v = m.qi[0];
#pragma unroll
              for (int q = 1; q < kMaxQi; ++q)
                if (q == e) v = m.qi[q];
              qidx = v;
            } else {
              qidx = a.edges[2 * (static_cast<int64_t>(m.edge0) + e)];
            }
            int64_t l64 = INT32_MAX;
            if (a.causal) {
              const int64_t ql = qidx - m.q0;
              l64 = a.causal == 2 || m.lk < m.qo ? ql : m.lk - m.qo + ql;
            }
            lim[r] = static_cast<int>(l64 < INT32_MAX ? l64 : INT32_MAX);
          }
        }
        float m_run[R], l_part[R];
        float4 o[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
          m_run[r] = -INFINITY;
          l_part[r] = 0.f;
          o[r] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        const int key = lane & 15;
        const int half = lane >> 4;
        for (int c = 0; c < cps; ++c) {
          const int stage = chunks_done % NST;
          const uint32_t parity = (chunks_done / NST) & 1u;
          const bool got = mbar_wait_bounded(bars + stage, parity);
          if (!__all_sync(0xffffffffu, got)) {
            if (lane == 0) report(status, SA_ERR_DEVICE_TIMEOUT);
            ok = false;
            break;
          }
          const unsigned char* kt = stages + stage * plan.stage_bytes;
          const unsigned char* vt = kt + plan.chunk_bytes;
          const int k0 = c * kKC;
          const int pos = m.bstart + k0 + key;
          const bool page_ok = ((m.pmask >> ((k0 + key) / ps)) & 1u) != 0;
          const bool key_ok = pos < m.bend && page_ok;
          if (__any_sync(0xffffffffu, key_ok)) {
            // Scores: this lane's key, half of the dims, all rows.
            float acc[R];
#pragma unroll
            for (int r = 0; r < R; ++r) acc[r] = 0.f;
#pragma unroll 4
            for (int cc = 0; cc < 16; ++cc) {
              const int dim = half * 64 + ((cc + key) & 15) * 4;
              const float4 kv = ld_row4<kBf16>(kt, key, dim);
#pragma unroll
              for (int r = 0; r < R; ++r)
                acc[r] += dot4(*reinterpret_cast<const float4*>(qg + r * kD + dim), kv);
            }
            float p[R], alpha[R];
#pragma unroll
            for (int r = 0; r < R; ++r) {
              float s = acc[r] + __shfl_xor_sync(0xffffffffu, acc[r], 16);
              s = (key_ok && r < rows_g && pos <= lim[r]) ? s * qscale : -INFINITY;
              float cm = s;
#pragma unroll
              for (int off = 1; off < 16; off <<= 1)
                cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, off));
              const float m_new = fmaxf(m_run[r], cm);
              alpha[r] = m_new == -INFINITY ? 1.f : exp2f(m_run[r] - m_new);
              p[r] = s == -INFINITY ? 0.f : exp2f(s - m_new);
              l_part[r] = l_part[r] * alpha[r] + (half == 0 ? p[r] : 0.f);
              m_run[r] = m_new;
              o[r].x *= alpha[r];
              o[r].y *= alpha[r];
              o[r].z *= alpha[r];
              o[r].w *= alpha[r];
            }
            // o += p V: lane = 4 output dims.
#pragma unroll 4
            for (int t = 0; t < kKC; ++t) {
              const float4 vv = ld_row4<kBf16>(vt, t, lane * 4);
#pragma unroll
              for (int r = 0; r < R; ++r) {
                const float pt = __shfl_sync(0xffffffffu, p[r], t);
                o[r].x = fmaf(pt, vv.x, o[r].x);
                o[r].y = fmaf(pt, vv.y, o[r].y);
                o[r].z = fmaf(pt, vv.z, o[r].z);
                o[r].w = fmaf(pt, vv.w, o[r].w);
              }
            }
          }
          ++chunks_done;
          // The stage is free once every lane has read it.
          __syncwarp();
          fence_proxy_async_smem();
          if (is_j < nb) issue_one();
        }
        if (!ok) break;
        ++groups_done;
        // Finish the group's rows.
        const int64_t row0 = static_cast<int64_t>(m.edge0) * qhead + g * R;
#pragma unroll
        for (int r = 0; r < R; ++r) {
          float l = l_part[r];
#pragma unroll
          for (int off = 1; off < 32; off <<= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
          if (r < rows_g) {
            store_o4(a.o_partial, a.o_bf16, (row0 + r) * kD + 4 * lane, o[r]);
            if (lane == 0) {
              a.m_partial[row0 + r] = m_run[r] == -INFINITY ? -INFINITY : m_run[r] * kLn2;
              a.l_partial[row0 + r] = l;
            }
          }
        }
      }
    }
    if (!ok) {
      // Let copies already in flight land before the warp leaves.
      while (chunks_done < chunks_issued) {
        mbar_wait_bounded(bars + chunks_done % NST, (chunks_done / NST) & 1u);
        ++chunks_done;
      }
    }
  }
}

template <int R, bool kBf16, int NST, int WARPS>
cudaError_t launch_dec(const ForwardArgs& a, cudaStream_t stream) {
  const WarpPlan p = warp_plan(R, a.kv_bf16, NST);
  const size_t smem = p.warp_bytes * WARPS;
  if (smem > 227 * 1024) return cudaErrorNotSupported;
  const void* fn = reinterpret_cast<const void*>(forward_dec_kernel<R, kBf16, NST, WARPS>);
  cudaError_t err =
      cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  err = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
  if (err != cudaSuccess) return err;
  int64_t grid = device_sm_count();
  const int64_t need = (a.max_splits + WARPS - 1) / WARPS;
  if (grid > need) grid = need;
  if (grid < 1) grid = 1;
  forward_dec_kernel<R, kBf16, NST, WARPS>
      <<<static_cast<unsigned>(grid), WARPS * 32, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

bool forward_dec_supported(int head_dim, int block_size, int page_size, int qhead, int kv_bf16) {
  (void)kv_bf16;
  if (head_dim != kD) return false;
  // at least two chunks per block keeps the Q buffers of the ring apart
  if (block_size % kKC != 0 || block_size < 2 * kKC) return false;
  if (page_size <= 0 || block_size % page_size) return false;
  if (block_size / page_size > kMaxPages) return false;
  if (page_size < kKC && kKC % page_size) return false;   // pieces of a chunk tile it exactly
  if (page_size > kKC && page_size % kKC) return false;
  if (qhead != 1 && qhead != 2 && qhead != 4 && qhead != 8) return false;
  return true;
}

cudaError_t launch_forward_dec(const ForwardArgs& a, cudaStream_t stream) {
  if (!forward_dec_supported(a.head_dim, a.block_size, a.page_size, a.qhead, a.kv_bf16))
    return cudaErrorNotSupported;
  if (a.qhead <= 4)
    return a.kv_bf16 ? launch_dec<4, true, 4, 5>(a, stream) : launch_dec<4, false, 3, 4>(a, stream);
  return a.kv_bf16 ? launch_dec<8, true, 3, 6>(a, stream) : launch_dec<8, false, 3, 3>(a, stream);
}

}  // namespace sa
