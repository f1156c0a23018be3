// Step 3 of KV-outer sparse attention: the log-sum-exp combine named in the
// module doc of forward.rs (alice-llm sparse_attention).  One warp per
// (query, q-head): lanes gather the row's partial positions through inv and
// reduce M = max m_r and L = sum exp(m_r - M) l_r; then the live partials are
// visited in ballot order, eight rows loaded at a time, and each lane
// accumulates four or eight of the head_dim outputs with 16-byte loads.
#include <cstdint>

#include "internal.h"
#include "sa_common.cuh"

namespace sa {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

template <int kChunks>  // float4 chunks per lane (head_dim <= 128 * kChunks)
__global__ void __launch_bounds__(kThreads) combine_kernel(CombineArgs a) {
  const int lane = threadIdx.x & 31;
  const int64_t hq = static_cast<int64_t>(a.hkv) * a.qhead;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  if (row >= a.tq * hq) return;
  const int64_t i = row / hq;
  const int hqa = static_cast<int>(row - i * hq);
  const int h = hqa / a.qhead;
  const int qh = hqa - h * a.qhead;
  const int d = a.head_dim;
  const int nc = d >> 2;
  const int32_t* inv_row = a.inv + (static_cast<int64_t>(h) * a.tq + i) * a.topk;
  const int64_t base = a.edge_head_base[h];

  float big_m = -INFINITY;
  for (int r = lane; r < a.topk; r += 32) {
    const int32_t p = inv_row[r];
    if (p >= 0) big_m = fmaxf(big_m, a.m_partial[(base + p) * a.qhead + qh]);
  }
#pragma unroll
  for (int off = 16; off; off >>= 1) big_m = fmaxf(big_m, __shfl_xor_sync(0xffffffffu, big_m, off));

  float4 acc[kChunks];
#pragma unroll
  for (int c = 0; c < kChunks; ++c) acc[c] = make_float4(0.f, 0.f, 0.f, 0.f);
  float big_l = 0.f;
  if (big_m != -INFINITY) {
    for (int r0 = 0; r0 < a.topk; r0 += 32) {
      const int r = r0 + lane;
      float wgt = 0.f;
      int64_t prow = 0;
      if (r < a.topk) {
        const int32_t p = inv_row[r];
        if (p >= 0) {
          prow = (base + p) * a.qhead + qh;
          const float m = a.m_partial[prow];
          if (m != -INFINITY) {
            wgt = __expf(m - big_m);
            big_l += wgt * a.l_partial[prow];
          }
        }
      }
      unsigned live = __ballot_sync(0xffffffffu, wgt > 0.f);
      // Up to kBatch partial rows are loaded before any is used, so their
      // latencies overlap.
      constexpr int kBatch = 8;
      while (live) {
        float wv[kBatch];
        float4 v[kBatch][kChunks];
#pragma unroll
        for (int t = 0; t < kBatch; ++t) {
          wv[t] = 0.f;
          int64_t pr = 0;
          if (live) {
            const int src = __ffs(live) - 1;
            live &= live - 1;
            wv[t] = __shfl_sync(0xffffffffu, wgt, src);
            pr = __shfl_sync(0xffffffffu, prow, src);
          }
          const float4* orow = reinterpret_cast<const float4*>(a.o_partial + pr * d);
#pragma unroll
          for (int c = 0; c < kChunks; ++c) {
            const int ch = lane + 32 * c;
            v[t][c] = (wv[t] > 0.f && ch < nc) ? orow[ch] : make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
#pragma unroll
        for (int t = 0; t < kBatch; ++t)
#pragma unroll
          for (int c = 0; c < kChunks; ++c) {
            acc[c].x = fmaf(wv[t], v[t][c].x, acc[c].x);
            acc[c].y = fmaf(wv[t], v[t][c].y, acc[c].y);
            acc[c].z = fmaf(wv[t], v[t][c].z, acc[c].z);
            acc[c].w = fmaf(wv[t], v[t][c].w, acc[c].w);
          }
      }
    }
#pragma unroll
    for (int off = 16; off; off >>= 1) big_l += __shfl_xor_sync(0xffffffffu, big_l, off);
  }
  const float inv_l = big_l > 0.f ? 1.f / big_l : 0.f;
  float4* orow = reinterpret_cast<float4*>(a.out + row * d);
#pragma unroll
  for (int c = 0; c < kChunks; ++c) {
    const int ch = lane + 32 * c;
    if (ch < nc)
      orow[ch] = make_float4(acc[c].x * inv_l, acc[c].y * inv_l, acc[c].z * inv_l,
                             acc[c].w * inv_l);
  }
  if (a.lse && lane == 0) a.lse[row] = big_l > 0.f ? big_m + logf(big_l) : -INFINITY;
}

}  // namespace

cudaError_t launch_combine(const CombineArgs& a, cudaStream_t stream) {
  const int64_t rows = a.tq * a.hkv * a.qhead;
  if (rows == 0) return cudaSuccess;
  const int64_t grid = (rows + kWarps - 1) / kWarps;
  if (a.head_dim <= 128)
    combine_kernel<1><<<static_cast<unsigned>(grid), kThreads, 0, stream>>>(a);
  else
    combine_kernel<2><<<static_cast<unsigned>(grid), kThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace sa
