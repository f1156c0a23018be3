// Step 3 of KV-outer sparse attention: the log-sum-exp combine named in the
// module doc of forward.rs (alice-llm sparse_attention).  One warp per
// (query, q-head): lanes gather the row's partial positions through inv and
// reduce M = max m_r and L = sum exp(m_r - M) l_r; then the live partials are
// visited in ballot order, eight rows loaded at a time, and each lane
// accumulates four or eight of the head_dim outputs with 16-byte loads.  bf16
// o partials (the opt-in 16-bit form) take a half-warp per row so that loads
// stay 16 bytes wide (8-byte loads where head_dim is not a multiple of 8).
#include <cstdint>

#include "internal.h"
#include "sa_common.cuh"

namespace sa {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

// kChunks: groups of four dims per lane (head_dim <= 128 * kChunks); kBf16:
// the o partials are bf16.
template <int kChunks, bool kBf16>
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
#pragma unroll
          for (int c = 0; c < kChunks; ++c) {
            const int ch = lane + 32 * c;
            v[t][c] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (wv[t] > 0.f && ch < nc) {
              if constexpr (kBf16)
                v[t][c] = bf16x4_to_f32(reinterpret_cast<const uint2*>(
                    static_cast<const uint16_t*>(a.o_partial) + pr * d)[ch]);
              else
                v[t][c] = reinterpret_cast<const float4*>(
                    static_cast<const float*>(a.o_partial) + pr * d)[ch];
            }
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

// bf16 o partials with head_dim a multiple of 8: a half-warp per partial row
// (lane = 8 dims, one 16-byte load), so one load instruction covers two rows
// and kBatch of them keep 2 * kBatch rows in flight; the halves add their
// sums at the end.
template <int kChunks>
__global__ void __launch_bounds__(kThreads) combine_bf16_kernel(CombineArgs a) {
  const int lane = threadIdx.x & 31;
  const int half = lane >> 4;
  const int hl = lane & 15;
  const int64_t hq = static_cast<int64_t>(a.hkv) * a.qhead;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  if (row >= a.tq * hq) return;
  const int64_t i = row / hq;
  const int hqa = static_cast<int>(row - i * hq);
  const int h = hqa / a.qhead;
  const int qh = hqa - h * a.qhead;
  const int d = a.head_dim;
  const int n8 = d >> 3;
  const int32_t* inv_row = a.inv + (static_cast<int64_t>(h) * a.tq + i) * a.topk;
  const int64_t base = a.edge_head_base[h];
  const uint16_t* o16 = static_cast<const uint16_t*>(a.o_partial);

  float big_m = -INFINITY;
  for (int r = lane; r < a.topk; r += 32) {
    const int32_t p = inv_row[r];
    if (p >= 0) big_m = fmaxf(big_m, a.m_partial[(base + p) * a.qhead + qh]);
  }
#pragma unroll
  for (int off = 16; off; off >>= 1) big_m = fmaxf(big_m, __shfl_xor_sync(0xffffffffu, big_m, off));

  float acc[kChunks][8];
#pragma unroll
  for (int c = 0; c < kChunks; ++c)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[c][j] = 0.f;
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
      constexpr int kBatch = 8;
      while (live) {
        float wv[kBatch];
        uint4 v[kBatch][kChunks];
#pragma unroll
        for (int t = 0; t < kBatch; ++t) {
          int s0 = -1, s1 = -1;
          if (live) {
            s0 = __ffs(live) - 1;
            live &= live - 1;
          }
          if (live) {
            s1 = __ffs(live) - 1;
            live &= live - 1;
          }
          const float w0 = __shfl_sync(0xffffffffu, wgt, s0 < 0 ? 0 : s0);
          const float w1 = __shfl_sync(0xffffffffu, wgt, s1 < 0 ? 0 : s1);
          const int64_t p0 = __shfl_sync(0xffffffffu, prow, s0 < 0 ? 0 : s0);
          const int64_t p1 = __shfl_sync(0xffffffffu, prow, s1 < 0 ? 0 : s1);
          const bool ok = half ? s1 >= 0 : s0 >= 0;
          wv[t] = ok ? (half ? w1 : w0) : 0.f;
          const int64_t pr = half ? p1 : p0;
#pragma unroll
          for (int c = 0; c < kChunks; ++c) {
            const int ch = hl + 16 * c;
            v[t][c] = make_uint4(0u, 0u, 0u, 0u);
            if (wv[t] > 0.f && ch < n8)
              v[t][c] = reinterpret_cast<const uint4*>(o16 + pr * d)[ch];
          }
        }
#pragma unroll
        for (int t = 0; t < kBatch; ++t)
#pragma unroll
          for (int c = 0; c < kChunks; ++c) {
            const uint32_t u[4] = {v[t][c].x, v[t][c].y, v[t][c].z, v[t][c].w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              acc[c][2 * j] = fmaf(wv[t], __uint_as_float(u[j] << 16), acc[c][2 * j]);
              acc[c][2 * j + 1] =
                  fmaf(wv[t], __uint_as_float(u[j] & 0xFFFF0000u), acc[c][2 * j + 1]);
            }
          }
      }
    }
#pragma unroll
    for (int off = 16; off; off >>= 1) big_l += __shfl_xor_sync(0xffffffffu, big_l, off);
#pragma unroll
    for (int c = 0; c < kChunks; ++c)
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[c][j] += __shfl_xor_sync(0xffffffffu, acc[c][j], 16);
  }
  const float inv_l = big_l > 0.f ? 1.f / big_l : 0.f;
  if (half == 0) {
    float4* orow = reinterpret_cast<float4*>(a.out + row * d);
#pragma unroll
    for (int c = 0; c < kChunks; ++c) {
      const int ch = hl + 16 * c;
      if (ch < n8) {
        orow[2 * ch] = make_float4(acc[c][0] * inv_l, acc[c][1] * inv_l, acc[c][2] * inv_l,
                                   acc[c][3] * inv_l);
        orow[2 * ch + 1] = make_float4(acc[c][4] * inv_l, acc[c][5] * inv_l, acc[c][6] * inv_l,
                                       acc[c][7] * inv_l);
      }
    }
  }
  if (a.lse && lane == 0) a.lse[row] = big_l > 0.f ? big_m + logf(big_l) : -INFINITY;
}

}  // namespace

cudaError_t launch_combine(const CombineArgs& a, cudaStream_t stream) {
  const int64_t rows = a.tq * a.hkv * a.qhead;
  if (rows == 0) return cudaSuccess;
  const int64_t grid = (rows + kWarps - 1) / kWarps;
  const unsigned g = static_cast<unsigned>(grid);
  if (a.o_bf16 && a.head_dim % 8 == 0) {
    if (a.head_dim <= 128)
      combine_bf16_kernel<1><<<g, kThreads, 0, stream>>>(a);
    else
      combine_bf16_kernel<2><<<g, kThreads, 0, stream>>>(a);
    return cudaGetLastError();
  }
  if (a.head_dim <= 128) {
    if (a.o_bf16)
      combine_kernel<1, true><<<g, kThreads, 0, stream>>>(a);
    else
      combine_kernel<1, false><<<g, kThreads, 0, stream>>>(a);
  } else {
    if (a.o_bf16)
      combine_kernel<2, true><<<g, kThreads, 0, stream>>>(a);
    else
      combine_kernel<2, false><<<g, kThreads, 0, stream>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace sa
