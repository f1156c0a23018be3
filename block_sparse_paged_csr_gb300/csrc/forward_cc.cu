// Step 2 of KV-outer sparse attention on CUDA cores: per-edge softmax partials
// (kvouter_forward / process_work_unit, forward.rs of alice-llm's
// sparse_attention), general over head_dim, block and page size.
//
// One CTA walks work splits (head, compact slot, edge range) with a grid
// stride.  For each split it stages the block's pages of K and V once into
// shared memory with 1-D bulk copies (one per page, completion on an
// mbarrier), then, 8 rows at a time (row = edge x GQA lane):
//   scores   one thread per (row, key): dot over head_dim from shared memory,
//            chunk order rotated by key so a warp's 16-byte reads spread over
//            all banks;
//   softmax  one warp per row: max and sum with shuffles, p = exp(s - m);
//   PV       one thread per (row, 4 output dims), p broadcast from shared.
// Masked keys (past the sequence's length, absent pages, right-aligned
// causal limit) score -inf; a row with no live key writes (0, -inf, 0).
#include <cfloat>
#include <cstdint>

#include "internal.h"
#include "sa_common.cuh"

namespace sa {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kRows = 8;               // rows per group
constexpr int kMaxDim = 256;

struct SmemPlan {
  size_t kv_bytes;   // one of K or V
  size_t k_off, v_off, q_off, p_off, pos_off, lim_off, total;
};

__host__ __device__ inline size_t align128(size_t x) { return (x + 127) & ~static_cast<size_t>(127); }

__host__ __device__ inline SmemPlan plan_smem(int block_size, int head_dim, int kv_bf16) {
  SmemPlan p{};
  const size_t elt = kv_bf16 ? 2 : 4;
  p.kv_bytes = static_cast<size_t>(block_size) * head_dim * elt;
  p.k_off = 128;  // [0, 16) holds the mbarrier
  p.v_off = align128(p.k_off + p.kv_bytes);
  p.q_off = align128(p.v_off + p.kv_bytes);
  p.p_off = align128(p.q_off + sizeof(float) * kRows * head_dim);
  p.pos_off = align128(p.p_off + sizeof(float) * kRows * block_size);
  p.lim_off = align128(p.pos_off + sizeof(int32_t) * block_size);
  p.total = align128(p.lim_off + sizeof(int32_t) * kRows);
  return p;
}

template <bool kBf16>
__device__ __forceinline__ float4 load4(const unsigned char* base, int row, int chunk,
                                        int head_dim) {
  if constexpr (kBf16) {
    const uint2 u = *reinterpret_cast<const uint2*>(
        base + (static_cast<size_t>(row) * head_dim + 4 * chunk) * 2);
    return bf16x4_to_f32(u);
  } else {
    return *reinterpret_cast<const float4*>(
        base + (static_cast<size_t>(row) * head_dim + 4 * chunk) * 4);
  }
}

template <bool kBf16>
__global__ void __launch_bounds__(kThreads)
forward_cc_kernel(ForwardArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  const SmemPlan plan = plan_smem(a.block_size, a.head_dim, kBf16 ? 1 : 0);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
  unsigned char* ks = smem + plan.k_off;
  unsigned char* vs = smem + plan.v_off;
  float* qs = reinterpret_cast<float*>(smem + plan.q_off);
  float* ps = reinterpret_cast<float*>(smem + plan.p_off);
  int32_t* kpos = reinterpret_cast<int32_t*>(smem + plan.pos_off);
  int32_t* rlim = reinterpret_cast<int32_t*>(smem + plan.lim_off);
  __shared__ uint32_t s_bytes;

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int d = a.head_dim;
  const int nc = d >> 2;                // float4 chunks per row
  const int bs = a.block_size;
  const int ps_ = a.page_size;
  const int qhead = a.qhead;
  const size_t elt = kBf16 ? 2 : 4;
  const size_t page_bytes = static_cast<size_t>(ps_) * d * elt;
  int64_t* status = a.totals + 3;

  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  // Rows of absent pages are never copied; PV multiplies them by p = 0, so
  // they must hold finite values: clear both tiles once.
  for (size_t off = 16u * tid; off < plan.kv_bytes; off += 16u * kThreads) {
    *reinterpret_cast<float4*>(ks + off) = make_float4(0.f, 0.f, 0.f, 0.f);
    *reinterpret_cast<float4*>(vs + off) = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  fence_proxy_async_smem();
  __syncthreads();
  uint32_t phase = 0;

  const int64_t n_splits = min(a.totals[1], a.max_splits);
  for (int64_t sp = blockIdx.x; sp < n_splits; sp += gridDim.x) {
    const int4 w = reinterpret_cast<const int4*>(a.splits)[sp];
    const int h = w.x;
    if (h < 0 || h >= a.hkv || w.y < 0 || w.y >= a.nbs || w.z < 0 || w.w < w.z) {
      if (tid == 0) report(status, SA_ERR_SHAPE);
      continue;
    }
    const int raw = a.sel_slots[static_cast<int64_t>(h) * a.nbs + w.y];
    if (raw < 0 || raw >= a.nbs) {
      if (tid == 0) report(status, SA_ERR_SHAPE);
      continue;
    }
    const int b = raw / a.msb;
    const int blk = raw % a.msb;
    const int64_t lk = a.used ? (a.used[b] > 0 ? a.used[b] : 0)
                              : static_cast<int64_t>(a.msb) * bs;
    const int64_t block_start = static_cast<int64_t>(blk) * bs;
    const int64_t block_end = min(block_start + bs, lk);
    const int64_t q0 = a.cu[b];
    const int64_t qo = a.cu[b + 1] - q0;
    const int32_t* bt_row = a.block_tables + static_cast<int64_t>(b) * a.max_pages +
                            static_cast<int64_t>(blk) * a.pages_per_block;

    __syncthreads();  // previous split's readers of K/V/Q/P are done
    // Key liveness: absolute position, or -1 (past the length / absent page).
    for (int t = tid; t < bs; t += kThreads) {
      const int64_t p = block_start + t;
      int32_t live = -1;
      if (p < block_end) {
        const int32_t pid = bt_row[t / ps_];
        if (pid >= 0 && pid < a.num_pages) live = static_cast<int32_t>(p);
      }
      kpos[t] = live;
    }
    if (tid == 0) {
      uint32_t bytes = 0;
      for (int pl = 0; pl < a.pages_per_block; ++pl) {
        const int64_t lo = block_start + static_cast<int64_t>(pl) * ps_;
        if (lo >= block_end) break;
        const int32_t pid = bt_row[pl];
        if (pid < 0) continue;
        if (pid >= a.num_pages) {
          report(status, SA_ERR_SHAPE);
          continue;
        }
        bytes += 2u * static_cast<uint32_t>(page_bytes);
      }
      s_bytes = bytes;
      if (bytes) {
        mbar_arrive_expect_tx(bar, bytes);
        for (int pl = 0; pl < a.pages_per_block; ++pl) {
          const int64_t lo = block_start + static_cast<int64_t>(pl) * ps_;
          if (lo >= block_end) break;
          const int32_t pid = bt_row[pl];
          if (pid < 0 || pid >= a.num_pages) continue;
          const size_t src = ((static_cast<size_t>(pid) * a.hkv + h) * ps_) * d * elt;
          bulk_g2s(ks + pl * page_bytes, static_cast<const unsigned char*>(a.k_pages) + src,
                   static_cast<uint32_t>(page_bytes), bar);
          bulk_g2s(vs + pl * page_bytes, static_cast<const unsigned char*>(a.v_pages) + src,
                   static_cast<uint32_t>(page_bytes), bar);
        }
      }
    }
    __syncthreads();
    if (s_bytes) {
      const bool ok = mbar_wait_bounded(bar, phase);
      if (__syncthreads_or(!ok)) {   // every thread leaves together
        if (tid == 0) report(status, SA_ERR_DEVICE_TIMEOUT);
        return;
      }
      phase ^= 1u;
    }

    const int64_t row0 = static_cast<int64_t>(w.z) * qhead;     // first partial row
    const int rows = (w.w - w.z) * qhead;
    for (int rg = 0; rg < rows; rg += kRows) {
      const int nr = min(kRows, rows - rg);
      // Q rows of this group and their causal limits.
      for (int idx = tid; idx < nr * nc; idx += kThreads) {
        const int r = idx / nc;
        const int c = idx - r * nc;
        const int row = rg + r;
        const int64_t e = w.z + row / qhead;
        const int qh = row % qhead;
        const int64_t qi = a.edges[2 * e];
        const float4 v = *reinterpret_cast<const float4*>(
            a.q + (qi * a.hq + static_cast<int64_t>(h) * qhead + qh) * d + 4 * c);
        reinterpret_cast<float4*>(qs + r * d)[c] = v;
        if (c == 0) {
          int64_t lim = INT32_MAX;
          if (a.causal) {
            const int64_t ql = qi - q0;
            lim = a.causal == 2 || lk < qo ? ql : lk - qo + ql;
          }
          rlim[r] = static_cast<int32_t>(lim < INT32_MAX ? lim : INT32_MAX);
        }
      }
      __syncthreads();
      // Scores.
      for (int idx = tid; idx < nr * bs; idx += kThreads) {
        const int r = idx / bs;
        const int t = idx - r * bs;
        const int32_t kp = kpos[t];
        float s = -INFINITY;
        if (kp >= 0 && kp <= rlim[r]) {
          const float4* qrow = reinterpret_cast<const float4*>(qs + r * d);
          float acc = 0.f;
          int c = t % nc;
          for (int cc = 0; cc < nc; ++cc) {
            const float4 kv = load4<kBf16>(ks, t, c, d);
            const float4 qv = qrow[c];
            acc = fmaf(qv.x, kv.x, acc);
            acc = fmaf(qv.y, kv.y, acc);
            acc = fmaf(qv.z, kv.z, acc);
            acc = fmaf(qv.w, kv.w, acc);
            if (++c == nc) c = 0;
          }
          s = acc * a.scale;
        }
        ps[r * bs + t] = s;
      }
      __syncthreads();
      // Softmax statistics, one warp per row.
      for (int r = warp; r < nr; r += kWarps) {
        float m = -INFINITY;
        for (int t = lane; t < bs; t += 32) m = fmaxf(m, ps[r * bs + t]);
#pragma unroll
        for (int off = 16; off; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
        float l = 0.f;
        for (int t = lane; t < bs; t += 32) {
          const float s = ps[r * bs + t];
          const float p = (m == -INFINITY || s == -INFINITY) ? 0.f : __expf(s - m);
          ps[r * bs + t] = p;
          l += p;
        }
#pragma unroll
        for (int off = 16; off; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
        if (lane == 0) {
          a.m_partial[row0 + rg + r] = m;
          a.l_partial[row0 + rg + r] = l;
        }
      }
      __syncthreads();
      // o = sum_t p_t v_t.
      for (int idx = tid; idx < nr * nc; idx += kThreads) {
        const int r = idx / nc;
        const int c = idx - r * nc;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        const float* prow = ps + r * bs;
        for (int t = 0; t < bs; ++t) {
          const float p = prow[t];
          const float4 vv = load4<kBf16>(vs, t, c, d);
          acc.x = fmaf(p, vv.x, acc.x);
          acc.y = fmaf(p, vv.y, acc.y);
          acc.z = fmaf(p, vv.z, acc.z);
          acc.w = fmaf(p, vv.w, acc.w);
        }
        store_o4(a.o_partial, a.o_bf16, (row0 + rg + r) * d + 4 * c, acc);
      }
      __syncthreads();
    }
  }
}

}  // namespace

bool forward_cc_supported(int head_dim, int block_size, int kv_bf16) {
  if (head_dim <= 0 || head_dim > kMaxDim) return false;
  if (head_dim % (kv_bf16 ? 8 : 4) != 0) return false;
  if (block_size <= 0) return false;
  const SmemPlan p = plan_smem(block_size, head_dim, kv_bf16);
  return p.kv_bytes * 2 <= 160 * 1024 && p.total <= 227 * 1024;
}

cudaError_t launch_forward_cc(const ForwardArgs& a, cudaStream_t stream) {
  if (!forward_cc_supported(a.head_dim, a.block_size, a.kv_bf16)) return cudaErrorNotSupported;
  const SmemPlan p = plan_smem(a.block_size, a.head_dim, a.kv_bf16);
  const void* fn = a.kv_bf16 ? reinterpret_cast<const void*>(forward_cc_kernel<true>)
                             : reinterpret_cast<const void*>(forward_cc_kernel<false>);
  cudaError_t err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(p.total));
  if (err != cudaSuccess) return err;
  err = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
  if (err != cudaSuccess) return err;
  int per_sm = 0;
  err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kThreads, p.total);
  if (err != cudaSuccess) return err;
  if (per_sm < 1) per_sm = 1;
  int64_t grid = static_cast<int64_t>(device_sm_count()) * per_sm;
  if (grid > a.max_splits) grid = a.max_splits;
  if (grid < 1) grid = 1;
  if (a.kv_bf16)
    forward_cc_kernel<true><<<static_cast<unsigned>(grid), kThreads, p.total, stream>>>(a);
  else
    forward_cc_kernel<false><<<static_cast<unsigned>(grid), kThreads, p.total, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace sa
