// Step 2 of KV-outer sparse attention for decode-shaped work with bf16 K/V:
// per-edge partials as in process_work_unit (forward.rs of alice-llm's
// sparse_attention), with the two products of every 16-key chunk on the
// tensor cores through warp-level mma.sync (m16n8k16, bf16 in, f32 out).
//
// Why warp-level MMA here: a decode unit has 8-16 rows (one query's GQA
// lanes), far below the 64/128-row tiles of tcgen05, and the kernel is bound
// by HBM; what it needs from the tensor cores is to take the per-key FMA work
// off the CUDA cores (with 8 rows that work would otherwise cap it near 30 %
// of HBM).  Precision: K and V are exact in bf16; Q and P are each split into
// a bf16 high part and a bf16 remainder and both parts are multiplied, so
// products carry about 16 mantissa bits and accumulation stays in f32.
//
// Structure (per warp, independent pipelines, as in forward_dec.cu): the warp
// streams its splits in chunks of 16 keys; lanes 0-15 / 16-31 bulk-copy one
// K / V row each (256 bytes) into a ring stage with rows padded to 272 bytes
// (conflict-free ldmatrix); the split's Q rows (f32) arrive with its first
// chunk.  Per chunk: S = Q K^T (ldmatrix K, 32 mma), online softmax on the
// accumulator fragments (row max over a 4-lane quad), P re-used in registers
// as the A operand of O += P V (ldmatrix.trans V, 32 mma).
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
using dec::bcast_scalars;
using dec::stash_meta_arrays;

constexpr int kD = 128;
constexpr int kKC = 16;             // keys per chunk
constexpr int kRow = 272;           // bytes per staged bf16 row (256 + 16 padding)
constexpr int kQBufs = 2;          // enough while NST <= chunks per block + 1
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__host__ __device__ inline size_t up128m(size_t x) { return (x + 127) & ~static_cast<size_t>(127); }

struct MmaPlan {
  size_t stage_bytes, q_bytes, warp_bytes;
};

__host__ __device__ inline MmaPlan mma_plan(int rows, int nst) {
  MmaPlan p{};
  p.stage_bytes = 2 * kKC * kRow;                          // K rows then V rows
  p.q_bytes = static_cast<size_t>(rows) * kD * 4;          // raw f32 Q rows
  p.warp_bytes = up128m(nst * p.stage_bytes + kQBufs * p.q_bytes + 8 * nst +
                       4 * 32 * (kMaxPages + kMaxQi));
  return p;
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// (lo, hi) f32 -> packed bf16x2, round to nearest even; lo in the low half.
__device__ __forceinline__ uint32_t bf2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float bf_lo_f(uint32_t p) { return __uint_as_float(p << 16); }
__device__ __forceinline__ float bf_hi_f(uint32_t p) { return __uint_as_float(p & 0xFFFF0000u); }

// Split two values into bf16 high parts and bf16 remainders.
__device__ __forceinline__ void split2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  hi = bf2(x0, x1);
  lo = bf2(x0 - bf_lo_f(hi), x1 - bf_hi_f(hi));
}

// kOBf16: the o partials are written as bf16.
template <int R, int NST, int WARPS, bool kOBf16>
__global__ void __launch_bounds__(WARPS * 32, 1)
forward_dec_mma_kernel(ForwardArgs a) {
  static_assert(R == 8 || R == 16, "rows per group");
  extern __shared__ __align__(128) unsigned char smem[];
  const MmaPlan plan = mma_plan(R, NST);
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  unsigned char* base = smem + warp * plan.warp_bytes;
  unsigned char* stages = base;
  float* qbuf = reinterpret_cast<float*>(base + NST * plan.stage_bytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + NST * plan.stage_bytes + kQBufs * plan.q_bytes);
  int* pid_tab = reinterpret_cast<int*>(bars + NST);     // [32][kMaxPages] of the current batch
  int* qi_tab = pid_tab + 32 * kMaxPages;                // [32][kMaxQi]

  const int qhead = a.qhead;
  const int ps = a.page_size;
  const int cps = a.block_size / kKC;
  const int staged_edges = R / qhead;
  int64_t* status = a.totals + 3;
  const int64_t n_splits = min(a.totals[1], a.max_splits);
  const int64_t tw = static_cast<int64_t>(gridDim.x) * WARPS;
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * WARPS + warp;
  const float qscale = a.scale * kLog2e;
  const int g = lane >> 2;          // fragment row (and row + 8)
  const int c = lane & 3;           // fragment column pair

  if (lane == 0) {
    for (int s = 0; s < NST; ++s) mbar_init(bars + s, 1);
    fence_mbar_init();
  }
  for (size_t off = 16u * lane; off < NST * plan.stage_bytes; off += 16u * 32)
    *reinterpret_cast<float4*>(stages + off) = make_float4(0.f, 0.f, 0.f, 0.f);
  fence_proxy_async_smem();
  __syncwarp();

  uint32_t chunks_issued = 0, chunks_done = 0, groups_issued = 0, groups_done = 0;
  bool ok = true;

  for (int64_t batch0 = 0; ok; batch0 += 32) {
    if (gw + batch0 * tw >= n_splits) break;
    SplitMeta mine;
    load_meta(a, gw + (batch0 + lane) * tw, n_splits, staged_edges, mine);
    __syncwarp();   // the previous batch is done with the tables
    stash_meta_arrays(mine, lane, pid_tab, qi_tab);
    __syncwarp();
    const int64_t left = (n_splits - gw - batch0 * tw + tw - 1) / tw;
    const int nb = static_cast<int>(left < 32 ? left : 32);

    int is_j = 0, is_g = 0, is_c = 0;
    SplitMeta im = bcast_scalars(mine, 0);
    auto issue_one = [&]() {
      const int stage = chunks_issued % NST;
      unsigned char* st = stages + stage * plan.stage_bytes;
      const int k0 = is_c * kKC;
      // lanes 0-15: K row k0+lane, lanes 16-31: V row k0+lane-16
      const int kk = lane & 15;
      const int j = k0 + kk;
      const int p = j / ps;
      const bool live = p < kMaxPages && ((im.pmask >> p) & 1u) && im.bstart + j < im.bend;
      const int pid = p < kMaxPages ? pid_tab[is_j * kMaxPages + p] : -1;
      uint32_t tx = live ? 256u : 0u;
      const int rows_g = min(R, im.nrows - is_g * R);
      const int ne = (rows_g + qhead - 1) / qhead;
      int my_qi = -1;
      if (is_c == 0 && lane < ne) {
        const int e = is_g * staged_edges + lane;
        my_qi = e < kMaxQi ? qi_tab[is_j * kMaxQi + e]
                           : a.edges[2 * (static_cast<int64_t>(im.edge0) + e)];
      }
      const uint32_t q_tx = my_qi >= 0 ? static_cast<uint32_t>(qhead * kD * 4) : 0u;
      uint32_t all = tx + q_tx;
#pragma unroll
      for (int off = 16; off; off >>= 1) all += __shfl_xor_sync(0xffffffffu, all, off);
      if (lane == 0) mbar_arrive_expect_tx(bars + stage, all);
      __syncwarp();
      if (live) {
        const size_t src = ((static_cast<size_t>(pid) * a.hkv + im.h) * ps + (j - p * ps)) * kD * 2;
        const void* base_ptr = lane < 16 ? a.k_pages : a.v_pages;
        bulk_g2s(st + (lane < 16 ? 0 : kKC * kRow) + kk * kRow,
                 static_cast<const unsigned char*>(base_ptr) + src, 256u, bars + stage);
      }
      if (my_qi >= 0) {
        float* dst = qbuf + static_cast<size_t>(groups_issued % kQBufs) * R * kD +
                     static_cast<size_t>(lane) * qhead * kD;
        const float* src = a.q + (static_cast<int64_t>(my_qi) * a.hq +
                                  static_cast<int64_t>(im.h) * qhead) * kD;
        bulk_g2s(dst, src, static_cast<uint32_t>(qhead * kD * 4), bars + stage);
      }
      ++chunks_issued;
      if (++is_c == cps) {
        is_c = 0;
        ++groups_issued;
        if (++is_g * R >= max(im.nrows, 1)) {
          is_g = 0;
          ++is_j;
          if (is_j < nb) im = bcast_scalars(mine, is_j);
        }
      }
    };

    while (is_j < nb && chunks_issued - chunks_done < static_cast<uint32_t>(NST)) issue_one();

    for (int jsp = 0; jsp < nb && ok; ++jsp) {
      const SplitMeta m = bcast_scalars(mine, jsp);
      const int ngroups = max((m.nrows + R - 1) / R, 1);
      for (int grp = 0; grp < ngroups && ok; ++grp) {
        const int rows_g = min(R, m.nrows - grp * R);
        const float* qg = qbuf + static_cast<size_t>(groups_done % kQBufs) * R * kD;
        // Causal limits of this thread's two fragment rows (g and g + 8).
        int lim[2];
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          const int r = g + 8 * h2;
          lim[h2] = -1;
          if (r < rows_g) {
            const int e = grp * staged_edges + r / qhead;
            int64_t qidx;
            qidx = e < kMaxQi ? qi_tab[jsp * kMaxQi + e]
                              : a.edges[2 * (static_cast<int64_t>(m.edge0) + e)];
            int64_t l64 = INT32_MAX;
            if (a.causal) {
              const int64_t ql = qidx - m.q0;
              l64 = a.causal == 2 || m.lk < m.qo ? ql : m.lk - m.qo + ql;
            }
            lim[h2] = static_cast<int>(l64 < INT32_MAX ? l64 : INT32_MAX);
          }
        }
        float m_run[2] = {-INFINITY, -INFINITY};
        float l_part[2] = {0.f, 0.f};
        float o[16][4];
#pragma unroll
        for (int nt = 0; nt < 16; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) o[nt][e] = 0.f;
        uint32_t qhi[8][4], qlo[8][4];
        bool have_q = false;

        for (int ch = 0; ch < cps; ++ch) {
          const int stage = chunks_done % NST;
          const uint32_t parity = (chunks_done / NST) & 1u;
          const bool got = mbar_wait_bounded(bars + stage, parity);
          if (!__all_sync(0xffffffffu, got)) {
            if (lane == 0) report(status, SA_ERR_DEVICE_TIMEOUT);
            ok = false;
            break;
          }
          if (!have_q) {
            // Q fragments (pre-scaled into the log2 domain), high and low parts.
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
#pragma unroll
              for (int part = 0; part < 4; ++part) {
                const int r = g + ((part & 1) ? 8 : 0);
                const int col = 16 * ks + 2 * c + ((part & 2) ? 8 : 0);
                float2 v = make_float2(0.f, 0.f);
                if (r < rows_g) v = *reinterpret_cast<const float2*>(qg + r * kD + col);
                split2(v.x * qscale, v.y * qscale, qhi[ks][part], qlo[ks][part]);
              }
            }
            have_q = true;
          }
          const unsigned char* kt = stages + stage * plan.stage_bytes;
          const unsigned char* vt = kt + kKC * kRow;
          const int k0 = ch * kKC;
          // Keys of this chunk that exist (inside the length, page present).
          const unsigned present = __ballot_sync(
              0xffffffffu, lane < kKC && m.bstart + k0 + lane < m.bend &&
                               ((m.pmask >> ((k0 + lane) / ps)) & 1u));
          if (present) {
            // ---- S = Q K^T for 16 keys (two n-tiles of 8) ----
            // Four independent accumulator chains per n-tile (high / low
            // parts of Q, even / odd k-steps), summed at the end.
            float sacc[2][4];
            {
              float part[4][2][4];
#pragma unroll
              for (int q = 0; q < 4; ++q)
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                  for (int e = 0; e < 4; ++e) part[q][nt][e] = 0.f;
              const int mi = lane >> 3, ri = lane & 7;
              const uint32_t rowaddr =
                  smem_u32(kt) + static_cast<uint32_t>(((mi >> 1) * 8 + ri) * kRow + (mi & 1) * 16);
#pragma unroll
              for (int ks = 0; ks < 8; ++ks) {
                uint32_t b[4];
                ldsm_x4(rowaddr + ks * 32, b);
                const int q = (ks & 1) * 2;
                mma16816(part[q][0], qhi[ks], b[0], b[1]);
                mma16816(part[q + 1][0], qlo[ks], b[0], b[1]);
                mma16816(part[q][1], qhi[ks], b[2], b[3]);
                mma16816(part[q + 1][1], qlo[ks], b[2], b[3]);
              }
#pragma unroll
              for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e)
                  sacc[nt][e] = (part[0][nt][e] + part[2][nt][e]) + (part[1][nt][e] + part[3][nt][e]);
            }
            // ---- mask, online softmax (rows g and g + 8) ----
            float pv[2][4];
            float alpha[2];
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
              float cm = -INFINITY;
#pragma unroll
              for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                  const int kk = 8 * nt + 2 * c + e;
                  const bool live = ((present >> kk) & 1u) && m.bstart + k0 + kk <= lim[h2];
                  float& sv = sacc[nt][2 * h2 + e];
                  sv = live ? sv : -INFINITY;
                  cm = fmaxf(cm, sv);
                }
              cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, 1));
              cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, 2));
              const float m_new = fmaxf(m_run[h2], cm);
              alpha[h2] = m_new == -INFINITY ? 1.f : exp2f(m_run[h2] - m_new);
              const float msub = m_new == -INFINITY ? 0.f : m_new;
              float lsum = 0.f;
#pragma unroll
              for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                  const float pe = exp2f(sacc[nt][2 * h2 + e] - msub);
                  pv[nt][2 * h2 + e] = pe;
                  lsum += pe;
                }
              l_part[h2] = l_part[h2] * alpha[h2] + lsum;
              m_run[h2] = m_new;
            }
            if (__any_sync(0xffffffffu, alpha[0] != 1.f || alpha[1] != 1.f)) {
#pragma unroll
              for (int nt = 0; nt < 16; ++nt) {
                o[nt][0] *= alpha[0];
                o[nt][1] *= alpha[0];
                o[nt][2] *= alpha[1];
                o[nt][3] *= alpha[1];
              }
            }
            // P as the A operand (rows g / g+8, keys 2c.. / 2c+8..), high and low parts.
            uint32_t phi[4], plo[4];
            split2(pv[0][0], pv[0][1], phi[0], plo[0]);
            split2(pv[0][2], pv[0][3], phi[1], plo[1]);
            split2(pv[1][0], pv[1][1], phi[2], plo[2]);
            split2(pv[1][2], pv[1][3], phi[3], plo[3]);
            // ---- O += P V (16 n-tiles of 8 dims) ----
            {
              const int mi = lane >> 3, ri = lane & 7;
              const uint32_t rowaddr =
                  smem_u32(vt) + static_cast<uint32_t>(((mi & 1) * 8 + ri) * kRow + (mi >> 1) * 16);
#pragma unroll
              for (int np = 0; np < 8; ++np) {
                uint32_t b[4];
                ldsm_x4_t(rowaddr + np * 32, b);
                mma16816(o[2 * np], phi, b[0], b[1]);
                mma16816(o[2 * np], plo, b[0], b[1]);
                mma16816(o[2 * np + 1], phi, b[2], b[3]);
                mma16816(o[2 * np + 1], plo, b[2], b[3]);
              }
            }
          }
          ++chunks_done;
          __syncwarp();
          fence_proxy_async_smem();
          if (is_j < nb) issue_one();
        }
        if (!ok) break;
        ++groups_done;
        // ---- the group's partial rows ----
        const int64_t row0 = static_cast<int64_t>(m.edge0) * qhead + grp * R;
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          float l = l_part[h2];
          l += __shfl_xor_sync(0xffffffffu, l, 1);
          l += __shfl_xor_sync(0xffffffffu, l, 2);
          const int r = g + 8 * h2;
          if (r < rows_g) {
            if constexpr (kOBf16) {
              uint16_t* dst = static_cast<uint16_t*>(a.o_partial) + (row0 + r) * kD + 2 * c;
#pragma unroll
              for (int nt = 0; nt < 16; ++nt)
                *reinterpret_cast<uint32_t*>(dst + 8 * nt) = bf2(o[nt][2 * h2], o[nt][2 * h2 + 1]);
            } else {
              float* dst = static_cast<float*>(a.o_partial) + (row0 + r) * kD + 2 * c;
#pragma unroll
              for (int nt = 0; nt < 16; ++nt)
                *reinterpret_cast<float2*>(dst + 8 * nt) = make_float2(o[nt][2 * h2], o[nt][2 * h2 + 1]);
            }
            if (c == 0) {
              a.m_partial[row0 + r] = m_run[h2] == -INFINITY ? -INFINITY : m_run[h2] * kLn2;
              a.l_partial[row0 + r] = l;
            }
          }
        }
      }
    }
    if (!ok) {
      while (chunks_done < chunks_issued) {
        mbar_wait_bounded(bars + chunks_done % NST, (chunks_done / NST) & 1u);
        ++chunks_done;
      }
    }
  }
}

template <int R, int NST, int WARPS, bool kOBf16>
cudaError_t launch_dec_mma(const ForwardArgs& a, cudaStream_t stream) {
  const MmaPlan p = mma_plan(R, NST);
  const size_t smem = p.warp_bytes * WARPS;
  if (smem > 227 * 1024) return cudaErrorNotSupported;
  const void* fn = reinterpret_cast<const void*>(forward_dec_mma_kernel<R, NST, WARPS, kOBf16>);
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
  forward_dec_mma_kernel<R, NST, WARPS, kOBf16>
      <<<static_cast<unsigned>(grid), WARPS * 32, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

bool forward_dec_mma_supported(int head_dim, int block_size, int page_size, int qhead,
                               int kv_bf16) {
  if (!kv_bf16 || head_dim != kD) return false;
  // at least two chunks per block keeps the two Q buffers apart
  if (block_size % kKC != 0 || block_size < 2 * kKC) return false;
  if (page_size <= 0 || block_size % page_size || block_size / page_size > kMaxPages) return false;
  return qhead == 1 || qhead == 2 || qhead == 4 || qhead == 8 || qhead == 16;
}

cudaError_t launch_forward_dec_mma(const ForwardArgs& a, cudaStream_t stream) {
  if (!forward_dec_mma_supported(a.head_dim, a.block_size, a.page_size, a.qhead, a.kv_bf16))
    return cudaErrorNotSupported;
  if (a.qhead <= 8)
    return a.o_bf16 ? launch_dec_mma<8, 3, 6, true>(a, stream)
                    : launch_dec_mma<8, 3, 6, false>(a, stream);
  return a.o_bf16 ? launch_dec_mma<16, 3, 4, true>(a, stream)
                  : launch_dec_mma<16, 3, 4, false>(a, stream);
}

}  // namespace sa
