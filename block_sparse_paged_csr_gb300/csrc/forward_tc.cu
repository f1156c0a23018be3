// Step 2 of KV-outer sparse attention on the 5th-generation tensor cores
// (tcgen05 + TMEM): per-edge partials as in process_work_unit (forward.rs of
// alice-llm's sparse_attention) for work units with many gathered rows
// (chunked prefill, skewed selections).
//
// A CTA (4 warps, thread t <-> accumulator row t; two CTAs per SM) takes
// (kv head, block) units round-robin, so the CTAs running together work on
// neighbouring blocks of one (kv head, sequence) and share its Q rows in L2.
// For each unit it converts the block's K and V rows (fetched through the
// block table, f32 or bf16) to bf16 once, in shared memory laid out for the
// tensor cores: K as [keys x 128] and V transposed as [128 x keys], both
// K-major with the 128-byte swizzle.  For every tile of up to 128 of the
// unit's rows (edge x GQA lane) it then
//   1. gathers the rows' Q (f32 -> bf16, same layout),
//   2. issues S = Q K^T (M=128, N=block, K=128) into TMEM,
//   3. reads S back one row per thread (tcgen05.ld), masks (block length,
//      absent pages, right-aligned causal limit), computes m, p = exp(s - m)
//      and l, and stores p as bf16 over the (now unused) Q tile,
//   4. issues O = P V (M=128, N=128, K=block) into TMEM,
//   5. reads O back one row per thread and writes the unnormalised partial
//      row with its m and l.
// One thread issues the MMAs; tcgen05.commit signals an mbarrier.  Operands
// are rounded to bf16 (tolerance class of the tensor-core path); S, O and
// the softmax statistics stay in f32.
#include <cstdint>

#include "internal.h"
#include "sa_common.cuh"

namespace sa {

namespace {

constexpr int kD = 128;
constexpr int kM = 128;            // rows per MMA tile
constexpr int kThreads = 128;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr uint32_t kTmemCols = 256;  // S at column 0 (<= 128 columns), O at column 128

// ---------------------------------------------------------------- PTX helpers

__device__ __forceinline__ void tmem_alloc(uint32_t* smem_result, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(smem_result)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D (TMEM) (+)= A (smem) x B (smem)^T, bf16 inputs, f32 accumulation.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// 32 consecutive f32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, 8-row
// core groups 1024 bytes apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);          // start address
  d |= static_cast<uint64_t>(1u) << 16;                         // leading byte offset (unused)
  d |= static_cast<uint64_t>((1024u >> 4) & 0x3FFFu) << 32;     // stride byte offset
  d |= static_cast<uint64_t>(1u) << 46;                         // descriptor version
  d |= static_cast<uint64_t>(2u) << 61;                         // 128-byte swizzle
  return d;
}

// Instruction descriptor: bf16 x bf16 -> f32, both operands K-major.
__host__ __device__ constexpr uint32_t idesc_bf16(int m, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(m >> 4) << 24);
}

// Byte offset of element pair/quad position inside a K-major, 128B-swizzled
// tile of `rows` rows: element k of row r (bf16 elements, 64 per panel row).
__device__ __forceinline__ uint32_t sw128_offset(int rows, int r, int k) {
  const int panel = k >> 6;
  const int chunk = (k & 63) >> 3;
  const int within = (k & 7) * 2;
  return static_cast<uint32_t>(panel * rows * 128 + r * 128 + ((chunk ^ (r & 7)) << 4) + within);
}

// Two f32 values to a packed bf16x2 (round to nearest even), `lo` in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2_rn(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

struct TcPlan {
  size_t k_off, v_off, qp_off, pos_off, off_off, total;
};

// Shared memory: K [BS][128] and V^T [128][BS] (bf16, swizzled), one tile
// buffer used first for Q [128][128] and then for P [128][BS], per-key
// positions and row offsets.
__host__ __device__ inline TcPlan tc_plan(int bs) {
  TcPlan p{};
  p.k_off = 1024;                                   // [0, 1024): barrier, TMEM slot, unit bases
  p.v_off = p.k_off + static_cast<size_t>(bs) * kD * 2;
  p.qp_off = p.v_off + static_cast<size_t>(kD) * bs * 2;
  p.pos_off = p.qp_off + static_cast<size_t>(kM) * kD * 2;
  p.off_off = p.pos_off + static_cast<size_t>(bs) * 4;
  p.total = p.off_off + static_cast<size_t>(bs) * 8 + 1024;   // + alignment slack
  return p;
}

template <bool kBf16>
__device__ __forceinline__ uint2 ld_kv4_bf16(const void* pages, int64_t elem_off) {
  if constexpr (kBf16) {
    return __ldg(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(pages) + elem_off));
  } else {
    const float4 v = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(pages) + elem_off));
    return make_uint2(pack_bf16x2_rn(v.x, v.y), pack_bf16x2_rn(v.z, v.w));
  }
}

template <bool kBf16>
__device__ __forceinline__ float ld_kv1(const void* pages, int64_t elem_off) {
  if constexpr (kBf16) {
    return bf16_to_f32(__ldg(static_cast<const uint16_t*>(pages) + elem_off));
  } else {
    return __ldg(static_cast<const float*>(pages) + elem_off);
  }
}

template <int BS, bool kBf16>
__global__ void __launch_bounds__(kThreads)
forward_tc_kernel(ForwardArgs a) {
  extern __shared__ unsigned char smem_raw[];
  // 1024-byte alignment for the swizzled tiles.
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const TcPlan plan = tc_plan(BS);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + 16);
  int32_t* unit_base = reinterpret_cast<int32_t*>(smem + 64);       // [hkv+1], hkv <= 200
  unsigned char* ks = smem + plan.k_off;     // K   [BS rows][128] bf16, K-major SW128
  unsigned char* vs = smem + plan.v_off;     // V^T [128 rows][BS] bf16, K-major SW128
  unsigned char* qp = smem + plan.qp_off;    // Q [128][128], later P [128][BS] bf16
  int32_t* kpos = reinterpret_cast<int32_t*>(smem + plan.pos_off);   // [BS] position or -1
  int64_t* koff = reinterpret_cast<int64_t*>(smem + plan.off_off);   // [BS] row offset or -1

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int qhead = a.qhead;
  const int ps = a.page_size;
  int64_t* status = a.totals + 3;
  const float qscale = a.scale * kLog2e;

  if (warp == 0) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
    int32_t acc = 0;
    for (int hh = 0; hh < a.hkv; ++hh) {
      unit_base[hh] = acc;
      acc += a.num_sel[hh];
    }
    unit_base[a.hkv] = acc;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t t_s = tmem;            // S: columns [0, BS)
  const uint32_t t_o = tmem + 128;      // O: columns [128, 256)
  const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
  const int64_t n_units = unit_base[a.hkv];
  uint32_t phase = 0;
  bool ok = true;

  // Units round-robin over CTAs: CTAs running at the same time work on
  // neighbouring blocks of one (kv head, sequence), whose Q rows stay in L2.
  for (int64_t u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
    int h = 0;
    while (h + 1 < a.hkv && unit_base[h + 1] <= u) ++h;
    const int j = static_cast<int>(u - unit_base[h]);
    const int raw = a.sel_slots[static_cast<int64_t>(h) * a.nbs + j];
    const int64_t ebase = a.edge_head_base[h];
    const int64_t e0 = ebase + a.sel_offsets[static_cast<int64_t>(h) * (a.nbs + 1) + j];
    const int64_t e1 = ebase + a.sel_offsets[static_cast<int64_t>(h) * (a.nbs + 1) + j + 1];
    if (raw < 0 || raw >= a.nbs || e1 < e0) {
      if (tid == 0) report(status, SA_ERR_SHAPE);
      continue;
    }
    const int b = raw / a.msb;
    const int blk = raw - b * a.msb;
    const int64_t lk = a.used ? max(a.used[b], 0) : static_cast<int64_t>(a.msb) * BS;
    const int64_t bstart = static_cast<int64_t>(blk) * BS;
    const int64_t bend = min(bstart + BS, lk);
    const int64_t q0 = a.cu[b];
    const int64_t qo = a.cu[b + 1] - q0;

    // ---- K and V^T of the unit ---------------------------------------------
    __syncthreads();   // the previous unit's MMAs were waited for: K / V are free
    const int32_t* bt = a.block_tables + static_cast<int64_t>(b) * a.max_pages +
                        static_cast<int64_t>(blk) * a.pages_per_block;
    for (int jj = tid; jj < BS; jj += kThreads) {
      const int64_t pos = bstart + jj;
      int32_t live = -1;
      int64_t off = -1;
      if (pos < bend) {
        const int pid = bt[jj / ps];
        if (pid >= a.num_pages) report(status, SA_ERR_SHAPE);
        if (pid >= 0 && pid < a.num_pages) {
          live = static_cast<int32_t>(pos);
          off = ((static_cast<int64_t>(pid) * a.hkv + h) * ps + jj % ps) * kD;
        }
      }
      kpos[jj] = live;
      koff[jj] = off;
    }
    __syncthreads();
    // K rows: warp-cooperative (lane = 4 dims), all of a warp's rows in flight.
    {
      uint2 kr[BS / 4];
#pragma unroll
      for (int q = 0; q < BS / 4; ++q) {
        const int64_t off = koff[warp + 4 * q];
        kr[q] = off >= 0 ? ld_kv4_bf16<kBf16>(a.k_pages, off + 4 * lane) : make_uint2(0u, 0u);
      }
#pragma unroll
      for (int q = 0; q < BS / 4; ++q)
        *reinterpret_cast<uint2*>(ks + sw128_offset(BS, warp + 4 * q, 4 * lane)) = kr[q];
    }
    // V^T: a warp takes 8 keys at a time; lane l loads dims 4l..4l+3 of each
    // (coalesced rows), then writes, for each of its 4 dims d, the 8 keys as
    // one 16-byte chunk of row d.  The order of the 4 dims is rotated by lane
    // so the 8 lanes of a store phase hit 8 different bank groups.
    for (int kc = warp; kc < BS / 8; kc += kThreads / 32) {
      float4 v[8];
#pragma unroll
      for (int uu = 0; uu < 8; ++uu) {
        const int64_t off = koff[kc * 8 + uu];
        v[uu] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (off >= 0) {
          if constexpr (kBf16) {
            v[uu] = bf16x4_to_f32(__ldg(reinterpret_cast<const uint2*>(
                static_cast<const uint16_t*>(a.v_pages) + off + 4 * lane)));
          } else {
            v[uu] = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(a.v_pages) + off) + lane);
          }
        }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int comp = ((lane >> 1) + i) & 3;
        float c8[8];
#pragma unroll
        for (int uu = 0; uu < 8; ++uu)
          c8[uu] = comp == 0 ? v[uu].x : comp == 1 ? v[uu].y : comp == 2 ? v[uu].z : v[uu].w;
        uint4 packed;
        packed.x = pack_bf16x2_rn(c8[0], c8[1]);
        packed.y = pack_bf16x2_rn(c8[2], c8[3]);
        packed.z = pack_bf16x2_rn(c8[4], c8[5]);
        packed.w = pack_bf16x2_rn(c8[6], c8[7]);
        const int d = 4 * lane + comp;
        *reinterpret_cast<uint4*>(vs + sw128_offset(kD, d, kc * 8)) = packed;
      }
    }

    // Keys present in the block (position inside the length, page not absent).
    uint32_t vmask[BS / 32];
#pragma unroll
    for (int c = 0; c < BS / 32; ++c) vmask[c] = __ballot_sync(0xffffffffu, kpos[c * 32 + lane] >= 0);

    const int rows = static_cast<int>((e1 - e0) * qhead);
    for (int rt = 0; rt < rows && ok; rt += kM) {
      const int nrows = min(kM, rows - rt);
      // ---- Q tile: lane l of warp w owns row 32w + l's query --------------------
      {
        const int r = warp * 32 + lane;
        int64_t my_src = -1;
        if (r < nrows) {
          const int row = rt + r;
          const int64_t qi = a.edges[2 * (e0 + row / qhead)];
          my_src = (qi * a.hq + static_cast<int64_t>(h) * qhead + row % qhead) * kD;
        }
        // All 32 row loads in flight before any is used.
        float4 v[32];
#pragma unroll
        for (int rr = 0; rr < 32; ++rr) {
          const int64_t src = __shfl_sync(0xffffffffu, my_src, rr);
          v[rr] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (src >= 0) v[rr] = __ldg(reinterpret_cast<const float4*>(a.q + src) + lane);
        }
#pragma unroll
        for (int rr = 0; rr < 32; ++rr) {
          const uint2 packed =
              make_uint2(pack_bf16x2_rn(v[rr].x, v[rr].y), pack_bf16x2_rn(v[rr].z, v[rr].w));
          *reinterpret_cast<uint2*>(qp + sw128_offset(kM, warp * 32 + rr, 4 * lane)) = packed;
        }
      }
      // This thread's row: last live key of the block under the causal limit.
      const bool row_ok = tid < nrows;
      int jlim = row_ok ? BS - 1 : -1;
      if (row_ok && a.causal) {
        const int row = rt + tid;
        const int64_t qi = a.edges[2 * (e0 + row / qhead)];
        const int64_t ql = qi - q0;
        const int64_t lim = lk >= qo ? lk - qo + ql : ql;
        const int64_t rel = lim - bstart;
        jlim = rel < -1 ? -1 : (rel > BS - 1 ? BS - 1 : static_cast<int>(rel));
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncthreads();
      tc_fence_after();

      // ---- S = Q K^T ------------------------------------------------------------
      if (tid == 0) {
        const uint32_t q_addr = smem_u32(qp);
        const uint32_t k_addr = smem_u32(ks);
#pragma unroll
        for (int st = 0; st < kD / 16; ++st) {
          const uint32_t panel = st >> 2;
          const uint32_t kb = (st & 3) * 32;
          mma_bf16(t_s, sw128_desc(q_addr + panel * kM * 128 + kb),
                   sw128_desc(k_addr + panel * BS * 128 + kb), idesc_bf16(kM, BS), st > 0);
        }
        mma_commit(bar);
      }
      bool got = mbar_wait_bounded(bar, phase);
      phase ^= 1u;
      if (__syncthreads_or(!got)) {
        if (tid == 0) report(status, SA_ERR_DEVICE_TIMEOUT);
        ok = false;
        break;
      }
      tc_fence_after();

      // ---- softmax of this thread's row; P overwrites the Q tile -----------------
      float m2 = -INFINITY;
      float sc[BS];
#pragma unroll
      for (int c = 0; c < BS / 32; ++c) {
        float v[32];
        tmem_ld32(t_s + lane_base + c * 32, v);
        tmem_ld_wait();
        // live keys of this chunk for this row: present and at or before jlim
        const int cut = jlim - c * 32;        // keys i <= cut are inside the limit
        const uint32_t inside = cut >= 31 ? 0xffffffffu : (cut < 0 ? 0u : ((2u << cut) - 1u));
        const uint32_t live = vmask[c] & inside;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          sc[c * 32 + i] = ((live >> i) & 1u) ? v[i] * qscale : -INFINITY;
          m2 = fmaxf(m2, sc[c * 32 + i]);
        }
      }
      const float msub = m2 == -INFINITY ? 0.f : m2;
      float l = 0.f;
#pragma unroll
      for (int j0 = 0; j0 < BS; j0 += 8) {
        float p8[8];
#pragma unroll
        for (int uu = 0; uu < 8; ++uu) {
          p8[uu] = exp2f(sc[j0 + uu] - msub);   // exp2(-inf) = 0
          l += p8[uu];
        }
        uint4 packed;
        packed.x = pack_bf16x2_rn(p8[0], p8[1]);
        packed.y = pack_bf16x2_rn(p8[2], p8[3]);
        packed.z = pack_bf16x2_rn(p8[4], p8[5]);
        packed.w = pack_bf16x2_rn(p8[6], p8[7]);
        *reinterpret_cast<uint4*>(qp + sw128_offset(kM, tid, j0)) = packed;
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncthreads();
      tc_fence_after();

      // ---- O = P V ----------------------------------------------------------------
      if (tid == 0) {
        const uint32_t p_addr = smem_u32(qp);
        const uint32_t v_addr = smem_u32(vs);
#pragma unroll
        for (int st = 0; st < BS / 16; ++st) {
          const uint32_t panel = st >> 2;
          const uint32_t kb = (st & 3) * 32;
          mma_bf16(t_o, sw128_desc(p_addr + panel * kM * 128 + kb),
                   sw128_desc(v_addr + panel * kD * 128 + kb), idesc_bf16(kM, kD), st > 0);
        }
        mma_commit(bar);
      }
      got = mbar_wait_bounded(bar, phase);
      phase ^= 1u;
      if (__syncthreads_or(!got)) {
        if (tid == 0) report(status, SA_ERR_DEVICE_TIMEOUT);
        ok = false;
        break;
      }
      tc_fence_after();

      // ---- epilogue: this thread's partial row -------------------------------------
      const int64_t prow = e0 * qhead + rt + tid;
#pragma unroll
      for (int c = 0; c < kD / 32; ++c) {
        float v[32];
        tmem_ld32(t_o + lane_base + c * 32, v);
        tmem_ld_wait();
        if (row_ok) {
          float4* dst = reinterpret_cast<float4*>(a.o_partial + prow * kD + c * 32);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
        }
      }
      if (row_ok) {
        a.m_partial[prow] = m2 == -INFINITY ? -INFINITY : m2 * kLn2;
        a.l_partial[prow] = l;
      }
      tc_fence_before();
      __syncthreads();   // S / O / the tile buffer are free for the next tile
      tc_fence_after();
    }
  }
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

template <int BS, bool kBf16>
cudaError_t launch_tc(const ForwardArgs& a, cudaStream_t stream) {
  const TcPlan p = tc_plan(BS);
  const void* fn = reinterpret_cast<const void*>(forward_tc_kernel<BS, kBf16>);
  cudaError_t err =
      cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(p.total));
  if (err != cudaSuccess) return err;
  err = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
  if (err != cudaSuccess) return err;
  // Two CTAs per SM when their shared memory fits (two CTAs x 256 TMEM
  // columns fill an SM's TMEM); the occupancy query is not used because it
  // reported one CTA where two fit.
  const int per_sm = 2 * (p.total + 1024) <= 228 * 1024 ? 2 : 1;
  int64_t grid = static_cast<int64_t>(device_sm_count()) * per_sm;
  if (grid > a.max_splits) grid = a.max_splits;
  if (grid < 1) grid = 1;
  forward_tc_kernel<BS, kBf16><<<static_cast<unsigned>(grid), kThreads, p.total, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

bool forward_tc_supported(int head_dim, int block_size, int page_size, int qhead) {
  if (head_dim != kD) return false;
  if (block_size != 64 && block_size != 128) return false;
  if (page_size <= 0 || block_size % page_size) return false;
  if (qhead <= 0 || kM % qhead) return false;
  return true;
}

cudaError_t launch_forward_tc(const ForwardArgs& a, cudaStream_t stream) {
  if (!forward_tc_supported(a.head_dim, a.block_size, a.page_size, a.qhead) || a.hkv > 200)
    return cudaErrorNotSupported;
  if (a.block_size == 64)
    return a.kv_bf16 ? launch_tc<64, true>(a, stream) : launch_tc<64, false>(a, stream);
  return a.kv_bf16 ? launch_tc<128, true>(a, stream) : launch_tc<128, false>(a, stream);
}

}  // namespace sa
