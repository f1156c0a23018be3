// Fused decode attention: steps 2 and 3 of KV-outer sparse attention
// (kvouter_forward and the log-sum-exp combine of its partials, forward.rs of
// alice-llm's sparse_attention) in one kernel, for batches in which every
// sequence holds at most one query.
//
// With one query per sequence, each work unit (kv head, block) carries edges
// of that query only, so all partials the combine merges for a (query, kv
// head) pair come from the pair's own kept ranks.  The kernel therefore walks
// the kept ranks of each pair and keeps the merge on chip: a "piece" is a
// range of ranks of one pair (normally all of them); its blocks stream through
// shared memory and one online softmax runs across them.  Where a pair is cut
// into several pieces (to fill the SMs in the last round of pairs, or when
// asked), they meet in a small global scratch (one (o, m, l) row per piece and
// GQA lane, normally still in L2); the last piece of the pair to finish
// merges them and writes out and lse.
// The causal mask is a no-op here: a sequence's only query sits at position
// lk - 1 and sees every key below lk.
//
// Warp roles of a CTA (persistent, one per SM, pieces round-robin):
//   warp 0    metadata: for each piece the query's sequence and KV length,
//             the kept ranks (inv >= 0) with their blocks and page ids, into
//             a ring of piece descriptors in shared memory;
//   warps 1-2 loads: for each 64-key chunk of a kept block, tensor-map copies
//             of its K and V pages with the 128-byte swizzle, plus the piece's
//             Q rows, into a ring of stages (the two warps take alternate
//             stages: the copies one warp issues alone fall well short of HBM
//             bandwidth);
//   warp 3    merge: merges the consumers' states of a finished piece and
//             writes the output (or the piece's scratch rows, the pair's
//             counter and, for the pair's last piece, the merge of its
//             scratch rows), beside the consumers;
//   warps 4.. consumers: each owns a slice of every chunk's keys and keeps its
//             own online-softmax state over the piece; at the end of a piece
//             they hand the states to the merge warp through shared memory
//             and go on (they wait for it only at their next piece's end).
// f32 K/V: 8 consumer warps x 8 keys on CUDA-core FMA; the piece's Q rows
// come with every stage (a 2 KB copy, from L2 after the first) in the same
// swizzled layout, so the scores read Q from shared memory without bank
// conflicts and hold no Q in registers.  bf16 K/V: 4 consumer warps x 16 keys
// on warp-level MMA (m16n8k16), Q and P split into bf16 high parts and
// remainders; with at most 8 q-heads per kv head the remainders ride in the
// tile's otherwise empty rows 8-15, so the split costs no extra MMA.
//
// Shared-memory layout of a stage (a 1024-byte aligned region per tensor):
//   f32:  [key][quarter of head_dim][32 floats], one 128-byte row per
//         (key, quarter), 16-byte chunks XOR-swizzled by (4 key + quarter) & 7;
//   bf16: [half of head_dim][key][64 bf16], one 128-byte row per (half, key),
//         chunks swizzled by key & 7.
// Both make the consumers' shared loads (and ldmatrix) bank-conflict free.
#include <cstdint>
#include <cuda.h>

#include "internal.h"
#include "sa_common.cuh"

namespace sa {

namespace {

constexpr int kD = 128;
constexpr int kCK = 64;              // keys per stage
constexpr int kMaxEP = 64;           // ranks per piece
constexpr int kMaxPPB = 8;           // pages per block
constexpr int kDescs = 4;            // piece descriptors in flight
constexpr uint32_t kFirst = 1u, kLast = 2u, kDone = 4u;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct TmaMaps {
  CUtensorMap k[2];   // f32: [0]; bf16: [0] low half, [1] high half of head_dim
  CUtensorMap v[2];
  CUtensorMap q;      // f32: q as rows of 32 floats (quarters of a head)
};

struct PieceDesc {
  int32_t item, k, i, h, lk, nr, pad0, pad1;
  int32_t blk[kMaxEP];                  // blocks of the kept ranks, in rank order
  int32_t pid[kMaxEP][kMaxPPB];         // their page ids (-1: absent)
};

struct StageHdr {
  uint32_t flags, mask_lo, mask_hi;     // keys of the chunk that exist
  int32_t item, k, pad0, pad1, pad2;
};

template <bool kBf16> struct Cfg;
// NC consumer warps (keys of a stage split between them), NL load warps
// (stages round-robin: one warp's copy issue alone does not keep HBM busy).
template <> struct Cfg<false> { static constexpr int NC = 8, NL = 2; };   // 8 keys per consumer
template <> struct Cfg<true> { static constexpr int NC = 4, NL = 3; };    // 16 keys per consumer

struct Layout {
  uint32_t tensor;     // bytes of K (or V) of one stage
  uint32_t stage;      // K + V
  uint32_t q, hdr, mo, mm, ml, desc, bars, flag, total;
};

__host__ __device__ constexpr uint32_t up_to(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

template <bool kBf16, int R, int S>
__host__ __device__ constexpr Layout fused_layout() {
  Layout L{};
  L.tensor = kCK * kD * (kBf16 ? 2 : 4);
  L.stage = 2 * L.tensor;
  L.q = S * L.stage;                                          // Q slots [S][R][128] f32
  L.hdr = L.q + S * R * kD * 4;                               // StageHdr[S]
  L.mo = up_to(L.hdr + S * static_cast<uint32_t>(sizeof(StageHdr)), 16);
  L.mm = L.mo + Cfg<kBf16>::NC * R * kD * 4;                  // merge rows [NC][R][128]
  L.ml = L.mm + Cfg<kBf16>::NC * R * 4;
  L.desc = up_to(L.ml + Cfg<kBf16>::NC * R * 4, 16);
  L.bars = up_to(L.desc + kDescs * static_cast<uint32_t>(sizeof(PieceDesc)), 8);
  L.flag = L.bars + (2 * S + 2 * kDescs + 2) * 8;           // merge info: item, k
  L.total = L.flag + 16;
  return L;
}

struct Smem {
  uint32_t spin;        // tries of every mbarrier wait
  unsigned char* base;
  float* qs;
  StageHdr* hdr;
  float* mo;
  float* mm;
  float* ml;
  PieceDesc* desc;
  uint64_t* full;
  uint64_t* empty;
  uint64_t* dfull;
  uint64_t* dempty;
  uint64_t* mready;     // consumers -> merge warp: the piece's states are in mo/mm/ml
  uint64_t* mfree;      // merge warp -> consumers: the states have been read
  volatile int* minfo;  // item, k of the piece being merged (-1: no more pieces)
};

// ------------------------------------------------------------------ metadata

// Sequence b of query i: the largest b with cu[b] <= i (cu[0] = 0 <= i <
// cu[batch]); 32 candidates per round.
__device__ __forceinline__ int warp_batch_of(const int64_t* cu, int batch, int64_t i, int lane) {
  int lo = 0, hi = batch;            // answer in [lo, hi)
  while (hi - lo > 1) {
    const int step = (hi - lo + 31) / 32;
    const int cand = lo + lane * step;
    const bool le = cand < hi && cu[cand] <= i;
    const unsigned bal = __ballot_sync(0xffffffffu, le);   // lane 0 (cand = lo) always set
    const int last = 31 - __clz(bal);
    const int nlo = lo + last * step;
    hi = min(nlo + step, hi);
    lo = nlo;
  }
  return lo;
}

__device__ void meta_warp(const FusedDecArgs& a, const Smem& sm, int64_t n_pieces, int lane) {
  uint32_t n = 0;
  for (int64_t g = blockIdx.x;; g += gridDim.x, ++n) {
    const int slot = static_cast<int>(n % kDescs);
    if (n >= static_cast<uint32_t>(kDescs) &&
        !mbar_wait_bounded(sm.dempty + slot, ((n / kDescs) - 1) & 1u, sm.spin)) {
      if (lane == 0) report(a.status, SA_ERR_DEVICE_TIMEOUT);
      return;
    }
    PieceDesc& d = sm.desc[slot];
    if (g >= n_pieces) {
      if (lane == 0) d.item = -1;
      __syncwarp();
      mbar_arrive(sm.dfull + slot);
      return;
    }
    int64_t item;
    int k, r0, nrange;
    if (g < a.whole_items) {            // a whole pair: all its ranks
      item = g;
      k = 0;
      r0 = 0;
      nrange = a.topk;
    } else {
      const int64_t t = g - a.whole_items;
      item = a.whole_items + t / a.pieces;
      k = static_cast<int>(t - (item - a.whole_items) * a.pieces);
      r0 = k * a.ranks_per_piece;
      nrange = min(a.ranks_per_piece, a.topk - r0);
    }
    const int64_t i = item / a.hkv;
    const int h = static_cast<int>(item - i * a.hkv);
    const int b = warp_batch_of(a.cu, a.batch, i, lane);
    const int lk = a.used ? max(a.used[b], 0) : a.msb * a.block_size;
    // Ranks r0 + lane and r0 + 32 + lane; kept ones compacted in rank order.
    int nkept = 0;
#pragma unroll
    for (int half = 0; half < kMaxEP / 32; ++half) {
      const int jr = 32 * half + lane;
      bool kept = false;
      int blk = 0;
      if (jr < nrange) {
        const int r = r0 + jr;
        // the index's rule for keeping an entry (its inv >= 0): a block id in
        // [0, msb) whose first key lies below the sequence's KV length
        blk = a.selected[(i * a.hkv + h) * a.topk + r];
        if (blk < -1 || blk >= a.msb) report(a.status, SA_ERR_SELECTED_RANGE);
        kept = blk >= 0 && blk < a.msb && static_cast<int64_t>(blk) * a.block_size < lk;
      }
      const unsigned km = __ballot_sync(0xffffffffu, kept);
      if (kept) {
        const int pos = nkept + __popc(km & ((1u << lane) - 1u));
        d.blk[pos] = blk;
        const int32_t* bt = a.block_tables + static_cast<int64_t>(b) * a.max_pages +
                            static_cast<int64_t>(blk) * a.pages_per_block;
        const int64_t key0 = static_cast<int64_t>(blk) * a.block_size;
#pragma unroll
        for (int p = 0; p < kMaxPPB; ++p) {
          int id = -1;
          if (p < a.pages_per_block && key0 + static_cast<int64_t>(p) * a.page_size < lk) {
            id = bt[p];
            if (id >= a.num_pages) {
              report(a.status, SA_ERR_SHAPE);
              id = -1;
            }
            if (id < 0) id = -1;
          }
          d.pid[pos][p] = id;
        }
      }
      nkept += __popc(km);
    }
    if (lane == 0) {
      d.item = static_cast<int>(item);
      d.k = k;
      d.i = static_cast<int>(i);
      d.h = h;
      d.lk = lk;
      d.nr = nkept;
    }
    __syncwarp();
    mbar_arrive(sm.dfull + slot);
  }
}

// ------------------------------------------------------------------ loads

// Load warp lw of NL: fills the stages whose running index is lw modulo NL.
template <bool kBf16, int R, int S>
__device__ void load_warp(const TmaMaps& maps, const FusedDecArgs& a, const Smem& sm, int lw,
                          int lane) {
  constexpr Layout L = fused_layout<kBf16, R, S>();
  constexpr uint32_t NL = Cfg<kBf16>::NL;
  const int ck = a.block_size < kCK ? a.block_size : kCK;           // keys per chunk
  const int cpb = a.block_size / ck;                                // chunks per block
  const int kb = a.page_size < ck ? a.page_size : ck;               // keys per page box
  const int nbox = ck / kb;
  const uint32_t box_bytes = static_cast<uint32_t>(kb) * kD * (kBf16 ? 2 : 4);
  const uint32_t q_bytes = static_cast<uint32_t>(a.qhead) * kD * 4;
  uint32_t n = 0, xs = 0;
  bool ok = true;
  if (a.stall) return;   // test hook: no stage is ever filled, so every wait on one runs out
  for (;;) {
    const int slot = static_cast<int>(n % kDescs);
    if (!mbar_wait_bounded(sm.dfull + slot, (n / kDescs) & 1u, sm.spin)) {
      ok = false;
      break;
    }
    const PieceDesc& d = sm.desc[slot];
    const int item = d.item;
    if (item < 0) {
      if (xs % NL != static_cast<uint32_t>(lw)) break;   // another load warp ends the ring
      const int s = static_cast<int>(xs % S);
      if (xs >= static_cast<uint32_t>(S) && !mbar_wait_bounded(sm.empty + s, ((xs / S) - 1) & 1u, sm.spin)) {
        ok = false;
        break;
      }
      if (lane == 0) {
        sm.hdr[s].flags = kDone;
        mbar_arrive(sm.full + s);
      }
      ++xs;
      break;
    }
    const int nr = d.nr, lk = d.lk, h = d.h;
    const int nst = nr == 0 ? 1 : nr * cpb;
    for (int u = 0; u < nst; ++u) {
      if (xs % NL != static_cast<uint32_t>(lw)) {    // another load warp's stage
        ++xs;
        continue;
      }
      const int j = u / cpb, c = u - j * cpb;
      const int s = static_cast<int>(xs % S);
      if (xs >= static_cast<uint32_t>(S) && !mbar_wait_bounded(sm.empty + s, ((xs / S) - 1) & 1u, sm.spin)) {
        ok = false;
        break;
      }
      const bool first = u == 0, last = u == nst - 1;
      uint32_t mlo = 0, mhi = 0;
      bool present = false;
      int row0 = 0;
      if (nr > 0) {
        const int blk = d.blk[j];
        const int64_t pos0 = static_cast<int64_t>(blk) * a.block_size + c * ck;
        // lanes t and t + 32: does chunk key t exist?
        int t = lane;
        const bool e0 = t < ck && pos0 + t < lk && d.pid[j][(c * ck + t) / a.page_size] >= 0;
        t = lane + 32;
        const bool e1 = t < ck && pos0 + t < lk && d.pid[j][(c * ck + t) / a.page_size] >= 0;
        mlo = __ballot_sync(0xffffffffu, e0);
        mhi = __ballot_sync(0xffffffffu, e1);
        if (lane < nbox) {
          const int kk0 = c * ck + lane * kb;           // block key of the box's first row
          const int p = kk0 / a.page_size;
          const int id = d.pid[j][p];
          present = id >= 0 && pos0 + lane * kb < lk;
          if (present)
            row0 = static_cast<int>((static_cast<int64_t>(id) * a.hkv + h) * a.page_size +
                                    (kk0 - p * a.page_size));
        }
      }
      const unsigned pm = __ballot_sync(0xffffffffu, present);
      const bool with_q = kBf16 ? (first && nr > 0) : nr > 0;
      const uint32_t tx =
          static_cast<uint32_t>(__popc(pm)) * 2u * box_bytes + (with_q ? q_bytes : 0u);
      if (lane == 0) {
        StageHdr& hd = sm.hdr[s];
        hd.flags = (first ? kFirst : 0u) | (last ? kLast : 0u);
        hd.mask_lo = mlo;
        hd.mask_hi = mhi;
        hd.item = item;
        hd.k = d.k;
        mbar_arrive_expect_tx(sm.full + s, tx);
      }
      __syncwarp();
      unsigned char* st = sm.base + s * L.stage;
      if (present) {
        if constexpr (kBf16) {
          const uint32_t off = static_cast<uint32_t>(lane * kb) * 128u;
          tma_load_2d(st + off, &maps.k[0], 0, row0, sm.full + s);
          tma_load_2d(st + kCK * 128 + off, &maps.k[1], 0, row0, sm.full + s);
          tma_load_2d(st + L.tensor + off, &maps.v[0], 0, row0, sm.full + s);
          tma_load_2d(st + L.tensor + kCK * 128 + off, &maps.v[1], 0, row0, sm.full + s);
        } else {
          const uint32_t off = static_cast<uint32_t>(lane * kb) * 512u;
          tma_load_3d(st + off, &maps.k[0], 0, 0, row0, sm.full + s);
          tma_load_3d(st + L.tensor + off, &maps.v[0], 0, 0, row0, sm.full + s);
        }
      }
      if (with_q && lane == 31) {
        const int64_t qrow = static_cast<int64_t>(d.i) * a.hq + static_cast<int64_t>(h) * a.qhead;
        if constexpr (kBf16)
          bulk_g2s(sm.qs + s * R * kD, a.q + qrow * kD, q_bytes, sm.full + s);
        else
          tma_load_2d(sm.qs + s * R * kD, &maps.q, 0, static_cast<int>(qrow * 4), sm.full + s);
      }
      ++xs;
    }
    if (!ok) break;
    __syncwarp();
    mbar_arrive(sm.dempty + slot);
    ++n;
  }
  if (!ok) {
    if (lane == 0) report(a.status, SA_ERR_DEVICE_TIMEOUT);
    // Let this warp's copies still in flight land before the CTA can exit.
    for (uint32_t x = xs > static_cast<uint32_t>(S) ? xs - S : 0u; x < xs; ++x)
      if (x % NL == static_cast<uint32_t>(lw)) mbar_wait_bounded(sm.full + x % S, (x / S) & 1u, sm.spin);
  }
}

// ------------------------------------------------------------------ piece end

__device__ __forceinline__ void write_row(const FusedDecArgs& a, int64_t row, int d4, float m2,
                                          float l, float4 o) {
  const float inv = l > 0.f ? 1.f / l : 0.f;
  reinterpret_cast<float4*>(a.out + row * kD)[d4] =
      make_float4(o.x * inv, o.y * inv, o.z * inv, o.w * inv);
  if (a.lse && d4 == 0) a.lse[row] = l > 0.f ? (m2 + log2f(l)) * kLn2 : -INFINITY;
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int off = 16; off; off >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, off));
  return x;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int off = 16; off; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
  return x;
}

// The merge warp.  Per piece: merge the NC consumer warps' states (m in the
// log2 domain) row by row, lane = 4 dims; release the state buffer; then
// either write the output rows (one piece per pair) or the piece's scratch
// rows, and if this piece is the pair's last to finish (a counter per pair),
// merge the pair's scratch rows into the output.  It runs beside the
// consumers, which only wait for it when they hand over their next piece.
template <int NC, int R>
__device__ void merge_warp(const FusedDecArgs& a, const Smem& sm, int lane) {
  const int qhead = a.qhead;
  for (uint32_t np = 0;; ++np) {
    if (!mbar_wait_bounded(sm.mready, np & 1u, sm.spin)) {
      if (lane == 0) report(a.status, SA_ERR_DEVICE_TIMEOUT);
      return;
    }
    const int item = sm.minfo[0];
    const int k = sm.minfo[1];
    if (item < 0) return;
    const int P = item < a.whole_items ? 1 : a.pieces;
    const int64_t i = item / a.hkv;
    const int h = item - static_cast<int>(i) * a.hkv;
    const int64_t row0 = i * a.hq + static_cast<int64_t>(h) * qhead;
    // scratch row of (pair, piece kk, lane r): (item * topk + kk) * qhead + r
    const int64_t prow = static_cast<int64_t>(item) * a.topk * qhead;
    for (int r = 0; r < qhead; ++r) {
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < NC; ++w) M = fmaxf(M, sm.mm[w * R + r]);
      float l = 0.f;
      float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
      if (M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < NC; ++w) {
          const float e = exp2f(sm.mm[w * R + r] - M);
          l = fmaf(e, sm.ml[w * R + r], l);
          const float4 v = reinterpret_cast<const float4*>(sm.mo + (w * R + r) * kD)[lane];
          o.x = fmaf(e, v.x, o.x);
          o.y = fmaf(e, v.y, o.y);
          o.z = fmaf(e, v.z, o.z);
          o.w = fmaf(e, v.w, o.w);
        }
      }
      if (P == 1) {
        write_row(a, row0 + r, lane, M, l, o);
      } else {
        const int64_t pr = prow + static_cast<int64_t>(k) * qhead + r;
        store_o4(a.part_o, a.part_bf16, pr * kD + 4 * lane, o);
        if (lane == 0) {
          a.part_m[pr] = M;
          a.part_l[pr] = l;
        }
      }
    }
    __syncwarp();
    mbar_arrive(sm.mfree);
    if (P == 1) continue;
    __threadfence();
    unsigned last = 0;
    if (lane == 0) {
      const unsigned old = atomicAdd(a.item_cnt + item, 1u);
      last = old == static_cast<unsigned>(P - 1);
      if (last) atomicExch(a.item_cnt + item, 0u);
    }
    last = __shfl_sync(0xffffffffu, last, 0);
    if (!last) continue;
    __threadfence();
    // The pair's P scratch rows per GQA lane: statistics one piece per lane,
    // then the o rows, eight loads in flight.
    for (int r = 0; r < qhead; ++r) {
      const int64_t pr0 = prow + r;
      float M = -INFINITY;
      for (int b = 0; b < P; b += 32)
        if (b + lane < P) M = fmaxf(M, __ldcg(a.part_m + pr0 + static_cast<int64_t>(b + lane) * qhead));
      M = warp_max(M);
      float l = 0.f;
      float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
      if (M != -INFINITY) {
        for (int b = 0; b < P; b += 32) {
          float e = 0.f;
          if (b + lane < P) {
            const int64_t pr = pr0 + static_cast<int64_t>(b + lane) * qhead;
            e = exp2f(__ldcg(a.part_m + pr) - M);
            l = fmaf(e, __ldcg(a.part_l + pr), l);
          }
          const int n = min(32, P - b);
          for (int t0 = 0; t0 < n; t0 += 8) {
            float wt[8];
            float4 v[8];
#pragma unroll
            for (int t = 0; t < 8; ++t) {
              wt[t] = __shfl_sync(0xffffffffu, e, (t0 + t) & 31);
              v[t] = make_float4(0.f, 0.f, 0.f, 0.f);
              if (t0 + t < n && wt[t] > 0.f) {
                const int64_t e = (pr0 + static_cast<int64_t>(b + t0 + t) * qhead) * kD + 4 * lane;
                v[t] = a.part_bf16
                           ? bf16x4_to_f32(__ldcg(reinterpret_cast<const uint2*>(
                                 static_cast<const uint16_t*>(a.part_o) + e)))
                           : __ldcg(reinterpret_cast<const float4*>(
                                 static_cast<const float*>(a.part_o) + e));
              }
            }
#pragma unroll
            for (int t = 0; t < 8; ++t) {
              const float ww = t0 + t < n ? wt[t] : 0.f;
              o.x = fmaf(ww, v[t].x, o.x);
              o.y = fmaf(ww, v[t].y, o.y);
              o.z = fmaf(ww, v[t].z, o.z);
              o.w = fmaf(ww, v[t].w, o.w);
            }
          }
        }
        l = warp_sum(l);
      }
      write_row(a, row0 + r, lane, M, l, o);
    }
  }
}

// Consumer side of a piece's end: wait until the merge warp has read the
// previous piece's states (bounded), then the caller writes its state.
__device__ __forceinline__ bool handoff_wait(const Smem& sm, uint32_t handed) {
  return handed == 0 || mbar_wait_bounded(sm.mfree, (handed - 1) & 1u, sm.spin);
}

// After the caller's state is written: consumer 0 names the piece, every
// consumer thread arrives.
__device__ __forceinline__ void handoff_signal(const Smem& sm, int w, int lane, int item, int k) {
  if (w == 0 && lane == 0) {
    sm.minfo[0] = item;
    sm.minfo[1] = k;
  }
  mbar_arrive(sm.mready);
}

// ------------------------------------------------------------------ f32 consumers

template <int R, int S>
__device__ void consumer_f32(const FusedDecArgs& a, const Smem& sm, int w, int lane) {
  constexpr Layout L = fused_layout<false, R, S>();
  const int ck = a.block_size < kCK ? a.block_size : kCK;
  const int kb = a.page_size < ck ? a.page_size : ck;
  const int lkb = __ffs(kb) - 1;                  // kb is a power of two
  // Scores: lane = (key k8 of the warp's 8, quarter qd of head_dim).
  const int k8 = lane >> 2, qd = lane & 3;
  const int t = 8 * w + k8;
  const uint32_t krow = static_cast<uint32_t>((t >> lkb) * kb * 4 + (t & (kb - 1)) * 4 + qd);
  const uint32_t koff = krow * 128u;
  const uint32_t kx = krow & 7u;
  // PV: lane = 4 output dims: quarter vq, 16-byte chunk vc.
  const int vq = lane >> 3, vc = lane & 7;
  const float qscale = a.scale * kLog2e;

  float m_run[R], l_run[R];
  float4 o[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    m_run[r] = -INFINITY;
    l_run[r] = 0.f;
    o[r] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  uint32_t xc = 0, handed = 0;
  for (;;) {
    const int s = static_cast<int>(xc % S);
    if (!mbar_wait_bounded(sm.full + s, (xc / S) & 1u, sm.spin)) {
      if (lane == 0) report(a.status, SA_ERR_DEVICE_TIMEOUT);
      return;
    }
    const StageHdr hd = sm.hdr[s];
    if (hd.flags & kDone) {
      if (handoff_wait(sm, handed)) handoff_signal(sm, w, lane, -1, 0);
      return;
    }
    const unsigned char* kt = sm.base + s * L.stage;
    const unsigned char* vt = kt + L.tensor;
    // Q rows of the piece: row 4 r + quarter, chunks swizzled like K.
    const unsigned char* qt = reinterpret_cast<const unsigned char*>(sm.qs + s * R * kD);
    if (hd.flags & kFirst) {
#pragma unroll
      for (int r = 0; r < R; ++r) {
        m_run[r] = -INFINITY;
        l_run[r] = 0.f;
        o[r] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    const uint32_t mk = ((w < 4 ? hd.mask_lo >> (8 * w) : hd.mask_hi >> (8 * (w - 4)))) & 0xFFu;
    if (mk) {
      float acc[R][2];
#pragma unroll
      for (int r = 0; r < R; ++r) acc[r][0] = acc[r][1] = 0.f;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const float4 kv = *reinterpret_cast<const float4*>(kt + koff + ((c ^ kx) << 4));
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const uint32_t qrow = static_cast<uint32_t>(4 * r + qd);
          const float4 qv =
              *reinterpret_cast<const float4*>(qt + qrow * 128u + ((c ^ (qrow & 7u)) << 4));
          float x = acc[r][c & 1];
          x = fmaf(qv.x, kv.x, x);
          x = fmaf(qv.y, kv.y, x);
          x = fmaf(qv.z, kv.z, x);
          x = fmaf(qv.w, kv.w, x);
          acc[r][c & 1] = x;
        }
      }
      const bool valid = (mk >> k8) & 1u;
      float p[R];
#pragma unroll
      for (int r = 0; r < R; ++r) {
        float sc = acc[r][0] + acc[r][1];
        sc += __shfl_xor_sync(0xffffffffu, sc, 1);
        sc += __shfl_xor_sync(0xffffffffu, sc, 2);
        sc = valid ? sc * qscale : -INFINITY;
        float cm = sc;
        cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, 4));
        cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, 8));
        cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, 16));
        // cm is finite: the warp has a key (mk != 0)
        const float m_new = fmaxf(m_run[r], cm);
        const float alpha = exp2f(m_run[r] - m_new);
        p[r] = valid ? exp2f(sc - m_new) : 0.f;
        l_run[r] = fmaf(l_run[r], alpha, p[r]);
        m_run[r] = m_new;
        o[r].x *= alpha;
        o[r].y *= alpha;
        o[r].z *= alpha;
        o[r].w *= alpha;
      }
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        if (!((mk >> jj) & 1u)) continue;             // warp-uniform
        const int tj = 8 * w + jj;
        const uint32_t vrow =
            static_cast<uint32_t>((tj >> lkb) * kb * 4 + (tj & (kb - 1)) * 4 + vq);
        const float4 vv =
            *reinterpret_cast<const float4*>(vt + vrow * 128u + ((vc ^ (vrow & 7u)) << 4));
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const float pj = __shfl_sync(0xffffffffu, p[r], jj * 4);
          o[r].x = fmaf(pj, vv.x, o[r].x);
          o[r].y = fmaf(pj, vv.y, o[r].y);
          o[r].z = fmaf(pj, vv.z, o[r].z);
          o[r].w = fmaf(pj, vv.w, o[r].w);
        }
      }
    }
    mbar_arrive(sm.empty + s);
    if (hd.flags & kLast) {
      if (!handoff_wait(sm, handed)) {
        if (lane == 0) report(a.status, SA_ERR_DEVICE_TIMEOUT);
        return;
      }
#pragma unroll
      for (int r = 0; r < R; ++r) {
        float lw = qd == 0 ? l_run[r] : 0.f;
        lw += __shfl_xor_sync(0xffffffffu, lw, 4);
        lw += __shfl_xor_sync(0xffffffffu, lw, 8);
        lw += __shfl_xor_sync(0xffffffffu, lw, 16);
        reinterpret_cast<float4*>(sm.mo + (w * R + r) * kD)[lane] = o[r];
        if (lane == 0) {
          sm.mm[w * R + r] = m_run[r];
          sm.ml[w * R + r] = lw;
        }
      }
      handoff_signal(sm, w, lane, hd.item, hd.k);
      ++handed;
    }
    ++xc;
  }
}

// ------------------------------------------------------------------ bf16 consumers

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

// Split two values into bf16 high parts and bf16 remainders.
__device__ __forceinline__ void split2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  hi = bf2(x0, x1);
  lo = bf2(x0 - __uint_as_float(hi << 16), x1 - __uint_as_float(hi & 0xFFFF0000u));
}

template <int R, int S>
__device__ void consumer_bf16(const FusedDecArgs& a, const Smem& sm, int w, int lane) {
  static_assert(R == 16, "rows g and g + 8 of the m16 tile are both query rows");
  constexpr Layout L = fused_layout<true, R, S>();
  const int g = lane >> 2, c = lane & 3;          // fragment row (and + 8), column pair
  const int mi = lane >> 3, ri = lane & 7;        // ldmatrix matrix and row
  // K rows for S = Q K^T: matrices (keys 0-7 | 8-15) x (dims lo | hi 8 of 16).
  const uint32_t krow = static_cast<uint32_t>(16 * w + (mi >> 1) * 8 + ri) * 128u;
  // V rows for O += P V (transposed): matrices (keys 0-7 | 8-15) x (dims).
  const uint32_t vrow = static_cast<uint32_t>(16 * w + (mi & 1) * 8 + ri) * 128u;
  const float qscale = a.scale * kLog2e;

  float m_run[2] = {-INFINITY, -INFINITY};
  float l_part[2] = {0.f, 0.f};
  float o[16][4];
  uint32_t qhi[8][4], qlo[8][4];
#pragma unroll
  for (int nt = 0; nt < 16; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[nt][e] = 0.f;
#pragma unroll
  for (int ks = 0; ks < 8; ++ks)
#pragma unroll
    for (int e = 0; e < 4; ++e) qhi[ks][e] = qlo[ks][e] = 0u;

  uint32_t xc = 0, handed = 0;
  for (;;) {
    const int s = static_cast<int>(xc % S);
    if (!mbar_wait_bounded(sm.full + s, (xc / S) & 1u, sm.spin)) {
      if (lane == 0) report(a.status, SA_ERR_DEVICE_TIMEOUT);
      return;
    }
    const StageHdr hd = sm.hdr[s];
    if (hd.flags & kDone) {
      if (handoff_wait(sm, handed)) handoff_signal(sm, w, lane, -1, 0);
      return;
    }
    const uint32_t kt = smem_u32(sm.base + s * L.stage);
    const uint32_t vt = kt + L.tensor;
    if (hd.flags & kFirst) {
      const float* qg = sm.qs + s * R * kD;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
#pragma unroll
        for (int part = 0; part < 4; ++part) {
          const int r = g + ((part & 1) ? 8 : 0);
          const int col = 16 * ks + 2 * c + ((part & 2) ? 8 : 0);
          float2 v = make_float2(0.f, 0.f);
          if (r < a.qhead) v = *reinterpret_cast<const float2*>(qg + r * kD + col);
          split2(v.x * qscale, v.y * qscale, qhi[ks][part], qlo[ks][part]);
        }
      }
      m_run[0] = m_run[1] = -INFINITY;
      l_part[0] = l_part[1] = 0.f;
#pragma unroll
      for (int nt = 0; nt < 16; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[nt][e] = 0.f;
    }
    const uint32_t mk = (w < 2 ? hd.mask_lo >> (16 * w) : hd.mask_hi >> (16 * (w - 2))) & 0xFFFFu;
    if (mk) {
      // ---- S = Q K^T for the warp's 16 keys (two n-tiles of 8) ----
      float sacc[2][4];
      {
        float part[4][2][4];
#pragma unroll
        for (int qq = 0; qq < 4; ++qq)
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) part[qq][nt][e] = 0.f;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t chunk = static_cast<uint32_t>(((ks & 3) << 1) | (mi & 1));
          uint32_t b[4];
          ldsm_x4(kt + (ks >> 2) * (kCK * 128) + krow + ((chunk ^ ri) << 4), b);
          const int qq = (ks & 1) * 2;
          mma16816(part[qq][0], qhi[ks], b[0], b[1]);
          mma16816(part[qq + 1][0], qlo[ks], b[0], b[1]);
          mma16816(part[qq][1], qhi[ks], b[2], b[3]);
          mma16816(part[qq + 1][1], qlo[ks], b[2], b[3]);
        }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e)
            sacc[nt][e] = (part[0][nt][e] + part[2][nt][e]) + (part[1][nt][e] + part[3][nt][e]);
      }
      // ---- online softmax on the fragments (rows g and g + 8) ----
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
            float& sv = sacc[nt][2 * h2 + e];
            sv = ((mk >> kk) & 1u) ? sv : -INFINITY;
            cm = fmaxf(cm, sv);
          }
        cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, 1));
        cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, 2));
        const float m_new = fmaxf(m_run[h2], cm);      // finite: the warp has a key
        alpha[h2] = exp2f(m_run[h2] - m_new);
        float lsum = 0.f;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float pe = exp2f(sacc[nt][2 * h2 + e] - m_new);
            pv[nt][2 * h2 + e] = pe;
            lsum += pe;
          }
        l_part[h2] = fmaf(l_part[h2], alpha[h2], lsum);
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
      uint32_t phi[4], plo[4];
      split2(pv[0][0], pv[0][1], phi[0], plo[0]);
      split2(pv[0][2], pv[0][3], phi[1], plo[1]);
      split2(pv[1][0], pv[1][1], phi[2], plo[2]);
      split2(pv[1][2], pv[1][3], phi[3], plo[3]);
      // ---- O += P V (16 n-tiles of 8 dims) ----
#pragma unroll
      for (int np = 0; np < 8; ++np) {
        const uint32_t chunk = static_cast<uint32_t>(((np & 3) << 1) | (mi >> 1));
        uint32_t b[4];
        ldsm_x4_t(vt + (np >> 2) * (kCK * 128) + vrow + ((chunk ^ ri) << 4), b);
        mma16816(o[2 * np], phi, b[0], b[1]);
        mma16816(o[2 * np], plo, b[0], b[1]);
        mma16816(o[2 * np + 1], phi, b[2], b[3]);
        mma16816(o[2 * np + 1], plo, b[2], b[3]);
      }
    }
    mbar_arrive(sm.empty + s);
    if (hd.flags & kLast) {
      if (!handoff_wait(sm, handed)) {
        if (lane == 0) report(a.status, SA_ERR_DEVICE_TIMEOUT);
        return;
      }
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        float l = l_part[h2];
        l += __shfl_xor_sync(0xffffffffu, l, 1);
        l += __shfl_xor_sync(0xffffffffu, l, 2);
        const int r = g + 8 * h2;
        if (r < R) {
          float* dst = sm.mo + (w * R + r) * kD + 2 * c;
#pragma unroll
          for (int nt = 0; nt < 16; ++nt)
            *reinterpret_cast<float2*>(dst + 8 * nt) = make_float2(o[nt][2 * h2], o[nt][2 * h2 + 1]);
          if (c == 0) {
            sm.mm[w * R + r] = m_run[h2];
            sm.ml[w * R + r] = l;
          }
        }
      }
      handoff_signal(sm, w, lane, hd.item, hd.k);
      ++handed;
    }
    ++xc;
  }
}

// Up to 8 query rows (qhead <= 8): rows g + 8 of the m16 tile carry the bf16
// remainders of rows g, for Q in S = Q K^T and for P in O += P V, so the
// split costs no extra MMA; accumulator rows g and g + 8 are summed.
template <int S>
__device__ void consumer_bf16_packed(const FusedDecArgs& a, const Smem& sm, int w, int lane) {
  constexpr int R = 8;
  constexpr Layout L = fused_layout<true, R, S>();
  const int g = lane >> 2, c = lane & 3;          // fragment row, column pair
  const int mi = lane >> 3, ri = lane & 7;        // ldmatrix matrix and row
  const uint32_t krow = static_cast<uint32_t>(16 * w + (mi >> 1) * 8 + ri) * 128u;
  const uint32_t vrow = static_cast<uint32_t>(16 * w + (mi & 1) * 8 + ri) * 128u;
  const float qscale = a.scale * kLog2e;

  float m_run = -INFINITY;
  float l_part = 0.f;
  float o[16][4];           // [n-tile][row g: 0-1 | row g + 8 (remainder part): 2-3]
  uint32_t qa[8][4];        // A fragments: high parts in rows g, remainders in rows g + 8
#pragma unroll
  for (int nt = 0; nt < 16; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[nt][e] = 0.f;
#pragma unroll
  for (int ks = 0; ks < 8; ++ks)
#pragma unroll
    for (int e = 0; e < 4; ++e) qa[ks][e] = 0u;

  uint32_t xc = 0, handed = 0;
  for (;;) {
    const int s = static_cast<int>(xc % S);
    if (!mbar_wait_bounded(sm.full + s, (xc / S) & 1u, sm.spin)) {
      if (lane == 0) report(a.status, SA_ERR_DEVICE_TIMEOUT);
      return;
    }
    const StageHdr hd = sm.hdr[s];
    if (hd.flags & kDone) {
      if (handoff_wait(sm, handed)) handoff_signal(sm, w, lane, -1, 0);
      return;
    }
    const uint32_t kt = smem_u32(sm.base + s * L.stage);
    const uint32_t vt = kt + L.tensor;
    if (hd.flags & kFirst) {
      const float* qg = sm.qs + s * R * kD;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          float2 v = make_float2(0.f, 0.f);
          if (g < a.qhead) v = *reinterpret_cast<const float2*>(qg + g * kD + 16 * ks + 2 * c + 8 * half);
          split2(v.x * qscale, v.y * qscale, qa[ks][2 * half], qa[ks][2 * half + 1]);
        }
      }
      m_run = -INFINITY;
      l_part = 0.f;
#pragma unroll
      for (int nt = 0; nt < 16; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[nt][e] = 0.f;
    }
    const uint32_t mk = (w < 2 ? hd.mask_lo >> (16 * w) : hd.mask_hi >> (16 * (w - 2))) & 0xFFFFu;
    if (mk) {
      // ---- S = Q K^T for the warp's 16 keys: two chains (even / odd k-steps) ----
      float sc[2][2];
      {
        float part[2][2][4];
#pragma unroll
        for (int qq = 0; qq < 2; ++qq)
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) part[qq][nt][e] = 0.f;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t chunk = static_cast<uint32_t>(((ks & 3) << 1) | (mi & 1));
          uint32_t b[4];
          ldsm_x4(kt + (ks >> 2) * (kCK * 128) + krow + ((chunk ^ ri) << 4), b);
          mma16816(part[ks & 1][0], qa[ks], b[0], b[1]);
          mma16816(part[ks & 1][1], qa[ks], b[2], b[3]);
        }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e)
            sc[nt][e] = (part[0][nt][e] + part[0][nt][e + 2]) + (part[1][nt][e] + part[1][nt][e + 2]);
      }
      // ---- online softmax of row g ----
      float cm = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int kk = 8 * nt + 2 * c + e;
          sc[nt][e] = ((mk >> kk) & 1u) ? sc[nt][e] : -INFINITY;
          cm = fmaxf(cm, sc[nt][e]);
        }
      cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, 1));
      cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, 2));
      const float m_new = fmaxf(m_run, cm);          // finite: the warp has a key
      const float alpha = exp2f(m_run - m_new);
      float pv[2][2];
      float lsum = 0.f;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          pv[nt][e] = exp2f(sc[nt][e] - m_new);
          lsum += pv[nt][e];
        }
      l_part = fmaf(l_part, alpha, lsum);
      m_run = m_new;
      if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
        for (int nt = 0; nt < 16; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) o[nt][e] *= alpha;
      }
      uint32_t pa[4];
      split2(pv[0][0], pv[0][1], pa[0], pa[1]);
      split2(pv[1][0], pv[1][1], pa[2], pa[3]);
      // ---- O += P V (16 n-tiles of 8 dims) ----
#pragma unroll
      for (int np = 0; np < 8; ++np) {
        const uint32_t chunk = static_cast<uint32_t>(((np & 3) << 1) | (mi >> 1));
        uint32_t b[4];
        ldsm_x4_t(vt + (np >> 2) * (kCK * 128) + vrow + ((chunk ^ ri) << 4), b);
        mma16816(o[2 * np], pa, b[0], b[1]);
        mma16816(o[2 * np + 1], pa, b[2], b[3]);
      }
    }
    mbar_arrive(sm.empty + s);
    if (hd.flags & kLast) {
      if (!handoff_wait(sm, handed)) {
        if (lane == 0) report(a.status, SA_ERR_DEVICE_TIMEOUT);
        return;
      }
      float l = l_part;
      l += __shfl_xor_sync(0xffffffffu, l, 1);
      l += __shfl_xor_sync(0xffffffffu, l, 2);
      float* dst = sm.mo + (w * R + g) * kD + 2 * c;
#pragma unroll
      for (int nt = 0; nt < 16; ++nt)
        *reinterpret_cast<float2*>(dst + 8 * nt) =
            make_float2(o[nt][0] + o[nt][2], o[nt][1] + o[nt][3]);
      if (c == 0) {
        sm.mm[w * R + g] = m_run;
        sm.ml[w * R + g] = l;
      }
      handoff_signal(sm, w, lane, hd.item, hd.k);
      ++handed;
    }
    ++xc;
  }
}

// ------------------------------------------------------------------ kernel

template <bool kBf16, int R, int S>
__global__ void __launch_bounds__((2 + Cfg<kBf16>::NL + Cfg<kBf16>::NC) * 32, 1)
fused_dec_kernel(const __grid_constant__ TmaMaps maps, const FusedDecArgs a) {
  extern __shared__ unsigned char smem_raw[];
  constexpr Layout L = fused_layout<kBf16, R, S>();
  constexpr int NC = Cfg<kBf16>::NC;
  constexpr int NL = Cfg<kBf16>::NL;
  unsigned char* base = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  Smem sm;
  sm.spin = a.spin_limit ? a.spin_limit : kSpinLimit;
  sm.base = base;
  sm.qs = reinterpret_cast<float*>(base + L.q);
  sm.hdr = reinterpret_cast<StageHdr*>(base + L.hdr);
  sm.mo = reinterpret_cast<float*>(base + L.mo);
  sm.mm = reinterpret_cast<float*>(base + L.mm);
  sm.ml = reinterpret_cast<float*>(base + L.ml);
  sm.desc = reinterpret_cast<PieceDesc*>(base + L.desc);
  sm.full = reinterpret_cast<uint64_t*>(base + L.bars);
  sm.empty = sm.full + S;
  sm.dfull = sm.empty + S;
  sm.dempty = sm.dfull + kDescs;
  sm.mready = sm.dempty + kDescs;
  sm.mfree = sm.mready + 1;
  sm.minfo = reinterpret_cast<volatile int*>(base + L.flag);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(sm.full + s, 1);
      mbar_init(sm.empty + s, NC * 32);
    }
    for (int d = 0; d < kDescs; ++d) {
      mbar_init(sm.dfull + d, 32);
      mbar_init(sm.dempty + d, 32 * Cfg<kBf16>::NL);
    }
    mbar_init(sm.mready, NC * 32);
    mbar_init(sm.mfree, 32);
    fence_mbar_init();
  }
  // Keys (and Q rows past qhead) that are never copied enter products that
  // are discarded or multiplied by p = 0: keep them finite.
  for (uint32_t off = threadIdx.x * 16u; off < L.hdr; off += blockDim.x * 16u)
    *reinterpret_cast<float4*>(base + off) = make_float4(0.f, 0.f, 0.f, 0.f);
  fence_proxy_async_smem();
  __syncthreads();

  const int64_t n_pieces = a.whole_items + (a.tq * a.hkv - a.whole_items) * a.pieces;
  if (warp == 0) {
    meta_warp(a, sm, n_pieces, lane);
  } else if (warp <= NL) {
    load_warp<kBf16, R, S>(maps, a, sm, warp - 1, lane);
  } else if (warp == NL + 1) {
    merge_warp<NC, R>(a, sm, lane);
  } else if constexpr (kBf16) {
    if constexpr (R == 8)
      consumer_bf16_packed<S>(a, sm, warp - NL - 2, lane);
    else
      consumer_bf16<R, S>(a, sm, warp - NL - 2, lane);
  } else {
    consumer_f32<R, S>(a, sm, warp - NL - 2, lane);
  }
  // Launched behind the index kernel (programmatic dependent launch): finish
  // only after it, so that later work of the stream sees both complete.
  if (a.pdl) griddep_wait();
}

// ------------------------------------------------------------------ host

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

// K or V pool [num_pages, hkv, page_size, 128] as rows of one key.
//   f32:  3-D (32 floats, 4 quarters, rows), box (32, 4, kb);
//   bf16: 2-D (64 bf16 of one half, rows) with row stride 256 bytes, one map
//         per half (base + 128 bytes for the high half), box (64, kb).
bool encode_pool(const void* pool, int64_t rows, int kb, bool bf16, CUtensorMap* maps) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  if (bf16) {
    for (int half = 0; half < 2; ++half) {
      const cuuint64_t dims[2] = {64, static_cast<cuuint64_t>(rows)};
      const cuuint64_t strides[1] = {256};
      const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(kb)};
      const cuuint32_t estr[2] = {1, 1};
      void* addr = const_cast<unsigned char*>(static_cast<const unsigned char*>(pool) + 128 * half);
      if (enc(maps + half, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, addr, dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    }
    return true;
  }
  const cuuint64_t dims[3] = {32, 4, static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[2] = {128, 512};
  const cuuint32_t box[3] = {32, 4, static_cast<cuuint32_t>(kb)};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(maps, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(pool), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool kBf16, int R, int S>
cudaError_t launch_fused(const FusedDecArgs& a, cudaStream_t stream) {
  constexpr Layout L = fused_layout<kBf16, R, S>();
  constexpr int NC = Cfg<kBf16>::NC;
  constexpr int NL = Cfg<kBf16>::NL;
  const size_t smem = L.total + 1024;
  if (smem > 227 * 1024) return cudaErrorNotSupported;
  const int ck = a.block_size < kCK ? a.block_size : kCK;
  const int kb = a.page_size < ck ? a.page_size : ck;
  const int64_t rows = a.num_pages * a.hkv * a.page_size;
  TmaMaps maps;
  if (!encode_pool(a.k_pages, rows, kb, kBf16, maps.k) ||
      !encode_pool(a.v_pages, rows, kb, kBf16, maps.v))
    return cudaErrorNotSupported;
  if constexpr (!kBf16) {
    // q [tq, hq, 128] as rows of 32 floats; box = the qhead rows of one kv head.
    const int64_t qrows = a.tq * a.hq * 4;
    const cuuint64_t dims[2] = {32, static_cast<cuuint64_t>(qrows)};
    const cuuint64_t strides[1] = {128};
    const cuuint32_t box[2] = {32, static_cast<cuuint32_t>(a.qhead * 4)};
    const cuuint32_t estr[2] = {1, 1};
    EncodeTiledFn enc = encode_fn();
    if (enc == nullptr || qrows > kFusedMaxRows ||
        enc(&maps.q, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(a.q), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorNotSupported;
  } else {
    maps.q = maps.k[0];   // unused
  }
  const void* fn = reinterpret_cast<const void*>(fused_dec_kernel<kBf16, R, S>);
  cudaError_t err =
      cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  const int64_t n_pieces = a.whole_items + (a.tq * a.hkv - a.whole_items) * a.pieces;
  int64_t grid = device_sm_count();
  if (grid > n_pieces) grid = n_pieces;
  if (grid < 1) return cudaSuccess;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3((2 + NL + NC) * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = a.pdl ? 1 : 0;
  FusedDecArgs args = a;
  int site = kStallNone;
  debug_stall_setting(&site, &args.spin_limit);
  args.stall = site == kStallFusedCopies;
  return cudaLaunchKernelEx(&cfg, fused_dec_kernel<kBf16, R, S>, maps, args);
}

}  // namespace

bool fused_dec_supported(int head_dim, int block_size, int page_size, int qhead, int kv_bf16) {
  if (head_dim != kD) return false;
  // page boxes: a power of two of at least 8 rows (the swizzle period)
  if (page_size < 8 || (page_size & (page_size - 1)) != 0) return false;
  if (block_size <= 0 || block_size % page_size != 0) return false;
  if (block_size / page_size > kMaxPPB) return false;
  const int ck = block_size < kCK ? block_size : kCK;
  if (block_size % ck != 0) return false;
  if (kv_bf16) return qhead >= 1 && qhead <= 16;
  return qhead >= 1 && qhead <= 4;
}

cudaError_t launch_fused_dec(const FusedDecArgs& a, cudaStream_t stream) {
  if (!fused_dec_supported(kD, a.block_size, a.page_size, a.qhead, a.kv_bf16))
    return cudaErrorNotSupported;
  if (a.ranks_per_piece < 1 || a.ranks_per_piece > kMaxEP || a.pieces < 1 ||
      static_cast<int64_t>(a.pieces) * a.ranks_per_piece < a.topk || a.whole_items < 0 ||
      a.whole_items > a.tq * a.hkv || (a.whole_items > 0 && a.topk > kMaxEP))
    return cudaErrorInvalidValue;
  if (a.num_pages < 1 || a.num_pages * a.hkv * a.page_size > kFusedMaxRows)
    return cudaErrorNotSupported;
  if (!a.kv_bf16) return launch_fused<false, 4, 3>(a, stream);
  if (a.qhead <= 8) return launch_fused<true, 8, 5>(a, stream);
  return launch_fused<true, 16, 4>(a, stream);
}

}  // namespace sa
