// Step 2 of KV-outer sparse attention on the 5th-generation tensor cores
// (tcgen05 + TMEM): per-edge partials as in process_work_unit (forward.rs of
// alice-llm's sparse_attention) for work units with many gathered rows
// (chunked prefill, skewed selections).
//
// A persistent CTA per SM claims (kv head, block) units in index order from a
// per-launch counter (whichever CTA is free takes the next unit, so the heavy
// units of a skewed selection spread out), so the SMs working at the same
// time cover neighbouring blocks of one (kv head, sequence) and share its Q
// rows in L2.  A unit's rows (edge x GQA lane) go through 128-row tiles.
// Warp roles, coupled by mbarriers:
//   warp 23    scheduler: claims units up to four ahead of the loaders and
//              resolves each unit's index entries (slot, edge range,
//              sequence, KV length), its keys' positions and page offsets
//              through the block table, and the Q row sources of its first
//              tile into a ring of unit slots, so that the loaders start
//              every unit with its global addresses at hand; an end-of-work
//              unit stops the other roles;
//   warps 1-14 loaders: per unit, the block's K and V rows (through the
//              block table, f32 or bf16) converted to bf16 once, both as
//              [keys x 128] rows with the 128-byte swizzle: K-major for S,
//              MN-major for O (two unit buffers, so the next unit loads
//              while this one computes); per tile, the rows' Q in the same
//              layout, from a bf16 copy of Q when the caller gives scratch
//              for one, else f32 rows converted (two or three tile buffers,
//              so the gathers' latency stays off the path);
//   warp 0     one thread issues S = Q K^T (M=128, N=block, K=128) into TMEM
//              and, once the softmax has turned S into P, O = P V (M=128,
//              N=128, K=block; P from TMEM); tcgen05.commit signals the
//              mbarriers;
//   warps 15-22 softmax and epilogue, two warpgroups taking alternate tiles
//              (and the matching S / O buffer), thread t <-> row t of the
//              tile (TMEM lane t): S back with tcgen05.ld, masks (block
//              length, absent pages, causal limit), m, p = 2^(s q - m), l,
//              and P as bf16 pairs back into S's TMEM columns (tcgen05.st),
//              where the second MMA takes it as its A operand; the tile
//              buffer thus holds Q only and frees as soon as S is done; then
//              the previous tile's O back from TMEM and its unnormalised
//              partial row through a swizzled staging tile, as TMA box
//              stores for full 32-row warps, and m and l to memory.
// S and O are double-buffered in TMEM (512 columns), so S of tile t + 1 and
// the epilogue of tile t - 1 overlap the softmax of tile t.  Operands are
// rounded to bf16 (tolerance class of the tensor-core path); S, O and the
// softmax statistics stay in f32.
#include <cstdint>

#include "internal.h"
#include "sa_common.cuh"

namespace sa {

namespace {

constexpr int kD = 128;
constexpr int kM = 128;            // rows per MMA tile
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr uint32_t kTmemCols = 512;  // S[2] at columns 0 / 128, O[2] at 256 / 384

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

// D (TMEM) (+)= A (TMEM, row i in lane i, two bf16 per column) x B (smem)^T.
__device__ __forceinline__ void mma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D (TMEM) (+)= A (smem) x B (smem)^T, tf32 inputs (f32 in shared memory),
// f32 accumulation.
__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 64 consecutive f32 columns of this thread's TMEM lane (one round trip).
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&v)[64]) {
  uint32_t r[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, "
      "%45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, "
      "%62, %63}, [%64];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]),
        "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]),
        "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]),
        "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]),
        "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]),
        "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}

// 32 consecutive 32-bit columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// 16 consecutive 32-bit columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
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

// Shared-memory descriptor of an MN-major operand stored as rows of one K
// index (128 bytes = 64 MN elements per row, 128-byte swizzle): 8 K rows per
// swizzle atom (stride 1024 bytes), the next 64 MN elements `lbo` bytes on.
__device__ __forceinline__ uint64_t sw128_desc_mn(uint32_t saddr, uint32_t lbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);          // start address
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;       // leading byte offset (MN)
  d |= static_cast<uint64_t>((1024u >> 4) & 0x3FFFu) << 32;     // stride byte offset (K)
  d |= static_cast<uint64_t>(1u) << 46;                         // descriptor version
  d |= static_cast<uint64_t>(2u) << 61;                         // 128-byte swizzle
  return d;
}

// Instruction descriptor: bf16 x bf16 -> f32, A K-major, B K-major or (b_mn)
// MN-major.
__host__ __device__ constexpr uint32_t idesc_bf16(int m, int n, bool b_mn = false) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (b_mn ? (1u << 16) : 0u) |
         (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(m >> 4) << 24);
}

// Instruction descriptor: tf32 x tf32 -> f32 (operand format 2), A K-major,
// B K-major or (b_mn) MN-major.
__host__ __device__ constexpr uint32_t idesc_tf32(int m, int n, bool b_mn = false) {
  return (1u << 4) | (2u << 7) | (2u << 10) | (b_mn ? (1u << 16) : 0u) |
         (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(m >> 4) << 24);
}

// Byte offset of a 16-byte chunk of f32 elements inside a K-major,
// 128B-swizzled tile of `rows` rows: element k (a multiple of 4) of row r,
// 32 f32 per panel row.
__device__ __forceinline__ uint32_t sw128_offset_f32(int rows, int r, int k) {
  const int panel = k >> 5;
  const int chunk = (k & 31) >> 2;
  return static_cast<uint32_t>(panel * rows * 128 + r * 128 + ((chunk ^ (r & 7)) << 4));
}

// Byte offset of element pair/quad position inside a K-major, 128B-swizzled
// tile of `rows` rows: element k of row r (bf16 elements, 64 per panel row).
__device__ __forceinline__ uint32_t sw128_offset(int rows, int r, int k) {
  const int panel = k >> 6;
  const int chunk = (k & 63) >> 3;
  const int within = (k & 7) * 2;
  return static_cast<uint32_t>(panel * rows * 128 + r * 128 + ((chunk ^ (r & 7)) << 4) + within);
}

// Four K/V elements (f32 or bf16) as packed bf16 (round to nearest even).
template <bool kBf16>
__device__ __forceinline__ uint2 ld_kv4_bf16(const void* pages, int64_t elem_off) {
  if constexpr (kBf16) {
    return __ldg(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(pages) + elem_off));
  } else {
    const float4 v = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(pages) + elem_off));
    return make_uint2(pack_bf16x2_rn(v.x, v.y), pack_bf16x2_rn(v.z, v.w));
  }
}

// Warp roles: 0 MMA issue, 1 scheduler, then the loaders, then two softmax /
// epilogue warpgroups (warp w reads TMEM lanes 32 (w % 4) ..).  Units of
// 64-key blocks (skewed selections: about one tile each) lean on the
// loaders' per-unit K/V pass: 14 loaders, 768 threads at 80 registers, S read
// 32 columns per TMEM load.  Units of 128-key blocks (prefill: many tiles
// each) lean on the softmax: 10 loaders, 640 threads at 96 registers, S read
// 64 columns per TMEM load.
template <int BS> struct TcWarps {
  static constexpr int kLoaders = BS == 64 ? 14 : 10;
  static constexpr int kThreads = 32 * (2 + kLoaders + 8);
  static constexpr int kLoadThreads = 32 * kLoaders;
  static constexpr int kRowsPerLoader = (kM + kLoaders - 1) / kLoaders;  // Q rows per loader lane
  static constexpr int kQBatch = kRowsPerLoader;                        // f32 Q rows in flight
  static constexpr int kKvBatch = (2 * BS + kLoaders - 1) / kLoaders < 13
                                      ? (2 * BS + kLoaders - 1) / kLoaders : 13;
  static constexpr int kSoftmaxWarp0 = 2 + kLoaders;
  static constexpr bool kWideS = BS == 128;
  static_assert(kSoftmaxWarp0 % 4 == 0, "softmax warpgroups aligned to TMEM lane quarters");
};

// kTf32: the scores S = Q K^T from Q and K kept in f32 (tcgen05 kind::tf32)
// instead of rounded to bf16, so their Q and K tiles are twice as large; P
// and V stay bf16 operands of O = P V either way.
template <int BS, bool kTf32 = false> struct TcCfg {
  static constexpr int E = kTf32 ? 4 : 2;         // bytes per Q / K element
  static constexpr int KVB = kTf32 && BS == 128 ? 1 : 2;     // unit buffers (K, V)
  static constexpr int NX = kTf32 ? 1 : (BS == 128 ? 2 : 3); // tile buffers (Q)
  // epilogue staging tiles per warp: two where shared memory allows (the
  // box store of one drains while the other fills)
  static constexpr int SB = BS == 64 ? 2 : 1;
};
constexpr int kMaxNX = 3;
constexpr int kRing = 4;                          // unit slots of the scheduler
constexpr int kSchedWarp = 1;
constexpr int kLoaderWarp0 = 2;

struct UnitInfo {
  int32_t rows;         // edges x qhead of the unit (0: skip)
  int32_t h;
  int64_t prow0;        // first partial row of the unit
  int64_t e0;           // first edge of the unit (absolute)
  int64_t q0, qo, lk;   // the sequence's first query, query count, KV length
  int64_t bstart;       // position of the block's first key
};

// Shared memory: KVB unit buffers (K, V), NX tile buffers (Q), key
// positions and unit info per unit buffer, the scheduler's ring of unit
// slots, the epilogue's staging tiles, barriers, the TMEM address and
// per-head unit bases.
struct TcPlan {
  size_t kv_bytes;      // one unit buffer: K [BS][128] + V [BS][128] bf16
  size_t slot_bytes;    // one unit slot (UnitSlot layout below)
  size_t kv, x, kpos, info, ring, stage, bars, misc, total;
};

// A unit slot of the scheduler ring: the unit's info, then per key its
// source offset in the pool (elements, -1 = no key) and position (-1 = no
// key), then the Q source offsets (elements, -1 = no row) of the unit's
// first tile.
template <int BS> struct SlotLayout {
  static constexpr size_t koff = 64;                       // int64 [BS]
  static constexpr size_t kpos = koff + 8 * BS;            // int32 [BS]
  static constexpr size_t qsrc = kpos + 4 * BS;            // int64 [kM]
  static constexpr size_t bytes = (qsrc + 8 * 128 + 127) / 128 * 128;
};

__host__ __device__ constexpr size_t tc_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Every region starts on a 128-byte boundary (the swizzled tiles on 1024):
// float4 staging, int64 offsets and mbarriers all need their alignment
// whatever the sizes of the regions before them.
template <int BS, bool kTf32>
__host__ __device__ inline TcPlan tc_plan() {
  using C = TcCfg<BS, kTf32>;
  const int bs = BS, kvb = C::KVB, nx = C::NX, sb = C::SB;
  TcPlan p{};
  p.kv_bytes = static_cast<size_t>(bs) * kD * (C::E + 2);               // K, then V (bf16)
  p.kv = 0;                                                             // 1024-aligned
  p.x = p.kv + kvb * p.kv_bytes;                                        // [nx] Q tiles
  p.kpos = tc_up(p.x + nx * static_cast<size_t>(kM) * kD * C::E, 128);  // int32 [kvb][BS]
  p.info = tc_up(p.kpos + kvb * static_cast<size_t>(bs) * 4, 128);      // UnitInfo [kvb]
  p.slot_bytes = bs == 128 ? SlotLayout<128>::bytes : SlotLayout<64>::bytes;
  p.ring = tc_up(p.info + kvb * sizeof(UnitInfo), 128);                 // slots [kRing]
  p.stage = tc_up(p.ring + kRing * p.slot_bytes, 1024);                 // f32 [8][sb][32][16]
  p.bars = tc_up(p.stage + 8 * sb * 32 * 16 * 4, 128);                  // uint64 [32]
  p.misc = tc_up(p.bars + 32 * 8, 128);                                 // TMEM slot, unit bases
  p.total = p.misc + 16 + 201 * 4 + 1024;                               // + alignment slack
  return p;
}
static_assert(sizeof(UnitInfo) % 8 == 0 && sizeof(UnitInfo) <= 64, "UnitInfo in a slot header");
static_assert(4 + 2 * kMaxNX + 10 + 1 + 2 * kRing <= 32, "mbarriers fit their 32 slots");

struct TcBars {
  uint64_t *kv_full, *kv_empty;        // [KVB]
  uint64_t *x_full, *x_empty;          // [NX]
  uint64_t *s_full, *s_free;           // [2] TMEM S buffers
  uint64_t *p_full, *o_full, *o_free;  // [2]
  uint64_t* done;
  uint64_t *slot_full, *slot_empty;    // [kRing]
};

// OR of `pred` over the loader warps (named barrier 1); also a barrier.
template <int kLoadThreads>
__device__ __forceinline__ bool loaders_or(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "barrier.red.or.pred q, 1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(pred ? 1u : 0u), "n"(kLoadThreads)
      : "memory");
  return r != 0;
}

// Unit u's head h and compact slot j from the per-head unit bases.
__device__ __forceinline__ void unit_head(const int32_t* unit_base, int hkv, int64_t u, int& h,
                                          int& j) {
  h = 0;
  while (h + 1 < hkv && unit_base[h + 1] <= u) ++h;
  j = static_cast<int>(u - unit_base[h]);
}

// ------------------------------------------------------------------ scheduler

// Fills slot U % kRing with unit U of this CTA once the loaders have freed
// it: the index lookups are spread over lanes so that each level of the
// chain (slot and edge range, then the sequence's lengths, then the block
// table and the edges) costs one memory round trip.
template <int BS>
__device__ void tc_scheduler(const ForwardArgs& a, unsigned char* smem, const TcPlan& P,
                             const TcBars& B, const int32_t* unit_base, int64_t n_units,
                             int lane) {
  using L = SlotLayout<BS>;
  constexpr unsigned kAll = 0xffffffffu;
  const int qhead = a.qhead;
  const int ps = a.page_size;
  int64_t* status = a.totals + 3;
  for (uint32_t U = 0;; ++U) {
    const int sl = static_cast<int>(U % kRing);
    unsigned char* slot = smem + P.ring + sl * P.slot_bytes;
    const bool got = U < static_cast<uint32_t>(kRing) ||
                     mbar_wait_bounded(B.slot_empty + sl, ((U / kRing) - 1) & 1u);
    if (!__all_sync(kAll, got)) {
      if (lane == 0) report(status, SA_ERR_DEVICE_TIMEOUT);
      return;
    }
    // The next unit: claimed from the forward's counter (whichever CTA is
    // free takes the next unit, so heavy units of a skewed selection do not
    // pile up on a few CTAs), in the order of the longest-first list when
    // there is one, else in index order; round-robin without a counter.
    int64_t u = 0;
    if (lane == 0) {
      if (a.unit_counter != nullptr) {
        const uint32_t k = atomicAdd(a.unit_counter, 1u);
        u = (a.unit_order != nullptr && k < n_units) ? static_cast<int64_t>(a.unit_order[k])
                                                     : static_cast<int64_t>(k);
      } else {
        u = blockIdx.x + static_cast<int64_t>(U) * gridDim.x;
      }
    }
    u = __shfl_sync(kAll, u, 0);
    if (u >= n_units) {
      // end of work: a unit with rows < 0 tells the other roles to stop
      if (lane == 0) reinterpret_cast<UnitInfo*>(slot)->rows = -1;
      mbar_arrive(B.slot_full + sl);
      return;
    }
    int h, j;
    unit_head(unit_base, a.hkv, u, h, j);
    int64_t x = 0;
    if (lane == 0) x = a.sel_slots[static_cast<int64_t>(h) * a.nbs + j];
    else if (lane == 1) x = a.sel_offsets[static_cast<int64_t>(h) * (a.nbs + 1) + j];
    else if (lane == 2) x = a.sel_offsets[static_cast<int64_t>(h) * (a.nbs + 1) + j + 1];
    else if (lane == 3) x = a.edge_head_base[h];
    const int raw = static_cast<int>(__shfl_sync(kAll, x, 0));
    const int64_t ebase = __shfl_sync(kAll, x, 3);
    const int64_t e0 = ebase + __shfl_sync(kAll, x, 1);
    const int64_t e1 = ebase + __shfl_sync(kAll, x, 2);
    const bool bad = raw < 0 || raw >= a.nbs || e1 < e0;
    if (bad && lane == 0) report(status, SA_ERR_SHAPE);
    const int b = bad ? 0 : raw / a.msb;
    const int blk = bad ? 0 : raw - b * a.msb;
    int64_t y = 0;
    if (lane == 0) y = a.used ? max(a.used[b], 0) : static_cast<int64_t>(a.msb) * BS;
    else if (lane == 1) y = a.cu[b];
    else if (lane == 2) y = a.cu[b + 1];
    const int64_t lk = __shfl_sync(kAll, y, 0);
    const int64_t q0 = __shfl_sync(kAll, y, 1);
    const int64_t qo = __shfl_sync(kAll, y, 2) - q0;
    const int rows = bad ? 0 : static_cast<int>((e1 - e0) * qhead);
    const int64_t bstart = static_cast<int64_t>(blk) * BS;
    const int64_t bend = min(bstart + BS, lk);
    // the keys: position (or -1) and source offset through the block table
    const int32_t* bt = a.block_tables + static_cast<int64_t>(b) * a.max_pages +
                        static_cast<int64_t>(blk) * a.pages_per_block;
    int64_t* koff = reinterpret_cast<int64_t*>(slot + L::koff);
    int32_t* kpos = reinterpret_cast<int32_t*>(slot + L::kpos);
    for (int jj = lane; jj < BS; jj += 32) {
      const int64_t pos = bstart + jj;
      int32_t live = -1;
      int64_t off = -1;
      if (!bad && pos < bend) {
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
    // the first tile's Q sources
    int64_t* qsrc = reinterpret_cast<int64_t*>(slot + L::qsrc);
    for (int r = lane; r < kM; r += 32) {
      int64_t src = -1;
      if (r < rows) {
        const int64_t qi = a.edges[2 * (e0 + r / qhead)];
        src = (qi * a.hq + static_cast<int64_t>(h) * qhead + r % qhead) * kD;
      }
      qsrc[r] = src;
    }
    if (lane == 0 && a.cta_stats != nullptr && static_cast<int>(blockIdx.x) < a.cta_stats_len) {
      unsigned long long* st = reinterpret_cast<unsigned long long*>(a.cta_stats) + 3 * blockIdx.x;
      atomicAdd(st, static_cast<unsigned long long>(rows));
      atomicAdd(st + 1, 1ull);
    }
    if (lane == 0) {
      UnitInfo* info = reinterpret_cast<UnitInfo*>(slot);
      info->rows = rows;
      info->h = h;
      info->prow0 = e0 * qhead;
      info->e0 = e0;
      info->q0 = q0;
      info->qo = qo;
      info->lk = lk;
      info->bstart = bstart;
    }
    mbar_arrive(B.slot_full + sl);
  }
}

// ------------------------------------------------------------------ loaders

template <int BS, bool kBf16, bool kTf32>
__device__ void tc_loader(const ForwardArgs& a, unsigned char* smem, const TcPlan& P,
                          const TcBars& B, int lw, int lane) {
  constexpr int KVB = TcCfg<BS, kTf32>::KVB;
  constexpr int kNX = TcCfg<BS, kTf32>::NX;
  constexpr int E = TcCfg<BS, kTf32>::E;
  using W = TcWarps<BS>;
  constexpr int kLoaders = W::kLoaders, kLoadThreads = W::kLoadThreads;
  constexpr int kRowsPerLoader = W::kRowsPerLoader, kQBatch = W::kQBatch, kKvBatch = W::kKvBatch;
  using L = SlotLayout<BS>;
  const int lt = lw * 32 + lane;
  const int qhead = a.qhead;
  int64_t* status = a.totals + 3;
  uint32_t T = 0;
  for (uint32_t U = 0;; ++U) {
    const int kvb = static_cast<int>(U % KVB);
    unsigned char* ks = smem + P.kv + kvb * P.kv_bytes;
    unsigned char* vs = ks + static_cast<size_t>(BS) * kD * E;
    int32_t* kpos = reinterpret_cast<int32_t*>(smem + P.kpos) + kvb * BS;
    UnitInfo* info = reinterpret_cast<UnitInfo*>(smem + P.info) + kvb;
    const int sl = static_cast<int>(U % kRing);
    const unsigned char* slot = smem + P.ring + sl * P.slot_bytes;

    bool got = mbar_wait_bounded(B.slot_full + sl, (U / kRing) & 1u);
    got = got && (U < static_cast<uint32_t>(KVB) ||
                  mbar_wait_bounded(B.kv_empty + kvb, ((U / KVB) - 1) & 1u));
    if (loaders_or<W::kLoadThreads>(!got)) {
      if (lt == 0) report(status, SA_ERR_DEVICE_TIMEOUT);
      return;
    }
    // ---- the unit, as the scheduler resolved it ------------------------------
    const UnitInfo si = *reinterpret_cast<const UnitInfo*>(slot);
    if (si.rows < 0) {
      // end of work: passed on to the MMA and softmax roles through the unit
      // buffer (freed above)
      if (lt == 0) info->rows = -1;
      mbar_arrive(B.kv_full + kvb);
      return;
    }
    const int rows = si.rows;
    const int h = si.h;
    const int64_t e0 = si.e0;
    const int64_t* koff = reinterpret_cast<const int64_t*>(slot + L::koff);
    const int32_t* skpos = reinterpret_cast<const int32_t*>(slot + L::kpos);
    for (int jj = lt; jj < BS; jj += kLoadThreads) kpos[jj] = skpos[jj];
    // K and V rows alike (lane = 4 dims, converted to bf16, except K rows
    // kept f32 for tf32 scores), 13 of a warp's rows in flight at a time:
    // rows [0, BS) are K, [BS, 2 BS) V, both stored [key][128] with the
    // 128-byte swizzle (V is the MMA's MN-major B operand).
    if constexpr (kTf32) {
      constexpr int kRows = (2 * BS + kLoaders - 1) / kLoaders;
#pragma unroll
      for (int q0 = 0; q0 < kRows; q0 += kKvBatch) {
        float4 kr[kKvBatch];
#pragma unroll
        for (int q = 0; q < kKvBatch; ++q) {
          const int r = lw + (q0 + q) * kLoaders;
          const int key = r < BS ? r : r - BS;
          const int64_t off = q0 + q < kRows && r < 2 * BS ? koff[key] : -1;
          kr[q] = off >= 0 ? __ldg(reinterpret_cast<const float4*>(
                                 static_cast<const float*>(r < BS ? a.k_pages : a.v_pages) + off) +
                             lane)
                           : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int q = 0; q < kKvBatch; ++q) {
          const int r = lw + (q0 + q) * kLoaders;
          if (q0 + q < kRows && r < 2 * BS) {
            if (r < BS)       // K: f32 rows (tf32 operand)
              *reinterpret_cast<float4*>(ks + sw128_offset_f32(BS, r, 4 * lane)) = kr[q];
            else              // V: bf16 rows (bf16 operand of O = P V)
              *reinterpret_cast<uint2*>(vs + sw128_offset(BS, r - BS, 4 * lane)) =
                  make_uint2(pack_bf16x2_rn(kr[q].x, kr[q].y), pack_bf16x2_rn(kr[q].z, kr[q].w));
          }
        }
      }
    } else {
      constexpr int kRows = (2 * BS + kLoaders - 1) / kLoaders;
#pragma unroll
      for (int q0 = 0; q0 < kRows; q0 += kKvBatch) {
        uint2 kr[kKvBatch];
#pragma unroll
        for (int q = 0; q < kKvBatch; ++q) {
          const int r = lw + (q0 + q) * kLoaders;
          const int key = r < BS ? r : r - BS;
          const int64_t off = q0 + q < kRows && r < 2 * BS ? koff[key] : -1;
          kr[q] = off >= 0 ? ld_kv4_bf16<kBf16>(r < BS ? a.k_pages : a.v_pages, off + 4 * lane)
                           : make_uint2(0u, 0u);
        }
#pragma unroll
        for (int q = 0; q < kKvBatch; ++q) {
          const int r = lw + (q0 + q) * kLoaders;
          if (q0 + q < kRows && r < 2 * BS) {
            const int key = r < BS ? r : r - BS;
            *reinterpret_cast<uint2*>((r < BS ? ks : vs) + sw128_offset(BS, key, 4 * lane)) =
                kr[q];
          }
        }
      }
    }
    if (lt == 0) *info = si;
    fence_proxy_async_smem();
    mbar_arrive(B.kv_full + kvb);

    // ---- tiles: Q rows and causal limits ------------------------------------
    // Warp lw gathers rows lw + kLoaders q of a tile: lane q holds row q's Q
    // source (found, and prefetched into L2, for the next tile while this
    // tile's rows are in flight), then the rows are loaded (lane = 4 dims of
    // a row).
    auto row_source = [&](int rt) -> int64_t {
      const int r = lw + lane * kLoaders;
      if (lane < kRowsPerLoader && r < kM && rt + r < rows) {
        const int row = rt + r;
        const int64_t qi = a.edges[2 * (e0 + row / qhead)];
        return (qi * a.hq + static_cast<int64_t>(h) * qhead + row % qhead) * kD;
      }
      return -1;
    };
    // the first tile's sources from the slot, which then goes back to the
    // scheduler
    int64_t my_src = -1;
    {
      const int r = lw + lane * kLoaders;
      if (lane < kRowsPerLoader && r < kM)
        my_src = reinterpret_cast<const int64_t*>(slot + L::qsrc)[r];
    }
    mbar_arrive(B.slot_empty + sl);
    for (int rt = 0; rt < rows; rt += kM, ++T) {
      const int xb = static_cast<int>(T % kNX);
      got = T < static_cast<uint32_t>(kNX) ||
            mbar_wait_bounded(B.x_empty + xb, ((T / kNX) - 1) & 1u);
      if (loaders_or<W::kLoadThreads>(!got)) {
        if (lt == 0) report(status, SA_ERR_DEVICE_TIMEOUT);
        return;
      }
      unsigned char* xq = smem + P.x + static_cast<size_t>(xb) * kM * kD * E;
      int64_t nxt_src = -1;
      if (!kTf32 && a.q16 != nullptr) {
        // bf16 rows (256 bytes): a half-warp per row, 8 dims per lane, two
        // of the warp's rows per load instruction
        constexpr int kPairs = (kRowsPerLoader + 1) / 2;
        const int hl = lane & 15;
        const int half = lane >> 4;
        uint4 w[kPairs];
#pragma unroll
        for (int i = 0; i < kPairs; ++i) {
          const int q = 2 * i + half;
          const int64_t src = __shfl_sync(0xffffffffu, my_src, q & 31);
          w[i] = make_uint4(0u, 0u, 0u, 0u);
          if (q < kRowsPerLoader && src >= 0)
            w[i] = __ldg(reinterpret_cast<const uint4*>(a.q16 + src) + hl);
        }
        if (rt + kM < rows) {
          nxt_src = row_source(rt + kM);
          if (nxt_src >= 0)
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(a.q16 + nxt_src),
                         "r"(static_cast<uint32_t>(kD * 2))
                         : "memory");
        }
#pragma unroll
        for (int i = 0; i < kPairs; ++i) {
          const int q = 2 * i + half;
          const int r = lw + q * kLoaders;
          if (q < kRowsPerLoader && r < kM)
            *reinterpret_cast<uint4*>(xq + sw128_offset(kM, r, 8 * hl)) = w[i];
        }
      } else {
        // f32 rows (512 bytes): lane = 4 dims, converted to bf16 (kept f32
        // for tf32 operands)
#pragma unroll
        for (int q0 = 0; q0 < kRowsPerLoader; q0 += kQBatch) {
          float4 v[kQBatch];
#pragma unroll
          for (int q = 0; q < kQBatch; ++q) {
            const int64_t src = __shfl_sync(0xffffffffu, my_src, (q0 + q) & 31);
            v[q] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (q0 + q < kRowsPerLoader && src >= 0)
              v[q] = __ldg(reinterpret_cast<const float4*>(a.q + src) + lane);
          }
          if (q0 == 0 && rt + kM < rows) {
            nxt_src = row_source(rt + kM);
            // the next tile's rows start for L2 now; their loads come a tile later
            if (nxt_src >= 0)
              asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(a.q + nxt_src),
                           "r"(static_cast<uint32_t>(kD * 4))
                           : "memory");
          }
#pragma unroll
          for (int q = 0; q < kQBatch; ++q) {
            const int r = lw + (q0 + q) * kLoaders;
            if (q0 + q < kRowsPerLoader && r < kM) {
              if constexpr (kTf32)
                *reinterpret_cast<float4*>(xq + sw128_offset_f32(kM, r, 4 * lane)) = v[q];
              else
                *reinterpret_cast<uint2*>(xq + sw128_offset(kM, r, 4 * lane)) =
                    make_uint2(pack_bf16x2_rn(v[q].x, v[q].y), pack_bf16x2_rn(v[q].z, v[q].w));
            }
          }
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(B.x_full + xb);
      my_src = nxt_src;
    }
  }
}

// ------------------------------------------------------------------ MMA issue

template <int BS, bool kTf32>
__device__ bool tc_issue_o(unsigned char* smem, const TcPlan& P, const TcBars& B, uint32_t tmem,
                           int kvb, uint32_t T) {
  const int sb = static_cast<int>(T & 1u);
  if (!mbar_wait_bounded(B.p_full + sb, (T >> 1) & 1u)) return false;
  if (T >= 2 && !mbar_wait_bounded(B.o_free + sb, ((T >> 1) - 1) & 1u)) return false;
  tc_fence_after();
  constexpr int E = TcCfg<BS, kTf32>::E;
  const uint32_t v_addr = smem_u32(smem + P.kv + kvb * P.kv_bytes + static_cast<size_t>(BS) * kD * E);
  const uint32_t t_p = tmem + 128 * sb;          // P (bf16 pairs) over S's columns
  const uint32_t t_o = tmem + 256 + 128 * sb;
  // P of keys 0..63 in columns 0..31, of keys 64..127 in columns 64..95
#pragma unroll
  for (int st = 0; st < BS / 16; ++st)   // 16 keys = 2048 bytes of V rows per step
    mma_bf16_ta(t_o, t_p + 8 * st + (st >= 4 ? 32 : 0),
                sw128_desc_mn(v_addr + st * 2048, BS * 128), idesc_bf16(kM, kD, true), st > 0);
  mma_commit(B.o_full + sb);
  mma_commit(B.s_free + sb);                     // P read: the S / P columns are free
  return true;
}

template <int BS, bool kTf32>
__device__ void tc_mma(const ForwardArgs& a, unsigned char* smem, const TcPlan& P,
                       const TcBars& B, uint32_t tmem) {
  constexpr int KVB = TcCfg<BS, kTf32>::KVB;
  constexpr int kNX = TcCfg<BS, kTf32>::NX;
  constexpr int E = TcCfg<BS, kTf32>::E;
  int64_t* status = a.totals + 3;
  uint32_t T = 0;
  for (uint32_t U = 0;; ++U) {
    const int kvb = static_cast<int>(U % KVB);
    if (!mbar_wait_bounded(B.kv_full + kvb, (U / KVB) & 1u)) {
      report(status, SA_ERR_DEVICE_TIMEOUT);
      return;
    }
    const UnitInfo* info = reinterpret_cast<const UnitInfo*>(smem + P.info) + kvb;
    const int rows = info->rows;
    if (rows < 0) return;                        // end of work
    const uint32_t k_addr = smem_u32(smem + P.kv + kvb * P.kv_bytes);
    tc_fence_after();
    const int tiles = (rows + kM - 1) / kM;
    for (int tt = 0; tt < tiles; ++tt, ++T) {
      const int sb = static_cast<int>(T & 1u);
      const int xb = static_cast<int>(T % kNX);
      if (!mbar_wait_bounded(B.x_full + xb, (T / kNX) & 1u) ||
          (T >= 2 && !mbar_wait_bounded(B.s_free + sb, ((T >> 1) - 1) & 1u))) {
        report(status, SA_ERR_DEVICE_TIMEOUT);
        return;
      }
      tc_fence_after();
      const uint32_t q_addr = smem_u32(smem + P.x + static_cast<size_t>(xb) * kM * kD * E);
      const uint32_t t_s = tmem + 128 * sb;
      // K steps of 32 bytes (16 bf16 or 8 tf32), four per 128-byte panel
#pragma unroll
      for (int st = 0; st < kD * E / 32; ++st) {
        const uint32_t panel = st >> 2;
        const uint32_t kb = (st & 3) * 32;
        if constexpr (kTf32)
          mma_tf32(t_s, sw128_desc(q_addr + panel * kM * 128 + kb),
                   sw128_desc(k_addr + panel * BS * 128 + kb), idesc_tf32(kM, BS), st > 0);
        else
          mma_bf16(t_s, sw128_desc(q_addr + panel * kM * 128 + kb),
                   sw128_desc(k_addr + panel * BS * 128 + kb), idesc_bf16(kM, BS), st > 0);
      }
      mma_commit(B.s_full + sb);
      mma_commit(B.x_empty + xb);                // Q read: the tile buffer is free
      if (tt > 0 && !tc_issue_o<BS, kTf32>(smem, P, B, tmem, kvb, T - 1)) {
        report(status, SA_ERR_DEVICE_TIMEOUT);
        return;
      }
    }
    if (tiles > 0 && !tc_issue_o<BS, kTf32>(smem, P, B, tmem, kvb, T - 1)) {
      report(status, SA_ERR_DEVICE_TIMEOUT);
      return;
    }
    mma_commit(B.kv_empty + kvb);
  }
}

// ------------------------------------------------------------------ softmax + epilogue

// 2^x by the special-function unit (ex2.approx: relative error about 2^-22;
// subnormal results flush to zero, below what bf16 P and f32 l resolve).
__device__ __forceinline__ float ex2_fast(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ float min3(float a, float b, float c) {
  float d;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Packed pairs of f32 (lo in the low half) and their elementwise a * b + c
// and a + b, one instruction per pair.
__device__ __forceinline__ uint64_t f32x2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}

__device__ __forceinline__ void f32x2_split(uint64_t r, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
}

__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// Softmax warpgroup g (0 or 1) takes the tiles whose running index has
// parity g, and with them TMEM buffers S[g], O[g].
template <int BS, bool kTf32>
__device__ void tc_softmax(const ForwardArgs& a, const CUtensorMap* omap, unsigned char* smem,
                           const TcPlan& P, const TcBars& B, uint32_t tmem, int warp,
                           int lane) {
  const uint32_t g = static_cast<uint32_t>((warp - TcWarps<BS>::kSoftmaxWarp0) >> 2);
  constexpr int KVB = TcCfg<BS, kTf32>::KVB;
  int64_t* status = a.totals + 3;
  const int row = (warp & 3) * 32 + lane;               // TMEM lane = tile row
  const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
  const float qscale = a.scale * kLog2e;
  // the warp's staging tiles (32 rows x 64 bytes each), used in turn
  constexpr int SB = TcCfg<BS, kTf32>::SB;
  float* const wst0 =
      reinterpret_cast<float*>(smem + P.stage) + (g * 4 + (warp & 3)) * SB * 32 * 16;
  uint32_t rnd = 0;
  // The previous tile's row, stored after this tile's softmax.
  bool prev = false;
  uint32_t prevT = 0;
  int64_t prev_prow = -1;
  float prev_m = -INFINITY, prev_l = 0.f;

  auto epilogue = [&](uint32_t Tp, int64_t prow, float m2, float l) -> bool {
    const int sb = static_cast<int>(Tp & 1u);
    const bool got = mbar_wait_bounded(B.o_full + sb, (Tp >> 1) & 1u);
    if (!__all_sync(0xffffffffu, got)) return false;
    tc_fence_after();
    const uint32_t t_o = tmem + 256 + 128 * sb + lane_base;
    // 64 bytes of a row at a time (16 f32 or 32 bf16 columns): each thread
    // puts them into the warp's staging tile (16-byte chunk i of row r at
    // i ^ ((r >> 1) & 3): the 64-byte swizzle of the tensor maps, and 8
    // consecutive rows hit 8 different bank groups).  A warp whose 32 rows
    // are all live hands the tile to the TMA engine (one 32 x 64-byte box
    // store, asynchronous: the warp goes on while the rows drain to L2);
    // otherwise it writes its live rows, 8 rows x 64 bytes per store
    // instruction.  Valid rows are a prefix of the tile, so a warp with a
    // valid row has lane 0 valid.
    const int64_t prow0 = __shfl_sync(0xffffffffu, prow, 0);
    const unsigned live = __ballot_sync(0xffffffffu, prow >= 0);
    const bool by_tma = a.o_tma && live == 0xffffffffu;
    // A round's staging tile is free once the box store last issued from
    // it has read it: with two tiles, the store of two rounds ago (one box
    // store per round, issued by lane 0; a round of plain stores waits for
    // every earlier box store instead); with one, the previous round's.
    float* wst = wst0;
    auto stage_free = [&]() {
      wst = wst0 + (rnd % SB) * 32 * 16;
      ++rnd;
      if (lane == 0) {
        if (SB == 2 && by_tma)
          bulk_wait_read_1();
        else
          bulk_wait_read_all();
      }
      __syncwarp();
    };
    auto stage_store = [&](int x) {
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_2d(omap, x, static_cast<int>(prow0), wst);
        bulk_commit();
      }
    };
    // O 32 columns at a time (the epilogue keeps the softmax loop's state
    // live, so a 64-column load would spill)
#pragma unroll 1
    for (int c = 0; c < kD / 32; ++c) {
      float v[32];
      tmem_ld32(t_o + c * 32, v);
      tmem_ld_wait();
      if (a.o_bf16) {
        stage_free();
#pragma unroll
        for (int i = 0; i < 4; ++i)
          reinterpret_cast<uint4*>(wst + lane * 16)[i ^ ((lane >> 1) & 3)] =
              make_uint4(pack_bf16x2_rn(v[8 * i], v[8 * i + 1]),
                         pack_bf16x2_rn(v[8 * i + 2], v[8 * i + 3]),
                         pack_bf16x2_rn(v[8 * i + 4], v[8 * i + 5]),
                         pack_bf16x2_rn(v[8 * i + 6], v[8 * i + 7]));
        if (by_tma) {
          stage_store(c * 32);
          continue;
        }
        __syncwarp();
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int r = 8 * k + (lane >> 2);
          const int ch = lane & 3;
          if ((live >> r) & 1u) {
            const uint4 val = reinterpret_cast<const uint4*>(wst + r * 16)[ch ^ ((r >> 1) & 3)];
            reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.o_partial) + (prow0 + r) * kD +
                                     c * 32)[ch] = val;
          }
        }
        continue;
      }
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        stage_free();
#pragma unroll
        for (int i = 0; i < 4; ++i)
          reinterpret_cast<float4*>(wst + lane * 16)[i ^ ((lane >> 1) & 3)] =
              make_float4(v[16 * hf + 4 * i], v[16 * hf + 4 * i + 1], v[16 * hf + 4 * i + 2],
                          v[16 * hf + 4 * i + 3]);
        if (by_tma) {
          stage_store(c * 32 + 16 * hf);
          continue;
        }
        __syncwarp();
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int r = 8 * k + (lane >> 2);
          const int ch = lane & 3;
          if ((live >> r) & 1u) {
            const float4 val = reinterpret_cast<const float4*>(wst + r * 16)[ch ^ ((r >> 1) & 3)];
            reinterpret_cast<float4*>(static_cast<float*>(a.o_partial) + (prow0 + r) * kD +
                                      c * 32 + 16 * hf)[ch] = val;
          }
        }
      }
    }
    tc_fence_before();
    mbar_arrive(B.o_free + sb);
    if (prow >= 0) {
      a.m_partial[prow] = m2 == -INFINITY ? -INFINITY : m2 * kLn2;
      a.l_partial[prow] = l;
    }
    return true;
  };

  uint32_t T = 0;
  for (uint32_t U = 0;; ++U) {
    const int kvb = static_cast<int>(U % KVB);
    const bool gk = mbar_wait_bounded(B.kv_full + kvb, (U / KVB) & 1u);
    if (!__all_sync(0xffffffffu, gk)) {
      if (lane == 0) report(status, SA_ERR_DEVICE_TIMEOUT);
      return;
    }
    const UnitInfo info = reinterpret_cast<const UnitInfo*>(smem + P.info)[kvb];
    if (info.rows < 0) return;                          // end of work
    const int32_t* kpos = reinterpret_cast<const int32_t*>(smem + P.kpos) + kvb * BS;
    uint32_t vmask[BS / 32];
#pragma unroll
    for (int c = 0; c < BS / 32; ++c) vmask[c] = __ballot_sync(0xffffffffu, kpos[c * 32 + lane] >= 0);
    mbar_arrive(B.kv_empty + kvb);                      // info and keys read
    const int tiles = (info.rows + kM - 1) / kM;
    for (int tt = 0; tt < tiles; ++tt, ++T) {
      if ((T & 1u) != g) continue;                      // the other warpgroup's tile
      // This warpgroup's previous tile's partial row first: its O buffer is
      // then free by the time this tile's P is ready.
      if (prev && !epilogue(prevT, prev_prow, prev_m, prev_l)) {
        if (lane == 0) report(status, SA_ERR_DEVICE_TIMEOUT);
        return;
      }
      prev = false;
      const int sb = static_cast<int>(T & 1u);
      // This row's last live key of the block under the causal limit (its
      // query read before S is awaited).
      const int nrows = min(kM, info.rows - tt * kM);
      int jlim = -1;
      if (row < nrows) {
        jlim = BS - 1;
        if (a.causal) {
          const int rr = tt * kM + row;
          const int64_t qi = a.edges[2 * (info.e0 + rr / a.qhead)];
          const int64_t ql = qi - info.q0;
          const int64_t lim = a.causal == 2 || info.lk < info.qo ? ql : info.lk - info.qo + ql;
          const int64_t rel = lim - info.bstart;
          jlim = rel < -1 ? -1 : (rel > BS - 1 ? BS - 1 : static_cast<int>(rel));
        }
      }
      const bool got = mbar_wait_bounded(B.s_full + sb, (T >> 1) & 1u);
      if (!__all_sync(0xffffffffu, got)) {
        if (lane == 0) report(status, SA_ERR_DEVICE_TIMEOUT);
        return;
      }
      tc_fence_after();
      const uint32_t t_s = tmem + 128 * sb + lane_base;
      uint64_t l2 = f32x2(0.f, 0.f);          // two partial sums of p
      float m2;
      if constexpr (TcWarps<BS>::kWideS) {
      // S in halves of 64 keys, each read with one TMEM load (one round trip):
      // pass 1 takes the row maximum of qscale * s over live keys, as qscale
      // times the largest (qscale >= 0) or smallest raw score (rounding is
      // monotonic, so the product is the same maximum; fully live chunks, the
      // common case, without per-key masks, three scores per instruction).
      // Pass 2 turns each half into p = exp(s - m), l, and P as bf16 pairs
      // (16 columns per 32 keys): the half pass 1 read last is still in
      // registers and goes first, its P into columns 64.. of S (already
      // read), then the first half's P into columns 0..; the P V MMA reads
      // keys 64.. from there.
      constexpr int NH = BS / 64;
      auto live_of = [&](int c) -> uint32_t {      // live keys of 32-key chunk c
        const int cut = jlim - c * 32;
        const uint32_t inside = cut >= 31 ? 0xffffffffu : (cut < 0 ? 0u : ((2u << cut) - 1u));
        return vmask[c] & inside;
      };
      const bool up = qscale >= 0.f;
      float ext = up ? -INFINITY : INFINITY;
      bool any = false;
      float v[64];
#pragma unroll
      for (int hh = 0; hh < NH; ++hh) {
        tmem_ld64(t_s + hh * 64, v);
        tmem_ld_wait();
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2) {
          const uint32_t live = live_of(2 * hh + c2);
          const float* x = v + 32 * c2;
          any = any || live != 0u;
          if (live == 0xffffffffu) {
            if (up) {
#pragma unroll
              for (int i = 0; i < 32; i += 2) ext = max3(ext, x[i], x[i + 1]);
            } else {
#pragma unroll
              for (int i = 0; i < 32; i += 2) ext = min3(ext, x[i], x[i + 1]);
            }
          } else if (live) {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if ((live >> i) & 1u) ext = up ? fmaxf(ext, x[i]) : fminf(ext, x[i]);
          }
        }
      }
      m2 = any ? ext * qscale : -INFINITY;
      const float msub = m2 == -INFINITY ? 0.f : m2;
      const uint64_t qs2 = f32x2(qscale, qscale);
      const uint64_t nm2 = f32x2(-msub, -msub);
      // P of half hh (v) into pk[32]
      auto p_half = [&](int hh, uint32_t (&pk)[32]) {
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2) {
          const uint32_t live = live_of(2 * hh + c2);
          const float* x = v + 32 * c2;
          if (live == 0xffffffffu) {
#pragma unroll
            for (int i2 = 0; i2 < 16; ++i2) {
              float x0, x1;
              f32x2_split(fma_f32x2(f32x2(x[2 * i2], x[2 * i2 + 1]), qs2, nm2), x0, x1);
              const float p0 = ex2_fast(x0);
              const float p1 = ex2_fast(x1);
              l2 = add_f32x2(l2, f32x2(p0, p1));
              pk[16 * c2 + i2] = pack_bf16x2_rn(p0, p1);
            }
          } else {
#pragma unroll
            for (int i2 = 0; i2 < 16; ++i2) {
              const int i = 2 * i2;
              float x0, x1;
              f32x2_split(fma_f32x2(f32x2(x[i], x[i + 1]), qs2, nm2), x0, x1);
              const float p0 = ((live >> i) & 1u) ? ex2_fast(x0) : 0.f;
              const float p1 = ((live >> (i + 1)) & 1u) ? ex2_fast(x1) : 0.f;
              l2 = add_f32x2(l2, f32x2(p0, p1));
              pk[16 * c2 + i2] = pack_bf16x2_rn(p0, p1);
            }
          }
        }
      };
      {
        uint32_t pk[32];
        if constexpr (NH == 2) {
          p_half(1, pk);                     // keys 64..127, still in registers
          tmem_st32(t_s + 64, pk);           // over S columns already read
          tmem_ld64(t_s, v);                 // keys 0..63
          tmem_ld_wait();
        }
        p_half(0, pk);
        tmem_st32(t_s, pk);
      }
      } else {
      // S 32 keys per TMEM load: pass 1 takes the row maximum of qscale * s
      // over live keys, as qscale times the largest (qscale >= 0) or
      // smallest raw score (rounding is monotonic, so the product is the same
      // maximum; fully live chunks, the common case, without per-key masks,
      // three scores per instruction); pass 2 reads each chunk again and
      // writes P as bf16 pairs over the S columns already read (chunk c's 16
      // columns lie at or before S chunk c).
      auto live_of = [&](int c) -> uint32_t {      // live keys of 32-key chunk c
        const int cut = jlim - c * 32;
        const uint32_t inside = cut >= 31 ? 0xffffffffu : (cut < 0 ? 0u : ((2u << cut) - 1u));
        return vmask[c] & inside;
      };
      const bool up = qscale >= 0.f;
      float ext = up ? -INFINITY : INFINITY;
      bool any = false;
#pragma unroll 1
      for (int c = 0; c < BS / 32; ++c) {
        float v[32];
        tmem_ld32(t_s + c * 32, v);
        tmem_ld_wait();
        const uint32_t live = live_of(c);
        any = any || live != 0u;
        if (live == 0xffffffffu) {
          if (up) {
#pragma unroll
            for (int i = 0; i < 32; i += 2) ext = max3(ext, v[i], v[i + 1]);
          } else {
#pragma unroll
            for (int i = 0; i < 32; i += 2) ext = min3(ext, v[i], v[i + 1]);
          }
        } else if (live) {
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if ((live >> i) & 1u) ext = up ? fmaxf(ext, v[i]) : fminf(ext, v[i]);
        }
      }
      m2 = any ? ext * qscale : -INFINITY;
      const float msub = m2 == -INFINITY ? 0.f : m2;
      const uint64_t qs2 = f32x2(qscale, qscale);
      const uint64_t nm2 = f32x2(-msub, -msub);
#pragma unroll 1
      for (int c = 0; c < BS / 32; ++c) {
        float v[32];
        tmem_ld32(t_s + c * 32, v);
        tmem_ld_wait();
        const uint32_t live = live_of(c);
        uint32_t pk[16];
        if (live == 0xffffffffu) {
#pragma unroll
          for (int i2 = 0; i2 < 16; ++i2) {
            float x0, x1;
            f32x2_split(fma_f32x2(f32x2(v[2 * i2], v[2 * i2 + 1]), qs2, nm2), x0, x1);
            const float p0 = ex2_fast(x0);
            const float p1 = ex2_fast(x1);
            l2 = add_f32x2(l2, f32x2(p0, p1));
            pk[i2] = pack_bf16x2_rn(p0, p1);
          }
        } else {
#pragma unroll
          for (int i2 = 0; i2 < 16; ++i2) {
            const int i = 2 * i2;
            float x0, x1;
            f32x2_split(fma_f32x2(f32x2(v[i], v[i + 1]), qs2, nm2), x0, x1);
            const float p0 = ((live >> i) & 1u) ? ex2_fast(x0) : 0.f;
            const float p1 = ((live >> (i + 1)) & 1u) ? ex2_fast(x1) : 0.f;
            l2 = add_f32x2(l2, f32x2(p0, p1));
            pk[i2] = pack_bf16x2_rn(p0, p1);
          }
        }
        tmem_st16(t_s + c * 16, pk);
      }
      }
      float la, lb;
      f32x2_split(l2, la, lb);
      const float l = la + lb;
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(B.p_full + sb);
      prev = true;
      prevT = T;
      prev_prow = row < nrows ? info.prow0 + static_cast<int64_t>(tt) * kM + row : -1;
      prev_m = m2;
      prev_l = l;
    }
    // The unit's last tile before the next unit's keys.
    if (prev && !epilogue(prevT, prev_prow, prev_m, prev_l)) {
      if (lane == 0) report(status, SA_ERR_DEVICE_TIMEOUT);
      return;
    }
    prev = false;
  }
}

// ------------------------------------------------------------------ kernel

template <int BS, bool kBf16, bool kTf32>
__global__ void __launch_bounds__(TcWarps<BS>::kThreads, 1)
forward_tc_kernel(const __grid_constant__ CUtensorMap omap, ForwardArgs a) {
  constexpr int KVB = TcCfg<BS, kTf32>::KVB;
  constexpr int kNX = TcCfg<BS, kTf32>::NX;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const TcPlan P = tc_plan<BS, kTf32>();
  using W = TcWarps<BS>;
  constexpr int kLoadThreads = W::kLoadThreads;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + P.bars);
  TcBars B;
  B.kv_full = bars;
  B.kv_empty = bars + 2;
  B.x_full = bars + 4;
  B.x_empty = bars + 4 + kMaxNX;
  B.s_full = bars + 4 + 2 * kMaxNX;
  B.s_free = B.s_full + 2;
  B.p_full = B.s_full + 4;
  B.o_full = B.s_full + 6;
  B.o_free = B.s_full + 8;
  B.done = B.s_full + 10;
  B.slot_full = B.done + 1;
  B.slot_empty = B.slot_full + kRing;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + P.misc);
  int32_t* unit_base = reinterpret_cast<int32_t*>(smem + P.misc + 16);   // [hkv + 1]

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const long long t_start = clock64();
  if (warp == 0) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  if (tid == 32) {
    for (int i = 0; i < KVB; ++i) {
      mbar_init(B.kv_full + i, kLoadThreads);
      // freed by the unit's last MMA and by both softmax warpgroups (which
      // read the unit's info and keys even when a one-tile unit gives them
      // no tile)
      mbar_init(B.kv_empty + i, 1 + 2 * kM);
    }
    for (int i = 0; i < kNX; ++i) {
      mbar_init(B.x_full + i, kLoadThreads);
      mbar_init(B.x_empty + i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(B.s_full + i, 1);
      mbar_init(B.s_free + i, 1);
      mbar_init(B.p_full + i, kM);
      mbar_init(B.o_full + i, 1);
      mbar_init(B.o_free + i, kM);
    }
    mbar_init(B.done, 1);
    for (int i = 0; i < kRing; ++i) {
      mbar_init(B.slot_full + i, 32);
      mbar_init(B.slot_empty + i, kLoadThreads);
    }
    fence_mbar_init();
    // (a head never has more units than slots; the bound only matters for an
    // index whose build did not finish)
    int32_t acc = 0;
    for (int hh = 0; hh < a.hkv; ++hh) {
      unit_base[hh] = acc;
      acc += static_cast<int32_t>(min(max(static_cast<int64_t>(a.num_sel[hh]), int64_t{0}), a.nbs));
    }
    if (a.unit_order != nullptr && acc > a.max_units) acc = static_cast<int32_t>(a.max_units);
    unit_base[a.hkv] = acc;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int64_t n_units = unit_base[a.hkv];
  if (warp >= W::kSoftmaxWarp0) {
    tc_softmax<BS, kTf32>(a, &omap, smem, P, B, tmem, warp, lane);
    // box stores issued by this thread have landed before the CTA leaves
    bulk_wait_all();
  } else {
    if (warp == 0) {
      if (lane == 0) {
        tc_mma<BS, kTf32>(a, smem, P, B, tmem);
        // Every MMA issued has completed before TMEM is released.
        mma_commit(B.done);
        if (!mbar_wait_bounded(B.done, 0)) report(a.totals + 3, SA_ERR_DEVICE_TIMEOUT);
      }
      __syncwarp();
    } else if (warp == kSchedWarp) {
      tc_scheduler<BS>(a, smem, P, B, unit_base, n_units, lane);
    } else {
      tc_loader<BS, kBf16, kTf32>(a, smem, P, B, warp - kLoaderWarp0, lane);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
  if (tid == 0 && a.cta_stats != nullptr && static_cast<int>(blockIdx.x) < a.cta_stats_len)
    a.cta_stats[3 * blockIdx.x + 2] = clock64() - t_start;
}

// The longest-first work list: every unit (kv head, compact slot) of the
// index, numbered across heads as the scheduler numbers them.  Cost model:
// a unit costs about its edges (each edge is qhead rows of the tile loop);
// a unit whose cost reaches a thirty-second of a CTA's mean share (E / ctas / 32
// edges) is heavy and could leave the SMs idle behind it if claimed late,
// so heavy units come first, in classes of descending size (2^c <= edges <
// 2^(c+1)); the light rest keep index order, where neighbouring blocks,
// claimed at the same time by different CTAs, share their queries' Q rows
// in L2 (an order by size alone scattered them and cost more than it
// balanced).  Inside a class, index order.  Two kernels over the same grid
// of 1024-unit chunks: the first counts each chunk's units per class, the
// second places each chunk's units after the larger classes and after the
// earlier chunks' units of its class, warp by warp, lane by lane.
constexpr int kOrderThreads = 1024;
constexpr int kOrderClasses = 16;

// Unit u's class (-1 past the end) from the per-head unit bases: 0 for a
// light unit, 1 + floor(log2(edges)) (at most the last class) for a heavy one.
__device__ __forceinline__ int unit_class(const ForwardArgs& a, const int32_t* ubase, int64_t n,
                                          int64_t u, int64_t heavy) {
  if (u >= n) return -1;
  int h = 0;
  while (h + 1 < a.hkv && ubase[h + 1] <= u) ++h;
  const int32_t* off = a.sel_offsets + static_cast<int64_t>(h) * (a.nbs + 1) + (u - ubase[h]);
  const int c = max(off[1] - off[0], 1);
  if (c < heavy) return 0;
  return min(1 + 31 - __clz(c), kOrderClasses - 1);
}

// Edges from which a unit is heavy: a thirty-second of a CTA's mean share.
__device__ __forceinline__ int64_t heavy_edges(const ForwardArgs& a) {
  const int64_t e = a.totals[0] > 0 ? a.totals[0] : 0;
  const int64_t share = e / (32 * static_cast<int64_t>(a.order_ctas > 0 ? a.order_ctas : 1));
  return share > 1 ? share : 1;
}

__device__ __forceinline__ int64_t order_unit_bases(const ForwardArgs& a, int32_t* ubase) {
  if (threadIdx.x == 0) {
    int32_t acc = 0;
    for (int hh = 0; hh < a.hkv; ++hh) {
      ubase[hh] = acc;
      acc += static_cast<int32_t>(min(max(static_cast<int64_t>(a.num_sel[hh]), int64_t{0}), a.nbs));
    }
    ubase[a.hkv] = acc > a.max_units ? static_cast<int32_t>(a.max_units) : acc;
  }
  __syncthreads();
  return ubase[a.hkv];
}

// counts[chunk][class] of the chunk's units
__global__ void __launch_bounds__(kOrderThreads) unit_class_count_kernel(ForwardArgs a) {
  __shared__ int32_t ubase[201];
  __shared__ uint32_t cnt[kOrderClasses];
  const int tid = threadIdx.x, lane = tid & 31;
  if (tid < kOrderClasses) cnt[tid] = 0;
  const int64_t n = order_unit_bases(a, ubase);
  const int c = unit_class(a, ubase, n, static_cast<int64_t>(blockIdx.x) * kOrderThreads + tid,
                          heavy_edges(a));
  const unsigned peers = __match_any_sync(0xffffffffu, c);
  if (c >= 0 && lane == __ffs(peers) - 1) atomicAdd(&cnt[c], static_cast<uint32_t>(__popc(peers)));
  __syncthreads();
  if (tid < kOrderClasses) a.order_counts[blockIdx.x * kOrderClasses + tid] = cnt[tid];
}

__global__ void __launch_bounds__(kOrderThreads) unit_order_kernel(ForwardArgs a) {
  __shared__ int32_t ubase[201];
  __shared__ uint32_t base[kOrderClasses], total[kOrderClasses], before[kOrderClasses];
  __shared__ uint32_t wcnt[kOrderThreads / 32][kOrderClasses];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid < kOrderClasses) total[tid] = before[tid] = 0;
  const int64_t n = order_unit_bases(a, ubase);
  // every chunk's class counts: per class the total, and the earlier chunks'
  for (int64_t e = tid; e < static_cast<int64_t>(gridDim.x) * kOrderClasses; e += kOrderThreads) {
    const uint32_t x = a.order_counts[e];
    const int cc = static_cast<int>(e % kOrderClasses);
    if (x) {
      atomicAdd(&total[cc], x);
      if (e / kOrderClasses < blockIdx.x) atomicAdd(&before[cc], x);
    }
  }
  __syncthreads();
  if (tid < kOrderClasses) {
    uint32_t larger = 0;
    for (int cc = tid + 1; cc < kOrderClasses; ++cc) larger += total[cc];
    base[tid] = larger + before[tid];
  }
  const int64_t u = static_cast<int64_t>(blockIdx.x) * kOrderThreads + tid;
  const int c = unit_class(a, ubase, n, u, heavy_edges(a));
  // rank among the warp's units of the same class, and the warp's counts
  const unsigned peers = __match_any_sync(0xffffffffu, c);
  const uint32_t rank = __popc(peers & ((1u << lane) - 1u));
  if (lane < kOrderClasses) wcnt[warp][lane] = 0;
  __syncwarp();
  if (c >= 0 && lane == __ffs(peers) - 1) wcnt[warp][c] = __popc(peers);
  __syncthreads();
  if (tid < kOrderClasses) {
    uint32_t run = base[tid];
    for (int w = 0; w < kOrderThreads / 32; ++w) {
      const uint32_t x = wcnt[w][tid];
      wcnt[w][tid] = run;
      run += x;
    }
  }
  __syncthreads();
  if (c >= 0) a.unit_order[wcnt[warp][c] + rank] = static_cast<int32_t>(u);
}

template <int BS, bool kBf16, bool kTf32>
cudaError_t launch_tc(const ForwardArgs& a, cudaStream_t stream) {
  const TcPlan p = tc_plan<BS, kTf32>();
  if (p.total > 227 * 1024) return cudaErrorNotSupported;
  const void* fn = reinterpret_cast<const void*>(forward_tc_kernel<BS, kBf16, kTf32>);
  cudaError_t err =
      cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(p.total));
  if (err != cudaSuccess) return err;
  err = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
  if (err != cudaSuccess) return err;
  // The partial o rows [capacity, 128] as a 2-D tensor map for the
  // epilogue's box stores (32 rows x 64 bytes, 64-byte swizzle); without one
  // (capacity outside int32 coordinates, or no encoder) every row goes out
  // through plain stores.
  ForwardArgs args = a;
  args.o_tma = 0;
  CUtensorMap omap{};
  const int64_t cap = a.max_splits * a.qhead;
  EncodeTiledFn enc = encode_fn();
  if (enc != nullptr && cap >= 32 && cap < (int64_t{1} << 31)) {
    const cuuint64_t dims[2] = {kD, static_cast<cuuint64_t>(cap)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kD) * (a.o_bf16 ? 2 : 4)};
    const cuuint32_t box[2] = {a.o_bf16 ? 32u : 16u, 32u};
    const cuuint32_t estr[2] = {1, 1};
    if (enc(&omap, a.o_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
            2, a.o_partial, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS)
      args.o_tma = 1;
  }
  // The work counter starts at zero for every launch, and walks the
  // longest-first list where the index workspace has room for one.
  if (args.unit_counter != nullptr) {
    const cudaError_t e = cudaMemsetAsync(args.unit_counter, 0, sizeof(uint32_t), stream);
    if (e != cudaSuccess) return e;
  } else {
    args.unit_order = nullptr;
  }
  // One CTA per SM: it holds all 512 TMEM columns.
  int64_t grid = device_sm_count();
  if (grid > a.max_splits) grid = a.max_splits;
  if (grid < 1) grid = 1;
  args.order_ctas = static_cast<int32_t>(grid);
  if (args.unit_order != nullptr) {
    const unsigned chunks = static_cast<unsigned>((args.max_units + kOrderThreads - 1) / kOrderThreads);
    unit_class_count_kernel<<<chunks, kOrderThreads, 0, stream>>>(args);
    unit_order_kernel<<<chunks, kOrderThreads, 0, stream>>>(args);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  forward_tc_kernel<BS, kBf16, kTf32>
      <<<static_cast<unsigned>(grid), TcWarps<BS>::kThreads, p.total, stream>>>(omap, args);
  return cudaGetLastError();
}

}  // namespace

namespace {

__global__ void __launch_bounds__(256) q_to_bf16_kernel(const float4* __restrict__ q,
                                                        uint4* __restrict__ q16, int64_t n8) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const float4 x = q[2 * i];
    const float4 y = q[2 * i + 1];
    q16[i] = make_uint4(pack_bf16x2_rn(x.x, x.y), pack_bf16x2_rn(x.z, x.w),
                        pack_bf16x2_rn(y.x, y.y), pack_bf16x2_rn(y.z, y.w));
  }
}

}  // namespace

cudaError_t launch_q_to_bf16(const float* q, uint16_t* q16, int64_t n, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  if (n % 8 != 0) return cudaErrorInvalidValue;
  const int64_t n8 = n / 8;
  int64_t grid = static_cast<int64_t>(device_sm_count()) * 8;
  const int64_t need = (n8 + 255) / 256;
  if (grid > need) grid = need;
  q_to_bf16_kernel<<<static_cast<unsigned>(grid), 256, 0, stream>>>(
      reinterpret_cast<const float4*>(q), reinterpret_cast<uint4*>(q16), n8);
  return cudaGetLastError();
}

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
  // tf32 operands only for f32 K/V (bf16 K/V are exact in bf16)
  const bool tf32 = a.tf32 && !a.kv_bf16;
  if (a.block_size == 64) {
    if (a.kv_bf16) return launch_tc<64, true, false>(a, stream);
    return tf32 ? launch_tc<64, false, true>(a, stream) : launch_tc<64, false, false>(a, stream);
  }
  if (a.kv_bf16) return launch_tc<128, true, false>(a, stream);
  return tf32 ? launch_tc<128, false, true>(a, stream) : launch_tc<128, false, false>(a, stream);
}

}  // namespace sa
