// Internal launch interfaces between the C ABI (api.cu) and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "sa.h"

namespace sa {

// Entries of one (kv head, sequence) segment handled by one CTA of the index
// kernel at a time.
constexpr int kChunkEntries = 4096;

// Layout of the index workspace (bytes from its start).
struct WorkspaceLayout {
  size_t barrier;       // uint32[2]: grid barrier counter and generation
  size_t unit_ctr;      // uint32: units claimed by a tensor-core forward (within the
                        // barrier's 256-byte block, outside the index build's use)
  size_t seg_done;      // uint32[hkv*batch]: chunks of the segment that finished phase 1
  size_t item_cnt;      // uint32[tq*hkv]: finished pieces per (query, kv head), fused decode
  size_t seg_tot;       // int32[hkv*batch][3]: edges, non-empty bins, work splits
  size_t seg_pre;       // int64[hkv*batch+1][3]: exclusive prefixes of seg_tot
  size_t hist;          // int32[hkv][slots][msb]: histograms of multi-chunk segments
  size_t zero_bytes;    // bytes cleared at the start of every build
  size_t total;
};

WorkspaceLayout workspace_layout(int32_t hkv, int32_t batch, int64_t tq,
                                 int64_t hist_slots_per_head, int32_t msb);

// The tensor-core forward's longest-first work list in the index workspace,
// after everything an index build of these sizes may use: `offset` bytes
// from the workspace start, `bytes` long (int32 per possible work unit).
struct LptRegion {
  size_t offset, bytes;     // the list (int32 per unit), then the sort's counts
  size_t counts;            // offset of the counts from `offset`
  int64_t units;
};
LptRegion lpt_region(int64_t tq, int32_t hkv, int32_t topk, int32_t batch, int32_t msb,
                     int64_t nbs);
// Chunks of one head (and, in *multi_slots, chunks of its multi-chunk segments).
int64_t index_chunks_per_head(const int64_t* cu_host, int32_t batch, int32_t topk,
                              int64_t* multi_slots);
// Upper bound of the multi-chunk histogram slots of one head.
int64_t index_hist_slot_bound(int64_t tq, int32_t topk);

// Test hook (sa_debug_stall): a site whose bounded wait is made to run out,
// and the tries a bounded wait takes before it gives up (0 = kSpinLimit).
enum StallSite { kStallNone = 0, kStallIndexBarrier = 1, kStallFusedCopies = 2 };
void debug_stall_setting(int* site, uint32_t* spin_limit);
// Test hook (sa_debug_cta_stats): where the tensor-core forward adds up each
// CTA's rows, units and busy cycles (NULL: nowhere), and its length in CTAs.
void debug_cta_stats(int64_t** buf, int32_t* n_ctas);

struct IndexArgs {
  const int32_t* selected;
  const int64_t* cu;
  const int32_t* used;      // nullable
  int64_t tq;
  int32_t hkv, topk, batch, msb, block_size, split_edges;
  int64_t nbs;
  sa_index idx;             // output arrays + workspace
  uint32_t spin_limit;      // tries of the grid barrier's wait (0 = kSpinLimit)
  int stall;                // test hook: the grid barrier is never released
  int small;                // every segment holds at most kSmallSegment entries
                            // (decode batches): one warp per segment
  int external_clear;       // the workspace counters and the status word were
                            // cleared by the caller, on the stream this build
                            // waits on (the build runs beside a fused decode
                            // kernel that may already report into the status)
};

// Largest segment (entries of one (kv head, sequence)) of the index kernel's
// warp-per-segment mode: two entries per lane.
constexpr int kSmallSegment = 64;

cudaError_t launch_build_index(const IndexArgs& a, int64_t chunks_per_head,
                               int64_t hist_slots_per_head, cudaStream_t stream);

// Clears `bytes` (a multiple of 16) of a 16-byte-aligned workspace and the
// status word in one launch.
cudaError_t launch_clear_for_build(void* workspace, size_t bytes, int64_t* status,
                                   cudaStream_t stream);

struct ForwardArgs {
  const float* q;
  const void* k_pages;
  const void* v_pages;
  int64_t num_pages;
  int kv_bf16;
  const int32_t* block_tables;
  const int64_t* cu;
  const int32_t* used;      // nullable
  int32_t hq, hkv, qhead, head_dim, block_size, page_size, pages_per_block, max_pages, msb;
  int64_t nbs;
  float scale;
  int causal;               // 0 none, 1 right-aligned, 2 left-aligned
  // index
  const int32_t* sel_slots;
  const int32_t* sel_offsets;
  const int32_t* num_sel;
  const int64_t* edge_head_base;
  const int32_t* edges;
  const int32_t* splits;
  int64_t* totals;          // [0] E, [1] splits, [3] status
  int64_t max_splits;       // capacity of the split list (upper bound of totals[1])
  // outputs
  void* o_partial;          // f32, or bf16 when o_bf16
  int o_bf16;
  int o_tma;                // set by a launcher: o rows may go out by tensor-map stores
  const uint16_t* q16;      // nullable: Q rounded to bf16, same layout (tensor-core kernel)
  int tf32;                 // tensor-core kernel: f32 K/V as tf32 operands (else bf16)
  uint32_t* unit_counter;   // nullable: the tensor-core kernel's work counter (in the
                            // index workspace; cleared by its launcher)
  int32_t* unit_order;      // nullable: room for one int32 per possible unit (in the
                            // index workspace): the launcher writes the units there in
                            // longest-first order and the counter walks that list
  int64_t max_units;        // entries unit_order has room for
  uint32_t* order_counts;   // [ceil(max_units / 1024)][16] scratch of the list's sort
  int32_t order_ctas;       // CTAs of the forward (the list's cost model)
  int64_t* cta_stats;       // nullable (test hook): per CTA rows, units, busy cycles
  int32_t cta_stats_len;    // CTAs cta_stats has room for
  float* m_partial;
  float* l_partial;
};

// Returns cudaErrorNotSupported when the shape has no kernel.
cudaError_t launch_forward_cc(const ForwardArgs& a, cudaStream_t stream);
bool forward_cc_supported(int head_dim, int block_size, int kv_bf16);

// Tensor-core (tcgen05) forward for units with many gathered rows.
cudaError_t launch_forward_tc(const ForwardArgs& a, cudaStream_t stream);
// q [n] f32 -> q16 [n] bf16 (round to nearest even); n a multiple of 8,
// both 16-byte aligned.
cudaError_t launch_q_to_bf16(const float* q, uint16_t* q16, int64_t n, cudaStream_t stream);
bool forward_tc_supported(int head_dim, int block_size, int page_size, int qhead);

// Decode-shaped forward with bf16 K/V on warp-level tensor-core MMA.
cudaError_t launch_forward_dec_mma(const ForwardArgs& a, cudaStream_t stream);
bool forward_dec_mma_supported(int head_dim, int block_size, int page_size, int qhead,
                               int kv_bf16);

// Pipelined decode-shaped forward (head_dim 128, few rows per split).
cudaError_t launch_forward_dec(const ForwardArgs& a, cudaStream_t stream);
bool forward_dec_supported(int head_dim, int block_size, int page_size, int qhead, int kv_bf16);

// Fused decode attention (forward and combine in one kernel) for batches in
// which every sequence holds at most one query.
struct FusedDecArgs {
  const float* q;
  const void* k_pages;
  const void* v_pages;
  int64_t num_pages;
  int kv_bf16;
  const int32_t* block_tables;
  const int64_t* cu;
  const int32_t* used;      // nullable
  const int32_t* selected;  // [tq, hkv, topk]
  const int32_t* inv;       // [hkv, tq, topk] of the built index
  int64_t tq;
  int32_t batch, hq, hkv, qhead, topk, block_size, page_size, pages_per_block, max_pages, msb;
  int64_t whole_items;      // (query, kv head) pairs [0, whole_items): one piece of all
                            // ranks each (topk <= 64); the rest: `pieces` pieces each
  int32_t pieces;           // pieces per pair from whole_items on
  int32_t ranks_per_piece;  // ranks of one of those pieces, at most 64
  float scale;
  int64_t* status;          // device status word
  uint32_t* item_cnt;       // [tq * hkv], zero on entry, left zero
  void* part_o;             // per-piece scratch rows (the partial buffers):
  int part_bf16;            // o rows f32, or bf16 when part_bf16
  float* part_m;
  float* part_l;
  float* out;
  float* lse;               // nullable
  int pdl;                  // launched right behind the index kernel that built the
                            // index: it may start while that kernel runs (it reads
                            // nothing the index writes) and waits for it at its end
  uint32_t spin_limit;      // tries of every mbarrier wait (0 = kSpinLimit)
  int stall;                // test hook: the load warps issue no copy at all
};

// Whether the fused decode kernel supports this shape (the caller also checks
// that every sequence holds at most one query and the pool size limits).
bool fused_dec_supported(int head_dim, int block_size, int page_size, int qhead, int kv_bf16);
// Largest pool (num_pages * hkv * page_size key rows) the kernel addresses.
constexpr int64_t kFusedMaxRows = (int64_t{1} << 31) - 1;
cudaError_t launch_fused_dec(const FusedDecArgs& a, cudaStream_t stream);

struct CombineArgs {
  const int32_t* inv;
  const int64_t* edge_head_base;
  const void* o_partial;    // f32, or bf16 when o_bf16
  int o_bf16;
  const float* m_partial;
  const float* l_partial;
  int64_t tq;
  int32_t hkv, topk, qhead, head_dim;
  float* out;
  float* lse;               // nullable
};

cudaError_t launch_combine(const CombineArgs& a, cudaStream_t stream);

int device_sm_count();

// The fixed scratch array of sa_build_index_no_alloc on the current device
// (no_alloc.cu): its device address and size.
sa_status static_index_scratch(void** ptr, size_t* bytes);

// cuTensorMapEncodeTiled from the driver (NULL if unavailable); looked up once.
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_fn();

}  // namespace sa
