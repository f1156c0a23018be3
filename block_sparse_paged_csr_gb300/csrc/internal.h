// Internal launch interfaces between the C ABI (api.cu) and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "sa.h"

namespace sa {

// Layout of the index workspace (bytes from its start).
struct WorkspaceLayout {
  size_t ticket;        // uint32: next segment ticket of the index kernel
  size_t seg_a;         // uint64[hkv*batch]: flag | edges
  size_t seg_b;         // uint64[hkv*batch]: flag | units | splits
  size_t head_units;    // int32[hkv]: non-empty units before head h
  size_t zero_bytes;    // bytes cleared at the start of every build
  size_t total;
};

WorkspaceLayout workspace_layout(int32_t hkv, int32_t batch);

struct IndexArgs {
  const int32_t* selected;
  const int64_t* cu;
  const int32_t* used;      // nullable
  int64_t tq;
  int32_t hkv, topk, batch, msb, block_size, split_edges;
  int64_t nbs;
  sa_index idx;             // output arrays + workspace
};

cudaError_t launch_build_index(const IndexArgs& a, cudaStream_t stream);

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
  int causal;
  // index
  const int32_t* sel_slots;
  const int32_t* edges;
  const int32_t* splits;
  int64_t* totals;          // [0] E, [1] splits, [3] status
  int64_t max_splits;       // capacity of the split list (upper bound of totals[1])
  // outputs
  float* o_partial;
  float* m_partial;
  float* l_partial;
};

// Returns cudaErrorNotSupported when the shape has no kernel.
cudaError_t launch_forward_cc(const ForwardArgs& a, cudaStream_t stream);
bool forward_cc_supported(int head_dim, int block_size, int kv_bf16);

// Pipelined decode-shaped forward (head_dim 128, few rows per split).
cudaError_t launch_forward_dec(const ForwardArgs& a, cudaStream_t stream);
bool forward_dec_supported(int head_dim, int block_size, int page_size, int qhead, int kv_bf16);

struct CombineArgs {
  const int32_t* inv;
  const int64_t* edge_head_base;
  const float* o_partial;
  const float* m_partial;
  const float* l_partial;
  int64_t tq;
  int32_t hkv, topk, qhead, head_dim;
  float* out;
  float* lse;               // nullable
};

cudaError_t launch_combine(const CombineArgs& a, cudaStream_t stream);

int device_sm_count();

}  // namespace sa
