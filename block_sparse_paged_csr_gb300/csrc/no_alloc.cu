// sa_build_index_no_alloc: the index build with its scratch memory taken from
// a fixed array compiled into this library instead of a caller-provided
// workspace.
//
// Who needs it: callers that must not allocate device memory at call time:
// an inference server whose memory pool is fixed at start-up, code running
// where a cudaMalloc would synchronise the device or fail under a memory cap,
// or a host runtime that has no allocator to hand.  They still own the index
// arrays and the selection inputs; only the scratch moves into the library.
//
// The scratch holds what the index build keeps outside the index arrays
// (workspace_layout in index.cu): the grid barrier, the segment tickets, one
// counter per (query, kv head) for the fused decode kernel, the segment
// totals and prefixes, and the histograms of multi-chunk segments.  An index
// built here carries SA_INDEX_STATIC_SCRATCH, and the forward entry points
// then take their counters from this array too (index_scratch in api.cu).
// Every GPU that loads this library keeps its own copy of the array until the
// process exits.
#include <cstdint>
#include <mutex>

#include "internal.h"
#include "sa.h"

namespace {

// 288 KiB.  Per (kv head, sequence) segment 40 bytes (ticket 4, totals 12,
// prefixes 24), per (query, kv head) 4 bytes, per 4096-entry chunk of a
// multi-chunk segment msb 4-byte bins, plus the barrier block and roundings
// to 256 bytes (workspace_layout in index.cu; the formula is in sa.h).
constexpr size_t kStaticScratchBytes = 288 * 1024;

static __device__ __align__(256) unsigned char g_index_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of g_index_scratch on the current device, looked up once per
// device.  The name g_index_scratch in host code is only a host-side stand-in,
// so the address must come from cudaGetSymbolAddress with that device current.
sa_status scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return SA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_index_scratch) != cudaSuccess || p == nullptr)
      return SA_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return SA_OK;
}

}  // namespace

namespace sa {

sa_status static_index_scratch(void** ptr, size_t* bytes) {
  const sa_status st = scratch_for_current_device(ptr);
  if (st == SA_OK) *bytes = kStaticScratchBytes;
  return st;
}

}  // namespace sa

extern "C" sa_status sa_build_index_no_alloc(const int32_t* selected, int64_t tq, int32_t hkv,
                                             int32_t topk, const int64_t* cu_seqlens_q_host,
                                             const int64_t* cu_seqlens_q, int32_t batch,
                                             const int32_t* used_kv_lens, int32_t max_pages,
                                             int32_t block_size, int32_t page_size,
                                             int32_t split_edges, sa_index* idx, void* stream) {
  if (idx == nullptr) return SA_ERR_INVALID_ARGUMENT;
  if (hkv > 0 && batch > 0 && topk > 0 && cu_seqlens_q_host != nullptr && block_size > 0 &&
      page_size > 0 && block_size % page_size == 0) {
    int64_t multi_slots = 0;
    sa::index_chunks_per_head(cu_seqlens_q_host, batch, topk, &multi_slots);
    const int64_t msb = max_pages / (block_size / page_size);
    if (sa::workspace_layout(hkv, batch, tq, multi_slots, static_cast<int32_t>(msb)).total >
        kStaticScratchBytes)
      return SA_ERR_UNSUPPORTED;  // the problem needs more scratch than the array holds
  }
  void* scratch = nullptr;
  if (hkv > 0 && batch > 0) {
    const sa_status st = scratch_for_current_device(&scratch);
    if (st != SA_OK) return st;
  }
  // Run the regular build on a copy of the caller's index whose workspace is
  // the static scratch; the build clears the part of it that must start at
  // zero on the stream before its kernels run.
  sa_index local = *idx;
  local.workspace = scratch;
  local.workspace_bytes = kStaticScratchBytes;
  const sa_status st =
      sa_build_index(selected, tq, hkv, topk, cu_seqlens_q_host, cu_seqlens_q, batch,
                     used_kv_lens, max_pages, block_size, page_size, split_edges, &local, stream);
  if (st == SA_OK) {
    void* keep_ws = idx->workspace;
    const size_t keep_bytes = idx->workspace_bytes;
    *idx = local;
    idx->workspace = keep_ws;
    idx->workspace_bytes = keep_bytes;
    idx->flags = SA_INDEX_STATIC_SCRATCH;
  }
  return st;
}
