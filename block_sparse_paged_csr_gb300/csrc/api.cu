// C ABI of libsa (declared in include/sa.h): argument checks in the order of
// kvouter_forward's "argument sanity" (forward.rs) and of the error enum
// (types.rs), then kernel launches on the caller's stream.
#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "internal.h"
#include "sa.h"
#include "sa_common.cuh"

namespace sa {

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

namespace {
std::atomic<int> g_stall_site{kStallNone};
std::atomic<uint32_t> g_spin_limit{0};
}  // namespace

namespace {
std::atomic<int64_t*> g_cta_stats{nullptr};
std::atomic<int32_t> g_cta_stats_len{0};
}  // namespace

void debug_cta_stats(int64_t** buf, int32_t* n_ctas) {
  *n_ctas = g_cta_stats_len.load(std::memory_order_relaxed);
  *buf = *n_ctas > 0 ? g_cta_stats.load(std::memory_order_relaxed) : nullptr;
}

void debug_stall_setting(int* site, uint32_t* spin_limit) {
  *site = g_stall_site.load(std::memory_order_relaxed);
  *spin_limit = g_spin_limit.load(std::memory_order_relaxed);
}

int device_sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (dev >= 0 && dev < 64 && cached[dev] > 0) return cached[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
    n = 1;
  if (dev >= 0 && dev < 64) cached[dev] = n;
  return n;
}

}  // namespace sa

namespace {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

enum class FwdKernel { kNone, kGeneral, kDecode, kDecodeMma, kTensor };

// The forward kernel a call takes.  Decode-shaped problems (tq at most twice
// the batch: about one query per sequence, so few rows per work split) go to
// the per-warp decode kernels (warp-level MMA for bf16 K/V, f32 FMA
// otherwise); problems whose units gather many rows go to the tcgen05
// kernel; the general f32 kernel takes whatever the others do not support.
FwdKernel choose_forward(int64_t tq, int32_t batch, int32_t qhead, int32_t head_dim,
                         int32_t block_size, int32_t page_size, int kv_bf16, sa_path path) {
  const bool decode_like = tq <= 2 * static_cast<int64_t>(batch);
  const bool tc_ok = sa::forward_tc_supported(head_dim, block_size, page_size, qhead);
  const bool mma_ok =
      sa::forward_dec_mma_supported(head_dim, block_size, page_size, qhead, kv_bf16);
  const bool dec_ok = sa::forward_dec_supported(head_dim, block_size, page_size, qhead, kv_bf16);
  const bool cc_ok = sa::forward_cc_supported(head_dim, block_size, kv_bf16);
  switch (path) {
    case SA_PATH_TENSOR_CORE:
    case SA_PATH_TENSOR_CORE_TF32:
      if (decode_like && mma_ok) return FwdKernel::kDecodeMma;
      return tc_ok ? FwdKernel::kTensor : FwdKernel::kNone;
    case SA_PATH_CUDA_CORE:
      if (!cc_ok) return FwdKernel::kNone;
      return dec_ok ? FwdKernel::kDecode : FwdKernel::kGeneral;
    case SA_PATH_CUDA_CORE_GENERAL:
      return cc_ok ? FwdKernel::kGeneral : FwdKernel::kNone;
    case SA_PATH_AUTO:
      if (!cc_ok) return FwdKernel::kNone;
      if (decode_like && mma_ok) return FwdKernel::kDecodeMma;
      if (decode_like && dec_ok) return FwdKernel::kDecode;
      if (!decode_like && tc_ok) return FwdKernel::kTensor;
      return FwdKernel::kGeneral;
    default:
      return FwdKernel::kNone;
  }
}

// Whether steps 2 and 3 run as the fused decode kernel: every sequence holds
// at most one query (then each work unit carries edges of one query only)
// and the shape is one the kernel supports.
bool fused_eligible(int64_t tq, int32_t batch, const int64_t* cu_host, int64_t num_pages,
                    int32_t hq, int32_t hkv, int32_t head_dim, int32_t block_size,
                    int32_t page_size, int kv_bf16) {
  if (cu_host == nullptr || batch < 1 || tq < 1 || hkv < 1 || hq % hkv != 0) return false;
  if (!sa::fused_dec_supported(head_dim, block_size, page_size, hq / hkv, kv_bf16)) return false;
  if (num_pages < 1 || num_pages > sa::kFusedMaxRows / (static_cast<int64_t>(hkv) * page_size))
    return false;
  if (tq * hq * 4 > sa::kFusedMaxRows) return false;
  for (int32_t b = 0; b < batch; ++b)
    if (cu_host[b + 1] - cu_host[b] > 1) return false;
  return true;
}

const char* forward_kernel_name(FwdKernel k) {
  switch (k) {
    case FwdKernel::kDecodeMma: return "forward_dec_mma_kernel";
    case FwdKernel::kTensor: return "forward_tc_kernel";
    case FwdKernel::kDecode: return "forward_dec_kernel";
    case FwdKernel::kGeneral: return "forward_cc_kernel";
    default: return nullptr;
  }
}

sa_status validate_cu_host(const int64_t* cu, int32_t batch) {
  if (cu == nullptr || batch < 1 || cu[0] != 0) return SA_ERR_CU_SEQLENS;
  for (int32_t b = 1; b <= batch; ++b)
    if (cu[b] < cu[b - 1]) return SA_ERR_CU_SEQLENS;
  return SA_OK;
}

sa_status check_geometry(int64_t tq, int32_t hkv, int32_t topk, int32_t batch, int32_t max_pages,
                         int32_t block_size, int32_t page_size, int64_t* msb_out,
                         int64_t* nbs_out) {
  if (block_size <= 0 || page_size <= 0 || block_size % page_size != 0) return SA_ERR_BLOCK_PAGE;
  if (tq == 0 || hkv == 0 || topk == 0) return SA_ERR_EMPTY;
  if (tq < 0 || hkv < 0 || topk < 0 || max_pages < 0) return SA_ERR_SHAPE;
  if (batch < 1) return SA_ERR_CU_SEQLENS;
  const int64_t ppb = block_size / page_size;
  const int64_t msb = max_pages / ppb;
  const int64_t n = tq * hkv * static_cast<int64_t>(topk);
  if (n >= (int64_t{1} << 31) || msb > sa::kMaxMsb || msb * block_size >= (int64_t{1} << 31))
    return SA_ERR_UNSUPPORTED;
  const int64_t nbs = batch * msb;
  if (static_cast<int64_t>(hkv) * (nbs + 1) >= (int64_t{1} << 31)) return SA_ERR_UNSUPPORTED;
  *msb_out = msb;
  *nbs_out = nbs;
  return SA_OK;
}

}  // namespace

extern "C" {

const char* sa_status_string(sa_status status) {
  switch (status) {
    case SA_OK: return "ok";
    case SA_ERR_HEAD_COUNT: return "Hq must be a positive multiple of Hkv";
    case SA_ERR_BLOCK_PAGE: return "block_size must be a positive multiple of page_size";
    case SA_ERR_CU_SEQLENS: return "cu_seqlens_q invalid (empty or not monotonic)";
    case SA_ERR_SHAPE: return "shape mismatch";
    case SA_ERR_SELECTED_RANGE: return "selected block id out of range [-1, msb)";
    case SA_ERR_HEAD_DIM: return "head dim mismatch across q/k_cache/v_cache";
    case SA_ERR_EMPTY: return "empty input";
    case SA_ERR_CUDA: return "CUDA runtime error";
    case SA_ERR_DEVICE_TIMEOUT: return "a bounded device wait ran out";
    case SA_ERR_UNSUPPORTED: return "shape not supported by the kernels";
    case SA_ERR_INVALID_ARGUMENT: return "invalid argument (null, misaligned or too small)";
  }
  return "unknown status";
}

const char* sa_version(void) { return "sa-gb300 0.1 (sm_103a)"; }

sa_status sa_index_query_sizes(int64_t tq, int32_t hkv, int32_t topk, int32_t batch,
                               int32_t max_pages, int32_t block_size, int32_t page_size,
                               sa_index_sizes* out) {
  if (out == nullptr) return SA_ERR_INVALID_ARGUMENT;
  int64_t msb = 0, nbs = 0;
  const sa_status st =
      check_geometry(tq, hkv, topk, batch, max_pages, block_size, page_size, &msb, &nbs);
  if (st != SA_OK) return st;
  const int64_t n = tq * hkv * static_cast<int64_t>(topk);
  std::memset(out, 0, sizeof(*out));
  out->msb = msb;
  out->nbs = nbs;
  out->sel_slots = nbs > 0 ? static_cast<int64_t>(hkv) * nbs : 1;
  out->sel_offsets = static_cast<int64_t>(hkv) * (nbs + 1);
  out->num_sel = hkv;
  out->edge_head_base = static_cast<int64_t>(hkv) + 1;
  out->edges = 2 * n;
  out->inv = n;
  out->splits = 4 * n;
  out->totals = 4;
  // the build's scratch, then the tensor-core forward's longest-first work list
  const sa::LptRegion lpt =
      sa::lpt_region(tq, hkv, topk, batch, static_cast<int32_t>(msb), nbs);
  out->workspace_bytes = lpt.offset + lpt.bytes;
  return SA_OK;
}

sa_status sa_index_workspace_size(int64_t tq, int32_t hkv, int32_t topk, int32_t batch,
                                  int32_t max_pages, int32_t block_size, int32_t page_size,
                                  size_t* bytes) {
  if (bytes == nullptr) return SA_ERR_INVALID_ARGUMENT;
  sa_index_sizes z;
  const sa_status st =
      sa_index_query_sizes(tq, hkv, topk, batch, max_pages, block_size, page_size, &z);
  if (st != SA_OK) return st;
  *bytes = z.workspace_bytes;
  return SA_OK;
}

namespace {

// Per host thread and device: the side stream an index build runs on beside
// the fused decode kernel (sa_attention), and the events of the fork and the
// join.  Created on first use; none (the build then runs in stream order)
// where creation fails.
struct SideStream {
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  bool tried = false, ok = false;
};

SideStream* side_stream() {
  constexpr int kMaxDevices = 64;
  thread_local SideStream per_device[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return nullptr;
  }
  SideStream& r = per_device[dev];
  if (!r.tried) {
    r.tried = true;
    r.ok = cudaStreamCreateWithFlags(&r.s, cudaStreamNonBlocking) == cudaSuccess &&
           cudaEventCreateWithFlags(&r.fork, cudaEventDisableTiming) == cudaSuccess &&
           cudaEventCreateWithFlags(&r.join, cudaEventDisableTiming) == cudaSuccess;
    if (!r.ok) cudaGetLastError();
  }
  return r.ok ? &r : nullptr;
}

// Step 1.  With `side`: the workspace counters and the status word are
// cleared on `stream`, then the build runs on the side stream, forked from
// `stream` (the caller joins it back after launching what runs beside it).
sa_status build_index_impl(const int32_t* selected, int64_t tq, int32_t hkv, int32_t topk,
                           const int64_t* cu_seqlens_q_host, const int64_t* cu_seqlens_q,
                           int32_t batch, const int32_t* used_kv_lens, int32_t max_pages,
                           int32_t block_size, int32_t page_size, int32_t split_edges,
                           sa_index* idx, void* stream, SideStream* side,
                           bool* forked = nullptr) {
  if (forked != nullptr) *forked = false;
  if (block_size <= 0 || page_size <= 0 || block_size % page_size != 0) return SA_ERR_BLOCK_PAGE;
  if (tq == 0 || hkv == 0 || topk == 0) return SA_ERR_EMPTY;
  sa_status st = validate_cu_host(cu_seqlens_q_host, batch);
  if (st != SA_OK) return st;
  if (cu_seqlens_q_host[batch] != tq) return SA_ERR_SHAPE;
  int64_t msb = 0, nbs = 0;
  st = check_geometry(tq, hkv, topk, batch, max_pages, block_size, page_size, &msb, &nbs);
  if (st != SA_OK) return st;
  if (split_edges < 0) return SA_ERR_INVALID_ARGUMENT;
  if (idx == nullptr || selected == nullptr || cu_seqlens_q == nullptr) return SA_ERR_INVALID_ARGUMENT;
  if (!idx->sel_slots || !idx->sel_offsets || !idx->num_sel || !idx->edge_head_base ||
      !idx->edges || !idx->inv || !idx->splits || !idx->totals || !idx->workspace)
    return SA_ERR_INVALID_ARGUMENT;
  if (!aligned16(idx->splits) || !aligned16(idx->edges) ||
      (reinterpret_cast<uintptr_t>(idx->workspace) & 255u) != 0)
    return SA_ERR_INVALID_ARGUMENT;
  int64_t multi_slots = 0;
  const int64_t chunks_per_head =
      sa::index_chunks_per_head(cu_seqlens_q_host, batch, topk, &multi_slots);
  const sa::WorkspaceLayout lay =
      sa::workspace_layout(hkv, batch, tq, multi_slots, static_cast<int32_t>(msb));
  if (idx->workspace_bytes < lay.total) return SA_ERR_INVALID_ARGUMENT;

  idx->tq = tq;
  idx->hkv = hkv;
  idx->topk = topk;
  idx->batch = batch;
  idx->max_pages = max_pages;
  idx->block_size = block_size;
  idx->page_size = page_size;
  idx->pages_per_block = block_size / page_size;
  idx->msb = static_cast<int32_t>(msb);
  idx->nbs = nbs;
  idx->split_edges = split_edges;
  idx->flags = 0;

  sa::IndexArgs a{};
  a.selected = selected;
  a.cu = cu_seqlens_q;
  a.used = used_kv_lens;
  a.tq = tq;
  a.hkv = hkv;
  a.topk = topk;
  a.batch = batch;
  a.msb = static_cast<int32_t>(msb);
  a.block_size = block_size;
  a.split_edges = split_edges;
  a.nbs = nbs;
  a.idx = *idx;
  // decode batches (every (kv head, sequence) segment of at most 64 entries)
  // take the kernel's warp-per-segment mode
  int64_t longest = 0;
  for (int32_t b = 0; b < batch; ++b)
    longest = std::max<int64_t>(longest, cu_seqlens_q_host[b + 1] - cu_seqlens_q_host[b]);
  a.small = longest * topk <= sa::kSmallSegment ? 1 : 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (side != nullptr) {
    if (sa::launch_clear_for_build(idx->workspace, lay.zero_bytes, idx->totals + 3, s) !=
            cudaSuccess ||
        cudaEventRecord(side->fork, s) != cudaSuccess ||
        cudaStreamWaitEvent(side->s, side->fork, 0) != cudaSuccess)
      return SA_ERR_CUDA;
    if (forked != nullptr) *forked = true;
    a.external_clear = 1;
    s = side->s;
  }
  const cudaError_t err = sa::launch_build_index(a, chunks_per_head, multi_slots, s);
  if (err == cudaErrorNotSupported) return SA_ERR_UNSUPPORTED;
  return err == cudaSuccess ? SA_OK : SA_ERR_CUDA;
}

}  // namespace

sa_status sa_build_index(const int32_t* selected, int64_t tq, int32_t hkv, int32_t topk,
                         const int64_t* cu_seqlens_q_host, const int64_t* cu_seqlens_q,
                         int32_t batch, const int32_t* used_kv_lens, int32_t max_pages,
                         int32_t block_size, int32_t page_size, int32_t split_edges,
                         sa_index* idx, void* stream) {
  return build_index_impl(selected, tq, hkv, topk, cu_seqlens_q_host, cu_seqlens_q, batch,
                          used_kv_lens, max_pages, block_size, page_size, split_edges, idx,
                          stream, nullptr);
}

namespace {

// The scratch an index's forward takes its counters from: the library's
// fixed array for an index built by sa_build_index_no_alloc, else the
// caller's workspace.  Returns false when there is none (NULL workspace).
bool index_scratch(const sa_index* idx, unsigned char** ws, size_t* bytes) {
  void* p = nullptr;
  size_t n = 0;
  if (idx->flags & SA_INDEX_STATIC_SCRATCH) {
    if (sa::static_index_scratch(&p, &n) != SA_OK) p = nullptr;
  } else {
    p = idx->workspace;
    n = idx->workspace_bytes;
  }
  *ws = static_cast<unsigned char*>(p);
  *bytes = p != nullptr ? n : 0;
  return p != nullptr;
}

// Step 2.  `q16_scratch` (nullable): room for tq * hq * head_dim bf16 values,
// 16-byte aligned, not overlapping q, that the tensor-core kernel may fill
// with Q rounded to bf16 and gather from (half the bytes of the f32 rows, no
// conversion per gather); its content afterwards is unspecified.
sa_status forward_impl(const float* q, const void* k_pages, const void* v_pages,
                       int64_t num_pages, sa_dtype kv_dtype, const sa_index* idx,
                       const int32_t* block_tables, const int64_t* cu_seqlens_q,
                       const int32_t* used_kv_lens, int32_t hq, int32_t hkv, int32_t head_dim,
                       int32_t block_size, int32_t page_size, float softmax_scale, int32_t causal,
                       sa_dtype partial_dtype, void* o_partial, float* m_partial,
                       float* l_partial, sa_path path, void* stream, void* q16_scratch) {
  if (hkv <= 0 || hq <= 0 || hq % hkv != 0) return SA_ERR_HEAD_COUNT;
  if (head_dim <= 0 || block_size <= 0 || page_size <= 0 || block_size % page_size != 0)
    return SA_ERR_BLOCK_PAGE;
  if (idx == nullptr) return SA_ERR_INVALID_ARGUMENT;
  if (idx->hkv != hkv || idx->pages_per_block != block_size / page_size ||
      idx->block_size != block_size || idx->page_size != page_size)
    return SA_ERR_SHAPE;
  if (num_pages < 0) return SA_ERR_SHAPE;
  if (kv_dtype != SA_DTYPE_F32 && kv_dtype != SA_DTYPE_BF16) return SA_ERR_INVALID_ARGUMENT;
  if (partial_dtype != SA_DTYPE_F32 && partial_dtype != SA_DTYPE_BF16)
    return SA_ERR_INVALID_ARGUMENT;
  if (causal < 0 || causal > 2) return SA_ERR_INVALID_ARGUMENT;
  const int kv_bf16 = kv_dtype == SA_DTYPE_BF16 ? 1 : 0;
  if (path == SA_PATH_FUSED_DECODE) return SA_ERR_UNSUPPORTED;   // writes no partials
  if (path != SA_PATH_AUTO && path != SA_PATH_CUDA_CORE && path != SA_PATH_CUDA_CORE_GENERAL &&
      path != SA_PATH_TENSOR_CORE && path != SA_PATH_TENSOR_CORE_TF32)
    return SA_ERR_INVALID_ARGUMENT;
  const FwdKernel kernel = choose_forward(idx->tq, idx->batch, hq / hkv, head_dim, block_size,
                                          page_size, kv_bf16, path);
  if (kernel == FwdKernel::kNone) return SA_ERR_UNSUPPORTED;
  if (!q || !k_pages || !v_pages || !block_tables || !cu_seqlens_q || !o_partial || !m_partial ||
      !l_partial)
    return SA_ERR_INVALID_ARGUMENT;
  if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(o_partial))
    return SA_ERR_INVALID_ARGUMENT;

  sa::ForwardArgs a{};
  a.q = q;
  a.k_pages = k_pages;
  a.v_pages = v_pages;
  a.num_pages = num_pages;
  a.kv_bf16 = kv_bf16;
  a.block_tables = block_tables;
  a.cu = cu_seqlens_q;
  a.used = used_kv_lens;
  a.hq = hq;
  a.hkv = hkv;
  a.qhead = hq / hkv;
  a.head_dim = head_dim;
  a.block_size = block_size;
  a.page_size = page_size;
  a.pages_per_block = block_size / page_size;
  a.max_pages = idx->max_pages;
  a.msb = idx->msb;
  a.nbs = idx->nbs;
  a.scale = softmax_scale;
  a.causal = causal;
  a.sel_slots = idx->sel_slots;
  a.sel_offsets = idx->sel_offsets;
  a.num_sel = idx->num_sel;
  a.edge_head_base = idx->edge_head_base;
  a.edges = idx->edges;
  a.splits = idx->splits;
  a.totals = idx->totals;
  a.max_splits = idx->tq * idx->hkv * static_cast<int64_t>(idx->topk);
  a.o_partial = o_partial;
  a.o_bf16 = partial_dtype == SA_DTYPE_BF16 ? 1 : 0;
  a.m_partial = m_partial;
  a.l_partial = l_partial;
  if (a.msb <= 0) return SA_OK;  // no block is addressable: every entry was dropped
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t err;
  unsigned char* ws = nullptr;
  size_t ws_bytes = 0;
  if (kernel == FwdKernel::kTensor && index_scratch(idx, &ws, &ws_bytes) && ws_bytes >= 256) {
    a.unit_counter =
        reinterpret_cast<uint32_t*>(ws + sa::workspace_layout(1, 1, 1, 0, 1).unit_ctr);
    const sa::LptRegion lpt =
        sa::lpt_region(idx->tq, idx->hkv, idx->topk, idx->batch, idx->msb, idx->nbs);
    if (ws_bytes >= lpt.offset + lpt.bytes) {
      a.unit_order = reinterpret_cast<int32_t*>(ws + lpt.offset);
      a.order_counts = reinterpret_cast<uint32_t*>(ws + lpt.offset + lpt.counts);
      a.max_units = lpt.units;
    }
  }
  if (kernel == FwdKernel::kTensor) sa::debug_cta_stats(&a.cta_stats, &a.cta_stats_len);
  // tf32 scores for f32 K/V where asked for; bf16 operands otherwise
  a.tf32 = kernel == FwdKernel::kTensor && !kv_bf16 && path == SA_PATH_TENSOR_CORE_TF32;
  if (kernel == FwdKernel::kTensor && !a.tf32 && q16_scratch != nullptr) {
    const int64_t n = idx->tq * static_cast<int64_t>(hq) * head_dim;
    err = sa::launch_q_to_bf16(q, static_cast<uint16_t*>(q16_scratch), n, s);
    if (err != cudaSuccess) return SA_ERR_CUDA;
    a.q16 = static_cast<const uint16_t*>(q16_scratch);
  }
  switch (kernel) {
    case FwdKernel::kDecodeMma: err = sa::launch_forward_dec_mma(a, s); break;
    case FwdKernel::kTensor: err = sa::launch_forward_tc(a, s); break;
    case FwdKernel::kDecode: err = sa::launch_forward_dec(a, s); break;
    default: err = sa::launch_forward_cc(a, s); break;
  }
  if (err == cudaErrorNotSupported) return SA_ERR_UNSUPPORTED;
  return err == cudaSuccess ? SA_OK : SA_ERR_CUDA;
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

}  // namespace

sa_status sa_forward_ex(const float* q, const void* k_pages, const void* v_pages,
                        int64_t num_pages, sa_dtype kv_dtype, const sa_index* idx,
                        const int32_t* block_tables, const int64_t* cu_seqlens_q,
                        const int32_t* used_kv_lens, int32_t hq, int32_t hkv, int32_t head_dim,
                        int32_t block_size, int32_t page_size, float softmax_scale,
                        int32_t causal, sa_dtype partial_dtype, void* o_partial,
                        float* m_partial, float* l_partial, sa_path path, void* stream,
                        void* q_scratch) {
  if (q_scratch != nullptr) {
    const size_t qbytes = idx ? static_cast<size_t>(idx->tq) * (hq > 0 ? hq : 0) *
                                    (head_dim > 0 ? head_dim : 0) * sizeof(float)
                              : 0;
    if (!aligned16(q_scratch) || head_dim % 8 != 0 || overlaps(q, qbytes, q_scratch, qbytes / 2))
      return SA_ERR_INVALID_ARGUMENT;
  }
  return forward_impl(q, k_pages, v_pages, num_pages, kv_dtype, idx, block_tables, cu_seqlens_q,
                      used_kv_lens, hq, hkv, head_dim, block_size, page_size, softmax_scale,
                      causal, partial_dtype, o_partial, m_partial, l_partial, path, stream,
                      q_scratch);
}

sa_status sa_forward(const float* q, const void* k_pages, const void* v_pages, int64_t num_pages,
                     sa_dtype kv_dtype, const sa_index* idx, const int32_t* block_tables,
                     const int64_t* cu_seqlens_q, const int32_t* used_kv_lens, int32_t hq,
                     int32_t hkv, int32_t head_dim, int32_t block_size, int32_t page_size,
                     float softmax_scale, int32_t causal, float* o_partial, float* m_partial,
                     float* l_partial, sa_path path, void* stream) {
  return sa_forward_ex(q, k_pages, v_pages, num_pages, kv_dtype, idx, block_tables, cu_seqlens_q,
                       used_kv_lens, hq, hkv, head_dim, block_size, page_size, softmax_scale,
                       causal, SA_DTYPE_F32, o_partial, m_partial, l_partial, path, stream,
                       nullptr);
}

const char* sa_forward_kernel_name(int64_t tq, int32_t batch, int32_t hq, int32_t hkv,
                                   int32_t head_dim, int32_t block_size, int32_t page_size,
                                   sa_dtype kv_dtype, sa_path path) {
  if (hkv <= 0 || hq <= 0 || hq % hkv != 0) return nullptr;
  if (head_dim <= 0 || block_size <= 0 || page_size <= 0 || block_size % page_size != 0)
    return nullptr;
  if (kv_dtype != SA_DTYPE_F32 && kv_dtype != SA_DTYPE_BF16) return nullptr;
  return forward_kernel_name(choose_forward(tq, batch, hq / hkv, head_dim, block_size, page_size,
                                            kv_dtype == SA_DTYPE_BF16 ? 1 : 0, path));
}

const char* sa_attention_kernel_name(int64_t tq, int32_t batch, const int64_t* cu_seqlens_q_host,
                                     int64_t num_pages, int32_t hq, int32_t hkv,
                                     int32_t head_dim, int32_t block_size, int32_t page_size,
                                     sa_dtype kv_dtype, int32_t causal, sa_path path) {
  if (kv_dtype != SA_DTYPE_F32 && kv_dtype != SA_DTYPE_BF16) return nullptr;
  if (causal < 0 || causal > 2) return nullptr;
  const int kv_bf16 = kv_dtype == SA_DTYPE_BF16 ? 1 : 0;
  if ((path == SA_PATH_AUTO || path == SA_PATH_FUSED_DECODE) && causal != 2) {
    if (hkv > 0 && hq > 0 && hq % hkv == 0 && head_dim > 0 && block_size > 0 && page_size > 0 &&
        block_size % page_size == 0 && validate_cu_host(cu_seqlens_q_host, batch) == SA_OK &&
        cu_seqlens_q_host[batch] == tq &&
        fused_eligible(tq, batch, cu_seqlens_q_host, num_pages, hq, hkv, head_dim, block_size,
                       page_size, kv_bf16))
      return "fused_dec_kernel";
  }
  if (path == SA_PATH_FUSED_DECODE) return nullptr;
  return sa_forward_kernel_name(tq, batch, hq, hkv, head_dim, block_size, page_size, kv_dtype,
                                path);
}

sa_status sa_combine_ex(const sa_index* idx, sa_dtype partial_dtype, const void* o_partial,
                        const float* m_partial, const float* l_partial, int32_t hq,
                        int32_t head_dim, float* out, float* lse, void* stream) {
  if (idx == nullptr) return SA_ERR_INVALID_ARGUMENT;
  if (partial_dtype != SA_DTYPE_F32 && partial_dtype != SA_DTYPE_BF16)
    return SA_ERR_INVALID_ARGUMENT;
  if (idx->hkv <= 0 || hq <= 0 || hq % idx->hkv != 0) return SA_ERR_HEAD_COUNT;
  if (head_dim <= 0) return SA_ERR_BLOCK_PAGE;
  if (head_dim % 4 != 0 || head_dim > 256) return SA_ERR_UNSUPPORTED;
  if (!o_partial || !m_partial || !l_partial || !out) return SA_ERR_INVALID_ARGUMENT;
  if (!aligned16(o_partial) || !aligned16(out)) return SA_ERR_INVALID_ARGUMENT;
  sa::CombineArgs a{};
  a.inv = idx->inv;
  a.edge_head_base = idx->edge_head_base;
  a.o_partial = o_partial;
  a.o_bf16 = partial_dtype == SA_DTYPE_BF16 ? 1 : 0;
  a.m_partial = m_partial;
  a.l_partial = l_partial;
  a.tq = idx->tq;
  a.hkv = idx->hkv;
  a.topk = idx->topk;
  a.qhead = hq / idx->hkv;
  a.head_dim = head_dim;
  a.out = out;
  a.lse = lse;
  const cudaError_t err = sa::launch_combine(a, static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? SA_OK : SA_ERR_CUDA;
}

sa_status sa_combine(const sa_index* idx, const float* o_partial, const float* m_partial,
                     const float* l_partial, int32_t hq, int32_t head_dim, float* out, float* lse,
                     void* stream) {
  return sa_combine_ex(idx, SA_DTYPE_F32, o_partial, m_partial, l_partial, hq, head_dim, out, lse,
                       stream);
}

namespace {

// Steps 2 and 3.  `behind_build`: the index build that made `idx` was the
// last launch on `stream` (sa_attention), so the fused decode kernel may be
// launched as its programmatic dependent.
sa_status forward_combine_impl(const float* q, const void* k_pages, const void* v_pages,
                               int64_t num_pages, sa_dtype kv_dtype, const sa_index* idx,
                               const int32_t* selected, const int64_t* cu_seqlens_q_host,
                               const int64_t* cu_seqlens_q, const int32_t* used_kv_lens,
                               const int32_t* block_tables, int32_t hq, int32_t head_dim,
                               int32_t block_size, int32_t page_size, float softmax_scale,
                               int32_t causal, int32_t split_edges, sa_dtype partial_dtype,
                               void* o_partial, float* m_partial, float* l_partial, float* out,
                               float* lse, sa_path path, void* stream, bool behind_build) {
  if (idx == nullptr) return SA_ERR_INVALID_ARGUMENT;
  if (partial_dtype != SA_DTYPE_F32 && partial_dtype != SA_DTYPE_BF16)
    return SA_ERR_INVALID_ARGUMENT;
  const int32_t hkv = idx->hkv;
  if (hkv <= 0 || hq <= 0 || hq % hkv != 0) return SA_ERR_HEAD_COUNT;
  if (head_dim <= 0 || block_size <= 0 || page_size <= 0 || block_size % page_size != 0)
    return SA_ERR_BLOCK_PAGE;
  if (idx->block_size != block_size || idx->page_size != page_size) return SA_ERR_SHAPE;
  if (kv_dtype != SA_DTYPE_F32 && kv_dtype != SA_DTYPE_BF16) return SA_ERR_INVALID_ARGUMENT;
  if (split_edges < 0) return SA_ERR_INVALID_ARGUMENT;
  if (causal < 0 || causal > 2) return SA_ERR_INVALID_ARGUMENT;
  const int kv_bf16 = kv_dtype == SA_DTYPE_BF16 ? 1 : 0;
  const int64_t tq = idx->tq;
  const int32_t batch = idx->batch;
  bool fused = false;
  if (path == SA_PATH_AUTO || path == SA_PATH_FUSED_DECODE) {
    // (left-aligned causal masks a lone query's keys: not the fused path's case)
    if (causal != 2 && validate_cu_host(cu_seqlens_q_host, batch) == SA_OK &&
        cu_seqlens_q_host[batch] == tq)
      fused = fused_eligible(tq, batch, cu_seqlens_q_host, num_pages, hq, hkv, head_dim,
                             block_size, page_size, kv_bf16);
    if (path == SA_PATH_FUSED_DECODE && !fused) return SA_ERR_UNSUPPORTED;
  }
  if (!fused) {
    // `out` is not written before the combine: the tensor-core forward may
    // keep a bf16 copy of Q there (in its first half), unless out and q
    // share memory.
    const size_t qbytes = static_cast<size_t>(tq) * hq * head_dim * sizeof(float);
    void* q16 = (out != nullptr && q != nullptr && qbytes > 0 && head_dim % 8 == 0 &&
                 aligned16(out) && !overlaps(q, qbytes, out, qbytes))
                    ? static_cast<void*>(out)
                    : nullptr;
    const sa_status st = forward_impl(q, k_pages, v_pages, num_pages, kv_dtype, idx,
                                      block_tables, cu_seqlens_q, used_kv_lens, hq, hkv, head_dim,
                                      block_size, page_size, softmax_scale, causal,
                                      partial_dtype, o_partial, m_partial, l_partial, path,
                                      stream, q16);
    if (st != SA_OK) return st;
    return sa_combine_ex(idx, partial_dtype, o_partial, m_partial, l_partial, hq, head_dim, out,
                         lse, stream);
  }
  if (!q || !k_pages || !v_pages || !block_tables || !cu_seqlens_q || !selected || !o_partial ||
      !m_partial || !l_partial || !out || !idx->inv || !idx->totals)
    return SA_ERR_INVALID_ARGUMENT;
  // The per-(query, kv head) piece counters live in the index's scratch,
  // cleared by the build that made the index.
  unsigned char* ws = nullptr;
  size_t ws_bytes = 0;
  const sa::WorkspaceLayout lay = sa::workspace_layout(hkv, batch, tq, 0, 1);
  if (!index_scratch(idx, &ws, &ws_bytes) || ws_bytes < lay.seg_tot)
    return SA_ERR_INVALID_ARGUMENT;
  if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(o_partial) ||
      !aligned16(out))
    return SA_ERR_INVALID_ARGUMENT;
  if (idx->msb <= 0) return SA_ERR_SHAPE;   // a built index over these sizes addresses blocks
  sa::FusedDecArgs a{};
  a.q = q;
  a.k_pages = k_pages;
  a.v_pages = v_pages;
  a.num_pages = num_pages;
  a.kv_bf16 = kv_bf16;
  a.block_tables = block_tables;
  a.cu = cu_seqlens_q;
  a.used = used_kv_lens;
  a.selected = selected;
  a.inv = idx->inv;
  a.tq = tq;
  a.batch = batch;
  a.hq = hq;
  a.hkv = hkv;
  a.qhead = hq / hkv;
  a.topk = idx->topk;
  a.block_size = block_size;
  a.page_size = page_size;
  a.pages_per_block = block_size / page_size;
  a.max_pages = idx->max_pages;
  a.msb = idx->msb;
  // Pieces.  split_edges > 0: every pair in pieces of split_edges ranks (at
  // most 64).  Otherwise whole pairs (all ranks, when topk <= 64) round-robin
  // over the SMs, and only the pairs of the last, partial round are cut, into
  // as many pieces as keep the otherwise idle SMs busy.
  const int64_t items = tq * hkv;
  int ep = split_edges;
  a.whole_items = 0;
  if (ep <= 0) {
    if (a.topk <= 64) {
      const int64_t sms = sa::device_sm_count();
      const int64_t tail = items % sms;
      int64_t pt = tail > 0 ? sms / tail : 1;
      if (pt > a.topk) pt = a.topk;
      if (pt < 1) pt = 1;
      a.whole_items = pt == 1 ? items : items - tail;
      ep = static_cast<int>((a.topk + pt - 1) / pt);
    } else {
      ep = 64;
    }
  }
  if (ep > 64) ep = 64;
  a.ranks_per_piece = ep;
  a.pieces = (a.topk + ep - 1) / ep;
  a.scale = softmax_scale;
  a.status = idx->totals + 3;
  a.item_cnt = reinterpret_cast<uint32_t*>(ws + lay.item_cnt);
  a.part_o = o_partial;
  a.part_bf16 = partial_dtype == SA_DTYPE_BF16 ? 1 : 0;
  a.part_m = m_partial;
  a.part_l = l_partial;
  a.out = out;
  a.lse = lse;
  a.pdl = behind_build ? 1 : 0;
  (void)causal;   // a no-op for one query per sequence (its position is lk - 1)
  const cudaError_t err = sa::launch_fused_dec(a, static_cast<cudaStream_t>(stream));
  if (err == cudaErrorNotSupported) return SA_ERR_UNSUPPORTED;
  return err == cudaSuccess ? SA_OK : SA_ERR_CUDA;
}

}  // namespace

sa_status sa_forward_combine_ex(const float* q, const void* k_pages, const void* v_pages,
                                int64_t num_pages, sa_dtype kv_dtype, const sa_index* idx,
                                const int32_t* selected, const int64_t* cu_seqlens_q_host,
                                const int64_t* cu_seqlens_q, const int32_t* used_kv_lens,
                                const int32_t* block_tables, int32_t hq, int32_t head_dim,
                                int32_t block_size, int32_t page_size, float softmax_scale,
                                int32_t causal, int32_t split_edges, sa_dtype partial_dtype,
                                void* o_partial, float* m_partial, float* l_partial, float* out,
                                float* lse, sa_path path, void* stream) {
  return forward_combine_impl(q, k_pages, v_pages, num_pages, kv_dtype, idx, selected,
                              cu_seqlens_q_host, cu_seqlens_q, used_kv_lens, block_tables, hq,
                              head_dim, block_size, page_size, softmax_scale, causal, split_edges,
                              partial_dtype, o_partial, m_partial, l_partial, out, lse, path,
                              stream, false);
}

sa_status sa_forward_combine(const float* q, const void* k_pages, const void* v_pages,
                             int64_t num_pages, sa_dtype kv_dtype, const sa_index* idx,
                             const int32_t* selected, const int64_t* cu_seqlens_q_host,
                             const int64_t* cu_seqlens_q, const int32_t* used_kv_lens,
                             const int32_t* block_tables, int32_t hq, int32_t head_dim,
                             int32_t block_size, int32_t page_size, float softmax_scale,
                             int32_t causal, int32_t split_edges, float* o_partial,
                             float* m_partial, float* l_partial, float* out, float* lse,
                             sa_path path, void* stream) {
  return sa_forward_combine_ex(q, k_pages, v_pages, num_pages, kv_dtype, idx, selected,
                               cu_seqlens_q_host, cu_seqlens_q, used_kv_lens, block_tables, hq,
                               head_dim, block_size, page_size, softmax_scale, causal,
                               split_edges, SA_DTYPE_F32, o_partial, m_partial, l_partial, out,
                               lse, path, stream);
}

sa_status sa_attention_ex(const float* q, const void* k_pages, const void* v_pages,
                          int64_t num_pages, sa_dtype kv_dtype, const int32_t* selected, int64_t tq,
                          int32_t topk, const int64_t* cu_seqlens_q_host,
                          const int64_t* cu_seqlens_q, int32_t batch, const int32_t* used_kv_lens,
                          const int32_t* block_tables, int32_t max_pages, int32_t hq, int32_t hkv,
                          int32_t head_dim, int32_t block_size, int32_t page_size,
                          float softmax_scale, int32_t causal, int32_t split_edges, sa_index* idx,
                          sa_dtype partial_dtype, void* o_partial, float* m_partial,
                          float* l_partial, float* out, float* lse, sa_path path, void* stream) {
  if (hkv <= 0 || hq <= 0 || hq % hkv != 0) return SA_ERR_HEAD_COUNT;
  if (head_dim <= 0 || block_size <= 0 || page_size <= 0 || block_size % page_size != 0)
    return SA_ERR_BLOCK_PAGE;
  if (kv_dtype != SA_DTYPE_F32 && kv_dtype != SA_DTYPE_BF16) return SA_ERR_INVALID_ARGUMENT;
  if (partial_dtype != SA_DTYPE_F32 && partial_dtype != SA_DTYPE_BF16)
    return SA_ERR_INVALID_ARGUMENT;
  if (causal < 0 || causal > 2) return SA_ERR_INVALID_ARGUMENT;
  const int kv_bf16 = kv_dtype == SA_DTYPE_BF16 ? 1 : 0;
  // Shape checks of the forward step, before any device work.
  bool fused = false;
  if (path == SA_PATH_AUTO || path == SA_PATH_FUSED_DECODE) {
    if (causal != 2 && tq > 0 && validate_cu_host(cu_seqlens_q_host, batch) == SA_OK)
      fused = fused_eligible(tq, batch, cu_seqlens_q_host, num_pages, hq, hkv, head_dim,
                             block_size, page_size, kv_bf16);
    if (path == SA_PATH_FUSED_DECODE && !fused) return SA_ERR_UNSUPPORTED;
  }
  if (!fused && !sa::forward_cc_supported(head_dim, block_size, kv_bf16) &&
      !((path == SA_PATH_TENSOR_CORE || path == SA_PATH_TENSOR_CORE_TF32) &&
        sa::forward_tc_supported(head_dim, block_size, page_size, hq / hkv)))
    return SA_ERR_UNSUPPORTED;
  // The fused decode kernel reads no output of the index build: the build
  // runs beside it on a side stream (both after the workspace counters and
  // the status word are cleared in stream order), joined back before the
  // call returns, so later work on `stream` sees both complete.  Without a
  // side stream the fused kernel is the build's programmatic dependent.
  SideStream* side = fused ? side_stream() : nullptr;
  bool forked = false;
  const sa_status st = build_index_impl(selected, tq, hkv, topk, cu_seqlens_q_host,
                                        cu_seqlens_q, batch, used_kv_lens, max_pages, block_size,
                                        page_size, split_edges, idx, stream, side, &forked);
  sa_status st2 = st;
  if (st == SA_OK)
    st2 = forward_combine_impl(q, k_pages, v_pages, num_pages, kv_dtype, idx, selected,
                               cu_seqlens_q_host, cu_seqlens_q, used_kv_lens, block_tables, hq,
                               head_dim, block_size, page_size, softmax_scale, causal,
                               split_edges, partial_dtype, o_partial, m_partial, l_partial, out,
                               lse, path, stream, side == nullptr);
  if (forked && (cudaEventRecord(side->join, side->s) != cudaSuccess ||
                          cudaStreamWaitEvent(static_cast<cudaStream_t>(stream), side->join, 0) !=
                              cudaSuccess))
    return SA_ERR_CUDA;
  return st2;
}

sa_status sa_attention(const float* q, const void* k_pages, const void* v_pages,
                       int64_t num_pages, sa_dtype kv_dtype, const int32_t* selected, int64_t tq,
                       int32_t topk, const int64_t* cu_seqlens_q_host,
                       const int64_t* cu_seqlens_q, int32_t batch, const int32_t* used_kv_lens,
                       const int32_t* block_tables, int32_t max_pages, int32_t hq, int32_t hkv,
                       int32_t head_dim, int32_t block_size, int32_t page_size,
                       float softmax_scale, int32_t causal, int32_t split_edges, sa_index* idx,
                       float* o_partial, float* m_partial, float* l_partial, float* out,
                       float* lse, sa_path path, void* stream) {
  return sa_attention_ex(q, k_pages, v_pages, num_pages, kv_dtype, selected, tq, topk,
                         cu_seqlens_q_host, cu_seqlens_q, batch, used_kv_lens, block_tables,
                         max_pages, hq, hkv, head_dim, block_size, page_size, softmax_scale,
                         causal, split_edges, idx, SA_DTYPE_F32, o_partial, m_partial, l_partial,
                         out, lse, path, stream);
}

sa_status sa_debug_stall(int32_t site, uint32_t spin_limit) {
  if (site < sa::kStallNone || site > sa::kStallFusedCopies) return SA_ERR_INVALID_ARGUMENT;
  sa::g_stall_site.store(site, std::memory_order_relaxed);
  sa::g_spin_limit.store(spin_limit, std::memory_order_relaxed);
  return SA_OK;
}

sa_status sa_debug_cta_stats(int64_t* stats, int32_t n_ctas) {
  if (n_ctas < 0 || (n_ctas > 0 && stats == nullptr)) return SA_ERR_INVALID_ARGUMENT;
  sa::g_cta_stats.store(n_ctas > 0 ? stats : nullptr, std::memory_order_relaxed);
  sa::g_cta_stats_len.store(n_ctas, std::memory_order_relaxed);
  return SA_OK;
}

sa_status sa_get_status(const sa_index* idx, void* stream) {
  if (idx == nullptr || idx->totals == nullptr) return SA_ERR_INVALID_ARGUMENT;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return SA_ERR_CUDA;
  int64_t code = 0;
  if (cudaMemcpy(&code, idx->totals + 3, sizeof(code), cudaMemcpyDeviceToHost) != cudaSuccess)
    return SA_ERR_CUDA;
  return static_cast<sa_status>(code);
}

sa_status sa_clear_status(const sa_index* idx, void* stream) {
  if (idx == nullptr || idx->totals == nullptr) return SA_ERR_INVALID_ARGUMENT;
  return cudaMemsetAsync(idx->totals + 3, 0, sizeof(int64_t), static_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? SA_OK
             : SA_ERR_CUDA;
}

}  // extern "C"
