/*
 * sa.h - C ABI of the KV-outer block-sparse attention library (libsa.so).
 *
 * The method (crate alice-llm 2.0.0, module sparse_attention) has three steps:
 *   1. sa_build_index: invert the per-query top-K block selection into a CSR
 *      index keyed by (kv head, sparse block)       - types.rs, KvOuterIndex
 *   2. sa_forward:     for each (kv head, block) work unit, load the block's
 *      pages once and emit unnormalised softmax partials (o, m, l) for every
 *      (query, rank) edge and GQA lane pointing at it  - forward.rs,
 *      kvouter_forward / process_work_unit
 *   3. sa_combine:     merge each (query, q-head)'s partials with the
 *      log-sum-exp rule                              - forward.rs, module doc
 * sa_attention runs the three in order on the caller's stream with no host
 * sync (on the fused decode path the build runs beside the fused kernel on a
 * side stream, joined back before the call returns); sa_forward_combine runs
 * steps 2 and 3 on a built index.
 *
 * Conventions for every entry point:
 *   - Array arguments are DEVICE pointers unless the name ends in _host.  The
 *     caller owns and allocates every buffer; the library allocates no device
 *     memory (it creates one side stream and two events per host thread and
 *     device, on the first sa_attention call that takes the fused decode
 *     path, and keeps them for the life of the process).
 *   - Layouts are row-major and contiguous; shapes are given in brackets.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Calls only enqueue work; they return after host-side checks.
 *   - Host-side checks (shapes, geometry, alignment) return an error status
 *     and enqueue nothing.  Errors that depend on device data (a selected id
 *     outside [-1, msb), a page id >= num_pages) are written to the device
 *     status word of the index (sa_index.totals[3]); outputs are then
 *     unspecified but every access stays in bounds.  sa_get_status reads it.
 *   - No kernel traps or waits without a bound: a wait that runs out sets
 *     SA_ERR_DEVICE_TIMEOUT in the status word and the kernel returns.
 */
#ifndef SA_H_
#define SA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Error kinds.  1..7 follow SparseAttentionError (types.rs) in order;
 * GpuInitFailed / GpuRuntimeError become SA_ERR_CUDA. */
typedef enum sa_status {
  SA_OK = 0,
  SA_ERR_HEAD_COUNT = 1,       /* hq, hkv >= 1 and hq % hkv == 0 required           */
  SA_ERR_BLOCK_PAGE = 2,       /* head_dim, block_size, page_size > 0 and
                                  block_size % page_size == 0 required             */
  SA_ERR_CU_SEQLENS = 3,       /* cu_seqlens_q: >= 2 entries, [0] == 0, non-decreasing */
  SA_ERR_SHAPE = 4,            /* a size disagrees (cu_seqlens_q[B] != tq, index vs
                                  call geometry), or a page id >= num_pages (device) */
  SA_ERR_SELECTED_RANGE = 5,   /* a selected id outside [-1, msb) (device)          */
  SA_ERR_HEAD_DIM = 6,         /* reserved: q / cache head dims disagree            */
  SA_ERR_EMPTY = 7,            /* tq == 0, hkv == 0 or topk == 0                    */
  SA_ERR_CUDA = 8,             /* a CUDA runtime call failed                        */
  SA_ERR_DEVICE_TIMEOUT = 9,   /* a bounded device wait ran out                     */
  SA_ERR_UNSUPPORTED = 10,     /* valid for the method, outside what the kernels
                                  implement (see sa_forward)                       */
  SA_ERR_INVALID_ARGUMENT = 11 /* NULL or misaligned pointer, too-small workspace   */
} sa_status;

typedef enum sa_dtype {
  SA_DTYPE_F32 = 0,
  SA_DTYPE_BF16 = 1
} sa_dtype;

/* Forward kernel choice (sa_forward / sa_attention `path`). */
typedef enum sa_path {
  SA_PATH_AUTO = 0,              /* pick per problem shape                          */
  SA_PATH_CUDA_CORE = 1,         /* f32 FMA kernels: the pipelined decode kernel
                                    where its shape limits allow, else the general one */
  SA_PATH_TENSOR_CORE = 2,       /* tensor cores, head_dim 128: decode-shaped
                                    problems with bf16 K/V use warp-level MMA (Q and
                                    P split into two bf16 parts); others use the
                                    tcgen05 kernel (block 64 or 128, qhead dividing
                                    128, bf16 operands); f32 accumulation;
                                    SA_ERR_UNSUPPORTED elsewhere                   */
  SA_PATH_CUDA_CORE_GENERAL = 3, /* the general f32 FMA kernel only                 */
  SA_PATH_FUSED_DECODE = 4,      /* sa_attention / sa_forward_combine only: forward
                                    and combine as one kernel when every sequence
                                    holds at most one query (see sa_attention);
                                    SA_ERR_UNSUPPORTED elsewhere and from
                                    sa_forward                                   */
  SA_PATH_TENSOR_CORE_TF32 = 5   /* as SA_PATH_TENSOR_CORE, but with f32 K/V the
                                    tcgen05 kernel forms the scores S = Q K^T from
                                    Q and K kept in f32 (tf32 operands) and only
                                    P and V are rounded to bf16: about half the
                                    error of bf16 operands, at the cost of twice
                                    the shared-memory bytes of Q and K          */
} sa_path;

/*
 * The KV-outer index (KvOuterIndex, types.rs) plus the work list of the
 * forward (WorkSplit, scheduler).  Geometry fields are written by
 * sa_build_index; the caller fills the array pointers (sizes from
 * sa_index_query_sizes) before the call and must keep them alive and
 * unmodified until the forward and combine that use the index have run.
 *
 *   msb  = floor(max_pages / pages_per_block) blocks per block-table row
 *   nbs  = batch * msb raw slots per kv head; raw slot = b * msb + block
 *   E    = number of kept (query, rank) edges          (totals[0])
 */
typedef struct sa_index {
  /* geometry (written by sa_build_index) */
  int64_t tq;
  int32_t hkv;
  int32_t topk;
  int32_t batch;
  int32_t max_pages;
  int32_t block_size;
  int32_t page_size;
  int32_t pages_per_block;
  int32_t msb;
  int64_t nbs;
  int32_t split_edges;       /* largest number of edges in one work split (0 = no cut) */
  int32_t flags;             /* SA_INDEX_* bits, written by the build entry points  */

  /* device arrays, caller-allocated */
  int32_t *sel_slots;        /* [hkv, nbs]   compact slot j -> raw slot; -1 for j >= num_sel[h] */
  int32_t *sel_offsets;      /* [hkv, nbs+1] head-local CSR offsets; equal to the head's
                                edge total for j >= num_sel[h] (plateau)                       */
  int32_t *num_sel;          /* [hkv]        non-empty compact slots per head                  */
  int64_t *edge_head_base;   /* [hkv+1]      head h owns edges [base[h], base[h+1])            */
  int32_t *edges;            /* [tq*hkv*topk, 2] (query, rank) pairs in CSR order; first E valid */
  int32_t *inv;              /* [hkv, tq, topk] head-local edge position, -1 = dropped          */
  int32_t *splits;           /* [tq*hkv*topk, 4] work list (head, compact slot, abs edge start,
                                abs edge end) in CSR order; first totals[1] valid               */
  int64_t *totals;           /* [4] E, number of splits, number of non-empty (head, slot) units,
                                device status (an sa_status, 0 = none)                         */
  void *workspace;           /* scratch, sa_index_sizes.workspace_bytes, 256-byte aligned       */
  size_t workspace_bytes;
} sa_index;

/* sa_index.flags bit: the index was built by sa_build_index_no_alloc, so its
 * scratch (the counters that the forward entry points read after the build)
 * lives in the library's fixed array on that device, not in idx->workspace. */
#define SA_INDEX_STATIC_SCRATCH 1

/* Element counts of each sa_index array and the workspace size in bytes. */
typedef struct sa_index_sizes {
  int64_t msb;
  int64_t nbs;
  int64_t sel_slots;         /* int32 elements */
  int64_t sel_offsets;       /* int32 elements */
  int64_t num_sel;           /* int32 elements */
  int64_t edge_head_base;    /* int64 elements */
  int64_t edges;             /* int32 elements (2 per edge)  */
  int64_t inv;               /* int32 elements */
  int64_t splits;            /* int32 elements (4 per split) */
  int64_t totals;            /* int64 elements */
  size_t workspace_bytes;
} sa_index_sizes;

/* Human-readable text of a status (the Display strings of
 * SparseAttentionError, types.rs, where one exists).  Never NULL. */
const char *sa_status_string(sa_status status);

/* Library version string. */
const char *sa_version(void);

/*
 * Sizes for an index over selected[tq, hkv, topk] with `batch` sequences and
 * block tables of `max_pages` columns.  Fails with SA_ERR_BLOCK_PAGE,
 * SA_ERR_EMPTY, SA_ERR_UNSUPPORTED (msb above 16384, or tq*hkv*topk >= 2^31)
 * or SA_ERR_INVALID_ARGUMENT (out == NULL).
 */
sa_status sa_index_query_sizes(int64_t tq, int32_t hkv, int32_t topk, int32_t batch,
                               int32_t max_pages, int32_t block_size, int32_t page_size,
                               sa_index_sizes *out);

/*
 * The workspace size alone (sa_index_query_sizes(...)->workspace_bytes):
 * bytes of device memory the caller hands sa_build_index in
 * sa_index.workspace for an index of these sizes.  Same errors as
 * sa_index_query_sizes; SA_ERR_INVALID_ARGUMENT when bytes == NULL.
 */
sa_status sa_index_workspace_size(int64_t tq, int32_t hkv, int32_t topk, int32_t batch,
                                  int32_t max_pages, int32_t block_size, int32_t page_size,
                                  size_t *bytes);

/*
 * Step 1: build the KV-outer CSR index (build_kvouter_index; fields of
 * KvOuterIndex in types.rs).
 *
 *   selected          [tq, hkv, topk] int32, -1 = padding (SparseSelection)
 *   cu_seqlens_q_host [batch+1] int64 on the HOST (validated here, no sync)
 *   cu_seqlens_q      [batch+1] int64 on the device, same values
 *   used_kv_lens      [batch] int32 or NULL (NULL: every sequence spans
 *                     msb * block_size keys)
 *   max_pages         columns of the block tables; msb = max_pages / (block_size / page_size)
 *   split_edges       cut each (head, slot) unit's edge range into work splits of
 *                     at most this many edges (0 = one split per unit)
 *
 * An entry (query i, head h, rank r) with block s is kept iff s >= 0 and
 * s * block_size < max(used_kv_lens[b], 0), b the sequence of i.  Compact
 * slots are in ascending raw-slot order and each slot's edges in ascending
 * (query, rank) order.  Checks, in order: BLOCK_PAGE, EMPTY, CU_SEQLENS,
 * SHAPE (cu_seqlens_q_host[batch] != tq), UNSUPPORTED, INVALID_ARGUMENT;
 * on device: SELECTED_RANGE.  Enqueues a memset and two kernels on `stream`.
 */
sa_status sa_build_index(const int32_t *selected, int64_t tq, int32_t hkv, int32_t topk,
                         const int64_t *cu_seqlens_q_host, const int64_t *cu_seqlens_q,
                         int32_t batch, const int32_t *used_kv_lens, int32_t max_pages,
                         int32_t block_size, int32_t page_size, int32_t split_edges,
                         sa_index *idx, void *stream);

/*
 * sa_build_index without a workspace: the pages have no counterpart; this is
 * a library convenience.  Same arguments, checks and results as
 * sa_build_index, except that the build's scratch comes from a 288 KiB array
 * compiled into the library (one copy per GPU that loads it, held until the
 * process exits) instead of idx->workspace, which may be NULL and is left
 * unchanged.  The call sets SA_INDEX_STATIC_SCRATCH in idx->flags;
 * sa_build_index clears it.
 *
 * For callers that cannot allocate device memory when they call: servers
 * whose device memory is reserved up front, code running under a memory cap,
 * or host runtimes without a device allocator.  The call itself allocates
 * nothing (no cudaMalloc, cudaFree or allocating library routine).
 *
 *   - Capacity.  With S = hkv * batch segments, M = the 4096-entry chunks of
 *     the sequences holding more than 4096 (query, rank) entries per kv head
 *     (sum over those sequences of ceil(qo_len * topk / 4096)), and up(x) =
 *     x rounded up to a multiple of 256, the scratch is
 *         a = up(256 + 4 S)            segment tickets
 *         b = up(a + 4 hkv tq)         counters per (query, kv head)
 *         c = up(b + 12 S)             segment totals
 *         d = up(c + 24 (S + 1))       segment prefixes
 *         total = up(d + 4 hkv M msb)  histograms of multi-chunk segments
 *     bytes; a problem with total > 294912 (288 KiB) returns
 *     SA_ERR_UNSUPPORTED before any device work.  With one query per
 *     sequence and topk <= 4096 (M = 0) that is about 40 bytes per segment
 *     plus 4 bytes per (query, kv head): up to 6,687 sequences at hkv = 1
 *     or 835 at hkv = 8.  The decode shapes (64 or 128 sequences of
 *     one query, hkv 8) fit; prefill-sized problems (thousands of queries
 *     per sequence) do not and need sa_build_index.
 *   - The forward entry points take the index's counters (the fused decode
 *     kernel's piece counters, which this build clears, and the tensor-core
 *     kernel's work counter) from the same array: run them on the index
 *     before the next sa_build_index_no_alloc call on that device, which
 *     reuses the array.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture on the device.
 *   - Every call shares the one array per device, and each call clears the
 *     part that must start at zero on its stream.  Calls whose work overlaps
 *     on the GPU (other streams, other threads) race on it: serialise them.
 */
sa_status sa_build_index_no_alloc(const int32_t *selected, int64_t tq, int32_t hkv,
                                  int32_t topk, const int64_t *cu_seqlens_q_host,
                                  const int64_t *cu_seqlens_q, int32_t batch,
                                  const int32_t *used_kv_lens, int32_t max_pages,
                                  int32_t block_size, int32_t page_size, int32_t split_edges,
                                  sa_index *idx, void *stream);

/*
 * Step 2: per-edge partials (kvouter_forward, forward.rs).
 *
 *   q             [tq, hq, head_dim] float32, 16-byte aligned
 *   k_pages,
 *   v_pages       [num_pages, hkv, page_size, head_dim] of kv_dtype, 16-byte aligned
 *   idx           an index built by sa_build_index on the same stream
 *   block_tables  [batch, max_pages] int32 physical page per logical page;
 *                 -1 = no page (its keys are skipped); only pages overlapping a
 *                 kept block's live range are read
 *   cu_seqlens_q, used_kv_lens  as for sa_build_index (device)
 *   softmax_scale scores are softmax_scale * <q, k>
 *   causal        1: key at absolute position p is live for query i of
 *                 sequence b iff p <= lk_b - qo_b + (i - cu[b]) when
 *                 lk_b >= qo_b, else p <= i - cu[b] (right-aligned, the rule
 *                 of forward.rs); 2: iff p <= i - cu[b] (left-aligned, the
 *                 forward.rs doc's reading for unknown KV lengths, an
 *                 opt-in); 0: no mask; other values SA_ERR_INVALID_ARGUMENT
 *   o_partial     [tq*hkv*topk*qhead, head_dim] float32; rows e*qhead + qh
 *   m_partial,
 *   l_partial     [tq*hkv*topk*qhead] float32
 *
 * Row e*qhead+qh of the partials (e an edge in CSR order, qh the GQA lane,
 * q-head h*qhead+qh) holds m = max_p s_p, l = sum_p exp(s_p - m),
 * o = sum_p exp(s_p - m) v_p over the live keys of its block; a row with no
 * live key holds (o = 0, m = -inf, l = 0).  Only the first E*qhead rows are
 * written.  Supported: head_dim a multiple of 4 (f32) or 8 (bf16), at most
 * 256, and block_size * head_dim * elt * 2 <= 160 KiB; otherwise
 * SA_ERR_UNSUPPORTED.  SA_PATH_AUTO sends decode-shaped problems (tq at most
 * twice the batch) to the pipelined CUDA-core kernel (f32 K/V) or to the
 * warp-level MMA kernel (bf16 K/V), and the others to the tcgen05 kernel
 * where supported (operands rounded to bf16; use SA_PATH_TENSOR_CORE_TF32 for
 * tf32 scores with f32 K/V, SA_PATH_CUDA_CORE for f32 arithmetic
 * throughout).  The tcgen05 kernel claims work units from a
 * counter in the first 256 bytes of the index's scratch (cleared on the
 * stream before each launch): idx->workspace when it is set and
 * idx->workspace_bytes is at least 256, the library's array for an index
 * with SA_INDEX_STATIC_SCRATCH; with neither it takes units round-robin.
 * When that scratch also has room for the work list that follows the build's
 * own use of it (sa_index_query_sizes counts it in workspace_bytes), a
 * one-CTA kernel first sorts the units by descending edge count and the
 * counter walks that longest-first list.  So one index serves one forward
 * at a time.  Checks: HEAD_COUNT, BLOCK_PAGE, SHAPE (idx geometry),
 * UNSUPPORTED, INVALID_ARGUMENT; on device: SHAPE (page id >= num_pages).
 */
sa_status sa_forward(const float *q, const void *k_pages, const void *v_pages,
                     int64_t num_pages, sa_dtype kv_dtype, const sa_index *idx,
                     const int32_t *block_tables, const int64_t *cu_seqlens_q,
                     const int32_t *used_kv_lens, int32_t hq, int32_t hkv, int32_t head_dim,
                     int32_t block_size, int32_t page_size, float softmax_scale, int32_t causal,
                     float *o_partial, float *m_partial, float *l_partial, sa_path path,
                     void *stream);

/*
 * sa_forward with the o partials stored as `partial_dtype`: SA_DTYPE_F32
 * (exactly sa_forward) or SA_DTYPE_BF16, where each o value is rounded to
 * nearest even bfloat16 as it is written and o_partial holds
 * [tq*hkv*topk*qhead, head_dim] uint16 bit patterns (16-byte aligned).  m and
 * l stay float32.  The pages keep all partials in f32 (forward.rs, the
 * o_partial / m_partial / l_partial buffers); the 16-bit form has no
 * counterpart there: it is an opt-in that halves the bytes the forward
 * writes and the combine reads, at a relative error of at most 2^-8 per o
 * value before the combine.  Every forward kernel supports it.  Other
 * partial_dtype values: SA_ERR_INVALID_ARGUMENT.
 *
 * q_scratch (nullable): device memory of tq * hq * head_dim * 2 bytes,
 * 16-byte aligned, not overlapping q (head_dim a multiple of 8), which the
 * tensor-core kernel may fill with Q rounded to bf16 (one extra pass over Q)
 * and gather its tiles from; the result is identical (that kernel rounds Q
 * to bf16 either way) and the scratch content afterwards unspecified.
 * sa_forward_combine and sa_attention pass the first half of `out` (written
 * only by the combine) unless out and q overlap.  Bad scratch:
 * SA_ERR_INVALID_ARGUMENT.
 */
sa_status sa_forward_ex(const float *q, const void *k_pages, const void *v_pages,
                        int64_t num_pages, sa_dtype kv_dtype, const sa_index *idx,
                        const int32_t *block_tables, const int64_t *cu_seqlens_q,
                        const int32_t *used_kv_lens, int32_t hq, int32_t hkv, int32_t head_dim,
                        int32_t block_size, int32_t page_size, float softmax_scale,
                        int32_t causal, sa_dtype partial_dtype, void *o_partial,
                        float *m_partial, float *l_partial, sa_path path, void *stream,
                        void *q_scratch);

/*
 * Name of the kernel sa_forward launches for a problem of tq queries in
 * `batch` sequences with these head counts, sizes, K/V type and `path`
 * ("forward_dec_mma_kernel", "forward_tc_kernel", "forward_dec_kernel" or
 * "forward_cc_kernel"), or NULL where sa_forward would refuse it (bad head
 * counts or block/page sizes, or SA_ERR_UNSUPPORTED).  Host only; the returned
 * string is static.  The pages have no counterpart: it tells a caller (or a
 * profiling script) which kernel serves a shape.
 */
const char *sa_forward_kernel_name(int64_t tq, int32_t batch, int32_t hq, int32_t hkv,
                                   int32_t head_dim, int32_t block_size, int32_t page_size,
                                   sa_dtype kv_dtype, sa_path path);

/*
 * The kernel that sa_attention / sa_forward_combine run for steps 2 and 3
 * with this `causal` mode: "fused_dec_kernel" on the fused decode path (see
 * sa_attention), else the name sa_forward_kernel_name gives; NULL where the
 * call would be refused.  Host only (reads cu_seqlens_q_host[0..batch]).
 */
const char *sa_attention_kernel_name(int64_t tq, int32_t batch, const int64_t *cu_seqlens_q_host,
                                     int64_t num_pages, int32_t hq, int32_t hkv,
                                     int32_t head_dim, int32_t block_size, int32_t page_size,
                                     sa_dtype kv_dtype, int32_t causal, sa_path path);

/*
 * Steps 2 and 3 on an index built by sa_build_index (same stream), with no
 * host synchronisation: the forward and the combine, or, on the fused decode
 * path described at sa_attention, the one kernel that does both.  Arguments
 * as for sa_forward and sa_combine, plus `selected` and cu_seqlens_q_host
 * (those given to sa_build_index) and split_edges (used by the fused path
 * only: ranks per piece).  The partial buffers are scratch on the fused path.
 * Errors as for sa_forward and sa_combine; SA_ERR_SHAPE when the index's
 * block or page size differ from the arguments.
 */
sa_status sa_forward_combine(const float *q, const void *k_pages, const void *v_pages,
                             int64_t num_pages, sa_dtype kv_dtype, const sa_index *idx,
                             const int32_t *selected, const int64_t *cu_seqlens_q_host,
                             const int64_t *cu_seqlens_q, const int32_t *used_kv_lens,
                             const int32_t *block_tables, int32_t hq, int32_t head_dim,
                             int32_t block_size, int32_t page_size, float softmax_scale,
                             int32_t causal, int32_t split_edges, float *o_partial,
                             float *m_partial, float *l_partial, float *out, float *lse,
                             sa_path path, void *stream);

/* sa_forward_combine with o partials of `partial_dtype` (see sa_forward_ex);
 * on the fused decode path the pieces' scratch o rows take that type. */
sa_status sa_forward_combine_ex(const float *q, const void *k_pages, const void *v_pages,
                                int64_t num_pages, sa_dtype kv_dtype, const sa_index *idx,
                                const int32_t *selected, const int64_t *cu_seqlens_q_host,
                                const int64_t *cu_seqlens_q, const int32_t *used_kv_lens,
                                const int32_t *block_tables, int32_t hq, int32_t head_dim,
                                int32_t block_size, int32_t page_size, float softmax_scale,
                                int32_t causal, int32_t split_edges, sa_dtype partial_dtype,
                                void *o_partial, float *m_partial, float *l_partial, float *out,
                                float *lse, sa_path path, void *stream);

/*
 * Step 3: log-sum-exp combine (forward.rs module doc: "standard FlashAttention
 * log-sum-exp update").  For query i and q-head hq (h = hq / qhead), over
 * ranks r with inv[h, i, r] >= 0: M = max m_r, L = sum exp(m_r - M) l_r,
 * out[i, hq] = sum exp(m_r - M) o_r / L, lse[i, hq] = M + log L.  A row with
 * no live partial gets out = 0 and lse = -inf.
 *
 *   out  [tq, hq, head_dim] float32 (16-byte aligned)
 *   lse  [tq, hq] float32 or NULL
 */
sa_status sa_combine(const sa_index *idx, const float *o_partial, const float *m_partial,
                     const float *l_partial, int32_t hq, int32_t head_dim, float *out,
                     float *lse, void *stream);

/* sa_combine over o partials of `partial_dtype` (SA_DTYPE_F32: exactly
 * sa_combine; SA_DTYPE_BF16: the uint16 rows sa_forward_ex writes), widened
 * to f32 as they are read; other values: SA_ERR_INVALID_ARGUMENT. */
sa_status sa_combine_ex(const sa_index *idx, sa_dtype partial_dtype, const void *o_partial,
                        const float *m_partial, const float *l_partial, int32_t hq,
                        int32_t head_dim, float *out, float *lse, void *stream);

/*
 * Steps 1-3 on one stream, no host synchronisation (kvouter_attention, the
 * fused public entry of the module).  Arguments as above; `idx` carries the
 * caller's index arrays and workspace and is filled in as by sa_build_index.
 * The partial buffers are scratch of the sizes sa_forward documents.
 *
 * Fused decode path (SA_PATH_AUTO or SA_PATH_FUSED_DECODE): when causal is
 * 0 or 1, every sequence holds at most one query (cu_seqlens_q_host),
 * head_dim is 128,
 * page_size is a power of two of at least 8, block_size / page_size <= 8,
 * block_size <= 64 or a multiple of 64, qhead <= 4 (f32 K/V) or <= 16 (bf16),
 * num_pages * hkv * page_size < 2^31 and tq * hq * 4 < 2^31, steps 2 and 3
 * run as one kernel that keeps each query's partials on chip: every work
 * unit of such a batch carries edges of a single query, so the combine only
 * ever merges a (query, kv head)'s own units.  The index is still built in
 * full.  With split_edges = 0 each (query, kv head) is one piece of work
 * (topk <= 64), except that the pairs of the last, partial round over the
 * SMs are cut into pieces to fill the SMs; split_edges > 0 cuts every pair
 * into pieces of split_edges ranks (at most 64).  Pieces of one pair are
 * merged through rows of the partial buffers, whose content afterwards is
 * unspecified, and counted in one 4-byte counter per (query, kv head) that
 * the index build clears in its scratch (idx->workspace, or the library's
 * array for an index with SA_INDEX_STATIC_SCRATCH) and the kernel leaves at
 * zero: sa_forward_combine on this path returns SA_ERR_INVALID_ARGUMENT when
 * that scratch is missing or smaller than the build's layout.  out and lse
 * equal those of the unfused path up to rounding.  On this path
 * sa_attention clears the build's counters and the status word in one launch
 * on `stream`, then runs the index build on its side stream (forked from
 * `stream` after the clear) while the fused kernel runs on `stream` (it reads
 * no output of the build), and makes `stream` wait for the build before it
 * returns: work enqueued on `stream` afterwards sees both, and a CUDA graph
 * captured from `stream` holds the fork and the join.  An error either kernel
 * reports stays in the status word.
 */
sa_status sa_attention(const float *q, const void *k_pages, const void *v_pages,
                       int64_t num_pages, sa_dtype kv_dtype, const int32_t *selected,
                       int64_t tq, int32_t topk, const int64_t *cu_seqlens_q_host,
                       const int64_t *cu_seqlens_q, int32_t batch, const int32_t *used_kv_lens,
                       const int32_t *block_tables, int32_t max_pages, int32_t hq, int32_t hkv,
                       int32_t head_dim, int32_t block_size, int32_t page_size,
                       float softmax_scale, int32_t causal, int32_t split_edges, sa_index *idx,
                       float *o_partial, float *m_partial, float *l_partial, float *out,
                       float *lse, sa_path path, void *stream);

/* sa_attention with o partials of `partial_dtype` (see sa_forward_ex); the
 * o_partial buffer is [tq*hkv*topk*qhead, head_dim] of that type. */
sa_status sa_attention_ex(const float *q, const void *k_pages, const void *v_pages,
                          int64_t num_pages, sa_dtype kv_dtype, const int32_t *selected,
                          int64_t tq, int32_t topk, const int64_t *cu_seqlens_q_host,
                          const int64_t *cu_seqlens_q, int32_t batch,
                          const int32_t *used_kv_lens, const int32_t *block_tables,
                          int32_t max_pages, int32_t hq, int32_t hkv, int32_t head_dim,
                          int32_t block_size, int32_t page_size, float softmax_scale,
                          int32_t causal, int32_t split_edges, sa_index *idx,
                          sa_dtype partial_dtype, void *o_partial, float *m_partial,
                          float *l_partial, float *out, float *lse, sa_path path, void *stream);

/*
 * Test hook for the bounded device waits (the pages have no counterpart:
 * their GpuRuntimeError stands for any device failure).  Every wait inside
 * the kernels gives up after a bounded number of tries, records
 * SA_ERR_DEVICE_TIMEOUT in the index's status word and lets the kernel
 * return.  This call makes one such wait run out on purpose, so that a test
 * can see the status and then check that the next clean call works:
 *   site 1: the index kernel's grid barrier is never released (every CTA of
 *           the build times out and returns; the index is left unfinished);
 *   site 2: the fused decode kernel's load warps issue no copy (its
 *           consumer, merge and metadata warps time out and return; no copy
 *           is ever in flight);
 *   site 0: normal operation.
 * spin_limit: tries of each bounded wait from now on (0 = the library's
 * default, about a second).  Process-wide, read at every launch; not for
 * production use and not safe to change while other threads launch.
 * Returns SA_ERR_INVALID_ARGUMENT for an unknown site.
 */
sa_status sa_debug_stall(int32_t site, uint32_t spin_limit);

/*
 * Test hook for the tensor-core forward's load balance (the pages have no
 * counterpart: their WorkSplit list is walked by a thread pool).  With
 * n_ctas > 0, every later tcgen05 forward adds, for each CTA c < n_ctas,
 * the rows (edge x GQA lane) and the units it claimed to stats[3 c] and
 * stats[3 c + 1], and writes the CTA's busy time in SM clock cycles (kernel
 * start to end) to stats[3 c + 2].  stats: device memory of 3 * n_ctas
 * int64 that the caller zeroes; n_ctas = 0 turns the hook off.
 * Process-wide, not for production use.  SA_ERR_INVALID_ARGUMENT for
 * n_ctas < 0 or a NULL stats with n_ctas > 0.
 */
sa_status sa_debug_cta_stats(int64_t *stats, int32_t n_ctas);

/* Synchronises `stream` and returns the first device-detected error recorded
 * in idx->totals[3] (SA_OK if none), or SA_ERR_CUDA if the stream failed. */
sa_status sa_get_status(const sa_index *idx, void *stream);

/* Clears the device status word of an index (enqueued on `stream`). */
sa_status sa_clear_status(const sa_index *idx, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* SA_H_ */
