// Device helpers shared by the kernels of libsa: status reporting, bounded
// mbarrier waits, 1-D bulk and tensor-map (TMA) copies into shared memory.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "sa.h"

namespace sa {

// Upper bounds of spin loops.  A wait that runs out records
// SA_ERR_DEVICE_TIMEOUT and lets the kernel return instead of hanging.
constexpr uint32_t kSpinLimit = 1u << 22;        // ~0.25-4 s with backoff
constexpr int kMaxMsb = 16384;                    // bins of the index kernel (3 per block in shared memory)

// Record the first device-side error of a call in the index status word.
__device__ __forceinline__ void report(int64_t* status_word, int code) {
  if (status_word != nullptr)
    atomicCAS(reinterpret_cast<unsigned long long*>(status_word), 0ull,
              static_cast<unsigned long long>(code));
}

// Programmatic dependent launch: a kernel lets the next kernel of its stream
// (launched with programmatic stream serialization) start before it ends;
// that kernel waits for its prerequisite grids to finish, and their memory to
// be visible, where it calls griddep_wait.  Both are no-ops without such a
// launch.
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Arrive once and announce `bytes` of transactions that the bulk copies
// issued next will complete.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// Plain arrival (release at CTA scope).
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for phase `parity` of `bar` to complete, at most `limit` tries
// (kSpinLimit by default).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint32_t limit = kSpinLimit) {
  for (uint32_t i = 0; i < limit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

// 1-D bulk copy global -> shared, completion counted on `bar`.  Both
// addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* smem_dst, const void* gmem_src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_u32(smem_dst)), "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Tiled tensor-map copies global -> shared (2-D and 3-D boxes), completion
// counted on `bar`.  `tmap` is the address of a CUtensorMap kernel parameter;
// the innermost coordinate x must be 16-byte aligned in bytes (the callers
// pass x = 0).
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const void* tmap, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];"
      ::"r"(smem_u32(smem_dst)), "l"(tmap), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* smem_dst, const void* tmap, int x, int y, int z,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];"
      ::"r"(smem_u32(smem_dst)), "l"(tmap), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ float bf16_to_f32(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// Unpack 4 bf16 (8 bytes) into floats.
__device__ __forceinline__ float4 bf16x4_to_f32(uint2 u) {
  float4 r;
  r.x = __uint_as_float(u.x << 16);
  r.y = __uint_as_float(u.x & 0xFFFF0000u);
  r.z = __uint_as_float(u.y << 16);
  r.w = __uint_as_float(u.y & 0xFFFF0000u);
  return r;
}

// Tiled tensor-map copy shared -> global (2-D box at (x, y)), tracked by the
// issuing thread's bulk groups.  x * element size must be a multiple of 16
// bytes and x, y non-negative; the source tile is laid out as the map's
// swizzle mode defines on absolute shared-memory address bits.
__device__ __forceinline__ void tma_store_2d(const void* tmap, int x, int y, const void* smem_src) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];"
               ::"l"(tmap), "r"(x), "r"(y), "r"(smem_u32(smem_src))
               : "memory");
}

__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// The issuing thread's committed bulk stores have read their shared-memory
// sources (the sources may be rewritten).
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// All but the most recent of the issuing thread's committed bulk stores
// have read their shared-memory sources.
__device__ __forceinline__ void bulk_wait_read_1() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}

// All but the N most recent of the issuing thread's committed bulk stores
// have read their shared-memory sources.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// The issuing thread's committed bulk stores have completed.
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Two f32 values to a packed bf16x2 (round to nearest even), `lo` in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2_rn(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Four consecutive elements of a partial o buffer, starting at element `off`
// (a multiple of 4): f32, or bf16 rounded to nearest even when the caller
// asked for 16-bit o partials.
__device__ __forceinline__ void store_o4(void* o, int bf16, int64_t off, float4 v) {
  if (bf16)
    *reinterpret_cast<uint2*>(static_cast<uint16_t*>(o) + off) =
        make_uint2(pack_bf16x2_rn(v.x, v.y), pack_bf16x2_rn(v.z, v.w));
  else
    *reinterpret_cast<float4*>(static_cast<float*>(o) + off) = v;
}

}  // namespace sa
