// Device fill for the seeded synthetic inputs: writes elements
// [start, start + count) of the counter-based generator documented in
// inputs/__init__.py (splitmix64 finaliser, Irwin-Hall sum of four 16-bit
// fields, one rounded float multiply), as float32 or as round-to-nearest-even
// bf16.  Input generation only; it holds no attention arithmetic.
#include <cstdint>
#include <cuda_runtime.h>

namespace {

__device__ __forceinline__ uint64_t splitmix64(uint64_t x) {
  uint64_t z = x + 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__device__ __forceinline__ float counter_value(uint64_t key, uint64_t idx) {
  const uint64_t z = splitmix64(idx + key * 0xD1B54A32D192ED03ull);
  const int64_t u = (int64_t)(z & 0xFFFF) + (int64_t)((z >> 16) & 0xFFFF) +
                    (int64_t)((z >> 32) & 0xFFFF) + (int64_t)((z >> 48) & 0xFFFF);
  // 1 / sqrt((65536^2 - 1) / 3) rounded to float (bits 0x37ddb3d7), the
  // same constant as the host side.
  const float scale = __uint_as_float(0x37ddb3d7u);
  return __fmul_rn((float)(u - 131070), scale);
}

__device__ __forceinline__ uint16_t to_bf16_rne(float f) {
  const uint32_t b = __float_as_uint(f);
  return (uint16_t)((b + 0x7FFFu + ((b >> 16) & 1u)) >> 16);
}

__global__ void fill_f32(float* __restrict__ dst, int64_t count, int64_t start, uint64_t key) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < count; i += stride)
    dst[i] = counter_value(key, (uint64_t)(start + i));
}

__global__ void fill_bf16(uint16_t* __restrict__ dst, int64_t count, int64_t start, uint64_t key) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < count; i += stride)
    dst[i] = to_bf16_rne(counter_value(key, (uint64_t)(start + i)));
}

}  // namespace

extern "C" int sa_inputs_fill(void* dst, int64_t count, int64_t start, uint64_t seed,
                              uint32_t stream_id, int bf16, void* stream) {
  if (count <= 0) return 0;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const uint64_t key = seed * 16ull + stream_id;
  const int threads = 256;
  int64_t blocks = (count + threads - 1) / threads;
  const int64_t cap = (int64_t)(sms > 0 ? sms : 1) * 16;
  if (blocks > cap) blocks = cap;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (bf16)
    fill_bf16<<<(unsigned)blocks, threads, 0, s>>>(static_cast<uint16_t*>(dst), count, start, key);
  else
    fill_f32<<<(unsigned)blocks, threads, 0, s>>>(static_cast<float*>(dst), count, start, key);
  return (int)cudaGetLastError();
}
