// Device fill kernels of the seeded synthetic-input generator.
//
// Same definition as synth/__init__.py (splitmix64 counter hash, twelve
// 24-bit uniforms, Irwin-Hall sum, fp32 scale, optional |x| and bf16 RNE),
// so a buffer filled here equals the host draws bit for bit. Input generation
// only: nothing of the FSDP step is computed here.
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace {

constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ull;

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__device__ __forceinline__ float draw(uint64_t key, uint64_t i, float scale, int absval) {
  int64_t s = 0;
  const uint64_t base = i * 6ull;
#pragma unroll
  for (int d = 0; d < 6; ++d) {
    uint64_t z = mix64(key + (base + (uint64_t)(d + 1)) * kGamma);
    s += (int64_t)(z >> 40);
    s += (int64_t)((z >> 16) & 0xFFFFFFull);
  }
  const int64_t c = s - (int64_t)(6ll << 24);
  float x = __fmul_rn(__ll2float_rn(c), scale);
  return absval ? fabsf(x) : x;
}

__global__ void fill_f32_kernel(float* out, int64_t n, int64_t idx0, int64_t n_valid,
                                uint64_t key, float scale, int absval) {
  for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < n;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int64_t i = idx0 + e;
    out[e] = (i < n_valid) ? draw(key, (uint64_t)i, scale, absval) : 0.0f;
  }
}

__global__ void fill_bf16_kernel(uint16_t* out, int64_t n, int64_t idx0, int64_t n_valid,
                                 uint64_t key, float scale, int absval) {
  for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < n;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int64_t i = idx0 + e;
    float x = (i < n_valid) ? draw(key, (uint64_t)i, scale, absval) : 0.0f;
    out[e] = __bfloat16_as_ushort(__float2bfloat16_rn(x));
  }
}

int grid_for(int64_t n) {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int64_t want = (n + 255) / 256;
  int64_t cap = (int64_t)(sms > 0 ? sms : 1) * 16;
  return (int)(want < cap ? (want > 0 ? want : 1) : cap);
}

}  // namespace

extern "C" int synth_fill_f32(void* out, int64_t n, int64_t idx0, int64_t n_valid,
                              uint64_t key, float scale, int absval, void* stream) {
  if (n <= 0) return 0;
  fill_f32_kernel<<<grid_for(n), 256, 0, (cudaStream_t)stream>>>(
      (float*)out, n, idx0, n_valid, key, scale, absval);
  return (int)cudaGetLastError();
}

extern "C" int synth_fill_bf16(void* out, int64_t n, int64_t idx0, int64_t n_valid,
                               uint64_t key, float scale, int absval, void* stream) {
  if (n <= 0) return 0;
  fill_bf16_kernel<<<grid_for(n), 256, 0, (cudaStream_t)stream>>>(
      (uint16_t*)out, n, idx0, n_valid, key, scale, absval);
  return (int)cudaGetLastError();
}
