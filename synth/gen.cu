// Seeded synthetic bf16 inputs, written straight into device memory.
//
// This library only makes inputs.  It holds none of the operator's
// arithmetic (no rank sum, no residual add, no normalisation, no
// round-to-nearest bf16 conversion) and is shared by the CUDA path and the
// CPU oracle's tests only as a source of input bytes.
//
// Generator (one counter-based stream per (seed, stream_id)):
//   SplitMix64 output mixing of Steele, Lea and Flood, "Fast Splittable
//   Pseudorandom Number Generators" (OOPSLA 2014): gamma 0x9E3779B97F4A7C15,
//   finaliser  z ^= z>>30; z *= 0xBF58476D1CE4E5B9; z ^= z>>27;
//              z *= 0x94D049BB133111EB; z ^= z>>31.
//   base      = mix(seed ^ mix(stream_id + gamma))
//   draw(j)   = mix(base + (j + 1) * gamma)
//   element i uses draws 3i (u1), 3i+1 (u2), 3i+2 (u3)
//   u(z)      = ((z >> 11) + 0.5) * 2^-53, in (0, 1)
//   normal    : mean + sqrt(var) * sqrt(-2 ln u1) * cos(2 pi u2)  (Box-Muller)
//   uniform   : a + (b - a) * u1
//   outlier   : value *= outlier_scale when u3 < outlier_p
//   value (fp64) -> fp32 (IEEE round to nearest) -> bf16 by truncation
//   (the upper 16 bits of the fp32 pattern).
// The numpy twin in synth/__init__.py evaluates the same recipe on the host.
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ull;

__host__ __device__ inline uint64_t mix64(uint64_t z) {
  z ^= z >> 30;
  z *= 0xBF58476D1CE4E5B9ull;
  z ^= z >> 27;
  z *= 0x94D049BB133111EBull;
  z ^= z >> 31;
  return z;
}

__device__ inline double unit(uint64_t z) {
  return ((double)(z >> 11) + 0.5) * 0x1.0p-53;
}

// One value of the recipe, element i of the stream with key `base`.
__device__ inline float draw(int64_t i, uint64_t base, int dist, double p0, double p1,
                             double outlier_p, double outlier_scale) {
  const double kTwoPi = 6.283185307179586476925286766559;
  uint64_t j = 3ull * (uint64_t)i;
  double u1 = unit(mix64(base + (j + 1) * kGamma));
  double u2 = unit(mix64(base + (j + 2) * kGamma));
  double v;
  if (dist == 0) {
    double z = sqrt(-2.0 * log(u1)) * cos(kTwoPi * u2);
    v = p0 + sqrt(p1) * z;
  } else {
    v = p0 + (p1 - p0) * u1;
  }
  if (outlier_p > 0.0) {
    double u3 = unit(mix64(base + (j + 3) * kGamma));
    if (u3 < outlier_p) v *= outlier_scale;
  }
  return (float)v;
}

__global__ void fill_f32_kernel(float* __restrict__ dst, int64_t n, uint64_t base, int dist,
                                double p0, double p1, double outlier_p,
                                double outlier_scale) {
  int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
    dst[i] = draw(i, base, dist, p0, p1, outlier_p, outlier_scale);
}

__global__ void fill_bf16_kernel(uint16_t* __restrict__ dst, int64_t n,
                                 uint64_t base, int dist, double p0, double p1,
                                 double outlier_p, double outlier_scale) {
  int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    const float f = draw(i, base, dist, p0, p1, outlier_p, outlier_scale);
    dst[i] = (uint16_t)(__float_as_uint(f) >> 16);
  }
}

}  // namespace

extern "C" {

// Fills dst[0..n) (device memory, bf16 patterns) on `stream`.
// dist 0: normal with mean p0 and variance p1;  dist 1: uniform on [p0, p1).
// Returns 0, -1 for a bad argument, -4 for a CUDA launch error.
int farn_synth_fill_bf16(void* dst, int64_t n, uint64_t seed,
                         uint64_t stream_id, int dist, double p0, double p1,
                         double outlier_p, double outlier_scale,
                         cudaStream_t stream) {
  if (n < 0 || (n > 0 && dst == nullptr) || (dist != 0 && dist != 1) ||
      (dist == 0 && !(p1 >= 0.0)) || !(outlier_p >= 0.0))
    return -1;
  if (n == 0) return 0;
  uint64_t base = mix64(seed ^ mix64(stream_id + kGamma));
  int threads = 256;
  int64_t want = (n + threads - 1) / threads;
  int blocks = (int)(want < 152 * 32 ? want : 152 * 32);
  fill_bf16_kernel<<<blocks, threads, 0, stream>>>(
      (uint16_t*)dst, n, base, dist, p0, p1, outlier_p, outlier_scale);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

// The same recipe kept in fp32 (no bf16 truncation): dst is float[n].
int farn_synth_fill_f32(void* dst, int64_t n, uint64_t seed, uint64_t stream_id, int dist,
                        double p0, double p1, double outlier_p, double outlier_scale,
                        cudaStream_t stream) {
  if (n < 0 || (n > 0 && dst == nullptr) || (dist != 0 && dist != 1) ||
      (dist == 0 && !(p1 >= 0.0)) || !(outlier_p >= 0.0))
    return -1;
  if (n == 0) return 0;
  uint64_t base = mix64(seed ^ mix64(stream_id + kGamma));
  int threads = 256;
  int64_t want = (n + threads - 1) / threads;
  int blocks = (int)(want < 152 * 32 ? want : 152 * 32);
  fill_f32_kernel<<<blocks, threads, 0, stream>>>((float*)dst, n, base, dist, p0, p1,
                                                  outlier_p, outlier_scale);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

}  // extern "C"
