// synth_gen.cu - device copy of the counter-based input generator (synth/rng.py).
//
// Fills a byte buffer with uniform integers in [lo, hi] drawn exactly as the
// host generator does: key = splitmix64(splitmix64(seed) ^ stream),
// u = splitmix64(key ^ i), value = lo + ((u >> 32) * (hi - lo + 1)) >> 32,
// stored as a two's-complement byte.  Holds no attention arithmetic; it only
// makes multi-GB synthetic caches without a host round trip.
#include <cstdint>
#include <cuda_runtime.h>

namespace {

__host__ __device__ __forceinline__ uint64_t splitmix64(uint64_t x) {
  uint64_t z = x + 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__global__ void fill_uniform_i8(uint8_t* dst, uint64_t start, uint64_t n, uint64_t key,
                                int32_t lo, uint64_t span) {
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    const uint64_t u = splitmix64(key ^ (start + i));
    const int64_t v = (int64_t)lo + (int64_t)(((u >> 32) * span) >> 32);
    dst[i] = (uint8_t)(int8_t)v;
  }
}

}  // namespace

extern "C" int synth_fill_uniform_i8(void* dst, uint64_t start, uint64_t n, uint64_t seed,
                                     uint64_t stream_id, int32_t lo, int32_t hi, void* stream) {
  if (n == 0) return 0;
  if (!dst || hi < lo) return 1;
  const uint64_t key = splitmix64(splitmix64(seed) ^ stream_id);
  const uint64_t span = (uint64_t)((int64_t)hi - lo + 1);
  const int threads = 256;
  uint64_t blocks = (n + threads - 1) / threads;
  if (blocks > 152ull * 64) blocks = 152ull * 64;
  fill_uniform_i8<<<(unsigned)blocks, threads, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<uint8_t*>(dst), start, n, key, lo, span);
  return cudaGetLastError() == cudaSuccess ? 0 : 2;
}
