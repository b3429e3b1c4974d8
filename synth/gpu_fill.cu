// Device copy of the seeded word stream of synth/gen.py: word 2i / 2i+1 is
// the low / high half of SplitMix64 draw i of a stream key.  Integer-only,
// so host and device produce identical bits.  Input generation only.
#include <cuda_runtime.h>
#include <stdint.h>

namespace {
__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z ^= z >> 30;
  z *= 0xBF58476D1CE4E5B9ull;
  z ^= z >> 27;
  z *= 0x94D049BB133111EBull;
  z ^= z >> 31;
  return z;
}

__global__ void fill_words_kernel(uint32_t *dst, uint64_t n_words, uint64_t key) {
  const uint64_t n_draws = (n_words + 1) / 2;
  for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < n_draws;
       i += (uint64_t)gridDim.x * blockDim.x) {
    const uint64_t d = mix64(key + (i + 1) * 0x9E3779B97F4A7C15ull);
    dst[2 * i] = (uint32_t)d;
    if (2 * i + 1 < n_words) dst[2 * i + 1] = (uint32_t)(d >> 32);
  }
}
}  // namespace

extern "C" int synth_fill_words(void *dst, unsigned long long n_words, unsigned long long key, void *stream) {
  if (!dst || ((uintptr_t)dst & 3)) return 1;
  if (n_words == 0) return 0;
  const unsigned long long draws = (n_words + 1) / 2;
  unsigned long long blocks = (draws + 255) / 256;
  if (blocks > 152ull * 16) blocks = 152ull * 16;
  fill_words_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>((uint32_t *)dst, n_words, key);
  return cudaGetLastError() == cudaSuccess ? 0 : 2;
}
