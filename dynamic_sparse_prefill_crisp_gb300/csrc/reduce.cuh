// Block-wide reductions and the exact top-k threshold search shared by the
// selection kernels.
#pragma once

#include <cstdint>

namespace crisp {

template <typename T>
__device__ __forceinline__ T warp_sum(T v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Sum over the block; every thread gets the result. `scratch` holds >= 32 T.
// Must be called by all threads of the block.
template <typename T>
__device__ __forceinline__ T block_sum(T v, T* scratch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) scratch[warp] = v;
  __syncthreads();
  T r = 0;
  for (int w = 0; w < nw; ++w) r += scratch[w];
  return r;
}

// Selection key: mass first, then the lower index; unique per position.
// Masses of a probability map are < 2^43 (a 128x128 tile of Q32 quanta), so
// mass << 13 | (8191 - c) fits in 56 bits; larger masses saturate.
constexpr int kKeyBits = 56;
__device__ __forceinline__ uint64_t sel_key(uint64_t m, int c) {
  const uint64_t cap = (1ull << 43) - 1;
  return ((m < cap ? m : cap) << 13) | static_cast<uint64_t>(8191 - c);
}

}  // namespace crisp
