// Block-wide reductions and the exact top-k threshold searches shared by the
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

// The largest 48-bit value x such that reach(W(x)) holds, where W(x) is the
// weight of the eligible elements c in [0, len) whose key(c) >= x. With
// unique keys and a reach that grows with W, this x is the key of the last
// member of the (key descending) prefix that first reaches the goal: the
// same answer as a bit-by-bit search from the top, found one 8-bit digit
// per pass (at most six passes) from a shared-memory histogram of weights.
// Each bin also counts its keys (bits 40 and up of the entry); once the
// chosen bin holds a single eligible key, that key is the answer and the
// remaining passes are skipped. Digit 0, where most small masses fall in the
// first passes, is summed per warp before its one shared atomic. Keys must be
// < 2^48 and the total eligible weight < 2^40; reach(total eligible weight)
// must hold (then every pass finds a digit). If reach(0) holds the result is
// 2^48 - 1 (no key reaches it). All threads of the block call it.
// hist: 256 entries; bcast: 4 entries (shared memory).
template <typename KeyFn, typename WeightFn, typename EligFn, typename ReachFn>
__device__ __forceinline__ uint64_t radix_max_key(int len, KeyFn key_of, WeightFn weight_of, EligFn eligible,
                                                  ReachFn reach, unsigned long long* hist,
                                                  unsigned long long* bcast) {
  constexpr unsigned long long kOne = 1ull << 40, kWeight = kOne - 1;  // count unit, weight field
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint64_t prefix = 0;            // digits decided so far
  unsigned long long above = 0;   // weight of eligible keys above the current bucket
  for (int shift = 40; shift >= 0; shift -= 8) {
    for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0ull;
    __syncthreads();
    unsigned long long w0 = 0;
    for (int c = threadIdx.x; c < len; c += blockDim.x) {
      if (!eligible(c)) continue;
      const uint64_t key = key_of(c);
      if ((key >> (shift + 8)) != prefix) continue;
      const int d = static_cast<int>((key >> shift) & 255u);
      const unsigned long long w = kOne + weight_of(c);
      if (d == 0)
        w0 += w;
      else
        atomicAdd(&hist[d], w);
    }
    w0 = warp_sum(w0);
    if (lane == 0 && w0 != 0ull) atomicAdd(&hist[0], w0);
    __syncthreads();
    if (warp == 0) {
      // Lane l holds bins 255-8l .. 248-8l (descending); cumulative weights
      // from the top find the largest digit whose suffix reaches the goal.
      unsigned long long v[8], cnt[8], mine = 0;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const unsigned long long e = hist[255 - 8 * lane - k];
        v[k] = e & kWeight;
        cnt[k] = e >> 40;
        mine += v[k];
      }
      unsigned long long before = mine;  // inclusive scan over lanes, then exclusive
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long t = __shfl_up_sync(0xffffffffu, before, o);
        if (lane >= o) before += t;
      }
      before -= mine;
      unsigned long long run = above + before;
      int found = -1;
      unsigned long long run_above = 0, found_cnt = 0;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        if (found < 0 && reach(run + v[k])) {
          found = 255 - 8 * lane - k;
          run_above = run;
          found_cnt = cnt[k];
        }
        run += v[k];
      }
      const unsigned int hits = __ballot_sync(0xffffffffu, found >= 0);
      const int first = hits ? __ffs(hits) - 1 : 31;
      if (lane == first) {
        bcast[0] = static_cast<unsigned long long>(found >= 0 ? found : 0);
        bcast[1] = found >= 0 ? run_above : above;
        bcast[2] = found >= 0 ? found_cnt : 0ull;
      }
    }
    __syncthreads();
    prefix = (prefix << 8) | bcast[0];
    above = bcast[1];
    if (bcast[2] == 1ull && shift > 0) {
      // One eligible key carries the decided digits: the goal is reached at
      // it and not above it, so it is the answer.
      for (int c = threadIdx.x; c < len; c += blockDim.x)
        if (eligible(c) && (key_of(c) >> shift) == prefix) bcast[3] = key_of(c);
      __syncthreads();
      const uint64_t x = bcast[3];
      __syncthreads();  // bcast is free for the caller's next search
      return x;
    }
    __syncthreads();
  }
  return prefix;
}

// The same search by one warp on its own (no block barrier): `hist` is the
// warp's own 256 entries and `last` 256 key indexes; weight_of(c, key) is
// given the key already formed. Every lane of the warp calls it with the
// same arguments and gets the result. Each pass records the index of one key
// of each digit (digit 0, summed in registers without atomics, in a register
// per lane): when the chosen digit holds a single key, that index names the
// answer without another read of the row.
template <typename KeyFn, typename WeightFn, typename EligFn, typename ReachFn>
__device__ __forceinline__ uint64_t warp_radix_max_key(int len, KeyFn key_of, WeightFn weight_of, EligFn eligible,
                                                       ReachFn reach, unsigned long long* hist,
                                                       unsigned short* last) {
  constexpr unsigned long long kOne = 1ull << 40, kWeight = kOne - 1;
  const int lane = threadIdx.x & 31;
  uint64_t prefix = 0;
  unsigned long long above = 0;
  for (int shift = 40; shift >= 0; shift -= 8) {
#pragma unroll
    for (int k = 0; k < 8; ++k) hist[lane + 32 * k] = 0ull;
    __syncwarp();
    unsigned long long w0 = 0;
    int c0 = 0;  // a key of digit 0 seen by this lane
    for (int c = lane; c < len; c += 32) {
      if (!eligible(c)) continue;
      const uint64_t key = key_of(c);
      if ((key >> (shift + 8)) != prefix) continue;
      const int d = static_cast<int>((key >> shift) & 255u);
      const unsigned long long w = kOne + weight_of(c, key);
      if (d == 0) {
        w0 += w;
        c0 = c;
      } else {
        atomicAdd(&hist[d], w);
        last[d] = static_cast<unsigned short>(c);  // any writer: read only when the digit holds one key
      }
    }
    const bool has0 = w0 != 0;
    w0 = warp_sum(w0);
    __syncwarp();
    if (lane == 0) hist[0] = w0;  // digit 0 takes no atomics
    __syncwarp();
    unsigned long long v[8], cnt[8], mine = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const unsigned long long e = hist[255 - 8 * lane - k];
      v[k] = e & kWeight;
      cnt[k] = e >> 40;
      mine += v[k];
    }
    unsigned long long before = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long t = __shfl_up_sync(0xffffffffu, before, o);
      if (lane >= o) before += t;
    }
    before -= mine;
    unsigned long long run = above + before, run_above = 0, found_cnt = 0;
    int found = -1;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      if (found < 0 && reach(run + v[k])) {
        found = 255 - 8 * lane - k;
        run_above = run;
        found_cnt = cnt[k];
      }
      run += v[k];
    }
    const unsigned int hits = __ballot_sync(0xffffffffu, found >= 0);
    const int first = hits ? __ffs(hits) - 1 : 31;
    const int digit = __shfl_sync(0xffffffffu, found >= 0 ? found : 0, first);
    const unsigned long long new_above = __shfl_sync(0xffffffffu, found >= 0 ? run_above : above, first);
    const unsigned long long single = __shfl_sync(0xffffffffu, found >= 0 ? found_cnt : 0ull, first);
    prefix = (prefix << 8) | static_cast<uint64_t>(digit);
    above = new_above;
    if (single == 1ull && shift > 0) {
      // One eligible key carries the decided digits: the goal is reached at
      // it and not above it, so it is the answer.
      int c;
      if (digit == 0) {
        const unsigned int own = __ballot_sync(0xffffffffu, has0);  // the one lane that saw it
        c = __shfl_sync(0xffffffffu, c0, own ? __ffs(own) - 1 : 0);
      } else {
        c = last[digit];
      }
      return key_of(c);
    }
    __syncwarp();  // every lane has read hist and last before the next pass writes them
  }
  return prefix;
}

}  // namespace crisp
