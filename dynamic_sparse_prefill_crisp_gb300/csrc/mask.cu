// A7. Per-head sparse block mask (ai-feeds page, "方法": the method's output
// is a per-head sparse attention mask), one bitset row per query block:
//   VS head: {kb <= qb : kb in V} U {qb - s, qb - s - 1 : s in S}
//   PE head: the pebits row qb
// and the attention work order: rows sorted by block count, largest first
// (longest-processing-time order for the attention grid).
//
// The slash part is built a word at a time: with Srev the slash set reversed
// (bit x of Srev = bit nb-1-x of S), bit b of word w of {qb - s} is Srev bit
// nb-1-qb+32w+b, a 32-bit window of Srev (a funnel shift of two words); the
// {qb - s - 1} part is the window one bit further.
#include "common.cuh"
#include "reduce.cuh"

namespace crisp {

namespace {

__global__ void srev_kernel(const uint32_t* __restrict__ sbits, const uint8_t* __restrict__ route, int nb,
                            uint32_t* __restrict__ srev) {
  const int h = blockIdx.x;
  const int W = (nb + 31) / 32;
  const uint32_t* S = sbits + static_cast<size_t>(h) * W;
  for (int w = threadIdx.x; w < W + 2; w += blockDim.x) {
    uint32_t word = 0;
    if (route[h]) {
      for (int b = 0; b < 32; ++b) {
        const int x = 32 * w + b;
        if (x < nb) {
          const int s = nb - 1 - x;
          word |= ((S[s >> 5] >> (s & 31)) & 1u) << b;
        }
      }
    }
    srev[static_cast<size_t>(h) * (W + 2) + w] = word;
  }
}

__device__ __forceinline__ uint32_t window32(const uint32_t* v, int p) {
  return __funnelshift_r(v[p >> 5], v[(p >> 5) + 1], p & 31);
}

// grid (nb, hq); one thread per bitset word.
__global__ void mask_kernel(const uint8_t* __restrict__ route, const uint32_t* __restrict__ vbits,
                            const uint32_t* __restrict__ srev, const uint32_t* __restrict__ pebits, int nb,
                            uint32_t* __restrict__ rowbits, int32_t* __restrict__ counts) {
  __shared__ int scratch[32];
  const int qb = blockIdx.x, h = blockIdx.y;
  const int W = (nb + 31) / 32, wq = qb >> 5;
  const bool vs = route[h] != 0;
  const uint32_t* V = vbits + static_cast<size_t>(h) * W;
  const uint32_t* R = srev + static_cast<size_t>(h) * (W + 2);
  const uint32_t* PE = pebits + (static_cast<size_t>(h) * nb + qb) * W;
  uint32_t* out = rowbits + (static_cast<size_t>(h) * nb + qb) * W;
  int cnt = 0;
  for (int w = threadIdx.x; w < W; w += blockDim.x) {
    uint32_t word = 0;
    if (w <= wq) {
      if (vs) {
        const int p = nb - 1 - qb + 32 * w;
        word = V[w] | window32(R, p) | window32(R, p + 1);
      } else {
        word = PE[w];
      }
      if (w == wq && (qb & 31) != 31) word &= (1u << ((qb & 31) + 1)) - 1u;
    }
    out[w] = word;
    cnt += __popc(word);
  }
  const int total = block_sum(cnt, scratch);
  if (threadIdx.x == 0) counts[static_cast<size_t>(h) * nb + qb] = total;
}

// Counting sort of the rows by count, descending.
__global__ void bucket_clear(int32_t* __restrict__ bucket, int len) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < len) bucket[i] = 0;
}

__global__ void count_hist(const int32_t* __restrict__ counts, int items, int nb, int32_t* __restrict__ bucket) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < items) atomicAdd(&bucket[min(max(counts[i], 0), nb)], 1);
}

// bucket[c] <- number of items with count > c (exclusive scan from the top).
__global__ void count_scan(int32_t* __restrict__ bucket, int nb) {
  __shared__ int32_t part[1024];
  const int per = (nb + 1 + blockDim.x - 1) / blockDim.x;
  // thread t owns counts [nb - (t+1)*per + 1, nb - t*per] (descending order)
  const int hi = nb - threadIdx.x * per;
  int32_t s = 0;
  for (int c = hi; c > hi - per && c >= 0; --c) s += bucket[c];
  part[threadIdx.x] = s;
  __syncthreads();
  if (threadIdx.x == 0) {
    int32_t run = 0;
    for (int t = 0; t < static_cast<int>(blockDim.x); ++t) {
      const int32_t v = part[t];
      part[t] = run;
      run += v;
    }
  }
  __syncthreads();
  int32_t run = part[threadIdx.x];
  for (int c = hi; c > hi - per && c >= 0; --c) {
    const int32_t v = bucket[c];
    bucket[c] = run;
    run += v;
  }
}

__global__ void count_scatter(const int32_t* __restrict__ counts, int items, int nb, int32_t* __restrict__ bucket,
                              int32_t* __restrict__ order) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < items) order[atomicAdd(&bucket[min(max(counts[i], 0), nb)], 1)] = i;
}

}  // namespace

cudaError_t launch_build_mask(const crisp_shape& s, const uint8_t* route, const uint32_t* vbits,
                              const uint32_t* sbits, const uint32_t* pebits, uint32_t* rowbits, int32_t* counts,
                              int32_t* order, char* ws, cudaStream_t st) {
  const ScratchLayout L = scratch_layout(s);
  const int nb = num_blocks(s.seq_len);
  const int items = s.hq * nb;
  auto* srev = reinterpret_cast<uint32_t*>(ws + L.srev);
  auto* bucket = reinterpret_cast<int32_t*>(ws + L.bucket);
  srev_kernel<<<s.hq, 128, 0, st>>>(sbits, route, nb, srev);
  mask_kernel<<<dim3(nb, s.hq), 128, 0, st>>>(route, vbits, srev, pebits, nb, rowbits, counts);
  // Schedule: row ids sorted by count, descending (counting sort).
  bucket_clear<<<(nb + 2 + 255) / 256, 256, 0, st>>>(bucket, nb + 2);
  count_hist<<<(items + 255) / 256, 256, 0, st>>>(counts, items, nb, bucket);
  count_scan<<<1, 1024, 0, st>>>(bucket, nb);
  count_scatter<<<(items + 255) / 256, 256, 0, st>>>(counts, items, nb, bucket, order);
  return cudaGetLastError();
}

}  // namespace crisp
