// A7. Per-head sparse block mask (ai-feeds page, "方法": the method's output
// is a per-head sparse attention mask), one bitset row per query block:
//   VS head: {kb <= qb : kb in V} U {qb - s, qb - s - 1 : s in S}
//   PE head: the pebits row qb
// and the attention work order: kv group by kv group; within a group query
// blocks descending, the group's heads consecutive. A causal row's block
// count grows with qb, so each group runs its longest rows first (the short
// rows of the last group's first query blocks fill the tail), and the CTAs in
// flight gather the K/V blocks of one kv group, which then stay in L2. Query
// blocks descending across all heads was measured slower where heads keep
// many blocks (7 % at 256k with 24 PE heads), and a strict sort by count
// slower still: both spread the CTAs in flight over every group's K/V.
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
                            uint32_t* __restrict__ srev, DevStatus* status) {
  const int h = blockIdx.x;
  const int W = (nb + 31) / 32;
  if (!CRISP_CHECK(h < static_cast<int>(gridDim.x), status, 0x510)) return;
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

// 32 bits of v starting at bit p (v holds `words` words).
__device__ __forceinline__ uint32_t window32(const uint32_t* v, int p, int words, DevStatus* status) {
  if (!CRISP_CHECK(p >= 0 && (p >> 5) + 1 < words, status, 0x511)) return 0u;
  return __funnelshift_r(v[p >> 5], v[(p >> 5) + 1], p & 31);
}

// One warp per row (h, qb), rows of a head consecutive; a lane per bitset
// word (strided).
constexpr int kMaskRowsPerCta = 8;
__global__ void mask_kernel(const uint8_t* __restrict__ route, const uint32_t* __restrict__ vbits,
                            const uint32_t* __restrict__ srev, const uint32_t* __restrict__ pebits, int hq, int nb,
                            int group, uint32_t* __restrict__ rowbits, int32_t* __restrict__ counts,
                            int32_t* __restrict__ order, DevStatus* status) {
  const int lane = threadIdx.x & 31;
  const int rowid = blockIdx.x * kMaskRowsPerCta + (threadIdx.x >> 5);
  if (rowid >= hq * nb) return;  // whole warps
  const int h = rowid / nb, qb = rowid % nb;
  const int W = (nb + 31) / 32, wq = qb >> 5;
  const bool vs = route[h] != 0;
  const uint32_t* V = vbits + static_cast<size_t>(h) * W;
  const uint32_t* R = srev + static_cast<size_t>(h) * (W + 2);
  const uint32_t* PE = pebits + (static_cast<size_t>(h) * nb + qb) * W;
  uint32_t* out = rowbits + (static_cast<size_t>(h) * nb + qb) * W;
  int cnt = 0;
  for (int w = lane; w < W; w += 32) {
    uint32_t word = 0;
    if (w <= wq) {
      if (vs) {
        const int p = nb - 1 - qb + 32 * w;
        word = V[w] | window32(R, p, W + 2, status) | window32(R, p + 1, W + 2, status);
      } else {
        word = PE[w];
      }
      if (w == wq && (qb & 31) != 31) word &= (1u << ((qb & 31) + 1)) - 1u;
    }
    out[w] = word;
    cnt += __popc(word);
  }
  const int total = warp_sum(cnt);
  if (lane == 0) {
    counts[static_cast<size_t>(h) * nb + qb] = total;
    const size_t g = h / group, j = h % group;
    const size_t o = (g * nb + (nb - 1 - qb)) * group + j;
    if (CRISP_CHECK(o < static_cast<size_t>(hq) * nb, status, 0x512)) order[o] = h * nb + qb;
  }
}

}  // namespace

cudaError_t launch_build_mask(const crisp_shape& s, const uint8_t* route, const uint32_t* vbits,
                              const uint32_t* sbits, const uint32_t* pebits, uint32_t* rowbits, int32_t* counts,
                              int32_t* order, char* ws, cudaStream_t st) {
  const ScratchLayout L = scratch_layout(s);
  const int nb = num_blocks(s.seq_len);
  auto* srev = reinterpret_cast<uint32_t*>(ws + L.srev);
  auto* status = reinterpret_cast<DevStatus*>(ws + L.status);
  srev_kernel<<<s.hq, 128, 0, st>>>(sbits, route, nb, srev, status);
  const int rows = s.hq * nb;
  mask_kernel<<<(rows + kMaskRowsPerCta - 1) / kMaskRowsPerCta, 32 * kMaskRowsPerCta, 0, st>>>(
      route, vbits, srev, pebits, s.hq, nb, s.hq / s.hkv, rowbits, counts, order, status);
  return cudaGetLastError();
}

}  // namespace crisp
