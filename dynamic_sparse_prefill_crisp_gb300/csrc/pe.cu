// A5 pooled attention estimate and A6 Pooled-Estimation block selection for
// the heads routed to PE (CRISP paper page on ai.info, "Overview" and
// "Methodology in Plain English": the PE path keeps FlexPrefill's pooled
// estimate and uses gamma = 0.95 coverage).
//
// A5: qbar_b / kbar_c = means over each block's tokens (128, or fewer in a
// short last block); pbar[b][c] = softmax
// over c <= b of scale * qbar_b . kbar_c (fp32; c > b stored as 0).
// A6: per row b, gamma coverage (or the noise floor) over Q32 quanta of pbar.
#include <cuda_bf16.h>

#include <algorithm>

#include "common.cuh"
#include "reduce.cuh"
#include "ptx.cuh"

namespace crisp {

namespace {

// Whether head y of the pooling list is pooled: y < hq is query head y (PE
// heads only), otherwise kv head y - hq (when any of its query heads is PE).
__device__ __forceinline__ bool pooled_head(const uint8_t* route, int hq, int G, int y) {
  if (y < hq) return route[y] == 0;
  bool any = false;
  for (int t = 0; t < G; ++t) any |= route[(y - hq) * G + t] == 0;
  return any;
}

// The first item index at or after `start` that is congruent to `id` modulo
// `stride`: where worker `id` of a grid-stride loop starts in a range of items.
__device__ __forceinline__ int64_t first_item(int64_t start, int64_t id, int64_t stride) {
  return start + (((id - start) % stride) + stride) % stride;
}

// The j-th head (0-based) whose route equals `want` (0: PE, 1: VS), found by
// the calling warp from ballots over 32 heads at a time.
__device__ __forceinline__ int nth_head(const uint8_t* route, int hq, bool want_vs, int j) {
  const int lane = threadIdx.x & 31;
  for (int base = 0; base < hq; base += 32) {
    const bool is_vs = base + lane < hq && route[base + lane] != 0;
    const uint32_t hits = __ballot_sync(0xffffffffu, base + lane < hq && is_vs == want_vs);
    const int cnt = __popc(hits);
    if (j < cnt) return base + static_cast<int>(__fns(hits, 0, j + 1));
    j -= cnt;
  }
  return hq;  // not reached for j below the head count
}

// Snake order: the k-th item of worker w of N is k*N + w in even rounds and
// k*N + N-1-w in odd ones, so that with items sorted by decreasing cost every
// worker gets a mix of long and short ones.
__device__ __forceinline__ int64_t snake_item(int64_t k, int64_t w, int64_t N) {
  return k * N + ((k & 1) ? N - 1 - w : w);
}

// Block means. Items (head y, block b), head-major: each CTA takes items
// blockIdx.x, blockIdx.x + gridDim.x, ... of the pooled heads only, so a
// layer with few PE heads launches no idle CTAs. Thread t sums dims
// 8(t % 16) .. 8(t % 16) + 7 of rows t / 16, t / 16 + 16, ... with 16-byte
// loads (eight in flight, the next item's issued before this item's sums
// are added); the 16 row groups are then added in order through shared
// memory.
__global__ void __launch_bounds__(256) pool_kernel(const __nv_bfloat16* __restrict__ q,
                                                   const __nv_bfloat16* __restrict__ k,
                                                   const uint8_t* __restrict__ route, int hq, int hkv, int n, int nb,
                                                   int64_t q_hs, int64_t q_ts, int64_t kv_hs, int64_t kv_ts,
                                                   float* __restrict__ qbar, float* __restrict__ kbar,
                                                   DevStatus* status) {
  __shared__ float red[16][kD + 4];
  const int G = hq / hkv;
  const int seg = threadIdx.x & 15, rg = threadIdx.x >> 4;
  for (int y = 0; y < hq + hkv; ++y) {
    if (!pooled_head(route, hq, G, y)) continue;
    const bool is_q = y < hq;
    const int64_t start = static_cast<int64_t>(y) * nb;
    const __nv_bfloat16* base = is_q ? q + static_cast<int64_t>(y) * q_hs : k + static_cast<int64_t>(y - hq) * kv_hs;
    const int64_t ts = is_q ? q_ts : kv_ts;  // elements, a multiple of 8
    // The next item's rows are requested before this item's sums go through
    // shared memory (eight 16-byte loads per thread in flight).
    uint4 raw[kB / 16];
    auto fetch = [&](int b) {
      const __nv_bfloat16* src = base + static_cast<int64_t>(b) * kB * ts;
      const int len = min(kB, n - b * kB);
#pragma unroll
      for (int j = 0; j < kB / 16; ++j) {
        const int r = rg + 16 * j;
        raw[j] = r < len ? *reinterpret_cast<const uint4*>(src + r * ts + 8 * seg) : make_uint4(0u, 0u, 0u, 0u);
      }
    };
    int64_t i = first_item(start, blockIdx.x, gridDim.x);
    if (i < start + nb) fetch(static_cast<int>(i - start));
    for (; i < start + nb; i += gridDim.x) {
      const int b = static_cast<int>(i - start);
      // (checking build) the block's tokens lie in [0, n)
      if (!CRISP_CHECK(b * kB < n, status, 0x410)) return;
      const int len = min(kB, n - b * kB);     // tokens of block b
      float acc[8] = {};
#pragma unroll
      for (int j = 0; j < kB / 16; ++j) {
        const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&raw[j]);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 v = __bfloat1622float2(h2[e]);
          acc[2 * e] += v.x;
          acc[2 * e + 1] += v.y;
        }
      }
      if (i + gridDim.x < start + nb) fetch(b + static_cast<int>(gridDim.x));
      __syncthreads();  // the previous item's sums have been read
#pragma unroll
      for (int e = 0; e < 8; ++e) red[rg][8 * seg + e] = acc[e];
      __syncthreads();
      if (threadIdx.x < kD) {
        float sum = 0.f;
#pragma unroll
        for (int g = 0; g < 16; ++g) sum += red[g][threadIdx.x];
        const size_t o = is_q ? (static_cast<size_t>(y) * nb + b) * kD : (static_cast<size_t>(y - hq) * nb + b) * kD;
        if (CRISP_CHECK(o + kD <= static_cast<size_t>(is_q ? hq : hkv) * nb * kD, status, 0x411))
          (is_q ? qbar : kbar)[o + threadIdx.x] = sum * (1.0f / static_cast<float>(len));  // exact for a whole block
      }
    }
  }
}

// Pooled logits in log2 units on the lower triangle (c <= b) of 128x128
// tiles: items (PE head h, tile t) with t over the T(T+1)/2 tiles (bt, ct <=
// bt), grid-stride like pool_kernel. Each of 256 threads computes 8x8 outputs
// (two 4x4 quadrants) from 16-deep slabs, double-buffered in shared memory:
// float4 reads of both operands, two fp32 fmas per instruction, the features
// added in ascending order. Entries above the diagonal are left to
// pooled_softmax, which writes whole rows.
constexpr int kPT = 128, kKS = 16;  // tile edge, depth of a shared-memory slab
__global__ void __launch_bounds__(256, 2) pooled_scores(const float* __restrict__ qbar, const float* __restrict__ kbar,
                                                        const uint8_t* __restrict__ route, int hq, int nb, int group,
                                                        float c_log2, float* __restrict__ pbar, DevStatus* status) {
  __shared__ __align__(16) float As[2][kKS][kPT + 4];
  __shared__ __align__(16) float Bs[2][kKS][kPT + 4];
  const int T = (nb + kPT - 1) / kPT;
  const int64_t per_head = static_cast<int64_t>(T) * (T + 1) / 2;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  for (int h = 0; h < hq; ++h) {
    if (route[h]) continue;
    const int64_t start = static_cast<int64_t>(h) * per_head;
    for (int64_t i = first_item(start, blockIdx.x, gridDim.x); i < start + per_head; i += gridDim.x) {
      const int t = static_cast<int>(i - start);
      int bt = static_cast<int>((sqrtf(8.0f * static_cast<float>(t) + 1.0f) - 1.0f) * 0.5f);
      while ((bt + 1) * (bt + 2) / 2 <= t) ++bt;
      while (bt * (bt + 1) / 2 > t) --bt;
      const int ct = t - bt * (bt + 1) / 2;
      // (checking build) the tile lies on or below the diagonal inside [0, nb)
      if (!CRISP_CHECK(bt < T && ct <= bt, status, 0x412)) return;
      float* out = pbar + static_cast<size_t>(h) * nb * nb;
      const float* A = qbar + static_cast<size_t>(h) * nb * kD;
      const float* Bm = kbar + static_cast<size_t>(h / group) * nb * kD;
      // Slab loads: thread f reads 4 consecutive features of row f / 4 (and of
      // row 64 + f / 4) of both operands with float4 loads.
      float4 ra[2], rb[2];
      auto load = [&](int d0) {
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int f = threadIdx.x + 256 * u, row = f >> 2, quad = f & 3;
          const int b = bt * kPT + row, c = ct * kPT + row;
          ra[u] = b < nb ? *reinterpret_cast<const float4*>(A + static_cast<size_t>(b) * kD + d0 + 4 * quad)
                         : make_float4(0.f, 0.f, 0.f, 0.f);
          rb[u] = c < nb ? *reinterpret_cast<const float4*>(Bm + static_cast<size_t>(c) * kD + d0 + 4 * quad)
                         : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      };
      auto store = [&](int buf) {
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int f = threadIdx.x + 256 * u, row = f >> 2, quad = f & 3;
          As[buf][4 * quad + 0][row] = ra[u].x;
          As[buf][4 * quad + 1][row] = ra[u].y;
          As[buf][4 * quad + 2][row] = ra[u].z;
          As[buf][4 * quad + 3][row] = ra[u].w;
          Bs[buf][4 * quad + 0][row] = rb[u].x;
          Bs[buf][4 * quad + 1][row] = rb[u].y;
          Bs[buf][4 * quad + 2][row] = rb[u].z;
          Bs[buf][4 * quad + 3][row] = rb[u].w;
        }
      };
      // Rows ty*4 .. +3 and 64 + ty*4 .. +3, columns tx*4 .. +3 and 64 + tx*4 .. +3.
      float acc[8][8] = {};
      __syncthreads();  // the previous item's last slab has been read
      load(0);
      store(0);
      __syncthreads();
      for (int sl = 0; sl < kD / kKS; ++sl) {
        const int buf = sl & 1;
        if (sl + 1 < kD / kKS) load((sl + 1) * kKS);
#pragma unroll
        for (int kk = 0; kk < kKS; ++kk) {
          const float4 a0 = *reinterpret_cast<const float4*>(&As[buf][kk][ty * 4]);
          const float4 a1 = *reinterpret_cast<const float4*>(&As[buf][kk][64 + ty * 4]);
          const float4 b0 = *reinterpret_cast<const float4*>(&Bs[buf][kk][tx * 4]);
          const float4 b1 = *reinterpret_cast<const float4*>(&Bs[buf][kk][64 + tx * 4]);
          const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
          const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
          for (int r = 0; r < 8; ++r)
#pragma unroll
            for (int j = 0; j < 8; j += 2)
              ptx::ffma2(acc[r][j], acc[r][j + 1], av[r], av[r], bv[j], bv[j + 1], acc[r][j], acc[r][j + 1]);
        }
        if (sl + 1 < kD / kKS) store(buf ^ 1);  // the other buffer was last read before the previous barrier
        __syncthreads();
      }
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        const int b = bt * kPT + (r < 4 ? ty * 4 + r : 64 + ty * 4 + r - 4);
        if (b >= nb) continue;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int c = ct * kPT + (j < 4 ? tx * 4 + j : 64 + tx * 4 + j - 4);
          if (c <= b) out[static_cast<size_t>(b) * nb + c] = acc[r][j] * c_log2;
        }
      }
    }
  }
}

// Row softmax over c <= b (base 2, logits already in log2 units) and zeros for
// b < c < nb; one warp per row of a PE head. Rows are numbered b descending
// (PE heads ascending within a b) and dealt to the warps in snake order.
__global__ void __launch_bounds__(256) pooled_softmax(const uint8_t* __restrict__ route, int hq, int nb,
                                                      float* __restrict__ pbar, DevStatus* status) {
  const int lane = threadIdx.x & 31;
  const int64_t wid = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  int n_pe = 0;
  for (int base = 0; base < hq; base += 32)
    n_pe += __popc(__ballot_sync(0xffffffffu, base + lane < hq && route[base + lane] == 0));
  const int64_t rows = static_cast<int64_t>(n_pe) * nb;
  for (int64_t k = 0;; ++k) {
    const int64_t r = snake_item(k, wid, nwarps);
    if (r >= rows) break;
    const int b = nb - 1 - static_cast<int>(r / n_pe);
    const int h = nth_head(route, hq, false, static_cast<int>(r % n_pe));
    if (!CRISP_CHECK(h < hq && b >= 0, status, 0x413)) return;
    float* z = pbar + (static_cast<size_t>(h) * nb + b) * nb;
    float mx = -INFINITY;
    for (int c = lane; c <= b; c += 32) mx = fmaxf(mx, z[c]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float sum = 0.f;
    for (int c = lane; c <= b; c += 32) sum += ptx::ex2_approx(z[c] - mx);
    sum = warp_sum(sum);
    const float inv = 1.0f / sum;
    for (int c = lane; c < nb; c += 32) z[c] = c <= b ? ptx::ex2_approx(z[c] - mx) * inv : 0.f;
  }
}

// A6: one warp per row (h, b), no block barrier. Warps are numbered PE rows
// first -- b descending (longest rows first), PE heads ascending within a b --
// then the VS heads' rows, which only get zeros; so the CTAs that search hold
// PE rows only. Each warp keeps its histogram (256 x 8 bytes) and its bitset
// (W words) in shared memory, and with kRowInShared its row of pbar (fp32,
// b + 1 entries) too; otherwise every pass reads the row again from global
// memory (L1/L2), which keeps more warps resident for long rows. Every pass
// re-forms the selection keys (quantum << 13 | 8191 - c) from the row. Bitset
// word i is the ballot of the lanes' keys 32i .. 32i + 31.
struct PeWarpLayout {
  int hist, chosen, vals, bytes;  // byte offsets inside one warp's slice
};
__host__ __device__ inline PeWarpLayout pe_warp_layout(int nb, bool row_in_shared) {
  PeWarpLayout L;
  L.hist = 0;
  L.chosen = 256 * 8;
  L.vals = L.chosen + (((nb + 31) / 32 + 3) / 4) * 16;
  L.bytes = L.vals + (row_in_shared ? ((nb + 3) / 4) * 16 : 0);
  return L;
}
constexpr int kPeRowsInShared = 1024;  // the longest row kept in shared memory

template <bool kRowInShared>
__global__ void __launch_bounds__(256, 4) select_pe_kernel(const float* __restrict__ pbar,
                                                           const uint8_t* __restrict__ route, int hq, int nb,
                                                           int pe_mode, uint32_t gamma_num, uint32_t gamma_den,
                                                           uint32_t alpha_num, uint32_t alpha_den, int kmin,
                                                           uint32_t* __restrict__ pebits, DevStatus* status) {
  extern __shared__ __align__(16) unsigned char pe_smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int n_pe = 0;
  for (int base = 0; base < hq; base += 32)
    n_pe += __popc(__ballot_sync(0xffffffffu, base + lane < hq && route[base + lane] == 0));
  const int W = (nb + 31) / 32;
  const PeWarpLayout L = pe_warp_layout(nb, kRowInShared);
  unsigned char* mine = pe_smem + static_cast<size_t>(warp) * L.bytes;
  auto* hist = reinterpret_cast<unsigned long long*>(mine + L.hist);
  auto* chosen = reinterpret_cast<uint32_t*>(mine + L.chosen);
  auto* vals = reinterpret_cast<float*>(mine + L.vals);
  const int row = blockIdx.x * (blockDim.x >> 5) + warp;
  if (row >= hq * nb) return;  // whole warps
  const bool vs_row = row >= n_pe * nb;
  const int j = vs_row ? row - n_pe * nb : row;
  const int nsel = vs_row ? hq - n_pe : n_pe;  // > 0 here
  const int b = vs_row ? j / nsel : nb - 1 - j / nsel;
  const int h = nth_head(route, hq, vs_row, j % nsel);
  // (checking build) the row lies inside pbar [hq][nb][nb] and pebits [hq][nb][W]
  if (!CRISP_CHECK(b >= 0 && b < nb && h < hq && W <= kMaxBlocks / 32, status, 0x414)) return;
  uint32_t* out = pebits + (static_cast<size_t>(h) * nb + b) * W;
  if (vs_row) {
    for (int w = lane; w < W; w += 32) out[w] = 0u;
    return;
  }
  const float* z = pbar + (static_cast<size_t>(h) * nb + b) * nb;
  const int len = b + 1;
  const bool gamma = pe_mode == CRISP_PE_GAMMA;
  // Pooled quanta are <= 2^33, so the keys fit in 48 bits and key >> 13 is
  // the quantum.
  uint64_t part = 0;
  for (int c = lane; c < len; c += 32) {
    const float p = z[c];
    if (kRowInShared) vals[c] = p;
    if (gamma || (c >= 1 && c <= b - 1)) part += q32(p);
  }
  const uint64_t T = warp_sum(part);
  __syncwarp();
  const float* row_vals = kRowInShared ? vals : z;
  auto mass_of = [&](int c) { return q32(row_vals[c]); };
  auto key_of = [&](int c) { return sel_key(mass_of(c), c); };
  auto mass_in_key = [](int, uint64_t key) { return key >> 13; };  // the quantum (< 2^43, kept whole)
  const int words = (len + 31) / 32;  // bitset words that can hold a set bit
  if (gamma) {
    const unsigned __int128 goal = static_cast<unsigned __int128>(gamma_num) * T;
    // Largest key x whose suffix mass reaches gamma of the row: the last
    // member of the shortest (mass desc, index asc) prefix.
    const uint64_t x = warp_radix_max_key(
        len, key_of, mass_in_key, [](int) { return true; },
        [&](unsigned long long f) { return static_cast<unsigned __int128>(gamma_den) * f >= goal; }, hist);
    for (int i = 0; i < words; ++i) {
      const int c = 32 * i + lane;
      const uint32_t word = __ballot_sync(0xffffffffu, c < len && key_of(c) >= x);
      if (lane == 0) chosen[i] = word;
    }
  } else {
    const int N = max(0, b - 1);  // candidates [1, b-1]; T is their mass
    const unsigned __int128 rhs = static_cast<unsigned __int128>(alpha_num) * T;
    for (int i = 0; i < words; ++i) {
      const int c = 32 * i + lane;
      const bool above = c >= 1 && c <= b - 1 &&
                         static_cast<unsigned __int128>(mass_of(c)) * static_cast<unsigned>(N) * alpha_den > rhs;
      const uint32_t word = __ballot_sync(0xffffffffu, above);
      if (lane == 0) chosen[i] = word;
    }
  }
  __syncwarp();
  if (lane == 0) {
    chosen[0] |= 1u;
    chosen[b >> 5] |= 1u << (b & 31);
  }
  __syncwarp();
  int pc = 0;
  for (int w = lane; w < words; w += 32) pc += __popc(chosen[w]);
  const int need = min(kmin, len) - warp_sum(pc);
  if (need > 0) {
    // k_min fill: the `need` unchosen blocks with the largest keys.
    auto unchosen = [&](int c) { return !((chosen[c >> 5] >> (c & 31)) & 1u); };
    const uint64_t x = warp_radix_max_key(
        len, key_of, [](int, uint64_t) { return 1ull; }, unchosen,
        [&](unsigned long long cnt) { return cnt >= static_cast<unsigned long long>(need); }, hist);
    for (int i = 0; i < words; ++i) {
      const int c = 32 * i + lane;
      const bool add = c < len && unchosen(c) && key_of(c) >= x;
      const uint32_t word = __ballot_sync(0xffffffffu, add);
      __syncwarp();  // every lane has read chosen[i] before lane 0 updates it
      if (lane == 0) chosen[i] |= word;
    }
    __syncwarp();
  }
  for (int w = lane; w < W; w += 32) out[w] = w < words ? chosen[w] : 0u;
}

}  // namespace

static int sm_count() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 152;
  return sms;
}

// CTAs of `threads` threads that stay resident on all SMs at once (at least
// one per SM), capped at `items`.
template <typename Kernel>
static unsigned resident_grid(Kernel kernel, int sms, int64_t items, int threads = 256, size_t smem = 0) {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem) != cudaSuccess || per_sm < 1)
    per_sm = 1;
  return static_cast<unsigned>(std::max<int64_t>(1, std::min(items, static_cast<int64_t>(sms) * per_sm)));
}

cudaError_t launch_pe_map(const crisp_shape& s, const void* q, const void* k, const uint8_t* route, float* pbar,
                          char* ws, cudaStream_t st) {
  const ScratchLayout L = scratch_layout(s);
  const int nb = num_blocks(s.seq_len);
  auto* qbar = reinterpret_cast<float*>(ws + L.qbar);
  auto* kbar = reinterpret_cast<float*>(ws + L.kbar);
  auto* status = reinterpret_cast<DevStatus*>(ws + L.status);
  // Grids of resident CTAs, each looping over its share of the PE heads'
  // items (VS heads cost a route read), so a layer with few PE heads launches
  // no idle CTAs.
  const int sms = sm_count();
  const int64_t pool_items = static_cast<int64_t>(s.hq + s.hkv) * nb;
  pool_kernel<<<resident_grid(pool_kernel, sms, pool_items), 256, 0, st>>>(
      static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k), route, s.hq, s.hkv, s.seq_len, nb,
      s.q_head_stride, s.q_tok_stride, s.kv_head_stride, s.kv_tok_stride, qbar, kbar, status);
  const int64_t T = (nb + kPT - 1) / kPT;
  const int64_t tiles = static_cast<int64_t>(s.hq) * T * (T + 1) / 2;
  pooled_scores<<<resident_grid(pooled_scores, sms, tiles), 256, 0, st>>>(
      qbar, kbar, route, s.hq, nb, s.hq / s.hkv, s.scale * 1.4426950408889634f, pbar, status);
  const int64_t rows = static_cast<int64_t>(s.hq) * nb;
  pooled_softmax<<<resident_grid(pooled_softmax, sms, (rows + 7) / 8), 256, 0, st>>>(route, s.hq, nb, pbar, status);
  return cudaGetLastError();
}

cudaError_t launch_select_pe(const crisp_shape& s, const crisp_params& p, const float* pbar, const uint8_t* route,
                             uint32_t* pebits, DevStatus* status, cudaStream_t st) {
  const int nb = num_blocks(s.seq_len);
  // One warp per row, 8 rows per CTA. Rows up to kPeRowsInShared entries stay
  // in shared memory (50 KB per CTA at most: four CTAs per SM); longer rows
  // are read again from global memory in each pass.
  const bool in_shared = nb <= kPeRowsInShared;
  const int smem = 8 * pe_warp_layout(nb, in_shared).bytes;
  auto kernel = in_shared ? select_pe_kernel<true> : select_pe_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int64_t rows = static_cast<int64_t>(s.hq) * nb;
  kernel<<<static_cast<unsigned>((rows + 7) / 8), 256, smem, st>>>(pbar, route, s.hq, nb, p.pe_mode, p.gamma_num,
                                                                   p.gamma_den, p.alpha_num, p.alpha_den,
                                                                   p.kmin_blocks, pebits, status);
  return cudaGetLastError();
}

}  // namespace crisp
