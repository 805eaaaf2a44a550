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

#include "common.cuh"
#include "reduce.cuh"
#include "ptx.cuh"

namespace crisp {

namespace {

// Block means. grid (nb, hq + hkv): y < hq pools query head y (PE heads
// only), otherwise kv head y - hq (when any of its query heads is PE).
__global__ void __launch_bounds__(256) pool_kernel(const __nv_bfloat162* __restrict__ q,
                                                   const __nv_bfloat162* __restrict__ k, const uint8_t* __restrict__ route,
                                                   int hq, int hkv, int n, int64_t q_hs, int64_t q_ts, int64_t kv_hs,
                                                   int64_t kv_ts, float* __restrict__ qbar, float* __restrict__ kbar,
                                                   DevStatus* status) {
  __shared__ float2 red[4][64];
  const int b = blockIdx.x, y = blockIdx.y, nb = gridDim.x;
  // (checking build) the block's tokens lie in [0, n) and the head in q or k
  if (!CRISP_CHECK(b * kB < n && y < hq + hkv, status, 0x410)) return;
  const int G = hq / hkv;
  const bool is_q = y < hq;
  if (is_q) {
    if (route[y]) return;
  } else {
    bool any = false;
    for (int t = 0; t < G; ++t) any |= route[(y - hq) * G + t] == 0;
    if (!any) return;
  }
  const int pair = threadIdx.x & 63, rg = threadIdx.x >> 6;
  // strides are in bf16 elements; the pointers here are bf16x2 (two elements)
  const __nv_bfloat162* src = is_q ? q + (static_cast<int64_t>(y) * q_hs + static_cast<int64_t>(b) * kB * q_ts) / 2
                                   : k + (static_cast<int64_t>(y - hq) * kv_hs + static_cast<int64_t>(b) * kB * kv_ts) / 2;
  const int64_t ts = (is_q ? q_ts : kv_ts) / 2;
  const int len = min(kB, n - b * kB);  // tokens of block b
  float2 acc = make_float2(0.f, 0.f);
  for (int r = rg * 32; r < min(rg * 32 + 32, len); ++r) {
    const float2 v = __bfloat1622float2(src[r * ts + pair]);
    acc.x += v.x;
    acc.y += v.y;
  }
  red[rg][pair] = acc;
  __syncthreads();
  if (rg == 0) {
    float2 s = red[0][pair];
    for (int t = 1; t < 4; ++t) {
      s.x += red[t][pair].x;
      s.y += red[t][pair].y;
    }
    const size_t o = is_q ? (static_cast<size_t>(y) * nb + b) * kD : (static_cast<size_t>(y - hq) * nb + b) * kD;
    if (!CRISP_CHECK(o + kD <= static_cast<size_t>(is_q ? hq : hkv) * nb * kD, status, 0x411)) return;
    float* dst = (is_q ? qbar : kbar) + o;
    const float inv = 1.0f / static_cast<float>(len);  // exact for a whole block
    dst[2 * pair] = s.x * inv;
    dst[2 * pair + 1] = s.y * inv;
  }
}

// Pooled logits in log2 units, 64x64 tiles: grid (tiles, tiles, hq); each of
// 256 threads computes 4x4 outputs. Tiles above the diagonal are zero-filled.
constexpr int kPT = 64;
__global__ void __launch_bounds__(256) pooled_scores(const float* __restrict__ qbar, const float* __restrict__ kbar,
                                                     const uint8_t* __restrict__ route, int nb, int group,
                                                     float c_log2, float* __restrict__ pbar, DevStatus* status) {
  __shared__ float As[32][kPT + 1];
  __shared__ float Bs[32][kPT + 1];
  const int bt = blockIdx.y, ct = blockIdx.x, h = blockIdx.z;
  // (checking build) the tile's rows and columns start inside [0, nb)
  if (!CRISP_CHECK(bt * kPT < nb && ct * kPT < nb, status, 0x412)) return;
  if (route[h]) return;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float* out = pbar + static_cast<size_t>(h) * nb * nb;
  if (ct > bt) {
    for (int e = threadIdx.x; e < kPT * kPT; e += 256) {
      const int b = bt * kPT + e / kPT, c = ct * kPT + e % kPT;
      if (b < nb && c < nb) out[static_cast<size_t>(b) * nb + c] = 0.f;
    }
    return;
  }
  const float* A = qbar + static_cast<size_t>(h) * nb * kD;
  const float* Bm = kbar + static_cast<size_t>(h / group) * nb * kD;
  float acc[4][4] = {};
  for (int d0 = 0; d0 < kD; d0 += 32) {
    for (int e = threadIdx.x; e < 32 * kPT; e += 256) {
      const int row = e / 32, dd = e % 32;
      const int b = bt * kPT + row, c = ct * kPT + row;
      As[dd][row] = b < nb ? A[static_cast<size_t>(b) * kD + d0 + dd] : 0.f;
      Bs[dd][row] = c < nb ? Bm[static_cast<size_t>(c) * kD + d0 + dd] : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int dd = 0; dd < 32; ++dd) {
      float a[4], bb[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        a[i] = As[dd][ty * 4 + i];
        bb[i] = Bs[dd][tx * 4 + i];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] += a[i] * bb[j];
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int b = bt * kPT + ty * 4 + i;
    if (b >= nb) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int c = ct * kPT + tx * 4 + j;
      if (c < nb) out[static_cast<size_t>(b) * nb + c] = c <= b ? acc[i][j] * c_log2 : 0.f;
    }
  }
}

// Row softmax over c <= b (base 2, logits already in log2 units), one warp per row.
__global__ void pooled_softmax(const uint8_t* __restrict__ route, int hq, int nb, float* __restrict__ pbar,
                               DevStatus* status) {
  const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= hq * nb) return;
  const int h = row / nb, b = row % nb;
  if (!CRISP_CHECK(static_cast<size_t>(row) * nb + b < static_cast<size_t>(hq) * nb * nb, status, 0x413)) return;
  if (route[h]) return;
  float* z = pbar + static_cast<size_t>(row) * nb;
  float mx = -INFINITY;
  for (int c = lane; c <= b; c += 32) mx = fmaxf(mx, z[c]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  float sum = 0.f;
  for (int c = lane; c <= b; c += 32) sum += ptx::ex2_approx(z[c] - mx);
  sum = warp_sum(sum);
  const float inv = 1.0f / sum;
  for (int c = lane; c <= b; c += 32) z[c] = ptx::ex2_approx(z[c] - mx) * inv;
}

// A6: one CTA per head and `rows` consecutive query blocks b (rows of one
// head have similar lengths; a VS head's CTA only writes empty rows, so long
// sequences group rows to launch fewer of those). Each row's selection keys
// (quantum << 13 | 8191 - c) are formed once into shared memory (nb x 8
// bytes, dynamic); every search pass then reads them from there.
constexpr int kPeThreads = 256;
__global__ void __launch_bounds__(kPeThreads) select_pe_kernel(const float* __restrict__ pbar,
                                                               const uint8_t* __restrict__ route, int nb,
                                                               int pe_mode, uint32_t gamma_num, uint32_t gamma_den,
                                                               uint32_t alpha_num, uint32_t alpha_den, int kmin,
                                                               int rows, uint32_t* __restrict__ pebits,
                                                               DevStatus* status) {
  extern __shared__ unsigned long long keys[];  // [b + 1]
  __shared__ uint32_t chosen[kMaxBlocks / 32];
  __shared__ uint64_t scratch64[32];
  __shared__ int scratch32[32];
  __shared__ unsigned long long hist[256], bcast[4];
  const int h = blockIdx.y;
  const int W = (nb + 31) / 32;
  const int b_end = min(nb, (static_cast<int>(blockIdx.x) + 1) * rows);
  // (checking build) the shared bitset holds a row; the rows [.., b_end) of
  // head h lie inside pbar [hq][nb][nb] and pebits [hq][nb][W]
  if (!CRISP_CHECK(W <= kMaxBlocks / 32 && h < static_cast<int>(gridDim.y) && b_end <= nb, status, 0x414)) return;
  if (route[h]) {
    for (int i = blockIdx.x * rows * W + threadIdx.x; i < b_end * W; i += blockDim.x)
      pebits[static_cast<size_t>(h) * nb * W + i] = 0u;
    return;
  }
  for (int b = blockIdx.x * rows; b < b_end; ++b) {
    uint32_t* out = pebits + (static_cast<size_t>(h) * nb + b) * W;
    __syncthreads();  // the previous row's reads of keys and chosen are done
    for (int w = threadIdx.x; w < W; w += blockDim.x) chosen[w] = 0u;
    const float* z = pbar + (static_cast<size_t>(h) * nb + b) * nb;
    // Pooled quanta are <= 2^33, so the keys fit in 48 bits and key >> 13 is
    // the quantum.
    uint64_t part = 0;
    for (int c = threadIdx.x; c <= b; c += blockDim.x) {
      const uint64_t m = q32(z[c]);
      keys[c] = sel_key(m, c);
      if (pe_mode == CRISP_PE_GAMMA || (c >= 1 && c <= b - 1)) part += m;
    }
    const uint64_t T = block_sum(part, scratch64);  // also orders the key writes before the reads below
    auto key_of = [&](int c) { return static_cast<uint64_t>(keys[c]); };
    if (pe_mode == CRISP_PE_GAMMA) {
      const unsigned __int128 goal = static_cast<unsigned __int128>(gamma_num) * T;
      // Largest key x whose suffix mass reaches gamma of the row: the last
      // member of the shortest (mass desc, index asc) prefix.
      const uint64_t x = radix_max_key(
          b + 1, key_of, [&](int c) { return keys[c] >> 13; }, [](int) { return true; },
          [&](unsigned long long f) { return static_cast<unsigned __int128>(gamma_den) * f >= goal; }, hist, bcast);
      for (int c = threadIdx.x; c <= b; c += blockDim.x)
        if (keys[c] >= x) atomicOr(&chosen[c >> 5], 1u << (c & 31));
      __syncthreads();
      if (threadIdx.x == 0) {
        chosen[0] |= 1u;
        chosen[b >> 5] |= 1u << (b & 31);
      }
    } else {
      const int N = max(0, b - 1);  // candidates [1, b-1]; T is their mass
      const unsigned __int128 rhs = static_cast<unsigned __int128>(alpha_num) * T;
      for (int c = 1 + threadIdx.x; c <= b - 1; c += blockDim.x) {
        const unsigned __int128 lhs = static_cast<unsigned __int128>(keys[c] >> 13) * static_cast<unsigned>(N) * alpha_den;
        if (lhs > rhs) atomicOr(&chosen[c >> 5], 1u << (c & 31));
      }
      __syncthreads();
      if (threadIdx.x == 0) {
        chosen[0] |= 1u;
        chosen[b >> 5] |= 1u << (b & 31);
      }
    }
    __syncthreads();
    int pc = 0;
    for (int w = threadIdx.x; w < W; w += blockDim.x) pc += __popc(chosen[w]);
    const int count = block_sum(pc, scratch32);
    const int need = min(kmin, b + 1) - count;
    if (need > 0) {
      // k_min fill: the `need` unchosen blocks with the largest keys.
      auto unchosen = [&](int c) { return !((chosen[c >> 5] >> (c & 31)) & 1u); };
      const uint64_t x = radix_max_key(
          b + 1, key_of, [](int) { return 1ull; }, unchosen,
          [&](unsigned long long cnt) { return cnt >= static_cast<unsigned long long>(need); }, hist, bcast);
      __syncthreads();
      for (int c = threadIdx.x; c <= b; c += blockDim.x)
        if (unchosen(c) && keys[c] >= x) atomicOr(&chosen[c >> 5], 1u << (c & 31));
    }
    __syncthreads();
    for (int w = threadIdx.x; w < W; w += blockDim.x) out[w] = chosen[w];
  }
}

}  // namespace

cudaError_t launch_pe_map(const crisp_shape& s, const void* q, const void* k, const uint8_t* route, float* pbar,
                          char* ws, cudaStream_t st) {
  const ScratchLayout L = scratch_layout(s);
  const int nb = num_blocks(s.seq_len);
  auto* qbar = reinterpret_cast<float*>(ws + L.qbar);
  auto* kbar = reinterpret_cast<float*>(ws + L.kbar);
  pool_kernel<<<dim3(nb, s.hq + s.hkv), 256, 0, st>>>(static_cast<const __nv_bfloat162*>(q),
                                                      static_cast<const __nv_bfloat162*>(k), route, s.hq, s.hkv,
                                                      s.seq_len, s.q_head_stride, s.q_tok_stride, s.kv_head_stride,
                                                      s.kv_tok_stride, qbar, kbar, reinterpret_cast<DevStatus*>(ws + L.status));
  const int tiles = (nb + kPT - 1) / kPT;
  auto* status = reinterpret_cast<DevStatus*>(ws + L.status);
  pooled_scores<<<dim3(tiles, tiles, s.hq), 256, 0, st>>>(qbar, kbar, route, nb, s.hq / s.hkv,
                                                          s.scale * 1.4426950408889634f, pbar, status);
  const int rows = s.hq * nb;
  pooled_softmax<<<(rows + 7) / 8, 256, 0, st>>>(route, s.hq, nb, pbar, status);
  return cudaGetLastError();
}

cudaError_t launch_select_pe(const crisp_shape& s, const crisp_params& p, const float* pbar, const uint8_t* route,
                             uint32_t* pebits, DevStatus* status, cudaStream_t st) {
  const int nb = num_blocks(s.seq_len);
  const size_t key_bytes = static_cast<size_t>(nb) * sizeof(unsigned long long);  // <= 64 KB (nb <= 8192)
  cudaError_t e = cudaFuncSetAttribute(select_pe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(key_bytes));
  if (e != cudaSuccess) return e;
  // Four rows per CTA from 1024 blocks (measured: 512k with no PE heads
  // 0.13 -> 0.03 ms); one below, where a CTA per row keeps more in flight.
  const int rows = nb >= 1024 ? 4 : 1;
  select_pe_kernel<<<dim3((nb + rows - 1) / rows, s.hq), kPeThreads, key_bytes, st>>>(
      pbar, route, nb, p.pe_mode, p.gamma_num, p.gamma_den, p.alpha_num, p.alpha_den, p.kmin_blocks, rows, pebits,
      status);
  return cudaGetLastError();
}

}  // namespace crisp
