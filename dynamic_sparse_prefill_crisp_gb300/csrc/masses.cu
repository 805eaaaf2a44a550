// A3 block masses, A2 C_struct routing and A4 Vertical-Slash noise-floor
// selection (CRISP paper page on ai.info, "Key Contributions" 2 and
// "Methodology in Plain English"; ai-feeds page, "方法").
//
// Every mass is an integer sum of Q32 quanta q(p) = round-half-even(p * 2^32),
// so the result does not depend on the order of the reduction and matches an
// element-by-element statement bit for bit.
#include "common.cuh"
#include "reduce.cuh"

namespace crisp {

namespace {

constexpr int kMassThreads = 256;

// One CTA per 128x128 tile (key block c, head h) of the proxy map (row
// stride ld floats). Thread t reads columns 4*(t%32)..+3 of rows
// 16*(t/32)..+15 (coalesced 512-byte rows) and sums the quanta by slash
// block. Row r is token i = n-128+r = (nb-2)*128 + tail + r and column jj
// of the tile is token j = 128c + jj, so the diagonal offset i - j falls in
// slash block nb-2-c + floor((tail + r - jj) / 128):
//   nb-1-c  where jj - r <= tail - 128   (the lower triangle when 128 | n)
//   nb-2-c  where tail - 128 < jj - r <= tail
//   nb-3-c  where jj - r > tail          (empty when 128 | n)
// The whole tile is the vertical mass of block c. Tile nb-2 also sums its
// columns jj >= tail, the part of the recency columns [n-128, n) that lies
// before the (short) last block. kRagged = false fixes tail = 128 (128
// divides n), where the third band and the recency part fold away.
template <bool kRagged>
__global__ void __launch_bounds__(kMassThreads) mass_tiles(const float* __restrict__ pmap, int64_t ld, int tail_arg,
                                                           uint64_t* __restrict__ vmass,
                                                           uint64_t* __restrict__ lower,
                                                           uint64_t* __restrict__ upper,
                                                           uint64_t* __restrict__ upper2,
                                                           uint64_t* __restrict__ rec, DevStatus* status) {
  __shared__ uint64_t red[4][kMassThreads / 32];
  const int tail = kRagged ? tail_arg : kB;
  const int c = blockIdx.x, h = blockIdx.y, nb = gridDim.x;
  const int cq = threadIdx.x & 31, rg = threadIdx.x >> 5;
  const size_t off = static_cast<size_t>(h) * kB * ld + static_cast<size_t>(c) * kB + cq * 4;
  // (checking build) the tile must lie inside the map [hq][128][ld]
  const bool tile_ok = CRISP_CHECK(off + static_cast<size_t>(kB - 1) * ld + 4 <= static_cast<size_t>(gridDim.y) * kB * ld &&
                                       static_cast<size_t>(c) * kB + kB <= static_cast<size_t>(ld),
                                   status, 0x310);
  const float* base = pmap + off;
  float4 p[16];
#pragma unroll
  for (int k = 0; k < 16; ++k)
    p[k] = tile_ok ? __ldcs(reinterpret_cast<const float4*>(base + static_cast<size_t>(rg * 16 + k) * ld))
                   : make_float4(0.f, 0.f, 0.f, 0.f);
  // Quanta below 2^23 (nearly all of them) are summed in 32 bits: 64 of them
  // stay below 2^29. Larger ones go to 64-bit sums.
  uint32_t all32 = 0, lo32 = 0, hi32 = 0;
  uint64_t all64 = 0, lo64 = 0, hi64 = 0;
  const int jj = cq * 4, b_lo = tail - kB, b_hi = tail;
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const int r = rg * 16 + k;
    const float x[4] = {p[k].x * 4294967296.0f, p[k].y * 4294967296.0f, p[k].z * 4294967296.0f,
                        p[k].w * 4294967296.0f};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int dj = jj + e - r;
      const bool in_lo = dj <= b_lo, in_hi = kRagged && dj > b_hi;
      if (x[e] < kTwo23) {
        const uint32_t f = q32_small(x[e]);
        all32 += f;
        lo32 += in_lo ? f : 0u;
        hi32 += in_hi ? f : 0u;
      } else {
        const uint64_t f = q32_large(x[e]);
        all64 += f;
        lo64 += in_lo ? f : 0ull;
        hi64 += in_hi ? f : 0ull;
      }
    }
  }
  const bool rec_tile = c == nb - 2 && tail < kB;
  uint64_t rs = 0;
  if (rec_tile) {
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const float x[4] = {p[k].x * 4294967296.0f, p[k].y * 4294967296.0f, p[k].z * 4294967296.0f,
                          p[k].w * 4294967296.0f};
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (jj + e >= tail) rs += x[e] < kTwo23 ? static_cast<uint64_t>(q32_small(x[e])) : q32_large(x[e]);
    }
  }
  uint64_t v[4] = {all64 + all32, lo64 + lo32, hi64 + hi32, rs};
#pragma unroll
  for (int t = 0; t < 4; ++t) v[t] = warp_sum(v[t]);
  if ((threadIdx.x & 31) == 0)
    for (int t = 0; t < 4; ++t) red[t][threadIdx.x >> 5] = v[t];
  __syncthreads();
  if (threadIdx.x == 0) {
    uint64_t sum[4] = {0, 0, 0, 0};
    for (int t = 0; t < 4; ++t)
      for (int w = 0; w < kMassThreads / 32; ++w) sum[t] += red[t][w];
    const size_t idx = static_cast<size_t>(h) * nb + c;
    if (CRISP_CHECK(idx < static_cast<size_t>(gridDim.y) * nb, status, 0x311)) {
      vmass[idx] = sum[0];
      lower[idx] = sum[1];
      upper[idx] = sum[0] - sum[1] - sum[2];
      upper2[idx] = sum[2];
    }
    if (rec_tile) rec[h] = sum[3];
  }
}

// smass[h][s] = lower[nb-1-s] + upper[nb-2-s] + upper2[nb-3-s], each over
// tiles >= 1: tile 0 holds the sink columns j < 128, which the slash
// direction leaves out. Thread s = 0 also forms the recency mass, the
// columns [n-128, n): the last block plus, when it is short, the rest of
// tile nb-2.
__global__ void assemble_slash(const uint64_t* __restrict__ vmass, const uint64_t* __restrict__ lower,
                               const uint64_t* __restrict__ upper, const uint64_t* __restrict__ upper2,
                               const uint64_t* __restrict__ rec, int nb, int tail, uint64_t* __restrict__ smass,
                               uint64_t* __restrict__ rmass, DevStatus* status) {
  const int h = blockIdx.y;
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  if (s >= nb) return;
  const size_t o = static_cast<size_t>(h) * nb;
  const int c1 = nb - 1 - s, c2 = nb - 2 - s, c3 = nb - 3 - s;
  if (!CRISP_CHECK(o + s < static_cast<size_t>(gridDim.y) * nb && c1 < nb, status, 0x312)) return;
  smass[o + s] = (c1 >= 1 ? lower[o + c1] : 0ull) + (c2 >= 1 ? upper[o + c2] : 0ull) +
                 (c3 >= 1 ? upper2[o + c3] : 0ull);
  if (s == 0) rmass[h] = vmass[o + nb - 1] + (tail < kB ? rec[h] : 0ull);
}

// C_struct = vmass[0] + rmass (columns [0,128) and [n-128,n), disjoint for
// n >= 256), total = sum of vmass; VS iff tau_den * C_struct >= tau_num * total.
__global__ void route_kernel(const uint64_t* __restrict__ vmass, const uint64_t* __restrict__ rmass, int nb,
                             uint32_t tau_num, uint32_t tau_den, uint64_t* __restrict__ cstruct,
                             uint64_t* __restrict__ total, uint8_t* __restrict__ route, DevStatus* status) {
  __shared__ uint64_t scratch[32];
  const int h = blockIdx.x;
  const uint64_t* v = vmass + static_cast<size_t>(h) * nb;
  uint64_t s = 0;
  for (int c = threadIdx.x; c < nb; c += blockDim.x)
    if (CRISP_CHECK(static_cast<size_t>(h) * nb + c < static_cast<size_t>(gridDim.x) * nb, status, 0x313)) s += v[c];
  const uint64_t T = block_sum(s, scratch);
  if (threadIdx.x == 0) {
    const uint64_t S = v[0] + rmass[h];
    cstruct[h] = S;
    total[h] = T;
    route[h] = static_cast<unsigned __int128>(tau_den) * S >= static_cast<unsigned __int128>(tau_num) * T ? 1 : 0;
  }
}

// C_struct from the proxy map itself, for any slice widths: one CTA per
// 128x128 tile (column block c, head h), 16-byte streaming loads as in
// mass_tiles; the tile's quanta go to the head's total and, for columns j in
// [0, sink) U [n - recency, n), to its slice sum (both zeroed beforehand;
// integer atomics, so the order of the tiles does not matter).
__global__ void __launch_bounds__(kMassThreads) cstruct_tiles(const float* __restrict__ pmap, int64_t ld, int n,
                                                              int sink, int recency, uint64_t* __restrict__ cstruct,
                                                              uint64_t* __restrict__ total, DevStatus* status) {
  __shared__ uint64_t red[2][kMassThreads / 32];
  const int c = blockIdx.x, h = blockIdx.y;
  const int cq = threadIdx.x & 31, rg = threadIdx.x >> 5;
  const size_t off = static_cast<size_t>(h) * kB * ld + static_cast<size_t>(c) * kB + cq * 4;
  const bool tile_ok = CRISP_CHECK(off + static_cast<size_t>(kB - 1) * ld + 4 <= static_cast<size_t>(gridDim.y) * kB * ld &&
                                       static_cast<size_t>(c) * kB + kB <= static_cast<size_t>(ld),
                                   status, 0x314);
  const float* base = pmap + off;
  const int j0 = c * kB + cq * 4;  // key token of this thread's first column
  bool in_slice[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) in_slice[e] = j0 + e < sink || (j0 + e >= n - recency && j0 + e < n);
  float4 p[16];
#pragma unroll
  for (int k = 0; k < 16; ++k)
    p[k] = tile_ok ? __ldcs(reinterpret_cast<const float4*>(base + static_cast<size_t>(rg * 16 + k) * ld))
                   : make_float4(0.f, 0.f, 0.f, 0.f);
  // As in mass_tiles: quanta below 2^23 summed in 32 bits (64 stay below 2^29).
  uint32_t all32 = 0, sl32 = 0;
  uint64_t all64 = 0, sl64 = 0;
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const float x[4] = {p[k].x * 4294967296.0f, p[k].y * 4294967296.0f, p[k].z * 4294967296.0f,
                        p[k].w * 4294967296.0f};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (x[e] < kTwo23) {
        const uint32_t f = q32_small(x[e]);
        all32 += f;
        sl32 += in_slice[e] ? f : 0u;
      } else {
        const uint64_t f = q32_large(x[e]);
        all64 += f;
        sl64 += in_slice[e] ? f : 0ull;
      }
    }
  }
  const uint64_t all = warp_sum(all64 + all32), sl = warp_sum(sl64 + sl32);
  if (cq == 0) {
    red[0][rg] = all;
    red[1][rg] = sl;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    uint64_t a = 0, b = 0;
    for (int w = 0; w < kMassThreads / 32; ++w) {
      a += red[0][w];
      b += red[1][w];
    }
    atomicAdd(reinterpret_cast<unsigned long long*>(total + h), static_cast<unsigned long long>(a));
    if (b != 0) atomicAdd(reinterpret_cast<unsigned long long*>(cstruct + h), static_cast<unsigned long long>(b));
  }
}

// VS iff tau_den * C_struct >= tau_num * total, one thread per head.
__global__ void route_decide(const uint64_t* __restrict__ cstruct, const uint64_t* __restrict__ total, int hq,
                             uint32_t tau_num, uint32_t tau_den, uint8_t* __restrict__ route) {
  const int h = blockIdx.x * blockDim.x + threadIdx.x;
  if (h >= hq) return;
  route[h] = static_cast<unsigned __int128>(tau_den) * cstruct[h] >= static_cast<unsigned __int128>(tau_num) * total[h]
                 ? 1
                 : 0;
}

// A4 for one (head, direction): direction 0 = vertical (always keeps {0,
// nb-1}), 1 = slash (always keeps {0}). Noise floor (CRISP): candidates
// [1, nb-2] above alpha times their mean. Cumulative coverage (FlexPrefill,
// the comparator): candidates [0, nb-1], the shortest (mass desc, index asc)
// prefix reaching gamma of their total. Both then fill to k_min.
constexpr int kSelThreads = 512;
__global__ void __launch_bounds__(kSelThreads) select_vs_kernel(const uint64_t* __restrict__ vmass,
                                                                const uint64_t* __restrict__ smass,
                                                                const uint8_t* __restrict__ route, int nb,
                                                                uint32_t alpha_num, uint32_t alpha_den, int kmin,
                                                                int vs_mode, uint32_t gamma_num, uint32_t gamma_den,
                                                                uint32_t* __restrict__ vbits,
                                                                uint32_t* __restrict__ sbits, DevStatus* status) {
  __shared__ uint32_t chosen[kMaxBlocks / 32];
  __shared__ uint64_t scratch64[32];
  __shared__ int scratch32[32];
  const int h = blockIdx.x, dir = blockIdx.y;
  const int W = (nb + 31) / 32;
  // (checking build) the bit rows fit the shared bitset; the head's mass rows
  // [h*nb, h*nb + nb) and bit words [h*W, h*W + W) lie inside [hq][nb] / [hq][W]
  if (!CRISP_CHECK(W <= kMaxBlocks / 32 && h < static_cast<int>(gridDim.x), status, 0x315)) return;
  uint32_t* out = (dir == 0 ? vbits : sbits) + static_cast<size_t>(h) * W;
  for (int w = threadIdx.x; w < W; w += blockDim.x) chosen[w] = 0u;
  __syncthreads();
  if (!route[h]) {
    for (int w = threadIdx.x; w < W; w += blockDim.x) out[w] = 0u;
    return;
  }
  const uint64_t* m = (dir == 0 ? vmass : smass) + static_cast<size_t>(h) * nb;
  const bool coverage = vs_mode == CRISP_VS_GAMMA;
  const int c_lo = coverage ? 0 : 1, c_hi = coverage ? nb - 1 : nb - 2;  // candidates [c_lo, c_hi]
  const int N = max(0, c_hi - c_lo + 1);
  const int nforced = (dir == 0 && nb >= 2) ? 2 : 1;
  if (threadIdx.x == 0) {
    chosen[0] |= 1u;
    if (dir == 0) chosen[(nb - 1) >> 5] |= 1u << ((nb - 1) & 31);
  }
  uint64_t part = 0;
  for (int c = c_lo + threadIdx.x; c <= c_hi; c += blockDim.x) part += m[c];
  const uint64_t sum = block_sum(part, scratch64);
  if (coverage) {
    // Largest key x whose suffix mass reaches gamma of the total: the last
    // member of the shortest (mass desc, index asc) prefix.
    const unsigned __int128 goal = static_cast<unsigned __int128>(gamma_num) * sum;
    uint64_t x = 0;
    for (int bit = kKeyBits - 1; bit >= 0; --bit) {
      const uint64_t cand = x | (1ull << bit);
      uint64_t f = 0;
      for (int c = c_lo + threadIdx.x; c <= c_hi; c += blockDim.x)
        if (sel_key(m[c], c) >= cand) f += m[c];
      if (static_cast<unsigned __int128>(gamma_den) * block_sum(f, scratch64) >= goal) x = cand;
    }
    for (int c = c_lo + threadIdx.x; c <= c_hi; c += blockDim.x)
      if (sel_key(m[c], c) >= x) atomicOr(&chosen[c >> 5], 1u << (c & 31));
  } else if (N > 0) {
    const unsigned __int128 rhs = static_cast<unsigned __int128>(alpha_num) * sum;
    for (int c = c_lo + threadIdx.x; c <= c_hi; c += blockDim.x) {
      const unsigned __int128 lhs = static_cast<unsigned __int128>(m[c]) * static_cast<unsigned>(N) * alpha_den;
      if (lhs > rhs) atomicOr(&chosen[c >> 5], 1u << (c & 31));
    }
  }
  __syncthreads();
  int pc = 0;
  for (int w = threadIdx.x; w < W; w += blockDim.x) pc += __popc(chosen[w]);
  const int count = block_sum(pc, scratch32);
  const int target = min(kmin, coverage ? nb : nforced + N);
  const int need = target - count;
  if (need > 0) {
    // Largest key x with #{unchosen candidates: key >= x} >= need; keys are
    // unique, so exactly `need` candidates reach it: the (mass desc, index
    // asc) order of the k_min fill.
    uint64_t x = 0;
    for (int bit = kKeyBits - 1; bit >= 0; --bit) {
      const uint64_t cand = x | (1ull << bit);
      int cnt = 0;
      for (int c = c_lo + threadIdx.x; c <= c_hi; c += blockDim.x)
        if (!((chosen[c >> 5] >> (c & 31)) & 1u) && sel_key(m[c], c) >= cand) ++cnt;
      if (block_sum(cnt, scratch32) >= need) x = cand;
    }
    __syncthreads();
    for (int c = c_lo + threadIdx.x; c <= c_hi; c += blockDim.x)
      if (!((chosen[c >> 5] >> (c & 31)) & 1u) && sel_key(m[c], c) >= x) atomicOr(&chosen[c >> 5], 1u << (c & 31));
  }
  __syncthreads();
  for (int w = threadIdx.x; w < W; w += blockDim.x) out[w] = chosen[w];
}

// FlexPrefill's routing rule (the comparator): Jensen-Shannon divergence
// between the last query block's block-pooled attention a (from the block
// masses) and its pooled estimate e (row nb-1 of the pooled map), in fp64.
__global__ void jsd_route_kernel(const uint64_t* __restrict__ vmass, const float* __restrict__ pbar, int nb,
                                 float tau, double* __restrict__ jsd, uint8_t* __restrict__ route, DevStatus* status) {
  __shared__ uint64_t scratch64[32];
  __shared__ double scratchd[32];
  const int h = blockIdx.x;
  if (!CRISP_CHECK(h < static_cast<int>(gridDim.x) && nb >= 1, status, 0x316)) return;
  const uint64_t* v = vmass + static_cast<size_t>(h) * nb;
  const float* e = pbar + (static_cast<size_t>(h) * nb + (nb - 1)) * nb;
  uint64_t part = 0;
  for (int c = threadIdx.x; c < nb; c += blockDim.x) part += v[c];
  const double T = static_cast<double>(block_sum(part, scratch64));
  double acc = 0.0;
  for (int c = threadIdx.x; c < nb; c += blockDim.x) {
    const double a = T > 0.0 ? static_cast<double>(v[c]) / T : 0.0;
    const double b = static_cast<double>(e[c]);
    const double mid = 0.5 * (a + b);
    if (a > 0.0) acc += a * log(a / mid);
    if (b > 0.0) acc += b * log(b / mid);
  }
  const double D = 0.5 * block_sum(acc, scratchd);
  if (threadIdx.x == 0) {
    if (jsd) jsd[h] = D;
    route[h] = sqrt(fmax(D, 0.0)) >= static_cast<double>(tau) ? 1 : 0;
  }
}

}  // namespace

cudaError_t launch_block_masses(const crisp_shape& s, const float* pmap, uint64_t* vmass, uint64_t* smass,
                                uint64_t* rmass, char* ws, cudaStream_t st) {
  const ScratchLayout L = scratch_layout(s);
  const int nb = num_blocks(s.seq_len);
  auto* kern = tail_len(s.seq_len) == kB ? mass_tiles<false> : mass_tiles<true>;
  kern<<<dim3(nb, s.hq), kMassThreads, 0, st>>>(
      pmap, map_ld(s.seq_len), tail_len(s.seq_len), vmass, reinterpret_cast<uint64_t*>(ws + L.mass_lower),
      reinterpret_cast<uint64_t*>(ws + L.mass_upper), reinterpret_cast<uint64_t*>(ws + L.mass_upper2),
      reinterpret_cast<uint64_t*>(ws + L.mass_rec), reinterpret_cast<DevStatus*>(ws + L.status));
  const cudaError_t e = cudaGetLastError();
  return e != cudaSuccess ? e : launch_assemble_slash(s, vmass, ws, smass, rmass, st);
}

cudaError_t launch_assemble_slash(const crisp_shape& s, const uint64_t* vmass, char* ws, uint64_t* smass,
                                  uint64_t* rmass, cudaStream_t st) {
  const ScratchLayout L = scratch_layout(s);
  const int nb = num_blocks(s.seq_len);
  assemble_slash<<<dim3((nb + 255) / 256, s.hq), 256, 0, st>>>(
      vmass, reinterpret_cast<const uint64_t*>(ws + L.mass_lower), reinterpret_cast<const uint64_t*>(ws + L.mass_upper),
      reinterpret_cast<const uint64_t*>(ws + L.mass_upper2), reinterpret_cast<const uint64_t*>(ws + L.mass_rec), nb,
      tail_len(s.seq_len), smass, rmass, reinterpret_cast<DevStatus*>(ws + L.status));
  return cudaGetLastError();
}

cudaError_t launch_route(const crisp_shape& s, const crisp_params& p, const uint64_t* vmass, const uint64_t* rmass,
                         uint64_t* cstruct, uint64_t* total, uint8_t* route, DevStatus* status, cudaStream_t st) {
  route_kernel<<<s.hq, 256, 0, st>>>(vmass, rmass, num_blocks(s.seq_len), p.tau_num, p.tau_den, cstruct, total,
                                     route, status);
  return cudaGetLastError();
}

cudaError_t launch_route_map(const crisp_shape& s, const crisp_params& p, const float* pmap, uint64_t* cstruct,
                             uint64_t* total, uint8_t* route, DevStatus* status, cudaStream_t st) {
  const size_t bytes = static_cast<size_t>(s.hq) * sizeof(uint64_t);
  cudaError_t e = cudaMemsetAsync(cstruct, 0, bytes, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(total, 0, bytes, st);
  if (e != cudaSuccess) return e;
  cstruct_tiles<<<dim3(num_blocks(s.seq_len), s.hq), kMassThreads, 0, st>>>(
      pmap, map_ld(s.seq_len), s.seq_len, p.sink_tokens, p.recency_tokens, cstruct, total, status);
  route_decide<<<(s.hq + 127) / 128, 128, 0, st>>>(cstruct, total, s.hq, p.tau_num, p.tau_den, route);
  return cudaGetLastError();
}

cudaError_t launch_select_vs(const crisp_shape& s, const crisp_params& p, const uint64_t* vmass,
                             const uint64_t* smass, const uint8_t* route, uint32_t* vbits, uint32_t* sbits,
                             DevStatus* status, cudaStream_t st) {
  select_vs_kernel<<<dim3(s.hq, 2), kSelThreads, 0, st>>>(vmass, smass, route, num_blocks(s.seq_len), p.alpha_num,
                                                          p.alpha_den, p.kmin_blocks, p.vs_mode, p.vs_gamma_num,
                                                          p.vs_gamma_den, vbits, sbits, status);
  return cudaGetLastError();
}

cudaError_t launch_route_jsd(const crisp_shape& s, const crisp_params& p, const uint64_t* vmass, const float* pbar,
                             double* jsd, uint8_t* route, DevStatus* status, cudaStream_t st) {
  jsd_route_kernel<<<s.hq, 256, 0, st>>>(vmass, pbar, num_blocks(s.seq_len), p.jsd_tau, jsd, route, status);
  return cudaGetLastError();
}

}  // namespace crisp
