// A5 pooled attention estimate and A6 Pooled-Estimation block selection for
// the heads routed to PE (CRISP paper page on ai.info, "Overview" and
// "Methodology in Plain English": the PE path keeps FlexPrefill's pooled
// estimate and uses gamma = 0.95 coverage).
//
// A5: qbar_b / kbar_c = means over each block's tokens (128, or fewer in a
// short last block); pbar[b][c] = softmax
// over c <= b of scale * qbar_b . kbar_c (fp32; c > b stored as 0). Two
// kernels: pool_kernel (the means, HBM-bound) and pooled_map (the products
// on the tensor cores with the row softmax fused).
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
// memory. Each mean m is stored as two bf16 values, hi = bf16(m) and
// lo = bf16(m - hi), the tensor-core operands of pooled_map.
__global__ void __launch_bounds__(256) pool_kernel(const __nv_bfloat16* __restrict__ q,
                                                   const __nv_bfloat16* __restrict__ k,
                                                   const uint8_t* __restrict__ route, int hq, int hkv, int n, int nb,
                                                   int64_t q_hs, int64_t q_ts, int64_t kv_hs, int64_t kv_ts,
                                                   __nv_bfloat16* __restrict__ qbar, __nv_bfloat16* __restrict__ kbar,
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
        if (CRISP_CHECK(o + kD <= static_cast<size_t>(is_q ? hq : hkv) * nb * kD, status, 0x411)) {
          // the mean as a sum of two bf16 values (hi + lo carries 16 bits)
          const float mean = sum * (1.0f / static_cast<float>(len));  // exact for a whole block
          const __nv_bfloat16 hi = __float2bfloat16_rn(mean);
          const __nv_bfloat16 lo = __float2bfloat16_rn(mean - __bfloat162float(hi));
          __nv_bfloat16* dst = is_q ? qbar : kbar;
          const size_t half = static_cast<size_t>(is_q ? hq : hkv) * nb * kD;  // lo after all hi rows
          dst[o + threadIdx.x] = hi;
          dst[half + o + threadIdx.x] = lo;
        }
      }
    }
  }
}

// Pooled map on the tensor cores, softmax fused: each block mean is held as
// hi + lo (two bf16 values) and qbar . kbar = hi.hi + hi.lo + lo.hi (the
// lo.lo term, 2^-16 of the product, is left out): three tcgen05 products of
// M = N = 128 over the 128 features into an fp32 TMEM accumulator. One CTA
// per SM takes items (PE head h, row tile bt), bt descending, in snake
// order. Per item it keeps A = qbar rows [128 bt, +128) in shared memory and
// walks the column tiles ct <= bt twice: pass 1 keeps each row's running max
// and sum of 2^(z - max) (z = scale log2(e) qbar . kbar), pass 2 forms the
// same products again and writes p = 2^(z - max) / sum for c <= b and 0 for
// b < c < nb (the zeros right of the row tile first, while the first
// products are in flight), so the logits never go to memory. TMA double-buffers
// B = kbar rows, the MMA thread alternates two TMEM accumulators, and eight
// epilogue warps (two per TMEM lane quarter, one per 64-column half) read
// the accumulators; each 32x16 piece of P goes through shared memory so that
// it leaves as 64-byte row segments.
constexpr int kPT = 128;                            // tile edge
constexpr uint32_t kPTile = kPT * kD * 2;           // 32 KB: one bf16 128x128 operand
constexpr uint32_t kPHalf = kPTile / 2;             // one 64-feature half
constexpr int kPStage = 32 * 20;                    // an epilogue warp's 32x16 fp32 transpose (padded rows)
constexpr int kMapThreads = 320;                 // TMA warp, MMA warp, 8 epilogue warps
constexpr uint32_t kMapSmem = 1024 + 6 * kPTile + 8 * kPStage * 4;  // A, two B stages, eight transposes

struct MapBars {
  uint64_t a_full, a_empty, b_full[2], b_empty[2], d_full[2], d_empty[2], xbar, drain;
  uint32_t tmem_base;
  int abort;
  float2 stats[2][kPT];  // (max, sum) of each row of the item's tile, per column half
};

__global__ void __launch_bounds__(kMapThreads, 1)
    pooled_map(const __grid_constant__ CUtensorMap tq_hi, const __grid_constant__ CUtensorMap tq_lo,
               const __grid_constant__ CUtensorMap tk_hi, const __grid_constant__ CUtensorMap tk_lo,
               const uint8_t* __restrict__ route, int hq, int nb, int group, float c_log2,
               float* __restrict__ pbar, DevStatus* status) {
  extern __shared__ uint8_t pe_tc_smem[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(pe_tc_smem) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = base;                 // hi, lo
  uint8_t* sB = base + 2 * kPTile;    // stage s: hi, lo at + 2 * kPTile * s
  float* sT = reinterpret_cast<float*>(base + 6 * kPTile);  // epilogue warp e: sT + e * kPStage
  __shared__ MapBars bars;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    bars.abort = 0;
    ptx::mbar_init(&bars.a_full, 1);
    ptx::mbar_init(&bars.a_empty, 1);
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&bars.b_full[i], 1);
      ptx::mbar_init(&bars.b_empty[i], 1);
      ptx::mbar_init(&bars.d_full[i], 1);
      ptx::mbar_init(&bars.d_empty[i], 8);
    }
    ptx::mbar_init(&bars.xbar, 256);
    ptx::mbar_init(&bars.drain, 1);
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(&bars.tmem_base, 256);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = bars.tmem_base;
  int n_pe = 0;
  for (int b0 = 0; b0 < hq; b0 += 32)
    n_pe += __popc(__ballot_sync(0xffffffffu, b0 + lane < hq && route[b0 + lane] == 0));
  const int T = (nb + kPT - 1) / kPT;
  const int64_t items = static_cast<int64_t>(n_pe) * T;
  const bool vec = (nb & 3) == 0 && (reinterpret_cast<uintptr_t>(pbar) & 15u) == 0;  // 16-byte row segments
  auto fail = [&](uint32_t where) {
    *reinterpret_cast<volatile int*>(&bars.abort) = 1;
    report_error(status, CRISP_ERR_TIMEOUT, where);
  };
  // phase counters (each role counts its own); `tile` counts tile passes
  uint32_t a_n = 0, b_n[2] = {0u, 0u}, d_n[2] = {0u, 0u}, x_n = 0, tile = 0;
  bool ok = true;
  for (int64_t k = 0; ok; ++k) {
    const int64_t r = snake_item(k, blockIdx.x, gridDim.x);
    if (r >= items) break;
    const int bt = T - 1 - static_cast<int>(r / n_pe);
    const int h = nth_head(route, hq, false, static_cast<int>(r % n_pe));
    // (checking build) the item's rows and its TMA coordinates lie in the maps
    if (!CRISP_CHECK(h < hq && bt >= 0 && bt * kPT < nb && h / group < hq / group, status, 0x412)) break;
    const int g = h / group;
    const int passes = 2 * (bt + 1);  // tile passes of this item
    if (warp == 0) {
      if (lane == 0) {
        if (!ptx::mbar_wait(&bars.a_empty, (a_n & 1u) ^ 1u, &bars.abort)) { fail(0x415); ok = false; }
        if (ok) {
          ptx::mbar_arrive_expect_tx(&bars.a_full, 2 * kPTile);
          ptx::tma_load_3d(sA, &tq_hi, &bars.a_full, 0, bt * kPT, h);
          ptx::tma_load_3d(sA + kPHalf, &tq_hi, &bars.a_full, 64, bt * kPT, h);
          ptx::tma_load_3d(sA + kPTile, &tq_lo, &bars.a_full, 0, bt * kPT, h);
          ptx::tma_load_3d(sA + kPTile + kPHalf, &tq_lo, &bars.a_full, 64, bt * kPT, h);
        }
        for (int t = 0; ok && t < passes; ++t) {
          const int ct = t % (bt + 1);
          const int st = static_cast<int>((tile + t) & 1u);
          if (!ptx::mbar_wait(&bars.b_empty[st], (b_n[st] & 1u) ^ 1u, &bars.abort)) { fail(0x416); ok = false; break; }
          ++b_n[st];
          uint8_t* dst = sB + 2 * kPTile * st;
          ptx::mbar_arrive_expect_tx(&bars.b_full[st], 2 * kPTile);
          ptx::tma_load_3d(dst, &tk_hi, &bars.b_full[st], 0, ct * kPT, g);
          ptx::tma_load_3d(dst + kPHalf, &tk_hi, &bars.b_full[st], 64, ct * kPT, g);
          ptx::tma_load_3d(dst + kPTile, &tk_lo, &bars.b_full[st], 0, ct * kPT, g);
          ptx::tma_load_3d(dst + kPTile + kPHalf, &tk_lo, &bars.b_full[st], 64, ct * kPT, g);
        }
      }
    } else if (warp == 1) {
      if (lane == 0) {
        constexpr uint32_t idesc = ptx::idesc_bf16_f32(128, 128, false, false);
        if (!ptx::mbar_wait(&bars.a_full, a_n & 1u, &bars.abort)) { fail(0x417); ok = false; }
        const uint32_t ah = ptx::smem_u32(sA), al = ptx::smem_u32(sA + kPTile);
        for (int t = 0; ok && t < passes; ++t) {
          const int u = static_cast<int>((tile + t) & 1u);  // B stage and accumulator
          if (!ptx::mbar_wait(&bars.b_full[u], b_n[u] & 1u, &bars.abort) ||
              !ptx::mbar_wait(&bars.d_empty[u], (d_n[u] & 1u) ^ 1u, &bars.abort)) {
            fail(0x418);
            ok = false;
            break;
          }
          ++b_n[u];
          ++d_n[u];
          ptx::tc_fence_after();
          const uint32_t bh = ptx::smem_u32(sB + 2 * kPTile * u), bl = bh + kPTile;
          const uint32_t d = tmem + u * 128;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t off = (kk >> 2) * kPHalf + (kk & 3) * 32;
            ptx::umma_ss(d, ptx::sdesc_sw128(ah + off, 16, 1024), ptx::sdesc_sw128(bh + off, 16, 1024), idesc, kk > 0);
            ptx::umma_ss(d, ptx::sdesc_sw128(ah + off, 16, 1024), ptx::sdesc_sw128(bl + off, 16, 1024), idesc, 1);
            ptx::umma_ss(d, ptx::sdesc_sw128(al + off, 16, 1024), ptx::sdesc_sw128(bh + off, 16, 1024), idesc, 1);
          }
          ptx::umma_commit(&bars.b_empty[u]);
          ptx::umma_commit(&bars.d_full[u]);
        }
        ptx::umma_commit(&bars.a_empty);
      }
    } else {
      // Epilogue warp e = warp - 2 reads TMEM lane quarter q = warp % 4 (rows
      // r0 .. r0 + 31 of the tile, one per lane) and the 64 columns of half
      // ch of each accumulator.
      const int e = warp - 2, q = warp & 3, ch = e >> 2;
      const int r0 = bt * kPT + q * 32, row = r0 + lane;
      const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
      float* tr = sT + e * kPStage;
      float* out = pbar + static_cast<size_t>(h) * nb * nb;
      // zeros right of the row tile: columns [128 (bt + 1), nb) of rows r0 ..
      // r0 + 31, the two warps of a quarter taking alternate 32-lane runs
      const int z0 = (bt + 1) * kPT;
      if (z0 < nb) {
        const int rows = min(32, nb - r0);
        for (int rr = 0; rr < rows; ++rr) {
          float* dst = out + static_cast<size_t>(r0 + rr) * nb;
          if (!CRISP_CHECK(static_cast<size_t>(h) * nb + r0 + rr < static_cast<size_t>(hq) * nb, status, 0x41b)) break;
          if (vec) {
            for (int c = z0 + 4 * (ch * 32 + lane); c < nb; c += 4 * 64)
              *reinterpret_cast<float4*>(dst + c) = make_float4(0.f, 0.f, 0.f, 0.f);
          } else {
            for (int c = z0 + ch * 32 + lane; c < nb; c += 64) dst[c] = 0.f;
          }
        }
      }
      float m = -INFINITY, l = 0.f, inv = 0.f;
      for (int t = 0; t < passes; ++t) {
        const bool second = t > bt;
        if (t == bt + 1) {
          // the two halves' (max, sum) of each row combine into the row's
          bars.stats[ch][q * 32 + lane] = make_float2(m, l);
          ptx::mbar_arrive(&bars.xbar);
          if (ok && !ptx::mbar_wait(&bars.xbar, x_n & 1u, &bars.abort)) {
            if (lane == 0) fail(0x41a);
            ok = false;
          }
          ++x_n;
          const float2 a = bars.stats[0][q * 32 + lane], b = bars.stats[1][q * 32 + lane];
          m = fmaxf(a.x, b.x);  // finite for rows < nb: column 0 is in half 0
          l = a.y * ptx::ex2_approx(a.x - m) + (b.x == -INFINITY ? 0.f : b.y * ptx::ex2_approx(b.x - m));
          inv = 1.0f / l;
        }
        if (!ok) break;
        const int ct = t % (bt + 1);
        const int u = static_cast<int>((tile + t) & 1u);
        if (!ptx::mbar_wait(&bars.d_full[u], d_n[u] & 1u, &bars.abort)) {
          if (lane == 0) fail(0x419);
          ok = false;
          break;
        }
        ++d_n[u];
        ptx::tc_fence_after();
        if (!second) {
#pragma unroll 1
          for (int pc = 0; pc < 2; ++pc) {
            const int c0 = ch * 64 + pc * 32, col = ct * kPT + c0;
            if (r0 >= nb || col >= nb || col > r0 + 31) break;  // past the map, or right of the diagonal
            uint32_t v[32];
            ptx::tmem_ld32(tmem + lane_addr + u * 128 + c0, v);
            float z[32], mp = -INFINITY;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              z[j] = col + j <= row ? __fmul_rn(__uint_as_float(v[j]), c_log2) : -INFINITY;
              mp = fmaxf(mp, z[j]);
            }
            if (mp != -INFINITY) {  // this row has entries c <= b in the piece
              const float mn = fmaxf(m, mp);
              float s0 = 0.f, s1 = 0.f;
#pragma unroll
              for (int j = 0; j < 32; j += 2) {
                s0 += ptx::ex2_approx(z[j] - mn);
                s1 += ptx::ex2_approx(z[j + 1] - mn);
              }
              l = (m == -INFINITY ? 0.f : l * ptx::ex2_approx(m - mn)) + (s0 + s1);
              m = mn;
            }
          }
        } else {
#pragma unroll 1
          for (int pc = 0; pc < 4; ++pc) {
            const int c0 = ch * 64 + pc * 16, col = ct * kPT + c0;
            if (r0 >= nb || col >= nb) break;  // rows or columns past the map
            const bool above = col > r0 + 31;  // the whole piece lies right of the diagonal
            uint32_t v[16];
            if (!above) ptx::tmem_ld16(tmem + lane_addr + u * 128 + c0, v);
#pragma unroll
            for (int j = 0; j < 16; j += 4) {
              float pj[4];
#pragma unroll
              for (int x = 0; x < 4; ++x)
                pj[x] = !above && col + j + x <= row
                            ? ptx::ex2_approx(__fmul_rn(__uint_as_float(v[j + x]), c_log2) - m) * inv
                            : 0.f;
              *reinterpret_cast<float4*>(tr + lane * 20 + j) = make_float4(pj[0], pj[1], pj[2], pj[3]);
            }
            __syncwarp();
            // rows r0 + 8i + lane / 4, columns col + 4 (lane % 4) .. + 3
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int rr = 8 * i + (lane >> 2), cc = 4 * (lane & 3);
              const float4 p = *reinterpret_cast<const float4*>(tr + rr * 20 + cc);
              if (r0 + rr < nb && col + cc < nb &&
                  CRISP_CHECK(static_cast<size_t>(h) * nb + r0 + rr < static_cast<size_t>(hq) * nb, status, 0x41c)) {
                float* dst = out + static_cast<size_t>(r0 + rr) * nb + col + cc;
                if (vec) {
                  *reinterpret_cast<float4*>(dst) = p;
                } else {
                  dst[0] = p.x;
                  if (col + cc + 1 < nb) dst[1] = p.y;
                  if (col + cc + 2 < nb) dst[2] = p.z;
                  if (col + cc + 3 < nb) dst[3] = p.w;
                }
              }
            }
            __syncwarp();
          }
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&bars.d_empty[u]);
      }
    }
    ++a_n;
    tile += static_cast<uint32_t>(passes);
    ok = __syncthreads_and(ok) != 0;
  }
  if (warp == 1 && lane == 0) {
    ptx::umma_commit(&bars.drain);
    const int never = 0;
    ptx::mbar_wait(&bars.drain, 0, &never);
  }
  if (warp == 0 && lane == 0) {
    // every copy has landed before the CTA exits (consumers may have given up)
    const int never = 0;
    if (a_n > 0) ptx::mbar_wait(&bars.a_full, (a_n - 1u) & 1u, &never);
    for (int i = 0; i < 2; ++i)
      if (b_n[i] > 0) ptx::mbar_wait(&bars.b_full[i], (b_n[i] - 1u) & 1u, &never);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc(tmem, 256);
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
  int hist, last, chosen, vals, bytes;  // byte offsets inside one warp's slice
};
__host__ __device__ inline PeWarpLayout pe_warp_layout(int nb, bool row_in_shared) {
  PeWarpLayout L;
  L.hist = 0;
  L.last = 256 * 8;
  L.chosen = L.last + 256 * 2;
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
  auto* last = reinterpret_cast<unsigned short*>(mine + L.last);
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
        [&](unsigned long long f) { return static_cast<unsigned __int128>(gamma_den) * f >= goal; }, hist, last);
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
        [&](unsigned long long cnt) { return cnt >= static_cast<unsigned long long>(need); }, hist, last);
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
  auto* qbar = reinterpret_cast<__nv_bfloat16*>(ws + L.qbar);  // hi [hq][nb][128], then lo
  auto* kbar = reinterpret_cast<__nv_bfloat16*>(ws + L.kbar);  // hi [hkv][nb][128], then lo
  auto* status = reinterpret_cast<DevStatus*>(ws + L.status);
  // Grids of resident CTAs, each looping over its share of the PE heads'
  // items (VS heads cost a route read), so a layer with few PE heads launches
  // no idle CTAs.
  const int sms = sm_count();
  const int64_t pool_items = static_cast<int64_t>(s.hq + s.hkv) * nb;
  pool_kernel<<<resident_grid(pool_kernel, sms, pool_items), 256, 0, st>>>(
      static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k), route, s.hq, s.hkv, s.seq_len, nb,
      s.q_head_stride, s.q_tok_stride, s.kv_head_stride, s.kv_tok_stride, qbar, kbar, status);
  CUtensorMap tq_hi, tq_lo, tk_hi, tk_lo;
  const size_t q_half = static_cast<size_t>(s.hq) * nb * kD, k_half = static_cast<size_t>(s.hkv) * nb * kD;
  if (!encode_bf16_rows(&tq_hi, qbar, s.hq, nb) || !encode_bf16_rows(&tq_lo, qbar + q_half, s.hq, nb) ||
      !encode_bf16_rows(&tk_hi, kbar, s.hkv, nb) || !encode_bf16_rows(&tk_lo, kbar + k_half, s.hkv, nb))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(pooled_map, cudaFuncAttributeMaxDynamicSharedMemorySize, kMapSmem);
  if (e != cudaSuccess) return e;
  const int64_t T = (nb + kPT - 1) / kPT;
  pooled_map<<<static_cast<unsigned>(std::min<int64_t>(sms, static_cast<int64_t>(s.hq) * T)), kMapThreads,
               kMapSmem, st>>>(tq_hi, tq_lo, tk_hi, tk_lo, route, s.hq, nb, s.hq / s.hkv,
                                  s.scale * 1.4426950408889634f, pbar, status);
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
