// A1. Proxy attention map of the last query block (CRISP paper page on
// ai.info, "Key Contributions" 2 / "Methodology": routing and Vertical-Slash
// selection read the proxy attention map of the last query block).
//
//   pmap[h][r][j] = softmax_j( scale * q_{n-128+r} . k_j ),  j <= n-128+r
//
// Key tiles are the 128-token blocks aligned at token 0 (the last one short
// when 128 does not divide n; TMA fills its missing rows with zeros and the
// causal mask hides them); the query rows are the last 128 tokens.
//
// Two passes over the keys with the same tile engine: pass 1 computes per-row
// (max, sum of exp) over each chunk of key blocks, a tiny kernel combines the
// chunks, pass 2 recomputes the logits and writes the normalised fp32 map.
// The logits S = Q K^T of one 128x128 tile come from tcgen05.mma into TMEM
// (two S buffers, so the MMA of tile t+1 overlaps the epilogue of tile t);
// operands arrive by TMA (128-byte swizzle). The map write is the dominant
// cost (4 * hq * 128 * n bytes), so the epilogue transposes each warp's
// 32x32 fp32 block through shared memory and writes full 128-byte lines.
#include "common.cuh"
#include "ptx.cuh"

namespace crisp {
using namespace ptx;

namespace {

constexpr int kEpiWarps = 8;                       // 2 warps per TMEM lane quarter (column halves)
constexpr int kThreads = (kEpiWarps + 2) * 32;     // + TMA warp + MMA warp
constexpr int kTmaWarp = kEpiWarps;
constexpr int kMmaWarp = kEpiWarps + 1;
constexpr uint32_t kTile = kB * kD * 2;            // one bf16 128x128 tile: 32 KB
constexpr uint32_t kHalf = kTile / 2;              // 64-feature half (TMA box)
constexpr int kMaxStages = 3;                      // K ring (at most)
constexpr uint32_t kStageBytes = 32 * 32 * 4;      // per-warp transpose buffer
constexpr uint32_t kTmemCols = 256;                // two 128-column S buffers

struct Bars {
  uint64_t q_full;
  uint64_t k_full[kMaxStages], k_empty[kMaxStages];
  uint64_t s_full[2], s_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, int* abort) {
  const bool ok = mbar_wait(bar, parity, abort);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void fail(int* abort, DevStatus* st, uint32_t where) {
  *reinterpret_cast<volatile int*>(abort) = 1;
  report_error(st, CRISP_ERR_TIMEOUT, where);
}

// Pass kinds: per-chunk row statistics, the map write, and the fused block
// masses (the same fp32 probabilities, quantised and summed per 128x128 tile
// the way the mass pass sums the written map, so the masses are identical).
enum : int { kStats = 0, kWriteMap = 1, kMasses = 2 };

// The map write keeps a three-deep K ring and a transpose buffer (one CTA per
// SM). The two passes that store nothing per element use a two-deep ring and
// no buffer, so two CTAs fit on an SM (2 x 97 KB shared, 2 x 256 TMEM
// columns) and twice the epilogue warps hide the exponential latency.
template <int kMode>
struct ProxyCfg {
  static constexpr int kStages = kMode == kWriteMap ? 3 : 2;
  static constexpr int kCtasPerSm = kMode == kWriteMap ? 1 : 2;
  static constexpr uint32_t kSmem =
      1024 + kTile + kStages * kTile + (kMode == kWriteMap ? kEpiWarps * kStageBytes : 0u);
};

// grid: (hq, chunks). CTA (h, chunk) covers key blocks [chunk*C, chunk*C + C).
// kRagged: 128 does not divide n. The whole-block instantiation has the tail
// fixed at 128, so the third slash band and the recency part fold away.
template <int kMode, bool kRagged>
__global__ void __launch_bounds__(kThreads, ProxyCfg<kMode>::kCtasPerSm)
    proxy_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk, int n, int group,
                 float c_log2, float* __restrict__ pmap, int64_t ld, float2* __restrict__ part,
                 const float2* __restrict__ stats, uint64_t* __restrict__ vmass, uint64_t* __restrict__ lower,
                 uint64_t* __restrict__ upper, uint64_t* __restrict__ upper2, uint64_t* __restrict__ rec,
                 DevStatus* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = base;
  uint8_t* sK = base + kTile;
  constexpr int kStages = ProxyCfg<kMode>::kStages;
  float* sStage = reinterpret_cast<float*>(base + kTile + kStages * kTile);
  __shared__ Bars bars;
  __shared__ unsigned long long tile_acc[2][4];  // [tile parity][whole, band lo, band hi, recency part]
  __shared__ unsigned int tile_cnt[2];           // warps that have added to the slot

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.x, chunk = blockIdx.y, nchunks = gridDim.y;
  const int g = h / group;
  const int nb = (n + kB - 1) / kB;
  const int tail = kRagged ? n - (nb - 1) * kB : kB;  // tokens of the last block, in [1, 128]
  const int kb0 = chunk * kProxyChunk;
  const int T = min(nb, kb0 + kProxyChunk) - kb0;

  if (threadIdx.x == 0) {
    bars.abort = 0;
    for (int b = 0; b < 2; ++b)
      for (int k = 0; k < 4; ++k) tile_acc[b][k] = 0ull;
    tile_cnt[0] = tile_cnt[1] = 0u;
    mbar_init(&bars.q_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars.k_full[s], 1);
      mbar_init(&bars.k_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars.s_full[b], 1);
      mbar_init(&bars.s_empty[b], kEpiWarps);
    }
    mbar_init(&bars.drain, 1);
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&bars.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars.tmem_base;

  if (warp == kTmaWarp) {
    if (lane == 0) {
      prefetch_tmap(&tq);
      prefetch_tmap(&tk);
      // (checking build) a tile outside q or k is not copied; its barrier
      // phase completes without data and the status word says why.
      if (CRISP_CHECK(n - kB >= 0 && h < static_cast<int>(gridDim.x), status, 0x110)) {
        mbar_arrive_expect_tx(&bars.q_full, kTile);
        tma_load_3d(sQ, &tq, &bars.q_full, 0, n - kB, h);
        tma_load_3d(sQ + kHalf, &tq, &bars.q_full, 64, n - kB, h);
      } else {
        mbar_arrive(&bars.q_full);
      }
      int issued = 0;  // K tiles whose copies were started
      for (int t = 0; t < T; ++t) {
        const int s = t % kStages;
        const uint32_t use = t / kStages;
        if (!mbar_wait(&bars.k_empty[s], (use & 1u) ^ 1u, &bars.abort)) {
          fail(&bars.abort, status, 0x101);
          break;
        }
        ++issued;
        if (!CRISP_CHECK((kb0 + t) * kB < n && g < static_cast<int>(gridDim.x) / group, status, 0x111)) {
          mbar_arrive(&bars.k_full[s]);
          continue;
        }
        mbar_arrive_expect_tx(&bars.k_full[s], kTile);
        uint8_t* dst = sK + s * kTile;
        tma_load_3d(dst, &tk, &bars.k_full[s], 0, (kb0 + t) * kB, g);
        tma_load_3d(dst + kHalf, &tk, &bars.k_full[s], 64, (kb0 + t) * kB, g);
      }
      // Every copy issued has landed before the CTA may exit (after a timeout
      // the consumers may not have waited for it): the last use of each slot.
      const int never = 0;
      mbar_wait(&bars.q_full, 0, &never);
      for (int s = 0; s < kStages && s < issued; ++s) {
        const int last_use = (issued - 1 - s) / kStages;  // uses of slot s: t = s, s + kStages, ...
        mbar_wait(&bars.k_full[s], static_cast<uint32_t>(last_use) & 1u, &never);
      }
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, 128, false, false);
      bool ok = mbar_wait(&bars.q_full, 0, &bars.abort);
      if (!ok) fail(&bars.abort, status, 0x102);
      for (int t = 0; ok && t < T; ++t) {
        const int s = t % kStages;
        const int b = t & 1;
        if (!mbar_wait(&bars.k_full[s], (t / kStages) & 1u, &bars.abort) ||
            !mbar_wait(&bars.s_empty[b], ((t >> 1) & 1u) ^ 1u, &bars.abort)) {
          fail(&bars.abort, status, 0x103);
          break;
        }
        tc_fence_after();
        const uint32_t qa = smem_u32(sQ), ka = smem_u32(sK + s * kTile);
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
          umma_ss(tmem + b * 128, sdesc_sw128(qa + off, 16, 1024), sdesc_sw128(ka + off, 16, 1024), idesc, kk > 0);
        }
        umma_commit(&bars.k_empty[s]);
        umma_commit(&bars.s_full[b]);
      }
      // Every MMA issued above has completed before TMEM is released.
      umma_commit(&bars.drain);
      if (!mbar_wait(&bars.drain, 0, &bars.abort)) fail(&bars.abort, status, 0x104);
    }
  } else {
    // Epilogue: warp w reads TMEM lanes 32*(w%4).. (rows) and column half w/4.
    const int quarter = warp & 3, half = warp >> 2;
    const int r = quarter * 32 + lane;  // row of the query block
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    float m_run = -INFINITY, l_run = 0.f;
    float M = 0.f, inv_l = 0.f, inv_l32 = 0.f;
    if (kMode != kStats && CRISP_CHECK(h < static_cast<int>(gridDim.x), status, 0x112)) {
      const float2 st = stats[static_cast<size_t>(h) * kB + r];
      M = st.x;
      inv_l = st.y;
      // p * 2^32 == e * (inv_l * 2^32) exactly for every normal p; a
      // subnormal p quantises to 0 either way.
      inv_l32 = st.y * 4294967296.0f;
    }
    float* stg = sStage + warp * (32 * 32);
    for (int t = 0; t < T; ++t) {
      const int b = t & 1;
      if (!warp_wait(&bars.s_full[b], (t >> 1) & 1u, &bars.abort)) {
        if (lane == 0) fail(&bars.abort, status, 0x105);
        break;
      }
      tc_fence_after();
      const int kb = kb0 + t;
      // Row r is token n-128+r = (nb-2)*128 + tail + r and column jj of this
      // tile is token 128*kb + jj: visible iff jj - r <= lim (causal edge in
      // the last one or two tiles).
      const int lim = (nb - 2 - kb) * kB + tail;
      const bool edge = lim < kB - 1;
      const bool rec_tile = kb == nb - 2 && tail < kB;  // holds recency columns jj >= tail
      // Q32 quanta of this row's 64 probabilities of the tile: below 2^23 in
      // 32 bits (64 of them stay below 2^29), larger ones in 64 bits.
      uint32_t all32 = 0, lo32 = 0, hi32 = 0;
      uint64_t all64 = 0, lo64 = 0, hi64 = 0, rec64 = 0;
#pragma unroll 1
      for (int cc = 0; cc < 2; ++cc) {
        const int col0 = half * 64 + cc * 32;
        uint32_t v[32];
        tmem_ld32(tmem + lane_addr + b * 128 + col0, v);
        // Raw logits S; on the causal edge keys j > n-128+r are -inf.
        float x[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) x[e] = __uint_as_float(v[e]);
        if (edge) {
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (col0 + e - r > lim) x[e] = -INFINITY;
        }
        if (kMode == kStats) {
          // Running (max, sum) in base-2 units: m = c_log2 * max S, l = sum
          // 2^(c_log2*S - m), with the exponent as one fma. Tree max and four
          // partial sums keep the dependency chains short.
          float t[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) t[i] = fmax3(x[4 * i], x[4 * i + 1], fmaxf(x[4 * i + 2], x[4 * i + 3]));
          const float mx = fmax3(fmax3(t[0], t[1], t[2]), fmax3(t[3], t[4], t[5]), fmaxf(t[6], t[7])) * c_log2;
          if (mx > m_run) {
            l_run *= ex2_approx(m_run - mx);
            m_run = mx;
          }
          if (m_run != -INFINITY) {
            float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
              float y[4];
              ffma2(y[0], y[1], x[e], x[e + 1], c_log2, c_log2, -m_run, -m_run);
              ffma2(y[2], y[3], x[e + 2], x[e + 3], c_log2, c_log2, -m_run, -m_run);
              fadd2_acc(s4[0], s4[1], ex2_approx(y[0]), ex2_approx(y[1]));
              fadd2_acc(s4[2], s4[3], ex2_approx(y[2]), ex2_approx(y[3]));
            }
            l_run += (s4[0] + s4[1]) + (s4[2] + s4[3]);
          }
        } else {
          // The base-2 exponent c_log2*S - M as one fma, so the map write
          // and the fused masses evaluate p = 2^(c_log2*S - M) / L alike.
#pragma unroll
          for (int e = 0; e < 32; e += 2) ffma2(x[e], x[e + 1], x[e], x[e + 1], c_log2, c_log2, -M, -M);
        }
        if (kMode == kWriteMap) {
          // Row `lane` of this warp's 32x32 block into the transpose buffer
          // (16-byte chunks XOR-swizzled by row to spread the banks).
#pragma unroll
          for (int c4 = 0; c4 < 8; ++c4) {
            float4 p;
            p.x = ex2_approx(x[4 * c4 + 0]) * inv_l;
            p.y = ex2_approx(x[4 * c4 + 1]) * inv_l;
            p.z = ex2_approx(x[4 * c4 + 2]) * inv_l;
            p.w = ex2_approx(x[4 * c4 + 3]) * inv_l;
            reinterpret_cast<float4*>(stg + lane * 32)[c4 ^ (lane & 7)] = p;
          }
          __syncwarp();
          const int c4 = lane & 7;
#pragma unroll
          for (int it = 0; it < 8; ++it) {
            const int R = it * 4 + (lane >> 3);
            const float4 p = reinterpret_cast<const float4*>(stg + R * 32)[c4 ^ (R & 7)];
            const size_t idx = (static_cast<size_t>(h) * kB + quarter * 32 + R) * static_cast<size_t>(ld) +
                               static_cast<size_t>(kb) * kB + col0 + c4 * 4;
            if (CRISP_CHECK(idx + 4 <= static_cast<size_t>(gridDim.x) * kB * static_cast<size_t>(ld) &&
                                static_cast<size_t>(kb) * kB + col0 + c4 * 4 + 4 <= static_cast<size_t>(ld),
                            status, 0x113))
              *reinterpret_cast<float4*>(pmap + idx) = p;
          }
          __syncwarp();
        } else if (kMode == kMasses) {
          // xq = p * 2^32 for the p the map write stores.
          float xq[32];
#pragma unroll
          for (int e = 0; e < 32; e += 2)
            fmul2(xq[e], xq[e + 1], ex2_approx(x[e]), ex2_approx(x[e + 1]), inv_l32, inv_l32);
          float t[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) t[i] = fmax3(xq[4 * i], xq[4 * i + 1], fmaxf(xq[4 * i + 2], xq[4 * i + 3]));
          const float mx = fmax3(fmax3(t[0], t[1], t[2]), fmax3(t[3], t[4], t[5]), fmaxf(t[6], t[7]));
          // Slash bands of the tile (as the mass pass over the map sums
          // them): band lo = entries with jj - r <= tail-128 (slash block
          // nb-1-kb; the lower triangle when 128 | n), band hi = jj - r >
          // tail (block nb-3-kb; empty when 128 | n), the rest block
          // nb-2-kb. Here jj - r = D0 + e - lane with D0 = col0 - 32*quarter,
          // so each band holds none, all or the e - lane side of a
          // warp-uniform threshold.
          const int D0 = col0 - quarter * 32;
          const int th_lo = tail - kB - D0, th_hi = tail - D0;
          const bool lo_all = th_lo >= 31, lo_part = !lo_all && th_lo >= -31;
          const bool hi_all = kRagged && th_hi < -31, hi_part = kRagged && !hi_all && th_hi < 31;
          if (!__any_sync(0xffffffffu, mx >= kTwo23)) {
            // Every quantum below 2^23: the bits of xq + 2^23 minus those of
            // 2^23, with the 32 subtractions taken once at the end (mod 2^32;
            // the true sums stay below 2^28).
            uint32_t a4[4] = {0u, 0u, 0u, 0u}, lo = 0, hi = 0;
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              float t0, t1;
              fadd2(t0, t1, xq[e], xq[e + 1], kTwo23, kTwo23);
              const uint32_t u0 = __float_as_uint(t0), u1 = __float_as_uint(t1);
              a4[e & 3] += u0;
              a4[(e + 1) & 3] += u1;
              if (lo_part) {
                lo += e - lane <= th_lo ? u0 : 0x4B000000u;
                lo += e + 1 - lane <= th_lo ? u1 : 0x4B000000u;
              }
              if (hi_part) {
                hi += e - lane > th_hi ? u0 : 0x4B000000u;
                hi += e + 1 - lane > th_hi ? u1 : 0x4B000000u;
              }
            }
            const uint32_t a = (a4[0] + a4[1]) + (a4[2] + a4[3]) - 32u * 0x4B000000u;
            all32 += a;
            lo32 += lo_part ? lo - 32u * 0x4B000000u : (lo_all ? a : 0u);
            hi32 += hi_part ? hi - 32u * 0x4B000000u : (hi_all ? a : 0u);
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const bool in_lo = e - lane <= th_lo, in_hi = kRagged && e - lane > th_hi;
              if (xq[e] < kTwo23) {
                const uint32_t f = q32_small(xq[e]);
                all32 += f;
                lo32 += in_lo ? f : 0u;
                hi32 += in_hi ? f : 0u;
              } else {
                const uint64_t f = q32_large(xq[e]);
                all64 += f;
                lo64 += in_lo ? f : 0ull;
                hi64 += in_hi ? f : 0ull;
              }
            }
          }
          if (rec_tile) {
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (col0 + e >= tail)
                rec64 += xq[e] < kTwo23 ? static_cast<uint64_t>(q32_small(xq[e])) : q32_large(xq[e]);
          }
        }
      }
      if (kMode == kMasses) {
        // Tile sums: the rows of this warp by shuffles, then the eight warps
        // by shared-memory atomics into the slot of this tile's parity; the
        // last warp to add publishes the sums and clears the slot (before it
        // releases S, so the slot's next use, two tiles later, sees it clear).
        unsigned long long all = all64 + all32, lo = lo64 + lo32, hi = hi64 + hi32, rc = rec64;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          all += __shfl_xor_sync(0xffffffffu, all, o);
          lo += __shfl_xor_sync(0xffffffffu, lo, o);
          if (kRagged) hi += __shfl_xor_sync(0xffffffffu, hi, o);
        }
        if (rec_tile) {
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) rc += __shfl_xor_sync(0xffffffffu, rc, o);
        }
        if (lane == 0) {
          atomicAdd(&tile_acc[b][0], all);
          atomicAdd(&tile_acc[b][1], lo);
          if (kRagged) atomicAdd(&tile_acc[b][2], hi);
          if (rec_tile) atomicAdd(&tile_acc[b][3], rc);
          __threadfence_block();
          if (atomicAdd(&tile_cnt[b], 1u) == kEpiWarps - 1) {
            __threadfence_block();
            const unsigned long long sa = atomicExch(&tile_acc[b][0], 0ull);
            const unsigned long long sl = atomicExch(&tile_acc[b][1], 0ull);
            const unsigned long long sh = kRagged ? atomicExch(&tile_acc[b][2], 0ull) : 0ull;
            const unsigned long long sr = atomicExch(&tile_acc[b][3], 0ull);
            atomicExch(&tile_cnt[b], 0u);
            const size_t idx = static_cast<size_t>(h) * nb + kb;
            if (CRISP_CHECK(idx < static_cast<size_t>(gridDim.x) * nb, status, 0x114)) {
              vmass[idx] = sa;
              lower[idx] = sl;
              upper[idx] = sa - sl - sh;
              upper2[idx] = sh;
            }
            if (rec_tile && CRISP_CHECK(h < static_cast<int>(gridDim.x), status, 0x115)) rec[h] = sr;
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.s_empty[b]);
    }
    if (kMode == kStats) {
      const size_t idx = (static_cast<size_t>(h) * kB + r) * (2 * nchunks) + 2 * chunk + half;
      if (CRISP_CHECK(idx < static_cast<size_t>(gridDim.x) * kB * 2 * nchunks, status, 0x116))
        part[idx] = make_float2(m_run, l_run);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
}

// Combines the per-chunk (max, sum) pairs of each row, one warp per row:
// M = max m_c, L = sum l_c * 2^(m_c - M); stores (M, 1/L).
__global__ void proxy_combine(const float2* __restrict__ part, float2* __restrict__ stats, int rows, int nparts,
                              DevStatus* status) {
  const int row = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (row >= rows) return;  // whole warps
  if (!CRISP_CHECK(static_cast<size_t>(row) * nparts + nparts <= static_cast<size_t>(rows) * nparts, status, 0x117))
    return;
  const float2* p = part + static_cast<size_t>(row) * nparts;
  float M = -INFINITY;
  for (int c = lane; c < nparts; c += 32) M = fmaxf(M, p[c].x);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float L = 0.f;
  for (int c = lane; c < nparts; c += 32)
    if (p[c].x != -INFINITY) L += p[c].y * ex2_approx(p[c].x - M);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
  if (lane == 0) stats[row] = make_float2(M, 1.0f / L);
}

}  // namespace

// Pass 1 (row statistics) and their combination; shared by both entry points.
static cudaError_t proxy_stats(const crisp_shape& s, const TmaMaps& maps, char* ws, cudaStream_t st) {
  const ScratchLayout L = scratch_layout(s);
  const int chunks = proxy_chunks(num_blocks(s.seq_len));
  auto* part = reinterpret_cast<float2*>(ws + L.proxy_part);
  auto* stats = reinterpret_cast<float2*>(ws + L.proxy_stats);
  auto* status = reinterpret_cast<DevStatus*>(ws + L.status);
  auto* kern = tail_len(s.seq_len) == kB ? proxy_kernel<kStats, false> : proxy_kernel<kStats, true>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, ProxyCfg<kStats>::kSmem);
  if (e != cudaSuccess) return e;
  kern<<<dim3(s.hq, chunks), kThreads, ProxyCfg<kStats>::kSmem, st>>>(
      maps.q, maps.k, s.seq_len, s.hq / s.hkv, s.scale * 1.4426950408889634f, nullptr, 0, part, stats, nullptr,
      nullptr, nullptr, nullptr, nullptr, status);
  const int rows = s.hq * kB;
  proxy_combine<<<(rows + 7) / 8, 256, 0, st>>>(part, stats, rows, 2 * chunks, status);  // 8 rows (warps) per CTA
  return cudaGetLastError();
}

cudaError_t launch_proxy(const crisp_shape& s, const TmaMaps& maps, float* pmap, char* ws, cudaStream_t st) {
  cudaError_t e = proxy_stats(s, maps, ws, st);
  if (e != cudaSuccess) return e;
  const ScratchLayout L = scratch_layout(s);
  const int chunks = proxy_chunks(num_blocks(s.seq_len));
  auto* kern = tail_len(s.seq_len) == kB ? proxy_kernel<kWriteMap, false> : proxy_kernel<kWriteMap, true>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, ProxyCfg<kWriteMap>::kSmem);
  if (e != cudaSuccess) return e;
  kern<<<dim3(s.hq, chunks), kThreads, ProxyCfg<kWriteMap>::kSmem, st>>>(
      maps.q, maps.k, s.seq_len, s.hq / s.hkv, s.scale * 1.4426950408889634f, pmap, map_ld(s.seq_len),
      reinterpret_cast<float2*>(ws + L.proxy_part), reinterpret_cast<const float2*>(ws + L.proxy_stats), nullptr,
      nullptr, nullptr, nullptr, nullptr, reinterpret_cast<DevStatus*>(ws + L.status));
  return cudaGetLastError();
}

cudaError_t launch_proxy_masses(const crisp_shape& s, const TmaMaps& maps, uint64_t* vmass, uint64_t* smass,
                                uint64_t* rmass, char* ws, cudaStream_t st) {
  cudaError_t e = proxy_stats(s, maps, ws, st);
  if (e != cudaSuccess) return e;
  const ScratchLayout L = scratch_layout(s);
  const int chunks = proxy_chunks(num_blocks(s.seq_len));
  auto* kern = tail_len(s.seq_len) == kB ? proxy_kernel<kMasses, false> : proxy_kernel<kMasses, true>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, ProxyCfg<kMasses>::kSmem);
  if (e != cudaSuccess) return e;
  kern<<<dim3(s.hq, chunks), kThreads, ProxyCfg<kMasses>::kSmem, st>>>(
      maps.q, maps.k, s.seq_len, s.hq / s.hkv, s.scale * 1.4426950408889634f, nullptr, 0,
      reinterpret_cast<float2*>(ws + L.proxy_part), reinterpret_cast<const float2*>(ws + L.proxy_stats), vmass,
      reinterpret_cast<uint64_t*>(ws + L.mass_lower), reinterpret_cast<uint64_t*>(ws + L.mass_upper),
      reinterpret_cast<uint64_t*>(ws + L.mass_upper2), reinterpret_cast<uint64_t*>(ws + L.mass_rec),
      reinterpret_cast<DevStatus*>(ws + L.status));
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_assemble_slash(s, vmass, ws, smass, rmass, st);
}

}  // namespace crisp
