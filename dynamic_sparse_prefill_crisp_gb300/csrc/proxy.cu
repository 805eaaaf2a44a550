// A1. Proxy attention map of the last query block (CRISP paper page on
// ai.info, "Key Contributions" 2 / "Methodology": routing and Vertical-Slash
// selection read the proxy attention map of the last query block).
//
//   pmap[h][r][j] = softmax_j( scale * q_{n-128+r} . k_j ),  j <= n-128+r
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
constexpr int kStages = 3;                         // K ring
constexpr uint32_t kStageBytes = 32 * 32 * 4;      // per-warp transpose buffer
constexpr uint32_t kSmemBytes = 1024 + kTile + kStages * kTile + kEpiWarps * kStageBytes;
constexpr uint32_t kTmemCols = 256;                // two 128-column S buffers

struct Bars {
  uint64_t q_full;
  uint64_t k_full[kStages], k_empty[kStages];
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

// grid: (hq, chunks). CTA (h, chunk) covers key blocks [chunk*C, chunk*C + C).
template <bool kWrite>
__global__ void __launch_bounds__(kThreads, 1)
    proxy_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk, int n, int group,
                 float c_log2, float* __restrict__ pmap, float2* __restrict__ part,
                 const float2* __restrict__ stats, DevStatus* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = base;
  uint8_t* sK = base + kTile;
  float* sStage = reinterpret_cast<float*>(base + kTile + kStages * kTile);
  __shared__ Bars bars;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.x, chunk = blockIdx.y, nchunks = gridDim.y;
  const int g = h / group;
  const int nb = n / kB;
  const int kb0 = chunk * kProxyChunk;
  const int T = min(nb, kb0 + kProxyChunk) - kb0;

  if (threadIdx.x == 0) {
    bars.abort = 0;
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
      mbar_arrive_expect_tx(&bars.q_full, kTile);
      tma_load_3d(sQ, &tq, &bars.q_full, 0, n - kB, h);
      tma_load_3d(sQ + kHalf, &tq, &bars.q_full, 64, n - kB, h);
      for (int t = 0; t < T; ++t) {
        const int s = t % kStages;
        const uint32_t use = t / kStages;
        if (!mbar_wait(&bars.k_empty[s], (use & 1u) ^ 1u, &bars.abort)) {
          fail(&bars.abort, status, 0x101);
          break;
        }
        mbar_arrive_expect_tx(&bars.k_full[s], kTile);
        uint8_t* dst = sK + s * kTile;
        tma_load_3d(dst, &tk, &bars.k_full[s], 0, (kb0 + t) * kB, g);
        tma_load_3d(dst + kHalf, &tk, &bars.k_full[s], 64, (kb0 + t) * kB, g);
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
    float M = 0.f, inv_l = 0.f;
    if (kWrite) {
      const float2 st = stats[static_cast<size_t>(h) * kB + r];
      M = st.x;
      inv_l = st.y;
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
      const bool diag = (kb == nb - 1);  // causal edge: keys j > n-128+r are masked
#pragma unroll 1
      for (int cc = 0; cc < 2; ++cc) {
        const int col0 = half * 64 + cc * 32;
        uint32_t v[32];
        tmem_ld32(tmem + lane_addr + b * 128 + col0, v);
        float x[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const float val = __uint_as_float(v[e]) * c_log2;
          x[e] = (diag && col0 + e > r) ? -INFINITY : val;
        }
        if (!kWrite) {
          float mx = x[0];
#pragma unroll
          for (int e = 1; e < 32; ++e) mx = fmaxf(mx, x[e]);
          if (mx > m_run) {
            l_run *= ex2_approx(m_run - mx);
            m_run = mx;
          }
          if (m_run != -INFINITY) {
            float sum = 0.f;
#pragma unroll
            for (int e = 0; e < 32; ++e) sum += ex2_approx(x[e] - m_run);
            l_run += sum;
          }
        } else {
          // Row `lane` of this warp's 32x32 block into the transpose buffer
          // (16-byte chunks XOR-swizzled by row to spread the banks).
#pragma unroll
          for (int c4 = 0; c4 < 8; ++c4) {
            float4 p;
            p.x = ex2_approx(x[4 * c4 + 0] - M) * inv_l;
            p.y = ex2_approx(x[4 * c4 + 1] - M) * inv_l;
            p.z = ex2_approx(x[4 * c4 + 2] - M) * inv_l;
            p.w = ex2_approx(x[4 * c4 + 3] - M) * inv_l;
            reinterpret_cast<float4*>(stg + lane * 32)[c4 ^ (lane & 7)] = p;
          }
          __syncwarp();
          const int c4 = lane & 7;
#pragma unroll
          for (int it = 0; it < 8; ++it) {
            const int R = it * 4 + (lane >> 3);
            const float4 p = reinterpret_cast<const float4*>(stg + R * 32)[c4 ^ (R & 7)];
            float* dst = pmap + (static_cast<size_t>(h) * kB + quarter * 32 + R) * static_cast<size_t>(n) +
                         static_cast<size_t>(kb) * kB + col0 + c4 * 4;
            *reinterpret_cast<float4*>(dst) = p;
          }
          __syncwarp();
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.s_empty[b]);
    }
    if (!kWrite) part[(static_cast<size_t>(h) * kB + r) * (2 * nchunks) + 2 * chunk + half] = make_float2(m_run, l_run);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
}

// Combines the per-chunk (max, sum) pairs of each row: M = max m_c,
// L = sum l_c * 2^(m_c - M); stores (M, 1/L).
__global__ void proxy_combine(const float2* __restrict__ part, float2* __restrict__ stats, int rows, int nparts) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= rows) return;
  const float2* p = part + static_cast<size_t>(idx) * nparts;
  float M = -INFINITY;
  for (int c = 0; c < nparts; ++c) M = fmaxf(M, p[c].x);
  float L = 0.f;
  for (int c = 0; c < nparts; ++c)
    if (p[c].x != -INFINITY) L += p[c].y * ex2_approx(p[c].x - M);
  stats[idx] = make_float2(M, 1.0f / L);
}

}  // namespace

cudaError_t launch_proxy(const crisp_shape& s, const TmaMaps& maps, float* pmap, char* ws, cudaStream_t st) {
  const ScratchLayout L = scratch_layout(s);
  const int nb = num_blocks(s.seq_len);
  const int chunks = proxy_chunks(nb);
  const float c_log2 = s.scale * 1.4426950408889634f;  // scale * log2(e): softmax in base 2
  auto* part = reinterpret_cast<float2*>(ws + L.proxy_part);
  auto* stats = reinterpret_cast<float2*>(ws + L.proxy_stats);
  auto* status = reinterpret_cast<DevStatus*>(ws + L.status);
  cudaError_t e = cudaFuncSetAttribute(proxy_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(proxy_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  const dim3 grid(s.hq, chunks);
  const int group = s.hq / s.hkv;
  proxy_kernel<false><<<grid, kThreads, kSmemBytes, st>>>(maps.q, maps.k, s.seq_len, group, c_log2, pmap, part,
                                                          stats, status);
  const int rows = s.hq * kB;
  proxy_combine<<<(rows + 127) / 128, 128, 0, st>>>(part, stats, rows, 2 * chunks);
  proxy_kernel<true><<<grid, kThreads, kSmemBytes, st>>>(maps.q, maps.k, s.seq_len, group, c_log2, pmap, part,
                                                         stats, status);
  return cudaGetLastError();
}

}  // namespace crisp
