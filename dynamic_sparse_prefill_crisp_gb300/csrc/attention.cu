// A8/A9. Causal GQA block-sparse (or dense) attention on the 5th-generation
// tensor cores (CRISP paper page on ai.info, "Why This Matters": exact
// softmax attention over the blocks the method selects; the dense path is the
// exact FlashAttention-style baseline the paper measures against).
//
// One CTA per (head h, query block qb), two CTAs per SM so that one CTA's
// softmax overlaps the other's matrix products. Per selected key block kb:
//   S  = Q K_kb^T        tcgen05.mma, A = Q (smem), B = K (smem), D = S (TMEM)
//   P  = 2^(S*c - m)     softmax warps: TMEM -> registers -> bf16 -> TMEM (each warp
//                        over its own S columns)
//   O += P V_kb          tcgen05.mma, A = P (TMEM), B = V (smem, MN-major), D = O (TMEM)
// K and V tiles arrive by TMA at row coordinate kb*128 (gather by block index);
// rows past n in a short last block are filled with zeros, the causal mask
// hides those keys and their query rows are not stored.
// The reference max m is the first block's exact row max and is raised
// lazily after that: each later block is exponentiated at the current m and
// stored chunk by chunk, with no agreement between the two warps of a row;
// only a warp that finds some chunk's row sum past 2^16 (so possibly one
// p > 2^16) holds back, waits for its partner's P, moves m to the max of its
// unstored scores, rescales the row's stored P, O and its row sum, and
// recomputes the rest; the partner follows the new m at its next block.
// Every p stays <= 2^16 and O/l is exact.
//
// Warp roles: 0-7 softmax + epilogue (warp w owns TMEM lanes / rows
// 32*(w%4)..+31 and columns 64*(w/4)..+63), 8 TMA producer, 9 MMA issuer (and
// TMEM owner).
#include <cuda_bf16.h>

#include "common.cuh"
#include "ptx.cuh"

namespace crisp {
using namespace ptx;

namespace {

constexpr int kSoftmaxWarps = 8;  // two per TMEM lane quarter (column halves)
constexpr int kThreads = (kSoftmaxWarps + 2) * 32;
constexpr int kTmaWarp = kSoftmaxWarps, kMmaWarp = kSoftmaxWarps + 1;
constexpr uint32_t kTile = kB * kD * 2;  // 32 KB bf16 tile
constexpr uint32_t kHalf = kTile / 2;
constexpr uint32_t kSmemBytes = 1024 + 3 * kTile;  // Q, K, V (+ alignment slack)
constexpr uint32_t kTmemCols = 256;                // S/P [0,128), O [128,256)
constexpr float kRescaleSum = 65536.0f;  // 2^16: the largest chunk row sum kept at the current reference

struct Bars {
  uint64_t q_full, k_full, k_empty, v_full, v_empty, s_full, p_full, pv_done, drain;
  uint64_t qdone[4];     // per lane quarter: both warps have stored their P of the block
  uint32_t tmem_base;
  int count;
  int has_diag;
  int abort;
  uint32_t qov[4][2];    // [lane quarter][column half]: j + 1 when that warp's block j needed a new reference
  float mrow[kB];        // the reference m of each row, as last moved
  float xmax[2][2][kB];  // [first block / both halves redone][column half][row]: partial row maxima
  float xsum[2][kB];     // [column half][row]: partial row sums (epilogue)
};

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, int* abort) {
  const bool ok = mbar_wait(bar, parity, abort);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void fail(int* abort, DevStatus* st, uint32_t where) {
  *reinterpret_cast<volatile int*>(abort) = 1;
  report_error(st, CRISP_ERR_TIMEOUT, where);
}

// p = 2^(s*c - m) for 32 scores of this thread's row: a packed FMA and a
// packed add per element pair, one MUFU per element. pk: bf16 pairs (even key
// low); sum += the fp32 sum of the 32 values.
__device__ __forceinline__ void p_exp32(const uint32_t (&sv)[32], float c, float neg_m, uint32_t* pk, float& sum) {
  float sa0 = 0.f, sa1 = 0.f, sb0 = 0.f, sb1 = 0.f;
#pragma unroll
  for (int e = 0; e < 32; e += 4) {
    float x0, x1, x2, x3;
    ffma2(x0, x1, __uint_as_float(sv[e]), __uint_as_float(sv[e + 1]), c, c, neg_m, neg_m);
    ffma2(x2, x3, __uint_as_float(sv[e + 2]), __uint_as_float(sv[e + 3]), c, c, neg_m, neg_m);
    const float p0 = ex2_approx(x0), p1 = ex2_approx(x1), p2 = ex2_approx(x2), p3 = ex2_approx(x3);
    fadd2_acc(sa0, sa1, p0, p1);
    fadd2_acc(sb0, sb1, p2, p3);
    pk[e / 2] = pack_bf16x2(p0, p1);
    pk[e / 2 + 1] = pack_bf16x2(p2, p3);
  }
  sum += (sa0 + sa1) + (sb0 + sb1);
}

// 32 S columns of this thread's row from TMEM; on the diagonal block the keys
// above the row (column index col0 + e > r) are set to -inf.
__device__ __forceinline__ void load_s32(uint32_t taddr, bool diag, int col0, int r, uint32_t (&sv)[32]) {
  tmem_ld32(taddr, sv);
  if (diag) {
#pragma unroll
    for (int e = 0; e < 32; ++e)
      if (col0 + e > r) sv[e] = 0xff800000u;  // -inf
  }
}

// Keys above the row on the diagonal block (column index col0 + e > r) -> -inf.
__device__ __forceinline__ void mask_diag32(int col0, int r, uint32_t (&sv)[32]) {
#pragma unroll
  for (int e = 0; e < 32; ++e)
    if (col0 + e > r) sv[e] = 0xff800000u;
}

// Largest of 32 raw scores.
__device__ __forceinline__ float max32(const uint32_t (&sv)[32]) {
  float ma = fmax3(__uint_as_float(sv[0]), __uint_as_float(sv[1]), __uint_as_float(sv[2]));
  float mb = fmax3(__uint_as_float(sv[3]), __uint_as_float(sv[4]), __uint_as_float(sv[5]));
#pragma unroll
  for (int e = 6; e + 3 < 32; e += 4) {
    ma = fmax3(ma, __uint_as_float(sv[e]), __uint_as_float(sv[e + 1]));
    mb = fmax3(mb, __uint_as_float(sv[e + 2]), __uint_as_float(sv[e + 3]));
  }
  return fmax3(fmax3(ma, mb, __uint_as_float(sv[30])), __uint_as_float(sv[31]), -INFINITY);
}

// 16 columns of bf16 pairs scaled by f (and repacked).
__device__ __forceinline__ void scale_bf16x32(uint32_t (&pk)[16], float f) {
#pragma unroll
  for (int e = 0; e < 16; ++e)
    pk[e] = pack_bf16x2(__uint_as_float(pk[e] << 16) * f, __uint_as_float(pk[e] & 0xffff0000u) * f);
}

// The reference and sum of one softmax row (a thread's partial sum).
struct RowState {
  float m, l;
};

// A new reference for the rows of lane quarter `quarter` (rare; out of line so
// that the common loop keeps its registers). Called by a warp in whose block
// some p would pass 2^16 (a chunk row sum past 2^16), or whose rows' reference
// the other warp moved in the last block, once the other warp of the rows has
// stored its P (qdone). The warp's scores are in TMEM: chunk 0 at columns
// 0..31, chunk 1 (put back) at 32..63. The rows' new reference is the max of
// the old one and these scores -- of both warps when both are here (then they
// exchange it through xmax and each fixes its own columns); otherwise this
// warp also rescales the other warp's P and O columns (TMEM lanes belong to
// the quarter, so it can) and the other warp follows the new reference (mrow)
// at its next block. The other warp's stored P holds p <= 2^16 at the old
// reference and is rescaled in place by f = 2^(m_old - m_new); this warp's P
// is formed again from its scores (chunk 1 first: its P goes over chunk 1's
// own scores, chunk 0's over chunk 1's first half). Every p stays below 2^16
// and O/l is exact. Returns the new reference and the row sum with this
// block's part.
__device__ __noinline__ RowState new_reference(RowState st, uint32_t tmem, uint32_t lane_addr, int half, int r,
                                               bool diag, bool both, float c_log2, float* xmine, const float* xother,
                                               int pair_bar, float* mrow) {
  const uint32_t s_addr = tmem + lane_addr + half * 64, p_addr = s_addr + 32;
  const int col0 = half * 64;
  uint32_t sv[32], pk[16];
  float mc = -INFINITY;
#pragma unroll 1
  for (int cc = 0; cc < 2; ++cc) {
    load_s32(s_addr + cc * 32, diag, col0 + cc * 32, r, sv);
    mc = fmaxf(mc, max32(sv));
  }
  if (both) {
    *xmine = mc;
    named_bar_sync(pair_bar, 64);
    mc = fmaxf(mc, *xother);
  }
  const float m_new = fmaxf(st.m, mc * c_log2);
  const float f = ex2_approx(st.m - m_new);
  float t = 0.f;
#pragma unroll 1
  for (int cc = 1; cc >= 0; --cc) {
    load_s32(s_addr + cc * 32, diag, col0 + cc * 32, r, sv);
    p_exp32(sv, c_log2, -m_new, pk, t);
    tmem_st16(p_addr + cc * 16, pk);
  }
  // O columns to rescale: this warp's half, and the other half too when the
  // other warp is not here (then also its stored P).
  if (!both) {
    const uint32_t other = tmem + lane_addr + (half ^ 1) * 64 + 32;
#pragma unroll 1
    for (int cc = 0; cc < 2; ++cc) {
      tmem_ld16(other + cc * 16, pk);
      scale_bf16x32(pk, f);
      tmem_st16(other + cc * 16, pk);
    }
  }
#pragma unroll 1
  for (int oh = 0; oh < (both ? 1 : 2); ++oh) {
    const uint32_t oa = tmem + lane_addr + 128 + (oh == 0 ? half : half ^ 1) * 64;
#pragma unroll 1
    for (int cc = 0; cc < 4; ++cc) {
      tmem_ld16(oa + cc * 16, pk);
#pragma unroll
      for (int e = 0; e < 16; ++e) pk[e] = __float_as_uint(__uint_as_float(pk[e]) * f);
      tmem_st16(oa + cc * 16, pk);
    }
  }
  *mrow = m_new;
  tmem_st_wait();
  return RowState{m_new, st.l * f + t};
}

// Bits of row word w restricted to key blocks <= qb (row: W words).
__device__ __forceinline__ uint32_t row_word(const uint32_t* row, bool dense, int w, int qb, int W,
                                             DevStatus* status) {
  uint32_t bits = dense ? 0xffffffffu : (CRISP_CHECK(w < W, status, 0x211) ? row[w] : 0u);
  if (w == (qb >> 5) && (qb & 31) != 31) bits &= (1u << ((qb & 31) + 1)) - 1u;
  return bits;
}

__global__ void __launch_bounds__(kThreads, 2)
    attention_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                     const __grid_constant__ CUtensorMap tv, int n, int group, float c_log2,
                     const uint32_t* __restrict__ rowbits, const int32_t* __restrict__ order, int dense,
                     __nv_bfloat16* __restrict__ out, int64_t o_hs, int64_t o_ts, DevStatus* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = base;
  uint8_t* sK = base + kTile;
  uint8_t* sV = base + 2 * kTile;
  __shared__ Bars bars;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nb = (n + kB - 1) / kB, W = (nb + 31) / 32;  // a short last block when 128 does not divide n
  // Work item: the schedule order[] or, without one, the same kv-group-major
  // order (kv group by kv group, query blocks descending within a group).
  int item;
  if (order != nullptr) {
    item = order[blockIdx.x];
    // (checking build) a work item outside [0, hq*nb) is replaced by 0
    if (!CRISP_CHECK(item >= 0 && item < static_cast<int>(gridDim.x), status, 0x210)) item = 0;
  } else {
    const int t = static_cast<int>(blockIdx.x), per_group = group * nb;
    const int rem = t % per_group;
    item = ((t / per_group) * group + rem % group) * nb + (nb - 1 - rem / group);
  }
  const int h = item / nb, qb = item % nb;
  const int g = h / group;
  const uint32_t* row = rowbits ? rowbits + static_cast<size_t>(item) * W : nullptr;
  const bool is_dense = dense != 0;

  if (threadIdx.x == 0) {
    bars.abort = 0;
    mbar_init(&bars.q_full, 1);
    mbar_init(&bars.k_full, 1);
    mbar_init(&bars.k_empty, 1);
    mbar_init(&bars.v_full, 1);
    mbar_init(&bars.v_empty, 1);
    mbar_init(&bars.s_full, 1);
    mbar_init(&bars.p_full, kSoftmaxWarps);
    mbar_init(&bars.pv_done, 1);
    for (int qq = 0; qq < 4; ++qq) {
      mbar_init(&bars.qdone[qq], 2);
      bars.qov[qq][0] = bars.qov[qq][1] = 0;
    }
    mbar_init(&bars.drain, 1);
    fence_mbar_init();
  }
  if (warp == kTmaWarp) {
    int cnt = 0;
    for (int w = lane; w <= (qb >> 5); w += 32) cnt += __popc(row_word(row, is_dense, w, qb, W, status));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
    if (lane == 0) {
      bars.count = cnt;
      bars.has_diag = (row_word(row, is_dense, qb >> 5, qb, W, status) >> (qb & 31)) & 1u;
    }
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&bars.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars.tmem_base;
  const int count = bars.count;

  if (warp == kTmaWarp) {
    if (lane == 0 && count > 0) {
      prefetch_tmap(&tq);
      prefetch_tmap(&tk);
      prefetch_tmap(&tv);
      // (checking build) a tile outside q, k or v is not copied; its barrier
      // phase completes without data and the status word says why.
      const int hq = static_cast<int>(gridDim.x) / nb;
      if (CRISP_CHECK(qb * kB < n && h < hq, status, 0x212)) {
        mbar_arrive_expect_tx(&bars.q_full, kTile);
        tma_load_3d(sQ, &tq, &bars.q_full, 0, qb * kB, h);
        tma_load_3d(sQ + kHalf, &tq, &bars.q_full, 64, qb * kB, h);
      } else {
        mbar_arrive(&bars.q_full);
      }
      const bool kv_ok = CRISP_CHECK(g < hq / group, status, 0x213);
      int j = 0, nk = 0, nv = 0;  // blocks started, K and V loads issued
      bool ok = true;
      for (int w = 0; ok && w <= (qb >> 5); ++w) {
        uint32_t bits = row_word(row, is_dense, w, qb, W, status);
        while (bits) {
          const int kb = w * 32 + __ffs(bits) - 1;
          bits &= bits - 1;
          const uint32_t par = (static_cast<uint32_t>(j) & 1u) ^ 1u;
          if (!mbar_wait(&bars.k_empty, par, &bars.abort)) {
            fail(&bars.abort, status, 0x201);
            ok = false;
            break;
          }
          const bool tile_ok = kv_ok && CRISP_CHECK(kb * kB < n, status, 0x214);
          ++nk;
          if (tile_ok) {
            mbar_arrive_expect_tx(&bars.k_full, kTile);
            tma_load_3d(sK, &tk, &bars.k_full, 0, kb * kB, g);
            tma_load_3d(sK + kHalf, &tk, &bars.k_full, 64, kb * kB, g);
          } else {
            mbar_arrive(&bars.k_full);
          }
          if (!mbar_wait(&bars.v_empty, par, &bars.abort)) {
            fail(&bars.abort, status, 0x202);
            ok = false;
            break;
          }
          ++nv;
          if (tile_ok) {
            mbar_arrive_expect_tx(&bars.v_full, kTile);
            tma_load_3d(sV, &tv, &bars.v_full, 0, kb * kB, g);
            tma_load_3d(sV + kHalf, &tv, &bars.v_full, 64, kb * kB, g);
          } else {
            mbar_arrive(&bars.v_full);
          }
          ++j;
        }
      }
      // Every copy issued has landed before the CTA may exit: on the normal
      // path the consumers already waited for them; after a timeout they may
      // not have. Bounded waits that ignore the abort flag.
      const int never = 0;
      mbar_wait(&bars.q_full, 0, &never);
      if (nk > 0) mbar_wait(&bars.k_full, static_cast<uint32_t>(nk - 1) & 1u, &never);
      if (nv > 0) mbar_wait(&bars.v_full, static_cast<uint32_t>(nv - 1) & 1u, &never);
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0 && count > 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(128, 128, false, true);
      bool ok = mbar_wait(&bars.q_full, 0, &bars.abort);
      if (!ok) fail(&bars.abort, status, 0x203);
      const uint32_t qa = smem_u32(sQ), ka = smem_u32(sK), va = smem_u32(sV);
      for (int j = 0; ok && j < count; ++j) {
        const uint32_t par = static_cast<uint32_t>(j) & 1u;
        // S (aliased by P_{j-1}) is free once PV_{j-1} has completed.
        if ((j > 0 && !mbar_wait(&bars.pv_done, par ^ 1u, &bars.abort)) ||
            !mbar_wait(&bars.k_full, par, &bars.abort)) {
          fail(&bars.abort, status, 0x204);
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
          umma_ss(tmem, sdesc_sw128(qa + off, 16, 1024), sdesc_sw128(ka + off, 16, 1024), idesc_qk, kk > 0);
        }
        umma_commit(&bars.k_empty);
        umma_commit(&bars.s_full);
        const bool got = mbar_wait(&bars.p_full, par, &bars.abort);
        if (!got || !mbar_wait(&bars.v_full, par, &bars.abort)) {
          fail(&bars.abort, status, 0x205);
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          // A = P rows in TMEM (bf16 pairs, 8 columns per 16 keys; keys
          // 0..63 at columns 32..63, keys 64..127 at columns 96..127);
          // B = V, 16 keys x 128 features, MN-major: 16 rows of 128 B per
          // step, the second 64-feature half kHalf bytes further.
          umma_ts(tmem + 128, tmem + (kk >> 2) * 64 + 32 + (kk & 3) * 8, sdesc_sw128(va + kk * 2048, kHalf, 1024),
                  idesc_pv,
                  (j > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(&bars.v_empty);
        umma_commit(&bars.pv_done);
      }
      // The last phase of s_full: O is final. After a failure the softmax
      // warps leave on the abort flag instead.
      if (!*reinterpret_cast<volatile int*>(&bars.abort)) umma_commit(&bars.s_full);
      umma_commit(&bars.drain);
      if (!mbar_wait(&bars.drain, 0, &bars.abort)) fail(&bars.abort, status, 0x206);
    }
  } else {
    // Softmax warps, two per TMEM lane quarter: warp w owns query rows
    // 32*(w%4)..+31 and score / output columns 64*(w/4)..+63. The two warps
    // of a quarter exchange partial row maxima through shared memory (named
    // barrier 1 + quarter); their partial row sums are added at the end.
    const int quarter = warp & 3, half = warp >> 2;
    const int r = quarter * 32 + lane;
    const int pair_bar = 1 + quarter;
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t s_addr = tmem + lane_addr + half * 64;        // 64 S columns
    const uint32_t p_addr = s_addr + 32;                         // 32 P columns (bf16 pairs) over the last of them
    const uint32_t o_addr = tmem + lane_addr + 128 + half * 64;  // 64 O columns
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    // One phase of s_full per block (its scores), then one when O is final.
    for (int j = 0; count > 0 && j <= count; ++j) {
      if (!warp_wait(&bars.s_full, static_cast<uint32_t>(j) & 1u, &bars.abort)) {
        if (lane == 0) fail(&bars.abort, status, 0x207);
        ok = false;
        break;
      }
      tc_fence_after();
      if (j == count) {
        // O is final; the row sum follows the last reference of the row.
        const float mr = bars.mrow[r];
        if (mr > m_ref) l *= ex2_approx(m_ref - mr);
        break;
      }
      const bool diag = bars.has_diag && j == count - 1;  // ascending order: qb is last
      const int col0 = half * 64;
      if (j == 0) {
        // First block: the exact row max over both column halves (partial
        // maxima exchanged through shared memory) is the reference m.
        float pm = -INFINITY;
#pragma unroll 1
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t sv[32];
          load_s32(s_addr + cc * 32, diag, col0 + cc * 32, r, sv);
          pm = fmaxf(pm, max32(sv));
        }
        bars.xmax[0][half][r] = pm;
        named_bar_sync(pair_bar, 64);
        m_ref = fmaxf(pm, bars.xmax[0][half ^ 1][r]) * c_log2;  // c > 0: max(s*c) = max(s)*c
        if (half == 0) bars.mrow[r] = m_ref;
        uint32_t pk[32];
        float bsum = 0.f;
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t sv[32];
          load_s32(s_addr + cc * 32, diag, col0 + cc * 32, r, sv);
          p_exp32(sv, c_log2, -m_ref, pk + cc * 16, bsum);
        }
        tmem_st32(p_addr, pk);
        l = bsum;
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.p_full);
        continue;
      }
      // Later blocks: P at the current reference, each 32-key chunk stored
      // as soon as it is formed, without waiting for the other warp of the
      // row and without a test first. P goes over chunk 1's scores (columns
      // 32..63): chunk 0's P once chunk 1's scores are in registers, chunk
      // 1's right after. A block in which some chunk row sum passes 2^16 (any
      // p that could pass 2^16, or a non-finite value), or whose reference
      // the other warp moved in the last block, takes the slow path below
      // with chunk 0's scores still in TMEM and chunk 1's put back from
      // registers.
      uint32_t sv[32], pk[16], pk1[16];
      float s0 = 0.f, s1 = 0.f;
      // The other warp may have moved the rows' reference (and rescaled this
      // warp's P and O) in the last block; the read overlaps the loads and
      // the exponentials.
      tmem_ld32_async(s_addr, sv);
      const float mr = bars.mrow[r];
      tmem_ld_wait32(sv);
      if (diag) mask_diag32(col0, r, sv);
      p_exp32(sv, c_log2, -m_ref, pk, s0);
      tmem_ld32_async(s_addr + 32, sv);
      tmem_ld_wait32(sv);
      tmem_st16(p_addr, pk);
      if (diag) mask_diag32(col0 + 32, r, sv);
      p_exp32(sv, c_log2, -m_ref, pk1, s1);
      tmem_st16(p_addr + 16, pk1);
      const bool moved = mr > m_ref;
      const bool ov = __any_sync(0xffffffffu, !(s0 <= kRescaleSum) || !(s1 <= kRescaleSum) || moved);
      if (ov) {
        if (lane == 0) *reinterpret_cast<volatile uint32_t*>(&bars.qov[quarter][half]) = j + 1;
        tmem_st32(s_addr + 32, sv);  // chunk 1's scores back (masked keys stay masked: -inf)
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (!ov) {
        l += s0 + s1;
        if (lane == 0) {
          mbar_arrive(&bars.p_full);
          mbar_arrive(&bars.qdone[quarter]);
        }
        continue;
      }
      // A new reference (rare): this warp holds back its arrival on p_full,
      // so PV waits, until its rows are consistent again. First catch up
      // with a reference the other warp moved in the last block.
      if (moved) {
        l *= ex2_approx(m_ref - mr);
        m_ref = mr;
      }
      if (lane == 0) mbar_arrive(&bars.qdone[quarter]);
      if (!warp_wait(&bars.qdone[quarter], static_cast<uint32_t>(j - 1) & 1u, &bars.abort)) {
        if (lane == 0) fail(&bars.abort, status, 0x209);
        ok = false;
        break;
      }
      tc_fence_after();
      const bool both =
          *reinterpret_cast<volatile uint32_t*>(&bars.qov[quarter][half ^ 1]) == static_cast<uint32_t>(j + 1);
      const RowState st = new_reference(RowState{m_ref, l}, tmem, lane_addr, half, r, diag, both, c_log2,
                                        &bars.xmax[1][half][r], &bars.xmax[1][half ^ 1][r], pair_bar, &bars.mrow[r]);
      m_ref = st.m;
      l = st.l;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.p_full);
    }
    // Epilogue: O / l -> bf16 for this warp's 64 columns, staged per warp
    // through shared memory (the K tile is no longer needed) so that each
    // store instruction writes four 128-byte row segments.
    const bool have = ok && count > 0;  // the loop ended on O's final phase
    bars.xsum[half][r] = l;
    named_bar_sync(pair_bar, 64);
    const float l_row = l + bars.xsum[half ^ 1][r];
    uint4* stg = reinterpret_cast<uint4*>(sK + warp * (32 * 128));  // 32 rows x 128 B
    const float inv_l = have && l_row > 0.f ? 1.0f / l_row : 0.f;
#pragma unroll 1
    for (int cc = 0; cc < 2; ++cc) {
      uint32_t v[32];
      if (have) {
        tmem_ld32(o_addr + cc * 32, v);
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] = 0u;
      }
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        uint4 u;
        u.x = pack_bf16x2(__uint_as_float(v[q4 * 8 + 0]) * inv_l, __uint_as_float(v[q4 * 8 + 1]) * inv_l);
        u.y = pack_bf16x2(__uint_as_float(v[q4 * 8 + 2]) * inv_l, __uint_as_float(v[q4 * 8 + 3]) * inv_l);
        u.z = pack_bf16x2(__uint_as_float(v[q4 * 8 + 4]) * inv_l, __uint_as_float(v[q4 * 8 + 5]) * inv_l);
        u.w = pack_bf16x2(__uint_as_float(v[q4 * 8 + 6]) * inv_l, __uint_as_float(v[q4 * 8 + 7]) * inv_l);
        const int chunk = cc * 4 + q4;  // 16-byte chunk of this warp's 128-byte row part
        stg[lane * 8 + (chunk ^ (lane & 7))] = u;
      }
    }
    __syncwarp();
    const int chunk = lane & 7;
#pragma unroll 4
    for (int it = 0; it < 8; ++it) {
      const int R = it * 4 + (lane >> 3);
      const uint4 u = stg[R * 8 + (chunk ^ (R & 7))];
      const int tok = qb * kB + quarter * 32 + R;
      if (tok >= n) continue;  // rows past the end of a short last block
      const int64_t idx = static_cast<int64_t>(h) * o_hs + static_cast<int64_t>(tok) * o_ts + half * 64 + chunk * 8;
      // extent of out under its strides: (hq - 1) * o_hs + (n - 1) * o_ts + 128 elements
      if (!CRISP_CHECK(idx >= 0 && idx + 8 <= (static_cast<int64_t>(gridDim.x) / nb - 1) * o_hs +
                                                   static_cast<int64_t>(n - 1) * o_ts + kD,
                       status, 0x215))
        continue;
      *reinterpret_cast<uint4*>(out + idx) = u;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

cudaError_t launch_attention(const crisp_shape& s, const TmaMaps& maps, const uint32_t* rowbits,
                             const int32_t* order, void* out, char* ws, bool dense, cudaStream_t st) {
  const ScratchLayout L = scratch_layout(s);
  const int nb = num_blocks(s.seq_len);
  auto* status = reinterpret_cast<DevStatus*>(ws + L.status);
  if (dense) order = nullptr;
  cudaError_t e = cudaFuncSetAttribute(attention_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  const int items = s.hq * nb;
  attention_kernel<<<items, kThreads, kSmemBytes, st>>>(
      maps.q, maps.k, maps.v, s.seq_len, s.hq / s.hkv, s.scale * 1.4426950408889634f,
      dense ? nullptr : rowbits, order, dense ? 1 : 0, static_cast<__nv_bfloat16*>(out), s.o_head_stride,
      s.o_tok_stride, status);
  return cudaGetLastError();
}

}  // namespace crisp
