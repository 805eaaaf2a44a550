// A8/A9. Causal GQA block-sparse (or dense) attention on the 5th-generation
// tensor cores (CRISP paper page on ai.info, "Why This Matters": exact
// softmax attention over the blocks the method selects; the dense path is the
// exact FlashAttention-style baseline the paper measures against).
//
// One CTA per (head h, query block qb), two CTAs per SM. Each selected key
// block kb is taken as two sub-blocks of 64 keys, and the two sub-blocks'
// scores have TMEM buffers of their own, so the scores of the next sub-block
// are formed while the softmax warps work on the current one:
//   S_s = Q K_kb,s^T     tcgen05.mma (N = 64), A = Q (smem), B = K (smem), D = S_s (TMEM)
//   P_s = 2^(S_s*c - m)  softmax warps: TMEM -> registers -> bf16 -> TMEM (over their own S columns)
//   O  += P_s V_kb,s     tcgen05.mma (K = 64), A = P_s (TMEM), B = V (smem, MN-major), D = O (TMEM)
// K and V arrive by TMA in 64-key halves at row coordinate kb*128 + 64s (a
// gather by block index); rows past n in a short last block are filled with
// zeros, the causal mask hides those keys and their query rows are not
// stored.
//
// The reference m of a row is the exact max of its first sub-block and stays
// fixed: later sub-blocks are exponentiated at it with no exchange between
// warps. A chunk whose row sum passes 2^64 (a score more than 64 above m in
// base-2 units, where bf16 P or the fp32 sums could overflow) marks the CTA;
// it then runs the row again in two passes: the exact row max over every
// selected block first (scores only), then the sum at that max (every p <= 1).
//
// Warp roles: 0-7 softmax + epilogue (warp w owns TMEM lanes / rows
// 32*(w%4)..+31, score columns 32*(w/4)..+31 of each sub-block and output
// columns 64*(w/4)..+63), 8 TMA producer, 9 MMA issuer (and TMEM owner).
#include <cuda_bf16.h>

#include "common.cuh"
#include "ptx.cuh"

namespace crisp {
using namespace ptx;

namespace {

constexpr int kSoftmaxWarps = 8;  // two per TMEM lane quarter (32-column chunks of a sub-block)
constexpr int kThreads = (kSoftmaxWarps + 2) * 32;
constexpr int kTmaWarp = kSoftmaxWarps, kMmaWarp = kSoftmaxWarps + 1;
constexpr int kSubKeys = kB / 2;                       // keys per sub-block
constexpr uint32_t kTile = kB * kD * 2;                // 32 KB bf16 tile (Q)
constexpr uint32_t kHalf = kTile / 2;                  // Q: one 64-feature half
constexpr uint32_t kSub = kTile / 2;                   // K or V: one 64-key sub-block (both feature halves)
constexpr uint32_t kSubHalf = kSub / 2;                // 64 keys x 64 features
constexpr uint32_t kSmemBytes = 1024 + kTile + 4 * kSub;  // Q, K[2], V[2] (+ alignment slack)
constexpr uint32_t kTmemCols = 256;                    // S/P [0,64) and [64,128), O [128,256)
constexpr float kOverflowSum = 0x1p64f;                // chunk row sum past which the row is redone

enum Mode : int { kFast = 0, kMaxOnly = 1, kFixed = 2 };

struct Bars {
  uint64_t q_full;
  uint64_t k_full[2], v_full[2], v_empty[2];  // a K slot is free again once s_full of its sub-block completes
  uint64_t s_full[2], p_full[2];
  uint64_t o_full, drain;
  uint64_t xbar[4];      // per lane quarter: both warps have written their partial row maxima
  uint32_t tmem_base;
  int count;
  int has_diag;
  int abort;
  int redo;              // a chunk row sum passed kOverflowSum (fast pass)
  float xmax[2][kB];     // [chunk][row]: partial row maxima
  float xsum[2][kB];     // [chunk][row]: partial row sums (epilogue)
};

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, int* abort) {
  const bool ok = mbar_wait(bar, parity, abort);
  return __all_sync(0xffffffffu, ok);
}

// Two 16-bit counters (one per slot s = 0, 1) in one register, so that a
// slot picked at run time costs shifts, not a local-memory array.
struct SlotCounts {
  uint32_t v = 0u;
  __device__ __forceinline__ uint32_t parity(int s) const { return (v >> (16 * s)) & 1u; }
  __device__ __forceinline__ void inc(int s) { v += 1u << (16 * s); }
};

__device__ __forceinline__ void fail(int* abort, DevStatus* st, uint32_t where) {
  *reinterpret_cast<volatile int*>(abort) = 1;
  report_error(st, CRISP_ERR_TIMEOUT, where);
}

// p = 2^(s*c - m) for 32 scores of this thread's row: a packed FMA and a
// packed add per element pair, one MUFU per element. pk: bf16 pairs (even key
// low); sum += the fp32 sum of the 32 values.
__device__ __forceinline__ void p_exp32(const uint32_t (&sv)[32], float c, float neg_m, uint32_t (&pk)[16],
                                        float& sum) {
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

// S = Q K^T over 128 features as eight K = 16 products in one asm block:
// step kk reads A (Q) and B (K) at descriptor start addresses advanced by
// 2 (kk % 4) + (kk / 4) * a_half (resp. b_half) 16-byte units; the first
// step overwrites D. One predicate pair serves all eight.
template <uint32_t kAHalf, uint32_t kBHalf>
__device__ __forceinline__ void umma_qk_x8(uint32_t d, uint64_t da, uint64_t db, uint32_t idesc) {
  asm volatile(
      "{\n\t.reg .pred f, t;\n\t.reg .b64 a, b;\n\t"
      "setp.ne.b32 f, %3, %3;\n\t"
      "setp.eq.b32 t, %3, %3;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, f;\n\t"
      "add.s64 a, %1, 2;\n\tadd.s64 b, %2, 2;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, t;\n\t"
      "add.s64 a, %1, 4;\n\tadd.s64 b, %2, 4;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, t;\n\t"
      "add.s64 a, %1, 6;\n\tadd.s64 b, %2, 6;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, t;\n\t"
      "add.s64 a, %1, %4;\n\tadd.s64 b, %2, %5;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, t;\n\t"
      "add.s64 a, %1, %4 + 2;\n\tadd.s64 b, %2, %5 + 2;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, t;\n\t"
      "add.s64 a, %1, %4 + 4;\n\tadd.s64 b, %2, %5 + 4;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, t;\n\t"
      "add.s64 a, %1, %4 + 6;\n\tadd.s64 b, %2, %5 + 6;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, t;\n\t}\n" ::"r"(d),
      "l"(da), "l"(db), "r"(idesc), "n"(kAHalf), "n"(kBHalf)
      : "memory");
}

// O += P V over 64 keys as four K = 16 products in one asm block: step kk
// reads P from TMEM column pa + 32 (kk / 2) + 8 (kk % 2) and V 16 keys
// (128 16-byte units) further on; the first step accumulates iff acc0.
__device__ __forceinline__ void umma_pv_x4(uint32_t d, uint32_t pa, uint64_t dv, uint32_t idesc, uint32_t acc0) {
  asm volatile(
      "{\n\t.reg .pred p, t;\n\t.reg .b32 ta;\n\t.reg .b64 b;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "setp.eq.b32 t, %3, %3;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t"
      "add.u32 ta, %1, 8;\n\tadd.s64 b, %2, 128;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], b, %3, t;\n\t"
      "add.u32 ta, %1, 32;\n\tadd.s64 b, %2, 256;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], b, %3, t;\n\t"
      "add.u32 ta, %1, 40;\n\tadd.s64 b, %2, 384;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], b, %3, t;\n\t}\n" ::"r"(d),
      "r"(pa), "l"(dv), "r"(idesc), "r"(acc0)
      : "memory");
}

// Keys above the row on the diagonal block (key index col0 + e > r) -> -inf.
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
  uint8_t* sK = base + kTile;            // K sub-block slots 0, 1
  uint8_t* sV = base + kTile + 2 * kSub;  // V sub-block slots 0, 1
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
    bars.redo = 0;
    mbar_init(&bars.q_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars.k_full[s], 1);
      mbar_init(&bars.v_full[s], 1);
      mbar_init(&bars.v_empty[s], 1);
      mbar_init(&bars.s_full[s], 1);
      mbar_init(&bars.p_full[s], kSoftmaxWarps);
    }
    mbar_init(&bars.o_full, 1);
    mbar_init(&bars.drain, 1);
    for (int qq = 0; qq < 4; ++qq) mbar_init(&bars.xbar[qq], 64);
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
  const int nsub = 2 * count;  // sub-blocks of one pass

  // Phase counters that persist across passes (each role counts its own).
  uint32_t kn[2] = {0u, 0u}, vn[2] = {0u, 0u};  // TMA: loads issued per slot; MMA: loads consumed per slot
  SlotCounts pn;                                // MMA: p_full phases consumed per slot
  SlotCounts sn;                                // softmax: s_full phases consumed per slot
  uint32_t drains = 0u, o_phase = 0u, x_phase = 0u;
  // Softmax state (per thread: one row, one 32-column chunk).
  const int quarter = warp & 3, chunk = warp >> 2;
  const int r = quarter * 32 + lane;
  const int pair_bar = 1 + quarter;
  // The row max over both chunks: each thread posts its partial max and
  // arrives; a bounded wait for the partner warp's 32 arrivals.
  auto row_max = [&](float partial, float& m) -> bool {
    bars.xmax[chunk][r] = partial;
    mbar_arrive(&bars.xbar[quarter]);
    const bool got = warp_wait(&bars.xbar[quarter], x_phase & 1u, &bars.abort);
    ++x_phase;
    m = fmaxf(bars.xmax[0][r], bars.xmax[1][r]);
    return got;
  };
  const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
  float m_ref = -INFINITY, l = 0.f;
  bool ok = true;

  int mode = kFast;
  for (int pass = 0; pass < 3 && count > 0; ++pass) {
    mode = pass;
    if (warp == kTmaWarp) {
      if (lane == 0) {
        // (checking build) a tile outside q, k or v is not copied; its
        // barrier phase completes without data and the status word says why.
        const int hq = static_cast<int>(gridDim.x) / nb;
        if (pass == 0) {
          prefetch_tmap(&tq);
          prefetch_tmap(&tk);
          prefetch_tmap(&tv);
          if (CRISP_CHECK(qb * kB < n && h < hq, status, 0x212)) {
            mbar_arrive_expect_tx(&bars.q_full, kTile);
            tma_load_3d(sQ, &tq, &bars.q_full, 0, qb * kB, h);
            tma_load_3d(sQ + kHalf, &tq, &bars.q_full, 64, qb * kB, h);
          } else {
            mbar_arrive(&bars.q_full);
          }
        }
        const bool kv_ok = CRISP_CHECK(g < hq / group, status, 0x213);
        (void)hq;
        // Sub-block t = 2j + s of selected block j. K runs one sub-block
        // ahead of V (K(t), then V(t-1)): the order in which the products
        // free their slots (QK(t-2) frees K slot t&1, PV(t-3) frees V slot
        // (t-1)&1). Two cursors walk the selected blocks in ascending order.
        struct Cursor {
          int w;
          uint32_t bits;
        };
        auto next_kb = [&](Cursor& c) -> int {
          while (c.bits == 0u && c.w < (qb >> 5)) {
            ++c.w;
            c.bits = row_word(row, is_dense, c.w, qb, W, status);
          }
          if (c.bits == 0u) return 0;  // not reached: exactly `count` blocks are taken
          const int kb = c.w * 32 + __ffs(c.bits) - 1;
          c.bits &= c.bits - 1u;
          return kb;
        };
        auto load = [&](bool is_k, int t, int kb) -> bool {
          const int s = t & 1;
          // K slot s is free once the scores of its last sub-block are formed
          uint64_t* empty = is_k ? &bars.s_full[s] : &bars.v_empty[s];
          uint64_t* full = is_k ? &bars.k_full[s] : &bars.v_full[s];
          uint32_t& cnt = is_k ? kn[s] : vn[s];
          if (!mbar_wait(empty, (cnt & 1u) ^ 1u, &bars.abort)) {
            fail(&bars.abort, status, is_k ? 0x201 : 0x202);
            return false;
          }
          ++cnt;
          uint8_t* dst = (is_k ? sK : sV) + s * kSub;
          const CUtensorMap* map = is_k ? &tk : &tv;
          if (kv_ok && CRISP_CHECK(kb * kB < n, status, 0x214)) {
            mbar_arrive_expect_tx(full, kSub);
            tma_load_3d(dst, map, full, 0, kb * kB + s * kSubKeys, g);
            tma_load_3d(dst + kSubHalf, map, full, 64, kb * kB + s * kSubKeys, g);
          } else {
            mbar_arrive(full);
          }
          return true;
        };
        Cursor ck{0, row_word(row, is_dense, 0, qb, W, status)};
        Cursor cv = ck;
        int kb_k = 0, kb_v = 0;
        bool go = true;
        for (int t = 0; go && t <= nsub; ++t) {
          if (t < nsub) {
            if ((t & 1) == 0) kb_k = next_kb(ck);
            go = load(true, t, kb_k);
          }
          if (go && t >= 1 && mode != kMaxOnly) {
            if (((t - 1) & 1) == 0) kb_v = next_kb(cv);
            go = load(false, t - 1, kb_v);
          }
        }
        // Every copy issued has landed before the pass ends (the consumers
        // waited for them on the normal path; after a timeout they may not
        // have). Bounded waits that ignore the abort flag.
        const int never = 0;
        mbar_wait(&bars.q_full, 0, &never);
        for (int s = 0; s < 2; ++s) {
          if (kn[s] > 0) mbar_wait(&bars.k_full[s], (kn[s] - 1u) & 1u, &never);
          if (vn[s] > 0) mbar_wait(&bars.v_full[s], (vn[s] - 1u) & 1u, &never);
        }
      }
    } else if (warp == kMmaWarp) {
      if (lane == 0) {
        constexpr uint32_t idesc_qk = idesc_bf16_f32(128, kSubKeys, false, false);
        constexpr uint32_t idesc_pv = idesc_bf16_f32(128, 128, false, true);
        bool go = mbar_wait(&bars.q_full, 0, &bars.abort);
        if (!go) fail(&bars.abort, status, 0x203);
        const uint64_t dq = sdesc_sw128(smem_u32(sQ), 16, 1024);
        const uint64_t dk0 = sdesc_sw128(smem_u32(sK), 16, 1024), dk1 = dk0 + (kSub >> 4);
        const uint64_t dv0 = sdesc_sw128(smem_u32(sV), kSubHalf, 1024), dv1 = dv0 + (kSub >> 4);
        // S_s = Q K_s^T (8 steps of 16 features) into buffer s.
        auto issue_qk = [&](int s) -> bool {
          if (!mbar_wait(&bars.k_full[s], kn[s] & 1u, &bars.abort)) return false;
          ++kn[s];
          tc_fence_after();
          const uint64_t dk = s ? dk1 : dk0;
          // the start-address field is (address >> 4) in the low 14 bits;
          // shared addresses stay below 2^18, so adding offset >> 4 never carries
          umma_qk_x8<(kHalf >> 4), (kSubHalf >> 4)>(tmem + s * kSubKeys, dq, dk, idesc_qk);
          umma_commit(&bars.s_full[s]);
          return true;
        };
        // O += P_s V_s (4 steps of 16 keys); P_s of chunk c at columns
        // 64s + 32c + 16 .. +15 (bf16 pairs, 8 columns per 16 keys).
        auto issue_pv = [&](int s, bool first) -> bool {
          if (!mbar_wait(&bars.p_full[s], pn.parity(s), &bars.abort)) return false;
          pn.inc(s);
          if (!mbar_wait(&bars.v_full[s], vn[s] & 1u, &bars.abort)) return false;
          ++vn[s];
          tc_fence_after();
          const uint64_t dv = s ? dv1 : dv0;
          umma_pv_x4(tmem + 128, tmem + s * kSubKeys + 16, dv, idesc_pv, first ? 0u : 1u);
          umma_commit(&bars.v_empty[s]);
          return true;
        };
        if (go && mode != kMaxOnly) {
          // QK(0,0) QK(0,1) | PV(j,0) QK(j+1,0) PV(j,1) QK(j+1,1) | ...: the QK
          // that writes buffer s is issued right behind the PV that reads P_s
          // from it (tcgen05 MMAs of one thread execute in order), so the
          // next sub-block's scores are formed while the softmax warps work.
          for (int s = 0; go && s < 2; ++s) go = issue_qk(s);
          for (int j = 0; go && j < count; ++j) {
            for (int s = 0; go && s < 2; ++s) {
              go = issue_pv(s, j == 0 && s == 0);
              if (go && j + 1 < count) go = issue_qk(s);
            }
          }
          if (go) umma_commit(&bars.o_full);
        } else if (go) {
          // Scores only: a buffer is free again once its scores have been
          // read (the softmax warps arrive on p_full).
          for (int i = 0; go && i < nsub; ++i) {
            const int s = i & 1;
            if (i >= 2) {
              go = mbar_wait(&bars.p_full[s], pn.parity(s), &bars.abort);
              if (go) pn.inc(s);
            }
            if (go) go = issue_qk(s);
          }
          for (int s = 0; go && s < 2 && s < nsub; ++s) {
            go = mbar_wait(&bars.p_full[s], pn.parity(s), &bars.abort);
            if (go) pn.inc(s);
          }
        }
        if (!go) fail(&bars.abort, status, 0x204);
        // Every MMA issued in this pass has completed before it ends (a
        // bounded wait that ignores the abort flag: TMEM is released later).
        umma_commit(&bars.drain);
        const int never = 0;
        if (!mbar_wait(&bars.drain, drains & 1u, &never)) fail(&bars.abort, status, 0x206);
        ++drains;
      }
    } else {
      // Softmax warps: warp (quarter, chunk) owns rows 32*quarter..+31 and
      // the 32 score columns 32*chunk..+31 of each sub-block.
      const uint32_t s_col = static_cast<uint32_t>(chunk * 32);
      float mx = -INFINITY;  // max-only pass: running raw max of this chunk
      if (mode != kMaxOnly) l = 0.f;
      for (int i = 0; ok && i < nsub; ++i) {
        const int s = i & 1, j = i >> 1;
        if (!warp_wait(&bars.s_full[s], sn.parity(s), &bars.abort)) {
          if (lane == 0) fail(&bars.abort, status, 0x207);
          ok = false;
          break;
        }
        sn.inc(s);
        tc_fence_after();
        const bool diag = bars.has_diag && j == count - 1;  // ascending order: qb is last
        const int key0 = s * kSubKeys + chunk * 32;          // key index in the block of column 0
        uint32_t sv[32];
        tmem_ld32(tmem + lane_addr + s * kSubKeys + s_col, sv);
        if (diag) mask_diag32(key0, r, sv);
        if (mode == kMaxOnly) {
          mx = fmaxf(mx, max32(sv));
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars.p_full[s]);
          continue;
        }
        if (mode == kFast && i == 0) {
          // First sub-block: its exact row max (both chunks) is the reference.
          float m0;
          if (!row_max(max32(sv), m0)) {
            if (lane == 0) fail(&bars.abort, status, 0x209);
            ok = false;
            break;
          }
          m_ref = m0 * c_log2;  // c > 0: max(s*c) = max(s)*c
        }
        uint32_t pk[16];
        float cs = 0.f;
        p_exp32(sv, c_log2, -m_ref, pk, cs);
        tmem_st16(tmem + lane_addr + s * kSubKeys + s_col + 16, pk);
        l += cs;
        if (mode == kFast && !(cs <= kOverflowSum)) *reinterpret_cast<volatile int*>(&bars.redo) = 1;
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.p_full[s]);
      }
      if (mode == kMaxOnly) {
        // The exact row max over every selected block (both chunks).
        float m1;
        if (!row_max(mx, m1)) {
          if (lane == 0) fail(&bars.abort, status, 0x20a);
          ok = false;
        }
        m_ref = m1 * c_log2;
      } else if (ok) {
        // O is final once every PV of the pass has completed.
        if (!warp_wait(&bars.o_full, o_phase & 1u, &bars.abort)) {
          if (lane == 0) fail(&bars.abort, status, 0x208);
          ok = false;
        }
        ++o_phase;
        tc_fence_after();
      }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // After the fast pass, a marked CTA runs the max-only and fixed passes.
    const bool stop = *reinterpret_cast<volatile int*>(&bars.abort) != 0;
    if (stop || (pass == kFast && *reinterpret_cast<volatile int*>(&bars.redo) == 0) || pass == kFixed) break;
  }

  if (warp < kSoftmaxWarps) {
    // Epilogue: O / l -> bf16 for this warp's 64 output columns, staged per
    // warp through shared memory (the K slots are no longer needed) so that
    // each store instruction writes four 128-byte row segments.
    const uint32_t o_addr = tmem + lane_addr + 128 + chunk * 64;
    const bool have = ok && count > 0 && *reinterpret_cast<volatile int*>(&bars.abort) == 0;
    bars.xsum[chunk][r] = l;
    named_bar_sync(pair_bar, 64);
    const float l_row = bars.xsum[0][r] + bars.xsum[1][r];
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
        const int c16 = cc * 4 + q4;  // 16-byte chunk of this warp's 128-byte row part
        stg[lane * 8 + (c16 ^ (lane & 7))] = u;
      }
    }
    __syncwarp();
    const int c16 = lane & 7;
#pragma unroll 4
    for (int it = 0; it < 8; ++it) {
      const int R = it * 4 + (lane >> 3);
      const uint4 u = stg[R * 8 + (c16 ^ (R & 7))];
      const int tok = qb * kB + quarter * 32 + R;
      if (tok >= n) continue;  // rows past the end of a short last block
      const int64_t idx = static_cast<int64_t>(h) * o_hs + static_cast<int64_t>(tok) * o_ts + chunk * 64 + c16 * 8;
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
      maps.q, maps.k64, maps.v, s.seq_len, s.hq / s.hkv, s.scale * 1.4426950408889634f,
      dense ? nullptr : rowbits, order, dense ? 1 : 0, static_cast<__nv_bfloat16*>(out), s.o_head_stride,
      s.o_tok_stride, status);
  return cudaGetLastError();
}

}  // namespace crisp
