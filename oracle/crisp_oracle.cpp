// CRISP sparse-prefill oracle: a plain, slow, fp64 CPU statement of what the
// method computes. TEST INFRASTRUCTURE ONLY: tests, the smoke check and the
// benchmark's CPU-baseline leg call it; the product path never does. It shares
// no code, header, helper or constant generator with the CUDA library.
//
// Source: "CRISP: Cliff-awaRe Input-adaptive Sparse Prefilling with
// Structural-Mass-Motivated Routing" (arXiv 2609.01925), as summarised on the
// ai.info paper page ("Key Contributions", "Methodology in Plain English") and
// the ai-feeds page ("方法"). The pages define the method in prose only; every
// step they leave open is taken at its plainest reading, noted where it is
// used.
//
// Notation: Hq query heads, Hkv kv heads, G = Hq/Hkv, d = 128, B = 128,
// n tokens, nb = ceil(n/B) blocks (block b holds tokens [bB, min(n, bB+B));
// only the last can be short), W = ceil(nb/32) bitset words. Query row r of
// the proxy block is token i = n - B + r: the last B tokens, which straddle
// two blocks when B does not divide n. All bf16 inputs are widened exactly to
// double. Bitsets: bit c of a row is word[c >> 5] >> (c & 31) & 1.
//
// Parity status: every function below is pinned by tests/test_oracle_*.py
// (closed forms, invariants, library special cases, brute force).
#include <algorithm>
#include <cfenv>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <functional>
#include <thread>
#include <vector>

namespace {

constexpr int kB = 128;  // block size, "block size B=128" (ai.info, Methodology)
constexpr int kD = 128;  // head dimension of the evaluated models

int num_blocks(int n) { return (n + kB - 1) / kB; }
// Tokens of block b: B, except a short last block.
int block_len(int n, int b) { return std::min(kB, n - b * kB); }

double bf16_to_double(uint16_t b) {
  uint32_t u = static_cast<uint32_t>(b) << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return static_cast<double>(f);
}

void parallel_for(int64_t count, int nthreads, const std::function<void(int64_t)>& body) {
  if (nthreads <= 1 || count <= 1) {
    for (int64_t t = 0; t < count; ++t) body(t);
    return;
  }
  std::vector<std::thread> pool;
  const int64_t nt = std::min<int64_t>(nthreads, count);
  for (int64_t w = 0; w < nt; ++w) {
    pool.emplace_back([&, w]() {
      for (int64_t t = w; t < count; t += nt) body(t);
    });
  }
  for (auto& th : pool) th.join();
}

// Q32 quantum of a probability: round-half-even(p * 2^32). Not on the pages:
// an exactness device so that every mass below is an integer sum, identical
// under any summation order. p * 2^32 is exact in double for fp32 p.
uint64_t q32(float p) {
  const double x = static_cast<double>(p) * 4294967296.0;
  return static_cast<uint64_t>(std::nearbyint(x));
}

// Softmax over a set of logits (plain definition).
void softmax_inplace(std::vector<double>& s) {
  double m = -INFINITY;
  for (double x : s) m = std::max(m, x);
  double z = 0.0;
  for (double& x : s) {
    x = std::exp(x - m);
    z += x;
  }
  for (double& x : s) x /= z;
}

bool bit(const uint32_t* row, int c) { return (row[c >> 5] >> (c & 31)) & 1u; }
void set_bit(uint32_t* row, int c) { row[c >> 5] |= 1u << (c & 31); }

// Fills `chosen` up to `target` members from `cands` (not yet chosen) in the
// order (mass descending, index ascending): the k_min rule's tie order.
void fill_to(std::vector<char>& chosen, int& count, int target, const std::vector<int>& cands,
             const std::vector<uint64_t>& m) {
  if (count >= target) return;
  std::vector<int> rest;
  for (int c : cands)
    if (!chosen[c]) rest.push_back(c);
  std::stable_sort(rest.begin(), rest.end(), [&](int a, int b) {
    if (m[a] != m[b]) return m[a] > m[b];
    return a < b;
  });
  for (int c : rest) {
    if (count >= target) break;
    chosen[c] = 1;
    ++count;
  }
}

// Sink-aware noise floor over one direction (ai.info, Methodology: "computes
// the expected background mass over the blocks that are not always retained,
// and selects each block that exceeds a multiple alpha of that expectation").
// Reading: expectation = mean mass of the candidate (not-always-retained)
// blocks; "exceeds" is strict; compared in integers as
// m[c] * N * alpha_den > alpha_num * sum. Forced blocks are always kept; the
// set is then filled to min(kmin, |forced| + |candidates|) by (mass desc,
// index asc) ("k_min=1024 tokens (8 blocks) per direction").
void noise_floor_select(const std::vector<uint64_t>& m, const std::vector<int>& forced,
                        const std::vector<int>& cands, uint32_t alpha_num, uint32_t alpha_den, int kmin,
                        std::vector<char>& chosen) {
  int count = 0;
  for (int c : forced)
    if (!chosen[c]) {
      chosen[c] = 1;
      ++count;
    }
  const unsigned __int128 N = cands.size();
  unsigned __int128 sum = 0;
  for (int c : cands) sum += m[c];
  if (N > 0) {
    for (int c : cands) {
      const unsigned __int128 lhs = static_cast<unsigned __int128>(m[c]) * N * alpha_den;
      const unsigned __int128 rhs = static_cast<unsigned __int128>(alpha_num) * sum;
      if (lhs > rhs && !chosen[c]) {
        chosen[c] = 1;
        ++count;
      }
    }
  }
  const int avail = static_cast<int>(forced.size() + cands.size());
  fill_to(chosen, count, std::min(kmin, avail), cands, m);
}

}  // namespace

extern "C" {

// ---------------------------------------------------------------------------
// A1. Proxy attention map of the last query block against all keys
// (ai.info, Key Contributions 2: C_struct is read off "the already-computed
// proxy attention map"). Reading: the last B query rows, causal, each row a
// softmax over its visible keys j <= i; P[h][r][j] = 0 for j > i.
// q: bf16 [hq][n][128], k: bf16 [hkv][n][128]; out: double [hq][128][n].
int oracle_proxy_map(int hq, int hkv, int n, const uint16_t* q, const uint16_t* k, double scale, double* out,
                     int nthreads) {
  if (hq <= 0 || hkv <= 0 || hq % hkv || n < kB) return 1;
  const int G = hq / hkv;
  parallel_for(static_cast<int64_t>(hq) * kB, nthreads, [&](int64_t t) {
    const int h = static_cast<int>(t / kB), r = static_cast<int>(t % kB);
    const int g = h / G;
    const int i = n - kB + r;
    double qi[kD];
    for (int c = 0; c < kD; ++c) qi[c] = bf16_to_double(q[(static_cast<int64_t>(h) * n + i) * kD + c]);
    std::vector<double> s(i + 1);
    for (int j = 0; j <= i; ++j) {
      const uint16_t* kj = k + (static_cast<int64_t>(g) * n + j) * kD;
      double acc = 0.0;
      for (int c = 0; c < kD; ++c) acc += qi[c] * bf16_to_double(kj[c]);
      s[j] = scale * acc;
    }
    softmax_inplace(s);
    double* row = out + (static_cast<int64_t>(h) * kB + r) * n;
    for (int j = 0; j < n; ++j) row[j] = j <= i ? s[j] : 0.0;
  });
  return 0;
}

// A1 for selected rows only: for each requested (head, r) the row
// pmap[h][r][0..n) of oracle_proxy_map, computed on its own (for long
// sequences where the full map is too large to state in fp64).
// out: double [count][n].
int oracle_proxy_rows(int hq, int hkv, int n, const uint16_t* q, const uint16_t* k, double scale, int64_t count,
                      const int32_t* heads, const int32_t* rows, double* out, int nthreads) {
  if (hq <= 0 || hkv <= 0 || hq % hkv || n < kB) return 1;
  for (int64_t t = 0; t < count; ++t)
    if (heads[t] < 0 || heads[t] >= hq || rows[t] < 0 || rows[t] >= kB) return 2;
  const int G = hq / hkv;
  parallel_for(count, nthreads, [&](int64_t t) {
    const int h = heads[t], g = h / G, i = n - kB + rows[t];
    double qi[kD];
    for (int c = 0; c < kD; ++c) qi[c] = bf16_to_double(q[(static_cast<int64_t>(h) * n + i) * kD + c]);
    std::vector<double> s(i + 1);
    for (int j = 0; j <= i; ++j) {
      const uint16_t* kj = k + (static_cast<int64_t>(g) * n + j) * kD;
      double acc = 0.0;
      for (int c = 0; c < kD; ++c) acc += qi[c] * bf16_to_double(kj[c]);
      s[j] = scale * acc;
    }
    softmax_inplace(s);
    double* row = out + t * n;
    for (int j = 0; j < n; ++j) row[j] = j <= i ? s[j] : 0.0;
  });
  return 0;
}

// Q32 quanta of an fp32 array (see q32 above).
void oracle_quantize(const float* p, int64_t count, uint64_t* out) {
  for (int64_t t = 0; t < count; ++t) out[t] = q32(p[t]);
}

// ---------------------------------------------------------------------------
// A2. C_struct routing (ai.info, Key Contributions 2 and Methodology: the
// share of the proxy map's mass in the sink slice, the first 128 key tokens,
// and the recency slice, the last 128; tau_proxy = 0.2). Reading: C_struct =
// S/T with S the quantised mass in columns [0, sink) U [n - recency, n) (the
// union, counted once; the pages fix sink = recency = 128, the two widths are
// parameters here so that other slices can be checked) and T the total
// quantised mass; a head is Vertical-Slash iff C_struct >= tau, compared in
// integers as tau_den * S >= tau_num * T.
// pmap: fp32 [hq][128][n] (the map under test); route[h] = 1 for VS, 0 for PE.
int oracle_route(int hq, int n, const float* pmap, uint32_t tau_num, uint32_t tau_den, int sink, int recency,
                 uint64_t* cstruct, uint64_t* total, uint8_t* route, int nthreads) {
  if (hq <= 0 || n < 2 * kB || tau_den == 0 || sink < 0 || recency < 0) return 1;
  parallel_for(hq, nthreads, [&](int64_t hh) {
    const int h = static_cast<int>(hh);
    uint64_t S = 0, T = 0;
    for (int r = 0; r < kB; ++r) {
      const float* row = pmap + (static_cast<int64_t>(h) * kB + r) * n;
      for (int j = 0; j < n; ++j) {
        const uint64_t m = q32(row[j]);
        T += m;
        if (j < sink || j >= n - recency) S += m;
      }
    }
    cstruct[h] = S;
    total[h] = T;
    route[h] = static_cast<unsigned __int128>(tau_den) * S >= static_cast<unsigned __int128>(tau_num) * T ? 1 : 0;
  });
  return 0;
}

// ---------------------------------------------------------------------------
// A3. Vertical and slash block masses from the proxy map (ai.info,
// Methodology; ai-feeds: mass at "Vertical-Slash compatible positions").
// Reading: vmass[c] = quantised mass of key columns in block c; the slash
// (diagonal) offset of entry (i, j) is i - j and its block s = floor((i-j)/B);
// smass[s] sums entries with j <= i and j >= 128: sink columns are left out of
// the slash direction (the "sink-aware" part: a sink cannot raise the
// diagonal noise floor). Written element by element, independent of any tiling.
int oracle_vs_masses(int hq, int n, const float* pmap, uint64_t* vmass, uint64_t* smass, int nthreads) {
  if (hq <= 0 || n < 2 * kB) return 1;
  const int nb = num_blocks(n);
  parallel_for(hq, nthreads, [&](int64_t hh) {
    const int h = static_cast<int>(hh);
    uint64_t* v = vmass + static_cast<int64_t>(h) * nb;
    uint64_t* s = smass + static_cast<int64_t>(h) * nb;
    std::fill(v, v + nb, 0ull);
    std::fill(s, s + nb, 0ull);
    for (int r = 0; r < kB; ++r) {
      const int i = n - kB + r;
      const float* row = pmap + (static_cast<int64_t>(h) * kB + r) * n;
      for (int j = 0; j < n; ++j) {
        const uint64_t m = q32(row[j]);
        v[j / kB] += m;
        if (j <= i && j >= 128) s[(i - j) / kB] += m;
      }
    }
  });
  return 0;
}

// ---------------------------------------------------------------------------
// A4. Vertical-Slash selection by the sink-aware noise floor. Always-retained
// blocks (reading): vertical {0 (sink), nb-1 (recency)}, slash {0 (local)};
// candidates [1, nb-2] in both directions.
// vbits/sbits: uint32 [hq][W]. Heads with route[h] == 0 get empty sets.
int oracle_select_vs(int hq, int nb, const uint64_t* vmass, const uint64_t* smass, const uint8_t* route,
                     uint32_t alpha_num, uint32_t alpha_den, int kmin, uint32_t* vbits, uint32_t* sbits) {
  if (hq <= 0 || nb < 2 || alpha_den == 0) return 1;
  const int W = (nb + 31) / 32;
  std::vector<int> cands;
  for (int c = 1; c <= nb - 2; ++c) cands.push_back(c);
  for (int h = 0; h < hq; ++h) {
    uint32_t* vb = vbits + static_cast<int64_t>(h) * W;
    uint32_t* sb = sbits + static_cast<int64_t>(h) * W;
    std::fill(vb, vb + W, 0u);
    std::fill(sb, sb + W, 0u);
    if (!route[h]) continue;
    std::vector<uint64_t> mv(vmass + static_cast<int64_t>(h) * nb, vmass + static_cast<int64_t>(h + 1) * nb);
    std::vector<uint64_t> ms(smass + static_cast<int64_t>(h) * nb, smass + static_cast<int64_t>(h + 1) * nb);
    std::vector<char> cv(nb, 0), cs(nb, 0);
    noise_floor_select(mv, {0, nb - 1}, cands, alpha_num, alpha_den, kmin, cv);
    noise_floor_select(ms, {0}, cands, alpha_num, alpha_den, kmin, cs);
    for (int c = 0; c < nb; ++c) {
      if (cv[c]) set_bit(vb, c);
      if (cs[c]) set_bit(sb, c);
    }
  }
  return 0;
}

// ---------------------------------------------------------------------------
// A4 comparator: FlexPrefill's cumulative coverage on Vertical-Slash heads,
// the rule CRISP replaces (ai.info, Key Findings: at gamma = 0.95 a large
// sink mass ends the selection inside the sink, "sink-only collapse").
// Reading: per direction every block [0, nb-1] is a candidate (the sink block
// included, which is what lets the sink fill the coverage); keep the shortest
// prefix in (mass desc, index asc) order whose mass reaches gamma of the
// direction total (gamma_den * prefix >= gamma_num * total); add the
// always-retained blocks of A4; fill to min(kmin, nb) in the same order.
int oracle_select_vs_gamma(int hq, int nb, const uint64_t* vmass, const uint64_t* smass, const uint8_t* route,
                           uint32_t gamma_num, uint32_t gamma_den, int kmin, uint32_t* vbits, uint32_t* sbits) {
  if (hq <= 0 || nb < 2 || gamma_den == 0 || gamma_num > gamma_den) return 1;
  const int W = (nb + 31) / 32;
  std::vector<int> all;
  for (int c = 0; c < nb; ++c) all.push_back(c);
  for (int h = 0; h < hq; ++h) {
    uint32_t* bits[2] = {vbits + static_cast<int64_t>(h) * W, sbits + static_cast<int64_t>(h) * W};
    std::fill(bits[0], bits[0] + W, 0u);
    std::fill(bits[1], bits[1] + W, 0u);
    if (!route[h]) continue;
    for (int dir = 0; dir < 2; ++dir) {
      const uint64_t* src = (dir == 0 ? vmass : smass) + static_cast<int64_t>(h) * nb;
      std::vector<uint64_t> m(src, src + nb);
      std::vector<int> order = all;
      std::stable_sort(order.begin(), order.end(), [&](int a, int b) {
        if (m[a] != m[b]) return m[a] > m[b];
        return a < b;
      });
      unsigned __int128 T = 0, cum = 0;
      for (uint64_t x : m) T += x;
      std::vector<char> chosen(nb, 0);
      for (int c : order) {
        if (static_cast<unsigned __int128>(gamma_den) * cum >= static_cast<unsigned __int128>(gamma_num) * T) break;
        chosen[c] = 1;
        cum += m[c];
      }
      chosen[0] = 1;
      if (dir == 0) chosen[nb - 1] = 1;
      int count = 0;
      for (char x : chosen) count += x;
      fill_to(chosen, count, std::min(kmin, nb), all, m);
      for (int c = 0; c < nb; ++c)
        if (chosen[c]) set_bit(bits[dir], c);
    }
  }
  return 0;
}

// ---------------------------------------------------------------------------
// A2 comparator: FlexPrefill's routing, which CRISP replaces (ai.info,
// Methodology in Plain English: FlexPrefill builds a pooled attention
// estimate and takes its Jensen-Shannon divergence from the per-query
// attention to decide whether a head is concentrated). Reading: the true
// distribution is the last query block's attention pooled into key blocks,
// a[c] = vmass[c] / sum(vmass) (the A3 masses); the estimate is row nb-1 of
// the A5 pooled map, e[c]; D = (KL(a||m) + KL(e||m)) / 2 with m = (a+e)/2
// and natural logarithms (0 log 0 = 0); the head is Vertical-Slash iff
// sqrt(D) >= tau (the block average misses the head's structure). The
// threshold value is not on the pages; 0.1 is our default.
// pbar_last: fp32 [hq][nb] (row nb-1 of each head); jsd: double [hq].
int oracle_route_jsd(int hq, int nb, const uint64_t* vmass, const float* pbar_last, double tau, double* jsd,
                     uint8_t* route) {
  if (hq <= 0 || nb < 1) return 1;
  for (int h = 0; h < hq; ++h) {
    const uint64_t* v = vmass + static_cast<int64_t>(h) * nb;
    const float* e = pbar_last + static_cast<int64_t>(h) * nb;
    long double T = 0.0L;
    for (int c = 0; c < nb; ++c) T += static_cast<long double>(v[c]);
    double kl_a = 0.0, kl_e = 0.0;
    for (int c = 0; c < nb; ++c) {
      const double a = static_cast<double>(static_cast<long double>(v[c]) / T);
      const double b = static_cast<double>(e[c]);
      const double m = 0.5 * (a + b);
      if (a > 0.0) kl_a += a * std::log(a / m);
      if (b > 0.0) kl_e += b * std::log(b / m);
    }
    const double D = 0.5 * (kl_a + kl_e);
    jsd[h] = D;
    route[h] = std::sqrt(std::max(D, 0.0)) >= tau ? 1 : 0;
  }
  return 0;
}

// ---------------------------------------------------------------------------
// A5. Pooled-Estimation map (the PE route CRISP keeps from FlexPrefill;
// ai.info, Overview/Methodology). Reading: mean-pool queries and keys over
// each block (a short last block over its own tokens), logits
// scale * Qbar[b] . Kbar[c] for c <= b, softmax over c in [0, b] per row;
// entries c > b are 0.
// out: double [hq][nb][nb].
int oracle_pe_map(int hq, int hkv, int n, const uint16_t* q, const uint16_t* k, double scale, double* out,
                  int nthreads) {
  if (hq <= 0 || hkv <= 0 || hq % hkv || n < 1) return 1;
  const int G = hq / hkv, nb = num_blocks(n);
  std::vector<double> qbar(static_cast<size_t>(hq) * nb * kD, 0.0), kbar(static_cast<size_t>(hkv) * nb * kD, 0.0);
  parallel_for(static_cast<int64_t>(hq) * nb, nthreads, [&](int64_t t) {
    double* dst = &qbar[t * kD];
    const int64_t h = t / nb, b = t % nb;
    const int len = block_len(n, static_cast<int>(b));
    for (int r = 0; r < len; ++r)
      for (int c = 0; c < kD; ++c) dst[c] += bf16_to_double(q[((h * n) + b * kB + r) * kD + c]);
    for (int c = 0; c < kD; ++c) dst[c] /= len;
  });
  parallel_for(static_cast<int64_t>(hkv) * nb, nthreads, [&](int64_t t) {
    double* dst = &kbar[t * kD];
    const int64_t g = t / nb, b = t % nb;
    const int len = block_len(n, static_cast<int>(b));
    for (int r = 0; r < len; ++r)
      for (int c = 0; c < kD; ++c) dst[c] += bf16_to_double(k[((g * n) + b * kB + r) * kD + c]);
    for (int c = 0; c < kD; ++c) dst[c] /= len;
  });
  parallel_for(static_cast<int64_t>(hq) * nb, nthreads, [&](int64_t t) {
    const int64_t h = t / nb, b = t % nb, g = h / G;
    std::vector<double> s(b + 1);
    for (int64_t c = 0; c <= b; ++c) {
      double acc = 0.0;
      for (int e = 0; e < kD; ++e) acc += qbar[(h * nb + b) * kD + e] * kbar[(g * nb + c) * kD + e];
      s[c] = scale * acc;
    }
    softmax_inplace(s);
    double* row = out + (h * nb + b) * nb;
    for (int64_t c = 0; c < nb; ++c) row[c] = c <= b ? s[c] : 0.0;
  });
  return 0;
}

// A5 for selected rows only: row b of head h of oracle_pe_map for each
// requested (head, b). out: double [count][nb].
int oracle_pe_rows(int hq, int hkv, int n, const uint16_t* q, const uint16_t* k, double scale, int64_t count,
                   const int32_t* heads, const int32_t* blocks, double* out, int nthreads) {
  if (hq <= 0 || hkv <= 0 || hq % hkv || n < 1) return 1;
  const int G = hq / hkv, nb = num_blocks(n);
  for (int64_t t = 0; t < count; ++t)
    if (heads[t] < 0 || heads[t] >= hq || blocks[t] < 0 || blocks[t] >= nb) return 2;
  // Mean-pooled keys of every block of every kv head (needed by any row).
  std::vector<double> kbar(static_cast<size_t>(hkv) * nb * kD, 0.0);
  parallel_for(static_cast<int64_t>(hkv) * nb, nthreads, [&](int64_t t) {
    double* dst = &kbar[t * kD];
    const int64_t g = t / nb, c = t % nb;
    const int len = block_len(n, static_cast<int>(c));
    for (int r = 0; r < len; ++r)
      for (int e = 0; e < kD; ++e) dst[e] += bf16_to_double(k[((g * n) + c * kB + r) * kD + e]);
    for (int e = 0; e < kD; ++e) dst[e] /= len;
  });
  parallel_for(count, nthreads, [&](int64_t t) {
    const int64_t h = heads[t], b = blocks[t], g = h / G;
    double qbar[kD] = {};
    const int len = block_len(n, static_cast<int>(b));
    for (int r = 0; r < len; ++r)
      for (int e = 0; e < kD; ++e) qbar[e] += bf16_to_double(q[((h * n) + b * kB + r) * kD + e]);
    for (int e = 0; e < kD; ++e) qbar[e] /= len;
    std::vector<double> s(b + 1);
    for (int64_t c = 0; c <= b; ++c) {
      double acc = 0.0;
      for (int e = 0; e < kD; ++e) acc += qbar[e] * kbar[(g * nb + c) * kD + e];
      s[c] = scale * acc;
    }
    softmax_inplace(s);
    double* row = out + t * nb;
    for (int64_t c = 0; c < nb; ++c) row[c] = c <= b ? s[c] : 0.0;
  });
  return 0;
}

// ---------------------------------------------------------------------------
// A6. Pooled-Estimation block selection per query block b, from an fp32
// pooled map [hq][nb][nb] (the one under test), quantised to Q32.
// pe_mode 0 (the pages' universal configuration, "gamma=0.95 for the PE path
// only"): order the visible blocks c in [0, b] by (mass desc, index asc) and
// keep the shortest prefix whose mass reaches gamma of the row total
// (gamma_den * prefix >= gamma_num * total); then add {0, b}.
// pe_mode 1: the noise floor of A4 with forced {0, b} and candidates [1, b-1].
// Both modes then fill to min(kmin, b+1) by (mass desc, index asc).
// pebits: uint32 [hq][nb][W]; heads with route[h] == 1 get empty rows.
int oracle_select_pe(int hq, int nb, const float* pbar, const uint8_t* route, int pe_mode, uint32_t gamma_num,
                     uint32_t gamma_den, uint32_t alpha_num, uint32_t alpha_den, int kmin, uint32_t* pebits,
                     int nthreads) {
  if (hq <= 0 || nb < 1 || gamma_den == 0 || alpha_den == 0 || gamma_num > gamma_den) return 1;
  const int W = (nb + 31) / 32;
  parallel_for(static_cast<int64_t>(hq) * nb, nthreads, [&](int64_t t) {
    const int h = static_cast<int>(t / nb), b = static_cast<int>(t % nb);
    uint32_t* out = pebits + t * W;
    std::fill(out, out + W, 0u);
    if (route[h]) return;
    const float* row = pbar + t * nb;
    std::vector<uint64_t> m(b + 1);
    for (int c = 0; c <= b; ++c) m[c] = q32(row[c]);
    std::vector<char> chosen(b + 1, 0);
    std::vector<int> all;
    for (int c = 0; c <= b; ++c) all.push_back(c);
    if (pe_mode == 0) {
      std::vector<int> order = all;
      std::stable_sort(order.begin(), order.end(), [&](int a, int c) {
        if (m[a] != m[c]) return m[a] > m[c];
        return a < c;
      });
      unsigned __int128 T = 0, cum = 0;
      for (uint64_t x : m) T += x;
      for (int c : order) {
        if (static_cast<unsigned __int128>(gamma_den) * cum >= static_cast<unsigned __int128>(gamma_num) * T) break;
        chosen[c] = 1;
        cum += m[c];
      }
      chosen[0] = 1;
      chosen[b] = 1;
      int count = 0;
      for (char x : chosen) count += x;
      fill_to(chosen, count, std::min(kmin, b + 1), all, m);
    } else {
      std::vector<int> forced = {0};
      if (b > 0) forced.push_back(b);
      std::vector<int> cands;
      for (int c = 1; c <= b - 1; ++c) cands.push_back(c);
      noise_floor_select(m, forced, cands, alpha_num, alpha_den, kmin, chosen);
    }
    for (int c = 0; c <= b; ++c)
      if (chosen[c]) set_bit(out, c);
  });
  return 0;
}

// ---------------------------------------------------------------------------
// A7. Per-head sparse attention mask (ai-feeds: the method's output is "a
// per-head sparse attention mask"), as key-block sets per query block qb.
// VS head: {kb <= qb : kb in V} U {qb - s, qb - s - 1 : s in S} restricted to
// [0, qb] (a B-wide diagonal band at offset block s crosses key blocks qb-s
// and qb-s-1). PE head: the pebits row qb.
// rowbits: uint32 [hq][nb][W].
int oracle_build_mask(int hq, int nb, const uint8_t* route, const uint32_t* vbits, const uint32_t* sbits,
                      const uint32_t* pebits, uint32_t* rowbits) {
  if (hq <= 0 || nb < 1) return 1;
  const int W = (nb + 31) / 32;
  for (int h = 0; h < hq; ++h) {
    for (int qb = 0; qb < nb; ++qb) {
      uint32_t* out = rowbits + (static_cast<int64_t>(h) * nb + qb) * W;
      std::fill(out, out + W, 0u);
      if (route[h]) {
        const uint32_t* vb = vbits + static_cast<int64_t>(h) * W;
        const uint32_t* sb = sbits + static_cast<int64_t>(h) * W;
        for (int kb = 0; kb <= qb; ++kb)
          if (bit(vb, kb)) set_bit(out, kb);
        for (int s = 0; s < nb; ++s) {
          if (!bit(sb, s)) continue;
          if (qb - s >= 0) set_bit(out, qb - s);
          if (qb - s - 1 >= 0) set_bit(out, qb - s - 1);
        }
      } else {
        const uint32_t* pr = pebits + (static_cast<int64_t>(h) * nb + qb) * W;
        for (int kb = 0; kb <= qb; ++kb)
          if (bit(pr, kb)) set_bit(out, kb);
      }
    }
  }
  return 0;
}

// ---------------------------------------------------------------------------
// A8/A9. Exact softmax attention over the selected blocks (ai.info, Industry
// relevance: the method "computes exact softmax attention over the blocks it
// selects"), causal, GQA (q-head h reads kv head h / G). For each requested
// (head, token) pair: O_i = sum_{j in A(i)} softmax_j(scale q_i.k_j) v_j with
// A(i) = {j <= i : block(j) in rowbits[h][block(i)]}. rowbits == nullptr
// gives dense causal attention (A(i) = [0, i]). An empty A(i) yields zeros.
// q: bf16 [hq][n][128]; k, v: bf16 [hkv][n][128]; out: double [count][128].
int oracle_attention_rows(int hq, int hkv, int n, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                          double scale, const uint32_t* rowbits, int64_t count, const int32_t* heads,
                          const int32_t* tokens, double* out, int nthreads) {
  if (hq <= 0 || hkv <= 0 || hq % hkv || n < 1) return 1;
  const int G = hq / hkv, nb = num_blocks(n), W = (nb + 31) / 32;
  for (int64_t t = 0; t < count; ++t)
    if (heads[t] < 0 || heads[t] >= hq || tokens[t] < 0 || tokens[t] >= n) return 2;
  parallel_for(count, nthreads, [&](int64_t t) {
    const int h = heads[t], i = tokens[t], g = h / G;
    const uint32_t* rb = rowbits ? rowbits + (static_cast<int64_t>(h) * nb + i / kB) * W : nullptr;
    double qi[kD];
    for (int c = 0; c < kD; ++c) qi[c] = bf16_to_double(q[(static_cast<int64_t>(h) * n + i) * kD + c]);
    std::vector<int> keys;
    std::vector<double> s;
    for (int j = 0; j <= i; ++j) {
      if (rb && !bit(rb, j / kB)) continue;
      const uint16_t* kj = k + (static_cast<int64_t>(g) * n + j) * kD;
      double acc = 0.0;
      for (int c = 0; c < kD; ++c) acc += qi[c] * bf16_to_double(kj[c]);
      keys.push_back(j);
      s.push_back(scale * acc);
    }
    double* o = out + t * kD;
    std::fill(o, o + kD, 0.0);
    if (keys.empty()) return;
    softmax_inplace(s);
    for (size_t u = 0; u < keys.size(); ++u) {
      const uint16_t* vj = v + (static_cast<int64_t>(g) * n + keys[u]) * kD;
      for (int c = 0; c < kD; ++c) o[c] += s[u] * bf16_to_double(vj[c]);
    }
  });
  return 0;
}

// Number of (row, key) pairs the attention over `rowbits` visits, i.e. the
// causal pairs of every selected block of n tokens: len(qb)*len(kb) off the
// diagonal, len(qb)(len(qb)+1)/2 on it (len = B except a short last block).
int64_t oracle_selected_pairs(int hq, int n, const uint32_t* rowbits) {
  const int nb = num_blocks(n), W = (nb + 31) / 32;
  int64_t pairs = 0;
  for (int h = 0; h < hq; ++h)
    for (int qb = 0; qb < nb; ++qb) {
      const uint32_t* rb = rowbits + (static_cast<int64_t>(h) * nb + qb) * W;
      const int64_t lq = block_len(n, qb);
      for (int kb = 0; kb <= qb; ++kb)
        if (bit(rb, kb)) pairs += kb == qb ? lq * (lq + 1) / 2 : lq * block_len(n, kb);
    }
  return pairs;
}

}  // extern "C"
