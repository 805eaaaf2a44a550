// Internal declarations shared by the CRISP CUDA translation units.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/crisp.h"

namespace crisp {

constexpr int kB = 128;  // block size (tokens), "block size B=128"
constexpr int kD = 128;  // head dimension
constexpr int kMaxSeq = 1 << 20;
constexpr int kMaxBlocks = kMaxSeq / kB;  // 8192
constexpr int kProxyChunk = 16;           // key blocks per proxy CTA

// Device status word at offset 0 of every workspace: first error wins.
struct DevStatus {
  uint32_t code;
  uint32_t detail;
};

__device__ __forceinline__ void report_error(DevStatus* st, uint32_t code, uint32_t detail) {
  if (atomicCAS(&st->code, 0u, code) == 0u) atomicExch(&st->detail, detail);
}

// Bounds checks of the checking build (compiled with -DCRISP_DEBUG): a
// global index or TMA coordinate outside its buffer records CRISP_ERR_BOUNDS
// with the site code in the status word (first error wins), and the caller
// skips the access; nothing traps. Each extent is derived from the shape the
// kernel was launched with, independently of the index it guards. The
// release build compiles every check to `true`.
#ifdef CRISP_DEBUG
__device__ __forceinline__ bool in_bounds(bool ok, DevStatus* st, uint32_t site) {
  if (!ok && st != nullptr) report_error(st, CRISP_ERR_BOUNDS, site);
  return ok;
}
#define CRISP_CHECK(cond, st, site) ::crisp::in_bounds((cond), (st), (site))
#else
#define CRISP_CHECK(cond, st, site) true
#endif

// Q32 quantum of a probability: round-half-even(p * 2^32); p * 2^32 is exact
// in fp32. No float->64-bit conversion instruction is used (on this GPU those
// run on the FP64 pipe): below 2^23, adding 2^23 in fp32 rounds the value to
// the nearest even integer, whose bits minus those of 2^23 are the result;
// from 2^23 up the product is already an integer, rebuilt from its exponent
// and mantissa.
constexpr float kTwo23 = 8388608.0f;
__device__ __forceinline__ uint32_t q32_small(float x) {  // x = p * 2^32 < 2^23
  return __float_as_uint(x + kTwo23) - 0x4B000000u;
}
__device__ __forceinline__ uint64_t q32_large(float x) {  // x = p * 2^32 >= 2^23
  const uint32_t b = __float_as_uint(x);
  const uint32_t sh = min((b >> 23) - 150u, 40u);
  return static_cast<uint64_t>((b & 0x7FFFFFu) | 0x800000u) << sh;
}
__device__ __forceinline__ uint64_t q32(float p) {
  const float x = p * 4294967296.0f;
  return x < kTwo23 ? static_cast<uint64_t>(q32_small(x)) : q32_large(x);
}

// Blocks are aligned at token 0; when 128 does not divide n the last block
// is short: it holds tail_len(n) in [1, 128] tokens.
inline int num_blocks(int n) { return (n + kB - 1) / kB; }
inline int tail_len(int n) { return n - (num_blocks(n) - 1) * kB; }
// Row stride (floats) of the proxy map: whole 128-column tiles.
inline int64_t map_ld(int n) { return static_cast<int64_t>(num_blocks(n)) * kB; }
inline int bit_words(int nb) { return (nb + 31) / 32; }
inline int proxy_chunks(int nb) { return (nb + kProxyChunk - 1) / kProxyChunk; }

// Scratch part of every workspace (offsets in bytes, each 256-aligned).
struct ScratchLayout {
  size_t status;       // DevStatus
  size_t proxy_part;   // float2 [hq][128][chunks]  per-chunk (max, sum) in log2 units
  size_t proxy_stats;  // float2 [hq][128]          (row max, 1/row sum)
  size_t mass_lower;   // uint64 [hq][nb]  tile c's entries with slash block nb-1-c
  size_t mass_upper;   // uint64 [hq][nb]  tile c's entries with slash block nb-2-c
  size_t mass_upper2;  // uint64 [hq][nb]  tile c's entries with slash block nb-3-c (short last block only)
  size_t mass_rec;     // uint64 [hq]      recency columns [n-128, n) that lie in tile nb-2
  size_t qbar;         // bf16 [hq][nb][128] hi, then the same for lo (block means as hi + lo)
  size_t kbar;         // bf16 [hkv][nb][128] hi, then lo
  size_t srev;         // uint32 [hq][W + 2]  slash bits reversed
  size_t rmass;        // uint64 [hq]      recency masses of crisp_select_vs (from the map)
  size_t rowbits;      // uint32 [hq][nb][W]  block mask built by crisp_sparse_prefill
  size_t counts;       // int32  [hq][nb]      blocks per row
  size_t order;        // int32  [hq*nb]       attention schedule
  size_t total;
};

// Intermediates of crisp_prefill_layer, placed after the scratch.
struct LayerLayout {
  size_t vmass, smass, rmass, cstruct, total_mass, route, vbits, sbits, pbar, pebits, rowbits, counts, order;
  size_t total;
};

ScratchLayout scratch_layout(const crisp_shape& s);
LayerLayout layer_layout(const crisp_shape& s);

bool encode_bf16_rows(CUtensorMap* m, const void* ptr, int heads, int rows);

struct TmaMaps {
  CUtensorMap q, k, v, k64;  // k: 128-token boxes (proxy); k64, v: 64-token boxes (attention)
};

// ---- launchers (one per translation unit); return cudaSuccess or the launch error
cudaError_t launch_proxy(const crisp_shape& s, const TmaMaps& maps, float* pmap, char* ws, cudaStream_t st);
cudaError_t launch_proxy_masses(const crisp_shape& s, const TmaMaps& maps, uint64_t* vmass, uint64_t* smass,
                                uint64_t* rmass, char* ws, cudaStream_t st);
cudaError_t launch_assemble_slash(const crisp_shape& s, const uint64_t* vmass, char* ws, uint64_t* smass,
                                  uint64_t* rmass, cudaStream_t st);
cudaError_t launch_block_masses(const crisp_shape& s, const float* pmap, uint64_t* vmass, uint64_t* smass,
                                uint64_t* rmass, char* ws, cudaStream_t st);
cudaError_t launch_route(const crisp_shape& s, const crisp_params& p, const uint64_t* vmass, const uint64_t* rmass,
                         uint64_t* cstruct, uint64_t* total, uint8_t* route, DevStatus* status, cudaStream_t st);
cudaError_t launch_route_map(const crisp_shape& s, const crisp_params& p, const float* pmap, uint64_t* cstruct,
                             uint64_t* total, uint8_t* route, DevStatus* status, cudaStream_t st);
cudaError_t launch_route_jsd(const crisp_shape& s, const crisp_params& p, const uint64_t* vmass, const float* pbar,
                             double* jsd, uint8_t* route, DevStatus* status, cudaStream_t st);
cudaError_t launch_select_vs(const crisp_shape& s, const crisp_params& p, const uint64_t* vmass,
                             const uint64_t* smass, const uint8_t* route, uint32_t* vbits, uint32_t* sbits,
                             DevStatus* status, cudaStream_t st);
cudaError_t launch_pe_map(const crisp_shape& s, const void* q, const void* k, const uint8_t* route, float* pbar,
                          char* ws, cudaStream_t st);
cudaError_t launch_select_pe(const crisp_shape& s, const crisp_params& p, const float* pbar, const uint8_t* route,
                             uint32_t* pebits, DevStatus* status, cudaStream_t st);
cudaError_t launch_build_mask(const crisp_shape& s, const uint8_t* route, const uint32_t* vbits,
                              const uint32_t* sbits, const uint32_t* pebits, uint32_t* rowbits, int32_t* counts,
                              int32_t* order, char* ws, cudaStream_t st);
cudaError_t launch_attention(const crisp_shape& s, const TmaMaps& maps, const uint32_t* rowbits,
                             const int32_t* order, void* out, char* ws, bool dense, cudaStream_t st);

}  // namespace crisp
