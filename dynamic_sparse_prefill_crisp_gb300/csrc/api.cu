// Host side of the C ABI declared in include/crisp.h: argument validation,
// workspace layout, TMA descriptors and the launch sequence of each step.
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>
#include <new>

#include <nvtx3/nvToolsExt.h>

#include "common.cuh"
#include "ptx.cuh"

namespace crisp {

namespace {

constexpr size_t kAlign = 256;
size_t up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// The method's steps need the sink block and at least one more (n >= 256);
// attention and the whole layer take any n from 0 (an empty input) up.
constexpr int kMinSeqMethod = 2 * kB;

crisp_status check_shape(const crisp_shape* s, int min_n = kMinSeqMethod) {
  if (!s) return CRISP_ERR_INVALID_ARG;
  if (s->hq <= 0 || s->hkv <= 0 || s->hq % s->hkv != 0) return CRISP_ERR_SHAPE;
  if (s->head_dim != kD || s->block != kB) return CRISP_ERR_SHAPE;
  if (s->seq_len < min_n || s->seq_len > kMaxSeq) return CRISP_ERR_SHAPE;
  if (s->hq > 4096) return CRISP_ERR_SHAPE;
  if (!(s->scale >= 0.f) || std::isinf(s->scale)) return CRISP_ERR_INVALID_ARG;
  if (s->seq_len == 0) return CRISP_OK;  // an empty input addresses no element: strides are not used
  const int64_t strides[6] = {s->q_head_stride, s->q_tok_stride, s->kv_head_stride,
                              s->kv_tok_stride, s->o_head_stride, s->o_tok_stride};
  for (int64_t st : strides)
    if (st <= 0 || st % 8 != 0 || st > (int64_t(1) << 38)) return CRISP_ERR_ALIGN;
  if (s->q_tok_stride < kD || s->kv_tok_stride < kD || s->o_tok_stride < kD) return CRISP_ERR_SHAPE;
  return CRISP_OK;
}

crisp_status check_params(const crisp_params* p) {
  if (!p) return CRISP_ERR_INVALID_ARG;
  if (p->tau_den == 0 || p->tau_num > p->tau_den) return CRISP_ERR_INVALID_ARG;
  if (p->alpha_den == 0 || p->alpha_den > 65535u || p->alpha_num > 65535u) return CRISP_ERR_INVALID_ARG;
  if (p->gamma_den == 0 || p->gamma_num > p->gamma_den) return CRISP_ERR_INVALID_ARG;
  if (p->kmin_blocks < 0 || p->kmin_blocks > kMaxBlocks) return CRISP_ERR_INVALID_ARG;
  if (p->pe_mode != CRISP_PE_GAMMA && p->pe_mode != CRISP_PE_NOISE) return CRISP_ERR_INVALID_ARG;
  if (p->route_mode != CRISP_ROUTE_CSTRUCT && p->route_mode != CRISP_ROUTE_JSD) return CRISP_ERR_INVALID_ARG;
  if (p->vs_mode != CRISP_VS_NOISE && p->vs_mode != CRISP_VS_GAMMA) return CRISP_ERR_INVALID_ARG;
  if (p->vs_gamma_den == 0 || p->vs_gamma_num > p->vs_gamma_den) return CRISP_ERR_INVALID_ARG;
  if (!(p->jsd_tau >= 0.f && p->jsd_tau <= 1.f)) return CRISP_ERR_INVALID_ARG;
  if (p->dense_below < 0) return CRISP_ERR_INVALID_ARG;
  if (p->sink_tokens < 0 || p->sink_tokens > kMaxSeq || p->recency_tokens < 0 || p->recency_tokens > kMaxSeq)
    return CRISP_ERR_INVALID_ARG;
  return CRISP_OK;
}

// Routing from block masses reads the sink slice as key block 0 and the
// recency slice as the recency mass: both slices must be one block wide.
crisp_status check_block_slices(const crisp_params* p) {
  return (p->sink_tokens == kB && p->recency_tokens == kB) ? CRISP_OK : CRISP_ERR_INVALID_ARG;
}

crisp_shape normalised(const crisp_shape& s) {
  crisp_shape t = s;
  if (t.scale == 0.f) t.scale = 1.0f / std::sqrt(static_cast<float>(kD));
  return t;
}

crisp_status check_device() {
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return CRISP_ERR_CUDA;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return CRISP_ERR_CUDA;
  return (major == 10 && minor == 3) ? CRISP_OK : CRISP_ERR_DEVICE;
}

crisp_status check_ws(const crisp_shape& s, const void* ws, size_t ws_bytes) {
  if (!ws || !aligned(ws, kAlign)) return ws ? CRISP_ERR_ALIGN : CRISP_ERR_WORKSPACE;
  return ws_bytes >= scratch_layout(s).total ? CRISP_OK : CRISP_ERR_WORKSPACE;
}

typedef CUresult (*EncodeTiled)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver entry point is looked up once; it is a constant afterwards.
EncodeTiled encode_fn() {
  static EncodeTiled fn = nullptr;
  static std::once_flag once;
  std::call_once(once, []() {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiled>(p);
  });
  return fn;
}

// bf16 [heads][n][128] with element strides; boxes of 64 features x `rows`
// tokens (one 128-byte swizzle row per token).
crisp_status make_map(CUtensorMap* m, const void* ptr, int heads, int n, int64_t hs, int64_t ts, int rows = kB) {
  EncodeTiled enc = encode_fn();
  if (!enc) return CRISP_ERR_CUDA;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(n), static_cast<cuuint64_t>(heads)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(ts) * 2, static_cast<cuuint64_t>(hs) * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(rows), 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? CRISP_OK : CRISP_ERR_ALIGN;
}

// The attention kernel's K and V maps: boxes of 64 tokens (a sub-block).
crisp_status make_kv_maps(TmaMaps* maps, const void* k, const void* v, const crisp_shape& s) {
  crisp_status st = make_map(&maps->k64, k, s.hkv, s.seq_len, s.kv_head_stride, s.kv_tok_stride, kB / 2);
  if (st != CRISP_OK) return st;
  return make_map(&maps->v, v, s.hkv, s.seq_len, s.kv_head_stride, s.kv_tok_stride, kB / 2);
}

crisp_status from_cuda(cudaError_t e) { return e == cudaSuccess ? CRISP_OK : CRISP_ERR_CUDA; }

// Tracing of the entry points: each call runs inside an NVTX range named
// after it (Nsight tools show the per-stage ranges; without a tool attached
// the range is a no-op), and with CRISP_LOG=1 in the environment each call
// writes its name, shape and returned status to stderr.
bool log_enabled() {
  static const bool on = [] {
    const char* v = std::getenv("CRISP_LOG");
    return v != nullptr && v[0] == '1';
  }();
  return on;
}

template <class Body>
crisp_status traced(const char* name, const crisp_shape* shape, Body&& body) {
  nvtxRangePushA(name);
  const crisp_status st = body();
  nvtxRangePop();
  if (log_enabled()) {
    if (shape != nullptr)
      std::fprintf(stderr, "[crisp] %s hq=%d hkv=%d n=%d -> %d (%s)\n", name, shape->hq, shape->hkv, shape->seq_len,
                   static_cast<int>(st), crisp_status_string(st));
    else
      std::fprintf(stderr, "[crisp] %s -> %d (%s)\n", name, static_cast<int>(st), crisp_status_string(st));
  }
  return st;
}

// The status word at the start of a workspace.
DevStatus* status_of(void* ws) { return static_cast<DevStatus*>(ws); }

}  // namespace

ScratchLayout scratch_layout(const crisp_shape& s) {
  const size_t hq = s.hq, hkv = s.hkv, nb = num_blocks(s.seq_len), W = bit_words(static_cast<int>(nb));
  const size_t chunks = proxy_chunks(static_cast<int>(nb));
  ScratchLayout L{};
  size_t o = 0;
  L.status = o;      o = up(o + sizeof(DevStatus));
  L.proxy_part = o;  o = up(o + hq * kB * 2 * chunks * sizeof(float2));
  L.proxy_stats = o; o = up(o + hq * kB * sizeof(float2));
  L.mass_lower = o;  o = up(o + hq * nb * 8);
  L.mass_upper = o;  o = up(o + hq * nb * 8);
  L.mass_upper2 = o; o = up(o + hq * nb * 8);
  L.mass_rec = o;    o = up(o + hq * 8);
  L.qbar = o;        o = up(o + hq * nb * kD * 4);   // bf16 hi and lo
  L.kbar = o;        o = up(o + hkv * nb * kD * 4);  // bf16 hi and lo
  L.srev = o;        o = up(o + hq * (W + 2) * 4);
  L.rmass = o;       o = up(o + hq * 8);
  L.rowbits = o;     o = up(o + hq * nb * W * 4);
  L.counts = o;      o = up(o + hq * nb * 4);
  L.order = o;       o = up(o + hq * nb * 4);
  L.total = o;
  return L;
}

LayerLayout layer_layout(const crisp_shape& s) {
  const size_t hq = s.hq, nb = num_blocks(s.seq_len), W = bit_words(static_cast<int>(nb));
  LayerLayout L{};
  const ScratchLayout S = scratch_layout(s);
  size_t o = S.total;
  L.vmass = o;      o = up(o + hq * nb * 8);
  L.smass = o;      o = up(o + hq * nb * 8);
  L.rmass = o;      o = up(o + hq * 8);
  L.cstruct = o;    o = up(o + hq * 8);
  L.total_mass = o; o = up(o + hq * 8);
  L.route = o;      o = up(o + hq);
  L.vbits = o;      o = up(o + hq * W * 4);
  L.sbits = o;      o = up(o + hq * W * 4);
  L.pbar = o;       o = up(o + hq * nb * nb * 4);
  L.pebits = o;     o = up(o + hq * nb * W * 4);
  // The mask and the schedule share the scratch regions crisp_sparse_prefill uses.
  L.rowbits = S.rowbits;
  L.counts = S.counts;
  L.order = S.order;
  L.total = o;
  return L;
}

// bf16 [heads][rows][128] with 128-row boxes (the pooled estimate's operands).
bool encode_bf16_rows(CUtensorMap* m, const void* ptr, int heads, int rows) {
  return make_map(m, ptr, heads, rows, static_cast<int64_t>(rows) * kD, kD, kB) == CRISP_OK;
}

}  // namespace crisp

using namespace crisp;

extern "C" {

void crisp_params_default(crisp_params* p) {
  if (!p) return;
  p->tau_num = 1;
  p->tau_den = 5;
  p->alpha_num = 1;
  p->alpha_den = 1;
  p->gamma_num = 19;
  p->gamma_den = 20;
  p->kmin_blocks = 8;
  p->pe_mode = CRISP_PE_GAMMA;
  p->route_mode = CRISP_ROUTE_CSTRUCT;
  p->vs_mode = CRISP_VS_NOISE;
  p->vs_gamma_num = 95;
  p->vs_gamma_den = 100;
  p->jsd_tau = 0.1f;
  p->dense_below = 0;
  p->sink_tokens = kB;
  p->recency_tokens = kB;
}

crisp_status crisp_workspace_size(const crisp_shape* shape, size_t* bytes) {
  return traced("crisp_workspace_size", shape, [&]() -> crisp_status {
    crisp_status st = check_shape(shape, 0);
    if (st != CRISP_OK) return st;
    if (!bytes) return CRISP_ERR_INVALID_ARG;
    *bytes = scratch_layout(*shape).total;
    return CRISP_OK;
  });
}

crisp_status crisp_layer_workspace_size(const crisp_shape* shape, size_t* bytes) {
  return traced("crisp_layer_workspace_size", shape, [&]() -> crisp_status {
    crisp_status st = check_shape(shape, 0);
    if (st != CRISP_OK) return st;
    if (!bytes) return CRISP_ERR_INVALID_ARG;
    *bytes = layer_layout(*shape).total;
    return CRISP_OK;
  });
}

crisp_status crisp_workspace_init(void* ws, size_t ws_bytes, crisp_stream_t stream) {
  return traced("crisp_workspace_init", nullptr, [&]() -> crisp_status {
    if (!ws) return CRISP_ERR_WORKSPACE;
    if (ws_bytes < sizeof(DevStatus)) return CRISP_ERR_WORKSPACE;
    return from_cuda(cudaMemsetAsync(ws, 0, sizeof(DevStatus), stream));
  });
}

crisp_status crisp_proxy_map(const crisp_shape* shape, const void* q, const void* k, float* pmap, void* ws,
                             size_t ws_bytes, crisp_stream_t stream) {
  return traced("crisp_proxy_map", shape, [&]() -> crisp_status {
    crisp_status st = check_shape(shape);
    if (st != CRISP_OK) return st;
    if (!q || !k || !pmap) return CRISP_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(pmap)) return CRISP_ERR_ALIGN;
    const crisp_shape s = normalised(*shape);
    if ((st = check_ws(s, ws, ws_bytes)) != CRISP_OK) return st;
    if ((st = check_device()) != CRISP_OK) return st;
    TmaMaps maps;
    if ((st = make_map(&maps.q, q, s.hq, s.seq_len, s.q_head_stride, s.q_tok_stride)) != CRISP_OK) return st;
    if ((st = make_map(&maps.k, k, s.hkv, s.seq_len, s.kv_head_stride, s.kv_tok_stride)) != CRISP_OK) return st;
    maps.v = maps.k;
    return from_cuda(launch_proxy(s, maps, pmap, static_cast<char*>(ws), stream));
  });
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Proxy map for callers that cannot allocate: the scratch of the proxy
// kernels (status word + per-chunk statistics, the first regions of the
// workspace layout) lives in this static device array instead of a caller
// workspace. Every GPU that loads the library holds it until exit.
namespace crisp {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;
constexpr int kMaxDevices = 64;
static __device__ __align__(256) unsigned char g_proxy_scratch[kNoAllocScratchBytes];

// Device address of g_proxy_scratch on the current device; looked up once per
// device (host code only sees a host-side stand-in for the symbol).
crisp_status noalloc_scratch(char** out) {
  static std::mutex mu;
  static void* addr[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return CRISP_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return CRISP_ERR_DEVICE;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_proxy_scratch) != cudaSuccess || p == nullptr) return CRISP_ERR_CUDA;
    addr[dev] = p;
  }
  *out = static_cast<char*>(addr[dev]);
  return CRISP_OK;
}

}  // namespace
}  // namespace crisp

extern "C" {

crisp_status crisp_proxy_map_noalloc(const crisp_shape* shape, const void* q, const void* k, float* pmap,
                                     crisp_stream_t stream) {
  return traced("crisp_proxy_map_noalloc", shape, [&]() -> crisp_status {
    crisp_status st = check_shape(shape);
    if (st != CRISP_OK) return st;
    if (!q || !k || !pmap) return CRISP_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(pmap)) return CRISP_ERR_ALIGN;
    const crisp_shape s = normalised(*shape);
    // The proxy kernels touch only the status word and the two statistics
    // regions, which end where the mass scratch begins.
    const ScratchLayout L = scratch_layout(s);
    if (L.mass_lower > kNoAllocScratchBytes) return CRISP_ERR_WORKSPACE;
    if ((st = check_device()) != CRISP_OK) return st;
    char* scratch = nullptr;
    if ((st = noalloc_scratch(&scratch)) != CRISP_OK) return st;
    TmaMaps maps;
    if ((st = make_map(&maps.q, q, s.hq, s.seq_len, s.q_head_stride, s.q_tok_stride)) != CRISP_OK) return st;
    if ((st = make_map(&maps.k, k, s.hkv, s.seq_len, s.kv_head_stride, s.kv_tok_stride)) != CRISP_OK) return st;
    maps.v = maps.k;
    // The array keeps the previous call's contents: start from a clear status.
    if (cudaMemsetAsync(scratch + L.status, 0, sizeof(DevStatus), stream) != cudaSuccess) return CRISP_ERR_CUDA;
    return from_cuda(launch_proxy(s, maps, pmap, scratch, stream));
  });
}

crisp_status crisp_noalloc_read_status(crisp_stream_t stream, crisp_status* status) {
  return traced("crisp_noalloc_read_status", nullptr, [&]() -> crisp_status {
    if (!status) return CRISP_ERR_INVALID_ARG;
    char* scratch = nullptr;
    crisp_status st = noalloc_scratch(&scratch);
    if (st != CRISP_OK) return st;
    DevStatus host{};
    if (cudaMemcpyAsync(&host, scratch, sizeof(host), cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess)
      return CRISP_ERR_CUDA;
    *status = static_cast<crisp_status>(host.code);
    return CRISP_OK;
  });
}

crisp_status crisp_block_masses(const crisp_shape* shape, const float* pmap, uint64_t* vmass, uint64_t* smass,
                                uint64_t* rmass, void* ws, size_t ws_bytes, crisp_stream_t stream) {
  return traced("crisp_block_masses", shape, [&]() -> crisp_status {
    crisp_status st = check_shape(shape);
    if (st != CRISP_OK) return st;
    if (!pmap || !vmass || !smass || !rmass) return CRISP_ERR_INVALID_ARG;
    if (!aligned16(pmap) || !aligned(vmass, 8) || !aligned(smass, 8) || !aligned(rmass, 8)) return CRISP_ERR_ALIGN;
    const crisp_shape s = normalised(*shape);
    if ((st = check_ws(s, ws, ws_bytes)) != CRISP_OK) return st;
    if ((st = check_device()) != CRISP_OK) return st;
    return from_cuda(launch_block_masses(s, pmap, vmass, smass, rmass, static_cast<char*>(ws), stream));
  });
}

crisp_status crisp_proxy_masses(const crisp_shape* shape, const void* q, const void* k, uint64_t* vmass,
                                uint64_t* smass, uint64_t* rmass, void* ws, size_t ws_bytes, crisp_stream_t stream) {
  return traced("crisp_proxy_masses", shape, [&]() -> crisp_status {
    crisp_status st = check_shape(shape);
    if (st != CRISP_OK) return st;
    if (!q || !k || !vmass || !smass || !rmass) return CRISP_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned(vmass, 8) || !aligned(smass, 8) || !aligned(rmass, 8))
      return CRISP_ERR_ALIGN;
    const crisp_shape s = normalised(*shape);
    if ((st = check_ws(s, ws, ws_bytes)) != CRISP_OK) return st;
    if ((st = check_device()) != CRISP_OK) return st;
    TmaMaps maps;
    if ((st = make_map(&maps.q, q, s.hq, s.seq_len, s.q_head_stride, s.q_tok_stride)) != CRISP_OK) return st;
    if ((st = make_map(&maps.k, k, s.hkv, s.seq_len, s.kv_head_stride, s.kv_tok_stride)) != CRISP_OK) return st;
    maps.v = maps.k;
    return from_cuda(launch_proxy_masses(s, maps, vmass, smass, rmass, static_cast<char*>(ws), stream));
  });
}

crisp_status crisp_route_cstruct(const crisp_shape* shape, const crisp_params* params, const float* pmap,
                                 uint64_t* cstruct, uint64_t* total, uint8_t* route, void* ws, size_t ws_bytes,
                                 crisp_stream_t stream) {
  return traced("crisp_route_cstruct", shape, [&]() -> crisp_status {
    crisp_status st = check_shape(shape);
    if (st != CRISP_OK) return st;
    if ((st = check_params(params)) != CRISP_OK) return st;
    if (!pmap || !cstruct || !total || !route) return CRISP_ERR_INVALID_ARG;
    if (!aligned16(pmap) || !aligned(cstruct, 8) || !aligned(total, 8)) return CRISP_ERR_ALIGN;
    const crisp_shape s = normalised(*shape);
    if ((st = check_ws(s, ws, ws_bytes)) != CRISP_OK) return st;
    if ((st = check_device()) != CRISP_OK) return st;
    return from_cuda(launch_route_map(s, *params, pmap, cstruct, total, route, status_of(ws), stream));
  });
}

crisp_status crisp_route_cstruct_masses(const crisp_shape* shape, const crisp_params* params, const uint64_t* vmass,
                                        const uint64_t* rmass, uint64_t* cstruct, uint64_t* total, uint8_t* route,
                                        void* ws, size_t ws_bytes, crisp_stream_t stream) {
  return traced("crisp_route_cstruct_masses", shape, [&]() -> crisp_status {
    crisp_status st = check_shape(shape);
    if (st != CRISP_OK) return st;
    if ((st = check_params(params)) != CRISP_OK) return st;
    if ((st = check_block_slices(params)) != CRISP_OK) return st;
    if (!vmass || !rmass || !cstruct || !total || !route) return CRISP_ERR_INVALID_ARG;
    if (!aligned(vmass, 8) || !aligned(rmass, 8) || !aligned(cstruct, 8) || !aligned(total, 8)) return CRISP_ERR_ALIGN;
    const crisp_shape s = normalised(*shape);
    if ((st = check_ws(s, ws, ws_bytes)) != CRISP_OK) return st;
    if ((st = check_device()) != CRISP_OK) return st;
    return from_cuda(launch_route(s, *params, vmass, rmass, cstruct, total, route, status_of(ws), stream));
  });
}

crisp_status crisp_route_jsd(const crisp_shape* shape, const crisp_params* params, const uint64_t* vmass,
                             const float* pbar, double* jsd, uint8_t* route, void* ws, size_t ws_bytes,
                             crisp_stream_t stream) {
  return traced("crisp_route_jsd", shape, [&]() -> crisp_status {
    crisp_status st = check_shape(shape);
    if (st != CRISP_OK) return st;
    if ((st = check_params(params)) != CRISP_OK) return st;
    if (!vmass || !pbar || !route) return CRISP_ERR_INVALID_ARG;
    if (!aligned(vmass, 8) || !aligned(pbar, 4) || (jsd && !aligned(jsd, 8))) return CRISP_ERR_ALIGN;
    const crisp_shape s = normalised(*shape);
    if ((st = check_ws(s, ws, ws_bytes)) != CRISP_OK) return st;
    if ((st = check_device()) != CRISP_OK) return st;
    return from_cuda(launch_route_jsd(s, *params, vmass, pbar, jsd, route, status_of(ws), stream));
  });
}

crisp_status crisp_select_vs_masses(const crisp_shape* shape, const crisp_params* params, const uint64_t* vmass,
                                    const uint64_t* smass, const uint8_t* route, uint32_t* vbits, uint32_t* sbits,
                                    void* ws, size_t ws_bytes, crisp_stream_t stream) {
  return traced("crisp_select_vs_masses", shape, [&]() -> crisp_status {
    crisp_status st = check_shape(shape);
    if (st != CRISP_OK) return st;
    if ((st = check_params(params)) != CRISP_OK) return st;
    if (!vmass || !smass || !route || !vbits || !sbits) return CRISP_ERR_INVALID_ARG;
    if (!aligned(vmass, 8) || !aligned(smass, 8) || !aligned(vbits, 4) || !aligned(sbits, 4)) return CRISP_ERR_ALIGN;
    const crisp_shape s = normalised(*shape);
    if ((st = check_ws(s, ws, ws_bytes)) != CRISP_OK) return st;
    if ((st = check_device()) != CRISP_OK) return st;
    return from_cuda(launch_select_vs(s, *params, vmass, smass, route, vbits, sbits, status_of(ws), stream));
  });
}

crisp_status crisp_select_vs(const crisp_shape* shape, const crisp_params* params, const float* pmap,
                             const uint8_t* route, uint64_t* vmass, uint64_t* smass, uint32_t* vbits,
                             uint32_t* sbits, void* ws, size_t ws_bytes, crisp_stream_t stream) {
  return traced("crisp_select_vs", shape, [&]() -> crisp_status {
    crisp_status st = check_shape(shape);
    if (st != CRISP_OK) return st;
    if ((st = check_params(params)) != CRISP_OK) return st;
    if (!pmap || !route || !vmass || !smass || !vbits || !sbits) return CRISP_ERR_INVALID_ARG;
    if (!aligned16(pmap) || !aligned(vmass, 8) || !aligned(smass, 8) || !aligned(vbits, 4) || !aligned(sbits, 4))
      return CRISP_ERR_ALIGN;
    const crisp_shape s = normalised(*shape);
    if ((st = check_ws(s, ws, ws_bytes)) != CRISP_OK) return st;
    if ((st = check_device()) != CRISP_OK) return st;
    char* wsb = static_cast<char*>(ws);
    auto* rmass = reinterpret_cast<uint64_t*>(wsb + scratch_layout(s).rmass);
    if (launch_block_masses(s, pmap, vmass, smass, rmass, wsb, stream) != cudaSuccess) return CRISP_ERR_CUDA;
    return from_cuda(launch_select_vs(s, *params, vmass, smass, route, vbits, sbits, status_of(ws), stream));
  });
}

crisp_status crisp_pe_pool(const crisp_shape* shape, const void* q, const void* k, const uint8_t* route, float* pbar,
                           void* ws, size_t ws_bytes, crisp_stream_t stream) {
  return traced("crisp_pe_pool", shape, [&]() -> crisp_status {
    crisp_status st = check_shape(shape);
    if (st != CRISP_OK) return st;
    if (!q || !k || !route || !pbar) return CRISP_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(pbar)) return CRISP_ERR_ALIGN;
    const crisp_shape s = normalised(*shape);
    if ((st = check_ws(s, ws, ws_bytes)) != CRISP_OK) return st;
    if ((st = check_device()) != CRISP_OK) return st;
    return from_cuda(launch_pe_map(s, q, k, route, pbar, static_cast<char*>(ws), stream));
  });
}

crisp_status crisp_select_pe(const crisp_shape* shape, const crisp_params* params, const float* pbar,
                             const uint8_t* route, uint32_t* pebits, void* ws, size_t ws_bytes,
                             crisp_stream_t stream) {
  return traced("crisp_select_pe", shape, [&]() -> crisp_status {
    crisp_status st = check_shape(shape);
    if (st != CRISP_OK) return st;
    if ((st = check_params(params)) != CRISP_OK) return st;
    if (!pbar || !route || !pebits) return CRISP_ERR_INVALID_ARG;
    if (!aligned(pbar, 4) || !aligned(pebits, 4)) return CRISP_ERR_ALIGN;
    const crisp_shape s = normalised(*shape);
    if ((st = check_ws(s, ws, ws_bytes)) != CRISP_OK) return st;
    if ((st = check_device()) != CRISP_OK) return st;
    return from_cuda(launch_select_pe(s, *params, pbar, route, pebits, status_of(ws), stream));
  });
}

crisp_status crisp_build_mask(const crisp_shape* shape, const uint8_t* route, const uint32_t* vbits,
                              const uint32_t* sbits, const uint32_t* pebits, uint32_t* rowbits, int32_t* counts,
                              int32_t* order, void* ws, size_t ws_bytes, crisp_stream_t stream) {
  return traced("crisp_build_mask", shape, [&]() -> crisp_status {
    crisp_status st = check_shape(shape);
    if (st != CRISP_OK) return st;
    if (!route || !vbits || !sbits || !pebits || !rowbits || !counts || !order) return CRISP_ERR_INVALID_ARG;
    if (!aligned(vbits, 4) || !aligned(sbits, 4) || !aligned(pebits, 4) || !aligned(rowbits, 4) ||
        !aligned(counts, 4) || !aligned(order, 4))
      return CRISP_ERR_ALIGN;
    const crisp_shape s = normalised(*shape);
    if ((st = check_ws(s, ws, ws_bytes)) != CRISP_OK) return st;
    if ((st = check_device()) != CRISP_OK) return st;
    return from_cuda(
        launch_build_mask(s, route, vbits, sbits, pebits, rowbits, counts, order, static_cast<char*>(ws), stream));
  });
}

static crisp_status attention_common(const crisp_shape* shape, const void* q, const void* k, const void* v,
                                     const uint32_t* rowbits, const int32_t* order, void* out, void* ws,
                                     size_t ws_bytes, crisp_stream_t stream, bool dense) {
  crisp_status st = check_shape(shape, 0);
  if (st != CRISP_OK) return st;
  if (shape->seq_len == 0) return CRISP_OK;  // an empty input: nothing to compute
  if (!q || !k || !v || !out || (!dense && !rowbits)) return CRISP_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return CRISP_ERR_ALIGN;
  if (!dense && (!aligned(rowbits, 4) || !aligned(order, 4))) return CRISP_ERR_ALIGN;
  const crisp_shape s = normalised(*shape);
  if ((st = check_ws(s, ws, ws_bytes)) != CRISP_OK) return st;
  if ((st = check_device()) != CRISP_OK) return st;
  TmaMaps maps;
  if ((st = make_map(&maps.q, q, s.hq, s.seq_len, s.q_head_stride, s.q_tok_stride)) != CRISP_OK) return st;
  if ((st = make_map(&maps.k, k, s.hkv, s.seq_len, s.kv_head_stride, s.kv_tok_stride)) != CRISP_OK) return st;
  if ((st = make_kv_maps(&maps, k, v, s)) != CRISP_OK) return st;
  return from_cuda(launch_attention(s, maps, rowbits, order, out, static_cast<char*>(ws), dense, stream));
}

crisp_status crisp_sparse_prefill_mask(const crisp_shape* shape, const void* q, const void* k, const void* v,
                                       const uint32_t* rowbits, const int32_t* order, void* out, void* ws,
                                       size_t ws_bytes, crisp_stream_t stream) {
  return traced("crisp_sparse_prefill_mask", shape, [&]() -> crisp_status {
    return attention_common(shape, q, k, v, rowbits, order, out, ws, ws_bytes, stream, false);
  });
}

crisp_status crisp_sparse_prefill(const crisp_shape* shape, const void* q, const void* k, const void* v,
                                  const uint8_t* route, const uint32_t* vbits, const uint32_t* sbits,
                                  const uint32_t* pebits, void* out, void* ws, size_t ws_bytes,
                                  crisp_stream_t stream) {
  return traced("crisp_sparse_prefill", shape, [&]() -> crisp_status {
    crisp_status st = check_shape(shape);
    if (st != CRISP_OK) return st;
    if (!q || !k || !v || !out || !route || !vbits || !sbits || !pebits) return CRISP_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return CRISP_ERR_ALIGN;
    if (!aligned(vbits, 4) || !aligned(sbits, 4) || !aligned(pebits, 4)) return CRISP_ERR_ALIGN;
    const crisp_shape s = normalised(*shape);
    if ((st = check_ws(s, ws, ws_bytes)) != CRISP_OK) return st;
    if ((st = check_device()) != CRISP_OK) return st;
    // A7 into the workspace, then A8 over that mask in its schedule.
    char* wsb = static_cast<char*>(ws);
    const ScratchLayout L = scratch_layout(s);
    auto* rowbits = reinterpret_cast<uint32_t*>(wsb + L.rowbits);
    auto* counts = reinterpret_cast<int32_t*>(wsb + L.counts);
    auto* order = reinterpret_cast<int32_t*>(wsb + L.order);
    TmaMaps maps;
    if ((st = make_map(&maps.q, q, s.hq, s.seq_len, s.q_head_stride, s.q_tok_stride)) != CRISP_OK) return st;
    if ((st = make_map(&maps.k, k, s.hkv, s.seq_len, s.kv_head_stride, s.kv_tok_stride)) != CRISP_OK) return st;
    if ((st = make_kv_maps(&maps, k, v, s)) != CRISP_OK) return st;
    if (launch_build_mask(s, route, vbits, sbits, pebits, rowbits, counts, order, wsb, stream) != cudaSuccess)
      return CRISP_ERR_CUDA;
    return from_cuda(launch_attention(s, maps, rowbits, order, out, wsb, false, stream));
  });
}

crisp_status crisp_dense_prefill(const crisp_shape* shape, const void* q, const void* k, const void* v, void* out,
                                 void* ws, size_t ws_bytes, crisp_stream_t stream) {
  return traced("crisp_dense_prefill", shape, [&]() -> crisp_status {
    return attention_common(shape, q, k, v, nullptr, nullptr, out, ws, ws_bytes, stream, true);
  });
}

crisp_status crisp_layer_views_get(const crisp_shape* shape, void* ws, crisp_layer_views* views) {
  return traced("crisp_layer_views_get", shape, [&]() -> crisp_status {
    crisp_status st = check_shape(shape, 0);
    if (st != CRISP_OK) return st;
    if (!ws || !views) return CRISP_ERR_INVALID_ARG;
    const LayerLayout L = layer_layout(*shape);
    char* b = static_cast<char*>(ws);
    views->vmass = reinterpret_cast<uint64_t*>(b + L.vmass);
    views->smass = reinterpret_cast<uint64_t*>(b + L.smass);
    views->rmass = reinterpret_cast<uint64_t*>(b + L.rmass);
    views->cstruct = reinterpret_cast<uint64_t*>(b + L.cstruct);
    views->total = reinterpret_cast<uint64_t*>(b + L.total_mass);
    views->route = reinterpret_cast<uint8_t*>(b + L.route);
    views->vbits = reinterpret_cast<uint32_t*>(b + L.vbits);
    views->sbits = reinterpret_cast<uint32_t*>(b + L.sbits);
    views->pbar = reinterpret_cast<float*>(b + L.pbar);
    views->pebits = reinterpret_cast<uint32_t*>(b + L.pebits);
    views->rowbits = reinterpret_cast<uint32_t*>(b + L.rowbits);
    views->counts = reinterpret_cast<int32_t*>(b + L.counts);
    views->order = reinterpret_cast<int32_t*>(b + L.order);
    return CRISP_OK;
  });
}

}  // extern "C"

namespace crisp {
namespace {

// A1..A8 for one (normalised, validated) shape; intermediates in ws.
crisp_status run_layer(const crisp_shape& s, const crisp_params& p, const void* q, const void* k, const void* v,
                       void* out, void* ws, cudaStream_t stream) {
  crisp_layer_views w;
  crisp_layer_views_get(&s, ws, &w);
  TmaMaps maps;
  crisp_status st;
  if ((st = make_map(&maps.q, q, s.hq, s.seq_len, s.q_head_stride, s.q_tok_stride)) != CRISP_OK) return st;
  if ((st = make_map(&maps.k, k, s.hkv, s.seq_len, s.kv_head_stride, s.kv_tok_stride)) != CRISP_OK) return st;
  if ((st = make_kv_maps(&maps, k, v, s)) != CRISP_OK) return st;
  char* wsb = static_cast<char*>(ws);
  // Length gate: below it the layer is plain dense attention. Below two
  // blocks the method has no candidates (and k_min keeps every block of up
  // to 8), so such layers are dense too.
  if (s.seq_len < p.dense_below || s.seq_len < kMinSeqMethod)
    return from_cuda(launch_attention(s, maps, nullptr, nullptr, out, wsb, true, stream));
  if (launch_proxy_masses(s, maps, w.vmass, w.smass, w.rmass, wsb, stream) != cudaSuccess) return CRISP_ERR_CUDA;
  if (p.route_mode == CRISP_ROUTE_JSD) {
    // The comparator needs the pooled estimate of every head before routing
    // (a zero route array selects all heads), then routes by divergence.
    if (cudaMemsetAsync(w.route, 0, static_cast<size_t>(s.hq), stream) != cudaSuccess ||
        launch_pe_map(s, q, k, w.route, w.pbar, wsb, stream) != cudaSuccess ||
        launch_route_jsd(s, p, w.vmass, w.pbar, nullptr, w.route, status_of(ws), stream) != cudaSuccess)
      return CRISP_ERR_CUDA;
  } else if (launch_route(s, p, w.vmass, w.rmass, w.cstruct, w.total, w.route, status_of(ws), stream) != cudaSuccess ||
             launch_pe_map(s, q, k, w.route, w.pbar, wsb, stream) != cudaSuccess) {
    return CRISP_ERR_CUDA;
  }
  if (launch_select_vs(s, p, w.vmass, w.smass, w.route, w.vbits, w.sbits, status_of(ws), stream) != cudaSuccess ||
      launch_select_pe(s, p, w.pbar, w.route, w.pebits, status_of(ws), stream) != cudaSuccess ||
      launch_build_mask(s, w.route, w.vbits, w.sbits, w.pebits, w.rowbits, w.counts, w.order, wsb, stream) !=
          cudaSuccess ||
      launch_attention(s, maps, w.rowbits, w.order, out, wsb, false, stream) != cudaSuccess)
    return CRISP_ERR_CUDA;
  return CRISP_OK;
}

bool contiguous(const crisp_shape& s) {
  const int64_t plane = static_cast<int64_t>(s.seq_len) * kD;
  return s.q_tok_stride == kD && s.kv_tok_stride == kD && s.o_tok_stride == kD && s.q_head_stride == plane &&
         s.kv_head_stride == plane && s.o_head_stride == plane;
}

}  // namespace
}  // namespace crisp

// Sequence length from which the host-buffer path uploads half a kv group
// per chunk (measured: 256k and 512k layers gain 1-4 ms, a 32k layer loses 1).
constexpr int kHalfGroupChunkLen = 131072;

// Streams and events of the host-buffer path (created by
// crisp_host_pipeline_create on the current device).
struct crisp_host_pipeline {
  static constexpr int kRing = 4;  // events are reused round-robin across kv groups
  int device;
  cudaStream_t in, out, comp;  // comp: the second compute stream
  cudaEvent_t start, done, comp_done;
  cudaEvent_t ev_in[kRing], ev_comp[kRing];
};

extern "C" {

crisp_status crisp_prefill_layer(const crisp_shape* shape, const crisp_params* params, const void* q, const void* k,
                                 const void* v, void* out, void* ws, size_t ws_bytes, crisp_stream_t stream) {
  return traced("crisp_prefill_layer", shape, [&]() -> crisp_status {
    crisp_status st = check_shape(shape, 0);
    if (st != CRISP_OK) return st;
    if ((st = check_params(params)) != CRISP_OK) return st;
    if ((st = check_block_slices(params)) != CRISP_OK) return st;
    if (shape->seq_len == 0) return CRISP_OK;  // an empty input: nothing to compute
    if (!q || !k || !v || !out) return CRISP_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return CRISP_ERR_ALIGN;
    const crisp_shape s = normalised(*shape);
    if (!ws) return CRISP_ERR_WORKSPACE;
    if (!aligned(ws, kAlign)) return CRISP_ERR_ALIGN;
    if (ws_bytes < layer_layout(s).total) return CRISP_ERR_WORKSPACE;
    if ((st = check_device()) != CRISP_OK) return st;
    return run_layer(s, *params, q, k, v, out, ws, stream);
  });
}

crisp_status crisp_host_pipeline_create(crisp_host_pipeline** pipeline) {
  return traced("crisp_host_pipeline_create", nullptr, [&]() -> crisp_status {
    if (!pipeline) return CRISP_ERR_INVALID_ARG;
    *pipeline = nullptr;
    crisp_status st = check_device();
    if (st != CRISP_OK) return st;
    auto* p = new (std::nothrow) crisp_host_pipeline();
    if (!p) return CRISP_ERR_CUDA;
    bool ok = cudaGetDevice(&p->device) == cudaSuccess &&
              cudaStreamCreateWithFlags(&p->in, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&p->out, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&p->comp, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&p->start, cudaEventDisableTiming) == cudaSuccess &&
              cudaEventCreateWithFlags(&p->done, cudaEventDisableTiming) == cudaSuccess &&
              cudaEventCreateWithFlags(&p->comp_done, cudaEventDisableTiming) == cudaSuccess;
    for (int i = 0; ok && i < crisp_host_pipeline::kRing; ++i)
      ok = cudaEventCreateWithFlags(&p->ev_in[i], cudaEventDisableTiming) == cudaSuccess &&
           cudaEventCreateWithFlags(&p->ev_comp[i], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
      crisp_host_pipeline_destroy(p);
      return CRISP_ERR_CUDA;
    }
    *pipeline = p;
    return CRISP_OK;
  });
}

crisp_status crisp_host_pipeline_destroy(crisp_host_pipeline* p) {
  return traced("crisp_host_pipeline_destroy", nullptr, [&]() -> crisp_status {
    if (!p) return CRISP_OK;
    // Objects never created are null handles; destroying those is skipped.
    if (p->in) cudaStreamSynchronize(p->in);
    if (p->out) cudaStreamSynchronize(p->out);
    if (p->comp) cudaStreamSynchronize(p->comp);
    for (int i = 0; i < crisp_host_pipeline::kRing; ++i) {
      if (p->ev_in[i]) cudaEventDestroy(p->ev_in[i]);
      if (p->ev_comp[i]) cudaEventDestroy(p->ev_comp[i]);
    }
    if (p->start) cudaEventDestroy(p->start);
    if (p->done) cudaEventDestroy(p->done);
    if (p->comp_done) cudaEventDestroy(p->comp_done);
    if (p->comp) cudaStreamDestroy(p->comp);
    if (p->in) cudaStreamDestroy(p->in);
    if (p->out) cudaStreamDestroy(p->out);
    delete p;
    return CRISP_OK;
  });
}

}  // extern "C"

namespace crisp {
namespace {
// The second sub-workspace's status word folded into the caller's (the
// first error stays).
__global__ void merge_status_kernel(DevStatus* dst, const DevStatus* src) {
  if (dst->code == 0 && src->code != 0) {
    dst->detail = src->detail;
    dst->code = src->code;
  }
}
}  // namespace
}  // namespace crisp

extern "C" {

crisp_status crisp_prefill_layer_host(crisp_host_pipeline* pipeline, const crisp_shape* shape,
                                      const crisp_params* params, const void* q_host, const void* k_host,
                                      const void* v_host, void* out_host, void* q, void* k, void* v, void* out,
                                      void* ws, size_t ws_bytes, crisp_stream_t stream) {
  return traced("crisp_prefill_layer_host", shape, [&]() -> crisp_status {
    if (!pipeline) return CRISP_ERR_INVALID_ARG;
    crisp_status st = check_shape(shape, 0);
    if (st != CRISP_OK) return st;
    if ((st = check_params(params)) != CRISP_OK) return st;
    if ((st = check_block_slices(params)) != CRISP_OK) return st;
    if (shape->seq_len == 0) return CRISP_OK;  // an empty input: nothing to compute
    if (!q_host || !k_host || !v_host || !out_host || !q || !k || !v || !out) return CRISP_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return CRISP_ERR_ALIGN;
    const crisp_shape s = normalised(*shape);
    if (!contiguous(s)) return CRISP_ERR_SHAPE;
    if (!ws) return CRISP_ERR_WORKSPACE;
    if (!aligned(ws, kAlign)) return CRISP_ERR_ALIGN;
    if (ws_bytes < layer_layout(s).total) return CRISP_ERR_WORKSPACE;
    if ((st = check_device()) != CRISP_OK) return st;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev != pipeline->device) return CRISP_ERR_DEVICE;

    // The layer in chunks of query heads within a kv group, the group's K and
    // V uploaded with its first chunk: the upload of chunk c+1 and the
    // download of chunk c-1 overlap the compute of chunk c, and consecutive
    // chunks alternate between two compute streams (each with its own part of
    // the workspace), so that one chunk's short selection kernels run beside
    // the previous chunk's attention. Long sequences use half a group per
    // chunk (when G is even), and ramp the chunks of the first and last
    // groups, so that the pipeline fills and drains with a single head;
    // shorter ones a whole group per chunk, where the extra launches and
    // copies would cost more than the shorter fill.
    const int G = s.hq / s.hkv;
    const int hc = (G % 2 == 0 && s.seq_len >= kHalfGroupChunkLen) ? G / 2 : G;  // query heads per chunk
    const size_t plane = static_cast<size_t>(s.seq_len) * kD * 2;  // bytes of one head
    crisp_shape sub = s;
    sub.hq = hc;
    sub.hkv = 1;
    auto* p = pipeline;
    cudaStream_t cs = stream;
    auto cb = [](const void* b, size_t off) { return static_cast<const char*>(b) + off; };
    auto mb = [](void* b, size_t off) { return static_cast<char*>(b) + off; };
    // Two compute streams, each with its own part of the workspace, when it
    // holds two chunks' intermediates and there are several chunks.
    const size_t sub_bytes = up(layer_layout(sub).total);
    const bool dual = hc < s.hq && 2 * sub_bytes <= ws_bytes;
    void* ws1 = static_cast<char*>(ws) + sub_bytes;
    // Work already on `stream` (earlier users of these buffers) comes first.
    if (cudaEventRecord(p->start, cs) != cudaSuccess || cudaStreamWaitEvent(p->in, p->start, 0) != cudaSuccess ||
        cudaStreamWaitEvent(p->out, p->start, 0) != cudaSuccess ||
        (dual && (cudaStreamWaitEvent(p->comp, p->start, 0) != cudaSuccess ||
                  cudaMemsetAsync(ws1, 0, sizeof(DevStatus), p->comp) != cudaSuccess)))
      return CRISP_ERR_CUDA;
    // Chunk sizes in heads, in order: the first kv group ramps up 1, 2, 4, ...
    // (each at most hc) and the last ramps down the same way, so that the
    // pipeline fills and drains with one head but few chunks are small; the
    // groups between take hc heads per chunk.
    const bool ramp = hc > 1 && s.seq_len >= kHalfGroupChunkLen;
    std::vector<int> up_ramp;
    for (int at = 0, sz = 1; at < G; sz = std::min(2 * sz, hc)) {
      up_ramp.push_back(std::min(sz, G - at));
      at += up_ramp.back();
    }
    std::vector<int> sizes;
    for (int grp = 0; grp < s.hkv; ++grp) {
      if (ramp && grp == 0)
        sizes.insert(sizes.end(), up_ramp.begin(), up_ramp.end());
      else if (ramp && grp == s.hkv - 1)
        sizes.insert(sizes.end(), up_ramp.rbegin(), up_ramp.rend());
      else
        sizes.insert(sizes.end(), G / hc, hc);
    }
    int c = 0;
    for (int h0 = 0; h0 < s.hq; ++c) {
      const int size = sizes[c];  // heads in this chunk (within one kv group)
      sub.hq = size;
      const int e = c % crisp_host_pipeline::kRing;
      const int g = h0 / G;  // the chunk's kv group
      const size_t kv_off = static_cast<size_t>(g) * plane, q_off = static_cast<size_t>(h0) * plane;
      if (h0 % G == 0 &&
          (cudaMemcpyAsync(mb(k, kv_off), cb(k_host, kv_off), plane, cudaMemcpyHostToDevice, p->in) != cudaSuccess ||
           cudaMemcpyAsync(mb(v, kv_off), cb(v_host, kv_off), plane, cudaMemcpyHostToDevice, p->in) != cudaSuccess))
        return CRISP_ERR_CUDA;
      cudaStream_t sc = (dual && (c & 1)) ? p->comp : cs;
      void* wsc = (dual && (c & 1)) ? ws1 : ws;
      if (cudaMemcpyAsync(mb(q, q_off), cb(q_host, q_off), size * plane, cudaMemcpyHostToDevice, p->in) != cudaSuccess ||
          cudaEventRecord(p->ev_in[e], p->in) != cudaSuccess || cudaStreamWaitEvent(sc, p->ev_in[e], 0) != cudaSuccess)
        return CRISP_ERR_CUDA;
      if ((st = run_layer(sub, *params, mb(q, q_off), mb(k, kv_off), mb(v, kv_off), mb(out, q_off), wsc, sc)) !=
          CRISP_OK)
        return st;
      if (cudaEventRecord(p->ev_comp[e], sc) != cudaSuccess || cudaStreamWaitEvent(p->out, p->ev_comp[e], 0) != cudaSuccess ||
          cudaMemcpyAsync(mb(out_host, q_off), cb(out, q_off), size * plane, cudaMemcpyDeviceToHost, p->out) != cudaSuccess)
        return CRISP_ERR_CUDA;
      h0 += size;
    }
    // `stream` completes after the last download, with the second compute
    // stream's status folded into the caller's.
    if (dual) {
      if (cudaEventRecord(p->comp_done, p->comp) != cudaSuccess || cudaStreamWaitEvent(cs, p->comp_done, 0) != cudaSuccess)
        return CRISP_ERR_CUDA;
      merge_status_kernel<<<1, 1, 0, cs>>>(static_cast<DevStatus*>(ws), static_cast<const DevStatus*>(ws1));
      if (cudaGetLastError() != cudaSuccess) return CRISP_ERR_CUDA;
    }
    if (cudaEventRecord(p->done, p->out) != cudaSuccess || cudaStreamWaitEvent(cs, p->done, 0) != cudaSuccess)
      return CRISP_ERR_CUDA;
    return CRISP_OK;
  });
}

}  // extern "C"

namespace crisp {
namespace {

// One thread waits on an mbarrier that nothing arrives at, through the same
// bounded wait the pipeline kernels use; the wait must give up and record
// CRISP_ERR_TIMEOUT in the status word, and the kernel must return.
__global__ void wait_selftest_kernel(DevStatus* status, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar, 1);
    ptx::fence_mbar_init();
    abort = 0;
  }
  __syncthreads();
  if (threadIdx.x == 0 && !ptx::mbar_wait(&bar, 0, &abort, limit_ns)) report_error(status, CRISP_ERR_TIMEOUT, 0xF01);
}

}  // namespace
}  // namespace crisp

extern "C" {

crisp_status crisp_wait_selftest(void* ws, size_t ws_bytes, int64_t limit_ns, crisp_stream_t stream) {
  return traced("crisp_wait_selftest", nullptr, [&]() -> crisp_status {
    if (!ws || ws_bytes < sizeof(DevStatus)) return CRISP_ERR_WORKSPACE;
    if (limit_ns <= 0 || limit_ns > 10000000000ll) return CRISP_ERR_INVALID_ARG;
    crisp_status st = check_device();
    if (st != CRISP_OK) return st;
    wait_selftest_kernel<<<1, 32, 0, stream>>>(static_cast<DevStatus*>(ws), static_cast<unsigned long long>(limit_ns));
    return from_cuda(cudaGetLastError());
  });
}

crisp_status crisp_read_status(const void* ws, crisp_stream_t stream, crisp_status* status) {
  return traced("crisp_read_status", nullptr, [&]() -> crisp_status {
    if (!ws || !status) return CRISP_ERR_INVALID_ARG;
    DevStatus host{};
    if (cudaMemcpyAsync(&host, ws, sizeof(host), cudaMemcpyDeviceToHost, stream) != cudaSuccess) return CRISP_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return CRISP_ERR_CUDA;
    *status = static_cast<crisp_status>(host.code);
    return CRISP_OK;
  });
}

const char* crisp_status_string(crisp_status status) {
  switch (status) {
    case CRISP_OK: return "ok";
    case CRISP_ERR_INVALID_ARG: return "invalid argument";
    case CRISP_ERR_SHAPE: return "unsupported shape";
    case CRISP_ERR_ALIGN: return "pointer or stride not 16-byte aligned";
    case CRISP_ERR_WORKSPACE: return "workspace missing or too small";
    case CRISP_ERR_CUDA: return "CUDA runtime error";
    case CRISP_ERR_TIMEOUT: return "device wait timed out";
    case CRISP_ERR_DEVICE: return "device is not sm_103";
    case CRISP_ERR_BOUNDS: return "device index outside its buffer (bounds-checking build)";
  }
  return "unknown status";
}

}  // extern "C"
