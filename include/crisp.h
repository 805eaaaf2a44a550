/*
 * crisp.h -- C ABI of the CRISP sparse-prefill library (GB300, sm_103a).
 *
 * CRISP ("CRISP: Cliff-awaRe Input-adaptive Sparse Prefilling with
 * Structural-Mass-Motivated Routing", arXiv 2609.01925) decides, per layer and
 * per attention head, which 128x128 blocks of the causal attention matrix to
 * compute, then computes exact softmax attention over those blocks:
 *
 *   A1 crisp_proxy_map          proxy attention map of the last query block
 *   A3 crisp_block_masses       vertical / slash block masses of that map
 *   A1+A3 crisp_proxy_masses    the same masses straight from q and k (map not stored)
 *   A2 crisp_route_cstruct      C_struct routing from the map: Vertical-Slash or Pooled-Estimation
 *      crisp_route_cstruct_masses  the same from the block masses (what the layer runs)
 *      crisp_route_jsd          FlexPrefill's divergence routing (the rule CRISP replaces)
 *   A4 crisp_select_vs          sink-aware noise-floor selection from the map (VS heads)
 *      crisp_select_vs_masses   the same from the block masses (what the layer runs)
 *   A5 crisp_pe_pool            pooled attention estimate (PE heads)
 *   A6 crisp_select_pe          PE block selection (gamma coverage or noise floor)
 *   A7 crisp_build_mask         per-head sparse block mask and attention schedule
 *   A8 crisp_sparse_prefill     causal GQA block-sparse attention over the index sets
 *      crisp_sparse_prefill_mask  the same over a block mask from crisp_build_mask
 *   A9 crisp_dense_prefill      the same kernel over every causal block
 *   crisp_prefill_layer         A1..A8 in order, intermediates in the workspace
 *   crisp_prefill_layer_host    the same from host buffers, copies overlapped with compute
 *   crisp_proxy_map_noalloc     A1 without a caller workspace (static scratch)
 *   crisp_wait_selftest         failure detection: a bounded wait that must time out
 *
 * Conventions (every function):
 *  - Pointers are DEVICE pointers unless marked "host". The caller owns and
 *    allocates every buffer, including the workspace; the library allocates
 *    and frees no memory, and creates CUDA objects only in
 *    crisp_host_pipeline_create (three streams and their events).
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *    stream); calls return without synchronising, except crisp_read_status.
 *  - Argument errors are detected on the host, returned synchronously, and
 *    nothing is launched. Errors found on the device (a bounded wait that ran
 *    out) are recorded in the workspace status word; read it with
 *    crisp_read_status. No C++ exception crosses this boundary.
 *  - Fixed sizes: head_dim = 128, block = 128 tokens, batch 1 (a batch is a
 *    loop over calls). seq_len = n <= 2^20, any n: blocks are aligned at
 *    token 0, nb = ceil(n/128), and when 128 does not divide n the last block
 *    is short (n - 128*(nb-1) tokens). The method's steps (A1..A7) need
 *    n >= 256 (the sink block and at least one more); attention, the whole
 *    layer and the workspace sizes take any n >= 0, and n = 0 (an empty
 *    input) launches nothing and returns CRISP_OK.
 *  - bf16 tensors are [heads][tokens][128] with element strides per head and
 *    per token (the 128 features contiguous). For the TMA copies every
 *    pointer must be 16-byte aligned and every stride a multiple of 8
 *    elements.
 *  - Bitsets: bit c of a row is (word[c >> 5] >> (c & 31)) & 1; a row of nb
 *    bits takes W = ceil(nb / 32) uint32 words.
 *  - Rational parameters (tau, alpha, gamma) are compared exactly in integer
 *    arithmetic; masses are integer sums of Q32 quanta, q(p) = round-half-
 *    even(p * 2^32), so index sets do not depend on summation order.
 */
#ifndef CRISP_H_
#define CRISP_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define CRISP_API __attribute__((visibility("default")))
#else
#define CRISP_API
#endif

typedef struct CUstream_st* crisp_stream_t; /* same type as cudaStream_t */

typedef enum crisp_status {
  CRISP_OK = 0,
  CRISP_ERR_INVALID_ARG = 1, /* null pointer or parameter out of range */
  CRISP_ERR_SHAPE = 2,       /* unsupported shape (see limits above) */
  CRISP_ERR_ALIGN = 3,       /* pointer or stride not 16-byte aligned */
  CRISP_ERR_WORKSPACE = 4,   /* workspace null or smaller than required */
  CRISP_ERR_CUDA = 5,        /* a CUDA runtime call failed (launch, copy) */
  CRISP_ERR_TIMEOUT = 6,     /* device: a bounded wait inside a kernel ran out */
  CRISP_ERR_DEVICE = 7,      /* the current device is not sm_103 */
  CRISP_ERR_BOUNDS = 8       /* device, bounds-checking build only: an index fell outside its
                                buffer; the access was skipped (the release build has no checks) */
} crisp_status;

typedef enum crisp_pe_mode {
  CRISP_PE_GAMMA = 0, /* cumulative coverage gamma (the paper's PE rule) */
  CRISP_PE_NOISE = 1  /* the noise-floor rule applied to each pooled row */
} crisp_pe_mode;

/* Head routing: CRISP's structural mass (default) or the Jensen-Shannon
 * divergence rule of FlexPrefill that CRISP replaces (a comparator). */
typedef enum crisp_route_mode {
  CRISP_ROUTE_CSTRUCT = 0,
  CRISP_ROUTE_JSD = 1
} crisp_route_mode;

/* Vertical-Slash block selection: CRISP's sink-aware noise floor (default)
 * or FlexPrefill's cumulative coverage (a comparator). */
typedef enum crisp_vs_mode {
  CRISP_VS_NOISE = 0,
  CRISP_VS_GAMMA = 1
} crisp_vs_mode;

/* Problem shape. Strides are in elements. scale = 0 selects 1/sqrt(128). */
typedef struct crisp_shape {
  int32_t hq;       /* query heads */
  int32_t hkv;      /* key/value heads; hq % hkv == 0 (GQA group G = hq/hkv) */
  int32_t head_dim; /* must be 128 */
  int32_t seq_len;  /* n */
  int32_t block;    /* must be 128 */
  int64_t q_head_stride, q_tok_stride;
  int64_t kv_head_stride, kv_tok_stride; /* shared by K and V */
  int64_t o_head_stride, o_tok_stride;
  float scale;
} crisp_shape;

/* Method parameters; crisp_params_default gives the paper's universal
 * configuration: tau_proxy = 1/5, alpha = 1, gamma = 19/20 (PE only),
 * k_min = 8 blocks (1024 tokens) per direction, pe_mode = CRISP_PE_GAMMA,
 * route_mode = CRISP_ROUTE_CSTRUCT, vs_mode = CRISP_VS_NOISE (the comparator
 * fields default to FlexPrefill's settings as we read them: vs_gamma =
 * 95/100, jsd_tau = 0.1), dense_below = 0 (no length gate; the measured
 * sparse/dense crossover on GB300 lies between 4096 and 8192 tokens, so
 * 8192 is the recommended gate), sink_tokens = recency_tokens = 128 (the
 * paper's two slices: the sink is the first 128 key tokens, the recency
 * window the last 128).
 * crisp_route_cstruct (from the map) takes any slice widths; every call that
 * routes from block masses (crisp_route_cstruct_masses, crisp_prefill_layer,
 * crisp_prefill_layer_host) needs both at 128, one block, and returns
 * CRISP_ERR_INVALID_ARG otherwise. */
typedef struct crisp_params {
  uint32_t tau_num, tau_den;     /* 0 <= tau <= 1, tau_den > 0 */
  uint32_t alpha_num, alpha_den; /* alpha_num, alpha_den <= 65535, alpha_den > 0 */
  uint32_t gamma_num, gamma_den; /* 0 <= gamma <= 1, gamma_den > 0 */
  int32_t kmin_blocks;           /* 0 <= kmin_blocks <= 8192 */
  int32_t pe_mode;               /* crisp_pe_mode */
  int32_t route_mode;            /* crisp_route_mode */
  int32_t vs_mode;               /* crisp_vs_mode */
  uint32_t vs_gamma_num, vs_gamma_den; /* coverage of CRISP_VS_GAMMA, 0 <= gamma <= 1 */
  float jsd_tau;                 /* CRISP_ROUTE_JSD: VS iff sqrt(JSD) >= jsd_tau; 0 <= jsd_tau <= 1 */
  int32_t dense_below;           /* crisp_prefill_layer*: n < dense_below runs dense attention only */
  int32_t sink_tokens;           /* C_struct sink slice: key columns [0, sink_tokens), 0 <= . <= 2^20 */
  int32_t recency_tokens;        /* C_struct recency slice: key columns [n - recency_tokens, n), 0 <= . <= 2^20 */
} crisp_params;

/* Fills *p (host) with the defaults above. */
CRISP_API void crisp_params_default(crisp_params* p);

/* Bytes of workspace the step functions need (status word and scratch). */
CRISP_API crisp_status crisp_workspace_size(const crisp_shape* shape, size_t* bytes /* host */);

/* Bytes of workspace crisp_prefill_layer needs (scratch + every intermediate). */
CRISP_API crisp_status crisp_layer_workspace_size(const crisp_shape* shape, size_t* bytes /* host */);

/* Clears the status word at the start of `ws` (asynchronously on `stream`).
 * Call once after allocating a workspace and after reading an error. */
CRISP_API crisp_status crisp_workspace_init(void* ws, size_t ws_bytes, crisp_stream_t stream);

/* A1. Proxy attention map of the last query block (ai.info page, "Key
 * Contributions" 2 and "Methodology": routing reads the proxy attention map
 * the method already computes). For q-head h (kv head h/G) and the rows
 * i = n-128+r, r in [0,128) (the last 128 tokens):
 *   pmap[h][r][j] = softmax_j(scale * q_i . k_j) over j <= i, and 0 for j > i.
 * q: bf16 [hq][n][128] (only the last 128 rows are read); k: bf16
 * [hkv][n][128]; pmap: fp32 [hq][128][ld], ld = 128*nb (= n when 128
 * divides n; columns n..ld-1 are written as 0), contiguous, 16-byte aligned. */
CRISP_API crisp_status crisp_proxy_map(const crisp_shape* shape, const void* q, const void* k, float* pmap, void* ws,
                             size_t ws_bytes, crisp_stream_t stream);

/* crisp_proxy_map without a caller-provided workspace. The paper has no
 * counterpart to this entry point; it exists for callers that cannot
 * allocate device memory when they run this step -- for example a serving
 * engine that hands all free device memory to its own pool at start-up, or
 * code that must not call cudaMalloc because it synchronises the device and
 * would stall work on other streams. Inputs and the output are as for
 * crisp_proxy_map; q, k and pmap are still the caller's buffers.
 *
 * Scratch: the per-chunk softmax statistics live in one 32 MiB array in the
 * library's static device memory, held on every GPU that loads the library
 * until the process exits. A shape needs 256 + 8*128*hq*(2*ceil(nb/16) + 1)
 * bytes of it, rounded up to 256-byte units (the 512k-token, 32-head layer
 * needs about 16.8 MB); larger shapes are rejected with CRISP_ERR_WORKSPACE
 * and nothing is launched. The first call on a device looks up the array's
 * device address (once per device, with that device current) and keeps it
 * for the life of the process, so make that first call before any stream
 * capture, and make no call on a device after cudaDeviceReset on it (the
 * reset releases the library's static memory and the kept address would
 * point at memory the process no longer owns). Every call shares the one
 * array: calls whose kernels overlap on the GPU (other streams, other
 * threads) race and corrupt each other's statistics; calls serialised on one
 * stream are safe. The status word in the array is cleared by every call; a
 * device wait that times out is recorded there: read it with
 * crisp_noalloc_read_status on the same stream before the next call.
 * Allocates nothing (no cudaMalloc/cudaFree, no allocating library call). */
CRISP_API crisp_status crisp_proxy_map_noalloc(const crisp_shape* shape, const void* q, const void* k, float* pmap,
                                               crisp_stream_t stream);

/* The status word of crisp_proxy_map_noalloc's static scratch on the current
 * device: synchronises `stream` and copies the word to *status (host),
 * CRISP_OK or CRISP_ERR_TIMEOUT after the last call. Allocates nothing.
 * Returns CRISP_ERR_CUDA if the stream or the copy failed. */
CRISP_API crisp_status crisp_noalloc_read_status(crisp_stream_t stream, crisp_status* status /* host */);

/* A3. Block masses of the proxy map ("mass at Vertical-Slash compatible
 * positions", ai-feeds page, "方法"). With q(p) the Q32 quantum and row r
 * standing for token i = n-128+r:
 *   vmass[h][c] = sum over rows r and key columns j of block c of q(pmap[h][r][j])
 *   smass[h][s] = sum over (r, j) with j <= i, j >= 128 and
 *                 floor((i - j)/128) == s of q(pmap[h][r][j])
 *   rmass[h]    = sum over rows r and the recency columns j in [n-128, n)
 *                 (= vmass[h][nb-1] when 128 divides n)
 * Sink columns (j < 128) are left out of the slash masses, so the sink cannot
 * raise the slash noise floor. pmap fp32 [hq][128][ld] as crisp_proxy_map
 * writes it; vmass, smass: uint64 [hq][nb]; rmass: uint64 [hq]. */
CRISP_API crisp_status crisp_block_masses(const crisp_shape* shape, const float* pmap, uint64_t* vmass, uint64_t* smass,
                                uint64_t* rmass, void* ws, size_t ws_bytes, crisp_stream_t stream);

/* A1 and A3 in one pass: the block masses of the proxy map, computed from q
 * and k without storing the map (routing and Vertical-Slash selection read
 * only these masses; ai.info page, "Key Contributions" 2; ai-feeds page,
 * "方法"). Each fp32 probability is formed exactly as crisp_proxy_map stores
 * it and quantised exactly as crisp_block_masses reads it, so vmass and
 * smass (and rmass) are bit-identical to crisp_block_masses(crisp_proxy_map(q,
 * k)). q, k as for crisp_proxy_map; vmass, smass uint64 [hq][nb], rmass
 * uint64 [hq], 8-byte aligned. Saves the 4*hq*128*n-byte map write and its
 * re-read. */
CRISP_API crisp_status crisp_proxy_masses(const crisp_shape* shape, const void* q, const void* k, uint64_t* vmass,
                                          uint64_t* smass, uint64_t* rmass, void* ws, size_t ws_bytes,
                                          crisp_stream_t stream);

/* A2. C_struct routing from the proxy map (ai.info page, "Key Contributions"
 * 2 and "Methodology in Plain English": the share of the map's mass that sits
 * in the sink slice, the first 128 key tokens, and the recency slice, the
 * last 128; tau_proxy = 0.2). With q(p) the Q32 quantum and the slice widths
 * of params (sink_tokens = S, recency_tokens = R; the paper's 128 and 128):
 *   cstruct[h] = sum over rows r and columns j in [0, S) U [n-R, n) of
 *                q(pmap[h][r][j])   (the union: a column in both counts once),
 *   total[h]   = sum over rows r and all columns j of q(pmap[h][r][j]),
 *   route[h]   = 1 (Vertical-Slash) iff tau_den * cstruct >= tau_num * total,
 *                0 (Pooled-Estimation) otherwise.
 * Reads the whole map once (HBM-bound). pmap fp32 [hq][128][ld] as
 * crisp_proxy_map writes it; cstruct, total uint64 [hq], 8-byte aligned;
 * route uint8 [hq]. */
CRISP_API crisp_status crisp_route_cstruct(const crisp_shape* shape, const crisp_params* params, const float* pmap,
                                           uint64_t* cstruct, uint64_t* total, uint8_t* route, void* ws,
                                           size_t ws_bytes, crisp_stream_t stream);

/* A2 from the block masses (what crisp_prefill_layer runs: the masses come
 * from the fused crisp_proxy_masses pass and the map is never stored). With
 * both slices 128 tokens wide the sink slice is key block 0 and the recency
 * slice the recency mass rmass (key block nb-1 when 128 divides n), disjoint
 * for n >= 256:
 *   cstruct[h] = vmass[h][0] + rmass[h],  total[h] = sum_c vmass[h][c],
 *   route[h] as for crisp_route_cstruct; bit-identical to it on the same map.
 * params->sink_tokens and recency_tokens must be 128 (else
 * CRISP_ERR_INVALID_ARG). vmass uint64 [hq][nb]; rmass, cstruct, total
 * uint64 [hq]; route uint8 [hq]. */
CRISP_API crisp_status crisp_route_cstruct_masses(const crisp_shape* shape, const crisp_params* params,
                                                  const uint64_t* vmass, const uint64_t* rmass, uint64_t* cstruct,
                                                  uint64_t* total, uint8_t* route, void* ws, size_t ws_bytes,
                                                  crisp_stream_t stream);

/* A2 comparator: FlexPrefill's routing, which CRISP replaces (ai.info page,
 * "Methodology in Plain English": a pooled attention estimate compared with
 * the per-query attention by Jensen-Shannon divergence). For head h, with
 *   a[c] = vmass[h][c] / sum_c vmass[h][c]   (the last query block's true
 *          attention pooled into key blocks, from the proxy map),
 *   e[c] = pbar[h][nb-1][c]                  (the pooled estimate of that block),
 *   D    = (KL(a || m) + KL(e || m)) / 2,  m = (a + e) / 2, natural log, in fp64,
 *   route[h] = 1 (Vertical-Slash) iff sqrt(D) >= jsd_tau, else 0.
 * pbar: fp32 [hq][nb][nb] holding row nb-1 of EVERY head (crisp_pe_pool with a
 * route array of zeros computes it); jsd: double [hq] (D), or NULL. */
CRISP_API crisp_status crisp_route_jsd(const crisp_shape* shape, const crisp_params* params, const uint64_t* vmass,
                                       const float* pbar, double* jsd, uint8_t* route, void* ws, size_t ws_bytes,
                                       crisp_stream_t stream);

/* A4. Sink-aware noise-floor selection for VS heads, from the block masses
 * (ai.info page, "Methodology in Plain English": a block is kept when its
 * mass is above alpha times the mean background mass of the blocks that are
 * not always retained; k_min is 1024 tokens, 8 blocks, in each direction).
 * Per direction: always-retained vertical {0, nb-1}, slash {0}; candidates
 * [1, nb-2], N of them, mass sum M; keep c iff m[c]*N*alpha_den >
 * alpha_num*M; then fill to min(kmin, available) by (mass desc, index asc).
 * PE heads get empty rows.
 * vs_mode = CRISP_VS_GAMMA (FlexPrefill's cumulative coverage, the rule CRISP
 * replaces): per direction, every block [0, nb-1] is a candidate; keep the
 * shortest (mass desc, index asc) prefix whose mass reaches vs_gamma of the
 * direction's total (vs_gamma_den * prefix >= vs_gamma_num * total), add the
 * always-retained blocks and fill to min(kmin, nb) the same way.
 * vmass, smass: uint64 [hq][nb] (crisp_block_masses or crisp_proxy_masses);
 * vbits, sbits: uint32 [hq][W]. */
CRISP_API crisp_status crisp_select_vs_masses(const crisp_shape* shape, const crisp_params* params,
                                              const uint64_t* vmass, const uint64_t* smass, const uint8_t* route,
                                              uint32_t* vbits, uint32_t* sbits, void* ws, size_t ws_bytes,
                                              crisp_stream_t stream);

/* A4 from the proxy map: crisp_block_masses (A3) then crisp_select_vs_masses,
 * with the masses written out. pmap fp32 [hq][128][ld] as crisp_proxy_map
 * writes it; route uint8 [hq]; vmass, smass uint64 [hq][nb] (outputs);
 * vbits, sbits uint32 [hq][W]. */
CRISP_API crisp_status crisp_select_vs(const crisp_shape* shape, const crisp_params* params, const float* pmap,
                                       const uint8_t* route, uint64_t* vmass, uint64_t* smass, uint32_t* vbits,
                                       uint32_t* sbits, void* ws, size_t ws_bytes, crisp_stream_t stream);

/* A5. Pooled attention estimate for PE heads (the Pooled-Estimation route
 * CRISP keeps from FlexPrefill; ai.info page, "Overview"): block means of q
 * and k (a short last block averaged over its own tokens),
 * pbar[h][b][c] = softmax over c <= b of scale * qbar_b . kbar_c, and 0 for
 * c > b. Rows of VS heads are not written. q, k bf16; pbar fp32
 * [hq][nb][nb], 16-byte aligned. Precision: the means are summed in fp32 and
 * held as hi + lo bf16 pairs (16 significant bits); the logits accumulate
 * hi.hi + hi.lo + lo.hi in fp32 on the tensor cores (lo.lo, 2^-16 of a
 * product, is left out). */
CRISP_API crisp_status crisp_pe_pool(const crisp_shape* shape, const void* q, const void* k, const uint8_t* route,
                                     float* pbar, void* ws, size_t ws_bytes, crisp_stream_t stream);

/* A6. PE block selection per query block b from pbar (ai.info page,
 * "Methodology in Plain English": gamma = 0.95 for the PE path only).
 * CRISP_PE_GAMMA: the shortest prefix of [0, b] ordered by (mass desc, index
 * asc) whose mass reaches gamma of the row (gamma_den*prefix >= gamma_num*
 * total), plus {0, b}. CRISP_PE_NOISE: forced {0, b}, candidates [1, b-1],
 * the A4 rule. Both fill to min(kmin, b+1). VS heads get empty rows.
 * pebits: uint32 [hq][nb][W]. */
CRISP_API crisp_status crisp_select_pe(const crisp_shape* shape, const crisp_params* params, const float* pbar,
                             const uint8_t* route, uint32_t* pebits, void* ws, size_t ws_bytes,
                             crisp_stream_t stream);

/* A7. The per-head sparse mask (ai-feeds page, "方法": the output is a
 * per-head sparse attention mask) as key-block sets per query block qb:
 *   VS head: {kb <= qb : kb in V} U {qb-s, qb-s-1 : s in S} within [0, qb]
 *            (a 128-wide diagonal band at offset block s crosses key blocks
 *            qb-s and qb-s-1);
 *   PE head: pebits row qb within [0, qb].
 * and the attention schedule: kv group by kv group (g = h / G), within a
 * group query blocks descending and the group's heads ascending (a causal
 * row's block count grows with qb, so each group's longest rows run first,
 * and the CTAs in flight gather one kv group's blocks, which stay in L2).
 * rowbits: uint32 [hq][nb][W]; counts: int32 [hq][nb] = blocks per row;
 * order: int32 [hq*nb], order[(g*nb + nb-1-qb)*G + h%G] = h*nb + qb. */
CRISP_API crisp_status crisp_build_mask(const crisp_shape* shape, const uint8_t* route, const uint32_t* vbits,
                                        const uint32_t* sbits, const uint32_t* pebits, uint32_t* rowbits,
                                        int32_t* counts, int32_t* order, void* ws, size_t ws_bytes,
                                        crisp_stream_t stream);

/* A8. Exact causal GQA softmax attention over the selected blocks (ai.info
 * page, "Why This Matters": the attention is exact softmax over the blocks
 * the method keeps), from the index sets of A2, A4 and A6: the mask and the
 * schedule of crisp_build_mask (A7) are built in `ws`, then for token i in
 * query block qb of head h,
 *   out_i = sum_{j in A(i)} softmax_j(scale * q_i . k_j) v_j,
 *   A(i) = { j <= i : block(j) in the head's set for qb (crisp_build_mask) }.
 * Rows with an empty A(i) are written as zeros; only rows i < n are written.
 * q bf16 [hq][n][128]; k, v bf16 [hkv][n][128]; route uint8 [hq]; vbits,
 * sbits uint32 [hq][W]; pebits uint32 [hq][nb][W]; out bf16 [hq][n][128]
 * (o strides). n >= 256 (the index sets need the method's steps). */
CRISP_API crisp_status crisp_sparse_prefill(const crisp_shape* shape, const void* q, const void* k, const void* v,
                                            const uint8_t* route, const uint32_t* vbits, const uint32_t* sbits,
                                            const uint32_t* pebits, void* out, void* ws, size_t ws_bytes,
                                            crisp_stream_t stream);

/* A8 over a block mask: for token i in query block qb of head h,
 *   out_i = sum_{j in A(i)} softmax_j(scale * q_i . k_j) v_j,
 *   A(i) = { j <= i : block(j) in rowbits[h][qb] }.
 * Bits above the diagonal block are ignored; rows with an empty A(i) are
 * written as zeros; only rows i < n are written; any n >= 0. rowbits uint32
 * [hq][nb][W] (crisp_build_mask, or any caller-made mask); order: the
 * schedule from crisp_build_mask, or NULL for the same kv-group-major order
 * (any permutation of the row ids gives the same result). */
CRISP_API crisp_status crisp_sparse_prefill_mask(const crisp_shape* shape, const void* q, const void* k,
                                                 const void* v, const uint32_t* rowbits, const int32_t* order,
                                                 void* out, void* ws, size_t ws_bytes, crisp_stream_t stream);

/* A9. Dense causal attention (A(i) = [0, i]): the exact dense
 * FlashAttention-style baseline the paper measures against (ai.info page,
 * "Methodology in Plain English"). */
CRISP_API crisp_status crisp_dense_prefill(const crisp_shape* shape, const void* q, const void* k, const void* v, void* out,
                                 void* ws, size_t ws_bytes, crisp_stream_t stream);

/* Device views of the intermediates crisp_prefill_layer leaves in `ws`. */
typedef struct crisp_layer_views {
  uint64_t *vmass, *smass, *rmass, *cstruct, *total;
  uint8_t* route;
  uint32_t *vbits, *sbits;
  float* pbar;
  uint32_t *pebits, *rowbits;
  int32_t *counts, *order;
} crisp_layer_views;

/* Fills *views (host) with pointers into `ws` for this shape. */
CRISP_API crisp_status crisp_layer_views_get(const crisp_shape* shape, void* ws, crisp_layer_views* views /* host */);

/* A1..A8 for one layer: block masses of the proxy map (crisp_proxy_masses;
 * the map itself is never stored), routing, VS and PE selection, mask,
 * sparse attention. ws must hold crisp_layer_workspace_size bytes. With
 * route_mode = CRISP_ROUTE_JSD the pooled map is computed for every head and
 * routing is crisp_route_jsd. If seq_len < params->dense_below, or
 * seq_len < 256 (too short for the method, and every block would be kept
 * anyway), the layer is dense attention only and the workspace
 * intermediates are not written. seq_len = 0 launches nothing. */
CRISP_API crisp_status crisp_prefill_layer(const crisp_shape* shape, const crisp_params* params, const void* q, const void* k,
                                 const void* v, void* out, void* ws, size_t ws_bytes, crisp_stream_t stream);

/* Prefill from HOST buffers: the streams and events the host-buffer path
 * uses, created on the current device (the one call of this library that
 * creates CUDA objects; destroy it with crisp_host_pipeline_destroy). */
typedef struct crisp_host_pipeline crisp_host_pipeline;
CRISP_API crisp_status crisp_host_pipeline_create(crisp_host_pipeline** pipeline /* host out */);
/* Waits for the pipeline's streams and destroys them; NULL is a no-op. */
CRISP_API crisp_status crisp_host_pipeline_destroy(crisp_host_pipeline* pipeline);

/* crisp_prefill_layer with q, k, v read from host memory and out written to
 * host memory. The layer is processed in chunks of the query heads of one
 * kv group (half of its G heads when G is even and n >= 131072, with the
 * first and last half group of the layer one head at a time; else all G;
 * every step of the method is per head), the group's K and V uploaded with
 * its first chunk: the upload of chunk c+1 and the download of chunk c-1 run
 * on two of the pipeline's streams while chunk c computes, so the copies
 * overlap the compute. Consecutive chunks compute alternately on `stream`
 * and on the pipeline's third stream, each with its own half of `ws` (when
 * ws holds two chunks' intermediates, as a layer workspace of several
 * chunks does); errors from both land in the status word of `ws`.
 * Results are bit-identical to crisp_prefill_layer.
 * q_host, k_host, v_host, out_host: host, contiguous [heads][n][128] bf16,
 * page-locked for the copies to be asynchronous. q, k, v, out: device
 * buffers of the same sizes (staging; afterwards they hold the inputs and
 * the output). shape: contiguous strides only (else CRISP_ERR_SHAPE). ws:
 * crisp_layer_workspace_size bytes. Ordered after earlier work on `stream`;
 * `stream` completes after the last download. The pipeline must belong to
 * the current device (else CRISP_ERR_DEVICE) and serves one call at a time
 * per stream order. */
CRISP_API crisp_status crisp_prefill_layer_host(crisp_host_pipeline* pipeline, const crisp_shape* shape,
                                                const crisp_params* params, const void* q_host, const void* k_host,
                                                const void* v_host, void* out_host, void* q, void* k, void* v,
                                                void* out, void* ws, size_t ws_bytes, crisp_stream_t stream);

/* Synchronises `stream` and copies the workspace status word to *status
 * (host). Returns CRISP_ERR_CUDA if the stream or the copy failed. */
CRISP_API crisp_status crisp_read_status(const void* ws, crisp_stream_t stream, crisp_status* status /* host */);

/* Failure-detection self-test: launches one kernel that waits, through the
 * same bounded mbarrier wait every pipeline kernel uses, on a barrier that
 * nothing arrives at, for limit_ns (0 < limit_ns <= 10 s). The wait gives up,
 * the kernel records CRISP_ERR_TIMEOUT in the status word of ws and returns,
 * and the context stays usable (crisp_read_status then reports the timeout;
 * crisp_workspace_init clears it). */
CRISP_API crisp_status crisp_wait_selftest(void* ws, size_t ws_bytes, int64_t limit_ns, crisp_stream_t stream);

/* Static description of a status code (never NULL). */
CRISP_API const char* crisp_status_string(crisp_status status);

#ifdef __cplusplus
}
#endif

#endif /* CRISP_H_ */
