/*
 * tq.h -- C ABI of the TurboQuant KV-cache library for GB300 (sm_103a).
 *
 * What it computes (sources are the three TurboQuant pages, cited by title and
 * section):
 *   - Quantize one K or V vector x (head_dim d): store n = ||x||, rotate
 *     u = x / n with the random-sign Walsh-Hadamard transform
 *     y = (1/sqrt d) H_d (s * u), map each y_i to the index of one of 2^b
 *     Lloyd-Max centroids, bit-pack the indices, and for keys optionally add a
 *     1-bit QJL sign sketch of the residual.
 *       "TurboQuant KV 캐시 압축 for llama.cpp", header (WHT + Lloyd-Max + QJL)
 *       and v1.7.0 design decision 4 (internal sign flip + butterfly WHT);
 *       "윈도우용 터보퀀트(TurboQuant) 구현을 개선하다", recap and finding 3
 *       (dense packing: a 3-bit d=128 vector is 48 B of codes + a 4 B norm);
 *       "[GitHub 탐방] TurboQuant 3-bit KV 캐시 압축 — 단일 GPU 재현 기록",
 *       "GPU 세대가 바뀌면" item (1) (2^bits Lloyd-Max centroids per coordinate).
 *   - Asymmetric K/V bit widths and protected boundary layers:
 *       write-up findings 2 and 4 (K4/V2; first and last 4 layers at 8 bits).
 *   - Residual window: the most recent W tokens stay bf16:
 *       single-GPU blog, "실험 설계" (rw = 0 / 128).
 *   - Decode attention: rotate q once, score it against the packed keys
 *     through the centroid table (the WHT cancels between Q and K by
 *     Parseval), softmax, sum V in the rotated domain and inverse-rotate once:
 *       README v1.7.0 decision 4; v1.5.2 changes 1, 2 (fp32 accumulation) and
 *       4 (V needs the inverse rotation at the output); v1.4.2 item 2 and the
 *       v1.5.2 sharpening text (QJL score term from transformed Q and the sign
 *       bits).
 *
 * Conventions fixed where the pages are silent (the library and its test
 * oracle implement each independently):
 *   - Sylvester H (natural order), orthonormal 1/sqrt(d), signs applied first.
 *   - Sign vector per (layer, K|V), shared by all heads; q uses the K signs.
 *   - Codebook: Lloyd-Max for N(0, 1/d), solved in extended precision, then
 *     rounded once to fp32; boundaries are the fp32-rounded midpoints.
 *   - code_i = #{ j : boundary_j < y_i }, compared in fp32 (a tie takes the
 *     lower code).  Norm stored fp32.
 *   - Packing: dense LSB-first bit stream; the code of coordinate i occupies
 *     bits [i*b, i*b+b), stream bit k is bit (k mod 8) of byte k/8.
 *   - Random streams: splitmix64 counter streams keyed per (seed, layer,
 *     K|V, purpose).  QJL matrix S (m x d) is Gaussian via Box-Muller and
 *     rounded to bf16; the residual r = n (y - c[idx]) is sketched in the
 *     rotated domain; bit_j = [ (S r)_j >= 0 ]; gamma = ||r|| stored fp32.
 *   - QJL score term: gamma * sqrt(pi/2) / m * sum_j (S q_rot)_j (2 bit_j - 1).
 *
 * Memory and ownership: the caller allocates every buffer (device memory for
 * planes, tables, workspace, inputs and outputs); the library allocates
 * nothing at run time.  The query and the output of the decode calls, and
 * the new tokens (k_new, v_new) of tq_decode_step, may instead be pinned host
 * memory that the device can address (any page-locked allocation on a system
 * with unified addressing): the kernels then read and write them across the
 * host link, which for a decode step's few kilobytes costs less than separate
 * copies.  The other calls take device memory.
 * Its device state is one error word per translation unit plus, on every GPU
 * that loads it, the fixed 8 MiB scratch array of tq_decode_attention_noalloc
 * (reserved at load time, held until exit).  Every device call is
 * asynchronous on the caller's stream (a cudaStream_t passed as void*; NULL =
 * legacy default stream).
 *
 * Errors: arguments are validated on the host before any launch; a bad
 * argument returns TQ_ERR_* and launches nothing.  A launch failure returns
 * TQ_ERR_CUDA.  Faults detected on the device (a bounded wait that ran out,
 * an index check) set the device error word, read by tq_get_device_error().
 */
#ifndef TQ_H_
#define TQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define TQ_VERSION 1

typedef enum {
  TQ_OK = 0,
  TQ_ERR_INVALID_ARG = 1,     /* null pointer, bad size, bad enum value */
  TQ_ERR_UNSUPPORTED = 2,     /* valid request this build does not implement */
  TQ_ERR_ALIGNMENT = 3,       /* a device pointer or stride is not 16-byte aligned */
  TQ_ERR_CUDA = 4,            /* a CUDA runtime call or launch failed */
  TQ_ERR_DEVICE_TIMEOUT = 5,  /* a bounded device-side wait ran out */
  TQ_ERR_DEVICE_BOUNDS = 6,   /* a device-side index check failed */
  TQ_ERR_BUFFER_TOO_SMALL = 7 /* workspace / table buffer smaller than required */
} tq_status;

/* Key modes.  TQ_MODE_MSE_QJL: the 1-bit QJL sketch of the residual
 * ("TurboQuant KV 캐시 압축 for llama.cpp", "QJL 보정 효과": TurboQuant_prod).
 * TQ_MODE_MSE_SIGN: the Direct Sign residual of the same page's v1.1.0
 * ("Direct Sign": the sign of each rotated residual coordinate is stored
 * directly, no projection), with the scale a = mean_i |r_i|; the score gains
 * a <q_rot, 2 bits - 1>. */
typedef enum { TQ_MODE_MSE = 0, TQ_MODE_MSE_QJL = 1, TQ_MODE_MSE_SIGN = 2 } tq_mode;
typedef enum { TQ_DENSITY_GAUSSIAN = 0, TQ_DENSITY_SPHERE_BETA = 1 } tq_density;
typedef enum { TQ_BF16 = 0, TQ_F32 = 1 } tq_dtype;
typedef enum { TQ_KIND_K = 0, TQ_KIND_V = 1 } tq_kind;

/* Problem statement of one model's KV cache.
 *   head_dim         d; a power of two.  The GPU kernels implement d = 128.
 *   n_layers         number of attention layers (>= 1).
 *   k_bits, v_bits   MSE code bits of unprotected layers, in {1,2,3,4,8}.
 *   k_mode           TQ_MODE_MSE, TQ_MODE_MSE_QJL or TQ_MODE_MSE_SIGN (keys
 *                    only; values are always MSE-only: the residual term
 *                    corrects Q.K, not the V sum).
 *   qjl_m            QJL projections per key (multiple of 32, <= 256; 128 is
 *                    the only size the GPU kernels implement).
 *   n_protect_first, n_protect_last, protect_bits
 *                    boundary layers stored at protect_bits (MSE only).
 *   residual_window  W >= 0: the last W tokens of a sequence stay bf16.
 *   density          TQ_DENSITY_GAUSSIAN (N(0,1/d)); SPHERE_BETA is the exact
 *                    coordinate density of a uniform unit vector.
 *   sparse_v         0: exact.  k in 1..120: decode skips the V sum of a 32-token
 *                    chunk when every softmax weight of the chunk is below 2^-k
 *                    of the running maximum (the sparse-V dequant skip that
 *                    "[GitHub 탐방] TurboQuant 3-bit KV 캐시 압축 — 단일 GPU 재현
 *                    기록" cites from a llama.cpp extension); the softmax
 *                    denominator still counts those tokens.  MSE-only keys
 *                    (TQ_ERR_UNSUPPORTED with a key residual term).
 *   seed             seeds every random sign vector and QJL matrix. */
typedef struct {
  int32_t head_dim;
  int32_t n_layers;
  int32_t k_bits;
  int32_t v_bits;
  int32_t k_mode;
  int32_t qjl_m;
  int32_t n_protect_first;
  int32_t n_protect_last;
  int32_t protect_bits;
  int32_t residual_window;
  int32_t density;
  int32_t sparse_v;
  uint64_t seed;
} tq_config;

/* Resolved bits of one layer. */
typedef struct {
  int32_t k_bits;
  int32_t v_bits;
  int32_t k_mode;
} tq_layer_spec;

/* Structure-of-arrays storage of one layer's K or V cache, all device memory,
 * each plane laid out [batch][n_kv_heads][capacity][...] with no padding:
 *   codes      uint8 [.., code_bytes]  code_bytes = head_dim * bits / 8
 *   norms      fp32  [..]              ||x||
 *   qjl_signs  uint8 [.., qjl_m / 8]   QJL keys: sketch bits; Direct Sign keys:
 *                                      [.., head_dim / 8] residual signs; else NULL
 *   qjl_rnorm  fp32  [..]              QJL keys: gamma = ||r||; Direct Sign keys:
 *                                      a = mean |r_i|; else NULL
 *   capacity   tokens per (sequence, kv-head).
 * Every plane pointer must be 16-byte aligned (TQ_ERR_ALIGNMENT). */
typedef struct {
  uint8_t* codes;
  float* norms;
  uint8_t* qjl_signs;
  float* qjl_rnorm;
  int64_t capacity;
} tq_planes;

/* ---------------------------------------------------------------- host */

int tq_version(void);
const char* tq_status_string(tq_status s);

/* Bits of layer `layer` under cfg (protected layers: protect_bits, MSE). */
tq_status tq_layer_spec_get(const tq_config* cfg, int layer, tq_layer_spec* out);

/* Lloyd-Max codebook of 2^bits levels for the rotated-coordinate density
 * ("[GitHub 탐방] TurboQuant 3-bit KV 캐시 압축 — 단일 GPU 재현 기록", "GPU 세대가
 * 바뀌면" (1): each coordinate maps to one of 2^bits Lloyd-Max centroids)
 * (host only).  density TQ_DENSITY_GAUSSIAN: N(0, 1/d);
 * TQ_DENSITY_SPHERE_BETA: the exact density (1 - y^2)^((d-3)/2) / B(1/2,
 * (d-1)/2) of one coordinate of a uniform unit vector in R^d.
 * centroids[2^bits] and boundaries[2^bits - 1] (host memory, caller-owned)
 * receive fp32 values, ascending; symmetric about 0.  bits in {1, 2, 3, 4,
 * 8}; head_dim a power of two >= 2.  TQ_ERR_INVALID_ARG otherwise. */
tq_status tq_make_codebook(int bits, int head_dim, int density, float* centroids,
                           float* boundaries);

/* The +-1 sign vector of (seed, layer, kind), as floats (host only). */
tq_status tq_make_signs(uint64_t seed, int layer, int kind, int head_dim, float* signs);

/* The QJL matrix S of (seed, layer), m x head_dim row-major, as bf16 bit
 * patterns (host only). */
tq_status tq_make_qjl_matrix(uint64_t seed, int layer, int m, int head_dim,
                             uint16_t* s_bf16);

/* Device tables (codebooks, sign vectors, QJL matrices) of a config.
 * tq_tables_bytes gives the size; tq_build_tables fills a HOST buffer of at
 * least that size, which the caller copies verbatim into device memory and
 * passes as `tables` to every device call below.  Layout is private. */
size_t tq_tables_bytes(const tq_config* cfg);
tq_status tq_build_tables(const tq_config* cfg, void* host_buf, size_t bytes);

/* Bytes of the four planes of layer/kind for batch x n_kv_heads x capacity
 * vectors: sizes[0] codes, [1] norms, [2] qjl_signs, [3] qjl_rnorm (0 when
 * the plane is not used).  A b-bit vector of head_dim coordinates takes
 * head_dim*b/8 code bytes plus a 4-byte norm ("윈도우용 터보퀀트(TurboQuant)
 * 구현을 개선하다", finding 3: 3 bits x 128 = 48 B + 4 B = 52 B); QJL keys add
 * m/8 sign bytes and a 4-byte residual norm ("TurboQuant KV 캐시 압축 for
 * llama.cpp", v1.4.2 item 2), Direct Sign keys head_dim/8 and a 4-byte scale
 * (v1.1.0).  Host only; returns TQ_ERR_INVALID_ARG for a bad config, layer,
 * kind or a negative size. */
tq_status tq_plane_bytes(const tq_config* cfg, int layer, int kind, int batch, int n_kv_heads,
                         int64_t capacity, size_t sizes[4]);

/* Bytes of device workspace that tq_decode_attention needs for these shapes
 * (the largest over the config's layers): the split partials (m, l, o) of
 * the split-K decode and one split counter per (sequence, kv-head).  The
 * log-sum-exp merge of per-split softmax partials is the combine step of the
 * pages' flash-decoding kernels ("TurboQuant KV 캐시 압축 for llama.cpp",
 * v1.5.2 items 1-2: partial sums accumulate in fp32).  Host only; 0 for
 * invalid arguments. */
size_t tq_workspace_bytes(const tq_config* cfg, int batch, int n_q_heads, int n_kv_heads,
                          int max_seq_len);

/* -------------------------------------------------------------- device */

/* Zero a decode workspace (async on stream; the workspace is the one
 * tq_workspace_bytes sizes for the split-K combine described there).  Needed
 * once after allocation; every decode leaves its split counters at zero when
 * it completes, including one whose bounded waits ran out.
 * TQ_ERR_INVALID_ARG for a NULL workspace, TQ_ERR_CUDA if the memset fails. */
tq_status tq_workspace_init(void* workspace, size_t workspace_bytes, void* stream);

/* Quantize src[b, h, j, :] for j < n_tokens into plane row
 * (b, h, dst_pos[b] + j) of `dst`, for layer/kind of cfg.
 *   src          device, dtype src_dtype (TQ_BF16 | TQ_F32), element strides
 *                src_strides = {batch, head, token}; the head_dim axis is
 *                contiguous; base and token stride 16-byte aligned.
 *   dst_pos      device int32 [batch] first plane row per sequence, or NULL
 *                (all zero).  Rows dst_pos[b] + n_tokens must be <= capacity;
 *                rows past capacity are not written and set
 *                TQ_ERR_DEVICE_BOUNDS.
 *   QJL keys also get their sign sketch and residual norm. */
tq_status tq_quantize_kv(const tq_config* cfg, const void* tables, int layer, int kind,
                         const void* src, int src_dtype, const int64_t src_strides[3],
                         int batch, int n_kv_heads, int n_tokens, const int32_t* dst_pos,
                         tq_planes dst, void* stream);

/* Streaming append of n_new tokens per sequence with the residual window
 * ("[GitHub 탐방] ... 단일 GPU 재현 기록", "실험 설계": recent tokens stay full
 * precision).  For sequence b with T0 = seq_lens_before[b] tokens (device
 * int32 [batch]) and T1 = T0 + n_new:
 *   - every token t in [max(T0-W,0), max(T1-W,0)) is quantized into plane row
 *     t, read from window slot t mod W if t < T0, else from the new input;
 *   - every new token t >= max(T1-W, T0) is written (bf16) into window slot
 *     t mod W of k_win / v_win ([batch][n_kv_heads][W][head_dim], device).
 * With W = 0 this is tq_quantize_kv at dst_pos = seq_lens_before.
 * seq_lens_before is not updated (the caller owns the lengths). */
tq_status tq_append_kv(const tq_config* cfg, const void* tables, int layer, const void* k_new,
                       const void* v_new, int src_dtype, const int64_t src_strides[3],
                       int batch, int n_kv_heads, int n_new, const int32_t* seq_lens_before,
                       uint16_t* k_win, uint16_t* v_win, tq_planes k, tq_planes v,
                       void* stream);

/* Reconstruct vectors from their planes (inspection and tests; decode never
 * materialises them).  dst[b, h, j, :] (fp32, device, contiguous
 * [batch][n_kv_heads][n_tokens][d]) = n R^T c[idx] for plane rows
 * j < n_tokens: the centroid lookup, the inverse WHT and the norm
 * ("TurboQuant KV 캐시 압축 for llama.cpp", v1.7.0 decision 4: the decoder
 * undoes the encoder's sign flip + butterfly; "윈도우용 터보퀀트(TurboQuant)
 * 구현을 개선하다", recap).  With include_qjl != 0 and a QJL key plane, plus
 * R^T (sqrt(pi/2)/m) gamma S^T (2 bits - 1) (v1.4.2 item 2); with a Direct
 * Sign key plane, plus R^T a (2 bits - 1).  Arguments are checked as for
 * tq_quantize_kv; n_tokens <= capacity. */
tq_status tq_dequantize(const tq_config* cfg, const void* tables, int layer, int kind,
                        tq_planes src, int batch, int n_kv_heads, int n_tokens,
                        int include_qjl, float* dst, void* stream);

/* One decode step of attention for layer `layer`:
 *   q        device [batch][n_q_heads][head_dim], dtype q_dtype.
 *   k, v     the layer's planes (quantized tokens t < T - W at row t).
 *   k_win, v_win  device bf16 [batch][n_kv_heads][W][head_dim] ring, token t
 *            in slot t mod W (NULL when W = 0).
 *   seq_lens device int32 [batch]: T per sequence, window included;
 *            each T <= max_seq_len (host bound used to size the grid).  A T
 *            outside [0, max_seq_len] is decoded as an empty sequence (zeros)
 *            and sets TQ_ERR_DEVICE_BOUNDS (tq_get_device_error).
 *   out      device fp32 [batch][n_q_heads][head_dim].
 *   Query head h reads kv-head h / (n_q_heads / n_kv_heads).  Scores are
 *   softmax_scale * q.k; a sequence with T = 0 writes zeros.
 *   workspace  device, >= tq_workspace_bytes(), zeroed once by
 *            tq_workspace_init.  Calls that share a workspace must not
 *            overlap on the device. */
tq_status tq_decode_attention(const tq_config* cfg, const void* tables, int layer, const void* q,
                              int q_dtype, float softmax_scale, int batch, int n_q_heads,
                              int n_kv_heads, tq_planes k, tq_planes v, const uint16_t* k_win,
                              const uint16_t* v_win, const int32_t* seq_lens, int max_seq_len,
                              float* out, void* workspace, size_t workspace_bytes,
                              void* stream);

/* Decode attention for n_queries query tokens per sequence at once
 * (speculative-draft verification, chunked decode; the multi-column path of
 * "TurboQuant KV 캐시 압축 for llama.cpp", v1.1.0 bug fixes: ncols = 2 for
 * prompt evaluation).  Query token j
 * of sequence b sits at position T_b - n_queries + j and attends causally to
 * tokens t <= T_b - n_queries + j of the same cache.
 *   q     device [batch][n_q_heads][n_queries][head_dim], dtype q_dtype.
 *   out   device fp32 [batch][n_q_heads][n_queries][head_dim].
 *   workspace  >= tq_workspace_bytes(cfg, batch, n_q_heads * n_queries,
 *         n_kv_heads, max_seq_len).
 * The tokens some query may not see must be window tokens: residual_window
 * >= n_queries - 1, else TQ_ERR_UNSUPPORTED; (n_q_heads / n_kv_heads) *
 * n_queries in {1, 2, 4, 8}, else TQ_ERR_UNSUPPORTED.  Other arguments and
 * errors as tq_decode_attention (which is this call with n_queries = 1). */
tq_status tq_decode_attention_multi(const tq_config* cfg, const void* tables, int layer,
                                    const void* q, int q_dtype, float softmax_scale, int batch,
                                    int n_q_heads, int n_kv_heads, int n_queries, tq_planes k,
                                    tq_planes v, const uint16_t* k_win, const uint16_t* v_win,
                                    const int32_t* seq_lens, int max_seq_len, float* out,
                                    void* workspace, size_t workspace_bytes, void* stream);

/* One decode step of a serving loop: tq_append_kv of one new token per
 * (sequence, kv-head) (k_new, v_new: [batch][n_kv_heads][1][head_dim] with
 * src_strides, as there), then tq_decode_attention over the seq_lens_before[b]
 * + 1 tokens of every sequence, with the same arguments and results as those
 * two calls ("[GitHub 탐방] TurboQuant 3-bit KV 캐시 압축 — 단일 GPU 재현 기록",
 * "실험 설계": the newest tokens stay in the bf16 window).  max_seq_len bounds
 * seq_lens_before[b] + 1.  One launch when the plan with the step's work
 * fits one wave of the GPU and gives the warps of the quantized splits no more
 * 32-token chunks than a plain decode's plan (see tq_decode_step_launches):
 * the quantized splits stop before the token that leaves the window (with
 * W = 0 the new token itself), and each pair's first window split (with
 * W = 0 a split of its own) quantizes that token into the planes with the same warp-per-vector
 * quantizer as tq_append_kv (so the same codes, norms and residual terms),
 * attends to its dequantized key and value, and with W > 0 writes the new
 * token into the ring slot that token leaves; the window splits read the new
 * token from k_new / v_new.  The output equals that of the two calls within
 * the decode's rounding (that token enters the attention through fp32
 * dequantized operands rather than fp16 MMA operands).  Otherwise (the splits
 * that append would run in a later wave, or with W = 0 their extra split per
 * pair would give the quantized splits' warps more chunks) two launches: the
 * append kernel and a decode that waits for it.  k_new / v_new are bf16, or
 * fp32 when W = 0 (the ring is bf16).  The planes, ring and workspace must not
 * be used by other work on the device meanwhile. */
tq_status tq_decode_step(const tq_config* cfg, const void* tables, int layer, const void* q,
                         int q_dtype, float softmax_scale, int batch, int n_q_heads,
                         int n_kv_heads, const void* k_new, const void* v_new, int src_dtype,
                         const int64_t src_strides[3], const int32_t* seq_lens_before,
                         int max_seq_len, uint16_t* k_win, uint16_t* v_win, tq_planes k,
                         tq_planes v, float* out, void* workspace, size_t workspace_bytes,
                         void* stream);

/* Kernel launches tq_decode_step makes for these sizes: 1 (the decode kernel
 * appends the token itself) or 2 (the append kernel, then the decode), or 0
 * for invalid arguments.  The pages have no counterpart; this is an
 * introspection helper for schedulers and benchmarks. */
int tq_decode_step_launches(const tq_config* cfg, int layer, int batch, int n_q_heads,
                            int n_kv_heads, int max_seq_len);

/* Synchronize `stream`, then read and clear the device error words that the
 * kernels set instead of faulting: a bounded wait that ran out
 * (TQ_ERR_DEVICE_TIMEOUT) or an index check (TQ_ERR_DEVICE_BOUNDS: a plane
 * row past capacity, a sequence length outside [0, max_seq_len]).  The pages
 * have no counterpart; the __syncthreads race on the query-WHT shared memory
 * that they fixed ("TurboQuant KV 캐시 압축 for llama.cpp", v1.1.0 bug fixes)
 * is the kind of fault such checks make visible without taking the GPU down.
 * Returns TQ_OK, TQ_ERR_DEVICE_TIMEOUT, TQ_ERR_DEVICE_BOUNDS or TQ_ERR_CUDA. */
tq_status tq_get_device_error(void* stream);

/* Test hook: cap on the polling iterations of every bounded device wait
 * (0 restores the default).  A tiny cap makes the timeout path run without
 * hanging anything. */
void tq_set_wait_limit(uint32_t iterations);

/* Test hook for failure detection without a GPU fault.  mode 1: every
 * staging barrier of the decode kernel is told to expect 16 bytes more than
 * its copies deliver, so each bounded wait can only end by running out; the
 * kernel then flags TQ_ERR_DEVICE_TIMEOUT, gives its copies in flight one more
 * bounded wait, and finishes the call with an undefined output (the split
 * counters still return to zero, so the workspace stays usable).
 * mode 0 (default) turns it off. */
void tq_set_fault_injection(int mode);

/* Allocation-free variant of tq_decode_attention.  The pages have no
 * counterpart: this is an integration convenience for callers that cannot
 * give the library a workspace -- for example a plugin inside a serving engine
 * that owns all device memory and hands over only tensor pointers, or a
 * latency-bound decode loop that must not call the CUDA allocator (cudaMalloc
 * may synchronize the whole device).
 *
 * Same arguments and results as tq_decode_attention, minus the workspace: the
 * split partials and counters live in a fixed device array of 8 MiB
 * (8388608 bytes) that the library reserves on every GPU that loads it and
 * holds until the process exits.
 * Nothing is allocated by the call.
 *   - A problem whose tq_workspace_bytes() exceeds that size is rejected with
 *     TQ_ERR_BUFFER_TOO_SMALL before anything is launched.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     outside any stream capture.
 *   - Each call clears the array's split counters for its shapes (an async
 *     memset of a few bytes on `stream`) before the decode launch; the
 *     split partials are always written before they are read.
 *   - The array's device address is cached per device for the life of the
 *     process: after cudaDeviceReset (or a new primary context) on that
 *     device the entry point may not be used again.
 *   - Every call on a device shares the one array: calls whose work can
 *     overlap on the GPU (different streams, no ordering between them) race
 *     and give wrong results.  Order them on one stream or by events. */
tq_status tq_decode_attention_noalloc(const tq_config* cfg, const void* tables, int layer,
                                      const void* q, int q_dtype, float softmax_scale, int batch,
                                      int n_q_heads, int n_kv_heads, tq_planes k, tq_planes v,
                                      const uint16_t* k_win, const uint16_t* v_win,
                                      const int32_t* seq_lens, int max_seq_len, float* out,
                                      void* stream);

#ifdef __cplusplus
}
#endif

#endif /* TQ_H_ */
