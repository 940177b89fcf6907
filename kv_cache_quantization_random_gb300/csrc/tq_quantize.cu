// Quantize, streaming append and dequantize kernels (sm_103a).
//
// Quantize ("윈도우용 터보퀀트(TurboQuant) 구현을 개선하다", recap: rotate, then
// quantize; "TurboQuant KV 캐시 압축 for llama.cpp", v1.7.0 decision 4: sign
// flip + butterfly WHT inside the encoder): one thread owns one vector.  Each
// warp streams its own tiles of 32 rows through two padded shared-memory
// buffers with cp.async, and each thread keeps its 128 coordinates in
// registers (see quantize_row in tq_quant_common.cuh): sign flip folded into
// the bf16 -> fp32 widening, sum of squares, the Walsh-Hadamard butterfly on
// packed fp32 pairs, code search on a uniform grid with one exact boundary
// compare, and packing into a dense LSB-first stream ("... 개선하다", finding
// 3: 3 bits x 128 = 48 B + 4 B norm).  Keys in MSE+QJL mode take the tensor-
// core kernel in tq_qjl.cu instead.
#include <cuda_runtime.h>
#include <stdint.h>

#include "tq_quant_common.cuh"

namespace tq {

__device__ unsigned g_quant_err;

// dynamic shared memory of quantize_kernel: per warp two buffers of 32 rows,
// the search grid and the boundaries
__host__ __device__ constexpr size_t quant_smem_bytes(bool f32, int cells, bool sgn) {
  return 2 * quant_rows_bytes(f32) + (size_t)cells * 8 + 256 * 4 + (sgn ? 256 * 4 : 0);
}

// SGN: keys in Direct Sign mode also get the sign of every rotated residual
// coordinate and the scale mean |r_i| ("TurboQuant KV 캐시 압축 for
// llama.cpp", v1.1.0 "Direct Sign").  RING: an append with a window (bf16
// rows), which also writes the new tokens that stay into the ring (see
// ring_copy_of); a variant of its own, so that the bulk path carries none of it.
// (the tiles that CTA `cta` of the `ncta` working on `a` takes)
template <int BITS, bool F32, bool CLAMP, bool SGN, bool RING>
__device__ __forceinline__ void quantize_tiles(const QuantArgs& a, uint32_t cta, uint32_t ncta) {
  constexpr int kPitch = RowCfg<F32>::kPitch;
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // this warp's two buffers of 32 rows
  uint8_t* wrows = smem + (size_t)warp * 2 * 32 * kPitch;
  float2* grid = (float2*)(smem + 2 * quant_rows_bytes(F32));
  float* bnd = (float*)(grid + a.grid_cells);
  float* cen = bnd + 256;                               // SGN only
  for (int i = tid; i < 256; i += kQRows) {
    bnd[i] = a.boundaries[i];
    if constexpr (SGN) cen[i] = a.centroids[i];
  }
  __syncthreads();
  build_grid<BITS>(a, bnd, grid, tid, kQRows);
  __syncthreads();
  const uint32_t grid_base = smem_u32(grid);
  const uint32_t kmax = (uint32_t)a.grid_cells - 1u;

  // every warp streams its own tiles of 32 vectors: no CTA barrier below
  const uint32_t total = (uint32_t)a.B * (uint32_t)a.H * (uint32_t)a.n;
  const uint32_t ntiles = (total + 31) / 32;
  const uint32_t stride = ncta * (kQRows / 32);
  uint32_t tile = cta * (kQRows / 32) + warp;
  const void* src = nullptr;
  long long drow = 0;
  bool valid = false;
  if (tile < ntiles) {
    const uint32_t v = tile * 32 + lane;
    valid = v < total && resolve_row(a, v, &src, &drow);
    stage_rows<F32>(src, valid, wrows, lane);
  }
  cp_async_commit();
  int buf = 0;
  for (; tile < ntiles; tile += stride) {
    const uint32_t next = tile + stride;
    const void* nsrc = nullptr;
    long long ndrow = 0;
    bool nvalid = false;
    if (next < ntiles) {                 // the other buffer was released by the last __syncwarp
      const uint32_t v = next * 32 + lane;
      nvalid = v < total && resolve_row(a, v, &nsrc, &ndrow);
      stage_rows<F32>(nsrc, nvalid, wrows + (buf ^ 1) * 32 * kPitch, lane);
    }
    cp_async_commit();
    cp_async_wait<1>();                  // this lane's copies of `tile` have landed
    __syncwarp();                        // ... and every other lane's
    // the ring slots whose tokens this tile has read take the new tokens
    if constexpr (RING) ring_copies(a, tile * 32 + lane, tile * 32 + lane < total, lane);
    const uint8_t* rows = wrows + buf * 32 * kPitch;
    if (valid) {
      float2 p[64];
      const float nrm = quantize_row<BITS, F32, CLAMP, SGN>(
          a, rows + lane * kPitch, grid_base, kmax, cen, a.codes + drow * (16 * BITS), p);
      a.norms[drow] = nrm;
      if constexpr (SGN) direct_sign(p, a.qjl_signs + drow * (kD / 8), a.qjl_rnorm + drow);
    }
    __syncwarp();      // every lane is done with this buffer before it is refilled
    buf ^= 1;
    src = nsrc;
    drow = ndrow;
    valid = nvalid;
  }
  cp_async_wait<0>();
}

template <int BITS, bool F32, bool CLAMP, bool SGN, bool RING>
__global__ void __launch_bounds__(kQRows, 3) quantize_kernel(const QuantArgs a) {
  quantize_tiles<BITS, F32, CLAMP, SGN, RING>(a, blockIdx.x, gridDim.x);
}

// An append of both kinds in one launch (bf16 rows, keys and values of the
// same bit width, so that one search grid size serves both): CTAs below nk
// take the keys, the others the values.  For a streaming chunk of a few
// thousand tokens per head each kind alone fills about half an SM wave.
template <int BITS, bool SGN, bool RING>
__global__ void __launch_bounds__(kQRows, 3)
    quantize_kv_kernel(const QuantArgs ak, const QuantArgs av, uint32_t nk) {
  if (blockIdx.x < nk)
    quantize_tiles<BITS, false, (BITS > 4), SGN, RING>(ak, blockIdx.x, nk);
  else
    quantize_tiles<BITS, false, (BITS > 4), false, RING>(av, blockIdx.x - nk, gridDim.x - nk);
}

// ---- tq_append_kv with a few new tokens: one CTA per (sequence, kv-head).
// Warp 0 quantizes the keys and warp 1 the values that leave the window (or
// go straight to the planes), see warp_quantize_row; lane l owns coordinates 4l..4l+3, so the
// Walsh-Hadamard butterfly takes two in-register stages and five shuffle
// stages.  QJL keys take three more warps (2-4): each of the four key warps
// quantizes the key (only warp 0 stores codes and norm) and computes a quarter
// of its sketch, so that the m = 128 projections run four at a time instead of
// one after another.  After a CTA barrier (every ring slot that is about to
// be overwritten has been read) all threads write the new tokens into the ring.
constexpr int kAppendQjlWarps = 5;

// Rows 32 s + lane of S r, for slice s of the QJL sketch of the key residual
// r (lane l: coordinates 4l..4l+3; "TurboQuant KV 캐시 압축 for llama.cpp",
// "QJL 보정 효과"): sign word s of the 16 sign bytes, and for s = 0 gamma =
// ||r||.  The products are summed in the order of warp_qjl_sketch, so both
// give the same bits.  rbuf: 128 floats of this warp's shared scratch.
__device__ __forceinline__ void append_qjl_slice(const float (&r)[4], const uint16_t* S, float* rbuf,
                                                 uint8_t* signs_dst, float* gamma_dst, int lane,
                                                 int s) {
  if (s == 0) {
    float g = r[0] * r[0];
    g = fmaf(r[1], r[1], g);
    g = fmaf(r[2], r[2], g);
    g = fmaf(r[3], r[3], g);
    const float gamma = sqrtf(warp_sum(g));
    if (lane == 0) *gamma_dst = gamma;
  }
  *(float4*)(rbuf + 4 * lane) = make_float4(r[0], r[1], r[2], r[3]);
  __syncwarp();
  const uint4* Sj = (const uint4*)(S + (size_t)(32 * s + lane) * kD);
  float z0 = 0.f, z1 = 0.f;
#pragma unroll 4
  for (int e = 0; e < kD / 8; ++e) {
    const uint4 s8 = __ldg(Sj + e);
    const float4 ra = *(const float4*)(rbuf + 8 * e);
    const float4 rb = *(const float4*)(rbuf + 8 * e + 4);
    z0 = fmaf(bf16lo(s8.x), ra.x, z0);
    z1 = fmaf(bf16hi(s8.x), ra.y, z1);
    z0 = fmaf(bf16lo(s8.y), ra.z, z0);
    z1 = fmaf(bf16hi(s8.y), ra.w, z1);
    z0 = fmaf(bf16lo(s8.z), rb.x, z0);
    z1 = fmaf(bf16hi(s8.z), rb.y, z1);
    z0 = fmaf(bf16lo(s8.w), rb.z, z0);
    z1 = fmaf(bf16hi(s8.w), rb.w, z1);
  }
  const uint32_t w = __ballot_sync(0xffffffffu, z0 + z1 >= 0.f);
  if (lane == 0) ((uint32_t*)signs_dst)[s] = w;
  __syncwarp();      // rbuf is read by every lane before it is written again
}

// One row of kind `kind` by one warp.  slice: which quarter of a QJL key's
// sketch this warp computes; the warp of slice 0 stores the codes and norm,
// the others quantize into their scratch (16 * 8 bytes of codes, one norm).
__device__ __forceinline__ void append_quantize_row(const AppendArgs& a, int kind, int slice,
                                                    const void* src, int f32, long long drow,
                                                    const float* bnd, const float* cen, float4 sg,
                                                    uint32_t* words, float* rbuf, uint8_t* scratch,
                                                    int lane) {
  constexpr int kDim = 128;
  float r[4], yq[4];
  const bool own = slice == 0;
  warp_quantize_row(src, f32, sg, a.bits[kind], bnd, cen,
                    own ? a.codes[kind] + drow * (16 * a.bits[kind]) : scratch,
                    own ? a.norms[kind] + drow : (float*)(scratch + 128), words, lane, r, yq);
  if (kind == 0 && a.dsign)
    warp_direct_sign(r, a.qjl_signs + drow * (kDim / 8), a.qjl_rnorm + drow, lane);
  if (kind == 0 && a.qjl)
    append_qjl_slice(r, a.S, rbuf, a.qjl_signs + drow * (kQjlM / 8), a.qjl_rnorm + drow, lane,
                     slice);
}

__global__ void __launch_bounds__(32 * kAppendQjlWarps) append_kernel(const AppendArgs a) {
  __shared__ float bnd[2][256];
  __shared__ float cen[2][256];
  __shared__ uint32_t words[kAppendQjlWarps][32];
  __shared__ __align__(16) float rbuf[4][kD];
  __shared__ __align__(16) uint8_t scratch[kAppendQjlWarps][16 * 8 + 16];
  // a decode launched after this kernel may start its prologue now (it reads
  // nothing this kernel writes before its griddepcontrol.wait)
  asm volatile("griddepcontrol.launch_dependents;");
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // warp 1 takes the values; warps 0, 2, 3, 4 the keys (slices 0-3 of a QJL sketch)
  const int kind = warp == 1 ? 1 : 0;
  const int slice = warp < 2 ? 0 : warp - 1;
  const int h = blockIdx.x % a.H, b = blockIdx.x / a.H;
  if (warp < 2) {
    for (int i = lane; i < 256; i += 32) {
      bnd[kind][i] = a.boundaries[kind][i];
      cen[kind][i] = a.centroids[kind][i];
    }
  }
  words[warp][lane] = 0u;
  const float4 sg = ((const float4*)a.rot_signs[kind])[lane];
  __syncthreads();                                    // the key warps share warp 0's tables
  const long long T0 = a.seq_before[b];
  const long long T1 = T0 + a.n;
  const long long q0 = T0 - a.W > 0 ? T0 - a.W : 0;
  const long long q1 = T1 - a.W > 0 ? T1 - a.W : 0;
  const int esz = a.src_f32 ? 4 : 2;
  for (long long pos = q0; pos < q1; ++pos) {
    const void* src;
    int f32 = a.src_f32;
    if (pos < T0) {                                   // leaves the window ring
      src = a.win[kind] + (((long long)b * a.H + h) * a.W + pos % a.W) * kD;
      f32 = 0;
    } else {
      src = (const uint8_t*)a.src[kind] + (b * a.sb + h * a.sh + (pos - T0) * a.st) * esz;
    }
    if (pos < 0 || pos >= a.cap[kind]) {
      if (lane == 0) atomicOr(a.err, kErrBounds);
      continue;
    }
    // bounds-checked build: the row lies inside the ring or the new input
    if (kBoundsChecks) {
      const bool ring = pos < T0;
      const size_t bytes = ring ? (size_t)a.B * a.H * a.W * kD * 2
                                : (size_t)((long long)(a.B - 1) * a.sb + (long long)(a.H - 1) * a.sh +
                                           (long long)(a.n - 1) * a.st + kD) * esz;
      if (!bchk_range(src, (size_t)kD * (ring ? 2 : esz), ring ? (const void*)a.win[kind] : a.src[kind],
                      bytes, a.err))
        continue;
    }
    const long long drow = ((long long)b * a.H + h) * a.cap[kind] + pos;
    append_quantize_row(a, kind, slice, src, f32, drow, bnd[kind], cen[kind], sg, words[warp],
                        rbuf[slice], scratch[warp], lane);
  }
  if (a.W == 0) return;
  __syncthreads();                                    // ring slots read before they are rewritten
  const long long first = T1 - a.W > T0 ? T1 - a.W : T0;   // first new token kept in the ring
  const int n_ring = (int)(T1 - first);
  for (int e = tid; e < 2 * n_ring * 16; e += (int)blockDim.x) {
    const int part = e & 15, row = e >> 4;
    const int k2 = row / n_ring;
    const long long t = first + row % n_ring;
    const uint4* s4 = (const uint4*)((const uint8_t*)a.src[k2] +
                                     (b * a.sb + h * a.sh + (t - T0) * a.st) * 2);
    uint4* d4 = (uint4*)(a.win[k2] + (((long long)b * a.H + h) * a.W + t % a.W) * kD);
    *bchk(d4 + part, a.win[k2], (size_t)a.B * a.H * a.W * kD * 2, a.err) = s4[part];
  }
}

template <int BITS, bool QJL>
__global__ void __launch_bounds__(128) dequantize_kernel(const DequantArgs a) {
  constexpr int NW = 4 * BITS;
  __shared__ float cen[256];
  __shared__ float sgn[kD];
  extern __shared__ __align__(16) float Sf[];      // QJL only: m x d fp32
  const int tid = threadIdx.x;
  for (int i = tid; i < 256; i += blockDim.x) cen[i] = a.centroids[i];
  for (int i = tid; i < kD; i += blockDim.x) sgn[i] = a.rot_signs[i];
  if constexpr (QJL)
    for (int e = tid; e < kQjlM * kD; e += blockDim.x) Sf[e] = __uint_as_float((uint32_t)a.S[e] << 16);
  __syncthreads();
  const long long v = (long long)blockIdx.x * blockDim.x + tid;
  const long long total = (long long)a.B * a.H * a.n;
  if (v >= total) return;
  const int j = (int)(v % a.n);
  const long long bh = v / a.n;
  const long long row = bh * a.cap + j;
  uint32_t w[NW];
  const uint4* src = bchk((const uint4(*)[BITS])(a.codes + row * (16 * BITS)), a.codes,
                          (size_t)a.B * a.H * a.cap * 16 * BITS, a.err)[0];
#pragma unroll
  for (int k = 0; k < BITS; ++k) {
    uint4 t = src[k];
    w[4 * k] = t.x; w[4 * k + 1] = t.y; w[4 * k + 2] = t.z; w[4 * k + 3] = t.w;
  }
  const float nrm = a.norms[row];
  float y[kD];
#pragma unroll
  for (int i = 0; i < kD; ++i) {
    const int p = i * BITS;
    uint32_t c = w[p >> 5] >> (p & 31);
    if ((p & 31) + BITS > 32) c |= w[(p >> 5) + 1] << (32 - (p & 31));
    y[i] = cen[c & ((1u << BITS) - 1u)] * nrm;
  }
  if (a.dsign) {
    // Direct Sign residual: r_i ~= a (2 bit_i - 1), rotated domain
    const uint4 sb4 = *(const uint4*)(a.qjl_signs + row * (kD / 8));
    const uint32_t sb[4] = {sb4.x, sb4.y, sb4.z, sb4.w};
    const float sc = a.qjl_rnorm[row];
#pragma unroll
    for (int i = 0; i < kD; ++i) y[i] += ((sb[i >> 5] >> (i & 31)) & 1u) ? sc : -sc;
  }
  if constexpr (QJL) {
    const uint4 sb4 = *(const uint4*)(a.qjl_signs + row * (kQjlM / 8));
    const uint32_t sb[4] = {sb4.x, sb4.y, sb4.z, sb4.w};
    const float coef = 1.2533141373155003f / (float)kQjlM * a.qjl_rnorm[row];   // sqrt(pi/2)/m * gamma
    for (int jj = 0; jj < kQjlM; ++jj) {
      const float sgnj = ((sb[jj >> 5] >> (jj & 31)) & 1u) ? coef : -coef;
      const float* Sj = Sf + jj * kD;
#pragma unroll
      for (int i = 0; i < kD; ++i) y[i] = fmaf(sgnj, Sj[i], y[i]);
    }
  }
  fwht_regs<kD>(y);                       // R^T = D_s H / sqrt(d): transform, then signs
  float4* dst = (float4*)(a.dst + v * kD);
  const float r = 0.08838834764831845f;   // 1/sqrt(128)
#pragma unroll
  for (int c = 0; c < kD / 4; ++c)
    dst[c] = make_float4(y[4 * c] * r * sgn[4 * c], y[4 * c + 1] * r * sgn[4 * c + 1],
                         y[4 * c + 2] * r * sgn[4 * c + 2], y[4 * c + 3] * r * sgn[4 * c + 3]);
}

// ---------------------------------------------------------------- launchers
int sm_count() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 152;
  }
  return n;
}

template <int BITS, bool F32, bool SGN, bool RING>
static int launch_q(const QuantArgs& a, cudaStream_t s) {
  auto k = quantize_kernel<BITS, F32, (BITS > 4), SGN, RING>;
  const size_t smem = quant_smem_bytes(F32, a.grid_cells, SGN);
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return 1;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kQRows, smem) != cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  const long long total = (long long)a.B * a.H * a.n;
  const long long ntiles = (total + kQRows - 1) / kQRows;
  long long grid = (long long)sm_count() * per_sm;
  if (grid > ntiles) grid = ntiles;
  k<<<(unsigned)grid, kQRows, smem, s>>>(a);
  return cudaGetLastError() != cudaSuccess;
}

template <int BITS>
static int launch_q_bits(const QuantArgs& a, cudaStream_t s) {
  if (a.qjl) return launch_quantize_qjl(a, s);
  if (a.append && a.W > 0) {               // the window ring holds bf16 rows
    if (a.src_f32) return 1;
    return a.dsign ? launch_q<BITS, false, true, true>(a, s) : launch_q<BITS, false, false, true>(a, s);
  }
  if (a.dsign)
    return a.src_f32 ? launch_q<BITS, true, true, false>(a, s) : launch_q<BITS, false, true, false>(a, s);
  return a.src_f32 ? launch_q<BITS, true, false, false>(a, s) : launch_q<BITS, false, false, false>(a, s);
}

template <int BITS, bool SGN, bool RING>
static int launch_qkv(const QuantArgs& ak, const QuantArgs& av, cudaStream_t s) {
  auto k = quantize_kv_kernel<BITS, SGN, RING>;
  const size_t smem = quant_smem_bytes(false, ak.grid_cells, SGN);
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return 1;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kQRows, smem) != cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  // CTAs in proportion to each kind's tiles of 128 vectors, at least one each
  const long long tk = ((long long)ak.B * ak.H * ak.n + kQRows - 1) / kQRows;
  const long long tv = ((long long)av.B * av.H * av.n + kQRows - 1) / kQRows;
  long long grid = (long long)sm_count() * per_sm;
  if (grid > tk + tv) grid = tk + tv;
  if (grid < 2) grid = 2;
  long long nk = (grid * tk + (tk + tv) / 2) / (tk + tv);
  if (nk < 1) nk = 1;
  if (nk > grid - 1) nk = grid - 1;
  k<<<(unsigned)grid, kQRows, smem, s>>>(ak, av, (uint32_t)nk);
  return cudaGetLastError() != cudaSuccess;
}

template <int BITS>
static int launch_qkv_bits(const QuantArgs& ak, const QuantArgs& av, cudaStream_t s) {
  const bool ring = ak.append && ak.W > 0;
  if (ak.dsign)
    return ring ? launch_qkv<BITS, true, true>(ak, av, s) : launch_qkv<BITS, true, false>(ak, av, s);
  return ring ? launch_qkv<BITS, false, true>(ak, av, s) : launch_qkv<BITS, false, false>(ak, av, s);
}

int launch_quantize_kv(const QuantArgs& ak, const QuantArgs& av, void* stream) {
  cudaStream_t s = (cudaStream_t)stream;
  switch (ak.bits) {
    case 2: return launch_qkv_bits<2>(ak, av, s);
    case 3: return launch_qkv_bits<3>(ak, av, s);
    case 4: return launch_qkv_bits<4>(ak, av, s);
    case 8: return launch_qkv_bits<8>(ak, av, s);
  }
  return 1;
}

int launch_quantize(const QuantArgs& a, void* stream) {
  cudaStream_t s = (cudaStream_t)stream;
  switch (a.bits) {
    case 2: return launch_q_bits<2>(a, s);
    case 3: return launch_q_bits<3>(a, s);
    case 4: return launch_q_bits<4>(a, s);
    case 8: return launch_q_bits<8>(a, s);
  }
  return 1;
}

int launch_append(const AppendArgs& a, void* stream) {
  const long long units = (long long)a.B * a.H;
  if (units <= 0) return 0;
  append_kernel<<<(unsigned)units, a.qjl ? 32 * kAppendQjlWarps : 64, 0, (cudaStream_t)stream>>>(a);
  return cudaGetLastError() != cudaSuccess;
}

template <int BITS, bool QJL>
static int launch_dq(const DequantArgs& a, cudaStream_t s) {
  auto k = dequantize_kernel<BITS, QJL>;
  const size_t smem = QJL ? (size_t)kQjlM * kD * 4 : 0;
  if (smem && cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
                  cudaSuccess)
    return 1;
  const long long total = (long long)a.B * a.H * a.n;
  k<<<(unsigned)((total + 127) / 128), 128, smem, s>>>(a);
  return cudaGetLastError() != cudaSuccess;
}

int launch_dequantize(const DequantArgs& a, void* stream) {
  cudaStream_t s = (cudaStream_t)stream;
  switch (a.bits) {
    case 2: return a.qjl ? launch_dq<2, true>(a, s) : launch_dq<2, false>(a, s);
    case 3: return a.qjl ? launch_dq<3, true>(a, s) : launch_dq<3, false>(a, s);
    case 4: return a.qjl ? launch_dq<4, true>(a, s) : launch_dq<4, false>(a, s);
    case 8: return a.qjl ? launch_dq<8, true>(a, s) : launch_dq<8, false>(a, s);
  }
  return 1;
}

unsigned* quant_error_ptr() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_quant_err) != cudaSuccess) return nullptr;
  return (unsigned*)p;
}

int quant_read_error(unsigned* out) {
  unsigned zero = 0;
  if (cudaMemcpyFromSymbol(out, g_quant_err, sizeof(unsigned)) != cudaSuccess) return 1;
  if (cudaMemcpyToSymbol(g_quant_err, &zero, sizeof(unsigned)) != cudaSuccess) return 1;
  return 0;
}

}  // namespace tq
