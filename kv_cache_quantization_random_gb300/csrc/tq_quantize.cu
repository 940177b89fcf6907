// Quantize, streaming append and dequantize kernels (sm_103a).
//
// Quantize ("윈도우용 터보퀀트(TurboQuant) 구현을 개선하다", recap: rotate, then
// quantize; "TurboQuant KV 캐시 압축 for llama.cpp", v1.7.0 decision 4: sign
// flip + butterfly WHT inside the encoder): one thread owns one vector.  A CTA
// stages 128 rows with bulk (TMA) copies into padded shared memory, then each
// thread keeps its 128 coordinates in registers: sign flip (folded into the
// bf16 -> fp32 widening), sum of squares, the 7-stage Walsh-Hadamard butterfly,
// scaling by 1/(||x|| sqrt d), branch-free binary search over the fp32
// boundaries, and packing into a dense LSB-first stream ("... 개선하다",
// finding 3: 3 bits x 128 = 48 B + 4 B norm).  Keys in MSE+QJL mode also form
// the rotated-domain residual r = n (y - c[idx]), its norm and the sign sketch
// of S r ("TurboQuant KV 캐시 압축 for llama.cpp", "QJL 보정 효과").
#include <cuda_runtime.h>
#include <stdint.h>

#include "tq_device.cuh"

namespace tq {

__device__ unsigned g_quant_err;

constexpr int kQRows = 128;           // vectors per tile = threads per CTA
constexpr int kD = 128;

template <bool F32>
struct RowCfg {
  static constexpr int kRowBytes = F32 ? kD * 4 : kD * 2;
  static constexpr int kPitch = kRowBytes + 16;   // odd multiple of 16 B: conflict-free rows
};

__host__ __device__ constexpr size_t quant_smem_bytes(bool f32, bool qjl) {
  return (size_t)kQRows * (f32 ? RowCfg<true>::kPitch : RowCfg<false>::kPitch)  // rows
         + 256 * 4 + 256 * 4 + kD * 4                                              // tables
         + 16                                                                      // mbarrier
         + (qjl ? (size_t)kQjlM * kD * 4 : 0);                                     // S (fp32)
}

// Resolve row r of the tile: its source address and destination plane row.
__device__ __forceinline__ bool resolve_row(const QuantArgs& a, long long v, const void** src,
                                            long long* dst_row) {
  const int n = a.n;
  const int j = (int)(v % n);
  const long long bh = v / n;
  const int h = (int)(bh % a.H);
  const int b = (int)(bh / a.H);
  const int esz = a.src_f32 ? 4 : 2;
  long long pos;
  if (!a.append) {
    pos = (a.dst_pos ? (long long)a.dst_pos[b] : 0) + j;
    *src = (const uint8_t*)a.src + (b * a.sb + h * a.sh + (long long)j * a.st) * esz;
  } else {
    const long long T0 = a.seq_before[b];
    const long long q0 = T0 - a.W > 0 ? T0 - a.W : 0;
    const long long T1 = T0 + n;
    const long long q1 = T1 - a.W > 0 ? T1 - a.W : 0;
    pos = q0 + j;
    if (pos >= q1) return false;                       // stays in (or enters) the window
    if (pos < T0) {                                     // leaves the window ring
      const long long slot = pos % a.W;
      *src = (const uint8_t*)a.win + (((long long)b * a.H + h) * a.W + slot) * kD * 2;
    } else {
      *src = (const uint8_t*)a.src + (b * a.sb + h * a.sh + (pos - T0) * a.st) * esz;
    }
  }
  if (pos < 0 || pos >= a.cap) {
    atomicOr(a.err, kErrBounds);
    return false;
  }
  *dst_row = ((long long)b * a.H + h) * a.cap + pos;
  return true;
}

template <int BITS, bool QJL, bool F32>
__global__ void __launch_bounds__(kQRows) quantize_kernel(const QuantArgs a) {
  constexpr int L = 1 << BITS;
  constexpr int NW = 4 * BITS;         // 32-bit code words per vector (128 * BITS / 32)
  constexpr int kRowBytes = RowCfg<F32>::kRowBytes;
  constexpr int kPitch = RowCfg<F32>::kPitch;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* rows = smem;
  float* bnd = (float*)(smem + kQRows * kPitch);
  float* cen = bnd + 256;
  uint32_t* smask = (uint32_t*)(cen + 256);
  uint64_t* bar = (uint64_t*)(smask + kD);
  float* Sf = (float*)(bar + 2);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int i = tid; i < 256; i += kQRows) {
    bnd[i] = a.boundaries[i];
    cen[i] = a.centroids[i];
  }
  smask[tid] = a.rot_signs[tid] < 0.f ? 0x80000000u : 0u;
  if constexpr (QJL) {
    for (int e = tid; e < kQjlM * kD; e += kQRows) Sf[e] = __uint_as_float((uint32_t)a.S[e] << 16);
  }
  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbarrier_init();
  }
  __syncthreads();

  const long long total = (long long)a.B * a.H * a.n;
  const long long ntiles = (total + kQRows - 1) / kQRows;
  const uint32_t limit = a.wait_limit ? a.wait_limit : kDefaultWaitLimit;
  uint32_t parity = 0;
  for (long long tile = blockIdx.x; tile < ntiles; tile += gridDim.x, parity ^= 1u) {
    const long long v0 = tile * kQRows;
    // ---- stage the tile's rows (warp 0 issues one bulk copy per row)
    if (warp == 0) {
      const void* srcs[kQRows / 32];
      long long dummy;
      uint32_t mine = 0, count = 0;
#pragma unroll
      for (int k = 0; k < kQRows / 32; ++k) {
        const long long v = v0 + lane + 32 * k;
        bool ok = v < total && resolve_row(a, v, &srcs[k], &dummy);
        mine |= (ok ? 1u : 0u) << k;
      }
      count = __reduce_add_sync(0xffffffffu, (uint32_t)__popc(mine));
      // a.extra_tx is a test hook: bytes that never arrive, so the wait below
      // can only end by running out of polls
      if (lane == 0) mbar_arrive_expect_tx(bar, count * kRowBytes + a.extra_tx);
      __syncwarp();
#pragma unroll
      for (int k = 0; k < kQRows / 32; ++k)
        if (mine & (1u << k)) bulk_g2s(rows + (lane + 32 * k) * kPitch, srcs[k], kRowBytes, bar);
    }
    const bool staged = __syncthreads_and(mbar_wait(bar, parity, limit, a.err));
    if (!staged) {
      // the staging wait ran out (error word already set): give copies still in
      // flight one more bounded wait, then leave without touching the planes
      for (uint32_t i = 0; i < limit && !mbar_try_wait(bar, parity); ++i) {
      }
      return;
    }
    const long long v = v0 + tid;
    const void* srcp;
    long long drow;
    if (v < total && resolve_row(a, v, &srcp, &drow)) {
      // ---- widen, flip signs, accumulate ||x||^2
      float x[kD];
      const uint8_t* row = rows + tid * kPitch;
      if constexpr (F32) {
#pragma unroll
        for (int c = 0; c < kD / 4; ++c) {
          uint4 w = lds128(row + 16 * c);
          uint4 m = lds128(smask + 4 * c);
          x[4 * c + 0] = __uint_as_float(w.x ^ m.x);
          x[4 * c + 1] = __uint_as_float(w.y ^ m.y);
          x[4 * c + 2] = __uint_as_float(w.z ^ m.z);
          x[4 * c + 3] = __uint_as_float(w.w ^ m.w);
        }
      } else {
#pragma unroll
        for (int c = 0; c < kD / 8; ++c) {
          uint4 w = lds128(row + 16 * c);
          uint4 m0 = lds128(smask + 8 * c);
          uint4 m1 = lds128(smask + 8 * c + 4);
          x[8 * c + 0] = __uint_as_float((w.x << 16) ^ m0.x);
          x[8 * c + 1] = __uint_as_float((w.x & 0xFFFF0000u) ^ m0.y);
          x[8 * c + 2] = __uint_as_float((w.y << 16) ^ m0.z);
          x[8 * c + 3] = __uint_as_float((w.y & 0xFFFF0000u) ^ m0.w);
          x[8 * c + 4] = __uint_as_float((w.z << 16) ^ m1.x);
          x[8 * c + 5] = __uint_as_float((w.z & 0xFFFF0000u) ^ m1.y);
          x[8 * c + 6] = __uint_as_float((w.w << 16) ^ m1.z);
          x[8 * c + 7] = __uint_as_float((w.w & 0xFFFF0000u) ^ m1.w);
        }
      }
      float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
      for (int i = 0; i < kD; i += 4) {
        s0 = fmaf(x[i], x[i], s0);
        s1 = fmaf(x[i + 1], x[i + 1], s1);
        s2 = fmaf(x[i + 2], x[i + 2], s2);
        s3 = fmaf(x[i + 3], x[i + 3], s3);
      }
      const float nrm = sqrtf((s0 + s1) + (s2 + s3));
      // ---- rotate: y = H (s * x) / (||x|| sqrt d)
      fwht_regs<kD>(x);
      const float inv = nrm > 0.f ? 1.0f / (nrm * 11.313708498984761f) : 0.f;
      // ---- code search and packing
      uint32_t words[NW];
#pragma unroll
      for (int k = 0; k < NW; ++k) words[k] = 0u;
#pragma unroll
      for (int i = 0; i < kD; ++i) {
        const float y = x[i] * inv;
        uint32_t idx = 0;
#pragma unroll
        for (int step = L / 2; step >= 1; step >>= 1)
          if (bnd[idx + step - 1] < y) idx += step;
        const int p = i * BITS;
        words[p >> 5] |= idx << (p & 31);
        if ((p & 31) + BITS > 32) words[(p >> 5) + 1] |= idx >> (32 - (p & 31));
        if constexpr (QJL) x[i] = nrm * (y - cen[idx]);   // rotated-domain residual
      }
      uint4* dc = (uint4*)(a.codes + drow * (16 * BITS));
#pragma unroll
      for (int k = 0; k < BITS; ++k)
        dc[k] = make_uint4(words[4 * k], words[4 * k + 1], words[4 * k + 2], words[4 * k + 3]);
      a.norms[drow] = nrm;
      if constexpr (QJL) {
        float g0 = 0.f, g1 = 0.f;
#pragma unroll
        for (int i = 0; i < kD; i += 2) {
          g0 = fmaf(x[i], x[i], g0);
          g1 = fmaf(x[i + 1], x[i + 1], g1);
        }
        const float gamma = sqrtf(g0 + g1);
        uint32_t sb[kQjlM / 32];
#pragma unroll
        for (int k = 0; k < kQjlM / 32; ++k) sb[k] = 0u;
        for (int j = 0; j < kQjlM; ++j) {
          const float* Sj = Sf + j * kD;
          float z0 = 0.f, z1 = 0.f, z2 = 0.f, z3 = 0.f;
#pragma unroll
          for (int k = 0; k < kD; k += 4) {
            float4 s = *(const float4*)(Sj + k);
            z0 = fmaf(s.x, x[k], z0);
            z1 = fmaf(s.y, x[k + 1], z1);
            z2 = fmaf(s.z, x[k + 2], z2);
            z3 = fmaf(s.w, x[k + 3], z3);
          }
          const float z = (z0 + z1) + (z2 + z3);
          sb[j >> 5] |= (z >= 0.f ? 1u : 0u) << (j & 31);
        }
        *(uint4*)(a.qjl_signs + drow * (kQjlM / 8)) = make_uint4(sb[0], sb[1], sb[2], sb[3]);
        a.qjl_rnorm[drow] = gamma;
      }
    }
    __syncthreads();   // every thread is done with the tile's rows before they are refilled
  }
}

// Window ring update of tq_append_kv: new token t >= T1 - W goes to slot t mod W.
__global__ void window_scatter_kernel(const WindowScatterArgs a) {
  const long long rows = (long long)a.B * a.H * a.n;
  const long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long r = gid >> 4;          // 16 threads per row of 128 bf16
  const int part = (int)(gid & 15);
  if (r >= rows) return;
  const int j = (int)(r % a.n);
  const long long bh = r / a.n;
  const int h = (int)(bh % a.H);
  const int b = (int)(bh / a.H);
  const long long T0 = a.seq_before[b];
  const long long t = T0 + j;
  const long long T1 = T0 + a.n;
  if (t < T1 - a.W) return;              // quantized directly, never enters the ring
  const uint4* s = (const uint4*)((const uint8_t*)a.src + (b * a.sb + h * a.sh + (long long)j * a.st) * 2);
  uint4* d = (uint4*)(a.win + (((long long)b * a.H + h) * a.W + t % a.W) * kD);
  d[part] = s[part];
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
  const uint4* src = (const uint4*)(a.codes + row * (16 * BITS));
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
static int sm_count() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 152;
  }
  return n;
}

template <int BITS, bool QJL, bool F32>
static int launch_q(const QuantArgs& a, cudaStream_t s) {
  auto k = quantize_kernel<BITS, QJL, F32>;
  const size_t smem = quant_smem_bytes(F32, QJL);
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
  if (a.qjl) return a.src_f32 ? launch_q<BITS, true, true>(a, s) : launch_q<BITS, true, false>(a, s);
  return a.src_f32 ? launch_q<BITS, false, true>(a, s) : launch_q<BITS, false, false>(a, s);
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

int launch_window_scatter(const WindowScatterArgs& a, void* stream) {
  const long long threads = (long long)a.B * a.H * a.n * 16;
  const int block = 256;
  window_scatter_kernel<<<(unsigned)((threads + block - 1) / block), block, 0, (cudaStream_t)stream>>>(a);
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
