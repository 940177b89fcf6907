// Keys in MSE+QJL mode: codes, norm and the 1-bit QJL sketch of the residual,
// with the Gaussian projection on the 5th-generation tensor cores (sm_103a).
//
// "TurboQuant KV 캐시 압축 for llama.cpp", "QJL 보정 효과" (QJL is
// TurboQuant_prod: a 1-bit correction of the residual) and v1.4.2 item 2 (the
// correction is formed from the sign bits and a stored residual scale).  Per
// key: r = ||x|| (y - c[idx]) in the rotated domain, gamma = ||r||, and
// bit_j = [(S r)_j >= 0] for the m = 128 rows of the Gaussian matrix S.
//
// One CTA = 128 threads = one tile of 128 keys; thread t owns key t.  Each
// thread quantizes its key in registers (tq_quant_common.cuh) and writes its
// residual, split into bf16 hi + lo parts (r ~= hi + lo to ~16 bits), as row t
// of two [128 x 128] K-major operand tiles in shared memory.  One thread then
// issues Z = R_hi S^T + R_lo S^T as 16 tcgen05.mma (M = N = 128, K = 16, bf16
// in, fp32 accumulate) into a 128-column TMEM accumulator; S (bf16, exact)
// stays in shared memory for the whole launch.  TMEM lane t holds z for key
// t, so after the commit each warp reads its 32 lanes with tcgen05.ld and
// every thread turns its own 128 projections into 4 words of sign bits.
// bf16 rows are staged in the R lo tile itself (a CTA barrier separates the
// last read of a row from the first residual write), which leaves room for
// two CTAs per SM; fp32 rows keep a buffer of their own and one CTA per SM.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "tq_quant_common.cuh"
#include "tq_umma.cuh"

namespace tq {

// bf16 rows are staged in the R lo tile (read into registers before R lo is
// written), so a CTA fits twice on an SM; fp32 rows need their own buffer.
__host__ __device__ constexpr size_t qjl_smem_bytes(bool f32, int cells) {
  return 1024                                    // alignment slack
         + 3 * (size_t)kOpBytes                  // R hi, R lo, S
         + (f32 ? quant_rows_bytes(true) : 0)    // staged fp32 rows (one tile)
         + (size_t)cells * 8 + 2 * 256 * 4       // grid, boundaries, centroids
         + 16;                                   // mbarrier + TMEM address
}

template <int BITS, bool F32>
__global__ void __launch_bounds__(kQRows, F32 ? 1 : 2) quantize_qjl_kernel(const QuantArgs a) {
  constexpr int kPitch = RowCfg<F32>::kPitch;
  extern __shared__ uint8_t smem_raw[];
  // operand tiles on a 1 KB boundary
  uint8_t* base = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* ahi = base;
  uint8_t* alo = base + kOpBytes;
  uint8_t* sop = base + 2 * kOpBytes;
  uint8_t* rows = F32 ? base + 3 * kOpBytes : alo;
  float2* grid = (float2*)(base + 3 * kOpBytes + (F32 ? quant_rows_bytes(true) : 0));
  float* bnd = (float*)(grid + a.grid_cells);
  float* cen = bnd + 256;
  uint64_t* bar = (uint64_t*)(cen + 256);
  uint32_t* tslot = (uint32_t*)(bar + 1);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 128;" ::"r"(
                     smem_u32(tslot))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  for (int i = tid; i < 256; i += kQRows) {
    bnd[i] = a.boundaries[i];
    cen[i] = a.centroids[i];
  }
  // S (bf16 [m][d]) as the B operand: row n = tid, 16 chunks of 8 values
  {
    const uint4* srow = (const uint4*)(a.S + (size_t)tid * kD);
#pragma unroll
    for (int c = 0; c < 16; ++c) *(uint4*)(sop + op_offset(tid, c)) = __ldg(srow + c);
  }
  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbarrier_init();
  }
  __syncthreads();
  build_grid<BITS>(a, bnd, grid, tid, kQRows);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t grid_base = smem_u32(grid);
  const uint32_t kmax = (uint32_t)a.grid_cells - 1u;
  const uint32_t limit = a.wait_limit ? a.wait_limit : kDefaultWaitLimit;

  const uint32_t total = (uint32_t)a.B * (uint32_t)a.H * (uint32_t)a.n;
  const uint32_t ntiles = (total + kQRows - 1) / kQRows;
  uint32_t phase = 0;
  bool failed = false;
  // stage: warp w copies rows 32w .. 32w+31 of a tile (the rows its threads
  // quantize); the next tile's rows are staged as soon as the tensor cores
  // have read this tile's R tiles, so their loads overlap the signs and stores
  auto stage = [&](uint32_t t, const void** src, long long* drow, bool* valid) {
    const uint32_t v = t * kQRows + tid;
    *valid = t < ntiles && v < total && resolve_row(a, v, src, drow);
    if constexpr (F32) stage_rows<F32>(*src, *valid, rows + warp * 32 * kPitch, lane);
    else stage_rows_swz(*src, *valid, rows, 32 * warp, lane);
    cp_async_commit();
  };
  const void* src = nullptr;
  long long drow = 0;
  bool valid = false;
  stage(blockIdx.x, &src, &drow, &valid);
  for (uint32_t tile = blockIdx.x; tile < ntiles && !failed; tile += gridDim.x, phase ^= 1u) {
    cp_async_wait<0>();
    __syncwarp();
    // append mode: the ring slots whose tokens this tile has read take the new tokens
    if (a.append && a.W > 0) ring_copies(a, tile * kQRows + tid, tile * kQRows + tid < total, lane);
    // ---- codes, norm and residual of this thread's key; residual rows of R
    float gamma = 0.f;
    {
      float2 p[64];
      if (valid) {
        const float nrm = quantize_row<BITS, F32, (BITS > 4), true, !F32>(
            a, rows + tid * (F32 ? kPitch : 256), grid_base, kmax, cen,
            a.codes + drow * (16 * BITS), p, tid & 7);
        a.norms[drow] = nrm;
        float2 g2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int j = 0; j < 64; ++j) g2 = __ffma2_rn(p[j], p[j], g2);
        gamma = sqrtf(g2.x + g2.y);
      } else {
#pragma unroll
        for (int j = 0; j < 64; ++j) p[j] = make_float2(0.f, 0.f);
      }
      // bf16 rows live in the R lo tile: every thread has read its row
      if constexpr (!F32) __syncthreads();
      // p[j] = (r_j, r_{j+64}); chunk c of the row holds coordinates 8c .. 8c+7
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        uint32_t hw[4], lw[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int i0 = 8 * c + 2 * u;                 // coordinates i0, i0 + 1
          const float r0 = i0 < 64 ? p[i0].x : p[i0 - 64].y;
          const float r1 = i0 + 1 < 64 ? p[i0 + 1].x : p[i0 + 1 - 64].y;
          // packed conversions: hi = bf16(r), lo = bf16(r - hi)
          const __nv_bfloat162 h = __floats2bfloat162_rn(r0, r1);
          const float2 hf = __bfloat1622float2(h);
          const __nv_bfloat162 l = __floats2bfloat162_rn(r0 - hf.x, r1 - hf.y);
          hw[u] = *(const uint32_t*)&h;
          lw[u] = *(const uint32_t*)&l;
        }
        *(uint4*)(ahi + op_offset(tid, c)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        *(uint4*)(alo + op_offset(tid, c)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
      }
    }
    // generic-proxy stores -> visible to the tensor cores' (async proxy) reads
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();
    // ---- Z = R_hi S^T + R_lo S^T: 8 K-steps of 16 for each part
    if (tid == 0) {
      tc_fence_after();
      const uint32_t ah = smem_u32(ahi), al = smem_u32(alo), sb = smem_u32(sop);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        umma_bf16(tmem, umma_desc(ah + ks * 2 * kCoreLbo), umma_desc(sb + ks * 2 * kCoreLbo),
                  ks > 0 ? 1u : 0u);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        umma_bf16(tmem, umma_desc(al + ks * 2 * kCoreLbo), umma_desc(sb + ks * 2 * kCoreLbo), 1u);
      umma_commit(bar);
    }
    __syncwarp();
    if (!__syncthreads_and(mbar_wait(bar, phase, limit, a.err))) {
      // the accumulator never completed (error word set): one more bounded
      // wait for the MMAs in flight, then free the TMEM and stop
      for (uint32_t i = 0; i < limit && !mbar_try_wait(bar, phase); ++i) {
      }
      failed = true;
      break;
    }
    tc_fence_after();
    // the tensor cores are done with R lo, which holds the staged bf16 rows:
    // stage the next tile now (fp32 rows have their own buffer, read already)
    const void* nsrc = nullptr;
    long long ndrow = 0;
    bool nvalid = false;
    stage(tile + gridDim.x, &nsrc, &ndrow, &nvalid);
    // ---- signs: warp w reads TMEM lanes 32w .. 32w+31 (its threads' keys)
    uint32_t sbits[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t z[32];
      tmem_ld32(tmem + ((uint32_t)(32 * warp) << 16) + 32u * q, z);
      asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
      uint32_t w = 0u;
#pragma unroll
      for (int j = 0; j < 32; ++j) w |= (__uint_as_float(z[j]) >= 0.f ? 1u : 0u) << j;
      sbits[q] = w;
    }
    if (valid) {
      *(uint4*)(a.qjl_signs + drow * (kQjlM / 8)) = make_uint4(sbits[0], sbits[1], sbits[2], sbits[3]);
      a.qjl_rnorm[drow] = gamma;
    }
    tc_fence_before();
    __syncthreads();   // TMEM and the R tiles are reused by the next tile
    src = nsrc;
    drow = ndrow;
    valid = nvalid;
  }
  cp_async_wait<0>();
  (void)failed;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 128;" ::"r"(tmem) : "memory");
}

template <int BITS, bool F32>
static int launch_qjl_t(const QuantArgs& a, cudaStream_t s) {
  auto k = quantize_qjl_kernel<BITS, F32>;
  const size_t smem = qjl_smem_bytes(F32, a.grid_cells);
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return 1;
  const long long total = (long long)a.B * a.H * a.n;
  const long long ntiles = (total + kQRows - 1) / kQRows;
  long long grid = (long long)sm_count() * (F32 ? 1 : 2);   // CTAs resident per SM
  if (grid > ntiles) grid = ntiles;
  k<<<(unsigned)grid, kQRows, smem, s>>>(a);
  return cudaGetLastError() != cudaSuccess;
}

int launch_quantize_qjl(const QuantArgs& a, cudaStream_t s) {
  switch (a.bits) {
    case 2: return a.src_f32 ? launch_qjl_t<2, true>(a, s) : launch_qjl_t<2, false>(a, s);
    case 3: return a.src_f32 ? launch_qjl_t<3, true>(a, s) : launch_qjl_t<3, false>(a, s);
    case 4: return a.src_f32 ? launch_qjl_t<4, true>(a, s) : launch_qjl_t<4, false>(a, s);
    case 8: return a.src_f32 ? launch_qjl_t<8, true>(a, s) : launch_qjl_t<8, false>(a, s);
  }
  return 1;
}

}  // namespace tq
