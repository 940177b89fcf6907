// Device pieces shared by the quantize kernels (tq_quantize.cu: codes and
// norms; tq_qjl.cu: codes, norms and the QJL sign sketch on the tensor cores).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "tq_device.cuh"

namespace tq {

constexpr int kQRows = 128;           // vectors per tile = threads per CTA
constexpr int kD = 128;

template <bool F32>
struct RowCfg {
  static constexpr int kRowBytes = F32 ? kD * 4 : kD * 2;
  static constexpr int kPitch = kRowBytes + 16;   // odd multiple of 16 B: conflict-free rows
};

// 128 padded rows (one tile)
__host__ __device__ constexpr size_t quant_rows_bytes(bool f32) {
  return (size_t)kQRows * (f32 ? RowCfg<true>::kPitch : RowCfg<false>::kPitch);
}

// Bytes spanned by the source tensor [B][H][n][d] of a quantize (strides in
// elements, non-negative), and by a bf16 window ring [B][H][W][d].
__device__ __forceinline__ size_t src_extent_bytes(const QuantArgs& a) {
  const long long e = (long long)(a.B - 1) * a.sb + (long long)(a.H - 1) * a.sh +
                      (long long)(a.n - 1) * a.st + kD;
  return (size_t)e * (a.src_f32 ? 4 : 2);
}
__device__ __forceinline__ size_t ring_bytes(int B, int H, int W) {
  return (size_t)B * H * W * kD * 2;
}

// Resolve vector v of the launch: its plane row and, for the stager, its
// source address.  All index arithmetic is 32-bit (a launch covers fewer than
// 2^31 vectors, checked on the host).
__device__ __forceinline__ bool resolve_row(const QuantArgs& a, uint32_t v, const void** src,
                                            long long* dst_row) {
  const uint32_t n = (uint32_t)a.n;
  const uint32_t bh = v / n;
  const uint32_t j = v - bh * n;
  const uint32_t b = bh / (uint32_t)a.H;
  const uint32_t h = bh - b * (uint32_t)a.H;
  const int esz = a.src_f32 ? 4 : 2;
  long long pos;
  if (!a.append) {
    pos = (a.dst_pos ? (long long)a.dst_pos[b] : 0) + j;
    *src = (const uint8_t*)a.src + ((long long)b * a.sb + (long long)h * a.sh + (long long)j * a.st) * esz;
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
      *src = (const uint8_t*)a.src + ((long long)b * a.sb + (long long)h * a.sh + (pos - T0) * a.st) * esz;
    }
  }
  if (pos < 0 || pos >= a.cap) {
    atomicOr(a.err, kErrBounds);
    return false;
  }
  // the source row lies inside the input tensor or the window ring
  // (bounds-checked build; a row outside is not quantized)
  if (kBoundsChecks) {
    const bool from_ring = a.append && pos < (long long)a.seq_before[b];
    const void* base = from_ring ? (const void*)a.win : a.src;
    const size_t bytes = from_ring ? ring_bytes(a.B, a.H, a.W) : src_extent_bytes(a);
    if (!bchk_range(*src, (size_t)kD * (a.src_f32 && !from_ring ? 4 : 2), base, bytes, a.err))
      return false;
  }
  *dst_row = ((long long)bh) * a.cap + pos;
  return true;
}

// Append mode with a window ring: which new token the launch writes into the
// ring for vector index v, and where.  Slot s of a (sequence, head) ring
// receives the newest token t of the append with t = s (mod W), if t is among
// the W newest.  Before the append the slot held the token tau = t - kW just
// below T0 (if tau >= 0): that token leaves the window, is quantized from the
// ring by this launch, and the lane that quantizes it writes t once its row
// has been read.  A slot that held no token (T0 < W) has no reader: the
// vector indices past the quantized range, one for each such slot, write those.
// So every slot has one writer, and none is written before its old token has
// been read.
__device__ __forceinline__ bool ring_copy_of(const QuantArgs& a, uint32_t v, const uint8_t** csrc,
                                             uint16_t** cdst) {
  const uint32_t n = (uint32_t)a.n;
  const uint32_t bh = v / n;
  const uint32_t j = v - bh * n;
  const uint32_t b = bh / (uint32_t)a.H;
  const uint32_t h = bh - b * (uint32_t)a.H;
  const long long W = a.W;
  const long long T0 = a.seq_before[b];
  const long long T1 = T0 + n;
  const long long q0 = T0 - W > 0 ? T0 - W : 0;
  const long long q1 = T1 - W > 0 ? T1 - W : 0;
  const long long pos = q0 + j;
  long long slot, t;
  if (pos < q1) {                          // a quantized token
    if (pos >= T0 || T1 - 1 - pos < W) return false;   // not in the ring, or no successor
    slot = pos % W;
    t = pos + W * ((T1 - 1 - pos) / W);
  } else {                                 // index j - (q1 - q0) of the empty slots
    slot = T0 + (pos - q1);
    if (slot >= W || slot >= T1) return false;
    t = slot + W * ((T1 - 1 - slot) / W);
  }
  *csrc = (const uint8_t*)a.src + ((long long)b * a.sb + (long long)h * a.sh + (t - T0) * a.st) * 2;
  *cdst = a.win + (((long long)b * a.H + h) * W + slot) * kD;
  if (kBoundsChecks)
    return bchk_range(*csrc, kD * 2, a.src, src_extent_bytes(a), a.err) &&
           bchk_range(*cdst, kD * 2, a.win, ring_bytes(a.B, a.H, a.W), a.err);
  return true;
}

// The ring writes of a warp's vectors v (lanes with in_range; see
// ring_copy_of).  Lane l copies 16-byte chunk l % 16 of the rows of lanes
// l / 16, l / 16 + 2, ...: all loads first, then all stores, so that the
// loads' latencies overlap.  Called after the warp's rows have landed in
// shared memory; not inlined, as only appends with a window take it.
static __device__ __noinline__ void ring_copies(const QuantArgs& a, uint32_t v, bool in_range,
                                                   int lane) {
  const uint8_t* cs = nullptr;
  uint16_t* cd = nullptr;
  const bool want = in_range && ring_copy_of(a, v, &cs, &cd);
  const uint32_t m = __ballot_sync(0xffffffffu, want);
  if (m == 0u) return;
  const int c = lane & 15, hf = lane >> 4;
  uint4 buf[16];
  uint4* dst[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const int r = 2 * k + hf;
    const uint4* s = (const uint4*)__shfl_sync(0xffffffffu, (unsigned long long)cs, r);
    dst[k] = (uint4*)__shfl_sync(0xffffffffu, (unsigned long long)cd, r);
    buf[k] = (m >> r) & 1u ? __ldg(s + c) : make_uint4(0u, 0u, 0u, 0u);
  }
#pragma unroll
  for (int k = 0; k < 16; ++k)
    if ((m >> (2 * k + hf)) & 1u) dst[k][c] = buf[k];
}

__device__ __forceinline__ float2 lds64f(uint32_t addr) {
  float2 v;
  asm("ld.shared.v2.f32 {%0,%1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr));
  return v;
}

// A warp stages the 32 rows of its next tile into one of its two row buffers
// with 16-byte asynchronous copies (cp.async): lane l resolved row l; each
// pass copies 512 contiguous source bytes (two bf16 rows or one fp32 row),
// one 16-byte chunk per lane.  Rows that resolve to nothing are not copied.
template <bool F32>
__device__ __forceinline__ void stage_rows(const void* src, bool valid, uint8_t* rows, int lane) {
  constexpr int kRowBytes = RowCfg<F32>::kRowBytes;
  constexpr int kPitch = RowCfg<F32>::kPitch;
  constexpr int kChunks = kRowBytes / 16;            // 16 (bf16) or 32 (fp32)
  constexpr int kRowsPerPass = 32 / kChunks;
  const uint32_t vmask = __ballot_sync(0xffffffffu, valid);
  const int c = lane % kChunks;
#pragma unroll 4
  for (int pass = 0; pass < 32 / kRowsPerPass; ++pass) {
    const int r = pass * kRowsPerPass + lane / kChunks;
    const uint8_t* sp = (const uint8_t*)__shfl_sync(0xffffffffu, (unsigned long long)src, r);
    if ((vmask >> r) & 1u) cp_async16(rows + r * kPitch + 16 * c, sp + 16 * c);
  }
}

// bf16 rows packed 256 bytes apart with their 16-byte chunks permuted: chunk
// c of row r sits at position (c & 8) | ((c ^ r) & 7), so that the 32 lanes
// of a warp, reading the same chunk of 32 consecutive rows, hit 8 different
// bank groups per quarter-warp.  A tile of 128 such rows fills 32 KB.
__device__ __forceinline__ int swz_chunk(int c, int r) { return (c & 8) | ((c ^ r) & 7); }

// stage_rows for the permuted bf16 layout (rows 256 bytes apart)
__device__ __forceinline__ void stage_rows_swz(const void* src, bool valid, uint8_t* rows,
                                               int row0, int lane) {
  const uint32_t vmask = __ballot_sync(0xffffffffu, valid);
  const int c = lane % 16;
#pragma unroll 4
  for (int pass = 0; pass < 16; ++pass) {
    const int r = pass * 2 + lane / 16;
    const uint8_t* sp = (const uint8_t*)__shfl_sync(0xffffffffu, (unsigned long long)src, r);
    if ((vmask >> r) & 1u)
      cp_async16(rows + (row0 + r) * 256 + 16 * swz_chunk(c, row0 + r), sp + 16 * c);
  }
}

// Rotated coordinates of one vector, held as pairs (y_j, y_{j+64}), j < 64,
// so that six of the seven butterfly stages run on packed fp32 pairs.
// SWZ: bf16 row in the permuted layout, rsw = its row index (mod 8).
template <bool F32, bool SWZ = false>
__device__ __forceinline__ float load_rotate(const QuantArgs& a, const uint8_t* row,
                                             float2 (&p)[64], int rsw = 0) {
  if constexpr (F32) {
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const uint4 lo = lds128(row + 16 * c);            // coordinates 4c .. 4c+3
      const uint4 hi = lds128(row + 256 + 16 * c);      // coordinates 64+4c ..
      p[4 * c + 0] = make_float2(__uint_as_float(lo.x ^ a.smask[4 * c + 0]), __uint_as_float(hi.x ^ a.smask[64 + 4 * c + 0]));
      p[4 * c + 1] = make_float2(__uint_as_float(lo.y ^ a.smask[4 * c + 1]), __uint_as_float(hi.y ^ a.smask[64 + 4 * c + 1]));
      p[4 * c + 2] = make_float2(__uint_as_float(lo.z ^ a.smask[4 * c + 2]), __uint_as_float(hi.z ^ a.smask[64 + 4 * c + 2]));
      p[4 * c + 3] = make_float2(__uint_as_float(lo.w ^ a.smask[4 * c + 3]), __uint_as_float(hi.w ^ a.smask[64 + 4 * c + 3]));
    }
  } else {
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const int pc = SWZ ? (c ^ rsw) & 7 : c;           // chunk position in the row
      const uint4 lo = lds128(row + 16 * pc);           // coordinates 8c .. 8c+7
      const uint4 hi = lds128(row + 128 + 16 * pc);     // coordinates 64+8c ..
      const uint32_t l[4] = {lo.x, lo.y, lo.z, lo.w};
      const uint32_t h[4] = {hi.x, hi.y, hi.z, hi.w};
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = 8 * c + 2 * u;
        // bf16 -> fp32 with the sign flip: adding 0x80000000 flips the sign bit
        p[i] = make_float2(__uint_as_float(l[u] * 65536u + a.smask[i]),
                           __uint_as_float(h[u] * 65536u + a.smask[64 + i]));
        p[i + 1] = make_float2(__uint_as_float((l[u] & 0xFFFF0000u) ^ a.smask[i + 1]),
                               __uint_as_float((h[u] & 0xFFFF0000u) ^ a.smask[64 + i + 1]));
      }
    }
  }
  float2 s0 = make_float2(0.f, 0.f), s1 = s0;
#pragma unroll
  for (int j = 0; j < 64; j += 2) {
    s0 = __ffma2_rn(p[j], p[j], s0);
    s1 = __ffma2_rn(p[j + 1], p[j + 1], s1);
  }
  const float2 s = __fadd2_rn(s0, s1);
  // butterflies between pairs: stages 1, 2, 4, ..., 32 of the index j
  const float2 neg1 = make_float2(-1.f, -1.f);
#pragma unroll
  for (int hs = 1; hs < 64; hs <<= 1) {
#pragma unroll
    for (int j = 0; j < 64; ++j) {
      if ((j & hs) == 0) {
        const float2 u = p[j], w = p[j + hs];
        p[j] = __fadd2_rn(u, w);
        p[j + hs] = __ffma2_rn(w, neg1, u);
      }
    }
  }
  // stage 64: inside each pair
#pragma unroll
  for (int j = 0; j < 64; ++j) p[j] = make_float2(p[j].x + p[j].y, p[j].x - p[j].y);
  return sqrtf(s.x + s.y);
}

// Search-grid table (see SearchGrid in tq_internal.h) from the boundaries in
// shared memory: entry k = (first boundary at or above the lower edge of cells
// k-1..k+1, number of boundaries below that edge).  Called by all threads of
// the CTA; the caller synchronises before using the table.
template <int BITS>
__device__ __forceinline__ void build_grid(const QuantArgs& a, const float* bnd, float2* grid,
                                           int tid, int nthreads) {
  const int off = a.grid_cells / 2;
  for (int k = tid; k < a.grid_cells; k += nthreads) {
    const float lo = ((float)(k - off) - 1.5f) / a.grid_scale;
    uint32_t idx = 0;
#pragma unroll
    for (int step = (1 << BITS) / 2; step >= 1; step >>= 1)
      if (bnd[idx + step - 1] < lo) idx += step;
    grid[k] = make_float2(bnd[idx], __uint_as_float(idx));
  }
}

// Code search and packing of one vector from its unnormalised rotated
// coordinates p (pairs (z_j, z_{j+64}) of z = H (s * x), H the +-1 Sylvester
// matrix) and its norm: y = z / (||x|| sqrt(d)); the codes go to codes_dst
// (16 * BITS bytes).  With RESID, p holds the rotated-domain residual
// ||x|| (y - c[idx]) afterwards, from the centroids `cen` in shared memory.
// GUARD bounds every grid index; without it the caller guarantees |y_i| <= 1
// (up to rounding), inside the grid of a 2-4 bit codebook.
template <int BITS, bool CLAMP, bool GUARD, bool RESID>
__device__ __forceinline__ void search_pack_t(const QuantArgs& a, float2 (&p)[64], float nrm,
                                              uint32_t grid_base, uint32_t kmax, const float* cen,
                                              uint8_t* codes_dst) {
  constexpr int NW = 4 * BITS;         // 32-bit code words per vector (128 * BITS / 32)
  const float inv = nrm > 0.f ? 1.0f / (nrm * 11.313708498984761f) : 0.f;
  const float2 inv2 = make_float2(inv, inv);
  const float2 gs2 = make_float2(a.grid_scale, a.grid_scale);
  const float2 gm2 = make_float2(a.grid_magic, a.grid_magic);
  const uint32_t bias = grid_base - 0x4B400000u * 8u;
  uint32_t words[NW];
#pragma unroll
  for (int k = 0; k < NW; ++k) words[k] = 0u;
#pragma unroll
  for (int j = 0; j < 64; ++j) {
    const float2 y = __fmul2_rn(p[j], inv2);
    float2 yc = y;
    if constexpr (CLAMP) {
      yc.x = fminf(fmaxf(y.x, -a.grid_clamp), a.grid_clamp);
      yc.y = fminf(fmaxf(y.y, -a.grid_clamp), a.grid_clamp);
    }
    const float2 t = __ffma2_rn(yc, gs2, gm2);
    uint32_t a0, a1;                                 // grid entry addresses
    if constexpr (GUARD) {
      a0 = grid_base + min(__float_as_uint(t.x) - 0x4B400000u, kmax) * 8u;
      a1 = grid_base + min(__float_as_uint(t.y) - 0x4B400000u, kmax) * 8u;
    } else {
      a0 = __float_as_uint(t.x) * 8u + bias;        // cell = bits(t) - bits(magic)
      a1 = __float_as_uint(t.y) * 8u + bias;
    }
    if constexpr (kBoundsChecks) {   // grid entries of this launch's table
      const uint32_t end = grid_base + (kmax + 1u) * 8u;
      if (a0 < grid_base || a0 + 8u > end || a1 < grid_base || a1 + 8u > end) {
        atomicOr(a.err, kErrBounds);
        a0 = a1 = grid_base;
      }
    }
    const float2 e0 = lds64f(a0);
    const float2 e1 = lds64f(a1);
    const uint32_t c0 = __float_as_uint(e0.y) + (e0.x < y.x ? 1u : 0u);
    const uint32_t c1 = __float_as_uint(e1.y) + (e1.x < y.y ? 1u : 0u);
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int i = j + 64 * half;                   // coordinate
      const uint32_t code = half ? c1 : c0;
      const int pb = i * BITS;
      // fields do not overlap: a multiply-add places the code
      words[pb >> 5] = code * (1u << (pb & 31)) + words[pb >> 5];
      if ((pb & 31) + BITS > 32) words[(pb >> 5) + 1] |= code >> (32 - (pb & 31));
    }
    if constexpr (RESID) p[j] = make_float2(nrm * (y.x - cen[c0]), nrm * (y.y - cen[c1]));
  }
  uint4* dc = (uint4*)codes_dst;
#pragma unroll
  for (int k = 0; k < BITS; ++k)
    dc[k] = make_uint4(words[4 * k], words[4 * k + 1], words[4 * k + 2], words[4 * k + 3]);
}

// A row whose norm is finite and of normal size has |y_i| <= 1 to within
// rounding, inside the search grid of a 2-4 bit codebook (8-bit grids clamp
// y): it takes the unguarded search.  Rows with inf or NaN, or so small that
// the sum of squares loses precision, take the guarded one.
template <int BITS, bool CLAMP, bool RESID>
__device__ __forceinline__ void search_pack(const QuantArgs& a, float2 (&p)[64], float nrm,
                                            uint32_t grid_base, uint32_t kmax, const float* cen,
                                            uint8_t* codes_dst) {
  if (!CLAMP && nrm <= 3.4e38f && nrm >= 1e-18f)
    search_pack_t<BITS, CLAMP, false, RESID>(a, p, nrm, grid_base, kmax, cen, codes_dst);
  else
    search_pack_t<BITS, CLAMP, true, RESID>(a, p, nrm, grid_base, kmax, cen, codes_dst);
}

// Norm, rotation, code search and packing of the vector in `row` (shared
// memory); the codes go to codes_dst (16 * BITS bytes).  Returns ||x||.  With
// RESID, p holds the rotated-domain residual n (y - c[idx]) afterwards (pairs
// (r_j, r_{j+64})), from the centroids `cen` in shared memory.
template <int BITS, bool F32, bool CLAMP, bool RESID, bool SWZ = false>
__device__ __forceinline__ float quantize_row(const QuantArgs& a, const uint8_t* row,
                                              uint32_t grid_base, uint32_t kmax,
                                              const float* cen, uint8_t* codes_dst,
                                              float2 (&p)[64], int rsw = 0) {
  const float nrm = load_rotate<F32, SWZ>(a, row, p, rsw);
  search_pack<BITS, CLAMP, RESID>(a, p, nrm, grid_base, kmax, cen, codes_dst);
  return nrm;
}

// Unnormalised Walsh-Hadamard transform (Sylvester order) of 128 values held
// by a warp, lane l holding 4l..4l+3: stages 1 and 2 inside the lane, 4..64
// across lanes.
__device__ __forceinline__ void warp_fwht4(float (&x)[4], int lane) {
  const float t0 = x[0] + x[1], t1 = x[0] - x[1], t2 = x[2] + x[3], t3 = x[2] - x[3];
  x[0] = t0 + t2; x[2] = t0 - t2; x[1] = t1 + t3; x[3] = t1 - t3;
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const bool hi = (lane & m) != 0;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const float p = __shfl_xor_sync(0xffffffffu, x[c], m);
      x[c] = hi ? p - x[c] : x[c] + p;
    }
  }
}

// One vector quantized by one warp: lane l holds coordinates 4l..4l+3 (x, in
// place: flipped by the signs sg, then rotated), two butterfly stages in the
// lane and five by shuffles.  Writes the codes
// (16 * bits bytes, dense LSB-first) and the norm, returns the norm and leaves
// the lane's centroids c[idx] in yq and rotated-domain residuals
// ||x|| (y - c[idx]) in r.  bnd / cen: the codebook's boundaries and
// centroids in shared memory; words: 32 words of shared scratch, zero on
// entry and left zero.
__device__ __forceinline__ float warp_quantize_vals(float (&x)[4], float4 sg, int bits,
                                                    const float* bnd, const float* cen,
                                                    uint8_t* codes_dst, float* norm_dst,
                                                    uint32_t* words, int lane, float (&r)[4],
                                                    float (&yq)[4]) {
  x[0] *= sg.x; x[1] *= sg.y; x[2] *= sg.z; x[3] *= sg.w;
  float ss = x[0] * x[0];
  ss = fmaf(x[1], x[1], ss);
  ss = fmaf(x[2], x[2], ss);
  ss = fmaf(x[3], x[3], ss);
  const float nrm = sqrtf(warp_sum(ss));
  warp_fwht4(x, lane);
  const float inv = nrm > 0.f ? 1.0f / (nrm * 11.313708498984761f) : 0.f;
  uint32_t packed = 0;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const float y = x[c] * inv;
    uint32_t idx = 0;
    for (int step = 1 << (bits - 1); step >= 1; step >>= 1)
      if (bnd[idx + step - 1] < y) idx += step;
    packed |= idx << (c * bits);
    yq[c] = cen[idx];
    r[c] = nrm * (y - yq[c]);
  }
  // dense LSB-first stream: lane l's 4*bits bits start at bit 4*bits*l
  const int pos = 4 * bits * lane;
  const int wi = pos >> 5, sh = pos & 31;
  atomicOr(&words[wi], packed << sh);
  if (sh + 4 * bits > 32) atomicOr(&words[wi + 1], packed >> (32 - sh));
  __syncwarp();
  if (lane < bits)
    ((uint4*)codes_dst)[lane] = make_uint4(words[4 * lane], words[4 * lane + 1],
                                           words[4 * lane + 2], words[4 * lane + 3]);
  if (lane == 0) *norm_dst = nrm;
  __syncwarp();
  if (lane < 4 * bits) words[lane] = 0u;
  __syncwarp();
  return nrm;
}
// the same from a row in memory (bf16, or fp32 when f32)
__device__ __forceinline__ float warp_quantize_row(const void* src, int f32, float4 sg, int bits,
                                                   const float* bnd, const float* cen,
                                                   uint8_t* codes_dst, float* norm_dst,
                                                   uint32_t* words, int lane, float (&r)[4],
                                                   float (&yq)[4]) {
  float x[4];
  if (f32) {
    const float4 v = ((const float4*)src)[lane];
    x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
  } else {
    const uint2 v = ((const uint2*)src)[lane];
    x[0] = bf16lo(v.x); x[1] = bf16hi(v.x); x[2] = bf16lo(v.y); x[3] = bf16hi(v.y);
  }
  return warp_quantize_vals(x, sg, bits, bnd, cen, codes_dst, norm_dst, words, lane, r, yq);
}

// Direct Sign of a residual held by a warp as in warp_quantize_row: bit i =
// [r_i >= 0] (lane l: coordinates 4l..4l+3), scale = mean |r_i|
// ("TurboQuant KV 캐시 압축 for llama.cpp", v1.1.0 "Direct Sign").  Returns
// the scale (in every lane).
__device__ __forceinline__ float warp_direct_sign(const float (&r)[4], uint8_t* signs_dst,
                                                  float* scale_dst, int lane) {
  uint32_t nib = 0u;
#pragma unroll
  for (int c = 0; c < 4; ++c) nib |= (r[c] >= 0.f ? 1u : 0u) << c;
  const float asum = warp_sum(fabsf(r[0]) + fabsf(r[1]) + fabsf(r[2]) + fabsf(r[3]));
  // lanes 8w .. 8w+7 fill word w; gather with shuffles
  uint32_t word = nib << (4 * (lane & 7));
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) word |= __shfl_xor_sync(0xffffffffu, word, o);
  const uint32_t w0 = __shfl_sync(0xffffffffu, word, 0), w1 = __shfl_sync(0xffffffffu, word, 8);
  const uint32_t w2 = __shfl_sync(0xffffffffu, word, 16), w3 = __shfl_sync(0xffffffffu, word, 24);
  const float scale = asum * (1.0f / kD);
  if (lane == 0) {
    *(uint4*)signs_dst = make_uint4(w0, w1, w2, w3);
    *scale_dst = scale;
  }
  return scale;
}

// QJL sketch of a residual held by a warp as in warp_quantize_vals (lane l:
// coordinates 4l..4l+3): gamma = ||r|| and bit j = [(S r)_j >= 0] for the
// kQjlM rows of S (bf16, [m][d]); lane l computes rows l, l + 32, l + 64,
// l + 96 ("TurboQuant KV 캐시 압축 for llama.cpp", "QJL 보정 효과").  rbuf: 128
// floats of shared scratch.  Writes the 16 sign bytes and gamma, leaves the
// sign words (bit j of word j / 32) in sb in every lane and returns gamma.
__device__ __forceinline__ float warp_qjl_sketch(const float (&r)[4], const uint16_t* S, float* rbuf,
                                                 uint8_t* signs_dst, float* gamma_dst, int lane,
                                                 uint32_t (&sb)[4]) {
  float g = r[0] * r[0];
  g = fmaf(r[1], r[1], g);
  g = fmaf(r[2], r[2], g);
  g = fmaf(r[3], r[3], g);
  const float gamma = sqrtf(warp_sum(g));
  *(float4*)(rbuf + 4 * lane) = make_float4(r[0], r[1], r[2], r[3]);
  __syncwarp();
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint4* Sj = (const uint4*)(S + (size_t)(32 * k + lane) * kD);
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
    sb[k] = __ballot_sync(0xffffffffu, z0 + z1 >= 0.f);
  }
  if (lane == 0) {
    *(uint4*)signs_dst = make_uint4(sb[0], sb[1], sb[2], sb[3]);
    *gamma_dst = gamma;
  }
  __syncwarp();      // rbuf is read by every lane before it is written again
  return gamma;
}

// Direct Sign sketch of a residual held as pairs p[j] = (r_j, r_{j+64}): bit
// i of the 128-bit sign vector is [r_i >= 0]; the scale is mean |r_i|
// ("TurboQuant KV 캐시 압축 for llama.cpp", v1.1.0 "Direct Sign").
__device__ __forceinline__ void direct_sign(const float2 (&p)[64], uint8_t* signs_dst,
                                            float* scale_dst) {
  uint32_t sw[4] = {0u, 0u, 0u, 0u};
  float asum = 0.f;
#pragma unroll
  for (int j = 0; j < 64; ++j) {
    sw[j >> 5] |= (p[j].x >= 0.f ? 1u : 0u) << (j & 31);
    sw[2 + (j >> 5)] |= (p[j].y >= 0.f ? 1u : 0u) << (j & 31);
    asum += fabsf(p[j].x) + fabsf(p[j].y);
  }
  *(uint4*)signs_dst = make_uint4(sw[0], sw[1], sw[2], sw[3]);
  *scale_dst = asum * (1.0f / kD);
}

}  // namespace tq
