// Decode attention over a TurboQuant-compressed KV cache (sm_103a): the kernel
// template, instantiated per (query heads per kv-head G, key bits, value bits,
// key residual term: none, QJL sketch or Direct Sign) in
// tq_decode_g{1,2,4,8}.cu so that each launch runs code for exactly one
// storage format.
//
// "TurboQuant KV 캐시 압축 for llama.cpp": v1.7.0 decision 4 (the decode kernel
// applies the encoders' WHT to Q, so q_rot . k_rot = q . k by Parseval);
// v1.5.2 changes 1-2 (accumulate in fp32, never half) and 4 (V is summed in
// the rotated domain and needs one inverse rotation at the output); v1.4.2
// items 1 and 2 (dequantized codes fed to tensor-core MMA; the QJL term is a
// correction from the sign bits and the stored residual scale).
//
// One CTA = (split, kv-head, sequence): with MSE keys one CTA per SM of 12
// (or 8) warps for G <= 4 query columns and of 8 warps for G = 8; with a key
// residual term two or three of 4 warps (decode_warps, decode_ctas_per_sm).  Prologue: the G query heads
// of the kv-head are scaled by softmax_scale*log2(e), rotated with the K sign
// vector and split into fp16 hi + lo MMA operands held in registers; QJL keys
// also get S q_rot as hi + lo operands.  Main loop, per warp and 32-token
// chunk (bulk copies into a 3- or 4-slot ring, bounded mbarrier waits), all on
// mma.sync m16n8k16 with fp32 accumulators:
//   scores   S[tokens x heads] = K_c[tokens x coords] Q[coords x heads]: the
//            packed codes are decoded in registers through tables of fp16
//            centroid hi/lo parts; hi*hi + lo*hi + hi*lo carry ~22 bits, so the
//            scores match fp32 arithmetic; times ||k|| (fp32), plus for QJL
//            keys gamma * sqrt(pi/2)/m * (+-1 signs)[tokens x m] (S q_rot);
//   softmax  online, per head, in the log2 domain, on the accumulator layout;
//   V sum    D[coords x heads] += V_c^T W with fp16 centroid pairs and fp16
//            weights scaled per chunk into range (error <= ~5e-4 relative).
// The split owning the residual window scores the bf16 window tokens in the
// original domain on CUDA cores.  Epilogue: warps merge by log-sum-exp, the
// CTA writes (m, l, o) for its split; the last CTA of the (sequence, kv-head)
// merges the splits, one warp per head, inverse-rotates with the V sign vector
// by an in-register butterfly and writes the output.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "tq_device.cuh"
#include "tq_quant_common.cuh"

namespace tq {

constexpr int kD2 = 128;
constexpr float kNegBig = -1.0e30f;
constexpr float kCScale = 64.f;   // centroids are scaled by 64 in the K tables
// the running softmax maxima are raised only when a score exceeds them by
// more than this (log2 units), so softmax weights are at most 2^kLazyMax
constexpr float kLazyMax = 8.f;

// 2^x on the MUFU unit (relative error about 2^-22; results below the fp32
// normal range flush to zero, as the softmax weights may)
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint32_t byte_of(uint32_t x, int b) {
  return __byte_perm(x, 0u, 0x4440u | (uint32_t)b);
}
__device__ __forceinline__ uint32_t half_of(uint32_t x, int h) {
  return __byte_perm(x, 0u, h ? 0x4432u : 0x4410u);
}
__device__ __forceinline__ uint32_t h16(float x) {
  return (uint32_t)__half_as_ushort(__float2half_rn(x));
}
// fp16 hi and lo parts of x (x ~= hi + lo to ~22 bits), packed hi | lo << 16
__device__ __forceinline__ uint32_t hilo(float x) {
  const __half h = __float2half_rn(x);
  return (uint32_t)__half_as_ushort(h) | (h16(x - __half2float(h)) << 16);
}
// pack two (hi | lo << 16) entries into the hi pair and the lo pair
__device__ __forceinline__ void pack_hilo(uint32_t e0, uint32_t e1, uint32_t& hi, uint32_t& lo) {
  hi = __byte_perm(e0, e1, 0x5410);
  lo = __byte_perm(e0, e1, 0x7632);
}
// the same hi pair and lo pair of (x0, x1) from packed conversions: two
// conversions for two values instead of four
__device__ __forceinline__ void hilo2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __floats2half2_rn(x0, x1);
  const float2 f = __half22float2(h);
  const __half2 l = __floats2half2_rn(x0 - f.x, x1 - f.y);
  hi = *(const uint32_t*)&h;
  lo = *(const uint32_t*)&l;
}
// ---- V sum on the tensor cores ------------------------------------------------
// D[coords x heads] += V^T[coords x tokens] W[tokens x heads] with
// mma.sync m16n8k16 (fp16 operands, fp32 accumulate).  The m index is a free
// permutation of the coordinates: thread (g = lane/4, tig = lane%4) owns rows
// g and g+8 of every m-tile k, mapped to coordinates 16g+2k and 16g+2k+1, so
// its 16 coordinates are contiguous in a packed row.  The k index is a free
// permutation of the tokens: columns 2j, 2j+1 of k-tile kt are tokens
// 16kt + j and 16kt + j + 8, the two tokens whose scores a lane of the score
// MMA holds, so that lane packs both weights into one B register; B holds the
// fp16 softmax weights.
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// Coordinate of accumulator row g (hi = 0) or g + 8 (hi = 1) of m-tile k for
// lane group g: 2-bit values pair coordinates c and c + 2 in one code byte
// (see vmma_ktile), wider values c and c + 1.
template <int VB>
__device__ __forceinline__ int vrow_coord(int g, int k, int hi) {
  if constexpr (VB == 2) return 16 * g + 4 * (k >> 1) + (k & 1) + 2 * hi;
  else return 16 * g + 2 * k + hi;
}

// A operands of k-tile kt for the 8 m-tiles, then the 8 MMAs.
// 2-bit values: vtab is the value half of the shared pair table (entry b at
// byte 256 b, lane l's replica 8 (l % 16) bytes into it, laneV = 128 + 8 (l %
// 16) being that replica's offset in the row): for a byte b of the codes of two
// tokens (bits 0-1 / 2-3: coordinate c of the first / second token, bits 4-5 /
// 6-7: coordinate c + 2), entry b is the operand pair (a0, a1) or (a2, a3) as
// loaded: half2 (c_V of the two tokens) for c and for c + 2.
// lutp: for 3-bit values, half2 (c[i0], c[i1]) indexed by the pair (i0 | i1 <<
// 3) of the codes of the two tokens of an operand register; for 4- and 8-bit
// values, fp16 c[i] in the low half (pairs are packed with a byte permute).
template <int VB>
__device__ __forceinline__ void vmma_ktile(const uint8_t* vbuf, const uint32_t* lutp,
                                           const uint8_t* vtab, uint32_t laneV, int kt,
                                           int g, int tig, uint32_t b0, uint32_t b1,
                                           float (&d)[8][4], unsigned* err) {
  constexpr int VROW = 16 * VB;
  // a0/a1: columns 2tig, 2tig+1 = tokens t0, t0 + 8; a2/a3: columns 2tig+8,
  // 2tig+9 = tokens t0 + 4, t0 + 12 (rows of the chunk's 32-row slot)
  const int t0 = 16 * kt + tig;
  const uint8_t* r0 = bchk((const uint8_t(*)[VROW])(vbuf + t0 * VROW), vbuf, 32 * VROW, err)[0];
  const uint8_t* r1 = bchk((const uint8_t(*)[VROW])(vbuf + (t0 + 8) * VROW), vbuf, 32 * VROW, err)[0];
  const uint8_t* r2 = bchk((const uint8_t(*)[VROW])(vbuf + (t0 + 4) * VROW), vbuf, 32 * VROW, err)[0];
  const uint8_t* r3 = bchk((const uint8_t(*)[VROW])(vbuf + (t0 + 12) * VROW), vbuf, 32 * VROW, err)[0];
  // lookups stay inside the 256-entry tables
  auto lut_u32 = [&](const uint32_t* lut, uint32_t off) {
    return *bchk((const uint32_t*)((const char*)lut + off), lut, 256 * 4, err);
  };
  if constexpr (VB == 2) {
    const uint32_t x0 = *(const uint32_t*)(r0 + 4 * g), x1 = *(const uint32_t*)(r1 + 4 * g);
    const uint32_t x2 = *(const uint32_t*)(r2 + 4 * g), x3 = *(const uint32_t*)(r3 + 4 * g);
    // byte b of zA: codes of coordinates 16g + 4b (bits 0-3) and 16g + 4b + 2
    // (bits 4-7) of tokens t0 and t0 + 8; zA2 the same for 16g + 4b + 1 and
    // + 3; zB, zB2 for tokens t0 + 4, t0 + 12.  m-tile k reads byte k / 2 of
    // zA (k even) or zA2 (k odd): rows g / g + 8 are coordinates c / c + 2.
    const uint32_t zA = (x0 & 0x33333333u) | ((x1 & 0x33333333u) << 2);
    const uint32_t zA2 = ((x0 >> 2) & 0x33333333u) | (x1 & 0xCCCCCCCCu);
    const uint32_t zB = (x2 & 0x33333333u) | ((x3 & 0x33333333u) << 2);
    const uint32_t zB2 = ((x2 >> 2) & 0x33333333u) | (x3 & 0xCCCCCCCCu);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint32_t sel = 0x5504u | ((uint32_t)(k >> 1) << 4);
      const uint2 ea = *bchk((const uint2*)(vtab + __byte_perm((k & 1) ? zA2 : zA, laneV, sel)),
                             vtab, 256 * 256, err);
      const uint2 eb = *bchk((const uint2*)(vtab + __byte_perm((k & 1) ? zB2 : zB, laneV, sel)),
                             vtab, 256 * 256, err);
      mma16816(d[k], ea.x, ea.y, eb.x, eb.y, b0, b1);
    }
  } else if constexpr (VB == 3) {
    // 48 bits of coordinates 16g..16g+15 start at byte 6g of a 48-byte row;
    // as two words: lo = bits 0-31, hi = bits 32-47
    const int bo = 6 * g;
    const int sh = 8 * (bo & 3);
    auto bits48 = [&](const uint8_t* r, uint32_t& lo, uint32_t& hi) {
      const uint32_t* w = (const uint32_t*)(r + (bo & ~3));
      lo = __funnelshift_r(w[0], w[1], sh);
      hi = w[1] >> sh;
    };
    uint32_t l0, h0, l1, h1, l2, h2, l3, h3;
    bits48(r0, l0, h0);
    bits48(r1, l1, h1);
    bits48(r2, l2, h2);
    bits48(r3, l3, h3);
    // the 3-bit field at bit P of (hi:lo) moved to bit Q (compile-time P, Q)
    auto field = [](uint32_t lo, uint32_t hi, int P, int Q) -> uint32_t {
      if (P < Q) return lo << (Q - P);
      if (P - Q < 32) return __funnelshift_r(lo, hi, P - Q);
      return hi >> (P - Q - 32);
    };
    // byte offset 4e of pair entry e = x | y << 3 for codes x (first token)
    // and y (second token)
    auto pair_off = [&](uint32_t la, uint32_t ha, uint32_t lb, uint32_t hb, int i) {
      return (field(la, ha, 3 * i, 2) & 0x1Cu) | (field(lb, hb, 3 * i, 5) & 0xE0u);
    };
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint32_t a0 = lut_u32(lutp, pair_off(l0, h0, l1, h1, 2 * k));
      const uint32_t a1 = lut_u32(lutp, pair_off(l0, h0, l1, h1, 2 * k + 1));
      const uint32_t a2 = lut_u32(lutp, pair_off(l2, h2, l3, h3, 2 * k));
      const uint32_t a3 = lut_u32(lutp, pair_off(l2, h2, l3, h3, 2 * k + 1));
      mma16816(d[k], a0, a1, a2, a3, b0, b1);
    }
  } else if constexpr (VB == 4) {
    const uint2 x0 = *(const uint2*)(r0 + 8 * g), x1 = *(const uint2*)(r1 + 8 * g);
    const uint2 x2 = *(const uint2*)(r2 + 8 * g), x3 = *(const uint2*)(r3 + 8 * g);
    const uint32_t w0[2] = {x0.x, x0.y}, w1[2] = {x1.x, x1.y}, w2[2] = {x2.x, x2.y},
                   w3[2] = {x3.x, x3.y};
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int wi = k >> 2, by = k & 3;
      // low nibble of byte k%4 of word k/4: coordinate 16g+2k; high nibble: 16g+2k+1
      auto lo = [&](uint32_t w) { return lut_u32(lutp, byte_of((w << 2) & 0x3C3C3C3Cu, by)); };
      auto hi = [&](uint32_t w) { return lut_u32(lutp, byte_of((w >> 2) & 0x3C3C3C3Cu, by)); };
      const uint32_t a0 = __byte_perm(lo(w0[wi]), lo(w1[wi]), 0x5410);
      const uint32_t a1 = __byte_perm(hi(w0[wi]), hi(w1[wi]), 0x5410);
      const uint32_t a2 = __byte_perm(lo(w2[wi]), lo(w3[wi]), 0x5410);
      const uint32_t a3 = __byte_perm(hi(w2[wi]), hi(w3[wi]), 0x5410);
      mma16816(d[k], a0, a1, a2, a3, b0, b1);
    }
  } else {   // VB == 8: one byte per coordinate, 16 bytes at byte 16g
    const uint4 x0 = *(const uint4*)(r0 + 16 * g), x1 = *(const uint4*)(r1 + 16 * g);
    const uint4 x2 = *(const uint4*)(r2 + 16 * g), x3 = *(const uint4*)(r3 + 16 * g);
    const uint32_t w0[4] = {x0.x, x0.y, x0.z, x0.w}, w1[4] = {x1.x, x1.y, x1.z, x1.w},
                   w2[4] = {x2.x, x2.y, x2.z, x2.w}, w3[4] = {x3.x, x3.y, x3.z, x3.w};
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int wi = k >> 1, hh = k & 1;
      // bytes 2(k%2) and 2(k%2)+1 of word k/2: coordinates 16g+2k, 16g+2k+1
      auto ev = [&](uint32_t w) { return lut_u32(lutp, half_of((w << 2) & 0x03FC03FCu, hh)); };
      auto od = [&](uint32_t w) { return lut_u32(lutp, half_of((w >> 6) & 0x03FC03FCu, hh)); };
      const uint32_t a0 = __byte_perm(ev(w0[wi]), ev(w1[wi]), 0x5410);
      const uint32_t a1 = __byte_perm(od(w0[wi]), od(w1[wi]), 0x5410);
      const uint32_t a2 = __byte_perm(ev(w2[wi]), ev(w3[wi]), 0x5410);
      const uint32_t a3 = __byte_perm(od(w2[wi]), od(w3[wi]), 0x5410);
      mma16816(d[k], a0, a1, a2, a3, b0, b1);
    }
  }
}

// ---- scores on the tensor cores ---------------------------------------------
// S[tokens x heads] = K_c[tokens x coords] Q[coords x heads].  The k index is a
// free permutation of the coordinates: thread (g, tig) supplies columns 2tig,
// 2tig+1 (and 2tig+8, 2tig+9) of k-tile kt, mapped to coordinates 32tig+4kt,
// +1 (and +2, +3), so its 32 coordinates are contiguous in a packed row.
// Key tables (centroids x kCScale): 2, 3 and 4 bits: uint2 (hi pair, lo pair)
// indexed by the code pair (c_i | c_{i+1} << KB); the 3- and 4-bit tables (64
// and 256 pairs) are the key halves of the shared pair table: 16 replicas
// interleaved 8 bytes apart in 256-byte rows, lane l reading replica l % 16,
// so a half-warp's 16 lookups never collide; 8 bits: u32 hi | lo << 16 per code.
template <int KB>
struct KCodes {  // one token's 32 codes for this thread, as table offsets
  uint32_t w[KB];
};

template <int KB>
__device__ __forceinline__ void load_kcodes(const uint8_t* slot, int r, int tig, KCodes<KB>& c,
                                            unsigned* err) {
  // row r of the chunk's 32-row slot
  const uint8_t* row =
      bchk((const uint8_t(*)[16 * KB])(slot + r * 16 * KB), slot, 32 * 16 * KB, err)[0];
  if constexpr (KB == 2) {
    const uint2 x = *(const uint2*)(row + 8 * tig);
    c.w[0] = x.x;
    c.w[1] = x.y;
  } else if constexpr (KB == 3) {
    const uint32_t* p = (const uint32_t*)(row + 12 * tig);
    c.w[0] = p[0];
    c.w[1] = p[1];
    c.w[2] = p[2];
  } else if constexpr (KB == 4) {
    const uint4 x = *(const uint4*)(row + 16 * tig);
    c.w[0] = x.x; c.w[1] = x.y; c.w[2] = x.z; c.w[3] = x.w;
  } else {
    const uint4 x = *(const uint4*)(row + 32 * tig);
    const uint4 y = *(const uint4*)(row + 32 * tig + 16);
    c.w[0] = x.x; c.w[1] = x.y; c.w[2] = x.z; c.w[3] = x.w;
    c.w[4] = y.x; c.w[5] = y.y; c.w[6] = y.z; c.w[7] = y.w;
  }
}

// (hi pair, lo pair) operand of coordinates 32tig + i, i+1 (i even, compile time).
// 3- and 4-bit keys: lut is the base of the pair table (entry p at byte 256 p,
// lane l's replica 8 (l % 16) bytes into it) and lane8 = 8 (lane % 16), so the
// byte offset (p << 8) | lane8 is one byte permute (4 bits: the pair is a
// byte of the codes) or one shift and one masked OR (3 bits) away from the codes.
template <int KB, int I>
__device__ __forceinline__ void kpair(const KCodes<KB>& c, const uint32_t* lut, uint32_t lane8,
                                      uint32_t& hi, uint32_t& lo, unsigned* err) {
  // extent of the table this format reads: the 3/4-bit pair table's key rows
  // (256-byte rows), else the kernel's 256-word table
  constexpr size_t kLutBytes = KB == 4 ? 256 * 256 : KB == 3 ? 64 * 256 : 256 * 4;
  if constexpr (KB == 2) {
    // nibble I/2 of the 64 code bits: byte (I/4) % 4 of word I/16, low or high nibble
    const uint32_t w = c.w[I / 16];
    const uint32_t off = (I / 2) % 2 == 0 ? byte_of((w << 3) & 0x78787878u, (I / 4) % 4)
                                          : byte_of((w >> 1) & 0x78787878u, (I / 4) % 4);
    const uint2 e = *bchk((const uint2*)((const char*)lut + off), lut, kLutBytes, err);
    hi = e.x;
    lo = e.y;
  } else if constexpr (KB == 3) {
    // the pair's 6 bits start at bit o of the 96 code bits: the field moved to
    // bit 8, masked, OR the lane's replica offset
    constexpr int o = 3 * I, wi = o / 32, b = o % 32;
    uint32_t v;
    if constexpr (b < 8) {
      v = c.w[wi] << (8 - b);
    } else if constexpr (b + 6 <= 32) {
      v = c.w[wi] >> (b - 8);
    } else {
      v = __funnelshift_r(c.w[wi], c.w[wi + 1], b - 8);
    }
    const uint2 e =
        *bchk((const uint2*)((const char*)lut + ((v & 0x3F00u) | lane8)), lut, kLutBytes, err);
    hi = e.x;
    lo = e.y;
  } else if constexpr (KB == 4) {
    // byte I/2 of the 128 code bits (word I/8, byte (I/2)%4) is the pair index
    // c_I | c_{I+1} << 4: the permute puts it in byte 1 and lane8 in byte 0
    const uint32_t off = __byte_perm(c.w[I / 8], lane8, 0x5504u | (((I / 2) % 4) << 4));
    const uint2 e = *bchk((const uint2*)((const char*)lut + off), lut, kLutBytes, err);
    hi = e.x;
    lo = e.y;
  } else {
    // bytes I, I+1 of the 256 code bits: word I/4, half (I/2)%2
    const uint32_t w = c.w[I / 4];
    const uint32_t e0 = *bchk((const uint32_t*)((const char*)lut + half_of((w << 2) & 0x03FC03FCu, (I / 2) % 2)), lut, kLutBytes, err);
    const uint32_t e1 = *bchk((const uint32_t*)((const char*)lut + half_of((w >> 6) & 0x03FC03FCu, (I / 2) % 2)), lut, kLutBytes, err);
    pack_hilo(e0, e1, hi, lo);
  }
}

// Scores of the chunk's 32 tokens: codes c[u] are token 8u + g.
// G = 8: columns are heads; m-tile mt has rows g / g+8 = tokens 16mt + g /
// 16mt + 8 + g, and the hi*hi, lo*hi and hi*lo products accumulate in
// separate chains (six independent chains of eight).
template <int KB, int KT>
__device__ __forceinline__ void score_ktile(const KCodes<KB> (&c)[4], const uint32_t* lut,
                                            uint32_t lane8, unsigned* err,
                                            const uint32_t (&bh)[8][2], const uint32_t (&bl)[8][2],
                                            float (&hh)[2][4], float (&lh)[2][4], float (&hl)[2][4]) {
#pragma unroll
  for (int mt = 0; mt < 2; ++mt) {
    uint32_t h0, l0, h1, l1, h2, l2, h3, l3;
    kpair<KB, 4 * KT>(c[2 * mt], lut, lane8, h0, l0, err);
    kpair<KB, 4 * KT>(c[2 * mt + 1], lut, lane8, h1, l1, err);
    kpair<KB, 4 * KT + 2>(c[2 * mt], lut, lane8, h2, l2, err);
    kpair<KB, 4 * KT + 2>(c[2 * mt + 1], lut, lane8, h3, l3, err);
    mma16816(hh[mt], h0, h1, h2, h3, bh[KT][0], bh[KT][1]);
    mma16816(lh[mt], l0, l1, l2, l3, bh[KT][0], bh[KT][1]);
    mma16816(hl[mt], h0, h1, h2, h3, bl[KT][0], bl[KT][1]);
  }
}

template <int KB, int KT>
__device__ __forceinline__ void score_all(const KCodes<KB> (&c)[4], const uint32_t* lut,
                                          uint32_t lane8, unsigned* err,
                                          const uint32_t (&bh)[8][2], const uint32_t (&bl)[8][2],
                                          float (&hh)[2][4], float (&lh)[2][4], float (&hl)[2][4]) {
  if constexpr (KT < 8) {
    score_ktile<KB, KT>(c, lut, lane8, err, bh, bl, hh, lh, hl);
    score_all<KB, KT + 1>(c, lut, lane8, err, bh, bl, hh, lh, hl);
  }
}

// G <= 4 ("folded"): the 8 MMA columns hold G heads twice, column 2h the
// query's hi part of head h and column 2h + 1 its lo part, and m-tile u holds
// token 8u + g twice: row g its K hi part, row g+8 its K lo part.  One MMA
// then yields hi*hi (row g, even columns), hi*lo (row g, odd), lo*hi (row
// g+8, even) and a negligible lo*lo, all of head tig in lane (g, tig), and
// each (hi pair, lo pair) table entry is the A operand pair (a0, a1) or
// (a2, a3) as loaded: 32 MMAs per chunk in four chains, against 48 in six.
template <int KB, int KT>
__device__ __forceinline__ void score_all_folded(const KCodes<KB> (&c)[4], const uint32_t* lut,
                                                 uint32_t lane8, unsigned* err,
                                                 const uint32_t (&bq)[8][2], float (&acc)[4][4]) {
  if constexpr (KT < 8) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      uint32_t h0, l0, h2, l2;
      kpair<KB, 4 * KT>(c[u], lut, lane8, h0, l0, err);
      kpair<KB, 4 * KT + 2>(c[u], lut, lane8, h2, l2, err);
      mma16816(acc[u], h0, l0, h2, l2, bq[KT][0], bq[KT][1]);
    }
    score_all_folded<KB, KT + 1>(c, lut, lane8, err, bq, acc);
  }
}

// Direct Sign: sum_i (2 bit_i - 1) q_rot,i for tokens ta, ta+8.  Bit i of
// the token's 128-bit sign vector belongs to rotated coordinate i, and the
// lane's 32 bits are coordinates 32 tig .. 32 tig + 31: the same k-index
// permutation as the key scores, so B is the query operand bh / bl (folded:
// bh alone, whose columns already carry both parts).
template <bool FOLD>
__device__ __forceinline__ void sign_scores(uint32_t sa, uint32_t sb, const uint32_t* slut,
                                            const uint32_t (&bh)[8][2],
                                            const uint32_t (&bl)[8][2], float (&d)[4],
                                            float (&dl)[4]) {
#pragma unroll
  for (int kt = 0; kt < 8; ++kt) {
    const uint32_t a0 = slut[(sa >> (4 * kt)) & 3u], a1 = slut[(sb >> (4 * kt)) & 3u];
    const uint32_t a2 = slut[(sa >> (4 * kt + 2)) & 3u], a3 = slut[(sb >> (4 * kt + 2)) & 3u];
    mma16816(d, a0, a1, a2, a3, bh[kt][0], bh[kt][1]);
    if constexpr (!FOLD) mma16816(dl, a0, a1, a2, a3, bl[kt][0], bl[kt][1]);
  }
}

// QJL: sum_j (2 bit_j - 1) (S q)_j for tokens ta, ta+8: A = exact +-1 signs,
// B = S q hi and lo from shared memory, k-tile-major so that a warp's 32
// lanes read contiguous words: unfolded, uint4 (b0 hi, b1 hi, b0 lo, b1 lo)
// at [kt][lane]; folded, the lane's part (hi or lo) as uint2 at [kt][lane].
template <bool FOLD>
__device__ __forceinline__ void qjl_scores(uint32_t sa, uint32_t sb, const uint32_t* slut,
                                           const void* qb, int lane, float (&d)[4],
                                           float (&dl)[4]) {
#pragma unroll
  for (int kt = 0; kt < 8; ++kt) {
    // sign bits 4kt, 4kt+1 (pair 0) and 4kt+2, 4kt+3 (pair 1) of this lane's 32
    const uint32_t a0 = slut[(sa >> (4 * kt)) & 3u], a1 = slut[(sb >> (4 * kt)) & 3u];
    const uint32_t a2 = slut[(sa >> (4 * kt + 2)) & 3u], a3 = slut[(sb >> (4 * kt + 2)) & 3u];
    if constexpr (FOLD) {
      const uint2 b = ((const uint2*)qb)[kt * 32 + lane];
      mma16816(d, a0, a1, a2, a3, b.x, b.y);
    } else {
      const uint4 b = ((const uint4*)qb)[kt * 32 + lane];
      mma16816(d, a0, a1, a2, a3, b.x, b.y);
      mma16816(dl, a0, a1, a2, a3, b.z, b.w);
    }
  }
}

// Bytes spanned by a decode step's new-token rows knew / vnew ([B][Hkv][.][d],
// element strides nsb, nsh), for the bounds-checked build.
__device__ __forceinline__ size_t new_rows_bytes(const DecodeArgs& a) {
  return (size_t)((long long)(a.B - 1) * a.nsb + (long long)(a.Hkv - 1) * a.nsh + kD2) *
         (a.new_f32 ? 4 : 2);
}

// Decode step in one launch (DecodeArgs::fused_step): the token L = T - 1 - W
// that leaves the window (with W = 0 the new token itself), handled by warp 0
// of its pair's first window split.  The warp reads L's rows (ring slot
// L mod W, bf16; with W = 0 the step's input), quantizes them into plane row L
// with the warp-per-vector quantizer of tq_append_kv (codes, norm and the
// key's residual term: Direct Sign bits and scale, or the QJL sketch and
// gamma), writes the new token T - 1 into the ring slot (W > 0), and returns
// L's dequantized key and value (lane l: coordinates 4l..4l+3) for the window
// split to attend to: the quantized splits of this launch stop before row L,
// so no CTA waits for another.  The codebooks' boundaries (2 KB), 32 words of
// packing scratch and 128 floats of residual scratch sit at byte scr of the
// dynamic shared memory.  Not inlined: it runs once per pair, off the main loop.
static __device__ __noinline__ void step_leaving_token(const DecodeArgs& a, long long pair, int L,
                                                       int scr, const float* kcen,
                                                       const float* vcen, float* kx, float* vx,
                                                       int lane) {
  extern __shared__ __align__(128) uint8_t smem[];
  const float* bnd = (const float*)(smem + scr);
  uint32_t* words = (uint32_t*)(smem + scr + 2048);
  float* rbuf = (float*)(smem + scr + 2048 + 128);
  const long long kr = pair * a.kcap + L, vr = pair * a.vcap + L;
  uint8_t* kc = (uint8_t*)a.kc + kr * 16 * a.kb;
  uint8_t* vc = (uint8_t*)a.vc + vr * 16 * a.vb;
  const long long ring = a.W > 0 ? (pair * a.W + L % a.W) * kD2 : 0;
  const long long noff = (pair / a.Hkv) * a.nsb + (pair % a.Hkv) * a.nsh;
  const size_t ring_bytes_ = (size_t)a.B * a.Hkv * a.W * kD2 * 2;
  const size_t nrow = (size_t)kD2 * (a.new_f32 ? 4 : 2);
  const uint8_t* kn_ = (const uint8_t*)a.knew + noff * (a.new_f32 ? 4 : 2);
  const uint8_t* vn_ = (const uint8_t*)a.vnew + noff * (a.new_f32 ? 4 : 2);
  if (!bchk_range(kc, 16 * a.kb, a.kc, (size_t)a.B * a.Hkv * a.kcap * 16 * a.kb, a.err) ||
      !bchk_range(vc, 16 * a.vb, a.vc, (size_t)a.B * a.Hkv * a.vcap * 16 * a.vb, a.err) ||
      !bchk_range(kn_, nrow, a.knew, new_rows_bytes(a), a.err) ||
      !bchk_range(vn_, nrow, a.vnew, new_rows_bytes(a), a.err) ||
      (a.W > 0 && !bchk_range(a.kwin + ring, kD2 * 2, a.kwin, ring_bytes_, a.err))) {
    for (int c = 0; c < 4; ++c) kx[c] = vx[c] = 0.f;
    return;
  }
  // the rows' loads first (with a window: the leaving token's key and value
  // and the new token's, for the ring), so that their latencies overlap
  float xk[4], xv[4];
  uint2 knw = make_uint2(0u, 0u), vnw = knw;
  if (a.W > 0) {
    const uint2 ko = ((const uint2*)(a.kwin + ring))[lane];
    const uint2 vo = ((const uint2*)(a.vwin + ring))[lane];
    knw = ((const uint2*)((const uint16_t*)a.knew + noff))[lane];
    vnw = ((const uint2*)((const uint16_t*)a.vnew + noff))[lane];
    xk[0] = bf16lo(ko.x); xk[1] = bf16hi(ko.x); xk[2] = bf16lo(ko.y); xk[3] = bf16hi(ko.y);
    xv[0] = bf16lo(vo.x); xv[1] = bf16hi(vo.x); xv[2] = bf16lo(vo.y); xv[3] = bf16hi(vo.y);
  } else if (a.new_f32) {
    const float4 ko = ((const float4*)((const float*)a.knew + noff))[lane];
    const float4 vo = ((const float4*)((const float*)a.vnew + noff))[lane];
    xk[0] = ko.x; xk[1] = ko.y; xk[2] = ko.z; xk[3] = ko.w;
    xv[0] = vo.x; xv[1] = vo.y; xv[2] = vo.z; xv[3] = vo.w;
  } else {
    const uint2 ko = ((const uint2*)((const uint16_t*)a.knew + noff))[lane];
    const uint2 vo = ((const uint2*)((const uint16_t*)a.vnew + noff))[lane];
    xk[0] = bf16lo(ko.x); xk[1] = bf16hi(ko.x); xk[2] = bf16lo(ko.y); xk[3] = bf16hi(ko.y);
    xv[0] = bf16lo(vo.x); xv[1] = bf16hi(vo.x); xv[2] = bf16lo(vo.y); xv[3] = bf16hi(vo.y);
  }
  const float4 sk = __ldg((const float4*)a.sk + lane), sv = __ldg((const float4*)a.sv + lane);
  const float sks[4] = {sk.x, sk.y, sk.z, sk.w}, svs_[4] = {sv.x, sv.y, sv.z, sv.w};
  float r[4], yq[4], t[4];
  // keys: quantize, then dequantize as a reader of the planes would (norm x
  // centroid plus the residual term; inverse rotation H / sqrt(d); signs)
  const float nk = warp_quantize_vals(xk, sk, a.kb, bnd, kcen, kc, (float*)a.kn + kr, words, lane,
                                      r, yq);
#pragma unroll
  for (int c = 0; c < 4; ++c) t[c] = nk * yq[c];
  if (a.dsign) {
    const float sc = warp_direct_sign(r, (uint8_t*)a.ks + kr * 16, (float*)a.kr + kr, lane);
#pragma unroll
    for (int c = 0; c < 4; ++c) t[c] += r[c] >= 0.f ? sc : -sc;
  } else if (a.qjl) {
    // residual estimate sqrt(pi/2) / m * gamma * S^T (2 bit - 1), coordinates 4l..4l+3
    uint32_t sb[4];
    const float gamma =
        warp_qjl_sketch(r, a.S, rbuf, (uint8_t*)a.ks + kr * 16, (float*)a.kr + kr, lane, sb);
    float e[4] = {0.f, 0.f, 0.f, 0.f};
    for (int j = 0; j < kQjlM; ++j) {
      const uint2 s4 = __ldg((const uint2*)(a.S + (size_t)j * kD2) + lane);
      const float sg = (sb[j >> 5] >> (j & 31)) & 1u ? 1.f : -1.f;
      e[0] = fmaf(sg, bf16lo(s4.x), e[0]);
      e[1] = fmaf(sg, bf16hi(s4.x), e[1]);
      e[2] = fmaf(sg, bf16lo(s4.y), e[2]);
      e[3] = fmaf(sg, bf16hi(s4.y), e[3]);
    }
    const float coef = 1.2533141373155003f / (float)kQjlM * gamma;   // sqrt(pi/2) / m
#pragma unroll
    for (int c = 0; c < 4; ++c) t[c] = fmaf(coef, e[c], t[c]);
  }
  warp_fwht4(t, lane);
#pragma unroll
  for (int c = 0; c < 4; ++c) kx[c] = t[c] * 0.08838834764831845f * sks[c];
  // values
  const float nv = warp_quantize_vals(xv, sv, a.vb, bnd + 256, vcen, vc, (float*)a.vn + vr, words,
                                      lane, r, yq);
#pragma unroll
  for (int c = 0; c < 4; ++c) t[c] = nv * yq[c];
  warp_fwht4(t, lane);
#pragma unroll
  for (int c = 0; c < 4; ++c) vx[c] = t[c] * 0.08838834764831845f * svs_[c];
  if (a.W > 0) {          // the new token into the slot (each lane rewrites the 8 bytes it read)
    ((uint2*)((uint16_t*)a.kwin + ring))[lane] = knw;
    ((uint2*)((uint16_t*)a.vwin + ring))[lane] = vnw;
  }
}

template <int G, int KB, int VB, int RES, bool SPARSE>
__global__ void __launch_bounds__(32 * decode_warps(G, KB, VB, RES),
                                  decode_ctas_per_sm(G, KB, VB, RES))
    decode_kernel(const DecodeArgs a) {
  constexpr int kDWarps = decode_warps(G, KB, VB, RES);   // warps of this CTA
  constexpr int kDT = kDWarps * 32;
  constexpr int KROW = 16 * KB, VROW = 16 * VB;
  __shared__ __align__(16) uint32_t lutk[256];   // K centroid tables (see kpair)
  __shared__ __align__(16) uint32_t lutv[256];   // V fp16 centroids (pairs for 2/3 bits)
  __shared__ uint32_t slut[4];                   // (+-1, +-1) fp16 pairs of two sign bits
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr bool QJL = RES == 1;        // QJL sketch of the key residual
  constexpr bool HAS_RES = RES != 0;
  // G <= 4 query heads leave half of the 8 MMA columns free: they carry the
  // query's lo part (see score_ktile)
  constexpr bool FOLD = G <= 4;
  constexpr DecodeSmem L(G, RES, KB, VB, kDWarps);
  float* qr = (float*)(smem + L.qr);
  float* qo = (float*)(smem + L.qo);
  float* svs = (float*)(smem + L.sv);
  int* is_last = (int*)(smem + L.total - 16);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // 1-D grid.  Several waves: the long quantized splits of every (sequence,
  // kv-head) first and the short window splits after them, so that CTAs start
  // longest first; one wave: each pair's splits together.
  int split, seq_head;
  {
    const int nq_total = a.B * a.Hkv * a.n_qsplits;
    const int i = (int)blockIdx.x;
    if (!a.long_first) {
      seq_head = i / a.n_splits;
      split = i - seq_head * a.n_splits;
    } else if (i < nq_total) {
      seq_head = i / a.n_qsplits;
      split = i - seq_head * a.n_qsplits;
    } else {
      const int nws = a.n_splits - a.n_qsplits;
      seq_head = (i - nq_total) / nws;
      split = a.n_qsplits + (i - nq_total - seq_head * nws);
    }
  }
  const int kvh = seq_head % a.Hkv, b = seq_head / a.Hkv;
  const int Hkv = a.Hkv;
  const uint32_t limit = a.wait_limit ? a.wait_limit : kDefaultWaitLimit;
  const int mg = lane >> 2, tig = lane & 3;   // MMA group / thread-in-group

  // A kernel launched after this one with programmatic dependent launch (the
  // next decode) may start its CTAs as soon as SMs free up and build its
  // tables while this grid's last CTAs merge; it still waits
  // (griddepcontrol.wait) for this grid to complete before it reads anything
  // this grid writes.  Only for one wave of one CTA per SM (a.pdl_trigger):
  // with two CTAs per SM or several waves, the early CTAs slowed this grid's
  // own (measured).
  if (a.pdl_trigger) asm volatile("griddepcontrol.launch_dependents;");

  // ------------------------------------------------------------- prologue
  // The codec tables are loaded and the lookup tables built before the
  // dependency wait; right after it come the loads of the sequence length and
  // the query, then the bulk copy of each warp's first chunk (before the
  // length has arrived), the query rotation overlaps the copies' flight, and
  // each warp's later chunks follow the CTA barrier of the query scale, so
  // that the first chunks of all warps are not queued behind them.
  __shared__ float cks[256], cvs[256];
  // fused decode step: the codebooks' boundaries and 32 words of packing
  // scratch after the dynamic shared memory (see step_leaving_token)
  constexpr int kScr = (L.total + 127) & ~127;
  if (a.fused_step) {
    float* qbnd = (float*)(smem + kScr);           // [2][256]
    for (int i = tid; i < 256; i += kDT) {
      qbnd[i] = __ldg(a.ck + 256 + i);
      qbnd[256 + i] = __ldg(a.cv + 256 + i);
    }
    if (tid < 32) ((uint32_t*)(smem + kScr + 2048))[tid] = 0u;
  }
  const int W = a.W;
  const bool window_split = split >= a.n_qsplits;
  constexpr int GW = (G + kDWarps - 1) / kDWarps;   // query heads rotated per warp
  for (int i = tid; i < 256; i += kDT) {
    cks[i] = i < (1 << KB) ? __ldg(a.ck + i) : 0.f;
    cvs[i] = i < (1 << VB) ? __ldg(a.cv + i) : 0.f;
  }
  if (tid < kD2) svs[tid] = __ldg(a.sv + tid);
  const float4 sk4 = __ldg((const float4*)a.sk + lane);
  uint8_t* wreg = smem + L.warps + warp * L.warp_stride;
  uint64_t* bar = (uint64_t*)(wreg + L.bar);
  constexpr int NS = ring_slots(KB, VB);
  if (lane == 0) {
#pragma unroll
    for (int i = 0; i < NS; ++i) mbar_init(bar + i, 1);
    fence_mbarrier_init();
  }
  __syncthreads();                                   // cks, cvs, svs
  // the shared lookup tables, built before the dependency wait so that they
  // overlap the previous kernel's tail (the tables buffer is written by the
  // host, never by a kernel on the stream)
  for (int i = tid; i < 256; i += kDT) {
    if constexpr (KB == 2) {
      if (i < 16) {
        uint32_t hp, lp;
        hilo2(cks[i & 3] * kCScale, cks[(i >> 2) & 3] * kCScale, hp, lp);
        lutk[2 * i] = hp;
        lutk[2 * i + 1] = lp;
      }
    } else if constexpr (KB == 3 || KB == 4) {
      // pair i = c_lo | c_hi << KB into the 16 key replicas of row i; at
      // step j lane l writes replica (l + j) % 16
      if (i < (1 << (2 * KB))) {
        constexpr int msk = (1 << KB) - 1;
        uint32_t hp, lp;
        hilo2(cks[i & msk] * kCScale, cks[i >> KB] * kCScale, hp, lp);
        uint2* row = (uint2*)(smem + L.lutk4) + i * 32;
#pragma unroll
        for (int j = 0; j < 16; ++j)
          *bchk(row + ((lane + j) & 15), smem + L.lutk4, L.warps - L.lutk4, a.err) =
              make_uint2(hp, lp);
      }
    } else {
      lutk[i] = hilo(cks[i] * kCScale);
    }
    if constexpr (VB == 2) {
      // value entry i of the pair table: (half2 of coordinate c, half2 of c + 2)
      // for the code byte i (see vmma_ktile), into replicas 16-31 of row i
      auto pe = [&](int n) {   // n = code of the first token | code of the second << 2
        return (h16(cvs[(n >> 2) & 3]) << 16) | h16(cvs[n & 3]);
      };
      const uint2 ve = make_uint2(pe(i & 15), pe(i >> 4));
      uint2* row = (uint2*)(smem + L.lutk4) + i * 32 + 16;
#pragma unroll
      for (int j = 0; j < 16; ++j)
        *bchk(row + ((lane + j) & 15), smem + L.lutk4, L.warps - L.lutk4, a.err) = ve;
    }
    uint32_t e;
    if constexpr (VB == 2 || VB == 3) {
      const int msk = (1 << VB) - 1;
      e = (h16(cvs[(i >> VB) & msk]) << 16) | h16(cvs[i & msk]);
    } else {
      e = h16(cvs[i]);
    }
    lutv[i] = e;
  }
  if (tid < 4) slut[tid] = ((tid & 2) ? 0x3C000000u : 0xBC000000u) | ((tid & 1) ? 0x3C00u : 0xBC00u);

  // this pair's plane rows and this split's first token
  const long long row0 = ((long long)b * Hkv + kvh);
  const uint8_t* kc = a.kc + row0 * a.kcap * KROW;
  const uint8_t* vc = a.vc + row0 * a.vcap * VROW;
  const float* knp = a.kn + row0 * a.kcap;
  const float* vnp = a.vn + row0 * a.vcap;
  const uint8_t* ksp = HAS_RES ? a.ks + row0 * a.kcap * 16 : nullptr;
  const float* krp = HAS_RES ? a.kr + row0 * a.kcap : nullptr;
  const int t_begin = split * a.split_tokens;
  // everything below may read what the previous kernel on the stream wrote
  // (sequence lengths, query, planes, window ring, workspace): wait for it
  // to finish
  asm volatile("griddepcontrol.wait;" ::: "memory");
  int T = *bchk(a.seq_lens + b, a.seq_lens, (size_t)a.B * 4, a.err) + a.step_new;
  // the query's loads go out before any bulk copy, so that they are not
  // queued behind the copies' burst
  const long long qbase = ((long long)b * a.Hq + (long long)kvh * G) * kD2;
  float qv[GW][4];
#pragma unroll
  for (int j = 0; j < GW; ++j) {
    const int g = warp + kDWarps * j;
    qv[j][0] = qv[j][1] = qv[j][2] = qv[j][3] = 0.f;
    if (g < G) {
      if (a.q_f32) {
        const float4 v = __ldg(bchk((const float4*)((const float*)a.q + qbase + g * kD2) + lane,
                                    a.q, (size_t)a.B * a.Hq * kD2 * 4, a.err));
        qv[j][0] = v.x; qv[j][1] = v.y; qv[j][2] = v.z; qv[j][3] = v.w;
      } else {
        const uint2 v = __ldg(bchk((const uint2*)((const uint16_t*)a.q + qbase + g * kD2) + lane,
                                   a.q, (size_t)a.B * a.Hq * kD2 * 2, a.err));
        qv[j][0] = bf16lo(v.x); qv[j][1] = bf16hi(v.x); qv[j][2] = bf16lo(v.y); qv[j][3] = bf16hi(v.y);
      }
    }
  }

  // rows c0 .. c0 + nv - 1 -> ring slot: codes by bulk copy; norms by bulk
  // copy when the 16-byte-rounded range stays inside the plane, else by plain
  // loads
  auto issue = [&](int c0, int slot, int nv) {
    const int n4 = (nv + 3) & ~3;
    // bulk copies need 16-byte aligned sources: the norm rows of a (sequence,
    // head) start at row0 * capacity floats, aligned only if capacity % 4 == 0
    // (chunks start at multiples of 32 tokens, so this holds for all or none)
    const bool norms_aligned = (((uintptr_t)knp | (uintptr_t)vnp |
                                 (HAS_RES ? (uintptr_t)krp : (uintptr_t)0)) & 15u) == 0;
    const bool bulk_norms =
        norms_aligned && (long long)c0 + n4 <= a.kcap && (long long)c0 + n4 <= a.vcap;
    uint8_t* kb_ = wreg + L.kbuf + slot * 32 * KROW;
    uint8_t* vb_ = wreg + L.vbuf + slot * 32 * VROW;
    float* kn_ = (float*)(wreg + L.kn + slot * 128);
    float* vn_ = (float*)(wreg + L.vn + slot * 128);
    if (!bulk_norms) {                     // warp-uniform
      if (lane < nv) {
        *bchk(kn_ + lane, kn_, 128, a.err) = *bchk(knp + c0 + lane, knp, (size_t)a.kcap * 4, a.err);
        *bchk(vn_ + lane, vn_, 128, a.err) = *bchk(vnp + c0 + lane, vnp, (size_t)a.vcap * 4, a.err);
        if constexpr (HAS_RES)
          *bchk((float*)(wreg + L.rn + slot * 128) + lane, wreg + L.rn + slot * 128, 128, a.err) =
              *bchk(krp + c0 + lane, krp, (size_t)a.kcap * 4, a.err);
      }
      __syncwarp();
    }
    if (lane == 0) {
      uint32_t bytes = nv * (KROW + VROW) + (bulk_norms ? 2 * n4 * 4 : 0);
      if constexpr (HAS_RES) bytes += nv * 16 + (bulk_norms ? n4 * 4 : 0);
      // a.extra_tx is a test hook: bytes that never arrive, so the wait on
      // this chunk can only end by running out of polls
      mbar_arrive_expect_tx(bar + slot, bytes + a.extra_tx);
      // a copy whose source leaves this pair's plane rows, or whose
      // destination leaves the slot, is dropped (bounds-checked build)
      auto copy = [&](void* dst, const void* dbase, size_t dbytes, const void* src,
                      const void* sbase, size_t sbytes, uint32_t n) {
        if (bchk_range(dst, n, dbase, dbytes, a.err) && bchk_range(src, n, sbase, sbytes, a.err))
          bulk_g2s(dst, src, n, bar + slot);
        else
          mbar_complete_tx(bar + slot, n);
      };
      copy(kb_, kb_, 32 * KROW, kc + (long long)c0 * KROW, kc, (size_t)a.kcap * KROW, nv * KROW);
      copy(vb_, vb_, 32 * VROW, vc + (long long)c0 * VROW, vc, (size_t)a.vcap * VROW, nv * VROW);
      if (bulk_norms) {
        copy(kn_, kn_, 128, knp + c0, knp, (size_t)a.kcap * 4, n4 * 4);
        copy(vn_, vn_, 128, vnp + c0, vnp, (size_t)a.vcap * 4, n4 * 4);
      }
      if constexpr (HAS_RES) {
        uint8_t* sdst = wreg + L.sbuf + slot * 512;
        copy(sdst, sdst, 512, ksp + (long long)c0 * 16, ksp, (size_t)a.kcap * 16, nv * 16);
        if (bulk_norms) {
          uint8_t* rdst = wreg + L.rn + slot * 128;
          copy(rdst, rdst, 128, krp + c0, krp, (size_t)a.kcap * 4, n4 * 4);
        }
      }
    }
  };
  // Each warp's first chunk of a quantized split goes in flight while the
  // sequence length is still on its way: 32 whole rows when they lie inside
  // the planes (rows past the split's last token are staged but never used:
  // their scores are masked and their value weights are zero).
  const int c_first = t_begin + 32 * warp;
  const bool spec0 =
      !window_split && (long long)c_first + 32 <= a.kcap && (long long)c_first + 32 <= a.vcap;
  if (spec0) issue(c_first, 0, 32);
  // a length outside the plan's range would read past this pair's plane rows
  // or ring: flag it and decode the sequence as empty
  if (T < 0 || T > a.max_seq_len) {
    if (tid == 0) atomicOr(a.err, kErrBounds);
    T = 0;
  }
  const int nq = T - W > 0 ? T - W : 0;
  // this split's token range (quantized splits); in a fused decode step the
  // window split takes row nq - 1, the token leaving the window
  int t_end = t_begin + a.split_tokens;
  if (t_end > nq - a.fused_step) t_end = nq - a.fused_step;
  auto rows_of = [&](int c0) { return t_end - c0 < 32 ? t_end - c0 : 32; };
  // a first chunk that reaches the planes' last rows goes in flight now, with
  // the rows the split holds; every warp's next NS - 2 chunks follow after the
  // CTA barrier below, so that the first chunks of all warps are not queued
  // behind the later ones
  if (!window_split && !spec0 && c_first < t_end) issue(c_first, 0, rows_of(c_first));

  // query rotation in registers: warp w rotates heads w (and w + 4), lane l
  // holds coordinates 4l .. 4l+3; two butterfly stages in the lane, five by shuffles
  float qmax = 0.f;
#pragma unroll
  for (int j = 0; j < GW; ++j) {
    const int g = warp + kDWarps * j;
    if (g < G) {
      float x[4];
      const float sgs[4] = {sk4.x, sk4.y, sk4.z, sk4.w};
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float v = qv[j][c] * a.qscale;
        *bchk(qo + (4 * lane + c) * G + g, qo, kD2 * G * 4, a.err) = v;
        x[c] = v * sgs[c];
      }
      warp_fwht4(x, lane);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float v = x[c] * 0.08838834764831845f;   // 1/sqrt(128)
        *bchk(qr + (4 * lane + c) * G + g, qr, kD2 * G * 4, a.err) = v;
        qmax = fmaxf(qmax, fabsf(v));
      }
    }
  }
  // power-of-two scale bringing max |q_rot| below 1 for the fp16 operands
  __shared__ float red[kDWarps];
  qmax = warp_max(qmax);
  if (lane == 0) red[warp] = qmax;
  __syncthreads();
  if (!window_split) {
#pragma unroll
    for (int j = 1; j < NS - 1; ++j) {
      const int c = t_begin + 32 * warp + 32 * kDWarps * j;
      if (c < t_end) issue(c, j, rows_of(c));
    }
  }
#pragma unroll
  for (int w = 0; w < kDWarps; ++w) qmax = fmaxf(qmax, red[w]);
  int qe = 0;
  (void)frexpf(qmax, &qe);
  const float qsp = qmax > 0.f ? ldexpf(1.f, -qe) : 1.f;
  // B operands (q hi/lo) of this lane, coordinates 32tig + 4kt + {0,1} / {2,3}:
  // unfolded, head mg in bh (hi) and bl (lo); folded, column mg is head mg / 2,
  // its hi part for even mg and its lo part for odd mg, all in bh
  const int qhead = FOLD ? (mg >> 1) : mg;
  uint32_t bh[8][2], bl[8][2];
#pragma unroll
  for (int kt = 0; kt < 8; ++kt) {
#pragma unroll
    for (int p = 0; p < 2; ++p) {
      uint32_t hp = 0u, lp = 0u;
      if (qhead < G) {
        const int c = 32 * tig + 4 * kt + 2 * p;
        hilo2(*bchk(qr + c * G + qhead, qr, kD2 * G * 4, a.err) * qsp,
              *bchk(qr + (c + 1) * G + qhead, qr, kD2 * G * 4, a.err) * qsp, hp, lp);
      }
      bh[kt][p] = FOLD && (mg & 1) ? lp : hp;
      bl[kt][p] = lp;
    }
  }
  float qsq = 1.f;                                   // scale of the S q operands
  if constexpr (QJL) {
    float* sq = (float*)(smem + L.sq);               // [G][m]
    float smax = 0.f;
    for (int j = tid; j < kQjlM; j += kDT) {
      float acc[G];
#pragma unroll
      for (int g = 0; g < G; ++g) acc[g] = 0.f;
      const uint4* Sj = (const uint4*)(a.S + (size_t)j * kD2);
#pragma unroll 2
      for (int c = 0; c < kD2 / 8; ++c) {
        const uint4 s8 = __ldg(Sj + c);
        const uint32_t sw[4] = {s8.x, s8.y, s8.z, s8.w};
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float sv = (u & 1) ? bf16hi(sw[u >> 1]) : bf16lo(sw[u >> 1]);
          const int k = 8 * c + u;
#pragma unroll
          for (int g = 0; g < G; ++g) acc[g] = fmaf(sv, qr[k * G + g], acc[g]);
        }
      }
#pragma unroll
      for (int g = 0; g < G; ++g) {
        *bchk(sq + g * kQjlM + j, sq, G * kQjlM * 4, a.err) = acc[g];
        smax = fmaxf(smax, fabsf(acc[g]));
      }
    }
    smax = warp_max(smax);
    __syncthreads();
    if (lane == 0) red[warp] = smax;
    __syncthreads();
#pragma unroll
    for (int w = 0; w < kDWarps; ++w) smax = fmaxf(smax, red[w]);
    int se = 0;
    (void)frexpf(smax, &se);
    qsq = smax > 0.f ? ldexpf(1.f, -se) : 1.f;
    // per k-tile, per lane: (b0 hi, b1 hi, b0 lo, b1 lo) of head lane/4 (folded:
    // head lane/8, and only the lane's part, hi for even lane/4), sketch
    // indices 32(lane%4) + 4kt + {0,1} / {2,3}
    for (int e = tid; e < 32 * 8; e += kDT) {
      const int kt = e / 32, ln = e % 32, g = FOLD ? ln >> 3 : ln >> 2, tg = ln & 3;
      uint4 o = make_uint4(0u, 0u, 0u, 0u);
      if (g < G) {
        const int c = 32 * tg + 4 * kt;
        const float4 s4q = *bchk((const float4*)(sq + g * kQjlM + c), sq, G * kQjlM * 4, a.err);
        hilo2(s4q.x * qsq, s4q.y * qsq, o.x, o.z);
        hilo2(s4q.z * qsq, s4q.w * qsq, o.y, o.w);
      }
      if constexpr (FOLD)
        *bchk((uint2*)(smem + L.qjlb) + e, smem + L.qjlb, 32 * 8 * 16, a.err) =
            ((ln >> 2) & 1) ? make_uint2(o.z, o.w) : make_uint2(o.x, o.y);
      else
        *bchk((uint4*)(smem + L.qjlb) + e, smem + L.qjlb, 32 * 8 * 16, a.err) = o;
    }
  }
  __syncthreads();

  // ------------------------------------------------------------- main loop
  float* cm = (float*)(smem + L.comb);   // [warps][G]      (merge area, after the loop)
  float* cl = cm + kDWarps * G;          // [warps][G]
  float* co = cl + kDWarps * G;          // [warps][G][128]
  constexpr size_t kCombBytes = (size_t)kDWarps * G * (2 + kD2) * 4;
  // bounds-checked accessors of the merge area (plain references otherwise)
  auto CM = [&](int i) -> float& { return *bchk(cm + i, cm, kCombBytes, a.err); };
  auto CL = [&](int i) -> float& { return *bchk(cl + i, cm, kCombBytes, a.err); };
  auto CO = [&](long long i) -> float& { return *bchk(co + i, cm, kCombBytes, a.err); };

  if (!window_split) {
    // online-softmax state: folded, of head tig (mfold, lfold); unfolded, of heads
    // 2tig, 2tig+1 (the accumulator columns)
    float mfold = kNegBig, lfold = 0.f;
    float m0 = kNegBig, m1 = kNegBig, l0 = 0.f, l1 = 0.f;
    float inv_d = 1.f;       // d holds the V sum divided by inv_d (a power of two)
    float scl = 1.f;         // folded path: fp16 weight scale (a power of two), inv_d = 1 / scl
    float vcap = 0.f;        // folded path: value-norm bound of the current weight scale
    float d[8][4];           // fp32 V-sum accumulators (MMA layout)
#pragma unroll
    for (int k = 0; k < 8; ++k)
#pragma unroll
      for (int j = 0; j < 4; ++j) d[k][j] = 0.f;
    const bool h0ok = 2 * tig < G, h1ok = 2 * tig + 1 < G;
    // the shared pair table: row p (256 bytes) holds 16 replicas of the key
    // pair entry p (bytes 0-127) and, for 2-bit values, 16 of the value entry p
    // (bytes 128-255); lane l reads replica l % 16, so a half-warp's 16
    // lookups hit 16 different bank pairs
    const uint8_t* ptab = smem + L.lutk4;
    const uint32_t* klut = KB == 3 || KB == 4 ? (const uint32_t*)ptab : lutk;
    const uint32_t lane8 = 8u * (uint32_t)(lane & 15);          // key replica offset
    const uint32_t laneV = 128u + 8u * (uint32_t)(lane & 15);   // value replica offset
    // [8 heads][16 pairs] fp16 weights: pair 8kt + j = tokens 16kt + j, 16kt + j + 8
    uint32_t* ws32 = (uint32_t*)(wreg + L.ws);
    const float kscale = 1.f / (kCScale * qsp);
    // residual-term scale: QJL sqrt(pi/2)/m over the S q operand scale;
    // Direct Sign 1 over the q operand scale
    const float res_scale = QJL ? 1.2533141373155003f / (float)kQjlM / qsq : 1.f / qsp;
    const void* qjlb = QJL ? (const void*)(smem + L.qjlb) : nullptr;

    int c0 = t_begin + 32 * warp;           // its copies were started in the prologue
    bool ok = true;
    int kq = 0;
    for (; c0 < t_end; c0 += 32 * kDWarps, ++kq) {
      const int slot = kq % NS;
      // the chunk NS - 1 ahead goes into the slot released at the end of the
      // previous iteration
      const int c1 = c0 + 32 * kDWarps * (NS - 1);
      if (c1 < t_end) issue(c1, (kq + NS - 1) % NS, rows_of(c1));
      ok = __all_sync(0xffffffffu, mbar_wait(bar + slot, (kq / NS) & 1, limit, a.err));
      if (!ok) break;
      const int nv = t_end - c0 < 32 ? t_end - c0 : 32;
      const uint8_t* kb_ = wreg + L.kbuf + slot * 32 * KROW;
      const float* kn_ = (const float*)(wreg + L.kn + slot * 128);
      const float* vn_ = (const float*)(wreg + L.vn + slot * 128);
      if constexpr (FOLD) {
        // value norms of this lane's tokens 8u + mg (u = 0..3; 0 past the end)
        float vn4[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
          vn4[u] = 8 * u + mg < nv ? *bchk(vn_ + 8 * u + mg, vn_, 128, a.err) : 0.f;
        // lazy weight scale: raised only when a norm exceeds the bound vcap
        float rs = 1.f;
        {
          const float nmax = fmaxf(fmaxf(vn4[0], vn4[1]), fmaxf(vn4[2], vn4[3]));
          if (__any_sync(0xffffffffu, nmax > vcap)) {
            const float wm = warp_max(nmax);
            // wm in [2^e, 2^(e+1)): vcap = 2^(e+1) and scl = 2^(6-e), so that
            // every weight p ||v|| scl (p <= 2^kLazyMax) stays below 2^15; the
            // exponent is clamped to [2^-60, 2^64] so that the accumulator, kept
            // in the current scale, stays finite
            const int be = (int)((__float_as_uint(wm) >> 23) & 0xFFu);
            int sexp = 133 - be;
            sexp = sexp > 64 ? 64 : sexp < -60 ? -60 : sexp;
            vcap = __int_as_float(((be < 253 ? be : 253) + 1) << 23);
            const float scl_new = __int_as_float((127 + sexp) << 23);
            rs = scl_new * inv_d;                    // a power of two, exact
            scl = scl_new;
            inv_d = __uint_as_float(0x7F000000u - __float_as_uint(scl));   // 1 / scl
          }
        }
        // ---- scores on the tensor cores: MMA column 2h is head h's query hi
        // part and column 2h + 1 its lo part, so lane (mg, tig) holds both
        // parts of head tig for the tokens of its rows.  m-tile u holds token
        // 8u + mg twice (row mg: K hi, row mg + 8: K lo), and
        //   score = hi*hi (acc[0]) + hi*lo (acc[1]) + lo*hi (acc[2])
        // (lo*lo, acc[3], is below fp32 rounding and dropped).
        float s4[4];
        {
          KCodes<KB> c[4];
#pragma unroll
          for (int r = 0; r < 4; ++r) load_kcodes<KB>(kb_, 8 * r + mg, tig, c[r], a.err);
          float acc[4][4];
#pragma unroll
          for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[u][j] = 0.f;
          score_all_folded<KB, 0>(c, klut, lane8, a.err, bh, acc);
#pragma unroll
          for (int u = 0; u < 4; ++u)
            s4[u] = (acc[u][0] + acc[u][1] + acc[u][2]) *
                    (*bchk(kn_ + 8 * u + mg, kn_, 128, a.err) * kscale);
        }
        if constexpr (HAS_RES) {
          // the residual MMA's rows are two tokens (16mt + mg, 16mt + mg + 8),
          // its columns the same hi / lo pairs
          const uint8_t* sb_ = wreg + L.sbuf + slot * 512;
          const float* rn_ = (const float*)(wreg + L.rn + slot * 128);
#pragma unroll
          for (int mt = 0; mt < 2; ++mt) {
            const int ta = 16 * mt + mg, tb = ta + 8;
            const uint32_t sa = *bchk((const uint32_t*)(sb_ + ta * 16 + 4 * tig), sb_, 512, a.err);
            const uint32_t sbits =
                *bchk((const uint32_t*)(sb_ + tb * 16 + 4 * tig), sb_, 512, a.err);
            float qa[4] = {0.f, 0.f, 0.f, 0.f}, ql[4] = {0.f, 0.f, 0.f, 0.f};
            if constexpr (QJL) qjl_scores<true>(sa, sbits, slut, qjlb, lane, qa, ql);
            else sign_scores<true>(sa, sbits, slut, bh, bl, qa, ql);
            s4[2 * mt] =
                fmaf(qa[0] + qa[1], *bchk(rn_ + ta, rn_, 128, a.err) * res_scale, s4[2 * mt]);
            s4[2 * mt + 1] = fmaf(qa[2] + qa[3], *bchk(rn_ + tb, rn_, 128, a.err) * res_scale,
                                  s4[2 * mt + 1]);
          }
        }
        // tokens past the end of a partial chunk get no weight; lanes of
        // absent heads (tig >= G) compute values that are never used
        if (nv < 32) {
#pragma unroll
          for (int u = 0; u < 4; ++u)
            if (8 * u + mg >= nv) s4[u] = kNegBig;
        }
        // ---- online softmax of head tig (log2 domain) with a lazy maximum:
        // mfold (uniform over the head's 8 lanes) is raised only when a score
        // exceeds it by more than kLazyMax (a warp vote), so the weights
        // p = 2^(s - mfold) are at most 2^kLazyMax and most chunks need no
        // reduction over lanes and no rescale
        const float smax = fmaxf(fmaxf(s4[0], s4[1]), fmaxf(s4[2], s4[3]));
        float al = 1.f, al0 = 1.f, al1 = 1.f;
        if (__any_sync(0xffffffffu, smax > mfold + kLazyMax)) {
          float x = smax;
#pragma unroll
          for (int o = 4; o < 32; o <<= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
          const float mn = fmaxf(mfold, x);
          al = ex2(mfold - mn);
          mfold = mn;
          // accumulator columns 2tig, 2tig + 1 are heads 2tig, 2tig + 1, whose
          // factors the score lanes of those heads hold
          al0 = __shfl_sync(0xffffffffu, al, 2 * tig);
          al1 = __shfl_sync(0xffffffffu, al, 2 * tig + 1);
        }
        float p[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) p[u] = ex2(s4[u] - mfold);
        lfold = fmaf(lfold, al, (p[0] + p[1]) + (p[2] + p[3]));
        bool skip_v = false;
        if constexpr (SPARSE)
          skip_v = warp_max(tig < G ? fmaxf(fmaxf(p[0], p[1]), fmaxf(p[2], p[3])) : 0.f) <
                   a.sparse_thr;
        // fp16 weights p ||v|| scl; pairs (tokens 8u + mg, 8u + 8 + mg) for u = 0, 2
        uint32_t pk[2];
#pragma unroll
        for (int kt = 0; kt < 2; ++kt) {
          const __half2 h = __floats2half2_rn(p[2 * kt] * (vn4[2 * kt] * scl),
                                              p[2 * kt + 1] * (vn4[2 * kt + 1] * scl));
          pk[kt] = *(const uint32_t*)&h;
        }
        // ---- rotated-domain V sum on the tensor cores: bring the accumulator
        // to the current maximum and scale first (rarely needed)
        const float2 pre = make_float2(al0 * rs, al1 * rs);
        if (__any_sync(0xffffffffu, pre.x != 1.f || pre.y != 1.f)) {
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const float2 lo = __fmul2_rn(make_float2(d[k][0], d[k][1]), pre);
            const float2 hi = __fmul2_rn(make_float2(d[k][2], d[k][3]), pre);
            d[k][0] = lo.x; d[k][1] = lo.y; d[k][2] = hi.x; d[k][3] = hi.y;
          }
        }
        // B operand of k-tile kt, lane (mg, tig): head mg's weight pairs
        // tig and tig + 4, i.e. tokens (16kt + tig, 16kt + tig + 8) and
        // (16kt + tig + 4, 16kt + tig + 12), packed by score lanes 4 tig + mg
        // and 4 (tig + 4) + mg
        const uint8_t* vb_ = wreg + L.vbuf + slot * 32 * VROW;
#pragma unroll
        for (int kt = 0; kt < 2; ++kt) {
          uint32_t b0 = __shfl_sync(0xffffffffu, pk[kt], 4 * tig + mg);
          uint32_t b1 = __shfl_sync(0xffffffffu, pk[kt], 4 * tig + mg + 16);
          if (mg >= G) b0 = b1 = 0u;
          if (!skip_v) vmma_ktile<VB>(vb_, lutv, ptab, laneV, kt, mg, tig, b0, b1, d, a.err);
        }
      } else {
      // ---- scores on the tensor cores: sc[mt][0,1] token 16mt+mg, sc[mt][2,3] token +8;
      //      columns 0 / 1 are heads 2tig / 2tig+1
      float sc[2][4];
      {
        KCodes<KB> c[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) load_kcodes<KB>(kb_, 8 * r + mg, tig, c[r], a.err);
        float hh[2][4], lh[2][4], hl[2][4];
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
          for (int j = 0; j < 4; ++j) hh[mt][j] = lh[mt][j] = hl[mt][j] = 0.f;
        score_all<KB, 0>(c, klut, lane8, a.err, bh, bl, hh, lh, hl);
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
          const int ta = 16 * mt + mg, tb = ta + 8;
          const float na = *bchk(kn_ + ta, kn_, 128, a.err) * kscale;
          const float nb = *bchk(kn_ + tb, kn_, 128, a.err) * kscale;
          sc[mt][0] = (hh[mt][0] + (lh[mt][0] + hl[mt][0])) * na;
          sc[mt][1] = (hh[mt][1] + (lh[mt][1] + hl[mt][1])) * na;
          sc[mt][2] = (hh[mt][2] + (lh[mt][2] + hl[mt][2])) * nb;
          sc[mt][3] = (hh[mt][3] + (lh[mt][3] + hl[mt][3])) * nb;
          if constexpr (HAS_RES) {
            const uint8_t* sb_ = wreg + L.sbuf + slot * 512;
            const float* rn_ = (const float*)(wreg + L.rn + slot * 128);
            const uint32_t sa = *bchk((const uint32_t*)(sb_ + ta * 16 + 4 * tig), sb_, 512, a.err);
            const uint32_t sbits =
                *bchk((const uint32_t*)(sb_ + tb * 16 + 4 * tig), sb_, 512, a.err);
            float qa[4] = {0.f, 0.f, 0.f, 0.f}, ql[4] = {0.f, 0.f, 0.f, 0.f};
            if constexpr (QJL) qjl_scores<false>(sa, sbits, slut, qjlb, lane, qa, ql);
            else sign_scores<false>(sa, sbits, slut, bh, bl, qa, ql);
            const float ga = *bchk(rn_ + ta, rn_, 128, a.err) * res_scale;
            const float gb = *bchk(rn_ + tb, rn_, 128, a.err) * res_scale;
            sc[mt][0] = fmaf(qa[0] + ql[0], ga, sc[mt][0]);
            sc[mt][1] = fmaf(qa[1] + ql[1], ga, sc[mt][1]);
            sc[mt][2] = fmaf(qa[2] + ql[2], gb, sc[mt][2]);
            sc[mt][3] = fmaf(qa[3] + ql[3], gb, sc[mt][3]);
          }
          // tokens past the end of a partial chunk get no weight; columns of
          // absent heads are never written or read back, so need no mask
          if (nv < 32) {
            if (ta >= nv) sc[mt][0] = sc[mt][1] = kNegBig;
            if (tb >= nv) sc[mt][2] = sc[mt][3] = kNegBig;
          }
        }
      }
      // ---- online softmax (log2 domain) per head column; reduce over mg.
      // (The lazy maxima of the folded path measured slower here: the
      // branches split the chunk's body, which the wider unfolded path needs
      // whole for its schedule.)
      float x0 = fmaxf(fmaxf(sc[0][0], sc[0][2]), fmaxf(sc[1][0], sc[1][2]));
      float x1 = fmaxf(fmaxf(sc[0][1], sc[0][3]), fmaxf(sc[1][1], sc[1][3]));
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, o));
        x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, o));
      }
      const float mn0 = fmaxf(m0, x0), mn1 = fmaxf(m1, x1);
      const float al0 = ex2(m0 - mn0), al1 = ex2(m1 - mn1);
      m0 = mn0;
      m1 = mn1;
      // fp16 weights scaled into range by a power of two: every weight
      // p ||v|| is at most the chunk's largest value norm (p <= 1), which maps
      // below 2^15; the exponent is clamped to [2^-60, 2^64] so that the
      // accumulator, kept in the latest chunk's scale, stays finite
      const float vmax = warp_max(lane < nv ? *bchk(vn_ + lane, vn_, 128, a.err) : 0.f);
      int sexp = 141 - (int)((__float_as_uint(vmax) >> 23) & 0xFFu);   // 14 - floor(log2 vmax)
      sexp = sexp > 64 ? 64 : sexp < -60 ? -60 : sexp;
      const float scl = __int_as_float((127 + sexp) << 23);
      float w[2][4];
      float ploc = 0.f, ps0 = 0.f, ps1 = 0.f;
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
        const int ta = 16 * mt + mg, tb = ta + 8;
        const float va = ta < nv ? *bchk(vn_ + ta, vn_, 128, a.err) * scl : 0.f;
        const float vb = tb < nv ? *bchk(vn_ + tb, vn_, 128, a.err) * scl : 0.f;
        const float p0 = ex2(sc[mt][0] - mn0), p1 = ex2(sc[mt][1] - mn1);
        const float p2 = ex2(sc[mt][2] - mn0), p3 = ex2(sc[mt][3] - mn1);
        ps0 += p0 + p2;
        ps1 += p1 + p3;
        if constexpr (SPARSE)
          ploc = fmaxf(ploc, fmaxf(h0ok ? fmaxf(p0, p2) : 0.f, h1ok ? fmaxf(p1, p3) : 0.f));
        w[mt][0] = p0 * va;
        w[mt][1] = p1 * va;
        w[mt][2] = p2 * vb;
        w[mt][3] = p3 * vb;
      }
      l0 = fmaf(l0, al0, ps0);
      l1 = fmaf(l1, al1, ps1);
      // sparse V: when every weight of the chunk is below the threshold
      // (relative to the running maximum), only the accumulator is rescaled
      bool skip_v = false;
      if constexpr (SPARSE) skip_v = warp_max(ploc) < a.sparse_thr;
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
        // tokens 16mt + mg and 16mt + mg + 8: weight pair 8mt + mg
        if (h0ok && !skip_v) {
          const __half2 h = __floats2half2_rn(w[mt][0], w[mt][2]);
          *bchk(ws32 + (2 * tig) * kWsStride + 8 * mt + mg, ws32, 8 * kWsStride * 4, a.err) =
              *(const uint32_t*)&h;
        }
        if (h1ok && !skip_v) {
          const __half2 h = __floats2half2_rn(w[mt][1], w[mt][3]);
          *bchk(ws32 + (2 * tig + 1) * kWsStride + 8 * mt + mg, ws32, 8 * kWsStride * 4, a.err) =
              *(const uint32_t*)&h;
        }
      }
      __syncwarp();
      // ---- rotated-domain V sum on the tensor cores: d holds the sum times
      // the current chunk's weight scale; rescale, then d += V^T W
      const float rs = skip_v ? 1.f : scl * inv_d;     // a power of two, exact
      if (!skip_v) inv_d = __uint_as_float(0x7F000000u - __float_as_uint(scl));   // 1 / scl
      const float2 pre = make_float2(al0 * rs, al1 * rs);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float2 lo = __fmul2_rn(make_float2(d[k][0], d[k][1]), pre);
        const float2 hi = __fmul2_rn(make_float2(d[k][2], d[k][3]), pre);
        d[k][0] = lo.x; d[k][1] = lo.y; d[k][2] = hi.x; d[k][3] = hi.y;
      }
      const uint8_t* vb_ = wreg + L.vbuf + slot * 32 * VROW;
#pragma unroll
      for (int kt = 0; kt < 2 && !skip_v; ++kt) {
        const uint32_t b0 =
            mg < G ? *bchk(ws32 + mg * kWsStride + 8 * kt + tig, ws32, 8 * kWsStride * 4, a.err) : 0u;
        const uint32_t b1 =
            mg < G ? *bchk(ws32 + mg * kWsStride + 8 * kt + tig + 4, ws32, 8 * kWsStride * 4, a.err)
                   : 0u;
        vmma_ktile<VB>(vb_, lutv, ptab, laneV, kt, mg, tig, b0, b1, d, a.err);
      }
      __syncwarp();
      }
    }
    {
      const float inv = inv_d;                    // back to the unscaled sum
#pragma unroll
      for (int k = 0; k < 8; ++k)
#pragma unroll
        for (int j = 0; j < 4; ++j) d[k][j] *= inv;
    }
    if (!ok) {
      // a staging wait ran out (error word set): wait for the copies still in
      // flight (chunks kq .. kq + NS - 1, one per ring slot) to land, each
      // wait bounded, then stop.  Under fault injection each barrier expects
      // a.extra_tx bytes that no copy delivers: retire them first, so that
      // the barrier completes exactly when the real copies have landed.
      for (int dd = 0; dd < NS; ++dd) {
        const int kk = kq + dd;
        if (t_begin + 32 * warp + kk * 32 * kDWarps >= t_end) break;
        if (lane == 0 && a.extra_tx != 0) mbar_complete_tx(bar + kk % NS, a.extra_tx);
        __syncwarp();
        for (uint32_t i = 0; i < limit && !mbar_try_wait(bar + kk % NS, (kk / NS) & 1); ++i) {
        }
      }
    }
    if (spec0 && c_first >= t_end) {
      // the first chunk went in flight before the length was known and holds
      // no token of this split: let it land (bounded wait) before the ring's
      // memory is reused
      if (lane == 0 && a.extra_tx != 0) mbar_complete_tx(bar, a.extra_tx);
      __syncwarp();
      for (uint32_t i = 0; i < limit && !mbar_try_wait(bar, 0); ++i) {
      }
    }
    // per-head l: sum over the 8 lanes of each column group
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      if constexpr (FOLD) {
        lfold += __shfl_xor_sync(0xffffffffu, lfold, o);
      } else {
        l0 += __shfl_xor_sync(0xffffffffu, l0, o);
        l1 += __shfl_xor_sync(0xffffffffu, l1, o);
      }
    }
    __syncthreads();                     // every warp is done with its ring buffers
    if constexpr (FOLD) {
      if (mg == 0 && tig < G) {
        CM(warp * G + tig) = mfold;
        CL(warp * G + tig) = lfold;
      }
    } else if (mg == 0) {
      if (h0ok) {
        CM(warp * G + 2 * tig) = m0;
        CL(warp * G + 2 * tig) = l0;
      }
      if (h1ok) {
        CM(warp * G + 2 * tig + 1) = m1;
        CL(warp * G + 2 * tig + 1) = l1;
      }
    }
    // thread (mg, tig): m-tile k rows mg, mg + 8 -> coordinates vrow_coord;
    // columns -> heads 2tig (+1)
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int c0 = vrow_coord<VB>(mg, k, 0), c1 = vrow_coord<VB>(mg, k, 1);
      if (h0ok) {
        const long long r = (long long)(warp * G + 2 * tig) * kD2;
        CO(r + c0) = d[k][0];
        CO(r + c1) = d[k][2];
      }
      if (h1ok) {
        const long long r = (long long)(warp * G + 2 * tig + 1) * kD2;
        CO(r + c0) = d[k][1];
        CO(r + c1) = d[k][3];
      }
    }
  } else {
    // residual window: tokens [T - nw, T) in slots t mod W, original domain
    float m[G], l[G], ow[G][4];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      m[g] = kNegBig;
      l[g] = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) ow[g][j] = 0.f;
    }
    const int nw = T < W ? T : W;                     // window tokens of this sequence
    const int tw0 = T - nw;
    const int kw0 = a.wsplit_tokens * (split - a.n_qsplits);   // this split's share
    const int kw1 = kw0 + a.wsplit_tokens < nw ? kw0 + a.wsplit_tokens : nw;
    const long long base = ((long long)b * Hkv + kvh) * W;
    // one token's key and value (lane l: coordinates 4l..4l+3, original
    // domain) into the warp's online softmax state
    auto attend = [&](const float (&kx)[4], const float (&vx)[4], int tpos) {
#pragma unroll
      for (int g = 0; g < G; ++g) {
        // several query tokens per sequence: column g is query token g % n_q
        // at position T - n_q + g % n_q, which sees tokens up to itself
        // (branch-free, so the per-column state stays in registers)
        const bool vis = tpos <= T - a.n_q + g % a.n_q;
        float part = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j)
          part = fmaf(*bchk(qo + (4 * lane + j) * G + g, qo, kD2 * G * 4, a.err), kx[j], part);
        const float s = warp_sum(part);
        const float mnew = vis ? fmaxf(m[g], s) : m[g];
        const float al = vis ? ex2(m[g] - mnew) : 1.f;
        const float p = vis ? ex2(s - mnew) : 0.f;
        l[g] = fmaf(l[g], al, p);
        m[g] = mnew;
#pragma unroll
        for (int j = 0; j < 4; ++j) ow[g][j] = fmaf(p, vx[j], ow[g][j] * al);
      }
    };
    // fused decode step: the new token T - 1 is read from the step's input (its
    // ring slot is written in this launch).  The pair's first window split also
    // takes the token leaving the window (row nq - 1, see step_leaving_token)
    // or, when none leaves (T <= W), writes the new token into slot T - 1,
    // which held none
    const uint16_t* knrow = nullptr;
    const uint16_t* vnrow = nullptr;
    if (a.fused_step && T >= 1) {
      const long long noff = (long long)b * a.nsb + (long long)kvh * a.nsh;
      knrow = (const uint16_t*)a.knew + noff;
      vnrow = (const uint16_t*)a.vnew + noff;
      // bounds-checked build: rows outside the step's input read its first row
      if (!bchk_range(knrow, kD2 * 2, a.knew, new_rows_bytes(a), a.err) ||
          !bchk_range(vnrow, kD2 * 2, a.vnew, new_rows_bytes(a), a.err)) {
        knrow = (const uint16_t*)a.knew;
        vnrow = (const uint16_t*)a.vnew;
      }
      if (split == a.n_qsplits && warp == 0) {
        if (nq > 0) {
          float kx[4], vx[4];
          step_leaving_token(a, (long long)b * Hkv + kvh, nq - 1, kScr, cks, cvs, kx, vx, lane);
          attend(kx, vx, nq - 1);
        } else {
          uint2* dk = (uint2*)(a.kwin + (base + T - 1) * kD2) + lane;
          uint2* dv = (uint2*)(a.vwin + (base + T - 1) * kD2) + lane;
          const size_t rb = (size_t)a.B * Hkv * W * kD2 * 2;
          if (bchk_range(dk, 8, a.kwin, rb, a.err) && bchk_range(dv, 8, a.vwin, rb, a.err)) {
            *dk = ((const uint2*)knrow)[lane];
            *dv = ((const uint2*)vnrow)[lane];
          }
        }
      }
    }
    // warp w takes window tokens w, w + warps, ...; 8 tokens' rows are loaded
    // before any is used, so the loads overlap instead of paying one latency
    // each.  Warp 0 of a split that took the leaving token takes none.
    const bool took = a.fused_step && T >= 1 && nq > 0 && split == a.n_qsplits;
    const int ww = took ? warp - 1 : warp, nww = took ? kDWarps - 1 : kDWarps;
    for (int k0 = kw0 + ww; ww >= 0 && k0 < kw1; k0 += 8 * nww) {
      uint2 kw[8], vw[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int k = k0 + u * nww;
        if (k < kw1) {
          const long long slotrow = (base + (tw0 + k) % W) * kD2;
          if (knrow != nullptr && tw0 + k == T - 1) {
            kw[u] = ((const uint2*)knrow)[lane];
            vw[u] = ((const uint2*)vnrow)[lane];
          } else {
            // this pair's W ring rows
            kw[u] = *bchk((const uint2*)(a.kwin + slotrow + 4 * lane), a.kwin + base * kD2,
                          (size_t)W * kD2 * 2, a.err);
            vw[u] = *bchk((const uint2*)(a.vwin + slotrow + 4 * lane), a.vwin + base * kD2,
                          (size_t)W * kD2 * 2, a.err);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (k0 + u * nww >= kw1) break;
        const float kx[4] = {bf16lo(kw[u].x), bf16hi(kw[u].x), bf16lo(kw[u].y), bf16hi(kw[u].y)};
        const float vx[4] = {bf16lo(vw[u].x), bf16hi(vw[u].x), bf16lo(vw[u].y), bf16hi(vw[u].y)};
        attend(kx, vx, tw0 + k0 + u * nww);
      }
    }
    __syncthreads();
#pragma unroll
    for (int g = 0; g < G; ++g) {
      if (lane == 0) {
        CM(warp * G + g) = m[g];
        CL(warp * G + g) = l[g];
      }
      *bchk((float4*)(co + (warp * G + g) * kD2 + 4 * lane), cm, kCombBytes, a.err) =
          make_float4(ow[g][0], ow[g][1], ow[g][2], ow[g][3]);
    }
  }

  // ------------------------------------------------------------- epilogue
  __syncthreads();
  const long long unit = (long long)b * Hkv + kvh;
  const int stride = kPartialStride;
  float* part = a.partials + (unit * a.n_splits + split) * G * stride;
  const size_t part_bytes = (size_t)a.B * Hkv * a.n_splits * G * stride * 4;
  auto PART = [&](int i) -> float& { return *bchk(part + i, a.partials, part_bytes, a.err); };
  // thread e of the G x 128 outputs: head e / 128, coordinate e % 128
  for (int e = tid; e < G * kD2; e += kDT) {
    const int g = e / kD2, c = e % kD2;
    float M = kNegBig;
#pragma unroll
    for (int w = 0; w < kDWarps; ++w) M = fmaxf(M, CM(w * G + g));
    float O = 0.f, Lsum = 0.f;
#pragma unroll
    for (int w = 0; w < kDWarps; ++w) {
      const float f = ex2(CM(w * G + g) - M);
      O = fmaf(CO((long long)(w * G + g) * kD2 + c), f, O);
      Lsum = fmaf(CL(w * G + g), f, Lsum);
    }
    PART(g * stride + 4 + c) = O;
    if (c == 0) {
      PART(g * stride) = M;
      PART(g * stride + 1) = Lsum;
    }
  }
  // the CTA's partial writes are ordered before the counter update by the
  // barrier and the update's release semantics (cumulative, gpu scope); its
  // acquire side orders the last CTA's reads of the other splits' partials
  __syncthreads();
  if (tid == 0) {
    unsigned prev;
    asm volatile("atom.add.acq_rel.gpu.u32 %0, [%1], 1;"
                 : "=r"(prev)
                 : "l"(bchk(a.counters + unit, a.counters, (size_t)a.B * Hkv * 4, a.err))
                 : "memory");
    *is_last = prev == (unsigned)(a.n_splits - 1);
  }
  __syncthreads();
  if (!*is_last) return;

  // last CTA of this (sequence, kv-head): every warp takes a share of the
  // merge.  Head g gets WH = kDWarps / G warps (at least one); warp k of the
  // head merges splits k, k + WH, ... in one pass with online rescaling
  // (lane s holds (m, l) of the batch's split s, every lane its 4 coordinates
  // of every row; NB rows in flight per batch).  Rows of quantized splits are
  // rotated-domain sums, rows of window splits original-domain sums: two
  // accumulators.  The WH warps of a head then combine through shared memory,
  // and the head's first warp inverse-rotates (R^T = D_s H / sqrt(d)) in
  // registers and writes the output.
  constexpr int WH = kDWarps / G > 0 ? kDWarps / G : 1;    // warps per head
  constexpr int NB = WH == 1 ? 32 : 8;                       // split rows per batch
  const float* base = a.partials + unit * a.n_splits * G * stride;
  float* mres = (float*)(smem + L.comb);     // [kDWarps][M, L, pad, pad, rot[128], win[128]]
  constexpr int kMres = 4 + 2 * kD2;
  auto MR = [&](int i) -> float& {
    return *bchk(mres + i, mres, (size_t)kDWarps * kMres * 4, a.err);
  };
  for (int g0 = warp / WH; g0 < G; g0 += kDWarps / WH) {
    const int g = g0, k = warp % WH;
    float M = kNegBig, Lsum = 0.f;
    float4 rot = make_float4(0.f, 0.f, 0.f, 0.f), win = rot;
    for (int s0 = k; s0 < a.n_splits; s0 += WH * NB) {
      const int sl = s0 + WH * lane;                // this lane's (m, l) row
      const bool lv = lane < NB && sl < a.n_splits;
      const float* pl = bchk(base + (lv ? sl : 0) * G * stride + g * stride, a.partials,
                             part_bytes, a.err);
      const float ml = lv ? __ldcg(pl) : kNegBig;
      const float ll = lv ? __ldcg(pl + 1) : 0.f;
      float4 v[NB];
#pragma unroll
      for (int u = 0; u < NB; ++u) {
        const int su = s0 + WH * u;
        v[u] = su < a.n_splits
                   ? __ldcg(bchk((const float4*)(base + (su * G + g) * stride + 4) + lane,
                                 a.partials, part_bytes, a.err))
                   : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      const float Mn = fmaxf(M, warp_max(ml));
      const float r = ex2(M - Mn);
      const float fl = ex2(ml - Mn);
      Lsum = fmaf(Lsum, r, warp_sum(ll * fl));
      rot = make_float4(rot.x * r, rot.y * r, rot.z * r, rot.w * r);
      win = make_float4(win.x * r, win.y * r, win.z * r, win.w * r);
#pragma unroll
      for (int u = 0; u < NB; ++u) {
        const float f = __shfl_sync(0xffffffffu, fl, u);
        const bool q = s0 + WH * u < a.n_qsplits;
        const float fq = q ? f : 0.f, fw = q ? 0.f : f;
        rot.x = fmaf(v[u].x, fq, rot.x);
        rot.y = fmaf(v[u].y, fq, rot.y);
        rot.z = fmaf(v[u].z, fq, rot.z);
        rot.w = fmaf(v[u].w, fq, rot.w);
        win.x = fmaf(v[u].x, fw, win.x);
        win.y = fmaf(v[u].y, fw, win.y);
        win.z = fmaf(v[u].z, fw, win.z);
        win.w = fmaf(v[u].w, fw, win.w);
      }
      M = Mn;
    }
    if constexpr (WH > 1) {
      if (lane == 0) {
        MR(warp * kMres) = M;
        MR(warp * kMres + 1) = Lsum;
      }
      *bchk((float4*)(mres + warp * kMres + 4) + lane, mres, (size_t)kDWarps * kMres * 4, a.err) = rot;
      *bchk((float4*)(mres + warp * kMres + 4 + kD2) + lane, mres, (size_t)kDWarps * kMres * 4,
            a.err) = win;
    }
    if constexpr (WH == 1) {
      // one warp per head: no combine step
      float x[4] = {rot.x, rot.y, rot.z, rot.w};
      warp_fwht4(x, lane);
      const float4 sv4 = *(const float4*)(svs + 4 * lane);
      const float rr = 0.08838834764831845f;
      const float inv = Lsum > 0.f ? 1.0f / Lsum : 0.f;
      const float4 res = make_float4((x[0] * rr * sv4.x + win.x) * inv, (x[1] * rr * sv4.y + win.y) * inv,
                                     (x[2] * rr * sv4.z + win.z) * inv, (x[3] * rr * sv4.w + win.w) * inv);
      *bchk((float4*)(a.out + ((long long)b * a.Hq + (long long)kvh * G + g) * kD2 + 4 * lane), a.out,
            (size_t)a.B * a.Hq * kD2 * 4, a.err) = res;
    }
  }
  if constexpr (WH > 1) {
    __syncthreads();
    // the first warp of each head combines its head's WH partial merges
    if (warp % WH == 0 && warp / WH < G) {
      const int g = warp / WH;
      float M = kNegBig;
#pragma unroll
      for (int k = 0; k < WH; ++k) M = fmaxf(M, MR((warp + k) * kMres));
      float Lsum = 0.f;
      float4 rot = make_float4(0.f, 0.f, 0.f, 0.f), win = rot;
#pragma unroll
      for (int k = 0; k < WH; ++k) {
        const float f = ex2(MR((warp + k) * kMres) - M);
        Lsum = fmaf(MR((warp + k) * kMres + 1), f, Lsum);
        const float4 rk = *bchk((const float4*)(mres + (warp + k) * kMres + 4) + lane, mres,
                                (size_t)kDWarps * kMres * 4, a.err);
        const float4 wk = *bchk((const float4*)(mres + (warp + k) * kMres + 4 + kD2) + lane, mres,
                                (size_t)kDWarps * kMres * 4, a.err);
        rot = make_float4(fmaf(rk.x, f, rot.x), fmaf(rk.y, f, rot.y), fmaf(rk.z, f, rot.z),
                          fmaf(rk.w, f, rot.w));
        win = make_float4(fmaf(wk.x, f, win.x), fmaf(wk.y, f, win.y), fmaf(wk.z, f, win.z),
                          fmaf(wk.w, f, win.w));
      }
      // butterfly over 128 values, 4 per lane (coordinates 4*lane .. 4*lane+3)
      float x[4] = {rot.x, rot.y, rot.z, rot.w};
      warp_fwht4(x, lane);
      const float4 sv4 = *(const float4*)(svs + 4 * lane);
      const float rr = 0.08838834764831845f;
      const float inv = Lsum > 0.f ? 1.0f / Lsum : 0.f;
      const float4 res = make_float4((x[0] * rr * sv4.x + win.x) * inv, (x[1] * rr * sv4.y + win.y) * inv,
                                     (x[2] * rr * sv4.z + win.z) * inv, (x[3] * rr * sv4.w + win.w) * inv);
      *bchk((float4*)(a.out + ((long long)b * a.Hq + (long long)kvh * G + g) * kD2 + 4 * lane), a.out,
            (size_t)a.B * a.Hq * kD2 * 4, a.err) = res;
    }
  }
  if (tid == 0)   // leave the counter ready for the next call
    *bchk(a.counters + unit, a.counters, (size_t)a.B * Hkv * 4, a.err) = 0u;
}


template <int G, int KB, int VB, int RES, bool SPARSE = false>
int launch_decode_t(const DecodeArgs& a, cudaStream_t s) {
  auto k = decode_kernel<G, KB, VB, RES, SPARSE>;
  constexpr int kWarps = decode_warps(G, KB, VB, RES);
  const size_t base = (size_t)DecodeSmem(G, RES, KB, VB, kWarps).total;
  const size_t smem = base + (a.fused_step ? kFusedScratchBytes : 0);
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)(base + kFusedScratchBytes)) != cudaSuccess)
    return 1;
  // programmatic dependent launch: the CTAs may start while the previous
  // kernel on the stream is still running; they read only the codec tables
  // before griddepcontrol.wait
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((long long)a.n_splits * a.Hkv * a.B), 1, 1);
  cfg.blockDim = dim3(32 * kWarps, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, k, a) != cudaSuccess) return 1;
  return cudaGetLastError() != cudaSuccess;
}

// Dispatch over (KB, VB, key residual) for one G; defined once per G
// translation unit.  Keys with a residual term (QJL, Direct Sign) use 2-4 bit codes.
template <int G>
int launch_decode_g(const DecodeArgs& a, cudaStream_t s) {
#define TQ_VB_CASES(KB_, RES_)                                               \
  switch (a.vb) {                                                          \
    case 2: return launch_decode_t<G, KB_, 2, RES_>(a, s);                 \
    case 3: return launch_decode_t<G, KB_, 3, RES_>(a, s);                 \
    case 4: return launch_decode_t<G, KB_, 4, RES_>(a, s);                 \
    case 8: return launch_decode_t<G, KB_, 8, RES_>(a, s);                 \
  }                                                                        \
  return 1;
  if (a.qjl || a.dsign) {
    if (a.qjl) {
      switch (a.kb) {
        case 2: { TQ_VB_CASES(2, 1) }
        case 3: { TQ_VB_CASES(3, 1) }
        case 4: { TQ_VB_CASES(4, 1) }
      }
    } else {
      switch (a.kb) {
        case 2: { TQ_VB_CASES(2, 2) }
        case 3: { TQ_VB_CASES(3, 2) }
        case 4: { TQ_VB_CASES(4, 2) }
      }
    }
    return 1;
  }
  if (a.sparse_thr > 0.f) {
#define TQ_VB_SPARSE(KB_)                                                    \
  switch (a.vb) {                                                          \
    case 2: return launch_decode_t<G, KB_, 2, 0, true>(a, s);              \
    case 3: return launch_decode_t<G, KB_, 3, 0, true>(a, s);              \
    case 4: return launch_decode_t<G, KB_, 4, 0, true>(a, s);              \
    case 8: return launch_decode_t<G, KB_, 8, 0, true>(a, s);              \
  }                                                                        \
  return 1;
    switch (a.kb) {
      case 2: { TQ_VB_SPARSE(2) }
      case 3: { TQ_VB_SPARSE(3) }
      case 4: { TQ_VB_SPARSE(4) }
      case 8: { TQ_VB_SPARSE(8) }
    }
#undef TQ_VB_SPARSE
    return 1;
  }
  switch (a.kb) {
    case 2: { TQ_VB_CASES(2, 0) }
    case 3: { TQ_VB_CASES(3, 0) }
    case 4: { TQ_VB_CASES(4, 0) }
    case 8: { TQ_VB_CASES(8, 0) }
  }
#undef TQ_VB_CASES
  return 1;
}

}  // namespace tq
