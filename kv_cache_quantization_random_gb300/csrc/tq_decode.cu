// Decode attention over a TurboQuant-compressed KV cache (sm_103a).
//
// "TurboQuant KV 캐시 압축 for llama.cpp": v1.7.0 decision 4 (the decode kernel
// applies the encoders' WHT to Q, so q_rot . k_rot = q . k by Parseval);
// v1.5.2 changes 1-2 (accumulate in fp32, never half) and 4 (V is summed in
// the rotated domain and needs one inverse rotation at the output); v1.4.2
// item 2 and the v1.5.2 sharpening text (the QJL term is a scalar correction
// from the sign bits and the stored residual scale).
//
// One CTA = (split, kv-head, sequence).  Prologue: load the G query heads that
// share the kv-head, fold in softmax_scale * log2(e), rotate them with the K
// sign vector (smem butterfly), load both centroid tables; QJL keys also get a
// byte-indexed table of signed partial sums of S q_rot.  Main loop: each warp
// streams 32-token chunks of packed codes and norms into a double-buffered
// shared-memory ring with cp.async; lane t scores token t against all G heads
// through the K centroid table (no dequantized K ever reaches memory), the warp
// runs an online softmax in the log2 domain, then lane l accumulates the
// rotated-domain V sum for coordinates 4l..4l+3.  The split that owns the
// residual window scores the bf16 window tokens in the original domain.
// Epilogue: warps merge by log-sum-exp, the CTA writes (m, l, o) for its split;
// the last CTA of the (sequence, kv-head) merges every split, inverse-rotates
// the rotated part with the V sign vector, adds the window part and writes out.
#include <cuda_runtime.h>
#include <stdint.h>

#include "tq_device.cuh"

namespace tq {

__device__ unsigned g_decode_err;

constexpr int kDT = kDecodeWarps * 32;   // threads per decode CTA
constexpr int kD2 = 128;
constexpr float kNegBig = -1.0e30f;

struct DecodeSmem {
  int qr, qo, lutk, lutv, sv, tbl, warps, warp_stride;
  int kbuf, vbuf, kn, vn, sbuf, rn, ws;   // offsets inside one warp's region
  int comb, total;
  __host__ __device__ DecodeSmem(int G, int qjl, int pk, int pv) {
    int off = 0;
    qr = off; off += kD2 * G * 4;
    qo = off; off += kD2 * G * 4;
    lutk = off; off += 256 * 4;
    lutv = off; off += 256 * 4;
    sv = off; off += kD2 * 4;
    tbl = off; off += qjl ? 16 * 256 * G * 4 : 0;
    warps = off;
    int w = 0;
    kbuf = w; w += 2 * 32 * pk;
    vbuf = w; w += 2 * 32 * pv;
    kn = w; w += 2 * 32 * 4;
    vn = w; w += 2 * 32 * 4;
    sbuf = w; w += qjl ? 2 * 32 * 16 : 0;
    rn = w; w += qjl ? 2 * 32 * 4 : 0;
    ws = w; w += 32 * G * 4;
    warp_stride = w;
    int region = kDecodeWarps * w;
    int comb_need = kDecodeWarps * G * (2 + kD2) * 4;
    int scratch_need = 2 * G * kD2 * 4;
    if (region < comb_need) region = comb_need;
    if (region < scratch_need) region = scratch_need;
    comb = warps;            // aliases the warp regions after the main loop
    off += region;
    total = off + 16;        // + is_last flag
  }
};

size_t decode_smem_bytes(int G, int kb, int vb, int qjl, int pk, int pv) {
  (void)kb;
  (void)vb;
  return (size_t)DecodeSmem(G, qjl, pk, pv).total;
}

template <int G>
__device__ __forceinline__ void load_vec(const float* p, float (&v)[G]) {
  if constexpr (G == 1) {
    v[0] = p[0];
  } else if constexpr (G == 2) {
    float2 t = *(const float2*)p;
    v[0] = t.x; v[1] = t.y;
  } else {
#pragma unroll
    for (int k = 0; k < G; k += 4) {
      float4 t = *(const float4*)(p + k);
      v[k] = t.x; v[k + 1] = t.y; v[k + 2] = t.z; v[k + 3] = t.w;
    }
  }
}

// Phase A: score of this lane's token against the G heads, through the K table.
template <int KB, int G, bool QJL>
__device__ __forceinline__ void score_token(const uint8_t* krow, const float* qr, const float* lutk,
                                            float kn, const uint8_t* srow, float rn,
                                            const float* tbl, float (&s)[G]) {
  constexpr int NW = 4 * KB;
  uint32_t w[NW];
#pragma unroll
  for (int c = 0; c < KB; ++c) {
    uint4 t = lds128(krow + 16 * c);
    w[4 * c] = t.x; w[4 * c + 1] = t.y; w[4 * c + 2] = t.z; w[4 * c + 3] = t.w;
  }
  float acc[G];
#pragma unroll
  for (int g = 0; g < G; ++g) acc[g] = 0.f;
#pragma unroll
  for (int i = 0; i < kD2; ++i) {
    constexpr uint32_t mask = (1u << KB) - 1u;
    const int p = i * KB;
    uint32_t code = w[p >> 5] >> (p & 31);
    if ((p & 31) + KB > 32) code |= w[(p >> 5) + 1] << (32 - (p & 31));
    const float c = lutk[code & mask];
    float qv[G];
    load_vec<G>(qr + i * G, qv);
#pragma unroll
    for (int g = 0; g < G; ++g) acc[g] = fmaf(c, qv[g], acc[g]);
  }
#pragma unroll
  for (int g = 0; g < G; ++g) s[g] = acc[g] * kn;
  if constexpr (QJL) {
    uint4 sb = lds128(srow);
    const uint32_t sw[4] = {sb.x, sb.y, sb.z, sb.w};
    float qa[G];
#pragma unroll
    for (int g = 0; g < G; ++g) qa[g] = 0.f;
#pragma unroll
    for (int p = 0; p < 16; ++p) {
      const uint32_t byte = (sw[p >> 2] >> (8 * (p & 3))) & 0xFFu;
      float tv[G];
      load_vec<G>(tbl + ((p << 8) | byte) * G, tv);
#pragma unroll
      for (int g = 0; g < G; ++g) qa[g] += tv[g];
    }
#pragma unroll
    for (int g = 0; g < G; ++g) s[g] = fmaf(rn, qa[g], s[g]);
  }
}

// Phase C: this lane's 4 coordinates of the rotated-domain V sum over nv tokens.
template <int VB, int G>
__device__ __forceinline__ void vsum_chunk(const uint8_t* vbuf, int pv, const float* ws,
                                           const float* lutv, int nv, int lane,
                                           float (&o)[G][4]) {
  constexpr uint32_t mask = (1u << VB) - 1u;
  for (int t = 0; t < nv; ++t) {
    const uint8_t* row = vbuf + t * pv;
    uint32_t bits;
    if constexpr (VB == 2) {
      bits = row[lane];
    } else if constexpr (VB == 4) {
      bits = *(const uint16_t*)(row + 2 * lane);
    } else if constexpr (VB == 8) {
      bits = *(const uint32_t*)(row + 4 * lane);
    } else {   // VB == 3: 12 bits at bit 12*lane of a 48-byte row
      const int bo = 12 * lane;
      const int wi = bo >> 5, sh = bo & 31;
      const uint32_t* rw = (const uint32_t*)row;
      const uint32_t lo = rw[wi];
      const uint32_t hi = rw[wi + 1 < 12 ? wi + 1 : 11];
      bits = (uint32_t)((((uint64_t)hi << 32) | lo) >> sh);
    }
    float c[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) c[j] = lutv[(bits >> (VB * j)) & mask];
    float wv[G];
    load_vec<G>(ws + t * G, wv);
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int j = 0; j < 4; ++j) o[g][j] = fmaf(wv[g], c[j], o[g][j]);
  }
}

template <int G, bool QJL>
__global__ void __launch_bounds__(kDT) decode_kernel(const DecodeArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const DecodeSmem L(G, QJL ? 1 : 0, a.pk, a.pv);
  float* qr = (float*)(smem + L.qr);
  float* qo = (float*)(smem + L.qo);
  float* lutk = (float*)(smem + L.lutk);
  float* lutv = (float*)(smem + L.lutv);
  float* svs = (float*)(smem + L.sv);
  float* tbl = (float*)(smem + L.tbl);
  int* is_last = (int*)(smem + L.total - 16);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int Hkv = a.Hkv;

  // ------------------------------------------------------------- prologue
  for (int i = tid; i < 256; i += kDT) {
    lutk[i] = a.ck[i];
    lutv[i] = a.cv[i];
  }
  svs[tid] = a.sv[tid];
  float* scratch = (float*)(smem + L.warps);        // [G][128], aliases warp buffers
  {
    const long long qbase = ((long long)b * a.Hq + (long long)kvh * G) * kD2;
    for (int e = tid; e < G * kD2; e += kDT) {
      const int g = e / kD2, i = e % kD2;
      float v = a.q_f32 ? ((const float*)a.q)[qbase + e]
                        : __uint_as_float((uint32_t)((const uint16_t*)a.q)[qbase + e] << 16);
      v *= a.qscale;
      qo[i * G + g] = v;
      scratch[g * kD2 + i] = v * a.sk[i];
    }
  }
  __syncthreads();
  for (int h = 1; h < kD2; h <<= 1) {               // butterfly, Sylvester order
    for (int e = tid; e < G * (kD2 / 2); e += kDT) {
      const int g = e / (kD2 / 2), r = e % (kD2 / 2);
      const int i = (r / h) * 2 * h + (r % h);
      float* x = scratch + g * kD2;
      const float u = x[i], v = x[i + h];
      x[i] = u + v;
      x[i + h] = u - v;
    }
    __syncthreads();
  }
  for (int e = tid; e < G * kD2; e += kDT) {
    const int g = e / kD2, i = e % kD2;
    qr[i * G + g] = scratch[e] * 0.08838834764831845f;   // 1/sqrt(128)
  }
  __syncthreads();
  if constexpr (QJL) {
    // sq[g][j] = sum_k S[j][k] q_rot[g][k];  table[p][byte][g] = coef * sum_bits +-sq
    float* sq = scratch;                                   // [G][m]
    for (int j = tid; j < kQjlM; j += kDT) {
      float acc[G];
#pragma unroll
      for (int g = 0; g < G; ++g) acc[g] = 0.f;
      const uint16_t* Sj = a.S + (size_t)j * kD2;
      for (int k = 0; k < kD2; ++k) {
        const float s = __uint_as_float((uint32_t)Sj[k] << 16);
#pragma unroll
        for (int g = 0; g < G; ++g) acc[g] = fmaf(s, qr[k * G + g], acc[g]);
      }
#pragma unroll
      for (int g = 0; g < G; ++g) sq[g * kQjlM + j] = acc[g];
    }
    __syncthreads();
    const float coef = 1.2533141373155003f / (float)kQjlM;   // sqrt(pi/2) / m
    for (int e = tid; e < 16 * 256; e += kDT) {
      const int p = e >> 8, byte = e & 255;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float acc = 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const float v = sq[g * kQjlM + 8 * p + k];
          acc += ((byte >> k) & 1) ? v : -v;
        }
        tbl[e * G + g] = coef * acc;
      }
    }
    __syncthreads();
  }

  // ------------------------------------------------------------- main loop
  const int T = a.seq_lens[b];
  const int W = a.W;
  const int nq = T - W > 0 ? T - W : 0;
  float m[G], l[G], o[G][4];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    m[g] = kNegBig;
    l[g] = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) o[g][j] = 0.f;
  }
  uint8_t* wreg = smem + L.warps + warp * L.warp_stride;
  float* ws = (float*)(wreg + L.ws);

  if (split < a.n_qsplits) {
    const int t_begin = split * a.split_tokens;
    int t_end = t_begin + a.split_tokens;
    if (t_end > nq) t_end = nq;
    const long long row0 = ((long long)b * Hkv + kvh);
    const uint8_t* kc = a.kc + row0 * a.kcap * (16 * a.kb);
    const uint8_t* vc = a.vc + row0 * a.vcap * (16 * a.vb);
    const float* knp = a.kn + row0 * a.kcap;
    const float* vnp = a.vn + row0 * a.vcap;
    const uint8_t* ksp = QJL ? a.ks + row0 * a.kcap * 16 : nullptr;
    const float* krp = QJL ? a.kr + row0 * a.kcap : nullptr;
    const int kb = a.kb, vb = a.vb, pk = a.pk, pv = a.pv;

    auto load_chunk = [&](int c0, int slot) {
      const int nv = t_end - c0 < 32 ? t_end - c0 : 32;
      uint8_t* kbuf = wreg + L.kbuf + slot * 32 * pk;
      uint8_t* vbuf = wreg + L.vbuf + slot * 32 * pv;
      for (int p = lane; p < nv * kb; p += 32) {
        const int r = p / kb, c = p - r * kb;
        cp_async16(kbuf + r * pk + c * 16, kc + (long long)(c0 + r) * (16 * kb) + c * 16);
      }
      for (int p = lane; p < nv * vb; p += 32) {
        const int r = p / vb, c = p - r * vb;
        cp_async16(vbuf + r * pv + c * 16, vc + (long long)(c0 + r) * (16 * vb) + c * 16);
      }
      if (lane < nv) {
        cp_async4(wreg + L.kn + slot * 128 + lane * 4, knp + c0 + lane);
        cp_async4(wreg + L.vn + slot * 128 + lane * 4, vnp + c0 + lane);
        if constexpr (QJL) {
          cp_async16(wreg + L.sbuf + slot * 512 + lane * 16, ksp + (long long)(c0 + lane) * 16);
          cp_async4(wreg + L.rn + slot * 128 + lane * 4, krp + c0 + lane);
        }
      }
      cp_async_commit();
    };

    int c0 = t_begin + 32 * warp;
    if (c0 < t_end) load_chunk(c0, 0);
    else cp_async_commit();
    int slot = 0;
    for (; c0 < t_end; c0 += 32 * kDecodeWarps, slot ^= 1) {
      const int c1 = c0 + 32 * kDecodeWarps;
      if (c1 < t_end) load_chunk(c1, slot ^ 1);
      else cp_async_commit();
      cp_async_wait<1>();
      __syncwarp();
      const int nv = t_end - c0 < 32 ? t_end - c0 : 32;
      const bool valid = lane < nv;
      const uint8_t* krow = wreg + L.kbuf + slot * 32 * pk + lane * pk;
      const float kn = ((const float*)(wreg + L.kn + slot * 128))[lane];
      const float vn = ((const float*)(wreg + L.vn + slot * 128))[lane];
      const uint8_t* srow = QJL ? wreg + L.sbuf + slot * 512 + lane * 16 : nullptr;
      const float rn = QJL ? ((const float*)(wreg + L.rn + slot * 128))[lane] : 0.f;
      float s[G];
      switch (kb) {
        case 2: score_token<2, G, QJL>(krow, qr, lutk, kn, srow, rn, tbl, s); break;
        case 3: score_token<3, G, QJL>(krow, qr, lutk, kn, srow, rn, tbl, s); break;
        case 4: score_token<4, G, QJL>(krow, qr, lutk, kn, srow, rn, tbl, s); break;
        default: score_token<8, G, QJL>(krow, qr, lutk, kn, srow, rn, tbl, s); break;
      }
      float alpha[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float sv = valid ? s[g] : kNegBig;
        const float mnew = fmaxf(m[g], warp_max(sv));
        alpha[g] = exp2f(m[g] - mnew);
        const float p = valid ? exp2f(sv - mnew) : 0.f;
        l[g] = fmaf(l[g], alpha[g], p);
        m[g] = mnew;
        ws[lane * G + g] = valid ? p * vn : 0.f;
      }
      __syncwarp();
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int j = 0; j < 4; ++j) o[g][j] *= alpha[g];
      const uint8_t* vbuf = wreg + L.vbuf + slot * 32 * pv;
      switch (vb) {
        case 2: vsum_chunk<2, G>(vbuf, pv, ws, lutv, nv, lane, o); break;
        case 3: vsum_chunk<3, G>(vbuf, pv, ws, lutv, nv, lane, o); break;
        case 4: vsum_chunk<4, G>(vbuf, pv, ws, lutv, nv, lane, o); break;
        default: vsum_chunk<8, G>(vbuf, pv, ws, lutv, nv, lane, o); break;
      }
      __syncwarp();
    }
    cp_async_wait<0>();
  } else {
    // residual window: tokens [T - nw, T) in slots t mod W, original domain
    const int nw = T < W ? T : W;
    const int tw0 = T - nw;
    const long long base = ((long long)b * Hkv + kvh) * W;
    for (int k = warp; k < nw; k += kDecodeWarps) {
      const int t = tw0 + k;
      const long long slotrow = (base + t % W) * kD2;
      const uint2 kw = *(const uint2*)(a.kwin + slotrow + 4 * lane);
      const uint2 vw = *(const uint2*)(a.vwin + slotrow + 4 * lane);
      const float kx[4] = {bf16lo(kw.x), bf16hi(kw.x), bf16lo(kw.y), bf16hi(kw.y)};
      const float vx[4] = {bf16lo(vw.x), bf16hi(vw.x), bf16lo(vw.y), bf16hi(vw.y)};
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float part = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) part = fmaf(qo[(4 * lane + j) * G + g], kx[j], part);
        const float sc = warp_sum(part);
        const float mnew = fmaxf(m[g], sc);
        const float al = exp2f(m[g] - mnew);
        const float p = exp2f(sc - mnew);
        l[g] = fmaf(l[g], al, lane == 0 ? p : 0.f);
        m[g] = mnew;
#pragma unroll
        for (int j = 0; j < 4; ++j) o[g][j] = fmaf(p, vx[j], o[g][j] * al);
      }
    }
  }

  // ------------------------------------------------------------- epilogue
  __syncthreads();                       // warp buffers become the merge area
  float* cm = (float*)(smem + L.comb);   // [warps][G]
  float* cl = cm + kDecodeWarps * G;     // [warps][G]
  float* co = cl + kDecodeWarps * G;     // [warps][G][128]
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const float ls = warp_sum(l[g]);
    if (lane == 0) {
      cm[warp * G + g] = m[g];
      cl[warp * G + g] = ls;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) co[(warp * G + g) * kD2 + 4 * lane + j] = o[g][j];
  }
  __syncthreads();
  const long long unit = (long long)b * Hkv + kvh;
  const int stride = 2 + kD2;
  float* part = a.partials + (unit * a.n_splits + split) * G * stride;
#pragma unroll
  for (int g = 0; g < G; ++g) {
    float M = kNegBig;
#pragma unroll
    for (int w = 0; w < kDecodeWarps; ++w) M = fmaxf(M, cm[w * G + g]);
    float O = 0.f, Lsum = 0.f;
#pragma unroll
    for (int w = 0; w < kDecodeWarps; ++w) {
      const float f = exp2f(cm[w * G + g] - M);
      O = fmaf(co[(w * G + g) * kD2 + tid], f, O);
      Lsum = fmaf(cl[w * G + g], f, Lsum);
    }
    part[g * stride + 2 + tid] = O;
    if (tid == 0) {
      part[g * stride] = M;
      part[g * stride + 1] = Lsum;
    }
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const unsigned prev = atomicAdd(&a.counters[unit], 1u);
    *is_last = prev == (unsigned)(a.n_splits - 1);
  }
  __syncthreads();
  if (!*is_last) return;
  __threadfence();

  // last CTA of this (sequence, kv-head): merge the splits, inverse-rotate V
  float* acc = cm;                       // reuse: [128]
  const float* base = a.partials + unit * a.n_splits * G * stride;
  for (int g = 0; g < G; ++g) {
    float M = kNegBig;
    for (int s = 0; s < a.n_splits; ++s) M = fmaxf(M, __ldcg(base + (s * G + g) * stride));
    float rot = 0.f, Lsum = 0.f;
    for (int s = 0; s < a.n_qsplits; ++s) {
      const float* ps = base + (s * G + g) * stride;
      const float f = exp2f(__ldcg(ps) - M);
      rot = fmaf(__ldcg(ps + 2 + tid), f, rot);
      Lsum = fmaf(__ldcg(ps + 1), f, Lsum);
    }
    float win = 0.f;
    if (a.n_splits > a.n_qsplits) {
      const float* ps = base + (a.n_qsplits * G + g) * stride;
      const float f = exp2f(__ldcg(ps) - M);
      win = __ldcg(ps + 2 + tid) * f;
      Lsum = fmaf(__ldcg(ps + 1), f, Lsum);
    }
    __syncthreads();
    acc[tid] = rot;
    __syncthreads();
    for (int h = 1; h < kD2; h <<= 1) {  // R^T = D_s H / sqrt(d)
      float u = 0.f, v = 0.f;
      const bool lower = (tid & h) == 0;
      if (lower) {
        u = acc[tid];
        v = acc[tid + h];
      }
      __syncthreads();
      if (lower) {
        acc[tid] = u + v;
        acc[tid + h] = u - v;
      }
      __syncthreads();
    }
    const float x = acc[tid] * 0.08838834764831845f * svs[tid];
    a.out[((long long)b * a.Hq + (long long)kvh * G + g) * kD2 + tid] =
        Lsum > 0.f ? (x + win) / Lsum : 0.f;
  }
  if (tid == 0) a.counters[unit] = 0u;   // leave the counter ready for the next call
}

// ---------------------------------------------------------------- launcher
template <int G, bool QJL>
static int launch_d(const DecodeArgs& a, cudaStream_t s) {
  auto k = decode_kernel<G, QJL>;
  const size_t smem = (size_t)DecodeSmem(G, QJL ? 1 : 0, a.pk, a.pv).total;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return 1;
  dim3 grid((unsigned)a.n_splits, (unsigned)a.Hkv, (unsigned)a.B);
  k<<<grid, kDT, smem, s>>>(a);
  return cudaGetLastError() != cudaSuccess;
}

int launch_decode(const DecodeArgs& a, void* stream) {
  cudaStream_t s = (cudaStream_t)stream;
  if (a.Hkv > 65535 || a.B > 65535) return 1;
  switch (a.G) {
    case 1: return a.qjl ? launch_d<1, true>(a, s) : launch_d<1, false>(a, s);
    case 2: return a.qjl ? launch_d<2, true>(a, s) : launch_d<2, false>(a, s);
    case 4: return a.qjl ? launch_d<4, true>(a, s) : launch_d<4, false>(a, s);
    case 8: return a.qjl ? launch_d<8, true>(a, s) : launch_d<8, false>(a, s);
  }
  return 1;
}

unsigned* decode_error_ptr() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_decode_err) != cudaSuccess) return nullptr;
  return (unsigned*)p;
}

int decode_read_error(unsigned* out) {
  unsigned zero = 0;
  if (cudaMemcpyFromSymbol(out, g_decode_err, sizeof(unsigned)) != cudaSuccess) return 1;
  if (cudaMemcpyToSymbol(g_decode_err, &zero, sizeof(unsigned)) != cudaSuccess) return 1;
  return 0;
}

}  // namespace tq

// ------------------------------------------------ allocation-free decode entry
// Some callers cannot hand this library a workspace: a plugin inside a
// serving engine that owns every device allocation and passes only tensor
// pointers, or a latency-bound decode loop that must not call the CUDA
// allocator (cudaMalloc can synchronize the whole device).  For them the
// decode split partials and split counters live in one fixed array in device
// memory that this library reserves when it is loaded.
#include <mutex>

namespace tq {

constexpr size_t kStaticScratchBytes = 8u << 20;   // 8 MiB per GPU
constexpr int kMaxDevices = 64;

// Reserved on every GPU that loads the library, held until the process exits.
// In host code this name is only a stand-in for the device object: its device
// address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

static void* g_static_scratch_addr[kMaxDevices];
static std::mutex g_static_scratch_mu;

// Device address of the array on the current device, looked up once per device.
static tq_status static_scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return TQ_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return TQ_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_static_scratch_mu);
  if (!g_static_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) return TQ_ERR_CUDA;
    g_static_scratch_addr[dev] = p;
  }
  *out = g_static_scratch_addr[dev];
  return TQ_OK;
}

}  // namespace tq

extern "C" tq_status tq_decode_attention_noalloc(
    const tq_config* cfg, const void* tables, int layer, const void* q, int q_dtype,
    float softmax_scale, int batch, int n_q_heads, int n_kv_heads, tq_planes k, tq_planes v,
    const uint16_t* k_win, const uint16_t* v_win, const int32_t* seq_lens, int max_seq_len,
    float* out, void* stream) {
  if (!cfg || batch < 0 || n_kv_heads < 1 || n_q_heads < n_kv_heads || max_seq_len < 0)
    return TQ_ERR_INVALID_ARG;
  const size_t need = tq_workspace_bytes(cfg, batch, n_q_heads, n_kv_heads, max_seq_len);
  if (need > tq::kStaticScratchBytes) return TQ_ERR_BUFFER_TOO_SMALL;
  void* scratch = nullptr;
  tq_status st = tq::static_scratch_address(&scratch);
  if (st != TQ_OK) return st;
  // the array keeps whatever the previous call left; the split counters must
  // start at zero, so clear the part this call uses
  if (need > 0 && cudaMemsetAsync(scratch, 0, need, (cudaStream_t)stream) != cudaSuccess)
    return TQ_ERR_CUDA;
  return tq_decode_attention(cfg, tables, layer, q, q_dtype, softmax_scale, batch, n_q_heads,
                             n_kv_heads, k, v, k_win, v_win, seq_lens, max_seq_len, out, scratch,
                             tq::kStaticScratchBytes, stream);
}
