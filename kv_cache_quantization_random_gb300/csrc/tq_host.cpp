// Host side of the TurboQuant library: argument validation, the Lloyd-Max
// codebook, the seeded sign vectors and QJL matrix, the device-table layout,
// and the C-ABI entry points that launch the kernels.
//
// Sources: "TurboQuant KV 캐시 압축 for llama.cpp" (header: WHT + Lloyd-Max +
// QJL; v1.7.0 decision 4: the encoders' own sign flip + butterfly WHT);
// "[GitHub 탐방] TurboQuant 3-bit KV 캐시 압축 — 단일 GPU 재현 기록", "GPU 세대가
// 바뀌면" item (1): 2^bits Lloyd-Max centroids per rotated coordinate.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include <cuda_runtime.h>

#include "tq_internal.h"

namespace tq {

uint32_t g_wait_limit = 0;
uint32_t g_fault_injection = 0;

// ------------------------------------------------------------------ splitmix64
// Generator of Steele, Lea and Flood (2014); output k of the stream seeded
// with `state` is mix(state + (k + 1) * gamma).
static constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ull;

static inline uint64_t sm64_mix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}
static inline uint64_t sm64_at(uint64_t state, uint64_t k) { return sm64_mix(state + (k + 1) * kGamma); }

// Key of the stream of (layer, kind, purpose): output number
// layer*256 + purpose*16 + kind of the stream seeded with `seed`.
static inline uint64_t stream_key(uint64_t seed, int layer, int kind, int purpose) {
  uint64_t tag = ((uint64_t)layer << 8) | ((uint64_t)purpose << 4) | (uint64_t)kind;
  return sm64_at(seed, tag);
}
constexpr int kPurposeSigns = 0;
constexpr int kPurposeQjl = 1;

static inline uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  uint32_t lsb = (u >> 16) & 1u;
  u = u + 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

// ------------------------------------------------------------ Lloyd-Max codebook
// The quantizer of N(0,1) meeting the midpoint condition
//   beta_j = (c_j + c_{j+1}) / 2
// and the centroid condition
//   c_j = E[Z | beta_{j-1} < Z <= beta_j] = (phi(beta_{j-1}) - phi(beta_j)) / P_j,
// solved in long double by Newton's method on F(c) = c - m(beta(c)) (the
// Jacobian is tridiagonal), with c_{L-1-j} = -c_j imposed after each step.
typedef long double ld;

static ld pdf_ld(ld x) {
  if (!std::isfinite(x)) return 0.0L;
  return std::exp(-0.5L * x * x) / std::sqrt(2.0L * 3.14159265358979323846264338327950288L);
}
// P(lo < Z <= hi), in the form that does not cancel
static ld mass_ld(ld lo, ld hi) {
  const ld r2 = 1.41421356237309504880168872420969808L;
  if (lo >= 0) return 0.5L * (std::erfc(lo / r2) - (std::isfinite(hi) ? std::erfc(hi / r2) : 0.0L));
  if (hi <= 0) return 0.5L * (std::erfc(-hi / r2) - (std::isfinite(lo) ? std::erfc(-lo / r2) : 0.0L));
  return 0.5L * (std::erf(hi / r2) - std::erf(lo / r2));
}
// phi(lo) - phi(hi)
static ld pdf_diff_ld(ld lo, ld hi) {
  if (!std::isfinite(lo)) return -pdf_ld(hi);
  if (!std::isfinite(hi)) return pdf_ld(lo);
  return -pdf_ld(lo) * std::expm1(-0.5L * (hi - lo) * (hi + lo));
}
static ld normal_quantile(ld p) {
  // bisection on the CDF; plenty for a starting point
  ld lo = -40, hi = 40;
  for (int i = 0; i < 200; ++i) {
    ld mid = 0.5L * (lo + hi);
    ld cdf = mid < 0 ? 0.5L * std::erfc(-mid / 1.41421356237309504880L)
                     : 1.0L - 0.5L * std::erfc(mid / 1.41421356237309504880L);
    if (cdf < p) lo = mid; else hi = mid;
  }
  return 0.5L * (lo + hi);
}

static void lloyd_max_gaussian(int bits, std::vector<ld>& c, std::vector<ld>& beta) {
  const int L = 1 << bits;
  const ld widen = L > 16 ? std::sqrt(3.0L) : 1.0L;   // point density ~ pdf^(1/3)
  c.assign(L, 0);
  for (int j = 0; j < L; ++j) c[j] = widen * normal_quantile(((ld)j + 0.5L) / (ld)L);
  std::vector<ld> b(L - 1), lo(L), hi(L), P(L), m(L), F(L), sub(L), diag(L), sup(L), cp(L), dp(L),
      dx(L);
  for (int it = 0; it < 80; ++it) {
    for (int j = 0; j + 1 < L; ++j) b[j] = 0.5L * (c[j] + c[j + 1]);
    for (int j = 0; j < L; ++j) {
      lo[j] = j == 0 ? -INFINITY : b[j - 1];
      hi[j] = j == L - 1 ? INFINITY : b[j];
      P[j] = mass_ld(lo[j], hi[j]);
      m[j] = pdf_diff_ld(lo[j], hi[j]) / P[j];
      F[j] = c[j] - m[j];
      sub[j] = 0;
      diag[j] = 1;
      sup[j] = 0;
    }
    for (int j = 0; j < L; ++j) {
      if (j < L - 1) {
        ld t = 0.5L * pdf_ld(b[j]) * (b[j] - m[j]) / P[j];
        diag[j] -= t;
        sup[j] -= t;
      }
      if (j > 0) {
        ld t = 0.5L * pdf_ld(b[j - 1]) * (m[j] - b[j - 1]) / P[j];
        sub[j] -= t;
        diag[j] -= t;
      }
    }
    cp[0] = sup[0] / diag[0];
    dp[0] = -F[0] / diag[0];
    for (int j = 1; j < L; ++j) {
      ld den = diag[j] - sub[j] * cp[j - 1];
      cp[j] = j < L - 1 ? sup[j] / den : 0;
      dp[j] = (-F[j] - sub[j] * dp[j - 1]) / den;
    }
    dx[L - 1] = dp[L - 1];
    for (int j = L - 2; j >= 0; --j) dx[j] = dp[j] - cp[j] * dx[j + 1];
    for (int j = 0; j < L; ++j) c[j] += dx[j];
    std::vector<ld> s(c);
    for (int j = 0; j < L; ++j) c[j] = 0.5L * (s[j] - s[L - 1 - j]);
  }
  beta.assign(L - 1, 0);
  for (int j = 0; j + 1 < L; ++j) beta[j] = 0.5L * (c[j] + c[j + 1]);
  if (L % 2 == 0) beta[L / 2 - 1] = 0;
}

// ---- Lloyd-Max on the exact rotated-coordinate density ---------------------
// One coordinate y of a uniformly random unit vector in R^d has density
// f(y) = C_d (1 - y^2)^((d-3)/2) on [-1, 1], C_d = Gamma(d/2) / (Gamma(1/2)
// Gamma((d-1)/2)); it tends to N(0, 1/d) as d grows.  With y = sin(t) the
// mass of a cell is C_d * integral of cos^(d-2)(t) dt, whose integrand is
// smooth everywhere (also at the ends of the support), so composite
// Gauss-Legendre quadrature on the angle is accurate to long-double round-off;
// the first moment has the closed form C_d / (d-1) [(1-lo^2)^((d-1)/2) -
// (1-hi^2)^((d-1)/2)].  The optimality conditions are solved by the same
// Newton iteration as the Gaussian case.
static void gauss_legendre(int n, std::vector<ld>& x, std::vector<ld>& w) {
  // nodes: roots of P_n by Newton from cos(pi (i - 1/4) / (n + 1/2));
  // weights 2 / ((1 - x^2) P_n'(x)^2)
  const ld pi = 3.14159265358979323846264338327950288L;
  x.assign(n, 0);
  w.assign(n, 0);
  for (int i = 0; i < n; ++i) {
    ld z = std::cos(pi * ((ld)i + 0.75L) / ((ld)n + 0.5L));
    ld dp = 0;
    for (int it = 0; it < 100; ++it) {
      ld p0 = 1, p1 = z;
      for (int k = 2; k <= n; ++k) {
        ld p2 = ((2 * k - 1) * z * p1 - (k - 1) * p0) / k;
        p0 = p1;
        p1 = p2;
      }
      dp = n * (z * p1 - p0) / (z * z - 1);
      ld dz = p1 / dp;
      z -= dz;
      if (std::fabs(dz) < 1e-19L) break;
    }
    x[i] = z;
    w[i] = 2 / ((1 - z * z) * dp * dp);
  }
}

static ld sphere_log_norm(int d) {
  return std::lgamma((ld)d / 2) - std::lgamma(0.5L) - std::lgamma(((ld)d - 1) / 2);
}

// C_d * integral over [asin lo, asin hi] of cos^(d-2)(t)
static ld sphere_mass(ld lo, ld hi, int d, const std::vector<ld>& gx, const std::vector<ld>& gw) {
  const ld t0 = std::asin(std::max(-1.0L, std::min(1.0L, lo)));
  const ld t1 = std::asin(std::max(-1.0L, std::min(1.0L, hi)));
  const int panels = 16;
  const ld h = (t1 - t0) / panels;
  ld sum = 0;
  for (int p = 0; p < panels; ++p) {
    const ld mid = t0 + (p + 0.5L) * h;
    ld part = 0;
    for (size_t i = 0; i < gx.size(); ++i) part += gw[i] * std::pow(std::cos(mid + 0.5L * h * gx[i]), (ld)(d - 2));
    sum += 0.5L * h * part;
  }
  return std::exp(sphere_log_norm(d)) * sum;
}

static ld sphere_first_moment(ld lo, ld hi, int d) {
  const ld e = ((ld)d - 1) / 2;
  auto g = [&](ld y) { return std::pow(std::max(0.0L, 1 - y * y), e); };
  return std::exp(sphere_log_norm(d)) / (d - 1) * (g(lo) - g(hi));
}

static ld sphere_pdf(ld y, int d) {
  return std::exp(sphere_log_norm(d)) * std::pow(std::max(0.0L, 1 - y * y), ((ld)d - 3) / 2);
}

static void lloyd_max_sphere(int bits, int d, std::vector<ld>& c, std::vector<ld>& beta) {
  const int L = 1 << bits;
  std::vector<ld> gx, gw;
  gauss_legendre(24, gx, gw);
  c.assign(L, 0);
  if (d <= 16) {
    for (int j = 0; j < L; ++j) c[j] = -1 + (2 * (ld)j + 1) / L;   // uniform start
  } else {
    std::vector<ld> g, gb;
    lloyd_max_gaussian(bits, g, gb);
    for (int j = 0; j < L; ++j) c[j] = g[j] / std::sqrt((ld)d);
  }
  std::vector<ld> b(L - 1), lo(L), hi(L), P(L), m(L), F(L), sub(L), diag(L), sup(L), cp(L), dp(L),
      dx(L);
  for (int it = 0; it < 80; ++it) {
    for (int j = 0; j + 1 < L; ++j) b[j] = 0.5L * (c[j] + c[j + 1]);
    for (int j = 0; j < L; ++j) {
      lo[j] = j == 0 ? -1.0L : b[j - 1];
      hi[j] = j == L - 1 ? 1.0L : b[j];
      P[j] = sphere_mass(lo[j], hi[j], d, gx, gw);
      m[j] = sphere_first_moment(lo[j], hi[j], d) / P[j];
      F[j] = c[j] - m[j];
      sub[j] = 0;
      diag[j] = 1;
      sup[j] = 0;
    }
    for (int j = 0; j < L; ++j) {
      if (j < L - 1) {
        ld t = 0.5L * sphere_pdf(b[j], d) * (b[j] - m[j]) / P[j];
        diag[j] -= t;
        sup[j] -= t;
      }
      if (j > 0) {
        ld t = 0.5L * sphere_pdf(b[j - 1], d) * (m[j] - b[j - 1]) / P[j];
        sub[j] -= t;
        diag[j] -= t;
      }
    }
    cp[0] = sup[0] / diag[0];
    dp[0] = -F[0] / diag[0];
    for (int j = 1; j < L; ++j) {
      ld den = diag[j] - sub[j] * cp[j - 1];
      cp[j] = j < L - 1 ? sup[j] / den : 0;
      dp[j] = (-F[j] - sub[j] * dp[j - 1]) / den;
    }
    dx[L - 1] = dp[L - 1];
    for (int j = L - 2; j >= 0; --j) dx[j] = dp[j] - cp[j] * dx[j + 1];
    for (int j = 0; j < L; ++j) c[j] += dx[j];
    std::vector<ld> s(c);
    for (int j = 0; j < L; ++j) c[j] = 0.5L * (s[j] - s[L - 1 - j]);
  }
  beta.assign(L - 1, 0);
  for (int j = 0; j + 1 < L; ++j) beta[j] = 0.5L * (c[j] + c[j + 1]);
  if (L % 2 == 0) beta[L / 2 - 1] = 0;
}

static bool valid_bits(int b) { return b == 1 || b == 2 || b == 3 || b == 4 || b == 8; }
static bool gpu_bits(int b) { return b == 2 || b == 3 || b == 4 || b == 8; }
static bool pow2(int d) { return d >= 2 && (d & (d - 1)) == 0; }

static tq_status check_config(const tq_config* cfg) {
  if (!cfg) return TQ_ERR_INVALID_ARG;
  if (!pow2(cfg->head_dim) || cfg->head_dim > 1024) return TQ_ERR_INVALID_ARG;
  if (cfg->n_layers < 1 || cfg->n_layers > 4096) return TQ_ERR_INVALID_ARG;
  if (!valid_bits(cfg->k_bits) || !valid_bits(cfg->v_bits)) return TQ_ERR_INVALID_ARG;
  if (cfg->k_mode != TQ_MODE_MSE && cfg->k_mode != TQ_MODE_MSE_QJL &&
      cfg->k_mode != TQ_MODE_MSE_SIGN)
    return TQ_ERR_INVALID_ARG;
  if (cfg->k_mode == TQ_MODE_MSE_QJL &&
      (cfg->qjl_m < 32 || cfg->qjl_m > 256 || cfg->qjl_m % 32 != 0))
    return TQ_ERR_INVALID_ARG;
  if (cfg->n_protect_first < 0 || cfg->n_protect_last < 0) return TQ_ERR_INVALID_ARG;
  if ((cfg->n_protect_first > 0 || cfg->n_protect_last > 0) && !valid_bits(cfg->protect_bits))
    return TQ_ERR_INVALID_ARG;
  if (cfg->residual_window < 0 || cfg->residual_window > (1 << 20)) return TQ_ERR_INVALID_ARG;
  if (cfg->density != TQ_DENSITY_GAUSSIAN && cfg->density != TQ_DENSITY_SPHERE_BETA)
    return TQ_ERR_INVALID_ARG;
  if (cfg->sparse_v < 0 || cfg->sparse_v > 120) return TQ_ERR_INVALID_ARG;
  return TQ_OK;
}

static tq_layer_spec spec_of(const tq_config* cfg, int layer) {
  tq_layer_spec s;
  if (layer < cfg->n_protect_first || layer >= cfg->n_layers - cfg->n_protect_last) {
    s.k_bits = cfg->protect_bits;
    s.v_bits = cfg->protect_bits;
    s.k_mode = TQ_MODE_MSE;
  } else {
    s.k_bits = cfg->k_bits;
    s.v_bits = cfg->v_bits;
    s.k_mode = cfg->k_mode;
  }
  return s;
}

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

static TableOffsets table_offsets(const tq_config* cfg) {
  TableOffsets o;
  o.signs = kTblCodebook + 8 * kTblCodebookSlot;
  size_t signs_bytes = (size_t)cfg->n_layers * 2 * cfg->head_dim * sizeof(float);
  o.qjl = align256(o.signs + signs_bytes);
  int nq = 0;
  for (int l = 0; l < cfg->n_layers; ++l) nq += spec_of(cfg, l).k_mode == TQ_MODE_MSE_QJL;
  o.total = align256(o.qjl + (size_t)nq * cfg->qjl_m * cfg->head_dim * sizeof(uint16_t));
  return o;
}

static int qjl_slot(const tq_config* cfg, int layer) {
  int s = 0;
  for (int l = 0; l < layer; ++l) s += spec_of(cfg, l).k_mode == TQ_MODE_MSE_QJL;
  return s;
}

static size_t code_bytes(int d, int bits) { return (size_t)d * bits / 8; }

static bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace tq

using namespace tq;

// ===================================================================== C ABI

extern "C" int tq_version(void) { return TQ_VERSION; }

extern "C" const char* tq_status_string(tq_status s) {
  switch (s) {
    case TQ_OK: return "ok";
    case TQ_ERR_INVALID_ARG: return "invalid argument";
    case TQ_ERR_UNSUPPORTED: return "unsupported";
    case TQ_ERR_ALIGNMENT: return "misaligned pointer or stride";
    case TQ_ERR_CUDA: return "CUDA error";
    case TQ_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    case TQ_ERR_DEVICE_BOUNDS: return "device index out of bounds";
    case TQ_ERR_BUFFER_TOO_SMALL: return "buffer too small";
  }
  return "unknown status";
}

extern "C" tq_status tq_layer_spec_get(const tq_config* cfg, int layer, tq_layer_spec* out) {
  tq_status st = check_config(cfg);
  if (st != TQ_OK) return st;
  if (!out || layer < 0 || layer >= cfg->n_layers) return TQ_ERR_INVALID_ARG;
  *out = spec_of(cfg, layer);
  return TQ_OK;
}

extern "C" tq_status tq_make_codebook(int bits, int head_dim, int density, float* centroids,
                                      float* boundaries) {
  if (!valid_bits(bits) || !pow2(head_dim) || !centroids || !boundaries) return TQ_ERR_INVALID_ARG;
  if (density != TQ_DENSITY_GAUSSIAN && density != TQ_DENSITY_SPHERE_BETA) return TQ_ERR_INVALID_ARG;
  std::vector<ld> c, b;
  ld sigma = 1.0L / std::sqrt((ld)head_dim);
  if (density == TQ_DENSITY_SPHERE_BETA) {
    lloyd_max_sphere(bits, head_dim, c, b);
    sigma = 1.0L;                        // already in units of the coordinate
  } else {
    lloyd_max_gaussian(bits, c, b);
  }
  const int L = 1 << bits;
  for (int j = 0; j < L; ++j) centroids[j] = (float)(double)(c[j] * sigma);
  for (int j = 0; j + 1 < L; ++j) boundaries[j] = (float)(double)(b[j] * sigma);
  return TQ_OK;
}

extern "C" tq_status tq_make_signs(uint64_t seed, int layer, int kind, int head_dim, float* signs) {
  if (!pow2(head_dim) || !signs || layer < 0 || (kind != 0 && kind != 1)) return TQ_ERR_INVALID_ARG;
  uint64_t key = stream_key(seed, layer, kind, kPurposeSigns);
  for (int i = 0; i < head_dim; ++i) signs[i] = (sm64_at(key, (uint64_t)i) & 1ull) ? -1.0f : 1.0f;
  return TQ_OK;
}

extern "C" tq_status tq_make_qjl_matrix(uint64_t seed, int layer, int m, int head_dim,
                                        uint16_t* s_bf16) {
  if (!pow2(head_dim) || !s_bf16 || layer < 0 || m < 1) return TQ_ERR_INVALID_ARG;
  uint64_t key = stream_key(seed, layer, 0, kPurposeQjl);
  const double two53 = 9007199254740992.0;
  for (int64_t e = 0; e < (int64_t)m * head_dim; ++e) {
    uint64_t o1 = sm64_at(key, 2 * (uint64_t)e), o2 = sm64_at(key, 2 * (uint64_t)e + 1);
    double u1 = ((double)(o1 >> 11) + 0.5) / two53;
    double u2 = (double)(o2 >> 11) / two53;
    double g = std::sqrt(-2.0 * std::log(u1)) * std::cos(2.0 * 3.14159265358979323846 * u2);
    s_bf16[e] = f32_to_bf16_rne((float)g);
  }
  return TQ_OK;
}

extern "C" size_t tq_tables_bytes(const tq_config* cfg) {
  if (check_config(cfg) != TQ_OK) return 0;
  return table_offsets(cfg).total;
}

extern "C" tq_status tq_build_tables(const tq_config* cfg, void* host_buf, size_t bytes) {
  tq_status st = check_config(cfg);
  if (st != TQ_OK) return st;
  if (!host_buf) return TQ_ERR_INVALID_ARG;
  TableOffsets o = table_offsets(cfg);
  if (bytes < o.total) return TQ_ERR_BUFFER_TOO_SMALL;
  uint8_t* base = (uint8_t*)host_buf;
  std::memset(base, 0, o.total);
  int32_t* hdr = (int32_t*)base;
  hdr[0] = (int32_t)kTblMagic;
  hdr[1] = TQ_VERSION;
  hdr[2] = cfg->head_dim;
  hdr[3] = cfg->n_layers;
  hdr[4] = cfg->qjl_m;
  // codebooks for every bit width any layer uses
  bool used[9] = {false};
  for (int l = 0; l < cfg->n_layers; ++l) {
    tq_layer_spec s = spec_of(cfg, l);
    used[s.k_bits] = used[s.v_bits] = true;
  }
  for (int bits = 1; bits <= 8; ++bits) {
    float* cb = (float*)(base + kTblCodebook + (bits - 1) * kTblCodebookSlot);
    for (int j = 0; j < 256; ++j) cb[256 + j] = INFINITY;
    if (!used[bits]) continue;
    st = tq_make_codebook(bits, cfg->head_dim, cfg->density, cb, cb + 256);
    if (st != TQ_OK) return st;
  }
  for (int l = 0; l < cfg->n_layers; ++l)
    for (int kind = 0; kind < 2; ++kind)
      tq_make_signs(cfg->seed, l, kind, cfg->head_dim,
                    (float*)(base + o.signs) + (size_t)(2 * l + kind) * cfg->head_dim);
  int slot = 0;
  for (int l = 0; l < cfg->n_layers; ++l) {
    if (spec_of(cfg, l).k_mode != TQ_MODE_MSE_QJL) continue;
    tq_make_qjl_matrix(cfg->seed, l, cfg->qjl_m, cfg->head_dim,
                       (uint16_t*)(base + o.qjl) + (size_t)slot * cfg->qjl_m * cfg->head_dim);
    ++slot;
  }
  return TQ_OK;
}

extern "C" tq_status tq_plane_bytes(const tq_config* cfg, int layer, int kind, int batch,
                                    int n_kv_heads, int64_t capacity, size_t sizes[4]) {
  tq_status st = check_config(cfg);
  if (st != TQ_OK) return st;
  if (!sizes || layer < 0 || layer >= cfg->n_layers || (kind != 0 && kind != 1) || batch < 0 ||
      n_kv_heads < 0 || capacity < 0)
    return TQ_ERR_INVALID_ARG;
  tq_layer_spec s = spec_of(cfg, layer);
  int bits = kind == 0 ? s.k_bits : s.v_bits;
  size_t rows = (size_t)batch * n_kv_heads * (size_t)capacity;
  sizes[0] = rows * code_bytes(cfg->head_dim, bits);
  sizes[1] = rows * sizeof(float);
  const bool qjl = kind == 0 && s.k_mode == TQ_MODE_MSE_QJL;
  const bool dsign = kind == 0 && s.k_mode == TQ_MODE_MSE_SIGN;
  sizes[2] = qjl ? rows * (size_t)(cfg->qjl_m / 8) : dsign ? rows * (size_t)(cfg->head_dim / 8) : 0;
  sizes[3] = qjl || dsign ? rows * sizeof(float) : 0;
  return TQ_OK;
}

// ------------------------------------------------------------------ decode plan
namespace tq {
struct DecodePlan {
  int n_qsplits, n_splits, split_tokens, wsplit_tokens, G, long_first;
  size_t partial_floats, counters_off, total;
};
// Splits of one decode launch for a layer of format s: one wave of about
// kDecodeSms x decode_ctas_per_sm CTAs of decode_warps(...) warps.  The window is
// cut into splits of at most 32 tokens per warp; the quantized tokens of each
// (sequence, kv-head) are split evenly in multiples of 32 tokens over the rest.
// step_split: a decode step in one launch with no window gets one split per
// pair for the new token (see DecodeArgs::fused_step)
static DecodePlan decode_plan(const tq_config* cfg, const tq_layer_spec& s, int batch,
                              int n_q_heads, int n_kv_heads, int max_seq_len,
                              bool step_split = false) {
  DecodePlan p;
  const int W = cfg->residual_window;
  long long max_nq = (long long)max_seq_len - W;
  if (max_nq < 0) max_nq = 0;
  const long long units = (long long)batch * n_kv_heads;
  p.G = n_kv_heads > 0 ? n_q_heads / n_kv_heads : 0;
  const int res = s.k_mode == TQ_MODE_MSE_QJL ? 1 : s.k_mode == TQ_MODE_MSE_SIGN ? 2 : 0;
  const int warps = decode_warps(p.G, s.k_bits, s.v_bits, res);
  int wst = (W + 31) / 32 * 32;
  if (wst > 32 * warps) wst = 32 * warps;
  p.wsplit_tokens = wst > 0 ? wst : 1;
  const int n_wsplits = W > 0 ? (W + wst - 1) / wst : step_split ? 1 : 0;
  const long long wave = (long long)kDecodeSms * decode_ctas_per_sm(p.G, s.k_bits, s.v_bits, res);
  long long slots = wave - units * n_wsplits;
  if (slots < units) {
    // more than one wave: the quantized splits alone fill the wave (the short
    // window splits run after them, longest first), at least one per pair
    slots = (wave / units > 0 ? wave / units : 1) * units;
  }
  // the same number of quantized splits for every pair, as many as the slots
  // allow: cutting the pairs' tokens into slots-many pieces instead leaves a
  // ragged second wave (measured on 128 pairs of 8,192 tokens at two CTAs per
  // SM: 89.2 us for 3 splits of 3,456 tokens in two waves, 80.1 us for 2
  // splits of 4,096 in one)
  const long long k = units > 0 ? slots / units : 1;
  long long per = k > 0 ? (max_nq + k - 1) / k : max_nq;
  long long st = (per + 31) / 32 * 32;
  if (st < 256) st = 256;
  p.split_tokens = (int)st;
  p.n_qsplits = (int)((max_nq + st - 1) / st);
  p.n_splits = p.n_qsplits + n_wsplits;
  p.long_first = units * p.n_splits > wave;
  p.partial_floats = (size_t)units * p.n_splits * p.G * kPartialStride;
  p.counters_off = align256(p.partial_floats * sizeof(float));
  p.total = p.counters_off + align256((size_t)units * sizeof(unsigned));
  return p;
}
}  // namespace tq

extern "C" size_t tq_workspace_bytes(const tq_config* cfg, int batch, int n_q_heads,
                                     int n_kv_heads, int max_seq_len) {
  if (check_config(cfg) != TQ_OK || batch < 0 || n_kv_heads < 1 || n_q_heads < n_kv_heads ||
      max_seq_len < 0)
    return 0;
  // the largest plan over the layers' formats, a plain decode's or a decode
  // step's (which with W = 0 has one split more per pair)
  size_t total = 0;
  for (int layer = 0; layer < cfg->n_layers; ++layer) {
    for (int step = 0; step < 2; ++step) {
      const size_t t = decode_plan(cfg, spec_of(cfg, layer), batch, n_q_heads, n_kv_heads,
                                   max_seq_len, step == 1).total;
      if (t > total) total = t;
    }
  }
  return total;
}

namespace tq {
// A decode step runs in one launch when its plan (with the splits that append
// the token) is one wave and gives the warps of the quantized splits no more
// 32-token chunks than a plain decode's plan: with W = 0 the step's extra split
// per pair can cost the pairs a quantized split (measured: on 128 pairs at
// three CTAs per SM, 3 splits of 2,752 tokens, 22 chunks a warp, became 2 of
// 4,096, 32 chunks a warp, and the step took 111 us against 90 us as an append
// and a decode).  Otherwise the append kernel runs first and a plain decode
// after it.
static bool step_one_launch(const tq_config* cfg, int layer, int batch, int n_q_heads,
                            int n_kv_heads, int max_seq_len) {
  const tq_layer_spec s = spec_of(cfg, layer);
  const DecodePlan ps = decode_plan(cfg, s, batch, n_q_heads, n_kv_heads, max_seq_len, true);
  const DecodePlan pd = decode_plan(cfg, s, batch, n_q_heads, n_kv_heads, max_seq_len, false);
  const int res = s.k_mode == TQ_MODE_MSE_QJL ? 1 : s.k_mode == TQ_MODE_MSE_SIGN ? 2 : 0;
  const long long warp_tokens = 32LL * decode_warps(ps.G, s.k_bits, s.v_bits, res);
  auto chunks = [&](int st) { return (st + warp_tokens - 1) / warp_tokens; };
  return !ps.long_first && chunks(ps.split_tokens) <= chunks(pd.split_tokens);
}
}  // namespace tq

namespace tq {
// Byte range [*off, *off + *bytes) of the split counters in the workspace of a
// tq_decode_attention call with these shapes: the only part of the workspace
// that must be zero when the decode starts (the partials are written before
// they are read).
tq_status decode_counters_range(const tq_config* cfg, int layer, int batch, int n_q_heads,
                                int n_kv_heads, int max_seq_len, size_t* off, size_t* bytes) {
  if (check_config(cfg) != TQ_OK || layer < 0 || layer >= cfg->n_layers || batch < 0 ||
      n_kv_heads < 1 || n_q_heads < n_kv_heads || max_seq_len < 0)
    return TQ_ERR_INVALID_ARG;
  const DecodePlan p =
      decode_plan(cfg, spec_of(cfg, layer), batch, n_q_heads, n_kv_heads, max_seq_len);
  *off = p.counters_off;
  *bytes = p.total - p.counters_off;
  return TQ_OK;
}
}  // namespace tq

extern "C" tq_status tq_workspace_init(void* workspace, size_t workspace_bytes, void* stream) {
  if (!workspace) return TQ_ERR_INVALID_ARG;
  if (cudaMemsetAsync(workspace, 0, workspace_bytes, (cudaStream_t)stream) != cudaSuccess)
    return TQ_ERR_CUDA;
  return TQ_OK;
}

// ---------------------------------------------------------------- entry points
namespace tq {
static const uint8_t* tbl_codebook(const void* tables, int bits) {
  return (const uint8_t*)tables + kTblCodebook + (size_t)(bits - 1) * kTblCodebookSlot;
}
static const float* tbl_signs(const tq_config* cfg, const void* tables, int layer, int kind) {
  TableOffsets o = table_offsets(cfg);
  return (const float*)((const uint8_t*)tables + o.signs) + (size_t)(2 * layer + kind) * cfg->head_dim;
}
static const uint16_t* tbl_qjl(const tq_config* cfg, const void* tables, int layer) {
  TableOffsets o = table_offsets(cfg);
  return (const uint16_t*)((const uint8_t*)tables + o.qjl) +
         (size_t)qjl_slot(cfg, layer) * cfg->qjl_m * cfg->head_dim;
}
static tq_status check_gpu_common(const tq_config* cfg, const void* tables, int layer) {
  tq_status st = check_config(cfg);
  if (st != TQ_OK) return st;
  if (!tables || layer < 0 || layer >= cfg->n_layers) return TQ_ERR_INVALID_ARG;
  if (!aligned16(tables)) return TQ_ERR_ALIGNMENT;
  if (cfg->head_dim != kHeadDim) return TQ_ERR_UNSUPPORTED;
  tq_layer_spec s = spec_of(cfg, layer);
  if (!gpu_bits(s.k_bits) || !gpu_bits(s.v_bits)) return TQ_ERR_UNSUPPORTED;
  if (s.k_mode == TQ_MODE_MSE_QJL && cfg->qjl_m != kQjlM) return TQ_ERR_UNSUPPORTED;
  return TQ_OK;
}
static tq_status check_planes(const tq_config* cfg, int layer, int kind, const tq_planes& p) {
  tq_layer_spec s = spec_of(cfg, layer);
  const bool qjl = kind == 0 && s.k_mode != TQ_MODE_MSE;   // QJL or Direct Sign planes
  if (!p.codes || !p.norms || p.capacity < 0) return TQ_ERR_INVALID_ARG;
  if (qjl && (!p.qjl_signs || !p.qjl_rnorm)) return TQ_ERR_INVALID_ARG;
  if (!aligned16(p.codes) || !aligned16(p.norms)) return TQ_ERR_ALIGNMENT;
  if (qjl && (!aligned16(p.qjl_signs) || !aligned16(p.qjl_rnorm))) return TQ_ERR_ALIGNMENT;
  return TQ_OK;
}
// Search grid of a codebook (see SearchGrid), from the same fp32 boundaries
// the device tables hold; cached per (bits, density, head_dim).
static SearchGrid search_grid(const tq_config* cfg, int bits) {
  static std::mutex mu;
  static std::vector<std::pair<uint64_t, SearchGrid>> cache;
  const uint64_t key = ((uint64_t)bits << 40) | ((uint64_t)cfg->density << 32) | (uint32_t)cfg->head_dim;
  {
    std::lock_guard<std::mutex> lock(mu);
    for (auto& e : cache)
      if (e.first == key) return e.second;
  }
  std::vector<float> c(256), b(256);
  SearchGrid g{0.f, 0.f, 0.f, 0};
  if (tq_make_codebook(bits, cfg->head_dim, cfg->density, c.data(), b.data()) != TQ_OK) return g;
  const int L = 1 << bits;
  double gap = 1.0, maxb = 0.0;
  for (int j = 0; j + 1 < L - 1; ++j) gap = std::min(gap, (double)b[j + 1] - (double)b[j]);
  for (int j = 0; j + 1 < L; ++j) maxb = std::max(maxb, std::fabs((double)b[j]));
  g.scale = (float)(4.0 / gap);
  // 2..4 bits: the grid spans |y| <= 1.01 (a unit vector's coordinates); 8
  // bits: only the span of the boundaries, with |y| clamped onto it
  const double span = bits <= 4 ? 1.01 : maxb + 3.0 / g.scale;
  g.clamp = bits <= 4 ? 0.f : (float)(maxb + 2.0 / g.scale);
  g.cells = 2 * (int)std::ceil(span * g.scale) + 4;
  g.magic = 12582912.0f + (float)(g.cells / 2);
  std::lock_guard<std::mutex> lock(mu);
  cache.push_back({key, g});
  return g;
}

static void fill_quant_codec(QuantArgs& a, const tq_config* cfg, const void* tables, int layer,
                             int kind) {
  tq_layer_spec s = spec_of(cfg, layer);
  a.bits = kind == 0 ? s.k_bits : s.v_bits;
  const uint8_t* cb = tbl_codebook(tables, a.bits);
  a.centroids = (const float*)cb;
  a.boundaries = (const float*)cb + 256;
  a.rot_signs = tbl_signs(cfg, tables, layer, kind);
  a.qjl = kind == 0 && s.k_mode == TQ_MODE_MSE_QJL;
  a.dsign = kind == 0 && s.k_mode == TQ_MODE_MSE_SIGN;
  a.S = a.qjl ? tbl_qjl(cfg, tables, layer) : nullptr;
  a.m = cfg->qjl_m;
  a.err = quant_error_ptr();
  a.wait_limit = g_wait_limit;
  const SearchGrid g = search_grid(cfg, a.bits);
  a.grid_scale = g.scale;
  a.grid_magic = g.magic;
  a.grid_clamp = g.clamp;
  a.grid_cells = g.cells;
  float sg[kHeadDim];
  tq_make_signs(cfg->seed, layer, kind, kHeadDim, sg);
  for (int i = 0; i < kHeadDim; ++i) a.smask[i] = sg[i] < 0.f ? 0x80000000u : 0u;
}
}  // namespace tq

extern "C" tq_status tq_quantize_kv(const tq_config* cfg, const void* tables, int layer, int kind,
                                    const void* src, int src_dtype, const int64_t src_strides[3],
                                    int batch, int n_kv_heads, int n_tokens,
                                    const int32_t* dst_pos, tq_planes dst, void* stream) {
  tq_status st = check_gpu_common(cfg, tables, layer);
  if (st != TQ_OK) return st;
  if (kind != 0 && kind != 1) return TQ_ERR_INVALID_ARG;
  if (batch < 0 || n_kv_heads < 0 || n_tokens < 0 || !src_strides) return TQ_ERR_INVALID_ARG;
  if (src_dtype != TQ_BF16 && src_dtype != TQ_F32) return TQ_ERR_INVALID_ARG;
  if ((long long)batch * n_kv_heads * n_tokens == 0) return TQ_OK;
  if (!src) return TQ_ERR_INVALID_ARG;
  st = check_planes(cfg, layer, kind, dst);
  if (st != TQ_OK) return st;
  const int esz = src_dtype == TQ_F32 ? 4 : 2;
  if (!aligned16(src)) return TQ_ERR_ALIGNMENT;
  for (int i = 0; i < 3; ++i)
    if (src_strides[i] < 0 || (src_strides[i] * esz) % 16 != 0) return TQ_ERR_ALIGNMENT;
  if (!dst_pos && n_tokens > dst.capacity) return TQ_ERR_INVALID_ARG;
  if ((long long)batch * n_kv_heads * n_tokens >= (1ll << 31)) return TQ_ERR_UNSUPPORTED;
  QuantArgs a{};
  a.src = src;
  a.src_f32 = src_dtype == TQ_F32;
  a.sb = src_strides[0];
  a.sh = src_strides[1];
  a.st = src_strides[2];
  a.B = batch;
  a.H = n_kv_heads;
  a.n = n_tokens;
  a.dst_pos = dst_pos;
  a.codes = dst.codes;
  a.norms = dst.norms;
  a.qjl_signs = dst.qjl_signs;
  a.qjl_rnorm = dst.qjl_rnorm;
  a.cap = dst.capacity;
  fill_quant_codec(a, cfg, tables, layer, kind);
  if (a.grid_cells <= 0 || a.grid_cells > kMaxGridCells) return TQ_ERR_UNSUPPORTED;
  return launch_quantize(a, stream) == 0 ? TQ_OK : TQ_ERR_CUDA;
}

extern "C" tq_status tq_append_kv(const tq_config* cfg, const void* tables, int layer,
                                  const void* k_new, const void* v_new, int src_dtype,
                                  const int64_t src_strides[3], int batch, int n_kv_heads,
                                  int n_new, const int32_t* seq_lens_before, uint16_t* k_win,
                                  uint16_t* v_win, tq_planes k, tq_planes v, void* stream) {
  tq_status st = check_gpu_common(cfg, tables, layer);
  if (st != TQ_OK) return st;
  if (batch < 0 || n_kv_heads < 0 || n_new < 0 || !src_strides) return TQ_ERR_INVALID_ARG;
  if (src_dtype != TQ_BF16 && src_dtype != TQ_F32) return TQ_ERR_INVALID_ARG;
  if ((long long)batch * n_kv_heads * n_new == 0) return TQ_OK;
  if (!k_new || !v_new || !seq_lens_before) return TQ_ERR_INVALID_ARG;
  const int W = cfg->residual_window;
  if (W > 0 && (!k_win || !v_win)) return TQ_ERR_INVALID_ARG;
  if (W > 0 && src_dtype != TQ_BF16) return TQ_ERR_UNSUPPORTED;  // the window ring is bf16
  if (W > 0 && (!aligned16(k_win) || !aligned16(v_win))) return TQ_ERR_ALIGNMENT;
  const int esz = src_dtype == TQ_F32 ? 4 : 2;
  if (!aligned16(k_new) || !aligned16(v_new)) return TQ_ERR_ALIGNMENT;
  for (int i = 0; i < 3; ++i)
    if (src_strides[i] < 0 || (src_strides[i] * esz) % 16 != 0) return TQ_ERR_ALIGNMENT;
  for (int kind = 0; kind < 2; ++kind) {
    st = check_planes(cfg, layer, kind, kind == 0 ? k : v);
    if (st != TQ_OK) return st;
  }
  if (n_new <= kAppendFusedMaxNew) {
    AppendArgs a{};
    a.src[0] = k_new;
    a.src[1] = v_new;
    a.src_f32 = src_dtype == TQ_F32;
    a.sb = src_strides[0];
    a.sh = src_strides[1];
    a.st = src_strides[2];
    a.B = batch;
    a.H = n_kv_heads;
    a.n = n_new;
    a.seq_before = seq_lens_before;
    a.W = W;
    a.win[0] = k_win;
    a.win[1] = v_win;
    for (int kind = 0; kind < 2; ++kind) {
      const tq_planes& p = kind == 0 ? k : v;
      QuantArgs q{};
      fill_quant_codec(q, cfg, tables, layer, kind);
      a.codes[kind] = p.codes;
      a.norms[kind] = p.norms;
      a.cap[kind] = p.capacity;
      a.bits[kind] = q.bits;
      a.centroids[kind] = q.centroids;
      a.boundaries[kind] = q.boundaries;
      a.rot_signs[kind] = q.rot_signs;
      if (kind == 0) {
        a.qjl = q.qjl;
        a.dsign = q.dsign;
        a.S = q.S;
        a.qjl_signs = p.qjl_signs;
        a.qjl_rnorm = p.qjl_rnorm;
        a.err = q.err;
      }
    }
    return launch_append(a, stream) != 0 ? TQ_ERR_CUDA : TQ_OK;
  }
  if ((long long)batch * n_kv_heads * n_new >= (1ll << 31)) return TQ_ERR_UNSUPPORTED;
  QuantArgs qa[2] = {};
  for (int kind = 0; kind < 2; ++kind) {
    const tq_planes& p = kind == 0 ? k : v;
    QuantArgs& a = qa[kind];
    a.src = kind == 0 ? k_new : v_new;
    a.src_f32 = src_dtype == TQ_F32;
    a.sb = src_strides[0];
    a.sh = src_strides[1];
    a.st = src_strides[2];
    a.B = batch;
    a.H = n_kv_heads;
    a.n = n_new;
    a.append = 1;
    a.seq_before = seq_lens_before;
    a.W = W;
    a.win = kind == 0 ? k_win : v_win;
    a.codes = p.codes;
    a.norms = p.norms;
    a.qjl_signs = p.qjl_signs;
    a.qjl_rnorm = p.qjl_rnorm;
    a.cap = p.capacity;
    fill_quant_codec(a, cfg, tables, layer, kind);
    if (a.grid_cells <= 0 || a.grid_cells > kMaxGridCells) return TQ_ERR_UNSUPPORTED;
  }
  // one launch for both kinds when they share the kernel variant's shape
  if (!qa[0].src_f32 && !qa[0].qjl && !qa[1].qjl && !qa[1].dsign && qa[0].bits == qa[1].bits &&
      qa[0].grid_cells == qa[1].grid_cells)
    return launch_quantize_kv(qa[0], qa[1], stream) != 0 ? TQ_ERR_CUDA : TQ_OK;
  for (int kind = 0; kind < 2; ++kind)
    if (launch_quantize(qa[kind], stream) != 0) return TQ_ERR_CUDA;
  return TQ_OK;
}

extern "C" tq_status tq_dequantize(const tq_config* cfg, const void* tables, int layer, int kind,
                                   tq_planes src, int batch, int n_kv_heads, int n_tokens,
                                   int include_qjl, float* dst, void* stream) {
  tq_status st = check_gpu_common(cfg, tables, layer);
  if (st != TQ_OK) return st;
  if ((kind != 0 && kind != 1) || batch < 0 || n_kv_heads < 0 || n_tokens < 0)
    return TQ_ERR_INVALID_ARG;
  if ((long long)batch * n_kv_heads * n_tokens == 0) return TQ_OK;
  if (!dst) return TQ_ERR_INVALID_ARG;
  if (!aligned16(dst)) return TQ_ERR_ALIGNMENT;
  st = check_planes(cfg, layer, kind, src);
  if (st != TQ_OK) return st;
  if (n_tokens > src.capacity) return TQ_ERR_INVALID_ARG;
  tq_layer_spec s = spec_of(cfg, layer);
  DequantArgs a{};
  a.codes = src.codes;
  a.norms = src.norms;
  a.qjl_signs = src.qjl_signs;
  a.qjl_rnorm = src.qjl_rnorm;
  a.cap = src.capacity;
  a.B = batch;
  a.H = n_kv_heads;
  a.n = n_tokens;
  a.bits = kind == 0 ? s.k_bits : s.v_bits;
  a.centroids = (const float*)tbl_codebook(tables, a.bits);
  a.rot_signs = tbl_signs(cfg, tables, layer, kind);
  a.qjl = include_qjl && kind == 0 && s.k_mode == TQ_MODE_MSE_QJL;
  a.dsign = include_qjl && kind == 0 && s.k_mode == TQ_MODE_MSE_SIGN;
  a.S = a.qjl ? tbl_qjl(cfg, tables, layer) : nullptr;
  a.m = cfg->qjl_m;
  a.dst = dst;
  a.err = quant_error_ptr();
  return launch_dequantize(a, stream) == 0 ? TQ_OK : TQ_ERR_CUDA;
}

// Decode with n_queries query tokens per sequence: the n_queries query
// vectors of a query head are laid out contiguously ([B][Hq][n_queries][d]),
// so the kernel sees n_q_heads * n_queries query columns in groups of
// G * n_queries per kv-head, and masks window tokens causally per column.
namespace tq {
// Checks and launch arguments of a decode; *empty: every sequence is empty
// (nothing to launch, the output is zero).
static tq_status decode_prepare(const tq_config* cfg, const void* tables, int layer, const void* q,
                                int q_dtype, float softmax_scale, int batch, int n_q_heads,
                                int n_kv_heads, int n_queries, tq_planes k, tq_planes v,
                                const uint16_t* k_win, const uint16_t* v_win,
                                const int32_t* seq_lens, int max_seq_len, float* out,
                                void* workspace, size_t workspace_bytes, int step_new,
                                bool step_split, DecodeArgs* args, bool* empty) {
  *empty = false;
  tq_status st = check_gpu_common(cfg, tables, layer);
  if (st != TQ_OK) return st;
  if (batch < 0 || n_kv_heads < 1 || n_q_heads < n_kv_heads || n_q_heads % n_kv_heads != 0 ||
      max_seq_len < 0 || n_queries < 1)
    return TQ_ERR_INVALID_ARG;
  const int G = n_q_heads / n_kv_heads * n_queries;   // query columns per kv-head
  if (G != 1 && G != 2 && G != 4 && G != 8) return TQ_ERR_UNSUPPORTED;
  // the tokens that some query must not see (the last n_queries - 1) have to
  // be window tokens
  if (n_queries > 1 && cfg->residual_window < n_queries - 1) return TQ_ERR_UNSUPPORTED;
  n_q_heads *= n_queries;
  if (q_dtype != TQ_BF16 && q_dtype != TQ_F32) return TQ_ERR_INVALID_ARG;
  if (!(std::isfinite(softmax_scale))) return TQ_ERR_INVALID_ARG;
  if (batch == 0) {
    *empty = true;
    return TQ_OK;
  }
  if (!q || !seq_lens || !out || !workspace) return TQ_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(out) || !aligned16(workspace)) return TQ_ERR_ALIGNMENT;
  const int W = cfg->residual_window;
  if (W > 0 && (!k_win || !v_win)) return TQ_ERR_INVALID_ARG;
  if (W > 0 && (!aligned16(k_win) || !aligned16(v_win))) return TQ_ERR_ALIGNMENT;
  for (int kind = 0; kind < 2; ++kind) {
    st = check_planes(cfg, layer, kind, kind == 0 ? k : v);
    if (st != TQ_OK) return st;
  }
  long long max_nq = (long long)max_seq_len - W;
  if (max_nq > k.capacity || max_nq > v.capacity) return TQ_ERR_INVALID_ARG;
  tq_layer_spec s = spec_of(cfg, layer);
  const DecodePlan p = decode_plan(cfg, s, batch, n_q_heads, n_kv_heads, max_seq_len, step_split);
  if (workspace_bytes < p.total) return TQ_ERR_BUFFER_TOO_SMALL;
  if ((long long)p.n_splits * n_kv_heads * batch >= (1ll << 31)) return TQ_ERR_UNSUPPORTED;
  DecodeArgs a{};
  a.q = q;
  a.q_f32 = q_dtype == TQ_F32;
  a.qscale = softmax_scale * 1.4426950408889634f;
  a.B = batch;
  a.Hq = n_q_heads;
  a.Hkv = n_kv_heads;
  a.G = G;
  a.kc = k.codes;
  a.kn = k.norms;
  a.ks = k.qjl_signs;
  a.kr = k.qjl_rnorm;
  a.kcap = k.capacity;
  a.vc = v.codes;
  a.vn = v.norms;
  a.vcap = v.capacity;
  a.kb = s.k_bits;
  a.vb = s.v_bits;
  a.qjl = s.k_mode == TQ_MODE_MSE_QJL;
  a.dsign = s.k_mode == TQ_MODE_MSE_SIGN;
  a.sparse_thr = cfg->sparse_v > 0 ? std::ldexp(1.0f, -cfg->sparse_v) : 0.0f;
  if (a.sparse_thr > 0.f && (a.qjl || a.dsign)) return TQ_ERR_UNSUPPORTED;   // MSE keys only
  a.m = cfg->qjl_m;
  a.kwin = k_win;
  a.vwin = v_win;
  a.W = W;
  a.seq_lens = seq_lens;
  a.max_seq_len = max_seq_len;
  a.n_qsplits = p.n_qsplits;
  a.n_splits = p.n_splits;
  a.split_tokens = p.split_tokens;
  a.wsplit_tokens = p.wsplit_tokens;
  a.long_first = p.long_first;
  {
    const int res = a.qjl ? 1 : a.dsign ? 2 : 0;
    a.pdl_trigger = !p.long_first && decode_ctas_per_sm(G, s.k_bits, s.v_bits, res) == 1;
  }
  a.ck = (const float*)tbl_codebook(tables, s.k_bits);
  a.cv = (const float*)tbl_codebook(tables, s.v_bits);
  a.sk = tbl_signs(cfg, tables, layer, 0);
  a.sv = tbl_signs(cfg, tables, layer, 1);
  a.S = a.qjl ? tbl_qjl(cfg, tables, layer) : nullptr;
  a.out = out;
  a.partials = (float*)workspace;
  a.counters = (unsigned*)((uint8_t*)workspace + p.counters_off);
  a.err = decode_error_ptr();
  a.wait_limit = g_wait_limit;
  a.extra_tx = g_fault_injection == 1 ? 16u : 0u;
  a.n_q = n_queries;
  a.step_new = step_new;
  *empty = p.n_splits == 0;
  *args = a;
  return TQ_OK;
}

static tq_status decode_common(const tq_config* cfg, const void* tables, int layer, const void* q,
                               int q_dtype, float softmax_scale, int batch, int n_q_heads,
                               int n_kv_heads, int n_queries, tq_planes k, tq_planes v,
                               const uint16_t* k_win, const uint16_t* v_win,
                               const int32_t* seq_lens, int max_seq_len, float* out,
                               void* workspace, size_t workspace_bytes, void* stream) {
  DecodeArgs a{};
  bool empty = false;
  tq_status st = decode_prepare(cfg, tables, layer, q, q_dtype, softmax_scale, batch, n_q_heads,
                                n_kv_heads, n_queries, k, v, k_win, v_win, seq_lens, max_seq_len,
                                out, workspace, workspace_bytes, 0, false, &a, &empty);
  if (st != TQ_OK) return st;
  if (batch == 0) return TQ_OK;
  if (empty) {
    // every sequence is empty: the output is zero
    if (cudaMemsetAsync(out, 0, (size_t)batch * n_q_heads * n_queries * kHeadDim * sizeof(float),
                        (cudaStream_t)stream) != cudaSuccess)
      return TQ_ERR_CUDA;
    return TQ_OK;
  }
  return launch_decode(a, stream) == 0 ? TQ_OK : TQ_ERR_CUDA;
}
}  // namespace tq

extern "C" tq_status tq_decode_attention(const tq_config* cfg, const void* tables, int layer,
                                         const void* q, int q_dtype, float softmax_scale,
                                         int batch, int n_q_heads, int n_kv_heads, tq_planes k,
                                         tq_planes v, const uint16_t* k_win,
                                         const uint16_t* v_win, const int32_t* seq_lens,
                                         int max_seq_len, float* out, void* workspace,
                                         size_t workspace_bytes, void* stream) {
  return decode_common(cfg, tables, layer, q, q_dtype, softmax_scale, batch, n_q_heads,
                       n_kv_heads, 1, k, v, k_win, v_win, seq_lens, max_seq_len, out, workspace,
                       workspace_bytes, stream);
}

extern "C" tq_status tq_decode_attention_multi(
    const tq_config* cfg, const void* tables, int layer, const void* q, int q_dtype,
    float softmax_scale, int batch, int n_q_heads, int n_kv_heads, int n_queries, tq_planes k,
    tq_planes v, const uint16_t* k_win, const uint16_t* v_win, const int32_t* seq_lens,
    int max_seq_len, float* out, void* workspace, size_t workspace_bytes, void* stream) {
  return decode_common(cfg, tables, layer, q, q_dtype, softmax_scale, batch, n_q_heads,
                       n_kv_heads, n_queries, k, v, k_win, v_win, seq_lens, max_seq_len, out,
                       workspace, workspace_bytes, stream);
}

extern "C" tq_status tq_decode_step(const tq_config* cfg, const void* tables, int layer,
                                    const void* q, int q_dtype, float softmax_scale, int batch,
                                    int n_q_heads, int n_kv_heads, const void* k_new,
                                    const void* v_new, int src_dtype, const int64_t src_strides[3],
                                    const int32_t* seq_lens_before, int max_seq_len,
                                    uint16_t* k_win, uint16_t* v_win, tq_planes k, tq_planes v,
                                    float* out, void* workspace, size_t workspace_bytes,
                                    void* stream) {
  if (batch == 0) return TQ_OK;
  if (max_seq_len < 1) return TQ_ERR_INVALID_ARG;
  tq_status st = check_gpu_common(cfg, tables, layer);
  if (st != TQ_OK) return st;
  // one launch: the decode kernel appends the step's token itself (see
  // DecodeArgs::fused_step); the inputs are checked as tq_append_kv checks them
  const int W = cfg->residual_window;
  if (!k_new || !v_new || !src_strides) return TQ_ERR_INVALID_ARG;
  if (src_dtype != TQ_BF16 && src_dtype != TQ_F32) return TQ_ERR_INVALID_ARG;
  if (W > 0 && src_dtype != TQ_BF16) return TQ_ERR_UNSUPPORTED;    // the ring is bf16
  const int esz = src_dtype == TQ_F32 ? 4 : 2;
  if (!aligned16(k_new) || !aligned16(v_new)) return TQ_ERR_ALIGNMENT;
  for (int i = 0; i < 2; ++i)
    if (src_strides[i] < 0 || (src_strides[i] * esz) % 16 != 0) return TQ_ERR_ALIGNMENT;
  DecodeArgs a{};
  bool empty = false;
  const bool one = batch > 0 && n_kv_heads >= 1 && n_q_heads >= n_kv_heads &&
                   step_one_launch(cfg, layer, batch, n_q_heads, n_kv_heads, max_seq_len);
  st = decode_prepare(cfg, tables, layer, q, q_dtype, softmax_scale, batch, n_q_heads, n_kv_heads,
                      1, k, v, k_win, v_win, seq_lens_before, max_seq_len, out, workspace,
                      workspace_bytes, 1, one, &a, &empty);
  if (st != TQ_OK) return st;
  if (empty) return TQ_ERR_INVALID_ARG;              // unreachable with max_seq_len >= 1
  if (!one) {   // see step_one_launch
    // the append kernel, then a plain decode of the grown sequences (which
    // waits for the append at its start)
    st = tq_append_kv(cfg, tables, layer, k_new, v_new, src_dtype, src_strides, batch, n_kv_heads,
                      1, seq_lens_before, k_win, v_win, k, v, stream);
    if (st != TQ_OK) return st;
    return launch_decode(a, stream) == 0 ? TQ_OK : TQ_ERR_CUDA;
  }
  a.fused_step = 1;
  a.knew = k_new;
  a.vnew = v_new;
  a.new_f32 = src_dtype == TQ_F32;
  a.nsb = src_strides[0];
  a.nsh = src_strides[1];
  return launch_decode(a, stream) == 0 ? TQ_OK : TQ_ERR_CUDA;
}

extern "C" int tq_decode_step_launches(const tq_config* cfg, int layer, int batch, int n_q_heads,
                                       int n_kv_heads, int max_seq_len) {
  if (check_config(cfg) != TQ_OK || layer < 0 || layer >= cfg->n_layers || batch < 1 ||
      n_kv_heads < 1 || n_q_heads < n_kv_heads || n_q_heads % n_kv_heads != 0 || max_seq_len < 1)
    return 0;
  const int G = n_q_heads / n_kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8) return 0;   // query groups the decode implements
  return step_one_launch(cfg, layer, batch, n_q_heads, n_kv_heads, max_seq_len) ? 1 : 2;
}

extern "C" tq_status tq_get_device_error(void* stream) {
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return TQ_ERR_CUDA;
  unsigned e1 = 0, e2 = 0;
  if (quant_read_error(&e1) != 0 || decode_read_error(&e2) != 0) return TQ_ERR_CUDA;
  unsigned e = e1 | e2;
  if (e & kErrTimeout) return TQ_ERR_DEVICE_TIMEOUT;
  if (e & kErrBounds) return TQ_ERR_DEVICE_BOUNDS;
  return TQ_OK;
}

extern "C" void tq_set_wait_limit(uint32_t iterations) { g_wait_limit = iterations; }

extern "C" void tq_set_fault_injection(int mode) { g_fault_injection = mode == 1 ? 1u : 0u; }
