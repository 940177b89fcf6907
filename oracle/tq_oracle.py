"""TurboQuant oracle: plain fp64 restatement of quantize, dequantize and decode attention.

TEST INFRASTRUCTURE ONLY -- see the package docstring.  Nothing in the product
path imports this file.

Sources (page title, then section):

* [README]  "TurboQuant KV 캐시 압축 for llama.cpp" (AmesianX/TurboQuant README):
  header (WHT + Lloyd-Max + QJL correction); v1.7.0 "핵심 설계 결정" item 4
  (encoders apply a sign flip then a butterfly WHT, and the decode kernel applies
  the same WHT to Q so the two cancel by Parseval); v1.5.2 "핵심 변경" items 1, 2
  (float accumulation) and 4 (V needs the inverse rotation at the output);
  v1.5.2 attention-sharpening discussion (QJL score term = scale x sum of
  transformed-Q times sign bits); v1.4.2 item 2 (QJL scalar correction from the
  sign bits and the stored residual scale); "QJL 보정 효과" (QJL = TurboQuant_prod,
  a 1-bit residual correction on keys).
* [WRITEUP] "윈도우용 터보퀀트(TurboQuant) 구현을 개선하다": recap (rotate, then
  quantize, plus a 1-bit QJL fix); finding 2 (keys get more bits than values,
  K4/V2); finding 3 (a 3-bit, 128-dim vector packs to 52 bytes); finding 4
  (first and last four layers protected at 8 bits); the English transcript's
  softmax example (10, 10.1, 9.9 -> 33/37/30 %).
* [BLOG]  "[GitHub 탐방] TurboQuant 3-bit KV 캐시 압축 — 단일 GPU 재현 기록":
  "실험 설계" (residual window rw of full-precision recent tokens);
  "GPU 세대가 바뀌면" item (1) (each coordinate maps to one of 2^bits Lloyd-Max
  centroids).

Conventions the pages leave open are fixed here exactly as the CUDA library
fixes them (independently, in its own code); each is listed with its reason in
the design notes:
  rotation y = (1/sqrt(d)) H_d (s * u), Sylvester H, signs per (layer, K|V);
  Lloyd-Max on N(0, 1/d); code = #{boundaries < y} decided in fp32;
  LSB-first dense bit stream; splitmix64 counter streams; QJL matrix rounded
  to bf16; QJL residual taken in the rotated domain.
"""

from __future__ import annotations

import functools
import math
from typing import Optional

import numpy as np

__all__ = [
    "GOLDEN_GAMMA", "mix64", "splitmix64_outputs", "stream_key",
    "PURPOSE_SIGNS", "PURPOSE_QJL", "KIND_K", "KIND_V",
    "rotation_signs", "qjl_matrix", "round_to_bf16", "round_to_fp32",
    "hadamard", "rotation_matrix", "rotate", "inverse_rotate",
    "lloyd_max_gaussian", "codebook_fp32", "gaussian_distortion",
    "sphere_pdf", "lloyd_max_sphere", "codebook_sphere_fp32", "quantizer_distortion",
    "quantize_vectors", "near_boundary", "pack_codes", "unpack_codes",
    "pack_bits", "unpack_bits", "qjl_residual", "qjl_sketch",
    "qjl_inner_product_estimate", "direct_sign_sketch", "direct_sign_estimate", "dequantize", "dequantize_qjl",
    "layer_bits", "softmax", "decode_attention", "decode_attention_multi", "exact_attention",
]

# --------------------------------------------------------------------------
# Seeded generators (splitmix64, Steele/Lea/Flood 2014; finaliser constants as
# published by Vigna).  Both sides implement this from the definition.
# --------------------------------------------------------------------------

GOLDEN_GAMMA = 0x9E3779B97F4A7C15
_M64 = (1 << 64) - 1

PURPOSE_SIGNS = 0
PURPOSE_QJL = 1
KIND_K = 0
KIND_V = 1


def mix64(z: int) -> int:
    """splitmix64 output function on one 64-bit integer."""
    z &= _M64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _M64
    return z ^ (z >> 31)


def splitmix64_outputs(state: int, start: int, count: int) -> np.ndarray:
    """Outputs start .. start+count-1 of splitmix64 seeded with ``state``.

    Output k is mix64(state + (k+1)*gamma): the k-th value the sequential
    generator (state += gamma; return mix64(state)) returns.  Vectorised over k;
    ``mix64`` above is the scalar form the tests compare it with.
    """
    k = np.arange(start, start + count, dtype=np.uint64)
    with np.errstate(over="ignore"):
        # uint64 array arithmetic wraps modulo 2^64, as the definition requires
        z = np.uint64(state & _M64) + (k + np.uint64(1)) * np.uint64(GOLDEN_GAMMA)
        z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
        z = z ^ (z >> np.uint64(31))
    return z


def stream_key(seed: int, layer: int, kind: int, purpose: int) -> int:
    """Key of the counter stream for (layer, K|V, purpose): output number
    tag = layer*256 + purpose*16 + kind of splitmix64 seeded with ``seed``."""
    tag = (layer << 8) | (purpose << 4) | kind
    return int(splitmix64_outputs(seed & _M64, tag, 1)[0])


def rotation_signs(seed: int, layer: int, kind: int, d: int) -> np.ndarray:
    """The +-1 vector s of the random-sign WHT ([README] v1.7.0 item 4, the
    encoders' internal sign flip).  s_i = +1 when bit 0 of output i is 0."""
    key = stream_key(seed, layer, kind, PURPOSE_SIGNS)
    bits = splitmix64_outputs(key, 0, d) & np.uint64(1)
    return np.where(bits == 0, 1.0, -1.0)


def round_to_fp32(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64).astype(np.float32)


def round_to_bf16(x) -> np.ndarray:
    """fp64 -> fp32 (round to nearest even) -> bf16 (round to nearest even),
    returned as fp64 values.  Written out on the bit pattern."""
    f = round_to_fp32(x)
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    u = (u + np.uint64(0x7FFF) + lsb) & np.uint64(0xFFFF0000)
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


def qjl_matrix(seed: int, layer: int, m: int, d: int) -> np.ndarray:
    """Dense Gaussian QJL projection S (m x d), entries rounded to bf16.

    Entry e = j*d + k takes outputs 2e and 2e+1 of the stream (layer, K, QJL):
    u1 = ((o >> 11) + 0.5) * 2^-53 in (0,1), u2 = (o' >> 11) * 2^-53, and
    g = sqrt(-2 ln u1) cos(2 pi u2) (Box-Muller, cosine branch).
    """
    key = stream_key(seed, layer, KIND_K, PURPOSE_QJL)
    o = splitmix64_outputs(key, 0, 2 * m * d)
    a = (o[0::2] >> np.uint64(11)).astype(np.float64)
    b = (o[1::2] >> np.uint64(11)).astype(np.float64)
    u1 = (a + 0.5) * 2.0 ** -53
    u2 = b * 2.0 ** -53
    g = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)
    return round_to_bf16(g).reshape(m, d)


# --------------------------------------------------------------------------
# Rotation ([README] v1.7.0 item 4; v1.5.0 Gemma 4 item 2: per-head WHT)
# --------------------------------------------------------------------------

def hadamard(d: int) -> np.ndarray:
    """Dense Sylvester Hadamard matrix, H[i, j] = (-1)^popcount(i & j)."""
    assert d >= 1 and (d & (d - 1)) == 0, "d must be a power of two"
    H = np.empty((d, d))
    for i in range(d):
        for j in range(d):
            H[i, j] = -1.0 if bin(i & j).count("1") % 2 else 1.0
    return H


def rotation_matrix(signs: np.ndarray) -> np.ndarray:
    """R = (1/sqrt(d)) H_d diag(s): sign flip first, then the transform."""
    d = signs.shape[0]
    return hadamard(d) * signs[None, :] / math.sqrt(d)


def rotate(u: np.ndarray, signs: np.ndarray) -> np.ndarray:
    """y = R u for the rows of u (dense matrix product, not a butterfly)."""
    return np.asarray(u, dtype=np.float64) @ rotation_matrix(signs).T


def inverse_rotate(y: np.ndarray, signs: np.ndarray) -> np.ndarray:
    """u = R^T y; R is orthogonal."""
    return np.asarray(y, dtype=np.float64) @ rotation_matrix(signs)


# --------------------------------------------------------------------------
# Lloyd-Max codebook ([BLOG] "GPU 세대" item (1); [README] header)
# --------------------------------------------------------------------------

_SQRT2 = math.sqrt(2.0)
_INV_SQRT_2PI = 1.0 / math.sqrt(2.0 * math.pi)


def _pdf(x: float) -> float:
    return _INV_SQRT_2PI * math.exp(-0.5 * x * x) if math.isfinite(x) else 0.0


def _cell_mass(lo: float, hi: float) -> float:
    """P(lo < Z <= hi) for Z ~ N(0,1), in the form that does not cancel."""
    if lo >= 0.0:
        return 0.5 * (math.erfc(lo / _SQRT2) - (math.erfc(hi / _SQRT2) if math.isfinite(hi) else 0.0))
    if hi <= 0.0:
        return 0.5 * (math.erfc(-hi / _SQRT2) - (math.erfc(-lo / _SQRT2) if math.isfinite(lo) else 0.0))
    return 0.5 * (math.erf(hi / _SQRT2) - math.erf(lo / _SQRT2))


def _normal_quantile(p: float) -> float:
    from statistics import NormalDist
    return NormalDist().inv_cdf(p)


def _lloyd_alternation(c, cell_mean, tol: float, window: int = 5000,
                       max_iter: int = 2_000_000):
    """Lloyd's alternation on the positive half of a symmetric density.

    ``c`` holds the L/2 positive centroids in increasing order.  One pass
    applies the two optimality conditions in turn:
      midpoint condition:  beta_j = (c_j + c_{j+1}) / 2,
      centroid condition:  c_j = E[Y | beta_{j-1} < Y <= beta_j],
    where the lowest positive cell starts at the middle boundary 0 (symmetry
    puts it there) and the highest one ends at the top of the support.
    ``cell_mean(edges)`` returns the conditional means of the cells between
    consecutive edges.  The passes stop when no centroid moves by more than
    ``tol``, or, once the moves have reached the fp64 rounding floor (6 bits
    and up), when the largest move has not shrunk by 10 % for ``window``
    passes.  Returns (centroids, passes)."""
    best, best_pass = math.inf, 0
    passes = 0
    for passes in range(1, max_iter + 1):
        beta = 0.5 * (c[:-1] + c[1:])
        new = cell_mean(np.concatenate([[0.0], beta, [np.inf]]))
        step = float(np.max(np.abs(new - c)))
        c = new
        if step <= tol:
            break
        if step < 0.9 * best:
            best, best_pass = step, passes
        elif passes - best_pass > window:
            break
    return c, passes


def _gaussian_cell_means(edges: np.ndarray) -> np.ndarray:
    """E[Z | lo < Z <= hi] for Z ~ N(0,1) on cells of the positive half line:
    (phi(lo) - phi(hi)) / (Phi(hi) - Phi(lo)), both differences taken in a
    form that does not cancel (upper-tail erfc; phi(lo) (1 - e^{-(hi-lo)(hi+lo)/2}))."""
    from scipy.special import erfc
    lo, hi = edges[:-1], edges[1:]
    top = np.isfinite(hi)
    h = np.where(top, hi, 0.0)
    tail = erfc(edges / _SQRT2)                 # 2 P(Z > edge); 0 at +inf
    mass = 0.5 * (tail[:-1] - tail[1:])
    dphi = _INV_SQRT_2PI * np.exp(-0.5 * lo * lo) * np.where(
        top, -np.expm1(-0.5 * (h - lo) * (h + lo)), 1.0)
    return dphi / mass


@functools.lru_cache(maxsize=None)
def _lloyd_max_gaussian_cached(bits: int):
    L = 1 << bits
    H = L // 2
    c = np.array([_normal_quantile((H + j + 0.5) / L) for j in range(H)])
    c, _ = _lloyd_alternation(c, _gaussian_cell_means, 1e-15)
    c = np.concatenate([-c[::-1], c])
    beta = 0.5 * (c[:-1] + c[1:])
    beta[H - 1] = 0.0
    return c, beta


def lloyd_max_gaussian(bits: int):
    """Lloyd-Max quantizer of N(0, 1), in fp64.

    The quantizer meets the midpoint and centroid conditions of
    ``_lloyd_alternation``; for a log-concave density their solution is
    unique.  The density is symmetric, so the middle boundary is 0 and
    c_{L-1-j} = -c_j: the alternation runs on the L/2 positive cells, from
    the quantile midpoints c_j = Phi^{-1}((j + 1/2) / L), until no centroid
    moves by more than 1e-15 (or the moves reach the fp64 rounding floor,
    about 1e-14 at 6-8 bits; 8 bits takes about 1.7e5 passes).
    Returns (centroids[L], boundaries[L-1]) for unit variance (copies of a
    per-process cache)."""
    c, beta = _lloyd_max_gaussian_cached(int(bits))
    return c.copy(), beta.copy()


def codebook_fp32(bits: int, d: int):
    """Codebook for the rotated-coordinate density N(0, 1/d), rounded to fp32.

    centroids = fp32(sigma * c), boundaries = fp32(sigma * beta) with
    sigma = 1/sqrt(d), each rounded once from fp64.  Returns fp32 arrays.
    """
    c, beta = lloyd_max_gaussian(bits)
    sigma = 1.0 / math.sqrt(d)
    return round_to_fp32(c * sigma), round_to_fp32(beta * sigma)


# --------------------------------------------------------------------------
# Exact rotated-coordinate density (the "sphere" codebook).  A coordinate y of
# a uniformly random unit vector in R^d has density
#   f(y) = (1 - y^2)^((d-3)/2) / B(1/2, (d-1)/2),  -1 <= y <= 1,
# which tends to N(0, 1/d) as d grows.  Lloyd-Max on f is the alternative
# reading of "Lloyd-Max on the rotated-coordinate density" to N(0, 1/d).
# --------------------------------------------------------------------------

def _sphere_log_norm(d: int) -> float:
    from scipy.special import gammaln
    return gammaln(d / 2.0) - gammaln(0.5) - gammaln((d - 1) / 2.0)


def sphere_pdf(y, d: int):
    """Density of one coordinate of a uniform unit vector in R^d."""
    y = np.asarray(y, dtype=np.float64)
    return np.exp(_sphere_log_norm(d)) * np.clip(1.0 - y * y, 0.0, None) ** ((d - 3) / 2.0)


def _sphere_first_moment_terms(y: np.ndarray, d: int) -> np.ndarray:
    """(1 - y^2)^((d-1)/2) C_d / (d - 1): int_lo^hi y f(y) dy is its value at lo
    minus its value at hi (the antiderivative of y (1 - y^2)^k is
    -(1 - y^2)^(k+1) / (2 (k+1)))."""
    return math.exp(_sphere_log_norm(d)) / (d - 1) * np.clip(1.0 - y * y, 0.0, None) ** ((d - 1) / 2.0)


def _sphere_cell_means(d: int):
    """Cell means E[Y | lo < Y <= hi] under the sphere-coordinate density on
    cells of [0, 1]: the mass from the regularized incomplete beta function,
    P(Y > y) = I_{1-y^2}((d-1)/2, 1/2) / 2 for y >= 0 (upper tail, no
    cancellation), and the first moment in closed form
    (_sphere_first_moment_terms)."""
    from scipy.special import betaincc
    a, b = 0.5, (d - 1) / 2.0

    def means(edges: np.ndarray) -> np.ndarray:
        y = np.minimum(edges, 1.0)
        tail = betaincc(a, b, y * y)            # 2 P(Y > y)
        mass = 0.5 * (tail[:-1] - tail[1:])
        g = _sphere_first_moment_terms(y, d)
        return (g[:-1] - g[1:]) / mass
    return means


@functools.lru_cache(maxsize=None)
def _lloyd_max_sphere_cached(bits: int, d: int):
    L = 1 << bits
    H = L // 2
    if d <= 16:      # far from Gaussian: start from the uniform quantizer of [-1, 1]
        c = np.array([-1.0 + (2 * (H + j) + 1) / L for j in range(H)])
    else:
        g, _ = lloyd_max_gaussian(bits)
        c = g[H:] / math.sqrt(d)
    c, _ = _lloyd_alternation(c, _sphere_cell_means(d), 1e-15 / math.sqrt(d))
    c = np.concatenate([-c[::-1], c])
    beta = 0.5 * (c[:-1] + c[1:])
    beta[H - 1] = 0.0
    return c, beta


def lloyd_max_sphere(bits: int, d: int):
    """Lloyd-Max quantizer of the sphere-coordinate density f (above), fp64.

    The same midpoint and centroid conditions as lloyd_max_gaussian, with
    cells [-1, beta_0], ..., [beta_{L-2}, 1], by the same alternation on the
    positive half (f is symmetric), until no centroid moves by more than
    1e-15 / sqrt(d) (or the rounding floor is reached).  Starting point: the
    uniform quantizer of [-1, 1] for d <= 16, else the N(0, 1/d) quantizer.
    At 256 levels this takes about 1.2e5-1.5e5 passes.
    Returns (centroids[L], boundaries[L-1]) in units of y (not scaled;
    copies of a per-process cache)."""
    c, beta = _lloyd_max_sphere_cached(int(bits), int(d))
    return c.copy(), beta.copy()


def codebook_sphere_fp32(bits: int, d: int):
    """Sphere-density codebook rounded to fp32 (centroids, boundaries)."""
    c, beta = lloyd_max_sphere(bits, d)
    return round_to_fp32(c), round_to_fp32(beta)


def quantizer_distortion(c, beta, pdf, lo=-np.inf, hi=np.inf) -> float:
    """E[(Y - Q(Y))^2] under density pdf for the quantizer (c, beta), by
    adaptive quadrature cell by cell (scipy.integrate.quad)."""
    from scipy.integrate import quad
    edges = [lo] + list(np.asarray(beta, dtype=np.float64)) + [hi]
    total = 0.0
    for j, cj in enumerate(np.asarray(c, dtype=np.float64)):
        v, _ = quad(lambda y: (y - cj) ** 2 * pdf(y), edges[j], edges[j + 1], limit=200,
                    epsabs=1e-15, epsrel=1e-12)
        total += v
    return total


def gaussian_distortion(bits: int) -> float:
    """E[(Z - Q(Z))^2] for Z ~ N(0,1) under the Lloyd-Max quantizer, by
    integrating each cell in closed form:
      E[Z^2; cell] = (Phi(hi)-Phi(lo)) + lo phi(lo) - hi phi(hi),
    so D = E[Z^2] - sum_j P_j c_j^2 (the centroid condition makes the cross term
    equal to sum_j P_j c_j^2)."""
    c, beta = lloyd_max_gaussian(bits)
    L = len(c)
    lo = [-math.inf] + list(beta)
    hi = list(beta) + [math.inf]
    total = 0.0
    for j in range(L):
        P = _cell_mass(lo[j], hi[j])
        total += P * c[j] ** 2
    return 1.0 - total


# --------------------------------------------------------------------------
# Quantize: norm, rotate, code search ([WRITEUP] recap; [README] v1.7.0 item 4)
# --------------------------------------------------------------------------

def quantize_vectors(X: np.ndarray, centroids32: np.ndarray, boundaries32: np.ndarray,
                     signs: np.ndarray):
    """Quantize the rows of X (shape [..., d]).

    n = ||x||_2 (fp64); u = x / n (u = 0 when n = 0); y = R u (fp64);
    code_i = #{j : beta_j < y_i}, the comparison taken in fp32 (y rounded to
    fp32 once, boundaries are the fp32 table), so an exact tie y = beta_j
    takes the lower code.  The norm is stored rounded to fp32.

    Returns dict(codes=int64[..., d], norms=fp32[...], norm64, y=fp64[..., d]).
    """
    X = np.asarray(X, dtype=np.float64)
    n = np.sqrt(np.sum(X * X, axis=-1))
    safe = np.where(n > 0, n, 1.0)
    U = np.where(n[..., None] > 0, X / safe[..., None], 0.0)
    Y = rotate(U, signs)
    y32 = Y.astype(np.float32)
    # count of boundaries strictly below y: a left-sided search in the sorted
    # fp32 boundary table (the tests check it against brute-force counting
    # and nearest-centroid search)
    b32 = np.asarray(boundaries32, dtype=np.float32)
    codes = np.searchsorted(b32, y32, side="left").astype(np.int64)
    return dict(codes=codes, norms=round_to_fp32(n), norm64=n, y=Y)


def near_boundary(y64: np.ndarray, boundaries32: np.ndarray, d: int, rel: float = 1e-6):
    """Mask of coordinates lying within rel * max(|beta_j|, sigma) of some
    boundary (sigma = 1/sqrt(d) floors the scale at the zero boundary)."""
    sigma = 1.0 / math.sqrt(d)
    mask = np.zeros(np.shape(y64), dtype=bool)
    for beta in np.asarray(boundaries32, dtype=np.float64):
        mask |= np.abs(y64 - beta) <= rel * max(abs(beta), sigma)
    return mask


# --------------------------------------------------------------------------
# Bit packing ([WRITEUP] finding 3: 3 bits x 128 = 48 B of codes + 4 B norm)
# --------------------------------------------------------------------------

def pack_codes(codes: np.ndarray, bits: int) -> np.ndarray:
    """Dense LSB-first stream: the code of coordinate i occupies stream bits
    [i*bits, i*bits + bits); stream bit k is bit (k mod 8) of byte k // 8."""
    codes = np.asarray(codes, dtype=np.int64)
    d = codes.shape[-1]
    nbytes = (d * bits + 7) // 8
    flat = codes.reshape(-1, d)
    out = np.zeros((flat.shape[0], nbytes), dtype=np.uint8)
    for i in range(d):
        for t in range(bits):
            k = i * bits + t
            bit = (flat[:, i] >> t) & 1
            out[:, k // 8] |= (bit << (k % 8)).astype(np.uint8)
    return out.reshape(codes.shape[:-1] + (nbytes,))


def unpack_codes(packed: np.ndarray, bits: int, d: int) -> np.ndarray:
    packed = np.asarray(packed, dtype=np.uint8)
    flat = packed.reshape(-1, packed.shape[-1]).astype(np.int64)
    codes = np.zeros((flat.shape[0], d), dtype=np.int64)
    for i in range(d):
        for t in range(bits):
            k = i * bits + t
            codes[:, i] |= ((flat[:, k // 8] >> (k % 8)) & 1) << t
    return codes.reshape(packed.shape[:-1] + (d,))


def pack_bits(b: np.ndarray) -> np.ndarray:
    """Sign bits, LSB-first: bit j -> bit (j mod 8) of byte j // 8."""
    return pack_codes(np.asarray(b, dtype=np.int64), 1)


def unpack_bits(packed: np.ndarray, m: int) -> np.ndarray:
    return unpack_codes(packed, 1, m)


# --------------------------------------------------------------------------
# QJL residual sketch ([README] "QJL 보정 효과", v1.4.2 item 2, v1.5.2
# sharpening text; [WRITEUP] recap and finding 1)
# --------------------------------------------------------------------------

def qjl_residual(y64: np.ndarray, codes: np.ndarray, norm64: np.ndarray,
                 centroids32: np.ndarray) -> np.ndarray:
    """Residual in the rotated domain, at the vector's scale: r = n (y - c[idx])."""
    c = np.asarray(centroids32, dtype=np.float64)
    return np.asarray(norm64, dtype=np.float64)[..., None] * (y64 - c[codes])


def qjl_sketch(r: np.ndarray, S: np.ndarray):
    """bit_j = [ (S r)_j >= 0 ], gamma = ||r||_2 (stored fp32).  Returns
    (bits int64[..., m], gamma fp32[...], z fp64[..., m])."""
    r = np.asarray(r, dtype=np.float64)
    z = r @ np.asarray(S, dtype=np.float64).T
    bits = (z >= 0).astype(np.int64)
    gamma = np.sqrt(np.sum(r * r, axis=-1))
    return bits, round_to_fp32(gamma), z


def qjl_inner_product_estimate(q_rot: np.ndarray, bits: np.ndarray, gamma, S: np.ndarray):
    """Unbiased estimate of <q_rot, r> from the sketch:
    gamma * sqrt(pi/2) / m * sum_j (S q_rot)_j (2 bit_j - 1).
    (For a Gaussian row g: E[sign(g.r) (g.q)] = sqrt(2/pi) <q, r> / ||r||.)"""
    S = np.asarray(S, dtype=np.float64)
    m = S.shape[0]
    sq = np.asarray(q_rot, dtype=np.float64) @ S.T
    sgn = 2.0 * np.asarray(bits, dtype=np.float64) - 1.0
    return np.asarray(gamma, dtype=np.float64) * math.sqrt(math.pi / 2.0) / m * np.sum(sq * sgn, axis=-1)


# --------------------------------------------------------------------------
# Direct Sign residual ([README] v1.1.0 "Direct Sign": at head_dim <= 128 the
# sign of each rotated residual coordinate is stored directly instead of a
# projected sketch; no second transform is needed on the query side)
# --------------------------------------------------------------------------

def direct_sign_sketch(r: np.ndarray):
    """bit_i = [r_i >= 0] for every rotated residual coordinate, and the scale
    a = mean_i |r_i| (stored fp32): the least-squares a for r ~= a (2 bit - 1).
    Returns (bits int64[..., d], scale fp32[...])."""
    r = np.asarray(r, dtype=np.float64)
    bits = (r >= 0).astype(np.int64)
    scale = np.mean(np.abs(r), axis=-1)
    return bits, round_to_fp32(scale)


def direct_sign_estimate(q_rot: np.ndarray, bits: np.ndarray, scale) -> np.ndarray:
    """Estimate of <q_rot, r> from the direct signs: a * sum_i q_i (2 bit_i - 1).
    For residual coordinates ~ N(0, s^2) its error variance per coordinate is
    s^2 (1 - 2/pi), against s^2 pi/2 d/m for the m-row QJL sketch: the ratio
    (1 - 2/pi) / (pi/2) = 0.23 at m = d."""
    sgn = 2.0 * np.asarray(bits, dtype=np.float64) - 1.0
    return np.asarray(scale, dtype=np.float64) * np.sum(np.asarray(q_rot, dtype=np.float64) * sgn,
                                                        axis=-1)


# --------------------------------------------------------------------------
# Dequantize
# --------------------------------------------------------------------------

def dequantize(codes: np.ndarray, norms: np.ndarray, centroids32: np.ndarray,
               signs: np.ndarray) -> np.ndarray:
    """x_hat = n R^T c[idx] (the norm as stored, fp32)."""
    c = np.asarray(centroids32, dtype=np.float64)
    yhat = c[np.asarray(codes)] * np.asarray(norms, dtype=np.float64)[..., None]
    return inverse_rotate(yhat, signs)


def dequantize_qjl(codes, norms, bits, gamma, centroids32, signs, S):
    """MSE part plus the unbiased QJL reconstruction of the residual,
    x_hat = R^T (n c[idx] + sqrt(pi/2)/m * gamma * S^T (2 bit - 1))."""
    S = np.asarray(S, dtype=np.float64)
    m = S.shape[0]
    c = np.asarray(centroids32, dtype=np.float64)
    yhat = c[np.asarray(codes)] * np.asarray(norms, dtype=np.float64)[..., None]
    sgn = 2.0 * np.asarray(bits, dtype=np.float64) - 1.0
    yhat = yhat + (math.sqrt(math.pi / 2.0) / m) * np.asarray(gamma, dtype=np.float64)[..., None] * (sgn @ S)
    return inverse_rotate(yhat, signs)


def layer_bits(layer: int, n_layers: int, k_bits: int, v_bits: int, k_qjl: bool,
               n_protect_first: int, n_protect_last: int, protect_bits: int = 8):
    """Bits per layer ([WRITEUP] finding 4): the first and last protected layers
    use protect_bits for K and V with MSE only; the rest use (k_bits, v_bits)."""
    if layer < n_protect_first or layer >= n_layers - n_protect_last:
        return protect_bits, protect_bits, False
    return k_bits, v_bits, k_qjl


# --------------------------------------------------------------------------
# Decode attention
# --------------------------------------------------------------------------

def softmax(s: np.ndarray) -> np.ndarray:
    s = np.asarray(s, dtype=np.float64)
    e = np.exp(s - np.max(s))
    return e / np.sum(e)


def decode_attention(q, k_codes, k_norms, v_codes, v_norms, ck32, cv32,
                     signs_k, signs_v, seq_lens, scale, window=0,
                     k_win=None, v_win=None, qjl=None, dsign=None):
    """One decode step of attention over a compressed cache.

    q        [B, Hq, d] query values (fp64 copy of the inputs)
    k_codes  [B, Hkv, cap, d] key codes;  k_norms [B, Hkv, cap]
    v_codes, v_norms  likewise for values
    seq_lens [B] tokens per sequence, window included
    window   W: tokens t in [T-W, T) are read from k_win / v_win
             ([B, Hkv, W, d], slot t mod W) in the original domain;
             tokens t < T-W come from the codes.
    qjl      None, or dict(bits=[B,Hkv,cap,m], gamma=[B,Hkv,cap], S=[m,d])
    dsign    None, or dict(bits=[B,Hkv,cap,d], scale=[B,Hkv,cap]): Direct Sign
             keys, s_t += scale * a_t <q_rot, 2 bit_t - 1>

    Per query head h (kv-head h // (Hq/Hkv)):
      q_rot = R_K q;
      quantized token:  s_t = scale * (n_t <q_rot, cK[idx_t]>
                                       + gamma_t sqrt(pi/2)/m <S q_rot, 2 bit_t - 1>);
      window token:     s_t = scale * <q, k_t>;
      p = softmax(s) in fp64;
      o = R_V^T (sum_quantized p_t n^V_t cV[idx^V_t]) + sum_window p_t v_t.
    A sequence of length 0 gives o = 0.  Returns fp64 [B, Hq, d].
    """
    q = np.asarray(q, dtype=np.float64)
    B, Hq, d = q.shape
    Hkv = k_codes.shape[1]
    g = Hq // Hkv
    RK = rotation_matrix(np.asarray(signs_k, dtype=np.float64))
    RV = rotation_matrix(np.asarray(signs_v, dtype=np.float64))
    ck = np.asarray(ck32, dtype=np.float64)
    cv = np.asarray(cv32, dtype=np.float64)
    out = np.zeros((B, Hq, d))
    for b in range(B):
        T = int(seq_lens[b])
        if T <= 0:
            continue
        nq = max(T - window, 0)
        win_tokens = list(range(nq, T))
        for h in range(Hq):
            kh = h // g
            qv = q[b, h]
            q_rot = RK @ qv
            scores = []
            if nq > 0:
                kc = np.asarray(k_codes[b, kh, :nq])
                s_q = np.asarray(k_norms[b, kh, :nq], dtype=np.float64) * (ck[kc] @ q_rot)
                if qjl is not None:
                    S = np.asarray(qjl["S"], dtype=np.float64)
                    m = S.shape[0]
                    sgn = 2.0 * np.asarray(qjl["bits"][b, kh, :nq], dtype=np.float64) - 1.0
                    gam = np.asarray(qjl["gamma"][b, kh, :nq], dtype=np.float64)
                    s_q = s_q + gam * math.sqrt(math.pi / 2.0) / m * (sgn @ (S @ q_rot))
                if dsign is not None:
                    sgn = 2.0 * np.asarray(dsign["bits"][b, kh, :nq], dtype=np.float64) - 1.0
                    a = np.asarray(dsign["scale"][b, kh, :nq], dtype=np.float64)
                    s_q = s_q + a * (sgn @ q_rot)
                scores.append(scale * s_q)
            if win_tokens:
                slots = [t % window for t in win_tokens]
                kw = np.asarray(k_win[b, kh, slots], dtype=np.float64)
                scores.append(scale * (kw @ qv))
            p = softmax(np.concatenate(scores))
            o = np.zeros(d)
            if nq > 0:
                vc = np.asarray(v_codes[b, kh, :nq])
                w = p[:nq] * np.asarray(v_norms[b, kh, :nq], dtype=np.float64)
                o_rot = w @ cv[vc]
                o = o + RV.T @ o_rot
            if win_tokens:
                vw = np.asarray(v_win[b, kh, slots], dtype=np.float64)
                o = o + p[nq:] @ vw
            out[b, h] = o
    return out


def decode_attention_multi(q, k_codes, k_norms, v_codes, v_norms, ck32, cv32,
                           signs_k, signs_v, seq_lens, scale, window=0,
                           k_win=None, v_win=None):
    """Several query tokens per sequence at once (speculative verification,
    chunked decode): q [B, Hq, n_q, d]; query j of sequence b is the token at
    position T_b - n_q + j and attends causally to tokens t <= T_b - n_q + j.
    The cache is the same as for decode_attention (tokens t < T_b - W in the
    codes, the last W in the window ring).  Returns fp64 [B, Hq, n_q, d]."""
    q = np.asarray(q, dtype=np.float64)
    B, Hq, nQ, d = q.shape
    Hkv = k_codes.shape[1]
    g = Hq // Hkv
    RK = rotation_matrix(np.asarray(signs_k, dtype=np.float64))
    RV = rotation_matrix(np.asarray(signs_v, dtype=np.float64))
    ck = np.asarray(ck32, dtype=np.float64)
    cv = np.asarray(cv32, dtype=np.float64)
    out = np.zeros((B, Hq, nQ, d))
    for b in range(B):
        T = int(seq_lens[b])
        nq = max(T - window, 0)
        for h in range(Hq):
            kh = h // g
            for j in range(nQ):
                last = T - nQ + j                  # last visible position
                if last < 0:
                    continue
                qv = q[b, h, j]
                q_rot = RK @ qv
                nqv = min(nq, last + 1)            # visible quantized tokens
                win = [t for t in range(nq, T) if t <= last]
                scores = []
                if nqv > 0:
                    kc = np.asarray(k_codes[b, kh, :nqv])
                    scores.append(scale * np.asarray(k_norms[b, kh, :nqv], dtype=np.float64) *
                                  (ck[kc] @ q_rot))
                if win:
                    kw = np.asarray(k_win[b, kh, [t % window for t in win]], dtype=np.float64)
                    scores.append(scale * (kw @ qv))
                p = softmax(np.concatenate(scores))
                o = np.zeros(d)
                if nqv > 0:
                    vc = np.asarray(v_codes[b, kh, :nqv])
                    w = p[:nqv] * np.asarray(v_norms[b, kh, :nqv], dtype=np.float64)
                    o = o + RV.T @ (w @ cv[vc])
                if win:
                    vw = np.asarray(v_win[b, kh, [t % window for t in win]], dtype=np.float64)
                    o = o + p[nqv:] @ vw
                out[b, h, j] = o
    return out


def exact_attention(q, K, V, scale):
    """Uncompressed softmax attention for one query per head.
    q [B,Hq,d], K,V [B,Hkv,T,d] -> [B,Hq,d], fp64."""
    q = np.asarray(q, dtype=np.float64)
    B, Hq, d = q.shape
    Hkv = K.shape[1]
    g = Hq // Hkv
    out = np.zeros((B, Hq, d))
    for b in range(B):
        for h in range(Hq):
            kh = h // g
            p = softmax(scale * (np.asarray(K[b, kh], dtype=np.float64) @ q[b, h]))
            out[b, h] = p @ np.asarray(V[b, kh], dtype=np.float64)
    return out
