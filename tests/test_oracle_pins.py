"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: a value the
pages print (fixtures under tests/golden/, each with its citation), a textbook
table, a closed form, an invariant, a library routine, or brute force on tiny
inputs.  They are chosen so that a plausible slip in the oracle (a dropped
term, a wrong sign or index, a transposed operand, signs applied after the
transform instead of before) fails at least one of them.
"""

import math
import os

import numpy as np
import pytest

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


# ---------------------------------------------------------------- generators

def test_splitmix64_published_vectors():
    for row in _golden_lines("splitmix64_vectors.txt"):
        seed = int(row[1])
        want = [int(v) for v in row[3:]]
        got = [int(v) for v in O.splitmix64_outputs(seed, 0, len(want))]
        assert got == want


def test_splitmix64_vectorised_matches_scalar_definition():
    state = 0xDEADBEEFCAFEF00D
    out = O.splitmix64_outputs(state, 7, 40)
    for i in range(40):
        assert int(out[i]) == O.mix64(state + (7 + i + 1) * O.GOLDEN_GAMMA)


def test_rotation_signs_are_balanced_and_distinct_per_layer_and_kind():
    s = O.rotation_signs(0, 0, O.KIND_K, 4096)
    assert set(np.unique(s)) <= {-1.0, 1.0}
    assert abs(s.mean()) < 4 / math.sqrt(4096)
    a = O.rotation_signs(0, 0, O.KIND_K, 128)
    b = O.rotation_signs(0, 0, O.KIND_V, 128)
    c = O.rotation_signs(0, 1, O.KIND_K, 128)
    d = O.rotation_signs(1, 0, O.KIND_K, 128)
    assert not np.array_equal(a, b) and not np.array_equal(a, c) and not np.array_equal(a, d)
    assert np.array_equal(a, O.rotation_signs(0, 0, O.KIND_K, 128))


def test_round_to_bf16_matches_torch_round_to_nearest_even():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(5)
    x = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-6, 6, 20000),
                        1 + np.array([2.0 ** -8, 3 * 2.0 ** -8, -2.0 ** -9])])
    ours = O.round_to_bf16(x)
    ref = torch.tensor(x.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(ours, ref)
    # ties go to the even mantissa
    assert O.round_to_bf16(np.array([1 + 2.0 ** -8]))[0] == 1.0
    assert O.round_to_bf16(np.array([1 + 3 * 2.0 ** -8]))[0] == 1 + 2.0 ** -6


def test_qjl_matrix_is_standard_gaussian_in_bf16():
    from scipy import stats
    S = O.qjl_matrix(0, 5, 256, 128)
    assert S.shape == (256, 128)
    assert np.array_equal(O.round_to_bf16(S), S)          # exactly bf16
    n = S.size
    assert abs(S.mean()) < 4 / math.sqrt(n)
    assert abs(S.var() - 1.0) < 4 * math.sqrt(2.0 / n)
    assert stats.kstest(S.ravel(), "norm").pvalue > 1e-3
    assert not np.array_equal(S[:128], O.qjl_matrix(0, 6, 128, 128))


# ------------------------------------------------------------------ rotation

def _butterfly_wht(v):
    """Independent in-place fast Walsh-Hadamard transform (natural order)."""
    v = np.array(v, dtype=np.float64)
    h = 1
    n = v.shape[-1]
    while h < n:
        for i in range(0, n, 2 * h):
            a = v[..., i:i + h].copy()
            b = v[..., i + h:i + 2 * h].copy()
            v[..., i:i + h] = a + b
            v[..., i + h:i + 2 * h] = a - b
        h *= 2
    return v


def test_hadamard_small_cases_and_library():
    from scipy.linalg import hadamard as scipy_hadamard
    assert np.array_equal(O.hadamard(1), [[1.0]])
    assert np.array_equal(O.hadamard(2), [[1.0, 1.0], [1.0, -1.0]])
    for d in (4, 8, 16, 128):
        H = O.hadamard(d)
        assert np.array_equal(H, scipy_hadamard(d))
        assert np.array_equal(H @ H.T, d * np.eye(d))


def test_rotation_is_orthogonal_and_sign_flip_comes_first():
    rng = np.random.default_rng(1)
    for d in (2, 4, 16, 128):
        s = O.rotation_signs(3, 2, O.KIND_K, d)
        R = O.rotation_matrix(s)
        assert np.allclose(R.T @ R, np.eye(d), atol=1e-13)
        a, b = rng.standard_normal((2, d))
        ya, yb = O.rotate(a, s), O.rotate(b, s)
        assert abs(np.linalg.norm(ya) - np.linalg.norm(a)) < 1e-13 * np.linalg.norm(a)
        assert abs(ya @ yb - a @ b) < 1e-12 * np.linalg.norm(a) * np.linalg.norm(b)
        # y = (1/sqrt d) H (s * u): compare with an independent butterfly
        assert np.allclose(ya, _butterfly_wht(s * a) / math.sqrt(d), atol=1e-13)
        assert np.allclose(O.inverse_rotate(ya, s), a, atol=1e-13)
    # d = 2 by hand: s = (+1, -1), u = (0.6, 0.8) -> (1/sqrt2)(0.6-0.8, 0.6+0.8)
    y = O.rotate(np.array([0.6, 0.8]), np.array([1.0, -1.0]))
    assert np.allclose(y, np.array([-0.2, 1.4]) / math.sqrt(2), atol=1e-15)


# ------------------------------------------------------------------ codebook

def _max_table():
    rows = {}
    for row in _golden_lines("max1960_gaussian.txt"):
        bits = int(row[1])
        i_c, i_b, i_m = row.index("centroids"), row.index("boundaries"), row.index("mse")
        rows[bits] = ([float(v) for v in row[i_c + 1:i_b]],
                      [float(v) for v in row[i_b + 1:i_m]], float(row[i_m + 1]))
    return rows


def test_codebook_matches_max_1960_table_and_closed_form():
    for bits, (cent, bnd, mse) in _max_table().items():
        c, beta = O.lloyd_max_gaussian(bits)
        L = 1 << bits
        assert np.allclose(c[L // 2:], cent, rtol=6e-4, atol=0)
        assert np.allclose(beta[L // 2:], bnd, rtol=6e-4, atol=0)
        assert abs(O.gaussian_distortion(bits) - mse) < 6e-4 * mse
    c1, _ = O.lloyd_max_gaussian(1)
    assert abs(c1[1] - math.sqrt(2 / math.pi)) < 1e-15
    assert abs(O.gaussian_distortion(1) - (1 - 2 / math.pi)) < 1e-15


@pytest.mark.parametrize("bits", [1, 2, 3, 4, 8])
def test_codebook_meets_centroid_and_midpoint_conditions(bits):
    from scipy import integrate
    c, beta = O.lloyd_max_gaussian(bits)
    L = 1 << bits
    assert np.all(np.diff(c) > 0) and np.all(np.diff(beta) > 0)
    assert np.array_equal(c, -c[::-1])
    assert np.allclose(beta, 0.5 * (c[:-1] + c[1:]), rtol=0, atol=1e-15)
    edges = np.concatenate([[-np.inf], beta, [np.inf]])
    phi = lambda x: math.exp(-x * x / 2) / math.sqrt(2 * math.pi)
    # independent quadrature of E[Z | cell]
    for j in range(L // 2, L):
        lo, hi = edges[j], edges[j + 1]
        mass = integrate.quad(phi, lo, hi, epsabs=0, epsrel=1e-13)[0]
        first = integrate.quad(lambda x: x * phi(x), lo, hi, epsabs=0, epsrel=1e-13)[0]
        assert abs(first / mass - c[j]) < 1e-10 * max(1.0, abs(c[j]))


def test_distortion_closed_form_matches_quadrature():
    from scipy import integrate
    for bits in (1, 2, 3, 4):
        c, beta = O.lloyd_max_gaussian(bits)
        edges = np.concatenate([[-np.inf], beta, [np.inf]])
        phi = lambda x: math.exp(-x * x / 2) / math.sqrt(2 * math.pi)
        D = sum(integrate.quad(lambda x, cj=cj: (x - cj) ** 2 * phi(x), lo, hi, epsrel=1e-12)[0]
                for cj, lo, hi in zip(c, edges[:-1], edges[1:]))
        assert abs(D - O.gaussian_distortion(bits)) < 1e-10


def test_codebook_fp32_scales_to_coordinate_density():
    c32, b32 = O.codebook_fp32(3, 128)
    c, beta = O.lloyd_max_gaussian(3)
    assert c32.dtype == np.float32 and b32.dtype == np.float32
    assert np.array_equal(c32, (c / math.sqrt(128)).astype(np.float32))
    assert np.array_equal(b32, (beta / math.sqrt(128)).astype(np.float32))
    assert b32[3] == 0.0


# --------------------------------------------------------------- code search

@pytest.mark.parametrize("bits", [1, 2, 3, 4, 8])
def test_code_search_is_nearest_centroid_on_tiny_inputs(bits):
    for d in (2, 4, 8, 16):
        c32, b32 = O.codebook_fp32(bits, d)
        s = O.rotation_signs(0, 0, O.KIND_K, d)
        rng = np.random.default_rng(d * 10 + bits)
        X = rng.standard_normal((3000, d))
        q = O.quantize_vectors(X, c32, b32, s)
        y32 = q["y"].astype(np.float32).astype(np.float64)
        brute = np.argmin(np.abs(y32[..., None] - c32.astype(np.float64)), axis=-1)
        far = ~O.near_boundary(q["y"], b32, d, rel=1e-6)
        assert np.array_equal(q["codes"][far], brute[far])
        # brute-force count of boundaries strictly below (fp32 decision)
        count = (b32[None, None, :] < q["y"].astype(np.float32)[..., None]).sum(-1)
        assert np.array_equal(q["codes"], count)


def test_code_search_exhaustive_grid_and_tie_rule():
    d = 4
    for bits in (1, 2, 3, 4):
        c32, b32 = O.codebook_fp32(bits, d)
        # exact boundary values take the lower code; one ulp above takes the upper
        for j, beta in enumerate(b32):
            assert np.searchsorted(b32, beta, side="left") == j
            up = np.nextafter(beta, np.float32(np.inf))
            assert int((b32 < up).sum()) == j + 1
        grid = np.linspace(-3, 3, 6001).astype(np.float32) / np.float32(math.sqrt(d))
        idx = np.array([int((b32 < y).sum()) for y in grid])
        mid = 0.5 * (c32[:-1].astype(np.float64) + c32[1:])
        brute = np.array([int(np.argmin(np.abs(float(y) - c32.astype(np.float64)))) for y in grid])
        ok = np.min(np.abs(grid[:, None].astype(np.float64) - mid[None, :]), axis=1) > 1e-6
        assert np.array_equal(idx[ok], brute[ok])


def test_quantize_hand_case_d2_and_zero_vector():
    c32, b32 = O.codebook_fp32(2, 2)
    s = np.array([1.0, -1.0])
    q = O.quantize_vectors(np.array([[3.0, 4.0], [0.0, 0.0]]), c32, b32, s)
    assert q["norms"][0] == np.float32(5.0)
    assert np.allclose(q["y"][0], np.array([-0.2, 1.4]) / math.sqrt(2), atol=1e-15)
    assert q["norms"][1] == 0.0 and np.all(q["y"][1] == 0.0)
    # y = 0 lies on the middle boundary, so the tie rule gives the lower code
    assert np.all(q["codes"][1] == (1 << 2) // 2 - 1)
    assert np.all(O.dequantize(q["codes"][1:], q["norms"][1:], c32, s) == 0.0)


def test_quantize_is_scale_invariant_in_codes():
    c32, b32 = O.codebook_fp32(4, 128)
    s = O.rotation_signs(0, 0, O.KIND_K, 128)
    X = np.random.default_rng(2).standard_normal((200, 128))
    a = O.quantize_vectors(X, c32, b32, s)
    b = O.quantize_vectors(X * 4.0, c32, b32, s)     # power of two: exact
    assert np.array_equal(a["codes"], b["codes"])
    assert np.array_equal(b["norms"], a["norms"] * 4)


# ------------------------------------------------------------------- packing

def test_packing_matches_page_52_bytes_and_hand_example():
    row = {r[0]: r[1:] for r in _golden_lines("packing_3bit_d128.txt")}
    bits, d = int(row["bits"][0]), int(row["d"][0])
    codes = np.tile([int(v) for v in row["codes_pattern"]], d // 8)
    packed = O.pack_codes(codes, bits)
    assert packed.shape == (int(row["code_bytes"][0]),)
    assert packed.size + int(row["norm_bytes"][0]) == int(row["total_bytes"][0]) == 52
    pattern = [int(v, 16) for v in row["bytes_pattern"]]
    assert list(packed) == pattern * (packed.size // 3)


@pytest.mark.parametrize("bits", [1, 2, 3, 4, 8])
def test_packing_round_trip_and_numpy_packbits(bits):
    rng = np.random.default_rng(bits)
    codes = rng.integers(0, 1 << bits, size=(50, 128))
    packed = O.pack_codes(codes, bits)
    assert packed.shape == (50, 128 * bits // 8)
    assert np.array_equal(O.unpack_codes(packed, bits, 128), codes)
    # independent: expand each code LSB-first into bits, let numpy pack them
    bitmat = ((codes[..., None] >> np.arange(bits)) & 1).reshape(50, -1).astype(np.uint8)
    assert np.array_equal(np.packbits(bitmat, axis=-1, bitorder="little"), packed)


# ---------------------------------------------------------------- distortion

@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_mean_distortion_of_unit_vectors_matches_max(bits):
    d = 128
    c32, b32 = O.codebook_fp32(bits, d)
    s = O.rotation_signs(7, 3, O.KIND_V, d)
    X = np.random.default_rng(100 + bits).standard_normal((20000, d))
    q = O.quantize_vectors(X, c32, b32, s)
    U = X / np.linalg.norm(X, axis=1, keepdims=True)
    Uhat = O.dequantize(q["codes"], np.ones(len(X), np.float32), c32, s)
    D = np.mean(np.sum((U - Uhat) ** 2, axis=1))
    assert abs(D - O.gaussian_distortion(bits)) < 0.03 * O.gaussian_distortion(bits)


# ----------------------------------------------------------------------- QJL

def test_qjl_estimator_is_unbiased_with_the_closed_form_variance():
    d, m, n_seeds = 128, 128, 1500
    rng = np.random.default_rng(11)
    q = rng.standard_normal(d)
    r = 0.3 * q + rng.standard_normal(d)      # correlated, so <q, r> is sizeable
    truth = q @ r
    est = np.empty(n_seeds)
    for k in range(n_seeds):
        S = O.qjl_matrix(1000 + k, 0, m, d)
        bits, gamma, _ = O.qjl_sketch(r, S)
        est[k] = O.qjl_inner_product_estimate(q, bits, float(np.linalg.norm(r)), S)
    var = ((math.pi / 2) * (q @ q) * (r @ r) - truth ** 2) / m
    assert abs(est.mean() - truth) < 4 * math.sqrt(var / n_seeds)
    assert abs(est.var() / var - 1) < 0.15


def test_qjl_sign_convention_and_residual():
    S = O.qjl_matrix(0, 0, 8, 4)
    r = np.zeros(4)
    bits, gamma, z = O.qjl_sketch(r, S)
    assert np.all(bits == 1) and gamma == 0.0      # z = 0 counts as non-negative
    c32, b32 = O.codebook_fp32(2, 4)
    y = np.array([[0.1, -0.2, 0.3, 0.05]])
    codes = np.array([[2, 0, 3, 2]])
    res = O.qjl_residual(y, codes, np.array([2.0]), c32)
    assert np.allclose(res, 2.0 * (y - c32.astype(np.float64)[codes]), atol=0)


def test_qjl_reconstruction_is_unbiased():
    d, m = 16, 128
    rng = np.random.default_rng(3)
    x = rng.standard_normal(d)
    c32, b32 = O.codebook_fp32(2, d)
    s = O.rotation_signs(0, 0, O.KIND_K, d)
    q = O.quantize_vectors(x[None], c32, b32, s)
    r = O.qjl_residual(q["y"], q["codes"], q["norm64"], c32)
    recs = []
    for k in range(600):
        S = O.qjl_matrix(5000 + k, 0, m, d)
        bits, gamma, _ = O.qjl_sketch(r, S)
        recs.append(O.dequantize_qjl(q["codes"], q["norm64"], bits, np.linalg.norm(r, axis=-1), c32, s, S)[0])
    recs = np.array(recs)
    se = recs.std(axis=0) / math.sqrt(len(recs))
    assert np.all(np.abs(recs.mean(axis=0) - x) < 5 * se + 1e-12)


# ------------------------------------------------------------------ attention

def test_softmax_worked_example_from_the_page():
    row = {r[0]: r[1:] for r in _golden_lines("softmax_worked_example.txt")}
    p = O.softmax(np.array([float(v) for v in row["scores"]]))
    assert list(np.rint(100 * p).astype(int)) == [int(v) for v in row["percent"]]
    assert abs(p.sum() - 1) < 1e-15


def _small_cache(rng, B=2, Hkv=2, g=2, T=40, d=16, kb=3, vb=2, seed=0, layer=1, k_scale=3.0):
    ck, bk = O.codebook_fp32(kb, d)
    cv, bv = O.codebook_fp32(vb, d)
    sk = O.rotation_signs(seed, layer, O.KIND_K, d)
    sv = O.rotation_signs(seed, layer, O.KIND_V, d)
    K = rng.standard_normal((B, Hkv, T, d)) * k_scale
    V = rng.standard_normal((B, Hkv, T, d))
    qk = O.quantize_vectors(K, ck, bk, sk)
    qv = O.quantize_vectors(V, cv, bv, sv)
    q = rng.standard_normal((B, Hkv * g, d))
    return dict(K=K, V=V, q=q, ck=ck, cv=cv, sk=sk, sv=sv, qk=qk, qv=qv)


def test_decode_equals_attention_over_dequantized_cache():
    """Parseval: scoring in the rotated domain and inverse-rotating the V sum
    equals plain attention over the dequantized K and V."""
    rng = np.random.default_rng(4)
    c = _small_cache(rng)
    T = c["K"].shape[2]
    seq = np.array([T, 17])
    out = O.decode_attention(c["q"], c["qk"]["codes"], c["qk"]["norms"], c["qv"]["codes"],
                             c["qv"]["norms"], c["ck"], c["cv"], c["sk"], c["sv"], seq, 0.25)
    Kh = O.dequantize(c["qk"]["codes"], c["qk"]["norms"], c["ck"], c["sk"])
    Vh = O.dequantize(c["qv"]["codes"], c["qv"]["norms"], c["cv"], c["sv"])
    ref0 = O.exact_attention(c["q"][:1], Kh[:1], Vh[:1], 0.25)
    ref1 = O.exact_attention(c["q"][1:], Kh[1:, :, :17], Vh[1:, :, :17], 0.25)
    assert np.allclose(out[:1], ref0, atol=1e-12, rtol=1e-12)
    assert np.allclose(out[1:], ref1, atol=1e-12, rtol=1e-12)


def test_decode_single_token_equal_scores_and_empty():
    rng = np.random.default_rng(5)
    c = _small_cache(rng, B=1, T=9)
    Vh = O.dequantize(c["qv"]["codes"], c["qv"]["norms"], c["cv"], c["sv"])
    args = (c["qk"]["codes"], c["qk"]["norms"], c["qv"]["codes"], c["qv"]["norms"],
            c["ck"], c["cv"], c["sk"], c["sv"])
    one = O.decode_attention(c["q"], *args, np.array([1]), 1.0)
    assert np.allclose(one[0, 0], Vh[0, 0, 0], atol=1e-13)
    flat = O.decode_attention(np.zeros_like(c["q"]), *args, np.array([9]), 1.0)
    assert np.allclose(flat[0, 0], Vh[0, 0].mean(axis=0), atol=1e-13)
    empty = O.decode_attention(c["q"], *args, np.array([0]), 1.0)
    assert np.all(empty == 0.0)


def test_decode_window_reproduces_exact_attention_and_mixes():
    rng = np.random.default_rng(6)
    B, Hkv, g, d, W = 1, 2, 2, 16, 8
    c = _small_cache(rng, B=B, Hkv=Hkv, g=g, T=30, d=d)
    args = (c["qk"]["codes"], c["qk"]["norms"], c["qv"]["codes"], c["qv"]["norms"],
            c["ck"], c["cv"], c["sk"], c["sv"])
    # window ring: slot t mod W holds token t for the last W tokens
    for T in (5, 8, 30):
        kw = np.zeros((B, Hkv, W, d))
        vw = np.zeros((B, Hkv, W, d))
        for t in range(max(T - W, 0), T):
            kw[:, :, t % W] = c["K"][:, :, t]
            vw[:, :, t % W] = c["V"][:, :, t]
        out = O.decode_attention(c["q"], *args, np.array([T]), 0.5, window=W, k_win=kw, v_win=vw)
        nq = max(T - W, 0)
        Kh = O.dequantize(c["qk"]["codes"], c["qk"]["norms"], c["ck"], c["sk"])[:, :, :nq]
        Vh = O.dequantize(c["qv"]["codes"], c["qv"]["norms"], c["cv"], c["sv"])[:, :, :nq]
        Kc = np.concatenate([Kh, c["K"][:, :, nq:T]], axis=2)
        Vc = np.concatenate([Vh, c["V"][:, :, nq:T]], axis=2)
        assert np.allclose(out, O.exact_attention(c["q"], Kc, Vc, 0.5), atol=1e-12)
        if T <= W:
            assert np.allclose(out, O.exact_attention(c["q"], c["K"][:, :, :T], c["V"][:, :, :T], 0.5),
                               atol=1e-12)


def test_decode_qjl_term_equals_attention_over_qjl_reconstruction():
    rng = np.random.default_rng(7)
    c = _small_cache(rng, B=1, Hkv=1, g=3, T=25, d=16, kb=2, vb=3)
    m = 32
    S = O.qjl_matrix(0, 1, m, 16)
    r = O.qjl_residual(c["qk"]["y"], c["qk"]["codes"], c["qk"]["norm64"], c["ck"])
    bits, gamma, _ = O.qjl_sketch(r, S)
    qjl = dict(bits=bits, gamma=gamma, S=S)
    out = O.decode_attention(c["q"], c["qk"]["codes"], c["qk"]["norms"], c["qv"]["codes"],
                             c["qv"]["norms"], c["ck"], c["cv"], c["sk"], c["sv"],
                             np.array([25]), 0.3, qjl=qjl)
    Kh = O.dequantize_qjl(c["qk"]["codes"], c["qk"]["norms"], bits, gamma, c["ck"], c["sk"], S)
    Vh = O.dequantize(c["qv"]["codes"], c["qv"]["norms"], c["cv"], c["sv"])
    assert np.allclose(out, O.exact_attention(c["q"], Kh, Vh, 0.3), atol=1e-12)


def test_decode_at_8_bits_is_close_to_exact_attention():
    rng = np.random.default_rng(8)
    # unit-variance scores, so the comparison measures the codec, not softmax gain
    c = _small_cache(rng, B=1, Hkv=2, g=2, T=200, d=128, kb=8, vb=8, k_scale=1.0)
    out = O.decode_attention(c["q"], c["qk"]["codes"], c["qk"]["norms"], c["qv"]["codes"],
                             c["qv"]["norms"], c["ck"], c["cv"], c["sk"], c["sv"],
                             np.array([200]), 1 / math.sqrt(128))
    ref = O.exact_attention(c["q"], c["K"], c["V"], 1 / math.sqrt(128))
    # 8-bit distortion is sqrt(D_8) ~ 0.65 % per vector; the output is a convex
    # combination of values, so measure its error against the value scale
    vscale = np.linalg.norm(c["V"], axis=-1).mean()
    err = np.linalg.norm(out - ref, axis=-1) / vscale
    assert err.max() < 1e-2
    # and 8 bits must beat 3 bits by a wide margin
    c3 = dict(c)
    ck3, bk3 = O.codebook_fp32(3, 128)
    cv3, bv3 = O.codebook_fp32(3, 128)
    qk3 = O.quantize_vectors(c["K"], ck3, bk3, c["sk"])
    qv3 = O.quantize_vectors(c["V"], cv3, bv3, c["sv"])
    out3 = O.decode_attention(c["q"], qk3["codes"], qk3["norms"], qv3["codes"], qv3["norms"],
                              ck3, cv3, c["sk"], c["sv"], np.array([200]), 1 / math.sqrt(128))
    assert np.linalg.norm(out3 - ref) > 5 * np.linalg.norm(out - ref)


def test_protected_layer_table():
    table = [O.layer_bits(l, 36, 4, 2, False, 4, 4) for l in range(36)]
    assert all(t == (8, 8, False) for t in table[:4] + table[32:])
    assert all(t == (4, 2, False) for t in table[4:32])
    assert O.layer_bits(10, 36, 2, 3, True, 4, 4) == (2, 3, True)


# ---------------------------------------------------------------- sphere density
# Lloyd-Max on the exact density of one coordinate of a uniform unit vector,
# f(y) = (1 - y^2)^((d-3)/2) / B(1/2, (d-1)/2): the pins below come from
# outside the oracle's own formulas (scipy quadrature, the uniform and
# Gaussian limits), not from its incomplete-beta or closed-form moments.

@pytest.mark.parametrize("bits", [1, 2, 3, 4, 8])
def test_sphere_codebook_at_d3_is_the_uniform_quantizer(bits):
    # d = 3: f = 1/2 on [-1, 1] (Archimedes), whose Lloyd-Max quantizer is the
    # uniform one: centroids -1 + (2j+1)/L, boundaries -1 + 2(j+1)/L
    c, beta = O.lloyd_max_sphere(bits, 3)
    L = 1 << bits
    j = np.arange(L)
    # (incomplete-beta and moment round-off: ~1e-12 at 256 levels)
    assert np.allclose(c, -1 + (2 * j + 1) / L, atol=1e-11, rtol=0)
    assert np.allclose(beta, -1 + 2 * (j[:-1] + 1) / L, atol=1e-11, rtol=0)


@pytest.mark.parametrize("d", [4, 8, 128])
def test_sphere_pdf_integrates_to_one_and_has_variance_1_over_d(d):
    from scipy.integrate import quad
    mass, _ = quad(lambda y: O.sphere_pdf(y, d), -1, 1, epsabs=1e-14, epsrel=1e-13, limit=200)
    var, _ = quad(lambda y: y * y * O.sphere_pdf(y, d), -1, 1, epsabs=1e-14, epsrel=1e-13,
                  limit=200)
    assert abs(mass - 1) < 1e-10
    assert abs(var - 1.0 / d) < 1e-10 / d        # E[y_i^2] = 1/d by symmetry of the sphere


@pytest.mark.parametrize("d,bits", [(8, 2), (8, 4), (128, 2), (128, 4), (64, 3)])
def test_sphere_codebook_meets_centroid_condition_by_quadrature(d, bits):
    from scipy.integrate import quad
    c, beta = O.lloyd_max_sphere(bits, d)
    edges = [-1.0] + list(beta) + [1.0]
    for j, cj in enumerate(c):
        num, _ = quad(lambda y: y * O.sphere_pdf(y, d), edges[j], edges[j + 1], epsabs=1e-16,
                      epsrel=1e-13, limit=200)
        den, _ = quad(lambda y: O.sphere_pdf(y, d), edges[j], edges[j + 1], epsabs=1e-16,
                      epsrel=1e-13, limit=200)
        assert abs(num / den - cj) < 1e-10 * max(1.0, abs(cj) * d)
    assert np.allclose(beta, 0.5 * (c[:-1] + c[1:]), atol=1e-15)


@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_sphere_codebook_tends_to_the_gaussian_one_for_large_d(bits):
    d = 1 << 16
    c, _ = O.lloyd_max_sphere(bits, d)
    g, _ = O.lloyd_max_gaussian(bits)
    assert np.allclose(c * math.sqrt(d), g, atol=2e-4 * max(1.0, abs(g).max()), rtol=0)


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_sphere_codebook_has_lower_distortion_under_the_true_density(bits):
    # Lloyd-Max optimality: under f, the quantizer designed for f has a lower
    # mean squared error than the N(0, 1/d) one; at d = 128 they are close
    for d, gap in ((16, None), (128, 0.01)):
        cs, bs = O.lloyd_max_sphere(bits, d)
        cg, bg = O.lloyd_max_gaussian(bits)
        cg, bg = cg / math.sqrt(d), bg / math.sqrt(d)
        pdf = lambda y: O.sphere_pdf(y, d)
        ds = O.quantizer_distortion(cs, bs, pdf, -1.0, 1.0)
        dg = O.quantizer_distortion(cg, bg, pdf, -1.0, 1.0)
        assert ds < dg
        if gap is not None:
            assert (dg - ds) / ds < gap


# ------------------------------------------------------------------- Direct Sign
def test_direct_sign_is_exact_when_all_residual_coordinates_have_equal_magnitude():
    rng = np.random.default_rng(31)
    s = np.where(rng.random(128) < 0.5, -1.0, 1.0)
    r = 0.37 * s
    q = rng.standard_normal(128)
    bits, a = O.direct_sign_sketch(r)
    assert np.array_equal(bits, (s > 0).astype(np.int64))
    assert O.direct_sign_estimate(q, bits, a) == pytest.approx(q @ r, rel=1e-6)


def test_direct_sign_scale_is_the_least_squares_one():
    # a = mean|r| minimises ||r - a sign(r)||^2; check against a 1-D search
    r = np.random.default_rng(32).standard_normal((3, 128))
    bits, a = O.direct_sign_sketch(r)
    sgn = 2.0 * bits - 1.0
    for k in range(3):
        grid = np.linspace(0.5 * a[k], 1.5 * a[k], 2001)
        err = [np.sum((r[k] - g * sgn[k]) ** 2) for g in grid]
        assert abs(grid[int(np.argmin(err))] - a[k]) <= 1e-3 * a[k]


def test_direct_sign_error_variance_is_0_23_of_qjl_at_m_equal_d():
    # the pages' ratio (1 - 2/pi)/(pi/2) = 0.231 for Gaussian residual
    # coordinates, measured over 4000 (q, r, S) draws
    rng = np.random.default_rng(33)
    d = 128
    e_ds, e_qjl = [], []
    for _ in range(4000):
        r = rng.standard_normal(d)
        q = rng.standard_normal(d)
        S = rng.standard_normal((d, d))
        bits, a = O.direct_sign_sketch(r)
        e_ds.append(O.direct_sign_estimate(q, bits, a) - q @ r)
        qb, gamma, _ = O.qjl_sketch(r, S)
        e_qjl.append(O.qjl_inner_product_estimate(q, qb, float(np.linalg.norm(r)), S) - q @ r)
    ratio = np.var(e_ds) / np.var(e_qjl)
    assert 0.20 < ratio < 0.26, ratio
    assert (1 - 2 / math.pi) / (math.pi / 2) == pytest.approx(0.2313, abs=1e-4)


# ------------------------------------------------------------ multi-query decode
def _tiny_cache(T, W, d=16, seed=41):
    rng = np.random.default_rng(seed)
    K = rng.standard_normal((1, 1, T, d))
    V = rng.standard_normal((1, 1, T, d))
    ck, bk = O.codebook_fp32(3, d)
    cv, bv = O.codebook_fp32(3, d)
    sk = O.rotation_signs(1, 0, 0, d)
    sv = O.rotation_signs(1, 0, 1, d)
    nq = T - W
    qk = O.quantize_vectors(K[:, :, :nq], ck, bk, sk)
    qv = O.quantize_vectors(V[:, :, :nq], cv, bv, sv)
    kw = np.zeros((1, 1, max(W, 1), d))
    vw = np.zeros_like(kw)
    for t in range(nq, T):
        kw[0, 0, t % W] = K[0, 0, t]
        vw[0, 0, t % W] = V[0, 0, t]
    return dict(K=K, V=V, ck=ck, cv=cv, sk=sk, sv=sv, qk=qk, qv=qv, kw=kw, vw=vw, nq=nq)


def test_multi_query_with_one_query_is_single_query_decode():
    c = _tiny_cache(T=40, W=8)
    q = np.random.default_rng(42).standard_normal((1, 2, 1, 16))
    a = O.decode_attention_multi(q, c["qk"]["codes"], c["qk"]["norms"], c["qv"]["codes"],
                                 c["qv"]["norms"], c["ck"], c["cv"], c["sk"], c["sv"], [40], 0.25,
                                 window=8, k_win=c["kw"], v_win=c["vw"])
    b = O.decode_attention(q[:, :, 0], c["qk"]["codes"], c["qk"]["norms"], c["qv"]["codes"],
                           c["qv"]["norms"], c["ck"], c["cv"], c["sk"], c["sv"], [40], 0.25,
                           window=8, k_win=c["kw"], v_win=c["vw"])
    assert np.allclose(a[:, :, 0], b, rtol=0, atol=1e-14)


def test_multi_query_is_causal_over_the_window():
    # query j sees exactly the tokens up to T - n_q + j: with every token in
    # the window (W >= T) this is exact causal attention, brute force
    T, nQ = 12, 3
    c = _tiny_cache(T=T, W=T)
    q = np.random.default_rng(43).standard_normal((1, 1, nQ, 16))
    got = O.decode_attention_multi(q, c["qk"]["codes"], c["qk"]["norms"], c["qv"]["codes"],
                                   c["qv"]["norms"], c["ck"], c["cv"], c["sk"], c["sv"], [T], 0.3,
                                   window=T, k_win=c["kw"], v_win=c["vw"])
    for j in range(nQ):
        last = T - nQ + j
        ref = O.exact_attention(q[:, :, j], c["K"][:, :, :last + 1], c["V"][:, :, :last + 1], 0.3)
        assert np.allclose(got[:, :, j], ref, rtol=0, atol=1e-12)
