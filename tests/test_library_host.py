"""Host-side checks of the C-ABI library (no GPU needed).

The library must load and export every function include/tq.h declares; its host
functions (codebook, sign vectors, QJL matrix, sizes) must agree with the
independently written oracle; argument validation must reject bad calls before
any launch.
"""

import os
import re

import numpy as np
import pytest

import oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def B():
    from kv_cache_quantization_random_gb300 import binding, build
    build.build()
    binding.load()
    return binding


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "tq.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tq_[a-z_0-9]+)\s*\(", text)))


def test_library_exports_every_declared_symbol(B):
    lib = B.load()
    declared = _declared_functions()
    assert len(declared) >= 15
    missing = [n for n in declared if not hasattr(lib, n)]
    assert not missing, missing
    assert sorted(B.EXPORTED) == declared
    assert lib.tq_version() == 1


@pytest.mark.parametrize("bits", [1, 2, 3, 4, 8])
def test_codebook_matches_oracle(B, bits):
    c, b = B.tq_make_codebook(bits, 128)
    oc, ob = O.codebook_fp32(bits, 128)
    assert np.array_equal(c, oc)
    assert np.array_equal(b, ob)


def test_codebook_other_dims(B):
    for d in (2, 16, 64, 256):
        c, b = B.tq_make_codebook(3, d)
        oc, ob = O.codebook_fp32(3, d)
        assert np.array_equal(c, oc) and np.array_equal(b, ob)


# 256 levels only at the pages' head size: the oracle's alternation needs
# about 1.2e5 passes of incomplete-beta evaluations there (tens of seconds)
@pytest.mark.parametrize("bits,d", [(b, d) for b in (1, 2, 3, 4) for d in (4, 8, 64, 128)]
                         + [(8, 128)])
def test_sphere_codebook_matches_oracle(B, bits, d):
    """fp32 values equal the oracle's, except that at 256 levels (where the
    optimality system is ill-conditioned and the fp64 oracle resolves the
    fixed point to ~1e-10) a value may round to the neighbouring fp32 number
    when the oracle's fp64 value lies within 1e-9 (relative) of the rounding tie."""
    c, b = B.tq_make_codebook(bits, d, density=B.TQ_DENSITY_SPHERE_BETA)
    oc64, ob64 = O.lloyd_max_sphere(bits, d)
    for got, ref64 in ((c, oc64), (b, ob64)):
        ref = ref64.astype(np.float32)
        diff = np.nonzero(got != ref)[0]
        assert bits == 8 or diff.size == 0
        for i in diff:
            nxt = np.nextafter(ref[i], got[i])
            assert got[i] == nxt                              # one ulp apart
            tie = 0.5 * (float(ref[i]) + float(nxt))
            assert abs(ref64[i] - tie) <= 1e-9 * abs(tie)


def test_sign_vectors_match_oracle(B):
    for seed in (0, 1, 123456789123):
        for layer in (0, 5, 35):
            for kind in (0, 1):
                s = B.tq_make_signs(seed, layer, kind, 128)
                assert np.array_equal(s.astype(np.float64), O.rotation_signs(seed, layer, kind, 128))


def test_qjl_matrix_matches_oracle(B):
    for seed, layer in ((0, 0), (0, 7), (99, 3)):
        s = B.tq_make_qjl_matrix(seed, layer, 128, 128)
        vals = (s.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        assert np.array_equal(vals, O.qjl_matrix(seed, layer, 128, 128))


def test_plane_sizes_match_the_pages_52_byte_vector(B):
    cfg = B.Config(k_bits=3, v_bits=3)
    sizes = B.tq_plane_bytes(cfg, 0, B.TQ_KIND_K, 1, 1, 1)
    assert sizes[0] + sizes[1] == 52 and sizes[2] == sizes[3] == 0
    cfg = B.Config(k_bits=2, v_bits=3, k_mode=B.TQ_MODE_MSE_QJL)
    k = B.tq_plane_bytes(cfg, 0, B.TQ_KIND_K, 1, 1, 1)
    v = B.tq_plane_bytes(cfg, 0, B.TQ_KIND_V, 1, 1, 1)
    assert sum(k) == 32 + 4 + 16 + 4 == 56 and v == (48, 4, 0, 0)
    cfg = B.Config(n_layers=36, k_bits=4, v_bits=2, n_protect_first=4, n_protect_last=4)
    assert sum(B.tq_plane_bytes(cfg, 0, 0, 1, 1, 1)) == 132
    assert sum(B.tq_plane_bytes(cfg, 10, 0, 1, 1, 1)) == 68
    assert sum(B.tq_plane_bytes(cfg, 10, 1, 1, 1, 1)) == 36
    assert sum(B.tq_plane_bytes(cfg, 35, 1, 1, 1, 1)) == 132


def test_layer_spec_matches_oracle_protection(B):
    cfg = B.Config(n_layers=36, k_bits=4, v_bits=2, n_protect_first=4, n_protect_last=4)
    for layer in range(36):
        kb, vb, mode = B.tq_layer_spec_get(cfg, layer)
        assert (kb, vb, bool(mode)) == O.layer_bits(layer, 36, 4, 2, False, 4, 4)


def test_tables_layout(B):
    cfg = B.Config(n_layers=3, k_bits=2, v_bits=3, k_mode=B.TQ_MODE_MSE_QJL, seed=5)
    buf = B.tq_build_tables(cfg)
    assert buf.size == B.tq_tables_bytes(cfg) and buf.size % 256 == 0
    hdr = buf[:32].view(np.int32)
    assert hdr[0] == 0x42545154 and hdr[2] == 128 and hdr[3] == 3
    cb2 = buf[256 + 2048: 256 + 2 * 2048].view(np.float32)
    oc, ob = O.codebook_fp32(2, 128)
    assert np.array_equal(cb2[:4], oc) and np.array_equal(cb2[256:259], ob)
    assert np.all(np.isinf(cb2[259:512]))


def test_workspace_bytes(B):
    cfg = B.Config(residual_window=128)
    n = B.tq_workspace_bytes(cfg, 1, 32, 8, 32768)
    assert n > 0 and n % 256 == 0
    assert B.tq_workspace_bytes(B.Config(), 1, 32, 8, 0) >= 0


def test_workspace_bytes_follow_the_split_plan(B):
    """The workspace holds (m, l, pad, pad, o[128]) fp32 per (pair, split,
    query head) and one counter per pair, each region rounded up to 256
    bytes.  The split counts pin the plan: every pair gets the same number of
    whole quantized splits in one wave.  Host logic only."""
    def expect(pairs, splits, G):
        part = pairs * splits * G * 132 * 4
        return -(-part // 256) * 256 + -(-pairs * 4 // 256) * 256
    # Llama-shaped 32K cache, window 128: 152 CTAs = 8 pairs x (18 quantized + 1 window)
    llama = B.Config(k_bits=4, v_bits=2, residual_window=128)
    assert B.tq_workspace_bytes(llama, 1, 32, 8, 32768) == expect(8, 19, 4)
    # 128 pairs with QJL keys (three CTAs per SM, 456 slots): 3 splits each for a
    # plain decode, 2 + the step's own for a step
    qjl = B.Config(k_bits=2, v_bits=3, k_mode=B.TQ_MODE_MSE_QJL)
    assert B.tq_workspace_bytes(qjl, 16, 32, 8, 8192) == expect(128, 3, 4)
    # more pairs than a wave: one quantized and one window split per pair (several waves)
    assert B.tq_workspace_bytes(llama, 64, 32, 8, 16384) == expect(512, 2, 4)


@pytest.mark.skipif(__import__("conftest").has_gpu(), reason="fake pointers are only used without a GPU")
def test_argument_validation_rejects_before_launch(B):
    import ctypes as C
    lib = B.load()
    cfg = B.Config()
    planes = B.tq_planes(4096, 8192, None, None, 100)
    strides = (C.c_int64 * 3)(128 * 100, 128 * 100, 128)
    call = lambda c, tables=4096, layer=0, kind=0, src=16384, dt=0, p=planes: lib.tq_quantize_kv(
        C.byref(c.c()), tables, layer, kind, src, dt, strides, 1, 1, 10, None, p, None)
    assert call(B.Config(head_dim=64)) == 2            # unsupported head_dim
    assert call(B.Config(k_bits=5)) == 1               # invalid bits
    assert call(B.Config(k_bits=1)) == 2               # host-only bit width
    assert call(cfg, layer=1) == 1                     # layer out of range
    assert call(cfg, tables=4100) == 3                 # misaligned tables
    assert call(cfg, src=16386) == 3                   # misaligned source
    assert call(cfg, dt=7) == 1                        # bad dtype
    assert call(cfg, p=B.tq_planes(4104, 8192, None, None, 100)) == 3
    assert call(B.Config(k_mode=1)) == 1               # QJL planes missing
    assert lib.tq_quantize_kv(None, 4096, 0, 0, 16384, 0, strides, 1, 1, 10, None, planes, None) == 1
    # decode: workspace too small, group size not supported
    out = 32768
    rc = lib.tq_decode_attention(C.byref(cfg.c()), 4096, 0, 16384, 0, 1.0, 1, 8, 8, planes, planes,
                                 None, None, 20480, 10, out, 65536, 16, None)
    assert rc == 7
    rc = lib.tq_decode_attention(C.byref(cfg.c()), 4096, 0, 16384, 0, 1.0, 1, 24, 8, planes, planes,
                                 None, None, 20480, 10, out, 65536, 1 << 20, None)
    assert rc == 2
    wcfg = B.Config(residual_window=16)
    rc = lib.tq_decode_attention(C.byref(wcfg.c()), 4096, 0, 16384, 0, 1.0, 1, 8, 8, planes,
                                 planes, None, None, 20480, 10, out, 65536, 1 << 20, None)
    assert rc == 1                                     # window buffers missing


def test_decode_step_validates_both_calls_before_launch(B):
    """tq_decode_step checks the decode's arguments and the append's before it
    launches either (so no half-done step): each rejection below returns
    before any CUDA call, which would fail on a host without a GPU."""
    import ctypes as C
    lib = B.load()
    cfg = B.Config()
    planes = B.tq_planes(4096, 8192, None, None, 100)
    strides = (C.c_int64 * 3)(128, 128, 128)

    def step(c=cfg, ws_bytes=1 << 20, max_len=10, knew=20480, dt=0, hq=8, tables=4096):
        return lib.tq_decode_step(C.byref(c.c()), tables, 0, 16384, 0, 1.0, 1, hq, 8, knew, 24576,
                                  dt, strides, 28672, max_len, None, None, planes, planes, 32768,
                                  65536, ws_bytes, None)

    assert step(max_len=0) == 1                        # the step adds a token: max_seq_len >= 1
    assert step(ws_bytes=16) == 7                      # workspace too small
    assert step(hq=24) == 2                            # group size 3
    assert step(tables=4100) == 3                      # misaligned tables
    assert step(B.Config(residual_window=16)) == 1     # window buffers missing
    assert step(knew=20482) == 3                       # misaligned new keys (append's check)
    assert step(dt=7) == 1                             # bad source dtype (append's check)
    assert lib.tq_decode_step(C.byref(cfg.c()), 4096, 0, 16384, 0, 1.0, 0, 8, 8, 20480, 24576, 0,
                              strides, 28672, 10, None, None, planes, planes, 32768, 65536,
                              1 << 20, None) == 0      # empty batch: nothing to do


def test_decode_step_launches(B):
    """tq_decode_step takes one launch when its plan, with the splits that
    append the token, fits one wave of the GPU, else two (the append kernel,
    then the decode); 0 flags invalid sizes.  Host logic only."""
    llama = B.Config(k_bits=4, v_bits=2, residual_window=128)
    assert B.tq_decode_step_launches(llama, 0, 1, 32, 8, 32768) == 1
    # no window: the step's split per pair leaves 18 quantized splits of 1,824
    # tokens instead of 19 of 1,728, the same 5 chunks for the busiest warp
    no_window = B.Config(k_bits=4, v_bits=2)
    assert B.tq_decode_step_launches(no_window, 0, 1, 32, 8, 32768) == 1
    long_ctx = B.Config(k_bits=3, v_bits=3, residual_window=256)
    assert B.tq_decode_step_launches(long_ctx, 0, 1, 64, 8, 1 << 20) == 1
    single = B.Config(k_bits=3, v_bits=3)
    assert B.tq_decode_step_launches(single, 0, 1, 1, 1, 1024) == 1
    # 128 pairs at three CTAs per SM: a plain decode gives each pair 3 quantized
    # splits, the step's plan (one split more per pair for the token) only 2
    for mode in (B.TQ_MODE_MSE_QJL, B.TQ_MODE_MSE_SIGN):
        cfg = B.Config(k_bits=2, v_bits=3, k_mode=mode)
        assert B.tq_decode_step_launches(cfg, 0, 16, 32, 8, 8192) == 2
    assert B.tq_decode_step_launches(llama, 0, 84, 8, 2, 700) == 2   # 168 pairs, one CTA per SM
    assert B.tq_decode_step_launches(llama, 0, 1, 32, 8, 0) == 0
    assert B.tq_decode_step_launches(llama, 1, 1, 32, 8, 100) == 0   # layer out of range
    assert B.tq_decode_step_launches(llama, 0, 1, 24, 8, 100) == 0   # group size 3
