"""GPU parity of quantize / append / dequantize against the oracle (through the C ABI)."""

import math

import numpy as np
import pytest

import oracle as O
from gpu_helpers import (binding, compare_codes, compare_norms, oq_slice, oracle_qjl,
                         oracle_quantize, to64, upload_oracle_planes)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    return binding()


def _run_quantize(B, cfg, layer, kind, X, capacity=None, dst_pos=None):
    import torch
    b, h, n, _ = X.shape
    cap = capacity or n
    tables = B.device_tables(cfg)
    planes = B.Planes(cfg, layer, kind, b, h, cap)
    B.tq_quantize_kv(cfg, tables, layer, kind, X, planes, dst_pos=dst_pos)
    torch.cuda.synchronize()
    assert B.tq_get_device_error() == B.TQ_OK
    return planes


def test_quantize_single_head_1k_fp32(B):
    from kv_cache_quantization_random_gb300 import workloads as W
    w = W.get("single_head_1k")
    K, V = W.make_kv(w)
    cfg = B.Config(k_bits=3, v_bits=3, seed=w.codec_seed)
    for kind, X in ((0, K), (1, V)):
        planes = _run_quantize(B, cfg, 0, kind, X.cuda())
        oq = oracle_quantize(to64(X), 3, w.codec_seed, 0, kind)
        n = compare_codes(planes.codes_view().cpu().numpy(), oq, 3)
        compare_norms(planes.norms_view().cpu().numpy(), oq["norms"])
        assert n <= 2


@pytest.mark.parametrize("bits", [2, 3, 4, 8])
@pytest.mark.parametrize("n", [1, 31, 129, 300])
def test_quantize_bits_and_ragged_tiles_bf16(B, bits, n):
    from kv_cache_quantization_random_gb300 import workloads as W
    w = W.scaled(W.get("llama8b_32k"), batch=2, n_kv_heads=3, context=n)
    K, V = W.make_kv(w)
    cfg = B.Config(k_bits=bits, v_bits=bits, seed=7)
    for kind, X in ((0, K), (1, V)):
        planes = _run_quantize(B, cfg, 0, kind, X.cuda())
        oq = oracle_quantize(to64(X), bits, 7, 0, kind)
        compare_codes(planes.codes_view().cpu().numpy(), oq, bits)
        compare_norms(planes.norms_view().cpu().numpy(), oq["norms"])


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_quantize_rows_of_extreme_magnitude(B, bits):
    """Rows scaled by 1e-15 and 1e15 quantize like the oracle's (same unit
    vector); zero rows, rows whose squares fall below the fp32 normal range,
    and rows with inf or NaN take the bounded search and raise no error."""
    import torch
    g = torch.Generator().manual_seed(11)
    base = torch.randn(1, 1, 8, 128, generator=g)
    scales = torch.tensor([1.0, 1e-15, 1e15, 1e-3, 0.0, 1e-21, 1.0, 1.0]).view(1, 1, 8, 1)
    X = (base * scales).to(torch.bfloat16)
    X[0, 0, 6, 5] = float("inf")
    X[0, 0, 7, 9] = float("nan")
    cfg = B.Config(k_bits=bits, v_bits=bits, seed=3)
    planes = _run_quantize(B, cfg, 0, 1, X.cuda())
    codes = planes.codes_view().cpu().numpy()
    fin = [0, 1, 2, 3]
    oq = oracle_quantize(to64(X[:, :, fin]), bits, 3, 0, 1)
    compare_codes(codes[:, :, fin], oq, bits)
    compare_norms(planes.norms_view().cpu().numpy()[:, :, fin], oq["norms"])
    got = O.unpack_codes(codes[0, 0], bits, 128)
    assert (got >= 0).all() and (got < (1 << bits)).all()
    assert planes.norms_view().cpu().numpy()[0, 0, 4] == 0.0


@pytest.mark.parametrize("bits", [2, 4])
def test_quantize_and_decode_with_the_sphere_density_codebook(B, bits):
    """Codebook from the exact coordinate density (TQ_DENSITY_SPHERE_BETA):
    the kernels are the same, the codes follow the sphere codebook, and decode
    attention matches the oracle's."""
    import torch
    from kv_cache_quantization_random_gb300 import workloads as W
    w = W.scaled(W.get("llama8b_32k"), batch=2, n_q_heads=8, n_kv_heads=2, context=700, window=0)
    K, V = W.make_kv(w)
    q = W.make_q(w)
    cfg = B.Config(k_bits=bits, v_bits=bits, seed=9, density=B.TQ_DENSITY_SPHERE_BETA)
    tables = B.device_tables(cfg)
    kp = B.Planes(cfg, 0, 0, 2, 2, 700)
    vp = B.Planes(cfg, 0, 1, 2, 2, 700)
    B.tq_quantize_kv(cfg, tables, 0, 0, K.cuda(), kp)
    B.tq_quantize_kv(cfg, tables, 0, 1, V.cuda(), vp)
    torch.cuda.synchronize()
    assert B.tq_get_device_error() == B.TQ_OK
    oqk = oracle_quantize(to64(K), bits, 9, 0, 0, density=1)
    oqv = oracle_quantize(to64(V), bits, 9, 0, 1, density=1)
    compare_codes(kp.codes_view().cpu().numpy(), oqk, bits)
    compare_codes(vp.codes_view().cpu().numpy(), oqv, bits)
    out = torch.empty(2, 8, 128, device="cuda")
    ws = B.new_workspace(cfg, 2, 8, 2, 700)
    seq = torch.tensor([700, 411], dtype=torch.int32, device="cuda")
    B.tq_decode_attention(cfg, tables, 0, q.cuda(), w.softmax_scale, kp, vp, seq, 700, out, ws)
    torch.cuda.synchronize()
    ref = O.decode_attention(to64(q), oqk["codes"], oqk["norms"], oqv["codes"], oqv["norms"],
                             oqk["c32"], oqv["c32"], oqk["signs"], oqv["signs"], [700, 411],
                             w.softmax_scale)
    got = to64(out)
    rel = np.linalg.norm(got - ref, axis=-1) / np.linalg.norm(ref, axis=-1)
    assert rel.max() < 2e-3


def test_quantize_strided_source_dst_pos_and_zero_rows(B):
    import torch
    g = torch.Generator().manual_seed(3)
    base = torch.randn(2, 40, 4, 128, generator=g).to(torch.bfloat16)   # [B, T, H, d] storage
    base[1, 5] = 0                                                       # zero vectors
    X = base.cuda().permute(0, 2, 1, 3)                                  # [B, H, T, d] view
    assert X.stride(2) == 4 * 128
    cfg = B.Config(k_bits=4, v_bits=4, seed=11, n_layers=3)
    pos = torch.tensor([0, 17], dtype=torch.int32, device="cuda")
    planes = _run_quantize(B, cfg, 2, 0, X, capacity=64, dst_pos=pos)
    oq = oracle_quantize(to64(X), 4, 11, 2, 0)
    codes = planes.codes_view().cpu().numpy()
    norms = planes.norms_view().cpu().numpy()
    compare_codes(codes[0, :, 0:40], oq_slice(oq, 0), 4)
    compare_codes(codes[1, :, 17:57], oq_slice(oq, 1), 4)
    compare_norms(norms[0, :, 0:40], oq["norms"][0])
    compare_norms(norms[1, :, 17:57], oq["norms"][1])
    assert np.all(norms[1, :, 22] == 0.0)                               # zero vectors
    assert np.all(codes[0, :, 40:] == 0) and np.all(codes[1, :, :17] == 0)


def test_quantize_rows_past_capacity_are_flagged_not_written(B):
    import torch
    X = torch.randn(1, 1, 8, 128).to(torch.bfloat16).cuda()
    cfg = B.Config(k_bits=2, v_bits=2)
    tables = B.device_tables(cfg)
    planes = B.Planes(cfg, 0, 0, 1, 1, 8)
    pos = torch.tensor([4], dtype=torch.int32, device="cuda")
    B.tq_quantize_kv(cfg, tables, 0, 0, X, planes, dst_pos=pos)
    assert B.tq_get_device_error() == 6               # TQ_ERR_DEVICE_BOUNDS
    assert B.tq_get_device_error() == B.TQ_OK         # cleared on read
    oq = oracle_quantize(to64(X), 2, 0, 0, 0)
    codes = planes.codes_view().cpu().numpy()
    compare_codes(codes[:, :, 4:8], oq_slice(oq, (slice(None), slice(None), slice(0, 4))), 2)
    assert np.all(codes[:, :, :4] == 0)


def test_quantize_qjl_keys(B):
    from kv_cache_quantization_random_gb300 import workloads as W
    w = W.scaled(W.get("qjl_b16_8k"), batch=2, context=200)
    K, _ = W.make_kv(w)
    cfg = B.Config(k_bits=2, v_bits=3, k_mode=B.TQ_MODE_MSE_QJL, qjl_m=128, seed=w.codec_seed)
    planes = _run_quantize(B, cfg, 0, 0, K.cuda())
    oq = oracle_quantize(to64(K), 2, w.codec_seed, 0, 0)
    compare_codes(planes.codes_view().cpu().numpy(), oq, 2)
    compare_norms(planes.norms_view().cpu().numpy(), oq["norms"])
    # the sketch is checked against the oracle's residual of the GPU's own codes
    # (codes may legitimately differ inside the boundary band)
    gcodes = O.unpack_codes(planes.codes_view().cpu().numpy(), 2, 128)
    S = O.qjl_matrix(w.codec_seed, 0, 128, 128)
    r = O.qjl_residual(oq["y"], gcodes, oq["norm64"], oq["c32"])
    bits, gamma, z = O.qjl_sketch(r, S)
    gbits = O.unpack_bits(planes.signs_view().cpu().numpy(), 128)
    compare_norms(planes.rnorm_view().cpu().numpy(), gamma, rel=2e-6)
    band = np.abs(z) <= 1e-5 * np.linalg.norm(S, axis=1) * gamma[..., None].astype(np.float64)
    bad = (gbits != bits) & ~band
    assert not bad.any(), int(bad.sum())


def _check_direct_sign(P, oq, bits, rows=None):
    """GPU signs and scale against the oracle's Direct Sign of the residual of
    the GPU's own codes (codes may differ inside the boundary band); a sign may
    differ only where |r_i| <= 1e-6 ||x||."""
    sl = (slice(None), slice(None), slice(None, rows))
    gcodes = O.unpack_codes(P.codes_view()[sl].cpu().numpy(), bits, 128)
    r = O.qjl_residual(oq["y"], gcodes, oq["norm64"], oq["c32"])
    sb, scale = O.direct_sign_sketch(r)
    gbits = O.unpack_bits(P.signs_view()[sl].cpu().numpy(), 128)
    band = np.abs(r) <= 1e-6 * oq["norm64"][..., None]
    assert not ((gbits != sb) & ~band).any()
    compare_norms(P.rnorm_view()[sl].cpu().numpy(), scale, rel=1e-5)


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_quantize_direct_sign_keys(B, bits):
    from kv_cache_quantization_random_gb300 import workloads as W
    w = W.scaled(W.get("sign_b16_8k"), batch=2, context=333)
    K, _ = W.make_kv(w)
    cfg = B.Config(k_bits=bits, v_bits=3, k_mode=B.TQ_MODE_MSE_SIGN, seed=4)
    planes = _run_quantize(B, cfg, 0, 0, K.cuda())
    oq = oracle_quantize(to64(K), bits, 4, 0, 0)
    compare_codes(planes.codes_view().cpu().numpy(), oq, bits)
    compare_norms(planes.norms_view().cpu().numpy(), oq["norms"])
    _check_direct_sign(planes, oq, bits)


@pytest.mark.parametrize("bits,qjl", [(2, False), (3, False), (4, False), (8, False), (2, True)])
def test_dequantize_matches_oracle(B, bits, qjl):
    import torch
    rng = np.random.default_rng(bits)
    X = rng.standard_normal((2, 2, 70, 128)) * 3.0
    seed, layer = 5, 0
    cfg = B.Config(k_bits=bits, v_bits=bits, seed=seed,
                   k_mode=B.TQ_MODE_MSE_QJL if qjl else B.TQ_MODE_MSE)
    tables = B.device_tables(cfg)
    oq = oracle_quantize(X, bits, seed, layer, 0)
    planes = B.Planes(cfg, layer, 0, 2, 2, 70)
    upload_oracle_planes(B, planes, oq)
    if qjl:
        qj = oracle_qjl(oq, seed, layer)
        planes.signs_view().copy_(torch.from_numpy(qj["packed"]))
        planes.rnorm_view().copy_(torch.from_numpy(qj["gamma"]))
        ref = O.dequantize_qjl(oq["codes"], oq["norms"], qj["bits"], qj["gamma"], oq["c32"],
                               oq["signs"], qj["S"])
    else:
        ref = O.dequantize(oq["codes"], oq["norms"], oq["c32"], oq["signs"])
    out = torch.empty(2, 2, 70, 128, device="cuda")
    B.tq_dequantize(cfg, tables, layer, 0, planes, 70, out, include_qjl=qjl)
    got = to64(out)
    scale = np.linalg.norm(ref, axis=-1, keepdims=True)
    assert np.all(np.abs(got - ref) <= 2e-6 * scale + 1e-30)


@pytest.mark.parametrize("W_", [0, 16])
def test_streaming_append_with_window(B, W_):
    import torch
    from kv_cache_quantization_random_gb300 import workloads as W
    Bsz, H, cap = 2, 2, 96
    cfg = B.Config(k_bits=4, v_bits=2, residual_window=W_, seed=3)
    tables = B.device_tables(cfg)
    kp = B.Planes(cfg, 0, 0, Bsz, H, cap)
    vp = B.Planes(cfg, 0, 1, Bsz, H, cap)
    kw = torch.zeros(Bsz, H, max(W_, 1), 128, dtype=torch.bfloat16, device="cuda")
    vw = torch.zeros_like(kw)
    w = W.scaled(W.get("llama8b_32k"), batch=Bsz, n_kv_heads=H, context=cap)
    K, V = W.make_kv(w)
    lens = np.zeros(Bsz, dtype=np.int64)
    for n_new in (1, 7, 20, 1, 40):
        kn = torch.empty(Bsz, H, n_new, 128, dtype=torch.bfloat16)
        vn = torch.empty_like(kn)
        for b in range(Bsz):
            t0 = int(lens[b])
            kn[b] = K[b, :, t0:t0 + n_new]
            vn[b] = V[b, :, t0:t0 + n_new]
        before = torch.tensor(lens, dtype=torch.int32, device="cuda")
        B.tq_append_kv(cfg, tables, 0, kn.cuda(), vn.cuda(), before, kw if W_ else None,
                       vw if W_ else None, kp, vp)
        torch.cuda.synchronize()
        assert B.tq_get_device_error() == B.TQ_OK
        lens += n_new
        if lens[0] + 40 > cap:
            break
    T = int(lens[0])
    nq = max(T - W_, 0)
    for kind, X, P in ((0, K, kp), (1, V, vp)):
        bits = 4 if kind == 0 else 2
        oq = oracle_quantize(to64(X[:, :, :nq]), bits, 3, 0, kind)
        compare_codes(P.codes_view()[:, :, :nq].cpu().numpy(), oq, bits)
        compare_norms(P.norms_view()[:, :, :nq].cpu().numpy(), oq["norms"])
    if W_:
        for t in range(nq, T):
            assert torch.equal(kw[:, :, t % W_].cpu(), K[:, :, t])
            assert torch.equal(vw[:, :, t % W_].cpu(), V[:, :, t])


@pytest.mark.parametrize("kb,vb,qjl,W_", [(3, 3, False, 8), (8, 8, False, 0), (2, 3, True, 0),
                                        (4, 2, True, 32), (2, 3, "sign", 0),
                                        (3, 2, "sign", 16)])
def test_append_one_launch_and_bulk_paths(B, kb, vb, qjl, W_):
    """Appends of at most 8 tokens per sequence run as one fused launch (warp
    per vector); larger ones take the bulk quantize kernel.  Both must give the
    oracle's codes, norms and (QJL keys) sign sketches."""
    import torch
    from kv_cache_quantization_random_gb300 import workloads as W
    Bsz, H, cap = 3, 2, 80
    cfg = B.Config(k_bits=kb, v_bits=vb, residual_window=W_, seed=11,
                   k_mode=(B.TQ_MODE_MSE_SIGN if qjl == "sign" else
                           B.TQ_MODE_MSE_QJL if qjl else B.TQ_MODE_MSE))
    tables = B.device_tables(cfg)
    kp = B.Planes(cfg, 0, 0, Bsz, H, cap)
    vp = B.Planes(cfg, 0, 1, Bsz, H, cap)
    kw = torch.zeros(Bsz, H, max(W_, 1), 128, dtype=torch.bfloat16, device="cuda")
    vw = torch.zeros_like(kw)
    w = W.scaled(W.get("llama8b_32k"), batch=Bsz, n_kv_heads=H, context=cap, data_seed=5)
    K, V = W.make_kv(w)
    lens = np.zeros(Bsz, dtype=np.int64)
    for n_new in (1, 8, 9, 3, 1, 30):
        if lens[0] + n_new > cap:
            break
        kn = K[:, :, int(lens[0]):int(lens[0]) + n_new].contiguous()
        vn = V[:, :, int(lens[0]):int(lens[0]) + n_new].contiguous()
        before = torch.tensor(lens, dtype=torch.int32, device="cuda")
        B.tq_append_kv(cfg, tables, 0, kn.cuda(), vn.cuda(), before, kw if W_ else None,
                       vw if W_ else None, kp, vp)
        torch.cuda.synchronize()
        assert B.tq_get_device_error() == B.TQ_OK
        lens += n_new
    T = int(lens[0])
    nq = max(T - W_, 0)
    for kind, X, P, bits in ((0, K, kp, kb), (1, V, vp, vb)):
        oq = oracle_quantize(to64(X[:, :, :nq]), bits, 11, 0, kind)
        compare_codes(P.codes_view()[:, :, :nq].cpu().numpy(), oq, bits)
        compare_norms(P.norms_view()[:, :, :nq].cpu().numpy(), oq["norms"])
        if kind == 0 and qjl == "sign":
            _check_direct_sign(P, oq, bits, rows=nq)
        elif kind == 0 and qjl:
            # sketch of the oracle's residual of the GPU's own codes (codes may
            # differ inside the boundary band); a sign may differ only where
            # |z_j| <= 1e-5 ||S_j|| gamma
            gcodes = O.unpack_codes(P.codes_view()[:, :, :nq].cpu().numpy(), bits, 128)
            S = O.qjl_matrix(11, 0, 128, 128)
            r = O.qjl_residual(oq["y"], gcodes, oq["norm64"], oq["c32"])
            sb, gamma, z = O.qjl_sketch(r, S)
            gbits = O.unpack_bits(P.signs_view()[:, :, :nq].cpu().numpy(), 128)
            compare_norms(P.rnorm_view()[:, :, :nq].cpu().numpy(), gamma, rel=2e-6)
            band = np.abs(z) <= 1e-5 * np.linalg.norm(S, axis=1) * gamma[..., None]
            assert not ((gbits != sb) & ~band).any()
    if W_:
        for t in range(nq, T):
            assert torch.equal(kw[:, :, t % W_].cpu(), K[:, :, t])
            assert torch.equal(vw[:, :, t % W_].cpu(), V[:, :, t])


def test_gpu_argument_validation_with_real_buffers(B):
    import torch
    cfg = B.Config(k_bits=3, v_bits=3)
    tables = B.device_tables(cfg)
    X = torch.randn(1, 1, 16, 136).to(torch.bfloat16).cuda()[..., 4:132]   # misaligned rows
    planes = B.Planes(cfg, 0, 0, 1, 1, 16)
    with pytest.raises(B.TQError) as e:
        B.tq_quantize_kv(cfg, tables, 0, 0, X, planes)
    assert e.value.status == 3
    with pytest.raises(B.TQError) as e:
        B.tq_quantize_kv(B.Config(head_dim=64), tables, 0, 0, X, planes)
    assert e.value.status == 2
