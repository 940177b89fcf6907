"""GPU parity of decode attention against the oracle (through the C ABI).

Most tests upload the oracle's own packed codes into the planes, so the
comparison isolates decode attention from quantize; the end-to-end tests run
the CUDA quantize too.  The bar is 2e-3 relative L2 per (sequence, query head).
"""

import math

import numpy as np
import pytest

import oracle as O
from gpu_helpers import (binding, compare_codes, oracle_qjl, oracle_quantize, rel_l2_per_head,
                         to64, upload_oracle_planes)

pytestmark = pytest.mark.gpu
TOL = 2e-3


@pytest.fixture(scope="module")
def B():
    return binding()


def _decode_case(B, *, batch, hq, hkv, seq, kb, vb, W=0, qjl=False, dsign=False, layer=0,
                 n_layers=1, protect=(0, 0), q_f32=False, seed=0, dist="llama", extra_cap=0,
                 data_seed=5):
    """Build a cache from seeded inputs, quantize it with the oracle, upload the
    oracle's planes, run the CUDA decode, run the oracle decode, return both."""
    import torch
    from kv_cache_quantization_random_gb300 import workloads as W_
    seq = np.asarray(seq, dtype=np.int64)
    Tmax = int(seq.max()) if len(seq) else 0
    cap = max(Tmax - W, 0) + extra_cap + 1
    w = W_.scaled(W_.get("llama8b_32k"), batch=batch, n_q_heads=hq, n_kv_heads=hkv,
                  context=max(Tmax, 1), dist=dist, data_seed=data_seed)
    K, V = W_.make_kv(w)
    q = W_.make_q(w)
    if q_f32:
        q = q.float()
    cfg = B.Config(k_bits=kb, v_bits=vb, residual_window=W, seed=seed, n_layers=n_layers,
                   n_protect_first=protect[0], n_protect_last=protect[1],
                   k_mode=(B.TQ_MODE_MSE_QJL if qjl else
                           B.TQ_MODE_MSE_SIGN if dsign else B.TQ_MODE_MSE))
    kb_l, vb_l, mode = B.tq_layer_spec_get(cfg, layer)
    tables = B.device_tables(cfg)
    K64, V64 = to64(K), to64(V)
    nq = max(Tmax - W, 0)
    oqk = oracle_quantize(K64[:, :, :nq], kb_l, seed, layer, 0)
    oqv = oracle_quantize(V64[:, :, :nq], vb_l, seed, layer, 1)
    kp = B.Planes(cfg, layer, 0, batch, hkv, cap)
    vp = B.Planes(cfg, layer, 1, batch, hkv, cap)
    qj = None
    if nq:
        upload_oracle_planes(B, kp, oqk)
        upload_oracle_planes(B, vp, oqv)
        if mode == B.TQ_MODE_MSE_QJL:
            qj = oracle_qjl(oqk, seed, layer)
            kp.signs_view()[:, :, :nq].copy_(torch.from_numpy(qj["packed"]))
            kp.rnorm_view()[:, :, :nq].copy_(torch.from_numpy(qj["gamma"]))
        if mode == B.TQ_MODE_MSE_SIGN:
            r = O.qjl_residual(oqk["y"], oqk["codes"], oqk["norm64"], oqk["c32"])
            dbits, dscale = O.direct_sign_sketch(r)
            kp.signs_view()[:, :, :nq].copy_(torch.from_numpy(O.pack_bits(dbits)))
            kp.rnorm_view()[:, :, :nq].copy_(torch.from_numpy(dscale))
    # window ring per sequence: token t in slot t mod W, for t in [T_b - W, T_b)
    kw = vw = None
    kw64 = vw64 = None
    if W:
        kw = torch.zeros(batch, hkv, W, 128, dtype=torch.bfloat16)
        vw = torch.zeros_like(kw)
        for b in range(batch):
            for t in range(max(int(seq[b]) - W, 0), int(seq[b])):
                kw[b, :, t % W] = K[b, :, t]
                vw[b, :, t % W] = V[b, :, t]
        kw64, vw64 = to64(kw), to64(vw)
        kw, vw = kw.cuda(), vw.cuda()
    # the oracle reads quantized tokens t < T_b - W; rows beyond are never used
    kcodes = np.zeros((batch, hkv, cap, 128), dtype=np.int64)
    vcodes = np.zeros_like(kcodes)
    kn = np.zeros((batch, hkv, cap), np.float32)
    vn = np.zeros_like(kn)
    if nq:
        kcodes[:, :, :nq], vcodes[:, :, :nq] = oqk["codes"], oqv["codes"]
        kn[:, :, :nq], vn[:, :, :nq] = oqk["norms"], oqv["norms"]
    qjl_arg = None
    if qj is not None:
        bits = np.zeros((batch, hkv, cap, 128), np.int64)
        gam = np.zeros((batch, hkv, cap), np.float32)
        bits[:, :, :nq], gam[:, :, :nq] = qj["bits"], qj["gamma"]
        qjl_arg = dict(bits=bits, gamma=gam, S=qj["S"])
    dsign_arg = None
    if mode == B.TQ_MODE_MSE_SIGN:
        bits_ = np.zeros((batch, hkv, cap, 128), np.int64)
        sc_ = np.zeros((batch, hkv, cap), np.float32)
        if nq:
            bits_[:, :, :nq], sc_[:, :, :nq] = dbits, dscale
        dsign_arg = dict(bits=bits_, scale=sc_)
    ck, _ = O.codebook_fp32(kb_l, 128)
    cv, _ = O.codebook_fp32(vb_l, 128)
    ref = O.decode_attention(to64(q), kcodes, kn, vcodes, vn, ck, cv,
                             O.rotation_signs(seed, layer, 0, 128),
                             O.rotation_signs(seed, layer, 1, 128), seq, w.softmax_scale,
                             window=W, k_win=kw64, v_win=vw64, qjl=qjl_arg, dsign=dsign_arg)
    out = torch.full((batch, hq, 128), float("nan"), device="cuda")
    ws = B.new_workspace(cfg, batch, hq, hkv, Tmax)
    seq_t = torch.tensor(seq, dtype=torch.int32, device="cuda")
    B.tq_decode_attention(cfg, tables, layer, q.cuda(), w.softmax_scale, kp, vp, seq_t, Tmax, out,
                          ws, k_win=kw, v_win=vw)
    torch.cuda.synchronize()
    assert B.tq_get_device_error() == B.TQ_OK
    return to64(out), ref, dict(cfg=cfg, tables=tables, kp=kp, vp=vp, q=q, seq_t=seq_t, Tmax=Tmax,
                                ws=ws, kw=kw, vw=vw, scale=w.softmax_scale)


@pytest.mark.parametrize("kb,vb", [(4, 2), (3, 3), (2, 2), (8, 8), (2, 4), (4, 8)])
def test_decode_bits(B, kb, vb):
    out, ref, _ = _decode_case(B, batch=2, hq=8, hkv=2, seq=[700, 333], kb=kb, vb=vb)
    assert rel_l2_per_head(out, ref).max() < TOL


@pytest.mark.parametrize("seq,W", [([1], 0), ([2], 0), ([31], 0), ([33], 16), ([255, 256, 257], 0),
                                   ([511, 512, 513], 8), ([1, 2, 3], 4), ([32, 64], 32)])
def test_decode_tiny_and_split_boundary_lengths(B, seq, W):
    """Tiny contexts and contexts one token either side of a split boundary
    (splits are multiples of 256 tokens here), with and without a window."""
    out, ref, _ = _decode_case(B, batch=len(seq), hq=8, hkv=2, seq=seq, kb=4, vb=2, W=W)
    assert rel_l2_per_head(out, ref).max() < TOL


@pytest.mark.parametrize("g", [1, 2, 4, 8])
def test_decode_group_sizes(B, g):
    out, ref, _ = _decode_case(B, batch=1, hq=2 * g, hkv=2, seq=[1500], kb=3, vb=3)
    assert rel_l2_per_head(out, ref).max() < TOL


def test_decode_single_head_1k_config(B):
    """The single-head 1024-token config: fp32 K/V with outliers, K3/V3, W=0,
    query prescaled by 1/sqrt(d) with softmax scale 1."""
    import torch
    from kv_cache_quantization_random_gb300 import workloads as W_
    w = W_.get("single_head_1k")
    K, V = W_.make_kv(w)
    q = W_.make_q(w)
    cfg = B.Config(k_bits=3, v_bits=3, seed=w.codec_seed)
    tables = B.device_tables(cfg)
    kp = B.Planes(cfg, 0, 0, 1, 1, 1024)
    vp = B.Planes(cfg, 0, 1, 1, 1, 1024)
    B.tq_quantize_kv(cfg, tables, 0, 0, K.cuda(), kp)
    B.tq_quantize_kv(cfg, tables, 0, 1, V.cuda(), vp)
    out = torch.empty(1, 1, 128, device="cuda")
    ws = B.new_workspace(cfg, 1, 1, 1, 1024)
    seq = torch.tensor([1024], dtype=torch.int32, device="cuda")
    B.tq_decode_attention(cfg, tables, 0, q.cuda(), 1.0, kp, vp, seq, 1024, out, ws)
    torch.cuda.synchronize()
    oqk = oracle_quantize(to64(K), 3, 0, 0, 0)
    oqv = oracle_quantize(to64(V), 3, 0, 0, 1)
    compare_codes(kp.codes_view().cpu().numpy(), oqk, 3)
    compare_codes(vp.codes_view().cpu().numpy(), oqv, 3)
    ref = O.decode_attention(to64(q), oqk["codes"], oqk["norms"], oqv["codes"], oqv["norms"],
                             oqk["c32"], oqv["c32"], oqk["signs"], oqv["signs"], [1024], 1.0)
    assert rel_l2_per_head(to64(out), ref).max() < TOL


def test_decode_ragged_edges_with_window(B):
    W = 16
    seq = [0, 1, W - 1, W, W + 1, 2 * W + 3, 300, 1027]
    out, ref, _ = _decode_case(B, batch=len(seq), hq=4, hkv=1, seq=seq, kb=4, vb=2, W=W)
    assert np.all(out[0] == 0.0)
    assert rel_l2_per_head(out[1:], ref[1:]).max() < TOL


@pytest.mark.parametrize("W", [100, 256, 520])
def test_decode_window_spread_over_several_splits(B, W):
    """A window of W tokens is split at most 32 tokens per warp of a CTA (520
    tokens take two 12-warp CTAs); sequences shorter than the window leave
    some of those splits partly or wholly empty."""
    seq = [5, 31, 33, 64, W - 1, W, W + 1, W + 64, 900]
    out, ref, _ = _decode_case(B, batch=len(seq), hq=8, hkv=2, seq=seq, kb=4, vb=2, W=W)
    assert rel_l2_per_head(out, ref).max() < TOL


def test_decode_ragged_no_window_and_empty(B):
    seq = [0, 1, 2, 31, 32, 33, 255, 256, 257, 2000]
    out, ref, _ = _decode_case(B, batch=len(seq), hq=8, hkv=2, seq=seq, kb=3, vb=2)
    assert np.all(out[0] == 0.0)
    assert rel_l2_per_head(out[1:], ref[1:]).max() < TOL


def test_decode_qjl_keys(B):
    out, ref, _ = _decode_case(B, batch=3, hq=8, hkv=2, seq=[900, 64, 1], kb=2, vb=3, qjl=True)
    assert rel_l2_per_head(out, ref).max() < TOL


@pytest.mark.parametrize("kb,vb,W", [(2, 3, 0), (3, 3, 64), (4, 2, 16)])
def test_decode_direct_sign_keys(B, kb, vb, W):
    out, ref, _ = _decode_case(B, batch=3, hq=8, hkv=2, seq=[900, 64, 1], kb=kb, vb=vb, W=W,
                               dsign=True)
    assert rel_l2_per_head(out, ref).max() < TOL


def test_decode_sparse_v_skip_stays_within_tolerance(B):
    """sparse_v = 20: the V sum of a 32-token chunk whose softmax weights are
    all below 2^-20 of the running maximum is skipped.  The output stays within
    the parity bar of the exact oracle, and close to the exact GPU output."""
    import copy
    import torch
    out, ref, c = _decode_case(B, batch=2, hq=8, hkv=2, seq=[4000, 2500], kb=4, vb=2, W=32)
    scfg = copy.copy(c["cfg"])
    scfg.sparse_v = 20
    got = torch.empty(2, 8, 128, device="cuda")
    B.tq_decode_attention(scfg, c["tables"], 0, c["q"].cuda(), c["scale"], c["kp"], c["vp"],
                          c["seq_t"], c["Tmax"], got, c["ws"], k_win=c["kw"], v_win=c["vw"])
    torch.cuda.synchronize()
    assert B.tq_get_device_error() == B.TQ_OK
    g = to64(got)
    assert rel_l2_per_head(g, ref).max() < TOL
    # the skipped weights are each below 2^-20 of the largest: the change is
    # far below the codec's own error
    assert rel_l2_per_head(g, out).max() < 1e-4


def test_decode_protected_layers(B):
    for layer in (0, 5, 11):
        out, ref, _ = _decode_case(B, batch=2, hq=8, hkv=2, seq=[600, 1200], kb=4, vb=2,
                                   n_layers=12, protect=(4, 4), layer=layer)
        assert rel_l2_per_head(out, ref).max() < TOL


def test_decode_fp32_query_and_repeat_calls_reuse_workspace(B):
    import torch
    out, ref, ctx = _decode_case(B, batch=2, hq=4, hkv=2, seq=[513, 2049], kb=4, vb=4, q_f32=True)
    assert rel_l2_per_head(out, ref).max() < TOL
    out2 = torch.empty(2, 4, 128, device="cuda")
    for _ in range(3):     # the split counters reset themselves
        B.tq_decode_attention(ctx["cfg"], ctx["tables"], 0, ctx["q"].cuda(), ctx["scale"], ctx["kp"],
                              ctx["vp"], ctx["seq_t"], ctx["Tmax"], out2, ctx["ws"])
    torch.cuda.synchronize()
    assert np.array_equal(to64(out2), out)


def test_decode_end_to_end_gpu_quantize(B):
    """CUDA quantize + CUDA decode against oracle quantize + oracle decode."""
    import torch
    from kv_cache_quantization_random_gb300 import workloads as W_
    w = W_.scaled(W_.get("llama8b_32k"), context=3000)
    K, V = W_.make_kv(w)
    q = W_.make_q(w)
    Wn = w.window
    T = w.context
    nq = T - Wn
    cfg = B.Config(k_bits=4, v_bits=2, residual_window=Wn, seed=w.codec_seed)
    tables = B.device_tables(cfg)
    kp = B.Planes(cfg, 0, 0, 1, 8, nq)
    vp = B.Planes(cfg, 0, 1, 1, 8, nq)
    B.tq_quantize_kv(cfg, tables, 0, 0, K[:, :, :nq].cuda(), kp)
    B.tq_quantize_kv(cfg, tables, 0, 1, V[:, :, :nq].cuda(), vp)
    kw = torch.empty(1, 8, Wn, 128, dtype=torch.bfloat16)
    vw = torch.empty_like(kw)
    for t in range(nq, T):
        kw[:, :, t % Wn] = K[:, :, t]
        vw[:, :, t % Wn] = V[:, :, t]
    out = torch.empty(1, 32, 128, device="cuda")
    ws = B.new_workspace(cfg, 1, 32, 8, T)
    seq = torch.tensor([T], dtype=torch.int32, device="cuda")
    B.tq_decode_attention(cfg, tables, 0, q.cuda(), w.softmax_scale, kp, vp, seq, T, out, ws,
                          k_win=kw.cuda(), v_win=vw.cuda())
    torch.cuda.synchronize()
    assert B.tq_get_device_error() == B.TQ_OK
    oqk = oracle_quantize(to64(K[:, :, :nq]), 4, 0, 0, 0)
    oqv = oracle_quantize(to64(V[:, :, :nq]), 2, 0, 0, 1)
    compare_codes(kp.codes_view().cpu().numpy(), oqk, 4)
    compare_codes(vp.codes_view().cpu().numpy(), oqv, 2)
    ref = O.decode_attention(to64(q), oqk["codes"], oqk["norms"], oqv["codes"], oqv["norms"],
                             oqk["c32"], oqv["c32"], oqk["signs"], oqv["signs"], [T],
                             w.softmax_scale, window=Wn, k_win=to64(kw), v_win=to64(vw))
    assert rel_l2_per_head(to64(out), ref).max() < TOL


def test_fault_injection_times_out_and_context_stays_usable(B):
    """The decode kernel's staging waits are told to expect bytes that never
    arrive: each bounded wait runs out, the call reports a device timeout, and
    the next call on the same workspace is correct again."""
    import torch
    got, ref, c = _decode_case(B, batch=2, hq=8, hkv=2, seq=[700, 300], kb=4, vb=2, W=16)
    assert rel_l2_per_head(got, ref).max() < TOL
    out = torch.empty(2, 8, 128, device="cuda")
    B.tq_set_wait_limit(2000)
    B.tq_set_fault_injection(1)
    try:
        B.tq_decode_attention(c["cfg"], c["tables"], 0, c["q"].cuda(), c["scale"], c["kp"], c["vp"],
                              c["seq_t"], c["Tmax"], out, c["ws"], k_win=c["kw"], v_win=c["vw"])
        assert B.tq_get_device_error() == 5          # TQ_ERR_DEVICE_TIMEOUT
    finally:
        B.tq_set_fault_injection(0)
        B.tq_set_wait_limit(0)
    B.tq_decode_attention(c["cfg"], c["tables"], 0, c["q"].cuda(), c["scale"], c["kp"], c["vp"],
                          c["seq_t"], c["Tmax"], out, c["ws"], k_win=c["kw"], v_win=c["vw"])
    assert B.tq_get_device_error() == B.TQ_OK
    assert rel_l2_per_head(to64(out), ref).max() < TOL


def test_decode_flags_lengths_outside_the_plan(B):
    """A sequence length above max_seq_len (or below zero) would make the
    kernel read past the pair's plane rows or window ring.  The kernel checks
    every length it reads: such a sequence is decoded as empty (zeros) and the
    call reports TQ_ERR_DEVICE_BOUNDS; the other sequences are unaffected, and
    the next call is clean."""
    import torch
    got, ref, c = _decode_case(B, batch=3, hq=8, hkv=2, seq=[700, 333, 512], kb=4, vb=2, W=16)
    assert rel_l2_per_head(got, ref).max() < TOL
    bad = torch.tensor([700, 5000, -3], dtype=torch.int32, device="cuda")
    out = torch.full((3, 8, 128), float("nan"), device="cuda")
    B.tq_decode_attention(c["cfg"], c["tables"], 0, c["q"].cuda(), c["scale"], c["kp"], c["vp"],
                          bad, c["Tmax"], out, c["ws"], k_win=c["kw"], v_win=c["vw"])
    assert B.tq_get_device_error() == B.TQ_ERR_DEVICE_BOUNDS
    o = to64(out)
    assert np.array_equal(o[0], got[0])           # same plan, same splits: bit-identical
    assert np.all(o[1:] == 0.0)
    B.tq_decode_attention(c["cfg"], c["tables"], 0, c["q"].cuda(), c["scale"], c["kp"], c["vp"],
                          c["seq_t"], c["Tmax"], out, c["ws"], k_win=c["kw"], v_win=c["vw"])
    assert B.tq_get_device_error() == B.TQ_OK
    assert np.array_equal(to64(out), got)


@pytest.mark.parametrize("hq,hkv,nq_tok,W", [(8, 2, 2, 16), (4, 2, 4, 8), (2, 2, 8, 64), (8, 8, 1, 0)])
def test_decode_multi_query_matches_causal_oracle(B, hq, hkv, nq_tok, W):
    """n_queries query tokens per sequence at once: query j sees tokens up to
    T - n_queries + j; against the oracle's causal multi-query decode."""
    import torch
    from kv_cache_quantization_random_gb300 import workloads as W_
    seq = np.array([700, 300, max(nq_tok, 5)], dtype=np.int64)
    batch, Tmax = len(seq), int(seq.max())
    w = W_.scaled(W_.get("llama8b_32k"), batch=batch, n_q_heads=hq, n_kv_heads=hkv,
                  context=Tmax, data_seed=9)
    K, V = W_.make_kv(w)
    gen = torch.Generator().manual_seed(77)
    q = torch.randn(batch, hq, nq_tok, 128, generator=gen).to(torch.bfloat16)
    cfg = B.Config(k_bits=4, v_bits=2, residual_window=W, seed=3)
    tables = B.device_tables(cfg)
    nq = max(Tmax - W, 0)
    kp = B.Planes(cfg, 0, 0, batch, hkv, max(nq, 1))
    vp = B.Planes(cfg, 0, 1, batch, hkv, max(nq, 1))
    if nq:
        B.tq_quantize_kv(cfg, tables, 0, 0, K[:, :, :nq].cuda(), kp)
        B.tq_quantize_kv(cfg, tables, 0, 1, V[:, :, :nq].cuda(), vp)
    kw = vw = None
    kw64 = vw64 = None
    if W:
        kw = torch.zeros(batch, hkv, W, 128, dtype=torch.bfloat16)
        vw = torch.zeros_like(kw)
        for b in range(batch):
            for t in range(max(int(seq[b]) - W, 0), int(seq[b])):
                kw[b, :, t % W] = K[b, :, t]
                vw[b, :, t % W] = V[b, :, t]
        kw64, vw64 = to64(kw), to64(vw)
        kw, vw = kw.cuda(), vw.cuda()
    out = torch.full((batch, hq, nq_tok, 128), float("nan"), device="cuda")
    ws = B.new_workspace(cfg, batch, hq * nq_tok, hkv, Tmax)
    seq_t = torch.tensor(seq, dtype=torch.int32, device="cuda")
    B.tq_decode_attention_multi(cfg, tables, 0, q.cuda(), w.softmax_scale, kp, vp, seq_t, Tmax,
                                out, ws, k_win=kw, v_win=vw)
    torch.cuda.synchronize()
    assert B.tq_get_device_error() == B.TQ_OK
    oqk = oracle_quantize(to64(K[:, :, :nq]), 4, 3, 0, 0)
    oqv = oracle_quantize(to64(V[:, :, :nq]), 2, 3, 0, 1)
    ref = O.decode_attention_multi(to64(q), oqk["codes"], oqk["norms"], oqv["codes"],
                                   oqv["norms"], oqk["c32"], oqv["c32"], oqk["signs"], oqv["signs"],
                                   seq, w.softmax_scale, window=W, k_win=kw64, v_win=vw64)
    got = to64(out)
    assert np.all(np.isfinite(got))
    rel = np.linalg.norm(got - ref, axis=-1) / np.linalg.norm(ref, axis=-1)
    assert rel.max() < TOL


def test_decode_multi_query_needs_the_hidden_tokens_in_the_window(B):
    import torch
    cfg = B.Config(k_bits=4, v_bits=2, residual_window=2)
    tables = B.device_tables(cfg)
    kp = B.Planes(cfg, 0, 0, 1, 2, 64)
    vp = B.Planes(cfg, 0, 1, 1, 2, 64)
    q = torch.zeros(1, 2, 4, 128, dtype=torch.bfloat16, device="cuda")     # 4 columns per kv-head
    out = torch.empty(1, 2, 4, 128, device="cuda")
    ws = B.new_workspace(cfg, 1, 8, 2, 66)
    kw = torch.zeros(1, 2, 2, 128, dtype=torch.bfloat16, device="cuda")
    seq = torch.tensor([66], dtype=torch.int32, device="cuda")
    with pytest.raises(B.TQError) as e:      # n_queries = 4 needs W >= 3
        B.tq_decode_attention_multi(cfg, tables, 0, q, 1.0, kp, vp, seq, 66, out, ws,
                                    k_win=kw, v_win=kw)
    assert e.value.status == 2


@pytest.mark.parametrize("mode,W", [("mse", 16), ("sign", 16), ("qjl", 0)])
def test_decode_step_with_host_mapped_inputs_and_output(B, mode, W):
    """The query, the new tokens and the output of tq_decode_step may be
    pinned host memory, which the kernel reads and writes across the host
    link.  Planes, ring and output must be bit-identical to the same step on
    device buffers."""
    import torch
    from kv_cache_quantization_random_gb300 import workloads as W_
    T0 = np.array([299, 37, max(W - 1, 0)], dtype=np.int64)
    batch, hkv, hq, C = len(T0), 2, 8, 300
    w = W_.scaled(W_.get("llama8b_32k"), batch=batch, n_q_heads=hq, n_kv_heads=hkv, context=C,
                  data_seed=23)
    K, V = W_.make_kv(w)
    q = W_.make_q(w)
    km = {"mse": B.TQ_MODE_MSE, "sign": B.TQ_MODE_MSE_SIGN, "qjl": B.TQ_MODE_MSE_QJL}[mode]
    cfg = B.Config(k_bits=4, v_bits=2, k_mode=km, residual_window=W, seed=8)
    tables = B.device_tables(cfg)
    Kd, Vd = K.cuda(), V.cuda()
    caches = []
    for _ in range(2):
        kp, vp = B.Planes(cfg, 0, 0, batch, hkv, C), B.Planes(cfg, 0, 1, batch, hkv, C)
        B.tq_quantize_kv(cfg, tables, 0, 0, Kd[:, :, :C - 1], kp)
        B.tq_quantize_kv(cfg, tables, 0, 1, Vd[:, :, :C - 1], vp)
        kw = torch.zeros(batch, hkv, max(W, 1), 128, dtype=torch.bfloat16, device="cuda")
        vw = torch.zeros_like(kw)
        for b in range(batch):
            for t in range(max(int(T0[b]) - W, 0), int(T0[b])):
                kw[b, :, t % W] = Kd[b, :, t]
                vw[b, :, t % W] = Vd[b, :, t]
        caches.append((kp, vp, kw if W else None, vw if W else None))
    kn = torch.stack([K[b, :, int(T0[b]):int(T0[b]) + 1] for b in range(batch)])
    vn = torch.stack([V[b, :, int(T0[b]):int(T0[b]) + 1] for b in range(batch)])
    before = torch.tensor(T0, dtype=torch.int32, device="cuda")
    ws = B.new_workspace(cfg, batch, hq, hkv, C)
    out_d = torch.empty(batch, hq, 128, device="cuda")
    out_h = torch.full((batch, hq, 128), float("nan")).pin_memory()
    kp, vp, kw, vw = caches[0]
    B.tq_decode_step(cfg, tables, 0, q.cuda(), w.softmax_scale, kn.cuda(), vn.cuda(), before, C,
                     kp, vp, out_d, ws, k_win=kw, v_win=vw)
    kp, vp, kw, vw = caches[1]
    B.tq_decode_step(cfg, tables, 0, q.pin_memory(), w.softmax_scale, kn.pin_memory(),
                     vn.pin_memory(), before, C, kp, vp, out_h, ws, k_win=kw, v_win=vw)
    torch.cuda.synchronize()
    assert B.tq_get_device_error() == B.TQ_OK
    (ka, va, kwa, vwa), (kb_, vb_, kwb, vwb) = caches
    for Pa, Pb in ((ka, kb_), (va, vb_)):
        assert torch.equal(Pa.codes.cpu(), Pb.codes.cpu())
        assert torch.equal(Pa.norms.cpu(), Pb.norms.cpu())
        if Pa.qjl_signs is not None:
            assert torch.equal(Pa.qjl_signs.cpu(), Pb.qjl_signs.cpu())
    if W:
        assert torch.equal(kwa.cpu(), kwb.cpu()) and torch.equal(vwa.cpu(), vwb.cpu())
    assert torch.equal(out_h, out_d.cpu())


@pytest.mark.parametrize("kb,vb,mode,W,rep,f32", [(4, 2, "mse", 16, 1, False),
                                                  (3, 3, "mse", 0, 1, False),
                                                  (4, 2, "mse", 0, 1, True),
                                                  (2, 3, "qjl", 0, 1, False),
                                                  (2, 3, "qjl", 16, 1, False),
                                                  (2, 3, "sign", 16, 1, False),
                                                  (3, 2, "sign", 0, 1, True),
                                                  (8, 8, "mse", 8, 1, False),
                                                  (4, 2, "mse", 128, 1, False),
                                                  (4, 2, "mse", 16, 2, False),
                                                  (4, 2, "mse", 16, 14, False),
                                                  (2, 3, "qjl", 0, 20, False)])
def test_decode_step_matches_append_then_decode(B, kb, vb, mode, W, rep, f32):
    """tq_decode_step (append of one token per sequence and decode, in one
    launch) writes the same planes and ring as tq_append_kv and returns the
    output of tq_decode_attention after it, within the decode tolerance (the
    token the step quantizes enters its attention through fp32 dequantized
    operands, not fp16 MMA operands).  The plane rows the append writes are
    zeroed beforehand, so a decode that read them before they were written
    would differ.  The lengths cover a token leaving the window from its ring
    slot (as the first and as the last row of the quantized part), a ring slot
    that held no token (T0 < W), and W = 0 (the new token goes straight to the
    planes, from bf16 or fp32 rows); keys in MSE, Direct Sign and QJL mode.
    rep = 2 gives 24 (sequence, kv-head) pairs; rep = 14 gives 168 and rep =
    20 gives 240, whose one-launch plans would take two waves (one CTA per SM
    for these MSE keys, three for these QJL keys), so the step takes two
    launches."""
    import torch
    from kv_cache_quantization_random_gb300 import workloads as W_
    T0 = np.tile(np.array([699, max(W - 1, 0), W, 0, 37, 300], dtype=np.int64), rep)
    batch, hkv, hq, C = len(T0), 2, 8, 700
    w = W_.scaled(W_.get("llama8b_32k"), batch=batch, n_q_heads=hq, n_kv_heads=hkv, context=C,
                  data_seed=17)
    K, V = W_.make_kv(w)
    q = W_.make_q(w).cuda()
    km = {"mse": B.TQ_MODE_MSE, "sign": B.TQ_MODE_MSE_SIGN, "qjl": B.TQ_MODE_MSE_QJL}[mode]
    cfg = B.Config(k_bits=kb, v_bits=vb, k_mode=km, residual_window=W, seed=6)
    tables = B.device_tables(cfg)
    Kd, Vd = K.cuda(), V.cuda()
    caches = []
    for _ in range(2):
        kp, vp = B.Planes(cfg, 0, 0, batch, hkv, C), B.Planes(cfg, 0, 1, batch, hkv, C)
        B.tq_quantize_kv(cfg, tables, 0, 0, Kd[:, :, :C - 1], kp)
        B.tq_quantize_kv(cfg, tables, 0, 1, Vd[:, :, :C - 1], vp)
        for b in range(batch):                    # rows the step's append writes, and later ones
            r0 = max(int(T0[b]) - W, 0)
            for P in (kp, vp):
                P.codes_view()[b, :, r0:] = 0
                P.norms_view()[b, :, r0:] = 0
                if P.qjl_signs is not None:
                    P.signs_view()[b, :, r0:] = 0
                    P.rnorm_view()[b, :, r0:] = 0
        kw = torch.zeros(batch, hkv, max(W, 1), 128, dtype=torch.bfloat16, device="cuda")
        vw = torch.zeros_like(kw)
        for b in range(batch):
            for t in range(max(int(T0[b]) - W, 0), int(T0[b])):
                kw[b, :, t % W] = Kd[b, :, t]
                vw[b, :, t % W] = Vd[b, :, t]
        caches.append((kp, vp, kw if W else None, vw if W else None))
    kn = torch.stack([K[b, :, int(T0[b]):int(T0[b]) + 1] for b in range(batch)]).cuda()
    vn = torch.stack([V[b, :, int(T0[b]):int(T0[b]) + 1] for b in range(batch)]).cuda()
    if f32:
        kn, vn = kn.float(), vn.float()
    before = torch.tensor(T0, dtype=torch.int32, device="cuda")
    after = before + 1
    ws = B.new_workspace(cfg, batch, hq, hkv, C)
    assert B.tq_decode_step_launches(cfg, 0, batch, hq, hkv, C) == (2 if rep > 2 else 1)
    outs = [torch.empty(batch, hq, 128, device="cuda") for _ in range(2)]
    kp, vp, kw, vw = caches[0]
    B.tq_append_kv(cfg, tables, 0, kn, vn, before, kw, vw, kp, vp)
    B.tq_decode_attention(cfg, tables, 0, q, w.softmax_scale, kp, vp, after, C, outs[0], ws,
                          k_win=kw, v_win=vw)
    kp, vp, kw, vw = caches[1]
    B.tq_decode_step(cfg, tables, 0, q, w.softmax_scale, kn, vn, before, C, kp, vp, outs[1], ws,
                     k_win=kw, v_win=vw)
    torch.cuda.synchronize()
    assert B.tq_get_device_error() == B.TQ_OK
    (ka, va, kwa, vwa), (kb_, vb_, kwb, vwb) = caches
    for Pa, Pb in ((ka, kb_), (va, vb_)):
        assert torch.equal(Pa.codes.cpu(), Pb.codes.cpu())
        assert torch.equal(Pa.norms.cpu(), Pb.norms.cpu())
        if Pa.qjl_signs is not None:
            assert torch.equal(Pa.qjl_signs.cpu(), Pb.qjl_signs.cpu())
            assert torch.equal(Pa.qjl_rnorm.cpu(), Pb.qjl_rnorm.cpu())
    if W:
        assert torch.equal(kwa.cpu(), kwb.cpu()) and torch.equal(vwa.cpu(), vwb.cpu())
    a, b = to64(outs[0]), to64(outs[1])
    assert rel_l2_per_head(b, a).max() < 2e-3
